// no_alloc.cu -- hkv_insert_or_assign_noalloc: insert_or_assign whose
// working memory is a fixed array compiled into the library, so the call
// itself never allocates.
//
// Why it exists: hkv_insert_or_assign takes its per-call working memory (the
// de-duplication map and the per-bucket grouping arrays) from a stream-
// ordered pool.  Some callers cannot let a library allocate device memory:
// a serving loop that must never enter the allocator (cudaMalloc/cudaFree can
// synchronise the device and take driver locks), a process whose memory is
// fully handed out up front to a framework's caching allocator, or a host
// that accounts for every byte of a fixed device-memory budget.  This entry
// point runs the same kernels with that working memory in a file-scope
// __device__ array instead.
//
// The array lives in this translation unit's module; each GPU that loads the
// module keeps its HKV_NOALLOC_SCRATCH_BYTES until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// a device (with that device current) asks the runtime for the address with
// cudaGetSymbolAddress and caches it per device.  The cache is not refreshed:
// after cudaDeviceReset the module may be loaded at another address, so the
// header tells callers not to use this function on a reset device.
#include <mutex>

#include "hkv.h"
#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[HKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on `device`, which must be current
// (set-up on the first call per device).
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

}  // namespace

extern "C" hkv_status hkv_insert_or_assign_noalloc(hkv_table* table, uint64_t n,
                                                   const uint64_t* keys, const float* values,
                                                   const uint64_t* scores, void* stream) {
  return hkv::NoAllocAccess::run(table, n, keys, values, scores, stream, &scratch_address);
}
