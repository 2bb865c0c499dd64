// access_probe.cu -- measurement helper for the benchmark (not part of the
// table library; built as its own libhkv_probe.so).
//
// The table's kernels are bound by random DRAM accesses (a digest line, a
// key/score sector and a value row per key at unpredictable addresses), not by
// streaming bandwidth.  This probe measures what the GPU sustains for that
// access pattern: reads of `granule` bytes at uniformly random, granule-
// aligned offsets of a buffer far larger than L2.  Granules of 32 bytes are
// read one per lane; larger granules by 8-lane tiles, 16 bytes per lane, the
// way the table kernels read digest lines and value rows.  Each thread or
// tile keeps kInFlight independent reads outstanding.
//
// Offsets come from a fixed integer mix of (thread, iteration) reduced modulo
// the number of granules, so every read stays inside the buffer.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr int kInFlight = 4;

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  x ^= x >> 33;
  x *= 0xff51afd7ed558ccdull;
  x ^= x >> 33;
  x *= 0xc4ceb9fe1a85ec53ull;
  x ^= x >> 33;
  return x;
}

__global__ void sector_reads(const uint8_t* buf, uint64_t granules, uint64_t iters,
                             unsigned long long* sink) {
  const uint64_t tid = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x;
  unsigned long long acc = 0;
  for (uint64_t it = 0; it < iters; ++it) {
    unsigned long long v[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const uint64_t g = mix64(tid * 0x9E3779B97F4A7C15ull + it * kInFlight + u) % granules;
      v[u] = __ldcg(reinterpret_cast<const unsigned long long*>(buf + g * 32));
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) acc ^= v[u];
  }
  if (acc == 0x5EEDull) *sink = acc;  // keeps the loads
}

__global__ void line_reads(const uint8_t* buf, uint64_t granules, uint32_t granule, uint64_t iters,
                           unsigned long long* sink) {
  const uint64_t tile = (blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x) >> 3;
  const uint32_t sub = threadIdx.x & 7u;
  uint32_t acc = 0;
  for (uint64_t it = 0; it < iters; ++it) {
    uint4 v[kInFlight];
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      v[u] = make_uint4(0, 0, 0, 0);
      const uint64_t g = mix64(tile * 0xD1B54A32D192ED03ull + it * kInFlight + u) % granules;
      const uint8_t* p = buf + g * granule;
      for (uint32_t c = sub; c < granule / 16; c += 8) {
        const uint4 w = __ldcg(reinterpret_cast<const uint4*>(p + 16 * c));
        v[u].x ^= w.x;
        v[u].w ^= w.w;
      }
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) acc ^= v[u].x ^ v[u].w;
  }
  if (acc == 0x5EEDu) *sink = acc;
}

}  // namespace

extern "C" {

// Measures random reads of `granule` bytes (32, or a multiple of 16 from 48
// to 4096) over a freshly allocated device buffer of `buffer_bytes` on the
// current device.  Writes the reads per second to *reads_per_s.  Returns 0,
// -1 on bad arguments, or the CUDA error code.  Allocates and frees its
// buffer; synchronises the device.
int hkv_probe_random_reads(uint32_t granule, uint64_t buffer_bytes, double* reads_per_s) {
  const bool ok_granule = granule == 32 || (granule % 16 == 0 && granule >= 48 && granule <= 4096);
  if (!reads_per_s || !ok_granule || buffer_bytes < (64ull << 20)) return -1;
  uint8_t* buf = nullptr;
  unsigned long long* sink = nullptr;
  cudaError_t e = cudaMalloc(&buf, buffer_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&sink, sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(buf, 1, buffer_bytes);
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaEvent_t a = nullptr, b = nullptr;
  if (e == cudaSuccess) e = cudaEventCreate(&a);
  if (e == cudaSuccess) e = cudaEventCreate(&b);
  if (e == cudaSuccess) {
    const unsigned threads = 256, grid = static_cast<unsigned>(sms) * 8;
    const uint64_t granules = buffer_bytes / granule;
    const uint64_t iters = 32;
    auto launch = [&]() {
      if (granule == 32)
        sector_reads<<<grid, threads>>>(buf, granules, iters, sink);
      else
        line_reads<<<grid, threads>>>(buf, granules, granule, iters, sink);
    };
    launch();  // warm-up
    cudaEventRecord(a);
    launch();
    cudaEventRecord(b);
    e = cudaEventSynchronize(b);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
    if (e == cudaSuccess) e = cudaGetLastError();
    const double lanes_per_read = granule == 32 ? 1.0 : 8.0;
    const double reads = static_cast<double>(grid) * threads / lanes_per_read * iters * kInFlight;
    if (e == cudaSuccess) *reads_per_s = ms > 0.f ? reads / (ms * 1e-3) : 0.0;
  }
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  if (buf) cudaFree(buf);
  if (sink) cudaFree(sink);
  return e == cudaSuccess ? 0 : static_cast<int>(e);
}

}  // extern "C"
