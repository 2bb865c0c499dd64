// access_probe.cu -- measurement helper for the benchmark (not part of the
// table library; built as its own libhkv_probe.so).
//
// The table's kernels are bound by random DRAM accesses (a digest line, a
// key/score sector and a value row per key at unpredictable addresses), not by
// streaming bandwidth.  This probe measures what the GPU sustains for that
// access pattern: reads of `granule` bytes at uniformly random, granule-
// aligned offsets of a buffer far larger than L2.  Granules of 32 bytes are
// read one per lane; larger granules by 8-lane tiles, 16 bytes per lane per
// 128 bytes, the way the table kernels read digest lines and value rows.
// Each thread or tile keeps D independent reads outstanding (D = 1..16), and
// the grid holds a chosen number of 256-thread blocks per SM, so the rate can
// be swept over the number of reads in flight until it stops growing.
//
// The buffer size is a power of two and offsets are a fixed integer mix of
// (thread, iteration) masked to the granule count, so every read stays inside
// the buffer and the address arithmetic costs a few instructions.
//
// A second probe measures the host link the way tiered mode uses it: SM loads
// and stores (not copy-engine transfers) of 16-byte vectors over mapped
// pinned host memory, either streaming (consecutive addresses) or as random
// rows of `granule` bytes.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  x ^= x >> 33;
  x *= 0xff51afd7ed558ccdull;
  x ^= x >> 33;
  x *= 0xc4ceb9fe1a85ec53ull;
  x ^= x >> 33;
  return x;
}

template <int D>
__global__ void sector_reads(const uint8_t* buf, uint64_t mask, uint32_t iters,
                             unsigned long long* sink) {
  const uint64_t tid = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x;
  unsigned long long acc = 0;
  for (uint32_t it = 0; it < iters; ++it) {
    unsigned long long v[D];
#pragma unroll
    for (int u = 0; u < D; ++u) {
      const uint64_t g = mix64(tid * 0x9E3779B97F4A7C15ull + it * D + u) & mask;
      v[u] = __ldcg(reinterpret_cast<const unsigned long long*>(buf + g * 32));
    }
#pragma unroll
    for (int u = 0; u < D; ++u) acc ^= v[u];
  }
  if (acc == 0x5EEDull) *sink = acc;  // keeps the loads
}

// Tile reads: granule = 128 * C bytes is read as C 16-byte loads per lane
// (granules of 48..112 bytes: lanes past the end stay idle).
template <int D, int C>
__global__ void line_reads(const uint8_t* buf, uint64_t mask, uint32_t granule, uint32_t iters,
                           unsigned long long* sink) {
  const uint64_t tile = (blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x) >> 3;
  const uint32_t sub = threadIdx.x & 7u;
  const uint32_t vecs = granule / 16;
  uint32_t acc = 0;
  for (uint32_t it = 0; it < iters; ++it) {
    uint4 v[D][C];
#pragma unroll
    for (int u = 0; u < D; ++u) {
      const uint64_t g = mix64(tile * 0xD1B54A32D192ED03ull + it * D + u) & mask;
      const uint8_t* p = buf + g * granule;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        const uint32_t q = sub + 8u * c;
        v[u][c] = q < vecs ? __ldcg(reinterpret_cast<const uint4*>(p + 16 * q))
                           : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < D; ++u)
#pragma unroll
      for (int c = 0; c < C; ++c) acc ^= v[u][c].x ^ v[u][c].w;
  }
  if (acc == 0x5EEDu) *sink = acc;
}

template <int D>
cudaError_t launch_reads(uint32_t granule, const uint8_t* buf, uint64_t mask, unsigned grid,
                         uint32_t iters, unsigned long long* sink) {
  if (granule == 32)
    sector_reads<D><<<grid, 256>>>(buf, mask, iters, sink);
  else if (granule <= 128)
    line_reads<D, 1><<<grid, 256>>>(buf, mask, granule, iters, sink);
  else if (granule <= 256)
    line_reads<D, 2><<<grid, 256>>>(buf, mask, granule, iters, sink);
  else
    line_reads<D, 4><<<grid, 256>>>(buf, mask, granule, iters, sink);
  return cudaGetLastError();
}

cudaError_t launch_depth(int depth, uint32_t granule, const uint8_t* buf, uint64_t mask,
                         unsigned grid, uint32_t iters, unsigned long long* sink) {
  switch (depth) {
    case 1: return launch_reads<1>(granule, buf, mask, grid, iters, sink);
    case 2: return launch_reads<2>(granule, buf, mask, grid, iters, sink);
    case 4: return launch_reads<4>(granule, buf, mask, grid, iters, sink);
    case 8: return launch_reads<8>(granule, buf, mask, grid, iters, sink);
    default: return launch_reads<16>(granule, buf, mask, grid, iters, sink);
  }
}

// Host-link probe kernels: 16-byte SM loads / stores over host memory, with
// the instructions the table's kernels use for rows of the host slab (plain
// loads, streaming stores; loads through the read-only path reach half the
// rate).  Streaming: the grid walks the buffer in consecutive 16-byte vectors.
__device__ __forceinline__ uint4 ld_row_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ void st_row_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__global__ void host_stream_read(const uint4* p, uint64_t nvec, unsigned long long* sink) {
  uint32_t acc = 0;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < nvec;
       i += stride) {
    const uint4 w = ld_row_v4(p + i);
    acc ^= w.x ^ w.w;
  }
  if (acc == 0x5EEDu) *sink = acc;
}

__global__ void host_stream_write(uint4* p, uint64_t nvec) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < nvec;
       i += stride)
    st_row_v4(p + i, make_uint4(static_cast<uint32_t>(i), 1u, 2u, 3u));
}

// Random rows of `granule` bytes (a multiple of 16, at most 512), one row per
// 8-lane tile at a time, 4 rows in flight per tile; row indices uniform in
// [0, rows) (the high half of a 64x64-bit product, always below rows).
__global__ void host_row_read(const uint8_t* p, uint64_t rows, uint32_t granule,
                              uint32_t iters, unsigned long long* sink) {
  const uint64_t tile = (blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x) >> 3;
  const uint32_t sub = threadIdx.x & 7u;
  const uint32_t vecs = granule / 16;
  uint32_t acc = 0;
  for (uint32_t it = 0; it < iters; ++it) {
    uint4 v[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint64_t g = __umul64hi(mix64(tile * 0xD1B54A32D192ED03ull + it * 4 + u), rows);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t q = sub + 8u * c;
        v[u][c] = q < vecs ? ld_row_v4(p + g * granule + 16 * q) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc ^= v[u][c].x ^ v[u][c].w;
  }
  if (acc == 0x5EEDu) *sink = acc;
}

__global__ void host_row_write(uint8_t* p, uint64_t rows, uint32_t granule, uint32_t iters) {
  const uint64_t tile = (blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x) >> 3;
  const uint32_t sub = threadIdx.x & 7u;
  const uint32_t vecs = granule / 16;
  for (uint32_t it = 0; it < iters; ++it) {
    const uint64_t g = __umul64hi(mix64(tile * 0xD1B54A32D192ED03ull + it), rows);
    for (uint32_t q = sub; q < vecs; q += 8)
      st_row_v4(p + g * granule + 16 * q, make_uint4(it, 1u, 2u, 3u));
  }
}

bool pow2(uint64_t x) { return x && !(x & (x - 1)); }

struct Timer {
  cudaEvent_t a = nullptr, b = nullptr;
  cudaError_t init() {
    cudaError_t e = cudaEventCreate(&a);
    return e == cudaSuccess ? cudaEventCreate(&b) : e;
  }
  ~Timer() {
    if (a) cudaEventDestroy(a);
    if (b) cudaEventDestroy(b);
  }
};

}  // namespace

extern "C" {

// Measures random reads of `granule` bytes (32, or a multiple of 16 from 48
// to 512) over a freshly allocated device buffer of `buffer_bytes` (a power
// of two, at least 64 MiB) on the current device, with `in_flight` (1, 2, 4,
// 8 or 16) independent reads outstanding per thread (32-byte granules) or per
// 8-lane tile (larger granules) and `blocks_per_sm` (1..8) blocks of 256
// threads per SM.  Writes the reads per second to *reads_per_s.  Returns 0,
// -1 on bad arguments, or the CUDA error code.  Allocates and frees its
// buffer; synchronises the device.
int hkv_probe_random_reads_at(uint32_t granule, uint64_t buffer_bytes, int in_flight,
                              int blocks_per_sm, double* reads_per_s) {
  const bool ok_granule = granule == 32 || (granule % 16 == 0 && granule >= 48 && granule <= 512);
  const bool ok_depth = in_flight == 1 || in_flight == 2 || in_flight == 4 || in_flight == 8 ||
                        in_flight == 16;
  if (!reads_per_s || !ok_granule || !ok_depth || blocks_per_sm < 1 || blocks_per_sm > 8 ||
      !pow2(buffer_bytes) || buffer_bytes < (64ull << 20))
    return -1;
  uint8_t* buf = nullptr;
  unsigned long long* sink = nullptr;
  cudaError_t e = cudaMalloc(&buf, buffer_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&sink, sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(buf, 1, buffer_bytes);
  int dev = 0, sms = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  Timer tm;
  if (e == cudaSuccess) e = tm.init();
  if (e == cudaSuccess) {
    const unsigned grid = static_cast<unsigned>(sms) * blocks_per_sm;
    // power-of-two granule count: the largest power of two of granules that
    // fits the buffer
    uint64_t granules = 1;
    while (granules * 2 * granule <= buffer_bytes) granules *= 2;
    const uint64_t mask = granules - 1;
    const double lanes_per_read = granule == 32 ? 1.0 : 8.0;
    // about 2^24 reads per launch, whatever the depth and the grid
    const double per_iter = static_cast<double>(grid) * 256 / lanes_per_read * in_flight;
    uint32_t iters = static_cast<uint32_t>((1 << 24) / per_iter);
    if (iters < 4) iters = 4;
    e = launch_depth(in_flight, granule, buf, mask, grid, iters, sink);  // warm-up
    if (e == cudaSuccess) e = cudaEventRecord(tm.a);
    if (e == cudaSuccess) e = launch_depth(in_flight, granule, buf, mask, grid, iters, sink);
    if (e == cudaSuccess) e = cudaEventRecord(tm.b);
    if (e == cudaSuccess) e = cudaEventSynchronize(tm.b);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, tm.a, tm.b);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) *reads_per_s = ms > 0.f ? per_iter * iters / (ms * 1e-3) : 0.0;
  }
  if (buf) cudaFree(buf);
  if (sink) cudaFree(sink);
  return e == cudaSuccess ? 0 : static_cast<int>(e);
}

// The earlier form: 4 reads in flight, 8 blocks per SM.
int hkv_probe_random_reads(uint32_t granule, uint64_t buffer_bytes, double* reads_per_s) {
  uint64_t p = 1;
  while (p * 2 <= buffer_bytes) p *= 2;
  return hkv_probe_random_reads_at(granule, p, 4, 8, reads_per_s);
}

// Pinned host memory the device reads and writes at the same address, drawn
// from a memory pool on the host NUMA node nearest the device, as a tiered
// table's value slab is.
static cudaError_t pool_host_buffer(int dev, uint64_t bytes, cudaMemPool_t* pool, void** p) {
  int numa = -1;
  if (cudaDeviceGetAttribute(&numa, cudaDevAttrHostNumaId, dev) != cudaSuccess) {
    cudaGetLastError();
    numa = -1;
  }
  cudaMemPoolProps props{};
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = numa >= 0 ? cudaMemLocationTypeHostNuma : cudaMemLocationTypeHost;
  props.location.id = numa >= 0 ? numa : 0;
  cudaError_t e = cudaMemPoolCreate(pool, &props);
  if (e != cudaSuccess) {
    *pool = nullptr;
    return e;
  }
  cudaMemAccessDesc access{};
  access.location.type = cudaMemLocationTypeDevice;
  access.location.id = dev;
  access.flags = cudaMemAccessFlagsProtReadWrite;
  e = cudaMemPoolSetAccess(*pool, &access, 1);
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(p, bytes, *pool, cudaStreamLegacy);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cudaStreamLegacy);
  return e;
}

// Measures SM access to pinned host memory, the path tiered mode's value
// rows take.  kind & 3: 0 = streaming 16-byte reads, 1 = streaming 16-byte
// writes, 2 = random reads of `granule`-byte rows, 3 = random writes of
// `granule`-byte rows (granule a multiple of 16, 16..512).  kind & 4: the
// buffer comes from a host-NUMA memory pool (as a tiered slab above
// HKV_HOST_SLAB_MAPPED_MAX does), else from cudaHostAllocMapped.
// `buffer_bytes` is a multiple of 64 MiB; the buffer is freed
// before return.  Writes to *bytes_per_s the best rate over 4, 8 and 16
// blocks of 256 threads per SM (each launch moves about buffer_bytes, at
// most 4 GiB for the random kinds; one untimed launch first).  Returns 0, -1
// on bad arguments, or the CUDA error code.  Synchronises the device.
int hkv_probe_host_link(int kind, uint32_t granule, uint64_t buffer_bytes, double* bytes_per_s) {
  if (!bytes_per_s || kind < 0 || kind > 7 || buffer_bytes == 0 ||
      buffer_bytes % (64ull << 20) != 0)
    return -1;
  const bool pooled = (kind & 4) != 0;
  kind &= 3;
  if (kind >= 2 && (granule % 16 != 0 || granule < 16 || granule > 512)) return -1;
  cudaMemPool_t pool = nullptr;
  void* host = nullptr;
  uint8_t* dp = nullptr;
  unsigned long long* sink = nullptr;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) {
    if (pooled) {
      e = pool_host_buffer(dev, buffer_bytes, &pool, reinterpret_cast<void**>(&dp));
    } else {
      e = cudaHostAlloc(&host, buffer_bytes, cudaHostAllocMapped | cudaHostAllocPortable);
      if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&dp), host, 0);
    }
  }
  if (e == cudaSuccess) e = cudaMalloc(&sink, sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  Timer tm;
  if (e == cudaSuccess) e = tm.init();
  double best = 0.0;
  const uint64_t nvec = buffer_bytes / 16;
  const uint64_t rows = buffer_bytes / granule;  // whole rows of the buffer
  for (int per_sm = 4; e == cudaSuccess && per_sm <= 16; per_sm *= 2) {
    const unsigned grid = static_cast<unsigned>(sms) * per_sm;
    const uint64_t tiles = static_cast<uint64_t>(grid) * 256 / 8;
    // random kinds: rows drawn from the whole buffer, about min(buffer_bytes,
    // 4 GiB) of them per launch
    const uint64_t moved = buffer_bytes < (4ull << 30) ? buffer_bytes : (4ull << 30);
    uint32_t iters = kind >= 2 ? static_cast<uint32_t>(moved / granule / tiles) : 0;
    if (kind == 2) iters = (iters + 3) / 4;  // 4 rows per iteration
    if (kind >= 2 && iters < 1) iters = 1;
    double bytes = 0;
    auto launch = [&]() {
      switch (kind) {
        case 0: host_stream_read<<<grid, 256>>>(reinterpret_cast<const uint4*>(dp), nvec, sink);
                bytes = static_cast<double>(buffer_bytes); break;
        case 1: host_stream_write<<<grid, 256>>>(reinterpret_cast<uint4*>(dp), nvec);
                bytes = static_cast<double>(buffer_bytes); break;
        case 2: host_row_read<<<grid, 256>>>(dp, rows, granule, iters, sink);
                bytes = static_cast<double>(tiles) * iters * 4 * granule; break;
        default: host_row_write<<<grid, 256>>>(dp, rows, granule, iters);
                 bytes = static_cast<double>(tiles) * iters * granule; break;
      }
      return cudaGetLastError();
    };
    e = launch();  // warm-up
    if (e == cudaSuccess) e = cudaEventRecord(tm.a);
    if (e == cudaSuccess) e = launch();
    if (e == cudaSuccess) e = cudaEventRecord(tm.b);
    if (e == cudaSuccess) e = cudaEventSynchronize(tm.b);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, tm.a, tm.b);
    if (e == cudaSuccess && ms > 0.f && bytes / (ms * 1e-3) > best) best = bytes / (ms * 1e-3);
  }
  if (e == cudaSuccess) *bytes_per_s = best;
  if (sink) cudaFree(sink);
  cudaDeviceSynchronize();
  if (host) cudaFreeHost(host);
  if (pool) {
    if (dp) cudaFree(dp);
    cudaMemPoolDestroy(pool);
  }
  return e == cudaSuccess ? 0 : static_cast<int>(e);
}

}  // extern "C"
