// find.cu -- the reader kernel: HierarchicalKV Algorithm 1 (digest-accelerated
// find) and its two-bucket form for dual mode (HKV §3.4, "two fixed-length
// transactions").
//
// Mapping on sm_103a: one 8-lane tile per key.  Each lane loads 16 bytes of
// the bucket's 128-byte digest line, so the tile reads the line with a single
// coalesced request; the byte compare is a SWAR zero-byte test (the role of
// the paper's 32 x __vcmpeq4).  A lane whose bytes match confirms the key
// with one 16-byte (key, score) load; a tile ballot picks the hit.  The same 8 lanes then
// move the value row in 16-byte vectors (one 128-byte row per instruction)
// with streaming stores.  The grid is a multiple of the SM count and each
// tile walks keys with a grid stride, loading its next keys one iteration
// ahead.
#include "launch.h"

namespace hkv {
namespace {

#ifndef HKV_FIND_KEYS_PER_TILE
#define HKV_FIND_KEYS_PER_TILE 2
#endif
#ifndef HKV_FIND_MIN_BLOCKS
#define HKV_FIND_MIN_BLOCKS 4
#endif
#ifndef HKV_FIND_NO_DIGEST
#define HKV_FIND_NO_DIGEST 0
#endif

constexpr int kFindKeysPerTile = HKV_FIND_KEYS_PER_TILE;

// Digest ablation (HKV §5.4, Table 7): the same probe without the digest
// line.  The tile compares the key against every slot's key: lane `sub`
// reads the (key, score) pairs of slots sub, sub+8, ..., 16 bytes per lane
// and 128 bytes per tile per step, until a step finds the key (a hit reads on
// average half of the bucket's 2 KiB of pairs, a miss all of it).  Built only
// with -DHKV_FIND_NO_DIGEST, for the ablation measurement.
template <int U>
__device__ __forceinline__ void tile_scan_many(const TableView& t, const uint64_t (&b)[U],
                                               const uint64_t (&k)[U], const bool (&act)[U],
                                               unsigned sub, unsigned tmask, int (&slot)[U],
                                               uint64_t (&score)[U]) {
  int hit[U];
  uint64_t hs[U];
  bool open[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    hit[u] = -1;
    hs[u] = 0;
    open[u] = act[u];
  }
  for (int c = 0; c < kSlots / 8; ++c) {
    ulonglong2 p[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (open[u]) p[u] = ld_nc_pair(key_at(t, b[u] * kSlots + c * 8 + sub));
    bool more = false;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (open[u] && p[u].x == k[u]) {
        hit[u] = c * 8 + static_cast<int>(sub);
        hs[u] = p[u].y;
      }
      open[u] = open[u] && !(__ballot_sync(tmask, hit[u] >= 0) & tmask);
      more = more || open[u];
    }
    if (!more) break;
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const unsigned bal = __ballot_sync(tmask, hit[u] >= 0) & tmask;
    const int lead = bal ? __ffs(bal) - 1 : static_cast<int>(lane_id());
    slot[u] = bal ? __shfl_sync(tmask, hit[u], lead) : -1;
    score[u] = __shfl_sync(tmask, hs[u], lead);
  }
}

// What a find writes per key besides the found flag (and the score).
enum FindOut { kOutValues = 0, kOutNone = 1, kOutPointer = 2 };

// One 8-lane tile handles U keys per iteration: keys i, i+T, ..., i+(U-1)T
// for T tiles in the grid; the next iteration's keys are loaded at the top
// of the current one.
template <bool kDual, int U, int kOut>
__global__ void __launch_bounds__(256, HKV_FIND_MIN_BLOCKS)
    find_kernel(TableView t, uint64_t n, const uint64_t* keys, float* values_out,
                float** ptrs_out, uint8_t* found_out, uint64_t* scores_out, bool vec) {
  pdl_wait();
  pdl_trigger();
  const unsigned lane = lane_id();
  const unsigned sub = lane & 7u;
  const unsigned tmask = 0xFFu << (lane & 24u);
  const uint64_t tiles = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 3;
  unsigned long long reserved = 0;
  uint64_t i0 = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  uint64_t kn[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint64_t i = i0 + u * tiles;
    kn[u] = i < n ? keys[i] : kEmptyKey;
  }
  for (; i0 < n; i0 += tiles * U) {
    uint64_t k[U], b[U];
    uint32_t pat[U];
    bool act[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      k[u] = kn[u];
      const uint64_t i = i0 + (U + u) * tiles;
      kn[u] = i < n ? keys[i] : kEmptyKey;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t i = i0 + u * tiles;
      act[u] = i < n && !is_reserved(k[u]);
      if (i < n && !act[u] && sub == 0) ++reserved;
      const uint64_t h = hash64(k[u]);
      pat[u] = digest_of_hash(h) * 0x01010101u;
      b[u] = bucket_of_hash(t, h);
    }
    int slot[U];
    uint64_t sc[U];
#if HKV_FIND_NO_DIGEST
    tile_scan_many<U>(t, b, k, act, sub, tmask, slot, sc);
#else
    tile_probe_many<U>(t, b, k, pat, act, sub, tmask, slot, sc);
#endif
    if (kDual) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (act[u] && slot[u] < 0) {
          b[u] = bucket2_of(t, k[u], b[u]);
          slot[u] = tile_probe<true>(t, b[u], k[u], pat[u], sub, tmask);
          if (slot[u] >= 0) sc[u] = ld_nc_u64(score_at(t, b[u] * kSlots + slot[u]));
        }
      }
    }
    if (kOut == kOutValues) {
      // Value rows: U loads in flight, then U streaming stores.
      const float* src[U];
      float* dst[U];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        ok[u] = slot[u] >= 0;
        src[u] = ok[u] ? row_ptr(t, b[u] * kSlots + slot[u]) : nullptr;
        dst[u] = values_out + (i0 + u * tiles) * t.dim;
      }
      tile_copy_rows<U>(dst, src, ok, t.dim, sub, vec);
    }
    if (sub == 0) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint64_t i = i0 + u * tiles;
        if (i >= n) continue;
        found_out[i] = slot[u] >= 0 ? 1 : 0;
        const uint64_t row = b[u] * kSlots + static_cast<uint64_t>(slot[u]);
        if (kOut == kOutPointer) ptrs_out[i] = slot[u] >= 0 ? row_ptr(t, row) : nullptr;
        if (slot[u] >= 0 && scores_out) scores_out[i] = sc[u];
      }
    }
  }
  if (reserved) atomicAdd(&t.stats->reserved, reserved);
}

template <bool kDual, int U, int kOut>
cudaError_t launch_find_u(const TableView& t, uint64_t n, const uint64_t* keys, float* values_out,
                          float** ptrs_out, uint8_t* found_out, uint64_t* scores_out, bool vec,
                          cudaStream_t st) {
  const int threads = 256;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, find_kernel<kDual, U, kOut>, threads, 0);
  if (per_sm < 1) per_sm = 1;
  uint64_t blocks = (n * 8 + threads * U - 1) / (threads * U);
  const uint64_t cap = static_cast<uint64_t>(sm_count()) * per_sm;
  if (blocks > cap) blocks = cap;
  return launch_chained(find_kernel<kDual, U, kOut>, static_cast<unsigned>(blocks), threads, 0, st,
                        t, n, keys, values_out, ptrs_out, found_out, scores_out, vec);
}

template <int kOut>
cudaError_t launch_find_mode(const TableView& t, uint64_t n, const uint64_t* keys,
                             float* values_out, float** ptrs_out, uint8_t* found_out,
                             uint64_t* scores_out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const bool vec = (t.dim % 4 == 0) && ((reinterpret_cast<uintptr_t>(values_out) & 15) == 0);
  if (t.dual)
    return launch_find_u<true, kFindKeysPerTile, kOut>(t, n, keys, values_out, ptrs_out,
                                                        found_out, scores_out, vec, st);
  return launch_find_u<false, kFindKeysPerTile, kOut>(t, n, keys, values_out, ptrs_out, found_out,
                                                       scores_out, vec, st);
}

}  // namespace

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 148;
  }
  return cached[dev];
}

cudaError_t launch_find(const TableView& t, uint64_t n, const uint64_t* keys, float* values_out,
                        uint8_t* found_out, uint64_t* scores_out, cudaStream_t st) {
  return launch_find_mode<kOutValues>(t, n, keys, values_out, nullptr, found_out, scores_out, st);
}

cudaError_t launch_contains(const TableView& t, uint64_t n, const uint64_t* keys,
                            uint8_t* found_out, cudaStream_t st) {
  return launch_find_mode<kOutNone>(t, n, keys, nullptr, nullptr, found_out, nullptr, st);
}

cudaError_t launch_find_ptr(const TableView& t, uint64_t n, const uint64_t* keys, float** ptrs_out,
                            uint8_t* found_out, uint64_t* scores_out, cudaStream_t st) {
  return launch_find_mode<kOutPointer>(t, n, keys, nullptr, ptrs_out, found_out, scores_out, st);
}

}  // namespace hkv
