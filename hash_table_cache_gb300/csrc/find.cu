// find.cu -- the reader kernel: HierarchicalKV Algorithm 1 (digest-accelerated
// find) and its two-bucket form for dual mode (HKV §3.4, "two fixed-length
// transactions").
//
// Mapping on sm_103a: one 8-lane tile per key.  Each lane loads 16 bytes of
// the bucket's 128-byte digest line, so the tile reads the line with a single
// coalesced request; the byte compare is a SWAR zero-byte test (the role of
// the paper's 32 x __vcmpeq4).  A lane whose bytes match confirms the key
// with one 8-byte load; a tile ballot picks the hit.  The same 8 lanes then
// move the value row in 16-byte vectors (one 128-byte row per instruction)
// with streaming stores.  The grid is a multiple of the SM count and each
// tile walks keys with a grid stride, prefetching its next key.
#include "launch.h"

namespace hkv {
namespace {

template <bool kDual>
__global__ void __launch_bounds__(256) find_kernel(TableView t, uint64_t n, const uint64_t* keys,
                                                   float* values_out, uint8_t* found_out,
                                                   uint64_t* scores_out, bool vec) {
  const unsigned lane = lane_id();
  const unsigned sub = lane & 7u;
  const unsigned tmask = 0xFFu << (lane & 24u);
  const uint64_t tiles = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 3;
  uint64_t i = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  uint64_t key = i < n ? keys[i] : 0;
  unsigned long long reserved = 0;
  for (; i < n; i += tiles) {
    const uint64_t k = key;
    if (i + tiles < n) key = keys[i + tiles];  // prefetch the next key of this tile
    int slot = -1;
    uint64_t b = 0;
    if (!is_reserved(k)) {
      const uint64_t h = hash64(k);
      const uint32_t pat = digest_of_hash(h) * 0x01010101u;
      b = bucket_of_hash(t, h);
      slot = tile_probe<true>(t, b, k, pat, sub, tmask);
      if (kDual && slot < 0) {
        b = bucket2_of(t, k, b);
        slot = tile_probe<true>(t, b, k, pat, sub, tmask);
      }
    } else if (sub == 0) {
      ++reserved;
    }
    if (slot >= 0) {
      const uint64_t row = b * kSlots + static_cast<uint64_t>(slot);
      tile_copy_row(values_out + i * t.dim, row_ptr(t, row), t.dim, sub, vec, true);
      if (sub == 0) {
        found_out[i] = 1;
        if (scores_out) scores_out[i] = t.scores[row];
      }
    } else if (sub == 0) {
      found_out[i] = 0;
    }
  }
  if (reserved) atomicAdd(&t.stats->reserved, reserved);
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
  if (n == 0) return cudaSuccess;
  const int threads = 256;
  const uint64_t tiles_needed = n;
  uint64_t blocks = (tiles_needed * 8 + threads - 1) / threads;
  const uint64_t cap = static_cast<uint64_t>(sm_count()) * 8;  // 8 blocks of 256 per SM
  if (blocks > cap) blocks = cap;
  const bool vec = (t.dim % 4 == 0) && ((reinterpret_cast<uintptr_t>(values_out) & 15) == 0);
  if (t.dual)
    find_kernel<true><<<static_cast<unsigned>(blocks), threads, 0, st>>>(t, n, keys, values_out,
                                                                          found_out, scores_out, vec);
  else
    find_kernel<false><<<static_cast<unsigned>(blocks), threads, 0, st>>>(t, n, keys, values_out,
                                                                           found_out, scores_out, vec);
  return cudaGetLastError();
}

}  // namespace hkv
