// find.cu -- the reader kernel: HierarchicalKV Algorithm 1 (digest-accelerated
// find) and its two-bucket form for dual mode (HKV §3.4, "two fixed-length
// transactions"); the same kernel serves contains and the pointer-returning
// find* (HKV §5.2-§5.3).
//
// Mapping on sm_103a: a warp takes 32 consecutive keys of the batch, one per
// lane.  Everything that is per key and not a 128-byte transfer runs one key
// per lane: the key's load, its hash, bucket and digest pattern, the
// confirmation of its candidate slots, and its found flag, score or row
// address (coalesced stores).  The 128-byte transfers run on 8-lane tiles,
// 16 bytes per lane, so each digest line and each 128 bytes of a value row
// is one request: tile j loads the digest lines of the warp's keys 8j..8j+7
// (DG lines in flight), compares their bytes with the keys' digests (a SWAR
// zero-byte test, the role of the paper's 32 x __vcmpeq4) and hands each
// key's 128-bit candidate mask to the key's lane through shared memory; the
// key's lane loads the (key, score) pairs of its first two candidate slots
// together (one 16-byte load each; the score comes with the key) and
// confirms the key; tile j then copies the value rows of its keys that were
// found, RG rows in flight, with streaming stores.  In dual mode the keys
// not found in their first bucket run the probe again on their second.
//
// Why this shape: the kernel is bound by random DRAM accesses (a key/score
// sector and a value row per hit) and needs many of them in flight.  The
// tile-per-key form spends eight lanes on every scalar step of every key;
// here those steps cost one lane, so a warp keeps up to 32 keys' accesses
// outstanding at a fraction of the instructions.
#include "launch.h"

namespace hkv {
namespace {

// Digest ablation (HKV §5.4, Table 7): -DHKV_FIND_NO_DIGEST=1 builds the
// same kernel without the digest line (libhkv_nodigest.so).
#ifndef HKV_FIND_NO_DIGEST
#define HKV_FIND_NO_DIGEST 0
#endif
// Blocks of 256 threads per SM (the register budget: 64 per thread).
#ifndef HKV_FIND_MIN_BLOCKS
#define HKV_FIND_MIN_BLOCKS 4
#endif
// Digest lines in flight per tile.
#ifndef HKV_FIND_DIGEST_GROUP
#define HKV_FIND_DIGEST_GROUP 2
#endif
// Value rows in flight per tile: rows of up to 32 floats, longer rows.
#ifndef HKV_FIND_ROW_GROUP
#define HKV_FIND_ROW_GROUP 4
#endif
#ifndef HKV_FIND_ROW_GROUP_WIDE
#define HKV_FIND_ROW_GROUP_WIDE 1
#endif

// What a find writes per key besides the found flag (and the score).
enum FindOut { kOutValues = 0, kOutNone = 1, kOutPointer = 2 };

// Row shapes: CH = 16-byte chunks per lane of a value row copied with rows
// in flight (a row of at most 8*CH chunks); kNoRow = no row copied;
// kAnyRow = any dim, one row at a time (4-byte words unless `vec`).
constexpr int kNoRow = 0;
constexpr int kAnyRow = -1;

constexpr unsigned kFull = 0xFFFFFFFFu;

#if !HKV_FIND_NO_DIGEST
// Candidate mask of this lane's 16 digest bytes: bit j set when byte j may
// equal the digest (every equal byte is set; see zero_byte_flags).
__device__ __forceinline__ uint32_t match16(const uint4& dg, uint32_t pat) {
  return byte_match4(dg.x, pat) | (byte_match4(dg.y, pat) << 4) | (byte_match4(dg.z, pat) << 8) |
         (byte_match4(dg.w, pat) << 12);
}

// Removes and returns the lowest set bit of a 128-bit mask (-1 when empty).
__device__ __forceinline__ int pop_slot(uint4& m) {
  if (m.x) {
    const int b = __ffs(m.x) - 1;
    m.x &= m.x - 1;
    return b;
  }
  if (m.y) {
    const int b = __ffs(m.y) - 1;
    m.y &= m.y - 1;
    return 32 + b;
  }
  if (m.z) {
    const int b = __ffs(m.z) - 1;
    m.z &= m.z - 1;
    return 64 + b;
  }
  if (m.w) {
    const int b = __ffs(m.w) - 1;
    m.w &= m.w - 1;
    return 96 + b;
  }
  return -1;
}

// Candidate slots of the warp's probing keys (bit s of a lane's result =
// slot s of its key's bucket `bkt`): tile j matches the digest lines of keys
// 8j..8j+7, DG lines in flight, and the masks reach the keys' lanes through
// `msk` (32 keys x 8 lanes x 16 bits).
__device__ __forceinline__ uint4 candidates(const TableView& t, unsigned probe, uint32_t bkt,
                                            uint32_t pat, unsigned lane, uint16_t (*msk)[8]) {
  const unsigned tile = lane >> 3, sub = lane & 7u;
  constexpr int DG = HKV_FIND_DIGEST_GROUP;
#pragma unroll
  for (int g = 0; g < 8; g += DG) {
    uint4 dg[DG];
#pragma unroll
    for (int m = 0; m < DG; ++m) {
      const unsigned src = tile * 8 + g + m;
      const uint32_t b = __shfl_sync(kFull, bkt, src);
      if ((probe >> src) & 1u)
        dg[m] = ld_nc_v4(t.digests + static_cast<uint64_t>(b) * kSlots + sub * 16);
    }
#pragma unroll
    for (int m = 0; m < DG; ++m) {
      const unsigned src = tile * 8 + g + m;
      const uint32_t p = __shfl_sync(kFull, pat, src);
      msk[src][sub] = static_cast<uint16_t>(((probe >> src) & 1u) ? match16(dg[m], p) : 0u);
    }
  }
  __syncwarp();
  const uint4 cand = *reinterpret_cast<const uint4*>(msk[lane]);
  __syncwarp();  // every lane has read its mask before the next probe writes
  return cand;
}
#endif

#if HKV_FIND_NO_DIGEST
// Digest ablation: the slot of each probing key found by comparing it with
// every slot's key, 8 slots (128 bytes of pairs) per tile step, two of the
// tile's keys' steps in flight together, until each key is found or its
// bucket is exhausted.  Returns the slot (or -1) and the score in the key's
// lane.
__device__ __forceinline__ int scan_without_digest(const TableView& t, unsigned probe,
                                                   uint32_t bkt, uint64_t k, unsigned lane,
                                                   uint64_t& score) {
  const unsigned tile = lane >> 3, sub = lane & 7u;
  int slot = -1;
#pragma unroll 1
  for (int g = 0; g < 8; g += 2) {
    unsigned open = 0x3u & (probe >> (tile * 8 + g));  // keys g, g+1 still searched
    for (int c = 0; c < kSlots / 8 && __any_sync(kFull, open != 0); ++c) {
      ulonglong2 p[2];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint32_t b = __shfl_sync(kFull, bkt, tile * 8 + g + m);
        if ((open >> m) & 1u)
          p[m] = ld_nc_pair(key_at(t, static_cast<uint64_t>(b) * kSlots + c * 8 + sub));
      }
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const unsigned owner = tile * 8 + g + m;
        const uint64_t km = __shfl_sync(kFull, k, owner);
        const bool hit = ((open >> m) & 1u) && p[m].x == km;
        const unsigned tb = (__ballot_sync(kFull, hit) >> (tile * 8)) & 0xFFu;
        // the key's lane takes the slot and score from the lane that matched
        const unsigned from = tb ? tile * 8 + (__ffs(tb) - 1) : lane;
        const uint64_t s = __shfl_sync(kFull, hit ? p[m].y : 0ull, from);
        if (lane == owner && tb) {
          slot = c * 8 + (__ffs(tb) - 1);
          score = s;
        }
        if (tb) open &= ~(1u << m);
      }
    }
  }
  return slot;
}
#endif

template <int CH>
__host__ __device__ constexpr int row_group() {
  return CH == 1 ? HKV_FIND_ROW_GROUP : HKV_FIND_ROW_GROUP_WIDE;
}

template <bool kDual, int CH, int kOut>
__global__ void __launch_bounds__(256, HKV_FIND_MIN_BLOCKS)
    find_kernel(TableView t, uint32_t n, const uint64_t* keys, float* values_out, float** ptrs_out,
                uint8_t* found_out, uint64_t* scores_out, bool vec) {
  __shared__ __align__(16) uint16_t masks_sh[8][32][8];
  pdl_wait();
  pdl_trigger();
  const unsigned lane = lane_id();
  const unsigned tile = lane >> 3;
  const unsigned sub = lane & 7u;
  uint16_t(*msk)[8] = masks_sh[threadIdx.x >> 5];
  const uint32_t wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nw = (gridDim.x * blockDim.x) >> 5;
  const uint32_t chunks = t.dim >> 2;
  uint32_t reserved = 0;
  for (uint32_t base = wid * 32u; base < n; base += nw * 32u) {
    const uint32_t i = base + lane;
    const bool valid = i < n;
    const uint64_t k = valid ? keys[i] : 0;
    const bool act = valid && !is_reserved(k);
    if (valid && !act) ++reserved;  // skipped: reported not found
    const uint64_t h = hash64(k);
    const uint32_t pat = digest_of_hash(h) * 0x01010101u;
    uint32_t bkt = static_cast<uint32_t>(bucket_of_hash(t, h));
    int slot = -1;
    uint64_t sc = 0;
    bool open = act;
#pragma unroll 1
    for (int round = 0; round < (kDual ? 2 : 1); ++round) {
      const unsigned probe = __ballot_sync(kFull, open);
      if (!probe) break;
#if HKV_FIND_NO_DIGEST
      (void)pat;
      (void)msk;
      slot = scan_without_digest(t, probe, bkt, k, lane, sc);
#else
      uint4 cand = candidates(t, probe, bkt, pat, lane, msk);
      if (open) {
        // the first two candidates' pairs in flight together, then the rest
        // (rare) one by one
        const uint64_t row0 = static_cast<uint64_t>(bkt) * kSlots;
        const int c1 = pop_slot(cand);
        const int c2 = pop_slot(cand);
        ulonglong2 p1 = make_ulonglong2(0, 0), p2 = make_ulonglong2(0, 0);
        if (c1 >= 0) p1 = ld_nc_pair(key_at(t, row0 + c1));
        if (c2 >= 0) p2 = ld_nc_pair(key_at(t, row0 + c2));
        if (c1 >= 0 && p1.x == k) {
          slot = c1;
          sc = p1.y;
        } else if (c2 >= 0 && p2.x == k) {
          slot = c2;
          sc = p2.y;
        } else if (c2 >= 0) {
          for (int c = pop_slot(cand); c >= 0; c = pop_slot(cand)) {
            const ulonglong2 p = ld_nc_pair(key_at(t, row0 + c));
            if (p.x == k) {
              slot = c;
              sc = p.y;
              break;
            }
          }
        }
      }
#endif
      open = open && slot < 0;
      if (kDual && open && round == 0) bkt = static_cast<uint32_t>(bucket2_of(t, k, bkt));
    }
    if (valid) {
      found_out[i] = slot >= 0 ? 1 : 0;
      if (slot >= 0 && scores_out) scores_out[i] = sc;
      if (kOut == kOutPointer)
        ptrs_out[i] = slot >= 0 ? row_ptr(t, static_cast<uint64_t>(bkt) * kSlots + slot) : nullptr;
    }
    if (CH == kNoRow) continue;
    // value rows of the found keys: tile j copies those of keys 8j..8j+7
    const unsigned hits = __ballot_sync(kFull, slot >= 0);
    if (CH == kAnyRow) {
      for (int m = 0; m < 8; ++m) {
        const unsigned src = tile * 8 + m;
        const int s = __shfl_sync(kFull, slot, src);
        const uint32_t b = __shfl_sync(kFull, bkt, src);
        const uint64_t row = static_cast<uint64_t>(b) * kSlots + s;
        if ((hits >> src) & 1u)
          tile_copy_row(values_out + static_cast<uint64_t>(base + src) * t.dim, row_ptr(t, row),
                        t.dim, sub, vec, true, row >= t.hbm_rows);
      }
      continue;
    }
    constexpr int C = CH > 0 ? CH : 1;
    constexpr int RG = row_group<CH>();
#pragma unroll
    for (int g = 0; g < 8; g += RG) {
      uint4 v[RG][C];
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const unsigned src = tile * 8 + g + r;
        const int s = __shfl_sync(kFull, slot, src);
        const uint32_t b = __shfl_sync(kFull, bkt, src);
        if ((hits >> src) & 1u) {
          const uint64_t row = static_cast<uint64_t>(b) * kSlots + s;
          const float* p = row_ptr(t, row);
          const bool host = row >= t.hbm_rows;  // a row of the tiered host slab
#pragma unroll
          for (int c = 0; c < C; ++c) {
            const uint32_t q = sub + 8u * c;
            if (q < chunks) v[r][c] = host ? ld_host_row_v4(p + 4 * q) : ld_stream_v4(p + 4 * q);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const unsigned src = tile * 8 + g + r;
        if ((hits >> src) & 1u) {
          float* d = values_out + static_cast<uint64_t>(base + src) * t.dim;
#pragma unroll
          for (int c = 0; c < C; ++c) {
            const uint32_t q = sub + 8u * c;
            if (q < chunks) st_stream_v4(d + 4 * q, v[r][c]);
          }
        }
      }
    }
  }
  if (__any_sync(kFull, reserved != 0)) {
    uint32_t r = reserved;
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(kFull, r, o);
    if (lane == 0) atomicAdd(&t.stats->reserved, static_cast<unsigned long long>(r));
  }
}

template <bool kDual, int CH, int kOut>
cudaError_t launch_find_kernel(const TableView& t, uint64_t n, const uint64_t* keys,
                               float* values_out, float** ptrs_out, uint8_t* found_out,
                               uint64_t* scores_out, bool vec, cudaStream_t st) {
  const int threads = 256;
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, find_kernel<kDual, CH, kOut>, threads, 0);
  if (per_sm < 1) per_sm = 1;
  uint64_t blocks = (n + threads - 1) / threads;  // 32 keys per warp
  const uint64_t cap = static_cast<uint64_t>(sm_count()) * per_sm;
  if (blocks > cap) blocks = cap;
  return launch_chained(find_kernel<kDual, CH, kOut>, static_cast<unsigned>(blocks), threads, 0, st,
                        t, static_cast<uint32_t>(n), keys, values_out, ptrs_out, found_out,
                        scores_out, vec);
}

template <bool kDual, int kOut>
cudaError_t launch_find_rows(const TableView& t, uint64_t n, const uint64_t* keys,
                             float* values_out, float** ptrs_out, uint8_t* found_out,
                             uint64_t* scores_out, cudaStream_t st) {
  if (kOut != kOutValues)
    return launch_find_kernel<kDual, kNoRow, kOut>(t, n, keys, values_out, ptrs_out, found_out,
                                                   scores_out, false, st);
  const bool vec = (t.dim % 4 == 0) && ((reinterpret_cast<uintptr_t>(values_out) & 15) == 0);
  const uint32_t chunks = t.dim / 4;
  if (vec && chunks <= 8)
    return launch_find_kernel<kDual, 1, kOut>(t, n, keys, values_out, ptrs_out, found_out,
                                              scores_out, vec, st);
  if (vec && chunks <= 16)
    return launch_find_kernel<kDual, 2, kOut>(t, n, keys, values_out, ptrs_out, found_out,
                                              scores_out, vec, st);
  if (vec && chunks <= 32)
    return launch_find_kernel<kDual, 4, kOut>(t, n, keys, values_out, ptrs_out, found_out,
                                              scores_out, vec, st);
  return launch_find_kernel<kDual, kAnyRow, kOut>(t, n, keys, values_out, ptrs_out, found_out,
                                                  scores_out, vec, st);
}

template <int kOut>
cudaError_t launch_find_mode(const TableView& t, uint64_t n, const uint64_t* keys,
                             float* values_out, float** ptrs_out, uint8_t* found_out,
                             uint64_t* scores_out, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  if (t.dual)
    return launch_find_rows<true, kOut>(t, n, keys, values_out, ptrs_out, found_out, scores_out,
                                        st);
  return launch_find_rows<false, kOut>(t, n, keys, values_out, ptrs_out, found_out, scores_out,
                                       st);
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
