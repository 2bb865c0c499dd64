// upsert.cu -- the inserter and updater kernels: HierarchicalKV Algorithm 2
// (upsert with bucket-local admission and eviction), Algorithm 3 (score-based
// dual-bucket upsert), assign and erase (HKV §3.5).
//
// Single-bucket insert_or_assign is organised around bucket ownership rather
// than the paper's per-key CAS protocol:
//   1. dedup: the keys of the batch go into a scratch hash map that keeps the
//      largest batch index of each key (duplicates collapse to their last
//      occurrence);
//   2. group: each surviving key is counted into its bucket, groups get
//      disjoint ranges of one index array, and the keys are scattered there;
//   3. process: one warp owns one bucket.  It loads the bucket's 128 keys
//      (32 bytes per lane, one coalesced kilobyte), applies the in-place
//      updates of resident keys, then places the absent keys: a free slot if
//      there is one, else the 128 scores are loaded once and a warp-shuffle
//      arg-min over the rank (score, key) decides admission and the victim.
//      Keys, scores and digests are written back once per bucket and the
//      value rows of the final occupants are copied by 8-lane tiles.
// With one owner per bucket there is no slot locking and no retry; the result
// of a bucket depends only on its residents and its group, never on thread
// scheduling, so it equals the oracle's serial result exactly.
//
// Dual mode couples two buckets per key, so ownership cannot be partitioned:
// resident keys are updated in place by a tile kernel, then each absent key
// is placed by one warp holding locks on both candidate buckets (taken in
// increasing bucket order, bounded spin).
#include "launch.h"

namespace hkv {
namespace {

constexpr int kThreads = 256;
constexpr uint32_t kHitMark = 0x80000000u;
constexpr int kSpinLimit = 1 << 20;

__device__ __forceinline__ uint32_t map_home(uint64_t key, uint32_t mask) {
  return static_cast<uint32_t>(hash64(key) >> 32) & mask;
}

// Locate `key` in the dedup map; it must have been inserted.
__device__ __forceinline__ uint32_t map_find(const uint64_t* mkeys, uint32_t mask, uint64_t key) {
  uint32_t s = map_home(key, mask);
  for (uint32_t p = 0; p <= mask; ++p) {
    const uint64_t v = mkeys[s];
    if (v == key || v == kEmptyKey) return s;
    s = (s + 1) & mask;
  }
  return kNone;
}

__device__ __forceinline__ bool is_last_occurrence(const UpsertScratch& sc, uint64_t key,
                                                   uint64_t i) {
  const uint32_t mask = sc.map_size - 1;
  const uint32_t s = map_find(sc.map_keys, mask, key);
  return s != kNone && sc.map_keys[s] == key && sc.map_idx[s] == static_cast<uint32_t>(i) + 1;
}

// ---------------------------------------------------------------------------
// 1. dedup: map[key] = max batch index + 1.  Lanes of a warp holding the same
// key are merged first (the highest lane holds the largest index).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) dedup_insert_kernel(UpsertScratch sc, uint64_t n,
                                                                const uint64_t* keys,
                                                                DeviceStats* stats) {
  const unsigned lane = lane_id();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  const uint32_t mask = sc.map_size - 1;
  unsigned long long reserved = 0;
  for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31u);
       base < n; base += stride) {
    const uint64_t i = base + lane;
    const bool active = i < n;
    const uint64_t k = active ? keys[i] : kEmptyKey;
    const bool valid = active && !is_reserved(k);
    if (active && !valid) ++reserved;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, k);
    const bool leader = valid && static_cast<unsigned>(31 - __clz(peers)) == lane;
    if (leader) {
      uint32_t s = map_home(k, mask);
      for (uint32_t p = 0; p <= mask; ++p) {
        const unsigned long long prev = atomicCAS(
            reinterpret_cast<unsigned long long*>(sc.map_keys + s), kEmptyKey, k);
        if (prev == kEmptyKey || prev == k) {
          atomicMax(sc.map_idx + s, static_cast<uint32_t>(i) + 1);
          break;
        }
        s = (s + 1) & mask;
      }
    }
  }
  warp_add(&stats->reserved, reserved);
}

// ---------------------------------------------------------------------------
// 2. group: count last occurrences per bucket, assign group ranges, scatter.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) group_count_kernel(TableView t, UpsertScratch sc,
                                                               uint64_t n, const uint64_t* keys) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const uint64_t k = keys[i];
    uint32_t b = kNone;
    if (!is_reserved(k) && is_last_occurrence(sc, k, i)) {
      b = static_cast<uint32_t>(bucket_of_hash(t, hash64(k)));
      sc.rnk[i] = atomicAdd(sc.cnt + b, 1u);
    }
    sc.bkt[i] = b;
  }
}

__global__ void __launch_bounds__(kThreads) group_offsets_kernel(UpsertScratch sc, uint64_t nb) {
  const unsigned lane = lane_id();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31u);
       base < nb; base += stride) {
    const uint64_t b = base + lane;
    const uint32_t c = b < nb ? sc.cnt[b] : 0;
    uint32_t incl = c;
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= static_cast<unsigned>(o)) incl += v;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    uint32_t start = 0;
    if (lane == 31 && total) start = atomicAdd(sc.cursor, total);
    start = __shfl_sync(0xFFFFFFFFu, start, 31);
    if (b < nb && c) sc.off[b] = start + incl - c;
  }
}

__global__ void __launch_bounds__(kThreads) group_scatter_kernel(UpsertScratch sc, uint64_t n) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const uint32_t b = sc.bkt[i];
    if (b != kNone) sc.group[sc.off[b] + sc.rnk[i]] = static_cast<uint32_t>(i);
  }
}

// Rank order (HKV Algorithm 2 arg-min, ties by key): true when (s1,k1) < (s2,k2).
__device__ __forceinline__ bool rank_less(uint64_t s1, uint64_t k1, uint64_t s2, uint64_t k2) {
  return s1 < s2 || (s1 == s2 && k1 < k2);
}

// ---------------------------------------------------------------------------
// 3. process: one warp per bucket (single mode).
// Lane l holds slots 4l..4l+3: key sk[q], score sc_[q] (valid when the slot
// is dirty or the scores were loaded), occ[q] = batch index whose value row
// the slot must receive (kNone = unchanged), bit q of `fresh` = the slot's
// occupant was admitted by this call.
// ---------------------------------------------------------------------------
struct CopyJob {
  uint32_t src;  // batch index
  uint32_t slot; // 0..127
};

__global__ void __launch_bounds__(kThreads) upsert_single_kernel(
    TableView t, UpsertScratch scr, const uint64_t* keys_in, const float* values_in,
    const uint64_t* scores_in, uint64_t step_score, bool vec) {
  __shared__ CopyJob jobs_all[kThreads / 32][kSlots];
  const unsigned lane = lane_id();
  const unsigned warp = threadIdx.x >> 5;
  CopyJob* jobs = jobs_all[warp];
  const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
  const uint64_t nb = t.num_buckets;
  unsigned long long n_upd = 0, n_adm = 0, n_evi = 0, n_rej = 0;  // lane 0 only

  for (uint64_t b = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; b < nb;
       b += nwarps) {
    const uint32_t g = scr.cnt[b];
    if (g == 0) continue;
    const uint32_t o = scr.off[b];
    const uint64_t base = b * kSlots + lane * 4;

    uint64_t sk[4], sc[4];
    uint32_t occ[4] = {kNone, kNone, kNone, kNone};
    uint32_t fresh = 0;
    {
      const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(t.keys + base);
      const ulonglong2 c = *reinterpret_cast<const ulonglong2*>(t.keys + base + 2);
      sk[0] = a.x; sk[1] = a.y; sk[2] = c.x; sk[3] = c.y;
    }
    bool have_scores = false;
    const bool small = g <= 32;
    // Entry registers of the first chunk are kept for the small case.
    uint32_t e0 = kNone;
    uint64_t k0 = kEmptyKey, s0 = 0;
    bool hit0 = false;

    // Phase A: keys already resident are updated in place (Algorithm 2,
    // found branch).  All updates happen before any placement.
    for (uint32_t c0 = 0; c0 < g; c0 += 32) {
      const uint32_t e = (c0 + lane < g) ? scr.group[o + c0 + lane] : kNone;
      const uint64_t ke = (e != kNone) ? keys_in[e] : kEmptyKey;
      const uint64_t se = (e != kNone) ? (scores_in ? scores_in[e] : step_score) : 0;
      const uint32_t cn = min(32u, g - c0);
      bool myhit = false;
      for (uint32_t j = 0; j < cn; ++j) {
        const uint64_t kj = __shfl_sync(0xFFFFFFFFu, ke, j);
        int qh = -1;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (sk[q] == kj) qh = q;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, qh >= 0);
        if (m) {
          const uint64_t sj = __shfl_sync(0xFFFFFFFFu, se, j);
          const uint32_t ej = __shfl_sync(0xFFFFFFFFu, e, j);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q == qh) {
              occ[q] = ej;
              sc[q] = sj;
            }
          if (lane == j) myhit = true;
        }
      }
      const unsigned hm = __ballot_sync(0xFFFFFFFFu, myhit);
      if (lane == 0) n_upd += __popc(hm);
      if (small) {
        e0 = e; k0 = ke; s0 = se; hit0 = myhit;
      } else if (myhit) {
        scr.group[o + c0 + lane] = e | kHitMark;
      }
    }

    // Phase B: absent keys (Algorithm 2, empty-slot / eviction / rejection).
    bool min_valid = false;
    uint64_t ms = 0, mk = 0;
    uint32_t mslot = 0;
    for (uint32_t c0 = 0; c0 < g; c0 += 32) {
      uint32_t e;
      uint64_t ke, se;
      bool miss;
      if (small) {
        e = e0; ke = k0; se = s0; miss = (e0 != kNone) && !hit0;
      } else {
        const uint32_t raw = (c0 + lane < g) ? scr.group[o + c0 + lane] : kNone;
        miss = raw != kNone && !(raw & kHitMark);
        e = miss ? raw : kNone;
        ke = miss ? keys_in[e] : kEmptyKey;
        se = miss ? (scores_in ? scores_in[e] : step_score) : 0;
      }
      unsigned mm = __ballot_sync(0xFFFFFFFFu, miss);
      while (mm) {
        const int j = __ffs(mm) - 1;
        mm &= mm - 1;
        const uint64_t kj = __shfl_sync(0xFFFFFFFFu, ke, j);
        const uint64_t sj = __shfl_sync(0xFFFFFFFFu, se, j);
        const uint32_t ej = __shfl_sync(0xFFFFFFFFu, e, j);
        // free slot: the first one in slot order
        int qf = -1;
#pragma unroll
        for (int q = 3; q >= 0; --q)
          if (sk[q] == kEmptyKey) qf = q;
        const unsigned fm = __ballot_sync(0xFFFFFFFFu, qf >= 0);
        if (fm) {
          if (lane == static_cast<unsigned>(__ffs(fm) - 1)) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (q == qf) {
                sk[q] = kj; sc[q] = sj; occ[q] = ej; fresh |= 1u << q;
              }
          }
          if (lane == 0) ++n_adm;
          continue;
        }
        // bucket full: lowest-ranked entry (loaded once per bucket)
        if (!have_scores) {
          const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(t.scores + base);
          const ulonglong2 c = *reinterpret_cast<const ulonglong2*>(t.scores + base + 2);
          const uint64_t ld[4] = {a.x, a.y, c.x, c.y};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (occ[q] == kNone) sc[q] = ld[q];
          have_scores = true;
        }
        if (!min_valid) {
          uint64_t bs = sc[0], bk = sk[0];
          uint32_t bslot = lane * 4;
#pragma unroll
          for (int q = 1; q < 4; ++q)
            if (rank_less(sc[q], sk[q], bs, bk)) { bs = sc[q]; bk = sk[q]; bslot = lane * 4 + q; }
          for (int off = 16; off > 0; off >>= 1) {
            const uint64_t os = __shfl_xor_sync(0xFFFFFFFFu, bs, off);
            const uint64_t ok = __shfl_xor_sync(0xFFFFFFFFu, bk, off);
            const uint32_t osl = __shfl_xor_sync(0xFFFFFFFFu, bslot, off);
            if (rank_less(os, ok, bs, bk)) { bs = os; bk = ok; bslot = osl; }
          }
          ms = bs; mk = bk; mslot = bslot;
          min_valid = true;
        }
        if (rank_less(sj, kj, ms, mk)) {  // admission control
          if (lane == 0) ++n_rej;
          continue;
        }
        // evict the minimum
        bool was_fresh = false;
        if (lane == (mslot >> 2)) {
          const int qv = static_cast<int>(mslot & 3);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q == qv) {
              was_fresh = (fresh >> q) & 1u;
              sk[q] = kj; sc[q] = sj; occ[q] = ej; fresh |= 1u << q;
            }
        }
        was_fresh = __shfl_sync(0xFFFFFFFFu, was_fresh, mslot >> 2);
        if (lane == 0) {
          if (was_fresh) ++n_rej;   // displaced a key admitted by this call
          else { ++n_evi; ++n_adm; }
        }
        min_valid = false;
      }
    }

    // Write back keys, digests and scores of the lane's slots, and queue the
    // value copies of the final occupants.
    uint32_t dirty = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (occ[q] != kNone) dirty |= 1u << q;
    if (dirty) {
      *reinterpret_cast<ulonglong2*>(t.keys + base) = make_ulonglong2(sk[0], sk[1]);
      *reinterpret_cast<ulonglong2*>(t.keys + base + 2) = make_ulonglong2(sk[2], sk[3]);
      uint32_t dw = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (sk[q] != kEmptyKey) dw |= digest_of_hash(hash64(sk[q])) << (8 * q);
      *reinterpret_cast<uint32_t*>(t.digests + base) = dw;
      if (have_scores) {
        *reinterpret_cast<ulonglong2*>(t.scores + base) = make_ulonglong2(sc[0], sc[1]);
        *reinterpret_cast<ulonglong2*>(t.scores + base + 2) = make_ulonglong2(sc[2], sc[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (occ[q] != kNone) t.scores[base + q] = sc[q];
      }
    }
    const uint32_t nd = __popc(dirty);
    uint32_t pos = nd;
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, pos, off);
      if (lane >= static_cast<unsigned>(off)) pos += v;
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, pos, 31);
    pos -= nd;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (occ[q] != kNone) jobs[pos++] = CopyJob{occ[q], lane * 4 + static_cast<uint32_t>(q)};
    __syncwarp();
    const unsigned sub = lane & 7u;
    for (uint32_t p = lane >> 3; p < total; p += 4) {
      const CopyJob jb = jobs[p];
      tile_copy_row(row_ptr(t, b * kSlots + jb.slot),
                    values_in + static_cast<uint64_t>(jb.src) * t.dim, t.dim, sub, vec, true);
    }
    __syncwarp();
  }
  if (lane == 0) {
    if (n_upd) atomicAdd(&t.stats->updated, n_upd);
    if (n_adm) atomicAdd(&t.stats->admitted, n_adm);
    if (n_evi) atomicAdd(&t.stats->evicted, n_evi);
    if (n_rej) atomicAdd(&t.stats->rejected, n_rej);
    if (n_adm != n_evi) atomicAdd(&t.stats->size, n_adm - n_evi);
  }
}

// ---------------------------------------------------------------------------
// Dual mode (Algorithm 3).
// ---------------------------------------------------------------------------
// Resident keys: update value (and score) in place; absent keys go to the
// miss list.  One 8-lane tile per key.
__global__ void __launch_bounds__(kThreads) dual_resident_kernel(
    TableView t, UpsertScratch sc, uint64_t n, const uint64_t* keys, const float* values,
    const uint64_t* scores, uint64_t step_score, bool vec) {
  const unsigned lane = lane_id();
  const unsigned sub = lane & 7u;
  const unsigned tmask = 0xFFu << (lane & 24u);
  const uint64_t tiles = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 3;
  unsigned long long upd = 0;
  for (uint64_t i = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3; i < n;
       i += tiles) {
    const uint64_t k = keys[i];
    if (is_reserved(k) || !is_last_occurrence(sc, k, i)) continue;
    const uint64_t h = hash64(k);
    const uint32_t pat = digest_of_hash(h) * 0x01010101u;
    uint64_t b = bucket_of_hash(t, h);
    int slot = tile_probe<true>(t, b, k, pat, sub, tmask);
    if (slot < 0) {
      b = bucket2_of(t, k, b);
      slot = tile_probe<true>(t, b, k, pat, sub, tmask);
    }
    if (slot >= 0) {
      const uint64_t row = b * kSlots + static_cast<uint64_t>(slot);
      tile_copy_row(row_ptr(t, row), values + i * t.dim, t.dim, sub, vec, true);
      if (sub == 0) {
        t.scores[row] = scores ? scores[i] : step_score;
        ++upd;
      }
    } else if (sub == 0) {
      sc.group[atomicAdd(sc.cursor + 1, 1u)] = static_cast<uint32_t>(i);
    }
  }
  warp_add(&t.stats->updated, upd);
}

__device__ __forceinline__ bool lock_bucket(uint32_t* lk) {
  for (int it = 0; it < kSpinLimit; ++it) {
    if (atomicCAS(lk, 0u, 1u) == 0u) {
      __threadfence();
      return true;
    }
    __nanosleep(it < 64 ? 32 : 256);
  }
  return false;
}

__device__ __forceinline__ void unlock_bucket(uint32_t* lk) {
  __threadfence();
  atomicExch(lk, 0u);
}

// Warp-wide arg-min of rank over one bucket's 128 slots; lane l holds slots
// 4l..4l+3 in (s[q], k[q]).  Returns the slot index; (ms, mk) get its rank.
__device__ __forceinline__ uint32_t warp_argmin(const uint64_t* s, const uint64_t* k, uint64_t& ms,
                                                uint64_t& mk) {
  const unsigned lane = lane_id();
  uint64_t bs = s[0], bk = k[0];
  uint32_t bslot = lane * 4;
#pragma unroll
  for (int q = 1; q < 4; ++q)
    if (rank_less(s[q], k[q], bs, bk)) { bs = s[q]; bk = k[q]; bslot = lane * 4 + q; }
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t os = __shfl_xor_sync(0xFFFFFFFFu, bs, off);
    const uint64_t ok = __shfl_xor_sync(0xFFFFFFFFu, bk, off);
    const uint32_t osl = __shfl_xor_sync(0xFFFFFFFFu, bslot, off);
    if (rank_less(os, ok, bs, bk)) { bs = os; bk = ok; bslot = osl; }
  }
  ms = bs; mk = bk;
  return bslot;
}

// Absent keys: one warp per key, both candidate buckets locked.
__global__ void __launch_bounds__(kThreads) dual_place_kernel(
    TableView t, UpsertScratch sc, const uint64_t* keys, const float* values,
    const uint64_t* scores, uint64_t step_score, bool vec) {
  const unsigned lane = lane_id();
  const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
  const uint32_t nmiss = *(volatile uint32_t*)(sc.cursor + 1);
  unsigned long long fills = 0, timeouts = 0;
  for (uint64_t w = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < nmiss;
       w += nwarps) {
    const uint32_t i = sc.group[w];
    const uint64_t k = keys[i];
    const uint64_t s = scores ? scores[i] : step_score;
    const uint64_t h = hash64(k);
    const uint64_t b1 = bucket_of_hash(t, h);
    const uint64_t b2 = bucket2_of(t, k, b1);
    const uint64_t lo = b1 < b2 ? b1 : b2, hi = b1 < b2 ? b2 : b1;
    bool ok = true;
    if (lane == 0) {
      ok = lock_bucket(t.locks + lo);
      if (ok && !lock_bucket(t.locks + hi)) {
        unlock_bucket(t.locks + lo);
        ok = false;
      }
      if (!ok) ++timeouts;
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) continue;
    __threadfence();  // acquire side for every lane

    uint64_t k1[4], k2[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      k1[q] = ld_cg_u64(t.keys + b1 * kSlots + lane * 4 + q);
      k2[q] = ld_cg_u64(t.keys + b2 * kSlots + lane * 4 + q);
    }
    int f1 = -1, f2 = -1, c1 = 0, c2 = 0;
#pragma unroll
    for (int q = 3; q >= 0; --q) {
      if (k1[q] == kEmptyKey) { f1 = q; ++c1; }
      if (k2[q] == kEmptyKey) { f2 = q; ++c2; }
    }
    int free1 = c1, free2 = c2;
    for (int off = 16; off > 0; off >>= 1) {
      free1 += __shfl_xor_sync(0xFFFFFFFFu, free1, off);
      free2 += __shfl_xor_sync(0xFFFFFFFFu, free2, off);
    }
    uint64_t tb = 0;
    int tslot = -1;
    if (free1 > 0 || free2 > 0) {
      // Phase D1: the less occupied bucket (more free slots), ties to b1.
      const bool use2 = free2 > free1;
      tb = use2 ? b2 : b1;
      const unsigned fm = __ballot_sync(0xFFFFFFFFu, (use2 ? f2 : f1) >= 0);
      const int fl = __ffs(fm) - 1;
      const int fq = __shfl_sync(0xFFFFFFFFu, use2 ? f2 : f1, fl);
      tslot = fl * 4 + fq;
      ++fills;
    } else {
      // Phase D2: compare the two bucket minima; admission against the lower.
      uint64_t s1[4], s2[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        s1[q] = ld_cg_u64(t.scores + b1 * kSlots + lane * 4 + q);
        s2[q] = ld_cg_u64(t.scores + b2 * kSlots + lane * 4 + q);
      }
      uint64_t ms1, mk1, ms2, mk2;
      const uint32_t m1 = warp_argmin(s1, k1, ms1, mk1);
      const uint32_t m2 = warp_argmin(s2, k2, ms2, mk2);
      const bool use2 = rank_less(ms2, mk2, ms1, mk1);
      const uint64_t ms = use2 ? ms2 : ms1, mk = use2 ? mk2 : mk1;
      if (rank_less(ms, mk, s, k)) {
        tb = use2 ? b2 : b1;
        tslot = static_cast<int>(use2 ? m2 : m1);
      }
    }
    if (tslot >= 0) {
      const uint64_t row = tb * kSlots + static_cast<uint64_t>(tslot);
      if (lane == 0) {
        t.keys[row] = k;
        t.scores[row] = s;
        t.digests[row] = static_cast<uint8_t>(digest_of_hash(h));
      }
      float* dst = row_ptr(t, row);
      const float* src = values + static_cast<uint64_t>(i) * t.dim;
      if (vec) {
        for (uint32_t c = lane; c < (t.dim >> 2); c += 32)
          st_stream_v4(dst + 4 * c, ld_stream_v4(src + 4 * c));
      } else {
        for (uint32_t c = lane; c < t.dim; c += 32) dst[c] = src[c];
      }
    }
    __threadfence();  // release side: every lane's writes before the unlock
    __syncwarp();
    if (lane == 0) {
      unlock_bucket(t.locks + hi);
      unlock_bucket(t.locks + lo);
    }
  }
  if (lane == 0) {
    if (fills) atomicAdd(&t.stats->fills, fills);
    if (timeouts) atomicAdd(&t.stats->timeouts, timeouts);
  }
}

// After placement: count admitted (resident) vs rejected absent keys.
__global__ void __launch_bounds__(kThreads) dual_count_kernel(TableView t, UpsertScratch sc,
                                                              const uint64_t* keys) {
  const unsigned lane = lane_id();
  const unsigned sub = lane & 7u;
  const unsigned tmask = 0xFFu << (lane & 24u);
  const uint64_t tiles = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 3;
  const uint32_t nmiss = sc.cursor[1];
  unsigned long long adm = 0, rej = 0;
  for (uint64_t w = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3; w < nmiss;
       w += tiles) {
    const uint64_t k = keys[sc.group[w]];
    const uint64_t h = hash64(k);
    const uint32_t pat = digest_of_hash(h) * 0x01010101u;
    const uint64_t b1 = bucket_of_hash(t, h);
    int slot = tile_probe<true>(t, b1, k, pat, sub, tmask);
    if (slot < 0) slot = tile_probe<true>(t, bucket2_of(t, k, b1), k, pat, sub, tmask);
    if (sub == 0) {
      if (slot >= 0) ++adm;
      else ++rej;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    adm += __shfl_xor_sync(0xFFFFFFFFu, adm, o);
    rej += __shfl_xor_sync(0xFFFFFFFFu, rej, o);
  }
  if (lane == 0) {
    if (adm) atomicAdd(&t.stats->admitted, adm);
    if (rej) atomicAdd(&t.stats->rejected, rej);
    // this call's admitted count; dual_finish_kernel turns it into evictions
    if (adm) atomicAdd(reinterpret_cast<unsigned long long*>(sc.cursor + 2), adm);
  }
}

// evicted = admitted - fills for the call; size grows by fills.
__global__ void dual_finish_kernel(TableView t, UpsertScratch sc) {
  const unsigned long long adm = *reinterpret_cast<unsigned long long*>(sc.cursor + 2);
  const unsigned long long fills = t.stats->fills;
  t.stats->evicted += adm - fills;
  t.stats->size += fills;
  t.stats->fills = 0;
}

// ---------------------------------------------------------------------------
// assign (updater) and erase (inserter).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) assign_kernel(TableView t, UpsertScratch sc, uint64_t n,
                                                          const uint64_t* keys, const float* values,
                                                          const uint64_t* scores, bool vec) {
  const unsigned lane = lane_id();
  const unsigned sub = lane & 7u;
  const unsigned tmask = 0xFFu << (lane & 24u);
  const uint64_t tiles = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 3;
  unsigned long long upd = 0;
  for (uint64_t i = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3; i < n;
       i += tiles) {
    const uint64_t k = keys[i];
    if (is_reserved(k) || !is_last_occurrence(sc, k, i)) continue;
    const uint64_t h = hash64(k);
    const uint32_t pat = digest_of_hash(h) * 0x01010101u;
    uint64_t b = bucket_of_hash(t, h);
    int slot = tile_probe<true>(t, b, k, pat, sub, tmask);
    if (t.dual && slot < 0) {
      b = bucket2_of(t, k, b);
      slot = tile_probe<true>(t, b, k, pat, sub, tmask);
    }
    if (slot < 0) continue;
    const uint64_t row = b * kSlots + static_cast<uint64_t>(slot);
    tile_copy_row(row_ptr(t, row), values + i * t.dim, t.dim, sub, vec, true);
    if (sub == 0) {
      if (scores) t.scores[row] = scores[i];
      ++upd;
    }
  }
  warp_add(&t.stats->updated, upd);
}

__global__ void __launch_bounds__(kThreads) erase_kernel(TableView t, uint64_t n,
                                                         const uint64_t* keys) {
  const unsigned lane = lane_id();
  const unsigned sub = lane & 7u;
  const unsigned tmask = 0xFFu << (lane & 24u);
  const uint64_t tiles = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 3;
  unsigned long long erased = 0, reserved = 0;
  for (uint64_t i = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3; i < n;
       i += tiles) {
    const uint64_t k = keys[i];
    if (is_reserved(k)) {
      if (sub == 0) ++reserved;
      continue;
    }
    const uint64_t h = hash64(k);
    const uint32_t pat = digest_of_hash(h) * 0x01010101u;
    uint64_t b = bucket_of_hash(t, h);
    int slot = tile_probe<false>(t, b, k, pat, sub, tmask);
    if (t.dual && slot < 0) {
      b = bucket2_of(t, k, b);
      slot = tile_probe<false>(t, b, k, pat, sub, tmask);
    }
    if (slot >= 0 && sub == 0) {
      const uint64_t row = b * kSlots + static_cast<uint64_t>(slot);
      // Duplicates of k in the batch race here; exactly one CAS wins.
      if (atomicCAS(reinterpret_cast<unsigned long long*>(t.keys + row), k, kEmptyKey) == k) {
        t.digests[row] = 0;
        t.scores[row] = 0;
        ++erased;
      }
    }
  }
  warp_add(&t.stats->erased, erased);
  warp_add(&t.stats->reserved, reserved);
  // size -= erased, as a two's-complement add
  unsigned long long s = erased;
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if (lane == 0 && s) atomicAdd(&t.stats->size, ~s + 1ull);
}

unsigned grid_for(uint64_t threads_needed, int per_sm = 8) {
  uint64_t blocks = (threads_needed + kThreads - 1) / kThreads;
  const uint64_t cap = static_cast<uint64_t>(sm_count()) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  return static_cast<unsigned>(blocks);
}

uint64_t next_pow2(uint64_t v) {
  uint64_t p = 1;
  while (p < v) p <<= 1;
  return p;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t upsert_scratch_bytes(uint64_t n, uint64_t num_buckets, bool need_groups) {
  const uint64_t m = next_pow2(n * 2 < 64 ? 64 : n * 2);
  size_t bytes = align256(m * 8) + align256(m * 4) + align256(64);
  if (need_groups) bytes += 3 * align256(n * 4) + 2 * align256(num_buckets * 4);
  return bytes;
}

UpsertScratch carve_upsert_scratch(void* base, uint64_t n, uint64_t num_buckets, bool need_groups) {
  UpsertScratch s{};
  const uint64_t m = next_pow2(n * 2 < 64 ? 64 : n * 2);
  char* p = static_cast<char*>(base);
  s.map_size = static_cast<uint32_t>(m);
  s.map_keys = reinterpret_cast<uint64_t*>(p); p += align256(m * 8);
  s.map_idx = reinterpret_cast<uint32_t*>(p); p += align256(m * 4);
  s.cursor = reinterpret_cast<uint32_t*>(p); p += align256(64);
  if (need_groups) {
    s.bkt = reinterpret_cast<uint32_t*>(p); p += align256(n * 4);
    s.rnk = reinterpret_cast<uint32_t*>(p); p += align256(n * 4);
    s.group = reinterpret_cast<uint32_t*>(p); p += align256(n * 4);
    s.cnt = reinterpret_cast<uint32_t*>(p); p += align256(num_buckets * 4);
    s.off = reinterpret_cast<uint32_t*>(p); p += align256(num_buckets * 4);
  }
  return s;
}

cudaError_t clear_upsert_scratch(const UpsertScratch& s, uint64_t num_buckets, bool need_groups,
                                 cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(s.map_keys, 0xFF, static_cast<size_t>(s.map_size) * 8, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(s.map_idx, 0, static_cast<size_t>(s.map_size) * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(s.cursor, 0, 64, st);
  if (e == cudaSuccess && need_groups) e = cudaMemsetAsync(s.cnt, 0, num_buckets * 4, st);
  return e;
}

cudaError_t launch_upsert(const TableView& t, const UpsertScratch& s, uint64_t n,
                          const uint64_t* keys, const float* values, const uint64_t* scores,
                          uint64_t step_score, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const bool vec = (t.dim % 4 == 0) && ((reinterpret_cast<uintptr_t>(values) & 15) == 0);
  dedup_insert_kernel<<<grid_for(n), kThreads, 0, st>>>(s, n, keys, t.stats);
  if (!t.dual) {
    group_count_kernel<<<grid_for(n), kThreads, 0, st>>>(t, s, n, keys);
    group_offsets_kernel<<<grid_for(t.num_buckets), kThreads, 0, st>>>(s, t.num_buckets);
    group_scatter_kernel<<<grid_for(n), kThreads, 0, st>>>(s, n);
    upsert_single_kernel<<<grid_for(t.num_buckets * 32), kThreads, 0, st>>>(
        t, s, keys, values, scores, step_score, vec);
  } else {
    dual_resident_kernel<<<grid_for(n * 8), kThreads, 0, st>>>(t, s, n, keys, values, scores,
                                                                step_score, vec);
    dual_place_kernel<<<grid_for(n * 32), kThreads, 0, st>>>(t, s, keys, values, scores, step_score,
                                                             vec);
    dual_count_kernel<<<grid_for(n * 8), kThreads, 0, st>>>(t, s, keys);
    dual_finish_kernel<<<1, 1, 0, st>>>(t, s);
  }
  return cudaGetLastError();
}

cudaError_t launch_assign(const TableView& t, const UpsertScratch& s, uint64_t n,
                          const uint64_t* keys, const float* values, const uint64_t* scores,
                          cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const bool vec = (t.dim % 4 == 0) && ((reinterpret_cast<uintptr_t>(values) & 15) == 0);
  dedup_insert_kernel<<<grid_for(n), kThreads, 0, st>>>(s, n, keys, t.stats);
  assign_kernel<<<grid_for(n * 8), kThreads, 0, st>>>(t, s, n, keys, values, scores, vec);
  return cudaGetLastError();
}

cudaError_t launch_erase(const TableView& t, uint64_t n, const uint64_t* keys, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  erase_kernel<<<grid_for(n * 8), kThreads, 0, st>>>(t, n, keys);
  return cudaGetLastError();
}

}  // namespace hkv
