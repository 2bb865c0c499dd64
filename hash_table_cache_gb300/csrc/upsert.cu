// upsert.cu -- the inserter and updater kernels: HierarchicalKV Algorithm 2
// (upsert with bucket-local admission and eviction), Algorithm 3 (score-based
// dual-bucket upsert), assign and erase (HKV §3.5).
//
// Single-bucket insert_or_assign is organised around bucket ownership rather
// than the paper's per-key CAS protocol.  Two kernels:
//   1. stage: every key of the batch is entered into a scratch open-addressing
//      table laid out bucket by bucket: table bucket b owns the positions
//      [S*b/B, S*(b+1)/B) of the S-entry stage and a key probes linearly from
//      a hashed position inside its bucket's range.  An entry keeps the largest
//      batch index of its key, so duplicates collapse to their last
//      occurrence, and the entries of one table bucket end up in one short
//      contiguous run of the stage.
//   2. process: one warp owns one table bucket.  It loads the bucket (128
//      key/score pairs, two kilobytes, and the digest line) into shared
//      memory, scans its stage run 32 positions at a time, applies the
//      in-place updates of resident keys, then places the absent keys: the
//      free slots in slot order first, then, for each remaining absent key, a
//      warp arg-min over the rank (score, new, key) decides admission and the
//      victim.  Keys, scores and digests are written back once per bucket and
//      the value rows of the final occupants are copied by 8-lane tiles.
// With one owner per bucket there is no slot locking and no retry; the result
// of a bucket depends only on its residents and its keys in the batch, never
// on thread scheduling, so it equals the oracle's serial result exactly.
//
// Dual mode couples two buckets per key.  The batch is de-duplicated in a
// scratch map; a route kernel (32 keys per warp, both candidate lines probed
// by 8-lane tiles) updates resident keys in place and routes each absent key
// to one of its buckets by Algorithm 3's rules on per-bucket summaries; the
// same bucket kernel then places every bucket's routed keys; keys that pass
// displaces are routed once more and placed in a second pass.  No locks:
// every bucket still has one owner per pass.
#include <cstddef>

#include "launch.h"

namespace hkv {
namespace {

constexpr int kThreads = 256;
#ifndef HKV_BUCKET_THREADS
#define HKV_BUCKET_THREADS 256
#endif
#ifndef HKV_UPSERT_MIN_BLOCKS
#define HKV_UPSERT_MIN_BLOCKS 3
#endif
constexpr int kBucketThreads = HKV_BUCKET_THREADS;  // bucket kernel block size
#ifndef HKV_UPSERT_PIPELINE
#define HKV_UPSERT_PIPELINE 0
#endif
// L2 prefetch of the warp's next bucket and of the entries' input rows
#ifndef HKV_UPSERT_PREFETCH
#define HKV_UPSERT_PREFETCH 1
#endif
// sparse batches (at most 4 keys per bucket) of plain insert_or_assign take
// the tile-per-bucket pass (upsert_tile_kernel); 0 sends every batch to the
// warp-per-bucket kernel
#ifndef HKV_UPSERT_SPARSE
#define HKV_UPSERT_SPARSE 1
#endif
constexpr uint32_t kHitMark = 0x80000000u;

// Saturating add of v to a per-call sum of LFU increments: one native
// atomicAdd, and if the old value shows that this add wrapped past 2^64 - 1,
// an atomicMax that pins the sum at 2^64 - 1 (every later add wraps again and
// pins it again; a sum that never reaches 2^64 never wraps and is exact).
// Unlike a compare-and-swap loop it costs one operation however many
// occurrences of one hot key add at once.
__device__ __forceinline__ void sum_add_sat64(uint64_t* p, uint64_t v) {
  unsigned long long* q = reinterpret_cast<unsigned long long*>(p);
  const unsigned long long old = atomicAdd(q, static_cast<unsigned long long>(v));
  if (old + v < old) atomicMax(q, ~0ull);
}

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

// Whether `key` is a key of the running dual-mode call that was absent when
// the call began (its dedup-map entry carries pass 1's absent flag).
__device__ __forceinline__ bool absent_in_call(const UpsertScratch& sc, uint64_t key) {
  const uint32_t s = map_find(sc.map_keys, sc.map_size - 1, key);
  return s != kNone && sc.map_keys[s] == key && sc.absent[s];
}

// Map entry of `key` when batch index i is its last occurrence, else kNone,
// looked up by one thread (the warp-per-32-keys kernels keep a warp's 32
// lookups in flight together).  Each probe position's key and index are read together.
// The lookup in two steps, so that a kernel can start it (the home
// position's key and index in flight), issue other loads, and finish it.
struct MapProbe {
  uint32_t s;    // position
  uint32_t idx;  // its index
  uint64_t v;    // its key
};
__device__ __forceinline__ MapProbe map_probe_start(const UpsertScratch& sc, uint64_t key) {
  const uint32_t s = map_home(key, sc.map_size - 1);
  return MapProbe{s, sc.map_idx[s], sc.map_keys[s]};
}
__device__ __forceinline__ uint32_t map_last_occurrence_from(const UpsertScratch& sc, uint64_t key,
                                                             uint64_t i, MapProbe f) {
  const uint32_t mask = sc.map_size - 1;
  for (uint32_t p = 0; p <= mask; ++p) {
    if (f.v == key) return f.idx == static_cast<uint32_t>(i) + 1 ? f.s : kNone;
    if (f.v == kEmptyKey) return kNone;
    f.s = (f.s + 1) & mask;
    f.v = sc.map_keys[f.s];
    f.idx = sc.map_idx[f.s];
  }
  return kNone;
}
__device__ __forceinline__ uint32_t map_last_occurrence(const UpsertScratch& sc, uint64_t key,
                                                        uint64_t i) {
  return map_last_occurrence_from(sc, key, i, map_probe_start(sc, key));
}

// Summed increment of a deduplicated entry (LFU policies; 0 otherwise).
__device__ __forceinline__ uint64_t entry_inc(const UpsertScratch& sc, uint32_t slot) {
  return sc.inc ? sc.inc[slot] : 0ull;
}

// ---------------------------------------------------------------------------
// 1. dedup: map[key] = max batch index + 1.  Lanes of a warp holding the same
// key are merged first (the highest lane holds the largest index).  Under the
// LFU policies every occurrence adds its increment (inc_in[i], or 1) to the
// entry's sum.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) dedup_insert_kernel(UpsertScratch sc, uint64_t n,
                                                                const uint64_t* keys,
                                                                const uint64_t* inc_in,
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
    const unsigned lead = static_cast<unsigned>(31 - __clz(peers));
    const bool leader = valid && lead == lane;
    uint32_t slot = kNone;
    if (leader) {
      uint32_t s = map_home(k, mask);
      for (uint32_t p = 0; p <= mask; ++p) {
        const unsigned long long prev = atomicCAS(
            reinterpret_cast<unsigned long long*>(sc.map_keys + s), kEmptyKey, k);
        if (prev == kEmptyKey || prev == k) {
          atomicMax(sc.map_idx + s, static_cast<uint32_t>(i) + 1);
          slot = s;
          break;
        }
        s = (s + 1) & mask;
      }
    }
    if (sc.inc) {  // warp-uniform
      slot = __shfl_sync(0xFFFFFFFFu, slot, lead);
      if (valid && slot != kNone) sum_add_sat64(sc.inc + slot, inc_in ? inc_in[i] : 1ull);
    }
  }
  warp_add(&stats->reserved, reserved);
}

// ---------------------------------------------------------------------------
// Single mode, 1. stage.  Bucket b's range of the S-entry stage starts at
// area_start(b) = S*b/B; `a` = its length (0 when the stage has fewer entries
// than the table has buckets).
// ---------------------------------------------------------------------------
constexpr int32_t kNoShift = 0x7FFFFFFF;

__device__ __forceinline__ uint64_t area_start(uint64_t b, uint64_t S, uint64_t B, int32_t shift) {
  if (shift == kNoShift) return (b * S) / B;
  return shift >= 0 ? (b << shift) : (b >> (-shift));
}

__device__ __forceinline__ uint64_t stage_home(uint64_t h, uint64_t lo, uint64_t a) {
  if (a == 0) return lo;
  const uint64_t r = h >> 40;
  return lo + ((a & (a - 1)) == 0 ? (r & (a - 1)) : (r % a));
}

#ifndef HKV_STAGE_KEYS_PER_THREAD
#define HKV_STAGE_KEYS_PER_THREAD 1
#endif
constexpr int kStageKeysPerThread = HKV_STAGE_KEYS_PER_THREAD;

// kWarpDedup: lanes of a warp holding the same key let only the highest
// (largest batch index) enter the stage, so a key repeated many times in a
// skewed batch costs fewer atomics on its one address (not under the LFU
// policies, where every occurrence adds its own increment).  Also, the warps
// take the batch's 32-key chunks from the last to the first, and an
// occurrence reads its stage position before touching it: it skips the CAS
// when the key is there already and the max when the recorded index is not
// below its own (a stale read is only ever lower than the true value, so a
// skip is always right), which leaves a hot key's later occurrences, most
// of them seen after its last one, no atomics at all.  Used for sparse
// batches (at most 4 keys per bucket), where skewed workloads over large
// tables live; dense batches run the plain kernel, which keeps more blocks
// resident and whose keys rarely repeat.
template <bool kWarpDedup>
__global__ void __launch_bounds__(kThreads) stage_kernel(TableView t, UpsertScratch sc, uint64_t n,
                                                         const uint64_t* keys,
                                                         const uint64_t* inc_in) {
  pdl_wait();
  pdl_trigger();
  constexpr int U = kStageKeysPerThread;
  const uint64_t S = sc.map_size, mask = S - 1, B = t.num_buckets;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  unsigned long long reserved = 0;
  const uint64_t chunks = (n + 31) / 32;  // kWarpDedup: visited last to first
  // (with kWarpDedup the trip count is warp-uniform: whole warps iterate)
  for (uint64_t j0 = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       (kWarpDedup ? j0 - lane_id() : j0) < n; j0 += stride * U) {
    uint64_t k[U], pos[U], b[U];
    bool v[U];
    uint64_t idx[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t j = j0 + u * stride;
      const uint64_t i = kWarpDedup ? (chunks - 1 - (j >> 5)) * 32 + (j & 31) : j;
      idx[u] = i;
      v[u] = i < n;
      k[u] = v[u] ? keys[i] : kEmptyKey;
      if (v[u] && is_reserved(k[u])) {
        ++reserved;
        v[u] = false;
      }
      if (kWarpDedup && !sc.inc &&
          (__match_any_sync(0xFFFFFFFFu, k[u]) >> lane_id()) > 1u)
        v[u] = false;
      const uint64_t h = hash64(k[u]);
      b[u] = bucket_of_hash(t, h);
      const uint64_t lo = area_start(b[u], S, B, sc.area_shift);
      pos[u] = stage_home(h, lo, area_start(b[u] + 1, S, B, sc.area_shift) - lo) & mask;
    }
    unsigned long long prev[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!v[u]) continue;
      unsigned long long* q = reinterpret_cast<unsigned long long*>(sc.map_keys + pos[u]);
      prev[u] = (kWarpDedup && __ldcg(q) == k[u]) ? k[u] : atomicCAS(q, kEmptyKey, k[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!v[u]) continue;
      uint64_t p = pos[u];
      unsigned long long pv = prev[u];
      // S >= 2n: a free position exists, so the probe ends within S steps
      for (uint64_t tries = 1; pv != kEmptyKey && pv != k[u] && tries < S; ++tries) {
        p = (p + 1) & mask;
        pv = atomicCAS(reinterpret_cast<unsigned long long*>(sc.map_keys + p), kEmptyKey, k[u]);
      }
      const uint32_t mine = static_cast<uint32_t>(idx[u]) + 1;
      if (!kWarpDedup || __ldcg(sc.map_idx + p) < mine) atomicMax(sc.map_idx + p, mine);
      // LFU policies: every occurrence adds its increment to the entry's sum
      if (sc.inc) sum_add_sat64(sc.inc + p, inc_in ? inc_in[idx[u]] : 1ull);
      // Sparse batches mark the buckets they touch (plain store) so that the
      // processing kernel skips the others without reading them; dense
      // batches skip the marks, which would only collide.
      if (sc.mark) sc.mark[b[u]] = 1;
    }
  }
  warp_add(&t.stats->reserved, reserved);
}

// Rank order of single mode: (score, new, key), where `new` marks an entry
// placed in the bucket by the current call.  HKV Algorithm 2 admits an absent
// key when its score is >= the bucket minimum, so an incoming key outranks an
// older entry of equal score; the key orders entries of equal score and age.
// Dual mode ranks by (score, key) (Algorithm 3 admits on score > minimum, the
// key breaks ties): the same order with every `new` bit 0.
__device__ __forceinline__ bool rank3_less(uint64_t s1, uint32_t n1, uint64_t k1, uint64_t s2,
                                           uint32_t n2, uint64_t k2) {
  if (s1 != s2) return s1 < s2;
  if (n1 != n2) return n1 < n2;
  return k1 < k2;
}

// ---------------------------------------------------------------------------
// 3. process: one warp per bucket (single mode).
// The warp stages its bucket in shared memory: the 128 keys, the digest line,
// the scores (loaded once the bucket needs an eviction decision, or up front
// for large groups), and per slot the batch index whose value row the slot
// must receive (occ; kNone = unchanged) and whether its occupant was admitted
// by this call (fresh).
// ---------------------------------------------------------------------------
constexpr int kWin = 4;  // stage chunks (32 positions each) held in registers

// Arrays read or written with 16-byte vector accesses are aligned to 16.
template <bool kLfu>
struct alignas(16) BucketStage {
  alignas(16) uint64_t ekey[kWin * 32];  // the bucket's batch entries, compacted
  alignas(16) uint32_t eidx[kWin * 32];
  alignas(16) uint64_t key[kSlots];
  alignas(16) uint64_t score[kSlots];
  alignas(16) uint32_t occ[kSlots];
  alignas(16) uint32_t dig[kSlots / 4];
  alignas(16) uint32_t fresh[kSlots / 32];
  alignas(16) uint32_t dhead[256];  // digest -> first slot carrying it (0xFF: none)
  uint8_t dnext[kSlots];            // next slot with the same digest (0xFF: end)
  uint8_t list[kSlots];             // free-slot list, later the dirty-slot list
  // insert_and_evict: the value rows of one extraction round to report
  // (output index, source batch index or kNone, slot), at most 32
  uint32_t ev_o[32];
  uint32_t ev_src[32];
  uint8_t ev_slot[32];
  alignas(16) uint64_t einc[kLfu ? kWin * 32 : 2];  // summed increments (LFU policies)
#if HKV_UPSERT_PIPELINE
  // The warp's next bucket, brought in by the copy engine while this one is
  // processed: its key/score pairs, its digest line and the copy's barrier.
  alignas(128) ulonglong2 next_pairs[kSlots];
  alignas(16) uint32_t next_dig[kSlots / 4];
  alignas(8) uint64_t bar;
#endif
};
#define HKV_STAGE_ALIGNED(L)                                                                     \
  static_assert(offsetof(BucketStage<L>, key) % 16 == 0 &&                                     \
                    offsetof(BucketStage<L>, score) % 16 == 0 &&                               \
                    offsetof(BucketStage<L>, occ) % 16 == 0 &&                                 \
                    offsetof(BucketStage<L>, dhead) % 16 == 0 && sizeof(BucketStage<L>) % 16 == 0, \
                "vector-accessed stage arrays must be 16-byte aligned")
HKV_STAGE_ALIGNED(false);
HKV_STAGE_ALIGNED(true);
#undef HKV_STAGE_ALIGNED
#if HKV_UPSERT_PIPELINE
static_assert(offsetof(BucketStage<false>, next_pairs) % 128 == 0 &&
                  offsetof(BucketStage<true>, next_pairs) % 128 == 0 &&
                  offsetof(BucketStage<false>, next_dig) % 16 == 0 &&
                  offsetof(BucketStage<true>, next_dig) % 16 == 0,
              "bulk-copy targets must be 16-byte aligned");
#endif

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive prefix over lanes of a per-lane count in 0..4 (three bit planes).
__device__ __forceinline__ uint32_t prefix_small(uint32_t c, uint32_t& total) {
  const unsigned lt = lanemask_lt();
  const unsigned p0 = __ballot_sync(0xFFFFFFFFu, c & 1u);
  const unsigned p1 = __ballot_sync(0xFFFFFFFFu, c & 2u);
  const unsigned p2 = __ballot_sync(0xFFFFFFFFu, c & 4u);
  total = __popc(p0) + 2 * __popc(p1) + 4 * __popc(p2);
  return __popc(p0 & lt) + 2 * __popc(p1 & lt) + 4 * __popc(p2 & lt);
}

// Warp minimum of a 64-bit value over the lanes with `valid`, by two 32-bit
// reductions; `sel` receives the lanes that hold it.
__device__ __forceinline__ uint64_t warp_min_u64(uint64_t v, bool valid, unsigned& sel) {
  const uint32_t hi = valid ? static_cast<uint32_t>(v >> 32) : 0xFFFFFFFFu;
  const uint32_t mh = __reduce_min_sync(0xFFFFFFFFu, hi);
  bool c = valid && hi == mh;
  const uint32_t lo = c ? static_cast<uint32_t>(v) : 0xFFFFFFFFu;
  const uint32_t ml = __reduce_min_sync(0xFFFFFFFFu, lo);
  c = c && static_cast<uint32_t>(v) == ml;
  sel = __ballot_sync(0xFFFFFFFFu, c);
  return (static_cast<uint64_t>(mh) << 32) | ml;
}

// Exact form of the E extractions of phase B (below), for a bucket whose
// 31-bit rank keys tie at the front: each extraction takes the warp's
// minimum 31-bit key, and among the elements that share it the lowest exact
// rank (score, new, key), first within the lane, then across the warp.
// f0..f3 are the lane's entries' keys, mf its pending key's (0xFFFFFFFF: no
// pending key).  Returns the lane's extracted entries (bits 0..3) and whether
// its pending key survived.  Kept out of line: it runs rarely.
struct ExactOut {
  uint32_t rem;
  bool pending;
};

template <class Stage>
__device__ __noinline__ ExactOut extract_exact(const Stage* st, unsigned lane, uint32_t E,
                                               uint32_t f0, uint32_t f1, uint32_t f2, uint32_t f3,
                                               uint32_t mf, bool pending, uint64_t se,
                                               uint64_t ke, bool with_new) {
  constexpr uint32_t kGone = 0xFFFFFFFFu;
  uint32_t rf[4] = {f0, f1, f2, f3};
  const uint32_t fw = with_new ? st->fresh[lane >> 3] >> ((lane * 4) & 31) : 0u;
  uint32_t rem = 0;
  for (uint32_t x = 0; x < E; ++x) {
    const uint32_t lf = min(min(min(rf[0], rf[1]), min(rf[2], rf[3])), mf);
    const uint32_t m = __reduce_min_sync(0xFFFFFFFFu, lf);
    const uint32_t eq = (rf[0] == m ? 1u : 0u) | (rf[1] == m ? 2u : 0u) |
                        (rf[2] == m ? 4u : 0u) | (rf[3] == m ? 8u : 0u) | (mf == m ? 16u : 0u);
    uint64_t bs = ~0ull, bk = ~0ull;
    uint32_t bn = 1u, bbit = 0;
#pragma unroll
    for (int q = 0; q < 5; ++q) {
      if (!((eq >> q) & 1u)) continue;
      const uint64_t cs = q < 4 ? st->score[lane * 4 + q] : se;
      const uint64_t ck = q < 4 ? st->key[lane * 4 + q] : ke;
      const uint32_t cn = q < 4 ? (fw >> q) & 1u : (with_new ? 1u : 0u);
      if (!bbit || rank3_less(cs, cn, ck, bs, bn, bk)) {
        bs = cs;
        bk = ck;
        bn = cn;
        bbit = 1u << q;
      }
    }
    unsigned sel_s, sel_k;
    warp_min_u64(bs, bbit != 0, sel_s);
    const unsigned old_s = __ballot_sync(0xFFFFFFFFu, ((sel_s >> lane) & 1u) && bn == 0u);
    const unsigned sel_n = old_s ? old_s : sel_s;
    warp_min_u64(bk, (sel_n >> lane) & 1u, sel_k);
    const uint32_t take = lane == static_cast<unsigned>(__ffs(sel_k) - 1) ? bbit : 0u;
    if (take & 16u) {
      pending = false;  // rejected
      mf = kGone;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (take & (1u << q)) rf[q] = kGone;
    rem |= take & 15u;
  }
  return {rem, pending};
}

// kLfu: the table sums increments (kLfu, kEpochLfu).  Otherwise every key of
// the call gets rule.in[e] or the constant rule.clock (the host folds the
// clock policies into that constant).
// kDual: the buckets of a dual-mode table, whose stage holds the absent keys
// routed to each bucket (their chosen bucket in stage_bkt).  Ranks are then
// (score, key) (Algorithm 3), no key is resident (phase A is skipped), the
// batch counts come from a later kernel (this one only adds the free slots it
// fills), and the kernel leaves each bucket's summary.
//
// Pipelined build (-DHKV_UPSERT_PIPELINE=1, the latency-hiding variant in
// the spirit of HKV §4.3's Pipeline kernel): each warp keeps its next bucket
// in flight.  While it works on bucket b, the copy engine moves the key/score
// pairs (2 KiB) and the digest line of the next bucket it owns into shared
// memory (cp.async.bulk, completion on an mbarrier).  The wait on the barrier
// is bounded: if it runs out the warp counts a timeout, loads its buckets
// directly from then on, and before exiting waits (bounded again) for the
// copy still in flight.  Measured slower than the default build on GB300
// (the kernel is bound by its instruction stream, not by the bucket loads),
// so it is kept as a build option for that measurement only.
#if HKV_UPSERT_PIPELINE
constexpr int kCopyWaitLimit = 1 << 14;
#endif

template <bool kLfu, bool kDual, bool kEvict>
__global__ void __launch_bounds__(kBucketThreads, HKV_UPSERT_MIN_BLOCKS) upsert_single_kernel(
    TableView t, UpsertScratch scr, const uint64_t* keys_in, const float* values_in,
    ScoreRule rule, bool vec, UpsertExtra ex) {
  (void)keys_in;  // entry keys come from the stage
#if HKV_UPSERT_PIPELINE
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BucketStage<kLfu>* stage_all = reinterpret_cast<BucketStage<kLfu>*>(smem_raw);
#else
  __shared__ BucketStage<kLfu> stage_all[kBucketThreads / 32];
#endif
  pdl_wait();
  pdl_trigger();
  const unsigned lane = lane_id();
  BucketStage<kLfu>& st = stage_all[threadIdx.x >> 5];
  auto score_of = [&](uint32_t e, uint64_t inc, bool resident, uint64_t old) -> uint64_t {
    if (kLfu) return policy_score(rule, e, inc, resident, old);
    return rule.in ? rule.in[e] : rule.clock;
  };
  const uint64_t nwarps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
  const uint64_t nb = t.num_buckets;
  const unsigned sub = lane & 7u;
  const uint64_t S = scr.map_size, smask = S - 1;
  unsigned long long n_upd = 0, n_adm = 0, n_evi = 0, n_rej = 0, n_fill = 0;  // lane 0 only
  constexpr uint32_t kNewBit = kDual ? 0u : 1u;  // rank (score, new, key) or (score, key)

#if HKV_UPSERT_PIPELINE
  // the warp's buckets with keys of the batch (sparse batches mark them)
  auto owned_from = [&](uint64_t x) -> uint64_t {
    while (x < nb && scr.mark && !(ex.mark_want ? scr.mark[x] == ex.mark_want : scr.mark[x] != 0))
      x += nwarps;
    return x;
  };
  auto copy_bucket = [&](uint64_t x) {  // lane 0 only
    mbar_arrive_expect_tx(&st.bar, kSlots * 16 + kSlots);
    bulk_load_smem(st.next_pairs, key_at(t, x * kSlots), kSlots * 16, &st.bar);
    bulk_load_smem(st.next_dig, t.digests + x * kSlots, kSlots, &st.bar);
  };
  auto wait_copy = [&](uint32_t par) {
    bool done = false;
    for (int it = 0; it < kCopyWaitLimit && !done; ++it) done = mbar_try_wait(&st.bar, par);
    return __all_sync(0xFFFFFFFFu, done);
  };
  bool engine = true;      // the copy engine serves this warp
  bool in_flight = false;  // a copy into next_* has not been waited for
  uint32_t parity = 0;
  uint64_t b = owned_from((static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (lane == 0) mbar_init(&st.bar, 1);
  __syncwarp();
  if (b < nb) {
    if (lane == 0) copy_bucket(b);
    in_flight = true;
  }
  uint64_t b_next = 0;
  for (; b < nb; b = b_next) {
    b_next = owned_from(b + nwarps);
#else
  // The warp's buckets b0, b0 + W, b0 + 2W, ... (W warps in the grid) that
  // hold a key of the batch (all of them without a mark array), 32 at a
  // time: one mark load per lane, then the set bits of the ballot in order.
  uint64_t g = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  auto marked = [&](uint64_t g0) -> unsigned {
    const uint64_t x = g0 + lane * nwarps;
    return __ballot_sync(0xFFFFFFFFu,
                         x < nb && (!scr.mark || (ex.mark_want ? scr.mark[x] == ex.mark_want
                                                               : scr.mark[x] != 0)));
  };
  unsigned todo = marked(g);
  auto next_bucket = [&]() -> uint64_t {
    while (!todo) {
      g += 32 * nwarps;
      if (g >= nb) return nb;
      todo = marked(g);
    }
    const uint64_t x = g + (__ffs(todo) - 1) * nwarps;
    todo &= todo - 1;
    return x;
  };
  for (uint64_t b = next_bucket(); b < nb; b = next_bucket()) {
#if HKV_UPSERT_PREFETCH
    if (todo) {  // the warp's next bucket: its pairs and digest line into L2
      const uint64_t bn = g + (__ffs(todo) - 1) * nwarps;
      if (lane < 16) prefetch_l2(key_at(t, bn * kSlots + lane * 8));
      else if (lane == 16) prefetch_l2(t.digests + bn * kSlots);
    }
#endif
#endif
    const uint64_t base = b * kSlots + lane * 4;
    // This bucket's stage run: from lo, past a_end, up to the first free
    // position at or after a_end (linear probing leaves no gap in a run).
    const uint64_t lo = area_start(b, S, nb, scr.area_shift);
    const uint64_t a_end = area_start(b + 1, S, nb, scr.area_shift);

    // Loads: the bucket (the lane's four key/score pairs and digest bytes)
    // and the first kWin chunks of the run, all issued before any use.  The
    // pipelined build takes the bucket from the copy engine's buffer.
    ulonglong2 kv[4];
    uint32_t dw;
#if HKV_UPSERT_PIPELINE
    bool have = false;
    if (engine) {
      if (wait_copy(parity)) {
        parity ^= 1u;
        in_flight = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) kv[q] = st.next_pairs[lane * 4 + q];
        dw = st.next_dig[lane];
        have = true;
      } else {
        engine = false;
        if (lane == 0) atomicAdd(&t.stats->timeouts, 1ull);
      }
    }
    if (!have)
#endif
    {
#pragma unroll
      for (int q = 0; q < 4; ++q) kv[q] = *reinterpret_cast<const ulonglong2*>(key_at(t, base + q));
      dw = *reinterpret_cast<const uint32_t*>(t.digests + base);
    }
    const uint64_t nw_need = (a_end - lo) / 32 + 1;
    const uint32_t nw = nw_need < kWin ? static_cast<uint32_t>(nw_need) : kWin;
    uint64_t wk[kWin];
    uint32_t wr[kWin], wb[kWin];
#pragma unroll
    for (int w = 0; w < kWin; ++w) {
      wk[w] = kEmptyKey;
      wr[w] = 0;
      wb[w] = 0;
      if (w < static_cast<int>(nw)) {
        const uint64_t j = (lo + 32ull * w + lane) & smask;
        wk[w] = scr.stage_keys[j];
        wr[w] = scr.stage_idx[j];
        if (kDual) wb[w] = scr.stage_bkt[j];
      }
    }
#if HKV_UPSERT_PIPELINE
    __syncwarp();  // every lane has read the buffer: refill it
    if (engine && b_next < nb) {
      if (lane == 0) {
        fence_proxy_async_smem();
        copy_bucket(b_next);
      }
      in_flight = true;
    }
#endif
    *reinterpret_cast<ulonglong2*>(&st.key[lane * 4]) = make_ulonglong2(kv[0].x, kv[1].x);
    *reinterpret_cast<ulonglong2*>(&st.key[lane * 4 + 2]) = make_ulonglong2(kv[2].x, kv[3].x);
    *reinterpret_cast<ulonglong2*>(&st.score[lane * 4]) = make_ulonglong2(kv[0].y, kv[1].y);
    *reinterpret_cast<ulonglong2*>(&st.score[lane * 4 + 2]) = make_ulonglong2(kv[2].y, kv[3].y);
    *reinterpret_cast<uint4*>(&st.occ[lane * 4]) = make_uint4(kNone, kNone, kNone, kNone);
    st.dig[lane] = dw;
    // Reverse digest index of the bucket: a chain of slots per digest value
    // (phase A's lookup; dual mode routes only absent keys and skips it).
    if (!kDual) {
      reinterpret_cast<uint4*>(st.dhead)[2 * lane] = make_uint4(0xFF, 0xFF, 0xFF, 0xFF);
      reinterpret_cast<uint4*>(st.dhead)[2 * lane + 1] = make_uint4(0xFF, 0xFF, 0xFF, 0xFF);
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t d = (dw >> (8 * q)) & 0xFFu;
        if (d)
          st.dnext[lane * 4 + q] = static_cast<uint8_t>(atomicExch(&st.dhead[d], lane * 4 + q));
      }
    }
    if (lane < 4) st.fresh[lane] = 0;

    // Entry of chunk c for this lane: batch index if the stage position holds
    // a key of bucket b before the end of the run (else kNone).  `stop`
    // carries the run end across chunks.
    bool run_ended = false;
    auto entry_of = [&](uint64_t c, uint64_t key, uint32_t raw, uint32_t bkt) -> uint32_t {
      const uint64_t j = lo + 32ull * c + lane;
      const bool empty = key == kEmptyKey;
      const unsigned stopm = __ballot_sync(0xFFFFFFFFu, empty && j >= a_end);
      const bool before = !run_ended && (stopm == 0 || lane < static_cast<unsigned>(__ffs(stopm) - 1));
      if (stopm) run_ended = true;
      if (32ull * (c + 1) >= S) run_ended = true;
      const bool mine = !empty && before &&
                        (kDual ? bkt == static_cast<uint32_t>(b) : bucket_of_hash(t, hash64(key)) == b);
      return mine ? (raw & ~kHitMark) - 1 : kNone;
    };
    uint32_t we[kWin];
#pragma unroll
    for (int w = 0; w < kWin; ++w)
      we[w] = w < static_cast<int>(nw) ? entry_of(w, wk[w], wr[w], wb[w]) : kNone;
    const bool in_window = run_ended;  // the run ends inside the loaded chunks
#if HKV_UPSERT_PREFETCH
    // the entries' input value rows (phase C copies them) into L2
#pragma unroll
    for (int w = 0; w < kWin; ++w) {
      if (we[w] == kNone) continue;
      const char* row = reinterpret_cast<const char*>(values_in + static_cast<uint64_t>(we[w]) * t.dim);
      for (uint32_t off = 0; off < 4 * t.dim; off += 128) prefetch_l2(row + off);
    }
#endif
    __syncwarp();

    // Phase A (Algorithm 2, found branch): a resident key gets its new value
    // and score.  The entry lane scans the staged digest line and confirms
    // matches against the staged keys.  Returns whether the entry hit.
    auto phase_a = [&](uint32_t e, uint64_t ke, uint64_t inc) -> bool {
      int hs = -1;
      if (e != kNone) {
        // walk the slots whose digest equals the key's (HKV Algorithm 1's
        // digest filter, through the bucket's reverse index)
        uint32_t sl = st.dhead[digest_of_hash(hash64(ke))];
        for (int guard = 0; sl != 0xFFu && guard < kSlots; ++guard) {
          if (st.key[sl] == ke) {
            hs = static_cast<int>(sl);
            break;
          }
          sl = st.dnext[sl];
        }
        if (hs >= 0 && ex.update_resident) {
          st.occ[hs] = e;
          st.score[hs] = score_of(e, inc, true, st.score[hs]);
        }
      }
      const unsigned hm = __ballot_sync(0xFFFFFFFFu, hs >= 0);
      if (lane == 0 && ex.update_resident) n_upd += __popc(hm);
      return hs >= 0;
    };

    // Phase B (Algorithm 2, empty slot / eviction / rejection) for the absent
    // keys of one chunk.  Free slots (in slot order) go to the first absent
    // keys.  For the E absent keys left, applying Algorithm 2 to each in turn
    // leaves the 128 highest ranks of (bucket entries + those keys), so the
    // warp drops the E lowest-ranked of that union directly: E extractions of
    // the union's minimum, each one 32-bit warp reduction over the lanes'
    // candidates (its four bucket entries and its own absent key).  Extracted
    // absent keys are rejected; the absent keys left take the slots of the
    // extracted entries.
    uint32_t nfree = 0, used = 0;
    auto phase_b = [&](uint32_t e, uint64_t ke, bool miss, uint64_t inc) {
      const uint64_t se = miss ? score_of(e, inc, false, 0) : 0;
      const unsigned mm = __ballot_sync(0xFFFFFFFFu, miss);
      if (!mm) return;
      const uint32_t rank = used + __popc(mm & lanemask_lt());
      if (miss && rank < nfree) {
        const uint32_t slot = st.list[rank];
        st.key[slot] = ke;
        st.score[slot] = se;
        st.occ[slot] = e;
        reinterpret_cast<uint8_t*>(st.dig)[slot] = static_cast<uint8_t>(digest_of_hash(hash64(ke)));
        atomicOr(&st.fresh[slot >> 5], 1u << (slot & 31));
      }
      const uint32_t placed = min(static_cast<uint32_t>(__popc(mm)), nfree - used);
      used += placed;
      if (lane == 0) {
        n_adm += placed;
        n_fill += placed;
      }
      bool pending = miss && rank >= nfree;  // this lane's absent key still competes
      const unsigned em = __ballot_sync(0xFFFFFFFFu, pending);
      if (!em) return;
      const uint32_t E = __popc(em);
      __syncwarp();
      // 31-bit keys that preserve the rank order (ties allowed): the score
      // relative to the union's minimum, with the new bit and the top 16 key
      // bits appended when the scores span less than 2^14, shifted right to
      // 31 bits when they span more than 2^31.  0xFFFFFFFF marks an element
      // that is no longer a candidate.  An entry's `new` bit is its fresh
      // mark; every pending key is new.
      constexpr uint32_t kGone = 0xFFFFFFFFu;
      uint64_t s4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) s4[q] = st.score[lane * 4 + q];
      const uint32_t fw = st.fresh[lane >> 3] >> ((lane * 4) & 31);  // the lane's 4 fresh bits
      uint64_t lo_s = min(min(s4[0], s4[1]), min(s4[2], s4[3]));
      uint64_t hi_s = max(max(s4[0], s4[1]), max(s4[2], s4[3]));
      if (pending) {
        lo_s = min(lo_s, se);
        hi_s = max(hi_s, se);
      }
      unsigned sel;
      const uint64_t smin = warp_min_u64(lo_s, true, sel);
      const uint64_t smax = ~warp_min_u64(~hi_s, true, sel);
      const uint64_t span = smax - smin;
      const int nbits = span ? 64 - __clzll(static_cast<long long>(span)) : 0;
      const int sh = nbits > 31 ? nbits - 31 : 0;
      auto fkey = [&](uint64_t sc, uint32_t nw, uint64_t k) -> uint32_t {
        if (span < 16384)
          return static_cast<uint32_t>(((sc - smin) << 17) | (static_cast<uint64_t>(nw) << 16) |
                                       (k >> 48));
        return static_cast<uint32_t>((sc - smin) >> sh);
      };
      uint32_t rf[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        rf[q] = fkey(s4[q], (fw >> q) & kNewBit, st.key[lane * 4 + q]);
      const uint32_t mf0 = pending ? fkey(se, kNewBit, ke) : kGone;
      const bool pending0 = pending;
      uint32_t mf = mf0;
      // E extractions of the union's minimum.  Fast pass: every element equal
      // to the warp minimum leaves; when the 31-bit keys of the extracted
      // elements are distinct that is exactly one element per extraction,
      // which the count at the end confirms.
      uint32_t rem = 0;  // the lane's bucket entries taken out
#pragma unroll 1
      for (uint32_t x = 0; x < E; ++x) {
        const uint32_t m =
            __reduce_min_sync(0xFFFFFFFFu, min(min(min(rf[0], rf[1]), min(rf[2], rf[3])), mf));
        // branch-free: every element equal to the minimum leaves
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const bool out_q = rf[q] == m;
          rf[q] = out_q ? kGone : rf[q];
          rem |= out_q ? (1u << q) : 0u;
        }
        const bool out_m = mf == m;
        mf = out_m ? kGone : mf;
        pending = pending && !out_m;
      }
      const uint32_t out = __popc(rem) + ((pending0 && !pending) ? 1u : 0u);
      if (__reduce_add_sync(0xFFFFFFFFu, out) != E) {
        // Equal 31-bit keys met at the front: redo with exact ranks.
        const ExactOut r = extract_exact(
            &st, lane, E, fkey(s4[0], fw & kNewBit, st.key[lane * 4]),
            fkey(s4[1], (fw >> 1) & kNewBit, st.key[lane * 4 + 1]),
            fkey(s4[2], (fw >> 2) & kNewBit, st.key[lane * 4 + 2]),
            fkey(s4[3], (fw >> 3) & kNewBit, st.key[lane * 4 + 3]), mf0, pending0, se, ke,
            kNewBit != 0);
        rem = r.rem;
        pending = r.pending;
      }
      // Extracted bucket entries: list them in slot order for the pending keys.
      uint32_t n_ext;
      uint32_t pos = prefix_small(static_cast<uint32_t>(__popc(rem)), n_ext);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (rem & (1u << q)) st.list[pos++] = static_cast<uint8_t>(lane * 4 + q);
      // extracted entries placed earlier this call (fresh) vs pre-call residents
      const uint32_t evm = rem & ~fw & 15u;
      const uint32_t ev = __popc(evm), fr = __popc(rem & fw & 15u);
      if (kEvict && ex.ev_keys) {
        // insert_and_evict: report the displaced pre-call residents as they
        // are now, at output positions taken with one atomic per warp
        uint32_t n_out;
        uint32_t at = prefix_small(ev, n_out);
        unsigned long long o0 = 0;
        if (lane == 0 && n_out) o0 = atomicAdd(ex.ev_count, static_cast<unsigned long long>(n_out));
        o0 = __shfl_sync(0xFFFFFFFFu, o0, 0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (!((evm >> q) & 1u)) continue;
          const uint32_t slot = lane * 4 + q;
          const unsigned long long o = o0 + at;
          ex.ev_keys[o] = st.key[slot];
          if (ex.ev_scores) ex.ev_scores[o] = st.score[slot];
          st.ev_o[at] = static_cast<uint32_t>(o);
          st.ev_src[at] = st.occ[slot];  // updated by this call: its input row
          st.ev_slot[at] = static_cast<uint8_t>(slot);
          ++at;
        }
        __syncwarp();
        if (ex.ev_values) {  // the rows, 8-lane tiles, 16-byte vectors when aligned
          const bool evec = vec && (reinterpret_cast<uintptr_t>(ex.ev_values) & 15) == 0;
          for (uint32_t j = lane >> 3; j < n_out; j += 4) {
            const uint32_t src_i = st.ev_src[j];
            const float* src = src_i != kNone
                                   ? values_in + static_cast<uint64_t>(src_i) * t.dim
                                   : row_ptr(t, b * kSlots + st.ev_slot[j]);
            tile_copy_row(ex.ev_values + static_cast<uint64_t>(st.ev_o[j]) * t.dim, src, t.dim,
                          sub, evec, true,
                          src_i == kNone && b * kSlots + st.ev_slot[j] >= t.hbm_rows);
          }
        }
        __syncwarp();
      }
      if (kDual && ex.collect_retry) {
        // keys of the batch this pass displaced (rejected absent keys and
        // entries it placed and then lost) are routed once more
        uint32_t mine = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) mine += (rem >> q) & (fw >> q) & 1u;
        const bool rej = pending0 && !pending;
        mine += rej ? 1u : 0u;
        uint32_t tot;
        uint32_t at = prefix_small(mine, tot);
        uint32_t base_r = 0;
        if (lane == 0 && tot) base_r = atomicAdd(scr.cursor + 4, tot);
        base_r = __shfl_sync(0xFFFFFFFFu, base_r, 0) + at;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if ((rem >> q) & (fw >> q) & 1u) scr.retry[base_r++] = st.occ[lane * 4 + q];
        if (rej) scr.retry[base_r] = e;
      }
      uint32_t fr_all = fr;
      if (kDual && !ex.collect_retry) {
        // second pass: an extracted entry that the first pass placed is a key
        // of this call that ends up absent, not an eviction
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (((evm >> q) & 1u) && absent_in_call(scr, st.key[lane * 4 + q])) ++fr_all;
      }
      const uint32_t n_ev = __reduce_add_sync(0xFFFFFFFFu, ev);
      const uint32_t n_fr = __reduce_add_sync(0xFFFFFFFFu, fr_all);
      if (lane == 0) {
        n_evi += n_ev;
        n_adm -= n_fr;
        n_rej += n_fr + (E - n_ext);  // displaced fresh keys + rejected absent keys
      }
      __syncwarp();
      // absent keys still pending take the extracted slots
      const unsigned am = __ballot_sync(0xFFFFFFFFu, pending);
      if (pending) {
        const uint32_t slot = st.list[__popc(am & lanemask_lt())];
        st.key[slot] = ke;
        st.score[slot] = se;
        st.occ[slot] = e;
        reinterpret_cast<uint8_t*>(st.dig)[slot] = static_cast<uint8_t>(digest_of_hash(hash64(ke)));
        atomicOr(&st.fresh[slot >> 5], 1u << (slot & 31));
      }
      if (lane == 0) n_adm += __popc(am);
      __syncwarp();
    };

    auto build_free_list = [&]() {
      // a free slot is a zero digest byte (phase A changes no digest)
      const uint32_t fm = byte_eq_mask4(dw, 0u);
      if (!__any_sync(0xFFFFFFFFu, fm != 0)) {  // full bucket: nothing to list
        nfree = 0;
        return;
      }
      uint32_t pos = prefix_small(__popc(fm), nfree);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (fm & (1u << q)) st.list[pos++] = static_cast<uint8_t>(lane * 4 + q);
      __syncwarp();
    };

    if (in_window) {
      // Compact the window's entries, then work on dense chunks of 32.
      uint32_t ne = 0;
#pragma unroll
      for (int w = 0; w < kWin; ++w) {
        const unsigned m = __ballot_sync(0xFFFFFFFFu, we[w] != kNone);
        if (we[w] != kNone) {
          const uint32_t p = ne + __popc(m & lanemask_lt());
          st.ekey[p] = wk[w];
          st.eidx[p] = we[w];
          if (kLfu) st.einc[p] = scr.stage_inc[(lo + 32ull * w + lane) & smask];
        }
        ne += __popc(m);
      }
      __syncwarp();
      // (loops kept rolled: one copy of each phase keeps the code in cache)
      uint32_t hits = 0;  // bit c: this lane's entry of dense chunk c hit
#pragma unroll 1
      for (uint32_t c = 0; !kDual && 32u * c < ne; ++c) {
        const bool v = 32u * c + lane < ne;
        const uint64_t inc = kLfu && v ? st.einc[32 * c + lane] : 0ull;
        if (phase_a(v ? st.eidx[32 * c + lane] : kNone, v ? st.ekey[32 * c + lane] : kEmptyKey,
                    inc))
          hits |= 1u << c;
      }
      __syncwarp();
      build_free_list();
#pragma unroll 1
      for (uint32_t c = 0; 32u * c < ne; ++c) {
        const bool v = 32u * c + lane < ne;
        const uint32_t e = v ? st.eidx[32 * c + lane] : kNone;
        const uint64_t inc = kLfu && v ? st.einc[32 * c + lane] : 0ull;
        phase_b(e, v ? st.ekey[32 * c + lane] : kEmptyKey, v && !((hits >> c) & 1u), inc);
      }
    } else {
      // Long run: walk it chunk by chunk from the stage, marking hits there.
      uint64_t nch = 0;
      run_ended = false;
      for (uint64_t c = 0; !run_ended; ++c) {
        const uint64_t j = (lo + 32ull * c + lane) & smask;
        const uint64_t key = scr.stage_keys[j];
        const uint32_t raw = scr.stage_idx[j];
        const uint32_t e = entry_of(c, key, raw, kDual ? scr.stage_bkt[j] : 0u);
        if (!kDual && phase_a(e, key, kLfu && e != kNone ? scr.stage_inc[j] : 0ull))
          scr.stage_idx[j] = raw | kHitMark;
        nch = c + 1;
      }
      __syncwarp();
      build_free_list();
      run_ended = false;
      for (uint64_t c = 0; c < nch; ++c) {
        const uint64_t j = (lo + 32ull * c + lane) & smask;
        const uint64_t key = scr.stage_keys[j];
        const uint32_t raw = scr.stage_idx[j];
        const uint32_t e = entry_of(c, key, raw, kDual ? scr.stage_bkt[j] : 0u);
        phase_b(e, key, e != kNone && !(raw & kHitMark),
                kLfu && e != kNone ? scr.stage_inc[j] : 0ull);
      }
    }
    __syncwarp();

    if (kDual) {  // the bucket's summary for the next routing
      uint32_t cnt = 0;
      uint64_t mn = ~0ull;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (st.key[lane * 4 + q] == kEmptyKey) continue;
        ++cnt;
        mn = min(mn, st.score[lane * 4 + q]);
      }
      unsigned sel;
      mn = warp_min_u64(mn, true, sel);
      cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
      if (lane == 0) {
        t.summary[b].min_score = cnt ? mn : 0ull;
        t.summary[b].count = cnt;
      }
    }

    // Phase C: write back the lane's changed slots and digest bytes, then
    // copy the value rows of the final occupants.
    const uint4 oc = *reinterpret_cast<const uint4*>(&st.occ[lane * 4]);
    const uint32_t dm = (oc.x != kNone ? 1u : 0u) | (oc.y != kNone ? 2u : 0u) |
                        (oc.z != kNone ? 4u : 0u) | (oc.w != kNone ? 8u : 0u);
    if (dm) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (!(dm & (1u << q))) continue;
        *reinterpret_cast<ulonglong2*>(key_at(t, base + q)) =
            make_ulonglong2(st.key[lane * 4 + q], st.score[lane * 4 + q]);
      }
      const uint32_t nd = st.dig[lane];
      if (nd != dw) *reinterpret_cast<uint32_t*>(t.digests + base) = nd;
    }
    uint32_t total;
    uint32_t pos = prefix_small(__popc(dm), total);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (dm & (1u << q)) st.list[pos++] = static_cast<uint8_t>(lane * 4 + q);
    __syncwarp();
    // four rows per tile per pass, loads in flight together; a bucket's rows
    // are contiguous and all in HBM or all in host memory (the split falls
    // on a bucket boundary)
    float* const rows = row_ptr(t, b * kSlots);
    for (uint32_t p0 = lane >> 3; p0 < total; p0 += 16) {
      float* dst[4];
      const float* src[4];
      bool ok[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t p = p0 + 4 * r;
        ok[r] = p < total;
        const uint32_t slot = ok[r] ? st.list[p] : 0;
        dst[r] = rows + slot * t.dim;
        src[r] = values_in + static_cast<uint64_t>(ok[r] ? st.occ[slot] : 0) * t.dim;
      }
      tile_copy_rows<4>(dst, src, ok, t.dim, sub, vec);
    }
    __syncwarp();
  }
#if HKV_UPSERT_PIPELINE
  if (in_flight) wait_copy(parity);  // only after a timed-out wait: let the copy land first
#endif
  if (lane == 0) {
    if (kDual) {  // dual_finish_kernel turns these into the call's counts
      if (n_fill) atomicAdd(&t.stats->fills, n_fill);
      // net admitted keys of this pass (two's complement: may be negative)
      if (n_adm) atomicAdd(reinterpret_cast<unsigned long long*>(scr.cursor + 2), n_adm);
    } else {
      if (n_upd) atomicAdd(&t.stats->updated, n_upd);
      if (n_adm) atomicAdd(&t.stats->admitted, n_adm);
      if (n_evi) atomicAdd(&t.stats->evicted, n_evi);
      if (n_rej) atomicAdd(&t.stats->rejected, n_rej);
      if (n_adm != n_evi) atomicAdd(&t.stats->size, n_adm - n_evi);
    }
  }
}

// ---------------------------------------------------------------------------
// Sparse-batch bucket pass (single mode, plain insert_or_assign, batches of
// at most four keys per table bucket on average: large tables fed skewed or
// modest batches).  Most touched buckets then hold one or two of the batch's
// keys, and a warp per bucket spends about a thousand instructions on set-up
// and warp-wide steps whatever the bucket receives.  Here an 8-lane tile
// owns a bucket (four buckets per warp):
//   1. it reads the first 16 positions of the bucket's stage run and lists
//      the bucket's keys (at most 8) in stage order;
//   2. every key is looked up through the digest line (HKV Algorithm 1) and
//      the (key, score) pairs of its candidate slots; a resident key gets its
//      new score (Algorithm 2, found branch), all before any placement;
//   3. the absent keys take the free slots (zero digest bytes) in slot order;
//   4. for the E absent keys left the tile removes, E times, the lowest rank
//      (score, new, key) among the bucket's slots and those keys: one pass
//      over the bucket's 128 pairs (16 per lane) and a tile arg-min per
//      removal (an incoming key outranks a resident of equal score); the
//      keys still pending take the removed slots;
//   5. key / score pairs and digest bytes are written as decided, and the
//      value rows of the keys that ended resident are copied, four in flight.
// A bucket whose run does not end within 16 positions, or that has more than
// 8 keys, is left untouched and marked for the general bucket kernel, which a
// second launch runs on those buckets only.  The results equal the general
// kernel's: each bucket ends with the 128 highest ranks of its residents
// (after their updates) and its absent keys.
// ---------------------------------------------------------------------------
#ifndef HKV_TILE_MIN_BLOCKS
#define HKV_TILE_MIN_BLOCKS 4
#endif
constexpr uint8_t kMarkDeferred = 2;

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}
constexpr int kTileRun = 16;       // stage positions a tile reads, two per lane
constexpr int kTileMaxEntries = 8;  // keys per bucket the tile path takes

// Lowest rank (score, new, key) over the 8 lanes of a tile, with its slot.
__device__ __forceinline__ void tile_min_rank(uint64_t& s, uint32_t& nw, uint64_t& k,
                                              uint32_t& slot, unsigned tmask) {
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) {
    const uint64_t s2 = __shfl_xor_sync(tmask, s, o);
    const uint32_t n2 = __shfl_xor_sync(tmask, nw, o);
    const uint64_t k2 = __shfl_xor_sync(tmask, k, o);
    const uint32_t l2 = __shfl_xor_sync(tmask, slot, o);
    if (rank3_less(s2, n2, k2, s, nw, k)) {
      s = s2;
      nw = n2;
      k = k2;
      slot = l2;
    }
  }
}

// kDual: the buckets of a dual-mode pass (the keys routed to each bucket, all
// absent; rank (score, key); keys the pass displaces go to the retry list
// in the first pass (collect_retry); each bucket's summary is rewritten).
template <bool kLfu, bool kDual>
__global__ void __launch_bounds__(kThreads, HKV_TILE_MIN_BLOCKS) upsert_tile_kernel(
    TableView t, UpsertScratch scr, const float* values_in, ScoreRule rule, bool vec,
    bool collect_retry) {
  // per tile, its bucket's keys in stage order: key, batch index, increment,
  // score (absent keys), the slot a resident key holds or an absent key
  // ends in (-1: none), and a resident key's old score
  constexpr int kTiles = kThreads / 8;
  __shared__ uint64_t ekey_sh[kTiles][kTileMaxEntries];
  __shared__ uint64_t einc_sh[kTiles][kTileMaxEntries];
  __shared__ uint64_t escore_sh[kTiles][kTileMaxEntries];
  __shared__ uint32_t eidx_sh[kTiles][kTileMaxEntries];
  __shared__ int32_t eslot_sh[kTiles][kTileMaxEntries];
  __shared__ uint8_t xslot_sh[kTiles][kTileMaxEntries];  // slots removed, in order
  __shared__ uint32_t retry_sh[kTiles][kTileMaxEntries];  // dual: keys to route again
  pdl_wait();
  pdl_trigger();
  const unsigned lane = lane_id();
  const unsigned sub = lane & 7u;
  const unsigned tb = lane & 24u;
  const unsigned tmask = 0xFFu << tb;
  const int tw = threadIdx.x >> 3;
  uint64_t* ekey = ekey_sh[tw];
  uint64_t* einc = einc_sh[tw];
  uint64_t* escore = escore_sh[tw];
  uint32_t* eidx = eidx_sh[tw];
  int32_t* eslot = eslot_sh[tw];
  uint8_t* xslot = xslot_sh[tw];
  uint32_t* rtry = retry_sh[tw];
  constexpr uint32_t kNew = kDual ? 0u : 1u;  // rank (score, new, key) or (score, key)
  auto score_of = [&](uint32_t e, uint64_t inc, bool resident, uint64_t old) -> uint64_t {
    if (kLfu) return policy_score(rule, e, inc, resident, old);
    return rule.in ? rule.in[e] : rule.clock;
  };
  const uint64_t T = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 3;
  const uint64_t tile = (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  const uint64_t nb = t.num_buckets;
  const uint64_t S = scr.map_size, smask = S - 1;
  uint32_t n_upd = 0, n_adm = 0, n_evi = 0, n_rej = 0;  // lane sub == 0 of each tile
  int32_t n_net = 0;
  uint32_t n_fill = 0;  // dual: net placements of the pass, free-slot placements

  // the tile's buckets tile, tile + T, ..., eight candidates per mark load
  for (uint64_t g0 = tile; g0 < nb; g0 += 8 * T) {
    const uint64_t x = g0 + sub * T;
    unsigned todo = (__ballot_sync(tmask, x < nb && scr.mark[x] == 1) >> tb) & 0xFFu;
    while (todo) {
      const uint64_t b = g0 + (__ffs(todo) - 1) * T;
      todo &= todo - 1;
      const uint64_t row0 = b * kSlots;
      // the bucket's (key, score) pairs into L1 now: the candidate checks and
      // the eviction rounds read them after the stage and digest loads
      prefetch_l1(key_at(t, row0 + 16 * sub));
      prefetch_l1(key_at(t, row0 + 16 * sub + 8));
      // ---- 1. the bucket's keys: stage positions lo + sub and lo + 8 + sub
      const uint64_t lo = area_start(b, S, nb, scr.area_shift);
      const uint64_t a_end = area_start(b + 1, S, nb, scr.area_shift);
      uint64_t key[2], inc[2];
      uint32_t raw[2], bkt[2];
      unsigned stop = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint64_t j = lo + 8 * h + sub;
        key[h] = scr.stage_keys[j & smask];
        raw[h] = scr.stage_idx[j & smask];
        inc[h] = kLfu ? scr.stage_inc[j & smask] : 0ull;
        bkt[h] = kDual ? scr.stage_bkt[j & smask] : 0u;
        stop |= ((__ballot_sync(tmask, key[h] == kEmptyKey && j >= a_end) >> tb) & 0xFFu) << (8 * h);
      }
      const int end = stop ? __ffs(stop) - 1 : kTileRun;  // first position past the run
      unsigned em = 0;
      uint64_t sin[2];  // non-LFU rules: the score of each of this lane's keys
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const bool mine =
            key[h] != kEmptyKey && static_cast<int>(8 * h + sub) < end &&
            (kDual ? bkt[h] == static_cast<uint32_t>(b) : bucket_of_hash(t, hash64(key[h])) == b);
        em |= ((__ballot_sync(tmask, mine) >> tb) & 0xFFu) << (8 * h);
        sin[h] = (!kLfu && mine && rule.in) ? rule.in[(raw[h] & ~kHitMark) - 1] : rule.clock;
      }
      const int ne = __popc(em);
      if (!stop || ne > kTileMaxEntries) {  // a long run or many keys: general kernel
        if (sub == 0) scr.mark[b] = kMarkDeferred;
        continue;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const unsigned pos = 8 * h + sub;
        if ((em >> pos) & 1u) {
          const int i = __popc(em & ((1u << pos) - 1u));
          ekey[i] = key[h];
          eidx[i] = (raw[h] & ~kHitMark) - 1;
          einc[i] = inc[h];
          if (!kLfu) escore[i] = sin[h];
        }
      }
      __syncwarp(tmask);
      // ---- 2. look every key up (this lane: digest bytes of slots 16 sub ..)
      const uint4 dg = *reinterpret_cast<const uint4*>(t.digests + row0 + sub * 16);
      unsigned hm = 0;  // entries resident (none in dual mode: routed keys are absent)
      for (int i = 0; i < ne; ++i) {
        if (kDual) {
          if (sub == 0) {
            eslot[i] = -1;
            if (kLfu) escore[i] = score_of(eidx[i], einc[i], false, 0ull);
          }
          continue;
        }
        const uint64_t ke = ekey[i];
        const uint32_t pat = digest_of_hash(hash64(ke)) * 0x01010101u;
        uint32_t cm = byte_match4(dg.x, pat) | (byte_match4(dg.y, pat) << 4) |
                      (byte_match4(dg.z, pat) << 8) | (byte_match4(dg.w, pat) << 12);
        int hs = -1;
        uint64_t old = 0;
        while (cm) {
          const int c = __ffs(cm) - 1;
          cm &= cm - 1;
          const ulonglong2 p = *reinterpret_cast<const ulonglong2*>(key_at(t, row0 + sub * 16 + c));
          if (p.x == ke) {
            hs = static_cast<int>(sub * 16 + c);
            old = p.y;
            break;
          }
        }
        const unsigned hb = (__ballot_sync(tmask, hs >= 0) >> tb) & 0xFFu;
        if (hb) {
          hm |= 1u << i;
          if (sub == static_cast<unsigned>(__ffs(hb) - 1)) {  // the lane that found it
            eslot[i] = hs;
            *score_at(t, row0 + hs) = kLfu ? score_of(eidx[i], einc[i], true, old) : escore[i];
          }
        } else if (sub == 0) {
          eslot[i] = -1;
          if (kLfu) escore[i] = score_of(eidx[i], einc[i], false, 0ull);
        }
      }
      const uint32_t nh = __popc(hm);
      const uint32_t A = ne - nh;
      if (sub == 0) n_upd += nh;
      // ---- 3. free slots (zero digest bytes; bit j = slot 16 sub + j) to the
      // absent keys in stage order, in slot order
      const uint32_t fm = byte_eq_mask4(dg.x, 0u) | (byte_eq_mask4(dg.y, 0u) << 4) |
                          (byte_eq_mask4(dg.z, 0u) << 8) | (byte_eq_mask4(dg.w, 0u) << 12);
      const uint32_t nf = __popc(fm);
      uint32_t pre = nf;  // inclusive prefix over the tile's lanes, then exclusive
#pragma unroll
      for (int d = 1; d < 8; d <<= 1) {
        const uint32_t y = __shfl_up_sync(tmask, pre, d, 8);
        if (sub >= static_cast<unsigned>(d)) pre += y;
      }
      const uint32_t F = __shfl_sync(tmask, pre, tb + 7);
      pre -= nf;
      __syncwarp(tmask);  // escore / eslot written above
      const unsigned amask = ((1u << ne) - 1u) & ~hm;  // absent entries
      unsigned pend = amask;                           // absent entries not placed yet
      {
        uint32_t r = 0;
        for (unsigned m = amask; m && r < F; m &= m - 1, ++r) {
          const int i = __ffs(m) - 1;
          pend &= ~(1u << i);
          if (pre <= r && r < pre + nf) {
            const uint32_t slot = sub * 16 + __fns(fm, 0, static_cast<int>(r - pre + 1));
            *reinterpret_cast<ulonglong2*>(key_at(t, row0 + slot)) =
                make_ulonglong2(ekey[i], escore[i]);
            t.digests[row0 + slot] = static_cast<uint8_t>(digest_of_hash(hash64(ekey[i])));
            eslot[i] = static_cast<int32_t>(slot);
          }
        }
      }
      // ---- 4. evictions: E = the absent keys left
      const uint32_t E = __popc(pend);
      uint32_t evicted = 0, displaced_earlier = 0, nretry = 0;
      if (E) {
        __syncwarp(tmask);  // the placements and new scores are visible
        // the slots free at entry (now holding keys of this call) rank as new:
        // this lane's slots 8 q + sub lie in lane q/2's digest bytes
        uint32_t newm = 0;  // bit q: slot 8 q + sub
#pragma unroll
        for (int l = 0; l < 8; ++l) {
          const uint32_t f = __shfl_sync(tmask, fm, tb + l);
          newm |= ((f >> sub) & 1u) << (2 * l);
          newm |= ((f >> (8 + sub)) & 1u) << (2 * l + 1);
        }
        uint32_t removed = 0;  // bit q: slot 8 q + sub taken out
        uint32_t nx = 0;       // slots taken out
        for (uint32_t x = 0; x < E; ++x) {
          uint64_t bs = ~0ull, bk = ~0ull;
          uint32_t bn = 1u, bl = kNone;
#pragma unroll
          for (int g = 0; g < 16; g += 4) {
            ulonglong2 p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              p[i] = *reinterpret_cast<const ulonglong2*>(key_at(t, row0 + 8 * (g + i) + sub));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int q = g + i;
              const uint32_t cn = (newm >> q) & kNew;
              if (!((removed >> q) & 1u) &&
                  (bl == kNone || rank3_less(p[i].y, cn, p[i].x, bs, bn, bk))) {
                bs = p[i].y;
                bk = p[i].x;
                bn = cn;
                bl = 8 * q + sub;
              }
            }
          }
          tile_min_rank(bs, bn, bk, bl, tmask);
          // the lowest pending key (rank (score, 1, key)), if any is left
          int pi = -1;
          uint64_t ps = 0, pk = 0;
          for (unsigned m = pend; m; m &= m - 1) {
            const int i = __ffs(m) - 1;
            if (pi < 0 || rank3_less(escore[i], kNew, ekey[i], ps, kNew, pk)) {
              pi = i;
              ps = escore[i];
              pk = ekey[i];
            }
          }
          if (pi >= 0 && rank3_less(ps, kNew, pk, bs, bn, bk)) {
            pend &= ~(1u << pi);  // rejected
            if (kDual && collect_retry && sub == 0) rtry[nretry] = eidx[pi];
            ++nretry;
            continue;
          }
          // the slot goes: a key of this call placed there is displaced, a
          // pre-call resident is evicted (also when this call updated it: a
          // resident key's new score can still be the lowest), and no key of
          // this call's row goes to it any more
          if ((bl & 7u) == sub) removed |= 1u << (bl >> 3);
          // placed by this pass (free at entry): a key of this call displaced
          const bool fresh = (__shfl_sync(tmask, fm, tb + (bl >> 4)) >> (bl & 15u)) & 1u;
          // dual mode's second pass: a key the first pass placed is also a
          // key of this call
          const bool earlier = kDual && !fresh && !collect_retry && absent_in_call(scr, bk);
          if (sub == 0) {
            xslot[nx] = static_cast<uint8_t>(bl);
            for (int i = 0; i < ne; ++i) {
              if (eslot[i] != static_cast<int32_t>(bl)) continue;
              eslot[i] = -1;
              if (kDual && collect_retry && fresh) rtry[nretry] = eidx[i];
            }
          }
          if (kDual && collect_retry && fresh) ++nretry;
          ++nx;
          if (earlier) ++displaced_earlier;
          else if (!fresh) ++evicted;
          __syncwarp(tmask);
        }
        // the pending keys left take the removed slots, in order
        uint32_t r = 0;
        for (unsigned m = pend; m; m &= m - 1, ++r) {
          const int i = __ffs(m) - 1;
          const uint32_t slot = xslot[r];
          if (sub == 0) {
            *reinterpret_cast<ulonglong2*>(key_at(t, row0 + slot)) =
                make_ulonglong2(ekey[i], escore[i]);
            t.digests[row0 + slot] = static_cast<uint8_t>(digest_of_hash(hash64(ekey[i])));
            eslot[i] = static_cast<int32_t>(slot);
          }
        }
      }
      __syncwarp(tmask);
      // counts: absent keys resident at the end are admitted
      uint32_t adm = 0;
      for (unsigned m = amask; m; m &= m - 1) adm += eslot[__ffs(m) - 1] >= 0 ? 1u : 0u;
      if (kDual) {
        // the pass's net placements (keys of earlier passes of this call it
        // displaced count against them), its free-slot placements, the keys
        // to route again, and the bucket's new summary
        const uint32_t placed_free = A < F ? A : F;
        if (sub == 0) {
          n_net += static_cast<int32_t>(adm) - static_cast<int32_t>(displaced_earlier);
          n_fill += placed_free;
        }
        if (collect_retry && nretry) {
          uint32_t at = 0;
          if (sub == 0) at = atomicAdd(scr.cursor + 4, nretry);
          at = __shfl_sync(tmask, at, tb);
          for (uint32_t r = sub; r < nretry; r += 8) scr.retry[at + r] = rtry[r];
        }
        uint32_t cnt = 0;
        uint64_t mn = ~0ull;
#pragma unroll
        for (int g = 0; g < 16; g += 4) {
          ulonglong2 p[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            p[i] = *reinterpret_cast<const ulonglong2*>(key_at(t, row0 + 8 * (g + i) + sub));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (p[i].x == kEmptyKey) continue;
            ++cnt;
            mn = min(mn, static_cast<uint64_t>(p[i].y));
          }
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
          cnt += __shfl_xor_sync(tmask, cnt, o);
          mn = min(mn, static_cast<uint64_t>(__shfl_xor_sync(tmask, mn, o)));
        }
        if (sub == 0) {
          t.summary[b].min_score = cnt ? mn : 0ull;
          t.summary[b].count = cnt;
        }
      } else if (sub == 0) {
        n_adm += adm;
        n_rej += A - adm;
        n_evi += evicted;
      }
      // ---- 5. the value rows of the keys resident at the end, four in flight
      float* const rows = row_ptr(t, row0);
      unsigned cm = 0;  // entries to copy
      for (int i = 0; i < ne; ++i) cm |= eslot[i] >= 0 ? (1u << i) : 0u;
      while (cm) {
        float* dst[4];
        const float* src[4];
        bool ok[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          ok[r] = cm != 0;
          const int i = ok[r] ? __ffs(cm) - 1 : 0;
          if (ok[r]) cm &= cm - 1;
          dst[r] = rows + (ok[r] ? eslot[i] : 0) * t.dim;
          src[r] = values_in + static_cast<uint64_t>(ok[r] ? eidx[i] : 0) * t.dim;
        }
        tile_copy_rows<4>(dst, src, ok, t.dim, sub, vec);
      }
      __syncwarp(tmask);  // the lists are read before the next bucket writes them
    }
  }
  const unsigned kFull = 0xFFFFFFFFu;
  using ull = unsigned long long;
  if (kDual) {  // dual_finish_kernel turns these into the call's counts
    const int32_t net = __reduce_add_sync(kFull, n_net);
    const uint32_t fills = __reduce_add_sync(kFull, n_fill);
    if (lane == 0) {
      if (fills) atomicAdd(&t.stats->fills, static_cast<ull>(fills));
      if (net) atomicAdd(reinterpret_cast<ull*>(scr.cursor + 2),
                         static_cast<ull>(static_cast<long long>(net)));
    }
    return;
  }
  const uint32_t u = __reduce_add_sync(kFull, n_upd), ad = __reduce_add_sync(kFull, n_adm);
  const uint32_t ev = __reduce_add_sync(kFull, n_evi), rj = __reduce_add_sync(kFull, n_rej);
  if (lane == 0) {
    if (u) atomicAdd(&t.stats->updated, static_cast<ull>(u));
    if (ad) atomicAdd(&t.stats->admitted, static_cast<ull>(ad));
    if (ev) atomicAdd(&t.stats->evicted, static_cast<ull>(ev));
    if (rj) atomicAdd(&t.stats->rejected, static_cast<ull>(rj));
    if (ad != ev) atomicAdd(&t.stats->size, static_cast<ull>(ad) - static_cast<ull>(ev));
  }
}

// ---------------------------------------------------------------------------
// Dual mode (Algorithm 3), as routing plus bucket ownership.
//
// Algorithm 3 sends an absent key to one of its two buckets: the less
// occupied one while either has room (D1), else the one whose lowest rank is
// lower, where it is admitted only if it outranks that minimum (D2).  The
// bucket then runs Algorithm 2's placement.  Here each absent key is routed
// by those rules on the bucket summaries (occupancy and lowest score, exact
// as of the last pass over the bucket) and staged in the chosen bucket's
// area; the bucket kernel of single mode then places every bucket's routed
// keys with one warp per bucket (free slots first, then the top 128 by rank
// (score, key) of entries and keys survive).  Keys that the first pass
// displaces get one more routing with the summaries that pass left, and a
// second pass.  Whatever the routing chose, a key that ends up absent lost to
// a full bucket all of whose entries outrank it, which is the invariant the
// tests check; the processing order, and so which keys win near the margin,
// is this design's, as it is any parallel kernel's.
// ---------------------------------------------------------------------------

// Algorithm 3's choice between b1 and b2 for a key of score s, from the
// summaries.  Returns kNoBucket when the key cannot enter either bucket: both
// full and s below both lowest scores (the summaries' lowest scores are never
// above the true ones, so such a key would be rejected anyway).
constexpr uint64_t kNoBucket = ~0ull;

__device__ __forceinline__ uint64_t route_bucket(const TableView& t, uint64_t b1, uint64_t b2,
                                                 uint64_t s) {
  const BucketSummary x = t.summary[b1], y = t.summary[b2];
  const uint32_t f1 = kSlots - min(x.count, static_cast<unsigned>(kSlots));
  const uint32_t f2 = kSlots - min(y.count, static_cast<unsigned>(kSlots));
  if (f1 || f2) return f2 > f1 ? b2 : b1;  // D1: the less occupied, ties to b1
  const bool use2 = y.min_score < x.min_score;  // D2: the lower minimum
  const uint64_t m = use2 ? y.min_score : x.min_score;
  if (s < m) return kNoBucket;
  return use2 ? b2 : b1;
}

// Stage key k (batch index i) in bucket target's area of the dual stage.
// Keys are unique here (the batch was de-duplicated), so a CAS that loses
// only means another key took the position.
__device__ __forceinline__ void stage_routed(const TableView& t, const UpsertScratch& sc,
                                             uint64_t target, uint64_t k, uint64_t h, uint64_t i,
                                             uint64_t inc) {
  const uint64_t S = sc.map_size, mask = S - 1, B = t.num_buckets;
  const uint64_t lo = area_start(target, S, B, sc.area_shift);
  uint64_t p = stage_home(h, lo, area_start(target + 1, S, B, sc.area_shift) - lo) & mask;
  // S >= 2n: a free position exists, so the probe ends within S steps
  for (uint64_t tries = 0; tries < S; ++tries) {
    if (atomicCAS(reinterpret_cast<unsigned long long*>(sc.stage_keys + p), kEmptyKey, k) ==
        kEmptyKey)
      break;
    p = (p + 1) & mask;
  }
  sc.stage_idx[p] = static_cast<uint32_t>(i) + 1;
  sc.stage_bkt[p] = static_cast<uint32_t>(target);
  if (sc.stage_inc) sc.stage_inc[p] = inc;
  sc.mark[target] = 1;
}

// Pass 1: resident keys update value (and score) in place; absent keys are
// flagged in the dedup map (for the counts) and routed.
#ifndef HKV_ASSIGN_MIN_BLOCKS
#define HKV_ASSIGN_MIN_BLOCKS 4
#endif
#ifndef HKV_ROUTE_MIN_BLOCKS
#define HKV_ROUTE_MIN_BLOCKS 4
#endif

// Candidate mask of 16 digest bytes: bit j set when byte j may equal the
// key's digest (`pat` = digest * 0x01010101).
__device__ __forceinline__ uint32_t digest_mask16(const uint4& dg, uint32_t pat) {
  return byte_match4(dg.x, pat) | (byte_match4(dg.y, pat) << 4) | (byte_match4(dg.z, pat) << 8) |
         (byte_match4(dg.w, pat) << 12);
}

// Removes and returns the lowest set bit of a 128-bit slot mask (-1: empty).
__device__ __forceinline__ int take_slot(uint4& m) {
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

// Candidate slots of the warp's probing keys (HKV Algorithm 1; both
// candidate buckets with kPair, HKV §3.4: two fixed-length line loads per
// key): tile j loads the digest lines of keys 8j..8j+7, four lines in flight,
// and each key's 128-bit masks reach its lane through `msk` (32 keys x 16 x
// 16 bits: b1's line, then b2's).  Read-only loads: no thread of the calling
// kernels writes digests.
template <bool kPair>
__device__ __forceinline__ void warp_candidates(const TableView& t, unsigned probe, uint32_t b1,
                                                uint32_t b2, uint32_t pat, unsigned lane,
                                                uint16_t (*msk)[16], uint4& c1, uint4& c2) {
  constexpr unsigned kFull = 0xFFFFFFFFu;
  constexpr int KG = kPair ? 2 : 4;  // keys per group
  const unsigned tile = lane >> 3, sub = lane & 7u;
#pragma unroll
  for (int g = 0; g < 8; g += KG) {
    uint4 d1[KG], d2[KG];
#pragma unroll
    for (int m = 0; m < KG; ++m) {
      const unsigned src = tile * 8 + g + m;
      const uint32_t x1 = __shfl_sync(kFull, b1, src);
      const uint32_t x2 = kPair ? __shfl_sync(kFull, b2, src) : 0u;
      if ((probe >> src) & 1u) {
        d1[m] = ld_nc_v4(t.digests + static_cast<uint64_t>(x1) * kSlots + sub * 16);
        if (kPair) d2[m] = ld_nc_v4(t.digests + static_cast<uint64_t>(x2) * kSlots + sub * 16);
      }
    }
#pragma unroll
    for (int m = 0; m < KG; ++m) {
      const unsigned src = tile * 8 + g + m;
      const uint32_t p = __shfl_sync(kFull, pat, src);
      const bool on = (probe >> src) & 1u;
      msk[src][sub] = static_cast<uint16_t>(on ? digest_mask16(d1[m], p) : 0u);
      if (kPair) msk[src][8 + sub] = static_cast<uint16_t>(on ? digest_mask16(d2[m], p) : 0u);
    }
  }
  __syncwarp();
  c1 = *reinterpret_cast<const uint4*>(&msk[lane][0]);
  c2 = kPair ? *reinterpret_cast<const uint4*>(&msk[lane][8]) : make_uint4(0, 0, 0, 0);
  __syncwarp();  // every lane has its masks before the next probe writes them
}

// The slot of the lane's key k (or -1) and the bucket holding it, from its
// candidate masks: the first candidate of each bucket confirmed together,
// then the rest (rare) in order; a key sits in at most one of its buckets.
// Keys are read with read-only loads: no thread of the calling kernels
// writes keys (the scores beside them are not read here).
__device__ __forceinline__ int confirm_slot(const TableView& t, uint64_t k, uint32_t b1,
                                            uint32_t b2, uint4 c1, uint4 c2, uint32_t& bk) {
  bk = b1;
  const int a1 = take_slot(c1), a2 = take_slot(c2);
  uint64_t k1 = 0, k2 = 0;
  if (a1 >= 0) k1 = ld_nc_u64(key_at(t, static_cast<uint64_t>(b1) * kSlots + a1));
  if (a2 >= 0) k2 = ld_nc_u64(key_at(t, static_cast<uint64_t>(b2) * kSlots + a2));
  if (a1 >= 0 && k1 == k) return a1;
  if (a2 >= 0 && k2 == k) {
    bk = b2;
    return a2;
  }
  for (int c = take_slot(c1); c >= 0; c = take_slot(c1))
    if (ld_nc_u64(key_at(t, static_cast<uint64_t>(b1) * kSlots + c)) == k) return c;
  for (int c = take_slot(c2); c >= 0; c = take_slot(c2)) {
    if (ld_nc_u64(key_at(t, static_cast<uint64_t>(b2) * kSlots + c)) == k) {
      bk = b2;
      return c;
    }
  }
  return -1;
}

// Resident keys of the warp's 32 (slot >= 0): tile j copies the input rows
// of keys 8j..8j+7 (batch indices base + 8j ..) over their table rows, two
// rows in flight (more hold registers the calling kernels need).
__device__ __forceinline__ void warp_copy_rows(const TableView& t, int slot, uint32_t bk,
                                               const float* values, uint64_t base, bool vec,
                                               unsigned lane) {
  const unsigned tile = lane >> 3, sub = lane & 7u;
  const unsigned tmask = 0xFFu << (tile * 8);
  unsigned rows = (__ballot_sync(0xFFFFFFFFu, slot >= 0) >> (tile * 8)) & 0xFFu;
  while (rows) {
    float* dst[2];
    const float* src[2];
    bool ok[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      ok[r] = rows != 0;
      const unsigned j = ok[r] ? __ffs(rows) - 1 : 0u;
      if (ok[r]) rows &= rows - 1;
      const unsigned from = tile * 8 + j;
      const int s_ = __shfl_sync(tmask, slot, from);
      const uint32_t b_ = __shfl_sync(tmask, bk, from);
      dst[r] = ok[r] ? row_ptr(t, static_cast<uint64_t>(b_) * kSlots + s_) : nullptr;
      src[r] = ok[r] ? values + (base + from) * t.dim : values;
    }
    tile_copy_rows<2>(dst, src, ok, t.dim, sub, vec);
  }
}

// A warp takes 32 consecutive keys, one per lane for everything scalar (the
// dedup lookup, hash, candidate confirmation, score update, routing and
// staging), so the 32 keys' accesses are in flight together; the 128-byte
// transfers (digest lines, value rows) run on the four 8-lane tiles.  The
// two bucket summaries of each key are brought into L2 at the start, for
// the routing of the keys found absent.
__global__ void __launch_bounds__(kThreads, HKV_ROUTE_MIN_BLOCKS) dual_route_kernel(
    TableView t, UpsertScratch sc, uint64_t n, const uint64_t* keys, const float* values,
    ScoreRule rule, bool vec) {
  __shared__ __align__(16) uint16_t masks_sh[kThreads / 32][32][16];
  pdl_wait();
  pdl_trigger();
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const unsigned lane = lane_id();
  uint16_t(*msk)[16] = masks_sh[threadIdx.x >> 5];
  const uint64_t warps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
  unsigned long long upd = 0, absent = 0;
  for (uint64_t base = ((static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * 32;
       base < n; base += warps * 32) {
    const uint64_t i = base + lane;
    const uint64_t k = i < n ? keys[i] : kEmptyKey;
    const uint32_t ms = i < n && !is_reserved(k) ? map_last_occurrence(sc, k, i) : kNone;
    const bool live = ms != kNone;  // the key's last occurrence in the batch
    const uint64_t h = hash64(k);
    const uint32_t b1 = static_cast<uint32_t>(bucket_of_hash(t, h));
    const uint32_t b2 = static_cast<uint32_t>(bucket2_of(t, k, b1));
    if (live) {
      prefetch_l2(t.summary + b1);
      prefetch_l2(t.summary + b2);
    }
    const unsigned probe = __ballot_sync(kFull, live);
    if (!probe) continue;
    uint4 c1, c2;
    warp_candidates<true>(t, probe, b1, b2, digest_of_hash(h) * 0x01010101u, lane, msk, c1, c2);
    uint32_t bk = b1;
    const int slot = live ? confirm_slot(t, k, b1, b2, c1, c2, bk) : -1;
    if (live) {
      sc.absent[ms] = slot < 0 ? 1 : 0;  // read by the second bucket pass
      const uint64_t inc = entry_inc(sc, ms);
      if (slot >= 0) {
        uint64_t* sp = score_at(t, static_cast<uint64_t>(bk) * kSlots + static_cast<uint64_t>(slot));
        *sp = policy_score(rule, i, inc, true, rule.lfu() ? *sp : 0ull);
        ++upd;
      } else {
        ++absent;
        const uint64_t target = route_bucket(t, b1, b2, policy_score(rule, i, inc, false, 0));
        if (target != kNoBucket) stage_routed(t, sc, target, k, h, i, inc);
      }
    }
    warp_copy_rows(t, slot, bk, values, base, vec, lane);
  }
  warp_add(&t.stats->updated, upd);
  // the call's absent keys; dual_finish_kernel splits them into admitted
  // and rejected
  warp_add(reinterpret_cast<unsigned long long*>(sc.cursor + 6), absent);
}

// Pass 2: the keys the first bucket pass displaced are routed again with the
// summaries that pass left.  One thread per key.
__global__ void __launch_bounds__(kThreads) dual_retry_kernel(TableView t, UpsertScratch sc,
                                                              const uint64_t* keys,
                                                              ScoreRule rule) {
  pdl_wait();
  pdl_trigger();
  const uint32_t nretry = sc.cursor[4];
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t w = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; w < nretry;
       w += stride) {
    const uint32_t i = sc.retry[w];
    const uint64_t k = keys[i];
    const uint64_t inc = sc.inc ? sc.inc[map_find(sc.map_keys, sc.map_size - 1, k)] : 0ull;
    const uint64_t h = hash64(k);
    const uint64_t b1 = bucket_of_hash(t, h);
    const uint64_t target =
        route_bucket(t, b1, bucket2_of(t, k, b1), policy_score(rule, i, inc, false, 0));
    if (target != kNoBucket) stage_routed(t, sc, target, k, h, i, inc);
  }
}

// The call's counts: admitted = the bucket passes' net placements (keys of
// the call resident at its end), rejected = absent keys - admitted, evicted =
// admitted - fills (every other admitted key displaced a resident); size
// grows by fills.
__global__ void dual_finish_kernel(TableView t, UpsertScratch sc) {
  const unsigned long long adm = *reinterpret_cast<unsigned long long*>(sc.cursor + 2);
  const unsigned long long absent = *reinterpret_cast<unsigned long long*>(sc.cursor + 6);
  const unsigned long long fills = t.stats->fills;
  t.stats->admitted += adm;
  t.stats->rejected += absent - adm;
  t.stats->evicted += adm - fills;
  t.stats->size += fills;
  t.stats->fills = 0;
}

// ---------------------------------------------------------------------------
// assign (updater) and erase (inserter).
// ---------------------------------------------------------------------------
template <bool kDual>
__global__ void __launch_bounds__(kThreads, HKV_ASSIGN_MIN_BLOCKS) assign_kernel(
    TableView t, UpsertScratch sc, uint64_t n, const uint64_t* keys, const float* values,
    ScoreRule rule, bool keep_scores, bool vec) {
  __shared__ __align__(16) uint16_t masks_sh[kThreads / 32][32][16];
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const unsigned lane = lane_id();
  uint16_t(*msk)[16] = masks_sh[threadIdx.x >> 5];
  const uint64_t warps = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5;
  unsigned long long upd = 0;
  for (uint64_t base = ((static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * 32;
       base < n; base += warps * 32) {
    const uint64_t i = base + lane;
    const uint64_t k = i < n ? keys[i] : kEmptyKey;
    const bool valid = i < n && !is_reserved(k);
    // the dedup lookup's first position is read while the digest lines load
    MapProbe mp{0, 0, 0};
    if (valid) mp = map_probe_start(sc, k);
    const uint64_t h = hash64(k);
    const uint32_t b1 = static_cast<uint32_t>(bucket_of_hash(t, h));
    const uint32_t b2 = kDual ? static_cast<uint32_t>(bucket2_of(t, k, b1)) : b1;
    const unsigned probe = __ballot_sync(kFull, valid);
    if (!probe) continue;
    uint4 c1, c2;
    warp_candidates<kDual>(t, probe, b1, b2, digest_of_hash(h) * 0x01010101u, lane, msk, c1, c2);
    const uint32_t ms = valid ? map_last_occurrence_from(sc, k, i, mp) : kNone;
    const bool live = ms != kNone;  // the key's last occurrence in the batch
    uint32_t bk = b1;
    const int slot = live ? confirm_slot(t, k, b1, b2, c1, c2, bk) : -1;
    if (slot >= 0) {
      if (!keep_scores) {
        uint64_t* sp = score_at(t, static_cast<uint64_t>(bk) * kSlots + static_cast<uint64_t>(slot));
        *sp = policy_score(rule, i, entry_inc(sc, ms), true, rule.lfu() ? *sp : 0ull);
      }
      ++upd;
    }
    warp_copy_rows(t, slot, bk, values, base, vec, lane);
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
      if (atomicCAS(reinterpret_cast<unsigned long long*>(key_at(t, row)), k, kEmptyKey) == k) {
        t.digests[row] = 0;
        if (t.summary) atomicSub(&t.summary[b].count, 1u);  // dual mode: keep occupancy exact
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

namespace {
// A batch of at most four keys per table bucket on average: the stage marks
// the buckets it touches (the bucket passes visit only those), collapses
// repeated keys inside each warp, and plain insert_or_assign takes the
// register-resident bucket pass.
bool sparse_batch(uint64_t n, uint64_t num_buckets) { return n <= 4 * num_buckets; }

#ifndef HKV_STAGE_FACTOR
#define HKV_STAGE_FACTOR 2
#endif
uint64_t stage_entries(uint64_t n) {
  return next_pow2(n * HKV_STAGE_FACTOR < 64 ? 64 : n * HKV_STAGE_FACTOR);
}
}  // namespace

size_t upsert_scratch_bytes(uint64_t n, uint64_t num_buckets, ScratchKind kind, bool lfu) {
  const uint64_t m = stage_entries(n);
  size_t bytes = align256(m * 8) + align256(m * 4) + align256(64);
  if (kind == ScratchKind::kSingleUpsert) bytes += align256(num_buckets);
  if (kind == ScratchKind::kDualUpsert)
    bytes += align256(m) + align256(n * 4) + align256(m * 8) + 2 * align256(m * 4) +
             align256(num_buckets);
  if (lfu) bytes += align256(m * 8) * (kind == ScratchKind::kDualUpsert ? 2 : 1);
  return bytes;
}

UpsertScratch carve_upsert_scratch(void* base, uint64_t n, uint64_t num_buckets, ScratchKind kind,
                                   bool lfu) {
  UpsertScratch s{};
  const uint64_t m = stage_entries(n);
  char* p = static_cast<char*>(base);
  auto take = [&](size_t bytes) {
    char* q = p;
    p += align256(bytes);
    return q;
  };
  s.map_size = static_cast<uint32_t>(m);
  s.area_shift = kNoShift;
  if ((num_buckets & (num_buckets - 1)) == 0) {
    int lb = 0, lm = 0;
    while ((1ull << lb) < num_buckets) ++lb;
    while ((1ull << lm) < m) ++lm;
    s.area_shift = lm - lb;
  }
  s.map_keys = reinterpret_cast<uint64_t*>(take(m * 8));
  s.map_idx = reinterpret_cast<uint32_t*>(take(m * 4));
  s.cursor = reinterpret_cast<uint32_t*>(take(64));
  if (kind == ScratchKind::kSingleUpsert) {
    s.mark = reinterpret_cast<uint8_t*>(take(num_buckets));
    if (!sparse_batch(n, num_buckets)) s.mark = nullptr;  // dense batch: no marks
  }
  if (lfu) s.inc = reinterpret_cast<uint64_t*>(take(m * 8));
  if (kind == ScratchKind::kDualUpsert) {
    s.absent = reinterpret_cast<uint8_t*>(take(m));
    s.retry = reinterpret_cast<uint32_t*>(take(n * 4));
    s.stage_keys = reinterpret_cast<uint64_t*>(take(m * 8));
    s.stage_idx = reinterpret_cast<uint32_t*>(take(m * 4));
    s.stage_bkt = reinterpret_cast<uint32_t*>(take(m * 4));
    s.mark = reinterpret_cast<uint8_t*>(take(num_buckets));
    if (lfu) s.stage_inc = reinterpret_cast<uint64_t*>(take(m * 8));
  } else {  // the single-mode stage is the dedup map itself
    s.stage_keys = s.map_keys;
    s.stage_idx = s.map_idx;
    s.stage_inc = s.inc;
  }
  s.bytes = static_cast<size_t>(p - static_cast<char*>(base));
  return s;
}

namespace {

// One launch clears every scratch array of a call: the map keys to EMPTY, the
// map indices (and LFU sums) to 0, the counters and the bucket marks to 0,
// and in dual mode the routed stage's keys to EMPTY.  stage_only clears just
// the routed stage and the marks (between the two dual-mode passes).
// map_size is a power of two >= 64, and every array starts 256-byte aligned.
__global__ void __launch_bounds__(kThreads) clear_scratch_kernel(UpsertScratch s,
                                                                 uint64_t mark_bytes,
                                                                 bool stage_only) {
  pdl_wait();
  pdl_trigger();
  const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  const uint64_t pairs = s.map_size / 2;
  const bool routed = s.stage_keys != s.map_keys;
  for (uint64_t i = tid; i < pairs; i += stride) {
    if (!stage_only) {
      reinterpret_cast<ulonglong2*>(s.map_keys)[i] = make_ulonglong2(kEmptyKey, kEmptyKey);
      reinterpret_cast<uint2*>(s.map_idx)[i] = make_uint2(0u, 0u);
      if (s.inc) reinterpret_cast<ulonglong2*>(s.inc)[i] = make_ulonglong2(0ull, 0ull);
    }
    if (routed) reinterpret_cast<ulonglong2*>(s.stage_keys)[i] = make_ulonglong2(kEmptyKey, kEmptyKey);
  }
  if (!stage_only && tid < 16) s.cursor[tid] = 0u;
  if (s.mark)
    for (uint64_t i = tid; i < mark_bytes; i += stride) s.mark[i] = 0;
}

template <bool kLfu, bool kDual, bool kEvict>
cudaError_t launch_bucket_kernel(unsigned grid, const TableView& t, const UpsertScratch& s,
                                 const uint64_t* keys, const float* values, const ScoreRule& r,
                                 bool vec, cudaStream_t st, const UpsertExtra& ex) {
  const size_t smem =
      HKV_UPSERT_PIPELINE ? sizeof(BucketStage<kLfu>) * (kBucketThreads / 32) : 0;
  if (smem) {
    const cudaError_t e =
        cudaFuncSetAttribute(upsert_single_kernel<kLfu, kDual, kEvict>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_chained(upsert_single_kernel<kLfu, kDual, kEvict>, grid, kBucketThreads, smem, st,
                        t, s, keys, values, r, vec, ex);
}

// One bucket pass (single or dual mode).  Non-LFU rules become one score per
// call (the clock, folded with the epoch) unless the caller gives scores.
// insert_and_evict (single mode only) runs its own instance of the kernel,
// so the plain upsert carries none of the reporting code.
template <bool kDual>
cudaError_t launch_bucket_pass(const TableView& t, const UpsertScratch& s, const uint64_t* keys,
                               const float* values, const ScoreRule& rule, bool vec,
                               cudaStream_t st, const UpsertExtra& ex) {
  // one warp per bucket, at most one wave of resident blocks
  uint64_t blocks = (t.num_buckets * 32 + kBucketThreads - 1) / kBucketThreads;
  const uint64_t cap = static_cast<uint64_t>(sm_count()) * HKV_UPSERT_MIN_BLOCKS;
  const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
  const bool evict = !kDual && ex.ev_keys != nullptr;
  if (rule.lfu())
    return evict ? launch_bucket_kernel<true, kDual, !kDual>(grid, t, s, keys, values, rule, vec,
                                                             st, ex)
                 : launch_bucket_kernel<true, kDual, false>(grid, t, s, keys, values, rule, vec,
                                                            st, ex);
  ScoreRule r = rule;
  if (rule.policy != kCustomized) r.in = nullptr;
  if (rule.policy == kEpochLru) r.clock = rule.epoch_hi | (rule.clock & 0xFFFFFFFFull);
  r.policy = kCustomized;
  return evict ? launch_bucket_kernel<false, kDual, !kDual>(grid, t, s, keys, values, r, vec, st,
                                                            ex)
               : launch_bucket_kernel<false, kDual, false>(grid, t, s, keys, values, r, vec, st,
                                                           ex);
}

// The sparse-batch pass (single mode, plain insert_or_assign; and every pass
// of dual mode): the tile kernel, then the general kernel on the buckets it
// deferred.
template <bool kDual>
cudaError_t launch_tile_pass(const TableView& t, const UpsertScratch& s, const uint64_t* keys,
                             const float* values, const ScoreRule& rule, bool vec, cudaStream_t st,
                             bool collect_retry) {
  uint64_t blocks = (t.num_buckets * 8 + kThreads - 1) / kThreads;
  const uint64_t cap = static_cast<uint64_t>(sm_count()) * HKV_TILE_MIN_BLOCKS;
  const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
  ScoreRule r = rule;
  if (!rule.lfu()) {
    if (rule.policy != kCustomized) r.in = nullptr;
    if (rule.policy == kEpochLru) r.clock = rule.epoch_hi | (rule.clock & 0xFFFFFFFFull);
    r.policy = kCustomized;
  }
  cudaError_t e = rule.lfu() ? launch_chained(upsert_tile_kernel<true, kDual>, grid, kThreads, 0,
                                              st, t, s, values, r, vec, collect_retry)
                             : launch_chained(upsert_tile_kernel<false, kDual>, grid, kThreads, 0,
                                              st, t, s, values, r, vec, collect_retry);
  if (e != cudaSuccess) return e;
  UpsertExtra deferred;
  deferred.mark_want = kMarkDeferred;
  deferred.collect_retry = collect_retry;
  return launch_bucket_pass<kDual>(t, s, keys, values, rule, vec, st, deferred);
}

}  // namespace

cudaError_t clear_upsert_scratch(const UpsertScratch& s, uint64_t num_buckets, ScratchKind kind,
                                 cudaStream_t st) {
  const uint64_t mark_bytes = s.mark ? num_buckets : 0;
  (void)kind;
  return launch_chained(clear_scratch_kernel, grid_for(s.map_size / 2), kThreads, 0, st, s,
                        mark_bytes, false);
}

cudaError_t launch_upsert(const TableView& t, const UpsertScratch& s, uint64_t n,
                          const uint64_t* keys, const float* values, const ScoreRule& rule,
                          cudaStream_t st, const UpsertExtra& ex) {
  if (n == 0) return cudaSuccess;
  const bool vec = (t.dim % 4 == 0) && ((reinterpret_cast<uintptr_t>(values) & 15) == 0);
  const uint64_t* inc_in = rule.lfu() ? rule.in : nullptr;
  cudaError_t e = cudaSuccess;
  if (!t.dual) {
    const unsigned sg = grid_for((n + kStageKeysPerThread - 1) / kStageKeysPerThread);
    const bool sparse = sparse_batch(n, t.num_buckets);
    e = sparse ? launch_chained(stage_kernel<true>, sg, kThreads, 0, st, t, s, n, keys, inc_in)
               : launch_chained(stage_kernel<false>, sg, kThreads, 0, st, t, s, n, keys, inc_in);
    const bool plain = ex.update_resident && !ex.ev_keys;
    if (e == cudaSuccess && sparse && plain && HKV_UPSERT_SPARSE)
      return launch_tile_pass<false>(t, s, keys, values, rule, vec, st, false);
    if (e == cudaSuccess) e = launch_bucket_pass<false>(t, s, keys, values, rule, vec, st, ex);
    return e;
  }
  // Dual mode: de-duplicate; update residents and route absent keys; place
  // them bucket by bucket; route the displaced ones once more and place
  // them; count.
  dedup_insert_kernel<<<grid_for(n), kThreads, 0, st>>>(s, n, keys, inc_in, t.stats);
  e = launch_chained(dual_route_kernel, grid_for(n, HKV_ROUTE_MIN_BLOCKS), kThreads, 0, st, t, s,
                     n, keys, values, rule, vec);
  UpsertExtra first = ex;
  first.collect_retry = true;
  if (e == cudaSuccess)
    e = HKV_UPSERT_SPARSE ? launch_tile_pass<true>(t, s, keys, values, rule, vec, st, true)
                          : launch_bucket_pass<true>(t, s, keys, values, rule, vec, st, first);
  if (e == cudaSuccess)
    e = launch_chained(clear_scratch_kernel, grid_for(s.map_size / 2), kThreads, 0, st, s,
                       t.num_buckets, true);
  if (e == cudaSuccess)
    e = launch_chained(dual_retry_kernel, grid_for(n), kThreads, 0, st, t, s, keys, rule);
  if (e == cudaSuccess)
    e = HKV_UPSERT_SPARSE ? launch_tile_pass<true>(t, s, keys, values, rule, vec, st, false)
                          : launch_bucket_pass<true>(t, s, keys, values, rule, vec, st, ex);
  if (e != cudaSuccess) return e;
  dual_finish_kernel<<<1, 1, 0, st>>>(t, s);
  return cudaGetLastError();
}

cudaError_t launch_assign(const TableView& t, const UpsertScratch& s, uint64_t n,
                          const uint64_t* keys, const float* values, const ScoreRule& rule,
                          bool keep_scores, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const bool vec = (t.dim % 4 == 0) && ((reinterpret_cast<uintptr_t>(values) & 15) == 0);
  dedup_insert_kernel<<<grid_for(n), kThreads, 0, st>>>(s, n, keys, rule.lfu() ? rule.in : nullptr,
                                                         t.stats);
  if (t.dual)
    assign_kernel<true><<<grid_for(n, HKV_ASSIGN_MIN_BLOCKS), kThreads, 0, st>>>(
        t, s, n, keys, values, rule, keep_scores, vec);
  else
    assign_kernel<false><<<grid_for(n, HKV_ASSIGN_MIN_BLOCKS), kThreads, 0, st>>>(
        t, s, n, keys, values, rule, keep_scores, vec);
  return cudaGetLastError();
}

cudaError_t launch_erase(const TableView& t, uint64_t n, const uint64_t* keys, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  erase_kernel<<<grid_for(n * 8), kThreads, 0, st>>>(t, n, keys);
  return cudaGetLastError();
}

}  // namespace hkv
