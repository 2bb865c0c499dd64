// common.cuh -- table layout, hashing and small device helpers shared by the
// kernels of the library.
//
// Layout in HBM (HierarchicalKV §3.2 Figure 4, §3.6, §4.2): structure of
// arrays over B buckets of 128 slots; slot j of bucket b is row r = b*128 + j.
//   digests[B*128]  uint8   one 128-byte line per bucket, 0 = free slot
//   slots[B*128]    {uint64 key, uint64 score}; EMPTY_KEY marks a free slot
//                   (key and score share one 32-byte sector, so a find hit
//                   reads its score with the key confirm)
//   values          float32 rows of `dim`; rows < hbm_rows in HBM, the rest in
//                   mapped pinned host memory (tiered mode)
// No per-entry pointer is stored: a value row is found from (bucket, slot).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace hkv {

constexpr int kSlots = 128;
constexpr uint64_t kEmptyKey = 0xFFFFFFFFFFFFFFFFull;
constexpr uint64_t kReservedLo = 0xFFFFFFFFFFFFFFF0ull;
constexpr uint64_t kDualSeed = 0x9E3779B97F4A7C15ull;
constexpr uint32_t kNone = 0xFFFFFFFFu;

// Device-resident counters of one table.  Fields are updated with atomics.
struct DeviceStats {
  unsigned long long reserved;   // reserved keys skipped
  unsigned long long timeouts;   // bounded waits that ran out (dual-mode locks, bucket copies)
  unsigned long long updated;
  unsigned long long admitted;
  unsigned long long evicted;
  unsigned long long rejected;
  unsigned long long erased;
  unsigned long long size;       // resident entries
  unsigned long long fills;      // dual mode: entries placed in free slots by the current call
};

// Dual mode: per bucket, its occupancy and the lowest score in it, as of the
// last upsert pass that processed the bucket (erase keeps the count exact;
// assign may leave min_score below the true minimum).  Upserts use them only
// to choose between a key's two buckets, never to decide admission.
struct BucketSummary {
  unsigned long long min_score;
  unsigned int count;
  unsigned int pad;
};

// Everything a kernel needs to address the table; passed by value.
struct TableView {
  uint8_t* digests;
  uint64_t* slots;        // 2 words per slot: key, score
  float* values_hbm;
  float* values_host;     // device pointer of the mapped host slab, or null
  uint64_t hbm_rows;      // rows below this index live in values_hbm
  uint64_t num_buckets;
  uint64_t bucket_mask;   // num_buckets - 1 when a power of two, else 0
  uint32_t dim;
  uint32_t dual;
  BucketSummary* summary; // dual mode: one per bucket (routing hints)
  DeviceStats* stats;
};

// Score policies (HKV §3.3 "Scoring policies"; Table 8 names kCustomized,
// kLru, kLfu, kEpochLru, kEpochLfu).  Values are the policy field of the
// table mode shifted down by 4.
enum Policy : uint32_t { kCustomized = 0, kLru = 1, kLfu = 2, kEpochLru = 3, kEpochLfu = 4 };

// How one call computes the scores it writes; passed by value.
struct ScoreRule {
  const uint64_t* in;  // caller scores (kCustomized) or increments (LFU kinds); may be null
  uint64_t clock;      // the call's step counter value
  uint64_t epoch_hi;   // epoch << 32
  uint32_t policy;
  __host__ __device__ bool lfu() const { return policy == kLfu || policy == kEpochLfu; }
};

__device__ __forceinline__ uint64_t add_sat64(uint64_t a, uint64_t b) {
  const uint64_t c = a + b;
  return c < a ? ~0ull : c;
}

// Score written for batch entry e.  `inc` is the entry's summed increment
// (LFU kinds); `old` the resident entry's score when `resident`.
__device__ __forceinline__ uint64_t policy_score(const ScoreRule& r, uint64_t e, uint64_t inc,
                                                 bool resident, uint64_t old) {
  switch (r.policy) {
    case kLru: return r.clock;
    case kEpochLru: return r.epoch_hi | (r.clock & 0xFFFFFFFFull);
    case kLfu: return resident ? add_sat64(old, inc) : inc;
    case kEpochLfu: {
      const uint64_t f = add_sat64(resident ? (old & 0xFFFFFFFFull) : 0ull, inc);
      return r.epoch_hi | (f > 0xFFFFFFFFull ? 0xFFFFFFFFull : f);
    }
    default: return r.in ? r.in[e] : r.clock;
  }
}

// Saturating atomic add of a 64-bit counter (lock-free: a failed CAS means
// another thread's add went through).
__device__ __forceinline__ void atomic_add_sat64(uint64_t* p, uint64_t v) {
  unsigned long long* q = reinterpret_cast<unsigned long long*>(p);
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(q);
  while (true) {
    const unsigned long long nv = add_sat64(old, v);
    const unsigned long long seen = atomicCAS(q, old, nv);
    if (seen == old) return;
    old = seen;
  }
}

// H(k): the 64-bit MurmurHash3 finalizer (HKV §3.1 names a Murmur3-derived
// hash; the finalizer is the published 64-bit mixing step).
__host__ __device__ __forceinline__ uint64_t hash64(uint64_t h) {
  h ^= h >> 33;
  h *= 0xff51afd7ed558ccdull;
  h ^= h >> 33;
  h *= 0xc4ceb9fe1a85ec53ull;
  h ^= h >> 33;
  return h;
}

__host__ __device__ __forceinline__ uint64_t bucket_of_hash(const TableView& t, uint64_t h) {
  return t.bucket_mask ? (h & t.bucket_mask) : (h % t.num_buckets);
}

// Second candidate bucket for dual mode (HKV §3.4, "two candidate buckets via
// independent hashes"); never equal to the first.
__host__ __device__ __forceinline__ uint64_t bucket2_of(const TableView& t, uint64_t key,
                                                        uint64_t b1) {
  uint64_t b2 = bucket_of_hash(t, hash64(key ^ kDualSeed));
  if (b2 == b1) b2 = (b1 + 1 == t.num_buckets) ? 0 : b1 + 1;
  return b2;
}

// 8-bit digest from bits 32..39 of the hash (HKV §3.2).  Byte 0 is kept for
// free slots, so a digest of 0 is stored as 1.
__host__ __device__ __forceinline__ uint32_t digest_of_hash(uint64_t h) {
  uint32_t d = static_cast<uint32_t>(h >> 32) & 0xFFu;
  return d ? d : 1u;
}

__device__ __forceinline__ bool is_reserved(uint64_t k) { return k >= kReservedLo; }

__device__ __forceinline__ uint64_t* key_at(const TableView& t, uint64_t row) {
  return t.slots + 2 * row;
}
__device__ __forceinline__ uint64_t* score_at(const TableView& t, uint64_t row) {
  return t.slots + 2 * row + 1;
}

__device__ __forceinline__ float* row_ptr(const TableView& t, uint64_t row) {
  return row < t.hbm_rows ? t.values_hbm + row * t.dim
                          : t.values_host + (row - t.hbm_rows) * t.dim;
}

// ---------------------------------------------------------------------------
// Memory access helpers (inline PTX for the cache hints).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// Hint: bring the 128-byte line holding p (global memory) into L2; no result.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Streaming read: no L1 allocation (value rows are touched once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// Streaming store (evict-first), for output rows and written value rows.
// A value row in the host slab of a tiered table is read with a plain
// (L1-cached) load: on a GB300 over NVLink-C2C, SM reads of host memory
// through the read-only path, with or without L1 allocation, reach half of
// the link's rate (105.6 GB/s for random 256-byte rows), plain loads the
// whole of it (211.1 GB/s).  HBM rows keep ld_stream_v4.
__device__ __forceinline__ uint4 ld_host_row_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint64_t ld_nc_u64(const uint64_t* p) {
  uint64_t r;
  asm volatile("ld.global.nc.u64 %0, [%1];" : "=l"(r) : "l"(p));
  return r;
}
// Read-only 16-byte load of a slot's (key, score) pair.
__device__ __forceinline__ ulonglong2 ld_nc_pair(const uint64_t* p) {
  ulonglong2 r;
  asm volatile("ld.global.nc.v2.u64 {%0,%1}, [%2];" : "=l"(r.x), "=l"(r.y) : "l"(p));
  return r;
}

// L2-coherent loads (bypass L1) for data other blocks may have written in
// the same kernel.
__device__ __forceinline__ uint64_t ld_cg_u64(const uint64_t* p) {
  uint64_t r;
  asm volatile("ld.global.cg.u64 %0, [%1];" : "=l"(r) : "l"(p) : "memory");
  return r;
}

__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p) : "memory");
  return r;
}

// Exact per-byte equality mask: bit i of the result is set when byte i of
// `w` equals byte i of `pat` (i = 0..3).  Branch-free SWAR test for a zero
// byte in w ^ pat.
__device__ __forceinline__ uint32_t byte_eq_mask4(uint32_t w, uint32_t pat) {
  uint32_t x = w ^ pat;
  uint32_t y = ((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x;  // high bit set iff byte != 0
  uint32_t z = ~y & 0x80808080u;                      // high bit set iff byte == 0
  return ((z >> 7) & 1u) | ((z >> 14) & 2u) | ((z >> 21) & 4u) | ((z >> 28) & 8u);
}

// Zero-byte flags of x: bit 8i+7 is set for every zero byte i of x, and may
// also be set for a byte directly above a zero byte (borrow).  A word with no
// zero byte gives 0.  Used on (digest word ^ pattern): a flagged byte is a
// candidate slot whose key is then compared, so an extra flag costs one key
// comparison and never a wrong result.
__device__ __forceinline__ uint32_t zero_byte_flags(uint32_t x) {
  return (x - 0x01010101u) & ~x & 0x80808080u;
}

// Candidate mask of the four bytes of w against the replicated digest `pat`:
// bit i set when byte i may equal the digest (every equal byte is set; see
// zero_byte_flags for the rare extra).  The multiply gathers the flag bits
// 7, 15, 23, 31 into bits 28..31 without carries.
__device__ __forceinline__ uint32_t byte_match4(uint32_t w, uint32_t pat) {
  return (zero_byte_flags(w ^ pat) * 0x00204081u) >> 28;
}

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// ---------------------------------------------------------------------------
// Bulk copies into shared memory by the copy engine (TMA, non-tensor form)
// with completion on a shared-memory mbarrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t arrivals) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(arrivals)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One arrival that also announces `bytes` of copies completing on `bar`.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_load_smem(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before
// later bulk copies into shared memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// One bounded probe of the barrier's phase `parity`; true once it completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Programmatic dependent launch (sm_90+).  A kernel launched with
// launch_chained() may become resident while the previous kernel of its
// stream is still running; pdl_wait() blocks until that kernel has completed
// and its memory writes are visible, and is a no-op for a normal launch.
// pdl_trigger() lets the next chained kernel be scheduled early.  Every
// kernel here calls pdl_wait() before it touches global memory, so chaining
// only hides the launch latency and the ramp between kernels.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Warp-aggregated atomic add of a per-lane contribution (any lane set).
__device__ __forceinline__ void warp_add(unsigned long long* p, unsigned long long v) {
  unsigned long long s = v;
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if (lane_id() == 0 && s) atomicAdd(p, s);
}

// Copy one value row of `dim` floats with the 8 lanes of a tile: lane `sub`
// (0..7) moves 16-byte chunks sub, sub+8, ...  `vec` selects the 16-byte path
// (both rows 16-byte aligned and dim % 4 == 0); otherwise 4-byte words.
__device__ __forceinline__ void tile_copy_row(float* dst, const float* src, uint32_t dim,
                                              unsigned sub, bool vec, bool stream_store,
                                              bool src_host = false) {
  if (vec) {
    const uint32_t chunks = dim >> 2;
    for (uint32_t c = sub; c < chunks; c += 8) {
      uint4 v = src_host ? ld_host_row_v4(src + 4 * c) : ld_stream_v4(src + 4 * c);
      if (stream_store) st_stream_v4(dst + 4 * c, v);
      else *reinterpret_cast<uint4*>(dst + 4 * c) = v;
    }
  } else {
    for (uint32_t c = sub; c < dim; c += 8) dst[c] = src[c];
  }
}

// Copy R value rows with the 8 lanes of a tile, all R loads of a chunk in
// flight before the stores (rows with ok[r] == false are skipped).
template <int R>
__device__ __forceinline__ void tile_copy_rows(float* const (&dst)[R], const float* const (&src)[R],
                                               const bool (&ok)[R], uint32_t dim, unsigned sub,
                                               bool vec) {
  if (vec) {
    const uint32_t chunks = dim >> 2;
    for (uint32_t c = sub; c < chunks; c += 8) {
      uint4 v[R];
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (ok[r]) v[r] = ld_stream_v4(src[r] + 4 * c);
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (ok[r]) st_stream_v4(dst[r] + 4 * c, v[r]);
    }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (ok[r])
        for (uint32_t c = sub; c < dim; c += 8) dst[r][c] = src[r][c];
  }
}

// Probe bucket b for `key` with the 8 lanes of a tile (HKV Algorithm 1):
// lane `sub` loads 16 bytes of the 128-byte digest line, byte-compares them
// with the key's digest (`pat` = digest * 0x01010101) and confirms each match
// with an 8-byte key load.  Returns the slot, or -1; uniform across the tile.
// kNC selects read-only loads, legal only when no thread of the running
// kernel writes keys or digests.
template <bool kNC>
__device__ __forceinline__ int tile_probe(const TableView& t, uint64_t b, uint64_t key, uint32_t pat,
                                          unsigned sub, unsigned tmask) {
  const uint8_t* dp = t.digests + b * kSlots + sub * 16;
  uint4 dg;
  if (kNC) dg = ld_nc_v4(dp);
  else dg = ld_cg_v4(dp);
  uint32_t m = byte_match4(dg.x, pat) | (byte_match4(dg.y, pat) << 4) |
               (byte_match4(dg.z, pat) << 8) | (byte_match4(dg.w, pat) << 12);
  int hit = -1;
  const uint64_t* kb = t.slots + 2 * (b * kSlots + sub * 16);
  while (m) {
    const int bit = __ffs(m) - 1;
    m &= m - 1;
    const uint64_t k = kNC ? ld_nc_u64(kb + 2 * bit) : ld_cg_u64(kb + 2 * bit);
    if (k == key) {
      hit = static_cast<int>(sub * 16 + bit);
      break;
    }
  }
  const unsigned bal = __ballot_sync(tmask, hit >= 0) & tmask;
  if (!bal) return -1;
  return __shfl_sync(tmask, hit, __ffs(bal) - 1);
}

}  // namespace hkv
