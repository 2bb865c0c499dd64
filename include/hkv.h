/*
 * hkv.h -- C ABI of a cache-semantic GPU key-value hash table (GB300, sm_103a).
 *
 * The operations follow "HierarchicalKV: A GPU Hash Table with Cache
 * Semantics for Continuous Online Embedding Storage" (arXiv 2603.17168v1),
 * cited below as HKV.  Keys are uint64, scores uint64, values float32 rows of
 * `dim` elements.  A table of capacity C has B = C / 128 buckets of 128 slots
 * (HKV §3.2).  Every key lives in one bucket b1 = H(k) mod B (single mode) or
 * in one of two buckets b1, b2 (dual mode, HKV §3.4), where H is the 64-bit
 * MurmurHash3 finalizer and b2 = H(k ^ 0x9E3779B97F4A7C15) mod B, moved to
 * (b1 + 1) mod B when it equals b1.
 *
 * Reserved keys: 0xFFFFFFFFFFFFFFF0 .. 0xFFFFFFFFFFFFFFFF are sentinels of
 * the table.  An input key in that range is skipped by every call (find
 * reports it not found) and counted; see hkv_get_error_counts.
 *
 * Ranks: admission and victim choice compare ranks, tuples compared
 * lexicographically as unsigned integers, so equal scores never leave a
 * choice open.  Single mode ranks an entry by (score, new, key), where `new`
 * is 1 for an entry placed by the current call and 0 for one that was
 * resident before it: an incoming key of equal score outranks an older
 * entry (HKV Algorithm 2 admits on score >= the bucket minimum), and the key
 * decides between entries of equal score and age.  Dual mode ranks by
 * (score, key) (HKV Algorithm 3 admits on score > the minimum).
 *
 * Batches: duplicate keys inside one insert_or_assign or assign batch
 * collapse to their last occurrence.  Inside one insert_or_assign call the
 * keys already resident are updated first, then the absent keys are placed;
 * in single mode the result is therefore a pure function of the table and the
 * batch (bucket b ends up with the 128 highest-ranked of its residents and of
 * the absent keys hashed to it).  In dual mode each absent key is routed to
 * one of its buckets by Algorithm 3's rules applied to per-bucket summaries
 * (occupancy and lowest score as of the bucket's last upsert pass), each
 * bucket then keeps the highest-ranked of its entries and its routed keys,
 * and the keys displaced by that pass are routed once more with the updated
 * summaries; which keys win near the margin depends on that processing
 * order, but a key that ends up absent always lost to a full bucket all of
 * whose entries outrank it.
 *
 * Memory: all pointer arguments except the `*_host` ones are device pointers
 * (or pointers the device can dereference: mapped or managed host memory).
 * The caller owns them; they must stay valid until the stream reaches the
 * call.  The table owns its storage.  Row-major value buffers hold n * dim
 * float32; a 16-byte aligned base and dim % 4 == 0 select the vector path.
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream).  Every batched call is asynchronous: it validates its arguments,
 * enqueues kernels and returns.  Argument errors are returned at once and
 * enqueue nothing.
 *
 * Score policies (HKV §3.3 "Scoring policies"; §5 Exp #3c, Table 8 names
 * kLru, kLfu, kEpochLru, kEpochLfu and kCustomized without defining their
 * update rules).  A table is created with one policy (mode bits 4-7), which
 * decides the score a call writes for a key (insert_or_assign,
 * insert_and_evict, find_or_insert, assign):
 *   HKV_POLICY_CUSTOMIZED  the caller's score; scores == NULL: the table's
 *                          step counter, which starts at 1 and grows by 1
 *                          per NULL-score call (assign with NULL keeps the
 *                          scores).
 *   HKV_POLICY_LRU         the table clock: the step counter, which under this
 *                          policy grows by 1 per score-writing call.  scores
 *                          must be NULL (else HKV_ERR_INVALID).
 *   HKV_POLICY_EPOCH_LRU   (epoch << 32) | (clock mod 2^32); scores NULL.
 *   HKV_POLICY_LFU         a frequency: scores are per-occurrence increments
 *                          (NULL: 1 each).  The increments of all occurrences
 *                          of a key in one call add up; a resident key gets
 *                          old score + sum, an absent key competes with sum;
 *                          sums saturate at 2^64 - 1.
 *   HKV_POLICY_EPOCH_LFU   (epoch << 32) | f, where f is the LFU rule applied
 *                          to the low 32 bits of the old score, saturating at
 *                          2^32 - 1 (the count survives epoch changes).
 * The epoch is a 32-bit value of the table (0 at creation, hkv_set_epoch),
 * read when a call is issued.  find_or_insert never changes a resident key.
 *
 * Roles (HKV §3.5, Table 4): find, size and export are readers; assign is an
 * updater; insert_or_assign and erase are inserters.  Calls of conflicting
 * roles issued on different streams are ordered by CUDA events in host issue
 * order: readers overlap readers, updaters overlap updaters, an inserter
 * overlaps nothing.  Calls on one table may come from several host threads.
 */
#ifndef HKV_H_
#define HKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hkv_table hkv_table; /* opaque, owned by the library */
typedef int hkv_status;

enum {
  HKV_MODE_SINGLE = 0, /* one candidate bucket per key (HKV §3.2) */
  HKV_MODE_DUAL = 1,   /* two candidate buckets, score-based choice (HKV §3.4) */
  HKV_MODE_TIERED = 2  /* flag: values above the HBM budget live in mapped host memory (HKV §3.6) */
};

/* Score policy, ORed into hkv_create's mode (see "Score policies"). */
enum {
  HKV_POLICY_CUSTOMIZED = 0x00,
  HKV_POLICY_LRU = 0x10,
  HKV_POLICY_LFU = 0x20,
  HKV_POLICY_EPOCH_LRU = 0x30,
  HKV_POLICY_EPOCH_LFU = 0x40,
  HKV_POLICY_MASK = 0xF0
};

enum {
  HKV_OK = 0,
  HKV_ERR_INVALID = -1,      /* bad argument; nothing was enqueued */
  HKV_ERR_OOM = -2,          /* device or pinned host allocation failed */
  HKV_ERR_CUDA = -3,         /* a CUDA runtime call failed */
  HKV_ERR_RESERVED_KEY = -4, /* hkv_get_error_counts: reserved keys were skipped */
  HKV_ERR_TIMEOUT = -5       /* hkv_get_error_counts: keys were abandoned after a bounded wait */
};

#define HKV_SLOTS_PER_BUCKET 128
#define HKV_RESERVED_KEY_LO 0xFFFFFFFFFFFFFFF0ull
#define HKV_MAX_BATCH 0x7FFFFFFFull /* largest n accepted by a batched call */

/* Create a table.  HKV §3.1-§3.2 (bucketed layout), §3.6/§4.2 (tiered).
 *  capacity        slots; a positive multiple of 128 (B = capacity / 128;
 *                  B >= 2 in dual mode).
 *  dim             float32 elements per value row, >= 1.
 *  mode            HKV_MODE_SINGLE or HKV_MODE_DUAL, optionally | HKV_MODE_TIERED,
 *                  | one HKV_POLICY_* (default HKV_POLICY_CUSTOMIZED).
 *  value_hbm_bytes with TIERED: HBM budget for value rows.  Rows of whole
 *                  buckets 0 .. R-1 (R = floor(budget / (128 * 4 * dim)) * 128)
 *                  live in HBM, the rest in pinned host memory the device
 *                  reads and writes directly (see HKV_HOST_SLAB_MAPPED_MAX).
 *                  Ignored without TIERED (all rows in HBM).
 *  device          CUDA device ordinal the table lives on.
 *  out             receives the table handle.
 * Keys, digests and scores always live in HBM.  The table starts empty.
 * Synchronous.  Errors: INVALID, OOM, CUDA (nothing is leaked). */
hkv_status hkv_create(uint64_t capacity, uint32_t dim, uint32_t mode, uint64_t value_hbm_bytes,
                      int device, hkv_table** out);

/* The host slab of a tiered table (the rows above the HBM budget) is
 * cudaHostAllocMapped memory when it holds at most this many bytes, and
 * pinned memory from a memory pool on the device's nearest host NUMA node
 * when it is larger.  Measured on a GB300 (Grace host, 64 KiB pages, NVLink-
 * C2C), random 256-byte row reads from the GPU: mapped memory reads at 183-208
 * GB/s while the process's mapped footprint is at most 16 GiB and at 7-12
 * GB/s beyond 24 GiB; pool memory reads at 26-28 GB/s from 8 GiB to 32 GiB.
 * Where the system offers no host memory pool, a larger slab is mapped
 * memory too.  Either way a row's device address is fixed for the table's
 * life. */
#define HKV_HOST_SLAB_MAPPED_MAX (16ull << 30)

/* Wait for all work on the table and free it.  NULL is a no-op. */
hkv_status hkv_destroy(hkv_table* table);

/* Reader.  HKV Algorithm 1 (digest-accelerated find; two buckets in dual
 * mode).  For each i < n: if keys[i] is resident, found_out[i] = 1,
 * values_out[i*dim .. +dim) = its value row and, when scores_out != NULL,
 * scores_out[i] = its score; otherwise found_out[i] = 0 and the value and
 * score outputs of row i are left untouched.  The table is not modified. */
hkv_status hkv_find(hkv_table* table, uint64_t n, const uint64_t* keys, float* values_out,
                    uint8_t* found_out, uint64_t* scores_out, void* stream);

/* Inserter.  HKV Algorithm 2 (single mode) / Algorithm 3 (dual mode):
 * upsert with bucket-local admission and eviction.  A resident key gets the
 * new value and score unconditionally.  An absent key takes a free slot of
 * its bucket (dual mode: the less occupied candidate, ties to b1); when the
 * bucket is full (dual: both full) it replaces the lowest-ranked entry of the
 * bucket (dual: of the candidate whose lowest rank is lower) if it ranks
 * higher than that entry, else it is rejected.  Dual mode applies these rules
 * batch-wise as described under "Batches".
 *  scores  per-key scores (LFU policies: increments) or NULL; the score an
 *          entry receives follows the table's policy (see "Score
 *          policies"); under HKV_POLICY_CUSTOMIZED, NULL gives every key of
 *          the call the step counter.
 * Outcome totals accumulate in hkv_get_op_counts. */
hkv_status hkv_insert_or_assign(hkv_table* table, uint64_t n, const uint64_t* keys,
                                const float* values, const uint64_t* scores, void* stream);

/* Inserter, single-bucket tables only (HKV §7: the dual-bucket mode covers
 * insert_or_assign and find).  HKV §4.1 insert_and_evict: the same update as
 * hkv_insert_or_assign, and every entry that was resident before the call
 * and is displaced by it is written to evicted_keys_out / evicted_values_out
 * / evicted_scores_out (values and scores may be NULL) as it was when
 * displaced (a key updated by this call and then displaced carries its new
 * value and score), at consecutive positions in unspecified order;
 * *evicted_count_out (device) receives their number.  Outputs need room for
 * n entries.  Dual-mode tables return HKV_ERR_INVALID. */
hkv_status hkv_insert_and_evict(hkv_table* table, uint64_t n, const uint64_t* keys,
                                const float* values, const uint64_t* scores,
                                uint64_t* evicted_keys_out, float* evicted_values_out,
                                uint64_t* evicted_scores_out, uint64_t* evicted_count_out,
                                void* stream);

/* Inserter, single-bucket tables only.  HKV §4.1 find_or_insert (lookup
 * with insertion for cold start): absent keys are inserted with their row of
 * values_inout and the score the table's policy gives them under
 * HKV Algorithm 2; resident keys are not modified.  Afterwards, for each i:
 * when keys[i] is resident, found_out[i] = 1 and row i of values_inout holds
 * its stored value; otherwise (admission rejected it) found_out[i] = 0 and
 * row i is left unchanged.  Dual-mode tables return HKV_ERR_INVALID. */
hkv_status hkv_find_or_insert(hkv_table* table, uint64_t n, const uint64_t* keys,
                              float* values_inout, const uint64_t* scores, uint8_t* found_out,
                              void* stream);

/* Reader.  HKV §3.5 contains: found_out[i] = 1 iff keys[i] is resident.
 * Reads digests and keys only, no value row. */
hkv_status hkv_contains(hkv_table* table, uint64_t n, const uint64_t* keys, uint8_t* found_out,
                        void* stream);

/* Reader.  HKV §5.2-§5.3 find*: like hkv_find, but instead of copying a
 * resident key's value row, values_ptr_out[i] receives the device address of
 * the row inside the table (HBM, or the mapped host slab in tiered mode);
 * NULL on a miss.  The addresses stay valid until the next inserter call on
 * the table (insert_or_assign, insert_and_evict, find_or_insert, erase). */
hkv_status hkv_find_ptr(hkv_table* table, uint64_t n, const uint64_t* keys, float** values_ptr_out,
                        uint8_t* found_out, uint64_t* scores_out, void* stream);

/* Updater.  HKV §3.5: overwrites the value and the score of resident keys
 * in place; absent keys are ignored; nothing is inserted, evicted or moved.
 * The score follows the table's policy (see "Score policies"); under
 * HKV_POLICY_CUSTOMIZED with scores == NULL the scores are left as they are
 * and the step counter does not move. */
hkv_status hkv_assign(hkv_table* table, uint64_t n, const uint64_t* keys, const float* values,
                      const uint64_t* scores, void* stream);

/* Inserter.  HKV §3.5: removes each resident key; its slot becomes free. */
hkv_status hkv_erase(hkv_table* table, uint64_t n, const uint64_t* keys, void* stream);

/* Reader.  HKV §3.5 (size): number of resident entries, written to the host
 * variable *size_host.  Synchronises with `stream`. */
hkv_status hkv_size(hkv_table* table, uint64_t* size_host, void* stream);

/* Reader.  HKV §4.1 export_batch_if with the predicate score >= min_score
 * (the score-threshold dump of the DynamicEmb API page).  Scans slots
 * [slot_begin, slot_end) (slot = bucket * 128 + position, end clamped to the
 * capacity) and writes each matching entry to keys_out / values_out /
 * scores_out (values_out and scores_out may be NULL) at consecutive
 * positions in unspecified order.  *count_out (device) receives the number
 * written; outputs must have room for slot_end - slot_begin entries. */
hkv_status hkv_export(hkv_table* table, uint64_t slot_begin, uint64_t slot_end, uint64_t min_score,
                      uint64_t* keys_out, float* values_out, uint64_t* scores_out,
                      uint64_t* count_out, void* stream);

/* Cumulative counts since creation, read synchronously (waits for the
 * table's outstanding work).  reserved_keys: input keys skipped because they
 * were reserved sentinels.  timeouts: bounded device-side waits that ran out
 * (none in the default build; the pipelined measurement build counts a bucket
 * copy that did not arrive in time, then loads that bucket directly).
 * Returns HKV_ERR_TIMEOUT when timeouts > 0, else HKV_ERR_RESERVED_KEY when
 * reserved_keys > 0, else HKV_OK; the counts are written in every case. */
hkv_status hkv_get_error_counts(hkv_table* table, uint64_t* reserved_keys_host,
                                uint64_t* timeouts_host);

/* Cumulative outcome totals of insert_or_assign / assign / erase since
 * creation (or the last reset), read synchronously.  For insert_or_assign:
 * updated = resident keys overwritten; admitted = absent keys resident after
 * their call; rejected = absent keys not resident after their call; evicted =
 * keys resident before a call that it displaced.  assign adds to updated,
 * erase to erased. */
typedef struct hkv_op_counts {
  uint64_t updated, admitted, evicted, rejected, erased;
} hkv_op_counts;
hkv_status hkv_get_op_counts(hkv_table* table, hkv_op_counts* out_host);
hkv_status hkv_reset_op_counts(hkv_table* table);

/* Static facts about a table.  Value row r (r = bucket * 128 + slot) lives
 * at device address hbm_values_addr + r * dim * 4 when r < hbm_value_rows,
 * else at host_values_addr + (r - hbm_value_rows) * dim * 4 (the mapped host
 * slab of a tiered table; 0 when there is none), so a row address returned
 * by hkv_find_ptr maps back to its row and bucket. */
typedef struct hkv_info {
  uint64_t capacity, num_buckets, hbm_value_rows;
  uint32_t dim, mode;
  int device;
  uint64_t hbm_values_addr, host_values_addr;
} hkv_info;
hkv_status hkv_get_info(hkv_table* table, hkv_info* out_host);

/* Set the table's 32-bit epoch (HKV §3.3 epoch-aware scoring; see "Score
 * policies").  Calls issued afterwards use it; calls already issued keep the
 * epoch they were issued with.  Any policy accepts it; only the EPOCH
 * policies read it.  Errors: INVALID (NULL table). */
hkv_status hkv_set_epoch(hkv_table* table, uint32_t epoch);

/* insert_or_assign for callers that cannot let the library allocate.
 *
 * The paper has no counterpart: this is a deployment variant of
 * hkv_insert_or_assign with the same arguments and the same results.  That
 * call takes its per-call working memory from a stream-ordered pool; this
 * one uses a fixed array of HKV_NOALLOC_SCRATCH_BYTES compiled into the
 * library, for callers whose device memory is already handed out (e.g. to a
 * framework's caching allocator), who keep a fixed memory budget, or whose
 * serving loop must never enter cudaMalloc/cudaFree (which can synchronise
 * the device).  It calls no allocation routine.
 *  - Limit: the batch's working memory must fit the array, i.e.
 *      a(8M) + a(4M) + 256 + a(B) bytes in single mode and
 *      2 a(8M) + 3 a(4M) + a(M) + 256 + a(4n) + a(B) bytes in dual mode,
 *    plus a(8M) under the LFU policies (2 a(8M) in dual mode), with M the
 *    smallest power of two >= max(64, 2n), B the bucket count and a(x) = x
 *    rounded up to a multiple of 256.  Larger batches return HKV_ERR_INVALID and enqueue
 *    nothing (split them, or use hkv_insert_or_assign).  In single mode that
 *    is up to 2^20 keys per call for tables of at most 2^23 - 256 buckets,
 *    and up to 2^19 keys under the LFU policies for tables of at most
 *    12 * 2^20 - 256 buckets; a call of 2^20 + 1 keys (2^19 + 1 under LFU)
 *    is refused on any table.
 *  - Sharing: every call on every table of a device uses the same array and
 *    clears it before use.  Calls whose kernels overlap on the GPU (on
 *    different streams, from any table) race on it and corrupt each other's
 *    results: keep such calls on one stream, or order them with events.
 *  - Ordering on the table: as for hkv_insert_or_assign (an inserter), using
 *    CUDA events the table created with it, so later calls on other streams,
 *    hkv_get_op_counts and hkv_destroy wait for this one.
 *  - Set-up: the first call on a device (made with any table of that device)
 *    looks up the array's device address with cudaGetSymbolAddress and keeps
 *    it for the life of the process; make that first call before any stream
 *    capture.  cudaDeviceReset on that device destroys its tables and may
 *    move the array; do not call this function on that device afterwards. */
#define HKV_NOALLOC_SCRATCH_BYTES (32ull << 20)
hkv_status hkv_insert_or_assign_noalloc(hkv_table* table, uint64_t n, const uint64_t* keys,
                                        const float* values, const uint64_t* scores, void* stream);

/* Human-readable name of a status code (static storage). */
const char* hkv_status_string(hkv_status status);

#ifdef __cplusplus
}
#endif

#endif /* HKV_H_ */
