// launch.h -- host-side launchers of the library's kernels (internal).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "hkv.h"

namespace hkv {

// Scratch of one insert_or_assign / assign call (device memory, call-owned).
struct UpsertScratch {
  uint64_t* map_keys;   // map_size entries, EMPTY-initialised: the single-mode
                        // stage, or the dedup map of dual mode and assign
  uint32_t* map_idx;    // last batch index + 1 per entry, 0-initialised
  uint32_t map_size;    // power of two, >= 2n
  int32_t area_shift;   // single mode, power-of-two bucket count B: log2(S/B)
                        // (negative: B > S); kNoShift otherwise
  uint32_t* cursor;     // small counters (0-initialised)
  uint8_t* mark;        // single mode, sparse batches: one byte per table bucket,
                        // 1 = holds batch keys (null for dense batches)
  uint8_t* absent;      // dual mode: per dedup-map entry, 1 = the key was absent
                        // before the call (written for every entry in use)
  uint32_t* retry;      // dual mode: absent keys displaced in the first pass
  uint64_t* inc;        // LFU policies: summed increments per map entry,
                        // 0-initialised (null under the other policies)
  // The stage read by the bucket kernel: one run of positions per bucket.
  // Single mode stages straight into the dedup arrays (stage_keys = map_keys,
  // stage_idx = map_idx, stage_inc = inc, stage_bkt = null); dual mode routes
  // each absent key to one of its two buckets and stages it in a second set
  // of arrays, with the chosen bucket in stage_bkt.
  uint64_t* stage_keys;
  uint32_t* stage_idx;
  uint32_t* stage_bkt;
  uint64_t* stage_inc;
  size_t bytes;         // bytes of the allocation the carving uses
};

// What a call needs scratch for.
enum class ScratchKind { kSingleUpsert, kDualUpsert, kAssign };

// Bytes of scratch a call of n keys needs, and the carving of one allocation
// into the UpsertScratch arrays.
// `lfu`: the table's policy sums increments (kLfu, kEpochLfu).
size_t upsert_scratch_bytes(uint64_t n, uint64_t num_buckets, ScratchKind kind, bool lfu);
UpsertScratch carve_upsert_scratch(void* base, uint64_t n, uint64_t num_buckets, ScratchKind kind,
                                   bool lfu);
// Enqueue the clears the scratch needs before use.
cudaError_t clear_upsert_scratch(const UpsertScratch& s, uint64_t num_buckets, ScratchKind kind,
                                 cudaStream_t st);

cudaError_t launch_find(const TableView& t, uint64_t n, const uint64_t* keys, float* values_out,
                        uint8_t* found_out, uint64_t* scores_out, cudaStream_t st);

cudaError_t launch_contains(const TableView& t, uint64_t n, const uint64_t* keys,
                            uint8_t* found_out, cudaStream_t st);

cudaError_t launch_find_ptr(const TableView& t, uint64_t n, const uint64_t* keys, float** ptrs_out,
                            uint8_t* found_out, uint64_t* scores_out, cudaStream_t st);

// Variants of the single-mode upsert: find_or_insert leaves resident keys
// untouched; insert_and_evict reports the pre-call residents it displaces.
struct UpsertExtra {
  bool update_resident = true;
  bool collect_retry = false;  // dual mode, first bucket pass: list displaced keys
  uint64_t* ev_keys = nullptr;
  float* ev_values = nullptr;
  uint64_t* ev_scores = nullptr;
  unsigned long long* ev_count = nullptr;
  uint8_t mark_want = 0;  // process only buckets whose mark equals this (0: any mark)
};

cudaError_t launch_upsert(const TableView& t, const UpsertScratch& s, uint64_t n,
                          const uint64_t* keys, const float* values, const ScoreRule& rule,
                          cudaStream_t st, const UpsertExtra& ex = UpsertExtra());

// keep_scores: write values only (kCustomized without caller scores).
cudaError_t launch_assign(const TableView& t, const UpsertScratch& s, uint64_t n,
                          const uint64_t* keys, const float* values, const ScoreRule& rule,
                          bool keep_scores, cudaStream_t st);

cudaError_t launch_erase(const TableView& t, uint64_t n, const uint64_t* keys, cudaStream_t st);

cudaError_t launch_export(const TableView& t, uint64_t slot_begin, uint64_t slot_end,
                          uint64_t min_score, uint64_t* keys_out, float* values_out,
                          uint64_t* scores_out, uint64_t* count_out, cudaStream_t st);

cudaError_t launch_clear_table(const TableView& t, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int sm_count();

// Launch `kernel` on `st` with programmatic stream serialization, so it can be
// scheduled while the stream's previous kernel drains (the kernel must call
// pdl_wait() before touching memory that kernel writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                           cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Runs insert_or_assign with caller-provided working memory (used by
// hkv_insert_or_assign_noalloc); get_scratch(device, &ptr) yields it.
struct NoAllocAccess {
  static int run(hkv_table* t, uint64_t n, const uint64_t* keys, const float* values,
                 const uint64_t* scores, void* stream, cudaError_t (*get_scratch)(int, void**));
};

}  // namespace hkv
