// export.cu -- reader kernel for export_batch_if (HierarchicalKV §4.1) with the
// predicate score >= min_score, and the table initialisation kernel.
#include "launch.h"

namespace hkv {
namespace {

constexpr int kThreads = 256;

// One 8-lane tile per slot: lane 0 tests the slot, the tile copies the row.
__global__ void __launch_bounds__(kThreads) export_kernel(TableView t, uint64_t slot_begin,
                                                          uint64_t slot_end, uint64_t min_score,
                                                          uint64_t* keys_out, float* values_out,
                                                          uint64_t* scores_out,
                                                          unsigned long long* count, bool vec) {
  const unsigned lane = lane_id();
  const unsigned sub = lane & 7u;
  const unsigned tmask = 0xFFu << (lane & 24u);
  const uint64_t tiles = (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 3;
  for (uint64_t row = slot_begin + ((static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3);
       row < slot_end; row += tiles) {
    const ulonglong2 ks = *reinterpret_cast<const ulonglong2*>(key_at(t, row));
    const uint64_t k = ks.x;
    const bool take = k < kReservedLo && ks.y >= min_score;
    if (!take) continue;  // tile-uniform
    unsigned long long pos = 0;
    if (sub == 0) {
      pos = atomicAdd(count, 1ull);
      keys_out[pos] = k;
      if (scores_out) scores_out[pos] = ks.y;
    }
    pos = __shfl_sync(tmask, pos, lane & 24u);
    if (values_out)
      tile_copy_row(values_out + pos * t.dim, row_ptr(t, row), t.dim, sub, vec, true,
                    row >= t.hbm_rows);
  }
}

}  // namespace

cudaError_t launch_export(const TableView& t, uint64_t slot_begin, uint64_t slot_end,
                          uint64_t min_score, uint64_t* keys_out, float* values_out,
                          uint64_t* scores_out, uint64_t* count_out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(count_out, 0, sizeof(uint64_t), st);
  if (e != cudaSuccess || slot_end <= slot_begin) return e;
  uint64_t blocks = ((slot_end - slot_begin) * 8 + kThreads - 1) / kThreads;
  const uint64_t cap = static_cast<uint64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  const bool vec = (t.dim % 4 == 0) && ((reinterpret_cast<uintptr_t>(values_out) & 15) == 0);
  export_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, st>>>(
      t, slot_begin, slot_end, min_score, keys_out, values_out, scores_out,
      reinterpret_cast<unsigned long long*>(count_out), vec);
  return cudaGetLastError();
}

cudaError_t launch_clear_table(const TableView& t, cudaStream_t st) {
  const uint64_t slots = t.num_buckets * kSlots;
  // every slot free: key = EMPTY (all ones); a free slot's score is never read
  cudaError_t e = cudaMemsetAsync(t.slots, 0xFF, slots * 16, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(t.digests, 0, slots, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(t.stats, 0, sizeof(DeviceStats), st);
  if (e == cudaSuccess && t.summary)
    e = cudaMemsetAsync(t.summary, 0, t.num_buckets * sizeof(BucketSummary), st);
  return e;
}

}  // namespace hkv
