// table.cu -- the C ABI (include/hkv.h): table construction, argument
// checking, scratch management and reader/updater/inserter ordering.
//
// Role ordering (HierarchicalKV §3.5 Table 4, §4.4): the paper mirrors three
// host atomic counters to the device with a one-thread kernel.  Here every
// call records a CUDA event on its stream and makes its stream wait, in host
// issue order, for the events of the earlier calls whose role conflicts with
// its own: readers wait for updaters and inserters, updaters for readers and
// inserters, inserters for everyone.  Compatible calls on different streams
// overlap; nothing spins on the device.
#include <cstddef>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "hkv.h"
#include "launch.h"

namespace {

enum class Role { kReader, kUpdater, kInserter };

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    int cur = -1;
    if (cudaGetDevice(&cur) == cudaSuccess && cur != dev) {
      prev = cur;
      cudaSetDevice(dev);
    }
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

// Events of the calls issued since the last inserter, by role.
class RoleTracker {
 public:
  cudaError_t before(Role r, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (last_inserter_) e = cudaStreamWaitEvent(s, last_inserter_, 0);
    if (e == cudaSuccess && r != Role::kUpdater)
      for (cudaEvent_t ev : updaters_)
        if ((e = cudaStreamWaitEvent(s, ev, 0)) != cudaSuccess) break;
    if (e == cudaSuccess && r != Role::kReader)
      for (cudaEvent_t ev : readers_)
        if ((e = cudaStreamWaitEvent(s, ev, 0)) != cudaSuccess) break;
    return e;
  }

  cudaError_t after(Role r, cudaStream_t s, cudaStream_t aux) {
    cudaEvent_t ev = nullptr;
    cudaError_t e = get(&ev);
    if (e == cudaSuccess) e = cudaEventRecord(ev, s);
    if (e != cudaSuccess) return e;
    if (r == Role::kInserter) {
      if (last_inserter_) free_.push_back(last_inserter_);
      for (cudaEvent_t x : readers_) free_.push_back(x);
      for (cudaEvent_t x : updaters_) free_.push_back(x);
      readers_.clear();
      updaters_.clear();
      last_inserter_ = ev;
      return cudaSuccess;
    }
    std::vector<cudaEvent_t>& list = (r == Role::kReader) ? readers_ : updaters_;
    list.push_back(ev);
    if (list.size() > 16) return join(list, aux);
    return cudaSuccess;
  }

  // Create k events ahead of use, so that later calls find them in the free
  // list.
  cudaError_t reserve(int k) {
    for (int i = 0; i < k; ++i) {
      cudaEvent_t ev = nullptr;
      cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
      free_.push_back(ev);
    }
    return cudaSuccess;
  }

  // Block the host until every recorded call has finished.
  cudaError_t wait_all() {
    cudaError_t e = cudaSuccess;
    if (last_inserter_) e = cudaEventSynchronize(last_inserter_);
    for (cudaEvent_t x : readers_)
      if (e == cudaSuccess) e = cudaEventSynchronize(x);
    for (cudaEvent_t x : updaters_)
      if (e == cudaSuccess) e = cudaEventSynchronize(x);
    return e;
  }

  void destroy() {
    if (last_inserter_) cudaEventDestroy(last_inserter_);
    for (cudaEvent_t x : readers_) cudaEventDestroy(x);
    for (cudaEvent_t x : updaters_) cudaEventDestroy(x);
    for (cudaEvent_t x : free_) cudaEventDestroy(x);
    last_inserter_ = nullptr;
    readers_.clear();
    updaters_.clear();
    free_.clear();
  }

 private:
  cudaError_t get(cudaEvent_t* ev) {
    if (!free_.empty()) {
      *ev = free_.back();
      free_.pop_back();
      return cudaSuccess;
    }
    return cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  }

  // Replace a long list by one event that completes after all of them.
  cudaError_t join(std::vector<cudaEvent_t>& list, cudaStream_t aux) {
    cudaError_t e = cudaSuccess;
    for (cudaEvent_t x : list)
      if ((e = cudaStreamWaitEvent(aux, x, 0)) != cudaSuccess) return e;
    cudaEvent_t j = nullptr;
    if ((e = get(&j)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(j, aux)) != cudaSuccess) return e;
    for (cudaEvent_t x : list) free_.push_back(x);
    list.assign(1, j);
    return cudaSuccess;
  }

  cudaEvent_t last_inserter_ = nullptr;
  std::vector<cudaEvent_t> readers_, updaters_, free_;
};

hkv_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return HKV_OK;
  if (e == cudaErrorMemoryAllocation) return HKV_ERR_OOM;
  return HKV_ERR_CUDA;
}

}  // namespace

struct hkv_table {
  hkv::TableView v{};
  int device = 0;
  uint32_t mode = 0;
  uint64_t capacity = 0;
  void* host_slab = nullptr;  // the tiered value slab as allocated (values_host: its device address)
  cudaMemPool_t host_pool = nullptr;  // its pool, for slabs above HKV_HOST_SLAB_MAPPED_MAX
  cudaMemPool_t pool = nullptr;
  cudaStream_t aux = nullptr;
  uint64_t step = 1;       // step counter / clock of the score policies
  uint32_t policy = 0;     // hkv::Policy
  uint32_t epoch = 0;
  RoleTracker roles;
  std::mutex mu;
};

namespace {

void release(hkv_table* t) {
  if (!t) return;
  DeviceGuard g(t->device);
  t->roles.wait_all();
  t->roles.destroy();
  if (t->aux) cudaStreamDestroy(t->aux);
  if (t->pool) cudaMemPoolDestroy(t->pool);
  cudaFree(t->v.digests);
  cudaFree(t->v.slots);
  cudaFree(t->v.values_hbm);
  cudaFree(t->v.summary);
  cudaFree(t->v.stats);
  // the table's work has finished (wait_all above): the slab is unused
  if (t->host_pool) {
    if (t->host_slab) cudaFree(t->host_slab);
    cudaMemPoolDestroy(t->host_pool);
  } else if (t->host_slab) {
    cudaFreeHost(t->host_slab);
  }
  delete t;
}

bool batch_ok(hkv_table* t, uint64_t n) { return t && n <= HKV_MAX_BATCH; }

// The tiered value slab, pinned host memory the device reads and writes at
// the same address.  Up to HKV_HOST_SLAB_MAPPED_MAX bytes it is
// cudaHostAllocMapped memory; a larger slab comes from a memory pool on the
// host NUMA node nearest the device (the host location where the system has
// no NUMA ids).  The two differ in how the device reaches random rows: mapped
// memory reads fastest while the process's mapped footprint stays small, and
// falls steeply past it; pool memory reads more slowly but holds its rate at
// any size (figures in include/hkv.h).
cudaError_t alloc_mapped_slab(size_t bytes, void** host, void** slab) {
  cudaError_t e = cudaHostAlloc(host, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer(slab, *host, 0);
  return e;
}

cudaError_t alloc_host_slab(int device, size_t bytes, cudaMemPool_t* pool, void** host,
                            void** slab) {
  *pool = nullptr;
  *host = nullptr;
  *slab = nullptr;
  if (bytes <= HKV_HOST_SLAB_MAPPED_MAX) return alloc_mapped_slab(bytes, host, slab);
  int numa = -1;
  if (cudaDeviceGetAttribute(&numa, cudaDevAttrHostNumaId, device) != cudaSuccess) {
    cudaGetLastError();
    numa = -1;
  }
  cudaMemPoolProps props{};
  props.allocType = cudaMemAllocationTypePinned;
  props.location.type = numa >= 0 ? cudaMemLocationTypeHostNuma : cudaMemLocationTypeHost;
  props.location.id = numa >= 0 ? numa : 0;
  cudaError_t e = cudaMemPoolCreate(pool, &props);
  if (e == cudaSuccess) {
    cudaMemAccessDesc access{};
    access.location.type = cudaMemLocationTypeDevice;
    access.location.id = device;
    access.flags = cudaMemAccessFlagsProtReadWrite;
    e = cudaMemPoolSetAccess(*pool, &access, 1);
  }
  if (e == cudaSuccess) e = cudaMallocFromPoolAsync(slab, bytes, *pool, cudaStreamLegacy);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cudaStreamLegacy);
  if (e == cudaSuccess) {
    *host = *slab;
    return e;
  }
  // no host memory pool here (or it could not hold the slab): mapped memory,
  // at its lower rate for random rows past HKV_HOST_SLAB_MAPPED_MAX
  if (*slab) cudaFree(*slab);
  if (*pool) cudaMemPoolDestroy(*pool);
  *pool = nullptr;
  *slab = nullptr;
  cudaGetLastError();
  return alloc_mapped_slab(bytes, host, slab);
}

bool clock_policy(const hkv_table* t) {
  return t->policy == hkv::kLru || t->policy == hkv::kEpochLru;
}

// Clock-driven policies take no caller scores.
bool scores_ok(const hkv_table* t, const uint64_t* scores) {
  return !(scores && clock_policy(t));
}

bool lfu_policy(const hkv_table* t) {
  return t->policy == hkv::kLfu || t->policy == hkv::kEpochLfu;
}

// The score rule of a call that writes scores, taken when the call is issued:
// it reads the clock and the epoch and advances the step counter where the
// policy says so (kCustomized without scores, the clock policies always).
hkv::ScoreRule take_rule(hkv_table* t, const uint64_t* scores) {
  hkv::ScoreRule r{};
  r.in = scores;
  r.clock = t->step;
  r.epoch_hi = static_cast<uint64_t>(t->epoch) << 32;
  r.policy = t->policy;
  if (clock_policy(t) || (t->policy == hkv::kCustomized && !scores)) ++t->step;
  return r;
}

// Order a call by role: wait for the conflicting calls, run `body`, record
// the call's role event.  The caller holds the table lock and has selected
// the device.
template <class F>
hkv_status run_ordered(hkv_table* t, Role r, cudaStream_t s, F&& body) {
  cudaError_t e = t->roles.before(r, s);
  if (e != cudaSuccess) return from_cuda(e);
  hkv_status st = body(s);
  e = t->roles.after(r, s, t->aux);
  if (st != HKV_OK) return st;
  return from_cuda(e);
}

// Common frame of a batched call: lock, select the device, order by role.
template <class F>
hkv_status run_call(hkv_table* t, Role r, void* stream, F&& body) {
  std::lock_guard<std::mutex> lk(t->mu);
  DeviceGuard g(t->device);
  return run_ordered(t, r, static_cast<cudaStream_t>(stream), body);
}

}  // namespace

namespace hkv {

int NoAllocAccess::run(hkv_table* t, uint64_t n, const uint64_t* keys, const float* values,
                       const uint64_t* scores, void* stream,
                       cudaError_t (*get_scratch)(int, void**)) {
  if (!batch_ok(t, n) || !scores_ok(t, scores)) return HKV_ERR_INVALID;
  if (n && (!keys || !values)) return HKV_ERR_INVALID;
  const ScratchKind kind = t->v.dual ? ScratchKind::kDualUpsert : ScratchKind::kSingleUpsert;
  if (upsert_scratch_bytes(n, t->v.num_buckets, kind, lfu_policy(t)) > HKV_NOALLOC_SCRATCH_BYTES)
    return HKV_ERR_INVALID;
  std::lock_guard<std::mutex> lk(t->mu);
  DeviceGuard g(t->device);
  void* mem = nullptr;
  cudaError_t e = get_scratch(t->device, &mem);
  if (e != cudaSuccess) return from_cuda(e);
  UpsertScratch sc{};
  if (n) {
    sc = carve_upsert_scratch(mem, n, t->v.num_buckets, kind, lfu_policy(t));
    // the carving itself must stay inside the array, whatever the formula
    // above says
    if (sc.bytes > HKV_NOALLOC_SCRATCH_BYTES) return HKV_ERR_INVALID;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return run_ordered(t, Role::kInserter, s, [&](cudaStream_t) -> hkv_status {
    const ScoreRule rule = take_rule(t, scores);
    if (n == 0) return HKV_OK;
    cudaError_t f = clear_upsert_scratch(sc, t->v.num_buckets, kind, s);
    if (f == cudaSuccess) f = launch_upsert(t->v, sc, n, keys, values, rule, s);
    return from_cuda(f);
  });
}

}  // namespace hkv

extern "C" {

hkv_status hkv_create(uint64_t capacity, uint32_t dim, uint32_t mode, uint64_t value_hbm_bytes,
                      int device, hkv_table** out) {
  if (!out) return HKV_ERR_INVALID;
  *out = nullptr;
  if (capacity == 0 || capacity % hkv::kSlots != 0 || dim == 0) return HKV_ERR_INVALID;
  if (mode & ~static_cast<uint32_t>(HKV_MODE_DUAL | HKV_MODE_TIERED | HKV_POLICY_MASK))
    return HKV_ERR_INVALID;
  if ((mode & HKV_POLICY_MASK) > HKV_POLICY_EPOCH_LFU) return HKV_ERR_INVALID;
  const uint64_t nb = capacity / hkv::kSlots;
  if (nb >= 0xFFFFFFFFull) return HKV_ERR_INVALID;
  const bool dual = (mode & HKV_MODE_DUAL) != 0;
  if (dual && nb < 2) return HKV_ERR_INVALID;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return HKV_ERR_INVALID;

  hkv_table* t = new (std::nothrow) hkv_table();
  if (!t) return HKV_ERR_OOM;
  t->device = device;
  t->mode = mode;
  t->policy = (mode & HKV_POLICY_MASK) >> 4;
  t->capacity = capacity;
  DeviceGuard g(device);

  uint64_t hbm_rows = capacity;
  if (mode & HKV_MODE_TIERED) {
    const uint64_t bucket_bytes = static_cast<uint64_t>(hkv::kSlots) * 4ull * dim;
    const uint64_t hb = value_hbm_bytes / bucket_bytes;
    hbm_rows = (hb < nb ? hb : nb) * hkv::kSlots;
  }
  hkv::TableView& v = t->v;
  v.num_buckets = nb;
  v.bucket_mask = (nb & (nb - 1)) == 0 ? nb - 1 : 0;
  v.dim = dim;
  v.dual = dual ? 1u : 0u;
  v.hbm_rows = hbm_rows;

  cudaError_t e = cudaMalloc(&v.digests, capacity);
  if (e == cudaSuccess) e = cudaMalloc(&v.slots, capacity * 16);
  if (e == cudaSuccess) e = cudaMalloc(&v.stats, sizeof(hkv::DeviceStats));
  if (e == cudaSuccess && hbm_rows) e = cudaMalloc(&v.values_hbm, hbm_rows * 4ull * dim);
  if (e == cudaSuccess && dual) e = cudaMalloc(&v.summary, nb * sizeof(hkv::BucketSummary));
  if (e == cudaSuccess && hbm_rows < capacity) {
    e = alloc_host_slab(device, (capacity - hbm_rows) * 4ull * dim, &t->host_pool, &t->host_slab,
                        reinterpret_cast<void**>(&v.values_host));
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&t->aux, cudaStreamNonBlocking);
  // role events for the first calls (a call reuses the events of the calls
  // an inserter has retired)
  if (e == cudaSuccess) e = t->roles.reserve(4);
  if (e == cudaSuccess) {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = device;
    e = cudaMemPoolCreate(&t->pool, &props);
    if (e == cudaSuccess) {
      uint64_t keep = ~0ull;  // keep scratch cached between calls
      e = cudaMemPoolSetAttribute(t->pool, cudaMemPoolAttrReleaseThreshold, &keep);
    }
  }
  if (e == cudaSuccess) e = hkv::launch_clear_table(v, t->aux);
  if (e == cudaSuccess) {
    // Grow the scratch pool once now, to what an insert_or_assign of
    // min(capacity, 2^20) keys needs, so the first batches do not pay for
    // the pool's first allocation (the pool keeps what it holds).
    const uint64_t n_warm = capacity < (1ull << 20) ? capacity : (1ull << 20);
    const hkv::ScratchKind kind = dual ? hkv::ScratchKind::kDualUpsert
                                       : hkv::ScratchKind::kSingleUpsert;
    void* warm = nullptr;
    e = cudaMallocFromPoolAsync(&warm, hkv::upsert_scratch_bytes(n_warm, nb, kind, lfu_policy(t)),
                                t->pool, t->aux);
    if (e == cudaSuccess) e = cudaFreeAsync(warm, t->aux);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(t->aux);
  if (e != cudaSuccess) {
    cudaGetLastError();
    release(t);
    return from_cuda(e);
  }
  *out = t;
  return HKV_OK;
}

hkv_status hkv_destroy(hkv_table* table) {
  if (!table) return HKV_OK;
  {
    std::lock_guard<std::mutex> lk(table->mu);
  }
  release(table);
  return HKV_OK;
}

hkv_status hkv_find(hkv_table* t, uint64_t n, const uint64_t* keys, float* values_out,
                    uint8_t* found_out, uint64_t* scores_out, void* stream) {
  if (!batch_ok(t, n)) return HKV_ERR_INVALID;
  if (n && (!keys || !values_out || !found_out)) return HKV_ERR_INVALID;
  return run_call(t, Role::kReader, stream, [&](cudaStream_t s) {
    return from_cuda(hkv::launch_find(t->v, n, keys, values_out, found_out, scores_out, s));
  });
}

namespace {

// Call-owned scratch from the table's stream-ordered memory pool; freed on
// the same stream after the kernels, so concurrent calls never share it.
hkv_status scratch_call(hkv_table* t, cudaStream_t s, uint64_t n, hkv::ScratchKind kind,
                        void** mem) {
  const size_t bytes = hkv::upsert_scratch_bytes(n, t->v.num_buckets, kind, lfu_policy(t));
  cudaError_t e = cudaMallocFromPoolAsync(mem, bytes, t->pool, s);
  return from_cuda(e);
}

}  // namespace

hkv_status hkv_insert_or_assign(hkv_table* t, uint64_t n, const uint64_t* keys, const float* values,
                                const uint64_t* scores, void* stream) {
  if (!batch_ok(t, n) || !scores_ok(t, scores)) return HKV_ERR_INVALID;
  if (n && (!keys || !values)) return HKV_ERR_INVALID;
  return run_call(t, Role::kInserter, stream, [&](cudaStream_t s) -> hkv_status {
    const hkv::ScoreRule rule = take_rule(t, scores);
    if (n == 0) return HKV_OK;
    const hkv::ScratchKind kind =
        t->v.dual ? hkv::ScratchKind::kDualUpsert : hkv::ScratchKind::kSingleUpsert;
    void* mem = nullptr;
    hkv_status st = scratch_call(t, s, n, kind, &mem);
    if (st != HKV_OK) return st;
    hkv::UpsertScratch sc = hkv::carve_upsert_scratch(mem, n, t->v.num_buckets, kind, lfu_policy(t));
    cudaError_t e = hkv::clear_upsert_scratch(sc, t->v.num_buckets, kind, s);
    if (e == cudaSuccess) e = hkv::launch_upsert(t->v, sc, n, keys, values, rule, s);
    cudaError_t f = cudaFreeAsync(mem, s);
    return from_cuda(e != cudaSuccess ? e : f);
  });
}

hkv_status hkv_contains(hkv_table* t, uint64_t n, const uint64_t* keys, uint8_t* found_out,
                        void* stream) {
  if (!batch_ok(t, n)) return HKV_ERR_INVALID;
  if (n && (!keys || !found_out)) return HKV_ERR_INVALID;
  return run_call(t, Role::kReader, stream, [&](cudaStream_t s) {
    return from_cuda(hkv::launch_contains(t->v, n, keys, found_out, s));
  });
}

hkv_status hkv_find_ptr(hkv_table* t, uint64_t n, const uint64_t* keys, float** values_ptr_out,
                        uint8_t* found_out, uint64_t* scores_out, void* stream) {
  if (!batch_ok(t, n)) return HKV_ERR_INVALID;
  if (n && (!keys || !values_ptr_out || !found_out)) return HKV_ERR_INVALID;
  return run_call(t, Role::kReader, stream, [&](cudaStream_t s) {
    return from_cuda(hkv::launch_find_ptr(t->v, n, keys, values_ptr_out, found_out, scores_out, s));
  });
}

namespace {

// Single-mode upsert variant with its own scratch (insert_and_evict,
// find_or_insert).
hkv_status upsert_variant(hkv_table* t, cudaStream_t s, uint64_t n, const uint64_t* keys,
                          const float* values, const uint64_t* scores,
                          const hkv::UpsertExtra& ex) {
  const hkv::ScoreRule rule = take_rule(t, scores);
  if (n == 0) return HKV_OK;
  void* mem = nullptr;
  hkv_status st = scratch_call(t, s, n, hkv::ScratchKind::kSingleUpsert, &mem);
  if (st != HKV_OK) return st;
  hkv::UpsertScratch sc = hkv::carve_upsert_scratch(mem, n, t->v.num_buckets,
                                                    hkv::ScratchKind::kSingleUpsert, lfu_policy(t));
  cudaError_t e =
      hkv::clear_upsert_scratch(sc, t->v.num_buckets, hkv::ScratchKind::kSingleUpsert, s);
  if (e == cudaSuccess) e = hkv::launch_upsert(t->v, sc, n, keys, values, rule, s, ex);
  cudaError_t f = cudaFreeAsync(mem, s);
  return from_cuda(e != cudaSuccess ? e : f);
}

}  // namespace

hkv_status hkv_insert_and_evict(hkv_table* t, uint64_t n, const uint64_t* keys,
                                const float* values, const uint64_t* scores,
                                uint64_t* evicted_keys_out, float* evicted_values_out,
                                uint64_t* evicted_scores_out, uint64_t* evicted_count_out,
                                void* stream) {
  if (!batch_ok(t, n) || t->v.dual || !scores_ok(t, scores)) return HKV_ERR_INVALID;
  if (n && (!keys || !values)) return HKV_ERR_INVALID;
  if (!evicted_keys_out || !evicted_count_out) return HKV_ERR_INVALID;
  return run_call(t, Role::kInserter, stream, [&](cudaStream_t s) -> hkv_status {
    cudaError_t e = cudaMemsetAsync(evicted_count_out, 0, sizeof(uint64_t), s);
    if (e != cudaSuccess) return from_cuda(e);
    hkv::UpsertExtra ex;
    ex.ev_keys = evicted_keys_out;
    ex.ev_values = evicted_values_out;
    ex.ev_scores = evicted_scores_out;
    ex.ev_count = reinterpret_cast<unsigned long long*>(evicted_count_out);
    return upsert_variant(t, s, n, keys, values, scores, ex);
  });
}

hkv_status hkv_find_or_insert(hkv_table* t, uint64_t n, const uint64_t* keys, float* values_inout,
                              const uint64_t* scores, uint8_t* found_out, void* stream) {
  if (!batch_ok(t, n) || t->v.dual || !scores_ok(t, scores)) return HKV_ERR_INVALID;
  if (n && (!keys || !values_inout || !found_out)) return HKV_ERR_INVALID;
  return run_call(t, Role::kInserter, stream, [&](cudaStream_t s) -> hkv_status {
    hkv::UpsertExtra ex;
    ex.update_resident = false;
    hkv_status st = upsert_variant(t, s, n, keys, values_inout, scores, ex);
    if (st != HKV_OK) return st;
    return from_cuda(hkv::launch_find(t->v, n, keys, values_inout, found_out, nullptr, s));
  });
}

hkv_status hkv_assign(hkv_table* t, uint64_t n, const uint64_t* keys, const float* values,
                      const uint64_t* scores, void* stream) {
  if (!batch_ok(t, n) || !scores_ok(t, scores)) return HKV_ERR_INVALID;
  if (n && (!keys || !values)) return HKV_ERR_INVALID;
  return run_call(t, Role::kUpdater, stream, [&](cudaStream_t s) -> hkv_status {
    // kCustomized without scores keeps the scores and the step counter
    const bool keep = t->policy == hkv::kCustomized && !scores;
    const hkv::ScoreRule rule = keep ? hkv::ScoreRule{} : take_rule(t, scores);
    if (n == 0) return HKV_OK;
    void* mem = nullptr;
    hkv_status st = scratch_call(t, s, n, hkv::ScratchKind::kAssign, &mem);
    if (st != HKV_OK) return st;
    hkv::UpsertScratch sc = hkv::carve_upsert_scratch(mem, n, t->v.num_buckets,
                                                      hkv::ScratchKind::kAssign, lfu_policy(t));
    cudaError_t e =
        hkv::clear_upsert_scratch(sc, t->v.num_buckets, hkv::ScratchKind::kAssign, s);
    if (e == cudaSuccess) e = hkv::launch_assign(t->v, sc, n, keys, values, rule, keep, s);
    cudaError_t f = cudaFreeAsync(mem, s);
    return from_cuda(e != cudaSuccess ? e : f);
  });
}

hkv_status hkv_erase(hkv_table* t, uint64_t n, const uint64_t* keys, void* stream) {
  if (!batch_ok(t, n)) return HKV_ERR_INVALID;
  if (n && !keys) return HKV_ERR_INVALID;
  return run_call(t, Role::kInserter, stream, [&](cudaStream_t s) {
    return from_cuda(hkv::launch_erase(t->v, n, keys, s));
  });
}

hkv_status hkv_size(hkv_table* t, uint64_t* size_host, void* stream) {
  if (!t || !size_host) return HKV_ERR_INVALID;
  unsigned long long v = 0;
  hkv_status st = run_call(t, Role::kReader, stream, [&](cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(&v, &t->v.stats->size, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return from_cuda(e);
  });
  if (st == HKV_OK) *size_host = v;
  return st;
}

hkv_status hkv_export(hkv_table* t, uint64_t slot_begin, uint64_t slot_end, uint64_t min_score,
                      uint64_t* keys_out, float* values_out, uint64_t* scores_out,
                      uint64_t* count_out, void* stream) {
  if (!t || !keys_out || !count_out) return HKV_ERR_INVALID;
  if (slot_end > t->capacity) slot_end = t->capacity;
  if (slot_begin > slot_end) slot_begin = slot_end;
  return run_call(t, Role::kReader, stream, [&](cudaStream_t s) {
    return from_cuda(hkv::launch_export(t->v, slot_begin, slot_end, min_score, keys_out, values_out,
                                        scores_out, count_out, s));
  });
}

static hkv_status read_stats(hkv_table* t, hkv::DeviceStats* out) {
  std::lock_guard<std::mutex> lk(t->mu);
  DeviceGuard g(t->device);
  cudaError_t e = t->roles.wait_all();
  if (e == cudaSuccess) e = cudaMemcpy(out, t->v.stats, sizeof(*out), cudaMemcpyDeviceToHost);
  return from_cuda(e);
}

hkv_status hkv_get_error_counts(hkv_table* t, uint64_t* reserved_keys_host, uint64_t* timeouts_host) {
  if (!t || !reserved_keys_host || !timeouts_host) return HKV_ERR_INVALID;
  hkv::DeviceStats s{};
  hkv_status st = read_stats(t, &s);
  if (st != HKV_OK) return st;
  *reserved_keys_host = s.reserved;
  *timeouts_host = s.timeouts;
  if (s.timeouts) return HKV_ERR_TIMEOUT;
  if (s.reserved) return HKV_ERR_RESERVED_KEY;
  return HKV_OK;
}

hkv_status hkv_get_op_counts(hkv_table* t, hkv_op_counts* out) {
  if (!t || !out) return HKV_ERR_INVALID;
  hkv::DeviceStats s{};
  hkv_status st = read_stats(t, &s);
  if (st != HKV_OK) return st;
  out->updated = s.updated;
  out->admitted = s.admitted;
  out->evicted = s.evicted;
  out->rejected = s.rejected;
  out->erased = s.erased;
  return HKV_OK;
}

hkv_status hkv_reset_op_counts(hkv_table* t) {
  if (!t) return HKV_ERR_INVALID;
  std::lock_guard<std::mutex> lk(t->mu);
  DeviceGuard g(t->device);
  cudaError_t e = t->roles.wait_all();
  // updated .. erased are contiguous in DeviceStats
  if (e == cudaSuccess)
    e = cudaMemset(&t->v.stats->updated, 0,
                   offsetof(hkv::DeviceStats, size) - offsetof(hkv::DeviceStats, updated));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return from_cuda(e);
}

hkv_status hkv_set_epoch(hkv_table* t, uint32_t epoch) {
  if (!t) return HKV_ERR_INVALID;
  std::lock_guard<std::mutex> lk(t->mu);
  t->epoch = epoch;
  return HKV_OK;
}

hkv_status hkv_get_info(hkv_table* t, hkv_info* out) {
  if (!t || !out) return HKV_ERR_INVALID;
  out->capacity = t->capacity;
  out->num_buckets = t->v.num_buckets;
  out->hbm_value_rows = t->v.hbm_rows;
  out->dim = t->v.dim;
  out->mode = t->mode;
  out->device = t->device;
  out->hbm_values_addr = reinterpret_cast<uint64_t>(t->v.values_hbm);
  out->host_values_addr = reinterpret_cast<uint64_t>(t->v.values_host);
  return HKV_OK;
}

const char* hkv_status_string(hkv_status s) {
  switch (s) {
    case HKV_OK: return "ok";
    case HKV_ERR_INVALID: return "invalid argument";
    case HKV_ERR_OOM: return "out of memory";
    case HKV_ERR_CUDA: return "CUDA error";
    case HKV_ERR_RESERVED_KEY: return "reserved keys were skipped";
    case HKV_ERR_TIMEOUT: return "keys abandoned after a bounded wait";
    default: return "unknown status";
  }
}

}  // extern "C"
