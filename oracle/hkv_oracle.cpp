// hkv_oracle.cpp -- reference model of the cache-semantic hash table.
//
// TEST INFRASTRUCTURE ONLY.  This file is the correctness oracle that the
// CUDA library is checked against.  Only the test suite, the smoke check in
// __graft_entry__.py and the cpu_baseline leg of bench.py may load it.  The
// product path (hash_table_cache_gb300/) never links, imports or calls it,
// and this file shares no header, helper or constant with that path.
//
// It is deliberately plain: single-threaded, one std::vector per bucket,
// linear scans, no blocking or reordering beyond what the method states.
//
// Source of the method: "HierarchicalKV: A GPU Hash Table with Cache
// Semantics for Continuous Online Embedding Storage" (arXiv 2603.17168v1),
// cited below as HKV with its section / algorithm / proposition numbers.
//
// Readings taken where the paper is silent or inconsistent (each one is also
// listed in the design notes of the repository):
//  R1 hash: the paper names it only as a Murmur3 derivative; we use the 64-bit
//     MurmurHash3 finalizer (Appleby, public domain) as H(k).
//  R2 bucket b1 = H(k) mod B.  Dual mode: b2 = H(k ^ 0x9E3779B97F4A7C15) mod B,
//     and b2 = (b1 + 1) mod B when the two coincide.
//  R3 the 16 keys 0xFFFFFFFFFFFFFFF0..0xFFFFFFFFFFFFFFFF are reserved
//     sentinels (EMPTY and LOCKED live there); inputs carrying them are
//     skipped and counted.
//  R4 ranks.  HKV Algorithm 2 admits an absent key into a full bucket when
//     its score is >= the bucket's minimum; Algorithm 3 only when it is >.
//     Single mode ranks an entry by (score, new, key): `new` marks entries
//     placed in the bucket by the current call, so an incoming key beats an
//     older entry of equal score (Algorithm 2's >=), and the key decides
//     between entries of equal score and age.  The victim is the entry of
//     lowest rank.  Dual mode ranks by (score, key) (Algorithm 3's >, with
//     the key as the deterministic tie-break).  Both orders are total, so a
//     bucket's result never depends on the order of the keys in a batch.
//  R5 duplicate keys inside one batch collapse to their last occurrence.
//  R6 within one batch, the unique keys are applied in this serial order:
//     first every key that is already resident (in-place update, HKV
//     Algorithm 2's found branch), then every absent key (the empty-slot /
//     eviction / rejection branches), each group in batch order.  The paper
//     runs a batch in parallel and fixes no order; this is one valid serial
//     order, and when no update lowers a rank it gives the same table as any
//     other serial order.
//  R7 scores == NULL: every key of the call gets the table's step counter,
//     which starts at 1 and increments once per insert_or_assign call (the
//     STEP strategy of the DynamicEmb API page).
//  R8 find of an absent key leaves the caller's value and score outputs
//     untouched and reports found = 0.
//  R9 slot positions are not modelled: a bucket is an unordered set of at
//     most 128 entries; nothing observable depends on positions.
//  R10 score policies.  HKV §3.3 ("Scoring policies") and §5 Exp #3c
//     (Table 8) name five ScoreFunctor variants -- kLru, kLfu, kEpochLru,
//     kEpochLfu, kCustomized -- but give none of their update rules.  A table
//     is created with one of them, and the score a call writes for a key is:
//       kCustomized  the caller's score; without scores the step counter (R7).
//       kLru         the table clock.  The clock is the step counter, which
//                    under this policy advances once per call that writes
//                    scores (insert_or_assign, insert_and_evict,
//                    find_or_insert, assign).  Callers pass no scores.
//       kEpochLru    (epoch << 32) | (clock mod 2^32), clock as for kLru.
//       kLfu         a frequency.  The caller's scores are per-occurrence
//                    increments (1 each without scores); the increments of
//                    all occurrences of a key in one call add up (R5 then
//                    keeps the last occurrence's value).  A resident key
//                    gets old + sum, an absent key competes with sum;
//                    additions saturate at 2^64 - 1.
//       kEpochLfu    (epoch << 32) | f with f the kLfu rule applied to the
//                    low 32 bits of the old score, saturating at 2^32 - 1:
//                    the count survives an epoch change, the epoch field
//                    records the epoch of the last write.
//     The epoch is a 32-bit value set on the table (0 at creation) and read
//     when the call is issued.  find_or_insert leaves resident keys as they
//     are under every policy (HKV §4.1).  With the epoch advanced once per
//     call, both epoch policies rank like kLru across calls, which is the
//     equality Table 8 shows for the three columns.
//  The 8-bit digest only accelerates lookups and never changes a result
//  (HKV §3.2), so the oracle does not model it.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <unordered_set>
#include <vector>

namespace {

constexpr int kSlots = 128;                                 // HKV §3.2: S = 128
constexpr uint64_t kReservedLo = 0xFFFFFFFFFFFFFFF0ull;    // R3
constexpr uint64_t kDualSeed = 0x9E3779B97F4A7C15ull;      // R2

// MurmurHash3 64-bit finalizer (R1).
uint64_t murmur_fmix64(uint64_t h) {
    h ^= h >> 33;
    h *= 0xff51afd7ed558ccdull;
    h ^= h >> 33;
    h *= 0xc4ceb9fe1a85ec53ull;
    h ^= h >> 33;
    return h;
}

bool is_reserved(uint64_t k) { return k >= kReservedLo; }

// R4: rank comparison.
bool rank_less(uint64_t s1, uint64_t k1, uint64_t s2, uint64_t k2) {
    return s1 < s2 || (s1 == s2 && k1 < k2);
}

// R4, single mode: (score, new, key).
bool rank_less_new(uint64_t s1, int n1, uint64_t k1, uint64_t s2, int n2, uint64_t k2) {
    if (s1 != s2) return s1 < s2;
    if (n1 != n2) return n1 < n2;
    return k1 < k2;
}

struct Bucket {
    // Parallel arrays, unordered, size <= kSlots (R9).
    std::vector<uint64_t> keys;
    std::vector<uint64_t> scores;
    std::vector<float> values;   // keys.size() * dim
    std::vector<uint8_t> fresh;  // 1 = placed by the current call (R4)

    int find(uint64_t k) const {
        for (size_t i = 0; i < keys.size(); ++i)
            if (keys[i] == k) return static_cast<int>(i);
        return -1;
    }
    int size() const { return static_cast<int>(keys.size()); }
    // Position of the minimum-rank entry (the arg-min over the bucket's
    // scores of HKV Algorithms 2 and 3, ties per R4: with_new selects the
    // single-mode rank).  Bucket must be non-empty.
    int argmin_rank(bool with_new) const {
        int m = 0;
        for (int i = 1; i < size(); ++i) {
            const bool lt = with_new
                ? rank_less_new(scores[i], fresh[i], keys[i], scores[m], fresh[m], keys[m])
                : rank_less(scores[i], keys[i], scores[m], keys[m]);
            if (lt) m = i;
        }
        return m;
    }
};

struct Counts {
    uint64_t updated = 0, admitted = 0, evicted = 0, rejected = 0, reserved = 0, filtered = 0,
             erased = 0;
};

// R10: score policies.
enum Policy : uint32_t { kCustomized = 0, kLru = 1, kLfu = 2, kEpochLru = 3, kEpochLfu = 4 };

uint64_t add_sat64(uint64_t a, uint64_t b) { return a + b < a ? ~0ull : a + b; }

struct Table {
    uint64_t num_buckets;
    uint32_t dim;
    bool dual;
    uint32_t policy = kCustomized;                       // R10
    uint32_t epoch = 0;                                  // R10
    uint64_t step = 1;                                   // R7
    std::unordered_map<uint64_t, Bucket> buckets;       // created on first use
    std::vector<uint64_t> placed_in;                    // buckets holding new entries (R4)
    bool filtered = false;
    std::unordered_set<uint64_t> filter;                // single mode only

    uint64_t bucket1(uint64_t k) const { return murmur_fmix64(k) % num_buckets; }
    uint64_t bucket2(uint64_t k) const {
        uint64_t b1 = bucket1(k);
        uint64_t b2 = murmur_fmix64(k ^ kDualSeed) % num_buckets;
        if (b2 == b1) b2 = (b1 + 1) % num_buckets;
        return b2;
    }
    bool simulated(uint64_t b) const { return !filtered || filter.count(b) != 0; }
    Bucket& at(uint64_t b) { return buckets[b]; }

    // Locate a resident key: returns bucket index and position, or false.
    bool locate(uint64_t k, uint64_t* b_out, int* pos_out) {
        uint64_t b1 = bucket1(k);
        auto it = buckets.find(b1);
        if (it != buckets.end()) {
            int p = it->second.find(k);
            if (p >= 0) { *b_out = b1; *pos_out = p; return true; }
        }
        if (dual) {
            uint64_t b2 = bucket2(k);
            auto it2 = buckets.find(b2);
            if (it2 != buckets.end()) {
                int p = it2->second.find(k);
                if (p >= 0) { *b_out = b2; *pos_out = p; return true; }
            }
        }
        return false;
    }

    void write_entry(Bucket& bk, int pos, uint64_t k, uint64_t s, const float* v) {
        bk.keys[pos] = k;
        bk.scores[pos] = s;
        std::memcpy(&bk.values[static_cast<size_t>(pos) * dim], v, sizeof(float) * dim);
    }
    void append_entry(Bucket& bk, uint64_t k, uint64_t s, const float* v) {
        bk.keys.push_back(k);
        bk.scores.push_back(s);
        bk.fresh.push_back(0);
        bk.values.insert(bk.values.end(), v, v + dim);
    }
    void remove_entry(Bucket& bk, int pos) {
        int last = bk.size() - 1;
        if (pos != last) {
            write_entry(bk, pos, bk.keys[last], bk.scores[last],
                        &bk.values[static_cast<size_t>(last) * dim]);
            bk.fresh[pos] = bk.fresh[last];
        }
        bk.keys.pop_back();
        bk.scores.pop_back();
        bk.fresh.pop_back();
        bk.values.resize(static_cast<size_t>(last) * dim);
    }

    // Outcome of one absent key (HKV Algorithm 2 / 3 return values).
    enum Outcome { kInserted, kEvicted, kRejected };

    // A displaced entry as it was at the moment of its displacement.
    struct Victim { uint64_t key = 0, score = 0; std::vector<float> value; };

    void take_victim(const Bucket& bk, int m, Victim* out) {
        out->key = bk.keys[m];
        out->score = bk.scores[m];
        out->value.assign(bk.values.begin() + static_cast<long>(m) * dim,
                          bk.values.begin() + static_cast<long>(m + 1) * dim);
    }

    // HKV Algorithm 2, branches after the (failed) lookup, on bucket b.
    // On kEvicted, *victim receives the displaced entry.
    Outcome insert_single(uint64_t b, uint64_t k, uint64_t s, const float* v, Victim* victim) {
        Bucket& bk = at(b);
        if (bk.size() < kSlots) {                 // first empty slot exists
            append_entry(bk, k, s, v);
            mark_new(b, bk, bk.size() - 1);
            return kInserted;
        }
        int m = bk.argmin_rank(true);             // bucket full: eviction path
        // admission control: the incoming key is new to the bucket (R4)
        if (rank_less_new(s, 1, k, bk.scores[m], bk.fresh[m], bk.keys[m]))
            return kRejected;
        take_victim(bk, m, victim);
        write_entry(bk, m, k, s, v);              // replace the minimum
        mark_new(b, bk, m);
        return kEvicted;
    }

    void mark_new(uint64_t b, Bucket& bk, int pos) {
        bk.fresh[pos] = 1;
        placed_in.push_back(b);
    }

    // HKV Algorithm 3 (score-based dual-bucket upsert), for an absent key.
    Outcome insert_dual(uint64_t k, uint64_t s, const float* v, Victim* victim) {
        uint64_t b1 = bucket1(k), b2 = bucket2(k);
        Bucket& x = at(b1);
        Bucket& y = at(b2);
        if (x.size() < kSlots || y.size() < kSlots) {        // phase D1
            Bucket& target = (y.size() < x.size()) ? y : x;  // less occupied, tie -> b1
            append_entry(target, k, s, v);
            return kInserted;
        }
        int m1 = x.argmin_rank(false), m2 = y.argmin_rank(false);  // phase D2
        bool pick2 = rank_less(y.scores[m2], y.keys[m2], x.scores[m1], x.keys[m1]);
        Bucket& bs = pick2 ? y : x;
        int m = pick2 ? m2 : m1;
        if (!rank_less(bs.scores[m], bs.keys[m], s, k))      // admission control
            return kRejected;
        take_victim(bs, m, victim);
        write_entry(bs, m, k, s, v);
        return kEvicted;
    }

    // Collapse a batch to the last occurrence of each valid key (R5) and
    // return the surviving indices in batch order.
    std::vector<uint64_t> last_occurrences(uint64_t n, const uint64_t* keys, Counts& c) {
        std::unordered_map<uint64_t, uint64_t> last;
        last.reserve(static_cast<size_t>(n) * 2 + 1);
        for (uint64_t i = 0; i < n; ++i) {
            if (is_reserved(keys[i])) { ++c.reserved; continue; }
            last[keys[i]] = i;
        }
        std::vector<uint64_t> idx;
        idx.reserve(last.size());
        for (uint64_t i = 0; i < n; ++i)
            if (!is_reserved(keys[i]) && last[keys[i]] == i) idx.push_back(i);
        return idx;
    }

    bool skip_for_filter(uint64_t k, Counts& c) {
        if (filtered && !simulated(bucket1(k))) { ++c.filtered; return true; }
        return false;
    }

    // The score rule of one call (R7, R10).  `scores` are the caller's
    // scores (kCustomized) or increments (kLfu, kEpochLfu).
    struct ScoreRule {
        uint32_t policy = kCustomized;
        uint64_t clock = 0;      // the call's step / clock value
        uint64_t epoch_hi = 0;   // epoch << 32
        const uint64_t* scores = nullptr;
        std::unordered_map<uint64_t, uint64_t> inc;   // kLfu kinds: summed increments

        bool lfu() const { return policy == kLfu || policy == kEpochLfu; }
        // Score of a key written by this call; `resident` with its old score.
        uint64_t score(uint64_t i, uint64_t k, bool resident, uint64_t old) const {
            switch (policy) {
                case kLru: return clock;
                case kEpochLru: return epoch_hi | (clock & 0xFFFFFFFFull);
                case kLfu: {
                    const uint64_t d = inc.at(k);
                    return resident ? add_sat64(old, d) : d;
                }
                case kEpochLfu: {
                    uint64_t f = add_sat64(resident ? (old & 0xFFFFFFFFull) : 0, inc.at(k));
                    if (f > 0xFFFFFFFFull) f = 0xFFFFFFFFull;
                    return epoch_hi | f;
                }
                default: return scores ? scores[i] : clock;
            }
        }
    };

    // Opens a call that writes scores: takes its clock and advances the step
    // counter where the policy says so (R7, R10).
    ScoreRule score_rule(uint64_t n, const uint64_t* keys, const uint64_t* scores) {
        ScoreRule r;
        r.policy = policy;
        r.clock = step;
        r.epoch_hi = static_cast<uint64_t>(epoch) << 32;
        r.scores = scores;
        if (policy == kLru || policy == kEpochLru || (policy == kCustomized && !scores)) ++step;
        if (r.lfu()) {
            for (uint64_t i = 0; i < n; ++i) {
                if (is_reserved(keys[i])) continue;
                uint64_t& d = r.inc[keys[i]];
                d = add_sat64(d, scores ? scores[i] : 1);
            }
        }
        return r;
    }

    // update_resident = false gives find_or_insert's insertion step: resident
    // keys are left as they are.  evicted_out, when given, receives every
    // entry that was resident before the call and is displaced by it
    // (insert_and_evict), as it was when displaced.
    Counts insert_or_assign(uint64_t n, const uint64_t* keys, const float* values,
                            const uint64_t* scores, bool update_resident = true,
                            std::vector<Victim>* evicted_out = nullptr) {
        Counts c;
        const ScoreRule rule = score_rule(n, keys, scores);
        std::vector<uint64_t> idx = last_occurrences(n, keys, c);
        std::vector<uint64_t> absent;
        for (uint64_t i : idx) {                  // R6: resident keys first
            uint64_t k = keys[i];
            if (skip_for_filter(k, c)) continue;
            uint64_t b; int p;
            if (locate(k, &b, &p)) {              // HKV Algorithm 2, found branch
                if (update_resident) {
                    const uint64_t s = rule.score(i, k, true, at(b).scores[p]);
                    write_entry(at(b), p, k, s, values + i * dim);
                    ++c.updated;
                }
            } else {
                absent.push_back(i);
            }
        }
        // Then the absent keys, batch order.  The counts are batch-level and
        // independent of the serial order: an absent key that is admitted and
        // displaced again within the same call counts as rejected, and
        // "evicted" counts only keys that were resident before the call.
        std::unordered_set<uint64_t> admitted;
        for (uint64_t i : absent) {
            uint64_t k = keys[i];
            const uint64_t s = rule.score(i, k, false, 0);
            Victim victim;
            Outcome o = dual ? insert_dual(k, s, values + i * dim, &victim)
                             : insert_single(bucket1(k), k, s, values + i * dim, &victim);
            if (o == kRejected) continue;
            admitted.insert(k);
            if (o == kEvicted) {
                if (admitted.erase(victim.key) == 0) {
                    ++c.evicted;
                    if (evicted_out) evicted_out->push_back(std::move(victim));
                }
            }
        }
        for (uint64_t b : placed_in) {            // R4: "new" lasts one call
            Bucket& bk = at(b);
            std::fill(bk.fresh.begin(), bk.fresh.end(), 0);
        }
        placed_in.clear();
        c.admitted = admitted.size();
        c.rejected = absent.size() - admitted.size();
        return c;
    }

    Counts assign(uint64_t n, const uint64_t* keys, const float* values, const uint64_t* scores) {
        Counts c;
        // kCustomized without scores keeps the scores (and the step counter);
        // every other case writes the policy's score (R10).
        const bool keep = policy == kCustomized && !scores;
        const ScoreRule rule = keep ? ScoreRule() : score_rule(n, keys, scores);
        std::vector<uint64_t> idx = last_occurrences(n, keys, c);
        for (uint64_t i : idx) {
            uint64_t k = keys[i];
            if (skip_for_filter(k, c)) continue;
            uint64_t b; int p;
            if (!locate(k, &b, &p)) continue;     // updater: absent keys are a no-op
            Bucket& bk = at(b);
            std::memcpy(&bk.values[static_cast<size_t>(p) * dim], values + i * dim,
                        sizeof(float) * dim);
            if (!keep) bk.scores[p] = rule.score(i, k, true, bk.scores[p]);
            ++c.updated;
        }
        return c;
    }

    Counts erase(uint64_t n, const uint64_t* keys) {
        Counts c;
        for (uint64_t i = 0; i < n; ++i) {
            uint64_t k = keys[i];
            if (is_reserved(k)) { ++c.reserved; continue; }
            if (skip_for_filter(k, c)) continue;
            uint64_t b; int p;
            if (!locate(k, &b, &p)) continue;
            remove_entry(at(b), p);
            ++c.erased;
        }
        return c;
    }

    // HKV Algorithm 1 (and its two-bucket form in dual mode): membership.
    uint64_t find(uint64_t n, const uint64_t* keys, float* values_out, uint8_t* found_out,
                  uint64_t* scores_out) {
        uint64_t hits = 0;
        for (uint64_t i = 0; i < n; ++i) {
            uint64_t k = keys[i];
            uint64_t b; int p;
            if (is_reserved(k) || !locate(k, &b, &p)) { found_out[i] = 0; continue; }
            Bucket& bk = at(b);
            found_out[i] = 1;
            std::memcpy(values_out + i * dim, &bk.values[static_cast<size_t>(p) * dim],
                        sizeof(float) * dim);
            if (scores_out) scores_out[i] = bk.scores[p];
            ++hits;
        }
        return hits;
    }

    uint64_t size() const {
        uint64_t s = 0;
        for (const auto& kv : buckets) s += kv.second.keys.size();
        return s;
    }
};

struct Row { uint64_t key, score; const float* v; };

}  // namespace

extern "C" {

struct oracle_counts {
    uint64_t updated, admitted, evicted, rejected, reserved, filtered, erased;
};

static void put(const Counts& c, oracle_counts* out) {
    if (!out) return;
    out->updated = c.updated; out->admitted = c.admitted; out->evicted = c.evicted;
    out->rejected = c.rejected; out->reserved = c.reserved; out->filtered = c.filtered;
    out->erased = c.erased;
}

// policy: 0 kCustomized, 1 kLru, 2 kLfu, 3 kEpochLru, 4 kEpochLfu (R10).
// Under kLru and kEpochLru the callers below must pass scores = NULL.
void* oracle_create(uint64_t num_buckets, uint32_t dim, int dual, uint32_t policy) {
    if (num_buckets == 0 || dim == 0 || (dual && num_buckets < 2) || policy > kEpochLfu)
        return nullptr;
    Table* t = new Table();
    t->num_buckets = num_buckets;
    t->dim = dim;
    t->dual = dual != 0;
    t->policy = policy;
    return t;
}

void oracle_set_epoch(void* h, uint32_t epoch) { static_cast<Table*>(h)->epoch = epoch; }

void oracle_destroy(void* h) { delete static_cast<Table*>(h); }

// Restrict the model to the listed buckets (single mode only); keys hashed
// elsewhere are ignored and counted as "filtered".
int oracle_set_bucket_filter(void* h, uint64_t n, const uint64_t* buckets) {
    Table* t = static_cast<Table*>(h);
    if (t->dual) return -1;
    t->filtered = true;
    t->filter.clear();
    for (uint64_t i = 0; i < n; ++i) t->filter.insert(buckets[i]);
    return 0;
}

uint64_t oracle_hash(uint64_t key) { return murmur_fmix64(key); }

uint64_t oracle_bucket(void* h, uint64_t key, int which) {
    Table* t = static_cast<Table*>(h);
    return which == 0 ? t->bucket1(key) : t->bucket2(key);
}

void oracle_buckets(void* h, uint64_t n, const uint64_t* keys, int which, uint64_t* out) {
    Table* t = static_cast<Table*>(h);
    for (uint64_t i = 0; i < n; ++i) out[i] = which == 0 ? t->bucket1(keys[i]) : t->bucket2(keys[i]);
}

uint64_t oracle_step(void* h) { return static_cast<Table*>(h)->step; }

void oracle_insert_or_assign(void* h, uint64_t n, const uint64_t* keys, const float* values,
                             const uint64_t* scores, oracle_counts* out) {
    put(static_cast<Table*>(h)->insert_or_assign(n, keys, values, scores), out);
}

void oracle_assign(void* h, uint64_t n, const uint64_t* keys, const float* values,
                   const uint64_t* scores, oracle_counts* out) {
    put(static_cast<Table*>(h)->assign(n, keys, values, scores), out);
}

void oracle_erase(void* h, uint64_t n, const uint64_t* keys, oracle_counts* out) {
    put(static_cast<Table*>(h)->erase(n, keys), out);
}

// insert_and_evict (HKV §4.1): insert_or_assign that also returns the entries
// resident before the call that it displaced, sorted by key.  Outputs need
// room for n entries; *count_out receives their number.
void oracle_insert_and_evict(void* h, uint64_t n, const uint64_t* keys, const float* values,
                             const uint64_t* scores, uint64_t* ev_keys, float* ev_values,
                             uint64_t* ev_scores, uint64_t* count_out, oracle_counts* out) {
    Table* t = static_cast<Table*>(h);
    std::vector<Table::Victim> ev;
    put(t->insert_or_assign(n, keys, values, scores, true, &ev), out);
    std::sort(ev.begin(), ev.end(),
              [](const Table::Victim& a, const Table::Victim& b) { return a.key < b.key; });
    for (size_t i = 0; i < ev.size(); ++i) {
        ev_keys[i] = ev[i].key;
        ev_scores[i] = ev[i].score;
        std::memcpy(ev_values + i * t->dim, ev[i].value.data(), sizeof(float) * t->dim);
    }
    *count_out = ev.size();
}

// find_or_insert (HKV §4.1): absent keys are inserted with their row of
// values_inout (and their score) under Algorithm 2; resident keys are left
// as they are.  Then every key that is resident after the call gets
// found_out = 1 and its stored row in values_inout; the others get
// found_out = 0 and keep their row.
void oracle_find_or_insert(void* h, uint64_t n, const uint64_t* keys, float* values_inout,
                           const uint64_t* scores, uint8_t* found_out, oracle_counts* out) {
    Table* t = static_cast<Table*>(h);
    put(t->insert_or_assign(n, keys, values_inout, scores, false, nullptr), out);
    t->find(n, keys, values_inout, found_out, nullptr);
}

// contains (HKV §3.5 reader): found_out[i] = 1 iff keys[i] is resident.
void oracle_contains(void* h, uint64_t n, const uint64_t* keys, uint8_t* found_out) {
    Table* t = static_cast<Table*>(h);
    for (uint64_t i = 0; i < n; ++i) {
        uint64_t b; int p;
        found_out[i] = (!is_reserved(keys[i]) && t->locate(keys[i], &b, &p)) ? 1 : 0;
    }
}

uint64_t oracle_find(void* h, uint64_t n, const uint64_t* keys, float* values_out,
                     uint8_t* found_out, uint64_t* scores_out) {
    return static_cast<Table*>(h)->find(n, keys, values_out, found_out, scores_out);
}

uint64_t oracle_size(void* h) { return static_cast<Table*>(h)->size(); }

uint64_t oracle_bucket_size(void* h, uint64_t b) {
    Table* t = static_cast<Table*>(h);
    auto it = t->buckets.find(b);
    return it == t->buckets.end() ? 0 : it->second.keys.size();
}

// Entries of buckets [b_begin, b_end) whose score is >= min_score, sorted by
// key.  Pass NULL outputs to only count.  Returns the number of entries.
uint64_t oracle_export(void* h, uint64_t b_begin, uint64_t b_end, uint64_t min_score,
                       uint64_t* keys_out, float* values_out, uint64_t* scores_out) {
    Table* t = static_cast<Table*>(h);
    std::vector<Row> rows;
    for (auto& kv : t->buckets) {
        if (kv.first < b_begin || kv.first >= b_end) continue;
        const Bucket& bk = kv.second;
        for (int i = 0; i < bk.size(); ++i)
            if (bk.scores[i] >= min_score)
                rows.push_back({bk.keys[i], bk.scores[i], &bk.values[static_cast<size_t>(i) * t->dim]});
    }
    std::sort(rows.begin(), rows.end(), [](const Row& a, const Row& b) { return a.key < b.key; });
    for (size_t i = 0; i < rows.size(); ++i) {
        if (keys_out) keys_out[i] = rows[i].key;
        if (scores_out) scores_out[i] = rows[i].score;
        if (values_out) std::memcpy(values_out + i * t->dim, rows[i].v, sizeof(float) * t->dim);
    }
    return rows.size();
}

}  // extern "C"
