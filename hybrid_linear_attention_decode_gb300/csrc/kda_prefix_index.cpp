// kda_prefix_index.cpp -- host-side prefix index and retention policies for KDA state checkpoints.
//
// What it implements ("A Preview of Production-Scale Kimi K3 Support on vLLM", section "The Hardest
// Part: Prefix Caching for KDA"; "vLLM Kimi K3 Support", section "Agentic Cache Retention Policies";
// "moonshotai/Kimi-K3" recipe, prefix-match unit 128):
//   * chained fine-grained hashes: the hash of boundary b covers the whole prefix (hash of boundary b-1
//     combined with the tokens of block b), so a hit identifies the entire prefix, not just its tail;
//   * a state is registered at a fine boundary (a multiple of the match unit) inside a larger pool;
//   * copy-on-write: a request that hits a cached state gets a private slot; the plan copies the cached
//     slot into it (kda_resume_from_slot) and prefills from the boundary;
//   * deferred same-step reuse: entries created by a plan become visible to lookups only at commit, so a
//     request planned in the same step cannot resume from a state that is still being written;
//   * retention policies: interval retention (boundaries at multiples of an interval, plus the last
//     boundary of the prompt) and selective second-hit retention (a boundary's state is kept only once
//     its prefix has been seen before).
// Pure host code: no CUDA calls, no allocation of device memory (slots are indices into the caller's pool).
#include <stdint.h>

#include <algorithm>
#include <list>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/kda.h"

namespace {

// splitmix64 finaliser; the block hash chains it over (previous hash, token ids, block index).
inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t block_hash(uint64_t prev, const int32_t *tokens, int32_t n) {
    uint64_t h = mix64(prev ^ 0x9E3779B97F4A7C15ull);
    for (int32_t i = 0; i < n; ++i) h = mix64(h + (uint64_t)(uint32_t)tokens[i] * 0x9E3779B97F4A7C15ull + (uint64_t)i);
    return h;
}

struct Entry {
    int32_t slot = -1;        // pool slot holding the state at this boundary (-1: ghost, seen but not kept)
    int64_t prefix_len = 0;   // the boundary (tokens in the prefix)
    int32_t pins = 0;         // plans that read this slot and have not committed yet
    bool visible = false;     // committed (usable by lookups)
    bool was_ghost = false;   // a committed ghost that a pending plan is turning into a kept state
    uint64_t plan_id = 0;     // plan that created it (while not visible)
    std::list<uint64_t>::iterator lru;  // position in the LRU list (visible, kept entries only)
};

struct PlanRec {
    std::vector<uint64_t> created;  // entries this plan registered (made visible at commit)
    uint64_t pinned = 0;            // entry whose slot this plan reads (0: none)
    bool has_pin = false;
    int32_t private_slot = -1;
};

}  // namespace

struct kda_prefix_index {
    int32_t num_slots = 0, unit = 128, policy = KDA_RETAIN_INTERVAL;
    int64_t interval = 0;
    std::vector<int32_t> free_slots;
    std::unordered_map<uint64_t, Entry> entries;
    std::list<uint64_t> lru;  // least recently used first (kept, visible, unpinned candidates)
    std::unordered_map<uint64_t, PlanRec> plans;
    uint64_t next_plan = 1;
    std::mutex mu;

    int32_t take_slot() {
        if (!free_slots.empty()) {
            const int32_t s = free_slots.back();
            free_slots.pop_back();
            return s;
        }
        // evict the least recently used visible, unpinned entry
        for (auto it = lru.begin(); it != lru.end(); ++it) {
            auto e = entries.find(*it);
            if (e == entries.end() || e->second.pins > 0 || e->second.slot < 0) continue;
            const int32_t s = e->second.slot;
            lru.erase(it);
            entries.erase(e);
            return s;
        }
        return -1;
    }
    void touch(uint64_t key, Entry &e) {
        if (e.visible && e.slot >= 0) {
            lru.erase(e.lru);
            e.lru = lru.insert(lru.end(), key);
        }
    }
};

extern "C" {

kda_prefix_index *kda_prefix_index_create(int32_t num_slots, int32_t match_unit, int32_t policy, int64_t interval) {
    if (num_slots <= 0 || match_unit <= 0) return nullptr;
    if (policy != KDA_RETAIN_INTERVAL && policy != KDA_RETAIN_SECOND_HIT) return nullptr;
    if (interval < 0 || (interval > 0 && interval % match_unit != 0)) return nullptr;
    kda_prefix_index *ix = new (std::nothrow) kda_prefix_index();
    if (!ix) return nullptr;
    ix->num_slots = num_slots;
    ix->unit = match_unit;
    ix->policy = policy;
    ix->interval = interval;
    ix->free_slots.reserve(num_slots);
    for (int32_t s = num_slots - 1; s >= 0; --s) ix->free_slots.push_back(s);
    return ix;
}

void kda_prefix_index_destroy(kda_prefix_index *ix) { delete ix; }

int32_t kda_prefix_index_free_slots(kda_prefix_index *ix) {
    if (!ix) return -1;
    std::lock_guard<std::mutex> g(ix->mu);
    return (int32_t)ix->free_slots.size();
}

int kda_prefix_plan(kda_prefix_index *ix, const int32_t *tokens, int64_t len, kda_prefix_plan_t *out,
                    int32_t *ckpt_slots, int32_t ckpt_capacity) {
    if (!ix || !out || (len > 0 && !tokens) || len < 0 || ckpt_capacity < 0 || (ckpt_capacity > 0 && !ckpt_slots))
        return KDA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(ix->mu);
    const int64_t U = ix->unit;
    const int64_t nb = len / U;  // complete blocks in the prompt
    // chained hashes of every complete block
    std::vector<uint64_t> hs((size_t)nb);
    uint64_t h = 0;
    for (int64_t b = 0; b < nb; ++b) {
        h = block_hash(h, tokens + b * U, (int32_t)U);
        hs[(size_t)b] = h;
    }
    // longest visible cached prefix (the prefix must leave at least one token to prefill)
    int64_t hit_block = -1;
    for (int64_t b = nb - 1; b >= 0; --b) {
        if ((b + 1) * U >= len) continue;
        auto it = ix->entries.find(hs[(size_t)b]);
        if (it != ix->entries.end() && it->second.visible && it->second.slot >= 0) {
            hit_block = b;
            break;
        }
    }
    const int64_t start = hit_block >= 0 ? (hit_block + 1) * U : 0;
    // checkpoint boundaries of this prefill: every multiple of the match unit in (start, len]
    const int64_t first = start / U + 1, last = len / U;
    const int64_t nck = last >= first ? last - first + 1 : 0;
    if (nck > ckpt_capacity) return KDA_ERR_INVALID_ARG;
    PlanRec rec;
    if (hit_block >= 0) {  // pin the source first so that taking slots below cannot evict it
        Entry &e = ix->entries[hs[(size_t)hit_block]];
        e.pins += 1;
        ix->touch(hs[(size_t)hit_block], e);
        rec.pinned = hs[(size_t)hit_block];
        rec.has_pin = true;
    }
    const int32_t priv = ix->take_slot();
    if (priv < 0) {  // pool exhausted by pinned / pending states
        if (rec.has_pin) ix->entries[rec.pinned].pins -= 1;
        return KDA_ERR_WORKSPACE;
    }
    const uint64_t pid = ix->next_plan++;
    rec.private_slot = priv;
    // second-hit retention: the longest boundary of this prompt whose prefix an earlier request has
    // already seen (a committed ghost entry) is the shared prefix worth keeping
    int64_t shared_last = -1;
    if (ix->policy == KDA_RETAIN_SECOND_HIT)
        for (int64_t b = last; b >= first; --b) {
            auto it = ix->entries.find(hs[(size_t)(b - 1)]);
            if (it != ix->entries.end() && it->second.visible && it->second.slot < 0) {
                shared_last = b * U;
                break;
            }
        }
    for (int64_t j = 0; j < nck; ++j) {
        const int64_t p = (first + j) * U;
        const uint64_t key = hs[(size_t)(p / U - 1)];
        int32_t slot = -1;
        auto it = ix->entries.find(key);
        const bool known = it != ix->entries.end();
        const bool on_interval = ix->interval > 0 && p % ix->interval == 0;
        bool keep = false;
        if (ix->policy == KDA_RETAIN_INTERVAL) {
            keep = on_interval || p == last * U;  // fixed intervals and the prompt's last boundary
        } else {  // kept only once seen before: the shared boundary, and seen interval boundaries
            const bool seen = known && it->second.visible && it->second.slot < 0;
            keep = seen && (p == shared_last || on_interval);
        }
        if (keep && (!known || it->second.slot < 0)) {
            slot = ix->take_slot();
            if (slot >= 0) {
                Entry &e = ix->entries[key];
                e.was_ghost = known;
                e.slot = slot;
                e.prefix_len = p;
                e.visible = false;
                e.plan_id = pid;
                rec.created.push_back(key);
            }
        } else if (!known && ix->policy == KDA_RETAIN_SECOND_HIT) {
            Entry &e = ix->entries[key];  // first sight: remember the prefix without keeping its state
            e.slot = -1;
            e.prefix_len = p;
            e.visible = false;
            e.plan_id = pid;
            rec.created.push_back(key);
        }
        ckpt_slots[j] = slot;
    }
    ix->plans[pid] = rec;
    out->plan_id = pid;
    out->src_slot = hit_block >= 0 ? ix->entries[hs[(size_t)hit_block]].slot : -1;
    out->private_slot = priv;
    out->start_pos = start;
    out->num_ckpts = (int32_t)nck;
    return KDA_OK;
}

int kda_prefix_commit(kda_prefix_index *ix, uint64_t plan_id) {
    if (!ix) return KDA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(ix->mu);
    auto it = ix->plans.find(plan_id);
    if (it == ix->plans.end()) return KDA_ERR_INVALID_ARG;
    for (uint64_t key : it->second.created) {
        auto e = ix->entries.find(key);
        if (e == ix->entries.end() || e->second.plan_id != plan_id) continue;
        e->second.visible = true;
        e->second.was_ghost = false;
        if (e->second.slot >= 0) e->second.lru = ix->lru.insert(ix->lru.end(), key);
    }
    if (it->second.has_pin) {
        auto e = ix->entries.find(it->second.pinned);
        if (e != ix->entries.end() && e->second.pins > 0) e->second.pins -= 1;
    }
    ix->plans.erase(it);
    return KDA_OK;
}

int kda_prefix_abort(kda_prefix_index *ix, uint64_t plan_id) {
    if (!ix) return KDA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(ix->mu);
    auto it = ix->plans.find(plan_id);
    if (it == ix->plans.end()) return KDA_ERR_INVALID_ARG;
    for (uint64_t key : it->second.created) {
        auto e = ix->entries.find(key);
        if (e == ix->entries.end() || e->second.plan_id != plan_id || e->second.visible) continue;
        if (e->second.slot >= 0) ix->free_slots.push_back(e->second.slot);
        if (e->second.was_ghost) {  // back to the committed ghost it was
            e->second.slot = -1;
            e->second.visible = true;
            e->second.was_ghost = false;
        } else {
            ix->entries.erase(e);
        }
    }
    if (it->second.has_pin) {
        auto e = ix->entries.find(it->second.pinned);
        if (e != ix->entries.end() && e->second.pins > 0) e->second.pins -= 1;
    }
    ix->free_slots.push_back(it->second.private_slot);
    ix->plans.erase(it);
    return KDA_OK;
}

int kda_prefix_release_slot(kda_prefix_index *ix, int32_t slot) {
    if (!ix || slot < 0 || slot >= ix->num_slots) return KDA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(ix->mu);
    for (const auto &kv : ix->entries)
        if (kv.second.slot == slot) return KDA_ERR_INVALID_ARG;  // cached states are released by eviction
    if (std::find(ix->free_slots.begin(), ix->free_slots.end(), slot) != ix->free_slots.end())
        return KDA_ERR_INVALID_ARG;
    ix->free_slots.push_back(slot);
    return KDA_OK;
}

}  // extern "C"
