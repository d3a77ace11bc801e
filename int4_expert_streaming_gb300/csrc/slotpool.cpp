// slotpool.cpp -- the bounded per-layer expert slot pool and its eviction policy.
//
// Swiftlet caches hot experts in a bounded pool evicted by "LFU + LRU"
// (article section 3 "Expert cache pool and LFU+LRU eviction") / "LFU plus
// recency" (README "How it works").  Reading taken here: the victim is the
// slot with the smallest (use count, last use, slot index) among slots whose
// expert is not requested by the same call; use counts start at 1 when an
// expert is loaded and are dropped on eviction; free slots fill lowest index
// first.  MOE_EVICT_LRU ranks by (last use, slot index) only.
//
// Two count lifetimes that the pages leave open are offered for comparison:
// MOE_EVICT_LFU_PERSIST keeps one all-time request count per expert (kept
// across evictions, raised for the whole request before any victim is
// chosen); MOE_EVICT_LFU_AGED halves every occupied slot's count, rounding
// down, when a call starts at a clock that is a positive multiple of the
// aging period.
#include <vector>

#include "moe_internal.h"

struct moe_slotpool {
    int32_t slots, n_experts, policy, aging;
    std::vector<int32_t> slot_expert;  // -1 = free
    std::vector<int64_t> freq, last;   // per slot
    std::vector<int64_t> count;        // per expert, all calls (LFU_PERSIST)
    std::vector<int32_t> expert_slot;  // -1 = not resident
    std::vector<uint8_t> requested;    // scratch: expert requested by the current call
    int32_t n_free;
    int64_t clock;
};

extern "C" int moe_slotpool_create(int32_t slots, int32_t n_experts, int32_t policy, int32_t aging_period,
                                   moe_slotpool** out) {
    if (!out || slots < 1 || n_experts < 1 || policy < MOE_EVICT_LFU_RECENCY || policy > MOE_EVICT_LFU_AGED)
        return MOE_EINVAL;
    moe_slotpool* p = new (std::nothrow) moe_slotpool;
    if (!p) return MOE_ENOMEM;
    p->slots = slots;
    p->n_experts = n_experts;
    p->policy = policy;
    p->aging = aging_period > 0 ? aging_period : 64;
    p->slot_expert.assign(slots, -1);
    p->count.assign(n_experts, 0);
    p->freq.assign(slots, 0);
    p->last.assign(slots, -1);
    p->expert_slot.assign(n_experts, -1);
    p->requested.assign(n_experts, 0);
    p->n_free = slots;
    p->clock = 0;
    *out = p;
    return MOE_OK;
}

extern "C" void moe_slotpool_destroy(moe_slotpool* p) { delete p; }

extern "C" int moe_slotpool_request(moe_slotpool* p, const int32_t* req, int32_t n, int32_t* events) {
    if (!p || n < 0 || (n > 0 && (!req || !events))) return MOE_EINVAL;
    if (n > p->slots) return MOE_EPOOL;
    for (int32_t i = 0; i < n; ++i)
        if (req[i] < 0 || req[i] >= p->n_experts || (i > 0 && req[i] <= req[i - 1])) return MOE_EINVAL;
    const int64_t t = p->clock;
    if (p->policy == MOE_EVICT_LFU_AGED && t > 0 && t % p->aging == 0)
        for (int32_t k = 0; k < p->slots; ++k)
            if (p->slot_expert[k] >= 0) p->freq[k] >>= 1;
    for (int32_t i = 0; i < n; ++i) p->requested[req[i]] = 1;
    if (p->policy == MOE_EVICT_LFU_PERSIST)
        for (int32_t i = 0; i < n; ++i) p->count[req[i]] += 1;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t e = req[i];
        int32_t* ev = events + 4 * i;
        const int32_t s = p->expert_slot[e];
        if (s >= 0) {
            p->freq[s] += 1;
            p->last[s] = t;
            ev[0] = e, ev[1] = 0, ev[2] = s, ev[3] = -1;
            continue;
        }
        int32_t victim = -1, evicted = -1;
        if (p->n_free > 0) {
            for (int32_t k = 0; k < p->slots; ++k)
                if (p->slot_expert[k] < 0) {
                    victim = k;
                    break;
                }
            p->n_free -= 1;
        } else {
            for (int32_t k = 0; k < p->slots; ++k) {
                if (p->requested[p->slot_expert[k]]) continue;
                if (victim < 0) {
                    victim = k;
                    continue;
                }
                if (p->policy == MOE_EVICT_LRU) {
                    if (p->last[k] < p->last[victim]) victim = k;
                    continue;
                }
                const int64_t fk = p->policy == MOE_EVICT_LFU_PERSIST ? p->count[p->slot_expert[k]] : p->freq[k];
                const int64_t fv =
                    p->policy == MOE_EVICT_LFU_PERSIST ? p->count[p->slot_expert[victim]] : p->freq[victim];
                if (fk < fv || (fk == fv && p->last[k] < p->last[victim])) victim = k;
            }
            evicted = p->slot_expert[victim];  // a victim exists: n <= slots and every requested expert pins one slot
            p->expert_slot[evicted] = -1;
        }
        p->slot_expert[victim] = e;
        p->freq[victim] = 1;
        p->last[victim] = t;
        p->expert_slot[e] = victim;
        ev[0] = e, ev[1] = 1, ev[2] = victim, ev[3] = evicted;
    }
    for (int32_t i = 0; i < n; ++i) p->requested[req[i]] = 0;
    p->clock += 1;
    return n;
}

// internal: number of resident experts
int32_t moe_slotpool_resident(const moe_slotpool* p) { return p->slots - p->n_free; }
