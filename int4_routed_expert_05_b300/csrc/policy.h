// policy.h -- slot policy of the bounded expert pool (host only, no CUDA).
//
// The pool caches hot experts in a fixed number of slots and evicts with LFU plus recency
// (paotong.dev commentary on Swiftlet: bounded pool, LFU + recency eviction, 43-70% hits;
// cheshm.ai item, scheduling paragraph). The pages do not give the exact rule; this one is:
//  - one pool over all layers, keyed by (layer, expert);
//  - every lookup call advances a tick; a hit adds one use and stamps the slot with the tick;
//  - a miss takes the lowest free slot, else evicts the unpinned slot with the smallest
//    (uses, last tick, slot index); the new entry starts with one use and the current tick;
//  - every expert looked up or loaded since the last release is pinned and cannot be evicted.
#pragma once
#include <cstdint>
#include <set>
#include <tuple>
#include <vector>

namespace moe {

class SlotPolicy {
public:
    SlotPolicy() = default;
    SlotPolicy(int n_layers, int n_experts, int n_slots)
        : L_(n_layers), E_(n_experts), S_(n_slots), table_((size_t)n_layers * n_experts, -1),
          owner_(n_slots, -1), uses_(n_slots, 0), last_(n_slots, 0), pinned_(n_slots, 0)
    {
        for (int s = 0; s < n_slots; ++s)
            free_.insert(s);
    }

    int slots() const { return S_; }
    int slot_of(int layer, int expert) const { return table_[(size_t)layer * E_ + expert]; }
    const std::vector<int32_t>& table() const { return table_; }
    uint64_t tick() const { return tick_; }

    // Lookup of n experts of one layer (one tick). out[i] = slot or -1. Hits are pinned.
    void lookup(int layer, const int32_t* experts, int n, int32_t* out, int64_t* hits, int64_t* misses)
    {
        ++tick_;
        for (int i = 0; i < n; ++i) {
            const int s = slot_of(layer, experts[i]);
            out[i] = s;
            if (s >= 0) {
                unlink(s);
                ++uses_[s];
                last_[s] = tick_;
                pin(s);
                ++*hits;
            } else {
                ++*misses;
            }
        }
    }

    // Choose the slot for a missing (layer, expert): -1 if every slot is pinned. *victim_key
    // receives the evicted entry's key (-1 if the slot was free). Does not change any state.
    int choose(int* victim_key) const
    {
        if (!free_.empty()) {
            *victim_key = -1;
            return *free_.begin();
        }
        if (evictable_.empty())
            return -1;
        const int s = std::get<2>(*evictable_.begin());
        *victim_key = owner_[s];
        return s;
    }

    // Install (layer, expert) in slot s chosen by choose(); the entry is pinned.
    void install(int layer, int expert, int s)
    {
        if (owner_[s] >= 0) {
            unlink(s);
            table_[owner_[s]] = -1;
        } else {
            free_.erase(s);
        }
        const int key = layer * E_ + expert;
        owner_[s] = key;
        table_[key] = s;
        uses_[s] = 1;
        last_[s] = tick_;
        pin(s);
    }

    // Resident placement: (layer, expert) lives in slot s, not pinned.
    void place(int layer, int expert, int s)
    {
        const int key = layer * E_ + expert;
        if (table_[key] >= 0 && table_[key] != s)
            drop(table_[key]);
        if (owner_[s] >= 0 && owner_[s] != key)
            table_[owner_[s]] = -1;
        if (owner_[s] < 0)
            free_.erase(s);
        unlink(s);
        owner_[s] = key;
        table_[key] = s;
        uses_[s] = 0;
        last_[s] = tick_;
        if (!pinned_[s])
            evictable_.insert(std::make_tuple(uses_[s], last_[s], s));
    }

    const std::vector<int>& pinned_list() const { return pin_list_; }

    void release()
    {
        for (int s : pin_list_) {
            pinned_[s] = 0;
            if (owner_[s] >= 0)
                evictable_.insert(std::make_tuple(uses_[s], last_[s], s));
        }
        pin_list_.clear();
    }

private:
    void pin(int s)
    {
        if (!pinned_[s]) {
            pinned_[s] = 1;
            pin_list_.push_back(s);
        }
    }
    void unlink(int s)
    {
        if (!pinned_[s] && owner_[s] >= 0)
            evictable_.erase(std::make_tuple(uses_[s], last_[s], s));
    }
    void drop(int s)
    {
        unlink(s);
        if (owner_[s] >= 0)
            table_[owner_[s]] = -1;
        owner_[s] = -1;
        uses_[s] = 0;
        free_.insert(s);
    }

    int L_ = 0, E_ = 0, S_ = 0;
    uint64_t tick_ = 0;
    std::vector<int32_t> table_;   // (layer * E + expert) -> slot
    std::vector<int> owner_;       // slot -> key or -1
    std::vector<uint64_t> uses_, last_;
    std::vector<char> pinned_;
    std::vector<int> pin_list_;
    std::set<int> free_;
    std::set<std::tuple<uint64_t, uint64_t, int>> evictable_;
};

}  // namespace moe
