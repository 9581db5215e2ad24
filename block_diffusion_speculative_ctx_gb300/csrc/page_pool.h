// Host-side allocator of the paged KV cache: one pool of physical pages shared
// by the sequence slots of a session.  A slot's logical page j (tokens
// [64 j, 64 j + 64) of its sequence) maps to a physical page through the page
// table; pages are handed out as the sequences grow and all return at the
// next reset (a new batch).  The last physical page is a scratch page that is
// never handed out: every table entry not backed by a page of its own points
// at it, so a speculative read past a sequence's end stays inside the cache.
// Plain C++ (no CUDA): the library mirrors table() to the device.
#pragma once

#include <algorithm>
#include <cstddef>
#include <vector>

namespace dfl {

class PagePool {
  public:
    // `pages` physical pages (the last one the scratch page), `slots` rows of
    // `per_slot` table entries.
    void init(int pages, int slots, int per_slot) {
        pages_ = pages;
        slots_ = slots;
        per_slot_ = per_slot;
        reset();
    }

    // Every page back to the pool, every entry on the scratch page; the whole
    // table needs uploading.
    void reset() {
        free_.clear();
        for (int p = scratch() - 1; p >= 0; --p) free_.push_back(p);  // page 0 is handed out first
        backed_.assign(slots_, 0);
        table_.assign((size_t)slots_ * per_slot_, scratch());
        full_dirty_ = true;
        pending_.clear();
    }

    // Back the slot's tokens [0, tokens) (at most per_slot pages) with pages of
    // its own.  False when the pool runs out; the pages taken before that stay
    // with the slot.
    bool ensure(int slot, long long tokens, int page_tokens) {
        const long long need_ll = (tokens + page_tokens - 1) / page_tokens;
        const int need = (int)std::min<long long>(need_ll, per_slot_);
        while (backed_[slot] < need) {
            if (free_.empty()) return false;
            const size_t e = (size_t)slot * per_slot_ + backed_[slot]++;
            table_[e] = free_.back();
            free_.pop_back();
            pending_.push_back((int)e);
        }
        return true;
    }

    // The slot's first `n` logical pages become `from`'s (shared physical pages:
    // the training forward's blocks read the clean sequence's context this way).
    void share(int slot, int from, int n) {
        for (int t = 0; t < n; ++t) {
            const size_t e = (size_t)slot * per_slot_ + t;
            table_[e] = table_[(size_t)from * per_slot_ + t];
            pending_.push_back((int)e);
        }
        backed_[slot] = std::max(backed_[slot], n);
    }

    int page(int slot, int logical) const { return table_[(size_t)slot * per_slot_ + logical]; }
    int scratch() const { return pages_ - 1; }
    int capacity() const { return pages_ - 1; }
    int in_use() const { return capacity() - (int)free_.size(); }
    int per_slot() const { return per_slot_; }
    const std::vector<int>& table() const { return table_; }

    // Entries changed since the last upload: all of them after a reset, else the list.
    bool full_dirty() const { return full_dirty_; }
    const std::vector<int>& pending() const { return pending_; }
    void uploaded() {
        full_dirty_ = false;
        pending_.clear();
    }

  private:
    int pages_ = 1, slots_ = 0, per_slot_ = 0;
    std::vector<int> free_;    // stack of pages not handed out
    std::vector<int> backed_;  // logical pages of each slot that have a page
    std::vector<int> table_;   // [slots][per_slot] physical page of each entry
    bool full_dirty_ = false;
    std::vector<int> pending_;
};

}  // namespace dfl
