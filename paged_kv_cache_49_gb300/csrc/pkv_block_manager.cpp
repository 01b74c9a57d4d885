// Host block manager: free list, reference counts, page-rounded admission
// with full output reservation, prefix groups, fork and copy-on-write.
//
// Policy sources: cs2680 Lecture 10, §10.3 (block pool and per-sequence block
// table, growth by one entry) and §10.4 (reference-counted sharing, copy on
// divergence); "KV cache systems", copy-on-write paragraph (the first writer
// of a shared block copies it); "Reserve the page a request has not written
// yet" (reserve ceil((prompt + output) / 16) pages at admission; reserve and
// admit as one serialised decision; charge shared prefix pages once; freeing
// changes ownership, not device memory).
#include <algorithm>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

namespace {

struct Sequence {
    std::vector<int32_t> table;
    int64_t ctx = 0;
    int group = -1;
};

struct Group {
    std::vector<int32_t> pages;
    int prefix_len = 0;
    int members = 0;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

struct pkv_bm {
    int num_blocks = 0;
    int block_tokens = 16;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> ref;
    std::vector<std::vector<int32_t>> spares;  // per block: pages reserved for its CoW
    std::unordered_map<int, Sequence> seqs;
    std::unordered_map<int, Group> groups;
    int next_id = 0;
    int64_t cow_copies = 0;
    int64_t spare_count = 0;
    std::mutex mu;

    int32_t pop() {
        int32_t b = free_stack.back();
        free_stack.pop_back();
        return b;
    }
    void push(int32_t b) { free_stack.push_back(b); }
    int num_free() const { return static_cast<int>(free_stack.size()); }
};

extern "C" {

pkv_bm* pkv_bm_create(int num_blocks, int block_tokens, const int32_t* free_order) {
    if (num_blocks <= 0 || (block_tokens != 8 && block_tokens != 16 && block_tokens != 32 && block_tokens != 64))
        return nullptr;
    auto* bm = new pkv_bm();
    bm->num_blocks = num_blocks;
    bm->block_tokens = block_tokens;
    bm->ref.assign(num_blocks, 0);
    bm->spares.assign(num_blocks, {});
    bm->free_stack.resize(num_blocks);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete bm;
                return nullptr;
            }
            seen[b] = 1;
            bm->free_stack[num_blocks - 1 - i] = b;
        }
    } else {
        for (int i = 0; i < num_blocks; ++i) bm->free_stack[num_blocks - 1 - i] = i;
    }
    return bm;
}

void pkv_bm_destroy(pkv_bm* bm) { delete bm; }

pkv_status pkv_bm_admit(pkv_bm* bm, int prompt_len, int max_new, int group, int prefix_len,
                        int* seq_id) {
    if (!bm || !seq_id) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    if (prompt_len < 0 || max_new < 0 || static_cast<int64_t>(prompt_len) + max_new <= 0)
        return PKV_EINVAL;
    const int64_t total = ceil_div(static_cast<int64_t>(prompt_len) + max_new, bm->block_tokens);
    int64_t n_shared = 0;
    const std::vector<int32_t>* shared = nullptr;
    Group* existing = nullptr;
    if (group >= 0) {
        if (prefix_len < 0 || prefix_len > prompt_len) return PKV_EINVAL;
        n_shared = prefix_len / bm->block_tokens;
        auto it = bm->groups.find(group);
        if (it != bm->groups.end()) {
            if (it->second.prefix_len != prefix_len) return PKV_EINVAL;
            existing = &it->second;
            shared = &existing->pages;
        }
    }
    const int64_t need = total - (shared ? static_cast<int64_t>(shared->size()) : 0);
    if (need > bm->num_free()) return PKV_ENOMEM;

    Sequence seq;
    seq.ctx = prompt_len;
    seq.group = group;
    seq.table.reserve(total);
    if (group >= 0 && !existing) {
        Group g;
        g.prefix_len = prefix_len;
        for (int64_t i = 0; i < n_shared; ++i) g.pages.push_back(bm->pop());
        existing = &(bm->groups[group] = std::move(g));
        shared = &existing->pages;
    }
    if (shared) seq.table.insert(seq.table.end(), shared->begin(), shared->end());
    while (static_cast<int64_t>(seq.table.size()) < total) seq.table.push_back(bm->pop());
    for (int32_t b : seq.table) bm->ref[b] += 1;
    if (existing) existing->members += 1;
    const int id = bm->next_id++;
    bm->seqs.emplace(id, std::move(seq));
    *seq_id = id;
    return PKV_OK;
}

pkv_status pkv_bm_fork(pkv_bm* bm, int parent_seq, int n, int32_t* child_ids) {
    if (!bm || n < 0 || (n > 0 && !child_ids)) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(parent_seq);
    if (it == bm->seqs.end()) return PKV_EINVAL;
    const Sequence parent = it->second;  // copy: emplacing children may rehash
    const int64_t written = ceil_div(parent.ctx, bm->block_tokens);
    const bool partial = parent.ctx % bm->block_tokens != 0;
    const int64_t per_child =
        (static_cast<int64_t>(parent.table.size()) - written) + (partial ? 1 : 0);
    if (static_cast<int64_t>(n) * per_child > bm->num_free()) return PKV_ENOMEM;
    for (int i = 0; i < n; ++i) {
        Sequence child;
        child.ctx = parent.ctx;
        child.group = parent.group;
        child.table.assign(parent.table.begin(), parent.table.begin() + written);
        while (child.table.size() < parent.table.size()) child.table.push_back(bm->pop());
        for (int32_t b : child.table) bm->ref[b] += 1;
        if (partial) {
            bm->spares[parent.table[written - 1]].push_back(bm->pop());
            bm->spare_count += 1;
        }
        if (parent.group >= 0) bm->groups[parent.group].members += 1;
        const int id = bm->next_id++;
        bm->seqs.emplace(id, std::move(child));
        child_ids[i] = id;
    }
    return PKV_OK;
}

pkv_status pkv_bm_prepare_append(pkv_bm* bm, const int32_t* seq_ids, int n,
                                 int64_t* slot_mapping_out, int32_t* cow_pairs_out,
                                 int* n_pairs_out) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slot_mapping_out || !cow_pairs_out)) ||
        !n_pairs_out)
        return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    std::vector<Sequence*> batch(n);
    {
        std::vector<int32_t> sorted(seq_ids, seq_ids + n);
        std::sort(sorted.begin(), sorted.end());
        if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return PKV_EINVAL;
    }
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_EINVAL;
        batch[i] = &it->second;
    }
    for (Sequence* s : batch)
        if (s->ctx / bm->block_tokens >= static_cast<int64_t>(s->table.size())) return PKV_ENOSPC;
    // Every copy-on-write below takes a reserved spare; check before mutating.
    {
        std::unordered_map<int32_t, int64_t> ref_left, spare_left;
        for (Sequence* s : batch) {
            int32_t b = s->table[s->ctx / bm->block_tokens];
            auto r = ref_left.emplace(b, bm->ref[b]).first;
            auto sp = spare_left.emplace(b, bm->spares[b].size()).first;
            if (r->second > 1) {
                if (sp->second == 0) return PKV_ESTATE;
                r->second -= 1;
                sp->second -= 1;
            }
        }
    }
    int pairs = 0;
    for (int i = 0; i < n; ++i) {
        Sequence* s = batch[i];
        const int64_t lb = s->ctx / bm->block_tokens;
        int32_t b = s->table[lb];
        if (bm->ref[b] > 1) {
            std::vector<int32_t>& sp = bm->spares[b];
            const int32_t dst = sp.back();
            sp.pop_back();
            bm->spare_count -= 1;
            bm->ref[b] -= 1;
            bm->ref[dst] = 1;
            s->table[lb] = dst;
            cow_pairs_out[2 * pairs] = b;
            cow_pairs_out[2 * pairs + 1] = dst;
            ++pairs;
            bm->cow_copies += 1;
            b = dst;
        }
        slot_mapping_out[i] = static_cast<int64_t>(b) * bm->block_tokens + s->ctx % bm->block_tokens;
        s->ctx += 1;
    }
    *n_pairs_out = pairs;
    return PKV_OK;
}

pkv_status pkv_bm_free(pkv_bm* bm, int seq_id) {
    if (!bm) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_EINVAL;
    Sequence s = std::move(it->second);
    bm->seqs.erase(it);
    for (int32_t b : s.table) {
        bm->ref[b] -= 1;
        std::vector<int32_t>& sp = bm->spares[b];
        if (!sp.empty() && static_cast<int64_t>(sp.size()) > bm->ref[b] - 1) {
            bm->push(sp.back());
            sp.pop_back();
            bm->spare_count -= 1;
        }
        if (bm->ref[b] == 0) bm->push(b);
    }
    if (s.group >= 0) {
        auto g = bm->groups.find(s.group);
        if (g != bm->groups.end() && --g->second.members == 0) bm->groups.erase(g);
    }
    return PKV_OK;
}

pkv_status pkv_bm_block_table(pkv_bm* bm, int seq_id, int32_t* out, int capacity, int* length) {
    if (!bm || !length || capacity < 0 || (capacity > 0 && !out)) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_EINVAL;
    const auto& t = it->second.table;
    *length = static_cast<int>(t.size());
    if (static_cast<int>(t.size()) > capacity) return PKV_ERANGE;
    std::copy(t.begin(), t.end(), out);
    return PKV_OK;
}

pkv_status pkv_bm_context_len(pkv_bm* bm, int seq_id, int* context_len) {
    if (!bm || !context_len) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_EINVAL;
    *context_len = static_cast<int>(it->second.ctx);
    return PKV_OK;
}

pkv_status pkv_bm_batch_tables(pkv_bm* bm, const int32_t* seq_ids, int n, int32_t* tables_out,
                               int width, int32_t* context_lens_out) {
    if (!bm || n < 0 || width < 0 ||
        (n > 0 && (!seq_ids || !context_lens_out || (width > 0 && !tables_out))))
        return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_EINVAL;
        if (static_cast<int>(it->second.table.size()) > width) return PKV_ERANGE;
    }
    for (int i = 0; i < n; ++i) {
        const Sequence& s = bm->seqs.find(seq_ids[i])->second;
        int32_t* row = tables_out + static_cast<int64_t>(i) * width;
        std::fill(row, row + width, -1);
        std::copy(s.table.begin(), s.table.end(), row);
        context_lens_out[i] = static_cast<int32_t>(s.ctx);
    }
    return PKV_OK;
}

pkv_status pkv_bm_stats(pkv_bm* bm, pkv_bm_stats_t* st) {
    if (!bm || !st) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    st->num_blocks = bm->num_blocks;
    st->free_blocks = bm->num_free();
    st->used_blocks = 0;
    st->shared_blocks = 0;
    st->ref_sum = 0;
    for (int32_t r : bm->ref) {
        st->used_blocks += r > 0;
        st->shared_blocks += r > 1;
        st->ref_sum += r;
    }
    st->spare_blocks = static_cast<int32_t>(bm->spare_count);
    st->num_seqs = static_cast<int32_t>(bm->seqs.size());
    st->cow_copies = bm->cow_copies;
    return PKV_OK;
}

int pkv_bm_refcount(pkv_bm* bm, int block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    std::lock_guard<std::mutex> lock(bm->mu);
    return bm->ref[block];
}

}  // extern "C"
