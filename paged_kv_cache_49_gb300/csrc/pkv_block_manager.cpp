// Host block manager: free list, reference counts, page-rounded admission
// (full reservation, or incremental with a watermark), prefix groups, fork,
// copy-on-write, preemption by recompute and a prefix-cache index.
//
// Policy sources: cs2680 Lecture 10, §10.3 (block pool and per-sequence block
// table, growth by one entry), §10.4 (reference-counted sharing, copy on
// divergence) and §10.5 (on-demand pages run out: refuse arrivals or preempt,
// keep a watermark of free pages, recompute a preempted sequence); "KV cache
// systems", copy-on-write paragraph (the first writer of a shared block
// copies it), prefix-hit paragraph (a block is reusable iff all its tokens
// and all earlier blocks match) and eviction paragraph (pinned blocks are
// never evicted; leaves go first); "Reserve the page a request has not
// written yet" (reserve ceil((prompt + output) / 16) pages at admission;
// reserve and admit as one serialised decision; charge shared prefix pages
// once; freeing changes ownership, not device memory).
//
// The prefix index keys a block by (the block holding the preceding tokens,
// its own tokens): because a cached block is evicted only once no cached
// block extends it, that parent id always names exactly one token prefix, so
// the key identifies the whole prefix without storing it.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/pkv.h"

namespace {

struct Sequence {
    std::vector<int32_t> table;
    int64_t ctx = 0;
    int64_t max_len = 0;
    int group = -1;
    bool running = true;
};

struct Group {
    std::vector<int32_t> pages;
    int prefix_len = 0;
    int members = 0;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Key of a cached block: its parent block (-1 for the first) then its tokens.
struct KeyHash {
    size_t operator()(const std::vector<int32_t>& k) const {
        uint64_t h = 1469598103934665603ull;  // FNV-1a, 64-bit
        for (int32_t v : k) {
            uint32_t u = static_cast<uint32_t>(v);
            for (int i = 0; i < 4; ++i) {
                h ^= (u >> (8 * i)) & 0xffu;
                h *= 1099511628211ull;
            }
        }
        return static_cast<size_t>(h);
    }
};

}  // namespace

struct pkv_bm {
    int num_blocks = 0;
    int block_tokens = 16;
    bool incremental = false;
    int watermark = 0;
    bool prefix_cache = false;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> ref;
    std::vector<std::vector<int32_t>> spares;  // per block: pages reserved for its CoW
    std::unordered_map<int, Sequence> seqs;
    std::unordered_map<int, Group> groups;
    int next_id = 0;
    int64_t cow_copies = 0;
    int64_t spare_count = 0;
    // prefix cache
    std::unordered_map<std::vector<int32_t>, int32_t, KeyHash> index;
    std::vector<std::vector<int32_t>> key;  // empty: block not indexed
    std::vector<int32_t> parent, children;
    std::vector<int64_t> last_use;
    std::set<std::pair<int64_t, int32_t>> evictable;  // indexed, ref 0, no indexed child
    int64_t clock = 0;
    int32_t cached = 0, cached_idle = 0;
    int64_t cache_hits = 0, evictions = 0;
    std::mutex mu;

    bool indexed(int32_t b) const { return !key[b].empty(); }
    int available() const { return static_cast<int>(free_stack.size()) + cached_idle; }

    // A free page if there is one, else the least recently released cached
    // leaf (callers have checked available()).
    int32_t alloc() {
        if (!free_stack.empty()) {
            int32_t b = free_stack.back();
            free_stack.pop_back();
            return b;
        }
        const int32_t b = evictable.begin()->second;
        evictable.erase(evictable.begin());
        index.erase(key[b]);
        key[b].clear();
        const int32_t p = parent[b];
        parent[b] = -1;
        if (p >= 0 && --children[p] == 0 && ref[p] == 0) evictable.emplace(last_use[p], p);
        cached -= 1;
        cached_idle -= 1;
        evictions += 1;
        return b;
    }

    // One more reference to a cached block that may be idle.
    void acquire_cached(int32_t b) {
        if (ref[b] == 0) {
            cached_idle -= 1;
            if (children[b] == 0) evictable.erase({last_use[b], b});
        }
        ref[b] += 1;
    }

    void release(const std::vector<int32_t>& table) {
        for (int32_t b : table) {
            ref[b] -= 1;
            std::vector<int32_t>& sp = spares[b];
            if (!sp.empty() && static_cast<int64_t>(sp.size()) > ref[b] - 1) {
                free_stack.push_back(sp.back());
                sp.pop_back();
                spare_count -= 1;
            }
            if (ref[b] == 0) {
                if (indexed(b)) {
                    last_use[b] = ++clock;
                    cached_idle += 1;
                    if (children[b] == 0) evictable.emplace(last_use[b], b);
                } else {
                    free_stack.push_back(b);
                }
            }
        }
    }

    void leave_group(Sequence& s) {
        if (s.group >= 0) {
            auto g = groups.find(s.group);
            if (g != groups.end() && --g->second.members == 0) groups.erase(g);
            s.group = -1;
        }
    }

    Sequence* running_seq(int id) {
        auto it = seqs.find(id);
        return it == seqs.end() || !it->second.running ? nullptr : &it->second;
    }
};

extern "C" {

pkv_bm* pkv_bm_create_ex(int num_blocks, int block_tokens, const int32_t* free_order,
                         int incremental, int watermark_blocks, int prefix_cache) {
    if (num_blocks <= 0 || watermark_blocks < 0 ||
        (block_tokens != 8 && block_tokens != 16 && block_tokens != 32 && block_tokens != 64))
        return nullptr;
    auto* bm = new pkv_bm();
    bm->num_blocks = num_blocks;
    bm->block_tokens = block_tokens;
    bm->incremental = incremental != 0;
    bm->watermark = watermark_blocks;
    bm->prefix_cache = prefix_cache != 0;
    bm->ref.assign(num_blocks, 0);
    bm->spares.assign(num_blocks, {});
    bm->key.assign(num_blocks, {});
    bm->parent.assign(num_blocks, -1);
    bm->children.assign(num_blocks, 0);
    bm->last_use.assign(num_blocks, 0);
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

pkv_bm* pkv_bm_create(int num_blocks, int block_tokens, const int32_t* free_order) {
    return pkv_bm_create_ex(num_blocks, block_tokens, free_order, 0, 0, 0);
}

void pkv_bm_destroy(pkv_bm* bm) { delete bm; }

static pkv_status admit_locked(pkv_bm* bm, const int32_t* tokens, int prompt_len, int max_new,
                               int group, int prefix_len, int* seq_id, int* reused_blocks) {
    if (prompt_len < 0 || max_new < 0 || static_cast<int64_t>(prompt_len) + max_new <= 0)
        return PKV_EINVAL;
    if (tokens && (!bm->prefix_cache || group >= 0)) return PKV_EINVAL;
    const int b = bm->block_tokens;
    const int64_t total =
        ceil_div(bm->incremental ? prompt_len : static_cast<int64_t>(prompt_len) + max_new, b);
    const std::vector<int32_t>* shared = nullptr;
    Group* existing = nullptr;
    bool new_group = false;
    if (group >= 0) {
        if (prefix_len < 0 || prefix_len > prompt_len) return PKV_EINVAL;
        auto it = bm->groups.find(group);
        if (it != bm->groups.end()) {
            if (it->second.prefix_len != prefix_len) return PKV_EINVAL;
            existing = &it->second;
            shared = &existing->pages;
        } else {
            new_group = true;
        }
    }
    // Prefix-cache hits: complete prompt blocks, from the first, up to the first miss.
    std::vector<int32_t> hits;
    std::vector<int32_t> k(1 + b);
    int64_t idle_hits = 0;
    if (tokens) {
        int32_t prev = -1;
        for (int i = 0; i < prompt_len / b; ++i) {
            k[0] = prev;
            std::memcpy(k.data() + 1, tokens + static_cast<int64_t>(i) * b, sizeof(int32_t) * b);
            auto it = bm->index.find(k);
            if (it == bm->index.end()) break;
            prev = it->second;
            hits.push_back(prev);
            idle_hits += bm->ref[prev] == 0;
        }
    }
    const int64_t n_shared = tokens ? static_cast<int64_t>(hits.size())
                                    : (shared ? static_cast<int64_t>(shared->size()) : 0);
    const int64_t need = total - n_shared;
    if (need + bm->watermark > bm->available() - idle_hits) return PKV_ENOMEM;

    Sequence seq;
    seq.ctx = prompt_len;
    seq.max_len = static_cast<int64_t>(prompt_len) + max_new;
    seq.group = group;
    seq.table.reserve(total);
    if (new_group) {
        Group g;
        g.prefix_len = prefix_len;
        for (int64_t i = 0; i < prefix_len / b; ++i) g.pages.push_back(bm->alloc());
        existing = &(bm->groups[group] = std::move(g));
        shared = &existing->pages;
    }
    for (int32_t h : hits) bm->acquire_cached(h);
    if (tokens) seq.table = hits;
    else if (shared) seq.table.assign(shared->begin(), shared->end());
    while (static_cast<int64_t>(seq.table.size()) < total) seq.table.push_back(bm->alloc());
    for (size_t i = tokens ? hits.size() : 0; i < seq.table.size(); ++i) bm->ref[seq.table[i]] += 1;
    if (existing) existing->members += 1;
    if (tokens) {
        for (int64_t i = static_cast<int64_t>(hits.size()); i < prompt_len / b; ++i) {
            const int32_t blk = seq.table[i];
            const int32_t par = i > 0 ? seq.table[i - 1] : -1;
            k[0] = par;
            std::memcpy(k.data() + 1, tokens + i * b, sizeof(int32_t) * b);
            bm->index.emplace(k, blk);
            bm->key[blk] = k;
            bm->parent[blk] = par;
            bm->children[blk] = 0;
            if (par >= 0) bm->children[par] += 1;
            bm->cached += 1;
        }
        bm->cache_hits += static_cast<int64_t>(hits.size());
    }
    const int id = bm->next_id++;
    bm->seqs.emplace(id, std::move(seq));
    *seq_id = id;
    if (reused_blocks) *reused_blocks = static_cast<int>(hits.size());
    return PKV_OK;
}

pkv_status pkv_bm_admit(pkv_bm* bm, int prompt_len, int max_new, int group, int prefix_len,
                        int* seq_id) {
    if (!bm || !seq_id) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    return admit_locked(bm, nullptr, prompt_len, max_new, group, prefix_len, seq_id, nullptr);
}

pkv_status pkv_bm_admit_tokens(pkv_bm* bm, const int32_t* tokens, int prompt_len, int max_new,
                               int* seq_id, int* reused_blocks) {
    if (!bm || !seq_id || !tokens) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    return admit_locked(bm, tokens, prompt_len, max_new, -1, 0, seq_id, reused_blocks);
}

pkv_status pkv_bm_fork(pkv_bm* bm, int parent_seq, int n, int32_t* child_ids) {
    if (!bm || n < 0 || (n > 0 && !child_ids)) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    const Sequence* p = bm->running_seq(parent_seq);
    if (!p) return PKV_EINVAL;
    const Sequence parent = *p;  // copy: emplacing children may rehash
    const int64_t written = ceil_div(parent.ctx, bm->block_tokens);
    const bool partial = parent.ctx % bm->block_tokens != 0 && !bm->incremental;
    const int64_t per_child = bm->incremental
        ? 0 : (static_cast<int64_t>(parent.table.size()) - written) + (partial ? 1 : 0);
    if (static_cast<int64_t>(n) * per_child > bm->available()) return PKV_ENOMEM;
    for (int i = 0; i < n; ++i) {
        Sequence child;
        child.ctx = parent.ctx;
        child.max_len = parent.max_len;
        child.group = parent.group;
        child.table.assign(parent.table.begin(), parent.table.begin() + written);
        while (child.table.size() < parent.table.size()) child.table.push_back(bm->alloc());
        for (int32_t b : child.table) bm->ref[b] += 1;
        if (partial) {
            bm->spares[parent.table[written - 1]].push_back(bm->alloc());
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
    const int bt = bm->block_tokens;
    std::vector<Sequence*> batch(n);
    {
        std::vector<int32_t> sorted(seq_ids, seq_ids + n);
        std::sort(sorted.begin(), sorted.end());
        if (std::adjacent_find(sorted.begin(), sorted.end()) != sorted.end()) return PKV_EINVAL;
    }
    for (int i = 0; i < n; ++i)
        if (!(batch[i] = bm->running_seq(seq_ids[i]))) return PKV_EINVAL;
    // Count the pages the step takes (new blocks, copies without a spare)
    // before changing anything.
    {
        int64_t need = 0;
        std::unordered_map<int32_t, int64_t> ref_left, spare_left;
        for (Sequence* s : batch) {
            const int64_t lb = s->ctx / bt;
            if (lb >= static_cast<int64_t>(s->table.size())) {
                if (!bm->incremental) return PKV_ENOSPC;
                need += 1;
                continue;
            }
            const int32_t b = s->table[lb];
            auto r = ref_left.emplace(b, bm->ref[b]).first;
            auto sp = spare_left.emplace(b, bm->spares[b].size()).first;
            if (r->second > 1) {
                r->second -= 1;
                if (sp->second > 0) sp->second -= 1;
                else if (bm->incremental) need += 1;
                else return PKV_ESTATE;
            }
        }
        if (need > bm->available()) return PKV_ENOMEM;
    }
    int pairs = 0;
    for (int i = 0; i < n; ++i) {
        Sequence* s = batch[i];
        const int64_t lb = s->ctx / bt;
        if (lb >= static_cast<int64_t>(s->table.size())) {
            const int32_t fresh = bm->alloc();
            bm->ref[fresh] = 1;
            s->table.push_back(fresh);
        }
        int32_t b = s->table[lb];
        if (bm->ref[b] > 1) {
            std::vector<int32_t>& sp = bm->spares[b];
            int32_t dst;
            if (!sp.empty()) {
                dst = sp.back();
                sp.pop_back();
                bm->spare_count -= 1;
            } else {
                dst = bm->alloc();
            }
            bm->ref[b] -= 1;
            bm->ref[dst] = 1;
            s->table[lb] = dst;
            cow_pairs_out[2 * pairs] = b;
            cow_pairs_out[2 * pairs + 1] = dst;
            ++pairs;
            bm->cow_copies += 1;
            b = dst;
        }
        slot_mapping_out[i] = static_cast<int64_t>(b) * bt + s->ctx % bt;
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
    if (s.running) {
        bm->release(s.table);
        bm->leave_group(s);
    }
    return PKV_OK;
}

pkv_status pkv_bm_preempt(pkv_bm* bm, int seq_id, int* released_blocks) {
    if (!bm) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    Sequence* s = bm->running_seq(seq_id);
    if (!s) return PKV_EINVAL;
    const int n = static_cast<int>(s->table.size());
    bm->release(s->table);
    bm->leave_group(*s);
    s->table.clear();
    s->running = false;
    if (released_blocks) *released_blocks = n;
    return PKV_OK;
}

pkv_status pkv_bm_resume(pkv_bm* bm, int seq_id) {
    if (!bm) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end() || it->second.running) return PKV_EINVAL;
    Sequence& s = it->second;
    const int64_t total = ceil_div(bm->incremental ? s.ctx : s.max_len, bm->block_tokens);
    if (total + bm->watermark > bm->available()) return PKV_ENOMEM;
    s.table.clear();
    for (int64_t i = 0; i < total; ++i) {
        const int32_t b = bm->alloc();
        bm->ref[b] = 1;
        s.table.push_back(b);
    }
    s.running = true;
    return PKV_OK;
}

pkv_status pkv_bm_slots(pkv_bm* bm, int seq_id, int first, int n, int64_t* slots_out) {
    if (!bm || first < 0 || n < 0 || (n > 0 && !slots_out)) return PKV_EINVAL;
    std::lock_guard<std::mutex> lock(bm->mu);
    const Sequence* s = bm->running_seq(seq_id);
    const int64_t bt = bm->block_tokens;
    if (!s || static_cast<int64_t>(first) + n > static_cast<int64_t>(s->table.size()) * bt)
        return PKV_EINVAL;
    for (int i = 0; i < n; ++i) {
        const int64_t pos = static_cast<int64_t>(first) + i;
        slots_out[i] = static_cast<int64_t>(s->table[pos / bt]) * bt + pos % bt;
    }
    return PKV_OK;
}

int pkv_bm_newest_running(pkv_bm* bm) {
    if (!bm) return -1;
    std::lock_guard<std::mutex> lock(bm->mu);
    int newest = -1;
    for (const auto& kv : bm->seqs)
        if (kv.second.running) newest = std::max(newest, kv.first);
    return newest;
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
        const Sequence* s = bm->running_seq(seq_ids[i]);
        if (!s) return PKV_EINVAL;
        if (static_cast<int>(s->table.size()) > width) return PKV_ERANGE;
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
    st->free_blocks = static_cast<int32_t>(bm->free_stack.size());
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
    st->cached_blocks = bm->cached;
    st->cached_idle_blocks = bm->cached_idle;
    st->preempted_seqs = 0;
    for (const auto& kv : bm->seqs) st->preempted_seqs += !kv.second.running;
    st->available_blocks = bm->available();
    st->cache_hits = bm->cache_hits;
    st->evictions = bm->evictions;
    return PKV_OK;
}

int pkv_bm_refcount(pkv_bm* bm, int block) {
    if (!bm || block < 0 || block >= bm->num_blocks) return -1;
    std::lock_guard<std::mutex> lock(bm->mu);
    return bm->ref[block];
}

}  // extern "C"
