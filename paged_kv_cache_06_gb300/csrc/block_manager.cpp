// Host-side block manager for the paged KV pool.
//
// "Paged attention" (danielfleming.xyz), section "What changed": a request
// takes its blocks off a free list when it is admitted and returns them when
// it finishes, and nothing is copied; reserve on admit takes every block the request could ever need
// (prompt + full token budget) or admits nothing.
// "SLM paged attention" (aicassindra.com), sections "The architecture" and
// "End-to-end flow": O(1) pop/push free list; without a reservation a
// sequence grows one block at a time when its current block fills; shared
// prefix blocks carry a reference count, are freed only when it reaches zero,
// and are copied on the first write into them.
// "PagedAttention" (deepconcepts.dev), section "So what does block_size
// trade?": blocks are shared whole, so a prefix shares floor(tokens / bs)
// blocks and the partial remainder stays private.
//
// Plain host memory; callers serialise access.
#include <algorithm>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "paged_kv.h"

namespace {

struct Sequence {
    std::vector<int32_t> table;     // physical ids of logical blocks 0..n-1
    std::vector<int32_t> reserved;  // private blocks held for later (reserve on admit)
    int64_t len = 0;                // tokens written
};

struct Prefix {
    std::vector<int32_t> blocks;
    bool live = false;
};

}  // namespace

struct pkv_block_manager {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    int32_t max_blocks_per_row = 0;
    std::vector<int32_t> free_list;  // LIFO stack: pop/push at the back, O(1)
    std::vector<int32_t> refcount;   // per physical block, 0 = on the free list
    std::unordered_map<int64_t, Sequence> seqs;
    std::vector<Prefix> prefixes;    // prefix id = index
    int64_t cow_copies = 0;
    int64_t pops_until_failure = -1; // fault injection; -1 = off

    bool can_pop(int64_t n) const {
        if (n < 0) return false;
        if ((int64_t)free_list.size() < n) return false;
        if (pops_until_failure >= 0 && pops_until_failure < n) return false;
        return true;
    }
    int32_t pop() {  // caller checked can_pop
        const int32_t id = free_list.back();
        free_list.pop_back();
        refcount[id] = 1;
        if (pops_until_failure > 0) --pops_until_failure;
        return id;
    }
    void unref(int32_t id) {
        if (--refcount[id] == 0) free_list.push_back(id);
    }
};

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

extern "C" {

int pkv_bm_create(int num_blocks, int block_size, int max_blocks_per_row,
                  pkv_block_manager** out) {
    if (!out || num_blocks < 0 || block_size <= 0 || max_blocks_per_row <= 0)
        return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_block_manager* bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return PKV_ERR_INVALID_ARG;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->max_blocks_per_row = max_blocks_per_row;
    bm->refcount.assign((size_t)num_blocks, 0);
    bm->free_list.reserve((size_t)num_blocks);
    // Lowest ids on top of the stack first.
    for (int32_t i = num_blocks - 1; i >= 0; --i) bm->free_list.push_back(i);
    *out = bm;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int pkv_bm_register_prefix(pkv_block_manager* bm, int prefix_tokens, int32_t* prefix_id_out,
                           int32_t* block_ids_out) {
    if (!bm || !prefix_id_out || prefix_tokens < 0) return PKV_ERR_INVALID_ARG;
    const int64_t n = prefix_tokens / bm->block_size;  // whole blocks only
    if (n > bm->max_blocks_per_row) return PKV_ERR_INVALID_ARG;
    if (!bm->can_pop(n)) return PKV_ERR_NO_BLOCKS;
    Prefix p;
    p.live = true;
    for (int64_t i = 0; i < n; ++i) p.blocks.push_back(bm->pop());
    if (block_ids_out)
        std::copy(p.blocks.begin(), p.blocks.end(), block_ids_out);
    bm->prefixes.push_back(std::move(p));
    *prefix_id_out = (int32_t)(bm->prefixes.size() - 1);
    return PKV_OK;
}

int pkv_bm_release_prefix(pkv_block_manager* bm, int32_t prefix_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    if (prefix_id < 0 || prefix_id >= (int32_t)bm->prefixes.size() || !bm->prefixes[prefix_id].live)
        return PKV_ERR_NOT_FOUND;
    Prefix& p = bm->prefixes[prefix_id];
    for (int32_t id : p.blocks) bm->unref(id);
    p.live = false;
    return PKV_OK;
}

int pkv_bm_admit(pkv_block_manager* bm, int64_t seq_id, int prompt_len, int max_new_tokens,
                 int32_t prefix_id, int reserve) {
    if (!bm || prompt_len < 0 || max_new_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (bm->seqs.count(seq_id)) return PKV_ERR_STATE;
    const int64_t bs = bm->block_size;
    const int64_t total_blocks = ceil_div((int64_t)prompt_len + max_new_tokens, bs);
    // A reservation must fit the table; without one only the prompt must.
    if ((reserve ? total_blocks : ceil_div(prompt_len, bs)) > bm->max_blocks_per_row)
        return PKV_ERR_INVALID_ARG;
    const Prefix* pre = nullptr;
    if (prefix_id >= 0) {
        if (prefix_id >= (int32_t)bm->prefixes.size() || !bm->prefixes[prefix_id].live)
            return PKV_ERR_NOT_FOUND;
        pre = &bm->prefixes[prefix_id];
    }
    const int64_t prompt_blocks = ceil_div(prompt_len, bs);
    const int64_t shared_used = pre ? std::min<int64_t>((int64_t)pre->blocks.size(), prompt_blocks) : 0;
    // The first write lands in a shared block when the prompt ends inside it.
    const bool will_cow = max_new_tokens > 0 && shared_used > 0 && prompt_len < shared_used * bs;
    const int64_t prompt_private = prompt_blocks - shared_used;
    const int64_t later = reserve ? (total_blocks - prompt_blocks) + (will_cow ? 1 : 0) : 0;
    if (!bm->can_pop(prompt_private + later)) return PKV_ERR_NO_BLOCKS;

    Sequence s;
    s.len = prompt_len;
    for (int64_t i = 0; i < shared_used; ++i) {
        const int32_t id = pre->blocks[(size_t)i];
        ++bm->refcount[id];
        s.table.push_back(id);
    }
    for (int64_t i = 0; i < prompt_private; ++i) s.table.push_back(bm->pop());
    for (int64_t i = 0; i < later; ++i) s.reserved.push_back(bm->pop());
    bm->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

int pkv_bm_append_slot(pkv_block_manager* bm, int64_t seq_id, int32_t* position_out,
                       int32_t* cow_src_out, int32_t* cow_dst_out) {
    if (!bm || !position_out) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_NOT_FOUND;
    Sequence& s = it->second;
    const int64_t pos = s.len;
    const int64_t lb = pos / bm->block_size;
    if (lb >= bm->max_blocks_per_row || pos > INT32_MAX) return PKV_ERR_STATE;
    int32_t src = -1, dst = -1;
    auto take = [&](int32_t* id) -> bool {
        if (!s.reserved.empty()) {
            *id = s.reserved.back();
            s.reserved.pop_back();
            return true;
        }
        if (!bm->can_pop(1)) return false;
        *id = bm->pop();
        return true;
    };
    if (lb == (int64_t)s.table.size()) {
        int32_t id;
        if (!take(&id)) return PKV_ERR_NO_BLOCKS;
        s.table.push_back(id);
    } else if (bm->refcount[s.table[(size_t)lb]] > 1) {
        // Copy on write: the writer gets a private block, readers keep theirs.
        if (!take(&dst)) return PKV_ERR_NO_BLOCKS;
        src = s.table[(size_t)lb];
        bm->unref(src);
        s.table[(size_t)lb] = dst;
        ++bm->cow_copies;
    }
    s.len = pos + 1;
    *position_out = (int32_t)pos;
    if (cow_src_out) *cow_src_out = src;
    if (cow_dst_out) *cow_dst_out = dst;
    return PKV_OK;
}

int pkv_bm_free(pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_NOT_FOUND;
    for (int32_t id : it->second.table) bm->unref(id);
    for (int32_t id : it->second.reserved) bm->unref(id);
    bm->seqs.erase(it);
    return PKV_OK;
}

int pkv_bm_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* row_out,
                 int32_t* seq_len_out) {
    if (!bm || !row_out) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_NOT_FOUND;
    const Sequence& s = it->second;
    for (int32_t i = 0; i < bm->max_blocks_per_row; ++i)
        row_out[i] = i < (int32_t)s.table.size() ? s.table[(size_t)i] : -1;
    if (seq_len_out) *seq_len_out = (int32_t)s.len;
    return PKV_OK;
}

int pkv_bm_stats(const pkv_block_manager* bm, pkv_bm_stats_t* out) {
    if (!bm || !out) return PKV_ERR_INVALID_ARG;
    pkv_bm_stats_t st{};
    st.num_blocks = bm->num_blocks;
    st.free_blocks = (int32_t)bm->free_list.size();
    st.used_blocks = bm->num_blocks - st.free_blocks;
    for (int32_t c : bm->refcount) st.shared_blocks += c > 1;
    st.sequences = (int32_t)bm->seqs.size();
    for (const Prefix& p : bm->prefixes) st.prefixes += p.live;
    for (const auto& kv : bm->seqs) {
        const Sequence& s = kv.second;
        st.live_tokens += s.len;
        const int64_t cap = (int64_t)s.table.size() * bm->block_size;
        st.reserved_slots += (int64_t)s.reserved.size() * bm->block_size + (cap > s.len ? cap - s.len : 0);
    }
    st.cow_copies = bm->cow_copies;
    *out = st;
    return PKV_OK;
}

int pkv_bm_refcount(const pkv_block_manager* bm, int32_t block_id, int32_t* count_out) {
    if (!bm || !count_out) return PKV_ERR_INVALID_ARG;
    if (block_id < 0 || block_id >= bm->num_blocks) return PKV_ERR_NOT_FOUND;
    *count_out = bm->refcount[(size_t)block_id];
    return PKV_OK;
}

int pkv_bm_inject_pop_failure(pkv_block_manager* bm, int pops) {
    if (!bm || pops < -1) return PKV_ERR_INVALID_ARG;
    bm->pops_until_failure = pops;
    return PKV_OK;
}

}  // extern "C"
