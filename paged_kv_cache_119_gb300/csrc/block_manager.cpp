// block_manager.cpp -- host-side KV block manager (C ABI in include/pa_block_manager.h).
//
// Reference counts, a first-in first-out free list, and the three primitives of
// "PagedAttention 完全拆解" section 三种原语：fork、append、free, with copy-on-write
// on append to a shared partially filled block (section 内存共享, Figure 8); and a
// CPU block pool for swapping whole sequence groups out and back in (section 调度与
// 抢占：内存不够时怎么办, 换出 (Swapping): all-or-nothing per group).
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pa_block_manager.h"

struct pa_block_manager {
    struct Seq {
        std::vector<int32_t> blocks;   // GPU block ids, or CPU block ids while swapped out
        int32_t tokens = 0;
        bool on_cpu = false;
    };
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> refs;
    std::unordered_map<int64_t, Seq> seqs;
    // CPU pool for swapped-out groups (empty until pa_bm_set_cpu_pool)
    std::deque<int32_t> cpu_free;
    std::vector<int32_t> cpu_refs;

    int64_t slot(const Seq& s, int32_t t) const
    {
        return (int64_t)s.blocks[t / block_size] * block_size + t % block_size;
    }
    int32_t take()
    {
        const int32_t b = free_list.front();
        free_list.pop_front();
        refs[b] = 1;
        return b;
    }
    void drop(int32_t b)
    {
        if (--refs[b] == 0)
            free_list.push_back(b);
    }
};

extern "C" {

pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t* alloc_order)
{
    if (num_blocks <= 0 || block_size <= 0)
        return nullptr;
    pa_block_manager* bm = new (std::nothrow) pa_block_manager;
    if (!bm)
        return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->refs.assign(num_blocks, 0);
    if (alloc_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            const int32_t b = alloc_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete bm;
                return nullptr;
            }
            seen[b] = 1;
            bm->free_list.push_back(b);
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i)
            bm->free_list.push_back(i);
    }
    return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, int32_t num_tokens, int64_t* slots_out)
{
    if (!bm || num_tokens < 0 || bm->seqs.count(seq_id))
        return PA_ERR_INVALID;
    const int32_t need = (num_tokens + bm->block_size - 1) / bm->block_size;
    if ((size_t)need > bm->free_list.size())
        return PA_ERR_INVALID;
    pa_block_manager::Seq s;
    for (int32_t i = 0; i < need; ++i)
        s.blocks.push_back(bm->take());
    s.tokens = num_tokens;
    if (slots_out)
        for (int32_t t = 0; t < num_tokens; ++t)
            slots_out[t] = bm->slot(s, t);
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

int pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id)
{
    if (!bm || parent_id == child_id || bm->seqs.count(child_id))
        return PA_ERR_INVALID;
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end() || it->second.on_cpu)
        return PA_ERR_INVALID;
    pa_block_manager::Seq child = it->second;
    for (int32_t b : child.blocks)
        ++bm->refs[b];
    bm->seqs.emplace(child_id, std::move(child));
    return PA_OK;
}

int pa_bm_append(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* slots_out,
                 int64_t* pairs_out, int32_t* num_pairs)
{
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots_out || !pairs_out)) || !num_pairs)
        return PA_ERR_INVALID;
    // Dry run: count the blocks this step takes, following the reference counts as
    // the earlier appends of the same step change them.
    std::unordered_set<int64_t> listed;
    std::unordered_map<int32_t, int32_t> released;   // block -> references dropped by CoW
    int32_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || it->second.on_cpu || !listed.insert(seq_ids[i]).second)
            return PA_ERR_INVALID;
        const auto& s = it->second;
        if (s.tokens % bm->block_size == 0) {
            ++need;                                   // the last block is full (or none yet)
        } else {
            const int32_t last = s.blocks.back();
            if (bm->refs[last] - released[last] > 1) {
                ++need;                               // shared partial block: copy-on-write
                ++released[last];
            }
        }
    }
    if ((size_t)need > bm->free_list.size())
        return PA_ERR_INVALID;
    int32_t pairs = 0;
    for (int32_t i = 0; i < n; ++i) {
        auto& s = bm->seqs[seq_ids[i]];
        if (s.tokens % bm->block_size == 0) {
            s.blocks.push_back(bm->take());
        } else {
            const int32_t last = s.blocks.back();
            if (bm->refs[last] > 1) {
                const int32_t fresh = bm->take();
                pairs_out[2 * pairs] = last;
                pairs_out[2 * pairs + 1] = fresh;
                ++pairs;
                bm->drop(last);
                s.blocks.back() = fresh;
            }
        }
        slots_out[i] = bm->slot(s, s.tokens);
        ++s.tokens;
    }
    *num_pairs = pairs;
    return PA_OK;
}

int pa_bm_free(pa_block_manager* bm, int64_t seq_id)
{
    if (!bm)
        return PA_ERR_INVALID;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end())
        return PA_ERR_INVALID;
    for (int32_t b : it->second.blocks) {
        if (!it->second.on_cpu)
            bm->drop(b);
        else if (--bm->cpu_refs[b] == 0)
            bm->cpu_free.push_back(b);
    }
    bm->seqs.erase(it);
    return PA_OK;
}

int pa_bm_block_tables(const pa_block_manager* bm, const int64_t* seq_ids, int32_t n,
                       int32_t* table_out, int32_t stride, int32_t* context_lens_out)
{
    if (!bm || n < 0 || stride <= 0 || (n > 0 && (!seq_ids || !table_out || !context_lens_out)))
        return PA_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || it->second.on_cpu || it->second.blocks.size() > (size_t)stride)
            return PA_ERR_INVALID;
    }
    for (int32_t i = 0; i < n; ++i) {
        const auto& s = bm->seqs.at(seq_ids[i]);
        int32_t* row = table_out + (int64_t)i * stride;
        for (int32_t j = 0; j < stride; ++j)
            row[j] = j < (int32_t)s.blocks.size() ? s.blocks[j] : -1;
        context_lens_out[i] = s.tokens;
    }
    return PA_OK;
}

int pa_bm_set_cpu_pool(pa_block_manager* bm, int32_t num_cpu_blocks)
{
    if (!bm || num_cpu_blocks <= 0 || !bm->cpu_refs.empty())
        return PA_ERR_INVALID;
    bm->cpu_refs.assign(num_cpu_blocks, 0);
    for (int32_t i = 0; i < num_cpu_blocks; ++i)
        bm->cpu_free.push_back(i);
    return PA_OK;
}

namespace {

// Moves a group's blocks between the pools: every distinct block of the listed
// sequences (first appearance order) gets one block of the other pool, a (from, to)
// pair is recorded, and the group's references move across.  to_cpu: GPU -> CPU.
int swap_group(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs_out,
               int32_t max_pairs, int32_t* num_pairs, bool to_cpu)
{
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !pairs_out)) || !num_pairs || bm->cpu_refs.empty())
        return PA_ERR_INVALID;
    std::unordered_set<int64_t> listed;
    std::vector<int32_t> order;                          // distinct source blocks
    std::unordered_map<int32_t, int32_t> uses;           // source block -> group references
    for (int32_t i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end() || it->second.on_cpu != !to_cpu || !listed.insert(seq_ids[i]).second)
            return PA_ERR_INVALID;
        for (int32_t b : it->second.blocks)
            if (uses[b]++ == 0)
                order.push_back(b);
    }
    std::deque<int32_t>& dst_free = to_cpu ? bm->cpu_free : bm->free_list;
    if (order.size() > dst_free.size() || (int64_t)order.size() > max_pairs)
        return PA_ERR_INVALID;                           // all or nothing
    std::vector<int32_t>& src_refs = to_cpu ? bm->refs : bm->cpu_refs;
    std::vector<int32_t>& dst_refs = to_cpu ? bm->cpu_refs : bm->refs;
    std::deque<int32_t>& src_free = to_cpu ? bm->free_list : bm->cpu_free;
    std::unordered_map<int32_t, int32_t> moved;          // source block -> destination block
    int32_t k = 0;
    for (int32_t b : order) {
        const int32_t d = dst_free.front();
        dst_free.pop_front();
        dst_refs[d] = uses[b];
        src_refs[b] -= uses[b];
        if (src_refs[b] == 0)
            src_free.push_back(b);
        moved[b] = d;
        pairs_out[2 * k] = b;
        pairs_out[2 * k + 1] = d;
        ++k;
    }
    for (int32_t i = 0; i < n; ++i) {
        auto& s = bm->seqs[seq_ids[i]];
        for (int32_t& b : s.blocks)
            b = moved[b];
        s.on_cpu = to_cpu;
    }
    *num_pairs = k;
    return PA_OK;
}

}  // namespace

int pa_bm_swap_out(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs_out,
                   int32_t max_pairs, int32_t* num_pairs)
{
    return swap_group(bm, seq_ids, n, pairs_out, max_pairs, num_pairs, true);
}

int pa_bm_swap_in(pa_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* pairs_out,
                  int32_t max_pairs, int32_t* num_pairs)
{
    return swap_group(bm, seq_ids, n, pairs_out, max_pairs, num_pairs, false);
}

int32_t pa_bm_num_free_cpu_blocks(const pa_block_manager* bm)
{
    return bm ? (int32_t)bm->cpu_free.size() : -1;
}

int32_t pa_bm_cpu_ref_count(const pa_block_manager* bm, int32_t block)
{
    if (!bm || block < 0 || block >= (int32_t)bm->cpu_refs.size())
        return -1;
    return bm->cpu_refs[block];
}

int32_t pa_bm_is_swapped(const pa_block_manager* bm, int64_t seq_id)
{
    if (!bm)
        return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : (it->second.on_cpu ? 1 : 0);
}

int32_t pa_bm_num_free_blocks(const pa_block_manager* bm)
{
    return bm ? (int32_t)bm->free_list.size() : -1;
}

int32_t pa_bm_ref_count(const pa_block_manager* bm, int32_t block)
{
    if (!bm || block < 0 || block >= bm->num_blocks)
        return -1;
    return bm->refs[block];
}

int32_t pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq_id)
{
    if (!bm)
        return -1;
    auto it = bm->seqs.find(seq_id);
    return it == bm->seqs.end() ? -1 : it->second.tokens;
}

}  // extern "C"
