// pa_kv_manager.cpp -- host-side KV block manager (C ABI in include/pa.h).
//
// The bookkeeping side of the paged KV cache, as the pages describe it:
// fixed-size blocks handed out from a free list, ceil(tokens / block_size)
// per request, with an out-of-memory error when the list is empty
// (doramagic.ai vLLM manual, "KVCacheManager 缓存管理"); a per-request block
// table mapping logical to physical blocks ("vLLM 2026 推理引擎全解", §2.1;
// mjmagnets.cn vLLM tutorial, §2.2); blocks shared between requests with a
// common system prompt, or between the samples of one prompt, counted by
// reference and freed at zero ("vLLM 2026 推理引擎全解", §2.3; mjmagnets.cn
// vLLM tutorial, §2.1; doramagic.ai vLLM manual, "共享机制").
//
// Writing into a block that another sequence still references would change
// that sequence's history, so an append that lands in a shared block first
// takes a fresh block and reports a (source, destination) copy for
// pa_copy_blocks -- copy-on-write.
//
// Pure host code: no CUDA call.  Not thread-safe; one manager per caller.
#include <stdint.h>

#include <deque>
#include <new>
#include <vector>

#include "pa.h"

struct pa_kv_manager {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    int32_t max_blocks_per_seq = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> refcount;
    struct Seq {
        bool live = false;
        int32_t len = 0;
        std::vector<int32_t> blocks;
    };
    std::vector<Seq> seqs;
    std::vector<int32_t> free_ids;

    bool valid_seq(int32_t id) const {
        return id >= 0 && id < static_cast<int32_t>(seqs.size()) && seqs[id].live;
    }
    int32_t new_id() {
        if (!free_ids.empty()) {
            const int32_t id = free_ids.back();
            free_ids.pop_back();
            return id;
        }
        seqs.emplace_back();
        return static_cast<int32_t>(seqs.size()) - 1;
    }
    bool pop(int32_t *b) {
        if (free_list.empty()) return false;
        *b = free_list.front();
        free_list.pop_front();
        refcount[*b] = 1;
        return true;
    }
    void release(int32_t b) {
        if (--refcount[b] == 0) free_list.push_back(b);
    }
    int32_t blocks_for(int64_t tokens) const {
        return static_cast<int32_t>((tokens + block_size - 1) / block_size);
    }
};

namespace {

// splitmix64: a small, fully specified generator for the free-list shuffle.
uint64_t splitmix64(uint64_t *state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

}  // namespace

extern "C" {

pa_kv_manager *pa_kvm_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                             uint64_t shuffle_seed) {
    if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0) return nullptr;
    pa_kv_manager *m = new (std::nothrow) pa_kv_manager;
    if (!m) return nullptr;
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->max_blocks_per_seq = max_blocks_per_seq;
    m->refcount.assign(num_blocks, 0);
    std::vector<int32_t> order(num_blocks);
    for (int32_t i = 0; i < num_blocks; ++i) order[i] = i;
    if (shuffle_seed != 0) {  // Fisher-Yates
        uint64_t state = shuffle_seed;
        for (int32_t i = num_blocks - 1; i > 0; --i) {
            const int32_t j = static_cast<int32_t>(splitmix64(&state) % static_cast<uint64_t>(i + 1));
            const int32_t t = order[i];
            order[i] = order[j];
            order[j] = t;
        }
    }
    m->free_list.assign(order.begin(), order.end());
    return m;
}

void pa_kvm_destroy(pa_kv_manager *m) { delete m; }

int32_t pa_kvm_num_free_blocks(const pa_kv_manager *m) {
    return m ? static_cast<int32_t>(m->free_list.size()) : -1;
}

int32_t pa_kvm_refcount(const pa_kv_manager *m, int32_t block) {
    if (!m || block < 0 || block >= m->num_blocks) return -1;
    return m->refcount[block];
}

int pa_kvm_add_sequence(pa_kv_manager *m, int32_t num_tokens, int32_t parent,
                        int32_t shared_blocks, int32_t *seq_out) {
    if (!m || !seq_out) return PA_ERR_NULL;
    if (num_tokens < 0 || shared_blocks < 0) return PA_ERR_SHAPE;
    const int32_t need = m->blocks_for(num_tokens);
    if (need > m->max_blocks_per_seq) return PA_ERR_SHAPE;
    if (parent >= 0) {
        if (!m->valid_seq(parent)) return PA_ERR_SHAPE;
        // only whole, filled blocks of the parent can be shared this way
        if (static_cast<int64_t>(shared_blocks) * m->block_size > m->seqs[parent].len ||
            static_cast<int64_t>(shared_blocks) * m->block_size > num_tokens)
            return PA_ERR_SHAPE;
    } else if (shared_blocks != 0) {
        return PA_ERR_SHAPE;
    }
    if (need - shared_blocks > static_cast<int32_t>(m->free_list.size())) return PA_ERR_OUT_OF_BLOCKS;
    const int32_t id = m->new_id();
    pa_kv_manager::Seq &s = m->seqs[id];
    s.live = true;
    s.len = num_tokens;
    s.blocks.clear();
    for (int32_t b = 0; b < shared_blocks; ++b) {
        const int32_t blk = m->seqs[parent].blocks[b];
        ++m->refcount[blk];
        s.blocks.push_back(blk);
    }
    for (int32_t b = shared_blocks; b < need; ++b) {
        int32_t blk = -1;
        m->pop(&blk);
        s.blocks.push_back(blk);
    }
    *seq_out = id;
    return PA_OK;
}

int pa_kvm_fork(pa_kv_manager *m, int32_t parent, int32_t *seq_out) {
    if (!m || !seq_out) return PA_ERR_NULL;
    if (!m->valid_seq(parent)) return PA_ERR_SHAPE;
    const int32_t id = m->new_id();
    pa_kv_manager::Seq &p = m->seqs[parent];  // new_id may grow seqs: take refs after
    pa_kv_manager::Seq &s = m->seqs[id];
    s.live = true;
    s.len = p.len;
    s.blocks = p.blocks;
    for (int32_t blk : s.blocks) ++m->refcount[blk];
    *seq_out = id;
    return PA_OK;
}

int pa_kvm_append(pa_kv_manager *m, int32_t seq, int32_t *slot_out, int32_t *copy_src_out,
                  int32_t *copy_dst_out) {
    if (!m || !slot_out || !copy_src_out || !copy_dst_out) return PA_ERR_NULL;
    if (!m->valid_seq(seq)) return PA_ERR_SHAPE;
    pa_kv_manager::Seq &s = m->seqs[seq];
    const int32_t pos = s.len;
    const int32_t logical = pos / m->block_size;
    *copy_src_out = -1;
    *copy_dst_out = -1;
    if (logical >= static_cast<int32_t>(s.blocks.size())) {  // a new block starts
        if (logical >= m->max_blocks_per_seq) return PA_ERR_SHAPE;
        int32_t blk = -1;
        if (!m->pop(&blk)) return PA_ERR_OUT_OF_BLOCKS;
        s.blocks.push_back(blk);
    } else if (m->refcount[s.blocks[logical]] > 1) {  // copy-on-write
        int32_t blk = -1;
        if (!m->pop(&blk)) return PA_ERR_OUT_OF_BLOCKS;
        *copy_src_out = s.blocks[logical];
        *copy_dst_out = blk;
        m->release(s.blocks[logical]);
        s.blocks[logical] = blk;
    }
    *slot_out = s.blocks[logical] * m->block_size + pos % m->block_size;
    s.len = pos + 1;
    return PA_OK;
}

int pa_kvm_free(pa_kv_manager *m, int32_t seq) {
    if (!m) return PA_ERR_NULL;
    if (!m->valid_seq(seq)) return PA_ERR_SHAPE;
    pa_kv_manager::Seq &s = m->seqs[seq];
    for (int32_t blk : s.blocks) m->release(blk);
    s.blocks.clear();
    s.len = 0;
    s.live = false;
    m->free_ids.push_back(seq);
    return PA_OK;
}

int32_t pa_kvm_context_len(const pa_kv_manager *m, int32_t seq) {
    if (!m || !m->valid_seq(seq)) return -1;
    return m->seqs[seq].len;
}

int pa_kvm_slot(const pa_kv_manager *m, int32_t seq, int32_t token, int32_t *slot_out) {
    if (!m || !slot_out) return PA_ERR_NULL;
    if (!m->valid_seq(seq) || token < 0 || token >= m->seqs[seq].len) return PA_ERR_SHAPE;
    const pa_kv_manager::Seq &s = m->seqs[seq];
    *slot_out = s.blocks[token / m->block_size] * m->block_size + token % m->block_size;
    return PA_OK;
}

int pa_kvm_block_tables(const pa_kv_manager *m, const int32_t *seqs, int32_t num_seqs,
                        int32_t *tables_out, int32_t row_len, int32_t *context_lens_out) {
    if (!m || (num_seqs > 0 && (!seqs || !tables_out || !context_lens_out))) return PA_ERR_NULL;
    if (num_seqs < 0 || row_len <= 0) return PA_ERR_SHAPE;
    for (int32_t i = 0; i < num_seqs; ++i) {
        int32_t *row = tables_out + static_cast<int64_t>(i) * row_len;
        for (int32_t b = 0; b < row_len; ++b) row[b] = -1;
        if (seqs[i] < 0) {  // an empty batch row (padding)
            context_lens_out[i] = 0;
            continue;
        }
        if (!m->valid_seq(seqs[i])) return PA_ERR_SHAPE;
        const pa_kv_manager::Seq &s = m->seqs[seqs[i]];
        if (static_cast<int32_t>(s.blocks.size()) > row_len) return PA_ERR_SHAPE;
        for (size_t b = 0; b < s.blocks.size(); ++b) row[b] = s.blocks[b];
        context_lens_out[i] = s.len;
    }
    return PA_OK;
}

int pa_kvm_prefix_groups(const pa_kv_manager *m, const int32_t *seqs, int32_t num_seqs,
                         int32_t *group_start_out, int32_t *group_prefix_out, int32_t max_groups,
                         int32_t *num_groups_out) {
    if (!m || !num_groups_out || (num_seqs > 0 && (!seqs || !group_start_out || !group_prefix_out)))
        return PA_ERR_NULL;
    if (num_seqs < 0 || max_groups < 0) return PA_ERR_SHAPE;
    for (int32_t i = 0; i < num_seqs; ++i)
        if (seqs[i] >= 0 && !m->valid_seq(seqs[i])) return PA_ERR_SHAPE;
    // leading blocks of row i that are full (a padding row has none)
    auto full = [&](int32_t i) -> int32_t {
        return seqs[i] < 0 ? 0 : m->seqs[seqs[i]].len / m->block_size;
    };
    // leading full blocks rows i and j have in common
    auto common = [&](int32_t i, int32_t j) -> int32_t {
        const int32_t n = full(i) < full(j) ? full(i) : full(j);
        if (n == 0) return 0;   // also every padding row
        const std::vector<int32_t> &a = m->seqs[seqs[i]].blocks, &b = m->seqs[seqs[j]].blocks;
        int32_t c = 0;
        while (c < n && a[c] == b[c]) ++c;
        return c;
    };
    int32_t g = 0;
    bool open_unshared = false;  // the last group holds rows that share nothing
    auto emit = [&](int32_t start, int32_t prefix) -> bool {
        if (g >= max_groups) return false;
        group_start_out[g] = start;
        group_prefix_out[g] = prefix;
        ++g;
        return true;
    };
    int32_t i = 0;
    while (i < num_seqs) {
        // the group's prefix is what row i shares with row i + 1; the run goes
        // on while later rows share at least that much with row i
        const int32_t P = i + 1 < num_seqs ? common(i, i + 1) : 0;
        int32_t j = i + 1;
        if (P > 0)
            while (j < num_seqs && common(i, j) >= P) ++j;
        if (P > 0) {
            if (!emit(i, P)) return PA_ERR_SHAPE;
            open_unshared = false;
            i = j;
        } else {
            if (!open_unshared && !emit(i, 0)) return PA_ERR_SHAPE;
            open_unshared = true;
            ++i;
        }
    }
    if (num_seqs > 0) {
        if (max_groups < g || !group_start_out) return PA_ERR_SHAPE;
        group_start_out[g] = num_seqs;
    } else if (group_start_out) {
        group_start_out[0] = 0;
    }
    *num_groups_out = g;
    return PA_OK;
}

}  // extern "C"
