// Host-side KV block pool and RoPE table (no GPU work).
//
// The pool is the free-block stack + per-sequence block tables of mini-infer's
// Paged KV Cache (mini-infer README, "项目概述" and "架构设计": KVCacheManager =
// BlockTable + FreeBlockPool), allocating ceil(tokens / block) blocks on
// demand like the allocate sketch of the nxmr.cn article (§2.1
// "KV缓存的内存革命"), but fixed in size: an allocation that does not fit fails
// and leaves the pool as it was.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "mi.h"

struct mi_kv_pool {
    int32_t num_blocks = 0;
    int32_t block_size = 16;
    int32_t max_blocks_per_seq = 0;
    std::vector<int32_t> free_stack;            // back() is the next block handed out
    std::vector<std::vector<int32_t>> tables;   // per sequence id
    std::vector<int32_t> tokens;                // per sequence id
    std::vector<uint8_t> live;                  // per sequence id: resident (holds its table)
    std::vector<uint8_t> swapped;               // per sequence id: blocks swapped out, tokens kept
    std::vector<int64_t> last_use;              // per sequence id: clock of the last use
    int64_t clock = 0;                          // LRU use counter

    void use(int32_t seq) { last_use[(size_t)seq] = clock; }
};

extern "C" const char* mi_status_string(mi_status s) {
    switch (s) {
        case MI_OK: return "ok";
        case MI_ERR_INVALID_ARG: return "invalid argument";
        case MI_ERR_OUT_OF_BLOCKS: return "out of KV blocks";
        case MI_ERR_UNKNOWN_SEQ: return "unknown sequence";
        case MI_ERR_UNSUPPORTED: return "unsupported shape";
        case MI_ERR_CUDA: return "CUDA error";
        case MI_ERR_DEVICE_BOUNDS: return "device-side bounds error";
        case MI_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

extern "C" mi_status mi_kv_pool_create(int32_t num_blocks, int32_t block_size, int32_t max_seqs,
                                       int32_t max_blocks_per_seq,
                                       const int32_t* initial_free_order, mi_kv_pool** out) {
    if (!out) return MI_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_blocks < 1 || max_seqs < 1 || max_blocks_per_seq < 1) return MI_ERR_INVALID_ARG;
    if (block_size != 16) return MI_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * block_size > INT32_MAX) return MI_ERR_INVALID_ARG;
    if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return MI_ERR_INVALID_ARG;
    mi_kv_pool* p = new (std::nothrow) mi_kv_pool();
    if (!p) return MI_ERR_INVALID_ARG;
    try {
        p->num_blocks = num_blocks;
        p->block_size = block_size;
        p->max_blocks_per_seq = max_blocks_per_seq;
        p->free_stack.resize((size_t)num_blocks);
        if (initial_free_order) {
            std::vector<uint8_t> seen((size_t)num_blocks, 0);
            for (int32_t i = 0; i < num_blocks; ++i) {
                const int32_t b = initial_free_order[i];
                if (b < 0 || b >= num_blocks || seen[(size_t)b]) { delete p; return MI_ERR_INVALID_ARG; }
                seen[(size_t)b] = 1;
                p->free_stack[(size_t)(num_blocks - 1 - i)] = b;
            }
        } else {
            for (int32_t i = 0; i < num_blocks; ++i) p->free_stack[(size_t)(num_blocks - 1 - i)] = i;
        }
        p->tables.resize((size_t)max_seqs);
        p->tokens.assign((size_t)max_seqs, 0);
        p->live.assign((size_t)max_seqs, 0);
        p->swapped.assign((size_t)max_seqs, 0);
        p->last_use.assign((size_t)max_seqs, 0);
    } catch (...) {
        delete p;
        return MI_ERR_INVALID_ARG;
    }
    *out = p;
    return MI_OK;
}

extern "C" void mi_kv_pool_destroy(mi_kv_pool* pool) { delete pool; }

extern "C" mi_status mi_kv_pool_alloc(mi_kv_pool* p, int32_t seq, int32_t num_tokens) {
    if (!p || seq < 0 || (size_t)seq >= p->tables.size() || num_tokens < 0) return MI_ERR_INVALID_ARG;
    if (p->swapped[(size_t)seq]) return MI_ERR_INVALID_ARG;  // swap it in first
    std::vector<int32_t>& t = p->tables[(size_t)seq];
    if (p->live[(size_t)seq] && num_tokens < p->tokens[(size_t)seq]) return MI_ERR_INVALID_ARG;
    const int64_t need = ((int64_t)num_tokens + p->block_size - 1) / p->block_size;
    if (need > p->max_blocks_per_seq) return MI_ERR_INVALID_ARG;
    const int64_t extra = need - (int64_t)t.size();
    if (extra > (int64_t)p->free_stack.size()) return MI_ERR_OUT_OF_BLOCKS;
    for (int64_t i = 0; i < extra; ++i) {
        t.push_back(p->free_stack.back());
        p->free_stack.pop_back();
    }
    p->tokens[(size_t)seq] = num_tokens;
    p->live[(size_t)seq] = 1;
    ++p->clock;
    p->use(seq);
    return MI_OK;
}

extern "C" mi_status mi_kv_pool_alloc_batch(mi_kv_pool* p, const int32_t* seq_ids, const int32_t* num_tokens,
                                            int32_t count) {
    if (!p || count < 0 || (count > 0 && (!seq_ids || !num_tokens))) return MI_ERR_INVALID_ARG;
    // check the whole batch first, earlier entries applied on a copy of the
    // state they touch, so that either every entry is made or none
    std::vector<int64_t> size(p->tables.size(), -1), toks(p->tables.size(), -1);
    int64_t extra_total = 0;
    for (int32_t i = 0; i < count; ++i) {
        const int32_t seq = seq_ids[i], n = num_tokens[i];
        if (seq < 0 || (size_t)seq >= p->tables.size() || n < 0) return MI_ERR_INVALID_ARG;
        if (p->swapped[(size_t)seq]) return MI_ERR_INVALID_ARG;
        const bool live = p->live[(size_t)seq] || size[(size_t)seq] >= 0;
        const int64_t have = size[(size_t)seq] >= 0 ? size[(size_t)seq] : (int64_t)p->tables[(size_t)seq].size();
        const int64_t held = toks[(size_t)seq] >= 0 ? toks[(size_t)seq] : p->tokens[(size_t)seq];
        if (live && n < held) return MI_ERR_INVALID_ARG;
        const int64_t need = ((int64_t)n + p->block_size - 1) / p->block_size;
        if (need > p->max_blocks_per_seq) return MI_ERR_INVALID_ARG;
        if (need > have) extra_total += need - have;
        size[(size_t)seq] = need > have ? need : have;
        toks[(size_t)seq] = n;
    }
    if (extra_total > (int64_t)p->free_stack.size()) return MI_ERR_OUT_OF_BLOCKS;
    for (int32_t i = 0; i < count; ++i) {
        const mi_status st = mi_kv_pool_alloc(p, seq_ids[i], num_tokens[i]);
        if (st != MI_OK) return st;  // not reached: the batch was checked above
    }
    return MI_OK;
}

extern "C" mi_status mi_kv_pool_free(mi_kv_pool* p, int32_t seq) {
    if (!p) return MI_ERR_INVALID_ARG;
    if (seq >= 0 && (size_t)seq < p->tables.size() && p->swapped[(size_t)seq]) {
        p->swapped[(size_t)seq] = 0;  // nothing on the device: just forget it
        p->tokens[(size_t)seq] = 0;
        return MI_OK;
    }
    if (seq < 0 || (size_t)seq >= p->tables.size() || !p->live[(size_t)seq]) return MI_ERR_UNKNOWN_SEQ;
    std::vector<int32_t>& t = p->tables[(size_t)seq];
    for (int32_t b : t) p->free_stack.push_back(b);
    t.clear();
    p->tokens[(size_t)seq] = 0;
    p->live[(size_t)seq] = 0;
    return MI_OK;
}

extern "C" int32_t mi_kv_pool_num_free(const mi_kv_pool* p) {
    return p ? (int32_t)p->free_stack.size() : -1;
}

extern "C" mi_status mi_kv_pool_batch_meta(const mi_kv_pool* p, const int32_t* seq_ids, int32_t B,
                                           int32_t* block_tables, int32_t* context_lens,
                                           int32_t* slot_mapping) {
    if (!p || B < 0 || (B > 0 && !seq_ids)) return MI_ERR_INVALID_ARG;
    const int32_t W = p->max_blocks_per_seq, BS = p->block_size;
    for (int32_t i = 0; i < B; ++i) {
        const int32_t s = seq_ids[i];
        if (s < 0 || (size_t)s >= p->tables.size() || !p->live[(size_t)s]) return MI_ERR_UNKNOWN_SEQ;
        const std::vector<int32_t>& t = p->tables[(size_t)s];
        const int32_t n = p->tokens[(size_t)s];
        if (block_tables) {
            int32_t* row = block_tables + (int64_t)i * W;
            const int32_t nb = (int32_t)t.size();
            if (nb) std::memcpy(row, t.data(), sizeof(int32_t) * (size_t)nb);
            for (int32_t j = nb; j < W; ++j) row[j] = -1;
        }
        if (context_lens) context_lens[i] = n;
        if (slot_mapping) slot_mapping[i] = n > 0 ? t[(size_t)((n - 1) / BS)] * BS + (n - 1) % BS : -1;
    }
    return MI_OK;
}

extern "C" int32_t mi_kv_pool_seq_blocks(const mi_kv_pool* p, int32_t seq, int32_t* out,
                                         int32_t max_out) {
    if (!p || seq < 0 || (size_t)seq >= p->tables.size() || !p->live[(size_t)seq]) return -1;
    const std::vector<int32_t>& t = p->tables[(size_t)seq];
    const int32_t n = (int32_t)t.size();
    if (out)
        for (int32_t i = 0; i < n && i < max_out; ++i) out[i] = t[(size_t)i];
    return n;
}

// RoPE table: (cos, sin) of p * theta^(-2i/d), double, rounded once to fp32.
extern "C" mi_status mi_rope_table(double theta, int32_t head_dim, int32_t max_pos, float* out) {
    if (!out || head_dim < 2 || (head_dim & 1) || max_pos < 1 || !(theta > 0.0)) return MI_ERR_INVALID_ARG;
    const int32_t half = head_dim / 2;
    std::vector<double> inv_freq((size_t)half);
    for (int32_t i = 0; i < half; ++i) inv_freq[(size_t)i] = 1.0 / std::pow(theta, (2.0 * i) / head_dim);
    for (int32_t p = 0; p < max_pos; ++p) {
        float* row = out + (int64_t)p * half * 2;
        for (int32_t i = 0; i < half; ++i) {
            const double a = (double)p * inv_freq[(size_t)i];
            row[2 * i] = (float)std::cos(a);
            row[2 * i + 1] = (float)std::sin(a);
        }
    }
    return MI_OK;
}

extern "C" mi_status mi_kv_pool_token_slots(const mi_kv_pool* p, int32_t seq, int32_t first_token,
                                            int32_t count, int32_t* slots_out) {
    if (!p || first_token < 0 || count < 0 || (count > 0 && !slots_out)) return MI_ERR_INVALID_ARG;
    if (seq < 0 || (size_t)seq >= p->tables.size() || !p->live[(size_t)seq]) return MI_ERR_UNKNOWN_SEQ;
    if ((int64_t)first_token + count > p->tokens[(size_t)seq]) return MI_ERR_INVALID_ARG;
    const std::vector<int32_t>& t = p->tables[(size_t)seq];
    const int32_t BS = p->block_size;
    for (int32_t i = 0; i < count; ++i) {
        const int32_t tok = first_token + i;
        slots_out[i] = t[(size_t)(tok / BS)] * BS + tok % BS;
    }
    return MI_OK;
}

extern "C" mi_status mi_kv_pool_admission(const mi_kv_pool* p, int32_t running_decodes, int32_t hard_bp,
                                          int32_t soft_bp, mi_admit_decision* out) {
    if (!p || !out || running_decodes < 0 || hard_bp < 0 || hard_bp > 10000 || soft_bp < 0 || soft_bp > 10000)
        return MI_ERR_INVALID_ARG;
    // free / total < bp / 10000, compared exactly in 64-bit integers
    const int64_t free_scaled = (int64_t)p->free_stack.size() * 10000;
    const int64_t total = p->num_blocks;
    if (free_scaled < (int64_t)hard_bp * total)
        *out = MI_ADMIT_HARD_BRAKE;
    else if (running_decodes > 0 && free_scaled < (int64_t)soft_bp * total)
        *out = MI_ADMIT_SOFT_BRAKE;
    else
        *out = MI_ADMIT_PROCEED;
    return MI_OK;
}

// ---------------------------------------------------------------- swap ----

extern "C" mi_status mi_kv_pool_touch(mi_kv_pool* p, const int32_t* seq_ids, int32_t n) {
    if (!p || n < 0 || (n > 0 && !seq_ids)) return MI_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t s = seq_ids[i];
        if (s < 0 || (size_t)s >= p->tables.size() || !p->live[(size_t)s]) return MI_ERR_UNKNOWN_SEQ;
    }
    ++p->clock;
    for (int32_t i = 0; i < n; ++i) p->use(seq_ids[i]);
    return MI_OK;
}

extern "C" int32_t mi_kv_pool_lru_victim(const mi_kv_pool* p, const int32_t* exclude, int32_t n_exclude) {
    if (!p || n_exclude < 0 || (n_exclude > 0 && !exclude)) return -1;
    int32_t best = -1;
    for (size_t s = 0; s < p->tables.size(); ++s) {
        if (!p->live[s] || p->tables[s].empty()) continue;
        bool skip = false;
        for (int32_t i = 0; i < n_exclude && !skip; ++i) skip = exclude[i] == (int32_t)s;
        if (skip) continue;
        if (best < 0 || p->last_use[s] < p->last_use[(size_t)best]) best = (int32_t)s;  // ties: lower id
    }
    return best;
}

extern "C" mi_status mi_kv_pool_swap_out(mi_kv_pool* p, int32_t seq, int32_t* blocks_out, int32_t max_out,
                                         int32_t* n_out) {
    if (!p || max_out < 0) return MI_ERR_INVALID_ARG;
    if (seq < 0 || (size_t)seq >= p->tables.size() || !p->live[(size_t)seq]) return MI_ERR_UNKNOWN_SEQ;
    std::vector<int32_t>& t = p->tables[(size_t)seq];
    if ((int64_t)t.size() > max_out || (!t.empty() && !blocks_out)) return MI_ERR_INVALID_ARG;
    for (size_t i = 0; i < t.size(); ++i) {
        blocks_out[i] = t[i];
        p->free_stack.push_back(t[i]);
    }
    if (n_out) *n_out = (int32_t)t.size();
    t.clear();
    p->live[(size_t)seq] = 0;
    p->swapped[(size_t)seq] = 1;
    return MI_OK;
}

extern "C" mi_status mi_kv_pool_swap_in(mi_kv_pool* p, int32_t seq, int32_t* blocks_out, int32_t max_out,
                                        int32_t* n_out) {
    if (!p || max_out < 0) return MI_ERR_INVALID_ARG;
    if (seq < 0 || (size_t)seq >= p->tables.size() || !p->swapped[(size_t)seq]) return MI_ERR_UNKNOWN_SEQ;
    const int64_t need = ((int64_t)p->tokens[(size_t)seq] + p->block_size - 1) / p->block_size;
    if (need > max_out || (need > 0 && !blocks_out)) return MI_ERR_INVALID_ARG;
    if (need > (int64_t)p->free_stack.size()) return MI_ERR_OUT_OF_BLOCKS;
    std::vector<int32_t>& t = p->tables[(size_t)seq];
    for (int64_t i = 0; i < need; ++i) {
        t.push_back(p->free_stack.back());
        p->free_stack.pop_back();
        blocks_out[i] = t.back();
    }
    if (n_out) *n_out = (int32_t)need;
    p->swapped[(size_t)seq] = 0;
    p->live[(size_t)seq] = 1;
    ++p->clock;
    p->use(seq);
    return MI_OK;
}
