/*
 * mi.h - paged KV cache decode step for one NVIDIA GB300 (sm_103a).
 *
 * One decode step per layer is: grow each request's block table on the host
 * (mi_kv_pool_*), apply RoPE to the new token's q/k and scatter k/v into the
 * paged cache (mi_paged_kv_append), then Grouped-Query decode attention over
 * every request's paged history (mi_paged_decode_attention).
 *
 * The step follows mini-infer's decode_batch (mini-infer README, "架构设计",
 * "decode_batch 关键步骤": gather_batch_kv -> model_forward -> write_decode_kv)
 * over its Paged KV Cache ("项目概述": BlockTable + free-block pool), with GQA
 * and RoPE as the NJU course brief "端侧大模型推理框架" §2.1 lists them for the
 * Qwen models. The gather is not materialised: the attention kernel reads each
 * block in place.
 *
 * Conventions for every entry point:
 *  - All sizes are int32 unless stated. bf16 tensors are passed as void*.
 *  - Device pointers are caller-owned memory on the current CUDA device, and
 *    must stay valid until the work queued on `stream` has finished. The
 *    library allocates no device memory and keeps no device pointer.
 *  - Every device entry point is asynchronous on `stream` (NULL = the legacy
 *    default stream). Host-side argument checks return synchronously, before
 *    anything is queued; a rejected call queues nothing.
 *  - Data-dependent faults found on the device (a block id outside
 *    [0, num_blocks), a slot outside the cache, a position outside the RoPE
 *    table, a context longer than a table row) never trap: the kernel skips the
 *    offending entry and ORs an MI_DEVERR_* bit into *dev_err (when dev_err is
 *    not NULL). The caller reads the word after synchronising; the library
 *    never clears it.
 *  - Thread safety: device entry points are reentrant. A pool handle must be
 *    used by one host thread at a time.
 */
#ifndef MI_H
#define MI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream), without the CUDA headers. */
typedef struct CUstream_st* mi_stream_t;

typedef enum mi_status {
    MI_OK = 0,
    MI_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned buffer */
    MI_ERR_OUT_OF_BLOCKS = 2,  /* the pool cannot grow the sequence; nothing changed */
    MI_ERR_UNKNOWN_SEQ = 3,    /* sequence id not allocated */
    MI_ERR_UNSUPPORTED = 4,    /* head_dim, block_size or GQA group outside what is built */
    MI_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
    MI_ERR_DEVICE_BOUNDS = 6,  /* reserved: a caller may map a nonzero *dev_err to it */
    MI_ERR_TIMEOUT = 7         /* reserved for bounded device-side waits */
} mi_status;

/* Bits ORed into *dev_err by the kernels. */
#define MI_DEVERR_BAD_BLOCK    0x1 /* block table entry outside [0, num_blocks) */
#define MI_DEVERR_BAD_SLOT     0x2 /* slot_mapping entry outside the cache */
#define MI_DEVERR_BAD_POS      0x4 /* position outside [0, max_pos) */
#define MI_DEVERR_BAD_CONTEXT  0x8 /* context length above max_blocks_per_seq * block_size */
#define MI_DEVERR_TIMEOUT      0x10 /* a staged copy did not land within the wait limit */
#define MI_DEVERR_BAD_SCALE    0x40 /* FP8 append: a KV head's scale is not a positive finite number */
#define MI_DEVERR_INTERNAL     0x80 /* a kernel could not lay out its shared memory (the call did nothing) */
#define MI_DEVERR_BAD_QUERY    0x20 /* prefill: query_start not within [0, total_q] and ascending,
                                       a request longer than max_query_len, or more
                                       new tokens than context */

/* Short human-readable name of a status. */
const char* mi_status_string(mi_status s);

/* ------------------------------------------------------------------------ */
/* Host block pool (mini-infer README "项目概述" / "架构设计" KVCacheManager;
 * nxmr.cn article §2.1 "KV缓存的内存革命" allocate sketch: pages_needed =
 * ceil(seq_len / PAGE_SIZE), each popped from the free list). The pool is
 * fixed: when the free list is empty a request fails instead of growing it.
 *
 * Semantics (exact, so that a model of the pool can reproduce every table):
 *  - The free list is a stack. On creation successive pops return
 *    initial_free_order[0], [1], ... (or 0, 1, 2, ... when it is NULL).
 *  - mi_kv_pool_alloc(seq, n) grows seq's table to ceil(n / block_size) blocks
 *    by popping the missing ones in order and appending them. All or nothing.
 *  - mi_kv_pool_free(seq) pushes seq's blocks in table order (so the next pop
 *    returns its last block) and forgets seq.
 * The pool is host memory only and never touches the GPU.
 * ------------------------------------------------------------------------ */
typedef struct mi_kv_pool mi_kv_pool; /* opaque; owned by the library */

/* num_blocks >= 1; block_size must be 16; max_seqs >= 1 (ids are 0..max_seqs-1);
 * max_blocks_per_seq >= 1 is the width of one block-table row.
 * initial_free_order: NULL or a permutation of [0, num_blocks) (checked).
 * On MI_OK *out holds a new pool; release it with mi_kv_pool_destroy. */
mi_status mi_kv_pool_create(int32_t num_blocks, int32_t block_size, int32_t max_seqs,
                            int32_t max_blocks_per_seq, const int32_t* initial_free_order,
                            mi_kv_pool** out);

/* Frees the pool and every table. NULL is ignored. */
void mi_kv_pool_destroy(mi_kv_pool* pool);

/* Grow sequence seq_id to hold num_tokens tokens (creating it if new).
 * MI_ERR_INVALID_ARG: seq_id outside [0, max_seqs), num_tokens < 0, fewer tokens
 * than the sequence already holds, or more blocks than a table row.
 * MI_ERR_OUT_OF_BLOCKS: not enough free blocks; the pool is unchanged. */
mi_status mi_kv_pool_alloc(mi_kv_pool* pool, int32_t seq_id, int32_t num_tokens);

/* mi_kv_pool_alloc for a whole batch (a decode step grows every request by
 * one token): entry i grows seq_ids[i] to num_tokens[i] tokens, in order, as
 * count calls of mi_kv_pool_alloc would (the same tables and use order), but
 * all or nothing: the batch is checked first, and on any error
 * (MI_ERR_INVALID_ARG for an entry mi_kv_pool_alloc would reject,
 * MI_ERR_OUT_OF_BLOCKS when the batch needs more blocks than are free) the
 * pool is unchanged. Host arrays of count entries; count 0 does nothing. */
mi_status mi_kv_pool_alloc_batch(mi_kv_pool* pool, const int32_t* seq_ids, const int32_t* num_tokens,
                                 int32_t count);

/* Return all blocks of seq_id to the free list. MI_ERR_UNKNOWN_SEQ if seq_id
 * holds no allocation. */
mi_status mi_kv_pool_free(mi_kv_pool* pool, int32_t seq_id);

/* Number of free blocks, or -1 for a NULL pool. */
int32_t mi_kv_pool_num_free(const mi_kv_pool* pool);

/* Host metadata for a decode batch of B sequences (host buffers, caller-owned):
 *  block_tables  [B][max_blocks_per_seq] int32: physical block ids, padded with -1;
 *  context_lens  [B] int32: tokens held (the post-append length in a decode step);
 *  slot_mapping  [B] int32: slot of the sequence's last token,
 *                table[(n-1)/16]*16 + (n-1)%16, or -1 when n == 0.
 * Any output pointer may be NULL to skip it. MI_ERR_UNKNOWN_SEQ if a sequence
 * is not allocated (outputs then undefined). */
mi_status mi_kv_pool_batch_meta(const mi_kv_pool* pool, const int32_t* seq_ids, int32_t B,
                                int32_t* block_tables, int32_t* context_lens,
                                int32_t* slot_mapping);

/* Slots of tokens first_token .. first_token+count-1 of sequence seq_id, in
 * order, into slots_out[0..count) (host): slot = table[t/16]*16 + t%16. This
 * is the slot_mapping of a chunked append (prefill of many tokens per
 * request; mini-infer README "项目概述", prefill and decode as separate
 * passes). MI_ERR_UNKNOWN_SEQ if seq_id holds no allocation;
 * MI_ERR_INVALID_ARG if first_token < 0, count < 0 or the range passes the
 * tokens the sequence holds. */
mi_status mi_kv_pool_token_slots(const mi_kv_pool* pool, int32_t seq_id, int32_t first_token,
                                 int32_t count, int32_t* slots_out);

/* Admission of a new prefill request from the pool's free space: the
 * three-level brake of the GitLink project report "mxdyymxgxtlkjdxtjyhysx"
 * (section "我们的解决方案：SLO感知与KV Cache保护调度器"):
 *   MI_ADMIT_HARD_BRAKE  free share of the pool below hard_bp / 10000
 *                        (report's example: 10%), whatever is running;
 *   MI_ADMIT_SOFT_BRAKE  running_decodes > 0 and free share below
 *                        soft_bp / 10000 (example: 30%);
 *   MI_ADMIT_PROCEED     otherwise.
 * "Below" is strict; the shares are compared exactly in integers
 * (free * 10000 < bp * num_blocks). Thresholds in basis points, 0..10000.
 * MI_ERR_INVALID_ARG for a NULL pool or out, running_decodes < 0 or a
 * threshold outside 0..10000. Host only; the pool is not changed. */
typedef enum mi_admit_decision {
    MI_ADMIT_PROCEED = 0,
    MI_ADMIT_SOFT_BRAKE = 1,
    MI_ADMIT_HARD_BRAKE = 2
} mi_admit_decision;
#define MI_ADMIT_HARD_BP_DEFAULT 1000
#define MI_ADMIT_SOFT_BP_DEFAULT 3000
mi_status mi_kv_pool_admission(const mi_kv_pool* pool, int32_t running_decodes, int32_t hard_bp,
                               int32_t soft_bp, mi_admit_decision* out);

/* ---- KV swap to host memory with LRU eviction (NJU course brief, optional
 * task 3 "KV Cache Offloading": inactive KV blocks move to CPU memory and come
 * back when needed, under an eviction policy such as LRU).
 * A sequence is resident (it holds a table) or swapped out (it holds no
 * block; its token count is kept). Swapped-out sequences are unknown to
 * batch_meta, token_slots and seq_blocks (MI_ERR_UNKNOWN_SEQ / -1), rejected
 * by alloc (MI_ERR_INVALID_ARG) and forgotten by free. The pool keeps a use
 * clock: every successful alloc, swap_in and touch call advances it by one
 * and stamps the sequences it names. */

/* Mark n resident sequences as used now. MI_ERR_UNKNOWN_SEQ (and no change)
 * if one is not resident. */
mi_status mi_kv_pool_touch(mi_kv_pool* pool, const int32_t* seq_ids, int32_t n);

/* The resident sequence with the oldest use stamp that holds at least one
 * block and is not among exclude[0..n_exclude) (ties: lower id), or -1. */
int32_t mi_kv_pool_lru_victim(const mi_kv_pool* pool, const int32_t* exclude, int32_t n_exclude);

/* Swap out a resident sequence: its table (in order) goes to
 * blocks_out[0..*n_out) and its blocks return to the free list as
 * mi_kv_pool_free returns them. The caller copies those blocks' contents
 * out (mi_kv_copy_blocks) before anything can reuse them. MI_ERR_INVALID_ARG
 * (no change) if max_out is below the block count. */
mi_status mi_kv_pool_swap_out(mi_kv_pool* pool, int32_t seq_id, int32_t* blocks_out, int32_t max_out,
                              int32_t* n_out);

/* Swap a sequence back in: pop ceil(tokens/16) blocks (as alloc pops them)
 * into its table and blocks_out[0..*n_out); the caller copies its contents
 * back into them. MI_ERR_OUT_OF_BLOCKS leaves the pool unchanged;
 * MI_ERR_UNKNOWN_SEQ if it is not swapped out. */
mi_status mi_kv_pool_swap_in(mi_kv_pool* pool, int32_t seq_id, int32_t* blocks_out, int32_t max_out,
                             int32_t* n_out);

/* Copy of one sequence's table into out[0..max_out) (host); returns the
 * number of blocks it holds, or -1 if unknown. */
int32_t mi_kv_pool_seq_blocks(const mi_kv_pool* pool, int32_t seq_id, int32_t* out,
                              int32_t max_out);

/* ------------------------------------------------------------------------ */
/* Shapes shared by the device entry points.
 *   B                   requests in the batch (decode attention: up to 65535;
 *                       prefill attention: any); for mi_paged_kv_append the
 *                       number of new-token rows (up to 2^24)
 *   Hq, Hkv             query / KV heads; Hq % Hkv == 0, G = Hq/Hkv in 1..8
 *   head_dim            64 or 128
 *   block_size          16
 *   num_blocks          physical blocks in k_cache / v_cache
 *   max_blocks_per_seq  width of a block-table row
 * Cache layout (both caches, bf16, contiguous, 16-byte aligned):
 *   [num_blocks][Hkv][block_size][head_dim]
 * so one (block, KV head) tile of 16 tokens is contiguous (4 KB at d = 128).
 * ------------------------------------------------------------------------ */
typedef struct mi_dims {
    int32_t B, Hq, Hkv, head_dim, block_size, num_blocks, max_blocks_per_seq;
} mi_dims;

/* RoPE table on the host: out[max_pos][head_dim/2][2] fp32 holds
 * (cos, sin) of p * theta^(-2i/head_dim), each evaluated in double and rounded
 * once to fp32 (NJU course brief §2.1, "RoPE construction and application";
 * theta = 1e6 for Qwen2.5/Qwen3). The caller copies it to the device for
 * mi_paged_kv_append. head_dim even and >= 2, max_pos >= 1, theta > 0. */
mi_status mi_rope_table(double theta, int32_t head_dim, int32_t max_pos, float* host_out);

/* Append one new token per request (mini-infer README "decode_batch 关键步骤",
 * write_decode_kv, with RoPE applied first as in NJU course brief §2.1).
 * Rows are independent, so the same call appends a prefill chunk: make each
 * new token a row b (dims.B = total new tokens) with its own position and
 * slot (mi_kv_pool_token_slots).
 * For row b at position p = positions[b]:
 *   q_out[b][j]                    = RoPE_p(q[b][j])   for j < Hq
 *   k_cache[blk][h][off][:]        = RoPE_p(k[b][h])   for h < Hkv
 *   v_cache[blk][h][off][:]        = v[b][h]
 * with blk = slot_mapping[b] / 16, off = slot_mapping[b] % 16. RoPE rotates the
 * pairs (i, i + d/2) by the table angle (rotate-half pairing):
 *   y[i] = x[i] c - x[i+d/2] s,  y[i+d/2] = x[i+d/2] c + x[i] s
 * computed in double from the bf16 inputs and fp32 table values, then rounded
 * once to bf16 (nearest, ties to even). No other cache byte is written.
 * Device buffers: q [B][Hq][d], k, v [B][Hkv][d], q_out [B][Hq][d] (bf16;
 * q_out may equal q), positions, slot_mapping [B] int32, rope_cos_sin
 * [max_pos][d/2][2] fp32 (from mi_rope_table), dev_err int32 or NULL.
 * A bad position skips the whole request (MI_DEVERR_BAD_POS); a bad slot skips
 * its cache writes (MI_DEVERR_BAD_SLOT). */
mi_status mi_paged_kv_append(const mi_dims* dims, const void* q, const void* k, const void* v,
                             const int32_t* positions, const int32_t* slot_mapping,
                             const float* rope_cos_sin, int32_t max_pos, void* q_out,
                             void* k_cache, void* v_cache, int32_t* dev_err, mi_stream_t stream);

/* Device workspace the attention call needs for these dims on the current
 * device (split-KV partials of the persistent grid): a size in bytes, or 0 when
 * the dims are not supported. */
size_t mi_paged_decode_workspace_bytes(const mi_dims* dims);

/* Paged GQA decode attention (mini-infer README "decode_batch 关键步骤": the
 * attention of model_forward over the KV that gather_batch_kv would collect,
 * read in place; NJU course brief §2.1 GQA: query head j uses KV head j / G).
 * For every request b and query head j, with n = context_lens[b] (the length
 * after append) and K_t, V_t read from block block_tables[b][t/16], offset t%16:
 *   out[b][j] = sum_t softmax_t(scale * <q[b][j], K_t>) V_t,   t < n
 * computed as a split-KV online softmax in fp32 followed by a log-sum-exp
 * combine of the splits, rounded to bf16. n <= 0 gives a zero row.
 * Device buffers: q [B][Hq][d] bf16 (RoPE already applied), k_cache, v_cache
 * (layout above), block_tables [B][max_blocks_per_seq] int32, context_lens [B]
 * int32, out [B][Hq][d] bf16, workspace of mi_paged_decode_workspace_bytes()
 * bytes (16-byte aligned; contents need no initialisation and are overwritten),
 * dev_err int32 or NULL. Only the first ceil(n/16) entries of a table row are
 * read. Tokens past n in the last block are never used (they may hold any bits,
 * NaN included). Results are bitwise independent of where blocks sit in the
 * cache. The call may be captured in a CUDA graph and the graph replayed any
 * number of times over the same workspace (each launch hands back its merge
 * counters zeroed); after a launch that set MI_DEVERR_TIMEOUT, zero the
 * workspace before the next replay. The same holds for the e4m3 and fused
 * step variants below. */
mi_status mi_paged_decode_attention(const mi_dims* dims, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    const int32_t* context_lens, float scale, void* out,
                                    void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                    mi_stream_t stream);

/* One decode step of a layer in one launch: exactly mi_paged_kv_append with
 * positions[b] = n - 1 and slot_mapping[b] = block_tables[b][(n-1)/16] * 16 +
 * (n-1) % 16 (n = context_lens[b], the length after the append), followed by
 * mi_paged_decode_attention on its outputs; q_out, the new cache rows and out
 * get the same bits as those two calls. Inside the attention kernel, every
 * CTA streaming a piece of request b's KV head h rotates that head group's q
 * itself, and the warp that streams the block holding the new token rotates
 * its k, writes k and v into that row of the staged tiles and of the cache,
 * and writes the rotated q to q_out. bf16 caches, the MMA tile.
 * Device buffers as for the two calls; q is the raw (unrotated) q and must
 * not overlap q_out (MI_ERR_INVALID_ARG). Requests with n <= 0 append nothing
 * and get zero rows; n - 1 >= max_pos sets MI_DEVERR_BAD_POS and leaves that
 * request's q zero.
 * flags: 0, or MI_STEP_EARLY_START (below); any other bit is
 * MI_ERR_INVALID_ARG. */
mi_status mi_paged_decode_step(const mi_dims* dims, const void* q, const void* k, const void* v,
                               const float* rope_cos_sin, int32_t max_pos, const int32_t* block_tables,
                               const int32_t* context_lens, float scale, void* q_out, void* k_cache,
                               void* v_cache, void* out, void* workspace, size_t workspace_bytes,
                               int32_t* dev_err, mi_stream_t stream, uint32_t flags);

/* Early start of a fused step (mi_paged_decode_step, mi_paged_decode_step_fp8).
 * Every call of this library waits for the kernel launched just before it on
 * the same stream before it reads anything, though it may be launched while
 * that kernel is finishing (programmatic dependent launch). With this flag
 * the step reads context_lens, block_tables, the cache rows of the history
 * and its plan entries in the workspace before that wait, and may write
 * those plan entries and report errors into dev_err: in a stack of layers,
 * each layer's plan and first KV copies then overlap the previous layer's
 * last CTAs. The results are bit for bit those without the flag.
 * The caller guarantees that the kernel launched just before the call on
 * the same stream writes none of this call's context_lens, block_tables,
 * k_cache and v_cache, does not clear dev_err (the library's own error
 * reports are atomic ORs, so consecutive steps may share one word), and
 * neither reads nor writes this call's workspace. So two consecutive
 * early-start calls take different workspaces (two, used in turn, suffice:
 * the step lets the next launch start only after its own wait, so a
 * launch never runs beside the one two before it), and a call directly
 * after mi_kv_copy_blocks, mi_kv_copy_rows or an append into the same
 * caches, or after a kernel of the caller's that fills the tables or
 * lengths, does not set the flag. */
#define MI_STEP_EARLY_START 1u

/* Kernel variant used by mi_paged_decode_attention_variant:
 *   MI_ATTN_MMA  bf16 tensor-core tiles (mma.sync m16n8k16: 16 tokens x 8 heads),
 *   MI_ATTN_FMA  fp32 CUDA-core FMA tiles.
 * Both share the staging pipeline, split plan and combine, and return results
 * within the same tolerance; mi_paged_decode_attention uses the default. */
typedef enum mi_attn_variant { MI_ATTN_DEFAULT = 0, MI_ATTN_MMA = 1, MI_ATTN_FMA = 2 } mi_attn_variant;

/* mi_paged_decode_attention with an explicit kernel variant and grid size:
 * ctas = 0 picks the persistent grid (all SMs at full occupancy); a positive
 * value caps the number of CTAs (and thus KV splits), which changes only the
 * fp32 rounding of the result. The workspace must be sized for ctas = 0. */
mi_status mi_paged_decode_attention_variant(const mi_dims* dims, const void* q,
                                            const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables,
                                            const int32_t* context_lens, float scale, void* out,
                                            void* workspace, size_t workspace_bytes,
                                            int32_t* dev_err, mi_stream_t stream,
                                            mi_attn_variant variant, int32_t ctas);

/* ---- FP8 (e4m3) KV cache (GitLink project report "mxdyymxgxtlkjdxtjyhysx",
 * section "技术探索：FP8 KV Cache量化效果分析": the KV cache held in FP8 to cut
 * the bytes each decode step moves). Layout as the bf16 caches with one byte
 * per element: [num_blocks][Hkv][16][head_dim] e4m3 (1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits, subnormals, no infinities, S.1111.111 = NaN,
 * largest finite 448). Each KV head h has fp32 scales k_scale[h], v_scale[h]
 * (device arrays [Hkv]): a cached code c stands for value(c) * scale[h]. */

/* mi_paged_kv_append into FP8 caches. q_out is as in mi_paged_kv_append; the
 * cache rows of the new token hold, for every element,
 *   k8 = e4m3(fp32(bf16(RoPE(k)) / k_scale[h])),  v8 = e4m3(fp32(v / v_scale[h]))
 * where bf16(RoPE(k)) is exactly what mi_paged_kv_append would store, the
 * quotient is an IEEE single-precision division, and e4m3() rounds to nearest
 * with ties to even, values beyond +-448 saturating to +-448. A scale that is
 * not a positive finite number skips that head's cache writes
 * (MI_DEVERR_BAD_SCALE; a bad V scale likewise skips its V rows). */
mi_status mi_paged_kv_append_fp8(const mi_dims* dims, const void* q, const void* k, const void* v,
                                 const int32_t* positions, const int32_t* slot_mapping,
                                 const float* rope_cos_sin, int32_t max_pos, void* q_out, void* k_cache,
                                 void* v_cache, const float* k_scale, const float* v_scale,
                                 int32_t* dev_err, mi_stream_t stream);

/* mi_paged_decode_attention over FP8 caches: the same definition with
 * K_t = value(k8_t) * k_scale[h] and V_t = value(v8_t) * v_scale[h]. The
 * products run on tensor cores in f16 (every e4m3 value is an f16 value; q is
 * converted to f16 with one rounding, so |q| must stay below 65504), with an
 * fp32 online softmax, as the bf16 call. Same workspace
 * (mi_paged_decode_workspace_bytes), errors and guarantees. */
mi_status mi_paged_decode_attention_fp8(const mi_dims* dims, const void* q, const void* k_cache,
                                        const void* v_cache, const float* k_scale, const float* v_scale,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        float scale, void* out, void* workspace, size_t workspace_bytes,
                                        int32_t* dev_err, mi_stream_t stream);

/* One decode step of a layer over FP8 caches in one launch: exactly
 * mi_paged_kv_append_fp8 with positions[b] = n - 1 and slot_mapping[b] =
 * block_tables[b][(n-1)/16] * 16 + (n-1) % 16 (n = context_lens[b], the
 * length after the append), followed by mi_paged_decode_attention_fp8 on its
 * outputs; q_out and the new cache rows (quantised as the FP8 append
 * quantises them) get the same bits as those two calls, and out is within
 * the attention's fp32 rounding of theirs (this kernel runs two CTAs per SM
 * where the e4m3 attention runs three, so the split differs). A K
 * or V scale that is not a positive finite number leaves that row of the
 * cache as it was (MI_DEVERR_BAD_SCALE). Other arguments, errors and
 * guarantees as mi_paged_decode_step (flags included); q must not overlap
 * q_out. */
mi_status mi_paged_decode_step_fp8(const mi_dims* dims, const void* q, const void* k, const void* v,
                                   const float* rope_cos_sin, int32_t max_pos, const int32_t* block_tables,
                                   const int32_t* context_lens, const float* k_scale, const float* v_scale,
                                   float scale, void* q_out, void* k_cache, void* v_cache, void* out,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_err, mi_stream_t stream,
                                   uint32_t flags);

/* ---- INT8 KV cache in 64-token groups (nxmr.cn article, §2.2
 * "量化压缩的实战选择": 8-bit KV quantised per group of 64 tokens rather than
 * per token, symmetric, scale = 127 / max|x|, the scaled values clamped to
 * [-128, 127] and cast to int8; per head).
 * A group is tokens 64g .. 64g+63 of one request and one KV head, over all
 * head_dim values; K and V are quantised separately. With m = max |x| over
 * the group's tokens (x the bf16 value the bf16 cache would hold, after RoPE
 * for K), a value is stored as the code
 *   c = trunc(clamp(fp32(x * fp32(127 / m)), -128, 127))
 * (both operations IEEE single precision, truncation toward zero; m = 0 gives
 * 0) and stands for c * m / 127. Buffers (device):
 *   k_cache, v_cache  int8 [num_blocks][Hkv][16][head_dim], 16-byte aligned;
 *   k_amax, v_amax    fp32 [num_blocks][Hkv]: m of the group each block's
 *                     tokens belong to (every block of a group holds it),
 *                     4-byte aligned;
 *   k_open, v_open    bf16 [num_open_slots][Hkv][64][head_dim]: the original
 *                     values of each sequence's last, still open group, at
 *                     the sequence's slot (open_slots[b] for request b).
 * A group that has fewer than 64 tokens (a sequence's last) is quantised over
 * the tokens it holds, and again from the open buffer whenever a token joins
 * it, so a full group ends up quantised over its 64 tokens. */

/* Decode append into INT8 caches, one new token per request: with n =
 * context_lens[b] (the length after the append; n <= 0 appends nothing) and
 * p = n - 1, q_out[b] = RoPE(q[b], p) as mi_paged_kv_append computes it; the
 * rotated k and the v of the new token go to row p % 64 of the request's open
 * slot, and the group of p (tokens 64(p/64) .. p) gets its codes and its m
 * as defined above, written through block_tables[b] (its blocks must be
 * allocated). Device errors: p >= max_pos (MI_DEVERR_BAD_POS) or n above
 * max_blocks_per_seq * 16 (MI_DEVERR_BAD_CONTEXT) skip the request; a slot
 * outside [0, num_open_slots) (MI_DEVERR_BAD_SLOT) or a block id of the
 * group out of range (MI_DEVERR_BAD_BLOCK) skip its cache writes. q, k, v,
 * q_out, rope_cos_sin and the open buffers 16-byte aligned; q_out may alias
 * q. */
mi_status mi_paged_kv_append_int8(const mi_dims* dims, const void* q, const void* k, const void* v,
                                  const float* rope_cos_sin, int32_t max_pos, const int32_t* block_tables,
                                  const int32_t* context_lens, const int32_t* open_slots,
                                  int32_t num_open_slots, void* q_out, void* k_cache, void* v_cache,
                                  float* k_amax, float* v_amax, void* k_open, void* v_open, int32_t* dev_err,
                                  mi_stream_t stream);

/* The INT8 append for many new tokens per request (a prompt, or a chunk of
 * one): dims.B = R requests; request r's m_r = query_start[r+1] -
 * query_start[r] new tokens are rows query_start[r] .. query_start[r+1]-1 of
 * q [T][Hq][d], k and v [T][Hkv][d] (T = total_tokens = query_start[R]),
 * at positions n_r - m_r .. n_r - 1 (n_r = context_lens[r], counting them).
 * The result is exactly that of m_r calls of mi_paged_kv_append_int8, one
 * token each, in order: q_out rows rotated, every group the new tokens touch
 * quantised over all its tokens (the open group's earlier ones from the open
 * buffer), its maxima written to all its blocks, and the last group's new
 * rows added to the open buffer (rows of a slot past its open group's tokens
 * are unspecified, and no call reads them). Device errors: query_start out of order or
 * past T, or m_r > n_r (MI_DEVERR_BAD_QUERY), n_r above max_blocks_per_seq *
 * 16 (MI_DEVERR_BAD_CONTEXT) or n_r - 1 >= max_pos (MI_DEVERR_BAD_POS) skip
 * the request; a bad open slot (MI_DEVERR_BAD_SLOT) or a bad block id of a
 * touched group (MI_DEVERR_BAD_BLOCK) skip its cache writes. Buffers and
 * alignment as mi_paged_kv_append_int8. */
mi_status mi_paged_kv_append_int8_tokens(const mi_dims* dims, int32_t total_tokens, const void* q, const void* k,
                                         const void* v, const float* rope_cos_sin, int32_t max_pos,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         const int32_t* query_start, const int32_t* open_slots,
                                         int32_t num_open_slots, void* q_out, void* k_cache, void* v_cache,
                                         float* k_amax, float* v_amax, void* k_open, void* v_open, int32_t* dev_err,
                                         mi_stream_t stream);

/* mi_paged_decode_attention over INT8 caches: the same definition with
 * K_t = c_t * k_amax[blk][h] / 127 and V_t = c_t * v_amax[blk][h] / 127,
 * blk = block_tables[b][t / 16]. The products run on tensor cores in f16
 * (every code is an f16 value; q is converted to f16 with one rounding, so
 * |q| must stay below 65504), with an fp32 online softmax; each block's V
 * factor scales the f16 probabilities relative to the largest factor seen so
 * far in the piece. Same workspace (mi_paged_decode_workspace_bytes), errors
 * and guarantees as mi_paged_decode_attention. */
mi_status mi_paged_decode_attention_int8(const mi_dims* dims, const void* q, const void* k_cache,
                                         const void* v_cache, const float* k_amax, const float* v_amax,
                                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                                         void* out, void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                         mi_stream_t stream);

/* Causal paged GQA attention for a prefill or chunked-prefill batch (NJU
 * course brief §2.1, the prefill stage of the prefill + decode loop; mini-infer
 * README "项目概述", prefill as its own pass). dims.B = R requests. Request r
 * contributes m_r = query_start[r+1] - query_start[r] new tokens, rows
 * query_start[r] .. query_start[r+1]-1 of q, and holds n_r = context_lens[r]
 * tokens counting them, so its new token i sits at position n_r - m_r + i:
 *   out[row][j] = sum_t softmax_t(scale * <q[row][j], K_t>) V_t,
 *                 t <= n_r - m_r + i,  K_t, V_t of KV head j / G
 * read through block_tables[r] as in mi_paged_decode_attention; fp32 online
 * softmax on bf16 tensor-core products, rounded to bf16.
 * Host arguments: total_q = query_start[R] (rows of q and out), max_query_len
 * >= every m_r (sizes the grid; 0 queues nothing).
 * Device buffers: q, out [total_q][Hq][d] bf16 (16-byte aligned; q with RoPE
 * applied), k_cache, v_cache, block_tables [R][max_blocks_per_seq] int32,
 * context_lens [R] int32, query_start [R+1] int32, dev_err int32 or NULL.
 * No workspace. Only the table entries covering positions < n_r are read;
 * cache tokens past n_r may hold any bits.
 * Device errors (MI_DEVERR_*): a bad query_start entry or m_r > max_query_len
 * skips request r (BAD_QUERY; its rows are left as they were); m_r > n_r gives
 * zero rows for the new tokens at negative positions (BAD_QUERY); n_r above a
 * table row clamps to it (BAD_CONTEXT); a bad block id drops that block's
 * keys (BAD_BLOCK). A request with m_r = 1 computes what
 * mi_paged_decode_attention computes for it. */
mi_status mi_paged_prefill_attention(const mi_dims* dims, int32_t total_q, int32_t max_query_len,
                                     const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, const int32_t* context_lens,
                                     const int32_t* query_start, float scale, void* out,
                                     int32_t* dev_err, mi_stream_t stream);

/* Kernel of mi_paged_prefill_attention_variant:
 *   MI_PREFILL_MMA      warp-level mma.sync tiles (64 rows per CTA; any G),
 *   MI_PREFILL_TCGEN05  fifth-generation tensor cores (tcgen05.mma with
 *                       tensor-memory accumulators; 128 / G whole tokens,
 *                       i.e. (128 / G) * G rows, per CTA; any G up to 8).
 *   MI_PREFILL_TCGEN05_PAIR  tcgen05 with two 128-row Q tiles per CTA
 *                       (one CTA per SM) sharing 128-key K / V stages,
 *                       one issuing thread alternating the tiles, 16
 *                       softmax warps (each lane: two rows, 32 keys).
 * MI_PREFILL_DEFAULT takes the pair kernel. All compute the same
 * definition within the same tolerance. */
#define MI_PREFILL_DEFAULT 0
#define MI_PREFILL_MMA 1
#define MI_PREFILL_TCGEN05 2
#define MI_PREFILL_TCGEN05_PAIR 3
mi_status mi_paged_prefill_attention_variant(const mi_dims* dims, int32_t total_q, int32_t max_query_len,
                                             const void* q, const void* k_cache, const void* v_cache,
                                             const int32_t* block_tables, const int32_t* context_lens,
                                             const int32_t* query_start, float scale, void* out,
                                             int32_t* dev_err, mi_stream_t stream, int32_t variant);

/* Block copies between two paged caches (the data movement of a swap):
 *   dst_k[dst_blocks[i]] = src_k[src_blocks[i]],
 *   dst_v[dst_blocks[i]] = src_v[src_blocks[i]]     for i < n,
 * a block being all Hkv heads' 16 token rows ([Hkv][16][head_dim] bf16; dims
 * supplies Hkv, head_dim and block_size; its other fields are not used).
 * src_* hold src_num_blocks blocks, dst_* dst_num_blocks. Each of the four
 * caches may be device memory or pinned host memory (cudaHostAlloc or
 * cudaHostRegister: the kernel reads and writes it in place); all 16-byte
 * aligned. src_blocks and dst_blocks are int32 [n] arrays the device can read
 * (device or pinned host). Pinned host pointers are translated to their
 * device addresses; pageable host memory is refused (MI_ERR_INVALID_ARG).
 * Destination blocks must be distinct and must not overlap the source
 * blocks. A pair with an id out of range is skipped (MI_DEVERR_BAD_BLOCK).
 * One kernel launch on `stream`; host buffers must stay pinned and untouched
 * by the host until it completes. */
mi_status mi_kv_copy_blocks(const mi_dims* dims, const void* src_k, const void* src_v,
                            int32_t src_num_blocks, const int32_t* src_blocks, void* dst_k, void* dst_v,
                            int32_t dst_num_blocks, const int32_t* dst_blocks, int32_t n,
                            int32_t* dev_err, mi_stream_t stream);

/* Copy n rows of row_bytes bytes each: row src_ids[i] of src (src_count rows
 * of row_bytes, back to back) to row dst_ids[i] of dst (dst_count rows).
 * The general form of mi_kv_copy_blocks for KV state whose rows are not
 * bf16 blocks: the blocks of one-byte (e4m3, INT8) caches (row =
 * Hkv * 16 * head_dim bytes), the INT8 group maxima of a block (row = Hkv
 * floats) and a sequence's INT8 open-group rows (row = Hkv * 64 * head_dim
 * bf16). row_bytes a positive multiple of 4, src and dst 4-byte aligned
 * (16-byte vectors are used when both are 16-byte aligned and row_bytes is
 * a multiple of 16). Memory, id arrays, overlap rules, errors
 * (MI_DEVERR_BAD_BLOCK for an id out of range, the pair skipped) and
 * streams as mi_kv_copy_blocks; one kernel launch. */
mi_status mi_kv_copy_rows(const void* src, int64_t src_count, const int32_t* src_ids, void* dst,
                          int64_t dst_count, const int32_t* dst_ids, int32_t n, int64_t row_bytes,
                          int32_t* dev_err, mi_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Allocation-free attention. The pages have no counterpart to this entry
 * point: it serves callers of this library that cannot call cudaMalloc (a
 * plugin whose host framework owns all device memory, a serving loop that
 * forbids allocator calls because they can synchronise the device, a process
 * held to a fixed device-memory budget). */

/* Size of the library's own scratch array (16 MiB, per GPU that loads the
 * library, held until the process exits). */
#define MI_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* mi_paged_decode_attention without a workspace argument: the split-KV
 * partials go to a fixed device array inside the library
 * (MI_NOALLOC_SCRATCH_BYTES). Same inputs, outputs, results and device error
 * bits as mi_paged_decode_attention. It calls no allocator.
 * Returns MI_ERR_UNSUPPORTED when the dims are not supported or need more
 * scratch than the array holds (mi_paged_decode_workspace_bytes(dims) >
 * MI_NOALLOC_SCRATCH_BYTES), before anything is queued.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture. The address is looked up again when the
 * device's context has changed (after a device reset, which also clears the
 * array). Every call on a device shares the one array and it keeps the last
 * call's contents; nothing in it needs to start at zero: each call tags the
 * merge counters it writes with its own epoch, so a counter left half-counted
 * by an earlier call (one that set MI_DEVERR_TIMEOUT) is ignored by the next.
 * Calls whose work overlaps on the GPU (other streams, other threads) race on
 * the array, so order them, e.g. on one stream. */
mi_status mi_paged_decode_attention_noalloc(const mi_dims* dims, const void* q,
                                            const void* k_cache, const void* v_cache,
                                            const int32_t* block_tables,
                                            const int32_t* context_lens, float scale, void* out,
                                            int32_t* dev_err, mi_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Failure-detection test hooks. Every mbarrier wait in the attention kernels
 * is bounded: when a staged copy or a partner warp does not arrive in time
 * the kernel ORs MI_DEVERR_TIMEOUT into *dev_err and returns instead of
 * hanging. These two process-wide settings let a test make such a wait run
 * out without faulting anything: they apply to every launch queued after the
 * call (not to launches already queued or captured), and a serving process
 * leaves them at their defaults. Not thread-safe against launches on other
 * host threads. */

/* Bound on each wait of later launches, in nanoseconds: 1 .. 2e9; 0 restores
 * the default (2 s). Waits for the launch's own copies or MMAs to finish
 * before it releases its memory keep a floor of 10 ms. MI_ERR_INVALID_ARG
 * outside 0 .. 2e9. */
mi_status mi_test_set_wait_limit(int64_t ns);

/* enable != 0: in later decode attention / fused step launches (bf16 and
 * e4m3), every CTA's producer neither copies nor announces the first block it
 * stages; in later tcgen05 prefill launches, every CTA's producer does so for
 * its first K stage. The waits on those stages then run out (set
 * MI_DEVERR_TIMEOUT) and the affected outputs are not valid. No copy is left
 * in flight. enable = 0 turns it off. Always MI_OK. */
mi_status mi_test_withhold_copy(int32_t enable);

#ifdef __cplusplus
}
#endif

#endif /* MI_H */
