// mi_paged_kv_append_int8: the decode append into INT8 KV caches quantised in
// groups of 64 tokens (nxmr.cn article, §2.2 "量化压缩的实战选择": 8-bit KV,
// quantised per 64-token group rather than per token, symmetric, scale =
// 127 / max|x|, the scaled values clamped to [-128, 127] and cast to int8,
// a cast that truncates toward zero; per head).
//
// A group is 64 consecutive tokens of one request and one KV head, over all
// dims, with K and V quantised separately. Its maximum m = max|x| (a bf16
// value, kept as fp32) is stored for every block of the group at
// amax[block][head]; a code c stands for c * m / 127. The last group of a
// request is open: its tokens keep their bf16 values in an open-group buffer
// [slot][Hkv][64][d] (one slot per sequence), and each new token is quantised
// with the group's current maximum. When the new row raises the maximum,
// every row of the group is quantised again from that buffer; otherwise only
// the new row is (with an unchanged maximum the other rows' codes come out
// the same), so a full group ends up quantised over its 64 tokens.
//
// One CTA per request, one warp per (KV head, K or V) item (8 to 16 warps;
// a warp takes a second item past 16):
// all threads rotate the request's q heads (RoPE as mi_paged_kv_append
// computes it, the same bits; each thread loads all its words before it
// stores any, so the loads overlap and q_out may alias q), then each warp
// takes its item: the new row (k rotated, v as given) into the open buffer,
// the row maximum by a warp reduction, and the codes of the new row or of
// the whole group. The open slot and the group's table entries are read
// before the q work, so their latency overlaps it.
#include "common.cuh"
#include "rope.cuh"

namespace mi {
namespace {

constexpr int kGroup = 64;
constexpr int kMaxThreads = 512;
constexpr int kQWords = 8;  // q words a thread holds at once
constexpr int kRequantRows = 16;  // open-buffer rows a lane loads at once when a group is quantised again
static_assert(kGroup % kRequantRows == 0, "a batch of rows never runs past the group's buffer");

struct Int8AppendParams {
    const uint16_t* q;             // [B][Hq][d] raw
    const uint16_t* k;             // [B][Hkv][d] raw
    const uint16_t* v;             // [B][Hkv][d]
    const float2* rope;            // [max_pos][d/2] (cos, sin)
    const int32_t* block_tables;   // [B][mbps]
    const int32_t* context_lens;   // [B], length after the append
    const int32_t* open_slots;     // [B]
    uint16_t* q_out;               // [B][Hq][d]
    int8_t* kc;                    // [num_blocks][Hkv][16][d]
    int8_t* vc;
    float* k_amax;                 // [num_blocks][Hkv]
    float* v_amax;
    uint16_t* k_open;              // [num_slots][Hkv][64][d]
    uint16_t* v_open;
    int32_t* dev_err;
    int Hq, Hkv, d, num_blocks, mbps, max_pos, num_slots;
};

// Code of one value with s = 127 / m: x * s in single precision, clamped to
// [-128, 127], truncated toward zero.
__device__ __forceinline__ uint32_t code_of(float x, float s) {
    const float y = fminf(fmaxf(__fmul_rn(x, s), -128.f), 127.f);
    return (uint32_t)__float2int_rz(y) & 0xFFu;
}

// Codes of a bf16 pair (one 32-bit word), first value in the low byte.
__device__ __forceinline__ uint32_t code_pair(uint32_t w, float s) {
    return code_of(bf16_lo(w), s) | (code_of(bf16_hi(w), s) << 8);
}

__device__ __forceinline__ float absmax_pair(uint32_t w) {
    return fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w)));
}

// g[j] for a run-time j < 4, without indexing the array in local memory.
__device__ __forceinline__ int pick4(const int (&g)[4], int j) {
    return j == 0 ? g[0] : (j == 1 ? g[1] : (j == 2 ? g[2] : g[3]));
}

__global__ void __launch_bounds__(kMaxThreads) append_int8_kernel(Int8AppendParams a) {
    // inputs may come from the kernel just before this one in the stream
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, half = d / 2, words = d / 4;  // words: 32-bit words per half row
    const int n = __ldg(a.context_lens + b);
    if (n <= 0) return;  // nothing to append
    const int p = n - 1;
    if (p >= a.max_pos || n > a.mbps * kBlock) {
        if (tid == 0) raise_err(a.dev_err, p >= a.max_pos ? MI_DEVERR_BAD_POS : MI_DEVERR_BAD_CONTEXT);
        return;
    }
    const float2* cs_row = a.rope + (long long)p * half;
    // read now, used after the q work
    const int slot = __ldg(a.open_slots + b);
    const int t0 = p / kGroup * kGroup, o = p - t0;  // the group's first token, the new token's offset
    const int j0 = t0 / kBlock, jp = p / kBlock;      // the group's first block, the new token's block
    const int32_t* bt = a.block_tables + (long long)b * a.mbps;
    int gblk[kGroup / kBlock];                        // the group's blocks so far
#pragma unroll
    for (int j = 0; j < kGroup / kBlock; ++j) gblk[j] = j0 + j <= jp ? __ldg(bt + j0 + j) : 0;

    // q heads: each word is one word of the first half and the matching word
    // of the second half of a head
    const int nq = a.Hq * words, nthr = blockDim.x;
    uint32_t xl[kQWords], xh[kQWords];
    float4 cs[kQWords];
#pragma unroll
    for (int k = 0; k < kQWords; ++k) {
        const int i = tid + k * nthr;
        if (i < nq) {
            const int head = i / words, w = i - head * words;
            const uint16_t* src = a.q + ((long long)b * a.Hq + head) * d;
            xl[k] = *reinterpret_cast<const uint32_t*>(src + 2 * w);
            xh[k] = *reinterpret_cast<const uint32_t*>(src + 2 * w + half);
            cs[k] = *reinterpret_cast<const float4*>(cs_row + 2 * w);
        }
    }
#pragma unroll
    for (int k = 0; k < kQWords; ++k) {
        const int i = tid + k * nthr;
        if (i < nq) {
            const int head = i / words, w = i - head * words;
            uint32_t yl, yh;
            if (rotate_word_fast(xl[k], xh[k], cs[k], yl, yh)) {
                const uint2 y = rotate_word_exact(xl[k], xh[k], cs[k]);
                yl = y.x;
                yh = y.y;
            }
            uint16_t* dst = a.q_out + ((long long)b * a.Hq + head) * d;
            *reinterpret_cast<uint32_t*>(dst + 2 * w) = yl;
            *reinterpret_cast<uint32_t*>(dst + 2 * w + half) = yh;
        }
    }
    // more q words than the threads hold at once (very wide heads): one at a time
    for (int i = tid + kQWords * nthr; i < nq; i += nthr) {
        const int head = i / words, w = i - head * words;
        const uint16_t* src = a.q + ((long long)b * a.Hq + head) * d;
        const uint32_t wl = *reinterpret_cast<const uint32_t*>(src + 2 * w);
        const uint32_t wh = *reinterpret_cast<const uint32_t*>(src + 2 * w + half);
        const float4 c4 = *reinterpret_cast<const float4*>(cs_row + 2 * w);
        uint32_t yl, yh;
        if (rotate_word_fast(wl, wh, c4, yl, yh)) {
            const uint2 y = rotate_word_exact(wl, wh, c4);
            yl = y.x;
            yh = y.y;
        }
        uint16_t* dst = a.q_out + ((long long)b * a.Hq + head) * d;
        *reinterpret_cast<uint32_t*>(dst + 2 * w) = yl;
        *reinterpret_cast<uint32_t*>(dst + 2 * w + half) = yh;
    }

    if (slot < 0 || slot >= a.num_slots) {
        if (tid == 0) raise_err(a.dev_err, MI_DEVERR_BAD_SLOT);
        return;
    }
    bool ok = true;
#pragma unroll
    for (int j = 0; j < kGroup / kBlock; ++j) ok &= j0 + j > jp || (gblk[j] >= 0 && gblk[j] < a.num_blocks);
    if (!ok) {
        if (tid == 0) raise_err(a.dev_err, MI_DEVERR_BAD_BLOCK);
        return;
    }

    // lane l owns words l (dims 2l, 2l+1) and l + words (dims half + 2l, +1)
    // of every row; lanes past `words` (d = 64) own nothing
    const bool own = lane < words;
    const int nw = blockDim.x >> 5;
    for (int item = warp; item < 2 * a.Hkv; item += nw) {
        const int h = item >> 1;
        const bool is_v = (item & 1) != 0;
        const long long nofs = ((long long)b * a.Hkv + h) * d;
        uint32_t yl = 0u, yh = 0u;
        if (own) {
            const uint16_t* src = (is_v ? a.v : a.k) + nofs;
            const uint32_t xl = *reinterpret_cast<const uint32_t*>(src + 2 * lane);
            const uint32_t xh = *reinterpret_cast<const uint32_t*>(src + 2 * lane + half);
            if (is_v) {
                yl = xl;
                yh = xh;
            } else {
                const float4 cs = *reinterpret_cast<const float4*>(cs_row + 2 * lane);
                if (rotate_word_fast(xl, xh, cs, yl, yh)) {
                    const uint2 y = rotate_word_exact(xl, xh, cs);
                    yl = y.x;
                    yh = y.y;
                }
            }
        }
        float* amax = is_v ? a.v_amax : a.k_amax;
        // the group's maximum so far (held by its first block), none for a new group
        const float m_old = o > 0 ? __ldcg(amax + (long long)gblk[0] * a.Hkv + h) : 0.f;
        uint16_t* grp = (is_v ? a.v_open : a.k_open) + ((long long)slot * a.Hkv + h) * kGroup * d;
        if (own) {
            *reinterpret_cast<uint32_t*>(grp + (long long)o * d + 2 * lane) = yl;
            *reinterpret_cast<uint32_t*>(grp + (long long)o * d + 2 * lane + half) = yh;
        }
        float rmax = own ? fmaxf(absmax_pair(yl), absmax_pair(yh)) : 0.f;
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, sh));
        int8_t* cache = is_v ? a.vc : a.kc;
        const float m = fmaxf(m_old, rmax);
        const float s = m > 0.f ? __fdiv_rn(127.f, m) : 0.f;  // m = 0: every code is 0
        if (o > 0 && m > m_old) {
            // the maximum grew: the whole group again, from its bf16 rows,
            // kRequantRows rows' loads in flight before their codes are
            // stored (one row at a time put o + 1 dependent trips to L2 on
            // the warp's path)
            __syncwarp();
            for (int tb = 0; tb <= o; tb += kRequantRows) {
                // rows tb .. tb + kRequantRows - 1 lie inside the group's
                // 64-row buffer (tb <= o < 64, kRequantRows divides 64), so
                // they load unconditionally; only rows up to o are stored
                uint32_t wl[kRequantRows], wh[kRequantRows];
#pragma unroll
                for (int u = 0; u < kRequantRows; ++u) {
                    const int t = tb + u;
                    if (own) {
                        wl[u] = *reinterpret_cast<const uint32_t*>(grp + (long long)t * d + 2 * lane);
                        wh[u] = *reinterpret_cast<const uint32_t*>(grp + (long long)t * d + 2 * lane + half);
                    }
                }
#pragma unroll
                for (int u = 0; u < kRequantRows; ++u) {
                    const int t = tb + u;
                    if (own && t <= o) {
                        const int blk = pick4(gblk, t / kBlock);
                        int8_t* row = cache + (((long long)blk * a.Hkv + h) * kBlock + (t0 + t) % kBlock) * d;
                        *reinterpret_cast<uint16_t*>(row + 2 * lane) = (uint16_t)code_pair(wl[u], s);
                        *reinterpret_cast<uint16_t*>(row + 2 * lane + half) = (uint16_t)code_pair(wh[u], s);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kGroup / kBlock; ++j)
                if (lane == j && j0 + j <= jp) amax[(long long)gblk[j] * a.Hkv + h] = m;
        } else {
            const int blk = pick4(gblk, jp - j0);
            int8_t* row = cache + (((long long)blk * a.Hkv + h) * kBlock + p % kBlock) * d;
            if (own) {
                *reinterpret_cast<uint16_t*>(row + 2 * lane) = (uint16_t)code_pair(yl, s);
                *reinterpret_cast<uint16_t*>(row + 2 * lane + half) = (uint16_t)code_pair(yh, s);
            }
            if (lane == 0) amax[(long long)blk * a.Hkv + h] = m;  // a new block of the group gets m too
        }
    }
}

// ------------------------------------------------- many tokens per request --
// mi_paged_kv_append_int8_tokens: request r's m = query_start[r+1] -
// query_start[r] new tokens at positions n - m .. n - 1 (n = context_lens[r],
// counting them), with the result of m decode appends in order: every group
// the new tokens touch is quantised over all its tokens (the open group's
// earlier ones from the open buffer), and the last group's new rows join the
// open buffer. One CTA per (request, KV head, K or V), eight warps; the G
// query heads of the KV head are rotated by its K and V CTAs, half each.

constexpr int kTokThreads = 256;
constexpr int kTokWarps = kTokThreads / 32;
constexpr int kRowsPerWarp = kGroup / kTokWarps;  // rows of a group per warp
constexpr int kQBatch = 8;                          // q words a thread loads before it stores

struct Int8TokParams {
    const uint16_t* q;             // [T][Hq][d] raw
    const uint16_t* k;             // [T][Hkv][d] raw
    const uint16_t* v;             // [T][Hkv][d]
    const float2* rope;
    const int32_t* block_tables;   // [R][mbps]
    const int32_t* context_lens;   // [R]
    const int32_t* query_start;    // [R + 1]
    const int32_t* open_slots;     // [R]
    uint16_t* q_out;               // [T][Hq][d]
    int8_t* kc;
    int8_t* vc;
    float* k_amax;
    float* v_amax;
    uint16_t* k_open;
    uint16_t* v_open;
    int32_t* dev_err;
    int Hq, Hkv, d, num_blocks, mbps, max_pos, num_slots, T;
};

__global__ void __launch_bounds__(kTokThreads) append_int8_tokens_kernel(Int8TokParams a) {
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = blockIdx.x / (2 * a.Hkv), h = (blockIdx.x >> 1) % a.Hkv;
    const bool is_v = (blockIdx.x & 1) != 0;
    const bool reporter = tid == 0 && blockIdx.x % (2 * a.Hkv) == 0;  // one error report per request
    const int d = a.d, half = d / 2, words = d / 4;
    const int n = __ldg(a.context_lens + r);
    const int q0 = __ldg(a.query_start + r), q1 = __ldg(a.query_start + r + 1);
    const int m = q1 - q0;
    if (q0 < 0 || q1 < q0 || q1 > a.T || m > (n > 0 ? n : 0)) {
        if (reporter) raise_err(a.dev_err, MI_DEVERR_BAD_QUERY);
        return;
    }
    if (m == 0) return;  // nothing to append
    if (n > a.mbps * kBlock || n - 1 >= a.max_pos) {
        if (reporter) raise_err(a.dev_err, n - 1 >= a.max_pos ? MI_DEVERR_BAD_POS : MI_DEVERR_BAD_CONTEXT);
        return;
    }
    const int p0 = n - m;

    // q rows of this CTA's share of the KV head's query heads, a batch of
    // words loaded per thread before any is stored (q_out may alias q)
    const int G = a.Hq / a.Hkv, gk = (G + 1) / 2;
    const int hq0 = h * G + (is_v ? gk : 0), nh = is_v ? G - gk : gk;
    const long long nqw = (long long)m * nh * words;
    for (long long i0 = tid; i0 < nqw; i0 += (long long)kQBatch * kTokThreads) {
        uint32_t xl[kQBatch], xh[kQBatch];
        float4 cs[kQBatch];
        long long ofs[kQBatch];
#pragma unroll
        for (int u = 0; u < kQBatch; ++u) {
            const long long i = i0 + (long long)u * kTokThreads;
            ofs[u] = -1;
            if (i < nqw) {
                const int w = (int)(i % words);
                const long long rest = i / words;
                const int hh = (int)(rest % nh), tok = (int)(rest / nh);
                ofs[u] = ((long long)(q0 + tok) * a.Hq + hq0 + hh) * d + 2 * w;
                xl[u] = *reinterpret_cast<const uint32_t*>(a.q + ofs[u]);
                xh[u] = *reinterpret_cast<const uint32_t*>(a.q + ofs[u] + half);
                cs[u] = *reinterpret_cast<const float4*>(a.rope + (long long)(p0 + tok) * half + 2 * w);
            }
        }
#pragma unroll
        for (int u = 0; u < kQBatch; ++u) {
            if (ofs[u] < 0) continue;
            uint32_t yl, yh;
            if (rotate_word_fast(xl[u], xh[u], cs[u], yl, yh)) {
                const uint2 y = rotate_word_exact(xl[u], xh[u], cs[u]);
                yl = y.x;
                yh = y.y;
            }
            *reinterpret_cast<uint32_t*>(a.q_out + ofs[u]) = yl;
            *reinterpret_cast<uint32_t*>(a.q_out + ofs[u] + half) = yh;
        }
    }

    const int slot = __ldg(a.open_slots + r);
    if (slot < 0 || slot >= a.num_slots) {
        if (reporter) raise_err(a.dev_err, MI_DEVERR_BAD_SLOT);
        return;
    }
    const int32_t* bt = a.block_tables + (long long)r * a.mbps;
    // every block of the groups the new tokens touch must be valid
    const int jfirst = p0 / kGroup * (kGroup / kBlock), jlast = (n - 1) / kBlock;
    bool ok = true;
    for (int j = jfirst + tid; j <= jlast; j += kTokThreads) {
        const int blk = __ldg(bt + j);
        ok &= blk >= 0 && blk < a.num_blocks;
    }
    if (!__syncthreads_and(ok)) {
        if (reporter) raise_err(a.dev_err, MI_DEVERR_BAD_BLOCK);
        return;
    }

    __shared__ float wmax[kTokWarps];
    uint16_t* grp = (is_v ? a.v_open : a.k_open) + ((long long)slot * a.Hkv + h) * kGroup * d;
    const uint16_t* in = is_v ? a.v : a.k;
    float* amax = is_v ? a.v_amax : a.k_amax;
    int8_t* cache = is_v ? a.vc : a.kc;
    const bool own = lane < words;  // lane l owns words l and l + words of every row
    for (int g = p0 / kGroup; g <= (n - 1) / kGroup; ++g) {
        const int t0 = g * kGroup, te = min(t0 + kGroup, n);
        uint32_t xl[kRowsPerWarp], xh[kRowsPerWarp];
        float lmax = 0.f;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int t = t0 + warp + kTokWarps * i;
            xl[i] = xh[i] = 0u;
            if (t < te && own) {
                if (t < p0) {
                    // a token of the open group from before this call: its bf16 row
                    const uint16_t* row = grp + (long long)(t - t0) * d;
                    xl[i] = *reinterpret_cast<const uint32_t*>(row + 2 * lane);
                    xh[i] = *reinterpret_cast<const uint32_t*>(row + 2 * lane + half);
                } else {
                    const uint16_t* row = in + ((long long)(q0 + t - p0) * a.Hkv + h) * d;
                    const uint32_t wl = *reinterpret_cast<const uint32_t*>(row + 2 * lane);
                    const uint32_t wh = *reinterpret_cast<const uint32_t*>(row + 2 * lane + half);
                    if (is_v) {
                        xl[i] = wl;
                        xh[i] = wh;
                    } else {
                        const float4 c4 = *reinterpret_cast<const float4*>(a.rope + (long long)t * half + 2 * lane);
                        uint32_t yl, yh;
                        if (rotate_word_fast(wl, wh, c4, yl, yh)) {
                            const uint2 y = rotate_word_exact(wl, wh, c4);
                            yl = y.x;
                            yh = y.y;
                        }
                        xl[i] = yl;
                        xh[i] = yh;
                    }
                }
                lmax = fmaxf(lmax, fmaxf(absmax_pair(xl[i]), absmax_pair(xh[i])));
            }
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, sh));
        if (lane == 0) wmax[warp] = lmax;
        __syncthreads();
        float mx = 0.f;
#pragma unroll
        for (int w = 0; w < kTokWarps; ++w) mx = fmaxf(mx, wmax[w]);
        const float sc = mx > 0.f ? __fdiv_rn(127.f, mx) : 0.f;  // m = 0: every code is 0
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int t = t0 + warp + kTokWarps * i;
            if (t < te && own) {
                const int blk = __ldg(bt + t / kBlock);
                int8_t* row = cache + (((long long)blk * a.Hkv + h) * kBlock + t % kBlock) * d;
                *reinterpret_cast<uint16_t*>(row + 2 * lane) = (uint16_t)code_pair(xl[i], sc);
                *reinterpret_cast<uint16_t*>(row + 2 * lane + half) = (uint16_t)code_pair(xh[i], sc);
                if (te == n && t >= p0) {
                    // the request's last group stays open: its new rows join the buffer
                    uint16_t* orow = grp + (long long)(t - t0) * d;
                    *reinterpret_cast<uint32_t*>(orow + 2 * lane) = xl[i];
                    *reinterpret_cast<uint32_t*>(orow + 2 * lane + half) = xh[i];
                }
            }
        }
        for (int j = t0 / kBlock + tid; j <= (te - 1) / kBlock; j += kTokThreads)
            amax[(long long)__ldg(bt + j) * a.Hkv + h] = mx;
        __syncthreads();  // wmax and the buffer rows are reused by the next group
    }
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace
}  // namespace mi

extern "C" mi_status mi_paged_kv_append_int8(const mi_dims* dims, const void* q, const void* k, const void* v,
                                             const float* rope_cos_sin, int32_t max_pos,
                                             const int32_t* block_tables, const int32_t* context_lens,
                                             const int32_t* open_slots, int32_t num_open_slots, void* q_out,
                                             void* k_cache, void* v_cache, float* k_amax, float* v_amax,
                                             void* k_open, void* v_open, int32_t* dev_err, mi_stream_t stream) {
    using namespace mi;
    if (!dims) return MI_ERR_INVALID_ARG;
    const mi_dims D = *dims;
    if (D.B < 0 || D.B > 0x7FFFFFFF || D.Hq < 1 || D.Hkv < 1 || D.num_blocks < 1 || D.max_blocks_per_seq < 1 ||
        max_pos < 1 || num_open_slots < 1)
        return MI_ERR_INVALID_ARG;
    if (D.block_size != kBlock || (D.head_dim != 64 && D.head_dim != 128) || D.Hq % D.Hkv != 0)
        return MI_ERR_UNSUPPORTED;
    if ((long long)D.num_blocks * D.Hkv * kBlock * D.head_dim > (1LL << 46)) return MI_ERR_INVALID_ARG;
    if (D.B == 0) return MI_OK;
    if (!q || !k || !v || !rope_cos_sin || !block_tables || !context_lens || !open_slots || !q_out || !k_cache ||
        !v_cache || !k_amax || !v_amax || !k_open || !v_open)
        return MI_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_out, 16) || !aligned(rope_cos_sin, 16) ||
        !aligned(k_open, 16) || !aligned(v_open, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(k_amax, 4) || !aligned(v_amax, 4))
        return MI_ERR_INVALID_ARG;
    Int8AppendParams a;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.rope = reinterpret_cast<const float2*>(rope_cos_sin);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.open_slots = open_slots;
    a.q_out = static_cast<uint16_t*>(q_out);
    a.kc = static_cast<int8_t*>(k_cache);
    a.vc = static_cast<int8_t*>(v_cache);
    a.k_amax = k_amax;
    a.v_amax = v_amax;
    a.k_open = static_cast<uint16_t*>(k_open);
    a.v_open = static_cast<uint16_t*>(v_open);
    a.dev_err = dev_err;
    a.Hq = D.Hq;
    a.Hkv = D.Hkv;
    a.d = D.head_dim;
    a.num_blocks = D.num_blocks;
    a.mbps = D.max_blocks_per_seq;
    a.max_pos = max_pos;
    a.num_slots = num_open_slots;
    // one warp per (KV head, K or V) item, at least 8 warps for the q work,
    // at most 16
    const int warps = 2 * D.Hkv < 8 ? 8 : (2 * D.Hkv > kMaxThreads / 32 ? kMaxThreads / 32 : 2 * D.Hkv);
    const cudaError_t e = launch_pdl(append_int8_kernel, (int)D.B, warps * 32, 0, (cudaStream_t)stream, a);
    return e == cudaSuccess ? MI_OK : MI_ERR_CUDA;
}

extern "C" mi_status mi_paged_kv_append_int8_tokens(const mi_dims* dims, int32_t total_tokens, const void* q,
                                                    const void* k, const void* v, const float* rope_cos_sin,
                                                    int32_t max_pos, const int32_t* block_tables,
                                                    const int32_t* context_lens, const int32_t* query_start,
                                                    const int32_t* open_slots, int32_t num_open_slots, void* q_out,
                                                    void* k_cache, void* v_cache, float* k_amax, float* v_amax,
                                                    void* k_open, void* v_open, int32_t* dev_err,
                                                    mi_stream_t stream) {
    using namespace mi;
    if (!dims) return MI_ERR_INVALID_ARG;
    const mi_dims D = *dims;
    if (D.B < 0 || D.Hq < 1 || D.Hkv < 1 || D.num_blocks < 1 || D.max_blocks_per_seq < 1 || max_pos < 1 ||
        num_open_slots < 1 || total_tokens < 0)
        return MI_ERR_INVALID_ARG;
    if (D.block_size != kBlock || (D.head_dim != 64 && D.head_dim != 128) || D.Hq % D.Hkv != 0)
        return MI_ERR_UNSUPPORTED;
    if ((long long)D.B * 2 * D.Hkv > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;
    if (D.B == 0 || total_tokens == 0) return MI_OK;
    if (!q || !k || !v || !rope_cos_sin || !block_tables || !context_lens || !query_start || !open_slots ||
        !q_out || !k_cache || !v_cache || !k_amax || !v_amax || !k_open || !v_open)
        return MI_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_out, 16) || !aligned(rope_cos_sin, 16) ||
        !aligned(k_open, 16) || !aligned(v_open, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(k_amax, 4) || !aligned(v_amax, 4))
        return MI_ERR_INVALID_ARG;
    Int8TokParams a;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.rope = reinterpret_cast<const float2*>(rope_cos_sin);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.open_slots = open_slots;
    a.q_out = static_cast<uint16_t*>(q_out);
    a.kc = static_cast<int8_t*>(k_cache);
    a.vc = static_cast<int8_t*>(v_cache);
    a.k_amax = k_amax;
    a.v_amax = v_amax;
    a.k_open = static_cast<uint16_t*>(k_open);
    a.v_open = static_cast<uint16_t*>(v_open);
    a.dev_err = dev_err;
    a.Hq = D.Hq;
    a.Hkv = D.Hkv;
    a.d = D.head_dim;
    a.num_blocks = D.num_blocks;
    a.mbps = D.max_blocks_per_seq;
    a.max_pos = max_pos;
    a.num_slots = num_open_slots;
    a.T = total_tokens;
    const cudaError_t e =
        launch_pdl(append_int8_tokens_kernel, (int)(D.B * 2 * D.Hkv), kTokThreads, 0, (cudaStream_t)stream, a);
    return e == cudaSuccess ? MI_OK : MI_ERR_CUDA;
}
