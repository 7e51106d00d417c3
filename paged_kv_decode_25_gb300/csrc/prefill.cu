// mi_paged_prefill_attention: causal GQA attention of many new tokens per
// request over the paged KV cache — the prefill step of the NJU course brief
// "端侧大模型推理框架" §2.1 (the prefill + decode main loop) and of the
// mini-infer README "项目概述" (prefill as its own forward pass), here also
// serving chunked prefill: the new tokens of request r are its last m_r
// context positions, n_r - m_r .. n_r - 1, and token n_r - m_r + i attends to
// cached tokens 0 .. n_r - m_r + i.
//
// Work decomposition:
//   * Rows are (new token i, query head g of the GQA group) pairs, row index
//     i * G + g, so one staged K/V tile serves every head of the group. A CTA
//     owns 64 consecutive rows of one (request, KV head); its 4 consumer warps
//     own 16 rows each.
//   * One producer warp walks the block table and streams 64-key stages (four
//     16-token blocks, one 4 KB 2-D TMA box per K or V tile, 128-byte swizzle)
//     through a 3-stage ring shared by the consumer warps (full barrier: one
//     arrival plus the copied bytes; empty barrier: one arrival per consumer
//     warp).
//   * Consumer warp tile (mma.sync m16n8k16, bf16 in, fp32 accumulate):
//     S[16 rows x 64 keys] = Q . K^T with Q held in registers as A fragments
//     and K read by ldmatrix as B fragments; causal mask and base-2 online
//     softmax on the accumulator fragments; the probabilities are repacked in
//     place as bf16 A fragments and O[16 x HD] += P . V with V read by
//     ldmatrix.trans.
//   * Grid: one CTA per (request r, KV head h, row tile k counted from the
//     request's end). Tiles come in groups of 8 consecutive k per (r, h), and
//     the groups run k-group by k-group over all (r, h): the hardware starts
//     the tiles with the most keys first, as a longest-first schedule wants,
//     while the 8 tiles of a group read the same K/V through L2 at about the
//     same time. Tiles past a request's last row exit at once.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "tma.cuh"

namespace mi {
namespace {

constexpr int kPWarps = 4;                      // consumer warps
constexpr int kPRows = kPWarps * 16;            // rows per CTA
constexpr int kStageBlocks = 4;                 // 16-token blocks per stage: 64 keys
constexpr int kSubBlocks = 2;                   // blocks per softmax sub-step: 32 keys
constexpr int kPStages = 3;
constexpr int kMaxGroup = 8;
constexpr int kTileGroup = 8;                   // row tiles of one (request, head) launched together

struct PrefillParams {
    const uint16_t* q;             // [T][Hq][HD], RoPE applied
    const int32_t* block_tables;   // [R][mbps]
    const int32_t* context_lens;   // [R], counting the new tokens
    const int32_t* query_start;    // [R + 1]
    uint16_t* out;                 // [T][Hq][HD]
    int32_t* dev_err;
    int R, Hq, Hkv, G, num_blocks, mbps, T, max_q;
    float sl2;                     // scale * log2(e)
};

template <int HD>
struct PrefillSmem {
    static constexpr int kTile = kBlock * HD * 2;                     // one 16-token K or V tile
    static constexpr int kStage = kStageBlocks * 2 * kTile;           // K and V of four blocks
    static constexpr int kFull = kPStages * kStage;
    static constexpr int kEmpty = kFull + kPStages * 8;
    static constexpr int kMask = kEmpty + kPStages * 8;
    static constexpr int kTotal = kMask + kPStages * 4 + 1024;        // slack: tiles start on 1024 bytes
};

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

template <int HD>
__global__ void __launch_bounds__((kPWarps + 1) * 32, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   PrefillParams p) {
    using SM = PrefillSmem<HD>;
    constexpr int kTile = SM::kTile;
    constexpr int kK = HD / 16;  // k-slices of Q . K^T
    constexpr int kN = HD / 8;   // 8-column tiles of O
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t full0 = sbase + SM::kFull, empty0 = sbase + SM::kEmpty, mask0 = sbase + SM::kMask;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // q, the tables and the lengths may come from the kernel before this one
    pdl_wait();
    pdl_trigger();

    // ------------------------------------------------------- work item ----
    const int kw = blockIdx.x % kTileGroup;
    const int rest0 = blockIdx.x / kTileGroup;
    const int h = rest0 % p.Hkv;
    const int rest = rest0 / p.Hkv;
    const int r = rest % p.R;
    const int k = (rest / p.R) * kTileGroup + kw;
    const bool reporter = k == 0 && h == 0 && threadIdx.x == 0;  // one error report per request
    const int q0 = __ldg(p.query_start + r), q1 = __ldg(p.query_start + r + 1);
    const int m = q1 - q0;
    if (q0 < 0 || q1 > p.T || m < 0 || m > p.max_q) {
        if (reporter) raise_err(p.dev_err, MI_DEVERR_BAD_QUERY);
        return;
    }
    const int nrows = m * p.G;
    const int tiles = (nrows + kPRows - 1) / kPRows;
    if (k >= tiles) return;
    int n = __ldg(p.context_lens + r);
    if (n > p.mbps * kBlock) {
        if (reporter) raise_err(p.dev_err, MI_DEVERR_BAD_CONTEXT);
        n = p.mbps * kBlock;
    }
    if (m > n && reporter) raise_err(p.dev_err, MI_DEVERR_BAD_QUERY);
    const int first = n - m;  // position of new token 0 (negative only when m > n)
    const int rho0 = (tiles - 1 - k) * kPRows;
    const int rows_here = min(kPRows, nrows - rho0);
    const int p_hi = first + (rho0 + rows_here - 1) / p.G;  // position of the CTA's last row
    const int nblk = p_hi >= 0 ? p_hi / kBlock + 1 : 0;    // blocks any row of the CTA reads
    const int nst = (nblk + kStageBlocks - 1) / kStageBlocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(full0 + s * 8, 1);
            mbar_init(empty0 + s * 8, kPWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kPWarps) {
        // ------------------------------------------------ producer warp --
        // Lanes 0..3 look up and copy the four blocks of a stage; lane 0 posts
        // the stage's block mask and byte count.
        const uint64_t policy = l2_policy_evict_normal();  // other row tiles of the request re-read these
        uint32_t stg = 0, ph = 1;  // a fresh barrier reads as having completed the phase before 0
        int issued = 0;
        for (int j = 0; j < nst; ++j) {
            // every lane waits; the warp gives up together if any lane ran out of
            // time (a consumer stopped taking stages: it timed out itself)
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(empty0 + stg * 8, ph))) {
                if (lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
                break;
            }
            const int x = j * kStageBlocks + lane;
            int blk = -1;
            bool ok = false;
            if (lane < kStageBlocks && x < nblk) {
                blk = __ldg(p.block_tables + (long long)r * p.mbps + x);
                ok = blk >= 0 && blk < p.num_blocks;
                if (!ok) raise_err(p.dev_err, MI_DEVERR_BAD_BLOCK);
            }
            const uint32_t msk = __ballot_sync(0xffffffffu, ok);
            const uint32_t bar = full0 + stg * 8;
            if (lane == 0) {
                sts_u32(mask0 + stg * 4, msk);
                mbar_arrive_expect_tx(bar, (uint32_t)__popc(msk) * 2u * kTile);
            }
            __syncwarp();
            if (ok) {
                const uint32_t dst = sbase + stg * SM::kStage + (uint32_t)lane * 2u * kTile;
                const int y = ((blk * p.Hkv + h) * kBlock) * (HD / 64);
                tma_load_2d(dst, &tmk, bar, 0, y, policy);
                tma_load_2d(dst + kTile, &tmv, bar, 0, y, policy);
            }
            ++issued;
            if (++stg == (uint32_t)kPStages) {
                stg = 0;
                ph ^= 1u;
            }
        }
        // Every copy issued must land before the CTA's shared memory goes away
        // (a no-op unless a consumer gave up early).
        if (lane == 0) {
            for (int s = 0; s < kPStages && s < issued; ++s) {
                const int fills = (issued - s + kPStages - 1) / kPStages;
                (void)mbar_wait_bounded(full0 + s * 8, (uint32_t)((fills - 1) & 1));
            }
        }
        return;
    }

    // --------------------------------------------------- consumer warps ----
    const int c = lane & 3;
    const int wr0 = rho0 + warp * 16;                  // first row of this warp
    const int rA = wr0 + (lane >> 2), rB = rA + 8;     // this thread's two rows
    const bool vA = rA < nrows, vB = rB < nrows;
    const int iA = rA / p.G, iB = rB / p.G;
    const int posA = vA ? first + iA : p_hi, posB = vB ? first + iB : p_hi;
    const int mposA = posA < 0 ? 0 : posA, mposB = posB < 0 ? 0 : posB;  // masking positions
    const int w_last = min(wr0 + 15, rho0 + rows_here - 1);
    const int pw_hi = w_last >= wr0 ? first + w_last / p.G : -1;
    const int pw_lo = first + wr0 / p.G;
    const int nblk_w = pw_hi >= 0 ? pw_hi / kBlock + 1 : 0;  // blocks this warp reads
    const int nb_ctx = (n + kBlock - 1) / kBlock;
    const int tail = n - (nb_ctx - 1) * kBlock;              // valid tokens in the context's last block

    // Q rows as A fragments (zero for rows past the request's last token)
    uint32_t qa[kK][4];
    {
        const long long headA = (long long)(q0 + (vA ? iA : 0)) * p.Hq + (long long)h * p.G + rA % p.G;
        const long long headB = (long long)(q0 + (vB ? iB : 0)) * p.Hq + (long long)h * p.G + rB % p.G;
        const uint32_t* qA = reinterpret_cast<const uint32_t*>(p.q + headA * HD);
        const uint32_t* qB = reinterpret_cast<const uint32_t*>(p.q + headB * HD);
#pragma unroll
        for (int ks = 0; ks < kK; ++ks) {
            qa[ks][0] = vA ? __ldg(qA + ks * 8 + c) : 0u;
            qa[ks][1] = vB ? __ldg(qB + ks * 8 + c) : 0u;
            qa[ks][2] = vA ? __ldg(qA + ks * 8 + 4 + c) : 0u;
            qa[ks][3] = vB ? __ldg(qB + ks * 8 + 4 + c) : 0u;
        }
    }

    float o[kN][4];
#pragma unroll
    for (int t = 0; t < kN; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    // ldmatrix lane addressing inside a staged tile
    const int k_key = ((lane >> 4) << 3) + (lane & 7), k_chk = (lane >> 3) & 1;   // K as B of Q.K^T
    const int v_key = (((lane >> 3) & 1) << 3) + (lane & 7), v_chk = lane >> 4;   // V as B of P.V

    uint32_t stg = 0, ph = 0;
    bool dead = false;
    for (int j = 0; j < nst; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(full0 + stg * 8, ph))) {
            if (lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
            dead = true;
            break;
        }
        const uint32_t present = lds_u32(mask0 + stg * 4);
        uint32_t used = 0;  // blocks of the stage this warp multiplies
#pragma unroll
        for (int l = 0; l < kStageBlocks; ++l)
            if (((present >> l) & 1u) && j * kStageBlocks + l < nblk_w) used |= 1u << l;
        // two 32-key sub-steps per stage keep the score and probability
        // fragments of only two blocks live at a time
#pragma unroll
        for (int hs = 0; hs < kStageBlocks / kSubBlocks; ++hs) {
            const uint32_t sub = (used >> (hs * kSubBlocks)) & ((1u << kSubBlocks) - 1u);
            if (!sub) continue;
            const int jb = j * kStageBlocks + hs * kSubBlocks;  // request block index of the first block
            const uint32_t sub_base = sbase + stg * SM::kStage + (uint32_t)(hs * kSubBlocks) * 2u * kTile;
            float s[kSubBlocks][2][4];
#pragma unroll
            for (int l = 0; l < kSubBlocks; ++l) {
#pragma unroll
                for (int e = 0; e < 4; ++e) s[l][0][e] = s[l][1][e] = 0.f;
                if (sub & (1u << l)) {
                    const uint32_t kt = sub_base + (uint32_t)l * 2u * kTile;
#pragma unroll
                    for (int ks = 0; ks < kK; ++ks) {
                        uint32_t b00, b01, b10, b11;
                        ldsm_x4(kt + swz<HD>(k_key, 2 * ks + k_chk), b00, b01, b10, b11);
                        mma_bf16_16816(s[l][0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
                        mma_bf16_16816(s[l][1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
                    }
                }
            }
            // scale to base 2, mask (blocks not multiplied, keys after a row's position)
            const int kbase = jb * kBlock;
            const bool causal = kbase + kSubBlocks * kBlock - 1 > pw_lo;
            float xA = -INFINITY, xB = -INFINITY;
#pragma unroll
            for (int l = 0; l < kSubBlocks; ++l) {
                const bool on = (sub >> l) & 1u;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = kbase + l * kBlock + t * 8 + 2 * c + (e & 1);
                        const int pos = e < 2 ? mposA : mposB;
                        const bool keep = on && (!causal || key <= pos);
                        s[l][t][e] = keep ? s[l][t][e] * p.sl2 : -INFINITY;
                    }
                    xA = fmaxf(xA, fmaxf(s[l][t][0], s[l][t][1]));
                    xB = fmaxf(xB, fmaxf(s[l][t][2], s[l][t][3]));
                }
            }
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 1));
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 2));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 1));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 2));
            const float nA = fmaxf(mA, xA), nB = fmaxf(mB, xB);
            const float uA = nA == -INFINITY ? 0.f : nA, uB = nB == -INFINITY ? 0.f : nB;
            const float aA = exp2f(mA - uA), aB = exp2f(mB - uB);
            mA = nA;
            mB = nB;
            if (__any_sync(0xffffffffu, aA != 1.f || aB != 1.f)) {
#pragma unroll
                for (int t = 0; t < kN; ++t) {
                    o[t][0] *= aA;
                    o[t][1] *= aA;
                    o[t][2] *= aB;
                    o[t][3] *= aB;
                }
            }
            lA *= aA;
            lB *= aB;
            // probabilities, repacked as the A fragments of P . V (16 keys per block)
            uint32_t pa[kSubBlocks][4];
#pragma unroll
            for (int l = 0; l < kSubBlocks; ++l) {
                float e[2][4];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    e[t][0] = exp2f(s[l][t][0] - uA);
                    e[t][1] = exp2f(s[l][t][1] - uA);
                    e[t][2] = exp2f(s[l][t][2] - uB);
                    e[t][3] = exp2f(s[l][t][3] - uB);
                    lA += e[t][0] + e[t][1];
                    lB += e[t][2] + e[t][3];
                }
                pa[l][0] = pack_bf16x2(e[0][0], e[0][1]);
                pa[l][1] = pack_bf16x2(e[0][2], e[0][3]);
                pa[l][2] = pack_bf16x2(e[1][0], e[1][1]);
                pa[l][3] = pack_bf16x2(e[1][2], e[1][3]);
            }
#pragma unroll
            for (int l = 0; l < kSubBlocks; ++l) {
                if (!(sub & (1u << l))) continue;
                const uint32_t vt = sub_base + (uint32_t)l * 2u * kTile + kTile;
                // keys past the context in its last block may hold any bits: zero them
                uint32_t zlo = 0xFFFFFFFFu, zhi = 0xFFFFFFFFu;
                if (jb + l == nb_ctx - 1 && tail < kBlock) {
                    const int k0 = 2 * c;
                    zlo = (k0 < tail ? 0x0000FFFFu : 0u) | (k0 + 1 < tail ? 0xFFFF0000u : 0u);
                    zhi = (k0 + 8 < tail ? 0x0000FFFFu : 0u) | (k0 + 9 < tail ? 0xFFFF0000u : 0u);
                }
#pragma unroll
                for (int dp = 0; dp < kN / 2; ++dp) {
                    uint32_t v0, v1, v2, v3;
                    ldsm_x4_trans(vt + swz<HD>(v_key, 2 * dp + v_chk), v0, v1, v2, v3);
                    v0 &= zlo;
                    v2 &= zlo;
                    v1 &= zhi;
                    v3 &= zhi;
                    mma_bf16_16816(o[2 * dp], pa[l][0], pa[l][1], pa[l][2], pa[l][3], v0, v1);
                    mma_bf16_16816(o[2 * dp + 1], pa[l][0], pa[l][1], pa[l][2], pa[l][3], v2, v3);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + stg * 8);
        if (++stg == (uint32_t)kPStages) {
            stg = 0;
            ph ^= 1u;
        }
    }
    if (dead) return;

    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    // rows before position 0 (more new tokens than context) are +0
    const uint32_t keepA = posA >= 0 ? 0xFFFFFFFFu : 0u, keepB = posB >= 0 ? 0xFFFFFFFFu : 0u;
    const float invA = lA > 0.f ? 1.f / lA : 0.f;
    const float invB = lB > 0.f ? 1.f / lB : 0.f;
    if (vA) {
        uint32_t* row = reinterpret_cast<uint32_t*>(
            p.out + ((long long)(q0 + iA) * p.Hq + (long long)h * p.G + rA % p.G) * HD);
#pragma unroll
        for (int t = 0; t < kN; ++t) row[t * 4 + c] = pack_bf16x2(o[t][0] * invA, o[t][1] * invA) & keepA;
    }
    if (vB) {
        uint32_t* row = reinterpret_cast<uint32_t*>(
            p.out + ((long long)(q0 + iB) * p.Hq + (long long)h * p.G + rB % p.G) * HD);
#pragma unroll
        for (int t = 0; t < kN; ++t) row[t * 4 + c] = pack_bf16x2(o[t][2] * invB, o[t][3] * invB) & keepB;
    }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <int HD>
bool prepare(int* smem) {
    // raise the kernel's dynamic shared-memory limit once per device
    static std::mutex mu;
    static bool done[256] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return false;
    *smem = PrefillSmem<HD>::kTotal;
    std::lock_guard<std::mutex> lk(mu);
    if (!done[dev]) {
        if (cudaFuncSetAttribute(reinterpret_cast<const void*>(prefill_kernel<HD>),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, *smem) != cudaSuccess)
            return false;
        done[dev] = true;
    }
    return true;
}

}  // namespace
}  // namespace mi

extern "C" mi_status mi_paged_prefill_attention(const mi_dims* dims, int32_t total_q, int32_t max_query_len,
                                                const void* q, const void* k_cache, const void* v_cache,
                                                const int32_t* block_tables, const int32_t* context_lens,
                                                const int32_t* query_start, float scale, void* out,
                                                int32_t* dev_err, mi_stream_t stream) {
    using namespace mi;
    if (!dims) return MI_ERR_INVALID_ARG;
    const mi_dims D = *dims;
    if (D.B < 0 || D.Hq < 1 || D.Hkv < 1 || D.num_blocks < 1 || D.max_blocks_per_seq < 1 || total_q < 0 ||
        max_query_len < 0)
        return MI_ERR_INVALID_ARG;
    if (D.block_size != kBlock || (D.head_dim != 64 && D.head_dim != 128) || D.Hq % D.Hkv != 0 ||
        D.Hq / D.Hkv > kMaxGroup)
        return MI_ERR_UNSUPPORTED;
    if ((long long)D.num_blocks * D.Hkv * kBlock * (D.head_dim / 64) > 0x7FFFFFFFLL ||
        (long long)D.max_blocks_per_seq * kBlock > 0x7FFFFFFFLL || (long long)total_q * D.Hq > 0x7FFFFFFFLL ||
        (long long)max_query_len * D.Hq > 0x7FFFFFFFLL)
        return MI_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return MI_ERR_INVALID_ARG;
    if (D.B == 0 || total_q == 0 || max_query_len == 0) return MI_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out)
        return MI_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache))
        return MI_ERR_INVALID_ARG;
    const int G = D.Hq / D.Hkv, HD = D.head_dim;
    const long long tiles_max = ((long long)max_query_len * G + kPRows - 1) / kPRows;
    const long long grid = (tiles_max + kTileGroup - 1) / kTileGroup * kTileGroup * D.B * D.Hkv;
    if (grid > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;

    int smem = 0;
    if (!(HD == 64 ? prepare<64>(&smem) : prepare<128>(&smem))) return MI_ERR_CUDA;
    CUtensorMap tk, tv;
    const long long rows = (long long)D.num_blocks * D.Hkv * kBlock;
    if (!make_tmap(&tk, k_cache, rows, HD) || !make_tmap(&tv, v_cache, rows, HD)) return MI_ERR_CUDA;

    PrefillParams p;
    p.q = static_cast<const uint16_t*>(q);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.query_start = query_start;
    p.out = static_cast<uint16_t*>(out);
    p.dev_err = dev_err;
    p.R = D.B;
    p.Hq = D.Hq;
    p.Hkv = D.Hkv;
    p.G = G;
    p.num_blocks = D.num_blocks;
    p.mbps = D.max_blocks_per_seq;
    p.T = total_q;
    p.max_q = max_query_len;
    p.sl2 = scale * 1.4426950408889634f;
    const cudaError_t e =
        HD == 64 ? launch_pdl(prefill_kernel<64>, (int)grid, (kPWarps + 1) * 32, smem, (cudaStream_t)stream, tk, tv, p)
                 : launch_pdl(prefill_kernel<128>, (int)grid, (kPWarps + 1) * 32, smem, (cudaStream_t)stream, tk, tv, p);
    return e == cudaSuccess ? MI_OK : MI_ERR_CUDA;
}
