// mi_paged_prefill_attention: causal GQA attention of many new tokens per
// request over the paged KV cache — the prefill step of the NJU course brief
// "端侧大模型推理框架" §2.1 (the prefill + decode main loop) and of the
// mini-infer README "项目概述" (prefill as its own forward pass), here also
// serving chunked prefill: the new tokens of request r are its last m_r
// context positions, n_r - m_r .. n_r - 1, and token n_r - m_r + i attends to
// cached tokens 0 .. n_r - m_r + i.
//
// Three kernels compute it: the two-tile tcgen05 kernel (the default,
// prefill_tc2_kernel), the single-tile tcgen05 kernel (prefill_tc_kernel) and
// the mma.sync kernel below (prefill_kernel), whose layout follows; the two
// tcgen05 kernels describe theirs where they are defined.
//
// mma.sync work decomposition:
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
//     softmax on the accumulator fragments, one 16-key block at a time; the probabilities are repacked in
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
#include "tc.cuh"
#include "tma.cuh"

namespace mi {
namespace {

constexpr int kPWarps = 4;                      // consumer warps
constexpr int kMT = 1;                          // 16-row m-tiles per consumer warp
constexpr int kPRows = kPWarps * 16 * kMT;      // rows per CTA
constexpr int kStageBlocks = 4;                 // 16-token blocks per stage: 64 keys
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
    long long wait_ns;             // bound on every mbarrier wait of the launch
    int withhold;                  // failure-detection test: each producer withholds its first K copy
};

// The work item of a CTA: row tile k (counted from the request's end) of
// (request r, KV head h), with `tile_rows` (token, head) rows per tile.
// Returns false when the CTA has nothing to do (past the request's last row,
// or a bad request, which is reported once).
struct Item {
    int r, h, q0, m, n, first, nrows, rho0, rows_here, p_hi, nblk;
};

__device__ __forceinline__ bool work_item(const PrefillParams& p, int tile_rows, Item& it) {
    const int kw = blockIdx.x % kTileGroup;
    const int rest0 = blockIdx.x / kTileGroup;
    it.h = rest0 % p.Hkv;
    const int rest = rest0 / p.Hkv;
    it.r = rest % p.R;
    const int k = (rest / p.R) * kTileGroup + kw;
    const bool reporter = k == 0 && it.h == 0 && threadIdx.x == 0;  // one error report per request
    it.q0 = __ldg(p.query_start + it.r);
    const int q1 = __ldg(p.query_start + it.r + 1);
    it.m = q1 - it.q0;
    if (it.q0 < 0 || q1 > p.T || it.m < 0 || it.m > p.max_q) {
        if (reporter) raise_err(p.dev_err, MI_DEVERR_BAD_QUERY);
        return false;
    }
    it.nrows = it.m * p.G;
    const int tiles = (it.nrows + tile_rows - 1) / tile_rows;
    if (k >= tiles) return false;
    int n = __ldg(p.context_lens + it.r);
    if (n > p.mbps * kBlock) {
        if (reporter) raise_err(p.dev_err, MI_DEVERR_BAD_CONTEXT);
        n = p.mbps * kBlock;
    }
    if (it.m > n && reporter) raise_err(p.dev_err, MI_DEVERR_BAD_QUERY);
    it.n = n;
    it.first = n - it.m;  // position of new token 0 (negative only when m > n)
    it.rho0 = (tiles - 1 - k) * tile_rows;
    it.rows_here = min(tile_rows, it.nrows - it.rho0);
    it.p_hi = it.first + (it.rho0 + it.rows_here - 1) / p.G;  // position of the CTA's last row
    it.nblk = it.p_hi >= 0 ? it.p_hi / kBlock + 1 : 0;        // blocks any row of the CTA reads
    return true;
}

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

// Every wait of the prefill kernels sleeps between polls (the hint of
// mbarrier.try_wait): their waiting warps share schedulers with the warps
// issuing MMAs and computing the softmax. 0.403 ms per Qwen3-8B layer
// against 0.412 ms polling.
__device__ __forceinline__ bool wait_pf(uint32_t bar, uint32_t parity, long long limit_ns) {
    return mbar_wait_bounded(bar, parity, limit_ns, kWaitSleepNs);
}

template <int HD>
__global__ void __launch_bounds__((kPWarps + 1) * 32, kMT == 1 ? 2 : 1)
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
    Item it;
    if (!work_item(p, kPRows, it)) return;
    const int h = it.h, r = it.r, q0 = it.q0, n = it.n, first = it.first, nrows = it.nrows;
    const int rho0 = it.rho0, rows_here = it.rows_here, p_hi = it.p_hi, nblk = it.nblk;
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
            if (!__all_sync(0xffffffffu, wait_pf(empty0 + stg * 8, ph, p.wait_ns))) {
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
                (void)wait_pf(full0 + s * 8, (uint32_t)((fills - 1) & 1), drain_limit(p.wait_ns));
            }
        }
        return;
    }

    // --------------------------------------------------- consumer warps ----
    // A warp owns kMT 16-row m-tiles; a thread holds rows lane/4 and lane/4 + 8
    // of each (index [mt][0] and [mt][1]).
    const int c = lane & 3;
    const int wr0 = rho0 + warp * 16 * kMT;            // first row of this warp
    int ridx[kMT][2], tok[kMT][2], pos[kMT][2], mpos[kMT][2];
    bool vrow[kMT][2];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int r = wr0 + mt * 16 + (lane >> 2) + 8 * hf;
            ridx[mt][hf] = r;
            vrow[mt][hf] = r < nrows;
            tok[mt][hf] = r / p.G;
            pos[mt][hf] = vrow[mt][hf] ? first + tok[mt][hf] : p_hi;
            mpos[mt][hf] = pos[mt][hf] < 0 ? 0 : pos[mt][hf];  // masking position
        }
    const int w_last = min(wr0 + 16 * kMT - 1, rho0 + rows_here - 1);
    const int pw_hi = w_last >= wr0 ? first + w_last / p.G : -1;
    const int pw_lo = first + wr0 / p.G;
    const int nblk_w = pw_hi >= 0 ? pw_hi / kBlock + 1 : 0;  // blocks this warp reads
    const int nb_ctx = (n + kBlock - 1) / kBlock;
    const int tail = n - (nb_ctx - 1) * kBlock;              // valid tokens in the context's last block

    // Q rows as A fragments (zero for rows past the request's last token)
    uint32_t qa[kMT][kK][4];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
        const uint32_t* qr[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const long long head = (long long)(q0 + (vrow[mt][hf] ? tok[mt][hf] : 0)) * p.Hq +
                                   (long long)h * p.G + ridx[mt][hf] % p.G;
            qr[hf] = reinterpret_cast<const uint32_t*>(p.q + head * HD);
        }
#pragma unroll
        for (int ks = 0; ks < kK; ++ks) {
            qa[mt][ks][0] = vrow[mt][0] ? __ldg(qr[0] + ks * 8 + c) : 0u;
            qa[mt][ks][1] = vrow[mt][1] ? __ldg(qr[1] + ks * 8 + c) : 0u;
            qa[mt][ks][2] = vrow[mt][0] ? __ldg(qr[0] + ks * 8 + 4 + c) : 0u;
            qa[mt][ks][3] = vrow[mt][1] ? __ldg(qr[1] + ks * 8 + 4 + c) : 0u;
        }
    }

    float o[kMT][kN][4];
    float mrow[kMT][2], lrow[kMT][2];
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt) {
#pragma unroll
        for (int t = 0; t < kN; ++t) o[mt][t][0] = o[mt][t][1] = o[mt][t][2] = o[mt][t][3] = 0.f;
        mrow[mt][0] = mrow[mt][1] = -INFINITY;
        lrow[mt][0] = lrow[mt][1] = 0.f;
    }

    // ldmatrix lane addressing inside a staged tile
    const int k_key = ((lane >> 4) << 3) + (lane & 7), k_chk = (lane >> 3) & 1;   // K as B of Q.K^T
    const int v_key = (((lane >> 3) & 1) << 3) + (lane & 7), v_chk = lane >> 4;   // V as B of P.V

    uint32_t stg = 0, ph = 0;
    bool dead = false;
    for (int j = 0; j < nst; ++j) {
        if (!__all_sync(0xffffffffu, wait_pf(full0 + stg * 8, ph, p.wait_ns))) {
            if (lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
            dead = true;
            break;
        }
        const uint32_t present = lds_u32(mask0 + stg * 4);
        // the stage is taken one 16-key block at a time, each block's K and V
        // fragments feeding every m-tile of the warp
#pragma unroll
        for (int l = 0; l < kStageBlocks; ++l) {
            const int jb = j * kStageBlocks + l;  // request block index
            if (!((present >> l) & 1u) || jb >= nblk_w) continue;
            const uint32_t kt = sbase + stg * SM::kStage + (uint32_t)l * 2u * kTile, vt = kt + kTile;
            float s[kMT][2][4];
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[mt][0][e] = s[mt][1][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < kK; ++ks) {
                uint32_t b00, b01, b10, b11;
                ldsm_x4(kt + swz<HD>(k_key, 2 * ks + k_chk), b00, b01, b10, b11);
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) {
                    mma_bf16_16816(s[mt][0], qa[mt][ks][0], qa[mt][ks][1], qa[mt][ks][2], qa[mt][ks][3], b00, b01);
                    mma_bf16_16816(s[mt][1], qa[mt][ks][0], qa[mt][ks][1], qa[mt][ks][2], qa[mt][ks][3], b10, b11);
                }
            }
            // scale to base 2, mask keys after a row's position, online softmax
            const int kbase = jb * kBlock;
            const bool causal = kbase + kBlock - 1 > pw_lo;
            uint32_t pa[kMT][4];
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
                float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = kbase + t * 8 + 2 * c + (e & 1);
                        const bool keep = !causal || key <= mpos[mt][e >> 1];
                        s[mt][t][e] = keep ? s[mt][t][e] * p.sl2 : -INFINITY;
                    }
                    x0 = fmaxf(x0, fmaxf(s[mt][t][0], s[mt][t][1]));
                    x1 = fmaxf(x1, fmaxf(s[mt][t][2], s[mt][t][3]));
                }
                x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
                x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
                x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
                x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
                const float n0 = fmaxf(mrow[mt][0], x0), n1 = fmaxf(mrow[mt][1], x1);
                const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
                const float a0 = exp2f(mrow[mt][0] - u0), a1 = exp2f(mrow[mt][1] - u1);
                mrow[mt][0] = n0;
                mrow[mt][1] = n1;
                if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                    for (int t = 0; t < kN; ++t) {
                        o[mt][t][0] *= a0;
                        o[mt][t][1] *= a0;
                        o[mt][t][2] *= a1;
                        o[mt][t][3] *= a1;
                    }
                }
                float e[2][4];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    e[t][0] = exp2f(s[mt][t][0] - u0);
                    e[t][1] = exp2f(s[mt][t][1] - u0);
                    e[t][2] = exp2f(s[mt][t][2] - u1);
                    e[t][3] = exp2f(s[mt][t][3] - u1);
                }
                lrow[mt][0] = lrow[mt][0] * a0 + (e[0][0] + e[0][1] + e[1][0] + e[1][1]);
                lrow[mt][1] = lrow[mt][1] * a1 + (e[0][2] + e[0][3] + e[1][2] + e[1][3]);
                // probabilities, repacked as the A fragment of P . V (16 keys)
                pa[mt][0] = pack_bf16x2(e[0][0], e[0][1]);
                pa[mt][1] = pack_bf16x2(e[0][2], e[0][3]);
                pa[mt][2] = pack_bf16x2(e[1][0], e[1][1]);
                pa[mt][3] = pack_bf16x2(e[1][2], e[1][3]);
            }
            // keys past the context in its last block may hold any bits: zero them
            uint32_t zlo = 0xFFFFFFFFu, zhi = 0xFFFFFFFFu;
            if (jb == nb_ctx - 1 && tail < kBlock) {
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
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) {
                    mma_bf16_16816(o[mt][2 * dp], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], v0, v1);
                    mma_bf16_16816(o[mt][2 * dp + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], v2, v3);
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

#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            float l = lrow[mt][hf];
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (!vrow[mt][hf]) continue;
            // rows before position 0 (more new tokens than context) are +0
            const uint32_t keep = pos[mt][hf] >= 0 ? 0xFFFFFFFFu : 0u;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint32_t* row = reinterpret_cast<uint32_t*>(
                p.out + ((long long)(q0 + tok[mt][hf]) * p.Hq + (long long)h * p.G + ridx[mt][hf] % p.G) * HD);
#pragma unroll
            for (int t = 0; t < kN; ++t)
                row[t * 4 + c] = pack_bf16x2(o[mt][t][2 * hf] * inv, o[mt][t][2 * hf + 1] * inv) & keep;
        }
}

// ------------------------------------------------- tcgen05 prefill kernel --
//
// 128 (token, head) rows per CTA on the fifth-generation tensor cores:
//   * warp 5 (producer) loads the Q tile once and streams 64-key stages (four
//     16-token blocks, each as HD/64 128-byte-wide TMA boxes) through separate
//     K and V rings of two stages, in the canonical 128-byte-swizzled layouts:
//     Q [HD/64][128 rows][128 B], K and V [HD/64][64 keys][128 B]. A K stage
//     is handed back as soon as S = Q . K^T has read it, a V stage once
//     P . V has; K of stage j is issued before V of stage j - 1. (With one
//     barrier pair for K and V together, each K load waited for the P . V of
//     two stages back, and the kernel ran 1.36x slower.)
//   * one thread of warp 4 issues S_j = Q . K_j^T (M 128, N 64, K-major A
//     and B) into one of two tensor-memory score buffers; one thread of
//     warp 6, once the softmax has written P_j, issues O += P_j . V_j (M 128,
//     N HD, A = P from tensor memory, B = V MN-major) into the tensor-memory
//     accumulator; tcgen05.commit signals the mbarriers;
//   * warps 0-3 (softmax): thread t owns row t, i.e. tensor-memory lane t. It
//     loads its 64 scores, masks (causal, missing blocks), updates the
//     running max and sum (on packed fp32 pairs), rescales its O row in
//     tensor memory when the max moved by more than 2^8, and writes its
//     probabilities as bf16 pairs over the consumed scores; warp 0 zeroes V
//     rows of keys that are not in the context. After the last stage each
//     thread reads its O row, normalises it and stores it.
// Tensor memory: 256 columns per CTA (O in columns 0..HD-1, the two score
// buffers at 128 and 192); two CTAs per SM.

constexpr int kTcRows = 128;
constexpr int kTcK = 2;  // K stages
constexpr int kTcV = 2;  // V stages
constexpr int kTcThreads = 224;
constexpr uint32_t kTcCols = 256;

template <int HD>
struct TcSmem {
    static constexpr int kH = HD / 64;                    // 128-byte column blocks of a row
    static constexpr int kQ = 0;                           // Q: kH x [128 rows][128 B]
    static constexpr int kKV = kH * 64 * 128;              // K (or V) of one stage: kH x [64 keys][128 B]
    static constexpr int kRingK = kQ + kH * kTcRows * 128;
    static constexpr int kRingV = kRingK + kTcK * kKV;
    static constexpr int kBar = kRingV + kTcV * kKV;
    // q_full, k_full[2 kTcK], k_empty[kTcK], v_full[kTcV], v_empty[kTcV], s_full[2], s_free[2], p_full[2],
    // o_done[2], fin_s, fin_o
    static constexpr int kNBar = 1 + 3 * kTcK + 2 * kTcV + 2 + 2 + 6;
    static constexpr int kMask = kBar + kNBar * 8;
    static constexpr int kTmem = kMask + 2 * kTcK * 4;     // block masks of stages j mod 2 kTcK
    static constexpr int kUsed = kTmem + 16;
    // the base is aligned up to 1024 B at run time; two CTAs per SM leave
    // 115,712 B each, so the slack is what remains of that (none needed when
    // the dynamic shared memory starts on a 1024-byte boundary)
    static constexpr int kSlack = 115712 - kUsed < 896 ? 115712 - kUsed : 896;
    static constexpr int kTotal = kUsed + kSlack;
    static_assert(kSlack >= 0, "shared memory plan exceeds two CTAs per SM");
};

__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, long long limit_ns) {
    return __all_sync(0xffffffffu, wait_pf(bar, parity, limit_ns));
}

template <int HD>
__global__ void __launch_bounds__(kTcThreads, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, PrefillParams p) {
    using SM = TcSmem<HD>;
    constexpr int kH = SM::kH;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_wait();
    pdl_trigger();

    // a tile holds whole tokens: 128 / G of them, G rows each (the UMMA rows
    // past tile_rows compute on stale shared memory and are never stored)
    const int tile_rows = (kTcRows / p.G) * p.G;
    Item it;
    if (!work_item(p, tile_rows, it)) return;
    if (sbase - raw > (uint32_t)SM::kSlack) {  // no room to align the tiles
        if (threadIdx.x == 0) raise_err(p.dev_err, MI_DEVERR_INTERNAL);
        return;
    }
    const int nst = (it.nblk + kStageBlocks - 1) / kStageBlocks;
    const uint32_t bar = sbase + SM::kBar;
    // K and V of a stage have their own barriers: a K stage is handed back as
    // soon as S = Q . K^T has read it, a V stage once P . V has. K of stage
    // j lands on k_full[j mod 2S]: the softmax warps wait on it too (for the
    // block mask), and with 2S barriers the next phase of the one a warp
    // waits on needs that warp's own P first, so no wait can see a phase
    // ahead of the one it means.
    const uint32_t q_full = bar, k_full0 = bar + 8, k_empty0 = k_full0 + 16 * kTcK;
    const uint32_t v_full0 = k_empty0 + 8 * kTcK, v_empty0 = v_full0 + 8 * kTcV;
    const uint32_t s_full0 = v_empty0 + 8 * kTcV, s_free0 = s_full0 + 16, p_full0 = s_free0 + 16;
    // o_done[b] completes when P . V of a stage with parity b has finished: one
    // barrier per parity keeps every wait within one phase of the barrier,
    // although softmax warps may run a stage apart
    const uint32_t o_done0 = p_full0 + 16, fin = o_done0 + 16, fin_o = fin + 8;
    const uint32_t mask0 = sbase + SM::kMask;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < 2 * kTcK; ++s) mbar_init(k_full0 + s * 8, 1);
        for (int s = 0; s < kTcK; ++s) mbar_init(k_empty0 + s * 8, 1);
        for (int s = 0; s < kTcV; ++s) {
            mbar_init(v_full0 + s * 8, 1);
            mbar_init(v_empty0 + s * 8, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full0 + b * 8, 1);
            mbar_init(s_free0 + b * 8, 1);
        }
        // P_j is ready when all 128 softmax threads have arrived on
        // p_full[j mod 2]: one barrier per stage parity, since a warp may
        // finish stage j + 1 before another has finished stage j
        mbar_init(p_full0, 128);
        mbar_init(p_full0 + 8, 128);
        mbar_init(o_done0, 1);
        mbar_init(o_done0 + 8, 1);
        mbar_init(fin, 1);
        mbar_init(fin_o, 1);
        fence_mbar_init();
    }
    if (warp == 4) {
        tc::alloc(sbase + SM::kTmem, kTcCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = lds_u32(sbase + SM::kTmem);

    if (warp == 5) {
        // ------------------------------------------------ producer warp --
        const uint64_t policy = l2_policy_evict_normal();
        if (lane == 0 && nst > 0) {
            mbar_arrive_expect_tx(q_full, kH * tile_rows * 128);
            for (int hh = 0; hh < kH; ++hh)
                tma_load_4d(sbase + SM::kQ + hh * kTcRows * 128, &tmq, q_full, 0, hh, it.h * p.G,
                            it.q0 + it.rho0 / p.G, policy);
        }
        // K of stage j is issued before V of stage j - 1: V is needed a
        // softmax later than K, and its stage frees up later
        int pblk = -1;
        bool pok = false;
        auto load_v = [&](int jv) -> bool {
            const int sl = jv % kTcV, u = jv / kTcV;
            if (!wait_all(v_empty0 + sl * 8, (uint32_t)((u & 1) ^ 1), p.wait_ns)) return false;
            const uint32_t msk = __ballot_sync(0xffffffffu, pok);
            const uint32_t fb = v_full0 + sl * 8;
            if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)__popc(msk) * kH * kBlock * 128u);
            __syncwarp();
            if (pok) {
                const uint32_t vd = sbase + SM::kRingV + sl * SM::kKV + lane * kBlock * 128;
                const int row0 = (pblk * p.Hkv + it.h) * kBlock;
                for (int hh = 0; hh < kH; ++hh) tma_load_3d(vd + hh * 64 * 128, &tmv, fb, 0, hh, row0, policy);
            }
            return true;
        };
        bool pgood = true;
        for (int j = 0; j < nst; ++j) {
            const int sl = j % kTcK, u = j / kTcK;
            if (!wait_all(k_empty0 + sl * 8, (uint32_t)((u & 1) ^ 1), p.wait_ns)) {
                pgood = false;
                break;
            }
            const int x = j * kStageBlocks + lane;
            int blk = -1;
            bool ok = false;
            if (lane < kStageBlocks && x < it.nblk) {
                blk = __ldg(p.block_tables + (long long)it.r * p.mbps + x);
                ok = blk >= 0 && blk < p.num_blocks;
                if (!ok) raise_err(p.dev_err, MI_DEVERR_BAD_BLOCK);
            }
            const uint32_t msk = __ballot_sync(0xffffffffu, ok);
            const uint32_t fb = k_full0 + (j % (2 * kTcK)) * 8;
            // failure-detection test: stage 0's K is neither copied nor
            // announced, so every wait on it runs out
            const bool held = p.withhold != 0 && j == 0;
            if (lane == 0 && !held) {
                sts32(mask0 + (j % (2 * kTcK)) * 4, msk);
                mbar_arrive_expect_tx(fb, (uint32_t)__popc(msk) * kH * kBlock * 128u);
            }
            __syncwarp();
            if (ok && !held) {
                const uint32_t kd = sbase + SM::kRingK + sl * SM::kKV + lane * kBlock * 128;
                const int row0 = (blk * p.Hkv + it.h) * kBlock;
                for (int hh = 0; hh < kH; ++hh) tma_load_3d(kd + hh * 64 * 128, &tmk, fb, 0, hh, row0, policy);
            }
            if (j > 0 && !load_v(j - 1)) {
                pgood = false;
                break;
            }
            pblk = blk;
            pok = ok;
        }
        if (pgood && nst > 0 && !load_v(nst - 1)) pgood = false;
        if (!pgood && lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
    } else if (warp == 4) {
        // ------------------------------------------------- MMA issuer ----
        if (lane == 0 && nst > 0) {
            constexpr uint32_t idS = tc::idesc_bf16(kTcRows, 64, false);
            bool ok = wait_pf(q_full, 0, p.wait_ns);
            auto issue_s = [&](int jj) {
                const int sl = jj % kTcK, b = jj & 1;
                const uint32_t kbase = sbase + SM::kRingK + sl * SM::kKV;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;  // 16 bf16 of the 128-byte row
                    const uint64_t a = tc::sdesc_sw128(sbase + SM::kQ + (kk >> 2) * kTcRows * 128 + off, 16, 1024);
                    const uint64_t bd = tc::sdesc_sw128(kbase + (kk >> 2) * 64 * 128 + off, 16, 1024);
                    tc::mma_ss(tbase + 128u + 64u * b, a, bd, idS, kk > 0);
                }
                tc::commit(s_full0 + b * 8);
                tc::commit(k_empty0 + sl * 8);  // S_jj has read its K stage
            };
            // S_j needs K_j and its score buffer back from P . V of stage
            // j - 2 (P_{j-2} lives there)
            for (int jj = 0; ok && jj < nst; ++jj) {
                const int u = jj >> 1;
                ok = wait_pf(k_full0 + (jj % (2 * kTcK)) * 8, (uint32_t)((jj / (2 * kTcK)) & 1), p.wait_ns);
                if (ok && u >= 1) ok = wait_pf(s_free0 + (jj & 1) * 8, (uint32_t)((u - 1) & 1), p.wait_ns);
                if (!ok) break;
                tc::fence_after();
                issue_s(jj);
            }
            if (!ok) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
            // every MMA issued has finished before tensor memory is released
            tc::commit(fin);
            (void)wait_pf(fin, 0, drain_limit(p.wait_ns));
        }
        __syncwarp();
    } else if (warp == 6) {
        // --------------------------------------------- P . V issuer ----
        // A second issuing thread, so that P . V of a stage goes out as soon
        // as its P is written instead of after the next S has been issued.
        if (lane == 0 && nst > 0) {
            constexpr uint32_t idO = tc::idesc_bf16(kTcRows, HD, true);
            bool ok = true;
            for (int j = 0; ok && j < nst; ++j) {
                if (!(ok = wait_pf(p_full0 + (j & 1) * 8, (uint32_t)((j >> 1) & 1), p.wait_ns))) break;
                if (!(ok = wait_pf(v_full0 + (j % kTcV) * 8, (uint32_t)((j / kTcV) & 1), p.wait_ns))) break;
                tc::fence_after();
                const uint32_t vbase = sbase + SM::kRingV + (j % kTcV) * SM::kKV;
                // P_j sits in the first 32 columns of its score buffer (bf16 pairs)
                const uint32_t pcol = tbase + 128u + 64u * (j & 1);
#pragma unroll
                for (int l = 0; l < kStageBlocks; ++l) {
                    const uint64_t bd = tc::sdesc_sw128(vbase + l * kBlock * 128, 64 * 128, 1024);
                    tc::mma_ts(tbase, pcol + 8u * l, bd, idO, j > 0 || l > 0);
                }
                tc::commit(o_done0 + (j & 1) * 8);
                tc::commit(s_free0 + (j & 1) * 8);  // the buffer's P has been read
                tc::commit(v_empty0 + (j % kTcV) * 8);
            }
            if (!ok) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
            tc::commit(fin_o);
            (void)wait_pf(fin_o, 0, drain_limit(p.wait_ns));
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax ----
        const int t = threadIdx.x;  // row of the tile, tensor-memory lane
        const int rr = it.rho0 + t;
        const bool vrow = t < tile_rows && rr < it.nrows;
        const int tok = rr / p.G;
        const int pos = vrow ? it.first + tok : it.p_hi;
        const int mpos = pos < 0 ? 0 : pos;
        const uint32_t tl = tbase + ((uint32_t)(warp * 32) << 16);
        const int nb_ctx = (it.n + kBlock - 1) / kBlock;
        const int tail = it.n - (nb_ctx - 1) * kBlock;
        float mrow = -INFINITY, lrow = 0.f;
        bool ok = true;
        for (int j = 0; j < nst; ++j) {
            const int sl = j % kTcV, b = j & 1;  // sl: the V stage
            ok = wait_all(k_full0 + (j % (2 * kTcK)) * 8, (uint32_t)((j / (2 * kTcK)) & 1), p.wait_ns) &&
                 wait_all(s_full0 + b * 8, (uint32_t)((j >> 1) & 1), p.wait_ns);
            if (!ok) break;
            tc::fence_after();
            uint32_t x[64];
            tc::ld32(tl + 128u + 64u * b, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
            tc::ld32(tl + 128u + 64u * b + 32u, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
            tc::wait_ld();
            const uint32_t present = lds_u32(mask0 + (j % (2 * kTcK)) * 4);
            const int kbase = j * kStageBlocks * kBlock;
            // eight independent partial maxima keep the dependency chains short.
            // With a positive scale (the usual case) the max is taken over the
            // raw scores and the scale folds into the exponent's fma; else the
            // scores are scaled first.
            const bool fold = p.sl2 > 0.f;
            float mp[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
            // stages wholly below every row's position with all blocks
            // present need no mask
            const bool nomask = __all_sync(0xffffffffu, present == 0xFu && kbase + kStageBlocks * kBlock - 1 <= mpos);
            if (fold && nomask) {
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    mp[c & 7] = tc::max3(mp[c & 7], __uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1]));
            } else if (fold) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const bool keep = ((present >> (c >> 4)) & 1u) && kbase + c <= mpos;
                    const float v = keep ? __uint_as_float(x[c]) : -INFINITY;
                    x[c] = __float_as_uint(v);
                    mp[c & 7] = fmaxf(mp[c & 7], v);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const bool keep = ((present >> (c >> 4)) & 1u) && kbase + c <= mpos;
                    const float v = keep ? __uint_as_float(x[c]) * p.sl2 : -INFINITY;
                    x[c] = __float_as_uint(v);
                    mp[c & 7] = fmaxf(mp[c & 7], v);
                }
            }
            const float mr = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                                   fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
            const float mx = fold ? mr * p.sl2 : mr;
            // Lazy rescaling: the reference max only moves when the new max
            // exceeds it by more than 2^8 (weights stay <= 256); O and l are
            // rescaled together, so the normalised result is unchanged.
            float alpha = 1.f;
            bool need = false;
            if (mrow == -INFINITY) {
                mrow = mx;  // nothing accumulated yet: O row and l are zero
            } else if (mx > mrow + 8.f) {
                alpha = exp2f(mrow - mx);
                mrow = mx;
                need = true;
            }
            const float un = mrow == -INFINITY ? 0.f : mrow;
            float ps[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) ps[i] = 0.f;
            uint32_t w[32];
            if (fold) {
                // exponent arguments and row sums on packed fp32 pairs
                const uint64_t sc2 = tc::f2(p.sl2, p.sl2), nu2 = tc::f2(-un, -un);
                uint64_t acc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = 0ull;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const uint64_t a2 = tc::fma2(tc::f2(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])), sc2, nu2);
                    const float e0 = ex2(tc::f2_lo(a2)), e1 = ex2(tc::f2_hi(a2));
                    acc[c & 3] = tc::add2(acc[c & 3], tc::f2(e0, e1));
                    w[c] = pack_bf16x2(e0, e1);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ps[2 * i] = tc::f2_lo(acc[i]);
                    ps[2 * i + 1] = tc::f2_hi(acc[i]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float e0 = ex2(__uint_as_float(x[2 * c]) - un);
                    const float e1 = ex2(__uint_as_float(x[2 * c + 1]) - un);
                    ps[c & 7] += e0 + e1;
                    w[c] = pack_bf16x2(e0, e1);
                }
            }
            const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            lrow = lrow * alpha + psum;
            if (__any_sync(0xffffffffu, need)) {
                // O may be touched once the previous P . V has finished
                if (!(ok = wait_all(o_done0 + ((j - 1) & 1) * 8, (uint32_t)(((j - 1) >> 1) & 1), p.wait_ns))) break;
                tc::fence_after();
#pragma unroll 1
                for (int ch = 0; ch < HD / 32; ++ch) {
                    uint32_t y[32];
                    tc::ld32(tl + 32u * ch, y);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) y[i] = __float_as_uint(__uint_as_float(y[i]) * alpha);
                    tc::st32(tl + 32u * ch, y);
                }
            }
            // P over the consumed scores: the A operand of O += P . V
            tc::st32(tl + 128u + 64u * b, w);
            tc::wait_st();
            if (warp == 0) {
                // V rows of keys outside the context (missing blocks, the
                // last block's tail) may hold any bits: zero them, once the
                // stage's V copies have landed
                const uint32_t vbase = sbase + SM::kRingV + sl * SM::kKV;
                bool any = false;
                for (int l = 0; l < kStageBlocks; ++l) {
                    const int blk = j * kStageBlocks + l;
                    any |= !((present >> l) & 1u) || (blk == nb_ctx - 1 && tail < kBlock);
                }
                if (any && !(ok = wait_all(v_full0 + sl * 8, (uint32_t)((j / kTcV) & 1), p.wait_ns))) break;
                for (int l = 0; any && l < kStageBlocks; ++l) {
                    const int blk = j * kStageBlocks + l;
                    const int from = !((present >> l) & 1u) ? 0 : (blk == nb_ctx - 1 && tail < kBlock ? tail : kBlock);
                    for (int i = lane; i < (kBlock - from) * kH * 8; i += 32) {
                        const int key = l * kBlock + from + i / (kH * 8), hh = (i / 8) % kH, ch = i % 8;
                        st_shared_zero16(vbase + hh * 64 * 128 + key * 128 + ch * 16);
                    }
                }
            }
            fence_proxy_async_smem();
            tc::fence_before();
            mbar_arrive(p_full0 + (j & 1) * 8);
        }
        if (!ok && threadIdx.x == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
        if (ok && nst > 0) ok = wait_all(o_done0 + ((nst - 1) & 1) * 8, (uint32_t)(((nst - 1) >> 1) & 1), p.wait_ns);
        tc::fence_after();
        const float inv = lrow > 0.f ? 1.f / lrow : 0.f;
        const uint32_t keep = pos >= 0 ? 0xFFFFFFFFu : 0u;  // rows before position 0 are +0
        uint16_t* orow = p.out + ((long long)(it.q0 + tok) * p.Hq + (long long)it.h * p.G + rr % p.G) * HD;
#pragma unroll 1
        for (int ch = 0; ch < HD / 32; ++ch) {
            uint32_t y[32];
            if (nst > 0 && ok) {
                tc::ld32(tl + 32u * ch, y);
                tc::wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) y[i] = 0u;
            }
            if (vrow && ok) {
                uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        pk[i] = pack_bf16x2(__uint_as_float(y[8 * q4 + 2 * i]) * inv,
                                            __uint_as_float(y[8 * q4 + 2 * i + 1]) * inv) & keep;
                    dst[q4] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 4) {
        tc::fence_after();
        tc::dealloc(tbase, kTcCols);
    }
}

// ----------------------------------------- tcgen05 prefill, two Q tiles --
//
// One CTA per SM holds two 128-row Q tiles of the same (request, KV head)
// (the second tile's rows are later positions) and streams 128-key stages
// that both tiles consume, so each K / V byte is staged once for 256 rows and
// each S = Q . K^T instruction is 128 x 128 (half the Q operand traffic per
// key of a 128 x 64 one). Tensor memory (512 columns): O_t at 256 t, S_t at
// 256 t + 128 (P_t, the bf16 probabilities, over the first 64 of its
// columns). One warp issues every MMA (converged, one elected lane),
// alternating the tiles so that one tile's softmax runs under the other
// tile's MMAs:
//   S_0(0), S_1(0); for each stage j: O_0 += P_0(j) V(j), S_0(j+1),
//   O_1 += P_1(j) V(j), S_1(j+1).
// S_t(j+1) overwrites P_t(j) after O_t += P_t(j) V(j) has read it: MMAs one
// thread issues run in issue order. Warps 0-15 run the softmax, eight per
// tile: warp w reads tensor-memory lanes 32 (w mod 4) + 16 (w / 8) ... + 15
// with the 16-lane shapes, each lane holding two rows x 32 keys of a stage;
// warp 16 issues the MMAs and owns the tensor memory; warp 17 loads Q once
// and streams K (two stages, a 2 KB copy per block half) and V (two stages,
// a 4 KB copy per block), K of stage j before V of stage j - 1.

constexpr int kT2Keys = 128;                 // keys per stage
constexpr int kT2Blocks = kT2Keys / kBlock;  // 16-token blocks per stage
constexpr int kT2MmaWarp = 16;  // warps 0-15 softmax, 16 MMA, 17 producer
constexpr int kT2Threads = (kT2MmaWarp + 2) * 32;
constexpr uint32_t kT2Cols = 512;
constexpr int kT2KSlots = 2;  // K ring depth (V: two); three measured no faster (0.389 against 0.386 ms)

template <int HD>
struct Tc2Smem {
    static constexpr int kH = HD / 64;
    static constexpr int kQT = kH * kTcRows * 128;            // one Q tile: kH x [128 rows][128 B]
    // one K or V stage: K as kH x [128 keys][128 B], V as 8 blocks x kH x [16 keys][128 B]
    static constexpr int kKV = kH * kT2Keys * 128;
    static constexpr int kQ = 0;
    static constexpr int kRingK = kQ + 2 * kQT;
    static constexpr int kRingV = kRingK + kT2KSlots * kKV;
    static constexpr int kBar = kRingV + 2 * kKV;
    // q_full, k_full[4], k_empty[kT2KSlots], v_full[2], v_empty[2], s_full[2], p_full[2], o_done[2], fin
    static constexpr int kNBar = 1 + 4 + kT2KSlots + 2 + 2 + 2 + 2 + 2 + 1;
    static constexpr int kMask = kBar + kNBar * 8;
    static constexpr int kTmem = kMask + 4 * 4;
    static constexpr int kTotal = kTmem + 16 + 1024;  // slack to align the base to 1024 B
};

template <int HD>
__global__ void __launch_bounds__(kT2Threads, 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, PrefillParams p) {
    using SM = Tc2Smem<HD>;
    constexpr int kH = SM::kH;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_wait();
    pdl_trigger();

    // a Q tile holds whole tokens: 128 / G of them, G rows each; the CTA's
    // two tiles are consecutive, tr rows apart
    const int tr = (kTcRows / p.G) * p.G;
    Item it;
    if (!work_item(p, 2 * tr, it)) return;
    const int nst = (it.nblk + kT2Blocks - 1) / kT2Blocks;
    const uint32_t bar = sbase + SM::kBar;
    const uint32_t q_full = bar, k_full0 = bar + 8, k_empty0 = k_full0 + 32, v_full0 = k_empty0 + 8 * kT2KSlots;
    const uint32_t v_empty0 = v_full0 + 16, s_full0 = v_empty0 + 16, p_full0 = s_full0 + 16;
    const uint32_t o_done0 = p_full0 + 16, fin = o_done0 + 16;
    const uint32_t mask0 = sbase + SM::kMask;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 4; ++i) mbar_init(k_full0 + i * 8, 1);
        for (int i = 0; i < kT2KSlots; ++i) mbar_init(k_empty0 + i * 8, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(v_full0 + i * 8, 1);
            mbar_init(v_empty0 + i * 8, 1);
            mbar_init(s_full0 + i * 8, 1);
            mbar_init(p_full0 + i * 8, 256);  // every softmax thread of the tile
            mbar_init(o_done0 + i * 8, 1);
        }
        mbar_init(fin, 1);
        fence_mbar_init();
    }
    if (warp == kT2MmaWarp) {
        tc::alloc(sbase + SM::kTmem, kT2Cols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = lds_u32(sbase + SM::kTmem);

    if (warp == kT2MmaWarp + 1) {
        // ------------------------------------------------ producer warp --
        const uint64_t policy = l2_policy_evict_normal();
        if (lane == 0 && nst > 0) {
            mbar_arrive_expect_tx(q_full, 2u * kH * (uint32_t)tr * 128u);
            for (int t = 0; t < 2; ++t)
                for (int hh = 0; hh < kH; ++hh)
                    tma_load_4d(sbase + SM::kQ + t * SM::kQT + hh * kTcRows * 128, &tmq, q_full, 0, hh, it.h * p.G,
                                it.q0 + (it.rho0 + t * tr) / p.G, policy);
        }
        int pblk = -1;
        bool pok = false;
        auto load_v = [&](int jv) -> bool {
            const int sl = jv & 1, u = jv >> 1;
            if (!wait_all(v_empty0 + sl * 8, (uint32_t)((u & 1) ^ 1), p.wait_ns)) return false;
            const uint32_t msk = __ballot_sync(0xffffffffu, pok);
            const uint32_t fb = v_full0 + sl * 8;
            if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)__popc(msk) * kH * kBlock * 128u);
            __syncwarp();
            if (pok) {
                // one copy per block: both 128-byte halves of its 16 rows
                const uint32_t vd = sbase + SM::kRingV + sl * SM::kKV + lane * kH * kBlock * 128;
                const int row0 = (pblk * p.Hkv + it.h) * kBlock;
                tma_load_3d(vd, &tmv, fb, 0, row0, 0, policy);
            }
            return true;
        };
        bool pgood = true;
        // block-table entries are read a stage ahead, before the wait for
        // the slot, so their load latency is hidden
        auto table_entry = [&](int jj) -> int {
            const int x = jj * kT2Blocks + lane;
            return (lane < kT2Blocks && x < it.nblk) ? __ldg(p.block_tables + (long long)it.r * p.mbps + x) : -1;
        };
        int nblk_next = table_entry(0);
        for (int j = 0; j < nst; ++j) {
            const int sl = j % kT2KSlots, u = j / kT2KSlots;
            const int x = j * kT2Blocks + lane;
            const int blk = nblk_next;
            if (j + 1 < nst) nblk_next = table_entry(j + 1);
            if (!wait_all(k_empty0 + sl * 8, (uint32_t)((u & 1) ^ 1), p.wait_ns)) {
                pgood = false;
                break;
            }
            bool ok = false;
            if (lane < kT2Blocks && x < it.nblk) {
                ok = blk >= 0 && blk < p.num_blocks;
                if (!ok) raise_err(p.dev_err, MI_DEVERR_BAD_BLOCK);
            }
            const uint32_t msk = __ballot_sync(0xffffffffu, ok);
            const uint32_t fb = k_full0 + (j & 3) * 8;
            // failure-detection test: stage 0's K is neither copied nor
            // announced, so every wait on it runs out
            const bool held = p.withhold != 0 && j == 0;
            if (lane == 0 && !held) {
                sts32(mask0 + (j & 3) * 4, msk);
                mbar_arrive_expect_tx(fb, (uint32_t)__popc(msk) * kH * kBlock * 128u);
            }
            __syncwarp();
            if (ok && !held) {
                const uint32_t kd = sbase + SM::kRingK + sl * SM::kKV + lane * kBlock * 128;
                const int row0 = (blk * p.Hkv + it.h) * kBlock;
                for (int hh = 0; hh < kH; ++hh) tma_load_3d(kd + hh * kT2Keys * 128, &tmk, fb, 0, hh, row0, policy);
            }
            if (j > 0 && !load_v(j - 1)) {
                pgood = false;
                break;
            }
            pblk = blk;
            pok = ok;
        }
        if (pgood && nst > 0 && !load_v(nst - 1)) pgood = false;
        if (!pgood && lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
    } else if (warp == kT2MmaWarp) {
        // -------------------------------------------------- MMA issuer --
        // The whole warp runs the loop; one elected lane issues each MMA
        // and commit.
        if (nst > 0) {
            constexpr uint32_t idS = tc::idesc_bf16(kTcRows, kT2Keys, false);
            constexpr uint32_t idO = tc::idesc_bf16(kTcRows, HD, true);
            auto issue_s = [&](int t, int j) {
                const uint32_t kbase = sbase + SM::kRingK + (j % kT2KSlots) * SM::kKV;
                const uint32_t qbase = sbase + SM::kQ + t * SM::kQT;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;  // 16 bf16 of the 128-byte row
                    const uint64_t a = tc::sdesc_sw128(qbase + (kk >> 2) * kTcRows * 128 + off, 16, 1024);
                    const uint64_t bd = tc::sdesc_sw128(kbase + (kk >> 2) * kT2Keys * 128 + off, 16, 1024);
                    tc::mma_ss_elect(tbase + 256u * t + 128u, a, bd, idS, kk > 0);
                }
                tc::commit_elect(s_full0 + t * 8);
            };
            auto issue_o = [&](int t, int j) {
                const uint32_t vbase = sbase + SM::kRingV + (j & 1) * SM::kKV;
                const uint32_t pcol = tbase + 256u * t + 128u;  // P_t(j): bf16 pairs over S_t's first 64 columns
#pragma unroll
                for (int l = 0; l < kT2Blocks; ++l) {
                    // block l: [kH][16 keys][128 B]; the 64-column halves of V
                    // are kBlock * 128 bytes apart
                    const uint64_t bd = tc::sdesc_sw128(vbase + l * kH * kBlock * 128, kBlock * 128, 1024);
                    tc::mma_ts_elect(tbase + 256u * t, pcol + 8u * l, bd, idO, j > 0 || l > 0);
                }
                tc::commit_elect(o_done0 + t * 8);
            };
            bool ok = wait_all(q_full, 0, p.wait_ns) && wait_all(k_full0, 0, p.wait_ns);
            if (ok) {
                tc::fence_after();
                issue_s(0, 0);
                issue_s(1, 0);
                tc::commit_elect(k_empty0);  // K(0) read by both tiles
            }
            for (int j = 0; ok && j < nst; ++j) {
                const uint32_t ph = (uint32_t)(j & 1);
                ok = wait_all(p_full0, ph, p.wait_ns) &&
                     wait_all(v_full0 + (j & 1) * 8, (uint32_t)((j >> 1) & 1), p.wait_ns);
                if (!ok) break;
                tc::fence_after();
                issue_o(0, j);
                const bool more = j + 1 < nst;
                if (more) {
                    if (!(ok = wait_all(k_full0 + ((j + 1) & 3) * 8, (uint32_t)(((j + 1) >> 2) & 1), p.wait_ns)))
                        break;
                    tc::fence_after();
                    issue_s(0, j + 1);
                }
                if (!(ok = wait_all(p_full0 + 8, ph, p.wait_ns))) break;
                tc::fence_after();
                issue_o(1, j);
                tc::commit_elect(v_empty0 + (j & 1) * 8);  // V(j) read by both tiles
                if (more) {
                    issue_s(1, j + 1);
                    tc::commit_elect(k_empty0 + ((j + 1) % kT2KSlots) * 8);
                }
            }
            if (!ok && lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
            // every MMA issued has finished before tensor memory is released
            tc::commit_elect(fin);
            (void)wait_all(fin, 0, drain_limit(p.wait_ns));
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax ----
        // Eight warps per tile. Warp w reads tensor-memory lanes lb ... lb + 15
        // (lb = 32 (w mod 4) + 16 (w / 8)) with the 16-lane shapes: lane i
        // holds rows a = lb + i/4 and b = a + 8, keys 8k + 2 (i mod 4) and the
        // next one of each 8-key group k, so a quad of lanes shares two rows'
        // scores (32 keys each per lane) and reduces them with shuffles.
        const int t = (warp >> 2) & 1;  // tile
        const int c4 = lane & 3;
        const int lb = (warp & 3) * 32 + (warp >> 3) * 16;
        const int rla = lb + (lane >> 2), rlb = rla + 8;  // rows of the tile
        const int rra = it.rho0 + t * tr + rla, rrb = it.rho0 + t * tr + rlb;
        const bool va = rla < tr && rra < it.nrows, vb = rlb < tr && rrb < it.nrows;
        const int toka = rra / p.G, tokb = rrb / p.G;
        const int posa = va ? it.first + toka : it.p_hi, posb = vb ? it.first + tokb : it.p_hi;
        const int mposa = posa < 0 ? 0 : posa, mposb = posb < 0 ? 0 : posb;
        const uint32_t tl = tbase + ((uint32_t)lb << 16) + 256u * t;  // O_t of these lanes
        const uint32_t ts = tl + 128u;                                // S_t / P_t
        const int nb_ctx = (it.n + kBlock - 1) / kBlock;
        const int tail = it.n - (nb_ctx - 1) * kBlock;
        const bool fold = p.sl2 > 0.f;
        float mra_run = -INFINITY, mrb_run = -INFINITY, lra = 0.f, lrb = 0.f;  // per lane: its 32 keys of the row
        bool ok = true;
        for (int j = 0; j < nst; ++j) {
            ok = wait_all(k_full0 + (j & 3) * 8, (uint32_t)((j >> 2) & 1), p.wait_ns) &&
                 wait_all(s_full0 + t * 8, (uint32_t)(j & 1), p.wait_ns);
            if (!ok) break;
            tc::fence_after();
            uint32_t x[2 * kT2Keys / 4];  // x[4k + e]: e = 0, 1 row a; e = 2, 3 row b
            tc::ld16x256_x8(ts, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
            tc::ld16x256_x8(ts + 64u, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
            tc::wait_ld();
            const uint32_t present = lds_u32(mask0 + (j & 3) * 4);
            const int kbase = j * kT2Keys;
            const bool nomask = __all_sync(0xffffffffu, present == (1u << kT2Blocks) - 1u &&
                                                            kbase + kT2Keys - 1 <= min(mposa, mposb));
            float alpha_a = 1.f, alpha_b = 1.f, psa, psb;
            bool need = false;
            float ma[4], mb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ma[i] = mb[i] = -INFINITY;
            if (fold && nomask) {
#pragma unroll
                for (int k = 0; k < kT2Keys / 8; ++k) {
                    ma[k & 3] = tc::max3(ma[k & 3], __uint_as_float(x[4 * k]), __uint_as_float(x[4 * k + 1]));
                    mb[k & 3] = tc::max3(mb[k & 3], __uint_as_float(x[4 * k + 2]), __uint_as_float(x[4 * k + 3]));
                }
            } else {
#pragma unroll
                for (int k = 0; k < kT2Keys / 8; ++k) {
                    const bool blk = (present >> (k >> 1)) & 1u;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = kbase + 8 * k + 2 * c4 + (e & 1);
                        const bool keep = blk && key <= (e < 2 ? mposa : mposb);
                        const float v = keep ? (fold ? __uint_as_float(x[4 * k + e])
                                                     : __uint_as_float(x[4 * k + e]) * p.sl2)
                                             : -INFINITY;
                        x[4 * k + e] = __float_as_uint(v);
                        if (e < 2)
                            ma[k & 3] = fmaxf(ma[k & 3], v);
                        else
                            mb[k & 3] = fmaxf(mb[k & 3], v);
                    }
                }
            }
            float mxa = fmaxf(fmaxf(ma[0], ma[1]), fmaxf(ma[2], ma[3]));
            float mxb = fmaxf(fmaxf(mb[0], mb[1]), fmaxf(mb[2], mb[3]));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
            if (fold) {
                mxa *= p.sl2;
                mxb *= p.sl2;
            }
            // lazy rescaling, per row: the reference max moves only when the
            // new max exceeds it by more than 2^8; O and l are rescaled
            // together (the four lanes of a quad take the same decision)
            if (mra_run == -INFINITY) {
                mra_run = mxa;
            } else if (mxa > mra_run + 8.f) {
                alpha_a = exp2f(mra_run - mxa);
                mra_run = mxa;
                need = true;
            }
            if (mrb_run == -INFINITY) {
                mrb_run = mxb;
            } else if (mxb > mrb_run + 8.f) {
                alpha_b = exp2f(mrb_run - mxb);
                mrb_run = mxb;
                need = true;
            }
            const float una = mra_run == -INFINITY ? 0.f : mra_run;
            const float unb = mrb_run == -INFINITY ? 0.f : mrb_run;
            if (fold) {
                const uint64_t sc2 = tc::f2(p.sl2, p.sl2);
                const uint64_t nua = tc::f2(-una, -una), nub = tc::f2(-unb, -unb);
                uint64_t acca[2] = {0ull, 0ull}, accb[2] = {0ull, 0ull};
#pragma unroll
                for (int k = 0; k < kT2Keys / 8; ++k) {
                    const uint64_t a2 = tc::fma2(tc::f2(__uint_as_float(x[4 * k]), __uint_as_float(x[4 * k + 1])),
                                                 sc2, nua);
                    const uint64_t b2 = tc::fma2(
                        tc::f2(__uint_as_float(x[4 * k + 2]), __uint_as_float(x[4 * k + 3])), sc2, nub);
                    const float ea0 = ex2(tc::f2_lo(a2)), ea1 = ex2(tc::f2_hi(a2));
                    const float eb0 = ex2(tc::f2_lo(b2)), eb1 = ex2(tc::f2_hi(b2));
                    acca[k & 1] = tc::add2(acca[k & 1], tc::f2(ea0, ea1));
                    accb[k & 1] = tc::add2(accb[k & 1], tc::f2(eb0, eb1));
                    // P words (column 4k + i mod 4 of rows a and b) over the
                    // consumed scores
                    x[2 * k] = pack_bf16x2(ea0, ea1);
                    x[2 * k + 1] = pack_bf16x2(eb0, eb1);
                }
                const uint64_t sa = tc::add2(acca[0], acca[1]), sb = tc::add2(accb[0], accb[1]);
                psa = tc::f2_lo(sa) + tc::f2_hi(sa);
                psb = tc::f2_lo(sb) + tc::f2_hi(sb);
            } else {
                float pa[2] = {0.f, 0.f}, pb[2] = {0.f, 0.f};
#pragma unroll
                for (int k = 0; k < kT2Keys / 8; ++k) {
                    const float ea0 = ex2(__uint_as_float(x[4 * k]) - una);
                    const float ea1 = ex2(__uint_as_float(x[4 * k + 1]) - una);
                    const float eb0 = ex2(__uint_as_float(x[4 * k + 2]) - unb);
                    const float eb1 = ex2(__uint_as_float(x[4 * k + 3]) - unb);
                    pa[k & 1] += ea0 + ea1;
                    pb[k & 1] += eb0 + eb1;
                    x[2 * k] = pack_bf16x2(ea0, ea1);
                    x[2 * k + 1] = pack_bf16x2(eb0, eb1);
                }
                psa = pa[0] + pa[1];
                psb = pb[0] + pb[1];
            }
            lra = lra * alpha_a + psa;
            lrb = lrb * alpha_b + psb;
            if (__any_sync(0xffffffffu, need)) {
                // O_t may be touched once its previous P . V has finished
                if (!(ok = wait_all(o_done0 + t * 8, (uint32_t)((j - 1) & 1), p.wait_ns))) break;
                tc::fence_after();
#pragma unroll 1
                for (int ch = 0; ch < HD / 32; ++ch) {
                    uint32_t y[16];
                    tc::ld16x256_x4(tl + 32u * ch, y);
                    tc::wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        y[i] = __float_as_uint(__uint_as_float(y[i]) * ((i & 2) ? alpha_b : alpha_a));
                    tc::st16x256_x4(tl + 32u * ch, y);
                }
            }
            // P_t(j): the A operand of O_t += P_t(j) . V(j)
            tc::st16x128_x16(ts, *reinterpret_cast<const uint32_t(*)[32]>(&x[0]));
            tc::wait_st();
            if (warp == 1) {
                // V rows of keys outside the context (missing blocks, the
                // last block's tail) may hold any bits: zero them once the
                // stage's V copies have landed, before tile 0's P . V (tile
                // 1's is issued after it). A warp of tile 0 off the MMA
                // warp's scheduler does it.
                const int last = nb_ctx - 1 - j * kT2Blocks;  // the context's last block, stage-local
                const bool any = present != (1u << kT2Blocks) - 1u || (last < kT2Blocks && tail < kBlock);
                if (any) {
                    if (!(ok = wait_all(v_full0 + (j & 1) * 8, (uint32_t)((j >> 1) & 1), p.wait_ns))) break;
                    const uint32_t vbase = sbase + SM::kRingV + (j & 1) * SM::kKV;
                    for (int l = 0; l < kT2Blocks; ++l) {
                        const int from = !((present >> l) & 1u) ? 0 : (l == last && tail < kBlock ? tail : kBlock);
                        for (int i = lane; i < (kBlock - from) * kH * 8; i += 32) {
                            const int r = from + i / (kH * 8), hh = (i / 8) % kH, ch = i % 8;
                            st_shared_zero16(vbase + (l * kH + hh) * kBlock * 128 + r * 128 + ch * 16);
                        }
                    }
                    fence_proxy_async_smem();  // generic-proxy writes read by the tensor cores
                }
            }
            tc::fence_before();
            mbar_arrive(p_full0 + t * 8);
        }
        if (!ok && lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
        if (ok && nst > 0) ok = wait_all(o_done0 + t * 8, (uint32_t)((nst - 1) & 1), p.wait_ns);
        tc::fence_after();
        lra += __shfl_xor_sync(0xffffffffu, lra, 1);
        lrb += __shfl_xor_sync(0xffffffffu, lrb, 1);
        lra += __shfl_xor_sync(0xffffffffu, lra, 2);
        lrb += __shfl_xor_sync(0xffffffffu, lrb, 2);
        const float inva = lra > 0.f ? 1.f / lra : 0.f, invb = lrb > 0.f ? 1.f / lrb : 0.f;
        const uint32_t keepa = posa >= 0 ? 0xFFFFFFFFu : 0u, keepb = posb >= 0 ? 0xFFFFFFFFu : 0u;  // rows before position 0 are +0
        uint16_t* orowa = p.out + ((long long)(it.q0 + toka) * p.Hq + (long long)it.h * p.G + rra % p.G) * HD;
        uint16_t* orowb = p.out + ((long long)(it.q0 + tokb) * p.Hq + (long long)it.h * p.G + rrb % p.G) * HD;
#pragma unroll 1
        for (int ch = 0; ch < HD / 32; ++ch) {
            uint32_t y[16];
            if (nst > 0 && ok) {
                tc::ld16x256_x4(tl + 32u * ch, y);
                tc::wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) y[i] = 0u;
            }
            if (ok) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int col = 32 * ch + 8 * k + 2 * c4;
                    if (va)
                        *reinterpret_cast<uint32_t*>(orowa + col) =
                            pack_bf16x2(__uint_as_float(y[4 * k]) * inva, __uint_as_float(y[4 * k + 1]) * inva) & keepa;
                    if (vb)
                        *reinterpret_cast<uint32_t*>(orowb + col) =
                            pack_bf16x2(__uint_as_float(y[4 * k + 2]) * invb, __uint_as_float(y[4 * k + 3]) * invb) &
                            keepb;
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == kT2MmaWarp) {
        tc::fence_after();
        tc::dealloc(tbase, kT2Cols);
    }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Raise a kernel's dynamic shared-memory limit once per device and context
// (a device reset makes a new context, which needs it again).
bool raise_smem_once(const void* fn, int smem, CUcontext* done, std::mutex& mu) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return false;
    std::lock_guard<std::mutex> lk(mu);
    const CUcontext ctx0 = current_context();
    if (ctx0 && done[dev] == ctx0) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
    done[dev] = current_context();
    return true;
}

template <int HD>
bool prepare_tc() {
    static std::mutex mu;
    static CUcontext done[256] = {};
    return raise_smem_once(reinterpret_cast<const void*>(prefill_tc_kernel<HD>), TcSmem<HD>::kTotal, done, mu);
}

template <int HD>
bool prepare_tc2() {
    static std::mutex mu;
    static CUcontext done[256] = {};
    return raise_smem_once(reinterpret_cast<const void*>(prefill_tc2_kernel<HD>), Tc2Smem<HD>::kTotal, done, mu);
}

template <int HD>
bool prepare(int* smem) {
    static std::mutex mu;
    static CUcontext done[256] = {};
    *smem = PrefillSmem<HD>::kTotal;
    return raise_smem_once(reinterpret_cast<const void*>(prefill_kernel<HD>), *smem, done, mu);
}

}  // namespace
}  // namespace mi

namespace mi {
namespace {

mi_status prefill(const mi_dims* dims, int32_t total_q, int32_t max_query_len, const void* q, const void* k_cache,
                  const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
                  const int32_t* query_start, float scale, void* out, int32_t* dev_err, mi_stream_t stream,
                  int32_t variant) {
    if (!dims) return MI_ERR_INVALID_ARG;
    if (variant < MI_PREFILL_DEFAULT || variant > MI_PREFILL_TCGEN05_PAIR) return MI_ERR_INVALID_ARG;
    const mi_dims D = *dims;
    if (D.B < 0 || D.Hq < 1 || D.Hkv < 1 || D.num_blocks < 1 || D.max_blocks_per_seq < 1 || total_q < 0 ||
        max_query_len < 0)
        return MI_ERR_INVALID_ARG;
    if (D.block_size != kBlock || (D.head_dim != 64 && D.head_dim != 128) || D.Hq % D.Hkv != 0 ||
        D.Hq / D.Hkv > kMaxGroup)
        return MI_ERR_UNSUPPORTED;
    const int G = D.Hq / D.Hkv, HD = D.head_dim;
    // the tcgen05 tile stacks 128 / G whole tokens of a group (G <= 8)
    const bool use_tc2 = variant == MI_PREFILL_TCGEN05_PAIR || variant == MI_PREFILL_DEFAULT;
    const bool use_tc = variant == MI_PREFILL_TCGEN05 || use_tc2;
    const int tc_rows = (kTcRows / G) * G;
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
    const int rows_per_tile = use_tc2 ? 2 * tc_rows : (use_tc ? tc_rows : kPRows);
    const long long tiles_max = ((long long)max_query_len * G + rows_per_tile - 1) / rows_per_tile;
    const long long grid = (tiles_max + kTileGroup - 1) / kTileGroup * kTileGroup * D.B * D.Hkv;
    if (grid > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;

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
    p.wait_ns = test_wait_limit_ns();
    p.withhold = use_tc && test_withhold_copy() ? 1 : 0;  // (the tcgen05 kernel's test hook)
    const long long rows = (long long)D.num_blocks * D.Hkv * kBlock;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (use_tc2) {
        if (!(HD == 64 ? prepare_tc2<64>() : prepare_tc2<128>())) return MI_ERR_CUDA;
        CUtensorMap tq, tk, tv;
        if (!make_tmap_q_group(&tq, q, total_q, D.Hq, HD, G, tc_rows) ||
            !make_tmap_kv_halves(&tk, k_cache, rows, HD) || !make_tmap_kv_blocks(&tv, v_cache, rows, HD))
            return MI_ERR_CUDA;
        e = HD == 64 ? launch_pdl(prefill_tc2_kernel<64>, (int)grid, kT2Threads, Tc2Smem<64>::kTotal, st, tq, tk, tv, p)
                     : launch_pdl(prefill_tc2_kernel<128>, (int)grid, kT2Threads, Tc2Smem<128>::kTotal, st, tq, tk,
                                  tv, p);
    } else if (use_tc) {
        if (!(HD == 64 ? prepare_tc<64>() : prepare_tc<128>())) return MI_ERR_CUDA;
        CUtensorMap tq, tk, tv;
        if (!make_tmap_q_group(&tq, q, total_q, D.Hq, HD, G, tc_rows) ||
            !make_tmap_kv_halves(&tk, k_cache, rows, HD) || !make_tmap_kv_halves(&tv, v_cache, rows, HD))
            return MI_ERR_CUDA;
        e = HD == 64 ? launch_pdl(prefill_tc_kernel<64>, (int)grid, kTcThreads, TcSmem<64>::kTotal, st, tq, tk, tv, p)
                     : launch_pdl(prefill_tc_kernel<128>, (int)grid, kTcThreads, TcSmem<128>::kTotal, st, tq, tk, tv,
                                  p);
    } else {
        int smem = 0;
        if (!(HD == 64 ? prepare<64>(&smem) : prepare<128>(&smem))) return MI_ERR_CUDA;
        CUtensorMap tk, tv;
        if (!make_tmap(&tk, k_cache, rows, HD) || !make_tmap(&tv, v_cache, rows, HD)) return MI_ERR_CUDA;
        e = HD == 64 ? launch_pdl(prefill_kernel<64>, (int)grid, (kPWarps + 1) * 32, smem, st, tk, tv, p)
                     : launch_pdl(prefill_kernel<128>, (int)grid, (kPWarps + 1) * 32, smem, st, tk, tv, p);
    }
    return e == cudaSuccess ? MI_OK : MI_ERR_CUDA;
}

}  // namespace
}  // namespace mi

extern "C" mi_status mi_paged_prefill_attention(const mi_dims* dims, int32_t total_q, int32_t max_query_len,
                                                const void* q, const void* k_cache, const void* v_cache,
                                                const int32_t* block_tables, const int32_t* context_lens,
                                                const int32_t* query_start, float scale, void* out,
                                                int32_t* dev_err, mi_stream_t stream) {
    return mi::prefill(dims, total_q, max_query_len, q, k_cache, v_cache, block_tables, context_lens, query_start,
                       scale, out, dev_err, stream, MI_PREFILL_DEFAULT);
}

extern "C" mi_status mi_paged_prefill_attention_variant(const mi_dims* dims, int32_t total_q,
                                                        int32_t max_query_len, const void* q, const void* k_cache,
                                                        const void* v_cache, const int32_t* block_tables,
                                                        const int32_t* context_lens, const int32_t* query_start,
                                                        float scale, void* out, int32_t* dev_err,
                                                        mi_stream_t stream, int32_t variant) {
    return mi::prefill(dims, total_q, max_query_len, q, k_cache, v_cache, block_tables, context_lens, query_start,
                       scale, out, dev_err, stream, variant);
}
