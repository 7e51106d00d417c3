// mi_paged_decode_attention: GQA decode attention over the paged KV cache.
//
// What it computes is the attention inside mini-infer's decode_batch
// model_forward (mini-infer README, "decode_batch 关键步骤"), over the history
// its gather_batch_kv would collect from the block tensor, with GQA as in the
// NJU course brief "端侧大模型推理框架" §2.1 (query head j reads KV head j / G).
// The gather is never materialised: blocks are read in place.
//
// Work decomposition (split-KV, flash-decoding style):
//   * A "unit" is one (request b, KV head h) pair; it owns ceil(n_b / 16) KV
//     blocks. Units are laid end to end in (b, h) order into one flat sequence
//     of TB blocks.
//   * A persistent grid (two CTAs per SM, three for e4m3 tiles) cuts that
//     sequence into equal contiguous ranges, one per CTA, so every CTA
//     streams the same number of bytes however skewed the context lengths
//     are.
//   * Warp specialisation: in each CTA one producer warp walks the block table
//     and issues 2-D TMA tensor copies (128-byte swizzle, one 4 KB box per K
//     or V tile) into a ring of shared-memory stages per consumer warp
//     (full/empty mbarriers); consumer warp w takes blocks w, w+W, ... of the
//     range. The producer never joins the consumers' barriers, so their merges
//     do not interrupt the stream.
//   * One 16-token K/V tile serves all G query heads of the KV head: scores
//     are 16 tokens x G heads on tensor cores (or fp32 FMAs), with an fp32
//     online softmax (base-2 exponent, scale * log2(e) folded into one
//     multiply).
//   * At every unit boundary the consumer warps merge their (max, sum, output)
//     states in shared memory. A unit wholly inside the range is written as
//     bf16 output; a unit cut by range edges leaves a normalised fp32 partial
//     and its log-sum-exp per piece in the workspace, then bumps the unit's
//     counter word (tagged with the call's epoch, so it never needs clearing);
//     the CTA that stores the last piece zeroes the word and merges the unit
//     (log-sum-exp combine). Each CTA streams the cut unit at its range end first, so
//     these merges happen early rather than at the end of the kernel.
// The split depends only on the context lengths and the grid size, so results
// are bitwise independent of which physical blocks a request holds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <random>

#include "common.cuh"
#include "rope.cuh"
#include "tma.cuh"

namespace mi {
namespace {

constexpr int kMaxG = 8;
// Per-unit cost of the split, in blocks (measured: e4m3 best at 12 on a
// Qwen3-8B layer and at 8 on a batch of one 32k and 255 short contexts;
// bf16 flat from 4 to 16 on the Qwen3-8B layer, best at 4-8 on the skewed
// batch)
constexpr int kUnitCostE4m3 = 10;
constexpr int kUnitCostBf16 = 6;
// Fewest blocks a CTA's range is cut to (measured on one layer of 8 requests
// of 200 tokens, 4 KV heads: 11 us with 32 CTAs against 17 us on all 304;
// larger batches keep the whole grid).
constexpr long long kMinBlocksPerCta = 12;
constexpr float kNegInf = -INFINITY;

// An e4m3 scale the FP8 append accepts: positive and finite.
__device__ __forceinline__ bool fp8_scale_ok(float s) { return s > 0.f && s <= 3.0e38f; }

struct AttnParams {
    const uint16_t* q;             // [B][Hq][HD]
    const int32_t* block_tables;   // [B][mbps]
    const int32_t* context_lens;   // [B]
    uint16_t* out;                 // [B][Hq][HD]
    float* part;                   // partial slots [CTAs][2][slot_floats]
    unsigned long long* unit_word; // [CTAs]: per cut unit (at its first piece's CTA): epoch | pieces stored
    unsigned long long epoch;      // distinct per call
    int32_t* dev_err;
    int B, Hq, Hkv, G, num_blocks, mbps, stages, slot_floats;
    int grid;                      // CTAs of the attention kernel
    float sl2;                     // scale * log2(e)
    const float* k_scale;          // [Hkv] e4m3 caches: per-head dequantisation scales
    const float* v_scale;          // [Hkv]
    const float* k_amax;           // [num_blocks][Hkv] INT8 caches: each block's 64-token group maximum
    const float* v_amax;
    // fused decode step only: the new token's raw q / k / v, the RoPE table,
    // q_out and the caches to write the new row into
    const uint16_t* qraw;          // [B][Hq][HD]
    const uint16_t* knew;          // [B][Hkv][HD]
    const uint16_t* vnew;          // [B][Hkv][HD]
    const float2* rope;            // [max_pos][HD/2] (cos, sin)
    uint16_t* q_out;               // [B][Hq][HD]
    uint16_t* kc;                  // [num_blocks][Hkv][16][HD]
    uint16_t* vc;
    int max_pos;
    unsigned char* plan_cache;     // [grid] entries of plan_stride bytes, or null (see PlanEntry)
    int plan_stride;
    int plan_kind;                 // which kernel the plans are for (variant, fused step)
    long long wait_ns;             // bound on every mbarrier wait of the launch
    int early;                     // fused step: plan and first copies before the wait on the kernel before
    int withhold;                  // failure-detection test: each producer withholds its first copy
};

// ------------------------------------------------------------- the plan ---

__device__ __forceinline__ int ctx_clamped(const AttnParams& p, int b) {
    int n = __ldg(p.context_lens + b);
    n = n < 0 ? 0 : n;
    const int cap = p.mbps * kBlock;
    return n > cap ? cap : n;
}

__device__ __forceinline__ int unit_blocks(const AttnParams& p, int b) {
    return b < p.B ? (ctx_clamped(p, b) + kBlock - 1) / kBlock : 0;
}

// A position in the flat unit sequence: unit (b, h) covers flat blocks
// [start, start + len).
struct Cursor {
    int b, h, len;
    long long start;   // first flat block
    long long cstart;  // cost position: every unit before it costs len + uc
    int uc;            // per-unit cost of the split, in blocks
    __device__ __forceinline__ void next(const AttnParams& p) {
        start += len;
        cstart += len + uc;
        if (++h == p.Hkv) {
            h = 0;
            ++b;
            len = unit_blocks(p, b);
            while (len == 0 && b < p.B) len = unit_blocks(p, ++b);
        }
    }
    __device__ __forceinline__ void advance_to(const AttnParams& p, long long x) {
        while (x >= start + len && b < p.B) next(p);
    }
};

// Block-wide exclusive scan of the per-thread values v (one per thread).
// Writes scratch[tid] = sum of v over threads < tid and scratch[nt] = total.
// `scratch` holds blockDim.x + 1 long longs plus 32 more for warp totals.
__device__ void block_exclusive_scan(long long v, long long* scratch) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = (blockDim.x + 31) >> 5;
    long long* wsum = scratch + blockDim.x + 1;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        long long t = lane < nw ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) wsum[lane] = t;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const long long before = (wid ? wsum[wid - 1] : 0) + x - v;
    scratch[tid] = before;
    if (tid == blockDim.x - 1) scratch[blockDim.x] = before + v;
    __syncthreads();
}

// The scan packs two sums in one word: flat blocks in the low kCntShift bits,
// the number of requests with at least one block above them (B < 2^17 and
// B * max_blocks_per_seq < 2^46, so neither field spills into the other).
constexpr int kCntShift = 46;
constexpr long long kBlkMask = (1LL << kCntShift) - 1;
__device__ __forceinline__ long long sc_blocks(long long v) { return v & kBlkMask; }
// cost = blocks + uc per unit with blocks (per KV head: multiply by Hkv)
__device__ __forceinline__ long long sc_cost(long long v, int uc) {
    return (v & kBlkMask) + (long long)uc * (v >> kCntShift);
}

// Each thread sums the unit lengths (and counts the non-empty requests) of a
// contiguous chunk of requests; after the scan, scan[t] holds the sums before
// chunk t and scan[nt] the totals. Returns TB = Hkv * total blocks and sets
// TC = Hkv * total cost, a unit costing its blocks plus uc.
__device__ __forceinline__ long long plan_scan(const AttnParams& p, int uc, long long* scan, long long& TC) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (p.B + nt - 1) / nt;
    const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
    long long s = 0, c = 0;
    for (int b = b0; b < b1; ++b) {
        const int L = unit_blocks(p, b);
        s += L;
        c += L > 0 ? 1 : 0;
    }
    block_exclusive_scan(s | (c << kCntShift), scan);
    TC = sc_cost(scan[nt], uc) * p.Hkv;
    return sc_blocks(scan[nt]) * p.Hkv;
}

// a / b for the plan's non-negative sizes: a 32-bit division when both fit
// (every workload of practical size), which is several times shorter than
// the 64-bit one.
__device__ __forceinline__ unsigned long long udiv(unsigned long long a, unsigned long long b) {
    if ((a | b) <= 0xFFFFFFFFull) return (unsigned)a / (unsigned)b;
    return a / b;
}

// Walks of one chunk of the scan (requests t*per .. of thread t): the unit
// holding flat block x, and the unit holding cost position y together with
// the flat block y maps to. The caller makes sure the chunk holds x (or y).

// The unit holding flat block x.
__device__ Cursor walk_block(const AttnParams& p, int uc, const long long* scan, int nt, int t, long long x) {
    const int per = (p.B + nt - 1) / nt;
    int b = t * per;
    long long acc = sc_blocks(scan[t]), cacc = sc_cost(scan[t], uc);
    int L = unit_blocks(p, b);
    while (x >= (acc + L) * p.Hkv) {
        acc += L;
        cacc += L > 0 ? L + uc : 0;
        L = unit_blocks(p, ++b);
    }
    Cursor c;
    c.b = b;
    c.len = L;
    c.h = (int)udiv((unsigned long long)(x - acc * p.Hkv), (unsigned long long)L);
    c.start = acc * p.Hkv + (long long)c.h * L;
    c.cstart = cacc * p.Hkv + (long long)c.h * (L + uc);
    c.uc = uc;
    return c;
}

// Units are laid out in cost space as uc of overhead followed by their
// blocks; a position in a unit's overhead maps to the unit's first block, so
// the map is monotone in y (the identity when uc = 0). Returns the unit
// holding that block and sets x to it.
__device__ Cursor walk_cost(const AttnParams& p, int uc, const long long* scan, int nt, int t, long long y,
                            long long& x) {
    const int per = (p.B + nt - 1) / nt;
    int b = t * per;
    long long acc = sc_blocks(scan[t]), cacc = sc_cost(scan[t], uc);
    int L = unit_blocks(p, b);
    long long W = L > 0 ? L + uc : 0;
    while (y >= (cacc + W) * p.Hkv) {
        acc += L;
        cacc += W;
        L = unit_blocks(p, ++b);
        W = L > 0 ? L + uc : 0;
    }
    const long long r = y - cacc * p.Hkv;
    const long long h = (long long)udiv((unsigned long long)r, (unsigned long long)W), o = r - h * W - uc;
    x = acc * p.Hkv + h * L + (o > 0 ? o : 0);
    Cursor c;
    c.b = b;
    c.len = L;
    c.h = (int)h;
    c.start = acc * p.Hkv + h * L;
    c.cstart = cacc * p.Hkv + h * W;
    c.uc = uc;
    return c;
}

// Range of CTA i of P over TB flat blocks.
__device__ __forceinline__ long long range_start(long long TB, int P, int i) {
    return (long long)udiv((unsigned long long)TB * (unsigned long long)i, (unsigned long long)P);
}

// The CTA whose range holds position x (0 <= x < TB); used on cost positions
// with TB = TC.
__device__ __forceinline__ int cta_of(long long TB, int P, long long x) {
    int c = (int)udiv((unsigned long long)x * (unsigned long long)P, (unsigned long long)TB);
    while (c > 0 && range_start(TB, P, c) > x) --c;
    while (c + 1 < P && range_start(TB, P, c + 1) <= x) ++c;
    return c;
}


// A CTA's share of the flat block sequence, in shared memory: the range
// [ra, rb) and the split point sl. When the range's last unit starts inside
// the range and continues past rb, it is streamed first: part 0 = [sl, rb),
// then part 1 = [ra, sl) (both pieces of every cut unit are then written
// early and their merge does not land at the end of the kernel); otherwise
// sl = rb. c0 is the unit holding sl (used when sl < rb), c1 the unit holding
// ra (used when ra < sl).
struct RangePlan {
    long long ra, rb, sl;
    Cursor c0, c1;
};

// A CTA's plan kept in the workspace for the next launch: the split depends
// only on the context lengths, the dims, the grid and the kernel, and every
// layer of a decode step has the same lengths, so each later layer's CTA
// finds its range here instead of recomputing the scan. An entry is used only
// when its key (which names the CTA) and its copy of all B lengths equal the
// launch's exactly and its hash matches its plan words, and a CTA reads and
// writes only its own entry. The CTA in the key matters when a workspace is
// given at another address over memory that still holds entries (a buffer
// freed and handed out again at a shifted offset): the entry found at a
// CTA's position may then be another CTA's. The hash catches an entry whose
// plan words were overwritten (the same memory used as the workspace of
// other dims) while its key and lengths survived. The lengths follow the
// header: int32 lens[B].
struct PlanEntry {
    int32_t key[8];                // kPlanMagic, kind, B, Hkv, mbps, grid, uc, CTA
    int32_t P;
    uint32_t sum;                  // plan_sum of (P, TB, TC, rp)
    long long TB, TC;
    RangePlan rp;
};
constexpr int32_t kPlanMagic = 0x6E616C50;  // "Plan"
constexpr int kPlanMaxB = 1024;               // larger batches always compute their plan
__host__ __device__ inline int plan_stride_for(int B) {
    return B > kPlanMaxB ? 0 : (int)((sizeof(PlanEntry) + 4 * (size_t)B + 127) / 128 * 128);
}

// Hash of an entry's plan words (P, TB, TC, then the range plan as 32-bit
// words, rp in shared memory), each mixed with its position; every lane of
// the calling warp gets the same value.
__device__ uint32_t plan_sum(int P, long long TB, long long TC, const RangePlan* rp, int lane) {
    constexpr int nrp = (int)(sizeof(RangePlan) / 4);
    uint32_t h = 0;
    for (int i = lane; i < 5 + nrp; i += 32) {
        uint32_t v;
        if (i == 0)
            v = (uint32_t)P;
        else if (i < 3)
            v = (uint32_t)((unsigned long long)TB >> (32 * (i - 1)));
        else if (i < 5)
            v = (uint32_t)((unsigned long long)TC >> (32 * (i - 3)));
        else
            v = reinterpret_cast<const uint32_t*>(rp)[i - 5];
        uint32_t x = (v ^ (0x9E3779B9u * (uint32_t)(i + 1))) * 0x85EBCA6Bu;
        x ^= x >> 15;
        h ^= x * 0xC2B2AE35u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) h ^= __shfl_xor_sync(0xffffffffu, h, o);
    return h;
}

// Every thread of the CTA calls this after plan_scan. The ranges are of equal
// cost (range_start over TC); each end is resolved by the one thread whose
// scan chunk holds it, with a barrier after each of the two steps, instead
// of a search by every thread.
__device__ void plan_ranges(const AttnParams& p, int uc, const long long* scan, long long TB, long long TC, int P,
                            RangePlan* rp) {
    const int t = threadIdx.x, nt = blockDim.x, cta = blockIdx.x;
    if (cta < P) {
        const long long ya = range_start(TC, P, cta), yb = range_start(TC, P, cta + 1);
        const long long lo = sc_cost(scan[t], uc) * p.Hkv, hi = sc_cost(scan[t + 1], uc) * p.Hkv;
        long long x = 0;
        if (ya >= lo && ya < hi) {
            rp->c1 = walk_cost(p, uc, scan, nt, t, ya, x);
            rp->ra = x;
        }
        if (yb >= lo && yb < hi) {
            (void)walk_cost(p, uc, scan, nt, t, yb, x);
            rp->rb = x;
        }
        if (t == 0) {
            if (ya >= TC) rp->ra = TB;
            if (yb >= TC) rp->rb = TB;
        }
    } else if (t == 0) {
        rp->ra = rp->rb = 0;
    }
    __syncthreads();
    const long long ra = rp->ra, rb = rp->rb;
    if (rb > ra) {
        const long long xl = rb - 1;
        if (xl >= sc_blocks(scan[t]) * p.Hkv && xl < sc_blocks(scan[t + 1]) * p.Hkv) {
            const Cursor cl = walk_block(p, uc, scan, nt, t, xl);
            rp->c0 = cl;
            rp->sl = (cl.start > ra && cl.start + cl.len > rb) ? cl.start : rb;
        }
    } else if (t == 0) {
        rp->sl = rb;
    }
    __syncthreads();
}

// prefetch.global.L2 of this CTA's share (1 / gridDim.x) of a buffer, one
// 128-byte line per lane step: the first reads after the plan then hit L2.
__device__ __forceinline__ void prefetch_share(const void* base, long long bytes, int lane) {
    if (!base || bytes <= 0) return;
    const long long lines = (bytes + 127) / 128;
    const long long a = lines * blockIdx.x / gridDim.x, b = lines * (blockIdx.x + 1) / gridDim.x;
    const char* c = static_cast<const char*>(base);
    for (long long l = a + lane; l < b; l += 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + l * 128));
}

// ------------------------------------------------------- smem layout ------

enum { kVarMma = 1, kVarFma = 2, kVarFp8 = 3, kVarInt8 = 4 };

// Bytes of one cache element: bf16, or one byte for the e4m3 and INT8 variants.
__host__ __device__ constexpr int elem_bytes(int var) { return var == kVarFp8 || var == kVarInt8 ? 1 : 2; }

template <int HD, int EB>
struct Tile {
    static constexpr int kBytes = kBlock * HD * EB;  // one 16-token K or V tile
};

struct SmemPlan {
    int tiles, full, empty, okf, amx, mbuf, lbuf, obuf, xbuf, scan, flag, rplan, qring, qbar, total;
};

// W consumer warps plus one producer warp (and, for the fused step, one RoPE
// warp); S stages per consumer warp. The weight-exchange buffer is only needed
// by the CUDA-core tile; the fused step adds a two-slot ring of rotated q rows
// ([G][HD] bf16 each) with full / empty barriers. INT8 tiles add, per stage,
// the block's K and V group maxima.
__host__ __device__ inline SmemPlan smem_plan(int W, int S, int HD, int G, bool fma, int eb = 2,
                                             bool fused = false, bool amx = false) {
    SmemPlan s;
    int off = 0;
    s.tiles = off; off += W * S * 2 * kBlock * HD * eb;
    s.full = off;  off += W * S * 8;
    s.empty = off; off += W * S * 8;
    s.okf = off;   off += W * S * 4;  // per stage: nonzero when its block id was valid and copied
    off = (off + 15) & ~15;
    s.amx = off;   off += amx ? W * S * 8 : 0;
    s.mbuf = off;  off += W * kMaxG * 4;
    s.lbuf = off;  off += W * kMaxG * 4;
    s.obuf = off;  off += W * G * HD * 4;
    s.xbuf = off;  off += fma ? W * (kBlock * kMaxG + kMaxG) * 4 : 0;
    off = (off + 15) & ~15;
    s.scan = off;  off += ((W + (fused ? 2 : 1)) * 32 + 1 + 32) * 8;
    s.flag = off;  off += 16;
    s.rplan = off; off += (int)((sizeof(RangePlan) + 15) & ~(size_t)15);
    s.qring = off; off += fused ? 2 * (G + 2) * HD * 2 : 0;  // per slot: q rows [G][HD], new k row, new v row
    s.qbar = off;  off += fused ? 6 * 8 : 0;  // q full [2], empty [2], k/v rows full [2]
    s.total = off + 1024;  // slack to align the tiles to 1024 bytes
    return s;
}

// ---------------------------------------------------- per-warp compute ----

// Tensor-core tile: S^T[16 tokens x 8 heads] = K[16 x HD] . Q^T[HD x 8] with
// mma.sync m16n8k16 (heads beyond G are zero columns), online softmax on the
// fragments, then O^T[HD x 8] += V^T[HD x 16] . P^T[16 x 8] (V^T by
// ldmatrix.trans, P^T by movmatrix.trans of the score fragments).
template <int HD>
struct MmaState {
    static constexpr int kK = HD / 16;
    uint32_t qb[kK][2];
    float o[kK][4];
    float m[2], l[2];

    __device__ __forceinline__ void begin_unit(const AttnParams& p, int b, int h, int lane) {
        const int n = lane >> 2;
        const bool ok = n < p.G;
        const uint16_t* qrow = p.q + ((long long)b * p.Hq + (long long)h * p.G + (ok ? n : 0)) * HD;
#pragma unroll
        for (int kk = 0; kk < kK; ++kk) {
            const int dcol = kk * 16 + (lane & 3) * 2;
            qb[kk][0] = ok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + dcol)) : 0u;
            qb[kk][1] = ok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + dcol + 8)) : 0u;
        }
#pragma unroll
        for (int mt = 0; mt < kK; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kNegInf;
        l[0] = l[1] = 0.f;
    }

    // The fused decode step: q of the unit's heads from rotated rows [G][HD]
    // bf16 in shared memory (the RoPE warp's ring slot).
    __device__ __forceinline__ void begin_unit_from(const uint16_t* qrows, const AttnParams& p, int /*h*/,
                                                    int lane) {
        const int n = lane >> 2;
        const bool ok = n < p.G;
        const uint16_t* qrow = qrows + (ok ? n : 0) * HD;
#pragma unroll
        for (int kk = 0; kk < kK; ++kk) {
            const int dcol = kk * 16 + (lane & 3) * 2;
            qb[kk][0] = ok ? *reinterpret_cast<const uint32_t*>(qrow + dcol) : 0u;
            qb[kk][1] = ok ? *reinterpret_cast<const uint32_t*>(qrow + dcol + 8) : 0u;
        }
#pragma unroll
        for (int mt = 0; mt < kK; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kNegInf;
        l[0] = l[1] = 0.f;
    }

    __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int valid, float sl2, int lane) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
            // two accumulation chains (even / odd k-slices) halve the
            // dependent MMA latency
            float c1[4] = {0.f, 0.f, 0.f, 0.f};
            const int tok = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int csel = lane >> 4;
#pragma unroll
            for (int kk = 0; kk < kK; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kt + swz<HD>(tok, kk * 2 + csel), a0, a1, a2, a3);
                mma_bf16_16816(kk & 1 ? c1 : c, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) c[i] += c1[i];
        }
        const int t0 = lane >> 2, t1 = t0 + 8;
        float s0 = t0 < valid ? c[0] * sl2 : kNegInf;  // head 2*(lane&3),   token t0
        float s1 = t0 < valid ? c[1] * sl2 : kNegInf;  // head 2*(lane&3)+1, token t0
        float s2 = t1 < valid ? c[2] * sl2 : kNegInf;  // head 2*(lane&3),   token t1
        float s3 = t1 < valid ? c[3] * sl2 : kNegInf;  // head 2*(lane&3)+1, token t1
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float r0 = mn0 == kNegInf ? 0.f : mn0, r1 = mn1 == kNegInf ? 0.f : mn1;
        const float al0 = ex2(m[0] - r0), al1 = ex2(m[1] - r1);
        m[0] = mn0;
        m[1] = mn1;
        const uint32_t x0 = pack_bf16x2(ex2(s0 - r0), ex2(s1 - r1));
        const uint32_t x1 = pack_bf16x2(ex2(s2 - r0), ex2(s3 - r1));
        // the sums use the same bf16-rounded weights the PV product uses
        l[0] = l[0] * al0 + (bf16_lo(x0) + bf16_lo(x1));
        l[1] = l[1] * al1 + (bf16_hi(x0) + bf16_hi(x1));
        // the running max rarely moves once a few blocks are in: skip the
        // rescale when no lane's factor differs from 1
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < kK; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
        }
        const uint32_t b0 = movmatrix_trans(x0), b1 = movmatrix_trans(x1);
        {
            const int qd = lane >> 3;
            const int tok = (lane & 7) + (qd >> 1) * 8;
            const int csel = qd & 1;
#pragma unroll
            for (int mt = 0; mt < kK; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(vt + swz<HD>(tok, mt * 2 + csel), a0, a1, a2, a3);
                mma_bf16_16816(o[mt], a0, a1, a2, a3, b0, b1);
            }
        }
    }

    // Reduce the per-thread sums and write (m, l, O) of this warp to smem.
    __device__ __forceinline__ void store(float* mbuf, float* lbuf, float* obuf, int G, int lane) {
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], sh);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], sh);
        }
        const int h0 = (lane & 3) * 2, h1 = h0 + 1;
        if (lane < 4) {
            if (h0 < G) { mbuf[h0] = m[0]; lbuf[h0] = l[0]; }
            if (h1 < G) { mbuf[h1] = m[1]; lbuf[h1] = l[1]; }
        }
        const int r = lane >> 2;
#pragma unroll
        for (int mt = 0; mt < kK; ++mt) {
            if (h0 < G) {
                obuf[h0 * HD + mt * 16 + r] = o[mt][0];
                obuf[h0 * HD + mt * 16 + r + 8] = o[mt][2];
            }
            if (h1 < G) {
                obuf[h1 * HD + mt * 16 + r] = o[mt][1];
                obuf[h1 * HD + mt * 16 + r + 8] = o[mt][3];
            }
        }
    }
};

// Tensor-core tile over e4m3 (FP8) K/V tiles, the MMA tile's arithmetic in
// f16 (every e4m3 value is an f16 value, and f16 keeps 11 bits of the
// probabilities). S^T = K . Q^T: ldmatrix hands each lane four consecutive K
// bytes of a token row, which convert to two f16 pairs; within every 16-dim
// k-slice the lane's k slots (2c, 2c+1) and (2c+8, 2c+9) are taken to be dims
// (4c, 4c+1) and (4c+2, 4c+3), and Q's fragments are loaded in the same order,
// so the dot products are unchanged. O^T = V^T . P^T: each lane reads four
// bytes (dims 4j..4j+3) of token rows 2c, 2c+1, 2c+8, 2c+9, byte-permutes
// them into (token pair, dim) pairs and converts; the 16 O^T rows of a tile
// pair are dims 4(8t + r) + {0, 1} (even tile) and + {2, 3} (odd tile).
// K's per-head scale folds into the exponent scale, V's into the output.
template <int HD>
struct Fp8State {
    static constexpr int kK = HD / 16;
    uint32_t qb[kK][2];
    float o[kK][4];
    float m[2], l[2];
    float sl2, vsc;

    __device__ __forceinline__ void begin_unit(const AttnParams& p, int b, int h, int lane) {
        const int n = lane >> 2, c = lane & 3;
        const bool ok = n < p.G;
        const uint16_t* qrow = p.q + ((long long)b * p.Hq + (long long)h * p.G + (ok ? n : 0)) * HD;
#pragma unroll
        for (int kk = 0; kk < kK; ++kk) {
            const uint2 w = ok ? __ldg(reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * c)) : make_uint2(0, 0);
            qb[kk][0] = pack_f16x2(bf16_lo(w.x), bf16_hi(w.x));  // dims 4c, 4c+1
            qb[kk][1] = pack_f16x2(bf16_lo(w.y), bf16_hi(w.y));  // dims 4c+2, 4c+3
        }
#pragma unroll
        for (int mt = 0; mt < kK; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kNegInf;
        l[0] = l[1] = 0.f;
        sl2 = p.sl2 * __ldg(p.k_scale + h);
        vsc = __ldg(p.v_scale + h);
    }

    // The fused decode step: q of the unit's heads from rotated rows [G][HD]
    // bf16 in shared memory (the RoPE warp's ring slot), in the same order.
    __device__ __forceinline__ void begin_unit_from(const uint16_t* qrows, const AttnParams& p, int h, int lane) {
        const int n = lane >> 2, c = lane & 3;
        const bool ok = n < p.G;
        const uint16_t* qrow = qrows + (ok ? n : 0) * HD;
#pragma unroll
        for (int kk = 0; kk < kK; ++kk) {
            const uint2 w = ok ? *reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * c) : make_uint2(0, 0);
            qb[kk][0] = pack_f16x2(bf16_lo(w.x), bf16_hi(w.x));
            qb[kk][1] = pack_f16x2(bf16_lo(w.y), bf16_hi(w.y));
        }
#pragma unroll
        for (int mt = 0; mt < kK; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kNegInf;
        l[0] = l[1] = 0.f;
        sl2 = p.sl2 * __ldg(p.k_scale + h);
        vsc = __ldg(p.v_scale + h);
    }

    __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int valid, float /*sl2 of bf16*/, int lane) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
            float c1[4] = {0.f, 0.f, 0.f, 0.f};  // second accumulation chain (odd k-slices)
            const int mi = lane >> 3;
            const int tok = (lane & 7) + (mi & 1) * 8;
#pragma unroll
            for (int kp = 0; kp < kK / 2; ++kp) {
                uint32_t r0, r1, r2, r3;  // tokens g / g+8 of k-slices 2kp / 2kp+1
                ldsm_x4(kt + swz8<HD>(tok, 2 * kp + (mi >> 1)), r0, r1, r2, r3);
                mma_f16_16816(c, e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                              e4m3x2_to_f16x2(r1 >> 16), qb[2 * kp][0], qb[2 * kp][1]);
                mma_f16_16816(c1, e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                              e4m3x2_to_f16x2(r3 >> 16), qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) c[i] += c1[i];
        }
        const int t0 = lane >> 2, t1 = t0 + 8;
        float s0 = t0 < valid ? c[0] * sl2 : kNegInf;
        float s1 = t0 < valid ? c[1] * sl2 : kNegInf;
        float s2 = t1 < valid ? c[2] * sl2 : kNegInf;
        float s3 = t1 < valid ? c[3] * sl2 : kNegInf;
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float r0 = mn0 == kNegInf ? 0.f : mn0, r1 = mn1 == kNegInf ? 0.f : mn1;
        const float al0 = ex2(m[0] - r0), al1 = ex2(m[1] - r1);
        m[0] = mn0;
        m[1] = mn1;
        const uint32_t x0 = pack_f16x2(ex2(s0 - r0), ex2(s1 - r1));
        const uint32_t x1 = pack_f16x2(ex2(s2 - r0), ex2(s3 - r1));
        l[0] = l[0] * al0 + (f16_lo(x0) + f16_lo(x1));
        l[1] = l[1] * al1 + (f16_hi(x0) + f16_hi(x1));
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < kK; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
        }
        const uint32_t b0 = movmatrix_trans(x0), b1 = movmatrix_trans(x1);
        {
            const int g = lane >> 2, cc = lane & 3;
#pragma unroll
            for (int t = 0; t < kK / 2; ++t) {
                // dims 4j .. 4j+3, j = 8t + g, of token rows 2cc, 2cc+1, 2cc+8, 2cc+9
                const int chunk = 2 * t + (g >> 2), inb = (g & 3) * 4;
                const uint32_t w0 = lds32(vt + swz8<HD>(2 * cc, chunk) + inb);
                const uint32_t w1 = lds32(vt + swz8<HD>(2 * cc + 1, chunk) + inb);
                const uint32_t w2 = lds32(vt + swz8<HD>(2 * cc + 8, chunk) + inb);
                const uint32_t w3 = lds32(vt + swz8<HD>(2 * cc + 9, chunk) + inb);
                const uint32_t lo01 = __byte_perm(w0, w1, 0x5140), hi01 = __byte_perm(w0, w1, 0x7362);
                const uint32_t lo89 = __byte_perm(w2, w3, 0x5140), hi89 = __byte_perm(w2, w3, 0x7362);
                mma_f16_16816(o[2 * t], e4m3x2_to_f16x2(lo01), e4m3x2_to_f16x2(lo01 >> 16), e4m3x2_to_f16x2(lo89),
                              e4m3x2_to_f16x2(lo89 >> 16), b0, b1);
                mma_f16_16816(o[2 * t + 1], e4m3x2_to_f16x2(hi01), e4m3x2_to_f16x2(hi01 >> 16),
                              e4m3x2_to_f16x2(hi89), e4m3x2_to_f16x2(hi89 >> 16), b0, b1);
            }
        }
    }

    // Reduce the per-thread sums and write (m, l, O * v_scale) of this warp to smem.
    __device__ __forceinline__ void store(float* mbuf, float* lbuf, float* obuf, int G, int lane) {
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], sh);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], sh);
        }
        const int h0 = (lane & 3) * 2, h1 = h0 + 1;
        if (lane < 4) {
            if (h0 < G) { mbuf[h0] = m[0]; lbuf[h0] = l[0]; }
            if (h1 < G) { mbuf[h1] = m[1]; lbuf[h1] = l[1]; }
        }
        const int r = lane >> 2;
#pragma unroll
        for (int t = 0; t < kK / 2; ++t) {
            const int d0 = 4 * (8 * t + r);
            if (h0 < G) {
                obuf[h0 * HD + d0] = o[2 * t][0] * vsc;
                obuf[h0 * HD + d0 + 1] = o[2 * t][2] * vsc;
                obuf[h0 * HD + d0 + 2] = o[2 * t + 1][0] * vsc;
                obuf[h0 * HD + d0 + 3] = o[2 * t + 1][2] * vsc;
            }
            if (h1 < G) {
                obuf[h1 * HD + d0] = o[2 * t][1] * vsc;
                obuf[h1 * HD + d0 + 1] = o[2 * t][3] * vsc;
                obuf[h1 * HD + d0 + 2] = o[2 * t + 1][1] * vsc;
                obuf[h1 * HD + d0 + 3] = o[2 * t + 1][3] * vsc;
            }
        }
    }
};

// Tensor-core tile over INT8 K/V tiles quantised in 64-token groups: the e4m3
// tile's data movement and fragment orders. Each code enters the MMAs as the
// f16 value 1152 + code (a byte permute, exact), and the bias is taken back
// off the results: from the scores, 1152 times the sum of the head's q (a
// constant per head, folded into the scaling FMA); from O, 1152 times the
// sum of the f16 probabilities that went into the PV products (summed per
// lane like the running sum and subtracted once, at the store). A block's
// codes stand for code * a / 127, a the maximum of its group (one per block
// and head, staged with the tile): K's factor multiplies the block's scores;
// V's factor is taken relative to a reference factor of the warp (the first
// block's, raised, with a rescale of O, when a block's factor exceeds it
// 256-fold) and multiplies the f16 probabilities of the block (at most 256,
// so within f16's range), while the running sum keeps the unscaled ones. O
// times the reference is the output.
template <int HD>
struct Int8State {
    static constexpr int kK = HD / 16;
    static constexpr uint32_t kFlip = 0x80808080u;  // sign bits: codes to offset binary
    static constexpr uint32_t kLo = 0x4140u, kHi = 0x4342u;
    static constexpr float kBias = 1152.f;
    uint32_t qb[kK][2];
    float o[kK][4];
    float m[2], l[2];
    float koff[2];  // kBias * sum of q over the dims, for this lane's two heads
    float sp[2];    // this lane's sum of the f16 probabilities fed to the PV products
    float sl2, vref, rvref;

    __device__ __forceinline__ void reset(const AttnParams& p, int lane) {
#pragma unroll
        for (int mt = 0; mt < kK; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m[0] = m[1] = kNegInf;
        l[0] = l[1] = 0.f;
        sp[0] = sp[1] = 0.f;
        sl2 = p.sl2 * (1.f / 127.f);
        vref = 0.f;
        rvref = 0.f;
        // q's sum per head: lane (n, c) holds dims 4c..4c+3 of every 16-dim
        // slice of head n; the quad reduces, then each lane takes the sums of
        // the heads its score columns hold (2c and 2c + 1)
        float qs = 0.f;
#pragma unroll
        for (int kk = 0; kk < kK; ++kk)
            qs += (f16_lo(qb[kk][0]) + f16_hi(qb[kk][0])) + (f16_lo(qb[kk][1]) + f16_hi(qb[kk][1]));
        qs += __shfl_xor_sync(0xffffffffu, qs, 1);
        qs += __shfl_xor_sync(0xffffffffu, qs, 2);
        koff[0] = kBias * __shfl_sync(0xffffffffu, qs, 8 * (lane & 3));
        koff[1] = kBias * __shfl_sync(0xffffffffu, qs, 8 * (lane & 3) + 4);
    }

    __device__ __forceinline__ void begin_unit(const AttnParams& p, int b, int h, int lane) {
        const int n = lane >> 2, c = lane & 3;
        const bool ok = n < p.G;
        const uint16_t* qrow = p.q + ((long long)b * p.Hq + (long long)h * p.G + (ok ? n : 0)) * HD;
#pragma unroll
        for (int kk = 0; kk < kK; ++kk) {
            const uint2 w = ok ? __ldg(reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * c)) : make_uint2(0, 0);
            qb[kk][0] = pack_f16x2(bf16_lo(w.x), bf16_hi(w.x));  // dims 4c, 4c+1
            qb[kk][1] = pack_f16x2(bf16_lo(w.y), bf16_hi(w.y));  // dims 4c+2, 4c+3
        }
        reset(p, lane);
    }

    __device__ __forceinline__ void begin_unit_from(const uint16_t*, const AttnParams& p, int, int lane) {
        reset(p, lane);
    }

    __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int valid, int lane, float ak, float av) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        {
            float c1[4] = {0.f, 0.f, 0.f, 0.f};  // second accumulation chain (odd k-slices)
            const int mi = lane >> 3;
            const int tok = (lane & 7) + (mi & 1) * 8;
#pragma unroll
            for (int kp = 0; kp < kK / 2; ++kp) {
                uint32_t r0, r1, r2, r3;  // tokens g / g+8 of k-slices 2kp / 2kp+1
                ldsm_x4(kt + swz8<HD>(tok, 2 * kp + (mi >> 1)), r0, r1, r2, r3);
                r0 ^= kFlip;
                r1 ^= kFlip;
                r2 ^= kFlip;
                r3 ^= kFlip;
                mma_f16_16816(c, i8x2_to_f16x2_biased(r0, kLo), i8x2_to_f16x2_biased(r1, kLo),
                              i8x2_to_f16x2_biased(r0, kHi), i8x2_to_f16x2_biased(r1, kHi), qb[2 * kp][0],
                              qb[2 * kp][1]);
                mma_f16_16816(c1, i8x2_to_f16x2_biased(r2, kLo), i8x2_to_f16x2_biased(r3, kLo),
                              i8x2_to_f16x2_biased(r2, kHi), i8x2_to_f16x2_biased(r3, kHi), qb[2 * kp + 1][0],
                              qb[2 * kp + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) c[i] += c1[i];
        }
        const float ks = sl2 * ak;  // scale * log2(e) * a_k / 127
        const float kb0 = ks * koff[0], kb1 = ks * koff[1];
        const int t0 = lane >> 2, t1 = t0 + 8;
        float s0 = t0 < valid ? fmaf(c[0], ks, -kb0) : kNegInf;
        float s1 = t0 < valid ? fmaf(c[1], ks, -kb1) : kNegInf;
        float s2 = t1 < valid ? fmaf(c[2], ks, -kb0) : kNegInf;
        float s3 = t1 < valid ? fmaf(c[3], ks, -kb1) : kNegInf;
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float r0 = mn0 == kNegInf ? 0.f : mn0, r1 = mn1 == kNegInf ? 0.f : mn1;
        float al0 = ex2(m[0] - r0), al1 = ex2(m[1] - r1);
        m[0] = mn0;
        m[1] = mn1;
        const float p0 = ex2(s0 - r0), p1 = ex2(s1 - r1), p2 = ex2(s2 - r0), p3 = ex2(s3 - r1);
        l[0] = l[0] * al0 + (p0 + p2);
        l[1] = l[1] * al1 + (p1 + p3);
        // V's factor relative to the reference (the same for every lane)
        const float fv = av * (1.f / 127.f);
        float ov0 = al0, ov1 = al1;  // O's factors for this block
        if (fv > vref * 256.f) {
            const float f = vref * (1.f / fv);  // 0 for the first nonzero factor (O is still 0)
            ov0 *= f;
            ov1 *= f;
            vref = fv;
            rvref = 1.f / fv;
        }
        const float rel = fv * rvref;
        const uint32_t x0 = pack_f16x2(p0 * rel, p1 * rel);
        const uint32_t x1 = pack_f16x2(p2 * rel, p3 * rel);
        sp[0] = sp[0] * ov0 + (f16_lo(x0) + f16_lo(x1));
        sp[1] = sp[1] * ov1 + (f16_hi(x0) + f16_hi(x1));
        if (__any_sync(0xffffffffu, ov0 != 1.f || ov1 != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < kK; ++mt) {
                o[mt][0] *= ov0;
                o[mt][1] *= ov1;
                o[mt][2] *= ov0;
                o[mt][3] *= ov1;
            }
        }
        const uint32_t b0 = movmatrix_trans(x0), b1 = movmatrix_trans(x1);
        {
            const int g = lane >> 2, cc = lane & 3;
#pragma unroll
            for (int t = 0; t < kK / 2; ++t) {
                // dims 4j .. 4j+3, j = 8t + g, of token rows 2cc, 2cc+1, 2cc+8, 2cc+9
                const int chunk = 2 * t + (g >> 2), inb = (g & 3) * 4;
                const uint32_t w0 = lds32(vt + swz8<HD>(2 * cc, chunk) + inb);
                const uint32_t w1 = lds32(vt + swz8<HD>(2 * cc + 1, chunk) + inb);
                const uint32_t w2 = lds32(vt + swz8<HD>(2 * cc + 8, chunk) + inb);
                const uint32_t w3 = lds32(vt + swz8<HD>(2 * cc + 9, chunk) + inb);
                const uint32_t lo01 = __byte_perm(w0, w1, 0x5140) ^ kFlip, hi01 = __byte_perm(w0, w1, 0x7362) ^ kFlip;
                const uint32_t lo89 = __byte_perm(w2, w3, 0x5140) ^ kFlip, hi89 = __byte_perm(w2, w3, 0x7362) ^ kFlip;
                mma_f16_16816(o[2 * t], i8x2_to_f16x2_biased(lo01, kLo), i8x2_to_f16x2_biased(lo01, kHi),
                              i8x2_to_f16x2_biased(lo89, kLo), i8x2_to_f16x2_biased(lo89, kHi), b0, b1);
                mma_f16_16816(o[2 * t + 1], i8x2_to_f16x2_biased(hi01, kLo), i8x2_to_f16x2_biased(hi01, kHi),
                              i8x2_to_f16x2_biased(hi89, kLo), i8x2_to_f16x2_biased(hi89, kHi), b0, b1);
            }
        }
    }

    // Reduce the per-thread sums and write (m, l, (O - bias * probability
    // sum) * reference) of this warp to smem.
    __device__ __forceinline__ void store(float* mbuf, float* lbuf, float* obuf, int G, int lane) {
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            l[0] += __shfl_xor_sync(0xffffffffu, l[0], sh);
            l[1] += __shfl_xor_sync(0xffffffffu, l[1], sh);
            sp[0] += __shfl_xor_sync(0xffffffffu, sp[0], sh);
            sp[1] += __shfl_xor_sync(0xffffffffu, sp[1], sh);
        }
        const int h0 = (lane & 3) * 2, h1 = h0 + 1;
        if (lane < 4) {
            if (h0 < G) { mbuf[h0] = m[0]; lbuf[h0] = l[0]; }
            if (h1 < G) { mbuf[h1] = m[1]; lbuf[h1] = l[1]; }
        }
        const float b0 = kBias * sp[0], b1 = kBias * sp[1];
        const int r = lane >> 2;
#pragma unroll
        for (int t = 0; t < kK / 2; ++t) {
            const int d0 = 4 * (8 * t + r);
            if (h0 < G) {
                obuf[h0 * HD + d0] = (o[2 * t][0] - b0) * vref;
                obuf[h0 * HD + d0 + 1] = (o[2 * t][2] - b0) * vref;
                obuf[h0 * HD + d0 + 2] = (o[2 * t + 1][0] - b0) * vref;
                obuf[h0 * HD + d0 + 3] = (o[2 * t + 1][2] - b0) * vref;
            }
            if (h1 < G) {
                obuf[h1 * HD + d0] = (o[2 * t][1] - b1) * vref;
                obuf[h1 * HD + d0 + 1] = (o[2 * t][3] - b1) * vref;
                obuf[h1 * HD + d0 + 2] = (o[2 * t + 1][1] - b1) * vref;
                obuf[h1 * HD + d0 + 3] = (o[2 * t + 1][3] - b1) * vref;
            }
        }
    }
};

// CUDA-core tile. Lane (r, c): c = lane % LPR picks a 16-byte chunk (8 dims)
// of a K/V row, r = lane / LPR a row group; the lane handles tokens r + RG*i.
// Partial dot products (TPL tokens x GP heads per lane) are summed over the
// LPR lanes of a row by a transposing butterfly that halves the values each
// lane carries at every step; afterwards lane c holds token r + RG*(c/2) for
// heads (c%2)*GP/2 .. +GP/2. Weights go through a per-warp smem exchange to
// the lanes that own each token's V chunk.
template <int HD, int GP>
struct FmaState {
    static constexpr int LPR = HD / 8;     // lanes per K/V row
    static constexpr int RG = 32 / LPR;    // row groups
    static constexpr int TPL = kBlock / RG;  // tokens per lane
    static constexpr int R = GP / 2;       // reduced values per lane
    static_assert(TPL * GP % LPR == 0 && TPL * GP / LPR == R, "layout");
    float q[GP][8];
    float o[GP][8];
    float m[R], l[R];

    __device__ __forceinline__ void begin_unit(const AttnParams& p, int b, int h, int lane) {
        const int c = lane % LPR;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            if (g < p.G) {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(
                    p.q + ((long long)b * p.Hq + (long long)h * p.G + g) * HD + c * 8));
                q[g][0] = bf16_lo(w.x); q[g][1] = bf16_hi(w.x);
                q[g][2] = bf16_lo(w.y); q[g][3] = bf16_hi(w.y);
                q[g][4] = bf16_lo(w.z); q[g][5] = bf16_hi(w.z);
                q[g][6] = bf16_lo(w.w); q[g][7] = bf16_hi(w.w);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) q[g][e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) o[g][e] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < R; ++k) { m[k] = kNegInf; l[k] = 0.f; }
    }

    __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int valid, float sl2, int lane,
                                          float* xp, int G) {
        const int c = lane % LPR, r = lane / LPR;
        float val[TPL * GP];
#pragma unroll
        for (int i = 0; i < TPL; ++i) {
            const int t = r + RG * i;
            uint32_t w0, w1, w2, w3;
            lds128(kt + swz<HD>(t, c), w0, w1, w2, w3);
            const float kf[8] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1),
                                 bf16_lo(w2), bf16_hi(w2), bf16_lo(w3), bf16_hi(w3)};
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(q[g][e], kf[e], acc);
                val[i * GP + g] = acc;
            }
        }
        // transposing butterfly over the LPR lanes of a row
#pragma unroll
        for (int msk = LPR / 2, n = TPL * GP; msk >= 1; msk >>= 1, n >>= 1) {
            const bool up = (lane & msk) != 0;
#pragma unroll
            for (int k = 0; k < n / 2; ++k) {
                const float lo = val[k], hi = val[k + n / 2];
                const float send = up ? lo : hi;
                const float keep = up ? hi : lo;
                val[k] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
            }
        }
        const int t = r + RG * (c >> 1);
        const int g0 = (c & 1) * R;
        float s[R], al[R];
#pragma unroll
        for (int k = 0; k < R; ++k) {
            s[k] = (t < valid && g0 + k < G) ? val[k] * sl2 : kNegInf;
            float mx = s[k];
#pragma unroll
            for (int sh = 2; sh < 32; sh <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
            const float mn = fmaxf(m[k], mx);
            const float ref = mn == kNegInf ? 0.f : mn;
            al[k] = exp2f(m[k] - ref);
            const float pk = exp2f(s[k] - ref);
            l[k] = l[k] * al[k] + pk;
            m[k] = mn;
            xp[t * GP + g0 + k] = pk;
        }
        if (lane < 2) {
#pragma unroll
            for (int k = 0; k < R; ++k) xp[kBlock * GP + g0 + k] = al[k];
        }
        __syncwarp();
        float alpha[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) alpha[g] = xp[kBlock * GP + g];
#pragma unroll
        for (int g = 0; g < GP; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) o[g][e] *= alpha[g];
#pragma unroll
        for (int i = 0; i < TPL; ++i) {
            const int tt = r + RG * i;
            if (tt < valid) {
                uint32_t w0, w1, w2, w3;
                lds128(vt + swz<HD>(tt, c), w0, w1, w2, w3);
                const float vf[8] = {bf16_lo(w0), bf16_hi(w0), bf16_lo(w1), bf16_hi(w1),
                                     bf16_lo(w2), bf16_hi(w2), bf16_lo(w3), bf16_hi(w3)};
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    const float pw = xp[tt * GP + g];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[g][e] = fmaf(pw, vf[e], o[g][e]);
                }
            }
        }
    }

    __device__ __forceinline__ void store(float* mbuf, float* lbuf, float* obuf, int G, int lane) {
        const int c = lane % LPR;
#pragma unroll
        for (int k = 0; k < R; ++k)
#pragma unroll
            for (int sh = 2; sh < 32; sh <<= 1) l[k] += __shfl_xor_sync(0xffffffffu, l[k], sh);
#pragma unroll
        for (int sh = LPR; sh < 32; sh <<= 1)
#pragma unroll
            for (int g = 0; g < GP; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) o[g][e] += __shfl_xor_sync(0xffffffffu, o[g][e], sh);
        if (lane < 2) {
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const int g = (lane & 1) * R + k;
                if (g < G) { mbuf[g] = m[k]; lbuf[g] = l[k]; }
            }
        }
        if (lane < LPR) {
#pragma unroll
            for (int g = 0; g < GP; ++g)
                if (g < G)
#pragma unroll
                    for (int e = 0; e < 8; ++e) obuf[g * HD + c * 8 + e] = o[g][e];
        }
    }
};



// ------------------------------------------------------ the main kernel ---

template <int HD, int VAR, int GP>
struct StateOf;
template <int HD, int GP>
struct StateOf<HD, kVarMma, GP> { using T = MmaState<HD>; };
template <int HD, int GP>
struct StateOf<HD, kVarFma, GP> { using T = FmaState<HD, GP>; };
template <int HD, int GP>
struct StateOf<HD, kVarFp8, GP> { using T = Fp8State<HD>; };
template <int HD, int GP>
struct StateOf<HD, kVarInt8, GP> { using T = Int8State<HD>; };

// A bounded wait by every lane of a warp; true when all of them saw the phase.
__device__ __forceinline__ bool wait_all_warp(uint32_t bar, uint32_t parity, long long limit_ns,
                                              uint32_t sleep_ns) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, limit_ns, sleep_ns));
}

__device__ __forceinline__ void consumer_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// W consumer warps (compute, merge) and one producer warp (block-table walk
// and TMA issue in lanes 0..W-1, zero rows for empty requests in the rest).
// Consumers synchronise among themselves on named barrier 1. The e4m3 tile
// runs three CTAs per SM (its per-block conversions make it latency-bound,
// so more resident warps pay; its tiles are half the size, so the stages
// still fit), the others two.
// FUSED (MMA tile only): the decode step of mi_paged_decode_step. An extra
// RoPE warp walks the CTA's units in the consumers' order and, ahead of them,
// fills a two-slot ring with each unit's rotated q rows and the new token's
// rotated k row and v row; when the block holding the new token is in this
// CTA's range it also writes that row of the cache and the unit's q_out. The
// consumer warp that streams that block copies the two rows into its staged
// tiles.
template <int HD, int VAR, int GP, int W, bool FUSED = false>
__global__ void __launch_bounds__((W + (FUSED ? 2 : 1)) * 32, (VAR == kVarFp8 || VAR == kVarInt8) && !FUSED ? 3 : 2)
    attn_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                const AttnParams p) {
    // e4m3 (and INT8) waits sleep between polls (the hint of
    // mbarrier.try_wait), bf16 ones poll: 2.415 against 2.440 ms per e4m3
    // step, 4.02 against 3.98 ms per bf16 step
    constexpr bool kOneByte = VAR == kVarFp8 || VAR == kVarInt8;
    constexpr uint32_t kSleep = kOneByte ? kWaitSleepNs : 0u;
    static_assert(!FUSED || VAR == kVarMma || VAR == kVarFp8, "the fused step runs the MMA or e4m3 tile");
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.stages;
    const SmemPlan sp = smem_plan(W, S, HD, p.G, VAR == kVarFma, elem_bytes(VAR), FUSED, VAR == kVarInt8);
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t* base = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    long long* scan = reinterpret_cast<long long*>(base + sp.scan);
    constexpr int kTile = Tile<HD, elem_bytes(VAR)>::kBytes;
    const uint32_t full0 = sbase + sp.full, empty0 = sbase + sp.empty;

    if (tid < W * S) {
        mbar_init(full0 + tid * 8, 1);
        mbar_init(empty0 + tid * 8, 1);
    }
    const uint32_t qfull0 = sbase + sp.qbar, qempty0 = qfull0 + 16, kvfull0 = qfull0 + 32;  // fused step: ring
    if (FUSED && tid < 2) {
        mbar_init(qfull0 + tid * 8, 1);
        mbar_init(qempty0 + tid * 8, W);
        mbar_init(kvfull0 + tid * 8, 1);
    }
    fence_mbar_init();
    // Inputs may come from the kernel just before this one in the stream:
    // what it wrote is visible only past pdl_wait. An early-start fused step
    // (the caller promises that kernel writes none of the lengths, the block
    // tables, the caches, the error word or this call's workspace) plans
    // and issues each producer lane's first S copies before its wait. Every
    // thread lets the next launch start only after its own wait has
    // returned, so that launch never runs beside the one before this.
    const bool early = FUSED && p.early != 0;
    if (!early) {
        pdl_wait();
        pdl_trigger();
    }
    // Warm L2 with this CTA's share of the block tables and of q (and, for
    // the fused step, of the new token's k and v rows): the lookups and loads
    // that follow the plan then hit L2 instead of going to DRAM.
    if (warp == W) {
        prefetch_share(p.block_tables, (long long)p.B * p.mbps * 4, lane);
        prefetch_share(p.q, (long long)p.B * p.Hq * HD * 2, lane);
        if (FUSED) {
            prefetch_share(p.knew, (long long)p.B * p.Hkv * HD * 2, lane);
            prefetch_share(p.vnew, (long long)p.B * p.Hkv * HD * 2, lane);
        }
    }

    // Ranges are cut by cost: a unit weighs its blocks plus a fixed number of
    // blocks for its per-unit work (q, the merge, the pipeline restart at its
    // boundary), which weighs more against the half-size one-byte blocks.
    constexpr int uc = kOneByte ? kUnitCostE4m3 : kUnitCostBf16;
    const int cta = blockIdx.x;
    RangePlan* rp = reinterpret_cast<RangePlan*>(base + sp.rplan);
    long long TB = 0, TC = 0;
    int P = 0;
    // this CTA's plan from an earlier launch with the same lengths, if any
    PlanEntry* pe = p.plan_cache ? reinterpret_cast<PlanEntry*>(p.plan_cache + (long long)cta * p.plan_stride)
                                 : nullptr;
    const int32_t key[8] = {kPlanMagic, p.plan_kind, p.B, p.Hkv, p.mbps, (int32_t)gridDim.x, uc, cta};
    bool hit = false;
    if (pe) {
        bool same = true;
        if (tid < 8) same = __ldcg(pe->key + tid) == key[tid];
        const int32_t* lens = reinterpret_cast<const int32_t*>(pe + 1);
        for (int b = tid; b < p.B; b += blockDim.x) same &= __ldcg(lens + b) == __ldg(p.context_lens + b);
        hit = __syncthreads_and(same) != 0;
    }
    if (hit) {
        if (tid == 0) {
            scan[0] = __ldcg(&pe->TB);
            scan[1] = __ldcg(&pe->TC);
            scan[2] = __ldcg(&pe->P);
            scan[3] = (long long)__ldcg(&pe->sum);
        }
        const int nw = (int)(sizeof(RangePlan) / 4);
        for (int i = tid; i < nw; i += blockDim.x)
            reinterpret_cast<int32_t*>(rp)[i] = __ldcg(reinterpret_cast<const int32_t*>(&pe->rp) + i);
        __syncthreads();
        TB = scan[0];
        TC = scan[1];
        P = (int)scan[2];
        if (warp == 0) {
            const uint32_t h = plan_sum(P, TB, TC, rp, lane);
            if (lane == 0) scan[4] = h == (uint32_t)scan[3] ? 1 : 0;
        }
        __syncthreads();
        hit = scan[4] != 0;  // a damaged entry: the plan is computed below
    }
    if (!hit) {
        TB = plan_scan(p, uc, scan, TC);  // (ends with a barrier of all warps)
        // CTAs that take part: the whole grid, unless that leaves fewer than
        // kMinBlocksPerCta blocks each (a small batch): every CTA's fixed cost
        // (the plan, the first copies, a merge) then outweighs its share of
        // streaming, and fewer, longer ranges finish sooner.
        const long long Pw = (TB + kMinBlocksPerCta - 1) / kMinBlocksPerCta;
        P = (int)(Pw < (long long)gridDim.x ? Pw : (long long)gridDim.x);
        plan_ranges(p, uc, scan, TB, TC, P, rp);  // (ends with a barrier of all warps)
        if (pe) {
            // the plan first, the lengths, then the key: an entry is
            // complete when its key matches
            int32_t* lens = reinterpret_cast<int32_t*>(pe + 1);
            for (int b = tid; b < p.B; b += blockDim.x) lens[b] = __ldg(p.context_lens + b);
            const int nw = (int)(sizeof(RangePlan) / 4);
            for (int i = tid; i < nw; i += blockDim.x)
                reinterpret_cast<int32_t*>(&pe->rp)[i] = reinterpret_cast<const int32_t*>(rp)[i];
            if (warp == 0) {
                const uint32_t h = plan_sum(P, TB, TC, rp, lane);
                if (lane == 0) {
                    pe->TB = TB;
                    pe->TC = TC;
                    pe->P = P;
                    pe->sum = h;
                    for (int i = 0; i < 8; ++i) pe->key[i] = key[i];
                }
            }
        }
    }
    const long long ra = rp->ra, rb = rp->rb, sl = rp->sl;
    if (early && !(warp == W && lane < W)) {
        pdl_wait();
        pdl_trigger();
    }

    if (FUSED && warp == W + 1) {
        // --------------------------------------------------- RoPE warp --
        // the consumers' unit order: part 0 = [sl, rb), then part 1 = [ra, sl)
        if (cta >= P) return;
        uint16_t* ring = reinterpret_cast<uint16_t*>(base + sp.qring);
        constexpr int kQW = kMaxG * HD / 4 / 32;   // q words per lane and half row, at most (one per head at d 128)
        constexpr int kVW = HD / 64;               // v words per lane
        const int kc = 2 * (lane % (HD / 4));      // this lane's column pair, the same in every head
        const bool klane = lane < HD / 4;          // lanes that rotate the new k (kc = 2 * lane there)
        int u = 0;
        bool good = true;
        for (int part = 0; good && part < 2; ++part) {
            const long long ps = part == 0 ? sl : ra, pe = part == 0 ? rb : sl;
            if (ps >= pe) continue;
            Cursor cu = part == 0 ? rp->c0 : rp->c1;
            for (; good && cu.start < pe && cu.b < p.B; cu.next(p), ++u) {
                const int slot = u & 1;
                int pos = ctx_clamped(p, cu.b) - 1;
                if (pos >= p.max_pos) pos = -1;
                // Every load of the unit is issued at once, ahead of the wait
                // for its slot: q (this lane's column pair in each head), the
                // new k and v rows and one cos/sin vector that serves both.
                uint32_t xl[kQW] = {}, xh[kQW] = {}, vv[kVW] = {}, kl = 0u, kh = 0u;
                float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (pos >= 0) {
                    c4 = __ldg(reinterpret_cast<const float4*>(p.rope + (long long)pos * (HD / 2) + kc));
                    const uint16_t* q0 = p.qraw + ((long long)cu.b * p.Hq + (long long)cu.h * p.G) * HD + kc;
#pragma unroll
                    for (int i = 0; i < kQW; ++i) {
                        const int w = lane + 32 * i;
                        if (w < p.G * HD / 4) {
                            const uint16_t* qr = q0 + (w / (HD / 4)) * HD;
                            xl[i] = __ldg(reinterpret_cast<const uint32_t*>(qr));
                            xh[i] = __ldg(reinterpret_cast<const uint32_t*>(qr + HD / 2));
                        }
                    }
                    const long long nofs = ((long long)cu.b * p.Hkv + cu.h) * HD;
                    if (klane) {
                        kl = __ldg(reinterpret_cast<const uint32_t*>(p.knew + nofs + kc));
                        kh = __ldg(reinterpret_cast<const uint32_t*>(p.knew + nofs + kc + HD / 2));
                    }
#pragma unroll
                    for (int j = 0; j < kVW; ++j)
                        vv[j] = __ldg(reinterpret_cast<const uint32_t*>(p.vnew + nofs + 2 * lane + 64 * j));
                }
                if (!wait_all_warp(qempty0 + slot * 8, (uint32_t)(((u >> 1) & 1) ^ 1), p.wait_ns, kSleep)) {
                    if (lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
                    good = false;
                    break;
                }
                uint16_t* qrows = ring + slot * (p.G + 2) * HD;
                uint16_t* krow = qrows + p.G * HD;
                uint16_t* vrow = krow + HD;
                unsigned need = 0;  // q words whose values need the exact route
#pragma unroll
                for (int i = 0; i < kQW; ++i) {
                    const int w = lane + 32 * i;
                    if (w < p.G * HD / 4) {
                        uint32_t yl = 0u, yh = 0u;
                        if (pos >= 0) need |= (unsigned)rotate_word_fast(xl[i], xh[i], c4, yl, yh) << i;
                        uint16_t* qd = qrows + (w / (HD / 4)) * HD + kc;
                        *reinterpret_cast<uint32_t*>(qd) = yl;
                        *reinterpret_cast<uint32_t*>(qd + HD / 2) = yh;
                    }
                }
                if (need) {
                    // rare: those words again by the exact route (the raw q
                    // is never written by this kernel, so it is re-read)
#pragma unroll 1
                    for (int i = 0; i < kQW; ++i) {
                        if (!((need >> i) & 1u)) continue;
                        const int row = (lane + 32 * i) / (HD / 4);
                        const uint16_t* qr =
                            p.qraw + ((long long)cu.b * p.Hq + (long long)cu.h * p.G + row) * HD + kc;
                        const uint2 y = rotate_word_exact(__ldg(reinterpret_cast<const uint32_t*>(qr)),
                                                          __ldg(reinterpret_cast<const uint32_t*>(qr + HD / 2)), c4);
                        uint16_t* qd = qrows + row * HD + kc;
                        *reinterpret_cast<uint32_t*>(qd) = y.x;
                        *reinterpret_cast<uint32_t*>(qd + HD / 2) = y.y;
                    }
                }
                // q first: the consumers need it where the unit starts, the
                // new token's rows only at its last block
                __syncwarp();
                if (lane == 0) mbar_arrive(qfull0 + slot * 8);
                // e4m3 caches: the rows are stored quantised with the head's
                // scales, as the FP8 append stores them; a row whose scale is
                // not a positive finite number is not written (a flag word in
                // the slot tells the consumers which rows to place)
                bool k_ok = true, v_ok = true;
                float ks = 1.f, vs = 1.f;
                if constexpr (VAR == kVarFp8) {
                    ks = __ldg(p.k_scale + cu.h);
                    vs = __ldg(p.v_scale + cu.h);
                    k_ok = fp8_scale_ok(ks);
                    v_ok = fp8_scale_ok(vs);
                    if (pos >= 0 && !(k_ok && v_ok) && lane == 0) raise_err(p.dev_err, MI_DEVERR_BAD_SCALE);
                }
                if (pos >= 0) {
                    if (klane) {
                        uint32_t yl, yh;
                        if (rotate_word_fast(kl, kh, c4, yl, yh)) {  // rare: the exact route
                            const uint2 y = rotate_word_exact(kl, kh, c4);
                            yl = y.x;
                            yh = y.y;
                        }
                        if constexpr (VAR == kVarFp8) {
                            uint8_t* k8 = reinterpret_cast<uint8_t*>(krow);
                            *reinterpret_cast<uint16_t*>(k8 + kc) =
                                (uint16_t)f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(yl), ks), __fdiv_rn(bf16_hi(yl), ks));
                            *reinterpret_cast<uint16_t*>(k8 + kc + HD / 2) =
                                (uint16_t)f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(yh), ks), __fdiv_rn(bf16_hi(yh), ks));
                        } else {
                            *reinterpret_cast<uint32_t*>(krow + kc) = yl;
                            *reinterpret_cast<uint32_t*>(krow + kc + HD / 2) = yh;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < kVW; ++j) {
                        if constexpr (VAR == kVarFp8) {
                            *reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(vrow) + 2 * lane + 64 * j) =
                                (uint16_t)f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(vv[j]), vs), __fdiv_rn(bf16_hi(vv[j]), vs));
                        } else {
                            *reinterpret_cast<uint32_t*>(vrow + 2 * lane + 64 * j) = vv[j];
                        }
                    }
                }
                if (VAR == kVarFp8 && lane == 0)
                    *reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(krow) + HD) = (k_ok ? 1u : 0u) | (v_ok ? 2u : 0u);
                __syncwarp();
                if (lane == 0) mbar_arrive(kvfull0 + slot * 8);
                if (pos >= 0) {
                    // the block holding the new token is streamed here: this
                    // CTA writes the cache row and the unit's q_out
                    const int jnew = pos / kBlock;
                    const long long jx = cu.start + jnew;
                    if (jx >= ra && jx < rb) {
                        const int blk = __ldg(p.block_tables + (long long)cu.b * p.mbps + jnew);
                        if (blk >= 0 && blk < p.num_blocks) {
                            const long long rofs = (((long long)blk * p.Hkv + cu.h) * kBlock + pos % kBlock) * HD;
                            if constexpr (VAR == kVarFp8) {
                                uint8_t* kc8 = reinterpret_cast<uint8_t*>(p.kc);
                                uint8_t* vc8 = reinterpret_cast<uint8_t*>(p.vc);
                                for (int k = 4 * lane; k < HD; k += 128) {
                                    if (k_ok)
                                        *reinterpret_cast<uint32_t*>(kc8 + rofs + k) =
                                            *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(krow) + k);
                                    if (v_ok)
                                        *reinterpret_cast<uint32_t*>(vc8 + rofs + k) =
                                            *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(vrow) + k);
                                }
                            } else {
                                for (int k = 2 * lane; k < HD; k += 64) {
                                    *reinterpret_cast<uint32_t*>(p.kc + rofs + k) = *reinterpret_cast<const uint32_t*>(krow + k);
                                    *reinterpret_cast<uint32_t*>(p.vc + rofs + k) = *reinterpret_cast<const uint32_t*>(vrow + k);
                                }
                            }
                        }
                        uint16_t* qo = p.q_out + ((long long)cu.b * p.Hq + (long long)cu.h * p.G) * HD;
                        for (int w = lane; w < p.G * HD / 2; w += 32)
                            reinterpret_cast<uint32_t*>(qo)[w] = reinterpret_cast<const uint32_t*>(qrows)[w];
                    }
                }
            }
        }
        return;
    }

    if (warp == W) {
        // ------------------------------------------------ producer warp --
        if (lane >= W) {
            // Rows of requests with no tokens are zero; CTA i owns b = i mod
            // gridDim (these rows belong to no unit, so nobody else writes them).
            const int nl = 32 - W;
            for (int b = cta; b < p.B; b += gridDim.x) {
                const int n = __ldg(p.context_lens + b);
                if (n > p.mbps * kBlock && lane == W) raise_err(p.dev_err, MI_DEVERR_BAD_CONTEXT);
                if (n <= 0) {
                    uint4* row = reinterpret_cast<uint4*>(p.out + (long long)b * p.Hq * HD);
                    for (int i = lane - W; i < p.Hq * HD / 8; i += nl) row[i] = make_uint4(0, 0, 0, 0);
                }
            }
            return;
        }
        // Lane w < W feeds consumer warp w: blocks ps + w, ps + w + W, ... of
        // each part [ps, pe) of this CTA's range. For each it waits for a free
        // stage of the warp's ring, looks the block up in the table and issues
        // the two copies.
        const uint64_t policy = l2_policy_evict_first();
        uint32_t stg = 0, ph = 1;  // a fresh barrier reads as having completed the phase before 0
        // failure-detection test: in every CTA, lane 0 neither copies nor
        // arrives for its first block, so consumer warp 0's wait on that
        // stage runs out (some CTAs may have no blocks at all)
        bool withhold = p.withhold != 0 && lane == 0;
        bool waited = !early;  // early start: this lane waits once its first S copies are issued
        int issued = 0;
        const uint32_t my_full = full0 + (uint32_t)(lane * S) * 8, my_empty = empty0 + (uint32_t)(lane * S) * 8;
        const uint32_t my_tiles = sbase + sp.tiles + (uint32_t)(lane * S) * (2 * kTile);
        for (int part = 0; part < 2; ++part) {
        const long long ps = part == 0 ? sl : ra, pe = part == 0 ? rb : sl;
        long long x = ps + lane;
        if (x >= pe) continue;
        Cursor cu = part == 0 ? rp->c0 : rp->c1;  // advanced to each block below
        // INT8 tiles: each block's table entry and group maxima are read one
        // block ahead, before the wait for its stage, so that the loads of
        // the maxima (which need the block id) stay off the issue path
        int nblk = 0, nh = 0;
        float nak = 0.f, nav = 0.f;
        if constexpr (VAR == kVarInt8) {
            cu.advance_to(p, x);
            nblk = __ldg(p.block_tables + (long long)cu.b * p.mbps + (x - cu.start));
            nh = cu.h;
            if (nblk >= 0 && nblk < p.num_blocks) {
                nak = __ldg(p.k_amax + (long long)nblk * p.Hkv + nh);
                nav = __ldg(p.v_amax + (long long)nblk * p.Hkv + nh);
            }
        }
        for (; x < pe; x += W) {
            int blk = 0, hh = 0;
            float ak = 0.f, av = 0.f;
            if constexpr (VAR == kVarInt8) {
                blk = nblk;
                hh = nh;
                ak = nak;
                av = nav;
                if (x + W < pe) {
                    cu.advance_to(p, x + W);
                    nblk = __ldg(p.block_tables + (long long)cu.b * p.mbps + (x + W - cu.start));
                    nh = cu.h;
                    if (nblk >= 0 && nblk < p.num_blocks) {
                        nak = __ldg(p.k_amax + (long long)nblk * p.Hkv + nh);
                        nav = __ldg(p.v_amax + (long long)nblk * p.Hkv + nh);
                    }
                }
            }
            if (!waited && issued == S) {
                pdl_wait();
                pdl_trigger();
                waited = true;
            }
            ++issued;
            if (!mbar_wait_bounded(my_empty + stg * 8, ph, p.wait_ns, kSleep)) {
                // the consumer stopped taking stages (it timed out itself)
                raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
                return;
            }
            if constexpr (VAR != kVarInt8) {
                cu.advance_to(p, x);
                blk = __ldg(p.block_tables + (long long)cu.b * p.mbps + (x - cu.start));
                hh = cu.h;
            }
            const uint32_t bar = my_full + stg * 8;
            const uint32_t okf = sbase + sp.okf + ((uint32_t)(lane * S) + stg) * 4;
            if (withhold) {
                withhold = false;  // nothing is copied into this stage and nothing arrives on it
            } else if (blk < 0 || blk >= p.num_blocks) {
                raise_err(p.dev_err, MI_DEVERR_BAD_BLOCK);
                sts32(okf, 0u);
                mbar_arrive(bar);  // the consumer skips the block
            } else {
                const uint32_t dst = my_tiles + stg * (2 * kTile);
                const int e = blk * p.Hkv + hh;
                const int y = e * (kTile / 128);  // the tile's first 128-byte line
                if constexpr (VAR == kVarInt8) {
                    // the tiles, then the block's K and V group maxima (read
                    // a block ahead; two more bulk copies per stage cost ~5
                    // us per Qwen3-8B layer) into the stage's slot; the
                    // arrive comes after them, so its release publishes them
                    // with the flag
                    const uint32_t am = sbase + sp.amx + ((uint32_t)(lane * S) + stg) * 8;
                    mbar_expect_tx(bar, 2 * kTile);
                    tma_load_2d(dst, &tmk, bar, 0, y, policy);
                    tma_load_2d(dst + kTile, &tmv, bar, 0, y, policy);
                    sts32(am, __float_as_uint(ak));
                    sts32(am + 4, __float_as_uint(av));
                    sts32(okf, 1u);
                    mbar_arrive(bar);
                } else {
                    sts32(okf, 1u);
                    mbar_arrive_expect_tx(bar, 2 * kTile);
                    tma_load_2d(dst, &tmk, bar, 0, y, policy);
                    tma_load_2d(dst + kTile, &tmv, bar, 0, y, policy);
                }
            }
            if (++stg == (uint32_t)S) {
                stg = 0;
                ph ^= 1u;
            }
        }
        }
        if (!waited) {
            pdl_wait();
            pdl_trigger();
        }
        return;
    }

    // ---------------------------------------------------- consumer warps --
    if (cta >= P) return;
    float* mbuf = reinterpret_cast<float*>(base + sp.mbuf);
    float* lbuf = reinterpret_cast<float*>(base + sp.lbuf);
    float* obuf = reinterpret_cast<float*>(base + sp.obuf);
    float* xbuf = reinterpret_cast<float*>(base + sp.xbuf) + warp * (kBlock * kMaxG + kMaxG);
    const int nc = W * 32;
    using State = typename StateOf<HD, VAR, GP>::T;
    State st;
    int unit_no = 0;  // fused step: units begun so far (q ring slot and phase)
    const uint16_t* qslot = nullptr;  // fused step: this unit's ring slot
    bool dead = false;  // a wait timed out: stop touching the pipeline
    uint32_t cstage = 0, cphase = 0;

    for (int part = 0; part < 2; ++part) {
    const long long ps = part == 0 ? sl : ra, pe = part == 0 ? rb : sl;
    if (ps >= pe) continue;
    Cursor cu = part == 0 ? rp->c0 : rp->c1;
    while (cu.start < pe && cu.b < p.B) {
        const long long sa = cu.start > ps ? cu.start : ps;
        const long long se = (cu.start + cu.len) < pe ? (cu.start + cu.len) : pe;
        const int nvalid = ctx_clamped(p, cu.b);
        // fused step: the new token sits at position nvalid - 1, in block jnew
        int pos = -1, jnew = -1;
        if constexpr (FUSED) {
            pos = nvalid - 1;
            jnew = pos / kBlock;
            if (pos >= p.max_pos) {
                if (lane == 0 && warp == 0) raise_err(p.dev_err, MI_DEVERR_BAD_POS);
                pos = -1;
                jnew = -1;
            }
            // this unit's rotated q from the RoPE warp's ring
            const int slot = unit_no & 1;
            if (!dead && !wait_all_warp(qfull0 + slot * 8, (uint32_t)((unit_no >> 1) & 1), p.wait_ns, kSleep)) {
                dead = true;
                if (lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
            }
            qslot = reinterpret_cast<const uint16_t*>(base + sp.qring) + slot * (p.G + 2) * HD;
            st.begin_unit_from(qslot, p, cu.h, lane);
        } else {
            st.begin_unit(p, cu.b, cu.h, lane);
        }
        long long x = sa + (((warp - (sa - ps)) % W) + W) % W;
        for (; x < se; x += W) {
            const uint32_t si = (uint32_t)(warp * S) + cstage;
            if (!dead) {
                const bool okw = mbar_wait_bounded(full0 + si * 8, cphase, p.wait_ns, kSleep);
                if (__any_sync(0xffffffffu, !okw)) {
                    dead = true;
                    if (lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
                }
            }
            const int j = (int)(x - cu.start);
            const int valid = min(kBlock, nvalid - j * kBlock);
            // the producer's flag (published by its arrive) says whether the block was copied
            const uint32_t okv = dead ? 0u : lds32(sbase + sp.okf + si * 4);
            if (okv != 0u) {
                const uint32_t kt = sbase + sp.tiles + si * (2 * kTile), vt = kt + kTile;
                // rows past the context may hold any bits: zero V there (they
                // meet zero weights, which clear every finite value; INT8
                // codes always are)
                if (VAR != kVarFma && VAR != kVarInt8 && valid < kBlock) {
                    constexpr int kChunks = HD * elem_bytes(VAR) / 16;  // 16-byte chunks per token row
                    for (int i = lane; i < (kBlock - valid) * kChunks; i += 32) {
                        const int row = valid + i / kChunks, ch = i % kChunks;
                        st_shared_zero16(vt + (VAR == kVarFp8 ? swz8<HD>(row, ch) : swz<HD>(row, ch)));
                    }
                    __syncwarp();
                }
                if constexpr (FUSED) {
                    if (j == jnew) {
                        // the new token: its rotated k and its v (from the
                        // RoPE warp's ring slot) into row valid - 1 of the tiles
                        const int row = valid - 1;
                        if (!wait_all_warp(kvfull0 + (unit_no & 1) * 8, (uint32_t)((unit_no >> 1) & 1), p.wait_ns, kSleep)) {
                            dead = true;
                            if (lane == 0) raise_err(p.dev_err, MI_DEVERR_TIMEOUT);
                        }
                        const uint16_t* krow = qslot + p.G * HD;
                        const uint16_t* vrow = krow + HD;
                        if constexpr (VAR == kVarFp8) {
                            const uint8_t* k8 = reinterpret_cast<const uint8_t*>(krow);
                            const uint8_t* v8 = reinterpret_cast<const uint8_t*>(vrow);
                            const uint32_t which = *reinterpret_cast<const uint32_t*>(k8 + HD);
                            for (int i = 4 * lane; i < HD; i += 128) {
                                if (which & 1u)
                                    sts32(kt + swz8<HD>(row, i >> 4) + (i & 15), *reinterpret_cast<const uint32_t*>(k8 + i));
                                if (which & 2u)
                                    sts32(vt + swz8<HD>(row, i >> 4) + (i & 15), *reinterpret_cast<const uint32_t*>(v8 + i));
                            }
                        } else {
                            for (int i = 2 * lane; i < HD; i += 64) {
                                sts32(kt + swz<HD>(row, i >> 3) + (i & 7) * 2, *reinterpret_cast<const uint32_t*>(krow + i));
                                sts32(vt + swz<HD>(row, i >> 3) + (i & 7) * 2, *reinterpret_cast<const uint32_t*>(vrow + i));
                            }
                        }
                        __syncwarp();
                    }
                }
                if constexpr (VAR == kVarInt8) {
                    // the block's K and V group maxima, staged with the tiles
                    const uint32_t am = sbase + sp.amx + si * 8;
                    st.block(kt, vt, valid, lane, __uint_as_float(lds32(am)), __uint_as_float(lds32(am + 4)));
                } else if constexpr (VAR != kVarFma) {
                    st.block(kt, vt, valid, p.sl2, lane);
                } else {
                    st.block(kt, vt, valid, p.sl2, lane, xbuf, p.G);
                }
            }
            __syncwarp();
            if (lane == 0 && !dead) {
                // this warp's reads of the stage are done: hand it back
                fence_proxy_async_smem();
                mbar_arrive(empty0 + si * 8);
            }
            if (++cstage == (uint32_t)S) {
                cstage = 0;
                cphase ^= 1u;
            }
        }
        if constexpr (FUSED) {
            // this warp is done with the unit's ring slot
            __syncwarp();
            if (lane == 0 && !dead) mbar_arrive(qempty0 + (unit_no & 1) * 8);
            ++unit_no;
        }
        // merge the warps' states for this unit (a warp without a block in
        // it stores its initial state: max -inf, sum 0, output 0)
        st.store(mbuf + warp * kMaxG, lbuf + warp * kMaxG, obuf + warp * p.G * HD, p.G, lane);
        consumer_sync(nc);
        const bool whole = (sa == cu.start) && (se == cu.start + cu.len);
        const int slot = (sa == ra) ? 0 : 1;
        float* part = p.part + ((long long)cta * 2 + slot) * p.slot_floats;
        // four consecutive outputs per thread (16-byte shared and global
        // accesses); each thread weighs the warps' states of its head itself
        for (int idx = 4 * tid; idx < p.G * HD; idx += 4 * nc) {
            const int g = idx / HD, dcol = idx - g * HD;
            float M = kNegInf;
            for (int w = 0; w < W; ++w) M = fmaxf(M, mbuf[w * kMaxG + g]);
            float fw[W];
            float L = 0.f;
            for (int w = 0; w < W; ++w) {
                fw[w] = (M == kNegInf) ? 0.f : exp2f(mbuf[w * kMaxG + g] - M);
                L += fw[w] * lbuf[w * kMaxG + g];
            }
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w = 0; w < W; ++w) {
                const float f = fw[w];
                if (f != 0.f) {
                    const float4 o = *reinterpret_cast<const float4*>(obuf + (w * p.G + g) * HD + dcol);
                    acc.x += f * o.x;
                    acc.y += f * o.y;
                    acc.z += f * o.z;
                    acc.w += f * o.w;
                }
            }
            const float r = L > 0.f ? 1.f / L : 0.f;
            const float4 v = make_float4(acc.x * r, acc.y * r, acc.z * r, acc.w * r);
            if (whole) {
                *reinterpret_cast<uint2*>(p.out + ((long long)cu.b * p.Hq + (long long)cu.h * p.G + g) * HD + dcol) =
                    make_uint2((uint32_t)f32_to_bf16(v.x) | ((uint32_t)f32_to_bf16(v.y) << 16),
                               (uint32_t)f32_to_bf16(v.z) | ((uint32_t)f32_to_bf16(v.w) << 16));
            } else {
                *reinterpret_cast<float4*>(part + idx) = v;
                if (dcol == 0) part[p.G * HD + g] = L > 0.f ? M + log2f(L) : kNegInf;
            }
        }
        if (!whole) {
            // pieces of this unit: CTAs cf..cl, found by cost position (the
            // unit's first block sits at cstart + uc, its last at cstart + uc
            // + len - 1); the first piece's slot is 1 when the unit starts
            // inside that CTA's range, every other piece is slot 0
            const long long c0 = cu.cstart + uc;
            const int cf = cta_of(TC, P, c0), cl = cta_of(TC, P, c0 + cu.len - 1);
            const int fs = (range_start(TC, P, cf) >= cu.cstart) ? 0 : 1;
            const int ns = cl - cf + 1;
            volatile int* mflag = reinterpret_cast<volatile int*>(base + sp.flag);
            consumer_sync(nc);  // this CTA's partial is stored
            if (tid == 0) {
                // one counter word per cut unit, at its first piece's CTA:
                // high 48 bits = the call's epoch, low 16 = pieces stored. A
                // word from another call counts as zero, so the buffer needs
                // no clearing. acq_rel: this CTA's partial is published
                // before the count, the others' partials are visible after it.
                unsigned long long* wd = p.unit_word + cf;
                const unsigned long long e48 = p.epoch & 0xFFFFFFFFFFFFull;
                unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(wd), nw, got;
                for (;;) {
                    nw = ((old >> 16) == e48) ? old + 1 : ((e48 << 16) | 1ull);
                    asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;"
                                 : "=l"(got) : "l"(wd), "l"(old), "l"(nw) : "memory");
                    if (got == old) break;
                    old = got;
                }
                const bool last = (int)(nw & 0xFFFFull) == ns;
                // The last piece hands the word back as zero (epochs are
                // never zero), so a replay of the same launch (a captured
                // graph keeps its epoch) starts every count afresh.
                if (last) *reinterpret_cast<volatile unsigned long long*>(wd) = 0ull;
                *mflag = last;
            }
            consumer_sync(nc);
            if (*mflag) {
                auto slot_of = [&](int c) {
                    return p.part + ((long long)c * 2 + (c == cf ? fs : 0)) * p.slot_floats;
                };
                // each thread weighs the pieces for its head itself: M = max
                // lse, out = sum 2^(lse-M) o / sum 2^(lse-M), pieces in order
                for (int idx = 4 * tid; idx < p.G * HD; idx += 4 * nc) {
                    const int g = idx / HD;
                    float M = kNegInf;
                    for (int c = cf; c <= cl; ++c) M = fmaxf(M, __ldcg(slot_of(c) + p.G * HD + g));
                    float den = 0.f;
                    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (M != kNegInf) {
#pragma unroll 4
                        for (int c = cf; c <= cl; ++c) {
                            const float wg = exp2f(__ldcg(slot_of(c) + p.G * HD + g) - M);
                            const float4 x = __ldcg(reinterpret_cast<const float4*>(slot_of(c) + idx));
                            den += wg;
                            num.x += wg * x.x;
                            num.y += wg * x.y;
                            num.z += wg * x.z;
                            num.w += wg * x.w;
                        }
                    }
                    const float r = den > 0.f ? 1.f / den : 0.f;
                    *reinterpret_cast<uint2*>(p.out + ((long long)cu.b * p.Hq + (long long)cu.h * p.G + g) * HD +
                                              (idx - g * HD)) =
                        make_uint2((uint32_t)f32_to_bf16(num.x * r) | ((uint32_t)f32_to_bf16(num.y * r) << 16),
                                   (uint32_t)f32_to_bf16(num.z * r) | ((uint32_t)f32_to_bf16(num.w * r) << 16));
                }
            }
        }
        consumer_sync(nc);
        cu.next(p);
    }
    }
    // After a timed-out wait, let the copies still in flight for this warp's
    // stages land (each wait bounded again) before shared memory goes away.
    if (dead && lane == 0) {
        for (int s2 = 0; s2 < S; ++s2) {
            const uint32_t si = (uint32_t)(warp * S) + (uint32_t)s2;
            (void)mbar_wait_bounded(full0 + si * 8, s2 < (int)cstage ? cphase ^ 1u : cphase, drain_limit(p.wait_ns));
        }
    }
}

// ------------------------------------------------------------- host side --

constexpr int kWarps = 4;                 // consumer warps; one producer warp more
constexpr int kMaxStages = 3;             // bf16 tiles; e4m3 tiles take twice as many
constexpr int kSmemLimit = 227 * 1024;    // per CTA
constexpr int kSmemTwoPerSm = 115712;     // per CTA so that two fit in an SM's 228 KB
constexpr int kSmemThreePerSm = 76800;    // per CTA so that three fit

// Stages per consumer warp: as many as fit with two CTAs per SM, else (very
// wide GQA groups) as many as fit one CTA. One-byte (e4m3, INT8) tiles are
// half the size, so they take up to twice the stages, and first try for
// three CTAs per SM with at least two stages each.
int pick_stages(int HD, int G, int var, bool fused = false) {
    const bool fma = var == kVarFma, amx = var == kVarInt8;
    const int eb = elem_bytes(var), top = kMaxStages * 2 / eb;
    if ((var == kVarFp8 || var == kVarInt8) && !fused)
        for (int S = top; S >= 2; --S)
            if (smem_plan(kWarps, S, HD, G, fma, eb, fused, amx).total <= kSmemThreePerSm) return S;
    for (int S = top; S >= 1; --S)
        if (smem_plan(kWarps, S, HD, G, fma, eb, fused, amx).total <= kSmemTwoPerSm) return S;
    for (int S = top; S >= 1; --S)
        if (smem_plan(kWarps, S, HD, G, fma, eb, fused, amx).total <= kSmemLimit) return S;
    return 0;
}

int smem_of(int HD, int G, int var, bool fused = false) {
    return smem_plan(kWarps, pick_stages(HD, G, var, fused), HD, G, var == kVarFma, elem_bytes(var), fused,
                     var == kVarInt8)
        .total;
}

int gp_of(int G) { return G <= 2 ? 2 : (G <= 4 ? 4 : 8); }

using KernelFn = void (*)(CUtensorMap, CUtensorMap, AttnParams);

template <int HD>
KernelFn fma_kernel_for(int GP) {
    switch (GP) {
        case 2: return attn_kernel<HD, kVarFma, 2, kWarps>;
        case 4: return attn_kernel<HD, kVarFma, 4, kWarps>;
        default: return attn_kernel<HD, kVarFma, 8, kWarps>;
    }
}

KernelFn pick_kernel(int HD, int var, int G) {
    // the MMA tiles always span 8 head columns; the FMA tile is sized to G
    if (var == kVarMma) return HD == 64 ? attn_kernel<64, kVarMma, 8, kWarps> : attn_kernel<128, kVarMma, 8, kWarps>;
    if (var == kVarFp8) return HD == 64 ? attn_kernel<64, kVarFp8, 8, kWarps> : attn_kernel<128, kVarFp8, 8, kWarps>;
    if (var == kVarInt8)
        return HD == 64 ? attn_kernel<64, kVarInt8, 8, kWarps> : attn_kernel<128, kVarInt8, 8, kWarps>;
    return HD == 64 ? fma_kernel_for<64>(gp_of(G)) : fma_kernel_for<128>(gp_of(G));
}

struct GridKey {
    int dev;
    CUcontext ctx;
    KernelFn fn;
    int smem;
};

// Persistent grid: SMs x resident CTAs of this kernel at this smem size.
// The first query for a (device, context, kernel) raises the kernel's dynamic
// shared-memory limit to the largest plan any shape uses, so a launch never
// depends on which shape was seen last; the grid is cached per smem size. A
// new context on the device (after a device reset) starts afresh.
int grid_for(KernelFn fn, int smem, int threads = (kWarps + 1) * 32) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static std::mutex mu;
    static GridKey keys[128];
    static int vals[128];
    static int nkeys = 0;
    std::lock_guard<std::mutex> lk(mu);
    const CUcontext ctx0 = current_context();
    for (int i = 0; i < nkeys; ++i)
        if (ctx0 && keys[i].dev == dev && keys[i].ctx == ctx0 && keys[i].fn == fn && keys[i].smem == smem)
            return vals[i];
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemLimit) != cudaSuccess)
        return 0;
    const CUcontext ctx = current_context();  // made current by the call above if it was not yet
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, reinterpret_cast<const void*>(fn), threads, smem) !=
        cudaSuccess)
        return 0;
    const int g = sms * (occ > 0 ? occ : 1);
    int slot = -1;
    for (int i = 0; i < nkeys && slot < 0; ++i)
        if (keys[i].dev == dev && keys[i].fn == fn && keys[i].smem == smem) slot = i;  // a stale context's entry
    if (slot < 0 && nkeys < 128) slot = nkeys++;
    if (slot >= 0 && ctx) {
        keys[slot] = GridKey{dev, ctx, fn, smem};
        vals[slot] = g;
    }
    return g;
}

mi_status check_dims(const mi_dims* dims) {
    if (!dims) return MI_ERR_INVALID_ARG;
    const mi_dims& D = *dims;
    if (D.B < 0 || D.B > 65535 || D.Hq < 1 || D.Hkv < 1 || D.num_blocks < 1 || D.max_blocks_per_seq < 1)
        return MI_ERR_INVALID_ARG;
    if (D.block_size != kBlock || (D.head_dim != 64 && D.head_dim != 128) || D.Hq % D.Hkv != 0 ||
        D.Hq / D.Hkv > kMaxG)
        return MI_ERR_UNSUPPORTED;
    if ((long long)D.num_blocks * D.Hkv * kBlock > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;
    if ((long long)D.max_blocks_per_seq * kBlock > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;
    return MI_OK;
}

int slot_floats(const mi_dims& D) { return (D.Hq / D.Hkv) * D.head_dim + 8; }

int max_grid(const mi_dims& D) {
    const int G = D.Hq / D.Hkv;
    int g = 0;
    for (int var : {kVarMma, kVarFma, kVarFp8, kVarInt8}) {
        if (!pick_stages(D.head_dim, G, var)) return 0;
        const int n = grid_for(pick_kernel(D.head_dim, var, G), smem_of(D.head_dim, G, var));
        if (n <= 0) return 0;
        g = n > g ? n : g;
    }
    return g;
}

// Unit counter words, one per CTA. A word carries the epoch of the call that
// wrote it and is zeroed by the unit's last piece, so nothing needs clearing
// between calls and a captured launch can be replayed with its one epoch.
size_t word_bytes(int grid) { return (((size_t)grid * 8) + 255) / 256 * 256; }

size_t partial_bytes(const mi_dims& D, int grid) { return (size_t)grid * 2 * (size_t)slot_floats(D) * sizeof(float); }

// Workspace: [unit counter words | partial slots | plan entries, one per CTA
// (none for batches above kPlanMaxB)].
size_t workspace_for(const mi_dims& D, int grid) {
    return word_bytes(grid) + (partial_bytes(D, grid) + 127) / 128 * 128 + (size_t)grid * plan_stride_for(D.B);
}

// A distinct value per call (in this process): a random start, then a
// counter, so a word left by earlier work in the buffer is never mistaken for
// this call's (the kernel compares the low 48 bits). The low bit is set, so an
// epoch is never the zero a finished unit leaves behind.
unsigned long long next_epoch() {
    static std::atomic<unsigned long long> ctr{0};
    static const unsigned long long start = [] {
        std::random_device rd;
        return ((unsigned long long)rd() << 32) ^ (unsigned long long)rd() ^
               (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count();
    }();
    return (start + 2 * ctr.fetch_add(1)) | 1ull;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

std::atomic<long long> g_test_wait_ns{0};  // 0: the default kWaitLimitNs
std::atomic<int> g_test_withhold{0};

}  // namespace

long long test_wait_limit_ns() {
    const long long v = g_test_wait_ns.load(std::memory_order_relaxed);
    return v > 0 ? v : kWaitLimitNs;
}

bool test_withhold_copy() { return g_test_withhold.load(std::memory_order_relaxed) != 0; }

}  // namespace mi

extern "C" mi_status mi_test_set_wait_limit(int64_t ns) {
    if (ns < 0 || ns > mi::kWaitLimitNs) return MI_ERR_INVALID_ARG;
    mi::g_test_wait_ns.store((long long)ns, std::memory_order_relaxed);
    return MI_OK;
}

extern "C" mi_status mi_test_withhold_copy(int32_t enable) {
    mi::g_test_withhold.store(enable ? 1 : 0, std::memory_order_relaxed);
    return MI_OK;
}

extern "C" size_t mi_paged_decode_workspace_bytes(const mi_dims* dims) {
    using namespace mi;
    if (check_dims(dims) != MI_OK) return 0;
    const int g = max_grid(*dims);
    if (g <= 0) return 0;
    return workspace_for(*dims, g);
}

namespace mi {
namespace {

// The new token's inputs of the fused decode step.
struct StepArgs {
    const void* k;
    const void* v;
    const float* rope;
    int32_t max_pos;
    void* q_out;
    uint32_t flags;  // MI_STEP_* bits
};

// Checks, plans and launches one attention call of variant `var` (bf16 caches
// for kVarMma / kVarFma, e4m3 caches with per-head scales for kVarFp8, INT8
// caches with per-block group maxima in k_scale / v_scale for kVarInt8);
// with `step`, the fused decode step (q is then the raw q; MMA tile).
mi_status attention(const mi_dims* dims, const void* q, const void* k_cache, const void* v_cache,
                    const float* k_scale, const float* v_scale, const int32_t* block_tables,
                    const int32_t* context_lens, float scale, void* out, void* workspace,
                    size_t workspace_bytes, int32_t* dev_err, mi_stream_t stream, int var, int32_t ctas,
                    const StepArgs* step = nullptr) {
    const mi_status ds = check_dims(dims);
    if (ds != MI_OK) return ds;
    const mi_dims D = *dims;
    if (D.B == 0) return MI_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
        return MI_ERR_INVALID_ARG;
    if ((var == kVarFp8 || var == kVarInt8) && (!k_scale || !v_scale)) return MI_ERR_INVALID_ARG;
    if (var == kVarInt8 && ((reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) & 3u))
        return MI_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q) || !aligned16(out) ||
        !aligned16(workspace))
        return MI_ERR_INVALID_ARG;
    if (ctas < 0 || !std::isfinite(scale)) return MI_ERR_INVALID_ARG;
    const int G = D.Hq / D.Hkv, HD = D.head_dim;
    if (step) {
        if ((var != kVarMma && var != kVarFp8) || !step->k || !step->v || !step->rope || !step->q_out ||
            step->max_pos < 1)
            return MI_ERR_INVALID_ARG;
        if (!aligned16(step->k) || !aligned16(step->v) || !aligned16(step->rope) || !aligned16(step->q_out))
            return MI_ERR_INVALID_ARG;
        // q is read by every CTA holding a piece of a unit, q_out written by
        // one of them: they must not overlap
        const uintptr_t qa = reinterpret_cast<uintptr_t>(q), oa = reinterpret_cast<uintptr_t>(step->q_out);
        const uintptr_t qbytes = (uintptr_t)D.B * D.Hq * HD * 2;
        if (qa < oa + qbytes && oa < qa + qbytes) return MI_ERR_INVALID_ARG;
    }
    const bool fused = step != nullptr;
    const int S = pick_stages(HD, G, var, fused);
    const int smem = smem_of(HD, G, var, fused);
    const int threads = (kWarps + (fused ? 2 : 1)) * 32;
    if (S <= 0) return MI_ERR_UNSUPPORTED;
    // the workspace is sized for the widest grid of any variant; this
    // kernel's own persistent grid is its SMs x resident CTAs
    const int gmax = max_grid(D);
    if (gmax <= 0) return MI_ERR_CUDA;
    if (workspace_bytes < workspace_for(D, gmax)) return MI_ERR_INVALID_ARG;
    KernelFn fn = !step ? pick_kernel(HD, var, G)
                : var == kVarFp8 ? (HD == 64 ? attn_kernel<64, kVarFp8, 8, kWarps, true>
                                             : attn_kernel<128, kVarFp8, 8, kWarps, true>)
                                 : (HD == 64 ? attn_kernel<64, kVarMma, 8, kWarps, true>
                                             : attn_kernel<128, kVarMma, 8, kWarps, true>);
    const int gown = grid_for(fn, smem, threads);
    if (gown <= 0 || gown > gmax) return MI_ERR_CUDA;
    const int grid = ctas > 0 && ctas < gown ? ctas : gown;

    CUtensorMap tk, tv;
    const long long rows = (long long)D.num_blocks * D.Hkv * kBlock;
    const bool maps = elem_bytes(var) == 1 ? make_tmap8(&tk, k_cache, rows, HD) && make_tmap8(&tv, v_cache, rows, HD)
                                           : make_tmap(&tk, k_cache, rows, HD) && make_tmap(&tv, v_cache, rows, HD);
    if (!maps) return MI_ERR_CUDA;

    AttnParams p;
    p.q = static_cast<const uint16_t*>(q);
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<uint16_t*>(out);
    p.unit_word = static_cast<unsigned long long*>(workspace);
    p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + word_bytes(gmax));
    p.plan_stride = plan_stride_for(D.B);
    p.plan_cache = p.plan_stride > 0 ? static_cast<uint8_t*>(workspace) + word_bytes(gmax) +
                                           (partial_bytes(D, gmax) + 127) / 128 * 128
                                     : nullptr;
    p.plan_kind = var * 2 + (step ? 1 : 0);
    p.epoch = next_epoch();
    p.dev_err = dev_err;
    p.B = D.B;
    p.Hq = D.Hq;
    p.Hkv = D.Hkv;
    p.G = G;
    p.num_blocks = D.num_blocks;
    p.mbps = D.max_blocks_per_seq;
    p.stages = S;
    p.slot_floats = slot_floats(D);
    p.grid = grid;
    p.sl2 = scale * 1.4426950408889634f;
    p.k_scale = var == kVarFp8 ? k_scale : nullptr;
    p.v_scale = var == kVarFp8 ? v_scale : nullptr;
    p.k_amax = var == kVarInt8 ? k_scale : nullptr;
    p.v_amax = var == kVarInt8 ? v_scale : nullptr;
    p.qraw = static_cast<const uint16_t*>(q);
    p.knew = step ? static_cast<const uint16_t*>(step->k) : nullptr;
    p.vnew = step ? static_cast<const uint16_t*>(step->v) : nullptr;
    p.rope = step ? reinterpret_cast<const float2*>(step->rope) : nullptr;
    p.q_out = step ? static_cast<uint16_t*>(step->q_out) : nullptr;
    p.kc = static_cast<uint16_t*>(const_cast<void*>(k_cache));
    p.vc = static_cast<uint16_t*>(const_cast<void*>(v_cache));
    p.max_pos = step ? step->max_pos : 0;
    p.wait_ns = test_wait_limit_ns();
    p.early = step && (step->flags & MI_STEP_EARLY_START) ? 1 : 0;
    p.withhold = test_withhold_copy() ? 1 : 0;

    cudaStream_t s = (cudaStream_t)stream;
    return launch_pdl(fn, grid, threads, smem, s, tk, tv, p) == cudaSuccess ? MI_OK : MI_ERR_CUDA;
}

}  // namespace
}  // namespace mi

extern "C" mi_status mi_paged_decode_attention_variant(const mi_dims* dims, const void* q,
                                                       const void* k_cache, const void* v_cache,
                                                       const int32_t* block_tables,
                                                       const int32_t* context_lens, float scale,
                                                       void* out, void* workspace,
                                                       size_t workspace_bytes, int32_t* dev_err,
                                                       mi_stream_t stream, mi_attn_variant variant,
                                                       int32_t ctas) {
    using namespace mi;
    if (variant != MI_ATTN_DEFAULT && variant != MI_ATTN_MMA && variant != MI_ATTN_FMA)
        return MI_ERR_INVALID_ARG;
    return attention(dims, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, scale, out,
                     workspace, workspace_bytes, dev_err, stream, variant == MI_ATTN_FMA ? kVarFma : kVarMma,
                     ctas);
}

extern "C" mi_status mi_paged_decode_step(const mi_dims* dims, const void* q, const void* k, const void* v,
                                        const float* rope_cos_sin, int32_t max_pos,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        float scale, void* q_out, void* k_cache, void* v_cache, void* out,
                                        void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                        mi_stream_t stream, uint32_t flags) {
    using namespace mi;
    if (flags & ~MI_STEP_EARLY_START) return MI_ERR_INVALID_ARG;
    const StepArgs step{k, v, rope_cos_sin, max_pos, q_out, flags};
    return attention(dims, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens, scale, out,
                     workspace, workspace_bytes, dev_err, stream, kVarMma, 0, &step);
}

extern "C" mi_status mi_paged_decode_step_fp8(const mi_dims* dims, const void* q, const void* k, const void* v,
                                            const float* rope_cos_sin, int32_t max_pos,
                                            const int32_t* block_tables, const int32_t* context_lens,
                                            const float* k_scale, const float* v_scale, float scale, void* q_out,
                                            void* k_cache, void* v_cache, void* out, void* workspace,
                                            size_t workspace_bytes, int32_t* dev_err, mi_stream_t stream,
                                            uint32_t flags) {
    using namespace mi;
    if (flags & ~MI_STEP_EARLY_START) return MI_ERR_INVALID_ARG;
    const StepArgs step{k, v, rope_cos_sin, max_pos, q_out, flags};
    return attention(dims, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
                     workspace, workspace_bytes, dev_err, stream, kVarFp8, 0, &step);
}

extern "C" mi_status mi_paged_decode_attention_fp8(const mi_dims* dims, const void* q, const void* k_cache,
                                                   const void* v_cache, const float* k_scale,
                                                   const float* v_scale, const int32_t* block_tables,
                                                   const int32_t* context_lens, float scale, void* out,
                                                   void* workspace, size_t workspace_bytes,
                                                   int32_t* dev_err, mi_stream_t stream) {
    using namespace mi;
    return attention(dims, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, out,
                     workspace, workspace_bytes, dev_err, stream, kVarFp8, 0);
}

extern "C" mi_status mi_paged_decode_attention(const mi_dims* dims, const void* q, const void* k_cache,
                                               const void* v_cache, const int32_t* block_tables,
                                               const int32_t* context_lens, float scale, void* out,
                                               void* workspace, size_t workspace_bytes,
                                               int32_t* dev_err, mi_stream_t stream) {
    return mi_paged_decode_attention_variant(dims, q, k_cache, v_cache, block_tables, context_lens, scale,
                                             out, workspace, workspace_bytes, dev_err, stream,
                                             MI_ATTN_DEFAULT, 0);
}

extern "C" mi_status mi_paged_decode_attention_int8(const mi_dims* dims, const void* q, const void* k_cache,
                                                    const void* v_cache, const float* k_amax, const float* v_amax,
                                                    const int32_t* block_tables, const int32_t* context_lens,
                                                    float scale, void* out, void* workspace,
                                                    size_t workspace_bytes, int32_t* dev_err, mi_stream_t stream) {
    using namespace mi;
    return attention(dims, q, k_cache, v_cache, k_amax, v_amax, block_tables, context_lens, scale, out,
                     workspace, workspace_bytes, dev_err, stream, kVarInt8, 0);
}
