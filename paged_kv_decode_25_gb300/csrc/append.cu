// mi_paged_kv_append: RoPE on the new token's q/k, then scatter k/v into the
// paged cache through slot_mapping (mini-infer README, "decode_batch 关键步骤",
// write_decode_kv; RoPE as the NJU course brief "端侧大模型推理框架" §2.1 lists
// it). The rotation is defined in double from bf16 inputs and fp32 table
// values (each product exact), then rounded once to bf16, so the result is a
// fixed function of the inputs; it is computed in single precision with
// error-free transformations when that provably gives the same bits, else in
// double.
#include "common.cuh"
#include "rope.cuh"

namespace mi {
namespace {

struct AppendParams {
    const uint16_t* q;
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* positions;
    const int32_t* slot_mapping;
    const float2* rope;  // [max_pos][d/2] (cos, sin)
    uint16_t* q_out;
    uint16_t* k_cache;             // bf16 caches
    uint16_t* v_cache;
    uint8_t* k_cache8;             // e4m3 caches (FP8 append)
    uint8_t* v_cache8;
    const float* k_scale;          // [Hkv] e4m3 quantisation scales
    const float* v_scale;
    int32_t* dev_err;
    int Hq, Hkv, d, num_blocks, max_pos;
};

// Eight bf16 values (packed pairs) / scale in IEEE single precision, then to
// e4m3 (nearest-even, saturating): eight codes, first value in the low byte.
__device__ __forceinline__ uint2 quantize8(const uint32_t (&x)[4], float scale) {
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        c[j] = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(x[j]), scale), __fdiv_rn(bf16_hi(x[j]), scale));
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__device__ __forceinline__ bool scale_ok(float s) { return s > 0.f && s <= 3.0e38f; }

// Words of NJ bf16 pairs (NJ = 4: 16 bytes, NJ = 1: 4 bytes).
template <int NJ>
__device__ __forceinline__ void load_words(const uint16_t* src, uint32_t (&x)[NJ]) {
    if constexpr (NJ == 4) {
        const uint4 w = *reinterpret_cast<const uint4*>(src);
        x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
    } else {
        x[0] = *reinterpret_cast<const uint32_t*>(src);
    }
}
template <int NJ>
__device__ __forceinline__ void store_words(uint16_t* dst, const uint32_t (&y)[NJ]) {
    if constexpr (NJ == 4) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(y[0], y[1], y[2], y[3]);
    } else {
        *reinterpret_cast<uint32_t*>(dst) = y[0];
    }
}
template <int NJ>
__device__ __forceinline__ void store_e4m3(uint8_t* dst, const uint32_t (&y)[NJ], float scale) {
    if constexpr (NJ == 4) {
        *reinterpret_cast<uint2*>(dst) = quantize8(y, scale);
    } else {
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)f32x2_to_e4m3x2(__fdiv_rn(bf16_lo(y[0]), scale),
                                                                      __fdiv_rn(bf16_hi(y[0]), scale));
    }
}

// The rare second pass of a thread's rotation: each word flagged in `need`
// is rotated again by the exact route and stored over the fast result (bf16
// words at lo / hi, or, with E4M3, its two e4m3 pairs quantised with
// `scale`). The inputs stay in registers (q_out may alias q, so the source
// cannot be re-read); a rolled loop with a select keeps this pass compact
// and keeps the out-of-line call away from the main rotation.
template <int NJ, bool E4M3, typename T>
__device__ __forceinline__ void exact_words(unsigned need, const uint32_t (&xl)[NJ], const uint32_t (&xh)[NJ],
                                         const float4 (&cs)[NJ], T* lo, T* hi, float scale) {
#pragma unroll 1
    for (int j = 0; j < NJ; ++j) {
        if (!((need >> j) & 1u)) continue;
        uint32_t wl = xl[0], wh = xh[0];
        float4 c = cs[0];
#pragma unroll
        for (int jj = 1; jj < NJ; ++jj)
            if (j == jj) {
                wl = xl[jj];
                wh = xh[jj];
                c = cs[jj];
            }
        const uint2 y = rotate_word_exact(wl, wh, c);
        if constexpr (E4M3) {
            const uint32_t yl1[1] = {y.x}, yh1[1] = {y.y};
            store_e4m3<1>(reinterpret_cast<uint8_t*>(lo) + 2 * j, yl1, scale);
            store_e4m3<1>(reinterpret_cast<uint8_t*>(hi) + 2 * j, yh1, scale);
        } else {
            *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(lo) + 2 * j) = y.x;
            *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(hi) + 2 * j) = y.y;
        }
    }
}

// One thread per (request, head, group of PPT rotation pairs): heads 0..Hq-1
// are query heads (to q_out), heads Hq..Hq+Hkv-1 key heads (to the cache).
// Each thread loads its two halves and its PPT (cos, sin) pairs before it
// computes or stores anything, so q_out may alias q. Threads past the
// rotation items copy 16-byte chunks of v into the cache. PPT = 8 for many
// rows (prefill), 2 for a decode batch (more threads, shorter chains).
template <bool FP8, int PPT>
__global__ void __launch_bounds__(128) append_kernel(AppendParams a, int B) {
    // inputs may come from the kernel just before this one in the stream
    pdl_wait();
    pdl_trigger();
    constexpr int NJ = PPT / 2;  // 32-bit words (bf16 pairs) per half
    const int half = a.d / 2;
    const int groups = half / PPT;  // PPT-pair groups per head
    const long long n_rot = (long long)B * (a.Hq + a.Hkv) * groups;
    const long long n_cpy = (long long)B * a.Hkv * (a.d / 8);
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    // d is 64 or 128: groups (d/2/PPT) and chunks (d/8) are powers of two,
    // and the remaining divisions run in 32 bits whenever the quotient range
    // fits
    const int lgc = a.d == 128 ? 4 : 3;
    const int lgg = lgc + 2 - (PPT == 8 ? 3 : 1);
    if (t < n_rot) {
        const int grp = (int)(t & (groups - 1));
        const long long bh = t >> lgg;
        const int HH = a.Hq + a.Hkv;
        int head, b;
        if (bh <= 0xFFFFFFFFLL) {
            const uint32_t u = (uint32_t)bh;
            head = (int)(u % (uint32_t)HH);
            b = (int)(u / (uint32_t)HH);
        } else {
            head = (int)(bh % HH);
            b = (int)(bh / HH);
        }
        const bool is_q = head < a.Hq;
        const uint16_t* src = is_q ? a.q + ((long long)b * a.Hq + head) * a.d
                                   : a.k + ((long long)b * a.Hkv + (head - a.Hq)) * a.d;
        const int i0 = grp * PPT;
        // issue the independent loads first
        uint32_t xl[NJ], xh[NJ];
        load_words<NJ>(src + i0, xl);
        load_words<NJ>(src + i0 + half, xh);
        const int p = a.positions[b];
        const int slot = is_q ? 0 : a.slot_mapping[b];
        if (p < 0 || p >= a.max_pos) {
            if (head == 0 && grp == 0) raise_err(a.dev_err, MI_DEVERR_BAD_POS);  // once per request
            return;
        }
        long long dst_off;
        if (is_q) {
            dst_off = ((long long)b * a.Hq + head) * a.d;
        } else {
            if (slot < 0 || slot >= a.num_blocks * kBlock) {
                if (head == a.Hq && grp == 0) raise_err(a.dev_err, MI_DEVERR_BAD_SLOT);
                return;
            }
            dst_off = (((long long)(slot / kBlock) * a.Hkv + (head - a.Hq)) * kBlock + slot % kBlock) * a.d;
        }
        const float4* cs4 = reinterpret_cast<const float4*>(a.rope + (long long)p * half + i0);
        float4 cs[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) cs[j] = cs4[j];
        uint32_t yl[NJ], yh[NJ];
        unsigned need = 0;  // words whose values need the exact route
#pragma unroll
        for (int j = 0; j < NJ; ++j) need |= (unsigned)rotate_word_fast(xl[j], xh[j], cs[j], yl[j], yh[j]) << j;
        if (FP8 && !is_q) {
            const float ks = a.k_scale[head - a.Hq];
            if (!scale_ok(ks)) {
                if (grp == 0) raise_err(a.dev_err, MI_DEVERR_BAD_SCALE);
                return;
            }
            uint8_t* dst8 = a.k_cache8 + dst_off;
            store_e4m3<NJ>(dst8 + i0, yl, ks);
            store_e4m3<NJ>(dst8 + i0 + half, yh, ks);
            if (need) exact_words<NJ, true>(need, xl, xh, cs, dst8 + i0, dst8 + i0 + half, ks);
            return;
        }
        uint16_t* dst = (is_q ? a.q_out : a.k_cache) + dst_off;
        store_words<NJ>(dst + i0, yl);
        store_words<NJ>(dst + i0 + half, yh);
        if (need) exact_words<NJ, false>(need, xl, xh, cs, dst + i0, dst + i0 + half, 0.f);
        return;
    }
    const long long c = t - n_rot;
    if (c >= n_cpy) return;
    const int chunks = a.d / 8;
    const int ch = (int)(c & (chunks - 1));
    const long long bh = c >> lgc;
    int h, b;
    if (bh <= 0xFFFFFFFFLL) {
        const uint32_t u = (uint32_t)bh;
        h = (int)(u % (uint32_t)a.Hkv);
        b = (int)(u / (uint32_t)a.Hkv);
    } else {
        h = (int)(bh % a.Hkv);
        b = (int)(bh / a.Hkv);
    }
    const int p = a.positions[b];
    const int slot = a.slot_mapping[b];
    if (p < 0 || p >= a.max_pos || slot < 0 || slot >= a.num_blocks * kBlock) return;
    const uint4 val = reinterpret_cast<const uint4*>(a.v + ((long long)b * a.Hkv + h) * a.d)[ch];
    const long long row = (((long long)(slot / kBlock) * a.Hkv + h) * kBlock + slot % kBlock) * a.d;
    if (FP8) {
        const float vs = a.v_scale[h];
        if (!scale_ok(vs)) {
            if (ch == 0) raise_err(a.dev_err, MI_DEVERR_BAD_SCALE);
            return;
        }
        const uint32_t x[4] = {val.x, val.y, val.z, val.w};
        reinterpret_cast<uint2*>(a.v_cache8 + row)[ch] = quantize8(x, vs);
    } else {
        reinterpret_cast<uint4*>(a.v_cache + row)[ch] = val;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mi

namespace mi {
namespace {

mi_status append(const mi_dims* dims, const void* q, const void* k, const void* v, const int32_t* positions,
                 const int32_t* slot_mapping, const float* rope_cos_sin, int32_t max_pos, void* q_out,
                 void* k_cache, void* v_cache, const float* k_scale, const float* v_scale, bool fp8,
                 int32_t* dev_err, mi_stream_t stream) {
    if (!dims) return MI_ERR_INVALID_ARG;
    const mi_dims D = *dims;
    if (D.B < 0 || D.B > (1 << 24) || D.Hq < 1 || D.Hkv < 1 || D.num_blocks < 1 || max_pos < 1)
        return MI_ERR_INVALID_ARG;
    if (D.block_size != kBlock || (D.head_dim != 64 && D.head_dim != 128) || D.Hq % D.Hkv != 0)
        return MI_ERR_UNSUPPORTED;
    if ((long long)D.num_blocks * kBlock > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;
    if (D.B == 0) return MI_OK;
    if (!q || !k || !v || !positions || !slot_mapping || !rope_cos_sin || !q_out || !k_cache || !v_cache)
        return MI_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale)) return MI_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out) || !aligned16(k_cache) ||
        !aligned16(v_cache) || !aligned16(rope_cos_sin))
        return MI_ERR_INVALID_ARG;
    AppendParams a;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.positions = positions;
    a.slot_mapping = slot_mapping;
    a.rope = reinterpret_cast<const float2*>(rope_cos_sin);
    a.q_out = static_cast<uint16_t*>(q_out);
    a.k_cache = fp8 ? nullptr : static_cast<uint16_t*>(k_cache);
    a.v_cache = fp8 ? nullptr : static_cast<uint16_t*>(v_cache);
    a.k_cache8 = fp8 ? static_cast<uint8_t*>(k_cache) : nullptr;
    a.v_cache8 = fp8 ? static_cast<uint8_t*>(v_cache) : nullptr;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.dev_err = dev_err;
    a.Hq = D.Hq;
    a.Hkv = D.Hkv;
    a.d = D.head_dim;
    a.num_blocks = D.num_blocks;
    a.max_pos = max_pos;
    // few rows (a decode batch): two pairs per thread, else eight
    const int ppt = D.B <= 256 ? 2 : 8;
    const long long threads = (long long)D.B * (D.Hq + D.Hkv) * (D.head_dim / 2 / ppt) +
                              (long long)D.B * D.Hkv * (D.head_dim / 8);
    const long long grid = (threads + 127) / 128;
    if (grid > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;
    const cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (ppt == 2)
        e = fp8 ? launch_pdl(append_kernel<true, 2>, (int)grid, 128, 0, st, a, (int)D.B)
                : launch_pdl(append_kernel<false, 2>, (int)grid, 128, 0, st, a, (int)D.B);
    else
        e = fp8 ? launch_pdl(append_kernel<true, 8>, (int)grid, 128, 0, st, a, (int)D.B)
                : launch_pdl(append_kernel<false, 8>, (int)grid, 128, 0, st, a, (int)D.B);
    return e == cudaSuccess ? MI_OK : MI_ERR_CUDA;
}

}  // namespace
}  // namespace mi

extern "C" mi_status mi_paged_kv_append(const mi_dims* dims, const void* q, const void* k,
                                        const void* v, const int32_t* positions,
                                        const int32_t* slot_mapping, const float* rope_cos_sin,
                                        int32_t max_pos, void* q_out, void* k_cache, void* v_cache,
                                        int32_t* dev_err, mi_stream_t stream) {
    return mi::append(dims, q, k, v, positions, slot_mapping, rope_cos_sin, max_pos, q_out, k_cache, v_cache,
                      nullptr, nullptr, false, dev_err, stream);
}

extern "C" mi_status mi_paged_kv_append_fp8(const mi_dims* dims, const void* q, const void* k,
                                            const void* v, const int32_t* positions,
                                            const int32_t* slot_mapping, const float* rope_cos_sin,
                                            int32_t max_pos, void* q_out, void* k_cache, void* v_cache,
                                            const float* k_scale, const float* v_scale, int32_t* dev_err,
                                            mi_stream_t stream) {
    return mi::append(dims, q, k, v, positions, slot_mapping, rope_cos_sin, max_pos, q_out, k_cache, v_cache,
                      k_scale, v_scale, true, dev_err, stream);
}
