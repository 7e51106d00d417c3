// mi_paged_kv_append: RoPE on the new token's q/k, then scatter k/v into the
// paged cache through slot_mapping (mini-infer README, "decode_batch 关键步骤",
// write_decode_kv; RoPE as the NJU course brief "端侧大模型推理框架" §2.1 lists
// it). The rotation is done in double from bf16 inputs and fp32 table values
// (each product exact), then rounded once to bf16, so the result is a fixed
// function of the inputs.
#include "common.cuh"

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
    uint16_t* k_cache;
    uint16_t* v_cache;
    int32_t* dev_err;
    int Hq, Hkv, d, num_blocks, max_pos;
};

// One CTA per request. Threads walk (head, pair) items: heads 0..Hq-1 are
// query heads (to q_out), heads Hq..Hq+Hkv-1 are key heads (to the cache);
// then 16-byte chunks of v are copied.
__global__ void __launch_bounds__(256) append_kernel(AppendParams a) {
    const int b = blockIdx.x;
    const int p = a.positions[b];
    if (p < 0 || p >= a.max_pos) {
        if (threadIdx.x == 0) raise_err(a.dev_err, MI_DEVERR_BAD_POS);
        return;
    }
    const int slot = a.slot_mapping[b];
    const bool slot_ok = slot >= 0 && slot < a.num_blocks * kBlock;
    if (!slot_ok && threadIdx.x == 0) raise_err(a.dev_err, MI_DEVERR_BAD_SLOT);
    const long long blk = slot_ok ? slot / kBlock : 0;
    const int off = slot_ok ? slot % kBlock : 0;
    const int half = a.d / 2;
    const float2* cs = a.rope + (long long)p * half;
    const int items = (a.Hq + a.Hkv) * half;
    for (int idx = threadIdx.x; idx < items; idx += blockDim.x) {
        const int head = idx / half;
        const int i = idx - head * half;
        const bool is_q = head < a.Hq;
        if (!is_q && !slot_ok) continue;
        const uint16_t* src = is_q ? a.q + ((long long)b * a.Hq + head) * a.d
                                   : a.k + ((long long)b * a.Hkv + (head - a.Hq)) * a.d;
        const double x1 = (double)bf16_to_f32(src[i]);
        const double x2 = (double)bf16_to_f32(src[i + half]);
        const float2 t = cs[i];
        const double c = (double)t.x, s = (double)t.y;
        const double y1 = x1 * c - x2 * s;  // products are exact in double
        const double y2 = x2 * c + x1 * s;
        uint16_t* dst = is_q ? a.q_out + ((long long)b * a.Hq + head) * a.d
                             : a.k_cache + ((blk * a.Hkv + (head - a.Hq)) * kBlock + off) * a.d;
        dst[i] = f64_to_bf16(y1);
        dst[i + half] = f64_to_bf16(y2);
    }
    if (!slot_ok) return;
    const int chunks = a.d / 8;  // 16-byte chunks per head vector
    for (int idx = threadIdx.x; idx < a.Hkv * chunks; idx += blockDim.x) {
        const int h = idx / chunks, c = idx - h * chunks;
        const uint4 val = reinterpret_cast<const uint4*>(a.v + ((long long)b * a.Hkv + h) * a.d)[c];
        reinterpret_cast<uint4*>(a.v_cache + ((blk * a.Hkv + h) * kBlock + off) * a.d)[c] = val;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mi

extern "C" mi_status mi_paged_kv_append(const mi_dims* dims, const void* q, const void* k,
                                        const void* v, const int32_t* positions,
                                        const int32_t* slot_mapping, const float* rope_cos_sin,
                                        int32_t max_pos, void* q_out, void* k_cache, void* v_cache,
                                        int32_t* dev_err, mi_stream_t stream) {
    using namespace mi;
    if (!dims) return MI_ERR_INVALID_ARG;
    const mi_dims D = *dims;
    if (D.B < 0 || D.B > 65535 || D.Hq < 1 || D.Hkv < 1 || D.num_blocks < 1 || max_pos < 1)
        return MI_ERR_INVALID_ARG;
    if (D.block_size != kBlock || (D.head_dim != 64 && D.head_dim != 128) || D.Hq % D.Hkv != 0)
        return MI_ERR_UNSUPPORTED;
    if ((long long)D.num_blocks * kBlock > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;
    if (D.B == 0) return MI_OK;
    if (!q || !k || !v || !positions || !slot_mapping || !rope_cos_sin || !q_out || !k_cache || !v_cache)
        return MI_ERR_INVALID_ARG;
    if (!aligned16(v) || !aligned16(v_cache) || !aligned16(rope_cos_sin)) return MI_ERR_INVALID_ARG;
    AppendParams a;
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.positions = positions;
    a.slot_mapping = slot_mapping;
    a.rope = reinterpret_cast<const float2*>(rope_cos_sin);
    a.q_out = static_cast<uint16_t*>(q_out);
    a.k_cache = static_cast<uint16_t*>(k_cache);
    a.v_cache = static_cast<uint16_t*>(v_cache);
    a.dev_err = dev_err;
    a.Hq = D.Hq;
    a.Hkv = D.Hkv;
    a.d = D.head_dim;
    a.num_blocks = D.num_blocks;
    a.max_pos = max_pos;
    append_kernel<<<D.B, 256, 0, (cudaStream_t)stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? MI_OK : MI_ERR_CUDA;
}
