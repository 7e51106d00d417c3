// Staging of 16-token KV tiles by TMA, shared by the decode and prefill
// attention kernels: the host-side tensor map over a paged cache and the
// device-side address of a 16-byte chunk inside a staged, 128-byte-swizzled
// tile.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace mi {

// Physical byte offset of 16-byte chunk `chunk` (0 .. HD/8-1) of token row
// `row` inside a tile written by one 128-byte-swizzled TMA box. The cache is
// viewed as 128-byte lines (HD/64 per token), so a 16-token tile is one
// contiguous box of 16*HD/64 lines; chunk c of line l sits at c ^ (l & 7).
// The tile must start on a 1024-byte boundary.
template <int HD>
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    const int line = row * (HD / 64) + (chunk >> 3);
    return (uint32_t)(line * 128 + (((chunk & 7) ^ (line & 7)) << 4));
}

// The same for a tile of one-byte (e4m3) elements: a token row is HD bytes,
// so a 128-byte line holds 128/HD token rows; chunk c (0 .. HD/16-1) of row r
// is byte r*HD + 16c of the tile before the swizzle.
template <int HD>
__device__ __forceinline__ uint32_t swz8(int row, int chunk) {
    const int byte = row * HD + chunk * 16;
    const int line = byte >> 7, cil = (byte >> 4) & 7;
    return (uint32_t)(line * 128 + ((cil ^ (line & 7)) << 4));
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda); nullptr when the driver does not provide it.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult qr;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// The calling thread's current CUDA context (cuCtxGetCurrent through the
// runtime's driver entry point), or nullptr when there is none yet. Caches of
// per-device set-up (kernel attributes, symbol addresses) are keyed by it: a
// device reset makes a new context, and the set-up is then done again.
inline CUcontext current_context() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult qr;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// 2-D map over a cache viewed as 128-byte lines: [rows * HD/64][64] bf16,
// box = one 16-token tile (16 * HD/64 lines x 64 columns), 128-byte swizzle.
// `rows` counts token rows of all blocks and KV heads (num_blocks * Hkv * 16).
inline bool make_tmap(CUtensorMap* m, const void* base, long long rows, int HD) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {64, (cuuint64_t)rows * (HD / 64)};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {64, (cuuint32_t)(kBlock * HD / 64)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D map over a one-byte (e4m3) cache viewed as 128-byte lines:
// [rows * HD/128][128] u8, box = one 16-token tile (16 * HD/128 lines), 128-byte
// swizzle.
inline bool make_tmap8(CUtensorMap* m, const void* base, long long rows, int HD) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {128, (cuuint64_t)rows * HD / 128};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, (cuuint32_t)(kBlock * HD / 128)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map over a bf16 cache for canonical K-major tiles: dims {64, HD/64,
// rows} (a token row split into 128-byte halves), box {64, 1, 16}: one
// 128-byte half of 16 token rows, landing as [16][128 B] with 128-byte swizzle.
inline bool make_tmap_kv_halves(CUtensorMap* m, const void* base, long long rows, int HD) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)(HD / 64), (cuuint64_t)rows};
    cuuint64_t strides[2] = {128, (cuuint64_t)HD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kBlock};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map over a bf16 cache for whole blocks: dims {64, rows, HD/64} (the
// 128-byte halves of a token row as the outer dimension), box {64, 16,
// HD/64}: all of a block's 16 token rows in one copy, landing as
// [HD/64][16][128 B] with 128-byte swizzle (each half's 16 rows together).
inline bool make_tmap_kv_blocks(CUtensorMap* m, const void* base, long long rows, int HD) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(HD / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)HD * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kBlock, (cuuint32_t)(HD / 64)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D map over q [T][Hq][HD] bf16: dims {64, HD/64, Hq, T}, box {64, 1, G,
// rows / G}: one 128-byte half of `rows` (token, head) rows of a GQA group,
// landing as [rows][128 B] with 128-byte swizzle; tokens past T read as zero.
inline bool make_tmap_q_group(CUtensorMap* m, const void* q, int T, int Hq, int HD, int G, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)(HD / 64), (cuuint64_t)Hq, (cuuint64_t)T};
    cuuint64_t strides[3] = {128, (cuuint64_t)HD * 2, (cuuint64_t)Hq * HD * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)G, (cuuint32_t)(rows / G)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mi
