// mi_kv_copy_blocks: copy whole KV blocks between two paged caches, the data
// movement of a KV swap (NJU course brief "端侧大模型推理框架", optional task 3
// "KV Cache Offloading": inactive blocks go to CPU memory and come back when
// needed). Either cache may live in device memory or in pinned host memory:
// on a Grace-Blackwell node the SMs reach host memory over the coherent
// chip-to-chip link, so one launch gathers or scatters any list of blocks
// with no per-block copy call.
//
// One CTA per (pair, K or V): 256 threads move the block's Hkv*16*d*2 bytes
// as 16-byte vectors, eight loads in flight per thread before the stores.
// mi_kv_copy_rows does the same for rows of any length (a multiple of 4
// bytes): the blocks of one-byte caches, and the INT8 group maxima and
// open-group rows that move with a sequence.
#include "common.cuh"

namespace mi {
namespace {

struct CopyParams {
    const uint4* src_k;
    const uint4* src_v;
    uint4* dst_k;
    uint4* dst_v;
    const int32_t* src_blocks;
    const int32_t* dst_blocks;
    int32_t* dev_err;
    long long block_vecs;  // 16-byte vectors per block (all KV heads)
    int src_num_blocks, dst_num_blocks, n;
};

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(CopyParams p) {
    pdl_wait();
    pdl_trigger();
    const int pair = blockIdx.x >> 1;
    const bool is_v = blockIdx.x & 1;
    if (pair >= p.n) return;
    const int s = __ldg(p.src_blocks + pair), d = __ldg(p.dst_blocks + pair);
    if (s < 0 || s >= p.src_num_blocks || d < 0 || d >= p.dst_num_blocks) {
        if (!is_v && threadIdx.x == 0) raise_err(p.dev_err, MI_DEVERR_BAD_BLOCK);
        return;
    }
    const uint4* src = (is_v ? p.src_v : p.src_k) + (long long)s * p.block_vecs;
    uint4* dst = (is_v ? p.dst_v : p.dst_k) + (long long)d * p.block_vecs;
    constexpr int kStep = kCopyThreads * kCopyUnroll;
    for (long long base = 0; base < p.block_vecs; base += kStep) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const long long i = base + u * kCopyThreads + threadIdx.x;
            if (i < p.block_vecs) v[u] = src[i];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const long long i = base + u * kCopyThreads + threadIdx.x;
            if (i < p.block_vecs) dst[i] = v[u];
        }
    }
}

// Rows of any length (mi_kv_copy_rows): one CTA per row, U = uint4 (16-byte
// vectors) or uint32_t (rows a multiple of 4 bytes only).
struct RowParams {
    const void* src;
    void* dst;
    const int32_t* src_ids;
    const int32_t* dst_ids;
    int32_t* dev_err;
    long long row_units;  // U-sized words per row
    long long src_count, dst_count;
    int n;
};

template <typename U>
__global__ void __launch_bounds__(kCopyThreads) copy_rows_kernel(RowParams p) {
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x;
    if (row >= p.n) return;
    const long long s = __ldg(p.src_ids + row), d = __ldg(p.dst_ids + row);
    if (s < 0 || s >= p.src_count || d < 0 || d >= p.dst_count) {
        if (threadIdx.x == 0) raise_err(p.dev_err, MI_DEVERR_BAD_BLOCK);
        return;
    }
    const U* src = static_cast<const U*>(p.src) + s * p.row_units;
    U* dst = static_cast<U*>(p.dst) + d * p.row_units;
    constexpr int kStep = kCopyThreads * kCopyUnroll;
    for (long long base = 0; base < p.row_units; base += kStep) {
        U v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const long long i = base + u * kCopyThreads + threadIdx.x;
            if (i < p.row_units) v[u] = src[i];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const long long i = base + u * kCopyThreads + threadIdx.x;
            if (i < p.row_units) dst[i] = v[u];
        }
    }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// The address the kernel uses for a device or pinned host pointer; nullptr
// for memory the device cannot reach (pageable host memory).
const void* device_alias(const void* ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return ptr;
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

}  // namespace
}  // namespace mi

extern "C" mi_status mi_kv_copy_blocks(const mi_dims* dims, const void* src_k, const void* src_v,
                                       int32_t src_num_blocks, const int32_t* src_blocks, void* dst_k,
                                       void* dst_v, int32_t dst_num_blocks, const int32_t* dst_blocks,
                                       int32_t n, int32_t* dev_err, mi_stream_t stream) {
    using namespace mi;
    if (!dims || n < 0 || src_num_blocks < 1 || dst_num_blocks < 1) return MI_ERR_INVALID_ARG;
    const mi_dims D = *dims;
    if (D.Hkv < 1) return MI_ERR_INVALID_ARG;
    if (D.block_size != kBlock || (D.head_dim != 64 && D.head_dim != 128)) return MI_ERR_UNSUPPORTED;
    if (n == 0) return MI_OK;
    if ((long long)n * 2 > 0x7FFFFFFFLL) return MI_ERR_INVALID_ARG;
    if (!src_k || !src_v || !dst_k || !dst_v || !src_blocks || !dst_blocks) return MI_ERR_INVALID_ARG;
    if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v))
        return MI_ERR_INVALID_ARG;
    const void* ptrs[6] = {src_k, src_v, dst_k, dst_v, src_blocks, dst_blocks};
    const void* dev[6];
    for (int i = 0; i < 6; ++i)
        if (!(dev[i] = device_alias(ptrs[i]))) return MI_ERR_INVALID_ARG;
    CopyParams p;
    p.src_k = static_cast<const uint4*>(dev[0]);
    p.src_v = static_cast<const uint4*>(dev[1]);
    p.dst_k = static_cast<uint4*>(const_cast<void*>(dev[2]));
    p.dst_v = static_cast<uint4*>(const_cast<void*>(dev[3]));
    p.src_blocks = static_cast<const int32_t*>(dev[4]);
    p.dst_blocks = static_cast<const int32_t*>(dev[5]);
    p.dev_err = dev_err;
    p.block_vecs = (long long)D.Hkv * kBlock * D.head_dim * 2 / 16;
    p.src_num_blocks = src_num_blocks;
    p.dst_num_blocks = dst_num_blocks;
    p.n = n;
    return launch_pdl(copy_blocks_kernel, 2 * n, kCopyThreads, 0, (cudaStream_t)stream, p) == cudaSuccess
               ? MI_OK
               : MI_ERR_CUDA;
}

extern "C" mi_status mi_kv_copy_rows(const void* src, int64_t src_count, const int32_t* src_ids, void* dst,
                                     int64_t dst_count, const int32_t* dst_ids, int32_t n, int64_t row_bytes,
                                     int32_t* dev_err, mi_stream_t stream) {
    using namespace mi;
    if (n < 0 || src_count < 1 || dst_count < 1 || row_bytes < 4 || row_bytes % 4 != 0) return MI_ERR_INVALID_ARG;
    if (n == 0) return MI_OK;
    if (!src || !dst || !src_ids || !dst_ids) return MI_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 3u) return MI_ERR_INVALID_ARG;
    const void* ptrs[4] = {src, dst, src_ids, dst_ids};
    const void* dev[4];
    for (int i = 0; i < 4; ++i)
        if (!(dev[i] = device_alias(ptrs[i]))) return MI_ERR_INVALID_ARG;
    RowParams p;
    p.src = dev[0];
    p.dst = const_cast<void*>(dev[1]);
    p.src_ids = static_cast<const int32_t*>(dev[2]);
    p.dst_ids = static_cast<const int32_t*>(dev[3]);
    p.dev_err = dev_err;
    p.src_count = src_count;
    p.dst_count = dst_count;
    p.n = n;
    const bool vec16 = row_bytes % 16 == 0 && aligned16(dev[0]) && aligned16(dev[1]);
    p.row_units = row_bytes / (vec16 ? 16 : 4);
    const cudaError_t e = vec16 ? launch_pdl(copy_rows_kernel<uint4>, n, kCopyThreads, 0, (cudaStream_t)stream, p)
                                : launch_pdl(copy_rows_kernel<uint32_t>, n, kCopyThreads, 0, (cudaStream_t)stream, p);
    return e == cudaSuccess ? MI_OK : MI_ERR_CUDA;
}
