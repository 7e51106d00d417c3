// mi_paged_decode_attention_noalloc: paged decode attention for callers that
// cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a plugin whose host
// framework owns every device allocation and hands out no scratch, a serving
// loop that forbids allocator calls because cudaMalloc can synchronise the
// device and stall it, or a process that runs under a fixed device-memory
// budget set at start-up. For them the attention's split-KV workspace lives in
// a fixed array in this library's own device memory instead of a caller
// buffer. The caller still passes every input and output.
#include <cuda_runtime.h>

#include <mutex>

#include "mi.h"
#include "tma.cuh"

namespace {

// Loaded with the library on every GPU that runs it and kept until the
// process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MI_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;

// Device address of the array, looked up with the device current on the
// first call there and again whenever the device's context has changed (a
// device reset gives the array a new address). In host code
// `g_noalloc_scratch` names a host-side stand-in, never the device memory,
// so only the looked-up address is passed on.
void* scratch_on_current_device(mi_status* st) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    static CUcontext ctx_of[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *st = MI_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    const CUcontext ctx = mi::current_context();
    if (!addr[dev] || !ctx || ctx != ctx_of[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            *st = MI_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
        ctx_of[dev] = mi::current_context();  // current now, if it was not before the lookup
    }
    *st = MI_OK;
    return addr[dev];
}

}  // namespace

extern "C" mi_status mi_paged_decode_attention_noalloc(const mi_dims* dims, const void* q,
                                                       const void* k_cache, const void* v_cache,
                                                       const int32_t* block_tables,
                                                       const int32_t* context_lens, float scale,
                                                       void* out, int32_t* dev_err, mi_stream_t stream) {
    if (!dims) return MI_ERR_INVALID_ARG;
    if (dims->B == 0) return MI_OK;
    const size_t need = mi_paged_decode_workspace_bytes(dims);
    if (need == 0) return MI_ERR_UNSUPPORTED;             // shape not built, or no usable device
    if (need > (size_t)MI_NOALLOC_SCRATCH_BYTES) return MI_ERR_UNSUPPORTED;  // beyond the fixed array
    mi_status st = MI_OK;
    void* ws = scratch_on_current_device(&st);
    if (!ws) return st;
    return mi_paged_decode_attention(dims, q, k_cache, v_cache, block_tables, context_lens, scale, out, ws,
                                     (size_t)MI_NOALLOC_SCRATCH_BYTES, dev_err, stream);
}
