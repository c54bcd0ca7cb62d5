// pkv_noalloc.cu -- paged decode attention for callers that cannot allocate.
//
// pkv_paged_decode_attn needs a caller-allocated workspace (the per-warp partial
// results of requests split across warps, and the page prefix table).  Some
// callers cannot allocate device memory at all: a plugin inside an engine that
// owns every byte of device memory and offers no workspace hook, or code on a
// latency-critical path that must not call cudaMalloc (it can synchronise the
// device).  For them this file keeps the scratch in a file-scope device array
// that is part of the library's module image: every GPU that loads the library
// holds these kNoAllocScratchBytes until the process exits.
//
// The entry point computes exactly what pkv_paged_decode_attn computes, with the
// same kernels and the same launch plan; it only substitutes the address of the
// static array for the workspace pointer.
#include <mutex>

#include <cuda.h>

#include "pkv_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

// Shared scratch of every no-alloc call on a device.  In host code this name is
// only a stand-in for the device symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*ctx_get_current_fn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (the library does not
// link libcuda directly); nullptr if the driver does not offer it.
ctx_get_current_fn ctx_get_current() {
    static ctx_get_current_fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<ctx_get_current_fn>(p);
    });
    return fn;
}

std::mutex g_mu;
struct ScratchSlot {
    CUcontext ctx;   // context the address was looked up in
    void* addr;      // device address of the array in that context
};
ScratchSlot g_slot[kMaxDevices];

// Device address of the scratch for the current device and context.  It is looked
// up on the first call made with that device current, and again whenever the
// device's current context differs from the one it was looked up in (after
// cudaDeviceReset the module is loaded anew and the old address is stale).
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    ctx_get_current_fn get = ctx_get_current();
    if (!get) return PKV_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchSlot& s = g_slot[dev];
    if (!ctx || !s.addr || s.ctx != ctx) {
        // the lookup also makes the device's primary context current when no
        // context was, so the context is read again after it
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return PKV_ERR_CUDA;
        s.ctx = ctx;
        s.addr = p;
    }
    *out = s.addr;
    return PKV_OK;
}

}  // namespace

extern "C" PKV_API int pkv_paged_decode_attn_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_table, int max_blocks_per_seq,
    const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int cache_dtype, float scale, void* out,
    pkv_stream_t stream) {
    int num_sms = 0;
    if (pkv_device_num_sms(&num_sms) != PKV_OK) return PKV_ERR_CUDA;
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                  block_size, cache_dtype, num_sms);
    if (batch <= 0 || need == 0) {
        // nothing to run, or arguments the workspace entry point refuses: it returns
        // the same status here, checked in the same order, before it would need a
        // workspace
        return pkv_paged_decode_attn(q, k_cache, v_cache, k_scale, v_scale, block_table,
                                     max_blocks_per_seq, seq_lens, batch, num_q_heads,
                                     num_kv_heads, head_dim, block_size, num_blocks, cache_dtype,
                                     scale, out, nullptr, 0, stream);
    }
    if (need > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;   // beyond the static maximum
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
    return pkv_paged_decode_attn(q, k_cache, v_cache, k_scale, v_scale, block_table,
                                 max_blocks_per_seq, seq_lens, batch, num_q_heads, num_kv_heads,
                                 head_dim, block_size, num_blocks, cache_dtype, scale, out, scratch,
                                 kNoAllocScratchBytes, stream);
}
