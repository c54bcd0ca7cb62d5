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

#include "pkv_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

// Shared scratch of every no-alloc call on a device.  In host code this name is
// only a stand-in for the device symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];   // device address of the array, per device

// Device address of the scratch on the current device; looked up on the first
// call made with that device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" PKV_API int pkv_paged_decode_attn_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_table, int max_blocks_per_seq,
    const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int cache_dtype, float scale, void* out,
    pkv_stream_t stream) {
    if (batch == 0) return PKV_OK;
    const size_t need = pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                  block_size, cache_dtype, 0);
    if (need == 0) return batch < 0 ? PKV_ERR_INVALID_ARG : PKV_ERR_UNSUPPORTED;
    if (need > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;   // beyond the static maximum
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
    return pkv_paged_decode_attn(q, k_cache, v_cache, k_scale, v_scale, block_table,
                                 max_blocks_per_seq, seq_lens, batch, num_q_heads, num_kv_heads,
                                 head_dim, block_size, num_blocks, cache_dtype, scale, out, scratch,
                                 kNoAllocScratchBytes, stream);
}
