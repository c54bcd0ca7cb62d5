// pkv_write.cu -- slot mapping and paged KV cache write (reshape_and_cache).
//
// Slot mapping ("深入LLM推理：从KV Cache到PD分离的Serving全景解析",
// "PagedAttention与Cache管理"): token at position pos of request r lives in
// physical block block_table[r][pos / BS] at offset pos % BS.
// Cache write ("ai-infra-7", "组合拳：一次请求的完整旅程": new K/V go back into
// the cache pool; FP8 storage per "优化三：KV 传输优化", 传输量化).
//
// The write is a pure copy (bf16) or a per-element quantisation (E4M3): one
// thread moves one 16-byte chunk (8 elements) of a (token, head) row, so a
// row of D=128 bf16 is 16 coalesced 16-byte loads and stores.
#include <cuda_fp8.h>

#include "pkv_internal.cuh"

namespace pkv {

__global__ void __launch_bounds__(256)
    pkv_slot_mapping_kernel(const int32_t* __restrict__ block_table, int MB,
                            const int32_t* __restrict__ req_idx,
                            const int32_t* __restrict__ positions, int T, int BS,
                            int64_t* __restrict__ slot_mapping) {
    pdl_launch_dependents();
    pdl_wait();   // inputs may come from the previous kernel in the stream
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int r = req_idx ? req_idx[t] : t;
    const int pos = positions[t];
    int64_t slot = -1;
    if (pos >= 0) {
        const int lb = pos / BS;
        if (lb < MB) slot = (int64_t)block_table[(int64_t)r * MB + lb] * BS + (pos - lb * BS);
    }
    slot_mapping[t] = slot;
}

template <bool FP8>
__global__ void __launch_bounds__(256)
    pkv_cache_write_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                           const int64_t* __restrict__ slot_mapping, int64_t total_chunks,
                           int Hkv, int D, int BS, int NB, uint8_t* __restrict__ k_cache,
                           uint8_t* __restrict__ v_cache, const float* __restrict__ k_scale,
                           const float* __restrict__ v_scale) {
    pdl_launch_dependents();
    pdl_wait();   // slots and rows may come from the previous kernel in the stream
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total_chunks) return;
    const int cpr = D / 8;                       // 16-byte source chunks per row
    const int64_t row = idx / cpr;               // (token, head)
    const int chunk = (int)(idx - row * cpr);
    const int64_t t = row / Hkv;
    const int h = (int)(row - t * Hkv);
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;
    const int64_t blk = slot / BS;
    if (blk >= NB) return;
    const int64_t off = slot - blk * BS;
    const int64_t dst_row = (blk * Hkv + h) * BS + off;   // cache row index
    const uint4 ks = *reinterpret_cast<const uint4*>(k + row * D + chunk * 8);
    const uint4 vs = *reinterpret_cast<const uint4*>(v + row * D + chunk * 8);
    if (!FP8) {
        *reinterpret_cast<uint4*>(k_cache + (dst_row * D + chunk * 8) * 2) = ks;
        *reinterpret_cast<uint4*>(v_cache + (dst_row * D + chunk * 8) * 2) = vs;
    } else {
        const float ksc = k_scale[blk * Hkv + h];
        const float vsc = v_scale[blk * Hkv + h];
        const uint32_t kw[4] = {ks.x, ks.y, ks.z, ks.w};
        const uint32_t vw[4] = {vs.x, vs.y, vs.z, vs.w};
        uint32_t ko[2], vo[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            // IEEE binary32 division (round to nearest), then E4M3 RNE + saturate
            const uint16_t k01 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo_to_f32(kw[2 * p]), ksc),
                                                 __fdiv_rn(bf16_hi_to_f32(kw[2 * p]), ksc));
            const uint16_t k23 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo_to_f32(kw[2 * p + 1]), ksc),
                                                 __fdiv_rn(bf16_hi_to_f32(kw[2 * p + 1]), ksc));
            const uint16_t v01 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo_to_f32(vw[2 * p]), vsc),
                                                 __fdiv_rn(bf16_hi_to_f32(vw[2 * p]), vsc));
            const uint16_t v23 = f32x2_to_e4m3x2(__fdiv_rn(bf16_lo_to_f32(vw[2 * p + 1]), vsc),
                                                 __fdiv_rn(bf16_hi_to_f32(vw[2 * p + 1]), vsc));
            ko[p] = (uint32_t)k01 | ((uint32_t)k23 << 16);
            vo[p] = (uint32_t)v01 | ((uint32_t)v23 << 16);
        }
        *reinterpret_cast<uint2*>(k_cache + dst_row * D + chunk * 8) = make_uint2(ko[0], ko[1]);
        *reinterpret_cast<uint2*>(v_cache + dst_row * D + chunk * 8) = make_uint2(vo[0], vo[1]);
    }
}

cudaError_t slot_mapping_launch(const int32_t* block_table, int MB, const int32_t* req_idx,
                                const int32_t* positions, int T, int BS, int64_t* out,
                                cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    return launch_pdl(pkv_slot_mapping_kernel, dim3((T + 255) / 256), dim3(256), 0, st,
                      block_table, MB, req_idx, positions, T, BS, out);
}

cudaError_t cache_write_launch(const void* k, const void* v, const int64_t* slots, int T,
                               int Hkv, int D, int BS, int NB, int fp8, void* k_cache,
                               void* v_cache, const float* k_scale, const float* v_scale,
                               cudaStream_t st) {
    const int64_t chunks = (int64_t)T * Hkv * (D / 8);
    if (chunks == 0) return cudaSuccess;
    const int64_t grid = (chunks + 255) / 256;
    const uint16_t* kk = static_cast<const uint16_t*>(k);
    const uint16_t* vv = static_cast<const uint16_t*>(v);
    uint8_t* kc = static_cast<uint8_t*>(k_cache);
    uint8_t* vc = static_cast<uint8_t*>(v_cache);
    if (fp8)
        return launch_pdl(pkv_cache_write_kernel<true>, dim3((unsigned)grid), dim3(256), 0, st, kk,
                          vv, slots, chunks, Hkv, D, BS, NB, kc, vc, k_scale, v_scale);
    return launch_pdl(pkv_cache_write_kernel<false>, dim3((unsigned)grid), dim3(256), 0, st, kk, vv,
                      slots, chunks, Hkv, D, BS, NB, kc, vc, (const float*)nullptr,
                      (const float*)nullptr);
}

}  // namespace pkv
