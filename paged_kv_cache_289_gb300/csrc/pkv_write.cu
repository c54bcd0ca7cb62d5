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

// Rescaling writes: every (block, head) that receives a row in this call gets
// scale = amax / QMAX over the |values| of those rows (QMAX 448 for E4M3, 127 for
// int8; NaN ignored; amax = 0 gives 1).  The amax is gathered in a workspace of
// uint32 float bit patterns: for non-negative floats the bit patterns order like
// unsigned integers, so atomicMax on the bits is a max on the values.
__global__ void __launch_bounds__(256)
    pkv_rescale_zero_kernel(const int64_t* __restrict__ slot_mapping, int64_t rows, int Hkv,
                            int BS, int NB, uint32_t* __restrict__ kmax,
                            uint32_t* __restrict__ vmax) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // (token, head)
    if (idx >= rows) return;
    const int64_t t = idx / Hkv;
    const int h = (int)(idx - t * Hkv);
    const int64_t slot = slot_mapping[t];
    if (slot < 0 || slot / BS >= NB) return;
    kmax[(slot / BS) * Hkv + h] = 0u;
    vmax[(slot / BS) * Hkv + h] = 0u;
}

__device__ __forceinline__ float absmax8(const uint4 w) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = fabsf(bf16_lo_to_f32(ws[i])), b = fabsf(bf16_hi_to_f32(ws[i]));
        if (a == a) m = fmaxf(m, a);   // NaN compares unequal and is skipped
        if (b == b) m = fmaxf(m, b);
    }
    return m;
}

__global__ void __launch_bounds__(256)
    pkv_rescale_amax_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                            const int64_t* __restrict__ slot_mapping, int64_t total_chunks,
                            int Hkv, int D, int BS, int NB, uint32_t* __restrict__ kmax,
                            uint32_t* __restrict__ vmax) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total_chunks) return;
    const int cpr = D / 8;
    const int64_t row = idx / cpr;
    const int chunk = (int)(idx - row * cpr);
    const int64_t t = row / Hkv;
    const int h = (int)(row - t * Hkv);
    const int64_t slot = slot_mapping[t];
    if (slot < 0 || slot / BS >= NB) return;
    const int64_t i = (slot / BS) * Hkv + h;
    const float km = absmax8(*reinterpret_cast<const uint4*>(k + row * D + chunk * 8));
    const float vm = absmax8(*reinterpret_cast<const uint4*>(v + row * D + chunk * 8));
    if (km > 0.f) atomicMax(kmax + i, __float_as_uint(km));
    if (vm > 0.f) atomicMax(vmax + i, __float_as_uint(vm));
}

// The K and V scale of cache entry i: read, or (RESCALE) derived from the gathered
// amax with a binary32 divide and stored by the row's first chunk.
template <int KT, bool RESCALE>
__device__ __forceinline__ void block_scales(int64_t i, int chunk, float* k_scale, float* v_scale,
                                             const uint32_t* kmax, const uint32_t* vmax,
                                             float& ksc, float& vsc) {
    if constexpr (!RESCALE) {
        ksc = k_scale[i];
        vsc = v_scale[i];
    } else {
        constexpr float QMAX = KT == 3 ? 7.f : (KT == 2 ? 127.f : 448.f);
        const float ka = __uint_as_float(kmax[i]), va = __uint_as_float(vmax[i]);
        ksc = ka > 0.f ? __fdiv_rn(ka, QMAX) : 1.f;
        vsc = va > 0.f ? __fdiv_rn(va, QMAX) : 1.f;
        if (chunk == 0) {   // every row of the block stores the same value
            k_scale[i] = ksc;
            v_scale[i] = vsc;
        }
    }
}

// KT: 0 bf16 copy, 1 E4M3 (RNE, saturate to +-448), 2 int8 (RNE, clamp to +-127),
// 3 int4 (RNE, clamp to +-7, stored offset-binary q + 8: value 2b in the low nibble of
// byte b of the row, value 2b+1 in its high nibble).
// RESCALE: the block scales come from the gathered amax (and are stored), else
// they are read from k_scale / v_scale.
template <int KT, bool RESCALE = false>
__global__ void __launch_bounds__(256)
    pkv_cache_write_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                           const int64_t* __restrict__ slot_mapping, int64_t total_chunks,
                           int Hkv, int D, int BS, int NB, uint8_t* __restrict__ k_cache,
                           uint8_t* __restrict__ v_cache, float* __restrict__ k_scale,
                           float* __restrict__ v_scale, const uint32_t* __restrict__ kmax = nullptr,
                           const uint32_t* __restrict__ vmax = nullptr) {
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
    if constexpr (KT == 0) {
        *reinterpret_cast<uint4*>(k_cache + (dst_row * D + chunk * 8) * 2) = ks;
        *reinterpret_cast<uint4*>(v_cache + (dst_row * D + chunk * 8) * 2) = vs;
    } else if constexpr (KT == 3) {
        float ksc, vsc;
        block_scales<KT, RESCALE>(blk * Hkv + h, chunk, k_scale, v_scale, kmax, vmax, ksc, vsc);
        const uint32_t kw[4] = {ks.x, ks.y, ks.z, ks.w};
        const uint32_t vw[4] = {vs.x, vs.y, vs.z, vs.w};
        uint32_t ko = 0u, vo = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t kb = (e & 1) ? (kw[e >> 1] & 0xFFFF0000u) : (kw[e >> 1] << 16);
            const uint32_t vb = (e & 1) ? (vw[e >> 1] & 0xFFFF0000u) : (vw[e >> 1] << 16);
            // IEEE binary32 division, round to nearest even, clamp to +-7 (NaN gives 0)
            const int kq = min(max(__float2int_rn(__fdiv_rn(__uint_as_float(kb), ksc)), -7), 7);
            const int vq = min(max(__float2int_rn(__fdiv_rn(__uint_as_float(vb), vsc)), -7), 7);
            ko |= (uint32_t)(kq + 8) << (4 * e);
            vo |= (uint32_t)(vq + 8) << (4 * e);
        }
        *reinterpret_cast<uint32_t*>(k_cache + (dst_row * D + chunk * 8) / 2) = ko;
        *reinterpret_cast<uint32_t*>(v_cache + (dst_row * D + chunk * 8) / 2) = vo;
    } else if constexpr (KT == 2) {
        float ksc, vsc;
        block_scales<KT, RESCALE>(blk * Hkv + h, chunk, k_scale, v_scale, kmax, vmax, ksc, vsc);
        const uint32_t kw[4] = {ks.x, ks.y, ks.z, ks.w};
        const uint32_t vw[4] = {vs.x, vs.y, vs.z, vs.w};
        uint32_t ko[2] = {0u, 0u}, vo[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t kb = (e & 1) ? (kw[e >> 1] & 0xFFFF0000u) : (kw[e >> 1] << 16);
            const uint32_t vb = (e & 1) ? (vw[e >> 1] & 0xFFFF0000u) : (vw[e >> 1] << 16);
            // IEEE binary32 division, round to nearest even, clamp to +-127
            const int kq = min(max(__float2int_rn(__fdiv_rn(__uint_as_float(kb), ksc)), -127), 127);
            const int vq = min(max(__float2int_rn(__fdiv_rn(__uint_as_float(vb), vsc)), -127), 127);
            ko[e >> 2] |= ((uint32_t)kq & 0xFFu) << (8 * (e & 3));
            vo[e >> 2] |= ((uint32_t)vq & 0xFFu) << (8 * (e & 3));
        }
        *reinterpret_cast<uint2*>(k_cache + dst_row * D + chunk * 8) = make_uint2(ko[0], ko[1]);
        *reinterpret_cast<uint2*>(v_cache + dst_row * D + chunk * 8) = make_uint2(vo[0], vo[1]);
    } else {
        float ksc, vsc;
        block_scales<KT, RESCALE>(blk * Hkv + h, chunk, k_scale, v_scale, kmax, vmax, ksc, vsc);
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
                               int Hkv, int D, int BS, int NB, int kt, void* k_cache,
                               void* v_cache, const float* k_scale, const float* v_scale,
                               cudaStream_t st) {
    const int64_t chunks = (int64_t)T * Hkv * (D / 8);
    if (chunks == 0) return cudaSuccess;
    const int64_t grid = (chunks + 255) / 256;
    const uint16_t* kk = static_cast<const uint16_t*>(k);
    const uint16_t* vv = static_cast<const uint16_t*>(v);
    uint8_t* kc = static_cast<uint8_t*>(k_cache);
    uint8_t* vc = static_cast<uint8_t*>(v_cache);
    const uint32_t* nz = nullptr;
    float* ks = const_cast<float*>(k_scale);   // read only without RESCALE
    float* vs = const_cast<float*>(v_scale);
    if (kt == 1)
        return launch_pdl(pkv_cache_write_kernel<1, false>, dim3((unsigned)grid), dim3(256), 0, st,
                          kk, vv, slots, chunks, Hkv, D, BS, NB, kc, vc, ks, vs, nz, nz);
    if (kt == 2)
        return launch_pdl(pkv_cache_write_kernel<2, false>, dim3((unsigned)grid), dim3(256), 0, st,
                          kk, vv, slots, chunks, Hkv, D, BS, NB, kc, vc, ks, vs, nz, nz);
    if (kt == 3)
        return launch_pdl(pkv_cache_write_kernel<3, false>, dim3((unsigned)grid), dim3(256), 0, st,
                          kk, vv, slots, chunks, Hkv, D, BS, NB, kc, vc, ks, vs, nz, nz);
    return launch_pdl(pkv_cache_write_kernel<0, false>, dim3((unsigned)grid), dim3(256), 0, st, kk,
                      vv, slots, chunks, Hkv, D, BS, NB, kc, vc, (float*)nullptr, (float*)nullptr,
                      nz, nz);
}

cudaError_t cache_write_rescale_launch(const void* k, const void* v, const int64_t* slots, int T,
                                       int Hkv, int D, int BS, int NB, int kt, void* k_cache,
                                       void* v_cache, float* k_scale, float* v_scale,
                                       void* workspace, cudaStream_t st) {
    const int64_t chunks = (int64_t)T * Hkv * (D / 8);
    if (chunks == 0) return cudaSuccess;
    uint32_t* kmax = static_cast<uint32_t*>(workspace);
    uint32_t* vmax = kmax + (int64_t)NB * Hkv;
    const uint16_t* kk = static_cast<const uint16_t*>(k);
    const uint16_t* vv = static_cast<const uint16_t*>(v);
    uint8_t* kc = static_cast<uint8_t*>(k_cache);
    uint8_t* vc = static_cast<uint8_t*>(v_cache);
    const int64_t rows = (int64_t)T * Hkv;
    cudaError_t e = launch_pdl(pkv_rescale_zero_kernel, dim3((unsigned)((rows + 255) / 256)),
                               dim3(256), 0, st, slots, rows, Hkv, BS, NB, kmax, vmax);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((chunks + 255) / 256);
    e = launch_pdl(pkv_rescale_amax_kernel, dim3(grid), dim3(256), 0, st, kk, vv, slots, chunks,
                   Hkv, D, BS, NB, kmax, vmax);
    if (e != cudaSuccess) return e;
    const uint32_t* ckm = kmax;
    const uint32_t* cvm = vmax;
    if (kt == 2)
        return launch_pdl(pkv_cache_write_kernel<2, true>, dim3(grid), dim3(256), 0, st, kk, vv,
                          slots, chunks, Hkv, D, BS, NB, kc, vc, k_scale, v_scale, ckm, cvm);
    if (kt == 3)
        return launch_pdl(pkv_cache_write_kernel<3, true>, dim3(grid), dim3(256), 0, st, kk, vv,
                          slots, chunks, Hkv, D, BS, NB, kc, vc, k_scale, v_scale, ckm, cvm);
    return launch_pdl(pkv_cache_write_kernel<1, true>, dim3(grid), dim3(256), 0, st, kk, vv, slots,
                      chunks, Hkv, D, BS, NB, kc, vc, k_scale, v_scale, ckm, cvm);
}

}  // namespace pkv
