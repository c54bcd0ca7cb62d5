// pkv_dequant.cu -- quantised pages of a batch's requests expanded to bf16, for prefill.
//
// Prefill over E4M3, int8 or int4 pages ("ai-infra-7", 优化三 传输量化 and 优化五 KV 本体
// 压缩: KV kept at low precision) reuses the bf16 tensor-core prefill.  This pass writes
// every cached page of the batch, value = code * scale[block][head] rounded to bf16, into
// a dense workspace pool in request order (request r, logical block j -> pool block
// r * MB + j) and fills an identity block table for it.  Prefill is compute-bound and
// reads each page many times, so one extra bandwidth-bound pass over the pages is cheap.
//
// One thread writes one 16-byte output chunk (8 bf16 values) of one page row.
#include <cuda_fp8.h>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

// 8 codes of page kind KT at `src` (8 bytes for E4M3 / int8, 4 bytes for int4) times
// `scale`, as 8 bf16 (round to nearest even) packed in a uint4.
template <int KT>
__device__ __forceinline__ uint4 dequant8(const uint8_t* src, float scale) {
    float v[8];
    if constexpr (KT == 3) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (float)((int)((w >> (4 * e)) & 0xFu) - 8) * scale;
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(src);
        const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t b = (ws[e >> 2] >> (8 * (e & 3))) & 0xFFu;
            if constexpr (KT == 2) {
                v[e] = (float)(int8_t)b * scale;
            } else {
                __nv_fp8_e4m3 f;
                f.__x = (__nv_fp8_storage_t)b;
                v[e] = (float)f * scale;
            }
        }
    }
    uint4 o;
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    o.z = pack_bf16x2(v[4], v[5]);
    o.w = pack_bf16x2(v[6], v[7]);
    return o;
}

}  // namespace

template <int KT>
__global__ void __launch_bounds__(256)
    pkv_dequant_pages_kernel(const uint8_t* __restrict__ k_cache, const uint8_t* __restrict__ v_cache,
                             const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                             const int32_t* __restrict__ block_table, const int32_t* __restrict__ seq_lens,
                             int N, int MB, int NB, int Hkv, int BS, int D, uint16_t* __restrict__ kout,
                             uint16_t* __restrict__ vout, int32_t* __restrict__ bt_out,
                             uint32_t* __restrict__ err) {
    pdl_launch_dependents();
    pdl_wait();
    const int chunks_per_page = BS * (D / 8);
    const int64_t per_block = (int64_t)Hkv * chunks_per_page;
    const int64_t total = (int64_t)N * MB * per_block;
    // identity table of the pool (a grid-stride pass over N * MB entries)
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)N * MB;
         i += (int64_t)gridDim.x * blockDim.x)
        bt_out[i] = (int32_t)i;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pb = idx / per_block;                 // pool block = r * MB + j
        const int rem = (int)(idx - pb * per_block);
        const int h = rem / chunks_per_page;
        const int c = rem - h * chunks_per_page;
        const int t = c / (D / 8);                          // token row in the page
        const int k8 = c - t * (D / 8);                     // 8-value chunk in the row
        const int r = (int)(pb / MB);
        const int j = (int)(pb - (int64_t)r * MB);
        int seq = seq_lens[r];
        if (seq > MB * BS) seq = MB * BS;
        if (j * BS >= seq) continue;                        // page past the request
        const int64_t orow = ((pb * Hkv + h) * BS + t) * D + k8 * 8;
        const int blk = block_table[(int64_t)r * MB + j];
        if (blk < 0 || blk >= NB) {
            if (err != nullptr && h == 0 && t == 0 && k8 == 0) atomicOr(err, PKV_DEVERR_BLOCK_RANGE);
            *reinterpret_cast<uint4*>(kout + orow) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(vout + orow) = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        const int64_t srow = (((int64_t)blk * Hkv + h) * BS + t) * D + k8 * 8;   // element index
        const int64_t sb = KT == 3 ? srow / 2 : srow;                             // byte index
        const float ks = k_scale[(int64_t)blk * Hkv + h], vs = v_scale[(int64_t)blk * Hkv + h];
        *reinterpret_cast<uint4*>(kout + orow) = dequant8<KT>(k_cache + sb, ks);
        *reinterpret_cast<uint4*>(vout + orow) = dequant8<KT>(v_cache + sb, vs);
    }
}

cudaError_t dequant_pages_launch(const void* k_cache, const void* v_cache, const float* k_scale,
                                 const float* v_scale, const int32_t* block_table,
                                 const int32_t* seq_lens, int N, int MB, int NB, int Hkv, int BS,
                                 int D, int kt, void* kout, void* vout, int32_t* bt_out,
                                 uint32_t* err, int num_sms, cudaStream_t st) {
    const int64_t total = (int64_t)N * MB * Hkv * BS * (D / 8);
    int64_t grid = (total + 255) / 256;
    if (grid > (int64_t)num_sms * 16) grid = (int64_t)num_sms * 16;
    if (grid < 1) grid = 1;
    const uint8_t* kc = static_cast<const uint8_t*>(k_cache);
    const uint8_t* vc = static_cast<const uint8_t*>(v_cache);
    uint16_t* ko = static_cast<uint16_t*>(kout);
    uint16_t* vo = static_cast<uint16_t*>(vout);
    if (kt == 1)
        return launch_pdl(pkv_dequant_pages_kernel<1>, dim3((unsigned)grid), dim3(256), 0, st, kc,
                          vc, k_scale, v_scale, block_table, seq_lens, N, MB, NB, Hkv, BS, D, ko,
                          vo, bt_out, err);
    if (kt == 2)
        return launch_pdl(pkv_dequant_pages_kernel<2>, dim3((unsigned)grid), dim3(256), 0, st, kc,
                          vc, k_scale, v_scale, block_table, seq_lens, N, MB, NB, Hkv, BS, D, ko,
                          vo, bt_out, err);
    return launch_pdl(pkv_dequant_pages_kernel<3>, dim3((unsigned)grid), dim3(256), 0, st, kc, vc,
                      k_scale, v_scale, block_table, seq_lens, N, MB, NB, Hkv, BS, D, ko, vo,
                      bt_out, err);
}

}  // namespace pkv
