// pkv_internal.cuh -- device helpers shared by the libpagedkv kernels (sm_103a).
//
// Thin inline-PTX wrappers: mbarrier waits with a time limit, bulk tensor
// copies (TMA), ldmatrix / movmatrix, mma.sync m16n8k16 and the fp8/fp16/bf16
// packs.  No math library internals are re-implemented here: exponentials use
// the CUDA exp2f function and conversions use the hardware cvt instructions.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// ---------------------------------------------------------------- launch plan
// The decode kernel's CTA shape for one (dtype, head_dim, block_size).  Chosen
// on the host; the same numbers size the workspace.
struct DecodePlan {
    int warps;          // independent consumer warps per CTA (each its own pipeline)
    int stages;         // pages in flight per warp
    int ctas_per_sm;    // resident CTAs per SM (persistent grid = SMs * ctas_per_sm)
    int stage_bytes;    // K page + V page of one (block, head)
    int smem_bytes;     // dynamic shared memory per CTA
    int total_warps;    // grid warps = W
};

constexpr int kGroupPad = 8;                 // query heads per GQA group padded to mma N = 8
constexpr int kMaxBatch = 16384;             // requests (page-prefix table lives in smem)
constexpr uint32_t kWorkspaceHeader = 256;   // error word + reserved

__host__ __device__ inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Byte offsets inside the decode workspace.
struct WorkspaceLayout {
    int64_t prefix_off;    // int32 [N + 1] page prefix over requests (times Hkv)
    int64_t partial_off;   // fp32 [slots][QT][kGroupPad][D + 4]: o[D], m, l, pad
    int64_t slots;         // N * Hkv + W
    int64_t total;
};

__host__ __device__ inline WorkspaceLayout workspace_layout(int batch, int num_kv_heads,
                                                            int head_dim, int total_warps,
                                                            int qt) {
    WorkspaceLayout L;
    L.prefix_off = kWorkspaceHeader;
    L.partial_off = align_up(L.prefix_off + 4 * (int64_t)(batch + 1), 256);
    L.slots = (int64_t)batch * num_kv_heads + total_warps;
    L.total = L.partial_off + L.slots * qt * kGroupPad * (head_dim + 4) * 4;
    return L;
}

// ---------------------------------------------------------------- host launchers
struct DecodeLaunch {
    const void* q;
    const int32_t* q_offsets;   // null: one query per request
    int max_q_len;
    const void* k_cache;
    const void* v_cache;
    const float* k_scale;
    const float* v_scale;
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* out;
    void* workspace;
    int N, Hq, Hkv, D, BS, MB, NB, fp8;   // fp8: any quantised page kind (E4M3, int8, int4)
    int kt;                               // page kind: 0 bf16, 1 E4M3, 2 int8, 3 int4
    float scale;
    int num_sms;
    // shared-prefix decode (one query position): the first skip_blocks blocks are left
    // to the prefix pass whose partials cascade_part holds, cascade_split per row
    int skip_blocks = 0;
    const float* cascade_part = nullptr;
    int cascade_split = 0;
    // append (bf16, one query): the newest token's K/V rows [N][Hkv][D], written by the
    // decode kernel into the cache and used in place of the page's stored row
    const void* k_new = nullptr;
    const void* v_new = nullptr;
    // when set, the merge waits for this event (recorded after work on another stream
    // whose results it reads, e.g. a prefix pass run beside the decode)
    cudaEvent_t merge_after = nullptr;
};

int query_tile(int fp8, int max_q_len);
DecodePlan decode_plan(int kt, int head_dim, int block_size, int num_sms, int batch, int qt);
int decode_launch(const DecodeLaunch& L, cudaStream_t st);
size_t decode_workspace_bytes(int batch, int num_kv_heads, int head_dim, int block_size, int kt,
                              int num_sms, int max_q_len);
cudaError_t slot_mapping_launch(const int32_t* block_table, int MB, const int32_t* req_idx,
                                const int32_t* positions, int T, int BS, int64_t* out,
                                cudaStream_t st);
cudaError_t cache_write_launch(const void* k, const void* v, const int64_t* slots, int T,
                               int Hkv, int D, int BS, int NB, int kt, void* k_cache,
                               void* v_cache, const float* k_scale, const float* v_scale,
                               cudaStream_t st);
cudaError_t cache_write_rescale_launch(const void* k, const void* v, const int64_t* slots, int T,
                                       int Hkv, int D, int BS, int NB, int kt, void* k_cache,
                                       void* v_cache, float* k_scale, float* v_scale,
                                       void* workspace, cudaStream_t st);
// prev_hashes / first_blocks == nullptr: the full chain from seed; else resumed
cudaError_t prefix_hash_launch(const int32_t* tokens, const int64_t* offsets, int num_seqs, int B,
                               uint64_t seed, const uint64_t* prev_hashes,
                               const int64_t* first_blocks, uint64_t* hashes,
                               const int64_t* hash_offsets, cudaStream_t st);
struct PrefillLaunch {
    const void* q;
    const int32_t* q_offsets;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* out;
    uint32_t* err;                     // device error word, may be null
    int total_q, max_q_len, N, Hq, Hkv, D, BS, MB, NB;
    float scale;
    // shared-prefix mode: the total_q rows all see block-table row 0's first prefix_len
    // tokens, split in prefix_split chunks of chunk_tokens; partials go to part
    int prefix_split = 0, prefix_len = 0, chunk_tokens = 0;
    float* part = nullptr;
};
bool prefill_shape_supported(int Hq, int Hkv, int D, int BS, int dtype);
cudaError_t dequant_pages_launch(const void* k_cache, const void* v_cache, const float* k_scale,
                                 const float* v_scale, const int32_t* block_table,
                                 const int32_t* seq_lens, int N, int MB, int NB, int Hkv, int BS,
                                 int D, int kt, void* kout, void* vout, int32_t* bt_out,
                                 uint32_t* err, int num_sms, cudaStream_t st);
int prefill_launch(const PrefillLaunch& L, cudaStream_t st);
cudaError_t copy_blocks_launch(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                               const int32_t* mapping, int pairs, int64_t block_bytes, int NB,
                               int Hkv, int num_sms, cudaStream_t st);

// Launch `kern` as a programmatic dependent of the previous kernel in `st`: its CTAs
// may be dispatched while that kernel finishes, and the kernel itself calls
// griddepcontrol.wait before touching memory a predecessor may have written.  Falls
// back to an ordinary launch where the attribute is refused.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        kern<<<grid, block, smem, st>>>(args...);
        e = cudaGetLastError();
    }
    return e;
}

// ---------------------------------------------------------------- smem / sync
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns` of wall
// time (measured with %globaltimer).  Returns false on time-out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// 2-D tiled bulk tensor copy global -> shared, completion on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Same, with an L2 cache policy (evict-first for streamed pages).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x,
                                                 int y, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: let the next kernel in the stream start launching,
// and (in that kernel) wait until the kernels it depends on have completed and their
// memory is visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- fragments
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Transpose an 8x8 matrix of 16-bit elements held one row-pair per thread.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with fp16 inputs.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 bytes (low 16 bits of x, low byte first) -> fp16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x) {
    uint32_t y;
    asm volatile(
        "{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(y)
        : "r"(x));
    return y;
}

// Two int8 (low 16 bits of x, low byte first) -> fp16x2, exactly.  fp16 holds
// 1024 + k exactly for integers 0 <= k < 1024 (exponent of 1024, k in the
// mantissa), so q + 128 is placed under that exponent and 1152 subtracted.
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t x) {
    const uint32_t y = __byte_perm(x ^ 0x8080u, 0x64646464u, 0x5140);
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(y), "r"(0x64806480u));
    return r;
}

// Two int8 codes picked from the 4 bytes of xs by a byte-permute selector SEL (low pair
// first), where xs is x with its sign bits flipped (x ^ 0x80808080, so byte = code + 128):
// the permute gathers and widens at once, to fp16 (1024 + code + 128) per half.  fp16
// 1024 + k (k < 1024) is the exponent of 1024 with k in the mantissa.  The offset 1152 is
// left in: a caller subtracts it once per sum.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t i8pick_raw(uint32_t xs) {
    return __byte_perm(xs, 0x64646464u, SEL);
}

// Two int4 codes picked from the 8 offset-binary nibbles n0..n7 of x (n_j at bits
// 4j..4j+3, n = code + 8), pairing nibbles (I, I + 4): the mask-or places nibble n
// directly in the mantissa of 1024 (I even, giving 1024 + n) or 16 n (I odd, giving
// 1024 + 16 n).  The offsets are left in: a caller prescales q by 1/16 for odd picks
// and subtracts the constant part once per sum.
template <int I>
__device__ __forceinline__ uint32_t i4pick_raw(uint32_t x) {
    const uint32_t w = (I >= 2) ? (x >> 8) : x;
    return ((I & 1) ? (w & 0x00F000F0u) : (w & 0x000F000Fu)) | 0x64006400u;
}

// The same picks as fp16 subnormals: the nibble (I even) or 16 x the nibble (I odd) is
// the whole mantissa under a zero exponent, so each half is n * 2^-24 or 16 n * 2^-24
// exactly, with no 1024 offset.  A sum over many of them keeps only the small offset of
// the offset-binary code (8 per unit of the weights), so it can run across pages in one
// fp32 accumulator without a large constant to cancel at the end.
template <int I>
__device__ __forceinline__ uint32_t i4pick_sub(uint32_t x) {
    const uint32_t w = (I >= 2) ? (x >> 8) : x;
    return (I & 1) ? (w & 0x00F000F0u) : (w & 0x000F000Fu);
}

// Two sign-flipped int8 codes (byte = code + 128) picked by SEL as fp16 subnormals:
// (code + 128) * 2^-24 per half, the high byte of each half zero.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t i8pick_sub(uint32_t xs) {
    return __byte_perm(xs, 0u, SEL);
}

// Two 8-bit cache codes -> fp16x2 for page kind KT (1 = E4M3, 2 = int8).
template <int KT>
__device__ __forceinline__ uint32_t b8x2_to_f16x2(uint32_t x) {
    if constexpr (KT == 2) return i8x2_to_f16x2(x);
    else return e4m3x2_to_f16x2(x);
}

// Two fp32 -> E4M3x2 with round-to-nearest-even and saturation to +-448;
// `lo` lands in the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t y;
    asm volatile("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(y) : "f"(hi), "f"(lo));
    return y;
}

// Two fp32 -> packed bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t y;
    asm volatile("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(y) : "f"(hi), "f"(lo));
    return y;
}

// Two fp32 -> packed fp16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t y;
    asm volatile("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(y) : "f"(hi), "f"(lo));
    return y;
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero): one instruction;
// -inf gives +0.  Relative error about 2^-22; results below 2^-126 flush to zero, far
// below what a softmax weight relative to its running maximum contributes.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16_lo_to_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t x) {
    return __uint_as_float(x & 0xFFFF0000u);
}

}  // namespace pkv
