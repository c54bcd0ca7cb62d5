// pkv_prefill.cu -- paged prefill attention on the 5th-generation tensor cores.
//
// Prefill is the compute-bound phase: every prompt token is a query
// ("深入LLM推理：从KV Cache到PD分离的Serving全景解析", 推理的两阶段计算形态).  A chunk of
// q_len new tokens of request r (positions ctx .. ctx + q_len - 1, ctx = seq_len - q_len,
// their K/V already written to the pages) attends causally to the request's paged
// cache: query i sees positions 0 .. ctx + i ("KV Cache：Transformer的循环状态",
// causal mask; "PagedAttention与Cache管理", block table).
//
// One CTA = one 128-row query tile of one (request, KV head): 128 / G query tokens x
// the G query heads of the group, so every K/V tile staged in shared memory serves
// the whole GQA group.  Per 256-token KV tile:
//   S = Q K^T      tcgen05.mma, M = 128, N = 256, K = D; A (Q) and B (K) K-major in
//                  shared memory (128-byte swizzle), S in tensor memory (256 columns)
//   softmax        2 x 4 warps, one TMEM lane (= one query row) per thread, each
//                  warpgroup one half (128 columns) of every row: online max and sum in
//                  the log2 domain, P rounded to bf16 into its own tensor-memory columns
//   O += P V       tcgen05.mma, M = 128, N = D, A = P read from tensor memory and B = V
//                  (MN-major: the page rows are tokens, d contiguous), in two 128-token
//                  halves
// The softmax warps release S as soon as they have loaded it, so the next tile's
// Q K^T runs during this tile's softmax.  Warp roles: warps 0-7 softmax + epilogue,
// warp 8 K producer (and TMEM owner), warp 9 V producer, warp 10 the Q K^T issuer and
// warp 11 the P V issuer (lane 0 of each).  Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pkv_internal.cuh"

namespace pkv {

namespace {

constexpr int kRows = 128;        // query rows per tile (TMEM lanes)
constexpr int kKvTile = 256;      // tokens per K tile (and per score tile)
constexpr int kVHalf = 128;       // tokens per V half-tile
constexpr int kThreads = 384;     // 12 warps: 2 x 4 softmax; K producer, V producer, 2 MMA issuers
// Registers per thread after the start-up: the producer/MMA warpgroup gives registers
// back and the softmax warpgroups take them (setmaxnreg).  The block is launched with
// kThreads x (launch registers, 168 under the launch bounds); the split must fit in that.
constexpr int kRegsSoftmax = 216;
constexpr int kRegsOther = 56;
constexpr int kRegsSplit = 2 * 128 * kRegsSoftmax + 128 * kRegsOther;   // 62,464
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kColS = 0, kColP = 256, kColO = 384, kTmemCols = 512;

// ------------------------------------------------------------ tcgen05 wrappers
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: start, leading / stride byte offsets (16-byte
// units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulate, bf16 A and B, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Packed fp32 pairs (sm_100 family): one instruction does two fp32 FMAs or adds, each
// rounded as its scalar form would be.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t r, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// max of three (sm_100 family); like fmaxf, a NaN operand is ignored
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 32 consecutive fp32 columns of this thread's lane.  The load and its wait sit in
// one asm statement, so no use of the outputs can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 fp32 columns of this thread's lane in one load (+ its wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]),"=r"(r[1]),"=r"(r[2]),"=r"(r[3]),"=r"(r[4]),"=r"(r[5]),"=r"(r[6]),"=r"(r[7]),"=r"(r[8]),"=r"(r[9]),"=r"(r[10]),"=r"(r[11]),"=r"(r[12]),"=r"(r[13]),"=r"(r[14]),"=r"(r[15]),"=r"(r[16]),"=r"(r[17]),"=r"(r[18]),"=r"(r[19]),"=r"(r[20]),"=r"(r[21]),"=r"(r[22]),"=r"(r[23]),"=r"(r[24]),"=r"(r[25]),"=r"(r[26]),"=r"(r[27]),"=r"(r[28]),"=r"(r[29]),"=r"(r[30]),"=r"(r[31]),"=r"(r[32]),"=r"(r[33]),"=r"(r[34]),"=r"(r[35]),"=r"(r[36]),"=r"(r[37]),"=r"(r[38]),"=r"(r[39]),"=r"(r[40]),"=r"(r[41]),"=r"(r[42]),"=r"(r[43]),"=r"(r[44]),"=r"(r[45]),"=r"(r[46]),"=r"(r[47]),"=r"(r[48]),"=r"(r[49]),"=r"(r[50]),"=r"(r[51]),"=r"(r[52]),"=r"(r[53]),"=r"(r[54]),"=r"(r[55]),"=r"(r[56]),"=r"(r[57]),"=r"(r[58]),"=r"(r[59]),"=r"(r[60]),"=r"(r[61]),"=r"(r[62]),"=r"(r[63])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 32-bit columns (bf16 pairs) of this thread's lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&w)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(w[0]),"r"(w[1]),"r"(w[2]),"r"(w[3]),"r"(w[4]),"r"(w[5]),"r"(w[6]),"r"(w[7]),"r"(w[8]),"r"(w[9]),"r"(w[10]),"r"(w[11]),"r"(w[12]),"r"(w[13]),"r"(w[14]),"r"(w[15]),"r"(w[16]),"r"(w[17]),"r"(w[18]),"r"(w[19]),"r"(w[20]),"r"(w[21]),"r"(w[22]),"r"(w[23]),"r"(w[24]),"r"(w[25]),"r"(w[26]),"r"(w[27]),"r"(w[28]),"r"(w[29]),"r"(w[30]),"r"(w[31])
        : "memory");
}


__device__ __forceinline__ void tmem_st32f(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
        "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
        "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
        "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
        "f"(v[29]), "f"(v[30]), "f"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void flag_err(uint32_t* err, uint32_t bits) {
    if (err != nullptr) atomicOr(err, bits);
}

// Barrier among `count` threads (whole warps) under hardware barrier `id` (not 0).
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// N (16 or 32) 32-bit columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_st_words(uint32_t taddr, const uint32_t (&w)[N]) {
    static_assert(N == 16 || N == 32, "16 or 32 columns");
    if constexpr (N == 32) {
        tmem_st32(taddr, w);
    } else {
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,"
            "%12,%13,%14,%15,%16};" ::"r"(taddr),
            "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
            "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]),
            "r"(w[14]), "r"(w[15])
            : "memory");
    }
}

// 3-D tiled bulk tensor copy global -> shared, completion on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

}  // namespace

struct PrefillArgs {
    const uint16_t* q;
    const int32_t* q_offsets;
    const int32_t* block_table;
    const int32_t* seq_lens;
    uint16_t* out;
    uint32_t* err;
    int N, Hq, Hkv, MB, NB, total_q, max_q_len, tiles;
    float scale_log2;
    // Shared-prefix mode (prefix_split > 0): the total_q query rows all see, unmasked, the
    // first prefix_len tokens of block-table row 0; blockIdx.z picks a chunk of
    // chunk_tokens of them, and each row writes its unnormalised partial over that chunk,
    // part[(row * Hq + head) * prefix_split + chunk] = (o[D], m, l), instead of an output.
    int prefix_split, prefix_len, chunk_tokens;
    float* part;
};

// Shared memory, one 1024-byte aligned block (128-byte swizzle atoms):
//   Q [KB][128 rows][128 B] | K [2 slots][KB][256 rows][128 B] | V [2 half-slots][KB][128 rows][128 B]
//   | row-max exchange [2 parities][2 halves][128 rows] fp32 | mbarriers | TMEM base, abort flag
// At D = 128 that is 231,568 bytes of the 232,448 a CTA may use, with no slack for
// realignment: the kernel checks that the block starts 1024-byte aligned.
template <int D>
struct PrefillSmem {
    static constexpr int KB = D / 64;
    static constexpr int Q_BYTES = KB * kRows * 128;
    static constexpr int K_TILE = KB * kKvTile * 128;
    static constexpr int V_HALF = KB * kVHalf * 128;
    static constexpr int NK = 2, NV = 2;           // K slots, V half-slots
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + Q_BYTES;
    static constexpr int V_OFF = K_OFF + NK * K_TILE;
    static constexpr int XCH_OFF = V_OFF + NV * V_HALF;
    static constexpr int BAR_OFF = XCH_OFF + 2 * 2 * kRows * 4;
    static constexpr int NBARS = 16;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = MISC_OFF + 16;
    static_assert(BYTES <= 232448, "shared memory of one CTA");
};

// TMEM columns: S at 0 (fp32 scores of one 256-token tile, 256 columns), P at 256 (bf16
// pairs, 128 columns), O at 384 (fp32, D columns).  P V reads its A operand (P) from
// tensor memory.
//
// Softmax: two warpgroups split every score row: warps 0-3 take columns 0-127 of the
// tile, warps 4-7 columns 128-255 (the same TMEM lanes, i.e. the same query rows).  The
// partners exchange their row max through shared memory once per tile; each keeps its
// own partial row sum, the halves are added at the end.
// SHARED: the shared-prefix pass (every row sees block-table row 0's first prefix_len
// tokens, partials out); otherwise causal prefill chunks with bf16 outputs.
template <int D, int BS, int G, bool SHARED>
__global__ void __launch_bounds__(kThreads, 1)
    pkv_prefill_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                       const PrefillArgs a) {
    using SM = PrefillSmem<D>;
    constexpr int KB = SM::KB;
    constexpr int TQ = kRows / G;            // query tokens per tile
    constexpr int PAGES = kKvTile / BS;      // pages per K tile
    constexpr int HPAGES = kVHalf / BS;      // pages per V half-tile
    constexpr int HALF = kKvTile / 2;        // score columns per softmax warpgroup
    constexpr int DH = D / 2;                // O / Q columns per warpgroup (d values)
    constexpr uint32_t ID_S = idesc_bf16(kRows, kKvTile, 0);
    constexpr uint32_t ID_O = idesc_bf16(kRows, D, 1);

    extern __shared__ __align__(1024) uint8_t smem_raw[];

    pdl_launch_dependents();
    pdl_wait();

    if (smem_u32(smem_raw) & 1023u) {        // the swizzled layout needs the alignment
        if (threadIdx.x == 0) flag_err(a.err, PKV_DEVERR_WAIT_TIMEOUT);
        return;
    }
    const int tile = a.tiles - 1 - (int)blockIdx.x;   // heavy (late) tiles first
    const int h = blockIdx.y;
    constexpr bool shared = SHARED;
    const int r = shared ? 0 : (int)blockIdx.z;
    const int zc = shared ? (int)blockIdx.z : 0;      // shared mode: KV chunk
    int q0 = 0, q_len = a.total_q, seq = a.prefix_len;
    if (!shared) {
        q0 = a.q_offsets[r];
        q_len = a.q_offsets[r + 1] - q0;
        seq = a.seq_lens[r];
        if (q_len < 0) q_len = 0;
        if (q0 < 0 || q0 + q_len > a.total_q) {
            if (threadIdx.x == 0 && tile == 0 && h == 0) flag_err(a.err, PKV_DEVERR_QLEN_CLAMPED);
            return;
        }
    }
    const int ctx = seq - q_len;             // tokens before the chunk (causal mode)
    if (q_len > a.max_q_len) {               // rows past max_q_len are not computed
        if (threadIdx.x == 0 && h == 0 && (int)blockIdx.x == 0)
            flag_err(a.err, PKV_DEVERR_QLEN_CLAMPED);
        q_len = a.max_q_len;
    }
    if (tile * TQ >= q_len) return;          // past this request's queries: no work
    // KV range of this CTA: tokens kv_lo .. kv_lo + kv_end - 1 of the request's cache
    int kv_lo = 0, kv_end;
    if (shared) {
        kv_lo = zc * a.chunk_tokens;
        kv_end = min(seq, kv_lo + a.chunk_tokens) - kv_lo;
        if (kv_lo + kv_end > a.MB * BS) kv_end = a.MB * BS - kv_lo;
    } else {
        kv_end = ctx + min(tile * TQ + TQ, q_len);   // tokens the tile's last query sees
        if (kv_end > seq) kv_end = seq;
        if (kv_end > a.MB * BS) kv_end = a.MB * BS;
    }
    if (kv_end < 0) kv_end = 0;
    const int pg0 = kv_lo / BS;              // first page of the range (kv_lo % BS == 0)
    const int n_tiles = (kv_end + kKvTile - 1) / kKvTile;
    // V halves: both halves of every tile but the last, whose second half is loaded
    // only if a token of it is visible
    const int last_valid = n_tiles > 0 ? kv_end - (n_tiles - 1) * kKvTile : 0;   // 1..256
    const int n_halves = n_tiles > 0 ? 2 * n_tiles - (last_valid <= kVHalf ? 1 : 0) : 0;
    const int tail_valid = n_halves > 0 ? kv_end - (n_halves - 1) * kVHalf : 0;  // 1..128

    uint8_t* sm = smem_raw;
    const uint32_t sQ = smem_u32(sm + SM::Q_OFF);
    const uint32_t sK = smem_u32(sm + SM::K_OFF);
    const uint32_t sV = smem_u32(sm + SM::V_OFF);
    float* xch = reinterpret_cast<float*>(sm + SM::XCH_OFF);   // [parity][half][row]
    const uint32_t bars = smem_u32(sm + SM::BAR_OFF);
    uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(sm + SM::MISC_OFF);
    volatile int* abort_v = reinterpret_cast<volatile int*>(sm + SM::MISC_OFF + 4);
    const uint32_t bar_q = bars + 0;            // Q stored to shared memory (8 warps)
    const uint32_t bar_s_full = bars + 8;       // S computed (commit)
    const uint32_t bar_s_free = bars + 16;      // S loaded by the softmax (8 warps)
    const uint32_t bar_p_ready = bars + 24;     // P stored (8 warps)
    const uint32_t bar_pv = bars + 32;          // P V done (commit)
    const uint32_t bar_v_tail = bars + 40;      // last V half's tail zeroed
    const uint32_t bar_k_full = bars + 48;      // [2]
    const uint32_t bar_k_empty = bars + 64;     // [2]
    const uint32_t bar_v_full = bars + 80;      // [2]
    const uint32_t bar_v_empty = bars + 96;     // [2]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        mbar_init(bar_q, 8);
        mbar_init(bar_s_full, 1);
        mbar_init(bar_s_free, 8);
        mbar_init(bar_p_ready, 8);
        mbar_init(bar_pv, 1);
        mbar_init(bar_v_tail, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_k_full + 8 * i, 1);
            mbar_init(bar_k_empty + 8 * i, 1);
            mbar_init(bar_v_full + 8 * i, 1);
            mbar_init(bar_v_empty + 8 * i, 1);
        }
        *abort_v = 0;
        fence_mbar_init();
    }
    if (warp == 8) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_base_s)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_s;

    // a bounded wait by lane 0, its outcome broadcast to the warp (a time-out also
    // raises the abort flag, which the other roles see at their next failed wait)
    auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
        bool ok = true;
        if (lane == 0) ok = mbar_wait_bounded(bar, parity, kWaitNs);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok && lane == 0) {
            flag_err(a.err, PKV_DEVERR_WAIT_TIMEOUT);
            *abort_v = 1;
        }
        return ok;
    };
    // the same for a single thread
    auto thread_wait = [&](uint32_t bar, uint32_t parity) -> bool {
        if (mbar_wait_bounded(bar, parity, kWaitNs)) return true;
        flag_err(a.err, PKV_DEVERR_WAIT_TIMEOUT);
        *abort_v = 1;
        return false;
    };

    // warps 8-11 (the two producers and the two MMA issuers) run on few registers, the two
    // softmax warpgroups on many; each warpgroup executes its setmaxnreg as a whole, at
    // the head of its own branch
    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
        if (warp == 8 || warp == 9) {
            // ---------------------------------------------------------- TMA producers
            // warp 8 feeds the K slots (one 256-token tile each), warp 9 the V half-slots
            // (128 tokens each); a K slot frees when its Q K^T completes, a V half-slot
            // when the P V MMAs reading it complete
            const bool is_k = warp == 8;
            if (lane == 0) prefetch_tensormap(is_k ? &tk : &tv);
            const CUtensorMap* map = is_k ? &tk : &tv;
            const uint32_t ring = is_k ? sK : sV;
            const int slot_bytes = is_k ? SM::K_TILE : SM::V_HALF;
            const int rows = is_k ? kKvTile : kVHalf;           // rows of one 64-d chunk region
            const int per = is_k ? PAGES : HPAGES;              // pages per item
            const uint32_t full = is_k ? bar_k_full : bar_v_full;
            const uint32_t empty = is_k ? bar_k_empty : bar_v_empty;
            const int items = is_k ? n_tiles : n_halves;
            const int64_t row_end = (int64_t)a.NB * a.Hkv * BS;   // first row past the pool
            // pages of item jj, and lane's block id for it: read one item ahead, so the
            // table read overlaps the wait for the slot instead of following it
            auto item_pages = [&](int jj) {
                const int np = (kv_end - jj * per * BS + BS - 1) / BS;
                return np > per ? per : np;
            };
            auto item_block = [&](int jj) {
                return lane < item_pages(jj)
                           ? a.block_table[(int64_t)r * a.MB + pg0 + jj * per + lane] : 0;
            };
            int blk_next = items > 0 ? item_block(0) : 0;
            for (int j = 0; j < items; ++j) {
                const int st = j & 1;
                const int blk = blk_next;
                if (j + 1 < items) blk_next = item_block(j + 1);
                if (j >= 2 && !warp_wait(empty + 8 * st, ((j >> 1) - 1) & 1)) break;
                if (*abort_v) break;
                const int npages = item_pages(j);
                if (lane == 0)
                    mbar_arrive_expect_tx(full + 8 * st, (uint32_t)(npages * KB * BS * 128));
                __syncwarp();
                if (lane < npages) {
                    int64_t row;
                    if (blk < 0 || blk >= a.NB) {
                        if (is_k) flag_err(a.err, PKV_DEVERR_BLOCK_RANGE);
                        row = row_end;                 // past the end: TMA fills zeros
                    } else {
                        row = ((int64_t)blk * a.Hkv + h) * BS;
                    }
                    if (is_k) {
                        // K: [chunk][256 rows][128 B], one box per page and chunk
                        const uint32_t off = (uint32_t)(lane * BS * 128);
#pragma unroll
                        for (int kb = 0; kb < KB; ++kb)
                            tma_load_2d(ring + st * slot_bytes + kb * rows * 128 + off, map,
                                        kb * 64, (int)row, full + 8 * st);
                    } else {
                        // V: [page][chunk][BS rows][128 B], one box per page (all of D)
                        tma_load_3d(ring + st * slot_bytes + (uint32_t)(lane * KB * BS * 128),
                                    map, 0, (int)row, 0, full + 8 * st);
                    }
                }
            }
            // the last V half: once it has landed, zero its rows at or past kv_end (the
            // partial page, pages past the request), so P = 0 never meets stale or NaN bytes
            const int tail = n_halves - 1;
            if (!is_k && n_halves > 0 && tail_valid < kVHalf && !*abort_v) {
                if (warp_wait(bar_v_full + 8 * (tail & 1), (tail >> 1) & 1)) {
                    uint8_t* vst = sm + SM::V_OFF + (tail & 1) * SM::V_HALF;
                    for (int kb = 0; kb < KB; ++kb)
                        for (int rr = tail_valid + (lane >> 3); rr < kVHalf; rr += 4)
                            *reinterpret_cast<uint4*>(vst + ((rr / BS) * KB + kb) * BS * 128 +
                                                      (rr % BS) * 128 + (lane & 7) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_v_tail);
                }
            }
        } else if (warp == 10 || warp == 11) {
            // ---------------------------------------------------------- MMA issuers (lane 0)
            // warp 10 issues every Q K^T, warp 11 every P V.  They write disjoint TMEM
            // columns (S; O), each commit tracks only its own thread's MMAs, and the
            // barriers order what depends on what: Q K^T(j + 1) waits for S(j) to be
            // loaded, P V(j) for P(j), and P(j + 1) is stored only after P V(j).
            if (lane == 0 && warp == 11) {
                auto issue_pv = [&](int t) -> bool {
                    if (!thread_wait(bar_p_ready, t & 1)) return false;
                    for (int hv = 0; hv < 2; ++hv) {
                        const int t2 = 2 * t + hv;
                        if (t2 >= n_halves) break;
                        const int vs = t2 & 1;
                        if (!thread_wait(bar_v_full + 8 * vs, (t2 >> 1) & 1)) return false;
                        if (t2 == n_halves - 1 && tail_valid < kVHalf &&
                            !thread_wait(bar_v_tail, 0))
                            return false;
                        tc_fence_after();
                        const uint32_t vbase = sV + vs * SM::V_HALF;
#pragma unroll
                        for (int k = 0; k < kVHalf / 16; ++k) {
                            // 16 tokens inside one page: rows at 128 B, chunks BS * 128 B apart
                            const uint32_t koff = (uint32_t)(((k * 16) / BS) * KB * BS * 128 +
                                                             ((k * 16) % BS) * 128);
                            const uint64_t b = smem_desc_sw128(vbase + koff, BS * 128, 1024);
                            mma_ts(tmem + kColO, tmem + kColP + (hv * (kVHalf / 16) + k) * 8, b,
                                   ID_O, (t > 0 || hv > 0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit(bar_v_empty + 8 * vs);
                    }
                    mma_commit(bar_pv);
                    return true;
                };
                for (int t = 0; t < n_tiles; ++t)
                    if (!issue_pv(t)) break;
            } else if (lane == 0) {
                bool ok = thread_wait(bar_q, 0);
                tc_fence_after();
                for (int j = 0; ok && j < n_tiles; ++j) {
                    const int ks = j & 1;
                    if (!thread_wait(bar_k_full + 8 * ks, (j >> 1) & 1)) { ok = false; break; }
                    if (j >= 1 && !thread_wait(bar_s_free, (j - 1) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t kbase = sK + ks * SM::K_TILE;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t col = (uint32_t)((k & 3) * 32);
                        mma_ss(tmem + kColS,
                               smem_desc_sw128(sQ + (k >> 2) * kRows * 128 + col, 16, 1024),
                               smem_desc_sw128(kbase + (k >> 2) * kKvTile * 128 + col, 16, 1024),
                               ID_S, k > 0 ? 1u : 0u);
                    }
                    mma_commit(bar_s_full);
                    mma_commit(bar_k_empty + 8 * ks);
                }
            }
            __syncwarp();
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        // ---------------------------------------------------------- softmax, 2 x 4 warps
        const int hf = warp >> 2;                // column half of every score row
        const int m = tid & 127;                 // query row = TMEM lane
        const int tq_i = m / G, g = m - (m / G) * G;
        const int qi = tile * TQ + tq_i;
        const bool row_valid = qi < q_len;
        int vis = row_valid ? (shared ? kv_end : ctx + qi + 1) : 0;   // tokens this row sees
        if (vis > kv_end) vis = kv_end;
        if (vis < 0) vis = 0;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int nbar = 1 + (warp & 3);         // named barrier of this warp pair
        // this half's D/2 values of the Q row into shared memory, in the 128-byte
        // swizzled K-major layout the MMA reads (16-byte unit c of row m at c ^ (m & 7))
        {
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + ((int64_t)(q0 + qi) * a.Hq + (int64_t)h * G + g) * D + hf * DH);
#pragma unroll
            for (int i = 0; i < DH / 8; ++i) {
                const int cu = hf * (DH / 8) + i;        // 16-byte unit of the D-value row
                const uint4 v4 = row_valid ? src[i] : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sm + SM::Q_OFF + (cu >> 3) * kRows * 128 + m * 128 +
                                          (((cu & 7) ^ (m & 7)) << 4)) = v4;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q);
        }
        float m_ref = -INFINITY;                 // reference max (log2 domain) of O and l
        float l = 0.f;                           // this half's partial row sum
        // A failed wait marks the rows bad (zero output, flagged) but never leaves the
        // loop: the partner warp must meet every named barrier below.
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            if (ok && !warp_wait(bar_s_full, j & 1)) ok = false;
            tc_fence_after();
            float s[HALF];
            tmem_ld64(lane_base + kColS + hf * HALF, *reinterpret_cast<float(*)[64]>(s));
            tmem_ld64(lane_base + kColS + hf * HALF + 64, *reinterpret_cast<float(*)[64]>(s + 64));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_s_free);
            // mask (diagonal and tail tiles only), partial max on raw scores (scale > 0)
            const int lim = vis - j * kKvTile - hf * HALF;   // columns >= lim are masked
            if (lim < HALF) {
#pragma unroll
                for (int c = 0; c < HALF; ++c) s[c] = c < lim ? s[c] : -INFINITY;
            }
            static_assert(HALF % 16 == 0, "score columns in groups of 16");
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
            for (int c = 16; c < HALF; c += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmax3f(m8[i], s[c + i], s[c + 8 + i]);
            const float pmx = fmaxf(fmax3f(m8[0], m8[1], m8[2]),
                                    fmax3f(fmax3f(m8[3], m8[4], m8[5]), m8[6], m8[7]));
            float* xj = xch + (j & 1) * 2 * kRows;
            xj[hf * kRows + m] = pmx;
            named_barrier_sync(nbar, 64);
            const float mx = fmaxf(pmx, xj[(hf ^ 1) * kRows + m]) * a.scale_log2;
            // raise the reference max only when a score passes it by more than 2^8
            // (both halves take the same decision from the same numbers)
            float alpha = 1.f;
            bool rescale = false;
            if (mx > m_ref + 8.f) {
                alpha = m_ref == -INFINITY ? 0.f : exp2f(m_ref - mx);
                m_ref = mx;
                rescale = j > 0;
                l *= alpha;
            }
            const float nmu = m_ref == -INFINITY ? 0.f : -m_ref;
            uint32_t p[HALF / 2];
            // column pairs: the exponent arguments by one packed FMA, the sums in four
            // packed accumulators
            const uint64_t sc2 = f32x2_pack(a.scale_log2, a.scale_log2);
            const uint64_t nmu2 = f32x2_pack(nmu, nmu);
            uint64_t l4[4] = {0ull, 0ull, 0ull, 0ull};   // (+0, +0) pairs
#pragma unroll
            for (int c = 0; c < HALF; c += 2) {
                float t0, t1;
                f32x2_unpack(f32x2_fma(f32x2_pack(s[c], s[c + 1]), sc2, nmu2), t0, t1);
                const float e0 = ex2_approx(t0);
                const float e1 = ex2_approx(t1);
                p[c / 2] = pack_bf16x2(e0, e1);
                l4[(c >> 1) & 3] = f32x2_add(l4[(c >> 1) & 3], f32x2_pack(e0, e1));
            }
            float l8[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) f32x2_unpack(l4[i], l8[2 * i], l8[2 * i + 1]);
            l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
            // P buffer and O are free once the previous P V has completed
            if (j >= 1) {
                if (ok && !warp_wait(bar_pv, (j - 1) & 1)) ok = false;
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, rescale)) {
                const float f = rescale ? alpha : 1.f;
#pragma unroll 1
                for (int c = 0; c < DH / 32; ++c) {
                    float o[32];
                    tmem_ld32(lane_base + kColO + hf * DH + c * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= f;
                    tmem_st32f(lane_base + kColO + hf * DH + c * 32, o);
                }
            }
            tmem_st32(lane_base + kColP + hf * (HALF / 2), *reinterpret_cast<uint32_t(*)[32]>(p));
            tmem_st32(lane_base + kColP + hf * (HALF / 2) + 32,
                      *reinterpret_cast<uint32_t(*)[32]>(p + 32));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p_ready);
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n_tiles > 0) {
            ok = warp_wait(bar_pv, (n_tiles - 1) & 1);
            tc_fence_after();
        }
        // the halves' partial sums, through the exchange parity no pending read uses
        float* xl = xch + (n_tiles & 1) * 2 * kRows;
        xl[hf * kRows + m] = l;
        named_barrier_sync(nbar, 64);
        const float lt = l + xl[(hf ^ 1) * kRows + m];
        if (shared) {
            // the row's unnormalised partial over this chunk: o, its reference max m
            // (log2 domain, scale applied) and sum l; no contribution if nothing was seen.
            // The tensor-memory loads are warp-collective: every lane takes part (n_tiles
            // and ok are the same across the warp), only the stores depend on the row.
            float* prow = a.part + (((int64_t)qi * a.Hq + (int64_t)h * G + g) * a.prefix_split +
                                    zc) * (D + 4);
            const bool has = n_tiles > 0 && ok && lt > 0.f;
#pragma unroll 1
            for (int c = 0; c < DH / 32; ++c) {
                float o[32];
                if (n_tiles > 0 && ok) {
                    tmem_ld32(lane_base + kColO + hf * DH + c * 32, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.f;
                }
                if (row_valid) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(prow + hf * DH + c * 32 + i) =
                            has ? make_float4(o[i], o[i + 1], o[i + 2], o[i + 3])
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            if (row_valid && hf == 0)
                *reinterpret_cast<float2*>(prow + D) =
                    has ? make_float2(m_ref, lt) : make_float2(-INFINITY, 0.f);
        }
        const float inv = (lt > 0.f && ok) ? 1.f / lt : 0.f;
        uint16_t* orow = a.out + ((int64_t)(q0 + qi) * a.Hq + (int64_t)h * G + g) * D + hf * DH;
#pragma unroll 1
        for (int c = 0; c < (shared ? 0 : DH / 32); ++c) {
            float o[32];
            if (n_tiles > 0 && ok) {
                tmem_ld32(lane_base + kColO + hf * DH + c * 32, o);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0.f;
            }
            if (row_valid) {
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 u4;
                    u4.x = pack_bf16x2(o[i] * inv, o[i + 1] * inv);
                    u4.y = pack_bf16x2(o[i + 2] * inv, o[i + 3] * inv);
                    u4.z = pack_bf16x2(o[i + 4] * inv, o[i + 5] * inv);
                    u4.w = pack_bf16x2(o[i + 6] * inv, o[i + 7] * inv);
                    *reinterpret_cast<uint4*>(orow + c * 32 + i) = u4;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 prefill_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult qr;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <typename K>
int launch_regs(K kern) {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? fa.numRegs : 0;
}

template <int D, int BS, int G>
cudaError_t prefill_launch_t(const PrefillLaunch& L, const PrefillArgs& a, const CUtensorMap& tk,
                             const CUtensorMap& tv, cudaStream_t st) {
    auto kern = a.prefix_split > 0 ? pkv_prefill_kernel<D, BS, G, true>
                                   : pkv_prefill_kernel<D, BS, G, false>;
    // the register split must fit in what the block is launched with, else the softmax
    // warps' setmaxnreg.inc could never be granted
    static const int regs_c = launch_regs(pkv_prefill_kernel<D, BS, G, false>);
    static const int regs_s = launch_regs(pkv_prefill_kernel<D, BS, G, true>);
    if ((a.prefix_split > 0 ? regs_s : regs_c) * kThreads < kRegsSplit)
        return cudaErrorInvalidConfiguration;
    // one CTA per SM (it holds all 512 TMEM columns); ask for enough shared memory
    // that no second CTA can be co-resident
    int smem = PrefillSmem<D>::BYTES;
    if (smem < 120 * 1024) smem = 120 * 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned gz = (unsigned)(a.prefix_split > 0 ? a.prefix_split : L.N);
    return launch_pdl(kern, dim3((unsigned)a.tiles, (unsigned)L.Hkv, gz), dim3(kThreads),
                      (size_t)smem, st, tk, tv, a);
}

template <int D, int BS>
cudaError_t prefill_launch_g(int G, const PrefillLaunch& L, const PrefillArgs& a,
                             const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    switch (G) {
        case 1: return prefill_launch_t<D, BS, 1>(L, a, tk, tv, st);
        case 2: return prefill_launch_t<D, BS, 2>(L, a, tk, tv, st);
        case 4: return prefill_launch_t<D, BS, 4>(L, a, tk, tv, st);
        case 8: return prefill_launch_t<D, BS, 8>(L, a, tk, tv, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool prefill_shape_supported(int Hq, int Hkv, int D, int BS, int dtype) {
    if (dtype != PKV_BF16) return false;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return false;
    const int G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return false;
    return (D == 64 || D == 128) && (BS == 16 || BS == 32);
}

int prefill_launch(const PrefillLaunch& L, cudaStream_t st) {
    auto fn = prefill_encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    const int G = L.Hq / L.Hkv;
    const int TQ = kRows / G;
    alignas(64) CUtensorMap tk, tv;
    const int64_t rows = (int64_t)L.NB * L.Hkv * L.BS;
    {   // K: 2-D, one box = one page's rows of one 64-d chunk
        cuuint64_t dims[2] = {(cuuint64_t)L.D, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)L.D * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)L.BS};
        cuuint32_t es[2] = {1, 1};
        if (fn(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(L.k_cache), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PKV_ERR_CUDA;
    }
    {   // V: 3-D (64 d, row, 64-d chunk), one box = one page's rows of all of D, laid
        // out chunk by chunk
        cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(L.D / 64)};
        cuuint64_t strides[2] = {(cuuint64_t)L.D * 2, 128};
        cuuint32_t box[3] = {64, (cuuint32_t)L.BS, (cuuint32_t)(L.D / 64)};
        cuuint32_t es[3] = {1, 1, 1};
        if (fn(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(L.v_cache), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PKV_ERR_CUDA;
    }
    PrefillArgs a;
    a.q = static_cast<const uint16_t*>(L.q);
    a.q_offsets = L.q_offsets;
    a.block_table = L.block_table;
    a.seq_lens = L.seq_lens;
    a.out = static_cast<uint16_t*>(L.out);
    a.err = L.err;
    a.N = L.N;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.MB = L.MB;
    a.NB = L.NB;
    a.total_q = L.total_q;
    a.max_q_len = L.max_q_len;
    a.tiles = (L.max_q_len + TQ - 1) / TQ;   // query tiles per request
    a.scale_log2 = L.scale * 1.4426950408889634f;
    a.prefix_split = L.prefix_split;
    a.prefix_len = L.prefix_len;
    a.chunk_tokens = L.chunk_tokens;
    a.part = L.part;
    if (a.tiles <= 0) return PKV_OK;
    cudaError_t e = cudaErrorInvalidValue;
    if (L.D == 128 && L.BS == 16) e = prefill_launch_g<128, 16>(G, L, a, tk, tv, st);
    else if (L.D == 128 && L.BS == 32) e = prefill_launch_g<128, 32>(G, L, a, tk, tv, st);
    else if (L.D == 64 && L.BS == 16) e = prefill_launch_g<64, 16>(G, L, a, tk, tv, st);
    else if (L.D == 64 && L.BS == 32) e = prefill_launch_g<64, 32>(G, L, a, tk, tv, st);
    else return PKV_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
