// pkv_decode.cu -- paged GQA decode attention for sm_103a, one or several query
// tokens per request.
//
// Computes, for every request r and query head hq (kv head h = hq / G),
//     out[r][hq] = softmax(scale * q K_r^T) V_r
// where K_r / V_r are the request's pages gathered through its block table
// ("深入LLM推理：从KV Cache到PD分离的Serving全景解析", sections "KV Cache：Transformer
// 的循环状态" and "PagedAttention与Cache管理"), with an online (running max / sum)
// softmax ("GPU推理深度拆解：KV Cache视角", 算子优化要点) and the KV length split
// across warps when the batch is small (same note: batch-1 decode leaves SMs idle).
// With several query tokens per request (verifying speculative drafts,
// "深入LLM推理：从KV Cache到PD分离的Serving全景解析", "投机解码：打破每步一token的假设"),
// query i of the request's q_len newest tokens attends causally to positions
// 0 .. seq_len - q_len + i.
//
// Work decomposition.  Unit u = (request r, kv head h) owns np_r = ceil(seq_r / BS)
// pages.  All units' pages form one flat list of P items (request-major, then
// head, then page).  A persistent grid of W warps (one CTA per SM) cuts the list
// into W equal contiguous ranges, so every warp streams the same number of bytes
// whatever the length mix.  A warp walks its range unit by unit ("segments");
// a segment that covers a whole unit writes the bf16 output directly, otherwise
// it writes an unnormalised partial (o, running max m, sum l) to workspace slot
// u + w (unique: unit and warp ranges are both ordered).  Every split unit is merged
// with log-sum-exp weights by a small follow-up kernel (one CTA per unit, one warp
// per query head and query position), launched behind this one.  No warp waits for or merges after
// another: a merge by the last warp to finish a unit kept that warp, and its SM,
// busy past its peers (measured on GB300: up to 13 us for one query position and 46
// us for four, with the step 2.5% and 14% slower).
//
// Per-warp pipeline.  Each warp owns `stages` shared-memory stages, each holding
// the K and V tile (TT tokens) of one (block, head) page (of one 64-token group of
// blocks for int4).  Lane 0 issues 2-D bulk
// tensor copies (TMA, 128-byte swizzle, box = 128 bytes x TT rows) that complete on
// the stage's mbarrier; all lanes wait on it (bounded), compute, and the stage is
// refilled with the tile `stages` ahead.  Block ids for the next 32 pages are looked
// up one batch ahead (one lane per page), so the issue path never waits on the
// block table.
//
// Math per tile (tensor cores, mma.sync m16n8k16, fp32 accumulators); one mma
// n-tile of 8 columns per query position, a column per query head of the group:
//   S^T[t][g] = K[t][:] . Q[g][:]     A = K tile (16 tokens x 16 d, ldmatrix),
//                                     B = Q^T of the GQA group (8 heads, registers)
//   O^T[d][g] += V^T[d][t] P^T[t][g]  A = V tile (ldmatrix.trans), B = P^T from
//                                     the S^T accumulators via movmatrix.trans
// Quantised pages are widened exactly to fp16 in registers: E4M3 by cvt e4m3x2 ->
// f16x2; int8 and int4 K codes by a byte permute or mask-or that yields 1024 plus the
// biased code, whose constant share is subtracted once per score; int8 and int4 V
// codes by the same picks under a zero exponent (fp16 subnormals, biased code *
// 2^-24), whose small constant share is subtracted once per output.  The
// per-(block, head) K scale multiplies S in fp32; the V scale multiplies P before P is
// rounded to fp16, so O accumulates every page in the same mma accumulators.  int4
// caches are worked 64 tokens (two or four blocks of one unit) per pipeline item.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <atomic>
#include <type_traits>

#include "pkv_internal.cuh"

namespace pkv {

struct DecodeArgs {
    const uint16_t* q;
    const int32_t* q_offsets;       // [N + 1] query rows of each request; null: row r
    uint16_t* out;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const float* k_scale;
    const float* v_scale;
    uint32_t* err;
    int32_t* g_prefix;              // page prefix over requests, for the merge kernel
    float* partials;
    int N, Hq, Hkv, G, MB, NB;
    float scale_log2;   // scale * log2(e): scores kept in the log2 domain
    int stages;
    int total_warps;
    // Shared-prefix decode: the first skip_blocks blocks of every request are attended
    // by the prefix pass, this kernel takes the rest; every unit then writes a partial
    // (none writes its output) and the cascade merge adds the prefix partials
    // cascade_part[(r * Hq + hq) * cascade_split + c].
    int skip_blocks;
    const float* cascade_part;
    int cascade_split;
    // Append (bf16 pages, one query): each request's newest token (position seq_len - 1)
    // has K/V rows k_new / v_new [N][Hkv][D]; the warp whose tile holds that position
    // writes them into the cache pages (k_cache_w / v_cache_w) and into its tile, so the
    // call needs no cache write before it.
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint16_t* k_cache_w;
    uint16_t* v_cache_w;
};

template <int D, int BS, int KT>
struct Cfg {
    static constexpr bool FP8 = KT != 0;                  // quantised pages (one scale each)
    static constexpr bool I4 = KT == 3;                   // int4: two codes per byte
    // int8 and int4 codes enter the mma with their offset (1024 + biased code); the
    // offset's share is removed once per score and once per output
    static constexpr bool FOLD = KT == 2 || KT == 3;
    static constexpr int ELT = FP8 ? 1 : 2;
    static constexpr int ROW_BYTES = I4 ? D / 2 : D * ELT;
    static constexpr int CH = I4 ? 1 : ROW_BYTES / 128;   // 128-byte column chunks per row
    static constexpr int CH_ELEMS = 128 / ELT;            // elements per chunk
    // int4 pages are worked on two or four cache blocks at a time (64 tokens): the
    // flat page list counts these groups, so each pipeline item carries twice the
    // math of a 32-token block for the same waits, shuffles and branches
    static constexpr int PPI = I4 ? 64 / BS : 1;          // cache blocks per list page
    static constexpr int SPB = BS * PPI;                  // tokens per list page
    static constexpr int TT = FP8 ? SPB : 16;             // tokens per pipeline tile
    static constexpr int SUB = SPB / TT;                  // tiles per list page (1 or 2)
    static constexpr int MTB = BS / 16;                   // 16-token mma tiles per block
    static constexpr int TILE_BYTES = TT * ROW_BYTES;     // K (or V) part of a stage
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;    // 8 KB at bf16 D=128 or E4M3 BS=32
    static constexpr int MT = TT / 16;                    // 16-token mma tiles per tile
    static constexpr int KS = D / 16;                     // QK k-steps
    static constexpr int DT = D / 16;                     // PV d-tiles
    // 8/16-bit rows are whole 128-byte swizzle lines; int4 rows are 64 bytes (D = 128),
    // stored with the 64-byte swizzle
    static_assert(I4 || ROW_BYTES % 128 == 0, "rows must be whole 128-byte swizzle lines");
    static_assert(!I4 || ROW_BYTES == 64, "int4 rows are 64 bytes");
    static_assert(BS % 16 == 0, "block size must be a multiple of 16");
    static_assert(SUB == 1 || SUB == 2, "one or two tiles per page");
    static_assert(SPB <= 255, "token count of a list page fits the 8-bit field");
};

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
// The running max of a head is raised only when a score exceeds it by more than
// this many log2 units; until then P is taken against the stale max (P <= 2^8).
constexpr float kRescaleSlack = 8.f;

// Byte offset of 16-byte chunk `kc` of token row `t` inside a tile of ROWS rows
// laid out by TMA with 128-byte swizzle: column chunk region, then rows of 128
// bytes whose 16-byte units are XOR-permuted by (row mod 8).
template <int ROWS>
__device__ __forceinline__ uint32_t swz(int t, int kc) {
    return (uint32_t)((kc >> 3) * (ROWS * 128) + t * 128 + (((kc & 7) ^ (t & 7)) << 4));
}

// Byte offset of 16-byte unit `u` (0-3) of row `t` inside an int4 tile of 64-byte rows
// laid out by TMA with the 64-byte swizzle: address bits 4-5 XOR bits 7-8, i.e. the unit
// index XOR (t / 2 mod 4).  The eight rows one ldmatrix matrix reads then fall in eight
// different 16-byte bank groups (unswizzled they would share two, a 4-way conflict).
__device__ __forceinline__ uint32_t swz64(int t, int u) {
    return (uint32_t)(t * 64 + ((u ^ ((t >> 1) & 3)) << 4));
}

// Per-lane description of one list page (PPI cache blocks) of a 32-page batch.
template <int PPI>
struct PageBatch {
    int row[PPI];  // TMA row of each block's first token / BS: id * Hkv + h (id = NB: past
                   // the end, read as zeros)
    int r, h;      // unit
    uint32_t fl;   // valid tokens | first << 8 | last << 9 | page index j << 10
    float ks[PPI], vs[PPI];  // per-block scales of quantised pages
};

template <int BS, int PPI, bool FP8>
__device__ __forceinline__ void load_batch(PageBatch<PPI>& b, int xbeg, int x1,
                                           const int32_t* s_prefix, const int32_t* s_seq,
                                           const DecodeArgs& a, uint32_t& errbits) {
    const int lane = threadIdx.x & 31;
    const int x = xbeg + lane;
    b.r = 0; b.h = 0; b.fl = 0;
#pragma unroll
    for (int p = 0; p < PPI; ++p) {
        b.row[p] = a.NB * a.Hkv;
        b.ks[p] = 1.f;
        b.vs[p] = 1.f;
    }
    if (x >= x1) return;
    int lo = 0, hi = a.N;   // s_prefix[lo] <= x < s_prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_prefix[mid] <= x) lo = mid; else hi = mid;
    }
    const int r = lo;
    const int np = (s_prefix[r + 1] - s_prefix[r]) / a.Hkv;
    const int off = x - s_prefix[r];
    const int h = off / np;
    const int j = off - h * np;
#pragma unroll
    for (int p = 0; p < PPI; ++p) {
        const int blk = j * PPI + p;
        if (blk * BS >= s_seq[r]) break;   // past the request: stays a zero block
        int id = __ldg(a.block_table + (int64_t)r * a.MB + a.skip_blocks + blk);
        if (id < 0 || id >= a.NB) {
            errbits |= PKV_DEVERR_BLOCK_RANGE;
            id = a.NB;   // TMA of rows past the tensor end reads zeros
        }
        b.row[p] = id * a.Hkv + h;
        if (FP8 && id < a.NB) {
            b.ks[p] = __ldg(a.k_scale + (int64_t)id * a.Hkv + h);
            b.vs[p] = __ldg(a.v_scale + (int64_t)id * a.Hkv + h);
        }
    }
    const int ntok = min(BS * PPI, s_seq[r] - j * BS * PPI);
    b.r = r;
    b.h = h;
    b.fl = (uint32_t)ntok | ((j == 0) ? 0x100u : 0u) | ((j == np - 1) ? 0x200u : 0u) |
           ((uint32_t)j << 10);
}

// The query rows of request r: first row and count (clamped to QT).
template <int QT>
__device__ __forceinline__ void query_rows(const DecodeArgs& a, int r, int& qb, int& qlen,
                                           uint32_t& errbits) {
    if (a.q_offsets == nullptr) {
        qb = r;
        qlen = 1;
        return;
    }
    qb = __ldg(a.q_offsets + r);
    qlen = __ldg(a.q_offsets + r + 1) - qb;
    if (qlen < 0 || qlen > QT) {
        errbits |= PKV_DEVERR_QLEN_CLAMPED;
        qlen = min(max(qlen, 0), QT);
    }
}

template <int D, int BS, int KT, int QT>
__global__ void __launch_bounds__(((KT != 0 && KT != 3) || QT > 1) ? 256 : 384, 1)
    pkv_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
    constexpr bool FP8 = KT != 0;   // quantised pages (E4M3, int8, int4) with per-(block, head) scales
    using C = Cfg<D, BS, KT>;
    // four query positions (bf16 pages only) keep the GQA group's q fragments in shared
    // memory instead of 64 registers per lane, read back per k-step
    constexpr bool QSMEM = QT == 4;
    constexpr int QB = QSMEM ? C::KS * QT * 32 * 8 : 0;   // bytes per warp
    extern __shared__ uint8_t smem_raw[];
    const int NW = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = a.stages;

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* basep = smem_raw + (base - raw);
    const uint32_t stage0 = base + (uint32_t)(warp * S * C::STAGE_BYTES);
    uint2* qs = reinterpret_cast<uint2*>(basep + NW * S * C::STAGE_BYTES + warp * QB);
    const uint32_t bars =
        base + (uint32_t)(NW * S * C::STAGE_BYTES + NW * QB) + (uint32_t)(warp * S * 8);
    int32_t* s_prefix =
        reinterpret_cast<int32_t*>(basep + NW * S * C::STAGE_BYTES + NW * QB + NW * S * 8);
    int32_t* s_seq = s_prefix + (a.N + 1);

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bars + 8u * s, 1);
        fence_mbar_init();
    }
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    // programmatic dependent launch: let the merge kernel launch now (it waits for this
    // grid to complete), and wait for the kernels before this one (e.g. the KV write)
    // before reading anything they may have written
    pdl_launch_dependents();
    pdl_wait();

    // ---- page prefix over requests (every CTA computes its own copy) ----
    uint32_t errbits = 0;
    const int maxlen = (a.MB - a.skip_blocks) * BS;
    for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
        const int s = __ldg(a.seq_lens + i) - a.skip_blocks * BS;   // tokens after the skip
        const int c = min(max(s, 0), maxlen);
        if (c != s) errbits |= PKV_DEVERR_SEQ_CLAMPED;
        s_seq[i] = c;
    }
    __syncthreads();
    if (warp == 0) {
        int running = 0;
        for (int b0 = 0; b0 < a.N; b0 += 32) {
            const int i = b0 + lane;
            int v = (i < a.N) ? a.Hkv * ((s_seq[i] + C::SPB - 1) / C::SPB) : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += n;
            }
            if (i < a.N) s_prefix[i + 1] = running + v;
            running += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) s_prefix[0] = 0;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i <= a.N; i += blockDim.x) a.g_prefix[i] = s_prefix[i];
    }
    // requests with no cached tokens get zero output rows (grid-strided over requests);
    // with a shared prefix the cascade merge writes every row
    for (int r = blockIdx.x; r < (a.cascade_part ? 0 : a.N); r += gridDim.x) {
        if (s_seq[r] != 0) continue;
        int qb, qlen;
        query_rows<QT>(a, r, qb, qlen, errbits);
        uint4* ob = reinterpret_cast<uint4*>(a.out + (int64_t)qb * a.Hq * D);
        for (int k = threadIdx.x; k < qlen * a.Hq * D / 8; k += blockDim.x)
            ob[k] = make_uint4(0u, 0u, 0u, 0u);
    }

    const int P = s_prefix[a.N];
    // With fewer pages than warps only P warps get work (one page each); otherwise
    // every warp owns at least one page, so the warps spanning a unit are exactly
    // the ones between the warps of its first and last page.
    const int W = min(a.total_warps, P);
    const int gw = blockIdx.x * NW + warp;
    const int x0 = gw < W ? (int)(((int64_t)gw * P) / W) : 0;
    const int x1 = gw < W ? (int)(((int64_t)(gw + 1) * P) / W) : 0;
    const int count = x1 - x0;
    if (count <= 0) {
        if (blockIdx.x == 0 && errbits) atomicOr(a.err, errbits);
        return;
    }

    PageBatch<C::PPI> cur, nxt;
    load_batch<BS, C::PPI, FP8>(cur, x0, x1, s_prefix, s_seq, a, errbits);
    load_batch<BS, C::PPI, FP8>(nxt, x0 + 32, x1, s_prefix, s_seq, a, errbits);
    int cb = 0;   // batch index held in `cur`
    const uint64_t policy = l2_policy_evict_first();

    // load item i (a tile) into stage s; the caller tracks s = i mod S
    auto issue = [&](int i, int s) {
        const int pi = (C::SUB == 2) ? (i >> 1) : i;   // page of item i
        const int sub = i & (C::SUB - 1);               // tile within the page
        const int bi = pi >> 5;
        const int src = pi & 31;
        int row[C::PPI];
#pragma unroll
        for (int p = 0; p < C::PPI; ++p)
            row[p] = __shfl_sync(0xffffffffu, bi == cb ? cur.row[p] : nxt.row[p], src);
        if (lane == 0) {
            const uint32_t bar = bars + 8u * s;
            const uint32_t dst = stage0 + (uint32_t)(s * C::STAGE_BYTES);
            const int y = row[0] * BS + sub * C::TT;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
            if constexpr (C::I4) {
                // one box per cache block: BS rows of D/2 bytes, 64-byte swizzle; the
                // blocks of a list page stack into one tile of PPI * BS rows
#pragma unroll
                for (int p = 0; p < C::PPI; ++p) {
                    const uint32_t off = (uint32_t)(p * BS * C::ROW_BYTES);
                    tma_load_2d_hint(dst + off, &tmK, 0, row[p] * BS, bar, policy);
                    tma_load_2d_hint(dst + C::TILE_BYTES + off, &tmV, 0, row[p] * BS, bar,
                                     policy);
                }
            } else {
#pragma unroll
                for (int ch = 0; ch < C::CH; ++ch)
                    tma_load_2d_hint(dst + ch * (C::TT * 128), &tmK, ch * C::CH_ELEMS, y, bar,
                                     policy);
#pragma unroll
                for (int ch = 0; ch < C::CH; ++ch)
                    tma_load_2d_hint(dst + C::TILE_BYTES + ch * (C::TT * 128), &tmV,
                                     ch * C::CH_ELEMS, y, bar, policy);
            }
        }
    };

    const int total = count * C::SUB;   // pipeline items (tiles)
    const int npro = min(S, total);
    for (int i = 0; i < npro; ++i) issue(i, i);

    const int g = lane >> 2;   // mma row group: head column of B / token row of A
    const int c = lane & 3;

    float o[C::DT][QT][4];
    uint32_t qf[QSMEM ? 1 : C::KS][QT][2];
    float m0[QT], m1[QT], l0[QT], l1[QT];   // heads 2c, 2c+1 of this lane, per query
    // int8 / int4 pages: K codes enter the mma with an offset (1024 + code + 128;
    // 1024 + n or 1024 + 16 n with n = code + 8), and cq = the scores' constant part per
    // head (q . offsets).  V codes enter as fp16 subnormals ((code + 128) 2^-24; n 2^-24
    // or 16 n 2^-24) against P * v_scale, so O accumulates across pages, and cr = the
    // sum over pages of sum(P * v_scale), which times 128 (int8) or 8 (int4) is the
    // output's constant part once O is scaled back by 2^24 (int4 odd picks: 2^20)
    float cq0[QT], cq1[QT], cr0[QT], cr1[QT];
    float qscale = a.scale_log2;
    bool seg_full = false;
    int seg_r = 0, seg_h = 0;
    int seg_qb = 0, seg_qlen = 1, seg_vis = 0;   // query rows; query qi sees positions <= seg_vis + qi

    int s = 0;           // stage of item i (i mod S), kept by increment
    uint32_t par = 0;    // phase of that stage's barrier ((i / S) & 1)
    for (int i = 0; i < total; ++i) {
        const int pi = (C::SUB == 2) ? (i >> 1) : i;
        const int sub = i & (C::SUB - 1);
        if (sub == 0 && pi > 0 && (pi & 31) == 0) {
            cur = nxt;
            ++cb;
            load_batch<BS, C::PPI, FP8>(nxt, x0 + (cb + 1) * 32, x1, s_prefix, s_seq, a, errbits);
        }
        const int src = pi & 31;
        const uint32_t fl = __shfl_sync(0xffffffffu, cur.fl, src);
        float ks[C::PPI], vs[C::PPI];   // scales of the page's blocks (quantised pages)
#pragma unroll
        for (int p = 0; p < C::PPI; ++p) {
            ks[p] = FP8 ? __shfl_sync(0xffffffffu, cur.ks[p], src) : 1.f;
            vs[p] = FP8 ? __shfl_sync(0xffffffffu, cur.vs[p], src) : 1.f;
        }
        // valid tokens of this tile (<= 0 only for the empty second half of a last page)
        const int ntok = (int)(fl & 0xFFu) - sub * C::TT;
        const bool first = ((fl >> 8) & 1u) && sub == 0;
        const bool last = ((fl >> 9) & 1u) && sub == C::SUB - 1;
        const int tpos0 = (int)(fl >> 10) * C::SPB + sub * C::TT;   // position of tile row 0

        // ---- segment start: load the GQA group's queries as mma B fragments ----
        if (i == 0 || first) {
            const int r = __shfl_sync(0xffffffffu, cur.r, src);
            const int h = __shfl_sync(0xffffffffu, cur.h, src);
            seg_full = first;
            seg_r = r;
            seg_h = h;
            query_rows<QT>(a, r, seg_qb, seg_qlen, errbits);
            seg_vis = s_seq[r] - seg_qlen;
#pragma unroll
            for (int qi = 0; qi < QT; ++qi) {
                m0[qi] = m1[qi] = -INFINITY;
                l0[qi] = l1[qi] = 0.f;
                cr0[qi] = cr1[qi] = 0.f;
#pragma unroll
                for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[dt][qi][e] = 0.f;
            }
            if (!FP8) {
#pragma unroll
                for (int qi = 0; qi < QT; ++qi) {
                    const bool gv = g < a.G && qi < seg_qlen;
                    const uint16_t* qrow =
                        a.q + ((int64_t)(seg_qb + qi) * a.Hq + (int64_t)h * a.G + g) * D;
#pragma unroll
                    for (int ks2 = 0; ks2 < C::KS; ++ks2) {
                        const uint32_t b0 = gv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + ks2 * 16 + 2 * c)) : 0u;
                        const uint32_t b1 = gv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + ks2 * 16 + 8 + 2 * c)) : 0u;
                        if constexpr (QSMEM) {
                            qs[(ks2 * QT + qi) * 32 + lane] = make_uint2(b0, b1);   // own slots
                        } else {
                            qf[ks2][qi][0] = b0;
                            qf[ks2][qi][1] = b1;
                        }
                    }
                }
                qscale = a.scale_log2;
            } else if constexpr (C::I4) {
                // k-slot mapping for int4 A fragments (see the K path): for mma (dblk, i),
                // slots 2c,2c+1 <-> d = 64 dblk + 8c + i, +4 and slots 8+2c,9+2c <->
                // d = 64 dblk + 32 + 8c + i, +4.  Group gi of this lane: d = 32 gi + 8c + 0..7.
                uint4 raw4[4][QT];
                float amax = 0.f;
#pragma unroll
                for (int qi = 0; qi < QT; ++qi) {
                    const bool gv = g < a.G && qi < seg_qlen;
                    const uint16_t* qrow =
                        a.q + ((int64_t)(seg_qb + qi) * a.Hq + (int64_t)h * a.G + g) * D;
#pragma unroll
                    for (int gi = 0; gi < 4; ++gi) {
                        raw4[gi][qi] = gv ? __ldg(reinterpret_cast<const uint4*>(qrow + 32 * gi + 8 * c))
                                          : make_uint4(0u, 0u, 0u, 0u);
                        const uint32_t w4[4] = {raw4[gi][qi].x, raw4[gi][qi].y, raw4[gi][qi].z,
                                                raw4[gi][qi].w};
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo_to_f32(w4[k])),
                                                     fabsf(bf16_hi_to_f32(w4[k]))));
                    }
                }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
                int E = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
                E = max(E, 15);
                const float sc = __uint_as_float((uint32_t)(268 - E) << 23);
                const float inv_sc = __uint_as_float((uint32_t)(E - 14) << 23);
                auto qv = [&](const uint4& u, int j) {   // bf16 value j (0..7) of u, as fp32
                    const uint32_t w = j < 2 ? u.x : (j < 4 ? u.y : (j < 6 ? u.z : u.w));
                    return (j & 1) ? bf16_hi_to_f32(w) : bf16_lo_to_f32(w);
                };
#pragma unroll
                for (int qi = 0; qi < QT; ++qi)
#pragma unroll
                    for (int dblk = 0; dblk < 2; ++dblk)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4& A = raw4[2 * dblk][qi];
                            const uint4& B = raw4[2 * dblk + 1][qi];
                            // odd picks hold 16 n: their q carries the 1/16 (exact)
                            const float si = (i & 1) ? sc * 0.0625f : sc;
                            qf[dblk * 4 + i][qi][0] = pack_f16x2(qv(A, i) * si, qv(A, i + 4) * si);
                            qf[dblk * 4 + i][qi][1] = pack_f16x2(qv(B, i) * si, qv(B, i + 4) * si);
                        }
                // the scores' constant part: the same mma over a tile of code-0 nibbles
                // (1032 for even picks, 1152 for odd), one value per head
#pragma unroll
                for (int qi = 0; qi < QT; ++qi) {
                    float cacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t k0 = (kk & 1) ? 0x64806480u : 0x64086408u;
                        mma_f16(cacc, k0, k0, k0, k0, qf[kk][qi][0], qf[kk][qi][1]);
                    }
                    cq0[qi] = cacc[0];
                    cq1[qi] = cacc[1];
                }
                qscale = a.scale_log2 * inv_sc;
            } else {
                // k-slot mapping for E4M3 A fragments: slots 2c,2c+1 <-> d = 4c,4c+1 and
                // slots 8+2c,9+2c <-> d = 4c+2,4c+3 of each 16-d step.
                uint2 raw_q[C::KS][QT];
                float amax = 0.f;
#pragma unroll
                for (int qi = 0; qi < QT; ++qi) {
                    const bool gv = g < a.G && qi < seg_qlen;
                    const uint16_t* qrow =
                        a.q + ((int64_t)(seg_qb + qi) * a.Hq + (int64_t)h * a.G + g) * D;
#pragma unroll
                    for (int ks2 = 0; ks2 < C::KS; ++ks2) {
                        raw_q[ks2][qi] = gv ? __ldg(reinterpret_cast<const uint2*>(qrow + ks2 * 16 + 4 * c))
                                            : make_uint2(0u, 0u);
                        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo_to_f32(raw_q[ks2][qi].x)),
                                                       fabsf(bf16_hi_to_f32(raw_q[ks2][qi].x))),
                                                 fmaxf(fabsf(bf16_lo_to_f32(raw_q[ks2][qi].y)),
                                                       fabsf(bf16_hi_to_f32(raw_q[ks2][qi].y)))));
                    }
                }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
                // power of two putting the largest |q| in [2^14, 2^15): exact rescale
                // (E >= 15 keeps both 2^(141-E) and 2^(E-141) normal binary32 numbers)
                int E = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
                E = max(E, 15);
                const float sc = __uint_as_float((uint32_t)(268 - E) << 23);
                const float inv_sc = __uint_as_float((uint32_t)(E - 14) << 23);
#pragma unroll
                for (int qi = 0; qi < QT; ++qi)
#pragma unroll
                    for (int ks2 = 0; ks2 < C::KS; ++ks2) {
                        qf[ks2][qi][0] = pack_f16x2(bf16_lo_to_f32(raw_q[ks2][qi].x) * sc,
                                                    bf16_hi_to_f32(raw_q[ks2][qi].x) * sc);
                        qf[ks2][qi][1] = pack_f16x2(bf16_lo_to_f32(raw_q[ks2][qi].y) * sc,
                                                    bf16_hi_to_f32(raw_q[ks2][qi].y) * sc);
                    }
                if constexpr (KT == 2) {
                    // the scores' constant part: the same mma over a tile of code-0 bytes
                    // (1024 + 128), one value per head
#pragma unroll
                    for (int qi = 0; qi < QT; ++qi) {
                        float cacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int ks2 = 0; ks2 < C::KS; ++ks2)
                            mma_f16(cacc, 0x64806480u, 0x64806480u, 0x64806480u, 0x64806480u,
                                    qf[ks2][qi][0], qf[ks2][qi][1]);
                        cq0[qi] = cacc[0];
                        cq1[qi] = cacc[1];
                    }
                }
                qscale = a.scale_log2 * inv_sc;
            }
        }

        // ---- wait for the tile ----
        bool ok = mbar_wait_bounded(bars + 8u * s, par, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) atomicOr(a.err, PKV_DEVERR_WAIT_TIMEOUT | errbits);
            for (int k = i; k < min(i + S, total); ++k)
                (void)mbar_wait_bounded(bars + 8u * (k % S), (uint32_t)((k / S) & 1), kWaitLimitNs);
            __syncwarp();
            return;
        }
        const uint32_t kpg = stage0 + (uint32_t)(s * C::STAGE_BYTES);
        const uint32_t vpg = kpg + C::TILE_BYTES;

        // rows past the request's length hold stale data: zero them in V so that
        // P = 0 times them stays 0 even if they hold NaN patterns
        if (C::I4 && ntok < C::TT) {
            uint8_t* vp = basep + (vpg - base);
            const int t0 = max(ntok, 0);
            constexpr int UPR = C::ROW_BYTES / 16;          // 16-byte units per row
            for (int u = lane; u < (C::TT - t0) * UPR; u += 32)
                *reinterpret_cast<uint4*>(vp + (t0 + u / UPR) * C::ROW_BYTES + (u % UPR) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            __syncwarp();
        } else if (ntok < C::TT) {
            uint8_t* vp = basep + (vpg - base);
            const int t0 = max(ntok, 0);
            const int units = (C::TT - t0) * C::CH * 8;   // 16-byte units
            for (int u = lane; u < units; u += 32) {
                const int ch = u / ((C::TT - t0) * 8);
                const int rem = u - ch * ((C::TT - t0) * 8);
                const int t = t0 + rem / 8;
                const int k16 = rem & 7;
                *reinterpret_cast<uint4*>(vp + ch * (C::TT * 128) + t * 128 + k16 * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }

        // ---- append: the request's newest token into the cache and into this tile ----
        if constexpr (KT == 0 && QT == 1) {
            if (a.k_new != nullptr && ((fl >> 9) & 1u) && ntok >= 1 && ntok <= C::TT &&
                tpos0 + ntok == s_seq[seg_r]) {
                const int tr = ntok - 1;                   // tile row of the token
                const int prow = __shfl_sync(0xffffffffu, cur.row[0], src);   // block * Hkv + h
                constexpr int EPL = D / 32;                // elements per lane
                const int d0 = lane * EPL;
                const int64_t in = ((int64_t)seg_r * a.Hkv + seg_h) * D + d0;
                // the 128-byte swizzled tile layout the TMA wrote
                const uint32_t so = (uint32_t)((d0 / 64) * (C::TT * 128) + tr * 128 +
                                               ((((d0 % 64) / 8) ^ (tr & 7)) << 4) + (d0 % 8) * 2);
                const bool in_pool = prow < a.NB * a.Hkv;
                const int64_t go = ((int64_t)prow * BS + (tpos0 % BS) + tr) * D + d0;
                if constexpr (EPL == 4) {
                    const uint2 kv = __ldg(reinterpret_cast<const uint2*>(a.k_new + in));
                    const uint2 vv = __ldg(reinterpret_cast<const uint2*>(a.v_new + in));
                    *reinterpret_cast<uint2*>(basep + (kpg - base) + so) = kv;
                    *reinterpret_cast<uint2*>(basep + (vpg - base) + so) = vv;
                    if (in_pool) {
                        *reinterpret_cast<uint2*>(a.k_cache_w + go) = kv;
                        *reinterpret_cast<uint2*>(a.v_cache_w + go) = vv;
                    }
                } else {
                    const uint32_t kv = __ldg(reinterpret_cast<const uint32_t*>(a.k_new + in));
                    const uint32_t vv = __ldg(reinterpret_cast<const uint32_t*>(a.v_new + in));
                    *reinterpret_cast<uint32_t*>(basep + (kpg - base) + so) = kv;
                    *reinterpret_cast<uint32_t*>(basep + (vpg - base) + so) = vv;
                    if (in_pool) {
                        *reinterpret_cast<uint32_t*>(a.k_cache_w + go) = kv;
                        *reinterpret_cast<uint32_t*>(a.v_cache_w + go) = vv;
                    }
                }
                __syncwarp();
            }
        }

        // ---- S^T = K Q^T (tokens x heads), one n-tile per query position ----
        float sacc[C::MT][QT][4];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
            float e0[QT][4], e1[QT][4];
#pragma unroll
            for (int qi = 0; qi < QT; ++qi)
#pragma unroll
                for (int e = 0; e < 4; ++e) e0[qi][e] = e1[qi][e] = 0.f;
            const int t = mt * 16 + (lane & 15);
            if (!FP8) {
#pragma unroll
                for (int ks2 = 0; ks2 < C::KS; ++ks2) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kpg + swz<C::TT>(t, 2 * ks2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
                    for (int qi = 0; qi < QT; ++qi) {
                        uint32_t b0, b1;
                        if constexpr (QSMEM) {
                            const uint2 bq = qs[(ks2 * QT + qi) * 32 + lane];
                            b0 = bq.x;
                            b1 = bq.y;
                        } else {
                            b0 = qf[ks2][qi][0];
                            b1 = qf[ks2][qi][1];
                        }
                        // two accumulator chains give the single-query case its ILP; with
                        // several query tiles the tiles themselves are independent
                        if (QT == 1 && (ks2 & 1)) mma_bf16(e1[qi], a0, a1, a2, a3, b0, b1);
                        else                      mma_bf16(e0[qi], a0, a1, a2, a3, b0, b1);
                    }
                }
            } else if constexpr (C::I4) {
                // int4 rows: a 32-byte d-block (64 values) of tokens 0-7 / 8-15, bytes
                // 0-15 / 16-31 as the four 8x8 b16 matrices; each 32-bit register holds 8
                // nibbles (d = 64 dblk + 8c + 0..7 of token g, or +32 / token g+8)
                const int tr = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int dblk = 0; dblk < D / 64; ++dblk) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(kpg + swz64(tr, dblk * 2 + (lane >> 4)), r0, r1, r2, r3);
#pragma unroll
                    for (int qi = 0; qi < QT; ++qi) {
                        mma_f16(e0[qi], i4pick_raw<0>(r0), i4pick_raw<0>(r1),
                                i4pick_raw<0>(r2), i4pick_raw<0>(r3),
                                qf[dblk * 4][qi][0], qf[dblk * 4][qi][1]);
                        mma_f16(QT == 1 ? e1[qi] : e0[qi], i4pick_raw<1>(r0),
                                i4pick_raw<1>(r1), i4pick_raw<1>(r2),
                                i4pick_raw<1>(r3), qf[dblk * 4 + 1][qi][0],
                                qf[dblk * 4 + 1][qi][1]);
                        mma_f16(e0[qi], i4pick_raw<2>(r0), i4pick_raw<2>(r1),
                                i4pick_raw<2>(r2), i4pick_raw<2>(r3),
                                qf[dblk * 4 + 2][qi][0], qf[dblk * 4 + 2][qi][1]);
                        mma_f16(QT == 1 ? e1[qi] : e0[qi], i4pick_raw<3>(r0),
                                i4pick_raw<3>(r1), i4pick_raw<3>(r2),
                                i4pick_raw<3>(r3), qf[dblk * 4 + 3][qi][0],
                                qf[dblk * 4 + 3][qi][1]);
                    }
                }
            } else {
#pragma unroll
                for (int kp = 0; kp < C::KS / 2; ++kp) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(kpg + swz<C::TT>(t, 2 * kp + (lane >> 4)), r0, r1, r2, r3);
                    uint32_t k00, k01, k02, k03, k10, k11, k12, k13;
                    if constexpr (KT == 2) {
                        // int8: one sign flip per register, then gather + widen per pair
                        const uint32_t s0 = r0 ^ 0x80808080u, s1 = r1 ^ 0x80808080u;
                        const uint32_t s2 = r2 ^ 0x80808080u, s3 = r3 ^ 0x80808080u;
                        k00 = i8pick_raw<0x5140>(s0); k02 = i8pick_raw<0x7362>(s0);
                        k01 = i8pick_raw<0x5140>(s1); k03 = i8pick_raw<0x7362>(s1);
                        k10 = i8pick_raw<0x5140>(s2); k12 = i8pick_raw<0x7362>(s2);
                        k11 = i8pick_raw<0x5140>(s3); k13 = i8pick_raw<0x7362>(s3);
                    } else {
                        k00 = b8x2_to_f16x2<KT>(r0); k01 = b8x2_to_f16x2<KT>(r1);
                        k02 = b8x2_to_f16x2<KT>(r0 >> 16); k03 = b8x2_to_f16x2<KT>(r1 >> 16);
                        k10 = b8x2_to_f16x2<KT>(r2); k11 = b8x2_to_f16x2<KT>(r3);
                        k12 = b8x2_to_f16x2<KT>(r2 >> 16); k13 = b8x2_to_f16x2<KT>(r3 >> 16);
                    }
#pragma unroll
                    for (int qi = 0; qi < QT; ++qi) {
                        mma_f16(e0[qi], k00, k01, k02, k03, qf[2 * kp][qi][0], qf[2 * kp][qi][1]);
                        mma_f16(QT == 1 ? e1[qi] : e0[qi], k10, k11, k12, k13, qf[2 * kp + 1][qi][0],
                                qf[2 * kp + 1][qi][1]);
                    }
                }
            }
#pragma unroll
            for (int qi = 0; qi < QT; ++qi)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[mt][qi][e] = e0[qi][e] + e1[qi][e];
        }

        // ---- online softmax (log2 domain), heads 2c and 2c+1 of this lane ----
        float mx0[QT], mx1[QT];
        bool need = false;
        // every row of a full tile is a cached token every query sees: no mask
        const bool full_tile = QT == 1 && ntok >= C::TT;
#pragma unroll
        for (int qi = 0; qi < QT; ++qi) {
            mx0[qi] = mx1[qi] = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                // the K scale of the block holding these 16 tokens; int8 / int4:
                // score = (sum - cq) * scale, one fma
                const float sc_page = FP8 ? qscale * ks[mt / C::MTB] : qscale;
                const float nc0 = C::FOLD ? -cq0[qi] * sc_page : 0.f;
                const float nc1 = C::FOLD ? -cq1[qi] * sc_page : 0.f;
                if (full_tile) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sacc[mt][qi][e] = C::FOLD ? fmaf(sacc[mt][qi][e], sc_page, (e & 1) ? nc1 : nc0)
                                                  : sacc[mt][qi][e] * sc_page;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tok = mt * 16 + g + ((e & 2) ? 8 : 0);
                        bool valid = tok < ntok;
                        if constexpr (QT > 1) valid = valid && (tpos0 + tok <= seg_vis + qi);
                        const float v = C::FOLD ? fmaf(sacc[mt][qi][e], sc_page, (e & 1) ? nc1 : nc0)
                                                : sacc[mt][qi][e] * sc_page;
                        sacc[mt][qi][e] = valid ? v : -INFINITY;
                    }
                }
                mx0[qi] = fmaxf(mx0[qi], fmaxf(sacc[mt][qi][0], sacc[mt][qi][2]));
                mx1[qi] = fmaxf(mx1[qi], fmaxf(sacc[mt][qi][1], sacc[mt][qi][3]));
            }
            // raise the running max (and rescale O and l) only when some lane's score
            // exceeds it by more than the slack; P <= 2^kRescaleSlack otherwise
            need = need || (mx0[qi] > m0[qi] + kRescaleSlack) || (mx1[qi] > m1[qi] + kRescaleSlack);
        }
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int qi = 0; qi < QT; ++qi) {
#pragma unroll
                for (int o2 = 4; o2 < 32; o2 <<= 1) {
                    mx0[qi] = fmaxf(mx0[qi], __shfl_xor_sync(0xffffffffu, mx0[qi], o2));
                    mx1[qi] = fmaxf(mx1[qi], __shfl_xor_sync(0xffffffffu, mx1[qi], o2));
                }
                const float mn0 = fmaxf(m0[qi], mx0[qi]), mn1 = fmaxf(m1[qi], mx1[qi]);
                float al0 = ex2_approx(m0[qi] - mn0), al1 = ex2_approx(m1[qi] - mn1);
                if constexpr (QT > 1) {
                    // a query that has seen no token yet keeps -inf without a NaN
                    if (mn0 == -INFINITY) al0 = 1.f;
                    if (mn1 == -INFINITY) al1 = 1.f;
                }
                m0[qi] = mn0;
                m1[qi] = mn1;
                l0[qi] *= al0;
                l1[qi] *= al1;
                cr0[qi] *= al0;
                cr1[qi] *= al1;
#pragma unroll
                for (int dt = 0; dt < C::DT; ++dt) {
                    o[dt][qi][0] *= al0;
                    o[dt][qi][2] *= al0;
                    o[dt][qi][1] *= al1;
                    o[dt][qi][3] *= al1;
                }
            }
        }
        uint32_t pb[C::MT][QT][2];
#pragma unroll
        for (int qi = 0; qi < QT; ++qi) {
            float r0m = m0[qi], r1m = m1[qi];
            if constexpr (QT > 1) {
                if (r0m == -INFINITY) r0m = 0.f;   // every score of that head is -inf here
                if (r1m == -INFINITY) r1m = 0.f;
            }
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                const float p0 = ex2_approx(sacc[mt][qi][0] - r0m), p1 = ex2_approx(sacc[mt][qi][1] - r1m);
                const float p2 = ex2_approx(sacc[mt][qi][2] - r0m), p3 = ex2_approx(sacc[mt][qi][3] - r1m);
                ps0 += p0 + p2;
                ps1 += p1 + p3;
                if (!FP8) {
                    pb[mt][qi][0] = movmatrix_trans(pack_bf16x2(p0, p1));
                    pb[mt][qi][1] = movmatrix_trans(pack_bf16x2(p2, p3));
                } else {
                    // quantised pages: P carries the block's V scale into the mma
                    const float vsb = vs[mt / C::MTB];
                    pb[mt][qi][0] = movmatrix_trans(pack_f16x2(p0 * vsb, p1 * vsb));
                    pb[mt][qi][1] = movmatrix_trans(pack_f16x2(p2 * vsb, p3 * vsb));
                }
            }
            l0[qi] += ps0;
            l1[qi] += ps1;
        }

        // ---- O^T += V^T P^T ----
        if (!FP8) {
#pragma unroll
            for (int dt = 0; dt < C::DT; ++dt) {
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    const int t = mt * 16 + (lane & 7) + ((lane >> 4) << 3);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_trans(vpg + swz<C::TT>(t, 2 * dt + ((lane >> 3) & 1)), a0, a1, a2, a3);
#pragma unroll
                    for (int qi = 0; qi < QT; ++qi)
                        mma_bf16(o[dt][qi], a0, a1, a2, a3, pb[mt][qi][0], pb[mt][qi][1]);
                }
            }
        } else {
            // P already holds P * v_scale (fp16), so every page accumulates into O
            if constexpr (C::I4) {
                // the K-path matrices, transposed per 8x8 b16 block by the load: a lane holds
                // tokens 2c, 2c+1 of b16 unit g (d = 64 dblk + 4g + 0..3), and nibble pair
                // (j, j + 4) is one d for both tokens.  mma (dblk, i): V^T row g <-> d =
                // 64 dblk + 4g + i, row g + 8 <-> d = 64 dblk + 32 + 4g + i.
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    const int tr = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int dblk = 0; dblk < D / 64; ++dblk) {
                        // m0: tokens 0-7, d + 0; m1: tokens 8-15, d + 0; m2: tokens 0-7,
                        // d + 32; m3: tokens 8-15, d + 32
                        uint32_t m0, m1, m2, m3;
                        ldsm_x4_trans(vpg + swz64(tr, dblk * 2 + (lane >> 4)), m0, m1, m2, m3);
#pragma unroll
                        for (int qi = 0; qi < QT; ++qi) {
                            mma_f16(o[dblk * 4][qi], i4pick_sub<0>(m0), i4pick_sub<0>(m2),
                                    i4pick_sub<0>(m1), i4pick_sub<0>(m3),
                                    pb[mt][qi][0], pb[mt][qi][1]);
                            mma_f16(o[dblk * 4 + 1][qi], i4pick_sub<1>(m0),
                                    i4pick_sub<1>(m2), i4pick_sub<1>(m1),
                                    i4pick_sub<1>(m3), pb[mt][qi][0], pb[mt][qi][1]);
                            mma_f16(o[dblk * 4 + 2][qi], i4pick_sub<2>(m0),
                                    i4pick_sub<2>(m2), i4pick_sub<2>(m1),
                                    i4pick_sub<2>(m3), pb[mt][qi][0], pb[mt][qi][1]);
                            mma_f16(o[dblk * 4 + 3][qi], i4pick_sub<3>(m0),
                                    i4pick_sub<3>(m2), i4pick_sub<3>(m1),
                                    i4pick_sub<3>(m3), pb[mt][qi][0], pb[mt][qi][1]);
                        }
                    }
                }
            } else {
#pragma unroll
            for (int dp = 0; dp < C::DT / 2; ++dp) {
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    const int t = mt * 16 + (lane & 15);
                    // the four 8x8 b16 blocks, each transposed by the load
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_trans(vpg + swz<C::TT>(t, 2 * dp + (lane >> 4)), r0, r1, r2, r3);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t x = half ? r2 : r0;   // tokens 0-7
                        const uint32_t y = half ? r3 : r1;   // tokens 8-15
                        uint32_t v0, v1, v2, v3;
                        if constexpr (KT == 2) {
                            // int8: the token regroup and the widening are one permute
                            const uint32_t xs = x ^ 0x80808080u, ys = y ^ 0x80808080u;
                            v0 = i8pick_sub<0x5240>(xs);
                            v1 = i8pick_sub<0x5341>(xs);
                            v2 = i8pick_sub<0x5240>(ys);
                            v3 = i8pick_sub<0x5341>(ys);
                        } else {
                            v0 = b8x2_to_f16x2<KT>(__byte_perm(x, 0u, 0x0020));
                            v1 = b8x2_to_f16x2<KT>(__byte_perm(x, 0u, 0x0031));
                            v2 = b8x2_to_f16x2<KT>(__byte_perm(y, 0u, 0x0020));
                            v3 = b8x2_to_f16x2<KT>(__byte_perm(y, 0u, 0x0031));
                        }
#pragma unroll
                        for (int qi = 0; qi < QT; ++qi)
                            mma_f16(o[2 * dp + half][qi], v0, v1, v2, v3, pb[mt][qi][0],
                                    pb[mt][qi][1]);
                    }
                }
            }
            }
            if constexpr (C::FOLD) {
                // sum(P * v_scale) per head as the mma sees it (fp16 against a tile of
                // ones): the offset part of this page's P.V is that times 128 (int8) or 8
                // (int4), in units of 2^-24
#pragma unroll
                for (int qi = 0; qi < QT; ++qi) {
                    float psum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int mt = 0; mt < C::MT; ++mt)
                        mma_f16(psum, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u,
                                pb[mt][qi][0], pb[mt][qi][1]);
                    cr0[qi] += psum[0];
                    cr1[qi] += psum[1];
                }
            }
        }

        // ---- segment end ----
        if (last || i == total - 1) {
            const int g0 = 2 * c, g1 = 2 * c + 1;
            const bool complete = seg_full && last && a.cascade_part == nullptr;
            const int64_t u = (int64_t)seg_r * a.Hkv + seg_h;
            const int64_t slot = u + gw;
#pragma unroll
            for (int qi = 0; qi < QT; ++qi) {
                if (qi >= seg_qlen) break;
                if constexpr (C::FOLD) {
                    // back from subnormal units (2^24; int4 odd picks held 16 n: 2^20),
                    // then remove the offsets' share: 128 (int8) or 8 (int4) per unit of cr
                    const float k = C::I4 ? 8.f : 128.f;
#pragma unroll
                    for (int dt = 0; dt < C::DT; ++dt) {
                        const float u = (C::I4 && (dt & 1)) ? 1048576.f : 16777216.f;
                        o[dt][qi][0] = fmaf(o[dt][qi][0], u, -k * cr0[qi]);
                        o[dt][qi][2] = fmaf(o[dt][qi][2], u, -k * cr0[qi]);
                        o[dt][qi][1] = fmaf(o[dt][qi][1], u, -k * cr1[qi]);
                        o[dt][qi][3] = fmaf(o[dt][qi][3], u, -k * cr1[qi]);
                    }
                }
                float L0 = l0[qi], L1 = l1[qi];
#pragma unroll
                for (int o2 = 4; o2 < 32; o2 <<= 1) {
                    L0 += __shfl_xor_sync(0xffffffffu, L0, o2);
                    L1 += __shfl_xor_sync(0xffffffffu, L1, o2);
                }
                if (complete) {
                    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f;
                    const float inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
                    uint16_t* ob =
                        a.out + ((int64_t)(seg_qb + qi) * a.Hq + (int64_t)seg_h * a.G) * D;
#pragma unroll
                    for (int dt = 0; dt < C::DT; ++dt) {
                        if constexpr (C::I4) {
                            // accumulator dt = 4 dblk + i: row g <-> d, row g + 8 <-> d + 32
                            const int d = (dt >> 2) * 64 + 4 * g + (dt & 3);
                            if (g0 < a.G) {
                                ob[g0 * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o[dt][qi][0] * inv0));
                                ob[g0 * D + d + 32] = __bfloat16_as_ushort(__float2bfloat16_rn(o[dt][qi][2] * inv0));
                            }
                            if (g1 < a.G) {
                                ob[g1 * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o[dt][qi][1] * inv1));
                                ob[g1 * D + d + 32] = __bfloat16_as_ushort(__float2bfloat16_rn(o[dt][qi][3] * inv1));
                            }
                        } else if (!FP8) {
                            const int d = dt * 16 + g;
                            if (g0 < a.G) {
                                ob[g0 * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o[dt][qi][0] * inv0));
                                ob[g0 * D + d + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(o[dt][qi][2] * inv0));
                            }
                            if (g1 < a.G) {
                                ob[g1 * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o[dt][qi][1] * inv1));
                                ob[g1 * D + d + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(o[dt][qi][3] * inv1));
                            }
                        } else {
                            const int d = dt * 16 + 2 * g;
                            if (g0 < a.G)
                                *reinterpret_cast<uint32_t*>(ob + g0 * D + d) =
                                    pack_bf16x2(o[dt][qi][0] * inv0, o[dt][qi][2] * inv0);
                            if (g1 < a.G)
                                *reinterpret_cast<uint32_t*>(ob + g1 * D + d) =
                                    pack_bf16x2(o[dt][qi][1] * inv1, o[dt][qi][3] * inv1);
                        }
                    }
                } else {
                    float* ps = a.partials + slot * (QT * kGroupPad * (D + 4)) +
                                qi * (kGroupPad * (D + 4));
#pragma unroll
                    for (int dt = 0; dt < C::DT; ++dt) {
                        if constexpr (C::I4) {
                            const int d = (dt >> 2) * 64 + 4 * g + (dt & 3);
                            ps[g0 * (D + 4) + d] = o[dt][qi][0];
                            ps[g0 * (D + 4) + d + 32] = o[dt][qi][2];
                            ps[g1 * (D + 4) + d] = o[dt][qi][1];
                            ps[g1 * (D + 4) + d + 32] = o[dt][qi][3];
                        } else if (!FP8) {
                            const int d = dt * 16 + g;
                            ps[g0 * (D + 4) + d] = o[dt][qi][0];
                            ps[g0 * (D + 4) + d + 8] = o[dt][qi][2];
                            ps[g1 * (D + 4) + d] = o[dt][qi][1];
                            ps[g1 * (D + 4) + d + 8] = o[dt][qi][3];
                        } else {
                            const int d = dt * 16 + 2 * g;
                            *reinterpret_cast<float2*>(ps + g0 * (D + 4) + d) = make_float2(o[dt][qi][0], o[dt][qi][2]);
                            *reinterpret_cast<float2*>(ps + g1 * (D + 4) + d) = make_float2(o[dt][qi][1], o[dt][qi][3]);
                        }
                    }
                    if (g == 0) {
                        *reinterpret_cast<float2*>(ps + g0 * (D + 4) + D) = make_float2(m0[qi], L0);
                        *reinterpret_cast<float2*>(ps + g1 * (D + 4) + D) = make_float2(m1[qi], L1);
                    }
                }
            }
        }

        // every lane orders its generic accesses of this stage (ldmatrix reads, the
        // zero fill) before the async-proxy refill lane 0 is about to issue
        fence_proxy_async_smem();
        __syncwarp();
        if (i + S < total) issue(i + S, s);   // item i + S reuses stage s
        if (++s == S) {
            s = 0;
            par ^= 1u;
        }
    }
    if (errbits) atomicOr(a.err, errbits);
}

// Log-sum-exp merge of the units split over several warps:
//   M = max_w m_w,  out = sum_w 2^(m_w - M) o_w / sum_w 2^(m_w - M) l_w
// ("GPU推理深度拆解：KV Cache视角", 系统层：Context Parallel: the online-softmax merge
// that ring attention also uses).  One CTA per unit and one warp per (query head of the
// group, query position); each lane owns D/32 columns.  Lane k holds partial k's (m, l),
// so the weights reach the column loop by shuffle instead of another round of loads, and
// the loop keeps several partials' loads in flight.  Runs after the decode kernel
// (programmatic dependent launch: it waits for the decode grid to complete).
template <int D, int QT>
__global__ void __launch_bounds__(kGroupPad * 32 * QT)
    pkv_decode_merge_kernel(const DecodeArgs a) {
    constexpr int PER = D / 32;
    constexpr int QS = kGroupPad * (D + 4);
    constexpr int SLOT = QT * QS;
    pdl_wait();
    const int u = blockIdx.x;
    const int wi = threadIdx.x >> 5;
    const int gg = wi % kGroupPad, qi = wi / kGroupPad;
    const int lane = threadIdx.x & 31;
    if (gg >= a.G) return;
    const int r = u / a.Hkv;
    const int h = u - r * a.Hkv;
    const int P = a.g_prefix[a.N];
    const int p0 = a.g_prefix[r], p1 = a.g_prefix[r + 1];
    int qb, qlen;
    uint32_t errbits = 0;
    query_rows<QT>(a, r, qb, qlen, errbits);
    const int W = min(a.total_warps, P);
    const int np = (p1 - p0) / a.Hkv;
    if (np == 0 || qi >= qlen) return;
    const int64_t U = (int64_t)p0 + (int64_t)h * np;
    const int64_t E = U + np - 1;
    const int wf = (int)(((U + 1) * W - 1) / P);
    const int wl = (int)(((E + 1) * W - 1) / P);
    const int n = wl - wf + 1;
    if (n == 1) return;   // a whole unit: the decode kernel wrote its output
    static_assert(PER == 2 || PER == 4, "head_dim 64 or 128");
    using Row = typename std::conditional<PER == 4, float4, float2>::type;
    const float* base = a.partials + ((int64_t)u + wf) * SLOT + qi * QS + gg * (D + 4);
    // the first eight partials' rows go out with the (m, l) loads: their addresses do not
    // depend on the maximum
    Row v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < n) v[j] = *reinterpret_cast<const Row*>(base + (int64_t)j * SLOT + lane * PER);
        else v[j] = Row{};
    }
    // (m, l) of partial `lane` (and of lane + 32, ... for wider units)
    const float2 ml0 = lane < n ? *reinterpret_cast<const float2*>(base + (int64_t)lane * SLOT + D)
                                : make_float2(-INFINITY, 0.f);
    float M = ml0.x;
    for (int k = lane + 32; k < n; k += 32)
        M = fmaxf(M, base[(int64_t)k * SLOT + D]);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float acc[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c) acc[c] = 0.f;
    float L = 0.f;
    if (M != -INFINITY) {   // else: the query saw no token: zero row
        const float w0 = lane < n ? exp2f(ml0.x - M) : 0.f;   // weight of partial `lane`
        L = w0 * ml0.y;
        for (int k = lane + 32; k < n; k += 32) {
            const float2 ml = *reinterpret_cast<const float2*>(base + (int64_t)k * SLOT + D);
            L = fmaf(exp2f(ml.x - M), ml.y, L);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
        // 32 partials at a time: lane j holds the weight of partial c0 + j.  Rows are loaded
        // eight at a time before any of them is used; a row past the end loads as zero and
        // its lane's weight is zero, so the sum over k keeps its order and value.
        for (int c0 = 0; c0 < n; c0 += 32) {
            const float wc = c0 == 0 ? w0
                             : (c0 + lane < n ? exp2f(base[(int64_t)(c0 + lane) * SLOT + D] - M)
                                              : 0.f);
            const int nc = min(n - c0, 32);
            for (int k = 0; k < nc; k += 8) {
                if (c0 != 0 || k != 0) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float* ps = base + (int64_t)(c0 + k + j) * SLOT + lane * PER;
                        if (k + j < nc) v[j] = *reinterpret_cast<const Row*>(ps);
                        else v[j] = Row{};
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float wt = __shfl_sync(0xffffffffu, wc, k + j);
                    const float* f = reinterpret_cast<const float*>(&v[j]);
#pragma unroll
                    for (int c = 0; c < PER; ++c) acc[c] = fmaf(wt, f[c], acc[c]);
                }
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* ob = a.out + ((int64_t)(qb + qi) * a.Hq + (int64_t)h * a.G + gg) * D;
#pragma unroll
    for (int c = 0; c < PER; c += 2)
        *reinterpret_cast<uint32_t*>(ob + lane * PER + c) =
            pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
}

// The shared-prefix merge: per (request, query head), the unit's decode partials over
// its private pages and the prefix pass's partials over the shared pages, merged with
// the same log-sum-exp weights as pkv_decode_merge_kernel (one query position).  One
// CTA per unit, one warp per query head; lane k holds partial k's (m, l) and each lane
// owns D/32 columns.
template <int D>
__global__ void __launch_bounds__(kGroupPad * 32)
    pkv_cascade_merge_kernel(const DecodeArgs a) {
    constexpr int PER = D / 32;
    constexpr int QS = kGroupPad * (D + 4);
    pdl_wait();
    const int u = blockIdx.x;
    const int gg = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (gg >= a.G) return;
    const int r = u / a.Hkv;
    const int h = u - r * a.Hkv;
    const int P = a.g_prefix[a.N];
    const int p0 = a.g_prefix[r], p1 = a.g_prefix[r + 1];
    const int np = (p1 - p0) / a.Hkv;
    int wf = 0, n = 0;   // the unit's decode partials: slots u + wf .. u + wf + n - 1
    if (np > 0) {
        const int W = min(a.total_warps, P);
        const int64_t U = (int64_t)p0 + (int64_t)h * np;
        const int64_t E = U + np - 1;
        wf = (int)(((U + 1) * W - 1) / P);
        n = (int)(((E + 1) * W - 1) / P) - wf + 1;
    }
    const int C = a.cascade_split;
    const int T = n + C;   // all partials of this (request, head)
    const float* dp = a.partials + ((int64_t)u + wf) * QS + gg * (D + 4);
    const float* pp = a.cascade_part + ((int64_t)r * a.Hq + (int64_t)h * a.G + gg) * C * (D + 4);
    auto row = [&](int k) { return k < n ? dp + (int64_t)k * QS : pp + (int64_t)(k - n) * (D + 4); };
    static_assert(PER == 2 || PER == 4, "head_dim 64 or 128");
    using Row = typename std::conditional<PER == 4, float4, float2>::type;
    // lane k holds partial k's (m, l); further partials (more than 32) are folded in by
    // the lane-strided loops
    float2 ml0 = make_float2(-INFINITY, 0.f);
    if (lane < T) ml0 = *reinterpret_cast<const float2*>(row(lane) + D);
    float M = ml0.x;
    for (int k = lane + 32; k < T; k += 32) M = fmaxf(M, row(k)[D]);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float acc[PER];
#pragma unroll
    for (int c = 0; c < PER; ++c) acc[c] = 0.f;
    float L = 0.f;
    if (M != -INFINITY) {
        const float w0 = lane < T ? exp2f(ml0.x - M) : 0.f;   // weight of partial `lane`
        L = w0 * ml0.y;
        for (int k = lane + 32; k < T; k += 32) {
            const float2 ml = *reinterpret_cast<const float2*>(row(k) + D);
            L = fmaf(exp2f(ml.x - M), ml.y, L);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
        // rows eight at a time, all loads issued before any is used; a row past the end
        // loads as zero with weight zero, so the sum keeps its order over k
        for (int k0 = 0; k0 < T; k0 += 8) {
            Row v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = k0 + j < T ? *reinterpret_cast<const Row*>(row(k0 + j) + lane * PER) : Row{};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int k = k0 + j;
                float wt = __shfl_sync(0xffffffffu, w0, k & 31);
                if (k >= 32) wt = k < T ? exp2f(row(k)[D] - M) : 0.f;
                if (k >= T) wt = 0.f;
                const float* f = reinterpret_cast<const float*>(&v[j]);
#pragma unroll
                for (int c = 0; c < PER; ++c) acc[c] = fmaf(wt, f[c], acc[c]);
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* ob = a.out + ((int64_t)r * a.Hq + (int64_t)h * a.G + gg) * D;
#pragma unroll
    for (int c = 0; c < PER; c += 2)
        *reinterpret_cast<uint32_t*>(ob + lane * PER + c) = pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
}

// ------------------------------------------------------------------ host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

// Compile-time query positions per request for a call with at most `max_q_len`
// queries per request (0 if unsupported).
int query_tile(int fp8, int max_q_len) {
    if (max_q_len <= 1) return 1;
    if (max_q_len <= 2) return 2;
    if (max_q_len <= 4 && !fp8) return 4;
    return 0;
}

// The CTA shape for a (dtype, D, BS, QT): `warps` independent pipelines of
// `stages` tiles each.
DecodePlan decode_plan(int kt, int head_dim, int block_size, int num_sms, int batch, int qt) {
    DecodePlan p;
    const int fp8 = kt != 0;
    const int row_bytes = kt == 3 ? head_dim / 2 : head_dim * (fp8 ? 1 : 2);
    // int4 tiles hold 64 tokens (two or four cache blocks); 8-bit tiles one block;
    // bf16 tiles 16 tokens
    const int tile_tokens = kt == 3 ? 64 : (fp8 ? block_size : 16);
    p.stage_bytes = 2 * tile_tokens * row_bytes;
    // Each warp streams its pages through its own 2-stage pipeline; the per-page
    // instruction chain of a warp, not the bytes in flight, limits the rate, so the
    // CTA runs several warps per SM sub-partition.  Measured on GB300: 7 warps for
    // single-query bf16 pages (6 and 8 ran slower), 8 for 8-bit pages (whose tiles carry
    // twice the tokens)
    // and for several query positions, 12 for single-query int4 pages (compute-bound:
    // 0.44 of the copy peak against 0.40 with 8; 10 warps split unevenly over the four
    // sub-partitions and run slower).
    // (within the launch bounds' register budget: 384 threads for single-query bf16
    // and int4 pages, 256 otherwise)
    // The plan is a pure function of its arguments: pkv_decode_workspace_size and the
    // launch must agree on it in every process.
    p.warps = (kt == 3 && qt == 1) ? 12 : ((fp8 || qt > 1) ? 8 : 7);
    int stages = 131072 / (p.warps * p.stage_bytes);
    if (stages > 16) stages = 16;
    if (stages < 2) stages = 2;
    const int fixed = 1024 + (int)align_up(4 * (2 * (int64_t)batch + 1), 16);
    const int qbytes = qt == 4 ? (head_dim / 16) * 4 * 32 * 8 : 0;   // per-warp q fragments
    auto bytes = [&](int w, int st) { return fixed + w * (st * (p.stage_bytes + 8) + qbytes); };
    while (stages > 2 && bytes(p.warps, stages) > 232448) --stages;
    while (p.warps > 1 && bytes(p.warps, stages) > 232448) --p.warps;
    p.stages = stages;
    p.smem_bytes = bytes(p.warps, stages);
    p.ctas_per_sm = 1;
    p.total_warps = num_sms * p.ctas_per_sm * p.warps;
    return p;
}

template <int D, int BS, int KT, int QT>
static cudaError_t launch_t(const DecodeLaunch& L, const DecodePlan& plan, const CUtensorMap& tk,
                            const CUtensorMap& tv, const DecodeArgs& args, cudaStream_t st) {
    auto kern = pkv_decode_kernel<D, BS, KT, QT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         plan.smem_bytes);
    if (e != cudaSuccess) return e;
    const int grid = L.num_sms * plan.ctas_per_sm;
    e = launch_pdl(kern, dim3(grid), dim3(plan.warps * 32), (size_t)plan.smem_bytes, st, tk, tv,
                   args);
    if (e != cudaSuccess) return e;
    if (L.merge_after != nullptr) {
        e = cudaStreamWaitEvent(st, L.merge_after, 0);
        if (e != cudaSuccess) return e;
    }
    // the wide-split merge, a programmatic dependent of the decode grid (with a shared
    // prefix: the merge of every unit with its prefix partials)
    if constexpr (QT == 1) {
        if (L.cascade_part != nullptr)
            return launch_pdl(pkv_cascade_merge_kernel<D>, dim3((unsigned)(L.N * L.Hkv)),
                              dim3(kGroupPad * 32), 0, st, args);
    }
    return launch_pdl(pkv_decode_merge_kernel<D, QT>, dim3((unsigned)(L.N * L.Hkv)),
                      dim3(kGroupPad * 32 * QT), 0, st, args);
}

template <int D, int BS, int KT>
static cudaError_t launch_q(int qt, const DecodeLaunch& L, const DecodePlan& plan,
                            const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& args,
                            cudaStream_t st) {
    if (qt == 1) return launch_t<D, BS, KT, 1>(L, plan, tk, tv, args, st);
    if (qt == 2) return launch_t<D, BS, KT, 2>(L, plan, tk, tv, args, st);
    if constexpr (KT == 0) {
        if (qt == 4) return launch_t<D, BS, KT, 4>(L, plan, tk, tv, args, st);
    }
    return cudaErrorInvalidValue;
}

static bool encode_cache_map(CUtensorMap* m, const void* base, int fp8, int D, int BS,
                             int64_t rows, int kt) {
    auto fn = encode_fn();
    if (!fn) return false;
    if (kt == 3) {   // int4 rows: D/2 = 64 bytes, one box of BS rows, 64-byte swizzle
        cuuint64_t dims[2] = {(cuuint64_t)(D / 2), (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)(D / 2)};
        cuuint32_t box[2] = {(cuuint32_t)(D / 2), (cuuint32_t)BS};
        cuuint32_t estr[2] = {1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const int elt = fp8 ? 1 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(D * elt)};
    cuuint32_t box[2] = {(cuuint32_t)(128 / elt), (cuuint32_t)(fp8 ? BS : 16)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Returns a pkv_status.  Arguments are validated by the caller.
int decode_launch(const DecodeLaunch& L, cudaStream_t st) {
    const int qt = query_tile(L.fp8, L.max_q_len);
    if (qt == 0) return PKV_ERR_UNSUPPORTED;
    const DecodePlan plan = decode_plan(L.kt, L.D, L.BS, L.num_sms, L.N, qt);
    const WorkspaceLayout WL = workspace_layout(L.N, L.Hkv, L.D, plan.total_warps, qt);
    const int64_t rows = (int64_t)L.NB * L.Hkv * L.BS;
    alignas(64) CUtensorMap tk, tv;
    if (!encode_cache_map(&tk, L.k_cache, L.fp8, L.D, L.BS, rows, L.kt) ||
        !encode_cache_map(&tv, L.v_cache, L.fp8, L.D, L.BS, rows, L.kt))
        return PKV_ERR_CUDA;
    DecodeArgs a;
    uint8_t* ws = static_cast<uint8_t*>(L.workspace);
    a.q = static_cast<const uint16_t*>(L.q);
    a.q_offsets = L.q_offsets;
    a.out = static_cast<uint16_t*>(L.out);
    a.block_table = L.block_table;
    a.seq_lens = L.seq_lens;
    a.k_scale = L.k_scale;
    a.v_scale = L.v_scale;
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.g_prefix = reinterpret_cast<int32_t*>(ws + WL.prefix_off);
    a.partials = reinterpret_cast<float*>(ws + WL.partial_off);
    a.N = L.N;
    a.Hq = L.Hq;
    a.Hkv = L.Hkv;
    a.G = L.Hq / L.Hkv;
    a.MB = L.MB;
    a.NB = L.NB;
    a.scale_log2 = L.scale * 1.4426950408889634f;
    a.stages = plan.stages;
    a.total_warps = plan.total_warps;
    a.skip_blocks = L.skip_blocks;
    a.cascade_part = L.cascade_part;
    a.cascade_split = L.cascade_split;
    a.k_new = static_cast<const uint16_t*>(L.k_new);
    a.v_new = static_cast<const uint16_t*>(L.v_new);
    a.k_cache_w = static_cast<uint16_t*>(const_cast<void*>(L.k_cache));
    a.v_cache_w = static_cast<uint16_t*>(const_cast<void*>(L.v_cache));
    cudaError_t e = cudaErrorInvalidValue;
    if (L.kt == 0) {
        if (L.D == 128 && L.BS == 16) e = launch_q<128, 16, 0>(qt, L, plan, tk, tv, a, st);
        else if (L.D == 128 && L.BS == 32) e = launch_q<128, 32, 0>(qt, L, plan, tk, tv, a, st);
        else if (L.D == 64 && L.BS == 16) e = launch_q<64, 16, 0>(qt, L, plan, tk, tv, a, st);
        else if (L.D == 64 && L.BS == 32) e = launch_q<64, 32, 0>(qt, L, plan, tk, tv, a, st);
        else return PKV_ERR_UNSUPPORTED;
    } else if (L.kt == 1) {
        if (L.D == 128 && L.BS == 16) e = launch_q<128, 16, 1>(qt, L, plan, tk, tv, a, st);
        else if (L.D == 128 && L.BS == 32) e = launch_q<128, 32, 1>(qt, L, plan, tk, tv, a, st);
        else return PKV_ERR_UNSUPPORTED;
    } else if (L.kt == 2) {
        if (L.D == 128 && L.BS == 16) e = launch_q<128, 16, 2>(qt, L, plan, tk, tv, a, st);
        else if (L.D == 128 && L.BS == 32) e = launch_q<128, 32, 2>(qt, L, plan, tk, tv, a, st);
        else return PKV_ERR_UNSUPPORTED;
    } else {
        if (L.D == 128 && L.BS == 16) e = launch_q<128, 16, 3>(qt, L, plan, tk, tv, a, st);
        else if (L.D == 128 && L.BS == 32) e = launch_q<128, 32, 3>(qt, L, plan, tk, tv, a, st);
        else return PKV_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t decode_workspace_bytes(int batch, int num_kv_heads, int head_dim, int block_size, int kt,
                              int num_sms, int max_q_len) {
    const int qt = query_tile(kt != 0, max_q_len);
    if (qt == 0) return 0;
    const DecodePlan plan = decode_plan(kt, head_dim, block_size, num_sms, batch, qt);
    return (size_t)workspace_layout(batch, num_kv_heads, head_dim, plan.total_warps, qt).total;
}

}  // namespace pkv
