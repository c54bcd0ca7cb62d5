// pkv_api.cu -- the extern "C" entry points of libpagedkv.
//
// Every entry point validates its host-side scalars and pointer alignment
// first and launches nothing when a check fails.  No entry point synchronises
// the device or copies device memory to the host.
#include <math.h>
#include <stdint.h>

#include <mutex>

#include <cuda.h>

#include "pkv_internal.cuh"


namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool shape_supported(int Hq, int Hkv, int D, int BS, int dtype) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq / Hkv > pkv::kGroupPad) return false;
    if (BS != 16 && BS != 32) return false;
    if (dtype == PKV_BF16) return D == 64 || D == 128;
    if (dtype == PKV_FP8_E4M3 || dtype == PKV_INT8 || dtype == PKV_INT4) return D == 128;
    return false;
}

int current_num_sms(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PKV_ERR_CUDA;
    *out = n;
    return PKV_OK;
}

}  // namespace

extern "C" {

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_NO_BLOCKS: return "PKV_ERR_NO_BLOCKS";
        default: return "PKV_UNKNOWN_STATUS";
    }
}

int pkv_version(void) { return 1 * 10000 + 0 * 100 + 0; }

int pkv_device_num_sms(int* num_sms) {
    if (!num_sms) return PKV_ERR_INVALID_ARG;
    return current_num_sms(num_sms);
}

int pkv_compute_slot_mapping(const int32_t* block_table, int max_blocks_per_seq,
                             const int32_t* req_idx, const int32_t* positions, int num_tokens,
                             int block_size, int64_t* slot_mapping, pkv_stream_t stream) {
    if (num_tokens < 0 || block_size <= 0 || max_blocks_per_seq <= 0) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!block_table || !positions || !slot_mapping) return PKV_ERR_INVALID_ARG;
    cudaError_t e = pkv::slot_mapping_launch(block_table, max_blocks_per_seq, req_idx, positions,
                                             num_tokens, block_size, slot_mapping,
                                             reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_kv_cache_write(const void* k, const void* v, const int64_t* slot_mapping, int num_tokens,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks,
                       int cache_dtype, void* k_cache, void* v_cache, const float* k_scale,
                       const float* v_scale, pkv_stream_t stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3 && cache_dtype != PKV_INT8 &&
        cache_dtype != PKV_INT4)
        return PKV_ERR_UNSUPPORTED;
    if (head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (cache_dtype != PKV_BF16 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PKV_ERR_INVALID_ARG;
    cudaError_t e = pkv::cache_write_launch(
        k, v, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, num_blocks,
        cache_dtype, k_cache, v_cache, k_scale, v_scale,
        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_rescale_workspace_size(int num_blocks, int num_kv_heads) {
    if (num_blocks <= 0 || num_kv_heads <= 0) return 0;
    return (size_t)2 * num_blocks * num_kv_heads * 4;
}

int pkv_kv_cache_write_rescale(const void* k, const void* v, const int64_t* slot_mapping,
                               int num_tokens, int num_kv_heads, int head_dim, int block_size,
                               int num_blocks, int cache_dtype, void* k_cache, void* v_cache,
                               float* k_scale, float* v_scale, void* workspace,
                               size_t workspace_bytes, pkv_stream_t stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (cache_dtype != PKV_FP8_E4M3 && cache_dtype != PKV_INT8 && cache_dtype != PKV_INT4)
        return PKV_ERR_UNSUPPORTED;
    if (head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pkv_rescale_workspace_size(num_blocks, num_kv_heads))
        return PKV_ERR_WORKSPACE;
    if (!aligned(workspace, 4)) return PKV_ERR_INVALID_ARG;
    cudaError_t e = pkv::cache_write_rescale_launch(
        k, v, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, num_blocks,
        cache_dtype, k_cache, v_cache, k_scale, v_scale, workspace,
        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_multiquery_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, int cache_dtype, int max_q_len,
                                     int num_sms) {
    if (batch < 0 || batch > pkv::kMaxBatch || max_q_len < 1) return 0;
    if (!shape_supported(num_q_heads, num_kv_heads, head_dim, block_size, cache_dtype)) return 0;
    if (num_sms <= 0 && current_num_sms(&num_sms) != PKV_OK) return 0;
    return pkv::decode_workspace_bytes(batch, num_kv_heads, head_dim, block_size,
                                       cache_dtype, num_sms, max_q_len);
}

size_t pkv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int cache_dtype, int num_sms) {
    return pkv_multiquery_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                                         cache_dtype, 1, num_sms);
}

int pkv_paged_multiquery_attn(const void* q, const int32_t* q_offsets, int max_q_len,
                              const void* k_cache, const void* v_cache, const float* k_scale,
                              const float* v_scale, const int32_t* block_table,
                              int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              int num_blocks, int cache_dtype, float scale, void* out,
                              void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
    if (batch < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || max_q_len < 1)
        return PKV_ERR_INVALID_ARG;
    if (cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3 && cache_dtype != PKV_INT8 &&
        cache_dtype != PKV_INT4)
        return PKV_ERR_UNSUPPORTED;
    if (!shape_supported(num_q_heads, num_kv_heads, head_dim, block_size, cache_dtype))
        return PKV_ERR_UNSUPPORTED;
    if (pkv::query_tile(cache_dtype != PKV_BF16, max_q_len) == 0) return PKV_ERR_UNSUPPORTED;
    if (batch > pkv::kMaxBatch) return PKV_ERR_UNSUPPORTED;
    if (batch == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (max_q_len > 1 && !q_offsets) return PKV_ERR_INVALID_ARG;
    if (cache_dtype != PKV_BF16 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PKV_ERR_INVALID_ARG;
    // flat page index and TMA row coordinates are int32
    const int64_t rows = ((int64_t)num_blocks + 1) * num_kv_heads * block_size;
    const int64_t max_pages = (int64_t)batch * num_kv_heads * max_blocks_per_seq;
    if (rows >= (int64_t)1 << 31 || max_pages >= (int64_t)1 << 31 ||
        (int64_t)max_blocks_per_seq * block_size >= (int64_t)1 << 22)
        return PKV_ERR_UNSUPPORTED;
    int num_sms = 0;
    if (current_num_sms(&num_sms) != PKV_OK) return PKV_ERR_CUDA;
    const size_t need = pkv::decode_workspace_bytes(batch, num_kv_heads, head_dim, block_size,
                                                    cache_dtype, num_sms,
                                                    max_q_len);
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;
    pkv::DecodeLaunch L;
    L.q = q;
    L.q_offsets = q_offsets;
    L.max_q_len = max_q_len;
    L.k_cache = k_cache;
    L.v_cache = v_cache;
    L.k_scale = k_scale;
    L.v_scale = v_scale;
    L.block_table = block_table;
    L.seq_lens = seq_lens;
    L.out = out;
    L.workspace = workspace;
    L.N = batch;
    L.Hq = num_q_heads;
    L.Hkv = num_kv_heads;
    L.D = head_dim;
    L.BS = block_size;
    L.MB = max_blocks_per_seq;
    L.NB = num_blocks;
    L.fp8 = cache_dtype != PKV_BF16;
    L.kt = cache_dtype;
    L.scale = scale;
    L.num_sms = num_sms;
    return pkv::decode_launch(L, reinterpret_cast<cudaStream_t>(stream));
}

int pkv_paged_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                          const float* k_scale, const float* v_scale,
                          const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
                          int head_dim, int block_size, int num_blocks, int cache_dtype,
                          float scale, void* out, void* workspace, size_t workspace_bytes,
                          pkv_stream_t stream) {
    return pkv_paged_multiquery_attn(q, nullptr, 1, k_cache, v_cache, k_scale, v_scale,
                                     block_table, max_blocks_per_seq, seq_lens, batch,
                                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                                     cache_dtype, scale, out, workspace, workspace_bytes, stream);
}

int pkv_prefix_block_hash(const int32_t* tokens, const int64_t* offsets, int num_seqs,
                          int block_size, uint64_t seed, uint64_t* hashes,
                          const int64_t* hash_offsets, pkv_stream_t stream) {
    if (num_seqs < 0 || block_size <= 0 || block_size > 1024) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!tokens || !offsets || !hashes || !hash_offsets) return PKV_ERR_INVALID_ARG;
    cudaError_t e = pkv::prefix_hash_launch(tokens, offsets, num_seqs, block_size, seed, nullptr,
                                            nullptr, hashes, hash_offsets,
                                            reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_prefix_block_hash_resume(const int32_t* tokens, const int64_t* offsets, int num_seqs,
                                 int block_size, const uint64_t* prev_hashes,
                                 const int64_t* first_blocks, uint64_t* hashes,
                                 const int64_t* hash_offsets, pkv_stream_t stream) {
    if (num_seqs < 0 || block_size <= 0 || block_size > 1024) return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!tokens || !offsets || !prev_hashes || !first_blocks || !hashes || !hash_offsets)
        return PKV_ERR_INVALID_ARG;
    cudaError_t e = pkv::prefix_hash_launch(tokens, offsets, num_seqs, block_size, 0, prev_hashes,
                                            first_blocks, hashes, hash_offsets,
                                            reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_paged_decode_attn_append(const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, const int32_t* block_table,
                                 int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                                 int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, float scale, void* out, void* workspace,
                                 size_t workspace_bytes, pkv_stream_t stream) {
    if (batch < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (!shape_supported(num_q_heads, num_kv_heads, head_dim, block_size, PKV_BF16))
        return PKV_ERR_UNSUPPORTED;
    if (batch > pkv::kMaxBatch) return PKV_ERR_UNSUPPORTED;
    if (batch == 0) return PKV_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(k_new, 16) || !aligned(v_new, 16))
        return PKV_ERR_INVALID_ARG;
    const int64_t rows = ((int64_t)num_blocks + 1) * num_kv_heads * block_size;
    const int64_t max_pages = (int64_t)batch * num_kv_heads * max_blocks_per_seq;
    if (rows >= (int64_t)1 << 31 || max_pages >= (int64_t)1 << 31 ||
        (int64_t)max_blocks_per_seq * block_size >= (int64_t)1 << 22)
        return PKV_ERR_UNSUPPORTED;
    int num_sms = 0;
    if (current_num_sms(&num_sms) != PKV_OK) return PKV_ERR_CUDA;
    const size_t need = pkv::decode_workspace_bytes(batch, num_kv_heads, head_dim, block_size,
                                                    PKV_BF16, num_sms, 1);
    if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return PKV_ERR_INVALID_ARG;
    pkv::DecodeLaunch L;
    L.q = q;
    L.q_offsets = nullptr;
    L.max_q_len = 1;
    L.k_cache = k_cache;
    L.v_cache = v_cache;
    L.k_scale = nullptr;
    L.v_scale = nullptr;
    L.block_table = block_table;
    L.seq_lens = seq_lens;
    L.out = out;
    L.workspace = workspace;
    L.N = batch;
    L.Hq = num_q_heads;
    L.Hkv = num_kv_heads;
    L.D = head_dim;
    L.BS = block_size;
    L.MB = max_blocks_per_seq;
    L.NB = num_blocks;
    L.fp8 = 0;
    L.kt = PKV_BF16;
    L.scale = scale;
    L.num_sms = num_sms;
    L.k_new = k_new;
    L.v_new = v_new;
    return pkv::decode_launch(L, reinterpret_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------------ shared prefix
namespace {

// KV chunks of the prefix pass: enough (query tile, KV head, chunk) CTAs to cover the
// SMs, each chunk a whole number of 256-token tiles.
// How the shared-prefix call divides the GPU.  The prefix pass has rows = batch x G query
// rows per KV head, in 128-row tiles: CTAs = tiles x Hkv x split.
//   sequential: the prefix pass split into chunks so that its CTAs fill the SMs, then the
//     tail decode over every SM, then the merge.
//   overlapped: the prefix pass with one chunk per CTA (few CTAs) on a second stream,
//     while the tail decode runs on the remaining SMs, then the merge.  Chosen when those
//     CTAs take at most a third of the SMs and, by a cost estimate, finish sooner: the
//     prefix pass at about 2.1 us per 256-token tile plus 6.5 us per CTA, the tails
//     streamed at about 6.5 TB/s, each tail taken as half the room the block table leaves
//     after the prefix (the host does not see the lengths).
struct SharedPrefixPlan {
    int split;        // chunks of the prefix (one per CTA along the third grid axis)
    int chunk;        // tokens per chunk
    int dec_sms;      // SMs the tail decode is sized for
    bool overlap;
};

SharedPrefixPlan shared_prefix_plan(int batch, int Hq, int Hkv, int D, int BS, int MB,
                                    int prefix_len, int num_sms) {
    SharedPrefixPlan p{0, 0, num_sms, false};
    const int G = Hq / Hkv;
    const int TQ = 128 / G;
    const int tiles = (batch + TQ - 1) / TQ;
    const int ktiles = (prefix_len + 255) / 256;
    if (ktiles == 0 || tiles == 0) return p;
    int want = (num_sms + tiles * Hkv - 1) / (tiles * Hkv);
    if (want < 1) want = 1;
    if (want > ktiles) want = ktiles;
    const int per = (ktiles + want - 1) / want;
    p.chunk = per * 256;
    p.split = (ktiles + per - 1) / per;
    const int k = tiles * Hkv;                  // prefix CTAs with one chunk each
    if (3 * k <= num_sms) {
        const double tile_us = 2.1, cta_us = 6.5, gbs = 6500.0;
        const double tail_tokens = 0.5 * ((double)MB * BS - prefix_len);
        const double tail_us =
            (double)batch * tail_tokens * Hkv * D * 2.0 * 2.0 / (gbs * 1e3);
        const double seq_us = per * tile_us + cta_us + tail_us;
        const double ovl_us = fmax(ktiles * tile_us + cta_us,
                                   tail_us * num_sms / (double)(num_sms - k));
        if (ovl_us < seq_us) {
            p.split = 1;
            p.chunk = ktiles * 256;
            p.dec_sms = num_sms - k;
            p.overlap = true;
        }
    }
    return p;
}

// A second stream and two events per device for the overlapped prefix pass, created on
// the first overlapped call with that device current (make that call outside stream
// capture) and again after the device's context changes.  One lock serialises the fork
// and join of concurrent callers.
typedef CUresult (*ctx_get_current_fn)(CUcontext*);

ctx_get_current_fn side_ctx_get_current() {
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

struct SideStream {
    CUcontext ctx = nullptr;
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxSideDevices = 64;
std::mutex g_side_mu;
SideStream g_side[kMaxSideDevices];

// With g_side_mu held.
int side_stream(SideStream** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxSideDevices) return PKV_ERR_UNSUPPORTED;
    ctx_get_current_fn get = side_ctx_get_current();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS || !ctx) return PKV_ERR_CUDA;
    SideStream& s = g_side[dev];
    if (s.ctx != ctx || !s.stream) {
        // a new context: the old handles belonged to a context that is gone
        SideStream n;
        if (cudaStreamCreateWithFlags(&n.stream, cudaStreamNonBlocking) != cudaSuccess)
            return PKV_ERR_CUDA;
        if (cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) != cudaSuccess)
            return PKV_ERR_CUDA;
        n.ctx = ctx;
        s = n;
    }
    *out = &s;
    return PKV_OK;
}

bool shared_prefix_supported(int Hq, int Hkv, int D, int BS) {
    return shape_supported(Hq, Hkv, D, BS, PKV_BF16) &&
           pkv::prefill_shape_supported(Hq, Hkv, D, BS, PKV_BF16);
}

}  // namespace

int pkv_shared_prefix_plan(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                           int block_size, int max_blocks_per_seq, int prefix_len, int num_sms,
                           int* prefix_ctas, int* decode_sms) {
    if (batch < 0 || max_blocks_per_seq <= 0 || prefix_len < 0) return PKV_ERR_INVALID_ARG;
    if (!shared_prefix_supported(num_q_heads, num_kv_heads, head_dim, block_size))
        return PKV_ERR_UNSUPPORTED;
    if (batch > pkv::kMaxBatch) return PKV_ERR_UNSUPPORTED;
    if (prefix_len % block_size != 0 || prefix_len > max_blocks_per_seq * block_size)
        return PKV_ERR_INVALID_ARG;
    if (num_sms <= 0 && current_num_sms(&num_sms) != PKV_OK) return PKV_ERR_CUDA;
    const SharedPrefixPlan p = shared_prefix_plan(batch, num_q_heads, num_kv_heads, head_dim,
                                                  block_size, max_blocks_per_seq, prefix_len,
                                                  num_sms);
    const int G = num_q_heads / num_kv_heads;
    const int tiles = (batch + 128 / G - 1) / (128 / G);
    if (prefix_ctas) *prefix_ctas = p.split > 0 ? tiles * num_kv_heads * p.split : 0;
    if (decode_sms) *decode_sms = p.dec_sms;
    return p.overlap ? 1 : 0;
}

size_t pkv_shared_prefix_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int prefix_len,
                                        int num_sms) {
    if (batch < 0 || batch > pkv::kMaxBatch || prefix_len < 0) return 0;
    if (!shared_prefix_supported(num_q_heads, num_kv_heads, head_dim, block_size)) return 0;
    if (num_sms <= 0 && current_num_sms(&num_sms) != PKV_OK) return 0;
    const size_t dec = pkv::decode_workspace_bytes(batch, num_kv_heads, head_dim, block_size,
                                                   PKV_BF16, num_sms, 1);
    // the prefix partials for the sequential plan's split, which is at least the
    // overlapped plan's one chunk; the decode part for every SM, at least the tail
    // decode's share of them
    const SharedPrefixPlan p = shared_prefix_plan(batch, num_q_heads, num_kv_heads, head_dim,
                                                  block_size, 0, prefix_len, num_sms);
    return (size_t)pkv::align_up((int64_t)dec, 256) +
           (size_t)batch * num_q_heads * p.split * (head_dim + 4) * 4;
}

int pkv_paged_decode_attn_shared_prefix(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, int max_blocks_per_seq,
                                        const int32_t* seq_lens, int batch, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int num_blocks, int prefix_len, float scale, void* out,
                                        void* workspace, size_t workspace_bytes,
                                        pkv_stream_t stream) {
    if (batch < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || prefix_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (!shared_prefix_supported(num_q_heads, num_kv_heads, head_dim, block_size))
        return PKV_ERR_UNSUPPORTED;
    if (batch > pkv::kMaxBatch) return PKV_ERR_UNSUPPORTED;
    if (block_size <= 0 || prefix_len % block_size != 0 ||
        prefix_len > max_blocks_per_seq * block_size)
        return PKV_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < INFINITY)) return PKV_ERR_INVALID_ARG;
    if (prefix_len == 0)   // nothing shared: the plain decode
        return pkv_paged_decode_attn(q, k_cache, v_cache, nullptr, nullptr, block_table,
                                     max_blocks_per_seq, seq_lens, batch, num_q_heads,
                                     num_kv_heads, head_dim, block_size, num_blocks, PKV_BF16,
                                     scale, out, workspace, workspace_bytes, stream);
    if (batch == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PKV_ERR_INVALID_ARG;
    const int64_t rows = ((int64_t)num_blocks + 1) * num_kv_heads * block_size;
    const int64_t max_pages = (int64_t)batch * num_kv_heads * max_blocks_per_seq;
    if (rows >= (int64_t)1 << 31 || max_pages >= (int64_t)1 << 31 ||
        (int64_t)max_blocks_per_seq * block_size >= (int64_t)1 << 22)
        return PKV_ERR_UNSUPPORTED;
    int num_sms = 0;
    if (current_num_sms(&num_sms) != PKV_OK) return PKV_ERR_CUDA;
    const size_t need = pkv_shared_prefix_workspace_size(batch, num_q_heads, num_kv_heads,
                                                         head_dim, block_size, prefix_len,
                                                         num_sms);
    if (!workspace || need == 0 || workspace_bytes < need) return PKV_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PKV_ERR_INVALID_ARG;
    const size_t dec = pkv::decode_workspace_bytes(batch, num_kv_heads, head_dim, block_size,
                                                   PKV_BF16, num_sms, 1);
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                           pkv::align_up((int64_t)dec, 256));
    const SharedPrefixPlan plan =
        shared_prefix_plan(batch, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_blocks_per_seq, prefix_len, num_sms);
    const int split = plan.split, chunk = plan.chunk;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // 1) the shared pages once for every request: all queries as the rows of a
    //    non-causal pass over block-table row 0's first prefix_len tokens
    pkv::PrefillLaunch P;
    P.q = q;
    P.q_offsets = nullptr;
    P.k_cache = k_cache;
    P.v_cache = v_cache;
    P.block_table = block_table;
    P.seq_lens = nullptr;
    P.out = nullptr;
    P.err = static_cast<uint32_t*>(workspace);   // the decode workspace's error word
    P.total_q = batch;
    P.max_q_len = batch;
    P.N = 1;
    P.Hq = num_q_heads;
    P.Hkv = num_kv_heads;
    P.D = head_dim;
    P.BS = block_size;
    P.MB = max_blocks_per_seq;
    P.NB = num_blocks;
    P.scale = scale;
    P.prefix_split = split;
    P.prefix_len = prefix_len;
    P.chunk_tokens = chunk;
    P.part = part;
    // overlapped: the prefix pass forks onto the side stream and joins before the merge
    std::unique_lock<std::mutex> side_lock;
    SideStream* side = nullptr;
    if (plan.overlap) {
        side_lock = std::unique_lock<std::mutex>(g_side_mu);
        const int sst = side_stream(&side);
        if (sst != PKV_OK) return sst;
        if (cudaEventRecord(side->fork, st) != cudaSuccess ||
            cudaStreamWaitEvent(side->stream, side->fork, 0) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    int stp = pkv::prefill_launch(P, side ? side->stream : st);
    if (stp != PKV_OK) return stp;
    if (side && cudaEventRecord(side->join, side->stream) != cudaSuccess) return PKV_ERR_CUDA;
    // 2) each request's private pages, every unit as a partial, 3) the merge
    pkv::DecodeLaunch L;
    L.q = q;
    L.q_offsets = nullptr;
    L.max_q_len = 1;
    L.k_cache = k_cache;
    L.v_cache = v_cache;
    L.k_scale = nullptr;
    L.v_scale = nullptr;
    L.block_table = block_table;
    L.seq_lens = seq_lens;
    L.out = out;
    L.workspace = workspace;
    L.N = batch;
    L.Hq = num_q_heads;
    L.Hkv = num_kv_heads;
    L.D = head_dim;
    L.BS = block_size;
    L.MB = max_blocks_per_seq;
    L.NB = num_blocks;
    L.fp8 = 0;
    L.kt = PKV_BF16;
    L.scale = scale;
    L.num_sms = plan.dec_sms;
    L.skip_blocks = prefix_len / block_size;
    L.cascade_part = part;
    L.cascade_split = split;
    L.merge_after = side ? side->join : nullptr;
    return pkv::decode_launch(L, st);
}

size_t pkv_prefill_workspace_size(int batch, int max_blocks_per_seq, int num_kv_heads,
                                  int head_dim, int block_size, int cache_dtype) {
    if (batch <= 0 || max_blocks_per_seq <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0)
        return 0;
    if (cache_dtype == PKV_BF16) return 0;
    const int64_t blocks = (int64_t)batch * max_blocks_per_seq;
    const int64_t pool = blocks * num_kv_heads * block_size * head_dim * 2;   // bf16, K or V
    return (size_t)(2 * pkv::align_up(pool, 256) + pkv::align_up(blocks * 4, 256));
}

int pkv_paged_prefill_attn(const void* q, const int32_t* q_offsets, int total_q, int max_q_len,
                           const void* k_cache, const void* v_cache, const float* k_scale,
                           const float* v_scale, const int32_t* block_table,
                           int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, int cache_dtype, float scale, void* out,
                           void* workspace, size_t workspace_bytes, uint32_t* error_word,
                           pkv_stream_t stream) {
    if (batch < 0 || total_q < 0 || max_q_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3 && cache_dtype != PKV_INT8 &&
        cache_dtype != PKV_INT4)
        return PKV_ERR_UNSUPPORTED;
    if (!pkv::prefill_shape_supported(num_q_heads, num_kv_heads, head_dim, block_size, PKV_BF16))
        return PKV_ERR_UNSUPPORTED;
    if (!(scale > 0.f) || scale > 3.0e38f) return PKV_ERR_INVALID_ARG;   // finite, > 0
    if (batch == 0 || total_q == 0 || max_q_len == 0) return PKV_OK;
    if ((int64_t)(num_blocks + 1) * num_kv_heads * block_size >= ((int64_t)1 << 31))
        return PKV_ERR_UNSUPPORTED;
    if (!q || !q_offsets || !k_cache || !v_cache || !block_table || !seq_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(error_word, 4))
        return PKV_ERR_INVALID_ARG;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    pkv::PrefillLaunch L;
    L.q = q;
    L.q_offsets = q_offsets;
    L.k_cache = k_cache;
    L.v_cache = v_cache;
    L.block_table = block_table;
    L.seq_lens = seq_lens;
    L.out = out;
    L.err = error_word;
    L.total_q = total_q;
    L.max_q_len = max_q_len;
    L.N = batch;
    L.Hq = num_q_heads;
    L.Hkv = num_kv_heads;
    L.D = head_dim;
    L.BS = block_size;
    L.MB = max_blocks_per_seq;
    L.NB = num_blocks;
    L.scale = scale;
    if (cache_dtype != PKV_BF16) {
        // quantised pages: expand the batch's pages to a bf16 pool, then the bf16 kernel
        if (!k_scale || !v_scale) return PKV_ERR_INVALID_ARG;
        const size_t need = pkv_prefill_workspace_size(batch, max_blocks_per_seq, num_kv_heads,
                                                       head_dim, block_size, cache_dtype);
        if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return PKV_ERR_INVALID_ARG;
        const int64_t blocks = (int64_t)batch * max_blocks_per_seq;
        if ((blocks + 1) * num_kv_heads * block_size >= ((int64_t)1 << 31))
            return PKV_ERR_UNSUPPORTED;
        const int64_t pool = pkv::align_up(blocks * num_kv_heads * block_size * head_dim * 2, 256);
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        int sms = 0;
        const int sst = current_num_sms(&sms);
        if (sst != PKV_OK) return sst;
        cudaError_t e = pkv::dequant_pages_launch(
            k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, batch, max_blocks_per_seq,
            num_blocks, num_kv_heads, block_size, head_dim, cache_dtype, ws, ws + pool,
            reinterpret_cast<int32_t*>(ws + 2 * pool), error_word, sms, st);
        if (e != cudaSuccess) return PKV_ERR_CUDA;
        L.k_cache = ws;
        L.v_cache = ws + pool;
        L.block_table = reinterpret_cast<const int32_t*>(ws + 2 * pool);
        L.NB = (int)blocks;
    }
    return pkv::prefill_launch(L, st);
}

int pkv_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                    const int32_t* block_mapping, int num_pairs, int num_kv_heads, int head_dim,
                    int block_size, int num_blocks, int cache_dtype, pkv_stream_t stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (cache_dtype != PKV_BF16 && cache_dtype != PKV_FP8_E4M3 && cache_dtype != PKV_INT8 &&
        cache_dtype != PKV_INT4)
        return PKV_ERR_UNSUPPORTED;
    const int64_t elems = (int64_t)num_kv_heads * block_size * head_dim;
    const int64_t block_bytes = cache_dtype == PKV_BF16 ? 2 * elems
                                : (cache_dtype == PKV_INT4 ? elems / 2 : elems);
    if (block_bytes % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !block_mapping) return PKV_ERR_INVALID_ARG;
    if (cache_dtype != PKV_BF16 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_mapping, 4))
        return PKV_ERR_INVALID_ARG;
    int sms = 0;
    const int st = current_num_sms(&sms);
    if (st != PKV_OK) return st;
    const bool q8 = cache_dtype != PKV_BF16;
    cudaError_t e = pkv::copy_blocks_launch(k_cache, v_cache, q8 ? k_scale : nullptr,
                                            q8 ? v_scale : nullptr, block_mapping, num_pairs,
                                            block_bytes, num_blocks, num_kv_heads, sms,
                                            reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // extern "C"
