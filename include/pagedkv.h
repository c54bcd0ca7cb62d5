/*
 * pagedkv.h -- C ABI of libpagedkv: the decode-step hot path over a paged KV
 * cache, hand-written CUDA for sm_103a (GB300).
 *
 * Sources, by page title and section:
 *   [P1] "深入LLM推理：从KV Cache到PD分离的Serving全景解析"
 *        "KV Cache：Transformer的循环状态"  Attention(Q,K,V) = softmax(QK^T/sqrt(d)) V;
 *                                           GQA: several query heads share one K/V head.
 *        "PagedAttention与Cache管理"        block table: logical block -> physical block,
 *                                           fixed blocks of 16 or 32 tokens.
 *   [P2] "GPU推理深度拆解：KV Cache视角"
 *        "算子优化要点"                      online softmax (FlashAttention); CUDA Graph
 *                                           needs static shapes and addresses; batch-1
 *                                           decode under-uses the SMs.
 *   [P3] "ai-infra-7"
 *        "优化一：Prefix Cache"               hash_i = H(hash_{i-1}, block tokens).
 *        "优化三：KV 传输优化" (3. 传输量化)    FP8 KV.
 *        "组合拳：一次请求的完整旅程"           new KV written back into the cache pool.
 *
 * Conventions for every entry point
 *   - Pointers named *_cache, q, k, v, out, block_table, seq_lens, slot_mapping,
 *     tokens, offsets, hashes, workspace are DEVICE pointers owned by the caller.
 *     The library allocates nothing and keeps no per-call state.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *     No call synchronises the device or copies device data to the host, so a
 *     sequence of calls can be captured in a CUDA graph.
 *   - Host-side scalars are validated before anything is launched; a failed
 *     check returns a negative pkv_status and launches nothing.  A launch
 *     failure returns PKV_ERR_CUDA.  Nothing throws, aborts or traps.
 *   - Device-side content (block ids, slots, lengths) is the caller's contract;
 *     the decode kernels clamp what they cannot trust and record it in the
 *     workspace error word (PKV_DEVERR_*), they never read out of bounds.
 *   - Layouts are row-major and contiguous:
 *       q, out          bf16 [N][Hq][D]
 *       k, v (new rows) bf16 [T][Hkv][D]
 *       k_cache,v_cache [NB][Hkv][BS][D]  bf16 or E4M3 bytes; one (block, head)
 *                       page of BS*D elements is contiguous
 *       k_scale,v_scale fp32 [NB][Hkv]    FP8 caches only
 *       block_table     int32 [N][MB]     physical block of logical block j of request r
 *       seq_lens        int32 [N]         tokens cached for request r, including the
 *                                         one written this step
 *   - Query head hq reads KV head hq / G, G = Hq / Hkv (consecutive groups).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *pkv_stream_t;

/* Cache element type. */
enum { PKV_BF16 = 0, PKV_FP8_E4M3 = 1 };

/* Return codes. */
enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,   /* null pointer, bad size, misaligned buffer */
    PKV_ERR_UNSUPPORTED = -2,   /* a shape this build has no kernel for */
    PKV_ERR_WORKSPACE = -3,     /* workspace missing or smaller than required */
    PKV_ERR_CUDA = -4           /* a CUDA runtime call or launch failed */
};

/* Bits of the device error word (first 4 bytes of the decode workspace).  The
 * word is sticky: kernels only OR bits in; the caller clears it. */
#define PKV_DEVERR_WAIT_TIMEOUT  0x1u  /* a pipeline wait gave up after ~2 s      */
#define PKV_DEVERR_SEQ_CLAMPED   0x2u  /* seq_lens[r] < 0 or > MB*BS was clamped  */
#define PKV_DEVERR_BLOCK_RANGE   0x4u  /* a block id outside [0, NB) was read     */
#define PKV_DEVERR_QLEN_CLAMPED  0x8u  /* a request's query count exceeded max_q_len */

/* Human-readable name of a pkv_status value (static string). */
PKV_API const char *pkv_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
PKV_API int pkv_version(void);

/* Number of SMs of the current CUDA device (written to *num_sms). */
PKV_API int pkv_device_num_sms(int *num_sms);

/*
 * Slot mapping ([P1] "PagedAttention与Cache管理").  For token t of request
 * r = req_idx[t] (req_idx may be NULL: r = t) at position pos = positions[t]:
 *     slot_mapping[t] = block_table[r][pos / BS] * BS + pos % BS
 * pos < 0 marks a padding token and yields -1; so does pos >= MB*BS.
 * block_table int32 [*, MB]; req_idx, positions int32 [T]; slot_mapping int64 [T].
 */
PKV_API int pkv_compute_slot_mapping(const int32_t *block_table, int max_blocks_per_seq,
                             const int32_t *req_idx, const int32_t *positions,
                             int num_tokens, int block_size, int64_t *slot_mapping,
                             pkv_stream_t stream);

/*
 * KV cache write, a.k.a. reshape_and_cache ([P3] "组合拳：一次请求的完整旅程":
 * newly generated K/V go back into the cache pool; FP8 per [P3] 传输量化).
 * Row (t, h) of k and v (bf16 [T][Hkv][D]) goes to cache row
 * [slot / BS][h][slot % BS][:] with slot = slot_mapping[t]; slot < 0 is skipped,
 * and so is a slot whose block is >= num_blocks.
 *   PKV_BF16:     bytes are copied unchanged.
 *   PKV_FP8_E4M3: byte = E4M3(float(x) / scale[blk][h]), IEEE binary32 divide,
 *                 round to nearest even, saturating to +-448 (k_scale/v_scale
 *                 fp32 [NB][Hkv], required).  A later token of a block reuses
 *                 the block's scale.
 * Bytes not addressed by a slot are untouched.  Two tokens with the same slot
 * race (last writer wins, undefined which).
 * Requirements: head_dim % 8 == 0; k, v, caches 16-byte aligned.
 */
PKV_API int pkv_kv_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                       int num_tokens, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int cache_dtype, void *k_cache, void *v_cache,
                       const float *k_scale, const float *v_scale, pkv_stream_t stream);

/*
 * Bytes of device workspace pkv_paged_decode_attn needs for this shape on a
 * device with `num_sms` SMs (num_sms <= 0: the current device's).  Returns 0
 * for an unsupported shape.  The first 4 bytes of the workspace are the device
 * error word (PKV_DEVERR_*): zero the workspace once after allocating it.
 */
PKV_API size_t pkv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim, int block_size, int cache_dtype,
                                 int num_sms);

/*
 * Paged GQA decode attention ([P1] "KV Cache：Transformer的循环状态" formula;
 * [P1] "PagedAttention与Cache管理" paged gather; [P2] "算子优化要点" online
 * softmax and split of the KV length when the batch is small).
 * For every request r and query head hq (kv head h = hq / G):
 *     s_t = scale * <q[r][hq], K_r[t]>,   t < seq_lens[r]
 *     out[r][hq] = sum_t softmax(s)_t * V_r[t]
 * where K_r[t] is row t % BS of page (block_table[r][t / BS], h) of k_cache
 * (likewise V), dequantised with k_scale/v_scale[block][h] for FP8 pages.
 * Accumulation is fp32; out is bf16.  seq_lens[r] == 0 gives out[r] = 0.
 * Supported: Hq % Hkv == 0, G = Hq / Hkv <= 8; block_size 16 or 32;
 *   PKV_BF16 with head_dim 64 or 128; PKV_FP8_E4M3 with head_dim 128
 *   (FP8: the group's bf16 q values are rescaled by a power of two so the
 *   largest lands in [2^14, 2^15) and converted to fp16; this is exact except
 *   for nonzero elements more than 2^31 times smaller than the group's
 *   largest, which round to the fp16 subnormal grid).
 * Requirements: q, out, caches, workspace 16-byte aligned; workspace_bytes >=
 *   pkv_decode_workspace_size(...) for the same shape and device.
 * The work is one flat list of (request, kv head, page) items split evenly over
 * a persistent grid of warps.  A (request, kv head) unit split over at most six
 * warps is merged, with log-sum-exp weights, by the last of them to finish; wider
 * splits are merged by a small second kernel launched right behind the first
 * (programmatic dependent launch).  No host synchronisation.  The workspace's
 * arrival counters carry a per-call tag, so the workspace needs no clearing
 * between calls; calls that share a workspace must not overlap on the GPU.
 */
PKV_API int pkv_paged_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                          const float *k_scale, const float *v_scale,
                          const int32_t *block_table, int max_blocks_per_seq,
                          const int32_t *seq_lens, int batch, int num_q_heads,
                          int num_kv_heads, int head_dim, int block_size, int num_blocks,
                          int cache_dtype, float scale, void *out, void *workspace,
                          size_t workspace_bytes, pkv_stream_t stream);

/*
 * Multi-query paged attention: q_len >= 1 new query tokens per request, as when a
 * speculative draft of several tokens is verified in one pass ([P1] "投机解码：打破
 * 每步一token的假设"; [P2] "投机解码").  Request r owns query rows
 * q_offsets[r] .. q_offsets[r+1]-1 of q (bf16 [T][Hq][D]; out has the same
 * layout).  Its query i is the token at position seq_lens[r] - q_len + i, whose
 * K/V are already in the cache, and it attends causally ([P1] "KV Cache：
 * Transformer的循环状态") to the cached positions 0 .. seq_lens[r] - q_len + i.
 * A query that sees no token gets a zero row.  Each KV page is read once for all
 * of a request's queries and heads of a group.
 * Supported: 1 <= max_q_len <= 4 with bf16 pages, <= 2 with FP8 pages; every
 * request must have q_offsets[r+1] - q_offsets[r] <= max_q_len (a larger count
 * is clamped and sets PKV_DEVERR_QLEN_CLAMPED; the rows past the clamp are not
 * written).  Everything else as pkv_paged_decode_attn; q_offsets is a device
 * int32 [N + 1] array.  The workspace comes from pkv_multiquery_workspace_size.
 */
PKV_API size_t pkv_multiquery_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                             int head_dim, int block_size, int cache_dtype,
                                             int max_q_len, int num_sms);
PKV_API int pkv_paged_multiquery_attn(const void *q, const int32_t *q_offsets, int max_q_len,
                                      const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_table, int max_blocks_per_seq,
                                      const int32_t *seq_lens, int batch, int num_q_heads,
                                      int num_kv_heads, int head_dim, int block_size,
                                      int num_blocks, int cache_dtype, float scale, void *out,
                                      void *workspace, size_t workspace_bytes,
                                      pkv_stream_t stream);

/*
 * Paged decode attention that allocates nothing.  The sources describe no such
 * call: it exists for callers that cannot call cudaMalloc -- for example a plugin
 * hosted by an engine that owns all device memory and offers no workspace hook,
 * or code on a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not acceptable.  Same arguments and results as
 * pkv_paged_decode_attn without the workspace: the scratch is a 16 MiB static
 * device array inside the library, which every GPU that loads the library holds
 * until the process exits.
 *   - Shapes whose pkv_decode_workspace_size exceeds 16 MiB return
 *     PKV_ERR_WORKSPACE and launch nothing (at head_dim 128 on a 152-SM GPU:
 *     batch * num_kv_heads up to about 3,300).
 *   - The first call on a device, made with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call before
 *     any stream capture.
 *   - Every call shares the one array and it keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls that overlap on the GPU (other
 *     streams, other threads) race on it: serialise them.  The device error word
 *     of this variant stays inside the shared array and is not reported.
 */
PKV_API int pkv_paged_decode_attn_noalloc(const void *q, const void *k_cache,
                                          const void *v_cache, const float *k_scale,
                                          const float *v_scale, const int32_t *block_table,
                                          int max_blocks_per_seq, const int32_t *seq_lens,
                                          int batch, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, int num_blocks,
                                          int cache_dtype, float scale, void *out,
                                          pkv_stream_t stream);

/*
 * Chained prefix block hash ([P3] "优化一：Prefix Cache", 工作原理：按块哈希):
 *     h_0 = seed,   h_i = H(h_{i-1}, tokens of block i),   i = 1 .. floor(L_s / B)
 * with H(p, blk) = fmix64(p XOR FNV1a64(little-endian bytes of the block's int32
 * tokens)), fmix64 = the SplitMix64 output mixer.  Sequence s is
 * tokens[offsets[s] .. offsets[s+1]); its hashes go to
 * hashes[hash_offsets[s] .. hash_offsets[s] + floor(L_s / B)).  A partial last
 * block gets no hash.  tokens int32, offsets/hash_offsets int64 [num_seqs + 1],
 * hashes uint64.  block_size in [1, 1024].
 */
PKV_API int pkv_prefix_block_hash(const int32_t *tokens, const int64_t *offsets, int num_seqs,
                          int block_size, uint64_t seed, uint64_t *hashes,
                          const int64_t *hash_offsets, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
