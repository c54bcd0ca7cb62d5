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
 *       k_cache,v_cache [NB][Hkv][BS][D]  bf16, E4M3 bytes or int8 codes, or
 *                       [NB][Hkv][BS][D/2] bytes of int4 codes; one (block, head)
 *                       page is contiguous
 *       k_scale,v_scale fp32 [NB][Hkv]    quantised caches only
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

/* Cache element type.  The quantised kinds carry one fp32 scale per (block, kv
 * head): element value = code * scale.  PKV_INT4 pages hold two codes per byte,
 * offset-binary (code = q + 8, q in [-7, 7]): value 2b of a row in the low nibble of
 * byte b, value 2b+1 in the high nibble; a row of D values is D/2 bytes
 * ([P3] "优化五：KV 本体压缩": FP16 -> FP8/INT8/INT4). */
enum { PKV_BF16 = 0, PKV_FP8_E4M3 = 1, PKV_INT8 = 2, PKV_INT4 = 3 };

/* Return codes. */
enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,   /* null pointer, bad size, misaligned buffer */
    PKV_ERR_UNSUPPORTED = -2,   /* a shape this build has no kernel for */
    PKV_ERR_WORKSPACE = -3,     /* workspace missing or smaller than required */
    PKV_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed */
    PKV_ERR_NO_BLOCKS = -5      /* block manager: not enough free blocks; nothing changed */
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
 *   PKV_INT8:     byte = clamp(round_half_even(float(x) / scale[blk][h]), -127, 127)
 *                 as int8, same division and scales ([P3] "优化五：KV 本体压缩":
 *                 FP16 -> FP8/INT8/INT4).  NaN inputs give 0.
 *   PKV_INT4:     code = clamp(round_half_even(float(x) / scale[blk][h]), -7, 7),
 *                 same division and scales, stored offset-binary (code + 8) two per
 *                 byte in the nibble layout of the cache-type note above.  NaN
 *                 inputs give code 0.
 * Bytes not addressed by a slot are untouched.  Two tokens with the same slot
 * race (last writer wins, undefined which).
 * Requirements: head_dim % 8 == 0; k, v, caches 16-byte aligned.
 */
PKV_API int pkv_kv_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                       int num_tokens, int num_kv_heads, int head_dim, int block_size,
                       int num_blocks, int cache_dtype, void *k_cache, void *v_cache,
                       const float *k_scale, const float *v_scale, pkv_stream_t stream);

/*
 * KV write that also sets the block scales ([P3] "优化五：KV 本体压缩" and 传输量化:
 * 8-bit KV with a scale; here the scale is derived from the data being written).
 * For every (block, kv head) that receives at least one row in this call, its scale
 * becomes amax / QMAX over the |values| of the rows written to it by this call
 * (QMAX = 448 for PKV_FP8_E4M3, 127 for PKV_INT8, 7 for PKV_INT4; binary32 divide; NaN values
 * ignored; an all-zero block gets 1); the rows are then coded exactly as
 * pkv_kv_cache_write does with those scales.  Scales of blocks receiving no row are
 * unchanged; bytes written to a touched block by earlier calls are not re-coded, so
 * use it for whole blocks (prefill) and pkv_kv_cache_write for later tokens.
 * k_scale / v_scale are read and written.  workspace: device, >=
 * pkv_rescale_workspace_size(num_blocks, num_kv_heads) bytes, 4-byte aligned, no
 * clearing needed.  Three launches, no host synchronisation.
 */
PKV_API size_t pkv_rescale_workspace_size(int num_blocks, int num_kv_heads);
PKV_API int pkv_kv_cache_write_rescale(const void *k, const void *v,
                                       const int64_t *slot_mapping, int num_tokens,
                                       int num_kv_heads, int head_dim, int block_size,
                                       int num_blocks, int cache_dtype, void *k_cache,
                                       void *v_cache, float *k_scale, float *v_scale,
                                       void *workspace, size_t workspace_bytes,
                                       pkv_stream_t stream);

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
 *   PKV_BF16 with head_dim 64 or 128; PKV_FP8_E4M3, PKV_INT8 and PKV_INT4 with
 *   head_dim 128 (quantised pages: the group's bf16 q values are rescaled by a
 *   power of two so the largest lands in [2^14, 2^15) and converted to fp16; this
 *   is exact except for nonzero elements more than 2^31 times smaller than the
 *   group's largest, which round to the fp16 subnormal grid.  INT8 and INT4 K codes
 *   enter the fp16 mma with their offset, 1024 plus the biased code, subtracted once
 *   per score.  V codes enter as fp16 subnormals (biased code * 2^-24) against
 *   P * v_scale rounded to fp16; the small offset of the biased code (128 or 8) is
 *   subtracted once per output.  E4M3 V codes are widened exactly and also meet
 *   P * v_scale in fp16).
 * Requirements: q, out, caches, workspace 16-byte aligned; workspace_bytes >=
 *   pkv_decode_workspace_size(...) for the same shape and device.
 * The work is one flat list of (request, kv head, page) items split evenly over
 * a persistent grid of warps.  The partial results of a (request, kv head) unit
 * split over several warps are merged, with log-sum-exp weights, by a small second
 * kernel launched right behind the first (programmatic dependent launch).  No host
 * synchronisation.  The workspace needs no clearing between calls; calls that
 * share a workspace must not overlap on the GPU.
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
 * Supported: 1 <= max_q_len <= 4 with bf16 pages, <= 2 with 8-bit pages; every
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
 * Decode with the step's cache write folded in (bf16 pages, one query per request):
 * the same result and the same cache contents as pkv_compute_slot_mapping +
 * pkv_kv_cache_write of each request's newest token (position seq_lens[r] - 1) followed
 * by pkv_paged_decode_attn ([P1] "KV Cache：Transformer的循环状态": the new token's K/V
 * join the cache and the query attends to them; [P3] "组合拳：一次请求的完整旅程": the
 * new K/V go back into the pool).  k_new, v_new: bf16 [batch][Hkv][D], the newest token's
 * rows.  The warp whose tile holds that position writes the rows into the token's slot
 * (block_table[r][(seq_lens[r]-1) / BS], row (seq_lens[r]-1) % BS; a block id outside the
 * pool is not written and is flagged) and uses them in place of the page's stored row, so
 * the attention needs no write kernel before it.  seq_lens[r] == 0: nothing is written,
 * out[r] = 0.  Shapes, workspace (pkv_decode_workspace_size with PKV_BF16) and every
 * other argument as pkv_paged_decode_attn; k_new / v_new 16-byte aligned.
 */
PKV_API int pkv_paged_decode_attn_append(const void *q, const void *k_new, const void *v_new,
                                         void *k_cache, void *v_cache,
                                         const int32_t *block_table, int max_blocks_per_seq,
                                         const int32_t *seq_lens, int batch, int num_q_heads,
                                         int num_kv_heads, int head_dim, int block_size,
                                         int num_blocks, float scale, void *out,
                                         void *workspace, size_t workspace_bytes,
                                         pkv_stream_t stream);

/*
 * Paged decode attention over a shared prefix ([P3] "优化一：Prefix Cache": requests whose
 * first blocks hash alike share those physical blocks; [P2] "缓存命中与复用").  The same
 * result as pkv_paged_decode_attn (bf16 pages, one query per request) when every request
 * of the batch begins with the same prefix_len tokens held in the same blocks: the
 * first prefix_len / block_size entries of every block-table row equal row 0's, and
 * seq_lens[r] >= prefix_len (the caller's contract, not checked on the device).  The
 * shared pages are read once for the whole batch instead of once per request:
 *   1. all the batch's queries, stacked as the rows of the tensor-core prefill kernel,
 *      attend without mask to row 0's first prefix_len tokens (split in a few KV chunks
 *      so that the SMs are covered); each (request, query head) leaves an unnormalised
 *      partial (o, m, l) per chunk in the workspace;
 *   2. the decode kernel attends each request to its tokens prefix_len .. seq_lens[r]-1
 *      and leaves a partial for every (request, KV head);
 *   3. a merge combines each row's partials with log-sum-exp weights into out.
 * When step 1 needs few CTAs (its 128-row query tiles x num_kv_heads at most a third of
 * the SMs) and, by a cost estimate that takes each tail as half the room the block table
 * leaves after the prefix, finishes sooner that way, it runs as one KV chunk per CTA on a
 * second stream the library keeps per device, while step 2 runs on stream sized to the
 * remaining SMs; stream waits for it before step 3.  That second stream and its two
 * events are created by the first such call with the device current (make that call
 * outside stream capture; later calls capture into a CUDA graph, the fork and join
 * becoming graph edges) and again after the device's context changes.
 * prefix_len must be a multiple of block_size and at most max_blocks_per_seq *
 * block_size (else PKV_ERR_INVALID_ARG); 0 runs the plain decode.  scale finite and > 0.
 * Supported: bf16 pages, head_dim 64 or 128, block_size 16 or 32, G = Hq / Hkv in
 * {1, 2, 4, 8}; otherwise PKV_ERR_UNSUPPORTED.  workspace: at least
 * pkv_shared_prefix_workspace_size(...) bytes (0 for an unsupported shape), 256-byte
 * aligned, no clearing needed; its first word is the device error word.  Three
 * launches, no host synchronisation; PKV_ERR_CUDA if the second stream or its events
 * cannot be created.
 */
PKV_API size_t pkv_shared_prefix_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                                int head_dim, int block_size, int prefix_len,
                                                int num_sms);
PKV_API int pkv_paged_decode_attn_shared_prefix(const void *q, const void *k_cache,
                                                const void *v_cache, const int32_t *block_table,
                                                int max_blocks_per_seq, const int32_t *seq_lens,
                                                int batch, int num_q_heads, int num_kv_heads,
                                                int head_dim, int block_size, int num_blocks,
                                                int prefix_len, float scale, void *out,
                                                void *workspace, size_t workspace_bytes,
                                                pkv_stream_t stream);
/*
 * The plan pkv_paged_decode_attn_shared_prefix takes for these arguments on a device with
 * num_sms SMs (num_sms <= 0: the current device's): 1 overlapped (the prefix pass on the
 * library's second stream beside the tail decode), 0 sequential; negative: the status the
 * call would return for an invalid or unsupported shape.  When not null, *prefix_ctas
 * receives the prefix pass's CTAs and *decode_sms the SMs the tail decode is sized for.
 * Host only: launches nothing.
 */
PKV_API int pkv_shared_prefix_plan(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, int prefix_len,
                                   int num_sms, int *prefix_ctas, int *decode_sms);

/*
 * Paged decode attention that allocates nothing.  The sources describe no such
 * call: it exists for callers that cannot call cudaMalloc -- for example a plugin
 * hosted by an engine that owns all device memory and offers no workspace hook,
 * or code on a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not acceptable.  Same arguments and results as
 * pkv_paged_decode_attn without the workspace: the scratch is a 16 MiB static
 * device array inside the library, which every GPU that loads the library holds
 * until the process exits.
 *   - The limit: a call runs when pkv_decode_workspace_size(batch, ..., 0) on the
 *     current device is at most 16 MiB; larger shapes return PKV_ERR_WORKSPACE and
 *     launch nothing.  That size grows with batch * num_kv_heads and with the
 *     device's SM count, so the bound depends on the GPU: on a 152-SM GPU at
 *     head_dim 128 it is batch * num_kv_heads up to about 2,900 for bf16 pages,
 *     2,750 for E4M3 and int8 pages and 2,140 for int4 pages (whose plans run more
 *     warps per SM).
 *   - Argument checks come in the same order and return the same statuses as
 *     pkv_paged_decode_attn's; a failed CUDA query returns PKV_ERR_CUDA.
 *   - The first call on a device, made with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call before
 *     any stream capture.  The address is kept per device and looked up again when
 *     the device's current context has changed (after cudaDeviceReset, say).
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
 * hashes[hash_offsets[s] .. hash_offsets[s] + floor(L_s / B)), and never more than
 * hash_offsets[s+1] - hash_offsets[s] of them.  A partial last block gets no hash.  tokens int32, offsets/hash_offsets int64 [num_seqs + 1],
 * hashes uint64.  block_size in [1, 1024].
 */
PKV_API int pkv_prefix_block_hash(const int32_t *tokens, const int64_t *offsets, int num_seqs,
                          int block_size, uint64_t seed, uint64_t *hashes,
                          const int64_t *hash_offsets, pkv_stream_t stream);

/*
 * The same chain, resumed ([P3] "优化一：Prefix Cache", 工作原理：按块哈希: h_i depends
 * only on h_{i-1} and block i).  A serving step that has hashed a sequence's first
 * k full blocks before passes h_k and k, and only the blocks filled since are read
 * and hashed: a decode step typically hashes zero or one block per sequence
 * instead of its whole history.
 *   tokens, offsets  as pkv_prefix_block_hash: all tokens of sequence s
 *   first_blocks     device int64 [num_seqs]: k_s, full blocks already hashed
 *                    (negative reads as 0; at or past floor(L_s / B): nothing to do)
 *   prev_hashes      device uint64 [num_seqs]: h_{k_s} (the seed when k_s = 0)
 *   hashes           receives h_{k_s+1}, h_{k_s+2}, ... at hash_offsets[s] ..
 *   hash_offsets     device int64 [num_seqs + 1]; sequence s gets at most
 *                    hash_offsets[s+1] - hash_offsets[s] hashes, normally
 *                    max(0, floor(L_s / B) - k_s).  Entries past what is written
 *                    are left untouched.
 * With k_s = 0 and prev_hashes[s] = seed this equals pkv_prefix_block_hash.
 * block_size in [1, 1024]; any NULL pointer (num_seqs > 0) is PKV_ERR_INVALID_ARG.
 */
PKV_API int pkv_prefix_block_hash_resume(const int32_t *tokens, const int64_t *offsets,
                                         int num_seqs, int block_size,
                                         const uint64_t *prev_hashes,
                                         const int64_t *first_blocks, uint64_t *hashes,
                                         const int64_t *hash_offsets, pkv_stream_t stream);

/*
 * Paged prefill attention ([P1] "推理的两阶段计算形态": prefill processes every prompt
 * token at once and is compute-bound; "KV Cache：Transformer的循环状态": causal
 * attention; "PagedAttention与Cache管理": the block table).  A chunk of new tokens per
 * request, their K/V already written to the pages (pkv_kv_cache_write): request r's
 * query rows are q[q_offsets[r] .. q_offsets[r+1]) (q_len_r rows, int32 q_offsets
 * [batch + 1], q_offsets[batch] <= total_q); row i is the token at position
 * seq_lens[r] - q_len_r + i and attends to positions 0 .. seq_lens[r] - q_len_r + i.
 * A row that sees no token is zero.  Same result as pkv_paged_multiquery_attn, any
 * q_len.  max_q_len bounds every q_len_r: rows past it are not computed and
 * PKV_DEVERR_QLEN_CLAMPED is set; a request whose rows run past total_q is skipped
 * and flagged the same way.  Runs on the tcgen05 tensor cores: one CTA per 128 query
 * rows (128/G tokens x the G heads of a KV head).
 *   q, out          bf16 [total_q][Hq][D], 16-byte aligned; rows of no request untouched
 *   k/v_cache       pages of cache_dtype (layouts above); k/v_scale for quantised kinds
 *   workspace       quantised kinds only: pkv_prefill_workspace_size bytes, 256-byte
 *                   aligned.  The batch's pages are first expanded to bf16 there
 *                   (code * scale, rounded to nearest even) in request order, then the
 *                   bf16 kernel runs on that pool.  bf16 pages need no workspace (NULL).
 *   error_word      device uint32 collecting PKV_DEVERR_* bits (sticky), or NULL
 * scale must be finite and > 0 (else PKV_ERR_INVALID_ARG).
 * Supported: head_dim 64 or 128, block_size 16 or 32, G in {1, 2, 4, 8}; other shapes
 * return PKV_ERR_UNSUPPORTED. */
PKV_API size_t pkv_prefill_workspace_size(int batch, int max_blocks_per_seq, int num_kv_heads,
                                          int head_dim, int block_size, int cache_dtype);
PKV_API int pkv_paged_prefill_attn(const void *q, const int32_t *q_offsets, int total_q,
                                   int max_q_len, const void *k_cache, const void *v_cache,
                                   const float *k_scale, const float *v_scale,
                                   const int32_t *block_table, int max_blocks_per_seq,
                                   const int32_t *seq_lens, int batch, int num_q_heads,
                                   int num_kv_heads, int head_dim, int block_size,
                                   int num_blocks, int cache_dtype, float scale, void *out,
                                   void *workspace, size_t workspace_bytes,
                                   uint32_t *error_word, pkv_stream_t stream);

/*
 * Copy whole blocks inside the cache pool, for copy-on-write of a shared block
 * ([P1] "PagedAttention与Cache管理": physical blocks are shared between
 * sequences, and a sequence that must change a shared block gets its own copy
 * first -- beam search).  For each pair i, block block_mapping[2i] (source) is
 * copied to block block_mapping[2i+1] (destination): all num_kv_heads pages of K
 * and of V, BS*D elements each, and for 8-bit caches the 2*num_kv_heads fp32
 * scales of the block.  block_mapping is a DEVICE int32 array [num_pairs][2].
 *   - Destinations must be distinct and must not be the source of another pair
 *     (the block manager below only ever names a fresh block as destination);
 *     overlapping pairs give an unspecified result, never an out-of-bounds access.
 *   - A pair with an id outside [0, num_blocks) or with source == destination is
 *     skipped.
 *   - num_pairs == 0 launches nothing.  k_scale/v_scale are required for the
 *     8-bit kinds and ignored for bf16.
 */
PKV_API int pkv_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                            const int32_t *block_mapping, int num_pairs, int num_kv_heads,
                            int head_dim, int block_size, int num_blocks, int cache_dtype,
                            pkv_stream_t stream);

/*
 * Host block manager: owns the ids of the physical blocks of one cache pool and
 * builds the block tables the kernels above read ([P1] "PagedAttention与Cache管理":
 * on-demand blocks, waste under one block per sequence, sharing and copy-on-write;
 * [P3] "优化一：Prefix Cache": full blocks found again by their chained hash;
 * [P2] "缓存命中与复用": block-granular hits that must be a prefix, LRU eviction,
 * blocks in use are never evicted).  Pure host code, touches no device memory and
 * no CUDA context; every call is thread-safe (one mutex per manager).
 *
 * States of a block: FREE (refcount 0, no hash), USED (refcount >= 1, hash or
 * not), CACHED (refcount 0, still registered under its hash, reusable by a hit,
 * evictable).  Deterministic policy:
 *   - a fresh block is the lowest-numbered FREE block; with none FREE, the least
 *     recently released CACHED block is evicted (its hash forgotten) and reused;
 *   - pkv_bm_add_sequence takes the leading blocks whose hashes are registered
 *     (stopping at the first miss), then fresh blocks for the rest; the first
 *     num_hashes fresh blocks are registered under their hashes;
 *   - pkv_bm_free_sequence releases the blocks last to first, so the tail of a
 *     prefix becomes CACHED before its head and is evicted first;
 *   - a hash is registered to at most one block: the first registration wins;
 *   - calls that need blocks are all-or-nothing and return PKV_ERR_NO_BLOCKS with
 *     no change when too few FREE + CACHED blocks remain.
 * Sequence ids are any int64 chosen by the caller; an unknown id, or adding an id
 * that exists, returns PKV_ERR_INVALID_ARG.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager of blocks 0 .. num_blocks-1, all FREE, of block_size tokens each. */
PKV_API int pkv_bm_create(int num_blocks, int block_size, pkv_block_manager **out);
PKV_API void pkv_bm_destroy(pkv_block_manager *m);
/* FREE + CACHED blocks (what a call may still take), or a negative status. */
PKV_API int pkv_bm_num_available(pkv_block_manager *m);
/* Register a sequence of num_tokens tokens whose first num_hashes full blocks have
 * the given chained hashes (num_hashes <= num_tokens / block_size; pass the
 * output of pkv_prefix_block_hash).  Writes ceil(num_tokens / block_size) block
 * ids to block_ids (host int32) and the number of leading blocks reused from the
 * cache to *cached_blocks (may be NULL). */
PKV_API int pkv_bm_add_sequence(pkv_block_manager *m, int64_t seq_id, int64_t num_tokens,
                                const uint64_t *block_hashes, int num_hashes,
                                int32_t *block_ids, int *cached_blocks);
/* The sequence now holds num_tokens tokens (>= before): appends fresh blocks as
 * needed; *new_block (may be NULL) gets the last block appended, or -1 if none. */
PKV_API int pkv_bm_grow(pkv_block_manager *m, int64_t seq_id, int64_t num_tokens,
                        int32_t *new_block);
/* Register the sequence's full logical block under hash (after it was filled). */
PKV_API int pkv_bm_commit_block_hash(pkv_block_manager *m, int64_t seq_id, int logical_block,
                                     uint64_t hash);
/* child_id gets the parent's blocks and token count; every block's refcount + 1. */
PKV_API int pkv_bm_fork(pkv_block_manager *m, int64_t parent_id, int64_t child_id);
/* Before writing into logical_block of seq_id: if its block is shared (refcount
 * > 1) or registered under a hash, the sequence gets a fresh block in its place
 * and *copy_src / *copy_dst name the copy to make first (pkv_copy_blocks);
 * otherwise both are -1 and the block may be written in place. */
PKV_API int pkv_bm_prepare_write(pkv_block_manager *m, int64_t seq_id, int logical_block,
                                 int32_t *copy_src, int32_t *copy_dst);
/* Release every block of the sequence and forget the id. */
PKV_API int pkv_bm_free_sequence(pkv_block_manager *m, int64_t seq_id);
/* Copies the sequence's block ids to block_ids (capacity entries available);
 * returns their number, or a negative status.  block_ids == NULL returns the
 * number only. */
PKV_API int pkv_bm_block_table(pkv_block_manager *m, int64_t seq_id, int32_t *block_ids,
                               int capacity);
/* Refcount of a block (0 for FREE and CACHED), or a negative status. */
PKV_API int pkv_bm_refcount(pkv_block_manager *m, int block);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
