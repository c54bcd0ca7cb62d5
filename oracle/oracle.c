/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the paged-KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library,
 * its Python binding) may include, link, load or call this file.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no code, header, table or constant generator with the CUDA path.
 *
 * Every function is the plain definition of one step, written as loops in
 * the order the sources state it.  Sources cited by page title and section:
 *
 *   [P1] "深入LLM推理：从KV Cache到PD分离的Serving全景解析" (kongchang.com)
 *   [P2] "GPU推理深度拆解：KV Cache视角" (cutenote.app)
 *   [P3] "ai-infra-7" (zer0e blog: KV Cache under PD disaggregation)
 *
 * Readings where the sources are silent (hash function, FP8 scale
 * granularity, cache layout, GQA head grouping) are stated at each function
 * and listed in the design notes of the repository.
 *
 * Layout conventions (shared *as a specification* with the library, not as
 * code):
 *   q        bf16  [N][Hq][D]
 *   caches   [NB][Hkv][BS][D]   cache_kind 0: bf16 (uint16 bit patterns),
 *                               1: E4M3 bytes, 2: int8
 *   scales   fp32  [NB][Hkv]    (8-bit kinds; one per (block, kv head), K and V separate)
 *   block_table int32 [N][MB], seq_lens int32 [N]
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (no -ffast-math: the fp32 divide in
 * the FP8 write must be the IEEE round-to-nearest divide).
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE-754 binary32 pattern; widening is
 * exact. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; the largest
 * finite magnitude is S.1111.110 = 1.75 * 2^8 = 448; exponent field 0 encodes
 * subnormals 2^-6 * m/8.  Decoding is exact in double.
 * (The FP8 KV format of [P3] "优化三：KV 传输优化", item 3 传输量化.) */
double orc_e4m3_to_double(uint8_t x)
{
    int s = (x >> 7) & 1;
    int e = (x >> 3) & 0xF;
    int m = x & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Encode a binary32 value to E4M3, rounding to nearest with ties to even and
 * saturating to the largest finite value (|x| >= 448 -> +-448, infinities
 * included).  NaN encodes as S.1111.111 with the input's sign. */
uint8_t orc_e4m3_from_float(float xf)
{
    double x = (double)xf;
    uint8_t sign = signbit(xf) ? 0x80 : 0x00;
    double a = fabs(x);
    if (isnan(xf))
        return (uint8_t)(sign | 0x7F);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; rint() rounds half to even in
         * the default rounding mode.  A result of 8 is the smallest normal
         * (code 0x08), which the code arithmetic yields directly. */
        double q = rint(a * 512.0);
        return (uint8_t)(sign | (uint8_t)q);
    }
    {
        int E;
        double f = frexp(a, &E);        /* a = f * 2^E, f in [0.5, 1) */
        int e = E - 1;                  /* a = (2f) * 2^e, 2f in [1, 2) */
        double mant = (2.0 * f - 1.0) * 8.0;  /* exact in double */
        double mr = rint(mant);
        if (mr >= 8.0) {                /* rounded up into the next binade */
            mr = 0.0;
            e += 1;
        }
        {
            int code = ((e + 7) << 3) | (int)mr;
            if (code > 0x7E)
                code = 0x7E;
            return (uint8_t)(sign | (uint8_t)code);
        }
    }
}

/* Symmetric int8 code of a binary32 value: round to nearest, ties to even, then
 * clamp to [-127, 127] (the KV quantisation to INT8 of [P3] "优化五：KV 本体压缩",
 * FP16 -> FP8/INT8/INT4; per-(block, head) scale, symmetric so that 0 maps to 0). */
int8_t orc_int8_from_float(float x)
{
    double r = rint((double)x);   /* x is a binary32 value: exact in double */
    if (isnan(x))
        return 0;
    if (r > 127.0)
        r = 127.0;
    if (r < -127.0)
        r = -127.0;
    return (int8_t)r;
}

/* Symmetric int4 code of a binary32 value, stored offset-binary in a nibble: the
 * value q = round-to-nearest-even(x) clamped to [-7, 7] (NaN -> 0) is kept as the
 * unsigned nibble q + 8 (the INT4 KV of [P3] "优化五：KV 本体压缩"; symmetric, one
 * scale per (block, head)).  A cache row of D values is D/2 bytes: value 2b sits
 * in the low nibble of byte b, value 2b+1 in its high nibble. */
uint8_t orc_int4_code_from_float(float x)
{
    double r = rint((double)x);
    if (isnan(x))
        r = 0.0;
    if (r > 7.0)
        r = 7.0;
    if (r < -7.0)
        r = -7.0;
    return (uint8_t)((int)r + 8);
}

/* ------------------------------------------------------------------------ */
/* KV size formula  ([P3] "KV Cache 到底有多大？", KV Size equation)          */
/* ------------------------------------------------------------------------ */

/* KV Size = 2 x L x H_kv x d x S x b : the leading 2 counts K and V. */
int64_t orc_kv_bytes(int64_t L, int64_t Hkv, int64_t d, int64_t S, int64_t b)
{
    return 2 * L * Hkv * d * S * b;
}

/* ------------------------------------------------------------------------ */
/* Slot mapping  ([P1] "PagedAttention与Cache管理": the block table maps a   */
/* request's logical block to a physical block of 16 or 32 tokens)          */
/* ------------------------------------------------------------------------ */

/* Token t belongs to request req_idx[t] at position positions[t].  Its
 * physical cache row ("slot") is
 *     block_table[r][pos / BS] * BS + pos % BS.
 * A negative position marks a padding token: slot -1 (not written). */
void orc_slot_mapping(const int32_t *block_table, int max_blocks_per_seq,
                      const int32_t *req_idx, const int32_t *positions,
                      int num_tokens, int block_size, int64_t *slot_mapping)
{
    for (int t = 0; t < num_tokens; ++t) {
        int r = req_idx[t];
        int pos = positions[t];
        if (pos < 0) {
            slot_mapping[t] = -1;
            continue;
        }
        int logical_block = pos / block_size;
        int offset = pos % block_size;
        int64_t physical_block =
            block_table[(int64_t)r * max_blocks_per_seq + logical_block];
        slot_mapping[t] = physical_block * block_size + offset;
    }
}

/* ------------------------------------------------------------------------ */
/* KV cache write  ([P3] "组合拳：一次请求的完整旅程": newly generated KV is   */
/* written back into the cache pool; FP8 per [P3] 传输量化)                   */
/* ------------------------------------------------------------------------ */

/* Writes row (t, h) of k and v (bf16 [T][Hkv][D]) to cache row
 * [slot / BS][h][slot % BS][:].  bf16 caches receive the bytes unchanged.
 * Quantised caches receive code(float(x) / scale[blk][h]) where the division is the
 * IEEE binary32 divide and code is E4M3 (RNE, saturating), int8 (RNE, clamp to
 * +-127) or int4 (RNE, clamp to +-7, two codes per byte).  Tokens with slot < 0
 * are skipped; every other byte of the caches is left as it was. */
void orc_kv_cache_write(const uint16_t *k, const uint16_t *v,
                        const int64_t *slot_mapping, int num_tokens,
                        int num_kv_heads, int head_dim, int block_size,
                        int cache_kind, void *k_cache, void *v_cache,
                        const float *k_scale, const float *v_scale)
{
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t src = ((int64_t)t * num_kv_heads + h) * head_dim;
            int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
            for (int d = 0; d < head_dim; ++d) {
                if (!cache_kind) {
                    ((uint16_t *)k_cache)[dst + d] = k[src + d];
                    ((uint16_t *)v_cache)[dst + d] = v[src + d];
                } else {
                    float ks = k_scale[blk * num_kv_heads + h];
                    float vs = v_scale[blk * num_kv_heads + h];
                    float kx = (float)orc_bf16_to_double(k[src + d]);
                    float vx = (float)orc_bf16_to_double(v[src + d]);
                    volatile float kq = kx / ks;  /* binary32 divide, RN */
                    volatile float vq = vx / vs;
                    if (cache_kind == 1) {
                        ((uint8_t *)k_cache)[dst + d] = orc_e4m3_from_float(kq);
                        ((uint8_t *)v_cache)[dst + d] = orc_e4m3_from_float(vq);
                    } else if (cache_kind == 3) {
                        int64_t byte = (dst + d) >> 1;
                        int shift = (d & 1) ? 4 : 0;
                        uint8_t keep = (uint8_t)(0xF0u >> shift);
                        uint8_t *kb = (uint8_t *)k_cache + byte, *vb = (uint8_t *)v_cache + byte;
                        *kb = (uint8_t)((*kb & keep) | (orc_int4_code_from_float(kq) << shift));
                        *vb = (uint8_t)((*vb & keep) | (orc_int4_code_from_float(vq) << shift));
                    } else {
                        ((int8_t *)k_cache)[dst + d] = orc_int8_from_float(kq);
                        ((int8_t *)v_cache)[dst + d] = orc_int8_from_float(vq);
                    }
                }
            }
        }
    }
}

/* KV write that first sets the scale of every (block, head) receiving rows in
 * this call: scale = amax / QMAX over the |values| of those rows (QMAX = 448 for
 * E4M3, 127 for int8, 7 for int4; binary32 divide; NaN values ignored; amax = 0
 * gives 1), then writes the rows as orc_kv_cache_write does.  Scales of blocks
 * receiving no row are unchanged, and bytes written to a touched block by earlier
 * calls are not re-coded.  cache_kind 1, 2 or 3. */
void orc_kv_cache_write_rescale(const uint16_t *k, const uint16_t *v,
                                const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                int head_dim, int block_size, int cache_kind, void *k_cache,
                                void *v_cache, float *k_scale, float *v_scale)
{
    int64_t nblk = 0;
    for (int t = 0; t < num_tokens; ++t)
        if (slot_mapping[t] >= 0 && slot_mapping[t] / block_size + 1 > nblk)
            nblk = slot_mapping[t] / block_size + 1;
    float *kmax = (float *)malloc(sizeof(float) * (size_t)(nblk * num_kv_heads + 1));
    float *vmax = (float *)malloc(sizeof(float) * (size_t)(nblk * num_kv_heads + 1));
    for (int64_t i = 0; i < nblk * num_kv_heads; ++i)
        kmax[i] = vmax[i] = -1.0f;              /* -1: not touched by this call */
    for (int t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t i = blk * num_kv_heads + h;
            if (kmax[i] < 0.0f)
                kmax[i] = vmax[i] = 0.0f;
            for (int d = 0; d < head_dim; ++d) {
                float kx = fabsf((float)orc_bf16_to_double(k[((int64_t)t * num_kv_heads + h) * head_dim + d]));
                float vx = fabsf((float)orc_bf16_to_double(v[((int64_t)t * num_kv_heads + h) * head_dim + d]));
                if (!isnan(kx) && kx > kmax[i])
                    kmax[i] = kx;
                if (!isnan(vx) && vx > vmax[i])
                    vmax[i] = vx;
            }
        }
    }
    volatile float qmax = cache_kind == 1 ? 448.0f : (cache_kind == 3 ? 7.0f : 127.0f);
    for (int64_t i = 0; i < nblk * num_kv_heads; ++i) {
        if (kmax[i] < 0.0f)
            continue;
        volatile float ks = kmax[i] > 0.0f ? kmax[i] / qmax : 1.0f;   /* binary32 divide */
        volatile float vs = vmax[i] > 0.0f ? vmax[i] / qmax : 1.0f;
        k_scale[i] = ks;
        v_scale[i] = vs;
    }
    free(kmax);
    free(vmax);
    orc_kv_cache_write(k, v, slot_mapping, num_tokens, num_kv_heads, head_dim, block_size,
                       cache_kind, k_cache, v_cache, k_scale, v_scale);
}

/* ------------------------------------------------------------------------ */
/* Paged decode attention  ([P1] "KV Cache：Transformer的循环状态":           */
/* Attention(Q,K,V) = softmax(QK^T/sqrt(d)) V with GQA query heads sharing a */
/* KV head; [P1] "PagedAttention与Cache管理": K/V gathered via block table)  */
/* ------------------------------------------------------------------------ */

/* Value of cache element (blk, h, off, d) in fp64, dequantised for fp8. */
static double cache_elem(const void *cache, int cache_kind, const float *scale,
                         int64_t blk, int h, int64_t off, int d,
                         int num_kv_heads, int block_size, int head_dim)
{
    int64_t idx = ((blk * num_kv_heads + h) * block_size + off) * head_dim + d;
    if (!cache_kind)
        return orc_bf16_to_double(((const uint16_t *)cache)[idx]);
    if (cache_kind == 1)
        return orc_e4m3_to_double(((const uint8_t *)cache)[idx]) *
               (double)scale[blk * num_kv_heads + h];
    if (cache_kind == 3) {   /* int4: nibble d % 2 of byte idx / 2, offset-binary */
        uint8_t byte = ((const uint8_t *)cache)[idx >> 1];
        int code = (idx & 1) ? (byte >> 4) : (byte & 0xF);
        return (double)(code - 8) * (double)scale[blk * num_kv_heads + h];
    }
    return (double)((const int8_t *)cache)[idx] * (double)scale[blk * num_kv_heads + h];
}

/* One (request r, query head hq) output row.  Query head hq reads KV head
 * hq / G with G = Hq / Hkv (consecutive query heads form a group).  The
 * request attends to all seq_lens[r] cached tokens, in logical order: token
 * t lives in physical block block_table[r][t / BS] at offset t % BS.
 *   s_t = scale * sum_d q[d] k_t[d]
 *   p_t = exp(s_t - max_s) / sum_u exp(s_u - max_s)
 *   o   = sum_t p_t v_t
 * out_row receives o (D doubles).  probs (nullable) receives p (seq_len
 * doubles).  lse (nullable) receives log(sum_t exp(s_t)).
 * seq_len <= 0 gives o = 0 and lse = -inf. */
void orc_decode_row(const uint16_t *q, const void *k_cache, const void *v_cache,
                    const float *k_scale, const float *v_scale,
                    const int32_t *block_table, int max_blocks_per_seq,
                    const int32_t *seq_lens, int num_q_heads, int num_kv_heads,
                    int head_dim, int block_size, int cache_kind, double scale,
                    int r, int hq, double *out_row, double *probs, double *lse)
{
    int G = num_q_heads / num_kv_heads;
    int h = hq / G;
    int S = seq_lens[r];
    const uint16_t *qrow = q + ((int64_t)r * num_q_heads + hq) * head_dim;
    for (int d = 0; d < head_dim; ++d)
        out_row[d] = 0.0;
    if (S <= 0) {
        if (lse)
            *lse = -INFINITY;
        return;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)S);
    double smax = -INFINITY;
    for (int t = 0; t < S; ++t) {
        int64_t blk = block_table[(int64_t)r * max_blocks_per_seq + t / block_size];
        int64_t off = t % block_size;
        double acc = 0.0;
        for (int d = 0; d < head_dim; ++d)
            acc += orc_bf16_to_double(qrow[d]) *
                   cache_elem(k_cache, cache_kind, k_scale, blk, h, off, d,
                              num_kv_heads, block_size, head_dim);
        s[t] = scale * acc;
        if (s[t] > smax)
            smax = s[t];
    }
    double denom = 0.0;
    for (int t = 0; t < S; ++t) {
        s[t] = exp(s[t] - smax);
        denom += s[t];
    }
    for (int t = 0; t < S; ++t) {
        double p = s[t] / denom;
        int64_t blk = block_table[(int64_t)r * max_blocks_per_seq + t / block_size];
        int64_t off = t % block_size;
        for (int d = 0; d < head_dim; ++d)
            out_row[d] += p * cache_elem(v_cache, cache_kind, v_scale, blk, h, off,
                                         d, num_kv_heads, block_size, head_dim);
        if (probs)
            probs[t] = p;
    }
    if (lse)
        *lse = smax + log(denom);
    free(s);
}

/* Multi-query paged attention: several new query tokens per request, the case of
 * verifying speculative draft tokens in one pass ([P1] "投机解码：打破每步一token的
 * 假设": the large model checks K drafted tokens in a single forward) with the
 * causal rule of [P1] "KV Cache：Transformer的循环状态" (a token sees itself and
 * everything before it).
 * Request r owns query rows q_offsets[r] .. q_offsets[r+1]-1 (q bf16 [T][Hq][D]);
 * with q_len = q_offsets[r+1] - q_offsets[r], its query i is the token at position
 * seq_lens[r] - q_len + i, whose K/V are already in the cache, and it attends to
 * the cached tokens at positions 0 .. seq_lens[r] - q_len + i.  Each row is the
 * attention of orc_decode_row restricted to that prefix of the request; a query
 * that sees no token gets a zero row.  out [T][Hq][D] doubles. */
void orc_multiquery_attn(const uint16_t *q, const int32_t *q_offsets, const void *k_cache,
                         const void *v_cache, const float *k_scale, const float *v_scale,
                         const int32_t *block_table, int max_blocks_per_seq,
                         const int32_t *seq_lens, int batch, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int cache_kind, double scale,
                         double *out)
{
    int64_t T = q_offsets[batch];
    int64_t rows = T * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t row = 0; row < rows; ++row) {
        int64_t tq = row / num_q_heads;          /* query token */
        int hq = (int)(row % num_q_heads);
        int r = 0;
        while (q_offsets[r + 1] <= tq)
            ++r;
        int q_len = q_offsets[r + 1] - q_offsets[r];
        int i = (int)(tq - q_offsets[r]);
        int visible = seq_lens[r] - q_len + i + 1;  /* tokens at positions 0..pos */
        if (visible < 0)
            visible = 0;
        if (visible > seq_lens[r])
            visible = seq_lens[r];
        /* the same computation as a single-query decode of a request whose cache
         * holds only the visible prefix, with this row's query */
        int32_t len1 = visible;
        const int32_t *bt_row = block_table + (int64_t)r * max_blocks_per_seq;
        orc_decode_row(q + tq * num_q_heads * head_dim, k_cache, v_cache, k_scale, v_scale,
                       bt_row, max_blocks_per_seq, &len1, num_q_heads, num_kv_heads, head_dim,
                       block_size, cache_kind, scale, 0, hq, out + row * head_dim, NULL,
                       NULL);
    }
}

/* Selected rows of orc_multiquery_attn: rows[i] = tq * Hq + hq for query token tq
 * (an index into q's T rows) and query head hq; out [count][D] doubles.  Each row
 * is computed exactly as in orc_multiquery_attn (the same visible prefix and the
 * same single-row attention); used where the whole output is too large to compute
 * on the host (long prefill chunks). */
void orc_multiquery_rows(const uint16_t *q, const int32_t *q_offsets, const void *k_cache,
                         const void *v_cache, const float *k_scale, const float *v_scale,
                         const int32_t *block_table, int max_blocks_per_seq,
                         const int32_t *seq_lens, int batch, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int cache_kind, double scale,
                         const int64_t *rows, int64_t count, double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < count; ++i) {
        int64_t tq = rows[i] / num_q_heads;
        int hq = (int)(rows[i] % num_q_heads);
        int r = 0;
        while (r < batch - 1 && q_offsets[r + 1] <= tq)
            ++r;
        int q_len = q_offsets[r + 1] - q_offsets[r];
        int qi = (int)(tq - q_offsets[r]);
        int visible = seq_lens[r] - q_len + qi + 1;
        if (visible < 0)
            visible = 0;
        if (visible > seq_lens[r])
            visible = seq_lens[r];
        int32_t len1 = visible;
        orc_decode_row(q + tq * num_q_heads * head_dim, k_cache, v_cache, k_scale, v_scale,
                       block_table + (int64_t)r * max_blocks_per_seq, max_blocks_per_seq, &len1,
                       num_q_heads, num_kv_heads, head_dim, block_size, cache_kind, scale, 0, hq,
                       out + i * head_dim, NULL, NULL);
    }
}

/* All rows of a batch: out [N][Hq][D] doubles.  Rows are independent, so they
 * are spread over threads; each row is computed exactly as above. */
void orc_paged_decode_attn(const uint16_t *q, const void *k_cache, const void *v_cache,
                           const float *k_scale, const float *v_scale,
                           const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *seq_lens, int batch, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size,
                           int cache_kind, double scale, double *out)
{
    int64_t rows = (int64_t)batch * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < rows; ++i) {
        int r = (int)(i / num_q_heads);
        int hq = (int)(i % num_q_heads);
        orc_decode_row(q, k_cache, v_cache, k_scale, v_scale, block_table,
                       max_blocks_per_seq, seq_lens, num_q_heads, num_kv_heads,
                       head_dim, block_size, cache_kind, scale, r, hq,
                       out + i * head_dim, NULL, NULL);
    }
}

/* Selected rows only: rows[i] = r * Hq + hq, out [count][D]. */
void orc_decode_rows(const uint16_t *q, const void *k_cache, const void *v_cache,
                     const float *k_scale, const float *v_scale,
                     const int32_t *block_table, int max_blocks_per_seq,
                     const int32_t *seq_lens, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int cache_kind, double scale,
                     const int64_t *rows, int64_t count, double *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < count; ++i) {
        int r = (int)(rows[i] / num_q_heads);
        int hq = (int)(rows[i] % num_q_heads);
        orc_decode_row(q, k_cache, v_cache, k_scale, v_scale, block_table,
                       max_blocks_per_seq, seq_lens, num_q_heads, num_kv_heads,
                       head_dim, block_size, cache_kind, scale, r, hq,
                       out + i * head_dim, NULL, NULL);
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads used by the parallel loops from now on (n >= 1); for timing the oracle
 * on one core as well as on all of them.  Changes no result: every output row is
 * computed by one thread in the same order whatever the count. */
void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Prefix block hash  ([P3] "优化一：Prefix Cache", 工作原理：按块哈希:        */
/* hash_i = H(hash_{i-1}, t_{(i-1)B+1}, ..., t_{iB}); token-exact matching)   */
/* ------------------------------------------------------------------------ */

/* FNV-1a, 64-bit (Fowler/Noll/Vo): start from the 64-bit offset basis; for
 * each byte, xor it in, then multiply by the 64-bit FNV prime, mod 2^64. */
uint64_t orc_fnv1a64(const uint8_t *bytes, int64_t n)
{
    uint64_t h = 14695981039346656037ULL;   /* FNV-64 offset basis */
    for (int64_t i = 0; i < n; ++i) {
        h ^= (uint64_t)bytes[i];
        h *= 1099511628211ULL;              /* FNV-64 prime 2^40 + 2^8 + 0xb3 */
    }
    return h;
}

/* The SplitMix64 output function (Steele, Lea, Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; the variant with the
 * 30/27/31 shifts): a bijective 64-bit mixer. */
uint64_t orc_fmix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

/* H(prev, block) = fmix64(prev XOR FNV-1a-64(bytes of the block's tokens)),
 * the tokens taken as little-endian 32-bit words.  h_0 = seed.  Only full
 * blocks get a hash (a partial tail block cannot be shared): sequence s
 * of length L_s yields floor(L_s / B) hashes, written at
 * hashes[hash_offsets[s] + i - 1] for i = 1 .. floor(L_s / B). */
void orc_prefix_block_hash(const int32_t *tokens, const int64_t *offsets,
                           int num_seqs, int block_size, uint64_t seed,
                           uint64_t *hashes, const int64_t *hash_offsets)
{
    uint8_t *buf = (uint8_t *)malloc((size_t)block_size * 4);
    for (int s = 0; s < num_seqs; ++s) {
        int64_t begin = offsets[s];
        int64_t len = offsets[s + 1] - begin;
        int64_t nblocks = len / block_size;
        uint64_t h = seed;
        for (int64_t i = 1; i <= nblocks; ++i) {
            for (int j = 0; j < block_size; ++j) {
                uint32_t tok = (uint32_t)tokens[begin + (i - 1) * block_size + j];
                buf[4 * j + 0] = (uint8_t)(tok & 0xFF);
                buf[4 * j + 1] = (uint8_t)((tok >> 8) & 0xFF);
                buf[4 * j + 2] = (uint8_t)((tok >> 16) & 0xFF);
                buf[4 * j + 3] = (uint8_t)((tok >> 24) & 0xFF);
            }
            h = orc_fmix64(h ^ orc_fnv1a64(buf, (int64_t)block_size * 4));
            hashes[hash_offsets[s] + i - 1] = h;
        }
    }
    free(buf);
}

/* Resuming the chain of [P3] "优化一：Prefix Cache" (工作原理：按块哈希): h_i depends
 * only on h_{i-1} and the tokens of block i, so a sequence whose first k full
 * blocks were hashed earlier continues from h_k and needs only the blocks after
 * them.  Sequence s is tokens[offsets[s] .. offsets[s+1]) (all of its tokens);
 * first_blocks[s] = k_s full blocks are already hashed and prev_hashes[s] = h_{k_s}
 * (the seed when k_s = 0; a negative k_s is read as 0).  The hashes h_{k_s+1},
 * h_{k_s+2}, ... of its later full blocks go to hashes[hash_offsets[s] ..], at most
 * hash_offsets[s+1] - hash_offsets[s] of them; nothing is written when k_s is at or
 * past floor(L_s / B).  The chain is re-derived here block by block from the
 * definition above, independently of orc_prefix_block_hash. */
void orc_prefix_block_hash_resume(const int32_t *tokens, const int64_t *offsets,
                                  int num_seqs, int block_size,
                                  const uint64_t *prev_hashes, const int64_t *first_blocks,
                                  uint64_t *hashes, const int64_t *hash_offsets)
{
    uint8_t *buf = (uint8_t *)malloc((size_t)block_size * 4);
    for (int s = 0; s < num_seqs; ++s) {
        int64_t len = offsets[s + 1] - offsets[s];
        int64_t full = len / block_size;            /* full blocks of the sequence */
        int64_t k = first_blocks[s] < 0 ? 0 : first_blocks[s];
        int64_t room = hash_offsets[s + 1] - hash_offsets[s];
        uint64_t h = prev_hashes[s];                /* h_k */
        int64_t written = 0;
        /* block i (1-based) holds tokens (i-1)B .. iB-1 of the sequence */
        for (int64_t i = k + 1; i <= full && written < room; ++i) {
            const int32_t *blk = tokens + offsets[s] + (i - 1) * block_size;
            for (int j = 0; j < block_size; ++j) {
                uint32_t tok = (uint32_t)blk[j];
                for (int b = 0; b < 4; ++b)
                    buf[4 * j + b] = (uint8_t)(tok >> (8 * b));
            }
            h = orc_fmix64(h ^ orc_fnv1a64(buf, (int64_t)block_size * 4));
            hashes[hash_offsets[s] + written] = h;
            ++written;
        }
    }
    free(buf);
}
