/*
 * CPU oracle for paged decode attention over a block-paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: it exists so that tests, the smoke check and the
 * benchmark's CPU baseline can compare the CUDA kernels with a plain,
 * slow, obviously correct restatement of what the method computes.  It
 * shares no code, header or table with the CUDA sources.
 *
 * Sources (the pages this follows):
 *  - MinivLLM guide "HowToApproachvLLM", §4.5 (prepare_prefill/decode):
 *    the KV cache is carved into blocks along a token axis, a block's
 *    tokens are kv_cache[..., block_id*block_size:(block_id+1)*block_size, ...],
 *    a new token's K/V go to the flat slot given by slot_mapping, and the
 *    attention kernel reads KV through block_tables.
 *  - "Nano-vLLM 源码学习(2)", §2 Config: attention heads and KV heads are
 *    distinct counts (grouped-query attention).
 *  - "VLLM-0.7.3 源码", §3.1: a block table maps a sequence's logical
 *    blocks to physical blocks scattered through memory.
 *  The pages do not write out the attention formula; this oracle takes the
 *  plain reading: for each sequence b and query head h, the output is
 *  softmax(scale * q . K^T) . V over the first context_lens[b] cached
 *  tokens of KV head h / (Hq/Hkv).
 *
 * Layouts (row-major):
 *   k_cache, v_cache : bf16 [NB, bs, Hkv, D]   (flat slot = block*bs + offset)
 *   q                : bf16 [B, Hq, D]
 *   block_tables     : int32 [B, MBS]
 *   context_lens     : int32 [B]
 *   k, v (new)       : bf16 [N, Hkv, D]
 *   slot_mapping     : int64 [N], -1 = padding (skipped)
 * bf16 values are passed as their uint16 bit patterns.
 *
 * Arithmetic is fp64 throughout; bf16 -> fp64 widening is exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * store_kvcache: for every i with slot_mapping[i] >= 0, copy the bf16 bits
 * of k[i] and v[i] (all Hkv*D elements) to flat slot slot_mapping[i], i.e.
 * block slot/bs, offset slot%bs (MinivLLM guide §4.5: slot_mapping says where
 * each new token's KV is written; padding slots are skipped).
 * Returns the number of slots that were out of range [0, NB*bs) and skipped.
 */
int64_t oracle_store_kvcache(const uint16_t *k, const uint16_t *v,
                             uint16_t *k_cache, uint16_t *v_cache,
                             const int64_t *slot_mapping, int64_t N,
                             int Hkv, int D, int64_t NB, int bs)
{
    int64_t bad = 0;
    int64_t row = (int64_t)Hkv * D;
    for (int64_t i = 0; i < N; i++) {
        int64_t slot = slot_mapping[i];
        if (slot == -1)
            continue;
        if (slot < 0 || slot >= NB * (int64_t)bs) {
            bad++;
            continue;
        }
        int64_t block = slot / bs;
        int64_t offset = slot % bs;
        for (int h = 0; h < Hkv; h++) {
            for (int d = 0; d < D; d++) {
                int64_t dst = ((block * bs + offset) * Hkv + h) * D + d;
                int64_t src = i * row + (int64_t)h * D + d;
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
        }
    }
    return bad;
}

/*
 * One (sequence b, query head h) of decode attention, written out from the
 * definition: gather the first n cached tokens of KV head kvh through the
 * block table, score s_t = scale * sum_d q_d K_td, take w_t = exp(s_t - max s),
 * and return sum_t w_t V_t / sum_t w_t.  n == 0 gives zeros.
 * Returns 0, or -1 when a block-table entry needed is outside [0, NB).
 */
static int decode_one(const uint16_t *q, const uint16_t *k_cache,
                      const uint16_t *v_cache, const int32_t *table, int n,
                      int Hkv, int kvh, int D, int64_t NB, int bs,
                      double scale, double *out, double *s)
{
    for (int d = 0; d < D; d++)
        out[d] = 0.0;
    if (n <= 0)
        return 0;
    /* scores */
    for (int t = 0; t < n; t++) {
        int64_t phys = table[t / bs];
        if (phys < 0 || phys >= NB)
            return -1;
        int64_t base = ((phys * bs + t % bs) * Hkv + kvh) * (int64_t)D;
        double dot = 0.0;
        for (int d = 0; d < D; d++)
            dot += bf16_to_f64(q[d]) * bf16_to_f64(k_cache[base + d]);
        s[t] = scale * dot;
    }
    /* softmax weights */
    double m = s[0];
    for (int t = 1; t < n; t++)
        if (s[t] > m)
            m = s[t];
    double l = 0.0;
    for (int t = 0; t < n; t++) {
        s[t] = exp(s[t] - m);
        l += s[t];
    }
    /* weighted sum of V */
    for (int t = 0; t < n; t++) {
        int64_t phys = table[t / bs];
        int64_t base = ((phys * bs + t % bs) * Hkv + kvh) * (int64_t)D;
        for (int d = 0; d < D; d++)
            out[d] += s[t] * bf16_to_f64(v_cache[base + d]);
    }
    for (int d = 0; d < D; d++)
        out[d] /= l;
    return 0;
}

/*
 * paged_attn_decode over the listed (b, h) pairs (pairs[2*i], pairs[2*i+1]);
 * out is [n_pairs, D] fp64.  Query head h reads KV head h / (Hq / Hkv).
 * Returns the number of pairs that hit an invalid block-table entry (their
 * output rows are left at zero).
 */
int64_t oracle_paged_attn_decode_pairs(const uint16_t *q, const uint16_t *k_cache,
                                       const uint16_t *v_cache,
                                       const int32_t *block_tables, int MBS,
                                       const int32_t *context_lens, int B, int Hq,
                                       int Hkv, int D, int64_t NB, int bs, float scale,
                                       const int32_t *pairs, int64_t n_pairs, double *out)
{
    int G = Hq / Hkv;
    int64_t bad = 0;
    int max_n = MBS * bs;
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_n > 0 ? max_n : 1));
    if (!s)
        return -1;
    for (int64_t i = 0; i < n_pairs; i++) {
        int b = pairs[2 * i];
        int h = pairs[2 * i + 1];
        int n = context_lens[b];
        if (n > max_n)
            n = max_n;
        const uint16_t *qh = q + ((int64_t)b * Hq + h) * D;
        const int32_t *table = block_tables + (int64_t)b * MBS;
        if (decode_one(qh, k_cache, v_cache, table, n, Hkv, h / G, D, NB, bs,
                       (double)scale, out + i * D, s) != 0) {
            for (int d = 0; d < D; d++)
                out[i * D + d] = 0.0;
            bad++;
        }
    }
    free(s);
    (void)B;
    return bad;
}

/* paged_attn_decode over every (b, h); out is [B, Hq, D] fp64. */
int64_t oracle_paged_attn_decode(const uint16_t *q, const uint16_t *k_cache,
                                 const uint16_t *v_cache, const int32_t *block_tables,
                                 int MBS, const int32_t *context_lens, int B, int Hq,
                                 int Hkv, int D, int64_t NB, int bs, float scale,
                                 double *out)
{
    int64_t n_pairs = (int64_t)B * Hq;
    int32_t *pairs = (int32_t *)malloc(sizeof(int32_t) * 2 * (size_t)(n_pairs > 0 ? n_pairs : 1));
    if (!pairs)
        return -1;
    for (int b = 0; b < B; b++)
        for (int h = 0; h < Hq; h++) {
            pairs[2 * ((int64_t)b * Hq + h)] = b;
            pairs[2 * ((int64_t)b * Hq + h) + 1] = h;
        }
    int64_t r = oracle_paged_attn_decode_pairs(q, k_cache, v_cache, block_tables, MBS,
                                               context_lens, B, Hq, Hkv, D, NB, bs, scale,
                                               pairs, n_pairs, out);
    free(pairs);
    return r;
}

/*
 * Dense attention over contiguous K/V [n, Hkv, D] (no paging): the result
 * the paged cache must reproduce, since caching history only replaces
 * recomputing it ("从零实现vLLM系列【9】：Engine", §5: v0 recomputes the full
 * sequence each step; a KV cache keeps past K/V instead).
 * q is [Hq, D]; out is [Hq, D] fp64.
 */
void oracle_dense_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, int n,
                       int Hq, int Hkv, int D, float scale, double *out)
{
    int G = Hq / Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int h = 0; h < Hq; h++) {
        int kvh = h / G;
        double *o = out + (int64_t)h * D;
        for (int d = 0; d < D; d++)
            o[d] = 0.0;
        if (n <= 0)
            continue;
        for (int t = 0; t < n; t++) {
            double dot = 0.0;
            for (int d = 0; d < D; d++)
                dot += bf16_to_f64(q[(int64_t)h * D + d]) *
                       bf16_to_f64(k[((int64_t)t * Hkv + kvh) * D + d]);
            s[t] = (double)scale * dot;
        }
        double m = s[0];
        for (int t = 1; t < n; t++)
            if (s[t] > m)
                m = s[t];
        double l = 0.0;
        for (int t = 0; t < n; t++) {
            s[t] = exp(s[t] - m);
            l += s[t];
        }
        for (int t = 0; t < n; t++)
            for (int d = 0; d < D; d++)
                o[d] += s[t] * bf16_to_f64(v[((int64_t)t * Hkv + kvh) * D + d]);
        for (int d = 0; d < D; d++)
            o[d] /= l;
    }
    free(s);
}

/*
 * FP8 KV cache ("VLLM-0.7.3 源码" section 5.3: the KV cache may be stored in
 * FP8 via kv_cache_dtype while the attention computes in higher precision).
 * The page gives no scale convention; this oracle takes the plain per-tensor
 * one: a cache value is the OCP E4M3 code of x * (1 / scale) (computed in
 * fp32), and its value is code_value * scale.
 *
 * E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent field 0 encodes subnormals m/8 * 2^-6; no infinities; the codes
 * S.1111.111 are NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
 * Quantization rounds to nearest, ties to even, and saturates finite
 * overflow (and infinities) to +-448; NaN maps to 0x7F with its sign.
 */
static double e4m3_value(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

uint8_t oracle_e4m3_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x))
        return sign | 0x7F;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    /* nearest of all finite magnitudes; ties to the even (mantissa LSB 0) code */
    uint8_t best = 0;
    double best_err = a;  /* code 0 has value 0 */
    for (int c = 1; c <= 0x7E; c++) {
        double err = fabs(e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_err = err;
        }
    }
    return sign | best;
}

double oracle_e4m3_decode(uint8_t code) { return e4m3_value(code); }

/*
 * store_kvcache into FP8 caches: every element of k[i] / v[i] (bf16 bits) is
 * widened, multiplied by 1/k_scale (resp. 1/v_scale) in fp32, and encoded as
 * E4M3 at the slot slot_mapping[i].  Returns the number of skipped
 * out-of-range slots.
 */
int64_t oracle_store_kvcache_fp8(const uint16_t *k, const uint16_t *v, uint8_t *k_cache,
                                 uint8_t *v_cache, const int64_t *slot_mapping, int64_t N,
                                 int Hkv, int D, int64_t NB, int bs, float k_scale, float v_scale)
{
    int64_t bad = 0, row = (int64_t)Hkv * D;
    float kinv = 1.0f / k_scale, vinv = 1.0f / v_scale;
    for (int64_t i = 0; i < N; i++) {
        int64_t slot = slot_mapping[i];
        if (slot == -1)
            continue;
        if (slot < 0 || slot >= NB * (int64_t)bs) {
            bad++;
            continue;
        }
        for (int64_t e = 0; e < row; e++) {
            float kx = (float)bf16_to_f64(k[i * row + e]) * kinv;
            float vx = (float)bf16_to_f64(v[i * row + e]) * vinv;
            k_cache[slot * row + e] = oracle_e4m3_encode(kx);
            v_cache[slot * row + e] = oracle_e4m3_encode(vx);
        }
    }
    return bad;
}

/* Dequantize FP8 caches to fp64 (code value * scale). */
void oracle_dequant_fp8(const uint8_t *codes, int64_t n, float scale, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = e4m3_value(codes[i]) * (double)scale;
}

/*
 * Decode attention over caches already holding fp64 values (for example
 * dequantized FP8 codes): the same definition as decode_one, reading K and V
 * as doubles.  out is [n_pairs, D]; returns the number of pairs that hit an
 * invalid block-table entry.
 */
int64_t oracle_paged_attn_decode_pairs_f64kv(const uint16_t *q, const double *k_cache,
                                             const double *v_cache, const int32_t *block_tables,
                                             int MBS, const int32_t *context_lens, int Hq,
                                             int Hkv, int D, int64_t NB, int bs, float scale,
                                             const int32_t *pairs, int64_t n_pairs, double *out)
{
    int G = Hq / Hkv;
    int64_t bad = 0;
    int max_n = MBS * bs;
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_n > 0 ? max_n : 1));
    if (!s)
        return -1;
    for (int64_t i = 0; i < n_pairs; i++) {
        int b = pairs[2 * i], h = pairs[2 * i + 1], kvh = h / G;
        int n = context_lens[b] > max_n ? max_n : context_lens[b];
        const uint16_t *qh = q + ((int64_t)b * Hq + h) * D;
        const int32_t *table = block_tables + (int64_t)b * MBS;
        double *o = out + i * D;
        for (int d = 0; d < D; d++)
            o[d] = 0.0;
        int ok = 1;
        for (int t = 0; t < n && ok; t++) {
            int64_t phys = table[t / bs];
            if (phys < 0 || phys >= NB) {
                ok = 0;
                break;
            }
            int64_t base = ((phys * bs + t % bs) * Hkv + kvh) * (int64_t)D;
            double dot = 0.0;
            for (int d = 0; d < D; d++)
                dot += bf16_to_f64(qh[d]) * k_cache[base + d];
            s[t] = (double)scale * dot;
        }
        if (!ok) {
            bad++;
            continue;
        }
        if (n <= 0)
            continue;
        double m = s[0];
        for (int t = 1; t < n; t++)
            if (s[t] > m)
                m = s[t];
        double l = 0.0;
        for (int t = 0; t < n; t++) {
            s[t] = exp(s[t] - m);
            l += s[t];
        }
        for (int t = 0; t < n; t++) {
            int64_t phys = table[t / bs];
            int64_t base = ((phys * bs + t % bs) * Hkv + kvh) * (int64_t)D;
            for (int d = 0; d < D; d++)
                o[d] += s[t] * v_cache[base + d];
        }
        for (int d = 0; d < D; d++)
            o[d] /= l;
    }
    free(s);
    return bad;
}

/*
 * Paged prefill (MinivLLM guide §4.5, prepare_prefill: the new tokens of all
 * sequences are flattened into one list whose boundaries cu_seqlens_q marks,
 * cu_seqlens_k marks each sequence's keys, slot_mapping writes only the
 * uncached tokens, and block_tables say where KV is read; "Nano-vLLM 源码学习
 * (2)" §2: the prefix-hit prefill path reads paged KV through block_table).
 * The pages give no mask; the plain reading for a causal language model:
 * sequence b has q_len = cu_q[b+1] - cu_q[b] new tokens and a context of
 * k_len = cu_k[b+1] - cu_k[b] tokens (cached prefix + the new tokens, all
 * already stored in the cache, q_len <= k_len); its query i sits at position
 * k_len - q_len + i and attends to the tokens at positions 0 .. that position.
 * Each (query row, head) is thus decode attention over its first position + 1
 * tokens, computed here by the same definition as decode_one.
 *
 * pairs: (token row r in [0, cu_q[B]), query head h); out is [n_pairs, D].
 * Returns the number of pairs left at zero because their lengths are
 * inconsistent or a needed block-table entry is outside [0, NB).
 */
int64_t oracle_paged_prefill_pairs(const uint16_t *q, const uint16_t *k_cache,
                                   const uint16_t *v_cache, const int32_t *block_tables,
                                   int MBS, const int32_t *cu_q, const int32_t *cu_k, int B,
                                   int Hq, int Hkv, int D, int64_t NB, int bs, float scale,
                                   const int32_t *pairs, int64_t n_pairs, double *out)
{
    int G = Hq / Hkv;
    int64_t bad = 0;
    int max_n = MBS * bs;
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_n > 0 ? max_n : 1));
    if (!s)
        return -1;
    for (int64_t i = 0; i < n_pairs; i++) {
        int r = pairs[2 * i], h = pairs[2 * i + 1];
        double *o = out + i * D;
        for (int d = 0; d < D; d++)
            o[d] = 0.0;
        int b = 0;
        while (b < B && cu_q[b + 1] <= r)
            b++;
        if (b == B || r < cu_q[b]) {
            bad++;
            continue;
        }
        int q_len = cu_q[b + 1] - cu_q[b];
        int k_len = cu_k[b + 1] - cu_k[b];
        if (k_len < q_len || k_len > max_n) {
            bad++;
            continue;
        }
        int n = k_len - q_len + (r - cu_q[b]) + 1;
        const uint16_t *qr = q + ((int64_t)r * Hq + h) * D;
        const int32_t *table = block_tables + (int64_t)b * MBS;
        if (decode_one(qr, k_cache, v_cache, table, n, Hkv, h / G, D, NB, bs, (double)scale,
                       o, s) != 0) {
            for (int d = 0; d < D; d++)
                o[d] = 0.0;
            bad++;
        }
    }
    free(s);
    return bad;
}

/*
 * Dense causal attention of one sequence over contiguous K/V, written apart
 * from the paged routines (explicit score row with -inf above the diagonal)
 * so that the paged prefill can be checked against it: the paged cache must
 * give the result of attending over the contiguous context.
 * q [Lq, Hq, D], k/v [Lk, Hkv, D] (Lq <= Lk; query i is at position
 * Lk - Lq + i); out [Lq, Hq, D] fp64.
 */
void oracle_dense_causal_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, int Lq,
                              int Lk, int Hq, int Hkv, int D, float scale, double *out)
{
    int G = Hq / Hkv;
    double *row = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
    for (int i = 0; i < Lq; i++) {
        int last = Lk - Lq + i; /* highest key position this query may see */
        for (int h = 0; h < Hq; h++) {
            int kvh = h / G;
            double *o = out + ((int64_t)i * Hq + h) * D;
            double m = -INFINITY;
            for (int j = 0; j < Lk; j++) {
                if (j > last) {
                    row[j] = -INFINITY;
                    continue;
                }
                double dot = 0.0;
                for (int d = 0; d < D; d++)
                    dot += bf16_to_f64(q[((int64_t)i * Hq + h) * D + d]) *
                           bf16_to_f64(k[((int64_t)j * Hkv + kvh) * D + d]);
                row[j] = (double)scale * dot;
                if (row[j] > m)
                    m = row[j];
            }
            double l = 0.0;
            for (int j = 0; j < Lk; j++) {
                row[j] = exp(row[j] - m); /* exp(-inf) = 0 for masked keys */
                l += row[j];
            }
            for (int d = 0; d < D; d++) {
                double acc = 0.0;
                for (int j = 0; j < Lk; j++)
                    acc += row[j] * bf16_to_f64(v[((int64_t)j * Hkv + kvh) * D + d]);
                o[d] = acc / l;
            }
        }
    }
    free(row);
}
