/*
 * fp64 CPU oracle for masked scaled dot-product self-attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and
 * bench.py's cpu_baseline / reference arm may load this library.  It shares
 * no code, header, table or helper with the CUDA path in
 * transformer_self_attention_gb300/, and the product never calls it.
 *
 * What it computes (the plain definition, no tiling, no online softmax):
 *
 *   For a query head a with key/value head g(a), position i:
 *     s_ij   = (q_i^(a) . k_j^(g(a))) * scale            for allowed (i, j)
 *     alpha  = softmax_j(s_ij)                             over allowed j only
 *     z_i    = sum_j alpha_ij v_j^(g(a))
 *     LSE_i  = ln sum_j exp(s_ij)                          (natural log)
 *
 *   - "Trasformer 浅析" (atffang.github.io), section 缩放点积注意力: the
 *     score e_ij = q_i.k_j / sqrt(d_k), row-wise Softmax, output = weights x V.
 *   - same page, section 填充掩码与因果掩码: the additive mask M with -inf;
 *     a -inf entry gets exactly zero weight, so skipping the pair is the same
 *     thing as adding -inf to it, which is what this file does.
 *   - "Transformer 架构及其变体" (aaai.latere.ai), section 带显式形状的因果自注意力:
 *     the shape-explicit form with H_q query heads, H_kv key/value heads and a
 *     query-head -> kv-head map g(a).  The page leaves g open; this oracle takes
 *     the contiguous-group reading g(a) = a / (H_q / H_kv), which is the uniform
 *     grouping described in "Transformer 演进与变体" (ai.icyfenix.cn), section
 *     GQA：分组查询注意力 (g = 1 is MQA, g = h is MHA).
 *   - Mask kinds, "Transformer 演进与变体", section 稀疏注意力: a sliding window
 *     of half-width w (position i sees |i - j| <= w, width 2w+1) and local +
 *     global attention where global tokens see every position and are seen by
 *     every position.  The causal window (0 <= i - j <= w) is the causal mask
 *     of the 填充掩码与因果掩码 section intersected with that window.
 *
 * Arithmetic is fp64 throughout; inputs arrive as float32 arrays (which hold
 * bf16 and fp32 values exactly) and are widened element by element.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* mask kinds: same numbering as the library's public header, restated here */
enum {
    ORACLE_MASK_FULL = 0,
    ORACLE_MASK_CAUSAL = 1,
    ORACLE_MASK_SLIDING = 2,        /* |i - j| <= w                       */
    ORACLE_MASK_CAUSAL_SLIDING = 3, /* 0 <= i - j <= w                    */
    ORACLE_MASK_LOCAL_GLOBAL = 4    /* |i - j| <= w  or  i in G or j in G */
};

/* Allowed(i, j) for one mask kind.  is_global is a 0/1 array of length S
 * (may be NULL when the kind is not LOCAL_GLOBAL).  Returns 1 or 0; returns
 * 0 for a kind this file does not know. */
int oracle_allowed(int kind, long i, long j, long S, long w,
                   const unsigned char* is_global)
{
    if (i < 0 || j < 0 || i >= S || j >= S) return 0;
    long diff = i - j;
    switch (kind) {
    case ORACLE_MASK_FULL: return 1;
    case ORACLE_MASK_CAUSAL: return j <= i;
    case ORACLE_MASK_SLIDING: return labs(diff) <= w;
    case ORACLE_MASK_CAUSAL_SLIDING: return diff >= 0 && diff <= w;
    case ORACLE_MASK_LOCAL_GLOBAL:
        if (labs(diff) <= w) return 1;
        return (is_global[i] != 0) || (is_global[j] != 0);
    default: return 0;
    }
}

static unsigned char* make_global_flags(long S, const int* G, int nG)
{
    unsigned char* f = (unsigned char*)calloc((size_t)(S > 0 ? S : 1), 1);
    if (!f) return NULL;
    for (int t = 0; t < nG; ++t)
        if (G[t] >= 0 && G[t] < S) f[G[t]] = 1;
    return f;
}

/*
 * Attention for an explicit list of query rows.
 *
 * K, V      : float32 [B, Hkv, S, d], contiguous.
 * Qrows     : float32 [n, d], the query vectors of the requested rows.
 * row_b/a/i : batch index, query-head index and position of each row.
 * O         : fp64 [n, d] output (z_i of the shape-explicit form).
 * LSE       : fp64 [n] output, ln sum_j exp(s_ij); -inf for a row with no
 *             allowed key (cannot happen for the five kinds, every row sees
 *             itself), in which case O is set to 0.
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int oracle_attention_rows_bias(const float* K, const float* V,
                               int B, int Hq, int Hkv, int S, int d,
                               double scale, int kind, int window,
                               const int* G, int nG, const double* alibi,
                               const float* Qrows, const int* row_b, const int* row_a,
                               const int* row_i, long n,
                               double* O, double* LSE);
int oracle_attention_rows_general(const float* K, const float* V,
                                  int B, int Hq, int Hkv, int S, int d,
                                  double scale, int kind, int window,
                                  const int* G, int nG, const double* alibi,
                                  const float* bias, int Bb, int Hb, long ld,
                                  const float* Qrows, const int* row_b, const int* row_a,
                                  const int* row_i, long n,
                                  double* O, double* LSE);

int oracle_attention_rows(const float* K, const float* V,
                          int B, int Hq, int Hkv, int S, int d,
                          double scale, int kind, int window,
                          const int* G, int nG,
                          const float* Qrows, const int* row_b, const int* row_a,
                          const int* row_i, long n,
                          double* O, double* LSE)
{
    return oracle_attention_rows_bias(K, V, B, Hq, Hkv, S, d, scale, kind, window, G, nG, NULL,
                                      Qrows, row_b, row_a, row_i, n, O, LSE);
}

int oracle_attention_rows_bias(const float* K, const float* V,
                               int B, int Hq, int Hkv, int S, int d,
                               double scale, int kind, int window,
                               const int* G, int nG, const double* alibi,
                               const float* Qrows, const int* row_b, const int* row_a,
                               const int* row_i, long n,
                               double* O, double* LSE)
{
    return oracle_attention_rows_general(K, V, B, Hq, Hkv, S, d, scale, kind, window, G, nG, alibi,
                                         NULL, 1, 1, 0, Qrows, row_b, row_a, row_i, n, O, LSE);
}

/*
 * The same with additive score biases b_ij (alibi == NULL and bias == NULL: none):
 *   logits_ij = scale * q_i . k_j + b_ij,   b_ij = -alibi[a] * |i - j| + bias[b', a', i, j]
 * - the additive-bias form: "Transformer 架构及其变体" (aaai.latere.ai), the
 *   unified view of sequence and graph attention, logits = q.k / sqrt(d_k) + b_ij;
 * - ALiBi's distance penalty, -m |i - j| with one fixed slope per head: "Trasformer
 *   浅析" (atffang.github.io), section 线性偏置注意力; written -m_h (i - j) for
 *   j <= i under the causal mask in "Transformer 架构及其变体", section 加性偏置：ALiBi,
 *   which is the same value there.
 * alibi: fp64 [Hq], one slope per query head (the pages give no values; callers
 * pass them).
 * bias: a given bias matrix, the general b_ij of the same unified form: fp32
 * [Bb, Hb, S, ld] with Bb in {1, B} and Hb in {1, Hq} (size 1 = the same for every
 * batch / query head), ld >= S the row stride; b' = (Bb == 1 ? 0 : b), a' likewise.
 */
int oracle_attention_rows_general(const float* K, const float* V,
                                  int B, int Hq, int Hkv, int S, int d,
                                  double scale, int kind, int window,
                                  const int* G, int nG, const double* alibi,
                                  const float* bias, int Bb, int Hb, long ld,
                                  const float* Qrows, const int* row_b, const int* row_a,
                                  const int* row_i, long n,
                                  double* O, double* LSE)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || S < 0 || d < 1 || Hq % Hkv != 0) return -1;
    if (bias && ((Bb != 1 && Bb != B) || (Hb != 1 && Hb != Hq) || ld < S)) return -1;
    unsigned char* is_global = make_global_flags(S, G, nG);
    if (!is_global) return -1;
    const int group = Hq / Hkv; /* query heads per kv head */
    int failed = 0;

#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s || !acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < n; ++r) {
            if (!s || !acc) continue;
            const int b = row_b[r], a = row_a[r];
            const long i = row_i[r];
            const int ga = a / group; /* g(a) */
            const float* q = Qrows + (size_t)r * d;
            const float* Kh = K + ((size_t)b * Hkv + ga) * (size_t)S * d;
            const float* Vh = V + ((size_t)b * Hkv + ga) * (size_t)S * d;

            /* scores s_ij over allowed j, and their maximum */
            double m = -INFINITY;
            for (long j = 0; j < S; ++j) {
                if (!oracle_allowed(kind, i, j, S, window, is_global)) continue;
                const float* k = Kh + (size_t)j * d;
                double dot = 0.0;
                for (int t = 0; t < d; ++t) dot += (double)q[t] * (double)k[t];
                s[j] = dot * scale;
                if (alibi) s[j] -= alibi[a] * (double)labs(i - j);
                if (bias) {
                    const size_t plane = (size_t)(Bb == 1 ? 0 : b) * Hb + (Hb == 1 ? 0 : a);
                    s[j] += (double)bias[(plane * (size_t)S + (size_t)i) * (size_t)ld + (size_t)j];
                }
                if (s[j] > m) m = s[j];
            }
            for (int t = 0; t < d; ++t) acc[t] = 0.0;
            double l = 0.0;
            if (m != -INFINITY) {
                /* softmax numerators exp(s_ij - m), their sum, and the
                   weighted sum of value rows */
                for (long j = 0; j < S; ++j) {
                    if (!oracle_allowed(kind, i, j, S, window, is_global)) continue;
                    const double e = exp(s[j] - m);
                    l += e;
                    const float* v = Vh + (size_t)j * d;
                    for (int t = 0; t < d; ++t) acc[t] += e * (double)v[t];
                }
            }
            double* o = O + (size_t)r * d;
            if (l > 0.0) {
                for (int t = 0; t < d; ++t) o[t] = acc[t] / l;
                LSE[r] = m + log(l);
            } else {
                for (int t = 0; t < d; ++t) o[t] = 0.0;
                LSE[r] = -INFINITY;
            }
        }
        free(s);
        free(acc);
    }
    free(is_global);
    return failed ? -1 : 0;
}

/* Number of allowed keys of every row i in [0, S): counts[i]. */
int oracle_row_counts(int kind, int S, int window, const int* G, int nG, long* counts)
{
    unsigned char* is_global = make_global_flags(S, G, nG);
    if (!is_global) return -1;
#pragma omp parallel for schedule(static)
    for (long i = 0; i < S; ++i) {
        long c = 0;
        for (long j = 0; j < S; ++j) c += oracle_allowed(kind, i, j, S, window, is_global);
        counts[i] = c;
    }
    free(is_global);
    return 0;
}

/*
 * Brute-force tile classes: for every (row tile, column tile) of size
 * tm x tn over the S x S pair grid, enumerate each (i, j) inside the tile
 * (pairs beyond S count as not allowed) and write
 *   0 = SKIP    (no allowed pair),
 *   1 = FULL    (every pair of the tm x tn tile lies inside S x S and is allowed),
 *   2 = PARTIAL (anything else).
 * classes is uint8 [ceil(S/tm), ceil(S/tn)], row-major.
 */
int oracle_tile_classes(int kind, int S, int window, const int* G, int nG,
                        int tm, int tn, unsigned char* classes)
{
    if (tm < 1 || tn < 1) return -1;
    unsigned char* is_global = make_global_flags(S, G, nG);
    if (!is_global) return -1;
    const long nt_m = (S + tm - 1) / tm, nt_n = (S + tn - 1) / tn;
#pragma omp parallel for schedule(dynamic, 1)
    for (long ti = 0; ti < nt_m; ++ti) {
        for (long tj = 0; tj < nt_n; ++tj) {
            long allowed = 0;
            for (long i = ti * tm; i < (ti + 1) * tm; ++i)
                for (long j = tj * tn; j < (tj + 1) * tn; ++j)
                    allowed += oracle_allowed(kind, i, j, S, window, is_global);
            unsigned char c;
            if (allowed == 0) c = 0;
            else if (allowed == (long)tm * tn) c = 1;
            else c = 2;
            classes[ti * nt_n + tj] = c;
        }
    }
    free(is_global);
    return 0;
}

/*
 * Decode / key-value-cache attention: S_q new query positions per sequence
 * against a cache that holds cache_len[b] positions of sequence b.
 *
 *   - "Trasformer 浅析" (atffang.github.io), section 推理：KV 缓存: the output at
 *     step t is Softmax(q_t K_{1:t}^T / sqrt(d_k)) V_{1:t}, the query of the new
 *     position against every cached key and value up to and including it.
 *   - "第 8 章 现代大模型架构" (theaiera.top), section 预填充创建缓存，解码复用缓存:
 *     prefill may run in chunks, decode handles one new position per sequence,
 *     and batches are ragged (sequence r holds S_r cached positions).  A chunk
 *     of S_q new positions is read here as the last S_q positions of the cache:
 *     row i of sequence b sits at position t = cache_len[b] - S_q + i, and its
 *     own key and value are already in the cache.
 *   - "Trasformer 浅析", section 交叉注意力: the same formula with queries from
 *     the decoder and keys/values from the encoder; the score matrix is
 *     n_dec x n_enc and every encoder position is visible (kind FULL).
 *
 * Kinds: FULL (all j < cache_len[b]), CAUSAL (j <= t), CAUSAL_SLIDING
 * (t - w <= j <= t).  Other kinds return -1.
 *
 * Q   : float32 [B, Hq, S_q, d]      K, V : float32 [B, Hkv, S_cap, d]
 * O   : fp64 [B, Hq, S_q, d]         LSE  : fp64 [B, Hq, S_q]
 * Cache entries at positions >= cache_len[b] are never read.
 * Returns 0, or -1 on bad arguments (a cache length outside [1, S_cap], or
 * below S_q for the causal kinds) or allocation failure.
 */
int oracle_decode_allowed(int kind, long t, long j, long L, long w)
{
    if (j < 0 || j >= L) return 0;
    switch (kind) {
    case ORACLE_MASK_FULL: return 1;
    case ORACLE_MASK_CAUSAL: return j <= t;
    case ORACLE_MASK_CAUSAL_SLIDING: return j <= t && t - j <= w;
    default: return 0;
    }
}

int oracle_decode_bias(const float* Q, const float* K, const float* V,
                       int B, int Hq, int Hkv, int S_q, int S_cap, int d,
                       double scale, int kind, int window, const int* cache_len,
                       const double* alibi, double* O, double* LSE);

int oracle_decode(const float* Q, const float* K, const float* V,
                  int B, int Hq, int Hkv, int S_q, int S_cap, int d,
                  double scale, int kind, int window, const int* cache_len,
                  double* O, double* LSE)
{
    return oracle_decode_bias(Q, K, V, B, Hq, Hkv, S_q, S_cap, d, scale, kind, window, cache_len, NULL, O, LSE);
}

/* Decode with the ALiBi bias -alibi[a] * |t - j| (t the row's position; NULL: none). */
int oracle_decode_bias(const float* Q, const float* K, const float* V,
                       int B, int Hq, int Hkv, int S_q, int S_cap, int d,
                       double scale, int kind, int window, const int* cache_len,
                       const double* alibi, double* O, double* LSE)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || S_q < 1 || S_cap < 1 || d < 1 || Hq % Hkv != 0) return -1;
    if (kind != ORACLE_MASK_FULL && kind != ORACLE_MASK_CAUSAL && kind != ORACLE_MASK_CAUSAL_SLIDING)
        return -1;
    if (kind == ORACLE_MASK_CAUSAL_SLIDING && window < 0) return -1;
    for (int b = 0; b < B; ++b) {
        if (cache_len[b] < 1 || cache_len[b] > S_cap) return -1;
        if (kind != ORACLE_MASK_FULL && cache_len[b] < S_q) return -1;
    }
    const int group = Hq / Hkv;
    const long n = (long)B * Hq * S_q;
    int failed = 0;

#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)S_cap);
        double* acc = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s || !acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < n; ++r) {
            if (!s || !acc) continue;
            const int b = (int)(r / ((long)Hq * S_q));
            const int a = (int)((r / S_q) % Hq);
            const long i = r % S_q;
            const long L = cache_len[b];
            const long t = L - S_q + i; /* position of this query row */
            const int ga = a / group;   /* g(a) */
            const float* q = Q + (size_t)r * d;
            const float* Kh = K + ((size_t)b * Hkv + ga) * (size_t)S_cap * d;
            const float* Vh = V + ((size_t)b * Hkv + ga) * (size_t)S_cap * d;

            double m = -INFINITY;
            for (long j = 0; j < L; ++j) {
                if (!oracle_decode_allowed(kind, t, j, L, window)) continue;
                const float* k = Kh + (size_t)j * d;
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += (double)q[c] * (double)k[c];
                s[j] = dot * scale;
                if (alibi) s[j] -= alibi[a] * (double)labs(t - j);
                if (s[j] > m) m = s[j];
            }
            for (int c = 0; c < d; ++c) acc[c] = 0.0;
            double l = 0.0;
            if (m != -INFINITY) {
                for (long j = 0; j < L; ++j) {
                    if (!oracle_decode_allowed(kind, t, j, L, window)) continue;
                    const double e = exp(s[j] - m);
                    l += e;
                    const float* v = Vh + (size_t)j * d;
                    for (int c = 0; c < d; ++c) acc[c] += e * (double)v[c];
                }
            }
            double* o = O + (size_t)r * d;
            if (l > 0.0) {
                for (int c = 0; c < d; ++c) o[c] = acc[c] / l;
                LSE[r] = m + log(l);
            } else {
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                LSE[r] = -INFINITY;
            }
        }
        free(s);
        free(acc);
    }
    return failed ? -1 : 0;
}

/*
 * Backward pass: the gradients of the forward attention above with respect to
 * Q, K and V, given the output gradient dO.  The pages give no formulas for it;
 * they say only that the tiled method is exact and serves training ("Transformer
 * 演进与变体", section Flash Attention), so this is the plain derivative of the
 * definition, row by row (same mask, same g(a), optional ALiBi slopes):
 *
 *   P_ij  = exp(s_ij - LSE_i)            over allowed j  (s_ij as in the forward)
 *   dV_j += P_ij dO_i                    summed over the query heads of kv head g
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij  (= dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j += scale sum_i dS_ij q_i        summed over the query heads of kv head g
 *
 * Q, dO : float32 [B, Hq, S, d]   K, V : float32 [B, Hkv, S, d]
 * dQ    : fp64 [B, Hq, S, d] (out)   dK, dV : fp64 [B, Hkv, S, d] (out, overwritten)
 * Rows are computed in parallel; the dK / dV sums over rows are kept per thread
 * and added at the end, in a fixed order.
 * Returns 0, or -1 on bad arguments or allocation failure.
 */
/*
 * The same gradients with a given additive bias matrix as well (bias == NULL: none): the
 * logits are scale * q_i . k_j - alibi[a] |i - j| + bias[b', a', i, j] (b' = b if Bb == B
 * else 0, a' = a if Hb == Hq else 0, row stride ld), the unified biased-logits form of
 * "Transformer 架构及其变体" (aaai.latere.ai).  The bias does not depend on Q, K or V, so it
 * enters only the weights P; dS, dQ, dK and dV keep their formulas.
 */
int oracle_backward_bias(const float* Q, const float* K, const float* V, const float* dO,
                         int B, int Hq, int Hkv, int S, int d, double scale, int kind, int window,
                         const int* G, int nG, const double* alibi,
                         const float* bias, int Bb, int Hb, long ld,
                         double* dQ, double* dK, double* dV);

int oracle_backward(const float* Q, const float* K, const float* V, const float* dO,
                    int B, int Hq, int Hkv, int S, int d, double scale, int kind, int window,
                    const int* G, int nG, const double* alibi,
                    double* dQ, double* dK, double* dV)
{
    return oracle_backward_bias(Q, K, V, dO, B, Hq, Hkv, S, d, scale, kind, window, G, nG, alibi,
                                NULL, 1, 1, 0, dQ, dK, dV);
}

int oracle_backward_bias(const float* Q, const float* K, const float* V, const float* dO,
                         int B, int Hq, int Hkv, int S, int d, double scale, int kind, int window,
                         const int* G, int nG, const double* alibi,
                         const float* bias, int Bb, int Hb, long ld,
                         double* dQ, double* dK, double* dV)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || d < 1 || Hq % Hkv != 0) return -1;
    if (bias && ((Bb != 1 && Bb != B) || (Hb != 1 && Hb != Hq) || ld < S)) return -1;
    unsigned char* is_global = make_global_flags(S, G, nG);
    if (!is_global) return -1;
    const int group = Hq / Hkv;
    const size_t kv_elems = (size_t)B * Hkv * S * d;
    int nthreads = 1;
#ifdef _OPENMP
    nthreads = omp_get_max_threads();
#endif
    double* part = (double*)calloc((size_t)nthreads * 2 * kv_elems, sizeof(double));
    if (!part) { free(is_global); return -1; }
    int failed = 0;
    const long n = (long)B * Hq * S;

#pragma omp parallel
    {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double* pdK = part + (size_t)tid * 2 * kv_elems;
        double* pdV = pdK + kv_elems;
        double* s = (double*)malloc(sizeof(double) * (size_t)S);
        double* o = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s || !o) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < n; ++r) {
            if (!s || !o) continue;
            const int b = (int)(r / ((long)Hq * S));
            const int a = (int)((r / S) % Hq);
            const long i = r % S;
            const int ga = a / group;
            const size_t kvh = ((size_t)b * Hkv + ga) * (size_t)S * d;
            const float* q = Q + (size_t)r * d;
            const float* go = dO + (size_t)r * d;
            /* forward quantities of the row: scores, max, sum, O */
            double m = -INFINITY;
            for (long j = 0; j < S; ++j) {
                if (!oracle_allowed(kind, i, j, S, window, is_global)) continue;
                double dot = 0.0;
                for (int c = 0; c < d; ++c) dot += (double)q[c] * (double)K[kvh + (size_t)j * d + c];
                s[j] = dot * scale;
                if (alibi) s[j] -= alibi[a] * (double)labs(i - j);
                if (bias) {
                    const size_t plane = (size_t)(Bb == 1 ? 0 : b) * Hb + (size_t)(Hb == 1 ? 0 : a);
                    s[j] += (double)bias[(plane * (size_t)S + (size_t)i) * (size_t)ld + (size_t)j];
                }
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            for (long j = 0; j < S; ++j) {
                if (!oracle_allowed(kind, i, j, S, window, is_global)) continue;
                const double e = exp(s[j] - m);
                l += e;
                for (int c = 0; c < d; ++c) o[c] += e * (double)V[kvh + (size_t)j * d + c];
            }
            double Di = 0.0;
            for (int c = 0; c < d; ++c) { o[c] /= l; Di += (double)go[c] * o[c]; }
            double* gq = dQ + (size_t)r * d;
            for (int c = 0; c < d; ++c) gq[c] = 0.0;
            for (long j = 0; j < S; ++j) {
                if (!oracle_allowed(kind, i, j, S, window, is_global)) continue;
                const double P = exp(s[j] - m) / l;
                double dP = 0.0;
                for (int c = 0; c < d; ++c) dP += (double)go[c] * (double)V[kvh + (size_t)j * d + c];
                const double dS = P * (dP - Di);
                for (int c = 0; c < d; ++c) {
                    gq[c] += scale * dS * (double)K[kvh + (size_t)j * d + c];
                    pdK[kvh + (size_t)j * d + c] += scale * dS * (double)q[c];
                    pdV[kvh + (size_t)j * d + c] += P * (double)go[c];
                }
            }
        }
        free(s);
        free(o);
    }
    if (!failed) {
        for (size_t e = 0; e < kv_elems; ++e) { dK[e] = 0.0; dV[e] = 0.0; }
        for (int t = 0; t < nthreads; ++t) {
            const double* pdK = part + (size_t)t * 2 * kv_elems;
            const double* pdV = pdK + kv_elems;
            for (size_t e = 0; e < kv_elems; ++e) { dK[e] += pdK[e]; dV[e] += pdV[e]; }
        }
    }
    free(part);
    free(is_global);
    return failed ? -1 : 0;
}
