/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the
 * CUDA library.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load or call it; the product path never does.  It
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Every function computes its result straight from the definition on the
 * source pages, materialising the score matrix (or the score row) in fp64:
 *
 *   [IOAE] auturnal.com, "注意機構からIOを考慮した実行へ" (From attention to
 *          IO-aware execution): §2 scaled dot-product attention
 *          softmax(QK^T/sqrt(d_k))V; §8 max subtraction leaves the
 *          probabilities unchanged; §9 KV-cache size 2*L*n*h_kv*d_h*b.
 *   [TCOS] papanda925.com, "Transformer計算量最適化戦略の最前線": "standard
 *          attention pseudocode" (scores = QK^T/sqrt(d_k), masked entries
 *          set to -inf, softmax over the last axis, then weights @ V, shapes
 *          [batch, heads, L, d]); "KV cache management concept" (new K/V
 *          appended to the cache each generated token); block-wise KV cache
 *          (fixed-size blocks) in "latest trends".
 *   [ACD]  code-journey.com, attention co-design for long-context inference,
 *          "Group Size (G)": G query heads share one KV head (G=1 is MHA).
 *   [FASL] marketmaker.cc, "Flash Attention und die Frage nach der
 *          Sequenzlänge", "Kausale Maskierung": keys in the future of the
 *          query are masked.
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes): query head h uses KV head h / G; a causal mask is aligned
 * bottom-right (query i sees keys j <= i + n_kv - n_q); lse is the natural
 * log of sum_j exp(s_ij) over the scaled scores; an empty decode sequence
 * yields O = 0 and lse = -inf.
 *
 * Element formats are decoded from their definitions (IEEE binary16, the
 * upper half of IEEE binary32 for bfloat16, OCP FP8 E4M3), not through any
 * library.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2, OR_E4M3 = 3, OR_F64 = 4 };

/* ---------------------------------------------------------------- formats */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1.0 + f / 1024.0, e - 15);
    return sign ? -v : v;
}

/* bfloat16 is the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

/* OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent bits (bias 7), 3 fraction bits,
 * no infinities, S.1111.111 is NaN, largest finite magnitude 448. */
double oracle_e4m3_to_f64(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int f = c & 0x7;
    double v;
    if (e == 15 && f == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)f, -9); /* subnormal: f/8 * 2^-6 */
    else
        v = ldexp(1.0 + f / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round an fp32 value to E4M3, nearest-even, saturating to +-448 (the
 * "satfinite" convention: finite overflow clamps to the largest finite
 * magnitude; NaN stays NaN). */
uint8_t oracle_f32_to_e4m3(float xf) {
    double x = (double)xf;
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7e; /* 448 = 1.75 * 2^8 : e=15, f=6 */
    double step;
    if (a < ldexp(1.0, -6)) {
        step = ldexp(1.0, -9); /* subnormal spacing */
    } else {
        int ex;
        frexp(a, &ex); /* a = m * 2^ex, m in [0.5, 1) */
        step = ldexp(1.0, (ex - 1) - 3);
    }
    double q = nearbyint(a / step) * step; /* exact scaling; ties to even */
    if (q > 448.0)
        q = 448.0;
    if (q == 0.0)
        return sign;
    if (q < ldexp(1.0, -6)) {
        int f = (int)(q / ldexp(1.0, -9));
        return sign | (uint8_t)f;
    }
    int ex;
    double m = frexp(q, &ex); /* q = m * 2^ex, m in [0.5,1) -> 2m in [1,2) */
    int e = (ex - 1) + 7;
    int f = (int)((2.0 * m - 1.0) * 8.0);
    return sign | (uint8_t)(e << 3) | (uint8_t)f;
}

/* Element-wise oracle_f32_to_e4m3 over an array. */
void oracle_encode_e4m3_array(const float *x, uint8_t *out, long long n) {
    for (long long i = 0; i < n; ++i)
        out[i] = oracle_f32_to_e4m3(x[i]);
}

static double load_elem(const void *p, int dtype, size_t i) {
    switch (dtype) {
    case OR_F16: return oracle_f16_to_f64(((const uint16_t *)p)[i]);
    case OR_BF16: return oracle_bf16_to_f64(((const uint16_t *)p)[i]);
    case OR_F32: return (double)((const float *)p)[i];
    case OR_E4M3: return oracle_e4m3_to_f64(((const uint8_t *)p)[i]);
    case OR_F64: return ((const double *)p)[i];
    default: return NAN;
    }
}

/* ------------------------------------------------------------- prefill */

/* One (batch, query head): the full n_q x n_kv score matrix is materialised,
 * masked, soft-maxed row by row with max subtraction, then multiplied by V.
 * q/k/v are already decoded to fp64, row-major [n][d].  counts, if given,
 * receives {multiply-adds, exp evaluations}. */
static void sdpa_one_head(const double *q, const double *k, const double *v,
                          double *o, double *lse, int nq, int nkv, int d,
                          int causal, double scale, long long *counts) {
    double *S = (double *)malloc((size_t)nq * (size_t)nkv * sizeof(double));
    long long macs = 0, exps = 0;
    /* 1. scores = Q K^T * scale   ([TCOS] standard attention, step 1) */
    for (int i = 0; i < nq; ++i)
        for (int j = 0; j < nkv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += q[(size_t)i * d + c] * k[(size_t)j * d + c];
            macs += d;
            S[(size_t)i * nkv + j] = acc * scale;
        }
    /* 2. mask: future keys -> -inf   ([TCOS] step 2, [FASL] causal) */
    if (causal)
        for (int i = 0; i < nq; ++i)
            for (int j = 0; j < nkv; ++j)
                if (j > i + (nkv - nq))
                    S[(size_t)i * nkv + j] = -INFINITY;
    /* 3. softmax over keys with the row max subtracted ([IOAE] §8),
     * 4. weights @ V. */
    for (int i = 0; i < nq; ++i) {
        double *row = S + (size_t)i * nkv;
        double m = -INFINITY;
        for (int j = 0; j < nkv; ++j)
            if (row[j] > m)
                m = row[j];
        if (m == -INFINITY) { /* no visible key */
            for (int c = 0; c < d; ++c)
                o[(size_t)i * d + c] = 0.0;
            if (lse)
                lse[i] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int j = 0; j < nkv; ++j) {
            row[j] = exp(row[j] - m);
            ++exps;
            l += row[j];
        }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < nkv; ++j)
                acc += (row[j] / l) * v[(size_t)j * d + c];
            o[(size_t)i * d + c] = acc;
        }
        macs += (long long)nkv * d;
        if (lse)
            lse[i] = m + log(l);
    }
    free(S);
    if (counts) {
        counts[0] += macs;
        counts[1] += exps;
    }
}

static double *decode_rows(const void *src, int dtype, size_t base, size_t n) {
    double *out = (double *)malloc(n * sizeof(double));
    for (size_t i = 0; i < n; ++i)
        out[i] = load_elem(src, dtype, base + i);
    return out;
}

/* Full attention over Q [B,Hq,nq,d], K/V [B,Hkv,nkv,d] (contiguous, element
 * type in_dtype) into O [B,Hq,nq,d] and lse [B,Hq,nq] (fp64; lse may be
 * NULL).  Returns 0, or -1 on invalid sizes.  counts (nullable) receives the
 * total {multiply-adds, exp evaluations}. */
int oracle_sdpa(const void *Q, const void *K, const void *V, int in_dtype,
                double *O, double *lse, int B, int Hq, int Hkv, int nq,
                int nkv, int d, int causal, double scale, int nthreads,
                long long *counts) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || nq <= 0 || nkv <= 0 || d <= 0 ||
        Hq % Hkv != 0)
        return -1;
    int G = Hq / Hkv;
    long long total[2] = {0, 0};
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int bh = 0; bh < B * Hq; ++bh) {
        int b = bh / Hq, h = bh % Hq;
        int hk = h / G; /* [ACD] G query heads share one KV head */
        double *q = decode_rows(Q, in_dtype, ((size_t)b * Hq + h) * nq * d,
                                (size_t)nq * d);
        double *k = decode_rows(K, in_dtype, ((size_t)b * Hkv + hk) * nkv * d,
                                (size_t)nkv * d);
        double *v = decode_rows(V, in_dtype, ((size_t)b * Hkv + hk) * nkv * d,
                                (size_t)nkv * d);
        long long c[2] = {0, 0};
        sdpa_one_head(q, k, v, O + ((size_t)b * Hq + h) * nq * d,
                      lse ? lse + ((size_t)b * Hq + h) * nq : NULL, nq, nkv, d,
                      causal, scale, c);
#ifdef _OPENMP
#pragma omp critical
#endif
        {
            total[0] += c[0];
            total[1] += c[1];
        }
        free(q);
        free(k);
        free(v);
    }
    if (counts) {
        counts[0] = total[0];
        counts[1] = total[1];
    }
    return 0;
}

/* The same definition evaluated for selected rows only: rows[3*r+0..2] =
 * (b, h, i).  Each row materialises its own 1 x n_kv score row.  O_rows is
 * [nrows][d], lse_rows [nrows] (nullable).  Rows are independent under the
 * definition, so this is how outputs of large problems are sampled. */
int oracle_sdpa_rows(const void *Q, const void *K, const void *V, int in_dtype,
                     const int64_t *rows, int nrows, double *O_rows,
                     double *lse_rows, int B, int Hq, int Hkv, int nq, int nkv,
                     int d, int causal, double scale, int nthreads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || nq <= 0 || nkv <= 0 || d <= 0 ||
        Hq % Hkv != 0)
        return -1;
    for (int r = 0; r < nrows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= nq)
            return -1;
    }
    int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int r = 0; r < nrows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        int hk = (int)(h / G);
        double *q = decode_rows(Q, in_dtype, (((size_t)b * Hq + h) * nq + i) * d,
                                (size_t)d);
        double *k = decode_rows(K, in_dtype, ((size_t)b * Hkv + hk) * nkv * d,
                                (size_t)nkv * d);
        double *v = decode_rows(V, in_dtype, ((size_t)b * Hkv + hk) * nkv * d,
                                (size_t)nkv * d);
        /* row i of the full problem: its mask offset uses the full n_q */
        double *srow = (double *)malloc((size_t)nkv * sizeof(double));
        for (int j = 0; j < nkv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += q[c] * k[(size_t)j * d + c];
            srow[j] = acc * scale;
            if (causal && j > i + (nkv - nq))
                srow[j] = -INFINITY;
        }
        double m = -INFINITY;
        for (int j = 0; j < nkv; ++j)
            if (srow[j] > m)
                m = srow[j];
        double *o = O_rows + (size_t)r * d;
        if (m == -INFINITY) {
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
            if (lse_rows)
                lse_rows[r] = -INFINITY;
        } else {
            double l = 0.0;
            for (int j = 0; j < nkv; ++j) {
                srow[j] = exp(srow[j] - m);
                l += srow[j];
            }
            for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int j = 0; j < nkv; ++j)
                    acc += (srow[j] / l) * v[(size_t)j * d + c];
                o[c] = acc;
            }
            if (lse_rows)
                lse_rows[r] = m + log(l);
        }
        free(srow);
        free(q);
        free(k);
        free(v);
    }
    return 0;
}

/* -------------------------------------------------------------- decode */

/* One query token per sequence against a block-paged KV cache.
 *   q        [num_seqs][Hq][d]                (q_dtype)
 *   Kc, Vc   [num_blocks][Hkv][block_size][d] (kv_dtype)
 *   block_table [num_seqs][max_blocks_per_seq], seq_lens [num_seqs]
 * Token t of sequence s lives in block block_table[s][t / block_size], slot
 * t % block_size.  For E4M3 caches the stored code is decoded and multiplied
 * by the per-KV-head scale (k_scale / v_scale, [Hkv]).  The keys of each
 * (sequence, head) are gathered into a contiguous row in token order and the
 * definition is applied with n_q = 1 (the query sees the whole cache).
 * seq_subset (nullable) restricts the work to n_subset sequences; outputs of
 * the other sequences are left untouched.  O [num_seqs][Hq][d], lse
 * [num_seqs][Hq] (nullable).  counts (nullable): {multiply-adds, exps}. */
int oracle_decode_paged(const void *q, int q_dtype, const void *Kc,
                        const void *Vc, int kv_dtype, const float *k_scale,
                        const float *v_scale, const int32_t *block_table,
                        const int32_t *seq_lens, double *O, double *lse,
                        int num_seqs, int Hq, int Hkv, int d, int block_size,
                        int max_blocks_per_seq, int num_blocks, double scale,
                        const int32_t *seq_subset, int n_subset, int nthreads,
                        long long *counts) {
    if (num_seqs <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || block_size <= 0 ||
        Hq % Hkv != 0)
        return -1;
    if (kv_dtype == OR_E4M3 && (!k_scale || !v_scale))
        return -1;
    int G = Hq / Hkv;
    int nwork = seq_subset ? n_subset : num_seqs;
    /* validate every block index the gather will touch */
    for (int w = 0; w < nwork; ++w) {
        int s = seq_subset ? seq_subset[w] : w;
        if (s < 0 || s >= num_seqs)
            return -1;
        int len = seq_lens[s];
        if (len < 0 || (len + block_size - 1) / block_size > max_blocks_per_seq)
            return -1;
        for (int t = 0; t < len; t += block_size) {
            int blk = block_table[(size_t)s * max_blocks_per_seq + t / block_size];
            if (blk < 0 || blk >= num_blocks)
                return -1;
        }
    }
    long long total[2] = {0, 0};
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int wh = 0; wh < nwork * Hq; ++wh) {
        int w = wh / Hq, h = wh % Hq;
        int s = seq_subset ? seq_subset[w] : w;
        int hk = h / G;
        int len = seq_lens[s];
        double ks = (kv_dtype == OR_E4M3) ? (double)k_scale[hk] : 1.0;
        double vs = (kv_dtype == OR_E4M3) ? (double)v_scale[hk] : 1.0;
        double *qq = decode_rows(q, q_dtype, ((size_t)s * Hq + h) * d, (size_t)d);
        double *k = (double *)malloc(((size_t)len * d + 1) * sizeof(double));
        double *v = (double *)malloc(((size_t)len * d + 1) * sizeof(double));
        for (int t = 0; t < len; ++t) {
            int blk = block_table[(size_t)s * max_blocks_per_seq + t / block_size];
            size_t base = (((size_t)blk * Hkv + hk) * block_size + t % block_size) * d;
            for (int c = 0; c < d; ++c) {
                k[(size_t)t * d + c] = load_elem(Kc, kv_dtype, base + c) * ks;
                v[(size_t)t * d + c] = load_elem(Vc, kv_dtype, base + c) * vs;
            }
        }
        double *o = O + ((size_t)s * Hq + h) * d;
        double l_out = -INFINITY;
        if (len == 0) {
            for (int c = 0; c < d; ++c)
                o[c] = 0.0;
        } else {
            long long c2[2] = {0, 0};
            sdpa_one_head(qq, k, v, o, &l_out, 1, len, d, 0, scale, c2);
#ifdef _OPENMP
#pragma omp critical
#endif
            {
                total[0] += c2[0];
                total[1] += c2[1];
            }
        }
        if (lse)
            lse[(size_t)s * Hq + h] = l_out;
        free(qq);
        free(k);
        free(v);
    }
    if (counts) {
        counts[0] = total[0];
        counts[1] = total[1];
    }
    return 0;
}

/* ------------------------------------------------------------ kv append */

/* Backward pass of exact attention (marketmaker.cc, "Rückwärtsdurchlauf":
 * the probabilities are recomputed from Q, K and the stored row statistics
 * instead of being kept).  With S = scale Q K^T (causal: future keys
 * masked), P = softmax(S) row-wise and O = P V, the gradients of a loss
 * with dL/dO = dO are
 *   dV = P^T dO,
 *   dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P * (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q,
 * with dK and dV of a KV head summed over the G query heads that read it.
 * Everything is materialised in fp64 per (b, h).  mag_* (optional) receive,
 * per gradient element, the sum of the absolute values of the terms it is a
 * sum of (|P_ij dO_ic| for dV, scale |dS_ij K_jc| for dQ, scale |dS_ij Q_ic|
 * for dK) -- the scale against which rounding errors are judged.
 * d_err (optional, [B, Hq, nq]) bounds a perturbation of each row's D_i (an
 * implementation that forms D_i from a rounded copy of O sees one); dsens_q,
 * dsens_k then receive the resulting bound on the change of every dQ, dK
 * element: dS_ij moves by P_ij |dD_i|, so dQ_ic by scale d_err_i
 * sum_j P_ij |K_jc| and dK_jc by scale sum_i P_ij d_err_i |Q_ic|. */
int oracle_backward(const void *Q, const void *K, const void *V, const void *dO, int in_dtype,
                    double *dQ, double *dK, double *dV, double *mag_q, double *mag_k,
                    double *mag_v, const double *d_err, double *dsens_q, double *dsens_k,
                    int B, int Hq, int Hkv, int nq, int nkv, int d, int causal, double scale,
                    int nthreads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || nq <= 0 || nkv <= 0 || d <= 0 || Hq % Hkv != 0)
        return -1;
    if (causal && nq > nkv)
        return -1;
    const int G = Hq / Hkv;
    const size_t kv_elems = (size_t)B * Hkv * nkv * d;
    memset(dK, 0, kv_elems * sizeof(double));
    memset(dV, 0, kv_elems * sizeof(double));
    if (mag_k)
        memset(mag_k, 0, kv_elems * sizeof(double));
    if (mag_v)
        memset(mag_v, 0, kv_elems * sizeof(double));
    if (dsens_k)
        memset(dsens_k, 0, kv_elems * sizeof(double));
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int bk = 0; bk < B * Hkv; ++bk) { /* one KV head: its G query heads in turn */
        const int b = bk / Hkv, hk = bk % Hkv;
        double *k = decode_rows(K, in_dtype, (size_t)bk * nkv * d, (size_t)nkv * d);
        double *v = decode_rows(V, in_dtype, (size_t)bk * nkv * d, (size_t)nkv * d);
        double *P = (double *)malloc((size_t)nq * nkv * sizeof(double));
        double *dS = (double *)malloc((size_t)nq * nkv * sizeof(double));
        double *dk = dK + (size_t)bk * nkv * d, *dv = dV + (size_t)bk * nkv * d;
        double *mk = mag_k ? mag_k + (size_t)bk * nkv * d : NULL;
        double *mv = mag_v ? mag_v + (size_t)bk * nkv * d : NULL;
        for (int g = 0; g < G; ++g) {
            const int h = hk * G + g;
            const size_t qoff = ((size_t)b * Hq + h) * nq * d;
            double *q = decode_rows(Q, in_dtype, qoff, (size_t)nq * d);
            double *go = decode_rows(dO, in_dtype, qoff, (size_t)nq * d);
            /* P = softmax(scale Q K^T), masked */
            for (int i = 0; i < nq; ++i) {
                double *row = P + (size_t)i * nkv;
                double m = -INFINITY;
                for (int j = 0; j < nkv; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c)
                        acc += q[(size_t)i * d + c] * k[(size_t)j * d + c];
                    row[j] = (causal && j > i + (nkv - nq)) ? -INFINITY : acc * scale;
                    if (row[j] > m)
                        m = row[j];
                }
                double l = 0.0;
                for (int j = 0; j < nkv; ++j) {
                    row[j] = exp(row[j] - m);
                    l += row[j];
                }
                for (int j = 0; j < nkv; ++j)
                    row[j] /= l;
            }
            /* dP = dO V^T, D = rowsum(P * dP), dS = P * (dP - D) */
            for (int i = 0; i < nq; ++i) {
                double Di = 0.0;
                for (int j = 0; j < nkv; ++j) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c)
                        acc += go[(size_t)i * d + c] * v[(size_t)j * d + c];
                    dS[(size_t)i * nkv + j] = acc; /* dP for now */
                    Di += P[(size_t)i * nkv + j] * acc;
                }
                for (int j = 0; j < nkv; ++j)
                    dS[(size_t)i * nkv + j] = P[(size_t)i * nkv + j] * (dS[(size_t)i * nkv + j] - Di);
            }
            /* sensitivity of dQ, dK to perturbed D_i (bounds, not gradients) */
            if (d_err && (dsens_q || dsens_k)) {
                const double *de = d_err + ((size_t)b * Hq + h) * nq;
                for (int i = 0; i < nq; ++i)
                    for (int c = 0; c < d; ++c) {
                        if (dsens_q) {
                            double a = 0.0;
                            for (int j = 0; j < nkv; ++j)
                                a += P[(size_t)i * nkv + j] * fabs(k[(size_t)j * d + c]);
                            dsens_q[qoff + (size_t)i * d + c] = scale * de[i] * a;
                        }
                    }
                if (dsens_k) {
                    double *sk = dsens_k + (size_t)bk * nkv * d;
                    for (int j = 0; j < nkv; ++j)
                        for (int c = 0; c < d; ++c) {
                            double a = 0.0;
                            for (int i = 0; i < nq; ++i)
                                a += P[(size_t)i * nkv + j] * de[i] * fabs(q[(size_t)i * d + c]);
                            sk[(size_t)j * d + c] += scale * a;
                        }
                }
            }
            /* dV += P^T dO, dK += scale dS^T Q */
            for (int j = 0; j < nkv; ++j)
                for (int c = 0; c < d; ++c) {
                    double av = 0.0, ak = 0.0, mav = 0.0, mak = 0.0;
                    for (int i = 0; i < nq; ++i) {
                        const double tv = P[(size_t)i * nkv + j] * go[(size_t)i * d + c];
                        const double tk = dS[(size_t)i * nkv + j] * q[(size_t)i * d + c];
                        av += tv;
                        ak += tk;
                        mav += fabs(tv);
                        mak += fabs(tk);
                    }
                    dv[(size_t)j * d + c] += av;
                    dk[(size_t)j * d + c] += scale * ak;
                    if (mv)
                        mv[(size_t)j * d + c] += mav;
                    if (mk)
                        mk[(size_t)j * d + c] += scale * mak;
                }
            /* dQ = scale dS K */
            for (int i = 0; i < nq; ++i)
                for (int c = 0; c < d; ++c) {
                    double aq = 0.0, maq = 0.0;
                    for (int j = 0; j < nkv; ++j) {
                        const double tq = dS[(size_t)i * nkv + j] * k[(size_t)j * d + c];
                        aq += tq;
                        maq += fabs(tq);
                    }
                    dQ[qoff + (size_t)i * d + c] = scale * aq;
                    if (mag_q)
                        mag_q[qoff + (size_t)i * d + c] = scale * maq;
                }
            free(q);
            free(go);
        }
        free(k);
        free(v);
        free(P);
        free(dS);
    }
    return 0;
}

/* Prefill over a block-paged cache (prefix caching / chunked prefill):
 * for every sequence b and query head h, the n_q query rows Q[b,h] attend
 * to the len = seq_lens[b] cached keys of KV head h / G, gathered in token
 * order from cache[block_table[b][t / block_size]][h_kv][t % block_size]
 * ([TCOS] block-wise KV cache).  With causal set, query i sees key j iff
 * j <= i + (len - n_q) -- the new tokens are the last n_q of the sequence
 * (bottom-right alignment, [FASL] causal masking).  Only query rows
 * [row_lo, row_hi) are computed; O is [B, Hq, row_hi - row_lo, d] and lse
 * [B, Hq, row_hi - row_lo].  The scores of a row are materialised in fp64,
 * the row max is subtracted before exp ([IOAE] §8). */
int oracle_prefill_paged(const void *Q, int q_dtype, const void *Kc, const void *Vc,
                         int kv_dtype, const int32_t *block_table, const int32_t *seq_lens,
                         double *O, double *lse, int B, int Hq, int Hkv, int n_q, int d,
                         int block_size, int max_blocks_per_seq, int num_blocks, int causal,
                         double scale, int row_lo, int row_hi, int nthreads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || n_q <= 0 || d <= 0 || block_size <= 0 ||
        Hq % Hkv != 0 || row_lo < 0 || row_hi > n_q || row_lo >= row_hi)
        return -1;
    if (kv_dtype == OR_E4M3)
        return -1;
    const int G = Hq / Hkv;
    const int nr = row_hi - row_lo;
    for (int b = 0; b < B; ++b) {
        const int len = seq_lens[b];
        if (len < (causal ? n_q : 1) || (len + block_size - 1) / block_size > max_blocks_per_seq)
            return -1;
        for (int t = 0; t < len; t += block_size) {
            const int blk = block_table[(size_t)b * max_blocks_per_seq + t / block_size];
            if (blk < 0 || blk >= num_blocks)
                return -1;
        }
    }
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int bh = 0; bh < B * Hq; ++bh) {
        const int b = bh / Hq, h = bh % Hq, hk = h / G;
        const int len = seq_lens[b];
        double *k = (double *)malloc(((size_t)len * d + 1) * sizeof(double));
        double *v = (double *)malloc(((size_t)len * d + 1) * sizeof(double));
        double *srow = (double *)malloc(((size_t)len + 1) * sizeof(double));
        for (int t = 0; t < len; ++t) {
            const int blk = block_table[(size_t)b * max_blocks_per_seq + t / block_size];
            const size_t base = (((size_t)blk * Hkv + hk) * block_size + t % block_size) * d;
            for (int c = 0; c < d; ++c) {
                k[(size_t)t * d + c] = load_elem(Kc, kv_dtype, base + c);
                v[(size_t)t * d + c] = load_elem(Vc, kv_dtype, base + c);
            }
        }
        for (int i = row_lo; i < row_hi; ++i) {
            double *q = decode_rows(Q, q_dtype, (((size_t)b * Hq + h) * n_q + i) * d, (size_t)d);
            /* scores of row i, future keys masked to -inf */
            double m = -INFINITY;
            for (int j = 0; j < len; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += q[c] * k[(size_t)j * d + c];
                srow[j] = (causal && j > i + (len - n_q)) ? -INFINITY : acc * scale;
                if (srow[j] > m)
                    m = srow[j];
            }
            double *o = O + (((size_t)b * Hq + h) * nr + (i - row_lo)) * d;
            double l = 0.0;
            for (int j = 0; j < len; ++j) {
                srow[j] = exp(srow[j] - m);
                l += srow[j];
            }
            for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int j = 0; j < len; ++j)
                    acc += (srow[j] / l) * v[(size_t)j * d + c];
                o[c] = acc;
            }
            if (lse)
                lse[((size_t)b * Hq + h) * nr + (i - row_lo)] = m + log(l);
            free(q);
        }
        free(k);
        free(v);
        free(srow);
    }
    return 0;
}

/* Write T new tokens into the paged cache ([TCOS] KV cache concept: the new
 * K/V of each generated token is added to the cache).  k_new/v_new
 * [T][Hkv][d] (src_dtype), token r goes to sequence seq_ids[r] at position
 * positions[r]: block block_table[seq][pos / block_size], slot
 * pos % block_size.  Same-format copies keep the bit pattern; an E4M3 cache
 * stores e4m3(x / scale[h]) with x/scale evaluated in fp32 (the precision
 * the quantised code is decided in).  Returns 0 or -1. */
int oracle_kv_append(const void *k_new, const void *v_new, int src_dtype,
                     void *Kc, void *Vc, int kv_dtype, const float *k_scale,
                     const float *v_scale, const int32_t *block_table,
                     const int32_t *seq_ids, const int32_t *positions, int T,
                     int Hkv, int d, int block_size, int max_blocks_per_seq,
                     int num_seqs, int num_blocks) {
    if (T < 0 || Hkv <= 0 || d <= 0 || block_size <= 0)
        return -1;
    if (kv_dtype == OR_E4M3 && (!k_scale || !v_scale))
        return -1;
    if (kv_dtype != OR_E4M3 && kv_dtype != src_dtype)
        return -1;
    for (int r = 0; r < T; ++r) {
        int s = seq_ids[r], pos = positions[r];
        if (s < 0 || s >= num_seqs || pos < 0 || pos / block_size >= max_blocks_per_seq)
            return -1;
        int blk = block_table[(size_t)s * max_blocks_per_seq + pos / block_size];
        if (blk < 0 || blk >= num_blocks)
            return -1;
        for (int h = 0; h < Hkv; ++h) {
            size_t src = ((size_t)r * Hkv + h) * d;
            size_t dst = (((size_t)blk * Hkv + h) * block_size + pos % block_size) * d;
            for (int c = 0; c < d; ++c) {
                if (kv_dtype == OR_E4M3) {
                    float xk = (float)load_elem(k_new, src_dtype, src + c);
                    float xv = (float)load_elem(v_new, src_dtype, src + c);
                    ((uint8_t *)Kc)[dst + c] = oracle_f32_to_e4m3(xk / k_scale[h]);
                    ((uint8_t *)Vc)[dst + c] = oracle_f32_to_e4m3(xv / v_scale[h]);
                } else {
                    ((uint16_t *)Kc)[dst + c] = ((const uint16_t *)k_new)[src + c];
                    ((uint16_t *)Vc)[dst + c] = ((const uint16_t *)v_new)[src + c];
                }
            }
        }
    }
    return 0;
}
