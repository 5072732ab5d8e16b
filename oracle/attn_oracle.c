/*
 * attn_oracle.c -- fp64 CPU oracle for split-KV flash attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library (the package
 * split_kv_flash_gb300 and its CUDA sources) includes, links or calls this
 * file.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline /
 * reference leg load it.  It shares no code with the CUDA path.
 *
 * What it computes (the plain definition of attention that the tiled,
 * split, online-softmax method reproduces exactly up to rounding order):
 *
 *   FlashAttention tiling chapter, section 1 (tiling overview): S_ij = Q_i K_j^T
 *   for blocks of rows; the result is softmax(s * Q K^T) V.
 *   "The Occupancy Awakening" (flash-decode with KV splitting): each split keeps
 *   partial softmax statistics over its slice of the prefix and a reduction merges
 *   them; the merged value equals the unsplit softmax.
 *   FlashAttention tiling chapter, section 3.1 (block-level mask skipping): causal
 *   rows are aligned bottom-right (key offset seqlen_k - seqlen_q) and the local
 *   window has a lower bound at offset window_size_left.
 *
 * For every batch b, query head h and query row i in [0, sq):
 *   hk = h / G with G = Hq / Hkv            (query heads share KV head h / G)
 *   visible keys j in [0, sk_b):
 *       causal      -> j <= i + sk_b - sq
 *       window wl>=0-> j >= i + sk_b - sq - wl   (key at exactly wl back is visible)
 *   x_j   = scale * <Q[b,i,h,:], K[off_b + j, hk, :]>
 *   LSE   = ln sum_j exp(x_j)     (evaluated as M + ln sum exp(x_j - M), M = max x_j)
 *   O     = sum_j exp(x_j - LSE) * V[off_b + j, hk, :]
 *   no visible key -> O = 0, LSE = -inf.
 * Keys and queries have d columns, values and outputs dv (dv = d except for the
 * latent-attention entry points: "The Occupancy Awakening", the absorbed-MLA
 * verify of Kimi K2.6 with 512 + 64 query/key columns and 512 value columns).
 *
 * Everything is double precision.  Inputs arrive as raw bf16 bit patterns
 * (uint16), widened exactly to double.  No tiling, no online rescaling: the
 * whole logit row is formed, then max, then the exponential sum, then x V.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Visibility of key j for query row i (tiling chapter section 3.1: bottom-right
 * causal alignment and the local lower bound).  With causal == 0 and a window,
 * only the left bound applies. */
static int key_visible(long i, long j, long sq, long sk, int causal, long wl) {
    long diag = i + sk - sq;
    if (j < 0 || j >= sk) return 0;
    if (causal && j > diag) return 0;
    if (wl >= 0 && j < diag - wl) return 0;
    return 1;
}

/* One output row restricted to keys in [j_lo, j_hi) (all keys: 0, sk).
 * Writes dv doubles to o_row and returns the log-sum-exp. */
static double attn_row(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       int Hq, int Hkv, int sq, int d, int dv, double scale, int causal,
                       int wl, long b, long h, long i, long sk, long off,
                       long j_lo, long j_hi, double* logits, double* o_row) {
    const long G = Hq / Hkv;
    const long hk = h / G;
    const uint16_t* qrow = q + (((size_t)b * sq + i) * Hq + h) * (size_t)d;
    long nvis = 0;
    double mx = -INFINITY;
    if (j_lo < 0) j_lo = 0;
    if (j_hi > sk) j_hi = sk;
    /* 1. logits x_j = scale * q . k_j for every visible key */
    for (long j = j_lo; j < j_hi; ++j) {
        if (!key_visible(i, j, sq, sk, causal, wl)) {
            logits[j - j_lo] = -INFINITY;
            continue;
        }
        const uint16_t* krow = k + (((size_t)(off + j)) * Hkv + hk) * (size_t)d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += bf16_bits_to_double(qrow[c]) * bf16_bits_to_double(krow[c]);
        double x = scale * dot;
        logits[j - j_lo] = x;
        if (x > mx) mx = x;
        ++nvis;
    }
    for (int c = 0; c < dv; ++c) o_row[c] = 0.0;
    if (nvis == 0) return -INFINITY;
    /* 2. softmax normaliser */
    double sum = 0.0;
    for (long j = j_lo; j < j_hi; ++j) {
        double x = logits[j - j_lo];
        if (x == -INFINITY) continue;
        sum += exp(x - mx);
    }
    double lse = mx + log(sum);
    /* 3. O = sum_j softmax_j * V_j */
    for (long j = j_lo; j < j_hi; ++j) {
        double x = logits[j - j_lo];
        if (x == -INFINITY) continue;
        double w = exp(x - lse);
        const uint16_t* vrow = v + (((size_t)(off + j)) * Hkv + hk) * (size_t)dv;
        for (int c = 0; c < dv; ++c) o_row[c] += w * bf16_bits_to_double(vrow[c]);
    }
    return lse;
}

static int check_args(int B, int Hq, int Hkv, int sq, const int* kv_len, int d) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || sq < 0 || d <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    for (int b = 0; b < B; ++b)
        if (kv_len[b] < 0) return -1;
    return 0;
}

/*
 * Selected rows of the attention output.  rows holds n_rows triples
 * (b, h, i); out_rows receives n_rows x dv doubles, lse_rows n_rows doubles.
 * Layouts: q [B, sq, Hq, d]; k [sum_b kv_len[b], Hkv, d] and v
 * [sum_b kv_len[b], Hkv, dv] packed by sequence (offset of sequence b = sum of
 * the lengths before it).  Returns 0, or -1 on bad arguments.
 */
int oracle_attn_rows_v(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       int B, int Hq, int Hkv, int sq, const int* kv_len, int d, int dv,
                       double scale, int causal, int window_left,
                       const int* rows, long n_rows, double* out_rows, double* lse_rows,
                       int nthreads) {
    if (check_args(B, Hq, Hkv, sq, kv_len, d) || dv <= 0) return -1;
    long* off = (long*)malloc(sizeof(long) * (size_t)(B + 1));
    long max_sk = 0;
    off[0] = 0;
    for (int b = 0; b < B; ++b) {
        off[b + 1] = off[b] + kv_len[b];
        if (kv_len[b] > max_sk) max_sk = kv_len[b];
    }
    for (long r = 0; r < n_rows; ++r) {
        int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= sq) { free(off); return -1; }
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double* logits = (double*)malloc(sizeof(double) * (size_t)(max_sk > 0 ? max_sk : 1));
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < n_rows; ++r) {
            long b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
            lse_rows[r] = attn_row(q, k, v, Hq, Hkv, sq, d, dv, scale, causal, window_left, b, h, i,
                                   kv_len[b], off[b], 0, kv_len[b], logits,
                                   out_rows + (size_t)r * dv);
        }
        free(logits);
    }
    free(off);
    return 0;
}

/* Keys and values of one width (the common case). */
int oracle_attn_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     int B, int Hq, int Hkv, int sq, const int* kv_len, int d,
                     double scale, int causal, int window_left,
                     const int* rows, long n_rows, double* out_rows, double* lse_rows,
                     int nthreads) {
    return oracle_attn_rows_v(q, k, v, B, Hq, Hkv, sq, kv_len, d, d, scale, causal, window_left,
                              rows, n_rows, out_rows, lse_rows, nthreads);
}

/*
 * Full attention forward: out [B, sq, Hq, dv] (double), lse [B, Hq, sq] (double).
 */
int oracle_attn_fwd_v(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      int B, int Hq, int Hkv, int sq, const int* kv_len, int d, int dv,
                      double scale, int causal, int window_left,
                      double* out, double* lse, int nthreads) {
    if (check_args(B, Hq, Hkv, sq, kv_len, d) || dv <= 0) return -1;
    long n = (long)B * Hq * sq;
    int* rows = (int*)malloc(sizeof(int) * 3 * (size_t)(n > 0 ? n : 1));
    double* o_rows = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * dv);
    double* l_rows = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    long r = 0;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h)
            for (int i = 0; i < sq; ++i) {
                rows[3 * r] = b; rows[3 * r + 1] = h; rows[3 * r + 2] = i; ++r;
            }
    int rc = oracle_attn_rows_v(q, k, v, B, Hq, Hkv, sq, kv_len, d, dv, scale, causal, window_left,
                                rows, n, o_rows, l_rows, nthreads);
    if (rc == 0) {
        r = 0;
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hq; ++h)
                for (int i = 0; i < sq; ++i) {
                    memcpy(out + (((size_t)b * sq + i) * Hq + h) * dv, o_rows + (size_t)r * dv,
                           sizeof(double) * dv);
                    lse[((size_t)b * Hq + h) * sq + i] = l_rows[r];
                    ++r;
                }
    }
    free(rows); free(o_rows); free(l_rows);
    return rc;
}

/* Keys and values of one width (the common case). */
int oracle_attn_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    int B, int Hq, int Hkv, int sq, const int* kv_len, int d,
                    double scale, int causal, int window_left,
                    double* out, double* lse, int nthreads) {
    return oracle_attn_fwd_v(q, k, v, B, Hq, Hkv, sq, kv_len, d, d, scale, causal, window_left,
                             out, lse, nthreads);
}

/*
 * Split reference, used only to check split invariance.  For batch b the key
 * axis is cut at bounds[b * (S + 1) + t], t = 0..S (non-decreasing, from 0 to
 * kv_len[b]); split t covers keys [bounds[t], bounds[t+1]).  Each split is
 * evaluated on its own (O_t, LSE_t as above, restricted to its keys; empty ->
 * O_t = 0, LSE_t = -inf) and the partials are merged by their log-sum-exps
 * ("The Occupancy Awakening", KV-split reduction; tiling chapter section 5.1,
 * the separate combine step):
 *   M   = max_t LSE_t
 *   LSE = M + ln sum_t exp(LSE_t - M)
 *   O   = sum_t exp(LSE_t - LSE) * O_t
 * All partials at -inf -> O = 0, LSE = -inf.
 */
int oracle_attn_fwd_split(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          int B, int Hq, int Hkv, int sq, const int* kv_len, int d,
                          double scale, int causal, int window_left,
                          int S, const int* bounds, double* out, double* lse, int nthreads) {
    if (check_args(B, Hq, Hkv, sq, kv_len, d) || S <= 0) return -1;
    long* off = (long*)malloc(sizeof(long) * (size_t)(B + 1));
    long max_sk = 0;
    off[0] = 0;
    for (int b = 0; b < B; ++b) {
        off[b + 1] = off[b] + kv_len[b];
        if (kv_len[b] > max_sk) max_sk = kv_len[b];
        const int* bd = bounds + (size_t)b * (S + 1);
        if (bd[0] != 0 || bd[S] != kv_len[b]) { free(off); return -1; }
        for (int t = 0; t < S; ++t)
            if (bd[t + 1] < bd[t]) { free(off); return -1; }
    }
    long n = (long)B * Hq * sq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double* logits = (double*)malloc(sizeof(double) * (size_t)(max_sk > 0 ? max_sk : 1));
        double* o_part = (double*)malloc(sizeof(double) * (size_t)S * d);
        double* l_part = (double*)malloc(sizeof(double) * (size_t)S);
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < n; ++r) {
            long b = r / ((long)Hq * sq);
            long h = (r / sq) % Hq;
            long i = r % sq;
            const int* bd = bounds + (size_t)b * (S + 1);
            double mx = -INFINITY;
            for (int t = 0; t < S; ++t) {
                l_part[t] = attn_row(q, k, v, Hq, Hkv, sq, d, d, scale, causal, window_left, b, h, i,
                                     kv_len[b], off[b], bd[t], bd[t + 1], logits,
                                     o_part + (size_t)t * d);
                if (l_part[t] > mx) mx = l_part[t];
            }
            double* o_row = out + (((size_t)b * sq + i) * Hq + h) * d;
            for (int c = 0; c < d; ++c) o_row[c] = 0.0;
            double total;
            if (mx == -INFINITY) {
                total = -INFINITY;
            } else {
                double acc = 0.0;
                for (int t = 0; t < S; ++t)
                    if (l_part[t] != -INFINITY) acc += exp(l_part[t] - mx);
                total = mx + log(acc);
                for (int t = 0; t < S; ++t) {
                    if (l_part[t] == -INFINITY) continue;
                    double w = exp(l_part[t] - total);
                    for (int c = 0; c < d; ++c) o_row[c] += w * o_part[(size_t)t * d + c];
                }
            }
            lse[((size_t)b * Hq + h) * sq + i] = total;
        }
        free(logits); free(o_part); free(l_part);
    }
    free(off);
    return 0;
}

/* Number of visible (query, key) pairs of one head, by enumeration of the
 * visibility rule above; used to pin the masks against closed-form counts. */
long long oracle_count_visible(int sq, int sk, int causal, int window_left) {
    long long n = 0;
    for (long i = 0; i < sq; ++i)
        for (long j = 0; j < sk; ++j)
            n += key_visible(i, j, sq, sk, causal, window_left);
    return n;
}
