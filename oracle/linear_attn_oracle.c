/*
 * linear_attn_oracle.c -- fp64 CPU oracle for chunk-parallel gated linear
 * attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes, links or
 * calls this file; only tests/, __graft_entry__.smoke() and bench.py's CPU
 * legs load it.  It shares no code with the CUDA path.
 *
 * Source: inclusionAI/cuLA issue #11 (linear-attention kernels at small batch,
 * head count and length): each (sequence, head) is split along T into N
 * segments that run in parallel and are merged by an affine combine (M, h_ext).
 * The pages do not print the recurrence itself.  The reading taken here is
 * gated linear attention with one decay per key channel, whose state update is
 * affine in the state, so a segment is summarised by (M, h_ext):
 *
 *   S_0 = 0                                   (dk x dv, per sequence and head)
 *   S_t = Diag(exp(g_t)) S_{t-1} + k_t v_t^T   (g_t <= 0: log decay per key channel)
 *   o_t = scale * S_t^T q_t
 *
 * A segment [t0, t1) started from S_in ends at M S_in + h_ext with
 *   M     = Diag(exp(sum_{t0 <= t < t1} g_t))
 *   h_ext = the state at t1 - 1 of the recurrence started from 0 at t0,
 * so S_in of segment i+1 = M_i S_in(i) + h_ext(i), S_in(0) = 0, and the outputs
 * of segment i come from re-running it from S_in(i).  Segment i covers
 * [i L, min((i + 1) L, T)) with L = ceil(T / N).
 *
 * Layouts: q, k [B, T, H, dk] and v [B, T, H, dv] as bf16 bit patterns;
 * g [B, T, H, dk] float32; out [B, T, H, dv] and state [B, H, dk, dv] double.
 * Everything is computed in double precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

static double la_bf16(uint16_t bits) {
    union {
        uint32_t u;
        float f;
    } x;
    x.u = ((uint32_t)bits) << 16;
    return (double)x.f;
}

static int la_check(int B, int T, int H, int dk, int dv) {
    return (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) ? 1 : 0;
}

/* One token of the recurrence on state S (dk x dv, row-major): decay, then the
 * outer product; if out is not NULL also o = scale * S^T q. */
static void la_token(double* S, const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* g,
                     int dk, int dv, double scale, double* out) {
    for (int i = 0; i < dk; ++i) {
        const double a = exp((double)g[i]);
        const double ki = la_bf16(k[i]);
        double* row = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) row[j] = a * row[j] + ki * la_bf16(v[j]);
    }
    if (out) {
        for (int j = 0; j < dv; ++j) out[j] = 0.0;
        for (int i = 0; i < dk; ++i) {
            const double qi = la_bf16(q[i]);
            const double* row = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j) out[j] += qi * row[j];
        }
        for (int j = 0; j < dv; ++j) out[j] *= scale;
    }
}

/* The recurrence token by token over the whole sequence. */
int oracle_gla_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* g, int B, int T,
                   int H, int dk, int dv, double scale, double* out, double* state, int nthreads) {
    if (la_check(B, T, H, dk, dv)) return 1;
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * H; ++bh) {
        const int b = bh / H, h = bh % H;
        double* S = (double*)calloc((size_t)dk * dv, sizeof(double));
        for (int t = 0; t < T; ++t) {
            const size_t row = ((size_t)b * T + t) * H + h;
            la_token(S, q + row * dk, k + row * dk, v + row * dv, g + row * dk, dk, dv, scale,
                     out ? out + row * dv : NULL);
        }
        if (state) memcpy(state + (size_t)bh * dk * dv, S, sizeof(double) * (size_t)dk * dv);
        free(S);
    }
    return 0;
}

/* The segment method in the issue's order: every segment's (M, h_ext) from a
 * zero state, the affine combine over the segments, then every segment's
 * outputs from its incoming state. */
int oracle_gla_fwd_segments(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* g, int B,
                            int T, int H, int dk, int dv, double scale, int nseg, double* out, int nthreads) {
    if (la_check(B, T, H, dk, dv) || nseg <= 0) return 1;
    if (nthreads > 0) omp_set_num_threads(nthreads);
    const int L = T > 0 ? (T + nseg - 1) / nseg : 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bh = 0; bh < B * H; ++bh) {
        const int b = bh / H, h = bh % H;
        const size_t SZ = (size_t)dk * dv;
        double* hext = (double*)calloc(SZ * nseg, sizeof(double));
        double* logm = (double*)calloc((size_t)dk * nseg, sizeof(double));
        double* sin = (double*)calloc(SZ * nseg, sizeof(double));
        /* 1. each segment alone: h_ext from zero, log of M's diagonal */
        for (int s = 0; s < nseg; ++s) {
            const int t0 = s * L, t1 = (s + 1) * L < T ? (s + 1) * L : T;
            for (int t = t0; t < t1; ++t) {
                const size_t row = ((size_t)b * T + t) * H + h;
                la_token(hext + SZ * s, NULL, k + row * dk, v + row * dv, g + row * dk, dk, dv, scale, NULL);
                for (int i = 0; i < dk; ++i) logm[(size_t)s * dk + i] += (double)g[row * dk + i];
            }
        }
        /* 2. affine combine: S_in(s + 1) = M_s S_in(s) + h_ext(s) */
        for (int s = 0; s + 1 < nseg; ++s)
            for (int i = 0; i < dk; ++i) {
                const double m = exp(logm[(size_t)s * dk + i]);
                for (int j = 0; j < dv; ++j)
                    sin[SZ * (s + 1) + (size_t)i * dv + j] =
                        m * sin[SZ * s + (size_t)i * dv + j] + hext[SZ * s + (size_t)i * dv + j];
            }
        /* 3. outputs: each segment re-run from its incoming state */
        double* S = (double*)malloc(SZ * sizeof(double));
        for (int s = 0; s < nseg; ++s) {
            const int t0 = s * L, t1 = (s + 1) * L < T ? (s + 1) * L : T;
            memcpy(S, sin + SZ * s, SZ * sizeof(double));
            for (int t = t0; t < t1; ++t) {
                const size_t row = ((size_t)b * T + t) * H + h;
                la_token(S, q + row * dk, k + row * dk, v + row * dv, g + row * dk, dk, dv, scale, out + row * dv);
            }
        }
        free(S);
        free(sin);
        free(logm);
        free(hext);
    }
    return 0;
}
