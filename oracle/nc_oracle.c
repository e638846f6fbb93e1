/*
 * fp64 CPU oracle for exact causal sliding-window softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so and is
 * called by the test suite, by the package's smoke check and by the CPU
 * baseline leg of the benchmark.  The CUDA library never links, includes or
 * calls it, and it shares no code, header or table with the CUDA sources.
 *
 * What it computes, and where that comes from:
 *   - "nanochat GPT-2 speedrun" post (page 2; repeated on page 5), paragraph
 *     on the biggest improvements: attention runs through FlashAttention-3
 *     with its `window_size` argument, which gives alternating local/global
 *     (sliding-window / full causal) attention per layer.  The pages give no
 *     formula, so the oracle is the textbook definition of exact softmax
 *     attention restricted to the causal window.
 *   - "nanochat" walkthrough (page 4, inference paragraph closing the
 *     pretraining section; page 1 launch post): inference uses an Engine with
 *     a KV cache and a prefill/decode split, so decode is one query token
 *     attending over the cached keys/values, and prefill is a run of new
 *     query tokens appended after the cached ones.
 *
 * Readings where the pages are silent (each one is restated in the design
 * notes of the repository):
 *   - visibility: key j is visible to query i iff j <= i and i - j < W, i.e.
 *     the window counts W keys including the query's own position;
 *   - W <= -1 (the value -1) or W >= T mean full causal attention;
 *   - layout: q, k, v, o, dO, dq, dk, dv are contiguous [B, T, H, D];
 *     lse is [B, H, T] and holds the natural log of the softmax normaliser
 *     of the *scaled* scores;
 *   - decode: the query of sequence n is position L_n - 1 whose key/value
 *     already sit in the cache; cache rows max(0, L_n - W) .. L_n - 1 are
 *     visible;
 *   - prefill: the same cache layout; the last Tq of a sequence's L_n rows are
 *     the new tokens, and new token t is the query at position L_n - Tq + t.
 *
 * Everything is computed from the definition in double precision with plain
 * loops: no tiling, no online softmax, no reordering beyond the sums as
 * written.  OpenMP only splits independent (b, h) slices across threads.
 *
 * Definition (per batch b, head h, query i, with V(i) the visible set):
 *   s_ij  = scale * sum_d q_id k_jd                      j in V(i)
 *   M_i   = max_j s_ij
 *   lse_i = M_i + ln sum_j exp(s_ij - M_i)
 *   p_ij  = exp(s_ij - lse_i)
 *   o_i   = sum_j p_ij v_j
 * Gradients of a loss L given dO = dL/dO:
 *   dv_j  = sum_{i : j in V(i)} p_ij dO_i
 *   dp_ij = dO_i . v_j
 *   Delta_i = sum_j p_ij dp_ij
 *   ds_ij = p_ij (dp_ij - Delta_i)
 *   dq_i  = scale * sum_j ds_ij k_j
 *   dk_j  = scale * sum_i ds_ij q_i
 *
 * Parity pins: every function here is pinned by the CPU tests against
 * closed forms, invariants, brute-force enumeration, a library routine for
 * the same definition and finite differences; none is "parity unpinned".
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of keys visible in a row of length T with window W (W <= 0 -> full). */
static long eff_window(long W, long T) {
    if (W <= 0 || W >= T) return T;
    return W;
}

/* Element (b, t, h, d) of a contiguous [B, T, H, D] array. */
static size_t idx_bthd(long b, long t, long h, long d, long T, long H, long D) {
    return (((size_t)b * T + t) * H + h) * D + d;
}

/* Softmax weights of one query row over its visible keys.
 * p[j - lo] = exp(s_ij - lse_i) for j in [lo, i]; returns lse_i. */
static double row_probs(const double* q, const double* k, long b, long i, long h,
                        long lo, long T, long H, long D, double scale, double* p) {
    long n = i - lo + 1;
    double M = -INFINITY;
    for (long j = lo; j <= i; ++j) {
        double s = 0.0;
        for (long d = 0; d < D; ++d)
            s += q[idx_bthd(b, i, h, d, T, H, D)] * k[idx_bthd(b, j, h, d, T, H, D)];
        s *= scale;
        p[j - lo] = s;
        if (s > M) M = s;
    }
    double sum = 0.0;
    for (long t = 0; t < n; ++t) sum += exp(p[t] - M);
    double lse = M + log(sum);
    for (long t = 0; t < n; ++t) p[t] = exp(p[t] - lse);
    return lse;
}

/* Forward: o [B,T,H,D], lse [B,H,T]. */
void oracle_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                long B, long T, long H, long D, long window, double scale) {
    long W = eff_window(window, T);
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)W);
#pragma omp for schedule(dynamic, 1) collapse(2)
        for (long b = 0; b < B; ++b)
            for (long h = 0; h < H; ++h) {
                for (long i = 0; i < T; ++i) {
                    long lo = i - W + 1 < 0 ? 0 : i - W + 1;
                    double l = row_probs(q, k, b, i, h, lo, T, H, D, scale, p);
                    lse[((size_t)b * H + h) * T + i] = l;
                    for (long d = 0; d < D; ++d) {
                        double acc = 0.0;
                        for (long j = lo; j <= i; ++j)
                            acc += p[j - lo] * v[idx_bthd(b, j, h, d, T, H, D)];
                        o[idx_bthd(b, i, h, d, T, H, D)] = acc;
                    }
                }
            }
        free(p);
    }
}

/* Backward from the definition: dq, dk, dv [B,T,H,D] for upstream dO.
 * The softmax weights are recomputed in fp64; nothing from a forward run is
 * reused, so the gradients are those of the exact function. */
void oracle_bwd(const double* q, const double* k, const double* v, const double* dO,
                double* dq, double* dk, double* dv,
                long B, long T, long H, long D, long window, double scale) {
    long W = eff_window(window, T);
    size_t n_all = (size_t)B * T * H * D;
    memset(dq, 0, sizeof(double) * n_all);
    memset(dk, 0, sizeof(double) * n_all);
    memset(dv, 0, sizeof(double) * n_all);
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)W);
        double* dp = (double*)malloc(sizeof(double) * (size_t)W);
#pragma omp for schedule(dynamic, 1) collapse(2)
        for (long b = 0; b < B; ++b)
            for (long h = 0; h < H; ++h) {
                for (long i = 0; i < T; ++i) {
                    long lo = i - W + 1 < 0 ? 0 : i - W + 1;
                    long n = i - lo + 1;
                    (void)row_probs(q, k, b, i, h, lo, T, H, D, scale, p);
                    /* dp_ij = dO_i . v_j and Delta_i = sum_j p_ij dp_ij */
                    double delta = 0.0;
                    for (long j = lo; j <= i; ++j) {
                        double s = 0.0;
                        for (long d = 0; d < D; ++d)
                            s += dO[idx_bthd(b, i, h, d, T, H, D)] * v[idx_bthd(b, j, h, d, T, H, D)];
                        dp[j - lo] = s;
                        delta += p[j - lo] * s;
                    }
                    for (long t = 0; t < n; ++t) {
                        long j = lo + t;
                        double ds = p[t] * (dp[t] - delta);
                        for (long d = 0; d < D; ++d) {
                            dq[idx_bthd(b, i, h, d, T, H, D)] += scale * ds * k[idx_bthd(b, j, h, d, T, H, D)];
                            dk[idx_bthd(b, j, h, d, T, H, D)] += scale * ds * q[idx_bthd(b, i, h, d, T, H, D)];
                            dv[idx_bthd(b, j, h, d, T, H, D)] += p[t] * dO[idx_bthd(b, i, h, d, T, H, D)];
                        }
                    }
                }
            }
        free(p);
        free(dp);
    }
}

/* Decode over a padded KV cache.
 * q [N,H,D]; kc, vc [N,Tmax,H,D]; lens [N] with 1 <= lens[n] <= Tmax;
 * o [N,H,D]; lse [N,H].  Returns 0, or -1 when a length is out of range
 * (the rows of that sequence are then left as NaN). */
int oracle_decode(const double* q, const double* kc, const double* vc, const int* lens,
                  double* o, double* lse, long N, long Tmax, long H, long D, long window,
                  double scale) {
    int bad = 0;
    for (long n = 0; n < N; ++n) {
        long L = lens[n];
        if (L < 1 || L > Tmax) {
            bad = 1;
            for (long h = 0; h < H; ++h) {
                lse[n * H + h] = NAN;
                for (long d = 0; d < D; ++d) o[(n * H + h) * D + d] = NAN;
            }
            continue;
        }
        long W = eff_window(window, L);
        long lo = L - W;
        for (long h = 0; h < H; ++h) {
            double* p = (double*)malloc(sizeof(double) * (size_t)W);
            double M = -INFINITY;
            for (long j = lo; j < L; ++j) {
                double s = 0.0;
                for (long d = 0; d < D; ++d)
                    s += q[(n * H + h) * D + d] * kc[idx_bthd(n, j, h, d, Tmax, H, D)];
                s *= scale;
                p[j - lo] = s;
                if (s > M) M = s;
            }
            double sum = 0.0;
            for (long t = 0; t < W; ++t) sum += exp(p[t] - M);
            double l = M + log(sum);
            lse[n * H + h] = l;
            for (long t = 0; t < W; ++t) p[t] = exp(p[t] - l);
            for (long d = 0; d < D; ++d) {
                double acc = 0.0;
                for (long j = lo; j < L; ++j) acc += p[j - lo] * vc[idx_bthd(n, j, h, d, Tmax, H, D)];
                o[(n * H + h) * D + d] = acc;
            }
            free(p);
        }
    }
    return bad ? -1 : 0;
}

/* Prefill (append) over a KV cache: sequence n holds L_n = lens[n] cache rows, the last Tq of
 * which are the new tokens, whose keys and values are already in the cache.  New token t
 * (0 <= t < Tq) is the query at position i = L_n - Tq + t; it sees cache rows
 * max(0, i - W + 1) .. i (all rows up to i for W <= 0).  With Tq = 1 this is oracle_decode.
 * q [N,Tq,H,D]; caches [N,Tmax,H,D]; o [N,Tq,H,D]; lse [N,H,Tq].  A length outside [Tq, Tmax]
 * gives NaN rows for that sequence, and the call returns -1. */
int oracle_prefill(const double* q, const double* kc, const double* vc, const int* lens,
                   double* o, double* lse, long N, long Tq, long Tmax, long H, long D, long window,
                   double scale) {
    int bad = 0;
    for (long n = 0; n < N; ++n)
        if (lens[n] < Tq || lens[n] > Tmax) bad = 1;
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)Tmax);
#pragma omp for schedule(dynamic, 1) collapse(2)
        for (long n = 0; n < N; ++n)
            for (long h = 0; h < H; ++h) {
                long L = lens[n];
                for (long t = 0; t < Tq; ++t) {
                    double* orow = o + ((size_t)(n * Tq + t) * H + h) * D;
                    double* lrow = lse + ((size_t)n * H + h) * Tq + t;
                    if (L < Tq || L > Tmax) {
                        *lrow = NAN;
                        for (long d = 0; d < D; ++d) orow[d] = NAN;
                        continue;
                    }
                    long i = L - Tq + t;
                    long lo = (window <= 0 || i - window + 1 < 0) ? 0 : i - window + 1;
                    const double* qrow = q + ((size_t)(n * Tq + t) * H + h) * D;
                    double M = -INFINITY;
                    for (long j = lo; j <= i; ++j) {
                        double s = 0.0;
                        for (long d = 0; d < D; ++d) s += qrow[d] * kc[idx_bthd(n, j, h, d, Tmax, H, D)];
                        s *= scale;
                        p[j - lo] = s;
                        if (s > M) M = s;
                    }
                    double sum = 0.0;
                    for (long j = lo; j <= i; ++j) sum += exp(p[j - lo] - M);
                    double l = M + log(sum);
                    *lrow = l;
                    for (long j = lo; j <= i; ++j) p[j - lo] = exp(p[j - lo] - l);
                    for (long d = 0; d < D; ++d) {
                        double acc = 0.0;
                        for (long j = lo; j <= i; ++j) acc += p[j - lo] * vc[idx_bthd(n, j, h, d, Tmax, H, D)];
                        orow[d] = acc;
                    }
                }
            }
        free(p);
    }
    return bad ? -1 : 0;
}

/* Rotary position embedding of x [B, T, H, D] with tables cosv, sinv [T, D/2] (row t is position t).
 * "nanochat" walkthrough (page 4, comment thread): the model is Llama-like but simpler.  Reading (the
 * pages give no formula): Llama's rotate-half pairing, dimension i with dimension i + D/2,
 *   y_i       = x_i c - x_{i+D/2} s
 *   y_{i+D/2} = x_i s + x_{i+D/2} c,        c = cos[t][i], s = sin[t][i],
 * i.e. the pair (x_i, x_{i+D/2}) turned by the angle whose cosine and sine the tables hold.  With
 * inverse != 0 the transpose is applied (the turn back), which maps the gradient with respect to the
 * rotated vector to the gradient with respect to x.  q and k are rotated, v is not. */
void oracle_rotary(const double* x, const double* cosv, const double* sinv, double* y,
                   long B, long T, long H, long D, int inverse) {
    long half = D / 2;
#pragma omp parallel for collapse(2)
    for (long b = 0; b < B; ++b)
        for (long t = 0; t < T; ++t)
            for (long h = 0; h < H; ++h)
                for (long i = 0; i < half; ++i) {
                    double c = cosv[(size_t)t * half + i];
                    double s = sinv[(size_t)t * half + i];
                    if (inverse) s = -s;
                    double x1 = x[idx_bthd(b, t, h, i, T, H, D)];
                    double x2 = x[idx_bthd(b, t, h, i + half, T, H, D)];
                    y[idx_bthd(b, t, h, i, T, H, D)] = x1 * c - x2 * s;
                    y[idx_bthd(b, t, h, i + half, T, H, D)] = x1 * s + x2 * c;
                }
}

/* The rotary turn evaluated in float32 the way the CUDA kernels evaluate it: with x (bf16 values)
 * and the fp32 tables exact in float,
 *   y_i       = fmaf(x_i, c, -(x_{i+D/2} * s))
 *   y_{i+D/2} = fmaf(x_i, s,   x_{i+D/2} * c),
 * each product and each fused multiply-add rounded once to float32.  The rotary attention rounds the
 * turned q and k to bf16, a quantisation that floating point decides; both sides take that decision
 * in the same precision, so the oracle rounds this float32 turn (oracle_round_bf16), not its exact one.
 * Everything after the rounding is fp64 again. */
void oracle_rotary_f32(const double* x, const double* cosv, const double* sinv, double* y,
                       long B, long T, long H, long D) {
    long half = D / 2;
#pragma omp parallel for collapse(2)
    for (long b = 0; b < B; ++b)
        for (long t = 0; t < T; ++t)
            for (long h = 0; h < H; ++h)
                for (long i = 0; i < half; ++i) {
                    float c = (float)cosv[(size_t)t * half + i];
                    float s = (float)sinv[(size_t)t * half + i];
                    float x1 = (float)x[idx_bthd(b, t, h, i, T, H, D)];
                    float x2 = (float)x[idx_bthd(b, t, h, i + half, T, H, D)];
                    float p2s = x2 * s, p2c = x2 * c;
                    y[idx_bthd(b, t, h, i, T, H, D)] = (double)fmaf(x1, c, -p2s);
                    y[idx_bthd(b, t, h, i + half, T, H, D)] = (double)fmaf(x1, s, p2c);
                }
}

/* Round every value to the nearest bfloat16 (8 significant bits), ties to even, straight from
 * double (no intermediate float, so no double rounding).  The rotary attention takes the turned q
 * and k as bf16 tensors, the dtype of the model's activations ("nanochat GPT-2 speedrun" post,
 * page 2: the attention runs through a bf16 FlashAttention kernel), so the oracle rounds its
 * float32 turn (oracle_rotary_f32) once before the attention.  Values are assumed inside bf16's range (|x| < 2^128); zeros,
 * infinities and NaN are left as they are. */
void oracle_round_bf16(double* x, long n) {
    for (long i = 0; i < n; ++i) {
        double v = x[i];
        if (v == 0.0 || !isfinite(v)) continue;
        int e;
        frexp(v, &e);          /* v = m 2^e, 0.5 <= |m| < 1: the leading bit has weight 2^(e-1) */
        int ue = e - 8;        /* weight of the 8th significant bit: bf16's unit in the last place */
        if (ue < -133) ue = -133; /* below 2^-126 bf16 is subnormal with a fixed unit 2^-133 */
        x[i] = ldexp(nearbyint(ldexp(v, -ue)), ue); /* nearest integer multiple, ties to even */
    }
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
