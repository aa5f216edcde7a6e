/*
 * TEST INFRASTRUCTURE — NOT PART OF THE PRODUCT PATH.
 *
 * Float64 token-by-token oracle for the Gated DeltaNet recurrent mixer.
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline may load this library. It shares no code, header or table with
 * the CUDA library.
 *
 * What it computes (the plain definition, one token at a time):
 *
 *   S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *   o_t = q_scale * S_t^T q_t
 *
 * per (sequence, value head), with the fp32 state S of shape [dk, dv].  This
 * is the one-token decoder step that the Qwen3.5 chunked-prefill pull request
 * ("perf(qwen3_5): prefill text prompts in multi-token chunks", Background and
 * Exit Criteria) keeps for decode and whose results the chunked rule must
 * reproduce ("Generated tokens match the token-by-token prefill").  The
 * chunked closed form of that page's Implementation section is an exact
 * algebraic rearrangement of this loop.
 *
 * Optional steps before the loop, in this order:
 *   1. depthwise causal short convolution over [previous conv state ++ the
 *      prompt's columns]; the new conv state is the last kernel-1 columns
 *      ("perf(mamba): prefill text prompts in multi-token chunks",
 *      Implementation, add_short_conv_rows; reused by the Qwen3.5 page's
 *      Implementation section), optionally followed by SiLU;
 *   2. L2 normalisation of every q and k head vector: x / sqrt(sum x^2 + eps).
 *
 * Everything is float64 with plain loops; OpenMP only distributes independent
 * (sequence, channel), (token, head) and (sequence, head) work items.
 * Compile with -ffp-contract=off so x86 and Arm give the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

/* Activation applied after the short convolution. 0 = none, 1 = SiLU. */
static double oracle_act(double y, int act)
{
    if (act == 1) return y / (1.0 + exp(-y));
    return y;
}

/*
 * Depthwise causal convolution of one channel of one sequence.
 *   xx = [state_in[0..K-2], x[0..L-1]]      (oldest first)
 *   y[t] = act(sum_{j<K} w[j] * xx[t + j])   (tap K-1 weighs the current token)
 *   state_out = last K-1 entries of xx
 * x and y are strided (stride = number of channels).  Returns 0, or 2 when
 * out of memory.
 */
static int oracle_conv_channel(const double* x, double* y, long stride, long L,
                               const double* w, int K, const double* state_in,
                               double* state_out, int act)
{
    long n = L + K - 1;
    double* xx = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!xx) return ORACLE_NO_MEMORY;
    for (int j = 0; j < K - 1; ++j) xx[j] = state_in ? state_in[j] : 0.0;
    for (long t = 0; t < L; ++t) xx[K - 1 + t] = x[t * stride];
    for (long t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int j = 0; j < K; ++j) acc += w[j] * xx[t + j];
        y[t * stride] = oracle_act(acc, act);
    }
    if (state_out)
        for (int j = 0; j < K - 1; ++j) state_out[j] = xx[n - (K - 1) + j];
    free(xx);
    return ORACLE_OK;
}

/*
 * oracle_short_conv — the short convolution over a packed batch.
 *   x, y            [T, C]   (y may not alias x)
 *   w               [C, K]
 *   state_in/out    [B, C, K-1], oldest first; state_in NULL = zeros,
 *                   state_out NULL = not written; they may alias.
 *   cu_seqlens      [B+1]
 */
int oracle_short_conv(const double* x, double* y, const double* w, int K,
                      const double* state_in, double* state_out, int act,
                      const int32_t* cu_seqlens, int B, long C)
{
    if (!x || !y || !w || !cu_seqlens || K < 1 || C < 1 || B < 0) return ORACLE_BAD_ARG;
    long work = (long)B * C;
    int fail = 0;
#pragma omp parallel for schedule(static)
    for (long it = 0; it < work; ++it) {
        long n = it / C, c = it % C;
        long t0 = cu_seqlens[n], L = cu_seqlens[n + 1] - t0;
        const double* sin = state_in ? state_in + (n * C + c) * (K - 1) : NULL;
        double* sout = state_out ? state_out + (n * C + c) * (K - 1) : NULL;
        if (oracle_conv_channel(x + t0 * C + c, y + t0 * C + c, C, L, w + c * K, K,
                                sin, sout, act) != ORACLE_OK) {
#pragma omp atomic write
            fail = 1;
        }
    }
    return fail ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* x <- x / sqrt(sum x^2 + eps), in place, n contiguous values. */
static void oracle_l2norm(double* x, int n, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < n; ++i) x[i] *= inv;
}

/* oracle_l2norm_rows — normalise `rows` vectors of length n, stored with
 * `stride` doubles between consecutive rows, in place. */
int oracle_l2norm_rows(double* x, long rows, int n, long stride, double eps)
{
    if (!x || rows < 0 || n < 1) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) oracle_l2norm(x + r * stride, n, eps);
    return ORACLE_OK;
}

/*
 * oracle_prefill — the whole mixer over a packed variable-length batch.
 *
 * Layouts (row-major, token-major packed):
 *   q, k      [T, Hk, dk]   (ignored when conv_x != NULL)
 *   v         [T, Hv, dv]   (ignored when conv_x != NULL)
 *   conv_x    [T, 2*Hk*dk + Hv*dv]  channels ordered q | k | v, or NULL
 *   conv_w    [channels, K]
 *   conv_state_in / conv_state_out  [B, channels, K-1] oldest first, may be NULL
 *   g, beta   [T, Hv]
 *   state_in / state_out  [B, Hv, dk, dv]; state_in NULL = zero state
 *   out       [T, Hv, dv]
 *   cu_seqlens [B+1], cu[0] = 0, non-decreasing, cu[B] = T
 * Value head h reads key head h / (Hv / Hk).
 */
int oracle_prefill(const double* q, const double* k, const double* v,
                   const double* conv_x, const double* conv_w,
                   const double* conv_state_in, double* conv_state_out,
                   int conv_K, int conv_act,
                   const double* g, const double* beta,
                   const double* state_in, double* state_out, double* out,
                   const int32_t* cu_seqlens, int B, int Hk, int Hv, int dk,
                   int dv, int use_l2norm, double eps, double q_scale,
                   int nthreads)
{
    if (B < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk != 0)
        return ORACLE_BAD_ARG;
    if (!cu_seqlens || !g || !beta || !out) return ORACLE_BAD_ARG;
    if (cu_seqlens[0] != 0) return ORACLE_BAD_ARG;
    for (int n = 0; n < B; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return ORACLE_BAD_ARG;
    if (conv_x && (!conv_w || conv_K < 1)) return ORACLE_BAD_ARG;
    if (!conv_x && (!q || !k || !v)) return ORACLE_BAD_ARG;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

    const long T = cu_seqlens[B];
    const long cq = (long)Hk * dk, cv = (long)Hv * dv;
    const long C = 2 * cq + cv;

    /* Working copies of q, k, v in [T, channels] float64. */
    double* qkv = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * (size_t)C);
    if (!qkv) return ORACLE_NO_MEMORY;

    if (conv_x) {
        /* Step 1: short convolution, one (sequence, channel) at a time. */
        int rc = oracle_short_conv(conv_x, qkv, conv_w, conv_K, conv_state_in,
                                   conv_state_out, conv_act, cu_seqlens, B, C);
        if (rc != ORACLE_OK) {
            free(qkv);
            return rc;
        }
    } else {
#pragma omp parallel for schedule(static)
        for (long t = 0; t < T; ++t) {
            memcpy(qkv + t * C, q + t * cq, sizeof(double) * (size_t)cq);
            memcpy(qkv + t * C + cq, k + t * cq, sizeof(double) * (size_t)cq);
            memcpy(qkv + t * C + 2 * cq, v + t * cv, sizeof(double) * (size_t)cv);
        }
    }

    /* Step 2: L2 normalisation of each q and k head vector (q heads occupy
     * channels [0, Hk*dk), k heads [Hk*dk, 2*Hk*dk)). */
    if (use_l2norm) {
        long work = T * 2 * Hk;
#pragma omp parallel for schedule(static)
        for (long it = 0; it < work; ++it) {
            long t = it / (2 * Hk), r = it % (2 * Hk);
            oracle_l2norm(qkv + t * C + r * dk, dk, eps);
        }
    }

    /* Step 3: the recurrence, one (sequence, value head) at a time. */
    const int group = Hv / Hk;
    long work = (long)B * Hv;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long it = 0; it < work; ++it) {
        long n = it / Hv;
        int h = (int)(it % Hv), kh = h / group;
        double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
        double* u = (double*)malloc(sizeof(double) * (size_t)dv);
        if (!S || !u) {
            free(S);
            free(u);
#pragma omp atomic write
            fail = 1;
            continue;
        }
        const double* s0 = state_in ? state_in + (n * Hv + h) * (long)dk * dv : NULL;
        for (long i = 0; i < (long)dk * dv; ++i) S[i] = s0 ? s0[i] : 0.0;

        for (long t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            const double* qt = qkv + t * C + kh * dk;
            const double* kt = qkv + t * C + cq + kh * dk;
            const double* vt = qkv + t * C + 2 * cq + (long)h * dv;
            double decay = exp(g[t * Hv + h]);
            double b = beta[t * Hv + h];
            /* S <- exp(g) S */
            for (long i = 0; i < (long)dk * dv; ++i) S[i] *= decay;
            /* u = beta (v - S^T k) */
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[(long)i * dv + j] * kt[i];
                u[j] = b * (vt[j] - acc);
            }
            /* S <- S + k u^T */
            for (int i = 0; i < dk; ++i)
                for (int j = 0; j < dv; ++j) S[(long)i * dv + j] += kt[i] * u[j];
            /* o = q_scale S^T q  (the updated state) */
            double* ot = out + (t * Hv + h) * (long)dv;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += S[(long)i * dv + j] * qt[i];
                ot[j] = q_scale * acc;
            }
        }
        if (state_out) {
            double* s1 = state_out + (n * Hv + h) * (long)dk * dv;
            memcpy(s1, S, sizeof(double) * (size_t)dk * dv);
        }
        free(S);
        free(u);
    }
    free(qkv);
    return fail ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Selective-scan rows ("perf(mamba): prefill text prompts in multi-token
 * chunks", Implementation, add_selective_scan_rows): the first-order linear
 * recurrence h_t = a_t h_{t-1} + b_t per channel, one row at a time, from the
 * incoming state h_0 = h_in[n, c] (zero when h_in is NULL).
 *   a, b, h_rows: [T, C] row-major (token-major); h_in, h_out: [B, C].
 *   h_rows[t, c] = h_t; h_out[n, c] = h after the last row of sequence n
 *   (h_0 for an empty sequence).
 */
int oracle_scan_rows(const double* a, const double* b, const double* h_in,
                     double* h_out, double* h_rows, const int32_t* cu,
                     int B, long C)
{
    if (!a || !b || !h_out || !h_rows || !cu || B < 0 || C < 0) return ORACLE_BAD_ARG;
    long items = (long)B * C;
#pragma omp parallel for schedule(static)
    for (long it = 0; it < items; ++it) {
        const long n = it / C, c = it % C;
        double h = h_in ? h_in[n * C + c] : 0.0;
        for (long t = cu[n]; t < cu[n + 1]; ++t) {
            h = a[t * C + c] * h + b[t * C + c];
            h_rows[t * C + c] = h;
        }
        h_out[n * C + c] = h;
    }
    return ORACLE_OK;
}

/*
 * RWKV-4 WKV rows ("perf(rwkv): prefill text prompts in multi-token chunks",
 * Implementation): the one-token decoder's recurrence, one row at a time.
 * Per channel the state is (num, den, max) with A = num exp(max) and
 * B = den exp(max) of
 *   A_t = exp(w) A_{t-1} + exp(k_t) v_t,   B_t = exp(w) B_{t-1} + exp(k_t),
 * and the output is
 *   wkv_t = (A_{t-1} + exp(u + k_t) v_t) / (B_{t-1} + exp(u + k_t)).
 * Every exponential is taken after subtracting the largest exponent of the
 * sum, as the decoder does.  An absent state is (0, 0, -1e38).
 *   k, v, wkv: [T, C]; w, u: [C]; state_in / state_out: [B, 3, C] holding
 *   num, den, max; state_in may be NULL.
 */
int oracle_wkv_rows(const double* k, const double* v, const double* w, const double* u,
                    const double* state_in, double* state_out, double* wkv,
                    const int32_t* cu, int B, long C)
{
    if (!k || !v || !w || !u || !state_out || !wkv || !cu || B < 0 || C < 0) return ORACLE_BAD_ARG;
    long items = (long)B * C;
#pragma omp parallel for schedule(static)
    for (long it = 0; it < items; ++it) {
        const long n = it / C, c = it % C;
        double num = 0.0, den = 0.0, mx = -1e38;
        if (state_in) {
            num = state_in[(n * 3 + 0) * C + c];
            den = state_in[(n * 3 + 1) * C + c];
            mx = state_in[(n * 3 + 2) * C + c];
        }
        for (long t = cu[n]; t < cu[n + 1]; ++t) {
            const double kt = k[t * C + c], vt = v[t * C + c];
            /* output: A_{t-1} and the bonus term */
            double ww = u[c] + kt;
            double p = mx > ww ? mx : ww;
            double e1 = exp(mx - p), e2 = exp(ww - p);
            wkv[t * C + c] = (e1 * num + e2 * vt) / (e1 * den + e2);
            /* state: decay, then add row t */
            ww = mx + w[c];
            p = ww > kt ? ww : kt;
            e1 = exp(ww - p);
            e2 = exp(kt - p);
            num = e1 * num + e2 * vt;
            den = e1 * den + e2;
            mx = p;
        }
        state_out[(n * 3 + 0) * C + c] = num;
        state_out[(n * 3 + 1) * C + c] = den;
        state_out[(n * 3 + 2) * C + c] = mx;
    }
    return ORACLE_OK;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
