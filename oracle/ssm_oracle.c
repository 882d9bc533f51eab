/*
 * Test infrastructure: the fp64 CPU oracle for the selective-scan and SSD forward passes.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may call it;
 * the product library never links or loads it.
 *
 * Plain, slow, sequential recurrences in double precision, one (batch, channel) or
 * (batch, head) sequence after another, with OpenMP only across those independent
 * sequences. No blocking, chunking or reordering of the time loop.
 *
 * Sources (pages on the selective state space model):
 *  - "Mamba/SSM complete guide" (youngju.dev), section 5 "Mamba", listing `selective_scan`
 *    in "Mambaの完全な実装": discretise with exp(delta*A) and delta*B*u, run the loop
 *    x = deltaA*x + deltaB_u, read out y = x.C, then add u*D; the block gates the result
 *    with silu(z) afterwards (MambaBlock.forward, "ゲーティング").
 *  - "論文解説: Mamba — 選択的状態空間モデル…" (0h-n0.github.io), "選択機構"
 *    (softplus(z) = log(1 + e^z) makes delta positive) and "Hardware-Aware Parallel Scan"
 *    (the same recurrence, state in zeros at t = 0).
 *  - "State Space Model / Mamba" (disassemble-channel.com), "Zero-Order Hold" and
 *    `discretize_zoh`: for diagonal A the exact ZOH input matrix is (1/a)(exp(a*delta)-1)*B;
 *    "Mamba風の選択的SSMの実装" uses the simplified B_bar = delta*B.
 *  - "Mamba-2 / Structured State Space Duality" (abeam), "基本アイデア": h_t = A_t h_{t-1}
 *    + B_t x_t, y_t = C_t h_t with a scalar A per head; "Mamba/SSM complete guide" section 6
 *    "SSD演算の概念" gives the same recurrence, and `Mamba2Block` a scalar A per head.
 *
 * Readings where the pages are silent or disagree (each is listed in the design notes):
 *  - B_bar = delta*B (every selective listing) unless `zoh` asks for the exact ZOH form.
 *  - y_t reads the state after x_t has entered it (y[0] = C.B_bar.u[0]).
 *  - softplus is applied to delta + bias when delta_softplus != 0.
 *  - D and z are optional; the gate multiplies after the D skip.
 *  - The initial state is zero unless h0 is given.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(v) = log(1 + e^v), evaluated as max(v, 0) + log1p(e^-|v|) so it neither
 * overflows for large v nor loses the small result for very negative v. */
static double softplus_f64(double v) {
    return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
}

static double silu_f64(double v) { return v / (1.0 + exp(-v)); }

/*
 * Mamba-1 selective scan, fp64. All arrays are dense, C-contiguous, fp64:
 *   x, delta, z, y : (batch, seqlen, dim)
 *   B, C           : (batch, seqlen, dstate)   shared by all channels
 *   A              : (dim, dstate)
 *   Dskip, delta_bias : (dim)                  optional (NULL)
 *   h0, h_last     : (batch, dim, dstate)      optional (NULL)
 * zoh     : 0 -> B_bar x = delta*B*x; 1 -> B_bar x = expm1(delta*a)/a * B * x (a != 0),
 *           delta*B*x where a == 0 (the limit).
 * reverse : 0 -> t runs 0..L-1; 1 -> t runs L-1..0 (h_last is the state after t = 0).
 * Returns 0, or -1 on a bad size.
 */
int oracle_ssm_scan_f64(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate,
                        const double* x, const double* delta, const double* A,
                        const double* B, const double* C, const double* Dskip,
                        const double* z, const double* delta_bias, int delta_softplus,
                        const double* h0, int zoh, int reverse,
                        double* y, double* h_last, int nthreads) {
    if (batch < 0 || seqlen < 0 || dim < 0 || dstate < 1 || dstate > 4096) return -1;
    if (nthreads < 1) nthreads = 1;
    const int64_t nchan = batch * dim;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t bd = 0; bd < nchan; ++bd) {
        const int64_t b = bd / dim, d = bd % dim;
        double h[4096];
        for (int64_t n = 0; n < dstate; ++n)
            h[n] = h0 ? h0[(b * dim + d) * dstate + n] : 0.0;
        for (int64_t step = 0; step < seqlen; ++step) {
            const int64_t t = reverse ? seqlen - 1 - step : step;
            const int64_t i = (b * seqlen + t) * dim + d;   /* (b, t, d) */
            const int64_t r = (b * seqlen + t) * dstate;    /* row of B, C */
            double dt = delta[i] + (delta_bias ? delta_bias[d] : 0.0);
            if (delta_softplus) dt = softplus_f64(dt);
            const double u = x[i];
            double acc = 0.0;
            for (int64_t n = 0; n < dstate; ++n) {
                const double a = A[d * dstate + n];
                const double abar = exp(dt * a);
                double bx;
                if (zoh && a != 0.0)
                    bx = expm1(dt * a) / a * B[r + n] * u;
                else
                    bx = dt * B[r + n] * u;
                h[n] = abar * h[n] + bx;
                acc += C[r + n] * h[n];
            }
            double out = acc;
            if (Dskip) out += Dskip[d] * u;
            if (z) out *= silu_f64(z[i]);
            y[i] = out;
        }
        if (h_last)
            for (int64_t n = 0; n < dstate; ++n) h_last[(b * dim + d) * dstate + n] = h[n];
    }
    return 0;
}

/*
 * Mamba-2 (SSD) recurrence with a scalar A per head, fp64, sequential in t.
 *   x, z, y        : (batch, seqlen, nheads, headdim)
 *   delta          : (batch, seqlen, nheads)
 *   A, Dskip, delta_bias : (nheads)            Dskip, delta_bias optional
 *   B, C           : (batch, seqlen, ngroups, dstate); head h reads group h / (nheads/ngroups)
 *   h0, h_last     : (batch, nheads, dstate, headdim)   optional
 * Per step: dt = softplus(delta + bias); S = exp(dt*A_h) S + dt * B_t (x) x_t;
 * y_t[p] = sum_n C_t[n] S[n][p] (+ D_h x_t[p]) (* silu(z_t[p])).
 * Returns 0, -1 on a bad size, -2 if a state buffer could not be allocated.
 */
int oracle_ssd_scan_f64(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                        int64_t dstate, int64_t ngroups,
                        const double* x, const double* delta, const double* A,
                        const double* B, const double* C, const double* Dskip,
                        const double* z, const double* delta_bias, int delta_softplus,
                        const double* h0, double* y, double* h_last, int nthreads) {
    if (batch < 0 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1)
        return -1;
    if (nheads % ngroups != 0) return -1;
    if (nthreads < 1) nthreads = 1;
    const int64_t heads_per_group = nheads / ngroups;
    const int64_t nbh = batch * nheads;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
    for (int64_t bh = 0; bh < nbh; ++bh) {
        const int64_t b = bh / nheads, hh = bh % nheads, g = hh / heads_per_group;
        const int64_t sz = dstate * headdim;
        double* S = (double*)malloc((size_t)sz * sizeof(double));
        if (!S) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        for (int64_t k = 0; k < sz; ++k)
            S[k] = h0 ? h0[(b * nheads + hh) * sz + k] : 0.0;
        for (int64_t t = 0; t < seqlen; ++t) {
            double dt = delta[(b * seqlen + t) * nheads + hh] + (delta_bias ? delta_bias[hh] : 0.0);
            if (delta_softplus) dt = softplus_f64(dt);
            const double abar = exp(dt * A[hh]);
            const double* xt = x + ((b * seqlen + t) * nheads + hh) * headdim;
            const double* Bt = B + ((b * seqlen + t) * ngroups + g) * dstate;
            const double* Ct = C + ((b * seqlen + t) * ngroups + g) * dstate;
            for (int64_t n = 0; n < dstate; ++n) {
                const double bn = dt * Bt[n];
                double* Sn = S + n * headdim;
                for (int64_t p = 0; p < headdim; ++p) Sn[p] = abar * Sn[p] + bn * xt[p];
            }
            double* yt = y + ((b * seqlen + t) * nheads + hh) * headdim;
            const double* zt = z ? z + ((b * seqlen + t) * nheads + hh) * headdim : NULL;
            for (int64_t p = 0; p < headdim; ++p) {
                double acc = 0.0;
                for (int64_t n = 0; n < dstate; ++n) acc += Ct[n] * S[n * headdim + p];
                if (Dskip) acc += Dskip[hh] * xt[p];
                if (zt) acc *= silu_f64(zt[p]);
                yt[p] = acc;
            }
        }
        if (h_last)
            for (int64_t k = 0; k < sz; ++k) h_last[(b * nheads + hh) * sz + k] = S[k];
        free(S);
    }
    return failed ? -2 : 0;
}

/* Threads OpenMP would use by default (for reporting the CPU baseline's core count). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
