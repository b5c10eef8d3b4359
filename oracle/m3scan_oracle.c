/*
 * m3scan oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded float64 CPU statement of the Mamba-1
 * selective-scan layer core, forward and backward.  Only the tests, the
 * package smoke check and the benchmark's CPU-baseline leg may load this
 * file; the product path never does.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it follows (the mamba-rs docs.rs source pages):
 *  - mamba-rs 0.3.1, src/mamba_ssm/gpu/forward_mixed.rs, the per-layer loop
 *    of gpu_forward_mamba_backbone_mixed: F4a causal depthwise conv1d, SiLU
 *    (the "post-SiLU conv output, SSM input" u), F4c softplus of delta_raw
 *    (dt_proj output plus its bias), F4d the selective scan writing y with
 *    the D skip, F4e gating gated = y * silu(gate).
 *  - the same page, GpuMambaLayerMixedActs: h is f32 state over d_state
 *    lanes per channel; da_exp = exp(delta * A).
 *  - mamba-rs 0.7.3, src/mamba_ssm/gpu/trainer.rs, recompute_a_neg_all:
 *    A = -exp(a_log); reset_state: recurrent state starts at zero.
 *  - the same forward page, GpuMambaMixedTrainScratch: the backward
 *    produces d_delta, d_u, d_B, d_C (reduced over d_inner), d_D,
 *    d_a_log, softplus backward and conv1d backward (d_x, weight, bias).
 *
 * The backward is the exact reverse-mode derivative of
 *     L = sum_{b,t,d} gated[b,t,d] * d_gated[b,t,d]
 * written out step by step (no autograd, no fusion).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - conv taps: c[t] = conv_b + sum_k w[k] * x[t-(W-1)+k] (w[W-1] multiplies
 *    the current token); x before t=0 is the carried conv state, zero when
 *    none is given.
 *  - the recurrent state before step 0 is the carried SSM state, zero when
 *    none is given (the trainer's reset_state).
 *  - the input term of the recurrence is delta*B*u (Euler for B, zero-order
 *    hold for A); y_t reads the state after the t-th update.
 *  - softplus(v) = log(1 + e^v) exactly, no threshold.
 *  - dt_bias is added to delta_raw inside the softplus.
 *  - du is dL/du through the D skip and the recurrence only.
 *
 * Layouts (row-major, channel fastest): x, delta_raw, z, d_gated and every
 * per-element output are [B, T, D]; Bm, Cm, dB, dC are [B, T, N]; conv_w
 * and d_conv_w are [D, W]; a_log and d_a_log are [D, N]; conv_b, dt_bias,
 * Dp and their grads are [D].  ckpt is [B, nc, N, D] with nc = ceil(T/K):
 * ckpt[b, c, :, d] is the state before step c*K.
 *
 * Carried state (all nullable; NULL inputs mean zero, NULL outputs are not
 * written).  ssm_state [B, N, D] is the state before step 0 (h_{-1});
 * conv_state [B, W-1, D] holds the conv inputs of the W-1 steps before step
 * 0, oldest first (row r is step r-(W-1)).  ssm_state_out and conv_state_out
 * have the same layouts and hold h_{T-1} and the inputs of steps T-W+1..T-1,
 * so that a sequence cut in two windows and run window by window, each
 * window starting from the previous one's outputs, gives the same results as
 * one run over the whole sequence.
 *
 * chan_mask (nullable, [D] bytes): when given, only channels with a nonzero
 * mask byte are computed; the others keep whatever the caller put in the
 * outputs, and contribute nothing to dB and dC.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define IDX3(b, t, d, T, D) (((int64_t)(b) * (T) + (t)) * (D) + (d))

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* log(1 + e^v) without overflow: max(v, 0) + log1p(e^-|v|) */
static double softplus(double v) {
    return (v > 0.0 ? v : 0.0) + log1p(exp(-fabs(v)));
}

static double silu(double v) { return v * sigmoid(v); }

/* d/dv of v * sigmoid(v) */
static double silu_grad(double v) {
    double s = sigmoid(v);
    return s + v * s * (1.0 - s);
}

static int channel_on(const uint8_t* mask, int64_t d) {
    return mask == NULL || mask[d] != 0;
}

/* The conv input of channel d at step s >= -(W-1): x for s >= 0, else the
   carried conv state (row s + W - 1), zero when there is none. */
static double x_at(const double* x, const double* conv_state, int64_t b,
                   int64_t s, int64_t d, int64_t T, int64_t D, int64_t W) {
    if (s >= 0) return x[IDX3(b, s, d, T, D)];
    if (conv_state == NULL) return 0.0;
    return conv_state[IDX3(b, s + (W - 1), d, W - 1, D)];
}

/* Per-channel forward quantities along time (conv output c, u, delta). */
static void channel_inputs(int64_t b, int64_t d, int64_t T, int64_t D, int64_t W,
                           const double* x, const double* conv_state,
                           const double* delta_raw,
                           const double* conv_w, const double* conv_b,
                           const double* dt_bias, double* c, double* u,
                           double* delta) {
    for (int64_t t = 0; t < T; ++t) {
        double acc = conv_b[d];
        for (int64_t k = 0; k < W; ++k) {
            int64_t s = t - (W - 1) + k;
            acc += conv_w[d * W + k] * x_at(x, conv_state, b, s, d, T, D, W);
        }
        c[t] = acc;
        u[t] = silu(acc);
        delta[t] = softplus(delta_raw[IDX3(b, t, d, T, D)] + dt_bias[d]);
    }
}

/* One step of the recurrence for every lane n:
 *   h_t[n] = exp(delta_t * A[n]) * h_{t-1}[n] + delta_t * B_t[n] * u_t   */
static void scan_step(int64_t N, const double* A, double delta, double u,
                      const double* Bt, const double* hprev, double* hnext) {
    for (int64_t n = 0; n < N; ++n)
        hnext[n] = exp(delta * A[n]) * hprev[n] + delta * Bt[n] * u;
}

/* y_t = sum_n C_t[n] h_t[n] + D u_t */
static double scan_output(int64_t N, const double* Ct, const double* h,
                          double Dd, double u) {
    double y = 0.0;
    for (int64_t n = 0; n < N; ++n) y += Ct[n] * h[n];
    return y + Dd * u;
}

/*
 * Forward.  gated, y, u_out, delta_out: [B,T,D] (y, u_out, delta_out and
 * ckpt nullable).  K is the checkpoint interval used for ckpt (ignored when
 * ckpt is NULL).  ssm_state, conv_state, ssm_state_out, conv_state_out: the
 * carried state described above (nullable).  Returns 0, or -1 on an
 * allocation failure.
 */
int m3o_forward(int64_t B, int64_t T, int64_t D, int64_t N, int64_t W,
                const double* x, const double* delta_raw, const double* z,
                const double* Bm, const double* Cm, const double* conv_w,
                const double* conv_b, const double* dt_bias,
                const double* a_log, const double* Dp,
                const uint8_t* chan_mask, double* gated, double* y_out,
                double* u_out, double* delta_out, double* ckpt, int64_t K,
                const double* ssm_state, const double* conv_state,
                double* ssm_state_out, double* conv_state_out) {
    double* c = malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double* u = malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double* delta = malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double* A = malloc(sizeof(double) * (size_t)N);
    double* h = malloc(sizeof(double) * (size_t)N);
    double* hn = malloc(sizeof(double) * (size_t)N);
    if (!c || !u || !delta || !A || !h || !hn) {
        free(c); free(u); free(delta); free(A); free(h); free(hn);
        return -1;
    }
    int64_t nc = (ckpt && K > 0) ? (T + K - 1) / K : 0;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            if (!channel_on(chan_mask, d)) continue;
            for (int64_t n = 0; n < N; ++n) A[n] = -exp(a_log[d * N + n]);
            channel_inputs(b, d, T, D, W, x, conv_state, delta_raw, conv_w,
                           conv_b, dt_bias, c, u, delta);
            for (int64_t n = 0; n < N; ++n)
                h[n] = ssm_state ? ssm_state[(b * N + n) * D + d] : 0.0;
            for (int64_t t = 0; t < T; ++t) {
                if (nc > 0 && t % K == 0) {
                    int64_t ci = t / K;
                    for (int64_t n = 0; n < N; ++n)
                        ckpt[((b * nc + ci) * N + n) * D + d] = h[n];
                }
                const double* Bt = Bm + (b * T + t) * N;
                const double* Ct = Cm + (b * T + t) * N;
                scan_step(N, A, delta[t], u[t], Bt, h, hn);
                memcpy(h, hn, sizeof(double) * (size_t)N);
                double yt = scan_output(N, Ct, h, Dp[d], u[t]);
                int64_t i = IDX3(b, t, d, T, D);
                gated[i] = yt * silu(z[i]);
                if (y_out) y_out[i] = yt;
                if (u_out) u_out[i] = u[t];
                if (delta_out) delta_out[i] = delta[t];
            }
            if (ssm_state_out)
                for (int64_t n = 0; n < N; ++n)
                    ssm_state_out[(b * N + n) * D + d] = h[n];
            if (conv_state_out)
                for (int64_t r = 0; r < W - 1; ++r)
                    conv_state_out[IDX3(b, r, d, W - 1, D)] =
                        x_at(x, conv_state, b, T - (W - 1) + r, d, T, D, W);
        }
    }
    free(c); free(u); free(delta); free(A); free(h); free(hn);
    return 0;
}

/*
 * Backward of L = sum gated * d_gated.
 *
 * K == 0: h is kept for every step (sequential mode).
 * K  > 0: only the state at each chunk start is kept during the forward
 *         sweep; the reverse sweep recomputes the states of one chunk at a
 *         time from its start state (chunked mode).  In exact arithmetic the
 *         two modes are the same computation.
 *
 * Per-element outputs d_x, d_delta_raw, dz, du: [B,T,D] (du nullable).
 * dB, dC: [B,T,N], accumulated into (the caller zeroes them).
 * Parameter grads d_conv_w [D,W], d_conv_b [D], d_dt_bias [D], d_a_log
 * [D,N], dD [D]: overwritten for every computed channel.
 *
 * With carried state the loss gains the terms of the state outputs,
 *     L += sum ssm_state_out * d_ssm_state_out
 *        + sum conv_state_out * d_conv_state_out,
 * (d_ssm_state_out, d_conv_state_out nullable = zero), and d_ssm_state,
 * d_conv_state (nullable) receive dL/d ssm_state and dL/d conv_state.
 *
 * d_u_extra ([B,T,D], nullable = zero) is a gradient reaching u from
 * outside the layer core -- in the mamba-rs backward the x_proj GEMM's
 * input gradient, which the page adds into d_u before the SiLU and conv1d
 * backward -- so the loss gains sum u * d_u_extra.  It changes d_x,
 * d_conv_w, d_conv_b and d_conv_state; du_out stays dL/du through the D
 * skip and the recurrence only.
 */
int m3o_backward(int64_t B, int64_t T, int64_t D, int64_t N, int64_t W,
                 const double* x, const double* delta_raw, const double* z,
                 const double* Bm, const double* Cm, const double* conv_w,
                 const double* conv_b, const double* dt_bias,
                 const double* a_log, const double* Dp, const double* d_gated,
                 const uint8_t* chan_mask, int64_t K, double* d_x,
                 double* d_delta_raw, double* dz, double* du_out, double* dB,
                 double* dC, double* d_conv_w, double* d_conv_b,
                 double* d_dt_bias, double* d_a_log, double* dD,
                 const double* ssm_state, const double* conv_state,
                 const double* d_ssm_state_out, const double* d_conv_state_out,
                 double* d_ssm_state, double* d_conv_state, const double* d_u_extra) {
    int64_t Tm = T > 0 ? T : 1;
    int64_t span = (K > 0) ? K : Tm;         /* states held at once */
    int64_t nc = (K > 0) ? (T + K - 1) / K : 1;
    double* c = malloc(sizeof(double) * (size_t)Tm);
    double* u = malloc(sizeof(double) * (size_t)Tm);
    double* delta = malloc(sizeof(double) * (size_t)Tm);
    double* dc = malloc(sizeof(double) * (size_t)Tm);
    double* A = malloc(sizeof(double) * (size_t)N);
    double* starts = malloc(sizeof(double) * (size_t)(nc * N));
    /* hs[j] = state after step t0+j-1 within the current span; hs[0] is the
       state before the span's first step. */
    double* hs = malloc(sizeof(double) * (size_t)((span + 1) * N));
    double* dh_next = malloc(sizeof(double) * (size_t)N);
    double* dA_next = malloc(sizeof(double) * (size_t)N);
    double* dAp = malloc(sizeof(double) * (size_t)N);
    double* h = malloc(sizeof(double) * (size_t)N);
    double* hn = malloc(sizeof(double) * (size_t)N);
    int ok = c && u && delta && dc && A && starts && hs && dh_next && dA_next &&
             dAp && h && hn;
    if (!ok) goto done;

    for (int64_t b = 0; b < B; ++b) {
        for (int64_t d = 0; d < D; ++d) {
            if (!channel_on(chan_mask, d)) continue;
            for (int64_t n = 0; n < N; ++n) A[n] = -exp(a_log[d * N + n]);
            channel_inputs(b, d, T, D, W, x, conv_state, delta_raw, conv_w,
                           conv_b, dt_bias, c, u, delta);

            /* forward sweep: keep the state before each span */
            for (int64_t n = 0; n < N; ++n)
                h[n] = ssm_state ? ssm_state[(b * N + n) * D + d] : 0.0;
            for (int64_t t = 0; t < T; ++t) {
                if (t % span == 0)
                    memcpy(starts + (t / span) * N, h, sizeof(double) * (size_t)N);
                scan_step(N, A, delta[t], u[t], Bm + (b * T + t) * N, h, hn);
                memcpy(h, hn, sizeof(double) * (size_t)N);
            }

            double dD_acc = 0.0, ddtb_acc = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                /* dA_next[n] * dh_next[n] is the gradient reaching h_t from
                   later steps; after the last step that is the upstream
                   gradient of the state output (zero when none) */
                dh_next[n] = d_ssm_state_out ? d_ssm_state_out[(b * N + n) * D + d] : 0.0;
                dA_next[n] = 1.0;
                dAp[n] = 0.0;      /* dL/dA[n] */
            }
            for (int64_t s = (T + span - 1) / span - 1; s >= 0; --s) {
                int64_t t0 = s * span;
                int64_t t1 = t0 + span < T ? t0 + span : T;
                /* recompute the span's states from its start state */
                memcpy(hs, starts + s * N, sizeof(double) * (size_t)N);
                for (int64_t t = t0; t < t1; ++t)
                    scan_step(N, A, delta[t], u[t], Bm + (b * T + t) * N,
                              hs + (t - t0) * N, hs + (t - t0 + 1) * N);
                /* reverse sweep over the span */
                for (int64_t t = t1 - 1; t >= t0; --t) {
                    int64_t i = IDX3(b, t, d, T, D);
                    const double* Bt = Bm + (b * T + t) * N;
                    const double* Ct = Cm + (b * T + t) * N;
                    const double* h_t = hs + (t - t0 + 1) * N;
                    const double* h_p = hs + (t - t0) * N;
                    double yt = scan_output(N, Ct, h_t, Dp[d], u[t]);
                    double g = d_gated[i];
                    /* gated = y * silu(z) */
                    double dy = g * silu(z[i]);
                    dz[i] = g * yt * silu_grad(z[i]);
                    /* y = C.h + D u */
                    double du = dy * Dp[d];
                    dD_acc += dy * u[t];
                    double ddelta = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        double dA_t = exp(delta[t] * A[n]);
                        /* h_{t+1} = dA_{t+1} h_t + ..., y_t = C_t.h_t + ... */
                        double dh = dy * Ct[n] + dA_next[n] * dh_next[n];
                        int64_t bn = (b * T + t) * N + n;
                        dC[bn] += dy * h_t[n];
                        dB[bn] += dh * delta[t] * u[t];
                        du += dh * delta[t] * Bt[n];
                        ddelta += dh * (Bt[n] * u[t] + A[n] * dA_t * h_p[n]);
                        dAp[n] += dh * delta[t] * dA_t * h_p[n];
                        dh_next[n] = dh;
                        dA_next[n] = dA_t;
                    }
                    if (du_out) du_out[i] = du;
                    /* delta = softplus(delta_raw + dt_bias) */
                    double ddr = ddelta * sigmoid(delta_raw[i] + dt_bias[d]);
                    d_delta_raw[i] = ddr;
                    ddtb_acc += ddr;
                    /* u = silu(c); u also feeds the x_proj path */
                    double du_total = du + (d_u_extra ? d_u_extra[i] : 0.0);
                    dc[t] = du_total * silu_grad(c[t]);
                }
            }

            /* h_{-1} = ssm_state feeds h_0 = exp(delta_0 A) h_{-1} + ... */
            if (d_ssm_state)
                for (int64_t n = 0; n < N; ++n)
                    d_ssm_state[(b * N + n) * D + d] = dA_next[n] * dh_next[n];

            /* conv1d backward: c[t] = conv_b + sum_k w[k] x[t-(W-1)+k] */
            double dcb = 0.0;
            for (int64_t t = 0; t < T; ++t) dcb += dc[t];
            if (b == 0) d_conv_b[d] = 0.0;
            d_conv_b[d] += dcb;
            for (int64_t k = 0; k < W; ++k) {
                double acc = 0.0;
                for (int64_t t = 0; t < T; ++t) {
                    int64_t s2 = t - (W - 1) + k;
                    acc += dc[t] * x_at(x, conv_state, b, s2, d, T, D, W);
                }
                if (b == 0) d_conv_w[d * W + k] = 0.0;
                d_conv_w[d * W + k] += acc;
            }
            /* the conv input at step s2 >= -(W-1) reaches the conv outputs
               of steps s2..s2+W-1 and, for s2 >= T-(W-1), the conv state
               output row s2-(T-(W-1)) */
            for (int64_t s2 = -(W - 1); s2 < T; ++s2) {
                double acc = 0.0;
                for (int64_t k = 0; k < W; ++k) {
                    int64_t t = s2 + (W - 1) - k;
                    if (t >= 0 && t < T) acc += dc[t] * conv_w[d * W + k];
                }
                int64_t r = s2 - (T - (W - 1));
                if (d_conv_state_out && r >= 0)
                    acc += d_conv_state_out[IDX3(b, r, d, W - 1, D)];
                if (s2 >= 0)
                    d_x[IDX3(b, s2, d, T, D)] = acc;
                else if (d_conv_state)
                    d_conv_state[IDX3(b, s2 + (W - 1), d, W - 1, D)] = acc;
            }
            /* A = -exp(a_log): dL/da_log = dL/dA * A */
            for (int64_t n = 0; n < N; ++n) {
                if (b == 0) d_a_log[d * N + n] = 0.0;
                d_a_log[d * N + n] += dAp[n] * A[n];
            }
            if (b == 0) { dD[d] = 0.0; d_dt_bias[d] = 0.0; }
            dD[d] += dD_acc;
            d_dt_bias[d] += ddtb_acc;
        }
    }
    ok = 1;
done:
    free(c); free(u); free(delta); free(dc); free(A); free(starts); free(hs);
    free(dh_next); free(dA_next); free(dAp); free(h); free(hn);
    return ok ? 0 : -1;
}
