/*
 * m3scan oracle, all-core timing driver -- TEST INFRASTRUCTURE ONLY.
 *
 * Not a second statement of the method and not pinned on its own: it
 * compiles the pinned single-threaded oracle (m3scan_oracle.c, included
 * below unchanged) together with one driver function that runs that
 * oracle's forward and backward on every host core at once, each thread on
 * its own block of channels (channels are independent recurrences; only dB
 * and dC are sums over channels).  Each thread accumulates dB and dC into a
 * buffer of its own; the buffers are added in thread order at the end.  The
 * benchmark times it beside the single-threaded oracle as the all-core CPU
 * baseline; the tests compare it with the single-threaded oracle.
 */
#include "m3scan_oracle.c"

#include <omp.h>

/* Forward (gated) and backward (d_x, d_delta_raw, dz, dB, dC and the
 * parameter gradients) of L = sum gated * d_gated, as m3o_forward and
 * m3o_backward give them with no carried state, on `nthreads` OpenMP
 * threads (0 = the OpenMP default).  Outputs as in those functions; dB and
 * dC are overwritten.  *threads_used receives the thread count.  Returns 0,
 * or -1 on an allocation failure. */
int m3o_fwd_bwd_par(int64_t B, int64_t T, int64_t D, int64_t N, int64_t W,
                    const double* x, const double* delta_raw, const double* z,
                    const double* Bm, const double* Cm, const double* conv_w,
                    const double* conv_b, const double* dt_bias,
                    const double* a_log, const double* Dp, const double* d_gated,
                    int nthreads, double* gated, double* d_x, double* d_delta_raw,
                    double* dz, double* dB, double* dC, double* d_conv_w,
                    double* d_conv_b, double* d_dt_bias, double* d_a_log, double* dD,
                    int* threads_used) {
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
    if (nt < 1) nt = 1;
    if (nt > D && D > 0) nt = (int)D;
    const size_t btn = (size_t)(B * T * N);
    double* part = calloc((size_t)nt * 2 * (btn > 0 ? btn : 1), sizeof(double));
    if (!part) return -1;
    int rc = 0;
#pragma omp parallel num_threads(nt) reduction(| : rc)
    {
        const int i = omp_get_thread_num();
        const int n = omp_get_num_threads();
        uint8_t* mask = calloc((size_t)(D > 0 ? D : 1), 1);
        if (!mask) {
            rc |= 1;
        } else {
            /* a contiguous block of channels per thread */
            const int64_t lo = D * i / n, hi = D * (i + 1) / n;
            for (int64_t d = lo; d < hi; ++d) mask[d] = 1;
            double* pb = part + (size_t)i * 2 * btn;
            double* pc = pb + btn;
            rc |= m3o_forward(B, T, D, N, W, x, delta_raw, z, Bm, Cm, conv_w, conv_b,
                              dt_bias, a_log, Dp, mask, gated, NULL, NULL, NULL, NULL, 0,
                              NULL, NULL, NULL, NULL) != 0;
            rc |= m3o_backward(B, T, D, N, W, x, delta_raw, z, Bm, Cm, conv_w, conv_b,
                               dt_bias, a_log, Dp, d_gated, mask, 0, d_x, d_delta_raw, dz,
                               NULL, pb, pc, d_conv_w, d_conv_b, d_dt_bias, d_a_log, dD,
                               NULL, NULL, NULL, NULL, NULL, NULL, NULL) != 0;
            free(mask);
        }
        if (i == 0) *threads_used = n;
    }
    for (size_t k = 0; k < btn; ++k) {
        double sb = 0.0, sc = 0.0;
        for (int i = 0; i < nt; ++i) {
            sb += part[(size_t)i * 2 * btn + k];
            sc += part[(size_t)i * 2 * btn + btn + k];
        }
        dB[k] = sb;
        dC[k] = sc;
    }
    free(part);
    return rc ? -1 : 0;
}
