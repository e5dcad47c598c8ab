/*
 * Oracle: channelwise CG tensor product and message-passing convolution, forward and
 * backward, in plain float64 loops.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline may load this library; the product path never does.
 *
 * Definitions ("e3j: An efficient and open-source backend for Euclidean equivariant
 * operations on GPU and TPU", App. E.1):
 *   Eq. (10)-(11), tensor product with per-path, per-channel weights:
 *     z[r, zoff_p + m3, q] = sum_p sum_{m1,m2} C_p[m1,m2,m3] x[r, xoff_p + m1, q]
 *                                             y[r, yoff_p + m2] w[r, p, q]
 *   Eq. (12)-(13), convolution over a receiver-sorted CSR edge list:
 *     m[b] = scale * sum_{e in [ptr[b], ptr[b+1])} TP(x[snd[e]], y[e], w[e])
 *   Eq. (15)-(16), the adjoints (exact partial derivatives of the trilinear form):
 *     dx = sum C y w dz,  dy = sum_q C x w dz,  dw = sum_{m1,m2,m3} C x y dz
 *     (conv: dz = scale * dm[receiver], dx scattered to the sender).
 * y carries no channel axis and dy is summed over channels (App. E.3, Alg. 2-3).
 *
 * Path description (per path p, 7 ints): xoff, yoff, zoff, n1, n2, n3, cg offset, where
 * n_k = 2 l_k + 1 and the dense block C_p[m1][m2][m3] starts at cg[cg offset].
 * Every loop follows the definition directly: no blocking, fusion or reordering; zero
 * coefficients are skipped. Rows / receivers / edges / senders are independent and are
 * split over OpenMP threads; inside one output element the sum order is the definition's.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PI(p, k) pinfo[(p) * 7 + (k)]

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* z[R, D, Nq] */
void orc_tp_forward(int64_t R, int d1, int d2, int D, int P, int Nq, const int *pinfo,
                    const double *cg, const double *x, const double *y, const double *w,
                    double *z) {
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; ++r) {
        double *zr = z + r * D * Nq;
        memset(zr, 0, sizeof(double) * D * Nq);
        for (int p = 0; p < P; ++p) {
            const int xo = PI(p, 0), yo = PI(p, 1), zo = PI(p, 2);
            const int n1 = PI(p, 3), n2 = PI(p, 4), n3 = PI(p, 5);
            const double *C = cg + PI(p, 6);
            for (int m3 = 0; m3 < n3; ++m3)
                for (int m1 = 0; m1 < n1; ++m1)
                    for (int m2 = 0; m2 < n2; ++m2) {
                        const double c = C[(m1 * n2 + m2) * n3 + m3];
                        if (c == 0.0) continue;
                        const double yv = y[r * d2 + yo + m2];
                        for (int q = 0; q < Nq; ++q)
                            zr[(zo + m3) * Nq + q] += c * x[(r * d1 + xo + m1) * Nq + q] * yv *
                                                      w[(r * P + p) * Nq + q];
                    }
        }
    }
}

/* dx[R,d1,Nq], dy[R,d2], dw[R,P,Nq] from dz[R,D,Nq] */
void orc_tp_backward(int64_t R, int d1, int d2, int D, int P, int Nq, const int *pinfo,
                     const double *cg, const double *x, const double *y, const double *w,
                     const double *dz, double *dx, double *dy, double *dw) {
    int64_t r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < R; ++r) {
        memset(dx + r * d1 * Nq, 0, sizeof(double) * d1 * Nq);
        memset(dy + r * d2, 0, sizeof(double) * d2);
        memset(dw + r * P * Nq, 0, sizeof(double) * P * Nq);
        for (int p = 0; p < P; ++p) {
            const int xo = PI(p, 0), yo = PI(p, 1), zo = PI(p, 2);
            const int n1 = PI(p, 3), n2 = PI(p, 4), n3 = PI(p, 5);
            const double *C = cg + PI(p, 6);
            for (int m3 = 0; m3 < n3; ++m3)
                for (int m1 = 0; m1 < n1; ++m1)
                    for (int m2 = 0; m2 < n2; ++m2) {
                        const double c = C[(m1 * n2 + m2) * n3 + m3];
                        if (c == 0.0) continue;
                        const double yv = y[r * d2 + yo + m2];
                        for (int q = 0; q < Nq; ++q) {
                            const double xv = x[(r * d1 + xo + m1) * Nq + q];
                            const double wv = w[(r * P + p) * Nq + q];
                            const double g = dz[(r * D + zo + m3) * Nq + q];
                            dx[(r * d1 + xo + m1) * Nq + q] += c * yv * wv * g;
                            dy[r * d2 + yo + m2] += c * xv * wv * g;
                            dw[(r * P + p) * Nq + q] += c * xv * yv * g;
                        }
                    }
        }
    }
}

/* m[n_out, D, Nq]; receiver j of the output owns edges [ptr[j], ptr[j+1]) of the edge
 * arrays snd / y / w (which hold only the edges of the requested receivers). */
void orc_conv_forward(int64_t n_out, const int64_t *ptr, const int32_t *snd, int d1, int d2,
                      int D, int P, int Nq, const int *pinfo, const double *cg,
                      const double *x, const double *y, const double *w, double scale,
                      double *m) {
    int64_t j;
#pragma omp parallel for schedule(dynamic, 16)
    for (j = 0; j < n_out; ++j) {
        double *mj = m + j * D * Nq;
        memset(mj, 0, sizeof(double) * D * Nq);
        for (int64_t e = ptr[j]; e < ptr[j + 1]; ++e) {
            const int64_t a = snd[e];
            for (int p = 0; p < P; ++p) {
                const int xo = PI(p, 0), yo = PI(p, 1), zo = PI(p, 2);
                const int n1 = PI(p, 3), n2 = PI(p, 4), n3 = PI(p, 5);
                const double *C = cg + PI(p, 6);
                for (int m3 = 0; m3 < n3; ++m3)
                    for (int m1 = 0; m1 < n1; ++m1)
                        for (int m2 = 0; m2 < n2; ++m2) {
                            const double c = C[(m1 * n2 + m2) * n3 + m3];
                            if (c == 0.0) continue;
                            const double yv = y[e * d2 + yo + m2];
                            for (int q = 0; q < Nq; ++q)
                                mj[(zo + m3) * Nq + q] += c * x[(a * d1 + xo + m1) * Nq + q] *
                                                          yv * w[(e * P + p) * Nq + q];
                        }
            }
        }
        for (int k = 0; k < D * Nq; ++k) mj[k] *= scale;
    }
}

/* Edge-local cotangents of the convolution for E_sel edges: dy[e,d2], dw[e,P,Nq].
 * snd[e] indexes x, dmrow[e] indexes dm (the receiver's row). */
void orc_conv_backward_edges(int64_t n_e, const int32_t *snd, const int32_t *dmrow, int d1,
                             int d2, int D, int P, int Nq, const int *pinfo, const double *cg,
                             const double *x, const double *y, const double *w,
                             const double *dm, double scale, double *dy, double *dw) {
    int64_t e;
#pragma omp parallel for schedule(static)
    for (e = 0; e < n_e; ++e) {
        const int64_t a = snd[e], b = dmrow[e];
        memset(dy + e * d2, 0, sizeof(double) * d2);
        memset(dw + e * P * Nq, 0, sizeof(double) * P * Nq);
        for (int p = 0; p < P; ++p) {
            const int xo = PI(p, 0), yo = PI(p, 1), zo = PI(p, 2);
            const int n1 = PI(p, 3), n2 = PI(p, 4), n3 = PI(p, 5);
            const double *C = cg + PI(p, 6);
            for (int m3 = 0; m3 < n3; ++m3)
                for (int m1 = 0; m1 < n1; ++m1)
                    for (int m2 = 0; m2 < n2; ++m2) {
                        const double c = C[(m1 * n2 + m2) * n3 + m3];
                        if (c == 0.0) continue;
                        const double yv = y[e * d2 + yo + m2];
                        for (int q = 0; q < Nq; ++q) {
                            const double xv = x[(a * d1 + xo + m1) * Nq + q];
                            const double wv = w[(e * P + p) * Nq + q];
                            const double g = scale * dm[(b * D + zo + m3) * Nq + q];
                            dy[e * d2 + yo + m2] += c * xv * wv * g;
                            dw[(e * P + p) * Nq + q] += c * xv * yv * g;
                        }
                    }
        }
    }
}

/* dx[n_out, d1, Nq]: sender j of the output owns edges [ptr[j], ptr[j+1]) of the edge
 * arrays dmrow / y / w (the edges whose sender is that node). */
void orc_conv_backward_dx(int64_t n_out, const int64_t *ptr, const int32_t *dmrow, int d1,
                          int d2, int D, int P, int Nq, const int *pinfo, const double *cg,
                          const double *y, const double *w, const double *dm, double scale,
                          double *dx) {
    int64_t j;
#pragma omp parallel for schedule(dynamic, 16)
    for (j = 0; j < n_out; ++j) {
        double *dxj = dx + j * d1 * Nq;
        memset(dxj, 0, sizeof(double) * d1 * Nq);
        for (int64_t e = ptr[j]; e < ptr[j + 1]; ++e) {
            const int64_t b = dmrow[e];
            for (int p = 0; p < P; ++p) {
                const int xo = PI(p, 0), yo = PI(p, 1), zo = PI(p, 2);
                const int n1 = PI(p, 3), n2 = PI(p, 4), n3 = PI(p, 5);
                const double *C = cg + PI(p, 6);
                for (int m3 = 0; m3 < n3; ++m3)
                    for (int m1 = 0; m1 < n1; ++m1)
                        for (int m2 = 0; m2 < n2; ++m2) {
                            const double c = C[(m1 * n2 + m2) * n3 + m3];
                            if (c == 0.0) continue;
                            const double yv = y[e * d2 + yo + m2];
                            for (int q = 0; q < Nq; ++q)
                                dxj[(xo + m1) * Nq + q] += c * yv * w[(e * P + p) * Nq + q] *
                                                           scale * dm[(b * D + zo + m3) * Nq + q];
                        }
            }
        }
    }
}
