// Radial edge scalars: the hidden layer of the network that turns an edge length into the
// per-edge, per-path, per-channel weights of the convolution.
//
// "e3j ..." (App. E.1, notation for the edge scalars s) says the weights are usually an MLP
// applied to a radial embedding of the interatomic distance and projected to the paths and
// channels of each edge; App. A.3 ("Linear mixing") names fusing that scalar mixing into
// message passing. The pages fix neither the embedding nor the network. The reading here:
//   b_n(d) = sqrt(2/r_c) sin(n pi d / r_c) / d * u(d / r_c),  n = 1..n_basis   (Bessel basis)
//   u(x)   = 1 - 28 x^6 + 48 x^7 - 21 x^8 for x < 1, else 0  (p = 6 polynomial envelope)
//   h_k    = silu(sum_n b_n W1[n, k])                          (hidden layer, no bias)
//   w[p,q] = sum_k h_k W2[k, p, q]                             (output layer, in the conv)
// The output layer is the large one (H x P x Nq per edge); the radial convolution kernels
// evaluate it per edge from a shared-memory copy of W2, so w never reaches HBM. This file
// produces h[E, H] and, for forces, the gradient of <dh, h> with respect to the edge vectors.
//
// The basis is evaluated in float64 (the argument n pi d / r_c of an fp32 sine carries an
// absolute rounding error of ~1e-6 at n = 8, which would show up in the convolution's fp32
// tolerance): |r|, one sincos of theta = pi |r| / r_c, the Chebyshev recurrence
// s_{n+1} = 2 cos(theta) s_n - s_{n-1} for sin(n theta) and cos(n theta), the envelope. The
// basis values are then rounded once and the hidden layer (a small matrix product and SiLU)
// runs in fp32.
#include "radial.cuh"

namespace e3gb {

namespace {

struct RadialBasis {
    double b[kRadialMaxBasis];    // b_n(d)
    double db[kRadialMaxBasis];   // db_n/dd
    double d;                     // |r|
};

template <int NBC>
__device__ __forceinline__ void radial_basis(double x, double y, double z, int nb_rt, double rc, bool grad,
                                             RadialBasis& o) {
    const int nb = NBC > 0 ? NBC : nb_rt;
    const double d = sqrt(x * x + y * y + z * z);
    o.d = d;
    const double c = sqrt(2.0 / rc);
    const double k1 = 3.14159265358979323846 / rc;
    if (d < 1e-12) {   // the d -> 0 limit: e_n = c n pi / r_c, flat (u(0) = 1, u'(0) = 0)
#pragma unroll
        for (int n = 0; n < nb; ++n) {
            o.b[n] = c * k1 * (n + 1);
            o.db[n] = 0.0;
        }
        return;
    }
    const double xr = d / rc;
    double u = 0.0, du = 0.0;
    if (xr < 1.0) {
        const double x2 = xr * xr, x5 = x2 * x2 * xr, x6 = x5 * xr;
        u = 1.0 + x6 * (-28.0 + xr * (48.0 - 21.0 * xr));
        du = x5 * (-168.0 + xr * (336.0 - 168.0 * xr)) / rc;   // du/dd
    }
    double s1, c1;
    sincos(k1 * d, &s1, &c1);
    double sp = 0.0, sn = s1;   // sin((n-1) theta), sin(n theta)
    double cp = 1.0, cn = c1;   // cos((n-1) theta), cos(n theta)
    const double inv_d = 1.0 / d;
#pragma unroll
    for (int n = 0; n < nb; ++n) {
        const double e = c * sn * inv_d;
        o.b[n] = e * u;
        if (grad) {
            const double de = c * (k1 * (n + 1) * cn * d - sn) * inv_d * inv_d;
            o.db[n] = de * u + e * du;
        }
        const double s2 = 2.0 * c1 * sn - sp, c2 = 2.0 * c1 * cn - cp;
        sp = sn;
        sn = s2;
        cp = cn;
        cn = c2;
    }
}

// NBC, HC > 0: the basis and hidden sizes fixed at compile time (the arrays stay in registers)
template <int NBC, int HC>
__global__ void __launch_bounds__(256) radial_hidden_kernel(int64_t E, const float* __restrict__ vec,
                                                            const float* __restrict__ W1, int nb_rt, int H_rt,
                                                            double rc, float* __restrict__ h) {
    const int nb = NBC > 0 ? NBC : nb_rt, H = HC > 0 ? HC : H_rt;
    __shared__ float w1[kRadialMaxBasis * kRadialMaxHidden];
    for (int i = threadIdx.x; i < nb * H; i += blockDim.x) w1[i] = W1[i];
    __syncthreads();
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < E; e += int64_t(gridDim.x) * blockDim.x) {
        RadialBasis rb;
        radial_basis<NBC>(vec[3 * e], vec[3 * e + 1], vec[3 * e + 2], nb, rc, false, rb);
        float b[kRadialMaxBasis];
#pragma unroll
        for (int n = 0; n < nb; ++n) b[n] = float(rb.b[n]);
#pragma unroll
        for (int k = 0; k < H; ++k) {
            float a = 0.f;
#pragma unroll
            for (int n = 0; n < nb; ++n) a = fmaf(b[n], w1[n * H + k], a);
            h[e * H + k] = a / (1.f + expf(-a));
        }
    }
}

// dvec[e] (+)= (sum_k dh[e,k] silu'(a_k) sum_n b'_n W1[n,k]) r_e / |r_e|; zero for |r_e| < 1e-12
template <int NBC, int HC>
__global__ void __launch_bounds__(256) radial_backward_kernel(int64_t E, const float* __restrict__ vec,
                                                              const float* __restrict__ W1, int nb_rt, int H_rt,
                                                              double rc, const float* __restrict__ dh,
                                                              float* __restrict__ dvec, int accumulate) {
    const int nb = NBC > 0 ? NBC : nb_rt, H = HC > 0 ? HC : H_rt;
    __shared__ float w1[kRadialMaxBasis * kRadialMaxHidden];
    for (int i = threadIdx.x; i < nb * H; i += blockDim.x) w1[i] = W1[i];
    __syncthreads();
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < E; e += int64_t(gridDim.x) * blockDim.x) {
        const float x = vec[3 * e], y = vec[3 * e + 1], z = vec[3 * e + 2];
        RadialBasis rb;
        radial_basis<NBC>(x, y, z, nb, rc, true, rb);
        float b[kRadialMaxBasis], db[kRadialMaxBasis];
#pragma unroll
        for (int n = 0; n < nb; ++n) {
            b[n] = float(rb.b[n]);
            db[n] = float(rb.db[n]);
        }
        float dd = 0.f;   // d <dh, h> / d |r|
#pragma unroll
        for (int k = 0; k < H; ++k) {
            float a = 0.f, da = 0.f;
#pragma unroll
            for (int n = 0; n < nb; ++n) {
                a = fmaf(b[n], w1[n * H + k], a);
                da = fmaf(db[n], w1[n * H + k], da);
            }
            const float s = 1.f / (1.f + expf(-a));
            dd = fmaf(dh[e * H + k] * s * (1.f + a * (1.f - s)), da, dd);
        }
        const float f = rb.d < 1e-12 ? 0.f : float(double(dd) / rb.d);
        const float g[3] = {f * x, f * y, f * z};
        for (int i = 0; i < 3; ++i) dvec[3 * e + i] = accumulate ? dvec[3 * e + i] + g[i] : g[i];
    }
}

inline int blocks_for(int64_t n, int block, int cap) {
    const int64_t g = (n + block - 1) / block;
    return int(g < cap ? (g > 0 ? g : 1) : cap);
}

}  // namespace

cudaError_t radial_hidden(int64_t E, const float* vec, const float* W1, int nb, int H, float rc, float* h,
                          cudaStream_t s) {
    if (E <= 0) return cudaSuccess;
    const int grid = blocks_for(E, 256, 8192);
    if (nb == 8 && H == 8)
        radial_hidden_kernel<8, 8><<<grid, 256, 0, s>>>(E, vec, W1, nb, H, double(rc), h);
    else
        radial_hidden_kernel<0, 0><<<grid, 256, 0, s>>>(E, vec, W1, nb, H, double(rc), h);
    return cudaGetLastError();
}

cudaError_t radial_backward(int64_t E, const float* vec, const float* W1, int nb, int H, float rc, const float* dh,
                            float* dvec, int accumulate, cudaStream_t s) {
    if (E <= 0) return cudaSuccess;
    const int grid = blocks_for(E, 256, 8192);
    if (nb == 8 && H == 8)
        radial_backward_kernel<8, 8><<<grid, 256, 0, s>>>(E, vec, W1, nb, H, double(rc), dh, dvec, accumulate);
    else
        radial_backward_kernel<0, 0><<<grid, 256, 0, s>>>(E, vec, W1, nb, H, double(rc), dh, dvec, accumulate);
    return cudaGetLastError();
}

}  // namespace e3gb
