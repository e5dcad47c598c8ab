// Real spherical harmonics of edge vectors, l <= 3, component normalisation.
//
// "e3j ...", App. A.3 Eq. (4) (Y_l = (Y_lm)_{m=-l..l}, concatenated over l) and App. G.1
// (the degree-l harmonic polynomials). Real basis: m < 0 sin-type, m > 0 cos-type, scaled so
// that sum_m Y_lm(u)^2 = 2l+1 on the unit sphere; l = 1 is sqrt(3) (y, z, x). The
// polynomials are evaluated in homogeneous form at u = v/|v| (u = 0 for |v| < 1e-12).
//
// One thread per edge; the block stages its output rows in shared memory and writes them
// back as contiguous 16-byte vectors, so the [n, (lmax+1)^2] store is fully coalesced.
//
// Backward (the VJP, for forces through the harmonics): with Y_lm(u) = P_lm(u), P_lm the
// degree-l homogeneous polynomial and u = v/|v|, the chain rule and Euler's identity
// (grad P . u = l P) give dY/dv = (grad P(u) - l P(u) u) / |v|, so
//   dvec = (sum_lm dy_lm grad P_lm(u) - (sum_lm l dy_lm Y_lm(u)) u) / |v|   (0 for |v| < 1e-12).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "cg_table.hpp"

namespace e3gb {

namespace {
constexpr int kShBlock = 256;

template <int LMAX>
__device__ __forceinline__ void sh_eval(float x, float y, float z, float* o) {
    constexpr float s3 = float(csqrt(3.0)), s5 = float(csqrt(5.0)), s7 = float(csqrt(7.0));
    constexpr float s15 = float(csqrt(15.0)), s42 = float(csqrt(42.0)), s70 = float(csqrt(70.0));
    constexpr float s105 = float(csqrt(105.0));
    o[0] = 1.f;
    if constexpr (LMAX >= 1) {
        o[1] = s3 * y;
        o[2] = s3 * z;
        o[3] = s3 * x;
    }
    if constexpr (LMAX >= 2) {
        const float xx = x * x, yy = y * y, zz = z * z;
        o[4] = s15 * x * y;
        o[5] = s15 * y * z;
        o[6] = 0.5f * s5 * (2.f * zz - xx - yy);
        o[7] = s15 * x * z;
        o[8] = 0.5f * s15 * (xx - yy);
        if constexpr (LMAX >= 3) {
            o[9] = 0.25f * s70 * y * (3.f * xx - yy);
            o[10] = s105 * x * y * z;
            o[11] = 0.25f * s42 * y * (4.f * zz - xx - yy);
            o[12] = 0.5f * s7 * z * (2.f * zz - 3.f * xx - 3.f * yy);
            o[13] = 0.25f * s42 * x * (4.f * zz - xx - yy);
            o[14] = 0.5f * s105 * z * (xx - yy);
            o[15] = 0.25f * s70 * x * (xx - 3.f * yy);
        }
    }
}

template <class T>
__device__ __forceinline__ T cvt(float v);
template <>
__device__ __forceinline__ float cvt<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <int LMAX, class T>
__global__ void __launch_bounds__(kShBlock) sh_kernel(int64_t n, const float* __restrict__ vec, T* __restrict__ out) {
    constexpr int K = (LMAX + 1) * (LMAX + 1);
    __shared__ __align__(16) T stage[kShBlock * K];
    const int64_t base = int64_t(blockIdx.x) * kShBlock;
    const int64_t e = base + threadIdx.x;
    if (e < n) {
        float v0 = __ldg(vec + 3 * e), v1 = __ldg(vec + 3 * e + 1), v2 = __ldg(vec + 3 * e + 2);
        const float r = sqrtf(v0 * v0 + v1 * v1 + v2 * v2);
        if (r < 1e-12f) {
            v0 = v1 = v2 = 0.f;
        } else {
            v0 = v0 / r; v1 = v1 / r; v2 = v2 / r;
        }
        float o[K];
        sh_eval<LMAX>(v0, v1, v2, o);
#pragma unroll
        for (int k = 0; k < K; ++k) stage[threadIdx.x * K + k] = cvt<T>(o[k]);
    }
    __syncthreads();
    const int64_t rows = (n - base) < kShBlock ? (n - base) : kShBlock;
    const int64_t total = rows * K;                 // elements of this block's output
    T* dst = out + base * K;
    // 16-byte vectors where the row block allows it, scalars for the tail
    constexpr int per16 = 16 / sizeof(T);
    const int64_t nvec = total / per16;
    const bool aligned16 = (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
    if (aligned16) {
        for (int64_t i = threadIdx.x; i < nvec; i += kShBlock)
            reinterpret_cast<uint4*>(dst)[i] = reinterpret_cast<const uint4*>(stage)[i];
        for (int64_t i = nvec * per16 + threadIdx.x; i < total; i += kShBlock) dst[i] = stage[i];
    } else {
        for (int64_t i = threadIdx.x; i < total; i += kShBlock) dst[i] = stage[i];
    }
}

// g += sum_m dy_m grad P_lm(u) and e += sum_m l dy_m Y_lm(u) for degrees 0..LMAX
template <int LMAX>
__device__ __forceinline__ void sh_grad_eval(float x, float y, float z, const float* d, float (&g)[3], float& e) {
    constexpr float s3 = float(csqrt(3.0)), s5 = float(csqrt(5.0)), s7 = float(csqrt(7.0));
    constexpr float s15 = float(csqrt(15.0)), s42 = float(csqrt(42.0)), s70 = float(csqrt(70.0));
    constexpr float s105 = float(csqrt(105.0));
    g[0] = g[1] = g[2] = 0.f;
    e = 0.f;
    if constexpr (LMAX >= 1) {
        // P_1 = sqrt3 (y, z, x)
        g[0] += s3 * d[3];
        g[1] += s3 * d[1];
        g[2] += s3 * d[2];
        e += s3 * (d[1] * y + d[2] * z + d[3] * x);
    }
    if constexpr (LMAX >= 2) {
        const float xx = x * x, yy = y * y, zz = z * z;
        // xy, yz, (2z^2 - x^2 - y^2)/2 sqrt5, xz, (x^2 - y^2)/2 sqrt15
        g[0] += s15 * (d[4] * y + d[7] * z + d[8] * x) - s5 * d[6] * x;
        g[1] += s15 * (d[4] * x + d[5] * z - d[8] * y) - s5 * d[6] * y;
        g[2] += s15 * (d[5] * y + d[7] * x) + 2.f * s5 * d[6] * z;
        const float y2 = s15 * (d[4] * x * y + d[5] * y * z + d[7] * x * z + 0.5f * d[8] * (xx - yy)) +
                         0.5f * s5 * d[6] * (2.f * zz - xx - yy);
        e += 2.f * y2;
        if constexpr (LMAX >= 3) {
            const float a = 0.25f * s70, b = s105, c = 0.25f * s42, h = 0.5f * s7, k = 0.5f * s105;
            // m=-3: a (3x^2 y - y^3)     m=-2: b xyz          m=-1: c (4yz^2 - x^2 y - y^3)
            // m=0:  h (2z^3 - 3x^2 z - 3y^2 z)                m=1:  c (4xz^2 - x^3 - xy^2)
            // m=2:  k (x^2 z - y^2 z)    m=3:  a (x^3 - 3xy^2)
            g[0] += a * d[9] * 6.f * x * y + b * d[10] * y * z - c * d[11] * 2.f * x * y - h * d[12] * 6.f * x * z +
                    c * d[13] * (4.f * zz - 3.f * xx - yy) + k * d[14] * 2.f * x * z + a * d[15] * 3.f * (xx - yy);
            g[1] += a * d[9] * 3.f * (xx - yy) + b * d[10] * x * z + c * d[11] * (4.f * zz - xx - 3.f * yy) -
                    h * d[12] * 6.f * y * z - c * d[13] * 2.f * x * y - k * d[14] * 2.f * y * z - a * d[15] * 6.f * x * y;
            g[2] += b * d[10] * x * y + c * d[11] * 8.f * y * z + h * d[12] * (6.f * zz - 3.f * xx - 3.f * yy) +
                    c * d[13] * 8.f * x * z + k * d[14] * (xx - yy);
            const float y3 = a * d[9] * y * (3.f * xx - yy) + b * d[10] * x * y * z + c * d[11] * y * (4.f * zz - xx - yy) +
                             h * d[12] * z * (2.f * zz - 3.f * xx - 3.f * yy) + c * d[13] * x * (4.f * zz - xx - yy) +
                             k * d[14] * z * (xx - yy) + a * d[15] * x * (xx - 3.f * yy);
            e += 3.f * y3;
        }
    }
}

template <class T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <int LMAX, class T>
__global__ void __launch_bounds__(kShBlock) sh_backward_kernel(int64_t n, const float* __restrict__ vec,
                                                               const T* __restrict__ dy, float* __restrict__ dvec) {
    constexpr int K = (LMAX + 1) * (LMAX + 1);
    const int64_t e = int64_t(blockIdx.x) * kShBlock + threadIdx.x;
    if (e >= n) return;
    float v0 = __ldg(vec + 3 * e), v1 = __ldg(vec + 3 * e + 1), v2 = __ldg(vec + 3 * e + 2);
    const float r = sqrtf(v0 * v0 + v1 * v1 + v2 * v2);
    float out[3] = {0.f, 0.f, 0.f};
    if (r >= 1e-12f) {
        v0 = v0 / r; v1 = v1 / r; v2 = v2 / r;
        float d[16];
#pragma unroll
        for (int k = 0; k < K; ++k) d[k] = to_f32<T>(dy[e * K + k]);
        float g[3], eu;
        sh_grad_eval<LMAX>(v0, v1, v2, d, g, eu);
        out[0] = (g[0] - eu * v0) / r;
        out[1] = (g[1] - eu * v1) / r;
        out[2] = (g[2] - eu * v2) / r;
    }
    dvec[3 * e] = out[0];
    dvec[3 * e + 1] = out[1];
    dvec[3 * e + 2] = out[2];
}

template <class T>
cudaError_t launch_sh_backward(int lmax, int64_t n, const float* vec, const void* dy, float* dvec, cudaStream_t s) {
    const int64_t grid = (n + kShBlock - 1) / kShBlock;
    if (grid == 0) return cudaSuccess;
    switch (lmax) {
        case 0: sh_backward_kernel<0, T><<<grid, kShBlock, 0, s>>>(n, vec, (const T*)dy, dvec); break;
        case 1: sh_backward_kernel<1, T><<<grid, kShBlock, 0, s>>>(n, vec, (const T*)dy, dvec); break;
        case 2: sh_backward_kernel<2, T><<<grid, kShBlock, 0, s>>>(n, vec, (const T*)dy, dvec); break;
        default: sh_backward_kernel<3, T><<<grid, kShBlock, 0, s>>>(n, vec, (const T*)dy, dvec); break;
    }
    return cudaGetLastError();
}

template <class T>
cudaError_t launch_sh(int lmax, int64_t n, const float* vec, void* y, cudaStream_t s) {
    const int64_t grid = (n + kShBlock - 1) / kShBlock;
    if (grid == 0) return cudaSuccess;
    switch (lmax) {
        case 0: sh_kernel<0, T><<<grid, kShBlock, 0, s>>>(n, vec, (T*)y); break;
        case 1: sh_kernel<1, T><<<grid, kShBlock, 0, s>>>(n, vec, (T*)y); break;
        case 2: sh_kernel<2, T><<<grid, kShBlock, 0, s>>>(n, vec, (T*)y); break;
        default: sh_kernel<3, T><<<grid, kShBlock, 0, s>>>(n, vec, (T*)y); break;
    }
    return cudaGetLastError();
}
}  // namespace

cudaError_t sh_forward(int lmax, int64_t n, const float* vec, void* y, int bf16, cudaStream_t s) {
    return bf16 ? launch_sh<__nv_bfloat16>(lmax, n, vec, y, s) : launch_sh<float>(lmax, n, vec, y, s);
}

cudaError_t sh_backward(int lmax, int64_t n, const float* vec, const void* dy, float* dvec, int bf16, cudaStream_t s) {
    return bf16 ? launch_sh_backward<__nv_bfloat16>(lmax, n, vec, dy, dvec, s)
                : launch_sh_backward<float>(lmax, n, vec, dy, dvec, s);
}

}  // namespace e3gb
