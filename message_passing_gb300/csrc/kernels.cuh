// Tensor-product and convolution kernels, specialised at compile time per irreps
// configuration (cg_table.hpp). Included by instances.cu once per configuration.
//
// Mapping ("e3j ...", App. E.2.1 "trailing channels"): lanes own channels, VEC = 4 adjacent
// channels per lane (one 16-byte fp32 vector or one 8-byte bf16 vector), G = Nq/4 lanes per
// row, 32/G rows per warp. Every lane walks the same unrolled sequence of CG couplings.
// Inputs (x, y, w, dz / dm) are stored as T (fp32 or bf16); arithmetic and every output are
// fp32.
//
// Per row / edge, the SH operand y is contracted first with the CG block of each path:
//   A_p[m3][m1] = sum_m2 C_p[m1][m2][m3] y[l2^2 + m2]        (lane-uniform, from immediates)
// and then applied to every channel:
//   z_p[m3][q] = sum_m1 A_p[m3][m1] x[l1 off + m1][q],  out[blk p][m3][q] += w[p][q] z_p[m3][q]
// (the weight multiplies whichever side, x or z_p, is shorter). This is Eq. (13) with the
// sum over i2 taken inside the per-edge uniform part, as Alg. 2 takes the sum over records
// before applying the edge scalar.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "cg_table.hpp"

namespace e3gb {

constexpr int kVec = 4;

// device error word bits
constexpr unsigned kErrSender = 1u, kErrRowptr = 2u, kErrRecv = 4u;

template <int... I, class F>
__device__ __forceinline__ void sfor_impl(std::integer_sequence<int, I...>, F&& f) {
    (f(std::integral_constant<int, I>{}), ...);
}
// static for: f(integral_constant<int, i>) for i = 0..N-1, fully unrolled
template <int N, class F>
__device__ __forceinline__ void sfor(F&& f) {
    sfor_impl(std::make_integer_sequence<int, N>{}, f);
}

// ------------------------------------------------------------------------------------------
// storage types
// ------------------------------------------------------------------------------------------
template <class T>
struct IO;

template <>
struct IO<float> {
    static __device__ __forceinline__ void load4(const float* __restrict__ p, float (&o)[4]) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(p));
        o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
    }
    static __device__ __forceinline__ void store4(float* __restrict__ p, const float (&o)[4]) {
        *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
    }
    static __device__ __forceinline__ float load1(const float* __restrict__ p) { return __ldg(p); }
    static __device__ __forceinline__ void store1(float* __restrict__ p, float v) { *p = v; }
};

template <>
struct IO<__nv_bfloat16> {
    static __device__ __forceinline__ void load4(const __nv_bfloat16* __restrict__ p, float (&o)[4]) {
        const uint2 t = __ldg(reinterpret_cast<const uint2*>(p));
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&t.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&t.y);
        const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
        o[0] = fa.x; o[1] = fa.y; o[2] = fb.x; o[3] = fb.y;
    }
    static __device__ __forceinline__ void store4(__nv_bfloat16* __restrict__ p, const float (&o)[4]) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]);
        const __nv_bfloat162 b = __floats2bfloat162_rn(o[2], o[3]);
        uint2 t;
        t.x = *reinterpret_cast<const uint32_t*>(&a);
        t.y = *reinterpret_cast<const uint32_t*>(&b);
        *reinterpret_cast<uint2*>(p) = t;
    }
    static __device__ __forceinline__ float load1(const __nv_bfloat16* __restrict__ p) {
        return __bfloat162float(p[0]);
    }
    static __device__ __forceinline__ void store1(__nv_bfloat16* __restrict__ p, float v) {
        *p = __float2bfloat16_rn(v);
    }
};

// V consecutive channels (V = 1 or 4) of one row
template <class T, int V>
__device__ __forceinline__ void loadv(const T* __restrict__ p, float (&o)[V]) {
    if constexpr (V == 4) IO<T>::load4(p, o);
    else
#pragma unroll
        for (int c = 0; c < V; ++c) o[c] = IO<T>::load1(p + c);
}
template <int V>
__device__ __forceinline__ void storev(float* __restrict__ p, const float (&o)[V]) {
    if constexpr (V == 4) IO<float>::store4(p, o);
    else
#pragma unroll
        for (int c = 0; c < V; ++c) p[c] = o[c];
}

// ------------------------------------------------------------------------------------------
// per-configuration constant helpers
// ------------------------------------------------------------------------------------------
template <class Cfg>
struct Off {
    // offsets of each path's A-entries and CG records inside Cfg::aents / Cfg::recs
    static constexpr std::array<int, Cfg::NP + 1> a = [] {
        std::array<int, Cfg::NP + 1> o{};
        for (int i = 0; i < Cfg::NA; ++i) o[Cfg::aents[i].path + 1]++;
        for (int p = 0; p < Cfg::NP; ++p) o[p + 1] += o[p];
        return o;
    }();
    static constexpr std::array<int, Cfg::NP + 1> r = [] {
        std::array<int, Cfg::NP + 1> o{};
        for (int i = 0; i < Cfg::NR; ++i) o[Cfg::recs[i].path + 1]++;
        for (int p = 0; p < Cfg::NP; ++p) o[p + 1] += o[p];
        return o;
    }();
    // first output offset of output block j
    static constexpr std::array<int, Cfg::NOUT + 1> z = [] {
        std::array<int, Cfg::NOUT + 1> o{};
        for (int j = 0; j < Cfg::NOUT; ++j) o[j + 1] = o[j] + 2 * Cfg::table.outs[j].l + 1;
        return o;
    }();
};

// A_p entries for path P (compile-time), from the row's y values.
template <class Cfg, int P>
__device__ __forceinline__ void build_A(const float (&yv)[Cfg::D2], float (&A)[Off<Cfg>::a[P + 1] - Off<Cfg>::a[P]]) {
    constexpr int a0 = Off<Cfg>::a[P];
    constexpr int na = Off<Cfg>::a[P + 1] - a0;
    constexpr int yo = Cfg::table.paths[P].yoff;
    sfor<na>([&](auto k) {
        constexpr AEnt e = Cfg::aents[a0 + decltype(k)::value];
        float s = e.c[0] * yv[yo + e.m2[0]];
        sfor<e.nt - 1>([&](auto t) {
            constexpr int tt = decltype(t)::value + 1;
            s = fmaf(e.c[tt], yv[yo + e.m2[tt]], s);
        });
        A[decltype(k)::value] = s;
    });
}

// acc[m3][c] += w[c] * sum_m1 A[m3][m1] x[xoff + m1][c] for path P.
template <class Cfg, int P, int NROWS, int V>
__device__ __forceinline__ void apply_path(const float (&A)[Off<Cfg>::a[P + 1] - Off<Cfg>::a[P]],
                                           const float (&xv)[Cfg::D1][V], const float (&wv)[V],
                                           float (&acc)[NROWS][V], int row0) {
    constexpr PathInfo pi = Cfg::table.paths[P];
    constexpr int a0 = Off<Cfg>::a[P];
    constexpr int na = Off<Cfg>::a[P + 1] - a0;
    constexpr int n1 = 2 * pi.l1 + 1, n3 = 2 * pi.l3 + 1;
    if constexpr (n1 <= n3) {
        float xw[n1][V];
#pragma unroll
        for (int m = 0; m < n1; ++m)
#pragma unroll
            for (int c = 0; c < V; ++c) xw[m][c] = wv[c] * xv[pi.xoff + m][c];
        sfor<na>([&](auto k) {
            constexpr AEnt e = Cfg::aents[a0 + decltype(k)::value];
#pragma unroll
            for (int c = 0; c < V; ++c)
                acc[row0 + e.m3][c] = fmaf(A[decltype(k)::value], xw[e.m1][c], acc[row0 + e.m3][c]);
        });
    } else {
        float t[n3][V];
#pragma unroll
        for (int m = 0; m < n3; ++m)
#pragma unroll
            for (int c = 0; c < V; ++c) t[m][c] = 0.f;
        sfor<na>([&](auto k) {
            constexpr AEnt e = Cfg::aents[a0 + decltype(k)::value];
#pragma unroll
            for (int c = 0; c < V; ++c)
                t[e.m3][c] = fmaf(A[decltype(k)::value], xv[pi.xoff + e.m1][c], t[e.m3][c]);
        });
#pragma unroll
        for (int m = 0; m < n3; ++m)
#pragma unroll
            for (int c = 0; c < V; ++c) acc[row0 + m][c] = fmaf(wv[c], t[m][c], acc[row0 + m][c]);
    }
}

struct Lanes {
    int G;        // lanes per row
    int grp;      // row slot inside the warp
    int gl;       // lane inside the row group
    int per_warp; // rows per warp
};

template <int V>
__device__ __forceinline__ Lanes lanes_for(int Nq) {
    Lanes L;
    L.G = Nq / V;
    const int lane = threadIdx.x & 31;
    L.grp = lane / L.G;
    L.gl = lane % L.G;
    L.per_warp = 32 / L.G;
    return L;
}

// ------------------------------------------------------------------------------------------
// TP forward on rows: output block by output block, so only one block's accumulators live.
// ------------------------------------------------------------------------------------------
template <class Cfg, class T, int V>
__global__ void __launch_bounds__(384) tp_forward_kernel(int64_t R, int Nq, const T* __restrict__ x,
                                                         const T* __restrict__ y, const T* __restrict__ w,
                                                         float* __restrict__ z) {
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    for (int64_t r = warp * L.per_warp + L.grp; r < R; r += nwarp * L.per_warp) {
        float yv[Cfg::D2];
#pragma unroll
        for (int i = 0; i < Cfg::D2; ++i) yv[i] = IO<T>::load1(y + r * Cfg::D2 + i);
        float xv[Cfg::D1][V];
#pragma unroll
        for (int i = 0; i < Cfg::D1; ++i) loadv<T, V>(x + (r * Cfg::D1 + i) * Nq + c0, xv[i]);
        sfor<Cfg::NOUT>([&](auto jj) {
            constexpr int j = decltype(jj)::value;
            constexpr int nrow = 2 * Cfg::table.outs[j].l + 1;
            float acc[nrow][V];
#pragma unroll
            for (int m = 0; m < nrow; ++m)
#pragma unroll
                for (int c = 0; c < V; ++c) acc[m][c] = 0.f;
            sfor<Cfg::NP>([&](auto pp) {
                constexpr int p = decltype(pp)::value;
                if constexpr (Cfg::table.paths[p].out_block == j) {
                    float A[Off<Cfg>::a[p + 1] - Off<Cfg>::a[p]];
                    build_A<Cfg, p>(yv, A);
                    float wv[V];
                    loadv<T, V>(w + (r * Cfg::NP + p) * Nq + c0, wv);
                    apply_path<Cfg, p, nrow, V>(A, xv, wv, acc, 0);
                }
            });
            constexpr int zo = Off<Cfg>::z[j];
#pragma unroll
            for (int m = 0; m < nrow; ++m) storev<V>(z + (r * Cfg::D + zo + m) * Nq + c0, acc[m]);
        });
    }
}

// ------------------------------------------------------------------------------------------
// Where the per-edge weights w[e][p][c] come from and where their cotangent dw goes.
// WMem: rows of a w array in memory, dw rows written back.
// WRad: the radial network's output layer evaluated in place (the fused edge-scalar producer:
// "e3j ...", App. E.1 notation for s, App. A.3 "Linear mixing"),
//   w[p][c] = sum_k h[k] W2[k][p][c],   dh[k] += sum_c W2[k][p][c] dw[p][c],
// with W2 [RH][NP][Nq] in shared memory and h the edge's hidden activations; w and dw never
// reach memory. dh holds the lane's partial sums over its own channels.
// ------------------------------------------------------------------------------------------
template <class T, int V>
struct WMem {
    const T* __restrict__ w_e;
    float* __restrict__ dw_e;
    int Nq, c0;
    __device__ __forceinline__ void get(int p, float (&wv)[V]) const { loadv<T, V>(w_e + p * Nq + c0, wv); }
    __device__ __forceinline__ void put(int p, const float (&dwv)[V]) { storev<V>(dw_e + p * Nq + c0, dwv); }
};

// V consecutive floats of a shared-memory row (plain loads: the read-only global path of
// loadv must not be given a shared address)
template <int V>
__device__ __forceinline__ void lds_v(const float* p, float (&o)[V]) {
    if constexpr (V == 4) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
    } else {
#pragma unroll
        for (int c = 0; c < V; ++c) o[c] = p[c];
    }
}

template <int NP, int RH, int V>
struct WRad {
    const float* __restrict__ w2s;   // shared memory, [RH][NP][Nq]
    float h[RH];
    float dh[RH];
    int Nq, c0;
    __device__ __forceinline__ void get(int p, float (&wv)[V]) const {
#pragma unroll
        for (int c = 0; c < V; ++c) wv[c] = 0.f;
#pragma unroll
        for (int k = 0; k < RH; ++k) {
            float w2[V];
            lds_v<V>(w2s + (k * NP + p) * Nq + c0, w2);
#pragma unroll
            for (int c = 0; c < V; ++c) wv[c] = fmaf(h[k], w2[c], wv[c]);
        }
    }
    __device__ __forceinline__ void put(int p, const float (&dwv)[V]) {
#pragma unroll
        for (int k = 0; k < RH; ++k) {
            float w2[V];
            lds_v<V>(w2s + (k * NP + p) * Nq + c0, w2);
            float s = 0.f;
#pragma unroll
            for (int c = 0; c < V; ++c) s = fmaf(w2[c], dwv[c], s);
            dh[k] += s;
        }
    }
};

// shared-memory copy of W2 [RH][NP][Nq] by the whole block (n floats; both ends 16-byte
// aligned): 16-byte copies, then the n % 4 floats left over
__device__ __forceinline__ void load_w2_shared(float* __restrict__ dst, const float* __restrict__ W2, int n) {
    const int n4 = n & ~3;
    for (int i = threadIdx.x * 4; i < n4; i += blockDim.x * 4)
        *reinterpret_cast<float4*>(dst + i) = __ldg(reinterpret_cast<const float4*>(W2 + i));
    for (int i = n4 + threadIdx.x; i < n; i += blockDim.x) dst[i] = __ldg(W2 + i);
    __syncthreads();
}

// ------------------------------------------------------------------------------------------
// Backward body for one (row or edge) e: given x (of the row / sender), y[e], w[e] and the
// cotangent rows g = scale * dz/dm (of the row / receiver), accumulate dx into dxa, the
// lane's partial dy (summed over its channels) into dyp, and write dw[e].
//   g_p[m1][q] = sum_m3 A_p[m3][m1] g[blk p][m3][q]
//   dw[e,p,q]  = sum_m1 x[m1][q] g_p[m1][q]
//   dx[m1][q] += w[p][q] g_p[m1][q]
//   dy[m2]    += sum_{records (m1,m2,m3,c)} c * sum_q x[m1][q] w[p][q] g[m3][q]
// ------------------------------------------------------------------------------------------
template <class Cfg, class T, int V, class WS>
__device__ __forceinline__ void backward_body(const float (&xv)[Cfg::D1][V], const float (&yv)[Cfg::D2], WS& ws,
                                              const T* __restrict__ g_row, float gscale, int Nq, int c0,
                                              float (&dxa)[Cfg::D1][V], float (&dyp)[Cfg::D2]) {
    sfor<Cfg::NOUT>([&](auto jj) {
        constexpr int j = decltype(jj)::value;
        constexpr int nrow = 2 * Cfg::table.outs[j].l + 1;
        constexpr int zo = Off<Cfg>::z[j];
        float g[nrow][V];
#pragma unroll
        for (int m = 0; m < nrow; ++m) {
            loadv<T, V>(g_row + (zo + m) * Nq + c0, g[m]);
#pragma unroll
            for (int c = 0; c < V; ++c) g[m][c] *= gscale;
        }
        sfor<Cfg::NP>([&](auto pp) {
            constexpr int p = decltype(pp)::value;
            constexpr PathInfo pi = Cfg::table.paths[p];
            if constexpr (pi.out_block == j) {
                constexpr int a0 = Off<Cfg>::a[p];
                constexpr int na = Off<Cfg>::a[p + 1] - a0;
                constexpr int n1 = 2 * pi.l1 + 1;
                float A[na];
                build_A<Cfg, p>(yv, A);
                float wv[V];
                ws.get(p, wv);
                float gp[n1][V];
                float xw[n1][V];
#pragma unroll
                for (int m = 0; m < n1; ++m)
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        gp[m][c] = 0.f;
                        xw[m][c] = xv[pi.xoff + m][c] * wv[c];
                    }
                sfor<na>([&](auto k) {
                    constexpr AEnt e = Cfg::aents[a0 + decltype(k)::value];
                    float s = 0.f;
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        gp[e.m1][c] = fmaf(A[decltype(k)::value], g[e.m3][c], gp[e.m1][c]);
                        s = fmaf(xw[e.m1][c], g[e.m3][c], s);
                    }
                    sfor<e.nt>([&](auto t) {
                        constexpr int tt = decltype(t)::value;
                        dyp[pi.yoff + e.m2[tt]] = fmaf(e.c[tt], s, dyp[pi.yoff + e.m2[tt]]);
                    });
                });
                float dwv[V];
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    float s = 0.f;
#pragma unroll
                    for (int m = 0; m < n1; ++m) {
                        s = fmaf(xv[pi.xoff + m][c], gp[m][c], s);
                        dxa[pi.xoff + m][c] = fmaf(wv[c], gp[m][c], dxa[pi.xoff + m][c]);
                    }
                    dwv[c] = s;
                }
                ws.put(p, dwv);
            }
        });
    });
}

// Sum dyp over the G lanes of a row group (fixed butterfly order, deterministic).
template <int N>
__device__ __forceinline__ void group_reduce(float (&v)[N], int G) {
    for (int off = G >> 1; off > 0; off >>= 1) {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], off);
    }
}

template <class Cfg, class T, int V>
__global__ void __launch_bounds__(256) tp_backward_kernel(int64_t R, int Nq, const T* __restrict__ x,
                                                          const T* __restrict__ y, const T* __restrict__ w,
                                                          const T* __restrict__ dz, float* __restrict__ dx,
                                                          float* __restrict__ dy, float* __restrict__ dw) {
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    // every lane of the warp runs the same trip count so the group shuffles stay converged
    const int64_t iters = (R + nwarp * L.per_warp - 1) / (nwarp * L.per_warp);
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = (it * nwarp + warp) * L.per_warp + L.grp;
        const bool live = r < R;
        const int64_t rr = live ? r : 0;
        float yv[Cfg::D2], xv[Cfg::D1][V], dxa[Cfg::D1][V], dyp[Cfg::D2];
#pragma unroll
        for (int i = 0; i < Cfg::D2; ++i) {
            yv[i] = live ? IO<T>::load1(y + rr * Cfg::D2 + i) : 0.f;
            dyp[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < Cfg::D1; ++i) {
            if (live) loadv<T, V>(x + (rr * Cfg::D1 + i) * Nq + c0, xv[i]);
            else
#pragma unroll
                for (int c = 0; c < V; ++c) xv[i][c] = 0.f;
#pragma unroll
            for (int c = 0; c < V; ++c) dxa[i][c] = 0.f;
        }
        if (live) {
            WMem<T, V> ws{w + rr * Cfg::NP * Nq, dw + rr * Cfg::NP * Nq, Nq, c0};
            backward_body<Cfg, T, V>(xv, yv, ws, dz + rr * Cfg::D * Nq, 1.f, Nq, c0, dxa, dyp);
        }
        group_reduce<Cfg::D2>(dyp, L.G);
        if (live) {
#pragma unroll
            for (int i = 0; i < Cfg::D1; ++i) storev<V>(dx + (rr * Cfg::D1 + i) * Nq + c0, dxa[i]);
            if (L.gl == 0)
#pragma unroll
                for (int i = 0; i < Cfg::D2; ++i) dy[rr * Cfg::D2 + i] = dyp[i];
        }
    }
}

// ------------------------------------------------------------------------------------------
// Convolution forward: one row group per receiver, all D output rows in registers, edges
// of the receiver in CSR order (Alg. 2 receiver-stationary aggregation).
// ------------------------------------------------------------------------------------------
// RH > 0: the radial form (weights from the hidden activations h [E][RH] and the output
// layer W2 [RH][NP][Nq], staged in dynamic shared memory; w unused)
template <class Cfg, class T, int V, int RH = 0>
__global__ void __launch_bounds__(256) conv_forward_kernel(int64_t N, int64_t E, int Nq,
                                                           const int32_t* __restrict__ rowptr,
                                                           const int32_t* __restrict__ sender,
                                                           const T* __restrict__ x, const T* __restrict__ y,
                                                           const T* __restrict__ w, float scale,
                                                           float* __restrict__ m, int64_t pad,
                                                           unsigned* __restrict__ err, int64_t cap,
                                                           const float* __restrict__ hrad = nullptr,
                                                           const float* __restrict__ W2 = nullptr) {
    extern __shared__ __align__(16) float w2s[];
    if constexpr (RH > 0) load_w2_shared(w2s, W2, RH * Cfg::NP * Nq);
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    for (int64_t b = warp * L.per_warp + L.grp; b < N; b += nwarp * L.per_warp) {
        float acc[Cfg::D][V];
#pragma unroll
        for (int i = 0; i < Cfg::D; ++i)
#pragma unroll
            for (int c = 0; c < V; ++c) acc[i][c] = 0.f;
        int64_t e0 = __ldg(rowptr + b), e1 = __ldg(rowptr + b + 1);
        if (e0 < 0 || e1 < e0 || e1 > E) {
            if (L.gl == 0) atomicOr(err, kErrRowptr);
            e1 = e0 = 0;
        }
        if (b == pad) e0 = e1 = 0;   // padding receiver: no messages
        if (e1 - e0 > cap) e1 = e0 + cap;   // the rest of a heavy receiver: the pieces kernel
        for (int64_t e = e0; e < e1; ++e) {
            const int64_t a = __ldg(sender + e);
            if (pad >= 0 && a == pad) continue;   // padding edge
            if (a < 0 || a >= N) {
                if (L.gl == 0) atomicOr(err, kErrSender);
                continue;
            }
            float yv[Cfg::D2];
#pragma unroll
            for (int i = 0; i < Cfg::D2; ++i) yv[i] = IO<T>::load1(y + e * Cfg::D2 + i);
            float xv[Cfg::D1][V];
#pragma unroll
            for (int i = 0; i < Cfg::D1; ++i) loadv<T, V>(x + (a * Cfg::D1 + i) * Nq + c0, xv[i]);
            auto paths = [&](const auto& ws) {
                sfor<Cfg::NP>([&](auto pp) {
                    constexpr int p = decltype(pp)::value;
                    float A[Off<Cfg>::a[p + 1] - Off<Cfg>::a[p]];
                    build_A<Cfg, p>(yv, A);
                    float wv[V];
                    ws.get(p, wv);
                    apply_path<Cfg, p, Cfg::D, V>(A, xv, wv, acc, Cfg::table.paths[p].zoff);
                });
            };
            if constexpr (RH > 0) {
                WRad<Cfg::NP, RH, V> ws;
                ws.w2s = w2s;
                ws.Nq = Nq;
                ws.c0 = c0;
#pragma unroll
                for (int k = 0; k < RH; ++k) ws.h[k] = __ldg(hrad + e * RH + k);
                paths(ws);
            } else {
                paths(WMem<T, V>{w + e * Cfg::NP * Nq, nullptr, Nq, c0});
            }
        }
#pragma unroll
        for (int i = 0; i < Cfg::D; ++i) {
#pragma unroll
            for (int c = 0; c < V; ++c) acc[i][c] *= scale;
            storev<V>(m + (b * Cfg::D + i) * Nq + c0, acc[i]);
        }
    }
}

// Convolution forward for configurations with many output rows (one output block per path,
// "multiplicities arise", App. E.1): the receiver's edges are walked once per output block, so
// only that block's rows (at most 2 l3 + 1) are live in registers. The x and y rows of an edge
// are re-read per block from L1/L2; each path's w row is read in the block it belongs to, so
// w still moves once. Fixed order per block: deterministic.
template <class Cfg, class T, int V>
__global__ void __launch_bounds__(256) conv_forward_blocks_kernel(int64_t N, int64_t E, int Nq,
                                                                  const int32_t* __restrict__ rowptr,
                                                                  const int32_t* __restrict__ sender,
                                                                  const T* __restrict__ x, const T* __restrict__ y,
                                                                  const T* __restrict__ w, float scale,
                                                                  float* __restrict__ m, int64_t pad,
                                                                  unsigned* __restrict__ err, int64_t cap) {
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    for (int64_t b = warp * L.per_warp + L.grp; b < N; b += nwarp * L.per_warp) {
        int64_t e0 = __ldg(rowptr + b), e1 = __ldg(rowptr + b + 1);
        if (e0 < 0 || e1 < e0 || e1 > E) {
            if (L.gl == 0) atomicOr(err, kErrRowptr);
            e1 = e0 = 0;
        }
        if (b == pad) e0 = e1 = 0;   // padding receiver: no messages
        if (e1 - e0 > cap) e1 = e0 + cap;   // the rest of a heavy receiver: the pieces kernel
        sfor<Cfg::NOUT>([&](auto jj) {
            constexpr int j = decltype(jj)::value;
            constexpr int nrow = 2 * Cfg::table.outs[j].l + 1;
            float acc[nrow][V];
#pragma unroll
            for (int i = 0; i < nrow; ++i)
#pragma unroll
                for (int c = 0; c < V; ++c) acc[i][c] = 0.f;
            for (int64_t e = e0; e < e1; ++e) {
                const int64_t a = __ldg(sender + e);
                if (pad >= 0 && a == pad) continue;   // padding edge
                if (a < 0 || a >= N) {
                    if (j == 0 && L.gl == 0) atomicOr(err, kErrSender);
                    continue;
                }
                float yv[Cfg::D2];
#pragma unroll
                for (int i = 0; i < Cfg::D2; ++i) yv[i] = IO<T>::load1(y + e * Cfg::D2 + i);
                float xv[Cfg::D1][V];
#pragma unroll
                for (int i = 0; i < Cfg::D1; ++i) loadv<T, V>(x + (a * Cfg::D1 + i) * Nq + c0, xv[i]);
                sfor<Cfg::NP>([&](auto pp) {
                    constexpr int p = decltype(pp)::value;
                    if constexpr (Cfg::table.paths[p].out_block == j) {
                        float A[Off<Cfg>::a[p + 1] - Off<Cfg>::a[p]];
                        build_A<Cfg, p>(yv, A);
                        float wv[V];
                        loadv<T, V>(w + (e * Cfg::NP + p) * Nq + c0, wv);
                        apply_path<Cfg, p, nrow, V>(A, xv, wv, acc, 0);
                    }
                });
            }
            constexpr int zo = Off<Cfg>::z[j];
#pragma unroll
            for (int i = 0; i < nrow; ++i) {
#pragma unroll
                for (int c = 0; c < V; ++c) acc[i][c] *= scale;
                storev<V>(m + (b * Cfg::D + zo + i) * Nq + c0, acc[i]);
            }
        });
    }
}

// ------------------------------------------------------------------------------------------
// Convolution backward in sender order (the transposed graph of Eq. 16): one row group per
// sender a; x[a] and the dx[a] accumulators stay in registers while the group walks the
// edges of a (csc_ptr / csc_edge / csc_recv), gathering dm of each receiver. dw and dy are
// edge-local and written once per edge.
// ------------------------------------------------------------------------------------------
// RH > 0: the radial form; dw is then dh [E][RH] (the cotangent of the hidden activations,
// sum over paths and channels of W2 dw) and w is unused
template <class Cfg, class T, int V, int RH = 0>
__global__ void __launch_bounds__(256) conv_backward_kernel(
    int64_t N, int64_t E, int Nq, const int32_t* __restrict__ csc_ptr, const int32_t* __restrict__ csc_edge,
    const int32_t* __restrict__ csc_recv, const T* __restrict__ x, const T* __restrict__ y,
    const T* __restrict__ w, const T* __restrict__ dm, float scale, float* __restrict__ dx,
    float* __restrict__ dy, float* __restrict__ dw, int64_t pad, unsigned* __restrict__ err,
    const float* __restrict__ hrad = nullptr, const float* __restrict__ W2 = nullptr) {
    extern __shared__ __align__(16) float w2s[];
    if constexpr (RH > 0) load_w2_shared(w2s, W2, RH * Cfg::NP * Nq);
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    const int64_t iters = (N + nwarp * L.per_warp - 1) / (nwarp * L.per_warp);
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t a = (it * nwarp + warp) * L.per_warp + L.grp;
        const bool live = a < N;
        const int64_t aa = live ? a : 0;
        float xv[Cfg::D1][V], dxa[Cfg::D1][V];
#pragma unroll
        for (int i = 0; i < Cfg::D1; ++i) {
            if (live) loadv<T, V>(x + (aa * Cfg::D1 + i) * Nq + c0, xv[i]);
            else
#pragma unroll
                for (int c = 0; c < V; ++c) xv[i][c] = 0.f;
#pragma unroll
            for (int c = 0; c < V; ++c) dxa[i][c] = 0.f;
        }
        int64_t k0 = 0, k1 = 0;
        if (live) {
            k0 = __ldg(csc_ptr + aa);
            k1 = __ldg(csc_ptr + aa + 1);
            if (k0 < 0 || k1 < k0 || k1 > E) {
                if (L.gl == 0) atomicOr(err, kErrRowptr);
                k0 = k1 = 0;
            }
            if (aa == pad) k0 = k1 = 0;   // padding sender: no messages
        }
        // the row groups of a warp may own different edge counts; loop to the warp maximum
        int64_t cnt = k1 - k0, wmax = cnt;
        for (int off = 16; off > 0; off >>= 1) {
            const int64_t o = __shfl_xor_sync(0xffffffffu, wmax, off);
            wmax = o > wmax ? o : wmax;
        }
        for (int64_t i = 0; i < wmax; ++i) {
            bool ok = i < cnt;
            int64_t e = 0, b = 0;
            if (ok) {
                e = __ldg(csc_edge + k0 + i);
                b = __ldg(csc_recv + k0 + i);
                if (pad >= 0 && b == pad) {
                    ok = false;   // padding edge: its dw, dy rows are zeroed separately
                } else if (e < 0 || e >= E || b < 0 || b >= N) {
                    if (L.gl == 0) atomicOr(err, kErrRecv);
                    ok = false;
                }
            }
            float dyp[Cfg::D2];
#pragma unroll
            for (int t = 0; t < Cfg::D2; ++t) dyp[t] = 0.f;
            if constexpr (RH > 0) {
                WRad<Cfg::NP, RH, V> ws;
                ws.w2s = w2s;
                ws.Nq = Nq;
                ws.c0 = c0;
#pragma unroll
                for (int k = 0; k < RH; ++k) {
                    ws.h[k] = ok ? __ldg(hrad + e * RH + k) : 0.f;
                    ws.dh[k] = 0.f;
                }
                if (ok) {
                    float yv[Cfg::D2];
#pragma unroll
                    for (int t = 0; t < Cfg::D2; ++t) yv[t] = IO<T>::load1(y + e * Cfg::D2 + t);
                    backward_body<Cfg, T, V>(xv, yv, ws, dm + b * Cfg::D * Nq, scale, Nq, c0, dxa, dyp);
                }
                group_reduce<RH>(ws.dh, L.G);
                if (ok && L.gl == 0)
#pragma unroll
                    for (int k = 0; k < RH; ++k) dw[e * RH + k] = ws.dh[k];
            } else if (ok) {
                float yv[Cfg::D2];
#pragma unroll
                for (int t = 0; t < Cfg::D2; ++t) yv[t] = IO<T>::load1(y + e * Cfg::D2 + t);
                WMem<T, V> ws{w + e * Cfg::NP * Nq, dw + e * Cfg::NP * Nq, Nq, c0};
                backward_body<Cfg, T, V>(xv, yv, ws, dm + b * Cfg::D * Nq, scale, Nq, c0, dxa, dyp);
            }
            group_reduce<Cfg::D2>(dyp, L.G);
            if (ok && L.gl == 0)
#pragma unroll
                for (int t = 0; t < Cfg::D2; ++t) dy[e * Cfg::D2 + t] = dyp[t];
        }
        if (live)
#pragma unroll
            for (int i = 0; i < Cfg::D1; ++i) storev<V>(dx + (aa * Cfg::D1 + i) * Nq + c0, dxa[i]);
    }
}

// ------------------------------------------------------------------------------------------
// Convolution double backward ("e3j ...", App. E.1 Eq. (17)-(18)) in two fused passes
// instead of three conv and three conv_bwd calls: no cotangent that Eq. (18) discards is
// computed, and each primal is streamed once per pass.
//
// Receiver pass (Eq. 17): delta_dm[b] = scale * sum_e [TP(ddx_a, y, w) + TP(x_a, ddy, w)
//                                                      + TP(x_a, y, ddw)].
// Sender pass (Eq. 18), with g = scale * dm[b] and, per path, the adjoint couplings
//   gy[m1] = sum_m3 A_p(y)[m3][m1] g[m3],   gd[m1] = sum_m3 A_p(ddy)[m3][m1] g[m3]:
//   delta_x[a]       += w_p gd + ddw_p gy
//   delta_w[e][p]     = sum_m1 ddx[m1] gy[m1] + x[m1] gd[m1]
//   delta_y[e][m2]   += sum_{records (m1,m2,m3,c)} c * sum_q (ddx[m1] w_p + x[m1] ddw_p) g[m3]
// The x and ddx rows of a path's l1 block are loaded per path (L1-resident), which keeps
// the accumulators in registers at four channels per lane.
// ------------------------------------------------------------------------------------------
// acc[row0 + m3][c] += w[c] * sum_m1 A[m3][m1] xr[m1][c] (xr: the path's l1 rows only)
template <class Cfg, int P, int NROWS, int V>
__device__ __forceinline__ void tp_rows_acc(const float (&A)[Off<Cfg>::a[P + 1] - Off<Cfg>::a[P]],
                                            const float (&xr)[2 * Cfg::table.paths[P].l1 + 1][V],
                                            const float (&wv)[V], float (&acc)[NROWS][V], int row0) {
    constexpr int a0 = Off<Cfg>::a[P];
    constexpr int na = Off<Cfg>::a[P + 1] - a0;
    constexpr int n3 = 2 * Cfg::table.paths[P].l3 + 1;
    float t[n3][V];
#pragma unroll
    for (int m = 0; m < n3; ++m)
#pragma unroll
        for (int c = 0; c < V; ++c) t[m][c] = 0.f;
    sfor<na>([&](auto k) {
        constexpr AEnt e = Cfg::aents[a0 + decltype(k)::value];
#pragma unroll
        for (int c = 0; c < V; ++c) t[e.m3][c] = fmaf(A[decltype(k)::value], xr[e.m1][c], t[e.m3][c]);
    });
#pragma unroll
    for (int m = 0; m < n3; ++m)
#pragma unroll
        for (int c = 0; c < V; ++c) acc[row0 + m][c] = fmaf(wv[c], t[m][c], acc[row0 + m][c]);
}

// One output block at a time (the receiver's edge list is walked once per block, the edge
// rows of a block's paths read once), so only that block's rows are accumulated.
template <class Cfg, class T, int V>
__global__ void __launch_bounds__(256) conv_ddm_kernel(int64_t N, int64_t E, int Nq, const int32_t* __restrict__ rowptr,
                                                       const int32_t* __restrict__ sender, const T* __restrict__ x,
                                                       const T* __restrict__ y, const T* __restrict__ w,
                                                       const T* __restrict__ ddx, const T* __restrict__ ddy,
                                                       const T* __restrict__ ddw, float scale,
                                                       float* __restrict__ ddm, int64_t pad,
                                                       unsigned* __restrict__ err) {
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    for (int64_t b = warp * L.per_warp + L.grp; b < N; b += nwarp * L.per_warp) {
        int64_t e0 = __ldg(rowptr + b), e1 = __ldg(rowptr + b + 1);
        if (e0 < 0 || e1 < e0 || e1 > E) {
            if (L.gl == 0) atomicOr(err, kErrRowptr);
            e1 = e0 = 0;
        }
        if (b == pad) e0 = e1 = 0;
        sfor<Cfg::NOUT>([&](auto jj) {
            constexpr int j = decltype(jj)::value;
            constexpr int nrow = 2 * Cfg::table.outs[j].l + 1;
            float acc[nrow][V];
#pragma unroll
            for (int i = 0; i < nrow; ++i)
#pragma unroll
                for (int c = 0; c < V; ++c) acc[i][c] = 0.f;
            for (int64_t e = e0; e < e1; ++e) {
                const int64_t a = __ldg(sender + e);
                if (pad >= 0 && a == pad) continue;
                if (a < 0 || a >= N) {
                    if (j == 0 && L.gl == 0) atomicOr(err, kErrSender);
                    continue;
                }
                float yv[Cfg::D2], dyv[Cfg::D2];
#pragma unroll
                for (int i = 0; i < Cfg::D2; ++i) {
                    yv[i] = IO<T>::load1(y + e * Cfg::D2 + i);
                    dyv[i] = IO<T>::load1(ddy + e * Cfg::D2 + i);
                }
                sfor<Cfg::NP>([&](auto pp) {
                    constexpr int p = decltype(pp)::value;
                    constexpr PathInfo pi = Cfg::table.paths[p];
                    if constexpr (pi.out_block == j) {
                        constexpr int n1 = 2 * pi.l1 + 1;
                        constexpr int na = Off<Cfg>::a[p + 1] - Off<Cfg>::a[p];
                        float A[na], Ad[na];
                        build_A<Cfg, p>(yv, A);
                        build_A<Cfg, p>(dyv, Ad);
                        float xr[n1][V], dr[n1][V], wv[V], dwv[V];
#pragma unroll
                        for (int m = 0; m < n1; ++m) {
                            loadv<T, V>(x + (a * Cfg::D1 + pi.xoff + m) * Nq + c0, xr[m]);
                            loadv<T, V>(ddx + (a * Cfg::D1 + pi.xoff + m) * Nq + c0, dr[m]);
                        }
                        loadv<T, V>(w + (e * Cfg::NP + p) * Nq + c0, wv);
                        loadv<T, V>(ddw + (e * Cfg::NP + p) * Nq + c0, dwv);
                        tp_rows_acc<Cfg, p, nrow, V>(A, dr, wv, acc, 0);    // TP(ddx, y, w)
                        tp_rows_acc<Cfg, p, nrow, V>(Ad, xr, wv, acc, 0);   // TP(x, ddy, w)
                        tp_rows_acc<Cfg, p, nrow, V>(A, xr, dwv, acc, 0);   // TP(x, y, ddw)
                    }
                });
            }
            constexpr int zo = Off<Cfg>::z[j];
#pragma unroll
            for (int i = 0; i < nrow; ++i) {
#pragma unroll
                for (int c = 0; c < V; ++c) acc[i][c] *= scale;
                storev<V>(ddm + (b * Cfg::D + zo + i) * Nq + c0, acc[i]);
            }
        });
    }
}

// one edge of the sender pass: accumulates delta_x into gxa, the lane's partial delta_y into
// gyp and writes delta_w[e]
template <class Cfg, class T, int V>
__device__ __forceinline__ void dbackward_body(const T* __restrict__ x_a, const T* __restrict__ ddx_a,
                                               const float (&yv)[Cfg::D2], const float (&dyv)[Cfg::D2],
                                               const T* __restrict__ w_e, const T* __restrict__ ddw_e,
                                               const T* __restrict__ g_row, float gscale, float* __restrict__ gw_e,
                                               int Nq, int c0, float (&gxa)[Cfg::D1][V], float (&gyp)[Cfg::D2]) {
    sfor<Cfg::NOUT>([&](auto jj) {
        constexpr int j = decltype(jj)::value;
        constexpr int nrow = 2 * Cfg::table.outs[j].l + 1;
        constexpr int zo = Off<Cfg>::z[j];
        float g[nrow][V];
#pragma unroll
        for (int m = 0; m < nrow; ++m) {
            loadv<T, V>(g_row + (zo + m) * Nq + c0, g[m]);
#pragma unroll
            for (int c = 0; c < V; ++c) g[m][c] *= gscale;
        }
        sfor<Cfg::NP>([&](auto pp) {
            constexpr int p = decltype(pp)::value;
            constexpr PathInfo pi = Cfg::table.paths[p];
            if constexpr (pi.out_block == j) {
                constexpr int a0 = Off<Cfg>::a[p];
                constexpr int na = Off<Cfg>::a[p + 1] - a0;
                constexpr int n1 = 2 * pi.l1 + 1;
                float A[na], Ad[na];
                build_A<Cfg, p>(yv, A);
                build_A<Cfg, p>(dyv, Ad);
                float wv[V], dwv[V];
                loadv<T, V>(w_e + p * Nq + c0, wv);
                loadv<T, V>(ddw_e + p * Nq + c0, dwv);
                float xr[n1][V], dr[n1][V], u[n1][V], gy[n1][V], gd[n1][V];
#pragma unroll
                for (int m = 0; m < n1; ++m) {
                    loadv<T, V>(x_a + (pi.xoff + m) * Nq + c0, xr[m]);
                    loadv<T, V>(ddx_a + (pi.xoff + m) * Nq + c0, dr[m]);
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        u[m][c] = fmaf(dr[m][c], wv[c], xr[m][c] * dwv[c]);
                        gy[m][c] = 0.f;
                        gd[m][c] = 0.f;
                    }
                }
                sfor<na>([&](auto k) {
                    constexpr AEnt e = Cfg::aents[a0 + decltype(k)::value];
                    float s = 0.f;
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        gy[e.m1][c] = fmaf(A[decltype(k)::value], g[e.m3][c], gy[e.m1][c]);
                        gd[e.m1][c] = fmaf(Ad[decltype(k)::value], g[e.m3][c], gd[e.m1][c]);
                        s = fmaf(u[e.m1][c], g[e.m3][c], s);
                    }
                    sfor<e.nt>([&](auto t) {
                        constexpr int tt = decltype(t)::value;
                        gyp[pi.yoff + e.m2[tt]] = fmaf(e.c[tt], s, gyp[pi.yoff + e.m2[tt]]);
                    });
                });
                float gwv[V];
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    float s = 0.f;
#pragma unroll
                    for (int m = 0; m < n1; ++m) {
                        s = fmaf(dr[m][c], gy[m][c], s);
                        s = fmaf(xr[m][c], gd[m][c], s);
                        gxa[pi.xoff + m][c] = fmaf(wv[c], gd[m][c], fmaf(dwv[c], gy[m][c], gxa[pi.xoff + m][c]));
                    }
                    gwv[c] = s;
                }
                storev<V>(gw_e + p * Nq + c0, gwv);
            }
        });
    });
}

template <class Cfg, class T, int V>
__global__ void __launch_bounds__(256) conv_dbwd_kernel(
    int64_t N, int64_t E, int Nq, const int32_t* __restrict__ csc_ptr, const int32_t* __restrict__ csc_edge,
    const int32_t* __restrict__ csc_recv, const T* __restrict__ x, const T* __restrict__ y, const T* __restrict__ w,
    const T* __restrict__ dm, const T* __restrict__ ddx, const T* __restrict__ ddy, const T* __restrict__ ddw,
    float scale, float* __restrict__ gx, float* __restrict__ gy, float* __restrict__ gw, int64_t pad,
    unsigned* __restrict__ err) {
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    const int64_t iters = (N + nwarp * L.per_warp - 1) / (nwarp * L.per_warp);
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t a = (it * nwarp + warp) * L.per_warp + L.grp;
        const bool live = a < N;
        const int64_t aa = live ? a : 0;
        float gxa[Cfg::D1][V];
#pragma unroll
        for (int i = 0; i < Cfg::D1; ++i)
#pragma unroll
            for (int c = 0; c < V; ++c) gxa[i][c] = 0.f;
        int64_t k0 = 0, k1 = 0;
        if (live) {
            k0 = __ldg(csc_ptr + aa);
            k1 = __ldg(csc_ptr + aa + 1);
            if (k0 < 0 || k1 < k0 || k1 > E) {
                if (L.gl == 0) atomicOr(err, kErrRowptr);
                k0 = k1 = 0;
            }
            if (aa == pad) k0 = k1 = 0;
        }
        // the row groups of a warp may own different edge counts; loop to the warp maximum
        int64_t cnt = k1 - k0, wmax = cnt;
        for (int off = 16; off > 0; off >>= 1) {
            const int64_t o = __shfl_xor_sync(0xffffffffu, wmax, off);
            wmax = o > wmax ? o : wmax;
        }
        for (int64_t i = 0; i < wmax; ++i) {
            bool ok = i < cnt;
            int64_t e = 0, b = 0;
            if (ok) {
                e = __ldg(csc_edge + k0 + i);
                b = __ldg(csc_recv + k0 + i);
                if (pad >= 0 && b == pad) {
                    ok = false;   // padding edge: its rows are zeroed separately
                } else if (e < 0 || e >= E || b < 0 || b >= N) {
                    if (L.gl == 0) atomicOr(err, kErrRecv);
                    ok = false;
                }
            }
            float gyp[Cfg::D2];
#pragma unroll
            for (int t = 0; t < Cfg::D2; ++t) gyp[t] = 0.f;
            if (ok) {
                float yv[Cfg::D2], dyv[Cfg::D2];
#pragma unroll
                for (int t = 0; t < Cfg::D2; ++t) {
                    yv[t] = IO<T>::load1(y + e * Cfg::D2 + t);
                    dyv[t] = IO<T>::load1(ddy + e * Cfg::D2 + t);
                }
                dbackward_body<Cfg, T, V>(x + aa * Cfg::D1 * Nq, ddx + aa * Cfg::D1 * Nq, yv, dyv,
                                          w + e * Cfg::NP * Nq, ddw + e * Cfg::NP * Nq, dm + b * Cfg::D * Nq, scale,
                                          gw + e * Cfg::NP * Nq, Nq, c0, gxa, gyp);
            }
            group_reduce<Cfg::D2>(gyp, L.G);
            if (ok && L.gl == 0)
#pragma unroll
                for (int t = 0; t < Cfg::D2; ++t) gy[e * Cfg::D2 + t] = gyp[t];
        }
        if (live)
#pragma unroll
            for (int i = 0; i < Cfg::D1; ++i) storev<V>(gx + (aa * Cfg::D1 + i) * Nq + c0, gxa[i]);
    }
}

// ------------------------------------------------------------------------------------------
// host-side launch table of one configuration
// ------------------------------------------------------------------------------------------
struct Launch {
    int grid, block;
};

struct ConfigOps {
    uint32_t xcode;
    int L2, L3, per_path;
    int NP, D1, D2, D, NOUT, NR;
    const PathInfo* paths;
    const OutBlock* outs;
    const Rec* recs;
    // kernels (dtype 0 = fp32, 1 = bf16); each returns cudaError_t of the launch
    cudaError_t (*tp_fwd[2])(int64_t, int, const void*, const void*, const void*, void*, cudaStream_t);
    cudaError_t (*tp_bwd[2])(int64_t, int, const void*, const void*, const void*, const void*, void*, void*,
                             void*, cudaStream_t);
    // conv forward: ..., scale, m, pad, err, cap (CSR positions of a receiver it sums), stream
    cudaError_t (*conv_fwd[2])(int64_t, int64_t, int, const int32_t*, const int32_t*, const void*,
                               const void*, const void*, float, void*, int64_t, unsigned*, int64_t, cudaStream_t);
    cudaError_t (*conv_bwd[2])(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                               const void*, const void*, const void*, const void*, float, void*, void*,
                               void*, int64_t, unsigned*, cudaStream_t);
    // double backward: receiver CSR and sender-major index; x, y, w, dm, ddx, ddy, ddw in;
    // delta_x, delta_y, delta_w, delta_dm out
    cudaError_t (*conv_dbwd[2])(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                                const int32_t*, const int32_t*, const void*, const void*, const void*,
                                const void*, const void*, const void*, const void*, float, void*, void*, void*,
                                void*, int64_t, unsigned*, cudaStream_t);
    // radial convolution (fp32, hidden width kRadialHidden): forward (..., x, y, h, W2, scale, m,
    // pad, err, stream) and backward (..., x, y, h, W2, dm, scale, dx, dy, dh, pad, err, stream)
    cudaError_t (*conv_fwd_rad)(int64_t, int64_t, int, const int32_t*, const int32_t*, const float*,
                                const float*, const float*, const float*, float, float*, int64_t, unsigned*,
                                cudaStream_t);
    cudaError_t (*conv_bwd_rad)(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                                const float*, const float*, const float*, const float*, const float*, float,
                                float*, float*, float*, int64_t, unsigned*, cudaStream_t);
    // the further pieces of receivers with more than cap positions (after conv_fwd with that
    // cap): N, E, Nq, rowptr, sender, x, y, w, scale, m, pad, cap, workspace, err, stream
    cudaError_t (*conv_fwd_pieces[2])(int64_t, int64_t, int, const int32_t*, const int32_t*, const void*,
                                      const void*, const void*, float, void*, int64_t, int64_t, void*, unsigned*,
                                      cudaStream_t);
};

// hidden width of the radial network that the radial convolution kernels are built for
constexpr int kRadialHidden = 8;

int grid_for(const void* kernel, int block, int64_t items_per_block_unit, int64_t units, int smem = 0);
// exclusive scan of a[0..n) in place (graph.cu); sums: scan_sums_count(n) ints of scratch
cudaError_t exclusive_scan_i32(int32_t* a, int64_t n, int32_t* sums, cudaStream_t s);
size_t scan_sums_count(int64_t n);
int sm_count();

}  // namespace e3gb
