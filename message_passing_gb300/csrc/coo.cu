// Tensor product with runtime sparse coefficients ("e3j ...", App. E.1 Eq. (10)-(11) and
// Alg. 1: a COO list of records (i0, i1, i2, path, c)), forward and backward on rows:
//   z[r,i0,q] = sum_k c_k w[r,path_k,q] x[r,i1_k,q] y[r,i2_k]
// for any coefficient list (the Clebsch-Gordan product is one choice of records).
//
// Lanes own channels as in the compile-time kernels (one row group of Nq/V lanes per row).
// The records are read by the whole warp in the same order (broadcast loads through L1);
// each row group accumulates its outputs in its own shared-memory rows, each lane touching
// only its own channels, so the records may come in any order, repeat, and no output row is
// left unwritten. Records whose indices fall outside (D, d1, d2, P) are skipped and flag the
// device error word (bit 8).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.cuh"

namespace e3gb {

constexpr unsigned kErrRecord = 8u;

namespace {

template <class T, int V>
__global__ void __launch_bounds__(256) coo_tp_forward_kernel(int64_t R, int d1, int d2, int D, int P, int Nq, int nrec,
                                                             const int4* __restrict__ rec,
                                                             const float* __restrict__ coef, const T* __restrict__ x,
                                                             const T* __restrict__ y, const T* __restrict__ w,
                                                             float* __restrict__ z, unsigned* __restrict__ err) {
    extern __shared__ float zs_all[];
    const Lanes L = lanes_for<V>(Nq);
    const int wib = threadIdx.x >> 5;
    float* zs = zs_all + (wib * L.per_warp + L.grp) * (D * Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    bool flagged = false;
    // same trip count for every lane of the warp (the record loop is warp-uniform)
    const int64_t iters = (R + nwarp * L.per_warp - 1) / (nwarp * L.per_warp);
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = (it * nwarp + warp) * L.per_warp + L.grp;
        const bool live = r < R;
        const int64_t rr = live ? r : 0;
        for (int i = 0; i < D; ++i)
#pragma unroll
            for (int c = 0; c < V; ++c) zs[i * Nq + c0 + c] = 0.f;
        for (int k = 0; k < nrec; ++k) {
            const int4 t = __ldg(rec + k);   // (i0, i1, i2, path)
            if ((unsigned)t.x >= (unsigned)D || (unsigned)t.y >= (unsigned)d1 || (unsigned)t.z >= (unsigned)d2 ||
                (unsigned)t.w >= (unsigned)P) {
                flagged = true;
                continue;
            }
            if (!live) continue;
            const float cy = __ldg(coef + k) * IO<T>::load1(y + rr * d2 + t.z);
            float xv[V], wv[V];
            loadv<T, V>(x + (rr * d1 + t.y) * Nq + c0, xv);
            loadv<T, V>(w + (rr * P + t.w) * Nq + c0, wv);
#pragma unroll
            for (int c = 0; c < V; ++c) zs[t.x * Nq + c0 + c] = fmaf(cy * wv[c], xv[c], zs[t.x * Nq + c0 + c]);
        }
        if (live)
            for (int i = 0; i < D; ++i) {
                float o[V];
#pragma unroll
                for (int c = 0; c < V; ++c) o[c] = zs[i * Nq + c0 + c];
                storev<V>(z + (rr * D + i) * Nq + c0, o);
            }
    }
    if (flagged && L.gl == 0) atomicOr(err, kErrRecord);
}

template <class T, int V>
__global__ void __launch_bounds__(256) coo_tp_backward_kernel(int64_t R, int d1, int d2, int D, int P, int Nq,
                                                              int nrec, const int4* __restrict__ rec,
                                                              const float* __restrict__ coef, const T* __restrict__ x,
                                                              const T* __restrict__ y, const T* __restrict__ w,
                                                              const T* __restrict__ dz, float* __restrict__ dx,
                                                              float* __restrict__ dy, float* __restrict__ dw,
                                                              unsigned* __restrict__ err) {
    extern __shared__ float s_all[];
    const Lanes L = lanes_for<V>(Nq);
    const int wib = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // per row group: dx rows [d1][Nq], dw rows [P][Nq], then per-lane dy partials [d2][32]
    const int group_floats = (d1 + P) * Nq;
    float* gs = s_all + (wib * L.per_warp + L.grp) * group_floats;
    float* dyl = s_all + (blockDim.x >> 5) * L.per_warp * group_floats + wib * (d2 * 32);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    bool flagged = false;
    const int64_t iters = (R + nwarp * L.per_warp - 1) / (nwarp * L.per_warp);
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = (it * nwarp + warp) * L.per_warp + L.grp;
        const bool live = r < R;
        const int64_t rr = live ? r : 0;
        for (int i = 0; i < d1 + P; ++i)
#pragma unroll
            for (int c = 0; c < V; ++c) gs[i * Nq + c0 + c] = 0.f;
        for (int i = 0; i < d2; ++i) dyl[i * 32 + lane] = 0.f;
        for (int k = 0; k < nrec; ++k) {
            const int4 t = __ldg(rec + k);
            if ((unsigned)t.x >= (unsigned)D || (unsigned)t.y >= (unsigned)d1 || (unsigned)t.z >= (unsigned)d2 ||
                (unsigned)t.w >= (unsigned)P) {
                flagged = true;
                continue;
            }
            if (!live) continue;
            const float ck = __ldg(coef + k);
            const float yv = IO<T>::load1(y + rr * d2 + t.z);
            float xv[V], wv[V], gv[V];
            loadv<T, V>(x + (rr * d1 + t.y) * Nq + c0, xv);
            loadv<T, V>(w + (rr * P + t.w) * Nq + c0, wv);
            loadv<T, V>(dz + (rr * D + t.x) * Nq + c0, gv);
            float s = 0.f;
#pragma unroll
            for (int c = 0; c < V; ++c) {
                const float g = ck * gv[c];
                const float gy = g * yv;
                gs[t.y * Nq + c0 + c] = fmaf(gy, wv[c], gs[t.y * Nq + c0 + c]);          // dx[i1]
                gs[(d1 + t.w) * Nq + c0 + c] = fmaf(gy, xv[c], gs[(d1 + t.w) * Nq + c0 + c]);   // dw[path]
                s = fmaf(g * wv[c], xv[c], s);                                            // dy[i2] partial
            }
            dyl[t.z * 32 + lane] += s;
        }
        if (live) {
            for (int i = 0; i < d1; ++i) {
                float o[V];
#pragma unroll
                for (int c = 0; c < V; ++c) o[c] = gs[i * Nq + c0 + c];
                storev<V>(dx + (rr * d1 + i) * Nq + c0, o);
            }
            for (int p = 0; p < P; ++p) {
                float o[V];
#pragma unroll
                for (int c = 0; c < V; ++c) o[c] = gs[(d1 + p) * Nq + c0 + c];
                storev<V>(dw + (rr * P + p) * Nq + c0, o);
            }
        }
        // dy: sum each partial over the G lanes of the row group (fixed butterfly order)
        for (int i = 0; i < d2; ++i) {
            float v = dyl[i * 32 + lane];
            for (int off = L.G >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (live && L.gl == 0) dy[rr * d2 + i] = v;
        }
    }
    if (flagged && L.gl == 0) atomicOr(err, kErrRecord);
}

int sm_count_here() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

constexpr int kCooBlock = 256;

}  // namespace

// shared-memory bytes of one launch (0: shape not supported)
size_t coo_smem_bytes(bool backward, int d1, int d2, int D, int P, int Nq) {
    const int V = Nq >= 64 ? 4 : 1;
    const int rows_per_block = (kCooBlock / 32) * (32 / (Nq / V));
    if (!backward) return size_t(rows_per_block) * D * Nq * 4;
    return size_t(rows_per_block) * (d1 + P) * Nq * 4 + size_t(kCooBlock / 32) * d2 * 32 * 4;
}

template <class T>
cudaError_t coo_tp(bool backward, int64_t R, int d1, int d2, int D, int P, int Nq, int nrec, const int32_t* rec,
                   const float* coef, const void* x, const void* y, const void* w, const void* dz, void* z_or_dx,
                   void* dy, void* dw, unsigned* err, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    const int V = Nq >= 64 ? 4 : 1;
    const size_t smem = coo_smem_bytes(backward, d1, d2, D, P, Nq);
    const int rows_per_block = (kCooBlock / 32) * (32 / (Nq / V));
    const int64_t need = (R + rows_per_block - 1) / rows_per_block;
    const int sms = sm_count_here();
    if (sms == 0) return cudaErrorInvalidDevice;
    const int grid = int(need < int64_t(sms) * 2 ? need : int64_t(sms) * 2);
    const int4* r4 = reinterpret_cast<const int4*>(rec);
    cudaError_t st;
    if (!backward) {
        auto k = V == 4 ? coo_tp_forward_kernel<T, 4> : coo_tp_forward_kernel<T, 1>;
        st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (st != cudaSuccess) return st;
        k<<<grid, kCooBlock, smem, s>>>(R, d1, d2, D, P, Nq, nrec, r4, coef, (const T*)x, (const T*)y, (const T*)w,
                                         (float*)z_or_dx, err);
    } else {
        auto k = V == 4 ? coo_tp_backward_kernel<T, 4> : coo_tp_backward_kernel<T, 1>;
        st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (st != cudaSuccess) return st;
        k<<<grid, kCooBlock, smem, s>>>(R, d1, d2, D, P, Nq, nrec, r4, coef, (const T*)x, (const T*)y, (const T*)w,
                                         (const T*)dz, (float*)z_or_dx, (float*)dy, (float*)dw, err);
    }
    return cudaGetLastError();
}

template cudaError_t coo_tp<float>(bool, int64_t, int, int, int, int, int, int, const int32_t*, const float*,
                                   const void*, const void*, const void*, const void*, void*, void*, void*, unsigned*,
                                   cudaStream_t);
template cudaError_t coo_tp<__nv_bfloat16>(bool, int64_t, int, int, int, int, int, int, const int32_t*, const float*,
                                           const void*, const void*, const void*, const void*, void*, void*, void*,
                                           unsigned*, cudaStream_t);

}  // namespace e3gb
