// Tensor product with runtime sparse coefficients ("e3j ...", App. E.1 Eq. (10)-(11) and
// Alg. 1: a COO list of records (i0, i1, i2, path, c)), forward and backward on rows:
//   z[r,i0,q] = sum_k c_k w[r,path_k,q] x[r,i1_k,q] y[r,i2_k]
// for any coefficient list (the Clebsch-Gordan product is one choice of records).
//
// Lanes own channels as in the compile-time kernels (one row group of Nq/V lanes per row).
// Two forms:
// - sorted plan (up to 8,192 records; index widths 11/10/11 bits): each block sorts the records
//   into its shared memory by output row (forward) or path (backward), stably, so the records
//   of one index form a run whose sum (z row; w and dw rows, and the dx row of consecutive
//   records of one x row) lives in registers;
// - the general form: the whole warp reads the records in the given order (broadcast loads
//   through L1) and each row group accumulates its outputs in its own shared-memory rows.
// In both, records may come in any order and repeat, every output row is written, each lane
// touches only its own channels, and the order of every sum is fixed (deterministic). Records
// whose indices fall outside (D, d1, d2, P) are skipped and flag the device error word (bit 8).
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

// ------------------------------------------------------------------------------------------
// Sorted-plan kernels. Every block first turns the record list into a plan in its shared
// memory: the valid records in stable order of one index (the forward's output row i0, the
// backward's path), each packed with its other three indices and its coefficient, plus
// the start of each index's run. A warp then walks the plan once per row: the run of one
// index accumulates in registers and is stored once, and the records of a run are
// independent, so the loop is unrolled and their loads overlap. The records come from
// shared memory instead of a dependent global load per record.
// ------------------------------------------------------------------------------------------
struct CooRec {
    uint32_t idx;   // the three other indices, 11 | 10 | 11 bits
    float c;
};
constexpr int kCooPlanMaxRec = 8192;

// warp 0 of the block: stable counting sort of the valid records by key into srec, run starts
// in rs[0..nkeys], scratch fill[nkeys]; returns true if a record was out of range. Forward:
// key i0, packed (i1, i2, path). Backward: key path, packed (i0, i2, i1).
__device__ bool coo_build_plan(bool bwd, int nrec, const int4* __restrict__ rec, const float* __restrict__ coef,
                               int D, int d1, int d2, int P, CooRec* srec, int* rs, int* fill) {
    const int lane = threadIdx.x & 31;
    const int nkeys = bwd ? P : D;
    bool flagged = false;
    for (int i = lane; i <= nkeys; i += 32) rs[i] = 0;
    for (int i = lane; i < nkeys; i += 32) fill[i] = 0;
    __syncwarp();
    for (int pass = 0; pass < 2; ++pass) {
        for (int base = 0; base < nrec; base += 32) {
            const int k = base + lane;
            bool valid = false;
            int key = 0;
            int4 t = make_int4(0, 0, 0, 0);
            if (k < nrec) {
                t = __ldg(rec + k);
                valid = (unsigned)t.x < (unsigned)D && (unsigned)t.y < (unsigned)d1 &&
                        (unsigned)t.z < (unsigned)d2 && (unsigned)t.w < (unsigned)P;
                flagged |= !valid;
                key = bwd ? t.w : t.x;
            }
            const unsigned vmask = __ballot_sync(0xffffffffu, valid);
            const unsigned peers = __match_any_sync(0xffffffffu, valid ? key : -1) & vmask;
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const bool leader = valid && rank == 0;
            if (pass == 0) {
                if (leader) rs[key + 1] += __popc(peers);
            } else if (valid) {
                const uint32_t packed = bwd ? (uint32_t(t.x) | uint32_t(t.z) << 11 | uint32_t(t.y) << 21)
                                            : (uint32_t(t.y) | uint32_t(t.z) << 11 | uint32_t(t.w) << 21);
                srec[rs[key] + fill[key] + rank] = CooRec{packed, __ldg(coef + k)};
            }
            __syncwarp();
            if (pass == 1 && leader) fill[key] += __popc(peers);
            __syncwarp();
        }
        if (pass == 0) {
            if (lane == 0)
                for (int i = 0; i < nkeys; ++i) rs[i + 1] += rs[i];
            __syncwarp();
        }
    }
    return __any_sync(0xffffffffu, flagged);
}

template <class T, int V>
__global__ void __launch_bounds__(256, 4) coo_plan_forward_kernel(int64_t R, int d1, int d2, int D, int P, int Nq,
                                                               int nrec, const int4* __restrict__ rec,
                                                               const float* __restrict__ coef,
                                                               const T* __restrict__ x, const T* __restrict__ y,
                                                               const T* __restrict__ w, float* __restrict__ z,
                                                               unsigned* __restrict__ err) {
    extern __shared__ __align__(16) unsigned char sm[];
    CooRec* srec = reinterpret_cast<CooRec*>(sm);
    int* rs = reinterpret_cast<int*>(srec + nrec);
    int* fill = rs + D + 1;
    if (threadIdx.x < 32) {
        const bool flagged = coo_build_plan(false, nrec, rec, coef, D, d1, d2, P, srec, rs, fill);
        if (flagged && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(err, kErrRecord);
    }
    __syncthreads();
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    const int64_t iters = (R + nwarp * L.per_warp - 1) / (nwarp * L.per_warp);
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = (it * nwarp + warp) * L.per_warp + L.grp;
        const bool live = r < R;
        const int64_t rr = live ? r : 0;
        const T* xr = x + rr * d1 * Nq + c0;
        const T* wr = w + rr * P * Nq + c0;
        const T* yr = y + rr * d2;
        for (int i0 = 0; i0 < D; ++i0) {
            const int k0 = rs[i0], k1 = rs[i0 + 1];
            float acc[V];
#pragma unroll
            for (int c = 0; c < V; ++c) acc[c] = 0.f;
#pragma unroll 4
            for (int k = k0; k < k1; ++k) {
                const CooRec q = srec[k];
                const int i1 = q.idx & 0x7ff, i2 = (q.idx >> 11) & 0x3ff, p = q.idx >> 21;
                float xv[V], wv[V];
                loadv<T, V>(xr + i1 * Nq, xv);
                loadv<T, V>(wr + p * Nq, wv);
                const float cy = q.c * IO<T>::load1(yr + i2);
#pragma unroll
                for (int c = 0; c < V; ++c) acc[c] = fmaf(cy * wv[c], xv[c], acc[c]);
            }
            if (live) storev<V>(z + (rr * D + i0) * Nq + c0, acc);
        }
    }
}

template <class T, int V>
__global__ void __launch_bounds__(256, 3) coo_plan_backward_kernel(int64_t R, int d1, int d2, int D, int P, int Nq,
                                                                   int nrec, const int4* __restrict__ rec,
                                                                   const float* __restrict__ coef,
                                                                   const T* __restrict__ x, const T* __restrict__ y,
                                                                   const T* __restrict__ w, const T* __restrict__ dz,
                                                                   float* __restrict__ dx, float* __restrict__ dy,
                                                                   float* __restrict__ dw, unsigned* __restrict__ err) {
    extern __shared__ __align__(16) unsigned char sm[];
    CooRec* srec = reinterpret_cast<CooRec*>(sm);
    int* rs = reinterpret_cast<int*>(srec + nrec);
    int* fill = rs + P + 1;
    // per warp: dx rows of its row groups [per_warp][d1][Nq] (each lane its own channels),
    // then per-lane dy partials [d2][32]; the path runs keep w and dw in registers
    const Lanes L = lanes_for<V>(Nq);
    const int wib = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const size_t plan_bytes = (size_t(nrec) * sizeof(CooRec) + size_t(2 * P + 1) * 4 + 15) / 16 * 16;
    float* wsm = reinterpret_cast<float*>(sm + plan_bytes) + size_t(wib) * (size_t(32 * V) * d1 + 32 * d2);
    float* gx = wsm + size_t(L.grp) * d1 * Nq;
    float* dyl = wsm + size_t(32 * V) * d1;
    if (threadIdx.x < 32) {
        const bool flagged = coo_build_plan(true, nrec, rec, coef, D, d1, d2, P, srec, rs, fill);
        if (flagged && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(err, kErrRecord);
    }
    __syncthreads();
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    const int64_t iters = (R + nwarp * L.per_warp - 1) / (nwarp * L.per_warp);
    for (int64_t it = 0; it < iters; ++it) {
        const int64_t r = (it * nwarp + warp) * L.per_warp + L.grp;
        const bool live = r < R;
        const int64_t rr = live ? r : 0;
        const T* xr = x + rr * d1 * Nq + c0;
        const T* dzr = dz + rr * D * Nq + c0;
        const T* yr = y + rr * d2;
        for (int i = 0; i < d1; ++i)
#pragma unroll
            for (int c = 0; c < V; ++c) gx[i * Nq + c0 + c] = 0.f;
        for (int i = 0; i < d2; ++i) dyl[i * 32 + lane] = 0.f;
        for (int p = 0; p < P; ++p) {
            const int k0 = rs[p], k1 = rs[p + 1];
            float wv[V], dwp[V];
            loadv<T, V>(w + (rr * P + p) * Nq + c0, wv);
#pragma unroll
            for (int c = 0; c < V; ++c) dwp[c] = 0.f;
            // consecutive records of one x row (the usual order inside a path) load it once and
            // add their dx share in registers, flushed to the shared dx row when the row changes
            int cur_i1 = -1;
            float xv[V], dxr[V];
#pragma unroll
            for (int c = 0; c < V; ++c) xv[c] = dxr[c] = 0.f;
#pragma unroll 4
            for (int k = k0; k < k1; ++k) {
                const CooRec q = srec[k];
                const int i0 = q.idx & 0x7ff, i2 = (q.idx >> 11) & 0x3ff, i1 = q.idx >> 21;
                if (i1 != cur_i1) {   // warp-uniform: every lane reads the same record
                    if (cur_i1 >= 0)
#pragma unroll
                        for (int c = 0; c < V; ++c) gx[cur_i1 * Nq + c0 + c] += dxr[c];
                    loadv<T, V>(xr + i1 * Nq, xv);
#pragma unroll
                    for (int c = 0; c < V; ++c) dxr[c] = 0.f;
                    cur_i1 = i1;
                }
                float gv[V];
                loadv<T, V>(dzr + i0 * Nq, gv);
                const float yv = IO<T>::load1(yr + i2);
                float s = 0.f;
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    const float g = q.c * gv[c];
                    const float gy = g * yv;
                    dxr[c] = fmaf(gy, wv[c], dxr[c]);     // dx[i1]
                    dwp[c] = fmaf(gy, xv[c], dwp[c]);     // dw[path]
                    s = fmaf(g * wv[c], xv[c], s);        // dy[i2] partial
                }
                dyl[i2 * 32 + lane] += s;
            }
            if (cur_i1 >= 0)
#pragma unroll
                for (int c = 0; c < V; ++c) gx[cur_i1 * Nq + c0 + c] += dxr[c];
            if (live) storev<V>(dw + (rr * P + p) * Nq + c0, dwp);   // every path row, zero without records
        }
        __syncwarp();
        if (live)
            for (int i = 0; i < d1; ++i) {
                float o[V];
#pragma unroll
                for (int c = 0; c < V; ++c) o[c] = gx[i * Nq + c0 + c];
                storev<V>(dx + (rr * d1 + i) * Nq + c0, o);
            }
        // dy: sum each partial over the G lanes of the row group (fixed butterfly order)
        for (int i = 0; i < d2; ++i) {
            float v = dyl[i * 32 + lane];
            for (int off = L.G >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (live && L.gl == 0) dy[rr * d2 + i] = v;
        }
        __syncwarp();
    }
}

int sm_count_here() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

constexpr int kCooBlock = 256;

}  // namespace

// shared-memory bytes of one launch of the original kernels (0: shape not supported)
size_t coo_smem_bytes(bool backward, int d1, int d2, int D, int P, int Nq) {
    const int V = Nq >= 64 ? 4 : 1;
    const int rows_per_block = (kCooBlock / 32) * (32 / (Nq / V));
    if (!backward) return size_t(rows_per_block) * D * Nq * 4;
    return size_t(rows_per_block) * (d1 + P) * Nq * 4 + size_t(kCooBlock / 32) * d2 * 32 * 4;
}

namespace {
// shared-memory bytes of a sorted-plan launch, or 0 when its limits are exceeded (the record
// count, the packed index widths, the block's shared memory)
size_t coo_plan_smem_bytes(bool backward, int nrec, int d1, int d2, int D, int P, int Nq) {
    if (nrec > kCooPlanMaxRec || d2 > 1024 || d1 > 2048 || (backward ? D : P) > 2048) return 0;
    const int keys = backward ? P : D;
    const size_t plan = (size_t(nrec) * sizeof(CooRec) + size_t(2 * keys + 1) * 4 + 15) / 16 * 16;
    const int V = Nq >= 64 ? 4 : 1;
    const size_t per_warp = backward ? (size_t(32 * V) * d1 + 32 * size_t(d2)) * 4 : 0;
    const size_t total = plan + (kCooBlock / 32) * per_warp;
    return total <= 232448 ? total : 0;
}
}  // namespace

template <class T>
cudaError_t coo_tp(bool backward, int64_t R, int d1, int d2, int D, int P, int Nq, int nrec, const int32_t* rec,
                   const float* coef, const void* x, const void* y, const void* w, const void* dz, void* z_or_dx,
                   void* dy, void* dw, unsigned* err, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    const int V = Nq >= 64 ? 4 : 1;
    const int rows_per_block = (kCooBlock / 32) * (32 / (Nq / V));
    const int64_t need = (R + rows_per_block - 1) / rows_per_block;
    const int sms = sm_count_here();
    if (sms == 0) return cudaErrorInvalidDevice;
    const int4* r4 = reinterpret_cast<const int4*>(rec);
    cudaError_t st;
    const size_t plan_smem = coo_plan_smem_bytes(backward, nrec, d1, d2, D, P, Nq);
    if (plan_smem > 0) {   // sorted plan in shared memory; persistent grid of resident blocks
        const void* k = !backward ? (V == 4 ? (const void*)coo_plan_forward_kernel<T, 4> : (const void*)coo_plan_forward_kernel<T, 1>)
                                  : (V == 4 ? (const void*)coo_plan_backward_kernel<T, 4> : (const void*)coo_plan_backward_kernel<T, 1>);
        st = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(plan_smem));
        if (st != cudaSuccess) return st;
        int per_sm = 0;
        st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kCooBlock, plan_smem);
        if (st != cudaSuccess) return st;
        if (per_sm < 1) per_sm = 1;
        const int grid = int(need < int64_t(sms) * per_sm ? need : int64_t(sms) * per_sm);
        if (!backward) {
            auto kk = V == 4 ? coo_plan_forward_kernel<T, 4> : coo_plan_forward_kernel<T, 1>;
            kk<<<grid, kCooBlock, plan_smem, s>>>(R, d1, d2, D, P, Nq, nrec, r4, coef, (const T*)x, (const T*)y,
                                                   (const T*)w, (float*)z_or_dx, err);
        } else {
            auto kk = V == 4 ? coo_plan_backward_kernel<T, 4> : coo_plan_backward_kernel<T, 1>;
            kk<<<grid, kCooBlock, plan_smem, s>>>(R, d1, d2, D, P, Nq, nrec, r4, coef, (const T*)x, (const T*)y,
                                                   (const T*)w, (const T*)dz, (float*)z_or_dx, (float*)dy,
                                                   (float*)dw, err);
        }
        return cudaGetLastError();
    }
    const size_t smem = coo_smem_bytes(backward, d1, d2, D, P, Nq);
    const int grid = int(need < int64_t(sms) * 2 ? need : int64_t(sms) * 2);
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
