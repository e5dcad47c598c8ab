// Heavy receivers for the receiver-stationary forwards (e3gb_conv_forward_split).
#pragma once

#include "kernels.cuh"

namespace e3gb {

// ------------------------------------------------------------------------------------------
// Heavy receivers. Receiver-stationary summation gives a receiver with many edges to one warp
// ("e3j ...", Sec. 4 "Message passing convolution": deterministic receiver-stationary kernels
// meet the receiver-degree imbalance). With a cap, the forward kernels sum only the first cap
// CSR positions of a receiver into m; each further piece [e0 + j cap, e0 + (j+1) cap) of a
// heavier receiver is summed here into a partial row set of its own, and
// conv_pieces_combine_kernel adds the pieces to m[b] in piece order (fixed order, no atomics).
// cnt[b] = number of further pieces of b (cnt[N] = 0); its exclusive scan ptr gives piece k's
// receiver by binary search.
// ------------------------------------------------------------------------------------------
static __global__ void __launch_bounds__(256) piece_count_kernel(int64_t N, int64_t E, const int32_t* __restrict__ rowptr,
                                                          int64_t pad, int64_t cap, int32_t* __restrict__ cnt) {
    for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b <= N; b += int64_t(gridDim.x) * blockDim.x) {
        int64_t deg = 0;
        if (b < N && b != pad) {
            const int64_t e0 = __ldg(rowptr + b), e1 = __ldg(rowptr + b + 1);
            if (e0 >= 0 && e1 >= e0 && e1 <= E) deg = e1 - e0;   // a bad segment is flagged by the forward
        }
        cnt[b] = deg > cap ? int32_t((deg - 1) / cap) : 0;
    }
}

template <class Cfg, class T, int V>
__global__ void __launch_bounds__(256) conv_forward_pieces_kernel(
    int64_t N, int64_t E, int Nq, const int32_t* __restrict__ rowptr, const int32_t* __restrict__ sender,
    const T* __restrict__ x, const T* __restrict__ y, const T* __restrict__ w, int64_t pad, int64_t cap,
    const int32_t* __restrict__ ptr, float* __restrict__ partials, unsigned* __restrict__ err) {
    const Lanes L = lanes_for<V>(Nq);
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    const int c0 = L.gl * V;
    const int64_t total = __ldg(ptr + N);
    for (int64_t k = warp * L.per_warp + L.grp; k < total; k += nwarp * L.per_warp) {
        int64_t lo = 0, hi = N;   // the receiver: ptr[lo] <= k < ptr[lo + 1]
        while (hi - lo > 1) {
            const int64_t mid = (lo + hi) >> 1;
            if (__ldg(ptr + mid) <= k) lo = mid; else hi = mid;
        }
        const int64_t b = lo;
        const int64_t j = k - __ldg(ptr + b) + 1;
        const int64_t r1 = __ldg(rowptr + b + 1);
        const int64_t e0 = __ldg(rowptr + b) + j * cap;
        const int64_t e1 = e0 + cap < r1 ? e0 + cap : r1;
        float acc[Cfg::D][V];
#pragma unroll
        for (int i = 0; i < Cfg::D; ++i)
#pragma unroll
            for (int c = 0; c < V; ++c) acc[i][c] = 0.f;
        // the piece's edges one by one, loads in place; the next edge's weight rows (one
        // contiguous block) and x rows are prefetched into L2 a step ahead
        constexpr int kLine = 128;
        const size_t wbytes = size_t(Cfg::NP) * Nq * sizeof(T), xbytes = size_t(Cfg::D1) * Nq * sizeof(T);
        auto prefetch_edge = [&](int64_t e) {
            const unsigned char* wb = reinterpret_cast<const unsigned char*>(w + e * Cfg::NP * Nq);
            for (size_t o = size_t(L.gl) * kLine; o < wbytes; o += size_t(L.G) * kLine)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(wb + o));
            const int64_t a = __ldg(sender + e);
            if (a >= 0 && a < N) {
                const unsigned char* xb = reinterpret_cast<const unsigned char*>(x + a * Cfg::D1 * Nq);
                for (size_t o = size_t(L.gl) * kLine; o < xbytes; o += size_t(L.G) * kLine)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(xb + o));
            }
        };
        if (e0 < e1) prefetch_edge(e0);
        for (int64_t e = e0; e < e1; ++e) {
            if (e + 1 < e1) prefetch_edge(e + 1);
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
            sfor<Cfg::NP>([&](auto pp) {
                constexpr int p = decltype(pp)::value;
                float A[Off<Cfg>::a[p + 1] - Off<Cfg>::a[p]];
                build_A<Cfg, p>(yv, A);
                float wv[V];
                loadv<T, V>(w + (e * Cfg::NP + p) * Nq + c0, wv);
                apply_path<Cfg, p, Cfg::D, V>(A, xv, wv, acc, Cfg::table.paths[p].zoff);
            });
        }
#pragma unroll
        for (int i = 0; i < Cfg::D; ++i) storev<V>(partials + (k * Cfg::D + i) * Nq + c0, acc[i]);
    }
}

// m[b] += scale * (piece 1 + piece 2 + ...) for every receiver with pieces, in piece order.
// Thread (blockIdx.y * 256 + threadIdx.x) owns one of the row's D * Nq outputs and blocks stride
// over receivers, so a hub's outputs are summed by row / 256 blocks in parallel, each output
// over its pieces in order (the same sequence of multiply-adds for any launch shape).
static __global__ void __launch_bounds__(256) conv_pieces_combine_kernel(int64_t N, int64_t row, const int32_t* __restrict__ ptr,
                                                                  const float* __restrict__ partials, float scale,
                                                                  float* __restrict__ m) {
    const int64_t i = int64_t(blockIdx.y) * blockDim.x + threadIdx.x;
    if (i >= row) return;
    for (int64_t b = blockIdx.x; b < N; b += gridDim.x) {
        const int64_t k0 = __ldg(ptr + b), k1 = __ldg(ptr + b + 1);
        if (k1 <= k0) continue;
        float s = m[b * row + i];
        for (int64_t k = k0; k < k1; ++k) s = fmaf(scale, __ldg(partials + k * row + i), s);
        m[b * row + i] = s;
    }
}

}  // namespace e3gb
