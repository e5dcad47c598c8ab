// Convolution forward for narrow rows (4 to 32 channels): edge slots.
//
// With few channels the couplings A_p[m3][m1] = sum_m2 C y of an edge ("e3j ...", Eq. (13),
// the sum over the SH index taken first, as Alg. 2 takes the sum over records before applying
// the edge scalar) cost as much as applying them, so they should be built once per edge and
// shared by as many channels as possible. Here a lane owns 4 channels (G = Nq / 4 lanes per
// edge) and a warp works on SPR edges of the same receiver at once ("edge slots", up to 8),
// plus further receivers when Nq is small (Nq = 4, 8: 4 and 2 receivers per warp). Slot s of
// receiver b takes its (non-padding) edges s, s + SPR, ... (receiver-stationary, Alg. 2),
// accumulating all output rows of its 4 channels in registers; at the end the SPR partial sums
// are added across the slots with a transposing butterfly (fixed order: deterministic) and
// each lane stores the rows it ends up holding. Each lane computes the couplings of its edge
// from compile-time CG values next to their use, so the G lanes of an edge repeat that work
// (G = 2 at 8 channels) instead of every channel lane (the plain kernels' 8). Each lane copies
// its 4 channels of the next edge's sender x rows into its own double-buffered shared-memory
// slice with cp.async (no warp barrier: a lane reads only what it copied) and prefetches that
// edge's weights into L2.
#pragma once

#include "conv_pipe.cuh"

namespace e3gb {

template <int NQ>
struct Slots {
    static_assert(NQ % 4 == 0 && NQ >= 4 && NQ <= 32, "edge slots cover 4..32 channels");
    static constexpr int G = NQ / 4;             // lanes per edge (4 channels each)
    static constexpr int S = 32 / G;             // edges per warp
    static constexpr int SPR = S < 8 ? S : 8;    // edges per node
    static constexpr int NPW = S / SPR;          // nodes per warp
};

constexpr int pow2_at_least(int v) {
    int p = 1;
    while (p < v) p *= 2;
    return p;
}
constexpr int ilog2(int v) {
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

template <class Cfg>
struct SlotsFit {   // the output rows of one receiver in registers; staged x rows <= 128 KB
    static constexpr bool value = Cfg::D <= 32 && Cfg::D1 <= 16;
};
// receivers handled by one 256-thread block
template <int NQ>
constexpr int slots_nodes_per_block() { return 8 * Slots<NQ>::NPW; }
// staged x rows: [buffer][row][lane][4 channels] per warp, each lane reading only its own slice
constexpr int kSlotRow = 32 * 4;   // elements between rows of one buffer
template <class Cfg, class T>
constexpr int slots_fwd_smem() { return 8 * 2 * Cfg::D1 * kSlotRow * int(sizeof(T)); }


// Add R per-lane row quads (R a power of two >= SPR) over the SPR edge slots of a node: every
// step halves the rows a lane holds (it keeps one half and adds the partner slot's copy of
// it). Returns the first of the R / SPR consecutive rows that this lane then holds in v[0..].
template <int R, int SPR, int G>
__device__ __forceinline__ int slot_sum_transposed(Q2 (&v)[R], int es) {
    static_assert(R >= SPR && (R & (R - 1)) == 0, "R must be a power of two >= SPR");
    int row0 = 0;
    sfor<ilog2(SPR)>([&](auto ss) {
        constexpr int st = decltype(ss)::value;
        constexpr int bit = SPR >> (st + 1);      // slot bit exchanged in this step
        constexpr int half = R >> (st + 1);
        const bool upper = (es & bit) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const Q2 send = upper ? v[i] : v[i + half];
            const Q2 keep = upper ? v[i + half] : v[i];
            Q2 got;
            got.lo.x = __shfl_xor_sync(0xffffffffu, send.lo.x, bit * G);
            got.lo.y = __shfl_xor_sync(0xffffffffu, send.lo.y, bit * G);
            got.hi.x = __shfl_xor_sync(0xffffffffu, send.hi.x, bit * G);
            got.hi.y = __shfl_xor_sync(0xffffffffu, send.hi.y, bit * G);
            v[i] = {__fadd2_rn(keep.lo, got.lo), __fadd2_rn(keep.hi, got.hi)};
        }
        row0 += upper ? half : 0;
    });
    return row0;
}

// one coupling A[m3][m1] = sum_m2 C y of an entry, from compile-time CG values
template <class Cfg, int YOFF, AEnt E>
__device__ __forceinline__ float coupling(const float (&yv)[Cfg::D2]) {
    float s = E.c[0] * yv[YOFF + E.m2[0]];
    sfor<E.nt - 1>([&](auto t) {
        constexpr int tt = decltype(t)::value + 1;
        s = fmaf(E.c[tt], yv[YOFF + E.m2[tt]], s);
    });
    return s;
}

// Bring BYTES contiguous bytes at p (16-byte aligned) into L2 ahead of their loads; one
// instruction, no completion to wait for. Skipped when BYTES is not a multiple of 16.
template <int BYTES>
__device__ __forceinline__ void prefetch_l2(const void* p) {
    if constexpr (BYTES % 16 == 0 && BYTES > 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "n"(BYTES) : "memory");
}

template <class T>
__device__ __forceinline__ Q2 ldg_q2(const T* p) {
    float v[4];
    IO<T>::load4(p, v);
    return q2_of(v);
}

// y[e] (D2 values) into registers
template <class Cfg, class T>
__device__ __forceinline__ void load_y(const T* __restrict__ ye, float (&yv)[Cfg::D2]) {
    if constexpr (sizeof(T) == 4 && Cfg::D2 % 4 == 0) {
#pragma unroll
        for (int i = 0; i < Cfg::D2; i += 4) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(ye + i));
            yv[i] = t.x; yv[i + 1] = t.y; yv[i + 2] = t.z; yv[i + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < Cfg::D2; ++i) yv[i] = IO<T>::load1(ye + i);
    }
}

// ------------------------------------------------------------------------------------------
// forward
// ------------------------------------------------------------------------------------------
// acc[zoff + m3] += w * sum_m1 A[m3][m1] x[m1] for every path of one edge (4 channels); xs is
// this lane's staged copy of the sender's x rows (row r at xs + r * kSlotRow)
template <class Cfg, class T, int NQ, int R>
__device__ __forceinline__ void slots_edge_fwd(const T* __restrict__ xs, const float (&yv)[Cfg::D2],
                                               const T* __restrict__ we, Q2 (&acc)[R]) {
    sfor<Cfg::NP>([&](auto pp) {
        constexpr int p = decltype(pp)::value;
        constexpr PathInfo pi = Cfg::table.paths[p];
        constexpr int a0 = Off<Cfg>::a[p];
        constexpr int na = Off<Cfg>::a[p + 1] - a0;
        constexpr int n1 = 2 * pi.l1 + 1, n3 = 2 * pi.l3 + 1;
        constexpr int Z = pi.zoff;
        const Q2 wv = ldg_q2<T>(we + p * NQ);
        Q2 xr[n1];
#pragma unroll
        for (int m = 0; m < n1; ++m) xr[m] = lds_q2<T>(xs + (pi.xoff + m) * kSlotRow);
        if constexpr (n1 <= n3) {
#pragma unroll
            for (int m = 0; m < n1; ++m) xr[m] = q2_mul(xr[m], wv);
            sfor<na>([&](auto k) {
                constexpr int kk = decltype(k)::value;
                constexpr AEnt e = Cfg::aents[a0 + kk];
                const float a = coupling<Cfg, pi.yoff, e>(yv);
                acc[Z + e.m3] = q2_fma(make_float2(a, a), xr[e.m1], acc[Z + e.m3]);
            });
        } else {
            Q2 t[n3];
#pragma unroll
            for (int m = 0; m < n3; ++m) t[m] = q2_zero();
            sfor<na>([&](auto k) {
                constexpr int kk = decltype(k)::value;
                constexpr AEnt e = Cfg::aents[a0 + kk];
                const float a = coupling<Cfg, pi.yoff, e>(yv);
                t[e.m3] = q2_fma(make_float2(a, a), xr[e.m1], t[e.m3]);
            });
#pragma unroll
            for (int m = 0; m < n3; ++m) acc[Z + m] = q2_fma(wv, t[m], acc[Z + m]);
        }
    });
}

template <class Cfg, class T, int NQ>
__global__ void __launch_bounds__(256) conv_forward_slots_kernel(int64_t N, int64_t E,
                                                                 const int32_t* __restrict__ rowptr,
                                                                 const int32_t* __restrict__ sender,
                                                                 const T* __restrict__ x, const T* __restrict__ y,
                                                                 const T* __restrict__ w, float scale,
                                                                 float* __restrict__ m, int64_t pad,
                                                                 unsigned* __restrict__ err, int64_t cap) {
    using SL = Slots<NQ>;
    constexpr int R = pow2_at_least(Cfg::D > SL::SPR ? Cfg::D : SL::SPR);
    const int lane = threadIdx.x & 31;
    const int gl = lane % SL::G, es = (lane / SL::G) % SL::SPR, nl = lane / (SL::G * SL::SPR);
    const int c0 = gl * 4;
    const int64_t warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarp = (int64_t(gridDim.x) * blockDim.x) >> 5;
    extern __shared__ __align__(128) unsigned char slots_smem[];
    T* xs = reinterpret_cast<T*>(slots_smem) + (threadIdx.x >> 5) * (2 * Cfg::D1 * kSlotRow) + lane * 4;
    for (int64_t b0 = warp * SL::NPW; b0 < N; b0 += nwarp * SL::NPW) {   // warp-uniform
        const int64_t b = b0 + nl;
        int64_t e0 = 0, e1 = 0;
        if (b < N && b != pad) {
            e0 = __ldg(rowptr + b);
            e1 = __ldg(rowptr + b + 1);
            if (!seg_ok(e0, e1, E)) {
                if (lane % (SL::G * SL::SPR) == 0) atomicOr(err, kErrRowptr);
                e0 = e1 = 0;
            }
            if (e1 - e0 > cap) e1 = e0 + cap;   // the rest of a heavy receiver: the pieces kernel
        }
        Q2 acc[R];
#pragma unroll
        for (int i = 0; i < R; ++i) acc[i] = q2_zero();
        // Slot es takes the real (non-padding) edges of ranks es, es + SPR, ... of the segment, in
        // CSR order. Without a padding node these are the positions e0 + es, e0 + es + SPR, ...;
        // with one, each slot finds them by counting the segment's real edges, so the per-slot
        // sums, and with them the outputs, are bitwise those of the graph without the padding.
        int64_t q = e0, rank = 0;   // scan cursor and real edges before it (padding only)
        auto next_edge = [&](int64_t it) -> int64_t {
            if (pad < 0) {
                const int64_t e = e0 + it * SL::SPR + es;
                return e < e1 ? e : -1;
            }
            while (q < e1) {
                const int64_t j = q++;
                if (__ldg(sender + j) == pad) continue;
                if ((rank++ & (SL::SPR - 1)) == es) return j;
            }
            return -1;
        };
        // the sender's x rows of edge e (this lane's 4 channels) into buffer j, one edge ahead;
        // the weights of that edge into L2
        auto stage = [&](int64_t e, int j) {
            if (e >= 0) {
                const int64_t a = __ldg(sender + e);
                if (a >= 0 && a < N) {
                    const T* src = x + a * Cfg::D1 * NQ + c0;
#pragma unroll
                    for (int r = 0; r < Cfg::D1; ++r) cp_async_slice<T>(xs + (j * Cfg::D1 + r) * kSlotRow, src + r * NQ);
                }
                if (gl == 0) prefetch_l2<Cfg::NP * NQ * int(sizeof(T))>(w + e * Cfg::NP * NQ);
            }
            cp_async_commit();
        };
        int64_t cur = next_edge(0);
        stage(cur, 0);
        for (int64_t it = 0;; ++it) {
            if (!__any_sync(0xffffffffu, cur >= 0)) break;   // the warp runs to its largest node
            const int64_t nxt = next_edge(it + 1);
            stage(nxt, int((it + 1) & 1));
            cp_async_wait<1>();   // this lane's copies for cur are complete
            if (cur >= 0) {
                const int64_t a = __ldg(sender + cur);
                if (a < 0 || a >= N) {
                    if (gl == 0) atomicOr(err, kErrSender);
                } else {
                    float yv[Cfg::D2];
                    load_y<Cfg, T>(y + cur * Cfg::D2, yv);
                    slots_edge_fwd<Cfg, T, NQ, R>(xs + int(it & 1) * Cfg::D1 * kSlotRow, yv,
                                                  w + cur * Cfg::NP * NQ + c0, acc);
                }
            }
            cur = nxt;
        }
        cp_async_wait<0>();
        const int row0 = slot_sum_transposed<R, SL::SPR, SL::G>(acc, es);
        if (b < N) {
            const float2 sc = make_float2(scale, scale);
#pragma unroll
            for (int i = 0; i < R / SL::SPR; ++i) {
                const int row = row0 + i;
                if (row < Cfg::D) {
                    const float2 lo = __fmul2_rn(acc[i].lo, sc), hi = __fmul2_rn(acc[i].hi, sc);
                    *reinterpret_cast<float4*>(m + (b * Cfg::D + row) * NQ + c0) = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
            }
        }
    }
}

}  // namespace e3gb
