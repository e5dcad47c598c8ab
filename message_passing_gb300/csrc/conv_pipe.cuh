// Convolution kernels for 128 channels with per-warp asynchronous prefetch.
//
// Every warp works alone on one receiver (forward, "e3j ...", Alg. 2: receiver-stationary
// accumulation) or one sender (backward, the transposed graph of Eq. 16), with all 128
// channels (4 per lane) and every output row in registers, exactly like the plain kernels in
// kernels.cuh. What changes is how operands arrive: the warp walks a flat sequence of
// "items" (pieces of its edges) and keeps the next NSLOT-1 items in flight in a private
// shared-memory ring with cp.async, each lane copying the 16-byte channel slice it will
// itself read. No warp ever waits for another warp, all warps run the same code, and the
// bytes in flight per SM are (warps per SM) x (NSLOT-1) items regardless of registers.
//
//   forward items per edge:   [x rows of the sender + y]  [w rows of paths chunk 0] ...
//   backward items per sender: [x rows of the sender]; per edge: [y + dm rows + w rows of the
//                              paths of output block 0] [output block 1] ...
//
// Per edge the warp first turns y into the couplings A_p[m3][m1] = sum_m2 C y (a few
// entries per lane from a recipe table, stored to the warp's shared A buffer); the channel
// loops then read A as broadcast float4 loads. A sequence position i always uses ring slot
// i % NSLOT; the issue of item i + NSLOT - 1 overwrites the slot of item i - 1, which this
// lane has finished reading.
#pragma once

#include "kernels.cuh"

namespace e3gb {

constexpr int kPipeNq = 128;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte (fp32 x4) or 8-byte (bf16 x4) asynchronous copy of one lane's channel slice
template <class T>
__device__ __forceinline__ void cp_async_slice(void* dst, const void* src);
template <>
__device__ __forceinline__ void cp_async_slice<float>(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
template <>
__device__ __forceinline__ void cp_async_slice<__nv_bfloat16>(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// L2 policy for operands read exactly once (the edge weights): their lines go first when L2
// needs room, which keeps the gathered node rows (x, dm) resident longer
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// cp_async_slice with an L2 cache policy
template <class T>
__device__ __forceinline__ void cp_async_slice_hint(void* dst, const void* src, uint64_t pol);
template <>
__device__ __forceinline__ void cp_async_slice_hint<float>(void* dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "l"(pol) : "memory");
}
template <>
__device__ __forceinline__ void cp_async_slice_hint<__nv_bfloat16>(void* dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2;" ::"r"(smem_u32(dst)), "l"(src), "l"(pol) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <class T>
__device__ __forceinline__ void lds4(const T* p, float (&o)[4]);
template <>
__device__ __forceinline__ void lds4<float>(const float* p, float (&o)[4]) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
}
template <>
__device__ __forceinline__ void lds4<__nv_bfloat16>(const __nv_bfloat16* p, float (&o)[4]) {
    const uint2 t = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.y));
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
}

// ------------------------------------------------------------------------------------------
// compile-time plan
// ------------------------------------------------------------------------------------------
template <class Cfg>
struct PipePlan {
    // A entries of path p at apos[p] (a multiple of 4 floats) in the warp's A buffer
    static constexpr std::array<int, Cfg::NP + 1> apos = [] {
        std::array<int, Cfg::NP + 1> a{};
        for (int p = 0; p < Cfg::NP; ++p) {
            const int na = Off<Cfg>::a[p + 1] - Off<Cfg>::a[p];
            a[p + 1] = a[p] + (na + 3) / 4 * 4;
        }
        return a;
    }();
    static constexpr int NAPAD = apos[Cfg::NP];
    // forward order of the A entries inside each path: m1-major, so that consecutive
    // multiply-adds update different accumulator rows (independent chains)
    static constexpr std::array<int, Cfg::NA> fwd_order = [] {
        std::array<int, Cfg::NA> o{};
        for (int p = 0; p < Cfg::NP; ++p) {
            int n = Off<Cfg>::a[p];
            for (int m1 = 0; m1 < 7; ++m1)
                for (int k = Off<Cfg>::a[p]; k < Off<Cfg>::a[p + 1]; ++k)
                    if (Cfg::aents[k].m1 == m1) o[n++] = k;
        }
        return o;
    }();
    // forward: w rows in NWC chunks of PPC paths
    static constexpr int PPC = 8;   // measured: 4 / 6 / 8 / 12 / 24 paths per chunk -> 8 fastest
    static constexpr int NWC = (Cfg::NP + PPC - 1) / PPC;
    // backward: the paths of each output block, in path order
    static constexpr std::array<int, Cfg::NOUT + 1> bpos = [] {   // offsets into bpath
        std::array<int, Cfg::NOUT + 1> o{};
        for (int p = 0; p < Cfg::NP; ++p) o[Cfg::table.paths[p].out_block + 1]++;
        for (int j = 0; j < Cfg::NOUT; ++j) o[j + 1] += o[j];
        return o;
    }();
    static constexpr std::array<int, Cfg::NP> bpath = [] {
        std::array<int, Cfg::NP> b{};
        int fill[Cfg::NOUT + 1] = {};
        for (int p = 0; p < Cfg::NP; ++p) {
            const int j = Cfg::table.paths[p].out_block;
            b[bpos[j] + fill[j]++] = p;
        }
        return b;
    }();
    static constexpr int max_block_rows = [] {
        int m = 0;
        for (int j = 0; j < Cfg::NOUT; ++j) {
            const int r = (2 * Cfg::table.outs[j].l + 1) + (bpos[j + 1] - bpos[j]);
            m = r > m ? r : m;
        }
        return m;
    }();
};

// one A entry: A[pos] = c0 y[i0] (+ c1 y[i1])
struct alignas(16) Recipe {
    float c0, c1;
    int idx;   // i0 | i1 << 8 | nterms << 16
    int pos;
};
template <class Cfg>
struct RecipeTable {
    Recipe r[Cfg::NA];
};
// FWD: entries placed in forward order (PipePlan::fwd_order), else in table order
template <class Cfg, bool FWD>
constexpr RecipeTable<Cfg> make_recipes() {
    RecipeTable<Cfg> t{};
    for (int p = 0; p < Cfg::NP; ++p) {
        const int a0 = Off<Cfg>::a[p];
        const int yo = Cfg::table.paths[p].yoff;
        for (int k = a0; k < Off<Cfg>::a[p + 1]; ++k) {
            const int src = FWD ? PipePlan<Cfg>::fwd_order[k] : k;
            const AEnt& e = Cfg::aents[src];
            Recipe r{};
            r.c0 = e.c[0];
            r.c1 = e.nt > 1 ? e.c[1] : 0.f;
            r.idx = (yo + e.m2[0]) | ((yo + (e.nt > 1 ? e.m2[1] : e.m2[0])) << 8) | (e.nt << 16);
            r.pos = PipePlan<Cfg>::apos[p] + (k - a0);
            t.r[k] = r;
        }
    }
    return t;
}
template <class Cfg, bool FWD>
__device__ const RecipeTable<Cfg> kRecipes = make_recipes<Cfg, FWD>();

// A entries of one edge, built by the 32 lanes of a warp from y in shared memory (the
// buffer is addressed as floats; the float2 type only gives it 8-byte units). The channel
// loops read four entries per 16-byte load and broadcast each into an (A, A) operand pair
// of the paired (f32x2) multiply-adds.
template <class Cfg, bool FWD, class T>
__device__ __forceinline__ void build_A_warp(const T* __restrict__ sy, float2* __restrict__ sA, int lane,
                                             float mul = 1.f) {
#pragma unroll   // fully unrolled: the recipe loads of all entries issue together (measured)
    for (int i = lane; i < Cfg::NA; i += 32) {
        const Recipe r = kRecipes<Cfg, FWD>.r[i];
        const int i0 = r.idx & 0xff, i1 = (r.idx >> 8) & 0xff;
        float v = r.c0 * float(sy[i0]);
        if ((r.idx >> 16) > 1) v = fmaf(r.c1, float(sy[i1]), v);
        reinterpret_cast<float*>(sA)[r.pos] = v * mul;
    }
}

// channel quads as two pairs
struct Q2 {
    float2 lo, hi;
};
__device__ __forceinline__ Q2 q2_of(const float (&v)[4]) { return {make_float2(v[0], v[1]), make_float2(v[2], v[3])}; }
__device__ __forceinline__ Q2 q2_mul(Q2 a, Q2 b) { return {__fmul2_rn(a.lo, b.lo), __fmul2_rn(a.hi, b.hi)}; }
__device__ __forceinline__ Q2 q2_fma(float2 a, Q2 b, Q2 c) { return {__ffma2_rn(a, b.lo, c.lo), __ffma2_rn(a, b.hi, c.hi)}; }
__device__ __forceinline__ Q2 q2_fma(Q2 a, Q2 b, Q2 c) { return {__ffma2_rn(a.lo, b.lo, c.lo), __ffma2_rn(a.hi, b.hi, c.hi)}; }
__device__ __forceinline__ Q2 q2_zero() { return {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}; }
template <class T>
__device__ __forceinline__ Q2 lds_q2(const T* p) {
    float v[4];
    lds4<T>(p, v);
    return q2_of(v);
}

// acc[Z + m3] += w * sum_m1 A[m3][m1] x[xoff + m1] for path P (4 channels as two pairs)
template <class Cfg, int P>
__device__ __forceinline__ void fwd_path(const float2* __restrict__ sA, const Q2 (&xv)[Cfg::D1], Q2 wv,
                                         Q2 (&acc)[Cfg::D]) {
    constexpr PathInfo pi = Cfg::table.paths[P];
    constexpr int a0 = Off<Cfg>::a[P];
    constexpr int na = Off<Cfg>::a[P + 1] - a0;
    constexpr int base = PipePlan<Cfg>::apos[P];
    constexpr int n1 = 2 * pi.l1 + 1, n3 = 2 * pi.l3 + 1;
    constexpr int Z = pi.zoff;
    if constexpr (n1 <= n3) {
        Q2 xw[n1];
#pragma unroll
        for (int m = 0; m < n1; ++m) xw[m] = q2_mul(xv[pi.xoff + m], wv);
        sfor<(na + 3) / 4>([&](auto qq) {
            constexpr int q = decltype(qq)::value;
            const float4 t4 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(sA) + base + 4 * q);
            const float2 av[4] = {make_float2(t4.x, t4.x), make_float2(t4.y, t4.y), make_float2(t4.z, t4.z),
                                  make_float2(t4.w, t4.w)};
            sfor<4>([&](auto cc) {
                constexpr int kk = 4 * q + decltype(cc)::value;
                if constexpr (kk < na) {
                    constexpr AEnt e = Cfg::aents[PipePlan<Cfg>::fwd_order[a0 + kk]];
                    acc[Z + e.m3] = q2_fma(av[decltype(cc)::value], xw[e.m1], acc[Z + e.m3]);
                }
            });
        });
    } else {
        Q2 t[n3];
#pragma unroll
        for (int m = 0; m < n3; ++m) t[m] = q2_zero();
        sfor<(na + 3) / 4>([&](auto qq) {
            constexpr int q = decltype(qq)::value;
            const float4 t4 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(sA) + base + 4 * q);
            const float2 av[4] = {make_float2(t4.x, t4.x), make_float2(t4.y, t4.y), make_float2(t4.z, t4.z),
                                  make_float2(t4.w, t4.w)};
            sfor<4>([&](auto cc) {
                constexpr int kk = 4 * q + decltype(cc)::value;
                if constexpr (kk < na) {
                    constexpr AEnt e = Cfg::aents[PipePlan<Cfg>::fwd_order[a0 + kk]];
                    t[e.m3] = q2_fma(av[decltype(cc)::value], xv[pi.xoff + e.m1], t[e.m3]);
                }
            });
        });
#pragma unroll
        for (int m = 0; m < n3; ++m) acc[Z + m] = q2_fma(wv, t[m], acc[Z + m]);
    }
}

__device__ __forceinline__ bool seg_ok(int64_t k0, int64_t k1, int64_t E) { return k0 >= 0 && k1 >= k0 && k1 <= E; }

// Sum each of N (a power of two <= 32) per-lane values over the 32 lanes of the warp with a
// transposing butterfly: every step halves the values a lane holds (it keeps one half and
// adds its partner's copy of that half), then plain butterfly steps finish the sum. The
// 32/N lanes that differ only in their low bits end with the same sum; *index receives
// which of the N sums this lane holds. Fixed order: deterministic. 16 values: 16 shuffles.
template <int N>
__device__ __forceinline__ float warp_sum_transposed(float (&v)[N], int lane, int* index) {
    static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "N must be a power of two <= 32");
    int idx = 0;
    sfor<__builtin_ctz(N)>([&](auto ss) {
        constexpr int st = decltype(ss)::value;
        constexpr int off = 16 >> st;
        constexpr int half = N >> (st + 1);
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        idx += upper ? half : 0;
    });
#pragma unroll
    for (int off = 16 >> __builtin_ctz(N); off > 0; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    *index = idx;
    return v[0];
}

// ------------------------------------------------------------------------------------------
// forward
// ------------------------------------------------------------------------------------------
// RH > 0 (the radial form): no w rows are streamed; the edge's item also carries its RH hidden
// activations h[e], and each path's weights are formed in registers from the block's shared
// copy of the output layer W2 [RH][NP][128]: w_p = sum_k h_k W2[k][p].
template <class Cfg, class T, int NSLOT, int RH = 0>
struct FwdPipe {
    using PP = PipePlan<Cfg>;
    static constexpr int NCH = RH > 0 ? 1 : 1 + PP::NWC;          // items per edge
    static constexpr int ROWB = kPipeNq * sizeof(T);              // bytes of one 128-channel row
    static constexpr int YB = ((Cfg::D2 * sizeof(T) + 15) / 16) * 16;
    static constexpr int HB = RH * 4;                             // the edge's hidden activations (fp32)
    static constexpr int ROWS = RH > 0 ? Cfg::D1 : (Cfg::D1 > PP::PPC ? Cfg::D1 : PP::PPC);
    static constexpr int SLOT = ((ROWS * ROWB + YB + HB) + 127) / 128 * 128;
    static constexpr int WARP_BYTES = NSLOT * SLOT + PP::NAPAD * 4;
    static constexpr int W2B = RH * Cfg::NP * kPipeNq * 4;        // shared copy of W2, ahead of the warps
};

// w_p = sum_k h_k W2[k][p] for the lane's four channels
template <class Cfg, int RH>
__device__ __forceinline__ Q2 radial_w(const float* __restrict__ w2s, const float (&hv)[RH], int p, int c0) {
    Q2 wv = q2_zero();
#pragma unroll
    for (int k = 0; k < RH; ++k) {
        const float2 hh = make_float2(hv[k], hv[k]);
        wv = q2_fma(hh, lds_q2<float>(w2s + (k * Cfg::NP + p) * kPipeNq + c0), wv);
    }
    return wv;
}

template <class Cfg, class T, int NSLOT, int WARPS, int RH = 0>
__global__ void __launch_bounds__(WARPS * 32, 1)
conv_forward_pipe_kernel(int64_t N, int64_t E, const int32_t* __restrict__ rowptr, const int32_t* __restrict__ sender,
                         const T* __restrict__ x, const T* __restrict__ y, const T* __restrict__ w, float scale,
                         float* __restrict__ m, int64_t pad, unsigned* __restrict__ err, int64_t cap,
                         const float* __restrict__ hrad = nullptr, const float* __restrict__ W2 = nullptr) {
    using F = FwdPipe<Cfg, T, NSLOT, RH>;
    using PP = PipePlan<Cfg>;
    extern __shared__ __align__(128) unsigned char smem[];
    const float* w2s = reinterpret_cast<const float*>(smem);
    if constexpr (RH > 0) load_w2_shared(reinterpret_cast<float*>(smem), W2, RH * Cfg::NP * kPipeNq);
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    unsigned char* wsm = smem + F::W2B + wid * F::WARP_BYTES;
    float2* sA = reinterpret_cast<float2*>(wsm + NSLOT * F::SLOT);
    const int c0 = lane * kVec;
    const int64_t gw = int64_t(blockIdx.x) * WARPS + wid;
    const int64_t nw = int64_t(gridDim.x) * WARPS;
    const uint64_t wpol = l2_policy_evict_first();

    // producer cursor: next item to issue = (edge pe of node pn, chunk pc)
    int64_t pn = gw, pe = 0, pend = 0;
    int pc = 0;
    bool pdone = false;
    // padding edges (receiver or sender == pad, pad >= 0) are never issued: the padding
    // receiver's segment is passed over whole, edges from the padding sender one by one
    auto p_seek = [&]() {   // make pe < pend (pe not a padding edge) or set pdone
        for (;;) {
            if (pad >= 0)
                while (pe < pend && __ldg(sender + pe) == pad) ++pe;
            if (pe < pend) return;
            if (pn >= N) { pdone = true; return; }
            const int64_t k0 = __ldg(rowptr + pn), k1 = __ldg(rowptr + pn + 1);
            const bool skip = pn == pad;
            pn += nw;
            if (!skip && seg_ok(k0, k1, E)) { pe = k0; pend = k1 - k0 > cap ? k0 + cap : k1; }
        }
    };
    auto issue = [&](int64_t i) {   // issue the producer's current item into slot i % NSLOT
        if (!pdone) {
            unsigned char* slot = wsm + int(i % NSLOT) * F::SLOT;
            if (pc == 0) {
                const int64_t a = __ldg(sender + pe);
                if (a >= 0 && a < N) {
#pragma unroll
                    for (int r = 0; r < Cfg::D1; ++r)
                        cp_async_slice<T>(slot + r * F::ROWB + c0 * sizeof(T), x + (a * Cfg::D1 + r) * kPipeNq + c0);
                }
                if (lane < F::YB / 16) cp_async16(slot + Cfg::D1 * F::ROWB + lane * 16,
                                                   reinterpret_cast<const unsigned char*>(y + pe * Cfg::D2) + lane * 16);
                if constexpr (RH > 0)
                    if (lane < F::HB / 16)
                        cp_async16(slot + Cfg::D1 * F::ROWB + F::YB + lane * 16, hrad + pe * RH + lane * 4);
            } else {
                const int p0 = (pc - 1) * PP::PPC;
                const int np = (Cfg::NP - p0) < PP::PPC ? (Cfg::NP - p0) : PP::PPC;
                const T* src = w + (pe * Cfg::NP + p0) * kPipeNq + c0;
#pragma unroll
                for (int r = 0; r < PP::PPC; ++r)
                    if (r < np) cp_async_slice_hint<T>(slot + r * F::ROWB + c0 * sizeof(T), src + r * kPipeNq, wpol);
            }
            if (++pc == F::NCH) {
                pc = 0;
                ++pe;
                p_seek();
            }
        }
        cp_async_commit();
    };
    p_seek();
    int64_t issued = 0;
    for (int s = 0; s < NSLOT - 1; ++s) issue(issued++);

    int64_t item = 0;
    for (int64_t b = gw; b < N; b += nw) {
        int64_t e0 = __ldg(rowptr + b), e1 = __ldg(rowptr + b + 1);
        if (!seg_ok(e0, e1, E)) {
            if (lane == 0) atomicOr(err, kErrRowptr);
            e0 = e1 = 0;
        }
        if (b == pad) e0 = e1 = 0;
        if (e1 - e0 > cap) e1 = e0 + cap;   // the rest of a heavy receiver: conv_forward_pieces_kernel
        Q2 acc[Cfg::D];
#pragma unroll
        for (int i = 0; i < Cfg::D; ++i) acc[i] = q2_zero();
        for (int64_t e = e0; e < e1; ++e) {
            const int64_t a = __ldg(sender + e);
            if (pad >= 0 && a == pad) continue;   // not issued by the producer either
            const bool ok = a >= 0 && a < N;
            if (!ok && lane == 0) atomicOr(err, kErrSender);
            Q2 xv[Cfg::D1];
            sfor<F::NCH>([&](auto cc) {
                constexpr int ch = decltype(cc)::value;
                issue(issued++);
                cp_async_wait<NSLOT - 1>();
                const unsigned char* slot = wsm + int(item % NSLOT) * F::SLOT;
                ++item;
                if constexpr (ch == 0) {
                    __syncwarp();   // y from the lanes that copied it
                    build_A_warp<Cfg, true, T>(reinterpret_cast<const T*>(slot + Cfg::D1 * F::ROWB), sA, lane);
#pragma unroll
                    for (int r = 0; r < Cfg::D1; ++r)
                        xv[r] = ok ? lds_q2<T>(reinterpret_cast<const T*>(slot + r * F::ROWB) + c0) : q2_zero();
                    __syncwarp();   // A visible to every lane
                    if constexpr (RH > 0) {
                        float hv[RH];
                        const float* sh = reinterpret_cast<const float*>(slot + Cfg::D1 * F::ROWB + F::YB);
#pragma unroll
                        for (int k = 0; k < RH; ++k) hv[k] = sh[k];
                        sfor<Cfg::NP>([&](auto pp) {
                            constexpr int p = decltype(pp)::value;
                            fwd_path<Cfg, p>(sA, xv, radial_w<Cfg, RH>(w2s, hv, p, c0), acc);
                        });
                        __syncwarp();   // A is rebuilt for the next edge
                    }
                } else {
                    constexpr int p0 = (ch - 1) * PP::PPC;
                    constexpr int np = (Cfg::NP - p0) < PP::PPC ? (Cfg::NP - p0) : PP::PPC;
                    sfor<np>([&](auto rr) {
                        constexpr int r = decltype(rr)::value;
                        const Q2 wv = lds_q2<T>(reinterpret_cast<const T*>(slot + r * F::ROWB) + c0);
                        fwd_path<Cfg, p0 + r>(sA, xv, wv, acc);
                    });
                    if constexpr (ch == F::NCH - 1) __syncwarp();   // A is rebuilt for the next edge
                }
            });
        }
        float* mb = m + b * (Cfg::D * kPipeNq);
        const float2 sc = make_float2(scale, scale);
#pragma unroll
        for (int i = 0; i < Cfg::D; ++i) {
            const float2 lo = __fmul2_rn(acc[i].lo, sc), hi = __fmul2_rn(acc[i].hi, sc);
            *reinterpret_cast<float4*>(mb + i * kPipeNq + c0) = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------------------------------
// backward (sender order)
// ------------------------------------------------------------------------------------------
// RH > 0 (the radial form): block items carry only the dm rows; the edge's first item also
// carries its hidden activations h[e]; w_p is formed from the shared copy of W2 and the
// cotangent dh[e][k] = sum_p sum_c W2[k][p][c] dw_p[c] replaces the dw row.
template <class Cfg, class T, int NSLOT, int RH = 0>
struct BwdPipe {
    using PP = PipePlan<Cfg>;
    static constexpr int ROWB = kPipeNq * sizeof(T);
    static constexpr int YB = ((Cfg::D2 * sizeof(T) + 15) / 16) * 16;
    static constexpr int HB = RH * 4;
    static constexpr int max_out_rows = [] {
        int r = 0;
        for (int j = 0; j < Cfg::NOUT; ++j) r = 2 * Cfg::table.outs[j].l + 1 > r ? 2 * Cfg::table.outs[j].l + 1 : r;
        return r;
    }();
    static constexpr int BROWS = RH > 0 ? max_out_rows : PP::max_block_rows;
    static constexpr int ROWS = Cfg::D1 > BROWS ? Cfg::D1 : BROWS;
    static constexpr int SLOT = ((ROWS * ROWB + YB + HB) + 127) / 128 * 128;
    static constexpr int XBUF = Cfg::D1 * kPipeNq * 4;            // the sender's x rows (fp32)
    // the A buffer is given 8 bytes per entry although it uses 4: this layout measured ~3%
    // faster than the compact one on the 64k-atom workload
    static constexpr int WARP_BYTES = NSLOT * SLOT + PP::NAPAD * 8 + XBUF;
    static constexpr int NCH = Cfg::NOUT;   // items per edge (one per output block)
    static constexpr int W2B = RH * Cfg::NP * kPipeNq * 4;
};

// radial backward's per-edge state: the hidden activations and the lane's partial dh
template <int RH>
struct RadEdge {
    float h[RH > 0 ? RH : 1];
    float dh[RH > 0 ? RH : 1];
    const float* w2s;
};

// the part of an edge's backward that belongs to output block J; g rows from the slot
// (the couplings in sA already carry the convolution scale; dy is scaled by the caller)
template <class Cfg, class T, int J, int RH = 0>
__device__ __forceinline__ void bwd_block(const unsigned char* __restrict__ slot, const float2* __restrict__ sA,
                                          const float* __restrict__ sx, Q2 (&dxa)[Cfg::D1], float (&dyp)[Cfg::D2],
                                          float* __restrict__ dw_e, int c0, RadEdge<RH>& rad) {
    using PP = PipePlan<Cfg>;
    constexpr int ROWB = kPipeNq * sizeof(T);
    constexpr int nrow = 2 * Cfg::table.outs[J].l + 1;
    constexpr int npb = PP::bpos[J + 1] - PP::bpos[J];
    Q2 g[nrow];
#pragma unroll
    for (int mm = 0; mm < nrow; ++mm) g[mm] = lds_q2<T>(reinterpret_cast<const T*>(slot + mm * ROWB) + c0);
    sfor<npb>([&](auto ii) {
        constexpr int p = PP::bpath[PP::bpos[J] + decltype(ii)::value];
        constexpr PathInfo pi = Cfg::table.paths[p];
        constexpr int a0 = Off<Cfg>::a[p];
        constexpr int na = Off<Cfg>::a[p + 1] - a0;
        constexpr int n1 = 2 * pi.l1 + 1;
        constexpr int base = PP::apos[p];
        Q2 wv;
        if constexpr (RH > 0) wv = radial_w<Cfg, RH>(rad.w2s, rad.h, p, c0);
        else wv = lds_q2<T>(reinterpret_cast<const T*>(slot + (nrow + decltype(ii)::value) * ROWB) + c0);
        Q2 gp[n1], xw[n1], xr[n1];
#pragma unroll
        for (int mm = 0; mm < n1; ++mm) {
            xr[mm] = lds_q2<float>(sx + (pi.xoff + mm) * kPipeNq + c0);
            gp[mm] = q2_zero();
            xw[mm] = q2_mul(xr[mm], wv);
        }
        sfor<(na + 3) / 4>([&](auto qq) {
            constexpr int q = decltype(qq)::value;
            const float4 t4 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(sA) + base + 4 * q);
            const float2 av[4] = {make_float2(t4.x, t4.x), make_float2(t4.y, t4.y), make_float2(t4.z, t4.z),
                                  make_float2(t4.w, t4.w)};
            sfor<4>([&](auto cc) {
                constexpr int kk = 4 * q + decltype(cc)::value;
                if constexpr (kk < na) {
                    constexpr AEnt e = Cfg::aents[a0 + kk];
                    gp[e.m1] = q2_fma(av[decltype(cc)::value], g[e.m3], gp[e.m1]);
                    // sum over the lane's 4 channels of x w g, for dy (two paired products, one add)
                    const float2 s2 = __ffma2_rn(xw[e.m1].hi, g[e.m3].hi, __fmul2_rn(xw[e.m1].lo, g[e.m3].lo));
                    const float s = s2.x + s2.y;
                    sfor<e.nt>([&](auto t) {
                        constexpr int tt = decltype(t)::value;
                        dyp[pi.yoff + e.m2[tt]] = fmaf(e.c[tt], s, dyp[pi.yoff + e.m2[tt]]);
                    });
                }
            });
        });
        Q2 dwv = q2_zero();
#pragma unroll
        for (int mm = 0; mm < n1; ++mm) {
            dwv = q2_fma(xr[mm], gp[mm], dwv);
            dxa[pi.xoff + mm] = q2_fma(wv, gp[mm], dxa[pi.xoff + mm]);
        }
        if constexpr (RH > 0) {
#pragma unroll
            for (int k = 0; k < RH; ++k) {   // the lane's share of dh[k] = sum_c W2[k][p][c] dw_p[c]
                const Q2 w2 = lds_q2<float>(rad.w2s + (k * Cfg::NP + p) * kPipeNq + c0);
                const float2 s2 = __ffma2_rn(w2.hi, dwv.hi, __fmul2_rn(w2.lo, dwv.lo));
                rad.dh[k] += s2.x + s2.y;
            }
        } else {
            __stcs(reinterpret_cast<float4*>(dw_e + p * kPipeNq + c0),
                   make_float4(dwv.lo.x, dwv.lo.y, dwv.hi.x, dwv.hi.y));
        }
    });
}

// IDENT: the identity graph of the row-wise tensor product backward (App. E.1 Eq. (15)): row r
// is a node with the single edge r from and to itself, scale 1; the index arrays are not read
// and may be null, and so may err (no index can be out of range).
// RH > 0: the radial form (w unused; dw receives dh [E][RH]); not combined with IDENT.
template <class Cfg, class T, int NSLOT, int WARPS, bool IDENT = false, int RH = 0>
__global__ void __launch_bounds__(WARPS * 32, 1)
conv_backward_pipe_kernel(int64_t N, int64_t E, const int32_t* __restrict__ cptr, const int32_t* __restrict__ cedge,
                          const int32_t* __restrict__ crecv, const T* __restrict__ x, const T* __restrict__ y,
                          const T* __restrict__ w, const T* __restrict__ dm, float scale, float* __restrict__ dx,
                          float* __restrict__ dy, float* __restrict__ dw, int64_t pad, unsigned* __restrict__ err,
                          const float* __restrict__ hrad = nullptr, const float* __restrict__ W2 = nullptr) {
    static_assert(!(IDENT && RH > 0), "the identity graph has no radial form");
    using B = BwdPipe<Cfg, T, NSLOT, RH>;
    using PP = PipePlan<Cfg>;
    extern __shared__ __align__(128) unsigned char smem[];
    if constexpr (RH > 0) load_w2_shared(reinterpret_cast<float*>(smem), W2, RH * Cfg::NP * kPipeNq);
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    unsigned char* wsm = smem + B::W2B + wid * B::WARP_BYTES;
    float2* sA = reinterpret_cast<float2*>(wsm + NSLOT * B::SLOT);
    float* sx = reinterpret_cast<float*>(wsm + NSLOT * B::SLOT + PP::NAPAD * 8);
    const int c0 = lane * kVec;
    const int64_t gw = int64_t(blockIdx.x) * WARPS + wid;
    const int64_t nw = int64_t(gridDim.x) * WARPS;
    const uint64_t wpol = l2_policy_evict_first();
    auto cp_at = [&](int64_t i) -> int64_t {
        if constexpr (IDENT) return i;
        else return __ldg(cptr + i);
    };
    auto ce_at = [&](int64_t k) -> int64_t {
        if constexpr (IDENT) return k;
        else return __ldg(cedge + k);
    };
    auto cr_at = [&](int64_t k) -> int64_t {
        if constexpr (IDENT) return k;
        else return __ldg(crecv + k);
    };
    auto flag = [&](unsigned bits) {
        if constexpr (!IDENT) atomicOr(err, bits);
    };

    // producer cursor: sender pa, edge position pk in [pk, pkend), item pc (-1: x rows of pa)
    int64_t pa = gw - nw, pk = 0, pkend = 0;
    int pc = 0;
    bool pdone = false;
    // padding edges (sender or receiver == pad, pad >= 0) are never issued: the padding
    // sender's segment is passed over whole (only its x item is issued), edges into the
    // padding receiver one by one
    auto p_skip_pad = [&]() {
        if (pad >= 0)
            while (pk < pkend && cr_at(pk) == pad) ++pk;
    };
    auto p_next_sender = [&]() {
        pa += nw;
        if (pa >= N) { pdone = true; return; }
        int64_t k0 = cp_at(pa), k1 = cp_at(pa + 1);
        if (!seg_ok(k0, k1, E) || pa == pad) k0 = k1 = 0;
        pk = k0;
        pkend = k1;
        p_skip_pad();
        pc = -1;
    };
    auto issue = [&](int64_t i) {
        if (!pdone) {
            unsigned char* slot = wsm + int(i % NSLOT) * B::SLOT;
            if (pc < 0) {   // x rows of the sender
#pragma unroll
                for (int r = 0; r < Cfg::D1; ++r)
                    cp_async_slice<T>(slot + r * B::ROWB + c0 * sizeof(T), x + (pa * Cfg::D1 + r) * kPipeNq + c0);
                pc = 0;
                if (pk >= pkend) p_next_sender();
            } else {
                const int64_t e = ce_at(pk), bb = cr_at(pk);
                const bool ok = e >= 0 && e < E && bb >= 0 && bb < N;
                if (ok) {
                    // rows of output block pc: dm rows, then w rows of its paths; y behind them
                    sfor<Cfg::NOUT>([&](auto jj) {
                        constexpr int j = decltype(jj)::value;
                        if (pc == j) {
                            constexpr int nrow = 2 * Cfg::table.outs[j].l + 1;
                            constexpr int zo = Off<Cfg>::z[j];
#pragma unroll
                            for (int r = 0; r < nrow; ++r)
                                cp_async_slice<T>(slot + r * B::ROWB + c0 * sizeof(T),
                                                  dm + (bb * Cfg::D + zo + r) * kPipeNq + c0);
                            if constexpr (RH == 0)
                                sfor<PP::bpos[j + 1] - PP::bpos[j]>([&](auto ii) {
                                    constexpr int p = PP::bpath[PP::bpos[j] + decltype(ii)::value];
                                    cp_async_slice_hint<T>(
                                        slot + (nrow + decltype(ii)::value) * B::ROWB + c0 * sizeof(T),
                                        w + (e * Cfg::NP + p) * kPipeNq + c0, wpol);
                                });
                        }
                    });
                    if (pc == 0 && lane < B::YB / 16)
                        cp_async16(slot + B::ROWS * B::ROWB + lane * 16,
                                   reinterpret_cast<const unsigned char*>(y + e * Cfg::D2) + lane * 16);
                    if constexpr (RH > 0)
                        if (pc == 0 && lane < B::HB / 16)
                            cp_async16(slot + B::ROWS * B::ROWB + B::YB + lane * 16, hrad + e * RH + lane * 4);
                }
                if (++pc == B::NCH) {
                    pc = 0;
                    ++pk;
                    p_skip_pad();
                    if (pk >= pkend) p_next_sender();
                }
            }
        }
        cp_async_commit();
    };
    p_next_sender();
    int64_t issued = 0;
    for (int s = 0; s < NSLOT - 1; ++s) issue(issued++);

    int64_t item = 0;
    for (int64_t a = gw; a < N; a += nw) {
        int64_t k0 = cp_at(a), k1 = cp_at(a + 1);
        if (!seg_ok(k0, k1, E)) {
            if (lane == 0) flag(kErrRowptr);
            k0 = k1 = 0;
        }
        if (a == pad) k0 = k1 = 0;
        Q2 dxa[Cfg::D1];
        {   // item: x rows of the sender -> the warp's x buffer (each lane its own channels)
            issue(issued++);
            cp_async_wait<NSLOT - 1>();
            const unsigned char* slot = wsm + int(item % NSLOT) * B::SLOT;
            ++item;
#pragma unroll
            for (int r = 0; r < Cfg::D1; ++r) {
                const Q2 v = lds_q2<T>(reinterpret_cast<const T*>(slot + r * B::ROWB) + c0);
                *reinterpret_cast<float4*>(sx + r * kPipeNq + c0) = make_float4(v.lo.x, v.lo.y, v.hi.x, v.hi.y);
                dxa[r] = q2_zero();
            }
        }
        for (int64_t k = k0; k < k1; ++k) {
            const int64_t e = ce_at(k), bb = cr_at(k);
            if (pad >= 0 && bb == pad) continue;   // not issued by the producer either
            const bool ok = e >= 0 && e < E && bb >= 0 && bb < N;
            if (!ok && lane == 0) flag(kErrRecv);
            float dyp[Cfg::D2];
#pragma unroll
            for (int t = 0; t < Cfg::D2; ++t) dyp[t] = 0.f;
            float* dw_e = dw + (ok ? e : 0) * (Cfg::NP * kPipeNq);
            RadEdge<RH> rad;
            if constexpr (RH > 0) {
                rad.w2s = reinterpret_cast<const float*>(smem);
#pragma unroll
                for (int k = 0; k < RH; ++k) rad.dh[k] = 0.f;
            }
            sfor<B::NCH>([&](auto jj) {
                constexpr int j = decltype(jj)::value;
                issue(issued++);
                cp_async_wait<NSLOT - 1>();
                const unsigned char* slot = wsm + int(item % NSLOT) * B::SLOT;
                ++item;
                if constexpr (j == 0) {
                    __syncwarp();
                    if (ok)
                        build_A_warp<Cfg, false, T>(reinterpret_cast<const T*>(slot + B::ROWS * B::ROWB), sA, lane,
                                                    scale);
                    if constexpr (RH > 0) {
                        const float* sh = reinterpret_cast<const float*>(slot + B::ROWS * B::ROWB + B::YB);
#pragma unroll
                        for (int k = 0; k < RH; ++k) rad.h[k] = sh[k];
                    }
                    __syncwarp();
                }
                if (ok) bwd_block<Cfg, T, j, RH>(slot, sA, sx, dxa, dyp, dw_e, c0, rad);
                if constexpr (j == B::NCH - 1) __syncwarp();
            });
            int di = 0;
            const float dsum = warp_sum_transposed<Cfg::D2>(dyp, lane, &di);
            if (ok && (lane & (32 / Cfg::D2 - 1)) == 0) dy[e * Cfg::D2 + di] = dsum * scale;
            if constexpr (RH > 0) {
                int hi = 0;
                const float hsum = warp_sum_transposed<RH>(rad.dh, lane, &hi);
                if (ok && (lane & (32 / RH - 1)) == 0) dw[e * RH + hi] = hsum;
            }
        }
#pragma unroll
        for (int r = 0; r < Cfg::D1; ++r)
            *reinterpret_cast<float4*>(dx + (a * Cfg::D1 + r) * kPipeNq + c0) =
                make_float4(dxa[r].lo.x, dxa[r].lo.y, dxa[r].hi.x, dxa[r].hi.y);
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------------------------------
// launch shapes
// ------------------------------------------------------------------------------------------
constexpr int kSmemLimit = 232448;   // 227 KiB per block

template <class Cfg, class T, bool BWD, int RH = 0>
struct PipeShape {
    // the radial form keeps a shared copy of W2 beside the warps' rings: fewer slots
    static constexpr int NSLOT = BWD ? (RH > 0 ? 2 : 3) : (RH > 0 ? 3 : 4);
    static constexpr int WARP_BYTES =
        BWD ? BwdPipe<Cfg, T, NSLOT, RH>::WARP_BYTES : FwdPipe<Cfg, T, NSLOT, RH>::WARP_BYTES;
    static constexpr int W2B = RH * Cfg::NP * kPipeNq * 4;
    static constexpr int by_smem = (kSmemLimit - W2B) / WARP_BYTES;
    static constexpr int WARPS = by_smem < 8 ? by_smem : 8;
    static constexpr int SMEM = W2B + WARPS * WARP_BYTES;
    // the forward keeps every output row of its receiver in registers: at most 32 of them
    static constexpr bool usable = (Cfg::D2 * sizeof(T)) % 16 == 0 && WARPS >= 4 && (BWD || Cfg::D <= 32);
};

}  // namespace e3gb
