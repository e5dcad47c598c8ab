// Convolution double backward ("e3j ...", App. E.1 Eq. (17)-(18)) for 128 channels, with the
// per-warp cp.async rings of conv_pipe.cuh.
//
// Receiver pass (Eq. 17), one warp per receiver, all 31 output rows in registers:
//   delta_dm[b] = scale * sum_e sum_p [A_p(y) (w_p ddx_a + ddw_p x_a) + A_p(ddy) (w_p x_a)]
// which is conv(ddx, y, w) + conv(x, ddy, w) + conv(x, y, ddw) with the per-channel weights
// moved inside the coupling sum (they commute with it): two multiply-adds per coupling entry
// instead of three conv passes.
//   items per edge: [x rows of the sender + y + ddy] [ddx rows] [w and ddw rows of PPC paths] ...
// Sender pass (Eq. 18), one warp per sender, delta_x[a] in registers:
//   per edge and path, with g = dm rows of the receiver and the adjoint couplings
//   gy = A_p(y)^T g, gd = A_p(ddy)^T g (the scale folded into the couplings):
//   delta_x += w gd + ddw gy;  delta_w[e,p] = sum_m1 ddx gy + x gd;
//   delta_y[e] += sum over records c * sum_q (ddx w + x ddw)[m1] g[m3]   (scaled at the store)
//   items per sender: [x rows] [ddx rows]; per edge: [y + ddy + dm, w and ddw rows of the
//   paths of output block 0] [output block 1] ...
// The sender's x and ddx rows are copied out of the ring into a per-warp fp32 buffer (each
// lane its own channels), as the first-order backward does with x.
#pragma once

#include "conv_pipe.cuh"

namespace e3gb {

// ------------------------------------------------------------------------------------------
// receiver pass
// ------------------------------------------------------------------------------------------
template <class Cfg, class T, int NSLOT>
struct DdmPipe {
    using PP = PipePlan<Cfg>;
    static constexpr int PPC = 4;                                   // paths per chunk
    static constexpr int NWC = (Cfg::NP + PPC - 1) / PPC;
    static constexpr int NCH = 2 + NWC;                             // items per edge
    static constexpr int ROWB = kPipeNq * sizeof(T);
    static constexpr int YB = ((Cfg::D2 * sizeof(T) + 15) / 16) * 16;
    static constexpr int ROWS = Cfg::D1 > 2 * PPC ? Cfg::D1 : 2 * PPC;
    static constexpr int SLOT = ((ROWS * ROWB + 2 * YB) + 127) / 128 * 128;
    static constexpr int ABUF = PP::NAPAD * 4;
    static constexpr int XROWS = Cfg::D1 * kPipeNq * 4;              // one fp32 copy of d1 rows
    static constexpr int WARP_BYTES = NSLOT * SLOT + 2 * ABUF + 2 * XROWS;
};

// acc[Z + m3] += sum_m1 A_y[m3][m1] (w ddx + ddw x)[m1] + A_dy[m3][m1] (w x)[m1]  for path P
template <class Cfg, int P>
__device__ __forceinline__ void ddm_path(const float* __restrict__ sAy, const float* __restrict__ sAd,
                                         const float* __restrict__ sx, const float* __restrict__ sdx, Q2 wv,
                                         Q2 dwv, Q2 (&acc)[Cfg::D], int c0) {
    constexpr PathInfo pi = Cfg::table.paths[P];
    constexpr int a0 = Off<Cfg>::a[P];
    constexpr int na = Off<Cfg>::a[P + 1] - a0;
    constexpr int base = PipePlan<Cfg>::apos[P];
    constexpr int n1 = 2 * pi.l1 + 1;
    constexpr int Z = pi.zoff;
    Q2 u[n1], v[n1];
#pragma unroll
    for (int m = 0; m < n1; ++m) {
        const Q2 xr = lds_q2<float>(sx + (pi.xoff + m) * kPipeNq + c0);
        const Q2 dr = lds_q2<float>(sdx + (pi.xoff + m) * kPipeNq + c0);
        v[m] = q2_mul(xr, wv);
        u[m] = q2_fma(xr, dwv, q2_mul(dr, wv));
    }
    sfor<(na + 3) / 4>([&](auto qq) {
        constexpr int q = decltype(qq)::value;
        const float4 ty = *reinterpret_cast<const float4*>(sAy + base + 4 * q);
        const float4 td = *reinterpret_cast<const float4*>(sAd + base + 4 * q);
        const float2 ay[4] = {make_float2(ty.x, ty.x), make_float2(ty.y, ty.y), make_float2(ty.z, ty.z),
                              make_float2(ty.w, ty.w)};
        const float2 ad[4] = {make_float2(td.x, td.x), make_float2(td.y, td.y), make_float2(td.z, td.z),
                              make_float2(td.w, td.w)};
        sfor<4>([&](auto cc) {
            constexpr int kk = 4 * q + decltype(cc)::value;
            if constexpr (kk < na) {
                constexpr AEnt e = Cfg::aents[PipePlan<Cfg>::fwd_order[a0 + kk]];
                acc[Z + e.m3] = q2_fma(ay[decltype(cc)::value], u[e.m1], acc[Z + e.m3]);
            }
        });
        sfor<4>([&](auto cc) {
            constexpr int kk = 4 * q + decltype(cc)::value;
            if constexpr (kk < na) {
                constexpr AEnt e = Cfg::aents[PipePlan<Cfg>::fwd_order[a0 + kk]];
                acc[Z + e.m3] = q2_fma(ad[decltype(cc)::value], v[e.m1], acc[Z + e.m3]);
            }
        });
    });
}

// copy D1 rows of this lane's channels from a ring slot into an fp32 row buffer
template <class Cfg, class T>
__device__ __forceinline__ void stage_rows(const unsigned char* __restrict__ slot, float* __restrict__ buf, int c0) {
    constexpr int ROWB = kPipeNq * sizeof(T);
#pragma unroll
    for (int r = 0; r < Cfg::D1; ++r) {
        const Q2 v = lds_q2<T>(reinterpret_cast<const T*>(slot + r * ROWB) + c0);
        *reinterpret_cast<float4*>(buf + r * kPipeNq + c0) = make_float4(v.lo.x, v.lo.y, v.hi.x, v.hi.y);
    }
}

template <class Cfg, class T, int NSLOT, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1)
conv_ddm_pipe_kernel(int64_t N, int64_t E, const int32_t* __restrict__ rowptr, const int32_t* __restrict__ sender,
                     const T* __restrict__ x, const T* __restrict__ y, const T* __restrict__ w,
                     const T* __restrict__ ddx, const T* __restrict__ ddy, const T* __restrict__ ddw, float scale,
                     float* __restrict__ ddm, int64_t pad, unsigned* __restrict__ err) {
    using F = DdmPipe<Cfg, T, NSLOT>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    unsigned char* wsm = smem + wid * F::WARP_BYTES;
    float* sAy = reinterpret_cast<float*>(wsm + NSLOT * F::SLOT);
    float* sAd = reinterpret_cast<float*>(wsm + NSLOT * F::SLOT + F::ABUF);
    float* sx = reinterpret_cast<float*>(wsm + NSLOT * F::SLOT + 2 * F::ABUF);
    float* sdx = reinterpret_cast<float*>(wsm + NSLOT * F::SLOT + 2 * F::ABUF + F::XROWS);
    const int c0 = lane * kVec;
    const int64_t gw = int64_t(blockIdx.x) * WARPS + wid;
    const int64_t nw = int64_t(gridDim.x) * WARPS;

    // producer cursor: next item = (edge pe of node pn, item pc); padding edges never issued
    int64_t pn = gw, pe = 0, pend = 0;
    int pc = 0;
    bool pdone = false;
    auto p_seek = [&]() {
        for (;;) {
            if (pad >= 0)
                while (pe < pend && __ldg(sender + pe) == pad) ++pe;
            if (pe < pend) return;
            if (pn >= N) { pdone = true; return; }
            const int64_t k0 = __ldg(rowptr + pn), k1 = __ldg(rowptr + pn + 1);
            const bool skip = pn == pad;
            pn += nw;
            if (!skip && seg_ok(k0, k1, E)) { pe = k0; pend = k1; }
        }
    };
    auto issue = [&](int64_t i) {
        if (!pdone) {
            unsigned char* slot = wsm + int(i % NSLOT) * F::SLOT;
            if (pc <= 1) {
                const int64_t a = __ldg(sender + pe);
                if (a >= 0 && a < N) {
                    const T* src = (pc == 0 ? x : ddx) + a * Cfg::D1 * kPipeNq + c0;
#pragma unroll
                    for (int r = 0; r < Cfg::D1; ++r)
                        cp_async_slice<T>(slot + r * F::ROWB + c0 * sizeof(T), src + r * kPipeNq);
                }
                if (pc == 0 && lane < 2 * (F::YB / 16)) {   // y then ddy behind the rows
                    const int h = lane / (F::YB / 16), o = lane % (F::YB / 16);
                    const T* ys = (h == 0 ? y : ddy) + pe * Cfg::D2;
                    cp_async16(slot + F::ROWS * F::ROWB + h * F::YB + o * 16,
                               reinterpret_cast<const unsigned char*>(ys) + o * 16);
                }
            } else {
                const int p0 = (pc - 2) * F::PPC;
                const int np = (Cfg::NP - p0) < F::PPC ? (Cfg::NP - p0) : F::PPC;
                const T* sw = w + (pe * Cfg::NP + p0) * kPipeNq + c0;
                const T* sd = ddw + (pe * Cfg::NP + p0) * kPipeNq + c0;
#pragma unroll
                for (int r = 0; r < F::PPC; ++r)
                    if (r < np) {
                        cp_async_slice<T>(slot + r * F::ROWB + c0 * sizeof(T), sw + r * kPipeNq);
                        cp_async_slice<T>(slot + (F::PPC + r) * F::ROWB + c0 * sizeof(T), sd + r * kPipeNq);
                    }
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
        Q2 acc[Cfg::D];
#pragma unroll
        for (int i = 0; i < Cfg::D; ++i) acc[i] = q2_zero();
        for (int64_t e = e0; e < e1; ++e) {
            const int64_t a = __ldg(sender + e);
            if (pad >= 0 && a == pad) continue;   // not issued by the producer either
            const bool ok = a >= 0 && a < N;
            if (!ok && lane == 0) atomicOr(err, kErrSender);
            sfor<F::NCH>([&](auto cc) {
                constexpr int ch = decltype(cc)::value;
                issue(issued++);
                cp_async_wait<NSLOT - 1>();
                const unsigned char* slot = wsm + int(item % NSLOT) * F::SLOT;
                ++item;
                if constexpr (ch == 0) {
                    __syncwarp();   // y, ddy from the lanes that copied them
                    const T* sy = reinterpret_cast<const T*>(slot + F::ROWS * F::ROWB);
                    build_A_warp<Cfg, true, T>(sy, reinterpret_cast<float2*>(sAy), lane);
                    build_A_warp<Cfg, true, T>(reinterpret_cast<const T*>(slot + F::ROWS * F::ROWB + F::YB),
                                               reinterpret_cast<float2*>(sAd), lane);
                    stage_rows<Cfg, T>(slot, sx, c0);
                    __syncwarp();   // A visible to every lane
                } else if constexpr (ch == 1) {
                    stage_rows<Cfg, T>(slot, sdx, c0);
                } else {
                    constexpr int p0 = (ch - 2) * F::PPC;
                    constexpr int np = (Cfg::NP - p0) < F::PPC ? (Cfg::NP - p0) : F::PPC;
                    if (ok)
                        sfor<np>([&](auto rr) {
                            constexpr int r = decltype(rr)::value;
                            const Q2 wv = lds_q2<T>(reinterpret_cast<const T*>(slot + r * F::ROWB) + c0);
                            const Q2 dwv = lds_q2<T>(reinterpret_cast<const T*>(slot + (F::PPC + r) * F::ROWB) + c0);
                            ddm_path<Cfg, p0 + r>(sAy, sAd, sx, sdx, wv, dwv, acc, c0);
                        });
                    if constexpr (ch == F::NCH - 1) __syncwarp();   // A is rebuilt for the next edge
                }
            });
        }
        float* mb = ddm + b * (Cfg::D * kPipeNq);
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
// sender pass
// ------------------------------------------------------------------------------------------
template <class Cfg, class T, int NSLOT>
struct DbwdPipe {
    using PP = PipePlan<Cfg>;
    static constexpr int ROWB = kPipeNq * sizeof(T);
    static constexpr int YB = ((Cfg::D2 * sizeof(T) + 15) / 16) * 16;
    static constexpr int max_rows = [] {
        int m = Cfg::D1;
        for (int j = 0; j < Cfg::NOUT; ++j) {
            const int r = (2 * Cfg::table.outs[j].l + 1) + 2 * (PP::bpos[j + 1] - PP::bpos[j]);
            m = r > m ? r : m;
        }
        return m;
    }();
    static constexpr int ROWS = max_rows;
    static constexpr int SLOT = ((ROWS * ROWB + 2 * YB) + 127) / 128 * 128;
    static constexpr int ABUF = PP::NAPAD * 4;
    static constexpr int XROWS = Cfg::D1 * kPipeNq * 4;
    static constexpr int WARP_BYTES = NSLOT * SLOT + 2 * ABUF + 2 * XROWS;
    static constexpr int NCH = Cfg::NOUT;   // items per edge
};

// output block J of one edge: g = dm rows (slot rows 0..nrow-1), w rows (nrow..), ddw rows
// (nrow + npb..); the couplings carry the scale, the lane's delta_y partial (dyp) does not
template <class Cfg, class T, int J>
__device__ __forceinline__ void dbwd_block(const unsigned char* __restrict__ slot, const float* __restrict__ sAy,
                                           const float* __restrict__ sAd, const float* __restrict__ sx,
                                           const float* __restrict__ sdx, Q2 (&gxa)[Cfg::D1], float (&dyp)[Cfg::D2],
                                           float* __restrict__ gw_e, int c0) {
    using PP = PipePlan<Cfg>;
    constexpr int ROWB = kPipeNq * sizeof(T);
    constexpr int nrow = 2 * Cfg::table.outs[J].l + 1;
    constexpr int npb = PP::bpos[J + 1] - PP::bpos[J];
    Q2 g[nrow];
#pragma unroll
    for (int mm = 0; mm < nrow; ++mm) g[mm] = lds_q2<T>(reinterpret_cast<const T*>(slot + mm * ROWB) + c0);
    sfor<npb>([&](auto ii) {
        constexpr int i = decltype(ii)::value;
        constexpr int p = PP::bpath[PP::bpos[J] + i];
        constexpr PathInfo pi = Cfg::table.paths[p];
        constexpr int a0 = Off<Cfg>::a[p];
        constexpr int na = Off<Cfg>::a[p + 1] - a0;
        constexpr int n1 = 2 * pi.l1 + 1;
        constexpr int base = PP::apos[p];
        const Q2 wv = lds_q2<T>(reinterpret_cast<const T*>(slot + (nrow + i) * ROWB) + c0);
        const Q2 dwv = lds_q2<T>(reinterpret_cast<const T*>(slot + (nrow + npb + i) * ROWB) + c0);
        Q2 gy[n1], gd[n1], u[n1];
#pragma unroll
        for (int mm = 0; mm < n1; ++mm) {
            const Q2 xr = lds_q2<float>(sx + (pi.xoff + mm) * kPipeNq + c0);
            const Q2 dr = lds_q2<float>(sdx + (pi.xoff + mm) * kPipeNq + c0);
            u[mm] = q2_fma(xr, dwv, q2_mul(dr, wv));
            gy[mm] = q2_zero();
            gd[mm] = q2_zero();
        }
        sfor<(na + 3) / 4>([&](auto qq) {
            constexpr int q = decltype(qq)::value;
            const float4 ty = *reinterpret_cast<const float4*>(sAy + base + 4 * q);
            const float4 td = *reinterpret_cast<const float4*>(sAd + base + 4 * q);
            const float2 ay[4] = {make_float2(ty.x, ty.x), make_float2(ty.y, ty.y), make_float2(ty.z, ty.z),
                                  make_float2(ty.w, ty.w)};
            const float2 ad[4] = {make_float2(td.x, td.x), make_float2(td.y, td.y), make_float2(td.z, td.z),
                                  make_float2(td.w, td.w)};
            sfor<4>([&](auto cc) {
                constexpr int kk = 4 * q + decltype(cc)::value;
                if constexpr (kk < na) {
                    constexpr AEnt e = Cfg::aents[a0 + kk];
                    gy[e.m1] = q2_fma(ay[decltype(cc)::value], g[e.m3], gy[e.m1]);
                    gd[e.m1] = q2_fma(ad[decltype(cc)::value], g[e.m3], gd[e.m1]);
                    // sum over the lane's 4 channels of (ddx w + x ddw) g, for delta_y
                    const float2 s2 = __ffma2_rn(u[e.m1].hi, g[e.m3].hi, __fmul2_rn(u[e.m1].lo, g[e.m3].lo));
                    const float s = s2.x + s2.y;
                    sfor<e.nt>([&](auto t) {
                        constexpr int tt = decltype(t)::value;
                        dyp[pi.yoff + e.m2[tt]] = fmaf(e.c[tt], s, dyp[pi.yoff + e.m2[tt]]);
                    });
                }
            });
        });
        Q2 gwv = q2_zero();
#pragma unroll
        for (int mm = 0; mm < n1; ++mm) {
            const Q2 xr = lds_q2<float>(sx + (pi.xoff + mm) * kPipeNq + c0);
            const Q2 dr = lds_q2<float>(sdx + (pi.xoff + mm) * kPipeNq + c0);
            gwv = q2_fma(dr, gy[mm], q2_fma(xr, gd[mm], gwv));
            gxa[pi.xoff + mm] = q2_fma(wv, gd[mm], q2_fma(dwv, gy[mm], gxa[pi.xoff + mm]));
        }
        __stcs(reinterpret_cast<float4*>(gw_e + p * kPipeNq + c0), make_float4(gwv.lo.x, gwv.lo.y, gwv.hi.x, gwv.hi.y));
    });
}

template <class Cfg, class T, int NSLOT, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1)
conv_dbwd_pipe_kernel(int64_t N, int64_t E, const int32_t* __restrict__ cptr, const int32_t* __restrict__ cedge,
                      const int32_t* __restrict__ crecv, const T* __restrict__ x, const T* __restrict__ y,
                      const T* __restrict__ w, const T* __restrict__ dm, const T* __restrict__ ddx,
                      const T* __restrict__ ddy, const T* __restrict__ ddw, float scale, float* __restrict__ gx,
                      float* __restrict__ gy, float* __restrict__ gw, int64_t pad, unsigned* __restrict__ err) {
    using B = DbwdPipe<Cfg, T, NSLOT>;
    using PP = PipePlan<Cfg>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    unsigned char* wsm = smem + wid * B::WARP_BYTES;
    float* sAy = reinterpret_cast<float*>(wsm + NSLOT * B::SLOT);
    float* sAd = reinterpret_cast<float*>(wsm + NSLOT * B::SLOT + B::ABUF);
    float* sx = reinterpret_cast<float*>(wsm + NSLOT * B::SLOT + 2 * B::ABUF);
    float* sdx = reinterpret_cast<float*>(wsm + NSLOT * B::SLOT + 2 * B::ABUF + B::XROWS);
    const int c0 = lane * kVec;
    const int64_t gw0 = int64_t(blockIdx.x) * WARPS + wid;
    const int64_t nw = int64_t(gridDim.x) * WARPS;

    // producer cursor: sender pa, edge position pk in [pk, pkend), item pc (-2: x rows of pa,
    // -1: ddx rows of pa, 0..NCH-1: output blocks of edge pk); padding edges never issued
    int64_t pa = gw0 - nw, pk = 0, pkend = 0;
    int pc = 0;
    bool pdone = false;
    auto p_skip_pad = [&]() {
        if (pad >= 0)
            while (pk < pkend && __ldg(crecv + pk) == pad) ++pk;
    };
    auto p_next_sender = [&]() {
        pa += nw;
        if (pa >= N) { pdone = true; return; }
        int64_t k0 = __ldg(cptr + pa), k1 = __ldg(cptr + pa + 1);
        if (!seg_ok(k0, k1, E) || pa == pad) k0 = k1 = 0;
        pk = k0;
        pkend = k1;
        p_skip_pad();
        pc = -2;
    };
    auto issue = [&](int64_t i) {
        if (!pdone) {
            unsigned char* slot = wsm + int(i % NSLOT) * B::SLOT;
            if (pc < 0) {   // x or ddx rows of the sender
                const T* src = (pc == -2 ? x : ddx) + pa * Cfg::D1 * kPipeNq + c0;
#pragma unroll
                for (int r = 0; r < Cfg::D1; ++r)
                    cp_async_slice<T>(slot + r * B::ROWB + c0 * sizeof(T), src + r * kPipeNq);
                if (++pc == 0 && pk >= pkend) p_next_sender();
            } else {
                const int64_t e = __ldg(cedge + pk), bb = __ldg(crecv + pk);
                const bool ok = e >= 0 && e < E && bb >= 0 && bb < N;
                if (ok) {
                    sfor<Cfg::NOUT>([&](auto jj) {
                        constexpr int j = decltype(jj)::value;
                        if (pc == j) {
                            constexpr int nrow = 2 * Cfg::table.outs[j].l + 1;
                            constexpr int npb = PP::bpos[j + 1] - PP::bpos[j];
                            constexpr int zo = Off<Cfg>::z[j];
#pragma unroll
                            for (int r = 0; r < nrow; ++r)
                                cp_async_slice<T>(slot + r * B::ROWB + c0 * sizeof(T),
                                                  dm + (bb * Cfg::D + zo + r) * kPipeNq + c0);
                            sfor<npb>([&](auto ii) {
                                constexpr int i = decltype(ii)::value;
                                constexpr int p = PP::bpath[PP::bpos[j] + i];
                                cp_async_slice<T>(slot + (nrow + i) * B::ROWB + c0 * sizeof(T),
                                                  w + (e * Cfg::NP + p) * kPipeNq + c0);
                                cp_async_slice<T>(slot + (nrow + npb + i) * B::ROWB + c0 * sizeof(T),
                                                  ddw + (e * Cfg::NP + p) * kPipeNq + c0);
                            });
                        }
                    });
                    if (pc == 0 && lane < 2 * (B::YB / 16)) {
                        const int h = lane / (B::YB / 16), o = lane % (B::YB / 16);
                        const T* ys = (h == 0 ? y : ddy) + e * Cfg::D2;
                        cp_async16(slot + B::ROWS * B::ROWB + h * B::YB + o * 16,
                                   reinterpret_cast<const unsigned char*>(ys) + o * 16);
                    }
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
    for (int64_t a = gw0; a < N; a += nw) {
        int64_t k0 = __ldg(cptr + a), k1 = __ldg(cptr + a + 1);
        if (!seg_ok(k0, k1, E)) {
            if (lane == 0) atomicOr(err, kErrRowptr);
            k0 = k1 = 0;
        }
        if (a == pad) k0 = k1 = 0;
        Q2 gxa[Cfg::D1];
#pragma unroll
        for (int r = 0; r < Cfg::D1; ++r) gxa[r] = q2_zero();
#pragma unroll
        for (int h = 0; h < 2; ++h) {   // items: x rows -> sx, ddx rows -> sdx
            issue(issued++);
            cp_async_wait<NSLOT - 1>();
            const unsigned char* slot = wsm + int(item % NSLOT) * B::SLOT;
            ++item;
            stage_rows<Cfg, T>(slot, h == 0 ? sx : sdx, c0);
        }
        for (int64_t k = k0; k < k1; ++k) {
            const int64_t e = __ldg(cedge + k), bb = __ldg(crecv + k);
            if (pad >= 0 && bb == pad) continue;   // not issued by the producer either
            const bool ok = e >= 0 && e < E && bb >= 0 && bb < N;
            if (!ok && lane == 0) atomicOr(err, kErrRecv);
            float dyp[Cfg::D2];
#pragma unroll
            for (int t = 0; t < Cfg::D2; ++t) dyp[t] = 0.f;
            float* gw_e = gw + (ok ? e : 0) * (Cfg::NP * kPipeNq);
            sfor<B::NCH>([&](auto jj) {
                constexpr int j = decltype(jj)::value;
                issue(issued++);
                cp_async_wait<NSLOT - 1>();
                const unsigned char* slot = wsm + int(item % NSLOT) * B::SLOT;
                ++item;
                if constexpr (j == 0) {
                    __syncwarp();
                    if (ok) {
                        const T* sy = reinterpret_cast<const T*>(slot + B::ROWS * B::ROWB);
                        build_A_warp<Cfg, false, T>(sy, reinterpret_cast<float2*>(sAy), lane, scale);
                        build_A_warp<Cfg, false, T>(reinterpret_cast<const T*>(slot + B::ROWS * B::ROWB + B::YB),
                                                    reinterpret_cast<float2*>(sAd), lane, scale);
                    }
                    __syncwarp();
                }
                if (ok) dbwd_block<Cfg, T, j>(slot, sAy, sAd, sx, sdx, gxa, dyp, gw_e, c0);
                if constexpr (j == B::NCH - 1) __syncwarp();
            });
            int di = 0;
            const float dsum = warp_sum_transposed<Cfg::D2>(dyp, lane, &di);
            if (ok && (lane & (32 / Cfg::D2 - 1)) == 0) gy[e * Cfg::D2 + di] = dsum * scale;
        }
#pragma unroll
        for (int r = 0; r < Cfg::D1; ++r)
            *reinterpret_cast<float4*>(gx + (a * Cfg::D1 + r) * kPipeNq + c0) =
                make_float4(gxa[r].lo.x, gxa[r].lo.y, gxa[r].hi.x, gxa[r].hi.y);
    }
    cp_async_wait<0>();
}

template <class Cfg, class T, bool SENDER>
struct DdPipeShape {
    // 2 slots for the sender pass (its items are 15 rows) and 3 for the receiver pass give
    // 8 warps per SM; measured on the 64k-atom workload: sender 3 -> 2 slots 69.4 -> 58.1 ms,
    // receiver 4 -> 3 slots a further ~2 ms
    static constexpr int NSLOT = SENDER ? 2 : 3;
    static constexpr int WARP_BYTES =
        SENDER ? DbwdPipe<Cfg, T, NSLOT>::WARP_BYTES : DdmPipe<Cfg, T, NSLOT>::WARP_BYTES;
    static constexpr int by_smem = kSmemLimit / WARP_BYTES;
    static constexpr int WARPS = by_smem < 8 ? by_smem : 8;
    static constexpr int SMEM = WARPS * WARP_BYTES;
    // the receiver pass keeps every output row of its receiver in registers: at most 32
    static constexpr bool usable = (Cfg::D2 * sizeof(T)) % 16 == 0 && WARPS >= 4 &&
                                   2 * (Cfg::D2 * sizeof(T) + 15) / 16 <= 32 && (SENDER || Cfg::D <= 32);
};

}  // namespace e3gb
