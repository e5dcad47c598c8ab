// One irreps configuration's kernels and launchers; compiled six times per entry of configs.def,
// with -DE3GB_CFG=<id> -DE3GB_PART=0 (forward kernels and the ops table e3gb::ops_<id>())
// -DE3GB_PART=1 (backward kernels), -DE3GB_PART=2 (double backward, plain kernels),
// -DE3GB_PART=3 (double backward, 128-channel pipelined kernels), -DE3GB_PART=4 (forward,
// edge-slot kernels for 4-32 channels) and -DE3GB_PART=5 (the radial convolution, forward and
// backward), so that the parts compile in parallel.
#include "conv_pipe.cuh"
#include "conv_pipe_dd.cuh"
#include "conv_slots.cuh"
#include "conv_split.cuh"
#include "kernels.cuh"

#include <type_traits>

#if !defined(E3GB_CFG) || !defined(E3GB_PART)
#error "compile with -DE3GB_CFG=<config id> -DE3GB_PART=<0|1|2|3|4|5>"
#endif
#define E3GB_CAT2(a, b) a##b
#define E3GB_CAT(a, b) E3GB_CAT2(a, b)

namespace e3gb {

template <class... B>
constexpr uint32_t xcode(B... b) {
    uint32_t c = 0;
    int i = 0;
    ((c |= uint32_t(b) << (4 * i++)), ...);
    return c;
}

template <int ID>
struct Pick;
#define E3GB_CONFIG(ID, XC, L2, L3, PP) \
    template <>                         \
    struct Pick<ID> {                   \
        using type = Config<XC, L2, L3, PP>; \
    };
#include "configs.def"
#undef E3GB_CONFIG

namespace E3GB_CAT(cfg, E3GB_CFG) {
using Cfg = typename Pick<E3GB_CFG>::type;
constexpr int kBlock = 256;

// channels per lane of the plain kernels: 4 for wide rows, 1 for narrow ones (keeps the
// accumulators of all output rows in registers without spilling)
constexpr int vec_for(int Nq) { return Nq >= 64 ? 4 : 1; }
static int rows_per_block(int Nq) { return (kBlock / 32) * (32 / (Nq / vec_for(Nq))); }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// configurations whose receiver outputs fit in registers (the receiver-stationary forwards keep
// all of them live); others (one output block per path) walk the edges once per output block
constexpr bool kRowsFit = Cfg::D <= 32;

// The bf16 pipelined backward faulted ("illegal instruction") on its first run on the 0e+1o
// configuration, and reading it did not show why; the bf16 pipelined kernels (conv forward
// and backward, the row backward on the identity graph, the double backward), which share its
// staging, are launched only on the configuration where they have run in every test and
// benchmark (x irreps 0e+1o+2e, SH and outputs l <= 3). Other bf16 configurations take the
// plain kernels.
template <class T>
constexpr bool pipe_cleared() {
    if constexpr (std::is_same_v<T, float>) return true;
    else return Cfg::xcode == xcode(xblock(0, 1), xblock(1, -1), xblock(2, 1)) && Cfg::L2 == 3 && Cfg::L3 == 3 &&
                !Cfg::per_path;
}

template <class T>
cudaError_t tp_fwd(int64_t R, int Nq, const void* x, const void* y, const void* w, void* z, cudaStream_t s);
template <class T>
cudaError_t tp_bwd(int64_t R, int Nq, const void* x, const void* y, const void* w, const void* dz, void* dx,
                   void* dy, void* dw, cudaStream_t s);
template <class T>
cudaError_t conv_fwd(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const void* x,
                     const void* y, const void* w, float scale, void* m, int64_t pad, unsigned* err, int64_t cap,
                     cudaStream_t s);
// the further pieces of heavy receivers (part 4)
template <class T>
cudaError_t conv_fwd_pieces(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const void* x,
                            const void* y, const void* w, float scale, void* m, int64_t pad, int64_t cap, void* ws,
                            unsigned* err, cudaStream_t s);
template <class T>
cudaError_t conv_bwd(int64_t N, int64_t E, int Nq, const int32_t* cptr, const int32_t* cedge, const int32_t* crecv,
                     const void* x, const void* y, const void* w, const void* dm, float scale, void* dx, void* dy,
                     void* dw, int64_t pad, unsigned* err, cudaStream_t s);
template <class T>
cudaError_t conv_dbwd(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const int32_t* cptr,
                      const int32_t* cedge, const int32_t* crecv, const void* x, const void* y, const void* w,
                      const void* dm, const void* ddx, const void* ddy, const void* ddw, float scale, void* gx,
                      void* gy, void* gw, void* gdm, int64_t pad, unsigned* err, cudaStream_t s);
// the edge-slot forward for 4-32 channels (part 4); returns false when the shape needs the
// plain kernels
template <class T>
bool conv_fwd_slots(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const void* x,
                    const void* y, const void* w, float scale, void* m, int64_t pad, unsigned* err, int64_t cap,
                    cudaStream_t s, cudaError_t* st);
// the radial convolution, fp32 (part 5): weights formed in the kernels from the hidden
// activations h [E][kRadialHidden] and the output layer W2 [kRadialHidden][NP][Nq]
cudaError_t conv_fwd_rad(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const float* x,
                         const float* y, const float* h, const float* W2, float scale, float* m, int64_t pad,
                         unsigned* err, cudaStream_t s);
cudaError_t conv_bwd_rad(int64_t N, int64_t E, int Nq, const int32_t* cptr, const int32_t* cedge,
                         const int32_t* crecv, const float* x, const float* y, const float* h, const float* W2,
                         const float* dm, float scale, float* dx, float* dy, float* dh, int64_t pad, unsigned* err,
                         cudaStream_t s);
// the pipelined double backward (part 3); returns false when the shape needs the plain kernels
template <class T>
bool conv_dbwd_pipe(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const int32_t* cptr,
                    const int32_t* cedge, const int32_t* crecv, const void* x, const void* y, const void* w,
                    const void* dm, const void* ddx, const void* ddy, const void* ddw, float scale, void* gx, void* gy,
                    void* gw, void* gdm, int64_t pad, unsigned* err, cudaStream_t s, cudaError_t* st);

#if E3GB_PART == 0
template <class T>
cudaError_t tp_fwd(int64_t R, int Nq, const void* x, const void* y, const void* w, void* z, cudaStream_t s) {
    auto k = vec_for(Nq) == 4 ? tp_forward_kernel<Cfg, T, 4> : tp_forward_kernel<Cfg, T, 1>;
    // 4 channels per lane: 12 warps per block (at <= 168 registers, three per scheduler), which
    // measured 11% faster than 8 on the 200k-row workload; one channel per lane: 8
    const int blk = vec_for(Nq) == 4 ? 384 : kBlock;
    const int grid = grid_for((const void*)k, blk, (blk / 32) * (32 / (Nq / vec_for(Nq))), R);
    if (grid == 0) return cudaSuccess;
    k<<<grid, blk, 0, s>>>(R, Nq, (const T*)x, (const T*)y, (const T*)w, (float*)z);
    return cudaGetLastError();
}

#endif  // part 0

#if E3GB_PART == 1
template <class T>
cudaError_t tp_bwd(int64_t R, int Nq, const void* x, const void* y, const void* w, const void* dz, void* dx,
                   void* dy, void* dw, cudaStream_t s) {
    using S = PipeShape<Cfg, T, true>;
    if constexpr (S::usable && pipe_cleared<T>()) {
        // 128 channels: the pipelined convolution backward on the identity graph (row r is node
        // r with the one edge r), which streams the rows through the per-warp cp.async ring
        if (Nq == kPipeNq && aligned16(x) && aligned16(y) && aligned16(w) && aligned16(dz)) {
            auto k = conv_backward_pipe_kernel<Cfg, T, S::NSLOT, S::WARPS, true>;
            cudaError_t st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (st != cudaSuccess) return st;
            const int64_t need = (R + S::WARPS - 1) / S::WARPS;
            const int grid = int(sm_count() < need ? sm_count() : need);
            if (grid == 0) return cudaSuccess;
            k<<<grid, S::WARPS * 32, S::SMEM, s>>>(R, R, nullptr, nullptr, nullptr, (const T*)x, (const T*)y,
                                                   (const T*)w, (const T*)dz, 1.f, (float*)dx, (float*)dy, (float*)dw,
                                                   -1, nullptr, nullptr, nullptr);
            return cudaGetLastError();
        }
    }
    auto k = vec_for(Nq) == 4 ? tp_backward_kernel<Cfg, T, 4> : tp_backward_kernel<Cfg, T, 1>;
    const int grid = grid_for((const void*)k, kBlock, rows_per_block(Nq), R);
    if (grid == 0) return cudaSuccess;
    k<<<grid, kBlock, 0, s>>>(R, Nq, (const T*)x, (const T*)y, (const T*)w, (const T*)dz, (float*)dx,
                              (float*)dy, (float*)dw);
    return cudaGetLastError();
}

#endif  // part 1

#if E3GB_PART == 0
template <class T>
cudaError_t conv_fwd_rows(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const void* x,
                          const void* y, const void* w, float scale, void* m, int64_t pad, unsigned* err,
                          int64_t cap, cudaStream_t s);

template <class T>
cudaError_t conv_fwd(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const void* x,
                     const void* y, const void* w, float scale, void* m, int64_t pad, unsigned* err, int64_t cap,
                     cudaStream_t s) {
    if constexpr (!kRowsFit) {
        auto k = vec_for(Nq) == 4 ? conv_forward_blocks_kernel<Cfg, T, 4> : conv_forward_blocks_kernel<Cfg, T, 1>;
        const int grid = grid_for((const void*)k, kBlock, rows_per_block(Nq), N);
        if (grid == 0) return cudaSuccess;
        k<<<grid, kBlock, 0, s>>>(N, E, Nq, rowptr, sender, (const T*)x, (const T*)y, (const T*)w, scale, (float*)m,
                                  pad, err, cap);
        return cudaGetLastError();
    } else {
        return conv_fwd_rows<T>(N, E, Nq, rowptr, sender, x, y, w, scale, m, pad, err, cap, s);
    }
}

template <class T>
cudaError_t conv_fwd_rows(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const void* x,
                          const void* y, const void* w, float scale, void* m, int64_t pad, unsigned* err,
                          int64_t cap, cudaStream_t s) {
    using S = PipeShape<Cfg, T, false>;
    if constexpr (S::usable && pipe_cleared<T>()) {
        if (Nq == kPipeNq && aligned16(x) && aligned16(y) && aligned16(w)) {
            auto k = conv_forward_pipe_kernel<Cfg, T, S::NSLOT, S::WARPS>;
            cudaError_t st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (st != cudaSuccess) return st;
            const int64_t need = (N + S::WARPS - 1) / S::WARPS;
            const int grid = int(sm_count() < need ? sm_count() : need);
            if (grid == 0) return cudaSuccess;
            k<<<grid, S::WARPS * 32, S::SMEM, s>>>(N, E, rowptr, sender, (const T*)x, (const T*)y, (const T*)w, scale,
                                                   (float*)m, pad, err, cap, nullptr, nullptr);
            return cudaGetLastError();
        }
    }
    cudaError_t sst = cudaSuccess;
    if (conv_fwd_slots<T>(N, E, Nq, rowptr, sender, x, y, w, scale, m, pad, err, cap, s, &sst)) return sst;
    auto k = vec_for(Nq) == 4 ? conv_forward_kernel<Cfg, T, 4> : conv_forward_kernel<Cfg, T, 1>;
    const int grid = grid_for((const void*)k, kBlock, rows_per_block(Nq), N);
    if (grid == 0) return cudaSuccess;
    k<<<grid, kBlock, 0, s>>>(N, E, Nq, rowptr, sender, (const T*)x, (const T*)y, (const T*)w, scale, (float*)m,
                              pad, err, cap, nullptr, nullptr);
    return cudaGetLastError();
}

#endif  // part 0

#if E3GB_PART == 4
template <class T, int NQ>
static cudaError_t launch_fwd_slots(int64_t N, int64_t E, const int32_t* rowptr, const int32_t* sender, const void* x,
                                    const void* y, const void* w, float scale, void* m, int64_t pad, unsigned* err,
                                    int64_t cap, cudaStream_t s) {
    auto k = conv_forward_slots_kernel<Cfg, T, NQ>;
    constexpr int smem = slots_fwd_smem<Cfg, T>();
    cudaError_t st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (st != cudaSuccess) return st;
    const int grid = grid_for((const void*)k, kBlock, slots_nodes_per_block<NQ>(), N);
    if (grid == 0) return cudaSuccess;
    k<<<grid, kBlock, smem, s>>>(N, E, rowptr, sender, (const T*)x, (const T*)y, (const T*)w, scale, (float*)m, pad,
                                 err, cap);
    return cudaGetLastError();
}

template <class T>
bool conv_fwd_slots(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const void* x,
                    const void* y, const void* w, float scale, void* m, int64_t pad, unsigned* err, int64_t cap,
                    cudaStream_t s, cudaError_t* st) {
    if constexpr (SlotsFit<Cfg>::value) {
        if (aligned16(x) && aligned16(y) && aligned16(w) && aligned16(m)) {
            switch (Nq) {
            case 4: *st = launch_fwd_slots<T, 4>(N, E, rowptr, sender, x, y, w, scale, m, pad, err, cap, s); return true;
            case 8: *st = launch_fwd_slots<T, 8>(N, E, rowptr, sender, x, y, w, scale, m, pad, err, cap, s); return true;
            case 16: *st = launch_fwd_slots<T, 16>(N, E, rowptr, sender, x, y, w, scale, m, pad, err, cap, s); return true;
            case 32: *st = launch_fwd_slots<T, 32>(N, E, rowptr, sender, x, y, w, scale, m, pad, err, cap, s); return true;
            default: break;
            }
        }
    }
    return false;
}

template bool conv_fwd_slots<float>(int64_t, int64_t, int, const int32_t*, const int32_t*, const void*, const void*,
                                     const void*, float, void*, int64_t, unsigned*, int64_t, cudaStream_t,
                                     cudaError_t*);
template bool conv_fwd_slots<__nv_bfloat16>(int64_t, int64_t, int, const int32_t*, const int32_t*, const void*,
                                             const void*, const void*, float, void*, int64_t, unsigned*, int64_t,
                                             cudaStream_t, cudaError_t*);

// heavy receivers: count the further pieces, scan, sum each piece, add the pieces to m in
// order. Workspace: piece pointers (N + 1 ints), the scan's block sums, the partial rows.
template <class T>
cudaError_t conv_fwd_pieces(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const void* x,
                            const void* y, const void* w, float scale, void* m, int64_t pad, int64_t cap, void* ws,
                            unsigned* err, cudaStream_t s) {
    if constexpr (!kRowsFit) {   // the host rejects these configurations
        return cudaErrorNotSupported;
    } else {
        if (N <= 0 || E <= cap) return cudaSuccess;
        int32_t* ptr = static_cast<int32_t*>(ws);
        int32_t* sums = ptr + (N + 1 + 63) / 64 * 64;
        float* partials = reinterpret_cast<float*>(sums + (scan_sums_count(N + 1) + 63) / 64 * 64);
        piece_count_kernel<<<int((N + 256) / 256 < 4096 ? (N + 256) / 256 : 4096), 256, 0, s>>>(N, E, rowptr, pad,
                                                                                                 cap, ptr);
        cudaError_t st = exclusive_scan_i32(ptr, N + 1, sums, s);
        if (st != cudaSuccess) return st;
        auto k = vec_for(Nq) == 4 ? conv_forward_pieces_kernel<Cfg, T, 4> : conv_forward_pieces_kernel<Cfg, T, 1>;
        const int grid = grid_for((const void*)k, kBlock, rows_per_block(Nq), E / cap + 1);
        k<<<grid, kBlock, 0, s>>>(N, E, Nq, rowptr, sender, (const T*)x, (const T*)y, (const T*)w, pad, cap, ptr,
                                  partials, err);
        st = cudaGetLastError();
        if (st != cudaSuccess) return st;
        const int64_t row = int64_t(Cfg::D) * Nq;
        const dim3 cgrid(unsigned(N < 2048 ? N : 2048), unsigned((row + 255) / 256));
        conv_pieces_combine_kernel<<<cgrid, 256, 0, s>>>(N, row, ptr, partials, scale, (float*)m);
        return cudaGetLastError();
    }
}

template cudaError_t conv_fwd_pieces<float>(int64_t, int64_t, int, const int32_t*, const int32_t*, const void*,
                                            const void*, const void*, float, void*, int64_t, int64_t, void*, unsigned*,
                                            cudaStream_t);
template cudaError_t conv_fwd_pieces<__nv_bfloat16>(int64_t, int64_t, int, const int32_t*, const int32_t*, const void*,
                                                    const void*, const void*, float, void*, int64_t, int64_t, void*,
                                                    unsigned*, cudaStream_t);
#endif  // part 4

#if E3GB_PART == 1
template <class T>
cudaError_t conv_bwd(int64_t N, int64_t E, int Nq, const int32_t* cptr, const int32_t* cedge, const int32_t* crecv,
                     const void* x, const void* y, const void* w, const void* dm, float scale, void* dx, void* dy,
                     void* dw, int64_t pad, unsigned* err, cudaStream_t s) {
    using S = PipeShape<Cfg, T, true>;
    if constexpr (S::usable && pipe_cleared<T>()) {
        if (Nq == kPipeNq && aligned16(x) && aligned16(y) && aligned16(w) && aligned16(dm)) {
            auto k = conv_backward_pipe_kernel<Cfg, T, S::NSLOT, S::WARPS>;
            cudaError_t st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (st != cudaSuccess) return st;
            const int64_t need = (N + S::WARPS - 1) / S::WARPS;
            const int grid = int(sm_count() < need ? sm_count() : need);
            if (grid == 0) return cudaSuccess;
            k<<<grid, S::WARPS * 32, S::SMEM, s>>>(N, E, cptr, cedge, crecv, (const T*)x, (const T*)y, (const T*)w,
                                                   (const T*)dm, scale, (float*)dx, (float*)dy, (float*)dw, pad, err,
                                                   nullptr, nullptr);
            return cudaGetLastError();
        }
    }
    auto k = vec_for(Nq) == 4 ? conv_backward_kernel<Cfg, T, 4> : conv_backward_kernel<Cfg, T, 1>;
    const int grid = grid_for((const void*)k, kBlock, rows_per_block(Nq), N);
    if (grid == 0) return cudaSuccess;
    k<<<grid, kBlock, 0, s>>>(N, E, Nq, cptr, cedge, crecv, (const T*)x, (const T*)y, (const T*)w,
                              (const T*)dm, scale, (float*)dx, (float*)dy, (float*)dw, pad, err, nullptr, nullptr);
    return cudaGetLastError();
}

template cudaError_t tp_bwd<float>(int64_t, int, const void*, const void*, const void*, const void*, void*, void*,
                                    void*, cudaStream_t);
template cudaError_t tp_bwd<__nv_bfloat16>(int64_t, int, const void*, const void*, const void*, const void*, void*,
                                            void*, void*, cudaStream_t);
template cudaError_t conv_bwd<float>(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                                      const void*, const void*, const void*, const void*, float, void*, void*, void*,
                                      int64_t, unsigned*, cudaStream_t);
template cudaError_t conv_bwd<__nv_bfloat16>(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                                              const void*, const void*, const void*, const void*, float, void*, void*,
                                              void*, int64_t, unsigned*, cudaStream_t);
#endif  // part 1
#if E3GB_PART == 2
template <class T>
cudaError_t conv_dbwd(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const int32_t* cptr,
                      const int32_t* cedge, const int32_t* crecv, const void* x, const void* y, const void* w,
                      const void* dm, const void* ddx, const void* ddy, const void* ddw, float scale, void* gx,
                      void* gy, void* gw, void* gdm, int64_t pad, unsigned* err, cudaStream_t s) {
    cudaError_t pst = cudaSuccess;
    if (conv_dbwd_pipe<T>(N, E, Nq, rowptr, sender, cptr, cedge, crecv, x, y, w, dm, ddx, ddy, ddw, scale, gx, gy,
                          gw, gdm, pad, err, s, &pst))
        return pst;
    auto kr = vec_for(Nq) == 4 ? conv_ddm_kernel<Cfg, T, 4> : conv_ddm_kernel<Cfg, T, 1>;
    const int gr = grid_for((const void*)kr, kBlock, rows_per_block(Nq), N);
    if (gr == 0) return cudaSuccess;
    kr<<<gr, kBlock, 0, s>>>(N, E, Nq, rowptr, sender, (const T*)x, (const T*)y, (const T*)w, (const T*)ddx,
                             (const T*)ddy, (const T*)ddw, scale, (float*)gdm, pad, err);
    cudaError_t st = cudaGetLastError();
    if (st != cudaSuccess) return st;
    auto ks = vec_for(Nq) == 4 ? conv_dbwd_kernel<Cfg, T, 4> : conv_dbwd_kernel<Cfg, T, 1>;
    const int gs = grid_for((const void*)ks, kBlock, rows_per_block(Nq), N);
    ks<<<gs, kBlock, 0, s>>>(N, E, Nq, cptr, cedge, crecv, (const T*)x, (const T*)y, (const T*)w, (const T*)dm,
                             (const T*)ddx, (const T*)ddy, (const T*)ddw, scale, (float*)gx, (float*)gy, (float*)gw,
                             pad, err);
    return cudaGetLastError();
}

template cudaError_t conv_dbwd<float>(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                                       const int32_t*, const int32_t*, const void*, const void*, const void*,
                                       const void*, const void*, const void*, const void*, float, void*, void*, void*,
                                       void*, int64_t, unsigned*, cudaStream_t);
template cudaError_t conv_dbwd<__nv_bfloat16>(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                                               const int32_t*, const int32_t*, const void*, const void*, const void*,
                                               const void*, const void*, const void*, const void*, float, void*,
                                               void*, void*, void*, int64_t, unsigned*, cudaStream_t);
#endif  // part 2
#if E3GB_PART == 3
template <class T>
bool conv_dbwd_pipe(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const int32_t* cptr,
                    const int32_t* cedge, const int32_t* crecv, const void* x, const void* y, const void* w,
                    const void* dm, const void* ddx, const void* ddy, const void* ddw, float scale, void* gx, void* gy,
                    void* gw, void* gdm, int64_t pad, unsigned* err, cudaStream_t s, cudaError_t* st) {
    using SR = DdPipeShape<Cfg, T, false>;
    using SS = DdPipeShape<Cfg, T, true>;
    if constexpr (SR::usable && SS::usable && pipe_cleared<T>()) {
        if (Nq == kPipeNq && aligned16(x) && aligned16(y) && aligned16(w) && aligned16(dm) && aligned16(ddx) &&
            aligned16(ddy) && aligned16(ddw)) {
            auto kr = conv_ddm_pipe_kernel<Cfg, T, SR::NSLOT, SR::WARPS>;
            auto ks = conv_dbwd_pipe_kernel<Cfg, T, SS::NSLOT, SS::WARPS>;
            cudaError_t e = cudaFuncSetAttribute((const void*)kr, cudaFuncAttributeMaxDynamicSharedMemorySize, SR::SMEM);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute((const void*)ks, cudaFuncAttributeMaxDynamicSharedMemorySize, SS::SMEM);
            if (e != cudaSuccess) { *st = e; return true; }
            const int64_t nr = (N + SR::WARPS - 1) / SR::WARPS, ns = (N + SS::WARPS - 1) / SS::WARPS;
            const int gr = int(sm_count() < nr ? sm_count() : nr), gs = int(sm_count() < ns ? sm_count() : ns);
            if (gr == 0) { *st = cudaSuccess; return true; }
            kr<<<gr, SR::WARPS * 32, SR::SMEM, s>>>(N, E, rowptr, sender, (const T*)x, (const T*)y, (const T*)w,
                                                     (const T*)ddx, (const T*)ddy, (const T*)ddw, scale, (float*)gdm,
                                                     pad, err);
            e = cudaGetLastError();
            if (e != cudaSuccess) { *st = e; return true; }
            ks<<<gs, SS::WARPS * 32, SS::SMEM, s>>>(N, E, cptr, cedge, crecv, (const T*)x, (const T*)y, (const T*)w,
                                                     (const T*)dm, (const T*)ddx, (const T*)ddy, (const T*)ddw, scale,
                                                     (float*)gx, (float*)gy, (float*)gw, pad, err);
            *st = cudaGetLastError();
            return true;
        }
    }
    return false;
}

template bool conv_dbwd_pipe<float>(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                                     const int32_t*, const int32_t*, const void*, const void*, const void*, const void*,
                                     const void*, const void*, const void*, float, void*, void*, void*, void*, int64_t,
                                     unsigned*, cudaStream_t, cudaError_t*);
template bool conv_dbwd_pipe<__nv_bfloat16>(int64_t, int64_t, int, const int32_t*, const int32_t*, const int32_t*,
                                             const int32_t*, const int32_t*, const void*, const void*, const void*,
                                             const void*, const void*, const void*, const void*, float, void*, void*,
                                             void*, void*, int64_t, unsigned*, cudaStream_t, cudaError_t*);
#endif  // part 3
#if E3GB_PART == 5
cudaError_t conv_fwd_rad(int64_t N, int64_t E, int Nq, const int32_t* rowptr, const int32_t* sender, const float* x,
                         const float* y, const float* h, const float* W2, float scale, float* m, int64_t pad,
                         unsigned* err, cudaStream_t s) {
    if constexpr (!kRowsFit) {   // the host rejects these configurations
        return cudaErrorNotSupported;
    } else {
    constexpr int RH = kRadialHidden;
    using S = PipeShape<Cfg, float, false, RH>;
    if constexpr (S::usable) {
        if (Nq == kPipeNq && aligned16(x) && aligned16(y) && aligned16(h) && aligned16(W2)) {
            auto k = conv_forward_pipe_kernel<Cfg, float, S::NSLOT, S::WARPS, RH>;
            cudaError_t st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (st != cudaSuccess) return st;
            const int64_t need = (N + S::WARPS - 1) / S::WARPS;
            const int grid = int(sm_count() < need ? sm_count() : need);
            if (grid == 0) return cudaSuccess;
            k<<<grid, S::WARPS * 32, S::SMEM, s>>>(N, E, rowptr, sender, x, y, nullptr, scale, m, pad, err, INT64_MAX,
                                                   h, W2);
            return cudaGetLastError();
        }
    }
    const int smem = RH * Cfg::NP * Nq * 4;
    if (smem > kSmemLimit) return cudaErrorInvalidValue;
    auto k = vec_for(Nq) == 4 ? conv_forward_kernel<Cfg, float, 4, RH> : conv_forward_kernel<Cfg, float, 1, RH>;
    cudaError_t st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (st != cudaSuccess) return st;
    const int grid = grid_for((const void*)k, kBlock, rows_per_block(Nq), N, smem);
    if (grid == 0) return cudaSuccess;
    k<<<grid, kBlock, smem, s>>>(N, E, Nq, rowptr, sender, x, y, nullptr, scale, m, pad, err, INT64_MAX, h, W2);
    return cudaGetLastError();
    }
}

cudaError_t conv_bwd_rad(int64_t N, int64_t E, int Nq, const int32_t* cptr, const int32_t* cedge,
                         const int32_t* crecv, const float* x, const float* y, const float* h, const float* W2,
                         const float* dm, float scale, float* dx, float* dy, float* dh, int64_t pad, unsigned* err,
                         cudaStream_t s) {
    constexpr int RH = kRadialHidden;
    using S = PipeShape<Cfg, float, true, RH>;
    if constexpr (S::usable) {
        if (Nq == kPipeNq && aligned16(x) && aligned16(y) && aligned16(h) && aligned16(W2) && aligned16(dm)) {
            auto k = conv_backward_pipe_kernel<Cfg, float, S::NSLOT, S::WARPS, false, RH>;
            cudaError_t st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
            if (st != cudaSuccess) return st;
            const int64_t need = (N + S::WARPS - 1) / S::WARPS;
            const int grid = int(sm_count() < need ? sm_count() : need);
            if (grid == 0) return cudaSuccess;
            k<<<grid, S::WARPS * 32, S::SMEM, s>>>(N, E, cptr, cedge, crecv, x, y, nullptr, dm, scale, dx, dy, dh, pad,
                                                   err, h, W2);
            return cudaGetLastError();
        }
    }
    const int smem = RH * Cfg::NP * Nq * 4;
    if (smem > kSmemLimit) return cudaErrorInvalidValue;
    auto k = vec_for(Nq) == 4 ? conv_backward_kernel<Cfg, float, 4, RH> : conv_backward_kernel<Cfg, float, 1, RH>;
    cudaError_t st = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (st != cudaSuccess) return st;
    const int grid = grid_for((const void*)k, kBlock, rows_per_block(Nq), N, smem);
    if (grid == 0) return cudaSuccess;
    k<<<grid, kBlock, smem, s>>>(N, E, Nq, cptr, cedge, crecv, x, y, nullptr, dm, scale, dx, dy, dh, pad, err, h, W2);
    return cudaGetLastError();
}
#endif  // part 5
}  // namespace cfg<id>

#if E3GB_PART == 0
namespace {
using namespace E3GB_CAT(cfg, E3GB_CFG);
const ConfigOps kOps = {
    Cfg::xcode, Cfg::L2, Cfg::L3, Cfg::per_path ? 1 : 0,
    Cfg::NP, Cfg::D1, Cfg::D2, Cfg::D, Cfg::NOUT, Cfg::NR,
    Cfg::table.paths.data(), Cfg::table.outs.data(), Cfg::recs.data(),
    {tp_fwd<float>, tp_fwd<__nv_bfloat16>},
    {tp_bwd<float>, tp_bwd<__nv_bfloat16>},
    {conv_fwd<float>, conv_fwd<__nv_bfloat16>},
    {conv_bwd<float>, conv_bwd<__nv_bfloat16>},
    {conv_dbwd<float>, conv_dbwd<__nv_bfloat16>},
    conv_fwd_rad,
    conv_bwd_rad,
    {conv_fwd_pieces<float>, conv_fwd_pieces<__nv_bfloat16>},
};
}  // namespace

const ConfigOps* E3GB_CAT(ops_, E3GB_CFG)() { return &kOps; }
#endif

}  // namespace e3gb
