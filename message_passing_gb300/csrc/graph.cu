// Sender-major (CSC) index of a receiver-sorted CSR graph, built on the device.
//
// The backward convolution ("e3j ...", App. E.1 Eq. 16) is a message-passing operation on
// the transposed graph: dx[a] sums over the edges whose sender is a. Walking the edges in
// sender order lets one row group own dx[a] and sum it in registers in a fixed order, with
// no atomics (the pages' TPU backward reduces dx keyed on senders for the same reason,
// App. E.4 Alg. 7). Steps:
//   1. count edges per sender (integer atomics: the counts do not depend on order);
//   2. exclusive scan of the counts -> csc_ptr (one block);
//   3. place each edge id into its sender's segment (any order);
//   4. sort every segment by edge id (rank counting), which makes the index stable and
//      deterministic;
//   5. csc_recv[k] = receiver of csc_edge[k] (binary search in rowptr).
// Workspace: the per-sender counters / cursors (n_nodes + 1 ints).
#include <cuda_runtime.h>

#include <cstdint>

namespace e3gb {

namespace {
constexpr unsigned kErrSender = 1u, kErrRowptr = 2u;

__global__ void count_kernel(int64_t N, int64_t E, const int32_t* __restrict__ sender, int32_t* __restrict__ cnt,
                             unsigned* __restrict__ err) {
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < E; e += int64_t(gridDim.x) * blockDim.x) {
        const int32_t s = sender[e];
        if (s < 0 || s >= N) {
            atomicOr(err, kErrSender);
            continue;
        }
        atomicAdd(cnt + s, 1);
    }
}

// exclusive scan of cnt[0..N) into ptr[0..N], and cnt <- ptr[0..N) (the placement cursors)
__global__ void __launch_bounds__(1024) scan_kernel(int64_t N, int32_t* __restrict__ cnt, int32_t* __restrict__ ptr) {
    __shared__ int64_t part[1024];
    const int t = threadIdx.x;
    const int64_t chunk = (N + 1023) / 1024;
    const int64_t lo = t * chunk, hi = (lo + chunk < N) ? lo + chunk : N;
    int64_t s = 0;
    for (int64_t i = lo; i < hi; ++i) s += cnt[i];
    part[t] = s;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
        const int64_t v = t >= off ? part[t - off] : 0;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    int64_t run = t > 0 ? part[t - 1] : 0;   // exclusive prefix of this thread's chunk
    for (int64_t i = lo; i < hi; ++i) {
        const int32_t c = cnt[i];
        ptr[i] = int32_t(run);
        cnt[i] = int32_t(run);
        run += c;
    }
    if (t == 1023) ptr[N] = int32_t(part[1023]);
}

__global__ void place_kernel(int64_t N, int64_t E, const int32_t* __restrict__ rowptr,
                             const int32_t* __restrict__ sender, const int32_t* __restrict__ ptr,
                             int32_t* __restrict__ cursor, int32_t* __restrict__ tmp,
                             unsigned* __restrict__ err) {
    for (int64_t b = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; b < N; b += int64_t(gridDim.x) * blockDim.x) {
        const int64_t e0 = rowptr[b], e1 = rowptr[b + 1];
        if (e0 < 0 || e1 < e0 || e1 > E) {
            atomicOr(err, kErrRowptr);
            continue;
        }
        for (int64_t e = e0; e < e1; ++e) {
            const int32_t s = sender[e];
            if (s < 0 || s >= N) continue;   // flagged by count_kernel
            const int32_t pos = atomicAdd(cursor + s, 1);
            if (pos >= ptr[s + 1]) {   // overlapping CSR segments: more placements than edges
                atomicOr(err, kErrRowptr);
                continue;
            }
            tmp[pos] = int32_t(e);
        }
    }
}

// one block per sender segment: out[ptr[a] + rank(v)] = v, rank = #values smaller than v
__global__ void rank_kernel(int64_t N, const int32_t* __restrict__ ptr, const int32_t* __restrict__ cursor,
                            const int32_t* __restrict__ tmp, int32_t* __restrict__ out) {
    for (int64_t a = blockIdx.x; a < N; a += gridDim.x) {
        const int64_t s = ptr[a];
        const int64_t cap = int64_t(ptr[a + 1]) - s;
        // edges of a rejected receiver segment never arrive: the cursor says how many did
        int64_t n = int64_t(cursor[a]) - s;
        n = n < cap ? n : cap;
        // slots that no valid edge fills stay marked invalid (-1)
        for (int64_t i = threadIdx.x; i < cap; i += blockDim.x) out[s + i] = -1;
        __syncthreads();
        for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
            const int32_t v = tmp[s + i];
            int64_t r = 0;
            for (int64_t j = 0; j < n; ++j) r += tmp[s + j] < v;
            out[s + r] = v;
        }
        __syncthreads();
    }
}

__global__ void recv_kernel(int64_t N, int64_t K, const int32_t* __restrict__ rowptr,
                            const int32_t* __restrict__ edge, int32_t* __restrict__ recv) {
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < K; k += int64_t(gridDim.x) * blockDim.x) {
        const int32_t e = edge[k];
        if (e < 0) {
            recv[k] = -1;
            continue;
        }
        // largest b with rowptr[b] <= e
        int64_t lo = 0, hi = N;   // invariant: rowptr[lo] <= e < rowptr[hi]
        while (hi - lo > 1) {
            const int64_t mid = (lo + hi) >> 1;
            if (rowptr[mid] <= e) lo = mid; else hi = mid;
        }
        recv[k] = int32_t(lo);
    }
}

// Zero the dw and dy rows of every padding edge: the edges into the padding receiver (found
// by a warp-wide ballot over csc_recv) and the padding sender's edges (its sender-major
// segment). Each padding edge appears once in the sender-major index, so each row has one
// writer. Edge ids out of range are left alone (the conv kernel flags them).
__global__ void zero_padding_kernel(int64_t N, int64_t E, const int32_t* __restrict__ cptr,
                                    const int32_t* __restrict__ cedge, const int32_t* __restrict__ crecv,
                                    int64_t pad, float* __restrict__ dw, int64_t dw_row, float* __restrict__ dy,
                                    int64_t dy_row) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = (int64_t(gridDim.x) * blockDim.x) >> 5;
    int64_t s0 = cptr[pad], s1 = cptr[pad + 1];
    if (s0 < 0 || s1 < s0 || s1 > E) s0 = s1 = 0;
    for (int64_t base = gw * 32; base < E; base += nw * 32) {   // warp-uniform trip count
        const int64_t k = base + lane;
        int64_t e = -1;
        if (k < E && (crecv[k] == pad || (k >= s0 && k < s1))) {
            e = cedge[k];
            if (e >= E) e = -1;
        }
        unsigned todo = __ballot_sync(0xffffffffu, e >= 0);
        while (todo) {
            const int src = __ffs(todo) - 1;
            todo &= todo - 1;
            const int64_t ee = __shfl_sync(0xffffffffu, e, src);
            float* r = dw + ee * dw_row;
            for (int64_t i = lane; i < dw_row; i += 32) __stcs(r + i, 0.f);
            for (int64_t i = lane; i < dy_row; i += 32) dy[ee * dy_row + i] = 0.f;
        }
    }
}

inline int grid1d(int64_t n, int block, int cap) {
    const int64_t g = (n + block - 1) / block;
    return int(g < cap ? (g > 0 ? g : 1) : cap);
}
}  // namespace

cudaError_t zero_padding_edges(int64_t N, int64_t E, const int32_t* csc_ptr, const int32_t* csc_edge,
                               const int32_t* csc_recv, int64_t pad, float* dw, int64_t dw_row, float* dy,
                               int64_t dy_row, cudaStream_t s) {
    if (E <= 0 || pad < 0 || pad >= N) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t st = cudaGetDevice(&dev);
    if (st == cudaSuccess) st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (st != cudaSuccess) return st;
    const int block = 256;
    zero_padding_kernel<<<grid1d((E + 7) / 8, block, sms * 8), block, 0, s>>>(N, E, csc_ptr, csc_edge, csc_recv, pad,
                                                                              dw, dw_row, dy, dy_row);
    return cudaGetLastError();
}

size_t graph_workspace_bytes(int64_t N) { return size_t((N + 1) * 4 + 255) / 256 * 256; }

cudaError_t graph_prepare(int64_t N, int64_t E, const int32_t* rowptr, const int32_t* sender, int32_t* csc_ptr,
                          int32_t* csc_edge, int32_t* csc_recv, void* ws, unsigned* err, cudaStream_t s) {
    int32_t* cnt = static_cast<int32_t*>(ws);
    cudaError_t st = cudaMemsetAsync(cnt, 0, size_t(N + 1) * 4, s);
    if (st != cudaSuccess) return st;
    if (E > 0) count_kernel<<<grid1d(E, 256, 4096), 256, 0, s>>>(N, E, sender, cnt, err);
    scan_kernel<<<1, 1024, 0, s>>>(N, cnt, csc_ptr);
    if (E > 0) {
        // csc_recv is the temporary for unsorted segments; it is overwritten in step 5
        place_kernel<<<grid1d(N, 256, 4096), 256, 0, s>>>(N, E, rowptr, sender, csc_ptr, cnt, csc_recv, err);
        rank_kernel<<<int(N < 65535 ? (N > 0 ? N : 1) : 65535), 64, 0, s>>>(N, csc_ptr, cnt, csc_recv, csc_edge);
        recv_kernel<<<grid1d(E, 256, 4096), 256, 0, s>>>(N, E, rowptr, csc_edge, csc_recv);
    }
    return cudaGetLastError();
}

}  // namespace e3gb
