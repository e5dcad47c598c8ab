// Sender-major (CSC) index of a receiver-sorted CSR graph, built on the device.
//
// The backward convolution ("e3j ...", App. E.1 Eq. 16) is a message-passing operation on
// the transposed graph: dx[a] sums over the edges whose sender is a. Walking the edges in
// sender order lets one row group own dx[a] and sum it in registers in a fixed order, with
// no atomics (the pages' TPU backward reduces dx keyed on senders for the same reason,
// App. E.4 Alg. 7). The index is the edge ids stably sorted by sender, built in O(E) work
// whatever the degree distribution (one padding node may send most of the edges):
//   1. a least-significant-digit radix sort of the edge ids by key = sender, 8 bits per
//      pass, ceil(bits(n_nodes) / 8) passes. Edges that belong to no receiver or have a
//      sender outside [0, n_nodes) get the key n_nodes and sort to the end. Each pass splits
//      the edges into tiles of T consecutive entries, one warp per tile: (a) per-tile digit
//      counts, (b) an exclusive scan of the counts in digit-major order, (c) a stable scatter
//      in which each warp walks its tile in order and ranks equal digits with a match mask.
//      Keys are never stored: each pass gathers sender[edge id] again. The two output arrays
//      csc_edge / csc_recv are the ping-pong buffers, and the last pass lands in csc_edge;
//   2. csc_ptr[a] = first sorted position whose key is >= a (a binary search per node);
//   3. csc_recv[k] = receiver of csc_edge[k] (binary search in rowptr); positions past the
//      valid edges get -1 in both arrays.
// Workspace: the per-tile digit counts (256 per tile) and the scan's block sums.
#include <cuda_runtime.h>

#include <cstdint>

namespace e3gb {

namespace {
constexpr unsigned kErrSender = 1u, kErrRowptr = 2u;
constexpr int kRadixBits = 8, kBins = 1 << kRadixBits;
constexpr int kScanBlock = 1024, kScanItems = 4;          // one scan block covers 4096 counts
constexpr int64_t kScanChunk = int64_t(kScanBlock) * kScanItems;
constexpr int kSortWarps = 8;                              // warps (tiles in flight) per sort block

// Which edges enter the index, and under which key.
struct EdgeKeys {
    int64_t N, E;
    const int32_t* sender;
    const int32_t* rowptr;

    // key = sender for an edge inside [rowptr[0], rowptr[N]) with a sender in [0, N), else N
    __device__ __forceinline__ int32_t key(int32_t e, int64_t lo, int64_t hi) const {
        const int32_t s = __ldg(sender + e);
        return (s >= 0 && s < N && e >= lo && e < hi) ? s : int32_t(N);
    }
    __device__ __forceinline__ void range(int64_t& lo, int64_t& hi) const {
        lo = __ldg(rowptr);
        hi = __ldg(rowptr + N);
        lo = lo < 0 ? 0 : lo;
        hi = hi > E ? E : hi;
    }
};

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// (a) per-tile digit counts: hist[d * n_tiles + tile]. Pass 0 reads the identity order
// (in == nullptr) and flags out-of-range senders.
__global__ void __launch_bounds__(32 * kSortWarps) radix_hist_kernel(EdgeKeys k, const int32_t* __restrict__ in,
                                                                      int64_t T, int64_t n_tiles, int shift,
                                                                      int32_t* __restrict__ hist,
                                                                      unsigned* __restrict__ err) {
    __shared__ int32_t cnt[kSortWarps][kBins];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    int64_t lo, hi;
    k.range(lo, hi);
    const int64_t nw = int64_t(gridDim.x) * kSortWarps;
    for (int64_t tile = int64_t(blockIdx.x) * kSortWarps + wib; tile < n_tiles; tile += nw) {
        for (int d = lane; d < kBins; d += 32) cnt[wib][d] = 0;
        __syncwarp();
        const int64_t b = tile * T, e = (b + T < k.E) ? b + T : k.E;
        bool bad = false;
        for (int64_t r = b; r < e; r += 32) {   // warp-uniform trip count
            const int64_t i = r + lane;
            int32_t d = -1;
            if (i < e) {
                const int32_t v = in ? in[i] : int32_t(i);
                if (!in) {
                    const int32_t s = __ldg(k.sender + v);
                    bad |= (s < 0 || s >= k.N);
                }
                d = (k.key(v, lo, hi) >> shift) & (kBins - 1);
            }
            // one shared-memory add per distinct digit of the round (a heavy sender makes
            // whole rounds share one digit)
            const unsigned peers = __match_any_sync(0xffffffffu, d);
            if (d >= 0 && (peers & lanemask_lt()) == 0) cnt[wib][d] += __popc(peers);
            __syncwarp();
        }
        if (bad) atomicOr(err, kErrSender);
        __syncwarp();
        for (int d = lane; d < kBins; d += 32) hist[int64_t(d) * n_tiles + tile] = cnt[wib][d];
        __syncwarp();
    }
}

// (c) stable scatter: out[off[d][tile] + (#earlier entries of the tile with digit d)] = v
__global__ void __launch_bounds__(32 * kSortWarps) radix_scatter_kernel(EdgeKeys k, const int32_t* __restrict__ in,
                                                                         int64_t T, int64_t n_tiles, int shift,
                                                                         const int32_t* __restrict__ off,
                                                                         int32_t* __restrict__ out) {
    constexpr int kAhead = 4;   // rounds of 32 entries whose loads are issued together
    __shared__ int32_t cur[kSortWarps][kBins];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const unsigned lt = lanemask_lt();
    int64_t lo, hi;
    k.range(lo, hi);
    const int64_t nw = int64_t(gridDim.x) * kSortWarps;
    for (int64_t tile = int64_t(blockIdx.x) * kSortWarps + wib; tile < n_tiles; tile += nw) {
        for (int d = lane; d < kBins; d += 32) cur[wib][d] = off[int64_t(d) * n_tiles + tile];
        __syncwarp();
        const int64_t b = tile * T, e = (b + T < k.E) ? b + T : k.E;
        for (int64_t r0 = b; r0 < e; r0 += 32 * kAhead) {
            int32_t v[kAhead], dg[kAhead];
#pragma unroll
            for (int j = 0; j < kAhead; ++j) {
                const int64_t i = r0 + 32 * j + lane;
                v[j] = i < e ? (in ? in[i] : int32_t(i)) : -1;
            }
#pragma unroll
            for (int j = 0; j < kAhead; ++j)
                dg[j] = v[j] >= 0 ? (k.key(v[j], lo, hi) >> shift) & (kBins - 1) : -1;
#pragma unroll
            for (int j = 0; j < kAhead; ++j) {
                const unsigned peers = __match_any_sync(0xffffffffu, dg[j]);
                int32_t base = 0;
                if (dg[j] >= 0) base = cur[wib][dg[j]];
                __syncwarp();
                if (dg[j] >= 0) {
                    out[base + __popc(peers & lt)] = v[j];
                    if ((peers & lt) == 0) cur[wib][dg[j]] = base + __popc(peers);   // the group's first lane
                }
                __syncwarp();
            }
        }
    }
}

// block-wide exclusive scan of one value per thread (blockDim.x == kScanBlock); returns the
// thread's exclusive prefix and sets *total
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* total) {
    __shared__ int64_t warp_sums[kScanBlock / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int64_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int64_t s = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t n = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += n;
        }
        warp_sums[lane] = s;   // inclusive over warps
    }
    __syncthreads();
    const int64_t before = wid > 0 ? warp_sums[wid - 1] : 0;
    *total = warp_sums[kScanBlock / 32 - 1];
    __syncthreads();   // warp_sums is reused by the next call
    return before + incl - v;
}

// (b) exclusive scan of a[0..n) in place, three launches: block sums, a scan of the block
// sums, then each block's scan plus its offset.
__global__ void __launch_bounds__(kScanBlock) scan_sums_kernel(const int32_t* __restrict__ a, int64_t n,
                                                               int32_t* __restrict__ sums) {
    const int64_t b = int64_t(blockIdx.x) * kScanChunk;
    int64_t s = 0;
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
        const int64_t i = b + int64_t(j) * kScanBlock + threadIdx.x;
        if (i < n) s += a[i];
    }
    int64_t total;
    block_exclusive_scan(s, &total);
    if (threadIdx.x == 0) sums[blockIdx.x] = int32_t(total);
}

__global__ void __launch_bounds__(kScanBlock) scan_top_kernel(int32_t* __restrict__ sums, int64_t n) {
    int64_t carry = 0;
    for (int64_t b = 0; b < n; b += kScanBlock) {
        const int64_t i = b + threadIdx.x;
        const int64_t v = i < n ? sums[i] : 0;
        int64_t total;
        const int64_t ex = block_exclusive_scan(v, &total);
        if (i < n) sums[i] = int32_t(carry + ex);
        carry += total;
    }
}

__global__ void __launch_bounds__(kScanBlock) scan_apply_kernel(int32_t* __restrict__ a, int64_t n,
                                                                const int32_t* __restrict__ sums) {
    const int64_t b = int64_t(blockIdx.x) * kScanChunk + int64_t(threadIdx.x) * kScanItems;
    int32_t v[kScanItems];
    int64_t s = 0;
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
        v[j] = b + j < n ? a[b + j] : 0;
        s += v[j];
    }
    int64_t total;
    int64_t run = block_exclusive_scan(s, &total) + sums[blockIdx.x];
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
        if (b + j < n) a[b + j] = int32_t(run);
        run += v[j];
    }
}

// csc_ptr[a] = first position of the sorted edge ids whose key is >= a, a in [0, N]; also
// checks every receiver segment of rowptr
__global__ void ptr_kernel(EdgeKeys k, const int32_t* __restrict__ sorted, int32_t* __restrict__ ptr,
                           unsigned* __restrict__ err) {
    int64_t lo, hi;
    k.range(lo, hi);
    for (int64_t a = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; a <= k.N; a += int64_t(gridDim.x) * blockDim.x) {
        if (a < k.N) {
            const int64_t e0 = k.rowptr[a], e1 = k.rowptr[a + 1];
            if (e0 < 0 || e1 < e0 || e1 > k.E) atomicOr(err, kErrRowptr);
        }
        int64_t l = 0, h = k.E;   // invariant: key(sorted[l-1]) < a <= key(sorted[h])
        while (l < h) {
            const int64_t mid = (l + h) >> 1;
            if (k.key(sorted[mid], lo, hi) < a) l = mid + 1; else h = mid;
        }
        ptr[a] = int32_t(l);
    }
}

// csc_recv[k] = receiver of csc_edge[k]; entries past csc_ptr[N] (edges left out) become -1
__global__ void recv_kernel(int64_t N, int64_t E, const int32_t* __restrict__ rowptr,
                            const int32_t* __restrict__ ptr, int32_t* __restrict__ edge,
                            int32_t* __restrict__ recv) {
    const int64_t n_valid = ptr[N];
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < E; k += int64_t(gridDim.x) * blockDim.x) {
        if (k >= n_valid) {
            edge[k] = -1;
            recv[k] = -1;
            continue;
        }
        const int32_t e = edge[k];
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

// Tile length (entries per warp) of the sort; tiles_cap > 0 bounds the tile count so that
// the counts fit a fixed scratch (the tile then grows with the edge count).
int64_t sort_tile(int64_t E, int64_t tiles_cap) {
    int64_t T = 1024;
    if (tiles_cap > 0)
        while ((E + T - 1) / T > tiles_cap) T *= 2;
    return T;
}

size_t scan_sums_count(int64_t n) { return size_t((n + kScanChunk - 1) / kScanChunk); }

cudaError_t exclusive_scan_i32(int32_t* a, int64_t n, int32_t* sums, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t nb = int64_t(scan_sums_count(n));
    scan_sums_kernel<<<int(nb), kScanBlock, 0, s>>>(a, n, sums);
    scan_top_kernel<<<1, kScanBlock, 0, s>>>(sums, nb);
    scan_apply_kernel<<<int(nb), kScanBlock, 0, s>>>(a, n, sums);
    return cudaGetLastError();
}

// int32 entries of the sort's scratch for tile length T: the digit counts, then the scan's block sums
size_t graph_scratch_ints(int64_t E, int64_t T) {
    const int64_t n_hist = int64_t(kBins) * ((E + T - 1) / T);
    return size_t(n_hist) + scan_sums_count(n_hist) + 1;
}

int64_t graph_static_tiles_cap(size_t scratch_ints) {
    // largest tile count whose counts and block sums fit
    int64_t t = int64_t(scratch_ints) / kBins;
    while (t > 0 && graph_scratch_ints(t * 1024, 1024) > scratch_ints) --t;
    return t;
}

size_t graph_workspace_bytes(int64_t N, int64_t E) {
    (void)N;
    return (graph_scratch_ints(E, sort_tile(E, 0)) * 4 + 255) / 256 * 256;
}

cudaError_t graph_prepare(int64_t N, int64_t E, const int32_t* rowptr, const int32_t* sender, int32_t* csc_ptr,
                          int32_t* csc_edge, int32_t* csc_recv, void* ws, int64_t tiles_cap, unsigned* err,
                          cudaStream_t s) {
    const EdgeKeys k{N, E, sender, rowptr};
    if (E > 0) {
        int dev = 0, sms = 0;
        cudaError_t st = cudaGetDevice(&dev);
        if (st == cudaSuccess) st = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (st != cudaSuccess) return st;
        const int64_t T = sort_tile(E, tiles_cap);
        const int64_t n_tiles = (E + T - 1) / T;
        const int64_t n_hist = int64_t(kBins) * n_tiles;
        int32_t* hist = static_cast<int32_t*>(ws);
        int32_t* sums = hist + n_hist;
        const int64_t n_sums = int64_t(scan_sums_count(n_hist));
        int bits = 0;
        while ((int64_t(1) << bits) <= N) ++bits;   // keys lie in [0, N]
        const int passes = bits > kRadixBits ? (bits + kRadixBits - 1) / kRadixBits : 1;
        const int sort_grid = grid1d((n_tiles + kSortWarps - 1) / kSortWarps, 1, sms * 16);
        const int32_t* in = nullptr;
        for (int p = 0; p < passes; ++p) {
            int32_t* out = ((passes - 1 - p) % 2 == 0) ? csc_edge : csc_recv;
            const int shift = p * kRadixBits;
            radix_hist_kernel<<<sort_grid, 32 * kSortWarps, 0, s>>>(k, in, T, n_tiles, shift, hist, err);
            scan_sums_kernel<<<int(n_sums), kScanBlock, 0, s>>>(hist, n_hist, sums);
            scan_top_kernel<<<1, kScanBlock, 0, s>>>(sums, n_sums);
            scan_apply_kernel<<<int(n_sums), kScanBlock, 0, s>>>(hist, n_hist, sums);
            radix_scatter_kernel<<<sort_grid, 32 * kSortWarps, 0, s>>>(k, in, T, n_tiles, shift, hist, out);
            in = out;
        }
    }
    ptr_kernel<<<grid1d(N + 1, 256, 4096), 256, 0, s>>>(k, csc_edge, csc_ptr, err);
    if (E > 0) recv_kernel<<<grid1d(E, 256, 4096), 256, 0, s>>>(N, E, rowptr, csc_ptr, csc_edge, csc_recv);
    return cudaGetLastError();
}

}  // namespace e3gb
