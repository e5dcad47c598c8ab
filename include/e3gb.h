/*
 * e3gb: channelwise Clebsch-Gordan tensor product and message-passing convolution on
 * NVIDIA GB300 (sm_103a). C ABI.
 *
 * The operations are those of "e3j: An efficient and open-source backend for Euclidean
 * equivariant operations on GPU and TPU" (arXiv HTML version), App. E.1:
 *   - Eq. (10)-(11): tensor product of l.h.s. features x with r.h.s. features y (real
 *     spherical harmonics, no channel axis), weighted per path and channel;
 *   - Eq. (12)-(13): message-passing convolution, the same product per edge with the sender's
 *     x, summed at the receiver over a receiver-sorted CSR edge list;
 *   - Eq. (15)-(16): their reverse-mode (VJP) rules.
 * Spherical harmonics: App. A.3 Eq. (4) and App. G.1. CG coefficients: App. G.2.
 *
 * Layouts (all row-major, channel axis innermost: "trailing channels", App. E.2.1):
 *   x  [rows or nodes][d1][Nq]   d1 = sum over x irreps blocks of (2l+1), blocks in the order
 *                                given to e3gb_table_create, m = -l..l inside a block
 *   y  [rows or edges][d2]       d2 = (sh_lmax+1)^2, Y_0, Y_1, ... concatenated
 *   w  [rows or edges][P][Nq]    P paths in table order
 *   z, m, dz, dm [rows or nodes][D][Nq]
 * Nq (the uniform multiplicity) must be 4, 8, 16, 32, 64 or 128.
 *
 * Memory and streams: every device buffer belongs to the caller; no call allocates device
 * memory. Work is enqueued on the caller's stream (a cudaStream_t passed as void*, NULL =
 * legacy default stream) and the call returns without synchronising. Channel-vector arrays
 * (x, w, dz, dm, and every fp32 output) must be 16-byte aligned, or 8-byte aligned when they
 * are bf16 inputs; y and dy need element alignment; buffers must not alias each other.
 * Every buffer must hold the elements its layout above implies for the given counts: the
 * library receives bare pointers and cannot check sizes (the Python binding checks tensor
 * shapes before each call). Outputs are always fp32 and are overwritten, never accumulated into.
 *
 * Errors: each call checks its arguments on the host and returns a status; the message of
 * the last failure on the calling thread is e3gb_last_error(). Index errors found on the
 * device (a sender or receiver outside [0, n_nodes), a decreasing or out-of-range CSR
 * pointer) never fault: the offending edge or segment is skipped and a device error word
 * is set; e3gb_check_device_status() reads and clears it.
 *
 * Determinism: for identical inputs and launch configuration results are bitwise identical
 * from run to run (fixed summation order, no floating-point atomics).
 */
#ifndef E3GB_H
#define E3GB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    E3GB_OK = 0,
    E3GB_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, bad dtype */
    E3GB_ERR_UNSUPPORTED = 2,   /* irreps configuration or channel count not built in */
    E3GB_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
    E3GB_ERR_BAD_GRAPH = 4,     /* CSR arrays inconsistent on the host side */
    E3GB_ERR_DEVICE_INDEX = 5   /* the device saw an out-of-range index (see above) */
} e3gb_status;

typedef enum {
    E3GB_F32 = 0,   /* fp32 inputs, fp32 arithmetic, fp32 outputs */
    E3GB_BF16 = 1   /* bf16 storage of the inputs x, y, w and dz/dm (half their bytes); fp32
                       arithmetic and fp32 outputs. (bf16 outputs would not meet a 2e-2 RMS
                       bound: rounding the exact result alone reaches 3.7e-2 RMS for dw.) */
} e3gb_dtype;

/* Irreps of x with a uniform multiplicity: n blocks, block i of degree l[i] in 0..3 and
 * parity parity[i] = +1 (even) or -1 (odd), each with mul channels. */
typedef struct {
    int32_t n;
    const int32_t *l;
    const int32_t *parity;
    int32_t mul;
} e3gb_irreps;

/* Opaque path table: the paths (x block, l2, l3) with their real CG blocks, baked into the
 * kernels at compile time for each supported configuration. Host-owned. */
typedef struct e3gb_table e3gb_table;

/* table_create flags */
#define E3GB_PATHS_SUMMED 0    /* one output block per distinct (l3, p3); default */
#define E3GB_PATHS_SEPARATE 1  /* one output block per path */

/* Build the path table for x irreps, SH degrees 0..sh_lmax and output degrees <= out_lmax
 * (App. A.3 Eq. 6: every l3 in |l1-l2|..l1+l2; App. B.1: output parity p1 (-1)^l2).
 * Paths are ordered by (x block, l2, l3). In summed mode the output blocks are the distinct
 * (l3, p3) ordered by l3 with the natural parity (-1)^l3 first.
 * Returns E3GB_ERR_UNSUPPORTED when the configuration has no compiled kernels
 * (e3gb_config_count / e3gb_config_describe list the built ones). *out is set on success
 * and must be released with e3gb_table_destroy. */
e3gb_status e3gb_table_create(const e3gb_irreps *x, int32_t sh_lmax, int32_t out_lmax,
                              int32_t flags, e3gb_table **out);
e3gb_status e3gb_table_destroy(e3gb_table *t);

/* Sizes of a table; any output pointer may be NULL. nnz = number of nonzero CG records. */
e3gb_status e3gb_table_info(const e3gb_table *t, int32_t *d1, int32_t *d2, int32_t *n_paths,
                            int32_t *D, int32_t *nnz, int32_t *mul);

/* Path descriptors, n_paths x 8 int32: x block, l1, p1, l2, l3, p3, output block, output
 * offset. NULL-safe sizes: paths must hold 8*n_paths ints. */
e3gb_status e3gb_table_paths(const e3gb_table *t, int32_t *paths);

/* CG records, nnz x 5 doubles: path, m1, m2, m3 (0-based, i.e. m + l), value (App. G.2
 * normalisation sum_{m1,m2} C^2 = 1 per m3; first row-major entry of each block > 0). */
e3gb_status e3gb_table_coefficients(const e3gb_table *t, double *records);

/* Built configurations: count, and for index i the x irreps (up to 8 blocks), sh_lmax,
 * out_lmax and flags. */
int32_t e3gb_config_count(void);
e3gb_status e3gb_config_describe(int32_t i, int32_t *n_blocks, int32_t *l, int32_t *parity,
                                 int32_t *sh_lmax, int32_t *out_lmax, int32_t *flags);

/* Real spherical harmonics (App. A.3 Eq. 4, App. G.1): y[e] = (Y_l(u_e))_{l=0..lmax},
 * u_e = vec[e]/|vec[e]| (u = 0 when |vec| < 1e-12, giving Y_0 = 1 and Y_l>0 = 0),
 * component normalisation sum_m Y_lm^2 = 2l+1, l = 1 ordered sqrt(3)(y, z, x).
 * vec: device fp32 [n, 3]; y: device [n, (lmax+1)^2] of dtype (bf16: rounded to nearest
 * even from fp32, to feed the bf16 variant). lmax in 0..3. */
e3gb_status e3gb_sh_forward(int32_t lmax, int64_t n, const float *vec, void *y,
                            e3gb_dtype dtype, void *stream);

/* Its VJP, the gradient through the harmonics that forces need: dvec[e] = sum_{l,m}
 * dy[e, l^2+l+m] dY_lm(vec[e]/|vec[e]|)/dvec[e] (zero where |vec| < 1e-12). vec: device fp32
 * [n, 3]; dy: device [n, (lmax+1)^2] of dtype; dvec: device fp32 [n, 3]. */
e3gb_status e3gb_sh_backward(int32_t lmax, int64_t n, const float *vec, const void *dy, float *dvec,
                             e3gb_dtype dtype, void *stream);

/* Tensor product on rows (Eq. 10-11): z[r] = sum_p w[r,p] * C_p(x[r], y[r]) into the
 * output block of path p. x [rows,d1,Nq], y [rows,d2], w [rows,P,Nq], z [rows,D,Nq]. */
e3gb_status e3gb_tp_forward(const e3gb_table *t, int64_t rows, const void *x, const void *y,
                            const void *w, void *z, e3gb_dtype dtype, void *stream);

/* Its VJP (Eq. 15 with the weights as a third operand): from dz [rows,D,Nq] computes
 * dx [rows,d1,Nq], dy [rows,d2] (summed over channels) and dw [rows,P,Nq] in one pass that
 * reads dz once. */
e3gb_status e3gb_tp_backward(const e3gb_table *t, int64_t rows, const void *x, const void *y,
                             const void *w, const void *dz, void *dx, void *dy, void *dw,
                             e3gb_dtype dtype, void *stream);

/* Workspace (bytes) that e3gb_graph_prepare needs for a graph of n_nodes nodes and n_edges
 * edges (about n_edges bytes: the sort's per-tile digit counts). */
size_t e3gb_graph_prepare_workspace_bytes(int64_t n_nodes, int64_t n_edges);

/* Sender-major index of a receiver-sorted CSR graph (rowptr [n_nodes+1], sender [n_edges],
 * receiver b owns edges [rowptr[b], rowptr[b+1])). Writes csc_ptr [n_nodes+1], and for the
 * k-th edge in sender order csc_edge[k] (its CSR edge id) and csc_recv[k] (its receiver);
 * edges of one sender keep increasing edge id (stable). Used by the backward convolution to
 * sum dx per sender without atomics (the transposed graph of Eq. 16). All arrays are
 * device arrays. The work is linear in n_edges + n_nodes whatever the degrees (a padding
 * node that sends most edges costs what any other edges cost): a stable radix sort of the
 * edge ids by sender, ceil(bits(n_nodes)/8) passes. Edges outside [rowptr[0], rowptr[n_nodes])
 * and edges whose sender is outside [0, n_nodes) are left out of the index (the latter also
 * flagged in the device error word); the entries past csc_ptr[n_nodes] are -1. A rowptr
 * segment with a negative start, a decreasing pointer or an end past n_edges is flagged; the
 * index is then unspecified but every entry stays in range. workspace: device memory of at
 * least e3gb_graph_prepare_workspace_bytes(n_nodes, n_edges) bytes, 16-byte aligned; its
 * contents on entry do not matter. */
e3gb_status e3gb_graph_prepare(int64_t n_nodes, int64_t n_edges, const int32_t *rowptr,
                               const int32_t *sender, int32_t *csc_ptr, int32_t *csc_edge,
                               int32_t *csc_recv, void *workspace, size_t ws_bytes,
                               void *stream);

/* Size of the library's own scratch array behind e3gb_graph_prepare_static. */
#define E3GB_STATIC_PREPARE_SCRATCH_BYTES (4u << 20)

/* e3gb_graph_prepare for callers that cannot allocate device memory. The paper has no
 * counterpart: this entry point exists for programs that must not call cudaMalloc after
 * start-up, for example a host that has handed all free device memory to its own pool, a
 * plugin inside a host that owns every allocation and offers it no allocator, or a
 * latency-critical loop that cannot afford cudaMalloc's implicit device-wide
 * synchronisation. It computes exactly what e3gb_graph_prepare computes, but keeps the
 * sort's digit counts in a 4 MiB array inside the library (E3GB_STATIC_PREPARE_SCRATCH_BYTES,
 * one per device that loads the library, held until the process exits) instead of a caller
 * workspace; it allocates nothing. The array holds the counts of at most ~4,000 tiles, so
 * above ~4 M edges each tile covers more edges (fewer warps share the sort, same result).
 * Sizes: n_nodes, n_edges < 2^31-1, else E3GB_ERR_INVALID_ARG. The first call on a device
 * looks up the array's device address on that device; make that first call before any
 * stream capture. All calls share the one array (every count is written before it is read,
 * so nothing needs clearing): calls that overlap on the GPU (on different streams, or from
 * different threads) race on it and must be serialised by the caller. */
e3gb_status e3gb_graph_prepare_static(int64_t n_nodes, int64_t n_edges, const int32_t *rowptr,
                                      const int32_t *sender, int32_t *csc_ptr, int32_t *csc_edge,
                                      int32_t *csc_recv, void *stream);

/* Message-passing convolution (Eq. 12-13): for every receiver b,
 *   m[b] = scale * sum_{e in [rowptr[b], rowptr[b+1])} TP(x[sender[e]], y[e], w[e]),
 * accumulated in a fixed order in registers, written once (receivers without edges get 0).
 * x [n_nodes,d1,Nq], y [n_edges,d2], w [n_edges,P,Nq], m [n_nodes,D,Nq].
 *
 * Padding edges (e3j, Sec. 4 "Message passing convolution" and App. E: static-shape graphs
 * route their unused edge slots to one padding node, and the kernels skip them): pad_node is
 * that node's index, or -1 for none. Every edge whose receiver or sender is pad_node is a
 * padding edge and is not read at all (its x, y, w may hold anything, NaN included); the
 * padding receiver's whole segment is passed over, so its valency costs nothing, and
 * m[pad_node] = 0. pad_node outside [-1, n_nodes) is E3GB_ERR_INVALID_ARG. */
e3gb_status e3gb_conv_forward(const e3gb_table *t, int64_t n_nodes, int64_t n_edges,
                              const int32_t *rowptr, const int32_t *sender, const void *x,
                              const void *y, const void *w, float scale, int64_t pad_node,
                              void *m, e3gb_dtype dtype, void *stream);

/* e3gb_conv_forward for graphs with heavy receivers. A receiver-stationary forward gives each
 * receiver to one warp, so one receiver with very many edges (a hub that is not the padding
 * node) makes the whole launch wait for that warp (e3j, Sec. 4 "Message passing convolution":
 * the receiver-degree imbalance that deterministic receiver-stationary kernels face). Here a
 * receiver's CSR segment is cut into pieces of chunk positions: the first piece is summed by the
 * usual kernels, every further piece by its own warp into a partial row set in the workspace,
 * and the partials are added to m[b] in piece order. Deterministic (fixed order, no atomics);
 * receivers with at most chunk positions get exactly e3gb_conv_forward's result, heavier ones
 * a different (fixed) summation order. Arguments as e3gb_conv_forward, plus chunk >= 1 and a
 * device workspace of at least e3gb_conv_forward_split_workspace_bytes bytes (16-byte
 * aligned; contents on entry do not matter). E3GB_ERR_UNSUPPORTED for configurations with more
 * than 32 output rows. Choosing chunk: each further piece is one warp's serial walk, so the
 * pieces finish in about chunk x (one warp's time per edge) when they fit in one wave of
 * warps; a chunk a few times the typical degree (256 for degree ~40) leaves ordinary
 * receivers whole and gives a hub of 200,000 edges ~780 warps. */
size_t e3gb_conv_forward_split_workspace_bytes(const e3gb_table *t, int64_t n_nodes, int64_t n_edges,
                                               int32_t chunk);
e3gb_status e3gb_conv_forward_split(const e3gb_table *t, int64_t n_nodes, int64_t n_edges,
                                    const int32_t *rowptr, const int32_t *sender, const void *x,
                                    const void *y, const void *w, float scale, int64_t pad_node,
                                    int32_t chunk, void *m, void *workspace, size_t ws_bytes,
                                    e3gb_dtype dtype, void *stream);

/* Its VJP (Eq. 16) from dm [n_nodes,D,Nq]:
 *   dw[e,p] = scale * sum_m3 dm[b][blk p, m3] * (C_p(x[a], y[e]))[m3],
 *   dy[e]   = scale * sum over paths and channels of the x, w, dm couplings,
 *   dx[a]   = scale * sum over the edges of sender a of the y, w, dm couplings,
 * walking the graph in sender order (csc_* from e3gb_graph_prepare) so that dx[a] is summed
 * in registers in a fixed order: deterministic, no atomics, no workspace.
 * dx [n_nodes,d1,Nq], dy [n_edges,d2], dw [n_edges,P,Nq].
 * pad_node as in e3gb_conv_forward: padding edges are not read, their dw and dy rows are
 * written as zeros (by a second, grid-wide launch on the same stream that scans csc_recv),
 * and dx[pad_node] = 0. */
e3gb_status e3gb_conv_backward(const e3gb_table *t, int64_t n_nodes, int64_t n_edges,
                               const int32_t *csc_ptr, const int32_t *csc_edge,
                               const int32_t *csc_recv, const void *x, const void *y,
                               const void *w, const void *dm, float scale, int64_t pad_node,
                               void *dx, void *dy, void *dw, e3gb_dtype dtype, void *stream);

/* Double backward of the convolution (e3j App. E.1 Eq. (17)-(18)). Given the primals x, y,
 * w, dm of e3gb_conv_backward and variations delta_dx [n_nodes,d1,Nq], delta_dy
 * [n_edges,d2], delta_dw [n_edges,P,Nq] of the cotangents it returned, computes the
 * gradient of <dx, delta_dx> + <dy, delta_dy> + <dw, delta_dw> with respect to the primals:
 *   delta_dm = conv(delta_dx, y, w) + conv(x, delta_dy, w) + conv(x, y, delta_dw)   (17)
 *   delta_x  = dx of conv_bwd(x, delta_dy, w, dm) + dx of conv_bwd(x, y, delta_dw, dm)
 *   delta_y  = dy of conv_bwd(delta_dx, y, w, dm) + dy of conv_bwd(x, y, delta_dw, dm)
 *   delta_w  = dw of conv_bwd(delta_dx, y, w, dm) + dw of conv_bwd(x, delta_dy, w, dm)   (18)
 * in two fused launches (a receiver-ordered pass for delta_dm over rowptr/sender, a
 * sender-ordered pass for the rest over csc_* from e3gb_graph_prepare) that compute none of
 * the cotangents Eq. (18) discards. delta_x [n_nodes,d1,Nq], delta_y [n_edges,d2], delta_w
 * [n_edges,P,Nq], delta_dm [n_nodes,D,Nq], fp32, fully overwritten; deterministic (fixed
 * summation order, no atomics). scale and pad_node as in e3gb_conv_forward (padding edges
 * get zero delta_y, delta_w rows). Inputs share one dtype. */
e3gb_status e3gb_conv_double_backward(const e3gb_table *t, int64_t n_nodes, int64_t n_edges,
                                      const int32_t *rowptr, const int32_t *sender,
                                      const int32_t *csc_ptr, const int32_t *csc_edge,
                                      const int32_t *csc_recv, const void *x, const void *y,
                                      const void *w, const void *dm, const void *delta_dx,
                                      const void *delta_dy, const void *delta_dw, float scale,
                                      int64_t pad_node, void *delta_x, void *delta_y,
                                      void *delta_w, void *delta_dm, e3gb_dtype dtype,
                                      void *stream);

/* Radial edge scalars (e3j, App. E.1 notation for the edge scalars s: "usually" an MLP on a
 * radial embedding of the interatomic distance, projected to the paths and channels of each
 * edge; App. A.3 "Linear mixing": that scalar mixing fused into message passing). The pages
 * fix neither the embedding nor the network; this library reads them as
 *   b_n(d) = sqrt(2/r_cut) sin(n pi d / r_cut) / d * u(d / r_cut),  n = 1..n_basis
 *   u(x)   = 1 - 28 x^6 + 48 x^7 - 21 x^8 (x < 1), 0 beyond    (smooth cutoff, p = 6)
 *   h[e,k] = silu(sum_n b_n(|vec[e]|) W1[n,k]),  w[e,p,q] = sum_k h[e,k] W2[k,p,q]
 * (no biases; d -> 0 takes the limit sqrt(2/r_cut) n pi / r_cut). The hidden layer is computed
 * here; the output layer, the large one, is evaluated inside e3gb_conv_*_radial so that w
 * never reaches device memory.
 *
 * e3gb_radial_hidden: h [n_edges, hidden] from vec [n_edges, 3] and W1 [n_basis, hidden]
 * (float64 arithmetic, fp32 result). n_basis and hidden in [1, 16], r_cut > 0, else
 * E3GB_ERR_INVALID_ARG. All pointers are device pointers. */
e3gb_status e3gb_radial_hidden(int64_t n_edges, const float *vec, const float *W1, int32_t n_basis,
                               int32_t hidden, float r_cut, float *h, void *stream);

/* e3gb_radial_backward: dvec[e] = d <dh[e], h[e]> / d vec[e], the force contribution of the
 * radial weights, from the cotangent dh [n_edges, hidden] (e3gb_conv_backward_radial's dh).
 * Radial: (sum_k dh[e,k] silu'(a_k) sum_n b_n'(d) W1[n,k]) vec[e] / |vec[e]|; zero for
 * |vec[e]| < 1e-12. accumulate != 0 adds to dvec (for example to e3gb_sh_backward's output)
 * instead of overwriting it. */
e3gb_status e3gb_radial_backward(int64_t n_edges, const float *vec, const float *W1, int32_t n_basis,
                                 int32_t hidden, float r_cut, const float *dh, float *dvec,
                                 int32_t accumulate, void *stream);

/* e3gb_conv_forward with the edge weights produced in the kernel from the hidden activations
 * h [n_edges, hidden] (16-byte aligned rows) and the output layer W2 [hidden, P, Nq] (device,
 * 16-byte aligned): w[e,p,q] = sum_k h[e,k] W2[k,p,q], never written out. Otherwise as
 * e3gb_conv_forward (padding, scale, fixed order, m fully overwritten). Built for fp32
 * (x, y, m) and hidden = 8: other values give E3GB_ERR_UNSUPPORTED, and so does a W2 larger
 * than one block's shared memory (hidden * P * Nq * 4 > 227 KiB). */
e3gb_status e3gb_conv_forward_radial(const e3gb_table *t, int64_t n_nodes, int64_t n_edges,
                                     const int32_t *rowptr, const int32_t *sender, const void *x,
                                     const void *y, const float *h, const float *W2, int32_t hidden,
                                     float scale, int64_t pad_node, void *m, e3gb_dtype dtype,
                                     void *stream);

/* Its VJP: dx and dy as e3gb_conv_backward, and instead of dw the cotangent of the hidden
 * activations dh[e,k] = sum_{p,q} W2[k,p,q] dw[e,p,q] [n_edges, hidden] (dw itself never
 * reaches memory). Padding edges get zero dy and dh rows. Deterministic, no atomics. Same
 * limits as e3gb_conv_forward_radial. */
e3gb_status e3gb_conv_backward_radial(const e3gb_table *t, int64_t n_nodes, int64_t n_edges,
                                      const int32_t *csc_ptr, const int32_t *csc_edge,
                                      const int32_t *csc_recv, const void *x, const void *y,
                                      const float *h, const float *W2, int32_t hidden,
                                      const void *dm, float scale, int64_t pad_node, void *dx,
                                      void *dy, float *dh, e3gb_dtype dtype, void *stream);

/* Tensor product with arbitrary sparse coefficients on rows (e3j App. E.1 Eq. (10)-(11),
 * Alg. 1: C as a COO list of records), the general bilinear primitive of which the CG
 * tensor product is one choice of records:
 *   z[r,i0,q] = sum over records k with i0_k = i0 of coef[k] * w[r,path_k,q] * x[r,i1_k,q] * y[r,i2_k]
 * rec: device int32 [n_rec][4] = (i0, i1, i2, path), 16-byte aligned, any order, repeats
 * add; coef: device float [n_rec]. x [rows,d1,mul], y [rows,d2], w [rows,n_paths,mul]
 * (dtype), z [rows,D,mul] fp32, fully overwritten (rows of z with no record are 0).
 * mul: a power of two <= 128. E3GB_ERR_UNSUPPORTED when one block's accumulators do not fit
 * in shared memory (forward: 1024 * D * (mul >= 64 ? 4 : 1) bytes). A record with an index
 * outside D, d1, d2, n_paths is skipped and sets bit 8 of the device error word. Records
 * and coefficients are caller-owned device memory; nothing is allocated. */
e3gb_status e3gb_coo_tp_forward(int64_t rows, int32_t d1, int32_t d2, int32_t D, int32_t n_paths,
                                int32_t mul, int32_t n_rec, const int32_t *rec, const float *coef,
                                const void *x, const void *y, const void *w, void *z,
                                e3gb_dtype dtype, void *stream);

/* Its adjoint from dz [rows,D,mul]: dx [rows,d1,mul], dy [rows,d2], dw [rows,n_paths,mul],
 * fp32, fully overwritten. Deterministic (fixed record order per row, fixed reduction of
 * dy over channels). */
e3gb_status e3gb_coo_tp_backward(int64_t rows, int32_t d1, int32_t d2, int32_t D, int32_t n_paths,
                                 int32_t mul, int32_t n_rec, const int32_t *rec, const float *coef,
                                 const void *x, const void *y, const void *w, const void *dz,
                                 void *dx, void *dy, void *dw, e3gb_dtype dtype, void *stream);

/* Synchronise stream, read and clear the device error word of the current device.
 * E3GB_OK when clean, E3GB_ERR_DEVICE_INDEX when a kernel skipped bad indices (*flags, if
 * not NULL, receives the bits: 1 bad sender, 2 bad CSR pointer, 4 bad receiver / edge id,
 * 8 bad COO record index). */
e3gb_status e3gb_check_device_status(void *stream, int32_t *flags);

/* Message of the last failed call on this thread ("" if none). */
const char *e3gb_last_error(void);

/* Library version string. */
const char *e3gb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* E3GB_H */
