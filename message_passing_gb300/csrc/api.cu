// C ABI of the library (include/e3gb.h): argument checks, table objects, dispatch to the
// per-configuration kernels, and the device error word.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <tuple>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/e3gb.h"
#include "kernels.cuh"
#include "radial.cuh"

namespace e3gb {
#define E3GB_CONFIG(ID, XC, L2, L3, PP) const ConfigOps* ops_##ID();
#include "configs.def"
#undef E3GB_CONFIG

static const ConfigOps* (*const kRegistry[])() = {
#define E3GB_CONFIG(ID, XC, L2, L3, PP) ops_##ID,
#include "configs.def"
#undef E3GB_CONFIG
};
constexpr int kNumConfigs = int(sizeof(kRegistry) / sizeof(kRegistry[0]));

cudaError_t sh_forward(int lmax, int64_t n, const float* vec, void* y, int bf16, cudaStream_t s);
cudaError_t sh_backward(int lmax, int64_t n, const float* vec, const void* dy, float* dvec, int bf16, cudaStream_t s);
size_t graph_workspace_bytes(int64_t N, int64_t E);
int64_t graph_static_tiles_cap(size_t scratch_ints);
cudaError_t graph_prepare(int64_t N, int64_t E, const int32_t* rowptr, const int32_t* sender, int32_t* csc_ptr,
                          int32_t* csc_edge, int32_t* csc_recv, void* ws, int64_t tiles_cap, unsigned* err,
                          cudaStream_t s);
size_t coo_smem_bytes(bool backward, int d1, int d2, int D, int P, int Nq);
template <class T>
cudaError_t coo_tp(bool backward, int64_t R, int d1, int d2, int D, int P, int Nq, int nrec, const int32_t* rec,
                   const float* coef, const void* x, const void* y, const void* w, const void* dz, void* z_or_dx,
                   void* dy, void* dw, unsigned* err, cudaStream_t s);
cudaError_t zero_padding_edges(int64_t N, int64_t E, const int32_t* csc_ptr, const int32_t* csc_edge,
                               const int32_t* csc_recv, int64_t pad, float* dw, int64_t dw_row, float* dy,
                               int64_t dy_row, cudaStream_t s);

// ------------------------------------------------------------------------------------------
// launch sizing: grid = min(blocks needed, resident blocks per SM x SMs), cached per kernel
// ------------------------------------------------------------------------------------------
int grid_for(const void* kernel, int block, int64_t per_block, int64_t units, int smem) {
    if (units <= 0) return 0;
    static std::mutex mu;
    static std::map<std::tuple<const void*, int, int>, int> resident;  // blocks per device, by kernel and smem
    int dev = 0;
    cudaGetDevice(&dev);
    int cap = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        const std::tuple<const void*, int, int> key(kernel, dev, smem);
        auto it = resident.find(key);
        if (it == resident.end()) {
            int per_sm = 0, sms = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, size_t(smem));
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            cap = (per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
            resident.emplace(key, cap);
        } else {
            cap = it->second;
        }
    }
    const int64_t need = (units + per_block - 1) / per_block;
    return int(need < cap ? need : cap);
}
int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}
}  // namespace e3gb

using namespace e3gb;

// the device error word (one per device that loads the library)
__device__ unsigned e3gb_device_error_word;

struct e3gb_table {
    const ConfigOps* ops;
    int cfg;
    int mul;
};

namespace {
thread_local std::string g_last_error;

e3gb_status fail(e3gb_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

e3gb_status ok() { return E3GB_OK; }

e3gb_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return E3GB_OK;
    return fail(E3GB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// device address of the error word for the current device (cached per device)
unsigned* error_word(e3gb_status* st) {
    static std::mutex mu;
    static std::unordered_map<int, unsigned*> addr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = cuda_status(e, "cudaGetDevice");
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) return it->second;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, e3gb_device_error_word);
    if (e != cudaSuccess) {
        *st = cuda_status(e, "cudaGetSymbolAddress(error word)");
        return nullptr;
    }
    addr.emplace(dev, static_cast<unsigned*>(p));
    return static_cast<unsigned*>(p);
}

bool valid_mul(int mul) { return mul == 4 || mul == 8 || mul == 16 || mul == 32 || mul == 64 || mul == 128; }

// a pointer must be device-accessible memory of this process, aligned as required
e3gb_status check_ptr(const void* p, const char* name, size_t align, bool needed) {
    if (!needed) return E3GB_OK;
    if (p == nullptr) return fail(E3GB_ERR_INVALID_ARG, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(p) % align != 0)
        return fail(E3GB_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
    cudaPointerAttributes at{};
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(E3GB_ERR_INVALID_ARG, "%s: cannot query pointer (%s)", name, cudaGetErrorString(e));
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return fail(E3GB_ERR_INVALID_ARG, "%s is not device memory", name);
    return E3GB_OK;
}

size_t elt_bytes(e3gb_dtype d) { return d == E3GB_BF16 ? 2 : 4; }
size_t vec_align(e3gb_dtype d) { return d == E3GB_BF16 ? 8 : 16; }

e3gb_status check_table(const e3gb_table* t, e3gb_dtype dtype) {
    if (t == nullptr || t->ops == nullptr) return fail(E3GB_ERR_INVALID_ARG, "table is NULL");
    if (dtype != E3GB_F32 && dtype != E3GB_BF16) return fail(E3GB_ERR_INVALID_ARG, "unknown dtype %d", int(dtype));
    return E3GB_OK;
}

#define E3GB_TRY(expr)                       \
    do {                                     \
        const e3gb_status _s = (expr);       \
        if (_s != E3GB_OK) return _s;        \
    } while (0)
}  // namespace

extern "C" {

const char* e3gb_last_error(void) { return g_last_error.c_str(); }
const char* e3gb_version(void) { return "e3gb 0.1.0 (sm_103a)"; }

int32_t e3gb_config_count(void) { return kNumConfigs; }

e3gb_status e3gb_config_describe(int32_t i, int32_t* n_blocks, int32_t* l, int32_t* parity, int32_t* sh_lmax,
                                 int32_t* out_lmax, int32_t* flags) {
    if (i < 0 || i >= kNumConfigs) return fail(E3GB_ERR_INVALID_ARG, "config index %d out of range", i);
    const ConfigOps* o = kRegistry[i]();
    const int nb = xcode_nblocks(o->xcode);
    if (n_blocks) *n_blocks = nb;
    for (int b = 0; b < nb; ++b) {
        if (l) l[b] = xcode_l(o->xcode, b);
        if (parity) parity[b] = xcode_p(o->xcode, b);
    }
    if (sh_lmax) *sh_lmax = o->L2;
    if (out_lmax) *out_lmax = o->L3;
    if (flags) *flags = o->per_path ? E3GB_PATHS_SEPARATE : E3GB_PATHS_SUMMED;
    return ok();
}

e3gb_status e3gb_table_create(const e3gb_irreps* x, int32_t sh_lmax, int32_t out_lmax, int32_t flags,
                              e3gb_table** out) {
    if (out == nullptr) return fail(E3GB_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (x == nullptr || x->l == nullptr || x->parity == nullptr) return fail(E3GB_ERR_INVALID_ARG, "irreps is NULL");
    if (x->n <= 0 || x->n > kMaxBlocks) return fail(E3GB_ERR_INVALID_ARG, "irreps: %d blocks (1..8)", x->n);
    if (flags != E3GB_PATHS_SUMMED && flags != E3GB_PATHS_SEPARATE) return fail(E3GB_ERR_INVALID_ARG, "bad flags");
    if (sh_lmax < 0 || sh_lmax > kLmax || out_lmax < 0 || out_lmax > kLmax)
        return fail(E3GB_ERR_UNSUPPORTED, "sh_lmax and out_lmax must be in 0..3");
    uint32_t code = 0;
    for (int i = 0; i < x->n; ++i) {
        if (x->l[i] < 0 || x->l[i] > kLmax) return fail(E3GB_ERR_UNSUPPORTED, "irreps block %d: l=%d not in 0..3", i, x->l[i]);
        if (x->parity[i] != 1 && x->parity[i] != -1) return fail(E3GB_ERR_INVALID_ARG, "irreps block %d: parity must be +-1", i);
        code |= xblock(x->l[i], x->parity[i]) << (4 * i);
    }
    if (!valid_mul(x->mul))
        return fail(E3GB_ERR_UNSUPPORTED, "multiplicity %d: supported channel counts are 4, 8, 16, 32, 64, 128", x->mul);
    for (int i = 0; i < kNumConfigs; ++i) {
        const ConfigOps* o = kRegistry[i]();
        if (o->xcode == code && o->L2 == sh_lmax && o->L3 == out_lmax && o->per_path == flags) {
            *out = new e3gb_table{o, i, x->mul};
            return ok();
        }
    }
    return fail(E3GB_ERR_UNSUPPORTED, "irreps configuration has no compiled kernels (see e3gb_config_describe)");
}

e3gb_status e3gb_table_destroy(e3gb_table* t) {
    delete t;
    return ok();
}

e3gb_status e3gb_table_info(const e3gb_table* t, int32_t* d1, int32_t* d2, int32_t* n_paths, int32_t* D,
                            int32_t* nnz, int32_t* mul) {
    if (t == nullptr) return fail(E3GB_ERR_INVALID_ARG, "table is NULL");
    if (d1) *d1 = t->ops->D1;
    if (d2) *d2 = t->ops->D2;
    if (n_paths) *n_paths = t->ops->NP;
    if (D) *D = t->ops->D;
    if (nnz) *nnz = t->ops->NR;
    if (mul) *mul = t->mul;
    return ok();
}

e3gb_status e3gb_table_paths(const e3gb_table* t, int32_t* paths) {
    if (t == nullptr || paths == nullptr) return fail(E3GB_ERR_INVALID_ARG, "NULL argument");
    for (int p = 0; p < t->ops->NP; ++p) {
        const PathInfo& q = t->ops->paths[p];
        const int32_t v[8] = {q.xblock, q.l1, q.p1, q.l2, q.l3, q.p3, q.out_block, q.zoff};
        std::memcpy(paths + 8 * p, v, sizeof(v));
    }
    return ok();
}

e3gb_status e3gb_table_coefficients(const e3gb_table* t, double* rec) {
    if (t == nullptr || rec == nullptr) return fail(E3GB_ERR_INVALID_ARG, "NULL argument");
    for (int i = 0; i < t->ops->NR; ++i) {
        const Rec& r = t->ops->recs[i];
        rec[5 * i + 0] = r.path;
        rec[5 * i + 1] = r.m1;
        rec[5 * i + 2] = r.m2;
        rec[5 * i + 3] = r.m3;
        rec[5 * i + 4] = r.cd;
    }
    return ok();
}

e3gb_status e3gb_sh_forward(int32_t lmax, int64_t n, const float* vec, void* y, e3gb_dtype dtype, void* stream) {
    if (lmax < 0 || lmax > kLmax) return fail(E3GB_ERR_UNSUPPORTED, "lmax %d not in 0..3", lmax);
    if (n < 0) return fail(E3GB_ERR_INVALID_ARG, "n < 0");
    if (dtype != E3GB_F32 && dtype != E3GB_BF16) return fail(E3GB_ERR_INVALID_ARG, "unknown dtype");
    if (n == 0) return ok();
    E3GB_TRY(check_ptr(vec, "vec", 4, true));
    E3GB_TRY(check_ptr(y, "y", elt_bytes(dtype), true));
    return cuda_status(sh_forward(lmax, n, vec, y, dtype == E3GB_BF16, (cudaStream_t)stream), "sh_forward launch");
}

e3gb_status e3gb_sh_backward(int32_t lmax, int64_t n, const float* vec, const void* dy, float* dvec, e3gb_dtype dtype,
                             void* stream) {
    if (lmax < 0 || lmax > kLmax) return fail(E3GB_ERR_UNSUPPORTED, "lmax %d not in 0..3", lmax);
    if (n < 0) return fail(E3GB_ERR_INVALID_ARG, "n < 0");
    if (dtype != E3GB_F32 && dtype != E3GB_BF16) return fail(E3GB_ERR_INVALID_ARG, "unknown dtype");
    if (n == 0) return ok();
    E3GB_TRY(check_ptr(vec, "vec", 4, true));
    E3GB_TRY(check_ptr(dy, "dy", elt_bytes(dtype), true));
    E3GB_TRY(check_ptr(dvec, "dvec", 4, true));
    return cuda_status(sh_backward(lmax, n, vec, dy, dvec, dtype == E3GB_BF16, (cudaStream_t)stream),
                       "sh_backward launch");
}

e3gb_status e3gb_tp_forward(const e3gb_table* t, int64_t rows, const void* x, const void* y, const void* w, void* z,
                            e3gb_dtype dtype, void* stream) {
    E3GB_TRY(check_table(t, dtype));
    if (rows < 0) return fail(E3GB_ERR_INVALID_ARG, "rows < 0");
    if (rows == 0) return ok();
    const size_t va = vec_align(dtype), ea = elt_bytes(dtype);
    E3GB_TRY(check_ptr(x, "x", va, true));
    E3GB_TRY(check_ptr(y, "y", ea, true));
    E3GB_TRY(check_ptr(w, "w", va, true));
    E3GB_TRY(check_ptr(z, "z", 16, true));
    return cuda_status(t->ops->tp_fwd[dtype](rows, t->mul, x, y, w, z, (cudaStream_t)stream), "tp_forward launch");
}

e3gb_status e3gb_tp_backward(const e3gb_table* t, int64_t rows, const void* x, const void* y, const void* w,
                             const void* dz, void* dx, void* dy, void* dw, e3gb_dtype dtype, void* stream) {
    E3GB_TRY(check_table(t, dtype));
    if (rows < 0) return fail(E3GB_ERR_INVALID_ARG, "rows < 0");
    if (rows == 0) return ok();
    const size_t va = vec_align(dtype), ea = elt_bytes(dtype);
    E3GB_TRY(check_ptr(x, "x", va, true));
    E3GB_TRY(check_ptr(y, "y", ea, true));
    E3GB_TRY(check_ptr(w, "w", va, true));
    E3GB_TRY(check_ptr(dz, "dz", va, true));
    E3GB_TRY(check_ptr(dx, "dx", 16, true));
    E3GB_TRY(check_ptr(dy, "dy", 4, true));
    E3GB_TRY(check_ptr(dw, "dw", 16, true));
    return cuda_status(t->ops->tp_bwd[dtype](rows, t->mul, x, y, w, dz, dx, dy, dw, (cudaStream_t)stream),
                       "tp_backward launch");
}

size_t e3gb_graph_prepare_workspace_bytes(int64_t n_nodes, int64_t n_edges) {
    return (n_nodes < 0 || n_edges < 0) ? 0 : graph_workspace_bytes(n_nodes, n_edges);
}

e3gb_status e3gb_graph_prepare(int64_t n_nodes, int64_t n_edges, const int32_t* rowptr, const int32_t* sender,
                               int32_t* csc_ptr, int32_t* csc_edge, int32_t* csc_recv, void* workspace,
                               size_t ws_bytes, void* stream) {
    if (n_nodes < 0 || n_edges < 0) return fail(E3GB_ERR_INVALID_ARG, "negative size");
    if (n_nodes >= INT32_MAX || n_edges >= INT32_MAX) return fail(E3GB_ERR_INVALID_ARG, "sizes must be < 2^31-1");
    if (n_nodes == 0 && n_edges > 0) return fail(E3GB_ERR_BAD_GRAPH, "edges without nodes");
    if (ws_bytes < graph_workspace_bytes(n_nodes, n_edges))
        return fail(E3GB_ERR_INVALID_ARG, "workspace of %zu bytes, need %zu", ws_bytes,
                    graph_workspace_bytes(n_nodes, n_edges));
    E3GB_TRY(check_ptr(rowptr, "rowptr", 4, true));
    E3GB_TRY(check_ptr(csc_ptr, "csc_ptr", 4, true));
    E3GB_TRY(check_ptr(workspace, "workspace", 16, true));
    E3GB_TRY(check_ptr(sender, "sender", 4, n_edges > 0));
    E3GB_TRY(check_ptr(csc_edge, "csc_edge", 4, n_edges > 0));
    E3GB_TRY(check_ptr(csc_recv, "csc_recv", 4, n_edges > 0));
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    return cuda_status(graph_prepare(n_nodes, n_edges, rowptr, sender, csc_ptr, csc_edge, csc_recv, workspace, 0,
                                     err, (cudaStream_t)stream),
                       "graph_prepare launch");
}

// Allocation-free variant of e3gb_graph_prepare (see the header for who needs it): the
// sort's per-tile digit counts live in this file-scope array. Host code must not pass the
// symbol itself to a kernel (in host code it names a host-side stand-in); the device address
// is looked up once per device with cudaGetSymbolAddress and passed on.
static __device__ __align__(256) int32_t e3gb_prepare_scratch[E3GB_STATIC_PREPARE_SCRATCH_BYTES / 4];

static int32_t* prepare_scratch(e3gb_status* st) {
    static std::mutex mu;
    static std::unordered_map<int, int32_t*> addr;   // device -> address of the array there
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = cuda_status(e, "cudaGetDevice");
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(mu);
    auto it = addr.find(dev);
    if (it != addr.end()) return it->second;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, e3gb_prepare_scratch);
    if (e != cudaSuccess || p == nullptr) {
        *st = cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol, "cudaGetSymbolAddress(prepare scratch)");
        return nullptr;
    }
    addr.emplace(dev, static_cast<int32_t*>(p));
    return static_cast<int32_t*>(p);
}

e3gb_status e3gb_graph_prepare_static(int64_t n_nodes, int64_t n_edges, const int32_t* rowptr, const int32_t* sender,
                                      int32_t* csc_ptr, int32_t* csc_edge, int32_t* csc_recv, void* stream) {
    if (n_nodes < 0 || n_edges < 0) return fail(E3GB_ERR_INVALID_ARG, "negative size");
    if (n_nodes >= INT32_MAX || n_edges >= INT32_MAX)
        return fail(E3GB_ERR_INVALID_ARG, "sizes must be < 2^31-1 (e3gb_graph_prepare_static)");
    if (n_nodes == 0 && n_edges > 0) return fail(E3GB_ERR_BAD_GRAPH, "edges without nodes");
    E3GB_TRY(check_ptr(rowptr, "rowptr", 4, true));
    E3GB_TRY(check_ptr(csc_ptr, "csc_ptr", 4, true));
    E3GB_TRY(check_ptr(sender, "sender", 4, n_edges > 0));
    E3GB_TRY(check_ptr(csc_edge, "csc_edge", 4, n_edges > 0));
    E3GB_TRY(check_ptr(csc_recv, "csc_recv", 4, n_edges > 0));
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    int32_t* scratch = prepare_scratch(&st);
    if (scratch == nullptr) return st;
    // the tile count is capped so that the counts fit the array; every count is written
    // before it is read, so the previous call's contents need no clearing
    static const int64_t cap = graph_static_tiles_cap(E3GB_STATIC_PREPARE_SCRATCH_BYTES / 4);
    return cuda_status(graph_prepare(n_nodes, n_edges, rowptr, sender, csc_ptr, csc_edge, csc_recv, scratch, cap,
                                     err, (cudaStream_t)stream),
                       "graph_prepare_static launch");
}

e3gb_status e3gb_conv_forward(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, const int32_t* rowptr,
                              const int32_t* sender, const void* x, const void* y, const void* w, float scale,
                              int64_t pad_node, void* m, e3gb_dtype dtype, void* stream) {
    E3GB_TRY(check_table(t, dtype));
    if (n_nodes < 0 || n_edges < 0) return fail(E3GB_ERR_INVALID_ARG, "negative size");
    if (n_nodes >= INT32_MAX || n_edges >= INT32_MAX) return fail(E3GB_ERR_INVALID_ARG, "sizes must be < 2^31-1");
    if (pad_node < -1 || pad_node >= n_nodes)
        return fail(E3GB_ERR_INVALID_ARG, "pad_node %lld outside [-1, n_nodes)", (long long)pad_node);
    if (n_nodes == 0) {
        if (n_edges > 0) return fail(E3GB_ERR_BAD_GRAPH, "edges without nodes");
        return ok();
    }
    const size_t va = vec_align(dtype), ea = elt_bytes(dtype);
    const bool edges = n_edges > 0;
    E3GB_TRY(check_ptr(rowptr, "rowptr", 4, true));
    E3GB_TRY(check_ptr(sender, "sender", 4, edges));
    E3GB_TRY(check_ptr(x, "x", va, true));
    E3GB_TRY(check_ptr(y, "y", ea, edges));
    E3GB_TRY(check_ptr(w, "w", va, edges));
    E3GB_TRY(check_ptr(m, "m", 16, true));
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    return cuda_status(t->ops->conv_fwd[dtype](n_nodes, n_edges, t->mul, rowptr, sender, x, y, w, scale, m, pad_node,
                                               err, INT64_MAX, (cudaStream_t)stream),
                       "conv_forward launch");
}

// the split forward's workspace: piece pointers, the scan's block sums, the partial rows
static size_t split_workspace_bytes(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, int32_t chunk) {
    const size_t ptr = size_t(n_nodes + 1 + 63) / 64 * 64;
    const size_t sums = (scan_sums_count(n_nodes + 1) + 63) / 64 * 64;
    const size_t pieces = size_t(n_edges / chunk + 1);
    return (ptr + sums) * 4 + pieces * size_t(t->ops->D) * size_t(t->mul) * 4;
}

size_t e3gb_conv_forward_split_workspace_bytes(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, int32_t chunk) {
    if (t == nullptr || t->ops == nullptr || n_nodes < 0 || n_edges < 0 || chunk < 1) return 0;
    return split_workspace_bytes(t, n_nodes, n_edges, chunk);
}

e3gb_status e3gb_conv_forward_split(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, const int32_t* rowptr,
                                    const int32_t* sender, const void* x, const void* y, const void* w, float scale,
                                    int64_t pad_node, int32_t chunk, void* m, void* workspace, size_t ws_bytes,
                                    e3gb_dtype dtype, void* stream) {
    E3GB_TRY(check_table(t, dtype));
    if (chunk < 1) return fail(E3GB_ERR_INVALID_ARG, "chunk must be >= 1");
    if (t->ops->D > 32)
        return fail(E3GB_ERR_UNSUPPORTED, "the split forward keeps at most 32 output rows per receiver (D = %d)",
                    t->ops->D);
    if (n_nodes < 0 || n_edges < 0) return fail(E3GB_ERR_INVALID_ARG, "negative size");
    if (n_nodes >= INT32_MAX || n_edges >= INT32_MAX) return fail(E3GB_ERR_INVALID_ARG, "sizes must be < 2^31-1");
    if (pad_node < -1 || pad_node >= n_nodes)
        return fail(E3GB_ERR_INVALID_ARG, "pad_node %lld outside [-1, n_nodes)", (long long)pad_node);
    if (n_nodes == 0) {
        if (n_edges > 0) return fail(E3GB_ERR_BAD_GRAPH, "edges without nodes");
        return ok();
    }
    const size_t need = split_workspace_bytes(t, n_nodes, n_edges, chunk);
    if (ws_bytes < need) return fail(E3GB_ERR_INVALID_ARG, "workspace of %zu bytes, need %zu", ws_bytes, need);
    const size_t va = vec_align(dtype), ea = elt_bytes(dtype);
    const bool edges = n_edges > 0;
    E3GB_TRY(check_ptr(rowptr, "rowptr", 4, true));
    E3GB_TRY(check_ptr(sender, "sender", 4, edges));
    E3GB_TRY(check_ptr(x, "x", va, true));
    E3GB_TRY(check_ptr(y, "y", ea, edges));
    E3GB_TRY(check_ptr(w, "w", va, edges));
    E3GB_TRY(check_ptr(m, "m", 16, true));
    E3GB_TRY(check_ptr(workspace, "workspace", 16, true));
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    E3GB_TRY(cuda_status(t->ops->conv_fwd[dtype](n_nodes, n_edges, t->mul, rowptr, sender, x, y, w, scale, m, pad_node,
                                                 err, chunk, (cudaStream_t)stream),
                         "conv_forward_split launch"));
    return cuda_status(t->ops->conv_fwd_pieces[dtype](n_nodes, n_edges, t->mul, rowptr, sender, x, y, w, scale, m,
                                                      pad_node, chunk, workspace, err, (cudaStream_t)stream),
                       "conv_forward_split pieces launch");
}

e3gb_status e3gb_conv_backward(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, const int32_t* csc_ptr,
                               const int32_t* csc_edge, const int32_t* csc_recv, const void* x, const void* y,
                               const void* w, const void* dm, float scale, int64_t pad_node, void* dx, void* dy,
                               void* dw, e3gb_dtype dtype, void* stream) {
    E3GB_TRY(check_table(t, dtype));
    if (n_nodes < 0 || n_edges < 0) return fail(E3GB_ERR_INVALID_ARG, "negative size");
    if (n_nodes >= INT32_MAX || n_edges >= INT32_MAX) return fail(E3GB_ERR_INVALID_ARG, "sizes must be < 2^31-1");
    if (pad_node < -1 || pad_node >= n_nodes)
        return fail(E3GB_ERR_INVALID_ARG, "pad_node %lld outside [-1, n_nodes)", (long long)pad_node);
    if (n_nodes == 0) {
        if (n_edges > 0) return fail(E3GB_ERR_BAD_GRAPH, "edges without nodes");
        return ok();
    }
    const size_t va = vec_align(dtype), ea = elt_bytes(dtype);
    const bool edges = n_edges > 0;
    E3GB_TRY(check_ptr(csc_ptr, "csc_ptr", 4, true));
    E3GB_TRY(check_ptr(csc_edge, "csc_edge", 4, edges));
    E3GB_TRY(check_ptr(csc_recv, "csc_recv", 4, edges));
    E3GB_TRY(check_ptr(x, "x", va, true));
    E3GB_TRY(check_ptr(y, "y", ea, edges));
    E3GB_TRY(check_ptr(w, "w", va, edges));
    E3GB_TRY(check_ptr(dm, "dm", va, true));
    E3GB_TRY(check_ptr(dx, "dx", 16, true));
    E3GB_TRY(check_ptr(dy, "dy", 4, edges));
    E3GB_TRY(check_ptr(dw, "dw", 16, edges));
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    E3GB_TRY(cuda_status(t->ops->conv_bwd[dtype](n_nodes, n_edges, t->mul, csc_ptr, csc_edge, csc_recv, x, y, w,
                                                 dm, scale, dx, dy, dw, pad_node, err, (cudaStream_t)stream),
                         "conv_backward launch"));
    return cuda_status(zero_padding_edges(n_nodes, n_edges, csc_ptr, csc_edge, csc_recv, pad_node, (float*)dw,
                                          int64_t(t->ops->NP) * t->mul, (float*)dy, t->ops->D2, (cudaStream_t)stream),
                       "zero_padding_edges launch");
}

// ------------------------------------------------------------------------------------------
// radial edge scalars and the radial convolution
// ------------------------------------------------------------------------------------------
static e3gb_status check_radial_net(int32_t n_basis, int32_t hidden, float r_cut) {
    if (n_basis < 1 || n_basis > kRadialMaxBasis)
        return fail(E3GB_ERR_INVALID_ARG, "n_basis %d outside [1, %d]", n_basis, kRadialMaxBasis);
    if (hidden < 1 || hidden > kRadialMaxHidden)
        return fail(E3GB_ERR_INVALID_ARG, "hidden %d outside [1, %d]", hidden, kRadialMaxHidden);
    if (!(r_cut > 0.f)) return fail(E3GB_ERR_INVALID_ARG, "r_cut must be positive");
    return E3GB_OK;
}

e3gb_status e3gb_radial_hidden(int64_t n_edges, const float* vec, const float* W1, int32_t n_basis, int32_t hidden,
                               float r_cut, float* h, void* stream) {
    if (n_edges < 0 || n_edges >= INT32_MAX) return fail(E3GB_ERR_INVALID_ARG, "n_edges outside [0, 2^31-1)");
    E3GB_TRY(check_radial_net(n_basis, hidden, r_cut));
    const bool edges = n_edges > 0;
    E3GB_TRY(check_ptr(vec, "vec", 4, edges));
    E3GB_TRY(check_ptr(W1, "W1", 4, true));
    E3GB_TRY(check_ptr(h, "h", 4, edges));
    return cuda_status(radial_hidden(n_edges, vec, W1, n_basis, hidden, r_cut, h, (cudaStream_t)stream),
                       "radial_hidden launch");
}

e3gb_status e3gb_radial_backward(int64_t n_edges, const float* vec, const float* W1, int32_t n_basis, int32_t hidden,
                                 float r_cut, const float* dh, float* dvec, int32_t accumulate, void* stream) {
    if (n_edges < 0 || n_edges >= INT32_MAX) return fail(E3GB_ERR_INVALID_ARG, "n_edges outside [0, 2^31-1)");
    E3GB_TRY(check_radial_net(n_basis, hidden, r_cut));
    const bool edges = n_edges > 0;
    E3GB_TRY(check_ptr(vec, "vec", 4, edges));
    E3GB_TRY(check_ptr(W1, "W1", 4, true));
    E3GB_TRY(check_ptr(dh, "dh", 4, edges));
    E3GB_TRY(check_ptr(dvec, "dvec", 4, edges));
    return cuda_status(radial_backward(n_edges, vec, W1, n_basis, hidden, r_cut, dh, dvec, accumulate ? 1 : 0,
                                       (cudaStream_t)stream),
                       "radial_backward launch");
}

static e3gb_status check_radial_conv(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, int32_t hidden,
                                     int64_t pad_node, e3gb_dtype dtype) {
    E3GB_TRY(check_table(t, dtype));
    if (dtype != E3GB_F32) return fail(E3GB_ERR_UNSUPPORTED, "the radial convolution is built for fp32 only");
    if (hidden != kRadialHidden)
        return fail(E3GB_ERR_UNSUPPORTED, "the radial convolution is built for hidden = %d (got %d)", kRadialHidden,
                    hidden);
    if (t->ops->D > 32)
        return fail(E3GB_ERR_UNSUPPORTED, "the radial convolution keeps at most 32 output rows per receiver (D = %d)",
                    t->ops->D);
    if (t->ops->conv_fwd_rad == nullptr || int64_t(kRadialHidden) * t->ops->NP * t->mul * 4 > 232448)
        return fail(E3GB_ERR_UNSUPPORTED, "W2 of %d x %d x %d floats does not fit in shared memory", kRadialHidden,
                    t->ops->NP, t->mul);
    if (n_nodes < 0 || n_edges < 0) return fail(E3GB_ERR_INVALID_ARG, "negative size");
    if (n_nodes >= INT32_MAX || n_edges >= INT32_MAX) return fail(E3GB_ERR_INVALID_ARG, "sizes must be < 2^31-1");
    if (pad_node < -1 || pad_node >= n_nodes)
        return fail(E3GB_ERR_INVALID_ARG, "pad_node %lld outside [-1, n_nodes)", (long long)pad_node);
    if (n_nodes == 0 && n_edges > 0) return fail(E3GB_ERR_BAD_GRAPH, "edges without nodes");
    return E3GB_OK;
}

e3gb_status e3gb_conv_forward_radial(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, const int32_t* rowptr,
                                     const int32_t* sender, const void* x, const void* y, const float* h,
                                     const float* W2, int32_t hidden, float scale, int64_t pad_node, void* m,
                                     e3gb_dtype dtype, void* stream) {
    E3GB_TRY(check_radial_conv(t, n_nodes, n_edges, hidden, pad_node, dtype));
    if (n_nodes == 0) return ok();
    const bool edges = n_edges > 0;
    E3GB_TRY(check_ptr(rowptr, "rowptr", 4, true));
    E3GB_TRY(check_ptr(sender, "sender", 4, edges));
    E3GB_TRY(check_ptr(x, "x", 16, true));
    E3GB_TRY(check_ptr(y, "y", 4, edges));
    E3GB_TRY(check_ptr(h, "h", 16, edges));
    E3GB_TRY(check_ptr(W2, "W2", 16, true));
    E3GB_TRY(check_ptr(m, "m", 16, true));
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    return cuda_status(t->ops->conv_fwd_rad(n_nodes, n_edges, t->mul, rowptr, sender, (const float*)x, (const float*)y,
                                            h, W2, scale, (float*)m, pad_node, err, (cudaStream_t)stream),
                       "conv_forward_radial launch");
}

e3gb_status e3gb_conv_backward_radial(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, const int32_t* csc_ptr,
                                      const int32_t* csc_edge, const int32_t* csc_recv, const void* x, const void* y,
                                      const float* h, const float* W2, int32_t hidden, const void* dm, float scale,
                                      int64_t pad_node, void* dx, void* dy, float* dh, e3gb_dtype dtype,
                                      void* stream) {
    E3GB_TRY(check_radial_conv(t, n_nodes, n_edges, hidden, pad_node, dtype));
    if (n_nodes == 0) return ok();
    const bool edges = n_edges > 0;
    E3GB_TRY(check_ptr(csc_ptr, "csc_ptr", 4, true));
    E3GB_TRY(check_ptr(csc_edge, "csc_edge", 4, edges));
    E3GB_TRY(check_ptr(csc_recv, "csc_recv", 4, edges));
    E3GB_TRY(check_ptr(x, "x", 16, true));
    E3GB_TRY(check_ptr(y, "y", 4, edges));
    E3GB_TRY(check_ptr(h, "h", 16, edges));
    E3GB_TRY(check_ptr(W2, "W2", 16, true));
    E3GB_TRY(check_ptr(dm, "dm", 16, true));
    E3GB_TRY(check_ptr(dx, "dx", 16, true));
    E3GB_TRY(check_ptr(dy, "dy", 4, edges));
    E3GB_TRY(check_ptr(dh, "dh", 16, edges));
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    E3GB_TRY(cuda_status(t->ops->conv_bwd_rad(n_nodes, n_edges, t->mul, csc_ptr, csc_edge, csc_recv, (const float*)x,
                                              (const float*)y, h, W2, (const float*)dm, scale, (float*)dx, (float*)dy,
                                              dh, pad_node, err, (cudaStream_t)stream),
                         "conv_backward_radial launch"));
    return cuda_status(zero_padding_edges(n_nodes, n_edges, csc_ptr, csc_edge, csc_recv, pad_node, dh, kRadialHidden,
                                          (float*)dy, t->ops->D2, (cudaStream_t)stream),
                       "zero_padding_edges launch");
}

e3gb_status e3gb_conv_double_backward(const e3gb_table* t, int64_t n_nodes, int64_t n_edges, const int32_t* rowptr,
                                      const int32_t* sender, const int32_t* csc_ptr, const int32_t* csc_edge,
                                      const int32_t* csc_recv, const void* x, const void* y, const void* w,
                                      const void* dm, const void* delta_dx, const void* delta_dy, const void* delta_dw,
                                      float scale, int64_t pad_node, void* delta_x, void* delta_y, void* delta_w,
                                      void* delta_dm, e3gb_dtype dtype, void* stream) {
    E3GB_TRY(check_table(t, dtype));
    if (n_nodes < 0 || n_edges < 0) return fail(E3GB_ERR_INVALID_ARG, "negative size");
    if (n_nodes >= INT32_MAX || n_edges >= INT32_MAX) return fail(E3GB_ERR_INVALID_ARG, "sizes must be < 2^31-1");
    if (pad_node < -1 || pad_node >= n_nodes)
        return fail(E3GB_ERR_INVALID_ARG, "pad_node %lld outside [-1, n_nodes)", (long long)pad_node);
    if (n_nodes == 0) {
        if (n_edges > 0) return fail(E3GB_ERR_BAD_GRAPH, "edges without nodes");
        return ok();
    }
    const size_t va = vec_align(dtype), ea = elt_bytes(dtype);
    const bool edges = n_edges > 0;
    E3GB_TRY(check_ptr(rowptr, "rowptr", 4, true));
    E3GB_TRY(check_ptr(sender, "sender", 4, edges));
    E3GB_TRY(check_ptr(csc_ptr, "csc_ptr", 4, true));
    E3GB_TRY(check_ptr(csc_edge, "csc_edge", 4, edges));
    E3GB_TRY(check_ptr(csc_recv, "csc_recv", 4, edges));
    E3GB_TRY(check_ptr(x, "x", va, true));
    E3GB_TRY(check_ptr(y, "y", ea, edges));
    E3GB_TRY(check_ptr(w, "w", va, edges));
    E3GB_TRY(check_ptr(dm, "dm", va, true));
    E3GB_TRY(check_ptr(delta_dx, "delta_dx", va, true));
    E3GB_TRY(check_ptr(delta_dy, "delta_dy", ea, edges));
    E3GB_TRY(check_ptr(delta_dw, "delta_dw", va, edges));
    E3GB_TRY(check_ptr(delta_x, "delta_x", 16, true));
    E3GB_TRY(check_ptr(delta_y, "delta_y", 4, edges));
    E3GB_TRY(check_ptr(delta_w, "delta_w", 16, edges));
    E3GB_TRY(check_ptr(delta_dm, "delta_dm", 16, true));
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    E3GB_TRY(cuda_status(t->ops->conv_dbwd[dtype](n_nodes, n_edges, t->mul, rowptr, sender, csc_ptr, csc_edge,
                                                  csc_recv, x, y, w, dm, delta_dx, delta_dy, delta_dw, scale, delta_x,
                                                  delta_y, delta_w, delta_dm, pad_node, err, (cudaStream_t)stream),
                         "conv_double_backward launch"));
    return cuda_status(zero_padding_edges(n_nodes, n_edges, csc_ptr, csc_edge, csc_recv, pad_node, (float*)delta_w,
                                          int64_t(t->ops->NP) * t->mul, (float*)delta_y, t->ops->D2,
                                          (cudaStream_t)stream),
                       "zero_padding_edges launch");
}

namespace {
e3gb_status coo_common(bool backward, int64_t rows, int32_t d1, int32_t d2, int32_t D, int32_t n_paths, int32_t mul,
                       int32_t n_rec, const int32_t* rec, const float* coef, const void* x, const void* y,
                       const void* w, const void* dz, void* out0, void* out1, void* out2, e3gb_dtype dtype,
                       void* stream) {
    if (dtype != E3GB_F32 && dtype != E3GB_BF16) return fail(E3GB_ERR_INVALID_ARG, "unknown dtype");
    if (rows < 0 || n_rec < 0) return fail(E3GB_ERR_INVALID_ARG, "negative size");
    if (d1 < 1 || d2 < 1 || D < 1 || n_paths < 1) return fail(E3GB_ERR_INVALID_ARG, "d1, d2, D, n_paths must be >= 1");
    if (!(mul == 1 || mul == 2 || mul == 4 || mul == 8 || mul == 16 || mul == 32 || mul == 64 || mul == 128))
        return fail(E3GB_ERR_UNSUPPORTED, "mul %d not a power of two <= 128", mul);
    if (coo_smem_bytes(backward, d1, d2, D, n_paths, mul) > 232448)
        return fail(E3GB_ERR_UNSUPPORTED, "output rows x channels too large for one block's shared memory");
    if (rows == 0) return ok();
    const size_t va = mul >= 64 ? vec_align(dtype) : elt_bytes(dtype), ea = elt_bytes(dtype);
    E3GB_TRY(check_ptr(rec, "records", 16, n_rec > 0));
    E3GB_TRY(check_ptr(coef, "coefficients", 4, n_rec > 0));
    E3GB_TRY(check_ptr(x, "x", va, true));
    E3GB_TRY(check_ptr(y, "y", ea, true));
    E3GB_TRY(check_ptr(w, "w", va, true));
    if (backward) {
        E3GB_TRY(check_ptr(dz, "dz", va, true));
        E3GB_TRY(check_ptr(out0, "dx", mul >= 64 ? 16 : 4, true));
        E3GB_TRY(check_ptr(out1, "dy", 4, true));
        E3GB_TRY(check_ptr(out2, "dw", mul >= 64 ? 16 : 4, true));
    } else {
        E3GB_TRY(check_ptr(out0, "z", mul >= 64 ? 16 : 4, true));
    }
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    const cudaError_t e =
        dtype == E3GB_F32
            ? coo_tp<float>(backward, rows, d1, d2, D, n_paths, mul, n_rec, rec, coef, x, y, w, dz, out0, out1, out2,
                            err, (cudaStream_t)stream)
            : coo_tp<__nv_bfloat16>(backward, rows, d1, d2, D, n_paths, mul, n_rec, rec, coef, x, y, w, dz, out0,
                                    out1, out2, err, (cudaStream_t)stream);
    return cuda_status(e, backward ? "coo_tp_backward launch" : "coo_tp_forward launch");
}
}  // namespace

e3gb_status e3gb_coo_tp_forward(int64_t rows, int32_t d1, int32_t d2, int32_t D, int32_t n_paths, int32_t mul,
                                int32_t n_rec, const int32_t* rec, const float* coef, const void* x, const void* y,
                                const void* w, void* z, e3gb_dtype dtype, void* stream) {
    return coo_common(false, rows, d1, d2, D, n_paths, mul, n_rec, rec, coef, x, y, w, nullptr, z, nullptr, nullptr,
                      dtype, stream);
}

e3gb_status e3gb_coo_tp_backward(int64_t rows, int32_t d1, int32_t d2, int32_t D, int32_t n_paths, int32_t mul,
                                 int32_t n_rec, const int32_t* rec, const float* coef, const void* x, const void* y,
                                 const void* w, const void* dz, void* dx, void* dy, void* dw, e3gb_dtype dtype,
                                 void* stream) {
    return coo_common(true, rows, d1, d2, D, n_paths, mul, n_rec, rec, coef, x, y, w, dz, dx, dy, dw, dtype, stream);
}

e3gb_status e3gb_check_device_status(void* stream, int32_t* flags) {
    if (flags) *flags = 0;
    e3gb_status st = E3GB_OK;
    unsigned* err = error_word(&st);
    if (err == nullptr) return st;
    cudaStream_t s = (cudaStream_t)stream;
    unsigned host = 0;
    E3GB_TRY(cuda_status(cudaMemcpyAsync(&host, err, sizeof(unsigned), cudaMemcpyDeviceToHost, s), "read error word"));
    E3GB_TRY(cuda_status(cudaMemsetAsync(err, 0, sizeof(unsigned), s), "clear error word"));
    E3GB_TRY(cuda_status(cudaStreamSynchronize(s), "cudaStreamSynchronize"));
    if (flags) *flags = int32_t(host);
    if (host != 0) return fail(E3GB_ERR_DEVICE_INDEX, "device saw out-of-range indices (flags 0x%x)", host);
    return ok();
}

}  // extern "C"
