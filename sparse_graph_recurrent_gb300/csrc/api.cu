// The C ABI of libck: argument checks, error reporting, and dispatch to the
// graph build (graph.cu) and the recurrence kernels (recurrence.cu).
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "ck_internal.h"

namespace ck {
namespace {
thread_local char g_msg[512] = "";
thread_local int64_t g_launches = 0;
}  // namespace

ck_status fail(ck_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

ck_status cuda_fail(cudaError_t e, const char *what) {
    cudaGetLastError();  // clear a non-sticky error so later calls can proceed
    return fail(CK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

Options &options() {
    static Options o;
    return o;
}

namespace {

ck_status check_graph(const ck_graph *g) {
    if (!g) return fail(CK_ERR_INVALID_ARG, "graph handle is NULL");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != g->device)
        return fail(CK_ERR_INVALID_ARG, "graph was built on device %d, current device is %d",
                    g->device, dev);
    return CK_OK;
}

bool misaligned(const void *p) { return ((uintptr_t)p & 31u) != 0; }

}  // namespace
}  // namespace ck

using namespace ck;

extern "C" {

const char *ck_status_string(ck_status s) {
    switch (s) {
        case CK_OK: return "CK_OK";
        case CK_ERR_INVALID_ARG: return "CK_ERR_INVALID_ARG";
        case CK_ERR_CUDA: return "CK_ERR_CUDA";
        case CK_ERR_OUT_OF_MEMORY: return "CK_ERR_OUT_OF_MEMORY";
        case CK_ERR_TIMEOUT: return "CK_ERR_TIMEOUT";
        case CK_ERR_WORKSPACE: return "CK_ERR_WORKSPACE";
        case CK_ERR_INTERNAL: return "CK_ERR_INTERNAL";
        case CK_ERR_UNSUPPORTED: return "CK_ERR_UNSUPPORTED";
    }
    return "CK_ERR_UNKNOWN";
}

const char *ck_last_error_message(void) { return g_msg; }

int64_t ck_last_launch_count(void) { return g_launches; }

ck_status ck_set_option(ck_option opt, int64_t v) {
    Options &o = options();
    switch (opt) {
        case CK_OPT_PERSISTENT: o.persistent = v != 0; return CK_OK;
        case CK_OPT_BARRIER_TIMEOUT_NS:
            if (v < 1000) return fail(CK_ERR_INVALID_ARG, "timeout must be >= 1000 ns");
            o.timeout_ns = v;
            return CK_OK;
        case CK_OPT_TEST_BARRIER_EXTRA:
            if (v < 0 || v > 1024) return fail(CK_ERR_INVALID_ARG, "barrier extra out of range");
            o.barrier_extra = (int)v;
            return CK_OK;
        case CK_OPT_GRAPH_IN_SMEM: o.graph_in_smem = v != 0; return CK_OK;
        case CK_OPT_ROWS_IN_SMEM: o.rows_in_smem = v != 0; return CK_OK;
        case CK_OPT_TEST_BOUNDS_PROBE: o.bounds_probe = v != 0; return CK_OK;
        case CK_OPT_TILED: o.tiled = v != 0; return CK_OK;
        case CK_OPT_RECOMPUTE_STEPS:
            if (v < 0 || v > (1 << 30)) return fail(CK_ERR_INVALID_ARG, "recompute steps must be in [0, 2^30]");
            o.recompute_steps = (int)v;
            return CK_OK;
    }
    return fail(CK_ERR_INVALID_ARG, "unknown option %d", (int)opt);
}

int64_t ck_get_option(ck_option opt) {
    const Options &o = options();
    switch (opt) {
        case CK_OPT_PERSISTENT: return o.persistent;
        case CK_OPT_BARRIER_TIMEOUT_NS: return o.timeout_ns;
        case CK_OPT_TEST_BARRIER_EXTRA: return o.barrier_extra;
        case CK_OPT_GRAPH_IN_SMEM: return o.graph_in_smem;
        case CK_OPT_RECOMPUTE_STEPS: return o.recompute_steps;
        case CK_OPT_ROWS_IN_SMEM: return o.rows_in_smem;
        case CK_OPT_TEST_BOUNDS_PROBE: return o.bounds_probe;
        case CK_OPT_TILED: return o.tiled;
    }
    return -1;
}

ck_status ck_graph_create(const int64_t *src, const int64_t *dst, int64_t E, int64_t N,
                          const int64_t *input_nodes, int64_t n_in, void *stream,
                          ck_graph **out) {
    return ck_graph_create_flags(src, dst, E, N, input_nodes, n_in, 0u, stream, out);
}

ck_status ck_graph_create_flags(const int64_t *src, const int64_t *dst, int64_t E, int64_t N,
                                const int64_t *input_nodes, int64_t n_in, uint32_t flags,
                                void *stream, ck_graph **out) {
    if (!out) return fail(CK_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (flags & ~(uint32_t)(CK_GRAPH_EDGES_IN_HOST_MEMORY | CK_GRAPH_TILING))
        return fail(CK_ERR_INVALID_ARG, "unknown graph flag bits 0x%x", (unsigned)flags);
    if (N < 1 || N >= ((int64_t)1 << 31) - 1) return fail(CK_ERR_INVALID_ARG, "N must be in [1, 2^31 - 1)");
    if (E < 0 || E >= ((int64_t)1 << 31) - 1) return fail(CK_ERR_INVALID_ARG, "E must be in [0, 2^31 - 1)");
    if (n_in < 0 || n_in > N) return fail(CK_ERR_INVALID_ARG, "n_in must be in [0, N]");
    if (E > 0 && (!src || !dst)) return fail(CK_ERR_INVALID_ARG, "src or dst is NULL");
    if (n_in > 0 && !input_nodes) return fail(CK_ERR_INVALID_ARG, "input_nodes is NULL");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    int coop = 0;
    e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    if (!coop) return fail(CK_ERR_UNSUPPORTED, "device %d has no cooperative launch", dev);
    ck_graph *g = new (std::nothrow) ck_graph;
    if (!g) return fail(CK_ERR_OUT_OF_MEMORY, "host allocation failed");
    std::memset(g, 0, sizeof(*g));
    g->device = dev;
    g->num_sms = sms;
    g->N = N;
    g->E = E;
    g->n_in = n_in;
    ck_status st = build_graph(g, src, dst, input_nodes, flags, (cudaStream_t)stream);
    if (st != CK_OK) {
        char keep[sizeof(g_msg)];
        std::memcpy(keep, g_msg, sizeof(keep));
        ck_graph_destroy(g);
        std::memcpy(g_msg, keep, sizeof(keep));
        return st;
    }
    *out = g;
    return CK_OK;
}

ck_status ck_graph_destroy(ck_graph *g) {
    if (!g) return CK_OK;
    cudaDeviceSynchronize();
    int *dev_ptrs[] = {g->row_ptr, g->rowT_ptr, g->slot};
    for (int *p : dev_ptrs)
        if (p) cudaFree(p);
    int *edge_ptrs[] = {g->col, g->perm, g->colT, g->permT, g->rowid, g->rowidT};
    for (int *p : edge_ptrs)
        if (p) g->edges_in_host ? cudaFreeHost(p) : cudaFree(p);
    for (int d = 0; d < 2; ++d)
        for (int v = 0; v < 3; ++v)
            if (g->piece[d][v]) cudaFree(g->piece[d][v]);
    for (int d = 0; d < 2; ++d) {
        Tiled &t = g->tiled[d];
        for (int *p : {t.meta, t.ptr})
            if (p) cudaFree(p);
        for (int *p : {t.col, t.perm, t.rowid})
            if (p) g->edges_in_host ? cudaFreeHost(p) : cudaFree(p);
    }
    delete g;
    return CK_OK;
}

ck_status ck_graph_info(const ck_graph *g, int64_t *N, int64_t *E, int64_t *n_in) {
    if (!g) return fail(CK_ERR_INVALID_ARG, "graph handle is NULL");
    if (N) *N = g->N;
    if (E) *E = g->E;
    if (n_in) *n_in = g->n_in;
    return CK_OK;
}

ck_status ck_graph_memory(const ck_graph *g, size_t *device_bytes, size_t *host_bytes) {
    if (!g) return fail(CK_ERR_INVALID_ARG, "graph handle is NULL");
    if (device_bytes) *device_bytes = g->device_bytes;
    if (host_bytes) *host_bytes = g->host_bytes;
    return CK_OK;
}

ck_status ck_graph_tiling(const ck_graph *g, int dir, int64_t info[8]) {
    if (!g || !info || dir < 0 || dir > 1) return fail(CK_ERR_INVALID_ARG, "bad graph, info or dir");
    const Tiled &t = g->tiled[dir];
    const int64_t ptr_len = t.C ? (int64_t)t.C * (g->N + t.G) : 0;
    const int64_t v[8] = {t.C, t.G, t.P, t.max_rows, t.max_fin, t.max_chunk, t.max_edges, ptr_len};
    for (int i = 0; i < 8; ++i) info[i] = v[i];
    return CK_OK;
}

ck_status ck_graph_export_tiling(const ck_graph *g, int dir, int32_t *meta, int32_t *ptr,
                                 int32_t *col, int32_t *perm, int32_t *rowid, void *stream) {
    if (!g || dir < 0 || dir > 1) return fail(CK_ERR_INVALID_ARG, "bad graph or dir");
    const Tiled &t = g->tiled[dir];
    if (t.C == 0) return fail(CK_ERR_INVALID_ARG, "direction %d has no tiling", dir);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t E = (size_t)g->E;
    struct {
        int32_t *dst;
        const int *src;
        size_t n;
    } cp[] = {{meta, t.meta, (size_t)t.P * kTileInts},
              {ptr, t.ptr, (size_t)t.C * (size_t)(g->N + t.G)},
              {col, t.col, E},
              {perm, t.perm, E},
              {rowid, t.rowid, E}};
    for (auto &c : cp) {
        if (!c.dst || c.n == 0) continue;
        cudaError_t e = cudaMemcpyAsync(c.dst, c.src, sizeof(int) * c.n, cudaMemcpyDefault, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (tiling export)");
    }
    return CK_OK;
}

ck_status ck_graph_export(const ck_graph *g, int32_t *row_ptr, int32_t *col, int32_t *perm,
                          int32_t *rowT_ptr, int32_t *colT, int32_t *permT, int32_t *slot,
                          void *stream) {
    ck_status st = check_graph(g);
    if (st != CK_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    struct {
        int32_t *dst;
        const int *src;
        int64_t n;
    } items[] = {{row_ptr, g->row_ptr, g->N + 1}, {col, g->col, g->E},     {perm, g->perm, g->E},
                 {rowT_ptr, g->rowT_ptr, g->N + 1}, {colT, g->colT, g->E}, {permT, g->permT, g->E},
                 {slot, g->slot, g->N}};
    for (auto &it : items) {
        if (!it.dst || it.n == 0) continue;
        cudaError_t e = cudaMemcpyAsync(it.dst, it.src, sizeof(int32_t) * it.n,
                                        g->edges_in_host ? cudaMemcpyDefault : cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (export)");
    }
    return CK_OK;
}

ck_status ck_workspace_size(const ck_graph *g, int64_t B, int64_t T, int64_t microsteps,
                            size_t *saved_bytes, size_t *scratch_bytes) {
    if (!g) return fail(CK_ERR_INVALID_ARG, "graph handle is NULL");
    Plan p;
    ck_status st = make_plan(g, B, T, microsteps, &p);
    if (st != CK_OK) return st;
    if (saved_bytes) *saved_bytes = p.saved_bytes;
    if (scratch_bytes) *scratch_bytes = p.scratch_bytes;
    return CK_OK;
}

ck_status ck_forward(const ck_graph *g, const float *edge_values, const float *leak,
                     const float *bias, const float *drives, const float *state0, int64_t B,
                     int64_t T, int64_t microsteps, float *states_out, void *saved,
                     size_t saved_bytes, void *scratch, size_t scratch_bytes, void *stream) {
    g_launches = 0;
    ck_status st = check_graph(g);
    if (st != CK_OK) return st;
    Plan p;
    st = make_plan(g, B, T, microsteps, &p);
    if (st != CK_OK) return st;
    if ((g->E > 0 && !edge_values) || !leak || !bias || !state0 || !states_out || !saved ||
        !scratch || (g->n_in > 0 && !drives))
        return fail(CK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (misaligned(saved) || misaligned(scratch))
        return fail(CK_ERR_INVALID_ARG, "saved and scratch must be 32-byte aligned");
    if (saved_bytes < p.saved_bytes || scratch_bytes < p.scratch_bytes)
        return fail(CK_ERR_WORKSPACE, "workspace too small: saved %zu < %zu or scratch %zu < %zu",
                    saved_bytes, p.saved_bytes, scratch_bytes, p.scratch_bytes);
    FwdIO io{edge_values, leak, bias, drives, state0, states_out, (float *)saved, scratch};
    return launch_forward(g, p, io, (cudaStream_t)stream, &g_launches);
}

ck_status ck_workspace_size_recompute(const ck_graph *g, int64_t B, int64_t T,
                                      int64_t microsteps, size_t *ckpt_bytes,
                                      size_t *scratch_bytes) {
    if (!g) return fail(CK_ERR_INVALID_ARG, "graph handle is NULL");
    Plan p;
    ck_status st = make_plan(g, B, T, microsteps, &p);
    if (st != CK_OK) return st;
    if (ckpt_bytes) *ckpt_bytes = p.ckpt_bytes;
    if (scratch_bytes) *scratch_bytes = p.scratch_bytes_rc;
    return CK_OK;
}

ck_status ck_forward_checkpointed(const ck_graph *g, const float *edge_values,
                                  const float *leak, const float *bias, const float *drives,
                                  const float *state0, int64_t B, int64_t T,
                                  int64_t microsteps, float *states_out, void *ckpt,
                                  size_t ckpt_bytes, void *scratch, size_t scratch_bytes,
                                  void *stream) {
    g_launches = 0;
    ck_status st = check_graph(g);
    if (st != CK_OK) return st;
    Plan p;
    st = make_plan(g, B, T, microsteps, &p);
    if (st != CK_OK) return st;
    if ((g->E > 0 && !edge_values) || !leak || !bias || !state0 || !states_out || !ckpt ||
        !scratch || (g->n_in > 0 && !drives))
        return fail(CK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (misaligned(ckpt) || misaligned(scratch))
        return fail(CK_ERR_INVALID_ARG, "ckpt and scratch must be 32-byte aligned");
    if (ckpt_bytes < p.ckpt_bytes || scratch_bytes < p.scratch_bytes_rc)
        return fail(CK_ERR_WORKSPACE, "workspace too small: ckpt %zu < %zu or scratch %zu < %zu",
                    ckpt_bytes, p.ckpt_bytes, scratch_bytes, p.scratch_bytes_rc);
    FwdIO io{edge_values, leak, bias, drives, state0, states_out, (float *)ckpt, scratch};
    return launch_forward_ckpt(g, p, io, (cudaStream_t)stream, &g_launches);
}

ck_status ck_backward_recompute(const ck_graph *g, const float *edge_values, const float *leak,
                                const float *bias, const float *drives, int64_t B, int64_t T,
                                int64_t microsteps, const void *ckpt, size_t ckpt_bytes,
                                const float *d_states, float *d_edge_values, float *d_leak,
                                float *d_bias, float *d_drives, float *d_state0, void *scratch,
                                size_t scratch_bytes, void *stream) {
    g_launches = 0;
    ck_status st = check_graph(g);
    if (st != CK_OK) return st;
    Plan p;
    st = make_plan(g, B, T, microsteps, &p);
    if (st != CK_OK) return st;
    if ((g->E > 0 && (!edge_values || !d_edge_values)) || !leak || !bias || !ckpt || !d_states ||
        !d_leak || !d_bias || !d_state0 || !scratch || (g->n_in > 0 && (!drives || !d_drives)))
        return fail(CK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (misaligned(ckpt) || misaligned(scratch))
        return fail(CK_ERR_INVALID_ARG, "ckpt and scratch must be 32-byte aligned");
    if (ckpt_bytes < p.ckpt_bytes || scratch_bytes < p.scratch_bytes_rc)
        return fail(CK_ERR_WORKSPACE, "workspace too small: ckpt %zu < %zu or scratch %zu < %zu",
                    ckpt_bytes, p.ckpt_bytes, scratch_bytes, p.scratch_bytes_rc);
    RcIO io{edge_values, leak, bias, drives, (const float *)ckpt, d_states, d_edge_values,
            d_leak, d_bias, d_drives, d_state0, scratch};
    return launch_backward_recompute(g, p, io, (cudaStream_t)stream, &g_launches);
}

ck_status ck_backward(const ck_graph *g, const float *edge_values, const float *leak, int64_t B,
                      int64_t T, int64_t microsteps, const void *saved, size_t saved_bytes,
                      const float *d_states, float *d_edge_values, float *d_leak,
                      float *d_bias, float *d_drives, float *d_state0, void *scratch,
                      size_t scratch_bytes, void *stream) {
    g_launches = 0;
    ck_status st = check_graph(g);
    if (st != CK_OK) return st;
    Plan p;
    st = make_plan(g, B, T, microsteps, &p);
    if (st != CK_OK) return st;
    if ((g->E > 0 && (!edge_values || !d_edge_values)) || !leak || !saved || !d_states ||
        !d_leak || !d_bias || !d_state0 || !scratch || (g->n_in > 0 && !d_drives))
        return fail(CK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (misaligned(saved) || misaligned(scratch))
        return fail(CK_ERR_INVALID_ARG, "saved and scratch must be 32-byte aligned");
    if (saved_bytes < p.saved_bytes || scratch_bytes < p.scratch_bytes)
        return fail(CK_ERR_WORKSPACE, "workspace too small: saved %zu < %zu or scratch %zu < %zu",
                    saved_bytes, p.saved_bytes, scratch_bytes, p.scratch_bytes);
    BwdIO io{edge_values, leak, (const float *)saved, d_states, d_edge_values, d_leak, d_bias,
             d_drives, d_state0, scratch};
    return launch_backward(g, p, io, (cudaStream_t)stream, &g_launches);
}

ck_status ck_query_status(const void *scratch, void *stream) {
    if (!scratch) return fail(CK_ERR_INVALID_ARG, "scratch is NULL");
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "pending CUDA error");
    int word = 0;
    e = cudaMemcpy(&word, (const char *)scratch + kStatusOffset, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy (status word)");
    if (word == kDevTimeout) return fail(CK_ERR_TIMEOUT, "a device-side wait timed out");
    if (word == kDevBounds)
        return fail(CK_ERR_INTERNAL, "an index out of bounds was caught and its access skipped "
                                     "(bounds-checked build)");
    if (word != kDevOk) return fail(CK_ERR_INTERNAL, "device status word %d", word);
    return CK_OK;
}

}  // extern "C"
