/*
 * ck.h -- C ABI of libck: training passes of a leaky-tanh recurrence over a
 * fixed sparse directed graph, for one NVIDIA GB300 (sm_103a).
 *
 * The method (connectome-kernels page, intro): every node i holds one scalar
 * state per batch column; one microstep computes
 *     proposal_i = tanh( sum_j W_ij h_j + drive_i + bias_i )
 *     h_i       <- (1 - leak_i) h_i + leak_i * proposal_i
 * and `microsteps` microsteps run per input step.  W is sparse with a fixed
 * pattern and one trainable scalar per (src, dst) edge; the drive enters only
 * at a designated set of input nodes.  Readings this library takes where the
 * page leaves a step open:
 *   - an edge src[e] -> dst[e] carries W[dst][src] = edge_values[e]; repeated
 *     (src, dst) pairs add up; self-loops are allowed;
 *   - all nodes of a microstep read the state left by the previous microstep;
 *   - the drive of input step t is added in each of its microsteps;
 *   - the output of input step t is the state after its last microstep;
 *   - leak is used exactly as passed (the caller squashes it, e.g. sigmoid).
 *
 * Conventions for every call below:
 *   - Pointers marked (device) are CUDA device pointers on the current device;
 *     arrays are dense, row-major, with the shapes given.  Nothing is retained
 *     after a call returns except by ck_graph_create.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work on it and return without waiting, except
 *     where a call says it synchronises.
 *   - Every call returns a ck_status; none aborts the process or throws.  On
 *     failure ck_last_error_message() gives a one-line reason (per thread).
 *   - There is no CPU fallback: without a usable CUDA device, calls fail with
 *     CK_ERR_CUDA.
 *   - Memory: the library allocates device memory only inside
 *     ck_graph_create (the graph arrays, freed by ck_graph_destroy) and
 *     temporarily during that call.  The caller owns and allocates `saved` and
 *     `scratch`, sized by ck_workspace_size.
 */
#ifndef CK_H
#define CK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CK_OK = 0,
    CK_ERR_INVALID_ARG = 1,    /* bad size, null pointer, index out of range, duplicate input node */
    CK_ERR_CUDA = 2,           /* a CUDA runtime call failed (message names it) */
    CK_ERR_OUT_OF_MEMORY = 3,  /* device allocation failed inside ck_graph_create */
    CK_ERR_TIMEOUT = 4,        /* a bounded device-side wait gave up (see ck_query_status) */
    CK_ERR_WORKSPACE = 5,      /* saved or scratch smaller than ck_workspace_size asks */
    CK_ERR_INTERNAL = 6,       /* an internal invariant failed */
    CK_ERR_UNSUPPORTED = 7     /* shape outside what this build supports (message says which) */
} ck_status;

/* Opaque graph handle; owned by the library. */
typedef struct ck_graph ck_graph;

/*
 * ck_graph_create -- build the graph once (connectome-kernels page, "Use":
 * SparseGraph(src, dst, num_nodes, input_nodes); "Design notes": a transposed
 * compressed-row copy serves the state gradient; "Use": edge parameters stay in
 * the caller's order and the internal permutation is invisible).
 *
 *   src, dst      (device) int64[E]; edge e runs src[e] -> dst[e]; 0 <= src, dst < N
 *   E             number of edges, 0 <= E < 2^31
 *   N             number of nodes, 1 <= N < 2^31
 *   input_nodes   (device) int64[n_in]; distinct node ids; drive row k enters
 *                 node input_nodes[k]; may be NULL when n_in == 0
 *   n_in          0 <= n_in <= N
 *   out           (host) receives the new handle; set to NULL on failure
 *
 * Builds on the GPU, with the library's own kernels, the rows keyed by dst
 * (row_ptr[N+1], col = src in row order, perm = caller's edge id of each row
 * position) and the same keyed by src (rowT_ptr, colT = dst, permT), both by a
 * stable sort (equal keys keep ascending edge id), and slot[N] (k where
 * input_nodes[k] = i, else -1).  Validates every index and input-node
 * uniqueness on the device; synchronises `stream` to read the result.
 * Errors: CK_ERR_INVALID_ARG (sizes, null pointers, an index out of range, a
 * repeated input node), CK_ERR_OUT_OF_MEMORY, CK_ERR_CUDA.
 */
ck_status ck_graph_create(const int64_t *src, const int64_t *dst, int64_t E, int64_t N,
                          const int64_t *input_nodes, int64_t n_in, void *stream,
                          ck_graph **out);

/* Graph flags for ck_graph_create_flags. */
typedef enum {
    CK_GRAPH_EDGES_IN_HOST_MEMORY = 1, /* the arrays indexed by edge (col, perm and each edge's
                                          row, both directions: 24 bytes per edge) go to pinned
                                          host memory that the kernels read in place over the
                                          CPU-GPU link (NVLink-C2C on a Grace-Blackwell node);
                                          row pointers, slots and piece tables (O(N)) stay in
                                          device memory.  Results are bitwise those of a
                                          device-resident graph; speed depends on whether the
                                          CTAs' slices fit in shared memory (read once per call)
                                          or stream every microstep.  The connectome runtime
                                          page ("Why this runtime") makes graph residency an
                                          explicit choice in the same way. */
    CK_GRAPH_TILING = 2                /* also build the shared-memory tilings (ck_graph_tiling)
                                          that the tiled kernels (CK_OPT_TILED) need: three more
                                          int32 arrays per edge and direction, built on the host.
                                          Without it a graph has no tiling and every call runs
                                          the L2-gather kernels. */
} ck_graph_flag;

/*
 * ck_graph_create_flags -- ck_graph_create with flags (a bitwise OR of
 * ck_graph_flag values; 0 is ck_graph_create).  Errors: as ck_graph_create,
 * plus CK_ERR_INVALID_ARG for an unknown flag bit and CK_ERR_UNSUPPORTED when
 * pinned host memory is not mapped at the same address on the device.
 */
ck_status ck_graph_create_flags(const int64_t *src, const int64_t *dst, int64_t E, int64_t N,
                                const int64_t *input_nodes, int64_t n_in, uint32_t flags,
                                void *stream, ck_graph **out);

/* Frees the handle and its arrays (synchronises the device first).  NULL is a no-op. */
ck_status ck_graph_destroy(ck_graph *g);

/* Sizes recorded in the handle (any output pointer may be NULL). */
ck_status ck_graph_info(const ck_graph *g, int64_t *N, int64_t *E, int64_t *n_in);

/* Memory the handle holds until ck_graph_destroy: device bytes and pinned host
 * bytes (nonzero with CK_GRAPH_EDGES_IN_HOST_MEMORY).  Either pointer may be NULL. */
ck_status ck_graph_memory(const ck_graph *g, size_t *device_bytes, size_t *host_bytes);

/*
 * ck_graph_export -- copy the graph arrays out, for tests: (device) int32
 * row_ptr[N+1], col[E], perm[E], rowT_ptr[N+1], colT[E], permT[E], slot[N].
 * Any pointer may be NULL to skip that array.  Asynchronous on `stream`.
 */
ck_status ck_graph_export(const ck_graph *g, int32_t *row_ptr, int32_t *col, int32_t *perm,
                          int32_t *rowT_ptr, int32_t *colT, int32_t *permT, int32_t *slot,
                          void *stream);

/*
 * ck_graph_tiling -- the shared-memory tiling of one direction (dir 0: rows
 * keyed by dst, the forward; 1: keyed by src, the backward), which the
 * kernels use when the padded batch is at most 32 columns (connectome-kernels
 * page, "Design notes": the state stored [N, B] is gathered row by row; here a
 * CTA gathers from a chunk of the state rows held in its shared memory).  The
 * column nodes are cut into C chunks and the rows into G blocks; CTA
 * t = g * C + j owns cell (g, j): the edges of block g whose column lies in
 * chunk j, in row order.  info receives {C, G, P = G * C, most rows in a block,
 * most rows a CTA finishes, most nodes in a chunk, most edges in a cell, length
 * of the row-pointer array}; all zero when the direction has no tiling (a
 * graph created without CK_GRAPH_TILING, or one whose state rows do not fit
 * eight CTAs' shared memory).
 */
ck_status ck_graph_tiling(const ck_graph *g, int dir, int64_t info[8]);

/*
 * ck_graph_export_tiling -- copy one direction's tiling out, for tests:
 * (device) int32 meta[P][12] (per CTA: first row, rows, first and end edge,
 * chunk's first node, chunk nodes, offset of its row pointers, first and end
 * row it finishes relative to the block, chunk, block, 0), ptr[ptr length]
 * (per CTA, rows + 1 positions into the edge arrays), col[E] (column node minus
 * its chunk's first node), perm[E] (caller's edge id), rowid[E] (row node).
 * Any pointer may be NULL.  Errors: CK_ERR_INVALID_ARG (dir, no tiling).
 */
ck_status ck_graph_export_tiling(const ck_graph *g, int dir, int32_t *meta, int32_t *ptr,
                                 int32_t *col, int32_t *perm, int32_t *rowid, void *stream);

/*
 * ck_workspace_size -- bytes of the two caller-owned buffers for batch B,
 * T input steps and `microsteps` microsteps per step, on the current device.
 *   saved_bytes    activations kept from ck_forward for ck_backward: the state
 *                  and the proposal tanh(pre-activation) after every microstep,
 *                  plus the initial state (connectome-kernels page, "Design
 *                  notes": 2 x T x M x N x B floats saved; the proposal stands in
 *                  for the pre-activation, which the backward needs only through
 *                  its tanh), rows padded to Bp floats: B rounded up to 8, to 32
 *                  when 16 < B <= 32, to 16 above 256
 *   scratch_bytes  temporary device memory for one ck_forward or ck_backward
 *                  call; one scratch buffer may serve both, but two calls that
 *                  run at the same time need two buffers
 * Both depend on the device's SM count: query on the device that will run the calls.
 * Errors: CK_ERR_INVALID_ARG (B, T, microsteps < 1), CK_ERR_UNSUPPORTED (B > 512,
 * sizes whose element offsets overflow the index types, or a graph whose
 * pieces finish more rows than a CTA's shared memory holds tables for: 24
 * bytes per row, about 4,000 rows per piece, i.e. about 1.2 million nodes at a
 * few edges per node on 152 SMs).
 */
ck_status ck_workspace_size(const ck_graph *g, int64_t B, int64_t T, int64_t microsteps,
                            size_t *saved_bytes, size_t *scratch_bytes);

/*
 * ck_forward -- run the whole window of T input steps x microsteps
 * (connectome-kernels page, intro equations; "Use": sparse_recurrence returns
 * out[T, B, N], the node states after each input step).
 *
 *   edge_values  (device) float[E], the caller's edge order
 *   leak, bias   (device) float[N]
 *   drives       (device) float[T][n_in][B]; may be NULL when n_in == 0
 *   state0       (device) float[B][N]
 *   states_out   (device) float[T][B][N], overwritten
 *   saved        (device) >= saved_bytes, 32-byte aligned; filled for ck_backward
 *   scratch      (device) >= scratch_bytes, 32-byte aligned (the kernels gather rows
 *                with 32-byte loads)
 * Runs as one persistent cooperative kernel with bounded grid-wide barriers
 * between microsteps.  Asynchronous.  A device-side wait that times out makes
 * the kernel stop early and is reported by ck_query_status.
 * Errors: CK_ERR_INVALID_ARG, CK_ERR_WORKSPACE, CK_ERR_UNSUPPORTED, CK_ERR_CUDA.
 */
ck_status ck_forward(const ck_graph *g, const float *edge_values, const float *leak,
                     const float *bias, const float *drives, const float *state0,
                     int64_t B, int64_t T, int64_t microsteps, float *states_out,
                     void *saved, size_t saved_bytes, void *scratch, size_t scratch_bytes,
                     void *stream);

/*
 * ck_backward -- gradients of L = sum_t <d_states[t], states_out[t]> with
 * respect to all five inputs of ck_forward (connectome-kernels page, intro:
 * three backward parts -- elementwise terms with per-node reductions, the
 * transposed sparse product for the state gradient, a per-edge dot product
 * over the batch for the edge gradient; "Use": differentiable in every
 * argument).
 *
 *   edge_values, leak   the same values given to ck_forward
 *   saved               (device) as filled by ck_forward with the same g, B, T, microsteps
 *   d_states            (device) float[T][B][N]
 *   d_edge_values       (device) float[E], caller's edge order, overwritten
 *   d_leak, d_bias      (device) float[N], overwritten
 *   d_drives            (device) float[T][n_in][B], overwritten; may be NULL when n_in == 0
 *   d_state0            (device) float[B][N], overwritten
 *   scratch             (device) >= scratch_bytes
 * Gradients are written, not accumulated into.  Asynchronous.
 * Errors: as ck_forward.
 */
ck_status ck_backward(const ck_graph *g, const float *edge_values, const float *leak,
                      int64_t B, int64_t T, int64_t microsteps,
                      const void *saved, size_t saved_bytes, const float *d_states,
                      float *d_edge_values, float *d_leak, float *d_bias, float *d_drives,
                      float *d_state0, void *scratch, size_t scratch_bytes, void *stream);

/*
 * Recomputing variant: the forward keeps only the state after every input
 * step (T + 1 checkpoints instead of 2 T M + 1 saved rows), and the backward
 * recomputes the microsteps of a window of K input steps (CK_OPT_RECOMPUTE_STEPS,
 * about sqrt(T) by default) from the window's first checkpoint before
 * differentiating them.  The pages save every microstep's state and
 * pre-activation ("Design notes": 2 x T x M x N x B floats); this trades one
 * more forward pass (and two launches per window) for T + 1 + 2 K M + 1 rows
 * instead of 2 T M + 1.  Results equal ck_forward / ck_backward's bit for bit,
 * for every K.
 *
 * ck_workspace_size_recompute -- bytes of the checkpoints and of the scratch
 *   buffer for the two calls below (the scratch holds a window of K M + 1
 *   states and K M proposals on top of ck_workspace_size's scratch).
 *   Errors: as ck_workspace_size.
 */
ck_status ck_workspace_size_recompute(const ck_graph *g, int64_t B, int64_t T,
                                      int64_t microsteps, size_t *ckpt_bytes,
                                      size_t *scratch_bytes);

/*
 * ck_forward_checkpointed -- ck_forward that writes, instead of `saved`, the
 * state after every input step:
 *   ckpt   (device) >= ckpt_bytes, 32-byte aligned: float[T+1][N][Bp], Bp = B
 *          rounded up as in `saved`; ckpt[0] is state0 transposed
 * Other arguments, ownership and errors as ck_forward (scratch sized by
 * ck_workspace_size_recompute).
 */
ck_status ck_forward_checkpointed(const ck_graph *g, const float *edge_values,
                                  const float *leak, const float *bias, const float *drives,
                                  const float *state0, int64_t B, int64_t T,
                                  int64_t microsteps, float *states_out, void *ckpt,
                                  size_t ckpt_bytes, void *scratch, size_t scratch_bytes,
                                  void *stream);

/*
 * ck_backward_recompute -- ck_backward from checkpoints: for windows [t, t1)
 * of K input steps from the top (the lowest may be shorter) it recomputes
 * microsteps tM .. t1 M - 1 from ckpt[t] (one launch) and runs the backward
 * microsteps of steps t .. t1 - 1 (a second launch).  Needs bias and drives
 * besides ck_backward's inputs, since it reruns the forward.
 *   ckpt   (device) as filled by ck_forward_checkpointed with the same g, B, T,
 *          microsteps and inputs
 * Other arguments, ownership and errors as ck_backward (scratch sized by
 * ck_workspace_size_recompute).
 */
ck_status ck_backward_recompute(const ck_graph *g, const float *edge_values, const float *leak,
                                const float *bias, const float *drives, int64_t B, int64_t T,
                                int64_t microsteps, const void *ckpt, size_t ckpt_bytes,
                                const float *d_states, float *d_edge_values, float *d_leak,
                                float *d_bias, float *d_drives, float *d_state0, void *scratch,
                                size_t scratch_bytes, void *stream);

/*
 * ck_sgd_update -- param <- param - lr * grad over n floats (device arrays,
 * both owned by the caller), so that a whole training step -- ck_forward,
 * ck_backward, then this update of edge_values, leak and bias -- runs on the
 * device and can be captured as one CUDA graph (TrainKernel page, intro: a
 * captured step holds the forward, the gradients and the SGD update).
 * Asynchronous on `stream`.  Errors: CK_ERR_INVALID_ARG (n < 0, NULL pointer
 * with n > 0), CK_ERR_CUDA.
 */
ck_status ck_sgd_update(float *param, const float *grad, int64_t n, float lr, void *stream);

/*
 * ck_adam_update -- one Adam step (Kingma and Ba, "Adam: A Method for
 * Stochastic Optimization", Algorithm 1) over n floats, the optional
 * optimizer of a captured training step:
 *     m <- beta1 m + (1 - beta1) grad;  v <- beta2 v + (1 - beta2) grad^2
 *     param <- param - lr (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
 * with t = *step, a (device) int64 the caller keeps (t >= 1; advance it with
 * ck_step_advance before each step, so that a captured graph advances its own
 * count on every replay).  param, m, v: (device) float[n], updated in place;
 * grad: (device) float[n]; m and v start at zero.  Asynchronous on `stream`.
 * Errors: CK_ERR_INVALID_ARG (n < 0, betas outside [0, 1), eps <= 0, lr not a
 * number, NULL pointer), CK_ERR_CUDA.
 *
 * ck_step_advance -- *step += 1 on the device (one thread), on `stream`.
 */
ck_status ck_adam_update(float *param, const float *grad, float *m, float *v, int64_t n, float lr,
                         float beta1, float beta2, float eps, const int64_t *step, void *stream);
ck_status ck_step_advance(int64_t *step, void *stream);

/*
 * ck_forward_static_scratch -- ck_forward without a scratch buffer: the
 * temporary workspace comes from a 32 MiB array of device memory compiled into
 * the library.  The pages have no counterpart for this call; it exists for
 * callers that cannot allocate device memory when they run the forward, such
 * as a plugin inside a host application whose memory manager owns the device
 * and refuses allocations it did not make, or a control loop that must not
 * allocate once running.  The caller still passes every input and output
 * (including `saved`, sized by ck_workspace_size) with the meanings of
 * ck_forward; `saved` then feeds ck_backward as usual.
 *
 *   - Allocates nothing and calls no allocating routine.
 *   - Every GPU that loads the library holds the 32 MiB array until the process
 *     exits.  Each call made outside a stream capture looks up the array's
 *     device address (cudaGetSymbolAddress) with the call's device current, so
 *     a reset of the device's primary context, which moves the array, is
 *     followed; a call inside a capture reuses the last address looked up on
 *     that device, so make a first call on each device before any capture, and
 *     none across a context reset inside a capture.
 *   - All calls share the one array: two calls whose work overlaps on the GPU
 *     (different streams, different threads) race and corrupt each other.
 *     Each call clears the words that must start at zero; the rest of the
 *     array keeps the previous call's contents until overwritten.
 *   - Shapes whose forward workspace exceeds the array (control words, one
 *     carry row per CTA, one float per edge and per padded node-batch element)
 *     are refused with CK_ERR_UNSUPPORTED and a message giving both sizes.
 *   - A device-side wait that times out makes the kernel stop early; this call
 *     still returns CK_OK (it does not wait for the kernel), so check
 *     ck_query_status_static before using the outputs or `saved`.
 * Errors: CK_ERR_INVALID_ARG, CK_ERR_WORKSPACE, CK_ERR_UNSUPPORTED, CK_ERR_CUDA.
 */
ck_status ck_forward_static_scratch(const ck_graph *g, const float *edge_values,
                                    const float *leak, const float *bias, const float *drives,
                                    const float *state0, int64_t B, int64_t T,
                                    int64_t microsteps, float *states_out, void *saved,
                                    size_t saved_bytes, void *stream);

/*
 * ck_query_status_static -- ck_query_status for ck_forward_static_scratch:
 * synchronise `stream` and report whether the last static-scratch forward on
 * the current device finished every device-side wait (CK_OK), or a bounded
 * wait gave up (CK_ERR_TIMEOUT: that forward stopped early; its outputs and
 * `saved` are not valid).  Reads the status word out of the static array with
 * cudaMemcpyFromSymbol; allocates nothing.  Also reports pending CUDA errors.
 */
ck_status ck_query_status_static(void *stream);

/*
 * ck_query_status -- synchronise `stream` and report whether the last
 * ck_forward / ck_backward that used `scratch` finished every device-side wait:
 * CK_OK, or CK_ERR_TIMEOUT if a bounded wait gave up (its kernel then stopped
 * early and its outputs are not valid).  Also reports pending CUDA errors.
 */
ck_status ck_query_status(const void *scratch, void *stream);

/* Tuning and test switches, process-wide; take effect on the next call. */
typedef enum {
    CK_OPT_PERSISTENT = 0,          /* 1 (default): one launch per call; 0: one launch per microstep */
    CK_OPT_BARRIER_TIMEOUT_NS = 1,  /* bound on any device-side wait (default 4e9 ns) */
    CK_OPT_TEST_BARRIER_EXTRA = 2,  /* test hook: barriers wait for this many extra arrivals
                                       that never come, so every wait runs out (default 0) */
    CK_OPT_GRAPH_IN_SMEM = 3,       /* 1 (default): keep each CTA's slice of the graph in
                                       shared memory when it fits; 0: always stream it */
    CK_OPT_RECOMPUTE_STEPS = 4,     /* input steps K one recomputation window spans
                                       (ck_workspace_size_recompute and the two calls
                                       after it must see the same value); 0 (default):
                                       round(sqrt(T)); clamped to [1, T] */
    CK_OPT_ROWS_IN_SMEM = 5,        /* 1 (default): keep each CTA's per-row partial sums in
                                       shared memory when they fit; 0: always in the
                                       scratch buffer (a test switch: results are bitwise
                                       the same either way) */
    CK_OPT_TEST_BOUNDS_PROBE = 6,   /* test hook for the bounds-checked build of the library
                                       (compiled with -DCK_DEBUG_BOUNDS, which checks every
                                       gathered row, table and carry index on the device and
                                       reports a bad one through ck_query_status as
                                       CK_ERR_INTERNAL instead of making the access): 1 makes
                                       each recurrence kernel check one deliberately
                                       out-of-range index, never used for an access, so a test
                                       sees the report; no effect in the ordinary build
                                       (default 0) */
    CK_OPT_TILED = 7                /* 1: when the graph has a shared-memory tiling
                                       (created with CK_GRAPH_TILING and small enough;
                                       ck_graph_tiling) and the padded batch is at most 32
                                       columns, run the tiled kernels; 0 (default): always
                                       the L2-gather kernels.  ck_workspace_size and the
                                       calls after it must see the same value */
} ck_option;

ck_status ck_set_option(ck_option opt, int64_t value);
int64_t ck_get_option(ck_option opt);

/* Number of kernel launches the last ck_forward / ck_backward on this thread enqueued. */
int64_t ck_last_launch_count(void);

/*
 * Bandwidth probes (no counterpart on the pages: they measure the L2 rates
 * that bound the recurrence kernels, which the device does not report).
 *   ck_probe_read    reads `bytes` of (device) `buf` (16-byte aligned) `reps`
 *                    times with 16-byte L2-cached loads.
 *   ck_probe_gather  reads nidx whole rows rows[idx[k]][0:row_floats] of a
 *                    (device) float[nrows][row_floats] table, row_floats in
 *                    {8, 16, 32, 64, 128}; every idx[k] must lie in [0, nrows)
 *                    (the kernel does not check it).
 * `sink` is a (device) float[1] the kernels may write.  Asynchronous; time
 * them with events on `stream`.
 */
ck_status ck_probe_read(const void *buf, size_t bytes, int64_t reps, float *sink, void *stream);
ck_status ck_probe_gather(const float *rows, int64_t nrows, int64_t row_floats,
                          const int32_t *idx, int64_t nidx, float *sink, void *stream);
/*
 * ck_probe_read_shape -- ck_probe_read with the load shape chosen: loads of
 * `load_bytes` bytes (16, or 32: the 256-bit vector load of sm_100 and later),
 * `depth` of them in flight per thread (2, 4, 8, or 16 with at most 512
 * threads), CTAs of `threads` threads (128, 256, 512 or 1024), `ctas_per_sm`
 * CTAs per SM (threads x ctas_per_sm <= 2048); `buf` 32-byte aligned.  A sweep
 * over shapes gives the highest L2 read rate of the device, the denominator of
 * the L2 roofline.  Errors: CK_ERR_INVALID_ARG for a shape outside those sets.
 */
ck_status ck_probe_read_shape(const void *buf, size_t bytes, int64_t reps, int64_t load_bytes,
                              int64_t depth, int64_t threads, int64_t ctas_per_sm, float *sink,
                              void *stream);

/*
 * ck_probe_grid_barrier -- times one grid-barrier scheme on its own (no
 * counterpart on the pages: it measures the latency under every microstep of
 * the persistent kernels).  `ctas` co-resident CTAs of 256 threads each cross
 * `crossings` barriers; before each crossing every CTA writes rows_per_cta
 * (0..64) rows of 32 floats to (device) `rows`, float[ctas * rows_per_cta * 32]
 * (may be NULL when rows_per_cta is 0).  `words` is (device)
 * uint32[CK_PROBE_BARRIER_WORDS] and `status` (device) int32[1]; the call
 * clears both on `stream`.  `cluster` is 1, or 2, 4 or 8 for the cluster
 * schemes (then ctas must be a multiple of it).  Every wait gives up after
 * CK_OPT_BARRIER_TIMEOUT_NS and sets *status to 1, and all CTAs then stop.
 * Asynchronous: time it with events on `stream`, then read *status.
 * Errors: CK_ERR_INVALID_ARG for an argument outside these sets,
 * CK_ERR_UNSUPPORTED when the CTAs cannot all be resident at once.
 */
#define CK_PROBE_BARRIER_WORDS 16384
typedef enum {
    CK_BARRIER_COUNTER = 0,           /* the recurrence kernels' barrier: one release add per CTA
                                         on a counter, one thread per CTA polls it (acquire) */
    CK_BARRIER_COUNTER_RETURNING = 1, /* the add returns the count; the last CTA skips the poll */
    CK_BARRIER_COUNTER_RELAXED = 2,   /* relaxed polls, an acquire fence once the count is seen */
    CK_BARRIER_FLAG = 3,              /* the last CTA (returning add) writes a release flag that
                                         the others poll, apart from the counter */
    CK_BARRIER_FLAGS8 = 4,            /* as 3 with eight flag copies, each polled by 1/8 of the CTAs */
    CK_BARRIER_CLUSTER_SYNC = 5,      /* hardware cluster barrier, then one arrival per cluster */
    CK_BARRIER_CLUSTER_MBARRIER = 6   /* remote mbarrier arrivals on the cluster leader's shared
                                         memory (bounded waits), one arrival per cluster */
} ck_barrier_scheme;
ck_status ck_probe_grid_barrier(int64_t scheme, int64_t ctas, int64_t cluster, int64_t crossings,
                                int64_t rows_per_cta, float *rows, uint32_t *words, int32_t *status,
                                void *stream);

/*
 * ck_phase_profile_read -- the per-microstep phase times of the L2-gather
 * recurrence kernels (the tiled kernels keep none), kept only by the profiling build of this library (libck_prof.so,
 * compiled with -DCK_PHASE_PROFILE; every other build returns
 * CK_ERR_UNSUPPORTED without touching the device).  No counterpart on the
 * pages: it measures where a microstep's time goes.  Synchronises the device,
 * copies uint64 host[2][CK_PHASE_PROFILE_CTAS][CK_PHASE_PROFILE_WORDS] (index
 * 0 forward, 1 backward; then the CTA) and, with `clear`, zeroes the counters.
 * Per CTA, summed over microsteps and calls since the last clear
 * (%globaltimer ns): [0] part A (the gather); [1] part A and the CTA's sync
 * after it; [2] the finish (to its last warp); [3] the grid barrier, from
 * arrival to release, with the work issued inside its wait; [4] microsteps;
 * [5] barriers; [6] the SM of the last call; [7] rows << 32 | edges of
 * the CTA's piece.  The stamps add a CTA sync after the finish, so times are
 * close to, not equal to, the ordinary build's.  Errors: CK_ERR_INVALID_ARG
 * for a NULL or short buffer, CK_ERR_CUDA.
 */
#define CK_PHASE_PROFILE_CTAS 1024
#define CK_PHASE_PROFILE_WORDS 8
ck_status ck_phase_profile_read(uint64_t *host, int64_t words, int64_t clear);

const char *ck_status_string(ck_status s);
const char *ck_last_error_message(void);

#ifdef __cplusplus
}
#endif
#endif /* CK_H */
