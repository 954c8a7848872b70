// Internal declarations shared by the translation units of libck.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ck.h"

struct ck_graph {
    int device;
    int num_sms;
    int64_t N, E, n_in;
    int *row_ptr, *col, *perm;     // rows keyed by dst: col = src
    int *rowT_ptr, *colT, *permT;  // rows keyed by src: colT = dst
    int *slot;                     // slot[i] = k if input_nodes[k] == i, else -1
    int *rowid, *rowidT;           // row of each row-ordered edge (dst[perm[k]], src[permT[k]])
    // Per direction (0: rows keyed by dst, 1: keyed by src), with the work cut
    // into num_pieces(g) equal pieces of the merge path of (row ends, edges): the
    // most rows any piece finishes and the most edges any piece holds.
    //
    // One cut per finish pass size v (kPassRows[v] rows finished at once by a
    // CTA's warps): a weighted merge path, where a row end counts as w items
    // and w is chosen so that few pieces hold more rows than one pass
    // finishes.  piece[d][v][c * kPieceInts + j] for CTA c: {r0, nrows, e0,
    // e1, c_lo, publish} (first row, rows finished, edge range, first earlier
    // CTA whose carries reach row r0, whether the piece ends inside a row it
    // must publish).
    int max_rows[2][3], max_edges[2][3], row_weight[2][3];
    int *piece[2][3];
    // 1 when col, perm, rowid and their transposes live in pinned, mapped host
    // memory (the pointers above are then the device's view of it).
    int edges_in_host;
};

namespace ck {

constexpr int kPieceInts = 8;
// Shape of the recurrence kernels: kCtasPerSm CTAs of kThreads threads on
// every SM, the work cut into SMs x kCtasPerSm pieces.
constexpr int kCtasPerSm = 2;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
inline int num_pieces(const ck_graph *g) { return g->num_sms * kCtasPerSm; }
// Rows one finish pass of a CTA covers (kWarps warps, four (row,
// column-chunk) elements per lane), by padded batch width: index 0 for
// Bp <= 32, 1 for Bp <= 64, 2 above.
constexpr int kPassRows[3] = {4 * kWarps, 2 * kWarps, kWarps};
inline int pass_index(int Bp) { return Bp <= 32 ? 0 : (Bp <= 64 ? 1 : 2); }

// Per-thread error reporting used by every ABI entry point.
ck_status fail(ck_status s, const char *fmt, ...);
ck_status cuda_fail(cudaError_t e, const char *what);

// Graph build (graph.cu).  Fills g's device arrays; synchronises `stream`.
ck_status build_graph(ck_graph *g, const int64_t *src, const int64_t *dst,
                      const int64_t *input_nodes, uint32_t graph_flags, cudaStream_t stream);

// Device-side status words written by the recurrence kernels.
enum : int { kDevOk = 0, kDevTimeout = 1, kDevInternal = 2 };

// Control block at the start of scratch: the barrier counter and, on its own
// 128-byte line, the status word.
constexpr size_t kStatusOffset = 128;
constexpr size_t kCtrlBytes = 256;

// Shared-memory layout of one direction's kernel (byte offsets).
struct SmemLayout {
    int o_srp, o_prm, o_slot, o_grp, o_carry, o_rows, o_tile, o_cw, o_gst, o_dw;
    size_t bytes;
    bool graph;  // the CTA's slice of the graph lives in shared memory
    bool rows;   // row sums live in shared memory (else in global scratch)
    bool stage;  // finish operands staged in shared memory
    int o_st0, o_st1, o_st2, o_st3, o_st4, o_inp, o_acc;
};

// Launch description of one ck_forward / ck_backward call (recurrence.cu).
struct Plan {
    int N, E, n_in;
    int B, Bp, LPE, EPW, NC, T, M, S;
    int P;            // CTAs (kCtasPerSm per SM), one piece each
    int threads;      // threads per CTA
    int warps;        // warps per CTA
    int groups;       // lane groups per CTA (warps * EPW)
    int cap[2];       // bound on edges in one CTA's piece (0: forward rows, 1: transposed)
    int rows_cap[2];  // bound on rows one CTA touches, plus 2
    SmemLayout lay_fwd, lay_bwd;
    SmemLayout lay_bwd_flat;  // backward without staging or graph slices (recomputing windows)
    // scratch layout (byte offsets)
    size_t off_ctrl, ctrl_bytes;
    size_t off_carry;   // float [P][Bp]
    size_t off_wperm;   // float [E]
    size_t off_dwperm;  // float [E]
    size_t off_G;       // float [N][Bp]
    size_t off_da;      // float [2][N][Bp]
    size_t off_rowsum;  // float [N][Bp]
    size_t off_lacc;    // float2 [N][32] per-lane d_leak / d_bias partials
    size_t scratch_bytes;
    size_t saved_bytes; // float [(S+1) + S][N][Bp]
    // checkpointing forward / recomputing backward
    int rc_steps;             // input steps one recomputation window spans (K)
    size_t off_hwin;          // float [KM+1][N][Bp] window of states (first two: the forward's slots)
    size_t off_pwin;          // float [KM][N][Bp] window of proposals
    size_t scratch_bytes_rc;  // scratch for those calls (regular scratch plus the windows)
    size_t ckpt_bytes;        // float [T+1][N][Bp] states after every input step
};

// Process-wide switches (ck_set_option).  Atomic, so that a thread setting one
// while another plans a call reads either value, never a torn one.
struct Options {
    std::atomic<int> persistent{1};
    std::atomic<long long> timeout_ns{4000000000LL};
    std::atomic<int> barrier_extra{0};
    std::atomic<int> graph_in_smem{1};
    std::atomic<int> recompute_steps{0};  // 0: about sqrt(T)
};
Options &options();

ck_status make_plan(const ck_graph *g, int64_t B, int64_t T, int64_t M, Plan *p);

struct FwdIO {
    const float *w, *leak, *bias, *drives, *state0;
    float *out;
    float *saved;
    void *scratch;
};

struct RcIO {
    const float *w, *leak, *bias, *drives;
    const float *ckpt;
    const float *dout;
    float *dw, *dleak, *dbias, *ddrives, *dstate0;
    void *scratch;
};

struct BwdIO {
    const float *w, *leak;
    const float *saved;
    const float *dout;
    float *dw, *dleak, *dbias, *ddrives, *dstate0;
    void *scratch;
};

ck_status launch_forward(const ck_graph *g, const Plan &p, const FwdIO &io, cudaStream_t s,
                         int64_t *launches);
ck_status launch_backward(const ck_graph *g, const Plan &p, const BwdIO &io, cudaStream_t s,
                          int64_t *launches);
ck_status launch_forward_ckpt(const ck_graph *g, const Plan &p, const FwdIO &io, cudaStream_t s,
                              int64_t *launches);
ck_status launch_backward_recompute(const ck_graph *g, const Plan &p, const RcIO &io,
                                    cudaStream_t s, int64_t *launches);

}  // namespace ck
