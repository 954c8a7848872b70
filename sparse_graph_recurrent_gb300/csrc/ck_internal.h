// Internal declarations shared by the translation units of libck.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <stddef.h>
#include <stdint.h>

#include "../../include/ck.h"

namespace ck {
// Shared-memory tiling of one direction's rows (see ck_graph::tiled): the
// column nodes cut into C chunks, the rows into G blocks; CTA t = g * C + j
// owns cell (g, j), the edges of block g whose column lies in chunk j, in row
// order (within a row, the compressed-row order).  C == 0: no tiling.
struct Tiled {
    int C, G, P;    // chunks, row blocks, CTAs (G * C)
    int max_rows;   // most rows in a block
    int max_fin;    // most rows one CTA finishes (a block's rows split over its C CTAs)
    int max_chunk;  // most nodes in a chunk
    int max_edges;  // most edges in a cell
    // per CTA, kTileInts ints: {r0, nrows, e0, e1, chunk's first node, chunk
    // nodes, offset of the cell's row pointers in ptr, first and end row it
    // finishes (block-relative), chunk j, block g}
    int *meta;
    int *ptr;    // cell row pointers: nrows + 1 entries per CTA, positions in col/perm/rowid
    int *col;    // [E] column node minus its chunk's first node
    int *perm;   // [E] caller's edge id
    int *rowid;  // [E] row node
};
constexpr int kTileInts = 12;
}  // namespace ck

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
    // bytes the handle holds: device memory, and pinned host memory
    size_t device_bytes, host_bytes;
    // Shared-memory tiling per direction (0: rows keyed by dst, 1: by src),
    // built when the graph is small enough that a chunk of the state rows
    // (padded to 32 columns) fits in one CTA's shared memory.
    ck::Tiled tiled[2];
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
enum : int { kDevOk = 0, kDevTimeout = 1, kDevInternal = 2, kDevBounds = 3 };

// Index checks of the bounds-checked build (compiled with -DCK_DEBUG_BOUNDS):
// CK_IN(err, i, n) is true when 0 <= i < n; otherwise it records kDevBounds in
// the status word `err` (the first error wins) and is false, and the caller
// replaces the index by a safe one, so the bad access is skipped rather than
// made.  In the ordinary build it is the constant true and costs nothing.
#if defined(__CUDACC__) && defined(CK_DEBUG_BOUNDS)
__device__ __forceinline__ bool ck_in(int *err, long long i, long long n) {
    if (i >= 0 && i < n) return true;
    atomicCAS(err, 0, (int)kDevBounds);
    return false;
}
#define CK_IN(err, i, n) ::ck::ck_in((err), (long long)(i), (long long)(n))
#else
#define CK_IN(err, i, n) true
#endif

// Phase profile of the profiling build (compiled with -DCK_PHASE_PROFILE): per
// direction and CTA, kPhaseWords counters (layout in ck.h,
// ck_phase_profile_read).
constexpr int kPhaseCtas = CK_PHASE_PROFILE_CTAS, kPhaseWords = CK_PHASE_PROFILE_WORDS;

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
    int o_chunk;  // tiled kernels: the chunk of gathered rows (0 otherwise)
    // a streamed graph slice's cp.async ring, per lane group: ring_n chunks of
    // (edges per batch << ring_chb_sh) {col, w} entries; ring_n == 0: no ring
    int o_ring, ring_n, ring_chb_sh;
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
    // tiled kernels (ck::Tiled): one CTA per SM, the gathered rows' chunk in
    // shared memory; the fields below are per direction
    int tiled;         // 1: both directions run the tiled kernels
    int tP[2];         // CTAs (blocks x chunks)
    int fin_cap[2];    // most rows one CTA finishes
    int chunk_cap[2];  // most nodes in a chunk
    int xrows;         // row stride of the exchange buffer (most rows in a block)
    // scratch layout (byte offsets)
    size_t off_ctrl, ctrl_bytes;
    size_t off_carry;   // float [P][Bp]
    size_t off_xbuf;    // u64 [P][xrows][Bp] tiled kernels' partial totals (right after the carries)
    size_t clear_bytes; // bytes from off_ctrl cleared before every launch (control, carries, xbuf)
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
    std::atomic<int> rows_in_smem{1};
    std::atomic<int> bounds_probe{0};
    std::atomic<int> tiled{0};
};
Options &options();

ck_status make_plan(const ck_graph *g, int64_t B, int64_t T, int64_t M, Plan *p);

// Threads of a tiled-kernel CTA (one CTA per SM) and the widest padded batch
// the tiled kernels take (the layout is sized for it).
constexpr int kTiledThreads = 512;
constexpr int kTiledMaxBp = 32;
// Whether direction dir's tiled kernel fits one CTA's shared memory for a
// tiling with these maxima at padded batch width Bp (the optional graph slice
// and row sums may then still go to global memory).
bool tiled_fits(int dir, int Bp, int max_rows, int max_fin, int max_chunk);

// A scratch offset that names no region: the kernels get a null pointer for it.
constexpr size_t kNoRegion = ~(size_t)0;

// Lay out in p only the scratch regions ck_forward touches (control words,
// carries, permuted edge values, row sums), back to back from offset 0; the
// backward-only regions become kNoRegion.  Sets p->scratch_bytes to the total.
void forward_only_scratch(Plan *p);

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
