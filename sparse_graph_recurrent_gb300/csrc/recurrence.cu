// Forward and backward of the leaky-tanh recurrence over a fixed sparse graph.
//
// connectome-kernels page:
//   intro           proposal = tanh(W h + drive + bias); h <- (1-leak) h +
//                   leak * proposal, `microsteps` times per input step; the
//                   backward has elementwise terms with per-node row
//                   reductions, a transposed sparse product for the state
//                   gradient and a per-edge dot product over the batch for the
//                   edge gradient.  Everything fp32.
//   "Design notes"  states stored [N, B] so a node's batch row is contiguous;
//                   rows with many edges split across warps with an on-chip
//                   reduction; transposed CSR for the state gradient; state and
//                   pre-activation saved after every microstep.
//
// Layout in device memory (fp32, rows padded to Bp: B rounded up to 8; to 32
// for 16 < B <= 32, which keeps four lanes per row; to 16 above 256):
//   H[s+1][N][Bp]  state after microstep s; H[0] = state0 transposed
//   Pr[s][N][Bp]   proposal tanh(pre-activation) of microstep s (the backward
//                  needs only the proposal, so it is saved instead of the
//                  pre-activation and the backward evaluates no tanh)
//   G[N][Bp]       running state gradient (backward)
//   da[2][N][Bp]   d(loss)/d(pre-activation), ping-pong between microsteps
// H[s] and Pr[s] are addressed through hrow / prow, which map s to a slot:
// the saved arrays by default, a window of K input steps when the backward
// recomputes, a two-slot ping-pong when the forward keeps only checkpoints.
// The caller's [T][B][N] outputs and output gradients are read and written one
// input step at a time, transposed through shared memory when staging is on.
//
// Work split.  kCtasPerSm CTAs per SM (ck_internal.h) and one persistent
// cooperative launch per call;
// microsteps are separated by a grid-wide barrier whose wait is bounded.  CTA
// c owns the c-th of P pieces of a row-weighted merge path of (row ends,
// edges), read from a table the graph build computed: a range of edges and
// the rows whose ends fall in its piece.  Inside the CTA the edge range is cut
// into G equal sub-ranges, one per lane group (LPE lanes that together hold
// one batch row as NC chunks of 16-byte loads; a warp holds 32 / LPE groups).
// Each microstep has two parts:
//   A  every group walks its edges in order, UNR at a time: all the gathers of
//      a batch are issued before any is used, whatever rows they belong to.
//      When the group passes the end edge of its current row, the running sum
//      goes to that row's slot in shared memory; the partial sum of the row it
//      stops inside goes to the group's carry slot, after the groups of a warp
//      that carry the same row have added theirs together (a segmented sum
//      over shuffles), so a row split over many groups leaves one carry per
//      warp.
//   B  after a CTA barrier, warps finish the CTA's rows, lane = batch column
//      (one row per warp iteration for B <= 32 with staged operands, else four
//      rows at a time): row slot, plus the carries of the groups that hold the
//      row's earlier edges (and, for the CTA's first row, the carries earlier
//      CTAs published), then the elementwise terms.  Every sum is taken in a
//      fixed order: results do not depend on timing.
// When a CTA's slice of the graph fits in shared memory it is loaded there
// once per call; otherwise it streams from global memory every microstep, each
// batch's {col, w} read one batch ahead of its gathers.  The graph's arrays
// indexed by edge may be device memory or pinned host memory (chosen when the
// graph is built); the kernels read both the same way.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <type_traits>

#include "ck_internal.h"

namespace ck {
namespace {

constexpr unsigned kFull = 0xffffffffu;
// Gathers of rows held as two 16-byte chunks per lane (NC = 2) use one 256-bit
// load (sm_100 and later) instead of two 128-bit ones.
constexpr bool kGatherV8 = true;
// A streamed graph slice (graphs beyond L2, or in host memory) comes through a
// per-group cp.async ring several chunks ahead when shared memory has room.
constexpr bool kStreamRing = true;
constexpr int kMaxSmem = 227 * 1024;      // shared memory one CTA may take
constexpr int kSmemPerSm = 228 * 1024;    // shared memory an SM holds
constexpr int kStaticSmem = 64;

struct KArgs {
    int N, E, n_in, B, Bp, LPE, EPW, LPE_P2, T, M, S;
    int P, G;               // CTAs; lane groups per CTA
    int cap, rows_cap;      // edges / rows (+2) bounds per CTA, for shared memory
    int rs_smem;            // row sums in shared memory (else in global scratch)
    // dynamic shared memory layout (byte offsets)
    int o_srp, o_prm, o_slot, o_grp, o_carry, o_rows, o_tile, o_cw, o_gst, o_dw;
    int stage;  // finish operands staged in shared memory (see Cta)
    int o_st0, o_st1, o_st2, o_st3, o_st4, o_inp, o_acc;
    const int *row_ptr, *col, *perm, *slot, *rowid;
    const int *piece;  // per-CTA piece description, kPieceInts ints each
    const float *w, *leak, *bias, *drives, *state0;
    float *out;
    float *H, *Pr;  // saved states and proposals (Pr null: proposals not kept)
    // H[s] lives in slot s - h_off of H (modulo h_mod when h_mod > 0) and
    // Pr[s] in slot s - p_off of Pr: the saved arrays by default, a window of
    // K input steps when the backward recomputes, a two-slot ping-pong when
    // the forward keeps only checkpoints
    int h_off, h_mod, p_off;
    float *ckpt;  // forward: also write the state after every input step here ([T+1][N][Bp])
    const float *dout;
    float *dw, *dleak, *dbias, *ddrives, *dstate0;
    float *G_, *da, *rowsum_g;
    float2 *lacc;  // [N][32] per-lane {d_leak, d_bias} partials (backward, unstaged)
    unsigned *bar;
    int *err;
    unsigned long long *carry;  // [P][Bp] {float bits, phase id} words
    float *wperm, *dwperm;
    int s_first, s_count, do_prologue, do_epilogue;
    int init_w, zero_dw;  // write the permuted edge values / clear the edge-gradient sums (global)
    unsigned bar_base, bar_extra;
    unsigned long long timeout_ns;
    int bounds_probe;  // bounds-checked build: check one out-of-range index (test hook)
    int o_ring, ring_n, ring_chb_sh;  // streamed graph: per-group cp.async ring (ring_n 0: none)
    // tiled kernels: per-CTA cell descriptions and row pointers, the chunk of
    // gathered rows in shared memory, the exchange of partial row totals
    const int *tmeta, *tptr;
    int o_chunk;       // shared-memory offset of the chunk of gathered rows
    int chunk_cap;     // most nodes in a chunk
    int fin_cap;       // most rows a CTA finishes
    int tC;            // chunks (CTAs per block)
    int xrows;         // row stride of the exchange buffer per CTA (most rows in a block)
    unsigned long long *xbuf;  // [P][xrows][Bp] {float bits, phase id} partial totals
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ float *hrow(const KArgs &a, int s) {
    int j = s - a.h_off;
    if (a.h_mod > 0) j %= a.h_mod;
    return a.H + (size_t)j * a.N * a.Bp;
}
__device__ __forceinline__ float *prow(const KArgs &a, int s) {
    return a.Pr + (size_t)(s - a.p_off) * a.N * a.Bp;
}

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ int ld_err(const int *p) { return *(volatile const int *)p; }

#ifdef CK_PHASE_PROFILE
// The profiling build's counters, summed over microsteps and calls until read
// and cleared (ck_phase_profile_read).
__device__ unsigned long long g_phase[2][kPhaseCtas][kPhaseWords];
#endif

__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }
// 32 bytes from global memory (32-byte aligned), cached in L1 and L2.
__device__ __forceinline__ void ld_ca_v8(const float *p, float4 &lo, float4 &hi) {
    asm volatile("ld.global.ca.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w), "=f"(hi.x), "=f"(hi.y), "=f"(hi.z),
                   "=f"(hi.w)
                 : "l"(p));
}
// The same, cached in L2 only.
__device__ __forceinline__ void ld_cg_v8(const float *p, float4 &lo, float4 &hi) {
    asm volatile("ld.global.cg.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(lo.x), "=f"(lo.y), "=f"(lo.z), "=f"(lo.w), "=f"(hi.x), "=f"(hi.y), "=f"(hi.z),
                   "=f"(hi.w)
                 : "l"(p));
}
__device__ __forceinline__ void fma4(float4 &a, float w, const float4 &x) {
    a.x = fmaf(w, x.x, a.x);
    a.y = fmaf(w, x.y, a.y);
    a.z = fmaf(w, x.z, a.z);
    a.w = fmaf(w, x.w, a.w);
}
__device__ __forceinline__ float dot4(const float4 &a, const float4 &b, float d) {
    d = fmaf(a.x, b.x, d);
    d = fmaf(a.y, b.y, d);
    d = fmaf(a.z, b.z, d);
    return fmaf(a.w, b.w, d);
}

// Grid-wide barrier, bounded by a.timeout_ns.  Each CTA adds one to a
// counter that only grows within a call; barrier idx waits for its total.
// (A two-level tree of counters measured slower here: its extra returning
// atomic costs more than the contention it removes.)  Returns false for the
// whole CTA once any CTA has recorded an error, so every CTA leaves together.
// `during` runs on every thread between the arrival and the wait: work that
// other CTAs do not depend on (output copies, staging of the next operands).
template <class F>
__device__ bool grid_sync(const KArgs &a, unsigned idx, int *s_ok, F &&during) {
    __syncthreads();
    const unsigned target = (a.bar_base + idx + 1u) * (unsigned)a.P + a.bar_extra;
    if (threadIdx.x == 0) red_release_add(a.bar, 1u);
    during();
    if (threadIdx.x == 0) {
        // the status word and the clock are checked every eighth poll, so a
        // poll costs one round trip to the counter
        const unsigned long long t0 = globaltimer();
        int e = 0;
        for (unsigned n = 0; ld_acquire(a.bar) < target; ++n) {
            if ((n & 7) != 7) continue;
            if ((e = ld_err(a.err)) != 0) break;
            if (globaltimer() - t0 > a.timeout_ns) {
                atomicCAS(a.err, 0, kDevTimeout);
                e = kDevTimeout;
                break;
            }
        }
        *s_ok = (e == 0 && ld_err(a.err) == 0) ? 1 : 0;
    }
    __syncthreads();
    return *s_ok != 0;
}
__device__ bool grid_sync(const KArgs &a, unsigned idx, int *s_ok) {
    return grid_sync(a, idx, s_ok, [] {});
}

// Another CTA's published carry for column b: a 64-bit word whose high half
// is the microstep's id, so the value and its validity arrive together (an
// aligned 64-bit access is single-copy atomic).  Bounded wait.
__device__ __forceinline__ float wait_carry(const KArgs &a, const unsigned long long *p,
                                            unsigned phase_id) {
    unsigned long long v = ld_relaxed64(p);
    if ((unsigned)(v >> 32) != phase_id) {
        const unsigned long long t0 = globaltimer();
        do {
            if (ld_err(a.err) != 0) return 0.f;
            if (globaltimer() - t0 > a.timeout_ns) {
                atomicCAS(a.err, 0, kDevTimeout);
                return 0.f;
            }
            v = ld_relaxed64(p);
        } while ((unsigned)(v >> 32) != phase_id);
    }
    return __uint_as_float((unsigned)v);
}

// Transposes between the caller's batch-major [B][N] arrays and the
// node-major [N][Bp] rows, for rows [r0, r1), through a 32x33 tile.
// Every thread of the CTA must call these.
template <int THREADS>
__device__ void to_rows(float *__restrict__ dst, const float *__restrict__ src, int r0, int r1,
                        int B, int Bp, int N, float *tile) {
    const int tid = threadIdx.x;
    for (int rb = r0; rb < r1; rb += 32) {
        for (int cb = 0; cb < Bp; cb += 32) {
            for (int x = tid; x < 32 * 32; x += THREADS) {
                const int rr = x & 31, bb = x >> 5;
                const int r = rb + rr, b = cb + bb;
                tile[bb * 33 + rr] = (r < r1 && b < B) ? __ldg(src + (size_t)b * N + r) : 0.f;
            }
            __syncthreads();
            for (int x = tid; x < 32 * 32; x += THREADS) {
                const int bb = x & 31, rr = x >> 5;
                const int r = rb + rr, b = cb + bb;
                if (r < r1 && b < Bp) dst[(size_t)r * Bp + b] = tile[bb * 33 + rr];
            }
            __syncthreads();
        }
    }
}

template <int THREADS>
__device__ void from_rows(float *__restrict__ dst, const float *__restrict__ src, int r0, int r1,
                          int B, int Bp, int N, float *tile) {
    const int tid = threadIdx.x;
    for (int rb = r0; rb < r1; rb += 32) {
        for (int cb = 0; cb < B; cb += 32) {
            for (int x = tid; x < 32 * 32; x += THREADS) {
                const int bb = x & 31, rr = x >> 5;
                const int r = rb + rr, b = cb + bb;
                tile[bb * 33 + rr] = (r < r1 && b < B) ? __ldcg(src + (size_t)r * Bp + b) : 0.f;
            }
            __syncthreads();
            for (int x = tid; x < 32 * 32; x += THREADS) {
                const int rr = x & 31, bb = x >> 5;
                const int r = rb + rr, b = cb + bb;
                if (r < r1 && b < B) __stcs(dst + (size_t)b * N + r, tile[bb * 33 + rr]);
            }
            __syncthreads();
        }
    }
}

// Per-CTA view of its piece of the work.  Its tables live in shared memory at
// offsets fixed per launch; the accessors below recompute their addresses
// from the shared-memory base instead of holding them in registers.
//   srp    row_ptr[r0 + i], i < nrows + 2 (clamped at N)
//   prm    {leak, bias} of rows r0 + i;  sslot: their input slots
//   sgrp   groups [ga, gb) whose carries belong to row r0 + i, {ga << 16 | gb,
//          first group of the next warp after ga's}
//   scarry [G][Bp] group carries;  tile: [32][33] transpose tile
//   scw, srow, sdw   {col, w bits}, row and edge-gradient sum of the CTA's edges
//   stage mode, rows r0 + i:
//     forward:  st0 = current state (resident, row stride Bp + 1), st1 =
//               drives of the CTA's input rows for the current input step
//               (row inp[i])
//     backward: st0 = G (resident), st1 = Pr[q], st2 = H[q], st3 = dOut[t(q)]
//               (row stride Bp + 1), st4 = H[s] (rows r0 .. r0 + nrows: the
//               source rows part A meets), acc = {d_leak, d_bias} running
//               sums per row and lane, [rows][32] (resident)
struct Cta {
    float *rows;  // [nrows][Bp] row slots (shared or global)
    bool stage;
    int n_inp;
    int r0, nrows, e0, e1, c_lo;
    bool publish;
    bool glob;  // row r0 also sums carries published by earlier CTAs
};

extern __shared__ __align__(16) unsigned char ck_smem[];
__device__ __forceinline__ int *S_srp(const KArgs &a) { return reinterpret_cast<int *>(ck_smem + a.o_srp); }
__device__ __forceinline__ float2 *S_prm(const KArgs &a) { return reinterpret_cast<float2 *>(ck_smem + a.o_prm); }
__device__ __forceinline__ int *S_sslot(const KArgs &a) { return reinterpret_cast<int *>(ck_smem + a.o_slot); }
__device__ __forceinline__ int2 *S_sgrp(const KArgs &a) { return reinterpret_cast<int2 *>(ck_smem + a.o_grp); }
__device__ __forceinline__ float *S_scarry(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_carry); }
__device__ __forceinline__ float *S_tile(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_tile); }
__device__ __forceinline__ int2 *S_scw(const KArgs &a) { return reinterpret_cast<int2 *>(ck_smem + a.o_cw); }
__device__ __forceinline__ int *S_gst(const KArgs &a) { return reinterpret_cast<int *>(ck_smem + a.o_gst); }
__device__ __forceinline__ float *S_sdw(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_dw); }
__device__ __forceinline__ float *S_st0(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_st0); }
__device__ __forceinline__ float *S_st1(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_st1); }
__device__ __forceinline__ float *S_st2(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_st2); }
__device__ __forceinline__ float *S_st3(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_st3); }
__device__ __forceinline__ float *S_st4(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_st4); }
__device__ __forceinline__ int *S_inp(const KArgs &a) { return reinterpret_cast<int *>(ck_smem + a.o_inp); }
__device__ __forceinline__ float2 *S_acc(const KArgs &a) { return reinterpret_cast<float2 *>(ck_smem + a.o_acc); }
__device__ __forceinline__ float *S_chunk(const KArgs &a) { return reinterpret_cast<float *>(ck_smem + a.o_chunk); }
__device__ __forceinline__ int2 *S_ring(const KArgs &a) { return reinterpret_cast<int2 *>(ck_smem + a.o_ring); }
// Row stride of the staged arrays that are also read or written across rows
// (forward st0, backward st3): Bp + 1 words, so a warp walking down a column
// touches 32 distinct banks as well as one walking along a row.
__device__ __forceinline__ int pstride(const KArgs &a) { return a.Bp + 1; }


__device__ __forceinline__ void cp_async16(void *sdst, const void *gsrc) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(sdst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async4(void *sdst, const void *gsrc) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(sdst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// all but the most recently committed group have landed
__device__ __forceinline__ void cp_async_wait_but_last() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
// all but the N most recently committed groups have landed
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Edges per gather batch of part A: four for NC = 2 in both directions (the
// forward, gathering through L2 only, measured fastest at four: three and five
// each lost on some workload, two and six on all; the backward's dot-product
// butterfly wants a power of two), two in the four-chunk backward, where more
// rows in flight per lane measured slower.
__host__ __device__ constexpr int edge_batch(bool bwd, int nc) {
    return bwd && nc != 2 ? 2 : 4;
}

// The helpers below spread their work over nt threads, this one being number
// t of them.

// Copy this CTA's rows [r0, r0 + nrows) of a node-major array into shared memory.
__device__ __forceinline__ void stage_rows(float *sdst, const float *gsrc, int nrows, int Bp, int t,
                                           int nt) {
    const int n16 = nrows * Bp / 4;
    for (int j = t; j < n16; j += nt) cp_async16(sdst + 4 * j, gsrc + 4 * j);
}

// Copy dOut of input step ts for this CTA's rows (a [B][N] slab, rows r0 + i
// contiguous per column) into st3 as rows of stride Bp + 1: consecutive
// threads read consecutive nodes of one column.
__device__ __forceinline__ void stage_dout(const KArgs &a, const Cta &c, int ts, int t, int nt) {
    const float *src = a.dout + (size_t)ts * a.B * a.N + c.r0;
    for (int j = t; j < c.nrows * a.B; j += nt) {
        const int b = j / c.nrows, i = j - b * c.nrows;
        cp_async4(S_st3(a) + i * pstride(a) + b, src + (size_t)b * a.N + i);
    }
}

// Write the state held in st0 to output step ts ([B][N] slab): consecutive
// threads write consecutive nodes of one column.
__device__ __forceinline__ void write_out(const KArgs &a, const Cta &c, int ts, int t, int nt) {
    if (!a.out) return;  // a recomputation writes no outputs
    float *dst = a.out + (size_t)ts * a.B * a.N + c.r0;
    for (int j = t; j < c.nrows * a.B; j += nt) {
        const int b = j / c.nrows, i = j - b * c.nrows;
        __stcs(dst + (size_t)b * a.N + i, S_st0(a)[i * pstride(a) + b]);
    }
}

// The lane group whose edge sub-range holds edge k of the CTA (n = e1 - e0 > 0).
__device__ __forceinline__ int group_of(const Cta &c, int G, int k) {
    const long long n = c.e1 - c.e0;
    const int g = (int)(((long long)(k - c.e0 + 1) * G - 1) / n);
    return g < G - 1 ? g : G - 1;
}

// ------------------------------------------------------------ part A

// Walk this lane group's edges: gather rows[col[k]] * w[k] into per-row sums,
// UNR edges per batch with all of a batch's gathers issued before any is used.
// Backward: also add each edge's
// dot product with the state h_{s-1} of its source row into the edge-gradient
// accumulator; that source row stays in registers, and the next row's is
// fetched as soon as the current one starts.
template <int NC, int UNR>
struct Batch {
    float w[UNR];
    float4 v[UNR][NC];
};

// Sum of d over the LPE lanes of each group.  With LPE a power of two and a
// multiple of UNR (a power of two), the first log2(UNR) exchanges (lane
// offsets LPE/2, LPE/4, ...) each keep half of the items, and the remaining
// ones (offsets LPE/(2 UNR) ... 1) add: lane lig then holds in d[0] the total
// of item lig / (LPE / UNR) (item lig when LPE == UNR).  Otherwise each item
// is reduced by a tree and lane 0 holds it.
__device__ __forceinline__ bool butterfly_dots(int lpe, int unr) {
    return lpe >= unr && (lpe & (lpe - 1)) == 0 && (unr & (unr - 1)) == 0;
}
template <int UNR>
__device__ __forceinline__ void group_dots(float (&d)[UNR], int lig, int lpe, int lpe_p2) {
    if (lpe == UNR && (UNR & (UNR - 1)) == 0) {  // the common case, offsets known at compile time
#pragma unroll
        for (int o = UNR / 2; o >= 1; o >>= 1) {
#pragma unroll
            for (int j = 0; j < o; ++j) {
                const bool hi = (lig & o) != 0;
                const float keep = hi ? d[j + o] : d[j];
                const float send = hi ? d[j] : d[j + o];
                d[j] = keep + __shfl_xor_sync(kFull, send, o);
            }
        }
    } else if (butterfly_dots(lpe, UNR)) {
        int off = lpe >> 1;
#pragma unroll
        for (int o = UNR / 2; o >= 1; o >>= 1, off >>= 1) {
#pragma unroll
            for (int j = 0; j < o; ++j) {
                const bool hi = (lig & off) != 0;
                const float keep = hi ? d[j + o] : d[j];
                const float send = hi ? d[j] : d[j + o];
                d[j] = keep + __shfl_xor_sync(kFull, send, off);
            }
        }
        for (; off >= 1; off >>= 1) d[0] += __shfl_xor_sync(kFull, d[0], off);
    } else {
#pragma unroll
        for (int q = 0; q < UNR; ++q) {
            for (int o = lpe_p2 >> 1; o >= 1; o >>= 1) {
                const float y = __shfl_down_sync(kFull, d[q], o);
                if (lig + o < lpe) d[q] += y;
            }
        }
    }
}

// TT: the gathered rows are the chunk in shared memory (tiled kernels; column
// indices then count from the chunk's first node), else `rows` in global memory.
// RG (streamed graph only): {col, w} come through the group's cp.async ring in
// shared memory, several chunks ahead, instead of registers one batch ahead.
template <int NC, bool SMEMG, bool BWD, int UNR, bool HS, bool TT = false, bool RG = false>
__device__ __forceinline__ void stream_piece(const KArgs &a, const Cta &c, int gam, int lig,
                                             bool active, const float *__restrict__ rows,
                                             const float *__restrict__ hprev) {
    static_assert(!(SMEMG && RG), "the ring serves a streamed graph only");
    constexpr bool REG = !SMEMG && !RG;  // {col, w} one batch ahead in registers
    const int Bp = a.Bp, CW = 4 * a.LPE;
    // Columns a lane holds: chunk ch covers LB + ch * CS .. + 3.  With 256-bit
    // gathers (V8) a lane's two chunks are contiguous (columns 8 lig .. 8 lig
    // + 7); otherwise chunk ch sits CW columns after chunk ch - 1.
    constexpr bool V8 = kGatherV8 && NC == 2 && !TT;
    const int LB = V8 ? lig * 8 : lig * 4;
    const int CS = V8 ? 4 : CW;
    const int n = c.e1 - c.e0;
    int k0 = c.e0, k1 = c.e0;
    if (active && n > 0) {
        k0 = c.e0 + (int)((long long)gam * n / a.G);
        k1 = c.e0 + (int)((long long)(gam + 1) * n / a.G);
    }
    const int len = k1 - k0;
    const int trips = (__reduce_max_sync(kFull, (unsigned)len) + UNR - 1) / UNR;
    auto row_at = [&](int k) -> int { return __ldg(a.rowid + k); };
    const int row0 = active ? S_gst(a)[gam] : -1;  // row of edge k0 (when k0 < e1), set up once
    int cur = len > 0 ? row0 : -1;
    int bnd = len > 0 ? S_srp(a)[cur - c.r0 + 1] : k1;  // end of cur's edges
    float4 acc[NC];
#pragma unroll
    for (int ch = 0; ch < NC; ++ch) acc[ch] = zero4();

    // backward: own-row state of the current source row and, when it is read
    // from global memory (HS false), of the next one, fetched ahead; with HS
    // the CTA's rows of h_{s-1} are staged in shared memory (st4)
    constexpr int HN = BWD ? NC : 1;
    struct HRow {
        float4 v[HN];
    };
    auto load_h = [&](int row) -> HRow {
        HRow h;
        if (HS) {
            int i = row - c.r0;
            const bool in = row >= 0 && i <= c.nrows;  // always, for a valid graph
            if (in && !CK_IN(a.err, i, a.rows_cap)) i = 0;
            const float *hp = S_st4(a) + (size_t)(in ? i : 0) * Bp + LB;
#pragma unroll
            for (int ch = 0; ch < HN; ++ch)
                h.v[ch] = in ? *reinterpret_cast<const float4 *>(hp + ch * CS) : zero4();
        } else {
            if (row >= 0 && !CK_IN(a.err, row, a.N)) row = 0;
            const float *hp = hprev + (size_t)(row < 0 ? 0 : row) * Bp + LB;
#pragma unroll
            for (int ch = 0; ch < HN; ++ch)
                h.v[ch] = row >= 0 ? __ldg(reinterpret_cast<const float4 *>(hp + ch * CS)) : zero4();
        }
        return h;
    };
    HRow hcur, hnext;
    int nxt = -1;
    auto next_row = [&](int row) -> int {  // the row after `row` that has edges in [k0, k1)
        int ir = row - c.r0 + 1;
        if (!CK_IN(a.err, ir, a.rows_cap)) ir = 0;
        const int pos = S_srp(a)[ir];
        return pos < k1 ? row_at(pos) : -1;
    };
    if (BWD) {
        hcur = load_h(cur);
        if (!HS) {
            nxt = cur >= 0 ? next_row(cur) : -1;
            hnext = load_h(nxt);
        }
    }

    auto flush = [&](int row) {
        const int i = row - c.r0;
        if (i >= 0 && i < c.nrows) {
            float *dst = c.rows + (size_t)i * Bp + LB;
#pragma unroll
            for (int ch = 0; ch < NC; ++ch) *reinterpret_cast<float4 *>(dst + ch * CS) = acc[ch];
        } else {
            atomicCAS(a.err, 0, kDevInternal);  // cannot happen for a valid graph
        }
#pragma unroll
        for (int ch = 0; ch < NC; ++ch) acc[ch] = zero4();
    };
    // Edges past the group's range (the warp runs to its longest group) load
    // the CTA's first edge and weigh 0, so every load is unconditional.  A
    // graph streamed from global memory is read one batch ahead (into gc,
    // gw), so a batch's gathers never wait on its own column loads.
    // backward: the edge-gradient reduction's layout (see group_dots)
    const bool bfly = BWD && butterfly_dots(a.LPE, UNR);
    int per_sh = 0;
    while (bfly && (UNR << per_sh) < a.LPE) ++per_sh;  // log2(LPE / UNR)
    const bool dw_owner = bfly && (lig & ((1 << per_sh) - 1)) == 0;  // writes item lig >> per_sh
    int gc[REG ? UNR : 1];
    float gw[REG ? UNR : 1];
    // streamed backward with the butterfly layout: the edge-gradient sum this
    // lane updates in a batch, read one batch ahead too, so the update is a
    // store (each edge's sum is touched by its own group only, once per
    // microstep)
    float gdw = 0.f, cdw = 0.f;
    auto load_graph = [&](int kb) {
        if (BWD && !SMEMG && dw_owner) {
            int kk = kb + (lig >> per_sh);
            if (kk < k1 && !CK_IN(a.err, kk, a.E)) kk = k1;
            gdw = kk < k1 ? __ldcg(a.dwperm + kk) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < (REG ? UNR : 0); ++q) {
            const int kk = kb + q;
            int kc = kk < k1 ? kk : c.e0;
            if (!CK_IN(a.err, kc, a.E)) kc = 0;
            gc[q] = __ldg(a.col + kc);
            gw[q] = __ldcg(a.wperm + kc);
        }
    };
    // The ring: RN chunks (a power of two) of CHE = UNR << chb_sh edges, as
    // {col, w bits}.  Chunk ch of the group's range goes to slot ch mod RN,
    // copied by the group's lanes RN - 1 chunks before it is read; only chunks
    // that start inside [k0, k1) are copied (their entries past k1 copy edge e0),
    // and every chunk boundary commits a group, empty or not, which keeps the
    // wait counts fixed.  Each lane waits for its own copies; a __syncwarp then
    // makes the group's copies visible to all its lanes.
    const int chb_sh = RG ? a.ring_chb_sh : 0;
    const int RN = RG ? a.ring_n : 1;
    const int CHE = UNR << chb_sh;
    int2 *ring = RG && active ? S_ring(a) + (size_t)gam * RN * CHE : nullptr;
    auto issue = [&](int ch) {
        const int base = k0 + ch * CHE;
        if (ring && base < k1) {
            int2 *dst = ring + (ch & (RN - 1)) * CHE;
            for (int e = lig; e < CHE; e += a.LPE) {
                const int kk = base + e;
                int kc = kk < k1 ? kk : c.e0;
                if (!CK_IN(a.err, kc, a.E)) kc = 0;
                cp_async4(&dst[e].x, a.col + kc);
                cp_async4(&dst[e].y, a.wperm + kc);
            }
        }
        cp_async_commit();
    };
    auto load = [&](Batch<NC, UNR> &bt, int kb, int it) {
        int cn[UNR];
        float wn[UNR];
        if (REG) {
#pragma unroll
            for (int q = 0; q < UNR; ++q) {
                cn[q] = gc[REG ? q : 0];
                wn[q] = gw[REG ? q : 0];
            }
        }
        if (RG) {
            const int pos = it & ((1 << chb_sh) - 1);
            if (pos == 0) {
                // this chunk's copies (all lanes') have landed, and every lane
                // is done with the slot the next copy refills
                if (RN == 4) cp_async_wait_group<2>();
                else cp_async_wait_group<0>();
                __syncwarp();
                issue((it >> chb_sh) + RN - 1);
            }
            const int2 *src = ring ? ring + ((it >> chb_sh) & (RN - 1)) * CHE + pos * UNR : nullptr;
#pragma unroll
            for (int q = 0; q < UNR; ++q) {
                const int2 cw = src ? src[q] : make_int2(0, 0);
                cn[q] = cw.x;
                wn[q] = __int_as_float(cw.y);
            }
        }
        if (!SMEMG) {
            if (BWD) cdw = gdw;
            load_graph(kb + UNR);  // next batch's edges (valid addresses past the end too)
        }
#pragma unroll
        for (int q = 0; q < UNR; ++q) {
            const int kk = kb + q;
            const bool ok = kk < k1;
            const int kc = ok ? kk : c.e0;  // n > 0 whenever a batch runs
            int cc;
            float wv;
            if (SMEMG) {
                int ks = kc - c.e0;
                if (!CK_IN(a.err, ks, a.cap)) ks = 0;
                const int2 cw = S_scw(a)[ks];
                cc = cw.x;
                wv = __int_as_float(cw.y);
            } else {
                // a ring slot past the group's range holds no copy: row 0
                // stands in (weight 0)
                cc = RG && !ok ? 0 : cn[q];
                wv = wn[q];
            }
            bt.w[q] = ok ? wv : 0.f;
            if constexpr (TT) {
                if (!CK_IN(a.err, cc, a.chunk_cap)) cc = 0;
                const float *rp = S_chunk(a) + cc * Bp + lig * 4;
#pragma unroll
                for (int ch = 0; ch < NC; ++ch) bt.v[q][ch] = *reinterpret_cast<const float4 *>(rp + ch * CW);
            } else {
                if (!CK_IN(a.err, cc, a.N)) cc = 0;
                const float *rp = rows + (size_t)cc * Bp + LB;
                if constexpr (V8) {
                    // the forward's rows hit L1 for 16% of sectors only: they go
                    // through L2 alone (measured 0.2-0.4% faster); the backward's
                    // d(pre-activation) rows hit L1 for half, and keep it
                    if (BWD) ld_ca_v8(rp, bt.v[q][0], bt.v[q][NC - 1]);
                    else ld_cg_v8(rp, bt.v[q][0], bt.v[q][NC - 1]);
                } else {
#pragma unroll
                    for (int ch = 0; ch < NC; ++ch)
                        bt.v[q][ch] = __ldca(reinterpret_cast<const float4 *>(rp + ch * CW));
                }
            }
        }
    };
    // The group's current row is cur and its edges end at bnd = row_ptr[cur +
    // 1]: an edge at or past bnd starts a later row (rows without edges are
    // skipped).  A batch that no group of the warp sees cross its bound takes
    // the path without per-edge checks.
    auto next_row_at = [&](int kk) {
        flush(cur);
        do {
            ++cur;
            if (!CK_IN(a.err, cur - c.r0 + 1, a.rows_cap)) {
                cur = c.r0 + a.rows_cap - 2;
                break;
            }
        } while (S_srp(a)[cur - c.r0 + 1] <= kk);
        bnd = S_srp(a)[cur - c.r0 + 1];
        if (BWD) {
            if (HS) {
                hcur = load_h(cur);
            } else {
                hcur = cur == nxt ? hnext : load_h(cur);
                nxt = next_row(cur);
                hnext = load_h(nxt);
            }
        }
    };
    auto consume = [&](const Batch<NC, UNR> &bt, int kb) {
        float d[UNR];
        const int lim = kb + UNR < k1 ? kb + UNR : k1;
        const bool inside = __all_sync(kFull, lim <= bnd);
#pragma unroll
        for (int q = 0; q < UNR; ++q) {
            d[q] = 0.f;
            if (!inside) {
                const int kk = kb + q;
                if (kk < k1 && kk >= bnd) next_row_at(kk);
            }
#pragma unroll
            for (int ch = 0; ch < NC; ++ch) fma4(acc[ch], bt.w[q], bt.v[q][ch]);
            if (BWD) {
#pragma unroll
                for (int ch = 0; ch < NC; ++ch) d[q] = dot4(bt.v[q][ch], hcur.v[BWD ? ch : 0], d[q]);
            }
        }
        if (BWD) {
            group_dots<UNR>(d, lig, a.LPE, a.LPE_P2);
            if (bfly) {
                // lanes lig = m * (LPE / UNR) hold item m
                const int kk = kb + (lig >> per_sh);
                if ((lig & ((1 << per_sh) - 1)) == 0 && kk < k1 &&
                    CK_IN(a.err, SMEMG ? kk - c.e0 : kk, SMEMG ? a.cap : a.E)) {
                    if (SMEMG) S_sdw(a)[kk - c.e0] += d[0];
                    else a.dwperm[kk] = cdw + d[0];
                }
            } else if (lig == 0) {
#pragma unroll
                for (int q = 0; q < UNR; ++q) {
                    const int kk = kb + q;
                    if (kk < k1 && CK_IN(a.err, SMEMG ? kk - c.e0 : kk, SMEMG ? a.cap : a.E)) {
                        if (SMEMG) S_sdw(a)[kk - c.e0] += d[q];
                        else a.dwperm[kk] += d[q];
                    }
                }
            }
        }
    };

    Batch<NC, UNR> bt;
    if (!SMEMG && trips > 0) load_graph(k0);
    if (RG && trips > 0)
        for (int ch = 0; ch < RN - 1; ++ch) issue(ch);
    for (int it = 0; it < trips; ++it) {
        const int kb = k0 + it * UNR;
        load(bt, kb, it);
        consume(bt, kb);
    }
    if (RG) {
        // every copy issued was waited for above; this only settles the
        // (empty) groups committed last
        cp_async_wait_all();
        __syncwarp();
    }
    // the row this group stops in: finished here if its last edge is ours and
    // its row end belongs to this CTA (the carry is then 0), else a carry
    int lab = -2;  // row of this group's carry; never equal for inactive lanes
    if (active) {
        const bool fin = len > 0 && cur >= c.r0 && cur < c.r0 + c.nrows &&
                         S_srp(a)[cur - c.r0 + 1] == k1;
        if (fin) flush(cur);
        // an empty group sits at edge k0 < e1 (n > 0): it takes that edge's row
        lab = len > 0 ? cur : row0;
    }
    // Segmented suffix sums over the warp's groups: a group adds the carry of
    // the group d places on while both carry the same row (labels do not
    // decrease along the groups, so equal ends mean an equal run).  Afterwards
    // the first group of each run in the warp holds the run's total, and a row
    // spread over many groups needs one carry read per warp it crosses.
    const int g = (threadIdx.x & 31) / a.LPE;
    for (int d = 1; d < a.EPW; d <<= 1) {
        const int sh = d * a.LPE;
        const int lo = __shfl_down_sync(kFull, lab, sh);
        const bool take = g + d < a.EPW && lo == lab;
#pragma unroll
        for (int ch = 0; ch < NC; ++ch) {
            float4 o;
            o.x = __shfl_down_sync(kFull, acc[ch].x, sh);
            o.y = __shfl_down_sync(kFull, acc[ch].y, sh);
            o.z = __shfl_down_sync(kFull, acc[ch].z, sh);
            o.w = __shfl_down_sync(kFull, acc[ch].w, sh);
            if (take) {
                acc[ch].x += o.x;
                acc[ch].y += o.y;
                acc[ch].z += o.z;
                acc[ch].w += o.w;
            }
        }
    }
    if (active && CK_IN(a.err, gam, a.G)) {
        float *dst = S_scarry(a) + (size_t)gam * Bp + LB;
#pragma unroll
        for (int ch = 0; ch < NC; ++ch) *reinterpret_cast<float4 *>(dst + ch * CS) = acc[ch];
    }
}

// Part A with the streamed graph's ring when the plan gave it room.
template <int NC, bool SMEMG, bool BWD, int UNR, bool HS>
__device__ __forceinline__ void part_a(const KArgs &a, const Cta &c, int gam, int lig, bool active,
                                       const float *__restrict__ rows, const float *__restrict__ hprev) {
    if constexpr (!SMEMG) {
        if (a.ring_n > 0) {
            stream_piece<NC, false, BWD, UNR, HS, false, true>(a, c, gam, lig, active, rows, hprev);
            return;
        }
    }
    stream_piece<NC, SMEMG, BWD, UNR, HS>(a, c, gam, lig, active, rows, hprev);
}

// ------------------------------------------------------------ part B

// Element layout of part B: a warp finishes RB rows at a time, lane = batch
// column, NCH 32-column chunks per row, at most four (row, chunk) elements per
// lane per batch.  Fixed per launch.
struct PB {
    int NCH, cpb, RB, CB;
    int ri[4], ci[4];
};

__device__ __forceinline__ PB make_pb(int Bp) {
    PB p;
    p.NCH = (Bp + 31) >> 5;
    p.cpb = p.NCH < 4 ? p.NCH : 4;
    p.RB = 4 / p.cpb;
    p.CB = (p.NCH + p.cpb - 1) / p.cpb;
#pragma unroll
    for (int el = 0; el < 4; ++el) {
        p.ri[el] = el / p.cpb;
        p.ci[el] = el - p.ri[el] * p.cpb;
    }
    return p;
}

// Column b of the carries of groups [ga, gb), all of one row, after part A's
// per-warp run sums: group ga's entry covers the row's groups in ga's warp,
// and the first group of every later warp below gb covers that warp's.  The
// first two reads are unconditional (clamped, masked) so they issue without
// waiting on branches.
__device__ __forceinline__ int next_warp_group(const KArgs &a, int ga) { return (ga / a.EPW + 1) * a.EPW; }
__device__ __forceinline__ float carry_sum(const KArgs &a, const float *sc, int ga, int gb, int h1) {
    const float v0 = sc[(size_t)min(ga, a.G - 1) * a.Bp];
    const float v1 = sc[(size_t)min(h1, a.G - 1) * a.Bp];
    float x = ga < gb ? v0 : 0.f;
    x += h1 < gb ? v1 : 0.f;
    for (int h = h1 + a.EPW; h < gb && CK_IN(a.err, h, a.G); h += a.EPW) x += sc[(size_t)h * a.Bp];
    return x;
}

// Row sums of four (row, column) elements: each row's slot (the part summed by
// the group holding its last edge here) plus the carries of the groups holding
// its earlier edges (carry_sum's terms and order); 0 for a row with no edges
// in this CTA.  Every load of the common case (at most two carry reads) is
// unconditional, so the four elements' loads issue together; rows that cross
// more warps finish in a second pass.
template <bool RS>
__device__ __forceinline__ void row_sums4(const KArgs &a, const Cta &c, const int (&ii)[4],
                                          const int (&bb)[4], float (&x)[4]) {
    const float *sc = S_scarry(a);
    float slot[4], cs[4];
    int gb[4], h2[4];
#pragma unroll
    for (int el = 0; el < 4; ++el) {
        const int2 g2 = S_sgrp(a)[ii[el]];
        const int gr = g2.x;
        const size_t o = (size_t)ii[el] * a.Bp + bb[el];
        const float sv = RS ? c.rows[o] : __ldcg(c.rows + o);
        const int ga = gr < 0 ? 0 : gr >> 16;
        gb[el] = gr < 0 ? 0 : (gr & 0xffff);
        const int h1 = g2.y;
        const float v0 = sc[(size_t)min(ga, a.G - 1) * a.Bp + bb[el]];
        const float v1 = sc[(size_t)min(h1, a.G - 1) * a.Bp + bb[el]];
        slot[el] = gr < 0 ? 0.f : sv;
        cs[el] = ga < gb[el] ? v0 : 0.f;
        cs[el] += h1 < gb[el] ? v1 : 0.f;
        h2[el] = h1 + a.EPW;
    }
#pragma unroll
    for (int el = 0; el < 4; ++el)
        for (int h = h2[el]; h < gb[el] && CK_IN(a.err, h, a.G); h += a.EPW)
            cs[el] += sc[(size_t)h * a.Bp + bb[el]];
#pragma unroll
    for (int el = 0; el < 4; ++el) x[el] = slot[el] + cs[el];
}

// Carries published by earlier CTAs for column b of the CTA's first row.
__device__ __forceinline__ float global_carry(const KArgs &a, const Cta &c, int b,
                                              unsigned phase_id) {
    float x = 0.f;
    for (int cc = c.c_lo; cc < (int)blockIdx.x; ++cc)
        if (CK_IN(a.err, cc, a.P) && CK_IN(a.err, b, a.Bp))
            x += wait_carry(a, a.carry + (size_t)cc * a.Bp + b, phase_id);
    return x;
}

// Ask L2 to fetch `bytes` from `p` (16-byte aligned, multiple of 16) ahead of use.
__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes) {
    if (bytes >= 16)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes & ~15u) : "memory");
}

// Call f with the staging and row-sum placement as compile-time flags, so the
// finish code has no per-element branches on them.
template <class F>
__device__ __forceinline__ void dispatch_modes(bool stage, bool rs, F &&f) {
    using T = std::true_type;
    using Fl = std::false_type;
    if (stage) {
        if (rs) f(T{}, T{});
        else f(T{}, Fl{});
    } else {
        if (rs) f(Fl{}, T{});
        else f(Fl{}, Fl{});
    }
}

// Forward finish of rows [lo, hi) among the batch starting at row i0:
// pre-activation, tanh, leak blend, saved copies.  Straight-line over the
// batch's elements so their loads and tanh evaluations overlap.  Without
// staging, the state that ends an input step is also written to the output
// here; with staging it is copied out of st0 during the next microstep.
template <bool ST, bool RS>
__device__ __forceinline__ void finish_fwd_batch(const KArgs &a, const Cta &c, const PB &pb,
                                                 int s, unsigned phase_id, int i0, int lo,
                                                 int hi) {
    const int lane = threadIdx.x & 31;
    const int Bp = a.Bp, B = a.B;
    const int t = s / a.M;
    const bool step_end = s - t * a.M == a.M - 1;
    const size_t NBp = (size_t)a.N * Bp;
    const float *hin = hrow(a, s);
    float *hout = hrow(a, s + 1);
    float *pout = a.Pr ? prow(a, s) : nullptr;
    for (int cb = 0; cb < pb.CB; ++cb) {
        int ii[4], bb[4];
        bool ok[4];
        float x[4], hp[4], dr[4];
        float2 pr[4];
#pragma unroll
        for (int el = 0; el < 4; ++el) {
            const int i = i0 + pb.ri[el], cc = cb * pb.cpb + pb.ci[el], b = cc * 32 + lane;
            ok[el] = pb.ri[el] < pb.RB && i >= lo && i < hi && cc < pb.NCH && b < Bp;
            ii[el] = ok[el] ? i : hi - 1;  // an initialised row, read but not used
            bb[el] = ok[el] ? b : 0;
        }
        row_sums4<RS>(a, c, ii, bb, x);
#pragma unroll
        for (int el = 0; el < 4; ++el) {
            const size_t o = (size_t)ii[el] * Bp + bb[el];
            pr[el] = S_prm(a)[ii[el]];
            hp[el] = ST ? S_st0(a)[ii[el] * pstride(a) + bb[el]] : __ldcg(hin + (size_t)c.r0 * Bp + o);
            // drive: loaded from a valid address whatever the row, kept only
            // for a live column of an input row
            const int bl = bb[el] < B ? bb[el] : B - 1;
            if (ST) {
                const int j = S_inp(a)[ii[el]];
                const float v = S_st1(a)[(size_t)(j < 0 ? 0 : j) * Bp + bl];
                dr[el] = ok[el] && j >= 0 && bb[el] < B ? v : 0.f;
            } else {
                const int sl = S_sslot(a)[ii[el]];
                dr[el] = 0.f;
                if (a.n_in > 0) {
                    const float v = __ldg(a.drives + ((size_t)t * a.n_in + (sl < 0 ? 0 : sl)) * B + bl);
                    dr[el] = ok[el] && sl >= 0 && bb[el] < B ? v : 0.f;
                }
            }
        }
        if (lo == 0 && i0 == 0 && c.glob) {
#pragma unroll
            for (int el = 0; el < 4; ++el)
                if (pb.ri[el] == 0 && pb.RB > 0) x[el] += global_carry(a, c, bb[el], phase_id);
        }
        float av[4], th[4];
#pragma unroll
        for (int el = 0; el < 4; ++el) av[el] = x[el] + pr[el].y + dr[el];
#pragma unroll
        for (int el = 0; el < 4; ++el) th[el] = tanhf(av[el]);
#pragma unroll
        for (int el = 0; el < 4; ++el) {
            const bool live = bb[el] < B;
            const float hv = live ? fmaf(pr[el].x, th[el], (1.f - pr[el].x) * hp[el]) : 0.f;
            const float p0 = live ? th[el] : 0.f;
            if (ok[el]) {
                const size_t o = (size_t)ii[el] * Bp + bb[el];
                if (ST) S_st0(a)[ii[el] * pstride(a) + bb[el]] = hv;
                else if (step_end && live && a.out)
                    __stcs(a.out + ((size_t)t * B + bb[el]) * a.N + c.r0 + ii[el], hv);
                hout[(size_t)c.r0 * Bp + o] = hv;
                if (pout) __stcs(pout + (size_t)c.r0 * Bp + o, p0);
                if (a.ckpt && step_end) a.ckpt[(size_t)(t + 1) * NBp + (size_t)c.r0 * Bp + o] = hv;
            }
        }
    }
}


// ---- finish for Bp <= 32 with staged operands and row slots in shared memory
// (every FlyGPT-shaped workload).  Warp w takes rows r0 + sh + w, + 16, ...,
// one row per iteration, lane = batch column, where sh = 1 when the first row
// waits for earlier CTAs' carries: that row goes to the last warp, after its
// others (the last warp has the fewest).  Shared-memory offsets are 32-bit,
// and the arithmetic is the batched finish's, term for term, so both give
// identical results.

// Row i's sum for column b (b < Bp): row_sums4's terms in its order.
__device__ __forceinline__ float row_sum1(const KArgs &a, const Cta &c, int i, int b) {
    if (!CK_IN(a.err, i, a.rows_cap)) i = 0;
    const int2 g2 = S_sgrp(a)[i];
    const int gr = g2.x;
    const float *sc = S_scarry(a) + b;
    const float sv = c.rows[i * a.Bp + b];
    const int ga = gr < 0 ? 0 : gr >> 16, gb = gr < 0 ? 0 : (gr & 0xffff), h1 = g2.y;
    const float v0 = sc[min(ga, a.G - 1) * a.Bp];
    const float v1 = sc[min(h1, a.G - 1) * a.Bp];
    float cs = ga < gb ? v0 : 0.f;
    cs += h1 < gb ? v1 : 0.f;
    for (int h = h1 + a.EPW; h < gb && CK_IN(a.err, h, a.G); h += a.EPW) cs += sc[h * a.Bp];
    return (gr < 0 ? 0.f : sv) + cs;
}

// The row total of a finished row i (relative to c.r0) in column b: rowx(i,
// b, lane_ok) -- the row slot plus carries (and earlier CTAs' carries) here,
// the sum of the chunks' partial totals in the tiled kernels.
template <int THREADS, class RowX>
__device__ __forceinline__ void finish_fwd_narrow(const KArgs &a, const Cta &c, int s,
                                                  RowX &&rowx) {
    constexpr int U = THREADS / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Bp = a.Bp, B = a.B, PS = Bp + 1;
    const size_t NBp = (size_t)a.N * Bp;
    const int t = s / a.M;
    const bool step_end = s - t * a.M == a.M - 1;
    float *hout = hrow(a, s + 1) + (size_t)c.r0 * Bp;
    float *pout = a.Pr ? prow(a, s) + (size_t)c.r0 * Bp : nullptr;
    float *ck = a.ckpt && step_end ? a.ckpt + (size_t)(t + 1) * NBp + (size_t)c.r0 * Bp : nullptr;
    const bool lane_ok = lane < Bp, live = lane < B;
    const int b = lane_ok ? lane : 0, bl = live ? lane : B - 1;
    const int sh = c.glob ? 1 : 0;
    auto row = [&](int i) {
        const float x = rowx(i, b, lane_ok);
        const float2 pr = S_prm(a)[i];
        const float hp = S_st0(a)[i * PS + b];
        int j = S_inp(a)[i];
        if (j >= 0 && !CK_IN(a.err, j, a.rows_cap)) j = -1;
        const float dv = S_st1(a)[(j < 0 ? 0 : j) * Bp + bl];
        const float dr = lane_ok && j >= 0 && live ? dv : 0.f;
        const float av = x + pr.y + dr;
        const float th = tanhf(av);
        const float hv = live ? fmaf(pr.x, th, (1.f - pr.x) * hp) : 0.f;
        if (lane_ok) {
            S_st0(a)[i * PS + b] = hv;
            hout[i * Bp + b] = hv;
            if (pout) __stcs(pout + i * Bp + b, live ? th : 0.f);
            if (ck) ck[i * Bp + b] = hv;
        }
    };
    for (int i = sh + warp; i < c.nrows; i += U) row(i);
    if (sh && warp == U - 1) row(0);
}

template <int THREADS, class RowX>
__device__ __forceinline__ void finish_bwd_narrow(const KArgs &a, const Cta &c, int s,
                                                  RowX &&rowx) {
    constexpr int U = THREADS / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Bp = a.Bp, B = a.B, M = a.M, PS = Bp + 1;
    const size_t NBp = (size_t)a.N * Bp;
    const bool pro = s == a.S;
    const int q = s - 1;
    const int tq = q >= 0 ? q / M : 0;
    const bool step_end = q >= 0 && q - tq * M == M - 1;  // also the first visit of step tq
    float *daq = a.da + (size_t)(q & 1) * NBp + (size_t)c.r0 * Bp;
    const bool lane_ok = lane < Bp, live = lane < B;
    const int b = lane_ok ? lane : 0, bl = live ? lane : B - 1;
    const int sh = c.glob ? 1 : 0;
    auto row = [&](int i) {
        const float x = pro ? 0.f : rowx(i, b, lane_ok);
        const float lam = S_prm(a)[i].x;
        const int o = i * Bp + b;
        const float g0 = S_st0(a)[o], o0 = S_st3(a)[i * PS + bl], p0 = S_st1(a)[o], h0 = S_st2(a)[o];
        const float gv = pro ? 0.f : g0;
        const float ov = step_end && live ? o0 : 0.f;
        const float p = q >= 0 ? p0 : 0.f, hv = q >= 0 ? h0 : 0.f;
        float gn = fmaf(gv, 1.f - lam, x) + ov;
        if (!live) gn = 0.f;
        if (lane_ok) S_st0(a)[o] = gn;
        if (q < 0) return;
        float dl = 0.f, db = 0.f, d = 0.f;
        if (lane_ok && live) {
            d = gn * lam * (1.f - p * p);
            dl = fmaf(gn, p - hv, dl);
            db += d;
            const int sl = S_sslot(a)[i];
            if (sl >= 0 && CK_IN(a.err, sl, a.n_in)) {
                float *dd = a.ddrives + ((size_t)tq * a.n_in + sl) * B + lane;
                *dd = step_end ? d : *dd + d;
            }
        }
        if (lane_ok) daq[o] = d;
        float2 *pa = S_acc(a) + i * 32 + lane;
        const float2 old = q == a.S - 1 ? make_float2(0.f, 0.f) : *pa;
        *pa = make_float2(old.x + (0.f + dl), old.y + (0.f + db));
    };
    for (int i = sh + warp; i < c.nrows; i += U) row(i);
    if (sh && warp == U - 1) row(0);
}

template <int THREADS>
__device__ void finish_fwd(const KArgs &a, const Cta &c, const PB &pb, int s, unsigned phase_id) {
    if (a.Bp <= 32 && c.stage && a.rs_smem) {
        finish_fwd_narrow<THREADS>(a, c, s, [&](int i, int b, bool lane_ok) {
            float x = row_sum1(a, c, i, b);
            if (i == 0 && c.glob && lane_ok) x += global_carry(a, c, b, phase_id);
            return x;
        });
        return;
    }
    constexpr int U = THREADS / 32;
    const int warp = threadIdx.x >> 5;
    // a first row that waits for earlier CTAs' carries goes last, to the last warp
    const int lo = c.glob ? 1 : 0;
    auto run = [&](auto st, auto rs) {
        constexpr bool ST = decltype(st)::value, RS = decltype(rs)::value;
        for (int i0 = warp * pb.RB; i0 < c.nrows; i0 += U * pb.RB)
            finish_fwd_batch<ST, RS>(a, c, pb, s, phase_id, i0, lo, c.nrows);
        if (c.glob && warp == U - 1) finish_fwd_batch<ST, RS>(a, c, pb, s, phase_id, 0, 0, 1);
    };
    dispatch_modes(c.stage, a.rs_smem != 0, run);
}

// Backward finish of rows [lo, hi) among the batch at i0, for microstep s:
// G_{s-1} = G_s (1 - leak) + row total (+ dOut of the step ending at s-1),
// then the elementwise terms of microstep q = s-1.  s == S is the prologue
// (G_{S-1} = dOut[T-1]); s == 0 leaves G_{-1} for the transpose into d_state0.
template <bool ST, bool RS>
__device__ __forceinline__ void finish_bwd_batch(const KArgs &a, const Cta &c, const PB &pb,
                                                 int s, unsigned phase_id, int i0, int lo,
                                                 int hi) {
    const int lane = threadIdx.x & 31;
    const int Bp = a.Bp, B = a.B, M = a.M;
    const size_t NBp = (size_t)a.N * Bp;
    const bool pro = s == a.S;
    const int q = s - 1;
    const int tq = q >= 0 ? q / M : 0;
    const bool step_end = q >= 0 && q - tq * M == M - 1;
    const bool first = q >= 0 && q - tq * M == M - 1;  // first visit of step tq going backwards
    const size_t ro = (size_t)c.r0 * Bp;
    const int qc = q >= a.p_off ? q : a.p_off;  // a valid slot when q < 0
    const float *Pq = prow(a, qc) + ro;
    const float *Hq = hrow(a, qc) + ro;
    const float *dO = a.dout + (size_t)tq * B * a.N + c.r0;  // [B][N] slab of step tq
    float *daq = a.da + (size_t)(q & 1) * NBp + ro;
    // d_leak, d_bias terms summed per element slot over the column chunks
    float dl[4] = {0.f, 0.f, 0.f, 0.f}, db[4] = {0.f, 0.f, 0.f, 0.f};
    for (int cb = 0; cb < pb.CB; ++cb) {
        int ii[4], bb[4];
        bool ok[4];
        float x[4], gv[4], ov[4], p[4], hv[4], lam[4];
#pragma unroll
        for (int el = 0; el < 4; ++el) {
            const int i = i0 + pb.ri[el], cc = cb * pb.cpb + pb.ci[el], b = cc * 32 + lane;
            ok[el] = pb.ri[el] < pb.RB && i >= lo && i < hi && cc < pb.NCH && b < Bp;
            ii[el] = ok[el] ? i : hi - 1;  // an initialised row, read but not used
            bb[el] = ok[el] ? b : 0;
        }
        // every load below is unconditional (from a valid address) and the
        // value is selected after, so the four elements' loads issue together
        row_sums4<RS>(a, c, ii, bb, x);
#pragma unroll
        for (int el = 0; el < 4; ++el) {
            const size_t o = (size_t)ii[el] * Bp + bb[el];
            const int bl = bb[el] < B ? bb[el] : B - 1;
            float g0, o0, p0, h0;
            lam[el] = S_prm(a)[ii[el]].x;
            if (ST) {
                g0 = S_st0(a)[o];
                o0 = S_st3(a)[ii[el] * pstride(a) + bl];
                p0 = S_st1(a)[o];
                h0 = S_st2(a)[o];
            } else {
                g0 = __ldcg(a.G_ + ro + o);
                o0 = __ldg(dO + (size_t)bl * a.N + ii[el]);
                p0 = __ldcs(Pq + o);
                h0 = __ldg(Hq + o);
            }
            x[el] = pro ? 0.f : x[el];
            gv[el] = pro ? 0.f : g0;
            ov[el] = step_end && bb[el] < B ? o0 : 0.f;
            p[el] = q >= 0 ? p0 : 0.f;
            hv[el] = q >= 0 ? h0 : 0.f;
        }
        if (!pro && lo == 0 && i0 == 0 && c.glob) {
#pragma unroll
            for (int el = 0; el < 4; ++el)
                if (pb.ri[el] == 0) x[el] += global_carry(a, c, bb[el], phase_id);
        }
        float gn[4];
#pragma unroll
        for (int el = 0; el < 4; ++el) {
            gn[el] = fmaf(gv[el], 1.f - lam[el], x[el]) + ov[el];
            if (bb[el] >= B) gn[el] = 0.f;
        }
#pragma unroll
        for (int el = 0; el < 4; ++el) {
            if (!ok[el]) continue;
            const size_t o = (size_t)ii[el] * Bp + bb[el];
            if (ST) S_st0(a)[o] = gn[el];
            else a.G_[ro + o] = gn[el];
            if (q < 0) continue;
            const bool live = bb[el] < B;
            const float d = live ? gn[el] * lam[el] * (1.f - p[el] * p[el]) : 0.f;
            if (live) {
                dl[el] = fmaf(gn[el], p[el] - hv[el], dl[el]);
                db[el] += d;
                const int sl = S_sslot(a)[ii[el]];
                if (sl >= 0 && CK_IN(a.err, sl, a.n_in)) {
                    float *dd = a.ddrives + ((size_t)tq * a.n_in + sl) * B + bb[el];
                    *dd = first ? d : *dd + d;
                }
            }
            daq[o] = d;
        }
    }
    if (q >= 0) {
        // d_leak, d_bias: per-lane partial sums per row (shared memory when
        // staged, else scratch), reduced across lanes once, in the epilogue
        float2 *lacc = ST ? S_acc(a) : a.lacc + (size_t)c.r0 * 32;
#pragma unroll
        for (int ri = 0; ri < 4; ++ri) {
            if (ri >= pb.RB) break;
            const int i = i0 + ri;
            if (i >= hi) break;
            if (i < lo) continue;
            // the element slots of row ri (value selects keep dl, db in registers)
            float sl = 0.f, sb = 0.f;
#pragma unroll
            for (int el = 0; el < 4; ++el) {
                sl += pb.ri[el] == ri ? dl[el] : 0.f;
                sb += pb.ri[el] == ri ? db[el] : 0.f;
            }
            float2 *pa = lacc + i * 32 + lane;
            const float2 o = q == a.S - 1 ? make_float2(0.f, 0.f) : *pa;
            *pa = make_float2(o.x + sl, o.y + sb);
        }
    }
}

template <int THREADS>
__device__ void finish_bwd(const KArgs &a, const Cta &c, const PB &pb, int s, unsigned phase_id) {
    if (a.Bp <= 32 && c.stage && a.rs_smem) {
        finish_bwd_narrow<THREADS>(a, c, s, [&](int i, int b, bool lane_ok) {
            float x = row_sum1(a, c, i, b);
            if (i == 0 && c.glob && lane_ok) x += global_carry(a, c, b, phase_id);
            return x;
        });
        return;
    }
    constexpr int U = THREADS / 32;
    const int warp = threadIdx.x >> 5;
    const bool defer = c.glob && s != a.S;  // the prologue has no carries to wait for
    const int lo = defer ? 1 : 0;
    auto run = [&](auto st, auto rs) {
        constexpr bool ST = decltype(st)::value, RS = decltype(rs)::value;
        for (int i0 = warp * pb.RB; i0 < c.nrows; i0 += U * pb.RB)
            finish_bwd_batch<ST, RS>(a, c, pb, s, phase_id, i0, lo, c.nrows);
        if (defer && warp == U - 1) finish_bwd_batch<ST, RS>(a, c, pb, s, phase_id, 0, 0, 1);
    };
    dispatch_modes(c.stage, a.rs_smem != 0, run);
}

// Publish this CTA's carry for the row its piece ends inside (row r0 + nrows):
// the sum of the carries of the groups holding that row's edges here.
__device__ __forceinline__ void publish_carry(const KArgs &a, const Cta &c, unsigned phase_id) {
    const int lane = threadIdx.x & 31;
    const int ka = S_srp(a)[c.nrows] > c.e0 ? S_srp(a)[c.nrows] : c.e0;
    const int ga = ka < c.e1 ? group_of(c, a.G, ka) : a.G;
    for (int b = lane; b < a.Bp; b += 32) {
        const float x = carry_sum(a, S_scarry(a) + b, ga, a.G, next_warp_group(a, ga));
        st_relaxed64(a.carry + (size_t)blockIdx.x * a.Bp + b,
                     ((unsigned long long)phase_id << 32) | __float_as_uint(x));
    }
}

// ------------------------------------------------------------------ kernel

template <int THREADS, int NC, bool SMEMG, bool BWD>
__global__ void __launch_bounds__(THREADS, kCtasPerSm) rec_kernel(const KArgs a) {
    constexpr int UNR = edge_batch(BWD, NC);
    __shared__ int s_ok, s_meta[8];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int N = a.N, Bp = a.Bp;
    const size_t NBp = (size_t)N * Bp;
    const int g = lane / a.LPE, lig = lane - (lane / a.LPE) * a.LPE;
    const bool active = g < a.EPW;
    const int gam = warp * a.EPW + g;  // this lane's group in the CTA (if active)

    const PB pb = make_pb(Bp);
    Cta c;
    c.stage = a.stage != 0;

    // bounds-checked build, test hook: one index out of range, never used
    if (a.bounds_probe && cta == 0 && tid == 0) (void)CK_IN(a.err, a.N, a.N);
    // ---- this CTA's piece of the merge path of (row ends, edges), computed
    // when the graph was built
    if (tid < 6) s_meta[tid] = __ldg(a.piece + (size_t)cta * kPieceInts + tid);
    __syncthreads();
    c.r0 = s_meta[0];
    c.nrows = s_meta[1];
    c.e0 = s_meta[2];
    c.e1 = s_meta[3];
    c.c_lo = s_meta[4];
    c.publish = s_meta[5] != 0;
    c.glob = c.c_lo < cta && c.nrows > 0;
    c.rows = a.rs_smem ? reinterpret_cast<float *>(ck_smem + a.o_rows) : a.rowsum_g + (size_t)c.r0 * Bp;
    if (c.nrows + 2 > a.rows_cap || (SMEMG && c.e1 - c.e0 > a.cap) ||
        !CK_IN(a.err, c.r0 + c.nrows, a.N + 1) || !CK_IN(a.err, c.e1, a.E + 1) ||
        !CK_IN(a.err, c.e0, c.e1 + 1)) {
        if (tid == 0) atomicCAS(a.err, 0, kDevInternal);
        return;  // every other CTA sees the error word at its next wait
    }
    for (int i = tid; i < c.nrows + 2; i += THREADS) S_srp(a)[i] = __ldg(a.row_ptr + min(c.r0 + i, N));
    for (int i = tid; i < c.nrows; i += THREADS) {
        const int r = c.r0 + i;
        S_prm(a)[i] = make_float2(__ldg(a.leak + r), BWD ? 0.f : __ldg(a.bias + r));
        S_sslot(a)[i] = __ldg(a.slot + r);
        // a row's last edge lies in this CTA iff it has edges here: then its slot
        // holds the tail, and the groups holding its earlier edges carry the rest
        const int rs = __ldg(a.row_ptr + r), re = __ldg(a.row_ptr + r + 1);
        int2 gr = make_int2(-1, 0);
        if (re > rs && re - 1 >= c.e0) {
            const int ga = group_of(c, a.G, rs > c.e0 ? rs : c.e0);
            const int gb = group_of(c, a.G, re - 1);
            gr = make_int2((ga << 16) | gb, next_warp_group(a, ga));
        }
        S_sgrp(a)[i] = gr;
    }
    // the row of each lane group's first edge (-1 past the CTA's edges)
    for (int gi = tid; gi < a.G; gi += THREADS) {
        const int n = c.e1 - c.e0;
        const int k0 = c.e0 + (int)((long long)gi * n / a.G);
        S_gst(a)[gi] = k0 < c.e1 ? __ldg(a.rowid + k0) : -1;
    }
    // the CTA's edges: {col, w[perm[k]]}, eight edges per thread
    // per pass so the independent loads (and then the dependent w loads) of a
    // pass are in flight together
    if (SMEMG || a.init_w) {
        for (int kb = c.e0 + tid; kb < c.e1; kb += 8 * THREADS) {
            int pm[8], cl[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int k = kb + j * THREADS;
                int kc = k < c.e1 ? k : c.e0;  // a valid edge, result unused
                if (!CK_IN(a.err, kc, a.E)) kc = 0;
                pm[j] = __ldg(a.perm + kc);
                cl[j] = SMEMG ? __ldg(a.col + kc) : 0;
                if (!CK_IN(a.err, pm[j], a.E)) pm[j] = 0;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int k = kb + j * THREADS;
                const float wv = __ldg(a.w + pm[j]);
                if (k >= c.e1) continue;
                if (SMEMG) {
                    S_scw(a)[k - c.e0] = make_int2(cl[j], __float_as_int(wv));
                    // a recomputing window after the first continues the sums
                    // the previous window left in dwperm
                    if (BWD) S_sdw(a)[k - c.e0] = a.zero_dw ? 0.f : __ldcg(a.dwperm + k);
                } else {
                    a.wperm[k] = wv;
                    if (BWD && a.zero_dw) a.dwperm[k] = 0.f;
                }
            }
        }
    }
    __syncthreads();
    if (c.stage && !BWD) {
        // index of each input row among this CTA's input rows (their drives are staged)
        if (tid == 0) {
            int n = 0;
            for (int i = 0; i < c.nrows; ++i) S_inp(a)[i] = S_sslot(a)[i] >= 0 ? n++ : -1;
            s_meta[6] = n;
        }
        __syncthreads();
    }
    c.n_inp = (c.stage && !BWD) ? s_meta[6] : 0;

    unsigned nbar = 0;
    if (a.do_prologue) {
        if (!BWD) {
            to_rows<THREADS>(hrow(a, 0), a.state0, c.r0, c.r0 + c.nrows, a.B, Bp, N, S_tile(a));
            for (int j = tid; j < c.nrows * Bp; j += THREADS) {
                const float v = __ldcg(hrow(a, 0) + (size_t)c.r0 * Bp + j);
                if (c.stage) {
                    const int i = j / Bp, b = j - i * Bp;
                    S_st0(a)[i * pstride(a) + b] = v;
                }
                if (a.ckpt) a.ckpt[(size_t)c.r0 * Bp + j] = v;
            }
        } else {
            if (c.stage) {
                const size_t ro = (size_t)c.r0 * Bp;
                stage_rows(S_st1(a), prow(a, a.S - 1) + ro, c.nrows, Bp, tid, THREADS);
                stage_rows(S_st2(a), hrow(a, a.S - 1) + ro, c.nrows, Bp, tid, THREADS);
                stage_dout(a, c, a.T - 1, tid, THREADS);
                cp_async_wait_all();
            }
            __syncthreads();
            finish_bwd<THREADS>(a, c, pb, a.S, 0u);
        }
        if (!grid_sync(a, nbar++, &s_ok)) return;
    }

    if (!BWD && c.stage && !a.do_prologue) {
        // a forward window that starts from a state already in H (the backward's
        // recomputation): it becomes the resident state
        for (int j = tid; j < c.nrows * Bp; j += THREADS) {
            const int i = j / Bp, b = j - i * Bp;
            S_st0(a)[i * pstride(a) + b] = __ldcg(hrow(a, a.s_first) + (size_t)c.r0 * Bp + j);
        }
        __syncthreads();
    }

    // stage mode: issue the copies of microstep s's part-B operands into
    // shared memory (threads t of nt); they land while part A runs
    auto stage_for = [&](int s, int t0, int nt) {
        const size_t ro = (size_t)c.r0 * Bp;
        if (BWD) {
            // part A's source rows: r0 .. r0 + nrows (the last one only if it exists)
            stage_rows(S_st4(a), hrow(a, s) + ro, c.r0 + c.nrows < N ? c.nrows + 1 : c.nrows,
                       Bp, t0, nt);
            cp_async_commit();  // its own group: part A waits for it alone
            if (s > 0) {
                const int q = s - 1, tq = q / a.M;
                stage_rows(S_st1(a), prow(a, q) + ro, c.nrows, Bp, t0, nt);
                stage_rows(S_st2(a), hrow(a, q) + ro, c.nrows, Bp, t0, nt);
                if (q - tq * a.M == a.M - 1) stage_dout(a, c, tq, t0, nt);
            }
        } else if (c.n_inp > 0 && s % a.M == 0) {
            const int t = s / a.M;
            for (int j = t0; j < c.nrows * a.B; j += nt) {
                const int i = j / a.B, b = j - i * a.B;
                const int ii = S_inp(a)[i];
                if (ii >= 0)
                    cp_async4(S_st1(a) + (size_t)ii * Bp + b,
                              a.drives + ((size_t)t * a.n_in + S_sslot(a)[i]) * a.B + b);
            }
        }
        cp_async_commit();
    };
    if (c.stage && a.s_count > 0) stage_for(a.s_first, tid, THREADS);

#ifdef CK_PHASE_PROFILE
    // this launch's phase sums, in registers until the microsteps end
    unsigned long long ph[4] = {0, 0, 0, 0};
    unsigned ph_steps = 0, ph_bars = 0;
#endif
    for (int it = 0; it < a.s_count; ++it) {
        const int s = BWD ? a.s_first - it : a.s_first + it;
        const unsigned phase_id = BWD ? (unsigned)(a.S - s) : (unsigned)(s + 1);
        const float *rows = BWD ? a.da + (size_t)(s & 1) * NBp : hrow(a, s);
#ifdef CK_PHASE_PROFILE
        const unsigned long long tp0 = globaltimer();
#endif
        if (!c.stage && tid == 0 && c.nrows > 0) {
            // part B's operands of this CTA's rows, fetched into L2 during part A
            const unsigned rb = (unsigned)((size_t)c.nrows * Bp * 4);
            const size_t ro = (size_t)c.r0 * Bp;
            if (BWD) {
                if (s > 0) {
                    prefetch_l2(prow(a, s - 1) + ro, rb);
                    prefetch_l2(hrow(a, s - 1) + ro, rb);
                }
            } else {
                prefetch_l2(hrow(a, s) + ro, rb);
            }
        }
        if (BWD && c.stage) {
            // st4 (h_{s-1} rows) must have landed before part A reads it; the
            // finish operands committed after it may still be in flight
            cp_async_wait_but_last();
            __syncthreads();
            part_a<NC, SMEMG, BWD, UNR, true>(a, c, gam, lig, active, rows, hrow(a, s));
        } else {
            part_a<NC, SMEMG, BWD, UNR, false>(a, c, gam, lig, active, rows, hrow(a, s));
        }
#ifdef CK_PHASE_PROFILE
        const unsigned long long tpa = globaltimer();
#endif
        if (c.stage) cp_async_wait_all();
        __syncthreads();
#ifdef CK_PHASE_PROFILE
        const unsigned long long tp1 = globaltimer();
#endif
        if (warp == THREADS / 32 - 2 && c.publish) publish_carry(a, c, phase_id);
        if (BWD) finish_bwd<THREADS>(a, c, pb, s, phase_id);
        else finish_fwd<THREADS>(a, c, pb, s, phase_id);
#ifdef CK_PHASE_PROFILE
        __syncthreads();  // the CTA's finish ends when its last warp's does
        {
            const unsigned long long tp2 = globaltimer();
            ph[0] += tpa - tp0;
            ph[1] += tp1 - tp0;
            ph[2] += tp2 - tp1;
            ++ph_steps;
        }
#endif
        if (it + 1 < a.s_count) {
            // while other CTAs finish: copy out the state that ended an input
            // step, and stage the next microstep's operands (this microstep's
            // part B has read the old ones)
            auto between = [&]() {
                if (!c.stage) return;
                if (!BWD && s % a.M == a.M - 1) write_out(a, c, s / a.M, tid, THREADS);
                stage_for(BWD ? s - 1 : s + 1, tid, THREADS);
            };
#ifdef CK_PHASE_PROFILE
            const unsigned long long tb0 = globaltimer();
#endif
            if (!grid_sync(a, nbar++, &s_ok, between)) {
                cp_async_wait_all();
                return;
            }
#ifdef CK_PHASE_PROFILE
            ph[3] += globaltimer() - tb0;
            ++ph_bars;
#endif
        }
    }
#ifdef CK_PHASE_PROFILE
    if (tid == 0 && cta < kPhaseCtas) {
        unsigned long long *q = g_phase[BWD ? 1 : 0][cta];
        unsigned sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        for (int j = 0; j < 4; ++j) q[j] += ph[j];
        q[4] += ph_steps;
        q[5] += ph_bars;
        q[6] = sm;
        q[7] = ((unsigned long long)c.nrows << 32) | (unsigned)(c.e1 - c.e0);
    }
#endif

    if (a.do_epilogue) {
        __syncthreads();
        if (!BWD) {
            if (c.stage) write_out(a, c, a.T - 1, tid, THREADS);
        } else {
            if (c.stage) {
                for (int j = tid; j < c.nrows * Bp; j += THREADS) a.G_[(size_t)c.r0 * Bp + j] = S_st0(a)[j];
                __syncthreads();
            }
            // d_leak, d_bias: each row's 32 per-lane partials, summed by a fixed
            // butterfly
            const float2 *lacc = c.stage ? S_acc(a) : a.lacc + (size_t)c.r0 * 32;
            for (int i = warp; i < c.nrows; i += THREADS / 32) {
                float2 v = lacc[i * 32 + lane];
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) {
                    v.x += __shfl_xor_sync(kFull, v.x, m);
                    v.y += __shfl_xor_sync(kFull, v.y, m);
                }
                if (lane == 0) {
                    a.dleak[c.r0 + i] = v.x;
                    a.dbias[c.r0 + i] = v.y;
                }
            }
            from_rows<THREADS>(a.dstate0, a.G_, c.r0, c.r0 + c.nrows, a.B, Bp, N, S_tile(a));
            // dw back to the caller's edge order, eight edges per thread per pass
            for (int kb = c.e0 + tid; kb < c.e1; kb += 8 * THREADS) {
                int pm[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k = kb + j * THREADS;
                    pm[j] = __ldg(a.perm + (k < c.e1 ? k : c.e0));
                    if (k < c.e1 && !CK_IN(a.err, pm[j], a.E)) pm[j] = -1;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int k = kb + j * THREADS;
                    if (k < c.e1 && pm[j] >= 0) a.dw[pm[j]] = SMEMG ? S_sdw(a)[k - c.e0] : a.dwperm[k];
                }
            }
        }
    } else if (SMEMG && BWD) {
        // a recomputing window that is not the last: its edge sums go on to the
        // next window through dwperm
        __syncthreads();
        for (int k = c.e0 + tid; k < c.e1; k += THREADS) a.dwperm[k] = S_sdw(a)[k - c.e0];
    }
}

// ------------------------------------------------------------ tiled kernels
//
// For graphs whose state rows fit a few CTAs' shared memory (chosen when the
// graph is built, ck::Tiled): the column nodes are cut into C chunks and the
// rows into G blocks, and CTA t = g * C + j (one per SM) owns cell (g, j) --
// the edges of block g whose column lies in chunk j.  Each microstep a CTA
// copies chunk j of the gathered rows (the state forward, d(pre-activation)
// backward) from global memory into shared memory with bulk asynchronous
// copies, then walks its cell exactly like part A above but gathers from
// shared memory: every gathered row is read from L2 once per CTA of its
// chunk's group, not once per edge.  The C CTAs of a block then exchange their
// partial row totals: each publishes, as {value, microstep id} words, the
// totals of the block rows the others finish, and finishes its own share of
// the block's rows with the C partials summed in chunk order (a fixed order:
// results do not depend on timing).

__device__ __forceinline__ unsigned smem_u32(const void *p) {
    return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long *m, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long *m, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(m)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(unsigned long long *m, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(m)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global to this CTA's shared memory, completing on mbarrier m.
__device__ __forceinline__ void bulk_g2s(void *sdst, const void *gsrc, unsigned bytes,
                                         unsigned long long *m) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(m))
        : "memory");
}
// Order this thread's view of memory written by other CTAs (made visible by
// an acquire) before its asynchronous-proxy copies, and the CTA's generic reads
// of shared memory before the copies overwrite it.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Wait, bounded by a.timeout_ns, for phase `parity` of mbarrier m.  Every
// thread may call it.  The copies it waits for always complete; the bound
// only guards against a fault elsewhere.
__device__ __forceinline__ bool mbar_wait(const KArgs &a, unsigned long long *m, unsigned parity) {
    if (mbar_try_wait(m, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(m, parity)) {
        if (globaltimer() - t0 > a.timeout_ns) {
            atomicCAS(a.err, 0, kDevTimeout);
            return false;
        }
    }
    return true;
}

// Issue (thread 0) the copy of `rows` rows of Bp floats from gsrc into sdst,
// in pieces of at most 32 KB; returns the bytes.
__device__ __forceinline__ unsigned bulk_rows(float *sdst, const float *gsrc, int rows, int Bp,
                                              unsigned long long *m) {
    const unsigned total = (unsigned)rows * (unsigned)Bp * 4u;
    constexpr unsigned kPiece = 32u << 10;
    for (unsigned o = 0; o < total; o += kPiece) {
        const unsigned n = total - o < kPiece ? total - o : kPiece;
        bulk_g2s(reinterpret_cast<char *>(sdst) + o, reinterpret_cast<const char *>(gsrc) + o, n, m);
    }
    return total;
}

// Partial total of block row li (block-relative) in column b published by
// CTA t of this block, waited for (bounded) until its microstep id matches.
__device__ __forceinline__ const unsigned long long *xword(const KArgs &a, int t, int li, int b) {
    return a.xbuf + ((size_t)t * a.xrows + li) * a.Bp + b;
}

template <int THREADS, bool SMEMG, bool BWD>
__global__ void __launch_bounds__(THREADS, 1) tiled_kernel(const KArgs a) {
    constexpr int NC = 1;
    constexpr int UNR = BWD ? 8 : 4;
    __shared__ int s_ok, s_meta[16];
    __shared__ __align__(8) unsigned long long s_mbar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int N = a.N, Bp = a.Bp;
    const int g = lane / a.LPE, lig = lane - (lane / a.LPE) * a.LPE;
    const bool active = g < a.EPW;
    const int gam = warp * a.EPW + g;

    if (a.bounds_probe && cta == 0 && tid == 0) (void)CK_IN(a.err, a.N, a.N);
    if (tid < kTileInts) s_meta[tid] = __ldg(a.tmeta + (size_t)cta * kTileInts + tid);
    if (tid == 0) mbar_init(&s_mbar, 1);
    __syncthreads();
    // cb: the block (part A); cf: the rows this CTA finishes
    Cta cb, cf;
    cb.r0 = s_meta[0];
    cb.nrows = s_meta[1];
    cb.e0 = s_meta[2];
    cb.e1 = s_meta[3];
    cb.c_lo = cta;
    cb.publish = false;
    cb.glob = false;
    cb.stage = true;
    cb.n_inp = 0;
    const int cn0 = s_meta[4], cnr = s_meta[5], poff = s_meta[6], f0 = s_meta[7], f1 = s_meta[8];
    const int cj = s_meta[9], cgb = s_meta[10];
    cb.rows = a.rs_smem ? reinterpret_cast<float *>(ck_smem + a.o_rows)
                        : a.rowsum_g + (size_t)cta * a.rows_cap * Bp;
    cf = cb;
    cf.r0 = cb.r0 + f0;
    cf.nrows = f1 - f0;
    if (cb.nrows + 2 > a.rows_cap || cf.nrows > a.fin_cap || f0 < 0 || f1 > cb.nrows ||
        cnr > a.chunk_cap || cnr < 0 || (SMEMG && cb.e1 - cb.e0 > a.cap) ||
        !CK_IN(a.err, cb.r0 + cb.nrows, a.N + 1) || !CK_IN(a.err, cn0 + cnr, a.N + 1) ||
        !CK_IN(a.err, cb.e1, a.E + 1) || !CK_IN(a.err, cb.e0, cb.e1 + 1) ||
        !CK_IN(a.err, cj, a.tC) || !CK_IN(a.err, cgb * a.tC + cj, a.P)) {
        if (tid == 0) atomicCAS(a.err, 0, kDevInternal);
        return;  // every other CTA sees the error word at its next wait
    }
    // ---- part A tables (block rows), from the cell's row pointers
    for (int i = tid; i < cb.nrows + 2; i += THREADS)
        S_srp(a)[i] = __ldg(a.tptr + poff + min(i, cb.nrows));
    for (int i = tid; i < cb.nrows; i += THREADS) {
        const int rs = __ldg(a.tptr + poff + i), re = __ldg(a.tptr + poff + i + 1);
        int2 gr = make_int2(-1, 0);
        if (re > rs) {
            const int ga = group_of(cb, a.G, rs);
            const int gb = group_of(cb, a.G, re - 1);
            gr = make_int2((ga << 16) | gb, next_warp_group(a, ga));
        }
        S_sgrp(a)[i] = gr;
    }
    for (int gi = tid; gi < a.G; gi += THREADS) {
        const int n = cb.e1 - cb.e0;
        const int k0 = cb.e0 + (int)((long long)gi * n / a.G);
        S_gst(a)[gi] = k0 < cb.e1 ? __ldg(a.rowid + k0) : -1;
    }
    // ---- finish tables (this CTA's rows)
    for (int i = tid; i < cf.nrows; i += THREADS) {
        const int r = cf.r0 + i;
        S_prm(a)[i] = make_float2(__ldg(a.leak + r), BWD ? 0.f : __ldg(a.bias + r));
        S_sslot(a)[i] = __ldg(a.slot + r);
    }
    // ---- the cell's edges: {column in chunk, w[perm[k]]} in shared memory, or
    // the permuted values in scratch (streamed)
    if (SMEMG || a.init_w) {
        for (int kb = cb.e0 + tid; kb < cb.e1; kb += 8 * THREADS) {
            int pm[8], cl[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int k = kb + j * THREADS;
                int kc = k < cb.e1 ? k : cb.e0;
                if (!CK_IN(a.err, kc, a.E)) kc = 0;
                pm[j] = __ldg(a.perm + kc);
                cl[j] = SMEMG ? __ldg(a.col + kc) : 0;
                if (!CK_IN(a.err, pm[j], a.E)) pm[j] = 0;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int k = kb + j * THREADS;
                const float wv = __ldg(a.w + pm[j]);
                if (k >= cb.e1) continue;
                if (SMEMG) {
                    S_scw(a)[k - cb.e0] = make_int2(cl[j], __float_as_int(wv));
                    if (BWD) S_sdw(a)[k - cb.e0] = a.zero_dw ? 0.f : __ldcg(a.dwperm + k);
                } else {
                    a.wperm[k] = wv;
                    if (BWD && a.zero_dw) a.dwperm[k] = 0.f;
                }
            }
        }
    }
    __syncthreads();
    if (!BWD) {
        if (tid == 0) {
            int n = 0;
            for (int i = 0; i < cf.nrows; ++i) S_inp(a)[i] = S_sslot(a)[i] >= 0 ? n++ : -1;
            s_meta[12] = n;
        }
        __syncthreads();
        cf.n_inp = s_meta[12];
    }

    // ---- the row total x of finished row i (relative to cf.r0), column b:
    // the C chunks' partials in chunk order, this CTA's own from its row slots
    auto tiled_x = [&](unsigned phase_id) {
        return [&a, &cb, f0, cj, cgb, phase_id](int i, int b, bool lane_ok) -> float {
            if (!lane_ok) return 0.f;
            const int li = f0 + i;
            unsigned long long w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < a.tC && j != cj) w[j] = ld_relaxed64(xword(a, cgb * a.tC + j, li, b));
            float x = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= a.tC) break;
                if (j == cj) {
                    x += row_sum1(a, cb, li, b);
                } else if ((unsigned)(w[j] >> 32) == phase_id) {
                    x += __uint_as_float((unsigned)w[j]);
                } else {
                    x += wait_carry(a, xword(a, cgb * a.tC + j, li, b), phase_id);
                }
            }
            return x;
        };
    };
    // finish operands of microstep s for this CTA's rows, copied into shared
    // memory (cp.async) while other CTAs finish
    auto stage_for = [&](int s, int t0, int nt) {
        const size_t ro = (size_t)cf.r0 * Bp;
        if (BWD) {
            if (s > 0) {
                const int q = s - 1, tq = q / a.M;
                stage_rows(S_st1(a), prow(a, q) + ro, cf.nrows, Bp, t0, nt);
                stage_rows(S_st2(a), hrow(a, q) + ro, cf.nrows, Bp, t0, nt);
                if (q - tq * a.M == a.M - 1) stage_dout(a, cf, tq, t0, nt);
            }
        } else if (cf.n_inp > 0 && s % a.M == 0) {
            const int t = s / a.M;
            for (int j = t0; j < cf.nrows * a.B; j += nt) {
                const int i = j / a.B, b = j - i * a.B;
                const int ii = S_inp(a)[i];
                if (ii >= 0)
                    cp_async4(S_st1(a) + (size_t)ii * Bp + b,
                              a.drives + ((size_t)t * a.n_in + S_sslot(a)[i]) * a.B + b);
            }
        }
        cp_async_commit();
    };

    unsigned nbar = 0;
    if (!BWD) {
        if (a.do_prologue) {
            to_rows<THREADS>(hrow(a, 0), a.state0, cf.r0, cf.r0 + cf.nrows, a.B, Bp, N, S_tile(a));
            for (int j = tid; j < cf.nrows * Bp; j += THREADS) {
                const float v = __ldcg(hrow(a, 0) + (size_t)cf.r0 * Bp + j);
                const int i = j / Bp, b = j - i * Bp;
                S_st0(a)[i * pstride(a) + b] = v;
                if (a.ckpt) a.ckpt[(size_t)cf.r0 * Bp + j] = v;
            }
            if (!grid_sync(a, nbar++, &s_ok)) return;
        } else {
            // a window that starts from a state already in H: it becomes the resident state
            for (int j = tid; j < cf.nrows * Bp; j += THREADS) {
                const int i = j / Bp, b = j - i * Bp;
                S_st0(a)[i * pstride(a) + b] = __ldcg(hrow(a, a.s_first) + (size_t)cf.r0 * Bp + j);
            }
            __syncthreads();
        }
    } else {
        if (a.do_prologue) {
            const size_t ro = (size_t)cf.r0 * Bp;
            stage_rows(S_st1(a), prow(a, a.S - 1) + ro, cf.nrows, Bp, tid, THREADS);
            stage_rows(S_st2(a), hrow(a, a.S - 1) + ro, cf.nrows, Bp, tid, THREADS);
            stage_dout(a, cf, a.T - 1, tid, THREADS);
            cp_async_wait_all();
            __syncthreads();
            finish_bwd_narrow<THREADS>(a, cf, a.S, [](int, int, bool) { return 0.f; });
            if (!grid_sync(a, nbar++, &s_ok)) return;
        } else {
            // a window that continues a backward: G and the per-lane sums from scratch
            for (int j = tid; j < cf.nrows * Bp; j += THREADS)
                S_st0(a)[j] = __ldcg(a.G_ + (size_t)cf.r0 * Bp + j);
            for (int j = tid; j < cf.nrows * 32; j += THREADS)
                S_acc(a)[j] = a.lacc[(size_t)cf.r0 * 32 + j];
            __syncthreads();
        }
    }
    if (a.s_count > 0) stage_for(a.s_first, tid, THREADS);

    for (int it = 0; it < a.s_count; ++it) {
        const int s = BWD ? a.s_first - it : a.s_first + it;
        const unsigned phase_id = BWD ? (unsigned)(a.S - s) : (unsigned)(s + 1);
        // ---- the chunk of gathered rows (and, backward, the block's rows of
        // the state entering microstep s) into shared memory
        if (tid == 0) {
            fence_proxy_async();
            const float *table = BWD ? a.da + (size_t)(s & 1) * N * Bp : hrow(a, s);
            const int hr = BWD ? min(cb.nrows + 1, N - cb.r0) : 0;
            const unsigned bytes = (unsigned)(cnr + hr) * (unsigned)Bp * 4u;
            mbar_expect_tx(&s_mbar, bytes);
            if (cnr > 0) bulk_rows(S_chunk(a), table + (size_t)cn0 * Bp, cnr, Bp, &s_mbar);
            if (hr > 0) bulk_rows(S_st4(a), hrow(a, s) + (size_t)cb.r0 * Bp, hr, Bp, &s_mbar);
        }
        if (!mbar_wait(a, &s_mbar, (unsigned)(it & 1))) {
            cp_async_wait_all();
            mbar_wait(a, &s_mbar, (unsigned)(it & 1));  // its copies, once more, before leaving
            return;
        }
        // ---- part A over the cell
        stream_piece<NC, SMEMG, BWD, UNR, BWD, true>(a, cb, gam, lig, active, nullptr, hrow(a, s));
        cp_async_wait_all();
        __syncthreads();
        // ---- publish the totals of the block rows the other CTAs finish
        for (int e = tid; e < cb.nrows * Bp; e += THREADS) {
            const int li = e / Bp, b = e - li * Bp;
            if (li >= f0 && li < f1) continue;
            const float x = row_sum1(a, cb, li, b);
            st_relaxed64(const_cast<unsigned long long *>(xword(a, cta, li, b)),
                         ((unsigned long long)phase_id << 32) | __float_as_uint(x));
        }
        // ---- finish this CTA's rows
        if (BWD) finish_bwd_narrow<THREADS>(a, cf, s, tiled_x(phase_id));
        else finish_fwd_narrow<THREADS>(a, cf, s, tiled_x(phase_id));
        if (it + 1 < a.s_count) {
            auto between = [&]() {
                if (!BWD && s % a.M == a.M - 1) write_out(a, cf, s / a.M, tid, THREADS);
                stage_for(BWD ? s - 1 : s + 1, tid, THREADS);
            };
            if (!grid_sync(a, nbar++, &s_ok, between)) {
                cp_async_wait_all();
                return;
            }
        }
    }

    __syncthreads();
    if (!BWD) {
        // the state that ends an input step, if the launch's last microstep ends one
        const int s_last = a.s_first + a.s_count - 1;
        if (a.s_count > 0 && s_last % a.M == a.M - 1) write_out(a, cf, s_last / a.M, tid, THREADS);
        return;
    }
    if (!a.do_epilogue) {
        // a window that a later one continues: G and the per-lane sums to scratch
        for (int j = tid; j < cf.nrows * Bp; j += THREADS) a.G_[(size_t)cf.r0 * Bp + j] = S_st0(a)[j];
        for (int j = tid; j < cf.nrows * 32; j += THREADS) a.lacc[(size_t)cf.r0 * 32 + j] = S_acc(a)[j];
        if (SMEMG)
            for (int k = cb.e0 + tid; k < cb.e1; k += THREADS) a.dwperm[k] = S_sdw(a)[k - cb.e0];
        return;
    }
    for (int j = tid; j < cf.nrows * Bp; j += THREADS) a.G_[(size_t)cf.r0 * Bp + j] = S_st0(a)[j];
    __syncthreads();
    for (int i = warp; i < cf.nrows; i += THREADS / 32) {
        float2 v = S_acc(a)[i * 32 + lane];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            v.x += __shfl_xor_sync(kFull, v.x, m);
            v.y += __shfl_xor_sync(kFull, v.y, m);
        }
        if (lane == 0) {
            a.dleak[cf.r0 + i] = v.x;
            a.dbias[cf.r0 + i] = v.y;
        }
    }
    from_rows<THREADS>(a.dstate0, a.G_, cf.r0, cf.r0 + cf.nrows, a.B, Bp, N, S_tile(a));
    // dw back to the caller's edge order
    for (int kb = cb.e0 + tid; kb < cb.e1; kb += 8 * THREADS) {
        int pm[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int k = kb + j * THREADS;
            pm[j] = __ldg(a.perm + (k < cb.e1 ? k : cb.e0));
            if (k < cb.e1 && !CK_IN(a.err, pm[j], a.E)) pm[j] = -1;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int k = kb + j * THREADS;
            if (k < cb.e1 && pm[j] >= 0) a.dw[pm[j]] = SMEMG ? S_sdw(a)[k - cb.e0] : a.dwperm[k];
        }
    }
}

// ------------------------------------------------------------------ host

using KernelFn = void (*)(const KArgs);

template <int THREADS, bool BWD>
KernelFn pick_nc(int nc, bool smem) {
    if (nc == 2) return smem ? rec_kernel<THREADS, 2, true, BWD> : rec_kernel<THREADS, 2, false, BWD>;
    return smem ? rec_kernel<THREADS, 4, true, BWD> : rec_kernel<THREADS, 4, false, BWD>;
}

KernelFn pick_kernel(int nc, bool smem, bool bwd) {
    return bwd ? pick_nc<kThreads, true>(nc, smem) : pick_nc<kThreads, false>(nc, smem);
}

KernelFn pick_tiled(bool smem, bool bwd) {
    if (bwd) return smem ? tiled_kernel<kTiledThreads, true, true> : tiled_kernel<kTiledThreads, false, true>;
    return smem ? tiled_kernel<kTiledThreads, true, false> : tiled_kernel<kTiledThreads, false, false>;
}

// The kernel, grid and block of one direction's launch under plan p.
struct LaunchShape {
    KernelFn fn;
    int grid, block, per_sm;
};
LaunchShape launch_shape(const Plan &p, const SmemLayout &L, bool bwd) {
    if (p.tiled) return {pick_tiled(L.graph, bwd), p.tP[bwd ? 1 : 0], kTiledThreads, 1};
    return {pick_kernel(p.NC, L.graph, bwd), p.P, p.threads, kCtasPerSm};
}

int pow2ceil(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// Shared-memory layout of one direction.
SmemLayout smem_layout(const Plan &p, int dir, bool want_graph, bool want_stage,
                       bool want_rows = true) {
    SmemLayout L;
    std::memset(&L, 0, sizeof(L));
    size_t o = 0;
    const int rc = p.rows_cap[dir];
    L.o_srp = (int)o; o = align16(o + 4 * (size_t)rc);
    L.o_prm = (int)o; o = align16(o + 8 * (size_t)rc);
    L.o_slot = (int)o; o = align16(o + 4 * (size_t)rc);
    L.o_grp = (int)o; o = align16(o + 8 * (size_t)rc);
    L.o_carry = (int)o; o = align16(o + 4 * (size_t)p.groups * p.Bp);
    L.o_tile = (int)o; o = align16(o + 4 * 32 * 33);
    L.o_gst = (int)o; o = align16(o + 4 * (size_t)p.groups);
    // kCtasPerSm CTAs share the SM's shared memory, 1 KB of it reserved per CTA
    const size_t budget = std::min<size_t>(kMaxSmem, kSmemPerSm / kCtasPerSm - 1024) - kStaticSmem;
    const size_t rows_b = align16(4 * (size_t)rc * p.Bp);
    const size_t rows_pb = align16(4 * (size_t)rc * (p.Bp + 1));  // row stride Bp + 1
    const size_t graph_b = (dir == 0 ? 8 : 12) * (size_t)p.cap[dir] + 32;
    // finish operands: forward state + drives; backward G, A, H, dOut + two sums
    const size_t stage_b = (dir == 0 ? 1 : 4) * rows_b + rows_pb + (dir == 1 ? 8 * 32 * (size_t)rc : 0) +
                           align16(4 * (size_t)rc);
    L.rows = want_rows && o + rows_b <= budget;
    if (L.rows) o += rows_b;
    L.o_rows = (int)(o - (L.rows ? rows_b : 0));
    L.graph = want_graph && o + graph_b <= budget;
    L.o_cw = (int)o; o = align16(o + (L.graph ? 8 * (size_t)p.cap[dir] : 0));

    L.o_dw = (int)o; o = align16(o + (L.graph && dir == 1 ? 4 * (size_t)p.cap[dir] : 0));
    L.stage = want_stage && o + stage_b <= budget;
    const size_t sb = L.stage ? rows_b : 0, spb = L.stage ? rows_pb : 0;
    L.o_st0 = (int)o; o += dir == 0 ? spb : sb;
    L.o_st1 = (int)o; o += sb;
    L.o_st2 = (int)o; o += dir == 1 ? sb : 0;
    L.o_st3 = (int)o; o += dir == 1 ? spb : 0;
    L.o_st4 = (int)o; o += dir == 1 ? sb : 0;
    L.o_acc = (int)o; o = align16(o + (L.stage && dir == 1 ? 8 * 32 * (size_t)rc : 0));
    L.o_inp = (int)o; o = align16(o + (L.stage ? 4 * (size_t)rc : 0));
    // a streamed graph's cp.async ring, in what is left: the largest of a few
    // (chunks, log2 batches per chunk) shapes that fits
    L.o_ring = (int)o;
    L.ring_n = L.ring_chb_sh = 0;
    if (!L.graph && kStreamRing) {
        const int unr = edge_batch(dir == 1, p.NC);
        static const int shapes[4][2] = {{4, 2}, {4, 1}, {2, 1}, {2, 0}};
        for (const auto &sh : shapes) {
            const size_t b = 8 * (size_t)p.groups * sh[0] * ((size_t)unr << sh[1]);
            if (o + b <= budget) {
                L.ring_n = sh[0];
                L.ring_chb_sh = sh[1];
                o = align16(o + b);
                break;
            }
        }
    }
    L.bytes = o;
    return L;
}

// Shared-memory layout of a tiled kernel (one CTA per SM).  Required: the
// chunk of gathered rows and, backward, the block's rows of the state (both
// bulk-copy destinations, 128-byte aligned), the part A tables, the finish
// tables and staged operands of the rows the CTA finishes.  Then, if they fit:
// the row slots (else in scratch) and the cell's graph slice (else streamed).
// `fits` is false when the required part exceeds the budget.
constexpr size_t kTiledBudget = (size_t)kMaxSmem - 512;  // static shared memory below 512 bytes

SmemLayout tiled_layout(int dir, int Bp, int groups, int rows_cap, int fin_cap, int chunk_cap,
                        int ecap, bool want_graph, bool want_rows, bool *fits) {
    SmemLayout L;
    std::memset(&L, 0, sizeof(L));
    auto a128 = [](size_t x) { return (x + 127) & ~(size_t)127; };
    size_t o = 0;
    L.o_chunk = (int)o; o = a128(o + 4 * (size_t)chunk_cap * Bp);
    L.o_st4 = (int)o; o = a128(o + (dir == 1 ? 4 * (size_t)rows_cap * Bp : 0));
    L.o_srp = (int)o; o = align16(o + 4 * (size_t)rows_cap);
    L.o_grp = (int)o; o = align16(o + 8 * (size_t)rows_cap);
    L.o_gst = (int)o; o = align16(o + 4 * (size_t)groups);
    L.o_carry = (int)o; o = align16(o + 4 * (size_t)groups * Bp);
    L.o_tile = (int)o; o = align16(o + 4 * 32 * 33);
    const size_t F = (size_t)fin_cap + 1;
    L.o_prm = (int)o; o = align16(o + 8 * F);
    L.o_slot = (int)o; o = align16(o + 4 * F);
    L.o_inp = (int)o; o = align16(o + (dir == 0 ? 4 * F : 0));
    const size_t fr = align16(4 * F * Bp), frp = align16(4 * F * (Bp + 1));
    L.o_st0 = (int)o; o += dir == 0 ? frp : fr;
    L.o_st1 = (int)o; o += fr;
    L.o_st2 = (int)o; o += dir == 1 ? fr : 0;
    L.o_st3 = (int)o; o += dir == 1 ? frp : 0;
    L.o_acc = (int)o; o = align16(o + (dir == 1 ? 8 * 32 * F : 0));
    L.stage = true;
    *fits = o <= kTiledBudget;
    const size_t rows_b = align16(4 * (size_t)rows_cap * Bp);
    L.rows = want_rows && o + rows_b <= kTiledBudget;
    L.o_rows = (int)o;
    if (L.rows) o += rows_b;
    const size_t graph_b = align16(8 * (size_t)ecap) + (dir == 1 ? align16(4 * (size_t)ecap) : 0);
    L.graph = want_graph && o + graph_b <= kTiledBudget;
    L.o_cw = (int)o; o = align16(o + (L.graph ? 8 * (size_t)ecap : 0));
    L.o_dw = (int)o; o = align16(o + (L.graph && dir == 1 ? 4 * (size_t)ecap : 0));
    L.bytes = o;
    return L;
}

void fill_common(KArgs &k, const ck_graph *g, const Plan &p, void *scratch, int dir,
                 const SmemLayout *layout = nullptr) {
    std::memset(&k, 0, sizeof(k));
    k.N = p.N;
    k.E = p.E;
    k.n_in = p.n_in;
    k.B = p.B;
    k.Bp = p.Bp;
    k.LPE = p.LPE;
    k.EPW = p.EPW;
    k.LPE_P2 = pow2ceil(p.LPE);
    k.T = p.T;
    k.M = p.M;
    k.S = p.S;
    k.P = p.P;
    k.G = p.groups;
    k.cap = p.cap[dir];
    k.rows_cap = p.rows_cap[dir];
    const SmemLayout &L = layout ? *layout : dir == 0 ? p.lay_fwd : p.lay_bwd;
    k.rs_smem = L.rows ? 1 : 0;
    k.o_srp = L.o_srp;
    k.o_prm = L.o_prm;
    k.o_slot = L.o_slot;
    k.o_grp = L.o_grp;
    k.o_carry = L.o_carry;
    k.o_rows = L.o_rows;
    k.o_tile = L.o_tile;
    k.o_cw = L.o_cw;
    k.o_gst = L.o_gst;
    k.o_dw = L.o_dw;
    k.stage = L.stage ? 1 : 0;
    k.o_st0 = L.o_st0;
    k.o_st1 = L.o_st1;
    k.o_st2 = L.o_st2;
    k.o_st3 = L.o_st3;
    k.o_st4 = L.o_st4;
    k.o_inp = L.o_inp;
    k.o_acc = L.o_acc;
    k.slot = g->slot;
    char *sc = (char *)scratch;
    auto region = [&](size_t off) -> char * { return off == kNoRegion ? nullptr : sc + off; };
    k.bar = (unsigned *)(sc + p.off_ctrl);
    k.err = (int *)(sc + p.off_ctrl + kStatusOffset);
    k.carry = (unsigned long long *)region(p.off_carry);
    k.wperm = (float *)region(p.off_wperm);
    k.dwperm = (float *)region(p.off_dwperm);
    k.G_ = (float *)region(p.off_G);
    k.da = (float *)region(p.off_da);
    k.rowsum_g = (float *)region(p.off_rowsum);
    k.lacc = (float2 *)region(p.off_lacc);
    k.bar_extra = (unsigned)options().barrier_extra;
    k.timeout_ns = (unsigned long long)options().timeout_ns;
    k.bounds_probe = options().bounds_probe;
    k.o_chunk = L.o_chunk;
    k.o_ring = L.o_ring;
    k.ring_n = L.ring_n;
    k.ring_chb_sh = L.ring_chb_sh;
    if (p.tiled) {
        const Tiled &t = g->tiled[dir];
        k.P = p.tP[dir];
        k.tmeta = t.meta;
        k.tptr = t.ptr;
        k.chunk_cap = p.chunk_cap[dir];
        k.fin_cap = p.fin_cap[dir];
        k.tC = t.C;
        k.xrows = p.xrows;
        k.xbuf = (unsigned long long *)region(p.off_xbuf);
    }
}

// The graph arrays of direction dir: the compressed rows (and their pieces),
// or the tiling's cells.
void set_graph(KArgs &k, const ck_graph *g, const Plan &p, int dir) {
    if (p.tiled) {
        const Tiled &t = g->tiled[dir];
        k.col = t.col;
        k.perm = t.perm;
        k.rowid = t.rowid;
        return;
    }
    k.row_ptr = dir == 0 ? g->row_ptr : g->rowT_ptr;
    k.piece = g->piece[dir][pass_index(p.Bp)];
    k.col = dir == 0 ? g->col : g->colT;
    k.perm = dir == 0 ? g->perm : g->permT;
    k.rowid = dir == 0 ? g->rowid : g->rowidT;
}

// One cooperative launch of the kernel for layout L with k's microstep range
// and flags as given; the control words are cleared first.
ck_status launch_once(KArgs &k, const Plan &p, const SmemLayout &L, bool bwd, cudaStream_t s) {
    const LaunchShape sh = launch_shape(p, L, bwd);
    cudaError_t e = cudaFuncSetAttribute((const void *)sh.fn,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    e = cudaMemsetAsync((char *)k.bar, 0, p.clear_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (control words)");
    void *args[] = {&k};
    e = cudaLaunchCooperativeKernel((const void *)sh.fn, dim3(sh.grid), dim3(sh.block), args, L.bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchCooperativeKernel");
    return CK_OK;
}

ck_status launch_all(KArgs &k, const Plan &p, bool bwd, cudaStream_t s, int64_t *launches) {
    const SmemLayout &L = bwd ? p.lay_bwd : p.lay_fwd;
    const LaunchShape sh = launch_shape(p, L, bwd);
    KernelFn fn = sh.fn;
    cudaError_t e = cudaFuncSetAttribute((const void *)fn,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void *)fn, sh.block, L.bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (per_sm < sh.per_sm)
        return fail(CK_ERR_UNSUPPORTED, "%d CTAs of %d threads and %zu B shared do not fit on an SM",
                    sh.per_sm, sh.block, L.bytes);
    // barrier counter, status word, published carries and partial totals start at zero
    e = cudaMemsetAsync((char *)k.bar, 0, p.clear_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (control words)");
    int64_t n = 0;
    const bool persistent = options().persistent != 0;
    const int S = p.S;
    const int steps = persistent ? 1 : S;
    for (int i = 0; i < steps; ++i) {
        KArgs ki = k;
        ki.init_w = ki.zero_dw = persistent || i == 0;
        if (persistent) {
            ki.s_first = bwd ? S - 1 : 0;
            ki.s_count = S;
            ki.do_prologue = 1;
            ki.do_epilogue = 1;
            ki.bar_base = 0;
        } else {
            ki.s_first = bwd ? S - 1 - i : i;
            ki.s_count = 1;
            ki.do_prologue = i == 0;
            ki.do_epilogue = i == S - 1;
            ki.bar_base = i == 0 ? 0u : 1u;
        }
        void *args[] = {&ki};
        e = cudaLaunchCooperativeKernel((const void *)fn, dim3(sh.grid), dim3(sh.block), args, L.bytes,
                                        s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchCooperativeKernel");
        ++n;
    }
    if (launches) *launches = n;
    return CK_OK;
}

}  // namespace

bool tiled_fits(int dir, int Bp, int max_rows, int max_fin, int max_chunk) {
    const int lpe = Bp / 4, epw = 32 / lpe;
    bool fits = false;
    tiled_layout(dir, Bp, (kTiledThreads / 32) * epw, max_rows + 3, max_fin, max_chunk, 0, false,
                 false, &fits);
    return fits;
}

ck_status make_plan(const ck_graph *g, int64_t B, int64_t T, int64_t M, Plan *p) {
    if (B < 1 || T < 1 || M < 1) return fail(CK_ERR_INVALID_ARG, "B, T and microsteps must be >= 1");
    if (B > 512) return fail(CK_ERR_UNSUPPORTED, "B = %lld > 512 is not supported", (long long)B);
    if (T * M > (int64_t)1 << 30) return fail(CK_ERR_UNSUPPORTED, "T * microsteps too large");
    Plan q;
    std::memset(&q, 0, sizeof(q));
    q.N = (int)g->N;
    q.E = (int)g->E;
    q.n_in = (int)g->n_in;
    q.B = (int)B;
    // a lane holds NC float4 chunks of a batch row; LPE lanes hold the row
    q.Bp = (int)(B > 16 && B <= 32 ? 32 : B <= 256 ? (B + 7) / 8 * 8 : (B + 15) / 16 * 16);
    q.NC = q.Bp <= 256 ? 2 : 4;
    q.LPE = q.Bp / (4 * q.NC);
    q.EPW = 32 / q.LPE;
    q.T = (int)T;
    q.M = (int)M;
    q.S = (int)(T * M);
    q.P = num_pieces(g);
    q.threads = kThreads;
    q.warps = q.threads / 32;
    q.groups = q.warps * q.EPW;
    for (int d = 0; d < 2; ++d) {
        q.cap[d] = g->max_edges[d][pass_index(q.Bp)] + 1;
        q.rows_cap[d] = g->max_rows[d][pass_index(q.Bp)] + 3;
    }
    const bool want_graph = options().graph_in_smem && options().persistent;
    const bool want_stage = options().persistent != 0;
    const bool want_rows = options().rows_in_smem != 0;
    // tiled kernels: a tiling in both directions and at most 32 padded columns
    q.tiled = options().tiled && g->tiled[0].C > 0 && g->tiled[1].C > 0 && B <= kTiledMaxBp;
    if (q.tiled) {
        q.Bp = (int)((B + 3) / 4 * 4);
        q.NC = 1;
        q.LPE = q.Bp / 4;
        q.EPW = 32 / q.LPE;
        q.threads = kTiledThreads;
        q.warps = q.threads / 32;
        q.groups = q.warps * q.EPW;
        q.xrows = 0;
        q.P = 0;
        bool ok = true;
        for (int d = 0; d < 2; ++d) {
            const Tiled &t = g->tiled[d];
            q.tP[d] = t.P;
            q.P = std::max(q.P, t.P);
            q.cap[d] = t.max_edges + 1;
            q.rows_cap[d] = t.max_rows + 3;
            q.fin_cap[d] = t.max_fin;
            q.chunk_cap[d] = t.max_chunk;
            q.xrows = std::max(q.xrows, t.max_rows);
        }
        bool f0 = false, f1 = false, f2 = false;
        // the graph slice stays in global memory with one launch per microstep, as above
        q.lay_fwd = tiled_layout(0, q.Bp, q.groups, q.rows_cap[0], q.fin_cap[0], q.chunk_cap[0],
                                 q.cap[0], want_graph, want_rows, &f0);
        q.lay_bwd = tiled_layout(1, q.Bp, q.groups, q.rows_cap[1], q.fin_cap[1], q.chunk_cap[1],
                                 q.cap[1], want_graph, want_rows, &f1);
        q.lay_bwd_flat = tiled_layout(1, q.Bp, q.groups, q.rows_cap[1], q.fin_cap[1],
                                      q.chunk_cap[1], q.cap[1], false, want_rows, &f2);
        ok = f0 && f1 && f2;
        if (!ok) return fail(CK_ERR_INTERNAL, "tiled layout does not fit although the build checked it");
    } else {
        q.lay_fwd = smem_layout(q, 0, want_graph, want_stage, want_rows);
        q.lay_bwd = smem_layout(q, 1, want_graph, want_stage, want_rows);
        // the recomputing backward runs in windows of K input steps (one launch
        // each): the CTA's graph slice and edge sums in shared memory when they
        // fit (the sums carried between windows through dwperm), every other
        // accumulator in global memory
        q.lay_bwd_flat = smem_layout(q, 1, want_graph, false, want_rows);
        const size_t cta_smem = std::min<size_t>(kMaxSmem, kSmemPerSm / kCtasPerSm - 1024) - kStaticSmem;
        if (q.lay_fwd.bytes > cta_smem || q.lay_bwd.bytes > cta_smem || q.lay_bwd_flat.bytes > cta_smem)
            return fail(CK_ERR_UNSUPPORTED, "per-CTA tables exceed shared memory (rows per SM too many)");
    }
    const size_t NBp = (size_t)q.N * q.Bp;
    const size_t E1 = (size_t)(q.E > 0 ? q.E : 1);
    size_t off = 0;
    q.off_ctrl = off;
    q.ctrl_bytes = kCtrlBytes;
    off += q.ctrl_bytes;
    q.off_carry = off;
    off = align256(off + 8 * (size_t)q.P * q.Bp);
    q.off_xbuf = off;
    off = align256(off + (q.tiled ? 8 * (size_t)q.P * q.xrows * q.Bp : 0));
    q.clear_bytes = off - q.off_ctrl;
    q.off_wperm = off;
    off = align256(off + 4 * E1);
    q.off_dwperm = off;
    off = align256(off + 4 * E1);
    q.off_G = off;
    off = align256(off + 4 * NBp);
    q.off_da = off;
    off = align256(off + 8 * NBp);
    q.off_rowsum = off;
    // row slots out of shared memory: per row, or (tiled) per CTA and block row
    off = align256(off + 4 * std::max(NBp, q.tiled ? (size_t)q.P * q.rows_cap[0] * q.Bp +
                                                         (size_t)q.P * q.rows_cap[1] * q.Bp : 0));
    q.off_lacc = off;
    off = align256(off + 8 * 32 * (size_t)q.N);
    q.scratch_bytes = off;
    // recomputation windows (after the regular scratch): KM + 1 states and KM
    // proposals of K input steps; the checkpointing forward's two state slots
    // use the first two.  K defaults to about sqrt(T), which balances the
    // windows against the checkpoints and makes 2 ceil(T / K) launches
    {
        const int want = options().recompute_steps;
        int K = want > 0 ? want : (int)std::lround(std::sqrt((double)q.T));
        q.rc_steps = std::max(1, std::min(K, q.T));
    }
    const size_t KM = (size_t)q.rc_steps * q.M;
    q.off_hwin = off;
    off = align256(off + 4 * NBp * (KM + 1));
    q.off_pwin = off;
    off = align256(off + 4 * NBp * KM);
    q.scratch_bytes_rc = off;
    q.ckpt_bytes = 4 * NBp * (size_t)(q.T + 1);
    q.saved_bytes = 4 * NBp * (size_t)(2 * q.S + 1);
    *p = q;
    return CK_OK;
}

void forward_only_scratch(Plan *q) {
    size_t off = 0;
    q->off_ctrl = off;
    off += q->ctrl_bytes;
    q->off_carry = off;
    off = align256(off + 8 * (size_t)q->P * q->Bp);
    q->off_xbuf = off;
    off = align256(off + (q->tiled ? 8 * (size_t)q->P * q->xrows * q->Bp : 0));
    q->clear_bytes = off - q->off_ctrl;
    q->off_wperm = off;
    off = align256(off + 4 * (size_t)(q->E > 0 ? q->E : 1));
    q->off_rowsum = off;
    off = align256(off + 4 * std::max((size_t)q->N * q->Bp,
                                      q->tiled ? (size_t)q->P * q->rows_cap[0] * q->Bp : 0));
    q->off_dwperm = q->off_G = q->off_da = q->off_lacc = kNoRegion;
    q->off_hwin = q->off_pwin = kNoRegion;
    q->scratch_bytes = off;
}

ck_status launch_forward(const ck_graph *g, const Plan &p, const FwdIO &io, cudaStream_t s,
                         int64_t *launches) {
    KArgs k;
    fill_common(k, g, p, io.scratch, 0);
    set_graph(k, g, p, 0);
    k.w = io.w;
    k.leak = io.leak;
    k.bias = io.bias;
    k.drives = io.drives;
    k.state0 = io.state0;
    k.out = io.out;
    k.H = io.saved;
    k.Pr = io.saved + (size_t)(p.S + 1) * p.N * p.Bp;
    return launch_all(k, p, false, s, launches);
}

ck_status launch_forward_ckpt(const ck_graph *g, const Plan &p, const FwdIO &io, cudaStream_t s,
                              int64_t *launches) {
    KArgs k;
    fill_common(k, g, p, io.scratch, 0);
    set_graph(k, g, p, 0);
    k.w = io.w;
    k.leak = io.leak;
    k.bias = io.bias;
    k.drives = io.drives;
    k.state0 = io.state0;
    k.out = io.out;
    k.H = (float *)((char *)io.scratch + p.off_hwin);  // two state slots, used in turn
    k.h_mod = 2;
    k.Pr = nullptr;
    k.ckpt = io.saved;
    return launch_all(k, p, false, s, launches);
}

ck_status launch_backward_recompute(const ck_graph *g, const Plan &p, const RcIO &io,
                                    cudaStream_t s, int64_t *launches) {
    const size_t NBp = (size_t)p.N * p.Bp;
    float *hwin = (float *)((char *)io.scratch + p.off_hwin);
    float *pwin = (float *)((char *)io.scratch + p.off_pwin);
    const int M = p.M, T = p.T, S = p.S, K = p.rc_steps;
    int64_t n = 0;
    // windows [t, t1) of K input steps from the top (the lowest may be shorter)
    for (int t1 = T; t1 > 0; t1 -= K) {
        const int t = t1 > K ? t1 - K : 0, k = t1 - t;
        // microsteps tM .. t1 M - 1 again, from the checkpoint of step t:
        // states into window slots 0..kM, proposals into slots 0..kM-1
        cudaError_t e = cudaMemcpyAsync(hwin, io.ckpt + (size_t)t * NBp, 4 * NBp,
                                        cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync (checkpoint)");
        KArgs kf;
        fill_common(kf, g, p, io.scratch, 0);
        set_graph(kf, g, p, 0);
        kf.w = io.w;
        kf.leak = io.leak;
        kf.bias = io.bias;
        kf.drives = io.drives;
        kf.H = hwin;
        kf.h_off = t * M;
        kf.Pr = pwin;
        kf.p_off = t * M;
        kf.s_first = t * M;
        kf.s_count = k * M;
        kf.do_prologue = 0;
        kf.do_epilogue = 0;
        kf.init_w = 1;  // the backward windows overwrite the shared permuted values
        ck_status st = launch_once(kf, p, p.lay_fwd, false, s);
        if (st != CK_OK) return st;
        ++n;
        // the backward iterations whose elementwise terms belong to steps t ..
        // t1 - 1: s = t1 M .. tM + 1 (the first is the prologue for the last
        // step), and s = 0 after step 0
        KArgs kb;
        fill_common(kb, g, p, io.scratch, 1, &p.lay_bwd_flat);
        set_graph(kb, g, p, 1);
        kb.w = io.w;
        kb.leak = io.leak;
        kb.H = hwin;
        kb.h_off = t * M;
        kb.Pr = pwin;
        kb.p_off = t * M;
        kb.dout = io.dout;
        kb.dw = io.dw;
        kb.dleak = io.dleak;
        kb.dbias = io.dbias;
        kb.ddrives = io.ddrives;
        kb.dstate0 = io.dstate0;
        const bool last_step = t1 == T;
        kb.do_prologue = last_step ? 1 : 0;
        kb.s_first = last_step ? S - 1 : t1 * M;
        kb.s_count = (last_step ? k * M - 1 : k * M) + (t == 0 ? 1 : 0);
        kb.do_epilogue = t == 0 ? 1 : 0;
        kb.init_w = 1;
        kb.zero_dw = last_step ? 1 : 0;
        st = launch_once(kb, p, p.lay_bwd_flat, true, s);
        if (st != CK_OK) return st;
        ++n;
    }
    if (launches) *launches = n;
    return CK_OK;
}

ck_status launch_backward(const ck_graph *g, const Plan &p, const BwdIO &io, cudaStream_t s,
                          int64_t *launches) {
    KArgs k;
    fill_common(k, g, p, io.scratch, 1);
    set_graph(k, g, p, 1);
    k.w = io.w;
    k.leak = io.leak;
    k.H = const_cast<float *>(io.saved);
    k.Pr = const_cast<float *>(io.saved) + (size_t)(p.S + 1) * p.N * p.Bp;
    k.dout = io.dout;
    k.dw = io.dw;
    k.dleak = io.dleak;
    k.dbias = io.dbias;
    k.ddrives = io.ddrives;
    k.dstate0 = io.dstate0;
    return launch_all(k, p, true, s, launches);
}

}  // namespace ck

using namespace ck;

extern "C" ck_status ck_phase_profile_read(uint64_t *host, int64_t words, int64_t clear) {
#ifndef CK_PHASE_PROFILE
    (void)host;
    (void)words;
    (void)clear;
    return fail(CK_ERR_UNSUPPORTED, "phase profile: only the profiling build (libck_prof.so) keeps one");
#else
    const size_t n = sizeof(g_phase) / sizeof(unsigned long long);
    if (!host || words < (int64_t)n)
        return fail(CK_ERR_INVALID_ARG, "phase profile: host buffer of %zu words needed", n);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize (phase profile)");
    e = cudaMemcpyFromSymbol(host, g_phase, sizeof(g_phase));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol (phase profile)");
    if (clear) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_phase);
        if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(g_phase));
        if (e != cudaSuccess) return cuda_fail(e, "clearing the phase profile");
    }
    return CK_OK;
#endif
}
