// Forward and backward of the leaky-tanh recurrence over a fixed sparse graph.
//
// connectome-kernels page:
//   intro           proposal = tanh(W h + drive + bias); h <- (1-leak) h +
//                   leak * proposal, `microsteps` times per input step; one
//                   fused forward per microstep; the backward has elementwise
//                   terms with per-node row reductions, a transposed sparse
//                   product for the state gradient and a per-edge dot product
//                   over the batch for the edge gradient.  Everything fp32.
//   "Design notes"  states stored [N, B] so a node's batch row is contiguous;
//                   rows with many edges split across warps with an on-chip
//                   reduction; transposed CSR for the state gradient; state and
//                   pre-activation saved after every microstep.
//
// Layout in device memory (all fp32, rows padded to Bp = B rounded up to 8):
//   H[s+1][N][Bp]  state after microstep s; H[0] = state0 transposed
//   A[s][N][Bp]    pre-activation of microstep s
//   G[N][Bp]       running state gradient (backward)
//   da[2][N][Bp]   d(loss)/d(pre-activation), ping-pong between microsteps
//
// Work split.  One CTA per SM, one persistent cooperative launch per call;
// microsteps are separated by a grid-wide barrier whose wait is bounded.  The
// rows and edges of the compressed layout are cut into P*U equal pieces along
// the merge path of (row ends, edges) -- every warp gets the same number of
// row ends plus edges, so a hub row is spread over as many warps (and CTAs) as
// its size asks for.  A warp sums whole rows itself; a row cut by a piece
// boundary leaves partial sums ("carries") that the warp owning the row's end
// adds up in a fixed order after a CTA barrier (shared memory) or, across
// CTAs, after a flag the producing CTA publishes (global memory).  No atomics
// touch values, and the summation order never depends on timing.
//
// Lanes.  A warp processes EPW edges at once; each edge's batch row is read by
// LPE lanes with 16-byte loads (LPE = Bp/4 when Bp <= 128, else 32 lanes that
// loop over NC column chunks of 128).
//
// When one CTA's slice of the graph fits in shared memory it is loaded there
// once per call (column ids, edge values in row order, and the edge-gradient
// accumulators in the backward); otherwise it is read from global memory in
// every microstep.
#include <algorithm>
#include <cstring>

#include "ck_internal.h"

namespace ck {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxSmem = 227 * 1024;
constexpr int kSmemReserve = 2048;  // static shared memory and slack

struct KArgs {
    int N, E, n_in, B, Bp, LPE, EPW, LPE_P2, EPW_P2, T, M, S;
    int P, U, cap;
    const int *row_ptr, *col, *perm, *slot;
    const float *w, *leak, *bias, *drives, *state0;
    float *out;
    float *H, *A;
    const float *dout;
    float *dw, *dleak, *dbias, *ddrives, *dstate0;
    float *G, *da;
    unsigned *bar;
    int *err;
    unsigned *flags;
    float *carry, *wperm, *dwperm;
    int s_first, s_count, do_prologue, do_epilogue;
    unsigned bar_base, bar_extra;
    unsigned long long timeout_ns;
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ int ld_err(const int *p) { return *(volatile const int *)p; }

__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ void fma4(float4 &a, float w, const float4 &x) {
    a.x = fmaf(w, x.x, a.x);
    a.y = fmaf(w, x.y, a.y);
    a.z = fmaf(w, x.z, a.z);
    a.w = fmaf(w, x.w, a.w);
}
__device__ __forceinline__ void add4(float4 &a, const float4 &x) {
    a.x += x.x;
    a.y += x.y;
    a.z += x.z;
    a.w += x.w;
}
__device__ __forceinline__ float4 shfl_down4(const float4 &v, int d) {
    return make_float4(__shfl_down_sync(kFull, v.x, d), __shfl_down_sync(kFull, v.y, d),
                       __shfl_down_sync(kFull, v.z, d), __shfl_down_sync(kFull, v.w, d));
}
__device__ __forceinline__ float f4get(const float4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}
__device__ __forceinline__ void f4set(float4 &v, int q, float x) {
    if (q == 0) v.x = x;
    else if (q == 1) v.y = x;
    else if (q == 2) v.z = x;
    else v.w = x;
}

// Lane roles inside a warp.
struct Lanes {
    int lane, g, lig;
    bool active;  // g < EPW
    bool lead;    // g == 0: writes a row's results
};

__device__ __forceinline__ Lanes make_lanes(const KArgs &a, int lane) {
    Lanes L;
    L.lane = lane;
    L.g = lane / a.LPE;
    L.lig = lane - L.g * a.LPE;
    L.active = L.g < a.EPW;
    L.lead = L.g == 0;
    return L;
}
template <int NC>
__device__ __forceinline__ int col_of(const Lanes &L, int c) {
    return c * 128 + L.lig * 4;
}

// Sum over the LPE lanes of each group; valid in the group's lane lig == 0.
__device__ __forceinline__ float group_sum(float v, const KArgs &a, const Lanes &L) {
    for (int o = a.LPE_P2 >> 1; o >= 1; o >>= 1) {
        float y = __shfl_down_sync(kFull, v, o);
        if (L.lig + o < a.LPE) v += y;
    }
    return v;
}

// Sum the EPW groups' partial rows into group 0.
template <int NC>
__device__ __forceinline__ void reduce_groups(float4 (&acc)[NC], const KArgs &a, const Lanes &L) {
    for (int o = a.EPW_P2 >> 1; o >= 1; o >>= 1) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            float4 y = shfl_down4(acc[c], o * a.LPE);
            if (L.g + o < a.EPW) add4(acc[c], y);
        }
    }
}

// Grid-wide barrier, bounded by a.timeout_ns.  Returns false (for the whole
// CTA) once any CTA has recorded an error, so every CTA leaves together.
__device__ bool grid_sync(const KArgs &a, unsigned idx, int *s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned target = (a.bar_base + idx + 1u) * (unsigned)a.P + a.bar_extra;
        __threadfence();
        atomicAdd(a.bar, 1u);
        const unsigned long long t0 = globaltimer();
        int e = 0;
        while (ld_acquire(a.bar) < target) {
            if ((e = ld_err(a.err)) != 0) break;
            if (globaltimer() - t0 > a.timeout_ns) {
                atomicCAS(a.err, 0, kDevTimeout);
                e = kDevTimeout;
                break;
            }
        }
        __threadfence();
        *s_ok = (e == 0 && ld_err(a.err) == 0) ? 1 : 0;
    }
    __syncthreads();
    return *s_ok != 0;
}

// Bounded wait for another CTA's carry flag.
__device__ __forceinline__ void wait_flag(const KArgs &a, const unsigned *f, unsigned want) {
    const unsigned long long t0 = globaltimer();
    while (ld_acquire(f) < want) {
        if (ld_err(a.err) != 0) return;
        if (globaltimer() - t0 > a.timeout_ns) {
            atomicCAS(a.err, 0, kDevTimeout);
            return;
        }
    }
}

__device__ __forceinline__ long long diag_of(long long gu, long long items, long long nsub) {
    return (gu * items) / nsub;
}
// Merge-path split: the largest r in [0, min(d, N)] with row_ptr[r] + r <= d.
__device__ __forceinline__ int merge_search(const int *row_ptr, int N, long long d) {
    int lo = 0, hi = (int)(d < (long long)N ? d : (long long)N);
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if ((long long)__ldg(row_ptr + mid) + mid <= d) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Where a warp's piece of the merge path starts and ends, and whom it waits for.
struct Piece {
    int r0, e0, r1, e1;
    bool head;   // row r0 is finished here but started in an earlier piece
    int u_lo;    // first local piece whose carry belongs to row r0
    int c_lo;    // first CTA whose published carry belongs to row r0 (== own CTA: none)
};

// ------------------------------------------------------------ gather loops

// Accumulate sum_k w[k] * rows[col[k]] over edges [elo, ehi) into acc (per
// group); in the backward also add each edge's dot product with the own row
// `hp` into the edge-gradient accumulator.
template <int NC, bool SMEMG, bool BWD, int UNR>
__device__ __forceinline__ void gather(const KArgs &a, const Lanes &L, const int *scol,
                                       const float *sw, float *sdw, int cta_e0,
                                       const float *__restrict__ rows, int elo, int ehi,
                                       float4 (&acc)[NC], const float4 (&hp)[NC]) {
    const int Bp = a.Bp;
    for (int base = elo; base < ehi; base += a.EPW * UNR) {
        int kk[UNR];
        float wv[UNR];
        float4 v[UNR][NC];
#pragma unroll
        for (int q = 0; q < UNR; ++q) {
            const int k = base + q * a.EPW + L.g;
            const bool ok = L.active && k < ehi;
            int c = 0;
            float wq = 0.f;
            if (ok) {
                if (SMEMG) {
                    c = scol[k - cta_e0];
                    wq = sw[k - cta_e0];
                } else {
                    c = __ldg(a.col + k);
                    wq = __ldcg(a.wperm + k);
                }
            }
            kk[q] = ok ? k : -1;
            wv[q] = wq;
            const float *rp = rows + (size_t)c * Bp;
#pragma unroll
            for (int ch = 0; ch < NC; ++ch) {
                const int col0 = col_of<NC>(L, ch);
                v[q][ch] = (ok && col0 < Bp) ? __ldcg(reinterpret_cast<const float4 *>(rp + col0))
                                             : zero4();
            }
        }
#pragma unroll
        for (int q = 0; q < UNR; ++q)
#pragma unroll
            for (int ch = 0; ch < NC; ++ch) fma4(acc[ch], wv[q], v[q][ch]);
        if (BWD) {
#pragma unroll
            for (int q = 0; q < UNR; ++q) {
                float d = 0.f;
#pragma unroll
                for (int ch = 0; ch < NC; ++ch) {
                    d = fmaf(v[q][ch].x, hp[ch].x, d);
                    d = fmaf(v[q][ch].y, hp[ch].y, d);
                    d = fmaf(v[q][ch].z, hp[ch].z, d);
                    d = fmaf(v[q][ch].w, hp[ch].w, d);
                }
                d = group_sum(d, a, L);
                if (L.lig == 0 && kk[q] >= 0) {
                    if (SMEMG) sdw[kk[q] - cta_e0] += d;
                    else a.dwperm[kk[q]] += d;
                }
            }
        }
    }
}

// ------------------------------------------------------- row finalisation

// Forward: pre-activation, tanh, leak blend, saved copies and the output.
template <int NC>
__device__ void fwd_finalize(const KArgs &a, const Lanes &L, int r, const float4 (&acc)[NC],
                             int s) {
    if (!L.lead) return;
    const int t = s / a.M, m = s - t * a.M;
    const int Bp = a.Bp, B = a.B;
    const size_t NBp = (size_t)a.N * Bp;
    const float *hin = a.H + (size_t)s * NBp + (size_t)r * Bp;
    float *hout = a.H + (size_t)(s + 1) * NBp + (size_t)r * Bp;
    float *aout = a.A + (size_t)s * NBp + (size_t)r * Bp;
    const float lam = __ldg(a.leak + r), bia = __ldg(a.bias + r);
    const int sl = __ldg(a.slot + r);
    const float *drv = sl >= 0 ? a.drives + ((size_t)t * a.n_in + sl) * B : nullptr;
    const bool emit = (m == a.M - 1);
#pragma unroll
    for (int ch = 0; ch < NC; ++ch) {
        const int col0 = col_of<NC>(L, ch);
        if (col0 >= Bp) continue;
        const float4 hp = __ldcg(reinterpret_cast<const float4 *>(hin + col0));
        float4 av = acc[ch], hn;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int b = col0 + q;
            float x = f4get(av, q) + bia, y = 0.f;
            if (b < B) {
                if (drv) x += __ldg(drv + b);
                const float p = tanhf(x);
                y = fmaf(lam, p, (1.f - lam) * f4get(hp, q));
                if (emit) __stcs(a.out + ((size_t)t * B + b) * a.N + r, y);
            } else {
                x = 0.f;
            }
            f4set(av, q, x);
            f4set(hn, q, y);
        }
        __stcs(reinterpret_cast<float4 *>(aout + col0), av);
        *reinterpret_cast<float4 *>(hout + col0) = hn;
    }
}

// Backward elementwise terms of microstep q for node j, given Gn = dL/dh_q[j]:
// da = Gn * leak * (1 - p^2), p = tanh(a_q); leak and bias row reductions;
// the drive gradient at input nodes.  All lanes call this (for the shuffles).
template <int NC>
__device__ void elementwise(const KArgs &a, const Lanes &L, int j, const float4 (&Gn)[NC], int q,
                            float lam) {
    const int Bp = a.Bp, B = a.B;
    const size_t NBp = (size_t)a.N * Bp;
    const float *Aq = a.A + (size_t)q * NBp + (size_t)j * Bp;
    const float *Hq = a.H + (size_t)q * NBp + (size_t)j * Bp;  // state entering microstep q
    float *daq = a.da + (size_t)(q & 1) * NBp + (size_t)j * Bp;
    const int sl = __ldg(a.slot + j);
    const int tq = q / a.M;
    const bool first = (q - tq * a.M) == a.M - 1;  // first visit of step tq going backwards
    float *dd = sl >= 0 ? a.ddrives + ((size_t)tq * a.n_in + sl) * B : nullptr;
    float dl = 0.f, db = 0.f;
#pragma unroll
    for (int ch = 0; ch < NC; ++ch) {
        const int col0 = col_of<NC>(L, ch);
        if (!L.lead || col0 >= Bp) continue;
        *reinterpret_cast<float4 *>(a.G + (size_t)j * Bp + col0) = Gn[ch];
        const float4 av = __ldcs(reinterpret_cast<const float4 *>(Aq + col0));
        const float4 hv = __ldg(reinterpret_cast<const float4 *>(Hq + col0));
        float4 d4;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b = col0 + k;
            float d = 0.f;
            if (b < B) {
                const float g = f4get(Gn[ch], k);
                const float p = tanhf(f4get(av, k));
                d = g * lam * (1.f - p * p);
                dl = fmaf(g, p - f4get(hv, k), dl);
                db += d;
                if (dd) dd[b] = first ? d : dd[b] + d;
            }
            f4set(d4, k, d);
        }
        *reinterpret_cast<float4 *>(daq + col0) = d4;
    }
    dl = group_sum(dl, a, L);
    db = group_sum(db, a, L);
    if (L.lead && L.lig == 0) {
        if (q == a.S - 1) {
            a.dleak[j] = dl;
            a.dbias[j] = db;
        } else {
            a.dleak[j] += dl;
            a.dbias[j] += db;
        }
    }
}

// Backward: finish G_{s-1}[j] = G_s[j] (1 - leak) + (W^T da_s)[j] (+ dOut of the
// step that ends at microstep s-1), then the elementwise terms of microstep s-1;
// at s == 0 the result is the gradient of state0.
template <int NC>
__device__ void bwd_finalize(const KArgs &a, const Lanes &L, int j, const float4 (&acc)[NC],
                             int s) {
    const int Bp = a.Bp, B = a.B;
    const float lam = __ldg(a.leak + j);
    const int q = s - 1;
    const int tq = q >= 0 ? q / a.M : 0;
    const bool add_dout = q >= 0 && (q - tq * a.M) == a.M - 1;
    float4 Gn[NC];
#pragma unroll
    for (int ch = 0; ch < NC; ++ch) {
        const int col0 = col_of<NC>(L, ch);
        Gn[ch] = zero4();
        if (!L.lead || col0 >= Bp) continue;
        const float4 g = __ldcg(reinterpret_cast<const float4 *>(a.G + (size_t)j * Bp + col0));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b = col0 + k;
            float x = 0.f;
            if (b < B) {
                x = fmaf(f4get(g, k), 1.f - lam, f4get(acc[ch], k));
                if (add_dout) x += __ldg(a.dout + ((size_t)tq * B + b) * a.N + j);
                if (s == 0) a.dstate0[(size_t)b * a.N + j] = x;
            }
            f4set(Gn[ch], k, x);
        }
    }
    if (s > 0) elementwise<NC>(a, L, j, Gn, q, lam);
}

// ------------------------------------------------------------------ kernel

template <int THREADS, int NC, bool SMEMG, bool BWD>
__global__ void __launch_bounds__(THREADS, 1) rec_kernel(const KArgs a) {
    constexpr int U = THREADS / 32;
    constexpr int UNR = NC == 1 ? 8 : (NC == 2 ? 4 : 2);
    extern __shared__ float4 smem_dyn[];
    __shared__ int sub_r[U + 1], sub_e[U + 1];
    __shared__ int s_ok;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const Lanes L = make_lanes(a, lane);
    const int N = a.N, Bp = a.Bp;
    const size_t NBp = (size_t)N * Bp;

    // ---- this warp's piece of the merge path
    const long long items = (long long)N + a.E, nsub = (long long)a.P * U;
    Piece pc;
    {
        int r0 = 0, e0 = 0, r1 = 0, e1 = 0;
        if (lane == 0) {
            const long long d0 = diag_of((long long)cta * U + warp, items, nsub);
            const long long d1 = diag_of((long long)cta * U + warp + 1, items, nsub);
            r0 = merge_search(a.row_ptr, N, d0);
            r1 = merge_search(a.row_ptr, N, d1);
            e0 = (int)(d0 - r0);
            e1 = (int)(d1 - r1);
        }
        pc.r0 = __shfl_sync(kFull, r0, 0);
        pc.e0 = __shfl_sync(kFull, e0, 0);
        pc.r1 = __shfl_sync(kFull, r1, 0);
        pc.e1 = __shfl_sync(kFull, e1, 0);
        if (lane == 0) {
            sub_r[warp] = pc.r0;
            sub_e[warp] = pc.e0;
            if (warp == U - 1) {
                sub_r[U] = pc.r1;
                sub_e[U] = pc.e1;
            }
        }
    }
    __syncthreads();
    const int cta_e0 = sub_e[0], cta_e1 = sub_e[U];
    {
        const int R = pc.r0;
        pc.head = pc.r0 < pc.r1 && pc.e0 > __ldg(a.row_ptr + R);
        pc.u_lo = warp;
        pc.c_lo = cta;
        if (pc.head) {
            int v = warp - 1;
            while (v >= 0) {
                pc.u_lo = v;
                if (sub_r[v] != R) break;
                --v;
            }
            if (v < 0 && cta > 0) {
                int c = cta - 1;
                if (lane == 0) {
                    while (c > 0 && merge_search(a.row_ptr, N, diag_of((long long)c * U, items, nsub)) == R)
                        --c;
                }
                pc.c_lo = __shfl_sync(kFull, c, 0);
            }
        }
    }
    // carries this CTA publishes: pieces [p_lo, U) all end inside row Rc
    const int Rc = sub_r[U];
    const bool publish = cta + 1 < a.P && Rc < N;
    int p_lo = U - 1;
    while (p_lo > 0 && sub_r[p_lo] == Rc) --p_lo;

    // ---- shared memory: carries, then this CTA's slice of the graph
    float *scarry = reinterpret_cast<float *>(smem_dyn);  // [U][Bp]
    int *scol = reinterpret_cast<int *>(scarry + (size_t)U * Bp);
    float *sw = reinterpret_cast<float *>(scol + a.cap);
    float *sdw = sw + a.cap;
    if (SMEMG && cta_e1 - cta_e0 > a.cap) {
        if (tid == 0) atomicCAS(a.err, 0, kDevInternal);
        return;  // the other CTAs see the error word at their next wait
    }
    for (int k = cta_e0 + tid; k < cta_e1; k += THREADS) {
        if (SMEMG) {
            scol[k - cta_e0] = __ldg(a.col + k);
            sw[k - cta_e0] = __ldg(a.w + __ldg(a.perm + k));
            if (BWD) sdw[k - cta_e0] = 0.f;
        } else if (a.do_prologue) {
            a.wperm[k] = __ldg(a.w + __ldg(a.perm + k));
            if (BWD) a.dwperm[k] = 0.f;
        }
    }
    __syncthreads();

    unsigned nbar = 0;
    if (a.do_prologue) {
        if (!BWD) {
            // state0 [B][N] -> H[0] [N][Bp], pad columns zero
            const size_t total = NBp;
            for (size_t i = (size_t)cta * THREADS + tid; i < total; i += (size_t)a.P * THREADS) {
                const int node = (int)(i / Bp), b = (int)(i - (size_t)node * Bp);
                a.H[i] = b < a.B ? __ldg(a.state0 + (size_t)b * N + node) : 0.f;
            }
        } else {
            // G_{S-1} = dOut[T-1]^T, then the elementwise terms of the last microstep
            for (int j = pc.r0; j < pc.r1; ++j) {
                float4 Gn[NC];
#pragma unroll
                for (int ch = 0; ch < NC; ++ch) {
                    const int col0 = col_of<NC>(L, ch);
                    Gn[ch] = zero4();
                    if (!L.lead || col0 >= Bp) continue;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int b = col0 + k;
                        if (b < a.B)
                            f4set(Gn[ch], k, __ldg(a.dout + ((size_t)(a.T - 1) * a.B + b) * N + j));
                    }
                }
                elementwise<NC>(a, L, j, Gn, a.S - 1, __ldg(a.leak + j));
            }
        }
        if (!grid_sync(a, nbar++, &s_ok)) return;
    }

    for (int it = 0; it < a.s_count; ++it) {
        const int s = BWD ? a.s_first - it : a.s_first + it;
        const unsigned phase_id = BWD ? (unsigned)(a.S - s) : (unsigned)(s + 1);
        const float *rows = BWD ? a.da + (size_t)(s & 1) * NBp : a.H + (size_t)s * NBp;
        float4 head[NC];
#pragma unroll
        for (int ch = 0; ch < NC; ++ch) head[ch] = zero4();

        for (int r = pc.r0; r <= pc.r1 && r < N; ++r) {
            const int elo = max(__ldg(a.row_ptr + r), pc.e0);
            const int ehi = min(__ldg(a.row_ptr + r + 1), pc.e1);
            float4 acc[NC], hp[NC];
#pragma unroll
            for (int ch = 0; ch < NC; ++ch) {
                acc[ch] = zero4();
                hp[ch] = zero4();
                if (BWD) {
                    const int col0 = col_of<NC>(L, ch);
                    if (L.active && col0 < Bp && elo < ehi)
                        hp[ch] = __ldg(reinterpret_cast<const float4 *>(
                            a.H + (size_t)s * NBp + (size_t)r * Bp + col0));
                }
            }
            gather<NC, SMEMG, BWD, UNR>(a, L, scol, sw, sdw, cta_e0, rows, elo, ehi, acc, hp);
            reduce_groups<NC>(acc, a, L);
            if (r == pc.r1) {
                if (L.lead) {
#pragma unroll
                    for (int ch = 0; ch < NC; ++ch) {
                        const int col0 = col_of<NC>(L, ch);
                        if (col0 < Bp)
                            *reinterpret_cast<float4 *>(scarry + (size_t)warp * Bp + col0) = acc[ch];
                    }
                }
            } else if (r == pc.r0 && pc.head) {
#pragma unroll
                for (int ch = 0; ch < NC; ++ch) head[ch] = acc[ch];
            } else {
                if (BWD) bwd_finalize<NC>(a, L, r, acc, s);
                else fwd_finalize<NC>(a, L, r, acc, s);
            }
        }
        __syncthreads();

        // publish this CTA's carry for row Rc
        if (publish && warp == U - 1) {
            if (L.lead) {
#pragma unroll
                for (int ch = 0; ch < NC; ++ch) {
                    const int col0 = col_of<NC>(L, ch);
                    if (col0 >= Bp) continue;
                    float4 sum = zero4();
                    for (int v = p_lo; v < U; ++v)
                        add4(sum, *reinterpret_cast<const float4 *>(scarry + (size_t)v * Bp + col0));
                    __stcg(reinterpret_cast<float4 *>(a.carry + (size_t)cta * Bp + col0), sum);
                }
                __threadfence();
            }
            __syncwarp();
            if (lane == 0) st_release(a.flags + cta, phase_id);
        }
        // finish the head row: earlier CTAs' carries, earlier local pieces, own part
        if (pc.head) {
            float4 tot[NC];
#pragma unroll
            for (int ch = 0; ch < NC; ++ch) tot[ch] = zero4();
            for (int c = pc.c_lo; c < cta; ++c) {
                wait_flag(a, a.flags + c, phase_id);
                if (L.lead) {
#pragma unroll
                    for (int ch = 0; ch < NC; ++ch) {
                        const int col0 = col_of<NC>(L, ch);
                        if (col0 < Bp)
                            add4(tot[ch], __ldcg(reinterpret_cast<const float4 *>(
                                              a.carry + (size_t)c * Bp + col0)));
                    }
                }
            }
            __syncwarp();
            if (L.lead) {
                for (int v = pc.u_lo; v < warp; ++v) {
#pragma unroll
                    for (int ch = 0; ch < NC; ++ch) {
                        const int col0 = col_of<NC>(L, ch);
                        if (col0 < Bp)
                            add4(tot[ch],
                                 *reinterpret_cast<const float4 *>(scarry + (size_t)v * Bp + col0));
                    }
                }
#pragma unroll
                for (int ch = 0; ch < NC; ++ch) add4(tot[ch], head[ch]);
            }
            if (BWD) bwd_finalize<NC>(a, L, pc.r0, tot, s);
            else fwd_finalize<NC>(a, L, pc.r0, tot, s);
        }
        if (it + 1 < a.s_count)
            if (!grid_sync(a, nbar++, &s_ok)) return;
    }

    if (BWD && a.do_epilogue) {
        // edge gradients back to the caller's edge order
        __syncthreads();
        for (int k = cta_e0 + tid; k < cta_e1; k += THREADS) {
            const float v = SMEMG ? sdw[k - cta_e0] : a.dwperm[k];
            a.dw[__ldg(a.perm + k)] = v;
        }
    }
}

// ------------------------------------------------------------------ host

using KernelFn = void (*)(const KArgs);

template <int THREADS, bool BWD>
KernelFn pick_nc(int nc, bool smem) {
    switch (nc) {
        case 1: return smem ? rec_kernel<THREADS, 1, true, BWD> : rec_kernel<THREADS, 1, false, BWD>;
        case 2: return smem ? rec_kernel<THREADS, 2, true, BWD> : rec_kernel<THREADS, 2, false, BWD>;
        default: return smem ? rec_kernel<THREADS, 4, true, BWD> : rec_kernel<THREADS, 4, false, BWD>;
    }
}

KernelFn pick_kernel(int threads, int nc, bool smem, bool bwd) {
    if (threads == 1024) return bwd ? pick_nc<1024, true>(nc, smem) : pick_nc<1024, false>(nc, smem);
    return bwd ? pick_nc<512, true>(nc, smem) : pick_nc<512, false>(nc, smem);
}

int pow2ceil(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

void fill_common(KArgs &k, const ck_graph *g, const Plan &p, void *scratch) {
    std::memset(&k, 0, sizeof(k));
    k.N = p.N;
    k.E = p.E;
    k.n_in = p.n_in;
    k.B = p.B;
    k.Bp = p.Bp;
    k.LPE = p.LPE;
    k.EPW = p.EPW;
    k.LPE_P2 = pow2ceil(p.LPE);
    k.EPW_P2 = pow2ceil(p.EPW);
    k.T = p.T;
    k.M = p.M;
    k.S = p.S;
    k.P = p.P;
    k.U = p.warps;
    k.cap = p.cap;
    k.slot = g->slot;
    char *sc = (char *)scratch;
    k.bar = (unsigned *)(sc + p.off_ctrl);
    k.err = (int *)(sc + p.off_ctrl + 4);
    k.flags = (unsigned *)(sc + p.off_ctrl + 256);
    k.carry = (float *)(sc + p.off_carry);
    k.wperm = (float *)(sc + p.off_wperm);
    k.dwperm = (float *)(sc + p.off_dwperm);
    k.G = (float *)(sc + p.off_G);
    k.da = (float *)(sc + p.off_da);
    k.bar_extra = (unsigned)options().barrier_extra;
    k.timeout_ns = (unsigned long long)options().timeout_ns;
}

ck_status launch_all(KArgs &k, const Plan &p, bool bwd, bool smem, size_t smem_bytes,
                     cudaStream_t s, int64_t *launches) {
    KernelFn fn = pick_kernel(p.threads, p.NC, smem, bwd);
    cudaError_t e = cudaFuncSetAttribute((const void *)fn,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, (const void *)fn, p.threads,
                                                      smem_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (per_sm < 1)
        return fail(CK_ERR_UNSUPPORTED, "kernel does not fit on an SM (%d threads, %zu B shared)",
                    p.threads, smem_bytes);
    e = cudaMemsetAsync((char *)k.bar, 0, p.ctrl_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (control words)");
    int64_t n = 0;
    const bool persistent = options().persistent != 0;
    const int S = p.S;
    const int steps = persistent ? 1 : S;
    for (int i = 0; i < steps; ++i) {
        KArgs ki = k;
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
        e = cudaLaunchCooperativeKernel((const void *)fn, dim3(p.P), dim3(p.threads), args,
                                        smem_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaLaunchCooperativeKernel");
        ++n;
    }
    if (launches) *launches = n;
    return CK_OK;
}

}  // namespace

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
    q.Bp = (int)((B + 7) / 8 * 8);
    q.NC = (q.Bp + 127) / 128;
    if (q.NC == 3) q.NC = 4;  // three chunks run in the four-chunk kernel with masking
    q.LPE = q.Bp <= 128 ? q.Bp / 4 : 32;
    q.EPW = 32 / q.LPE;
    q.T = (int)T;
    q.M = (int)M;
    q.S = (int)(T * M);
    q.P = g->num_sms;
    q.threads = options().threads == 1024 ? 1024 : 512;
    q.warps = q.threads / 32;
    const int64_t items = g->N + g->E;
    q.cap = (int)(items / q.P + 2);
    const size_t carry_smem = (size_t)q.warps * q.Bp * 4;
    const size_t budget = kMaxSmem - kSmemReserve;
    const bool allow = options().graph_in_smem && options().persistent;
    q.smem_fwd = carry_smem + (size_t)q.cap * 8;
    q.smem_bwd = carry_smem + (size_t)q.cap * 12;
    q.smem_graph_fwd = allow && q.smem_fwd <= budget;
    q.smem_graph_bwd = allow && q.smem_bwd <= budget;
    if (!q.smem_graph_fwd) q.smem_fwd = carry_smem;
    if (!q.smem_graph_bwd) q.smem_bwd = carry_smem;
    if (carry_smem > budget) return fail(CK_ERR_UNSUPPORTED, "carry buffers exceed shared memory");
    const size_t NBp = (size_t)q.N * q.Bp;
    const size_t E1 = (size_t)(q.E > 0 ? q.E : 1);
    size_t off = 0;
    q.off_ctrl = off;
    q.ctrl_bytes = align256(256 + 4 * (size_t)q.P);
    off += q.ctrl_bytes;
    q.off_carry = off;
    off = align256(off + 4 * (size_t)q.P * q.Bp);
    q.off_wperm = off;
    off = align256(off + 4 * E1);
    q.off_dwperm = off;
    off = align256(off + 4 * E1);
    q.off_G = off;
    off = align256(off + 4 * NBp);
    q.off_da = off;
    off = align256(off + 8 * NBp);
    q.scratch_bytes = off;
    q.saved_bytes = 4 * NBp * (size_t)(2 * q.S + 1);
    *p = q;
    return CK_OK;
}

ck_status launch_forward(const ck_graph *g, const Plan &p, const FwdIO &io, cudaStream_t s,
                         int64_t *launches) {
    KArgs k;
    fill_common(k, g, p, io.scratch);
    k.row_ptr = g->row_ptr;
    k.col = g->col;
    k.perm = g->perm;
    k.w = io.w;
    k.leak = io.leak;
    k.bias = io.bias;
    k.drives = io.drives;
    k.state0 = io.state0;
    k.out = io.out;
    k.H = io.saved;
    k.A = io.saved + (size_t)(p.S + 1) * p.N * p.Bp;
    return launch_all(k, p, false, p.smem_graph_fwd, p.smem_fwd, s, launches);
}

ck_status launch_backward(const ck_graph *g, const Plan &p, const BwdIO &io, cudaStream_t s,
                          int64_t *launches) {
    KArgs k;
    fill_common(k, g, p, io.scratch);
    k.row_ptr = g->rowT_ptr;
    k.col = g->colT;
    k.perm = g->permT;
    k.w = io.w;
    k.leak = io.leak;
    k.H = const_cast<float *>(io.saved);
    k.A = const_cast<float *>(io.saved) + (size_t)(p.S + 1) * p.N * p.Bp;
    k.dout = io.dout;
    k.dw = io.dw;
    k.dleak = io.dleak;
    k.dbias = io.dbias;
    k.ddrives = io.ddrives;
    k.dstate0 = io.dstate0;
    return launch_all(k, p, true, p.smem_graph_bwd, p.smem_bwd, s, launches);
}

}  // namespace ck
