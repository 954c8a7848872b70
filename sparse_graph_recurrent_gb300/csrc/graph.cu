// Graph build on the GPU: validation, the input-slot map, and two stable sorts
// of the edge list (by dst for the forward rows, by src for the transposed rows).
//
// connectome-kernels page, "Use": the graph is built once from int64 (src, dst)
// lists on the GPU; edge parameters stay in the caller's order and the internal
// compressed-row permutation is invisible.  "Design notes": the state gradient
// runs over a precomputed transposed copy.
//
// The sort is a least-significant-digit radix sort with 8-bit digits.  Each
// pass is a counting sort over tiles of 4096 keys: a per-tile digit histogram,
// an exclusive scan of the histograms in (digit, tile) order, and a scatter in
// which every key's rank among equal digits of its tile comes from warp match
// masks taken in element order.  Every pass keeps equal keys in their previous
// order, so the result lists each row's edges in ascending caller edge id.
#include <algorithm>
#include <cstring>
#include <vector>

#include "ck_internal.h"

namespace ck {
namespace {

constexpr int kTile = 4096;      // keys per CTA in a radix pass
constexpr int kSortThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;    // per thread
constexpr int kScanBlock = kScanThreads * kScanItems;

enum : unsigned { kBadEdge = 1u, kBadInput = 2u, kDupInput = 4u };

__global__ void k_validate(const int64_t *__restrict__ src, const int64_t *__restrict__ dst,
                           int64_t E, int64_t N, int *__restrict__ key_dst,
                           int *__restrict__ key_src, int *__restrict__ ids,
                           int *__restrict__ ids2, unsigned *__restrict__ flags) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < E;
         e += (int64_t)gridDim.x * blockDim.x) {
        int64_t s = src[e], d = dst[e];
        if (s < 0 || s >= N || d < 0 || d >= N) {
            atomicOr(flags, kBadEdge);
            s = 0;
            d = 0;
        }
        key_src[e] = (int)s;
        key_dst[e] = (int)d;
        ids[e] = (int)e;
        ids2[e] = (int)e;
    }
}

__global__ void k_slots(const int64_t *__restrict__ inp, int64_t n_in, int64_t N,
                        int *__restrict__ slot, unsigned *__restrict__ flags) {
    for (int64_t k = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; k < n_in;
         k += (int64_t)gridDim.x * blockDim.x) {
        int64_t v = inp[k];
        if (v < 0 || v >= N) {
            atomicOr(flags, kBadInput);
            continue;
        }
        if (atomicCAS(&slot[v], -1, (int)k) != -1) atomicOr(flags, kDupInput);
    }
}

// Per-tile digit counts, stored digit-major: hist[digit * ntiles + tile].
__global__ void __launch_bounds__(kSortThreads) k_radix_hist(const int *__restrict__ keys, int n,
                                                             int shift, int *__restrict__ hist,
                                                             int ntiles) {
    __shared__ int h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    const int base = blockIdx.x * kTile;
    for (int i = threadIdx.x; i < kTile; i += kSortThreads) {
        int idx = base + i;
        if (idx < n) atomicAdd(&h[(keys[idx] >> shift) & 255], 1);
    }
    __syncthreads();
    hist[threadIdx.x * ntiles + blockIdx.x] = h[threadIdx.x];
}

// Stable scatter of one tile: element order inside the tile decides ranks.
__global__ void __launch_bounds__(kSortThreads) k_radix_scatter(
    const int *__restrict__ kin, const int *__restrict__ vin, int *__restrict__ kout,
    int *__restrict__ vout, int n, int shift, const int *__restrict__ offs, int ntiles) {
    constexpr int W = kSortThreads / 32;
    __shared__ int run[256];
    __shared__ int wcnt[W][256];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned lt = (1u << lane) - 1u;
    run[tid] = offs[tid * ntiles + blockIdx.x];
    const int base = blockIdx.x * kTile;
    for (int c = 0; c < kTile; c += kSortThreads) {
#pragma unroll
        for (int w = 0; w < W; ++w) wcnt[w][tid] = 0;
        __syncthreads();
        const int idx = base + c + tid;
        const bool valid = idx < n;
        int key = 0, val = 0, digit = -1;
        if (valid) {
            key = kin[idx];
            val = vin[idx];
            digit = (key >> shift) & 255;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        const int rank = __popc(peers & lt);
        if (valid && (__ffs(peers) - 1) == lane) wcnt[warp][digit] = __popc(peers);
        __syncthreads();
        {
            int r = run[tid];
#pragma unroll
            for (int w = 0; w < W; ++w) {
                int cnt = wcnt[w][tid];
                wcnt[w][tid] = r;
                r += cnt;
            }
            run[tid] = r;
        }
        __syncthreads();
        if (valid) {
            const int pos = wcnt[warp][digit] + rank;
            kout[pos] = key;
            vout[pos] = val;
        }
        __syncthreads();
    }
}

// Exclusive scan, three kernels: per-block scan + block totals, scan of the
// totals (recursively), add the scanned totals back.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;  // inclusive
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    if (total && threadIdx.x == blockDim.x - 1) *total = before + v;
    return before;
}

__global__ void __launch_bounds__(kScanThreads) k_scan_block(const int *__restrict__ in,
                                                             int *__restrict__ out, int n,
                                                             int *__restrict__ block_sums) {
    __shared__ int warp_sums[32];
    __shared__ int tot;
    const int base = blockIdx.x * kScanBlock + threadIdx.x * kScanItems;
    int v[kScanItems];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
        v[i] = (base + i < n) ? in[base + i] : 0;
        sum += v[i];
    }
    int run = block_exclusive_scan(sum, warp_sums, &tot);
#pragma unroll
    for (int i = 0; i < kScanItems; ++i) {
        if (base + i < n) out[base + i] = run;
        run += v[i];
    }
    __syncthreads();
    if (threadIdx.x == 0) block_sums[blockIdx.x] = tot;
}

__global__ void k_scan_add(int *__restrict__ out, int n, const int *__restrict__ block_offs) {
    const int b = blockIdx.x;
    const int add = block_offs[b];
    const int base = b * kScanBlock;
    for (int i = threadIdx.x; i < kScanBlock; i += blockDim.x)
        if (base + i < n) out[base + i] += add;
}

// In-place safe: each block reads its inputs before any block's output is added to.
cudaError_t exclusive_scan(const int *in, int *out, int n, int *tmp, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int nb = (n + kScanBlock - 1) / kScanBlock;
    int *sums = tmp;
    int *sums_scanned = tmp + nb;
    k_scan_block<<<nb, kScanThreads, 0, s>>>(in, out, n, sums);
    if (nb > 1) {
        cudaError_t e = exclusive_scan(sums, sums_scanned, nb, tmp + 2 * nb, s);
        if (e != cudaSuccess) return e;
        k_scan_add<<<nb, kScanThreads, 0, s>>>(out, n, sums_scanned);
    }
    return cudaGetLastError();
}

size_t scan_tmp_ints(int n) {
    size_t t = 0;
    while (n > 0) {
        int nb = (n + kScanBlock - 1) / kScanBlock;
        t += 2 * (size_t)nb;
        if (nb <= 1) break;
        n = nb;
    }
    return t + 2;
}

// row_ptr[i] = first position whose key >= i, for i in [0, N].
__global__ void k_row_ptr(const int *__restrict__ sorted_keys, int E, int N,
                          int *__restrict__ row_ptr) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= N; i += gridDim.x * blockDim.x) {
        int lo = 0, hi = E;
        while (lo < hi) {
            int mid = (lo + hi) >> 1;
            if (sorted_keys[mid] < i) lo = mid + 1;
            else hi = mid;
        }
        row_ptr[i] = lo;
    }
}

__global__ void k_gather_other(const int64_t *__restrict__ other, const int *__restrict__ perm,
                               int E, int *__restrict__ col) {
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < E; k += gridDim.x * blockDim.x)
        col[k] = (int)other[perm[k]];
}

// First row and edge of each of P equal pieces of the merge path of
// (row ends, edges): the largest r with row_ptr[r] + r <= floor(c (N+E) / P).
// One cut of the weighted merge path of (row ends, edges) into P pieces: a
// row end counts as `wt` items, an edge as one.  Piece c starts at diagonal
// d = c (E + wt N) / P: r = the rows whose ends come before d (the largest r
// with row_ptr[r] + wt r <= d) and e = the edges before d, which lie between
// row_ptr[r] and row_ptr[r + 1].  With wt = 1 this is the plain merge path.
struct Cut {
    std::vector<int> r, e;  // P + 1 bounds
    int max_rows = 0, max_edges = 0;
};

// CTAs P/2 .. P-1 are the second of their SM's two to be dispatched, and on
// the same work they finish 2-4% later than the first (per-CTA timings, both
// directions, across boxes and with the pieces rotated: the delay follows the
// block, not its data or its SM).  Their pieces get kLateShare per mille less
// of the weighted items, the first half's as much more.
constexpr int kLateShare = 15;

// Sum of the shares of pieces [0, c), in per mille of an even share.
long long share_prefix(int c, int P) {
    const int h = P / 2;
    return c <= h ? (long long)c * (1000 + kLateShare)
                  : (long long)h * (1000 + kLateShare) + (long long)(c - h) * (1000 - kLateShare);
}

Cut cut_pieces(const std::vector<int> &rp, int N, int E, int P, int wt) {
    Cut k;
    k.r.resize(P + 1);
    k.e.resize(P + 1);
    const long long items = (long long)E + (long long)wt * N;
    const long long total = share_prefix(P, P);
    for (int c = 0; c <= P; ++c) {
        const long long d = c == P ? items : items * share_prefix(c, P) / total;
        int lo = 0, hi = N;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)rp[mid] + (long long)wt * mid <= d) lo = mid;
            else hi = mid - 1;
        }
        const long long e = d - (long long)wt * lo;
        const int cap = rp[lo < N ? lo + 1 : N];
        k.r[c] = lo;
        k.e[c] = (int)(e < cap ? e : cap);
    }
    for (int c = 0; c < P; ++c) {
        k.max_rows = std::max(k.max_rows, k.r[c + 1] - k.r[c]);
        k.max_edges = std::max(k.max_edges, k.e[c + 1] - k.e[c]);
    }
    return k;
}

// Estimated time of the slowest piece, for choosing the row weight: part A
// grows with a piece's edges, part B with the finish passes its rows need; the
// second-dispatched half runs slower by the factor its smaller share offsets.
double cut_cost(const Cut &k, int P, int pass_rows, double edge_us, double pass_us) {
    double worst = 0.0;
    const double late = (1000.0 + kLateShare) / (1000.0 - kLateShare);
    for (int c = 0; c < P; ++c) {
        const int rows = k.r[c + 1] - k.r[c], edges = k.e[c + 1] - k.e[c];
        const int passes = (rows + pass_rows - 1) / pass_rows;
        const double t = edges * edge_us + (passes > 0 ? passes : 1) * pass_us;
        worst = std::max(worst, c >= P / 2 ? t * late : t);
    }
    return worst;
}

// Per-CTA piece descriptions (ck_graph::piece) of one cut.
std::vector<int> piece_meta(const Cut &k, const std::vector<int> &rp, int N, int P) {
    std::vector<int> m((size_t)P * kPieceInts, 0);
    for (int c = 0; c < P; ++c) {
        const int r0 = k.r[c], r1 = k.r[c + 1], e0 = k.e[c], e1 = k.e[c + 1];
        int clo = c;
        if (c > 0 && e0 > rp[r0]) {  // row r0 has edges in earlier pieces
            clo = c - 1;
            while (clo > 0 && k.r[clo] == r0) --clo;
        }
        int *q = m.data() + (size_t)c * kPieceInts;
        q[0] = r0;
        q[1] = r1 - r0;
        q[2] = e0;
        q[3] = e1;
        q[4] = clo;
        q[5] = (c + 1 < P && r1 < N) ? 1 : 0;
    }
    return m;
}

// Cut [0, n) into k contiguous ranges of about equal total weight (prefix
// weights pre[0..n], pre[0] = 0): range r ends at the first index whose prefix
// reaches (r + 1) / k of the total.  Returns k + 1 bounds.
std::vector<int> balanced_cuts(const std::vector<long long> &pre, int n, int k) {
    std::vector<int> b(k + 1, n);
    b[0] = 0;
    const long long total = pre[n];
    int i = 0;
    for (int r = 1; r < k; ++r) {
        const long long target = (total * r + k - 1) / k;
        while (i < n && pre[i] < target) ++i;
        b[r] = std::max(b[r - 1], i);
    }
    return b;
}

// Host-side tiling of one direction (ck::Tiled), from its compressed rows.
// Returns the layout in host vectors; C == 0 when no tiling fits.
struct TiledHost {
    Tiled t;
    std::vector<int> meta, ptr, col, perm, rowid;
};

TiledHost tile_direction(int dir, int N, int E, int sms, const std::vector<int> &rp,
                         const std::vector<int> &col, const std::vector<int> &perm) {
    TiledHost h;
    std::memset(&h.t, 0, sizeof(h.t));
    // column degrees (edges whose column is each node)
    std::vector<long long> colpre(N + 1, 0);
    for (int k = 0; k < E; ++k) colpre[col[k] + 1] += 1;
    for (int i = 0; i < N; ++i) colpre[i + 1] += colpre[i] + 1;  // + 1: a node's row of the chunk
    std::vector<long long> rowpre(N + 1, 0);
    for (int i = 0; i < N; ++i) rowpre[i + 1] = rowpre[i] + (rp[i + 1] - rp[i]) + 4;
    static const int kChunks[] = {1, 2, 3, 4, 5, 6, 8};
    for (int C : kChunks) {
        if (C > N) break;
        const int G = std::min(sms / C, N);
        if (G < 1) break;
        std::vector<int> cb = balanced_cuts(colpre, N, C);
        int max_chunk = 0;
        for (int j = 0; j < C; ++j) max_chunk = std::max(max_chunk, cb[j + 1] - cb[j]);
        if (!tiled_fits(dir, kTiledMaxBp, 0, 0, max_chunk)) {
            // edge-balanced chunks too uneven: equal node ranges
            for (int j = 0; j <= C; ++j) cb[j] = (int)((long long)N * j / C);
            max_chunk = 0;
            for (int j = 0; j < C; ++j) max_chunk = std::max(max_chunk, cb[j + 1] - cb[j]);
        }
        const std::vector<int> rb = balanced_cuts(rowpre, N, G);
        int max_rows = 0;
        for (int g = 0; g < G; ++g) max_rows = std::max(max_rows, rb[g + 1] - rb[g]);
        const int max_fin = (max_rows + C - 1) / C;
        if (!tiled_fits(dir, kTiledMaxBp, max_rows, max_fin, max_chunk)) continue;
        // chunk of every column node
        std::vector<int> chunk_of(N);
        for (int j = 0; j < C; ++j)
            for (int i = cb[j]; i < cb[j + 1]; ++i) chunk_of[i] = j;
        const int P = G * C;
        std::vector<long long> cnt(P + 1, 0);
        for (int g = 0; g < G; ++g)
            for (int k = rp[rb[g]]; k < rp[rb[g + 1]]; ++k) cnt[g * C + chunk_of[col[k]] + 1] += 1;
        for (int t = 0; t < P; ++t) cnt[t + 1] += cnt[t];
        std::vector<long long> pos(cnt.begin(), cnt.end() - 1);
        std::vector<int> off(P + 1, 0);
        for (int t = 0; t < P; ++t) off[t + 1] = off[t] + (rb[t / C + 1] - rb[t / C]) + 1;
        h.ptr.assign(off[P], 0);
        const size_t E1 = E > 0 ? (size_t)E : 1;
        h.col.assign(E1, 0);
        h.perm.assign(E1, 0);
        h.rowid.assign(E1, 0);
        int max_edges = 0;
        for (int g = 0; g < G; ++g) {
            for (int i = rb[g]; i < rb[g + 1]; ++i) {
                for (int j = 0; j < C; ++j) h.ptr[off[g * C + j] + (i - rb[g])] = (int)pos[g * C + j];
                for (int k = rp[i]; k < rp[i + 1]; ++k) {
                    const int j = chunk_of[col[k]];
                    const long long q = pos[g * C + j]++;
                    h.col[q] = col[k] - cb[j];
                    h.perm[q] = perm[k];
                    h.rowid[q] = i;
                }
            }
            for (int j = 0; j < C; ++j) {
                const int t = g * C + j;
                h.ptr[off[t] + (rb[g + 1] - rb[g])] = (int)pos[t];
                max_edges = std::max(max_edges, (int)(cnt[t + 1] - cnt[t]));
            }
        }
        h.meta.assign((size_t)P * kTileInts, 0);
        for (int t = 0; t < P; ++t) {
            const int g = t / C, j = t % C, R = rb[g + 1] - rb[g];
            int *m = &h.meta[(size_t)t * kTileInts];
            m[0] = rb[g];
            m[1] = R;
            m[2] = (int)cnt[t];
            m[3] = (int)cnt[t + 1];
            m[4] = cb[j];
            m[5] = cb[j + 1] - cb[j];
            m[6] = off[t];
            m[7] = (int)((long long)R * j / C);
            m[8] = (int)((long long)R * (j + 1) / C);
            m[9] = j;
            m[10] = g;
        }
        h.t.C = C;
        h.t.G = G;
        h.t.P = P;
        h.t.max_rows = max_rows;
        h.t.max_fin = max_fin;
        h.t.max_chunk = max_chunk;
        h.t.max_edges = max_edges;
        return h;
    }
    return h;  // no tiling fits
}

struct DevBuf {
    void *p = nullptr;
    ~DevBuf() {
        if (p) cudaFree(p);
    }
};

// Stable sort of (keys, vals) by key; *in_b tells which pair holds the result.
cudaError_t radix_sort(int *ka, int *va, int *kb, int *vb, int n, int key_bits, int *hist,
                       int *scan_tmp, cudaStream_t s, bool *in_b) {
    const int ntiles = (n + kTile - 1) / kTile;
    *in_b = false;
    for (int shift = 0; shift < key_bits; shift += 8) {
        k_radix_hist<<<ntiles, kSortThreads, 0, s>>>(ka, n, shift, hist, ntiles);
        cudaError_t e = exclusive_scan(hist, hist, 256 * ntiles, scan_tmp, s);
        if (e != cudaSuccess) return e;
        k_radix_scatter<<<ntiles, kSortThreads, 0, s>>>(ka, va, kb, vb, n, shift, hist, ntiles);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        int *t = ka; ka = kb; kb = t;
        t = va; va = vb; vb = t;
        *in_b = !*in_b;
    }
    return cudaSuccess;
}

}  // namespace

ck_status build_graph(ck_graph *g, const int64_t *src, const int64_t *dst,
                      const int64_t *input_nodes, uint32_t graph_flags, cudaStream_t s) {
    const int N = (int)g->N, E = (int)g->E, n_in = (int)g->n_in;
    cudaError_t e;
#define CK_TRY(call, what)                                                              \
    do {                                                                                \
        e = (call);                                                                     \
        if (e != cudaSuccess)                                                           \
            return (e == cudaErrorMemoryAllocation)                                     \
                       ? fail(CK_ERR_OUT_OF_MEMORY, "%s: %s", what, cudaGetErrorString(e)) \
                       : cuda_fail(e, what);                                            \
    } while (0)

    const size_t E1 = std::max<size_t>((size_t)E, 2 * (size_t)g->num_sms + 8);
    CK_TRY(cudaMalloc((void **)&g->row_ptr, sizeof(int) * (N + 1)), "cudaMalloc row_ptr");
    CK_TRY(cudaMalloc((void **)&g->rowT_ptr, sizeof(int) * (N + 1)), "cudaMalloc rowT_ptr");
    CK_TRY(cudaMalloc((void **)&g->slot, sizeof(int) * N), "cudaMalloc slot");
    CK_TRY(cudaMalloc((void **)&g->col, sizeof(int) * E1), "cudaMalloc col");
    CK_TRY(cudaMalloc((void **)&g->perm, sizeof(int) * E1), "cudaMalloc perm");
    CK_TRY(cudaMalloc((void **)&g->colT, sizeof(int) * E1), "cudaMalloc colT");
    CK_TRY(cudaMalloc((void **)&g->permT, sizeof(int) * E1), "cudaMalloc permT");
    CK_TRY(cudaMalloc((void **)&g->rowid, sizeof(int) * E1), "cudaMalloc rowid");
    CK_TRY(cudaMalloc((void **)&g->rowidT, sizeof(int) * E1), "cudaMalloc rowidT");
    g->device_bytes += sizeof(int) * (3 * (size_t)N + 2 + 6 * E1);

    const int ntiles = (E + kTile - 1) / kTile;
    const size_t n_hist = 256 * (size_t)(ntiles > 0 ? ntiles : 1);
    const size_t n_tmp = scan_tmp_ints((int)n_hist);
    // key_dst, key_src, ids, ids2, kb, vb; histograms; scan temp; flags
    const size_t ints = 6 * E1 + n_hist + n_tmp + 4;
    DevBuf tmp;
    CK_TRY(cudaMalloc(&tmp.p, ints * sizeof(int)), "cudaMalloc build temp");
    int *key_dst = (int *)tmp.p;
    int *key_src = key_dst + E1;
    int *ids = key_src + E1;
    int *ids2 = ids + E1;
    int *kb = ids2 + E1;
    int *vb = kb + E1;
    int *hist = vb + E1;
    int *scan_tmp = hist + n_hist;
    unsigned *flags = (unsigned *)(scan_tmp + n_tmp);

    CK_TRY(cudaMemsetAsync(flags, 0, sizeof(unsigned), s), "cudaMemsetAsync flags");
    CK_TRY(cudaMemsetAsync(g->slot, 0xff, sizeof(int) * N, s), "cudaMemsetAsync slot");
    const int blocks = g->num_sms * 4;
    if (E > 0)
        k_validate<<<blocks, 256, 0, s>>>(src, dst, E, N, key_dst, key_src, ids, ids2, flags);
    if (n_in > 0) k_slots<<<blocks, 256, 0, s>>>(input_nodes, n_in, N, g->slot, flags);
    CK_TRY(cudaGetLastError(), "validate launch");
    unsigned hflags = 0;
    CK_TRY(cudaMemcpyAsync(&hflags, flags, sizeof(unsigned), cudaMemcpyDeviceToHost, s),
           "cudaMemcpyAsync flags");
    CK_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize (validation)");
    if (hflags & kBadEdge) return fail(CK_ERR_INVALID_ARG, "an edge endpoint is outside [0, N)");
    if (hflags & kBadInput) return fail(CK_ERR_INVALID_ARG, "an input node is outside [0, N)");
    if (hflags & kDupInput) return fail(CK_ERR_INVALID_ARG, "input_nodes repeats a node");

    int key_bits = 0;  // keys are < N
    while (key_bits < 31 && ((int64_t)1 << key_bits) < (int64_t)N) ++key_bits;
    struct Side {
        int *keys, *vals, *row_ptr, *col, *perm, *rowid;
        const int64_t *other, *own;
    } sides[2] = {{key_dst, ids, g->row_ptr, g->col, g->perm, g->rowid, src, dst},
                  {key_src, ids2, g->rowT_ptr, g->colT, g->permT, g->rowidT, dst, src}};
    for (auto &sd : sides) {
        int *ks = sd.keys, *vs = sd.vals;
        if (E > 0) {
            bool in_b = false;
            CK_TRY(radix_sort(sd.keys, sd.vals, kb, vb, E, key_bits, hist, scan_tmp, s, &in_b),
                   "radix sort");
            if (in_b) {
                ks = kb;
                vs = vb;
            }
            CK_TRY(cudaMemcpyAsync(sd.perm, vs, sizeof(int) * E, cudaMemcpyDeviceToDevice, s),
                   "copy perm");
            k_gather_other<<<blocks, 256, 0, s>>>(sd.other, sd.perm, E, sd.col);
            k_gather_other<<<blocks, 256, 0, s>>>(sd.own, sd.perm, E, sd.rowid);
        }
        k_row_ptr<<<(N + 256) / 256, 256, 0, s>>>(ks, E, N, sd.row_ptr);
        CK_TRY(cudaGetLastError(), "row_ptr launch");
        // the second side reuses kb/vb; stream order already serialises it
    }
    // Pieces, one per CTA (kCtasPerSm per SM), for each finish pass size.  The row weight is the
    // one (of a few) whose slowest piece is estimated fastest: part A at about
    // 1.5 ns per edge per 32 batch columns (1.2 ns in the forward, whose gathers
    // go through L2 alone in batches of four), a finish pass at about 0.8 us
    // (measured on the FlyGPT-shaped graph); ties go to the smaller weight.
    {
        const int P = num_pieces(g);
        std::vector<int> rp(N + 1);
        const int *rps[2] = {g->row_ptr, g->rowT_ptr};
        static const int weights[] = {1, 2, 3, 4, 6, 8, 12, 16, 20, 24};
        for (int d = 0; d < 2; ++d) {
            CK_TRY(cudaMemcpyAsync(rp.data(), rps[d], sizeof(int) * (N + 1), cudaMemcpyDeviceToHost, s),
                   "copy row pointers");
            CK_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize (row pointers)");
            std::vector<Cut> cuts;
            for (int wt : weights) cuts.push_back(cut_pieces(rp, (int)N, (int)E, P, wt));
            for (int v = 0; v < 3; ++v) {
                const double edge_us = (d == 0 ? 1.2e-3 : 1.5e-3) * (v == 0 ? 1 : v == 1 ? 2 : 4);
                int best = 0;
                double best_cost = 0.0;
                for (int i = 0; i < (int)cuts.size(); ++i) {
                    const double cost = cut_cost(cuts[i], P, kPassRows[v], edge_us, 0.8);
                    if (i == 0 || cost < best_cost) {
                        best = i;
                        best_cost = cost;
                    }
                }
                const std::vector<int> m = piece_meta(cuts[best], rp, (int)N, P);
                CK_TRY(cudaMalloc((void **)&g->piece[d][v], sizeof(int) * m.size()), "cudaMalloc piece");
                g->device_bytes += sizeof(int) * m.size();
                CK_TRY(cudaMemcpy(g->piece[d][v], m.data(), sizeof(int) * m.size(), cudaMemcpyHostToDevice),
                       "copy piece descriptions");
                g->max_rows[d][v] = cuts[best].max_rows;
                g->max_edges[d][v] = cuts[best].max_edges;
                g->row_weight[d][v] = weights[best];
            }
        }
    }
    // Shared-memory tilings (ck::Tiled), one per direction, when the caller asks
    // for them and the graph's state rows fit a few CTAs' shared memory: built
    // on the host from the compressed rows.
    if (graph_flags & CK_GRAPH_TILING) {
        CK_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize (graph build)");
        std::vector<int> rp(N + 1), cl((size_t)E), pm((size_t)E);
        const int *rps[2] = {g->row_ptr, g->rowT_ptr};
        const int *cls[2] = {g->col, g->colT};
        const int *pms[2] = {g->perm, g->permT};
        for (int d = 0; d < 2; ++d) {
            // a chunk of at least one node per C, at 32 columns, must fit: skip large graphs early
            if (!tiled_fits(d, kTiledMaxBp, 0, 0, (N + 7) / 8)) continue;
            CK_TRY(cudaMemcpy(rp.data(), rps[d], sizeof(int) * (N + 1), cudaMemcpyDeviceToHost),
                   "copy row pointers (tiling)");
            if (E > 0) {
                CK_TRY(cudaMemcpy(cl.data(), cls[d], sizeof(int) * E, cudaMemcpyDeviceToHost),
                       "copy columns (tiling)");
                CK_TRY(cudaMemcpy(pm.data(), pms[d], sizeof(int) * E, cudaMemcpyDeviceToHost),
                       "copy permutation (tiling)");
            }
            TiledHost th = tile_direction(d, N, E, g->num_sms, rp, cl, pm);
            if (th.t.C == 0) continue;
            Tiled &t = g->tiled[d];
            t = th.t;
            struct Arr {
                int **dst;
                const std::vector<int> *src;
            } arrs[] = {{&t.meta, &th.meta}, {&t.ptr, &th.ptr}, {&t.col, &th.col},
                        {&t.perm, &th.perm}, {&t.rowid, &th.rowid}};
            for (auto &a : arrs) {
                const size_t bytes = sizeof(int) * a.src->size();
                CK_TRY(cudaMalloc((void **)a.dst, bytes), "cudaMalloc tiling");
                g->device_bytes += bytes;
                CK_TRY(cudaMemcpy(*a.dst, a.src->data(), bytes, cudaMemcpyHostToDevice), "copy tiling");
            }
        }
    }
    // Edge-indexed arrays to pinned host memory, read in place by the kernels
    // (on a Grace-Blackwell node over the coherent CPU-GPU link): the graph
    // then holds O(N) device memory.  Every array is complete before the copy
    // (the piece cut above synchronised the stream after the last kernel).
    if (graph_flags & CK_GRAPH_EDGES_IN_HOST_MEMORY) {
        CK_TRY(cudaStreamSynchronize(s), "cudaStreamSynchronize (graph build)");
        const size_t Et = E > 0 ? (size_t)E : 1;  // tiled arrays' length
        int **arrays[12] = {&g->col, &g->perm, &g->colT, &g->permT, &g->rowid, &g->rowidT};
        size_t lens[12] = {E1, E1, E1, E1, E1, E1};
        int na = 6;
        for (int d = 0; d < 2; ++d) {
            if (g->tiled[d].C == 0) continue;
            for (int **p : {&g->tiled[d].col, &g->tiled[d].perm, &g->tiled[d].rowid}) {
                arrays[na] = p;
                lens[na++] = Et;
            }
        }
        void *h[12] = {};
        auto drop = [&]() {
            for (void *p : h)
                if (p) cudaFreeHost(p);
        };
        // all copies first, so that a failure leaves the device arrays in place
        for (int i = 0; i < na; ++i) {
            e = cudaHostAlloc(&h[i], sizeof(int) * lens[i], cudaHostAllocMapped | cudaHostAllocPortable);
            if (e == cudaSuccess) e = cudaMemcpy(h[i], *arrays[i], sizeof(int) * lens[i], cudaMemcpyDeviceToHost);
            void *dv = nullptr;
            if (e == cudaSuccess) e = cudaHostGetDevicePointer(&dv, h[i], 0);
            if (e != cudaSuccess) {
                drop();
                return (e == cudaErrorMemoryAllocation)
                           ? fail(CK_ERR_OUT_OF_MEMORY, "graph in host memory: %s", cudaGetErrorString(e))
                           : cuda_fail(e, "graph in host memory");
            }
            if (dv != h[i]) {
                // the kernels take the pointer as is and the handle frees it
                // with cudaFreeHost: both need the unified address space
                drop();
                return fail(CK_ERR_UNSUPPORTED, "host memory is not mapped at the same address on the device");
            }
        }
        for (int i = 0; i < na; ++i) {
            cudaFree(*arrays[i]);
            *arrays[i] = (int *)h[i];
            g->device_bytes -= sizeof(int) * lens[i];
            g->host_bytes += sizeof(int) * lens[i];
        }
        g->edges_in_host = 1;
    }
#undef CK_TRY
    return CK_OK;
}

}  // namespace ck
