// Bandwidth probes: the denominators of the L2 roofline.
//
// The recurrence kernels read almost all their bytes from L2 (the state rows
// they gather and the graph stay resident there), so their ceiling is the
// rate at which the SMs can pull data out of L2, which the device properties
// do not state.  These two kernels measure it on the running GPU with the same
// load instruction the hot path uses (16-byte L2-cached loads):
//   k_probe_read    streams over a buffer `reps` times (dense read);
//   k_probe_gather  reads whole rows picked by an index list, LPE lanes per
//                   row, like the forward gather.
// Each thread folds what it read into one value and writes it only if it
// equals a value no input produces, so the loads cannot be dropped.
//
// A third probe, k_probe_barrier*, times grid-barrier schemes on their own:
// the latency floor under the recurrence kernels' microsteps, and the
// alternatives to their counter barrier, each measured the same way.
#include <cooperative_groups.h>

#include "ck_internal.h"

namespace ck {
namespace {

constexpr int kProbeThreads = 512;

__global__ void __launch_bounds__(kProbeThreads) k_probe_read(const float4 *__restrict__ buf,
                                                             size_t n4, int reps,
                                                             float *__restrict__ sink) {
    float acc = 0.f;
    const size_t stride = (size_t)gridDim.x * kProbeThreads;
    for (int r = 0; r < reps; ++r) {
        size_t i = (size_t)blockIdx.x * kProbeThreads + threadIdx.x;
        for (; i + 3 * stride < n4; i += 4 * stride) {
            float4 a = __ldcg(buf + i), b = __ldcg(buf + i + stride);
            float4 c = __ldcg(buf + i + 2 * stride), d = __ldcg(buf + i + 3 * stride);
            acc += (a.x + b.y) + (c.z + d.w);
        }
        for (; i < n4; i += stride) {
            float4 a = __ldcg(buf + i);
            acc += a.x;
        }
    }
    if (acc == 1.2345e-30f) sink[0] = acc;
}

__global__ void __launch_bounds__(kProbeThreads) k_probe_gather(
    const float *__restrict__ rows, int row_floats, const int *__restrict__ idx, size_t nidx,
    float *__restrict__ sink) {
    const int lpe = row_floats / 4;  // lanes per row
    const int epw = 32 / lpe;        // rows per warp instruction
    const int lane = threadIdx.x & 31, g = lane / lpe, lig = lane - g * lpe;
    const size_t warp = ((size_t)blockIdx.x * kProbeThreads + threadIdx.x) >> 5;
    const size_t nwarps = ((size_t)gridDim.x * kProbeThreads) >> 5;
    float acc = 0.f;
    if (g < epw) {
        for (size_t base = warp * epw * 8; base < nidx; base += nwarps * epw * 8) {
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const size_t k = base + (size_t)q * epw + g;
                v[q] = k < nidx ? __ldcg(reinterpret_cast<const float4 *>(
                                      rows + (size_t)__ldg(idx + k) * row_floats) + lig)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) acc += v[q].x + v[q].w;
        }
    }
    if (acc == 1.2345e-30f) sink[0] = acc;
}

// Dense read with a chosen shape: DEPTH independent loads of W bytes (16, or
// 32 with the 256-bit vector load of sm_100 and later) in flight per thread
// before any is used, `ctas_per_sm` CTAs of blockDim.x threads on every SM.  A
// sweep over these shapes finds the highest rate the SMs can pull from L2, so a
// fraction against it is not flattered by a weak probe.
template <int DEPTH, int MAXT, int W>
__global__ void __launch_bounds__(MAXT) k_probe_read_shape(const float *__restrict__ buf,
                                                          size_t nv, int reps,
                                                          float *__restrict__ sink) {
    float acc = 0.f;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (int r = 0; r < reps; ++r) {
        size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
        for (; i + (DEPTH - 1) * stride < nv; i += DEPTH * stride) {
            if constexpr (W == 16) {
                const float4 *b4 = reinterpret_cast<const float4 *>(buf);
                float4 v[DEPTH];
#pragma unroll
                for (int d = 0; d < DEPTH; ++d) v[d] = __ldcg(b4 + i + d * stride);
#pragma unroll
                for (int d = 0; d < DEPTH; ++d) acc += v[d].x + v[d].w;
            } else {
                float v[DEPTH][8];
#pragma unroll
                for (int d = 0; d < DEPTH; ++d)
                    asm volatile("ld.global.cg.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                                 : "=f"(v[d][0]), "=f"(v[d][1]), "=f"(v[d][2]), "=f"(v[d][3]),
                                   "=f"(v[d][4]), "=f"(v[d][5]), "=f"(v[d][6]), "=f"(v[d][7])
                                 : "l"(buf + (i + d * stride) * 8));
#pragma unroll
                for (int d = 0; d < DEPTH; ++d) acc += v[d][0] + v[d][7];
            }
        }
        // the tail (every byte the caller counts is read)
        for (; i < nv; i += stride) {
            if constexpr (W == 16) {
                acc += __ldcg(reinterpret_cast<const float4 *>(buf) + i).y;
            } else {
                float v[8];
                asm volatile("ld.global.cg.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                             : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]),
                               "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                             : "l"(buf + i * 8));
                acc += v[1];
            }
        }
    }
    if (acc == 1.2345e-30f) sink[0] = acc;
}

// ------------------------------------------------------ grid-barrier probe
//
// `ctas` persistent CTAs of kBarThreads threads; each crossing, every CTA
// writes rows_per_cta rows of 32 floats (like a finish pass publishing its
// rows) and then crosses a grid barrier of the chosen scheme.  Words: [0] the
// arrival counter, [kFlagBase + k * kFlagStride] the release flags.  Every
// wait gives up after `lim` ns, records 1 in *status and makes its CTA (and,
// through the status word, every CTA) stop; the cluster schemes release their
// members on every path, so each CTA reaches the final cluster barrier.
constexpr int kBarThreads = 256;
constexpr int kFlagBase = 1024, kFlagStride = 1040;
static_assert(kFlagBase + 7 * kFlagStride < CK_PROBE_BARRIER_WORDS, "flag words");

__device__ __forceinline__ unsigned long long pb_clock() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void pb_red_release(unsigned *p) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p) : "memory");
}
__device__ __forceinline__ unsigned pb_atom_release(unsigned *p) {
    unsigned o;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], 1;" : "=r"(o) : "l"(p) : "memory");
    return o;
}
__device__ __forceinline__ unsigned pb_atom_acq_rel(unsigned *p) {
    unsigned o;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(o) : "l"(p) : "memory");
    return o;
}
__device__ __forceinline__ unsigned pb_ld(const unsigned *p, bool relaxed) {
    unsigned v;
    if (relaxed) asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    else asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void pb_fence() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void pb_st(unsigned *p, unsigned v, bool release) {
    if (release) asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
    else asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int pb_status(const int *s) { return *(volatile const int *)s; }

// poll until *w >= target (acquire); false once the limit passes or another
// CTA recorded a timeout
__device__ bool pb_poll(const unsigned *w, unsigned target, bool relaxed, int *status,
                        unsigned long long lim) {
    const unsigned long long t0 = pb_clock();
    for (unsigned n = 0; pb_ld(w, relaxed) < target; ++n) {
        if ((n & 7) != 7) continue;
        if (pb_status(status) != 0) return false;
        if (pb_clock() - t0 > lim) {
            atomicExch(status, 1);
            return false;
        }
    }
    if (relaxed) pb_fence();
    return true;
}

__device__ __forceinline__ void pb_write_rows(float *rows, int rows_per_cta, int it) {
    float *r = rows + (size_t)blockIdx.x * rows_per_cta * 32;
    for (int i = threadIdx.x; i < rows_per_cta * 32; i += blockDim.x) r[i] = (float)(it + i);
}

// schemes without clusters (ck_barrier_scheme 0..4)
__global__ void __launch_bounds__(kBarThreads) k_probe_barrier(int scheme, unsigned *words,
                                                               int *status, float *rows,
                                                               int crossings, int rows_per_cta,
                                                               unsigned long long lim) {
    __shared__ int s_ok;
    const unsigned P = gridDim.x;
    for (int it = 0; it < crossings; ++it) {
        pb_write_rows(rows, rows_per_cta, it);
        __syncthreads();
        if (threadIdx.x == 0) {
            const unsigned target = (unsigned)(it + 1) * P;
            bool ok = true;
            if (scheme == CK_BARRIER_COUNTER || scheme == CK_BARRIER_COUNTER_RELAXED) {
                pb_red_release(words);
                ok = pb_poll(words, target, scheme == CK_BARRIER_COUNTER_RELAXED, status, lim);
            } else if (scheme == CK_BARRIER_COUNTER_RETURNING) {
                if (pb_atom_release(words) + 1u >= target) pb_fence();
                else ok = pb_poll(words, target, false, status, lim);
            } else {  // counter + release flag(s)
                const int K = scheme == CK_BARRIER_FLAG ? 1 : 8;
                if (pb_atom_acq_rel(words) + 1u >= target) {
                    if (K > 1) pb_fence();
                    for (int k = 0; k < K; ++k) pb_st(words + kFlagBase + k * kFlagStride, (unsigned)it + 1, K == 1);
                } else {
                    ok = pb_poll(words + kFlagBase + (blockIdx.x % K) * kFlagStride, (unsigned)it + 1,
                                 false, status, lim);
                }
            }
            s_ok = ok && pb_status(status) == 0;
        }
        __syncthreads();
        if (!s_ok) break;
    }
}

__device__ __forceinline__ unsigned pb_smem(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void pb_remote_arrive(unsigned long long *mb, unsigned rank) {
    unsigned r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(pb_smem(mb)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(r) : "memory");
}
__device__ bool pb_mb_wait(unsigned long long *mb, unsigned parity, int *status, unsigned long long lim) {
    const unsigned long long t0 = pb_clock();
    for (unsigned n = 0;; ++n) {
        unsigned done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
            "selp.u32 %0, 1, 0, p; }"
            : "=r"(done) : "r"(pb_smem(mb)), "r"(parity) : "memory");
        if (done) return true;
        if ((n & 7) != 7) continue;
        if (pb_status(status) != 0) return false;
        if (pb_clock() - t0 > lim) {
            atomicExch(status, 1);
            return false;
        }
    }
}

// cluster schemes: CS CTAs first meet inside their cluster (MB false: the
// hardware cluster barrier; MB true: remote mbarrier arrivals on the leader),
// the leader makes the cluster's one arrival on the counter and polls it,
// then releases its members the same way.
template <int CS, bool MB>
__global__ void __launch_bounds__(kBarThreads) k_probe_barrier_cluster(unsigned *words, int *status,
                                                                       float *rows, int crossings,
                                                                       int rows_per_cta,
                                                                       unsigned long long lim) {
    namespace cgr = cooperative_groups;
    __shared__ __align__(8) unsigned long long mb_in, mb_out;
    __shared__ int s_ok;
    cgr::cluster_group cl = cgr::this_cluster();
    const unsigned Q = gridDim.x / CS, rank = cl.block_rank();
    if (MB && threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(pb_smem(&mb_in)), "r"(CS - 1) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(pb_smem(&mb_out)), "r"(1) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    cl.sync();
    for (int it = 0; it < crossings; ++it) {
        pb_write_rows(rows, rows_per_cta, it);
        if (MB) {
            __syncthreads();
            if (threadIdx.x == 0) {
                bool ok;
                if (rank == 0) {
                    ok = pb_mb_wait(&mb_in, it & 1, status, lim);
                    if (ok) {
                        pb_red_release(words);
                        ok = pb_poll(words, (unsigned)(it + 1) * Q, false, status, lim);
                    }
                    for (unsigned r = 1; r < CS; ++r) pb_remote_arrive(&mb_out, r);  // on every path
                } else {
                    pb_remote_arrive(&mb_in, 0);
                    ok = pb_mb_wait(&mb_out, it & 1, status, lim);
                }
                s_ok = ok && pb_status(status) == 0;
            }
            __syncthreads();
            if (!s_ok) break;
        } else {
            cl.sync();
            if (rank == 0 && threadIdx.x == 0) {
                pb_red_release(words);
                s_ok = pb_poll(words, (unsigned)(it + 1) * Q, false, status, lim) ? 1 : 0;
            }
            cl.sync();
            // every CTA of the cluster takes the leader's decision
            if (!*cl.map_shared_rank(&s_ok, 0)) break;
        }
    }
    cl.sync();  // no CTA leaves while a peer may still reach its shared memory
}

int probe_blocks() {
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms * 2;
}

}  // namespace
}  // namespace ck

using namespace ck;

extern "C" ck_status ck_probe_read(const void *buf, size_t bytes, int64_t reps, float *sink,
                                   void *stream) {
    if (!buf || !sink || reps < 1 || bytes < 16 || ((uintptr_t)buf & 15u))
        return fail(CK_ERR_INVALID_ARG, "probe_read: bad buffer, size or reps");
    k_probe_read<<<probe_blocks(), kProbeThreads, 0, (cudaStream_t)stream>>>(
        (const float4 *)buf, bytes / 16, (int)reps, sink);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "k_probe_read launch");
}

extern "C" ck_status ck_probe_gather(const float *rows, int64_t nrows, int64_t row_floats,
                                     const int32_t *idx, int64_t nidx, float *sink,
                                     void *stream) {
    if (!rows || !idx || !sink || nrows < 1 || nidx < 1 ||
        (row_floats != 8 && row_floats != 16 && row_floats != 32 && row_floats != 64 &&
         row_floats != 128) || ((uintptr_t)rows & 15u))
        return fail(CK_ERR_INVALID_ARG, "probe_gather: bad rows, row width (8..128) or index list");
    k_probe_gather<<<probe_blocks(), kProbeThreads, 0, (cudaStream_t)stream>>>(
        rows, (int)row_floats, idx, (size_t)nidx, sink);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "k_probe_gather launch");
}

extern "C" ck_status ck_probe_read_shape(const void *buf, size_t bytes, int64_t reps,
                                         int64_t load_bytes, int64_t depth, int64_t threads,
                                         int64_t ctas_per_sm, float *sink, void *stream) {
    if (!buf || !sink || reps < 1 || bytes < 32 || ((uintptr_t)buf & 31u))
        return fail(CK_ERR_INVALID_ARG, "probe_read_shape: bad buffer (32-byte aligned), size or reps");
    if ((threads != 128 && threads != 256 && threads != 512 && threads != 1024) ||
        ctas_per_sm < 1 || threads * ctas_per_sm > 2048)
        return fail(CK_ERR_INVALID_ARG,
                    "probe_read_shape: threads in {128, 256, 512, 1024}, threads x ctas_per_sm <= 2048");
    using Fn = void (*)(const float *, size_t, int, float *);
    Fn fn = nullptr;
    const bool big = threads > 512;  // 1024-thread CTAs get at most 64 registers a thread
#define CK_PICK(W)                                                                        \
    switch (depth) {                                                                      \
    case 2: fn = big ? k_probe_read_shape<2, 1024, W> : k_probe_read_shape<2, 512, W>; break; \
    case 4: fn = big ? k_probe_read_shape<4, 1024, W> : k_probe_read_shape<4, 512, W>; break; \
    case 8: fn = big ? k_probe_read_shape<8, 1024, W> : k_probe_read_shape<8, 512, W>; break; \
    case 16: fn = big ? nullptr : k_probe_read_shape<16, 512, W>; break;                  \
    default: break;                                                                       \
    }
    if (load_bytes == 16) {
        CK_PICK(16)
    } else if (load_bytes == 32) {
        CK_PICK(32)
    }
#undef CK_PICK
    if (!fn)
        return fail(CK_ERR_INVALID_ARG,
                    "probe_read_shape: load_bytes in {16, 32}, depth in {2, 4, 8, 16} (16 only "
                    "with <= 512 threads)");
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    fn<<<sms * (int)ctas_per_sm, (int)threads, 0, (cudaStream_t)stream>>>(
        (const float *)buf, bytes / (size_t)load_bytes, (int)reps, sink);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "k_probe_read_shape launch");
}

#define PB_TRY(call, what)                       \
    do {                                         \
        const cudaError_t e_ = (call);           \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

extern "C" ck_status ck_probe_grid_barrier(int64_t scheme, int64_t ctas, int64_t cluster,
                                           int64_t crossings, int64_t rows_per_cta, float *rows,
                                           uint32_t *words, int32_t *status, void *stream) {
    const bool clustered = scheme == CK_BARRIER_CLUSTER_SYNC || scheme == CK_BARRIER_CLUSTER_MBARRIER;
    if (scheme < CK_BARRIER_COUNTER || scheme > CK_BARRIER_CLUSTER_MBARRIER)
        return fail(CK_ERR_INVALID_ARG, "probe_grid_barrier: unknown scheme %lld", (long long)scheme);
    if (clustered ? (cluster != 2 && cluster != 4 && cluster != 8) : cluster != 1)
        return fail(CK_ERR_INVALID_ARG, "probe_grid_barrier: cluster 1 (2, 4 or 8 for the cluster schemes)");
    if (ctas < 1 || ctas % cluster != 0 || crossings < 1 || crossings > (1 << 24) || rows_per_cta < 0 ||
        rows_per_cta > 64 || !words || !status || (rows_per_cta > 0 && !rows))
        return fail(CK_ERR_INVALID_ARG,
                    "probe_grid_barrier: ctas a multiple of cluster, 1 <= crossings <= 2^24, "
                    "0 <= rows_per_cta <= 64, buffers present");
    int dev = 0, sms = 1;
    PB_TRY(cudaGetDevice(&dev), "cudaGetDevice");
    PB_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
    const cudaStream_t s = (cudaStream_t)stream;
    PB_TRY(cudaMemsetAsync(words, 0, sizeof(uint32_t) * CK_PROBE_BARRIER_WORDS, s), "clear words");
    PB_TRY(cudaMemsetAsync(status, 0, sizeof(int32_t), s), "clear status");
    int it = (int)crossings, rpc = (int)rows_per_cta;
    unsigned long long lim = (unsigned long long)options().timeout_ns.load();
    if (!clustered) {
        int occ = 0;
        PB_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_probe_barrier, kBarThreads, 0),
               "occupancy");
        if ((int64_t)occ * sms < ctas)
            return fail(CK_ERR_UNSUPPORTED, "probe_grid_barrier: %lld CTAs are not co-resident", (long long)ctas);
        int sc = (int)scheme;
        void *args[] = {&sc, &words, &status, &rows, &it, &rpc, &lim};
        PB_TRY(cudaLaunchCooperativeKernel((const void *)k_probe_barrier, dim3((unsigned)ctas), dim3(kBarThreads),
                                           args, 0, s),
               "k_probe_barrier launch");
        return CK_OK;
    }
    using Fn = void (*)(unsigned *, int *, float *, int, int, unsigned long long);
    const bool mb = scheme == CK_BARRIER_CLUSTER_MBARRIER;
    Fn fn = cluster == 2 ? (mb ? k_probe_barrier_cluster<2, true> : k_probe_barrier_cluster<2, false>)
          : cluster == 4 ? (mb ? k_probe_barrier_cluster<4, true> : k_probe_barrier_cluster<4, false>)
                         : (mb ? k_probe_barrier_cluster<8, true> : k_probe_barrier_cluster<8, false>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(kBarThreads);
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeCooperative;
    at[1].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    int nclusters = 0;
    PB_TRY(cudaOccupancyMaxActiveClusters(&nclusters, (const void *)fn, &cfg), "cluster occupancy");
    if ((int64_t)nclusters * cluster < ctas)
        return fail(CK_ERR_UNSUPPORTED, "probe_grid_barrier: %lld CTAs in clusters of %lld are not co-resident",
                    (long long)ctas, (long long)cluster);
    unsigned *w = words;
    int *st = status;
    PB_TRY(cudaLaunchKernelEx(&cfg, fn, w, st, rows, it, rpc, lim), "k_probe_barrier_cluster launch");
    return CK_OK;
}
#undef PB_TRY
