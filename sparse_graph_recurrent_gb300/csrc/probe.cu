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
