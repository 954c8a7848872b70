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
