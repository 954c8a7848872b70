// ck_sgd_update: the plain SGD step param <- param - lr * grad, so that a whole
// training step (forward, backward, update) can run on the device and be
// captured as one CUDA graph (TrainKernel page, intro: a captured step holds
// the forward, gradients and the SGD update).
#include "ck_internal.h"

namespace ck {
namespace {

__global__ void k_sgd(float *__restrict__ p, const float *__restrict__ g, int64_t n, float lr) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (((uintptr_t)p | (uintptr_t)g) % 16 == 0) {
        const int64_t n4 = n / 4;
        float4 *p4 = reinterpret_cast<float4 *>(p);
        const float4 *g4 = reinterpret_cast<const float4 *>(g);
        for (int64_t i = i0; i < n4; i += stride) {
            float4 a = p4[i];
            const float4 b = g4[i];
            a.x = fmaf(-lr, b.x, a.x);
            a.y = fmaf(-lr, b.y, a.y);
            a.z = fmaf(-lr, b.z, a.z);
            a.w = fmaf(-lr, b.w, a.w);
            p4[i] = a;
        }
        for (int64_t i = 4 * n4 + i0; i < n; i += stride) p[i] = fmaf(-lr, g[i], p[i]);
    } else {
        for (int64_t i = i0; i < n; i += stride) p[i] = fmaf(-lr, g[i], p[i]);
    }
}

}  // namespace
}  // namespace ck

using namespace ck;

extern "C" ck_status ck_sgd_update(float *param, const float *grad, int64_t n, float lr,
                                   void *stream) {
    if (n < 0) return fail(CK_ERR_INVALID_ARG, "n = %lld < 0", (long long)n);
    if (n == 0) return CK_OK;
    if (!param || !grad) return fail(CK_ERR_INVALID_ARG, "a required pointer is NULL");
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    const int64_t want = (n / 4 + 255) / 256;
    const int blocks = (int)(want < 4 * sms ? (want > 0 ? want : 1) : 4 * sms);
    k_sgd<<<blocks, 256, 0, (cudaStream_t)stream>>>(param, grad, n, lr);
    e = cudaGetLastError();
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "k_sgd launch");
}
