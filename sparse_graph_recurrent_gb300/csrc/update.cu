// ck_sgd_update: the plain SGD step param <- param - lr * grad, and
// ck_adam_update / ck_step_advance: an Adam step (Kingma and Ba, "Adam: A
// Method for Stochastic Optimization", Algorithm 1) whose step number lives in
// device memory, so that a whole training step (forward, backward, update) can
// run on the device and be captured as one CUDA graph that advances its own
// step count (TrainKernel page, intro: a captured step holds the forward,
// gradients and the parameter update).
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

// Adam over n floats at step t = *step (>= 1): first and second moments
// updated in place, then the bias-corrected step, in the order the
// definition gives it.
__global__ void k_adam(float *__restrict__ p, const float *__restrict__ g, float *__restrict__ m,
                       float *__restrict__ v, int64_t n, float lr, float b1, float b2, float eps,
                       const int64_t *__restrict__ step) {
    const float t = (float)*step;
    const float c1 = 1.f - powf(b1, t), c2 = 1.f - powf(b2, t);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float gi = g[i];
        const float mi = b1 * m[i] + (1.f - b1) * gi;
        const float vi = b2 * v[i] + (1.f - b2) * gi * gi;
        m[i] = mi;
        v[i] = vi;
        p[i] = p[i] - lr * (mi / c1) / (sqrtf(vi / c2) + eps);
    }
}

__global__ void k_step_advance(int64_t *step) { *step += 1; }

int update_blocks(int64_t n) {
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 1;
    const int64_t want = (n + 255) / 256;
    return (int)(want < 4 * sms ? (want > 0 ? want : 1) : 4 * sms);
}

}  // namespace
}  // namespace ck

using namespace ck;

extern "C" ck_status ck_adam_update(float *param, const float *grad, float *m, float *v, int64_t n,
                                    float lr, float beta1, float beta2, float eps,
                                    const int64_t *step, void *stream) {
    if (n < 0) return fail(CK_ERR_INVALID_ARG, "n = %lld < 0", (long long)n);
    if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) || !(eps > 0.f) ||
        !(lr == lr))
        return fail(CK_ERR_INVALID_ARG, "adam: betas in [0, 1), eps > 0, lr a number");
    if (!step) return fail(CK_ERR_INVALID_ARG, "adam: step is NULL");
    if (n == 0) return CK_OK;
    if (!param || !grad || !m || !v) return fail(CK_ERR_INVALID_ARG, "a required pointer is NULL");
    k_adam<<<update_blocks(n), 256, 0, (cudaStream_t)stream>>>(param, grad, m, v, n, lr, beta1, beta2,
                                                               eps, step);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "k_adam launch");
}

extern "C" ck_status ck_step_advance(int64_t *step, void *stream) {
    if (!step) return fail(CK_ERR_INVALID_ARG, "step is NULL");
    k_step_advance<<<1, 1, 0, (cudaStream_t)stream>>>(step);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "k_step_advance launch");
}

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
