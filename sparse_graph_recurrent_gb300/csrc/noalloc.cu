// ck_forward_static_scratch: the forward pass with its temporary memory taken
// from an array compiled into the library instead of a buffer the caller
// allocates.
//
// Some callers cannot allocate device memory when they run the forward: a
// plugin loaded into a host application whose memory manager owns the whole
// device and refuses allocations it did not make, or a control loop that must
// not allocate once it is running.  They still own their inputs and outputs;
// only the temporary workspace comes from here.
//
// The array is file-scope device memory of a fixed size: every GPU that loads
// the library holds it until the process exits, and every call of this entry
// point shares it.
#include <cstring>
#include <mutex>

#include "ck_internal.h"

namespace ck {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_forward_scratch[kStaticScratchBytes];

// Device address of g_forward_scratch on each device.  In host code the
// array's name only stands in for the symbol; kernels need this address.  It
// is looked up again on every call made outside a stream capture (a reset of
// the device's primary context reloads the module and moves the array), and
// the last address is reused inside a capture, where the lookup may not run.
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

ck_status static_scratch(int dev, cudaStream_t stream, void **out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(CK_ERR_UNSUPPORTED, "device id %d out of range", dev);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cap == cudaStreamCaptureStatusNone || !g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_forward_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress (static forward scratch)");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return CK_OK;
}

}  // namespace
}  // namespace ck

using namespace ck;

extern "C" ck_status ck_forward_static_scratch(const ck_graph *g, const float *edge_values,
                                               const float *leak, const float *bias,
                                               const float *drives, const float *state0,
                                               int64_t B, int64_t T, int64_t microsteps,
                                               float *states_out, void *saved,
                                               size_t saved_bytes, void *stream) {
    if (!g) return fail(CK_ERR_INVALID_ARG, "graph handle is NULL");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != g->device)
        return fail(CK_ERR_INVALID_ARG, "graph was built on device %d, current device is %d",
                    g->device, dev);
    Plan p;
    ck_status st = make_plan(g, B, T, microsteps, &p);
    if (st != CK_OK) return st;
    if ((g->E > 0 && !edge_values) || !leak || !bias || !state0 || !states_out || !saved ||
        (g->n_in > 0 && !drives))
        return fail(CK_ERR_INVALID_ARG, "a required pointer is NULL");
    if (((uintptr_t)saved & 31u) != 0) return fail(CK_ERR_INVALID_ARG, "saved must be 32-byte aligned");
    if (saved_bytes < p.saved_bytes)
        return fail(CK_ERR_WORKSPACE, "saved too small: %zu < %zu", saved_bytes, p.saved_bytes);

    // the regions the forward touches, laid out back to back in the array
    Plan q = p;
    forward_only_scratch(&q);
    if (q.scratch_bytes > kStaticScratchBytes)
        return fail(CK_ERR_UNSUPPORTED,
                    "this shape needs %zu bytes of forward scratch; the static array holds %zu "
                    "(use ck_forward with a caller-allocated scratch buffer)",
                    q.scratch_bytes, kStaticScratchBytes);
    void *scratch = nullptr;
    st = static_scratch(dev, (cudaStream_t)stream, &scratch);
    if (st != CK_OK) return st;
    FwdIO io{edge_values, leak, bias, drives, state0, states_out, (float *)saved, scratch};
    int64_t launches = 0;
    return launch_forward(g, q, io, (cudaStream_t)stream, &launches);
}

extern "C" ck_status ck_query_status_static(void *stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "pending CUDA error");
    int word = 0;
    // the control block sits at offset 0 of the array (forward_only_scratch)
    e = cudaMemcpyFromSymbol(&word, g_forward_scratch, sizeof(int), kStatusOffset,
                             cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol (status word)");
    if (word == kDevTimeout) return fail(CK_ERR_TIMEOUT, "a device-side wait timed out");
    if (word == kDevBounds)
        return fail(CK_ERR_INTERNAL, "an index out of bounds was caught and its access skipped "
                                     "(bounds-checked build)");
    if (word != kDevOk) return fail(CK_ERR_INTERNAL, "device status word %d", word);
    return CK_OK;
}
