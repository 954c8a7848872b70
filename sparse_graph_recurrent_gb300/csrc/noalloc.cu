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

// Device address of g_forward_scratch, looked up once per device.  In host
// code the array's name only stands in for the symbol; kernels need this.
constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

ck_status static_scratch(int dev, void **out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(CK_ERR_UNSUPPORTED, "device id %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_forward_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress (static forward scratch)");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return CK_OK;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

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
    if (((uintptr_t)saved & 15u) != 0) return fail(CK_ERR_INVALID_ARG, "saved must be 16-byte aligned");
    if (saved_bytes < p.saved_bytes)
        return fail(CK_ERR_WORKSPACE, "saved too small: %zu < %zu", saved_bytes, p.saved_bytes);

    // The forward touches only these scratch regions: control words, carries,
    // permuted edge values and row sums.  Lay them out back to back.
    Plan q = p;
    size_t off = 0;
    q.off_ctrl = off;
    off += q.ctrl_bytes;
    q.off_carry = off;
    off = up256(off + 8 * (size_t)q.P * q.Bp);
    q.off_wperm = off;
    off = up256(off + 4 * (size_t)(q.E > 0 ? q.E : 1));
    q.off_rowsum = off;
    off = up256(off + 4 * (size_t)q.N * q.Bp);
    q.off_dwperm = q.off_G = q.off_da = q.off_lacc = 0;  // backward-only regions, unused here
    q.scratch_bytes = off;
    if (off > kStaticScratchBytes)
        return fail(CK_ERR_UNSUPPORTED,
                    "this shape needs %zu bytes of forward scratch; the static array holds %zu "
                    "(use ck_forward with a caller-allocated scratch buffer)",
                    off, kStaticScratchBytes);
    void *scratch = nullptr;
    st = static_scratch(dev, &scratch);
    if (st != CK_OK) return st;
    FwdIO io{edge_values, leak, bias, drives, state0, states_out, (float *)saved, scratch};
    int64_t launches = 0;
    return launch_forward(g, q, io, (cudaStream_t)stream, &launches);
}
