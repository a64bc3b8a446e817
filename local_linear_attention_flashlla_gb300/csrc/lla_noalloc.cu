// lla_forward_noalloc: the tensor-core forward pass with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory at the point where they run the forward pass:
// for example a host program whose device memory is entirely owned by another allocator
// (a framework that reserves the GPU's memory up front, so cudaMalloc fails or fragments its
// pool), or a service with a fixed latency budget that must not pay for an allocation, which
// can synchronise the device.  For them this entry point keeps the tensor path's scratch
// (fp16 operand copies, kbar and the CG iterate) in a file-scope __device__ array that exists
// for as long as the library is loaded, and it calls no allocating routine.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "../../include/lla.h"
#include "lla_internal.h"

namespace lla {
namespace {

// Fixed scratch; every GPU that loads the library holds it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LLA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context.  In host code the array's name
// is only a host-side stand-in, not a device address, so the runtime is asked for the address
// with the caller's device current.  The lookup is repeated on every call rather than cached:
// the address belongs to the context that loaded the module, and a cached value would dangle
// after cudaDeviceReset (or any teardown of the primary context) reloads the module elsewhere.
// The lookup allocates nothing.
cudaError_t scratch_address(void** out) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace lla

extern "C" int lla_forward_noalloc(const void* q, const void* k, const void* v, void* out, float* rho,
                                   float* denom, int B, int H, int n, int d, float tau, float lambda,
                                   int cg_max_iters, float cg_tol, void* stream) {
    if (d != 64 && d != 128)
        return lla::set_error(LLA_ERR_UNSUPPORTED, "lla_forward_noalloc: head dim d must be 64 or 128");
    if (B < 1 || H < 1 || n < 1)
        return lla::set_error(LLA_ERR_INVALID_ARG, "lla_forward_noalloc: B, H, n must be >= 1");
    const size_t need = lla_workspace_size(LLA_DTYPE_BF16, LLA_PATH_TENSOR, B, H, n, d);
    if (need > (size_t)LLA_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "lla_forward_noalloc: this problem needs %zu bytes of scratch, more than the fixed "
                 "%zu bytes (LLA_NOALLOC_SCRATCH_BYTES); use lla_forward or lla_forward_ex",
                 need, (size_t)LLA_NOALLOC_SCRATCH_BYTES);
        return lla::set_error(LLA_ERR_INVALID_ARG, msg);
    }
    void* ws = nullptr;
    cudaError_t e = lla::scratch_address(&ws);
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof(msg), "lla_forward_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        return lla::set_error(LLA_ERR_CUDA, msg);
    }
    // With a caller-provided workspace lla_forward_ex allocates nothing.
    return lla_forward_ex(LLA_DTYPE_BF16, LLA_PATH_TENSOR, q, k, v, out, rho, denom, nullptr, B, H, n, d, tau, lambda,
                          cg_max_iters, cg_tol, ws, (size_t)LLA_NOALLOC_SCRATCH_BYTES, stream);
}
