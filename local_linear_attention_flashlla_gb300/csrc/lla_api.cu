// C ABI of liblla.so: argument checks, path selection, scratch handling, error reporting.
// The operation itself is described in include/lla.h.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "../../include/lla.h"
#include "lla_internal.h"
#include "tc_ptx.cuh"

namespace lla {

namespace {
thread_local char g_msg[512] = "";

int fail(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(LLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

int set_error(int status, const char* message) { return fail(status, "%s", message); }

__device__ unsigned g_device_error = 0;

namespace {
// Profiling events (call begin, main kernel begin, main kernel end, call end).
bool g_prof_on = false;
bool g_prof_valid = false;
cudaEvent_t g_ev[4] = {nullptr, nullptr, nullptr, nullptr};
}  // namespace

unsigned* device_error_word() {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    return static_cast<unsigned*>(ptr);
}

cudaError_t read_and_clear_device_error(unsigned* out, cudaStream_t stream) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_device_error, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*out) {
        e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return e;
        e = cudaStreamSynchronize(stream);
    }
    return e;
}


// Self-test of the timeout path.  One thread waits, through the same bounded, abortable mbarrier
// wait the tensor kernels use, for a phase of a barrier that nothing arrives on.  The wait gives up
// after its limit (about two seconds of wall time), raises the launch-wide abort word and returns;
// the thread then records the timeout in the device error word exactly as a tensor kernel's CTA
// does before it exits.  The kernel ends normally: no trap, no fault, nothing left waiting.
__device__ int g_selftest_abort = 0;

__global__ void lla_selftest_wait_kernel(unsigned* dev_err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int err;
    if (threadIdx.x == 0) {
        err = 0;
        tc::mbar_init(&bar, 1);
        tc::mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !tc::mbar_wait_abortable(&bar, 0, &err, &g_selftest_abort) && err)
        atomicOr(dev_err, (unsigned)kDevErrMbarTimeout);
}

// Launch a validated problem on the resolved path (workspace: caller's buffer, or null to take
// one from the stream-ordered pool for the duration of the call).
static int run_problem(Problem& p, int rpath, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (g_prof_on) {
        for (int i = 0; i < 4; ++i)
            if (!g_ev[i]) {
                cudaError_t e = cudaEventCreate(&g_ev[i]);
                if (e != cudaSuccess) return cuda_fail(e, "profiling event");
            }
        p.ev_main_begin = g_ev[1];
        p.ev_main_end = g_ev[2];
        cudaError_t e = cudaEventRecord(g_ev[0], stream);
        if (e != cudaSuccess) return cuda_fail(e, "profiling event record");
    }

    if (rpath == LLA_PATH_FP32) {
        cudaError_t e = launch_simt(p, stream);
        if (e != cudaSuccess) return cuda_fail(e, "fp32 path launch");
        if (g_prof_on) {
            e = cudaEventRecord(g_ev[3], stream);
            if (e != cudaSuccess) return cuda_fail(e, "profiling event record");
            g_prof_valid = true;
        }
        return LLA_OK;
    }

    const size_t need = tensor_workspace_bytes(p.B, p.H, p.n, p.d);
    void* ws = workspace;
    bool owned = false;
    if (ws) {
        if (workspace_bytes < need)
            return fail(LLA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
        if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
            return fail(LLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    } else {
        cudaError_t e = cudaMallocAsync(&ws, need, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
        owned = true;
    }
    const char* why = nullptr;
    cudaError_t e = launch_tensor(p, ws, stream, &why);
    if (owned) {
        cudaError_t e2 = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess && e2 != cudaSuccess) return cuda_fail(e2, "cudaFreeAsync(workspace)");
    }
    if (e != cudaSuccess) return cuda_fail(e, why ? why : "tensor path launch");
    if (g_prof_on) {
        e = cudaEventRecord(g_ev[3], stream);
        if (e != cudaSuccess) return cuda_fail(e, "profiling event record");
        g_prof_valid = true;
    }
    return LLA_OK;
}

// Scalar and shape checks shared by the forward entry points (pointers are checked by each).
static int check_forward_args(int dtype, int path, int B, int H, int n, int d, float tau, float lambda,
                              int cg_max_iters, float cg_tol, int* rpath_out) {
    if (B < 1 || H < 1 || n < 1) return fail(LLA_ERR_INVALID_ARG, "B, H, n must be >= 1 (got %d, %d, %d)", B, H, n);
    if ((long long)B * H > 65535LL) return fail(LLA_ERR_INVALID_ARG, "B*H must be <= 65535 (one grid row per slice)");
    if ((long long)B * H * n * d > (1LL << 40)) return fail(LLA_ERR_INVALID_ARG, "problem too large");
    if (d != 16 && d != 32 && d != 64 && d != 128)
        return fail(LLA_ERR_INVALID_ARG, "head dim d must be 16, 32, 64 or 128 (got %d)", d);
    if (!(tau > 0.f) || !(tau < 1e30f)) return fail(LLA_ERR_INVALID_ARG, "tau must be finite and > 0");
    if (!(lambda > 0.f) || !(lambda < 1e30f)) return fail(LLA_ERR_INVALID_ARG, "lambda must be finite and > 0");
    if (cg_max_iters < 1 || cg_max_iters > 4096) return fail(LLA_ERR_INVALID_ARG, "cg_max_iters must be in [1, 4096]");
    if (!(cg_tol >= 0.f) || !(cg_tol < 1e30f)) return fail(LLA_ERR_INVALID_ARG, "cg_tol must be finite and >= 0");
    if (dtype != LLA_DTYPE_BF16 && dtype != LLA_DTYPE_FP32) return fail(LLA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (path < LLA_PATH_AUTO || path > LLA_PATH_FP32) return fail(LLA_ERR_INVALID_ARG, "unknown path %d", path);
    int rpath = path;
    if (rpath == LLA_PATH_AUTO) rpath = (dtype == LLA_DTYPE_BF16 && (d == 64 || d == 128)) ? LLA_PATH_TENSOR : LLA_PATH_FP32;
    if (rpath == LLA_PATH_TENSOR && (dtype != LLA_DTYPE_BF16 || (d != 64 && d != 128)))
        return fail(LLA_ERR_UNSUPPORTED, "tensor path needs bf16 inputs and d in {64, 128}");
    *rpath_out = rpath;
    return LLA_OK;
}

// Scalar and shape checks of the backward entry points (pointers are checked by each).
static int check_backward_args(int dtype, int path, int B, int H, int n, int d, float tau, float lambda,
                               int cg_max_iters, float cg_tol, int* rpath_out) {
    if (B < 1 || H < 1 || n < 1) return fail(LLA_ERR_INVALID_ARG, "B, H, n must be >= 1 (got %d, %d, %d)", B, H, n);
    if ((long long)B * H > 65535LL) return fail(LLA_ERR_INVALID_ARG, "B*H must be <= 65535");
    return check_forward_args(dtype, path, B, H, n, d, tau, lambda, cg_max_iters, cg_tol, rpath_out);
}

// ---------------------------------------------------------------------------------------------
// Host-buffer forward: the (b, h) slices go through the device in chunks, on two library streams
// (chunk c on stream c % 2, with its own half of the device buffer), so chunk c's copy in runs
// while chunk c-1 computes and chunk c-1's copy out runs while chunk c computes.
namespace {
cudaStream_t g_hs[2] = {nullptr, nullptr};
cudaEvent_t g_he[3] = {nullptr, nullptr, nullptr};   // start (caller stream), done of stream 0 and 1

int host_streams() {
    for (int i = 0; i < 2; ++i)
        if (!g_hs[i]) {
            cudaError_t e = cudaStreamCreateWithFlags(&g_hs[i], cudaStreamNonBlocking);
            if (e != cudaSuccess) return cuda_fail(e, "host-buffer forward: stream");
        }
    for (int i = 0; i < 3; ++i)
        if (!g_he[i]) {
            cudaError_t e = cudaEventCreateWithFlags(&g_he[i], cudaEventDisableTiming);
            if (e != cudaSuccess) return cuda_fail(e, "host-buffer forward: event");
        }
    return LLA_OK;
}

inline size_t a256(size_t x) { return (x + 255) & ~size_t(255); }

// One half of the device buffer: q, k, v, out, rho, denom, cg_iters and the tensor workspace of a
// chunk of C slices.
struct HostChunk {
    size_t tin, trho, tden, ws, half;
    HostChunk(int dtype, int rpath, int C, int n, int d) {
        const size_t es = dtype == LLA_DTYPE_BF16 ? 2 : 4;
        tin = a256((size_t)C * n * d * es);
        trho = a256((size_t)C * n * d * 4);
        tden = a256((size_t)C * n * 4);
        ws = rpath == LLA_PATH_TENSOR ? a256(tensor_workspace_bytes(C, 1, n, d)) : 0;
        half = 4 * tin + trho + 2 * tden + ws;
    }
};

// The backward's half of the device buffer: q, k, v, dout (dtype), rho, dq, dk, dv (fp32),
// denom and cg_iters, and the backward workspace of a chunk of C slices.
struct HostBwdChunk {
    size_t tin, tf, tden, ws, half;
    HostBwdChunk(int dtype, int rpath, int C, int n, int d) {
        const size_t es = dtype == LLA_DTYPE_BF16 ? 2 : 4;
        tin = a256((size_t)C * n * d * es);
        tf = a256((size_t)C * n * d * 4);
        tden = a256((size_t)C * n * 4);
        ws = a256(backward_workspace_bytes(rpath, C, 1, n, d));
        half = 4 * tin + 4 * tf + 2 * tden + ws;
    }
};

int host_chunk_slices(int S, int chunk_slices) {
    if (chunk_slices > 0) return chunk_slices < S ? chunk_slices : S;
    const int c = (S + 7) / 8;   // about eight chunks
    return c < 1 ? 1 : c;
}
}  // namespace
}  // namespace lla

using lla::fail;
using lla::aligned16;

// Dynamic shared memory a block may have on sm_103a (227 KB).
#define LLA_DECODE_SMEM_LIMIT 232448

extern "C" {

int lla_version(void) { return 10000; }

const char* lla_last_error(void) { return lla::g_msg; }

int lla_resolve_path(int dtype, int path, int d) {
    if (path != LLA_PATH_AUTO) return path;
    if (dtype == LLA_DTYPE_BF16 && (d == 64 || d == 128)) return LLA_PATH_TENSOR;
    return LLA_PATH_FP32;
}

size_t lla_workspace_size(int dtype, int path, int B, int H, int n, int d) {
    if (B < 1 || H < 1 || n < 1 || d < 1) return 0;
    if (lla_resolve_path(dtype, path, d) != LLA_PATH_TENSOR) return 0;
    return lla::tensor_workspace_bytes(B, H, n, d);
}

int lla_forward_ex(int dtype, int path, const void* q, const void* k, const void* v, void* out, float* rho,
                   float* denom, int* cg_iters, int B, int H, int n, int d, float tau, float lambda,
                   int cg_max_iters, float cg_tol, void* workspace, size_t workspace_bytes, void* stream_) {
    lla::g_msg[0] = '\0';
    if (!q || !k || !v || !out || !rho || !denom) return fail(LLA_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(rho) ||
        !aligned16(denom))
        return fail(LLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    int rpath = 0;
    const int st = lla::check_forward_args(dtype, path, B, H, n, d, tau, lambda, cg_max_iters, cg_tol, &rpath);
    if (st != LLA_OK) return st;

    lla::Problem p{q, k, v, out, rho, denom, cg_iters, B, H, n, d, tau, lambda, cg_max_iters, cg_tol, dtype,
                   nullptr, nullptr, nullptr};
    return lla::run_problem(p, rpath, workspace, workspace_bytes, static_cast<cudaStream_t>(stream_));
}

size_t lla_forward_host_buffer_size(int dtype, int path, int B, int H, int n, int d, int chunk_slices) {
    int rpath = 0;
    if (lla::check_forward_args(dtype, path, B, H, n, d, 1.f, 1.f, 1, 0.f, &rpath) != LLA_OK || chunk_slices < 0)
        return 0;
    const int C = lla::host_chunk_slices(B * H, chunk_slices);
    return 2 * lla::HostChunk(dtype, rpath, C, n, d).half;
}

int lla_forward_host(int dtype, int path, const void* q, const void* k, const void* v, void* out, float* rho,
                     float* denom, int* cg_iters, int B, int H, int n, int d, float tau, float lambda,
                     int cg_max_iters, float cg_tol, int chunk_slices, void* device_buffer,
                     size_t device_buffer_bytes, void* stream_) {
    lla::g_msg[0] = '\0';
    if (!q || !k || !v || !out || !rho || !denom) return fail(LLA_ERR_INVALID_ARG, "null host pointer");
    int rpath = 0;
    int st = lla::check_forward_args(dtype, path, B, H, n, d, tau, lambda, cg_max_iters, cg_tol, &rpath);
    if (st != LLA_OK) return st;
    if (chunk_slices < 0) return fail(LLA_ERR_INVALID_ARG, "chunk_slices must be >= 0 (0: automatic)");
    const int S = B * H;
    const int C = lla::host_chunk_slices(S, chunk_slices);
    const lla::HostChunk hc(dtype, rpath, C, n, d);
    const size_t need = 2 * hc.half;
    if (device_buffer) {
        if (device_buffer_bytes < need)
            return fail(LLA_ERR_INVALID_ARG, "device buffer too small: %zu < %zu bytes", device_buffer_bytes, need);
        if ((reinterpret_cast<uintptr_t>(device_buffer) & 255u) != 0)
            return fail(LLA_ERR_INVALID_ARG, "device buffer must be 256-byte aligned");
    }
    if ((st = lla::host_streams()) != LLA_OK) return st;

    cudaStream_t cs = static_cast<cudaStream_t>(stream_);
    unsigned char* buf = static_cast<unsigned char*>(device_buffer);
    cudaError_t e = cudaSuccess;
    if (!buf && (e = cudaMallocAsync(reinterpret_cast<void**>(&buf), need, cs)) != cudaSuccess)
        return lla::cuda_fail(e, "cudaMallocAsync(host-forward buffer)");
    // both library streams start after the caller's stream reaches this point (a pool buffer is
    // released again on the caller's stream if that cannot be arranged)
    e = cudaEventRecord(lla::g_he[0], cs);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(lla::g_hs[i], lla::g_he[0], 0);
    if (e != cudaSuccess) {
        if (!device_buffer) cudaFreeAsync(buf, cs);
        return lla::cuda_fail(e, "host forward: stream ordering");
    }

    const size_t es = dtype == LLA_DTYPE_BF16 ? 2 : 4;
    const unsigned char* hq = static_cast<const unsigned char*>(q);
    const unsigned char* hk = static_cast<const unsigned char*>(k);
    const unsigned char* hv = static_cast<const unsigned char*>(v);
    unsigned char* ho = static_cast<unsigned char*>(out);
    int rc = LLA_OK;
    for (int c = 0, s0 = 0; s0 < S && rc == LLA_OK; ++c, s0 += C) {
        const int cnt = S - s0 < C ? S - s0 : C;
        cudaStream_t sc = lla::g_hs[c & 1];
        unsigned char* base = buf + (size_t)(c & 1) * hc.half;
        unsigned char* dq = base;
        unsigned char* dk = dq + hc.tin;
        unsigned char* dv = dk + hc.tin;
        unsigned char* dout = dv + hc.tin;
        float* drho = reinterpret_cast<float*>(dout + hc.tin);
        float* dden = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(drho) + hc.trho);
        int* dits = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(dden) + hc.tden);
        void* dws = reinterpret_cast<unsigned char*>(dits) + hc.tden;
        const size_t tbytes = (size_t)cnt * n * d * es, off = (size_t)s0 * n * d * es;
        const size_t rbytes = (size_t)cnt * n * d * 4, roff = (size_t)s0 * n * d;
        const size_t dbytes = (size_t)cnt * n * 4, doff = (size_t)s0 * n;
        if ((e = cudaMemcpyAsync(dq, hq + off, tbytes, cudaMemcpyHostToDevice, sc)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dk, hk + off, tbytes, cudaMemcpyHostToDevice, sc)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dv, hv + off, tbytes, cudaMemcpyHostToDevice, sc)) != cudaSuccess) {
            rc = lla::cuda_fail(e, "host forward: copy in");
            break;
        }
        lla::Problem p{dq, dk, dv, dout, drho, dden, cg_iters ? dits : nullptr, cnt, 1, n, d, tau, lambda,
                       cg_max_iters, cg_tol, dtype, nullptr, nullptr, nullptr};
        const char* why = nullptr;
        e = rpath == LLA_PATH_FP32 ? lla::launch_simt(p, sc) : lla::launch_tensor(p, dws, sc, &why);
        if (e != cudaSuccess) {
            rc = lla::cuda_fail(e, why ? why : "host forward: launch");
            break;
        }
        if ((e = cudaMemcpyAsync(ho + off, dout, tbytes, cudaMemcpyDeviceToHost, sc)) != cudaSuccess ||
            (e = cudaMemcpyAsync(rho + roff, drho, rbytes, cudaMemcpyDeviceToHost, sc)) != cudaSuccess ||
            (e = cudaMemcpyAsync(denom + doff, dden, dbytes, cudaMemcpyDeviceToHost, sc)) != cudaSuccess ||
            (cg_iters && (e = cudaMemcpyAsync(cg_iters + doff, dits, dbytes, cudaMemcpyDeviceToHost, sc)) != cudaSuccess)) {
            rc = lla::cuda_fail(e, "host forward: copy out");
            break;
        }
    }
    // the caller's stream continues after both library streams (also on an error, so that a
    // pool buffer is released only after the work queued on it)
    for (int i = 0; i < 2; ++i) {
        cudaError_t e1 = cudaEventRecord(lla::g_he[1 + i], lla::g_hs[i]);
        if (e1 == cudaSuccess) e1 = cudaStreamWaitEvent(cs, lla::g_he[1 + i], 0);
        if (e1 != cudaSuccess && rc == LLA_OK) rc = lla::cuda_fail(e1, "host forward: join");
    }
    if (!device_buffer) {
        cudaError_t e2 = cudaFreeAsync(buf, cs);
        if (e2 != cudaSuccess && rc == LLA_OK) rc = lla::cuda_fail(e2, "cudaFreeAsync(host-forward buffer)");
    }
    return rc;
}

int lla_selftest_device_timeout(void* stream) {
    lla::g_msg[0] = '\0';
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* word = lla::device_error_word();
    if (!word) return fail(LLA_ERR_CUDA, "lla_selftest_device_timeout: device error word not found");
    const int zero = 0;
    cudaError_t e = cudaMemcpyToSymbolAsync(lla::g_selftest_abort, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return lla::cuda_fail(e, "lla_selftest_device_timeout: abort word reset");
    lla::lla_selftest_wait_kernel<<<1, 32, 0, s>>>(word);
    e = cudaGetLastError();
    if (e != cudaSuccess) return lla::cuda_fail(e, "lla_selftest_device_timeout: launch");
    return LLA_OK;
}

int lla_profile_enable(int on) {
    lla::g_prof_on = on != 0;
    return LLA_OK;
}

int lla_profile_read(float* main_ms, float* total_ms) {
    lla::g_msg[0] = '\0';
    if (!lla::g_prof_valid) return fail(LLA_ERR_INVALID_ARG, "no profiled call yet");
    cudaError_t e = cudaEventSynchronize(lla::g_ev[3]);
    if (e != cudaSuccess) return lla::cuda_fail(e, "lla_profile_read");
    if (main_ms && (e = cudaEventElapsedTime(main_ms, lla::g_ev[1], lla::g_ev[2])) != cudaSuccess)
        return lla::cuda_fail(e, "lla_profile_read");
    if (total_ms && (e = cudaEventElapsedTime(total_ms, lla::g_ev[0], lla::g_ev[3])) != cudaSuccess)
        return lla::cuda_fail(e, "lla_profile_read");
    return LLA_OK;
}

int lla_forward(const void* q, const void* k, const void* v, void* out, float* rho, float* denom, int B, int H,
                int n, int d, float tau, float lambda, int cg_max_iters, float cg_tol, void* stream) {
    return lla_forward_ex(LLA_DTYPE_BF16, LLA_PATH_AUTO, q, k, v, out, rho, denom, nullptr, B, H, n, d, tau,
                          lambda, cg_max_iters, cg_tol, nullptr, 0, stream);
}

int lla_parallax_forward(int dtype, int path, const void* q, const void* k, const void* v, const float* probe,
                         void* out, int B, int H, int n, int d, float tau, void* workspace, size_t workspace_bytes,
                         void* stream) {
    lla::g_msg[0] = '\0';
    if (!q || !k || !v || !probe || !out) return fail(LLA_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(probe) || !aligned16(out))
        return fail(LLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    if (B < 1 || H < 1 || n < 1) return fail(LLA_ERR_INVALID_ARG, "B, H, n must be >= 1 (got %d, %d, %d)", B, H, n);
    if ((long long)B * H > 65535LL) return fail(LLA_ERR_INVALID_ARG, "B*H must be <= 65535 (one grid row per slice)");
    if ((long long)B * H * n * d > (1LL << 40)) return fail(LLA_ERR_INVALID_ARG, "problem too large");
    if (d != 16 && d != 32 && d != 64 && d != 128)
        return fail(LLA_ERR_INVALID_ARG, "head dim d must be 16, 32, 64 or 128 (got %d)", d);
    if (!(tau > 0.f) || !(tau < 1e30f)) return fail(LLA_ERR_INVALID_ARG, "tau must be finite and > 0");
    if (dtype != LLA_DTYPE_BF16 && dtype != LLA_DTYPE_FP32) return fail(LLA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (path < LLA_PATH_AUTO || path > LLA_PATH_FP32) return fail(LLA_ERR_INVALID_ARG, "unknown path %d", path);
    const int rpath = lla_resolve_path(dtype, path, d);
    if (rpath == LLA_PATH_TENSOR && (dtype != LLA_DTYPE_BF16 || (d != 64 && d != 128)))
        return fail(LLA_ERR_UNSUPPORTED, "tensor path needs bf16 inputs and d in {64, 128}");
    // no regression solve: lambda only enters the skipped CG; 1 keeps the shared code finite
    lla::Problem p{q, k, v, out, nullptr, nullptr, nullptr, B, H, n, d, tau, 1.f, 0, 0.f, dtype,
                   nullptr, nullptr, probe};
    return lla::run_problem(p, rpath, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

constexpr int kDecodeMomentAutoMaxN = 16384;

static_assert(LLA_DECODE_AUTO == lla::kDecodeAuto && LLA_DECODE_MOMENT == lla::kDecodeMoment &&
                  LLA_DECODE_STREAM == lla::kDecodeStream && LLA_DECODE_CLUSTER == lla::kDecodeCluster,
              "decode form values");

int lla_decode(int dtype, const void* q, const void* k, const void* v, void* out, float* rho, float* denom,
               int* cg_iters, int B, int H, int n, int n_cap, int d, float tau, float lambda, int cg_max_iters,
               float cg_tol, void* stream_) {
    return lla_decode_ex(LLA_DECODE_AUTO, dtype, q, k, v, out, rho, denom, cg_iters, B, H, n, n_cap, d, tau, lambda,
                         cg_max_iters, cg_tol, stream_);
}

int lla_decode_ex(int form, int dtype, const void* q, const void* k, const void* v, void* out, float* rho,
                  float* denom, int* cg_iters, int B, int H, int n, int n_cap, int d, float tau, float lambda,
                  int cg_max_iters, float cg_tol, void* stream_) {
    lla::g_msg[0] = '\0';
    if (!q || !k || !v || !out || !rho || !denom) return fail(LLA_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(rho) ||
        !aligned16(denom))
        return fail(LLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    if (B < 1 || H < 1 || n < 1) return fail(LLA_ERR_INVALID_ARG, "B, H, n must be >= 1 (got %d, %d, %d)", B, H, n);
    if (n_cap < n) return fail(LLA_ERR_INVALID_ARG, "cache capacity n_cap (%d) must be >= n (%d)", n_cap, n);
    if ((long long)B * H > (1LL << 31) - 1) return fail(LLA_ERR_INVALID_ARG, "B*H too large");
    if ((long long)B * H * n_cap * d > (1LL << 40)) return fail(LLA_ERR_INVALID_ARG, "problem too large");
    if (d != 16 && d != 32 && d != 64 && d != 128)
        return fail(LLA_ERR_INVALID_ARG, "head dim d must be 16, 32, 64 or 128 (got %d)", d);
    if (!(tau > 0.f) || !(tau < 1e30f)) return fail(LLA_ERR_INVALID_ARG, "tau must be finite and > 0");
    if (!(lambda > 0.f) || !(lambda < 1e30f)) return fail(LLA_ERR_INVALID_ARG, "lambda must be finite and > 0");
    if (cg_max_iters < 1 || cg_max_iters > 4096) return fail(LLA_ERR_INVALID_ARG, "cg_max_iters must be in [1, 4096]");
    if (!(cg_tol >= 0.f) || !(cg_tol < 1e30f)) return fail(LLA_ERR_INVALID_ARG, "cg_tol must be finite and >= 0");
    if (dtype != LLA_DTYPE_BF16 && dtype != LLA_DTYPE_FP32) return fail(LLA_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (form < LLA_DECODE_AUTO || form > LLA_DECODE_CLUSTER) return fail(LLA_ERR_INVALID_ARG, "unknown decode form %d", form);
    lla::DecodeProblem p{q, k, v, out, rho, denom, cg_iters, B, H, n, n_cap, d, tau, lambda, cg_max_iters, cg_tol,
                         dtype, nullptr, nullptr, form, nullptr};
    // AUTO: the moment form's fp32 moment sums drift with the cache length (denom measured 2e-5
    // relative at 4096 keys, 1e-4 at 16384, 2e-4 at 32768, 3.4e-4 at 53952, where the CUDA-core forms
    // stay below 1e-6), so past kDecodeMomentAutoMaxN it takes a CUDA-core form while one fits
    if (form == LLA_DECODE_AUTO)
        p.form = lla::decode_moment_supported(p) &&
                         (n <= kDecodeMomentAutoMaxN || lla::decode_smem_bytes(n, d) > (size_t)LLA_DECODE_SMEM_LIMIT)
                     ? LLA_DECODE_MOMENT
                     : LLA_DECODE_AUTO;
    if (p.form == LLA_DECODE_MOMENT) {
        if (!lla::decode_moment_supported(p))
            return fail(LLA_ERR_UNSUPPORTED, "the moment form needs bf16 caches and d = 128");
        p.dev_err = lla::device_error_word();
        if (!p.dev_err) return fail(LLA_ERR_CUDA, "lla_decode: device error word not found");
    } else {
        if (lla::decode_smem_bytes(n, d) > (size_t)LLA_DECODE_SMEM_LIMIT)
            return fail(LLA_ERR_UNSUPPORTED,
                        "the CUDA-core decode forms keep the n weights in shared memory: n = %d is above the limit %d",
                        n, lla_decode_max_n(d));
        if (p.form == LLA_DECODE_CLUSTER && !lla::decode_cluster_fits(n, d, dtype))
            return fail(LLA_ERR_UNSUPPORTED, "the cluster form holds an eighth of the cache per CTA: n = %d is too long",
                        n);
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (lla::g_prof_on) {
        for (int i = 0; i < 4; ++i)
            if (!lla::g_ev[i]) {
                cudaError_t e = cudaEventCreate(&lla::g_ev[i]);
                if (e != cudaSuccess) return lla::cuda_fail(e, "profiling event");
            }
        p.ev_main_begin = lla::g_ev[1];
        p.ev_main_end = lla::g_ev[2];
        cudaError_t e = cudaEventRecord(lla::g_ev[0], stream);
        if (e != cudaSuccess) return lla::cuda_fail(e, "profiling event record");
    }
    cudaError_t e = lla::launch_decode(p, stream);
    if (e != cudaSuccess) return lla::cuda_fail(e, "decode launch");
    if (lla::g_prof_on) {
        e = cudaEventRecord(lla::g_ev[3], stream);
        if (e != cudaSuccess) return lla::cuda_fail(e, "profiling event record");
        lla::g_prof_valid = true;
    }
    return LLA_OK;
}

size_t lla_backward_workspace_size(int dtype, int path, int B, int H, int n, int d) {
    if (B < 1 || H < 1 || n < 1 || d < 1) return 0;
    return lla::backward_workspace_bytes(lla_resolve_path(dtype, path, d), B, H, n, d);
}

int lla_backward(int dtype, int path, const void* q, const void* k, const void* v, const float* rho,
                 const float* denom, const void* dout, float* dq, float* dk, float* dv, int* cg_iters, int B, int H,
                 int n, int d, float tau, float lambda, int cg_max_iters, float cg_tol, void* workspace,
                 size_t workspace_bytes, void* stream_) {
    lla::g_msg[0] = '\0';
    if (!q || !k || !v || !rho || !denom || !dout || !dq || !dk || !dv)
        return fail(LLA_ERR_INVALID_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(rho) || !aligned16(denom) ||
        !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return fail(LLA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
    int rpath = 0;
    const int st = lla::check_backward_args(dtype, path, B, H, n, d, tau, lambda, cg_max_iters, cg_tol, &rpath);
    if (st != LLA_OK) return st;
    const size_t need = lla::backward_workspace_bytes(rpath, B, H, n, d);
    if (workspace) {
        if (workspace_bytes < need)
            return fail(LLA_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", workspace_bytes, need);
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
            return fail(LLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    lla::BackwardProblem p{q, k, v, dout, rho, denom, dq, dk, dv, cg_iters, B, H, n, d, tau, lambda,
                           cg_max_iters, cg_tol, dtype, nullptr, nullptr};
    if (lla::g_prof_on) {
        for (int i = 0; i < 4; ++i)
            if (!lla::g_ev[i]) {
                cudaError_t e = cudaEventCreate(&lla::g_ev[i]);
                if (e != cudaSuccess) return lla::cuda_fail(e, "profiling event");
            }
        p.ev_main_begin = lla::g_ev[1];
        p.ev_main_end = lla::g_ev[2];
        cudaError_t e = cudaEventRecord(lla::g_ev[0], stream);
        if (e != cudaSuccess) return lla::cuda_fail(e, "profiling event record");
    }
    void* ws = workspace;
    if (!ws) {
        cudaError_t e = cudaMallocAsync(&ws, need, stream);
        if (e != cudaSuccess) return lla::cuda_fail(e, "cudaMallocAsync(workspace)");
    }
    const char* why = nullptr;
    cudaError_t e = lla::launch_backward(p, rpath, ws, stream, &why);
    if (!workspace) {
        cudaError_t e2 = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess && e2 != cudaSuccess) return lla::cuda_fail(e2, "cudaFreeAsync(workspace)");
    }
    if (e != cudaSuccess) return lla::cuda_fail(e, why ? why : "backward launch");
    if (lla::g_prof_on) {
        e = cudaEventRecord(lla::g_ev[3], stream);
        if (e != cudaSuccess) return lla::cuda_fail(e, "profiling event record");
        lla::g_prof_valid = true;
    }
    return LLA_OK;
}

size_t lla_backward_host_buffer_size(int dtype, int path, int B, int H, int n, int d, int chunk_slices) {
    int rpath = 0;
    if (lla::check_backward_args(dtype, path, B, H, n, d, 1.f, 1.f, 1, 0.f, &rpath) != LLA_OK || chunk_slices < 0)
        return 0;
    const int C = lla::host_chunk_slices(B * H, chunk_slices);
    return 2 * lla::HostBwdChunk(dtype, rpath, C, n, d).half;
}

int lla_backward_host(int dtype, int path, const void* q, const void* k, const void* v, const float* rho,
                      const float* denom, const void* dout, float* dq, float* dk, float* dv, int* cg_iters, int B,
                      int H, int n, int d, float tau, float lambda, int cg_max_iters, float cg_tol, int chunk_slices,
                      void* device_buffer, size_t device_buffer_bytes, void* stream_) {
    lla::g_msg[0] = '\0';
    if (!q || !k || !v || !rho || !denom || !dout || !dq || !dk || !dv) return fail(LLA_ERR_INVALID_ARG, "null host pointer");
    int rpath = 0;
    int st = lla::check_backward_args(dtype, path, B, H, n, d, tau, lambda, cg_max_iters, cg_tol, &rpath);
    if (st != LLA_OK) return st;
    if (chunk_slices < 0) return fail(LLA_ERR_INVALID_ARG, "chunk_slices must be >= 0 (0: automatic)");
    const int S = B * H;
    const int C = lla::host_chunk_slices(S, chunk_slices);
    const lla::HostBwdChunk hc(dtype, rpath, C, n, d);
    const size_t need = 2 * hc.half;
    if (device_buffer) {
        if (device_buffer_bytes < need)
            return fail(LLA_ERR_INVALID_ARG, "device buffer too small: %zu < %zu bytes", device_buffer_bytes, need);
        if ((reinterpret_cast<uintptr_t>(device_buffer) & 255u) != 0)
            return fail(LLA_ERR_INVALID_ARG, "device buffer must be 256-byte aligned");
    }
    if ((st = lla::host_streams()) != LLA_OK) return st;

    cudaStream_t cs = static_cast<cudaStream_t>(stream_);
    unsigned char* buf = static_cast<unsigned char*>(device_buffer);
    cudaError_t e = cudaSuccess;
    if (!buf && (e = cudaMallocAsync(reinterpret_cast<void**>(&buf), need, cs)) != cudaSuccess)
        return lla::cuda_fail(e, "cudaMallocAsync(host-backward buffer)");
    // both library streams start after the caller's stream reaches this point (a pool buffer is
    // released again on the caller's stream if that cannot be arranged)
    e = cudaEventRecord(lla::g_he[0], cs);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(lla::g_hs[i], lla::g_he[0], 0);
    if (e != cudaSuccess) {
        if (!device_buffer) cudaFreeAsync(buf, cs);
        return lla::cuda_fail(e, "host backward: stream ordering");
    }

    const size_t es = dtype == LLA_DTYPE_BF16 ? 2 : 4;
    const unsigned char* hin[4] = {static_cast<const unsigned char*>(q), static_cast<const unsigned char*>(k),
                                   static_cast<const unsigned char*>(v), static_cast<const unsigned char*>(dout)};
    float* hout[3] = {dq, dk, dv};
    int rc = LLA_OK;
    for (int c = 0, s0 = 0; s0 < S && rc == LLA_OK; ++c, s0 += C) {
        const int cnt = S - s0 < C ? S - s0 : C;
        cudaStream_t sc = lla::g_hs[c & 1];
        unsigned char* base = buf + (size_t)(c & 1) * hc.half;
        unsigned char* din[4] = {base, base + hc.tin, base + 2 * hc.tin, base + 3 * hc.tin};
        float* drho = reinterpret_cast<float*>(base + 4 * hc.tin);
        float* dg[3] = {reinterpret_cast<float*>(base + 4 * hc.tin + hc.tf),
                        reinterpret_cast<float*>(base + 4 * hc.tin + 2 * hc.tf),
                        reinterpret_cast<float*>(base + 4 * hc.tin + 3 * hc.tf)};
        float* dden = reinterpret_cast<float*>(base + 4 * hc.tin + 4 * hc.tf);
        int* dits = reinterpret_cast<int*>(base + 4 * hc.tin + 4 * hc.tf + hc.tden);
        void* dws = base + 4 * hc.tin + 4 * hc.tf + 2 * hc.tden;
        const size_t tbytes = (size_t)cnt * n * d * es, off = (size_t)s0 * n * d * es;
        const size_t fbytes = (size_t)cnt * n * d * 4, foff = (size_t)s0 * n * d;
        const size_t dbytes = (size_t)cnt * n * 4, doff = (size_t)s0 * n;
        for (int t = 0; t < 4 && rc == LLA_OK; ++t)
            if ((e = cudaMemcpyAsync(din[t], hin[t] + off, tbytes, cudaMemcpyHostToDevice, sc)) != cudaSuccess)
                rc = lla::cuda_fail(e, "host backward: copy in");
        if (rc == LLA_OK && ((e = cudaMemcpyAsync(drho, rho + foff, fbytes, cudaMemcpyHostToDevice, sc)) != cudaSuccess ||
                             (e = cudaMemcpyAsync(dden, denom + doff, dbytes, cudaMemcpyHostToDevice, sc)) != cudaSuccess))
            rc = lla::cuda_fail(e, "host backward: copy in");
        if (rc != LLA_OK) break;
        lla::BackwardProblem p{din[0], din[1], din[2], din[3], drho, dden, dg[0], dg[1], dg[2],
                               cg_iters ? dits : nullptr, cnt, 1, n, d, tau, lambda, cg_max_iters, cg_tol, dtype,
                               nullptr, nullptr};
        const char* why = nullptr;
        if ((e = lla::launch_backward(p, rpath, dws, sc, &why)) != cudaSuccess) {
            rc = lla::cuda_fail(e, why ? why : "host backward: launch");
            break;
        }
        for (int t = 0; t < 3 && rc == LLA_OK; ++t)
            if ((e = cudaMemcpyAsync(hout[t] + foff, dg[t], fbytes, cudaMemcpyDeviceToHost, sc)) != cudaSuccess)
                rc = lla::cuda_fail(e, "host backward: copy out");
        if (rc == LLA_OK && cg_iters &&
            (e = cudaMemcpyAsync(cg_iters + doff, dits, dbytes, cudaMemcpyDeviceToHost, sc)) != cudaSuccess)
            rc = lla::cuda_fail(e, "host backward: copy out");
    }
    for (int i = 0; i < 2; ++i) {
        cudaError_t e1 = cudaEventRecord(lla::g_he[1 + i], lla::g_hs[i]);
        if (e1 == cudaSuccess) e1 = cudaStreamWaitEvent(cs, lla::g_he[1 + i], 0);
        if (e1 != cudaSuccess && rc == LLA_OK) rc = lla::cuda_fail(e1, "host backward: join");
    }
    if (!device_buffer) {
        cudaError_t e2 = cudaFreeAsync(buf, cs);
        if (e2 != cudaSuccess && rc == LLA_OK) rc = lla::cuda_fail(e2, "cudaFreeAsync(host-backward buffer)");
    }
    return rc;
}

int lla_decode_max_n(int d) {
    if (d != 16 && d != 32 && d != 64 && d != 128) return 0;
    const size_t base = lla::decode_smem_bytes(0, d);
    return (int)(((size_t)LLA_DECODE_SMEM_LIMIT - base) / sizeof(float));
}

int lla_sync_status(void* stream) {
    lla::g_msg[0] = '\0';
    unsigned word = 0;
    cudaError_t e = lla::read_and_clear_device_error(&word, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return lla::cuda_fail(e, "lla_sync_status");
    if (word & lla::kDevErrSmemAlign)
        return fail(LLA_ERR_CUDA, "tensor kernel: dynamic shared memory not 1024-byte aligned, no work done (error word 0x%x)",
                    word);
    if (word & lla::kDevErrMbarTimeout)
        return fail(LLA_ERR_DEVICE_TIMEOUT, "a bounded device-side wait gave up (error word 0x%x)", word);
    return LLA_OK;
}

}  // extern "C"
