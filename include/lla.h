/*
 * lla.h -- C ABI of the causal Local Linear Attention (LLA) forward pass on GB300 (sm_103a).
 *
 * What is computed (Local Linear Attention reading notes, section 2.1, Eqs. (6)-(8); section
 * 2.2, Eqs. (10)-(12) and the FlashLLA three-phase query-tile sweep of Algorithm 1):
 * for every batch b, head h and query position i, over the causal prefix j <= i,
 *
 *     w_ij    = exp(tau q_i.k_j - m_i),  m_i = max_{l<=i} tau q_i.k_l     (largest weight is 1)
 *     omega_i = sum_j w_ij,   mu_i = sum_j w_ij (k_j - q_i),
 *     Sigma_i = sum_j w_ij (k_j - q_i)(k_j - q_i)^T + lambda I,   Sigma_i rho_i = mu_i,
 *     denom_i = omega_i - mu_i.rho_i,
 *     out_i   = sum_j w_ij (1 - (k_j - q_i).rho_i) v_j / denom_i.
 *
 * rho_i is found by conjugate gradient (section 2.2, "matrix-free CG").  The CG runs on the
 * centred key scatter: with kbar_i = sum_j w_ij k_j / omega_i and delta_i = kbar_i - q_i,
 * Sigma_i = C_i + omega_i delta_i delta_i^T exactly, so CG solves
 * (C_i / omega_i) rho'_i = delta_i and rho_i = rho'_i / (1 + delta_i.rho'_i),
 * denom_i = omega_i / (1 + delta_i.rho'_i) (Sherman-Morrison).  At convergence this is the same
 * rho_i; at a fixed iteration cap the centred system, having no dominant mean direction,
 * converges further and is stable in low precision.
 *
 * Layout: q, k, v, out are contiguous row-major [B, H, n, d]; rho is [B, H, n, d] fp32;
 * denom and cg_iters are [B, H, n].  All pointers are DEVICE pointers on the current device,
 * 16-byte aligned.  The caller owns every buffer.  All calls are asynchronous on `stream`
 * (a cudaStream_t passed as void*; NULL = legacy default stream).
 *
 * Errors: every entry point returns an lla_status.  Invalid arguments are rejected on the host
 * before anything is launched; no exception crosses this boundary.  lla_last_error() gives a
 * message for the calling thread's last failure.
 */
#ifndef LLA_H_
#define LLA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LLA_OK = 0,
    LLA_ERR_INVALID_ARG = 1,     /* null pointer, bad size, tau/lambda <= 0, cap < 1, ... */
    LLA_ERR_UNSUPPORTED = 2,     /* head dim or dtype/path combination not built */
    LLA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed; see lla_last_error() */
    LLA_ERR_DEVICE_TIMEOUT = 4   /* a bounded device-side wait gave up (reported by lla_sync_status) */
} lla_status;

typedef enum {
    LLA_DTYPE_BF16 = 0,          /* q, k, v, out are bfloat16 */
    LLA_DTYPE_FP32 = 1           /* q, k, v, out are float32 */
} lla_dtype;

typedef enum {
    LLA_PATH_AUTO = 0,           /* bf16 -> LLA_PATH_TENSOR when d in {64,128}, else LLA_PATH_FP32 */
    LLA_PATH_TENSOR = 1,         /* tcgen05/TMEM/TMA kernel, fp16 operands, fp32 accumulate/state */
    LLA_PATH_FP32 = 2            /* CUDA-core fp32 kernel: every product and the CG state in fp32 */
} lla_path;

/*
 * lla_forward -- causal LLA forward, bf16 q/k/v/out, LLA_PATH_AUTO.
 *
 * q, k, v   [B,H,n,d] bf16, read only.      out   [B,H,n,d] bf16, written.
 * rho       [B,H,n,d] fp32, written: rho_i.  denom [B,H,n] fp32, written: omega_i - mu_i.rho_i.
 * B, H, n >= 1 with B*H <= 65535 (one grid row per (b, h) slice); d in {16, 32, 64, 128};
 * tau > 0 (logit scale); lambda > 0 (ridge, absolute,
 * applied to the max-normalised weights); cg_max_iters >= 1; cg_tol >= 0: a query stops once
 * ||r|| <= cg_tol ||delta_i|| (cg_tol == 0: exactly cg_max_iters iterations).  CG runs on the
 * centred system (C_i/omega_i) rho'_i = delta_i, delta_i = kbar_i - q_i, which Sherman-Morrison maps
 * exactly to Eq. (7)'s Sigma_i rho_i = mu_i; the tolerance is relative to ||delta_i||, and iteration
 * counts are those of the centred iteration.
 * With cg_tol > 0 the tensor path runs its precise form: the moment weights, the CG coefficients
 * and the CG direction are carried as fp16 hi + lo pairs (about 22 bits; two more MMAs per CG block),
 * which solving to a relative residual needs where lambda/omega_i is small against the keys' scatter.
 * With cg_tol == 0 (a fixed iteration count) it runs the fp16 form.
 * Scratch (the tensor path's fp16 operand copies) is taken from the CUDA stream-ordered pool
 * with cudaMallocAsync/cudaFreeAsync on `stream`; use lla_forward_ex to pass it instead.
 */
int lla_forward(const void* q, const void* k, const void* v, void* out, float* rho, float* denom,
                int B, int H, int n, int d, float tau, float lambda, int cg_max_iters, float cg_tol,
                void* stream);

/*
 * lla_forward_ex -- as lla_forward with the dtype and path chosen by the caller.
 *
 * dtype      LLA_DTYPE_BF16 or LLA_DTYPE_FP32 (q, k, v and out share it).
 * path       an lla_path value.  LLA_PATH_TENSOR needs bf16 and d in {64, 128}.
 * cg_iters   NULL, or [B,H,n] int32 device buffer: CG iterations each query executed.
 * workspace  NULL (scratch from the stream-ordered pool) or a device buffer of at least
 *            lla_workspace_size(...) bytes, 256-byte aligned, not used concurrently by
 *            another call.
 */
int lla_forward_ex(int dtype, int path, const void* q, const void* k, const void* v, void* out,
                   float* rho, float* denom, int* cg_iters, int B, int H, int n, int d, float tau,
                   float lambda, int cg_max_iters, float cg_tol, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Bytes of scratch lla_forward_ex needs for these arguments (0 for the fp32 path). */
size_t lla_workspace_size(int dtype, int path, int B, int H, int n, int d);

/* The path LLA_PATH_AUTO resolves to for (dtype, d): LLA_PATH_TENSOR or LLA_PATH_FP32. */
int lla_resolve_path(int dtype, int path, int d);

/*
 * lla_forward_host -- lla_forward_ex with q, k, v read from HOST memory and out, rho, denom
 * (and cg_iters) written to HOST memory, the transfers overlapped with the computation.
 *
 * The B*H (b, h) slices are processed in chunks of chunk_slices consecutive slices (0: about
 * eight chunks).  Chunk c runs on one of two library-owned CUDA streams with its own half of
 * the device buffer: its inputs are copied in while chunk c-1 computes, and chunk c-1's results
 * are copied out while chunk c computes.  Both library streams start after the work already on
 * `stream`, and `stream` continues after both; the call returns once everything is queued, so
 * the host buffers must stay valid, and out/rho/denom must not be read, until `stream` has
 * reached that point (cudaStreamSynchronize or lla_sync_status).
 *
 * Each chunk's result is the result of lla_forward_ex on that chunk's slices (B = its slice
 * count, H = 1): the tensor path chooses its fp16 operand scales per chunk, so its last bits
 * can differ from one lla_forward_ex call on all slices; the fp32 path's results are identical.
 *
 * q, k, v      [B,H,n,d] host buffers of dtype; out the same; rho [B,H,n,d] and denom [B,H,n]
 *              fp32; cg_iters NULL or [B,H,n] int32.  Pinned memory (cudaHostAlloc, or torch's
 *              pin_memory) lets the copies run asynchronously; pageable memory works, slower.
 * device_buffer NULL (taken from the stream-ordered pool for the call) or a device buffer of
 *              lla_forward_host_buffer_size(...) bytes, 256-byte aligned, used by no other call
 *              until `stream` has passed this one.
 * Other arguments and errors as for lla_forward_ex; chunk_slices < 0 or a device buffer too
 * small or misaligned gives LLA_ERR_INVALID_ARG before anything is queued.  The two library
 * streams are shared by all calls: do not call this from several host threads at once.
 */
int lla_forward_host(int dtype, int path, const void* q, const void* k, const void* v, void* out,
                     float* rho, float* denom, int* cg_iters, int B, int H, int n, int d, float tau,
                     float lambda, int cg_max_iters, float cg_tol, int chunk_slices,
                     void* device_buffer, size_t device_buffer_bytes, void* stream);

/* Bytes of device buffer lla_forward_host needs for these arguments (0 for invalid ones). */
size_t lla_forward_host_buffer_size(int dtype, int path, int B, int H, int n, int d, int chunk_slices);

/*
 * lla_sync_status -- synchronise `stream`, then report and clear the library's device error
 * word: set when a bounded wait inside a kernel gave up (LLA_ERR_DEVICE_TIMEOUT), or when the
 * tensor kernel found its dynamic shared memory not 1024-byte aligned and did no work
 * (LLA_ERR_CUDA).
 */
int lla_sync_status(void* stream);

/*
 * lla_selftest_device_timeout -- self-test of the timeout reporting above.  Launches on `stream`
 * one small kernel whose single waiting thread calls the same bounded mbarrier wait the tensor
 * kernels use, on a barrier that nothing arrives on.  After the wait's limit (about two seconds)
 * the kernel records the timeout in the device error word and returns normally, so the next
 * lla_sync_status(stream) returns LLA_ERR_DEVICE_TIMEOUT and clears the word; the CUDA context
 * stays usable.  Returns LLA_OK once the kernel is launched (LLA_ERR_CUDA if the launch fails).
 * For tests of a caller's error handling; it does no other work.
 */
int lla_selftest_device_timeout(void* stream);

/*
 * lla_profile_enable -- on != 0: every later call records CUDA events on its stream around its
 * dominant kernel (the fused sweep kernel) and around the whole call; on == 0 stops.
 * lla_profile_read -- elapsed milliseconds of the most recent profiled call: main_ms for the
 * dominant kernel, total_ms for the whole call (either pointer may be NULL).  Waits for that
 * call's events.  Returns LLA_ERR_INVALID_ARG if no call was profiled yet.  Measurement support
 * for benchmarks; not thread-safe across concurrent profiled calls.
 */
int lla_profile_enable(int on);
int lla_profile_read(float* main_ms, float* total_ms);

/*
 * lla_forward_noalloc -- lla_forward (bf16, tensor path, d in {64, 128}) for callers that cannot
 * allocate device memory when they run it.  The paper has no counterpart: this is an interface
 * for hosts whose device memory is owned by another allocator (for example a framework that
 * reserves the GPU's memory up front) or that must not pay for an allocation on this path.
 *
 * Scratch lives in a fixed device array of LLA_NOALLOC_SCRATCH_BYTES that every GPU loading the
 * library holds until the process exits; the call makes no cudaMalloc/cudaFree or other
 * allocating call.  Arguments and outputs are as for lla_forward; q, k, v, out, rho, denom are
 * still the caller's buffers.  A problem whose lla_workspace_size(LLA_DTYPE_BF16,
 * LLA_PATH_TENSOR, ...) exceeds the array is rejected with LLA_ERR_INVALID_ARG before anything is
 * launched; d outside {64, 128} gives LLA_ERR_UNSUPPORTED.
 *
 * Every call looks up the array's device address in the current context (cudaGetSymbolAddress
 * with the caller's device current; no allocation), so the address stays right after a
 * cudaDeviceReset.  The first lookup on a device may load the library's device code: make the
 * first call on each device before any stream capture.  All calls share the array: calls that
 * overlap on the GPU (on different streams, or from different threads) race on it and must be
 * serialised by the caller.  Each call re-initialises what must start at zero.
 */
#define LLA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int lla_forward_noalloc(const void* q, const void* k, const void* v, void* out, float* rho, float* denom,
                        int B, int H, int n, int d, float tau, float lambda, int cg_max_iters, float cg_tol,
                        void* stream);

/*
 * lla_parallax_forward -- Parallax-form causal attention with a caller-supplied probe
 * (Parallax: Parameterized Local Linear Attention, the "softmax output minus a covariance
 * correction" rewrite of LLA; the page learns the probe as rho = RMSNorm(W_R x), here the
 * caller supplies it, and the page's boundary factor eta is dropped as the page does):
 *
 *     wbar_ij     = exp(tau q_i.k_j - m_i) / omega_i     (the causal softmax weights, j <= i)
 *     Sigma_KV,i  = sum_j wbar_ij (v_j - vbar_i)(k_j - kbar_i)^T
 *     out_i       = sum_j wbar_ij v_j - Sigma_KV,i probe_i
 *                 = sum_j wbar_ij (1 - (k_j - kbar_i).probe_i) v_j.
 *
 * With probe = 0 this is causal softmax attention.  With probe_i = omega_i rho_i / denom_i
 * (the LLA solution and denominator of lla_forward) it equals the LLA output.
 *
 * dtype, path, q, k, v, out, B, H, n, d, tau, workspace, workspace_bytes, stream: as for
 * lla_forward_ex (lla_workspace_size gives the same scratch size).  probe: [B,H,n,d] fp32
 * device buffer, read only, 16-byte aligned.  No regression is solved, so there is no lambda,
 * no iteration count and no rho/denom output.  Errors as for lla_forward_ex.
 */
int lla_parallax_forward(int dtype, int path, const void* q, const void* k, const void* v, const float* probe,
                         void* out, int B, int H, int n, int d, float tau, void* workspace, size_t workspace_bytes,
                         void* stream);

typedef enum {
    LLA_DECODE_AUTO = 0,         /* LLA_DECODE_MOMENT for bf16 caches at d = 128 with n <= 16384 or n past
                                    lla_decode_max_n(128), else a CUDA-core form */
    LLA_DECODE_MOMENT = 1,       /* tcgen05: the weighted moments of the cache in one pass, CG on them */
    LLA_DECODE_STREAM = 2,       /* CUDA cores, a CTA per head, K re-read every CG iteration */
    LLA_DECODE_CLUSTER = 3       /* CUDA cores, an 8-CTA cluster per head holding K in shared memory */
} lla_decode_form;

/*
 * lla_decode -- one decode step: a new query per (b, h) against its key/value cache (Local
 * Linear Attention reading notes, section 2.2: the FlashLLA cache is Theta(n d); the new
 * query's causal prefix is the whole cache).  The result equals row n-1 of lla_forward on the
 * sequence whose keys and values are the cache, computed by the same centred CG with fp32
 * accumulation and CG state (one query row per head: the step is bound by reading the cache).
 *
 * q       [B,H,d] in dtype, the new position's query.
 * k, v    [B,H,n_cap,d] in dtype: rows 0..n-1 are the cache (the new key/value at n-1); rows
 *         n..n_cap-1 are not read.  n_cap >= n is the row stride, so a preallocated cache can
 *         be passed as it grows.
 * out     [B,H,d] in dtype.  rho [B,H,d] fp32.  denom [B,H] fp32.  cg_iters NULL or [B,H] int32.
 * tau, lambda, cg_max_iters, cg_tol: as for lla_forward.
 * All pointers are device pointers, 16-byte aligned, owned by the caller.  No scratch.  Errors
 * as for lla_forward_ex.  The form is LLA_DECODE_AUTO (see lla_decode_ex): for bf16 caches at
 * d = 128 the moment form up to n = 16384 and past lla_decode_max_n(128); otherwise a CUDA-core
 * form, which keeps the n weights of a head in shared memory, so n above lla_decode_max_n(d) gives
 * LLA_ERR_UNSUPPORTED for fp32 caches or d < 128.
 */
int lla_decode(int dtype, const void* q, const void* k, const void* v, void* out, float* rho, float* denom,
               int* cg_iters, int B, int H, int n, int n_cap, int d, float tau, float lambda, int cg_max_iters,
               float cg_tol, void* stream);

/*
 * lla_decode_ex -- lla_decode with the form chosen by the caller (an lla_decode_form value).
 * Every form computes the same step, the centred CG of the reading notes' section 2.2 on the
 * new query's system, and differs only in how the operator C is applied:
 *   LLA_DECODE_MOMENT   (bf16 caches, d = 128 only) reads K twice and V once: a first pass gives
 *       the logits' maximum, omega and kbar; the second forms, on the tensor cores,
 *       Cc = sum_j w_j (k_j - kbar) k_j^T and Hc = sum_j w_j (k_j - kbar) v_j^T (d x d, fp32
 *       accumulation, the weighted centred keys carried as three bf16 terms), with
 *       r = sum_j w_j (k_j - kbar) and nu = sum_j w_j v_j; then runs the CG on the d x d moments:
 *       C p = Cc p - r (kbar.p), and the output sum_j u_j v_j = nu - Hc^T rho',
 *       sum_j u_j = omega - r.rho'.  No limit on n; its moment sums drift with n (denom measured
 *       1e-4 relative at 16384 keys, 3.4e-4 at 53952, where the CUDA-core forms stay below 1e-6),
 *       hence AUTO's rule.
 *   LLA_DECODE_STREAM   applies C with a pass over the cache per CG iteration (K read T+2 times).
 *   LLA_DECODE_CLUSTER  as STREAM, with an eighth of K held in each CTA of an 8-CTA cluster; n must
 *       leave an eighth of the cache within a CTA's shared memory, else LLA_ERR_UNSUPPORTED.
 * An unsupported dtype or d for the chosen form gives LLA_ERR_UNSUPPORTED.
 */
int lla_decode_ex(int form, int dtype, const void* q, const void* k, const void* v, void* out, float* rho,
                  float* denom, int* cg_iters, int B, int H, int n, int n_cap, int d, float tau, float lambda,
                  int cg_max_iters, float cg_tol, void* stream);

/* Largest cache length n that the CUDA-core decode forms accept for head dim d (0 when d is
 * unsupported).  The moment form (bf16, d = 128) has no such limit. */
int lla_decode_max_n(int d);

/*
 * lla_backward -- gradients of the causal LLA forward: with L = sum_{b,h,i} dout_i.out_i,
 * dq = dL/dq, dk = dL/dk, dv = dL/dv.  The Local Linear Attention reading notes name the
 * backward pass (appendix D: it needs further linear systems) without giving it; it is the
 * derivative of Eqs. (6)-(8) (section 2.1) through the exact solve, written in centred form.
 * Per query i (g_i = dout_i, wbar_ij = w_ij/omega_i, c_ij = k_j - kbar_i, h_ij = g_i.v_j,
 * hbar_i = sum_j wbar_ij h_ij), one adjoint system on the forward's centred operator:
 *
 *     (C_i / omega_i) y_i = sum_j wbar_ij h_ij c_ij,     rho'_i = rho_i omega_i / denom_i,
 *
 * and per pair  Ahat = 1 - c.rho'_i,  Bhat = (h - hbar_i) - c.y_i,  ds = wbar Ahat Bhat:
 *     dv_j += wbar Ahat g_i,   dk_j += tau ds q_i - wbar (Ahat y_i + Bhat rho'_i),
 *     dq_i  = tau sum_j ds k_j + y_i,
 * plus the path through the row maximum m_i (to the first key index attaining it), whose
 * weight is sum_j ds = -(lambda/omega_i) rho'_i.y_i.
 *
 * Three stages: stats (row maximum and its index, omega, kbar, hbar, the adjoint right-hand side
 * and the adjoint CG), dq (a query-major sweep) and dk/dv (a key-major sweep).  On
 * LLA_PATH_TENSOR the stats stage is the forward's tcgen05 kernel in its backward mode (fp16
 * operands, fp32 accumulation and CG state); the dq and dk/dv stages, and every stage of
 * LLA_PATH_FP32, are fp32 on CUDA cores.
 *
 * dtype      LLA_DTYPE_BF16 or LLA_DTYPE_FP32: q, k, v, dout share it.
 * path       an lla_path value, resolved as for lla_forward_ex (LLA_PATH_TENSOR needs bf16 and
 *            d in {64, 128}).
 * q, k, v    [B,H,n,d], the forward call's inputs.
 * rho        [B,H,n,d] fp32, denom [B,H,n] fp32: the forward call's outputs for these inputs
 *            (any path); the backward is exact to the extent they are.
 * dout       [B,H,n,d] in dtype: dL/dout.
 * dq, dk, dv [B,H,n,d] fp32, written (not accumulated into).
 * cg_iters   NULL, or [B,H,n] int32: adjoint CG iterations each query executed.
 * tau, lambda as for the forward call; cg_max_iters, cg_tol: the adjoint CG's cap and relative
 *            tolerance (||r|| <= cg_tol ||sum_j wbar_ij h_ij c_ij||), as for lla_forward.
 * workspace  NULL (scratch from the stream-ordered pool) or a device buffer of at least
 *            lla_backward_workspace_size(dtype, path, B, H, n, d) bytes, 256-byte aligned, not used
 *            concurrently by another call.
 * B*H <= 65535.  All pointers are device pointers, 16-byte aligned, owned by the caller.
 * Errors as for lla_forward_ex.
 */
int lla_backward(int dtype, int path, const void* q, const void* k, const void* v, const float* rho,
                 const float* denom, const void* dout, float* dq, float* dk, float* dv, int* cg_iters, int B, int H,
                 int n, int d, float tau, float lambda, int cg_max_iters, float cg_tol, void* workspace,
                 size_t workspace_bytes, void* stream);

/* Bytes of scratch lla_backward needs for these arguments (per-query records, the adjoint
 * vectors y and, on the tensor path, the fp16 operand copies and CG scratch). */
size_t lla_backward_workspace_size(int dtype, int path, int B, int H, int n, int d);

/*
 * lla_backward_host -- lla_backward with q, k, v, dout, rho, denom read from HOST memory and dq,
 * dk, dv (and cg_iters) written to HOST memory, the transfers overlapped with the computation,
 * exactly as lla_forward_host does for the forward: chunks of chunk_slices (b, h) slices (0:
 * ceil(B*H/8)) on the two library streams, each chunk's result that of lla_backward on its slices
 * (B = its slice count, H = 1; the tensor path chooses its operand scales per chunk), `stream`
 * ordered before and after, host buffers valid until `stream` has passed the call, pinned memory
 * for asynchronous copies.  device_buffer: NULL (stream-ordered pool) or
 * lla_backward_host_buffer_size(...) bytes, 256-byte aligned.  Errors as for lla_backward, plus
 * LLA_ERR_INVALID_ARG for chunk_slices < 0 or a device buffer too small or misaligned.  Not for
 * concurrent use from several host threads (the library streams are shared).
 */
int lla_backward_host(int dtype, int path, const void* q, const void* k, const void* v, const float* rho,
                      const float* denom, const void* dout, float* dq, float* dk, float* dv, int* cg_iters,
                      int B, int H, int n, int d, float tau, float lambda, int cg_max_iters, float cg_tol,
                      int chunk_slices, void* device_buffer, size_t device_buffer_bytes, void* stream);

/* Bytes of device buffer lla_backward_host needs for these arguments (0 for invalid ones). */
size_t lla_backward_host_buffer_size(int dtype, int path, int B, int H, int n, int d, int chunk_slices);

/* Message for the calling thread's most recent failure ("" if none). Owned by the library. */
const char* lla_last_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
int lla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LLA_H_ */
