// Internal declarations shared by the translation units of liblla.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace lla {

// Problem description handed from the C ABI to a path's launcher (already validated).
struct Problem {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    float* rho;
    float* denom;
    int* cg_iters;       // may be null
    int B, H, n, d;
    float tau, lambda;
    int cg_max_iters;
    float cg_tol;
    int dtype;           // lla_dtype
    cudaEvent_t ev_main_begin;   // recorded just before / after the dominant kernel when profiling
    cudaEvent_t ev_main_end;     // (null otherwise)
    // Parallax form: the caller's probe [B,H,n,d] fp32.  Non-null: no CG (cg_max_iters is 0),
    // the output sweep takes this probe as rho', and rho / denom / cg_iters are not written.
    const float* probe;
};

// Device error word: bit flags set by kernels that gave up (a bounded wait ran out, or the
// tensor kernel found its dynamic shared memory misaligned and did no work).
enum DeviceError : unsigned { kDevErrMbarTimeout = 1u, kDevErrSmemAlign = 2u };

// Decode step: one new query per (b, h) against a key/value cache of n rows (row stride n_cap).
struct DecodeProblem {
    const void* q;       // [B,H,d]
    const void* k;       // [B,H,n_cap,d], rows 0..n-1 valid
    const void* v;
    void* out;           // [B,H,d]
    float* rho;          // [B,H,d]
    float* denom;        // [B,H]
    int* cg_iters;       // [B,H] or null
    int B, H, n, n_cap, d;
    float tau, lambda;
    int cg_max_iters;
    float cg_tol;
    int dtype;           // lla_dtype
    cudaEvent_t ev_main_begin, ev_main_end;
    int form;            // DecodeForm, resolved (never kDecodeAuto)
    unsigned* dev_err;   // the device error word (the moment form's bounded waits)
};
// Decode forms (the values of lla_decode_form in include/lla.h).
enum DecodeForm : int { kDecodeAuto = 0, kDecodeMoment = 1, kDecodeStream = 2, kDecodeCluster = 3 };
size_t decode_smem_bytes(int n, int d);
bool decode_cluster_fits(int n, int d, int dtype);
bool decode_moment_supported(const DecodeProblem& p);
cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t stream);
cudaError_t launch_decode_moment(const DecodeProblem& p, cudaStream_t stream);

// Backward pass: gradients of sum_i dout_i.out_i with respect to q, k, v (all fp32 outputs).
struct BackwardProblem {
    const void* q;       // [B,H,n,d] in dtype
    const void* k;
    const void* v;
    const void* dout;
    const float* rho;    // [B,H,n,d] fp32, the forward's rho
    const float* denom;  // [B,H,n] fp32, the forward's denom
    float* dq;           // [B,H,n,d] fp32
    float* dk;
    float* dv;
    int* cg_iters;       // [B,H,n] adjoint CG iterations, or null
    int B, H, n, d;
    float tau, lambda;
    int cg_max_iters;
    float cg_tol;
    int dtype;           // lla_dtype
    cudaEvent_t ev_main_begin, ev_main_end;   // around the query-major kernel when profiling
};
// Per-query record of the backward pass, written by the stats stage (fp32 or tensor path) and
// read by the dq and key-major stages.
struct __align__(16) BwdRowRec {
    float m;         // row maximum of tau q_i.k_j (natural units: w_ij = exp(tau q_i.k_j - m))
    int jm;          // first key index attaining it
    float inv_omega; // 1 / omega
    float hbar;      // sum_j wbar_j dout_i.v_j
    float kb_rp;     // kbar.rho'
    float kb_y;      // kbar.y
    float sd;        // -(lambda/omega) rho'.y
    float rp_scale;  // omega / denom: rho' = rp_scale rho
};
size_t backward_records_bytes(int B, int H, int n, int d);   // records + y, 256-byte aligned parts
size_t backward_workspace_bytes(int path, int B, int H, int n, int d);
// Whole backward on the given path (LLA_PATH_FP32 or LLA_PATH_TENSOR).
cudaError_t launch_backward(const BackwardProblem& p, int path, void* workspace, cudaStream_t stream,
                            const char** why);
// The fp16 operand copies the tensor stats stage leaves in its workspace, and their scales
// (float bits of max |q|, |k|, |v|, |dout|; each copy is x 2^(14 - ceil log2 max)).
struct TensorOperands {
    const unsigned* maxabs;
    const void* q16;
    const void* k16;
    const void* v16;
    const void* g16;
};
TensorOperands tensor_backward_operands(void* ws, int B, int H, int n, int d);
// The dq and dk/dv stages on tcgen05 (lla_bwd_tc.cu): scratch bytes and launches.  kmax (per key,
// the largest dk and dv coefficient in scaled units, float bits) is written by the dq kernel.
size_t tensor_kv_bytes(int B, int H, int n, int d);
struct KvScratch {
    unsigned* hdr;        // float bits of max |rho'|, max |y|; an abort word
    void *rh, *rl, *yh, *yl;
    unsigned* kmax;       // [B*H*n][2]
};
KvScratch tensor_kv_scratch(void* ws, int B, int H, int n, int d);
cudaError_t launch_tensor_kv_prep(const BackwardProblem& p, const BwdRowRec* rec, const float* yvec,
                                  const KvScratch& kv, cudaStream_t stream);
cudaError_t launch_tensor_kv(const BackwardProblem& p, const BwdRowRec* rec, const TensorOperands& ops,
                             const KvScratch& kv, cudaStream_t stream, const char** why);
// The dq stage on tcgen05 (also records kmax for the dk/dv stage).
cudaError_t launch_tensor_dq(const BackwardProblem& p, const BwdRowRec* rec, const float* yvec,
                             const TensorOperands& ops, const KvScratch& kv, cudaStream_t stream, const char** why);

// The stats stage (max, moments, adjoint CG) on the tensor path; writes rec and yvec.
size_t tensor_backward_stats_bytes(int B, int H, int n, int d);
cudaError_t launch_tensor_backward_stats(const BackwardProblem& p, void* ws, BwdRowRec* rec, float* yvec,
                                         cudaStream_t stream, const char** why);

// fp32 CUDA-core path (any d in {16,32,64,128}, fp32 or bf16 inputs).
cudaError_t launch_simt(const Problem& p, cudaStream_t stream);

// Tensor-core path (bf16 inputs, d in {64,128}).
size_t tensor_workspace_bytes(int B, int H, int n, int d);
cudaError_t launch_tensor(const Problem& p, void* workspace, cudaStream_t stream, const char** why);

#ifdef __CUDACC__
// Dispatch order of the causal kernels.  A tile's cost grows with the length of its causal range,
// so a grid of (tile, head) CTAs is dispatched heaviest first: the CTAs that start last are the
// lightest, and the tail in which SMs idle is short.  The order runs over groups of heads whose
// operands (head_bytes each) fit in 32 MB together, so the CTAs running at once read L2-resident
// keys and values.  Block (x, y) of a grid (tiles, heads) maps to rank (0 = the heaviest tile of its
// head) and head; the map is a bijection of the grid.
__device__ __forceinline__ void causal_order(size_t head_bytes, int& rank, int& head) {
    const int nt = (int)gridDim.x, nh = (int)gridDim.y;
    const int lin = (int)blockIdx.x + (int)blockIdx.y * nt;
    const size_t fit = (size_t(32) << 20) / (head_bytes > 0 ? head_bytes : 1);
    const int group = (int)(fit < 1 ? 1 : fit > (size_t)nh ? (size_t)nh : fit);
    const int g0 = lin / (group * nt) * group;            // first head of this CTA's group
    const int gh = min(group, nh - g0);                   // heads in the group
    const int w = lin - g0 * nt;                          // position in the group, < gh * nt
    rank = w / gh;
    head = g0 + w % gh;
}
#endif

// Record a failure for lla_last_error() and return status (defined in lla_api.cu).
int set_error(int status, const char* message);

// Library-owned device error word (defined in lla_api.cu).
cudaError_t read_and_clear_device_error(unsigned* out, cudaStream_t stream);
unsigned* device_error_word();

}  // namespace lla
