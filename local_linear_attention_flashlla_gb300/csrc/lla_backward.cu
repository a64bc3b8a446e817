// fp32 CUDA-core backward pass of the causal LLA forward.
//
// Gradients of L = sum_i g_i.out_i (g = dL/dout) with respect to q, k and v, obtained by
// differentiating Eqs. (6)-(8) of the Local Linear Attention reading notes (section 2.1)
// through the exact solve; the notes name the backward pass (appendix D: it needs further
// linear systems) but print no formulas.  Centred form, per query i: w_j = exp(tau q_i.k_j - m_i),
// omega = sum_j w_j, wbar_j = w_j/omega, kbar = sum_j wbar_j k_j, c_j = k_j - kbar,
// C/omega = sum_j wbar_j c_j c_j^T + (lambda/omega) I (the forward's centred operator),
// rho' = (C/omega)^{-1}(kbar - q_i) = rho_i omega/denom_i (from the forward's outputs),
// h_j = g_i.v_j, hbar = sum_j wbar_j h_j, tbar = sum_j wbar_j h_j c_j, and
//   y       = (C/omega)^{-1} tbar                    (the adjoint solve: one CG on the same operator)
//   Ahat_j  = 1 - c_j.rho',   Bhat_j = (h_j - hbar) - c_j.y,   ds_j = wbar_j Ahat_j Bhat_j
//   dv_j   += wbar_j Ahat_j g_i
//   dk_j   += tau ds_j q_i - wbar_j (Ahat_j y + Bhat_j rho')
//   dq_i    = tau sum_j ds_j k_j + y
// and, through the row maximum m_i = tau q_i.k_jm (jm the first index attaining it; lambda is
// absolute, so the output depends on m_i), with sd = sum_j ds_j = -(lambda/omega) rho'.y:
// dq_i -= tau sd k_jm and dk_jm -= tau sd q_i.
// The centred form is the exact gradient rewritten with delta.y = rho'.tbar (both equal
// delta^T (C/omega)^{-1} tbar): every factor is O(1), whereas the uncentred factors 1 - z_j.rho
// and the adjoint u = -(1 + delta.rho') y/omega carry the factor 1 + delta.rho', which is in the
// thousands for a query outside the span of its keys and costs fp32 most of its digits.
//
// Three kernels and no atomics, so the result does not depend on scheduling:
//  * stats, query-major, one CTA per tile of BQ queries of one (b, h): the row maximum and its
//    index, the moments omega, kbar, hbar, tbar (one sweep over keys and values) and CG for y.
//    Per-row scalars (RowRec) and y go to the workspace.
//  * dq, query-major: one sweep over keys and values that forms dq_i from the records.
//  * key-major, one CTA per block of BK keys: sweeps the query tiles at or after the block,
//    forms Ahat, Bhat, ds for every pair from the records and sums dk_j and dv_j in registers.
// Every product, sum and CG quantity is fp32.  Thread layout as in the fp32 forward path:
// 256 threads, the 8 consecutive lanes 8r..8r+7 own row r (a query row in the first kernel, a
// key row in the second); pair tiles split the other side's rows j = lane8 + 8c, d-vectors
// split coordinates e = lane8 + 8c.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "lla_internal.h"

namespace lla {
namespace {

constexpr int BQ = 32;
constexpr int BK = 32;       // equal to BQ: query tile t and key block t start at the same row
constexpr int NT = 256;
constexpr int JPT = BK / 8;  // pair columns per lane

using RowRec = BwdRowRec;

__device__ __forceinline__ float ld_f(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float row_sum8(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

// Stage rows [row0, row0+rows) of a [n, D] slice into dst (zero beyond n).
template <int D, typename T>
__device__ __forceinline__ void load_rows(float (*dst)[D + 1], const T* src, int row0, int rows, int n) {
    for (int idx = threadIdx.x; idx < rows * D; idx += NT) {
        const int r = idx / D, e = idx - r * D;
        const int g = row0 + r;
        dst[r][e] = (g < n) ? ld_f(src + (size_t)g * D + e) : 0.f;
    }
}

// o_a[c] = xa[r] . blk[l8 + 8c] for NX row arrays xa against one block.
template <int D, int NX>
__device__ __forceinline__ void dots_rows(const float (*x0)[D + 1], const float (*x1)[D + 1],
                                          const float (*x2)[D + 1], const float (*blk)[D + 1], int r, int l8,
                                          float (&o0)[JPT], float (&o1)[JPT], float (&o2)[JPT]) {
#pragma unroll
    for (int c = 0; c < JPT; ++c) { o0[c] = 0.f; o1[c] = 0.f; o2[c] = 0.f; }
#pragma unroll 8
    for (int e = 0; e < D; ++e) {
        const float a0 = x0[r][e];
        const float a1 = NX > 1 ? x1[r][e] : 0.f;
        const float a2 = NX > 2 ? x2[r][e] : 0.f;
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            const float b = blk[l8 + 8 * c][e];
            o0[c] = fmaf(a0, b, o0[c]);
            if (NX > 1) o1[c] = fmaf(a1, b, o1[c]);
            if (NX > 2) o2[c] = fmaf(a2, b, o2[c]);
        }
    }
}

// o_a[c] = x[r] . blka[l8 + 8c] for one row against NB blocks.
template <int D, int NB>
__device__ __forceinline__ void dots_blocks(const float (*x)[D + 1], const float (*b0)[D + 1],
                                            const float (*b1)[D + 1], const float (*b2)[D + 1], int r, int l8,
                                            float (&o0)[JPT], float (&o1)[JPT], float (&o2)[JPT]) {
#pragma unroll
    for (int c = 0; c < JPT; ++c) { o0[c] = 0.f; o1[c] = 0.f; o2[c] = 0.f; }
#pragma unroll 4
    for (int e = 0; e < D; ++e) {
        const float a = x[r][e];
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            o0[c] = fmaf(a, b0[l8 + 8 * c][e], o0[c]);
            if (NB > 1) o1[c] = fmaf(a, b1[l8 + 8 * c][e], o1[c]);
            if (NB > 2) o2[c] = fmaf(a, b2[l8 + 8 * c][e], o2[c]);
        }
    }
}

// acc[c'] += sum_j coef[r][j] * blk[j][e], e = l8 + 8c'.
template <int D>
__device__ __forceinline__ void acc_rows(const float (*coef)[BK + 1], const float (*blk)[D + 1], int r, int l8,
                                         float (&acc)[D / 8]) {
#pragma unroll 4
    for (int j = 0; j < BK; ++j) {
        const float cj = coef[r][j];
#pragma unroll
        for (int c = 0; c < D / 8; ++c) acc[c] = fmaf(cj, blk[j][l8 + 8 * c], acc[c]);
    }
}

// acc1 += sum_j c1[r][j] blk[j], acc2 += sum_j c2[r][j] blk[j].
template <int D>
__device__ __forceinline__ void acc_rows2(const float (*c1)[BK + 1], const float (*c2)[BK + 1],
                                          const float (*blk)[D + 1], int r, int l8, float (&acc1)[D / 8],
                                          float (&acc2)[D / 8]) {
#pragma unroll 4
    for (int j = 0; j < BK; ++j) {
        const float a = c1[r][j], b = c2[r][j];
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const float x = blk[j][l8 + 8 * c];
            acc1[c] = fmaf(a, x, acc1[c]);
            acc2[c] = fmaf(b, x, acc2[c]);
        }
    }
}

template <int D>
struct QSmem {
    float q[BQ][D + 1];    // query rows
    float g[BQ][D + 1];    // output cotangent rows
    float p[BQ][D + 1];    // CG direction, then rho'
    float u[BQ][D + 1];    // adjoint solution y
    float kb[BK][D + 1];   // key block
    float vb[BK][D + 1];   // value block
    float m[BQ][BK + 1];   // per-pair coefficients of the current block
    float m2[BQ][BK + 1];
};

template <int D>
struct KSmem {
    float k[BK][D + 1];    // this CTA's key rows
    float v[BK][D + 1];    // and value rows
    float q[BQ][D + 1];    // current query tile: q, g, rho', y
    float g[BQ][D + 1];
    float rho[BQ][D + 1];
    float u[BQ][D + 1];
    float cq[BK][BQ + 1];  // per-pair coefficients of q_i, y_i, rho'_i (for dk) and g_i (for dv)
    float cu[BK][BQ + 1];
    float cr[BK][BQ + 1];
    float cv[BK][BQ + 1];
    RowRec rec[BQ];
};

template <int D, typename T>
__global__ void __launch_bounds__(NT, 1)
lla_bwd_stats_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                     const T* __restrict__ dout, const float* __restrict__ rho, const float* __restrict__ denom,
                     RowRec* __restrict__ rec, float* __restrict__ uvec,
                     int* __restrict__ cg_iters, int n, int n_tiles, float tau, float lambda, int cg_max_iters,
                     float cg_tol) {
    constexpr int E = D / 8;  // coordinates per lane
    extern __shared__ __align__(16) unsigned char smem_raw[];
    QSmem<D>& sm = *reinterpret_cast<QSmem<D>*>(smem_raw);

    const int tile = n_tiles - 1 - (int)blockIdx.x;  // longest causal ranges first
    const size_t head = blockIdx.y;
    const T* qh = q + head * (size_t)n * D;
    const T* kh = k + head * (size_t)n * D;
    const T* vh = v + head * (size_t)n * D;
    const T* gh = dout + head * (size_t)n * D;

    const int tid = threadIdx.x;
    const int r = tid >> 3;
    const int l8 = tid & 7;
    const int i0 = tile * BQ;
    const int i = i0 + r;
    const bool row_ok = i < n;
    const int last_key = min(n - 1, i0 + BQ - 1);
    const int n_blocks = last_key / BK + 1;
    const size_t rbase = (head * (size_t)n + (row_ok ? i : 0)) * D;

    load_rows<D>(sm.q, qh, i0, BQ, n);
    load_rows<D>(sm.g, gh, i0, BQ, n);

    // ---- row maximum of the logits and the first index attaining it ------------------------
    float m_row = -INFINITY;
    int jm = 0x7fffffff;
    for (int kb = 0; kb < n_blocks; ++kb) {
        __syncthreads();
        load_rows<D>(sm.kb, kh, kb * BK, BK, n);
        __syncthreads();
        float s[JPT], o1[JPT], o2[JPT];
        dots_rows<D, 1>(sm.q, nullptr, nullptr, sm.kb, r, l8, s, o1, o2);
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            const int j = kb * BK + l8 + 8 * c;
            const float x = tau * s[c];
            if (j <= i && row_ok && x > m_row) { m_row = x; jm = j; }  // j grows, so the first index wins
        }
    }
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m_row, off);
        const int oj = __shfl_xor_sync(0xffffffffu, jm, off);
        if (om > m_row || (om == m_row && oj < jm)) { m_row = om; jm = oj; }
    }

    // ---- moments: omega, sum w k, sum w h, sum w h k ----------------------------------------
    float acc1[E], acc2[E];
#pragma unroll
    for (int c = 0; c < E; ++c) { acc1[c] = 0.f; acc2[c] = 0.f; }
    float om_part = 0.f, wh_part = 0.f;
    for (int kb = 0; kb < n_blocks; ++kb) {
        __syncthreads();
        load_rows<D>(sm.kb, kh, kb * BK, BK, n);
        load_rows<D>(sm.vb, vh, kb * BK, BK, n);
        __syncthreads();
        float s[JPT], hh[JPT], o1[JPT], o2[JPT];
        dots_rows<D, 1>(sm.q, nullptr, nullptr, sm.kb, r, l8, s, o1, o2);
        dots_rows<D, 1>(sm.g, nullptr, nullptr, sm.vb, r, l8, hh, o1, o2);
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            const int j = kb * BK + l8 + 8 * c;
            const float w = (j <= i && row_ok) ? expf(tau * s[c] - m_row) : 0.f;
            const float wh = w * hh[c];
            om_part += w;
            wh_part += wh;
            sm.m[r][l8 + 8 * c] = w;
            sm.m2[r][l8 + 8 * c] = wh;
        }
        __syncwarp();
        acc_rows2<D>(sm.m, sm.m2, sm.kb, r, l8, acc1, acc2);
    }
    const float omega_sum = row_sum8(om_part);
    const float swh = row_sum8(wh_part);
    const float omega = row_ok ? omega_sum : 1.f;
    const float inv_omega = 1.f / omega;
    const float hbar = swh * inv_omega;
    const float den = row_ok ? denom[head * (size_t)n + i] : 1.f;
    const float rp_scale = omega / den;    // 1 + delta.rho'
    float kbar[E], b[E], rp[E];
#pragma unroll
    for (int c = 0; c < E; ++c) {
        kbar[c] = acc1[c] * inv_omega;
        b[c] = fmaf(acc2[c], inv_omega, -kbar[c] * hbar);   // tbar = sum_j wbar_j h_j (k_j - kbar)
        rp[c] = row_ok ? rho[rbase + l8 + 8 * c] * rp_scale : 0.f;
    }

    // ---- CG on (C/omega) y = tbar (the forward's centred operator) -------------------------
    float x[E], res[E], pv[E];
    float g2a = 0.f;
#pragma unroll
    for (int c = 0; c < E; ++c) {
        x[c] = 0.f;
        res[c] = row_ok ? b[c] : 0.f;
        pv[c] = res[c];
        g2a = fmaf(res[c], res[c], g2a);
    }
    float gamma = row_sum8(g2a);
    const float rn0 = sqrtf(gamma);
    bool active = row_ok && gamma > 0.f && !(sqrtf(gamma) <= cg_tol * rn0);
    int iters = 0;
    const float lam_n = lambda * inv_omega;

    for (int it = 0; it < cg_max_iters; ++it) {
        if (!__syncthreads_or(active ? 1 : 0)) break;
#pragma unroll
        for (int c = 0; c < E; ++c) sm.p[r][l8 + 8 * c] = pv[c];
        float kp = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) kp = fmaf(kbar[c], pv[c], kp);
        kp = row_sum8(kp);
#pragma unroll
        for (int c = 0; c < E; ++c) acc1[c] = 0.f;
        float msum_part = 0.f;
        for (int kb = 0; kb < n_blocks; ++kb) {
            __syncthreads();
            load_rows<D>(sm.kb, kh, kb * BK, BK, n);
            __syncthreads();
            float s[JPT], a[JPT], o2[JPT];
            dots_rows<D, 2>(sm.q, sm.p, nullptr, sm.kb, r, l8, s, a, o2);
#pragma unroll
            for (int c = 0; c < JPT; ++c) {
                const int j = kb * BK + l8 + 8 * c;
                const float w = (j <= i && row_ok) ? expf(tau * s[c] - m_row) : 0.f;
                const float mm = w * (a[c] - kp);
                msum_part += mm;
                sm.m[r][l8 + 8 * c] = mm;
            }
            __syncwarp();
            acc_rows<D>(sm.m, sm.kb, r, l8, acc1);
        }
        const float msum = row_sum8(msum_part);
        float cp[E];
        float pcp = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) {
            cp[c] = (acc1[c] - kbar[c] * msum) * inv_omega + lam_n * pv[c];
            pcp = fmaf(pv[c], cp[c], pcp);
        }
        pcp = row_sum8(pcp);
        const bool upd = active && (pcp > 0.f);
        const float alpha = upd ? gamma / pcp : 0.f;
        float g2 = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) {
            if (upd) {
                x[c] = fmaf(alpha, pv[c], x[c]);
                res[c] = fmaf(-alpha, cp[c], res[c]);
            }
            g2 = fmaf(res[c], res[c], g2);
        }
        g2 = row_sum8(g2);
        if (upd) {
            const float beta = g2 / gamma;
#pragma unroll
            for (int c = 0; c < E; ++c) pv[c] = fmaf(beta, pv[c], res[c]);
            gamma = g2;
            ++iters;
            if (gamma == 0.f || sqrtf(gamma) <= cg_tol * rn0) active = false;
        } else {
            active = false;
        }
    }

    // ---- per-row record and y ------------------------------------------------------------------
    float kr = 0.f, ky = 0.f, ry = 0.f;
#pragma unroll
    for (int c = 0; c < E; ++c) {
        kr = fmaf(kbar[c], rp[c], kr);
        ky = fmaf(kbar[c], x[c], ky);
        ry = fmaf(rp[c], x[c], ry);
    }
    kr = row_sum8(kr);
    ky = row_sum8(ky);
    ry = row_sum8(ry);
    if (row_ok) {
#pragma unroll
        for (int c = 0; c < E; ++c) uvec[rbase + l8 + 8 * c] = x[c];
        if (l8 == 0) {
            if (jm < 0 || jm > i) jm = 0;   // only when every logit of the row is NaN
            RowRec o;
            o.m = m_row;
            o.jm = jm;
            o.inv_omega = inv_omega;
            o.hbar = hbar;
            o.kb_rp = kr;
            o.kb_y = ky;
            o.sd = -lambda * inv_omega * ry;   // sum_j ds_j, the path through the row maximum
            o.rp_scale = rp_scale;
            rec[head * (size_t)n + i] = o;
            if (cg_iters) cg_iters[head * (size_t)n + i] = iters;
        }
    }
}

// dq_i = tau (sum_j ds_ij k_j - sd_i k_jm) + y_i, one CTA per tile of BQ queries, from the
// per-row records and y.
template <int D, typename T>
__global__ void __launch_bounds__(NT, 1)
lla_bwd_dq_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const T* __restrict__ dout, const float* __restrict__ rho, const RowRec* __restrict__ rec,
                  const float* __restrict__ uvec, float* __restrict__ dq, int n, int n_tiles, float tau) {
    constexpr int E = D / 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    QSmem<D>& sm = *reinterpret_cast<QSmem<D>*>(smem_raw);

    const int tile = n_tiles - 1 - (int)blockIdx.x;
    const size_t head = blockIdx.y;
    const size_t hoff = head * (size_t)n * D;
    const T* kh = k + hoff;
    const T* vh = v + hoff;
    const int tid = threadIdx.x;
    const int r = tid >> 3;
    const int l8 = tid & 7;
    const int i0 = tile * BQ;
    const int i = i0 + r;
    const bool row_ok = i < n;
    const int last_key = min(n - 1, i0 + BQ - 1);
    const int n_blocks = last_key / BK + 1;

    RowRec R{};
    if (row_ok) R = rec[head * (size_t)n + i];
    load_rows<D>(sm.q, q + hoff, i0, BQ, n);
    load_rows<D>(sm.g, dout + hoff, i0, BQ, n);
    load_rows<D>(sm.u, uvec + hoff, i0, BQ, n);
#pragma unroll
    for (int c = 0; c < E; ++c) {   // rho' = (omega/denom) rho; each row is read by its own lanes only
        const int e = l8 + 8 * c;
        sm.p[r][e] = row_ok ? __ldg(rho + hoff + (size_t)i * D + e) * R.rp_scale : 0.f;
    }
    float dqa[E];
#pragma unroll
    for (int c = 0; c < E; ++c) dqa[c] = 0.f;
    for (int kb = 0; kb < n_blocks; ++kb) {
        __syncthreads();
        load_rows<D>(sm.kb, kh, kb * BK, BK, n);
        load_rows<D>(sm.vb, vh, kb * BK, BK, n);
        __syncthreads();
        float s[JPT], a1[JPT], a2[JPT], hh[JPT], o1[JPT], o2[JPT];
        dots_rows<D, 3>(sm.q, sm.p, sm.u, sm.kb, r, l8, s, a1, a2);
        dots_rows<D, 1>(sm.g, nullptr, nullptr, sm.vb, r, l8, hh, o1, o2);
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            const int j = kb * BK + l8 + 8 * c;
            const float wb = (j <= i && row_ok) ? expf(tau * s[c] - R.m) * R.inv_omega : 0.f;
            const float Ah = 1.f - (a1[c] - R.kb_rp);
            const float Bh = (hh[c] - R.hbar) - (a2[c] - R.kb_y);
            sm.m[r][l8 + 8 * c] = wb * Ah * Bh;
        }
        __syncwarp();
        acc_rows<D>(sm.m, sm.kb, r, l8, dqa);
    }
    if (row_ok) {
        const T* kjm = kh + (size_t)R.jm * D;
        const size_t rbase = hoff + (size_t)i * D;
#pragma unroll
        for (int c = 0; c < E; ++c) {
            const int e = l8 + 8 * c;
            dq[rbase + e] = fmaf(tau, dqa[c] - R.sd * ld_f(kjm + e), sm.u[r][e]);
        }
    }
}

template <int D, typename T>
__global__ void __launch_bounds__(NT, 1)
lla_bwd_key_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ dout, const float* __restrict__ rho, const RowRec* __restrict__ rec,
                   const float* __restrict__ uvec, float* __restrict__ dk, float* __restrict__ dv, int n,
                   int n_tiles, float tau) {
    constexpr int E = D / 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    KSmem<D>& sm = *reinterpret_cast<KSmem<D>*>(smem_raw);

    const int kblk = (int)blockIdx.x;  // the earliest keys have the longest query range: first
    const size_t head = blockIdx.y;
    const size_t hoff = head * (size_t)n * D;
    const int tid = threadIdx.x;
    const int r = tid >> 3;
    const int l8 = tid & 7;
    const int j0 = kblk * BK;
    const int j = j0 + r;
    const bool key_ok = j < n;

    load_rows<D>(sm.k, k + hoff, j0, BK, n);
    load_rows<D>(sm.v, v + hoff, j0, BK, n);
    float dka[E], dva[E];
#pragma unroll
    for (int c = 0; c < E; ++c) { dka[c] = 0.f; dva[c] = 0.f; }

    for (int qt = kblk; qt < n_tiles; ++qt) {
        const int i0 = qt * BQ;
        __syncthreads();
        if (tid < BQ) {
            RowRec z{};
            sm.rec[tid] = (i0 + tid < n) ? rec[head * (size_t)n + i0 + tid] : z;
        }
        load_rows<D>(sm.q, q + hoff, i0, BQ, n);
        load_rows<D>(sm.g, dout + hoff, i0, BQ, n);
        load_rows<D>(sm.u, uvec + hoff, i0, BQ, n);
        __syncthreads();
        for (int idx = tid; idx < BQ * D; idx += NT) {   // rho' = (omega/denom) rho
            const int rr = idx / D, e = idx - rr * D;
            const int gi = i0 + rr;
            sm.rho[rr][e] = (gi < n) ? __ldg(rho + hoff + (size_t)gi * D + e) * sm.rec[rr].rp_scale : 0.f;
        }
        __syncthreads();
        float s[JPT], kr[JPT], ky[JPT], hh[JPT], o1[JPT], o2[JPT];
        dots_blocks<D, 3>(sm.k, sm.q, sm.rho, sm.u, r, l8, s, kr, ky);
        dots_blocks<D, 1>(sm.v, sm.g, nullptr, nullptr, r, l8, hh, o1, o2);
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            const int ii = l8 + 8 * c;
            const int i = i0 + ii;
            const RowRec& R = sm.rec[ii];
            const bool valid = key_ok && i < n && j <= i;
            const float wb = valid ? expf(tau * s[c] - R.m) * R.inv_omega : 0.f;
            const float Ah = 1.f - (kr[c] - R.kb_rp);
            const float Bh = (hh[c] - R.hbar) - (ky[c] - R.kb_y);
            const float ds = wb * Ah * Bh;
            const float corr = (valid && j == R.jm) ? R.sd : 0.f;  // through the row maximum
            sm.cq[r][ii] = tau * (ds - corr);
            sm.cu[r][ii] = -wb * Ah;
            sm.cr[r][ii] = -wb * Bh;
            sm.cv[r][ii] = wb * Ah;
        }
        __syncwarp();
#pragma unroll 2
        for (int ii = 0; ii < BQ; ++ii) {
            const float a = sm.cq[r][ii], bu = sm.cu[r][ii], br = sm.cr[r][ii], bv = sm.cv[r][ii];
#pragma unroll
            for (int c = 0; c < E; ++c) {
                const int e = l8 + 8 * c;
                float t = fmaf(a, sm.q[ii][e], dka[c]);
                t = fmaf(bu, sm.u[ii][e], t);
                dka[c] = fmaf(br, sm.rho[ii][e], t);
                dva[c] = fmaf(bv, sm.g[ii][e], dva[c]);
            }
        }
    }
    if (key_ok) {
        const size_t base = hoff + (size_t)j * D;
#pragma unroll
        for (int c = 0; c < E; ++c) {
            dk[base + l8 + 8 * c] = dka[c];
            dv[base + l8 + 8 * c] = dva[c];
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int D, typename T>
cudaError_t launch_stats_typed(const BackwardProblem& p, RowRec* rec, float* uvec, cudaStream_t stream) {
    const int n_tiles = (p.n + BQ - 1) / BQ;
    auto ks = lla_bwd_stats_kernel<D, T>;
    const size_t smq = sizeof(QSmem<D>);
    cudaError_t err = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smq);
    if (err != cudaSuccess) return err;
    const dim3 grid(n_tiles, p.B * p.H);
    if (p.ev_main_begin && (err = cudaEventRecord(p.ev_main_begin, stream)) != cudaSuccess) return err;
    ks<<<grid, NT, smq, stream>>>(static_cast<const T*>(p.q), static_cast<const T*>(p.k), static_cast<const T*>(p.v),
                                  static_cast<const T*>(p.dout), p.rho, p.denom, rec, uvec, p.cg_iters, p.n, n_tiles,
                                  p.tau, p.lambda, p.cg_max_iters, p.cg_tol);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (p.ev_main_end && (err = cudaEventRecord(p.ev_main_end, stream)) != cudaSuccess) return err;
    return cudaSuccess;
}

template <int D, typename T>
cudaError_t launch_rest_typed(const BackwardProblem& p, const RowRec* rec, const float* uvec, cudaStream_t stream) {
    const int n_tiles = (p.n + BQ - 1) / BQ;
    auto kd = lla_bwd_dq_kernel<D, T>;
    auto kk = lla_bwd_key_kernel<D, T>;
    const size_t smq = sizeof(QSmem<D>), smk = sizeof(KSmem<D>);
    cudaError_t err = cudaFuncSetAttribute(kd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smq);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
    if (err != cudaSuccess) return err;
    const dim3 grid(n_tiles, p.B * p.H);
    const T* q = static_cast<const T*>(p.q);
    const T* k = static_cast<const T*>(p.k);
    const T* v = static_cast<const T*>(p.v);
    const T* g = static_cast<const T*>(p.dout);
    kd<<<grid, NT, smq, stream>>>(q, k, v, g, p.rho, rec, uvec, p.dq, p.n, n_tiles, p.tau);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    kk<<<grid, NT, smk, stream>>>(q, k, v, g, p.rho, rec, uvec, p.dk, p.dv, p.n, n_tiles, p.tau);
    return cudaGetLastError();
}

template <typename T>
cudaError_t stats_dim(const BackwardProblem& p, RowRec* rec, float* uvec, cudaStream_t stream) {
    switch (p.d) {
        case 16: return launch_stats_typed<16, T>(p, rec, uvec, stream);
        case 32: return launch_stats_typed<32, T>(p, rec, uvec, stream);
        case 64: return launch_stats_typed<64, T>(p, rec, uvec, stream);
        case 128: return launch_stats_typed<128, T>(p, rec, uvec, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t rest_dim(const BackwardProblem& p, const RowRec* rec, const float* uvec, cudaStream_t stream) {
    switch (p.d) {
        case 16: return launch_rest_typed<16, T>(p, rec, uvec, stream);
        case 32: return launch_rest_typed<32, T>(p, rec, uvec, stream);
        case 64: return launch_rest_typed<64, T>(p, rec, uvec, stream);
        case 128: return launch_rest_typed<128, T>(p, rec, uvec, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t backward_records_bytes(int B, int H, int n, int d) {
    const size_t rows = (size_t)B * H * n;
    return align256(rows * sizeof(RowRec)) + align256(rows * (size_t)d * sizeof(float));
}

size_t backward_workspace_bytes(int path, int B, int H, int n, int d) {
    const size_t recs = backward_records_bytes(B, H, n, d);
    return path == 1 ? recs + tensor_backward_stats_bytes(B, H, n, d) : recs;
}

cudaError_t launch_backward_rest(const BackwardProblem& p, const BwdRowRec* rec, const float* yvec,
                                 cudaStream_t stream) {
    if (p.dtype == 1) return rest_dim<float>(p, rec, yvec, stream);
    return rest_dim<__nv_bfloat16>(p, rec, yvec, stream);
}

cudaError_t launch_backward(const BackwardProblem& p, int path, void* workspace, cudaStream_t stream,
                            const char** why) {
    const size_t rows = (size_t)p.B * p.H * p.n;
    RowRec* rec = static_cast<RowRec*>(workspace);
    float* yvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * sizeof(RowRec)));
    cudaError_t err;
    if (path == 1) {
        void* tws = static_cast<char*>(workspace) + backward_records_bytes(p.B, p.H, p.n, p.d);
        err = launch_tensor_backward_stats(p, tws, rec, yvec, stream, why);
        if (err != cudaSuccess) return err;
    } else {
        err = p.dtype == 1 ? stats_dim<float>(p, rec, yvec, stream) : stats_dim<__nv_bfloat16>(p, rec, yvec, stream);
        if (err != cudaSuccess) { *why = "fp32 backward stats launch"; return err; }
    }
    err = launch_backward_rest(p, rec, yvec, stream);
    if (err != cudaSuccess) *why = "backward dq / key-major launch";
    return err;
}

}  // namespace lla
