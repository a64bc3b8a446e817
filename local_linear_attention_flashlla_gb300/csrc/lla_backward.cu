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

    int rank, head_i;
    causal_order(3 * (size_t)n * D * sizeof(T), rank, head_i);   // keys, values and upstream gradients
    const int tile = n_tiles - 1 - rank;
    const size_t head = (size_t)head_i;
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

// ---- dq and dk/dv: register-tiled fp32 sweeps over the records ----------------------------
// Both kernels form, for a block of (query, key) pairs, the four dot products s = q.k,
// a1 = rho'.k, a2 = y.k, h = g.v (phase A), the per-pair coefficients (phase B) and then the
// gradient sums (phase C).  Each thread owns a small register tile of pairs or outputs and
// reads its shared-memory operands as float4, so an FMA costs an eighth of a load instead of
// one: q, rho', y, g rows are stored [row][coordinate], key rows [coordinate][key].
constexpr int KB2 = 64;        // keys per CTA of the dk/dv kernel
constexpr int QB2 = 32;        // queries per step of the dk/dv kernel
constexpr int QB3 = 64;        // queries per CTA of the dq kernel
constexpr int KS3 = 32;        // keys per step of the dq kernel

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float at4(const float4& v, int u) { return u == 0 ? v.x : u == 1 ? v.y : u == 2 ? v.z : v.w; }

// Phase C coordinates of thread group eg (0..15): EC = D/16 per thread.  With EC = 8 the two
// float4 halves sit at 4 eg and D/2 + 4 eg, so the 16 groups of a warp read contiguous 256-byte
// runs (no bank conflicts); otherwise EC consecutive coordinates from EC eg.
template <int D, int EC>
__device__ __forceinline__ int ec_col(int eg, int h) {
    return EC == 8 ? (h < 4 ? 4 * eg + h : D / 2 + 4 * eg + h - 4) : EC * eg + h;
}
template <int D, int EC>
__device__ __forceinline__ void load_ec(const float* row, int eg, float (&o)[EC]) {
    if constexpr (EC == 8) {
        const float4 a = ld4(row + 4 * eg), b = ld4(row + D / 2 + 4 * eg);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    } else if constexpr (EC == 4) {
        const float4 a = ld4(row + 4 * eg);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    } else {
#pragma unroll
        for (int h = 0; h < EC; ++h) o[h] = row[EC * eg + h];
    }
}
template <int D, int EC>
__device__ __forceinline__ void store_ec(float* row, int eg, const float (&o)[EC]) {
    if constexpr (EC == 8) {
        *reinterpret_cast<float4*>(row + 4 * eg) = make_float4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<float4*>(row + D / 2 + 4 * eg) = make_float4(o[4], o[5], o[6], o[7]);
    } else if constexpr (EC == 4) {
        *reinterpret_cast<float4*>(row + 4 * eg) = make_float4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int h = 0; h < EC; ++h) row[EC * eg + h] = o[h];
    }
}

// rows [row0, row0+rows) of a [n, D] slice into dst[row][0..D) (row stride DP), zero beyond n
template <int D, int DP, typename T>
__device__ __forceinline__ void stage_rows(float* dst, const T* src, int row0, int rows, int n, const RowRec* rec = nullptr) {
    for (int idx = threadIdx.x; idx < rows * D; idx += NT) {
        const int r = idx / D, e = idx - r * D;
        const int gr = row0 + r;
        float x = (gr < n) ? ld_f(src + (size_t)gr * D + e) : 0.f;
        if (rec) x *= rec[r].rp_scale;        // rho' = (omega/denom) rho
        dst[r * DP + e] = x;
    }
}
// rows [row0, row0+rows) transposed into dst[coordinate][row] (row stride KP), zero beyond n
template <int D, int KP, typename T>
__device__ __forceinline__ void stage_cols(float* dst, const T* src, int row0, int rows, int n) {
    for (int idx = threadIdx.x; idx < rows * D; idx += NT) {
        const int r = idx / D, e = idx - r * D;
        const int gr = row0 + r;
        dst[e * KP + r] = (gr < n) ? ld_f(src + (size_t)gr * D + e) : 0.f;
    }
}

// Phase A for two query rows (qa, qb: [row][coordinate] with stride DP) against four keys
// (kT, vT: [coordinate][key] with stride KP, starting at the thread's first key).
template <int D, int DP, int KP>
__device__ __forceinline__ void pair_dots(const float* qa, const float* ra, const float* ya, const float* ga,
                                          const float* kT, const float* vT, float (&s)[2][4], float (&a1)[2][4],
                                          float (&a2)[2][4], float (&h)[2][4]) {
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int c = 0; c < 4; ++c) { s[u][c] = 0.f; a1[u][c] = 0.f; a2[u][c] = 0.f; h[u][c] = 0.f; }
#pragma unroll 2
    for (int e = 0; e < D; e += 4) {
        const float4 q0 = ld4(qa + e), q1 = ld4(qa + DP + e);
        const float4 r0 = ld4(ra + e), r1 = ld4(ra + DP + e);
        const float4 y0 = ld4(ya + e), y1 = ld4(ya + DP + e);
        const float4 g0 = ld4(ga + e), g1 = ld4(ga + DP + e);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float4 kk = ld4(kT + (e + u) * KP), vv = ld4(vT + (e + u) * KP);
            const float kc[4] = {kk.x, kk.y, kk.z, kk.w}, vc[4] = {vv.x, vv.y, vv.z, vv.w};
            const float qe[2] = {at4(q0, u), at4(q1, u)}, re[2] = {at4(r0, u), at4(r1, u)};
            const float ye[2] = {at4(y0, u), at4(y1, u)}, ge[2] = {at4(g0, u), at4(g1, u)};
#pragma unroll
            for (int w = 0; w < 2; ++w)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    s[w][c] = fmaf(qe[w], kc[c], s[w][c]);
                    a1[w][c] = fmaf(re[w], kc[c], a1[w][c]);
                    a2[w][c] = fmaf(ye[w], kc[c], a2[w][c]);
                    h[w][c] = fmaf(ge[w], vc[c], h[w][c]);
                }
        }
    }
}

// Phase B for one pair: wbar Ahat, -wbar Bhat and ds - (path through the row maximum)
__device__ __forceinline__ void pair_coef(const RowRec& R, bool valid, bool at_max, float tau, float s, float a1,
                                          float a2, float h, float& cq, float& cw, float& cr) {
    const float wb = valid ? expf(tau * s - R.m) * R.inv_omega : 0.f;
    const float Ah = 1.f - (a1 - R.kb_rp);
    const float Bh = (h - R.hbar) - (a2 - R.kb_y);
    const float ds = wb * Ah * Bh;
    cq = tau * (ds - (valid && at_max ? R.sd : 0.f));
    cw = wb * Ah;
    cr = -wb * Bh;
}

template <int D>
struct K2Smem {
    static constexpr int KP = KB2 + 4, DP = D + 4;
    float kT[D * KP];              // this CTA's keys and values, [coordinate][key]
    float vT[D * KP];
    float q[QB2 * DP];             // the current query step, [query][coordinate]
    float r[QB2 * DP];             // rho'
    float y[QB2 * DP];
    float g[QB2 * DP];
    float cq[QB2 * KP];            // tau (ds - max path), [query][key]
    float cw[QB2 * KP];            // wbar Ahat
    float cr[QB2 * KP];            // -wbar Bhat
    RowRec rec[QB2];
};

// dk_j = sum_{i >= j} [cq_ij q_i - cw_ij y_i + cr_ij rho'_i],  dv_j = sum_{i >= j} cw_ij g_i.
template <int D, typename T>
__global__ void __launch_bounds__(NT, 1)
lla_bwd_key_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const T* __restrict__ dout, const float* __restrict__ rho, const RowRec* __restrict__ rec,
                   const float* __restrict__ uvec, float* __restrict__ dk, float* __restrict__ dv, int n, float tau) {
    using S = K2Smem<D>;
    constexpr int KP = S::KP, DP = S::DP;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    S& sm = *reinterpret_cast<S*>(smem_raw);
    const int tid = threadIdx.x;
    int rank, head_i;                           // the earliest keys have the longest query range
    causal_order(3 * (size_t)n * D * sizeof(T), rank, head_i);   // queries, upstream gradients, u
    const int j0 = rank * KB2;
    const size_t head = (size_t)head_i;
    const size_t hoff = head * (size_t)n * D;

    stage_cols<D, KP>(sm.kT, k + hoff, j0, KB2, n);
    stage_cols<D, KP>(sm.vT, v + hoff, j0, KB2, n);
    // phase A/B tile: 4 keys x 2 queries; phase C tile: 4 keys x EC coordinates
    constexpr int EC = D / 16;
    const int kg = tid & 15, qg = tid >> 4;
    const int kc2 = tid >> 4, eg = tid & 15;
    float dka[4][EC], dva[4][EC];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < EC; ++e) { dka[c][e] = 0.f; dva[c][e] = 0.f; }

    for (int i0 = j0; i0 < n; i0 += QB2) {
        __syncthreads();
        if (tid < QB2) {
            RowRec z{};
            sm.rec[tid] = (i0 + tid < n) ? rec[head * (size_t)n + i0 + tid] : z;
        }
        stage_rows<D, DP>(sm.q, q + hoff, i0, QB2, n);
        stage_rows<D, DP>(sm.g, dout + hoff, i0, QB2, n);
        stage_rows<D, DP>(sm.y, uvec + hoff, i0, QB2, n);
        __syncthreads();
        stage_rows<D, DP>(sm.r, rho + hoff, i0, QB2, n, sm.rec);
        __syncthreads();
        {   // phases A and B
            float s_[2][4], a1[2][4], a2[2][4], h[2][4];
            const int ql = 2 * qg;
            pair_dots<D, DP, KP>(sm.q + ql * DP, sm.r + ql * DP, sm.y + ql * DP, sm.g + ql * DP, sm.kT + 4 * kg,
                                 sm.vT + 4 * kg, s_, a1, a2, h);
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const RowRec& R = sm.rec[ql + w];
                const int i = i0 + ql + w;
                float cq[4], cw[4], cr[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = j0 + 4 * kg + c;
                    const bool valid = j < n && i < n && j <= i;
                    pair_coef(R, valid, j == R.jm, tau, s_[w][c], a1[w][c], a2[w][c], h[w][c], cq[c], cw[c], cr[c]);
                }
                *reinterpret_cast<float4*>(sm.cq + (ql + w) * KP + 4 * kg) = make_float4(cq[0], cq[1], cq[2], cq[3]);
                *reinterpret_cast<float4*>(sm.cw + (ql + w) * KP + 4 * kg) = make_float4(cw[0], cw[1], cw[2], cw[3]);
                *reinterpret_cast<float4*>(sm.cr + (ql + w) * KP + 4 * kg) = make_float4(cr[0], cr[1], cr[2], cr[3]);
            }
        }
        __syncthreads();
        // phase C
#pragma unroll 2
        for (int il = 0; il < QB2; ++il) {
            const float4 cq4 = ld4(sm.cq + il * KP + 4 * kc2), cw4 = ld4(sm.cw + il * KP + 4 * kc2);
            const float4 cr4 = ld4(sm.cr + il * KP + 4 * kc2);
            const float cq[4] = {cq4.x, cq4.y, cq4.z, cq4.w}, cw[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
            const float cr[4] = {cr4.x, cr4.y, cr4.z, cr4.w};
            float qv[EC], yv[EC], rv[EC], gv[EC];
            load_ec<D, EC>(sm.q + il * DP, eg, qv);
            load_ec<D, EC>(sm.y + il * DP, eg, yv);
            load_ec<D, EC>(sm.r + il * DP, eg, rv);
            load_ec<D, EC>(sm.g + il * DP, eg, gv);
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < EC; ++e) {
                    float t = fmaf(cq[c], qv[e], dka[c][e]);
                    t = fmaf(-cw[c], yv[e], t);
                    dka[c][e] = fmaf(cr[c], rv[e], t);
                    dva[c][e] = fmaf(cw[c], gv[e], dva[c][e]);
                }
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int j = j0 + 4 * kc2 + c;
        if (j < n) {
            store_ec<D, EC>(dk + hoff + (size_t)j * D, eg, dka[c]);
            store_ec<D, EC>(dv + hoff + (size_t)j * D, eg, dva[c]);
        }
    }
}

template <int D>
struct Q3Smem {
    static constexpr int KP = KS3 + 4, DP = D + 4, QP = QB3 + 4;
    float q[QB3 * DP];             // this CTA's queries, [query][coordinate]
    float r[QB3 * DP];
    float y[QB3 * DP];
    float g[QB3 * DP];
    float kT[D * KP];              // the current key step, [coordinate][key]
    float vT[D * KP];
    float k[KS3 * DP];             // the same keys, [key][coordinate]
    float ds[KS3 * QP];            // ds, [key][query]
    RowRec rec[QB3];
};

// dq_i = tau (sum_j ds_ij k_j - sd_i k_jm) + y_i over the keys j <= i.
template <int D, typename T>
__global__ void __launch_bounds__(NT, 1)
lla_bwd_dq_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                  const T* __restrict__ dout, const float* __restrict__ rho, const RowRec* __restrict__ rec,
                  const float* __restrict__ uvec, float* __restrict__ dq, int n, int n_tiles, float tau) {
    using S = Q3Smem<D>;
    constexpr int KP = S::KP, DP = S::DP, QP = S::QP;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    S& sm = *reinterpret_cast<S*>(smem_raw);
    const int tid = threadIdx.x;
    int rank, head_i;
    causal_order(2 * (size_t)n * D * sizeof(T), rank, head_i);   // keys and values of a head
    const int i0 = (n_tiles - 1 - rank) * QB3;
    const size_t head = (size_t)head_i;
    const size_t hoff = head * (size_t)n * D;
    const int last_key = min(n - 1, i0 + QB3 - 1);

    if (tid < QB3) {
        RowRec z{};
        sm.rec[tid] = (i0 + tid < n) ? rec[head * (size_t)n + i0 + tid] : z;
    }
    stage_rows<D, DP>(sm.q, q + hoff, i0, QB3, n);
    stage_rows<D, DP>(sm.g, dout + hoff, i0, QB3, n);
    stage_rows<D, DP>(sm.y, uvec + hoff, i0, QB3, n);
    __syncthreads();
    stage_rows<D, DP>(sm.r, rho + hoff, i0, QB3, n, sm.rec);
    // phase A/B tile: 2 queries x 4 keys; phase C tile: 4 queries x EC coordinates
    constexpr int EC = D / 16;
    const int kg = tid & 7, qg = tid >> 3;
    const int qc = (tid >> 4) * 4, eg = tid & 15;
    float dqa[4][EC];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < EC; ++e) dqa[c][e] = 0.f;

    for (int j0 = 0; j0 <= last_key; j0 += KS3) {
        __syncthreads();
        stage_cols<D, KP>(sm.kT, k + hoff, j0, KS3, n);
        stage_cols<D, KP>(sm.vT, v + hoff, j0, KS3, n);
        stage_rows<D, DP>(sm.k, k + hoff, j0, KS3, n);
        __syncthreads();
        {
            float s_[2][4], a1[2][4], a2[2][4], h[2][4];
            const int ql = 2 * qg;
            pair_dots<D, DP, KP>(sm.q + ql * DP, sm.r + ql * DP, sm.y + ql * DP, sm.g + ql * DP, sm.kT + 4 * kg,
                                 sm.vT + 4 * kg, s_, a1, a2, h);
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const RowRec& R = sm.rec[ql + w];
                const int i = i0 + ql + w;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int j = j0 + 4 * kg + c;
                    const bool valid = j < n && i < n && j <= i;
                    const float wb = valid ? expf(tau * s_[w][c] - R.m) * R.inv_omega : 0.f;
                    const float Ah = 1.f - (a1[w][c] - R.kb_rp);
                    const float Bh = (h[w][c] - R.hbar) - (a2[w][c] - R.kb_y);
                    sm.ds[(4 * kg + c) * QP + ql + w] = wb * Ah * Bh;
                }
            }
        }
        __syncthreads();
#pragma unroll 2
        for (int jl = 0; jl < KS3; ++jl) {
            const float4 d4 = ld4(sm.ds + jl * QP + qc);
            const float dsv[4] = {d4.x, d4.y, d4.z, d4.w};
            float kv[EC];
            load_ec<D, EC>(sm.k + jl * DP, eg, kv);
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < EC; ++e) dqa[c][e] = fmaf(dsv[c], kv[e], dqa[c][e]);
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int il = qc + c, i = i0 + il;
        if (i < n) {
            const RowRec& R = sm.rec[il];
            const T* kjm = k + hoff + (size_t)R.jm * D;
            float o[EC];
#pragma unroll
            for (int e = 0; e < EC; ++e) {
                const int col = ec_col<D, EC>(eg, e);
                o[e] = fmaf(tau, dqa[c][e] - R.sd * ld_f(kjm + col), sm.y[il * DP + col]);
            }
            store_ec<D, EC>(dq + hoff + (size_t)i * D, eg, o);
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
cudaError_t launch_dq_typed(const BackwardProblem& p, const RowRec* rec, const float* uvec, cudaStream_t stream) {
    auto kd = lla_bwd_dq_kernel<D, T>;
    const size_t smd = sizeof(Q3Smem<D>);
    cudaError_t err = cudaFuncSetAttribute(kd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smd);
    if (err != cudaSuccess) return err;
    const int dq_tiles = (p.n + QB3 - 1) / QB3;
    kd<<<dim3(dq_tiles, p.B * p.H), NT, smd, stream>>>(static_cast<const T*>(p.q), static_cast<const T*>(p.k),
                                                       static_cast<const T*>(p.v), static_cast<const T*>(p.dout),
                                                       p.rho, rec, uvec, p.dq, p.n, dq_tiles, p.tau);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t launch_key_typed(const BackwardProblem& p, const RowRec* rec, const float* uvec, cudaStream_t stream) {
    auto kk = lla_bwd_key_kernel<D, T>;
    const size_t smk = sizeof(K2Smem<D>);
    cudaError_t err = cudaFuncSetAttribute(kk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
    if (err != cudaSuccess) return err;
    kk<<<dim3((p.n + KB2 - 1) / KB2, p.B * p.H), NT, smk, stream>>>(
        static_cast<const T*>(p.q), static_cast<const T*>(p.k), static_cast<const T*>(p.v),
        static_cast<const T*>(p.dout), p.rho, rec, uvec, p.dk, p.dv, p.n, p.tau);
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
cudaError_t dq_dim(const BackwardProblem& p, const RowRec* rec, const float* uvec, cudaStream_t stream) {
    switch (p.d) {
        case 16: return launch_dq_typed<16, T>(p, rec, uvec, stream);
        case 32: return launch_dq_typed<32, T>(p, rec, uvec, stream);
        case 64: return launch_dq_typed<64, T>(p, rec, uvec, stream);
        case 128: return launch_dq_typed<128, T>(p, rec, uvec, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t key_dim(const BackwardProblem& p, const RowRec* rec, const float* uvec, cudaStream_t stream) {
    switch (p.d) {
        case 16: return launch_key_typed<16, T>(p, rec, uvec, stream);
        case 32: return launch_key_typed<32, T>(p, rec, uvec, stream);
        case 64: return launch_key_typed<64, T>(p, rec, uvec, stream);
        case 128: return launch_key_typed<128, T>(p, rec, uvec, stream);
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
    return path == 1 ? recs + tensor_backward_stats_bytes(B, H, n, d) + tensor_kv_bytes(B, H, n, d) : recs;
}

cudaError_t launch_backward(const BackwardProblem& p, int path, void* workspace, cudaStream_t stream,
                            const char** why) {
    const size_t rows = (size_t)p.B * p.H * p.n;
    RowRec* rec = static_cast<RowRec*>(workspace);
    float* yvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * sizeof(RowRec)));
    cudaError_t err;
    if (path == 1) {
        // stats, dq (recording the per-key coefficient maxima) and dk/dv on tcgen05
        char* tws = static_cast<char*>(workspace) + backward_records_bytes(p.B, p.H, p.n, p.d);
        err = launch_tensor_backward_stats(p, tws, rec, yvec, stream, why);
        if (err != cudaSuccess) return err;
        const TensorOperands ops = tensor_backward_operands(tws, p.B, p.H, p.n, p.d);
        const KvScratch kv = tensor_kv_scratch(tws + tensor_backward_stats_bytes(p.B, p.H, p.n, p.d), p.B, p.H, p.n, p.d);
        if ((err = launch_tensor_kv_prep(p, rec, yvec, kv, stream)) != cudaSuccess) { *why = "dk/dv prep"; return err; }
        if ((err = launch_tensor_dq(p, rec, yvec, ops, kv, stream, why)) != cudaSuccess) return err;
        return launch_tensor_kv(p, rec, ops, kv, stream, why);
    }
    err = p.dtype == 1 ? stats_dim<float>(p, rec, yvec, stream) : stats_dim<__nv_bfloat16>(p, rec, yvec, stream);
    if (err != cudaSuccess) { *why = "fp32 backward stats launch"; return err; }
    if ((err = p.dtype == 1 ? dq_dim<float>(p, rec, yvec, stream) : dq_dim<__nv_bfloat16>(p, rec, yvec, stream)) !=
        cudaSuccess) {
        *why = "backward dq launch";
        return err;
    }
    err = p.dtype == 1 ? key_dim<float>(p, rec, yvec, stream) : key_dim<__nv_bfloat16>(p, rec, yvec, stream);
    if (err != cudaSuccess) *why = "backward key-major launch";
    return err;
}

}  // namespace lla
