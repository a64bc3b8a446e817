// fp32 CUDA-core path of the causal LLA forward pass.
//
// One CTA owns a tile of BQ consecutive queries of one (b, h) and runs the FlashLLA
// phases of the Local Linear Attention reading notes (section 2.2, Algorithm 1) over the
// causal key range of the tile, streaming key/value blocks of BK rows through shared
// memory:
//   (0) exact row maximum m_i of tau q_i.k_j (a logits-only sweep, so every later
//       weight is w_ij = exp(tau q_i.k_j - m_i) with the final maximum; lambda is
//       absolute, so the normalisation must be exact),
//   (1) moments omega_i = sum_j w_ij and mu~_i = sum_j w_ij k_j (Eq. (10)),
//   (2) conjugate gradient on the centred system (C_i/omega_i) rho'_i = delta_i,
//       delta_i = kbar_i - q_i, kbar_i = mu~_i/omega_i, with the matrix-free product
//       (C_i/omega_i) p = [sum_j w_ij ((k_j - kbar_i).p) k_j - kbar_i sum_j w_ij ((k_j - kbar_i).p)]/omega_i
//                         + (lambda/omega_i) p         (Eqs. (11)-(12) with the mean in place of q),
//   (3) rho_i = rho'_i/(1 + delta_i.rho'_i), denom_i = omega_i/(1 + delta_i.rho'_i) and the
//       output sweep out_i = sum_j u_ij v_j / sum_j u_ij, u_ij = w_ij (1 - (k_j - kbar_i).rho'_i),
//       which is Eq. (8); sum_j u_ij equals omega_i exactly because sum_j w_ij (k_j - kbar_i) = 0,
//       and normalising by the computed sum keeps sum_j s_ij = 1 in rounding as well.
// Parallax form (a caller-supplied probe, Parallax page): phases (0), (1) and the output
// sweep of (3) with the probe as rho', i.e. out_i = sum_j wbar_ij (1 - (k_j - kbar_i).probe_i) v_j,
// the softmax output minus the softmax-weighted value/key covariance times the probe.
// Every product, sum and CG quantity is fp32.  No global scratch.
//
// Thread layout (256 threads): row r = tid / 8 is owned by the 8 consecutive lanes
// 8r .. 8r+7 of one warp.  For pair tiles each lane handles keys j = lane8 + 8c; for
// d-vectors each lane handles groups of VW = min(4, d/8) consecutive coordinates,
// e = VW (lane8 + 8 g) + u.  Shared rows are padded to d + 4 floats, so the vector loads of the 8
// lanes of a row group fall in distinct 16-byte bank slots and every shared-memory operand is read
// VW values per instruction.  Row reductions are 3 xor shuffles; the per-row CG vectors live in
// registers.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "lla_internal.h"

namespace lla {
namespace {

constexpr int BQ = 32;
constexpr int BK = 32;
constexpr int NT = 256;
constexpr int JPT = BK / 8;  // keys per lane in a pair tile

// Row pitch of the shared tiles (floats) and the lane's vector width along the head dimension.
template <int D>
struct Lay {
    static constexpr int E = D / 8;               // coordinates per lane
    static constexpr int VW = E < 4 ? E : 4;      // consecutive coordinates per vector access
    static constexpr int LD = D + 4;              // padded pitch
    // coordinate of this lane's slot c
    static __device__ __forceinline__ int coord(int l8, int c) { return VW * (l8 + 8 * (c / VW)) + c % VW; }
};

template <int VW>
struct Vec;
template <>
struct Vec<4> {
    static __device__ __forceinline__ void ld(const float* p, float (&o)[4]) {
        const float4 t = *reinterpret_cast<const float4*>(p);
        o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
    }
};
template <>
struct Vec<2> {
    static __device__ __forceinline__ void ld(const float* p, float (&o)[2]) {
        const float2 t = *reinterpret_cast<const float2*>(p);
        o[0] = t.x; o[1] = t.y;
    }
};

__device__ __forceinline__ float ld_f(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float row_sum8(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}
__device__ __forceinline__ float row_max8(float v) {
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    return v;
}

template <int D>
struct Smem {
    static constexpr int LD = Lay<D>::LD;
    __align__(16) float q[BQ][LD];    // query rows
    __align__(16) float p[BQ][LD];    // second operand rows: CG direction p, then rho'
    __align__(16) float kb[BK][LD];   // key block
    __align__(16) float vb[BK][LD];   // value block (output sweep)
    float m[BQ][BK + 1];              // per-pair coefficients of the current block
};

// 8 consecutive elements of a row as fp32 (one 16-byte load for bf16, two for fp32).
__device__ __forceinline__ void ld8(const float* src, float (&o)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(src));
    const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void ld8(const __nv_bfloat16* src, float (&o)[8]) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(h[u]);
        o[2 * u] = f.x;
        o[2 * u + 1] = f.y;
    }
}

// Stage rows [row0, row0+rows) of a [n, D] slice into dst (zero beyond n), 8 elements per access.
template <int D, typename T>
__device__ __forceinline__ void load_rows(float (*dst)[Lay<D>::LD], const T* src, int row0, int rows, int n) {
    for (int idx = threadIdx.x; idx < rows * (D / 8); idx += NT) {
        const int r = idx / (D / 8), e = (idx - r * (D / 8)) * 8;
        const int g = row0 + r;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (g < n) ld8(src + (size_t)g * D + e, v);
        *reinterpret_cast<float4*>(&dst[r][e]) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(&dst[r][e + 4]) = make_float4(v[4], v[5], v[6], v[7]);
    }
}

// One BK-row block of a [n, D] slice held in registers (8 elements per group, PER groups per
// thread): loaded while the previous block is computed, stored to shared memory after it.  For
// d <= 32 the registers would cost the second resident CTA, so there the block is staged
// synchronously at store() (load() only records where it comes from).
template <int D, typename T, bool PF = (D >= 64)>
struct BlockPrefetch {
    static constexpr int G = BK * (D / 8);
    static constexpr int PER = (G + NT - 1) / NT;
    float v[PER][8];
    __device__ __forceinline__ void load(const T* src, int row0, int n) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int idx = threadIdx.x + u * NT;
            const int r = idx / (D / 8), e = (idx - r * (D / 8)) * 8;
            const int g = row0 + r;
#pragma unroll
            for (int t = 0; t < 8; ++t) v[u][t] = 0.f;
            if (idx < G && g < n) ld8(src + (size_t)g * D + e, v[u]);
        }
    }
    __device__ __forceinline__ void store(float (*dst)[Lay<D>::LD]) const {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int idx = threadIdx.x + u * NT;
            if (idx < G) {
                const int r = idx / (D / 8), e = (idx - r * (D / 8)) * 8;
                *reinterpret_cast<float4*>(&dst[r][e]) = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
                *reinterpret_cast<float4*>(&dst[r][e + 4]) = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
            }
        }
    }
};
template <int D, typename T>
struct BlockPrefetch<D, T, false> {
    const T* src_ = nullptr;
    int row0_ = 0, n_ = 0;
    __device__ __forceinline__ void load(const T* src, int row0, int n) { src_ = src; row0_ = row0; n_ = n; }
    __device__ __forceinline__ void store(float (*dst)[Lay<D>::LD]) const { load_rows<D>(dst, src_, row0_, BK, n_); }
};

// Pair tile: for this lane's keys j = lane8 + 8c, s[c] = q_r.k_j and a[c] = p_r.k_j.
template <int D, bool SECOND>
__device__ __forceinline__ void pair_tile(const Smem<D>& sm, int r, int l8, float (&s)[JPT], float (&a)[JPT]) {
    constexpr int VW = Lay<D>::VW;
#pragma unroll
    for (int c = 0; c < JPT; ++c) { s[c] = 0.f; a[c] = 0.f; }
#pragma unroll 2
    for (int e = 0; e < D; e += VW) {
        float qv[VW], pv[VW];
        Vec<VW>::ld(&sm.q[r][e], qv);
        if (SECOND) Vec<VW>::ld(&sm.p[r][e], pv);
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            float kv[VW];
            Vec<VW>::ld(&sm.kb[l8 + 8 * c][e], kv);
#pragma unroll
            for (int u = 0; u < VW; ++u) {
                s[c] = fmaf(qv[u], kv[u], s[c]);
                if (SECOND) a[c] = fmaf(pv[u], kv[u], a[c]);
            }
        }
    }
}

// acc[c] += sum_j m[r][j] * blk[j][e(c)] over this lane's coordinates.
template <int D>
__device__ __forceinline__ void accumulate_rows(const Smem<D>& sm, const float (*blk)[Lay<D>::LD], int r, int l8,
                                                float (&acc)[D / 8]) {
    constexpr int VW = Lay<D>::VW, E = D / 8;
#pragma unroll 4
    for (int j = 0; j < BK; ++j) {
        const float mj = sm.m[r][j];
#pragma unroll
        for (int g = 0; g < E / VW; ++g) {
            float bv[VW];
            Vec<VW>::ld(&blk[j][VW * (l8 + 8 * g)], bv);
#pragma unroll
            for (int u = 0; u < VW; ++u) acc[g * VW + u] = fmaf(mj, bv[u], acc[g * VW + u]);
        }
    }
}

template <int D, typename T>
__global__ void __launch_bounds__(NT, 1)
lla_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ out,
                float* __restrict__ rho, float* __restrict__ denom, int* __restrict__ cg_iters, int n, int n_tiles,
                float tau, float lambda, int cg_max_iters, float cg_tol, const float* __restrict__ probe) {
    constexpr int E = D / 8;  // coordinates per lane
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem<D>& sm = *reinterpret_cast<Smem<D>*>(smem_raw);

    int rank, head_i;
    causal_order(2 * (size_t)n * D * sizeof(T), rank, head_i);   // keys and values of a head
    const int tile = n_tiles - 1 - rank;
    const size_t head = (size_t)head_i;
    const T* qh = q + head * (size_t)n * D;
    const T* kh = k + head * (size_t)n * D;
    const T* vh = v + head * (size_t)n * D;

    const int tid = threadIdx.x;
    const int r = tid >> 3;      // row owned
    const int l8 = tid & 7;      // lane within the row group
    const int i0 = tile * BQ;
    const int i = i0 + r;        // query position of this row
    const bool row_ok = i < n;
    const int last_key = min(n - 1, i0 + BQ - 1);
    const int n_blocks = last_key / BK + 1;

    load_rows<D>(sm.q, qh, i0, BQ, n);

    // ---- (0) exact row maximum of the logits ---------------------------------------------
    BlockPrefetch<D, T> pk;
    float m_row = -INFINITY;
    pk.load(kh, 0, n);
    for (int kb = 0; kb < n_blocks; ++kb) {
        __syncthreads();
        pk.store(sm.kb);
        if (kb + 1 < n_blocks) pk.load(kh, (kb + 1) * BK, n);   // in flight while this block computes
        __syncthreads();
        float s[JPT], a[JPT];
        pair_tile<D, false>(sm, r, l8, s, a);
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            const int j = kb * BK + l8 + 8 * c;
            if (j <= i && row_ok) m_row = fmaxf(m_row, tau * s[c]);
        }
    }
    m_row = row_max8(m_row);

    // ---- (1) moments omega and mu~ ---------------------------------------------------------
    float acc[E];
#pragma unroll
    for (int c = 0; c < E; ++c) acc[c] = 0.f;
    float omega_part = 0.f;
    pk.load(kh, 0, n);
    for (int kb = 0; kb < n_blocks; ++kb) {
        __syncthreads();
        pk.store(sm.kb);
        if (kb + 1 < n_blocks) pk.load(kh, (kb + 1) * BK, n);
        __syncthreads();
        float s[JPT], a[JPT];
        pair_tile<D, false>(sm, r, l8, s, a);
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            const int j = kb * BK + l8 + 8 * c;
            const float w = (j <= i && row_ok) ? expf(tau * s[c] - m_row) : 0.f;
            omega_part += w;
            sm.m[r][l8 + 8 * c] = w;
        }
        __syncwarp();
        accumulate_rows<D>(sm, sm.kb, r, l8, acc);
    }
    const float omega_sum = row_sum8(omega_part);   // shuffles stay outside divergent code
    const float omega = row_ok ? omega_sum : 1.f;
    const float inv_omega = 1.f / omega;
    float kbar[E], delta[E];
#pragma unroll
    for (int c = 0; c < E; ++c) {
        kbar[c] = acc[c] * inv_omega;
        delta[c] = kbar[c] - sm.q[r][Lay<D>::coord(l8, c)];
    }

    // ---- (2) CG on (C/omega) rho' = delta ----------------------------------------------------
    float x[E], res[E], pv[E];
    float g = 0.f;
#pragma unroll
    for (int c = 0; c < E; ++c) {
        x[c] = 0.f;
        res[c] = row_ok ? delta[c] : 0.f;
        pv[c] = res[c];
        g = fmaf(res[c], res[c], g);
    }
    float gamma = row_sum8(g);
    const float rn0 = sqrtf(gamma);
    bool active = row_ok && gamma > 0.f && !(sqrtf(gamma) <= cg_tol * rn0);
    int iters = 0;
    const float lam_n = lambda * inv_omega;

    for (int it = 0; it < cg_max_iters; ++it) {
        if (!__syncthreads_or(active ? 1 : 0)) break;
#pragma unroll
        for (int c = 0; c < E; ++c) sm.p[r][Lay<D>::coord(l8, c)] = pv[c];
        float kp = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) kp = fmaf(kbar[c], pv[c], kp);
        kp = row_sum8(kp);
#pragma unroll
        for (int c = 0; c < E; ++c) acc[c] = 0.f;
        float msum_part = 0.f;
        pk.load(kh, 0, n);
        for (int kb = 0; kb < n_blocks; ++kb) {
            __syncthreads();
            pk.store(sm.kb);
            if (kb + 1 < n_blocks) pk.load(kh, (kb + 1) * BK, n);
            __syncthreads();
            float s[JPT], a[JPT];
            pair_tile<D, true>(sm, r, l8, s, a);
#pragma unroll
            for (int c = 0; c < JPT; ++c) {
                const int j = kb * BK + l8 + 8 * c;
                const float w = (j <= i && row_ok) ? expf(tau * s[c] - m_row) : 0.f;
                const float mm = w * (a[c] - kp);
                msum_part += mm;
                sm.m[r][l8 + 8 * c] = mm;
            }
            __syncwarp();
            accumulate_rows<D>(sm, sm.kb, r, l8, acc);
        }
        const float msum = row_sum8(msum_part);
        float cp[E];
        float pcp = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) {
            cp[c] = (acc[c] - kbar[c] * msum) * inv_omega + lam_n * pv[c];
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
            active = false;  // converged earlier, or no positive curvature left
        }
    }

    // ---- (3) finalise and output sweep ---------------------------------------------------------
    // Parallax form: no solve (cg_max_iters is 0); the caller's probe plays rho'
    if (probe) {
        const float* pr = probe + (head * (size_t)n + (row_ok ? i : 0)) * D;
#pragma unroll
        for (int c = 0; c < E; ++c) x[c] = row_ok ? pr[Lay<D>::coord(l8, c)] : 0.f;
    }
    float dx = 0.f, kx = 0.f;
#pragma unroll
    for (int c = 0; c < E; ++c) {
        dx = fmaf(delta[c], x[c], dx);
        kx = fmaf(kbar[c], x[c], kx);
    }
    dx = row_sum8(dx);
    kx = row_sum8(kx);
    __syncthreads();
#pragma unroll
    for (int c = 0; c < E; ++c) sm.p[r][Lay<D>::coord(l8, c)] = x[c];
#pragma unroll
    for (int c = 0; c < E; ++c) acc[c] = 0.f;
    float usum_part = 0.f;
    const float c1 = 1.f + kx;
    BlockPrefetch<D, T> pv_;
    pk.load(kh, 0, n);
    pv_.load(vh, 0, n);
    for (int kb = 0; kb < n_blocks; ++kb) {
        __syncthreads();
        pk.store(sm.kb);
        pv_.store(sm.vb);
        if (kb + 1 < n_blocks) {
            pk.load(kh, (kb + 1) * BK, n);
            pv_.load(vh, (kb + 1) * BK, n);
        }
        __syncthreads();
        float s[JPT], a[JPT];
        pair_tile<D, true>(sm, r, l8, s, a);
#pragma unroll
        for (int c = 0; c < JPT; ++c) {
            const int j = kb * BK + l8 + 8 * c;
            const float w = (j <= i && row_ok) ? expf(tau * s[c] - m_row) : 0.f;
            const float u = w * (c1 - a[c]);
            usum_part += u;
            sm.m[r][l8 + 8 * c] = u;
        }
        __syncwarp();
        accumulate_rows<D>(sm, sm.vb, r, l8, acc);
    }
    const float usum = row_sum8(usum_part);
    if (row_ok) {
        const size_t base = (head * (size_t)n + i) * D;
        const float inv_u = 1.f / usum;
        const float inv_g = 1.f / (1.f + dx);
#pragma unroll
        for (int c = 0; c < E; ++c) {
            const int e = Lay<D>::coord(l8, c);
            st_f(out + base + e, acc[c] * inv_u);
            if (!probe) rho[base + e] = x[c] * inv_g;
        }
        if (l8 == 0 && !probe) {
            denom[head * (size_t)n + i] = omega * inv_g;
            if (cg_iters) cg_iters[head * (size_t)n + i] = iters;
        }
    }
}

template <int D, typename T>
cudaError_t launch_typed(const Problem& p, cudaStream_t stream) {
    const int n_tiles = (p.n + BQ - 1) / BQ;
    const size_t smem = sizeof(Smem<D>);
    auto kern = lla_simt_kernel<D, T>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid(n_tiles, p.B * p.H);
    if (p.ev_main_begin && (err = cudaEventRecord(p.ev_main_begin, stream)) != cudaSuccess) return err;
    kern<<<grid, NT, smem, stream>>>(static_cast<const T*>(p.q), static_cast<const T*>(p.k),
                                     static_cast<const T*>(p.v), static_cast<T*>(p.out), p.rho, p.denom,
                                     p.cg_iters, p.n, n_tiles, p.tau, p.lambda, p.cg_max_iters, p.cg_tol, p.probe);
    err = cudaGetLastError();
    if (err == cudaSuccess && p.ev_main_end) err = cudaEventRecord(p.ev_main_end, stream);
    return err;
}

template <typename T>
cudaError_t launch_dim(const Problem& p, cudaStream_t stream) {
    switch (p.d) {
        case 16: return launch_typed<16, T>(p, stream);
        case 32: return launch_typed<32, T>(p, stream);
        case 64: return launch_typed<64, T>(p, stream);
        case 128: return launch_typed<128, T>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_simt(const Problem& p, cudaStream_t stream) {
    if (p.dtype == 1) return launch_dim<float>(p, stream);
    return launch_dim<__nv_bfloat16>(p, stream);
}

}  // namespace lla
