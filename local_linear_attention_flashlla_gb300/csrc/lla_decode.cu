// Decode step of causal LLA: one new query per (b, h) against its key/value cache.
//
// The query at position n-1 sees every cached key j <= n-1, so the step is row n-1 of the
// forward pass (Local Linear Attention reading notes, section 2.1, Eqs. (6)-(8); section 2.2:
// "a KV cache of size Theta(n d)").  Per (b, h) it runs the FlashLLA phases over the cache:
//   (1) one pass over K: logits s_j = tau q.k_j with an online maximum, the weights kept in
//       shared memory, omega = sum_j w_j and mu~ = sum_j w_j k_j (rescaled as the maximum grows);
//   (2) conjugate gradient on the centred system (C/omega) rho' = delta, delta = kbar - q, one
//       pass over K per iteration: a_j = p.k_j, M_j = w_j (a_j - kbar.p), Y = sum_j M_j k_j,
//       (C/omega) p = (Y - kbar sum_j M_j)/omega + (lambda/omega) p;
//   (3) rho = rho'/(1 + delta.rho'), denom = omega/(1 + delta.rho') and one pass over K and V:
//       out = sum_j u_j v_j / sum_j u_j, u_j = w_j (1 - (k_j - kbar).rho').
// Every product, sum and CG quantity is fp32.
//
// With one query row the work per key is two length-d dot/axpy products per pass: the step is
// bound by reading the cache (K once per pass, V once), so it runs on CUDA cores, not tensor
// cores.  Two forms: the streaming form below, and a cluster form (further down) that keeps
// K in the shared memory of an 8-CTA cluster.  Streaming form: one CTA of 256 threads per
// (b, h): 32 groups of 8 lanes; group g takes keys
// j = g, g+32, ...; lane l of a group holds coordinates l*D/8 .. l*D/8 + D/8-1, so a group reads
// a key row as one contiguous segment and reduces its dot products with 3 shuffles.  Weights
// live in shared memory (n floats).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <cooperative_groups.h>

#include "lla_internal.h"

namespace cg = cooperative_groups;

namespace lla {
namespace {

constexpr int DT = 256;              // threads per CTA
constexpr int kMaxDynSmem = 232448;  // dynamic shared memory a block may have (227 KB)
constexpr int NG = DT / 8;           // key groups

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// E = D/8 consecutive elements of a row (lane l of a group holds elements l*E .. l*E + E-1) as raw
// bits.  Every pass fetches several rows into these before using any of them, so each thread keeps
// that many loads in flight and works on independent rows: with one row at a time, two streaming
// CTAs per SM hold too few bytes in flight to cover the HBM latency, and a cluster CTA's pass over
// its shared-memory slice is one long dependent chain (load, dot, shuffles) per row.
template <int E, typename T>
struct RawSeg {
    static constexpr int W = E * (int)sizeof(T) / 4;   // 32-bit words: 1 .. 16
    uint32_t w[W];
};

// Rows fetched ahead per pass: about 128 bytes per thread, at most 8 rows.
template <int E, typename T>
__host__ __device__ constexpr int rows_ahead() {
    return E * (int)sizeof(T) >= 128 ? 1 : (128 / (E * (int)sizeof(T)) > 8 ? 8 : 128 / (E * (int)sizeof(T)));
}

// Load the segment at p (aligned to its size rounded down to a power of two, at most 16 bytes),
// or zeros when !valid (p is then not read).
template <int E, typename T>
__device__ __forceinline__ void fetch_seg(const T* p, bool valid, RawSeg<E, T>& r) {
    constexpr int W = RawSeg<E, T>::W;
    const uint32_t* s = reinterpret_cast<const uint32_t*>(p);
    if (!valid) {
#pragma unroll
        for (int c = 0; c < W; ++c) r.w[c] = 0u;
    } else if constexpr (W % 4 == 0) {
#pragma unroll
        for (int c = 0; c < W; c += 4) {
            const uint4 t = *reinterpret_cast<const uint4*>(s + c);
            r.w[c] = t.x; r.w[c + 1] = t.y; r.w[c + 2] = t.z; r.w[c + 3] = t.w;
        }
    } else if constexpr (W == 2) {
        const uint2 t = *reinterpret_cast<const uint2*>(s);
        r.w[0] = t.x; r.w[1] = t.y;
    } else {
        r.w[0] = *s;
    }
}

template <int E>
__device__ __forceinline__ void unpack_seg(const RawSeg<E, float>& r, float (&o)[E]) {
#pragma unroll
    for (int c = 0; c < E; ++c) o[c] = __uint_as_float(r.w[c]);
}
template <int E>
__device__ __forceinline__ void unpack_seg(const RawSeg<E, __nv_bfloat16>& r, float (&o)[E]) {
#pragma unroll
    for (int c = 0; c < E / 2; ++c) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.w[c]));
        o[2 * c] = f.x; o[2 * c + 1] = f.y;
    }
}

// x . segment, with two interleaved partial sums: half the dependent FMA chain of one running sum.
template <int E, typename T>
__device__ __forceinline__ float dot_seg(const float (&x)[E], const RawSeg<E, T>& r) {
    float kv[E];
    unpack_seg<E>(r, kv);
    float t0 = 0.f, t1 = 0.f;
#pragma unroll
    for (int c = 0; c < E; c += 2) {
        t0 = fmaf(x[c], kv[c], t0);
        t1 = fmaf(x[c + 1], kv[c + 1], t1);
    }
    return t0 + t1;
}

// x . segment as one running sum (the streaming form measured faster with it than with dot_seg;
// its passes are bound by memory, not by this chain).
template <int E, typename T>
__device__ __forceinline__ float dot_seg1(const float (&x)[E], const RawSeg<E, T>& r) {
    float kv[E];
    unpack_seg<E>(r, kv);
    float t = 0.f;
#pragma unroll
    for (int c = 0; c < E; ++c) t = fmaf(x[c], kv[c], t);
    return t;
}

// Store a fetched segment at p (the alignment fetch_seg needs).
template <int E, typename T>
__device__ __forceinline__ void store_seg(T* p, const RawSeg<E, T>& r) {
    constexpr int W = RawSeg<E, T>::W;
    uint32_t* d = reinterpret_cast<uint32_t*>(p);
    if constexpr (W % 4 == 0) {
#pragma unroll
        for (int c = 0; c < W; c += 4) *reinterpret_cast<uint4*>(d + c) = make_uint4(r.w[c], r.w[c + 1], r.w[c + 2], r.w[c + 3]);
    } else if constexpr (W == 2) {
        *reinterpret_cast<uint2*>(d) = make_uint2(r.w[0], r.w[1]);
    } else {
        d[0] = r.w[0];
    }
}

__device__ __forceinline__ float group_sum(float x) {   // over the 8 lanes of a group
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    return x;
}

template <int D>
struct DecSmem {
    float part[NG][D];      // per-group partial vectors (Y, mu~, O)
    float gs[NG][4];        // per-group partial scalars
    float q[D], kbar[D], delta[D], x[D], r[D], p[D], cp[D];
    float red[DT / 32][4];  // warp partials of block reductions
    float bc[8];            // broadcast scalars
};

// Sum of v over the block (every thread passes its value; every thread gets the total).
template <int D>
__device__ __forceinline__ float block_sum(DecSmem<D>& sm, float v, int slot) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5][slot] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < DT / 32; ++w) t += sm.red[w][slot];
    __syncthreads();
    return t;
}

// Column sums of part[NG][D] into dst[D] (thread t sums column t; D <= DT).
template <int D>
__device__ __forceinline__ void reduce_parts(DecSmem<D>& sm, float* dst) {
    __syncthreads();
    if (threadIdx.x < D) {
        float t = 0.f;
#pragma unroll 8
        for (int g = 0; g < NG; ++g) t += sm.part[g][threadIdx.x];
        dst[threadIdx.x] = t;
    }
    __syncthreads();
}

// Two CTAs per SM (at most 128 registers a thread): with the rows fetched ahead, two CTAs
// keep enough loads in flight, and the register cap keeps the prefetched rows from spilling.
__device__ __forceinline__ float warp_sum(float x) {
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// One CG step on the D-vector state in shared memory, by one warp (lane l: coordinates l, l+32,
// ...; the dot products are warp reductions, so no block barrier is needed inside the step):
//   cp = (Y - kbar msum)/omega + (lambda/omega) p,  alpha = gamma / p.cp,  x += alpha p,
//   r -= alpha cp,  gamma' = r.r,  p = r + (gamma'/gamma) p.
// y_of(c) gives coordinate c of Y.  Returns false, with nothing changed, when p.cp <= 0 (no
// positive curvature left); otherwise updates x, r, p and gamma.
template <int D, typename YF>
__device__ __forceinline__ bool cg_step_warp(DecSmem<D>& sm, YF y_of, float msum, float inv_om, float lam_n,
                                             float& gamma) {
    constexpr int NPL = (D + 31) / 32;
    const int lane = threadIdx.x & 31;
    float cpv[NPL];
    float pcp = 0.f;
#pragma unroll
    for (int u = 0; u < NPL; ++u) {
        const int c = lane + 32 * u;
        cpv[u] = 0.f;
        if (c < D) {
            cpv[u] = (y_of(c) - sm.kbar[c] * msum) * inv_om + lam_n * sm.p[c];
            pcp = fmaf(sm.p[c], cpv[u], pcp);
        }
    }
    pcp = warp_sum(pcp);
    if (!(pcp > 0.f)) return false;
    const float alpha = gamma / pcp;
    float g2 = 0.f;
#pragma unroll
    for (int u = 0; u < NPL; ++u) {
        const int c = lane + 32 * u;
        if (c < D) {
            sm.x[c] = fmaf(alpha, sm.p[c], sm.x[c]);
            const float rv = fmaf(-alpha, cpv[u], sm.r[c]);
            sm.r[c] = rv;
            g2 = fmaf(rv, rv, g2);
        }
    }
    g2 = warp_sum(g2);
    const float beta = g2 / gamma;
    gamma = g2;
#pragma unroll
    for (int u = 0; u < NPL; ++u) {
        const int c = lane + 32 * u;
        if (c < D) sm.p[c] = fmaf(beta, sm.p[c], sm.r[c]);
    }
    return true;
}

template <int D, typename T>
__global__ void __launch_bounds__(DT, 2)
lla_decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, T* __restrict__ out,
                  float* __restrict__ rho, float* __restrict__ denom, int* __restrict__ cg_iters, int n, int n_cap,
                  float tau, float lambda, int cg_max_iters, float cg_tol) {
    constexpr int E = D / 8;
    constexpr int U = rows_ahead<E, T>();           // K rows in flight per thread (moments, CG)
    constexpr int UO = U > 1 ? U / 2 : 1;           // K and V rows in flight (output)
    extern __shared__ __align__(16) unsigned char smem_raw[];
    DecSmem<D>& sm = *reinterpret_cast<DecSmem<D>*>(smem_raw);
    float* wts = reinterpret_cast<float*>(smem_raw + sizeof(DecSmem<D>));   // n weights

    const size_t head = blockIdx.x;
    const T* kh = k + head * (size_t)n_cap * D;
    const T* vh = v + head * (size_t)n_cap * D;
    const int tid = threadIdx.x, g = tid >> 3, l8 = tid & 7;
    const int c0 = l8 * E;                          // first coordinate of this lane

    if (tid < D) sm.q[tid] = ldf(q + head * D + tid);
    __syncthreads();
    float qv[E];
#pragma unroll
    for (int c = 0; c < E; ++c) qv[c] = sm.q[c0 + c];

    // ---- (1) logits, online maximum, omega and mu~ in one pass ----------------------------
    float mg = -INFINITY, og = 0.f, acc[E];
#pragma unroll
    for (int c = 0; c < E; ++c) acc[c] = 0.f;
    // Every group runs the same number of iterations (the shuffles inside need all 32 lanes of
    // the warp); a group whose key is past the end does no work in that iteration.  Group g takes
    // the keys j = it NG + g in increasing it, U of them per step, all U fetched first.
    const int n_it = (n + NG - 1) / NG;
    auto key_of = [&](int it) { return it * NG + g; };
    for (int it = 0; it < n_it; it += U) {
        RawSeg<E, T> kr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = key_of(it + u);
            fetch_seg<E>(kh + (size_t)(j < n ? j : 0) * D + c0, j < n, kr[u]);
        }
        float s[U];
#pragma unroll
        for (int u = 0; u < U; ++u) s[u] = dot_seg1<E>(qv, kr[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) s[u] = tau * group_sum(s[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = key_of(it + u);
            if (j >= n) continue;
            if (l8 == 0) wts[j] = s[u];             // logit for now; weight after the pass
            if (s[u] > mg) {                        // rescale this group's sums to the new maximum
                const float f = expf(mg - s[u]);
                og *= f;
#pragma unroll
                for (int c = 0; c < E; ++c) acc[c] *= f;
                mg = s[u];
            }
            const float w = expf(s[u] - mg);
            og += w;
            float kv[E];
            unpack_seg<E>(kr[u], kv);
#pragma unroll
            for (int c = 0; c < E; ++c) acc[c] = fmaf(w, kv[c], acc[c]);
        }
    }
    if (l8 == 0) sm.gs[g][0] = mg;
    __syncthreads();
    float m = -INFINITY;
#pragma unroll 8
    for (int t = 0; t < NG; ++t) m = fmaxf(m, sm.gs[t][0]);
    {
        const float f = (mg == -INFINITY) ? 0.f : expf(mg - m);   // groups that saw no key add 0
#pragma unroll
        for (int c = 0; c < E; ++c) sm.part[g][c0 + c] = acc[c] * f;
        if (l8 == 0) sm.gs[g][1] = og * f;
    }
    __syncthreads();
    for (int j = tid; j < n; j += DT) wts[j] = expf(wts[j] - m);
    float omega = 0.f;
#pragma unroll 8
    for (int t = 0; t < NG; ++t) omega += sm.gs[t][1];
    reduce_parts<D>(sm, sm.kbar);                   // mu~ for now
    const float inv_om = 1.f / omega;
    if (tid < D) {
        const float kb = sm.kbar[tid] * inv_om;
        sm.kbar[tid] = kb;
        sm.delta[tid] = kb - sm.q[tid];
        sm.x[tid] = 0.f;
        sm.r[tid] = sm.delta[tid];
        sm.p[tid] = sm.delta[tid];
    }
    __syncthreads();

    // ---- (2) CG on (C/omega) rho' = delta -------------------------------------------------------
    float gamma = block_sum<D>(sm, tid < D ? sm.r[tid] * sm.r[tid] : 0.f, 0);
    const float rn0 = sqrtf(gamma);
    bool active = gamma > 0.f && !(rn0 <= cg_tol * rn0);
    int iters = 0;
    const float lam_n = lambda * inv_om;
    for (int it = 0; it < cg_max_iters && active; ++it) {   // active is uniform over the block
        float pv[E];
#pragma unroll
        for (int c = 0; c < E; ++c) pv[c] = sm.p[c0 + c];
        float kp = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) kp = fmaf(sm.kbar[c0 + c], pv[c], kp);
        kp = group_sum(kp);
        float ms = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) acc[c] = 0.f;
        for (int it2 = 0; it2 < n_it; it2 += U) {
            RawSeg<E, T> kr[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = key_of(it2 + u);
                fetch_seg<E>(kh + (size_t)(j < n ? j : 0) * D + c0, j < n, kr[u]);
            }
            float a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) a[u] = dot_seg1<E>(pv, kr[u]);
#pragma unroll
            for (int u = 0; u < U; ++u) a[u] = group_sum(a[u]);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = key_of(it2 + u);
                if (j >= n) continue;
                const float mm = wts[j] * (a[u] - kp);
                ms += mm;
                float kv[E];
                unpack_seg<E>(kr[u], kv);
#pragma unroll
                for (int c = 0; c < E; ++c) acc[c] = fmaf(mm, kv[c], acc[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < E; ++c) sm.part[g][c0 + c] = acc[c];
        if (l8 == 0) sm.gs[g][2] = ms;
        reduce_parts<D>(sm, sm.cp);                 // Y
        // the CG step by warp 0, then one barrier that publishes p and the outcome
        if (tid < 32) {
            float msum = 0.f;
#pragma unroll 8
            for (int t = 0; t < NG; ++t) msum += sm.gs[t][2];
            const bool stepped = cg_step_warp<D>(sm, [&](int c) { return sm.cp[c]; }, msum, inv_om, lam_n, gamma);
            if (tid == 0) {
                sm.bc[0] = stepped ? 1.f : 0.f;
                sm.bc[1] = gamma;
            }
        }
        __syncthreads();
        if (sm.bc[0] == 0.f) break;                 // no positive curvature left (uniform)
        gamma = sm.bc[1];
        ++iters;
        if (gamma == 0.f || sqrtf(gamma) <= cg_tol * rn0) active = false;
    }

    // ---- (3) finalise and output pass -------------------------------------------------------------
    const float dx = block_sum<D>(sm, tid < D ? sm.delta[tid] * sm.x[tid] : 0.f, 0);
    const float kx = block_sum<D>(sm, tid < D ? sm.kbar[tid] * sm.x[tid] : 0.f, 1);
    float xv[E];
#pragma unroll
    for (int c = 0; c < E; ++c) xv[c] = sm.x[c0 + c];
    const float c1 = 1.f + kx;
    float us = 0.f;
#pragma unroll
    for (int c = 0; c < E; ++c) acc[c] = 0.f;
    for (int it = 0; it < n_it; it += UO) {
        RawSeg<E, T> kr[UO], vr[UO];
#pragma unroll
        for (int u = 0; u < UO; ++u) {
            const int j = key_of(it + u);
            const size_t off = (size_t)(j < n ? j : 0) * D + c0;
            fetch_seg<E>(kh + off, j < n, kr[u]);
            fetch_seg<E>(vh + off, j < n, vr[u]);
        }
        float t[UO];
#pragma unroll
        for (int u = 0; u < UO; ++u) t[u] = dot_seg1<E>(xv, kr[u]);
#pragma unroll
        for (int u = 0; u < UO; ++u) t[u] = group_sum(t[u]);
#pragma unroll
        for (int u = 0; u < UO; ++u) {
            const int j = key_of(it + u);
            if (j >= n) continue;
            const float uj = wts[j] * (c1 - t[u]);
            us += uj;
            float vv[E];
            unpack_seg<E>(vr[u], vv);
#pragma unroll
            for (int c = 0; c < E; ++c) acc[c] = fmaf(uj, vv[c], acc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < E; ++c) sm.part[g][c0 + c] = acc[c];
    if (l8 == 0) sm.gs[g][3] = us;
    reduce_parts<D>(sm, sm.cp);                     // O
    float usum = 0.f;
#pragma unroll 8
    for (int t = 0; t < NG; ++t) usum += sm.gs[t][3];
    if (tid < D) {
        const float inv_g = 1.f / (1.f + dx);
        stf(out + head * D + tid, sm.cp[tid] / usum);
        rho[head * D + tid] = sm.x[tid] * inv_g;
        if (tid == 0) {
            denom[head] = omega * inv_g;
            if (cg_iters) cg_iters[head] = iters;
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Cluster form: the cache of one (b, h) is split over the CL CTAs of a thread-block cluster, each
// holding its slice of K in shared memory for the whole step, so K is read from HBM once instead
// of once per pass.  Partial sums (the moments, each CG product, the output) are combined through
// distributed shared memory: every CTA writes its partial to a double-buffered exchange slot,
// the cluster synchronises once, and every CTA adds the CL slots in rank order, so all CTAs hold
// bitwise identical CG state and take the same branches without a broadcast.
constexpr int CL = 8;                // CTAs per cluster (portable cluster size)

template <int D>
struct ClSmem {
    DecSmem<D> base;
    float xbuf[2][D + 4];            // exchange slots: vector partial + up to 4 scalars
};

template <int D>
__host__ __device__ constexpr size_t cl_off_w() { return (sizeof(ClSmem<D>) + 15) & ~size_t(15); }

template <int D>
__device__ __forceinline__ void cl_combine(cg::cluster_group& cl, ClSmem<D>& sm, int slot, float* vec_out,
                                           float (&sc)[4]) {
    // all CTAs' slot `slot` is complete after this sync; the read happens before this CTA's next
    // arrival, which is what a peer's next write to the same slot waits for (two slots in turn)
    cl.sync();
    for (int c = threadIdx.x; c < D; c += DT) {
        float t = 0.f;
        for (int r = 0; r < CL; ++r) t += cl.map_shared_rank(&sm.xbuf[slot][0], r)[c];
        vec_out[c] = t;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        float t = 0.f;
        for (int r = 0; r < CL; ++r) t += cl.map_shared_rank(&sm.xbuf[slot][0], r)[D + u];
        sc[u] = t;
    }
    __syncthreads();
}

template <int D, typename T>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(DT, 1)
lla_decode_cluster_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                          T* __restrict__ out, float* __restrict__ rho, float* __restrict__ denom,
                          int* __restrict__ cg_iters, int n, int n_cap, int S, float tau, float lambda,
                          int cg_max_iters, float cg_tol) {
    constexpr int E = D / 8;
    cg::cluster_group cl = cg::this_cluster();
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ClSmem<D>& cs = *reinterpret_cast<ClSmem<D>*>(smem_raw);
    DecSmem<D>& sm = cs.base;
    float* wts = reinterpret_cast<float*>(smem_raw + cl_off_w<D>());              // S weights
    T* ks = reinterpret_cast<T*>(smem_raw + cl_off_w<D>() + (size_t)S * sizeof(float));   // S x D keys (S % 4 == 0)

    const int rank = (int)cl.block_rank();
    const size_t head = blockIdx.x / CL;
    const int j0 = rank * S;                                  // first key of this CTA's slice
    const int ns = max(0, min(S, n - j0));                    // keys in the slice
    const T* kh = k + head * (size_t)n_cap * D;
    const T* vh = v + head * (size_t)n_cap * D;
    const int tid = threadIdx.x, g = tid >> 3, l8 = tid & 7;
    const int c0 = l8 * E;
    const int n_it = (S + NG - 1) / NG;                       // same trip count in every group
    // rows fetched ahead per thread, as in the streaming form (K and V alike in the output pass)
    constexpr int U = rows_ahead<E, T>();
    constexpr int UO = U > 1 ? U / 2 : 1;
    auto key_of = [&](int it) { return it * NG + g; };

    if (tid < D) sm.q[tid] = ldf(q + head * D + tid);
    __syncthreads();
    float qv[E];
#pragma unroll
    for (int c = 0; c < E; ++c) qv[c] = sm.q[c0 + c];

    // ---- (1) slice: copy K to shared memory, logits, online maximum, omega and mu~ -------------
    float mg = -INFINITY, og = 0.f, acc[E];
#pragma unroll
    for (int c = 0; c < E; ++c) acc[c] = 0.f;
    for (int it = 0; it < n_it; it += U) {
        RawSeg<E, T> kr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jj = key_of(it + u);
            fetch_seg<E>(kh + (size_t)(j0 + (jj < ns ? jj : 0)) * D + c0, jj < ns, kr[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jj = key_of(it + u);
            if (jj < ns) store_seg<E>(ks + (size_t)jj * D + c0, kr[u]);
        }
        float sv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) sv[u] = dot_seg<E>(qv, kr[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) sv[u] = tau * group_sum(sv[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jj = key_of(it + u);
            if (jj >= ns) continue;
            if (l8 == 0) wts[jj] = sv[u];
            if (sv[u] > mg) {
                const float f = expf(mg - sv[u]);
                og *= f;
#pragma unroll
                for (int c = 0; c < E; ++c) acc[c] *= f;
                mg = sv[u];
            }
            const float w = expf(sv[u] - mg);
            og += w;
            float kv[E];
            unpack_seg<E>(kr[u], kv);
#pragma unroll
            for (int c = 0; c < E; ++c) acc[c] = fmaf(w, kv[c], acc[c]);
        }
    }
    if (l8 == 0) sm.gs[g][0] = mg;
    __syncthreads();
    float m_cta = -INFINITY;
#pragma unroll 8
    for (int t = 0; t < NG; ++t) m_cta = fmaxf(m_cta, sm.gs[t][0]);
    {
        const float f = (mg == -INFINITY) ? 0.f : expf(mg - m_cta);
#pragma unroll
        for (int c = 0; c < E; ++c) sm.part[g][c0 + c] = acc[c] * f;
        if (l8 == 0) sm.gs[g][1] = og * f;
    }
    reduce_parts<D>(sm, sm.cp);
    float om_cta = 0.f;
#pragma unroll 8
    for (int t = 0; t < NG; ++t) om_cta += sm.gs[t][1];
    // the cluster-wide maximum first (a max, so no rescaling order issue), then the sums
    if (tid == 0) cs.xbuf[0][D] = m_cta;
    cl.sync();
    float m = -INFINITY;
    for (int r = 0; r < CL; ++r) m = fmaxf(m, cl.map_shared_rank(&cs.xbuf[0][0], r)[D]);
    const float f_cta = (m_cta == -INFINITY) ? 0.f : expf(m_cta - m);
    cl.sync();                                                // everyone has read slot 0's maximum
    for (int c = tid; c < D; c += DT) cs.xbuf[0][c] = sm.cp[c] * f_cta;
    if (tid == 0) cs.xbuf[0][D] = om_cta * f_cta;
    for (int jj = tid; jj < ns; jj += DT) wts[jj] = expf(wts[jj] - m);
    float scal[4];
    cl_combine<D>(cl, cs, 0, sm.kbar, scal);                  // mu~ and omega
    const float omega = scal[0];
    const float inv_om = 1.f / omega;
    if (tid < D) {
        const float kb = sm.kbar[tid] * inv_om;
        sm.kbar[tid] = kb;
        sm.delta[tid] = kb - sm.q[tid];
        sm.x[tid] = 0.f;
        sm.r[tid] = sm.delta[tid];
        sm.p[tid] = sm.delta[tid];
    }
    __syncthreads();

    // ---- (2) CG; every CTA carries the same state --------------------------------------------------
    float gamma = block_sum<D>(sm, tid < D ? sm.r[tid] * sm.r[tid] : 0.f, 0);
    const float rn0 = sqrtf(gamma);
    bool active = gamma > 0.f && !(rn0 <= cg_tol * rn0);
    int iters = 0, slot = 1;
    const float lam_n = lambda * inv_om;
    float kbv[E];
#pragma unroll
    for (int c = 0; c < E; ++c) kbv[c] = sm.kbar[c0 + c];
    for (int it = 0; it < cg_max_iters && active; ++it) {
        float pv[E];
#pragma unroll
        for (int c = 0; c < E; ++c) pv[c] = sm.p[c0 + c];
        float kp = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) kp = fmaf(kbv[c], pv[c], kp);
        kp = group_sum(kp);
        float ms = 0.f;
#pragma unroll
        for (int c = 0; c < E; ++c) acc[c] = 0.f;
        for (int it2 = 0; it2 < n_it; it2 += U) {
            RawSeg<E, T> kr[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int jj = key_of(it2 + u);
                fetch_seg<E>(ks + (size_t)(jj < ns ? jj : 0) * D + c0, jj < ns, kr[u]);
            }
            float a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) a[u] = dot_seg<E>(pv, kr[u]);
#pragma unroll
            for (int u = 0; u < U; ++u) a[u] = group_sum(a[u]);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int jj = key_of(it2 + u);
                if (jj >= ns) continue;
                const float mm = wts[jj] * (a[u] - kp);
                ms += mm;
                float kv[E];
                unpack_seg<E>(kr[u], kv);
#pragma unroll
                for (int c = 0; c < E; ++c) acc[c] = fmaf(mm, kv[c], acc[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < E; ++c) sm.part[g][c0 + c] = acc[c];
        if (l8 == 0) sm.gs[g][2] = ms;
        __syncthreads();
        // this CTA's partial Y and msum straight into its exchange slot (groups summed in order)
        for (int c = tid; c < D; c += DT) {
            float t = 0.f;
#pragma unroll 8
            for (int q2 = 0; q2 < NG; ++q2) t += sm.part[q2][c];
            cs.xbuf[slot][c] = t;
        }
        if (tid == 0) {
            float t = 0.f;
#pragma unroll 8
            for (int q2 = 0; q2 < NG; ++q2) t += sm.gs[q2][2];
            cs.xbuf[slot][D] = t;
        }
        // every slot of the cluster is complete after this barrier; warp 0 reads them before this
        // CTA's next arrival, which a peer's next write to the same slot waits for (two slots in turn)
        cl.sync();
        if (tid < 32) {
            const float* xb[CL];
#pragma unroll
            for (int r = 0; r < CL; ++r) xb[r] = cl.map_shared_rank(&cs.xbuf[slot][0], r);
            float msum = 0.f;
#pragma unroll
            for (int r = 0; r < CL; ++r) msum += xb[r][D];
            auto y_of = [&](int c) {
                float t = 0.f;
#pragma unroll
                for (int r = 0; r < CL; ++r) t += xb[r][c];
                return t;
            };
            // the CG step on the cluster's sums, in rank order: identical in every CTA
            const bool stepped = cg_step_warp<D>(sm, y_of, msum, inv_om, lam_n, gamma);
            if (tid == 0) {
                sm.bc[0] = stepped ? 1.f : 0.f;
                sm.bc[1] = gamma;
            }
        }
        slot ^= 1;
        __syncthreads();
        if (sm.bc[0] == 0.f) break;
        gamma = sm.bc[1];
        ++iters;
        if (gamma == 0.f || sqrtf(gamma) <= cg_tol * rn0) active = false;
    }

    // ---- (3) finalise and output over the slice (K from shared memory, V streamed) ----------------
    const float dx = block_sum<D>(sm, tid < D ? sm.delta[tid] * sm.x[tid] : 0.f, 0);
    const float kx = block_sum<D>(sm, tid < D ? sm.kbar[tid] * sm.x[tid] : 0.f, 1);
    float xv[E];
#pragma unroll
    for (int c = 0; c < E; ++c) xv[c] = sm.x[c0 + c];
    const float c1 = 1.f + kx;
    float us = 0.f;
#pragma unroll
    for (int c = 0; c < E; ++c) acc[c] = 0.f;
    for (int it = 0; it < n_it; it += UO) {
        RawSeg<E, T> kr[UO], vr[UO];
#pragma unroll
        for (int u = 0; u < UO; ++u) {
            const int jj = key_of(it + u);
            const bool valid = jj < ns;
            fetch_seg<E>(ks + (size_t)(valid ? jj : 0) * D + c0, valid, kr[u]);
            fetch_seg<E>(vh + (size_t)(j0 + (valid ? jj : 0)) * D + c0, valid, vr[u]);
        }
        float t[UO];
#pragma unroll
        for (int u = 0; u < UO; ++u) t[u] = dot_seg<E>(xv, kr[u]);
#pragma unroll
        for (int u = 0; u < UO; ++u) t[u] = group_sum(t[u]);
#pragma unroll
        for (int u = 0; u < UO; ++u) {
            const int jj = key_of(it + u);
            if (jj >= ns) continue;
            const float uj = wts[jj] * (c1 - t[u]);
            us += uj;
            float vv[E];
            unpack_seg<E>(vr[u], vv);
#pragma unroll
            for (int c = 0; c < E; ++c) acc[c] = fmaf(uj, vv[c], acc[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < E; ++c) sm.part[g][c0 + c] = acc[c];
    if (l8 == 0) sm.gs[g][3] = us;
    reduce_parts<D>(sm, sm.cp);
    float us_cta = 0.f;
#pragma unroll 8
    for (int t = 0; t < NG; ++t) us_cta += sm.gs[t][3];
    for (int c = tid; c < D; c += DT) cs.xbuf[slot][c] = sm.cp[c];
    if (tid == 0) cs.xbuf[slot][D] = us_cta;
    cl_combine<D>(cl, cs, slot, sm.cp, scal);                // O and sum_j u_j over the cache
    if (rank == 0 && tid < D) {
        const float inv_g = 1.f / (1.f + dx);
        stf(out + head * D + tid, sm.cp[tid] / scal[0]);
        rho[head * D + tid] = sm.x[tid] * inv_g;
        if (tid == 0) {
            denom[head] = omega * inv_g;
            if (cg_iters) cg_iters[head] = iters;
        }
    }
    cl.sync();                       // no CTA leaves while a peer may still read its slots
}

template <int D, typename T>
cudaError_t launch_dec(const DecodeProblem& p, cudaStream_t stream) {
    const size_t smem = sizeof(DecSmem<D>) + (size_t)p.n * sizeof(float);
    auto kern = lla_decode_kernel<D, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (p.ev_main_begin && (e = cudaEventRecord(p.ev_main_begin, stream)) != cudaSuccess) return e;
    kern<<<p.B * p.H, DT, smem, stream>>>(static_cast<const T*>(p.q), static_cast<const T*>(p.k),
                                          static_cast<const T*>(p.v), static_cast<T*>(p.out), p.rho, p.denom,
                                          p.cg_iters, p.n, p.n_cap, p.tau, p.lambda, p.cg_max_iters, p.cg_tol);
    e = cudaGetLastError();
    if (e == cudaSuccess && p.ev_main_end) e = cudaEventRecord(p.ev_main_end, stream);
    return e;
}

// Keys per CTA of the cluster form (a multiple of 4, so the key slice stays 16-byte aligned).
inline int cl_slice(int n) { return ((n + CL - 1) / CL + 3) & ~3; }

template <int D, typename T>
size_t cl_smem_bytes(int n) {
    const size_t S = (size_t)cl_slice(n);
    return cl_off_w<D>() + S * sizeof(float) + S * D * sizeof(T);
}

template <int D, typename T>
cudaError_t launch_dec_cluster(const DecodeProblem& p, cudaStream_t stream) {
    const int S = cl_slice(p.n);
    const size_t smem = cl_smem_bytes<D, T>(p.n);
    auto kern = lla_decode_cluster_kernel<D, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (p.ev_main_begin && (e = cudaEventRecord(p.ev_main_begin, stream)) != cudaSuccess) return e;
    kern<<<p.B * p.H * CL, DT, smem, stream>>>(static_cast<const T*>(p.q), static_cast<const T*>(p.k),
                                               static_cast<const T*>(p.v), static_cast<T*>(p.out), p.rho, p.denom,
                                               p.cg_iters, p.n, p.n_cap, S, p.tau, p.lambda, p.cg_max_iters,
                                               p.cg_tol);
    e = cudaGetLastError();
    if (e == cudaSuccess && p.ev_main_end) e = cudaEventRecord(p.ev_main_end, stream);
    return e;
}

// The cluster form reads K from HBM once but pays a cluster-wide exchange per pass; the streaming
// form re-reads K every pass but keeps every SM busy with whole heads.  Measured on GB300 (bf16,
// n = 4096, d = 128, 16 CG iterations), cluster vs streaming: 16 heads 0.17 vs 0.43 ms, 32 heads
// 0.26 vs 0.44 ms, 48 heads 0.34 vs 0.44 ms, 64 heads 0.43 vs 0.44 ms, 128 heads 0.75 vs 0.67 ms.
// The cluster form wins while there are too few heads to fill the GPU, up to about 64 heads.
constexpr long long kClusterMaxHeads = 64;

template <int D, typename T>
cudaError_t launch_dec_pick(const DecodeProblem& p, cudaStream_t stream) {
    const bool fits = cl_smem_bytes<D, T>(p.n) <= (size_t)kMaxDynSmem;
    if (p.form == kDecodeCluster) return fits ? launch_dec_cluster<D, T>(p, stream) : cudaErrorInvalidValue;
    if (p.form != kDecodeStream && fits && (long long)p.B * p.H <= kClusterMaxHeads)
        return launch_dec_cluster<D, T>(p, stream);
    return launch_dec<D, T>(p, stream);
}

template <typename T>
cudaError_t launch_dec_dim(const DecodeProblem& p, cudaStream_t stream) {
    switch (p.d) {
        case 16: return launch_dec_pick<16, T>(p, stream);
        case 32: return launch_dec_pick<32, T>(p, stream);
        case 64: return launch_dec_pick<64, T>(p, stream);
        case 128: return launch_dec_pick<128, T>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t decode_smem_bytes(int n, int d) {
    size_t base = 0;
    switch (d) {
        case 16: base = sizeof(DecSmem<16>); break;
        case 32: base = sizeof(DecSmem<32>); break;
        case 64: base = sizeof(DecSmem<64>); break;
        default: base = sizeof(DecSmem<128>); break;
    }
    return base + (size_t)n * sizeof(float);
}

template <typename T>
size_t cl_smem_dim(int n, int d) {
    switch (d) {
        case 16: return cl_smem_bytes<16, T>(n);
        case 32: return cl_smem_bytes<32, T>(n);
        case 64: return cl_smem_bytes<64, T>(n);
        default: return cl_smem_bytes<128, T>(n);
    }
}

bool decode_cluster_fits(int n, int d, int dtype) {
    const size_t b = dtype == 1 ? cl_smem_dim<float>(n, d) : cl_smem_dim<__nv_bfloat16>(n, d);
    return b <= (size_t)kMaxDynSmem;
}

cudaError_t launch_decode(const DecodeProblem& p, cudaStream_t stream) {
    if (p.form == kDecodeMoment) return launch_decode_moment(p, stream);
    if (p.dtype == 1) return launch_dec_dim<float>(p, stream);
    return launch_dec_dim<__nv_bfloat16>(p, stream);
}

}  // namespace lla
