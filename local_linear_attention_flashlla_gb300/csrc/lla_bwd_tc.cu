// tcgen05 dq and dk/dv stages of the LLA backward pass (tensor path, bf16 inputs, d in {64, 128}).
//
// For a block of 128 keys j (one CTA, MMA M = 128) and every step of 32 queries i >= j (MMA N / K =
// 32), the per-pair quantities of the backward (Local Linear Attention reading notes, section
// 2.1, Eqs. (6)-(8), differentiated in centred form; the formulas are in lla_backward.cu):
//   products (SS, fp16 operands, fp32 in TMEM):  S = K Q^T,  A1 = K (R'_hi + R'_lo)^T,
//            A2 = K (Y_hi + Y_lo)^T,  H = V G^T
//   coefficients (elementwise warps, fp32):  cq = tau (ds - max path), cw = wbar Ahat,
//            cr = -wbar Bhat, stored back into the product columns as fp16 hi + lo pairs
//   sums (TS, coefficients from TMEM):  dK += Cq Q - Cw (Y_hi + Y_lo) + Cr (R'_hi + R'_lo),
//            dV += Cw G, accumulated in TMEM over all query steps and read once at the end.
// q, k, v and dout are the stats stage's fp16 copies (exact for bf16 inputs, per-tensor power-of
// -two scales); rho' = rho omega/denom and y are split into fp16 hi + lo pairs (about 22 bits) at
// per-tensor scales by the prep kernels here.  Each key row's coefficients are scaled by a power
// of two fixed from that row's largest coefficient, which the dq kernel (below) records while it
// forms the same coefficients; the row's sums are unscaled once.  With hi + lo coefficients and
// operands every product keeps about 22 bits, so the stage is as accurate as fp32 arithmetic.
//
// Roles (320 threads): warps 0-7 elementwise (thread = key row, half of the 32 queries), warp 8
// lane 0 TMA (K, V once; the six query-side tiles of each step into two stages), warp 9 lane 0
// MMA issue (and the TMEM allocation).  TMEM: two product buffers of 4 x 32 columns, dK and dV
// accumulators of d columns each.  Every mbarrier wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "lla_internal.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace lla {
namespace {
using namespace tc;

constexpr int KB = 128;       // keys per CTA (MMA M)
constexpr int QS = 32;        // queries per step (N of the products, K of the sums)
constexpr int NTH = 320;
constexpr int NEW = 256;      // elementwise threads
constexpr int NTILE = 6;      // q, g, rh, rl, yh, yl

size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

// exponent s with x 2^s <= 2^14 (0 for x == 0): the rule of the stats stage's operand copies
__device__ __forceinline__ int sc_exp(float m) {
    if (!(m > 0.f)) return 0;
    int e;
    const float f = frexpf(m, &e);
    const int cl = f == 0.5f ? e - 1 : e;
    const int s = 14 - cl;
    return s < -100 ? -100 : (s > 100 ? 100 : s);
}

// ---- prep: max |rho'| and max |y|, then their fp16 hi + lo copies ------------------------------
template <int D>
__global__ void lla_bwd_rymax_kernel(const float* __restrict__ rho, const BwdRowRec* __restrict__ rec,
                                     const float* __restrict__ y, size_t rows, unsigned* hdr) {
    float mr = 0.f, my = 0.f;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < rows * D;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t r = idx / D;
        mr = fmaxf(mr, fabsf(__ldg(rho + idx) * __ldg(&rec[r].rp_scale)));
        my = fmaxf(my, fabsf(__ldg(y + idx)));
    }
    for (int o = 16; o; o >>= 1) {
        mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
        my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, o));
    }
    if ((threadIdx.x & 31) == 0) {
        atomicMax(&hdr[0], __float_as_uint(mr));
        atomicMax(&hdr[1], __float_as_uint(my));
    }
}

template <int D>
__global__ void lla_bwd_ry16_kernel(const float* __restrict__ rho, const BwdRowRec* __restrict__ rec,
                                    const float* __restrict__ y, size_t rows, const unsigned* __restrict__ hdr,
                                    __half* rh, __half* rl, __half* yh, __half* yl) {
    const float sr = pow2i(sc_exp(__uint_as_float(hdr[0]))), sy = pow2i(sc_exp(__uint_as_float(hdr[1])));
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < rows * D;
         idx += (size_t)gridDim.x * blockDim.x) {
        const size_t r = idx / D;
        const float x = __ldg(rho + idx) * __ldg(&rec[r].rp_scale) * sr;
        const __half xh = __float2half_rn(x);
        rh[idx] = xh;
        rl[idx] = __float2half_rn(x - __half2float(xh));
        const float z = __ldg(y + idx) * sy;
        const __half zh = __float2half_rn(z);
        yh[idx] = zh;
        yl[idx] = __float2half_rn(z - __half2float(zh));
    }
}

// ---- the dk/dv kernel -----------------------------------------------------------------------------
// Stages of the query-side ring: each step's six tiles (48 KB at d = 128) come from L2, and two
// stages left the products waiting on their loads.
constexpr int KV_STAGES = 3;

template <int D>
struct KvSmem {
    static constexpr int KT = KB * D * 2;     // [128 x D] fp16, SW128 boxes of 64 columns
    static constexpr int QT = QS * D * 2;     // [32 x D] fp16
    unsigned char k[KT];
    unsigned char v[KT];
    unsigned char st[KV_STAGES][NTILE][QT];   // stages of q, g, rh, rl, yh, yl
    BwdRowRec rec[KV_STAGES][QS];             // and the step's per-query records
    uint64_t kv_full, st_full[KV_STAGES], st_empty[KV_STAGES], prod_full[2], coef_ready[2], acc_free[2], acc_done;
    uint32_t tmem_base;
    int err;
};
static_assert(sizeof(KvSmem<128>) <= 232448, "shared memory layout too large");

struct KvParams {
    const BwdRowRec* rec;
    const unsigned* kmax;     // [B*H*n][2] float bits
    const unsigned* maxabs;   // q, k, v, dout
    const unsigned* ry;       // rho', y; word 2 is the abort flag
    float* dk;
    float* dv;
    unsigned* dev_err;
    int n;
    float tau;
};

// S-type product: D[tmem, 128 x 32] (+)= A[128 x D] B[32 x D]^T, both K-major SW128.
template <int D>
__device__ __forceinline__ void gemm_prod(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, bool acc) {
    constexpr uint32_t ID = idesc_f16(KB, QS, false);
    const uint64_t a0 = sdesc_sw128(a_addr, 16, 1024), b0 = sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t ao = (uint64_t)((((ks >> 2) * (KB * 128)) + (ks & 3) * 32) >> 4);
        const uint64_t bo = (uint64_t)((((ks >> 2) * (QS * 128)) + (ks & 3) * 32) >> 4);
        if (ks == 0 && !acc) umma_ss_c<false>(d_tmem, a0 + ao, b0 + bo, ID);
        else umma_ss_c<true>(d_tmem, a0 + ao, b0 + bo, ID);
    }
}
// Sum: D[tmem, 128 x D] (+)= C[tmem, 128 x 32] B[32 x D], B read MN-major.  The coefficients of
// query step k (16 queries) sit at c_tmem + 16k: hi pairs at +0..7, lo pairs at +8..15.
template <int D>
__device__ __forceinline__ void gemm_sum(uint32_t d_tmem, uint32_t c_tmem, uint32_t b_addr, bool acc) {
    constexpr uint32_t ID = idesc_f16(KB, D, true);
    const uint64_t b0 = sdesc_sw128(b_addr, QS * 128, 1024);
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < QS / 16; ++ks) {
            const uint64_t bk = b0 + (uint64_t)((ks * 2048) >> 4);
            if (part == 0 && ks == 0 && !acc) umma_ts_c<false>(d_tmem, c_tmem + 16 * ks + 8 * part, bk, ID);
            else umma_ts_c<true>(d_tmem, c_tmem + 16 * ks + 8 * part, bk, ID);
        }
}

// Plain bulk copy global -> shared (16-byte aligned, bytes a multiple of 16) on an mbarrier.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 2000000000ull) return;
}

template <int D>
__global__ void __launch_bounds__(NTH, 1)
lla_bwd_kv_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g,
                     const __grid_constant__ CUtensorMap tm_rh, const __grid_constant__ CUtensorMap tm_rl,
                     const __grid_constant__ CUtensorMap tm_yh, const __grid_constant__ CUtensorMap tm_yl,
                     const KvParams prm) {
    using S = KvSmem<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(prm.dev_err, (unsigned)kDevErrSmemAlign);
        return;
    }
    S& s = *reinterpret_cast<S*>(smem_raw);
    volatile int* err = &s.err;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(const_cast<unsigned*>(prm.ry) + 2);
#define WAIT(bar, par) mbar_wait_abortable(bar, par, err, abort_flag)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = prm.n;
    int rank, head;                                // the earliest keys have the longest query range
    causal_order((size_t)6 * n * D, rank, head);   // fp16 queries, upstream gradients and rho' of a head
    const int j0 = rank * KB;
    const int nst = (n - j0 + QS - 1) / QS;        // query steps i0 = j0 + QS t, t < nst

    if (tid == 0) {
        s.err = *abort_flag ? 1 : 0;
        mbar_init(&s.kv_full, 1);
        for (int i = 0; i < KV_STAGES; ++i) {
            mbar_init(&s.st_full[i], 1);
            mbar_init(&s.st_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.prod_full[i], 1);
            mbar_init(&s.coef_ready[i], NEW / 32);
            mbar_init(&s.acc_free[i], 1);
        }
        mbar_init(&s.acc_done, 1);
        mbar_fence_init();
    }
    if (warp == 9) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tP = s.tmem_base, tDK = s.tmem_base + 256, tDV = s.tmem_base + 256 + D;

    if (warp == 8) {
        // ================================ TMA producer ================================
        if (lane == 0) {
            const CUtensorMap* maps[NTILE] = {&tm_q, &tm_g, &tm_rh, &tm_rl, &tm_yh, &tm_yl};
            mbar_arrive_expect_tx(&s.kv_full, 2 * S::KT);
            for (int bx = 0; bx < D / 64; ++bx) {
                tma_load_3d(s.k + bx * KB * 128, &tm_k, &s.kv_full, bx * 64, j0, head);
                tma_load_3d(s.v + bx * KB * 128, &tm_v, &s.kv_full, bx * 64, j0, head);
            }
            for (int t = 0; t < nst && !*err; ++t) {
                const int st = t % KV_STAGES, f = t / KV_STAGES;
                if (f >= 1 && !WAIT(&s.st_empty[st], (f - 1) & 1)) break;
                const int i0 = j0 + QS * t;
                const uint32_t rbytes = (uint32_t)(min(QS, n - i0) * sizeof(BwdRowRec));   // rows past n: not read
                mbar_arrive_expect_tx(&s.st_full[st], NTILE * S::QT + rbytes);
                for (int m = 0; m < NTILE; ++m)
                    for (int bx = 0; bx < D / 64; ++bx)
                        tma_load_3d(s.st[st][m] + bx * QS * 128, maps[m], &s.st_full[st], bx * 64, i0, head);
                bulk_load(s.rec[st], prm.rec + (size_t)head * n + i0, rbytes, &s.st_full[st]);
            }
            for (int t = nst > KV_STAGES ? nst - KV_STAGES : 0; t < nst; ++t)
                drain(&s.st_full[t % KV_STAGES], (t / KV_STAGES) & 1);
            drain(&s.kv_full, 0);
        }
    } else if (warp == 9) {
        // ================================= MMA issuer =================================
        if (lane == 0) {
            const uint32_t ka = smem_u32(s.k), va = smem_u32(s.v);
            bool ok = WAIT(&s.kv_full, 0);
            for (int t = 0; t <= nst && ok; ++t) {
                if (t < nst) {   // products of step t into buffer t & 1
                    const int st = t % KV_STAGES, pb = t & 1;
                    if (!(ok = WAIT(&s.st_full[st], (t / KV_STAGES) & 1))) break;
                    // the buffer's coefficients of step t - 2 were read by that step's sums
                    if (t >= 2 && !(ok = WAIT(&s.acc_free[pb], ((t - 2) >> 1) & 1))) break;
                    tc_fence_after();
                    const uint32_t base = tP + pb * 128;
                    gemm_prod<D>(base, ka, smem_u32(s.st[st][0]), false);            // S = K Q^T
                    gemm_prod<D>(base + 32, ka, smem_u32(s.st[st][2]), false);       // A1 = K R'^T
                    gemm_prod<D>(base + 32, ka, smem_u32(s.st[st][3]), true);
                    gemm_prod<D>(base + 64, ka, smem_u32(s.st[st][4]), false);       // A2 = K Y^T
                    gemm_prod<D>(base + 64, ka, smem_u32(s.st[st][5]), true);
                    gemm_prod<D>(base + 96, va, smem_u32(s.st[st][1]), false);       // H = V G^T
                    umma_commit(&s.prod_full[pb]);
                }
                if (t >= 1) {    // sums of step t - 1
                    const int u = t - 1, st = u % KV_STAGES, pb = u & 1;
                    if (!(ok = WAIT(&s.coef_ready[pb], (u >> 1) & 1))) break;
                    tc_fence_after();
                    const uint32_t base = tP + pb * 128;
                    const bool acc = u > 0;
                    gemm_sum<D>(tDK, base, smem_u32(s.st[st][0]), acc);              // Cq Q
                    gemm_sum<D>(tDK, base + 64, smem_u32(s.st[st][4]), true);        // Cy Y (Cy = -cw)
                    gemm_sum<D>(tDK, base + 64, smem_u32(s.st[st][5]), true);
                    gemm_sum<D>(tDK, base + 32, smem_u32(s.st[st][2]), true);        // Cr R'
                    gemm_sum<D>(tDK, base + 32, smem_u32(s.st[st][3]), true);
                    gemm_sum<D>(tDV, base + 96, smem_u32(s.st[st][1]), acc);         // Cv G
                    umma_commit(&s.st_empty[st]);
                    umma_commit(&s.acc_free[pb]);
                }
            }
            umma_commit(&s.acc_done);
            drain(&s.acc_done, 0);
        }
    } else {
        // ============================ elementwise warps ============================
        const int quad = warp & 3, half = warp >> 2;
        const int row = quad * 32 + lane;
        const int j = j0 + row;
        const bool key_ok = j < n;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int eq = sc_exp(__uint_as_float(prm.maxabs[0])), ek = sc_exp(__uint_as_float(prm.maxabs[1]));
        const int ev = sc_exp(__uint_as_float(prm.maxabs[2])), eg = sc_exp(__uint_as_float(prm.maxabs[3]));
        const int er = sc_exp(__uint_as_float(prm.ry[0])), ey = sc_exp(__uint_as_float(prm.ry[1]));
        const size_t kidx = ((size_t)head * n + (key_ok ? j : 0)) * 2;
        const int sK = key_ok ? sc_exp(__uint_as_float(prm.kmax[kidx]) * 1.01f) : 0;
        const int sV = key_ok ? sc_exp(__uint_as_float(prm.kmax[kidx + 1]) * 1.01f) : 0;
        const float tau = prm.tau;
        const float fs = tau * pow2i(-(eq + ek)), f1 = pow2i(-(ek + er)), f2 = pow2i(-(ek + ey)), fh = pow2i(-(ev + eg));
        const float fs2 = fs * 1.4426950408889634f;      // the logits' scale in log2 units (weights via ex2)
        const float gq = pow2i(sK - eq), gy = -pow2i(sK - ey), gr = pow2i(sK - er), gv = pow2i(sV - eg);
        bool ok = true;
        for (int t = 0; t < nst; ++t) {
            const int pb = t & 1;
            ok = ok && WAIT(&s.prod_full[pb], (t >> 1) & 1);
            tc_fence_after();
            const uint32_t base = tP + pb * 128 + lane_off + 16 * half;
            float sv[16], a1[16], a2[16], hv[16];
            tmem_ld16(base, sv);
            tmem_ld16(base + 32, a1);
            tmem_ld16(base + 64, a2);
            tmem_ld16(base + 96, hv);
            tmem_ld_wait();
            uint32_t cq[16], cr[16], cy[16], cv[16];       // hi pairs in 0..7, lo pairs in 8..15
            const int ib = j0 + QS * t + 16 * half;
#pragma unroll
            for (int qq = 0; qq < 16; qq += 2) {
                float vq[2], vy[2], vr[2], vv[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int i = ib + qq + w;
                    const bool valid = key_ok && i < n && j <= i;
                    float c_q = 0.f, c_w = 0.f, c_r = 0.f;
                    if (valid) {
                        const float4* rp = reinterpret_cast<const float4*>(&s.rec[t % KV_STAGES][16 * half + qq + w]);
                        const float4 r0 = rp[0], r1 = rp[1];
                        // r0 = (m, jm, inv_omega, hbar), r1 = (kb_rp, kb_y, sd, rp_scale)
                        const float wb = ex2(fmaf(sv[qq + w], fs2, -r0.x * 1.4426950408889634f)) * r0.z;
                        const float Ah = 1.f - fmaf(a1[qq + w], f1, -r1.x);
                        const float Bh = fmaf(hv[qq + w], fh, -r0.w) - fmaf(a2[qq + w], f2, -r1.y);
                        const float ds = wb * Ah * Bh;
                        c_q = tau * (ds - (j == __float_as_int(r0.y) ? r1.z : 0.f));
                        c_w = wb * Ah;
                        c_r = -wb * Bh;
                    }
                    vq[w] = c_q * gq;
                    vy[w] = c_w * gy;
                    vr[w] = c_r * gr;
                    vv[w] = c_w * gv;
                }
                const int pidx = qq >> 1;
#define LLA_SPLIT(ARR, X)                                                                             \
                {                                                                                     \
                    ARR[pidx] = pack_half2(X[0], X[1]);                                               \
                    const float2 h_ = __half22float2(*reinterpret_cast<const __half2*>(&ARR[pidx]));   \
                    ARR[8 + pidx] = pack_half2(X[0] - h_.x, X[1] - h_.y);                             \
                }
                LLA_SPLIT(cq, vq)
                LLA_SPLIT(cy, vy)
                LLA_SPLIT(cr, vr)
                LLA_SPLIT(cv, vv)
#undef LLA_SPLIT
            }
            tmem_st16(base, cq);
            tmem_st16(base + 32, cr);
            tmem_st16(base + 64, cy);
            tmem_st16(base + 96, cv);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.coef_ready[pb]);
        }
        ok = ok && WAIT(&s.acc_done, 0);
        tc_fence_after();
        const float uk = pow2i(-sK), uv = pow2i(-sV);
        const size_t obase = ((size_t)head * n + (key_ok ? j : 0)) * D + half * (D / 2);
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) {
            float a[32], b[32];
            tmem_ld32(tDK + lane_off + half * (D / 2) + c, a);
            tmem_ld32(tDV + lane_off + half * (D / 2) + c, b);
            tmem_ld_wait();
            if (key_ok && ok) {
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    *reinterpret_cast<float4*>(prm.dk + obase + c + e) =
                        make_float4(a[e] * uk, a[e + 1] * uk, a[e + 2] * uk, a[e + 3] * uk);
                    *reinterpret_cast<float4*>(prm.dv + obase + c + e) =
                        make_float4(b[e] * uv, b[e + 1] * uv, b[e + 2] * uv, b[e + 3] * uv);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) {
        __syncwarp();
        tmem_dealloc(s.tmem_base, 512);
    }
    if (tid == 0 && s.err) atomicOr(prm.dev_err, (unsigned)kDevErrMbarTimeout);
#undef WAIT
}

// ---- the dq kernel ----------------------------------------------------------------------------------
// For a tile of 128 queries (M = 128) and every step of 32 keys j up to the tile's last query, the
// same four products with the roles of the two sides exchanged (S = Q K^T, A1 = R' K^T, A2 = Y K^T,
// H = G V^T, the query-side tiles resident), the coefficient ds of every pair, and
// dq_i += sum_j ds_ij k_j by a TS product into one of two TMEM partial-sum buffers.  A row's
// coefficients of one step share a power-of-two scale fixed from their maximum; the elementwise
// warps read each step's partial sums back, unscale them and add them in registers.  The kernel
// also records, per key, the largest coefficient of the dk and dv sums (kmax, scaled units of the
// dk/dv kernel).  At the end dq_i = tau (sum - sd_i k_jm) + y_i.
template <int D>
struct DqSmem {
    static constexpr int RT = KB * D * 2;     // [128 x D] fp16 resident tile
    static constexpr int ST = QS * D * 2;     // [32 x D] fp16 key-step tile
    unsigned char res[NTILE][RT];             // q, g, rh, rl, yh, yl of the query tile
    unsigned char st[2][2][ST];               // two stages of k, v
    uint64_t res_full, st_full[2], st_empty[2], prod_full[2], coef_ready[2], acc_free[2], sum_full[2], dq_free[2];
    unsigned kmx[2][QS][2];                   // per key of a step: largest dk / dv coefficient (float bits)
    float xch[2][2][KB];                      // row maxima of the two halves (two steps in turn)
    uint32_t tmem_base;
    int err;
};
static_assert(sizeof(DqSmem<128>) <= 232448, "shared memory layout too large");

struct DqParams {
    const BwdRowRec* rec;
    const __nv_bfloat16* k;    // the bf16 keys (dq's path through the row maximum)
    const float* y;            // [B*H*n][D]
    float* dq;
    unsigned* kmax;
    const unsigned* maxabs;
    const unsigned* ry;
    unsigned* dev_err;
    int n, n_tiles;
    float tau;
};

template <int D>
__global__ void __launch_bounds__(NTH, 1)
lla_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g,
                     const __grid_constant__ CUtensorMap tm_rh, const __grid_constant__ CUtensorMap tm_rl,
                     const __grid_constant__ CUtensorMap tm_yh, const __grid_constant__ CUtensorMap tm_yl,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const DqParams prm) {
    using S = DqSmem<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(prm.dev_err, (unsigned)kDevErrSmemAlign);
        return;
    }
    S& s = *reinterpret_cast<S*>(smem_raw);
    volatile int* err = &s.err;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(const_cast<unsigned*>(prm.ry) + 2);
#define WAIT(bar, par) mbar_wait_abortable(bar, par, err, abort_flag)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = prm.n;
    int rank, head;
    causal_order((size_t)4 * n * D, rank, head);                // fp16 keys and values of a head
    const int i0 = (prm.n_tiles - 1 - rank) * KB;
    const int last = min(n - 1, i0 + KB - 1);
    const int nst = last / QS + 1;                              // key steps j0 = QS t

    if (tid == 0) {
        s.err = *abort_flag ? 1 : 0;
        mbar_init(&s.res_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.st_full[i], 1);
            mbar_init(&s.st_empty[i], 1);
            mbar_init(&s.prod_full[i], 1);
            mbar_init(&s.coef_ready[i], NEW / 32);
            mbar_init(&s.acc_free[i], 1);
            mbar_init(&s.sum_full[i], 1);
            mbar_init(&s.dq_free[i], NEW / 32);
        }
        mbar_fence_init();
    }
    if (tid < 2 * QS * 2) (&s.kmx[0][0][0])[tid] = 0u;
    if (warp == 9) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tP = s.tmem_base, tQ = s.tmem_base + 256;   // two product buffers, two dq buffers

    if (warp == 8) {
        // ================================ TMA producer ================================
        if (lane == 0) {
            const CUtensorMap* maps[NTILE] = {&tm_q, &tm_g, &tm_rh, &tm_rl, &tm_yh, &tm_yl};
            mbar_arrive_expect_tx(&s.res_full, NTILE * S::RT);
            for (int m = 0; m < NTILE; ++m)
                for (int bx = 0; bx < D / 64; ++bx) tma_load_3d(s.res[m] + bx * KB * 128, maps[m], &s.res_full, bx * 64, i0, head);
            for (int t = 0; t < nst && !*err; ++t) {
                const int st = t & 1, f = t >> 1;
                if (f >= 1 && !WAIT(&s.st_empty[st], (f - 1) & 1)) break;
                mbar_arrive_expect_tx(&s.st_full[st], 2 * S::ST);
                for (int bx = 0; bx < D / 64; ++bx) {
                    tma_load_3d(s.st[st][0] + bx * QS * 128, &tm_k, &s.st_full[st], bx * 64, QS * t, head);
                    tma_load_3d(s.st[st][1] + bx * QS * 128, &tm_v, &s.st_full[st], bx * 64, QS * t, head);
                }
            }
            for (int t = nst > 2 ? nst - 2 : 0; t < nst; ++t) drain(&s.st_full[t & 1], (t >> 1) & 1);
            drain(&s.res_full, 0);
        }
    } else if (warp == 9) {
        // ================================= MMA issuer =================================
        if (lane == 0) {
            const uint32_t qa = smem_u32(s.res[0]), ga = smem_u32(s.res[1]);
            const uint32_t rha = smem_u32(s.res[2]), rla = smem_u32(s.res[3]);
            const uint32_t yha = smem_u32(s.res[4]), yla = smem_u32(s.res[5]);
            bool ok = WAIT(&s.res_full, 0);
            for (int t = 0; t <= nst && ok; ++t) {
                if (t < nst) {   // products of key step t into buffer t & 1
                    const int st = t & 1, pb = t & 1;
                    if (!(ok = WAIT(&s.st_full[st], (t >> 1) & 1))) break;
                    if (t >= 2 && !(ok = WAIT(&s.acc_free[pb], ((t - 2) >> 1) & 1))) break;
                    tc_fence_after();
                    const uint32_t base = tP + pb * 128, ka = smem_u32(s.st[st][0]), va = smem_u32(s.st[st][1]);
                    gemm_prod<D>(base, qa, ka, false);          // S = Q K^T
                    gemm_prod<D>(base + 32, rha, ka, false);    // A1 = R' K^T
                    gemm_prod<D>(base + 32, rla, ka, true);
                    gemm_prod<D>(base + 64, yha, ka, false);    // A2 = Y K^T
                    gemm_prod<D>(base + 64, yla, ka, true);
                    gemm_prod<D>(base + 96, ga, va, false);     // H = G V^T
                    umma_commit(&s.prod_full[pb]);
                }
                if (t >= 1) {    // partial dq of step t - 1
                    const int u = t - 1, st = u & 1, pb = u & 1;
                    if (!(ok = WAIT(&s.coef_ready[pb], (u >> 1) & 1))) break;
                    if (u >= 2 && !(ok = WAIT(&s.dq_free[pb], ((u - 2) >> 1) & 1))) break;
                    tc_fence_after();
                    gemm_sum<D>(tQ + pb * D, tP + pb * 128, smem_u32(s.st[st][0]), false);   // ds K
                    umma_commit(&s.sum_full[pb]);
                    umma_commit(&s.st_empty[st]);
                    umma_commit(&s.acc_free[pb]);
                }
            }
            for (int u = nst > 2 ? nst - 2 : 0; u < nst; ++u) drain(&s.sum_full[u & 1], (u >> 1) & 1);
        }
    } else {
        // ============================ elementwise warps ============================
        const int quad = warp & 3, half = warp >> 2;
        const int row = quad * 32 + lane;
        const int i = i0 + row;
        const bool row_ok = i < n;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int eq = sc_exp(__uint_as_float(prm.maxabs[0])), ek = sc_exp(__uint_as_float(prm.maxabs[1]));
        const int ev = sc_exp(__uint_as_float(prm.maxabs[2])), eg = sc_exp(__uint_as_float(prm.maxabs[3]));
        const int er = sc_exp(__uint_as_float(prm.ry[0])), ey = sc_exp(__uint_as_float(prm.ry[1]));
        const float tau = prm.tau;
        const float fs = tau * pow2i(-(eq + ek)), f1 = pow2i(-(ek + er)), f2 = pow2i(-(ek + ey)), fh = pow2i(-(ev + eg));
        const float fs2 = fs * 1.4426950408889634f;      // the logits' scale in log2 units (weights via ex2)
        const float gq = pow2i(-eq), gy = pow2i(-ey), gr = pow2i(-er), gvv = pow2i(-eg), gk = pow2i(-ek);
        BwdRowRec R{};
        if (row_ok) R = prm.rec[(size_t)head * n + i];
        const float m2 = R.m * 1.4426950408889634f;     // the row maximum in log2 units
        float acc[D / 2];
#pragma unroll
        for (int e = 0; e < D / 2; ++e) acc[e] = 0.f;
        float usc[2] = {1.f, 1.f};     // the unscale factors of the two partial-sum buffers
        bool ok = true;
        for (int t = 0; t <= nst; ++t) {
            if (t < nst) {
                const int pb = t & 1;
                ok = ok && WAIT(&s.prod_full[pb], (t >> 1) & 1);
                tc_fence_after();
                const uint32_t base = tP + pb * 128 + lane_off + 16 * half;
                float sv[16], a1[16], a2[16], hv[16];
                tmem_ld16(base, sv);
                tmem_ld16(base + 32, a1);
                tmem_ld16(base + 64, a2);
                tmem_ld16(base + 96, hv);
                tmem_ld_wait();
                const int jb = QS * t + 16 * half;
                float dsv[16];
                float mx = 0.f;
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = jb + jj;
                    const bool valid = row_ok && j <= i;
                    float ds = 0.f, mk = 0.f, mv = 0.f;
                    if (valid) {
                        const float wb = ex2(fmaf(sv[jj], fs2, -m2)) * R.inv_omega;
                        const float Ah = 1.f - fmaf(a1[jj], f1, -R.kb_rp);
                        const float Bh = fmaf(hv[jj], fh, -R.hbar) - fmaf(a2[jj], f2, -R.kb_y);
                        ds = wb * Ah * Bh;
                        const float cq = tau * (ds - (j == R.jm ? R.sd : 0.f));
                        const float cw = wb * Ah, cr = -wb * Bh;
                        mk = fmaxf(fabsf(cq) * gq, fmaxf(fabsf(cw) * gy, fabsf(cr) * gr));
                        mv = fabsf(cw) * gvv;
                    }
                    dsv[jj] = ds * gk;             // the k copy's scale folded in
                    mx = fmaxf(mx, fabsf(dsv[jj]));
                    // largest coefficient of key j over the warp's 32 query rows (non-negative floats
                    // order as their bit patterns)
                    const unsigned wk = __reduce_max_sync(0xffffffffu, __float_as_uint(mk));
                    const unsigned wv = __reduce_max_sync(0xffffffffu, __float_as_uint(mv));
                    if (lane == 0 && (wk | wv)) {
                        atomicMax(&s.kmx[t & 1][16 * half + jj][0], wk);
                        atomicMax(&s.kmx[t & 1][16 * half + jj][1], wv);
                    }
                }
                // the row's scale for this step: both halves' maxima
                // (buffer t & 1: a thread rewrites it at step t + 2, after the next barrier, which its
                // partner reaches only after reading this step's value)
                s.xch[t & 1][half][row] = mx;
                named_bar_sync(1, NEW);
                const float rmx = fmaxf(mx, s.xch[t & 1][1 - half][row]);
                const int sq = sc_exp(rmx * 1.01f);
                const float up = pow2i(sq);
                usc[pb] = pow2i(-sq);
                uint32_t pk[16];
#pragma unroll
                for (int jj = 0; jj < 16; jj += 2) {
                    const float x0 = dsv[jj] * up, x1 = dsv[jj + 1] * up;
                    pk[jj >> 1] = pack_half2(x0, x1);
                    const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&pk[jj >> 1]));
                    pk[8 + (jj >> 1)] = pack_half2(x0 - h.x, x1 - h.y);
                }
                tmem_st16(base, pk);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.coef_ready[pb]);
                // every warp's key maxima of this step are in: push them (two threads per key)
                if (tid < 2 * QS) {
                    const int j = QS * t + (tid >> 1);
                    unsigned* slot = &s.kmx[t & 1][tid >> 1][tid & 1];
                    if (j < n && *slot) atomicMax(prm.kmax + ((size_t)head * n + j) * 2 + (tid & 1), *slot);
                    *slot = 0u;
                }
            }
            if (t >= 1) {    // add step t - 1's partial sums
                const int u = t - 1, pb = u & 1;
                ok = ok && WAIT(&s.sum_full[pb], (u >> 1) & 1);
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 2; c += 32) {
                    float v[32];
                    tmem_ld32(tQ + pb * D + lane_off + half * (D / 2) + c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) acc[c + e] = fmaf(v[e], usc[pb], acc[c + e]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.dq_free[pb]);
            }
        }
        if (row_ok && ok) {
            const size_t rb = ((size_t)head * n + i) * D + half * (D / 2);
            const __nv_bfloat16* kjm = prm.k + ((size_t)head * n + R.jm) * D + half * (D / 2);
#pragma unroll
            for (int e = 0; e < D / 2; e += 4) {
                float o[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    o[u] = fmaf(tau, acc[e + u] - R.sd * __bfloat162float(kjm[e + u]), __ldg(prm.y + rb + e + u));
                *reinterpret_cast<float4*>(prm.dq + rb + e) = make_float4(o[0], o[1], o[2], o[3]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) {
        __syncwarp();
        tmem_dealloc(s.tmem_base, 512);
    }
    if (tid == 0 && s.err) atomicOr(prm.dev_err, (unsigned)kDevErrMbarTimeout);
#undef WAIT
}

template <int D>
cudaError_t launch_dq_d(const BackwardProblem& p, const BwdRowRec* rec, const float* yvec, const TensorOperands& ops,
                        const KvScratch& kv, cudaStream_t stream, const char** why) {
    const uint64_t slices = (uint64_t)p.B * p.H;
    CUtensorMap tq, tg, trh, trl, tyh, tyl, tk, tv;
    if (!make_tmap_f16_3d(&tq, ops.q16, D, p.n, slices, KB) || !make_tmap_f16_3d(&tg, ops.g16, D, p.n, slices, KB) ||
        !make_tmap_f16_3d(&trh, kv.rh, D, p.n, slices, KB) || !make_tmap_f16_3d(&trl, kv.rl, D, p.n, slices, KB) ||
        !make_tmap_f16_3d(&tyh, kv.yh, D, p.n, slices, KB) || !make_tmap_f16_3d(&tyl, kv.yl, D, p.n, slices, KB) ||
        !make_tmap_f16_3d(&tk, ops.k16, D, p.n, slices, QS) || !make_tmap_f16_3d(&tv, ops.v16, D, p.n, slices, QS)) {
        *why = "cuTensorMapEncodeTiled (dq)";
        return cudaErrorInvalidValue;
    }
    DqParams prm;
    prm.rec = rec;
    prm.k = static_cast<const __nv_bfloat16*>(p.k);
    prm.y = yvec;
    prm.dq = p.dq;
    prm.kmax = kv.kmax;
    prm.maxabs = ops.maxabs;
    prm.ry = kv.hdr;
    prm.dev_err = device_error_word();
    prm.n = p.n;
    prm.n_tiles = (p.n + KB - 1) / KB;
    prm.tau = p.tau;
    if (!prm.dev_err) { *why = "device error word"; return cudaErrorInvalidSymbol; }
    const size_t smem = sizeof(DqSmem<D>);
    auto kern = lla_bwd_dq_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) { *why = "dq kernel shared-memory attribute"; return e; }
    kern<<<dim3(prm.n_tiles, (unsigned)slices), NTH, smem, stream>>>(tq, tg, trh, trl, tyh, tyl, tk, tv, prm);
    e = cudaGetLastError();
    if (e != cudaSuccess) *why = "dq kernel launch";
    return e;
}

template <int D>
cudaError_t launch_kv_d(const BackwardProblem& p, const BwdRowRec* rec, const TensorOperands& ops,
                        const KvScratch& kv, cudaStream_t stream, const char** why) {
    const uint64_t slices = (uint64_t)p.B * p.H;
    CUtensorMap tk, tv, tq, tg, trh, trl, tyh, tyl;
    if (!make_tmap_f16_3d(&tk, ops.k16, D, p.n, slices, KB) || !make_tmap_f16_3d(&tv, ops.v16, D, p.n, slices, KB) ||
        !make_tmap_f16_3d(&tq, ops.q16, D, p.n, slices, QS) || !make_tmap_f16_3d(&tg, ops.g16, D, p.n, slices, QS) ||
        !make_tmap_f16_3d(&trh, kv.rh, D, p.n, slices, QS) || !make_tmap_f16_3d(&trl, kv.rl, D, p.n, slices, QS) ||
        !make_tmap_f16_3d(&tyh, kv.yh, D, p.n, slices, QS) || !make_tmap_f16_3d(&tyl, kv.yl, D, p.n, slices, QS)) {
        *why = "cuTensorMapEncodeTiled (dk/dv)";
        return cudaErrorInvalidValue;
    }
    KvParams prm;
    prm.rec = rec;
    prm.kmax = kv.kmax;
    prm.maxabs = ops.maxabs;
    prm.ry = kv.hdr;
    prm.dk = p.dk;
    prm.dv = p.dv;
    prm.dev_err = device_error_word();
    prm.n = p.n;
    prm.tau = p.tau;
    if (!prm.dev_err) { *why = "device error word"; return cudaErrorInvalidSymbol; }
    const size_t smem = sizeof(KvSmem<D>);
    auto kern = lla_bwd_kv_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) { *why = "dk/dv kernel shared-memory attribute"; return e; }
    kern<<<dim3((p.n + KB - 1) / KB, (unsigned)slices), NTH, smem, stream>>>(tk, tv, tq, tg, trh, trl, tyh, tyl, prm);
    e = cudaGetLastError();
    if (e != cudaSuccess) *why = "dk/dv kernel launch";
    return e;
}

}  // namespace

size_t tensor_kv_bytes(int B, int H, int n, int d) {
    const size_t N = (size_t)B * H * n * d, rows = (size_t)B * H * n;
    return 256 + 4 * a256(N * 2) + a256(rows * 8);
}

KvScratch tensor_kv_scratch(void* ws, int B, int H, int n, int d) {
    const size_t N = (size_t)B * H * n * d;
    unsigned char* base = static_cast<unsigned char*>(ws);
    KvScratch k;
    k.hdr = reinterpret_cast<unsigned*>(base);
    size_t off = 256;
    k.rh = base + off; off += a256(N * 2);
    k.rl = base + off; off += a256(N * 2);
    k.yh = base + off; off += a256(N * 2);
    k.yl = base + off; off += a256(N * 2);
    k.kmax = reinterpret_cast<unsigned*>(base + off);
    return k;
}

cudaError_t launch_tensor_kv_prep(const BackwardProblem& p, const BwdRowRec* rec, const float* yvec,
                                  const KvScratch& kv, cudaStream_t stream) {
    const size_t rows = (size_t)p.B * p.H * p.n;
    cudaError_t e = cudaMemsetAsync(kv.hdr, 0, 256, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(kv.kmax, 0, rows * 8, stream);
    if (e != cudaSuccess) return e;
    const size_t total = rows * p.d;
    const int blocks = (int)((total + 255) / 256 < 152 * 8 ? (total + 255) / 256 : 152 * 8);
    __half *rh = static_cast<__half*>(kv.rh), *rl = static_cast<__half*>(kv.rl);
    __half *yh = static_cast<__half*>(kv.yh), *yl = static_cast<__half*>(kv.yl);
    if (p.d == 128) {
        lla_bwd_rymax_kernel<128><<<blocks, 256, 0, stream>>>(p.rho, rec, yvec, rows, kv.hdr);
        lla_bwd_ry16_kernel<128><<<blocks, 256, 0, stream>>>(p.rho, rec, yvec, rows, kv.hdr, rh, rl, yh, yl);
    } else {
        lla_bwd_rymax_kernel<64><<<blocks, 256, 0, stream>>>(p.rho, rec, yvec, rows, kv.hdr);
        lla_bwd_ry16_kernel<64><<<blocks, 256, 0, stream>>>(p.rho, rec, yvec, rows, kv.hdr, rh, rl, yh, yl);
    }
    return cudaGetLastError();
}

cudaError_t launch_tensor_dq(const BackwardProblem& p, const BwdRowRec* rec, const float* yvec,
                             const TensorOperands& ops, const KvScratch& kv, cudaStream_t stream, const char** why) {
    if (p.d == 128) return launch_dq_d<128>(p, rec, yvec, ops, kv, stream, why);
    if (p.d == 64) return launch_dq_d<64>(p, rec, yvec, ops, kv, stream, why);
    *why = "tensor path supports d in {64, 128}";
    return cudaErrorInvalidValue;
}

cudaError_t launch_tensor_kv(const BackwardProblem& p, const BwdRowRec* rec, const TensorOperands& ops,
                             const KvScratch& kv, cudaStream_t stream, const char** why) {
    if (p.d == 128) return launch_kv_d<128>(p, rec, ops, kv, stream, why);
    if (p.d == 64) return launch_kv_d<64>(p, rec, ops, kv, stream, why);
    *why = "tensor path supports d in {64, 128}";
    return cudaErrorInvalidValue;
}

}  // namespace lla
