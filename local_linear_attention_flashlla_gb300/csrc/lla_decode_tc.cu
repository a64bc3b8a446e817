// Decode step of causal LLA, moment form on tcgen05 (bf16 caches, d = 128).
//
// The step is row n-1 of the forward pass (Local Linear Attention reading notes, section 2.1,
// Eqs. (6)-(8)): one query against the whole cache.  Its linear system is only d x d,
//     (C/omega + lambda/omega I) rho' = delta,   C = sum_j w_j (k_j - kbar)(k_j - kbar)^T,
// so instead of applying C to each CG direction with a pass over the cache (the CUDA-core forms
// in lla_decode.cu read K T+2 times), this form reads K twice and V once:
//   pass 1 (K): the logits s_j = tau q.k_j, their maximum m, omega = sum_j w_j and kbar =
//       sum_j w_j k_j / omega with w_j = exp(s_j - m) (an online maximum per thread, combined at
//       the end of the pass);
//   pass 2 (K, V): the centred moments, on the tensor cores,
//       Cc = sum_j w_j (k_j - kbar) k_j^T,   Hc = sum_j w_j (k_j - kbar) v_j^T     (d x d, fp32 in TMEM),
//       and, on CUDA cores, r = sum_j w_j (k_j - kbar) (zero in real arithmetic, kept so that the
//       rounding of kbar cancels) and nu = sum_j w_j v_j;
// then the same centred CG on the d x d moments:  C p = Cc p - r (kbar.p), and with x = rho',
// u_j = w_j (1 - (k_j - kbar).x):  sum_j u_j v_j = nu - Hc^T x,  sum_j u_j = omega - r.x.
// These are identities of real arithmetic, so the result is the CUDA-core forms' result up to
// rounding.  Centring every key against the exact kbar before the products keeps that rounding
// first order in |k|/spread(k), as in the CUDA-core forms; moments about any other point would
// cancel at second order when the keys share a large common component.
//
// Products: per chunk of 64 keys, D[128 x 256] += A^T [K | V], A = w o (K - kbar) (key row j
// scaled by w_j) as three bf16 terms hi + mid + lo (24 bits: the fp32 value), K and V the cache's
// own bf16 values (exact), fp32 accumulation: the sums keep fp32 accuracy.  Both operands are
// MN-major, keys as rows: the elementwise warps write A in the 128-byte-swizzle layout in which
// TMA delivers K and V.
//
// Roles (512 threads, one CTA per SM; a CTA takes heads blockIdx.x, blockIdx.x + gridDim.x, ...):
//   warp 0, lane 0   TMA: chunks of 128 keys of K (pass 1) and of 64 keys of K and V (pass 2), a
//                    32 KB stage each, into a 3-stage ring; rows past n read as zeros;
//   warp 1, lane 0   MMA issue (warp 1 owns TMEM: two 256-column accumulators, heads in turn);
//                    every chunk of either pass is handed back through it, in order;
//   warps 4-11       elementwise, 4 threads per key row (32 coordinates each): logits, weights,
//                    omega and kbar (pass 1); the three terms of A, r and nu (pass 2);
//   warps 12-15      the head's epilogue, thread = row of D: CG on the moments and the output,
//                    overlapped with the next head's passes.
// setmaxnreg gives the elementwise warpgroups 184 registers a thread (48 to the first warpgroup,
// 96 to the epilogue's: 48 + 2 x 184 + 96 = 4 x 128, the launch's share).
// Every mbarrier wait is bounded; a CTA whose pipeline broke drains and reports through the
// library's device error word.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "lla_internal.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace lla {
namespace {
using namespace tc;

constexpr int DM = 128;               // head dim: the MMA's M
constexpr int CK = 64;                // keys per chunk
constexpr int NSTAGE = 3;             // K/V chunk ring
constexpr int NTERM = 3;              // bf16 terms of w o K
constexpr int NEW = 256;              // elementwise threads
constexpr int NEP = 128;              // epilogue threads
constexpr int NTH = 128 + NEW + NEP;  // warpgroups: TMA/MMA, elementwise x 2, epilogue
constexpr int BOX = CK * 128;         // bytes of a [64 keys x 64 coordinates] bf16 box
// registers a thread after setmaxnreg: TMA/MMA warpgroup, each elementwise warpgroup, epilogue
constexpr int REG_IO = 48, REG_EW = 184, REG_EP = 96, REG_LAUNCH = 65536 / NTH;
static_assert(128 * (REG_IO + 2 * REG_EW + REG_EP) == REG_LAUNCH * NTH,
              "the split must hand out exactly the registers the block was launched with");

struct MomSmem {
    unsigned char kv[NSTAGE][4][BOX];     // K cols 0-63, K cols 64-127, V cols 0-63, V cols 64-127
    unsigned char a[2][NTERM][2][BOX];    // the terms of w o (K - kbar) (2 boxes each), chunks in turn
    float r[2][8][DM];                    // per elementwise warp: r and nu (heads in turn)
    float nu[2][8][DM];
    float kb[2][DM];                      // kbar, omega and the maximum (heads in turn)
    float om[2], mx[2];
    float p1[8][DM];                      // pass 1: per-warp sums of w_j k_j against the warp's maximum
    float p1s[8][2];                      //         the warp's maximum and omega
    float p[DM];                          // epilogue: the CG direction
    float red[4][4][4];                   // epilogue: reductions (slots in turn x warps x values)
    float hx[4][DM];                      // epilogue: per-warp column sums of Hc^T x
    uint64_t st_full[NSTAGE], st_empty[NSTAGE], a_full[2], a_free[2], d_full[2], mom_full[2], acc_free[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int err;
};
static_assert(sizeof(MomSmem) <= 232448, "shared memory layout too large");

struct MomParams {
    const __nv_bfloat16* q;   // [heads][128]
    __nv_bfloat16* out;       // [heads][128]
    float* rho;               // [heads][128]
    float* denom;             // [heads]
    int* cg_iters;            // [heads] or null
    unsigned* dev_err;
    int nheads, n, cg_max_iters;
    float tau, lambda, cg_tol;
};

// tma_load_3d with an L2 cache policy (from createpolicy) for the loaded lines.
__device__ __forceinline__ void tma_load_3d_hint(void* smem_dst, const void* tmap, uint64_t* bar, int x, int y, int z,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;"
        ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z),
          "l"(policy)
        : "memory");
}
// L2 policies for all of an access's lines: keep them (a later pass reads them again) or let them
// go first (last use).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 2000000000ull) return;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t bf_pack(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// x0, x1 -> three packed bf16 pairs whose sum is x (to 2^-24 relative): hi, then the rounded
// remainders.  Each subtraction is exact in fp32.
__device__ __forceinline__ void split3(float x0, float x1, uint32_t& h, uint32_t& m, uint32_t& l) {
    h = bf_pack(x0, x1);
    const float r0 = x0 - bf_lo(h), r1 = x1 - bf_hi(h);
    m = bf_pack(r0, r1);
    l = bf_pack(r0 - bf_lo(m), r1 - bf_hi(m));
}

__global__ void __launch_bounds__(NTH, 1)
lla_decode_mom_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const MomParams prm) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(prm.dev_err, (unsigned)kDevErrSmemAlign);
        return;
    }
    MomSmem& s = *reinterpret_cast<MomSmem*>(smem_raw);
    volatile int* err = &s.err;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch1 = (prm.n + 2 * CK - 1) / (2 * CK);      // pass-1 chunks (128 keys of K)
    const int nch = (prm.n + CK - 1) / CK;                 // pass-2 chunks (64 keys of K and V)
    const int nloc = (prm.nheads - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;   // grid <= heads

    if (tid == 0) {
        s.err = 0;
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&s.st_full[i], 1);
            mbar_init(&s.st_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.a_full[i], NEW / 32);
            mbar_init(&s.a_free[i], 1);
            mbar_init(&s.d_full[i], 1);
            mbar_init(&s.mom_full[i], NEW / 32);
            mbar_init(&s.acc_free[i], NEP / 32);
        }
        mbar_init(&s.mma_done, 1);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;

    // each role's code is dominated by its own setmaxnreg, so it is compiled to that budget
    if (warp < 4) {
        setmaxnreg_dec<REG_IO>();
        if (warp == 0 && lane == 0) {
            // ================================ TMA producer ================================
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            // pass 1's K is read again by pass 2: keep it in L2; pass 2's K and V are last uses
            const uint64_t keep = l2_policy_evict_last(), last = l2_policy_evict_first();
            int g = 0;
            bool ok = true;
            for (int hl = 0; hl < nloc && ok; ++hl) {
                const int head = (int)blockIdx.x + hl * (int)gridDim.x;
                for (int c2 = 0; c2 < nch1 + nch; ++c2) {
                    const int st = g % NSTAGE, f = g / NSTAGE;
                    if (f >= 1 && !(ok = mbar_wait(&s.st_empty[st], (f - 1) & 1, err))) break;
                    mbar_arrive_expect_tx(&s.st_full[st], 4 * BOX);
                    for (int bx = 0; bx < 2; ++bx) {
                        if (c2 < nch1) {   // K rows y .. y+63 into boxes 0, 1 and y+64 .. y+127 into 2, 3
                            tma_load_3d_hint(s.kv[st][bx], &tm_k, &s.st_full[st], bx * 64, c2 * 2 * CK, head, keep);
                            tma_load_3d_hint(s.kv[st][2 + bx], &tm_k, &s.st_full[st], bx * 64, c2 * 2 * CK + CK, head,
                                             keep);
                        } else {           // pass 2 from the last chunk down: the latest-read K first
                            const int c = nch - 1 - (c2 - nch1);
                            tma_load_3d_hint(s.kv[st][bx], &tm_k, &s.st_full[st], bx * 64, c * CK, head, last);
                            tma_load_3d_hint(s.kv[st][2 + bx], &tm_v, &s.st_full[st], bx * 64, c * CK, head, last);
                        }
                    }
                    ++g;
                }
            }
            // every armed stage's last fill lands before the CTA exits
            for (int t = g > NSTAGE ? g - NSTAGE : 0; t < g; ++t) drain(&s.st_full[t % NSTAGE], (t / NSTAGE) & 1);
        } else if (warp == 1 && lane == 0) {
            // ================================= MMA issuer =================================
            // Every chunk comes back through here: after its products (pass 2) or at once (pass 1),
            // a commit releases its stage and its A buffer, so both barriers complete in chunk order.
            const uint32_t idesc = idesc_bf16(DM, 256, true, true);
            int g = 0;
            bool ok = true;
            for (int hl = 0; hl < nloc && ok; ++hl) {
                const int db = hl & 1;
                const uint32_t tD = tbase + db * 256;
                for (int c2 = 0; c2 < nch1 + nch; ++c2) {
                    const int st = g % NSTAGE, ab = g & 1, c = c2 - nch1;
                    if (!(ok = mbar_wait(&s.st_full[st], (g / NSTAGE) & 1, err))) break;
                    if (!(ok = mbar_wait(&s.a_full[ab], (g >> 1) & 1, err))) break;
                    if (c >= 0) {
                        // the accumulator's previous head has been read by its epilogue
                        if (c == 0 && hl >= 2 && !(ok = mbar_wait(&s.acc_free[db], ((hl - 2) >> 1) & 1, err))) break;
                        tc_fence_after();
                        const uint32_t b0 = smem_u32(s.kv[st][0]);
#pragma unroll
                        for (int ks = 0; ks < CK / 16; ++ks)
#pragma unroll
                            for (int t = 0; t < NTERM; ++t)
                                umma_ss(tD, sdesc_sw128(smem_u32(s.a[ab][t][0]) + ks * 2048, BOX, 1024),
                                        sdesc_sw128(b0 + ks * 2048, BOX, 1024), idesc, (c | ks | t) != 0);
                    }
                    umma_commit(&s.st_empty[st]);
                    umma_commit(&s.a_free[ab]);
                    if (c == nch - 1) umma_commit(&s.d_full[db]);
                    ++g;
                }
            }
            umma_commit(&s.mma_done);
            drain(&s.mma_done, 0);
        }
    } else if (warp < 12) {
        setmaxnreg_inc<REG_EW>();
        // ============================ elementwise warps ============================
        // Thread: key row r of the chunk, coordinates box*64 + (qd & 1)*32 + [0, 32) as four 16-byte
        // groups.  Slot i holds group j = (i + 2*box) & 3: the rotation puts the four threads of a
        // row, and the two rows of a quarter-warp, on distinct banks in every 16-byte access.
        const int te = tid - 128, ew = warp - 4;
        const int r = te >> 2, qd = te & 3, box = qd >> 1;
        uint32_t goff[4];    // byte offset of slot i's group within a box (swizzled)
        int gcol[4];         // first coordinate of slot i's group
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = (i + 2 * box) & 3, lc = (qd & 1) * 4 + j;
            goff[i] = (uint32_t)(r * 128 + ((lc ^ (r & 7)) << 4));
            gcol[i] = box * 64 + (qd & 1) * 32 + 8 * j;
        }
        const float tau = prm.tau;
        // the logit of this thread's key in a box pair (its 32 coordinates left in kp)
        auto logit = [&](const unsigned char* kbx, const uint32_t (&qp)[16], uint32_t (&kp)[16]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 t = *reinterpret_cast<const uint4*>(kbx + goff[i]);
                kp[4 * i] = t.x; kp[4 * i + 1] = t.y; kp[4 * i + 2] = t.z; kp[4 * i + 3] = t.w;
            }
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                d0 = fmaf(bf_lo(qp[u]), bf_lo(kp[u]), d0);
                d1 = fmaf(bf_hi(qp[u]), bf_hi(kp[u]), d1);
            }
            float dot = d0 + d1;
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            dot += __shfl_xor_sync(0xffffffffu, dot, 2);
            return tau * dot;
        };
        int g = 0;
        for (int hl = 0; hl < nloc; ++hl) {
            const int head = (int)blockIdx.x + hl * (int)gridDim.x;
            const int db = hl & 1;
            uint32_t qp[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 t = *reinterpret_cast<const uint4*>(prm.q + (size_t)head * DM + gcol[i]);
                qp[4 * i] = t.x; qp[4 * i + 1] = t.y; qp[4 * i + 2] = t.z; qp[4 * i + 3] = t.w;
            }
            // ---- pass 1: maximum, omega, sum_j w_j k_j (online, against this thread's maximum) ----
            float acc[32], om = 0.f, mt = -INFINITY;   // acc: then kbar, this thread's 32 coordinates
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = 0.f;
            for (int c = 0; c < nch1; ++c, ++g) {
                const int st = g % NSTAGE, ab = g & 1;
                mbar_wait(&s.st_full[st], (g / NSTAGE) & 1, err);
#pragma unroll 1
                for (int h2 = 0; h2 < 2; ++h2) {         // keys r and r + 64 of the chunk's 128
                    uint32_t kp[16];
                    const float sj = logit(s.kv[st][2 * h2 + box], qp, kp);
                    if (c * 2 * CK + h2 * CK + r < prm.n) {
                        if (sj > mt) {
                            const float f = expf(mt - sj);    // 0 while nothing was summed
                            om *= f;
#pragma unroll
                            for (int e = 0; e < 32; ++e) acc[e] *= f;
                            mt = sj;
                        }
                        const float w = expf(sj - mt);
                        om += w;
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            acc[2 * u] = fmaf(w, bf_lo(kp[u]), acc[2 * u]);
                            acc[2 * u + 1] = fmaf(w, bf_hi(kp[u]), acc[2 * u + 1]);
                        }
                    }
                }
                // hand the stage back through the MMA issuer once it has taken chunk g - 2's hand-off
                // (the barrier then never runs two phases ahead of its waiter)
                if (g >= 2) mbar_wait(&s.a_free[ab], ((g - 2) >> 1) & 1, err);
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.a_full[ab]);   // the stage's reads are done
            }
            // combine: the warp's 8 rows against the warp's maximum, then the 8 warps
            {
                float mw = mt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
                const float f = mt == -INFINITY ? 0.f : expf(mt - mw);
                float omw = qd == 0 ? om * f : 0.f;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) omw += __shfl_xor_sync(0xffffffffu, omw, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float x = acc[e] * f;
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                    acc[e] = x;
                }
                if (lane < 4) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int e = 0; e < 8; ++e) s.p1[ew][gcol[i] + e] = acc[8 * i + e];
                    if (lane == 0) {
                        s.p1s[ew][0] = mw;
                        s.p1s[ew][1] = omw;
                    }
                }
            }
            named_bar_sync(1, NEW);
            float m = s.p1s[0][0];
#pragma unroll
            for (int w2 = 1; w2 < 8; ++w2) m = fmaxf(m, s.p1s[w2][0]);
            float fw[8];
            float omega = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < 8; ++w2) {
                fw[w2] = s.p1s[w2][0] == -INFINITY ? 0.f : expf(s.p1s[w2][0] - m);
                omega += s.p1s[w2][1] * fw[w2];
            }
            const float inv_om = 1.f / omega;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float t = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < 8; ++w2) t = fmaf(s.p1[w2][gcol[i] + e], fw[w2], t);
                    acc[8 * i + e] = t * inv_om;
                }
            named_bar_sync(1, NEW);                       // p1 may be written again (next head)
            // ---- pass 2: the products' A = w o (K - kbar), r = sum_j w_j (k_j - kbar), nu -------------
            float rs[32], nu[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) rs[e] = nu[e] = 0.f;
            for (int c = nch - 1; c >= 0; --c, ++g) {      // the chunks in the order TMA delivers them
                const int st = g % NSTAGE, ab = g & 1;
                mbar_wait(&s.st_full[st], (g / NSTAGE) & 1, err);
                uint32_t kp[16];
                const float sj = logit(s.kv[st][box], qp, kp);
                const float w = c * CK + r < prm.n ? expf(sj - m) : 0.f;
                // this chunk's A buffer was last read by the products of chunk g - 2
                if (g >= 2) mbar_wait(&s.a_free[ab], ((g - 2) >> 1) & 1, err);
                const unsigned char* vb = s.kv[st][2 + box];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t th[4], tm[4], tl[4];
                    const uint4 vv = *reinterpret_cast<const uint4*>(vb + goff[i]);
                    const uint32_t vp[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int e0 = 8 * i + 2 * u;
                        const float x0 = w * (bf_lo(kp[4 * i + u]) - acc[e0]);
                        const float x1 = w * (bf_hi(kp[4 * i + u]) - acc[e0 + 1]);
                        split3(x0, x1, th[u], tm[u], tl[u]);
                        rs[e0] += x0;
                        rs[e0 + 1] += x1;
                        nu[e0] = fmaf(w, bf_lo(vp[u]), nu[e0]);
                        nu[e0 + 1] = fmaf(w, bf_hi(vp[u]), nu[e0 + 1]);
                    }
                    *reinterpret_cast<uint4*>(s.a[ab][0][box] + goff[i]) = make_uint4(th[0], th[1], th[2], th[3]);
                    *reinterpret_cast<uint4*>(s.a[ab][1][box] + goff[i]) = make_uint4(tm[0], tm[1], tm[2], tm[3]);
                    *reinterpret_cast<uint4*>(s.a[ab][2][box] + goff[i]) = make_uint4(tl[0], tl[1], tl[2], tl[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.a_full[ab]);
            }
            // the head's sums, over the warp's 8 rows, into buffer db (released by the epilogue of
            // head hl - 2)
            if (hl >= 2) mbar_wait(&s.acc_free[db], ((hl - 2) >> 1) & 1, err);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    rs[e] += __shfl_xor_sync(0xffffffffu, rs[e], o);
                    nu[e] += __shfl_xor_sync(0xffffffffu, nu[e], o);
                }
            }
            if (lane < 4) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        s.r[db][ew][gcol[i] + e] = rs[8 * i + e];
                        s.nu[db][ew][gcol[i] + e] = nu[8 * i + e];
                        if (ew == 0) s.kb[db][gcol[i] + e] = acc[8 * i + e];
                    }
                if (ew == 0 && lane == 0) {
                    s.om[db] = omega;
                    s.mx[db] = m;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.mom_full[db]);
        }
    } else {
        setmaxnreg_dec<REG_EP>();
        // ================================ epilogue warps ================================
        const int quarter = warp & 3, wq = quarter;
        const int a = 32 * quarter + lane;    // row of D (TMEM lane) = coordinate
        int rsl = 0;                          // reduction slot
        // sums over the 128 epilogue threads of up to three values, in a fixed order (every
        // thread gets the same bits, so every branch on them is uniform)
        auto bsum3 = [&](float v0, float v1, float v2, float& o0, float& o1, float& o2) {
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                v0 += __shfl_xor_sync(0xffffffffu, v0, o);
                v1 += __shfl_xor_sync(0xffffffffu, v1, o);
                v2 += __shfl_xor_sync(0xffffffffu, v2, o);
            }
            if (lane == 0) {
                s.red[rsl][wq][0] = v0;
                s.red[rsl][wq][1] = v1;
                s.red[rsl][wq][2] = v2;
            }
            named_bar_sync(2, NEP);
            o0 = ((s.red[rsl][0][0] + s.red[rsl][1][0]) + s.red[rsl][2][0]) + s.red[rsl][3][0];
            o1 = ((s.red[rsl][0][1] + s.red[rsl][1][1]) + s.red[rsl][2][1]) + s.red[rsl][3][1];
            o2 = ((s.red[rsl][0][2] + s.red[rsl][1][2]) + s.red[rsl][2][2]) + s.red[rsl][3][2];
            rsl = (rsl + 1) & 3;
        };
        for (int hl = 0; hl < nloc; ++hl) {
            const int head = (int)blockIdx.x + hl * (int)gridDim.x;
            const int db = hl & 1;
            mbar_wait(&s.mom_full[db], (hl >> 1) & 1, err);
            mbar_wait(&s.d_full[db], (hl >> 1) & 1, err);
            tc_fence_after();
            float r_a = 0.f, nu_a = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < 8; ++w2) {
                r_a += s.r[db][w2][a];
                nu_a += s.nu[db][w2][a];
            }
            const float omega = s.om[db], kb = s.kb[db][a];
            const float inv_om = 1.f / omega, lam_n = prm.lambda / omega;
            const float dl = kb - __bfloat162float(prm.q[(size_t)head * DM + a]);
            const uint32_t trow = tbase + db * 256 + ((uint32_t)(32 * quarter) << 16);
            float x = 0.f, rr = dl, pp = dl, gamma, t1, t2;
            bsum3(rr * rr, 0.f, 0.f, gamma, t1, t2);
            const float rn0 = sqrtf(gamma);
            bool active = gamma > 0.f && !(rn0 <= prm.cg_tol * rn0);
            int iters = 0;
            for (int it = 0; it < prm.cg_max_iters && active; ++it) {
                s.p[a] = pp;
                named_bar_sync(2, NEP);
                float y0 = 0.f, y1 = 0.f;
#pragma unroll 1
                for (int cc = 0; cc < DM; cc += 32) {
                    float cv[32];
                    tmem_ld32(trow + cc, cv);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        y0 = fmaf(cv[e], s.p[cc + e], y0);
                        y1 = fmaf(cv[e + 1], s.p[cc + e + 1], y1);
                    }
                }
                float kp;
                bsum3(kb * pp, 0.f, 0.f, kp, t1, t2);
                const float cp = ((y0 + y1) - r_a * kp) * inv_om + lam_n * pp;
                float pcp;
                bsum3(pp * cp, 0.f, 0.f, pcp, t1, t2);
                if (!(pcp > 0.f)) break;             // no positive curvature left (uniform)
                const float alpha = gamma / pcp;
                x = fmaf(alpha, pp, x);
                rr = fmaf(-alpha, cp, rr);
                float g2;
                bsum3(rr * rr, 0.f, 0.f, g2, t1, t2);
                const float beta = g2 / gamma;
                gamma = g2;
                pp = fmaf(beta, pp, rr);
                ++iters;
                if (gamma == 0.f || sqrtf(gamma) <= prm.cg_tol * rn0) active = false;
            }
            float dx, rx;
            bsum3(dl * x, r_a * x, 0.f, dx, rx, t2);
            // Hc^T x: x_a times row a of Hc, summed over the rows: within a warp by a butterfly that
            // leaves column cc + l in lane l, then over the four warps
#pragma unroll 1
            for (int cc = 0; cc < DM; cc += 32) {
                float hv[32];
                tmem_ld32(trow + DM + cc, hv);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) hv[e] *= x;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const bool up = (lane & o) != 0;
#pragma unroll
                    for (int e = 0; e < o; ++e) {
                        const float send = up ? hv[e] : hv[e + o];
                        const float keep = up ? hv[e + o] : hv[e];
                        hv[e] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
                s.hx[wq][cc + lane] = hv[0];
            }
            named_bar_sync(2, NEP);
            const float hx = ((s.hx[0][a] + s.hx[1][a]) + s.hx[2][a]) + s.hx[3][a];
            const float inv_g = 1.f / (1.f + dx);
            prm.out[(size_t)head * DM + a] = __float2bfloat16_rn((nu_a - hx) / (omega - rx));
            prm.rho[(size_t)head * DM + a] = x * inv_g;
            if (a == 0) {
                prm.denom[head] = omega * inv_g;
                if (prm.cg_iters) prm.cg_iters[head] = iters;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.acc_free[db]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tbase, 512);
    }
    if (tid == 0 && s.err) atomicOr(prm.dev_err, (unsigned)kDevErrMbarTimeout);
}

int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
    }
    return n;
}

}  // namespace

bool decode_moment_supported(const DecodeProblem& p) {
    return p.dtype == 0 && p.d == DM;
}

cudaError_t launch_decode_moment(const DecodeProblem& p, cudaStream_t stream) {
    if (!decode_moment_supported(p)) return cudaErrorInvalidValue;
    const long long heads = (long long)p.B * p.H;
    CUtensorMap tk, tv;
    if (!make_tmap_16b_3d_strided(&tk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, DM, (uint64_t)p.n, (uint64_t)heads,
                                  (uint64_t)p.n_cap, CK) ||
        !make_tmap_16b_3d_strided(&tv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, DM, (uint64_t)p.n, (uint64_t)heads,
                                  (uint64_t)p.n_cap, CK))
        return cudaErrorInvalidValue;
    MomParams prm;
    prm.q = static_cast<const __nv_bfloat16*>(p.q);
    prm.out = static_cast<__nv_bfloat16*>(p.out);
    prm.rho = p.rho;
    prm.denom = p.denom;
    prm.cg_iters = p.cg_iters;
    prm.dev_err = p.dev_err;
    prm.nheads = (int)heads;
    prm.n = p.n;
    prm.cg_max_iters = p.cg_max_iters;
    prm.tau = p.tau;
    prm.lambda = p.lambda;
    prm.cg_tol = p.cg_tol;
    const size_t smem = sizeof(MomSmem);
    cudaError_t e = cudaFuncSetAttribute(lla_decode_mom_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // setmaxnreg.inc waits for registers the decreasing warpgroups give back: the split adds up
    // only if the kernel was built to the launch's full share
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, lla_decode_mom_kernel)) != cudaSuccess) return e;
    if (fa.numRegs != REG_LAUNCH) return cudaErrorInvalidConfiguration;
    const int grid = (int)(heads < sm_count() ? heads : sm_count());
    if (p.ev_main_begin && (e = cudaEventRecord(p.ev_main_begin, stream)) != cudaSuccess) return e;
    lla_decode_mom_kernel<<<grid, NTH, smem, stream>>>(tk, tv, prm);
    e = cudaGetLastError();
    if (e == cudaSuccess && p.ev_main_end) e = cudaEventRecord(p.ev_main_end, stream);
    return e;
}

}  // namespace lla
