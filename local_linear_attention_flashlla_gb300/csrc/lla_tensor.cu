// Tensor-core path of the causal LLA forward pass on sm_103a (tcgen05 + TMEM + TMA).
//
// Operands.  A pre-pass scales q, k, v (bf16) by per-tensor powers of two and stores them
// as fp16 (exact for every value in fp16's normal range; the scale puts each tensor's
// largest magnitude at or below 2^14).  fp16 is used instead of bf16 because the CG
// products need the extra mantissa bits: the matrix-vector products of CG are only as
// accurate as their rounded operands.  Every in-kernel operand (CG direction p, the
// per-pair coefficients, rho') is likewise stored as fp16 times a per-row power of two
// chosen from a bound on its magnitude, so nothing overflows and the exact unscaling is a
// multiplication by a power of two.
//
// Kernel.  One CTA owns a tile of 128 queries of one (b, h) and runs the FlashLLA sweeps
// of the Local Linear Attention reading notes (section 2.2, Algorithm 1) over the causal
// key blocks of 128 keys (tile t sees blocks 0..t, the last one masked):
//   MAX     S = Q K^T                                   -> exact row maxima m_i
//   MOMENT  S, W = 2^(S*c - m) -> Y = W K                 -> omega_i, kbar_i = mu~_i / omega_i
//   CG xT   S, A' = P K^T, M = W o (A' - kbar.p) -> Y = M K  -> (C_i/omega_i) p, CG update
//   OUT     S, T = (R_hi + R_lo) K^T, U = W o (c - T) -> Y = U V -> out_i
// CG runs on the centred system (C_i/omega_i) rho'_i = delta_i with delta_i = kbar_i - q_i;
// rho_i = rho'_i / (1 + delta_i.rho'_i), denom_i = omega_i / (1 + delta_i.rho'_i), and
// out_i = sum_j w_ij (1 - (k_j - kbar_i).rho'_i) v_j / sum_j w_ij (1 - (k_j - kbar_i).rho'_i)
// (Eqs. (6)-(8) with Sigma_i = C_i + omega_i delta_i delta_i^T, Sherman-Morrison).
//
// Parallax form (caller-supplied probe, Parallax page): MAX, MOMENT and OUT with the probe as
// rho' (no CG sweep), i.e. out_i = sum_j wbar_ij (1 - (k_j - kbar_i).probe_i) v_j, the softmax
// output minus the softmax-weighted value/key covariance times the probe.
//
// Roles (384 threads, three warpgroups): warp 0 lane 0 issues TMA (Q once, then K/V blocks
// into a 3-slot ring); lane 0 of warps 1, 3 and 2 issues the S, the A'/T and the Y products
// (three issue streams, synchronised through mbarriers: each MMA-issuing warp shares its
// sub-partition's scheduler with two elementwise warps, so one stream per warp keeps up);
// warpgroups 1-2 (256 threads) do the elementwise work and the CG vector updates, thread =
// (query row, half of the key block / half of the head dimension).  setmaxnreg moves
// registers from warpgroup 0 (72 each) to the elementwise warpgroups (216 each):
// 128 x 72 + 256 x 216 = 384 x 168, the launch allocation.  TMEM (512 columns): S double buffer (2 x 128), A' (128),
// Y accumulator (d).  The pairwise weights never leave TMEM/registers; working memory in
// HBM is the fp16 operand copies, the CG iterate (kept in the rho output) and kbar.
// Every mbarrier wait is bounded (about 2 s); on a timeout the CTA drains its in-flight
// copies and MMAs, frees TMEM and records the failure in the library's device error word.
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

constexpr int BQ = 128;            // queries per tile (MMA M)
constexpr int BK = 128;            // keys per block (MMA N of QK^T, K of the Y product)
constexpr int NTHREADS = 384;
constexpr int NEW = 256;           // elementwise threads
constexpr int NSLOT = 3;           // K/V ring slots
constexpr int EW_BAR = 1;          // named barrier of the elementwise warps
constexpr int HDR_BYTES = 256;

enum SweepType : int { SW_MAX = 0, SW_MOMENT = 1, SW_CG = 2, SW_OUT = 3, SW_TBAR = 4, SW_END = 5 };

// Sweep order without a tolerance: MAX, MOMENT, (backward: TBAR), T x CG, then OUT (forward) or
// the end (backward).  With a tolerance the elementwise threads publish each later sweep's type.
// NO_MAX (the precise and Parallax forms, TcParams::mode 1): the same without the MAX sweep; the
// MOMENT sweep finds the row maximum itself (a reference from its first block, the exact maximum by
// its end).
template <bool BWD>
__device__ __forceinline__ int static_sweep(int sweep, int cg_sweeps, int T, bool no_max) {
    if (!BWD && no_max) ++sweep;
    if (sweep == 0) return SW_MAX;
    if (sweep == 1) return SW_MOMENT;
    if (BWD && sweep == 2) return SW_TBAR;
    return cg_sweeps < T ? SW_CG : (BWD ? SW_END : SW_OUT);
}
// Sweeps that read a V block after each K block.
template <bool BWD>
__device__ __forceinline__ bool two_loads(int type) {
    return type == SW_OUT || (BWD && (type == SW_MOMENT || type == SW_TBAR));
}

struct Header {
    unsigned maxabs[4];            // float bits of max |q|, max |k|, max |v|, max |dout| (backward)
    int abort;                     // set by a CTA whose bounded wait gave up: the others stop early
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ceil(log2(x)) for finite x > 0
__device__ __forceinline__ int ceil_log2f(float x) {
    int e;
    const float f = frexpf(x, &e);      // x = f 2^e, f in [0.5, 1)
    return f == 0.5f ? e - 1 : e;
}
// exponent s such that x 2^s <= 2^14 with x 2^s > 2^13 (0 when x == 0)
__device__ __forceinline__ int scale_exp(float maxabs) {
    if (!(maxabs > 0.f)) return 0;
    int s = 14 - ceil_log2f(maxabs);
    return s < -100 ? -100 : (s > 100 ? 100 : s);
}

// ------------------------------------------------------------------------------------------
// Pre-pass: max |x| per tensor, then scaled fp16 copies.
// NTEN = 3: q, k, v; NTEN = 4 (backward): also dout.
template <int NTEN>
__global__ void lla_maxabs_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                                  const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
                                  size_t count8, Header* hdr) {
    float m[4] = {0.f, 0.f, 0.f, 0.f};
    const __nv_bfloat16* src[4] = {q, k, v, g};
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < count8; idx += (size_t)gridDim.x * blockDim.x) {
#pragma unroll
        for (int t = 0; t < NTEN; ++t) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src[t]) + idx);
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h[u]);
                m[t] = fmaxf(m[t], fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NTEN; ++t) {
        float x = m[t];
        for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
        if ((threadIdx.x & 31) == 0) atomicMax(&hdr->maxabs[t], __float_as_uint(x));
    }
}

// Scaled fp16 copies, and |k_j|^2 of every key row (natural units, fp32) into knorm [slices][npad]
// (rows of G = d/8 consecutive 8-element groups, summed over G lanes of a warp).  The loop's trip
// count is uniform per warp, so every lane takes part in the row sums' shuffles.
template <int NTEN>
__global__ void lla_to_half_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                                   const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
                                   __half* q16, __half* k16, __half* v16, __half* g16, size_t count8,
                                   const Header* __restrict__ hdr, float* __restrict__ knorm, int G, int n, int npad) {
    const __nv_bfloat16* src[4] = {q, k, v, g};
    __half* dst[4] = {q16, k16, v16, g16};
    float sc[4];
#pragma unroll
    for (int t = 0; t < NTEN; ++t) sc[t] = pow2i(scale_exp(__uint_as_float(hdr->maxabs[t])));
    const int lane = threadIdx.x & 31;
    const size_t stride = (size_t)gridDim.x * blockDim.x;      // a multiple of 32
    for (size_t base = blockIdx.x * (size_t)blockDim.x + (threadIdx.x & ~31u); base < count8; base += stride) {
        const size_t idx = base + lane;
        const bool in = idx < count8;
        float ss = 0.f;
        if (in) {
#pragma unroll
            for (int t = 0; t < NTEN; ++t) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src[t]) + idx);
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
                uint4 o;
                uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 f = __bfloat1622float2(h[u]);
                    ow[u] = pack_half2(f.x * sc[t], f.y * sc[t]);
                    if (t == 1) ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
                }
                reinterpret_cast<uint4*>(dst[t])[idx] = o;
            }
        }
        for (int o = G >> 1; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (in && (idx % (size_t)G) == 0) {
            const size_t r = idx / (size_t)G;          // key row over all slices
            knorm[(r / (size_t)n) * (size_t)npad + r % (size_t)n] = ss;
        }
    }
}

// |k_j|^2 of the 32 keys key0 .. key0+31 (key0 a multiple of 32; rows past n read the zeroed pad)
__device__ __forceinline__ void load_knorm32(const float* __restrict__ kn_row, int key0, float (&kn)[32]) {
    const float4* p = reinterpret_cast<const float4*>(kn_row + key0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float4 t = __ldg(p + u);
        kn[4 * u] = t.x;
        kn[4 * u + 1] = t.y;
        kn[4 * u + 2] = t.z;
        kn[4 * u + 3] = t.w;
    }
}

// Pulls the two 128-byte lines of a thread half's 64 key norms of a block into L1 (lanes 0 and 1),
// a block ahead of their loads: all lanes of a warp then read them at L1 latency, not L2's.
__device__ __forceinline__ void prefetch_knorm64(const float* kn_row, int key0, int lane) {
    if (lane < 2) asm volatile("prefetch.global.L1 [%0];" ::"l"(kn_row + key0 + 32 * lane));
}

// ------------------------------------------------------------------------------------------
template <int D>
struct TcSmem {
    static constexpr int NB = D / 64;                  // 64-column (128-byte) boxes per row
    static constexpr int TILE = BQ * D * 2;            // bytes of a [128 x D] fp16 tile
    unsigned char q[TILE];                             // queries (TMA)
    unsigned char p[TILE];                             // CG direction P, then R_hi (rho', threads)
    // R_lo (output sweep); P_lo (CG sweeps of tile 0); in the CG sweeps of the other tiles, the
    // fp32 CG iterate x of coordinates 0 .. D/2-1 as [coordinate][row]
    unsigned char rlo[TILE];
    unsigned char xb[TILE];                            // x of coordinates D/2 .. D-1 (tiles > 0)
    unsigned char slot[NSLOT][TILE];                   // K / V blocks (TMA)
    uint64_t slot_full[NSLOT], slot_empty[NSLOT];
    uint64_t q_full, s_full[2], ew_done[2], m_free[2], a_free, y_done, p_ready, final_s, final_a, final_y;
    uint64_t max_done;                                 // backward: the elementwise warps finished the MAX sweep
    float xch[2][2][BQ];                               // row-scalar exchange between the two halves
    uint32_t tmem_base;
    int err;
    int next_type;
    int out_split;                                     // the output sweep's T takes R_lo as well
};

// 227 KB: the most dynamic shared memory a block may have on sm_103a
static_assert(sizeof(TcSmem<128>) <= 232448 && sizeof(TcSmem<64>) <= 232448, "shared memory layout too large");

struct TcParams {
    Header* hdr;
    float* kbar;          // kbar, tile-transposed: [B*H][n_tiles][D][128] fp32 scratch
    float* xs;            // CG iterate rho', same layout
    const float* knorm;   // |k_j|^2 per key row: [B*H][n_tiles * 128] fp32 (zero past n)
    __nv_bfloat16* out;
    float* rho;
    float* denom;
    int* cg_iters;
    const float* probe;   // Parallax form: caller's probe [B,H,n,D] fp32 (null for LLA)
    // backward mode: the forward's rho [B,H,n,D] and denom [B,H,n] in, records and y out
    const float* rho_in;
    const float* denom_in;
    BwdRowRec* rec;
    float* yvec;          // [B,H,n,D] fp32
    unsigned* dev_err;
    // 0 = every tile with its MAX sweep; 1 (precise and Parallax forms) = no MAX sweep, each tile
    // writes tile_flag (1: a row's maximum exceeded its first block's by more than the weights' fp16
    // headroom, the tile's results are void); 2 = every tile whose flag is set, with its MAX sweep
    // (the others return).
    int mode;
    int* tile_flag;       // [B*H][n_tiles]
    int n, n_tiles;
    float tau, lambda, cg_tol;
    int cg_max_iters;
};

// Sum (or max) of a per-row value over the two half-threads of the row.  Two buffers used in
// turn suffice: a thread writes a buffer again only after the next exchange's barrier, which its
// partner reaches only after reading that buffer.
struct Xch {
    float (*buf)[2][BQ];
    int idx, half, row;
    __device__ float swap(float v) {
        const float* b = put(v);
        named_bar_sync(EW_BAR, NEW);
        return take(b);
    }
    // The two halves of a swap, for an exchange that rides on a barrier taken anyway.
    __device__ const float* put(float v) {
        float* b = &buf[idx][0][0];
        idx ^= 1;
        b[half * BQ + row] = v;
        return b;
    }
    __device__ float take(const float* b) const { return b[(1 - half) * BQ + row]; }
    __device__ float sum(float v) { return v + swap(v); }
    __device__ float max(float v) { return fmaxf(v, swap(v)); }
};

__device__ __forceinline__ bool ew_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, 256, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// Drain wait: ignores the error flag, bounded by its own timer (used only on exit).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 2000000000ull) return;
}

// fp16 element (row, col) of a swizzled [128 x D] tile
__device__ __forceinline__ __half* tile_half(const unsigned char* t, int row, int col) {
    return reinterpret_cast<__half*>(const_cast<unsigned char*>(t) + sw128_offset(row, col, BQ));
}

// 8 consecutive coordinates (from col) of this thread's row of a direction tile, unscaled:
// o = (hi [+ lo]) * sc.  split: the tile carries an fp16 remainder in lo (about 22 bits in all).
__device__ __forceinline__ void load_dir8(const unsigned char* hi, const unsigned char* lo, bool split, int row, int col,
                                          float sc, float (&o)[8]) {
    const uint4 h = *reinterpret_cast<const uint4*>(tile_half(hi, row, col));
    const __half2* h2 = reinterpret_cast<const __half2*>(&h);
    const uint64_t sc2 = f2_pack(sc, sc);
    if (split) {
        const uint4 l = *reinterpret_cast<const uint4*>(tile_half(lo, row, col));
        const __half2* l2 = reinterpret_cast<const __half2*>(&l);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 a = __half22float2(h2[u]), b = __half22float2(l2[u]);
            f2_unpack(f2_mul(f2_add(f2_pack(a.x, a.y), f2_pack(b.x, b.y)), sc2), o[2 * u], o[2 * u + 1]);
        }
    } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 a = __half22float2(h2[u]);
            f2_unpack(f2_mul(f2_pack(a.x, a.y), sc2), o[2 * u], o[2 * u + 1]);
        }
    }
}

// The 8 fp16 values of h, times sc.
__device__ __forceinline__ void dir8_hi(const uint4& h, float sc, float (&o)[8]) {
    const __half2* h2 = reinterpret_cast<const __half2*>(&h);
    const uint64_t sc2 = f2_pack(sc, sc);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 a = __half22float2(h2[u]);
        f2_unpack(f2_mul(f2_pack(a.x, a.y), sc2), o[2 * u], o[2 * u + 1]);
    }
}

// One 16-coordinate chunk C of this thread's DH coordinates of
//   cp = (C/omega) p_hat = Y ysc - kbar msc + lam_n p_hat
// (and, with DOT, the partial dot p_hat.cp as two fp32 partial sums).  SPLIT: the direction tile
// carries an fp16 remainder (hi + lo); a compile-time form, so the caller's loops hold no branch on it.
template <int C, int DH, bool DOT, bool SPLIT>
__device__ __forceinline__ void cg_apply_chunk(uint32_t ty, const unsigned char* ptile, const unsigned char* plo,
                                               int row, int col, const float (&kv)[DH], float ysc, float msc, float lam_n,
                                               float psc, float (&cp)[16], uint64_t& pcp2) {
    float y[16], p0[8], p1[8];
    tmem_ld16(ty + C * 16, y);
    load_dir8(ptile, plo, SPLIT, row, col + C * 16, psc, p0);
    load_dir8(ptile, plo, SPLIT, row, col + C * 16 + 8, psc, p1);
    tmem_ld_wait();
    const uint64_t ysc2 = f2_pack(ysc, ysc), nmsc2 = f2_pack(-msc, -msc), lam2 = f2_pack(lam_n, lam_n);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
        const uint64_t ph = j < 8 ? f2_pack(p0[j], p0[j + 1]) : f2_pack(p1[j - 8], p1[j - 7]);
        const uint64_t kb = f2_pack(kv[C * 16 + j], kv[C * 16 + j + 1]);
        const uint64_t c2 = f2_fma(f2_pack(y[j], y[j + 1]), ysc2, f2_fma(kb, nmsc2, f2_mul(ph, lam2)));
        f2_unpack(c2, cp[j], cp[j + 1]);
        if (DOT) pcp2 = f2_fma(ph, c2, pcp2);
    }
}

// Per-pair coefficients of one 32-key chunk (chunk C of this thread's 64 keys):
//   HAS_A:  out_j = 2^(s_j c - off) (base + sign a_j)     (CG: base = -kbar.p, sign = +1;
//                                                          output: base = c, sign = -1)
//   !HAS_A: out_j = 2^(s_j c - off)                       (moments)
// zero where MASKED and key column > lim.  Packs pairs to fp16 and accumulates their sum into
// two running fp32 partial sums (even and odd keys).  Key pairs go through f32x2 arithmetic.
// SPLIT: also the fp16 remainder of every coefficient in pl (hi + lo carry about 22 bits).
template <bool MASKED, bool HAS_A, int C, bool SPLIT = false>
__device__ __forceinline__ void coef_chunk(const float (&v)[32], const float (&a)[64], float c_log2, float off,
                                           float base, float sign, int col0, int lim, uint64_t& sum2,
                                           uint32_t (&pk)[16], uint32_t* pl = nullptr) {
    const uint64_t cc = f2_pack(c_log2, c_log2), oo = f2_pack(-off, -off);
    const uint64_t bb = f2_pack(base, base), sg = f2_pack(sign, sign);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(v[j], v[j + 1]), cc, oo), x0, x1);
        uint64_t m = f2_pack(ex2(x0), ex2(x1));
        if (HAS_A) m = f2_mul(m, f2_fma(sg, f2_pack(a[C * 32 + j], a[C * 32 + j + 1]), bb));
        float m0, m1;
        f2_unpack(m, m0, m1);
        if (MASKED) {
            m0 = (col0 + j <= lim) ? m0 : 0.f;
            m1 = (col0 + j + 1 <= lim) ? m1 : 0.f;
            m = f2_pack(m0, m1);
        }
        sum2 = f2_add(sum2, m);
        pk[j >> 1] = pack_half2(m0, m1);
        if (SPLIT) {
            const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&pk[j >> 1]));
            pl[j >> 1] = pack_half2(m0 - h.x, m1 - h.y);
        }
    }
}

// Forward moment sweep: weights out_j = 2^(s_j c - off), with the running sums of out_j and of
// out_j |k_j|^2 (kn: the chunk's 32 key norms).  SPLIT: also the fp16 remainder of every weight.
template <bool MASKED, bool SPLIT>
__device__ __forceinline__ void coef_chunk_wk(const float (&v)[32], const float (&kn)[32], float c_log2, float off,
                                              int col0, int lim, uint64_t& sum2, uint64_t& tk2, uint32_t (&pk)[16],
                                              uint32_t* pl = nullptr) {
    const uint64_t cc = f2_pack(c_log2, c_log2), oo = f2_pack(-off, -off);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(v[j], v[j + 1]), cc, oo), x0, x1);
        float m0 = ex2(x0), m1 = ex2(x1);
        if (MASKED) {
            m0 = (col0 + j <= lim) ? m0 : 0.f;
            m1 = (col0 + j + 1 <= lim) ? m1 : 0.f;
        }
        const uint64_t m = f2_pack(m0, m1);
        sum2 = f2_add(sum2, m);
        tk2 = f2_fma(m, f2_pack(kn[j], kn[j + 1]), tk2);
        pk[j >> 1] = pack_half2(m0, m1);
        if (SPLIT) {
            const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&pk[j >> 1]));
            pl[j >> 1] = pack_half2(m0 - h.x, m1 - h.y);
        }
    }
}

// Backward moment sweep: out_j = 2^(s_j c - off) (the weights, as the moment sweep), with the
// running sums of out_j and of out_j a_j (a = H = G V^T, the per-pair dout.v).
template <bool MASKED, int C>
__device__ __forceinline__ void coef_chunk_wh(const float (&v)[32], const float (&a)[64], float c_log2, float off,
                                              int col0, int lim, uint64_t& sum2, uint64_t& wh2, uint32_t (&pk)[16],
                                              uint32_t (&pl)[16]) {
    const uint64_t cc = f2_pack(c_log2, c_log2), oo = f2_pack(-off, -off);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(v[j], v[j + 1]), cc, oo), x0, x1);
        float m0 = ex2(x0), m1 = ex2(x1);
        if (MASKED) {
            m0 = (col0 + j <= lim) ? m0 : 0.f;
            m1 = (col0 + j + 1 <= lim) ? m1 : 0.f;
        }
        const uint64_t m = f2_pack(m0, m1);
        sum2 = f2_add(sum2, m);
        wh2 = f2_fma(m, f2_pack(a[C * 32 + j], a[C * 32 + j + 1]), wh2);
        pk[j >> 1] = pack_half2(m0, m1);
        const float2 h = __half22float2(*reinterpret_cast<const __half2*>(&pk[j >> 1]));
        pl[j >> 1] = pack_half2(m0 - h.x, m1 - h.y);
    }
}

__device__ __forceinline__ float f2_total(uint64_t s2) {
    float lo, hi;
    f2_unpack(s2, lo, hi);
    return lo + hi;
}

// One 128 x 128 x D product D[tmem] = A[smem] B[smem]^T, both K-major SW128 tiles, D/16 k-steps.
// Descriptors are built once; each k-step adds a compile-time start-address offset (bytes >> 4),
// which never carries out of the 14-bit field for tiles inside the 228 KB of shared memory.
template <int D, bool ACC_FIRST>
__device__ __forceinline__ void gemm_qk(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr) {
    constexpr uint32_t ID = idesc_f16(BQ, BK, false);
    const uint64_t a0 = sdesc_sw128(a_addr, 16, 1024), b0 = sdesc_sw128(b_addr, 16, 1024);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t off = (uint64_t)((((ks >> 2) * (BQ * 128)) + (ks & 3) * 32) >> 4);
        if (ks == 0 && !ACC_FIRST) umma_ss_c<false>(d_tmem, a0 + off, b0 + off, ID);
        else umma_ss_c<true>(d_tmem, a0 + off, b0 + off, ID);
    }
}
// Y[tmem] (+)= M[tmem] (128 x 128 keys, fp16 pairs at columns 64h + 0..31 per key half h) x B,
// B = a [128 keys x D] K/V slot read MN-major.
template <int D>
__device__ __forceinline__ void gemm_y(uint32_t y_tmem, uint32_t m_tmem, uint32_t b_addr, bool acc) {
    constexpr uint32_t ID = idesc_f16(BQ, D, true);
    const uint64_t b0 = sdesc_sw128(b_addr, BK * 128, 1024);
    if (acc) umma_ts_c<true>(y_tmem, m_tmem, b0, ID);
    else umma_ts_c<false>(y_tmem, m_tmem, b0, ID);
#pragma unroll
    for (int ks = 1; ks < BK / 16; ++ks)
        umma_ts_c<true>(y_tmem, m_tmem + (ks >> 2) * 64 + (ks & 3) * 8, b0 + (uint64_t)((ks * 2048) >> 4), ID);
}

// As gemm_y with hi + lo coefficients: key chunk c (32 keys) of key half h holds its fp16 hi pairs at
// columns 64h + 32c + 0..15 and the lo pairs at 64h + 32c + 16..31.
template <int D>
__device__ __forceinline__ void gemm_y_split(uint32_t y_tmem, uint32_t m_tmem, uint32_t b_addr, bool acc) {
    constexpr uint32_t ID = idesc_f16(BQ, D, true);
    const uint64_t b0 = sdesc_sw128(b_addr, BK * 128, 1024);
#pragma unroll
    for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
            const uint32_t col = (ks >> 2) * 64 + ((ks & 3) >> 1) * 32 + (ks & 1) * 8 + part * 16;
            const uint64_t bk = b0 + (uint64_t)((ks * 2048) >> 4);
            if (part == 0 && ks == 0 && !acc) umma_ts_c<false>(y_tmem, m_tmem + col, bk, ID);
            else umma_ts_c<true>(y_tmem, m_tmem + col, bk, ID);
        }
    }
}

// PREC (forward only): the precise form used in tolerance mode.  The moment sweep's weights and the
// CG sweeps' per-pair coefficients are fp16 hi + lo pairs (two TS products per block) and the CG
// direction is hi + lo in every tile, so each carries about 22 bits, as in the backward mode.
// PROBE: the Parallax form (caller's probe, no CG).  It needs no key-scatter trace: its output sweep's
// coefficient bound comes from max|k| alone, and it always carries the probe's fp16 remainder.
template <int D, bool BWD, bool PREC = false, bool PROBE = false>
__global__ void __launch_bounds__(NTHREADS, 1)
lla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g, const TcParams prm) {
    using S = TcSmem<D>;
    constexpr int NB = S::NB;
    constexpr int DH = D / 2;                       // head-dim coordinates per elementwise thread
    constexpr bool SPLITM = BWD || PREC;            // hi + lo weights and CG coefficients
    // The forms launched without MAX sweeps (mode 1, then mode 2 for the marked tiles): the precise
    // form and the Parallax form.  The fixed-cap form keeps them: without, its CG updates measured
    // about 1 000 cycles slower each (their row exchanges), more than the MAX sweep costs.
    constexpr bool NO_MAX_FORM = !BWD && (PREC || PROBE);

    // The swizzled tiles need 1024-byte alignment.  Dynamic shared memory begins 1024-aligned
    // (right after the block's reserved kilobyte), so no padding is requested; a launch where it
    // does not is refused here, by every thread alike, before anything is touched.
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(prm.dev_err, (unsigned)kDevErrSmemAlign);
        return;
    }
    S& s = *reinterpret_cast<S*>(smem_raw);
    volatile int* err = &s.err;
    volatile int* abort_flag = &prm.hdr->abort;
#define WAIT(bar, par, e) mbar_wait_abortable(bar, par, e, abort_flag)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int rank, head;
    causal_order((size_t)4 * prm.n * D, rank, head);    // fp16 keys and values of a head
    const int tile = prm.n_tiles - 1 - rank;
    // the second forward launch redoes only the tiles the first one marked (uniform per CTA, before
    // any barrier or TMEM allocation)
    if (NO_MAX_FORM && prm.mode == 2 && prm.tile_flag[(size_t)head * prm.n_tiles + tile] == 0) return;
    const int n = prm.n;
    const int nkb = tile + 1;
    const bool dynamic = prm.cg_tol > 0.f;
    const bool no_max = NO_MAX_FORM && prm.mode == 1;
    const int n_static = BWD ? 3 : (no_max ? 1 : 2);   // leading sweeps of a fixed type in every mode

    if (tid == 0) {
        s.err = *abort_flag ? 1 : 0;           // another CTA of this launch already gave up
        s.next_type = SW_CG;
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(&s.slot_full[i], 1);
            mbar_init(&s.slot_empty[i], 1);
        }
        mbar_init(&s.q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.s_full[i], 2);             // the S product and the A'/T product
            mbar_init(&s.ew_done[i], NEW / 32);       // one arrive per elementwise warp
        }
        mbar_init(&s.a_free, NEW / 32);
        for (int i = 0; i < 2; ++i) mbar_init(&s.m_free[i], 1);
        mbar_init(&s.y_done, 1);
        mbar_init(&s.p_ready, 1);                   // one arrive after the elementwise threads' barrier
        mbar_init(&s.final_s, 1);
        mbar_init(&s.final_a, 1);
        mbar_init(&s.final_y, 1);
        mbar_init(&s.max_done, NEW / 32);
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS0 = s.tmem_base, tA = s.tmem_base + 256, tY = s.tmem_base + 384;

    if (warp < 4) {
    // warpgroup 0: the register release dominates the producer and MMA code, so both are
    // compiled within 72 registers
    setmaxnreg_dec72();
    if (warp == 0) {
        // =============================== TMA producer ===============================
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            // backward: dout's tile goes to the direction tile, the A operand of H = G V^T in
            // the MOMENT and TBAR sweeps (the direction is first written after TBAR)
            mbar_arrive_expect_tx(&s.q_full, BWD ? 2 * S::TILE : S::TILE);
            for (int bx = 0; bx < NB; ++bx) tma_load_3d(s.q + bx * BQ * 128, &tm_q, &s.q_full, bx * 64, tile * BQ, head);
            if (BWD)
                for (int bx = 0; bx < NB; ++bx) tma_load_3d(s.p + bx * BQ * 128, &tm_g, &s.q_full, bx * 64, tile * BQ, head);
            uint32_t fill = 0, pr = 0;
            int cg_sweeps = 0;
            for (int sweep = 0; !*err; ++sweep) {
                int type;
                if (sweep < n_static || !dynamic) type = static_sweep<BWD>(sweep, cg_sweeps, prm.cg_max_iters, no_max);
                else {
                    if (!WAIT(&s.p_ready, pr & 1, err)) break;
                    ++pr;
                    type = s.next_type;
                }
                if (type == SW_END) break;
                if (type == SW_CG) ++cg_sweeps;
                const int nload = two_loads<BWD>(type) ? 2 : 1;
                for (int kb = 0; kb < nkb && !*err; ++kb) {
                    for (int l = 0; l < nload; ++l) {
                        const int sl = fill % NSLOT;
                        if (!WAIT(&s.slot_empty[sl], ((fill / NSLOT) & 1) ^ 1, err)) break;
                        mbar_arrive_expect_tx(&s.slot_full[sl], S::TILE);
                        const CUtensorMap* tm = l == 0 ? &tm_k : &tm_v;
                        for (int bx = 0; bx < NB; ++bx)
                            tma_load_3d(s.slot[sl] + bx * BK * 128, tm, &s.slot_full[sl], bx * 64, kb * BK, head);
                        ++fill;
                    }
                }
                if (type == SW_OUT) break;
            }
            // drain: every armed slot's last fill must land before the CTA exits
            for (uint32_t f = fill > NSLOT ? fill - NSLOT : 0; f < fill; ++f)
                mbar_drain(&s.slot_full[f % NSLOT], (f / NSLOT) & 1);
            mbar_drain(&s.q_full, 0);
        }
    } else if (warp == 1) {
        // ============================ MMA issuer 1: S = Q K^T ============================
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(s.q);
            uint32_t fill = 0, pr = 0, g = 0;
            bool ok = WAIT(&s.q_full, 0, err);
            int cg_sweeps = 0;
            for (int sweep = 0; ok; ++sweep) {
                int type;
                if (sweep < n_static || !dynamic) type = static_sweep<BWD>(sweep, cg_sweeps, prm.cg_max_iters, no_max);
                else {
                    if (!(ok = WAIT(&s.p_ready, pr & 1, err))) break;
                    ++pr;
                    type = s.next_type;
                }
                if (type == SW_END) break;
                if (type == SW_CG) ++cg_sweeps;
                const bool two = two_loads<BWD>(type);
                // a sweep with no A'/T/H product: S completes both arrivals of s_full
                const bool lone_s = type == SW_MAX || (!BWD && type == SW_MOMENT);
                for (int kb = 0; kb < nkb; ++kb, ++g) {
                    const uint32_t fk = fill++;
                    if (two) ++fill;                      // the V block of this key block
                    const int sk = fk % NSLOT;
                    const uint32_t b = g & 1;
                    // S buffer b was last used by block g - 2: its coefficients must have been read.  Waited
                    // before the slot: block g - 2's Y product has then consumed every fill before this
                    // block's K (in a two-load sweep the slot's previous fill is block g - 2's V), so the
                    // parity wait below cannot be answered by an older phase of the same slot.
                    if (g >= 2 && !(ok = WAIT(&s.m_free[b], ((g - 2) >> 1) & 1, err))) break;
                    if (!(ok = WAIT(&s.slot_full[sk], (fk / NSLOT) & 1, err))) break;
                    tc_fence_after();
                    gemm_qk<D, false>(tS0 + b * 128, q_addr, smem_u32(s.slot[sk]));
                    umma_commit(&s.s_full[b]);
                    if (lone_s) umma_commit(&s.s_full[b]);
                    if (type == SW_MAX) umma_commit(&s.slot_empty[sk]);   // read by S alone
                }
                if (type == SW_OUT) break;
            }
            umma_commit(&s.final_s);
            mbar_drain(&s.final_s, 0);
        }
    } else if (warp == 3) {
        // ======= MMA issuer 3: A' = P K^T (CG), T = R K^T (output) or H = G V^T (backward) =======
        if (lane == 0) {
            const uint32_t p_addr = smem_u32(s.p), rlo_addr = smem_u32(s.rlo);
            uint32_t fill = 0, pr = 0, g = 0, ga = 0;
            bool ok = true, have_g = false;
            int cg_sweeps = 0;
            for (int sweep = 0; ok; ++sweep) {
                int type;
                bool have_p = false;
                if (sweep < n_static || !dynamic) type = static_sweep<BWD>(sweep, cg_sweeps, prm.cg_max_iters, no_max);
                else {
                    if (!(ok = WAIT(&s.p_ready, pr & 1, err))) break;
                    ++pr;
                    have_p = true;
                    type = s.next_type;
                }
                if (type == SW_END) break;
                if (type == SW_CG) ++cg_sweeps;
                if (type == SW_MAX || (!BWD && type == SW_MOMENT)) {   // no product of this issuer
                    fill += nkb;
                    g += nkb;
                    continue;
                }
                const bool hprod = BWD && (type == SW_MOMENT || type == SW_TBAR);   // H = G V^T
                const bool two = two_loads<BWD>(type);
                // This issuer skips the fills of the sweeps above.  Before its first slot wait it learns
                // that all of them landed, so no parity wait below is answered by an older phase of
                // the same slot; from here on it waits every fill in order.  CG / output: P or R is
                // published after the previous sweep's last Y product.  Backward moments: the
                // elementwise warps have read every S product of the MAX sweep.
                if (!hprod && !have_p) {
                    if (!(ok = WAIT(&s.p_ready, pr & 1, err))) break;
                    ++pr;
                    have_p = true;
                }
                if (hprod && !have_g) {
                    if (!(ok = WAIT(&s.q_full, 0, err)) || !(ok = WAIT(&s.max_done, 0, err))) break;
                    have_g = true;
                }
                for (int kb = 0; kb < nkb; ++kb, ++g) {
                    const uint32_t fk = fill++;
                    const uint32_t fv = two ? fill++ : 0;
                    // the output sweep's T reads only K: its V fills are waited one block late (the
                    // order still holds: V(kb-1) precedes K(kb+1) in the slot that both use), so T
                    // never waits for a V load
                    if (type == SW_OUT && kb > 0 && !(ok = WAIT(&s.slot_full[(fk - 1) % NSLOT], ((fk - 1) / NSLOT) & 1, err))) break;
                    if (!(ok = WAIT(&s.slot_full[fk % NSLOT], (fk / NSLOT) & 1, err))) break;
                    if (hprod && !(ok = WAIT(&s.slot_full[fv % NSLOT], (fv / NSLOT) & 1, err))) break;
                    // A' is single-buffered: the elementwise threads release it as soon as they
                    // have copied the previous block's A' into registers
                    if (ga >= 1 && !(ok = WAIT(&s.a_free, (ga - 1) & 1, err))) break;
                    ++ga;
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(s.slot[(hprod ? fv : fk) % NSLOT]);
                    gemm_qk<D, false>(tA, p_addr, b_addr);
                    // A' = (P_hi + P_lo) K^T where the direction carries a remainder (first tile, backward,
                    // precise form); T = (R_hi + R_lo) K^T where the elementwise threads asked for it
                    const bool lo_prod = type == SW_OUT ? *reinterpret_cast<volatile int*>(&s.out_split) != 0
                                                        : (tile == 0 || BWD || PREC);
                    if (!hprod && lo_prod) gemm_qk<D, true>(tA, rlo_addr, b_addr);
                    umma_commit(&s.s_full[g & 1]);
                }
                if (type == SW_OUT) break;
            }
            umma_commit(&s.final_a);
            mbar_drain(&s.final_a, 0);
        }
    } else if (warp == 2) {
        // ===== MMA issuer 2: Y += M K (moments, CG; backward TBAR) or U V (output) =====
        if (lane == 0) {
            uint32_t fill = 0, pr = 0, g = 0;
            bool ok = WAIT(&s.q_full, 0, err);
            int cg_sweeps = 0;
            for (int sweep = 0; ok; ++sweep) {
                int type;
                if (sweep < n_static || !dynamic) type = static_sweep<BWD>(sweep, cg_sweeps, prm.cg_max_iters, no_max);
                else {
                    if (!(ok = WAIT(&s.p_ready, pr & 1, err))) break;
                    ++pr;
                    type = s.next_type;
                }
                if (type == SW_END) break;
                if (type == SW_CG) ++cg_sweeps;
                const bool two = two_loads<BWD>(type);
                const uint32_t ty_acc = tY;
                for (int kb = 0; kb < nkb; ++kb, ++g) {
                    const uint32_t fk = fill++;
                    const uint32_t fv = two ? fill++ : 0;
                    const uint32_t b = g & 1;
                    if (!(ok = WAIT(&s.ew_done[b], (g >> 1) & 1, err))) break;
                    if (type != SW_MAX) {
                        if (type == SW_OUT && !(ok = WAIT(&s.slot_full[fv % NSLOT], (fv / NSLOT) & 1, err))) break;
                        tc_fence_after();
                        const uint32_t fsrc = type == SW_OUT ? fv : fk;   // V for the output, K otherwise
                        if (BWD || (PREC && type != SW_OUT))
                            gemm_y_split<D>(ty_acc, tS0 + b * 128, smem_u32(s.slot[fsrc % NSLOT]), kb > 0);
                        else gemm_y<D>(ty_acc, tS0 + b * 128, smem_u32(s.slot[fsrc % NSLOT]), kb > 0);
                        umma_commit(&s.slot_empty[fsrc % NSLOT]);
                        // the other block of a two-block sweep (the output's K, the backward's V): its
                        // products completed before the elementwise warps could finish this block
                        if (two) umma_commit(&s.slot_empty[(type == SW_OUT ? fk : fv) % NSLOT]);
                        if (kb == nkb - 1) umma_commit(&s.y_done);
                    }
                    umma_commit(&s.m_free[b]);
                }
                if (type == SW_OUT) break;
            }
            umma_commit(&s.final_y);
            mbar_drain(&s.final_y, 0);
        }
    }
    } else {
        // =========================== elementwise + CG warps ===========================
        setmaxnreg_inc216();
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int half = (warp - 4) >> 2;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const int i = tile * BQ + row;
        const bool row_ok = i < n;
        const bool tile_full = (tile + 1) * BQ <= n;     // every row of the tile exists
        // the first tile holds the rows i < d whose key scatter is rank-deficient: there the CG
        // direction is kept to about 22 bits (hi + lo fp16 halves, one extra MMA per CG block);
        // the precise form does so in every tile
        const bool split_p = BWD || PREC || tile == 0;
        const size_t row_g = ((size_t)head * n + (row_ok ? i : 0)) * D + half * DH;
        // tile-transposed fp32 scratch: coordinate e of this thread's row at [e * BQ] (coalesced)
        const size_t tbase = ((size_t)(head * prm.n_tiles + tile) * D + half * DH) * BQ + row;
        // CG iterate x = rho': shared memory ([coordinate][row], rlo for the first half of the
        // coordinates and xb for the second), except in the first tile, whose rlo holds P_lo
        // and whose x uses the global scratch (same layout)
        float* xt = split_p ? prm.xs + tbase
                            : reinterpret_cast<float*>(half == 0 ? s.rlo : s.xb) + row;
        float* kbt = prm.kbar + tbase;          // kbar
        Xch xch{s.xch, 0, half, row};

        const float mk = __uint_as_float(prm.hdr->maxabs[1]);
        const int eq = scale_exp(__uint_as_float(prm.hdr->maxabs[0]));
        const int ek = scale_exp(mk);
        const int ev = scale_exp(__uint_as_float(prm.hdr->maxabs[2]));
        const float c_log2 = prm.tau * 1.4426950408889634f * pow2i(-(eq + ek));
        uint32_t g = 0, yd = 0;
        bool ok = WAIT(&s.q_full, 0, err);
        const float a_none[64] = {};                   // placeholder operand of the moment sweep
        // last valid key column of block kb for this row (-1: none)
        auto lim_of = [&](int kb) { return row_ok ? (kb < tile ? BK - 1 : i - kb * BK) : -1; };
        auto wait_s = [&](uint32_t gg) {
            const bool r = WAIT(&s.s_full[gg & 1], (gg >> 1) & 1, err);
            tc_fence_after();
            return r;
        };
        // Per-block signals are one arrive per warp (not per thread): fewer atomics on the
        // barrier word the MMA thread polls.
        auto done_block = [&](uint32_t gg) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.ew_done[gg & 1]);
        };
        auto release_a = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.a_free);
        };
        // P/R tile written: every thread fences its generic-proxy writes for the async proxy, the
        // elementwise threads meet, and one thread arrives.  With WITH_V the meeting also sums v over
        // the row's two halves (an exchange without a barrier of its own); returns that sum.
        auto publish_p = [&](int next_type, bool with_v = false, float v = 0.f) {
            const float* b = with_v ? xch.put(v) : nullptr;
            fence_proxy_async_smem();
            named_bar_sync(EW_BAR, NEW);
            if (tid == 128) {
                s.next_type = next_type;
                mbar_arrive(&s.p_ready);
            }
            return with_v ? v + xch.take(b) : 0.f;
        };
        auto wait_y = [&]() {
            const bool r = WAIT(&s.y_done, yd & 1, err);
            ++yd;
            tc_fence_after();
            return r;
        };

        // the moment sweep's key norms (forward): this half's 64 keys of every block
        const float* kn_row = prm.knorm + (size_t)head * (prm.n_tiles * BQ) + half * 64;
        if (!BWD && !PROBE) prefetch_knorm64(kn_row, 0, lane);

        // largest valid entry of one 32-key chunk of S (columns col0 .. col0 + 31; -inf for none)
        auto vmax32 = [&](const float (&v)[32], bool masked, int col0, int lim) {
            float m = -INFINITY;
            if (!masked) {
#pragma unroll
                for (int j = 0; j < 32; ++j) m = fmaxf(m, v[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) m = fmaxf(m, (col0 + j <= lim) ? v[j] : -INFINITY);
            }
            return m;
        };
        // The row maximum m2 (log2 units).  The moment sweep's weights are w 2^wsc in fp16 relative
        // to a reference mref2: the maximum itself after a MAX sweep (wsc = 14, w <= 1); without one,
        // the first block's maximum, with 2^6 of headroom for the later blocks (wsc = 8), the exact
        // maximum taken along the sweep.
        float m2 = 0.f, mref2 = 0.f;
        int wsc = 14;
        float mx = -INFINITY;
        int jmx = 0;                        // backward: first key index attaining the maximum
        if (no_max) {
            ok = ok && wait_s(g);           // the moment sweep's first block (waited again there)
            const uint32_t tS = tS0 + (g & 1) * 128 + lane_off + half * 64;
            float v0[32], v1[32];
            tmem_ld32(tS, v0);
            tmem_ld32(tS + 32, v1);
            tmem_ld_wait();
            const int lim = lim_of(0);
            const bool masked = !(tile_full && 0 < tile);
            const float bm = xch.max(fmaxf(vmax32(v0, masked, half * 64, lim), vmax32(v1, masked, half * 64 + 32, lim)));
            mref2 = (row_ok && bm > -INFINITY) ? bm * c_log2 : 0.f;
            wsc = 8;
        } else {
        // ---------------- MAX sweep ----------------
        for (int kb = 0; kb < nkb; ++kb, ++g) {
            ok = ok && wait_s(g);
            const uint32_t tS = tS0 + (g & 1) * 128 + lane_off + half * 64;
            float v0[32], v1[32];
            tmem_ld32(tS, v0);
            tmem_ld32(tS + 32, v1);
            tmem_ld_wait();
            done_block(g);
            const int lim = lim_of(kb);
            if (BWD) {                      // columns in increasing order: a strict > keeps the first
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (half * 64 + j <= lim && v0[j] > mx) { mx = v0[j]; jmx = kb * BK + half * 64 + j; }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (half * 64 + 32 + j <= lim && v1[j] > mx) { mx = v1[j]; jmx = kb * BK + half * 64 + 32 + j; }
            } else if (tile_full && kb < tile) {
#pragma unroll
                for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fmaxf(v0[j], v1[j]));
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    mx = fmaxf(mx, (half * 64 + j <= lim) ? v0[j] : -INFINITY);
                    mx = fmaxf(mx, (half * 64 + 32 + j <= lim) ? v1[j] : -INFINITY);
                }
            }
        }
        if (BWD) {                          // half 0 holds the lower columns of every block
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.max_done);
            const float omx = xch.swap(mx);
            const int ojm = __float_as_int(xch.swap(__int_as_float(jmx)));
            if (omx > mx || (omx == mx && ojm < jmx)) { mx = omx; jmx = ojm; }
        } else {
            mx = xch.max(mx);
        }
        m2 = row_ok ? mx * c_log2 : 0.f;
        mref2 = m2;
        }
        float mrun = -INFINITY;             // no MAX sweep: the largest valid S entry so far

        // ---------------- MOMENT sweep ----------------
        uint64_t om_part = 0;              // two fp32 partial sums (bit pattern 0 = +0.0f, +0.0f)
        uint64_t wh_part = 0;              // backward: sum of w h
        uint64_t tk_part = 0;              // sum of w |k|^2 (the key scatter's trace, below)
        for (int kb = 0; kb < nkb; ++kb, ++g) {
            if (!BWD && !PROBE && kb + 1 < nkb) prefetch_knorm64(kn_row, (kb + 1) * BK, lane);
            ok = ok && wait_s(g);
            const uint32_t tS = tS0 + (g & 1) * 128 + lane_off + half * 64;
            const int lim = lim_of(kb);
            const bool masked = !(tile_full && kb < tile);
            float v[32], kn[32];
            uint32_t pk[16];
            if (BWD) {
                float a[64];
                tmem_ld32(tA + lane_off + half * 64, *reinterpret_cast<float(*)[32]>(&a[0]));
                tmem_ld32(tA + lane_off + half * 64 + 32, *reinterpret_cast<float(*)[32]>(&a[32]));
                tmem_ld32(tS, v);
                tmem_ld_wait();
                release_a();
                uint32_t pl[16];            // hi + lo weights, split layout (gemm_y_split)
                if (masked) coef_chunk_wh<true, 0>(v, a, c_log2, mref2 - (float)wsc, half * 64, lim, om_part, wh_part, pk, pl);
                else coef_chunk_wh<false, 0>(v, a, c_log2, mref2 - (float)wsc, 0, 0, om_part, wh_part, pk, pl);
                tmem_st16(tS, pk);
                tmem_st16(tS + 16, pl);
                tmem_ld32(tS + 32, v);
                tmem_ld_wait();
                if (masked) coef_chunk_wh<true, 1>(v, a, c_log2, mref2 - (float)wsc, half * 64 + 32, lim, om_part, wh_part, pk, pl);
                else coef_chunk_wh<false, 1>(v, a, c_log2, mref2 - (float)wsc, 0, 0, om_part, wh_part, pk, pl);
                tmem_st16(tS + 32, pk);
                tmem_st16(tS + 48, pl);
            } else if constexpr (PREC) {    // hi + lo weights, split layout (gemm_y_split)
                uint32_t pl[16];
                tmem_ld32(tS, v);
                load_knorm32(kn_row, kb * BK, kn);
                tmem_ld_wait();
                if (no_max) mrun = fmaxf(mrun, vmax32(v, masked, half * 64, lim));
                if (masked) coef_chunk_wk<true, true>(v, kn, c_log2, mref2 - (float)wsc, half * 64, lim, om_part, tk_part, pk, pl);
                else coef_chunk_wk<false, true>(v, kn, c_log2, mref2 - (float)wsc, 0, 0, om_part, tk_part, pk, pl);
                tmem_st16(tS, pk);
                tmem_st16(tS + 16, pl);
                tmem_ld32(tS + 32, v);
                load_knorm32(kn_row, kb * BK + 32, kn);
                tmem_ld_wait();
                if (no_max) mrun = fmaxf(mrun, vmax32(v, masked, half * 64 + 32, lim));
                if (masked) coef_chunk_wk<true, true>(v, kn, c_log2, mref2 - (float)wsc, half * 64 + 32, lim, om_part, tk_part, pk, pl);
                else coef_chunk_wk<false, true>(v, kn, c_log2, mref2 - (float)wsc, 0, 0, om_part, tk_part, pk, pl);
                tmem_st16(tS + 32, pk);
                tmem_st16(tS + 48, pl);
            } else if constexpr (PROBE) {   // weights only (the probe form takes no key norms)
                tmem_ld32(tS, v);
                tmem_ld_wait();
                if (no_max) mrun = fmaxf(mrun, vmax32(v, masked, half * 64, lim));
                if (masked) coef_chunk<true, false, 0>(v, a_none, c_log2, mref2 - (float)wsc, 0.f, 0.f, half * 64, lim, om_part, pk);
                else coef_chunk<false, false, 0>(v, a_none, c_log2, mref2 - (float)wsc, 0.f, 0.f, 0, 0, om_part, pk);
                tmem_st16(tS, pk);
                tmem_ld32(tS + 32, v);
                tmem_ld_wait();
                if (no_max) mrun = fmaxf(mrun, vmax32(v, masked, half * 64 + 32, lim));
                if (masked) coef_chunk<true, false, 0>(v, a_none, c_log2, mref2 - (float)wsc, 0.f, 0.f, half * 64 + 32, lim, om_part, pk);
                else coef_chunk<false, false, 0>(v, a_none, c_log2, mref2 - (float)wsc, 0.f, 0.f, 0, 0, om_part, pk);
                tmem_st16(tS + 16, pk);
            } else {
                tmem_ld32(tS, v);
                load_knorm32(kn_row, kb * BK, kn);
                tmem_ld_wait();
                if (no_max) mrun = fmaxf(mrun, vmax32(v, masked, half * 64, lim));
                if (masked) coef_chunk_wk<true, false>(v, kn, c_log2, mref2 - (float)wsc, half * 64, lim, om_part, tk_part, pk);
                else coef_chunk_wk<false, false>(v, kn, c_log2, mref2 - (float)wsc, 0, 0, om_part, tk_part, pk);
                tmem_st16(tS, pk);
                tmem_ld32(tS + 32, v);
                load_knorm32(kn_row, kb * BK + 32, kn);
                tmem_ld_wait();
                if (no_max) mrun = fmaxf(mrun, vmax32(v, masked, half * 64 + 32, lim));
                if (masked) coef_chunk_wk<true, false>(v, kn, c_log2, mref2 - (float)wsc, half * 64 + 32, lim, om_part, tk_part, pk);
                else coef_chunk_wk<false, false>(v, kn, c_log2, mref2 - (float)wsc, 0, 0, om_part, tk_part, pk);
                tmem_st16(tS + 16, pk);
            }
            tmem_st_wait();
            done_block(g);
        }
        ok = ok && wait_y();
        const float om_all = xch.sum(f2_total(om_part));      // every elementwise thread joins the exchange
        const float tk_all = xch.sum(f2_total(tk_part));      // sum_j w_j |k_j|^2, weights in units of 2^-wsc
        float wunit = pow2i(-14);                             // the moment sums' unit, relative to the maximum
        if (no_max) {
            const float mt = xch.max(mrun);
            m2 = (row_ok && mt > -INFINITY) ? mt * c_log2 : 0.f;
            // a weight 2^(m2 - mref2 + 8) in fp16 stays below 2^15.5 (65504 is the largest finite value):
            // past that the tile's moments may hold an overflow, and its results are redone with a MAX sweep
            const bool over = ew_any(row_ok && m2 - mref2 > 7.5f);
            if (tid == 128) prm.tile_flag[(size_t)head * prm.n_tiles + tile] = over ? 1 : 0;
            wunit = pow2i(-wsc) * exp2f(mref2 - m2);
        }
        const float omega = row_ok ? om_all * wunit : 1.f;
        const float inv_om = 1.f / omega;
        const float lam_n = prm.lambda * inv_om;
        // backward: hbar in units of H (dout.v 2^(eg+ev)); TBAR's right-hand side, in res
        const int eg = BWD ? scale_exp(__uint_as_float(prm.hdr->maxabs[3])) : 0;
        const float wh_all = BWD ? xch.sum(f2_total(wh_part)) : 0.f;
        const float hbar_a = (BWD && row_ok && om_all > 0.f) ? wh_all / om_all : 0.f;

        // kbar, delta, CG initialisation (this thread: coordinates half*DH .. half*DH+DH-1)
        float res[DH];
        float gamma, rn0;
        bool active;
        int iters = 0;
        int sp = 0, sM = 0;                  // scale exponents of the direction tile and of M
        float kp_acc = 0.f, offM = 0.f;      // per-row parameters of the next CG sweep
        // kbar.res (a dot product each iteration) and kbar.p (by recurrence, p = res + beta p_old),
        // whole row.  kbar.p only centres the per-pair coefficients (the kbar msum term of the
        // update cancels any offset exactly), so it need not match the rounded direction bit for
        // bit; kbar.res is recomputed, not updated, because a converging residual cancels.
        float kbr = 0.f, kpx = 0.f;
        int cg_sweeps = 0;
        // Bound for the fp16 scales of the per-pair coefficients: |w_j (k_j - kbar).u| <= cbound |u|_2.
        // With the key scatter's trace T = sum_j w_j |k_j - kbar|^2 = sum_j w_j |k_j|^2 - omega |kbar|^2
        // and w_j <= 1, w_j |k_j - kbar| <= sqrt(w_j |k_j - kbar|^2) <= sqrt(T).
        // T is taken with 2^-9 of sum_j w_j |k_j|^2 added (it covers the cancellation, and kbar's error
        // from its fp16 weights), and 2^-8 |kbar| covers the rounded direction's kbar.u offset.  Rows whose
        // weights sit on a few keys far from the others keep their coefficients in fp16's normal range,
        // which a bound from max|k| alone does not.
        float cbound = 0.f, tr_om = 0.f;     // tr_om: the trace over omega, sum_j wbar_j |k_j - kbar|^2
        auto set_cbound = [&](float kk) {
            if constexpr (BWD) {   // hi + lo coefficients throughout: the bound from max|k| suffices
                cbound = (2.f * sqrtf((float)D) * mk + sqrtf(kk) * pow2i(-8)) * 1.001f;
                return;
            }
            const float tsum = row_ok ? tk_all * wunit : 0.f;
            const float tr = fmaxf(tsum - omega * kk, 0.f) + tsum * pow2i(-9);
            cbound = (sqrtf(tr) + sqrtf(kk) * pow2i(-8)) * 1.001f;
            tr_om = tr * inv_om;
        };
        // New direction p = res + beta p_old, stored in the direction tile as fp16 x 2^sp (hi, and lo when
        // SPLITC, the direction's form), in one pass.  MPB (row-level) bounds |p|_2, hence max|p|, so the
        // scale needs no exchange of the row maximum: |p|_2 <= |res|_2 + |beta| |p_old|_2, with |p_old|_2
        // carried as its own bound (pn2).  With XUPD the pass also updates this thread's x = rho' to
        // x + ALPHA p_old (XO: a previous x exists; else it starts from 0), p_old being the direction of the
        // sweep just finished.  The scale sM of the
        // next sweep's coefficients follows from the same bound; kbar.p (kp_acc) is set by set_kp once
        // kbar.res of the whole row is known.  The fp16-only form reads every p_old group before it
        // writes any (one batch of shared loads instead of a load per group behind the stores).
        float pn2 = 0.f;
#define LLA_SET_DIRECTION(BETA, KEEP, XUPD, ALPHA, XO, SPLITC, MPB)                                        \
        {                                                                                                  \
            const float osc_ = pow2i(-sp);                                                                 \
            const uint64_t b2_ = f2_pack((BETA), (BETA));                                                  \
            const int sp_new_ = min(scale_exp((MPB) * 1.001f), 100 - ek);   /* keeps 2^(sp+ek) finite */  \
            const uint64_t nsc2_ = f2_pack(pow2i(sp_new_), pow2i(sp_new_));                                \
            if (!(SPLITC)) {                                                                               \
                uint4 ph_[DH / 8];                                                                         \
                _Pragma("unroll") for (int g_ = 0; g_ < DH / 8; ++g_)                                      \
                    ph_[g_] = (KEEP) ? *reinterpret_cast<const uint4*>(tile_half(s.p, row, half * DH + 8 * g_)) \
                                     : make_uint4(0u, 0u, 0u, 0u);                                         \
                _Pragma("unroll") for (int g_ = 0; g_ < DH / 8; ++g_) {                                    \
                    const int e0 = 8 * g_;                                                                 \
                    float po_[8];                                                                          \
                    dir8_hi(ph_[g_], osc_, po_);                                                           \
                    if (XUPD) {                                                                            \
                        _Pragma("unroll") for (int u = 0; u < 8; ++u)                                      \
                            xt[(e0 + u) * BQ] = fmaf((ALPHA), po_[u], (XO) ? xt[(e0 + u) * BQ] : 0.f);      \
                    }                                                                                      \
                    uint32_t* hw_ = reinterpret_cast<uint32_t*>(&ph_[g_]);                                 \
                    _Pragma("unroll") for (int u = 0; u < 8; u += 2) {                                     \
                        float x0_, x1_;                                                                    \
                        f2_unpack(f2_mul(f2_fma(b2_, f2_pack(po_[u], po_[u + 1]),                          \
                                                f2_pack(res[e0 + u], res[e0 + u + 1])), nsc2_), x0_, x1_); \
                        hw_[u >> 1] = pack_half2(x0_, x1_);                                                \
                    }                                                                                      \
                }                                                                                          \
                _Pragma("unroll") for (int g_ = 0; g_ < DH / 8; ++g_)                                      \
                    *reinterpret_cast<uint4*>(tile_half(s.p, row, half * DH + 8 * g_)) = ph_[g_];          \
            } else                                                                                         \
            _Pragma("unroll") for (int e0 = 0; e0 < DH; e0 += 8) {                                         \
                float po_[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};                                   \
                if (KEEP) load_dir8(s.p, s.rlo, SPLITC, row, half * DH + e0, osc_, po_);                   \
                if (XUPD) {                                                                                \
                    _Pragma("unroll") for (int u = 0; u < 8; ++u)                                          \
                        xt[(e0 + u) * BQ] = fmaf((ALPHA), po_[u], (XO) ? xt[(e0 + u) * BQ] : 0.f);          \
                }                                                                                          \
                uint4 hk_, lk_;                                                                            \
                uint32_t* hw_ = reinterpret_cast<uint32_t*>(&hk_);                                         \
                uint32_t* lw_ = reinterpret_cast<uint32_t*>(&lk_);                                         \
                _Pragma("unroll") for (int u = 0; u < 8; u += 2) {                                         \
                    float x0_, x1_;                                                                        \
                    f2_unpack(f2_mul(f2_fma(b2_, f2_pack(po_[u], po_[u + 1]),                              \
                                            f2_pack(res[e0 + u], res[e0 + u + 1])), nsc2_), x0_, x1_);     \
                    hw_[u >> 1] = pack_half2(x0_, x1_);                                                    \
                    const float2 hf_ = __half22float2(*reinterpret_cast<const __half2*>(&hw_[u >> 1]));   \
                    lw_[u >> 1] = pack_half2(x0_ - hf_.x, x1_ - hf_.y);                                    \
                }                                                                                          \
                *reinterpret_cast<uint4*>(tile_half(s.p, row, half * DH + e0)) = hk_;                      \
                if (SPLITC) *reinterpret_cast<uint4*>(tile_half(s.rlo, row, half * DH + e0)) = lk_;        \
            }                                                                                              \
            sp = sp_new_;                                                                                  \
            pn2 = (MPB);                                                                                   \
            sM = scale_exp(cbound * (MPB));                                                                \
            offM = m2 - (float)sM + (float)sp + (float)ek;                                                 \
        }
        // kbar.p of the new direction by recurrence (p = res + beta p_old), in the units of the A' product
        auto set_kp = [&](float beta) {
            kpx = kbr + beta * kpx;
            kp_acc = kpx * pow2i(sp + ek);
        };
        if constexpr (BWD) {
            // kbar from the moment sweep's Y, before the TBAR sweep reuses the accumulator
            {
                const float ysc = wunit * pow2i(-ek) * inv_om;
                float kk = 0.f;
#pragma unroll
                for (int c = 0; c < DH / 32; ++c) {
                    float v[32];
                    tmem_ld32(tY + lane_off + half * DH + c * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        kbt[(c * 32 + j) * BQ] = v[j] * ysc;
                        kk = fmaf(v[j] * ysc, v[j] * ysc, kk);
                    }
                }
                set_cbound(xch.sum(row_ok ? kk : 0.f));
            }
            // ---------------- TBAR sweep: Y = sum_j w_j (h_j - hbar) k_j ----------------
            // coefficient w (h - hbar) 2^sT; |h - hbar| <= 2 D max|dout| max|v| fixes sT
            const int sT = scale_exp(2.f * (float)D * __uint_as_float(prm.hdr->maxabs[3]) *
                                     __uint_as_float(prm.hdr->maxabs[2]) * 1.001f);
            const float offT = m2 - (float)sT + (float)(eg + ev);
            uint64_t ts_part = 0;
            for (int kb = 0; kb < nkb; ++kb, ++g) {
                ok = ok && wait_s(g);
                const uint32_t tS = tS0 + (g & 1) * 128 + lane_off + half * 64;
                const uint32_t tAh = tA + lane_off + half * 64;
                const int lim = lim_of(kb);
                const bool masked = !(tile_full && kb < tile);
                float a[64], v[32];
                uint32_t pk[16];
                tmem_ld32(tAh, *reinterpret_cast<float(*)[32]>(&a[0]));
                tmem_ld32(tAh + 32, *reinterpret_cast<float(*)[32]>(&a[32]));
                tmem_ld32(tS, v);
                tmem_ld_wait();
                release_a();
                uint32_t pl[16];
                if (masked) coef_chunk<true, true, 0, true>(v, a, c_log2, offT, -hbar_a, 1.f, half * 64, lim, ts_part, pk, pl);
                else coef_chunk<false, true, 0, true>(v, a, c_log2, offT, -hbar_a, 1.f, 0, 0, ts_part, pk, pl);
                tmem_st16(tS, pk);
                tmem_st16(tS + 16, pl);
                tmem_ld32(tS + 32, v);
                tmem_ld_wait();
                if (masked) coef_chunk<true, true, 1, true>(v, a, c_log2, offT, -hbar_a, 1.f, half * 64 + 32, lim, ts_part, pk, pl);
                else coef_chunk<false, true, 1, true>(v, a, c_log2, offT, -hbar_a, 1.f, 0, 0, ts_part, pk, pl);
                tmem_st16(tS + 32, pk);
                tmem_st16(tS + 48, pl);
                tmem_st_wait();
                done_block(g);
            }
            ok = ok && wait_y();
            // right-hand side tbar = [Y 2^-(sT+ek) - kbar (sum of coefficients) 2^-sT] / omega
            const float tsum = xch.sum(f2_total(ts_part));
            const float tysc = pow2i(-(sT + ek)) * inv_om, tksc = tsum * pow2i(-sT) * inv_om;
            float gp = 0.f, kr = 0.f;
#pragma unroll
            for (int c = 0; c < DH / 32; ++c) {
                float v[32];
                tmem_ld32(tY + lane_off + half * DH + c * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float kb_ = kbt[(c * 32 + j) * BQ];
                    const float r_ = row_ok ? fmaf(v[j], tysc, -kb_ * tksc) : 0.f;
                    res[c * 32 + j] = r_;
                    gp = fmaf(r_, r_, gp);
                    kr = fmaf(kb_, r_, kr);
                }
            }
            gamma = xch.sum(gp);
            kbr = xch.sum(kr);
            rn0 = sqrtf(gamma);
            active = row_ok && gamma > 0.f && !(sqrtf(gamma) <= prm.cg_tol * rn0);
            LLA_SET_DIRECTION(0.f, false, false, 0.f, false, split_p, sqrtf(gamma));
            set_kp(0.f);
        } else {
            float kv[DH];
            const float ysc = wunit * pow2i(-ek) * inv_om;
            const float qsc = pow2i(-eq);
#pragma unroll
            for (int c = 0; c < DH / 32; ++c) {
                float v[32];
                tmem_ld32(tY + lane_off + half * DH + c * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    const uint4 qr = *reinterpret_cast<const uint4*>(tile_half(s.q, row, half * DH + c * 32 + j));
                    const __half* qh = reinterpret_cast<const __half*>(&qr);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float kb_ = v[j + u] * ysc;
                        kv[c * 32 + j + u] = kb_;
                        kbt[(c * 32 + j + u) * BQ] = kb_;
                        res[c * 32 + j + u] = row_ok ? kb_ - __half2float(qh[u]) * qsc : 0.f;
                    }
                }
            }
            float gp = 0.f, kr = 0.f, kk = 0.f;
#pragma unroll
            for (int e = 0; e < DH; ++e) {
                gp = fmaf(res[e], res[e], gp);
                kr = fmaf(kv[e], res[e], kr);
                kk = fmaf(kv[e], kv[e], kk);
            }
            gamma = xch.sum(gp);
            kbr = xch.sum(kr);
            set_cbound(xch.sum(row_ok ? kk : 0.f));
            rn0 = sqrtf(gamma);
            active = row_ok && gamma > 0.f && !(sqrtf(gamma) <= prm.cg_tol * rn0);
            LLA_SET_DIRECTION(0.f, false, false, 0.f, false, split_p, sqrtf(gamma));
            set_kp(0.f);
        }

        // ---------------- CG sweeps ----------------
        const float* kr_pend = nullptr;        // this half's kbar.res of the last update, in the exchange buffer
        float beta_pend = 0.f;
        while (true) {                         // uniform across the elementwise threads
            bool go;
            if (!dynamic) go = cg_sweeps < prm.cg_max_iters;
            else go = ew_any(active) && cg_sweeps < prm.cg_max_iters;
            if (!go) break;
            // the publishing barrier also sums kbar.res over the row, for kbar.p of the new direction
            publish_p(SW_CG);
            if (cg_sweeps > 0) {
                kbr = xch.take(kr_pend) + kr_pend[half * BQ + row];
                set_kp(beta_pend);
            }
            ++cg_sweeps;
            uint64_t msum_part = 0;
            for (int kb = 0; kb < nkb; ++kb, ++g) {
                ok = ok && wait_s(g);
                const uint32_t tS = tS0 + (g & 1) * 128 + lane_off + half * 64;
                const uint32_t tAh = tA + lane_off + half * 64;
                const int lim = lim_of(kb);
                const bool masked = !(tile_full && kb < tile);
                float a[64], v[32];
                uint32_t pk[16];
                tmem_ld32(tAh, *reinterpret_cast<float(*)[32]>(&a[0]));
                tmem_ld32(tAh + 32, *reinterpret_cast<float(*)[32]>(&a[32]));
                tmem_ld32(tS, v);
                tmem_ld_wait();
                release_a();
                if constexpr (SPLITM) {   // hi + lo coefficients, split layout (gemm_y_split)
                    uint32_t pl[16];
                    if (masked) coef_chunk<true, true, 0, true>(v, a, c_log2, offM, -kp_acc, 1.f, half * 64, lim, msum_part, pk, pl);
                    else coef_chunk<false, true, 0, true>(v, a, c_log2, offM, -kp_acc, 1.f, 0, 0, msum_part, pk, pl);
                    tmem_st16(tS, pk);
                    tmem_st16(tS + 16, pl);
                    tmem_ld32(tS + 32, v);
                    tmem_ld_wait();
                    if (masked) coef_chunk<true, true, 1, true>(v, a, c_log2, offM, -kp_acc, 1.f, half * 64 + 32, lim, msum_part, pk, pl);
                    else coef_chunk<false, true, 1, true>(v, a, c_log2, offM, -kp_acc, 1.f, 0, 0, msum_part, pk, pl);
                    tmem_st16(tS + 32, pk);
                    tmem_st16(tS + 48, pl);
                } else {
                    if (masked) coef_chunk<true, true, 0>(v, a, c_log2, offM, -kp_acc, 1.f, half * 64, lim, msum_part, pk);
                    else coef_chunk<false, true, 0>(v, a, c_log2, offM, -kp_acc, 1.f, 0, 0, msum_part, pk);
                    tmem_st16(tS, pk);
                    tmem_ld32(tS + 32, v);
                    tmem_ld_wait();
                    if (masked) coef_chunk<true, true, 1>(v, a, c_log2, offM, -kp_acc, 1.f, half * 64 + 32, lim, msum_part, pk);
                    else coef_chunk<false, true, 1>(v, a, c_log2, offM, -kp_acc, 1.f, 0, 0, msum_part, pk);
                    tmem_st16(tS + 16, pk);
                }
                tmem_st_wait();
                done_block(g);
            }
            // kbar for the update, loaded while the sweep's last Y products run
            float kv[DH];
#pragma unroll
            for (int e = 0; e < DH; ++e) kv[e] = kbt[e * BQ];
            ok = ok && wait_y();
            // ---- CG update: (C/omega) p = [Y 2^-(sM+ek) - kbar msum 2^-sM] / omega + (lambda/omega) p
            const float msum = xch.sum(f2_total(msum_part));
            const float ysc = pow2i(-(sM + ek)) * inv_om;
            const float msc = msum * pow2i(-sM) * inv_om;
            const float psc = pow2i(-sp);
            const uint32_t ty = tY + lane_off + half * DH;
            // first pass: Cp and p.Cp; Cp goes to the A' columns of TMEM, idle until the next
            // sweep's first A' product (which waits for this update's direction)
            const uint32_t tcp = tA + lane_off + half * 64;
            uint64_t pcp2 = 0;
#define LLA_CG_CHUNK(C, SPLITC)                                                                            \
            if constexpr ((C) * 16 < DH) {                                                                 \
                float cp_[16];                                                                             \
                uint32_t cb_[16];                                                                          \
                cg_apply_chunk<C, DH, true, SPLITC>(ty, s.p, s.rlo, row, half * DH, kv, ysc, msc, lam_n,    \
                                                    psc, cp_, pcp2);                                       \
                _Pragma("unroll") for (int j = 0; j < 16; ++j) cb_[j] = __float_as_uint(cp_[j]);          \
                tmem_st16(tcp + (C) * 16, cb_);                                                            \
            }
            if (split_p) {
                LLA_CG_CHUNK(0, true);
                LLA_CG_CHUNK(1, true);
                LLA_CG_CHUNK(2, true);
                LLA_CG_CHUNK(3, true);
            } else {
                LLA_CG_CHUNK(0, false);
                LLA_CG_CHUNK(1, false);
                LLA_CG_CHUNK(2, false);
                LLA_CG_CHUNK(3, false);
            }
#undef LLA_CG_CHUNK
            tmem_st_wait();
            const float pcp = xch.sum(f2_total(pcp2));
            const bool upd = active && pcp > 0.f;
            const float alpha = upd ? gamma / pcp : 0.f;
            // second pass: res -= alpha Cp, res.res, kbar.res
            uint64_t g22 = 0, kr2 = 0;
            {
                const uint64_t na2 = f2_pack(-alpha, -alpha);
                float c0[16], c1[16];
                tmem_ld16(tcp, c0);
                tmem_ld_wait();
#define LLA_CG_STEP(C, CC, CN)                                                                             \
                if constexpr ((C) * 16 < DH) {                                                             \
                    if constexpr (((C) + 1) * 16 < DH) tmem_ld16(tcp + ((C) + 1) * 16, CN);                \
                    _Pragma("unroll") for (int j = 0; j < 16; j += 2) {                                    \
                        uint64_t r2 = f2_pack(res[(C) * 16 + j], res[(C) * 16 + j + 1]);                   \
                        if (upd) r2 = f2_fma(na2, f2_pack(CC[j], CC[j + 1]), r2);                          \
                        f2_unpack(r2, res[(C) * 16 + j], res[(C) * 16 + j + 1]);                           \
                        g22 = f2_fma(r2, r2, g22);                                                         \
                        kr2 = f2_fma(f2_pack(kv[(C) * 16 + j], kv[(C) * 16 + j + 1]), r2, kr2);            \
                    }                                                                                      \
                    tmem_ld_wait();                                                                        \
                }
                LLA_CG_STEP(0, c0, c1);
                LLA_CG_STEP(1, c1, c0);
                LLA_CG_STEP(2, c0, c1);
                LLA_CG_STEP(3, c1, c0);
#undef LLA_CG_STEP
            }
            const float g2 = xch.sum(f2_total(g22));       // res.res
            float beta = 0.f;
            if (upd) {
                beta = g2 / gamma;
                gamma = g2;
                ++iters;
                if (gamma == 0.f || sqrtf(gamma) <= prm.cg_tol * rn0) active = false;
            } else {
                active = false;
            }
            if (!active) {
#pragma unroll
                for (int e = 0; e < DH; ++e) res[e] = 0.f;   // finished rows keep a zero direction
                beta = 0.f;
            }
            // this half's kbar.res goes to the exchange buffer now and is read after the next publishing
            // barrier.  Buffers alternate: this one last held the p.Cp exchange, which the partner read
            // before the res.res barrier above; the next write to it comes after the following sweep's
            // y_done, which needs both halves past the read.
            kr_pend = xch.put(active ? f2_total(kr2) : 0.f);
            beta_pend = beta;
            const float mpb = active ? sqrtf(gamma) + fabsf(beta) * pn2 : 0.f;   // bounds |p_new|_2
            // the form as a constant: the loops over the coordinates carry no branch on it
            const bool have_xo = cg_sweeps > 1;
            if (split_p) LLA_SET_DIRECTION(beta, true, true, alpha, have_xo, true, mpb)
            else LLA_SET_DIRECTION(beta, true, true, alpha, have_xo, false, mpb)
        }

        if constexpr (BWD) {
            // ---------------- backward: y and the per-row record ----------------
            // rho' = rho omega/denom from the forward's outputs; kbar.rho', kbar.y, rho'.y
            const bool have_x = row_ok && cg_sweeps > 0;   // no sweep ran: y = 0
            const float den = row_ok ? prm.denom_in[(size_t)head * n + i] : 1.f;
            const float rp_scale = omega / den;
            float kr = 0.f, ky = 0.f, ry = 0.f;
#pragma unroll
            for (int e0 = 0; e0 < DH; e0 += 4) {
                float xv[4], rv[4];
                const float4 r4 = row_ok ? *reinterpret_cast<const float4*>(prm.rho_in + row_g + e0)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                rv[0] = r4.x * rp_scale; rv[1] = r4.y * rp_scale; rv[2] = r4.z * rp_scale; rv[3] = r4.w * rp_scale;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    xv[u] = have_x ? xt[(e0 + u) * BQ] : 0.f;
                    const float kb_ = kbt[(e0 + u) * BQ];
                    kr = fmaf(kb_, rv[u], kr);
                    ky = fmaf(kb_, xv[u], ky);
                    ry = fmaf(rv[u], xv[u], ry);
                }
                if (row_ok) *reinterpret_cast<float4*>(prm.yvec + row_g + e0) = make_float4(xv[0], xv[1], xv[2], xv[3]);
            }
            kr = xch.sum(kr);
            ky = xch.sum(ky);
            ry = xch.sum(ry);
            if (row_ok && half == 0) {
                BwdRowRec o;
                o.m = mx * prm.tau * pow2i(-(eq + ek));
                o.jm = jmx;
                o.inv_omega = inv_om;
                o.hbar = hbar_a * pow2i(-(eg + ev));
                o.kb_rp = kr;
                o.kb_y = ky;
                o.sd = -prm.lambda * inv_om * ry;
                o.rp_scale = rp_scale;
                prm.rec[(size_t)head * n + i] = o;
                if (prm.cg_iters) prm.cg_iters[(size_t)head * n + i] = iters;
            }
            publish_p(SW_END);
        } else {
            // ---------------- finalise rho, denom; R = rho' (hi + lo) for the output sweep ----------------
            // x and kbar in registers, loaded in one batch (x from this thread's own scratch)
            float xv[DH], kv[DH];
            const bool have_x = row_ok && cg_sweeps > 0;   // no sweep ran: x = 0
#pragma unroll
            for (int e = 0; e < DH; ++e) {
                xv[e] = have_x ? xt[e * BQ] : 0.f;
                kv[e] = kbt[e * BQ];
            }
            if (prm.probe && row_ok) {   // Parallax form: the caller's probe plays rho'
#pragma unroll
                for (int e0 = 0; e0 < DH; e0 += 4) {
                    const float4 t = *reinterpret_cast<const float4*>(prm.probe + row_g + e0);
                    xv[e0] = t.x; xv[e0 + 1] = t.y; xv[e0 + 2] = t.z; xv[e0 + 3] = t.w;
                }
            }
            float dx = 0.f, xx = 0.f;
            {
                const float qsc = pow2i(-eq);
#pragma unroll
                for (int e0 = 0; e0 < DH; e0 += 8) {
                    const uint4 qr = *reinterpret_cast<const uint4*>(tile_half(s.q, row, half * DH + e0));
                    const __half* qh = reinterpret_cast<const __half*>(&qr);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        dx = fmaf(kv[e0 + u] - __half2float(qh[u]) * qsc, xv[e0 + u], dx);
                        xx = fmaf(xv[e0 + u], xv[e0 + u], xx);
                    }
                }
                if (!row_ok) { dx = 0.f; xx = 0.f; }
            }
            dx = xch.sum(dx);
            const float xn = sqrtf(xch.sum(xx));                 // |rho'|_2, which bounds max|rho'|
            const float inv_g = 1.f / (1.f + dx);
            const int sr = min(scale_exp(xn * 1.001f), 100 - ek);
            // R_lo (one more product per output block) only where rounding rho' to fp16 could move the
            // output by more than 2^-9 RMS(v): the output moves by the value/key covariance times the
            // rounding error, at most sqrt(tr_om) |rho'|_2 2^-11 (in RMS(v)).  The first tile (rank-
            // deficient scatter) and the precise form always take it.
            bool split_r;
            if constexpr (PROBE) split_r = true;
            else split_r = PREC || tile == 0 || ew_any(row_ok && sqrtf(tr_om) * xn > 4.f);
            float kx = 0.f;
            {
                const float rs = pow2i(sr), ris = pow2i(-sr);
#pragma unroll
                for (int e0 = 0; e0 < DH; e0 += 8) {
                    uint4 pk, pl;
                    uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
                    uint32_t* plw = reinterpret_cast<uint32_t*>(&pl);
#pragma unroll
                    for (int u = 0; u < 8; u += 2) {
                        const float x0 = xv[e0 + u] * rs, x1 = xv[e0 + u + 1] * rs;
                        pw[u >> 1] = pack_half2(x0, x1);
                        const float2 xh = __half22float2(*reinterpret_cast<const __half2*>(&pw[u >> 1]));
                        plw[u >> 1] = pack_half2(x0 - xh.x, x1 - xh.y);
                        const float2 xl = split_r ? __half22float2(*reinterpret_cast<const __half2*>(&plw[u >> 1]))
                                                  : make_float2(0.f, 0.f);
                        kx = fmaf(kv[e0 + u], (xh.x + xl.x) * ris, kx);        // kbar . R as the products see R
                        kx = fmaf(kv[e0 + u + 1], (xh.y + xl.y) * ris, kx);
                    }
                    *reinterpret_cast<uint4*>(tile_half(s.p, row, half * DH + e0)) = pk;
                    if (split_r) *reinterpret_cast<uint4*>(tile_half(s.rlo, row, half * DH + e0)) = pl;
                    if (row_ok && !prm.probe) {   // rho = rho' / (1 + delta.rho'), row-major output
                        *reinterpret_cast<float4*>(prm.rho + row_g + e0) =
                            make_float4(xv[e0] * inv_g, xv[e0 + 1] * inv_g, xv[e0 + 2] * inv_g, xv[e0 + 3] * inv_g);
                        *reinterpret_cast<float4*>(prm.rho + row_g + e0 + 4) =
                            make_float4(xv[e0 + 4] * inv_g, xv[e0 + 5] * inv_g, xv[e0 + 6] * inv_g, xv[e0 + 7] * inv_g);
                    }
                }
                if (!row_ok) kx = 0.f;
            }
            kx = xch.sum(kx);
            if (row_ok && half == 0 && !prm.probe) {
                prm.denom[(size_t)head * n + i] = omega * inv_g;
                if (prm.cg_iters) prm.cg_iters[(size_t)head * n + i] = iters;
            }
            int sU;
            // the probe form: |k_j - kbar|_2 <= 2 sqrt(D) max|k| (no key scatter trace was taken)
            if constexpr (PROBE) sU = scale_exp((1.f + 2.f * sqrtf((float)D) * mk * xn) * 1.001f);
            else sU = scale_exp((1.f + cbound * xn) * 1.001f);
            const float offU = m2 - (float)sU + (float)sr + (float)ek;
            const float c_acc = (1.f + kx) * pow2i(sr + ek);
            if (tid == 128) s.out_split = split_r ? 1 : 0;      // read by the T issuer after the publishing barrier
            publish_p(SW_OUT);

            // ---------------- OUT sweep ----------------
            uint64_t us_part = 0;
            for (int kb = 0; kb < nkb; ++kb, ++g) {
                ok = ok && wait_s(g);
                const uint32_t tS = tS0 + (g & 1) * 128 + lane_off + half * 64;
                const uint32_t tAh = tA + lane_off + half * 64;
                const int lim = lim_of(kb);
                const bool masked = !(tile_full && kb < tile);
                float a[64], v[32];
                uint32_t pk[16];
                tmem_ld32(tAh, *reinterpret_cast<float(*)[32]>(&a[0]));
                tmem_ld32(tAh + 32, *reinterpret_cast<float(*)[32]>(&a[32]));
                tmem_ld32(tS, v);
                tmem_ld_wait();
                release_a();
                if (masked) coef_chunk<true, true, 0>(v, a, c_log2, offU, c_acc, -1.f, half * 64, lim, us_part, pk);
                else coef_chunk<false, true, 0>(v, a, c_log2, offU, c_acc, -1.f, 0, 0, us_part, pk);
                tmem_st16(tS, pk);
                tmem_ld32(tS + 32, v);
                tmem_ld_wait();
                if (masked) coef_chunk<true, true, 1>(v, a, c_log2, offU, c_acc, -1.f, half * 64 + 32, lim, us_part, pk);
                else coef_chunk<false, true, 1>(v, a, c_log2, offU, c_acc, -1.f, 0, 0, us_part, pk);
                tmem_st16(tS + 16, pk);
                tmem_st_wait();
                done_block(g);
            }
            ok = ok && wait_y();
            const float usum = xch.sum(f2_total(us_part));
            const float osc = pow2i(-ev) / usum;
#pragma unroll
            for (int c = 0; c < DH / 32; ++c) {
                float v[32];
                tmem_ld32(tY + lane_off + half * DH + c * 32, v);
                tmem_ld_wait();
                if (row_ok) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 o;
                        __nv_bfloat162* ob = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
                        for (int u = 0; u < 4; ++u) ob[u] = __floats2bfloat162_rn(v[j + 2 * u] * osc, v[j + 2 * u + 1] * osc);
                        *reinterpret_cast<uint4*>(prm.out + row_g + c * 32 + j) = o;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();                           // the dealloc is warp-wide and aligned
        tmem_dealloc(s.tmem_base, 512);
    }
    if (tid == 0 && s.err) atomicOr(prm.dev_err, (unsigned)kDevErrMbarTimeout);
#undef WAIT
#undef LLA_SET_DIRECTION
}

// Workspace: header, fp16 copies of q, k, v (and dout for the backward), kbar and x scratch.
struct TcWs {
    Header* hdr;
    __half *q16, *k16, *v16, *g16;
    float *kbar, *xs, *knorm;
    int* tile_flag;
};
// Parts, each 256-byte aligned: header, q16, k16, v16, (g16), kbar and x ([slices][tiles][D][128]
// fp32), knorm ([slices][tiles * 128] fp32), tile flags ([slices][tiles] int).  N = B H n D,
// NT = B H (tiles * 128) D.
TcWs carve(void* ws, size_t N, size_t NT, int D, bool bwd) {
    unsigned char* base = static_cast<unsigned char*>(ws);
    TcWs w;
    w.hdr = reinterpret_cast<Header*>(base);
    size_t off = HDR_BYTES;
    w.q16 = reinterpret_cast<__half*>(base + off); off += align256(N * 2);
    w.k16 = reinterpret_cast<__half*>(base + off); off += align256(N * 2);
    w.v16 = reinterpret_cast<__half*>(base + off); off += align256(N * 2);
    w.g16 = nullptr;
    if (bwd) { w.g16 = reinterpret_cast<__half*>(base + off); off += align256(N * 2); }
    w.kbar = reinterpret_cast<float*>(base + off); off += align256(NT * 4);
    w.xs = reinterpret_cast<float*>(base + off); off += align256(NT * 4);
    w.knorm = reinterpret_cast<float*>(base + off); off += align256(NT / D * 4);
    w.tile_flag = reinterpret_cast<int*>(base + off);
    return w;
}

// Pre-pass, tensor maps and the sweep kernel.  BWD: the backward's stats stage (g = dout).
template <int D, bool BWD, bool PREC = false, bool PROBE = false>
cudaError_t launch_d(int B, int H, int n, const void* qv, const void* kv, const void* vv, const void* gv,
                     TcParams prm, void* ws, cudaEvent_t ev_begin, cudaEvent_t ev_end, cudaStream_t stream,
                     const char** why) {
    const size_t N = (size_t)B * H * n * D;
    const size_t NT = (size_t)B * H * ((n + BQ - 1) / BQ) * BQ * D;   // padded to whole tiles
    const TcWs w = carve(ws, N, NT, D, BWD);
    cudaError_t e = cudaMemsetAsync(w.hdr, 0, HDR_BYTES, stream);
    if (e != cudaSuccess) { *why = "workspace header clear"; return e; }
    const int n_tiles = (n + BQ - 1) / BQ;
    const size_t knorm_bytes = (size_t)B * H * n_tiles * BQ * 4;
    if (n % BQ && (e = cudaMemsetAsync(w.knorm, 0, knorm_bytes, stream)) != cudaSuccess) {   // the pad past n
        *why = "workspace key-norm clear";
        return e;
    }
    const size_t count8 = N / 8;
    const int pre_blocks = (int)((count8 + 255) / 256 < 152 * 8 ? (count8 + 255) / 256 : 152 * 8);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(qv);
    const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(kv);
    const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(vv);
    const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(gv);
    lla_maxabs_kernel<BWD ? 4 : 3><<<pre_blocks, 256, 0, stream>>>(q, k, v, g, count8, w.hdr);
    lla_to_half_kernel<BWD ? 4 : 3><<<pre_blocks, 256, 0, stream>>>(q, k, v, g, w.q16, w.k16, w.v16, w.g16, count8, w.hdr,
                                                                     w.knorm, D / 8, n, n_tiles * BQ);
    e = cudaGetLastError();
    if (e != cudaSuccess) { *why = "operand pre-pass launch"; return e; }

    CUtensorMap tq, tk, tv, tg;
    const uint64_t slices = (uint64_t)B * H;
    if (!make_tmap_f16_3d(&tq, w.q16, D, n, slices, BQ) || !make_tmap_f16_3d(&tk, w.k16, D, n, slices, BK) ||
        !make_tmap_f16_3d(&tv, w.v16, D, n, slices, BK) ||
        !make_tmap_f16_3d(&tg, BWD ? w.g16 : w.q16, D, n, slices, BQ)) {
        *why = "cuTensorMapEncodeTiled";
        return cudaErrorInvalidValue;
    }
    prm.hdr = w.hdr;
    prm.kbar = w.kbar;
    prm.xs = w.xs;
    prm.knorm = w.knorm;
    prm.tile_flag = w.tile_flag;
    prm.dev_err = device_error_word();
    prm.n = n;
    prm.n_tiles = (n + BQ - 1) / BQ;
    if (!prm.dev_err) { *why = "device error word"; return cudaErrorInvalidSymbol; }

    const size_t smem = sizeof(TcSmem<D>);
    auto kern = lla_tc_kernel<D, BWD, PREC, PROBE>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) { *why = "tensor kernel shared-memory attribute"; return e; }
    dim3 grid(prm.n_tiles, (unsigned)slices);
    if (ev_begin && (e = cudaEventRecord(ev_begin, stream)) != cudaSuccess) {
        *why = "profiling event record";
        return e;
    }
    // The precise and Parallax forms: a launch without MAX sweeps, then one that redoes, with them,
    // the tiles it marked (the marks are rare; the second launch's other CTAs return at once).  The
    // fixed-cap form and the backward: one launch with MAX sweeps.
    constexpr bool two = !BWD && (PREC || PROBE);
    for (int mode = two ? 1 : 0; mode <= (two ? 2 : 0); ++mode) {
        prm.mode = mode;
        kern<<<grid, NTHREADS, smem, stream>>>(tq, tk, tv, tg, prm);
        e = cudaGetLastError();
        if (e != cudaSuccess) { *why = "tensor kernel launch"; return e; }
    }
    if (ev_end && (e = cudaEventRecord(ev_end, stream)) != cudaSuccess) *why = "profiling event record";
    return e;
}

TcParams forward_params(const Problem& p) {
    TcParams prm{};
    prm.out = static_cast<__nv_bfloat16*>(p.out);
    prm.rho = p.rho;
    prm.denom = p.denom;
    prm.cg_iters = p.cg_iters;
    prm.probe = p.probe;
    prm.tau = p.tau;
    prm.lambda = p.lambda;
    prm.cg_tol = p.cg_tol;
    prm.cg_max_iters = p.cg_max_iters;
    return prm;
}

}  // namespace

size_t tensor_workspace_bytes(int B, int H, int n, int d) {
    const size_t N = (size_t)B * H * n * d;
    const size_t NT = (size_t)B * H * ((n + BQ - 1) / BQ) * BQ * d;
    return HDR_BYTES + 3 * align256(N * 2) + 2 * align256(NT * 4) + align256(NT / d * 4) +
           align256(NT / d / BQ * 4);
}

// Tolerance mode (cg_tol > 0) takes the precise form: CG run to a relative residual needs matrix-vector
// products accurate well beyond fp16's 11 bits wherever lambda/omega is small against the key scatter.
cudaError_t launch_tensor(const Problem& p, void* ws, cudaStream_t stream, const char** why) {
    const TcParams prm = forward_params(p);
    const bool prec = p.cg_tol > 0.f && !p.probe;
    if (p.d == 128) {
        if (p.probe)
            return launch_d<128, false, false, true>(p.B, p.H, p.n, p.q, p.k, p.v, nullptr, prm, ws, p.ev_main_begin,
                                                     p.ev_main_end, stream, why);
        return prec ? launch_d<128, false, true>(p.B, p.H, p.n, p.q, p.k, p.v, nullptr, prm, ws, p.ev_main_begin,
                                                 p.ev_main_end, stream, why)
                    : launch_d<128, false>(p.B, p.H, p.n, p.q, p.k, p.v, nullptr, prm, ws, p.ev_main_begin,
                                           p.ev_main_end, stream, why);
    }
    if (p.d == 64) {
        if (p.probe)
            return launch_d<64, false, false, true>(p.B, p.H, p.n, p.q, p.k, p.v, nullptr, prm, ws, p.ev_main_begin,
                                                    p.ev_main_end, stream, why);
        return prec ? launch_d<64, false, true>(p.B, p.H, p.n, p.q, p.k, p.v, nullptr, prm, ws, p.ev_main_begin,
                                                p.ev_main_end, stream, why)
                    : launch_d<64, false>(p.B, p.H, p.n, p.q, p.k, p.v, nullptr, prm, ws, p.ev_main_begin,
                                          p.ev_main_end, stream, why);
    }
    *why = "tensor path supports d in {64, 128}";
    return cudaErrorInvalidValue;
}

TensorOperands tensor_backward_operands(void* ws, int B, int H, int n, int d) {
    const size_t N = (size_t)B * H * n * d;
    const size_t NT = (size_t)B * H * ((n + BQ - 1) / BQ) * BQ * d;
    const TcWs w = carve(ws, N, NT, d, true);
    TensorOperands o;
    o.maxabs = w.hdr->maxabs;
    o.q16 = w.q16;
    o.k16 = w.k16;
    o.v16 = w.v16;
    o.g16 = w.g16;
    return o;
}

size_t tensor_backward_stats_bytes(int B, int H, int n, int d) {
    return tensor_workspace_bytes(B, H, n, d) + align256((size_t)B * H * n * d * 2);
}

cudaError_t launch_tensor_backward_stats(const BackwardProblem& p, void* ws, BwdRowRec* rec, float* yvec,
                                         cudaStream_t stream, const char** why) {
    TcParams prm{};
    prm.cg_iters = p.cg_iters;
    prm.rho_in = p.rho;
    prm.denom_in = p.denom;
    prm.rec = rec;
    prm.yvec = yvec;
    prm.tau = p.tau;
    prm.lambda = p.lambda;
    prm.cg_tol = p.cg_tol;
    prm.cg_max_iters = p.cg_max_iters;
    if (p.d == 128)
        return launch_d<128, true>(p.B, p.H, p.n, p.q, p.k, p.v, p.dout, prm, ws, p.ev_main_begin, p.ev_main_end,
                                   stream, why);
    if (p.d == 64)
        return launch_d<64, true>(p.B, p.H, p.n, p.q, p.k, p.v, p.dout, prm, ws, p.ev_main_begin, p.ev_main_end,
                                  stream, why);
    *why = "tensor path supports d in {64, 128}";
    return cudaErrorInvalidValue;
}

}  // namespace lla
