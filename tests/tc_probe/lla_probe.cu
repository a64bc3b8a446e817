// Single-CTA tcgen05 probe: see lla_probe.h.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tc_host.h"
#include "tc_ptx.cuh"
#include "lla_probe.h"

namespace {
using namespace lla::tc;

struct __align__(1024) ProbeSmem {
    __half a[128 * 128];    // TMA, K-major SW128 (2 boxes of 128 rows x 64)
    __half b[128 * 128];    // TMA, K-major SW128
    __half b2[128 * 128];   // TMA, rows = k, 64-column boxes: MN-major view
    __half a3[128 * 128];   // written by threads, K-major SW128
    uint64_t bar_tma, bar_mma;
    uint32_t tmem_base;
    int err;
};

__global__ void __launch_bounds__(128, 1)
probe_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
             const __grid_constant__ CUtensorMap tm_b2, const __half* __restrict__ A, float* D1, float* D2,
             float* D3, int* status) {
    extern __shared__ unsigned char raw[];
    ProbeSmem& s = *reinterpret_cast<ProbeSmem*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        s.err = 0;
        mbar_init(&s.bar_tma, 1);
        mbar_init(&s.bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;
    const uint32_t tD1 = tbase, tD2 = tbase + 128, tD3 = tbase + 256, tA = tbase + 384;

    if (tid == 0) {
        mbar_arrive_expect_tx(&s.bar_tma, 3 * 128 * 128 * 2);
        for (int bx = 0; bx < 2; ++bx) {
            tma_load_3d(s.a + bx * 128 * 64, &tm_a, &s.bar_tma, bx * 64, 0, 0);
            tma_load_3d(s.b + bx * 128 * 64, &tm_b, &s.bar_tma, bx * 64, 0, 0);
            tma_load_3d(s.b2 + bx * 128 * 64, &tm_b2, &s.bar_tma, bx * 64, 0, 0);
        }
    }
    // every thread: its row of A into the swizzled a3 tile and, packed, into TMEM columns tA..tA+63
    const int row = warp * 32 + lane;
    unsigned char* a3 = reinterpret_cast<unsigned char*>(s.a3);
    for (int c = 0; c < 128; ++c) *reinterpret_cast<__half*>(a3 + sw128_offset(row, c, 128)) = A[row * 128 + c];
    for (int g = 0; g < 4; ++g) {
        uint32_t r[16];
        for (int j = 0; j < 16; ++j) {
            const __half lo = A[row * 128 + g * 32 + 2 * j], hi = A[row * 128 + g * 32 + 2 * j + 1];
            r[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
        }
        tmem_st16(tA + ((uint32_t)(warp * 32) << 16) + g * 16, r);
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        if (mbar_wait(&s.bar_tma, 0, &s.err)) {
            const uint32_t id_k = idesc_f16(128, 128, false), id_mn = idesc_f16(128, 128, true);
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t koff = (ks >> 2) * 16384 + (ks & 3) * 32;
                umma_ss(tD1, sdesc_sw128(smem_u32(s.a) + koff, 16, 1024), sdesc_sw128(smem_u32(s.b) + koff, 16, 1024),
                        id_k, ks > 0);
                umma_ss(tD3, sdesc_sw128(smem_u32(s.a3) + koff, 16, 1024),
                        sdesc_sw128(smem_u32(s.b) + koff, 16, 1024), id_k, ks > 0);
                umma_ts(tD2, tA + ks * 8, sdesc_sw128(smem_u32(s.b2) + ks * 2048, 16384, 1024), id_mn, ks > 0);
            }
        }
        umma_commit(&s.bar_mma);
    }
    __syncwarp();
    mbar_wait(&s.bar_mma, 0, &s.err);
    tc_fence_after();
    float v[32];
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float* outs[3] = {D1, D2, D3};
    const uint32_t cols[3] = {tD1, tD2, tD3};
    for (int m = 0; m < 3; ++m)
        for (int g = 0; g < 4; ++g) {
            tmem_ld32(cols[m] + lane_base + g * 32, v);
            tmem_ld_wait();
            for (int j = 0; j < 32; ++j) outs[m][row * 128 + g * 32 + j] = v[j];
        }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
    if (tid == 0) *status = s.err;
}
// ---- moment product: D[128 x 256] = At^T [K | V], bf16, A and B both MN-major ----------------
// At, K, V are [64 rows][128] (a row = one key).  A (At viewed as [M = 128][K = 64 keys]) is written
// by threads in the 128-byte-swizzle layout of 64-row boxes; K and V arrive by TMA as four
// [64 x 64] boxes at a uniform 8 KB stride (K cols 0-63, K cols 64-127, V cols 0-63, V cols 64-127),
// read as one N = 256 operand.
struct __align__(1024) ProbeMnSmem {
    __nv_bfloat16 a[64 * 128];
    __nv_bfloat16 b[64 * 256];
    uint64_t bar_tma, bar_mma;
    uint32_t tmem_base;
    int err;
};

__global__ void __launch_bounds__(128, 1)
probe_mn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __nv_bfloat16* __restrict__ At, float* D, int* status) {
    extern __shared__ unsigned char raw[];
    ProbeMnSmem& s = *reinterpret_cast<ProbeMnSmem*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        s.err = 0;
        mbar_init(&s.bar_tma, 1);
        mbar_init(&s.bar_mma, 1);
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 256);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tD = s.tmem_base;
    if (tid == 0) {
        mbar_arrive_expect_tx(&s.bar_tma, 64 * 256 * 2);
        for (int bx = 0; bx < 2; ++bx) {
            tma_load_3d(s.b + bx * 64 * 64, &tm_k, &s.bar_tma, bx * 64, 0, 0);
            tma_load_3d(s.b + (2 + bx) * 64 * 64, &tm_v, &s.bar_tma, bx * 64, 0, 0);
        }
    }
    {   // thread: half a key row of At
        const int r = tid >> 1, c0 = (tid & 1) * 64;
        unsigned char* a = reinterpret_cast<unsigned char*>(s.a);
        for (int c = c0; c < c0 + 64; ++c)
            *reinterpret_cast<__nv_bfloat16*>(a + sw128_offset(r, c, 64)) = At[r * 128 + c];
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        if (mbar_wait(&s.bar_tma, 0, &s.err)) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 256, true, true);
            for (int ks = 0; ks < 4; ++ks)
                umma_ss(tD, sdesc_sw128(smem_u32(s.a) + ks * 2048, 8192, 1024),
                        sdesc_sw128(smem_u32(s.b) + ks * 2048, 8192, 1024), id, ks > 0);
        }
        umma_commit(&s.bar_mma);
    }
    __syncwarp();
    mbar_wait(&s.bar_mma, 0, &s.err);
    tc_fence_after();
    const int row = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float v[32];
    for (int g = 0; g < 8; ++g) {
        tmem_ld32(tD + lane_base + g * 32, v);
        tmem_ld_wait();
        for (int j = 0; j < 32; ++j) D[row * 256 + g * 32 + j] = v[j];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tD, 256);
    if (tid == 0) *status = s.err;
}
}  // namespace

extern "C" int lla_probe_umma(const void* A, const void* B, const void* B2, float* D1, float* D2, float* D3) {
    CUtensorMap ta, tb, tb2;
    if (!lla::make_tmap_f16_3d(&ta, A, 128, 128, 1, 128) || !lla::make_tmap_f16_3d(&tb, B, 128, 128, 1, 128) ||
        !lla::make_tmap_f16_3d(&tb2, B2, 128, 128, 1, 128))
        return (int)cudaErrorInvalidValue;
    int* status = nullptr;
    cudaError_t e = cudaMalloc(&status, sizeof(int));
    if (e != cudaSuccess) return (int)e;
    const size_t smem = sizeof(ProbeSmem) + 1024;
    e = cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) {
        probe_kernel<<<1, 128, smem>>>(ta, tb, tb2, static_cast<const __half*>(A), D1, D2, D3, status);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int h = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(status);
    if (e != cudaSuccess) return (int)e;
    return h ? 9999 : 0;
}

extern "C" int lla_probe_umma_mn(const void* At, const void* K, const void* V, float* D) {
    CUtensorMap tk, tv;
    if (!lla::make_tmap_16b_3d_strided(&tk, K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 128, 64, 1, 64, 64) ||
        !lla::make_tmap_16b_3d_strided(&tv, V, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 128, 64, 1, 64, 64))
        return (int)cudaErrorInvalidValue;
    int* status = nullptr;
    cudaError_t e = cudaMalloc(&status, sizeof(int));
    if (e != cudaSuccess) return (int)e;
    const size_t smem = sizeof(ProbeMnSmem) + 1024;
    e = cudaFuncSetAttribute(probe_mn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) {
        probe_mn_kernel<<<1, 128, smem>>>(tk, tv, static_cast<const __nv_bfloat16*>(At), D, status);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int h = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(status);
    if (e != cudaSuccess) return (int)e;
    return h ? 9999 : 0;
}
