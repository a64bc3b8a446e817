/* Test-only probe library (liblla_probe.so): checks the tcgen05 descriptor encodings and the
 * TMA/TMEM helpers the LLA tensor kernel uses, on single 128x128x128 fp16 products.
 * Not part of the LLA API.
 *
 * A, B, B2: device fp16 [128][128] row-major.  D1, D2, D3: device fp32 [128][128].
 *   D1 = A B^T      (A and B by TMA, both K-major, SMEM x SMEM)
 *   D2 = A B2       (A written to TMEM by threads, B2 by TMA read MN-major, TMEM x SMEM)
 *   D3 = A B^T      (A written to SMEM by threads in the 128-byte-swizzle layout)
 * Returns 0 on success, else a CUDA error code.  Synchronous.
 *
 * lla_probe_umma_mn: At, K, V device bf16 [64][128] row-major, D device fp32 [128][256]:
 *   D = At^T [K | V]  (At written to SMEM by threads, K and V by TMA; both operands MN-major,
 *                      bf16, one M = 128, N = 256 product per 16 rows). */
#ifndef LLA_PROBE_H_
#define LLA_PROBE_H_
#ifdef __cplusplus
extern "C" {
#endif
int lla_probe_umma(const void* A, const void* B, const void* B2, float* D1, float* D2, float* D3);
int lla_probe_umma_mn(const void* At, const void* K, const void* V, float* D);
#ifdef __cplusplus
}
#endif
#endif
