// Unit probe of the tcgen05 building blocks in csrc/ptx.cuh: one CTA stages A and B in the
// 128-byte-swizzled shared-memory layouts the chunk kernel uses, issues the MMAs, and reads
// the TMEM accumulator back. Built and driven by tests/test_gpu_tc_probe.py.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ptx.cuh"

using namespace kda::ptx;

// mode 0: tf32, A K-major [128][K], B K-major [N][K]        D = A B^T
// mode 1: tf32, A K-major [128][K], B MN-major given [K][N] D = A B
// mode 2: tf32, A MN-major given [K][128], B K-major [N][K] D = A^T B^T
// mode 3: bf16, A K-major [128][K], B K-major [N][K]        D = A B^T
// mode 4: bf16, A K-major [128][K], B MN-major given [K][N] D = A B
// mode 5: bf16, A MN-major given [K][128], B K-major [N][K] D = A^T B^T
// mode 6: tf32, A in TMEM [128 lanes][K cols], B K-major    D = A B^T
__global__ void __launch_bounds__(128) probe_kernel(int mode, const float* A, const float* B,
                                                    float* Dout, int N, int K, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x;
  const bool bf = mode == 3 || mode == 4 || mode == 5;
  const bool a_mn = mode == 2 || mode == 5, b_mn = mode == 1 || mode == 4;
  const uint32_t rowbytes_k = bf ? 64 : 32;    // elements per 128-byte row
  // A region: 128 rows; K-blocks of 128 rows x 128 B = 16 KiB
  uint8_t* sA = smem;
  const uint32_t a_kblk = 128 * 128;
  const int a_blocks = (K + rowbytes_k - 1) / rowbytes_k;
  uint8_t* sB = smem + a_blocks * a_kblk;
  // B region: K-major: N rows, K-blocks of N*128 B; MN-major: K rows, N-blocks of K*128 B
  const uint32_t b_kblk = b_mn ? (uint32_t)K * 128 : (uint32_t)N * 128;
  const uint32_t esz = bf ? 2 : 4;

  for (int e = tid; e < 128 * K && mode != 6; e += 128) {
    const int m = e / K, k = e % K;
    float x = a_mn ? A[k * 128 + m] : A[m * K + k];
    if (a_mn) {
      // MN-major: rows are k, contiguous index m
      if (bf) *(__nv_bfloat16*)(sA + sw128_off16(k, m, (uint32_t)K * 128)) = __float2bfloat16_rn(x);
      else *(float*)(sA + sw128_off32(k, m, (uint32_t)K * 128)) = x;
    } else if (bf) {
      *(__nv_bfloat16*)(sA + sw128_off16(m, k, a_kblk)) = __float2bfloat16_rn(x);
    } else {
      *(float*)(sA + sw128_off32(m, k, a_kblk)) = x;
    }
  }
  for (int e = tid; e < N * K; e += 128) {
    if (b_mn) {
      const int k = e / N, n = e % N;
      if (bf) *(__nv_bfloat16*)(sB + sw128_off16(k, n, b_kblk)) = __float2bfloat16_rn(B[k * N + n]);
      else *(float*)(sB + sw128_off32(k, n, b_kblk)) = B[k * N + n];
    } else {
      const int n = e / K, k = e % K;
      if (bf) *(__nv_bfloat16*)(sB + sw128_off16(n, k, b_kblk)) = __float2bfloat16_rn(B[n * K + k]);
      else *(float*)(sB + sw128_off32(n, k, b_kblk)) = B[n * K + k];
    }
  }
  fence_proxy_async_smem();
  if (tid < 32) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  if (mode == 6) {  // A into TMEM columns 128.. (lane = row m)
    const int warp = tid >> 5;
    for (int c0 = 0; c0 < K; c0 += 32) {
      float v[32];
      for (int j = 0; j < 32; ++j) v[j] = A[tid * K + c0 + j];
      tmem_st32(tbase + ((uint32_t)(warp * 32) << 16) + 128 + c0, v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (tid == 0) {
    const uint32_t idesc = idesc_make(bf ? kFmtBF16 : kFmtTF32, 128, N, a_mn, b_mn);
    const int kstep = bf ? 16 : 8;
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    for (int s = 0; s < K / kstep; ++s) {
      uint64_t ad, bd;
      // MN-major: one instruction covers kstep K-rows = kstep/8 atoms of 1024 B
      if (a_mn) ad = sdesc_sw128(a0 + s * (kstep / 8) * 1024, (uint32_t)K * 128, 1024);
      else ad = sdesc_sw128(a0 + (s * kstep / rowbytes_k) * a_kblk + ((s * kstep) % rowbytes_k) * esz, 16, 1024);
      if (b_mn) bd = sdesc_sw128(b0 + s * (kstep / 8) * 1024, b_kblk, 1024);
      else bd = sdesc_sw128(b0 + (s * kstep / rowbytes_k) * b_kblk + ((s * kstep) % rowbytes_k) * esz, 16, 1024);
      if (mode == 6) mma_tf32_ts(tbase, tbase + 128 + s * kstep, bd, idesc, s > 0);
      else if (bf) mma_f16(tbase, ad, bd, idesc, s > 0);
      else mma_tf32(tbase, ad, bd, idesc, s > 0);
    }
    mma_commit(&bar);
  }
  __syncwarp();
  if (!mbar_wait(&bar, 0, 200000000ull)) {
    if (tid == 0) atomicOr(err, 1);
  }
  tc_fence_after();
  const int warp = tid >> 5;
  for (int c0 = 0; c0 < N; c0 += 32) {
    float v[32];
    tmem_ld32(tbase + ((uint32_t)(warp * 32) << 16) + c0, v);
    for (int j = 0; j < 32; ++j) Dout[tid * N + c0 + j] = v[j];
  }
  tc_fence_before();
  __syncthreads();
  if (tid < 32) tmem_dealloc(tbase, 256);
}

extern "C" int probe_mma(int mode, const float* A, const float* B, float* D, int N, int K,
                         int* err) {
  // bounds the probe supports: N in {32, 64, 128}, K multiple of 64, <= 128
  if (!(N == 32 || N == 64 || N == 128) || K % 64 != 0 || K > 128 || mode < 0 || mode > 6)
    return -1;
  size_t smem = 1024 + 128 * 128 * 4 + 128 * 128 * 4;
  cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  probe_kernel<<<1, 128, smem>>>(mode, A, B, D, N, K, err);
  return (int)cudaGetLastError();
}
