// CUDA-core (FFMA) GEMM with the block's fused epilogues.
//
// This is the fp32 path of the library (no TF32: fp32 inputs are multiplied
// and accumulated in fp32), and the bf16 path's fallback for shapes the tensor
// core kernel does not take. C[M, N] = A[M, K] . B[N, K]^T, both operands
// K-contiguous ([out, in] weight layout).

#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace xmod {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, THREADS = 256;

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

template <typename T>
__device__ __forceinline__ void epilogue_store(const Epilogue& e, int M, int N, int m, int n,
                                               float acc, float acc2) {
  if (m >= M || n >= N) return;
  switch (e.kind) {
    case EPI_STORE:
      if (e.out_f32) ((float*)e.out)[(int64_t)m * e.ldo + n] = acc;
      else st_f((T*)e.out + (int64_t)m * e.ldo + n, acc);
      break;
    case EPI_OPROJ: {
      const int64_t b = m / e.n_per_seq;
      const int64_t t = e.idx ? (int64_t)e.idx[m] : (m - b * e.n_per_seq);
      const float xv = ld_f((const T*)e.x + (b * e.T + t) * e.d + n);
      if (e.out) st_f((T*)e.out + (int64_t)m * e.ldo + n, acc);
      if (e.out2) ((float*)e.out2)[(int64_t)m * e.ldo2 + n] = xv + acc;
      break;
    }
    case EPI_SWIGLU:
      st_f((T*)e.out + (int64_t)m * e.ldo + n, silu(acc) * acc2);
      break;
    case EPI_DOWN_SCATTER: {
      const int64_t b = m / e.n_per_seq;
      const int64_t t = e.idx ? (int64_t)e.idx[m] : (m - b * e.n_per_seq);
      T* xp = (T*)e.x + (b * e.T + t) * e.d + n;
      const float xv = ld_f(xp);
      const float av = e.a ? ld_f((const T*)e.a + (int64_t)m * e.d + n) : 0.0f;
      float y;
      if (e.gate == XMOD_GATE_XMOD) y = xv + e.varsigma * e.r_sel[m] * (av + acc);  // Eq. 7
      else if (e.gate == XMOD_GATE_MOD) y = (xv + av) + e.r_sel[m] * acc;         // Eq. 6
      else y = (xv + av) + acc;                                                    // dense
      st_f(xp, y);
      if (e.out) st_f((T*)e.out + (int64_t)m * e.ldo + n, y);
      break;
    }
  }
}

template <typename T, bool DUAL>
__global__ void __launch_bounds__(THREADS)
gemm_simt_kernel(int M, int N, int K, const T* __restrict__ A, int lda, const T* __restrict__ B,
                 int ldb, const T* __restrict__ B2, Epilogue e) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ float B2s[DUAL ? BK : 1][DUAL ? BN + 4 : 1];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4] = {}, acc2[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    // 64 x 16 tile of A and of B: 1024 elements each, 4 per thread
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int li = tid + i * THREADS;
      const int r = li / BK, kk = li % BK;
      const int gm = m0 + r, gn = n0 + r, gk = k0 + kk;
      As[kk][r] = (gm < M && gk < K) ? ld_f(A + (int64_t)gm * lda + gk) : 0.f;
      Bs[kk][r] = (gn < N && gk < K) ? ld_f(B + (int64_t)gn * ldb + gk) : 0.f;
      if (DUAL) B2s[kk][r] = (gn < N && gk < K) ? ld_f(B2 + (int64_t)gn * ldb + gk) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], bb[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bb[j] = Bs[kk][tx + 16 * j];
        if (DUAL) b2[j] = B2s[kk][tx + 16 * j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
          if (DUAL) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      epilogue_store<T>(e, M, N, m0 + ty + 16 * i, n0 + tx + 16 * j, acc[i][j], acc2[i][j]);
}

}  // namespace

cudaError_t launch_gemm_simt(const Ctx& c, xmod_dtype dt, int M, int N, int K, const void* A,
                             int lda, const void* B, int ldb, const void* B2,
                             const Epilogue& e) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  const bool dual = e.kind == EPI_SWIGLU;
  if (dt == XMOD_BF16) {
    using T = __nv_bfloat16;
    if (dual)
      gemm_simt_kernel<T, true><<<grid, THREADS, 0, c.stream>>>(M, N, K, (const T*)A, lda,
                                                                (const T*)B, ldb, (const T*)B2, e);
    else
      gemm_simt_kernel<T, false><<<grid, THREADS, 0, c.stream>>>(M, N, K, (const T*)A, lda,
                                                                 (const T*)B, ldb, nullptr, e);
  } else {
    using T = float;
    if (dual)
      gemm_simt_kernel<T, true><<<grid, THREADS, 0, c.stream>>>(M, N, K, (const T*)A, lda,
                                                                (const T*)B, ldb, (const T*)B2, e);
    else
      gemm_simt_kernel<T, false><<<grid, THREADS, 0, c.stream>>>(M, N, K, (const T*)A, lda,
                                                                 (const T*)B, ldb, nullptr, e);
  }
  return cudaGetLastError();
}

}  // namespace xmod
