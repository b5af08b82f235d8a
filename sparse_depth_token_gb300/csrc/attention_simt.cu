// CUDA-core causal GQA attention (fp32 arithmetic, online softmax).
//
// The fp32 path of the library, and the fallback for head sizes the tensor-core
// kernel does not take. Attention runs among the B*n rows of the compact
// buffer, sequence by sequence; the compact order is the position order, so the
// causal mask over compact indices is the causal mask over original positions
// (X-MoD notes, section "mechanism controls": a sparse layer attends within its
// selected subset; "Mixture-of-Depths explained": the gather keeps position order).
// Query head h reads key/value head h / (hq / hkv).
// With qpos (Selected-Q / full-KV, X-MoD notes "mechanism controls"): query row i of
// sequence b sits at position qpos[b * n + i] and attends to the keys at positions
// <= it among the nkv keys of its sequence (k, v rows b * nkv ...).

#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace xmod {

namespace {

constexpr int ROWS = 16;       // query rows per CTA, one warp each
constexpr int KT = 32;         // keys per shared-memory tile, one lane each

template <typename T, int HD>
__global__ void __launch_bounds__(ROWS * 32)
attention_simt_kernel(int n, int hq, int hkv, const T* __restrict__ q, int ldq,
                      const T* __restrict__ k, const T* __restrict__ v, int ldkv,
                      T* __restrict__ o, const int32_t* __restrict__ qpos, int nkv) {
  __shared__ float Qs[ROWS][HD];
  __shared__ float Ks[KT][HD + 1];
  __shared__ float Vs[KT][HD];
  constexpr int PER = HD / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (hq / hkv);
  const int i0 = blockIdx.x * ROWS;
  const int i = i0 + warp;
  const int64_t seq0 = (int64_t)b * n;
  const int64_t kseq0 = (int64_t)b * nkv;
  const float scale = rsqrtf((float)HD);
  // last key position row i may see (rows past n: none)
  const int li = i < n ? (qpos ? qpos[seq0 + i] : i) : -1;

  for (int e = threadIdx.x; e < ROWS * HD; e += ROWS * 32) {
    const int r = e / HD, c = e % HD;
    Qs[r][c] = (i0 + r < n) ? ld_f(q + (seq0 + i0 + r) * ldq + h * HD + c) : 0.f;
  }
  float m = -INFINITY, l = 0.f, acc[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p) acc[p] = 0.f;

  const int last_row = min(n - 1, i0 + ROWS - 1);
  const int last = qpos ? qpos[seq0 + last_row] : last_row;   // positions ascend with rows
  for (int j0 = 0; j0 <= last; j0 += KT) {
    __syncthreads();
    for (int e = threadIdx.x; e < KT * HD; e += ROWS * 32) {
      const int r = e / HD, c = e % HD;
      const bool ok = j0 + r < nkv;
      Ks[r][c] = ok ? ld_f(k + (kseq0 + j0 + r) * ldkv + g * HD + c) : 0.f;
      Vs[r][c] = ok ? ld_f(v + (kseq0 + j0 + r) * ldkv + g * HD + c) : 0.f;
    }
    __syncthreads();
    if (i >= n || j0 > li) continue;
    const int j = j0 + lane;
    float sc = -INFINITY;
    if (j <= li) {
      float dot = 0.f;
#pragma unroll 8
      for (int c = 0; c < HD; ++c) dot = fmaf(Qs[warp][c], Ks[lane][c], dot);
      sc = dot * scale;
    }
    const float m_new = fmaxf(m, warp_max(sc));
    const float p = (j <= li) ? expf(sc - m_new) : 0.f;
    const float corr = expf(m - m_new);
    l = l * corr + warp_sum(p);
#pragma unroll
    for (int pp = 0; pp < PER; ++pp) acc[pp] *= corr;
    const int jmax = min(KT, li - j0 + 1);
    for (int jj = 0; jj < jmax; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
      for (int pp = 0; pp < PER; ++pp) acc[pp] = fmaf(pj, Vs[jj][lane + 32 * pp], acc[pp]);
    }
    m = m_new;
  }
  if (i < n) {
    const float inv = 1.0f / l;
#pragma unroll
    for (int pp = 0; pp < PER; ++pp)
      st_f(o + (seq0 + i) * (int64_t)(hq * HD) + h * HD + lane + 32 * pp, acc[pp] * inv);
  }
}

template <typename T>
cudaError_t dispatch(const Ctx& c, int B, int n, int hq, int hkv, int hd, const void* q, int ldq,
                     const void* k, const void* v, int ldkv, void* o, const int32_t* qpos,
                     int nkv) {
  dim3 grid((n + ROWS - 1) / ROWS, hq, B);
  switch (hd) {
    case 32:
      attention_simt_kernel<T, 32><<<grid, ROWS * 32, 0, c.stream>>>(
          n, hq, hkv, (const T*)q, ldq, (const T*)k, (const T*)v, ldkv, (T*)o, qpos, nkv);
      break;
    case 64:
      attention_simt_kernel<T, 64><<<grid, ROWS * 32, 0, c.stream>>>(
          n, hq, hkv, (const T*)q, ldq, (const T*)k, (const T*)v, ldkv, (T*)o, qpos, nkv);
      break;
    case 128:
      attention_simt_kernel<T, 128><<<grid, ROWS * 32, 0, c.stream>>>(
          n, hq, hkv, (const T*)q, ldq, (const T*)k, (const T*)v, ldkv, (T*)o, qpos, nkv);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_simt(const Ctx& c, xmod_dtype dt, int B, int n, int hq, int hkv,
                                  int hd, const void* q, int ldq, const void* k, const void* v,
                                  int ldkv, void* o, const int32_t* qpos, int nkv) {
  if (B <= 0 || n <= 0) return cudaSuccess;
  if (!qpos) nkv = n;
  if (dt == XMOD_BF16)
    return dispatch<__nv_bfloat16>(c, B, n, hq, hkv, hd, q, ldq, k, v, ldkv, o, qpos, nkv);
  return dispatch<float>(c, B, n, hq, hkv, hd, q, ldq, k, v, ldkv, o, qpos, nkv);
}

}  // namespace xmod
