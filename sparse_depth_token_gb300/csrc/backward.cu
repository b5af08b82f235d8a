// Backward of one sparse-depth layer: the gradient of sum(dy * y) + route_coef * L_route
// with respect to the layer input and every weight, the top-(T/K) selection held fixed.
//
// Sources: "X-MoD: Practical Scaling Laws for Sparse-Depth Routing Beyond
// Mixture-of-Depths" reading notes -- Eq. 8 (router logit, sigmoid gate), Eq. 6 and
// Eq. 7 (gated residuals, the only place the gate r and varsigma enter), Eq. 9 (the
// binary cross-entropy between the top-k decisions and the threshold predictor,
// section "top-k in training, causal threshold at evaluation"); the block of the
// "backbone configuration" (pre-norm RMSNorm, GQA attention, SwiGLU FFN).
//
// The layer's forward is recomputed from x with the forward kernels (router, top-k,
// gather + RMSNorm1, projections, attention), keeping the intermediates the backward
// reads; then every step is differentiated in reverse order. Weight gradients are
// GEMMs over the token dimension and activation gradients GEMMs with the weights: for
// bf16 the tcgen05 GEMM reads dY, X and W as stored (MN-major operands); otherwise (fp32
// on the FFMA GEMM, or bf16 dimensions that are not multiples of 64 on the K-major
// tcgen05 GEMM) they are transposed into K-contiguous buffers, the token dimension padded
// with zero tokens to a multiple of 8.
// Column sums (RMSNorm gains,
// router vector) are taken in a fixed order: partial sums per row chunk, then the
// chunks in order, so every result is deterministic.

#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <initializer_list>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace xmod {

namespace {

constexpr int BW_WARPS = 8;   // warps per CTA of the row kernels

__device__ __forceinline__ int64_t bw_stream_row(int64_t m, int T, int n, const int32_t* idx) {
  const int64_t b = m / n;
  const int64_t t = idx ? (int64_t)idx[m] : (m - b * n);
  return b * T + t;
}

// Four consecutive elements (16 bytes of fp32, 8 of bf16) as a float4, and back.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float softplus_f(float z) {
  return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z)));
}

// ---------------------------------------------------------------- transpose
// out[c, r] = in[r, c] for r < R, c < C; out[c, r] = 0 for R <= r < Rpad (zero tokens).
// The kernel moves bits (U = a 2- or 4-byte word; 0 bits are +0.0 in bf16 and fp32).
// 64 x 64 tiles, 256 threads. Both phases move 16-byte chunks (V words) where the
// pointers, strides and bounds allow it (vec_in / vec_out), word by word otherwise. In
// shared memory chunk ch of tile row r sits at chunk ch ^ ((r / V) % (64 / V)): the
// read phase gathers one word from each of V consecutive rows, and across a warp those
// rows fall in distinct chunks, so neither phase has bank conflicts.
constexpr int TR_T = 64;

// One 64 x 64 tile at (r0, c0) of out = in^T, through the shared tile `tile`.
template <typename U>
__device__ __forceinline__ void transpose_tile(int R, int Rpad, int C, const U* __restrict__ in,
                                               int64_t ldi, U* __restrict__ out, int64_t ldo,
                                               int r0, int c0, int vec_in, int vec_out, U* tile) {
  constexpr int V = 16 / sizeof(U), CH = TR_T / V;
  for (int e = threadIdx.x; e < TR_T * CH; e += 256) {
    const int r = e / CH, ch = e - r * CH, gr = r0 + r, gc = c0 + ch * V;
    U* dst = tile + r * TR_T + ((ch ^ ((r / V) & (CH - 1))) * V);
    if (vec_in && gr < R && gc + V <= C) {
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(in + (int64_t)gr * ldi + gc);
    } else {
#pragma unroll
      for (int k = 0; k < V; ++k) dst[k] = (gr < R && gc + k < C) ? in[(int64_t)gr * ldi + gc + k] : U(0);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < TR_T * CH; e += 256) {
    const int c = e / CH, ch = e - c * CH, gc = c0 + c, gr = r0 + ch * V;
    if (gc >= C) continue;
    // rows ch * V + k all have r / V == ch: their chunk c / V sits at (c / V) ^ ch
    const U* src = tile + ((c / V) ^ ch) * V + (c % V);
    union {
      uint4 q;
      U w[V];
    } v;
#pragma unroll
    for (int k = 0; k < V; ++k) v.w[k] = src[(ch * V + k) * TR_T];
    U* dst = out + (int64_t)gc * ldo + gr;
    if (vec_out && gr + V <= Rpad) {
      *reinterpret_cast<uint4*>(dst) = v.q;
    } else {
#pragma unroll
      for (int k = 0; k < V; ++k)
        if (gr + k < Rpad) dst[k] = v.w[k];
    }
  }
}

// grid.z runs over a batch of such matrices, in_bs / out_bs elements apart.
template <typename U>
__global__ void __launch_bounds__(256)
transpose_kernel(int R, int Rpad, int C, const U* __restrict__ in, int64_t ldi,
                 U* __restrict__ out, int64_t ldo, int64_t in_bs, int64_t out_bs, int vec_in,
                 int vec_out) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) U tile[TR_T * TR_T];
  transpose_tile<U>(R, Rpad, C, in + blockIdx.z * in_bs, ldi, out + blockIdx.z * out_bs, ldo,
                    blockIdx.y * TR_T, blockIdx.x * TR_T, vec_in, vec_out, tile);
}

// Several independent transposes in one launch: job k owns the tiles [start, start +
// tiles_x * tiles_y) of grid.x (tile (bx, by) of its own matrix); grid.y runs over a
// batch common to the jobs (in_bs / out_bs elements apart per job).
struct TrJob {
  const void* in;
  void* out;
  int64_t ldi, ldo, in_bs, out_bs;
  int R, Rpad, C, tiles_x, start, vec_in, vec_out;
};
constexpr int kTrMaxJobs = 8;
struct TrJobs {
  TrJob j[kTrMaxJobs];
  int n;
};

template <typename U>
__global__ void __launch_bounds__(256)
transpose_multi_kernel(const __grid_constant__ TrJobs jobs) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(16) U tile[TR_T * TR_T];
  int k = 0;
  while (k + 1 < jobs.n && (int)blockIdx.x >= jobs.j[k + 1].start) ++k;
  const TrJob& J = jobs.j[k];
  const int t = (int)blockIdx.x - J.start;
  const int by = t / J.tiles_x, bx = t - by * J.tiles_x;
  transpose_tile<U>(J.R, J.Rpad, J.C, (const U*)J.in + blockIdx.y * J.in_bs, J.ldi,
                    (U*)J.out + blockIdx.y * J.out_bs, J.ldo, by * TR_T, bx * TR_T, J.vec_in,
                    J.vec_out, tile);
}

// ---------------------------------------------------------------- gated residual backward
// Selected row m (stream row of idx): Eq. 7 y = x + vs r (a + f): df = vs r dy (also the
// gradient reaching a), dr = vs <dy, a + f>, dvs_m = r <dy, a + f>. Eq. 6 y = x + a + r f:
// dae = dy (gradient reaching a), df = r dy, dr = <dy, f>.
template <typename T>
__global__ void __launch_bounds__(BW_WARPS * 32)
scatter_bwd_kernel(int64_t M, int seqT, int n, int d, const T* __restrict__ dy,
                   const int32_t* __restrict__ idx, const float* __restrict__ r_sel,
                   const T* __restrict__ a, const T* __restrict__ f, float vs, int gate,
                   T* __restrict__ df, T* __restrict__ dae, float* __restrict__ dr,
                   float* __restrict__ dvs) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * BW_WARPS + warp;
  if (m >= M) return;
  const T* g = dy + bw_stream_row(m, seqT, n, idx) * d;
  const float r = r_sel[m];
  constexpr int V = Vec16<T>::N;
  float dot = 0.0f;
  for (int c = lane * V; c < d; c += 32 * V) {
    const Vec16<T> gv = ld_vec(g + c), fv = ld_vec(f + m * d + c);
    Vec16<T> o;
    if (gate == XMOD_GATE_XMOD) {
      Vec16<T> av;
      av.raw = make_uint4(0, 0, 0, 0);   // bit pattern 0 is 0 in bf16 and fp32
      if (a) av = ld_vec(a + m * d + c);
#pragma unroll
      for (int k = 0; k < V; ++k) {
        dot += gv.get(k) * (av.get(k) + fv.get(k));
        o.set(k, vs * r * gv.get(k));
      }
    } else {
#pragma unroll
      for (int k = 0; k < V; ++k) {
        dot += gv.get(k) * fv.get(k);
        o.set(k, r * gv.get(k));
      }
      st_vec(dae + m * d + c, gv);
    }
    st_vec(df + m * d + c, o);
  }
  dot = warp_sum(dot);
  if (lane == 0) {
    dr[m] = gate == XMOD_GATE_XMOD ? vs * dot : dot;
    dvs[m] = gate == XMOD_GATE_XMOD ? r * dot : 0.0f;
  }
}

// ---------------------------------------------------------------- router logit gradient
// One CTA per sequence: ds[t] = coef_n * (sigmoid(s_t) - q_t) + (selected) dr * r (1 - r),
// and loss_part[b] = sum_t of the Eq. 9 terms (-log p for q = 1, -log(1 - p) for q = 0).
// Shared memory: T floats (the gate term of each selected token) and T flags.
__global__ void __launch_bounds__(1024)
route_bwd_kernel(int T, int n, const float* __restrict__ s, const int32_t* __restrict__ idx,
                 const float* __restrict__ r_sel, const float* __restrict__ dr, float coef_n,
                 float* __restrict__ ds, float* __restrict__ loss_part) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float gsh[];
  uint8_t* sel = reinterpret_cast<uint8_t*>(gsh + T);
  __shared__ float red[32];
  const int b = blockIdx.x;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    gsh[t] = 0.0f;
    sel[t] = 0;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int64_t m = (int64_t)b * n + j;
    const int t = idx[m];
    const float r = r_sel[m];
    gsh[t] = dr[m] * r * (1.0f - r);
    sel[t] = 1;
  }
  __syncthreads();
  float loss = 0.0f;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const float z = s[(int64_t)b * T + t];
    const float p = 1.0f / (1.0f + expf(-z));
    const bool q = sel[t] != 0;
    ds[(int64_t)b * T + t] = coef_n * (p - (q ? 1.0f : 0.0f)) + gsh[t];
    loss += q ? softplus_f(-z) : softplus_f(z);
  }
  loss = warp_sum(loss);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = loss;
  __syncthreads();
  if (warp == 0) {
    float v = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
    v = warp_sum(v);
    if (lane == 0) loss_part[b] = v;
  }
}

// dx = dy + ds[row] * w_r (every stream row).
template <typename T>
__global__ void __launch_bounds__(BW_WARPS * 32)
dx_init_kernel(int64_t rows, int d, const T* __restrict__ dy, const float* __restrict__ ds,
               const T* __restrict__ w_r, T* __restrict__ dx) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * BW_WARPS + warp;
  if (row >= rows) return;
  const float g = ds[row];
  constexpr int V = Vec16<T>::N;
  for (int c = lane * V; c < d; c += 32 * V) {
    const Vec16<T> yv = ld_vec(dy + row * d + c), wv = ld_vec(w_r + c);
    Vec16<T> o;
#pragma unroll
    for (int k = 0; k < V; ++k) o.set(k, yv.get(k) + g * wv.get(k));
    st_vec(dx + row * d + c, o);
  }
}

// ---------------------------------------------------------------- column reductions
// part[chunk, c] = sum over the chunk's rows m of (A ? A[m, c] : 1) * Bv[row(m), c] *
// (w ? w[m] : 1), rows in order; row(m) is the stream row of compact row m (idx NULL:
// m). One thread per 16-byte vector of columns; grid (column blocks, row chunks).
template <typename TB>
__global__ void __launch_bounds__(256)
coldot_kernel(int64_t M, int d, const float* __restrict__ A, const TB* __restrict__ Bv,
              const int32_t* __restrict__ idx, int seqT, int n, const float* __restrict__ w,
              int64_t rows_per_chunk, float* __restrict__ part) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<TB>::N;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * V;
  if (c >= d) return;
  const int64_t m0 = (int64_t)blockIdx.y * rows_per_chunk;
  const int64_t m1 = min(M, m0 + rows_per_chunk);
  float acc[V];
#pragma unroll
  for (int k = 0; k < V; ++k) acc[k] = 0.0f;
#pragma unroll 8
  for (int64_t m = m0; m < m1; ++m) {
    const int64_t row = idx ? bw_stream_row(m, seqT, n, idx) : m;
    const Vec16<TB> bv = ld_vec(Bv + row * d + c);
    const float wm = w ? w[m] : 1.0f;
    if (A) {
#pragma unroll
      for (int k = 0; k < V; k += 4) {
        const float4 a = *reinterpret_cast<const float4*>(A + m * d + c + k);
        acc[k] += a.x * bv.get(k) * wm;
        acc[k + 1] += a.y * bv.get(k + 1) * wm;
        acc[k + 2] += a.z * bv.get(k + 2) * wm;
        acc[k + 3] += a.w * bv.get(k + 3) * wm;
      }
    } else {
#pragma unroll
      for (int k = 0; k < V; ++k) acc[k] += bv.get(k) * wm;
    }
  }
#pragma unroll
  for (int k = 0; k < V; ++k) part[(int64_t)blockIdx.y * d + c + k] = acc[k];
}

// out[c] = sum over chunks k of part[k, c] in a fixed order: a CTA of 32 x 32 threads
// serves 32 columns; thread (x, y) sums the chunks k = y, y + 32, ... of column x in
// order, then the 32 partial sums are added in order of y.
__global__ void __launch_bounds__(1024)
colsum_kernel(int nchunks, int d, const float* __restrict__ part, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sh[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + tx;
  float acc = 0.0f;
  if (c < d) {
#pragma unroll 4
    for (int k = ty; k < nchunks; k += 32) acc += part[(int64_t)k * d + c];
  }
  sh[ty][tx] = acc;
  __syncthreads();
  if (ty == 0 && c < d) {
    float t = 0.0f;
    for (int y = 0; y < 32; ++y) t += sh[y][tx];
    out[c] = t;
  }
}

// out[0] = scale * sum of in[0 .. n): each thread sums a fixed strided subset in order,
// then a fixed tree; one CTA of 1024 threads.
__global__ void __launch_bounds__(1024)
sum_kernel(int64_t n, const float* __restrict__ in, float scale, float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sh[1024];
  float acc = 0.0f;
  for (int64_t i = threadIdx.x; i < n; i += 1024) acc += in[i];
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 512; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[0] = sh[0] * scale;
}

// ---------------------------------------------------------------- SwiGLU
// gu [M, 2F]: the gate pre-activation G in columns [0, F), the up projection U in [F, 2F).
// One 16-byte vector (V elements) per thread and step; F % V == 0.
template <typename T>
__global__ void swiglu_fwd_kernel(int64_t M, int F, const T* __restrict__ gu, T* __restrict__ H) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int FV = F / V;
  const int64_t total = M * FV;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / FV;
    const int e = (int)(i - m * FV) * V;
    const Vec16<T> g = ld_vec(gu + m * 2 * F + e), u = ld_vec(gu + m * 2 * F + F + e);
    Vec16<T> h;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float gv = g.get(k);
      h.set(k, gv / (1.0f + expf(-gv)) * u.get(k));
    }
    st_vec(H + m * F + e, h);
  }
}

// dG = dH U silu'(G), dU = dH silu(G); silu'(z) = sigmoid(z) (1 + z (1 - sigmoid(z))).
template <typename T>
__global__ void swiglu_bwd_kernel(int64_t M, int F, const T* __restrict__ gu,
                                  const float* __restrict__ dH, T* __restrict__ dgu) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int FV = F / V;
  const int64_t total = M * FV;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / FV;
    const int e = (int)(i - m * FV) * V;
    const Vec16<T> g = ld_vec(gu + m * 2 * F + e), u = ld_vec(gu + m * 2 * F + F + e);
    float dh[V];
#pragma unroll
    for (int k = 0; k < V; k += 4) {
      const float4 q = *reinterpret_cast<const float4*>(dH + m * F + e + k);
      dh[k] = q.x; dh[k + 1] = q.y; dh[k + 2] = q.z; dh[k + 3] = q.w;
    }
    Vec16<T> dg, du;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const float gv = g.get(k), uv = u.get(k);
      const float sg = 1.0f / (1.0f + expf(-gv));
      dg.set(k, dh[k] * uv * sg * (1.0f + gv * (1.0f - sg)));
      du.set(k, dh[k] * gv * sg);
    }
    st_vec(dgu + m * 2 * F + e, dg);
    st_vec(dgu + m * 2 * F + F + e, du);
  }
}

// ---------------------------------------------------------------- RMSNorm backward
// Row m of z = x rho g (rho = (mean x^2 + eps)^-1/2), x = xin[row(m)] (TIN; row(m) the
// stream row through idx, or m): grad = rho (dz g - xhat mean(dz g xhat)).
// RMSNorm2 use (dh_out): dh_out[m] = grad; da_out[m] = grad + dae[m].
// RMSNorm1 use (dx_io): dx_io[row(m)] += dadd[m] + grad.
// rstd_out[m] = rho.
template <typename TIN, typename T>
__global__ void __launch_bounds__(BW_WARPS * 32)
rms_bwd_kernel(int64_t M, int d, const float* __restrict__ dz, const T* __restrict__ g,
               const TIN* __restrict__ xin, const int32_t* __restrict__ idx, int seqT, int n,
               float eps, const T* __restrict__ dae, float* __restrict__ dh_out,
               T* __restrict__ da_out, const float* __restrict__ dadd, T* __restrict__ dx_io,
               float* __restrict__ rstd_out) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * BW_WARPS + warp;
  if (m >= M) return;
  const int64_t row = idx ? bw_stream_row(m, seqT, n, idx) : m;
  const TIN* xr = xin + row * d;
  const float* dzr = dz + m * d;
  float ss = 0.0f;
  for (int c = lane * 4; c < d; c += 128) {
    const float4 v = ld4(xr + c);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  const float rho = rsqrtf(warp_sum(ss) / (float)d + eps);
  float dot = 0.0f;
  for (int c = lane * 4; c < d; c += 128) {
    const float4 z = *reinterpret_cast<const float4*>(dzr + c), gg = ld4(g + c), x = ld4(xr + c);
    dot += (z.x * gg.x * x.x + z.y * gg.y * x.y + z.z * gg.z * x.z + z.w * gg.w * x.w) * rho;
  }
  const float mean = warp_sum(dot) / (float)d;
  for (int c = lane * 4; c < d; c += 128) {
    const float4 z = *reinterpret_cast<const float4*>(dzr + c), gg = ld4(g + c), x = ld4(xr + c);
    float4 gr;
    gr.x = rho * (z.x * gg.x - x.x * rho * mean);
    gr.y = rho * (z.y * gg.y - x.y * rho * mean);
    gr.z = rho * (z.z * gg.z - x.z * rho * mean);
    gr.w = rho * (z.w * gg.w - x.w * rho * mean);
    if (dh_out) {
      *reinterpret_cast<float4*>(dh_out + m * d + c) = gr;
      const float4 e = ld4(dae + m * d + c);
      st4(da_out + m * d + c, make_float4(gr.x + e.x, gr.y + e.y, gr.z + e.z, gr.w + e.w));
    } else {
      T* p = dx_io + row * d + c;
      const float4 cur = ld4(p);
      const float4 ad = dadd ? *reinterpret_cast<const float4*>(dadd + m * d + c)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      st4(p, make_float4(cur.x + (ad.x + gr.x), cur.y + (ad.y + gr.y), cur.z + (ad.z + gr.z),
                         cur.w + (ad.w + gr.w)));
    }
  }
  if (lane == 0) rstd_out[m] = rho;
}


// Selected-Q / full-KV: the RMSNorm1 output u of a selected token feeds its query and its
// key / value. Selected compact row m (stream row t) adds its query-side gradient
// du_sel[m] into du[t] (the keys' and values' part, every token) and puts dh[m] (the
// gradient through h = x + a) in dadd[t], which the caller zeroed.
__global__ void __launch_bounds__(BW_WARPS * 32)
fullkv_merge_kernel(int64_t M, int seqT, int n, int d, const int32_t* __restrict__ idx,
                    const float* __restrict__ du_sel, const float* __restrict__ dh,
                    float* __restrict__ du, float* __restrict__ dadd) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * BW_WARPS + warp;
  if (m >= M) return;
  const int64_t t = bw_stream_row(m, seqT, n, idx);
  for (int c = lane * 4; c < d; c += 128) {
    const float4 q = *reinterpret_cast<const float4*>(du_sel + m * d + c);
    float4* pu = reinterpret_cast<float4*>(du + t * d + c);
    const float4 u = *pu;
    *pu = make_float4(u.x + q.x, u.y + q.y, u.z + q.z, u.w + q.w);
    *reinterpret_cast<float4*>(dadd + t * d + c) =
        *reinterpret_cast<const float4*>(dh + m * d + c);
  }
}

// Selected-Q / full-KV, for the tcgen05 dk / dv kernel: qposS [B, ldS] = the query
// positions qpos [B, n] padded with -1, and qstart [B, nkb] = the first query positioned
// at or after key block kb's first key kb * kvb (n if none). One CTA per sequence.
__global__ void __launch_bounds__(256)
fullkv_qindex_kernel(int n, int ldS, int nkb, int kvb, const int32_t* __restrict__ qpos,
                     int32_t* __restrict__ qposS, int32_t* __restrict__ qstart) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  const int32_t* p = qpos + (int64_t)b * n;
  for (int i = threadIdx.x; i < ldS; i += blockDim.x) qposS[(int64_t)b * ldS + i] = i < n ? p[i] : -1;
  for (int kb = threadIdx.x; kb < nkb; kb += blockDim.x) {
    const int k0 = kb * kvb;
    int lo = 0, hi = n;   // positions ascend: binary search for the first >= k0
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (p[mid] >= k0) hi = mid; else lo = mid + 1;
    }
    qstart[(int64_t)b * nkb + kb] = lo;
  }
}

// ---------------------------------------------------------------- attention backward
// Causal GQA attention on each sequence's n compact rows (query head h reads KV head
// h / (hq / hkv)), or on n queries at ascending positions over nk keys, each query seeing
// the keys at or before its position (Selected-Q / full-KV); FFMA tiles of 32 queries x
// 32 keys in shared memory (fp32).
// bwd_q: per (32-query tile, head, sequence): the row statistics lse = m + log l, D =
//        <dO, O>, then dQ = scale * sum_j P (dP - D) K_j with P = exp(scale q.k - lse),
//        dP = dO . v_j.
// bwd_kv: per (32-key tile, KV head, sequence), over the group's query heads and the
//        queries from the first one positioned at or after the tile's first key: dV =
//        sum_i P dO_i, dK = scale * sum_i
//        P (dP - D) q_i. Every key row is owned by one CTA: no atomics.
struct AttnBwd {
  int n, hq, hkv;      // n queries per sequence
  int nk;              // keys per sequence
  const int32_t* qpos; // [B*n] ascending positions of the queries among the nk keys; query
                       // i sees keys j <= qpos[i] (NULL: j <= i, nk == n)
  const void* q;       // q of head h at column h*HD of [B*n, ldq]
  int ldq;
  const void* k;       // k of KV head g at column g*HD of [B*nk, ldk]
  int ldk;
  const void* v;       // vt_mode 0: v of KV head g at column g*HD of [B*nk, ldv];
  int vt_mode;         // 1: v transposed, [B, hkv, HD, vt_ld] (keys contiguous)
  int ldv, vt_ld;
  const void* o;       // [B*n, hq*HD]
  const float* dO;     // [B*n, hq*HD]
  float* lse;          // [B*n, hq]
  float* Dd;           // [B*n, hq]
  void* dq;            // dq of head h at column h*HD of [B*n, ldgq]
  int ldgq;
  void* dk;            // dk, dv of KV head g at column g*HD of [B*nk, ldgk]
  void* dv;
  int ldgk;
  float scale;
};

constexpr int AB_T = 32;   // queries and keys per tile

template <typename T, int HD>
__device__ __forceinline__ float ab_v(const AttnBwd& p, int b, int g, int j, int c) {
  if (p.vt_mode)
    return Elem<T>::to_f(((const T*)p.v)[(((int64_t)b * p.hkv + g) * HD + c) * p.vt_ld + j]);
  return Elem<T>::to_f(((const T*)p.v)[((int64_t)b * p.nk + j) * p.ldv + g * HD + c]);
}

// position of query i of sequence b among its keys
__device__ __forceinline__ int ab_qpos(const AttnBwd& p, int b, int i) {
  return p.qpos ? p.qpos[(int64_t)b * p.n + i] : i;
}

template <typename T, int HD>
__global__ void __launch_bounds__(256)
attn_bwd_q_kernel(const AttnBwd p) {
  pdl_trigger();
  pdl_wait();
  constexpr int P = HD + 1, KC = HD / 32;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* dOs = Qs + AB_T * P;
  float* Ks = dOs + AB_T * P;
  float* Vs = Ks + AB_T * P;
  float* dSs = Vs + AB_T * P;   // [AB_T][AB_T + 1]
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (p.hq / p.hkv);
  const int qw = p.hq * HD;
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int q0 = qt * AB_T;
  const T* Q = (const T*)p.q;
  const T* Kp = (const T*)p.k;
  for (int e = tid; e < AB_T * HD; e += 256) {
    const int i = e / HD, c = e - i * HD, qi = q0 + i;
    const int64_t row = (int64_t)b * p.n + qi;
    Qs[i * P + c] = qi < p.n ? Elem<T>::to_f(Q[row * p.ldq + h * HD + c]) : 0.0f;
    dOs[i * P + c] = qi < p.n ? p.dO[row * qw + h * HD + c] : 0.0f;
  }
  __syncthreads();
  float Dr[4], mr[4], lr[4];
  int qp[4];   // the rows' positions (-1 past the sequence: no key)
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = ty + 8 * r, qi = q0 + i;
    float acc = 0.0f;
    if (qi < p.n)
      for (int c = tx; c < HD; c += 32)
        acc += dOs[i * P + c] *
               Elem<T>::to_f(((const T*)p.o)[((int64_t)b * p.n + qi) * qw + h * HD + c]);
    Dr[r] = warp_sum(acc);
    mr[r] = -INFINITY;
    lr[r] = 0.0f;
    qp[r] = qi < p.n ? ab_qpos(p, b, qi) : -1;
  }
  // the key tiles up to the tile's last query position (positions ascend)
  const int kmax = ab_qpos(p, b, min(q0 + AB_T, p.n) - 1);
  const int nkt = kmax / AB_T + 1;
  // pass 1: row max and sum over the keys at or before each query
  for (int kt = 0; kt < nkt; ++kt) {
    const int k0 = kt * AB_T;
    for (int e = tid; e < AB_T * HD; e += 256) {
      const int j = e / HD, c = e - j * HD, kj = k0 + j;
      Ks[j * P + c] = kj < p.nk
          ? Elem<T>::to_f(Kp[((int64_t)b * p.nk + kj) * p.ldk + g * HD + c]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = ty + 8 * r, kj = k0 + tx;
      float s = 0.0f;
#pragma unroll 8
      for (int c = 0; c < HD; ++c) s += Qs[i * P + c] * Ks[tx * P + c];
      s *= p.scale;
      const bool ok = kj < p.nk && kj <= qp[r];
      const float mx = warp_max(ok ? s : -INFINITY);
      if (mx > -INFINITY) {   // uniform over the warp (one row per warp)
        const float mn = fmaxf(mr[r], mx);
        const float add = warp_sum(ok ? expf(s - mn) : 0.0f);
        lr[r] = lr[r] * expf(mr[r] - mn) + add;
        mr[r] = mn;
      }
    }
    __syncthreads();
  }
  float lse[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = ty + 8 * r, qi = q0 + i;
    lse[r] = mr[r] + logf(lr[r]);
    if (tx == 0 && qi < p.n) {
      p.lse[((int64_t)b * p.n + qi) * p.hq + h] = lse[r];
      p.Dd[((int64_t)b * p.n + qi) * p.hq + h] = Dr[r];
    }
  }
  // pass 2: dQ
  float dq[4][KC];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int k = 0; k < KC; ++k) dq[r][k] = 0.0f;
  for (int kt = 0; kt < nkt; ++kt) {
    const int k0 = kt * AB_T;
    for (int e = tid; e < AB_T * HD; e += 256) {
      const int j = e / HD, c = e - j * HD, kj = k0 + j;
      const bool ok = kj < p.nk;
      Ks[j * P + c] = ok
          ? Elem<T>::to_f(Kp[((int64_t)b * p.nk + kj) * p.ldk + g * HD + c]) : 0.0f;
      Vs[j * P + c] = ok ? ab_v<T, HD>(p, b, g, kj, c) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = ty + 8 * r, kj = k0 + tx;
      float s = 0.0f, dp = 0.0f;
#pragma unroll 8
      for (int c = 0; c < HD; ++c) {
        s += Qs[i * P + c] * Ks[tx * P + c];
        dp += dOs[i * P + c] * Vs[tx * P + c];
      }
      const bool ok = kj < p.nk && kj <= qp[r];
      const float pr = ok ? expf(s * p.scale - lse[r]) : 0.0f;
      dSs[i * (AB_T + 1) + tx] = pr * (dp - Dr[r]);
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = ty + 8 * r;
#pragma unroll
      for (int k = 0; k < KC; ++k) {
        const int c = tx + 32 * k;
        float acc = 0.0f;
#pragma unroll 8
        for (int j = 0; j < AB_T; ++j) acc += dSs[i * (AB_T + 1) + j] * Ks[j * P + c];
        dq[r][k] += acc;
      }
    }
    __syncthreads();
  }
  T* out = (T*)p.dq;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int qi = q0 + ty + 8 * r;
    if (qi >= p.n) continue;
#pragma unroll
    for (int k = 0; k < KC; ++k)
      out[((int64_t)b * p.n + qi) * p.ldgq + h * HD + tx + 32 * k] =
          Elem<T>::from_f(dq[r][k] * p.scale);
  }
}

template <typename T, int HD>
__global__ void __launch_bounds__(256)
attn_bwd_kv_kernel(const AttnBwd p) {
  pdl_trigger();
  pdl_wait();
  constexpr int P = HD + 1, KC = HD / 32;
  extern __shared__ float sm[];
  float* Ks = sm;
  float* Vs = Ks + AB_T * P;
  float* Qs = Vs + AB_T * P;
  float* dOs = Qs + AB_T * P;
  float* Ps = dOs + AB_T * P;          // [key][query], AB_T + 1 wide
  float* dSs = Ps + AB_T * (AB_T + 1);
  float* lse_s = dSs + AB_T * (AB_T + 1);
  float* D_s = lse_s + AB_T;
  int* qp_s = (int*)(D_s + AB_T);
  const int kt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = p.hq / p.hkv;
  const int qw = p.hq * HD;
  const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
  const int k0 = kt * AB_T;
  const T* Q = (const T*)p.q;
  const T* Kp = (const T*)p.k;
  for (int e = tid; e < AB_T * HD; e += 256) {
    const int j = e / HD, c = e - j * HD, kj = k0 + j;
    const bool ok = kj < p.nk;
    Ks[j * P + c] = ok
        ? Elem<T>::to_f(Kp[((int64_t)b * p.nk + kj) * p.ldk + g * HD + c]) : 0.0f;
    Vs[j * P + c] = ok ? ab_v<T, HD>(p, b, g, kj, c) : 0.0f;
  }
  // the first query at or after the tile's first key: positions ascend, so a binary search
  // (the same in every thread)
  int qstart = p.n;
  {
    int lo = 0, hi = p.n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (ab_qpos(p, b, mid) >= k0) hi = mid; else lo = mid + 1;
    }
    qstart = lo;
  }
  float dk[4][KC], dv[4][KC];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int k = 0; k < KC; ++k) dk[r][k] = dv[r][k] = 0.0f;
  for (int hh = 0; hh < G; ++hh) {
    const int h = g * G + hh;
    for (int q0 = qstart; q0 < p.n; q0 += AB_T) {
      __syncthreads();   // the previous tile's readers are done
      for (int e = tid; e < AB_T * HD; e += 256) {
        const int i = e / HD, c = e - i * HD, qi = q0 + i;
        const int64_t row = (int64_t)b * p.n + qi;
        Qs[i * P + c] = qi < p.n ? Elem<T>::to_f(Q[row * p.ldq + h * HD + c]) : 0.0f;
        dOs[i * P + c] = qi < p.n ? p.dO[row * qw + h * HD + c] : 0.0f;
      }
      if (tid < AB_T) {
        const int qi = q0 + tid;
        lse_s[tid] = qi < p.n ? p.lse[((int64_t)b * p.n + qi) * p.hq + h] : 0.0f;
        D_s[tid] = qi < p.n ? p.Dd[((int64_t)b * p.n + qi) * p.hq + h] : 0.0f;
        qp_s[tid] = qi < p.n ? ab_qpos(p, b, qi) : -1;
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = ty + 8 * r, kj = k0 + j;
        float s = 0.0f, dp = 0.0f;
#pragma unroll 8
        for (int c = 0; c < HD; ++c) {
          s += Ks[j * P + c] * Qs[tx * P + c];
          dp += Vs[j * P + c] * dOs[tx * P + c];
        }
        const bool ok = kj < p.nk && kj <= qp_s[tx];
        const float pr = ok ? expf(s * p.scale - lse_s[tx]) : 0.0f;
        Ps[j * (AB_T + 1) + tx] = pr;
        dSs[j * (AB_T + 1) + tx] = pr * (dp - D_s[tx]);
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = ty + 8 * r;
#pragma unroll
        for (int k = 0; k < KC; ++k) {
          const int c = tx + 32 * k;
          float av = 0.0f, ak = 0.0f;
#pragma unroll 8
          for (int i = 0; i < AB_T; ++i) {
            av += Ps[j * (AB_T + 1) + i] * dOs[i * P + c];
            ak += dSs[j * (AB_T + 1) + i] * Qs[i * P + c];
          }
          dv[r][k] += av;
          dk[r][k] += ak;
        }
      }
    }
  }
  T* odk = (T*)p.dk;
  T* odv = (T*)p.dv;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int kj = k0 + ty + 8 * r;
    if (kj >= p.nk) continue;
    const int64_t row = ((int64_t)b * p.nk + kj) * p.ldgk;
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const int c = tx + 32 * k;
      odk[row + g * HD + c] = Elem<T>::from_f(dk[r][k] * p.scale);
      odv[row + g * HD + c] = Elem<T>::from_f(dv[r][k]);
    }
  }
}

// ---------------------------------------------------------------- host side

constexpr size_t kBwAlign = 256;
inline size_t bw_align(size_t v) { return (v + kBwAlign - 1) / kBwAlign * kBwAlign; }
inline int64_t round8(int64_t v) { return (v + 7) / 8 * 8; }

// Workspace carve-up of the backward; M = B*T rows cover a dense layer.
struct BwLayout {
  size_t status, s, r, idx, r_sel, dr, dvs, ds, lossp, u, qkv, vt, o, a, h, v2, gu, H, f, df,
      dae, dH, dGU, dv2, dh, da, dO, lse, Dd, dqkv, du, rstd1, rstd2, tA, tB, tW, part, qkpre,
      dgq, dgk, lseT, DdT, qposS, qstart, total;
};

constexpr int kMaxChunks = 1024;   // row chunks of the column reductions

BwLayout bw_layout(const xmod_dims* dm) {
  BwLayout L{};
  const size_t es = dm->dtype == XMOD_BF16 ? 2 : 4;
  const size_t BT = (size_t)dm->B * dm->T, M = BT, Mp = (size_t)round8((int64_t)M);
  const size_t d = dm->d, F = dm->d_ff, hq = dm->n_heads, hd = dm->head_dim;
  const size_t qw = hq * hd, kw = (size_t)dm->n_kv_heads * hd, qkv_w = qw + 2 * kw;
  const size_t vtl = (size_t)round8(dm->T);
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = bw_align(off + bytes); return o; };
  L.status = take(kBwAlign);
  L.s = take(4 * BT);
  L.r = take(4 * BT);
  L.idx = take(4 * BT);
  L.r_sel = take(4 * BT);
  L.dr = take(4 * BT);
  L.dvs = take(4 * BT);
  L.ds = take(4 * BT);
  L.lossp = take(4 * (size_t)dm->B);
  L.u = take(es * M * d);
  L.qkv = take(es * M * qkv_w);
  L.vt = take(es * (size_t)dm->B * dm->n_kv_heads * hd * vtl);
  L.o = take(es * M * qw);
  L.a = take(es * M * d);
  L.h = take(4 * M * d);
  L.v2 = take(es * M * d);
  L.gu = take(es * M * 2 * F);
  L.H = take(es * M * F);
  L.f = take(es * M * d);
  L.df = take(es * M * d);
  L.dae = take(es * M * d);
  L.dH = take(4 * M * F);
  L.dGU = take(es * M * 2 * F);
  L.dv2 = take(4 * M * d);
  L.dh = take(4 * M * d);
  L.da = take(es * M * d);
  L.dO = take(4 * M * qw);
  L.lse = take(4 * M * hq);
  L.Dd = take(4 * M * hq);
  L.dqkv = take(es * M * qkv_w);
  L.du = take(4 * M * d);
  L.rstd1 = take(4 * M);
  L.rstd2 = take(4 * M);
  L.tA = take(es * Mp * std::max(std::max(d, 2 * F), qkv_w));
  L.tB = take(es * Mp * std::max(std::max(d, F), qw));
  L.tW = take(es * d * (3 * F + qw + qkv_w));   // every transposed weight of a layer
  L.part = take(4 * (size_t)kMaxChunks * std::max(d, (size_t)1));
  L.qkpre = take(es * M * (qw + kw));   // q | k before the QK-norm / rotation
  L.dgq = take(4 * M * hd);
  L.dgk = take(4 * M * hd);
  const size_t lds = ((size_t)dm->T + 63) / 64 * 64;
  L.lseT = take(4 * (size_t)dm->B * hq * lds);
  L.DdT = take(4 * (size_t)dm->B * hq * lds);
  L.qposS = take(4 * (size_t)dm->B * lds);   // full-KV: query positions, padded
  L.qstart = take(4 * (size_t)dm->B * (((size_t)dm->T + kAttnBwdKvBlock - 1) / kAttnBwdKvBlock));
  L.total = off;
  return L;
}

inline char* bat(void* ws, size_t off) { return (char*)ws + off; }

#define BW_RUN(kind, expr)                        \
  do {                                            \
    cudaError_t _e;                               \
    {                                             \
      ProfScope _p(kind, c.stream);               \
      _e = (expr);                                \
    }                                             \
    count_launch();                               \
    if (_e != cudaSuccess) return XMOD_ERR_CUDA;  \
  } while (0)

// out[c, r] = in[r, c] (zero for R <= r < Rpad) of T-typed matrices (2- or 4-byte).
template <typename T>
cudaError_t transpose_t(const Ctx& c, int R, int Rpad, int C, const void* in, int64_t ldi,
                        void* out, int64_t ldo, int batch, int64_t in_bs, int64_t out_bs) {
  if (R <= 0 || C <= 0 || batch <= 0) return cudaSuccess;
  using U = typename std::conditional<sizeof(T) == 2, uint16_t, uint32_t>::type;
  constexpr int V = 16 / sizeof(U);
  const int vec_in = ((uintptr_t)in % 16 == 0 && ldi % V == 0 && in_bs % V == 0) ? 1 : 0;
  const int vec_out = ((uintptr_t)out % 16 == 0 && ldo % V == 0 && out_bs % V == 0) ? 1 : 0;
  const dim3 grid((C + TR_T - 1) / TR_T, (Rpad + TR_T - 1) / TR_T, batch);
  return launch_pdl(transpose_kernel<U>, grid, dim3(256), 0, c.stream, R, Rpad, C,
                    (const U*)in, ldi, (U*)out, ldo, in_bs, out_bs, vec_in, vec_out);
}

// One transpose of a multi-transpose launch: out[c, r] = in[r, c] (zero for R <= r < Rpad),
// per batch entry in_bs / out_bs elements further.
struct TrSpec {
  const void* in;
  int64_t ldi;
  void* out;
  int64_t ldo;
  int R, Rpad, C;
  int64_t in_bs, out_bs;
};

// Up to kTrMaxJobs independent transposes of T-typed matrices in one launch.
template <typename T>
cudaError_t transpose_multi_t(const Ctx& c, const TrSpec* specs, int nspecs, int batch) {
  using U = typename std::conditional<sizeof(T) == 2, uint16_t, uint32_t>::type;
  constexpr int V = 16 / sizeof(U);
  if (nspecs > kTrMaxJobs || batch <= 0) return cudaErrorInvalidValue;
  TrJobs jobs{};
  int total = 0;
  for (int i = 0; i < nspecs; ++i) {
    const TrSpec& s = specs[i];
    if (s.R <= 0 || s.C <= 0) continue;
    TrJob& J = jobs.j[jobs.n++];
    J.in = s.in;
    J.out = s.out;
    J.ldi = s.ldi;
    J.ldo = s.ldo;
    J.in_bs = s.in_bs;
    J.out_bs = s.out_bs;
    J.R = s.R;
    J.Rpad = s.Rpad;
    J.C = s.C;
    J.tiles_x = (s.C + TR_T - 1) / TR_T;
    J.start = total;
    J.vec_in = ((uintptr_t)s.in % 16 == 0 && s.ldi % V == 0 && s.in_bs % V == 0) ? 1 : 0;
    J.vec_out = ((uintptr_t)s.out % 16 == 0 && s.ldo % V == 0 && s.out_bs % V == 0) ? 1 : 0;
    total += J.tiles_x * ((s.Rpad + TR_T - 1) / TR_T);
  }
  if (jobs.n == 0) return cudaSuccess;
  return launch_pdl(transpose_multi_kernel<U>, dim3(total, batch), dim3(256), 0, c.stream, jobs);
}

cudaError_t transpose_multi(const Ctx& c, xmod_dtype dt, const TrSpec* specs, int nspecs,
                            int batch = 1) {
  return dt == XMOD_BF16 ? transpose_multi_t<__nv_bfloat16>(c, specs, nspecs, batch)
                         : transpose_multi_t<float>(c, specs, nspecs, batch);
}
cudaError_t transpose_multi(const Ctx& c, xmod_dtype dt, std::initializer_list<TrSpec> specs,
                            int batch = 1) {
  return transpose_multi(c, dt, specs.begin(), (int)specs.size(), batch);
}

// The transposed weights of a layer's backward, each in its own part of the tW scratch:
// W_down^T [F, d]; [W_gate | W_up]^T [d, 2F]; W_o^T [qw, d]; [W_q | W_k | W_v]^T
// [d, qkv_w] (Selected-Q / full-KV: W_q^T [d, qw], then [W_k | W_v]^T [d, 2 kw]).
template <typename E>
struct TwParts {
  E *d, *gu, *o, *qkv;
};
template <typename E>
TwParts<E> tw_parts(const xmod_dims* dm, E* tW) {
  const size_t d = dm->d, F = dm->d_ff, qw = (size_t)dm->n_heads * dm->head_dim;
  return {tW, tW + F * d, tW + 3 * F * d, tW + (3 * F + qw) * d};
}

// C[M, N] = A[M, K] B[N, K]^T, both K-contiguous, stored plain (fp32 if f32out, else
// the layer's type): tcgen05 for bf16 when the shape allows, FFMA otherwise.
cudaError_t bw_gemm(const Ctx& c, xmod_dtype dt, int M, int N, int K, const void* A, int lda,
                    const void* Bm, int ldb, void* out, int ldo, bool f32out) {
  Epilogue e;
  e.kind = EPI_STORE;
  e.out = out;
  e.ldo = ldo;
  e.out_f32 = f32out;
  if (dt == XMOD_BF16) {
    GemmTcProblem p;
    p.M = M; p.N = N; p.K = K; p.A = A; p.lda = lda; p.B[0] = Bm; p.ldb = ldb;
    if (gemm_tc_supported(p, e)) return launch_gemm_tc(c, p, e);
  }
  return launch_gemm_simt(c, dt, M, N, K, A, lda, Bm, ldb, nullptr, e);
}

// The fp32 weight gradients of weights stacked along M in one GEMM: C = A B^T with rows
// [0, s0) to o0, [s0, s1) to o1 and [s1, M) to o2 (s1 = 0: rows [s0, M) to o1), each
// [rows, N] with row stride ldo. tcgen05 when the shape allows (one launch), else one
// GEMM per part.
cudaError_t bw_gemm_dw_split(const Ctx& c, xmod_dtype dt, int M, int N, int K, const void* A,
                             int lda, const void* Bm, int ldb, float* o0, float* o1, float* o2,
                             int s0, int s1, int ldo) {
  if (dt == XMOD_BF16) {
    Epilogue e;
    e.kind = EPI_STORE;
    e.out = o0;
    e.ldo = ldo;
    e.out_f32 = true;
    e.row_split[0] = s0;
    e.out_rows[0] = o1;
    if (s1 > 0) {
      e.row_split[1] = s1;
      e.out_rows[1] = o2;
    }
    GemmTcProblem p;
    p.M = M; p.N = N; p.K = K; p.A = A; p.lda = lda; p.B[0] = Bm; p.ldb = ldb;
    if (gemm_tc_supported(p, e)) return launch_gemm_tc(c, p, e);
  }
  const size_t es = dt == XMOD_BF16 ? 2 : 4;
  const int parts = s1 > 0 ? 3 : 2;
  const int ends[3] = {s0, s1 > 0 ? s1 : M, M};
  float* outs[3] = {o0, o1, o2};
  int r0 = 0;
  for (int i = 0; i < parts; ++i) {
    if (i > 0) count_launch();   // the caller counts one launch
    const cudaError_t err = bw_gemm(c, dt, ends[i] - r0, N, K, (const char*)A + es * (size_t)r0 * lda,
                                    lda, Bm, ldb, outs[i], ldo, true);
    if (err != cudaSuccess) return err;
    r0 = ends[i];
  }
  return cudaSuccess;
}

// A weight gradient dW = Y^T X in fp32 straight from the token-major Y [rows, Mo] (row
// stride ldy) and X [rows, N] (row stride ldx): the tensor-core GEMM reads both as stored
// (MN-major operands, the contraction over the token rows; rows past `rows` read as 0),
// so no token-contiguous copies are made. Rows [0, s0) of dW go to o0, [s0, s1) (or
// [s0, Mo) when s1 = 0) to o1, [s1, Mo) to o2; s0 = 0: all of dW to o0; row stride ldo.
// ok is false where that GEMM does not take the type or shape (the caller transposes).
struct DwDirect {
  GemmTcProblem p;
  Epilogue e;
  bool ok = false;
};
DwDirect dw_direct(xmod_dtype dt, int Mo, int N, int rows, const void* Y, int ldy, const void* X,
                   int ldx, float* o0, float* o1, float* o2, int s0, int s1, int ldo) {
  DwDirect w;
  w.e.kind = EPI_STORE;
  w.e.out = o0;
  w.e.ldo = ldo;
  w.e.out_f32 = true;
  if (s0 > 0) {
    w.e.row_split[0] = s0;
    w.e.out_rows[0] = o1;
    if (s1 > 0) {
      w.e.row_split[1] = s1;
      w.e.out_rows[1] = o2;
    }
  }
  w.p.M = Mo;
  w.p.N = N;
  w.p.K = rows;
  w.p.A = Y;
  w.p.lda = ldy;
  w.p.B[0] = X;
  w.p.ldb = ldx;
  w.p.a_mn = 1;
  w.p.b_mn = 1;
  w.ok = dt == XMOD_BF16 && rows > 0 && gemm_tc_supported(w.p, w.e);
  return w;
}

// An activation gradient dX [rows, N] = dY [rows, K] W (row strides ldy, ldo; fp32 out if
// f32out), W a projection's weights stacked along K -- w0 for k < k1, w1 for k1 <= k < k2
// (or < K when w2 is null), w2 for k >= k2, each [part rows, N] with row stride ldw:
// the tensor-core GEMM reads the weights as stored (an MN-major B operand, one tensor
// map per part), so they are not transposed. ok is false where that GEMM does not take
// the type or shape.
struct DxDirect {
  GemmTcProblem p;
  Epilogue e;
  bool ok = false;
};
DxDirect dx_direct(xmod_dtype dt, int rows, int N, int K, const void* dY, int ldy, const void* w0,
                   const void* w1, const void* w2, int k1, int k2, int ldw, void* out, int ldo,
                   bool f32out) {
  DxDirect x;
  x.e.kind = EPI_STORE;
  x.e.out = out;
  x.e.ldo = ldo;
  x.e.out_f32 = f32out;
  x.p.M = rows;
  x.p.N = N;
  x.p.K = K;
  x.p.A = dY;
  x.p.lda = ldy;
  x.p.B[0] = w0;
  x.p.B[1] = w1;
  x.p.B[2] = w2;
  x.p.nB = w2 ? 3 : w1 ? 2 : 1;
  x.p.split[0] = k1;
  x.p.split[1] = k2;
  x.p.ldb = ldw;
  x.p.b_mn = 1;
  x.ok = dt == XMOD_BF16 && rows > 0 && gemm_tc_supported(x.p, x.e);
  return x;
}

// Column sums out[c] = sum_m (A ? A[m, c] : 1) * Bv[row(m), c] * (w ? w[m] : 1).
template <typename TB>
int bw_coldot(const Ctx& c, int64_t M, int d, const float* A, const TB* Bv, const int32_t* idx,
              int seqT, int n, const float* w, float* part, float* out) {
  constexpr int V = 16 / sizeof(TB);
  int64_t chunks = std::min<int64_t>(kMaxChunks, std::max<int64_t>(1, (M + 15) / 16));
  const int64_t rpc = (M + chunks - 1) / chunks;
  chunks = (M + rpc - 1) / rpc;
  const dim3 grid((d / V + 255) / 256, (unsigned)chunks);
  BW_RUN("bwd_reduce", launch_pdl(coldot_kernel<TB>, grid, dim3(256), 0, c.stream, M, d, A, Bv,
                                  idx, seqT, n, w, rpc, part));
  BW_RUN("bwd_reduce", launch_pdl(colsum_kernel, dim3((d + 31) / 32), dim3(1024), 0, c.stream,
                                  (int)chunks, d, (const float*)part, out));
  return XMOD_OK;
}

template <typename T, int HD>
cudaError_t launch_attn_bwd_t(const Ctx& c, int B, const AttnBwd& p) {
  constexpr int P = HD + 1;
  const size_t smq = sizeof(float) * (4 * AB_T * P + AB_T * (AB_T + 1));
  const size_t smk = sizeof(float) * (4 * AB_T * P + 2 * AB_T * (AB_T + 1) + 3 * AB_T);
  cudaFuncSetAttribute(attn_bwd_q_kernel<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smq);
  cudaFuncSetAttribute(attn_bwd_kv_kernel<T, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smk);
  const int qtiles = (p.n + AB_T - 1) / AB_T, ktiles = (p.nk + AB_T - 1) / AB_T;
  cudaError_t e = launch_pdl(attn_bwd_q_kernel<T, HD>, dim3(qtiles, p.hq, B), dim3(256), smq,
                             c.stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_bwd_kv_kernel<T, HD>, dim3(ktiles, p.hkv, B), dim3(256), smk, c.stream,
                    p);
}

cudaError_t launch_attn_bwd(const Ctx& c, xmod_dtype dt, int B, int hd, const AttnBwd& p) {
  if (dt == XMOD_BF16) {
    switch (hd) {
      case 32: return launch_attn_bwd_t<__nv_bfloat16, 32>(c, B, p);
      case 64: return launch_attn_bwd_t<__nv_bfloat16, 64>(c, B, p);
      case 128: return launch_attn_bwd_t<__nv_bfloat16, 128>(c, B, p);
    }
  } else {
    switch (hd) {
      case 32: return launch_attn_bwd_t<float, 32>(c, B, p);
      case 64: return launch_attn_bwd_t<float, 64>(c, B, p);
      case 128: return launch_attn_bwd_t<float, 128>(c, B, p);
    }
  }
  return cudaErrorInvalidValue;
}

// The Selected-Q / full-KV layer's backward from the attention down (X-MoD notes,
// "mechanism controls"): the selected tokens' queries qb [M, qw] (M = B * T/K rows, at
// positions idx) over the keys and values kvb [B*T, 2kw] of every token (v also
// transposed, in vt, when v_transposed); dO [M, qw] (bf16 with mma, else fp32) and dh
// [M, d] (the gradient through h = x_sel + a) come from the block's backward above. The
// attention backward runs on the warp-level tensor-core MMA with mma (bf16, head_dim 64 or
// 128), on FFMA tiles otherwise. Every token's row of dx receives the gradient through its
// key and value; the selected ones, through their query too.
template <typename E>
int fullkv_tail(const Ctx& c, const xmod_dims* dm, int n, const xmod_layer_weights* w,
                const void* x, const int32_t* idx, void* dx, const xmod_layer_grads* gr,
                void* ws, const BwLayout& L, const E* kvb, const E* qb, const E* kpre,
                const E* qpre, const E* vt, bool v_transposed, const E* o, const void* dO,
                bool mma, const float* dh, bool dx_mn) {
  const xmod_dtype dt = dm->dtype;
  const int B = dm->B, T = dm->T, d = dm->d, hq = dm->n_heads, hkv = dm->n_kv_heads,
            hd = dm->head_dim;
  const int qw = hq * hd, kw = hkv * hd;
  const int M = B * n, Mp = (int)round8(M);
  const int BT = B * T, BTp = (int)round8(BT);
  E* dqkv = (E*)bat(ws, L.dqkv);
  E* dkv = dqkv;                               // [BT, 2kw]: dk | dv of every token
  E* dqb = dqkv + (size_t)BT * 2 * kw;         // [M, qw]: dq of the selected tokens
  E* tA = (E*)bat(ws, L.tA);
  E* tB = (E*)bat(ws, L.tB);
  const TwParts<E> tw = tw_parts<E>(dm, (E*)bat(ws, L.tW));   // transposed by the caller
  float* part = (float*)bat(ws, L.part);

  // ======== attention: n queries per sequence over its T keys
  const int ldS = (n + 63) / 64 * 64;
  const bool tc_bwd = mma && v_transposed && attn_bwd_dq_tc_supported(hd, qw, qw);
  if (tc_bwd) {   // tcgen05 (the forward wrote lse): dq, then dk and dv over every key
    float* lseT = (float*)bat(ws, L.lseT);
    float* DdT = (float*)bat(ws, L.DdT);
    int32_t* qposS = (int32_t*)bat(ws, L.qposS);
    int32_t* qstart = (int32_t*)bat(ws, L.qstart);
    const int nkb = (T + kAttnBwdKvBlock - 1) / kAttnBwdKvBlock;
    // the rows' lse per sequence and head, queries contiguous [hq, n]
    BW_RUN("bwd_transpose", transpose_t<float>(c, n, n, hq, bat(ws, L.lse), hq, lseT, ldS, B,
                                               (int64_t)n * hq, (int64_t)hq * ldS));
    BW_RUN("bwd_rows", launch_pdl(fullkv_qindex_kernel, dim3(B), dim3(256), 0, c.stream, n, ldS,
                                  nkb, kAttnBwdKvBlock, idx, qposS, qstart));
    BW_RUN("bwd_attention",
           launch_attn_bwd_dq_tc_kv(c, B, n, T, idx, hq, hkv, qb, qw, kvb, 2 * kw, 0, kw, o, dO,
                                    (const float*)bat(ws, L.lse), (float*)bat(ws, L.Dd), dqb, qw,
                                    DdT, ldS));
    BW_RUN("bwd_attention",
           launch_attn_bwd_dkv_tc_kv(c, B, n, T, qposS, qstart, hq, hkv, qb, qw, kvb, 2 * kw, 0,
                                     kw, dO, lseT, DdT, ldS, dkv, dkv + kw, 2 * kw));
  } else if (mma) {
    BW_RUN("bwd_attention",
           launch_attn_bwd_mma_kv(c, B, n, T, idx, hq, hkv, hd, qb, qw, kvb, 2 * kw, kvb + kw,
                                  2 * kw, o, dO, (float*)bat(ws, L.lse), (float*)bat(ws, L.Dd),
                                  dqb, qw, dkv, dkv + kw, 2 * kw));
  } else {
  AttnBwd p;
  p.n = n;
  p.nk = T;
  p.qpos = idx;
  p.hq = hq;
  p.hkv = hkv;
  p.q = qb;
  p.ldq = qw;
  p.k = kvb;
  p.ldk = 2 * kw;
  p.v = v_transposed ? (const void*)vt : (const void*)(kvb + kw);
  p.vt_mode = v_transposed ? 1 : 0;
  p.ldv = 2 * kw;
  p.vt_ld = (int)round8(T);
  p.o = o;
  p.dO = (const float*)dO;
  p.lse = (float*)bat(ws, L.lse);
  p.Dd = (float*)bat(ws, L.Dd);
  p.dq = dqb;
  p.ldgq = qw;
  p.dk = dkv;
  p.dv = dkv + kw;
  p.ldgk = 2 * kw;
  p.scale = 1.0f / sqrtf((float)hd);
  BW_RUN("bwd_attention", launch_attn_bwd(c, dt, B, hd, p));
  }

  if (w->q_norm || w->k_norm || w->rope_theta > 0.0f) {   // back through the QK-norm, rotation
    float* dgq = w->q_norm ? (float*)bat(ws, L.dgq) : nullptr;
    float* dgk = w->k_norm ? (float*)bat(ws, L.dgk) : nullptr;
    BW_RUN("bwd_rows", launch_qk_transform_bwd(c, dt, M, dqb, qw, 0, hq, w->q_norm, 0, 0, nullptr,
                                               qpre, qw, hd, dm->rms_eps, w->rope_theta, idx, T,
                                               dgq, nullptr));
    BW_RUN("bwd_rows", launch_qk_transform_bwd(c, dt, BT, dkv, 2 * kw, 0, 0, nullptr, 0, hkv,
                                               w->k_norm, kpre, kw, hd, dm->rms_eps,
                                               w->rope_theta, nullptr, T, nullptr, dgk));
    if (dgq) {
      const int st = bw_coldot<float>(c, M, hd, nullptr, dgq, nullptr, T, n, nullptr, part,
                                      gr->q_norm);
      if (st) return st;
    }
    if (dgk) {
      const int st = bw_coldot<float>(c, BT, hd, nullptr, dgk, nullptr, T, T, nullptr, part,
                                      gr->k_norm);
      if (st) return st;
    }
  }

  // ======== q = u_sel Wq^T (u_sel again in the RMSNorm2 buffer, which the FFN is done with)
  E* u = (E*)bat(ws, L.u);
  E* usel = (E*)bat(ws, L.v2);
  BW_RUN("gather_rmsnorm",
         launch_gather_rmsnorm(c, dt, B, T, n, d, x, idx, w->rms1, dm->rms_eps, usel));
  const DwDirect dwq = dw_direct(dt, qw, d, M, dqb, qw, usel, d, gr->wq, nullptr, nullptr, 0, 0, d);
  if (dwq.ok) {
    BW_RUN("bwd_gemm_dw", launch_gemm_tc(c, dwq.p, dwq.e));
  } else {   // dq^T [qw, Mp], u_sel^T [d, Mp]
    BW_RUN("bwd_transpose", transpose_multi(c, dt, {{dqb, qw, tA, Mp, M, Mp, qw, 0, 0},
                                                    {usel, d, tB, Mp, M, Mp, d, 0, 0}}));
    BW_RUN("bwd_gemm_dw", bw_gemm(c, dt, qw, d, Mp, tA, Mp, tB, Mp, gr->wq, d, true));
  }
  float* du_sel = (float*)bat(ws, L.dv2);
  if (dx_mn) {
    const DxDirect x = dx_direct(dt, M, d, qw, dqb, qw, w->wq, nullptr, nullptr, 0, 0, d, du_sel,
                                 d, true);
    if (!x.ok) return XMOD_ERR_UNSUPPORTED;
    BW_RUN("bwd_gemm_dx", launch_gemm_tc(c, x.p, x.e));
  } else {
    BW_RUN("bwd_gemm_dx", bw_gemm(c, dt, M, d, qw, dqb, qw, tw.qkv, qw, du_sel, d, true));
  }
  // ======== k, v = u [Wk | Wv]^T on every token
  const DwDirect dwkv = dw_direct(dt, 2 * kw, d, (int)BT, dkv, 2 * kw, u, d, gr->wk, gr->wv,
                                  nullptr, kw, 0, d);
  if (dwkv.ok) {
    BW_RUN("bwd_gemm_dw", launch_gemm_tc(c, dwkv.p, dwkv.e));
  } else {   // [dk | dv]^T [2kw, BTp], u^T [d, BTp]
    BW_RUN("bwd_transpose",
           transpose_multi(c, dt, {{dkv, 2 * kw, tA, BTp, BT, BTp, 2 * kw, 0, 0},
                                   {u, d, tB, BTp, BT, BTp, d, 0, 0}}));
    BW_RUN("bwd_gemm_dw", bw_gemm_dw_split(c, dt, 2 * kw, d, BTp, tA, BTp, tB, BTp, gr->wk,
                                           gr->wv, nullptr, kw, 0, d));
  }
  float* du = (float*)bat(ws, L.du);
  if (dx_mn) {
    const DxDirect x = dx_direct(dt, BT, d, 2 * kw, dkv, 2 * kw, w->wk, w->wv, nullptr, kw, 0, d,
                                 du, d, true);
    if (!x.ok) return XMOD_ERR_UNSUPPORTED;
    BW_RUN("bwd_gemm_dx", launch_gemm_tc(c, x.p, x.e));
  } else {
    BW_RUN("bwd_gemm_dx", bw_gemm(c, dt, BT, d, 2 * kw, dkv, 2 * kw, tw.qkv + (size_t)d * qw,
                                  2 * kw, du, d, true));
  }
  // ======== u = RMSNorm(x) g1 on every token; the selected rows add their query's part
  // and the gradient through h
  float* dadd = (float*)bat(ws, L.h);
  if (cudaMemsetAsync(dadd, 0, sizeof(float) * (size_t)BT * d, c.stream) != cudaSuccess)
    return XMOD_ERR_CUDA;
  BW_RUN("bwd_rows", launch_pdl(fullkv_merge_kernel, dim3((unsigned)((M + BW_WARPS - 1) / BW_WARPS)),
                                dim3(BW_WARPS * 32), 0, c.stream, (int64_t)M, T, n, d, idx,
                                (const float*)du_sel, dh, du, dadd));
  float* rstd1 = (float*)bat(ws, L.rstd1);
  BW_RUN("bwd_rows", launch_pdl(rms_bwd_kernel<E, E>, dim3((unsigned)((BT + BW_WARPS - 1) / BW_WARPS)),
                                dim3(BW_WARPS * 32), 0, c.stream, (int64_t)BT, d, (const float*)du,
                                (const E*)w->rms1, (const E*)x, (const int32_t*)nullptr, T, T,
                                dm->rms_eps, (const E*)nullptr, (float*)nullptr, (E*)nullptr,
                                (const float*)dadd, (E*)dx, rstd1));
  return bw_coldot<E>(c, BT, d, du, (const E*)x, nullptr, T, T, rstd1, part, gr->rms1);
}

template <typename E>
int layer_bwd_t(const Ctx& c, const xmod_dims* dm, int kind, int K, int gate,
                const xmod_layer_weights* w, const void* x, const float* bias, const void* dy,
                float route_coef, void* dx, const xmod_layer_grads* gr, void* ws,
                const BwLayout& L) {
  const xmod_dtype dt = dm->dtype;
  const int B = dm->B, T = dm->T, d = dm->d, hq = dm->n_heads, hkv = dm->n_kv_heads,
            hd = dm->head_dim, F = dm->d_ff;
  // routed: the layer selects top-(T/K) tokens; attn / ffn: which halves of the block run
  // (FullAttn layers: the attention half on every token, y = x + a; Routed-FFN layers:
  // the FFN half on RMSNorm(x_sel) rms2 with a = 0 in the gated residual); fullkv: the
  // Selected-Q / full-KV control, whose selected queries see every token's keys and values
  const bool fullkv = kind == XMOD_LAYER_SPARSE_FULLKV;
  const bool sparse = kind == XMOD_LAYER_SPARSE || kind == XMOD_LAYER_ROUTED_FFN || fullkv;
  const bool attn = kind != XMOD_LAYER_ROUTED_FFN;
  const bool ffn = kind != XMOD_LAYER_ATTN;
  const int n = sparse ? T / K : T;
  const int M = B * n;
  const int Mp = (int)round8(M);
  const int64_t BT = (int64_t)B * T;
  const int qw = hq * hd, kw = hkv * hd, qkv_w = qw + 2 * kw;
  const size_t es = sizeof(E);
  const bool tc = dt == XMOD_BF16;
  if (tc && !tma_available()) return XMOD_ERR_UNSUPPORTED;   // no FFMA route for bf16 GEMMs
  // route_bwd_kernel keeps a float and a flag per token of a sequence in shared memory
  if (sparse && (size_t)T * (sizeof(float) + 1) > 200 * 1024) return XMOD_ERR_UNSUPPORTED;
  float* s = (float*)bat(ws, L.s);
  float* rr = (float*)bat(ws, L.r);
  int32_t* idx = sparse ? (int32_t*)bat(ws, L.idx) : nullptr;
  float* r_sel = (float*)bat(ws, L.r_sel);
  E* u = (E*)bat(ws, L.u);
  E* qkv = (E*)bat(ws, L.qkv);
  E* vt = (E*)bat(ws, L.vt);
  E* o = (E*)bat(ws, L.o);
  E* a = (E*)bat(ws, L.a);
  float* h = (float*)bat(ws, L.h);
  E* v2 = (E*)bat(ws, L.v2);
  E* gu = (E*)bat(ws, L.gu);
  E* H = (E*)bat(ws, L.H);
  E* f = (E*)bat(ws, L.f);
  E* tA = (E*)bat(ws, L.tA);
  E* tB = (E*)bat(ws, L.tB);
  E* tW = (E*)bat(ws, L.tW);
  float* part = (float*)bat(ws, L.part);
  const unsigned rowblk = (unsigned)((M + BW_WARPS - 1) / BW_WARPS);

  // ======== forward recompute
  if (sparse) {
    BW_RUN("router", launch_router(c, dt, BT, d, x, w->w_router, bias, s, rr));
    BW_RUN("topk", launch_topk(c, B, T, n, s, idx, r_sel));
  }
  const bool extras = attn && (w->q_norm || w->k_norm || w->rope_theta > 0.0f);
  E* qkpre = (E*)bat(ws, L.qkpre);
  const bool tc_attn = tc && attention_tc_supported(hd, n, qkv_w);
  bool v_transposed = false;   // v kept only in its transposed layout (tensor-core path)
  // Selected-Q / full-KV buffers: k | v of every token [BT, 2kw] and the selected tokens'
  // q [M, qw] in the qkv buffer, their gradients alike in dqkv; the projections before
  // the QK-norm / rotation (k [BT, kw], then q [M, qw]) in qkpre
  E* kvb = qkv;
  E* qb = qkv + (size_t)BT * 2 * kw;
  E* kpre = qkpre;
  E* qpre = qkpre + (size_t)BT * kw;
  if (fullkv) {
    // RMSNorm1 of every token (keys, values) and of the selected ones (queries; the
    // RMSNorm2 buffer holds them until the o-projection)
    BW_RUN("gather_rmsnorm",
           launch_gather_rmsnorm(c, dt, B, T, T, d, x, nullptr, w->rms1, dm->rms_eps, u));
    BW_RUN("gather_rmsnorm",
           launch_gather_rmsnorm(c, dt, B, T, n, d, x, idx, w->rms1, dm->rms_eps, v2));
    Epilogue ek;
    ek.kind = EPI_STORE;
    ek.out = kvb;
    ek.ldo = 2 * kw;
    GemmTcProblem pk;
    pk.M = (int)BT; pk.N = 2 * kw; pk.K = d; pk.A = u; pk.lda = d; pk.ldb = d;
    pk.B[0] = w->wk; pk.B[1] = w->wv; pk.nB = 2; pk.split[0] = kw;
    const bool tc_kv = tc && attention_tc_supported(hd, n, qw) &&
                       attention_tc_supported(hd, T, 2 * kw);
    if (tc_kv) {   // v transposed for the tensor-core attention, and by rows as well
      ek.vt = vt;
      ek.vt_col0 = kw;
      ek.vt_hd = hd;
      ek.vt_hkv = hkv;
      ek.vt_ld = (int)round8(T);
      ek.n_per_seq = T;
      ek.vt_rows = true;
      v_transposed = gemm_tc_supported(pk, ek);
    }
    if (v_transposed) {
      BW_RUN("gemm_qkv", launch_gemm_tc(c, pk, ek));
    } else {
      BW_RUN("gemm_qkv", bw_gemm(c, dt, (int)BT, kw, d, u, d, w->wk, d, kvb, 2 * kw, false));
      BW_RUN("gemm_qkv", bw_gemm(c, dt, (int)BT, kw, d, u, d, w->wv, d, kvb + kw, 2 * kw, false));
    }
    BW_RUN("gemm_qkv", bw_gemm(c, dt, M, qw, d, v2, d, w->wq, d, qb, qw, false));
    if (extras) {   // keys at every position, queries at the selected ones; projections kept
      if (cudaMemcpy2DAsync(kpre, es * kw, kvb, es * 2 * kw, es * kw, (size_t)BT,
                            cudaMemcpyDeviceToDevice, c.stream) != cudaSuccess ||
          cudaMemcpyAsync(qpre, qb, es * (size_t)M * qw, cudaMemcpyDeviceToDevice, c.stream) !=
              cudaSuccess)
        return XMOD_ERR_CUDA;
      BW_RUN("qk_norm_rope", launch_qk_transform(c, dt, BT, nullptr, kvb, 2 * kw, 0, 0, nullptr,
                                                 0, hkv, w->k_norm, hd, dm->rms_eps,
                                                 w->rope_theta, nullptr, nullptr, T));
      BW_RUN("qk_norm_rope", launch_qk_transform(c, dt, M, nullptr, qb, qw, 0, hq, w->q_norm, 0,
                                                 0, nullptr, hd, dm->rms_eps, w->rope_theta, idx,
                                                 nullptr, T));
    }
    if (v_transposed) {
      AttnKv akv;
      akv.k = kvb;
      akv.ldk = 2 * kw;
      akv.nkv = T;
      akv.qpos = idx;
      BW_RUN("attention", launch_attention_tc(c, B, n, hq, hkv, qb, qw, vt, (int)round8(T), o,
                                              nullptr, nullptr, &akv, (float*)bat(ws, L.lse)));
    } else {
      BW_RUN("attention", launch_attention_simt(c, dt, B, n, hq, hkv, hd, qb, qw, kvb, kvb + kw,
                                                2 * kw, o, idx, T));
    }
  } else if (attn) {
  BW_RUN("gather_rmsnorm",
         launch_gather_rmsnorm(c, dt, B, T, n, d, x, idx, w->rms1, dm->rms_eps, u));
  {
    Epilogue e;
    e.kind = EPI_STORE;
    e.out = qkv;
    e.ldo = qkv_w;
    if (tc_attn) {   // v transposed for the forward attention, and by rows for the backward
      e.vt = vt;
      e.vt_col0 = qw + kw;
      e.vt_hd = hd;
      e.vt_hkv = hkv;
      e.vt_ld = (int)round8(n);
      e.n_per_seq = n;
      e.vt_rows = true;
    }
    GemmTcProblem pq;
    pq.M = M; pq.N = qkv_w; pq.K = d; pq.A = u; pq.lda = d; pq.ldb = d;
    pq.B[0] = w->wq; pq.B[1] = w->wk; pq.B[2] = w->wv; pq.nB = 3;
    pq.split[0] = qw; pq.split[1] = qw + kw;
    v_transposed = tc_attn && gemm_tc_supported(pq, e);
    if (v_transposed) {
      BW_RUN("gemm_qkv", launch_gemm_tc(c, pq, e));
    } else {
      e.vt = nullptr;
      BW_RUN("gemm_qkv", launch_gemm_simt(c, dt, M, qw, d, u, d, w->wq, d, nullptr, e));
      e.out = (char*)qkv + es * qw;
      BW_RUN("gemm_qkv", launch_gemm_simt(c, dt, M, kw, d, u, d, w->wk, d, nullptr, e));
      e.out = (char*)qkv + es * (qw + kw);
      BW_RUN("gemm_qkv", launch_gemm_simt(c, dt, M, kw, d, u, d, w->wv, d, nullptr, e));
    }
    if (extras) {   // QK-norm and rotation at the original positions, projections kept
      if (cudaMemcpy2DAsync(qkpre, es * (qw + kw), qkv, es * qkv_w, es * (qw + kw), M,
                            cudaMemcpyDeviceToDevice, c.stream) != cudaSuccess)
        return XMOD_ERR_CUDA;
      BW_RUN("qk_norm_rope", launch_qk_transform(c, dt, M, nullptr, qkv, qkv_w, 0, hq, w->q_norm,
                                                 qw, hkv, w->k_norm, hd, dm->rms_eps,
                                                 w->rope_theta, idx, nullptr, n));
    }
    if (v_transposed)   // also the rows' log-sum-exp, which the backward reuses
      BW_RUN("attention", launch_attention_tc(c, B, n, hq, hkv, qkv, qkv_w, vt, (int)round8(n), o,
                                              nullptr, nullptr, nullptr,
                                              (float*)bat(ws, L.lse)));
    else
      BW_RUN("attention", launch_attention_simt(c, dt, B, n, hq, hkv, hd, qkv, qkv_w,
                                                (char*)qkv + es * qw, (char*)qkv + es * (qw + kw),
                                                qkv_w, o));
  }
  }
  if (attn && ffn) {
    Epilogue eo;
    eo.kind = EPI_OPROJ;
    eo.out = a;
    eo.ldo = d;
    eo.out2 = h;
    eo.ldo2 = d;
    eo.x = (void*)x;
    eo.idx = idx;
    eo.T = T;
    eo.n_per_seq = n;
    eo.d = d;
    GemmTcProblem po;
    po.M = M; po.N = d; po.K = qw; po.A = o; po.lda = qw; po.ldb = qw; po.B[0] = w->wo;
    if (tc && gemm_tc_supported(po, eo))
      BW_RUN("gemm_o_residual", launch_gemm_tc(c, po, eo));
    else
      BW_RUN("gemm_o_residual", launch_gemm_simt(c, dt, M, d, qw, o, qw, w->wo, qw, nullptr, eo));
  }
  if (ffn) {
  if (attn)
    BW_RUN("rmsnorm2", launch_rmsnorm_f32in(c, dt, M, d, h, w->rms2, dm->rms_eps, v2));
  else   // Routed-FFN: the FFN input is RMSNorm(x_sel) rms2
    BW_RUN("gather_rmsnorm",
           launch_gather_rmsnorm(c, dt, B, T, n, d, x, idx, w->rms2, dm->rms_eps, v2));
  {   // H = silu(G) U with G | U = v2 [W_gate | W_up]^T: one tensor-core GEMM whose
      // SwiGLU epilogue also stores the pre-activations [G | U] for the SwiGLU backward
    Epilogue e;
    e.kind = EPI_SWIGLU;
    e.out = H;
    e.ldo = F;
    e.out2 = gu;
    e.ldo2 = 2 * F;
    GemmTcProblem p;
    p.M = M; p.N = F; p.K = d; p.A = v2; p.lda = d; p.ldb = d;
    p.B[0] = w->w_gate; p.B[1] = w->w_up; p.nB = 2;
    if (tc && gemm_tc_supported(p, e)) {
      BW_RUN("gemm_gate_up", launch_gemm_tc(c, p, e));
    } else {   // [G | U] stored, then H from them
      BW_RUN("gemm_gate_up", bw_gemm(c, dt, M, F, d, v2, d, w->w_gate, d, gu, 2 * F, false));
      BW_RUN("gemm_gate_up", bw_gemm(c, dt, M, F, d, v2, d, w->w_up, d, gu + F, 2 * F, false));
      const int64_t tot = (int64_t)M * F / (16 / sizeof(E));
      const unsigned blk = (unsigned)std::min<int64_t>((tot + 255) / 256, 8192);
      BW_RUN("swiglu", launch_pdl(swiglu_fwd_kernel<E>, dim3(blk), dim3(256), 0, c.stream,
                                  (int64_t)M, F, (const E*)gu, H));
    }
  }
  BW_RUN("gemm_down", bw_gemm(c, dt, M, d, F, H, F, w->w_down, F, f, d, false));
  }

  // ======== backward: residual rule and router
  E* df;
  const E* dae;
  if (sparse) {
    df = (E*)bat(ws, L.df);
    E* dae_buf = (E*)bat(ws, L.dae);
    float* dr = (float*)bat(ws, L.dr);
    float* dvs = (float*)bat(ws, L.dvs);
    float* ds = (float*)bat(ws, L.ds);
    float* lossp = (float*)bat(ws, L.lossp);
    BW_RUN("bwd_rows", launch_pdl(scatter_bwd_kernel<E>, dim3(rowblk), dim3(BW_WARPS * 32), 0,
                                  c.stream, (int64_t)M, T, n, d, (const E*)dy, (const int32_t*)idx,
                                  (const float*)r_sel, attn ? (const E*)a : (const E*)nullptr,
                                  (const E*)f, w->varsigma, gate,
                                  df, dae_buf, dr, dvs));
    dae = gate == XMOD_GATE_XMOD ? df : dae_buf;
    const size_t smr = (size_t)T * (sizeof(float) + 1);
    cudaFuncSetAttribute(route_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smr);
    BW_RUN("bwd_rows", launch_pdl(route_bwd_kernel, dim3(B), dim3(1024), smr, c.stream, T, n,
                                  (const float*)s, (const int32_t*)idx, (const float*)r_sel,
                                  (const float*)dr, route_coef / (float)BT, ds, lossp));
    BW_RUN("bwd_rows", launch_pdl(dx_init_kernel<E>, dim3((unsigned)((BT + BW_WARPS - 1) / BW_WARPS)),
                                  dim3(BW_WARPS * 32), 0, c.stream, BT, d, (const E*)dy,
                                  (const float*)ds, (const E*)w->w_router, (E*)dx));
    int st = bw_coldot<E>(c, BT, d, nullptr, (const E*)x, nullptr, T, T, ds, part, gr->w_router);
    if (st) return st;
    BW_RUN("bwd_reduce", launch_pdl(sum_kernel, dim3(1), dim3(1024), 0, c.stream, (int64_t)M,
                                    (const float*)dvs, 1.0f, gr->varsigma));
    if (gr->route_loss)
      BW_RUN("bwd_reduce", launch_pdl(sum_kernel, dim3(1), dim3(1024), 0, c.stream, (int64_t)B,
                                      (const float*)lossp, 1.0f / (float)BT, gr->route_loss));
  } else {   // dense: y = x + a + f (FullAttn: x + a), every residual receives dy; dx = dy
    df = (E*)dy;
    dae = (const E*)dy;
    if (cudaMemcpyAsync(dx, dy, es * (size_t)BT * d, cudaMemcpyDeviceToDevice, c.stream) !=
        cudaSuccess)
      return XMOD_ERR_CUDA;
    if (cudaMemsetAsync(gr->varsigma, 0, sizeof(float), c.stream) != cudaSuccess)
      return XMOD_ERR_CUDA;
    if (gr->w_router &&
        cudaMemsetAsync(gr->w_router, 0, sizeof(float) * (size_t)d, c.stream) != cudaSuccess)
      return XMOD_ERR_CUDA;
    if (gr->route_loss && cudaMemsetAsync(gr->route_loss, 0, sizeof(float), c.stream) != cudaSuccess)
      return XMOD_ERR_CUDA;
  }

  // gradients of weights a kind does not use are zero
  auto zero = [&](float* g, size_t cnt) {
    return !g || cudaMemsetAsync(g, 0, sizeof(float) * cnt, c.stream) == cudaSuccess;
  };
  if (!ffn && !(zero(gr->rms2, d) && zero(gr->w_gate, (size_t)F * d) &&
                zero(gr->w_up, (size_t)F * d) && zero(gr->w_down, (size_t)d * F)))
    return XMOD_ERR_CUDA;
  if (!attn && !(zero(gr->rms1, d) && zero(gr->wq, (size_t)qw * d) && zero(gr->wk, (size_t)kw * d) &&
                 zero(gr->wv, (size_t)kw * d) && zero(gr->wo, (size_t)d * qw) &&
                 zero(gr->q_norm, hd) && zero(gr->k_norm, hd)))
    return XMOD_ERR_CUDA;
  float* dh = nullptr;   // the gradient reaching h = x_sel + a through the FFN half
  const E* da = dae;     // the gradient reaching a (FullAttn: dy itself)

  // ======== the weights the activation gradients multiply by: read as stored when the
  // tensor-core GEMM takes every such product of this layer (dx_mn), else all transposed
  // in one launch. (The checks use the aligned scratch for the gradients' addresses.)
  const TwParts<E> tw = tw_parts<E>(dm, tW);
  bool dx_mn = dt == XMOD_BF16;
  if (dx_mn && ffn)
    dx_mn = dx_direct(dt, M, F, d, tW, d, w->w_down, nullptr, nullptr, 0, 0, F, tW, F, true).ok &&
            dx_direct(dt, M, d, 2 * F, tW, 2 * F, w->w_gate, w->w_up, nullptr, F, 0, d, tW, d,
                      true).ok;
  if (dx_mn && attn) {
    dx_mn = dx_direct(dt, M, qw, d, tW, d, w->wo, nullptr, nullptr, 0, 0, qw, tW, qw, true).ok;
    if (fullkv)
      dx_mn = dx_mn &&
              dx_direct(dt, M, d, qw, tW, qw, w->wq, nullptr, nullptr, 0, 0, d, tW, d, true).ok &&
              dx_direct(dt, B * T, d, 2 * kw, tW, 2 * kw, w->wk, w->wv, nullptr, kw, 0, d, tW, d,
                        true).ok;
    else
      dx_mn = dx_mn && dx_direct(dt, M, d, qkv_w, tW, qkv_w, w->wq, w->wk, w->wv, qw, qw + kw, d,
                                 tW, d, true).ok;
  }
  if (!dx_mn) {
    TrSpec sp[7];
    int ns = 0;
    if (ffn) {
      sp[ns++] = {w->w_down, F, tw.d, d, d, d, F, 0, 0};          // [F, d]
      sp[ns++] = {w->w_gate, d, tw.gu, 2 * F, F, F, d, 0, 0};     // [d, 2F]
      sp[ns++] = {w->w_up, d, tw.gu + F, 2 * F, F, F, d, 0, 0};
    }
    if (attn) {
      sp[ns++] = {w->wo, qw, tw.o, d, d, d, qw, 0, 0};            // [qw, d]
      if (fullkv) {   // [d, qw] and [d, 2kw]
        sp[ns++] = {w->wq, d, tw.qkv, qw, qw, qw, d, 0, 0};
        sp[ns++] = {w->wk, d, tw.qkv + (size_t)d * qw, 2 * kw, kw, kw, d, 0, 0};
        sp[ns++] = {w->wv, d, tw.qkv + (size_t)d * qw + kw, 2 * kw, kw, kw, d, 0, 0};
      } else {        // [d, qkv_w]
        sp[ns++] = {w->wq, d, tw.qkv, qkv_w, qw, qw, d, 0, 0};
        sp[ns++] = {w->wk, d, tw.qkv + qw, qkv_w, kw, kw, d, 0, 0};
        sp[ns++] = {w->wv, d, tw.qkv + qw + kw, qkv_w, kw, kw, d, 0, 0};
      }
    }
    BW_RUN("bwd_transpose", transpose_multi(c, dt, sp, ns));
  }

  if (ffn) {
  // ======== FFN: f = H Wd^T, H = silu(G) U, [G | U] = v2 [Wg | Wu]^T
  const DwDirect dwd = dw_direct(dt, d, F, M, df, d, H, F, gr->w_down, nullptr, nullptr, 0, 0, F);
  if (dwd.ok) {
    BW_RUN("bwd_gemm_dw", launch_gemm_tc(c, dwd.p, dwd.e));
  } else {   // df^T [d, Mp], H^T [F, Mp]
    BW_RUN("bwd_transpose", transpose_multi(c, dt, {{df, d, tA, Mp, M, Mp, d, 0, 0},
                                                    {H, F, tB, Mp, M, Mp, F, 0, 0}}));
    BW_RUN("bwd_gemm_dw", bw_gemm(c, dt, d, F, Mp, tA, Mp, tB, Mp, gr->w_down, F, true));
  }
  float* dH = (float*)bat(ws, L.dH);
  if (dx_mn) {
    const DxDirect x = dx_direct(dt, M, F, d, df, d, w->w_down, nullptr, nullptr, 0, 0, F, dH, F,
                                 true);
    if (!x.ok) return XMOD_ERR_UNSUPPORTED;
    BW_RUN("bwd_gemm_dx", launch_gemm_tc(c, x.p, x.e));
  } else {
    BW_RUN("bwd_gemm_dx", bw_gemm(c, dt, M, F, d, df, d, tw.d, d, dH, F, true));
  }
  E* dGU = (E*)bat(ws, L.dGU);
  {
    const int64_t tot = (int64_t)M * F / (16 / sizeof(E));
    const unsigned blk = (unsigned)std::min<int64_t>((tot + 255) / 256, 8192);
    BW_RUN("swiglu", launch_pdl(swiglu_bwd_kernel<E>, dim3(blk), dim3(256), 0, c.stream,
                                (int64_t)M, F, (const E*)gu, (const float*)dH, dGU));
  }
  const DwDirect dwgu = dw_direct(dt, 2 * F, d, M, dGU, 2 * F, v2, d, gr->w_gate, gr->w_up,
                                  nullptr, F, 0, d);
  if (dwgu.ok) {
    BW_RUN("bwd_gemm_dw", launch_gemm_tc(c, dwgu.p, dwgu.e));
  } else {   // [dG | dU]^T [2F, Mp], v2^T [d, Mp]
    BW_RUN("bwd_transpose", transpose_multi(c, dt, {{dGU, 2 * F, tA, Mp, M, Mp, 2 * F, 0, 0},
                                                    {v2, d, tB, Mp, M, Mp, d, 0, 0}}));
    BW_RUN("bwd_gemm_dw", bw_gemm_dw_split(c, dt, 2 * F, d, Mp, tA, Mp, tB, Mp, gr->w_gate,
                                           gr->w_up, nullptr, F, 0, d));
  }
  float* dv2 = (float*)bat(ws, L.dv2);
  if (dx_mn) {
    const DxDirect x = dx_direct(dt, M, d, 2 * F, dGU, 2 * F, w->w_gate, w->w_up, nullptr, F, 0,
                                 d, dv2, d, true);
    if (!x.ok) return XMOD_ERR_UNSUPPORTED;
    BW_RUN("bwd_gemm_dx", launch_gemm_tc(c, x.p, x.e));
  } else {
    BW_RUN("bwd_gemm_dx", bw_gemm(c, dt, M, d, 2 * F, dGU, 2 * F, tw.gu, 2 * F, dv2, d, true));
  }
  float* rstd2 = (float*)bat(ws, L.rstd2);
  if (attn) {
    // v2 = RMSNorm(h) g2; h = x_sel + a: dh reaches x_sel and (with dae) a
    dh = (float*)bat(ws, L.dh);
    E* da_buf = (E*)bat(ws, L.da);
    BW_RUN("bwd_rows", launch_pdl(rms_bwd_kernel<float, E>, dim3(rowblk), dim3(BW_WARPS * 32), 0,
                                  c.stream, (int64_t)M, d, (const float*)dv2, (const E*)w->rms2,
                                  (const float*)h, (const int32_t*)nullptr, T, n, dm->rms_eps, dae,
                                  dh, da_buf, (const float*)nullptr, (E*)nullptr, rstd2));
    da = da_buf;
    const int st = bw_coldot<float>(c, M, d, dv2, h, nullptr, T, n, rstd2, part, gr->rms2);
    if (st) return st;
  } else {
    // Routed-FFN: v2 = RMSNorm(x_sel) rms2, the gradient goes straight to the token's row
    BW_RUN("bwd_rows", launch_pdl(rms_bwd_kernel<E, E>, dim3(rowblk), dim3(BW_WARPS * 32), 0,
                                  c.stream, (int64_t)M, d, (const float*)dv2, (const E*)w->rms2,
                                  (const E*)x, (const int32_t*)idx, T, n, dm->rms_eps,
                                  (const E*)nullptr, (float*)nullptr, (E*)nullptr,
                                  (const float*)nullptr, (E*)dx, rstd2));
    return bw_coldot<E>(c, M, d, dv2, (const E*)x, idx, T, n, rstd2, part, gr->rms2);
  }
  }

  // ======== a = o Wo^T
  const DwDirect dwo = dw_direct(dt, d, qw, M, da, d, o, qw, gr->wo, nullptr, nullptr, 0, 0, qw);
  if (dwo.ok) {
    BW_RUN("bwd_gemm_dw", launch_gemm_tc(c, dwo.p, dwo.e));
  } else {   // da^T [d, Mp], o^T [qw, Mp]
    BW_RUN("bwd_transpose", transpose_multi(c, dt, {{da, d, tA, Mp, M, Mp, d, 0, 0},
                                                    {o, qw, tB, Mp, M, Mp, qw, 0, 0}}));
    BW_RUN("bwd_gemm_dw", bw_gemm(c, dt, d, qw, Mp, tA, Mp, tB, Mp, gr->wo, qw, true));
  }
  float* dO = (float*)bat(ws, L.dO);
  const bool mma_attn = tc && attn_bwd_mma_supported(hd, fullkv ? qw : qkv_w, qw);
  if (dx_mn) {
    const DxDirect x = dx_direct(dt, M, qw, d, da, d, w->wo, nullptr, nullptr, 0, 0, qw, dO, qw,
                                 !mma_attn);
    if (!x.ok) return XMOD_ERR_UNSUPPORTED;
    BW_RUN("bwd_gemm_dx", launch_gemm_tc(c, x.p, x.e));
  } else {
    BW_RUN("bwd_gemm_dx", bw_gemm(c, dt, M, qw, d, da, d, tw.o, d, dO, qw, !mma_attn));
  }

  // ======== attention
  E* dqkv = (E*)bat(ws, L.dqkv);
  const bool dq_tc = mma_attn && v_transposed && attn_bwd_dq_tc_supported(hd, qkv_w, qw);
  if (fullkv)
    return fullkv_tail<E>(c, dm, n, w, x, idx, dx, gr, ws, L, kvb, qb, kpre, qpre, vt,
                          v_transposed, o, dO, mma_attn, dh, dx_mn);
  if (dq_tc) {   // tcgen05 (lse from the forward): dq, then dk and dv
    float* lseT = (float*)bat(ws, L.lseT);
    float* DdT = (float*)bat(ws, L.DdT);
    const int ldS = (n + 63) / 64 * 64;
    // the rows' lse per sequence and head, queries contiguous [hq, queries]
    BW_RUN("bwd_transpose", transpose_t<float>(c, n, n, hq, bat(ws, L.lse), hq, lseT, ldS, B,
                                               (int64_t)n * hq, (int64_t)hq * ldS));
    BW_RUN("bwd_attention", launch_attn_bwd_dq_tc(c, B, n, hq, hkv, qkv, qkv_w, o, dO,
                                                  (const float*)bat(ws, L.lse),
                                                  (float*)bat(ws, L.Dd), dqkv, qkv_w, DdT, ldS));
    BW_RUN("bwd_attention", launch_attn_bwd_dkv_tc(c, B, n, hq, hkv, qkv, qkv_w, dO, lseT, DdT,
                                                   ldS, dqkv, qkv_w));
  } else if (mma_attn) {   // bf16: warp-level tensor-core MMA, v rows and dO in bf16
    BW_RUN("bwd_attention", launch_attn_bwd_mma(c, B, n, hq, hkv, hd, qkv, qkv_w, o, dO,
                                                (float*)bat(ws, L.lse), (float*)bat(ws, L.Dd),
                                                dqkv, qkv_w));
  } else {
    AttnBwd p;
    p.n = n;
    p.nk = n;
    p.qpos = nullptr;
    p.hq = hq;
    p.hkv = hkv;
    p.q = qkv;
    p.ldq = qkv_w;
    p.k = qkv + qw;
    p.ldk = qkv_w;
    p.v = v_transposed ? (const void*)vt : (const void*)(qkv + qw + kw);
    p.vt_mode = v_transposed ? 1 : 0;
    p.ldv = qkv_w;
    p.vt_ld = (int)round8(n);
    p.o = o;
    p.dO = dO;
    p.lse = (float*)bat(ws, L.lse);
    p.Dd = (float*)bat(ws, L.Dd);
    p.dq = dqkv;
    p.ldgq = qkv_w;
    p.dk = dqkv + qw;
    p.dv = dqkv + qw + kw;
    p.ldgk = qkv_w;
    p.scale = 1.0f / sqrtf((float)hd);
    BW_RUN("bwd_attention", launch_attn_bwd(c, dt, B, hd, p));
  }

  if (extras) {   // back through the rotation and the QK-norm to the projections
    float* dgq = w->q_norm ? (float*)bat(ws, L.dgq) : nullptr;
    float* dgk = w->k_norm ? (float*)bat(ws, L.dgk) : nullptr;
    BW_RUN("bwd_rows", launch_qk_transform_bwd(c, dt, M, dqkv, qkv_w, 0, hq, w->q_norm, qw, hkv,
                                               w->k_norm, qkpre, qw + kw, hd, dm->rms_eps,
                                               w->rope_theta, idx, n, dgq, dgk));
    if (dgq) {
      const int st = bw_coldot<float>(c, M, hd, nullptr, dgq, nullptr, T, n, nullptr, part,
                                      gr->q_norm);
      if (st) return st;
    }
    if (dgk) {
      const int st = bw_coldot<float>(c, M, hd, nullptr, dgk, nullptr, T, n, nullptr, part,
                                      gr->k_norm);
      if (st) return st;
    }
  }

  // ======== q, k, v = u [Wq | Wk | Wv]^T
  const DwDirect dwqkv = dw_direct(dt, qkv_w, d, M, dqkv, qkv_w, u, d, gr->wq, gr->wk, gr->wv,
                                   qw, qw + kw, d);
  if (dwqkv.ok) {
    BW_RUN("bwd_gemm_dw", launch_gemm_tc(c, dwqkv.p, dwqkv.e));
  } else {   // [dq | dk | dv]^T [qkv_w, Mp], u^T [d, Mp]
    BW_RUN("bwd_transpose",
           transpose_multi(c, dt, {{dqkv, qkv_w, tA, Mp, M, Mp, qkv_w, 0, 0},
                                   {u, d, tB, Mp, M, Mp, d, 0, 0}}));
    BW_RUN("bwd_gemm_dw", bw_gemm_dw_split(c, dt, qkv_w, d, Mp, tA, Mp, tB, Mp, gr->wq, gr->wk,
                                           gr->wv, qw, qw + kw, d));
  }
  float* du = (float*)bat(ws, L.du);
  if (dx_mn) {
    const DxDirect x = dx_direct(dt, M, d, qkv_w, dqkv, qkv_w, w->wq, w->wk, w->wv, qw, qw + kw,
                                 d, du, d, true);
    if (!x.ok) return XMOD_ERR_UNSUPPORTED;
    BW_RUN("bwd_gemm_dx", launch_gemm_tc(c, x.p, x.e));
  } else {
    BW_RUN("bwd_gemm_dx", bw_gemm(c, dt, M, d, qkv_w, dqkv, qkv_w, tw.qkv, qkv_w, du, d, true));
  }
  // u = RMSNorm(x_sel) g1; the gather's backward adds into the token's row of dx
  float* rstd1 = (float*)bat(ws, L.rstd1);
  BW_RUN("bwd_rows", launch_pdl(rms_bwd_kernel<E, E>, dim3(rowblk), dim3(BW_WARPS * 32), 0,
                                c.stream, (int64_t)M, d, (const float*)du, (const E*)w->rms1,
                                (const E*)x, (const int32_t*)idx, T, n, dm->rms_eps,
                                (const E*)nullptr, (float*)nullptr, (E*)nullptr,
                                (const float*)dh, (E*)dx, rstd1));
  return bw_coldot<E>(c, M, d, du, (const E*)x, idx, T, n, rstd1, part, gr->rms1);
}

}  // namespace

size_t bwd_workspace_bytes(const xmod_dims* dm) { return bw_layout(dm).total; }

int run_layer_bwd(cudaStream_t stream, const xmod_dims* dm, int kind, int K, int gate,
                  const xmod_layer_weights* w, const void* x, const float* bias, const void* dy,
                  float route_coef, void* dx, const xmod_layer_grads* gr, void* ws) {
  const BwLayout L = bw_layout(dm);
  Ctx c{stream, (int*)bat(ws, L.status)};
  if (dm->dtype == XMOD_BF16)
    return layer_bwd_t<__nv_bfloat16>(c, dm, kind, K, gate, w, x, bias, dy, route_coef, dx, gr,
                                      ws, L);
  return layer_bwd_t<float>(c, dm, kind, K, gate, w, x, bias, dy, route_coef, dx, gr, ws, L);
}

}  // namespace xmod
