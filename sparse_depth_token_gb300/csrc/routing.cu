// Memory-bound kernels of a sparse layer: router GEMV, per-sequence top-(T/K)
// selection, position-ordered gather (optionally fused with RMSNorm), and the
// gated residual scatter.
//
// Sources: "X-MoD: Practical Scaling Laws for Sparse-Depth Routing Beyond
// Mixture-of-Depths" reading notes -- Eq. 8 (router logit with token bias,
// sigmoid gate), section "MoD structural limit" (top-1/K tokens per sequence),
// Eq. 6 and Eq. 7 (gated residuals); "Mixture-of-Depths explained" -- the
// MoDLayer listing (floor(T * ratio) tokens, position-ordered boolean gather).

#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace xmod {

// ================================================================ router GEMV
//
// One warp per token row, 16-byte streaming loads of x (read exactly once), the
// router vector staged once per CTA in shared memory as fp32.

constexpr int ROUTER_WARPS = 8;

template <typename T>
__global__ void __launch_bounds__(ROUTER_WARPS * 32)
router_kernel(int64_t rows, int d, const T* __restrict__ x, const T* __restrict__ w_r,
              const float* __restrict__ bias, float* __restrict__ s, float* __restrict__ r) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float4 wsh4[];
  float* wsh = reinterpret_cast<float*>(wsh4);
  for (int i = threadIdx.x; i < d; i += blockDim.x) wsh[i] = ld_f(w_r + i);
  __syncthreads();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * ROUTER_WARPS;
  for (int64_t row = (int64_t)blockIdx.x * ROUTER_WARPS + warp; row < rows; row += stride) {
    const T* xr = x + row * d;
    float acc0 = 0.f, acc1 = 0.f;
    int c = lane * V;
    // two independent 16-byte loads in flight per lane per iteration
    for (; c + 32 * V < d; c += 64 * V) {
      Vec16<T> v0 = ld_vec_stream(xr + c);
      Vec16<T> v1 = ld_vec_stream(xr + c + 32 * V);
#pragma unroll
      for (int e = 0; e < V; e += 4) {
        float4 w0 = *reinterpret_cast<const float4*>(wsh + c + e);
        float4 w1 = *reinterpret_cast<const float4*>(wsh + c + 32 * V + e);
        acc0 = fmaf(v0.get(e), w0.x, acc0);
        acc0 = fmaf(v0.get(e + 1), w0.y, acc0);
        acc0 = fmaf(v0.get(e + 2), w0.z, acc0);
        acc0 = fmaf(v0.get(e + 3), w0.w, acc0);
        acc1 = fmaf(v1.get(e), w1.x, acc1);
        acc1 = fmaf(v1.get(e + 1), w1.y, acc1);
        acc1 = fmaf(v1.get(e + 2), w1.z, acc1);
        acc1 = fmaf(v1.get(e + 3), w1.w, acc1);
      }
    }
    for (; c < d; c += 32 * V) {
      Vec16<T> v0 = ld_vec_stream(xr + c);
#pragma unroll
      for (int e = 0; e < V; e += 4) {
        float4 w0 = *reinterpret_cast<const float4*>(wsh + c + e);
        acc0 = fmaf(v0.get(e), w0.x, acc0);
        acc0 = fmaf(v0.get(e + 1), w0.y, acc0);
        acc0 = fmaf(v0.get(e + 2), w0.z, acc0);
        acc0 = fmaf(v0.get(e + 3), w0.w, acc0);
      }
    }
    float acc = warp_sum(acc0 + acc1);
    if (lane == 0) {
      if (bias) acc += bias[row];
      s[row] = acc;
      if (r) r[row] = sigmoidf_acc(acc);
    }
  }
}

static int g_num_sms = 0;
static int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 1;
  }
  return g_num_sms;
}

// Register-cached variant for rows of at most 32 * VPL 16-byte vectors: a warp
// issues every load of its row before reducing, so a whole row is in flight at once.
template <typename T, int VPL>
__global__ void __launch_bounds__(ROUTER_WARPS * 32)
router_rows_kernel(int64_t rows, int d, const T* __restrict__ x, const T* __restrict__ w_r,
                   const float* __restrict__ bias, float* __restrict__ s, float* __restrict__ r) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float4 wsh4[];
  float* wsh = reinterpret_cast<float*>(wsh4);
  for (int i = threadIdx.x; i < d; i += blockDim.x) wsh[i] = ld_f(w_r + i);
  __syncthreads();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * ROUTER_WARPS;
  for (int64_t row = (int64_t)blockIdx.x * ROUTER_WARPS + warp; row < rows; row += stride) {
    const T* xr = x + row * d;
    Vec16<T> v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int c = (i * 32 + lane) * V;
      if (c < d) v[i] = ld_vec_stream(xr + c);
    }
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int c = (i * 32 + lane) * V;
      if (c < d) {
#pragma unroll
        for (int e = 0; e < V; e += 4) {
          const float4 w = wsh4[(c + e) >> 2];
          acc = fmaf(v[i].get(e), w.x, acc);
          acc = fmaf(v[i].get(e + 1), w.y, acc);
          acc = fmaf(v[i].get(e + 2), w.z, acc);
          acc = fmaf(v[i].get(e + 3), w.w, acc);
        }
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) {
      if (bias) acc += bias[row];
      s[row] = acc;
      if (r) r[row] = sigmoidf_acc(acc);
    }
  }
}

// Smallest supported vectors-per-lane count covering `vecs` 16-byte vectors per row
// (0 if the row is too long for the register-cached kernels).
static int pick_vpl(int vecs_per_lane) {
  const int opts[] = {1, 2, 4, 6, 8, 12, 16};
  for (int o : opts)
    if (vecs_per_lane <= o) return o;
  return 0;
}

template <typename T>
static cudaError_t launch_router_rows(const Ctx& c, int vpl, unsigned blocks, size_t smem,
                                      int64_t rows, int d, const T* x, const T* w_r,
                                      const float* bias, float* s, float* r) {
#define XMOD_ROUTER_CASE(N)                                                                  \
  case N: {                                                                                  \
    auto k = router_rows_kernel<T, N>;                                                       \
    if (smem > 48 * 1024)                                                                    \
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);       \
    launch_pdl(k, dim3(blocks), dim3(ROUTER_WARPS * 32), smem, c.stream, rows, d, x, w_r, bias, s, r);           \
    break;                                                                                   \
  }
  switch (vpl) {
    XMOD_ROUTER_CASE(1)
    XMOD_ROUTER_CASE(2)
    XMOD_ROUTER_CASE(4)
    XMOD_ROUTER_CASE(6)
    XMOD_ROUTER_CASE(8)
    XMOD_ROUTER_CASE(12)
    XMOD_ROUTER_CASE(16)
    default:
      return cudaErrorInvalidValue;
  }
#undef XMOD_ROUTER_CASE
  return cudaGetLastError();
}

cudaError_t launch_router(const Ctx& c, xmod_dtype dt, int64_t rows, int d, const void* x,
                          const void* w_r, const float* bias, float* s, float* r) {
  if (rows <= 0) return cudaSuccess;
  int64_t blocks = (rows + ROUTER_WARPS - 1) / ROUTER_WARPS;
  const int64_t cap = (int64_t)num_sms() * 8;  // 8 resident CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  const size_t smem = sizeof(float) * (size_t)d;
  const int vec = dt == XMOD_BF16 ? 8 : 4;
  const int vpl = pick_vpl((d / vec + 31) / 32);
  if (vpl) {
    if (dt == XMOD_BF16)
      return launch_router_rows<__nv_bfloat16>(c, vpl, (unsigned)blocks, smem, rows, d,
                                               (const __nv_bfloat16*)x,
                                               (const __nv_bfloat16*)w_r, bias, s, r);
    return launch_router_rows<float>(c, vpl, (unsigned)blocks, smem, rows, d, (const float*)x,
                                     (const float*)w_r, bias, s, r);
  }
  if (dt == XMOD_BF16) {
    auto k = router_kernel<__nv_bfloat16>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_pdl(k, dim3((unsigned)blocks), dim3(ROUTER_WARPS * 32), smem, c.stream, 
        rows, d, (const __nv_bfloat16*)x, (const __nv_bfloat16*)w_r, bias, s, r);
  } else {
    auto k = router_kernel<float>;
    if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_pdl(k, dim3((unsigned)blocks), dim3(ROUTER_WARPS * 32), smem, c.stream, rows, d, (const float*)x,
                                                               (const float*)w_r, bias, s, r);
  }
  return cudaGetLastError();
}

// ================================================================ top-(T/K)
//
// One CTA per sequence. Logits become order-preserving 32-bit keys in shared
// memory (-0 folded onto +0, so equal values compare equal). A radix select over
// three digits (12, 12 and 8 bits from the top) finds the n-th largest key K* and
// how many of the keys equal to K* are taken; since ties go to the lower position,
// those are the first `remaining` equal keys in position order. Each lane then
// owns a run of consecutive positions: one warp scan and one block scan of the
// per-lane counts of keys above and equal to K* give every selected key its output
// slot, and the selected positions come out in ascending order.
//
// The first digit's histogram is counted while the logits are loaded (16-byte loads
// of every plane); the later digits count only the keys that share the digits found
// so far. A 12-bit first digit (sign, exponent and three mantissa bits) spreads router
// logits over tens of bins, where an 8-bit one puts most of them in two or three and
// the shared-memory atomics on those bins serialise.

constexpr int TOPK_THREADS = 1024;
constexpr int TOPK_MAX_T = 48 * 1024;  // 192 KB of keys in shared memory
constexpr int TOPK_BINS = 4096;        // 12-bit digits

int topk_max_T() { return TOPK_MAX_T; }

__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u & 0x7fffffffu) == 0u) u = 0u;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Largest T whose logits are kept in shared memory beside the keys (for the gates of
// the selected tokens); longer sequences read them again from global memory.
constexpr int TOPK_CACHE_MAX_T = 24 * 1024;

// Adds to hist[d] the number of keys of src[0, len) whose bits under `mask` equal
// `prefix`, d = (key >> shift) & dmask.
__device__ __forceinline__ void radix_count(const uint32_t* src, int len, uint32_t mask,
                                            uint32_t prefix, int shift, uint32_t dmask,
                                            uint32_t* hist) {
  for (int t = threadIdx.x; t < len; t += TOPK_THREADS) {
    const uint32_t k = src[t];
    if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & dmask], 1u);
  }
}

// Scans hist[0, NB) from the largest digit down and finds the digit D at which the
// running count reaches `remaining`; every thread returns D and the count still to
// take among the keys with digit D. Thread i owns digits NB-1-i*P .. NB-P-i*P.
template <int NB>
__device__ __forceinline__ void radix_find(const uint32_t* hist, uint32_t remaining,
                                           uint32_t* warp_sums, uint32_t* result,
                                           uint32_t* digit, uint32_t* rem_out) {
  constexpr int P = NB >= TOPK_THREADS ? NB / TOPK_THREADS : 1;
  constexpr int ACTIVE = NB / P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t c[P], tot = 0;
#pragma unroll
  for (int e = 0; e < P; ++e) {
    c[e] = threadIdx.x < ACTIVE ? hist[NB - 1 - (threadIdx.x * P + e)] : 0u;
    tot += c[e];
  }
  uint32_t inc = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = warp_sums[lane];
    uint32_t wi = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - v;   // exclusive prefix of the warps above
  }
  __syncthreads();
  const uint32_t excl = warp_sums[warp] + inc - tot;
  if (threadIdx.x < ACTIVE && excl < remaining && remaining <= excl + tot) {
    uint32_t run = excl;
#pragma unroll
    for (int e = 0; e < P; ++e) {
      if (run + c[e] >= remaining) {
        result[0] = (uint32_t)(NB - 1 - (threadIdx.x * P + e));
        result[1] = remaining - run;
        break;
      }
      run += c[e];
    }
  }
  __syncthreads();
  *digit = result[0];
  *rem_out = result[1];
}

// The ranked logit of position t from its planes' sum v: minus the block's
// accumulated token-choice bias; its key goes to shared memory and into the first
// digit's histogram.
__device__ __forceinline__ void topk_take(int t, float v, const int32_t* cnt, float bias_step,
                                          uint32_t* keys, float* lsh, uint32_t* hist,
                                          int* bad) {
  const float x = cnt ? v - bias_step * (float)cnt[t] : v;
  if (!isfinite(x)) *bad = 1;
  const uint32_t k = order_key(x);
  keys[t] = k;
  if (lsh) lsh[t] = x;
  atomicAdd(&hist[k >> 20], 1u);
}

// TRACK: the token-choice bias state / statistics of tr are used (else tr is ignored
// and the kernel is the plain top-(T/K)).
template <bool TRACK>
__global__ void __launch_bounds__(TOPK_THREADS)
topk_kernel(int T, int n, const float* __restrict__ s, int32_t* __restrict__ idx,
            float* __restrict__ r_sel, int* status, RouteTrack tr, int nplanes, int64_t plane) {
  if (!TRACK) tr = RouteTrack{};
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t keys[];
  float* lsh = T <= TOPK_CACHE_MAX_T ? reinterpret_cast<float*>(keys + T) : nullptr;
  __shared__ uint32_t hist[TOPK_BINS];
  __shared__ uint32_t scan_sh[2][32];
  __shared__ uint32_t sh_result[2];
  __shared__ int sh_bad;
  __shared__ uint32_t sh_stat[3];   // threshold-selected, agreeing, also selected before
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* sb = s + (int64_t)b * T;
  int32_t* cnt = tr.count ? tr.count + (int64_t)b * T : nullptr;
  int32_t* last = tr.last ? tr.last + (int64_t)b * T : nullptr;
  if (threadIdx.x == 0) sh_bad = 0;
  if (threadIdx.x < 3) sh_stat[threadIdx.x] = 0u;
  for (int i = threadIdx.x; i < TOPK_BINS; i += TOPK_THREADS) hist[i] = 0u;
  __syncthreads();
  // The logit this layer ranks: s (the sum of its planes, in order) minus the block's
  // accumulated token-choice bias. With T a multiple of 4 every plane of the sequence
  // starts on a 16-byte boundary: four positions per load, four loads per plane in
  // flight, every plane's loads issued before any is used.
  if ((T & 3) == 0) {
    const int T4 = T >> 2;
    const float4* s4 = reinterpret_cast<const float4*>(sb);
    const int64_t plane4 = plane >> 2;
    for (int q0 = threadIdx.x; q0 < T4; q0 += 4 * TOPK_THREADS) {
      float4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = q0 + i * TOPK_THREADS;
        v[i] = q < T4 ? s4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int k = 1; k < nplanes; ++k) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = q0 + i * TOPK_THREADS;
          if (q < T4) {
            const float4 u = s4[k * plane4 + q];
            v[i].x += u.x;
            v[i].y += u.y;
            v[i].z += u.z;
            v[i].w += u.w;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = q0 + i * TOPK_THREADS;
        if (q < T4) {
          float4 x = v[i];
          if (cnt) {
            x.x -= tr.bias_step * (float)cnt[4 * q];
            x.y -= tr.bias_step * (float)cnt[4 * q + 1];
            x.z -= tr.bias_step * (float)cnt[4 * q + 2];
            x.w -= tr.bias_step * (float)cnt[4 * q + 3];
          }
          if (!isfinite(x.x) || !isfinite(x.y) || !isfinite(x.z) || !isfinite(x.w)) sh_bad = 1;
          const uint4 k = make_uint4(order_key(x.x), order_key(x.y), order_key(x.z), order_key(x.w));
          reinterpret_cast<uint4*>(keys)[q] = k;
          if (lsh) reinterpret_cast<float4*>(lsh)[q] = x;
          atomicAdd(&hist[k.x >> 20], 1u);
          atomicAdd(&hist[k.y >> 20], 1u);
          atomicAdd(&hist[k.z >> 20], 1u);
          atomicAdd(&hist[k.w >> 20], 1u);
        }
      }
    }
  } else {
    for (int t0 = threadIdx.x; t0 < T; t0 += 4 * TOPK_THREADS) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = t0 + i * TOPK_THREADS;
        v[i] = t < T ? sb[t] : 0.0f;
      }
      for (int k = 1; k < nplanes; ++k) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = t0 + i * TOPK_THREADS;
          if (t < T) v[i] += sb[k * plane + t];
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = t0 + i * TOPK_THREADS;
        if (t < T) topk_take(t, v[i], cnt, tr.bias_step, keys, lsh, hist, &sh_bad);
      }
    }
  }
  __syncthreads();
  if (sh_bad && threadIdx.x == 0) report_status(status, XMOD_ERR_DEVICE_CHECK);

  // Digit 1 (bits 31..20) was counted during the load.
  uint32_t d1, remaining;
  radix_find<TOPK_BINS>(hist, (uint32_t)n, scan_sh[0], sh_result, &d1, &remaining);
  uint32_t prefix = d1 << 20, mask = 0xfff00000u;
  for (int i = threadIdx.x; i < TOPK_BINS; i += TOPK_THREADS) hist[i] = 0u;
  __syncthreads();
  // Digit 2: bits 19..8 among the keys that match digit 1.
  radix_count(keys, T, mask, prefix, 8, 0xfffu, hist);
  __syncthreads();
  uint32_t d2;
  radix_find<TOPK_BINS>(hist, remaining, scan_sh[1], sh_result, &d2, &remaining);
  prefix |= d2 << 8;
  mask |= 0x000fff00u;
  for (int i = threadIdx.x; i < 256; i += TOPK_THREADS) hist[i] = 0u;
  __syncthreads();
  // Digit 3: bits 7..0.
  radix_count(keys, T, mask, prefix, 0, 0xffu, hist);
  __syncthreads();
  uint32_t d3;
  radix_find<256>(hist, remaining, scan_sh[0], sh_result, &d3, &remaining);
  const uint32_t kth = prefix | d3;

  // Lane l of warp w owns positions [lo, hi): PL consecutive positions starting at
  // (32 w + l) PL, recorded as bit masks (bit j = position lo + j) of the keys above,
  // equal to and (for the statistics) at or above 0 in logit. The lanes visit their
  // positions rotated by (l PL) / 32 so that a warp's shared-memory reads fall in
  // distinct banks. A key's output slot is the number of keys above K* before it plus
  // the number of keys equal to K* before it, capped at `remaining` (ties go to the
  // lower position).
  const int PL = (T + TOPK_THREADS - 1) / TOPK_THREADS;   // <= 48: fits a 64-bit mask
  const int lo = (warp * 32 + lane) * PL;
  const int cnt_here = max(0, min(T, lo + PL) - lo);
  const int rot = (lane * PL) >> 5;
  uint64_t gt_m = 0ull, eq_m = 0ull, thr_m = 0ull;
  for (int jj = 0; jj < PL; ++jj) {
    int j = jj + rot;
    if (j >= PL) j -= PL;
    if (j < cnt_here) {
      const uint32_t k = keys[lo + j];
      const uint64_t bit = 1ull << j;
      if (k > kth) gt_m |= bit;
      if (k == kth) eq_m |= bit;
      if (k >= 0x80000000u) thr_m |= bit;   // logit >= 0, i.e. r >= 1/2
    }
  }
  const uint32_t my_gt = (uint32_t)__popcll(gt_m), my_eq = (uint32_t)__popcll(eq_m);
  uint32_t gi = my_gt, ei = my_eq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t yg = __shfl_up_sync(0xffffffffu, gi, o);
    const uint32_t ye = __shfl_up_sync(0xffffffffu, ei, o);
    if (lane >= o) {
      gi += yg;
      ei += ye;
    }
  }
  if (lane == 31) {
    scan_sh[0][warp] = gi;
    scan_sh[1][warp] = ei;
  }
  __syncthreads();
  if (warp < 2) {
    const uint32_t v = scan_sh[warp][lane];
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    scan_sh[warp][lane] = inc - v;
  }
  __syncthreads();
  const uint32_t gt_before = scan_sh[0][warp] + gi - my_gt;
  const uint32_t eq_before = scan_sh[1][warp] + ei - my_eq;
  // the equal keys this lane takes: its first min(my_eq, remaining - eq_before)
  uint64_t sel_m = gt_m;
  {
    const uint32_t take = eq_before < remaining ? min(my_eq, remaining - eq_before) : 0u;
    uint64_t e = eq_m;
    for (uint32_t i = 0; i < take; ++i) {
      sel_m |= e & (~e + 1ull);   // lowest remaining equal key
      e &= e - 1ull;
    }
  }
  uint32_t n_thr = 0, n_agree = 0, n_again = 0;
  if (tr.stats) {
    const uint64_t valid = cnt_here >= 64 ? ~0ull : ((1ull << cnt_here) - 1ull);
    n_thr = (uint32_t)__popcll(thr_m);
    n_agree = (uint32_t)(cnt_here - __popcll((thr_m ^ sel_m) & valid));
  }
  for (uint64_t m = sel_m; m; m &= m - 1ull) {
    const int j = __ffsll((long long)m) - 1;
    const int t = lo + j;
    const uint64_t below = (1ull << j) - 1ull;
    const uint32_t o = gt_before + (uint32_t)__popcll(gt_m & below) +
                       min(eq_before + (uint32_t)__popcll(eq_m & below), remaining);
    if (tr.stats && last && last[t] == tr.layer - 1) ++n_again;
    if (o < (uint32_t)n) {
      idx[(int64_t)b * n + o] = t;
      if (r_sel) {
        float x;
        if (lsh) {
          x = lsh[t];
        } else {
          x = sb[t];
          for (int k2 = 1; k2 < nplanes; ++k2) x += sb[k2 * plane + t];
          if (cnt) x -= tr.bias_step * (float)cnt[t];
        }
        r_sel[(int64_t)b * n + o] = sigmoidf_acc(x);
      }
    }
    // this thread alone owns position t: record the selection for the block's later
    // layers after its last read of cnt[t] and last[t] above
    if (cnt) cnt[t] += 1;
    if (last) last[t] = tr.layer;
  }
  if (tr.stats) {
    n_thr = __reduce_add_sync(0xffffffffu, n_thr);
    n_agree = __reduce_add_sync(0xffffffffu, n_agree);
    n_again = __reduce_add_sync(0xffffffffu, n_again);
    if (lane == 0) {
      atomicAdd(&sh_stat[0], n_thr);
      atomicAdd(&sh_stat[1], n_agree);
      atomicAdd(&sh_stat[2], n_again);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int32_t* st = tr.stats + (int64_t)b * 4;
      st[0] = n;
      st[1] = (int32_t)sh_stat[0];
      st[2] = (int32_t)sh_stat[1];
      st[3] = (int32_t)sh_stat[2];
    }
  }
}

cudaError_t launch_topk(const Ctx& c, int B, int T, int n, const float* s, int32_t* idx,
                        float* r_sel, const RouteTrack* tr, int nplanes, int64_t plane) {
  if (nplanes < 1) return cudaErrorInvalidValue;
  if (B <= 0) return cudaSuccess;
  // keys, and the logits too up to TOPK_CACHE_MAX_T
  const size_t smem = sizeof(uint32_t) * (size_t)T * (T <= TOPK_CACHE_MAX_T ? 2 : 1);
  const int smem_max = (int)(sizeof(uint32_t) * (size_t)TOPK_MAX_T);
  static_assert(2 * TOPK_CACHE_MAX_T <= TOPK_MAX_T, "cached logits fit the key budget");
  cudaFuncSetAttribute(topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
  cudaFuncSetAttribute(topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
  if (tr)
    launch_pdl(topk_kernel<true>, dim3(B), dim3(TOPK_THREADS), smem, c.stream, T, n, s, idx,
               r_sel, c.status, *tr, nplanes, plane);
  else
    launch_pdl(topk_kernel<false>, dim3(B), dim3(TOPK_THREADS), smem, c.stream, T, n, s, idx,
               r_sel, c.status, RouteTrack{}, nplanes, plane);
  return cudaGetLastError();
}

// ================================================================ causal threshold rule
//
// X-MoD notes, "top-k in training, causal threshold at evaluation": token t enters the
// layer when its routing probability is at least 1/2, i.e. its ranked logit
// s - bias_step * count is >= 0 (-0 included), each token on its own. One CTA per
// sequence walks it in 1024-token chunks and writes its picks, in position order, to a
// per-sequence scratch row block; a second kernel gives each sequence its compact row
// offset (the counts of the sequences before it) and copies the picks there, so the
// compact rows come out in (sequence, position) order: tok[m] = b * T + t, r_sel[m] =
// sigmoid of the logit, seq_count[b], seq_off[b] and *M_out = total.

// Sum of one value per thread over the CTA: (exclusive prefix of this thread's warp,
// CTA total), both uniform within a warp.
__device__ __forceinline__ uint2 warps_scan_total(uint32_t v, uint32_t* sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = sh[lane];
    uint32_t inc = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    sh[lane] = inc - t;
    if (lane == 31) sh[32] = inc;
  }
  __syncthreads();
  const uint2 r = make_uint2(sh[warp], sh[32]);
  __syncthreads();
  return r;
}

// Sequence b = blockIdx.x: its picks' positions and gates to pos[b * T + i], gate[b * T
// + i] for i < seq_count[b].
__global__ void __launch_bounds__(TOPK_THREADS)
threshold_count_kernel(int T, const float* __restrict__ s, int32_t* __restrict__ pos,
                       float* __restrict__ gate, int32_t* __restrict__ seq_count, int* status,
                       RouteTrack tr, int nplanes, int64_t plane) {
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t sh[33];
  __shared__ int sh_bad;
  const int lane = threadIdx.x & 31;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) sh_bad = 0;
  __syncthreads();
  const float* sb = s + (int64_t)b * T;
  int32_t* cnt = tr.count ? tr.count + (int64_t)b * T : nullptr;
  int32_t* last = tr.last ? tr.last + (int64_t)b * T : nullptr;
  int32_t* pb = pos + (int64_t)b * T;
  float* gb = gate + (int64_t)b * T;
  uint32_t out = 0, again = 0;   // out: picks so far (the same in every thread)
  for (int t0 = 0; t0 < T; t0 += TOPK_THREADS) {
    const int t = t0 + (int)threadIdx.x;
    float v = 0.0f;
    bool take = false;
    if (t < T) {
      v = sb[t];
      for (int k = 1; k < nplanes; ++k) v += sb[k * plane + t];
      if (cnt) v -= tr.bias_step * (float)cnt[t];
      if (!isfinite(v)) sh_bad = 1;
      take = v >= 0.0f;
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, take);
    const uint2 sc = warps_scan_total((uint32_t)__popc(bal), sh);
    if (take) {
      const uint32_t i = out + sc.x + (uint32_t)__popc(bal & lt_mask);
      pb[i] = t;
      gb[i] = sigmoidf_acc(v);
      if (last && last[t] == tr.layer - 1) ++again;
      if (cnt) cnt[t] += 1;
      if (last) last[t] = tr.layer;
    }
    out += sc.y;
  }
  if (tr.stats) {   // reduce `again` over the CTA (only the stats use it)
    const uint2 sc = warps_scan_total((uint32_t)__reduce_add_sync(0xffffffffu, again), sh);
    if (threadIdx.x == 0) {
      int32_t* st = tr.stats + (int64_t)b * 4;
      st[0] = (int32_t)out;
      st[1] = (int32_t)out;   // the rule's own picks are its threshold picks
      st[2] = T;
      st[3] = (int32_t)sc.y;
    }
  }
  if (threadIdx.x == 0) {
    seq_count[b] = (int32_t)out;
    if (sh_bad) report_status(status, XMOD_ERR_DEVICE_CHECK);
  }
}

// Sequence b = blockIdx.x: offset = the counts of sequences 0 .. b-1 (added in order),
// its picks copied to the compact rows from there.
__global__ void __launch_bounds__(256)
threshold_compact_kernel(int B, int T, const int32_t* __restrict__ pos,
                         const float* __restrict__ gate, const int32_t* __restrict__ seq_count,
                         int32_t* __restrict__ tok, float* __restrict__ r_sel,
                         int32_t* __restrict__ seq_off, int32_t* __restrict__ M_out) {
  pdl_trigger();
  pdl_wait();
  __shared__ int32_t sh_off;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    int32_t off = 0;
    for (int i = 0; i < b; ++i) off += seq_count[i];
    sh_off = off;
    seq_off[b] = off;
    if (b == B - 1) *M_out = off + seq_count[b];
  }
  __syncthreads();
  const int32_t off = sh_off, n = seq_count[b];
  const int32_t* pb = pos + (int64_t)b * T;
  const float* gb = gate + (int64_t)b * T;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    tok[off + i] = b * T + pb[i];
    r_sel[off + i] = gb[i];
  }
}

cudaError_t launch_threshold_select(const Ctx& c, int B, int T, const float* s, int32_t* tok,
                                    float* r_sel, int32_t* seq_count, int32_t* seq_off,
                                    int32_t* M_out, const RouteTrack* tr, int nplanes,
                                    int64_t plane, int32_t* scratch_pos, float* scratch_gate) {
  if (B <= 0 || T <= 0 || nplanes < 1 || !scratch_pos || !scratch_gate)
    return cudaErrorInvalidValue;
  const RouteTrack none{};
  cudaError_t e = launch_pdl(threshold_count_kernel, dim3(B), dim3(TOPK_THREADS), 0, c.stream,
                             T, s, scratch_pos, scratch_gate, seq_count, c.status,
                             tr ? *tr : none, nplanes, plane);
  if (e != cudaSuccess) return e;
  count_launch();
  return launch_pdl(threshold_compact_kernel, dim3(B), dim3(256), 0, c.stream, B, T,
                    (const int32_t*)scratch_pos, (const float*)scratch_gate,
                    (const int32_t*)seq_count, tok, r_sel, seq_off, M_out);
}

// update_hist[b, c] = number of tokens of sequence b whose count is c (0 <= c <= max_count).
__global__ void count_hist_kernel(int T, int max_count, const int32_t* __restrict__ count,
                                  int32_t* __restrict__ update_hist) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint32_t h[];
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i <= max_count; i += blockDim.x) h[i] = 0u;
  __syncthreads();
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const int c = count[(int64_t)b * T + t];
    atomicAdd(&h[c < 0 ? 0 : (c > max_count ? max_count : c)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= max_count; i += blockDim.x)
    update_hist[(int64_t)b * (max_count + 1) + i] = (int32_t)h[i];
}

cudaError_t launch_count_hist(const Ctx& c, int B, int T, int max_count, const int32_t* count,
                              int32_t* update_hist) {
  if (B <= 0) return cudaSuccess;
  return launch_pdl(count_hist_kernel, dim3(B), dim3(512), sizeof(uint32_t) * (size_t)(max_count + 1),
                    c.stream, T, max_count, count, update_hist);
}

// ================================================================ gather (+ RMSNorm)

constexpr int ROW_WARPS = 8;

__device__ __forceinline__ int64_t stream_row(int64_t m, int T, int n, const int32_t* idx) {
  const int64_t b = m / n;
  const int64_t t = idx ? (int64_t)idx[m] : (m - b * n);
  return b * T + t;
}

// Positions from the caller (or top-k): row m, the (m % n)-th row of its sequence, must
// name a position in [0, seqT) above the one of the row before it in the sequence. A row
// that does not is skipped -- nothing is read or written for it -- and the status word
// records XMOD_ERR_DEVICE_CHECK.
__device__ __forceinline__ bool row_idx_ok(int64_t m, int seqT, int n, const int32_t* idx,
                                           int* status) {
  if (!idx) return true;
  const int32_t t = idx[m];
  const bool ok = t >= 0 && t < seqT && (m % n == 0 || t > idx[m - 1]);
  if (!ok) report_status(status, XMOD_ERR_DEVICE_CHECK);
  return ok;
}

template <typename T>
__global__ void __launch_bounds__(ROW_WARPS * 32)
gather_kernel(int64_t M, int seqT, int n, int d, const T* __restrict__ x,
              const int32_t* __restrict__ idx, T* __restrict__ xs, int* status) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= M || !row_idx_ok(m, seqT, n, idx, status)) return;
  const T* src = x + stream_row(m, seqT, n, idx) * d;
  T* dst = xs + m * d;
  for (int c = lane * V; c < d; c += 32 * V) st_vec(dst + c, ld_vec(src + c));
}

template <typename T>
__global__ void __launch_bounds__(ROW_WARPS * 32)
gather_rmsnorm_kernel(int64_t M, int seqT, int n, int d, const T* __restrict__ x,
                      const int32_t* __restrict__ idx, const T* __restrict__ gamma, float eps,
                      T* __restrict__ u, int* status) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= M || !row_idx_ok(m, seqT, n, idx, status)) return;
  const T* src = x + stream_row(m, seqT, n, idx) * d;
  float ss = 0.f;
  for (int c = lane * V; c < d; c += 32 * V) {
    Vec16<T> v = ld_vec(src + c);
#pragma unroll
    for (int e = 0; e < V; ++e) ss = fmaf(v.get(e), v.get(e), ss);
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)d + eps);
  T* dst = u + m * d;
  for (int c = lane * V; c < d; c += 32 * V) {
    Vec16<T> v = ld_vec(src + c);
    Vec16<T> g = ld_vec(gamma + c);
    Vec16<T> o;
#pragma unroll
    for (int e = 0; e < V; ++e) o.set(e, v.get(e) * inv * g.get(e));
    st_vec(dst + c, o);
  }
}

// Register-cached variant (rows of at most 32 * VPL 16-byte vectors): the row is
// read once with every load in flight, then normalised from registers. Rows of up to
// eight vectors a lane (2048 bf16, 1024 fp32) run four CTAs per SM (at most 64
// registers a thread): a sparse layer's 4096 rows are then all in flight in one wave
// on 152 SMs (three per SM, at 74 registers, left a second partial wave; A3K16 shape
// 14.6 -> 12.9 us). Longer rows would spill under that bound.
template <typename T, int VPL>
__global__ void __launch_bounds__(ROW_WARPS * 32, VPL <= 8 ? 4 : 1)
gather_rmsnorm_rows_kernel(int64_t M, int seqT, int n, int d, const T* __restrict__ x,
                           const int32_t* __restrict__ idx, const T* __restrict__ gamma,
                           float eps, T* __restrict__ u, RowMap rm, int* status) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= rm.rows(M)) return;
  if (!rm.tok && !row_idx_ok(m, seqT, n, idx, status)) return;
  const T* src = x + (rm.tok ? (int64_t)rm.tok[m] : stream_row(m, seqT, n, idx)) * d;
  Vec16<T> v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = (i * 32 + lane) * V;
    if (c < d) v[i] = ld_vec(src + c);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = (i * 32 + lane) * V;
    if (c < d) {
#pragma unroll
      for (int e = 0; e < V; ++e) ss = fmaf(v[i].get(e), v[i].get(e), ss);
    }
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)d + eps);
  T* dst = u + m * d;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = (i * 32 + lane) * V;
    if (c < d) {
      const Vec16<T> g = ld_vec(gamma + c);
      Vec16<T> o;
#pragma unroll
      for (int e = 0; e < V; ++e) o.set(e, v[i].get(e) * inv * g.get(e));
      st_vec(dst + c, o);
    }
  }
}

template <typename T>
static cudaError_t launch_gather_rmsnorm_rows(const Ctx& c, int vpl, unsigned blocks, int64_t M,
                                              int seqT, int n, int d, const T* x,
                                              const int32_t* idx, const T* gamma, float eps,
                                              T* u, RowMap rm) {
#define XMOD_GR_CASE(N)                                                                     \
  case N:                                                                                   \
    launch_pdl(gather_rmsnorm_rows_kernel<T, N>, dim3(blocks), dim3(ROW_WARPS * 32), 0,     \
               c.stream, M, seqT, n, d, x, idx, gamma, eps, u, rm, c.status);               \
    break;
  switch (vpl) {
    XMOD_GR_CASE(1)
    XMOD_GR_CASE(2)
    XMOD_GR_CASE(4)
    XMOD_GR_CASE(6)
    XMOD_GR_CASE(8)
    XMOD_GR_CASE(12)
    XMOD_GR_CASE(16)
    default:
      return cudaErrorInvalidValue;
  }
#undef XMOD_GR_CASE
  return cudaGetLastError();
}

// ================================================================ router vectors as rows

// dst[j, :] = rows.p[j][:] for j < count; rows [count, total) are zeroed. bf16 rows
// of d elements, d % 8 == 0, one 16-byte vector per thread.
__global__ void stack_rows_kernel(RowPtrs rows, int count, int total, int d, uint4* dst) {
  pdl_trigger();
  pdl_wait();
  const int vecs = d / 8;
  const int64_t n = (int64_t)total * vecs;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i / vecs), v = (int)(i - (int64_t)j * vecs);
    dst[i] = j < count ? reinterpret_cast<const uint4*>(rows.p[j])[v] : make_uint4(0, 0, 0, 0);
  }
}

cudaError_t launch_stack_rows(const Ctx& c, const RowPtrs& rows, int count, int total, int d,
                              void* dst) {
  if (count < 0 || count > RowPtrs::kMax || total < count || d % 8) return cudaErrorInvalidValue;
  const int64_t n = (int64_t)total * (d / 8);
  if (n <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 1024);
  return launch_pdl(stack_rows_kernel, dim3(blocks), dim3(256), 0, c.stream, rows, count, total,
                    d, (uint4*)dst);
}

// Register-cached gather (rows of at most 32 * VPL 16-byte vectors): every load of a
// row is issued before its first store, so a whole row is in flight per warp.
template <typename T, int VPL>
__global__ void __launch_bounds__(ROW_WARPS * 32)
gather_rows_kernel(int64_t M, int seqT, int n, int d, const T* __restrict__ x,
                   const int32_t* __restrict__ idx, T* __restrict__ xs, int* status) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= M || !row_idx_ok(m, seqT, n, idx, status)) return;
  const T* src = x + stream_row(m, seqT, n, idx) * d;
  T* dst = xs + m * d;
  Vec16<T> v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = (i * 32 + lane) * V;
    if (c < d) v[i] = ld_vec(src + c);
  }
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = (i * 32 + lane) * V;
    if (c < d) st_vec(dst + c, v[i]);
  }
}

cudaError_t launch_gather(const Ctx& c, xmod_dtype dt, int B, int T, int n, int d,
                          const void* x, const int32_t* idx, void* xs) {
  const int64_t M = (int64_t)B * n;
  if (M <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((M + ROW_WARPS - 1) / ROW_WARPS);
  const int vpl = pick_vpl((d / (dt == XMOD_BF16 ? 8 : 4) + 31) / 32);
  if (vpl) {
#define XMOD_GA_CASE(TT, N)                                                                  \
  case N:                                                                                    \
    return launch_pdl(gather_rows_kernel<TT, N>, dim3(blocks), dim3(ROW_WARPS * 32), 0,      \
                      c.stream, M, T, n, d, (const TT*)x, idx, (TT*)xs, c.status);
    if (dt == XMOD_BF16) {
      switch (vpl) {
        XMOD_GA_CASE(__nv_bfloat16, 1) XMOD_GA_CASE(__nv_bfloat16, 2)
        XMOD_GA_CASE(__nv_bfloat16, 4) XMOD_GA_CASE(__nv_bfloat16, 6)
        XMOD_GA_CASE(__nv_bfloat16, 8) XMOD_GA_CASE(__nv_bfloat16, 12)
        XMOD_GA_CASE(__nv_bfloat16, 16)
      }
    } else {
      switch (vpl) {
        XMOD_GA_CASE(float, 1) XMOD_GA_CASE(float, 2) XMOD_GA_CASE(float, 4)
        XMOD_GA_CASE(float, 6) XMOD_GA_CASE(float, 8) XMOD_GA_CASE(float, 12)
        XMOD_GA_CASE(float, 16)
      }
    }
#undef XMOD_GA_CASE
    return cudaErrorInvalidValue;
  }
  if (dt == XMOD_BF16)
    launch_pdl(gather_kernel<__nv_bfloat16>, dim3(blocks), dim3(ROW_WARPS * 32), 0, c.stream,
               M, T, n, d, (const __nv_bfloat16*)x, idx, (__nv_bfloat16*)xs, c.status);
  else
    launch_pdl(gather_kernel<float>, dim3(blocks), dim3(ROW_WARPS * 32), 0, c.stream, M, T, n,
               d, (const float*)x, idx, (float*)xs, c.status);
  return cudaGetLastError();
}

cudaError_t launch_gather_rmsnorm(const Ctx& c, xmod_dtype dt, int B, int T, int n, int d,
                                  const void* x, const int32_t* idx, const void* gamma,
                                  float eps, void* u, RowMap rm) {
  const int64_t M = (int64_t)B * n;
  if (M <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((M + ROW_WARPS - 1) / ROW_WARPS);
  const int vpl = pick_vpl((d / (dt == XMOD_BF16 ? 8 : 4) + 31) / 32);
  if (vpl) {
    if (dt == XMOD_BF16)
      return launch_gather_rmsnorm_rows<__nv_bfloat16>(
          c, vpl, blocks, M, T, n, d, (const __nv_bfloat16*)x, idx, (const __nv_bfloat16*)gamma,
          eps, (__nv_bfloat16*)u, rm);
    return launch_gather_rmsnorm_rows<float>(c, vpl, blocks, M, T, n, d, (const float*)x, idx,
                                             (const float*)gamma, eps, (float*)u, rm);
  }
  if (rm.tok || rm.M_dev) return cudaErrorInvalidValue;   // rows beyond the cached widths
  if (dt == XMOD_BF16)
    launch_pdl(gather_rmsnorm_kernel<__nv_bfloat16>, dim3(blocks), dim3(ROW_WARPS * 32), 0,
               c.stream, M, T, n, d, (const __nv_bfloat16*)x, idx, (const __nv_bfloat16*)gamma,
               eps, (__nv_bfloat16*)u, c.status);
  else
    launch_pdl(gather_rmsnorm_kernel<float>, dim3(blocks), dim3(ROW_WARPS * 32), 0, c.stream,
               M, T, n, d, (const float*)x, idx, (const float*)gamma, eps, (float*)u, c.status);
  return cudaGetLastError();
}

template <typename T>
__global__ void __launch_bounds__(ROW_WARPS * 32)
rmsnorm_f32in_kernel(int64_t M, int d, const float* __restrict__ h, const T* __restrict__ gamma,
                     float eps, T* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= M) return;
  const float* src = h + m * d;
  float ss = 0.f;
  for (int c = lane * 4; c < d; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(src + c);
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)d + eps);
  T* dst = out + m * d;
  for (int c = lane * V; c < d; c += 32 * V) {
    Vec16<T> g = ld_vec(gamma + c);
    Vec16<T> o;
#pragma unroll
    for (int e = 0; e < V; ++e) o.set(e, src[c + e] * inv * g.get(e));
    st_vec(dst + c, o);
  }
}

// Register-cached variant: units of V = 16 / sizeof(T) elements (one 16-byte output
// vector, V/4 float4 inputs), at most VPL units per lane.
template <typename T, int VPL>
__global__ void __launch_bounds__(ROW_WARPS * 32)
rmsnorm_f32in_rows_kernel(int64_t M, int d, const float* __restrict__ h,
                          const T* __restrict__ gamma, float eps, T* __restrict__ out,
                          const int32_t* __restrict__ M_dev) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= M || (M_dev && m >= *M_dev)) return;
  const float* src = h + m * d;
  float4 v[VPL][V / 4];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = (i * 32 + lane) * V;
    if (c < d) {
#pragma unroll
      for (int q = 0; q < V / 4; ++q) v[i][q] = *reinterpret_cast<const float4*>(src + c + 4 * q);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = (i * 32 + lane) * V;
    if (c < d) {
#pragma unroll
      for (int q = 0; q < V / 4; ++q)
        ss = fmaf(v[i][q].x, v[i][q].x,
                  fmaf(v[i][q].y, v[i][q].y, fmaf(v[i][q].z, v[i][q].z, fmaf(v[i][q].w, v[i][q].w, ss))));
    }
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / (float)d + eps);
  T* dst = out + m * d;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int c = (i * 32 + lane) * V;
    if (c < d) {
      const Vec16<T> g = ld_vec(gamma + c);
      Vec16<T> o;
#pragma unroll
      for (int q = 0; q < V / 4; ++q) {
        o.set(4 * q + 0, v[i][q].x * inv * g.get(4 * q + 0));
        o.set(4 * q + 1, v[i][q].y * inv * g.get(4 * q + 1));
        o.set(4 * q + 2, v[i][q].z * inv * g.get(4 * q + 2));
        o.set(4 * q + 3, v[i][q].w * inv * g.get(4 * q + 3));
      }
      st_vec(dst + c, o);
    }
  }
}

template <typename T>
static cudaError_t launch_rmsnorm_f32in_rows(const Ctx& c, int vpl, unsigned blocks, int64_t M,
                                             int d, const float* h, const T* gamma, float eps,
                                             T* out, const int32_t* M_dev) {
#define XMOD_RN_CASE(N)                                                                    \
  case N:                                                                                  \
    launch_pdl(rmsnorm_f32in_rows_kernel<T, N>, dim3(blocks), dim3(ROW_WARPS * 32), 0, c.stream, M, d, h, gamma, \
                                                                            eps, out, M_dev); \
    break;
  switch (vpl) {
    XMOD_RN_CASE(1)
    XMOD_RN_CASE(2)
    XMOD_RN_CASE(4)
    XMOD_RN_CASE(6)
    XMOD_RN_CASE(8)
    XMOD_RN_CASE(12)
    XMOD_RN_CASE(16)
    default:
      return cudaErrorInvalidValue;
  }
#undef XMOD_RN_CASE
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_f32in(const Ctx& c, xmod_dtype dt, int64_t M, int d, const float* h,
                                 const void* gamma, float eps, void* out, const int32_t* M_dev) {
  if (M <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((M + ROW_WARPS - 1) / ROW_WARPS);
  const int vpl = pick_vpl((d / (dt == XMOD_BF16 ? 8 : 4) + 31) / 32);
  if (vpl) {
    if (dt == XMOD_BF16)
      return launch_rmsnorm_f32in_rows<__nv_bfloat16>(c, vpl, blocks, M, d, h,
                                                      (const __nv_bfloat16*)gamma, eps,
                                                      (__nv_bfloat16*)out, M_dev);
    return launch_rmsnorm_f32in_rows<float>(c, vpl, blocks, M, d, h, (const float*)gamma, eps,
                                            (float*)out, M_dev);
  }
  if (M_dev) return cudaErrorInvalidValue;   // rows beyond the cached widths
  if (dt == XMOD_BF16)
    launch_pdl(rmsnorm_f32in_kernel<__nv_bfloat16>, dim3(blocks), dim3(ROW_WARPS * 32), 0, c.stream, 
        M, d, h, (const __nv_bfloat16*)gamma, eps, (__nv_bfloat16*)out);
  else
    launch_pdl(rmsnorm_f32in_kernel<float>, dim3(blocks), dim3(ROW_WARPS * 32), 0, c.stream, M, d, h, (const float*)gamma,
                                                                 eps, (float*)out);
  return cudaGetLastError();
}

// ================================================================ QK-norm and rotary embedding

// One warp per row of x [rows, ld] (bf16 or fp32), QK_HEADS heads loaded at a time:
// the q heads (columns from q_col0, gains q_gain) come before the k heads (k_col0,
// k_gain), each head of hd (a multiple of 32) elements. Each lane holds E = hd / 32 consecutive elements, so the rotation
// partner c + hd/2 of a lane's element c sits in lane ^ 16 at the same slot.
// Position of row m: pos_idx ? pos_idx[m] : pos_tok ? pos_tok[m] % seqT : m % seqT.
// The angle pos * theta^(-2c/hd) is taken modulo one turn without losing the position's
// bits: per pair c the turns per position, theta^(-2c/hd) / (2 pi), are kept as a
// float hi + lo sum, and pos * hi is split exactly with an fma.
constexpr int QK_HEADS = 4;   // 8 in flight measured slower (A4K8 sparse layer: 28.6 against 21.7 us)

// E consecutive elements of one lane: one 8- or 16-byte access when they fill one
// (the rows, head offsets and lane offsets are multiples of E elements).
template <typename T, int E>
__device__ __forceinline__ void ld_lane(const T* p, float (&v)[E]) {
  if constexpr (sizeof(T) == 2 && E == 4) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  } else if constexpr (sizeof(T) == 4 && E == 4) {
    const float4 r = *reinterpret_cast<const float4*>(p);
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = Elem<T>::to_f(p[e]);
  }
}
template <typename T, int E>
__device__ __forceinline__ void st_lane(T* p, const float (&v)[E]) {
  if constexpr (sizeof(T) == 2 && E == 4) {
    __nv_bfloat162 r[2] = {__floats2bfloat162_rn(v[0], v[1]), __floats2bfloat162_rn(v[2], v[3])};
    *reinterpret_cast<uint2*>(p) = *reinterpret_cast<const uint2*>(r);
  } else if constexpr (sizeof(T) == 4 && E == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) p[e] = Elem<T>::from_f(v[e]);
  }
}

template <typename T, int E>
__global__ void __launch_bounds__(ROW_WARPS * 32)
qk_transform_kernel(int64_t M, const int32_t* __restrict__ M_dev, T* __restrict__ x, int ld,
                    int q_col0, int q_heads, const T* __restrict__ q_gain, int k_col0,
                    int k_heads, const T* __restrict__ k_gain, float eps, double theta,
                    const int32_t* __restrict__ pos_idx, const int32_t* __restrict__ pos_tok,
                    int seqT) {
  pdl_trigger();
  constexpr int HD = 32 * E;
  __shared__ float2 turns[HD / 2];
  for (int c = threadIdx.x; c < HD / 2; c += blockDim.x) {
    const double r = theta > 0.0 ? exp2(-(2.0 * c / HD) * log2(theta)) / 6.283185307179586 : 0.0;
    const float hi = (float)r;
    turns[c] = make_float2(hi, (float)(r - (double)hi));
  }
  __syncthreads();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= M || (M_dev && m >= *M_dev)) return;
  const int64_t pos = pos_idx ? pos_idx[m] : pos_tok ? pos_tok[m] % seqT : m % seqT;
  const float pf = (float)pos;   // exact: positions stay below 2^24
  const bool first = lane < 16;
  // the angles depend on the position and the pair only: once per row for every head
  float cs[E], sn[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    cs[e] = 1.0f;
    sn[e] = 0.0f;
    if (theta > 0.0) {
      const float2 t = turns[(first ? lane : lane - 16) * E + e];
      const float a = pf * t.x;
      const float frac = (a - rintf(a)) + fmaf(pf, t.y, fmaf(pf, t.x, -a));
      __sincosf(frac * 6.2831853f, &sn[e], &cs[e]);   // |angle| <= pi: the fast form suffices
    }
  }
  const int heads = q_heads + k_heads;
  for (int h0 = 0; h0 < heads; h0 += QK_HEADS) {
    const int h_end = min(heads, h0 + QK_HEADS);
    T* hp[QK_HEADS];   // QK_HEADS heads loaded together
    float v[QK_HEADS][E];
#pragma unroll
    for (int i = 0; i < QK_HEADS; ++i) {
      const int h = h0 + i;
      hp[i] = nullptr;
      if (h < h_end) {
        const bool is_q = h < q_heads;
        hp[i] = x + m * ld + (is_q ? q_col0 + h * HD : k_col0 + (h - q_heads) * HD) + lane * E;
        ld_lane<T, E>(hp[i], v[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < QK_HEADS; ++i) {
      const int h = h0 + i;
      if (h >= h_end) break;
      const bool is_q = h < q_heads;
      const T* gain = is_q ? q_gain : k_gain;
      if (gain) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(v[i][e], v[i][e], ss);
        const float inv = rsqrtf(warp_sum(ss) / (float)HD + eps);
#pragma unroll
        for (int e = 0; e < E; ++e) v[i][e] = v[i][e] * inv * Elem<T>::to_f(gain[lane * E + e]);
      }
      if (theta > 0.0) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float other = __shfl_xor_sync(0xffffffffu, v[i][e], 16);
          v[i][e] = first ? v[i][e] * cs[e] - other * sn[e] : other * sn[e] + v[i][e] * cs[e];
        }
      }
      st_lane<T, E>(hp[i], v[i]);
    }
  }
}

// Backward of qk_transform_kernel (no variable row count): g [M, ld] holds the gradient
// at the transformed q heads (from q_col0) and k heads (from k_col0); pre [M, ldp] the
// projections before the transform, the q heads from column 0 and the k heads right
// after them. g becomes, in place, the gradient at the projections: the rotation is
// orthogonal, so its gradient rotates back by the same angle; through the QK-norm,
// rho (dn gain - vhat mean(dn gain vhat)). dgq / dgk [M, HD] (NULL: that gain is absent)
// receive per row the gain gradient dn * vhat summed over the row's q (k) heads.
template <typename T, int E>
__global__ void __launch_bounds__(ROW_WARPS * 32)
qk_transform_bwd_kernel(int64_t M, T* __restrict__ g, int ld, int q_col0, int q_heads,
                        const T* __restrict__ q_gain, int k_col0, int k_heads,
                        const T* __restrict__ k_gain, const T* __restrict__ pre, int ldp,
                        float eps, double theta, const int32_t* __restrict__ pos_idx, int seqT,
                        float* __restrict__ dgq, float* __restrict__ dgk) {
  pdl_trigger();
  constexpr int HD = 32 * E;
  __shared__ float2 turns[HD / 2];
  for (int c = threadIdx.x; c < HD / 2; c += blockDim.x) {
    const double r = theta > 0.0 ? exp2(-(2.0 * c / HD) * log2(theta)) / 6.283185307179586 : 0.0;
    const float hi = (float)r;
    turns[c] = make_float2(hi, (float)(r - (double)hi));
  }
  __syncthreads();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= M) return;
  const int64_t pos = pos_idx ? pos_idx[m] : m % seqT;
  const float pf = (float)pos;
  const bool first = lane < 16;
  float cs[E], sn[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {   // the forward's angles, computed the same way
    cs[e] = 1.0f;
    sn[e] = 0.0f;
    if (theta > 0.0) {
      const float2 t = turns[(first ? lane : lane - 16) * E + e];
      const float a = pf * t.x;
      const float frac = (a - rintf(a)) + fmaf(pf, t.y, fmaf(pf, t.x, -a));
      __sincosf(frac * 6.2831853f, &sn[e], &cs[e]);
    }
  }
  float accq[E], acck[E];
#pragma unroll
  for (int e = 0; e < E; ++e) accq[e] = acck[e] = 0.0f;
  const int heads = q_heads + k_heads;
  for (int h = 0; h < heads; ++h) {
    const bool is_q = h < q_heads;
    T* gp = g + m * ld + (is_q ? q_col0 + h * HD : k_col0 + (h - q_heads) * HD) + lane * E;
    const T* vp = pre + m * ldp + h * HD + lane * E;
    const T* gain = is_q ? q_gain : k_gain;
    float gv[E], v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      gv[e] = Elem<T>::to_f(gp[e]);
      v[e] = Elem<T>::to_f(vp[e]);
    }
    if (theta > 0.0) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, gv[e], 16);
        gv[e] = first ? gv[e] * cs[e] + other * sn[e] : gv[e] * cs[e] - other * sn[e];
      }
    }
    if (gain) {
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
      const float rho = rsqrtf(warp_sum(ss) / (float)HD + eps);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot += gv[e] * Elem<T>::to_f(gain[lane * E + e]) * v[e] * rho;
      const float mean = warp_sum(dot) / (float)HD;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float vh = v[e] * rho;
        if (is_q) accq[e] += gv[e] * vh;
        else acck[e] += gv[e] * vh;
        gv[e] = rho * (gv[e] * Elem<T>::to_f(gain[lane * E + e]) - vh * mean);
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) gp[e] = Elem<T>::from_f(gv[e]);
  }
  if (dgq)
#pragma unroll
    for (int e = 0; e < E; ++e) dgq[m * HD + lane * E + e] = accq[e];
  if (dgk)
#pragma unroll
    for (int e = 0; e < E; ++e) dgk[m * HD + lane * E + e] = acck[e];
}

cudaError_t launch_qk_transform_bwd(const Ctx& c, xmod_dtype dt, int64_t M, void* g, int ld,
                                    int q_col0, int q_heads, const void* q_gain, int k_col0,
                                    int k_heads, const void* k_gain, const void* pre, int ldp,
                                    int hd, float eps, float theta, const int32_t* pos_idx,
                                    int seqT, float* dgq, float* dgk) {
  if (M <= 0 || q_heads + k_heads <= 0) return cudaSuccess;
  if (hd % 32 || hd > 128 || seqT <= 0 || seqT >= (1 << 24)) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)((M + ROW_WARPS - 1) / ROW_WARPS);
#define XMOD_QKB_CASE(TT, EE)                                                                 \
  return launch_pdl(qk_transform_bwd_kernel<TT, EE>, dim3(blocks), dim3(ROW_WARPS * 32), 0,    \
                    c.stream, M, (TT*)g, ld, q_col0, q_heads, (const TT*)q_gain, k_col0,       \
                    k_heads, (const TT*)k_gain, (const TT*)pre, ldp, eps, (double)theta,       \
                    pos_idx, seqT, dgq, dgk);
  if (dt == XMOD_BF16) {
    switch (hd / 32) {
      case 1: XMOD_QKB_CASE(__nv_bfloat16, 1)
      case 2: XMOD_QKB_CASE(__nv_bfloat16, 2)
      case 4: XMOD_QKB_CASE(__nv_bfloat16, 4)
    }
  } else {
    switch (hd / 32) {
      case 1: XMOD_QKB_CASE(float, 1)
      case 2: XMOD_QKB_CASE(float, 2)
      case 4: XMOD_QKB_CASE(float, 4)
    }
  }
#undef XMOD_QKB_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_qk_transform(const Ctx& c, xmod_dtype dt, int64_t M, const int32_t* M_dev,
                                void* x, int ld, int q_col0, int q_heads, const void* q_gain,
                                int k_col0, int k_heads, const void* k_gain, int hd, float eps,
                                float theta, const int32_t* pos_idx, const int32_t* pos_tok,
                                int seqT) {
  if (M <= 0 || q_heads + k_heads <= 0) return cudaSuccess;
  if (hd % 32 || hd > 128 || seqT <= 0 || seqT >= (1 << 24)) return cudaErrorInvalidValue;
  const unsigned blocks = (unsigned)((M + ROW_WARPS - 1) / ROW_WARPS);
#define XMOD_QK_CASE(TT, EE)                                                                  \
  return launch_pdl(qk_transform_kernel<TT, EE>, dim3(blocks), dim3(ROW_WARPS * 32), 0,        \
                    c.stream, M, M_dev, (TT*)x, ld, q_col0, q_heads, (const TT*)q_gain,        \
                    k_col0, k_heads, (const TT*)k_gain, eps, (double)theta, pos_idx, pos_tok,  \
                    seqT);
  if (dt == XMOD_BF16) {
    switch (hd / 32) {
      case 1: XMOD_QK_CASE(__nv_bfloat16, 1)
      case 2: XMOD_QK_CASE(__nv_bfloat16, 2)
      case 4: XMOD_QK_CASE(__nv_bfloat16, 4)
    }
  } else {
    switch (hd / 32) {
      case 1: XMOD_QK_CASE(float, 1)
      case 2: XMOD_QK_CASE(float, 2)
      case 4: XMOD_QK_CASE(float, 4)
    }
  }
#undef XMOD_QK_CASE
  return cudaErrorInvalidValue;
}

// ================================================================ caller positions

// out[m] = idx[m] where row m passes row_idx_ok; a row that does not gets its position
// clamped into [0, seqT) (so every later access stays inside the stream) and the status
// word records XMOD_ERR_DEVICE_CHECK.
__global__ void idx_sanitize_kernel(int64_t M, int seqT, int n, const int32_t* __restrict__ idx,
                                    int32_t* __restrict__ out, int* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const int32_t t = idx[m];
  out[m] = row_idx_ok(m, seqT, n, idx, status) ? t : min(max(t, 0), seqT - 1);
}

cudaError_t launch_idx_sanitize(const Ctx& c, int B, int T, int n, const int32_t* idx,
                                int32_t* out) {
  const int64_t M = (int64_t)B * n;
  if (M <= 0) return cudaSuccess;
  return launch_pdl(idx_sanitize_kernel, dim3((unsigned)((M + 255) / 256)), dim3(256), 0,
                    c.stream, M, T, n, idx, out, c.status);
}

// ================================================================ gated scatter

// One warp per selected row, the row taken in chunks of SCATTER_CHUNK 16-byte vectors
// per lane: every load of a chunk (x, a and f) is issued before the chunk's first store.
constexpr int SCATTER_CHUNK = 8;

template <typename T>
__global__ void __launch_bounds__(ROW_WARPS * 32)
gated_scatter_kernel(int64_t M, int seqT, int n, int d, T* __restrict__ x,
                     const int32_t* __restrict__ idx, const float* __restrict__ r_sel,
                     const T* __restrict__ a, const T* __restrict__ f, float varsigma, int gate,
                     int* status) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Vec16<T>::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m = (int64_t)blockIdx.x * ROW_WARPS + warp;
  if (m >= M || !row_idx_ok(m, seqT, n, idx, status)) return;
  T* row = x + stream_row(m, seqT, n, idx) * d;
  const T* arow = a + m * d;
  const T* frow = f ? f + m * d : nullptr;
  const float r = (gate >= 0) ? r_sel[m] : 1.0f;
  const float g7 = varsigma * r;
  for (int c0 = lane * V; c0 < d; c0 += SCATTER_CHUNK * 32 * V) {
    Vec16<T> xv[SCATTER_CHUNK], av[SCATTER_CHUNK], fv[SCATTER_CHUNK];
#pragma unroll
    for (int i = 0; i < SCATTER_CHUNK; ++i) {
      const int c = c0 + i * 32 * V;
      if (c < d) {
        xv[i] = ld_vec(row + c);
        av[i] = ld_vec_stream(arow + c);
        if (frow) fv[i] = ld_vec_stream(frow + c);
      }
    }
#pragma unroll
    for (int i = 0; i < SCATTER_CHUNK; ++i) {
      const int c = c0 + i * 32 * V;
      if (c >= d) break;
      Vec16<T> o;
      if (frow) {
#pragma unroll
        for (int e = 0; e < V; ++e) {
          const float xa = xv[i].get(e), aa = av[i].get(e), ff = fv[i].get(e);
          float y;
          if (gate == XMOD_GATE_XMOD) y = xa + g7 * (aa + ff);       // Eq. 7
          else if (gate == XMOD_GATE_MOD) y = xa + aa + r * ff;      // Eq. 6
          else y = xa + aa + ff;                                      // dense layer
          o.set(e, y);
        }
      } else {  // a holds a + f (Eq. 7 only)
#pragma unroll
        for (int e = 0; e < V; ++e) o.set(e, xv[i].get(e) + g7 * av[i].get(e));
      }
      st_vec(row + c, o);
    }
  }
}

cudaError_t launch_gated_scatter(const Ctx& c, xmod_dtype dt, int B, int T, int n, int d,
                                 void* x, const int32_t* idx, const float* r_sel, const void* a,
                                 const void* f, float varsigma, int gate) {
  const int64_t M = (int64_t)B * n;
  if (M <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((M + ROW_WARPS - 1) / ROW_WARPS);
  if (dt == XMOD_BF16)
    launch_pdl(gated_scatter_kernel<__nv_bfloat16>, dim3(blocks), dim3(ROW_WARPS * 32), 0, c.stream, 
        M, T, n, d, (__nv_bfloat16*)x, idx, r_sel, (const __nv_bfloat16*)a,
        (const __nv_bfloat16*)f, varsigma, gate, c.status);
  else
    launch_pdl(gated_scatter_kernel<float>, dim3(blocks), dim3(ROW_WARPS * 32), 0, c.stream, 
        M, T, n, d, (float*)x, idx, r_sel, (const float*)a, (const float*)f, varsigma, gate,
        c.status);
  return cudaGetLastError();
}

}  // namespace xmod
