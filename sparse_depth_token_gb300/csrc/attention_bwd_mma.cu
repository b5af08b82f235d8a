// Backward of the causal GQA attention among each sequence's n compact rows (bf16), on
// the warp-level tensor-core MMA (mma.sync m16n8k16, bf16 operands, fp32 accumulation).
//
// Source: the block of the X-MoD notes' "backbone configuration" (GQA attention over the
// selected tokens, section "mechanism controls": attention among the selected tokens
// only). The gradients are those of softmax attention, o = P v with P = softmax(scale q.k^T)
// over the keys at or before each query: with D_i = <dO_i, o_i>,
//   dP = dO v^T,   dS = P * (dP - D),   dq = scale dS k,   dk = scale dS^T q,   dv = P^T dO.
//
// The Selected-Q / full-KV control (same section) is the general form: n queries per
// sequence at ascending positions qpos among nk keys, query i seeing the keys j <=
// qpos[i]; the compact case is qpos[i] = i, nk = n.
//
// Two kernels, each a CTA of four warps and 64-row tiles (16 rows per warp):
//   attn_bwd_q_mma: per (64-query tile, query head, sequence). Pass 1 recomputes the row
//     statistics lse = m + log(l) over the key tiles up to the tile's last query position;
//     pass 2
//     forms P, dP, dS and accumulates dq. Writes lse and D for the second kernel.
//   attn_bwd_kv_mma: per (64-key tile, KV head, sequence), over the group's query heads
//     and the queries from the first one positioned at or after the tile's first key:
//     S^T = k q^T and dP^T = v dO^T, then
//     dv += P^T dO and dk += dS^T q. Every key row belongs to one CTA: no atomics.
// Operands are staged in shared memory with rows padded by 8 elements (16 bytes), so the
// eight rows an ldmatrix reads fall in distinct 16-byte bank groups.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace xmod {

namespace {

constexpr int AM_T = 64;        // rows (queries or keys) per tile
constexpr int AM_WARPS = 4;     // 16 rows per warp

__device__ __forceinline__ uint32_t am_smem(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// d += a b (16x8x16, bf16 -> fp32)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t am_pack(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// rows [r0, r0 + 64) of a bf16 matrix (row stride ld elements, columns col0 .. col0 + HD)
// into shared memory [64][HD + 8]; rows at or beyond n are zero.
template <int HD>
__device__ __forceinline__ void am_load_tile(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                             int64_t ld, int r0, int n, int col0) {
  constexpr int P = HD + 8, V = HD / 8;   // 16-byte vectors per row
  for (int e = threadIdx.x; e < AM_T * V; e += AM_WARPS * 32) {
    const int r = e / V, v = e - r * V;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r0 + r < n) val = *reinterpret_cast<const uint4*>(src + (int64_t)(r0 + r) * ld + col0 + 8 * v);
    *reinterpret_cast<uint4*>(dst + r * P + 8 * v) = val;
  }
}

// Asynchronous copies (cp.async): 16 bytes, or 4; an invalid source is zero-filled (no
// bytes read; the address given is still a valid one).
__device__ __forceinline__ void cp16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(am_smem(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(am_smem(dst)), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// am_load_tile with asynchronous copies (complete at the caller's cp_wait).
template <int HD>
__device__ __forceinline__ void am_load_tile_async(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                                   int64_t ld, int r0, int n, int col0) {
  constexpr int P = HD + 8, V = HD / 8;
  for (int e = threadIdx.x; e < AM_T * V; e += AM_WARPS * 32) {
    const int r = e / V, v = e - r * V;
    const bool ok = r0 + r < n;
    cp16(dst + r * P + 8 * v, src + (ok ? (int64_t)(r0 + r) * ld + col0 + 8 * v : 0), ok);
  }
}

// A fragments of the 16 rows [row0, row0 + 16) x columns [k0, k0 + 16) of a [.][P] tile.
template <int P>
__device__ __forceinline__ void am_lda(const __nv_bfloat16* s, int row0, int k0,
                                       uint32_t (&a)[4]) {
  const int t = threadIdx.x & 31;
  const int row = row0 + (t & 7) + ((t >> 3) & 1) * 8, col = k0 + (t >> 4) * 8;
  ldsm_x4(am_smem(s + row * P + col), a);
}
// B fragments (two 8-column n-blocks) for B[k][n] = S[n][k], S a [.][P] tile with rows n:
// n in [n0, n0 + 16), k in [k0, k0 + 16). b[0], b[1]: n-block 0; b[2], b[3]: n-block 1.
template <int P>
__device__ __forceinline__ void am_ldb_nk(const __nv_bfloat16* s, int n0, int k0,
                                          uint32_t (&b)[4]) {
  const int t = threadIdx.x & 31;
  const int row = n0 + (t & 7) + (t >> 4) * 8, col = k0 + ((t >> 3) & 1) * 8;
  ldsm_x4(am_smem(s + row * P + col), b);
}
// B fragments for B[k][n] = S[k][n], S a [.][P] tile with rows k: k in [k0, k0 + 16),
// n in [n0, n0 + 16).
template <int P>
__device__ __forceinline__ void am_ldb_kn(const __nv_bfloat16* s, int k0, int n0,
                                          uint32_t (&b)[4]) {
  const int t = threadIdx.x & 31;
  const int row = k0 + (t & 7) + ((t >> 3) & 1) * 8, col = n0 + (t >> 4) * 8;
  ldsm_x4_t(am_smem(s + row * P + col), b);
}

// acc[16 x 64] = A rows [row0, +16) of sa . (rows [0, 64) of sb)^T over HD columns.
template <int HD>
__device__ __forceinline__ void am_qk(const __nv_bfloat16* sa, int row0,
                                      const __nv_bfloat16* sb, float (&acc)[8][4]) {
  constexpr int P = HD + 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
#pragma unroll
  for (int kc = 0; kc < HD / 16; ++kc) {
    uint32_t a[4];
    am_lda<P>(sa, row0, kc * 16, a);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b[4];
      am_ldb_nk<P>(sb, np * 16, kc * 16, b);
      mma16816(acc[2 * np], a, b[0], b[1]);
      mma16816(acc[2 * np + 1], a, b[2], b[3]);
    }
  }
}

// out[16 x HD] += A[16 x 64] . S[64 x HD], A given as fp32 C fragments (cast to bf16),
// S rows [0, 64) of a [.][P] tile.
template <int HD>
__device__ __forceinline__ void am_pv(const float (&pa)[8][4], const __nv_bfloat16* s,
                                      float (&out)[HD / 8][4]) {
  constexpr int P = HD + 8;
#pragma unroll
  for (int kb = 0; kb < 4; ++kb) {   // 16 rows of S (k) at a time
    uint32_t a[4];
    a[0] = am_pack(pa[2 * kb][0], pa[2 * kb][1]);
    a[1] = am_pack(pa[2 * kb][2], pa[2 * kb][3]);
    a[2] = am_pack(pa[2 * kb + 1][0], pa[2 * kb + 1][1]);
    a[3] = am_pack(pa[2 * kb + 1][2], pa[2 * kb + 1][3]);
#pragma unroll
    for (int np = 0; np < HD / 16; ++np) {
      uint32_t b[4];
      am_ldb_kn<P>(s, kb * 16, np * 16, b);
      mma16816(out[2 * np], a, b[0], b[1]);
      mma16816(out[2 * np + 1], a, b[2], b[3]);
    }
  }
}

struct AmArgs {
  int n, hq, hkv;             // n queries per sequence
  int nk;                     // keys per sequence
  const int32_t* qpos;        // [B*n] ascending query positions (NULL: i, nk == n)
  const __nv_bfloat16* q;     // q of head h at column h*HD of [B*n, ldq]
  int ldq;
  const __nv_bfloat16* k;     // k, v of KV head g at column g*HD of [B*nk, ldk], [B*nk, ldv]
  const __nv_bfloat16* v;
  int ldk, ldv;
  const __nv_bfloat16* o;     // [B*n, hq*HD]
  const __nv_bfloat16* dO;    // [B*n, hq*HD]
  float* lse;                 // [B*n, hq]
  float* Dd;                  // [B*n, hq]
  __nv_bfloat16* dq;          // dq of head h at column h*HD of [B*n, ldgq]
  int ldgq;
  __nv_bfloat16* dk;          // dk, dv of KV head g at column g*HD of [B*nk, ldgk]
  __nv_bfloat16* dv;
  int ldgk;
  float scale;
};

__device__ __forceinline__ int am_qpos(const AmArgs& p, int b, int i) {
  return p.qpos ? p.qpos[(int64_t)b * p.n + i] : i;
}

template <int HD>
__global__ void __launch_bounds__(AM_WARPS * 32)
attn_bwd_q_mma(const AmArgs p) {
  pdl_trigger();
  pdl_wait();
  constexpr int P = HD + 8;
  extern __shared__ __align__(16) unsigned char am_raw[];
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(am_raw);
  __nv_bfloat16* dOs = Qs + AM_T * P;
  __nv_bfloat16* Kb = dOs + AM_T * P;   // two key tiles
  __nv_bfloat16* Vb = Kb + 2 * AM_T * P;   // two value tiles
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (p.hq / p.hkv);
  const int qw = p.hq * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = qt * AM_T;
  const __nv_bfloat16* kbase = p.k + (int64_t)b * p.nk * p.ldk;
  const __nv_bfloat16* vbase = p.v + (int64_t)b * p.nk * p.ldv;
  // Key tiles up to the tile's last query position (positions ascend): nkt of them in
  // pass 1 (keys only), then again with values (pass 2); item i loads into buffer i % 2
  // while item i - 1 is computed.
  const int nkt = am_qpos(p, b, min(q0 + AM_T, p.n) - 1) / AM_T + 1;
  const int items = 2 * nkt;
  auto issue = [&](int it) {
    const int kt = it < nkt ? it : it - nkt, buf = it & 1;
    am_load_tile_async<HD>(Kb + buf * AM_T * P, kbase, p.ldk, kt * AM_T, p.nk, g * HD);
    if (it >= nkt)
      am_load_tile_async<HD>(Vb + buf * AM_T * P, vbase, p.ldv, kt * AM_T, p.nk, g * HD);
    cp_commit();
  };
  am_load_tile_async<HD>(Qs, p.q + (int64_t)b * p.n * p.ldq, p.ldq, q0, p.n, h * HD);
  am_load_tile_async<HD>(dOs, p.dO + (int64_t)b * p.n * qw, qw, q0, p.n, h * HD);
  issue(0);
  // D_i = <dO_i, o_i>: four lanes per row of this warp's 16 (rows lane/4 and lane/4 + 8
  // are this lane's rows in the MMA fragments)
  float Dr[2];
  int qp[2];   // the rows' positions (-1 past the sequence: no key)
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int i = warp * 16 + (lane >> 2) + 8 * hr, qi = q0 + i;
    qp[hr] = qi < p.n ? am_qpos(p, b, qi) : -1;
    float acc = 0.0f;
    if (qi < p.n) {
      const __nv_bfloat16* orow = p.o + ((int64_t)b * p.n + qi) * qw + h * HD;
      const __nv_bfloat16* grow = p.dO + ((int64_t)b * p.n + qi) * qw + h * HD;
      for (int c = (lane & 3) * 2; c < HD; c += 8) {
        const float2 ov = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(orow + c));
        const float2 gv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(grow + c));
        acc += ov.x * gv.x + ov.y * gv.y;
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    Dr[hr] = acc;
  }
  const float sl2 = p.scale * 1.4426950408889634f;   // scale in log2 units
  // pass 1: row max and sum in log2 units
  float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.0f, 0.0f};
  for (int kt = 0; kt < nkt; ++kt) {
    const int k0 = kt * AM_T;
    const __nv_bfloat16* Ks = Kb + (kt & 1) * AM_T * P;
    issue(kt + 1);   // the next item exists: pass 2 follows
    cp_wait<1>();
    __syncthreads();
    float s[8][4];
    am_qk<HD>(Qs, warp * 16, Ks, s);
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kj = k0 + j * 8 + (lane & 3) * 2 + e;
          const bool ok = kj <= qp[hr];   // qp < nk
          const float v = ok ? s[j][2 * hr + e] * sl2 : -INFINITY;
          s[j][2 * hr + e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      // every lane takes the shuffles (rows past n have no valid key and add nothing)
      const float mn = fmaxf(mr[hr], mx);
      const float mref = mn > -INFINITY ? mn : 0.0f;
      float add = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        add += exp2f(s[j][2 * hr] - mref) + exp2f(s[j][2 * hr + 1] - mref);
      add += __shfl_xor_sync(0xffffffffu, add, 1);
      add += __shfl_xor_sync(0xffffffffu, add, 2);
      if (mn > -INFINITY) {
        lr[hr] = lr[hr] * exp2f(mr[hr] - mn) + add;
        mr[hr] = mn;
      }
    }
    __syncthreads();   // this buffer is refilled by the item after next
  }
  float lse2[2];   // log2-sum-exp2 of the scaled logits
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lse2[hr] = mr[hr] + log2f(lr[hr]);
    const int qi = q0 + warp * 16 + (lane >> 2) + 8 * hr;
    if ((lane & 3) == 0 && qi < p.n) {
      p.lse[((int64_t)b * p.n + qi) * p.hq + h] = lse2[hr];
      p.Dd[((int64_t)b * p.n + qi) * p.hq + h] = Dr[hr];
    }
  }
  // pass 2: dq
  float dq[HD / 8][4];
#pragma unroll
  for (int j = 0; j < HD / 8; ++j) dq[j][0] = dq[j][1] = dq[j][2] = dq[j][3] = 0.0f;
  for (int kt = 0; kt < nkt; ++kt) {
    const int k0 = kt * AM_T, it = nkt + kt;
    const __nv_bfloat16* Ks = Kb + (it & 1) * AM_T * P;
    const __nv_bfloat16* Vs = Vb + (it & 1) * AM_T * P;
    if (it + 1 < items) {
      issue(it + 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    float s[8][4], dp[8][4];
    am_qk<HD>(Qs, warp * 16, Ks, s);
    am_qk<HD>(dOs, warp * 16, Vs, dp);
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hr = e >> 1;
        const int kj = k0 + j * 8 + (lane & 3) * 2 + (e & 1);
        const bool ok = kj <= qp[hr];
        const float pr = ok ? exp2f(s[j][e] * sl2 - lse2[hr]) : 0.0f;
        s[j][e] = pr * (dp[j][e] - Dr[hr]);   // dS
      }
    am_pv<HD>(s, Ks, dq);
    __syncthreads();
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int qi = q0 + warp * 16 + (lane >> 2) + 8 * hr;
    if (qi >= p.n) continue;
    __nv_bfloat16* out = p.dq + ((int64_t)b * p.n + qi) * p.ldgq + h * HD;
#pragma unroll
    for (int j = 0; j < HD / 8; ++j)
      *reinterpret_cast<uint32_t*>(out + j * 8 + (lane & 3) * 2) =
          am_pack(dq[j][2 * hr] * p.scale, dq[j][2 * hr + 1] * p.scale);
  }
}

template <int HD>
__global__ void __launch_bounds__(AM_WARPS * 32)
attn_bwd_kv_mma(const AmArgs p) {
  pdl_trigger();
  pdl_wait();
  constexpr int P = HD + 8;
  extern __shared__ __align__(16) unsigned char am_raw[];
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(am_raw);
  __nv_bfloat16* Vs = Ks + AM_T * P;
  __nv_bfloat16* Qb = Vs + AM_T * P;        // two query tiles
  __nv_bfloat16* dOb = Qb + 2 * AM_T * P;   // two dO tiles
  float* lse_b = reinterpret_cast<float*>(dOb + 2 * AM_T * P);   // [2][AM_T]
  float* D_b = lse_b + 2 * AM_T;                                   // [2][AM_T]
  int* qp_b = reinterpret_cast<int*>(D_b + 2 * AM_T);              // [2][AM_T]
  const int kt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = p.hq / p.hkv;
  const int qw = p.hq * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = kt * AM_T;
  const __nv_bfloat16* qbase = p.q + (int64_t)b * p.n * p.ldq;
  // the first query positioned at or after the tile's first key: a binary search over the
  // ascending positions, the same in every thread
  int qstart;
  {
    int lo = 0, hi = p.n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (am_qpos(p, b, mid) >= k0) hi = mid; else lo = mid + 1;
    }
    qstart = lo;
  }
  // items: (query head of the group, query tile from qstart); item i loads into buffer
  // i % 2 while item i - 1 is computed
  const int nq = (p.n - qstart + AM_T - 1) / AM_T;
  const int items = G * nq;
  auto issue = [&](int it) {
    const int h = g * G + it / nq, q0 = qstart + (it % nq) * AM_T, buf = it & 1;
    am_load_tile_async<HD>(Qb + buf * AM_T * P, qbase, p.ldq, q0, p.n, h * HD);
    am_load_tile_async<HD>(dOb + buf * AM_T * P, p.dO + (int64_t)b * p.n * qw, qw, q0, p.n,
                           h * HD);
    for (int i = threadIdx.x; i < AM_T; i += AM_WARPS * 32) {
      const int qi = q0 + i;
      const bool ok = qi < p.n;
      const int64_t o = ok ? ((int64_t)b * p.n + qi) * p.hq + h : 0;
      cp4(lse_b + buf * AM_T + i, p.lse + o, ok);
      cp4(D_b + buf * AM_T + i, p.Dd + o, ok);
      if (p.qpos)
        cp4(qp_b + buf * AM_T + i, p.qpos + (ok ? (int64_t)b * p.n + qi : 0), ok);
      else
        qp_b[buf * AM_T + i] = qi;   // read after the barrier that follows the wait
    }
    cp_commit();
  };
  if (items > 0) {   // no query sees this key tile: its dk, dv stay zero (written below)
    am_load_tile_async<HD>(Ks, p.k + (int64_t)b * p.nk * p.ldk, p.ldk, k0, p.nk, g * HD);
    am_load_tile_async<HD>(Vs, p.v + (int64_t)b * p.nk * p.ldv, p.ldv, k0, p.nk, g * HD);
    issue(0);
  }
  const float sl2 = p.scale * 1.4426950408889634f;
  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int j = 0; j < HD / 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[j][e] = dv[j][e] = 0.0f;
  for (int it = 0; it < items; ++it) {
    const int q0 = qstart + (it % nq) * AM_T, buf = it & 1;
    const __nv_bfloat16* Qs = Qb + buf * AM_T * P;
    const __nv_bfloat16* dOs = dOb + buf * AM_T * P;
    const float* lse_s = lse_b + buf * AM_T;
    const float* D_s = D_b + buf * AM_T;
    const int* qp_s = qp_b + buf * AM_T;
    if (it + 1 < items) {
      issue(it + 1);
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();
    float s[8][4], dp[8][4];
    am_qk<HD>(Ks, warp * 16, Qs, s);    // S^T: rows keys, columns queries
    am_qk<HD>(Vs, warp * 16, dOs, dp);  // dP^T
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kj = k0 + warp * 16 + (lane >> 2) + 8 * (e >> 1);
        const int ci = j * 8 + (lane & 3) * 2 + (e & 1);   // query within the tile
        const int qi = q0 + ci;
        const bool ok = qi < p.n && kj < p.nk && kj <= qp_s[ci];
        const float pr = ok ? exp2f(s[j][e] * sl2 - lse_s[ci]) : 0.0f;
        s[j][e] = pr;
        dp[j][e] = pr * (dp[j][e] - D_s[ci]);   // dS^T
      }
    am_pv<HD>(s, dOs, dv);
    am_pv<HD>(dp, Qs, dk);
    __syncthreads();   // this buffer is refilled by the item after next
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int kj = k0 + warp * 16 + (lane >> 2) + 8 * hr;
    if (kj >= p.nk) continue;
    const int64_t row = ((int64_t)b * p.nk + kj) * p.ldgk + g * HD;
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) {
      const int c = j * 8 + (lane & 3) * 2;
      *reinterpret_cast<uint32_t*>(p.dk + row + c) =
          am_pack(dk[j][2 * hr] * p.scale, dk[j][2 * hr + 1] * p.scale);
      *reinterpret_cast<uint32_t*>(p.dv + row + c) = am_pack(dv[j][2 * hr], dv[j][2 * hr + 1]);
    }
  }
}

template <int HD>
cudaError_t launch_am(int B, const AmArgs& a, cudaStream_t st, bool with_q) {
  constexpr int P = HD + 8;
  const size_t smq = sizeof(__nv_bfloat16) * 6 * AM_T * P;
  const size_t smk = smq + sizeof(float) * 6 * AM_T;
  cudaFuncSetAttribute(attn_bwd_q_mma<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smq);
  cudaFuncSetAttribute(attn_bwd_kv_mma<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
  const int qtiles = (a.n + AM_T - 1) / AM_T, ktiles = (a.nk + AM_T - 1) / AM_T;
  if (with_q) {
    const cudaError_t e = launch_pdl(attn_bwd_q_mma<HD>, dim3(qtiles, a.hq, B),
                                     dim3(AM_WARPS * 32), smq, st, a);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(attn_bwd_kv_mma<HD>, dim3(ktiles, a.hkv, B), dim3(AM_WARPS * 32), smk, st,
                    a);
}

}  // namespace

bool attn_bwd_mma_supported(int hd, int ldq, int ldo) {
  return (hd == 64 || hd == 128) && ldq % 8 == 0 && ldo % 8 == 0;
}

cudaError_t launch_attn_bwd_mma_kv(const Ctx& c, int B, int n, int nk, const int32_t* qpos,
                                   int hq, int hkv, int hd, const void* q, int ldq,
                                   const void* k, int ldk, const void* v, int ldv, const void* o,
                                   const void* dO, float* lse, float* Dd, void* dq, int ldgq,
                                   void* dk, void* dv, int ldgk, bool with_q) {
  if (!attn_bwd_mma_supported(hd, ldq, hq * hd) || ldk % 8 || ldv % 8 || ldgq % 2 || ldgk % 2)
    return cudaErrorInvalidValue;
  AmArgs a;
  a.n = n;
  a.nk = nk;
  a.qpos = qpos;
  a.hq = hq;
  a.hkv = hkv;
  a.q = (const __nv_bfloat16*)q;
  a.ldq = ldq;
  a.k = (const __nv_bfloat16*)k;
  a.v = (const __nv_bfloat16*)v;
  a.ldk = ldk;
  a.ldv = ldv;
  a.o = (const __nv_bfloat16*)o;
  a.dO = (const __nv_bfloat16*)dO;
  a.lse = lse;
  a.Dd = Dd;
  a.dq = (__nv_bfloat16*)dq;
  a.ldgq = ldgq;
  a.dk = (__nv_bfloat16*)dk;
  a.dv = (__nv_bfloat16*)dv;
  a.ldgk = ldgk;
  a.scale = 1.0f / sqrtf((float)hd);
  return hd == 128 ? launch_am<128>(B, a, c.stream, with_q) : launch_am<64>(B, a, c.stream, with_q);
}

cudaError_t launch_attn_bwd_mma(const Ctx& c, int B, int n, int hq, int hkv, int hd,
                                const void* qkv, int ldq, const void* o, const void* dO,
                                float* lse, float* Dd, void* dqkv, int ldg, bool with_q) {
  const int qw = hq * hd, kw = hkv * hd;
  const __nv_bfloat16* x = (const __nv_bfloat16*)qkv;
  __nv_bfloat16* g = (__nv_bfloat16*)dqkv;
  return launch_attn_bwd_mma_kv(c, B, n, n, nullptr, hq, hkv, hd, x, ldq, x + qw, ldq,
                                x + qw + kw, ldq, o, dO, lse, Dd, g, ldg, g + qw, g + qw + kw,
                                ldg, with_q);
}

}  // namespace xmod
