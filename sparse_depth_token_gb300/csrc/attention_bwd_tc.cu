// dQ of the causal GQA attention backward on the tcgen05 tensor cores (bf16, head_dim
// 128): dq = scale * sum_j dS_ij k_j with dS = P * (dP - D), P = exp2(scale_log2 q.k -
// lse), dP = dO v^T, D_i = <dO_i, o_i>.
//
// Source: the block of the X-MoD notes' "backbone configuration" (GQA attention among
// the selected tokens); the gradient is that of softmax attention.
//
// One CTA per (128-query block, query head, sequence), laid out as the forward kernel:
//   warp 0      TMA: the Q and dO tiles once, then per 64-key block the rows of K and of
//               V into a four-stage ring (the K rows serve S = Q K^T as a K-major
//               operand and dQ += dS K as an MN-major one, so no transposed copy)
//   warp 1      TMEM owner; one lane issues S_j = Q K_j^T and dP_j = dO V_j^T into one
//               of two TMEM buffer pairs, and dQ += dS_j K_j once dS_j is written, with
//               dS_j read from TMEM as the MMA's A operand
//   warps 2..5  one query row per thread (a TMEM lane is a row): D and lse of the row,
//               then per key block P and dS from S and dP in registers; dS goes back to
//               TMEM as bf16 pairs over the first half of S_j's columns
// The row statistics lse come from the forward pass (its log2-sum-exp2 output); D is
// computed here and written for the key/value kernel.
//
// Both kernels also take the Selected-Q / full-KV control of the same notes ("mechanism
// controls"): n queries per sequence at ascending positions qpos among nk keys, query i
// seeing the keys j <= qpos[i], keys and values read from their own rows; the compact
// case is qpos[i] = i, nk = n.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace xmod {

namespace {

using namespace tc;

constexpr int QB = 128;                  // query rows per CTA
constexpr int HD = 128;                  // head dim
constexpr int KB = 64;                   // keys per block
constexpr int NST = 4;                   // stages of the key ring
constexpr int THREADS = 192;
constexpr int CHUNK = 128 * 128;         // 128 rows x 64 bf16 columns, 128-byte swizzle
constexpr int QTILE = 2 * CHUNK;         // 128 x 128
constexpr int K_CHUNK = KB * 128;        // 64 rows x 64 columns
constexpr int K_TILE = 2 * K_CHUNK;      // 64 keys x 128 head dims
constexpr int STAGE = 2 * K_TILE;        // K and V rows
constexpr int DATA = 2 * QTILE + NST * STAGE;
constexpr int SMEM = DATA + 1024;
constexpr int TMEM_COLS = 512;           // S0, S1, dP0, dP1 (64 each), dQ (128)
static_assert((1 + 2 * NST + 8) * 8 + 16 <= 256, "barrier block overflows");

struct DqArgs {
  int n, hq, hkv, nqb;
  int nk;                     // keys per sequence
  const int32_t* qpos;        // [B*n] query positions (NULL: i)
  int k_col0, v_col0;         // columns of KV head 0's k and v in the key map's rows
  int qw;
  float scale_log2, scale;
  const float* lse;           // [B*n, hq], log2 units
  const __nv_bfloat16* o;     // [B*n, qw]
  const __nv_bfloat16* dO;    // [B*n, qw]
  float* Dd;                  // [B*n, hq] out
  float* DdT;                 // [B*hq, ldS] out (per head, queries contiguous) or NULL
  int ldS;
  __nv_bfloat16* dq;          // q columns of [B*n, ldg]
  int ldg;
  int* status;
};

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(THREADS, 1)
attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmDO,
                      const __grid_constant__ CUtensorMap tmK,
                      const DqArgs a) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sQ = base, sDO = base + QTILE;
  const uint32_t sSt0 = base + 2 * QTILE;   // stage s: K rows, V rows, K^T
  const uint32_t sBar = (base - raw >= 256u) ? raw : base + (uint32_t)DATA;
  const uint32_t QD_FULL = sBar;
  const uint32_t ST_FULL0 = sBar + 8, ST_EMPTY0 = ST_FULL0 + 8 * NST;
  const uint32_t S_FULL0 = ST_EMPTY0 + 8 * NST, S_EMPTY0 = S_FULL0 + 16;
  const uint32_t P_FULL0 = S_EMPTY0 + 16, P_EMPTY0 = P_FULL0 + 16;
  const uint32_t sTmem = P_EMPTY0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + (sTmem - raw));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + (sTmem - raw) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = a.nqb - 1 - (int)blockIdx.z;   // longest query blocks first
  const int h = blockIdx.x, b = blockIdx.y;
  const int g = h / (a.hq / a.hkv);
  const int q0 = qb * QB;

  if (threadIdx.x == 0) {
    mbar_init(QD_FULL, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(ST_FULL0 + 8 * s, 1);
      mbar_init(ST_EMPTY0 + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(S_FULL0 + 8 * s, 1);
      mbar_init(S_EMPTY0 + 8 * s, 128);
      mbar_init(P_FULL0 + 8 * s, 128);
      mbar_init(P_EMPTY0 + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmDO);
    prefetch_tensormap(&tmK);
  }
  if (warp == 1) tmem_alloc(sTmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tDQ = tmem + 256u;
  pdl_wait();
  const int last_q = min(q0 + QB, a.n) - 1;
  // key blocks up to the block's last query position (positions ascend)
  const int last_key = a.qpos && q0 < a.n ? a.qpos[(int64_t)b * a.n + last_q] : last_q;
  const int nkb = q0 < a.n ? last_key / KB + 1 : 0;

  if (warp == 0) {
    if (lane == 0 && nkb > 0) {
      mbar_arrive_expect_tx(QD_FULL, 2 * QTILE);
      tma_load_3d(sQ, &tmQ, QD_FULL, h * HD, q0, b);
      tma_load_3d(sQ + CHUNK, &tmQ, QD_FULL, h * HD + 64, q0, b);
      tma_load_3d(sDO, &tmDO, QD_FULL, h * HD, q0, b);
      tma_load_3d(sDO + CHUNK, &tmDO, QD_FULL, h * HD + 64, q0, b);
      for (int j = 0; j < nkb; ++j) {
        const int s = j % NST;
        if (!mbar_wait(ST_EMPTY0 + 8 * s, ((uint32_t)(j / NST) & 1u) ^ 1u, abort_flag, a.status))
          break;
        const uint32_t st = sSt0 + s * STAGE;
        mbar_arrive_expect_tx(ST_FULL0 + 8 * s, STAGE);
        tma_load_3d(st, &tmK, ST_FULL0 + 8 * s, a.k_col0 + g * HD, j * KB, b);
        tma_load_3d(st + K_CHUNK, &tmK, ST_FULL0 + 8 * s, a.k_col0 + g * HD + 64, j * KB, b);
        tma_load_3d(st + K_TILE, &tmK, ST_FULL0 + 8 * s, a.v_col0 + g * HD, j * KB, b);
        tma_load_3d(st + K_TILE + K_CHUNK, &tmK, ST_FULL0 + 8 * s, a.v_col0 + g * HD + 64,
                    j * KB, b);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, KB);
      constexpr uint32_t idesc_q = idesc_bf16_f32(128, HD) | kIdescBMajorMN;   // B = K rows
      bool ok = nkb > 0 && mbar_wait(QD_FULL, 0, abort_flag, a.status);
      int ns = 0, nd = 0;
      uint64_t t0 = global_timer_ns();
      uint32_t spins = 0;
      while (ok && nd < nkb) {
        bool progressed = false;
        // S_{j+2} and dP_{j+2} reuse buffer j & 1, whose first half holds dS_j: issued
        // after dQ += dS_j K_j (the MMAs of one thread run in order)
        if (ns < nkb && ns <= nd + 1) {
          const int s = ns & 1, st = ns % NST;
          if (mbar_test_wait(ST_FULL0 + 8 * st, (uint32_t)(ns / NST) & 1u) &&
              mbar_test_wait(S_EMPTY0 + 8 * s, ((uint32_t)(ns >> 1) & 1u) ^ 1u)) {
            tc_fence_after();
            const uint32_t stg = sSt0 + st * STAGE;
            const uint32_t dS = tmem + (uint32_t)(s * KB), dP = tmem + 128u + (uint32_t)(s * KB);
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
              const uint64_t aq = smem_desc_sw128(sQ + kc * CHUNK);
              const uint64_t ao = smem_desc_sw128(sDO + kc * CHUNK);
              const uint64_t bk = smem_desc_sw128(stg + kc * K_CHUNK);
              const uint64_t bv = smem_desc_sw128(stg + K_TILE + kc * K_CHUNK);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                mma_bf16(dS, aq + 2ull * k, bk + 2ull * k, idesc_s, (kc | k) != 0 ? 1u : 0u);
                mma_bf16(dP, ao + 2ull * k, bv + 2ull * k, idesc_s, (kc | k) != 0 ? 1u : 0u);
              }
            }
            mma_commit(S_FULL0 + 8 * s);
            ++ns;
            progressed = true;
          }
        }
        if (nd < ns) {
          const int s = nd & 1, st = nd % NST;
          if (mbar_test_wait(P_FULL0 + 8 * s, (uint32_t)(nd >> 1) & 1u)) {
            tc_fence_after();
            const uint32_t tp = tmem + (uint32_t)(s * KB);
            // B = K_j [64 keys, 128 head dims] as stored: MN-major, 64-dim atoms one
            // chunk apart, 16 keys (2 KB) per MMA
            const uint64_t bd = smem_desc_sw128_mn(sSt0 + st * STAGE, K_CHUNK);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_tmem_a(tDQ, tp + (uint32_t)(8 * k), bd + 128ull * k, idesc_q,
                              (nd | k) != 0 ? 1u : 0u);
            mma_commit(P_EMPTY0 + 8 * s);
            mma_commit(ST_EMPTY0 + 8 * st);
            ++nd;
            progressed = true;
          }
        }
        if (progressed) {
          t0 = global_timer_ns();
          spins = 0;
          continue;
        }
        if ((++spins & 255u) == 0u) {
          if (*abort_flag) break;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            report_status(a.status, XMOD_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
      }
    }
  } else {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int qi = q0 + row;
    const bool valid = qi < a.n;
    const int64_t grow = (int64_t)b * a.n + (valid ? qi : 0);
    const int qp = valid ? (a.qpos ? a.qpos[grow] : qi) : -1;   // the row's last key
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    // D_i = <dO_i, o_i> and the row's lse (log2 units)
    float D = 0.f, lse2 = 0.f;
    if (valid && nkb > 0) {
      const uint4* op = reinterpret_cast<const uint4*>(a.o + grow * a.qw + h * HD);
      const uint4* gp = reinterpret_cast<const uint4*>(a.dO + grow * a.qw + h * HD);
#pragma unroll 4
      for (int v = 0; v < HD / 8; ++v) {
        const uint4 ov = op[v], gv = gp[v];
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __bfloat1622float2(o2[e]), y = __bfloat1622float2(g2[e]);
          D = fmaf(x.x, y.x, fmaf(x.y, y.y, D));
        }
      }
      lse2 = a.lse[grow * a.hq + h];
      a.Dd[grow * a.hq + h] = D;
      if (a.DdT) a.DdT[(int64_t)(b * a.hq + h) * a.ldS + qi] = D;
    }
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      if (!mbar_wait(S_FULL0 + 8 * s, (uint32_t)(j >> 1) & 1u, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[KB], dp[KB];
      const uint32_t srow = tmem + lane_off + (uint32_t)(s * KB);
      const uint32_t prow = tmem + lane_off + 128u + (uint32_t)(s * KB);
      tmem_ld32(srow, *reinterpret_cast<float(*)[32]>(sv));
      tmem_ld32(srow + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
      tmem_ld32(prow, *reinterpret_cast<float(*)[32]>(dp));
      tmem_ld32(prow + 32, *reinterpret_cast<float(*)[32]>(dp + 32));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(S_EMPTY0 + 8 * s);
      const int key0 = j * KB;
      float pk[32];
#pragma unroll
      for (int i = 0; i < KB; i += 2) {
        const bool ok0 = key0 + i <= qp, ok1 = key0 + i + 1 <= qp;
        const float p0 = ok0 ? ex2f(fmaf(sv[i], a.scale_log2, -lse2)) : 0.f;
        const float p1 = ok1 ? ex2f(fmaf(sv[i + 1], a.scale_log2, -lse2)) : 0.f;
        pk[i / 2] = __uint_as_float(pack_bf16x2(p0 * (dp[i] - D), p1 * (dp[i + 1] - D)));
      }
      // dS_j over the first half of S_j's columns (S_j has been read; dS_{j-2}, which the
      // buffer held before S_j, was consumed by then)
      tmem_st32(srow, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(P_FULL0 + 8 * s);
    }
    if (nkb == 0) ok = false;
    if (ok) {
      const int jl = nkb - 1;
      ok = mbar_wait(P_EMPTY0 + 8 * (jl & 1), (uint32_t)(jl >> 1) & 1u, abort_flag, a.status);
    }
    if (ok) {
      tc_fence_after();
      __nv_bfloat16* dst = a.dq + grow * a.ldg + h * HD;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(tDQ + lane_off + c * 32, v);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 q;
            q.x = pack_bf16x2(v[e] * a.scale, v[e + 1] * a.scale);
            q.y = pack_bf16x2(v[e + 2] * a.scale, v[e + 3] * a.scale);
            q.z = pack_bf16x2(v[e + 4] * a.scale, v[e + 5] * a.scale);
            q.w = pack_bf16x2(v[e + 6] * a.scale, v[e + 7] * a.scale);
            *reinterpret_cast<uint4*>(dst + c * 32 + e) = q;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // a wait ran out: let copies and MMAs in flight land before the memory is released
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 20000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- dK, dV
// One CTA per (128-key block, KV head, sequence), over the group's query heads and the
// 64-query blocks from the one holding the first query positioned at or after the key
// block's first key:
//   warp 0      TMA: the K and V tiles (rows) once, then per query block the rows of Q
//               and dO into a four-stage ring (K-major operands of S^T and dP^T, MN-major
//               ones of dK and dV, so no transposed copies)
//   warp 1      one lane issues S^T = K Q^T and dP^T = V dO^T (keys in the TMEM lanes)
//               into two buffer pairs, then dV += P^T dO and dK += dS^T Q with P^T and
//               dS^T read from TMEM
//   warps 2..5  one key row per thread: P^T = exp2(scale_log2 s - lse[query]) under the
//               causal mask, dS^T = P^T (dP^T - D[query]), both back to TMEM as bf16
//               pairs over the first halves of their buffers
constexpr int KVB = kAttnBwdKvBlock;      // keys per CTA (128)
constexpr int QBK = 64;                   // queries per block
constexpr int KV_TILE = 2 * CHUNK;        // 128 keys x 128 head dims
constexpr int Q_CHUNK = QBK * 128;        // 64 rows x 64 columns
constexpr int Q_TILE = 2 * Q_CHUNK;       // 64 queries x 128 head dims
constexpr int KST2 = 4;                   // stages of the query ring
constexpr int QSTAGE = 2 * Q_TILE;        // Q, dO
constexpr int KV_DATA = 2 * KV_TILE + KST2 * QSTAGE;
constexpr int KV_SMEM = KV_DATA + 1024;
static_assert((1 + 2 * KST2 + 8) * 8 + 16 <= 256, "barrier block overflows");

struct DkvArgs {
  int n, hq, hkv;
  int nk;                     // keys per sequence
  int k_col0, v_col0;         // columns of KV head 0's k and v in the key map's rows
  // Selected-Q / full-KV (NULL both for the compact case): qposS [B, ldS] the query
  // positions, -1 past n; qstart [B, key blocks] the first query positioned at or after
  // each key block's first key
  const int32_t* qposS;
  const int32_t* qstart;
  float scale_log2, scale;
  const float* lseT;          // [B*hq, ldS]: lse (log2 units), per head, queries contiguous
  const float* DdT;           // [B*hq, ldS]: D, same layout
  int ldS;                    // a multiple of 64 at least n
  __nv_bfloat16* dk;          // dk, dv of KV head g at column g*HD of [B*nk, ldgk]
  __nv_bfloat16* dv;
  int ldgk;
  int* status;
};

__global__ void __launch_bounds__(THREADS, 1)
attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tmKV,
                       const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmDO, const DkvArgs a) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sK = base, sV = base + KV_TILE;
  const uint32_t sSt0 = base + 2 * KV_TILE;   // stage s: Q rows, dO rows, Q^T, dO^T
  const uint32_t sBar = (base - raw >= 256u) ? raw : base + (uint32_t)KV_DATA;
  const uint32_t KV_FULL = sBar;
  const uint32_t ST_FULL0 = sBar + 8, ST_EMPTY0 = ST_FULL0 + 8 * KST2;
  const uint32_t S_FULL0 = ST_EMPTY0 + 8 * KST2, S_EMPTY0 = S_FULL0 + 16;
  const uint32_t P_FULL0 = S_EMPTY0 + 16, P_EMPTY0 = P_FULL0 + 16;
  const uint32_t sTmem = P_EMPTY0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + (sTmem - raw));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + (sTmem - raw) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x, b = blockIdx.y, kb = blockIdx.z;   // key block 0 has most work
  const int G = a.hq / a.hkv;
  const int k0 = kb * KVB;
  // the first query that can see key k0 (compact case: query k0), its 64-query block
  const int qs = a.qstart ? a.qstart[(int64_t)b * gridDim.z + kb] : min(k0, a.n);
  const int qb0 = qs / QBK;
  const int nqb = (a.n + QBK - 1) / QBK - qb0;      // query blocks per head
  const int items = k0 < a.nk && qs < a.n ? G * nqb : 0;

  if (threadIdx.x == 0) {
    mbar_init(KV_FULL, 1);
    for (int s = 0; s < KST2; ++s) {
      mbar_init(ST_FULL0 + 8 * s, 1);
      mbar_init(ST_EMPTY0 + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(S_FULL0 + 8 * s, 1);
      mbar_init(S_EMPTY0 + 8 * s, 128);
      mbar_init(P_FULL0 + 8 * s, 128);
      mbar_init(P_EMPTY0 + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmKV);
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmDO);
  }
  if (warp == 1) tmem_alloc(sTmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;   // S^T 0/1: [0, 128); dP^T 0/1: [128, 256); dV, dK
  const uint32_t tDV = tmem + 256u, tDK = tmem + 384u;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0 && items > 0) {
      mbar_arrive_expect_tx(KV_FULL, 2 * KV_TILE);
      tma_load_3d(sK, &tmKV, KV_FULL, a.k_col0 + g * HD, k0, b);
      tma_load_3d(sK + CHUNK, &tmKV, KV_FULL, a.k_col0 + g * HD + 64, k0, b);
      tma_load_3d(sV, &tmKV, KV_FULL, a.v_col0 + g * HD, k0, b);
      tma_load_3d(sV + CHUNK, &tmKV, KV_FULL, a.v_col0 + g * HD + 64, k0, b);
      for (int it = 0; it < items; ++it) {
        const int s = it % KST2;
        const int h = g * G + it / nqb, q0 = (qb0 + it % nqb) * QBK;
        if (!mbar_wait(ST_EMPTY0 + 8 * s, ((uint32_t)(it / KST2) & 1u) ^ 1u, abort_flag,
                       a.status))
          break;
        const uint32_t st = sSt0 + s * QSTAGE;
        mbar_arrive_expect_tx(ST_FULL0 + 8 * s, QSTAGE);
        tma_load_3d(st, &tmQ, ST_FULL0 + 8 * s, h * HD, q0, b);
        tma_load_3d(st + Q_CHUNK, &tmQ, ST_FULL0 + 8 * s, h * HD + 64, q0, b);
        tma_load_3d(st + Q_TILE, &tmDO, ST_FULL0 + 8 * s, h * HD, q0, b);
        tma_load_3d(st + Q_TILE + Q_CHUNK, &tmDO, ST_FULL0 + 8 * s, h * HD + 64, q0, b);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, QBK);
      // dV += P^T dO and dK += dS^T Q: B = the dO / Q rows as stored, MN-major
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, HD) | kIdescBMajorMN;
      bool ok = items > 0 && mbar_wait(KV_FULL, 0, abort_flag, a.status);
      int ns = 0, nd = 0;
      uint64_t t0 = global_timer_ns();
      uint32_t spins = 0;
      while (ok && nd < items) {
        bool progressed = false;
        // S^T / dP^T of item i + 2 reuse buffer i & 1, holding P^T_i and dS^T_i: issued
        // after the dV / dK MMAs of item i (the MMAs of one thread run in order)
        if (ns < items && ns <= nd + 1) {
          const int s = ns & 1, st = ns % KST2;
          if (mbar_test_wait(ST_FULL0 + 8 * st, (uint32_t)(ns / KST2) & 1u) &&
              mbar_test_wait(S_EMPTY0 + 8 * s, ((uint32_t)(ns >> 1) & 1u) ^ 1u)) {
            tc_fence_after();
            const uint32_t stg = sSt0 + st * QSTAGE;
            const uint32_t dS = tmem + (uint32_t)(s * QBK), dP = tmem + 128u + (uint32_t)(s * QBK);
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
              const uint64_t ak = smem_desc_sw128(sK + kc * CHUNK);
              const uint64_t av = smem_desc_sw128(sV + kc * CHUNK);
              const uint64_t bq = smem_desc_sw128(stg + kc * Q_CHUNK);
              const uint64_t bo = smem_desc_sw128(stg + Q_TILE + kc * Q_CHUNK);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                mma_bf16(dS, ak + 2ull * k, bq + 2ull * k, idesc_s, (kc | k) != 0 ? 1u : 0u);
                mma_bf16(dP, av + 2ull * k, bo + 2ull * k, idesc_s, (kc | k) != 0 ? 1u : 0u);
              }
            }
            mma_commit(S_FULL0 + 8 * s);
            ++ns;
            progressed = true;
          }
        }
        if (nd < ns) {
          const int s = nd & 1, st = nd % KST2;
          if (mbar_test_wait(P_FULL0 + 8 * s, (uint32_t)(nd >> 1) & 1u)) {
            tc_fence_after();
            const uint32_t stg = sSt0 + st * QSTAGE;
            const uint32_t tp = tmem + (uint32_t)(s * QBK);
            const uint32_t tds = tmem + 128u + (uint32_t)(s * QBK);
            // Q and dO [64 queries, 128 head dims]: 64-dim atoms one chunk apart, 16
            // queries (2 KB) per MMA
            const uint64_t bq = smem_desc_sw128_mn(stg, Q_CHUNK);
            const uint64_t bo = smem_desc_sw128_mn(stg + Q_TILE, Q_CHUNK);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              mma_bf16_tmem_a(tDV, tp + (uint32_t)(8 * k), bo + 128ull * k, idesc_o,
                              (nd | k) != 0 ? 1u : 0u);
              mma_bf16_tmem_a(tDK, tds + (uint32_t)(8 * k), bq + 128ull * k, idesc_o,
                              (nd | k) != 0 ? 1u : 0u);
            }
            mma_commit(P_EMPTY0 + 8 * s);
            mma_commit(ST_EMPTY0 + 8 * st);
            ++nd;
            progressed = true;
          }
        }
        if (progressed) {
          t0 = global_timer_ns();
          spins = 0;
          continue;
        }
        if ((++spins & 255u) == 0u) {
          if (*abort_flag) break;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            report_status(a.status, XMOD_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
      }
    }
  } else {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int key = k0 + row;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    bool ok = true;
    for (int it = 0; it < items; ++it) {
      const int s = it & 1;
      const int h = g * G + it / nqb, q0 = (qb0 + it % nqb) * QBK;
      // this query block's lse and D (per head, queries contiguous; entries past n are
      // never used: their probabilities are masked to 0)
      const float* lrow = a.lseT + (int64_t)(b * a.hq + h) * a.ldS + q0;
      const float* drow = a.DdT + (int64_t)(b * a.hq + h) * a.ldS + q0;
      const int32_t* prow_q = a.qposS ? a.qposS + (int64_t)b * a.ldS + q0 : nullptr;
      if (!mbar_wait(S_FULL0 + 8 * s, (uint32_t)(it >> 1) & 1u, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[QBK], dp[QBK];
      const uint32_t srow = tmem + lane_off + (uint32_t)(s * QBK);
      const uint32_t prow = tmem + lane_off + 128u + (uint32_t)(s * QBK);
      tmem_ld32(srow, *reinterpret_cast<float(*)[32]>(sv));
      tmem_ld32(srow + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
      tmem_ld32(prow, *reinterpret_cast<float(*)[32]>(dp));
      tmem_ld32(prow + 32, *reinterpret_cast<float(*)[32]>(dp + 32));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(S_EMPTY0 + 8 * s);
      float pp[32], pd[32];
#pragma unroll
      for (int c4 = 0; c4 < QBK; c4 += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lrow + c4);
        const float4 d4 = *reinterpret_cast<const float4*>(drow + c4);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
        int qpv[4];   // the queries' positions, -1 past n
        if (prow_q) {
          const int4 p4 = *reinterpret_cast<const int4*>(prow_q + c4);
          qpv[0] = p4.x; qpv[1] = p4.y; qpv[2] = p4.z; qpv[3] = p4.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) qpv[e] = q0 + c4 + e < a.n ? q0 + c4 + e : -1;
        }
        float pv[4], dsv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool okp = key < a.nk && key <= qpv[e];
          const float p = okp ? ex2f(fmaf(sv[c4 + e], a.scale_log2, -lv[e])) : 0.f;
          pv[e] = p;
          dsv[e] = okp ? p * (dp[c4 + e] - dv[e]) : 0.f;
        }
        pp[c4 / 2] = __uint_as_float(pack_bf16x2(pv[0], pv[1]));
        pp[c4 / 2 + 1] = __uint_as_float(pack_bf16x2(pv[2], pv[3]));
        pd[c4 / 2] = __uint_as_float(pack_bf16x2(dsv[0], dsv[1]));
        pd[c4 / 2 + 1] = __uint_as_float(pack_bf16x2(dsv[2], dsv[3]));
      }
      // P^T and dS^T over the first halves of their buffers (read above; what the
      // buffers held two items ago was consumed by then)
      tmem_st32(srow, pp);
      tmem_st32(prow, pd);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(P_FULL0 + 8 * s);
    }
    if (items == 0) {   // no query sees these keys: their gradients are zero
      ok = false;
      if (key < a.nk) {
        const int64_t orow = ((int64_t)b * a.nk + key) * a.ldgk + g * HD;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 4
        for (int e = 0; e < HD; e += 8) {
          *reinterpret_cast<uint4*>(a.dk + orow + e) = z;
          *reinterpret_cast<uint4*>(a.dv + orow + e) = z;
        }
      }
    }
    if (ok) {
      const int il = items - 1;
      ok = mbar_wait(P_EMPTY0 + 8 * (il & 1), (uint32_t)(il >> 1) & 1u, abort_flag, a.status);
    }
    if (ok) {
      tc_fence_after();
      const int64_t orow = ((int64_t)b * a.nk + key) * a.ldgk + g * HD;
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {   // dK (scaled), then dV
        const uint32_t src = (part == 0 ? tDK : tDV) + lane_off;
        const float sc = part == 0 ? a.scale : 1.0f;
        __nv_bfloat16* dst = (part == 0 ? a.dk : a.dv) + orow;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float v[32];
          tmem_ld32(src + c * 32, v);
          tmem_ld_wait();
          if (key < a.nk) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 q;
              q.x = pack_bf16x2(v[e] * sc, v[e + 1] * sc);
              q.y = pack_bf16x2(v[e + 2] * sc, v[e + 3] * sc);
              q.z = pack_bf16x2(v[e + 4] * sc, v[e + 5] * sc);
              q.w = pack_bf16x2(v[e + 6] * sc, v[e + 7] * sc);
              *reinterpret_cast<uint4*>(dst + c * 32 + e) = q;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 20000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

bool attn_bwd_dq_tc_supported(int hd, int ldq, int qw) {
  return hd == HD && ldq % 8 == 0 && qw % 8 == 0 && tma_available();
}

cudaError_t launch_attn_bwd_dq_tc_kv(const Ctx& c, int B, int n, int nk, const int32_t* qpos,
                                     int hq, int hkv, const void* q, int ldq, const void* kv,
                                     int ldk, int k_col0, int v_col0, const void* o,
                                     const void* dO, const float* lse, float* Dd, void* dq,
                                     int ldg, float* DdT, int ldS) {
  if (B <= 0 || n <= 0) return cudaSuccess;
  const int qw = hq * HD;
  if (!attn_bwd_dq_tc_supported(HD, ldq, qw) || ldk % 8 || ldg % 8 || nk <= 0 ||
      (!qpos && nk != n))
    return cudaErrorInvalidValue;
  CUtensorMap mQ, mDO, mK;
  {
    const int64_t dims[3] = {ldq, n, B};
    const int64_t strides[2] = {(int64_t)ldq * 2, (int64_t)n * ldq * 2};
    const int qbox[3] = {64, QB, 1};
    if (!tma_map_bf16(&mQ, q, 3, dims, strides, qbox)) return cudaErrorInvalidValue;
  }
  {
    const int64_t dims[3] = {ldk, nk, B};
    const int64_t strides[2] = {(int64_t)ldk * 2, (int64_t)nk * ldk * 2};
    const int kbox[3] = {64, KB, 1};
    if (!tma_map_bf16(&mK, kv, 3, dims, strides, kbox)) return cudaErrorInvalidValue;
  }
  {
    const int64_t dims[3] = {qw, n, B};
    const int64_t strides[2] = {(int64_t)qw * 2, (int64_t)n * qw * 2};
    const int box[3] = {64, QB, 1};
    if (!tma_map_bf16(&mDO, dO, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  DqArgs a;
  a.n = n;
  a.hq = hq;
  a.hkv = hkv;
  a.nqb = (n + QB - 1) / QB;
  a.nk = nk;
  a.qpos = qpos;
  a.k_col0 = k_col0;
  a.v_col0 = v_col0;
  a.qw = qw;
  a.scale = 1.0f / sqrtf((float)HD);
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  a.lse = lse;
  a.o = (const __nv_bfloat16*)o;
  a.dO = (const __nv_bfloat16*)dO;
  a.Dd = Dd;
  a.DdT = DdT;
  a.ldS = ldS;
  a.dq = (__nv_bfloat16*)dq;
  a.ldg = ldg;
  a.status = c.status;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(attn_bwd_dq_tc_kernel, dim3(hq, B, a.nqb), dim3(THREADS), SMEM, c.stream,
                    mQ, mDO, mK, a);
}

cudaError_t launch_attn_bwd_dq_tc(const Ctx& c, int B, int n, int hq, int hkv, const void* qkv,
                                  int ldq, const void* o, const void* dO, const float* lse,
                                  float* Dd, void* dqkv, int ldg, float* DdT, int ldS) {
  const int qw = hq * HD, kw = hkv * HD;
  return launch_attn_bwd_dq_tc_kv(c, B, n, n, nullptr, hq, hkv, qkv, ldq, qkv, ldq, qw, qw + kw,
                                  o, dO, lse, Dd, dqkv, ldg, DdT, ldS);
}

cudaError_t launch_attn_bwd_dkv_tc_kv(const Ctx& c, int B, int n, int nk, const int32_t* qposS,
                                      const int32_t* qstart, int hq, int hkv, const void* q,
                                      int ldq, const void* kv, int ldk, int k_col0, int v_col0,
                                      const void* dO, const float* lseT, const float* DdT,
                                      int ldS, void* dk, void* dv, int ldgk) {
  if (B <= 0 || n <= 0 || nk <= 0) return cudaSuccess;
  const int qw = hq * HD;
  if (ldq % 8 || ldk % 8 || ldgk % 8 || ldS % QBK || ldS < n || hq % hkv ||
      !tma_available() || (!qposS) != (!qstart) || (!qposS && nk != n))
    return cudaErrorInvalidValue;
  CUtensorMap mKV, mQ, mDO;
  {
    const int64_t dims[3] = {ldk, nk, B};
    const int64_t strides[2] = {(int64_t)ldk * 2, (int64_t)nk * ldk * 2};
    const int kvbox[3] = {64, KVB, 1};
    if (!tma_map_bf16(&mKV, kv, 3, dims, strides, kvbox)) return cudaErrorInvalidValue;
  }
  {
    const int64_t dims[3] = {ldq, n, B};
    const int64_t strides[2] = {(int64_t)ldq * 2, (int64_t)n * ldq * 2};
    const int qbox[3] = {64, QBK, 1};
    if (!tma_map_bf16(&mQ, q, 3, dims, strides, qbox)) return cudaErrorInvalidValue;
  }
  {
    const int64_t dims[3] = {qw, n, B};
    const int64_t strides[2] = {(int64_t)qw * 2, (int64_t)n * qw * 2};
    const int box[3] = {64, QBK, 1};
    if (!tma_map_bf16(&mDO, dO, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  DkvArgs a;
  a.n = n;
  a.hq = hq;
  a.hkv = hkv;
  a.nk = nk;
  a.k_col0 = k_col0;
  a.v_col0 = v_col0;
  a.qposS = qposS;
  a.qstart = qstart;
  a.scale = 1.0f / sqrtf((float)HD);
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  a.lseT = lseT;
  a.DdT = DdT;
  a.ldS = ldS;
  a.dk = (__nv_bfloat16*)dk;
  a.dv = (__nv_bfloat16*)dv;
  a.ldgk = ldgk;
  a.status = c.status;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkv_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, KV_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_pdl(attn_bwd_dkv_tc_kernel, dim3(hkv, B, (nk + KVB - 1) / KVB), dim3(THREADS),
                    KV_SMEM, c.stream, mKV, mQ, mDO, a);
}

cudaError_t launch_attn_bwd_dkv_tc(const Ctx& c, int B, int n, int hq, int hkv, const void* qkv,
                                   int ldq, const void* dO, const float* lseT, const float* DdT,
                                   int ldS, void* dqkv, int ldg) {
  const int qw = hq * HD, kw = hkv * HD;
  __nv_bfloat16* g = (__nv_bfloat16*)dqkv;
  return launch_attn_bwd_dkv_tc_kv(c, B, n, n, nullptr, nullptr, hq, hkv, qkv, ldq, qkv, ldq, qw,
                                   qw + kw, dO, lseT, DdT, ldS, g + qw, g + qw + kw, ldg);
}

}  // namespace xmod
