// Tensor-core causal GQA attention for sm_103a (tcgen05 + TMEM + TMA), bf16,
// head_dim 128, fp32 softmax statistics.
//
// Attention runs among the n tokens of one sequence -- the selected tokens of a
// sparse layer (X-MoD notes, section "mechanism controls": attention within the
// selected subset) or all tokens of a dense layer. Compact order equals position
// order, so the causal mask over compact indices is the causal mask over
// positions. Query head h reads key/value head h / (hq / hkv).
//
// One CTA per (128-query block, query head, sequence):
//   warp 0      TMA: the Q tile once, then K_j and V_j^T for each 128-key block j
//               into a two-stage ring
//   warp 1      TMEM owner; one lane issues S_j = Q K_j^T into one of two TMEM
//               S buffers (S_{j+1} is issued before P_j V_j so the tensor core works
//               on the next scores while the softmax runs), then P_j V_j^T
//   warps 2..5  softmax, one query row per thread (a TMEM lane is a row, so row
//               max and row sum are thread-local): online max in log2 units,
//               P_j = exp2(s*scale - m) written as bf16 into shared memory in the
//               swizzled K-major layout the MMA reads, and O = O*alpha + P_j V_j
//               accumulated in registers.
// V arrives transposed ([hd, keys], keys contiguous), written that way by the
// q/k/v projection's epilogue, so both MMAs read K-major operands.

#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"
#include "tc_common.cuh"

namespace xmod {

namespace {

using namespace tc;

constexpr int QB = 128;     // query rows per CTA
constexpr int KB = 128;     // keys per block
constexpr int HD = 128;     // head dim
constexpr int THREADS = 192;
constexpr int CHUNK = 128 * 128;        // bytes of a 128 x 64 bf16 swizzled chunk
constexpr int TILE = 2 * CHUNK;         // a 128 x 128 bf16 tile
constexpr int SMEM = 6 * TILE + 1024 + 256;

struct AttnArgs {
  int n, hq, hkv, nqb;
  int qw;                 // column of k head 0 inside a q|k|v row
  float scale_log2;       // log2(e) / sqrt(hd)
  __nv_bfloat16* o;
  int ldo;
  int* status;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmQK, const __grid_constant__ CUtensorMap tmVt,
                    const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sP = base + TILE;
  const uint32_t sK0 = base + 2 * TILE;   // K stages at sK0 + s * TILE
  const uint32_t sV0 = base + 4 * TILE;   // V^T stages at sV0 + s * TILE
  const uint32_t sBar = base + 6 * TILE;
  // barriers
  const uint32_t Q_FULL = sBar + 0;
  const uint32_t KV_FULL0 = sBar + 8, KV_EMPTY0 = sBar + 24;
  const uint32_t S_FULL0 = sBar + 40, S_EMPTY0 = sBar + 56;
  const uint32_t P_FULL = sBar + 72, P_EMPTY = sBar + 80;
  const uint32_t PV_FULL = sBar + 88, PV_EMPTY = sBar + 96;
  const uint32_t sTmem = sBar + 112;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (sTmem - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (sTmem - base) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = a.nqb - 1 - (int)blockIdx.x;   // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (a.hq / a.hkv);
  const int q0 = qb * QB;
  const int last_q = min(q0 + QB, a.n) - 1;
  const int nkb = last_q / KB + 1;

  if (threadIdx.x == 0) {
    mbar_init(Q_FULL, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(KV_FULL0 + 8 * s, 1);
      mbar_init(KV_EMPTY0 + 8 * s, 1);
      mbar_init(S_FULL0 + 8 * s, 1);
      mbar_init(S_EMPTY0 + 8 * s, 128);
    }
    mbar_init(P_FULL, 128);
    mbar_init(P_EMPTY, 1);
    mbar_init(PV_FULL, 1);
    mbar_init(PV_EMPTY, 128);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmQK);
    prefetch_tensormap(&tmVt);
  }
  if (warp == 1) tmem_alloc(sTmem, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;   // S0: cols 0..127, S1: 128..255, PV: 256..383

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(Q_FULL, TILE);
      tma_load_3d(sQ, &tmQK, Q_FULL, h * HD, q0, b);
      tma_load_3d(sQ + CHUNK, &tmQK, Q_FULL, h * HD + 64, q0, b);
      const int vt_row = (b * a.hkv + g) * HD;
      for (int j = 0; j < nkb; ++j) {
        const int s = j & 1;
        const uint32_t ph = (uint32_t)(j >> 1) & 1u;
        if (!mbar_wait(KV_EMPTY0 + 8 * s, ph ^ 1u, abort_flag, a.status)) break;
        mbar_arrive_expect_tx(KV_FULL0 + 8 * s, 2 * TILE);
        const uint32_t kdst = sK0 + s * TILE, vdst = sV0 + s * TILE;
        tma_load_3d(kdst, &tmQK, KV_FULL0 + 8 * s, a.qw + g * HD, j * KB, b);
        tma_load_3d(kdst + CHUNK, &tmQK, KV_FULL0 + 8 * s, a.qw + g * HD + 64, j * KB, b);
        tma_load_2d(vdst, &tmVt, KV_FULL0 + 8 * s, j * KB, vt_row);
        tma_load_2d(vdst + CHUNK, &tmVt, KV_FULL0 + 8 * s, j * KB + 64, vt_row);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      bool ok = mbar_wait(Q_FULL, 0, abort_flag, a.status);
      auto issue_s = [&](int j) -> bool {
        const int s = j & 1;
        const uint32_t ph = (uint32_t)(j >> 1) & 1u;
        if (!mbar_wait(KV_FULL0 + 8 * s, ph, abort_flag, a.status)) return false;
        if (!mbar_wait(S_EMPTY0 + 8 * s, ph ^ 1u, abort_flag, a.status)) return false;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(s * 128);
#pragma unroll
        for (int kc = 0; kc < 2; ++kc) {
          const uint64_t ad = smem_desc_sw128(sQ + kc * CHUNK);
          const uint64_t bd = smem_desc_sw128(sK0 + s * TILE + kc * CHUNK);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(d, ad + 2ull * k, bd + 2ull * k, idesc, (kc | k) != 0 ? 1u : 0u);
        }
        mma_commit(S_FULL0 + 8 * s);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nkb; ++j) {
        if (j + 1 < nkb && !issue_s(j + 1)) break;
        const uint32_t pj = (uint32_t)j & 1u;
        if (!mbar_wait(P_FULL, pj, abort_flag, a.status)) break;
        if (!mbar_wait(PV_EMPTY, pj ^ 1u, abort_flag, a.status)) break;
        tc_fence_after();
        const int s = j & 1;
#pragma unroll
        for (int kc = 0; kc < 2; ++kc) {
          const uint64_t ad = smem_desc_sw128(sP + kc * CHUNK);
          const uint64_t bd = smem_desc_sw128(sV0 + s * TILE + kc * CHUNK);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16(tmem + 256u, ad + 2ull * k, bd + 2ull * k, idesc, (kc | k) != 0 ? 1u : 0u);
        }
        mma_commit(PV_FULL);
        mma_commit(P_EMPTY);
        mma_commit(KV_EMPTY0 + 8 * s);
      }
    }
  } else {
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int qi = q0 + row;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    float o[HD];
#pragma unroll
    for (int i = 0; i < HD; ++i) o[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    const uint32_t prow = sP + (uint32_t)row * 128u;
    const uint32_t sw = (uint32_t)(row & 7);
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      if (!mbar_wait(S_FULL0 + 8 * s, ph, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t srow = tmem + lane_off + (uint32_t)(s * 128);
      const int key0 = j * KB;
      // pass 1: row max of the unmasked scores
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(srow + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (key0 + c * 32 + i <= qi) mx = fmaxf(mx, v[i]);
      }
      const float m_new = fmaxf(m, mx * a.scale_log2);
      const float alpha = exp2f(m - m_new);
      // pass 2: probabilities into the shared-memory P tile (after P_{j-1} was consumed)
      if (!mbar_wait(P_EMPTY, ((uint32_t)j & 1u) ^ 1u, abort_flag, a.status)) {
        ok = false;
        break;
      }
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(srow + c * 32, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = (key0 + c * 32 + i <= qi) ? exp2f(v[i] * a.scale_log2 - m_new) : 0.f;
          const float p1 =
              (key0 + c * 32 + i + 1 <= qi) ? exp2f(v[i + 1] * a.scale_log2 - m_new) : 0.f;
          sum += p0 + p1;
          pk[i / 2] = pack_bf16x2(p0, p1);
        }
        const uint32_t chunk = prow + (uint32_t)(c >> 1) * CHUNK;
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const uint32_t unit = (uint32_t)((c & 1) * 4 + u4);
          st_shared_v4(chunk + ((unit ^ sw) << 4), pk[4 * u4], pk[4 * u4 + 1], pk[4 * u4 + 2],
                       pk[4 * u4 + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(S_EMPTY0 + 8 * s);
      mbar_arrive(P_FULL);
      l = l * alpha + sum;
      m = m_new;
      // O = O * alpha + P_j V_j
      if (!mbar_wait(PV_FULL, (uint32_t)j & 1u, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(tmem + lane_off + 256u + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c * 32 + i] = fmaf(o[c * 32 + i], alpha, v[i]);
      }
      tc_fence_before();
      mbar_arrive(PV_EMPTY);
    }
    if (ok && qi < a.n) {
      const float inv = 1.0f / l;
      __nv_bfloat16* dst = a.o + ((int64_t)b * a.n + qi) * a.ldo + h * HD;
#pragma unroll
      for (int c = 0; c < HD; c += 8) {
        uint4 q;
        q.x = pack_bf16x2(o[c] * inv, o[c + 1] * inv);
        q.y = pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv);
        q.z = pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv);
        q.w = pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv);
        *reinterpret_cast<uint4*>(dst + c) = q;
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 20000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool attention_tc_supported(int hd, int n, int ldq) {
  return hd == HD && n > 0 && ldq % 8 == 0 && tma_available();
}

cudaError_t launch_attention_tc(const Ctx& c, int B, int n, int hq, int hkv, const void* qkv,
                                int ldq, const void* vt, int vt_ld, void* o) {
  if (B <= 0 || n <= 0) return cudaSuccess;
  CUtensorMap mQK, mVt;
  {
    const int64_t dims[3] = {ldq, n, B};
    const int64_t strides[2] = {(int64_t)ldq * 2, (int64_t)n * ldq * 2};
    const int box[3] = {64, QB, 1};
    if (!tma_map_bf16(&mQK, qkv, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const int64_t dims[2] = {n, (int64_t)B * hkv * HD};
    const int64_t strides[1] = {(int64_t)vt_ld * 2};
    const int box[2] = {64, HD};
    if (!tma_map_bf16(&mVt, vt, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  AttnArgs a;
  a.n = n;
  a.hq = hq;
  a.hkv = hkv;
  a.nqb = (n + QB - 1) / QB;
  a.qw = hq * HD;
  a.scale_log2 = 1.4426950408889634f / sqrtf((float)HD);
  a.o = (__nv_bfloat16*)o;
  a.ldo = hq * HD;
  a.status = c.status;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(a.nqb, hq, B);
  attention_tc_kernel<<<grid, THREADS, SMEM, c.stream>>>(mQK, mVt, a);
  return cudaGetLastError();
}

}  // namespace xmod
