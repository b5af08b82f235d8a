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
//   warp 0      TMA: the Q tile once, then K_j and V_j^T of each key block j, each
//               into its own two-stage ring (a K stage comes free when S_j has been
//               computed, a V stage when P_j V_j has), whichever has a free stage first
//   warp 1      TMEM owner; one lane issues S_j = Q K_j^T into one of two TMEM S
//               buffers and O += P_j V_j (output accumulator O resident in TMEM), each
//               as soon as its inputs are ready, so S_{j+1} overlaps the softmax of S_j
//   warps 2..5  softmax, one query row per thread (a TMEM lane is a row, so row max
//               and row sum are thread-local), in one pass over the scores held in
//               registers: P_j = exp2(s*scale - m) is written as bf16 into one of two
//               shared-memory P buffers in the swizzled K-major layout the MMA reads.
//               The running max m only moves when a row's max grows by more than 2^8
//               (P then stays below 256); when it moves, the row of O in TMEM is
//               rescaled once P_{j-1} V_{j-1} has landed.
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
constexpr int HD = 128;     // head dim
constexpr int THREADS = 192;
constexpr int CHUNK = 128 * 128;        // bytes of a 128-row x 64-column bf16 swizzled chunk
constexpr int QTILE = 2 * CHUNK;        // the Q tile, 128 x 128
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// KB keys per block; PBUF shared-memory P buffers. <128, 2> suits long sequences
// (one CTA per SM); <64, 1> needs half the shared memory and TMEM so that two CTAs
// share an SM and hide each other's load and set-up latency (short sequences).
template <int KB, int PBUF>
struct AttnCfg {
  static constexpr int K_CHUNK = KB * 128;          // KB rows x 64 head dims
  static constexpr int K_STAGE = 2 * K_CHUNK;       // KB x 128 head dims
  static constexpr int V_STAGE = (KB / 64) * CHUNK; // 128 head dims x KB keys
  static constexpr int P_BYTES = (KB / 64) * CHUNK; // 128 rows x KB keys
  static constexpr int TMEM_COLS = 2 * KB + 128 <= 256 ? 256 : 512;
  static constexpr int DATA = QTILE + PBUF * P_BYTES + 2 * K_STAGE + 2 * V_STAGE;
  // 1024 bytes cover both the alignment of the tiles and the 256-byte barrier
  // block: the barriers sit in the alignment gap when it is at least 256 bytes,
  // else after the tiles (then the gap is under 256 bytes).
  static constexpr int SMEM = DATA + 1024;
  // two CTAs fit in the 228 KB of an SM (each also takes 1 KB reserved by the system)
  static constexpr int MIN_BLOCKS = 2 * (SMEM + 1024) <= 228 * 1024 ? 2 : 1;
};

struct AttnArgs {
  int n, hq, hkv, nqb;
  int qw;                 // column of k head 0 inside a q|k|v row
  float scale_log2;       // log2(e) / sqrt(hd)
  __nv_bfloat16* o;
  int ldo;
  int* status;
  // Variable tokens per sequence (threshold routing): sequence b has seq_count[b]
  // (<= n) rows starting at compact row seq_off[b]; the Q and K maps are then 2-D over
  // the compact rows. NULL: every sequence has n rows at b * n.
  const int32_t* seq_count;
  const int32_t* seq_off;
  // Selected-Q / full-KV: query row q of sequence b sits at position qpos[b * n + q]
  // (ascending in q) and attends to the keys at positions <= it among nkv keys per
  // sequence, read from a separate K map (columns from k_col0). qpos NULL: the keys
  // are the n query rows themselves (causal among them), nkv = n.
  const int32_t* qpos;
  int nkv;
  int k_col0;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 2^x by the PTX ex2.approx instruction: its error is far below the bf16 rounding the
// probabilities get right after. Inputs are <= 0 here; -inf gives 0.
#ifndef XMOD_ATTN_EX2_APPROX
#define XMOD_ATTN_EX2_APPROX 1
#endif
__device__ __forceinline__ float exp2_p(float x) {
#if XMOD_ATTN_EX2_APPROX
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
#else
  return exp2f(x);
#endif
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int KB, int PBUF>
__global__ void __launch_bounds__(THREADS, (AttnCfg<KB, PBUF>::MIN_BLOCKS))
attention_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmVt, const AttnArgs a) {
  using C = AttnCfg<KB, PBUF>;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sP0 = sQ + QTILE;                    // P buffers at sP0 + b * P_BYTES
  const uint32_t sK0 = sP0 + PBUF * C::P_BYTES;       // K stages at sK0 + s * K_STAGE
  const uint32_t sV0 = sK0 + 2 * C::K_STAGE;          // V^T stages at sV0 + s * V_STAGE
  const uint32_t sBar = (base - raw >= 256u) ? raw : base + (uint32_t)C::DATA;
  // K_j and V_j^T have separate stages and barriers: a K stage is free again once
  // S_j = Q K_j^T has completed, a V stage once P_j V_j has, so K loads run ahead of
  // the P V MMAs instead of waiting for them.
  const uint32_t Q_FULL = sBar + 0;
  const uint32_t K_FULL0 = sBar + 8, K_EMPTY0 = sBar + 24;
  const uint32_t S_FULL0 = sBar + 40, S_EMPTY0 = sBar + 56;
  const uint32_t P_FULL0 = sBar + 72, P_EMPTY0 = sBar + 88;
  const uint32_t V_FULL0 = sBar + 104, V_EMPTY0 = sBar + 120;
  const uint32_t sTmem = sBar + 144;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + (sTmem - raw));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + (sTmem - raw) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = a.nqb - 1 - (int)blockIdx.x;   // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (a.hq / a.hkv);
  const int q0 = qb * QB;

  if (threadIdx.x == 0) {
    mbar_init(Q_FULL, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(K_FULL0 + 8 * s, 1);
      mbar_init(K_EMPTY0 + 8 * s, 1);
      mbar_init(V_FULL0 + 8 * s, 1);
      mbar_init(V_EMPTY0 + 8 * s, 1);
      mbar_init(S_FULL0 + 8 * s, 1);
      mbar_init(S_EMPTY0 + 8 * s, 128);
    }
    for (int pb = 0; pb < PBUF; ++pb) {
      mbar_init(P_FULL0 + 8 * pb, 128);
      mbar_init(P_EMPTY0 + 8 * pb, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmVt);
  }
  if (warp == 1) tmem_alloc(sTmem, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;   // S0: cols [0, KB), S1: [KB, 2KB), O: [2KB, 2KB+128)
  const uint32_t tO = tmem + 2u * KB;
  pdl_wait();  // everything above overlapped the previous kernel's tail
  int n_b = a.n;
  int64_t row0 = (int64_t)b * a.n;   // compact row of the sequence's first token
  if (a.seq_count) {
    n_b = min(max(a.seq_count[b], 0), a.n);
    row0 = a.seq_off[b];
  }
  const int last_q = min(q0 + QB, n_b) - 1;
  // last key position any row of the block may see
  const int last_key = a.qpos && q0 < n_b ? a.qpos[(int64_t)b * a.n + last_q] : last_q;
  const int nkb = q0 < n_b ? last_key / KB + 1 : 0;   // 0: this query block is empty

  if (warp == 0) {
    if (lane == 0 && nkb > 0) {
      mbar_arrive_expect_tx(Q_FULL, QTILE);
      if (a.seq_count) {
        tma_load_2d(sQ, &tmQ, Q_FULL, h * HD, (int)(row0 + q0));
        tma_load_2d(sQ + CHUNK, &tmQ, Q_FULL, h * HD + 64, (int)(row0 + q0));
      } else {
        tma_load_3d(sQ, &tmQ, Q_FULL, h * HD, q0, b);
        tma_load_3d(sQ + CHUNK, &tmQ, Q_FULL, h * HD + 64, q0, b);
      }
      const int vt_row = (b * a.hkv + g) * HD;
      // issue whichever of the next K block and the next V block has a free stage
      int jk = 0, jv = 0;
      uint64_t t0 = global_timer_ns();
      uint32_t spins = 0;
      while (jv < nkb) {
        bool progressed = false;
        if (jk < nkb) {
          const int s = jk & 1;
          if (mbar_try_wait(K_EMPTY0 + 8 * s, ((uint32_t)(jk >> 1) & 1u) ^ 1u)) {
            mbar_arrive_expect_tx(K_FULL0 + 8 * s, C::K_STAGE);
            const uint32_t kdst = sK0 + s * C::K_STAGE;
            if (a.seq_count) {
              tma_load_2d(kdst, &tmK, K_FULL0 + 8 * s, a.k_col0 + g * HD, (int)(row0 + jk * KB));
              tma_load_2d(kdst + C::K_CHUNK, &tmK, K_FULL0 + 8 * s, a.k_col0 + g * HD + 64,
                          (int)(row0 + jk * KB));
            } else {
              tma_load_3d(kdst, &tmK, K_FULL0 + 8 * s, a.k_col0 + g * HD, jk * KB, b);
              tma_load_3d(kdst + C::K_CHUNK, &tmK, K_FULL0 + 8 * s, a.k_col0 + g * HD + 64,
                          jk * KB, b);
            }
            ++jk;
            progressed = true;
          }
        }
        if (jv < jk) {
          const int s = jv & 1;
          if (mbar_try_wait(V_EMPTY0 + 8 * s, ((uint32_t)(jv >> 1) & 1u) ^ 1u)) {
            mbar_arrive_expect_tx(V_FULL0 + 8 * s, C::V_STAGE);
            const uint32_t vdst = sV0 + s * C::V_STAGE;
#pragma unroll
            for (int kc = 0; kc < KB / 64; ++kc)
              tma_load_2d(vdst + kc * CHUNK, &tmVt, V_FULL0 + 8 * s, jv * KB + 64 * kc, vt_row);
            ++jv;
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
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, KB);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, HD);
      bool ok = nkb > 0 && mbar_wait(Q_FULL, 0, abort_flag, a.status);
      // Issue S_j = Q K_j^T and O += P_j V_j in whatever order their inputs arrive:
      // S_{j+1} as soon as K_{j+1} is resident (so it overlaps the softmax of S_j),
      // P_j V_j as soon as the softmax has written P_j -- never one waiting behind the
      // other's input.
      int ns = 0, npv = 0;
      uint64_t t0 = global_timer_ns();
      uint32_t spins = 0;
      while (ok && npv < nkb) {
        bool progressed = false;
        if (ns < nkb && ns <= npv + 1) {
          const int s = ns & 1;
          const uint32_t ph = (uint32_t)(ns >> 1) & 1u;
          if (mbar_try_wait(K_FULL0 + 8 * s, ph) && mbar_try_wait(S_EMPTY0 + 8 * s, ph ^ 1u)) {
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(s * KB);
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
              const uint64_t ad = smem_desc_sw128(sQ + kc * CHUNK);
              const uint64_t bd = smem_desc_sw128(sK0 + s * C::K_STAGE + kc * C::K_CHUNK);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16(d, ad + 2ull * k, bd + 2ull * k, idesc_s, (kc | k) != 0 ? 1u : 0u);
            }
            mma_commit(S_FULL0 + 8 * s);
            mma_commit(K_EMPTY0 + 8 * s);
            ++ns;
            progressed = true;
          }
        }
        if (npv < ns) {
          const int s = npv & 1;                         // V stage
          const int pb = npv % PBUF;                     // P buffer
          const uint32_t pph = (uint32_t)(npv / PBUF) & 1u;
          if (mbar_try_wait(P_FULL0 + 8 * pb, pph) &&
              mbar_try_wait(V_FULL0 + 8 * s, (uint32_t)(npv >> 1) & 1u)) {
            tc_fence_after();
#pragma unroll
            for (int kc = 0; kc < KB / 64; ++kc) {
              const uint64_t ad = smem_desc_sw128(sP0 + pb * C::P_BYTES + kc * CHUNK);
              const uint64_t bd = smem_desc_sw128(sV0 + s * C::V_STAGE + kc * CHUNK);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16(tO, ad + 2ull * k, bd + 2ull * k, idesc_o,
                         (npv | kc | k) != 0 ? 1u : 0u);
            }
            mma_commit(P_EMPTY0 + 8 * pb);
            mma_commit(V_EMPTY0 + 8 * s);
            ++npv;
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
    const int qi = q0 + row;   // compact query row
    // position that bounds this row's keys, and the smallest one in the block (rows
    // past the sequence's end repeat its last position; their output is not stored)
    int qp = qi, qp_min = q0;
    if (a.qpos && nkb > 0) {
      const int64_t base_row = (int64_t)b * a.n;
      qp = a.qpos[base_row + min(qi, n_b - 1)];
      qp_min = a.qpos[base_row + q0];
    }
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t sw = (uint32_t)(row & 7);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int s = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      if (!mbar_wait(S_FULL0 + 8 * s, ph, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[KB];
      {
        const uint32_t srow = tmem + lane_off + (uint32_t)(s * KB);
#pragma unroll
        for (int c = 0; c < KB / 32; ++c)
          tmem_ld32(srow + c * 32, *reinterpret_cast<float(*)[32]>(v + c * 32));
        tmem_ld_wait();
      }
      tc_fence_before();
      mbar_arrive(S_EMPTY0 + 8 * s);
      const int key0 = j * KB;
      const bool diag = key0 + KB - 1 > qp_min;   // only blocks reaching past a row need the mask
      float mx = -INFINITY;
      if (diag) {
#pragma unroll
        for (int i = 0; i < KB; ++i) {
          if (key0 + i > qp) v[i] = -INFINITY;
          mx = fmaxf(mx, v[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < KB; ++i) mx = fmaxf(mx, v[i]);
      }
      const float m_cand = mx * a.scale_log2;
      const bool grow = m_cand > m + kRescaleThreshold;
      const float m_new = grow ? m_cand : m;
      const float alpha = grow ? exp2f(m - m_new) : 1.0f;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O holds P_0..j-1 V: wait until the last of those MMAs landed, then rescale.
        const int jp = j - 1;
        if (!mbar_wait(P_EMPTY0 + 8 * (jp % PBUF), (uint32_t)(jp / PBUF) & 1u, abort_flag,
                       a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          float ov[32];
          tmem_ld32(tO + lane_off + c * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] *= alpha;
          tmem_st32(tO + lane_off + c * 32, ov);
        }
        tmem_st_wait();
      }
      m = m_new;
      // this P buffer is free once P_{j-PBUF} V_{j-PBUF} has completed
      const int pb = j % PBUF;
      if (!mbar_wait(P_EMPTY0 + 8 * pb, ((uint32_t)(j / PBUF) & 1u) ^ 1u, abort_flag, a.status)) {
        ok = false;
        break;
      }
      const uint32_t prow = sP0 + pb * C::P_BYTES + (uint32_t)row * 128u;
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < KB / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = exp2_p(fmaf(v[c * 32 + i], a.scale_log2, -m));
          const float p1 = exp2_p(fmaf(v[c * 32 + i + 1], a.scale_log2, -m));
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
      l = l * alpha + sum;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(P_FULL0 + 8 * pb);
    }
    if (nkb == 0) ok = false;   // nothing was computed for this query block
    if (ok) {
      const int jl = nkb - 1;
      ok = mbar_wait(P_EMPTY0 + 8 * (jl % PBUF), (uint32_t)(jl / PBUF) & 1u, abort_flag, a.status);
    }
    if (ok) {
      tc_fence_after();
      const float inv = 1.0f / l;
      __nv_bfloat16* dst = a.o + (row0 + qi) * a.ldo + h * HD;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float ov[32];
        tmem_ld32(tO + lane_off + c * 32, ov);
        tmem_ld_wait();
        if (qi < n_b) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 q;
            q.x = pack_bf16x2(ov[e] * inv, ov[e + 1] * inv);
            q.y = pack_bf16x2(ov[e + 2] * inv, ov[e + 3] * inv);
            q.z = pack_bf16x2(ov[e + 4] * inv, ov[e + 5] * inv);
            q.w = pack_bf16x2(ov[e + 6] * inv, ov[e + 7] * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + e) = q;
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
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int KB, int PBUF>
cudaError_t launch_attention_cfg(const Ctx& c, int B, int n, int hq, const void* qkv, int ldq,
                                 const CUtensorMap& mVt, const AttnArgs& a, const AttnKv* kv) {
  using Cf = AttnCfg<KB, PBUF>;
  CUtensorMap mQ, mK;
  if (kv) {   // queries [B, n, ldq]; keys [B, nkv, ldk] from their own tensor
    const int64_t qdims[3] = {ldq, n, B};
    const int64_t qstrides[2] = {(int64_t)ldq * 2, (int64_t)n * ldq * 2};
    const int qbox[3] = {64, QB, 1};
    const int64_t kdims[3] = {kv->ldk, kv->nkv, B};
    const int64_t kstrides[2] = {(int64_t)kv->ldk * 2, (int64_t)kv->nkv * kv->ldk * 2};
    const int kbox[3] = {64, KB, 1};
    if (!tma_map_bf16(&mQ, qkv, 3, qdims, qstrides, qbox)) return cudaErrorInvalidValue;
    if (!tma_map_bf16(&mK, kv->k, 3, kdims, kstrides, kbox)) return cudaErrorInvalidValue;
  } else if (a.seq_count) {   // 2-D over the B * n compact rows
    const int64_t dims[2] = {ldq, (int64_t)B * n};
    const int64_t strides[1] = {(int64_t)ldq * 2};
    const int qbox[2] = {64, QB};
    const int kbox[2] = {64, KB};
    if (!tma_map_bf16(&mQ, qkv, 2, dims, strides, qbox)) return cudaErrorInvalidValue;
    if (!tma_map_bf16(&mK, qkv, 2, dims, strides, kbox)) return cudaErrorInvalidValue;
  } else {
    const int64_t dims[3] = {ldq, n, B};
    const int64_t strides[2] = {(int64_t)ldq * 2, (int64_t)n * ldq * 2};
    const int qbox[3] = {64, QB, 1};
    const int kbox[3] = {64, KB, 1};
    if (!tma_map_bf16(&mQ, qkv, 3, dims, strides, qbox)) return cudaErrorInvalidValue;
    if (!tma_map_bf16(&mK, qkv, 3, dims, strides, kbox)) return cudaErrorInvalidValue;
  }
  auto k = attention_tc_kernel<KB, PBUF>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(a.nqb, hq, B);
  return launch_pdl(k, grid, dim3(THREADS), Cf::SMEM, c.stream, mQ, mK, mVt, a);
}

}  // namespace

// A sequence of at most this many tokens is one 128-key block: it runs the
// <128, 2> configuration; longer ones the two-CTAs-per-SM <64, 1> configuration,
// which measured 7-15% faster from 256 to 16384 tokens (GB300, 12/4 and 16/4 heads).
#ifndef XMOD_ATTN_ONE_BLOCK_MAX_N
#define XMOD_ATTN_ONE_BLOCK_MAX_N 128
#endif

bool attention_tc_supported(int hd, int n, int ldq) {
  return hd == HD && n > 0 && ldq % 8 == 0 && tma_available();
}

cudaError_t launch_attention_tc(const Ctx& c, int B, int n, int hq, int hkv, const void* qkv,
                                int ldq, const void* vt, int vt_ld, void* o,
                                const int32_t* seq_count, const int32_t* seq_off,
                                const AttnKv* kv) {
  if (B <= 0 || n <= 0) return cudaSuccess;
  if (kv && (seq_count || !kv->qpos || kv->nkv <= 0 || kv->ldk % 8)) return cudaErrorInvalidValue;
  const int nkv = kv ? kv->nkv : n;
  CUtensorMap mVt;
  {
    const int64_t dims[2] = {nkv, (int64_t)B * hkv * HD};
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
  a.seq_count = seq_count;
  a.seq_off = seq_off;
  a.qpos = kv ? kv->qpos : nullptr;
  a.nkv = nkv;
  a.k_col0 = kv ? 0 : a.qw;
  if (nkv <= XMOD_ATTN_ONE_BLOCK_MAX_N)
    return launch_attention_cfg<128, 2>(c, B, n, hq, qkv, ldq, mVt, a, kv);
  return launch_attention_cfg<64, 1>(c, B, n, hq, qkv, ldq, mVt, a, kv);
}

}  // namespace xmod
