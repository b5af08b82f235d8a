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
//               registers: P_j = exp2(s*scale - m) goes back to TMEM as bf16 pairs, over
//               the first half of S_j's own columns, and the P V MMA reads its A operand
//               from there (no shared-memory P buffer; that space holds a third V stage).
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

// KB keys per block; KST K stages and VST V stages. <128, 3, 3> (one CTA per SM) serves
// sequences of one key block; <64, 3, 2> needs half the shared memory and TMEM so that
// two CTAs share an SM and hide each other's load and set-up latency.
template <int KB, int KST, int VST>
struct AttnCfg {
  static constexpr int K_CHUNK = KB * 128;          // KB rows x 64 head dims
  static constexpr int K_STAGE = 2 * K_CHUNK;       // KB x 128 head dims
  static constexpr int V_STAGE = (KB / 64) * CHUNK; // 128 head dims x KB keys
  static constexpr int TMEM_COLS = 2 * KB + 128 <= 256 ? 256 : 512;
  static constexpr int DATA = QTILE + KST * K_STAGE + VST * V_STAGE;
  // 1024 bytes cover both the alignment of the tiles and the 256-byte barrier
  // block: the barriers sit in the alignment gap when it is at least 256 bytes,
  // else after the tiles (then the gap is under 256 bytes).
  static constexpr int SMEM = DATA + 1024;
  // two CTAs fit in the 228 KB of an SM (each also takes 1 KB reserved by the system)
  static constexpr int MIN_BLOCKS = 2 * (SMEM + 1024) <= 228 * 1024 ? 2 : 1;
  // barriers: Q, K full/empty per stage, V full/empty per stage, S and P full/empty x2;
  // then the TMEM address and the abort flag
  static_assert((1 + 2 * KST + 2 * VST + 8) * 8 + 16 <= 256, "barrier block overflows");
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
  // optional: each row's log2-sum-exp2 of its scaled logits, [rows, hq] (the backward
  // recomputes P from it)
  float* lse;
};

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

// Blackwell's paired fp32 arithmetic (two lanes per instruction, each rounded as the
// scalar instruction would) and three-input max: the softmax warps share their
// schedulers with the warps that issue the MMAs and the TMA loads, so fewer softmax
// instructions leave those more issue slots.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <int KB, int KST, int VST>
__global__ void __launch_bounds__(THREADS, (AttnCfg<KB, KST, VST>::MIN_BLOCKS))
attention_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmVt, const AttnArgs a) {
  using C = AttnCfg<KB, KST, VST>;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK0 = sQ + QTILE;                    // K stages at sK0 + s * K_STAGE
  const uint32_t sV0 = sK0 + KST * C::K_STAGE;        // V^T stages at sV0 + s * V_STAGE
  const uint32_t sBar = (base - raw >= 256u) ? raw : base + (uint32_t)C::DATA;
  // K_j and V_j^T have separate stages and barriers: a K stage is free again once
  // S_j = Q K_j^T has completed, a V stage once P_j V_j has, so K loads run ahead of
  // the P V MMAs instead of waiting for them.
  // P_FULL(b): P_j is in TMEM buffer b = j & 1; P_EMPTY(b): P_j V_j has completed.
  const uint32_t Q_FULL = sBar + 0;
  const uint32_t K_FULL0 = sBar + 8, K_EMPTY0 = K_FULL0 + 8 * KST;
  const uint32_t V_FULL0 = K_EMPTY0 + 8 * KST, V_EMPTY0 = V_FULL0 + 8 * VST;
  const uint32_t S_FULL0 = V_EMPTY0 + 8 * VST, S_EMPTY0 = S_FULL0 + 16;
  const uint32_t P_FULL0 = S_EMPTY0 + 16, P_EMPTY0 = P_FULL0 + 16;
  const uint32_t sTmem = P_EMPTY0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + (sTmem - raw));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + (sTmem - raw) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTAs start in blockIdx order, x fastest: every (head, sequence) pair's last query
  // block (the most keys) first, then the next-to-last ones, ... (longest first)
  const int qb = a.nqb - 1 - (int)blockIdx.z;
  const int h = blockIdx.x, b = blockIdx.y;
  const int g = h / (a.hq / a.hkv);
  const int q0 = qb * QB;

  if (threadIdx.x == 0) {
    mbar_init(Q_FULL, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(K_FULL0 + 8 * s, 1);
      mbar_init(K_EMPTY0 + 8 * s, 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(V_FULL0 + 8 * s, 1);
      mbar_init(V_EMPTY0 + 8 * s, 1);
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
          const int s = jk % KST;
          if (mbar_test_wait(K_EMPTY0 + 8 * s, ((uint32_t)(jk / KST) & 1u) ^ 1u)) {
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
          const int s = jv % VST;
          if (mbar_test_wait(V_EMPTY0 + 8 * s, ((uint32_t)(jv / VST) & 1u) ^ 1u)) {
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
        // S_{j+2} overwrites buffer j & 1, which holds P_j: it is issued after P_j V_j
        // (MMAs of one thread run in order)
        if (ns < nkb && ns <= npv + 1) {
          const int s = ns & 1, ks = ns % KST;
          const uint32_t ph = (uint32_t)(ns >> 1) & 1u;
          if (mbar_test_wait(K_FULL0 + 8 * ks, (uint32_t)(ns / KST) & 1u) &&
              mbar_test_wait(S_EMPTY0 + 8 * s, ph ^ 1u)) {
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(s * KB);
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
              const uint64_t ad = smem_desc_sw128(sQ + kc * CHUNK);
              const uint64_t bd = smem_desc_sw128(sK0 + ks * C::K_STAGE + kc * C::K_CHUNK);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16(d, ad + 2ull * k, bd + 2ull * k, idesc_s, (kc | k) != 0 ? 1u : 0u);
            }
            mma_commit(S_FULL0 + 8 * s);
            mma_commit(K_EMPTY0 + 8 * ks);
            ++ns;
            progressed = true;
          }
        }
        if (npv < ns) {
          const int pb = npv & 1, vs = npv % VST;       // P buffer (TMEM), V stage
          if (mbar_test_wait(P_FULL0 + 8 * pb, (uint32_t)(npv >> 1) & 1u) &&
              mbar_test_wait(V_FULL0 + 8 * vs, (uint32_t)(npv / VST) & 1u)) {
            tc_fence_after();
            // A = P_j from TMEM: 16 keys (8 columns of bf16 pairs) per MMA
            const uint32_t tp = tmem + (uint32_t)(pb * KB);
#pragma unroll
            for (int kc = 0; kc < KB / 64; ++kc) {
              const uint64_t bd = smem_desc_sw128(sV0 + vs * C::V_STAGE + kc * CHUNK);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_bf16_tmem_a(tO, tp + (uint32_t)(32 * kc + 8 * k), bd + 2ull * k, idesc_o,
                                (npv | kc | k) != 0 ? 1u : 0u);
            }
            mma_commit(P_EMPTY0 + 8 * pb);
            mma_commit(V_EMPTY0 + 8 * vs);
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
        for (int c = 0; c < KB / 64; ++c) tmem_ld64(srow + c * 64, v + c * 64);   // 1.5-2% faster
        tmem_ld_wait();                                                           // than 2 x32
      }
      tc_fence_before();
      mbar_arrive(S_EMPTY0 + 8 * s);
      const int key0 = j * KB;
      const bool diag = key0 + KB - 1 > qp_min;   // only blocks reaching past a row need the mask
      if (diag) {
#pragma unroll
        for (int i = 0; i < KB; ++i)
          if (key0 + i > qp) v[i] = -INFINITY;
      }
      // row max (exact in any order): KB / 16 chains of three-input max over 16 scores
      float mc[KB / 16];
#pragma unroll
      for (int r = 0; r < KB / 16; ++r) {
        const float* w = v + 16 * r;
        float t = max3(w[0], w[1], w[2]);
#pragma unroll
        for (int i = 3; i < 15; i += 2) t = max3(t, w[i], w[i + 1]);
        mc[r] = fmaxf(t, w[15]);
      }
      float mx = mc[0];
#pragma unroll
      for (int r = 1; r + 1 < KB / 16; r += 2) mx = max3(mx, mc[r], mc[r + 1]);
      if ((KB / 16) % 2 == 0) mx = fmaxf(mx, mc[KB / 16 - 1]);
      const float m_cand = mx * a.scale_log2;
      const bool grow = m_cand > m + kRescaleThreshold;
      const float m_new = grow ? m_cand : m;
      const float alpha = grow ? exp2f(m - m_new) : 1.0f;
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O holds P_0..j-1 V: wait until the last of those MMAs landed, then rescale.
        const int jp = j - 1;
        if (!mbar_wait(P_EMPTY0 + 8 * (jp & 1), (uint32_t)(jp >> 1) & 1u, abort_flag,
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
      // P_j as bf16 pairs over the first KB / 2 columns of S_j's buffer (S_j has been
      // read; P_{j-2}, which the buffer held before S_j, was consumed by then)
      // p = 2^(s * scale - m), two keys per paired instruction; the row sum in two
      // paired accumulators (four interleaved partial sums)
      const uint64_t scale2 = f2_pack(a.scale_log2, a.scale_log2);
      const uint64_t negm2 = f2_pack(-m, -m);
      uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
      const uint32_t prow = tmem + lane_off + (uint32_t)(s * KB);
#pragma unroll
      for (int c = 0; c < KB / 64; ++c) {
        float pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          float x0, x1;
          f2_unpack(fma_f2(f2_pack(v[c * 64 + i], v[c * 64 + i + 1]), scale2, negm2), x0, x1);
          const float p0 = exp2_p(x0);
          const float p1 = exp2_p(x1);
          acc2[(i >> 1) & 1] = add_f2(acc2[(i >> 1) & 1], f2_pack(p0, p1));
          pk[i / 2] = __uint_as_float(pack_bf16x2(p0, p1));
        }
        tmem_st32(prow + (uint32_t)(32 * c), pk);
      }
      tmem_st_wait();
      float s0, s1, s2, s3;
      f2_unpack(acc2[0], s0, s1);
      f2_unpack(acc2[1], s2, s3);
      l = l * alpha + ((s0 + s2) + (s1 + s3));
      tc_fence_before();
      mbar_arrive(P_FULL0 + 8 * s);
    }
    if (nkb == 0) ok = false;   // nothing was computed for this query block
    if (ok) {
      const int jl = nkb - 1;
      ok = mbar_wait(P_EMPTY0 + 8 * (jl & 1), (uint32_t)(jl >> 1) & 1u, abort_flag, a.status);
    }
    if (ok) {
      tc_fence_after();
      const float inv = 1.0f / l;
      if (a.lse && qi < n_b) a.lse[(row0 + qi) * a.hq + h] = m + log2f(l);
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

template <int KB, int KST, int VST>
cudaError_t launch_attention_cfg(const Ctx& c, int B, int n, int hq, const void* qkv, int ldq,
                                 const CUtensorMap& mVt, const AttnArgs& a, const AttnKv* kv) {
  using Cf = AttnCfg<KB, KST, VST>;
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
  auto k = attention_tc_kernel<KB, KST, VST>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(hq, B, a.nqb);
  return launch_pdl(k, grid, dim3(THREADS), Cf::SMEM, c.stream, mQ, mK, mVt, a);
}

}  // namespace

// A sequence of at most this many tokens is one 128-key block: it runs the
// <128, 3, 3> configuration; longer ones the two-CTAs-per-SM <64, 3, 2> configuration,
// which measured 7-15% faster from 256 to 16384 tokens (GB300, 12/4 and 16/4 heads).
// K stages of the 64-key configuration (the V stages take the rest of the five its
// shared memory holds).
#ifndef XMOD_ATTN_K_STAGES
#define XMOD_ATTN_K_STAGES 3
#endif
#ifndef XMOD_ATTN_ONE_BLOCK_MAX_N
#define XMOD_ATTN_ONE_BLOCK_MAX_N 128
#endif

bool attention_tc_supported(int hd, int n, int ldq) {
  return hd == HD && n > 0 && ldq % 8 == 0 && tma_available();
}

cudaError_t launch_attention_tc(const Ctx& c, int B, int n, int hq, int hkv, const void* qkv,
                                int ldq, const void* vt, int vt_ld, void* o,
                                const int32_t* seq_count, const int32_t* seq_off,
                                const AttnKv* kv, float* lse) {
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
  a.lse = lse;
  if (nkv <= XMOD_ATTN_ONE_BLOCK_MAX_N)
    return launch_attention_cfg<128, 3, 3>(c, B, n, hq, qkv, ldq, mVt, a, kv);
  return launch_attention_cfg<64, XMOD_ATTN_K_STAGES, 5 - XMOD_ATTN_K_STAGES>(c, B, n, hq, qkv,
                                                                            ldq, mVt, a, kv);
}

}  // namespace xmod
