// Tensor-core GEMM for sm_103a (tcgen05 + TMEM + TMA) with the block's fused
// epilogues. bf16 operands, fp32 accumulation.
//
//   C[M, N] = A[M, K] . B[N, K]^T      (A activations, B weights in [out, in] layout)
//
// Persistent CTAs (one per SM) walk the output tiles; inside a CTA the work is
// split by warp:
//   warp 0      TMA producer: streams 128 x 64 A tiles and BN x 64 B tiles into a
//               ring of shared-memory stages (128-byte swizzle)
//   warp 1      allocates TMEM; one lane issues tcgen05.mma (128 x BN x 16) into one
//               of two TMEM accumulators, committing each stage back to the producer
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator (TMEM lane = output
//               row, 32 columns at a time), the fused epilogue math, and 16-byte global
//               loads and stores of that row segment. The other accumulator meanwhile
//               receives the next tile's MMAs.
// Gathered-RMSNorm variant (q | k | v of a sparse layer): the A tile rows are the
// selected tokens' rows of the residual stream itself, brought in by TMA gather4 (four
// rows per copy), and four more warps apply RMSNorm1 on the way: each thread owns one
// row of the A tile, multiplies it by the gain in shared memory before the MMA reads it
// and sums its squares over the k-blocks; the epilogue scales the row's outputs by
// 1 / rms (RMSNorm(x) g . W^T = (1 / rms) (x g) . W^T), so no gathered copy is written.
// Fused epilogues: plain store (optionally q | k | v from three weight tensors, with
// v written transposed for the attention kernel), O-projection (a in bf16; h = x_sel
// + a in fp32 when a separate RMSNorm needs it, or h * rms2 and h's sums of squares
// when RMSNorm2 is folded), SwiGLU (gate and up halves of one tile), and the down
// projection's gated scatter back into the residual stream at the selected rows
// (X-MoD notes Eq. 7 / Eq. 6; a dense layer adds a + f), which reads a back.

#include <cuda.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdlib.h>
#include <string.h>

#include "internal.h"
#include "tc_common.cuh"

namespace xmod {

namespace {

using namespace tc;

constexpr int BM = 128, BK = 64;
// Epilogue warps: two per TMEM lane quadrant, each taking every other 32-column
// chunk of the tile, so the epilogue of a CTA's last tile finishes sooner.
#ifndef XMOD_EPI_WARPS
#define XMOD_EPI_WARPS 8
#endif
constexpr int EPI_WARPS = XMOD_EPI_WARPS;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
// RMSNorm warps of the gathered-A variant (one thread per A tile row), and the shared
// memory they add: 1 / rms of both accumulators' rows, then their barriers.
constexpr int XF_WARPS = 4;
constexpr int XF_SMEM = 2 * 128 * 4 + 256;

template <int BN>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (200 * 1024) / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
  // the last 256 bytes: 2 * STAGES + 5 mbarriers, the TMEM address and the abort flag
  static_assert((2 * STAGES + 5) * 8 + 12 <= 256, "barrier block overflows");
};

struct TcArgs {
  int M, N, K;
  int mode;                // EpiKind
  int n_split1, n_split2;  // STORE: first accumulator column served by B map 1 / map 2
  int tiles_m, tiles_n, tiles;   // tiles counts every k slice
  int ksplit;              // k slices per output tile (ROUTER only; else 1)
  const int32_t* M_dev;    // if set, the rows are min(*M_dev, M), read on the device
  int v8;                  // epilogue row segments may use 32-byte accesses
  // gathered-A variant: row m of A is row (m / g_n) * g_T + g_idx[m] of the stream
  const int32_t* g_idx;
  int g_T, g_n;
  const __nv_bfloat16* g_gamma;
  float g_eps;
  // Stream-K (see Work): the tiles' k-blocks split evenly over the CTAs
  int sk;
  int64_t units;           // tiles x k-blocks
  float* sk_part;          // per-CTA partial accumulator slots, BM x BN fp32 each
  int* sk_flag;            // per-CTA "slot published" flags, 0 between launches
  int band2;               // CTA-pair kernel: 256-row blocks per band of the tile order
  int k_split1, k_split2;  // MN-major B stacked along K: first k of B map 1 / map 2
  Epilogue e;
  int* status;
};

// Row blocks per band of the tile order. Tiles are numbered band by band; inside a
// band the row block varies fastest. The tiles that run at the same time (one per
// CTA) then cover a band of XMOD_TILE_BAND row blocks by about 152 / XMOD_TILE_BAND
// column blocks, so A and B are both re-read from L2 rather than from DRAM when the
// operands do not fit in L2 together.
#ifndef XMOD_TILE_BAND
#define XMOD_TILE_BAND 16
#endif

// An operand stored [K, rows] (its rows contiguous) reaches shared memory in one TMA
// load through a 3-D tensor map (64 rows, k, 64-row chunk): chunk j holds rows 64j ..
// 64j + 63 for the 64 k of the block, one 128-byte line (64 rows) per k under the
// 128-byte swizzle, 8 KB a chunk.
// The MMA reads it as an MN-major operand (smem_desc_sw128_mn: 64-row atoms one chunk
// apart, groups of 8 k 1 KB apart), the instruction descriptor marking it MN-major.
constexpr int MN_BOX_BYTES = 64 * BK * 2;

// The kernels take the operand layout as a template parameter LAY, so the K-major
// kernels' MMA-issuing loop keeps compile-time descriptors: LAY_KK both operands K-major,
// LAY_MM both MN-major (weight gradients dY^T X from token-major dY and X), LAY_KM A
// K-major and B MN-major (activation gradients dY W from W as stored).
enum { LAY_KK = 0, LAY_MM = 1, LAY_KM = 2 };
template <int LAY> constexpr bool kAMn = LAY == LAY_MM;
template <int LAY> constexpr bool kBMn = LAY != LAY_KK;
template <int LAY>
constexpr uint32_t kIdescMajor =
    (kAMn<LAY> ? kIdescAMajorMN : 0u) | (kBMn<LAY> ? kIdescBMajorMN : 0u);
// Descriptor of an operand tile and its advance per 16-deep MMA step (in 16-byte units):
// K-major 32 bytes along each row, MN-major 2 KB (two groups of 8 k).
template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t addr) {
  if constexpr (MN) return smem_desc_sw128_mn(addr, MN_BOX_BYTES);
  else return smem_desc_sw128(addr);
}
template <bool MN>
constexpr uint64_t kOperandStep = MN ? 128ull : 2ull;
// The loads of `rows` rows of an operand tile from row r0, k from k0.
template <bool MN>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int k0, int r0, int rows) {
  if constexpr (!MN) {
    tma_load_2d(dst, map, bar, k0, r0);
  } else {
    tma_load_3d(dst, map, bar, 0, k0, r0 / 64);
  }
}
// The same for a CTA of a pair, the bytes counted on a barrier of either CTA.
template <bool MN>
__device__ __forceinline__ void load_operand_pair(uint32_t dst, const CUtensorMap* map,
                                                  uint32_t bar, int k0, int r0, int rows) {
  if constexpr (!MN) {
    tma_load_2d_pair(dst, map, bar, k0, r0);
  } else {
    tma_load_3d_pair(dst, map, bar, 0, k0, r0 / 64);
  }
}
// An MN-major B stacked along K from up to three maps: the map holding k-block kb and
// the block's first k inside it.
__device__ __forceinline__ const CUtensorMap* b_map_at_k(const TcArgs& a, const CUtensorMap* m0,
                                                         const CUtensorMap* m1,
                                                         const CUtensorMap* m2, int kb, int& k0) {
  k0 = kb * BK;
  if (k0 >= a.k_split2) {
    k0 -= a.k_split2;
    return m2;
  }
  if (k0 >= a.k_split1) {
    k0 -= a.k_split1;
    return m1;
  }
  return m0;
}

__device__ __forceinline__ void tile_coords(const TcArgs& a, int tiles_m, int tile, int& m_blk,
                                            int& n_blk, int band_rows = XMOD_TILE_BAND) {
  const int per_band = band_rows * a.tiles_n;
  const int band = tile / per_band;
  const int r = tile - band * per_band;
  const int m_first = band * band_rows;
  const int rows = min(band_rows, tiles_m - m_first);
  m_blk = m_first + r % rows;
  n_blk = r / rows;
}

// Rows and tiles of one launch: fixed at launch, or -- with M_dev -- the row count
// written by an earlier kernel (a variable number of routed tokens), read after
// griddepcontrol.wait. Tiles past it are skipped.
struct Extent {
  int M, tiles_m, tiles;
};
__device__ __forceinline__ Extent launch_extent(const TcArgs& a, int tile_rows) {
  Extent x{a.M, a.tiles_m, a.tiles};
  if (a.M_dev) {
    const int m = *a.M_dev;
    x.M = m < 0 ? 0 : (m < a.M ? m : a.M);
    x.tiles_m = (x.M + tile_rows - 1) / tile_rows;
    x.tiles = x.tiles_m * a.tiles_n * a.ksplit;
  }
  return x;
}

// What one CTA does next: output tile `tile` (k slice `ks` for the router), k-blocks
// [kb0, kb1). Data-parallel launches give every CTA whole tiles, round robin.
//
// Stream-K launches line up the k-blocks of all tiles, tile after tile, and give
// CTA c the c-th of gridDim.x equal shares, so every SM issues the same number of
// MMAs whatever the tile count (no partial last wave). A tile cut between CTAs c and
// c + 1 is finished by c, which holds its first k-blocks and reaches it last, at the
// end of its share (WORK_OWNER); c + 1 takes the tile's last k-blocks first, leaves
// its fp32 accumulator in slot c + 1 and raises flag c + 1 (WORK_PART). The owner
// waits for the flag (bounded), adds the slot into its TMEM accumulator -- one fixed
// order, so results do not depend on timing -- clears the flag for the next launch
// and runs the epilogue. A CTA starts inside a tile at most once per launch, and the
// host takes this path only when each share covers a whole tile's k-blocks, so a tile
// spans at most two CTAs and each slot serves one tile. The producer, the MMA issuer
// and the epilogue walk the same sequence.
enum { WORK_FULL = 0, WORK_PART = 1, WORK_OWNER = 2 };
struct Work {
  int tile, ks, kb0, kb1, role;
};
__device__ __forceinline__ bool work_at(const TcArgs& a, const Extent& ext, int nk, int i,
                                        Work& w) {
  if (a.sk) {
    const int64_t P = gridDim.x, cta = blockIdx.x;
    const int64_t u0 = cta * a.units / P, u1 = (cta + 1) * a.units / P;
    const int64_t tile = u0 / nk + i;
    const int64_t s = max(u0, tile * nk), e = min(u1, (tile + 1) * nk);
    if (s >= e) return false;
    w.tile = (int)tile;
    w.ks = 0;
    w.kb0 = (int)(s - tile * nk);
    w.kb1 = (int)(e - tile * nk);
    w.role = w.kb0 > 0 ? WORK_PART : (w.kb1 < nk ? WORK_OWNER : WORK_FULL);
    return true;
  }
  const int t = (int)blockIdx.x + i * (int)gridDim.x;
  if (t >= ext.tiles) return false;
  w.ks = t % a.ksplit;
  w.tile = t / a.ksplit;
  w.kb0 = w.ks * nk / a.ksplit;
  w.kb1 = (w.ks + 1) * nk / a.ksplit;
  w.role = WORK_FULL;
  return true;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Bounded wait for a neighbour's published slot (as mbar_wait: on timeout the status
// word gets XMOD_ERR_TIMEOUT and the CTA's abort flag is raised).
__device__ __noinline__ bool flag_wait(const int* f, volatile int* abort_flag, int* status) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire_gpu(f) != 0) return true;
    if ((i & 63u) == 63u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        report_status(status, XMOD_ERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
    __nanosleep(100);
  }
}

// All epilogue warps meet (an mbarrier of EPI_WARPS arrivals, so the wait is bounded);
// n counts the meetings for the phase parity.
__device__ __forceinline__ bool epi_meet(uint32_t bar, int& n, int lane, volatile int* abort_flag,
                                         int* status) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = mbar_wait(bar, (uint32_t)(n & 1), abort_flag, status);
  ++n;
  return ok;
}

// silu(z) = z * sigmoid(z) with the fast exponential and approximate division (a few
// ulp of fp32, far below the bf16 rounding of the result). A full-precision division
// here made the SwiGLU epilogue the bottleneck of the gate/up GEMM.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ int64_t stream_row_of(const Epilogue& e, int m) {
  if (e.tok) return e.tok[m];
  const int64_t b = m / e.n_per_seq;
  const int64_t t = e.idx ? (int64_t)e.idx[m] : (m - b * e.n_per_seq);
  return b * e.T + t;
}

// Row-segment helpers of the direct epilogue: 32 consecutive columns of one row, of
// which the first `rem` exist (rem a multiple of 8, or >= 32). With `v8` (every
// tensor the epilogue touches is 32-byte aligned with 32-byte-multiple row strides)
// a lane moves 32 bytes per access -- a whole sector -- instead of 16.
__device__ __forceinline__ void st_v8(void* p, const uint4& a, const uint4& b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}
__device__ __forceinline__ void ld_v8(const void* p, uint4& a, uint4& b) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                 "=r"(b.w)
               : "l"(p));
}

// bf16 segment: q[g] holds columns 8g .. 8g+7.
__device__ __forceinline__ void st_seg_bf16(__nv_bfloat16* p, const uint4 (&q)[4], int rem,
                                            bool v8) {
  if (v8) {
#pragma unroll
    for (int g = 0; g < 4; g += 2) {
      if (8 * g + 16 <= rem) st_v8(p + 8 * g, q[g], q[g + 1]);
      else if (8 * g < rem) *reinterpret_cast<uint4*>(p + 8 * g) = q[g];
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (8 * g < rem) *reinterpret_cast<uint4*>(p + 8 * g) = q[g];
  }
}
__device__ __forceinline__ void ld_seg_bf16(const __nv_bfloat16* p, uint4 (&q)[4], int rem,
                                            bool v8) {
  if (v8) {
#pragma unroll
    for (int g = 0; g < 4; g += 2) {
      if (8 * g + 16 <= rem) ld_v8(p + 8 * g, q[g], q[g + 1]);
      else if (8 * g < rem) q[g] = *reinterpret_cast<const uint4*>(p + 8 * g);
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (8 * g < rem) q[g] = *reinterpret_cast<const uint4*>(p + 8 * g);
  }
}
// fp32 segment: f[g] holds columns 4g .. 4g+3.
__device__ __forceinline__ void st_seg_f32(float* p, const float4 (&f)[8], int rem, bool v8) {
  if (v8) {
#pragma unroll
    for (int g = 0; g < 8; g += 2) {
      if (4 * g + 8 <= rem)
        st_v8(p + 4 * g, reinterpret_cast<const uint4&>(f[g]), reinterpret_cast<const uint4&>(f[g + 1]));
      else if (4 * g < rem) *reinterpret_cast<float4*>(p + 4 * g) = f[g];
    }
  } else {
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (4 * g < rem) *reinterpret_cast<float4*>(p + 4 * g) = f[g];
  }
}
__device__ __forceinline__ void ld_seg_f32(const float* p, float4 (&f)[8], int rem, bool v8) {
  if (v8) {
#pragma unroll
    for (int g = 0; g < 8; g += 2) {
      if (4 * g + 8 <= rem)
        ld_v8(p + 4 * g, reinterpret_cast<uint4&>(f[g]), reinterpret_cast<uint4&>(f[g + 1]));
      else if (4 * g < rem) f[g] = *reinterpret_cast<const float4*>(p + 4 * g);
    }
  } else {
#pragma unroll
    for (int g = 0; g < 8; ++g)
      if (4 * g < rem) f[g] = *reinterpret_cast<const float4*>(p + 4 * g);
  }
}

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* p, const float (&v)[32], int rem,
                                             bool v8) {
  uint4 q[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    q[g].x = pack_bf16x2(v[8 * g + 0], v[8 * g + 1]);
    q[g].y = pack_bf16x2(v[8 * g + 2], v[8 * g + 3]);
    q[g].z = pack_bf16x2(v[8 * g + 4], v[8 * g + 5]);
    q[g].w = pack_bf16x2(v[8 * g + 6], v[8 * g + 7]);
  }
  st_seg_bf16(p, q, rem, v8);
}

// Relative cost per output column of a tile of width 256 / 192 / 128 (the narrower
// tiles read more shared memory per FLOP), calibrated on the A4K8 block's GEMMs;
// used to pick the tile width.
#ifndef XMOD_COST_256
#define XMOD_COST_256 1.0
#endif
#ifndef XMOD_COST_192
#define XMOD_COST_192 1.15
#endif
#ifndef XMOD_COST_128
#define XMOD_COST_128 1.33
#endif
// Waves of 256 x 256 tiles from which a GEMM runs on CTA pairs.
#ifndef XMOD_PAIR_MIN_WAVES
#define XMOD_PAIR_MIN_WAVES 6
#endif
// Cost per column of a 256 x 256 pair tile (per SM, the single-CTA tiles' units), and
// the margin by which the pair estimate must beat the best single-CTA one below
// XMOD_PAIR_MIN_WAVES.
#ifndef XMOD_COST_PAIR
#define XMOD_COST_PAIR 0.82
#endif
// The same for 256 x 192 pair tiles (each SM reads 28 KB of operands from shared memory
// per 64-deep k-block of its 128 x 192 half, against 32 KB per 128 x 256 half of a
// 256 x 256 pair tile and 40 KB per 128 x 192 single-CTA tile).
#ifndef XMOD_COST_PAIR192
#define XMOD_COST_PAIR192 0.88
#endif
#ifndef XMOD_PAIR_MARGIN
#define XMOD_PAIR_MARGIN 0.10
#endif
// 0 disables the CTA-pair kernels.
#ifndef XMOD_GEMM_PAIRS
#define XMOD_GEMM_PAIRS 1
#endif

// WORK_PART: this lane's accumulator row, every 32-column chunk of this warp's share,
// into the CTA's slot (row-major, BN floats per row).
template <int BN>
__device__ __forceinline__ void sk_leave_partial(const TcArgs& a, int row, uint32_t t_row,
                                                 int part, int nparts) {
  float* dst = a.sk_part + ((int64_t)blockIdx.x * BM + row) * BN;
#pragma unroll 1
  for (int c = part; c < BN / 32; c += nparts) {
    float v[32];
    tmem_ld32(t_row + c * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int g = 0; g < 32; g += 8)
      st_v8(dst + c * 32 + g,
            make_uint4(__float_as_uint(v[g]), __float_as_uint(v[g + 1]), __float_as_uint(v[g + 2]),
                       __float_as_uint(v[g + 3])),
            make_uint4(__float_as_uint(v[g + 4]), __float_as_uint(v[g + 5]),
                       __float_as_uint(v[g + 6]), __float_as_uint(v[g + 7])));
  }
}

// WORK_OWNER: add the next CTA's slot into this lane's accumulator row in TMEM, the
// slot's next chunk loaded while the current one is added.
template <int BN>
__device__ __forceinline__ void sk_add_partial(const TcArgs& a, int row, uint32_t t_row, int part,
                                               int nparts) {
  const float* src = a.sk_part + ((int64_t)(blockIdx.x + 1) * BM + row) * BN;
  float4 pc[8], pn[8];
#pragma unroll
  for (int g = 0; g < 8; ++g) pc[g] = ld_cg_f4(src + part * 32 + 4 * g);
#pragma unroll 1
  for (int c = part; c < BN / 32; c += nparts) {
    if (c + nparts < BN / 32) {
#pragma unroll
      for (int g = 0; g < 8; ++g) pn[g] = ld_cg_f4(src + (c + nparts) * 32 + 4 * g);
    }
    float v[32];
    tmem_ld32(t_row + c * 32, v);
    tmem_ld_wait();
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      v[4 * g] += pc[g].x;
      v[4 * g + 1] += pc[g].y;
      v[4 * g + 2] += pc[g].z;
      v[4 * g + 3] += pc[g].w;
    }
    tmem_st32(t_row + c * 32, v);
#pragma unroll
    for (int g = 0; g < 8; ++g) pc[g] = pn[g];
  }
  tmem_st_wait();
}

// L2 prefetch of `bytes` bytes at p (16-byte aligned, a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// The epilogue inputs of this lane's row of the next tile -- the x row segment and,
// for the down projection, the a row segment -- brought into L2 while the tile's MMAs
// run, so that the epilogue's loads (issued only once the accumulator is complete)
// do not wait on DRAM. Row segments are 16-byte aligned: d and N are multiples of 8.
template <int BN, int MODE>
__device__ __forceinline__ void epi_prefetch(const TcArgs& a, int M, int m, int n_blk, int part) {
  if (MODE != EPI_OPROJ && MODE != EPI_DOWN_SCATTER) return;
  const Epilogue& e = a.e;
  const int col0 = n_blk * BN;
  if (m >= M || col0 >= a.N) return;
  const uint32_t bytes = 2u * (uint32_t)min(BN, a.N - col0);
  if (part == 0)
    prefetch_l2((const __nv_bfloat16*)e.x + stream_row_of(e, m) * e.d + col0, bytes);
  else if (MODE == EPI_DOWN_SCATTER && e.a)
    prefetch_l2((const __nv_bfloat16*)e.a + (int64_t)m * e.d + col0, bytes);
}

// Inputs of the O-projection / down-projection epilogues for one 32-column chunk of
// one row: x and, for the down projection, a (bf16). They are loaded one chunk ahead
// so that their memory latency overlaps the previous chunk's work.
struct EpiIn {
  uint4 x[4];
  uint4 a[4];
};

// Staged epilogue inputs (CTA-pair kernel, o-projection and down projection): a loader
// warp brings the tile's x rows (TMA gather4 at their stream rows) and, for the down
// projection, its a rows (a TMA tile) into shared memory, 64 columns at a time into
// one of two buffers, while the accumulator is still being computed; the epilogue reads
// them from there instead of loading one row per lane from global memory. A buffer
// holds STG_TENSORS 128-row x 64-column bf16 tiles (128-byte swizzle, as TMA writes
// them: 16-byte chunk k of row r sits at chunk k ^ (r & 7)).
constexpr int STG_COLS = 64;
constexpr int STG_TILE = BM * STG_COLS * 2;   // 16 KB
template <int MODE>
__host__ __device__ constexpr int stg_tensors() {
  return MODE == EPI_DOWN_SCATTER ? 2 : (MODE == EPI_OPROJ ? 1 : 0);
}
template <int MODE>
__host__ __device__ constexpr int stg_bytes() {
  return 2 * stg_tensors<MODE>() * STG_TILE;
}

// Where the epilogue finds a staged chunk: the buffers' base, their full / empty
// barriers (two each, 8 bytes apart) and the global index of the tile's first
// 64-column pair (buffer = index & 1).
struct EpiStage {
  uint32_t base, full0, empty0;
  int gp0;
  volatile int* abort_flag;
  int* status;
};

// This lane's row (row r of the CTA tile) of the 32 columns of chunk c from the staged
// buffer; false if the wait ran out.
template <int MODE>
__device__ __forceinline__ bool epi_load_staged(const EpiStage& st, int c, int r, EpiIn& in) {
  const int g = st.gp0 + (c >> 1);
  const uint32_t u = (uint32_t)(g & 1);
  if (!mbar_wait(st.full0 + 8u * u, (uint32_t)(g >> 1) & 1u, st.abort_flag, st.status))
    return false;
  const uint32_t row = st.base + u * (uint32_t)(stg_tensors<MODE>() * STG_TILE) + (uint32_t)r * 128u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t off = (uint32_t)((((c & 1) * 4 + j) ^ (r & 7)) << 4);
    in.x[j] = lds128(row + off);
    if (MODE == EPI_DOWN_SCATTER) in.a[j] = lds128(row + STG_TILE + off);
  }
  return true;
}

template <int MODE>
__device__ __forceinline__ void epi_load_in(const TcArgs& a, int M, int m, int col0, int64_t xrow,
                                            EpiIn& in) {
  const Epilogue& e = a.e;
  if (m >= M || col0 >= a.N) return;
  const int rem = a.N - col0;
  ld_seg_bf16((const __nv_bfloat16*)e.x + xrow + col0, in.x, rem, a.v8);
  if (MODE == EPI_DOWN_SCATTER && e.a)
    ld_seg_bf16((const __nv_bfloat16*)e.a + (int64_t)m * e.d + col0, in.a, rem, a.v8);
}

__device__ __forceinline__ void unpack_x(const EpiIn& in, float (&xv)[32]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&in.x[g]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h2[i]);
      xv[8 * g + 2 * i] = f.x;
      xv[8 * g + 2 * i + 1] = f.y;
    }
  }
}

// This lane writes its own row's 32 columns. (Passing each 32 x 32 chunk through
// shared memory to store along rows instead measured 1.3-1.5 ms per step slower on
// the A4K8 block: the extra shared-memory traffic competes with the MMA operand
// reads, and one epilogue warp per scheduler cannot hide the added latency.)
template <int MODE>
__device__ __forceinline__ void epilogue_chunk_direct(const TcArgs& a, int M, int m, int col0,
                                                      int64_t xrow, float r, float (&v)[32],
                                                      const EpiIn& in, int ks) {
  const Epilogue& e = a.e;
  if (m >= M || col0 >= a.N) return;
  const int rem = a.N - col0;
  if (MODE == EPI_STORE && e.out_f32) {
    float4 fv[8];
#pragma unroll
    for (int g = 0; g < 8; ++g)
      fv[g] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
    float* base = (float*)e.out;
    int row = m;
    if (e.row_split[1] > 0 && m >= e.row_split[1]) {
      base = (float*)e.out_rows[1];
      row = m - e.row_split[1];
    } else if (e.row_split[0] > 0 && m >= e.row_split[0]) {
      base = (float*)e.out_rows[0];
      row = m - e.row_split[0];
    }
    st_seg_f32(base + (int64_t)row * e.ldo + col0, fv, rem, a.v8);
  } else if (MODE == EPI_STORE || MODE == EPI_SWIGLU) {
    store32_bf16((__nv_bfloat16*)e.out + (int64_t)m * e.ldo + col0, v, rem, a.v8);
  } else if (MODE == EPI_OPROJ) {
    if (e.out) store32_bf16((__nv_bfloat16*)e.out + (int64_t)m * e.ldo + col0, v, rem, a.v8);
    float4 hv[8];   // h = x + a
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&in.x[g]);
      const float2 f0 = __bfloat1622float2(x2[0]), f1 = __bfloat1622float2(x2[1]);
      const float2 f2 = __bfloat1622float2(x2[2]), f3 = __bfloat1622float2(x2[3]);
      hv[2 * g] = make_float4(f0.x + v[8 * g], f0.y + v[8 * g + 1], f1.x + v[8 * g + 2],
                              f1.y + v[8 * g + 3]);
      hv[2 * g + 1] = make_float4(f2.x + v[8 * g + 4], f2.y + v[8 * g + 5], f3.x + v[8 * g + 6],
                                  f3.y + v[8 * g + 7]);
    }
    if (e.out2) st_seg_f32((float*)e.out2 + (int64_t)m * e.ldo2 + col0, hv, rem, a.v8);
    if (e.out3) {   // RMSNorm2 folded: h * g2 in bf16, and this chunk's sum of squares
      const uint4* gp = reinterpret_cast<const uint4*>((const __nv_bfloat16*)e.g2 + col0);
      uint4 q[4];
      float ss = 0.0f;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const uint4 gg = 8 * g < rem ? gp[g] : make_uint4(0, 0, 0, 0);
        const __nv_bfloat162* g2v = reinterpret_cast<const __nv_bfloat162*>(&gg);
        const float4 h0 = hv[2 * g], h1 = hv[2 * g + 1];
        const float2 a0 = __bfloat1622float2(g2v[0]), a1 = __bfloat1622float2(g2v[1]);
        const float2 a2 = __bfloat1622float2(g2v[2]), a3 = __bfloat1622float2(g2v[3]);
        if (8 * g < rem)
          ss += h0.x * h0.x + h0.y * h0.y + h0.z * h0.z + h0.w * h0.w + h1.x * h1.x +
                h1.y * h1.y + h1.z * h1.z + h1.w * h1.w;
        q[g].x = pack_bf16x2(h0.x * a0.x, h0.y * a0.y);
        q[g].y = pack_bf16x2(h0.z * a1.x, h0.w * a1.y);
        q[g].z = pack_bf16x2(h1.x * a2.x, h1.y * a2.y);
        q[g].w = pack_bf16x2(h1.z * a3.x, h1.w * a3.y);
      }
      st_seg_bf16((__nv_bfloat16*)e.out3 + (int64_t)m * e.ldo2 + col0, q, rem, a.v8);
      e.rowss[(int64_t)m * (e.norm_d / 32) + col0 / 32] = ss;
    }
  } else if (MODE == EPI_ROUTER) {   // xrow is the stream token here; k slice ks -> plane ks
    float* sp = (float*)e.out + ks * e.plane + (int64_t)col0 * e.ldo + xrow;
    const float b = e.bias && ks == 0 ? e.bias[xrow] : 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < rem) sp[(int64_t)i * e.ldo] = v[i] + b;
  } else {  // EPI_DOWN_SCATTER with the attention residual a (none: a = 0)
    const float g7 = e.varsigma * r;
    uint4 qo[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {   // 8 columns at a time
      const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&in.x[g]);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&in.a[g]);
      float y[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(x2[i]);
        const float2 af = e.a ? __bfloat1622float2(a2[i]) : make_float2(0.0f, 0.0f);
        const float xx[2] = {f.x, f.y}, aa[2] = {af.x, af.y};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = 2 * i + k;
          const float fv = v[8 * g + j];
          if (e.gate == XMOD_GATE_XMOD) y[j] = xx[k] + g7 * (aa[k] + fv);   // Eq. 7
          else if (e.gate == XMOD_GATE_MOD) y[j] = (xx[k] + aa[k]) + r * fv;   // Eq. 6
          else y[j] = (xx[k] + aa[k]) + fv;                                      // dense
        }
      }
      qo[g].x = pack_bf16x2(y[0], y[1]);
      qo[g].y = pack_bf16x2(y[2], y[3]);
      qo[g].z = pack_bf16x2(y[4], y[5]);
      qo[g].w = pack_bf16x2(y[6], y[7]);
    }
    st_seg_bf16((__nv_bfloat16*)e.x + xrow + col0, qo, rem, a.v8);
    if (e.out) st_seg_bf16((__nv_bfloat16*)e.out + (int64_t)m * e.ldo + col0, qo, rem, a.v8);
  }
}

// Epilogue of one tile for this warp's 32-row slab [wrow0, wrow0 + 32). RS: every
// accumulator value of this lane's row is scaled by rscale first (gathered RMSNorm).
template <int BN, int MODE, bool RS = false, bool STG = false>
__device__ __forceinline__ bool epilogue_tile(const TcArgs& a, int M, int wrow0, int lane,
                                              int n_blk, uint32_t t_row, int part, int nparts,
                                              int ks = 0, float rscale = 1.0f,
                                              const EpiStage* stg = nullptr, int trow0 = 0) {
  const Epilogue& e = a.e;
  constexpr bool swiglu = MODE == EPI_SWIGLU;
  // the row this lane owns in TMEM: its stream row and gate
  const int m_own = wrow0 + lane;
  int64_t xrow_own = 0;
  float r_own = 1.0f;
  if ((MODE == EPI_OPROJ || MODE == EPI_DOWN_SCATTER) && m_own < M) {
    xrow_own = stream_row_of(e, m_own) * e.d;
    if (MODE == EPI_DOWN_SCATTER && e.gate >= 0) r_own = e.r_sel[m_own];
  }
  if (MODE == EPI_ROUTER && m_own < M) xrow_own = stream_row_of(e, m_own);
  // RMSNorm2 folded (see Epilogue::rowss): the row's 1 / rms for the SwiGLU inputs,
  // its chunk sums added in order
  float rstd_own = 1.0f;
  if (MODE == EPI_SWIGLU && e.rowss && m_own < M) {
    const float4* p = reinterpret_cast<const float4*>(e.rowss + (int64_t)m_own * (e.norm_d / 32));
    float ss = 0.0f;
    for (int i = 0; i < e.norm_d / 128; ++i) {
      const float4 q = p[i];
      ss += q.x;
      ss += q.y;
      ss += q.z;
      ss += q.w;
    }
    rstd_own = rsqrtf(ss / (float)e.norm_d + e.eps);
  }
  constexpr int NCH_FULL = BN / 32;
  const int nch = swiglu ? NCH_FULL / 2 : NCH_FULL;
  const int col_tile0 = swiglu ? n_blk * (BN / 2) : n_blk * BN;
  constexpr bool needs_in = (MODE == EPI_OPROJ || MODE == EPI_DOWN_SCATTER) && !STG;
  EpiIn cur, nxt;
  if (needs_in && part < nch) epi_load_in<MODE>(a, M, m_own, col_tile0 + part * 32, xrow_own, cur);
#pragma unroll 1
  for (int c = part; c < nch; c += nparts) {
    if (needs_in && c + nparts < nch)
      epi_load_in<MODE>(a, M, m_own, col_tile0 + (c + nparts) * 32, xrow_own, nxt);
    if (STG && !epi_load_staged<MODE>(*stg, c, wrow0 - trow0 + lane, cur)) return false;
    float v[32];
    if (swiglu) {
      float u[32];
      tmem_ld32(t_row + c * 32, v);
      tmem_ld32(t_row + BN / 2 + c * 32, u);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] *= rstd_own;
        u[i] *= rstd_own;
      }
      const int colh = col_tile0 + c * 32;
      if (e.out2 && m_own < M && colh < a.N) {   // the pre-activations G | U as well
        __nv_bfloat16* pg = (__nv_bfloat16*)e.out2 + (int64_t)m_own * e.ldo2 + colh;
        store32_bf16(pg, v, a.N - colh, a.v8);
        store32_bf16(pg + a.N, u, a.N - colh, a.v8);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = silu_f(v[i]) * u[i];
    } else {
      tmem_ld32(t_row + c * 32, v);
      tmem_ld_wait();
      if (RS) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= rscale;
      }
    }
    const int col0 = col_tile0 + c * 32;
    if (MODE == EPI_STORE && e.vt && col0 >= e.vt_col0) {
      // v^T: token m of sequence b goes to column t of rows (b, g, dim). For each dim
      // the warp's 32 consecutive tokens form one contiguous run, so no staging.
      if (m_own < M && col0 < a.N) {
        const int cv = col0 - e.vt_col0;
        const int g = cv / e.vt_hd, dim0 = cv % e.vt_hd;
        int64_t b, t;
        if (e.tok) {   // variable tokens per sequence: local index from the row offsets
          b = e.tok[m_own] / e.T;
          t = m_own - e.seq_off[b];
        } else {
          b = m_own / e.n_per_seq;
          t = m_own - b * e.n_per_seq;
        }
        __nv_bfloat16* p =
            (__nv_bfloat16*)e.vt + ((b * e.vt_hkv + g) * e.vt_hd + dim0) * (int64_t)e.vt_ld + t;
#pragma unroll
        for (int i = 0; i < 32; ++i) p[(int64_t)i * e.vt_ld] = __float2bfloat16_rn(v[i]);
      }
      if (!e.vt_rows) continue;
    }
    epilogue_chunk_direct<MODE>(a, M, m_own, col0, xrow_own, r_own, v, cur, ks);
    if (STG) {   // this warp is done with the chunk's staged rows
      __syncwarp();
      if (lane == 0) mbar_arrive(stg->empty0 + 8u * (uint32_t)((stg->gp0 + (c >> 1)) & 1));
    }
    cur = nxt;
  }
  return true;
}

template <int BN, int MODE, bool GATHER = false, int LAY = LAY_KK>
__global__ void __launch_bounds__(NUM_THREADS + (GATHER ? 32 * XF_WARPS : 0), 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
               const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
               const TcArgs args) {
  using C = Cfg<BN>;
  static_assert(!GATHER || MODE == EPI_STORE, "the gathered RMSNorm feeds a plain store");
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + C::STAGES * C::A_BYTES;
  const uint32_t sBar = sB + C::STAGES * C::B_BYTES;
  const uint32_t sTmem = sBar + 8 * (2 * C::STAGES + 5);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (sTmem - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (sTmem - base) + 8);
#define FULL(s) (sBar + 8u * (s))
#define EMPTY(s) (sBar + 8u * (C::STAGES + (s)))
#define ACC_FULL(a) (sBar + 8u * (2 * C::STAGES + (a)))
#define ACC_EMPTY(a) (sBar + 8u * (2 * C::STAGES + 2 + (a)))
#define EPI_MEET (sBar + 8u * (2 * C::STAGES + 4))
  // gathered-A variant only: 1 / rms of the rows of accumulator a at sXf + 512 a, then
  // XFORM(s) (stage s holds RMSNorm-gained rows) and RSTD_FULL(a) (1 / rms of a's rows
  // written)
  const uint32_t sXf = sBar + 256;
  float* rstd_buf = reinterpret_cast<float*>(gbase + (sXf - base));
#define XFORM(s) (sXf + 1024u + 8u * (s))
#define RSTD_FULL(a) (sXf + 1024u + 8u * (C::STAGES + (a)))
  static_assert(!GATHER || 8 * (C::STAGES + 2) <= XF_SMEM - 1024, "RMSNorm barriers overflow");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (args.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), 1);
      if (GATHER) mbar_init(XFORM(s), XF_WARPS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(ACC_FULL(a), 1);
      mbar_init(ACC_EMPTY(a), 32 * EPI_WARPS);
      if (GATHER) mbar_init(RSTD_FULL(a), XF_WARPS);
    }
    mbar_init(EPI_MEET, EPI_WARPS);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB0);
    if (MODE == EPI_SWIGLU || args.n_split1 < args.N) prefetch_tensormap(&tmB1);
    if (MODE != EPI_SWIGLU && args.n_split2 < args.N) prefetch_tensormap(&tmB2);
  }
  if (warp == 1) tmem_alloc(sTmem, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // everything above overlapped the previous kernel's tail
  const Extent ext = launch_extent(args, BM);

  if (warp == 0 && GATHER) {
    // The whole warp loads: lane l gathers rows 4l .. 4l+3 of each A tile, lane 0 also
    // the B tile.
    int it = 0;
    Work w;
    bool run = true;
    for (int i = 0; run && work_at(args, ext, nk, i, w); ++i) {
      int m_blk, n_blk;
      tile_coords(args, ext.tiles_m, w.tile, m_blk, n_blk);
      const int m0 = m_blk * BM;
      int r[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {   // rows past M repeat a valid row; never stored
        const int m = m0 + 4 * lane + q;
        r[q] = m < ext.M ? (m / args.g_n) * args.g_T + args.g_idx[m] : 0;
      }
      const CUtensorMap* mp = &tmB0;
      int brow = n_blk * BN;
      if (brow >= args.n_split2) {
        mp = &tmB2;
        brow -= args.n_split2;
      } else if (brow >= args.n_split1) {
        mp = &tmB1;
        brow -= args.n_split1;
      }
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
        int ok = 1;
        if (lane == 0) {
          ok = !*abort_flag && mbar_wait(EMPTY(s), ph ^ 1u, abort_flag, args.status);
          if (ok) mbar_arrive_expect_tx(FULL(s), C::STAGE_BYTES);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          run = false;
          break;
        }
        tma_gather4(sA + s * C::A_BYTES + lane * 512, &tmA, FULL(s), kb * BK, r[0], r[1], r[2],
                    r[3]);
        if (lane == 0) tma_load_2d(sB + s * C::B_BYTES, mp, FULL(s), kb * BK, brow);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      Work w;
      for (int i = 0; work_at(args, ext, nk, i, w) && !*abort_flag; ++i) {
        int m_blk, n_blk;
        tile_coords(args, ext.tiles_m, w.tile, m_blk, n_blk);
        const int kb0 = w.kb0, kb1 = w.kb1;
        const int m0 = m_blk * BM;
        const CUtensorMap* mp = &tmB0;
        int brow = n_blk * BN;
        if (MODE != EPI_SWIGLU) {
          if (brow >= args.n_split2) {
            mp = &tmB2;
            brow -= args.n_split2;
          } else if (brow >= args.n_split1) {
            mp = &tmB1;
            brow -= args.n_split1;
          }
        }
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait(EMPTY(s), ph ^ 1u, abort_flag, args.status)) break;
          mbar_arrive_expect_tx(FULL(s), C::STAGE_BYTES);
          load_operand<kAMn<LAY>>(sA + s * C::A_BYTES, &tmA, FULL(s), kb * BK, m0, BM);
          if (MODE == EPI_SWIGLU) {
            const int h0 = n_blk * (BN / 2);
            tma_load_2d(sB + s * C::B_BYTES, &tmB0, FULL(s), kb * BK, h0);
            tma_load_2d(sB + s * C::B_BYTES + (BN / 2) * 128, &tmB1, FULL(s), kb * BK, h0);
          } else {
            int k0 = kb * BK;
            const CUtensorMap* bm = mp;
            if constexpr (kBMn<LAY>) bm = b_map_at_k(args, &tmB0, &tmB1, &tmB2, kb, k0);
            load_operand<kBMn<LAY>>(sB + s * C::B_BYTES, bm, FULL(s), k0, brow, BN);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN) | kIdescMajor<LAY>;
      constexpr uint64_t astep = kOperandStep<kAMn<LAY>>, bstep = kOperandStep<kBMn<LAY>>;
      int it = 0;
      Work w;
      for (int lt = 0; work_at(args, ext, nk, lt, w) && !*abort_flag; ++lt) {
        const int acc = lt & 1;
        const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
        if (!mbar_wait(ACC_EMPTY(acc), aph ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int kb0 = w.kb0, kb1 = w.kb1;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait(GATHER ? XFORM(s) : FULL(s), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = operand_desc<kAMn<LAY>>(sA + s * C::A_BYTES);
          const uint64_t bd = operand_desc<kBMn<LAY>>(sB + s * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16(d_tmem, ad + astep * k, bd + bstep * k, idesc, (kb != kb0 || k) ? 1u : 0u);
          mma_commit(EMPTY(s));
        }
        if (!ok) break;
        mma_commit(ACC_FULL(acc));
      }
    }
  } else if (GATHER && warp >= 2 + EPI_WARPS) {
    // RMSNorm1 on the gathered rows: this thread owns row xr of every A tile. Each stage:
    // the row's 64 columns times the gain, back in place (the 128-byte swizzle puts
    // 16-byte chunk c of row r at chunk c ^ (r & 7)), and their squares summed in column
    // order. After a tile's last k-block: 1 / rms for the epilogue.
    const int xr = (warp - 2 - EPI_WARPS) * 32 + lane;
    const float inv_d = 1.0f / (float)args.K;
    int it = 0;
    Work w;
    for (int lt = 0; work_at(args, ext, nk, lt, w); ++lt) {
      const int acc = lt & 1;
      const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
      float ss = 0.0f;
      bool ok = true;
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
        if (!mbar_wait(FULL(s), ph, abort_flag, args.status)) {
          ok = false;
          break;
        }
        uint8_t* row = gbase + (sA - base) + s * C::A_BYTES + xr * 128;
        // columns past K are the map's zero fill: nothing to add or scale there
        const int nc = min(8, (args.K - kb * BK) / 8);
        // two halves of four 16-byte chunks, every load of a half issued before its math
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint4 v[4], g[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cc = 4 * h + c;
            if (cc < nc) {
              v[c] = *reinterpret_cast<const uint4*>(row + ((cc ^ (xr & 7)) << 4));
              g[c] = __ldg(reinterpret_cast<const uint4*>(args.g_gamma + kb * BK + 8 * cc));
            }
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cc = 4 * h + c;
            if (cc < nc) {
              uint32_t* vw = reinterpret_cast<uint32_t*>(&v[c]);
              const uint32_t* gw = reinterpret_cast<const uint32_t*>(&g[c]);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float2 xf =
                    __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vw[q]));
                const float2 gf =
                    __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[q]));
                ss = fmaf(xf.x, xf.x, ss);
                ss = fmaf(xf.y, xf.y, ss);
                vw[q] = pack_bf16x2(xf.x * gf.x, xf.y * gf.y);
              }
              *reinterpret_cast<uint4*>(row + ((cc ^ (xr & 7)) << 4)) = v[c];
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(XFORM(s));
      }
      if (!ok) break;
      // the buffer of accumulator acc is free once the epilogue of tile lt - 2 is done
      if (!mbar_wait(ACC_EMPTY(acc), aph ^ 1u, abort_flag, args.status)) break;
      rstd_buf[acc * 128 + xr] = 1.0f / sqrtf(ss * inv_d + args.g_eps);
      __syncwarp();
      if (lane == 0) mbar_arrive(RSTD_FULL(acc));
    }
  } else {
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31 belong to this warp
    const int part = (warp - 2) / 4, nparts = EPI_WARPS / 4;
    int meets = 0;
    Work w;
    for (int lt = 0; work_at(args, ext, nk, lt, w); ++lt) {
      const int acc = lt & 1;
      const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
      int m_blk, n_blk;
      tile_coords(args, ext.tiles_m, w.tile, m_blk, n_blk);
      const int wrow0 = m_blk * BM + quad * 32;
      if (w.role != WORK_PART) epi_prefetch<BN, MODE>(args, ext.M, wrow0 + lane, n_blk, part);
      if (!mbar_wait(ACC_FULL(acc), aph, abort_flag, args.status)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
      bool ok = true;
      if (w.role == WORK_PART) {
        sk_leave_partial<BN>(args, quad * 32 + lane, t_row, part, nparts);
        __threadfence();
        ok = epi_meet(EPI_MEET, meets, lane, abort_flag, args.status);
        if (ok && warp == 2 && lane == 0) st_release_gpu(args.sk_flag + blockIdx.x, 1);
      } else {
        if (w.role == WORK_OWNER) {
          if (warp == 2 && lane == 0 &&
              flag_wait(args.sk_flag + blockIdx.x + 1, abort_flag, args.status))
            args.sk_flag[blockIdx.x + 1] = 0;   // consumed: clear for the next launch
          ok = epi_meet(EPI_MEET, meets, lane, abort_flag, args.status) && !*abort_flag;
          if (ok) sk_add_partial<BN>(args, quad * 32 + lane, t_row, part, nparts);
        }
        if (GATHER) {
          ok = ok && mbar_wait(RSTD_FULL(acc), aph, abort_flag, args.status);
          if (ok)
            epilogue_tile<BN, MODE, true>(args, ext.M, wrow0, lane, n_blk, t_row, part, nparts,
                                          w.ks, rstd_buf[acc * 128 + quad * 32 + lane]);
        } else if (ok) {
          epilogue_tile<BN, MODE>(args, ext.M, wrow0, lane, n_blk, t_row, part, nparts, w.ks);
        }
      }
      tc_fence_before();
      mbar_arrive(ACC_EMPTY(acc));
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait ran out: give copies and MMAs still in flight time to land before the
    // shared memory and TMEM are released.
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 20000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
#undef FULL
#undef EMPTY
#undef ACC_FULL
#undef ACC_EMPTY
#undef EPI_MEET
#undef XFORM
#undef RSTD_FULL
}

// ---------------------------------------------------------------- CTA-pair variant
//
// The same GEMM on 256 x BN tiles shared by the two CTAs of a (2, 1, 1) cluster
// (tcgen05 cta_group::2). CTA r of the pair loads rows [128 r, 128 r + 128) of the A
// tile and rows [r BN/2, (r+1) BN/2) of the B tile (for SwiGLU: the gate rows in CTA 0,
// the up rows in CTA 1), so each SM streams half the B bytes per FLOP of the
// single-CTA kernel. CTA 0 issues every MMA; completion of a stage is signalled to
// both CTAs' producers, completion of a tile to both CTAs' epilogues, which then
// work exactly as in the single-CTA kernel on their own 128 TMEM lanes.
template <int BN>
struct Cfg2 {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (BN / 2) * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (200 * 1024) / STAGE_BYTES;
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
};
// The same with STG bytes of staged epilogue inputs, the stage ring filling what is
// left of the 227 KB a CTA may hold (the staged epilogue needs little L1 cache).
template <int BN, int STG>
struct Cfg2S : Cfg2<BN> {
  static constexpr int STAGES =
      STG ? (227 * 1024 - 1024 - 256 - STG) / Cfg2<BN>::STAGE_BYTES : Cfg2<BN>::STAGES;
  static constexpr int SMEM = STAGES * Cfg2<BN>::STAGE_BYTES + STG + 1024 + 256;
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Row blocks (of 256) per band of the pair kernel's tile order: as many as keep the
// band's A rows within XMOD_BAND_A_BYTES, between 4 and XMOD_TILE_BAND2. Inside a band
// every column tile reads the band's A rows again, so they must stay in L2 across the
// band; the B operand (the weights) is read from DRAM about once per band, since between
// bands the output stream evicts it. A dense layer's gate/up at d_ff = 5632, B = 4, T =
// 16384 read its 46 MB of weights 32 times with 8-block bands (1.35 GB read against 314
// MB of operands), 8 times with 32-block bands; the down projection (K = 5632: 2.9 MB of
// A per row block) read its hidden operand over and over with 32-block bands (919 MB
// against 342 MB at B = 1), which 11-block bands (32 MB of A) avoid.
#ifndef XMOD_TILE_BAND2
#define XMOD_TILE_BAND2 32
#endif
#ifndef XMOD_BAND_A_BYTES
#define XMOD_BAND_A_BYTES (32 << 20)
#endif
int band2_rows(int K) {
  const long per_block = 2L * BM * K * 2;   // bf16 A rows of one 256-row block
  const long r = (long)XMOD_BAND_A_BYTES / (per_block > 0 ? per_block : 1);
  return (int)(r < 4 ? 4 : (r > XMOD_TILE_BAND2 ? XMOD_TILE_BAND2 : r));
}

// STG: the o-projection's / down projection's epilogue inputs are staged in shared
// memory by one more warp (the loader), see EpiStage.
template <int BN, int MODE, bool STG = false, int LAY = LAY_KK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS + (STG ? 32 : 0), 1)
gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmAr,
                const TcArgs args) {
  static_assert(!STG || MODE == EPI_OPROJ || MODE == EPI_DOWN_SCATTER, "staged inputs");
  static_assert(!STG || EPI_WARPS == 8, "a staged buffer is released by eight warps");
  using C = Cfg2S<BN, STG ? stg_bytes<MODE>() : 0>;
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = sA + C::STAGES * C::A_BYTES;
  const uint32_t sStg = sB + C::STAGES * C::B_BYTES;   // 1024-aligned: stages are
  const uint32_t sBar = sStg + (STG ? stg_bytes<MODE>() : 0);
  const uint32_t sTmem = sBar + 8 * (2 * C::STAGES + 8);
  // staged inputs: IN_FULL(u) (the loader's copies landed), IN_EMPTY(u) (eight epilogue
  // warps read the buffer)
  const uint32_t IN_FULL0 = sBar + 8 * (2 * C::STAGES + 4), IN_EMPTY0 = IN_FULL0 + 16;
  static_assert(8 * (2 * C::STAGES + 8) + 12 <= 256, "barrier block overflows");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (sTmem - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (sTmem - base) + 8);
#define FULL(s) (sBar + 8u * (s))
#define EMPTY(s) (sBar + 8u * (C::STAGES + (s)))
#define ACC_FULL(a) (sBar + 8u * (2 * C::STAGES + (a)))
#define ACC_EMPTY(a) (sBar + 8u * (2 * C::STAGES + 2 + (a)))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (args.K + BK - 1) / BK;
  const uint32_t rank = cluster_ctarank();
  const int pair = (int)cluster_id_x(), npairs = (int)cluster_count_x();

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(FULL(s), 1);     // used in CTA 0: its producer's arrival + both CTAs' bytes
      mbar_init(EMPTY(s), 1);    // one multicast commit per use
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(ACC_FULL(a), 1);
      mbar_init(ACC_EMPTY(a), 2 * EPI_WARPS);   // used in CTA 0: one lane per epilogue warp
      if (STG) {
        mbar_init(IN_FULL0 + 8 * a, 1);
        mbar_init(IN_EMPTY0 + 8 * a, EPI_WARPS);
      }
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB0);
    if (STG) {
      prefetch_tensormap(&tmX);
      if (MODE == EPI_DOWN_SCATTER) prefetch_tensormap(&tmAr);
    }
    if (MODE == EPI_SWIGLU || args.n_split1 < args.N) prefetch_tensormap(&tmB1);
    if (MODE != EPI_SWIGLU && args.n_split2 < args.N) prefetch_tensormap(&tmB2);
  }
  if (warp == 1) tmem_alloc_pair(sTmem, C::TMEM_COLS);
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers initialised, TMEM address written
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // everything above overlapped the previous kernel's tail

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      for (int tile = pair; tile < args.tiles && !*abort_flag; tile += npairs) {
        int m_blk, n_blk;
        tile_coords(args, args.tiles_m, tile, m_blk, n_blk, args.band2);
        const int m0 = m_blk * (2 * BM) + (int)rank * BM;
        const CUtensorMap* mp = &tmB0;
        int brow = n_blk * BN;
        if (MODE == EPI_SWIGLU) {
          if (rank) mp = &tmB1;          // up rows in CTA 1, gate rows in CTA 0
          brow = n_blk * (BN / 2);
        } else {
          if (brow >= args.n_split2) {
            mp = &tmB2;
            brow -= args.n_split2;
          } else if (brow >= args.n_split1) {
            mp = &tmB1;
            brow -= args.n_split1;
          }
          brow += (int)rank * (BN / 2);
        }
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait_cluster(EMPTY(s), ph ^ 1u, abort_flag, args.status)) break;
          const uint32_t full0 = mapa_shared(FULL(s), 0);
          if (rank == 0) mbar_arrive_expect_tx(FULL(s), 2 * C::STAGE_BYTES);
          load_operand_pair<kAMn<LAY>>(sA + s * C::A_BYTES, &tmA, full0, kb * BK, m0, BM);
          int k0 = kb * BK;
          const CUtensorMap* bm = mp;
          if constexpr (kBMn<LAY>) bm = b_map_at_k(args, &tmB0, &tmB1, &tmB2, kb, k0);
          load_operand_pair<kBMn<LAY>>(sB + s * C::B_BYTES, bm, full0, k0, brow, BN / 2);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN) | kIdescMajor<LAY>;
      constexpr uint64_t astep = kOperandStep<kAMn<LAY>>, bstep = kOperandStep<kBMn<LAY>>;
      int it = 0, lt = 0;
      for (int tile = pair; tile < args.tiles && !*abort_flag; tile += npairs, ++lt) {
        const int acc = lt & 1;
        const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
        if (!mbar_wait_cluster(ACC_EMPTY(acc), aph ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % C::STAGES;
          const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
          if (!mbar_wait_cluster(FULL(s), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = operand_desc<kAMn<LAY>>(sA + s * C::A_BYTES);
          const uint64_t bd = operand_desc<kBMn<LAY>>(sB + s * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_bf16_pair(d_tmem, ad + astep * k, bd + bstep * k, idesc, (kb | k) != 0 ? 1u : 0u);
          mma_commit_pair(EMPTY(s));
        }
        if (!ok) break;
        mma_commit_pair(ACC_FULL(acc));
      }
    }
  } else if (STG && warp == 2 + EPI_WARPS) {
    // The loader: for each tile of this CTA and each 64-column pair of its chunks, the
    // CTA's 128 x rows by TMA gather4 (lane l: tile rows 4l .. 4l+3, at their stream
    // rows) and, for the down projection, the 128 a rows as one tile, into buffer
    // u = pair index & 1 once the epilogue has released it.
    int gp = 0;
    bool run = true;
    for (int tile = pair; run && tile < args.tiles; tile += npairs) {
      int m_blk, n_blk;
      tile_coords(args, args.tiles_m, tile, m_blk, n_blk, args.band2);
      const int m0 = m_blk * (2 * BM) + (int)rank * BM;
      int r[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {   // rows past M repeat a valid row; never used
        const int m = m0 + 4 * lane + q;
        r[q] = m < args.M ? (int)stream_row_of(args.e, m) : 0;
      }
      for (int cp = 0; cp < BN / STG_COLS; ++cp, ++gp) {
        const int u = gp & 1;
        int ok = 1;
        if (lane == 0) {
          ok = !*abort_flag &&
               mbar_wait(IN_EMPTY0 + 8 * u, ((uint32_t)(gp >> 1) & 1u) ^ 1u, abort_flag,
                         args.status);
          if (ok) mbar_arrive_expect_tx(IN_FULL0 + 8 * u, stg_tensors<MODE>() * STG_TILE);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          run = false;
          break;
        }
        const uint32_t buf = sStg + (uint32_t)(u * stg_tensors<MODE>() * STG_TILE);
        const int col = n_blk * BN + cp * STG_COLS;
        tma_gather4(buf + lane * 512, &tmX, IN_FULL0 + 8 * u, col, r[0], r[1], r[2], r[3]);
        if (MODE == EPI_DOWN_SCATTER && lane == 0)
          tma_load_2d(buf + STG_TILE, &tmAr, IN_FULL0 + 8 * u, col, m0);
      }
    }
  } else {
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31 belong to this warp
    int lt = 0;
    for (int tile = pair; tile < args.tiles; tile += npairs, ++lt) {
      const int acc = lt & 1;
      const uint32_t aph = (uint32_t)(lt >> 1) & 1u;
      int m_blk, n_blk;
      tile_coords(args, args.tiles_m, tile, m_blk, n_blk, args.band2);
      const int trow0 = m_blk * (2 * BM) + (int)rank * BM;
      const int wrow0 = trow0 + quad * 32;
      if (!STG) epi_prefetch<BN, MODE>(args, args.M, wrow0 + lane, n_blk, (warp - 2) / 4);
      if (!mbar_wait_cluster(ACC_FULL(acc), aph, abort_flag, args.status)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN);
      if (STG) {
        const EpiStage st{sStg, IN_FULL0, IN_EMPTY0, lt * (BN / STG_COLS), abort_flag,
                          args.status};
        if (!epilogue_tile<BN, MODE, false, true>(args, args.M, wrow0, lane, n_blk, t_row,
                                                  (warp - 2) / 4, EPI_WARPS / 4, 0, 1.0f, &st,
                                                  trow0))
          break;
      } else {
        epilogue_tile<BN, MODE>(args, args.M, wrow0, lane, n_blk, t_row, (warp - 2) / 4,
                                EPI_WARPS / 4);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(ACC_EMPTY(acc), 0));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // A wait ran out: give copies and MMAs still in flight time to land before the
    // shared memory and TMEM are released.
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 20000000ull) {
    }
  }
  cluster_sync_all();   // neither CTA leaves while the pair's MMAs or arrivals may touch it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
#undef FULL
#undef EMPTY
#undef ACC_FULL
#undef ACC_EMPTY
}

// ---------------------------------------------------------------- host side

// 2-D bf16 tensor map over a row-major [rows, inner] matrix with row stride `ld`
// elements; box = box_rows x 64 elements, 128-byte swizzle, zero fill outside.
bool make_map(CUtensorMap* m, const void* base, int64_t inner, int64_t rows, int64_t ld,
              int box_rows) {
  const int64_t dims[2] = {inner, rows};
  const int64_t strides[1] = {ld * 2};
  const int box[2] = {BK, box_rows};
  return tma_map_bf16(m, base, 2, dims, strides, box);
}

// 3-D bf16 tensor map over a row-major [rows, mn] matrix (mn a multiple of 64) read as
// (64 columns, row, 64-column chunk): a box of 64 rows x `chunks` chunks lands as
// `chunks` consecutive 64 x 64 swizzled tiles, the MN-major operand layout.
bool make_map_mn(CUtensorMap* m, const void* base, int64_t mn, int64_t rows, int64_t ld,
                 int chunks) {
  const int64_t dims[3] = {64, rows, mn / 64};
  const int64_t strides[2] = {ld * 2, 128};
  const int box[3] = {64, BK, chunks};
  return tma_map_bf16(m, base, 3, dims, strides, box);
}

int g_sms = 0;
int sm_count() {
  if (!g_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms <= 0) g_sms = 1;
  }
  return g_sms;
}

// Tensor maps and kernel arguments for tiles of tile_m x BN. B tiles are loaded
// b_box rows at a time (BN, or BN / 2 when a CTA pair splits them).
template <int BN>
bool setup(const Ctx& c, const GemmTcProblem& p, const Epilogue& e, int tile_m, int b_box,
           CUtensorMap& mA, CUtensorMap& mB0, CUtensorMap& mB1, CUtensorMap& mB2, TcArgs& a) {
  memset(&mB1, 0, sizeof(mB1));
  memset(&mB2, 0, sizeof(mB2));
  a.g_idx = p.gather_idx;
  a.g_T = p.gather_T;
  a.g_n = p.gather_n;
  a.g_gamma = (const __nv_bfloat16*)p.gather_gamma;
  a.g_eps = p.gather_eps;
  if (p.gather_idx) {   // the stream's rows, one-row boxes for gather4
    if (!make_map(&mA, p.A, p.K, p.gather_rows, p.lda, 1)) return false;
  } else if (p.a_mn) {  // [K, M]: a CTA's BM rows, 64 x 64 tiles, in one load
    if (!make_map_mn(&mA, p.A, p.M, p.K, p.lda, BM / 64)) return false;
  } else if (!make_map(&mA, p.A, p.K, p.M, p.lda, BM)) {
    return false;
  }
  a.M = p.M;
  a.M_dev = p.M_dev;
  a.ksplit = p.ksplit > 1 ? p.ksplit : 1;
  a.N = p.N;
  a.K = p.K;
  a.mode = e.kind;
  a.e = e;
  a.status = c.status;
  a.sk = 0;
  a.units = 0;
  a.sk_part = nullptr;
  a.sk_flag = nullptr;
  a.n_split1 = INT_MAX;
  a.n_split2 = INT_MAX;
  a.k_split1 = INT_MAX;
  a.k_split2 = INT_MAX;
  // 32-byte epilogue accesses need every row segment the epilogue touches aligned
  auto seg_ok = [](const void* base, int64_t row_bytes) {
    return ((uintptr_t)base & 31) == 0 && row_bytes % 32 == 0;
  };
  bool v8 = true;
  if (e.out && e.kind != EPI_ROUTER)
    v8 = v8 && seg_ok(e.out, (int64_t)e.ldo * (e.out_f32 ? 4 : 2));
  for (int i = 0; i < 2; ++i)
    if (e.row_split[i] > 0) v8 = v8 && seg_ok(e.out_rows[i], (int64_t)e.ldo * 4);
  if (e.out2 && e.kind == EPI_SWIGLU)   // bf16 [G | U] rows, the U half N columns on
    v8 = v8 && seg_ok(e.out2, (int64_t)e.ldo2 * 2) &&
         seg_ok((const __nv_bfloat16*)e.out2 + p.N, (int64_t)e.ldo2 * 2);
  else if (e.out2)
    v8 = v8 && seg_ok(e.out2, (int64_t)e.ldo2 * 4);
  if (e.x) v8 = v8 && seg_ok(e.x, (int64_t)e.d * 2);
  if (e.a) v8 = v8 && seg_ok(e.a, (int64_t)e.d * 2);
  a.v8 = v8 ? 1 : 0;
  a.tiles_m = (p.M + tile_m - 1) / tile_m;
  int tiles_n;
  if (e.kind == EPI_SWIGLU) {
    if (!make_map(&mB0, p.B[0], p.K, p.N, p.ldb, BN / 2)) return false;
    if (!make_map(&mB1, p.B[1], p.K, p.N, p.ldb, BN / 2)) return false;
    mB2 = mB0;
    tiles_n = (p.N + BN / 2 - 1) / (BN / 2);
  } else {
    const int rows0 = p.nB > 1 ? p.split[0] : (p.b_rows > 0 ? p.b_rows : p.N);
    if (p.b_mn) {   // [K, N] in up to three parts stacked along K: b_box / 64 tiles a load
      const int k1 = p.nB > 1 ? p.split[0] : p.K;
      const int k2 = p.nB > 2 ? p.split[1] : p.K;
      if (!make_map_mn(&mB0, p.B[0], p.N, k1, p.ldb, b_box / 64)) return false;
      if (p.nB > 1) {
        a.k_split1 = k1;
        if (!make_map_mn(&mB1, p.B[1], p.N, k2 - k1, p.ldb, b_box / 64)) return false;
      }
      if (p.nB > 2) {
        a.k_split2 = k2;
        if (!make_map_mn(&mB2, p.B[2], p.N, p.K - k2, p.ldb, b_box / 64)) return false;
      }
    } else if (!make_map(&mB0, p.B[0], p.K, rows0, p.ldb, b_box)) {
      return false;
    }
    if (p.nB > 1 && !p.b_mn) {
      a.n_split1 = p.split[0];
      const int rows1 = (p.nB > 2 ? p.split[1] : p.N) - p.split[0];
      if (!make_map(&mB1, p.B[1], p.K, rows1, p.ldb, b_box)) return false;
    }
    if (p.nB > 2 && !p.b_mn) {
      a.n_split2 = p.split[1];
      if (!make_map(&mB2, p.B[2], p.K, p.N - p.split[1], p.ldb, b_box)) return false;
    }
    if (p.nB < 2) mB1 = mB0;
    if (p.nB < 3) mB2 = mB0;
    tiles_n = (p.N + BN - 1) / BN;
  }
  a.tiles_n = tiles_n;
  a.tiles = a.tiles_m * tiles_n * a.ksplit;
  return true;
}

// Stream-K grid for a launch of `tiles` tiles of nk k-blocks: one CTA per SM (at most
// the scratch slots), and only when every CTA's share spans a whole tile's k-blocks
// (then a tile spans at most two CTAs); 0 when stream-K does not apply.
// XMOD_STREAM_K_CTAS (read at every launch) caps the grid, so that small problems
// can exercise tiles cut at many places.
int stream_k_grid(const Ctx& c, long tiles, int nk) {
  if (!c.sk_part || !c.sk_flag || c.sk_slots <= 0 || nk <= 0) return 0;
  int P = sm_count() < c.sk_slots ? sm_count() : c.sk_slots;
  const char* v = getenv("XMOD_STREAM_K_CTAS");
  if (v && *v) {
    char* end = nullptr;
    const long cap = strtol(v, &end, 10);
    if (end && *end == '\0' && cap > 0 && cap < P) P = (int)cap;
  }
  return tiles >= P ? P : 0;
}

template <int BN>
cudaError_t launch_bn(const Ctx& c, const GemmTcProblem& p, const Epilogue& e, bool sk = false) {
  using Cf = Cfg<BN>;
  if ((e.kind == EPI_ROUTER) != (BN == 32)) return cudaErrorInvalidValue;
  CUtensorMap mA, mB0, mB1, mB2;
  TcArgs a;
  if (!setup<BN>(c, p, e, BM, BN, mA, mB0, mB1, mB2, a)) return cudaErrorInvalidValue;
  if (a.tiles <= 0) return cudaSuccess;
  int grid = a.tiles < sm_count() ? a.tiles : sm_count();
  if (sk) {
    const int nk = (p.K + BK - 1) / BK;
    grid = p.M_dev || a.ksplit != 1 ? 0 : stream_k_grid(c, a.tiles, nk);
    if (grid <= 0) return cudaErrorInvalidValue;
    a.sk = 1;
    a.units = (int64_t)a.tiles * nk;
    a.sk_part = c.sk_part;
    a.sk_flag = c.sk_flag;
  }
  void (*k)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
            const TcArgs) = nullptr;
  if constexpr (BN != 32) {
    if (p.gather_idx) {   // RMSNorm of gathered rows in the A operand (STORE only)
      if (e.kind != EPI_STORE || sk) return cudaErrorInvalidValue;
      k = gemm_tc_kernel<BN, EPI_STORE, true>;
      static bool gattr = false;
      if (!gattr) {
        cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               Cf::SMEM + XF_SMEM);
        if (err != cudaSuccess) return err;
        gattr = true;
      }
      return launch_pdl(k, dim3(grid), dim3(NUM_THREADS + 32 * XF_WARPS), Cf::SMEM + XF_SMEM,
                        c.stream, mA, mB0, mB1, mB2, a);
    }
  }
  if constexpr (BN == 32) {
    k = gemm_tc_kernel<BN, EPI_ROUTER>;
  } else {
    switch (e.kind) {
      case EPI_STORE:
        k = p.a_mn   ? gemm_tc_kernel<BN, EPI_STORE, false, LAY_MM>
            : p.b_mn ? gemm_tc_kernel<BN, EPI_STORE, false, LAY_KM>
                     : gemm_tc_kernel<BN, EPI_STORE>;
        break;
      case EPI_OPROJ: k = gemm_tc_kernel<BN, EPI_OPROJ>; break;
      case EPI_SWIGLU: k = gemm_tc_kernel<BN, EPI_SWIGLU>; break;
      case EPI_DOWN_SCATTER: k = gemm_tc_kernel<BN, EPI_DOWN_SCATTER>; break;
      default: return cudaErrorInvalidValue;
    }
  }
  if (!k) return cudaErrorInvalidValue;
  static bool attr_set[3][5] = {};   // [layout][epilogue]: one entry per kernel
  const int mn = p.a_mn ? LAY_MM : p.b_mn ? LAY_KM : LAY_KK;
  if (!attr_set[mn][e.kind]) {
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    if (err != cudaSuccess) return err;
    attr_set[mn][e.kind] = true;
  }
  return launch_pdl(k, dim3(grid), dim3(NUM_THREADS), Cf::SMEM, c.stream, mA, mB0, mB1, mB2, a);
}

// CTA pairs that fit on the device at once with the pair kernel's shared memory
// (SMs of a GPC that cannot be paired stay unused).
template <int BN>
int max_pairs() {
  static int cached = 0;
  if (!cached) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)sm_count());
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = Cfg2<BN>::SMEM;
    auto k = gemm_tc2_kernel<BN, EPI_STORE>;
    int n = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg2<BN>::SMEM) ==
            cudaSuccess &&
        cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n > 0)
      cached = n;
    else
      cached = sm_count() / 2;
    (void)cudaGetLastError();
  }
  return cached;
}

// Staged epilogue inputs on the CTA-pair kernel (o-projection, down projection); the
// environment variable XMOD_EPI_STAGE=0, read at every launch, turns them off.
bool epi_stage_enabled() {
  const char* v = getenv("XMOD_EPI_STAGE");
  return !(v && v[0] == '0' && v[1] == '\0');
}

template <int BN>
cudaError_t launch_bn2(const Ctx& c, const GemmTcProblem& p, const Epilogue& e) {
  if (e.kind == EPI_ROUTER) return cudaErrorInvalidValue;
  CUtensorMap mA, mB0, mB1, mB2, mX, mAr;
  memset(&mX, 0, sizeof(mX));
  memset(&mAr, 0, sizeof(mAr));
  TcArgs a;
  if (!setup<BN>(c, p, e, 2 * BM, BN / 2, mA, mB0, mB1, mB2, a)) return cudaErrorInvalidValue;
  if (a.tiles <= 0) return cudaSuccess;
  a.band2 = band2_rows(p.K);
  // staged inputs: the stream's rows (one-row boxes for gather4) and a's 128-row tiles
  bool stg = epi_stage_enabled() && !e.tok && e.x && e.n_per_seq > 0 && e.T >= e.n_per_seq &&
             p.M % e.n_per_seq == 0 && p.N == e.d &&
             (e.kind == EPI_OPROJ || (e.kind == EPI_DOWN_SCATTER && e.a));
  if (stg) {
    const int64_t x_rows = (int64_t)(p.M / e.n_per_seq) * e.T;
    stg = make_map(&mX, e.x, e.d, x_rows, e.d, 1) &&
          (e.kind != EPI_DOWN_SCATTER || make_map(&mAr, e.a, e.d, p.M, e.d, BM));
  }
  void (*k)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
            const CUtensorMap, const CUtensorMap, const TcArgs) = nullptr;
  int smem = 0, threads = NUM_THREADS;
  switch (e.kind) {
    case EPI_STORE:
      if constexpr (BN == 256) {   // MN-major B halves need whole 64-row boxes
        k = p.a_mn   ? gemm_tc2_kernel<BN, EPI_STORE, false, LAY_MM>
            : p.b_mn ? gemm_tc2_kernel<BN, EPI_STORE, false, LAY_KM>
                     : gemm_tc2_kernel<BN, EPI_STORE>;
      } else {
        if (p.b_mn) return cudaErrorInvalidValue;
        k = gemm_tc2_kernel<BN, EPI_STORE>;
      }
      smem = Cfg2<BN>::SMEM;
      break;
    case EPI_SWIGLU:
      if constexpr (BN == 256) {   // gate / up halves of 128 columns each
        k = gemm_tc2_kernel<BN, EPI_SWIGLU>;
        smem = Cfg2<BN>::SMEM;
        break;
      } else {
        return cudaErrorInvalidValue;
      }
    case EPI_OPROJ:
      if (stg) {
        k = gemm_tc2_kernel<BN, EPI_OPROJ, true>;
        smem = Cfg2S<BN, stg_bytes<EPI_OPROJ>()>::SMEM;
        threads += 32;
      } else {
        k = gemm_tc2_kernel<BN, EPI_OPROJ>;
        smem = Cfg2<BN>::SMEM;
      }
      break;
    case EPI_DOWN_SCATTER:
      if (stg) {
        k = gemm_tc2_kernel<BN, EPI_DOWN_SCATTER, true>;
        smem = Cfg2S<BN, stg_bytes<EPI_DOWN_SCATTER>()>::SMEM;
        threads += 32;
      } else {
        k = gemm_tc2_kernel<BN, EPI_DOWN_SCATTER>;
        smem = Cfg2<BN>::SMEM;
      }
      break;
    default: return cudaErrorInvalidValue;
  }
  static bool attr_set[3][2][4] = {};   // [layout][staged inputs][epilogue]: per kernel
  const int mn = p.a_mn ? LAY_MM : p.b_mn ? LAY_KM : LAY_KK;
  if (!attr_set[mn][stg][e.kind]) {
    cudaError_t err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    attr_set[mn][stg][e.kind] = true;
  }
  const int pairs = a.tiles < max_pairs<BN>() ? a.tiles : max_pairs<BN>();
  return launch_pdl(k, dim3(2 * pairs), dim3(threads), smem, c.stream, mA, mB0, mB1, mB2, mX,
                    mAr, a);
}

// Tile widths a problem may use: the q|k|v boundaries must fall on tile edges.
bool bn_ok(const GemmTcProblem& p, const Epilogue& e, int bn) {
  if (e.kind == EPI_SWIGLU) return bn == 256;   // (pair tiles of 192 included)
  // Router logits: 32-wide tiles only, so that a logit's arithmetic never depends on
  // how many router vectors share its launch.
  if (e.kind == EPI_ROUTER) return bn == 32 && p.N <= 32 && p.nB == 1;
  if (p.b_mn) return true;   // its B parts are stacked along K, not N
  for (int i = 1; i < p.nB; ++i)
    if (p.split[i - 1] % bn) return false;
  return true;
}

}  // namespace

bool gemm_tc_supported(const GemmTcProblem& p, const Epilogue& e) {
  if (!tma_available()) return false;
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return false;
  if (p.gather_idx &&
      (e.kind != EPI_STORE || p.M_dev || p.gather_n <= 0 || p.gather_T < p.gather_n ||
       p.gather_rows <= 0 || p.lda != p.K || !p.gather_gamma ||
       ((uintptr_t)p.gather_gamma & 15)))
    return false;
  if (p.a_mn || p.b_mn) {   // plain stores; MN-major A only with MN-major B of one part
    if (!p.b_mn || e.kind != EPI_STORE || p.gather_idx || p.ksplit > 1 || p.b_rows ||
        (p.a_mn && p.nB != 1))
      return false;
    // MN-major operands are read in 64-row chunks of whole rows
    if (p.N % 64 || (p.a_mn && p.M % 64)) return false;
    // parts of B stacked along K: whole 64-deep k-blocks each
    if (p.nB > 1 && (p.split[0] % BK || p.split[0] <= 0 || p.split[0] >= p.K)) return false;
    if (p.nB > 2 && (p.split[1] % BK || p.split[1] <= p.split[0] || p.split[1] >= p.K))
      return false;
  }
  if ((p.K % 8 && !(p.a_mn && p.b_mn)) || p.lda % 8 || p.ldb % 8) return false;
  if (p.N % 8 && e.kind != EPI_ROUTER) return false;   // the others store 8-column groups
  if (p.b_rows && (p.b_rows < p.N || p.nB != 1)) return false;
  if (p.ksplit > 1 && (e.kind != EPI_ROUTER || p.ksplit > (p.K + BK - 1) / BK)) return false;
  if (((uintptr_t)p.A & 15) || ((uintptr_t)p.B[0] & 15)) return false;
  if (e.kind == EPI_SWIGLU && (p.nB != 2 || ((uintptr_t)p.B[1] & 15))) return false;
  if (e.kind != EPI_SWIGLU)
    for (int i = 1; i < p.nB; ++i)
      if ((uintptr_t)p.B[i] & 15) return false;
  return bn_ok(p, e, 32) || bn_ok(p, e, 128) || bn_ok(p, e, 256);
}

// The pair threshold in waves; the environment variable XMOD_PAIR_MIN_WAVES (read at
// every launch) overrides it, e.g. 0 to run every eligible GEMM on CTA pairs.
int pair_min_waves() {
  const char* v = getenv("XMOD_PAIR_MIN_WAVES");
  if (v && *v) {
    char* end = nullptr;
    const long w = strtol(v, &end, 10);
    if (end && *end == '\0' && w >= 0 && w < 1000000) return (int)w;
  }
  return XMOD_PAIR_MIN_WAVES;
}

// Pair tile width: XMOD_PAIR_BN=256 or 192 (read at every launch) limits the CTA-pair
// tilings to that width; otherwise the cheaper of the two is taken.
int pair_bn_forced() {
  const char* v = getenv("XMOD_PAIR_BN");
  if (v && strcmp(v, "256") == 0) return 256;
  if (v && strcmp(v, "192") == 0) return 192;
  return 0;
}

// Stream-K choice: XMOD_STREAM_K=1 (read at every launch) runs every GEMM it applies
// to as stream-K; otherwise none.
int stream_k_mode() {
  const char* v = getenv("XMOD_STREAM_K");
  if (v && (v[0] == '0' || v[0] == '1') && v[1] == '\0') return v[0] - '0';
  return -1;
}

cudaError_t launch_gemm_tc(const Ctx& c, const GemmTcProblem& p, const Epilogue& e) {
  if (e.kind == EPI_ROUTER) return launch_bn<32>(c, p, e);
  const int sms = sm_count();
  // The single-CTA tile width with the shortest estimated time: waves x tile width,
  // with narrower tiles charged for their higher shared-memory traffic per FLOP.
  const int tiles_m = (p.M + BM - 1) / BM;
  const int widths[3] = {256, 192, 128};
  const double cost_per_col[3] = {XMOD_COST_256, XMOD_COST_192, XMOD_COST_128};
  int best = -1;
  double best_cost = 0.0;
  for (int i = 0; i < 3; ++i) {
    const int bn = widths[i];
    if (!bn_ok(p, e, bn)) continue;
    const int cols = e.kind == EPI_SWIGLU ? bn / 2 : bn;
    const long tiles = (long)tiles_m * ((p.N + cols - 1) / cols);
    const double cost = (double)((tiles + sms - 1) / sms) * bn * cost_per_col[i];
    if (best < 0 || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  // CTA pairs on 256 x 256 tiles: each SM of a pair streams half of the B tile, so a
  // pair tile costs about 18% less time per SM than a 128 x 256 single-CTA tile (cost
  // XMOD_COST_PAIR per column in the units above), for about 5 us more per launch.
  // They run from six waves up (gate/up at M = 4096, every dense-layer GEMM), and below
  // that when the same waves-times-width estimate puts them at least XMOD_PAIR_MARGIN
  // ahead of the best single-CTA tiling. Measured on GB300 at M = 4096: with d = 2048,
  // d_ff = 5632 (2 pair waves against 2 single waves of 256) down 83.6 -> 70.2 us,
  // q|k|v 43.8 -> 40.2, o-proj 41.6 -> 39.4; with d = 1536, d_ff = 4096 (a second pair
  // wave on a quarter of the pairs against 192-wide single tiles) pairs lost 2-4 us on
  // the o-proj and down GEMMs, which the margin keeps single. 256 x 192 pair tiles
  // (cost XMOD_COST_PAIR192) serve those: at d = 1536 they give two waves of 128 pair
  // tiles, and measured o-proj 30.6 -> 29.0 us, down 53.1 -> 50.8 us against the
  // 192-wide single-CTA tiles.
  if (p.gather_idx) {   // the gathered-RMSNorm variant exists for single-CTA tiles only
    if (best == 256) return launch_bn<256>(c, p, e);
    if (best == 192) return launch_bn<192>(c, p, e);
    return launch_bn<128>(c, p, e);
  }
  if (XMOD_GEMM_PAIRS && p.M > BM && !p.M_dev) {
    // the cheaper of the 256 x 256 and 256 x 192 pair tilings
    const long ptiles_m = (p.M + 2 * BM - 1) / (2 * BM);
    int pbn = 0;
    long ptiles = 0, pairs = 0;
    double pair_cost = 0.0;
    const int forced = pair_bn_forced();
    for (int bn : {256, 192}) {
      if (!bn_ok(p, e, bn) || (forced && bn != forced)) continue;
      if (p.b_mn && bn != 256) continue;   // a CTA's B half must be whole 64-row boxes
      const int cols = e.kind == EPI_SWIGLU ? bn / 2 : bn;
      const long tiles = ptiles_m * ((p.N + cols - 1) / cols);
      const long np = bn == 256 ? max_pairs<256>() : max_pairs<192>();
      const double cost = (double)((tiles + np - 1) / np) * bn *
                          (bn == 256 ? XMOD_COST_PAIR : XMOD_COST_PAIR192);
      if (!pbn || cost < pair_cost) {
        pbn = bn;
        ptiles = tiles;
        pairs = np;
        pair_cost = cost;
      }
    }
    if (pbn && (ptiles >= (long)pair_min_waves() * pairs ||
                (best > 0 && pair_cost * (1.0 + XMOD_PAIR_MARGIN) <= best_cost)))
      return pbn == 256 ? launch_bn2<256>(c, p, e) : launch_bn2<192>(c, p, e);
  }
  // Stream-K at 256-wide tiles, on request only: on the A4K8 block's sparse-layer GEMMs
  // (1.3-2.1 waves) it measured 10-50% slower than the tiling above -- storing and
  // re-reading the fp32 partial tiles (128 KB per CTA, all CTAs at once) costs more
  // than the partial last wave it removes.
  if (stream_k_mode() == 1 && bn_ok(p, e, 256) && !p.M_dev && p.ksplit <= 1 && !p.a_mn &&
      !p.b_mn) {
    const int cols = e.kind == EPI_SWIGLU ? 128 : 256;
    const long tiles = (long)tiles_m * ((p.N + cols - 1) / cols);
    if (stream_k_grid(c, tiles, (p.K + BK - 1) / BK) > 0) return launch_bn<256>(c, p, e, true);
  }
  if (best == 256) return launch_bn<256>(c, p, e);
  if (best == 192) return launch_bn<192>(c, p, e);
  return launch_bn<128>(c, p, e);
}

}  // namespace xmod
