// Host-side launchers shared between the translation units of the library.
// Every launcher only enqueues work on ctx.stream and returns the launch status.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "xmod.h"

namespace xmod {

struct Ctx {
  cudaStream_t stream;
  int* status;  // device status word (first error wins)
  // Stream-K scratch of the tensor-core GEMMs: sk_slots partial accumulators of
  // 128 x 256 fp32 and as many flags, all zero between launches. NULL: no stream-K.
  float* sk_part = nullptr;
  int* sk_flag = nullptr;
  int sk_slots = 0;
};

// Launch with programmatic stream serialization: the kernel may begin while the
// previous kernel on the stream drains; it must call pdl_wait() (common.cuh) before
// touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- TMA tensor maps

bool tma_available();
// bf16 tensor map of the given rank (2 or 3): dims[0] is the contiguous extent,
// strides_bytes[i] the byte stride of dimension i+1; box in elements; 128-byte
// swizzle; reads outside the tensor return zeros.
bool tma_map_bf16(CUtensorMap* m, const void* base, int rank, const int64_t* dims,
                  const int64_t* strides_bytes, const int* box);

// ---------------------------------------------------------------- measurement

void count_launch();

// Records a CUDA event pair around one launch on `s` while profiling is enabled.
class ProfScope {
 public:
  ProfScope(const char* kind, cudaStream_t s);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  const char* kind_;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
};

// ---------------------------------------------------------------- routing and row kernels

// s[i] = w_r . x_i + bias[i] (fp32), r[i] = sigmoid(s[i]) if r != NULL.
cudaError_t launch_router(const Ctx& c, xmod_dtype dt, int64_t rows, int d, const void* x,
                          const void* w_r, const float* bias, float* s, float* r);

// Largest topk supported T (keys held in shared memory).
int topk_max_T();

// Token-choice bias state of a sparse-dense block (all pointers may be NULL).
//   count [B, T]  times each token was selected by the block's earlier sparse layers;
//                 the layer ranks s - bias_step * count, and its selection adds 1;
//   last  [B, T]  index of the last sparse layer that selected the token;
//   stats [B, 4]  this layer's selected count, tokens with a ranked logit >= 0,
//                 tokens where the two rules agree, and selected tokens the previous
//                 sparse layer (index layer - 1) also selected.
struct RouteTrack {
  int32_t* count = nullptr;
  int32_t* last = nullptr;
  float bias_step = 0.0f;
  int layer = 0;
  int32_t* stats = nullptr;
};

// Per-sequence top-n of s [B, T]; ties to the lower position; ascending idx [B, n].
// r_sel [B, n] = sigmoid(ranked logit at idx) if not NULL. With nplanes > 1 the logit
// is the in-order sum of the planes s + k * plane (partial sums of a k-split GEMM).
cudaError_t launch_topk(const Ctx& c, int B, int T, int n, const float* s, int32_t* idx,
                        float* r_sel, const RouteTrack* tr = nullptr, int nplanes = 1,
                        int64_t plane = 0);
// QK-norm (gains [hd], NULL: none) and rotary embedding (theta, 0: none), in place, of
// q_heads heads from column q_col0 and k_heads heads from k_col0 (hd columns each) in
// rows x [M, ld] (only m < *M_dev if given). Row m sits at position pos_idx[m], else
// pos_tok[m] % seqT, else m % seqT.
cudaError_t launch_qk_transform(const Ctx& c, xmod_dtype dt, int64_t M, const int32_t* M_dev,
                                void* x, int ld, int q_col0, int q_heads, const void* q_gain,
                                int k_col0, int k_heads, const void* k_gain, int hd, float eps,
                                float theta, const int32_t* pos_idx, const int32_t* pos_tok,
                                int seqT);

// Backward of launch_qk_transform (all M rows): g [M, ld], the gradient at the
// transformed q (from q_col0) and k (from k_col0) heads, becomes in place the gradient
// at the projections pre [M, ldp] (q heads from column 0, k heads after them); dgq / dgk
// [M, hd] fp32 (NULL: no such gain) receive each row's gain gradient over its heads.
cudaError_t launch_qk_transform_bwd(const Ctx& c, xmod_dtype dt, int64_t M, void* g, int ld,
                                    int q_col0, int q_heads, const void* q_gain, int k_col0,
                                    int k_heads, const void* k_gain, const void* pre, int ldp,
                                    int hd, float eps, float theta, const int32_t* pos_idx,
                                    int seqT, float* dgq, float* dgk);

// Causal threshold rule over s [B, T] (ranked logit s - bias_step * count >= 0):
// compact rows tok [<= B*T] (= b * T + t, sequence then position order), r_sel
// [<= B*T], seq_count [B], seq_off [B] and the total in *M_out (all device).
// scratch_pos [B*T] int32 and scratch_gate [B*T] fp32 hold each sequence's picks
// before the compaction. Two launches (counting, one CTA per sequence; compaction).
cudaError_t launch_threshold_select(const Ctx& c, int B, int T, const float* s, int32_t* tok,
                                    float* r_sel, int32_t* seq_count, int32_t* seq_off,
                                    int32_t* M_out, const RouteTrack* tr, int nplanes,
                                    int64_t plane, int32_t* scratch_pos, float* scratch_gate);
// update_hist [B, max_count + 1]: histogram of count [B, T] per sequence.
cudaError_t launch_count_hist(const Ctx& c, int B, int T, int max_count, const int32_t* count,
                              int32_t* update_hist);

// xs[b*n + j] = x[b, idx[b, j]] (idx NULL: identity, n == T).
cudaError_t launch_gather(const Ctx& c, xmod_dtype dt, int B, int T, int n, int d,
                          const void* x, const int32_t* idx, void* xs);

// Compact rows with a variable count (threshold routing): row m reads stream row
// tok[m], and only rows below *M_dev exist. Both NULL: the fixed layout.
struct RowMap {
  const int32_t* tok = nullptr;
  const int32_t* M_dev = nullptr;
  __device__ __forceinline__ int64_t rows(int64_t M) const {
    if (!M_dev) return M;
    const int64_t m = *M_dev;
    return m < M ? m : M;
  }
};

// u[b*n + j] = RMSNorm(x[b, idx[b, j]]) * gamma (idx NULL: identity); with rm.tok,
// u[m] = RMSNorm(x[tok[m]]) * gamma for the rows rm gives.
cudaError_t launch_gather_rmsnorm(const Ctx& c, xmod_dtype dt, int B, int T, int n, int d,
                                  const void* x, const int32_t* idx, const void* gamma,
                                  float eps, void* u, RowMap rm = RowMap{});

// out[m] = RMSNorm(h[m]) * gamma for fp32 rows h [M, d] (only m < *M_dev if given);
// out in the element type.
cudaError_t launch_rmsnorm_f32in(const Ctx& c, xmod_dtype dt, int64_t M, int d, const float* h,
                                 const void* gamma, float eps, void* out,
                                 const int32_t* M_dev = nullptr);

// Gated residual in place, see xmod_gated_scatter. gate < 0: dense update x + a + f.
// Copy of the caller's positions idx [B * n] with every row that is out of [0, T) or
// not above the previous row of its sequence clamped into range, recorded as
// XMOD_ERR_DEVICE_CHECK in the status word.
cudaError_t launch_idx_sanitize(const Ctx& c, int B, int T, int n, const int32_t* idx,
                                int32_t* out);
cudaError_t launch_gated_scatter(const Ctx& c, xmod_dtype dt, int B, int T, int n, int d,
                                 void* x, const int32_t* idx, const float* r_sel, const void* a,
                                 const void* f, float varsigma, int gate);

// Up to kMax row pointers passed by value to a kernel.
struct RowPtrs {
  static constexpr int kMax = 32;
  const void* p[kMax];
};
// dst [total, d] bf16 = the `count` rows, then zero rows up to `total`.
cudaError_t launch_stack_rows(const Ctx& c, const RowPtrs& rows, int count, int total, int d,
                              void* dst);

// ---------------------------------------------------------------- GEMM with fused epilogues

enum EpiKind {
  EPI_STORE = 0,         // out[m, n] = acc
  EPI_OPROJ = 1,         // out[m, n] = a = acc if out; out2[m, n] = h = x_row(m)[n] + acc
                         // (fp32) if out2
  EPI_SWIGLU = 2,        // out[m, n] = silu(acc_gate) * acc_up
  EPI_DOWN_SCATTER = 3,  // x_row(m)[n] = gated residual of (a[m, n], f = acc);
                         // also out[m, n] = that new row value when out is set
  EPI_ROUTER = 4,        // out[n * ldo + stream token of m] = acc + bias[token] (fp32);
                         // tensor-core path only, 32-wide tiles, any N <= 32
};

// Compact row m of a block belongs to sequence b = m / n_per_seq at position
// t = idx ? idx[m] : m % n_per_seq; its stream row is x[(b * T + t) * d].
struct Epilogue {
  int kind = EPI_STORE;
  void* out = nullptr;
  int ldo = 0;
  void* out2 = nullptr;          // OPROJ: h (fp32); SWIGLU: the pre-activations [G | U]
  int ldo2 = 0;                  //   (bf16 [M, 2N]) when not NULL
  void* x = nullptr;            // residual stream [B, T, d] (read for OPROJ, updated for DOWN)
  const int32_t* idx = nullptr;
  int T = 0, n_per_seq = 0, d = 0;
  // Variable tokens per sequence (threshold routing): the stream row of compact row m
  // is tok[m] (= b * T + t), and seq_off[b] is sequence b's first compact row.
  const int32_t* tok = nullptr;
  const int32_t* seq_off = nullptr;
  const void* a = nullptr;      // DOWN: the attention residual a [M, d] (the layer's dtype,
                                //       row stride d); NULL: none (a = 0)
  const float* r_sel = nullptr; // DOWN: gates [M]
  const float* bias = nullptr;  // ROUTER: per-token logit bias [B*T] or NULL (k slice 0)
  int64_t plane = 0;            // ROUTER with k slices: elements between slice planes
  // RMSNorm2 folded into the GEMMs (tensor-core path, norm_d % 128 == 0): OPROJ also
  // writes out3[m, n] = bf16(h * g2[n]) and, per 32-column chunk c, the chunk's
  // sum of h^2 to rowss[m * norm_d / 32 + c]; SWIGLU then adds a row's chunk sums in
  // order (deterministic, unlike atomics) and scales both accumulators of the row by
  // rsqrt(sum / norm_d + eps) -- RMSNorm(h) * g2 projected, by linearity.
  void* out3 = nullptr;
  const void* g2 = nullptr;
  float* rowss = nullptr;
  float eps = 0.0f;
  int norm_d = 0;
  float varsigma = 1.0f;
  int gate = -1;                // DOWN: XMOD_GATE_XMOD, XMOD_GATE_MOD, or -1 for dense
  // STORE (tensor-core path): columns >= vt_col0 are the values v; they are written
  // transposed to vt [B, hkv, hd, vt_ld] (keys contiguous) instead of to `out`.
  void* vt = nullptr;
  int vt_col0 = 0, vt_hd = 0, vt_hkv = 0, vt_ld = 0;
  bool vt_rows = false;         // with vt: write the values' columns to `out` as well
  // STORE: write the fp32 accumulator itself (out is float [M, ldo]) instead of
  // rounding it to the layer's element type
  bool out_f32 = false;
  // STORE with out_f32: rows from row_split[0] (when > 0) go to out_rows[0] and rows from
  // row_split[1] (when > 0) to out_rows[1], renumbered from 0 there (same ldo): one
  // GEMM writes the gradients of weights stacked along M, e.g. [W_q; W_k; W_v]
  int row_split[2] = {0, 0};
  void* out_rows[2] = {nullptr, nullptr};
};

// C[M, N] = A[M, K] . B[N, K]^T (fp32 accumulate), then the epilogue. For
// EPI_SWIGLU, B2 [N, K] is the up projection and B the gate projection.
cudaError_t launch_gemm_simt(const Ctx& c, xmod_dtype dt, int M, int N, int K, const void* A,
                             int lda, const void* B, int ldb, const void* B2,
                             const Epilogue& e);

// Tensor-core (tcgen05) GEMM, bf16 only. Up to three weight tensors can feed one
// launch: accumulator columns [0, split[0]) come from B[0], [split[0], split[1])
// from B[1], the rest from B[2] (q | k | v). For EPI_SWIGLU, B[0] is the gate and
// B[1] the up projection, each [N, K].
struct GemmTcProblem {
  int M = 0, N = 0, K = 0;
  const void* A = nullptr;
  int lda = 0;
  const void* B[3] = {nullptr, nullptr, nullptr};
  int nB = 1;
  int split[2] = {0, 0};
  int ldb = 0;
  int b_rows = 0;  // rows of B[0] the tensor map spans (0: N); may exceed N
  // If set, the launch covers M rows of buffers sized for M, but only the first
  // min(*M_dev, M) rows (a count an earlier kernel wrote) are computed.
  const int32_t* M_dev = nullptr;
  // ROUTER only: the K range split in ksplit slices (at most the number of 64-deep
  // k-blocks); slice k's partial sums go to the output plane k (Epilogue::plane apart).
  int ksplit = 1;
  // RMSNorm of gathered rows fused into the A operand (STORE epilogue only): row m of A
  // is row (m / gather_n) * gather_T + gather_idx[m] of the [gather_rows, K] matrix A
  // (the residual stream, lda = K), and the GEMM computes
  //   C[m, :] = rstd_m * (x_m * gather_gamma) . B^T,  rstd_m = (mean(x_m^2) + eps)^-1/2,
  // i.e. RMSNorm(x_m) * gamma times B^T, without a gathered copy of the rows.
  const int32_t* gather_idx = nullptr;
  int gather_T = 0, gather_n = 0;
  int64_t gather_rows = 0;
  const void* gather_gamma = nullptr;
  float gather_eps = 0.f;
  // Operands stored with the contraction index as the row (STORE epilogue, one B):
  // a_mn: A is [K, M] (M contiguous, lda elements per row k); b_mn: B is [K, N]. With
  // both set K is free (rows past K read as zero), e.g. weight gradients dW = dY^T X
  // straight from token-major dY and X.
  int a_mn = 0, b_mn = 0;
};
bool gemm_tc_supported(const GemmTcProblem& p, const Epilogue& e);
cudaError_t launch_gemm_tc(const Ctx& c, const GemmTcProblem& p, const Epilogue& e);

// ---------------------------------------------------------------- attention

// Causal GQA attention within each of B sequences of n tokens.
// q [B*n, ldq] (head h at column h*hd), k and v [B*n, ldkv] (KV head g at g*hd),
// o [B*n, hq*hd].
// With qpos [B, n] (ascending positions): query row i sees the keys at positions <=
// qpos[b * n + i] among nkv keys per sequence in k, v [B * nkv, ldkv].
cudaError_t launch_attention_simt(const Ctx& c, xmod_dtype dt, int B, int n, int hq, int hkv,
                                  int hd, const void* q, int ldq, const void* k, const void* v,
                                  int ldkv, void* o, const int32_t* qpos = nullptr,
                                  int nkv = 0);

// Tensor-core attention (bf16, head_dim 128). q and k come from the q|k|v rows
// [B*n, ldq] (k of KV head g at column hq*128 + g*128); v comes transposed,
// vt [B, hkv, 128, vt_ld] with keys contiguous; o [B*n, hq*128].
// With seq_count / seq_off (device [B]): sequence b has seq_count[b] <= n tokens at
// compact rows seq_off[b] ...; its keys past seq_count[b] in vt must be finite.
// With kv (Selected-Q / full-KV): the n query rows of sequence b sit at positions
// qpos[b * n + q] (ascending); keys come from k [B, nkv, ldk] (KV head g at column
// g * 128) and vt covers nkv keys; query row q sees the keys at positions <= its own.
struct AttnKv {
  const void* k = nullptr;
  int ldk = 0;
  int nkv = 0;
  const int32_t* qpos = nullptr;
};
bool attention_tc_supported(int hd, int n, int ldq);
// lse (optional, [B*n, hq] fp32): each row's log2-sum-exp2 of its scaled logits.
cudaError_t launch_attention_tc(const Ctx& c, int B, int n, int hq, int hkv, const void* qkv,
                                int ldq, const void* vt, int vt_ld, void* o,
                                const int32_t* seq_count = nullptr,
                                const int32_t* seq_off = nullptr, const AttnKv* kv = nullptr,
                                float* lse = nullptr);

// ---------------------------------------------------------------- backward of one layer

// Attention backward on the warp-level tensor-core MMA (bf16, head_dim 64 or 128):
// qkv rows [B*n, ldq] (q, k AND v columns written), o and dO [B*n, hq*hd] bf16;
// writes lse / Dd [B*n, hq] (log2 units / <dO, o>) and dq, dk, dv into the q, k, v
// columns of dqkv [B*n, ldg].
bool attn_bwd_mma_supported(int hd, int ldq, int ldo);
// with_q false: only dk, dv (lse and Dd already written, e.g. by the tcgen05 dq kernel).
cudaError_t launch_attn_bwd_mma(const Ctx& c, int B, int n, int hq, int hkv, int hd,
                                const void* qkv, int ldq, const void* o, const void* dO,
                                float* lse, float* Dd, void* dqkv, int ldg, bool with_q = true);
// The general form (Selected-Q / full-KV): n queries per sequence at ascending positions
// qpos [B*n] (NULL: i, nk == n) over nk keys, query i seeing the keys j <= qpos[i];
// q [B*n, ldq], k [B*nk, ldk], v [B*nk, ldv] (head h / KV head g at column h*hd / g*hd);
// dq [B*n, ldgq], dk and dv [B*nk, ldgk] likewise.
cudaError_t launch_attn_bwd_mma_kv(const Ctx& c, int B, int n, int nk, const int32_t* qpos,
                                   int hq, int hkv, int hd, const void* q, int ldq,
                                   const void* k, int ldk, const void* v, int ldv, const void* o,
                                   const void* dO, float* lse, float* Dd, void* dq, int ldgq,
                                   void* dk, void* dv, int ldgk, bool with_q = true);
// dq of the attention backward on tcgen05 (bf16, head_dim 128): qkv rows [B*n, ldq] (q, k,
// v columns; the key rows serve both S = Q K^T and dQ += dS K, the latter as an MN-major
// operand), o and dO [B*n, hq*128] bf16, lse [B*n, hq] from the forward (log2 units);
// writes Dd [B*n, hq] (<dO, o>) and dq into the q columns of dqkv [B*n, ldg].
bool attn_bwd_dq_tc_supported(int hd, int ldq, int qw);
cudaError_t launch_attn_bwd_dq_tc(const Ctx& c, int B, int n, int hq, int hkv, const void* qkv,
                                  int ldq, const void* o, const void* dO, const float* lse,
                                  float* Dd, void* dqkv, int ldg, float* DdT = nullptr,
                                  int ldS = 0);
// dk and dv on tcgen05 (the query and dO rows read as stored); lseT and DdT [B*hq, ldS]
// (ldS a multiple of 64, >= n) the rows' lse and D per head; writes the k and v columns
// of dqkv [B*n, ldg].
cudaError_t launch_attn_bwd_dkv_tc(const Ctx& c, int B, int n, int hq, int hkv, const void* qkv,
                                   int ldq, const void* dO, const float* lseT, const float* DdT,
                                   int ldS, void* dqkv, int ldg);
// The general forms (Selected-Q / full-KV): n queries per sequence at ascending
// positions over nk keys, query i seeing the keys j <= its position. q [B*n, ldq]; the
// keys' and values' rows kv [B*nk, ldk] (KV head g's k at column k_col0 + g*128, v at
// v_col0 + g*128). dq_tc_kv: qpos [B*n] (NULL:
// i, nk == n), dq [B*n, ldg]. dkv_tc_kv: qposS [B, ldS] the positions padded with -1 and
// qstart [B, ceil(nk / kAttnBwdKvBlock)] the first query positioned at or after each key
// block's first key (both NULL: the compact case), dk and dv [B*nk, ldgk].
constexpr int kAttnBwdKvBlock = 128;   // keys per CTA of the tcgen05 dk / dv kernel
cudaError_t launch_attn_bwd_dq_tc_kv(const Ctx& c, int B, int n, int nk, const int32_t* qpos,
                                     int hq, int hkv, const void* q, int ldq, const void* kv,
                                     int ldk, int k_col0, int v_col0, const void* o,
                                     const void* dO, const float* lse, float* Dd, void* dq,
                                     int ldg, float* DdT, int ldS);
cudaError_t launch_attn_bwd_dkv_tc_kv(const Ctx& c, int B, int n, int nk, const int32_t* qposS,
                                      const int32_t* qstart, int hq, int hkv, const void* q,
                                      int ldq, const void* kv, int ldk, int k_col0, int v_col0,
                                      const void* dO, const float* lseT, const float* DdT,
                                      int ldS, void* dk, void* dv, int ldgk);

// Workspace bytes of run_layer_bwd for these sizes (covers a dense layer).
size_t bwd_workspace_bytes(const xmod_dims* dm);
// See xmod_layer_bwd; arguments already validated by the caller.
int run_layer_bwd(cudaStream_t stream, const xmod_dims* dm, int kind, int K, int gate,
                  const xmod_layer_weights* w, const void* x, const float* bias, const void* dy,
                  float route_coef, void* dx, const xmod_layer_grads* gr, void* ws);

}  // namespace xmod
