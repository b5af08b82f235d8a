// C ABI of the sparse-depth layer library: argument checks, workspace layout,
// and the layer / stack schedules built from the kernels.
//
// Layer semantics follow "X-MoD: Practical Scaling Laws for Sparse-Depth Routing
// Beyond Mixture-of-Depths" (reading notes): Eq. 8 router, top-1/K selection,
// attention within the selected subset, Eq. 6 / Eq. 7 gated residuals, Eq. 3
// stack layout; and "Mixture-of-Depths explained" (MoDLayer listing) for the
// floor(T * ratio) count and position-ordered gather.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "internal.h"
#include "xmod.h"

namespace xmod {

namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline size_t esize(xmod_dtype dt) { return dt == XMOD_BF16 ? 2 : 4; }
inline bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }
inline bool aligned16_or_null(const void* p) { return !p || ((uintptr_t)p & 15u) == 0; }

bool dims_ok(const xmod_dims* dm) {
  if (!dm) return false;
  if (dm->dtype != XMOD_BF16 && dm->dtype != XMOD_FP32) return false;
  if (dm->B <= 0 || dm->T <= 0 || dm->d <= 0 || dm->n_heads <= 0 || dm->n_kv_heads <= 0 ||
      dm->head_dim <= 0 || dm->d_ff <= 0)
    return false;
  if (dm->n_heads % dm->n_kv_heads) return false;
  if (dm->d % 8 || dm->d_ff % 8 || (dm->n_heads * dm->head_dim) % 8 ||
      (dm->n_kv_heads * dm->head_dim) % 8)
    return false;
  if (!(dm->rms_eps >= 0.0f) || !isfinite(dm->rms_eps)) return false;
  return true;
}

bool head_dim_supported(int hd) { return hd == 32 || hd == 64 || hd == 128; }

// Row stride (elements) of the transposed values for n tokens: 16-byte multiple.
inline int vt_ld(int n) { return (n + 7) / 8 * 8; }

// Sparse layers whose router logits one pass over the stream computes (the widest
// router GEMM tile), and the zero rows that follow them in the stacked router
// vectors (a 32-row tile read from any starting layer stays inside the buffer).
constexpr int kRouterRun = RowPtrs::kMax;
constexpr int kRouterRows = 2 * kRouterRun;
// k slices of the router-logit GEMM: the refresh after a layer has only B*T/K rows,
// so splitting the d-long dot products spreads it over 4x the SMs; the selection
// kernels add the slices' planes in order.
#ifndef XMOD_ROUTER_SPLIT
#define XMOD_ROUTER_SPLIT 4
#endif
constexpr int kRouterSplit = XMOD_ROUTER_SPLIT;
inline int router_split(const xmod_dims* dm) {
  const int nk = (dm->d + 63) / 64;
  return nk < kRouterSplit ? nk : kRouterSplit;
}

// Workspace carve-up. M rows of block scratch cover a dense layer (M = B*T).
struct Layout {
  size_t status, s, idx, r_sel, u, qkv, vt, o, h, a, hidden, wr, count, last, seq, thr, rowss,
      skflag, skpart, total;
};

// Stream-K scratch of the tensor-core GEMMs (bf16 layouts): one 128 x 256 fp32 partial
// accumulator and one flag per CTA, for up to kSkSlots CTAs (one per SM).
constexpr int kSkSlots = 192;

Layout layout(const xmod_dims* dm, int K) {
  Layout L{};
  const size_t es = esize(dm->dtype);
  const size_t BT = (size_t)dm->B * dm->T;
  (void)K;  // one layout serves every K: selections are sized for n <= T
  const size_t Bn = BT;
  const size_t M = BT;
  const size_t qkv_w = (size_t)(dm->n_heads + 2 * dm->n_kv_heads) * dm->head_dim;
  size_t off = 0;
  L.status = off; off += kAlign;
  // logits [k slice, run layer, B*T]
  L.s = off;      off = align_up(off + 4 * BT * kRouterRun * kRouterSplit);
  L.idx = off;    off = align_up(off + 4 * Bn);
  L.r_sel = off;  off = align_up(off + 4 * Bn);
  L.u = off;      off = align_up(off + es * M * dm->d);
  L.qkv = off;    off = align_up(off + es * M * qkv_w);
  // v transposed for the tensor-core attention: [B, hkv, hd, vt_ld(T)]
  L.vt = off;     off = align_up(off + es * (size_t)dm->B * dm->n_kv_heads * dm->head_dim *
                                           (size_t)vt_ld(dm->T));
  L.o = off;      off = align_up(off + es * M * dm->n_heads * dm->head_dim);
  L.h = off;      off = align_up(off + 4 * M * dm->d);   // h = x_sel + a kept in fp32
  L.a = off;      off = align_up(off + es * M * dm->d);  // a, the attention residual
  L.hidden = off; off = align_up(off + es * M * dm->d_ff);
  L.wr = off;     off = align_up(off + es * (size_t)kRouterRows * dm->d);   // stacked w_r
  L.count = off;  off = align_up(off + 4 * BT);   // token-choice bias state of a block
  L.last = off;   off = align_up(off + 4 * BT);
  L.seq = off;    off = align_up(off + 4 * (2 * (size_t)dm->B + 1));   // threshold rows
  L.thr = off;    off = align_up(off + 8 * BT);   // threshold picks per sequence (pos, gate)
  L.rowss = off;  off = align_up(off + 4 * M * (size_t)(dm->d / 32));   // h^2 sums per chunk
  const size_t slots = dm->dtype == XMOD_BF16 ? kSkSlots : 0;
  L.skflag = off; off = align_up(off + 4 * slots);
  L.skpart = off; off = align_up(off + 4 * slots * 128 * 256);
  L.total = off;
  return L;
}

inline char* at(void* ws, size_t off) { return (char*)ws + off; }

// The launch context of an entry point: its stream, the status word and the GEMMs'
// stream-K scratch, whose flags are cleared here (each launch leaves them clear, but
// a launch that gave up on a wait may not have, and the workspace starts unset).
int make_ctx(const xmod_dims* dm, void* ws, const Layout& L, void* stream, Ctx& c) {
  c = Ctx{(cudaStream_t)stream, (int*)at(ws, L.status)};
  if (dm->dtype != XMOD_BF16) return XMOD_OK;
  c.sk_flag = (int*)at(ws, L.skflag);
  c.sk_part = (float*)at(ws, L.skpart);
  c.sk_slots = kSkSlots;
  return cudaMemsetAsync(c.sk_flag, 0, 4 * (size_t)kSkSlots, c.stream) == cudaSuccess
             ? XMOD_OK
             : XMOD_ERR_CUDA;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? XMOD_OK : XMOD_ERR_CUDA; }

// One kernel launch: counted, optionally timed, and checked.
#define XMOD_RUN(kind, expr)                         \
  do {                                               \
    cudaError_t _e;                                  \
    {                                                \
      ProfScope _p(kind, c.stream);                  \
      _e = (expr);                                   \
    }                                                \
    count_launch();                                  \
    if (_e != cudaSuccess) return XMOD_ERR_CUDA;     \
  } while (0)

bool routed(int kind) {
  return kind == XMOD_LAYER_SPARSE || kind == XMOD_LAYER_ROUTED_FFN ||
         kind == XMOD_LAYER_SPARSE_FULLKV;
}
bool kind_ok(int kind) { return kind >= XMOD_LAYER_DENSE && kind <= XMOD_LAYER_SPARSE_FULLKV; }
// Which part of the block runs: all of it, the attention half (its residual written
// straight into the stream: x += a, for ATTN layers), the FFN half on RMSNorm(x) *
// rms2 with a = 0 (ROUTED_FFN layers), or all of it with every token's keys and
// values (SPARSE_FULLKV layers).
enum BlockPart { PART_ALL = 0, PART_ATTN = 1, PART_FFN = 2, PART_FULLKV = 3 };

int block_part(int kind) {
  return kind == XMOD_LAYER_ROUTED_FFN ? PART_FFN
         : kind == XMOD_LAYER_SPARSE_FULLKV ? PART_FULLKV : PART_ALL;
}

// The weights a layer kind uses must be present and 16-byte aligned.
bool weights_ok(const xmod_layer_weights* w, int kind) {
  if (!w || !kind_ok(kind)) return false;
  if (routed(kind) && !aligned16(w->w_router)) return false;
  if (kind != XMOD_LAYER_ROUTED_FFN) {
    const void* ps[] = {w->rms1, w->wq, w->wk, w->wv, w->wo};
    for (const void* p : ps)
      if (!aligned16(p)) return false;
  }
  if (kind != XMOD_LAYER_ATTN) {
    const void* ps[] = {w->rms2, w->w_gate, w->w_up, w->w_down};
    for (const void* p : ps)
      if (!aligned16(p)) return false;
  }
  if (!aligned16_or_null(w->q_norm) || !aligned16_or_null(w->k_norm)) return false;
  if (!isfinite(w->rope_theta) || w->rope_theta < 0.0f) return false;
  return isfinite(w->varsigma);
}

// The block on B*n compact rows (rows of x selected by idx, or identity when
// idx == NULL and n == T). Writes a to a_out when given, and either
// scatters the gated residual into x (scatter == true) or stores f to f_out.
// Rows of a threshold-routed layer: a variable count per sequence, known only on the
// device. tok [B*T]: compact row -> stream row; seq_count / seq_off [B]; M [1].
struct Ragged {
  const int32_t* tok = nullptr;
  const int32_t* seq_count = nullptr;
  const int32_t* seq_off = nullptr;
  const int32_t* M = nullptr;
};

// With scatter, xs_new (if not NULL) receives the updated compact rows [B*n, d].
// With rg (threshold routing), n is T: buffers are sized for every token, kernels
// compute the rows the routing picked (tensor-core path only).

bool qk_extras(const xmod_layer_weights* w) {
  return w->q_norm || w->k_norm || w->rope_theta > 0.0f;
}

// QK-norm and rotary embedding of a projection's q heads (from q_col0) and k heads
// (from k_col0) in the same rows, in place.
int qk_extras_run(const Ctx& c, const xmod_dims* dm, int64_t M, const int32_t* M_dev, void* x,
                  int ld, int q_col0, int q_heads, int k_col0, int k_heads,
                  const xmod_layer_weights* w, const int32_t* pos_idx, const int32_t* pos_tok,
                  int seqT) {
  XMOD_RUN("qk_norm_rope",
           launch_qk_transform(c, dm->dtype, M, M_dev, x, ld, q_col0, q_heads, w->q_norm, k_col0,
                               k_heads, w->k_norm, dm->head_dim, dm->rms_eps, w->rope_theta,
                               pos_idx, pos_tok, seqT));
  return XMOD_OK;
}

// Attention of a Selected-Q / full-KV layer (X-MoD notes, "mechanism controls": the
// selected tokens are the queries, every token provides keys and values): o [B*n, qw]
// for the n selected rows of each sequence (idx, ascending positions), each attending
// to every token at or before its own position.
int fullkv_attention(const Ctx& c, const xmod_dims* dm, const Layout& L, void* ws, int n,
                     const void* x, const int32_t* idx, const xmod_layer_weights* w) {
  const xmod_dtype dt = dm->dtype;
  const int B = dm->B, T = dm->T, d = dm->d, hq = dm->n_heads, hkv = dm->n_kv_heads,
            hd = dm->head_dim;
  const int qw = hq * hd, kw = hkv * hd;
  const size_t es = esize(dt);
  // scratch: RMSNorm1 of every token in u, their k | v in qkv (v transposed into vt on
  // the tensor-core path), the selected tokens' RMSNorm1 and q in the fp32 h buffer
  char* u_all = at(ws, L.u);
  char* kv = at(ws, L.qkv);
  char* vt = at(ws, L.vt);
  char* o = at(ws, L.o);
  char* u_sel = at(ws, L.h);
  char* q = u_sel + align_up(es * (size_t)B * n * d);
  if (align_up(es * (size_t)B * n * d) + es * (size_t)B * n * qw > 4 * (size_t)B * T * d)
    return XMOD_ERR_UNSUPPORTED;
  XMOD_RUN("gather_rmsnorm", launch_gather_rmsnorm(c, dt, B, T, T, d, x, nullptr, w->rms1,
                                                   dm->rms_eps, u_all));
  Epilogue ek;
  ek.kind = EPI_STORE;
  ek.out = kv;
  ek.ldo = 2 * kw;
  GemmTcProblem pk;
  pk.M = B * T; pk.N = 2 * kw; pk.K = d; pk.A = u_all; pk.lda = d; pk.ldb = d;
  pk.B[0] = w->wk; pk.B[1] = w->wv; pk.nB = 2; pk.split[0] = kw;
  Epilogue eq;
  eq.kind = EPI_STORE;
  eq.out = q;
  eq.ldo = qw;
  GemmTcProblem pq;
  pq.M = B * n; pq.N = qw; pq.K = d; pq.A = u_sel; pq.lda = d; pq.ldb = d; pq.B[0] = w->wq;
  bool tc = dt == XMOD_BF16 && attention_tc_supported(hd, n, qw) &&
            attention_tc_supported(hd, T, 2 * kw) && gemm_tc_supported(pq, eq);
  if (tc) {
    ek.vt = vt;
    ek.vt_col0 = kw;
    ek.vt_hd = hd;
    ek.vt_hkv = hkv;
    ek.vt_ld = vt_ld(T);
    ek.n_per_seq = T;
    tc = gemm_tc_supported(pk, ek);
  }
  if (tc) {
    XMOD_RUN("gemm_qkv", launch_gemm_tc(c, pk, ek));
  } else {
    ek.vt = nullptr;
    XMOD_RUN("gemm_qkv", launch_gemm_simt(c, dt, B * T, kw, d, u_all, d, w->wk, d, nullptr, ek));
    ek.out = kv + es * kw;
    XMOD_RUN("gemm_qkv", launch_gemm_simt(c, dt, B * T, kw, d, u_all, d, w->wv, d, nullptr, ek));
  }
  if (qk_extras(w)) {   // keys of every token at their positions
    const int st = qk_extras_run(c, dm, (int64_t)B * T, nullptr, kv, 2 * kw, 0, 0, 0, hkv, w,
                                 nullptr, nullptr, T);
    if (st) return st;
  }
  XMOD_RUN("gather_rmsnorm", launch_gather_rmsnorm(c, dt, B, T, n, d, x, idx, w->rms1,
                                                   dm->rms_eps, u_sel));
  if (tc)
    XMOD_RUN("gemm_qkv", launch_gemm_tc(c, pq, eq));
  else
    XMOD_RUN("gemm_qkv", launch_gemm_simt(c, dt, B * n, qw, d, u_sel, d, w->wq, d, nullptr, eq));
  if (qk_extras(w)) {   // queries at their original positions
    const int st = qk_extras_run(c, dm, (int64_t)B * n, nullptr, q, qw, 0, hq, 0, 0, w, idx,
                                 nullptr, T);
    if (st) return st;
  }
  if (tc) {
    AttnKv akv;
    akv.k = kv;
    akv.ldk = 2 * kw;
    akv.nkv = T;
    akv.qpos = idx;
    XMOD_RUN("attention", launch_attention_tc(c, B, n, hq, hkv, q, qw, vt, vt_ld(T), o, nullptr,
                                              nullptr, &akv));
  } else {
    XMOD_RUN("attention", launch_attention_simt(c, dt, B, n, hq, hkv, hd, q, qw, kv,
                                                kv + es * kw, 2 * kw, o, idx, T));
  }
  return XMOD_OK;
}

// The standalone gather + RMSNorm1 kernel and a GEMM on its compact output (default),
// or the gathered RMSNorm inside the q|k|v GEMM's operand load: the environment variable
// XMOD_GATHER_FUSED=1, read at every call, selects the latter (both compute the block;
// they differ only in rounding order). The fused form measured slower on GB300 (see the
// gathered-RMSNorm GEMM in gemm_tc.cu), so it is not the default.
bool gather_fused_enabled() {
  const char* v = getenv("XMOD_GATHER_FUSED");
  return v && v[0] == '1' && v[1] == '\0';
}

int run_block(const Ctx& c, const xmod_dims* dm, const Layout& L, void* ws, int n,
              const void* x_src, const int32_t* idx, const xmod_layer_weights* w, void* a_out,
              void* f_out, bool scatter, void* x_inout, const float* r_sel, int gate,
              void* xs_new = nullptr, const Ragged* rg = nullptr, int part = PART_ALL) {
  const xmod_dtype dt = dm->dtype;
  const int B = dm->B, T = dm->T, d = dm->d, hq = dm->n_heads, hkv = dm->n_kv_heads,
            hd = dm->head_dim, F = dm->d_ff;
  const int M = B * n;
  const int32_t* M_dev = rg ? rg->M : nullptr;
  const int qw = hq * hd, kw = hkv * hd, qkv_w = qw + 2 * kw;
  const size_t es = esize(dt);
  char* u = at(ws, L.u);
  char* qkv = at(ws, L.qkv);
  char* o = at(ws, L.o);
  char* h = at(ws, L.h);
  char* hidden = at(ws, L.hidden);
  const bool tc = dt == XMOD_BF16;
  // bf16 projections run on the tensor cores only (no FFMA route for them): without the
  // TMA tensor-map entry point the call is refused rather than run on FFMA kernels
  if (tc && !tma_available()) return XMOD_ERR_UNSUPPORTED;
  char* v2 = u;   // RMSNorm2 output, in the buffer of u (consumed by the q/k/v projection)
  // a, the attention residual, for the down projection's scatter (the caller's a_out
  // when given); NULL for an FFN-only block (a = 0)
  void* a_res = a_out ? a_out : (void*)at(ws, L.a);
  RowMap rm;
  if (rg) {
    rm.tok = rg->tok;
    rm.M_dev = M_dev;
  }
  // RMSNorm2 folded into the o-projection and gate/up epilogues (tensor-core path)
  float* rowss = (float*)at(ws, L.rowss);
  Epilogue eg;   // 6. hidden = silu(v2 Wg^T) * (v2 Wu^T), set up here for the fold test
  eg.kind = EPI_SWIGLU;
  eg.out = hidden;
  eg.ldo = F;
  GemmTcProblem pg;
  pg.M = M; pg.N = F; pg.K = d; pg.A = v2; pg.lda = d; pg.ldb = d;
  pg.B[0] = w->w_gate; pg.B[1] = w->w_up; pg.nB = 2;
  pg.M_dev = M_dev;
  const bool gate_up_tc = tc && gemm_tc_supported(pg, eg);
  bool fold2 = gate_up_tc && part == PART_ALL && d % 128 == 0;
  if (part == PART_FFN) {   // FFN half only: v2 = RMSNorm(x_sel) * rms2, a = 0
    XMOD_RUN("gather_rmsnorm",
             launch_gather_rmsnorm(c, dt, B, T, n, d, x_src, idx, w->rms2, dm->rms_eps, v2, rm));
    a_res = nullptr;
  } else {
    if (part == PART_FULLKV) {   // steps 1-3 with every token's keys and values
      if (rg || !idx) return XMOD_ERR_UNSUPPORTED;
      const int st = fullkv_attention(c, dm, L, ws, n, x_src, idx, w);
      if (st) return st;
    } else {
      // 2. q, k, v projections into one [M, qkv_w] buffer
      char* vt = at(ws, L.vt);
      const bool tc_attn = tc && attention_tc_supported(hd, n, qkv_w);
      Epilogue e;
      e.kind = EPI_STORE;
      e.ldo = qkv_w;
      e.out = qkv;
      if (tc_attn) {  // v goes straight to its transposed layout
        e.vt = vt;
        e.vt_col0 = qw + kw;
        e.vt_hd = hd;
        e.vt_hkv = hkv;
        e.vt_ld = vt_ld(n);
        e.n_per_seq = n;
      }
      GemmTcProblem pq;
      pq.M = M; pq.N = qkv_w; pq.K = d; pq.A = u; pq.lda = d; pq.ldb = d;
      pq.B[0] = w->wq; pq.B[1] = w->wk; pq.B[2] = w->wv; pq.nB = 3;
      pq.split[0] = qw; pq.split[1] = qw + kw;
      // 1. gather + RMSNorm1: for the routed rows of a stream (idx given, a fixed count per
      // sequence) inside the q|k|v GEMM's operand load, else a gathered copy u
      bool fused_gather = false;
      if (tc && idx && !rg && gather_fused_enabled()) {
        GemmTcProblem pg = pq;
        pg.A = x_src;
        pg.gather_idx = idx;
        pg.gather_T = T;
        pg.gather_n = n;
        pg.gather_rows = (int64_t)B * T;
        pg.gather_gamma = w->rms1;
        pg.gather_eps = dm->rms_eps;
        if (gemm_tc_supported(pg, e)) {
          pq = pg;
          fused_gather = true;
        }
      }
      if (!fused_gather)
        XMOD_RUN("gather_rmsnorm", launch_gather_rmsnorm(c, dt, B, T, n, d, x_src, idx, w->rms1,
                                                         dm->rms_eps, u, rm));
      const bool tc_qkv = tc && gemm_tc_supported(pq, e);
      if (rg) {
        if (!tc_qkv || !tc_attn) return XMOD_ERR_UNSUPPORTED;
        e.tok = rg->tok;
        e.seq_off = rg->seq_off;
        e.T = T;
        pq.M_dev = M_dev;
        // keys past a sequence's count are read (and multiplied by zero weights): keep
        // them finite
        if (cudaMemsetAsync(vt, 0, es * (size_t)B * hkv * hd * vt_ld(n), c.stream) != cudaSuccess)
          return XMOD_ERR_CUDA;
      }
      if (tc_qkv) {
        XMOD_RUN("gemm_qkv", launch_gemm_tc(c, pq, e));
      } else {
        e.vt = nullptr;
        XMOD_RUN("gemm_qkv", launch_gemm_simt(c, dt, M, qw, d, u, d, w->wq, d, nullptr, e));
        e.out = qkv + es * qw;
        XMOD_RUN("gemm_qkv", launch_gemm_simt(c, dt, M, kw, d, u, d, w->wk, d, nullptr, e));
        e.out = qkv + es * (qw + kw);
        XMOD_RUN("gemm_qkv", launch_gemm_simt(c, dt, M, kw, d, u, d, w->wv, d, nullptr, e));
      }
      if (qk_extras(w)) {   // q and k heads at the tokens' original positions
        const int32_t* ptok = rg ? rg->tok : nullptr;
        const int seqT = rg ? T : n;
        const int st =
            qk_extras_run(c, dm, M, M_dev, qkv, qkv_w, 0, hq, qw, hkv, w, idx, ptok, seqT);
        if (st) return st;
      }
      // 3. causal GQA attention among the n rows of each sequence
      if (tc_qkv && tc_attn)
        XMOD_RUN("attention", launch_attention_tc(c, B, n, hq, hkv, qkv, qkv_w, vt, vt_ld(n), o,
                                                  rg ? rg->seq_count : nullptr,
                                                  rg ? rg->seq_off : nullptr));
      else
        XMOD_RUN("attention", launch_attention_simt(c, dt, B, n, hq, hkv, hd, qkv, qkv_w,
                                                    qkv + es * qw, qkv + es * (qw + kw), qkv_w, o));
    }
    if (part == PART_ATTN) {   // x += a straight into the stream: the down epilogue's
      Epilogue ea;            // dense form y = h + f with no h (h = x) and f = a
      ea.kind = EPI_DOWN_SCATTER;
      ea.x = x_inout;
      ea.idx = idx;
      ea.T = T;
      ea.n_per_seq = n;
      ea.d = d;
      ea.gate = -1;
      GemmTcProblem pa;
      pa.M = M; pa.N = d; pa.K = qw; pa.A = o; pa.lda = qw; pa.ldb = qw; pa.B[0] = w->wo;
      if (tc && gemm_tc_supported(pa, ea))
        XMOD_RUN("gemm_o_residual", launch_gemm_tc(c, pa, ea));
      else
        XMOD_RUN("gemm_o_residual", launch_gemm_simt(c, dt, M, d, qw, o, qw, w->wo, qw, nullptr, ea));
      return XMOD_OK;
    }
    // 4. a = o Wo^T, h = x_sel + a
    Epilogue eo;
    eo.kind = EPI_OPROJ;
    eo.out = scatter || a_out ? a_res : nullptr;
    eo.ldo = d;
    eo.out2 = h;
    eo.ldo2 = d;
    eo.x = (void*)x_src;
    eo.idx = idx;
    eo.T = T;
    eo.n_per_seq = n;
    eo.d = d;
    GemmTcProblem po;
    po.M = M; po.N = d; po.K = qw; po.A = o; po.lda = qw; po.ldb = qw; po.B[0] = w->wo;
    if (rg) {
      eo.tok = rg->tok;
      po.M_dev = M_dev;
      if (!gemm_tc_supported(po, eo)) return XMOD_ERR_UNSUPPORTED;
    }
    const bool oproj_tc = tc && gemm_tc_supported(po, eo);
    fold2 = fold2 && oproj_tc;
    if (fold2) {   // 5. folded: the epilogue writes h * rms2 and the row sums (no h)
      eo.out2 = nullptr;
      eo.out3 = v2;
      eo.g2 = w->rms2;
      eo.rowss = rowss;
      eo.norm_d = d;
    }
    if (oproj_tc)
      XMOD_RUN("gemm_o_residual", launch_gemm_tc(c, po, eo));
    else
      XMOD_RUN("gemm_o_residual", launch_gemm_simt(c, dt, M, d, qw, o, qw, w->wo, qw, nullptr, eo));
    // 5. v2 = RMSNorm(h) * rms2
    if (!fold2)
      XMOD_RUN("rmsnorm2", launch_rmsnorm_f32in(c, dt, M, d, (const float*)h, w->rms2,
                                                dm->rms_eps, v2, M_dev));
  }
  // 6. hidden = silu(v2 Wg^T) * (v2 Wu^T) (or, folded, of (h * rms2) scaled by 1 / rms(h))
  if (fold2) {
    eg.rowss = rowss;
    eg.eps = dm->rms_eps;
    eg.norm_d = d;
  }
  if (rg && !gate_up_tc) return XMOD_ERR_UNSUPPORTED;
  if (gate_up_tc)
    XMOD_RUN("gemm_gate_up_swiglu", launch_gemm_tc(c, pg, eg));
  else
    XMOD_RUN("gemm_gate_up_swiglu",
             launch_gemm_simt(c, dt, M, F, d, v2, d, w->w_gate, d, w->w_up, eg));
  // 7. f = hidden Wd^T, then the gated residual (or f stored)
  Epilogue ed;
  if (scatter) {
    ed.kind = EPI_DOWN_SCATTER;
    ed.x = x_inout;
    ed.idx = idx;
    ed.T = T;
    ed.n_per_seq = n;
    ed.d = d;
    ed.a = a_res;
    ed.r_sel = r_sel;
    ed.varsigma = w->varsigma;
    ed.gate = gate;
    ed.out = xs_new;
    ed.ldo = d;
  } else {
    ed.kind = EPI_STORE;
    ed.out = f_out;
    ed.ldo = d;
  }
  GemmTcProblem pd;
  pd.M = M; pd.N = d; pd.K = F; pd.A = hidden; pd.lda = F; pd.ldb = F; pd.B[0] = w->w_down;
  if (rg) {
    ed.tok = rg->tok;
    pd.M_dev = M_dev;
    if (!gemm_tc_supported(pd, ed)) return XMOD_ERR_UNSUPPORTED;
  }
  const char* down_name = scatter ? "gemm_down_scatter" : "gemm_down";
  if (tc && gemm_tc_supported(pd, ed))
    XMOD_RUN(down_name, launch_gemm_tc(c, pd, ed));
  else
    XMOD_RUN(down_name, launch_gemm_simt(c, dt, M, d, F, hidden, F, w->w_down, F, nullptr, ed));
  return XMOD_OK;
}

int check_ws(const xmod_dims* dm, int K, void* ws, size_t ws_bytes) {
  if (!aligned16(ws)) return XMOD_ERR_WORKSPACE;
  if (ws_bytes < layout(dm, K).total) return XMOD_ERR_WORKSPACE;
  return XMOD_OK;
}

// Router-logit GEMM: S[j, token(m)] = w_j . rows[m] + bias[token(m)] for the
// n_vec vectors stacked at wr (bf16, [>= 32 rows from wr, d]).
GemmTcProblem router_problem(const xmod_dims* dm, int M, const void* rows, const void* wr,
                             int wr_rows, int n_vec) {
  GemmTcProblem p;
  p.M = M; p.N = n_vec; p.K = dm->d; p.A = rows; p.lda = dm->d;
  p.B[0] = wr; p.ldb = dm->d; p.b_rows = wr_rows;
  p.ksplit = router_split(dm);
  return p;
}
Epilogue router_epilogue(const xmod_dims* dm, int n_per_seq, const int32_t* idx, float* S,
                         const float* bias) {
  Epilogue e;
  e.kind = EPI_ROUTER;
  e.out = S;
  e.ldo = dm->B * dm->T;
  e.plane = (int64_t)kRouterRun * dm->B * dm->T;
  e.idx = idx;
  e.T = dm->T;
  e.n_per_seq = n_per_seq;
  e.bias = bias;
  return e;
}

// Consecutive sparse layers lw[0..count) (count <= kRouterRun) with the router logits
// kept current incrementally. Each layer's logits are w_r . x + b on that layer's
// input stream, and a layer changes only the rows it selected. So one pass over the
// stream computes the logits of every layer of the run, and after each layer only
// its B*(T/K) updated rows get their logits for the later layers recomputed (from
// the compact copy of the new rows that the down-projection epilogue writes).
// A single sparse layer is a run of one; idx_out / r_sel_out (NULL: workspace) then
// receive its selection. track (NULL: none) carries the block's token-choice bias
// state; its `layer` is the stack index of lw[0] among the sparse layers, and its
// stats pointer addresses that layer's [B, 4] statistics.
RouteTrack track_for(const RouteTrack* track, int j, int B) {
  RouteTrack t = *track;
  t.layer += j;
  if (t.stats) t.stats += (int64_t)j * B * 4;
  return t;
}

// threshold: the causal threshold rule instead of top-(T/K) (K unused); the layers
// then take a variable number of tokens per sequence (device-side row counts).
int sparse_run(const Ctx& c, const xmod_dims* dm, const Layout& L, void* ws, int K,
               xmod_gate gate, const xmod_layer_weights* lw, int count, void* x,
               const float* bias, int32_t* idx_out = nullptr, float* r_sel_out = nullptr,
               const RouteTrack* track = nullptr, bool threshold = false, int part = PART_ALL) {
  const int B = dm->B, T = dm->T, d = dm->d, n = threshold ? T : T / K;
  const int64_t BT = (int64_t)B * T;
  float* S = (float*)at(ws, L.s);
  int32_t* idx = idx_out ? idx_out : (int32_t*)at(ws, L.idx);
  float* r_sel = r_sel_out ? r_sel_out : (float*)at(ws, L.r_sel);
  int32_t* seq = (int32_t*)at(ws, L.seq);   // seq_count [B], seq_off [B], M
  Ragged rg;
  rg.tok = idx;
  rg.seq_count = seq;
  rg.seq_off = seq + B;
  rg.M = seq + 2 * B;
  char* wr = at(ws, L.wr);
  void* xs_new = at(ws, L.u);   // free once the gate/up GEMM has read v2
  RowPtrs rows{};
  for (int j = 0; j < count; ++j) rows.p[j] = lw[j].w_router;
  XMOD_RUN("router_stack", launch_stack_rows(c, rows, count, kRouterRows, d, wr));
  XMOD_RUN("router", launch_gemm_tc(c, router_problem(dm, (int)BT, x, wr, kRouterRows, count),
                                    router_epilogue(dm, T, nullptr, S, bias)));
  for (int j = 0; j < count; ++j) {
    const RouteTrack tj = track ? track_for(track, j, B) : RouteTrack{};
    const int planes = router_split(dm);
    const int64_t plane = (int64_t)kRouterRun * BT;
    if (threshold)
      XMOD_RUN("threshold",
               launch_threshold_select(c, B, T, S + j * BT, idx, r_sel, seq, seq + B, seq + 2 * B,
                                       track ? &tj : nullptr, planes, plane,
                                       (int32_t*)at(ws, L.thr), (float*)at(ws, L.thr) + BT));
    else
      XMOD_RUN("topk", launch_topk(c, B, T, n, S + j * BT, idx, r_sel, track ? &tj : nullptr,
                                   planes, plane));
    const bool refresh = j + 1 < count;
    const int st = run_block(c, dm, L, ws, n, x, threshold ? nullptr : idx, &lw[j], nullptr,
                             nullptr, true, x, r_sel, (int)gate, refresh ? xs_new : nullptr,
                             threshold ? &rg : nullptr, part);
    if (st) return st;
    if (refresh) {
      GemmTcProblem p = router_problem(dm, B * n, xs_new, wr + (size_t)(j + 1) * d * 2,
                                       kRouterRows - (j + 1), count - 1 - j);
      Epilogue e = router_epilogue(dm, n, threshold ? nullptr : idx, S + (j + 1) * BT, bias);
      if (threshold) {
        p.M_dev = rg.M;
        e.tok = rg.tok;
      }
      XMOD_RUN("router_refresh", launch_gemm_tc(c, p, e));
    }
  }
  return XMOD_OK;
}

// Whether sparse_run can serve runs of these dimensions (bf16 tensor-core GEMMs).
bool sparse_run_supported(const xmod_dims* dm, void* ws, const Layout& L) {
  if (dm->dtype != XMOD_BF16) return false;
  if ((int64_t)dm->B * dm->T > INT32_MAX) return false;
  const GemmTcProblem p = router_problem(dm, dm->B * dm->T, at(ws, L.u), at(ws, L.wr),
                                         kRouterRows, kRouterRun);
  return gemm_tc_supported(p, router_epilogue(dm, dm->T, nullptr, (float*)at(ws, L.s), nullptr));
}

// Whether the threshold rule can run: the variable-length block needs the tensor-core
// GEMMs and attention.
bool threshold_supported(const xmod_dims* dm, void* ws, const Layout& L) {
  const int qkv_w = (dm->n_heads + 2 * dm->n_kv_heads) * dm->head_dim;
  return sparse_run_supported(dm, ws, L) && attention_tc_supported(dm->head_dim, dm->T, qkv_w);
}

int layer_impl(const Ctx& c, const xmod_dims* dm, xmod_layer_kind kind, int K, xmod_gate gate,
               const xmod_layer_weights* w, void* x, const float* bias, int32_t* idx_out,
               float* r_sel_out, void* ws, const Layout& L, const RouteTrack* track = nullptr) {
  if (kind == XMOD_LAYER_DENSE)
    return run_block(c, dm, L, ws, dm->T, x, nullptr, w, nullptr, nullptr, true, x, nullptr, -1);
  if (kind == XMOD_LAYER_ATTN)
    return run_block(c, dm, L, ws, dm->T, x, nullptr, w, nullptr, nullptr, true, x, nullptr, -1,
                     nullptr, nullptr, PART_ATTN);
  const int part = block_part(kind);
  if (sparse_run_supported(dm, ws, L))
    return sparse_run(c, dm, L, ws, K, gate, w, 1, x, bias, idx_out, r_sel_out, track, false,
                      part);
  const int n = dm->T / K;
  float* s = (float*)at(ws, L.s);
  int32_t* idx = idx_out ? idx_out : (int32_t*)at(ws, L.idx);
  float* r_sel = r_sel_out ? r_sel_out : (float*)at(ws, L.r_sel);
  XMOD_RUN("router", launch_router(c, dm->dtype, (int64_t)dm->B * dm->T, dm->d, x, w->w_router, bias, s,
                         nullptr));
  XMOD_RUN("topk", launch_topk(c, dm->B, dm->T, n, s, idx, r_sel, track));
  return run_block(c, dm, L, ws, n, x, idx, w, nullptr, nullptr, true, x, r_sel, (int)gate,
                   nullptr, nullptr, part);
}

// A stack in the given layer order. A block is the set of routed layers (SPARSE or
// ROUTED_FFN) between two dense layers (or the stack's ends): the token-choice bias
// state is cleared at its first routed layer, and update_hist has one [B, L_max + 1]
// slab per block, L_max the most routed layers of a block. Consecutive routed layers
// of one kind share their router-logit pass (sparse_run).
int stack_impl(const xmod_dims* dm, int K, const int32_t* kinds, int n_layers, xmod_gate gate,
               const xmod_layer_weights* layers, void* x_inout, const float* bias,
               const xmod_stack_opts* opts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (gate != XMOD_GATE_XMOD && gate != XMOD_GATE_MOD) return XMOD_ERR_INVALID_ARG;
  if (!aligned16(x_inout) || !aligned16_or_null(bias)) return XMOD_ERR_INVALID_ARG;
  if (opts && (!isfinite(opts->bias_step) || opts->bias_step < 0.0f)) return XMOD_ERR_INVALID_ARG;
  if (opts && (((uintptr_t)opts->layer_stats & 3) || ((uintptr_t)opts->update_hist & 3)))
    return XMOD_ERR_INVALID_ARG;
  if (opts && opts->routing != XMOD_ROUTE_TOPK && opts->routing != XMOD_ROUTE_THRESHOLD)
    return XMOD_ERR_INVALID_ARG;
  const bool threshold = opts && opts->routing == XMOD_ROUTE_THRESHOLD;
  // block of each routed layer, and whether it is the block's last routed layer
  std::vector<int> block_of(n_layers, -1);
  std::vector<char> block_last(n_layers, 0);
  bool any_routed = false;
  int max_block = 0, blocks = 0, in_block = 0, last_routed = -1;
  for (int l = 0; l < n_layers; ++l) {
    if (!weights_ok(&layers[l], kinds[l])) return XMOD_ERR_INVALID_ARG;
    if (threshold && routed(kinds[l]) && kinds[l] != XMOD_LAYER_SPARSE)
      return XMOD_ERR_UNSUPPORTED;
    if (kinds[l] == XMOD_LAYER_DENSE) {
      if (last_routed >= 0) block_last[last_routed] = 1;
      last_routed = -1;
      in_block = 0;
    } else if (routed(kinds[l])) {
      if (last_routed < 0) ++blocks;
      block_of[l] = blocks - 1;
      last_routed = l;
      any_routed = true;
      max_block = ++in_block > max_block ? in_block : max_block;
    }
  }
  if (last_routed >= 0) block_last[last_routed] = 1;
  if (!head_dim_supported(dm->head_dim)) return XMOD_ERR_UNSUPPORTED;
  if (any_routed && dm->T > topk_max_T()) return XMOD_ERR_UNSUPPORTED;
  int st = check_ws(dm, K, ws, ws_bytes);
  if (st) return st;
  const Layout L = layout(dm, K);
  const bool runs = sparse_run_supported(dm, ws, L);
  if (threshold && !threshold_supported(dm, ws, L)) return XMOD_ERR_UNSUPPORTED;
  Ctx c;
  st = make_ctx(dm, ws, L, stream, c);
  if (st) return st;
  const int64_t BT = (int64_t)dm->B * dm->T;
  // Token-choice bias state, only when an option needs it (else the plain top-k).
  const bool tracked = opts && (opts->bias_step != 0.0f || opts->layer_stats || opts->update_hist);
  RouteTrack track;
  if (tracked) {
    track.count = (int32_t*)at(ws, L.count);
    track.last = (int32_t*)at(ws, L.last);
    track.bias_step = opts->bias_step;
    track.stats = opts->layer_stats;
  }
  int routed_index = 0, cur_block = -1;
  for (int l = 0; l < n_layers;) {
    const int kind = kinds[l];
    if (!routed(kind)) {
      st = layer_impl(c, dm, (xmod_layer_kind)kind, K, gate, &layers[l], x_inout, bias, nullptr,
                      nullptr, ws, L);
      if (st) return st;
      ++l;
      continue;
    }
    if (tracked && block_of[l] != cur_block) {   // a new block: clear the bias state
      cur_block = block_of[l];
      if (cudaMemsetAsync(track.count, 0, 4 * BT, c.stream) != cudaSuccess) return XMOD_ERR_CUDA;
      if (cudaMemsetAsync(track.last, 0x80, 4 * BT, c.stream) != cudaSuccess) return XMOD_ERR_CUDA;
    }
    // the following layers of the same kind, at most kRouterRun at a time
    int count = 1;
    if (runs)
      while (count < kRouterRun && l + count < n_layers && kinds[l + count] == kind) ++count;
    RouteTrack tl = track;
    tl.layer = routed_index;
    if (tl.stats) tl.stats += (int64_t)routed_index * dm->B * 4;
    const int part = block_part(kind);
    if (runs)
      st = sparse_run(c, dm, L, ws, K, gate, &layers[l], count, x_inout, bias, nullptr, nullptr,
                      tracked ? &tl : nullptr, threshold, part);
    else
      st = layer_impl(c, dm, (xmod_layer_kind)kind, K, gate, &layers[l], x_inout, bias, nullptr,
                      nullptr, ws, L, tracked ? &tl : nullptr);
    if (st) return st;
    l += count;
    routed_index += count;
    if (tracked && opts->update_hist && block_last[l - 1])
      XMOD_RUN("update_hist",
               launch_count_hist(c, dm->B, dm->T, max_block, track.count,
                                 opts->update_hist + (int64_t)block_of[l - 1] * dm->B *
                                                         (max_block + 1)));
  }
  return XMOD_OK;
}

}  // namespace
}  // namespace xmod

using namespace xmod;

extern "C" {

const char* xmod_version(void) { return "xmod-gb300 0.1 (sm_103a)"; }

const char* xmod_status_string(int st) {
  switch (st) {
    case XMOD_OK: return "ok";
    case XMOD_ERR_INVALID_ARG: return "invalid argument";
    case XMOD_ERR_UNSUPPORTED: return "unsupported combination";
    case XMOD_ERR_CUDA: return "CUDA runtime error";
    case XMOD_ERR_TIMEOUT: return "device-side wait timed out";
    case XMOD_ERR_DEVICE_CHECK: return "device-side check failed (non-finite logit or bad index)";
    case XMOD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}

size_t xmod_workspace_bytes(const xmod_dims* dm, int K) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T) return 0;
  return layout(dm, K).total;
}

int xmod_reset_status(void* ws, size_t ws_bytes, void* stream) {
  if (!aligned16(ws) || ws_bytes < kAlign) return XMOD_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(int), (cudaStream_t)stream));
}

int xmod_sync_status(void* ws, void* stream) {
  if (!aligned16(ws)) return XMOD_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return XMOD_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return XMOD_ERR_CUDA;
  return h;
}

int xmod_router_topk(const xmod_dims* dm, int K, const void* x, const void* w_r,
                     const float* bias, float* logits, float* r, int32_t* idx, float* r_sel,
                     void* ws, size_t ws_bytes, void* stream) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T) return XMOD_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_r) || !aligned16(idx) || !aligned16_or_null(bias) ||
      !aligned16_or_null(logits) || !aligned16_or_null(r) || !aligned16_or_null(r_sel))
    return XMOD_ERR_INVALID_ARG;
  if (dm->T > topk_max_T()) return XMOD_ERR_UNSUPPORTED;
  int st = check_ws(dm, K, ws, ws_bytes);
  if (st) return st;
  const Layout L = layout(dm, K);
  Ctx c{(cudaStream_t)stream, (int*)at(ws, L.status)};
  float* s = logits ? logits : (float*)at(ws, L.s);
  XMOD_RUN("router", launch_router(c, dm->dtype, (int64_t)dm->B * dm->T, dm->d, x, w_r, bias, s, r));
  XMOD_RUN("topk", launch_topk(c, dm->B, dm->T, dm->T / K, s, idx, r_sel));
  return XMOD_OK;
}

int xmod_topk(const xmod_dims* dm, int K, const float* logits, int32_t* idx, float* r_sel,
              void* ws, size_t ws_bytes, void* stream) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T) return XMOD_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(idx) || !aligned16_or_null(r_sel))
    return XMOD_ERR_INVALID_ARG;
  if (dm->T > topk_max_T()) return XMOD_ERR_UNSUPPORTED;
  int st = check_ws(dm, K, ws, ws_bytes);
  if (st) return st;
  const Layout L = layout(dm, K);
  Ctx c{(cudaStream_t)stream, (int*)at(ws, L.status)};
  XMOD_RUN("topk", launch_topk(c, dm->B, dm->T, dm->T / K, logits, idx, r_sel));
  return XMOD_OK;
}

int xmod_gather(const xmod_dims* dm, int K, const void* x, const int32_t* idx, void* xs,
                int* status_out, void* stream) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T) return XMOD_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(idx) || !aligned16(xs) || ((uintptr_t)status_out & 3u))
    return XMOD_ERR_INVALID_ARG;
  Ctx c{(cudaStream_t)stream, status_out};
  XMOD_RUN("gather", launch_gather(c, dm->dtype, dm->B, dm->T, dm->T / K, dm->d, x, idx, xs));
  return XMOD_OK;
}

int xmod_block_fwd(const xmod_dims* dm, int n_per_seq, const void* xs, const int32_t* idx,
                   const xmod_layer_weights* w, void* a_out, void* f_out, void* ws,
                   size_t ws_bytes, void* stream) {
  if (!dims_ok(dm) || n_per_seq <= 0 || n_per_seq > dm->T) return XMOD_ERR_INVALID_ARG;
  if (!aligned16(xs) || !aligned16_or_null(idx) || !aligned16(a_out) || !aligned16(f_out) ||
      !weights_ok(w, XMOD_LAYER_DENSE))
    return XMOD_ERR_INVALID_ARG;
  if (!head_dim_supported(dm->head_dim)) return XMOD_ERR_UNSUPPORTED;
  const int K = dm->T / n_per_seq;
  int st = check_ws(dm, K, ws, ws_bytes);
  if (st) return st;
  const Layout L = layout(dm, K);
  Ctx c;
  st = make_ctx(dm, ws, L, stream, c);
  if (st) return st;
  // Without idx the rows come from the compact buffer: view it as B sequences of
  // n_per_seq tokens. With idx, the caller's positions are checked on the device first
  // and a copy with every bad row clamped into range is used, so no access leaves the
  // stream; the status word records the bad rows.
  xmod_dims local = *dm;
  if (!idx) local.T = n_per_seq;
  const int32_t* use_idx = idx;
  if (idx) {
    int32_t* safe = (int32_t*)at(ws, L.idx);
    XMOD_RUN("idx_check", launch_idx_sanitize(c, dm->B, dm->T, n_per_seq, idx, safe));
    use_idx = safe;
  }
  return run_block(c, &local, L, ws, n_per_seq, xs, use_idx, w, a_out, f_out, false, nullptr,
                   nullptr, -1);
}

int xmod_gated_scatter(const xmod_dims* dm, int K, void* x_inout, const int32_t* idx,
                       const float* r_sel, const void* a, const void* f, float varsigma,
                       xmod_gate gate, int* status_out, void* stream) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T) return XMOD_ERR_INVALID_ARG;
  if (gate != XMOD_GATE_XMOD && gate != XMOD_GATE_MOD) return XMOD_ERR_INVALID_ARG;
  if (!aligned16(x_inout) || !aligned16(idx) || !aligned16(r_sel) || !aligned16(a) ||
      !aligned16_or_null(f) || !isfinite(varsigma))
    return XMOD_ERR_INVALID_ARG;
  if (!f && gate != XMOD_GATE_XMOD) return XMOD_ERR_INVALID_ARG;
  if ((uintptr_t)status_out & 3u) return XMOD_ERR_INVALID_ARG;
  Ctx c{(cudaStream_t)stream, status_out};
  XMOD_RUN("gated_scatter", launch_gated_scatter(c, dm->dtype, dm->B, dm->T, dm->T / K, dm->d,
                                                 x_inout, idx, r_sel, a, f, varsigma, (int)gate));
  return XMOD_OK;
}

size_t xmod_bwd_workspace_bytes(const xmod_dims* dm, int K) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T) return 0;
  return bwd_workspace_bytes(dm);
}

int xmod_layer_bwd(const xmod_dims* dm, xmod_layer_kind kind, int K, xmod_gate gate,
                   const xmod_layer_weights* w, const void* x, const float* bias, const void* dy,
                   float route_coef, void* dx, const xmod_layer_grads* g, void* ws,
                   size_t ws_bytes, void* stream) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T) return XMOD_ERR_INVALID_ARG;
  if (!kind_ok(kind)) return XMOD_ERR_INVALID_ARG;
  if (gate != XMOD_GATE_XMOD && gate != XMOD_GATE_MOD) return XMOD_ERR_INVALID_ARG;
  if (!weights_ok(w, kind) || !aligned16(x) || !aligned16(dy) || !aligned16(dx) ||
      !aligned16_or_null(bias) || !g || !isfinite(route_coef))
    return XMOD_ERR_INVALID_ARG;
  if (dx == x || dx == dy) return XMOD_ERR_INVALID_ARG;
  // the gradients of the weights the kind uses are required; the others may be NULL
  const bool uses_attn = kind != XMOD_LAYER_ROUTED_FFN, uses_ffn = kind != XMOD_LAYER_ATTN;
  const float* ga[] = {g->rms1, g->wq, g->wk, g->wv, g->wo};
  const float* gf[] = {g->rms2, g->w_gate, g->w_up, g->w_down};
  for (const float* p : ga)
    if (uses_attn ? !aligned16(p) : !aligned16_or_null(p)) return XMOD_ERR_INVALID_ARG;
  for (const float* p : gf)
    if (uses_ffn ? !aligned16(p) : !aligned16_or_null(p)) return XMOD_ERR_INVALID_ARG;
  if (!g->varsigma || (routed(kind) && !aligned16(g->w_router)) ||
      !aligned16_or_null(g->w_router) || !aligned16_or_null(g->q_norm) ||
      !aligned16_or_null(g->k_norm))
    return XMOD_ERR_INVALID_ARG;
  if ((w->q_norm && !aligned16(g->q_norm)) || (w->k_norm && !aligned16(g->k_norm)))
    return XMOD_ERR_INVALID_ARG;
  if (!head_dim_supported(dm->head_dim)) return XMOD_ERR_UNSUPPORTED;
  if (routed(kind) && dm->T > topk_max_T()) return XMOD_ERR_UNSUPPORTED;
  if (!aligned16(ws) || ws_bytes < bwd_workspace_bytes(dm)) return XMOD_ERR_WORKSPACE;
  return run_layer_bwd((cudaStream_t)stream, dm, kind, K, gate, w, x, bias, dy, route_coef, dx,
                       g, ws);
}

// The stack backward's workspace: one region the forward recompute and then the
// backward use in turn (both keep the status word at offset 0), then two gradient
// buffers [B, T, d] that the layers' dy / dx alternate between.
static size_t stack_bwd_region(const xmod_dims* dm, int K) {
  const size_t f = layout(dm, K).total, b = bwd_workspace_bytes(dm);
  return align_up(f > b ? f : b);
}

size_t xmod_stack_bwd_workspace_bytes(const xmod_dims* dm, int K) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T) return 0;
  const size_t g = align_up(esize(dm->dtype) * (size_t)dm->B * dm->T * dm->d);
  return stack_bwd_region(dm, K) + 2 * g;
}

int xmod_stack_bwd(const xmod_dims* dm, int K, double A, int N0, int N1, xmod_gate gate,
                   const xmod_layer_weights* layers, int n_layers, const void* x,
                   const float* bias, const void* dy, float route_coef, void* dx,
                   const xmod_layer_grads* grads, void* checkpoints, void* ws, size_t ws_bytes,
                   void* stream) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T || N0 < 0 || N1 < 0 || !layers || !grads)
    return XMOD_ERR_INVALID_ARG;
  if (!isfinite(A) || A <= 0) return XMOD_ERR_INVALID_ARG;
  const double akd = A * (double)K;
  const long AK = lround(akd);
  if (AK < 1 || fabs(akd - (double)AK) > 1e-9) return XMOD_ERR_INVALID_ARG;
  if (n_layers < 1 || (long)n_layers != (long)N0 + (long)N1 * (AK + 1))
    return XMOD_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || !aligned16(checkpoints) ||
      !aligned16_or_null(bias))
    return XMOD_ERR_INVALID_ARG;
  const size_t sz = esize(dm->dtype) * (size_t)dm->B * dm->T * dm->d;
  const char* ck = (const char*)checkpoints;
  if (dx == x || dx == dy || ((const char*)dx + sz > ck && (const char*)dx < ck + sz * n_layers))
    return XMOD_ERR_INVALID_ARG;
  if (!aligned16(ws) || ws_bytes < xmod_stack_bwd_workspace_bytes(dm, K))
    return XMOD_ERR_WORKSPACE;
  const size_t region = stack_bwd_region(dm, K);
  char* gbuf[2] = {(char*)ws + region, (char*)ws + region + align_up(sz)};
  cudaStream_t st = (cudaStream_t)stream;
  auto kind_of = [&](int l) {
    return (l >= N0 && ((l - N0) % (AK + 1)) < AK) ? XMOD_LAYER_SPARSE : XMOD_LAYER_DENSE;
  };
  // forward: checkpoint l is the input of layer l
  char* ckp = (char*)checkpoints;
  if (cudaMemcpyAsync(ckp, x, sz, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return XMOD_ERR_CUDA;
  for (int l = 0; l + 1 < n_layers; ++l) {
    char* nxt = ckp + sz * (l + 1);
    if (cudaMemcpyAsync(nxt, ckp + sz * l, sz, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return XMOD_ERR_CUDA;
    const int k = kind_of(l);
    const int r = xmod_layer_fwd(dm, (xmod_layer_kind)k, K, gate, &layers[l], nxt,
                                 k == XMOD_LAYER_SPARSE ? bias : nullptr, nullptr, nullptr, ws,
                                 region, stream);
    if (r) return r;
  }
  // backward, last layer first
  const void* g = dy;
  for (int l = n_layers - 1; l >= 0; --l) {
    void* out = l == 0 ? dx : (void*)gbuf[l & 1];
    const int k = kind_of(l);
    const int r = xmod_layer_bwd(dm, (xmod_layer_kind)k, K, gate, &layers[l], ckp + sz * l,
                                 k == XMOD_LAYER_SPARSE ? bias : nullptr, g, route_coef, out,
                                 &grads[l], ws, region, stream);
    if (r) return r;
    g = out;
  }
  return XMOD_OK;
}

int xmod_layer_fwd(const xmod_dims* dm, xmod_layer_kind kind, int K, xmod_gate gate,
                   const xmod_layer_weights* w, void* x_inout, const float* bias,
                   int32_t* idx_out, float* r_sel_out, void* ws, size_t ws_bytes, void* stream) {
  if (!dims_ok(dm)) return XMOD_ERR_INVALID_ARG;
  if (!kind_ok(kind)) return XMOD_ERR_INVALID_ARG;
  if (gate != XMOD_GATE_XMOD && gate != XMOD_GATE_MOD) return XMOD_ERR_INVALID_ARG;
  if (routed(kind) && (K <= 0 || K > dm->T)) return XMOD_ERR_INVALID_ARG;
  if (!aligned16(x_inout) || !aligned16_or_null(bias) || !aligned16_or_null(idx_out) ||
      !aligned16_or_null(r_sel_out) || !weights_ok(w, kind))
    return XMOD_ERR_INVALID_ARG;
  if (!head_dim_supported(dm->head_dim)) return XMOD_ERR_UNSUPPORTED;
  if (routed(kind) && dm->T > topk_max_T()) return XMOD_ERR_UNSUPPORTED;
  const int Kw = routed(kind) ? K : 1;
  int st = check_ws(dm, Kw, ws, ws_bytes);
  if (st) return st;
  const Layout L = layout(dm, Kw);
  Ctx c;
  st = make_ctx(dm, ws, L, stream, c);
  if (st) return st;
  return layer_impl(c, dm, kind, Kw, gate, w, x_inout, bias, idx_out, r_sel_out, ws, L);
}

int xmod_layer_fwd_threshold(const xmod_dims* dm, xmod_gate gate, const xmod_layer_weights* w,
                             void* x_inout, const float* bias, int32_t* count_out, void* ws,
                             size_t ws_bytes, void* stream) {
  if (!dims_ok(dm) || !weights_ok(w, XMOD_LAYER_SPARSE)) return XMOD_ERR_INVALID_ARG;
  if (gate != XMOD_GATE_XMOD && gate != XMOD_GATE_MOD) return XMOD_ERR_INVALID_ARG;
  if (!aligned16(x_inout) || !aligned16_or_null(bias) || ((uintptr_t)count_out & 3))
    return XMOD_ERR_INVALID_ARG;
  if (!head_dim_supported(dm->head_dim)) return XMOD_ERR_UNSUPPORTED;
  int st = check_ws(dm, 1, ws, ws_bytes);
  if (st) return st;
  const Layout L = layout(dm, 1);
  if (!threshold_supported(dm, ws, L)) return XMOD_ERR_UNSUPPORTED;
  Ctx c;
  st = make_ctx(dm, ws, L, stream, c);
  if (st) return st;
  st = sparse_run(c, dm, L, ws, 1, gate, w, 1, x_inout, bias, nullptr, nullptr, nullptr, true);
  if (st) return st;
  if (count_out && cudaMemcpyAsync(count_out, at(ws, L.seq), sizeof(int32_t) * dm->B,
                                   cudaMemcpyDeviceToDevice, c.stream) != cudaSuccess)
    return XMOD_ERR_CUDA;
  return XMOD_OK;
}

int xmod_stack_fwd(const xmod_dims* dm, int K, double A, int N0, int N1, xmod_gate gate,
                   const xmod_layer_weights* layers, int n_layers, void* x_inout,
                   const float* bias, void* ws, size_t ws_bytes, void* stream) {
  return xmod_stack_fwd_ex(dm, K, A, N0, N1, gate, layers, n_layers, x_inout, bias, nullptr, ws,
                           ws_bytes, stream);
}

int xmod_stack_fwd_ex(const xmod_dims* dm, int K, double A, int N0, int N1, xmod_gate gate,
                      const xmod_layer_weights* layers, int n_layers, void* x_inout,
                      const float* bias, const xmod_stack_opts* opts, void* ws, size_t ws_bytes,
                      void* stream) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T || N0 < 0 || N1 < 0 || !layers) return XMOD_ERR_INVALID_ARG;
  if (!isfinite(A) || A <= 0) return XMOD_ERR_INVALID_ARG;
  const double akd = A * (double)K;
  const long AK = lround(akd);
  if (AK < 1 || fabs(akd - (double)AK) > 1e-9) return XMOD_ERR_INVALID_ARG;
  if ((long)n_layers != (long)N0 + (long)N1 * (AK + 1)) return XMOD_ERR_INVALID_ARG;
  // Eq. 3 order: N0 dense, then N1 blocks of AK sparse layers and one dense anchor.
  std::vector<int32_t> kinds(n_layers);
  for (int l = 0; l < n_layers; ++l)
    kinds[l] = (l >= N0 && ((l - N0) % (AK + 1)) < AK) ? XMOD_LAYER_SPARSE : XMOD_LAYER_DENSE;
  return stack_impl(dm, K, kinds.data(), n_layers, gate, layers, x_inout, bias, opts, ws, ws_bytes,
                    (cudaStream_t)stream);
}

int xmod_stack_fwd_sched(const xmod_dims* dm, int K, const int32_t* kinds, int n_layers,
                         xmod_gate gate, const xmod_layer_weights* layers, void* x_inout,
                         const float* bias, const xmod_stack_opts* opts, void* ws,
                         size_t ws_bytes, void* stream) {
  if (!dims_ok(dm) || K <= 0 || K > dm->T || !kinds || n_layers < 0 || !layers)
    return XMOD_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (!kind_ok(kinds[l])) return XMOD_ERR_INVALID_ARG;
  return stack_impl(dm, K, kinds, n_layers, gate, layers, x_inout, bias, opts, ws, ws_bytes,
                    (cudaStream_t)stream);
}

}  // extern "C"
