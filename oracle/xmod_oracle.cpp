// CPU oracle for the X-MoD / MoD sparse-depth layer forward pass.
//
// TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and the
// cpu_baseline / reference legs of bench.py may load this library. The CUDA
// library never includes, links or calls anything in this directory, and this
// file includes nothing from the CUDA library.
//
// Everything is computed in double precision with plain loops, in the order the
// method states its steps. Loops over independent rows or (sequence, head)
// pairs are spread over OpenMP threads; that changes no arithmetic.
//
// Sources (page: "X-MoD: Practical Scaling Laws for Sparse-Depth Routing Beyond
// Mixture-of-Depths", reading notes; page: "Mixture-of-Depths explained"):
//   router            X-MoD notes, Eq. 8 (router logit plus token-choice bias, sigmoid gate);
//                     MoD blog, "MoDLayer" listing (router = Linear(d, 1) + sigmoid)
//   top-(T/K)         X-MoD notes, "MoD structural limit" section and Eq. 1 (top-1/K tokens);
//                     MoD blog listing (topk over int(seq_len * capacity))
//   gather            MoD blog listing (boolean-mask gather keeps position order)
//   block             X-MoD notes, "backbone configuration" (GQA attention, standard FFN,
//                     Table 4); textbook chapter on dense Transformers (SwiGLU: three d x d_ff
//                     matrices, no bias); pre-norm RMSNorm before attention and before FFN
//   gated residual    X-MoD notes, Eq. 6 (MoD) and Eq. 7 (X-MoD); skip path y = x
//
// Readings where the pages are silent (each also listed in the design notes):
//   * the bias is passed already signed and is ADDED to the logit (Eq. 8 writes s - tau*b);
//   * the gate r includes the bias, as Eq. 8 defines r;
//   * selection ranks the logit s, not r = sigmoid(s) (same order in exact arithmetic);
//     ties go to the lower position; -0.0 equals +0.0; a non-finite logit is an error;
//   * n = floor(T / K) tokens are selected per sequence;
//   * no positional encoding, natural-exp softmax with scale 1/sqrt(head_dim);
//   * FFN input is h = x_sel + a (the ungated in-block residual);
//   * dense layers: y = x + a + f for every token.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

typedef struct {
  int B, T, d, hq, hkv, hd, F;
  double eps;
} oracle_dims;

// Matrices are [out, in] row-major (the nn.Linear layout):
//   wq [hq*hd, d], wk [hkv*hd, d], wv [hkv*hd, d], wo [d, hq*hd],
//   wg [F, d], wu [F, d], wd [d, F]; w_r, g1, g2 are [d].
// Optional, Qwen3-style (X-MoD notes, "backbone configuration": Qwen3 backbones):
//   gq, gk [hd]   QK-norm gains: each head's q and k vector is RMS-normalised and
//                 scaled by them before the rotation (NULL: no QK-norm);
//   rope_theta    rotary position embedding base (0: none), applied to q and k at the
//                 token's original position in its sequence.
typedef struct {
  const double *w_r, *g1, *wq, *wk, *wv, *wo, *g2, *wg, *wu, *wd;
  double varsigma;
  const double *gq, *gk;
  double rope_theta;
} oracle_layer_w;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = -1, ORACLE_NONFINITE = -5 };
enum { ORACLE_GATE_XMOD = 0, ORACLE_GATE_MOD = 1 };
// Layer kinds. ATTN and RFFN are the two halves of the Routed-FFN variant of X-MoD
// notes "mechanism controls" (Table 2 / Table 7): attention over the full sequence with
// its residual, and an FFN-only refinement applied to the top-(T/K) tokens.
// FULLKV is the Selected-Q / full-KV control of the same section: a sparse layer
// whose selected tokens attend to every token at or before their position.
enum { ORACLE_DENSE = 0, ORACLE_SPARSE = 1, ORACLE_ATTN = 2, ORACLE_RFFN = 3, ORACLE_FULLKV = 4 };

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

// Round to the nearest bfloat16 value (8 significant bits), ties to even.
// Used only to mirror a bf16 residual stream between layers.
double oracle_round_bf16(double v) {
  if (v == 0.0 || !std::isfinite(v)) return v;
  int e;
  std::frexp(v, &e);                      // v = m * 2^e, 0.5 <= |m| < 1
  double ulp = std::ldexp(1.0, e - 8);    // 8 significant bits
  return std::nearbyint(v / ulp) * ulp;   // default rounding mode: nearest-even
}

// The same rounding applied to n values in place.
void oracle_round_bf16_n(int64_t n, double* v) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) v[i] = oracle_round_bf16(v[i]);
}

// Eq. 8: s_i = w_r . x_i + b_i, r_i = sigmoid(s_i).
void oracle_router(int64_t rows, int d, const double* x, const double* w_r,
                   const double* bias, double* s, double* r) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows; ++i) {
    double acc = 0.0;
    for (int j = 0; j < d; ++j) acc += w_r[j] * x[i * d + j];
    if (bias) acc += bias[i];
    s[i] = acc;
    if (r) r[i] = 1.0 / (1.0 + std::exp(-acc));
  }
}

// Per-sequence top-k: the k largest logits, ties to the lower position, returned
// as ascending positions. Brute force: order all positions by (-s, position).
int oracle_topk(int B, int T, int k, const double* s, int32_t* idx) {
  if (B < 0 || T <= 0 || k <= 0 || k > T) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < (int64_t)B * T; ++i)
    if (!std::isfinite(s[i])) return ORACLE_NONFINITE;
  for (int b = 0; b < B; ++b) {
    const double* sb = s + (int64_t)b * T;
    std::vector<int32_t> order(T);
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(), [sb](int32_t p, int32_t q) {
      if (sb[p] != sb[q]) return sb[p] > sb[q];
      return p < q;
    });
    std::sort(order.begin(), order.begin() + k);
    for (int j = 0; j < k; ++j) idx[(int64_t)b * k + j] = order[j];
  }
  return ORACLE_OK;
}

// RMSNorm: out = x / sqrt(mean(x^2) + eps) * gamma.
void oracle_rmsnorm(int64_t rows, int d, const double* x, const double* gamma,
                    double eps, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows; ++i) {
    double ss = 0.0;
    for (int j = 0; j < d; ++j) ss += x[i * d + j] * x[i * d + j];
    double inv = 1.0 / std::sqrt(ss / d + eps);
    for (int j = 0; j < d; ++j) out[i * d + j] = x[i * d + j] * inv * gamma[j];
  }
}

// y[rows, out] = x[rows, in] . W[out, in]^T
void oracle_linear(int64_t rows, int in, int out, const double* x, const double* W,
                   double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < rows; ++i) {
    for (int o = 0; o < out; ++o) {
      double acc = 0.0;
      for (int j = 0; j < in; ++j) acc += x[i * in + j] * W[(int64_t)o * in + j];
      y[i * out + o] = acc;
    }
  }
}

// Causal grouped-query attention over one sequence of n tokens.
// q [n, hq*hd], k and v [n, hkv*hd]; query head h reads KV head h / (hq/hkv).
// o[i, h] = sum_{j<=i} softmax_j(q_i.k_j / sqrt(hd)) v_j.
// Only the rows listed in `rows` (nrows of them) are computed; rows == NULL means all.
// QK-norm and rotary embedding of `rows` vectors x [rows, heads * hd] in place. Row i
// sits at position pos[i] (NULL: i). QK-norm: x_h <- x_h / sqrt(mean(x_h^2) + eps) *
// gain. Rotation (the rotate-half pairing of the Qwen / LLaMA family): for
// c < hd/2, angle = pos * theta^(-2c/hd), (x_c, x_{c+hd/2}) <- (x_c cos - x_{c+hd/2} sin,
// x_c sin + x_{c+hd/2} cos).
void oracle_qk_transform(int rows, int heads, int hd, double* x, const double* gain, double eps,
                         double theta, const int32_t* pos) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < rows; ++i) {
    const double p = pos ? (double)pos[i] : (double)i;
    for (int h = 0; h < heads; ++h) {
      double* v = x + ((int64_t)i * heads + h) * hd;
      if (gain) {
        double ss = 0.0;
        for (int c = 0; c < hd; ++c) ss += v[c] * v[c];
        const double inv = 1.0 / std::sqrt(ss / hd + eps);
        for (int c = 0; c < hd; ++c) v[c] = v[c] * inv * gain[c];
      }
      if (theta > 0.0) {
        const int half = hd / 2;
        for (int c = 0; c < half; ++c) {
          const double ang = p * std::pow(theta, -2.0 * c / hd);
          const double cs = std::cos(ang), sn = std::sin(ang);
          const double a = v[c], b = v[c + half];
          v[c] = a * cs - b * sn;
          v[c + half] = a * sn + b * cs;
        }
      }
    }
  }
}

void oracle_attention_rows(int n, int hq, int hkv, int hd, const double* q,
                           const double* k, const double* v, double* o,
                           const int32_t* rows, int nrows) {
  const int G = hq / hkv;
  const double scale = 1.0 / std::sqrt((double)hd);
  const int nr = rows ? nrows : n;
  const int qs = hq * hd, ks = hkv * hd;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int ri = 0; ri < nr; ++ri) {
    for (int h = 0; h < hq; ++h) {
      const int i = rows ? rows[ri] : ri;
      const int g = h / G;
      std::vector<double> sc(i + 1);
      double m = -INFINITY;
      for (int j = 0; j <= i; ++j) {
        double acc = 0.0;
        for (int c = 0; c < hd; ++c)
          acc += q[(int64_t)i * qs + h * hd + c] * k[(int64_t)j * ks + g * hd + c];
        sc[j] = acc * scale;
        m = std::max(m, sc[j]);
      }
      double denom = 0.0;
      for (int j = 0; j <= i; ++j) {
        sc[j] = std::exp(sc[j] - m);
        denom += sc[j];
      }
      for (int c = 0; c < hd; ++c) {
        double acc = 0.0;
        for (int j = 0; j <= i; ++j) acc += sc[j] * v[(int64_t)j * ks + g * hd + c];
        o[(int64_t)ri * qs + h * hd + c] = acc / denom;
      }
    }
  }
}

static inline double silu(double z) { return z / (1.0 + std::exp(-z)); }

// Gated residual of one selected row (Eq. 7 for gate == XMOD, Eq. 6 for gate == MOD):
//   Eq. 7: y = x + varsigma * r * (a + f);   Eq. 6: y = x + a + r * f.
static inline double gated(double x, double a, double f, double r, double varsigma, int gate) {
  if (gate == ORACLE_GATE_XMOD) return x + varsigma * r * (a + f);
  return x + a + r * f;
}

// The scatter step on its own: rows[m] of x [rows_total, d] receives the gated
// residual of a[m], f[m] with gate value r[m]; other rows are left as they are.
// f == NULL means `a` already holds a + f (Eq. 7 only).
void oracle_gated_scatter(int64_t M, int d, double* x, const int64_t* rows, const double* a,
                          const double* f, const double* r, double varsigma, int gate) {
  for (int64_t m = 0; m < M; ++m)
    for (int c = 0; c < d; ++c) {
      double* px = x + rows[m] * d + c;
      const double am = a[m * d + c];
      *px = f ? gated(*px, am, f[m * d + c], r[m], varsigma, gate)
              : gated(*px, am, 0.0, r[m], varsigma, ORACLE_GATE_XMOD);
    }
}

// The transformer block on ONE sequence's compact buffer xs [n, d] (rows in
// position order). Produces the attention residual a and the FFN residual f
// for the requested compact rows (rows == NULL: all n rows), written densely
// in request order: a_out, f_out are [nrows, d].
//   u = RMSNorm(xs) * g1;  q,k,v = u Wq^T, u Wk^T, u Wv^T
//   o = causal GQA attention;  a = o Wo^T;  h = xs + a
//   v2 = RMSNorm(h) * g2;  f = (silu(v2 Wg^T) * (v2 Wu^T)) Wd^T
// As oracle_block_rows; compact row j sits at original position pos[j] (NULL: j),
// which only the rotary embedding sees.
void oracle_block_rows_pos(const oracle_dims* dm, int n, const double* xs,
                           const oracle_layer_w* w, const int32_t* rows, int nrows,
                           double* a_out, double* f_out, const int32_t* pos);

void oracle_block_rows(const oracle_dims* dm, int n, const double* xs,
                       const oracle_layer_w* w, const int32_t* rows, int nrows,
                       double* a_out, double* f_out) {
  oracle_block_rows_pos(dm, n, xs, w, rows, nrows, a_out, f_out, nullptr);
}

void oracle_block_rows_pos(const oracle_dims* dm, int n, const double* xs,
                           const oracle_layer_w* w, const int32_t* rows, int nrows,
                           double* a_out, double* f_out, const int32_t* pos) {
  const int d = dm->d, hq = dm->hq, hkv = dm->hkv, hd = dm->hd, F = dm->F;
  const int nr = rows ? nrows : n;
  if (nr <= 0) return;
  // Keys and values are needed for every compact row up to the last requested one.
  int last = n - 1;
  if (rows) {
    last = 0;
    for (int i = 0; i < nr; ++i) last = std::max(last, rows[i]);
  }
  const int nkv = last + 1;
  std::vector<double> u((int64_t)nkv * d);
  oracle_rmsnorm(nkv, d, xs, w->g1, dm->eps, u.data());
  std::vector<double> kk((int64_t)nkv * hkv * hd), vv((int64_t)nkv * hkv * hd);
  oracle_linear(nkv, d, hkv * hd, u.data(), w->wk, kk.data());
  oracle_linear(nkv, d, hkv * hd, u.data(), w->wv, vv.data());
  if (w->gk || w->rope_theta > 0.0)
    oracle_qk_transform(nkv, hkv, hd, kk.data(), w->gk, dm->eps, w->rope_theta, pos);
  // Queries for the requested rows only.
  std::vector<double> ur((int64_t)nr * d), xr((int64_t)nr * d);
  for (int i = 0; i < nr; ++i) {
    const int src = rows ? rows[i] : i;
    std::memcpy(&ur[(int64_t)i * d], &u[(int64_t)src * d], sizeof(double) * d);
    std::memcpy(&xr[(int64_t)i * d], &xs[(int64_t)src * d], sizeof(double) * d);
  }
  std::vector<double> qfull((int64_t)nkv * hq * hd, 0.0);
  {
    std::vector<double> qr((int64_t)nr * hq * hd);
    oracle_linear(nr, d, hq * hd, ur.data(), w->wq, qr.data());
    if (w->gq || w->rope_theta > 0.0) {
      std::vector<int32_t> qpos(nr);
      for (int i = 0; i < nr; ++i) {
        const int src = rows ? rows[i] : i;
        qpos[i] = pos ? pos[src] : src;
      }
      oracle_qk_transform(nr, hq, hd, qr.data(), w->gq, dm->eps, w->rope_theta, qpos.data());
    }
    for (int i = 0; i < nr; ++i) {
      const int dst = rows ? rows[i] : i;
      std::memcpy(&qfull[(int64_t)dst * hq * hd], &qr[(int64_t)i * hq * hd],
                  sizeof(double) * hq * hd);
    }
  }
  std::vector<double> o((int64_t)nr * hq * hd);
  std::vector<int32_t> all;
  const int32_t* rr = rows;
  if (!rows) {
    all.resize(n);
    std::iota(all.begin(), all.end(), 0);
    rr = all.data();
  }
  oracle_attention_rows(nkv, hq, hkv, hd, qfull.data(), kk.data(), vv.data(), o.data(),
                        rr, nr);
  oracle_linear(nr, hq * hd, d, o.data(), w->wo, a_out);
  std::vector<double> h((int64_t)nr * d), v2((int64_t)nr * d);
  for (int64_t i = 0; i < (int64_t)nr * d; ++i) h[i] = xr[i] + a_out[i];
  oracle_rmsnorm(nr, d, h.data(), w->g2, dm->eps, v2.data());
  std::vector<double> g((int64_t)nr * F), up((int64_t)nr * F), hid((int64_t)nr * F);
  oracle_linear(nr, d, F, v2.data(), w->wg, g.data());
  oracle_linear(nr, d, F, v2.data(), w->wu, up.data());
  for (int64_t i = 0; i < (int64_t)nr * F; ++i) hid[i] = silu(g[i]) * up[i];
  oracle_linear(nr, F, d, hid.data(), w->wd, f_out);
}

// FFN of the block without attention, on nr rows xs [nr, d]:
//   f = W_down(silu(W_gate v2) * (W_up v2)), v2 = RMSNorm(xs) * g2.
void oracle_ffn_rows(const oracle_dims* dm, int nr, const double* xs, const oracle_layer_w* w,
                     double* f_out) {
  const int d = dm->d, F = dm->F;
  if (nr <= 0) return;
  std::vector<double> v2((int64_t)nr * d);
  oracle_rmsnorm(nr, d, xs, w->g2, dm->eps, v2.data());
  std::vector<double> g((int64_t)nr * F), up((int64_t)nr * F), hid((int64_t)nr * F);
  oracle_linear(nr, d, F, v2.data(), w->wg, g.data());
  oracle_linear(nr, d, F, v2.data(), w->wu, up.data());
  for (int64_t i = 0; i < (int64_t)nr * F; ++i) hid[i] = silu(g[i]) * up[i];
  oracle_linear(nr, F, d, hid.data(), w->wd, f_out);
}

// Block of a Selected-Q / full-KV layer for one sequence x_seq [T, d]: the n selected
// tokens (ascending positions pos) are the queries; every token provides keys and
// values (RMSNorm1 of every token); query j attends to the positions <= pos[j].
// a_out, f_out [n, d].
void oracle_block_fullkv(const oracle_dims* dm, int T, const double* x_seq,
                         const oracle_layer_w* w, const int32_t* pos, int n, double* a_out,
                         double* f_out) {
  const int d = dm->d, hq = dm->hq, hkv = dm->hkv, hd = dm->hd, F = dm->F;
  if (n <= 0) return;
  std::vector<double> u((int64_t)T * d);
  oracle_rmsnorm(T, d, x_seq, w->g1, dm->eps, u.data());
  std::vector<double> kk((int64_t)T * hkv * hd), vv((int64_t)T * hkv * hd);
  oracle_linear(T, d, hkv * hd, u.data(), w->wk, kk.data());
  oracle_linear(T, d, hkv * hd, u.data(), w->wv, vv.data());
  if (w->gk || w->rope_theta > 0.0)
    oracle_qk_transform(T, hkv, hd, kk.data(), w->gk, dm->eps, w->rope_theta, nullptr);
  std::vector<double> us((int64_t)n * d), xr((int64_t)n * d), qs((int64_t)n * hq * hd);
  for (int j = 0; j < n; ++j) {
    std::memcpy(&us[(int64_t)j * d], &u[(int64_t)pos[j] * d], sizeof(double) * d);
    std::memcpy(&xr[(int64_t)j * d], &x_seq[(int64_t)pos[j] * d], sizeof(double) * d);
  }
  oracle_linear(n, d, hq * hd, us.data(), w->wq, qs.data());
  if (w->gq || w->rope_theta > 0.0)
    oracle_qk_transform(n, hq, hd, qs.data(), w->gq, dm->eps, w->rope_theta, pos);
  std::vector<double> qfull((int64_t)T * hq * hd, 0.0);
  for (int j = 0; j < n; ++j)
    std::memcpy(&qfull[(int64_t)pos[j] * hq * hd], &qs[(int64_t)j * hq * hd],
                sizeof(double) * hq * hd);
  std::vector<double> o((int64_t)n * hq * hd);
  oracle_attention_rows(T, hq, hkv, hd, qfull.data(), kk.data(), vv.data(), o.data(), pos, n);
  oracle_linear(n, hq * hd, d, o.data(), w->wo, a_out);
  std::vector<double> h((int64_t)n * d), v2((int64_t)n * d);
  for (int64_t i = 0; i < (int64_t)n * d; ++i) h[i] = xr[i] + a_out[i];
  oracle_rmsnorm(n, d, h.data(), w->g2, dm->eps, v2.data());
  std::vector<double> g((int64_t)n * F), up((int64_t)n * F), hid((int64_t)n * F);
  oracle_linear(n, d, F, v2.data(), w->wg, g.data());
  oracle_linear(n, d, F, v2.data(), w->wu, up.data());
  for (int64_t i = 0; i < (int64_t)n * F; ++i) hid[i] = silu(g[i]) * up[i];
  oracle_linear(n, F, d, hid.data(), w->wd, f_out);
}

// One layer of the stack on x_in [B, T, d] -> y [B, T, d].
//   sparse: router (Eq. 8) -> top-(T/K) -> gather -> block -> gated residual
//           (Eq. 7 if gate == XMOD, Eq. 6 if gate == MOD); unselected rows y = x.
//   dense:  block on all T tokens, y = x + a + f.
//   attn:   attention half of the block on all T tokens, y = x + a.
//   rffn:   router -> top-(T/K) -> gather -> FFN half on the selected tokens ->
//           gated residual with a = 0 (Eq. 7: x + varsigma r f; Eq. 6: x + r f).
//   fullkv: as sparse, but the selected tokens attend to every token (keys and values
//           of all T) at or before their own position.
// Optional arguments:
//   bias      [B, T]  signed per-token router bias, added to the logit;
//   s_out     [B, T]  router logits; r_out [B, T] gates;
//   idx_out   [B, n]  selected positions (ascending); rsel_out [B, n] their gates;
//   idx_force [B, n]  use these positions instead of the oracle's own top-k (used to
//                     decouple block parity from near-tie routing decisions; must
//                     be ascending and in range);
//   row_mask  [B, T]  nonzero marks output rows that are wanted; other rows are
//                     copied from x_in (NULL: all rows computed).
// Returns ORACLE_OK, ORACLE_BAD_ARG or ORACLE_NONFINITE.
int oracle_layer_fwd(const oracle_dims* dm, int kind, int K, int gate,
                     const oracle_layer_w* w, const double* x_in, const double* bias,
                     double* y, double* s_out, double* r_out, int32_t* idx_out,
                     double* rsel_out, const int32_t* idx_force, const int32_t* row_mask) {
  const int B = dm->B, T = dm->T, d = dm->d;
  if (B <= 0 || T <= 0 || d <= 0 || dm->hq % dm->hkv != 0) return ORACLE_BAD_ARG;
  const int64_t BT = (int64_t)B * T;
  std::memcpy(y, x_in, sizeof(double) * BT * d);
  if (kind == ORACLE_DENSE || kind == ORACLE_ATTN) {
    for (int b = 0; b < B; ++b) {
      std::vector<int32_t> rows;
      for (int t = 0; t < T; ++t)
        if (!row_mask || row_mask[(int64_t)b * T + t]) rows.push_back(t);
      if (rows.empty()) continue;
      const double* xb = x_in + (int64_t)b * T * d;
      std::vector<double> a(rows.size() * (size_t)d), f(rows.size() * (size_t)d);
      oracle_block_rows(dm, T, xb, w, rows.data(), (int)rows.size(), a.data(), f.data());
      for (size_t i = 0; i < rows.size(); ++i)
        for (int c = 0; c < d; ++c) {
          const int64_t o = ((int64_t)b * T + rows[i]) * d + c;
          y[o] = kind == ORACLE_ATTN ? x_in[o] + a[i * d + c] : x_in[o] + a[i * d + c] + f[i * d + c];
        }
    }
    return ORACLE_OK;
  }
  if ((kind != ORACLE_SPARSE && kind != ORACLE_RFFN && kind != ORACLE_FULLKV) || K <= 0)
    return ORACLE_BAD_ARG;
  const int n = T / K;
  if (n <= 0) return ORACLE_BAD_ARG;
  std::vector<double> s(BT), r(BT);
  oracle_router(BT, d, x_in, w->w_r, bias, s.data(), r.data());
  if (s_out) std::memcpy(s_out, s.data(), sizeof(double) * BT);
  if (r_out) std::memcpy(r_out, r.data(), sizeof(double) * BT);
  std::vector<int32_t> idx((int64_t)B * n);
  if (idx_force) {
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < n; ++j) {
        const int32_t p = idx_force[(int64_t)b * n + j];
        if (p < 0 || p >= T || (j > 0 && p <= idx_force[(int64_t)b * n + j - 1]))
          return ORACLE_BAD_ARG;
        idx[(int64_t)b * n + j] = p;
      }
  } else {
    int st = oracle_topk(B, T, n, s.data(), idx.data());
    if (st != ORACLE_OK) return st;
  }
  if (idx_out) std::memcpy(idx_out, idx.data(), sizeof(int32_t) * B * n);
  if (rsel_out)
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < n; ++j)
        rsel_out[(int64_t)b * n + j] = r[(int64_t)b * T + idx[(int64_t)b * n + j]];
  for (int b = 0; b < B; ++b) {
    // gather in position order
    std::vector<double> xs((int64_t)n * d);
    for (int j = 0; j < n; ++j)
      std::memcpy(&xs[(int64_t)j * d], x_in + ((int64_t)b * T + idx[(int64_t)b * n + j]) * d,
                  sizeof(double) * d);
    std::vector<int32_t> rows;
    for (int j = 0; j < n; ++j)
      if (!row_mask || row_mask[(int64_t)b * T + idx[(int64_t)b * n + j]]) rows.push_back(j);
    if (rows.empty()) continue;
    std::vector<double> a(rows.size() * (size_t)d, 0.0), f(rows.size() * (size_t)d);
    if (kind == ORACLE_FULLKV) {
      if (rows.size() != (size_t)n) return ORACLE_BAD_ARG;   // no row mask here
      oracle_block_fullkv(dm, T, x_in + (int64_t)b * T * d, w, &idx[(int64_t)b * n], n, a.data(),
                          f.data());
    } else if (kind == ORACLE_RFFN) {   // FFN only, row by row: attention context plays no part
      std::vector<double> xr(rows.size() * (size_t)d);
      for (size_t i = 0; i < rows.size(); ++i)
        std::memcpy(&xr[i * d], &xs[(int64_t)rows[i] * d], sizeof(double) * d);
      oracle_ffn_rows(dm, (int)rows.size(), xr.data(), w, f.data());
    } else {
      oracle_block_rows_pos(dm, n, xs.data(), w, rows.data(), (int)rows.size(), a.data(), f.data(),
                            &idx[(int64_t)b * n]);   // original positions for the rotation
    }
    for (size_t i = 0; i < rows.size(); ++i) {
      const int j = rows[i];
      const int t = idx[(int64_t)b * n + j];
      const double rt = r[(int64_t)b * T + t];
      for (int c = 0; c < d; ++c) {
        const int64_t o = ((int64_t)b * T + t) * d + c;
        y[o] = gated(x_in[o], a[i * d + c], f[i * d + c], rt, w->varsigma, gate);
      }
    }
  }
  return ORACLE_OK;
}

// Whole stack: layers applied in the given order (kinds[l] = DENSE or SPARSE).
// The same bias is used by every sparse layer. With mirror_bf16 != 0 the
// residual stream is rounded to bf16 after every layer, as a bf16 stream stores it.
// seq_mask [B] (nullable): only sequences with a nonzero entry are computed;
// the others keep their input values. x is updated in place.
int oracle_stack_fwd(const oracle_dims* dm, int K, int gate, int n_layers, const int* kinds,
                     const oracle_layer_w* layers, double* x, const double* bias,
                     int mirror_bf16, const int32_t* seq_mask) {
  const int64_t BT = (int64_t)dm->B * dm->T;
  const int64_t N = BT * dm->d;
  std::vector<int32_t> row_mask;
  if (seq_mask) {
    row_mask.resize(BT);
    for (int b = 0; b < dm->B; ++b)
      for (int t = 0; t < dm->T; ++t) row_mask[(int64_t)b * dm->T + t] = seq_mask[b] ? 1 : 0;
  }
  std::vector<double> y(N);
  for (int l = 0; l < n_layers; ++l) {
    int st = oracle_layer_fwd(dm, kinds[l], K, gate, &layers[l], x, bias, y.data(), nullptr,
                              nullptr, nullptr, nullptr, nullptr,
                              seq_mask ? row_mask.data() : nullptr);
    if (st != ORACLE_OK) return st;
    if (mirror_bf16)
      for (int64_t i = 0; i < N; ++i) y[i] = oracle_round_bf16(y[i]);
    std::memcpy(x, y.data(), sizeof(double) * N);
  }
  return ORACLE_OK;
}

// Sparse layer under the causal threshold rule of X-MoD notes "top-k in training,
// causal threshold at evaluation": token i enters the block when its routing
// probability r_i = sigmoid(s_i) is at least 1/2, i.e. s_i >= 0 (-0 counts as 0),
// each token deciding alone, so a sequence takes a variable number of tokens (none
// at all is allowed: then the sequence is unchanged). The selected tokens go through
// the block in position order, attention causal among them, and the gated residual
// (Eq. 7 / Eq. 6) with their own r. mask_out [B, T] (nullable) receives the decisions.
int oracle_layer_threshold(const oracle_dims* dm, int gate, const oracle_layer_w* w,
                           const double* x_in, const double* bias, double* y, double* s_out,
                           int32_t* mask_out) {
  const int B = dm->B, T = dm->T, d = dm->d;
  if (B <= 0 || T <= 0 || d <= 0 || dm->hq % dm->hkv != 0) return ORACLE_BAD_ARG;
  const int64_t BT = (int64_t)B * T;
  std::memcpy(y, x_in, sizeof(double) * BT * d);
  std::vector<double> s(BT), r(BT);
  oracle_router(BT, d, x_in, w->w_r, bias, s.data(), r.data());
  for (int64_t i = 0; i < BT; ++i)
    if (!std::isfinite(s[i])) return ORACLE_NONFINITE;
  if (s_out) std::memcpy(s_out, s.data(), sizeof(double) * BT);
  for (int b = 0; b < B; ++b) {
    std::vector<int32_t> pos;   // ascending positions
    for (int t = 0; t < T; ++t) {
      const bool take = s[(int64_t)b * T + t] >= 0.0;
      if (mask_out) mask_out[(int64_t)b * T + t] = take ? 1 : 0;
      if (take) pos.push_back(t);
    }
    const int n = (int)pos.size();
    if (n == 0) continue;
    std::vector<double> xs((int64_t)n * d);
    for (int j = 0; j < n; ++j)
      std::memcpy(&xs[(int64_t)j * d], x_in + ((int64_t)b * T + pos[j]) * d, sizeof(double) * d);
    std::vector<int32_t> rows(n);
    std::iota(rows.begin(), rows.end(), 0);
    std::vector<double> a((size_t)n * d), f((size_t)n * d);
    oracle_block_rows_pos(dm, n, xs.data(), w, rows.data(), n, a.data(), f.data(), pos.data());
    for (int j = 0; j < n; ++j) {
      const int t = pos[j];
      const double rt = r[(int64_t)b * T + t];
      for (int c = 0; c < d; ++c) {
        const int64_t o = ((int64_t)b * T + t) * d + c;
        y[o] = gated(x_in[o], a[(size_t)j * d + c], f[(size_t)j * d + c], rt, w->varsigma, gate);
      }
    }
  }
  return ORACLE_OK;
}

// Stack with the token-choice bias dynamics of X-MoD notes Eq. 8 and the paragraph
// after it: inside a sparse-dense block, every time token i is selected its bias
// b_i grows, and it is cleared at the next dense anchor. The pages give neither the
// increment nor tau; the reading taken here: the logit of sparse layer l is
//   s_i = w_r . x_i + bias0_i - bias_step * c_i,
// where c_i counts the earlier sparse layers of the current block (since the last
// dense layer or the start of the stack) that selected token i, and bias_step stands
// for tau times the increment. bias_step = 0 is the constant-bias stack.
// Optional outputs, per sparse layer in stack order (n_sparse of them):
//   idx_out [n_sparse, B, n]  its selection;
//   s_out   [n_sparse, B, T]  its logits (with the bias above).
// routing 0: top-(T/K) per sequence; 1: the causal threshold rule above (then K is
// unused by the sparse layers and idx_out must be NULL).
// mask_out [n_sparse, B, T] (nullable): each sparse layer's decisions.
int oracle_stack_dyn(const oracle_dims* dm, int K, int gate, int n_layers, const int* kinds,
                     const oracle_layer_w* layers, double* x, const double* bias0,
                     double bias_step, int mirror_bf16, int32_t* idx_out, double* s_out,
                     int routing, int32_t* mask_out) {
  if (routing != 0 && (routing != 1 || idx_out)) return ORACLE_BAD_ARG;
  const int64_t BT = (int64_t)dm->B * dm->T;
  const int64_t N = BT * dm->d;
  const int n = K > 0 ? dm->T / K : 0;
  std::vector<double> y(N), bias(BT), s(BT);
  std::vector<int32_t> count(BT, 0), idx((int64_t)dm->B * (n > 0 ? n : 1)), mask(BT);
  int ls = 0;
  for (int l = 0; l < n_layers; ++l) {
    const bool sparse = kinds[l] == ORACLE_SPARSE || kinds[l] == ORACLE_RFFN ||
                        kinds[l] == ORACLE_FULLKV;   // routed
    if (sparse)
      for (int64_t i = 0; i < BT; ++i)
        bias[i] = (bias0 ? bias0[i] : 0.0) - bias_step * (double)count[i];
    int st;
    if (sparse && routing == 1) {
      if (kinds[l] != ORACLE_SPARSE) return ORACLE_BAD_ARG;
      st = oracle_layer_threshold(dm, gate, &layers[l], x, bias.data(), y.data(), s.data(),
                                  mask.data());
    } else {
      st = oracle_layer_fwd(dm, kinds[l], K, gate, &layers[l], x, sparse ? bias.data() : nullptr,
                            y.data(), sparse ? s.data() : nullptr, nullptr,
                            sparse ? idx.data() : nullptr, nullptr, nullptr, nullptr);
      if (sparse) {
        std::fill(mask.begin(), mask.end(), 0);
        for (int b = 0; b < dm->B; ++b)
          for (int j = 0; j < n; ++j) mask[(int64_t)b * dm->T + idx[(int64_t)b * n + j]] = 1;
      }
    }
    if (st != ORACLE_OK) return st;
    if (sparse) {
      for (int64_t i = 0; i < BT; ++i) count[i] += mask[i];
      if (mask_out) std::memcpy(mask_out + (int64_t)ls * BT, mask.data(), sizeof(int32_t) * BT);
      if (idx_out) std::memcpy(idx_out + (int64_t)ls * dm->B * n, idx.data(), sizeof(int32_t) * dm->B * n);
      if (s_out) std::memcpy(s_out + (int64_t)ls * BT, s.data(), sizeof(double) * BT);
      ++ls;
    } else if (kinds[l] == ORACLE_DENSE) {
      std::fill(count.begin(), count.end(), 0);   // the dense anchor clears the bias
    }
    if (mirror_bf16)
      for (int64_t i = 0; i < N; ++i) y[i] = oracle_round_bf16(y[i]);
    std::memcpy(x, y.data(), sizeof(double) * N);
  }
  return ORACLE_OK;
}

}  // extern "C"
