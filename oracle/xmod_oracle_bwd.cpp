// CPU oracle for the backward pass of one sparse-depth layer.
//
// TEST INFRASTRUCTURE ONLY (same rules as xmod_oracle.cpp): only tests/,
// __graft_entry__.smoke() and the cpu_baseline / reference legs of bench.py may load
// it; the CUDA library never includes, links or calls anything here.
//
// What is differentiated. For a layer y = layer(x) (X-MoD notes: Eq. 8 router, top-1/K
// selection, the block, Eq. 6 / Eq. 7 gated residual; dense layers y = x + a + f) and a
// caller-given upstream gradient dy, the scalar objective is
//     J = sum(dy * y) + route_coef * L_route,
// where L_route is the binary cross-entropy of Eq. 9 ("top-k in training, causal
// threshold at evaluation"): -(1/N) sum_i [q_i log p_i + (1 - q_i) log(1 - p_i)], with
// q_i = 1 when token i is among the layer's top-(T/K), p_i = sigmoid(s_i) on the same
// (biased) logit the selection ranks, and N = B*T, every token of the layer's input.
// The selection is piecewise constant in the inputs: it is held fixed, so the router is
// trained only through the gate r of the residual (Eq. 6 / Eq. 7) and through Eq. 9.
// The function returns dJ/dx and dJ/d(every weight), plus L_route itself.
//
// Every derivative is the chain rule through the forward steps, written out in double
// with plain loops, in reverse order of the forward:
//   forward  u = RMSNorm(xs) g1; q, k, v = u Wq^T, u Wk^T, u Wv^T; o = attention;
//            a = o Wo^T; h = xs + a; v2 = RMSNorm(h) g2; G, U = v2 Wg^T, v2 Wu^T;
//            H = silu(G) U; f = H Wd^T
//   RMSNorm  z = x rho g with rho = (mean(x^2) + eps)^(-1/2):
//            dx = rho (dz g - xhat mean(dz g xhat)), xhat = x rho; dg = sum dz xhat
//   softmax  dS_ij = P_ij (dP_ij - sum_j' P_ij' dP_ij')
//   silu     silu'(z) = sigma(z) (1 + z (1 - sigma(z)))
//   BCE      d/ds [-q log sigma(s) - (1 - q) log(1 - sigma(s))] = sigma(s) - q
// The pins of this file are finite differences of the forward oracle (tests).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

extern "C" {

typedef struct {
  int B, T, d, hq, hkv, hd, F;
  double eps;
} oracle_dims;

typedef struct {
  const double *w_r, *g1, *wq, *wk, *wv, *wo, *g2, *wg, *wu, *wd;
  double varsigma;
  const double *gq, *gk;
  double rope_theta;
} oracle_layer_w;

// Gradients, shaped as the weights; every array is overwritten. gq, gk [hd] (the
// QK-norm gains' gradients) may be NULL when the layer has no QK-norm.
typedef struct {
  double *w_r, *g1, *wq, *wk, *wv, *wo, *g2, *wg, *wu, *wd;
  double varsigma;
  double *gq, *gk;
} oracle_layer_grad;

// forward helpers of xmod_oracle.cpp
void oracle_router(int64_t rows, int d, const double* x, const double* w_r,
                   const double* bias, double* s, double* r);
int oracle_topk(int B, int T, int k, const double* s, int32_t* idx);
void oracle_linear(int64_t rows, int in, int out, const double* x, const double* W, double* y);
void oracle_qk_transform(int rows, int heads, int hd, double* x, const double* gain, double eps,
                         double theta, const int32_t* pos);
void oracle_ffn_rows(const oracle_dims* dm, int nr, const double* xs, const oracle_layer_w* w,
                     double* f_out);
void oracle_block_fullkv(const oracle_dims* dm, int T, const double* x_seq,
                         const oracle_layer_w* w, const int32_t* pos, int n, double* a_out,
                         double* f_out);

}  // extern "C"

namespace {

enum { OK = 0, BAD_ARG = -1 };
enum { DENSE = 0, SPARSE = 1, ATTN = 2, RFFN = 3, FULLKV = 4 };
enum { GATE_XMOD = 0, GATE_MOD = 1 };

double sigmoid(double z) { return 1.0 / (1.0 + std::exp(-z)); }

// z = x rho g per row; keeps xhat = x rho and rho for the backward.
void rms_fwd(int n, int d, const double* x, const double* g, double eps, double* z,
             double* xhat, double* rho) {
  for (int i = 0; i < n; ++i) {
    double ss = 0.0;
    for (int c = 0; c < d; ++c) ss += x[(int64_t)i * d + c] * x[(int64_t)i * d + c];
    rho[i] = 1.0 / std::sqrt(ss / d + eps);
    for (int c = 0; c < d; ++c) {
      xhat[(int64_t)i * d + c] = x[(int64_t)i * d + c] * rho[i];
      z[(int64_t)i * d + c] = xhat[(int64_t)i * d + c] * g[c];
    }
  }
}

// dx += rho (dz g - xhat mean(dz g xhat)); dg += sum_i dz xhat.
void rms_bwd(int n, int d, const double* dz, const double* g, const double* xhat,
             const double* rho, double* dx, double* dg) {
  for (int i = 0; i < n; ++i) {
    double dot = 0.0;
    for (int c = 0; c < d; ++c) dot += dz[(int64_t)i * d + c] * g[c] * xhat[(int64_t)i * d + c];
    const double mean = dot / d;
    for (int c = 0; c < d; ++c) {
      const int64_t o = (int64_t)i * d + c;
      dx[o] += rho[i] * (dz[o] * g[c] - xhat[o] * mean);
      dg[c] += dz[o] * xhat[o];
    }
  }
}

// dW[out, in] += dy[n, out]^T x[n, in]
void linear_dw(int n, int in, int out, const double* dy, const double* x, double* dW) {
  for (int o = 0; o < out; ++o)
    for (int j = 0; j < in; ++j) {
      double acc = 0.0;
      for (int i = 0; i < n; ++i) acc += dy[(int64_t)i * out + o] * x[(int64_t)i * in + j];
      dW[(int64_t)o * in + j] += acc;
    }
}

// dx[n, in] += dy[n, out] W[out, in]
void linear_dx(int n, int in, int out, const double* dy, const double* W, double* dx) {
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < in; ++j) {
      double acc = 0.0;
      for (int o = 0; o < out; ++o) acc += dy[(int64_t)i * out + o] * W[(int64_t)o * in + j];
      dx[(int64_t)i * in + j] += acc;
    }
}

// Backward of the QK-norm and rotation of oracle_qk_transform (z = R(p) (v rho g) per
// head vector v of hd, rho = (mean(v^2) + eps)^(-1/2), R(p) rotating the pairs
// (c, c + hd/2) by the angle p * theta^(-2c/hd)): dz [rows, heads * hd] becomes dv in
// place (R is orthogonal: its transpose rotates back); the gain gradient is added to
// dgain [hd].
void qk_bwd(int rows, int heads, int hd, const double* pre, const double* gain, double eps,
            double theta, const int32_t* pos, double* dz, double* dgain) {
  const int half = hd / 2;
  for (int i = 0; i < rows; ++i) {
    const double p = pos ? (double)pos[i] : (double)i;
    for (int h = 0; h < heads; ++h) {
      const double* v = pre + ((int64_t)i * heads + h) * hd;
      double* g = dz + ((int64_t)i * heads + h) * hd;
      if (theta > 0.0)
        for (int c = 0; c < half; ++c) {
          const double ang = p * std::pow(theta, -2.0 * c / hd);
          const double cs = std::cos(ang), sn = std::sin(ang);
          const double a = g[c], b = g[c + half];
          g[c] = a * cs + b * sn;
          g[c + half] = -a * sn + b * cs;
        }
      if (gain) {
        double ss = 0.0;
        for (int c = 0; c < hd; ++c) ss += v[c] * v[c];
        const double rho = 1.0 / std::sqrt(ss / hd + eps);
        double dot = 0.0;
        for (int c = 0; c < hd; ++c) dot += g[c] * gain[c] * v[c] * rho;
        const double mean = dot / hd;
        for (int c = 0; c < hd; ++c) {
          const double vh = v[c] * rho;
          if (dgain) dgain[c] += g[c] * vh;
          g[c] = rho * (g[c] * gain[c] - vh * mean);
        }
      }
    }
  }
}

// The block's backward for one sequence. Keys and values come from the nkv rows
// xkv [nkv, d]; the nq queries are the rows qrow[i] of xkv (NULL: i, nq == nkv), in
// ascending order, and query i sees the keys j <= qrow[i]. The residual rows of the
// block are xs_i = xkv[qrow[i]], and the gradients reaching its two residuals are da_ext
// and df [nq, d]. Adds to dxkv [nkv, d] and to gw. Row j of xkv sits at original
// position kvpos[j] (NULL: j), which only the rotation sees.
//   sparse layer: xkv = the compact selected rows, qrow = NULL, kvpos = their positions;
//   dense layer:  xkv = the whole sequence, qrow = NULL, kvpos = NULL;
//   Selected-Q / full-KV (X-MoD notes, "mechanism controls"): xkv = the whole sequence,
//                 qrow = the selected positions, kvpos = NULL.
// attn / ffn select the halves (same section: a FullAttn layer is the attention half with
// its residual, a Routed-FFN layer the FFN half on RMSNorm(xs) g2, i.e. a = 0); both: the
// whole block.
void block_bwd(const oracle_dims* dm, int nkv, const double* xkv, const oracle_layer_w* w,
               int nq, const int32_t* qrow, const double* da_ext, const double* df,
               double* dxkv, oracle_layer_grad* gw, const int32_t* kvpos, bool attn = true,
               bool ffn = true) {
  const int d = dm->d, hq = dm->hq, hkv = dm->hkv, hd = dm->hd, F = dm->F;
  const int G = hq / hkv, qw = hq * hd, kw = hkv * hd;
  const double scale = 1.0 / std::sqrt((double)hd);
  std::vector<int32_t> qr(nq), qpos(nq);   // query i: its row of xkv and its position
  for (int i = 0; i < nq; ++i) {
    qr[i] = qrow ? qrow[i] : i;
    qpos[i] = kvpos ? kvpos[qr[i]] : qr[i];
  }
  std::vector<double> xs((int64_t)nq * d);
  for (int i = 0; i < nq; ++i)
    std::memcpy(&xs[(int64_t)i * d], xkv + (int64_t)qr[i] * d, sizeof(double) * d);
  // ---- forward, keeping what the backward reads
  std::vector<double> u((int64_t)nkv * d), x1((int64_t)nkv * d), rho1(nkv), uq((int64_t)nq * d);
  std::vector<double> q((int64_t)nq * qw), k((int64_t)nkv * kw), v((int64_t)nkv * kw);
  std::vector<double> q_pre, k_pre;
  std::vector<double> P, o;
  std::vector<double> a((int64_t)nq * d, 0.0), hh((int64_t)nq * d);
  const bool extras = w->gq || w->gk || w->rope_theta > 0.0;
  if (attn) {
  rms_fwd(nkv, d, xkv, w->g1, dm->eps, u.data(), x1.data(), rho1.data());
  for (int i = 0; i < nq; ++i)
    std::memcpy(&uq[(int64_t)i * d], &u[(int64_t)qr[i] * d], sizeof(double) * d);
  oracle_linear(nq, d, qw, uq.data(), w->wq, q.data());
  oracle_linear(nkv, d, kw, u.data(), w->wk, k.data());
  oracle_linear(nkv, d, kw, u.data(), w->wv, v.data());
  // QK-norm and rotation at the original positions, the projections kept for the backward
  if (extras) {
    q_pre = q;
    k_pre = k;
    oracle_qk_transform(nq, hq, hd, q.data(), w->gq, dm->eps, w->rope_theta, qpos.data());
    oracle_qk_transform(nkv, hkv, hd, k.data(), w->gk, dm->eps, w->rope_theta, kvpos);
  }
  // P[h][i][j] over the keys j <= qr[i], and o
  P.assign((int64_t)hq * nq * nkv, 0.0);
  o.assign((int64_t)nq * qw, 0.0);
  for (int h = 0; h < hq; ++h) {
    const int g = h / G;
    for (int i = 0; i < nq; ++i) {
      double* p = &P[((int64_t)h * nq + i) * nkv];
      double m = -INFINITY;
      for (int j = 0; j <= qr[i]; ++j) {
        double acc = 0.0;
        for (int c = 0; c < hd; ++c)
          acc += q[(int64_t)i * qw + h * hd + c] * k[(int64_t)j * kw + g * hd + c];
        p[j] = acc * scale;
        m = std::max(m, p[j]);
      }
      double den = 0.0;
      for (int j = 0; j <= qr[i]; ++j) {
        p[j] = std::exp(p[j] - m);
        den += p[j];
      }
      for (int j = 0; j <= qr[i]; ++j) p[j] /= den;
      for (int c = 0; c < hd; ++c) {
        double acc = 0.0;
        for (int j = 0; j <= qr[i]; ++j) acc += p[j] * v[(int64_t)j * kw + g * hd + c];
        o[(int64_t)i * qw + h * hd + c] = acc;
      }
    }
  }
  oracle_linear(nq, qw, d, o.data(), w->wo, a.data());
  }
  for (int64_t i = 0; i < (int64_t)nq * d; ++i) hh[i] = xs[i] + a[i];
  std::vector<double> dh((int64_t)nq * d, 0.0);
  if (ffn) {
  const int n = nq;
  std::vector<double> v2((int64_t)n * d), x2((int64_t)n * d), rho2(n);
  rms_fwd(n, d, hh.data(), w->g2, dm->eps, v2.data(), x2.data(), rho2.data());
  std::vector<double> Gp((int64_t)n * F), Up((int64_t)n * F), H((int64_t)n * F);
  oracle_linear(n, d, F, v2.data(), w->wg, Gp.data());
  oracle_linear(n, d, F, v2.data(), w->wu, Up.data());
  for (int64_t i = 0; i < (int64_t)n * F; ++i) H[i] = Gp[i] * sigmoid(Gp[i]) * Up[i];

  // ---- FFN: f = H Wd^T, H = silu(G) U
  linear_dw(n, F, d, df, H.data(), gw->wd);
  std::vector<double> dH((int64_t)n * F, 0.0);
  linear_dx(n, F, d, df, w->wd, dH.data());
  std::vector<double> dG((int64_t)n * F), dU((int64_t)n * F);
  for (int64_t i = 0; i < (int64_t)n * F; ++i) {
    const double sg = sigmoid(Gp[i]);
    dU[i] = dH[i] * Gp[i] * sg;
    dG[i] = dH[i] * Up[i] * sg * (1.0 + Gp[i] * (1.0 - sg));
  }
  linear_dw(n, d, F, dG.data(), v2.data(), gw->wg);
  linear_dw(n, d, F, dU.data(), v2.data(), gw->wu);
  std::vector<double> dv2((int64_t)n * d, 0.0);
  linear_dx(n, d, F, dG.data(), w->wg, dv2.data());
  linear_dx(n, d, F, dU.data(), w->wu, dv2.data());
  // ---- v2 = RMSNorm(h) g2, h = xs + a
  rms_bwd(n, d, dv2.data(), w->g2, x2.data(), rho2.data(), dh.data(), gw->g2);
  }
  for (int i = 0; i < nq; ++i)   // h = xs + a: dh reaches the query's own row
    for (int c = 0; c < d; ++c) dxkv[(int64_t)qr[i] * d + c] += dh[(int64_t)i * d + c];
  if (!attn) return;
  std::vector<double> da((int64_t)nq * d);
  for (int64_t i = 0; i < (int64_t)nq * d; ++i) da[i] = dh[i] + da_ext[i];
  // ---- a = o Wo^T
  linear_dw(nq, qw, d, da.data(), o.data(), gw->wo);
  std::vector<double> dO((int64_t)nq * qw, 0.0);
  linear_dx(nq, qw, d, da.data(), w->wo, dO.data());
  // ---- attention
  std::vector<double> dq((int64_t)nq * qw, 0.0), dk((int64_t)nkv * kw, 0.0),
      dv((int64_t)nkv * kw, 0.0);
  for (int h = 0; h < hq; ++h) {
    const int g = h / G;
    for (int i = 0; i < nq; ++i) {
      const double* p = &P[((int64_t)h * nq + i) * nkv];
      std::vector<double> dP(qr[i] + 1);
      double Di = 0.0;
      for (int j = 0; j <= qr[i]; ++j) {
        double acc = 0.0;
        for (int c = 0; c < hd; ++c)
          acc += dO[(int64_t)i * qw + h * hd + c] * v[(int64_t)j * kw + g * hd + c];
        dP[j] = acc;
        Di += p[j] * acc;
      }
      for (int j = 0; j <= qr[i]; ++j) {
        const double dS = p[j] * (dP[j] - Di);
        for (int c = 0; c < hd; ++c) {
          dv[(int64_t)j * kw + g * hd + c] += p[j] * dO[(int64_t)i * qw + h * hd + c];
          dq[(int64_t)i * qw + h * hd + c] += scale * dS * k[(int64_t)j * kw + g * hd + c];
          dk[(int64_t)j * kw + g * hd + c] += scale * dS * q[(int64_t)i * qw + h * hd + c];
        }
      }
    }
  }
  if (extras) {   // back through the rotation and the QK-norm
    qk_bwd(nq, hq, hd, q_pre.data(), w->gq, dm->eps, w->rope_theta, qpos.data(), dq.data(), gw->gq);
    qk_bwd(nkv, hkv, hd, k_pre.data(), w->gk, dm->eps, w->rope_theta, kvpos, dk.data(), gw->gk);
  }
  // ---- q = u_q Wq^T (the queries' rows of u), k, v = u [Wk | Wv]^T (every row)
  linear_dw(nq, d, qw, dq.data(), uq.data(), gw->wq);
  linear_dw(nkv, d, kw, dk.data(), u.data(), gw->wk);
  linear_dw(nkv, d, kw, dv.data(), u.data(), gw->wv);
  std::vector<double> du((int64_t)nkv * d, 0.0), duq((int64_t)nq * d, 0.0);
  linear_dx(nq, d, qw, dq.data(), w->wq, duq.data());
  for (int i = 0; i < nq; ++i)
    for (int c = 0; c < d; ++c) du[(int64_t)qr[i] * d + c] += duq[(int64_t)i * d + c];
  linear_dx(nkv, d, kw, dk.data(), w->wk, du.data());
  linear_dx(nkv, d, kw, dv.data(), w->wv, du.data());
  // ---- u = RMSNorm(xkv) g1
  rms_bwd(nkv, d, du.data(), w->g1, x1.data(), rho1.data(), dxkv, gw->g1);
}

// a and f of the block on compact rows xs [n, d] (all rows), for the gate derivatives.
void block_af(const oracle_dims* dm, int n, const double* xs, const oracle_layer_w* w,
              double* a_out, double* f_out, const int32_t* pos);

}  // namespace

extern "C" {

void oracle_block_rows_pos(const oracle_dims* dm, int n, const double* xs,
                           const oracle_layer_w* w, const int32_t* rows, int nrows,
                           double* a_out, double* f_out, const int32_t* pos);

// Backward of one layer (any kind: DENSE, SPARSE, the FullAttn / Routed-FFN halves ATTN
// and RFFN, the Selected-Q / full-KV FULLKV; Eq. 7 or Eq. 6 gating), see the file comment.
// x_in, dy, dx [B, T, d]; bias [B, T] or NULL; idx_force [B, n] or NULL (the
// oracle's own top-(T/K) then); idx_out [B, n] or NULL receives the selection used.
// route_loss (sparse only, NULL allowed) receives L_route of Eq. 9.
int oracle_layer_bwd(const oracle_dims* dm, int kind, int K, int gate, const oracle_layer_w* w,
                     const double* x_in, const double* bias, const int32_t* idx_force,
                     const double* dy, double route_coef, double* dx, oracle_layer_grad* gw,
                     int32_t* idx_out, double* route_loss) {
  const int B = dm->B, T = dm->T, d = dm->d, F = dm->F;
  const int qw = dm->hq * dm->hd, kw = dm->hkv * dm->hd;
  if (B <= 0 || T <= 0 || d <= 0 || dm->hq % dm->hkv) return BAD_ARG;
  if (kind < DENSE || kind > FULLKV) return BAD_ARG;
  if ((w->gq && !gw->gq) || (w->gk && !gw->gk)) return BAD_ARG;
  const int64_t BT = (int64_t)B * T;
  std::memset(gw->w_r, 0, sizeof(double) * d);
  std::memset(gw->g1, 0, sizeof(double) * d);
  std::memset(gw->g2, 0, sizeof(double) * d);
  std::memset(gw->wq, 0, sizeof(double) * (int64_t)qw * d);
  std::memset(gw->wk, 0, sizeof(double) * (int64_t)kw * d);
  std::memset(gw->wv, 0, sizeof(double) * (int64_t)kw * d);
  std::memset(gw->wo, 0, sizeof(double) * (int64_t)d * qw);
  std::memset(gw->wg, 0, sizeof(double) * (int64_t)F * d);
  std::memset(gw->wu, 0, sizeof(double) * (int64_t)F * d);
  std::memset(gw->wd, 0, sizeof(double) * (int64_t)d * F);
  gw->varsigma = 0.0;
  if (gw->gq) std::memset(gw->gq, 0, sizeof(double) * dm->hd);
  if (gw->gk) std::memset(gw->gk, 0, sizeof(double) * dm->hd);
  if (route_loss) *route_loss = 0.0;
  // the skip path: y = x + (residual) for every token
  std::memcpy(dx, dy, sizeof(double) * BT * d);

  if (kind == DENSE || kind == ATTN) {   // y = x + a + f (or x + a) on every token
    for (int b = 0; b < B; ++b) {
      const double* xb = x_in + (int64_t)b * T * d;
      const double* gb = dy + (int64_t)b * T * d;
      block_bwd(dm, T, xb, w, T, nullptr, gb, gb, dx + (int64_t)b * T * d, gw, nullptr, true,
                kind == DENSE);
    }
    return OK;
  }

  if (K <= 0 || T / K <= 0) return BAD_ARG;
  const int n = T / K;
  std::vector<double> s(BT), r(BT);
  oracle_router(BT, d, x_in, w->w_r, bias, s.data(), r.data());
  std::vector<int32_t> idx((int64_t)B * n);
  if (idx_force) {
    for (int64_t i = 0; i < (int64_t)B * n; ++i) idx[i] = idx_force[i];
  } else {
    const int st = oracle_topk(B, T, n, s.data(), idx.data());
    if (st != OK) return st;
  }
  if (idx_out) std::memcpy(idx_out, idx.data(), sizeof(int32_t) * B * n);
  std::vector<double> ds(BT, 0.0);
  // Eq. 9 on every token, q_i from the selection
  if (route_coef != 0.0 || route_loss) {
    std::vector<char> sel(BT, 0);
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < n; ++j) sel[(int64_t)b * T + idx[(int64_t)b * n + j]] = 1;
    double L = 0.0;
    for (int64_t i = 0; i < BT; ++i) {
      const double p = r[i];
      L -= sel[i] ? std::log(p) : std::log(1.0 - p);
      ds[i] += route_coef * (p - (sel[i] ? 1.0 : 0.0)) / (double)BT;
    }
    if (route_loss) *route_loss = L / (double)BT;
  }
  for (int b = 0; b < B; ++b) {
    const int32_t* ib = &idx[(int64_t)b * n];
    std::vector<double> xs((int64_t)n * d), a((int64_t)n * d), f((int64_t)n * d);
    for (int j = 0; j < n; ++j)
      std::memcpy(&xs[(int64_t)j * d], x_in + ((int64_t)b * T + ib[j]) * d, sizeof(double) * d);
    if (kind == RFFN)   // FFN half only: f = FFN(RMSNorm(xs) g2), a = 0
      oracle_ffn_rows(dm, n, xs.data(), w, f.data());
    else if (kind == FULLKV)
      oracle_block_fullkv(dm, T, x_in + (int64_t)b * T * d, w, ib, n, a.data(), f.data());
    else
      block_af(dm, n, xs.data(), w, a.data(), f.data(), ib);
    std::vector<double> da_ext((int64_t)n * d), df((int64_t)n * d), dxs((int64_t)n * d, 0.0);
    for (int j = 0; j < n; ++j) {
      const int64_t t = (int64_t)b * T + ib[j];
      const double* g = dy + t * d;
      const double rt = r[t];
      double dr = 0.0;
      for (int c = 0; c < d; ++c) {
        const int64_t o = (int64_t)j * d + c;
        if (gate == GATE_XMOD) {   // y = x + varsigma r (a + f)
          da_ext[o] = df[o] = w->varsigma * rt * g[c];
          dr += w->varsigma * g[c] * (a[o] + f[o]);
          gw->varsigma += rt * g[c] * (a[o] + f[o]);
        } else {                   // y = x + a + r f
          da_ext[o] = g[c];
          df[o] = rt * g[c];
          dr += g[c] * f[o];
        }
      }
      ds[t] += dr * rt * (1.0 - rt);
    }
    if (kind == FULLKV) {   // keys and values from every token: straight into the sequence's dx
      block_bwd(dm, T, x_in + (int64_t)b * T * d, w, n, ib, da_ext.data(), df.data(),
                dx + (int64_t)b * T * d, gw, nullptr);
      continue;
    }
    block_bwd(dm, n, xs.data(), w, n, nullptr, da_ext.data(), df.data(), dxs.data(), gw, ib,
              kind != RFFN, true);
    for (int j = 0; j < n; ++j)   // the gather's backward: back to the token's row
      for (int c = 0; c < d; ++c) dx[((int64_t)b * T + ib[j]) * d + c] += dxs[(int64_t)j * d + c];
  }
  // s = w_r . x + b
  for (int64_t i = 0; i < BT; ++i) {
    if (ds[i] == 0.0) continue;
    for (int c = 0; c < d; ++c) {
      dx[i * d + c] += ds[i] * w->w_r[c];
      gw->w_r[c] += ds[i] * x_in[i * d + c];
    }
  }
  return OK;
}

}  // extern "C"

namespace {
void block_af(const oracle_dims* dm, int n, const double* xs, const oracle_layer_w* w,
              double* a_out, double* f_out, const int32_t* pos) {
  oracle_block_rows_pos(dm, n, xs, w, nullptr, n, a_out, f_out, pos);
}
}  // namespace
