/*
 * xmod.h -- C ABI of the X-MoD / MoD sparse-depth layer stack on one GPU (forward, and
 * the backward of dense and sparse layers for training).
 *
 * The method (page "X-MoD: Practical Scaling Laws for Sparse-Depth Routing Beyond
 * Mixture-of-Depths", reading notes): every sparse layer scores each token with a
 * router (Eq. 8), keeps the top 1/K tokens of every sequence (section "MoD
 * structural limit", Eq. 1), runs the transformer block on those tokens only --
 * attention among the selected tokens (section "mechanism controls") -- and writes
 * them back with the gated residual of Eq. 7 (X-MoD) or Eq. 6 (MoD). Unselected
 * tokens pass through unchanged. Layers follow Eq. 3:
 * [Dense] x N0 + ([Sparse(K)] x AK + [Dense]) x N1.
 * The page "Mixture-of-Depths explained" (its MoDLayer listing) fixes the
 * position-ordered gather and the floor(T / K) selection count.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers, owned by the caller. The library
 *     never allocates, frees or synchronises (except xmod_sync_status).
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).
 *   - Residual-stream tensors and weights are in dims->dtype (bf16 or fp32),
 *     row-major. Router logits, gates and biases are always fp32; indices int32.
 *   - Matrices use the [out, in] row-major layout: wq [hq*hd, d], wk and wv
 *     [hkv*hd, d], wo [d, hq*hd], w_gate and w_up [F, d], w_down [d, F];
 *     w_router, rms1, rms2 are [d].
 *   - Host-detected errors return a negative xmod_status before anything is
 *     launched. Errors found on the device (a non-finite router logit, a bounded
 *     wait that ran out) are recorded in the workspace status word and returned
 *     by xmod_sync_status; kernels never trap.
 *   - Pointers must be 16-byte aligned; d, hq*hd, hkv*hd and F must be
 *     multiples of 8.
 *   - Which kernels run. bf16: every projection on the tcgen05 tensor cores (bf16
 *     operands, fp32 accumulation); the attention on the tcgen05 attention kernel when
 *     head_dim is 128, and on an FFMA kernel (bf16 operands, fp32 accumulation, much
 *     slower) for any other head_dim. fp32: FFMA kernels throughout (no TF32). The
 *     routing, gather and scatter kernels are the same in both. There is no other
 *     fallback: a bf16 call on a system without the TMA tensor-map entry point returns
 *     XMOD_ERR_UNSUPPORTED instead of running its projections on FFMA kernels.
 *   - Entry points are stateless and may run concurrently on different streams
 *     with different workspaces. They are capture-safe: a call recorded into a CUDA
 *     graph and replayed computes the same results as the eager call.
 *   - Tuning overrides, read from the environment at every launch (the defaults are
 *     the measured choices; the results are the same bit for bit except under
 *     stream-K, which changes the order of fp32 additions, and the fused gather, which
 *     scales the GEMM's output rows by 1 / rms instead of rounding normalised rows to
 *     bf16 first): XMOD_PAIR_MIN_WAVES (waves of 256 x 256 tiles
 *     from which GEMMs always run on CTA pairs; 0 puts every eligible GEMM on
 *     pairs), XMOD_PAIR_BN (256 or 192: the only CTA-pair tile width tried),
 *     XMOD_STREAM_K=1 (stream-K single-CTA GEMMs where they apply) and
 *     XMOD_STREAM_K_CTAS (their grid cap), XMOD_EPI_STAGE=0 (the pair GEMMs' epilogue
 *     inputs read from global memory instead of staged in shared memory),
 *     XMOD_GATHER_FUSED=1 (a sparse layer's gather + RMSNorm1 folded into the q|k|v
 *     GEMM's operand load).
 */
#ifndef XMOD_H
#define XMOD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define XMOD_API __attribute__((visibility("default")))
#else
#define XMOD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  XMOD_OK = 0,
  XMOD_ERR_INVALID_ARG = -1,   /* bad pointer, size or combination; nothing launched */
  XMOD_ERR_UNSUPPORTED = -2,   /* valid but not implemented (e.g. T beyond the top-k limit) */
  XMOD_ERR_CUDA = -3,          /* a CUDA runtime call failed */
  XMOD_ERR_TIMEOUT = -4,       /* a bounded device-side wait ran out (device status) */
  XMOD_ERR_DEVICE_CHECK = -5,  /* non-finite router logit or bad index seen on device */
  XMOD_ERR_WORKSPACE = -6      /* workspace missing or smaller than xmod_workspace_bytes */
} xmod_status;

typedef enum { XMOD_BF16 = 0, XMOD_FP32 = 1 } xmod_dtype;

/* Residual gate: Eq. 7 (X-MoD) x + varsigma * r * (a + f); Eq. 6 (MoD) x + a + r * f. */
typedef enum { XMOD_GATE_XMOD = 0, XMOD_GATE_MOD = 1 } xmod_gate;

/* Layer kinds. DENSE: the block on every token. SPARSE: the block on the routed tokens.
 * ATTN and ROUTED_FFN are the two halves of the Routed-FFN variant of X-MoD notes
 * "mechanism controls" (Table 2, Table 7; ([FullAttn] + [Routed-FFN] x K) x A between
 * dense anchors): ATTN is the attention half on every token, x += a (weights used:
 * rms1, wq, wk, wv, wo); ROUTED_FFN routes top-(T/K) tokens through the FFN half only,
 * f = FFN(RMSNorm(x) * rms2), with the gated residual taken with a = 0 (Eq. 7:
 * x + varsigma r f; Eq. 6: x + r f) (weights used: w_router, rms2, w_gate, w_up,
 * w_down, varsigma). Weights a kind does not use may be NULL.
 * SPARSE_FULLKV is the Selected-Q / full-KV control of the same section: routed like
 * SPARSE, but every token of the sequence provides keys and values (RMSNorm(x) * rms1
 * of all T tokens through wk, wv) and a selected token attends to every token at or
 * before its own position; the rest of the block and the residual are SPARSE's. */
typedef enum {
  XMOD_LAYER_DENSE = 0,
  XMOD_LAYER_SPARSE = 1,
  XMOD_LAYER_ATTN = 2,
  XMOD_LAYER_ROUTED_FFN = 3,
  XMOD_LAYER_SPARSE_FULLKV = 4
} xmod_layer_kind;

/* Problem sizes in the pages' notation: B sequences of T tokens, model width d,
 * n_heads query heads and n_kv_heads key/value heads of head_dim (GQA), SwiGLU
 * hidden width d_ff. rms_eps is the RMSNorm epsilon. */
typedef struct {
  int B, T, d, n_heads, n_kv_heads, head_dim, d_ff;
  xmod_dtype dtype;
  float rms_eps;
} xmod_dims;

/* One layer's weights (device pointers, dims->dtype). w_router is used by sparse
 * layers only; varsigma is the per-layer scalar of Eq. 7.
 * Optional Qwen3-style attention extras (the X-MoD notes name Qwen3 backbones; the
 * NEXT item "RoPE at original positions, QK-norm"), all off when zero / NULL:
 *   q_norm, k_norm  [head_dim] QK-norm gains: every head's q (k) vector is
 *                   RMS-normalised (rms_eps) and scaled by them after the projection;
 *   rope_theta      rotary embedding base: after QK-norm, q and k are rotated at the
 *                   token's ORIGINAL position t in its sequence (not its compact index),
 *                   pairing dimension c with c + head_dim/2 at angle
 *                   t * rope_theta^(-2c/head_dim). */
typedef struct {
  const void *w_router, *rms1, *wq, *wk, *wv, *wo, *rms2, *w_gate, *w_up, *w_down;
  float varsigma;
  const void *q_norm, *k_norm;
  float rope_theta;
} xmod_layer_weights;

/* Library version string. */
XMOD_API const char* xmod_version(void);

/* Human-readable name of an xmod_status value. */
XMOD_API const char* xmod_status_string(int status);

/* Bytes of device workspace the calls below need for these sizes and sparsity K
 * (K = 1 sizes a dense layer; the stack needs the size for its own K, which
 * covers its dense layers). Returns 0 for invalid dims. The workspace is
 * caller-owned scratch; its first 256 bytes hold the device status word. */
XMOD_API size_t xmod_workspace_bytes(const xmod_dims* dims, int K);

/* Clear the device status word of a workspace (asynchronous). */
XMOD_API int xmod_reset_status(void* ws, size_t ws_bytes, void* stream);

/* Synchronise `stream` and return the device status word of the workspace
 * (XMOD_OK or the first device-side error recorded since the last reset), or
 * XMOD_ERR_CUDA if synchronisation itself failed. */
XMOD_API int xmod_sync_status(void* ws, void* stream);

/* Router and per-sequence top-(T/K) selection (X-MoD notes Eq. 8; MoD blog listing).
 *   x        [B, T, d]   residual stream (dtype)
 *   w_r      [d]         router vector (dtype)
 *   bias     [B, T] fp32 signed per-token bias added to the logit, or NULL
 *   logits   [B, T] fp32 out: s = w_r . x + bias (NULL: kept in the workspace)
 *   r        [B, T] fp32 out: sigmoid(s) (NULL: not written)
 *   idx      [B, n] int32 out: the n = floor(T/K) positions with the largest s,
 *                    ties to the lower position, ascending
 *   r_sel    [B, n] fp32 out: sigmoid(s) at idx (NULL: not written)
 * A non-finite logit records XMOD_ERR_DEVICE_CHECK in the status word. */
XMOD_API int xmod_router_topk(const xmod_dims* dims, int K, const void* x, const void* w_r,
                     const float* bias, float* logits, float* r, int32_t* idx, float* r_sel,
                     void* ws, size_t ws_bytes, void* stream);

/* Top-(T/K) selection on given fp32 logits [B, T] (same rule and outputs as
 * xmod_router_topk; r_sel may be NULL). */
XMOD_API int xmod_topk(const xmod_dims* dims, int K, const float* logits, int32_t* idx, float* r_sel,
              void* ws, size_t ws_bytes, void* stream);

/* Position-ordered gather: xs[b*n + j, :] = x[b, idx[b, j], :], n = floor(T/K).
 * The positions are checked on the device: a row whose position is outside [0, T) or
 * not above the previous row's in its sequence is skipped (its xs row is not written)
 * and, when status_out (a device int, or NULL) is given, XMOD_ERR_DEVICE_CHECK is
 * stored there if it still holds 0 (the caller zeroes it; the first error stays). */
XMOD_API int xmod_gather(const xmod_dims* dims, int K, const void* x, const int32_t* idx, void* xs,
                int* status_out, void* stream);

/* The transformer block on n_per_seq tokens of every sequence (X-MoD notes,
 * backbone configuration: GQA attention, SwiGLU FFN; pre-norm RMSNorm):
 *   u = RMSNorm(xs) * rms1; q, k, v = u Wq^T, u Wk^T, u Wv^T
 *   o = causal GQA softmax attention among the n_per_seq tokens of a sequence,
 *       scale 1/sqrt(head_dim), query head h reads KV head h / (n_heads/n_kv_heads)
 *   a = o Wo^T; h = xs + a; f = (silu(v2 Wg^T) * (v2 Wu^T)) Wd^T, v2 = RMSNorm(h) * rms2
 * With idx == NULL, `xs` is the compact buffer [B * n_per_seq, d]; otherwise `xs`
 * is the full stream x [B, T, d] and row j of sequence b is x[b, idx[b, j]]; the
 * positions are checked on the device first (in [0, T), ascending within a sequence):
 * a bad row records XMOD_ERR_DEVICE_CHECK in the status word and is read at its
 * position clamped into [0, T), so nothing outside the stream is touched (its a_out,
 * f_out rows and those of the rows attending to it are then meaningless).
 * a_out, f_out: [B * n_per_seq, d] (dtype). Workspace: xmod_workspace_bytes with
 * K = T / n_per_seq rounded down. */
XMOD_API int xmod_block_fwd(const xmod_dims* dims, int n_per_seq, const void* xs, const int32_t* idx,
                   const xmod_layer_weights* w, void* a_out, void* f_out, void* ws,
                   size_t ws_bytes, void* stream);

/* Gated scatter back into the stream, in place (X-MoD notes Eq. 6 / Eq. 7):
 *   gate XMOD: x[b, idx[b,j]] += varsigma * r_sel[b,j] * (a + f)
 *   gate MOD:  x[b, idx[b,j]] += a + r_sel[b,j] * f
 * a, f: [B * n, d] (dtype). f may be NULL under XMOD, in which case `a` holds a + f.
 * Rows not in idx are not touched. The positions are checked as for xmod_gather: a
 * bad row is skipped (no stream row is written for it) and reported through
 * status_out (a device int, or NULL) as XMOD_ERR_DEVICE_CHECK. */
XMOD_API int xmod_gated_scatter(const xmod_dims* dims, int K, void* x_inout, const int32_t* idx,
                       const float* r_sel, const void* a, const void* f, float varsigma,
                       xmod_gate gate, int* status_out, void* stream);

/* One layer in place on x [B, T, d]. Sparse: router + top-(T/K) + block on the
 * selected tokens + gated residual; unselected rows untouched. Dense: the block on
 * all tokens and x += a + f. bias: [B, T] fp32 or NULL. idx_out ([B, n] int32) and
 * r_sel_out ([B, n] fp32) optionally receive the sparse layer's selection. */
XMOD_API int xmod_layer_fwd(const xmod_dims* dims, xmod_layer_kind kind, int K, xmod_gate gate,
                   const xmod_layer_weights* w, void* x_inout, const float* bias,
                   int32_t* idx_out, float* r_sel_out, void* ws, size_t ws_bytes, void* stream);

/* The Eq. 3 stack in place: [Dense] x N0 + ([Sparse(K)] x AK + [Dense]) x N1 with
 * AK = round(A * K) (must equal A * K and be >= 1). `layers` holds n_layers =
 * N0 + N1 * (AK + 1) weight sets in execution order. Every sparse layer uses the
 * same bias (NULL: none). MoD's Eq. 1 stack is N0 = 0, A = 1/K. */
XMOD_API int xmod_stack_fwd(const xmod_dims* dims, int K, double A, int N0, int N1, xmod_gate gate,
                   const xmod_layer_weights* layers, int n_layers, void* x_inout,
                   const float* bias, void* ws, size_t ws_bytes, void* stream);

/* Token selection rule of a sparse layer. TOPK: the top-(T/K) of each sequence
 * (training rule). THRESHOLD: the causal rule of X-MoD notes "top-k in training,
 * causal threshold at evaluation" -- every token whose routing probability
 * r = sigmoid(s) is at least 1/2 (s >= 0; -0 counts as 0) enters the layer, each token
 * deciding alone, so a sequence takes a variable number of tokens (possibly none);
 * the selected tokens attend causally among themselves in position order and get the
 * gated residual with their own r. THRESHOLD needs bf16 and head_dim 128 (the
 * tensor-core path; otherwise XMOD_ERR_UNSUPPORTED). */
typedef enum { XMOD_ROUTE_TOPK = 0, XMOD_ROUTE_THRESHOLD = 1 } xmod_routing;

/* One sparse layer under the causal threshold rule (see xmod_routing), in place on
 * x [B, T, d] (bf16). bias: [B, T] fp32 or NULL, added to the logit. count_out: NULL
 * or device int32 [B], the number of tokens each sequence routed through the layer.
 * Workspace: xmod_workspace_bytes(dims, any K). */
XMOD_API int xmod_layer_fwd_threshold(const xmod_dims* dims, xmod_gate gate,
                                      const xmod_layer_weights* w, void* x_inout,
                                      const float* bias, int32_t* count_out, void* ws,
                                      size_t ws_bytes, void* stream);

/* Options of xmod_stack_fwd_ex.
 *
 * bias_step: the token-choice bias dynamics of X-MoD notes Eq. 8 and the paragraph
 *   after it -- inside a sparse-dense block a token's bias grows each time it is
 *   selected and is cleared at the next dense anchor. The pages publish neither the
 *   increment nor tau; here a sparse layer ranks and gates with
 *     s_i = w_r . x_i + bias_i - bias_step * c_i,
 *   c_i = how many earlier sparse layers of the block selected token i. 0 gives the
 *   constant-bias stack of xmod_stack_fwd; must be finite and >= 0.
 * layer_stats: NULL or device int32 [n_sparse, B, 4], per routed layer (SPARSE or
 *   ROUTED_FFN, stack order) and sequence: tokens selected (T / K); tokens whose ranked logit is >= 0 (the
 *   causal threshold rule r >= 1/2 of X-MoD notes "top-k in training, causal threshold
 *   at evaluation"); tokens on which the two rules agree (both select or both skip);
 *   selected tokens that the previous sparse layer of the block also selected.
 * update_hist: NULL or device int32 [N1, B, AK + 1]: for each sparse-dense block (the
 *   routed layers between two dense layers) and sequence, how many tokens the block's
 *   AK routed layers updated 0, 1, ..., AK times.
 * These are the inputs of the routing diagnostics of X-MoD notes Table 10 (coverage,
 * adjacent-layer Jaccard overlap, threshold / top-k mask agreement, update counts).
 * Under THRESHOLD routing the selected count is the threshold count and every
 * decision agrees; update_hist then needs no K (the selections vary).
 * routing: xmod_routing of every sparse layer (K still fixes the Eq. 3 schedule). */
typedef struct {
  float bias_step;
  int32_t* layer_stats;
  int32_t* update_hist;
  int routing;
} xmod_stack_opts;

/* xmod_stack_fwd with options (opts NULL: exactly xmod_stack_fwd). The workspace
 * size is the same (xmod_workspace_bytes). Invalid options: XMOD_ERR_INVALID_ARG. */
XMOD_API int xmod_stack_fwd_ex(const xmod_dims* dims, int K, double A, int N0, int N1,
                               xmod_gate gate, const xmod_layer_weights* layers, int n_layers,
                               void* x_inout, const float* bias, const xmod_stack_opts* opts,
                               void* ws, size_t ws_bytes, void* stream);

/* A stack in an explicit layer order: kinds (host array of n_layers values,
 * an xmod_layer_kind) and `layers` in execution order. This is
 * how the heterogeneous segment stacks of X-MoD notes Eq. 35 and Eq. 36 (a shorter
 * first sparse segment, then A4K8 / A3K16 segments), MoD's Eq. 34 and the Routed-FFN
 * control (([ATTN] + [ROUTED_FFN] x K) x A between dense anchors) run. A block is the
 * set of routed layers between two dense layers; each routed layer selects T / K
 * tokens (or follows opts->routing; THRESHOLD with ROUTED_FFN is unsupported). With opts->update_hist the histogram has one
 * [B, L_max + 1] slab per block, L_max the longest block; layer_stats is as for
 * xmod_stack_fwd_ex. opts may be NULL. */
XMOD_API int xmod_stack_fwd_sched(const xmod_dims* dims, int K, const int32_t* kinds,
                                  int n_layers, xmod_gate gate, const xmod_layer_weights* layers,
                                  void* x_inout, const float* bias, const xmod_stack_opts* opts,
                                  void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- backward of one layer
 * The gradient of one layer (Eq. 7 or Eq. 6 gating) for training: for
 * the layer y = layer(x) of xmod_layer_fwd and a caller-given upstream gradient dy,
 * the call returns the gradients of the scalar
 *     J = sum(dy * y) + route_coef * L_route
 * with respect to x and to every weight of the layer. L_route is the binary
 * cross-entropy of X-MoD notes Eq. 9 (section "top-k in training, causal threshold at
 * evaluation"), which aligns the router with the deployable threshold rule:
 *     L_route = -(1/N) sum_i [q_i log p_i + (1 - q_i) log(1 - p_i)],
 * q_i = 1 for the layer's top-(T/K) tokens, p_i = sigmoid(s_i) on the same biased logit
 * the selection ranks, N = B*T (every token of the layer's input). The pages sweep the
 * coefficient over 1e-2 .. 1e-5 and keep 1e-4; route_coef = 0 leaves Eq. 9 out. The
 * top-(T/K) selection is piecewise constant and is held fixed: the router learns
 * through the gate r of the residual and through Eq. 9.
 *
 * The call recomputes the layer's forward from x (routing included) and then runs
 * the backward; it does not modify x.
 *   x, dy     [B, T, d]  the layer's input and the gradient at its output (dtype)
 *   bias      [B, T] fp32 as for xmod_layer_fwd, or NULL
 *   dx        [B, T, d]  out (dtype): dJ/dx; may not alias x or dy
 *   grads     fp32 device arrays shaped as the weights (overwritten); w_router is
 *             ignored for DENSE layers; varsigma (one float) receives dJ/dvarsigma (0
 *             under Eq. 6 and for DENSE); route_loss (one float, NULL allowed)
 *             receives L_route (the routed kinds; 0 for DENSE and ATTN)
 *   ws        at least xmod_bwd_workspace_bytes(dims, K) bytes
 * With the QK-norm / rotary extras the gradient also flows back through them (the
 * rotation at the tokens' original positions, as in the forward) and q_norm / k_norm
 * receive the gains' gradients. The mechanism controls' halves are differentiated too:
 * ATTN (y = x + a on every token) and ROUTED_FFN (the FFN half on the top-(T/K) tokens
 * with a = 0 in the gated residual); the gradients of the weights a kind does not use
 * may be NULL and are zeroed when given. SPARSE_FULLKV (the Selected-Q / full-KV
 * control) sends the gradient through every token's key and value as well: rows the
 * layer did not select receive more than dy when a selected query sees them. Its
 * attention backward runs on the tcgen05 kernels in bf16 with head_dim 128 (query
 * positions over a separate key set), on warp-level MMA kernels in bf16 with head_dim
 * 64 and on FFMA kernels in fp32. An unknown kind returns XMOD_ERR_INVALID_ARG.
 * bf16 runs the projections and their gradients on the tensor cores (bf16 operands,
 * fp32 accumulation, fp32 weight gradients); fp32 runs FFMA kernels throughout. */
typedef struct {
  float *w_router, *rms1, *wq, *wk, *wv, *wo, *rms2, *w_gate, *w_up, *w_down;
  float* varsigma;
  float* route_loss;
  float *q_norm, *k_norm;   /* [head_dim] each; required when the layer has that gain */
} xmod_layer_grads;

XMOD_API size_t xmod_bwd_workspace_bytes(const xmod_dims* dims, int K);

XMOD_API int xmod_layer_bwd(const xmod_dims* dims, xmod_layer_kind kind, int K, xmod_gate gate,
                            const xmod_layer_weights* w, const void* x, const float* bias,
                            const void* dy, float route_coef, void* dx,
                            const xmod_layer_grads* grads, void* ws, size_t ws_bytes,
                            void* stream);

/* Backward of the Eq. 3 stack, for training: every layer's input is recomputed with
 * xmod_layer_fwd (the layer-by-layer forward, equal bit for bit to xmod_stack_fwd) into
 * `checkpoints` ([n_layers, B, T, d], dtype; checkpoint l = the input of layer l), then
 * xmod_layer_bwd runs from the last layer to the first, each layer's dx becoming the dy
 * of the layer before it.
 *   x, bias, K, A, N0, N1, gate, layers, n_layers: as for xmod_stack_fwd (x is not
 *             modified; every sparse layer uses the same bias)
 *   dy        [B, T, d]  the gradient at the stack's output (dtype)
 *   route_coef the Eq. 9 coefficient of every sparse layer
 *   dx        [B, T, d]  out: the gradient at the stack's input; may not alias x, dy or
 *             the checkpoints
 *   grads     host array of n_layers xmod_layer_grads, layer order (device arrays,
 *             overwritten; as for xmod_layer_bwd)
 *   ws        at least xmod_stack_bwd_workspace_bytes(dims, K) bytes */
XMOD_API size_t xmod_stack_bwd_workspace_bytes(const xmod_dims* dims, int K);

XMOD_API int xmod_stack_bwd(const xmod_dims* dims, int K, double A, int N0, int N1,
                            xmod_gate gate, const xmod_layer_weights* layers, int n_layers,
                            const void* x, const float* bias, const void* dy, float route_coef,
                            void* dx, const xmod_layer_grads* grads, void* checkpoints,
                            void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- allocation-free routing
 * The paper has no counterpart to this entry point: it exists for callers that
 * cannot allocate device memory -- a plugin inside another runtime that is given
 * only its input and output buffers, a serving loop that must not allocate once
 * running (an allocation can synchronise the device), or a process whose device
 * memory is held by another framework's caching allocator so that cudaMalloc
 * fails. It computes exactly what xmod_router_topk computes (router logits with
 * bias, sigmoid gates at the selected positions, per-sequence top-(T/K) with ties
 * to the lower position) without a caller workspace.
 *
 * Its scratch (fp32 logits and a status word) is a fixed array inside the library
 * image, sized for at most XMOD_NOALLOC_MAX_TOKENS = B*T tokens (8 MiB of logits),
 * which every device that loads the library holds until the process exits. Larger
 * problems are rejected with XMOD_ERR_UNSUPPORTED before anything is launched.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *
 * All calls on a device share that array and it keeps the last call's contents;
 * each call clears the status word first and rewrites every logit it reads, so
 * back-to-back calls on one stream are independent. Calls that overlap on the GPU
 * (different streams with no ordering between them) race on the array.
 * A call looks up the array's device address with its device current whenever its
 * stream is not being captured, and remembers it per device; a call made during
 * stream capture uses the remembered address. So make one call on a device before
 * any capture, and again after a device reset (which moves the array); a captured
 * call on a device never called outside capture returns XMOD_ERR_INVALID_ARG.
 *
 *   x, w_r, bias, idx, r_sel: as for xmod_router_topk (device pointers, bias and
 *   r_sel may be NULL). status_out: NULL or a device int that receives the device
 *   status of this call (XMOD_OK, or XMOD_ERR_DEVICE_CHECK for a non-finite logit),
 *   written asynchronously on `stream`. */
#define XMOD_NOALLOC_MAX_TOKENS (2 * 1024 * 1024)

XMOD_API int xmod_router_topk_noalloc(const xmod_dims* dims, int K, const void* x,
                                      const void* w_r, const float* bias, int32_t* idx,
                                      float* r_sel, int* status_out, void* stream);

/* ---------------------------------------------------------------- failure detection
 * Not part of the method. Every wait inside the library's tcgen05 kernels (on an
 * mbarrier, or on a flag another CTA sets) gives up after 2 s without progress: the
 * waiting thread records XMOD_ERR_TIMEOUT in the status word, the CTA lets its copies in
 * flight land, frees its tensor memory and returns, so the CUDA context stays usable and
 * xmod_sync_status reports the error.
 *
 * Self-test of that path (no fault, no trap): one CTA waits, through the kernels' own
 * bounded wait, on an mbarrier phase that nothing completes, for the 2 s limit, then
 * returns. Afterwards the status word of `ws` (reset it first) holds XMOD_ERR_TIMEOUT,
 * and the ints at ws + 4 and ws + 8 hold the wait's result (0: it gave up) and the
 * CTA's abort flag (1: raised).
 *   ws        device buffer of at least 256 bytes, 16-byte aligned
 * Returns XMOD_OK once launched, XMOD_ERR_INVALID_ARG for a bad buffer. */
XMOD_API int xmod_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- measurement
 * Not part of the method: support for benchmarking the calls above. */

/* Per-kernel-kind timing record filled by xmod_profile_read. */
typedef struct {
  char name[32];     /* kernel kind, e.g. "gemm_gate_up" */
  int launches;      /* launches recorded since the last read */
  double total_ms;   /* summed CUDA-event time of those launches */
} xmod_kernel_time;

/* Host-side count of kernel launches this library has issued so far. */
XMOD_API uint64_t xmod_launch_count(void);

/* Turn per-launch CUDA-event recording on (1) or off (0). While on, every
 * launch is bracketed by two events on its own stream. Process-wide. */
XMOD_API int xmod_profile_enable(int enable);

/* Wait for the recorded events, aggregate them per kernel kind into out[0..max),
 * set *n_kinds, and clear the records. Returns XMOD_ERR_CUDA if an event failed. */
XMOD_API int xmod_profile_read(xmod_kernel_time* out, int max_kinds, int* n_kinds);

#ifdef __cplusplus
}
#endif

#endif /* XMOD_H */
