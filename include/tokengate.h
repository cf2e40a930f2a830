/*
 * tokengate.h -- C ABI of libtokengate.so: the gated-prefill hot path of
 * TokenGate-style learned token pruning, as hand-written CUDA for sm_103a.
 *
 * The method (five web pages about "TokenGate: Adapting LLMs for Fast and
 * Memory-Efficient Prefill with Learned Token Pruning"):
 *   [DE] spke.com, "TokenGate – Token-Gated Attention macht das Vollfüllen
 *        von langen Kontexten bis zu 11,3-mal schneller", sections "Wie hat
 *        TokenGate das Pruning von Tokens verstanden?" (three phases: full
 *        layers below gate layer L, a gate MLP + top-K at L, pruned layers
 *        above; only the document part may be pruned) and "Was ist
 *        token-gated Attention?" (the kept token's score becomes a bias on
 *        the attention logits, with a per-head gain and a temperature).
 *   [TH] ai4bro.com, "Stanford เปิดตัว TokenGate เร่งความเร็ว Prefill ใน LLM
 *        สูงสุด 11.3 เท่า", section "กลไกการทำงานของ Learned Token Pruning".
 *   [IT] ai.info, "TokenGate riporta un prefill fino a 11,3 volte più veloce
 *        sui contesti lunghi", section "TokenGate impara quali token
 *        mantenere" (only the kept rows go to the upper layers).
 * The pages give no formula; this library fixes the logit as
 *   l_ij = t * (q_i . k_j) / sqrt(dh) + g_h * log(sigmoid(s_j)),
 * causal on original positions, with grouped-query attention.
 *
 * Conventions for every call:
 *  - Pointers are DEVICE pointers unless marked "host".  The caller owns all
 *    buffers; the library allocates no device memory on any call.
 *  - Matrices are row-major with densely packed rows.  bf16 buffers hold
 *    IEEE bfloat16; fp32 buffers IEEE binary32.  Every device pointer must
 *    be 16-byte aligned, and every row's byte length a multiple of 16.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and never synchronise, except tg_get_device_status.
 *  - Argument errors (NULL pointers, misalignment, sizes out of range,
 *    unsupported shapes) return before anything is launched.
 *  - Data errors found on the device (a NaN score in the document span, a
 *    kept index outside [0, N), a wait that gave up) set bits in a sticky
 *    per-device status word read by tg_get_device_status.  Kernels never
 *    trap; on such an error their outputs are unspecified.
 *  - Outputs must not overlap inputs unless a call says otherwise.
 */
#ifndef TOKENGATE_H
#define TOKENGATE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t, declared so that C callers need no CUDA
 * headers. */
typedef struct CUstream_st* tg_stream_t;

typedef enum tg_status {
  TG_OK = 0,
  TG_ERR_INVALID_ARG = 1,  /* bad pointer, size, span, alignment           */
  TG_ERR_UNSUPPORTED = 2,  /* valid but not implemented (shape, dtype)     */
  TG_ERR_CUDA = 3,         /* a CUDA runtime call failed                    */
  TG_ERR_NAN_SCORE = 4,    /* device: NaN score inside the document span    */
  TG_ERR_BAD_INDEX = 5,    /* device: a gathered index outside [0, N)       */
  TG_ERR_TIMEOUT = 6       /* device: a pipeline wait gave up (bounded)     */
} tg_status;

typedef enum tg_dtype { TG_F32 = 0, TG_BF16 = 1 } tg_dtype;

/* Human-readable name of a status code.  Never NULL. */
const char* tg_status_string(int status);

/* ABI version of this header (bumped on any signature change). */
#define TG_ABI_VERSION 3
int tg_abi_version(void);

/* Message of the last TG_ERR_INVALID_ARG / TG_ERR_UNSUPPORTED / TG_ERR_CUDA
 * returned on the calling host thread ("" if none).  Host pointer, valid
 * until the next call on this thread. */
const char* tg_last_error_message(void);

/*
 * Gate MLP ([DE] "Wie hat TokenGate das Pruning von Tokens verstanden?",
 * Gate-Modul; [TH] phase 2): one scalar score per token from its residual
 * row at the gate layer,
 *   s_i = sum_k w2[k] * GELU(sum_c W1[k][c] * X[i][c] + b1[k]) + b2,
 * GELU(z) = z * Phi(z) (the exact erf form).
 *
 *  X       [N][d] in `dtype` (TG_BF16: tcgen05 tensor-core path, fp32
 *          accumulation; TG_F32: CUDA-core fp32 path).
 *  W1      [Hg][d] in `dtype` (nn.Linear layout, out x in).
 *  b1      [Hg] fp32, or NULL for zero.
 *  w2      [Hg] fp32.   b2: scalar.
 *  scores  [N] fp32 output.
 *  select_ws, doc_begin, doc_end: optional fusion with the next
 *          tg_select_topk.  When select_ws (a select workspace, see below)
 *          is given on the TG_BF16 path, the epilogue that produces the
 *          scores also counts the first radix pass of the selection (the top
 *          11 bits of each score key in [doc_begin, doc_end)) into it and
 *          stamps it with (N, doc_begin, doc_end); a tg_select_topk on the
 *          same span and workspace then skips that pass.  NULL: no fusion
 *          (doc_begin, doc_end ignored).  TG_F32 ignores the workspace.
 * Limits: N >= 0 (N == 0 launches nothing); d % 64 == 0 for TG_BF16
 * (d % 4 == 0 for TG_F32); 16 <= Hg <= 256 and Hg % 16 == 0 for TG_BF16,
 * 1 <= Hg <= 1024 for TG_F32; with select_ws, 0 <= doc_begin <= doc_end <= N.
 */
tg_status tg_gate_score(const void* X, tg_dtype dtype, int64_t N, int32_t d,
                        const void* W1, const float* b1, int32_t Hg,
                        const float* w2, float b2, float* scores,
                        void* select_ws, int64_t doc_begin, int64_t doc_end,
                        tg_stream_t stream);

/*
 * Bytes of the select workspace (device memory the caller owns, 256-byte
 * aligned, used by tg_select_topk and optionally filled by tg_gate_score):
 * 104 KiB for any N.  It must be zeroed once before its first use
 * (cudaMemset); every tg_select_topk that returns TG_OK and whose kernel
 * finishes without a device error leaves it ready for the next call: its
 * histograms (including one a tg_gate_score put there), header and barrier
 * counter are back at zero (per-CTA counts, a barrier generation word and
 * the candidate keys of long spans carry over and need no reset), so it can
 * be reused call after call on one stream.  A tg_gate_score that filled it must be followed by a
 * tg_select_topk on the same workspace before the next tg_gate_score.
 * After TG_ERR_TIMEOUT, zero it again.  Calls that share a workspace must
 * not overlap on the GPU (use one workspace per stream).
 */
size_t tg_select_workspace_bytes(int64_t N);

/*
 * Top-K select ([DE] same section: after scoring, the gate keeps the K
 * best-scoring tokens, and only document tokens are candidates for removal,
 * never the question; [TH] phases 2-3).
 *
 * Keeps every token outside [doc_begin, doc_end) and the K document tokens
 * that come first in the order (fp32 score bit pattern as a total order
 * descending, -0.0 below +0.0, then lower index first), and writes their
 * indices to kept_idx in ascending order.  The result is unique, so the
 * call is deterministic and bit-exact.
 *
 *  scores     [N] fp32.
 *  kept_idx   [M] int32 output, M = N - (doc_end - doc_begin) + K.
 *  M_out      host pointer (nullable): receives M, computed on the host, so
 *             no device synchronisation is needed to size the next calls.
 *  workspace  device, workspace_bytes >= tg_select_workspace_bytes(N),
 *             256-byte aligned, zeroed before its first use (see above).
 * Limits: 0 <= doc_begin <= doc_end <= N < 2^31, 0 <= K <= doc_end -
 * doc_begin.  M == 0 launches nothing.  A NaN score inside the span sets
 * TG_ERR_NAN_SCORE in the device status word (NaN then ranks above +inf).
 * One launch: a span of at most 4096 keys takes a single CTA (its keys in
 * shared memory, no grid barrier); a longer one takes one CTA per ~2048
 * keys, at most one per SM, and those CTAs meet at grid barriers in the
 * workspace whose waits are bounded (a barrier that never completes sets
 * TG_ERR_TIMEOUT instead of hanging).
 */
tg_status tg_select_topk(const float* scores, int64_t N, int64_t doc_begin,
                         int64_t doc_end, int64_t K, int32_t* kept_idx,
                         int64_t* M_out, void* workspace, size_t workspace_bytes,
                         tg_stream_t stream);

/*
 * tg_select_topk without a workspace argument, for callers that cannot
 * allocate device memory or hand the library a buffer: a host that owns all
 * device memory and allows no allocation after start-up, a plug-in inside
 * another framework's allocator, a C caller with no allocator at hand, or a
 * latency-critical path (cudaMalloc can synchronise the device, cudaFree
 * does).  The pages have no counterpart: this is a deployment variant of the
 * select above, with the same arguments (minus the workspace), the same
 * result and the same limits.  It allocates nothing: its scratch is a
 * 104 KiB array compiled into the library, which every GPU that loads the
 * library holds until the process exits.  A call whose scratch would not fit
 * in the array returns TG_ERR_UNSUPPORTED (no N < 2^31 needs more today).
 * The first call on each device looks up that device's array address
 * (cudaGetSymbolAddress) while the device is current; make that first call
 * outside any stream capture.  Each call clears the array on `stream`
 * (cudaMemsetAsync) before its kernel.  All calls share the one array per
 * device: calls that overlap on the GPU race and must not be made.  The
 * gate's fused first-pass histogram (tg_gate_score's select_ws) is not used.
 */
tg_status tg_select_topk_noalloc(const float* scores, int64_t N,
                                 int64_t doc_begin, int64_t doc_end, int64_t K,
                                 int32_t* kept_idx, int64_t* M_out,
                                 tg_stream_t stream);

/*
 * Row gather ([IT] "TokenGate impara quali token mantenere": only the kept
 * tokens' representations go up; [DE] "Was ist token-gated Attention?":
 * their scores become the attention bias):
 *   Y[m] = X[idx[m]]                      (exact copy, or bf16 -> fp32 widen)
 *   logsig_kept[m] = log(sigmoid(scores[idx[m]]))   (fp32, stable form)
 *
 *  X      [N][d] in x_dtype.     idx: [M] int32, or NULL for the identity
 *         (then M must equal N).
 *  Y      [M][d] in y_dtype; (x_dtype, y_dtype) is (bf16, bf16), (f32, f32)
 *         or (bf16, f32).
 *  scores [N] fp32 and logsig_kept [M] fp32: both NULL or both given.
 * M == 0 launches nothing.  An index outside [0, N) sets TG_ERR_BAD_INDEX
 * and that row is zeroed.
 */
tg_status tg_gather_rows(const void* X, tg_dtype x_dtype, int64_t N,
                         int32_t d, const int32_t* idx, int64_t M, void* Y,
                         tg_dtype y_dtype, const float* scores,
                         float* logsig_kept, tg_stream_t stream);

/*
 * RMSNorm of a pruned layer's input (the pages' pruned layers are ordinary
 * decoder layers run on the kept rows, [DE] "Prune-Front-Behandlung"):
 *   Y[i][c] = X[i][c] * gamma[c] / sqrt(mean_c(X[i][c]^2) + eps)
 *  X [M][d] in x_dtype (f32 or bf16); Y [M][d] in y_dtype (bf16 or f32).
 *  gamma [d] fp32.  d % 8 == 0.
 */
tg_status tg_rmsnorm(const void* X, tg_dtype x_dtype, int64_t M, int32_t d,
                     const float* gamma, float eps, void* Y, tg_dtype y_dtype,
                     tg_stream_t stream);

/*
 * QKV projection of the kept rows (layers above L, [DE] "Prune-Front-
 * Behandlung": no KV is produced for pruned tokens):
 *   QKV = X * Wqkv^T,  Wqkv [(Hq + 2 Hkv) * dh][d] (nn.Linear layout):
 *   output columns [0, Hq dh) are q heads, then Hkv dh of k, then Hkv dh
 *   of v.  TG_BF16: tcgen05 GEMM, fp32 accumulation, bf16 output rounded
 *   to nearest-even.  TG_F32: fp32 CUDA-core GEMM.
 *  X [M][d], QKV [M][(Hq + 2 Hkv) dh], both in `dtype`.
 * Limits: d % 64 == 0 and (Hq + 2 Hkv) dh % 16 == 0 for TG_BF16;
 * d % 4 == 0 for TG_F32.
 */
tg_status tg_qkv_proj(const void* X, tg_dtype dtype, int64_t M, int32_t d,
                      const void* Wqkv, int32_t Hq, int32_t Hkv, int32_t dh,
                      void* QKV, tg_stream_t stream);

/*
 * ---- A full decoder layer above the gate on the kept rows ([DE] "Wie hat
 * TokenGate das Pruning von Tokens verstanden?": the layers above L process
 * only the kept tokens; [IT] "TokenGate impara quali token mantenere": only
 * their representations go up).  The layer's internals are the base model's
 * (Qwen3): RMSNorm -> q|k|v -> per-head RMSNorm of q and k -> rotary
 * embedding -> token-gated attention -> o-projection + residual -> RMSNorm
 * -> SwiGLU MLP + residual.  The one pruning-specific choice: every kept row
 * keeps its ORIGINAL prompt position for the rotary embedding (a kept row's
 * result then equals the full prompt's at that row with the pruned keys
 * masked).  bf16 operands, fp32 accumulation, an fp32 residual stream.
 */

/*
 * Rotary table of the kept rows: for c < dh / 2,
 *   table[m][c] = (cos, sin)(positions[m] * base^(-2c / dh)),
 * [M][dh / 2][2] fp32, built once per prompt and shared by every layer.
 * The angle is formed and reduced modulo 2 pi in fp64; its cosine and sine
 * are taken in fp32.
 *  positions  [M] int32, the rows' positions in the prompt (the kept
 *             indices of tg_select_topk).
 * Limits: dh even, 2..1024; base > 1.
 */
tg_status tg_rope_table(const int32_t* positions, int64_t M, int32_t dh, double base,
                        float* table, tg_stream_t stream);

/*
 * QKV projection with Qwen3's per-head q/k RMSNorm and the rotary
 * embedding, fused into the GEMM epilogue (the accumulator never leaves
 * fp32 before the final bf16 store):
 *   qkv = X Wqkv^T;  for each q head (gamma_q) and k head (gamma_k), row m:
 *   y = x / sqrt(mean(x^2) + eps) * gamma;  then for c < dh / 2
 *   (y_c, y_{c+dh/2}) <- (y_c cos - y_{c+dh/2} sin, y_{c+dh/2} cos + y_c sin)
 *   with (cos, sin) = rope_table[m][c];  v heads unchanged.
 *  X [M][d] bf16; Wqkv [(Hq + 2 Hkv) dh][d] bf16; QKV [M][(Hq + 2 Hkv) dh]
 *  bf16 (layout of tg_qkv_proj); gamma_q, gamma_k [dh] fp32; rope_table as
 *  tg_rope_table wrote it.
 * Limits: dh == 128, d % 64 == 0, eps >= 0.
 */
tg_status tg_qkv_proj_qknorm_rope(const void* X, int64_t M, int32_t d, const void* Wqkv,
                                  int32_t Hq, int32_t Hkv, int32_t dh, const float* gamma_q,
                                  const float* gamma_k, float eps, const float* rope_table,
                                  void* QKV, tg_stream_t stream);

/*
 * A projection added into the residual stream (the o-projection and the
 * MLP's down-projection):  residual[m][n] += sum_k X[m][k] W[n][k].
 *  X [M][K] bf16; W [N][K] bf16 (nn.Linear layout); residual [M][N] fp32,
 *  updated in place.  Limits: K % 64 == 0, N % 32 == 0.
 */
tg_status tg_linear_residual(const void* X, int64_t M, int32_t K, const void* W, int32_t N,
                             float* residual, tg_stream_t stream);

/*
 * The SwiGLU hidden layer:  Y = silu(X W_gate^T) * (X W_up^T),
 * silu(z) = z / (1 + exp(-z)).  One GEMM: each CTA pair computes 128
 * columns of both products, one CTA loading W_gate's rows, the other
 * W_up's, and the epilogue multiplies them.
 *  X [M][d] bf16; W_gate, W_up [F][d] bf16; Y [M][F] bf16.
 * Limits: d % 64 == 0, F % 32 == 0.
 */
tg_status tg_swiglu(const void* X, int64_t M, int32_t d, const void* W_gate, const void* W_up,
                    int32_t F, void* Y, tg_stream_t stream);

/*
 * Token-gated causal attention over the kept rows ([DE] "Was ist
 * token-gated Attention?"; [TH] token-gated attention, per-head gain and
 * learnable temperature; [RU] "Механизм token-gated attention"):
 *   l_ij = t * (q_i . k_j) / sqrt(dh) + g_h * logsig_kept[j],  j <= i
 *   o_i  = sum_j softmax_j(l_ij) v_j,   kv head of q head h = h / (Hq/Hkv)
 * Rows are the kept tokens in ascending original order, so causality on
 * row numbers equals causality on original positions.
 *
 *  QKV          [M][(Hq + 2 Hkv) dh] in `dtype` (layout of tg_qkv_proj).
 *  logsig_kept  [M] fp32, or NULL for no bias (plain causal attention, the
 *               full-prefill path).
 *  gain         [Hq] fp32 (ignored when logsig_kept is NULL).
 *  temperature  scalar t.
 *  O            [M][Hq dh] in `dtype`, or NULL when residual is given.
 *  residual     [M][Hq dh] fp32 or NULL: when given, residual += o in fp32
 *               (the layer's residual add), fused into the epilogue.
 * Limits: Hq % Hkv == 0.  TG_BF16: dh == 128, (Hq / Hkv) even, and t finite
 * and > 0 (the kernel folds the bias into the q.k product as
 * g_h logsig_kept[j] sqrt(dh) / t, and takes row maxima of q.k; both need
 * t > 0); other t return TG_ERR_UNSUPPORTED.
 * TG_F32: dh <= 128 and dh % 4 == 0.
 */
tg_status tg_keybias_attn(const void* QKV, tg_dtype dtype, int64_t M,
                          int32_t Hq, int32_t Hkv, int32_t dh,
                          const float* logsig_kept, const float* gain,
                          float temperature, void* O, float* residual,
                          tg_stream_t stream);

/*
 * tg_keybias_attn, and also the per-row normaliser that a backward pass
 * re-uses:  lse[h][i] = log sum_{j <= i} exp(l_ij)  (natural log), fp32,
 * [Hq][M] densely packed (row h starts at lse + h * M).  Same arguments and
 * limits as tg_keybias_attn; lse must not be NULL when M > 0.
 */
tg_status tg_keybias_attn_lse(const void* QKV, tg_dtype dtype, int64_t M,
                              int32_t Hq, int32_t Hkv, int32_t dh,
                              const float* logsig_kept, const float* gain,
                              float temperature, void* O, float* residual,
                              float* lse, tg_stream_t stream);

/*
 * ---- The gradient the bias carries back to the scorer ([DE] "Was ist
 * token-gated Attention?": the kept token's score becomes a bias on the
 * attention logits, which gives the gradient a path back to the scorer;
 * [TH] the same, MoE-router style).  With b_hj = g_h * logsig_kept[j] and an
 * upstream gradient dO = dL/dO of the attention output, the chain rule gives
 *   dL/db_hj = sum_{i >= j} P_ij (dO_i . v_j - D_i),  D_i = dO_i . o_i,
 * with P_ij = exp(l_ij - lse_i) and dO_i, o_i the dh columns of head h.
 * The four calls, in order: tg_keybias_attn_lse (forward), tg_attn_bwd_delta,
 * tg_keybias_attn_bias_grad, tg_bias_grad_reduce.
 */

/*
 * D[h][i] = sum_c dO[i][h dh + c] * O[i][h dh + c], accumulated in fp32.
 *  dO, O   [M][Hq dh] in `dtype` (O as written by the forward).
 *  delta   [Hq][M] fp32 output, densely packed.
 * Limits: TG_BF16: dh in {64, 128, 256}; TG_F32: dh in {32, 64, 128}.
 */
tg_status tg_attn_bwd_delta(const void* dO, const void* O, tg_dtype dtype,
                            int64_t M, int32_t Hq, int32_t dh, float* delta,
                            tg_stream_t stream);

/*
 * dbias[h][j] = dL/db_hj for every q head h and kept row j (fp32, [Hq][M]
 * densely packed): P is recomputed from QKV, logsig_kept, gain, temperature
 * and lse (as tg_keybias_attn_lse wrote it), and D comes from
 * tg_attn_bwd_delta.  TG_BF16: tcgen05 tensor cores, fp32 accumulation;
 * TG_F32: CUDA cores.
 *  QKV          [M][(Hq + 2 Hkv) dh] in `dtype`; dO [M][Hq dh] in `dtype`.
 *  logsig_kept  [M] fp32 or NULL (no bias: b = 0); gain [Hq] fp32.
 *  lse, delta   [Hq][M] fp32.
 * Limits: Hq % Hkv == 0; t finite; TG_BF16: dh == 128; TG_F32: dh in
 * {32, 64, 128}.
 */
tg_status tg_keybias_attn_bias_grad(const void* QKV, const void* dO,
                                    tg_dtype dtype, int64_t M, int32_t Hq,
                                    int32_t Hkv, int32_t dh,
                                    const float* logsig_kept,
                                    const float* gain, float temperature,
                                    const float* lse, const float* delta,
                                    float* dbias, tg_stream_t stream);

/*
 * From dbias [Hq][M] (all fp32):
 *   dlogsig[j] = sum_h gain[h] * dbias[h][j]            (dL/d logsig_kept)
 *   dgain[h]   = sum_j logsig_kept[j] * dbias[h][j]     (dL/dg)
 *   dscore[j]  = dlogsig[j] * sigmoid(-s_j)              (dL/ds of kept token j,
 *                with sigmoid(-s) = -expm1(logsig_kept[j]); NULL to skip)
 * Pruned tokens get no gradient through this path.  Fixed summation order:
 * the results are bitwise reproducible.  M == 0 writes dgain = 0.
 */
tg_status tg_bias_grad_reduce(const float* dbias, int64_t M, int32_t Hq,
                              const float* logsig_kept, const float* gain,
                              float* dlogsig, float* dgain, float* dscore,
                              tg_stream_t stream);

/*
 * ---- Gated-DeltaNet layers of a hybrid model ([TH] "การใช้งานกับโมเดล
 * hybrid-attention"; [DE] "Wird es auf Hybrid-Attention-Modellen
 * funktionieren?"; [IT] "I modelli ibridi ampliano le possibilità di
 * selezione dei token": the gate can sit in a Gated-DeltaNet layer of a
 * hybrid model, and the DeltaNet layers above it are pruned too).  The pages
 * give no formula; the recurrence is the published gated delta rule, per
 * head h with a state S in R^{dv x dk}:
 *   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *   o_t = S_t q_t.
 * A pruned layer calls it on the kept tokens only (rows in prompt order):
 * a pruned token neither decays nor writes the state.
 *
 *  q, k  [T][H][dk] in `dtype` (the caller normalises k; bf16 or fp32).
 *  v     [T][H][dv] in `dtype`.
 *  alpha [T][H] fp32 in (0, 1];  beta [T][H] fp32 in [0, 1].
 *  S0    [H][dv][dk] fp32 initial state, or NULL for zero.
 *  o     [T][H][dv] output in `dtype`.
 *  S_out [H][dv][dk] fp32 final state, or NULL.
 *  workspace  device, tg_gated_delta_rule_workspace_bytes(T, H) bytes (no
 *             zeroing needed; every call overwrites what it reads).
 * Evaluated in chunks of 64 tokens, fp32 arithmetic throughout.
 * Limits: dk == dv == 128.
 */
size_t tg_gated_delta_rule_workspace_bytes(int64_t T, int32_t H);
tg_status tg_gated_delta_rule(const void* q, const void* k, const void* v, tg_dtype dtype,
                              const float* alpha, const float* beta, int64_t T, int32_t H,
                              int32_t dk, int32_t dv, const float* S0, void* o, float* S_out,
                              void* workspace, size_t workspace_bytes, tg_stream_t stream);

/*
 * ---- The gated layer as one CUDA graph ([DE] "Wie hat TokenGate das
 * Pruning von Tokens verstanden?": score every token, keep the top K, run
 * the layers above on the kept rows).  A plan captures the five calls of one
 * gated layer on fixed buffers -- tg_gate_score (counting the select's first
 * radix pass into the select workspace), tg_select_topk, tg_gather_rows,
 * tg_qkv_proj, tg_keybias_attn -- into a CUDA graph once; tg_plan_launch
 * replays it with one launch per prompt, so a new prompt is written into X
 * and the graph runs again.  bf16 path only.
 */
typedef struct tg_gated_layer_desc {
  const void* X;           /* [N][d] bf16 residual at the gate layer            */
  int64_t N;
  int32_t d;
  const void* W1;          /* [Hg][d] bf16                                      */
  const float* b1;         /* [Hg] or NULL                                      */
  int32_t Hg;
  const float* w2;         /* [Hg]                                              */
  float b2;
  int64_t doc_begin, doc_end, K;
  const void* Wqkv;        /* [(Hq + 2 Hkv) dh][d] bf16                         */
  int32_t Hq, Hkv, dh;
  const float* gain;       /* [Hq]                                              */
  float temperature;
  /* outputs and scratch, all owned by the caller */
  float* scores;           /* [N]                                               */
  void* select_ws;         /* tg_select_workspace_bytes(N) bytes, zeroed once   */
  size_t select_ws_bytes;
  int32_t* kept_idx;       /* [M], M = N - (doc_end - doc_begin) + K            */
  void* Xk;                /* [M][d] bf16                                       */
  float* logsig_kept;      /* [M]                                               */
  void* QKV;               /* [M][(Hq + 2 Hkv) dh] bf16                         */
  void* O;                 /* [M][Hq dh] bf16                                   */
} tg_gated_layer_desc;

typedef struct tg_plan_s* tg_plan_t;

/* Captures the gated layer described by *desc (every argument check of the
 * five calls runs here, once) and instantiates the graph.  *plan receives a
 * handle to release with tg_plan_destroy.  Uses the current device. */
tg_status tg_gated_layer_plan_create(const tg_gated_layer_desc* desc, tg_plan_t* plan);
/* Replays the plan's graph on `stream` (asynchronous). */
tg_status tg_plan_launch(tg_plan_t plan, tg_stream_t stream);
/* Releases the graph; plan must not be in use on the GPU. */
tg_status tg_plan_destroy(tg_plan_t plan);

/*
 * Synchronises `stream`, then returns and clears the sticky device status
 * of the current device: TG_OK, or the first of TG_ERR_NAN_SCORE,
 * TG_ERR_BAD_INDEX, TG_ERR_TIMEOUT that is set.  TG_ERR_CUDA if the
 * synchronisation itself failed.  The word is per device and shared by all
 * streams; it is read and cleared in one atomic exchange on `stream`, so a
 * bit that a kernel on another stream sets meanwhile is either returned now
 * or kept for the next call, never lost.
 */
tg_status tg_get_device_status(tg_stream_t stream);

/*
 * Self-check of the failure path (the pages have no counterpart: this is the
 * library's own diagnostic).  Every pipeline wait in this library is bounded:
 * a wait that gives up sets TG_ERR_TIMEOUT in the device status word and an
 * abort flag that makes the CTA's other waiters leave, so a lost arrival
 * becomes an error status instead of a hung GPU.  This call launches one CTA
 * with an mbarrier that nothing completes: one thread waits on it with a
 * bound of `timeout_us` microseconds and gives up; a second thread waits on
 * it with the pipelines' own bound (2 s) and must leave early because of the
 * abort flag.  Afterwards tg_get_device_status returns TG_ERR_TIMEOUT (once),
 * and the device stays usable.
 *  timeout_us  1 .. 1000000.
 *  report      device, 4 x uint64, or NULL: for the short-bound waiter then
 *              the abort-driven waiter, (1 if its wait succeeded else 0,
 *              nanoseconds it waited).  8-byte aligned.
 */
tg_status tg_selftest_bounded_wait(uint32_t timeout_us, unsigned long long* report,
                                   tg_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* TOKENGATE_H */
