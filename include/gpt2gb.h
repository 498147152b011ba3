/*
 * gpt2gb.h -- C ABI of the GB300 (sm_103a) GPT-2 Pre-LN forward library
 * (libgpt2gb.so).
 *
 * The operations are those of the GPT-2 Pre-LN Transformer as the pages
 * describe it:
 *   "Hidden State 如何流过 GPT-2 Block", section "GPT-2 Block":
 *       A = Attention(LN_attn(X)); H = X + A; M = MLP(LN_ffn(H)); X' = H + M
 *   "逐行拆GPT-2源码": GPT2Config (eps = 1e-5, n_inner = 4 * n_embd),
 *       Conv1D (bias + x @ W, W stored [in, out]), GPT2Attention (fused c_attn,
 *       Q|K|V split, 64-wide heads, scores / sqrt(head_dim), causal mask,
 *       softmax, merge, c_proj), GPT2MLP (c_fc, gelu_new, c_proj),
 *       GPT2Model (wte + wpe, position ids from past_length, ln_f),
 *       GPT2LMHeadModel (lm_head tied to wte, no bias), KV cache.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership: the caller owns every buffer (weights, activations, caches,
 *   workspace).  The library never allocates or frees device memory on these
 *   calls, keeps no model state, and never synchronises the stream it is
 *   given.  All pointers are DEVICE pointers unless stated otherwise;
 *   host-side structs (gpt2_dims, gpt2_block_weights, gpt2_model_weights and
 *   the blocks array) are read during the call only.
 * Streams: work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream).  Calls contain no host synchronisation, so a sequence of
 *   them can be captured in a CUDA graph.
 * Errors: every call returns a gpt2_status.  Argument checks happen before
 *   anything is enqueued (nothing runs when a check fails).  Faults that the
 *   device detects (a bounded wait that ran out, an index out of range) set a
 *   device error word and make the kernel return early; gpt2_last_error()
 *   reads it.  No C++ exception crosses this interface.
 * Layout: row-major everywhere.  Hidden states are [B, T, D] (M = B*T rows of
 *   D), linear weights are [in, out] as the Hugging Face Conv1D stores them.
 * Number types (gpt2_dtype): the BF16 path keeps weights, LayerNorm outputs,
 *   QKV, attention output and MLP hidden in bf16, accumulates in fp32 and
 *   keeps the residual stream, LayerNorm statistics and the softmax in fp32.
 *   The F16 path is the same with fp16 in place of bf16 (fp16 carries 3 more
 *   mantissa bits; bf16 weights convert to fp16 exactly down to magnitude
 *   2^-17, so a bf16 model runs on it unchanged in practice).  The F32 path
 *   keeps everything in fp32.
 * Supported shapes: head_dim = d_model / n_head must be 64; d_model a
 *   multiple of 64; d_ff a multiple of 64; T <= n_pos.  Anything else returns
 *   GPT2_ERR_UNSUPPORTED (shape) or GPT2_ERR_ARG (a null or inconsistent
 *   argument).  Device pointers must be 16-byte aligned.
 */
#ifndef GPT2GB_H
#define GPT2GB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *gpt2_stream_t;

typedef enum {
  GPT2_OK = 0,
  GPT2_ERR_ARG = 1,          /* null pointer, negative size, inconsistent dims */
  GPT2_ERR_UNSUPPORTED = 2,  /* a shape or type combination the library does not run */
  GPT2_ERR_WORKSPACE = 3,    /* workspace smaller than gpt2_*_workspace_bytes() */
  GPT2_ERR_CUDA = 4,         /* a CUDA runtime call or a kernel launch failed */
  GPT2_ERR_TIMEOUT = 5,      /* device side: a bounded wait ran out */
  GPT2_ERR_RANGE = 6         /* device side: a token id or position out of range */
} gpt2_status;

typedef enum { GPT2_F32 = 0, GPT2_BF16 = 1, GPT2_F16 = 2 } gpt2_dtype;

/* Switches of GPT2Config ("逐行拆GPT-2源码", GPT2Config section), OR-ed
 * into gpt2_dims.flags; 0 is GPT-2 as released.
 *   GPT2_SCALE_ATTN_BY_INVERSE_LAYER_IDX: the attention scores of layer l
 *     (counted from 0) are divided by l + 1 on top of the 1/sqrt(64) scale
 *     (scale_attn_by_inverse_layer_idx).
 *   GPT2_GELU_EXACT: the MLP uses GELU itself, x Phi(x) =
 *     0.5 x (1 + erf(x / sqrt(2))) (llm.c notes 4.2), in place of its tanh
 *     approximation gelu_new. */
enum { GPT2_SCALE_ATTN_BY_INVERSE_LAYER_IDX = 1, GPT2_GELU_EXACT = 2 };

/* Model hyper-parameters (GPT2Config on "逐行拆GPT-2源码": n_layer, n_embd,
 * n_head, n_inner = d_ff (4 * n_embd by default; any multiple of 64 runs),
 * vocab_size, n_positions, layer_norm_epsilon).  `dtype` selects the number
 * path described above; `flags` holds the switches above (an unknown bit is
 * GPT2_ERR_ARG).  Zero-initialise the struct so that flags start at 0. */
typedef struct {
  int n_layer;
  int d_model;
  int n_head;
  int d_ff;
  int vocab;
  int n_pos;
  float eps;
  gpt2_dtype dtype;
  unsigned flags;
} gpt2_dims;

/* One block's 12 tensors (6 groups of weight + bias, the safetensors key
 * list on "逐行拆GPT-2源码").  Element type = dims.dtype.
 *   ln1_g, ln1_b [D]; w_qkv [D, 3D]; b_qkv [3D]; w_o [D, D]; b_o [D];
 *   ln2_g, ln2_b [D]; w_fc [D, F]; b_fc [F]; w_proj [F, D]; b_proj [D]. */
typedef struct {
  const void *ln1_g, *ln1_b;
  const void *w_qkv, *b_qkv;
  const void *w_o, *b_o;
  const void *ln2_g, *ln2_b;
  const void *w_fc, *b_fc;
  const void *w_proj, *b_proj;
} gpt2_block_weights;

/* Whole model.  wte [V, D] (also the tied lm_head), wpe [n_pos, D],
 * lnf_g / lnf_b [D]; element type = dims.dtype.  `blocks` is a HOST array of
 * n_layer entries whose pointers are device pointers. */
typedef struct {
  const void *wte;
  const void *wpe;
  const void *lnf_g, *lnf_b;
  const gpt2_block_weights *blocks;
} gpt2_model_weights;

/* Epilogues of gpt2_linear. */
typedef enum {
  GPT2_EPI_NONE = 0,            /* y = x W                               */
  GPT2_EPI_BIAS = 1,            /* y = x W + b                           */
  GPT2_EPI_BIAS_GELU = 2,       /* y = gelu_new(x W + b)                 */
  GPT2_EPI_BIAS_RESIDUAL = 3,   /* y = r + x W + b  (y, r fp32)          */
  GPT2_EPI_BIAS_GELU_EXACT = 4  /* y = gelu(x W + b), gelu(u) = u Phi(u) */
} gpt2_epilogue;

/* Orientation of the weight of gpt2_linear. */
typedef enum {
  GPT2_W_IN_OUT = 0,  /* W is [K, N] (Conv1D, every block weight)      */
  GPT2_W_OUT_IN = 1   /* W is [N, K] (wte used as the tied lm_head)    */
} gpt2_weight_layout;

/* Library version of this interface (increments on any signature change). */
int gpt2_abi_version(void);

/* Human-readable text for a gpt2_status (static storage). */
const char *gpt2_status_string(int status);

/* First device-side fault recorded since the previous call, then cleared.
 * Synchronises the whole device first, so call it outside stream capture.
 * Returns GPT2_OK, GPT2_ERR_TIMEOUT or GPT2_ERR_RANGE (or GPT2_ERR_CUDA if
 * the read itself failed).  If `site` is not NULL it receives a code naming
 * the kernel and the wait that failed (0 when there is none). */
int gpt2_last_error(int *site);

/* Self-test of the failure detection above; the pages have no counterpart
 * (they describe no GPU code).  Enqueues one GPU thread that waits, through
 * the same bounded mbarrier wait every kernel of the library uses, on a
 * barrier that nothing ever arrives on, with a wait limit of `limit_ns`
 * nanoseconds of GPU wall time (1 .. 2e9; the library's own kernels use
 * 2e9) in place of the library's.  When the limit runs out the thread
 * records GPT2_ERR_TIMEOUT with site 18 in the device error word and the
 * kernel returns; nothing faults, traps or hangs, and the context stays
 * usable.  A following gpt2_last_error() returns GPT2_ERR_TIMEOUT and site
 * 18 (and clears the word).  Returns GPT2_ERR_ARG for a limit outside the
 * range (nothing enqueued), GPT2_ERR_CUDA if the launch failed. */
int gpt2_selftest_wait_timeout(uint64_t limit_ns, gpt2_stream_t stream);

/* LayerNorm over the last axis: y = gamma * (x - mean) / sqrt(var + eps) + beta,
 * var the population variance ("Hidden State 如何流过 GPT-2 Block", section
 * "Pre-Norm"; llm.c notes section 3.2: eps added to the variance).
 *   x [rows, D] of type x_t; y [rows, D] of type y_t; gamma, beta [D] of type
 *   y_t.  Statistics in fp32.  rows >= 0 (0 is a no-op), 4 <= D <= 4096 and
 *   D a multiple of 4.  x and y must not overlap. */
int gpt2_layernorm(const void *x, const void *gamma, const void *beta, void *y, int64_t rows, int D, float eps,
                   gpt2_dtype x_t, gpt2_dtype y_t, gpt2_stream_t stream);

/* Conv1D with a fused epilogue ("逐行拆GPT-2源码", GPT2Attention section:
 * Conv1D is addmm(bias, x, W)).  x [M, K] and W (see `w_layout`) of type
 * `dtype`; bias [N] of type `dtype` (ignored for GPT2_EPI_NONE); residual
 * [M, N] fp32 with row stride N (GPT2_EPI_BIAS_RESIDUAL only, may equal y);
 * y [M, ldy] of type y_t (fp32 when the epilogue is BIAS_RESIDUAL).
 * The BF16 path runs on the tcgen05 tensor cores (fp32 accumulate in tensor
 * memory); the F32 path on CUDA cores in fp32.
 *   M >= 0, N >= 1, K a multiple of 64, ldy >= N.  BF16 path: ldy times the
 *   size of y_t a multiple of 16 bytes (y is written by TMA bulk stores),
 *   N a multiple of 8 for GPT2_W_IN_OUT; BIAS_RESIDUAL: N a multiple of 4.
 *   Otherwise GPT2_ERR_UNSUPPORTED.  On the BF16 path the padding columns of
 *   each row of y from N up to the next 16-byte boundary are written with
 *   zeros; columns beyond that boundary are never written. */
int gpt2_linear(const void *x, const void *w, const void *bias, const float *residual, void *y, int64_t M, int N,
                int K, int64_t ldy, gpt2_weight_layout w_layout, gpt2_epilogue epilogue, gpt2_dtype dtype,
                gpt2_dtype y_t, gpt2_stream_t stream);

/* Causal multi-head self-attention on a packed QKV projection
 * ("逐行拆GPT-2源码", GPT2Attention ``_split_heads`` / ``_attn`` /
 * ``_merge_heads``; llm.c notes 2.2-2.3):
 *   for each batch b, head h and query i:
 *     out[b, i, h*64 + d] = sum_{j <= i} softmax_j(q_i . k_j / 8) v_j[d]
 *   with q_i = qkv[b, i, h*64 : h*64+64], k_j = qkv[b, j, D + h*64 : ...],
 *   v_j = qkv[b, j, 2D + h*64 : ...], D = n_head * head_dim.
 *   qkv [B, T, 3D] and out [B, T, D] of type `dtype`; softmax in fp32.
 *   head_dim must be 64.  B, T >= 0. */
int gpt2_attention_causal(const void *qkv, void *out, int B, int T, int n_head, int head_dim, gpt2_dtype dtype,
                          gpt2_stream_t stream);

/* gpt2_attention_causal with the scores q_i . k_j multiplied by
 * `score_scale` instead of 1/8 (with GPT2Config's
 * scale_attn_by_inverse_layer_idx, layer l uses 1 / (8 (l + 1))).
 * score_scale must be finite and > 0, else GPT2_ERR_ARG. */
int gpt2_attention_causal_scaled(const void *qkv, void *out, int B, int T, int n_head, int head_dim,
                                 float score_scale, gpt2_dtype dtype, gpt2_stream_t stream);

/* gpt2_attention_causal_scaled that also keeps, for the backward, each
 * query row's log-sum-exp of its scaled scores: lse[b, h, t] (fp32
 * [B, n_head, T]) = log2 sum_{j <= t} 2^(score_scale * log2(e) * q_t . k_j),
 * so that p_tj = 2^(score_scale * log2(e) * q_t . k_j - lse[b, h, t]).
 * 16-bit dtypes only (GPT2_ERR_UNSUPPORTED for GPT2_F32). */
int gpt2_attention_causal_lse(const void *qkv, void *out, float *lse, int B, int T, int n_head, int head_dim,
                              float score_scale, gpt2_dtype dtype, gpt2_stream_t stream);

/* Backward of the causal attention (llm.c notes 5.3: the softmax gradient
 * of the max-subtracted forward, no gradient at masked positions):
 *   dv = p^T do, dp = do v^T, ds = p (dp - rowsum(do * o)),
 *   dq = c ds k, dk = c ds^T q   (c = score_scale, per head)
 * qkv [B, T, 3D] and out [B, T, D] are the forward's input and output, lse
 * its row statistics (gpt2_attention_causal_lse), dout [B, T, D] the
 * gradient of out; dqkv [B, T, 3D] receives the gradients of Q | K | V in
 * the layout of qkv.  16-bit dtypes (all of qkv, out, dout, dqkv), fp32
 * accumulation on the tensor cores; p and ds are rounded to the 16-bit type
 * before they multiply.  The result does not depend on timing (no atomics).
 * ws: device workspace of gpt2_attention_backward_workspace_bytes(B, T,
 * n_head) bytes, 256-byte aligned. */
size_t gpt2_attention_backward_workspace_bytes(int B, int T, int n_head);
int gpt2_attention_causal_backward(const void *qkv, const void *out, const float *lse, const void *dout, void *dqkv,
                                   int B, int T, int n_head, int head_dim, float score_scale, void *ws,
                                   size_t ws_bytes, gpt2_dtype dtype, gpt2_stream_t stream);

/* Workspace needed by gpt2_mlp for M rows (the [M, F] hidden activation). */
size_t gpt2_mlp_workspace_bytes(int64_t M, int F, gpt2_dtype dtype);

/* MLP sublayer on an already normalised input ("逐行拆GPT-2源码", GPT2MLP:
 * c_fc -> gelu_new -> c_proj), with the residual add of GPT2Block fused:
 *   out = residual + gelu_new(x W_fc + b_fc) W_proj + b_proj
 *   x [M, D] of type dtype; w_fc [D, F]; b_fc [F]; w_proj [F, D]; b_proj [D]
 *   (type dtype); residual [M, D] fp32 or NULL (then out = the MLP output);
 *   out [M, D] fp32, may equal residual.  ws: device workspace of at least
 *   gpt2_mlp_workspace_bytes(M, F, dtype) bytes, 256-byte aligned. */
int gpt2_mlp(const void *x, const void *w_fc, const void *b_fc, const void *w_proj, const void *b_proj,
             const float *residual, float *out, int64_t M, int D, int F, void *ws, size_t ws_bytes,
             gpt2_dtype dtype, gpt2_stream_t stream);

/* gpt2_mlp without a workspace argument, for callers that cannot allocate
 * device memory when they call in (for example a plug-in whose host
 * framework has reserved the GPU's memory in its own pool, or code running
 * while a stream is captured into a CUDA graph, where cudaMalloc is not
 * allowed).  The pages have no counterpart of this call: it is a deployment
 * convenience over gpt2_mlp, with identical arguments apart from the
 * workspace and identical results.
 *   The [M, F] hidden activation is kept in a scratch array in device memory
 *   that the library owns: gpt2_mlp_noalloc_max_scratch_bytes() bytes per
 *   GPU (16 MiB), held from the library's first use on a device until the
 *   process exits.  M * F * (2 for BF16, 4 for F32) above that size returns
 *   GPT2_ERR_WORKSPACE and runs nothing.  Nothing is allocated by the call.
 *   The first call on each device looks up the scratch array's device
 *   address (cudaGetSymbolAddress); make that first call outside stream
 *   capture.  All calls on a device share the one array: calls whose GPU
 *   work may overlap (unordered streams) race on it; calls ordered on one
 *   stream are safe.  No part of the array needs clearing between calls.
 *   The looked-up address is kept for the life of the process: after a
 *   cudaDeviceReset of a device, do not call this entry point on it again
 *   in the same process (the new context's array may lie elsewhere). */
size_t gpt2_mlp_noalloc_max_scratch_bytes(void);
int gpt2_mlp_noalloc(const void *x, const void *w_fc, const void *b_fc, const void *w_proj, const void *b_proj,
                     const float *residual, float *out, int64_t M, int D, int F, gpt2_dtype dtype,
                     gpt2_stream_t stream);

/* Workspace needed by gpt2_block_forward and gpt2_forward_logits for a
 * [B, T] batch (0 if the dims are invalid). */
size_t gpt2_workspace_bytes(const gpt2_dims *dims, int B, int T);

/* One Pre-LN block ("Hidden State 如何流过 GPT-2 Block", section "GPT-2
 * Block"; "逐行拆GPT-2源码", GPT2Block.forward):
 *   H = X + c_proj(attn(c_attn(LN_1(X)))); X' = H + mlp(LN_2(H)).
 *   x_in, x_out: fp32 [B, T, D] residual stream (x_out may equal x_in);
 *   weights of type dims->dtype; ws of gpt2_workspace_bytes(dims, B, T)
 *   bytes.  dims->n_layer, vocab and n_pos are not used.  The block is
 *   taken as layer 0 (this matters only with
 *   GPT2_SCALE_ATTN_BY_INVERSE_LAYER_IDX). */
int gpt2_block_forward(const gpt2_dims *dims, const gpt2_block_weights *w, const float *x_in, float *x_out, int B,
                       int T, void *ws, size_t ws_bytes, gpt2_stream_t stream);

/* gpt2_block_forward for the block at index `layer` >= 0 of the stack
 * (counted from 0): with GPT2_SCALE_ATTN_BY_INVERSE_LAYER_IDX its attention
 * scores are divided by layer + 1. */
int gpt2_block_forward_layer(const gpt2_dims *dims, const gpt2_block_weights *w, int layer, const float *x_in,
                             float *x_out, int B, int T, void *ws, size_t ws_bytes, gpt2_stream_t stream);

/* Whole forward to logits ("逐行拆GPT-2源码", GPT2Model + GPT2LMHeadModel;
 * "Transformer Stack" page, GPT.forward):
 *   x0 = wte[tokens] + wpe[0..T-1]; n_layer blocks; logits = LN_f(x) wte^T.
 *   tokens: int32 [B, T] device, each in [0, vocab) (else GPT2_ERR_RANGE on
 *   the device; that row's embedding is taken as zero); logits [B, T, ld] of
 *   type logits_t, ld >= vocab, ld times the element size a multiple of 16
 *   bytes on the BF16 path; T <= n_pos. */
int gpt2_forward_logits(const gpt2_dims *dims, const gpt2_model_weights *w, const int32_t *tokens, void *logits,
                        int64_t ld, gpt2_dtype logits_t, int B, int T, void *ws, size_t ws_bytes,
                        gpt2_stream_t stream);

/* Gradients of one block's 12 tensors, fp32 device buffers shaped like the
 * tensors of gpt2_block_weights (written, not accumulated). */
typedef struct {
  float *ln1_g, *ln1_b;
  float *w_qkv, *b_qkv;
  float *w_o, *b_o;
  float *ln2_g, *ln2_b;
  float *w_fc, *b_fc;
  float *w_proj, *b_proj;
} gpt2_block_grads;

/* Workspace needed by gpt2_block_backward for a [B, T] batch (0 if the dims
 * are invalid or not the F32 path). */
size_t gpt2_block_backward_workspace_bytes(const gpt2_dims *dims, int B, int T);

/* Backward pass of one Pre-LN block on the F32 path (llm.c notes section
 * 5.3: LayerNorm gradients through the mean, the variance and the
 * normalised value, with gamma's and beta's own; the softmax gradient;
 * zero gradient at causally masked positions).  Given the block's input
 * x_in [B, T, D] and the gradient dx_out [B, T, D] of a scalar loss with
 * respect to its output, writes dx_in [B, T, D] (the gradient with respect
 * to the input) and every weight gradient into `grads`.  The forward
 * intermediates are recomputed into the workspace.  `layer` as in
 * gpt2_block_forward_layer (the index of the block in its stack).
 *   dims->dtype must be GPT2_F32 (else GPT2_ERR_UNSUPPORTED); T <= 4096 and
 *   B <= 65535;
 *   dx_in must not overlap x_in or dx_out; ws of
 *   gpt2_block_backward_workspace_bytes(dims, B, T) bytes, 256-byte
 *   aligned.  fp32 CUDA cores throughout; the sums over rows run in a
 *   fixed order, so results are deterministic. */
int gpt2_block_backward(const gpt2_dims *dims, const gpt2_block_weights *w, int layer, const float *x_in,
                        const float *dx_out, float *dx_in, const gpt2_block_grads *grads, int B, int T, void *ws,
                        size_t ws_bytes, gpt2_stream_t stream);

/* Gradients of the whole model, fp32 device buffers of the weights' shapes
 * (blocks: a HOST array of n_layer gpt2_block_grads). */
typedef struct {
  float *wte;   /* [V, D]: the tied lm_head and the embedding together */
  float *wpe;   /* [n_pos, D]: rows >= T are set to zero */
  float *lnf_g, *lnf_b;
  const gpt2_block_grads *blocks;
} gpt2_model_grads;

/* Workspace of gpt2_forward_backward for a [B, T] batch (0 if the dims are
 * invalid or not GPT2_BF16). */
size_t gpt2_train_workspace_bytes(const gpt2_dims *dims, int B, int T);

/* One training step's arithmetic: the forward of gpt2_forward_loss, keeping
 * every block's intermediates (llm.c notes 5.2), the mean shifted
 * cross-entropy into *mean_loss (device fp32), and the gradient of that
 * loss with respect to every parameter into `grads` (written, not added;
 * llm.c notes 5.3 for the LayerNorm and softmax gradients; "逐行拆GPT-2源码",
 * GPT2LMHeadModel: wte receives the lm_head's and the embedding's
 * gradient).  dL/dz at position t < T-1 is (softmax(z) - onehot(label of
 * t+1)) / (B (T-1)), zero at the last position of each sequence.
 *   dims->dtype must be GPT2_BF16 (else GPT2_ERR_UNSUPPORTED): bf16 operands
 *   on the tensor cores with fp32 accumulation (the products of every
 *   linear layer, of the lm_head and of the attention backward), fp32
 *   LayerNorm, residual-stream and bias gradients; sums over rows in a fixed
 *   order (results do not depend on timing).  tokens / labels as in
 *   gpt2_forward_loss (labels NULL = tokens); T >= 2; ws of
 *   gpt2_train_workspace_bytes(dims, B, T) bytes, 256-byte aligned (about
 *   0.2 GB per layer at GPT-2 small width and B T = 8192, plus the
 *   [B T, vocab] bf16 loss gradient). */
int gpt2_forward_backward(const gpt2_dims *dims, const gpt2_model_weights *w, const int32_t *tokens,
                          const int32_t *labels, const gpt2_model_grads *grads, float *mean_loss, int B, int T,
                          void *ws, size_t ws_bytes, gpt2_stream_t stream);

/* Workspace needed by gpt2_forward_loss for a [B, T] batch (0 if the dims
 * are invalid). */
size_t gpt2_loss_workspace_bytes(const gpt2_dims *dims, int B, int T);

/* Whole forward to the language-model loss ("逐行拆GPT-2源码",
 * GPT2LMHeadModel.forward with labels): the forward of gpt2_forward_logits,
 * then position t of each sequence is scored against labels[b, t + 1] (the
 * shift happens here, so labels may be the input ids themselves) by the
 * cross-entropy lse(z) - z[label], lse(z) = log sum_v exp(z_v) over the
 * vocabulary, and the mean is taken over all B (T - 1) positions.  The
 * [B, T, vocab] logits are never written: on the 16-bit paths with
 * B T > 128 the lm_head GEMM reduces each row to log-sum-exp partials and
 * the target logit in its epilogue.
 *   tokens: int32 [B, T] device (as gpt2_forward_logits); labels: NULL
 *   (= tokens) or int32 [B, T] device, each used label in [0, vocab) (else
 *   GPT2_ERR_RANGE on the device and a NaN loss at that position);
 *   token_loss: NULL or fp32 [B, T - 1] device; lse: NULL or fp32 [B, T]
 *   device (log-sum-exp of every position's logits, so that
 *   p(v) = exp(z_v - lse)); mean_loss: NULL or one fp32 on the device, the
 *   mean of the B (T - 1) losses summed in a fixed order (deterministic).
 *   At least one output must be given.  2 <= T <= n_pos; ws of
 *   gpt2_loss_workspace_bytes(dims, B, T) bytes, 256-byte aligned. */
int gpt2_forward_loss(const gpt2_dims *dims, const gpt2_model_weights *w, const int32_t *tokens,
                      const int32_t *labels, float *token_loss, float *lse, float *mean_loss, int B, int T, void *ws,
                      size_t ws_bytes, gpt2_stream_t stream);

/* Bytes of a KV cache laid out [n_layer, 2 (K, V), B, n_head, T_max, 64] in
 * the path's element type (2 bytes for BF16 and F16, 4 for F32). */
size_t gpt2_kv_cache_bytes(const gpt2_dims *dims, int B, int T_max);

/* Workspace needed by gpt2_prefill for a [B, T] prompt batch. */
size_t gpt2_prefill_workspace_bytes(const gpt2_dims *dims, int B, int T);

/* Prompt processing ahead of gpt2_decode_step ("逐行拆GPT-2源码",
 * GPT2Attention with use_cache: `present` keeps each layer's K and V of the
 * positions processed so far; GPT2Model: positions start at 0 without a
 * cache): the forward of gpt2_forward_logits over tokens [B, T], which also
 * writes every layer's K and V of positions 0..T-1 into cache slots 0..T-1
 * of each sequence; then LN_f and the tied lm_head on each sequence's last
 * position only, argmax (lowest index on ties) -> next_tokens[b], and
 * past_len[b] = T.  A following gpt2_decode_step with tokens = next_tokens
 * continues the greedy sequence at position T.
 *   kv_cache: [n_layer, 2, B, n_head, T_max, 64] (gpt2_kv_cache_bytes; slots
 *   >= T are not touched); past_len, next_tokens: int32 [B] device (written);
 *   logits_opt: NULL or fp32 [B, ld] device receiving the last position's
 *   logits (ld >= vocab, a multiple of 4); 1 <= T <= min(n_pos, T_max);
 *   ws of gpt2_prefill_workspace_bytes(dims, B, T) bytes.  16-bit paths
 *   only, and 2 * B * n_head * T_max < 2^31. */
int gpt2_prefill(const gpt2_dims *dims, const gpt2_model_weights *w, const int32_t *tokens, int B, int T,
                 void *kv_cache, int T_max, int32_t *past_len, int32_t *next_tokens, float *logits_opt, int64_t ld,
                 void *ws, size_t ws_bytes, gpt2_stream_t stream);

/* Workspace needed by gpt2_decode_step for a batch of B sequences. */
size_t gpt2_decode_workspace_bytes(const gpt2_dims *dims, int B);

/* One greedy decode step with a KV cache ("逐行拆GPT-2源码": position ids
 * continue at past_length; the new K, V are concatenated after the cached
 * ones; the query attends over all of them; huaweicloud page section 九:
 * the next token is chosen from the lm_head scores).  For each sequence b:
 *   pos = past_len[b]; x = wte[tokens[b]] + wpe[pos]; per layer: LN_1, c_attn,
 *   write k, v into cache slot pos, attend over slots 0..pos, c_proj +
 *   residual, LN_2, MLP + residual; then LN_f, tied lm_head, argmax (lowest
 *   index on ties) -> next_tokens[b]; finally past_len[b] += 1.
 *   kv_cache: [n_layer, 2, B, n_head, T_max, 64] (gpt2_kv_cache_bytes);
 *   past_len: int32 [B] device, read and incremented in place; needs
 *   past_len[b] < T_max and < n_pos (else GPT2_ERR_RANGE on the device, and
 *   that sequence is left unchanged); tokens, next_tokens: int32 [B] device
 *   (they may be the same buffer); logits_opt: NULL or fp32 [B, ld] device
 *   receiving the step's logits (ld >= vocab, a multiple of 4); ws of
 *   gpt2_decode_workspace_bytes(dims, B) bytes.  16-bit paths only (BF16,
 *   F16: GPT2_ERR_UNSUPPORTED for F32), and 2 * B * n_head * T_max < 2^31.
 *   Everything runs on `stream` and allocates nothing, so after a first call
 *   on a device (which sets kernel attributes) the call may be captured into
 *   a CUDA graph and replayed. */
int gpt2_decode_step(const gpt2_dims *dims, const gpt2_model_weights *w, void *kv_cache, int B, int T_max,
                     int32_t *past_len, const int32_t *tokens, int32_t *next_tokens, float *logits_opt, int64_t ld,
                     void *ws, size_t ws_bytes, gpt2_stream_t stream);

/* ------------------------------------------------------------ profiling
 * Per-kernel timing of the calls made between gpt2_profile_begin() and
 * gpt2_profile_end(): the library records a CUDA event on the launching
 * stream before and after each kernel it launches and tags the pair with
 * the kernel's name and its algorithmic work (flops and bytes, counted from
 * the shapes, not measured).  begin() creates the events (host-side CUDA
 * objects, no device memory); call it outside stream capture.  Launches
 * beyond `max_launches` are not recorded (still run).  read() waits for the
 * recorded events and returns one entry per kernel name, in first-launch
 * order; it fails with GPT2_ERR_ARG if recording is still on. */
typedef struct {
  char name[48];
  int launches;
  double ms;      /* sum over launches of (end event - start event) */
  double flops;   /* algorithmic floating-point operations, summed */
  double bytes;   /* algorithmic DRAM bytes (inputs read + outputs written), summed */
} gpt2_profile_entry;

int gpt2_profile_begin(int max_launches);
int gpt2_profile_end(void);
int gpt2_profile_read(gpt2_profile_entry *out, int max_entries, int *n_entries);

#ifdef __cplusplus
}
#endif

#endif /* GPT2GB_H */
