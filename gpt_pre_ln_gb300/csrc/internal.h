// Host-side declarations shared by the translation units of libgpt2gb.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gpt2gb.h"

namespace gpt2 {

// Device error word of the current device (see gpt2_last_error).
unsigned* device_error_word();
// Number of SMs of the current device (cached per device).
int num_sms();

// Launches `kern` with programmatic stream serialisation (see griddep_wait in
// common.cuh) and, when cluster_x > 0, thread-block clusters of cluster_x
// CTAs along x (0: no cluster attribute).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  unsigned n = 1;
  if (cluster_x > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// 2-D TMA map over a row-major [outer, inner] matrix with the given row pitch
// in bytes; boxes of [box_outer, box_inner] elements, 128-byte swizzle,
// out-of-range elements read as zero.  False if the driver rejects it.
bool encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);

// Each launcher validates nothing beyond what its kernel needs (the C-ABI
// layer has checked the arguments) and returns the launch status.
cudaError_t launch_layernorm(const void* x, const void* gamma, const void* beta, void* y, int64_t rows, int D,
                             float eps, gpt2_dtype x_t, gpt2_dtype y_t, cudaStream_t stream);

// x[m] = wte[tokens[m]] + wpe[pos0 + m % T] (fp32), y = LN(x) (type dt).
cudaError_t launch_embed_ln(const int32_t* tokens, const void* wte, const void* wpe, const void* gamma,
                            const void* beta, float* x, void* y, int B, int T, int D, int V, float eps, gpt2_dtype dt,
                            cudaStream_t stream);

// 16-bit tensor-core GEMM with a fused epilogue (tcgen05 + TMA); dt is
// GPT2_BF16 or GPT2_F16 (x, w, bias of that type), y_t is dt or GPT2_F32.
cudaError_t launch_gemm_16(gpt2_dtype dt, const void* x, const void* w, const void* bias, const float* residual,
                           void* y, int64_t M, int N, int K, int64_t ldy, bool w_out_in, int epilogue, gpt2_dtype y_t,
                           cudaStream_t stream);

// The lm_head of the loss: z = x . w^T (w [N, K], K-major), never stored.
// Per row r and column slice p: part[p * M + r] = (max_z, sum exp(z - max_z))
// over the slice; tgt[r] = z at column labels[r + 1] when r % T != T - 1 and
// that label is in [0, N) (not written otherwise).  *n_part = slices per
// row (at most lse_max_partials(N)).  M > kMaxRowsGemm only.
inline int lse_max_partials(int N) { return 2 * ((N + 127) / 128); }
cudaError_t launch_gemm_lse_16(gpt2_dtype dt, const void* x, const void* w, int64_t M, int N, int K,
                               const int32_t* labels, int T, float2* part, float* tgt, int* n_part,
                               cudaStream_t stream);

// The GEMM for the backward (bf16 operands, no epilogue; gemm_grad.cu):
//   y[M, N] = op(A) op(W) with A [M, K] (pitch lda) or, with a_mn, [K, M];
//   W [N, K] (pitch ldw) or, with w_kn, [K, N]; K any positive extent.
//   y fp32, or bf16 when neither a_mn nor w_kn.
//   With a_mn (weight gradients: few output tiles, K = the batch's rows) K
//   may be split over the SMs into fp32 partial slabs in `scratch` (at least
//   gemm_grad_scratch_bytes(M, N, K)), summed afterwards in a fixed order.
cudaError_t launch_gemm_grad(const void* a, long long lda, bool a_mn, const void* w, long long ldw, bool w_kn,
                             void* y, long long ldy, gpt2_dtype y_t, int M, int N, int K, cudaStream_t s,
                             float* scratch = nullptr, size_t scratch_bytes = 0);
size_t gemm_grad_scratch_bytes(int M, int N, int K);
// The loss gradient with respect to the logits z = xf wte^T (bf16 [M, D] x
// [V, D]), written as bf16 dz [M, lddz]: (exp(z - row_lse) - [v == label])
// * inv_n at row r with label labels[r + 1]; zero in the last row of every
// sequence of T rows.
cudaError_t launch_gemm_dlogits(const void* xf, const void* wte, int M, int V, int D, const float* row_lse,
                                const int32_t* labels, int T, float inv_n, void* dz, long long lddz, cudaStream_t s);

// The same GEMM for M <= kMaxRowsGemm rows (operands swapped, K split over a
// thread-block cluster); launch_gemm_16 hands such calls to it.  With
// argmax_cand (epilogue NONE, fp32 y, which may then be null) it also writes
// per-row argmax candidates: argmax_cand[m * rows_argmax_candidates(N) + c]
// = (value, index bits), to be reduced by launch_argmax_candidates.
constexpr int64_t kMaxRowsGemm = 128;
inline int rows_argmax_candidates(int N) { return 4 * ((N + 127) / 128); }
cudaError_t launch_gemm_rows_16(gpt2_dtype dt, const void* x, const void* w, const void* bias, const float* residual,
                                void* y, int64_t M, int N, int K, int64_t ldy, bool w_out_in, int epilogue,
                                gpt2_dtype y_t, cudaStream_t stream, float2* argmax_cand = nullptr);

// The MLP sublayer of gpt2_mlp: hidden = gelu_new(x W_fc + b_fc) (type dt,
// [M, F], caller memory), then out = residual + hidden W_proj + b_proj (fp32;
// no residual when it is null).  Both GEMMs go through the library's linear
// layer (per-kernel profiling included).
cudaError_t launch_mlp(gpt2_dtype dt, const void* x, const void* w_fc, const void* b_fc, const void* w_proj,
                       const void* b_proj, const float* residual, float* out, int64_t M, int D, int F, void* hidden,
                       cudaStream_t s);

// fp32 CUDA-core GEMM with the same epilogues.
cudaError_t launch_gemm_f32(const float* x, const float* w, const float* bias, const float* residual, float* y,
                            int64_t M, int N, int K, int64_t ldy, bool w_out_in, int epilogue, cudaStream_t stream);

// tcgen05 version (S and O in tensor memory), head_dim 64; dt GPT2_BF16 or
// GPT2_F16.
// Scores are q.k times score_scale (1/sqrt(64) for GPT-2).  With lse
// (fp32 [B, n_head, T]) each row's log2 sum_j 2^(s_j log2(e)) is kept for
// the backward.
cudaError_t launch_attention_tc(gpt2_dtype dt, const void* qkv, void* out, int B, int T, int n_head, float score_scale,
                                cudaStream_t stream, float* lse = nullptr);
// Causal attention backward (16-bit paths, tcgen05): dqkv [B, T, 3D] from
// qkv, the forward's output `out` and its lse (above), and dout [B, T, D];
// delta is [B, n_head, T] fp32 scratch.
cudaError_t launch_attention_backward_tc(gpt2_dtype dt, const void* qkv, const void* out, const float* lse,
                                         const void* dout, void* dqkv, float* delta, int B, int T, int n_head,
                                         float score_scale, cudaStream_t stream);
cudaError_t launch_attention_f32(const float* qkv, float* out, int B, int T, int n_head, float score_scale,
                                 cudaStream_t stream);

// Decode-step kernels (16-bit paths; dt GPT2_BF16 or GPT2_F16).
cudaError_t launch_decode_embed_ln(gpt2_dtype dt, const int32_t* tokens, const int32_t* past_len, const void* wte,
                                   const void* wpe, const void* gamma, const void* beta, float* x, void* y, int B,
                                   int D, int V, int n_pos, int T_max, float eps, int* valid, cudaStream_t stream);
// Rows 0..B-1 of qkv / out / past_len / valid are sequences b_cache0 ..
// b_cache0 + B - 1 of a cache laid out for B_cache sequences.
cudaError_t launch_decode_attention(gpt2_dtype dt, const void* qkv, void* kv_layer, void* out, const int32_t* past_len,
                                    const int* valid, int B, int b_cache0, int B_cache, int n_head, int T_max,
                                    float score_scale, cudaStream_t stream);
// Prefill: K and V of rows b T + t of qkv [B T, 3D] into cache slots t of
// sequences b (layer layout [2, B, n_head, T_max, 64]).
cudaError_t launch_kv_from_qkv(gpt2_dtype dt, const void* qkv, void* kv_layer, int B, int T, int n_head, int T_max,
                               cudaStream_t stream);
// x_last[b] = x[b T + T - 1] (fp32 [B, D]), valid[b] = 1, past_len[b] = T.
cudaError_t launch_prefill_last_rows(const float* x, int B, int T, int D, float* x_last, int* valid,
                                     int32_t* past_len, cudaStream_t stream);
// past_len may be null in the two argmax launchers (no increment).
cudaError_t launch_argmax_rows(const float* logits, int64_t ld, int B, int V, const int* valid, int32_t* next_tokens,
                               int32_t* past_len, cudaStream_t stream);
// The same from the candidates of launch_gemm_rows_16 (n_cand per row).
// Loss from log-sum-exp partials (n_part per row, layout of
// launch_gemm_lse_16) and target logits: lse[r] (nullable), token_loss
// [B, T-1] = lse - z_target (nullable), mean over the B (T-1) positions
// into *mean_loss (nullable).  A label outside [0, V) records kErrRange and
// gives a NaN loss.
cudaError_t launch_loss_rows(const float2* part, int n_part, const float* tgt, const int32_t* labels, int B, int T,
                             int V, float* lse, float* token_loss, float* mean_loss, cudaStream_t stream);
// Log-sum-exp partials (n_part = 1) and target logits from stored fp32 logits
// [M, ld], for the paths that write logits.
cudaError_t launch_lse_from_logits(const float* logits, int64_t ld, int64_t M, int V, const int32_t* labels, int T,
                                   float2* part, float* tgt, cudaStream_t stream);
cudaError_t launch_argmax_candidates(const float2* cand, int n_cand, int B, const int* valid, int32_t* next_tokens,
                                     int32_t* past_len, cudaStream_t stream);

// 16-bit backward kernels (backward_16.cu; bf16).
// out[N] = column sums of in[M, N] (row pitch ld; fp32 or, with in16, bf16),
// in a fixed order; partial: colsum_partial_bytes(M, N) of scratch.
size_t colsum_partial_bytes(long long M, int N);
cudaError_t launch_colsum(const void* in, bool in16, long long M, int N, long long ld, float* partial, float* out,
                          cudaStream_t s);
// g = act(u) over n bf16 values (n a multiple of 8, buffers 16-byte
// aligned); act gelu_new or, with exact, x Phi(x).
cudaError_t launch_gelu_fwd_16(const void* u, void* g, long long n, bool exact, cudaStream_t s);
// du = dg * act'(u) over [M, F] bf16 (F a multiple of 8, buffers 16-byte
// aligned) and dbias = the column sums of du; scratch:
// colsum_partial_bytes(M, F).
cudaError_t launch_gelu_bwd_sums_16(const void* dg, const void* u, void* du, long long M, int F, bool exact,
                                    float* dbias, float* scratch, cudaStream_t s);
// LayerNorm backward (gamma bf16): dx = LN'(x)^T dy (+ dres), dx16 (nullable)
// its bf16 copy, and the column sums dgamma = sum dy * xhat, dbeta = sum dy,
// dbias (nullable) = sum dx; scratch: ln_bwd_scratch_bytes(rows, D).
size_t ln_bwd_scratch_bytes(long long M, int D);
cudaError_t launch_ln_bwd_sums_16(const float* dy, const float* x, const void* gamma, const float* dres, float* dx,
                                  void* dx16, float* dgamma, float* dbeta, float* dbias, long long rows, int D,
                                  float eps, float* scratch, cudaStream_t s);
// dwte[tokens[m]] += dx0[m] (each row in position order), dwpe[t] = sum_b
// dx0[b, t] for t < T, 0 for T <= t < n_pos.
cudaError_t launch_embed_bwd(const int32_t* tokens, const float* dx0, float* dwte, float* dwpe, int B, int T, int D,
                             int V, int n_pos, cudaStream_t s);

// Backward of one block on the fp32 path (backward_f32.cu).
// dw[K, N] = x[M, K]^T dy[M, N].
cudaError_t launch_gemm_at_f32(const float* x, const float* dy, float* dw, int64_t M, int K, int N,
                               cudaStream_t stream);
// LayerNorm backward: dx = LN'(x)^T dy (+ dres when not null), prod = dy * xhat.
cudaError_t launch_ln_backward_f32(const float* dy, const float* x, const float* gamma, const float* dres, float* dx,
                                   float* prod, int64_t rows, int D, float eps, cudaStream_t stream);
// g = gelu(u) and du = dg * gelu'(u), the exact GELU or gelu_new.
cudaError_t launch_gelu_f32(const float* u, float* g, int64_t n, bool exact, cudaStream_t stream);
cudaError_t launch_gelu_backward_f32(const float* dg, const float* u, float* du, int64_t n, bool exact,
                                     cudaStream_t stream);
// Causal attention backward: dqkv [B, T, 3D] from qkv and dout [B, T, D];
// lse, delta: [B, n_head, T] scratch.  T <= 4096.
cudaError_t launch_attention_backward_f32(const float* qkv, const float* dout, float* dqkv, float* lse, float* delta,
                                          int B, int T, int n_head, float score_scale, cudaStream_t stream);

}  // namespace gpt2
