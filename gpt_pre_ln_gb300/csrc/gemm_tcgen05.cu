// Instantiations of the tcgen05 GEMM (gemm_tcgen05.cuh) for the forward:
// the block's four projections and the lm_head, with their epilogues, and
// the log-sum-exp lm_head of the loss.
#include "gemm_tcgen05.cuh"

namespace gpt2 {

namespace {

template <bool B_MN, typename T16>
cudaError_t dispatch(int v, const T16* x, const T16* w, const T16* bias, const float* residual, void* y, int M, int N,
                     int K, long long ldy, int epi, gpt2_dtype y_t, cudaStream_t s) {
  unsigned* err = device_error_word();
  const Ops<T16> op{x, K, w, B_MN ? N : K, K};
  if (epi == EPI_RES) {
    EpiArgs<float, T16> ea{bias, residual, static_cast<float*>(y), ldy, M, N, err};
    return run_variant<false, B_MN, EPI_RES, float, T16>(v, op, ea, s);
  }
  if (y_t != GPT2_F32) {
    EpiArgs<T16, T16> ea{bias, residual, static_cast<T16*>(y), ldy, M, N, err};
    ea.gelu_exact = epi == GPT2_EPI_BIAS_GELU_EXACT;
    switch (epi) {
      case EPI_NONE: return run_variant<false, B_MN, EPI_NONE, T16, T16>(v, op, ea, s);
      case EPI_BIAS: return run_variant<false, B_MN, EPI_BIAS, T16, T16>(v, op, ea, s);
      default: return run_variant<false, B_MN, EPI_GELU, T16, T16>(v, op, ea, s);
    }
  }
  EpiArgs<float, T16> ea{bias, residual, static_cast<float*>(y), ldy, M, N, err};
  ea.gelu_exact = epi == GPT2_EPI_BIAS_GELU_EXACT;
  switch (epi) {
    case EPI_NONE: return run_variant<false, B_MN, EPI_NONE, float, T16>(v, op, ea, s);
    case EPI_BIAS: return run_variant<false, B_MN, EPI_BIAS, float, T16>(v, op, ea, s);
    default: return run_variant<false, B_MN, EPI_GELU, float, T16>(v, op, ea, s);
  }
}

template <typename T16>
cudaError_t launch(const void* x, const void* w, const void* bias, const float* residual, void* y, int64_t M, int N,
                   int K, int64_t ldy, bool w_out_in, int epilogue, gpt2_dtype y_t, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  if (M <= kMaxRowsGemm)
    return launch_gemm_rows_16(Type16<T16>::kFormat == 0 ? GPT2_F16 : GPT2_BF16, x, w, bias, residual, y, M, N, K,
                               ldy, w_out_in, epilogue, y_t, stream);
  const int m = static_cast<int>(M);
  const int v = pick_variant(m, N, K, epilogue == GPT2_EPI_BIAS_RESIDUAL);
  const T16* X = static_cast<const T16*>(x);
  const T16* W = static_cast<const T16*>(w);
  const T16* Bv = static_cast<const T16*>(bias);
  return w_out_in ? dispatch<false, T16>(v, X, W, Bv, residual, y, m, N, K, ldy, epilogue, y_t, stream)
                  : dispatch<true, T16>(v, X, W, Bv, residual, y, m, N, K, ldy, epilogue, y_t, stream);
}

template <typename T16>
cudaError_t launch_lse(const void* x, const void* w, int64_t M, int N, int K, const int32_t* labels, int T,
                       float2* part, float* tgt, int* n_part, cudaStream_t stream) {
  const int m = static_cast<int>(M);
  const int v = pick_variant(m, N);
  const int bn = variant_bn(v);
  *n_part = 2 * ((N + bn - 1) / bn);
  EpiArgs<float, T16> ea{nullptr, nullptr, nullptr, 0, m, N, device_error_word(), labels, T, part, tgt};
  const Ops<T16> op{static_cast<const T16*>(x), K, static_cast<const T16*>(w), K, K};
  return run_variant<false, false, EPI_LSE, float, T16>(v, op, ea, stream);
}

}  // namespace

cudaError_t launch_gemm_lse_16(gpt2_dtype dt, const void* x, const void* w, int64_t M, int N, int K,
                               const int32_t* labels, int T, float2* part, float* tgt, int* n_part,
                               cudaStream_t stream) {
  if (M <= kMaxRowsGemm) return cudaErrorNotSupported;
  if (dt == GPT2_F16) return launch_lse<__half>(x, w, M, N, K, labels, T, part, tgt, n_part, stream);
  return launch_lse<__nv_bfloat16>(x, w, M, N, K, labels, T, part, tgt, n_part, stream);
}

cudaError_t launch_gemm_16(gpt2_dtype dt, const void* x, const void* w, const void* bias, const float* residual,
                           void* y, int64_t M, int N, int K, int64_t ldy, bool w_out_in, int epilogue, gpt2_dtype y_t,
                           cudaStream_t stream) {
  if (dt == GPT2_F16)
    return launch<__half>(x, w, bias, residual, y, M, N, K, ldy, w_out_in, epilogue, y_t, stream);
  return launch<__nv_bfloat16>(x, w, bias, residual, y, M, N, K, ldy, w_out_in, epilogue, y_t, stream);
}

}  // namespace gpt2
