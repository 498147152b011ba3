// Instantiations of the tcgen05 GEMM (gemm_tcgen05.cuh) for the backward of
// the 16-bit path: products with an fp32 or 16-bit output and no epilogue,
// with A read K-major or MN-major and W read either way, and the lm_head
// with the loss-gradient epilogue.  bf16 only.
//
//   dX  = dY W^T      A = dY [M, out] K-major, W [in, out] read as [N, K]
//   dW  = X^T dY      A = X [rows, in] read MN-major ([K, M]), B = dY [K, N]
//   dxf = dz wte      A = dz [M, V] K-major, wte [V, D] read as [K, N]
//   dz  = (softmax(LN_f(x) wte^T) - onehot) / N   (EPI_DZ)
#include "gemm_tcgen05.cuh"

namespace gpt2 {

namespace {

using T16 = __nv_bfloat16;

// The pair kernel where the output is wide and tall, else single-CTA tiles of
// 128 x 192 (fewer instantiations than the forward's choice; the backward's
// shapes are the forward's transposes).
int pick_grad_variant(int M, int N) { return (M >= 2 * kBM && N > 1024) ? 0 : 192; }

template <bool A_MN, bool B_MN, typename OutT>
cudaError_t run_plain(const Ops<T16>& op, void* y, long long ldy, int M, int N, cudaStream_t s) {
  EpiArgs<OutT, T16> ea{nullptr, nullptr, static_cast<OutT*>(y), ldy, M, N, device_error_word()};
  const int v = pick_grad_variant(M, N);
  if (v == 0) return run_2sm<A_MN, B_MN, EPI_NONE, OutT, T16>(op, ea, s);
  return run_1sm<192, A_MN, B_MN, EPI_NONE, OutT, T16>(op, ea, s);
}

}  // namespace

cudaError_t launch_gemm_grad(const void* a, long long lda, bool a_mn, const void* w, long long ldw, bool w_kn,
                             void* y, long long ldy, gpt2_dtype y_t, int M, int N, int K, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  const Ops<T16> op{static_cast<const T16*>(a), lda, static_cast<const T16*>(w), ldw, K};
  if (a_mn) {
    if (!w_kn || y_t != GPT2_F32) return cudaErrorNotSupported;
    return run_plain<true, true, float>(op, y, ldy, M, N, s);
  }
  if (w_kn) {
    if (y_t != GPT2_F32) return cudaErrorNotSupported;
    return run_plain<false, true, float>(op, y, ldy, M, N, s);
  }
  if (y_t == GPT2_F32) return run_plain<false, false, float>(op, y, ldy, M, N, s);
  return run_plain<false, false, T16>(op, y, ldy, M, N, s);
}

cudaError_t launch_gemm_dlogits(const void* xf, const void* wte, int M, int V, int D, const float* row_lse,
                                const int32_t* labels, int T, float inv_n, void* dz, long long lddz,
                                cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  EpiArgs<T16, T16> ea{nullptr, nullptr, static_cast<T16*>(dz), lddz, M, V, device_error_word(), labels, T,
                       nullptr, nullptr};
  ea.row_lse = row_lse;
  ea.inv_n = inv_n;
  const Ops<T16> op{static_cast<const T16*>(xf), D, static_cast<const T16*>(wte), D, D};
  if (pick_grad_variant(M, V) == 0) return run_2sm<false, false, EPI_DZ, T16, T16>(op, ea, s);
  return run_1sm<192, false, false, EPI_DZ, T16, T16>(op, ea, s);
}

}  // namespace gpt2
