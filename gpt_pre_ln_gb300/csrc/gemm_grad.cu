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
cudaError_t run_plain(const Ops<T16>& op, void* y, long long ldy, int M, int N, int splits, cudaStream_t s) {
  EpiArgs<OutT, T16> ea{nullptr, nullptr, static_cast<OutT*>(y), ldy, M, N, device_error_word()};
  ea.splits = splits;
  const int v = pick_grad_variant(M, N);
  if (v == 0) return run_2sm<kPairBN, A_MN, B_MN, EPI_NONE, OutT, T16>(op, ea, s);
  // the D-wide input gradients over a long K (dX of c_fc and c_attn, and
  // dxf over the vocabulary): the 192-wide pair tile
  if constexpr (!A_MN && sizeof(OutT) == 4) {
    if (use_pair192(M, N, op.K)) return run_2sm<192, A_MN, B_MN, EPI_NONE, OutT, T16>(op, ea, s);
  }
  return run_1sm<192, A_MN, B_MN, EPI_NONE, OutT, T16>(op, ea, s);
}

// The K split of a weight-gradient product: fewer output tiles than SMs (or
// CTA pairs) over a long K (the rows of the batch) leave SMs idle, so K is
// split S ways: S minimising ceil(tiles S / units) / S over 1..6, each split
// keeping at least four k-blocks; no split once the tiles fill a round (the
// partial slabs would cost more traffic than the last round saves).
constexpr int kMaxSplits = 6;
int pick_splits(int M, int N, int K) {
  const int v = pick_grad_variant(M, N);
  const long long tiles = v == 0 ? static_cast<long long>((M + 255) / 256) * ((N + 255) / 256)
                                 : static_cast<long long>((M + kBM - 1) / kBM) * ((N + 191) / 192);
  const long long units = v == 0 ? num_sms() / 2 : num_sms();
  const int kb = (K + kBK - 1) / kBK;
  int best = 1;
  if (tiles >= units) return best;
  double best_cost = 1.0;
  for (int S = 2; S <= kMaxSplits && kb / S >= 4; ++S) {
    const double cost = static_cast<double>((tiles * S + units - 1) / units) / S;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

// out[r, c] = sum over s of part[s M + r, c] (slabs in order).
__global__ void splitk_reduce(const float* __restrict__ part, int S, int M, int N, float* __restrict__ out,
                              long long ldo) {
  griddep_wait();
  griddep_launch_dependents();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long n4 = static_cast<long long>(M) * N / 4;
  if (i >= n4) return;
  const long long e = i * 4;
  const int r = static_cast<int>(e / N), c = static_cast<int>(e % N);
  // every slab's load in flight together (S <= kMaxSplits), then the sum
  // in slab order
  float4 v[kMaxSplits];
#pragma unroll
  for (int sp = 0; sp < kMaxSplits; ++sp)
    v[sp] = sp < S ? reinterpret_cast<const float4*>(part + static_cast<long long>(sp) * M * N)[i]
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 a = v[0];
#pragma unroll
  for (int sp = 1; sp < kMaxSplits; ++sp) {
    if (sp < S) {
      a.x += v[sp].x;
      a.y += v[sp].y;
      a.z += v[sp].z;
      a.w += v[sp].w;
    }
  }
  *reinterpret_cast<float4*>(out + r * ldo + c) = a;
}

}  // namespace

size_t gemm_grad_scratch_bytes(int M, int N, int K) {
  if (M % 32 != 0) return 0;
  const int S = pick_splits(M, N, K);
  return S > 1 ? static_cast<size_t>(S) * M * N * 4 : 0;
}

cudaError_t launch_gemm_grad(const void* a, long long lda, bool a_mn, const void* w, long long ldw, bool w_kn,
                             void* y, long long ldy, gpt2_dtype y_t, int M, int N, int K, cudaStream_t s,
                             float* scratch, size_t scratch_bytes) {
  if (M == 0 || N == 0) return cudaSuccess;
  const Ops<T16> op{static_cast<const T16*>(a), lda, static_cast<const T16*>(w), ldw, K};
  if (a_mn) {
    if (!w_kn || y_t != GPT2_F32) return cudaErrorNotSupported;
    const int S = pick_splits(M, N, K);
    // (slabs only when M is a multiple of the epilogue's 32-row store box,
    // so that no box of one slab reaches into the next)
    if (S > 1 && M % 32 == 0 && scratch && scratch_bytes >= static_cast<size_t>(S) * M * N * 4 && N % 4 == 0 &&
        ldy % 4 == 0) {
      cudaError_t e = run_plain<true, true, float>(op, scratch, N, M, N, S, s);
      if (e != cudaSuccess) return e;
      const long long n4 = static_cast<long long>(M) * N / 4;
      return launch_pdl(splitk_reduce, dim3(static_cast<unsigned>((n4 + 255) / 256)), 256, 0, s, 0,
                        static_cast<const float*>(scratch), S, M, N, static_cast<float*>(y), ldy);
    }
    return run_plain<true, true, float>(op, y, ldy, M, N, 1, s);
  }
  if (w_kn) {
    if (y_t != GPT2_F32) return cudaErrorNotSupported;
    return run_plain<false, true, float>(op, y, ldy, M, N, 1, s);
  }
  if (y_t == GPT2_F32) return run_plain<false, false, float>(op, y, ldy, M, N, 1, s);
  return run_plain<false, false, T16>(op, y, ldy, M, N, 1, s);
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
  if (pick_grad_variant(M, V) == 0) return run_2sm<kPairBN, false, false, EPI_DZ, T16, T16>(op, ea, s);
  return run_1sm<192, false, false, EPI_DZ, T16, T16>(op, ea, s);
}

}  // namespace gpt2
