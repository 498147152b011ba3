// The language-model loss of GPT2LMHeadModel ("逐行拆GPT-2源码",
// GPT2LMHeadModel section): position t of each sequence is scored against the
// label of position t + 1 by the cross-entropy lse(z) - z[label], and the
// mean is taken over all B (T-1) positions.
//
// The logits themselves are never needed whole: the lm_head GEMM's LSE
// epilogue leaves, per row, a (max, sum of exp(z - max)) pair for each of its
// column slices and the target logit.  loss_rows merges a row's pairs into
// lse = max + log(sum), then loss = lse - z_target; loss_mean sums the
// per-position losses in a fixed order (float64), so the result does not
// depend on scheduling.  lse_from_logits makes the same pairs from stored
// fp32 logits for the paths that write them (the fp32 model, few rows).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kRowsPerBlock = 32;
constexpr int kSliceWarps = 8;

// (m, s) <- the log-sum-exp pair of the union of the two column sets
__device__ __forceinline__ void lse_merge(float& m, float& s, float2 q) {
  if (q.y > 0.f) {
    const float nm = fmaxf(m, q.x);
    s = s * expf(m - nm) + q.y * expf(q.x - nm);  // m = -inf at first: 0
    m = nm;
  }
}

// One block per 32 rows; warp j merges slices j, j + 8, ... of each row
// (lane = row, so every load instruction reads 32 consecutive pairs), then
// warp 0 merges the eight results in a fixed order.
__global__ void __launch_bounds__(32 * kSliceWarps) loss_rows(const float2* __restrict__ part, int n_part,
                                                              const float* __restrict__ tgt,
                                                              const int32_t* __restrict__ labels, int B, int T, int V,
                                                              float* __restrict__ lse, float* __restrict__ token_loss,
                                                              unsigned* err) {
  __shared__ float2 red[kSliceWarps][kRowsPerBlock];
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long M = static_cast<long long>(B) * T;
  const long long r = static_cast<long long>(blockIdx.x) * kRowsPerBlock + lane;
  float m = -INFINITY, s = 0.f;
  if (r < M)
    for (int p = warp; p < n_part; p += kSliceWarps) lse_merge(m, s, part[p * M + r]);
  red[warp][lane] = make_float2(m, s);
  __syncthreads();
  if (warp != 0 || r >= M) return;
  m = -INFINITY;
  s = 0.f;
#pragma unroll
  for (int j = 0; j < kSliceWarps; ++j) lse_merge(m, s, red[j][lane]);
  const float l = m + logf(s);  // s >= 1: the maximum contributes exp(0)
  if (lse) lse[r] = l;
  const int t = static_cast<int>(r % T);
  if (t == T - 1) return;
  const int lbl = labels[r + 1];
  float loss;
  if (lbl < 0 || lbl >= V) {
    record_error(err, kErrRange, kSiteLossLabel);
    loss = __int_as_float(0x7fc00000);  // NaN
  } else {
    loss = l - tgt[r];
  }
  token_loss[(r / T) * (T - 1) + t] = loss;
}

// Mean of n values, one block: per-thread float64 partial sums over a fixed
// stride, then a fixed tree.
__global__ void __launch_bounds__(1024) loss_mean(const float* __restrict__ v, long long n, float* __restrict__ out) {
  __shared__ double acc[1024];
  griddep_wait();
  griddep_launch_dependents();
  double a = 0.0;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) a += v[i];
  acc[threadIdx.x] = a;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) acc[threadIdx.x] += acc[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = static_cast<float>(acc[0] / static_cast<double>(n));
}

// One warp per row of stored logits: lanes stride over the columns keeping
// their own (m, s), then merge across the warp by shuffles.
__global__ void __launch_bounds__(256) lse_from_logits(const float* __restrict__ logits, long long ld, long long M,
                                                       int V, const int32_t* __restrict__ labels, int T,
                                                       float2* __restrict__ part, float* __restrict__ tgt) {
  griddep_wait();
  griddep_launch_dependents();
  const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= M) return;
  const float* z = logits + r * ld;
  float m = -INFINITY, s = 0.f;
  for (int c = lane; c < V; c += 32) lse_merge(m, s, make_float2(z[c], 1.f));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, make_float2(om, os));
  }
  if (lane == 0) {
    part[r] = make_float2(m, s);
    if (static_cast<int>(r % T) != T - 1) {
      const int lbl = labels[r + 1];
      if (lbl >= 0 && lbl < V) tgt[r] = z[lbl];
    }
  }
}

}  // namespace

cudaError_t launch_loss_rows(const float2* part, int n_part, const float* tgt, const int32_t* labels, int B, int T,
                             int V, float* lse, float* token_loss, float* mean_loss, cudaStream_t stream) {
  const long long M = static_cast<long long>(B) * T;
  const unsigned blocks = static_cast<unsigned>((M + kRowsPerBlock - 1) / kRowsPerBlock);
  cudaError_t e = launch_pdl(loss_rows, dim3(blocks), dim3(32 * kSliceWarps), 0, stream, 0u, part, n_part, tgt,
                             labels, B, T, V, lse, token_loss, device_error_word());
  if (e != cudaSuccess || !mean_loss) return e;
  return launch_pdl(loss_mean, dim3(1), dim3(1024), 0, stream, 0u, static_cast<const float*>(token_loss),
                    static_cast<long long>(B) * (T - 1), mean_loss);
}

cudaError_t launch_lse_from_logits(const float* logits, int64_t ld, int64_t M, int V, const int32_t* labels, int T,
                                   float2* part, float* tgt, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((M + 7) / 8);
  return launch_pdl(lse_from_logits, dim3(blocks), dim3(256), 0, stream, 0u, logits, static_cast<long long>(ld),
                    static_cast<long long>(M), V, labels, T, part, tgt);
}

}  // namespace gpt2
