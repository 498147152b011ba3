// fp32 GEMM on the CUDA cores with the same fused epilogues as the tensor-core
// path.  It serves the F32 number path, whose tolerance (max relative error
// 1e-4 on hidden states) rules out TF32 tensor cores (10-bit mantissa).
//
//   y[M, N] = epilogue( x[M, K] . W ),  W [K, N] (Conv1D) or [N, K] (lm_head)
//
// 64 x 64 output tile per 256-thread block, 4 x 4 outputs per thread, fp32
// FMA accumulation in k order.
#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kT = 64;
constexpr int kKt = 16;

template <bool W_OUT_IN, int EPI>
__global__ void __launch_bounds__(256) gemm_f32_simt(const float* __restrict__ x, const float* __restrict__ w,
                                                     const float* __restrict__ bias, const float* residual, float* y,
                                                     int M, int N, int K, long long ldy) {
  __shared__ float As[kKt][kT + 4];
  __shared__ float Bs[kKt][kT + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15;
  const int ty = tid >> 4;
  const int m0 = blockIdx.y * kT;
  const int n0 = blockIdx.x * kT;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kKt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * 256;
      const int m = idx >> 4, k = idx & 15;
      const int gm = m0 + m, gk = k0 + k;
      As[k][m] = (gm < M && gk < K) ? x[static_cast<long long>(gm) * K + gk] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * 256;
      if (!W_OUT_IN) {
        const int k = idx >> 6, n = idx & 63;
        const int gk = k0 + k, gn = n0 + n;
        Bs[k][n] = (gk < K && gn < N) ? w[static_cast<long long>(gk) * N + gn] : 0.f;
      } else {
        const int n = idx >> 4, k = idx & 15;
        const int gk = k0 + k, gn = n0 + n;
        Bs[k][n] = (gk < K && gn < N) ? w[static_cast<long long>(gn) * K + gk] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kKt; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[k][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    if (row >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx * 4 + j;
      if (col >= N) continue;
      float v = acc[i][j];
      if (EPI != 0) v += bias[col];
      if (EPI == 2) v = gelu_new_accurate(v);
      if (EPI == 4) v = gelu_exact(v);
      if (EPI == 3) v += residual[static_cast<long long>(row) * N + col];
      y[static_cast<long long>(row) * ldy + col] = v;
    }
  }
}

template <bool W_OUT_IN>
cudaError_t dispatch(const float* x, const float* w, const float* bias, const float* residual, float* y, int M,
                     int N, int K, long long ldy, int epi, cudaStream_t s) {
  dim3 grid((N + kT - 1) / kT, (M + kT - 1) / kT);
  switch (epi) {
    case 0: gemm_f32_simt<W_OUT_IN, 0><<<grid, 256, 0, s>>>(x, w, bias, residual, y, M, N, K, ldy); break;
    case 1: gemm_f32_simt<W_OUT_IN, 1><<<grid, 256, 0, s>>>(x, w, bias, residual, y, M, N, K, ldy); break;
    case 2: gemm_f32_simt<W_OUT_IN, 2><<<grid, 256, 0, s>>>(x, w, bias, residual, y, M, N, K, ldy); break;
    case 4: gemm_f32_simt<W_OUT_IN, 4><<<grid, 256, 0, s>>>(x, w, bias, residual, y, M, N, K, ldy); break;
    default: gemm_f32_simt<W_OUT_IN, 3><<<grid, 256, 0, s>>>(x, w, bias, residual, y, M, N, K, ldy); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_f32(const float* x, const float* w, const float* bias, const float* residual, float* y,
                            int64_t M, int N, int K, int64_t ldy, bool w_out_in, int epilogue, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int m = static_cast<int>(M);
  return w_out_in ? dispatch<true>(x, w, bias, residual, y, m, N, K, ldy, epilogue, stream)
                  : dispatch<false>(x, w, bias, residual, y, m, N, K, ldy, epilogue, stream);
}

}  // namespace gpt2
