// Backward pass of one Pre-LN block on the fp32 CUDA-core path: the
// kernels that the forward has no counterpart for.  The block's dataflow and
// its gradients (llm.c notes section 5.3: the LayerNorm gradient through
// the mean, the variance and the normalised value, with gamma's and beta's
// own; the softmax gradient; zero gradient at causally masked positions):
//
//   LayerNorm   dx = rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat)),
//               dxhat = dy gamma; dgamma = sum_rows dy xhat, dbeta = sum_rows dy
//   GELU        du = dg * act'(u) (gelu_new or the exact GELU)
//   Conv1D      dx = dy W^T (the forward GEMM with W read as [N, K]),
//               dW = x^T dy, db = sum_rows dy
//   attention   per head: p = softmax(c q k^T) over j <= i, o = p v;
//               dv_j = sum_i p_ij do_i, dp_ij = do_i . v_j,
//               ds_ij = p_ij (dp_ij - sum_j p_ij dp_ij),
//               dq_i = c sum_j ds_ij k_j, dk_j = c sum_i ds_ij q_i;
//               masked pairs (j > i) are never visited, so their
//               gradient is exactly zero
//
// Every sum over rows is taken in a fixed order (one thread per column,
// rows in sequence), so results are deterministic.  fp32 throughout.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kT = 64;   // output tile of the x^T dy GEMM
constexpr int kMt = 16;  // rows of x and dy per step
constexpr int kHd = 64;
constexpr int kBwdWarps = 4;

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// dW[K, N] = x[M, K]^T dy[M, N]: a 64 x 64 tile of dW per 256-thread block,
// 4 x 4 per thread, accumulated over m in order.
__global__ void __launch_bounds__(256) gemm_at_f32(const float* __restrict__ x, const float* __restrict__ dy,
                                                   float* __restrict__ dw, int M, int K, int N) {
  __shared__ float As[kMt][kT + 4];
  __shared__ float Bs[kMt][kT + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15;
  const int ty = tid >> 4;
  const int k0 = blockIdx.y * kT;
  const int n0 = blockIdx.x * kT;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int m0 = 0; m0 < M; m0 += kMt) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * 256;  // 0 .. 1023 = 16 rows x 64 columns
      const int m = idx >> 6, c = idx & 63;
      const int gm = m0 + m;
      As[m][c] = (gm < M && k0 + c < K) ? x[static_cast<long long>(gm) * K + k0 + c] : 0.f;
      Bs[m][c] = (gm < M && n0 + c < N) ? dy[static_cast<long long>(gm) * N + n0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kMt; ++m) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[m][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[m][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int k = k0 + ty * 4 + i;
    if (k >= K) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) dw[static_cast<long long>(k) * N + n] = acc[i][j];
    }
  }
}

// One warp per row: dx = rstd (dxhat - mean(dxhat) - xhat mean(dxhat xhat))
// (+ dres, the gradient arriving through the residual path, when given);
// prod[row] = dy * xhat for the dgamma column sums.
__global__ void __launch_bounds__(128) ln_backward_f32(const float* __restrict__ dy, const float* __restrict__ x,
                                                       const float* __restrict__ gamma, const float* dres,
                                                       float* dx, float* __restrict__ prod, int rows, int D,
                                                       float eps) {
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const long long base = static_cast<long long>(row) * D;
  float s = 0.f;
  for (int c = lane; c < D; c += 32) s += x[base + c];
  const float mean = warp_sum_f(s) / static_cast<float>(D);
  float q = 0.f;
  for (int c = lane; c < D; c += 32) {
    const float d = x[base + c] - mean;
    q = fmaf(d, d, q);
  }
  const float rstd = rsqrtf(warp_sum_f(q) / static_cast<float>(D) + eps);
  float s1 = 0.f, s2 = 0.f;
  for (int c = lane; c < D; c += 32) {
    const float xh = (x[base + c] - mean) * rstd;
    const float g = dy[base + c] * gamma[c];
    s1 += g;
    s2 = fmaf(g, xh, s2);
  }
  const float m1 = warp_sum_f(s1) / static_cast<float>(D);
  const float m2 = warp_sum_f(s2) / static_cast<float>(D);
  for (int c = lane; c < D; c += 32) {
    const float xh = (x[base + c] - mean) * rstd;
    const float g = dy[base + c] * gamma[c];
    float v = rstd * (g - m1 - xh * m2);
    if (dres) v += dres[base + c];
    dx[base + c] = v;
    prod[base + c] = dy[base + c] * xh;
  }
}

// g = act(u) (forward) and du = dg * act'(u) (backward), elementwise.
__global__ void gelu_forward_f32(const float* __restrict__ u, float* __restrict__ g, long long n, int exact) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float x = u[i];
  g[i] = exact ? gelu_exact(x) : gelu_new_accurate(x);
}

__global__ void gelu_backward_f32(const float* __restrict__ dg, const float* __restrict__ u, float* __restrict__ du,
                                  long long n, int exact) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float x = u[i];
  float d;
  if (exact) {
    // Phi(x) + x phi(x)
    const float Phi = 0.5f * (1.f + erff(x * 0.7071067811865476f));
    d = Phi + x * 0.3989422804014327f * expf(-0.5f * x * x);
  } else {
    const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
    const float t = tanhf(k0 * (x + 0.044715f * x * x * x));
    d = 0.5f * (1.f + t) + 0.5f * x * (1.f - t * t) * k0 * (1.f + 3.f * 0.044715f * x * x);
  }
  du[i] = dg[i] * d;
}

// Attention backward, pass over query rows: one warp per (b, h, i).
// Recomputes the row's probabilities, stores lse_i and
// delta_i = sum_j p_ij dp_ij ([B, H, T] each), and writes dq_i into the
// Q columns of dqkv.  sbuf: T floats per warp.
__global__ void __launch_bounds__(kBwdWarps * 32) attn_bwd_rows_f32(const float* __restrict__ qkv,
                                                                    const float* __restrict__ dout,
                                                                    float* __restrict__ dqkv,
                                                                    float* __restrict__ lse,
                                                                    float* __restrict__ delta, int T, int H,
                                                                    float c) {
  extern __shared__ float sbuf_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * kBwdWarps + warp;
  if (gw >= static_cast<long long>(H) * T) return;
  const int i = static_cast<int>(gw % T), h = static_cast<int>(gw / T), b = blockIdx.y;
  float* sb = sbuf_all + warp * T;
  const int D = H * kHd;
  const long long rs = 3LL * D;
  const float* base = qkv + static_cast<long long>(b) * T * rs;
  const float* q = base + static_cast<long long>(i) * rs + h * kHd;
  const float* dor = dout + (static_cast<long long>(b) * T + i) * D + h * kHd;
  float mx = -INFINITY;
  for (int j = lane; j <= i; j += 32) {
    const float* k = base + static_cast<long long>(j) * rs + D + h * kHd;
    float s = 0.f;
    for (int d = 0; d < kHd; ++d) s = fmaf(q[d], k[d], s);
    s *= c;
    sb[j] = s;
    mx = fmaxf(mx, s);
  }
  mx = warp_max_f(mx);
  float sum = 0.f;
  for (int j = lane; j <= i; j += 32) {
    const float e = expf(sb[j] - mx);
    sb[j] = e;
    sum += e;
  }
  sum = warp_sum_f(sum);
  const float inv = 1.f / sum;
  float dl = 0.f;
  for (int j = lane; j <= i; j += 32) {
    const float* v = base + static_cast<long long>(j) * rs + 2 * D + h * kHd;
    float dp = 0.f;
    for (int d = 0; d < kHd; ++d) dp = fmaf(dor[d], v[d], dp);
    const float p = sb[j] * inv;
    dl = fmaf(p, dp, dl);
    sb[j] = p;
  }
  dl = warp_sum_f(dl);
  for (int j = lane; j <= i; j += 32) {
    const float* v = base + static_cast<long long>(j) * rs + 2 * D + h * kHd;
    float dp = 0.f;
    for (int d = 0; d < kHd; ++d) dp = fmaf(dor[d], v[d], dp);
    sb[j] = sb[j] * (dp - dl);  // ds_ij
  }
  __syncwarp();
  float a0 = 0.f, a1 = 0.f;
  for (int j = 0; j <= i; ++j) {
    const float* k = base + static_cast<long long>(j) * rs + D + h * kHd;
    a0 = fmaf(sb[j], k[lane], a0);
    a1 = fmaf(sb[j], k[lane + 32], a1);
  }
  float* dq = dqkv + (static_cast<long long>(b) * T + i) * rs + h * kHd;
  dq[lane] = c * a0;
  dq[lane + 32] = c * a1;
  if (lane == 0) {
    const long long si = (static_cast<long long>(b) * H + h) * T + i;
    lse[si] = mx + logf(sum);
    delta[si] = dl;
  }
}

// Attention backward, pass over key rows: one warp per (b, h, j); p_ij and
// ds_ij for i >= j from lse_i and delta_i; writes dk_j and dv_j.  sbuf:
// 2 T floats per warp (p and ds).
__global__ void __launch_bounds__(kBwdWarps * 32) attn_bwd_cols_f32(const float* __restrict__ qkv,
                                                                    const float* __restrict__ dout,
                                                                    float* __restrict__ dqkv,
                                                                    const float* __restrict__ lse,
                                                                    const float* __restrict__ delta, int T, int H,
                                                                    float c) {
  extern __shared__ float sbuf_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * kBwdWarps + warp;
  if (gw >= static_cast<long long>(H) * T) return;
  const int j = static_cast<int>(gw % T), h = static_cast<int>(gw / T), b = blockIdx.y;
  float* pb = sbuf_all + warp * 2 * T;
  float* db = pb + T;
  const int D = H * kHd;
  const long long rs = 3LL * D;
  const float* base = qkv + static_cast<long long>(b) * T * rs;
  const float* k = base + static_cast<long long>(j) * rs + D + h * kHd;
  const float* v = base + static_cast<long long>(j) * rs + 2 * D + h * kHd;
  const long long st = (static_cast<long long>(b) * H + h) * T;
  for (int i = j + lane; i < T; i += 32) {
    const float* q = base + static_cast<long long>(i) * rs + h * kHd;
    const float* dor = dout + (static_cast<long long>(b) * T + i) * D + h * kHd;
    float s = 0.f, dp = 0.f;
    for (int d = 0; d < kHd; ++d) {
      s = fmaf(q[d], k[d], s);
      dp = fmaf(dor[d], v[d], dp);
    }
    const float p = expf(s * c - lse[st + i]);
    pb[i] = p;
    db[i] = p * (dp - delta[st + i]);
  }
  __syncwarp();
  float k0 = 0.f, k1 = 0.f, v0 = 0.f, v1 = 0.f;
  for (int i = j; i < T; ++i) {
    const float* q = base + static_cast<long long>(i) * rs + h * kHd;
    const float* dor = dout + (static_cast<long long>(b) * T + i) * D + h * kHd;
    k0 = fmaf(db[i], q[lane], k0);
    k1 = fmaf(db[i], q[lane + 32], k1);
    v0 = fmaf(pb[i], dor[lane], v0);
    v1 = fmaf(pb[i], dor[lane + 32], v1);
  }
  float* drow = dqkv + (static_cast<long long>(b) * T + j) * rs + h * kHd;
  drow[D + lane] = c * k0;
  drow[D + lane + 32] = c * k1;
  drow[2 * D + lane] = v0;
  drow[2 * D + lane + 32] = v1;
}

template <typename Kern>
cudaError_t set_smem(Kern kern, size_t smem) {
  if (smem <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
}

}  // namespace

cudaError_t launch_gemm_at_f32(const float* x, const float* dy, float* dw, int64_t M, int K, int N,
                               cudaStream_t stream) {
  if (K == 0 || N == 0) return cudaSuccess;
  dim3 grid((N + kT - 1) / kT, (K + kT - 1) / kT);
  gemm_at_f32<<<grid, 256, 0, stream>>>(x, dy, dw, static_cast<int>(M), K, N);
  return cudaGetLastError();
}


cudaError_t launch_ln_backward_f32(const float* dy, const float* x, const float* gamma, const float* dres, float* dx,
                                   float* prod, int64_t rows, int D, float eps, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((rows + 3) / 4);
  ln_backward_f32<<<blocks, 128, 0, stream>>>(dy, x, gamma, dres, dx, prod, static_cast<int>(rows), D, eps);
  return cudaGetLastError();
}

cudaError_t launch_gelu_f32(const float* u, float* g, int64_t n, bool exact, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  gelu_forward_f32<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(u, g, n, exact ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_gelu_backward_f32(const float* dg, const float* u, float* du, int64_t n, bool exact,
                                     cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  gelu_backward_f32<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(dg, u, du, n, exact ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_attention_backward_f32(const float* qkv, const float* dout, float* dqkv, float* lse, float* delta,
                                          int B, int T, int n_head, float score_scale, cudaStream_t stream) {
  if (B == 0 || T == 0) return cudaSuccess;
  const long long rows = static_cast<long long>(n_head) * T;
  dim3 grid(static_cast<unsigned>((rows + kBwdWarps - 1) / kBwdWarps), B);
  const size_t smem_r = static_cast<size_t>(kBwdWarps) * T * sizeof(float);
  const size_t smem_c = 2 * smem_r;
  cudaError_t e = set_smem(attn_bwd_rows_f32, smem_r);
  if (e != cudaSuccess) return e;
  e = set_smem(attn_bwd_cols_f32, smem_c);
  if (e != cudaSuccess) return e;
  attn_bwd_rows_f32<<<grid, kBwdWarps * 32, smem_r, stream>>>(qkv, dout, dqkv, lse, delta, T, n_head, score_scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_cols_f32<<<grid, kBwdWarps * 32, smem_c, stream>>>(qkv, dout, dqkv, lse, delta, T, n_head, score_scale);
  return cudaGetLastError();
}

}  // namespace gpt2
