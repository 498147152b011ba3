// Causal multi-head self-attention on the packed c_attn output, fp32 path.
//
//   out[b, i, h*64 + d] = sum_{j <= i} softmax_j(q_i . k_j / sqrt(64)) v_j[d]
//
// ("逐行拆GPT-2源码", GPT2Attention ``_split_heads`` / ``_attn`` /
// ``_merge_heads``; llm.c notes 2.2-2.3: scale 1/sqrt(d_k), future positions
// masked before the softmax, row maximum subtracted.)  The Q|K|V split and
// the head split are index arithmetic on the [B, T, 3D] input; the head merge
// is the store into [B, T, D].
//
// One warp per query row, exact two-pass softmax with expf: the correctness
// path of the F32 configuration.  The 16-bit paths run attention_tc.cu.
#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kHd = 64;
// fp32 reference-precision attention: one warp per (b, h, i).
constexpr int kF32Warps = 4;

__global__ void __launch_bounds__(kF32Warps * 32) attn_causal_f32(const float* __restrict__ qkv,
                                                                  float* __restrict__ out, int T, int H,
                                                                  float score_scale) {
  extern __shared__ float sc[];  // kF32Warps x T scores
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * kF32Warps + warp;
  const int D = H * kHd;
  const long long total = static_cast<long long>(gridDim.y) * H * T;  // gridDim.y = B
  (void)total;
  const int i = static_cast<int>(gw % T);
  const int h = static_cast<int>((gw / T) % H);
  const int b = blockIdx.y;
  if (gw >= static_cast<long long>(H) * T) return;
  float* s = sc + warp * T;
  const long long rs = 3LL * D;
  const float* base = qkv + static_cast<long long>(b) * T * rs;
  const float* q = base + static_cast<long long>(i) * rs + h * kHd;
  // scores (lane j handles keys j, j+32, ...)
  float mx = -INFINITY;
  for (int j = lane; j <= i; j += 32) {
    const float* k = base + static_cast<long long>(j) * rs + D + h * kHd;
    float acc = 0.f;
#pragma unroll 16
    for (int d = 0; d < kHd; ++d) acc = fmaf(q[d], k[d], acc);
    acc *= score_scale;
    s[j] = acc;
    mx = fmaxf(mx, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.f;
  for (int j = lane; j <= i; j += 32) {
    const float e = expf(s[j] - mx);
    s[j] = e;
    sum += e;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncwarp();
  const float inv = 1.f / sum;
  float a0 = 0.f, a1 = 0.f;
  for (int j = 0; j <= i; ++j) {
    const float* v = base + static_cast<long long>(j) * rs + 2 * D + h * kHd;
    a0 = fmaf(s[j], v[lane], a0);
    a1 = fmaf(s[j], v[lane + 32], a1);
  }
  float* orow = out + (static_cast<long long>(b) * T + i) * D + h * kHd;
  orow[lane] = a0 * inv;
  orow[lane + 32] = a1 * inv;
}

}  // namespace

cudaError_t launch_attention_f32(const float* qkv, float* out, int B, int T, int n_head, float score_scale,
                                 cudaStream_t stream) {
  if (B == 0 || T == 0) return cudaSuccess;
  const long long rows = static_cast<long long>(n_head) * T;
  dim3 grid(static_cast<unsigned>((rows + kF32Warps - 1) / kF32Warps), B);
  const size_t smem = static_cast<size_t>(kF32Warps) * T * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_causal_f32, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  attn_causal_f32<<<grid, kF32Warps * 32, smem, stream>>>(qkv, out, T, n_head, score_scale);
  return cudaGetLastError();
}

}  // namespace gpt2
