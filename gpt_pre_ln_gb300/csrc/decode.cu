// Kernels of the KV-cache decode step (bf16 path).
//
// "逐行拆GPT-2源码", GPT2Model / GPT2Attention: with past_key_values the
// new token's position is past_length; its k, v are concatenated after the
// cached ones along the sequence axis and its query attends over all of
// them.  Here the cache is a preallocated [L, 2, B, H, T_max, 64] bf16 arena
// and "concatenate" is a write into slot past_len[b].  The next token is the
// argmax of the tied lm_head scores (huaweicloud page, section 九), lowest
// index on ties.
//
// The attention over the cache reads every cached key and value once: it is
// bound by HBM bandwidth.
#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kHd = 64;
constexpr int kDecThreads = 256;  // 8 warps per (b, h)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per sequence: valid[b] = position and token in range;
// x = wte[token] + wpe[pos]; y = LN(x).
__global__ void decode_embed_ln(const int32_t* __restrict__ tokens, const int32_t* __restrict__ past_len,
                                const __nv_bfloat16* __restrict__ wte, const __nv_bfloat16* __restrict__ wpe,
                                const __nv_bfloat16* __restrict__ gamma, const __nv_bfloat16* __restrict__ beta,
                                float* __restrict__ x, __nv_bfloat16* __restrict__ y, int B, int D, int V, int n_pos,
                                int T_max, float eps, int* __restrict__ valid, unsigned* err) {
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  const int lane = threadIdx.x & 31;
  const int pos = past_len[b];
  const int tok = tokens[b];
  const bool pos_ok = pos >= 0 && pos < n_pos && pos < T_max;
  const bool tok_ok = tok >= 0 && tok < V;
  if (lane == 0) {
    valid[b] = (pos_ok && tok_ok) ? 1 : 0;
    if (!pos_ok) record_error(err, kErrRange, kSiteDecodePos);
    if (!tok_ok) record_error(err, kErrRange, kSiteDecodeToken);
  }
  const bool ok = pos_ok && tok_ok;
  const __nv_bfloat16* er = wte + static_cast<long long>(ok ? tok : 0) * D;
  const __nv_bfloat16* pr = wpe + static_cast<long long>(ok ? pos : 0) * D;
  float* xr = x + static_cast<long long>(b) * D;
  float s = 0.f;
  for (int c = lane; c < D; c += 32) {
    const float v = ok ? (__bfloat162float(er[c]) + __bfloat162float(pr[c])) : 0.f;
    xr[c] = v;
    s += v;
  }
  const float mean = warp_sum(s) / D;
  float q = 0.f;
  for (int c = lane; c < D; c += 32) {
    const float d = xr[c] - mean;
    q = fmaf(d, d, q);
  }
  const float rstd = rsqrtf(warp_sum(q) / D + eps);
  __nv_bfloat16* yr = y + static_cast<long long>(b) * D;
  for (int c = lane; c < D; c += 32)
    yr[c] = __float2bfloat16_rn((xr[c] - mean) * rstd * __bfloat162float(gamma[c]) + __bfloat162float(beta[c]));
}

// One CTA per (b, h): append k, v of the new token at slot pos, then
// out = softmax_j(q . k_j / 8) v_j over slots 0..pos.  Each warp takes a
// contiguous range of slots; within a warp 8 lanes share one key (16 bytes
// of the 128-byte row each), 4 keys per step; online softmax per lane group,
// merged across groups and warps at the end.
__global__ void __launch_bounds__(kDecThreads)
    decode_attn(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* kv_layer, __nv_bfloat16* __restrict__ out,
                const int32_t* __restrict__ past_len, const int* __restrict__ valid, int B, int H, int T_max) {
  __shared__ float s_m[kDecThreads / 8], s_l[kDecThreads / 8];
  __shared__ float s_acc[kDecThreads / 8][kHd];
  const int bh = blockIdx.x;
  const int b = bh / H;
  const int h = bh % H;
  const int D = H * kHd;
  const int tid = threadIdx.x;
  if (!valid[b]) {
    if (tid < kHd) out[static_cast<long long>(b) * D + h * kHd + tid] = __float2bfloat16_rn(0.f);
    return;
  }
  const int pos = past_len[b];
  const __nv_bfloat16* row = qkv + static_cast<long long>(b) * 3 * D;
  const long long kv_stride = static_cast<long long>(B) * H * T_max * kHd;  // K block -> V block
  __nv_bfloat16* kc = kv_layer + (static_cast<long long>(b) * H + h) * T_max * kHd;
  __nv_bfloat16* vc = kc + kv_stride;
  if (tid < kHd) {
    kc[static_cast<long long>(pos) * kHd + tid] = row[D + h * kHd + tid];
    vc[static_cast<long long>(pos) * kHd + tid] = row[2 * D + h * kHd + tid];
  }
  __syncthreads();  // the new slot is visible to the whole block

  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int grp = lane >> 3;  // key within the step
  const int sub = lane & 7;   // 16-byte chunk of the row
  float q[8];
  {
    uint4 u = *reinterpret_cast<const uint4*>(row + h * kHd + sub * 8);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = __bfloat1622float2(p[e]);
      q[2 * e] = f.x * 0.125f;  // fold 1/sqrt(64) into q
      q[2 * e + 1] = f.y * 0.125f;
    }
  }
  const int n_keys = pos + 1;
  const int per_warp = (n_keys + (kDecThreads / 32) - 1) / (kDecThreads / 32);
  const int j_begin = warp * per_warp;
  const int j_end = min(n_keys, j_begin + per_warp);
  float m = -1e30f, l = 0.f, acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  constexpr int kUnroll = 4;
  for (int j0 = j_begin; j0 < j_end; j0 += 4 * kUnroll) {
    uint4 kr[kUnroll], vr[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = j0 + u * 4 + grp;
      if (j < j_end) {
        kr[u] = *reinterpret_cast<const uint4*>(kc + static_cast<long long>(j) * kHd + sub * 8);
        vr[u] = *reinterpret_cast<const uint4*>(vc + static_cast<long long>(j) * kHd + sub * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = j0 + u * 4 + grp;
      const __nv_bfloat162* kp = reinterpret_cast<const __nv_bfloat162*>(&kr[u]);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(kp[e]);
        d = fmaf(q[2 * e], f.x, d);
        d = fmaf(q[2 * e + 1], f.y, d);
      }
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      d += __shfl_xor_sync(0xffffffffu, d, 4);
      if (j < j_end) {
        const float m_new = fmaxf(m, d);
        const float alpha = __expf(m - m_new);
        const float p = __expf(d - m_new);
        l = l * alpha + p;
        const __nv_bfloat162* vp = reinterpret_cast<const __nv_bfloat162*>(&vr[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f = __bfloat1622float2(vp[e]);
          acc[2 * e] = fmaf(p, f.x, acc[2 * e] * alpha);
          acc[2 * e + 1] = fmaf(p, f.y, acc[2 * e + 1] * alpha);
        }
        m = m_new;
      }
    }
  }
  // one partial (m, l, acc[64]) per lane group of 8
  const int g = tid >> 3;
  if (sub == 0) {
    s_m[g] = m;
    s_l[g] = l;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) s_acc[g][sub * 8 + e] = acc[e];
  __syncthreads();
  if (tid < kHd) {
    float M = -1e30f;
    for (int i = 0; i < kDecThreads / 8; ++i) M = fmaxf(M, s_m[i]);
    float L = 0.f, A = 0.f;
    for (int i = 0; i < kDecThreads / 8; ++i) {
      const float w = __expf(s_m[i] - M);
      L += s_l[i] * w;
      A += s_acc[i][tid] * w;
    }
    out[static_cast<long long>(b) * D + h * kHd + tid] = __float2bfloat16_rn(A / L);
  }
}

// One CTA per row: lowest index of the maximum; then past_len[b] += 1.
__global__ void __launch_bounds__(1024) argmax_rows(const float* __restrict__ logits, long long ld, int V,
                                                    const int* __restrict__ valid, int32_t* __restrict__ next_tokens,
                                                    int32_t* __restrict__ past_len) {
  __shared__ float s_v[32];
  __shared__ int s_i[32];
  const int b = blockIdx.x;
  const float* r = logits + static_cast<long long>(b) * ld;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = threadIdx.x; c < V; c += blockDim.x) {
    const float v = r[c];
    if (v > best) {  // strictly greater keeps the first (lowest) index per thread
      best = v;
      bi = c;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) {
      best = ov;
      bi = oi;
    }
  }
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    s_v[warp] = best;
    s_i[warp] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    best = s_v[0];
    bi = s_i[0];
    for (int w = 1; w < (blockDim.x >> 5); ++w)
      if (s_v[w] > best || (s_v[w] == best && s_i[w] < bi)) {
        best = s_v[w];
        bi = s_i[w];
      }
    if (valid[b]) {
      next_tokens[b] = bi;
      past_len[b] += 1;
    }
  }
}

}  // namespace

cudaError_t launch_decode_embed_ln(const int32_t* tokens, const int32_t* past_len, const __nv_bfloat16* wte,
                                   const __nv_bfloat16* wpe, const __nv_bfloat16* gamma, const __nv_bfloat16* beta,
                                   float* x, __nv_bfloat16* y, int B, int D, int V, int n_pos, int T_max, float eps,
                                   int* valid, cudaStream_t stream) {
  const int warps = 4;
  decode_embed_ln<<<(B + warps - 1) / warps, warps * 32, 0, stream>>>(tokens, past_len, wte, wpe, gamma, beta, x, y,
                                                                      B, D, V, n_pos, T_max, eps, valid,
                                                                      device_error_word());
  return cudaGetLastError();
}

cudaError_t launch_decode_attention(const __nv_bfloat16* qkv, __nv_bfloat16* kv_layer, __nv_bfloat16* out,
                                    const int32_t* past_len, const int* valid, int B, int n_head, int T_max,
                                    cudaStream_t stream) {
  decode_attn<<<B * n_head, kDecThreads, 0, stream>>>(qkv, kv_layer, out, past_len, valid, B, n_head, T_max);
  return cudaGetLastError();
}

cudaError_t launch_argmax_rows(const float* logits, int64_t ld, int B, int V, const int* valid, int32_t* next_tokens,
                               int32_t* past_len, cudaStream_t stream) {
  argmax_rows<<<B, 1024, 0, stream>>>(logits, ld, V, valid, next_tokens, past_len);
  return cudaGetLastError();
}

}  // namespace gpt2
