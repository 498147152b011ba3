// Kernels of the KV-cache decode step (16-bit paths: bf16 or fp16 storage).
//
// "逐行拆GPT-2源码", GPT2Model / GPT2Attention: with past_key_values the
// new token's position is past_length; its k, v are concatenated after the
// cached ones along the sequence axis and its query attends over all of
// them.  Here the cache is a preallocated [L, 2, B, H, T_max, 64] 16-bit arena
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
template <typename T16>
__global__ void decode_embed_ln(const int32_t* __restrict__ tokens, const int32_t* __restrict__ past_len,
                                const T16* __restrict__ wte, const T16* __restrict__ wpe,
                                const T16* __restrict__ gamma, const T16* __restrict__ beta, float* __restrict__ x,
                                T16* __restrict__ y, int B, int D, int V, int n_pos, int T_max, float eps,
                                int* __restrict__ valid, unsigned* err) {
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
  const T16* er = wte + static_cast<long long>(ok ? tok : 0) * D;
  const T16* pr = wpe + static_cast<long long>(ok ? pos : 0) * D;
  float* xr = x + static_cast<long long>(b) * D;
  float s = 0.f;
  for (int c = lane; c < D; c += 32) {
    const float v = ok ? (to_f32<T16>(er[c]) + to_f32<T16>(pr[c])) : 0.f;
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
  T16* yr = y + static_cast<long long>(b) * D;
  for (int c = lane; c < D; c += 32)
    yr[c] = from_f32<T16>((xr[c] - mean) * rstd * to_f32<T16>(gamma[c]) + to_f32<T16>(beta[c]));
}

// One CTA per (b, h): append k, v of the new token at slot pos, then
// out = softmax_j(q . k_j / 8) v_j over slots 0..pos.  Each warp takes a
// contiguous range of slots; within a warp 8 lanes share one key (16 bytes
// of the 128-byte row each), 4 keys per step; online softmax per lane group,
// merged across groups and warps at the end.
template <typename T16>
__global__ void __launch_bounds__(kDecThreads)
    decode_attn(const T16* __restrict__ qkv, T16* kv_layer, T16* __restrict__ out,
                const int32_t* __restrict__ past_len, const int* __restrict__ valid, int B, int H, int T_max) {
  __shared__ float s_m[kDecThreads / 8], s_l[kDecThreads / 8];
  __shared__ float s_acc[kDecThreads / 8][kHd];
  const int bh = blockIdx.x;
  const int b = bh / H;
  const int h = bh % H;
  const int D = H * kHd;
  const int tid = threadIdx.x;
  if (!valid[b]) {
    if (tid < kHd) out[static_cast<long long>(b) * D + h * kHd + tid] = from_f32<T16>(0.f);
    return;
  }
  const int pos = past_len[b];
  const T16* row = qkv + static_cast<long long>(b) * 3 * D;
  const long long kv_stride = static_cast<long long>(B) * H * T_max * kHd;  // K block -> V block
  T16* kc = kv_layer + (static_cast<long long>(b) * H + h) * T_max * kHd;
  T16* vc = kc + kv_stride;
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
    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = Type16<T16>::unpack2(uw[e]);
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
      kr[u] = vr[u] = make_uint4(0u, 0u, 0u, 0u);
      if (j < j_end) {
        kr[u] = *reinterpret_cast<const uint4*>(kc + static_cast<long long>(j) * kHd + sub * 8);
        vr[u] = *reinterpret_cast<const uint4*>(vc + static_cast<long long>(j) * kHd + sub * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = j0 + u * 4 + grp;
      const uint32_t kw[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 f = Type16<T16>::unpack2(kw[e]);
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
        const uint32_t vw[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f = Type16<T16>::unpack2(vw[e]);
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
    out[static_cast<long long>(b) * D + h * kHd + tid] = from_f32<T16>(A / L);
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

cudaError_t launch_decode_embed_ln(gpt2_dtype dt, const int32_t* tokens, const int32_t* past_len, const void* wte,
                                   const void* wpe, const void* gamma, const void* beta, float* x, void* y, int B,
                                   int D, int V, int n_pos, int T_max, float eps, int* valid, cudaStream_t stream) {
  const int warps = 4;
  const dim3 grid((B + warps - 1) / warps), block(warps * 32);
  unsigned* err = device_error_word();
  if (dt == GPT2_F16) {
    using T = __half;
    decode_embed_ln<T><<<grid, block, 0, stream>>>(tokens, past_len, static_cast<const T*>(wte),
                                                   static_cast<const T*>(wpe), static_cast<const T*>(gamma),
                                                   static_cast<const T*>(beta), x, static_cast<T*>(y), B, D, V, n_pos,
                                                   T_max, eps, valid, err);
  } else {
    using T = __nv_bfloat16;
    decode_embed_ln<T><<<grid, block, 0, stream>>>(tokens, past_len, static_cast<const T*>(wte),
                                                   static_cast<const T*>(wpe), static_cast<const T*>(gamma),
                                                   static_cast<const T*>(beta), x, static_cast<T*>(y), B, D, V, n_pos,
                                                   T_max, eps, valid, err);
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_attention(gpt2_dtype dt, const void* qkv, void* kv_layer, void* out, const int32_t* past_len,
                                    const int* valid, int B, int n_head, int T_max, cudaStream_t stream) {
  if (dt == GPT2_F16) {
    using T = __half;
    decode_attn<T><<<B * n_head, kDecThreads, 0, stream>>>(static_cast<const T*>(qkv), static_cast<T*>(kv_layer),
                                                           static_cast<T*>(out), past_len, valid, B, n_head, T_max);
  } else {
    using T = __nv_bfloat16;
    decode_attn<T><<<B * n_head, kDecThreads, 0, stream>>>(static_cast<const T*>(qkv), static_cast<T*>(kv_layer),
                                                           static_cast<T*>(out), past_len, valid, B, n_head, T_max);
  }
  return cudaGetLastError();
}

cudaError_t launch_argmax_rows(const float* logits, int64_t ld, int B, int V, const int* valid, int32_t* next_tokens,
                               int32_t* past_len, cudaStream_t stream) {
  argmax_rows<<<B, 1024, 0, stream>>>(logits, ld, V, valid, next_tokens, past_len);
  return cudaGetLastError();
}

}  // namespace gpt2
