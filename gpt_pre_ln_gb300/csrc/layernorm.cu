// LayerNorm over the last axis, one warp per row, and the embedding
// (wte[token] + wpe[position]) fused with the first LayerNorm.
//
//   LN(x) = gamma * (x - mean) / sqrt(var + eps) + beta,  var = mean((x-mean)^2)
//
// ("Hidden State 如何流过 GPT-2 Block", section "Pre-Norm"; llm.c notes
// section 3.2: mean first, then the variance, eps inside the square root.)
// The row stays in registers between the two passes, so x is read once and
// y written once: the kernel is bound by HBM (or L2) bandwidth.
#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kLnThreads = 128;  // 4 rows per block

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  float4 f = *reinterpret_cast<const float4*>(p);
  v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.x));
  float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}

template <>
__device__ __forceinline__ void load4<__half>(const __half* p, float (&v)[4]) {
  uint2 u = *reinterpret_cast<const uint2*>(p);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&u.x));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}

template <typename T>
__device__ __forceinline__ void store4(T* p, const float (&v)[4]);
template <>
__device__ __forceinline__ void store4<float>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[4]) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

template <>
__device__ __forceinline__ void store4<__half>(__half* p, const float (&v)[4]) {
  __half2 a = __floats2half2_rn(v[0], v[1]);
  __half2 b = __floats2half2_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// gamma / beta for 4 consecutive columns, kept in their storage type until
// use (bf16: 8 bytes) so that preloading them costs few registers.
template <typename T> struct Raw4;
template <> struct Raw4<float> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ float get(int e) const { return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w; }
};
template <> struct Raw4<__nv_bfloat16> {
  uint2 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ float get(int e) const {
    const uint32_t w = e < 2 ? v.x : v.y;
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};

template <> struct Raw4<__half> {
  uint2 v;
  __device__ __forceinline__ void load(const __half* p) { v = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ float get(int e) const {
    const uint32_t w = e < 2 ? v.x : v.y;
    const unsigned short h = (e & 1) ? static_cast<unsigned short>(w >> 16) : static_cast<unsigned short>(w & 0xffffu);
    return __half2float(__ushort_as_half(h));
  }
};

// Normalises the row held in v (NV groups of 4 per lane, lane-strided) and
// writes it to yr.  Groups beyond D/4 hold zeros and are skipped.  gamma and
// beta (ln_load_affine) are loaded first, before the kernel's dependency
// wait, so that their latency overlaps the previous kernel.
template <typename YT, int NV>
__device__ __forceinline__ void ln_load_affine(int lane, int D, const YT* gamma, const YT* beta, Raw4<YT> (&g)[NV],
                                               Raw4<YT> (&bb)[NV]) {
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = (lane + i * 32) * 4;
    if (c < D) {
      g[i].load(gamma + c);
      bb[i].load(beta + c);
    }
  }
}

template <typename YT, int NV>
__device__ __forceinline__ void ln_finish(float (&v)[NV][4], int lane, int D, float eps, const Raw4<YT> (&g)[NV],
                                          const Raw4<YT> (&bb)[NV], YT* yr) {
  const int nvec = D >> 2;
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) s += (v[i][0] + v[i][1]) + (v[i][2] + v[i][3]);
  const float mean = warp_sum(s) / static_cast<float>(D);
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    if (lane + i * 32 < nvec) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float d = v[i][e] - mean;
        q = fmaf(d, d, q);
      }
    }
  }
  const float var = warp_sum(q) / static_cast<float>(D);
  const float rstd = rsqrtf(var + eps);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int c = (lane + i * 32) * 4;
    if (c < D) {
      float o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = fmaf((v[i][e] - mean) * rstd, g[i].get(e), bb[i].get(e));
      store4<YT>(yr + c, o);
    }
  }
}

template <typename XT, typename YT, int NV>
__global__ void __launch_bounds__(kLnThreads) layernorm_rows(const XT* __restrict__ x, const YT* __restrict__ gamma,
                                                             const YT* __restrict__ beta, YT* __restrict__ y,
                                                             long long rows, int D, float eps) {
  const long long row = static_cast<long long>(blockIdx.x) * (kLnThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  Raw4<YT> g[NV], bb[NV];
  ln_load_affine<YT, NV>(lane, D, gamma, beta, g, bb);
  griddep_wait();
  griddep_launch_dependents();
  if (row >= rows) return;
  const XT* xr = x + row * D;
  const int nvec = D >> 2;
  float v[NV][4];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = lane + i * 32;
    if (idx < nvec) {
      load4<XT>(xr + idx * 4, v[i]);
    } else {
      v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.f;
    }
  }
  ln_finish<YT, NV>(v, lane, D, eps, g, bb, y + row * D);
}

// x[m] = wte[tokens[m]] + wpe[m % T]; y[m] = LN(x[m]).  A token id outside
// [0, V) records GPT2_ERR_RANGE and contributes a zero embedding row.
template <typename WT, int NV>
__global__ void __launch_bounds__(kLnThreads)
    embed_ln_rows(const int32_t* __restrict__ tokens, const WT* __restrict__ wte, const WT* __restrict__ wpe,
                  const WT* __restrict__ gamma, const WT* __restrict__ beta, float* __restrict__ x,
                  WT* __restrict__ y, long long rows, int T, int D, int V, float eps, unsigned* err) {
  const long long row = static_cast<long long>(blockIdx.x) * (kLnThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  Raw4<WT> g[NV], bb[NV];
  ln_load_affine<WT, NV>(lane, D, gamma, beta, g, bb);
  griddep_wait();
  griddep_launch_dependents();
  if (row >= rows) return;
  const int pos = static_cast<int>(row % T);
  int tok = tokens[row];
  const bool tok_ok = tok >= 0 && tok < V;
  if (!tok_ok) {
    if (lane == 0) record_error(err, kErrRange, kSiteEmbedToken);
    tok = 0;
  }
  const WT* er = wte + static_cast<long long>(tok) * D;
  const WT* pr = wpe + static_cast<long long>(pos) * D;
  float* xr = x + row * D;
  const int nvec = D >> 2;
  float v[NV][4];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = lane + i * 32;
    if (idx < nvec) {
      float a[4], b[4];
      load4<WT>(er + idx * 4, a);
      load4<WT>(pr + idx * 4, b);
#pragma unroll
      for (int e = 0; e < 4; ++e) v[i][e] = (tok_ok ? a[e] : 0.f) + b[e];
      store4<float>(xr + idx * 4, v[i]);
    } else {
      v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.f;
    }
  }
  ln_finish<WT, NV>(v, lane, D, eps, g, bb, y + row * D);
}

template <typename XT, typename YT>
cudaError_t ln_dispatch(const void* x, const void* g, const void* b, void* y, long long rows, int D, float eps,
                        cudaStream_t s) {
  const unsigned blocks = static_cast<unsigned>((rows + kLnThreads / 32 - 1) / (kLnThreads / 32));
  auto X = static_cast<const XT*>(x);
  auto G = static_cast<const YT*>(g);
  auto Bt = static_cast<const YT*>(b);
  auto Y = static_cast<YT*>(y);
  if (D <= 512)
    return launch_pdl(layernorm_rows<XT, YT, 4>, blocks, kLnThreads, 0, s, 0, X, G, Bt, Y, rows, D, eps);
  else if (D <= 768)
    return launch_pdl(layernorm_rows<XT, YT, 6>, blocks, kLnThreads, 0, s, 0, X, G, Bt, Y, rows, D, eps);
  else if (D <= 1024)
    return launch_pdl(layernorm_rows<XT, YT, 8>, blocks, kLnThreads, 0, s, 0, X, G, Bt, Y, rows, D, eps);
  else if (D <= 1664)
    return launch_pdl(layernorm_rows<XT, YT, 13>, blocks, kLnThreads, 0, s, 0, X, G, Bt, Y, rows, D, eps);
  else if (D <= 2048)
    return launch_pdl(layernorm_rows<XT, YT, 16>, blocks, kLnThreads, 0, s, 0, X, G, Bt, Y, rows, D, eps);
  else
    return launch_pdl(layernorm_rows<XT, YT, 32>, blocks, kLnThreads, 0, s, 0, X, G, Bt, Y, rows, D, eps);
  return cudaGetLastError();
}

template <typename WT>
cudaError_t embed_dispatch(const int32_t* tokens, const void* wte, const void* wpe, const void* g, const void* b,
                           float* x, void* y, long long rows, int T, int D, int V, float eps, cudaStream_t s) {
  const unsigned blocks = static_cast<unsigned>((rows + kLnThreads / 32 - 1) / (kLnThreads / 32));
  auto E = static_cast<const WT*>(wte);
  auto P = static_cast<const WT*>(wpe);
  auto G = static_cast<const WT*>(g);
  auto Bt = static_cast<const WT*>(b);
  auto Y = static_cast<WT*>(y);
  unsigned* err = device_error_word();
  if (D <= 512)
    return launch_pdl(embed_ln_rows<WT, 4>, blocks, kLnThreads, 0, s, 0, tokens, E, P, G, Bt, x, Y, rows, T, D,
                      V, eps, err);
  else if (D <= 768)
    return launch_pdl(embed_ln_rows<WT, 6>, blocks, kLnThreads, 0, s, 0, tokens, E, P, G, Bt, x, Y, rows, T, D,
                      V, eps, err);
  else if (D <= 1024)
    return launch_pdl(embed_ln_rows<WT, 8>, blocks, kLnThreads, 0, s, 0, tokens, E, P, G, Bt, x, Y, rows, T, D,
                      V, eps, err);
  else if (D <= 2048)
    return launch_pdl(embed_ln_rows<WT, 16>, blocks, kLnThreads, 0, s, 0, tokens, E, P, G, Bt, x, Y, rows, T, D,
                      V, eps, err);
  else
    return launch_pdl(embed_ln_rows<WT, 32>, blocks, kLnThreads, 0, s, 0, tokens, E, P, G, Bt, x, Y, rows, T, D,
                      V, eps, err);
  return cudaGetLastError();
}

template <typename XT>
cudaError_t ln_by_y(const void* x, const void* g, const void* b, void* y, long long rows, int D, float eps,
                    gpt2_dtype y_t, cudaStream_t s) {
  if (y_t == GPT2_F32) return ln_dispatch<XT, float>(x, g, b, y, rows, D, eps, s);
  if (y_t == GPT2_F16) return ln_dispatch<XT, __half>(x, g, b, y, rows, D, eps, s);
  return ln_dispatch<XT, __nv_bfloat16>(x, g, b, y, rows, D, eps, s);
}

}  // namespace

cudaError_t launch_layernorm(const void* x, const void* gamma, const void* beta, void* y, int64_t rows, int D,
                             float eps, gpt2_dtype x_t, gpt2_dtype y_t, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (x_t == GPT2_F32) return ln_by_y<float>(x, gamma, beta, y, rows, D, eps, y_t, stream);
  if (x_t == GPT2_F16) return ln_by_y<__half>(x, gamma, beta, y, rows, D, eps, y_t, stream);
  return ln_by_y<__nv_bfloat16>(x, gamma, beta, y, rows, D, eps, y_t, stream);
}

cudaError_t launch_embed_ln(const int32_t* tokens, const void* wte, const void* wpe, const void* gamma,
                            const void* beta, float* x, void* y, int B, int T, int D, int V, float eps, gpt2_dtype dt,
                            cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * T;
  if (rows == 0) return cudaSuccess;
  if (dt == GPT2_F32) return embed_dispatch<float>(tokens, wte, wpe, gamma, beta, x, y, rows, T, D, V, eps, stream);
  if (dt == GPT2_F16) return embed_dispatch<__half>(tokens, wte, wpe, gamma, beta, x, y, rows, T, D, V, eps, stream);
  return embed_dispatch<__nv_bfloat16>(tokens, wte, wpe, gamma, beta, x, y, rows, T, D, V, eps, stream);
}

}  // namespace gpt2
