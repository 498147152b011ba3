// Element-wise and row-wise kernels of the 16-bit backward (the products
// run on the tensor cores: gemm_grad.cu, attention_bwd_tc.cu), and the
// column sums every backward uses for bias, gamma and beta gradients.
//
// llm.c notes 5.2-5.3: the LayerNorm gradient couples the mean, the
// variance and the normalised value, and gamma and beta have gradients of
// their own (sums over rows); the GELU derivative multiplies the incoming
// gradient element by element.  "逐行拆GPT-2源码", GPT2Model: the embedding
// is wte[token] + wpe[position], so wte rows collect the gradient of every
// position that used the token and wpe rows that of every sequence.
//
// Every sum over rows runs in a fixed order (two levels: row chunks, then
// the chunks in order), so results do not depend on timing.
#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T> __device__ __forceinline__ float ld_f(const T* p) { return to_f32<T>(*p); }

// g = act(u): gelu_new (the hardware tanh, as the c_fc epilogue) or the
// exact GELU; 16-bit in and out, eight values per thread.
template <typename T16>
__global__ void gelu_fwd_16(const T16* __restrict__ u, T16* __restrict__ g, long long n8, int exact) {
  griddep_wait();
  griddep_launch_dependents();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint4 in = reinterpret_cast<const uint4*>(u)[i];
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = Type16<T16>::unpack2(w[e]);
    o[e] = exact ? Type16<T16>::pack2(gelu_exact(x.x), gelu_exact(x.y))
                 : Type16<T16>::pack2(gelu_new_fast(x.x), gelu_new_fast(x.y));
  }
  reinterpret_cast<uint4*>(g)[i] = make_uint4(o[0], o[1], o[2], o[3]);
}

// du = dg * act'(u): d/du of 0.5 u (1 + tanh(k (u + 0.044715 u^3))), or of
// u Phi(u) = Phi(u) + u phi(u).
__device__ __forceinline__ float gelu_grad(float x, int exact) {
  if (exact) {
    const float Phi = 0.5f * (1.f + erff(x * 0.7071067811865476f));
    return Phi + x * 0.3989422804014327f * expf(-0.5f * x * x);
  }
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float t = tanhf(k0 * fmaf(0.044715f * x, x * x, x));
  return 0.5f * (1.f + t) + 0.5f * x * (1.f - t * t) * k0 * fmaf(3.f * 0.044715f, x * x, 1.f);
}
template <typename T16>
__global__ void gelu_bwd_16(const T16* __restrict__ dg, const T16* __restrict__ u, T16* __restrict__ du, long long n8,
                            int exact) {
  griddep_wait();
  griddep_launch_dependents();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint4 xu = reinterpret_cast<const uint4*>(u)[i];
  const uint4 xg = reinterpret_cast<const uint4*>(dg)[i];
  const uint32_t wu[4] = {xu.x, xu.y, xu.z, xu.w}, wg[4] = {xg.x, xg.y, xg.z, xg.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = Type16<T16>::unpack2(wu[e]);
    const float2 d = Type16<T16>::unpack2(wg[e]);
    o[e] = Type16<T16>::pack2(d.x * gelu_grad(x.x, exact), d.y * gelu_grad(x.y, exact));
  }
  reinterpret_cast<uint4*>(du)[i] = make_uint4(o[0], o[1], o[2], o[3]);
}

// LayerNorm backward, one warp per row (the row is re-read from L1 between
// passes): with xhat = (x - mean) rstd and g = dy * gamma,
//   dx = rstd (g - mean(g) - xhat mean(g xhat)) (+ dres),
//   prod = dy * xhat (its column sums are dgamma; those of dy are dbeta).
// dx fp32; dx16 (nullable) the same rounded to 16 bits for the next GEMM.
template <typename T16>
__global__ void __launch_bounds__(256) ln_bwd_16(const float* __restrict__ dy, const float* __restrict__ x,
                                                 const T16* __restrict__ gamma, const float* __restrict__ dres,
                                                 float* __restrict__ dx, T16* __restrict__ dx16,
                                                 float* __restrict__ prod, long long rows, int D, float eps) {
  griddep_wait();
  griddep_launch_dependents();
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float* xr = x + r * D;
  const float* gr = dy + r * D;
  float s = 0.f;
  for (int c = lane; c < D; c += 32) s += xr[c];
  const float mean = warp_sum(s) / static_cast<float>(D);
  float q = 0.f;
  for (int c = lane; c < D; c += 32) {
    const float d = xr[c] - mean;
    q = fmaf(d, d, q);
  }
  const float rstd = rsqrtf(warp_sum(q) / static_cast<float>(D) + eps);
  float sg = 0.f, sgx = 0.f;
  for (int c = lane; c < D; c += 32) {
    const float xh = (xr[c] - mean) * rstd;
    const float g = gr[c] * to_f32<T16>(gamma[c]);
    sg += g;
    sgx = fmaf(g, xh, sgx);
  }
  const float mg = warp_sum(sg) / static_cast<float>(D);
  const float mgx = warp_sum(sgx) / static_cast<float>(D);
  for (int c = lane; c < D; c += 32) {
    const float xh = (xr[c] - mean) * rstd;
    const float dyv = gr[c];
    float v = rstd * (dyv * to_f32<T16>(gamma[c]) - mg - xh * mgx);
    if (dres) v += dres[r * D + c];
    dx[r * D + c] = v;
    if (dx16) dx16[r * D + c] = from_f32<T16>(v);
    prod[r * D + c] = dyv * xh;
  }
}

// The same with the row held in registers (NV groups of four columns per
// lane, 16-byte loads; groups past D/4 idle): x and dy are read once.
template <typename T16, int NV>
__global__ void __launch_bounds__(256) ln_bwd_16_reg(const float* __restrict__ dy, const float* __restrict__ x,
                                                     const T16* __restrict__ gamma, const float* __restrict__ dres,
                                                     float* __restrict__ dx, T16* __restrict__ dx16,
                                                     float* __restrict__ prod, long long rows, int D, float eps) {
  griddep_wait();
  griddep_launch_dependents();
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const int nvec = D >> 2;
  float4 xv[NV], gv[NV];
  float gm[NV][4];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int g = lane + 32 * i;
    if (g < nvec) {
      xv[i] = reinterpret_cast<const float4*>(x + r * D)[g];
      gv[i] = reinterpret_cast<const float4*>(dy + r * D)[g];
      const uint2 gw = reinterpret_cast<const uint2*>(gamma)[g];
      const float2 g01 = Type16<T16>::unpack2(gw.x), g23 = Type16<T16>::unpack2(gw.y);
      gm[i][0] = g01.x;
      gm[i][1] = g01.y;
      gm[i][2] = g23.x;
      gm[i][3] = g23.y;
    } else {
      xv[i] = gv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      gm[i][0] = gm[i][1] = gm[i][2] = gm[i][3] = 0.f;
    }
    s += (xv[i].x + xv[i].y) + (xv[i].z + xv[i].w);
  }
  const float mean = warp_sum(s) / static_cast<float>(D);
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    if (lane + 32 * i < nvec) {
      const float a = xv[i].x - mean, b = xv[i].y - mean, c = xv[i].z - mean, d = xv[i].w - mean;
      q = fmaf(a, a, fmaf(b, b, fmaf(c, c, fmaf(d, d, q))));
    }
  }
  const float rstd = rsqrtf(warp_sum(q) / static_cast<float>(D) + eps);
  float sg = 0.f, sgx = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const float xs[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w}, ds[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float g = ds[e] * gm[i][e];
      sg += g;
      sgx = fmaf(g, (xs[e] - mean) * rstd, sgx);
    }
  }
  const float mg = warp_sum(sg) / static_cast<float>(D);
  const float mgx = warp_sum(sgx) / static_cast<float>(D);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int g = lane + 32 * i;
    if (g >= nvec) continue;
    const float xs[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w}, ds[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
    float o[4], pr[4];
    const float4 rr = dres ? reinterpret_cast<const float4*>(dres + r * D)[g] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float rs[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float xh = (xs[e] - mean) * rstd;
      o[e] = rstd * (ds[e] * gm[i][e] - mg - xh * mgx) + rs[e];
      pr[e] = ds[e] * xh;
    }
    reinterpret_cast<float4*>(dx + r * D)[g] = make_float4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<float4*>(prod + r * D)[g] = make_float4(pr[0], pr[1], pr[2], pr[3]);
    if (dx16)
      reinterpret_cast<uint2*>(dx16 + r * D)[g] =
          make_uint2(Type16<T16>::pack2(o[0], o[1]), Type16<T16>::pack2(o[2], o[3]));
  }
}

// Column sums, level 1: block (column tile of 64, row chunk of kChunk rows):
// 4 groups of 64 threads take rows group, group + 4, ... of the chunk (16
// rows each, loaded together and added in a fixed tree), then the 4 group
// sums are added in order.  partial[chunk][col].
constexpr int kChunk = 64;
template <typename T>
__global__ void __launch_bounds__(256) colsum_partial(const T* __restrict__ in, long long M, int N, long long ld,
                                                      float* __restrict__ partial) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float part[4][64];
  const int col = blockIdx.x * 64 + (threadIdx.x & 63);
  const int grp = threadIdx.x >> 6;
  const long long r0 = static_cast<long long>(blockIdx.y) * kChunk + grp;
  float v[kChunk / 4];
#pragma unroll
  for (int i = 0; i < kChunk / 4; ++i) {
    const long long r = r0 + 4 * i;
    v[i] = (col < N && r < M) ? ld_f(in + r * ld + col) : 0.f;
  }
#pragma unroll
  for (int w = kChunk / 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) v[i] += v[i + w];
  part[grp][threadIdx.x & 63] = v[0];
  __syncthreads();
  if (grp == 0 && col < N)
    partial[static_cast<long long>(blockIdx.y) * N + col] = ((part[0][threadIdx.x] + part[1][threadIdx.x]) +
                                                             part[2][threadIdx.x]) + part[3][threadIdx.x];
}
// level 2: out[col] = sum of the chunks' partials in chunk order.
__global__ void colsum_final(const float* __restrict__ partial, int chunks, int N, float* __restrict__ out) {
  griddep_wait();
  griddep_launch_dependents();
  const int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= N) return;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  int c = 0;
  for (; c + 4 <= chunks; c += 4)
#pragma unroll
    for (int u = 0; u < 4; ++u) a[u] += partial[static_cast<long long>(c + u) * N + col];
  for (; c < chunks; ++c) a[0] += partial[static_cast<long long>(c) * N + col];
  out[col] = (a[0] + a[1]) + (a[2] + a[3]);
}

// dwte[token] += the gradient of every position that used the token: the
// warp of position m adds the rows of all positions with m's token, in
// increasing order, when m is the token's first position (so each row is
// written by one warp, in a fixed order).  Tokens out of range are skipped
// (the forward reported them).
__global__ void embed_bwd_wte(const int32_t* __restrict__ tokens, const float* __restrict__ dx0, float* dwte,
                              int M, int D, int V) {
  griddep_wait();
  griddep_launch_dependents();
  const int m = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (m >= M) return;
  const int tok = tokens[m];
  if (tok < 0 || tok >= V) return;
  // is m the first position with this token?
  bool first = true;
  for (int b = 0; b < m && first; b += 32) {
    const int i = b + lane;
    const bool same = i < m && tokens[i] == tok;
    first = !__any_sync(0xffffffffu, same);
  }
  if (!first) return;
  // this warp alone writes the row: add the positions m, ... with the token
  // in increasing order, 32 candidates per ballot
  float* out = dwte + static_cast<long long>(tok) * D;
  for (int b = m; b < M; b += 32) {
    const int i = b + lane;
    unsigned hit = __ballot_sync(0xffffffffu, i < M && tokens[i] == tok);
    while (hit) {
      const int p = b + __ffs(hit) - 1;
      hit &= hit - 1;
      const float* src = dx0 + static_cast<long long>(p) * D;
      for (int c = lane; c < D; c += 32) out[c] += src[c];
    }
  }
}

// dwpe[t] = sum over the batch of the position-t gradients (in batch order);
// rows t >= T are zero.
__global__ void embed_bwd_wpe(const float* __restrict__ dx0, float* __restrict__ dwpe, int B, int T, int D,
                              int n_pos) {
  griddep_wait();
  griddep_launch_dependents();
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(n_pos) * D) return;
  const int t = static_cast<int>(i / D), c = static_cast<int>(i % D);
  float s = 0.f;
  if (t < T)
    for (int b = 0; b < B; ++b) s += dx0[(static_cast<long long>(b) * T + t) * D + c];
  dwpe[i] = s;
}

unsigned blocks_for(long long n, int per) { return static_cast<unsigned>((n + per - 1) / per); }

}  // namespace

size_t colsum_partial_bytes(long long M, int N) { return static_cast<size_t>((M + kChunk - 1) / kChunk) * N * 4; }

cudaError_t launch_colsum(const void* in, bool in16, long long M, int N, long long ld, float* partial, float* out,
                          cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const int chunks = static_cast<int>((M + kChunk - 1) / kChunk);
  if (chunks == 0) return cudaMemsetAsync(out, 0, static_cast<size_t>(N) * 4, s);
  const dim3 grid((N + 63) / 64, chunks);
  cudaError_t e = in16 ? launch_pdl(colsum_partial<__nv_bfloat16>, grid, 256, 0, s, 0,
                                    static_cast<const __nv_bfloat16*>(in), M, N, ld, partial)
                       : launch_pdl(colsum_partial<float>, grid, 256, 0, s, 0, static_cast<const float*>(in), M, N,
                                    ld, partial);
  if (e != cudaSuccess) return e;
  return launch_pdl(colsum_final, dim3(blocks_for(N, 256)), 256, 0, s, 0, static_cast<const float*>(partial),
                    chunks, N, out);
}

cudaError_t launch_gelu_fwd_16(const void* u, void* g, long long n, bool exact, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return launch_pdl(gelu_fwd_16<__nv_bfloat16>, dim3(blocks_for(n / 8, 256)), 256, 0, s, 0,
                    static_cast<const __nv_bfloat16*>(u), static_cast<__nv_bfloat16*>(g), n / 8, exact ? 1 : 0);
}

cudaError_t launch_gelu_bwd_16(const void* dg, const void* u, void* du, long long n, bool exact, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return launch_pdl(gelu_bwd_16<__nv_bfloat16>, dim3(blocks_for(n / 8, 256)), 256, 0, s, 0,
                    static_cast<const __nv_bfloat16*>(dg), static_cast<const __nv_bfloat16*>(u),
                    static_cast<__nv_bfloat16*>(du), n / 8, exact ? 1 : 0);
}

template <int NV>
cudaError_t ln_bwd_reg(const float* dy, const float* x, const void* gamma, const float* dres, float* dx, void* dx16,
                       float* prod, long long rows, int D, float eps, cudaStream_t s) {
  return launch_pdl(ln_bwd_16_reg<__nv_bfloat16, NV>, dim3(blocks_for(rows, 8)), 256, 0, s, 0, dy, x,
                    static_cast<const __nv_bfloat16*>(gamma), dres, dx, static_cast<__nv_bfloat16*>(dx16), prod, rows,
                    D, eps);
}

cudaError_t launch_ln_bwd_16(const float* dy, const float* x, const void* gamma, const float* dres, float* dx,
                             void* dx16, float* prod, long long rows, int D, float eps, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  // the row in registers up to 13 float4 groups per lane (D <= 1664)
  const int nv = (D + 127) / 128;
  if (nv <= 2) return ln_bwd_reg<2>(dy, x, gamma, dres, dx, dx16, prod, rows, D, eps, s);
  if (nv <= 4) return ln_bwd_reg<4>(dy, x, gamma, dres, dx, dx16, prod, rows, D, eps, s);
  if (nv <= 6) return ln_bwd_reg<6>(dy, x, gamma, dres, dx, dx16, prod, rows, D, eps, s);
  if (nv <= 8) return ln_bwd_reg<8>(dy, x, gamma, dres, dx, dx16, prod, rows, D, eps, s);
  if (nv <= 13) return ln_bwd_reg<13>(dy, x, gamma, dres, dx, dx16, prod, rows, D, eps, s);
  return launch_pdl(ln_bwd_16<__nv_bfloat16>, dim3(blocks_for(rows, 8)), 256, 0, s, 0, dy, x,
                    static_cast<const __nv_bfloat16*>(gamma), dres, dx, static_cast<__nv_bfloat16*>(dx16), prod, rows,
                    D, eps);
}

cudaError_t launch_embed_bwd(const int32_t* tokens, const float* dx0, float* dwte, float* dwpe, int B, int T, int D,
                             int V, int n_pos, cudaStream_t s) {
  const int M = B * T;
  cudaError_t e = launch_pdl(embed_bwd_wte, dim3(blocks_for(M, 8)), 256, 0, s, 0, tokens, dx0, dwte, M, D, V);
  if (e != cudaSuccess) return e;
  return launch_pdl(embed_bwd_wpe, dim3(blocks_for(static_cast<long long>(n_pos) * D, 256)), 256, 0, s, 0, dx0,
                    dwpe, B, T, D, n_pos);
}

}  // namespace gpt2
