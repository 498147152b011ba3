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

// act'(u): d/du of 0.5 u (1 + tanh(k (u + 0.044715 u^3))), or of u Phi(u)
// = Phi(u) + u phi(u).
__device__ __forceinline__ float gelu_grad(float x, int exact) {
  if (exact) {
    const float Phi = 0.5f * (1.f + erff(x * 0.7071067811865476f));
    return Phi + x * 0.3989422804014327f * expf(-0.5f * x * x);
  }
  // tanh(v) = 1 - 2 / (1 + e^(2v)) on the hardware exp2 and reciprocal
  // (absolute error about 1e-7; saturates for large |v|)
  const float k0 = 0.7978845608028654f;         // sqrt(2/pi)
  const float two_log2e = 2.8853900817779268f;  // 2 / ln(2)
  const float t = fmaf(-2.f, rcp_approx(1.f + ex2_approx(two_log2e * k0 * fmaf(0.044715f * x, x * x, x))), 1.f);
  return 0.5f * (1.f + t) + 0.5f * x * (1.f - t * t) * k0 * fmaf(3.f * 0.044715f, x * x, 1.f);
}
// LayerNorm backward for rows too wide for registers, one warp per row (the
// row is re-read from L1 between passes): with xhat = (x - mean) rstd and g = dy * gamma,
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

// Column sums, level 1: a block of 8 warps sums a chunk of kChunk rows over
// 32 x VEC columns (VEC columns of 16 bytes per lane: warp loads are whole
// 512-byte row segments); warp w takes rows w, w + 8, ... of the chunk (all
// its loads in flight together, added in a fixed tree), then the 8 warp sums
// are added in warp order.  partial[chunk][col].
constexpr int kChunk = 64;
template <typename T, int VEC>
__global__ void __launch_bounds__(256) colsum_partial(const T* __restrict__ in, long long M, int N, long long ld,
                                                      float* __restrict__ partial) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8][32 * VEC];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = (blockIdx.x * 32 + lane) * VEC;
  const long long r0 = static_cast<long long>(blockIdx.y) * kChunk + warp;
  constexpr int R = kChunk / 8;
  float v[R][VEC];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const long long r = r0 + 8 * i;
    const T* src = in + r * ld + c0;
    if (r < M && c0 + VEC <= N) {
      if constexpr (VEC == 1) {
        v[i][0] = ld_f(src);
      } else if constexpr (sizeof(T) == 4) {
        const float4 q = *reinterpret_cast<const float4*>(src);
        v[i][0] = q.x;
        v[i][1] = q.y;
        v[i][2] = q.z;
        v[i][3] = q.w;
      } else {
        const uint4 q = *reinterpret_cast<const uint4*>(src);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = Type16<T>::unpack2(w[e]);
          v[i][2 * e] = f.x;
          v[i][2 * e + 1] = f.y;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) v[i][e] = (r < M && c0 + e < N) ? ld_f(src + e) : 0.f;
    }
  }
#pragma unroll
  for (int w = R / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i)
#pragma unroll
      for (int e = 0; e < VEC; ++e) v[i][e] += v[i + w][e];
#pragma unroll
  for (int e = 0; e < VEC; ++e) red[warp][lane * VEC + e] = v[0][e];
  __syncthreads();
  for (int t = threadIdx.x; t < 32 * VEC; t += 256) {
    const int col = blockIdx.x * 32 * VEC + t;
    float s = red[0][t];
#pragma unroll
    for (int w = 1; w < 8; ++w) s += red[w][t];
    if (col < N) partial[static_cast<long long>(blockIdx.y) * N + col] = s;
  }
}

// Level 2: column c of partial [rows, N] summed over the rows in a fixed
// order: warp w of 32 takes rows w, w + 32, ... in batches of 16 (then 4,
// then single rows) whose loads are all in flight together and whose values
// are added in a fixed tree; then the 32 warp sums in warp order.  The
// result goes to out_q[c - q seg] for q = c / seg (three outputs at most; a
// null output is skipped).
__global__ void __launch_bounds__(1024) colsum_final(const float* __restrict__ partial, int rows, int N, int seg,
                                                     float* __restrict__ out0, float* __restrict__ out1,
                                                     float* __restrict__ out2) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[32][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = blockIdx.x * 32 + lane;
  float acc = 0.f;
  if (col < N) {
    const float* p = partial + col;
    int r = warp;
    for (; r + 15 * 32 < rows; r += 16 * 32) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = p[static_cast<long long>(r + 32 * i) * N];
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) v[i] += v[i + w];
      acc += v[0];
    }
    for (; r + 3 * 32 < rows; r += 4 * 32) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = p[static_cast<long long>(r + 32 * i) * N];
      acc += (v[0] + v[2]) + (v[1] + v[3]);
    }
    for (; r < rows; r += 32) acc += p[static_cast<long long>(r) * N];
  }
  red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && col < N) {
    float s = red[0][lane];
    for (int w = 1; w < 32; ++w) s += red[w][lane];
    const int q = col / seg;
    float* o = q == 0 ? out0 : (q == 1 ? out1 : out2);
    if (o) o[col - q * seg] = s;
  }
}

// LayerNorm backward with its column sums: one warp per row with the row in
// registers (NV groups of four columns per lane, 16-byte loads; x and dy are
// read once), 16 rows per block, and no per-row product written out.  The
// block adds up, over its rows and in warp order, dy * xhat (the gamma
// gradient), dy (beta) and dx (the bias gradient of the residual branch that
// produced the LayerNorm's input), through a shared [16][D] buffer one
// quantity at a time: partial[block][q][D].
constexpr int kLnColsWarps = 16;
template <typename T16, int NV>
__global__ void __launch_bounds__(kLnColsWarps * 32) ln_bwd_cols(const float* __restrict__ dy,
                                                                const float* __restrict__ x,
                                                                const T16* __restrict__ gamma,
                                                                const float* __restrict__ dres, float* __restrict__ dx,
                                                                T16* __restrict__ dx16, float* __restrict__ partial,
                                                                long long rows, int D, float eps) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ float red[];  // [kLnColsWarps][D]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kLnColsWarps + warp;
  const bool valid = r < rows;
  const int nvec = D >> 2;
  float4 xv[NV], gv[NV];
  float gm[NV][4];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int g = lane + 32 * i;
    if (valid && g < nvec) {
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
  // xv becomes dy * xhat, gm becomes dx (zero in rows past the end)
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int g = lane + 32 * i;
    float xs[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
    const float ds[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
    const float4 rr = (valid && dres && g < nvec) ? reinterpret_cast<const float4*>(dres + r * D)[g]
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    const float rs[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float xh = (xs[e] - mean) * rstd;
      gm[i][e] = valid ? rstd * (ds[e] * gm[i][e] - mg - xh * mgx) + rs[e] : 0.f;
      xs[e] = ds[e] * xh;
    }
    xv[i] = make_float4(xs[0], xs[1], xs[2], xs[3]);
    if (valid && g < nvec) {
      reinterpret_cast<float4*>(dx + r * D)[g] = make_float4(gm[i][0], gm[i][1], gm[i][2], gm[i][3]);
      if (dx16)
        reinterpret_cast<uint2*>(dx16 + r * D)[g] =
            make_uint2(Type16<T16>::pack2(gm[i][0], gm[i][1]), Type16<T16>::pack2(gm[i][2], gm[i][3]));
    }
  }
  float* out = partial + static_cast<long long>(blockIdx.x) * 3 * D;
#pragma unroll
  for (int qn = 0; qn < 3; ++qn) {
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int g = lane + 32 * i;
      if (g < nvec) {
        const float4 v = qn == 0 ? xv[i] : (qn == 1 ? gv[i] : make_float4(gm[i][0], gm[i][1], gm[i][2], gm[i][3]));
        reinterpret_cast<float4*>(red + warp * D)[g] = v;
      }
    }
    __syncthreads();
    for (int c = threadIdx.x; c < D; c += kLnColsWarps * 32) {
      float t = red[c];
#pragma unroll
      for (int w = 1; w < kLnColsWarps; ++w) t += red[w * D + c];
      out[qn * D + c] = t;
    }
    __syncthreads();
  }
}

// du = dg * act'(u) with the column sums of du (the c_fc bias gradient):
// block = 8 warps over a chunk of kChunk rows and 256 columns (8 per lane,
// 16-byte loads); warp w takes rows w, w + 8, ...; the 8 warp sums are added
// in warp order.  partial[chunk][col].  F a multiple of 8.
template <typename T16>
__global__ void __launch_bounds__(256) gelu_bwd_cols(const T16* __restrict__ dg, const T16* __restrict__ u,
                                                     T16* __restrict__ du, long long M, int F, int exact,
                                                     float* __restrict__ partial) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float red[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c0 = blockIdx.x * 256 + lane * 8;
  const long long r0 = static_cast<long long>(blockIdx.y) * kChunk + warp;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if (c0 < F) {
#pragma unroll 4
    for (int i = 0; i < kChunk / 8; ++i) {
      const long long r = r0 + 8 * i;
      if (r >= M) break;
      const long long off = (r * F + c0) / 8;
      const uint4 xu = reinterpret_cast<const uint4*>(u)[off];
      const uint4 xg = reinterpret_cast<const uint4*>(dg)[off];
      const uint32_t wu[4] = {xu.x, xu.y, xu.z, xu.w}, wg[4] = {xg.x, xg.y, xg.z, xg.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 xx = Type16<T16>::unpack2(wu[e]);
        const float2 d = Type16<T16>::unpack2(wg[e]);
        const float a = d.x * gelu_grad(xx.x, exact), b = d.y * gelu_grad(xx.y, exact);
        acc[2 * e] += a;
        acc[2 * e + 1] += b;
        o[e] = Type16<T16>::pack2(a, b);
      }
      reinterpret_cast<uint4*>(du)[off] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) red[warp][lane * 8 + e] = acc[e];
  __syncthreads();
  const int col = blockIdx.x * 256 + threadIdx.x;
  float s = red[0][threadIdx.x];
#pragma unroll
  for (int w = 1; w < 8; ++w) s += red[w][threadIdx.x];
  if (col < F) partial[static_cast<long long>(blockIdx.y) * F + col] = s;
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

namespace {

cudaError_t colsum_finish(const float* partial, int rows, int N, int seg, float* o0, float* o1, float* o2,
                          cudaStream_t s) {
  return launch_pdl(colsum_final, dim3(blocks_for(N, 32)), 1024, 0, s, 0, partial, rows, N, seg, o0, o1, o2);
}

template <typename T>
cudaError_t colsum_level1(const T* in, long long M, int N, long long ld, float* partial, cudaStream_t s) {
  constexpr int VEC = 16 / sizeof(T);
  const unsigned chunks = static_cast<unsigned>((M + kChunk - 1) / kChunk);
  const bool vec_ok = (reinterpret_cast<uintptr_t>(in) & 15u) == 0 && ld % VEC == 0;
  if (vec_ok)
    return launch_pdl(colsum_partial<T, VEC>, dim3(blocks_for(N, 32 * VEC), chunks), 256, 0, s, 0, in, M, N, ld,
                      partial);
  return launch_pdl(colsum_partial<T, 1>, dim3(blocks_for(N, 32), chunks), 256, 0, s, 0, in, M, N, ld, partial);
}

}  // namespace

cudaError_t launch_colsum(const void* in, bool in16, long long M, int N, long long ld, float* partial, float* out,
                          cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  const int chunks = static_cast<int>((M + kChunk - 1) / kChunk);
  if (chunks == 0) return cudaMemsetAsync(out, 0, static_cast<size_t>(N) * 4, s);
  cudaError_t e = in16 ? colsum_level1(static_cast<const __nv_bfloat16*>(in), M, N, ld, partial, s)
                       : colsum_level1(static_cast<const float*>(in), M, N, ld, partial, s);
  if (e != cudaSuccess) return e;
  return colsum_finish(partial, chunks, N, N, out, nullptr, nullptr, s);
}

cudaError_t launch_gelu_fwd_16(const void* u, void* g, long long n, bool exact, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  return launch_pdl(gelu_fwd_16<__nv_bfloat16>, dim3(blocks_for(n / 8, 256)), 256, 0, s, 0,
                    static_cast<const __nv_bfloat16*>(u), static_cast<__nv_bfloat16*>(g), n / 8, exact ? 1 : 0);
}

cudaError_t launch_gelu_bwd_sums_16(const void* dg, const void* u, void* du, long long M, int F, bool exact,
                                    float* dbias, float* scratch, cudaStream_t s) {
  if (F == 0) return cudaSuccess;
  const int chunks = static_cast<int>((M + kChunk - 1) / kChunk);
  if (chunks == 0) return cudaMemsetAsync(dbias, 0, static_cast<size_t>(F) * 4, s);
  cudaError_t e = launch_pdl(gelu_bwd_cols<__nv_bfloat16>, dim3(blocks_for(F, 256), chunks), 256, 0, s, 0,
                             static_cast<const __nv_bfloat16*>(dg), static_cast<const __nv_bfloat16*>(u),
                             static_cast<__nv_bfloat16*>(du), M, F, exact ? 1 : 0, scratch);
  if (e != cudaSuccess) return e;
  return colsum_finish(scratch, chunks, F, F, dbias, nullptr, nullptr, s);
}

namespace {

// the row in registers up to 13 float4 groups per lane (D <= 1664)
constexpr int kLnRegMaxD = 13 * 128;

template <int NV>
cudaError_t ln_bwd_cols_launch(const float* dy, const float* x, const void* gamma, const float* dres, float* dx,
                               void* dx16, float* partial, long long rows, int D, float eps, cudaStream_t s) {
  auto kern = ln_bwd_cols<__nv_bfloat16, NV>;
  const int smem = kLnColsWarps * D * 4;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLnColsWarps * kLnRegMaxD * 4);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return launch_pdl(kern, dim3(blocks_for(rows, kLnColsWarps)), kLnColsWarps * 32, smem, s, 0, dy, x,
                    static_cast<const __nv_bfloat16*>(gamma), dres, dx, static_cast<__nv_bfloat16*>(dx16), partial,
                    rows, D, eps);
}

}  // namespace

size_t ln_bwd_scratch_bytes(long long M, int D) {
  if (D <= kLnRegMaxD) return static_cast<size_t>((M + kLnColsWarps - 1) / kLnColsWarps) * 3 * D * 4;
  // wide rows: the per-row product dy * xhat, then the generic column sums
  return static_cast<size_t>(M) * D * 4 + colsum_partial_bytes(M, D);
}

cudaError_t launch_ln_bwd_sums_16(const float* dy, const float* x, const void* gamma, const float* dres, float* dx,
                                  void* dx16, float* dgamma, float* dbeta, float* dbias, long long rows, int D,
                                  float eps, float* scratch, cudaStream_t s) {
  if (rows == 0) {
    cudaError_t e = cudaMemsetAsync(dgamma, 0, static_cast<size_t>(D) * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, static_cast<size_t>(D) * 4, s);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, static_cast<size_t>(D) * 4, s);
    return e;
  }
  const int nv = (D + 127) / 128;
  cudaError_t e = cudaSuccess;
  if (nv <= 2) e = ln_bwd_cols_launch<2>(dy, x, gamma, dres, dx, dx16, scratch, rows, D, eps, s);
  else if (nv <= 4) e = ln_bwd_cols_launch<4>(dy, x, gamma, dres, dx, dx16, scratch, rows, D, eps, s);
  else if (nv <= 6) e = ln_bwd_cols_launch<6>(dy, x, gamma, dres, dx, dx16, scratch, rows, D, eps, s);
  else if (nv <= 8) e = ln_bwd_cols_launch<8>(dy, x, gamma, dres, dx, dx16, scratch, rows, D, eps, s);
  else if (nv <= 13) e = ln_bwd_cols_launch<13>(dy, x, gamma, dres, dx, dx16, scratch, rows, D, eps, s);
  else {
    float* prod = scratch;
    float* part = scratch + rows * D;
    e = launch_pdl(ln_bwd_16<__nv_bfloat16>, dim3(blocks_for(rows, 8)), 256, 0, s, 0, dy, x,
                   static_cast<const __nv_bfloat16*>(gamma), dres, dx, static_cast<__nv_bfloat16*>(dx16), prod, rows,
                   D, eps);
    if (e == cudaSuccess) e = launch_colsum(prod, false, rows, D, D, part, dgamma, s);
    if (e == cudaSuccess) e = launch_colsum(dy, false, rows, D, D, part, dbeta, s);
    if (e == cudaSuccess && dbias) e = launch_colsum(dx, false, rows, D, D, part, dbias, s);
    return e;
  }
  if (e != cudaSuccess) return e;
  const int blocks = static_cast<int>((rows + kLnColsWarps - 1) / kLnColsWarps);
  return colsum_finish(scratch, blocks, 3 * D, D, dgamma, dbeta, dbias, s);
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
