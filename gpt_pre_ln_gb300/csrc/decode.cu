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
  griddep_wait();
  griddep_launch_dependents();
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

// Attention of the new token over the cache, one CTA of four warps per
// (b, h).  The cached keys 0..pos-1 are cut into chunks of 16; warp w takes
// chunks w, w+4, w+8, ...  Each warp double-buffers its chunks in shared
// memory: its lane 0 loads a chunk's 16 K rows and 16 V rows as two TMA
// boxes with the 128-byte swizzle (16-byte unit u of row r lands at unit
// u ^ (r & 7)), which makes the reads below free of bank conflicts.
// Scores take two lanes per key (32 dimensions each, one shuffle to add) and
// live in log2 units (q carries log2(e) / sqrt(64)); the probabilities go
// through shared memory to the P.V phase, where lane (par, dq) accumulates
// dimensions 4dq..4dq+3 over the chunk's keys of parity par (the two halves
// of the warp are added once at the end).  Each warp keeps an online-softmax
// partial (running max, sum, accumulator); the new token's k, v are written
// to cache slot pos and enter as one more partial from registers, so no load
// of this launch reads a value it writes.
constexpr int kDaWarps = 4;
constexpr int kDaChunk = 16;
constexpr int kDaStages = 2;
constexpr int kDaBox = kDaChunk * kHd * 2;  // one box: 16 rows of 64 16-bit values
constexpr int kDaStageBytes = 2 * kDaBox;   // K and V of one chunk
constexpr int kDaSmem = kDaWarps * kDaStages * kDaStageBytes + 1024;  // + slack for 1024-byte alignment

template <typename T16>
__global__ void __launch_bounds__(kDaWarps * 32, 6)
    decode_attn_tma(const __grid_constant__ CUtensorMap kv_map, const T16* __restrict__ qkv, T16* kv_layer,
                    T16* __restrict__ out, const int32_t* __restrict__ past_len, const int* __restrict__ valid,
                    int b_cache0, int B_cache, int H, int T_max, float q_scale, unsigned* err) {
  extern __shared__ uint8_t da_smem_raw[];
  __shared__ __align__(8) uint64_t bars[kDaWarps][kDaStages];
  __shared__ float s_q[kHd];
  __shared__ __align__(16) float s_p[kDaWarps][kDaChunk];  // key k at (k & 1) * 8 + (k >> 1)
  __shared__ float s_m[kDaWarps + 1], s_l[kDaWarps + 1];
  __shared__ __align__(16) float s_acc[kDaWarps + 1][kHd];
  const int b = blockIdx.x / H;  // sequence within this call's rows
  const int h = blockIdx.x % H;
  const int bc = b_cache0 + b;   // and its index in the cache
  const int D = H * kHd;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  T16* orow = out + static_cast<long long>(b) * D + h * kHd;
  // valid and past_len were written at the start of the step, two or more
  // kernels back: readable before the dependency wait, and so are the cached
  // keys and values of slots below pos (earlier steps)
  const bool is_valid = valid[b] != 0;
  const int pos = is_valid ? past_len[b] : 0;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(da_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wbuf = smem + warp * kDaStages * kDaStageBytes;
  const int n_chunks = (pos + kDaChunk - 1) / kDaChunk;
  const int my_chunks = n_chunks > warp ? (n_chunks - warp + kDaWarps - 1) / kDaWarps : 0;
  const int row_k = (bc * H + h) * T_max;      // row of slot 0 of this (b, h) in the K half
  const int row_v = row_k + B_cache * H * T_max;  // and in the V half
  auto issue = [&](int i) {
    const int st = i % kDaStages;
    const int j0 = (warp + i * kDaWarps) * kDaChunk;
    const uint32_t bar = smem_u32(&bars[warp][st]);
    const uint32_t dst = smem_u32(wbuf + st * kDaStageBytes);
    mbar_arrive_expect_tx(bar, kDaStageBytes);
    tma_load_2d(dst, &kv_map, bar, 0, row_k + j0);
    tma_load_2d(dst + kDaBox, &kv_map, bar, 0, row_v + j0);
  };
  if (lane == 0) {
    for (int st = 0; st < kDaStages; ++st) mbar_init(smem_u32(&bars[warp][st]), 1);
    fence_barrier_init();
    for (int i = 0; i < kDaStages && i < my_chunks; ++i) issue(i);
  }
  griddep_wait();  // q, k, v of the new token come from the kernel before
  griddep_launch_dependents();
  if (!is_valid) {
    if (tid < kHd) orow[tid] = from_f32<T16>(0.f);
    return;
  }
  const T16* row = qkv + static_cast<long long>(b) * 3 * D;
  // q_scale = the score scale (1/sqrt(64) for GPT-2) times log2(e)
  if (tid < kHd) s_q[tid] = to_f32<T16>(row[h * kHd + tid]) * q_scale;
  __syncthreads();

  const int key = lane >> 1;  // score phase: key of the chunk
  const int hf = lane & 1;    // and which 32 of its 64 dimensions
  float2 q2[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) q2[e] = make_float2(s_q[hf * 32 + 2 * e], s_q[hf * 32 + 2 * e + 1]);
  const int par = lane >> 4;  // P.V phase: keys of this parity
  const int dq = lane & 15;   // dimensions 4dq..4dq+3: 8 bytes of the row
  float m = -1e30f, l = 0.f;
  float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
  int i = 0;
  for (; i < my_chunks; ++i) {
    const int st = i % kDaStages;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp][st]), (i / kDaStages) & 1));
    if (!ok) {
      if (lane == 0) record_error(err, kErrTimeout, kSiteDecodeAttn);
      break;
    }
    const uint8_t* kb = wbuf + st * kDaStageBytes;
    const uint8_t* vb = kb + kDaBox;
    const int cnt = min(kDaChunk, pos - (warp + i * kDaWarps) * kDaChunk);
    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint4 u = *reinterpret_cast<const uint4*>(kb + key * 128 + (((hf * 4 + t) ^ (key & 7)) << 4));
      s2 = fma_f32x2(q2[4 * t + 0], Type16<T16>::unpack2(u.x), s2);
      s2 = fma_f32x2(q2[4 * t + 1], Type16<T16>::unpack2(u.y), s2);
      s2 = fma_f32x2(q2[4 * t + 2], Type16<T16>::unpack2(u.z), s2);
      s2 = fma_f32x2(q2[4 * t + 3], Type16<T16>::unpack2(u.w), s2);
    }
    float s = s2.x + s2.y;
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    if (key >= cnt) s = -INFINITY;
    float cm = s;
#pragma unroll
    for (int o = 2; o < 32; o <<= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
    const float m_new = fmaxf(m, cm);
    const float alpha = ex2_approx(m - m_new);
    const float p = ex2_approx(s - m_new);
    l = fmaf(l, alpha, hf == 0 ? p : 0.f);  // each key counted by one lane of its pair
    if (hf == 0) s_p[warp][(key & 1) * 8 + (key >> 1)] = p;
    m = m_new;
    const float2 a2 = make_float2(alpha, alpha);
    acc01 = mul_f32x2(acc01, a2);
    acc23 = mul_f32x2(acc23, a2);
    __syncwarp();
    const float4 pa = *reinterpret_cast<const float4*>(&s_p[warp][par * 8]);
    const float4 pb = *reinterpret_cast<const float4*>(&s_p[warp][par * 8 + 4]);
    const float pk[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int kk = 2 * t + par;
      if (kk < cnt) {
        const uint2 w = *reinterpret_cast<const uint2*>(vb + kk * 128 + (((dq >> 1) ^ (kk & 7)) << 4) + (dq & 1) * 8);
        const float2 p2 = make_float2(pk[t], pk[t]);
        acc01 = fma_f32x2(p2, Type16<T16>::unpack2(w.x), acc01);
        acc23 = fma_f32x2(p2, Type16<T16>::unpack2(w.y), acc23);
      }
    }
    __syncwarp();
    if (lane == 0 && i + kDaStages < my_chunks) {
      fence_proxy_async_smem();
      issue(i + kDaStages);
    }
  }
  if (i < my_chunks && lane == 0) {
    // timed out: wait (bounded) for this warp's loads still in flight
    for (int k = i; k < my_chunks && k < i + kDaStages; ++k)
      (void)mbar_wait(smem_u32(&bars[warp][k % kDaStages]), (k / kDaStages) & 1);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  acc01.x += __shfl_xor_sync(0xffffffffu, acc01.x, 16);  // add the two key parities
  acc01.y += __shfl_xor_sync(0xffffffffu, acc01.y, 16);
  acc23.x += __shfl_xor_sync(0xffffffffu, acc23.x, 16);
  acc23.y += __shfl_xor_sync(0xffffffffu, acc23.y, 16);
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
  if (par == 0) *reinterpret_cast<float4*>(&s_acc[warp][4 * dq]) = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);
  if (warp == 0) {
    // the new token: score, value, and its slot in the cache
    const uint32_t kw = reinterpret_cast<const uint32_t*>(row + D + h * kHd)[lane];
    const uint32_t vw = reinterpret_cast<const uint32_t*>(row + 2 * D + h * kHd)[lane];
    const float2 kf = Type16<T16>::unpack2(kw);
    float sn = fmaf(s_q[2 * lane], kf.x, s_q[2 * lane + 1] * kf.y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sn += __shfl_xor_sync(0xffffffffu, sn, o);
    const float2 vf = Type16<T16>::unpack2(vw);
    if (lane == 0) {
      s_m[kDaWarps] = sn;
      s_l[kDaWarps] = 1.f;
    }
    s_acc[kDaWarps][2 * lane] = vf.x;
    s_acc[kDaWarps][2 * lane + 1] = vf.y;
    reinterpret_cast<uint32_t*>(kv_layer + (static_cast<long long>(row_k) + pos) * kHd)[lane] = kw;
    reinterpret_cast<uint32_t*>(kv_layer + (static_cast<long long>(row_v) + pos) * kHd)[lane] = vw;
  }
  __syncthreads();
  if (tid < kHd) {
    float M = s_m[0];
#pragma unroll
    for (int w = 1; w <= kDaWarps; ++w) M = fmaxf(M, s_m[w]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w <= kDaWarps; ++w) {
      const float c = ex2_approx(s_m[w] - M);
      L = fmaf(s_l[w], c, L);
      A = fmaf(s_acc[w][tid], c, A);
    }
    orow[tid] = from_f32<T16>(A / L);
  }
}

// (best, bi) of every thread of the block -> the block's maximum with the
// lowest index on ties, returned to thread 0.
__device__ __forceinline__ void block_argmax(float& best, int& bi) {
  __shared__ float s_v[32];
  __shared__ int s_i[32];
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
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w)
      if (s_v[w] > best || (s_v[w] == best && s_i[w] < bi)) {
        best = s_v[w];
        bi = s_i[w];
      }
  }
}

// One CTA per row: lowest index of the maximum; then past_len[b] += 1
// (unless past_len is null).
__global__ void __launch_bounds__(1024) argmax_rows(const float* __restrict__ logits, long long ld, int V,
                                                    const int* __restrict__ valid, int32_t* __restrict__ next_tokens,
                                                    int32_t* __restrict__ past_len) {
  griddep_wait();
  griddep_launch_dependents();
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
  block_argmax(best, bi);
  if (threadIdx.x == 0 && valid[b]) {
    next_tokens[b] = bi;
    if (past_len) past_len[b] += 1;
  }
}

// The same from the per-row candidates (value, index bits) of the lm_head
// GEMM's epilogue: every candidate is the maximum of a disjoint set of
// columns with its lowest index, so the maximum candidate with the lowest
// index is the row's argmax.
__global__ void __launch_bounds__(256) argmax_candidates(const float2* __restrict__ cand, int n_cand,
                                                         const int* __restrict__ valid,
                                                         int32_t* __restrict__ next_tokens,
                                                         int32_t* __restrict__ past_len) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x;
  const float2* c = cand + static_cast<long long>(b) * n_cand;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int k = threadIdx.x; k < n_cand; k += blockDim.x) {
    const float2 e = c[k];
    const int ei = __float_as_int(e.y);
    if (e.x > best || (e.x == best && ei < bi)) {
      best = e.x;
      bi = ei;
    }
  }
  block_argmax(best, bi);
  if (threadIdx.x == 0 && valid[b]) {
    next_tokens[b] = bi;
    if (past_len) past_len[b] += 1;
  }
}

// The prompt's K and V into the cache (the `present` of GPT2Attention after
// a forward over positions 0..T-1): row m = b T + t of qkv [M, 3D] holds
// k at columns D + h 64 + d and v at 2D + h 64 + d; they go to slots
// [0|1][b_cache][h][t][d] of the layer's [2, B_cache, n_head, T_max, 64]
// cache.  One CTA per row, one 16-byte chunk (8 elements) per thread.
template <typename T16>
__global__ void kv_from_qkv(const T16* __restrict__ qkv, T16* __restrict__ kv_layer, int T, int n_head, int T_max,
                            int B_cache) {
  griddep_wait();
  griddep_launch_dependents();
  const long long m = blockIdx.x;
  const int D = n_head * kHd;
  const int j = threadIdx.x;  // chunk of the row's 2D k|v elements
  if (j >= 2 * D / 8) return;
  const int b = static_cast<int>(m / T), t = static_cast<int>(m % T);
  const int kv = j * 8 >= D ? 1 : 0;
  const int c = j * 8 - kv * D;  // column within k or v
  const int h = c / kHd, d = c % kHd;
  const uint4 u = *reinterpret_cast<const uint4*>(qkv + m * 3 * D + D + j * 8);
  const long long dst = ((static_cast<long long>(kv) * B_cache + b) * n_head + h) * T_max * kHd +
                        static_cast<long long>(t) * kHd + d;
  *reinterpret_cast<uint4*>(kv_layer + dst) = u;
}

// After the prompt: x_last[b] = x[b T + T - 1] (the residual stream of each
// sequence's last position), valid[b] = 1, past_len[b] = T.
__global__ void prefill_last_rows(const float* __restrict__ x, int T, int D, float* __restrict__ x_last,
                                  int* __restrict__ valid, int32_t* __restrict__ past_len) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x;
  const float* src = x + (static_cast<long long>(b) * T + T - 1) * D;
  for (int i = threadIdx.x * 4; i < D; i += blockDim.x * 4)
    *reinterpret_cast<float4*>(x_last + static_cast<long long>(b) * D + i) =
        *reinterpret_cast<const float4*>(src + i);
  if (threadIdx.x == 0) {
    valid[b] = 1;
    past_len[b] = T;
  }
}

}  // namespace

cudaError_t launch_kv_from_qkv(gpt2_dtype dt, const void* qkv, void* kv_layer, int B, int T, int n_head, int T_max,
                               cudaStream_t stream) {
  const unsigned rows = static_cast<unsigned>(static_cast<long long>(B) * T);
  const int threads = (2 * n_head * kHd / 8 + 31) / 32 * 32;
  if (dt == GPT2_F16)
    return launch_pdl(kv_from_qkv<__half>, rows, threads, 0, stream, 0, static_cast<const __half*>(qkv),
                      static_cast<__half*>(kv_layer), T, n_head, T_max, B);
  return launch_pdl(kv_from_qkv<__nv_bfloat16>, rows, threads, 0, stream, 0,
                    static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(kv_layer), T, n_head, T_max,
                    B);
}

cudaError_t launch_prefill_last_rows(const float* x, int B, int T, int D, float* x_last, int* valid,
                                     int32_t* past_len, cudaStream_t stream) {
  return launch_pdl(prefill_last_rows, B, 256, 0, stream, 0, x, T, D, x_last, valid, past_len);
}

cudaError_t launch_decode_embed_ln(gpt2_dtype dt, const int32_t* tokens, const int32_t* past_len, const void* wte,
                                   const void* wpe, const void* gamma, const void* beta, float* x, void* y, int B,
                                   int D, int V, int n_pos, int T_max, float eps, int* valid, cudaStream_t stream) {
  const int warps = 4;
  const dim3 grid((B + warps - 1) / warps), block(warps * 32);
  unsigned* err = device_error_word();
  if (dt == GPT2_F16) {
    using T = __half;
    return launch_pdl(decode_embed_ln<T>, grid, block, 0, stream, 0, tokens, past_len, static_cast<const T*>(wte),
                      static_cast<const T*>(wpe), static_cast<const T*>(gamma), static_cast<const T*>(beta), x,
                      static_cast<T*>(y), B, D, V, n_pos, T_max, eps, valid, err);
  }
  using T = __nv_bfloat16;
  return launch_pdl(decode_embed_ln<T>, grid, block, 0, stream, 0, tokens, past_len, static_cast<const T*>(wte),
                    static_cast<const T*>(wpe), static_cast<const T*>(gamma), static_cast<const T*>(beta), x,
                    static_cast<T*>(y), B, D, V, n_pos, T_max, eps, valid, err);
}

namespace {
template <typename T16>
cudaError_t launch_decode_attn_t(const void* qkv, void* kv_layer, void* out, const int32_t* past_len, const int* valid,
                                 int B, int b_cache0, int B_cache, int n_head, int T_max, float score_scale,
                                 cudaStream_t stream) {
  // the layer's K and V halves as one [2 * B_cache * n_head * T_max, 64] matrix
  const uint64_t rows = 2ull * B_cache * n_head * static_cast<uint64_t>(T_max);
  if (rows >= (1ull << 31)) return cudaErrorInvalidValue;
  CUtensorMap map;
  if (!encode_tma_2d(&map, Type16<T16>::kTma, kv_layer, kHd, rows, kHd * 2, kHd, kDaChunk))
    return cudaErrorInvalidValue;
  return launch_pdl(decode_attn_tma<T16>, B * n_head, kDaWarps * 32, kDaSmem, stream, 0, map,
                    static_cast<const T16*>(qkv), static_cast<T16*>(kv_layer), static_cast<T16*>(out), past_len,
                    valid, b_cache0, B_cache, n_head, T_max, score_scale * 1.4426950408889634f, device_error_word());
}
}  // namespace

cudaError_t launch_decode_attention(gpt2_dtype dt, const void* qkv, void* kv_layer, void* out, const int32_t* past_len,
                                    const int* valid, int B, int b_cache0, int B_cache, int n_head, int T_max,
                                    float score_scale, cudaStream_t stream) {
  if (dt == GPT2_F16)
    return launch_decode_attn_t<__half>(qkv, kv_layer, out, past_len, valid, B, b_cache0, B_cache, n_head, T_max,
                                        score_scale, stream);
  return launch_decode_attn_t<__nv_bfloat16>(qkv, kv_layer, out, past_len, valid, B, b_cache0, B_cache, n_head,
                                             T_max, score_scale, stream);
}

cudaError_t launch_argmax_candidates(const float2* cand, int n_cand, int B, const int* valid, int32_t* next_tokens,
                                     int32_t* past_len, cudaStream_t stream) {
  return launch_pdl(argmax_candidates, B, 256, 0, stream, 0, cand, n_cand, valid, next_tokens, past_len);
}

cudaError_t launch_argmax_rows(const float* logits, int64_t ld, int B, int V, const int* valid, int32_t* next_tokens,
                               int32_t* past_len, cudaStream_t stream) {
  return launch_pdl(argmax_rows, B, 1024, 0, stream, 0, logits, static_cast<long long>(ld), V, valid, next_tokens,
                    past_len);
}

}  // namespace gpt2
