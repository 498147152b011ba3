// Causal multi-head self-attention on the packed c_attn output.
//
//   out[b, i, h*64 + d] = sum_{j <= i} softmax_j(q_i . k_j / sqrt(64)) v_j[d]
//
// ("逐行拆GPT-2源码", GPT2Attention ``_split_heads`` / ``_attn`` /
// ``_merge_heads``; llm.c notes 2.2-2.3: scale 1/sqrt(d_k), future positions
// masked before the softmax, row maximum subtracted.)  The Q|K|V split and
// the head split are index arithmetic on the [B, T, 3D] input; the head merge
// is the store into [B, T, D].
//
// bf16 path: flash-style tiles of 64 queries x 64 keys.  S = Q K^T and O += P V
// run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate); the
// softmax is online in fp32 registers.  Key tiles entirely above the
// diagonal are never visited; only the diagonal tile evaluates the mask.
// Query tiles are scheduled heaviest first.
//
// fp32 path: one warp per query row, exact two-pass softmax with expf; it is
// the correctness path of the F32 configuration.
#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kHd = 64;
constexpr int kBq = 64;
constexpr int kBkv = 64;
constexpr int kAttnThreads = 128;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int n = pred ? 16 : 0;  // 0 bytes read -> the 16 bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float exp2_hw(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory tile of 64 rows x 64 bf16 (128 B per row), 16-byte chunks
// XOR-swizzled by (row & 7) so that ldmatrix reads are conflict free.
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Loads rows [r0, r0+64) of one 64-wide column block of qkv into a tile.
__device__ __forceinline__ void load_tile(uint32_t s_tile, const __nv_bfloat16* base, long long row_stride, int r0,
                                          int T, int tid) {
#pragma unroll
  for (int i = 0; i < (kBkv * 8) / kAttnThreads; ++i) {
    const int idx = tid + i * kAttnThreads;
    const int row = idx >> 3;
    const int chunk = idx & 7;
    const int g = r0 + row;
    const bool ok = g < T;
    const __nv_bfloat16* src = base + static_cast<long long>(ok ? g : 0) * row_stride + chunk * 8;
    cp_async16(s_tile + tile_off(row, chunk), src, ok);
  }
}

__global__ void __launch_bounds__(kAttnThreads) attn_causal_bf16(const __nv_bfloat16* __restrict__ qkv,
                                                                 __nv_bfloat16* __restrict__ out, int T, int H) {
  __shared__ __align__(128) uint8_t smem[kBq * 128 + 4 * kBkv * 128];
  const int bh = blockIdx.x;
  const int b = bh / H;
  const int h = bh % H;
  const int n_qt = (T + kBq - 1) / kBq;
  const int qt = n_qt - 1 - static_cast<int>(blockIdx.y);  // heaviest tiles first
  const int q0 = qt * kBq;
  const int D = H * kHd;
  const long long rs = 3LL * D;
  const __nv_bfloat16* base = qkv + static_cast<long long>(b) * T * rs;
  const __nv_bfloat16* qb = base + h * kHd;
  const __nv_bfloat16* kb = base + D + h * kHd;
  const __nv_bfloat16* vb = base + 2 * D + h * kHd;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t sQ = smem_u32(smem);
  // stage s of K at sK0 + s * kStage, of V at sV0 + s * kStage
  constexpr uint32_t kStage = kBkv * 128;
  const uint32_t sK0 = sQ + kBq * 128;
  const uint32_t sV0 = sK0 + 2 * kStage;

  load_tile(sQ, qb, rs, q0, T, tid);
  load_tile(sK0, kb, rs, 0, T, tid);
  load_tile(sV0, vb, rs, 0, T, tid);
  cp_async_commit();

  const float scale_log2 = 1.4426950408889634f * 0.125f;  // log2(e) / sqrt(64)
  float o[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_r[2] = {-1e30f, -1e30f};
  float l_r[2] = {0.f, 0.f};
  uint32_t qf[4][4];

  const int n_kv = qt + 1;  // key tiles 0..qt; the rest are fully masked
  for (int j = 0; j < n_kv; ++j) {
    const int cur = j & 1;
    if (j + 1 < n_kv) {
      load_tile(sK0 + (cur ^ 1) * kStage, kb, rs, (j + 1) * kBkv, T, tid);
      load_tile(sV0 + (cur ^ 1) * kStage, vb, rs, (j + 1) * kBkv, T, tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (j == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int row = warp * 16 + (lane & 15);
        const int chunk = 2 * kk + (lane >> 4);
        ldsm_x4(sQ + tile_off(row, chunk), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    // S = Q K^T for this warp's 16 queries x 64 keys
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = np * 16 + ((lane >> 4) << 3) + (lane & 7);
        const int chunk = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK0 + cur * kStage + tile_off(key, chunk), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qf[kk], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qf[kk], b2, b3);
      }
    }
    // causal mask on the diagonal tile only
    const int qrow0 = q0 + warp * 16 + (lane >> 2);
    if (j == qt) {
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int key = j * kBkv + n * 8 + 2 * (lane & 3);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int qi = qrow0 + ((e >> 1) << 3);
          const int kj = key + (e & 1);
          if (kj > qi) s[n][e] = -INFINITY;
        }
      }
    }
    // online softmax, rows r0 = lane/4 and r1 = lane/4 + 8
    float mx[2] = {m_r[0], m_r[1]};
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      mx[0] = fmaxf(mx[0], fmaxf(s[n][0], s[n][1]));
      mx[1] = fmaxf(mx[1], fmaxf(s[n][2], s[n][3]));
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float alpha[2], rsum[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      alpha[r] = exp2_hw((m_r[r] - mx[r]) * scale_log2);
      m_r[r] = mx[r];
    }
    uint32_t pf[4][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float p0 = exp2_hw((s[n][0] - mx[0]) * scale_log2);
      const float p1 = exp2_hw((s[n][1] - mx[0]) * scale_log2);
      const float p2 = exp2_hw((s[n][2] - mx[1]) * scale_log2);
      const float p3 = exp2_hw((s[n][3] - mx[1]) * scale_log2);
      rsum[0] += p0 + p1;
      rsum[1] += p2 + p3;
      pf[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
      pf[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) l_r[r] = l_r[r] * alpha[r] + rsum[r];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    // O += P V: P (16 x 64 keys) from registers, V^T fragments by ldmatrix.trans
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t a[4] = {pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3]};
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {
        const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int chunk = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sV0 + cur * kStage + tile_off(key, chunk), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], a, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], a, b2, b3);
      }
    }
    __syncthreads();  // this stage is overwritten by the next prefetch
  }

  // the row sums are spread over the 4 threads of a quad
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
  }
  const float inv0 = 1.f / l_r[0];
  const float inv1 = 1.f / l_r[1];
  const int qa = q0 + warp * 16 + (lane >> 2);
  const int qb2 = qa + 8;
  __nv_bfloat16* ob = out + static_cast<long long>(b) * T * D + h * kHd;
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const int d = n * 8 + 2 * (lane & 3);
    if (qa < T)
      *reinterpret_cast<__nv_bfloat162*>(ob + static_cast<long long>(qa) * D + d) =
          __floats2bfloat162_rn(o[n][0] * inv0, o[n][1] * inv0);
    if (qb2 < T)
      *reinterpret_cast<__nv_bfloat162*>(ob + static_cast<long long>(qb2) * D + d) =
          __floats2bfloat162_rn(o[n][2] * inv1, o[n][3] * inv1);
  }
}

// fp32 reference-precision attention: one warp per (b, h, i).
constexpr int kF32Warps = 4;

__global__ void __launch_bounds__(kF32Warps * 32) attn_causal_f32(const float* __restrict__ qkv,
                                                                  float* __restrict__ out, int T, int H) {
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
    acc *= 0.125f;
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

cudaError_t launch_attention_bf16(const __nv_bfloat16* qkv, __nv_bfloat16* out, int B, int T, int n_head,
                                  cudaStream_t stream) {
  if (B == 0 || T == 0) return cudaSuccess;
  dim3 grid(B * n_head, (T + kBq - 1) / kBq);
  attn_causal_bf16<<<grid, kAttnThreads, 0, stream>>>(qkv, out, T, n_head);
  return cudaGetLastError();
}

cudaError_t launch_attention_f32(const float* qkv, float* out, int B, int T, int n_head, cudaStream_t stream) {
  if (B == 0 || T == 0) return cudaSuccess;
  const long long rows = static_cast<long long>(n_head) * T;
  dim3 grid(static_cast<unsigned>((rows + kF32Warps - 1) / kF32Warps), B);
  const size_t smem = static_cast<size_t>(kF32Warps) * T * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_causal_f32, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  attn_causal_f32<<<grid, kF32Warps * 32, smem, stream>>>(qkv, out, T, n_head);
  return cudaGetLastError();
}

}  // namespace gpt2
