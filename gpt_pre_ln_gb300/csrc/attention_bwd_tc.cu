// Causal multi-head attention backward on the 5th-generation tensor cores.
//
// With c the score scale (1/sqrt(64) for GPT-2), s = c q k^T, p = softmax
// over the visible keys (j <= i), o = p v and do the gradient of o:
//   dv = p^T do,  dp = do v^T,  ds = p * (dp - delta),  delta_i = do_i . o_i
//   dq = c ds k,  dk = c ds^T q
// (llm.c notes 5.3: the softmax gradient follows the max-subtracted forward;
// positions the causal mask hides get no gradient.)  p is recomputed from q,
// k and the forward's per-row log-sum-exp, so no [T, T] matrix is stored.
//
// Two kernels, each one CTA per (batch, head, tile), two CTAs per SM (256
// tensor-memory columns and ~66 KB of shared memory each):
//   attn_bwd_dq   thread = query row (tensor-memory lane), 128 queries per
//                 CTA; per 64-key tile j <= the diagonal:
//                   S = Q K^T, dP = dO V^T      (M=128 N=64 K=64, smem operands)
//                   dS = P (dP - delta) c       written as 16-bit over S
//                   dQ += dS K                  (A = dS in tensor memory, K MN-major)
//   attn_bwd_dkv  thread = key row, 128 keys per CTA; per 64-query tile at
//                 or after the diagonal, the transposed products
//                   S^T = K Q^T, dP^T = V dO^T
//                   P^T over S^T, dS^T over dP^T (16-bit, in tensor memory)
//                   dV += P^T dO, dK += dS^T Q  (A in tensor memory, B MN-major)
// so every product is a plain tcgen05.mma with its operands where the
// previous step left them, and each output row is summed in one CTA in a
// fixed order (no atomics; the result does not depend on timing).  Work
// items are issued heaviest first.  Rows past T read whatever TMA returns
// there (zeros past the buffer, else the next sequence's rows) and are
// masked out of every sum; nothing is stored for them.
//
// Waits are bounded (common.cuh); a timeout records GPT2_ERR_TIMEOUT and the
// roles unwind, draining their copies; tensor memory is freed on every path.
#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kHd = 64;
constexpr int kThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2-5 element-wise
constexpr int kBox = 64 * kHd * 2;  // one TMA box: 64 rows of 64 16-bit values (8 KB)
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColDP = 64, kColA0 = 128, kColA1 = 192;
constexpr int kSmemBytes = 1024 + 8 * kBox + 2048;  // eight 8 KB tiles, lse / delta slots and barriers

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// K-major operand of 64 16-bit values per row (128-byte swizzle), step kk of
// K = 16; and the MN-major operand of 64 columns, K rows kk*16 .. + 15.
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int kk) { return sdesc_sw128(base + kk * 32, 16, 1024); }
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int kk) { return sdesc_sw128(base + kk * 2048, 8192, 1024); }

// delta[b, h, t] = sum_d dout[b, t, h*64 + d] * out[b, t, h*64 + d]: eight
// lanes per (b, t, h) row of 64 values (16-byte loads, the 8 products added
// in a fixed tree, then the lanes by xor shuffles), kDeltaRows rows per
// group of lanes with all their loads in flight together.
constexpr int kDeltaRows = 4;
template <typename T16>
__global__ void __launch_bounds__(256) attn_bwd_delta(const T16* __restrict__ out, const T16* __restrict__ dout,
                                                      float* __restrict__ delta, int B, int T, int H) {
  griddep_wait();
  griddep_launch_dependents();
  const long long n = static_cast<long long>(B) * T * H;
  const long long grp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;
  const long long n_grp = (static_cast<long long>(gridDim.x) * blockDim.x) >> 3;
  const int g = threadIdx.x & 7;
  uint4 o[kDeltaRows], d[kDeltaRows];
#pragma unroll
  for (int i = 0; i < kDeltaRows; ++i) {
    const long long w = grp + i * n_grp;  // (b t) H + h
    if (w < n) {
      o[i] = *reinterpret_cast<const uint4*>(out + w * kHd + g * 8);
      d[i] = *reinterpret_cast<const uint4*>(dout + w * kHd + g * 8);
    } else {
      o[i] = d[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int i = 0; i < kDeltaRows; ++i) {
    const uint32_t ow[4] = {o[i].x, o[i].y, o[i].z, o[i].w}, dw[4] = {d[i].x, d[i].y, d[i].z, d[i].w};
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 a = Type16<T16>::unpack2(ow[e]), b = Type16<T16>::unpack2(dw[e]);
      p[e] = fmaf(a.x, b.x, a.y * b.y);
    }
    float sum = (p[0] + p[1]) + (p[2] + p[3]);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    const long long w = grp + i * n_grp;
    if (g == 0 && w < n) {
      const int h = static_cast<int>(w % H);
      const long long bt = w / H;
      const long long b = bt / T, t = bt % T;
      delta[(b * H + h) * T + t] = sum;
    }
  }
}

// Packs two fp32 values of one row (masked ones as 0).
template <typename T16>
__device__ __forceinline__ uint32_t pack_masked(float a, float b, bool va, bool vb) {
  return Type16<T16>::pack2(va ? a : 0.f, vb ? b : 0.f);
}

// ------------------------------------------------------------------ dQ
template <typename T16>
__global__ void __launch_bounds__(kThreads, 2)
    attn_bwd_dq(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                const float* __restrict__ lse, const float* __restrict__ delta, T16* __restrict__ dqkv, int B, int T,
                int H, float scale_log2, float score_scale, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);   // 128 query rows (two boxes)
  const uint32_t sDO = sQ + 2 * kBox;   // their output gradients
  const uint32_t sK0 = sDO + 2 * kBox;  // K slots 0, 1 (64 keys each)
  const uint32_t sV0 = sK0 + 2 * kBox;  // V slots 0, 1
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 8 * kBox);
  const uint32_t qd_full = smem_u32(bars + 0);
  auto kv_full = [&](int s) { return smem_u32(bars + 1 + s); };
  auto kv_empty = [&](int s) { return smem_u32(bars + 3 + s); };
  const uint32_t sdp_full = smem_u32(bars + 5);
  const uint32_t ds_ready = smem_u32(bars + 6);
  const uint32_t dq_done = smem_u32(bars + 7);
  const uint32_t drain = smem_u32(bars + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int D = H * kHd;
  const int BH = B * H;
  const int n_qt = (T + 127) / 128;
  const int w = blockIdx.x;
  const int qt = n_qt - 1 - w / BH;  // heaviest (longest) rows first
  const int bh = w % BH, b = bh / H, h = bh % H;
  const int row_base = b * T;
  const int n_kt = min(2 * qt + 2, (T + 63) / 64);  // 64-key tiles at or below the diagonal, holding keys < T

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_do);
    mbar_init(qd_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(ds_ready, 4);  // one arrival per element-wise warp
    mbar_init(dq_done, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  griddep_wait();  // qkv, dout, lse and delta come from earlier kernels; tensor memory only after they completed
  griddep_launch_dependents();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const int r0 = row_base + qt * 128;
      mbar_arrive_expect_tx(qd_full, 4 * kBox);
      tma_load_2d(sQ, &tm_qkv, qd_full, h * kHd, r0);
      tma_load_2d(sQ + kBox, &tm_qkv, qd_full, h * kHd, r0 + 64);
      tma_load_2d(sDO, &tm_do, qd_full, h * kHd, r0);
      tma_load_2d(sDO + kBox, &tm_do, qd_full, h * kHd, r0 + 64);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kt; ++j) {
        const int st = j & 1;
        if (!mbar_wait(kv_empty(st), static_cast<uint32_t>((j >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(kv_full(st), 2 * kBox);
        tma_load_2d(sK0 + st * kBox, &tm_qkv, kv_full(st), D + h * kHd, row_base + j * 64);
        tma_load_2d(sV0 + st * kBox, &tm_qkv, kv_full(st), 2 * D + h * kHd, row_base + j * 64);
        ++issued;
      }
      // copies still in flight
      bool drained = mbar_wait(qd_full, 0);
      for (int x = issued > 2 ? issued - 2 : 0; x < issued && drained; ++x)
        drained = mbar_wait(kv_full(x & 1), static_cast<uint32_t>((x >> 1) & 1));
      if (!ok || !drained) record_error(err, kErrTimeout, kSiteAttnBwd);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_s = idesc_f16kind_f32(128, 64, false, false, Type16<T16>::kFormat);
      constexpr uint32_t idesc_acc = idesc_f16kind_f32(128, 64, false, true, Type16<T16>::kFormat);
      bool ok = mbar_wait(qd_full, 0);
      bool any = false;
      // dQ += dS(j) K(j): dS in the S columns, K(j) as the MN-major B
      auto dq = [&](int j) {
        if (!mbar_wait(ds_ready, static_cast<uint32_t>(j & 1))) return false;
        tc_fence_after();
        const uint32_t kb = sK0 + (j & 1) * kBox;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts(tmem + kColA0, tmem + kColS + kk * 8, mnmaj(kb, kk), idesc_acc, (j | kk) != 0 ? 1u : 0u);
        umma_commit(dq_done);
        umma_commit(kv_empty(j & 1));
        return true;
      };
      for (int j = 0; j < n_kt && ok; ++j) {
        if (j > 0) {
          // S(j) overwrites dS(j - 1): its product must have completed
          if (!dq(j - 1) || !mbar_wait(dq_done, static_cast<uint32_t>((j - 1) & 1))) {
            ok = false;
            break;
          }
        }
        if (!mbar_wait(kv_full(j & 1), static_cast<uint32_t>((j >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t kb = sK0 + (j & 1) * kBox, vb = sV0 + (j & 1) * kBox;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + kColS, kmaj(sQ, kk), kmaj(kb, kk), idesc_s, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + kColDP, kmaj(sDO, kk), kmaj(vb, kk), idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(sdp_full);
        any = true;
      }
      if (ok && n_kt > 0 && !dq(n_kt - 1)) ok = false;
      if (!ok) record_error(err, kErrTimeout, kSiteAttnBwd);
      if (any) {
        umma_commit(drain);
        if (!mbar_wait(drain, 0)) record_error(err, kErrTimeout, kSiteAttnBwd);
      }
    }
  } else {
    // ------------------------------------------------ element-wise (warps 2..5)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int q = qt * 128 + r;
    const bool q_ok = q < T;
    const long long stat = (static_cast<long long>(b) * H + h) * T + q;
    const float lse2 = q_ok ? lse[stat] : 0.f;
    const float dl = q_ok ? delta[stat] : 0.f;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS, tDP = tmem + lane_off + kColDP;
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(sdp_full, static_cast<uint32_t>(j & 1)))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        // 32 keys from key0 against this warp's 32 rows from row0:
        // d >= 32 none visible, d == 0 key i visible to lane L iff i <= L,
        // d <= -32 all visible
        const int d = (j * 64 + c * 32) - (qt * 128 + quad * 32);
        uint32_t pk[16];
        if (d > 0) {
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = 0u;
        } else {
          uint32_t rs[32], rp[32];
          tmem_ld_32x32b_x32(tS + c * 32, rs);
          tmem_ld_32x32b_x32(tDP + c * 32, rp);
          tmem_ld_wait();
          // p = 2^(s c log2(e) - lse), ds = p (dp - delta) c on paired fp32
          // instructions (the same operations as scalar code)
          const float2 sl2 = make_float2(scale_log2, scale_log2), nl2 = make_float2(-lse2, -lse2);
          const float2 nd2 = make_float2(-dl, -dl), sc2 = make_float2(score_scale, score_scale);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = fma_f32x2(make_float2(__uint_as_float(rs[2 * i]), __uint_as_float(rs[2 * i + 1])), sl2, nl2);
            const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            const float2 ds = mul_f32x2(
                mul_f32x2(pp, add_f32x2(make_float2(__uint_as_float(rp[2 * i]), __uint_as_float(rp[2 * i + 1])), nd2)),
                sc2);
            pk[i] = pack_masked<T16>(ds.x, ds.y, d < 0 || 2 * i <= lane, d < 0 || 2 * i + 1 <= lane);
          }
        }
        tmem_st_32x32b_x16(tS + c * 16, pk);  // over S columns already read
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
    }
    if (ok && n_kt > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(dq_done, static_cast<uint32_t>((n_kt - 1) & 1)))) {
        ok = false;
      } else {
        tc_fence_after();
        T16* row = dqkv + (static_cast<long long>(row_base) + q) * 3 * D + h * kHd;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t raw[32];
          tmem_ld_32x32b_x32(tmem + lane_off + kColA0 + c * 32, raw);
          tmem_ld_wait();
          if (q_ok) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t wv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                wv[e] = Type16<T16>::pack2(__uint_as_float(raw[v * 8 + 2 * e]), __uint_as_float(raw[v * 8 + 2 * e + 1]));
              *reinterpret_cast<uint4*>(row + c * 32 + v * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
        }
      }
    }
    if (!ok && lane == 0) record_error(err, kErrTimeout, kSiteAttnBwd);
  }

  // every warp arrives converged (the producer and MMA roles ran on one lane):
  // a CTA barrier reached by a diverged warp need not hold the others, and
  // the tensor memory is freed only after the epilogue's last read
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- dK, dV
template <typename T16>
__global__ void __launch_bounds__(kThreads, 2)
    attn_bwd_dkv(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_do,
                 const float* __restrict__ lse, const float* __restrict__ delta, T16* __restrict__ dqkv, int B, int T,
                 int H, float scale_log2, float score_scale, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_u32(smem);   // 128 key rows (two boxes)
  const uint32_t sV = sK + 2 * kBox;    // their values
  const uint32_t sQ0 = sV + 2 * kBox;   // Q slots 0, 1 (64 queries each)
  const uint32_t sD0 = sQ0 + 2 * kBox;  // dO slots 0, 1
  float* s_lse = reinterpret_cast<float*>(smem + 8 * kBox);  // [2 slots][64]
  float* s_dl = s_lse + 128;                                 // [2 slots][64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 8 * kBox + 512 * 2);
  const uint32_t kv_full = smem_u32(bars + 0);
  auto qd_full = [&](int s) { return smem_u32(bars + 1 + s); };
  auto qd_empty = [&](int s) { return smem_u32(bars + 3 + s); };
  const uint32_t sdp_full = smem_u32(bars + 5);
  const uint32_t pds_ready = smem_u32(bars + 6);
  const uint32_t dkv_done = smem_u32(bars + 7);
  const uint32_t drain = smem_u32(bars + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int D = H * kHd;
  const int BH = B * H;
  const int w = blockIdx.x;
  const int kt = w / BH;  // heaviest (earliest keys, most queries) first
  const int bh = w % BH, b = bh / H, h = bh % H;
  const int row_base = b * T;
  const int qi0 = 2 * kt;                 // first 64-query tile at or after the diagonal
  const int n_i = (T + 63) / 64 - qi0;    // query tiles holding queries < T

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_do);
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(qd_full(s), 1);
      mbar_init(qd_empty(s), 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(pds_ready, 4);  // one arrival per element-wise warp
    mbar_init(dkv_done, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  griddep_wait();
  griddep_launch_dependents();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const int r0 = row_base + kt * 128;
      mbar_arrive_expect_tx(kv_full, 4 * kBox);
      tma_load_2d(sK, &tm_qkv, kv_full, D + h * kHd, r0);
      tma_load_2d(sK + kBox, &tm_qkv, kv_full, D + h * kHd, r0 + 64);
      tma_load_2d(sV, &tm_qkv, kv_full, 2 * D + h * kHd, r0);
      tma_load_2d(sV + kBox, &tm_qkv, kv_full, 2 * D + h * kHd, r0 + 64);
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < n_i; ++i) {
        const int st = i & 1;
        if (!mbar_wait(qd_empty(st), static_cast<uint32_t>((i >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(qd_full(st), 2 * kBox);
        const int qr = row_base + (qi0 + i) * 64;
        tma_load_2d(sQ0 + st * kBox, &tm_qkv, qd_full(st), h * kHd, qr);
        tma_load_2d(sD0 + st * kBox, &tm_do, qd_full(st), h * kHd, qr);
        ++issued;
      }
      bool drained = mbar_wait(kv_full, 0);
      for (int x = issued > 2 ? issued - 2 : 0; x < issued && drained; ++x)
        drained = mbar_wait(qd_full(x & 1), static_cast<uint32_t>((x >> 1) & 1));
      if (!ok || !drained) record_error(err, kErrTimeout, kSiteAttnBwd);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_s = idesc_f16kind_f32(128, 64, false, false, Type16<T16>::kFormat);
      constexpr uint32_t idesc_acc = idesc_f16kind_f32(128, 64, false, true, Type16<T16>::kFormat);
      bool ok = mbar_wait(kv_full, 0);
      bool any = false;
      // dV += P^T(i) dO(i), dK += dS^T(i) Q(i): A in the S / dP columns
      auto acc = [&](int i) {
        if (!mbar_wait(pds_ready, static_cast<uint32_t>(i & 1))) return false;
        tc_fence_after();
        const uint32_t qb = sQ0 + (i & 1) * kBox, db = sD0 + (i & 1) * kBox;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts(tmem + kColA0, tmem + kColS + kk * 8, mnmaj(db, kk), idesc_acc, (i | kk) != 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_ts(tmem + kColA1, tmem + kColDP + kk * 8, mnmaj(qb, kk), idesc_acc, (i | kk) != 0 ? 1u : 0u);
        umma_commit(dkv_done);
        umma_commit(qd_empty(i & 1));
        return true;
      };
      for (int i = 0; i < n_i && ok; ++i) {
        if (i > 0) {
          if (!acc(i - 1) || !mbar_wait(dkv_done, static_cast<uint32_t>((i - 1) & 1))) {
            ok = false;
            break;
          }
        }
        if (!mbar_wait(qd_full(i & 1), static_cast<uint32_t>((i >> 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t qb = sQ0 + (i & 1) * kBox, db = sD0 + (i & 1) * kBox;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + kColS, kmaj(sK, kk), kmaj(qb, kk), idesc_s, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + kColDP, kmaj(sV, kk), kmaj(db, kk), idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(sdp_full);
        any = true;
      }
      if (ok && n_i > 0 && !acc(n_i - 1)) ok = false;
      if (!ok) record_error(err, kErrTimeout, kSiteAttnBwd);
      if (any) {
        umma_commit(drain);
        if (!mbar_wait(drain, 0)) record_error(err, kErrTimeout, kSiteAttnBwd);
      }
    }
  } else {
    // ------------------------------------------------ element-wise (warps 2..5)
    const int quad = warp & 3;
    const int t = threadIdx.x - 64;  // 0..127
    const int r = quad * 32 + lane;
    const int k = kt * 128 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + kColS, tDP = tmem + lane_off + kColDP;
    const long long stat0 = (static_cast<long long>(b) * H + h) * T;
    bool ok = true;
    // Every iteration passes the named barrier, also after a timeout (the
    // four warps then only keep the barrier count, so none is left waiting).
    for (int i = 0; i < n_i; ++i) {
      const int q0 = (qi0 + i) * 64;
      const int sl = i & 1;
      {
        // this tile's 64 row statistics, negated, into the slot (rows past
        // T: zero)
        const int qq = q0 + (t & 63);
        const float v = qq < T ? (t < 64 ? lse[stat0 + qq] : delta[stat0 + qq]) : 0.f;
        (t < 64 ? s_lse : s_dl)[sl * 64 + (t & 63)] = -v;
      }
      named_bar_sync(1, 128);
      if (!ok) continue;
      if (!__all_sync(0xffffffffu, mbar_wait(sdp_full, static_cast<uint32_t>(i & 1)))) {
        ok = false;
        continue;
      }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        // 32 queries from qc0 against this warp's 32 keys from k0:
        // d < 0 none visible, d == 0 query i visible to key lane L iff
        // L <= i, d >= 32 all visible (queries past T never)
        const int qc0 = q0 + c * 32;
        const int d = qc0 - (kt * 128 + quad * 32);
        uint32_t pk[16], dk[16];
        if (d < 0) {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = dk[e] = 0u;
        } else {
          uint32_t rs[32], rp[32];
          tmem_ld_32x32b_x32(tS + c * 32, rs);
          tmem_ld_32x32b_x32(tDP + c * 32, rp);
          tmem_ld_wait();
          const float2* nls = reinterpret_cast<const float2*>(s_lse + sl * 64 + c * 32);  // -lse
          const float2* nds = reinterpret_cast<const float2*>(s_dl + sl * 64 + c * 32);   // -delta
          const float2 sl2 = make_float2(scale_log2, scale_log2), sc2 = make_float2(score_scale, score_scale);
          // p and ds on paired fp32 instructions (the same operations as
          // scalar code)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            bool vis[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) vis[u] = (d > 0 || lane <= 2 * e + u) && qc0 + 2 * e + u < T;
            const float2 x =
                fma_f32x2(make_float2(__uint_as_float(rs[2 * e]), __uint_as_float(rs[2 * e + 1])), sl2, nls[e]);
            const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            const float2 ds = mul_f32x2(
                mul_f32x2(p, add_f32x2(make_float2(__uint_as_float(rp[2 * e]), __uint_as_float(rp[2 * e + 1])), nds[e])),
                sc2);
            pk[e] = pack_masked<T16>(p.x, p.y, vis[0], vis[1]);
            dk[e] = pack_masked<T16>(ds.x, ds.y, vis[0], vis[1]);
          }
        }
        tmem_st_32x32b_x16(tS + c * 16, pk);   // P^T over S^T columns already read
        tmem_st_32x32b_x16(tDP + c * 16, dk);  // dS^T over dP^T columns already read
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pds_ready);
    }
    if (ok && n_i > 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(dkv_done, static_cast<uint32_t>((n_i - 1) & 1)))) {
        ok = false;
      } else {
        tc_fence_after();
        T16* row = dqkv + (static_cast<long long>(row_base) + k) * 3 * D + h * kHd;
#pragma unroll
        for (int which = 0; which < 2; ++which) {  // dV (columns 2D..), dK (columns D..)
          T16* dst = row + (which == 0 ? 2 * D : D);
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t raw[32];
            tmem_ld_32x32b_x32(tmem + lane_off + (which == 0 ? kColA0 : kColA1) + c * 32, raw);
            tmem_ld_wait();
            if (k < T) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint32_t wv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  wv[e] = Type16<T16>::pack2(__uint_as_float(raw[v * 8 + 2 * e]),
                                             __uint_as_float(raw[v * 8 + 2 * e + 1]));
                *reinterpret_cast<uint4*>(dst + c * 32 + v * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
              }
            }
          }
        }
      }
    }
    if (!ok && lane == 0) record_error(err, kErrTimeout, kSiteAttnBwd);
  }

  // every warp arrives converged (the producer and MMA roles ran on one lane):
  // a CTA barrier reached by a diverged warp need not hold the others, and
  // the tensor memory is freed only after the epilogue's last read
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename Kern>
cudaError_t smem_once(Kern kern, int (&configured)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return cudaSuccess;
}

template <typename T16>
cudaError_t launch_bwd(const void* qkv, const void* out, const float* lse, const void* dout, void* dqkv, float* delta,
                       int B, int T, int H, float score_scale, cudaStream_t s) {
  if (B == 0 || T == 0) return cudaSuccess;
  const uint64_t D = static_cast<uint64_t>(H) * kHd;
  const uint64_t rows = static_cast<uint64_t>(B) * T;
  CUtensorMap tq, td;
  if (!encode_tma_2d(&tq, Type16<T16>::kTma, qkv, 3 * D, rows, 3 * D * 2, kHd, 64) ||
      !encode_tma_2d(&td, Type16<T16>::kTma, dout, D, rows, D * 2, kHd, 64))
    return cudaErrorInvalidValue;
  static int conf_q[64] = {0}, conf_kv[64] = {0};
  cudaError_t e = smem_once(attn_bwd_dq<T16>, conf_q);
  if (e == cudaSuccess) e = smem_once(attn_bwd_dkv<T16>, conf_kv);
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(rows) * H;  // rows of 64 values, 8 lanes and kDeltaRows rows each
  const long long groups = (items + kDeltaRows - 1) / kDeltaRows;
  e = launch_pdl(attn_bwd_delta<T16>, dim3(static_cast<unsigned>((groups * 8 + 255) / 256)), 256, 0, s, 0,
                 static_cast<const T16*>(out), static_cast<const T16*>(dout), delta, B, T, H);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f * score_scale;
  const int n_qt = (T + 127) / 128;
  e = launch_pdl(attn_bwd_dq<T16>, dim3(B * H * n_qt), kThreads, kSmemBytes, s, 0, tq, td, lse,
                 static_cast<const float*>(delta), static_cast<T16*>(dqkv), B, T, H, scale_log2, score_scale,
                 device_error_word());
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_bwd_dkv<T16>, dim3(B * H * n_qt), kThreads, kSmemBytes, s, 0, tq, td, lse,
                    static_cast<const float*>(delta), static_cast<T16*>(dqkv), B, T, H, scale_log2, score_scale,
                    device_error_word());
}

}  // namespace

cudaError_t launch_attention_backward_tc(gpt2_dtype dt, const void* qkv, const void* out, const float* lse,
                                         const void* dout, void* dqkv, float* delta, int B, int T, int n_head,
                                         float score_scale, cudaStream_t stream) {
  if (dt == GPT2_F16)
    return launch_bwd<__half>(qkv, out, lse, dout, dqkv, delta, B, T, n_head, score_scale, stream);
  return launch_bwd<__nv_bfloat16>(qkv, out, lse, dout, dqkv, delta, B, T, n_head, score_scale, stream);
}

}  // namespace gpt2
