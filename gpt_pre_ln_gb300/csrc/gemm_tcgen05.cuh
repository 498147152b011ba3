// bf16 GEMM on the 5th-generation tensor cores (tcgen05) with fused
// epilogues: the Conv1D projections of the GPT-2 block (c_attn, attention
// c_proj, c_fc, MLP c_proj) and the tied lm_head.
//
//   y[M, N] = epilogue( x[M, K] . W )      W = [K, N] ("in, out", Conv1D)
//                                          or  [N, K] (wte as the lm_head)
//   epilogues: none | + bias | gelu_new or exact GELU (+ bias) | + bias +
//   residual (fp32)
//              | log-sum-exp partials (the lm_head of the loss: no output)
//              | the loss gradient (softmax(z) - onehot) / N (16-bit)
//   For the backward, A may also be read MN-major (x [K, M]: the weight
//   gradient X^T dY reads X [rows, in] as it is stored), operands may have
//   row pitches of their own, and K need not be a multiple of 64 (the
//   k-blocks past K read zeros).
//
// Two persistent kernels share one design (10 warps per CTA):
//   warp 0      TMA producer: 128-byte-swizzled A and B tiles of 64 K per
//               stage into a STAGES-deep shared-memory ring.
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma into
//               one of two fp32 accumulators in tensor memory and commits
//               the stage / accumulator barriers.
//   warps 2-9   epilogue in two halves of four warps (one thread per
//               accumulator row in each half); half h owns the column chunks
//               h, h+2, ... (128 bytes of output per row each): tcgen05.ld,
//               bias / GELU / residual in fp32, then each warp writes its
//               32 rows into a private swizzled staging area and reads them
//               back transposed, so that every global store instruction
//               covers four full 128-byte lines.  The fp32 residual is read
//               the same coalesced way.  No barrier spans more than a warp.
// gemm_1sm: one CTA per tile of 128 x BN (BN = 128, 192 or 256), MMA
//   M = 128, N = BN.
// gemm_2sm: a cluster of two CTAs per tile of 256 x 256; each CTA stages its
//   128 rows of A and its 128 columns of B, the even CTA issues the pair MMA
//   (tcgen05.mma.cta_group::2, M = 256, N = 256) and every commit arrives on
//   the barriers of both CTAs.  Per MMA cycle each SM takes in a third less
//   operand data than with 128 x 256 tiles, which is what limits these
//   K = 768 GEMMs (operand delivery, not the tensor core, sets their pace).
// The two accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1.  A is always K-major; W [K, N] is consumed MN-major straight from
// its Conv1D layout (no transpose), wte [N, K] K-major.
//
// Every mbarrier wait is bounded (common.cuh); on a timeout the thread
// records GPT2_ERR_TIMEOUT, stops issuing work, waits (bounded) for the
// copies and MMAs it already issued, and the CTA frees its tensor memory.
// Epilogue lanes combine their wait results with a warp vote, so a warp
// always takes the same branch.
#pragma once

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                 // one 128-byte swizzle atom of bf16 along K
constexpr int kEpiWarps = 8;            // two per tensor-memory lane quadrant
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kWarpStageBytes = 4096;   // 32 rows x 128 bytes per epilogue warp
constexpr int kSmemLimit = 232448;      // 227 KB opt-in maximum per block

enum Epi : int { EPI_NONE = 0, EPI_BIAS = 1, EPI_GELU = 2, EPI_RES = 3, EPI_LSE = 4, EPI_DZ = 5 };

// BN: output columns per CTA tile; B_COLS: columns of B staged per CTA
// (BN for one CTA, BN / 2 for a pair).
template <int BN, int B_COLS>
struct GemmCfg {
  static constexpr int A_BYTES = kBM * kBK * 2;
  static constexpr int B_BYTES = B_COLS * kBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // the bias of a tile, 16-bit, one buffer per accumulator
  static constexpr int BIAS_BYTES = 2 * BN * 2;
  static constexpr int BAR_BYTES = 192;
  static constexpr int FIXED = 1024 + kEpiWarps * kWarpStageBytes + BIAS_BYTES + BAR_BYTES;
  static constexpr int STAGES_FIT = (kSmemLimit - FIXED) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;  // power of two >= 2 * BN
  static constexpr int SMEM_BYTES = FIXED + STAGES * STAGE_BYTES;
  static_assert(STAGES >= 3, "pipeline too shallow");
  static_assert(SMEM_BYTES <= kSmemLimit, "shared memory");
  static_assert((2 * STAGES + 9) * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(BN % 64 == 0 && BN <= 256 && B_COLS % 64 == 0, "tile width");
};

// Byte offset of 16-byte chunk j of row r in a 128-byte-swizzled staging
// area (8-row groups, chunk index XOR row).
__device__ __forceinline__ uint32_t swz(int r, int j) { return static_cast<uint32_t>(r * 128 + ((j ^ (r & 7)) << 4)); }

template <typename OutT>
struct OutTraits {
  static constexpr int CW = 128 / sizeof(OutT);  // output columns per chunk
  static constexpr int LD = CW / 32;            // tcgen05.ld x32 per chunk
};

template <int EPI, typename OutT, typename T16>
__device__ __forceinline__ void apply_bias_act(float (&v)[OutTraits<OutT>::CW], const T16* __restrict__ bias,
                                               int col0, int N, bool gelu_exact_on = false) {
  constexpr int CW = OutTraits<OutT>::CW;
  if constexpr (EPI != EPI_NONE) {
    // all 16-byte bias loads first (independent, so their latencies
    // overlap), then the adds; a group that crosses column N is read
    // element by element
    uint4 raw[CW / 8];
#pragma unroll
    for (int q = 0; q < CW / 8; ++q) {
      const int c = col0 + q * 8;
      raw[q] = c + 8 <= N ? __ldg(reinterpret_cast<const uint4*>(bias + c)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < CW / 8; ++q) {
      const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = Type16<T16>::unpack2(w[e]);
        v[q * 8 + 2 * e] += f.x;
        v[q * 8 + 2 * e + 1] += f.y;
      }
    }
    if (col0 + CW > N) {
#pragma unroll
      for (int q = 0; q < CW / 8; ++q) {
        const int c = col0 + q * 8;
        if (c < N && c + 8 > N) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (c + e < N) v[q * 8 + e] += to_f32<T16>(bias[c + e]);
        }
      }
    }
  }
  // 16-bit outputs: one hardware tanh per element (absolute error below
  // 2^-11, under the rounding that follows); fp32 outputs: tanhf; the exact
  // GELU (a warp-uniform switch) with erff
  if constexpr (EPI == EPI_GELU) mlp_act_chunk<sizeof(OutT) == 2>(v, gelu_exact_on);
}

// The same with the bias of the chunk read from shared memory (16-bit, zero
// beyond column N), where the epilogue stages each tile's bias once.
template <int EPI, typename OutT, typename T16>
__device__ __forceinline__ void apply_bias_act_smem(float (&v)[OutTraits<OutT>::CW], uint32_t bias_addr,
                                                    bool gelu_exact_on) {
  constexpr int CW = OutTraits<OutT>::CW;
  uint4 raw[CW / 8];
#pragma unroll
  for (int q = 0; q < CW / 8; ++q)
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(raw[q].x), "=r"(raw[q].y), "=r"(raw[q].z), "=r"(raw[q].w)
                 : "r"(bias_addr + q * 16));
#pragma unroll
  for (int q = 0; q < CW / 8; ++q) {
    const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = add_f32x2(make_float2(v[q * 8 + 2 * e], v[q * 8 + 2 * e + 1]), Type16<T16>::unpack2(w[e]));
      v[q * 8 + 2 * e] = f.x;
      v[q * 8 + 2 * e + 1] = f.y;
    }
  }
  if constexpr (EPI == EPI_GELU) mlp_act_chunk<sizeof(OutT) == 2>(v, gelu_exact_on);
}

template <typename OutT, typename T16>
struct EpiArgs {
  const T16* bias;
  const float* residual;
  OutT* out;
  long long ldo;
  int M, N;
  unsigned* err;
  // EPI_LSE: row r's target column is labels[r + 1] unless r % T == T - 1
  // (the next token of the same sequence); part[p * M + r] = (max, sum of
  // exp(z - max)) of row r over column slice p; tgt[r] = z at the target
  const int32_t* labels;
  int T;
  float2* part;
  float* tgt;
  // EPI_GELU: the exact GELU x Phi(x) in place of gelu_new
  int gelu_exact;
  // EPI_DZ: the gradient of the mean shifted cross-entropy with respect to
  // the logits, (softmax(z) - onehot(label)) * inv_n, from each row's
  // log-sum-exp row_lse (natural log); zero in the last row of every
  // sequence (labels, T as for EPI_LSE)
  const float* row_lse;
  float inv_n;
  // split K (EPI_NONE with fp32 output only; M a multiple of 32, so that
  // no 32-row store box crosses into the next slab): S > 1 splits the
  // k-blocks of every tile into S ranges, tile (t, s) accumulating range s
  // and storing its partial into rows s M .. s M + M - 1 of the output (S
  // stacked [M, N] slabs, summed afterwards); 0 or 1: no split
  int splits;
};

// EPI_LSE: one 32-column chunk of a row's logits into the running (m, s) of
// a log-sum-exp (s = sum of exp(z - m) over the columns seen so far;
// columns >= N lie outside the vocabulary and are left out), and the target
// logit when its column falls in the chunk.  exp(z - m) = 2^((z - m) log2 e)
// on the hardware exp2.
__device__ __forceinline__ void lse_chunk(float (&v)[32], int col0, int N, int lbl, float& m, float& s,
                                          float* tgt_row) {
  constexpr float kLog2e = 1.4426950408889634f;
  if (col0 + 32 > N) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i >= N) v[i] = -INFINITY;
  }
  if (lbl >= col0 && lbl < col0 + 32) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) t = (col0 + i == lbl) ? v[i] : t;
    *tgt_row = t;
  }
  float cm = v[0];
#pragma unroll
  for (int i = 1; i < 31; i += 2) cm = max3f(cm, v[i], v[i + 1]);
  cm = fmaxf(cm, v[31]);
  const float nm = fmaxf(m, cm);  // finite: column col0 < N is in the chunk
  const float nml = -nm * kLog2e;
  float2 acc = make_float2(s * ex2_approx(fmaf(m, kLog2e, nml)), 0.f);  // m = -inf at first: 0
  const float2 l2 = make_float2(kLog2e, kLog2e), sh = make_float2(nml, nml);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 e = fma_f32x2(make_float2(v[i], v[i + 1]), l2, sh);
    acc = add_f32x2(acc, make_float2(ex2_approx(e.x), ex2_approx(e.y)));
  }
  m = nm;
  s = acc.x + acc.y;
}

// Epilogue role (warps 2-9).  Tiles tile_begin, tile_begin + tile_stride, ...
// < num_tiles; tile t covers rows (t % m_units) * unit_rows + row_off
// .. + 127 and columns (t / m_units) * BN .. + BN - 1.  Every thread arrives
// once per tile on the accumulator-empty barrier of the tile's accumulator:
// locally, or at a cluster address when CLUSTER_ARRIVE (the barrier of the
// pair's even CTA).
//   The arrival comes after the thread's last read of the tile's
//   accumulator, and means "free for the tile after next".
//   EPI_RES: residual + bias are added at read-out.  A warp loads the
//   residual of its 32 rows for a chunk with coalesced loads one chunk ahead
//   of the read-out (the first chunk of a tile before the wait for its
//   MMAs), and transposes it through its staging area just before the
//   chunk's output goes there: the loads overlap the MMAs, which never wait
//   for them.
template <int BN, int EPI, typename OutT, typename T16, bool CLUSTER_ARRIVE, bool SPLITK>
__device__ __forceinline__ void epilogue_role(const EpiArgs<OutT, T16>& a, const CUtensorMap* tmY, int warp, int lane,
                                              uint32_t stage_base, uint32_t bias_s, uint32_t bias_full0,
                                              uint32_t bias_full1, uint32_t bias_empty0, uint32_t bias_empty1,
                                              uint32_t tmem_base, uint32_t tfull0, uint32_t tfull1, uint32_t tempty0,
                                              uint32_t tempty1, int tile_begin, int tile_stride, int num_tiles,
                                              int m_units, int unit_rows, int row_off) {
  using OT = OutTraits<OutT>;
  constexpr int CW = OT::CW;
  const int quad = warp & 3;  // tensor-memory lanes this warp may access
  const int half = (warp - 2) >> 2;
  const uint32_t stage_w = stage_base + (warp - 2) * kWarpStageBytes;
  const int M = a.M, N = a.N;
  // the staging area is rewritten only once the TMA store of its previous
  // contents has read it
  auto staging_free = [&]() {
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  };
  // one arrival per warp, once all its lanes have read, made by lane 31:
  // lane 0 issues the warp's TMA stores, and an arrival (a release) from
  // that lane waited for its stores in flight to reach memory (3-6k cycles
  // per tile)
  auto arrive_empty = [&](int acc) {
    tc_fence_before();
    __syncwarp();
    if (lane == 31) {
      const uint32_t tempty = acc ? tempty1 : tempty0;
      if (CLUSTER_ARRIVE)
        mbar_arrive_cluster(tempty);
      else
        mbar_arrive(tempty);
    }
  };

  // EPI_RES: the residual of a chunk (32 fp32 columns from col0) of this
  // warp's 32 rows, coalesced: load i of lane L covers row i * 4 + L / 8,
  // columns 4 (L % 8) .. + 3 (four full 128-byte lines per instruction);
  // zero outside [M, N) (N is a multiple of 4)
  auto load_res = [&](float4 (&r)[8], int row0_, int col0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = row0_ + i * 4 + (lane >> 3);
      const int cc = col0 + (lane & 7) * 4;
      r[i] = (rr < M && cc < N) ? __ldg(reinterpret_cast<const float4*>(a.residual + static_cast<long long>(rr) * N + cc))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };

  const int n_splits = SPLITK && a.splits > 1 ? a.splits : 1;
  const int tiles_per_split = num_tiles / n_splits;
  int t_local = 0;
  for (int tile = tile_begin; tile < num_tiles; tile += tile_stride, ++t_local) {
    const int acc = t_local & 1;
    const uint32_t acc_par = (t_local >> 1) & 1;
    const int tt = SPLITK ? tile % tiles_per_split : tile;
    const int row_shift = SPLITK ? (tile / tiles_per_split) * M : 0;  // the split's slab
    const int m0 = (tt % m_units) * unit_rows + row_off;
    const int n0 = (tt / m_units) * BN;
    const int row0 = m0 + quad * 32;  // first row of this warp
    const int valid_cols = N - n0 < BN ? N - n0 : BN;
    const int nch = (valid_cols + CW - 1) / CW;
    // EPI_BIAS / EPI_GELU: the tile's bias into the shared buffer of this
    // accumulator (loaded by warp 2 while the MMAs run; the buffer is free
    // once all eight warps have released it after its previous tile)
    constexpr bool kBiasSmem = EPI == EPI_BIAS || EPI == EPI_GELU || EPI == EPI_RES;
    const uint32_t bias_b = bias_s + acc * (BN * 2);
    if constexpr (kBiasSmem) {
      if (warp == 2) {
        const bool free_ok = t_local < 2 || __all_sync(0xffffffffu, mbar_wait(acc ? bias_empty1 : bias_empty0,
                                                                                acc_par ^ 1));
        if (!free_ok) {
          if (lane == 0) {
            record_error(a.err, kErrTimeout, kSiteGemmEpilogue);
            bulk_wait_group<0>();
          }
          return;
        }
        for (int i = lane; i < BN / 8; i += 32) {
          const int col = n0 + i * 8;
          uint4 u = make_uint4(0u, 0u, 0u, 0u);
          if (col + 8 <= N) {
            u = __ldg(reinterpret_cast<const uint4*>(a.bias + col));
          } else if (col < N) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = Type16<T16>::pack2(col + 2 * e < N ? to_f32<T16>(a.bias[col + 2 * e]) : 0.f,
                                        col + 2 * e + 1 < N ? to_f32<T16>(a.bias[col + 2 * e + 1]) : 0.f);
            u = make_uint4(w[0], w[1], w[2], w[3]);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(bias_b + i * 16), "r"(u.x), "r"(u.y),
                       "r"(u.z), "r"(u.w)
                       : "memory");
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(acc ? bias_full1 : bias_full0);
      }
    }
    float4 res_next[EPI == EPI_RES ? 8 : 1];
    if constexpr (EPI == EPI_RES) {
      if (half < nch) load_res(res_next, row0, n0 + half * CW);
    }
    const bool got = mbar_wait(acc ? tfull1 : tfull0, acc_par);
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) {
        record_error(a.err, kErrTimeout, kSiteGemmEpilogue);
        bulk_wait_group<0>();
      }
      return;
    }
    tc_fence_after();
    if constexpr (kBiasSmem) {
      if (!__all_sync(0xffffffffu, mbar_wait(acc ? bias_full1 : bias_full0, acc_par))) {
        if (lane == 0) {
          record_error(a.err, kErrTimeout, kSiteGemmEpilogue);
          bulk_wait_group<0>();
        }
        return;
      }
    }
    // the last chunk of this half in the tile, after which its accumulator
    // columns are no longer read (-1: none)
    const int last_c = (nch - 1 - half) >= 0 ? nch - 1 - ((nch - 1 - half) & 1) : -1;
    const uint32_t t_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
    if (last_c < 0) arrive_empty(acc);
    // EPI_LSE: this lane's row, its target column (-1: none) and running
    // log-sum-exp over this half's chunks
    const int row = row0 + lane;
    int lbl = -1;
    float lse_m = -INFINITY, lse_s = 0.f;
    if constexpr (EPI == EPI_LSE || EPI == EPI_DZ) {
      if (row < M && row % a.T != a.T - 1) lbl = __ldg(a.labels + row + 1);
    }
    // EPI_DZ: this row's log-sum-exp in log2 units; rows without a target
    // (the last of a sequence, or past M) get zero gradients
    float lse2 = 0.f;
    bool dz_row = false;
    if constexpr (EPI == EPI_DZ) {
      dz_row = row < M && row % a.T != a.T - 1;
      if (dz_row) lse2 = __ldg(a.row_lse + row) * 1.4426950408889634f;
    }
#pragma unroll 1
    for (int c = half; c < nch; c += 2) {
      const int col0 = n0 + c * CW;
      float v[CW];
      {
        uint32_t raw[OT::LD][32];
#pragma unroll
        for (int l = 0; l < OT::LD; ++l) tmem_ld_32x32b_x32(t_addr + c * CW + l * 32, raw[l]);
        tmem_ld_wait();
#pragma unroll
        for (int l = 0; l < OT::LD; ++l)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[l * 32 + i] = __uint_as_float(raw[l][i]);
      }
      if (c == last_c) arrive_empty(acc);  // this half has read its last columns
      if constexpr (EPI == EPI_LSE) {
        lse_chunk(v, col0, N, lbl, lse_m, lse_s, a.tgt + row);
        continue;
      }
      if constexpr (EPI == EPI_DZ) {
        constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          const float p = ex2_approx(fmaf(v[i], kLog2e, -lse2));
          const float g = (p - (col0 + i == lbl ? 1.f : 0.f)) * a.inv_n;
          v[i] = (dz_row && col0 + i < N) ? g : 0.f;
        }
      }
      if constexpr (EPI == EPI_RES) {
        // this chunk's residual transposed through the staging area (row =
        // lane), then the next chunk's loads put in flight
        staging_free();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(stage_w + swz(i * 4 + (lane >> 3), lane & 7)),
                       "f"(res_next[i].x), "f"(res_next[i].y), "f"(res_next[i].z), "f"(res_next[i].w)
                       : "memory");
        __syncwarp();
        if (c + 2 < nch) load_res(res_next, row0, n0 + (c + 2) * CW);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float4 q;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(q.x), "=f"(q.y), "=f"(q.z), "=f"(q.w)
                       : "r"(stage_w + swz(lane, j)));
          v[4 * j] += q.x;
          v[4 * j + 1] += q.y;
          v[4 * j + 2] += q.z;
          v[4 * j + 3] += q.w;
        }
        __syncwarp();  // every lane has read the staging area before it is rewritten below
      }
      if constexpr (kBiasSmem)
        apply_bias_act_smem<EPI, OutT, T16>(v, bias_b + static_cast<uint32_t>(c * CW * 2), a.gelu_exact != 0);
      else if constexpr (EPI == EPI_NONE)
        apply_bias_act<EPI, OutT, T16>(v, a.bias, col0, N);
      // this lane's row (128 bytes) into the staging area (the 128-byte
      // swizzled layout of a [32 x 128 B] TMA box)
      staging_free();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t w0, w1, w2, w3;
        if constexpr (sizeof(OutT) == 2) {
          w0 = Type16<OutT>::pack2(v[8 * j], v[8 * j + 1]);
          w1 = Type16<OutT>::pack2(v[8 * j + 2], v[8 * j + 3]);
          w2 = Type16<OutT>::pack2(v[8 * j + 4], v[8 * j + 5]);
          w3 = Type16<OutT>::pack2(v[8 * j + 6], v[8 * j + 7]);
        } else {
          w0 = __float_as_uint(v[4 * j]);
          w1 = __float_as_uint(v[4 * j + 1]);
          w2 = __float_as_uint(v[4 * j + 2]);
          w3 = __float_as_uint(v[4 * j + 3]);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage_w + swz(lane, j)), "r"(w0), "r"(w1),
                     "r"(w2), "r"(w3)
                     : "memory");
      }
      // and out to global memory by one TMA store of the warp's 32 rows; the
      // tensor map ends at the 16-byte boundary after column N (that padding
      // receives the zeros computed there) and at row M
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && row0 < M) {  // (a box wholly below row M writes nothing)
        tma_store_2d(tmY, stage_w, col0, row0 + row_shift);
        bulk_commit_group();
      }
    }
    if constexpr (kBiasSmem) {
      __syncwarp();
      if (lane == 31) mbar_arrive(acc ? bias_empty1 : bias_empty0);  // this warp has read the tile's bias (lane 0: see arrive_empty)
    }
    if constexpr (EPI == EPI_LSE) {
      // slice (n0 / BN) * 2 + half; lanes write consecutive rows
      if (row < M) a.part[static_cast<long long>((n0 / BN) * 2 + half) * M + row] = make_float2(lse_m, lse_s);
    }
  }
  if (lane == 0) bulk_wait_group<0>();  // this warp's stores are complete
}

// Producer drain: wait for the copies still in flight (the last STAGES
// issued) on the local full barriers.
template <int STAGES, typename FullBar>
__device__ __forceinline__ void drain_loads(long long issued, FullBar full_bar, unsigned* err) {
  const long long first = issued > STAGES ? issued - STAGES : 0;
  for (long long i = first; i < issued; ++i) {
    const int s = static_cast<int>(i % STAGES);
    const uint32_t par = static_cast<uint32_t>((i / STAGES) & 1);
    if (!mbar_wait(full_bar(s), par)) {
      record_error(err, kErrTimeout, kSiteGemmDrain);
      break;
    }
  }
}

// ------------------------------------------------------------------ 1 SM
// One CTA per 128 x BN tile, persistent over the tiles; every CTA loads its
// own A and W tiles (no operand is shared between CTAs).
template <int BN, bool A_MN, bool B_MN, int EPI, typename OutT, typename T16>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_1sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmY, const EpiArgs<OutT, T16> ea, int K) {
  using Cfg = GemmCfg<BN, BN>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  uint8_t* sOut = sB + STAGES * Cfg::B_BYTES;  // per-warp staging areas, 1024-aligned
  uint8_t* sBias = sOut + kEpiWarps * kWarpStageBytes;  // two tiles' bias
  uint64_t* bars = reinterpret_cast<uint64_t*>(sBias + Cfg::BIAS_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 9);
  auto bias_full_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 5 + a); };
  auto bias_empty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 7 + a); };
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 2 + a); };
  const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);
  unsigned* err = ea.err;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int M = ea.M, N = ea.N;
  const int m_tiles = (M + kBM - 1) / kBM;
  const int n_tiles = (N + BN - 1) / BN;
  // split K only in the weight-gradient instantiations (A MN-major)
  constexpr bool kSplit = A_MN;
  const int n_splits = kSplit && ea.splits > 1 ? ea.splits : 1;
  const int tiles_per_split = m_tiles * n_tiles;
  const int num_tiles = tiles_per_split * n_splits;
  const int tile0 = blockIdx.x, tile_step = gridDim.x;
  const int k_blocks = (K + kBK - 1) / kBK;  // k-blocks past K read zeros
  // k-blocks [kb_lo, kb_hi) of a tile (its split's share)
  auto kb_range = [&](int tile, int& kb_lo, int& kb_hi) {
    if constexpr (kSplit) {
      const int sp = tile / tiles_per_split;
      kb_lo = sp * k_blocks / n_splits;
      kb_hi = (sp + 1) * k_blocks / n_splits;
    } else {
      kb_lo = 0;
      kb_hi = k_blocks;
    }
  };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmY);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);  // the MMA commit that has read the stage
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiWarps);  // every epilogue warp, once per tile
      mbar_init(bias_full_bar(a), 1);
      mbar_init(bias_empty_bar(a), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    fence_barrier_init();
  }
  griddep_wait();  // x (and the residual) come from earlier kernels; tensor memory only after they completed
  griddep_launch_dependents();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = tile0; tile < num_tiles && ok; tile += tile_step) {
        const int tt = kSplit ? tile % tiles_per_split : tile;
        const int m0 = (tt % m_tiles) * kBM;
        const int n0 = (tt / m_tiles) * BN;
        int kb_lo, kb_hi;
        kb_range(tile, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1)) {
            record_error(err, kErrTimeout, kSiteGemmProducer);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), Cfg::STAGE_BYTES);
          const uint32_t a_dst = smem_u32(sA + stage * Cfg::A_BYTES);
          if constexpr (A_MN) {
            // A [K, M]: two boxes of 64 M-columns x 64 k-rows
            tma_load_2d(a_dst, &tmA, full_bar(stage), m0, kb * kBK);
            tma_load_2d(a_dst + kBK * 128, &tmA, full_bar(stage), m0 + 64, kb * kBK);
          } else {
            tma_load_2d(a_dst, &tmA, full_bar(stage), kb * kBK, m0);
          }
          const uint32_t b_dst = smem_u32(sB + stage * Cfg::B_BYTES);
          if constexpr (B_MN) {
            // W [K, N]: one box of 64 N-columns x 64 K-rows per 64-wide atom
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(b_dst + j * (kBK * 128), &tmB, full_bar(stage), n0 + j * 64, kb * kBK);
          } else {
            tma_load_2d(b_dst, &tmB, full_bar(stage), kb * kBK, n0);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      drain_loads<STAGES>(issued, full_bar, err);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_f16kind_f32(kBM, BN, A_MN, B_MN, Type16<T16>::kFormat);
      int stage = 0;
      uint32_t phase = 0;
      int t_local = 0;
      bool ok = true;
      bool any = false;
      for (int tile = tile0; tile < num_tiles && ok; tile += tile_step, ++t_local) {
        const int acc = t_local & 1;
        const uint32_t acc_par = (t_local >> 1) & 1;
        // wait for the read-out of the tile before last (none at first)
        if (!mbar_wait(tempty_bar(acc), acc_par ^ 1)) {
          record_error(err, kErrTimeout, kSiteGemmMma);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        int kb_lo, kb_hi;
        kb_range(tile, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(full_bar(stage), phase)) {
            record_error(err, kErrTimeout, kSiteGemmMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * Cfg::A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * Cfg::B_BYTES);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // A K-major: rows of 128 B, 8-row groups 1024 B apart, +32 B per
            // K=16; MN-major: 64-wide M atoms kBK*128 B apart, K=16 = 2048 B
            const uint64_t adesc = A_MN ? sdesc_sw128(a_base + k * 2048, kBK * 128, 1024)
                                        : sdesc_sw128(a_base + k * 32, 16, 1024);
            uint64_t bdesc;
            if constexpr (B_MN) {
              // B MN-major: 64-wide N atoms kBK*128 B apart (LBO), 8-row K
              // groups 1024 B apart (SBO); K=16 spans two groups = 2048 B
              bdesc = sdesc_sw128(b_base + k * 2048, kBK * 128, 1024);
            } else {
              bdesc = sdesc_sw128(b_base + k * 32, 16, 1024);
            }
            umma_bf16(d_tmem, adesc, bdesc, idesc, (kb != kb_lo || k != 0) ? 1u : 0u);
            any = true;
          }
          umma_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
      }
      // wait until every MMA issued has finished writing tensor memory
      if (any) {
        umma_commit(drain_bar);
        if (!mbar_wait(drain_bar, 0)) record_error(err, kErrTimeout, kSiteGemmDrain);
      }
    }
  } else {
    epilogue_role<BN, EPI, OutT, T16, false, A_MN>(ea, &tmY, warp, lane, smem_u32(sOut), smem_u32(sBias), bias_full_bar(0),
                                         bias_full_bar(1), bias_empty_bar(0), bias_empty_bar(1), tmem_base,
                                         tfull_bar(0), tfull_bar(1),
                                         tempty_bar(0), tempty_bar(1), tile0, tile_step, num_tiles, m_tiles, kBM, 0);
  }

  // every warp arrives converged (the producer and MMA roles ran on one lane):
  // a CTA barrier reached by a diverged warp need not hold the others, and
  // the tensor memory is freed only after the epilogue's last read
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------ CTA pair
// Pair tiles of 256 x PBN: PBN = 256 for wide outputs, 192 for the D-wide
// ones (N = 768: 128 tiles for 76 pairs, two rounds of 1.68 tiles, where
// the 256-wide tile leaves 96 tiles and the same two rounds of a longer
// tile).  Each CTA holds 128 rows of the tile and stages PBN / 2 columns of
// B per k-block; with B MN-major those are whole 64-column swizzle atoms
// (128 columns, of which the MMA reads PBN / 2).
constexpr int kPairBN = 256;

template <int PBN, bool A_MN, bool B_MN, int EPI, typename OutT, typename T16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_2sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmY, const EpiArgs<OutT, T16> ea, int K) {
  static_assert(PBN == 256 || PBN == 192, "pair tile width");
  using Cfg = GemmCfg<PBN, 128>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int kBAtoms = (PBN / 2 + 63) / 64;  // MN-major B: 64-column boxes per CTA
  constexpr int kBLoadBytes = B_MN ? kBAtoms * 64 * kBK * 2 : (PBN / 2) * kBK * 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  uint8_t* sOut = sB + STAGES * Cfg::B_BYTES;
  uint8_t* sBias = sOut + kEpiWarps * kWarpStageBytes;  // two tiles' bias
  uint64_t* bars = reinterpret_cast<uint64_t*>(sBias + Cfg::BIAS_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 9);
  auto bias_full_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 5 + a); };
  auto bias_empty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 7 + a); };
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 2 + a); };
  const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);
  unsigned* err = ea.err;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;  // 0: the CTA that issues the MMAs
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const int M = ea.M, N = ea.N;
  const int m_units = (M + 2 * kBM - 1) / (2 * kBM);
  const int n_tiles = (N + PBN - 1) / PBN;
  constexpr bool kSplit = A_MN;  // split K only for the weight gradients
  const int n_splits = kSplit && ea.splits > 1 ? ea.splits : 1;
  const int tiles_per_split = m_units * n_tiles;
  const int num_tiles = tiles_per_split * n_splits;
  const int k_blocks = (K + kBK - 1) / kBK;  // k-blocks past K read zeros
  auto kb_range = [&](int tile, int& kb_lo, int& kb_hi) {
    if constexpr (kSplit) {
      const int sp = tile / tiles_per_split;
      kb_lo = sp * k_blocks / n_splits;
      kb_hi = (sp + 1) * k_blocks / n_splits;
    } else {
      kb_lo = 0;
      kb_hi = k_blocks;
    }
  };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmY);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // the even CTA's expect_tx; both CTAs' bytes
      mbar_init(empty_bar(s), 1);  // the pair MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * kEpiWarps);  // both CTAs' epilogue warps
      mbar_init(bias_full_bar(a), 1);
      mbar_init(bias_empty_bar(a), kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    fence_barrier_init();
  }
  griddep_wait();  // x (and the residual) come from earlier kernels; tensor memory only after they completed
  griddep_launch_dependents();
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before either uses them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs) {
        const int tt = kSplit ? tile % tiles_per_split : tile;
        const int m0 = (tt % m_units) * (2 * kBM) + static_cast<int>(rank) * kBM;
        const int nb = (tt / m_units) * PBN + static_cast<int>(rank) * (PBN / 2);
        int kb_lo, kb_hi;
        kb_range(tile, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1)) {
            record_error(err, kErrTimeout, kSiteGemmProducer);
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(full_bar(stage), 0);  // the even CTA's barrier
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * (Cfg::A_BYTES + kBLoadBytes));
          const uint32_t a_dst = smem_u32(sA + stage * Cfg::A_BYTES);
          if constexpr (A_MN) {
            tma_load_2d_pair(a_dst, &tmA, fb, m0, kb * kBK);
            tma_load_2d_pair(a_dst + kBK * 128, &tmA, fb, m0 + 64, kb * kBK);
          } else {
            tma_load_2d_pair(a_dst, &tmA, fb, kb * kBK, m0);
          }
          const uint32_t b_dst = smem_u32(sB + stage * Cfg::B_BYTES);
          if constexpr (B_MN) {
#pragma unroll
            for (int j = 0; j < kBAtoms; ++j)
              tma_load_2d_pair(b_dst + j * (kBK * 128), &tmB, fb, nb + j * 64, kb * kBK);
          } else {
            tma_load_2d_pair(b_dst, &tmB, fb, kb * kBK, nb);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // the even CTA's full barriers count both CTAs' bytes
      if (rank == 0) drain_loads<STAGES>(issued, full_bar, err);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------ pair MMA issuer
      constexpr uint32_t idesc = idesc_f16kind_f32(2 * kBM, PBN, A_MN, B_MN, Type16<T16>::kFormat);
      constexpr uint16_t kBoth = 0x3;
      int stage = 0;
      uint32_t phase = 0;
      int t_local = 0;
      bool ok = true;
      bool any = false;
      for (int tile = pair; tile < num_tiles && ok; tile += num_pairs, ++t_local) {
        const int acc = t_local & 1;
        const uint32_t acc_par = (t_local >> 1) & 1;
        // wait for the read-out of the tile before last (none at first)
        if (!mbar_wait(tempty_bar(acc), acc_par ^ 1)) {
          record_error(err, kErrTimeout, kSiteGemmMma);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * PBN;
        int kb_lo, kb_hi;
        kb_range(tile, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait(full_bar(stage), phase)) {
            record_error(err, kErrTimeout, kSiteGemmMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * Cfg::A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * Cfg::B_BYTES);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t adesc = A_MN ? sdesc_sw128(a_base + k * 2048, kBK * 128, 1024)
                                        : sdesc_sw128(a_base + k * 32, 16, 1024);
            uint64_t bdesc;
            if constexpr (B_MN) {
              bdesc = sdesc_sw128(b_base + k * 2048, kBK * 128, 1024);
            } else {
              bdesc = sdesc_sw128(b_base + k * 32, 16, 1024);
            }
            umma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb != kb_lo || k != 0) ? 1u : 0u);
            any = true;
          }
          umma_commit_pair_multicast(empty_bar(stage), kBoth);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair_multicast(tfull_bar(acc), kBoth);
      }
      if (any) {
        umma_commit_pair(drain_bar);
        if (!mbar_wait(drain_bar, 0)) record_error(err, kErrTimeout, kSiteGemmDrain);
      }
    }
  } else {
    epilogue_role<PBN, EPI, OutT, T16, true, A_MN>(ea, &tmY, warp, lane, smem_u32(sOut), smem_u32(sBias),
                                            bias_full_bar(0), bias_full_bar(1), bias_empty_bar(0), bias_empty_bar(1),
                                            tmem_base, tfull_bar(0), tfull_bar(1),
                                            mapa_shared(tempty_bar(0), 0), mapa_shared(tempty_bar(1), 0), pair,
                                            num_pairs, num_tiles, m_units, 2 * kBM, static_cast<int>(rank) * kBM);
  }

  __syncwarp();
  tc_fence_before();
  // neither CTA leaves while the pair's MMAs may still read its shared memory
  // or write its tensor memory
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
// Row-major 16-bit [outer, inner] matrix with a row pitch of `pitch`
// elements; boxes of [box_outer, 64] elements, 128-byte swizzle; reads past
// the extents return zeros.
bool make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint64_t pitch, uint32_t box_outer) {
  return encode_tma_2d(map, dt, base, inner, outer, pitch * 2, 64, box_outer);
}

// The operands of one launch: A [M, K] (K contiguous; A_MN: [K, M], M
// contiguous) with a row pitch of lda elements; W [N, K] (K contiguous;
// B_MN: [K, N], N contiguous) with pitch ldw; K the inner extent, any
// positive value (the k-blocks past it read zeros).
template <typename T16>
struct Ops {
  const T16* a;
  long long lda;
  const T16* w;
  long long ldw;
  int K;
};

template <bool A_MN, bool B_MN, typename T16>
bool make_operand_maps(CUtensorMap* ta, CUtensorMap* tb, const Ops<T16>& op, int M, int N, uint32_t b_box) {
  constexpr CUtensorMapDataType dt = Type16<T16>::kTma;
  const uint64_t K = static_cast<uint64_t>(op.K);
  const bool a_ok = A_MN ? make_map(ta, dt, op.a, M, K, op.lda, kBK) : make_map(ta, dt, op.a, K, M, op.lda, kBM);
  const bool b_ok = B_MN ? make_map(tb, dt, op.w, N, K, op.ldw, kBK) : make_map(tb, dt, op.w, K, N, op.ldw, b_box);
  return a_ok && b_ok;
}

// Output y [M, ldo] as the target of the epilogue warps' TMA stores: boxes
// of 32 rows x 128 bytes, 128-byte swizzle; the map ends at the 16-byte
// boundary after column N and at row M.
template <typename OutT>
constexpr CUtensorMapDataType out_tma_type() {
  if constexpr (sizeof(OutT) == 4)
    return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  else
    return Type16<OutT>::kTma;
}
template <typename OutT, typename T16>
bool make_out_map(CUtensorMap* map, const EpiArgs<OutT, T16>& ea) {
  constexpr int esz = static_cast<int>(sizeof(OutT));
  const uint64_t n16 = (static_cast<uint64_t>(ea.N) * esz + 15) / 16 * 16 / esz;
  const uint64_t slabs = ea.splits > 1 ? static_cast<uint64_t>(ea.splits) : 1;
  return encode_tma_2d(map, out_tma_type<OutT>(), ea.out, n16, static_cast<uint64_t>(ea.M) * slabs,
                       static_cast<uint64_t>(ea.ldo) * esz, 128 / esz, 32);
}

template <typename Kern>
cudaError_t set_smem_once(Kern kern, int bytes, int (&configured)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return cudaSuccess;
}

template <int BN, bool A_MN, bool B_MN, int EPI, typename OutT, typename T16>
cudaError_t run_1sm(const Ops<T16>& op, const EpiArgs<OutT, T16>& ea, cudaStream_t stream) {
  using Cfg = GemmCfg<BN, BN>;
  auto kern = gemm_1sm<BN, A_MN, B_MN, EPI, OutT, T16>;
  static int configured[64] = {0};
  cudaError_t e = set_smem_once(kern, Cfg::SMEM_BYTES, configured);
  if (e != cudaSuccess) return e;
  const int M = ea.M, N = ea.N;
  const int m_tiles = (M + kBM - 1) / kBM;
  CUtensorMap ta, tb;
  if (!make_operand_maps<A_MN, B_MN>(&ta, &tb, op, M, N, BN)) return cudaErrorInvalidValue;
  const int tiles = m_tiles * ((N + BN - 1) / BN) * (ea.splits > 1 ? ea.splits : 1);
  const int ctas = tiles < num_sms() ? tiles : num_sms();
  CUtensorMap ty = ta;  // EPI_LSE stores no tile (a valid map, never used)
  if (EPI != EPI_LSE && !make_out_map(&ty, ea)) return cudaErrorInvalidValue;
  return launch_pdl(kern, ctas, kThreads, Cfg::SMEM_BYTES, stream, 0, ta, tb, ty, ea, op.K);
}

template <int PBN, bool A_MN, bool B_MN, int EPI, typename OutT, typename T16>
cudaError_t run_2sm(const Ops<T16>& op, const EpiArgs<OutT, T16>& ea, cudaStream_t stream) {
  using Cfg = GemmCfg<PBN, 128>;
  auto kern = gemm_2sm<PBN, A_MN, B_MN, EPI, OutT, T16>;
  static int configured[64] = {0};
  cudaError_t e = set_smem_once(kern, Cfg::SMEM_BYTES, configured);
  if (e != cudaSuccess) return e;
  const int M = ea.M, N = ea.N;
  CUtensorMap ta, tb;
  if (!make_operand_maps<A_MN, B_MN>(&ta, &tb, op, M, N, PBN / 2)) return cudaErrorInvalidValue;
  // pairs that can be resident at once (a pair needs two SMs of one GPC)
  static int max_pairs[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && max_pairs[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = num_sms() / 2;
    max_pairs[dev] = n < num_sms() / 2 ? n : num_sms() / 2;
  }
  const int pairs_max = (dev >= 0 && dev < 64) ? max_pairs[dev] : num_sms() / 2;
  const int tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + PBN - 1) / PBN) * (ea.splits > 1 ? ea.splits : 1);
  const int pairs = tiles < pairs_max ? tiles : pairs_max;
  CUtensorMap ty = ta;  // EPI_LSE stores no tile (a valid map, never used)
  if (EPI != EPI_LSE && !make_out_map(&ty, ea)) return cudaErrorInvalidValue;
  return launch_pdl(kern, 2 * pairs, kThreads, Cfg::SMEM_BYTES, stream, 0, ta, tb, ty, ea, op.K);
}

// The 256 x 192 pair tile for a D-wide output (N <= 1024) with a long K:
// these products are bound by the operand stream from L2 (M = 8192,
// N = 768, K = 3072: ~500 MB from L2 per launch with 128 x 192 tiles), and
// the pair reads a fifth less per output; at K = 768 the pair's start-up
// costs more than that saves (measured: 37.6 against 38.9 us at K = 3072,
// 16.2 against 14.4 us at K = 768).
bool use_pair192(int M, int N, int K) { return M >= 2 * kBM && N > 128 && N <= 1024 && K >= 2048; }

// Kernel variant for an M x N problem: 0 = CTA pair with 256 x 256 tiles,
// 1 = CTA pair with 256 x 192 tiles, otherwise the tile width of the
// single-CTA kernel.  Measured on the GPT-2 shapes: the pair wins wherever
// the output is wide (c_attn, c_fc, lm_head: its per-SM operand traffic is
// lower); for D-wide outputs (N <= 1024) its 256-wide tiles leave too few
// tiles for 76 pairs: the 192-wide pair tile where use_pair192 says so (and
// the caller offers it: the residual epilogue), else the single-CTA tile
// width that needs the fewest rounds.
constexpr int kVariantPair192 = 1;
int variant_bn(int v) { return v == 0 ? 256 : v == kVariantPair192 ? 192 : v; }
int pick_variant(int M, int N, int K = 0, bool pair192 = false) {
#ifdef GPT2_GEMM_FORCE_BN
  (void)M;
  (void)N;
  (void)K;
  (void)pair192;
  return GPT2_GEMM_FORCE_BN;
#else
  if (M >= 2 * kBM && N > 1024) return 0;
  if (pair192 && use_pair192(M, N, K)) return kVariantPair192;
  const int sms = num_sms();
  int best = 192;
  long long best_cost = -1;
  for (int bn : {192, 128, 256}) {
    const long long tiles = static_cast<long long>((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
    const long long rounds = (tiles + sms - 1) / sms;
    // cycles per k-block: operand bytes at ~60 B per cycle per SM, at least the MMA time
    const long long per_kb = std::max<long long>(bn * 2, (kBM + bn) * kBK * 2 / 60);
    const long long cost = rounds * per_kb;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
#endif
}

template <bool A_MN, bool B_MN, int EPI, typename OutT, typename T16>
cudaError_t run_variant(int v, const Ops<T16>& op, const EpiArgs<OutT, T16>& ea, cudaStream_t s) {
  if constexpr (EPI == EPI_RES) {
    if (v == kVariantPair192) return run_2sm<192, A_MN, B_MN, EPI, OutT, T16>(op, ea, s);
  } else {
    if (v == kVariantPair192) v = 192;
  }
  switch (v) {
    case 0: return run_2sm<kPairBN, A_MN, B_MN, EPI, OutT, T16>(op, ea, s);
    case 128: return run_1sm<128, A_MN, B_MN, EPI, OutT, T16>(op, ea, s);
    case 192: return run_1sm<192, A_MN, B_MN, EPI, OutT, T16>(op, ea, s);
    default: return run_1sm<256, A_MN, B_MN, EPI, OutT, T16>(op, ea, s);
  }
}

}  // namespace

}  // namespace gpt2
