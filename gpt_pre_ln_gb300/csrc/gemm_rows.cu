// Conv1D / lm_head GEMM for few rows (M <= 128: one token per sequence in a
// decode step) on the tcgen05 tensor cores.
//
//   y[M, N] = epilogue( x[M, K] . W ),  same epilogues and layouts as the
//   large-M kernel (gemm_tcgen05.cu).
//
// With few rows the work is a stream of the weights (1.2 to 77 MB for the
// GPT-2 small shapes) past a small block of activations, so the design is
// about spreading that stream over the SMs:
//   * operands swapped: a 128-feature slice of W is the MMA's M side (A),
//     the M rows of x, padded to MP = 16..128, its N side (B); the
//     accumulator in tensor memory holds y transposed, lane = feature,
//     column = row.  W [K, N] is read MN-major straight from its Conv1D
//     layout, wte [N, K] K-major; x K-major.
//   * split K across a thread-block cluster of S CTAs (S <= 16; more than 8
//     is a non-portable cluster size, all CTAs in one GPC), one
//     128-feature tile per cluster: each CTA multiplies its share of the 64-
//     wide k-blocks; the partial sums are reduce-scattered through
//     distributed shared memory (CTA r of the cluster receives the partials
//     of rows [r*cw, r*cw + cw) from every CTA, adds them and applies the
//     epilogue), so no partial goes through global memory and the result
//     does not depend on timing.
//   * wide outputs (tiles >= half the SM count, e.g. the lm_head's 393
//     tiles) run with S = 1 as a persistent grid over the tiles instead,
//     with two accumulators so the epilogue of one tile overlaps the loads
//     and MMAs of the next.
// Roles: warp 0 TMA producer (one 16 KB weight box or two 8 KB ones plus the
// x box per k-block, into a 3-deep ring), warp 1 tensor-memory allocation
// and MMA issue, warps 2-5 epilogue (warp w reads lanes 32 (w % 4) ..).
// Every mbarrier wait is bounded; on a timeout a role records the error,
// stops, and still reaches the cluster barriers and the final teardown.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kRF = 128;  // output features per tile (MMA M)
constexpr int kRK = 64;   // K per k-block: one 128-byte swizzle atom of 16-bit values
constexpr int kRThreads = 192;
constexpr int kRStages = 3;      // ring depth with a K split (two CTAs per SM)
constexpr int kRStagesMax = 8;   // ring depth of the persistent form (one CTA per SM, no receive area)
#ifndef GPT2_ROWS_MAX_CLUSTER
#define GPT2_ROWS_MAX_CLUSTER 16
#endif
constexpr int kRMaxCluster = 16;                      // receive-area sizing
constexpr int kRClusterCap = GPT2_ROWS_MAX_CLUSTER;  // largest K split launched (<= kRMaxCluster)

enum RowsEpi : int { R_NONE = 0, R_BIAS = 1, R_GELU = 2, R_RES = 3 };

template <int MP>
struct RowsCfg {
  static_assert(MP == 16 || MP == 32 || MP == 64 || MP == 128, "padded rows");
  static constexpr int A_BYTES = kRF * kRK * 2;
  static constexpr int B_BYTES = MP * kRK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // receive area of the split-K reduction: S sources x cw rows x 128 features
  // (S * cw <= M + S - 1 <= MP + kRMaxCluster - 1 rows in all)
  static constexpr int RECV_BYTES = kRF * (MP + kRMaxCluster - 1) * 4;
  // layout: ring (A stages, B stages), receive area (split-K form only),
  // barriers
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM_BYTES = 1024 + kRStages * STAGE_BYTES + RECV_BYTES + BAR_BYTES;
  static constexpr int NST_PERSIST_FIT = (232448 - 1024 - BAR_BYTES) / STAGE_BYTES;
  static constexpr int NST_PERSIST = NST_PERSIST_FIT < kRStagesMax ? NST_PERSIST_FIT : kRStagesMax;
  static constexpr int SMEM_BYTES_PERSIST = 1024 + NST_PERSIST * STAGE_BYTES + BAR_BYTES;
  static constexpr int TMEM_COLS = 2 * MP < 64 ? 64 : 2 * MP;  // two accumulators; x32 loads stay inside
  static_assert((2 * kRStagesMax + 6) * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(NST_PERSIST >= kRStages, "persistent ring");
  static_assert(kRStages * STAGE_BYTES >= MP * kRF * 4, "the partial fits over the ring");
};

template <typename OutT, typename T16>
struct RowsArgs {
  const T16* bias;
  const float* residual;  // [M, N] fp32, row stride N
  OutT* out;              // [M, ldo]; may be null when `cand` is set
  long long ldo;
  int M, N, K;
  unsigned* err;
  // optional (S = 1 only): per row m and per (tile, epilogue warp) q, the
  // largest output value of the warp's 32 features and its lowest index, at
  // cand[m * 4 * n_tiles + q] (value, index bits)
  float2* cand;
  // R_GELU: the exact GELU x Phi(x) in place of gelu_new
  int gelu_exact;
};

// Argmax over the lanes of a warp for 32 rows at once: v[j], i[j] are this
// lane's value and index for row j.  Each of the 5 steps trades half of the
// rows still held with the lane `o` apart; afterwards lane L holds the
// maximum of row L (lowest index on ties) in v[0], i[0].
__device__ __forceinline__ void warp_argmax_rows32(float (&v)[32], int (&i)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int half = 16 >> step;  // rows kept after this step
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float kv = upper ? v[j + half] : v[j];
      const int ki = upper ? i[j + half] : i[j];
      const float sv = upper ? v[j] : v[j + half];
      const int si = upper ? i[j] : i[j + half];
      const float ov = __shfl_xor_sync(0xffffffffu, sv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, si, o);
      const bool take = ov > kv || (ov == kv && oi < ki);
      v[j] = take ? ov : kv;
      i[j] = take ? oi : ki;
    }
  }
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// One output element: bias, activation, residual (the value r, loaded ahead
// by the caller), conversion, store.
template <int EPI, typename OutT, typename T16>
__device__ __forceinline__ void rows_store(const RowsArgs<OutT, T16>& a, int m, int n, float v, float b, float r) {
  if constexpr (EPI != R_NONE) v += b;
  if constexpr (EPI == R_GELU) v = mlp_act<sizeof(OutT) == 2>(v, a.gelu_exact != 0);
  if constexpr (EPI == R_RES) v += r;
  a.out[static_cast<long long>(m) * a.ldo + n] = from_f32<OutT>(v);
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to
// shared memory of a CTA of the cluster; completes the bytes on the mbarrier
// at `bar` (a shared::cluster address in the destination CTA).
__device__ __forceinline__ void bulk_copy_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

template <int MP, bool W_MN, int EPI, typename OutT, typename T16>
__global__ void __launch_bounds__(kRThreads, 1)
    gemm_rows(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const RowsArgs<OutT, T16> ea) {
  using Cfg = RowsCfg<MP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = static_cast<int>(cluster_nctarank());  // K split; 1 = persistent over tiles
  const int nst = S == 1 ? Cfg::NST_PERSIST : kRStages;  // ring depth
  uint8_t* sA = smem;
  uint8_t* sB = sA + nst * Cfg::A_BYTES;
  // split K: this CTA's partial, rows x 128 features fp32, staged over the
  // operand ring once every MMA has completed
  float* part = reinterpret_cast<float*>(smem);
  float* recv = reinterpret_cast<float*>(sB + nst * Cfg::B_BYTES);  // split-K form only
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(recv) + (S > 1 ? Cfg::RECV_BYTES : 0));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kRStagesMax + 6);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kRStagesMax + s); };
  auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * kRStagesMax + a); };
  auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * kRStagesMax + 2 + a); };
  const uint32_t drain_bar = smem_u32(bars + 2 * kRStagesMax + 4);
  const uint32_t recv_bar = smem_u32(bars + 2 * kRStagesMax + 5);
  unsigned* err = ea.err;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int M = ea.M, N = ea.N;
  const int rank = static_cast<int>(cluster_ctarank());
  const int n_tiles = (N + kRF - 1) / kRF;
  const int KB = ea.K / kRK;
  const int kb0 = rank * KB / S, kb1 = (rank + 1) * KB / S;
  const int tile0 = blockIdx.x / S, tile_step = gridDim.x / S;
  const int cw = (M + S - 1) / S;  // rows owned by each CTA of the cluster
  const int own0 = min(M, rank * cw), own1 = min(M, rank * cw + cw);

  // producer state (thread 0).  The weight boxes of the first stages go out
  // before the dependency wait (weights are never written by a kernel), the
  // activation boxes after it.
  int p_stage = 0;
  uint32_t p_phase = 0;
  long long issued = 0;
  int p_tile = tile0, p_kb = kb0;
  auto load_w = [&](int stage, int tile, int kb) {
    const int n0 = tile * kRF;
    const uint32_t a_dst = smem_u32(sA + stage * Cfg::A_BYTES);
    if constexpr (W_MN) {
      // W [K, N]: two boxes of 64 features x 64 k-rows
      tma_load_2d(a_dst, &tmW, full_bar(stage), n0, kb * kRK);
      tma_load_2d(a_dst + kRK * 128, &tmW, full_bar(stage), n0 + 64, kb * kRK);
    } else {
      tma_load_2d(a_dst, &tmW, full_bar(stage), kb * kRK, n0);  // W [N, K]: 128 rows x 64 k
    }
  };
  auto load_x = [&](int stage, int kb) {
    tma_load_2d(smem_u32(sB + stage * Cfg::B_BYTES), &tmX, full_bar(stage), kb * kRK, 0);
  };
  auto advance = [&]() {
    ++issued;
    if (++p_stage == nst) {
      p_stage = 0;
      p_phase ^= 1;
    }
    if (++p_kb == kb1) {
      p_kb = kb0;
      p_tile += tile_step;
    }
  };

  int n_pro = 0;  // stages whose W boxes were loaded before the wait
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    for (int s = 0; s < nst; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    mbar_init(recv_bar, 1);
    fence_barrier_init();
    // the partials of this CTA's rows from all S CTAs (none when S = 1)
    mbar_arrive_expect_tx(recv_bar, S > 1 ? static_cast<uint32_t>(S * (own1 - own0) * kRF * 4) : 0u);
    for (; n_pro < nst && p_tile < n_tiles; ++n_pro) {  // fresh ring: no waits
      mbar_arrive_expect_tx(full_bar(p_stage), Cfg::STAGE_BYTES);
      load_w(p_stage, p_tile, p_kb);
      advance();
    }
  }
  griddep_wait();  // x and the residual come from earlier kernels; tensor memory only after they completed
  griddep_launch_dependents();
  if (threadIdx.x == 0)
    for (int i = 0; i < n_pro; ++i) load_x(i, kb0 + i % (kb1 - kb0));  // stage i holds k-block kb0 + i mod (kb1 - kb0)
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // every CTA of the cluster has started (and initialised its barriers)
  // before any copy into its shared memory (the matching wait comes first)
  cluster_arrive_relaxed();
  bool waited = false;  // this thread's matching cluster wait taken

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      while (p_tile < n_tiles) {
        if (!mbar_wait(empty_bar(p_stage), p_phase ^ 1)) {
          record_error(err, kErrTimeout, kSiteRowsProducer);
          break;
        }
        mbar_arrive_expect_tx(full_bar(p_stage), Cfg::STAGE_BYTES);
        load_w(p_stage, p_tile, p_kb);
        load_x(p_stage, p_kb);
        advance();
      }
      // wait for the copies still in flight
      const long long first = issued > nst ? issued - nst : 0;
      for (long long i = first; i < issued; ++i)
        if (!mbar_wait(full_bar(static_cast<int>(i % nst)), static_cast<uint32_t>((i / nst) & 1))) {
          record_error(err, kErrTimeout, kSiteRowsProducer);
          break;
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_f16kind_f32(kRF, MP, W_MN, false, Type16<T16>::kFormat);
      int stage = 0;
      uint32_t phase = 0;
      int t_local = 0;
      bool ok = true;
      bool any = false;
      for (int tile = tile0; tile < n_tiles && ok; tile += tile_step, ++t_local) {
        const int acc = t_local & 1;
        if (!mbar_wait(tempty_bar(acc), ((t_local >> 1) & 1) ^ 1)) {
          record_error(err, kErrTimeout, kSiteRowsMma);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * MP;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(full_bar(stage), phase)) {
            record_error(err, kErrTimeout, kSiteRowsMma);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * Cfg::A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * Cfg::B_BYTES);
#pragma unroll
          for (int k = 0; k < kRK / 16; ++k) {
            uint64_t adesc;
            if constexpr (W_MN) {
              // features MN-major: 64-feature atoms kRK*128 B apart (LBO),
              // 8-row K groups 1024 B apart (SBO); K=16 spans 2048 B
              adesc = sdesc_sw128(a_base + k * 2048, kRK * 128, 1024);
            } else {
              adesc = sdesc_sw128(a_base + k * 32, 16, 1024);  // K-major rows of 128 B
            }
            const uint64_t bdesc = sdesc_sw128(b_base + k * 32, 16, 1024);
            umma_bf16(d_tmem, adesc, bdesc, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
            any = true;
          }
          umma_commit(empty_bar(stage));
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));
      }
      if (any) {
        umma_commit(drain_bar);
        if (!mbar_wait(drain_bar, 0)) record_error(err, kErrTimeout, kSiteRowsMma);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2-5)
    const int quad = warp & 3;
    const int f = quad * 32 + lane;  // feature of this thread within the tile
    constexpr int kPer16 = 16 / static_cast<int>(sizeof(OutT));
    const int n16 = (N + kPer16 - 1) / kPer16 * kPer16;  // padding up to the 16-byte boundary gets zeros
    int t_local = 0;
    for (int tile = tile0; tile < n_tiles; tile += tile_step, ++t_local) {
      const int acc = t_local & 1;
      const int n = tile * kRF + f;
      float b = 0.f;
      if constexpr (EPI != R_NONE) b = n < N ? to_f32<T16>(ea.bias[n]) : 0.f;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), (t_local >> 1) & 1));
      if (!ok) {
        if (lane == 0) record_error(err, kErrTimeout, kSiteRowsEpilogue);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * MP;
      if (S == 1) {
        for (int c0 = 0; c0 < M; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c0, r);
          float res[32];
          if constexpr (EPI == R_RES) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              res[j] = (c0 + j < M && n < N) ? ea.residual[static_cast<long long>(c0 + j) * N + n] : 0.f;
          }
          tmem_ld_wait();
          if (ea.out) {
            if (n < N) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c0 + j < M)
                  rows_store<EPI, OutT, T16>(ea, c0 + j, n, __uint_as_float(r[j]), b, EPI == R_RES ? res[j] : 0.f);
            } else if (n < n16) {
              for (int j = 0; j < 32 && c0 + j < M; ++j)
                ea.out[static_cast<long long>(c0 + j) * ea.ldo + n] = from_f32<OutT>(0.f);
            }
          }
          if constexpr (EPI == R_NONE) {
            if (ea.cand) {
              float cv[32];
              int ci[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float x = __uint_as_float(r[j]);
                cv[j] = (n < N && x == x) ? x : -INFINITY;  // a NaN never wins, as in argmax_rows
                ci[j] = n;
              }
              warp_argmax_rows32(cv, ci, lane);
              if (c0 + lane < M)
                ea.cand[static_cast<long long>(c0 + lane) * 4 * n_tiles + tile * 4 + quad] =
                    make_float2(cv[0], __int_as_float(ci[0]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc));
      } else {
        // 1. this CTA's partial to shared memory, rows x 128 features
        for (int c0 = 0; c0 < M; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < M) part[(c0 + j) * kRF + f] = __uint_as_float(r[j]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        // 2. rows [r*cw, r*cw + cw) to CTA r, into its slot for this rank
        if (warp == 2) {
          cluster_wait();  // every CTA of the cluster is running
          waited = true;
        }
        if (warp == 2 && lane == 0) {
          const uint32_t part_s = smem_u32(part);
          const uint32_t recv_s = smem_u32(recv) + static_cast<uint32_t>(rank * cw * kRF * 4);
          for (int r = 0; r < S; ++r) {
            const int r0 = min(M, r * cw), r1 = min(M, r * cw + cw);
            if (r1 > r0)
              bulk_copy_s2cluster(mapa_shared(recv_s, r), part_s + static_cast<uint32_t>(r0 * kRF * 4),
                                  static_cast<uint32_t>((r1 - r0) * kRF * 4), mapa_shared(recv_bar, r));
          }
          bulk_commit_group();
        }
        // 3. sum the S partials of this CTA's rows, in rank order
        for (int m0 = own0; m0 < own1; m0 += 8) {
          float res[8];
          if constexpr (EPI == R_RES) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              res[e] = (m0 + e < own1 && n < N) ? ea.residual[static_cast<long long>(m0 + e) * N + n] : 0.f;
          }
          if (m0 == own0) {
            const bool got = __all_sync(0xffffffffu, mbar_wait(recv_bar, 0));
            if (!got) {
              if (lane == 0) record_error(err, kErrTimeout, kSiteRowsEpilogue);
              break;
            }
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int m = m0 + e;
            if (m < own1) {
              if (n < N) {
                float v = 0.f;
#pragma unroll
                for (int s = 0; s < kRMaxCluster; ++s)
                  if (s < S) v += recv[(s * cw + m - own0) * kRF + f];
                rows_store<EPI, OutT, T16>(ea, m, n, v, b, EPI == R_RES ? res[e] : 0.f);
              } else if (n < n16) {
                ea.out[static_cast<long long>(m) * ea.ldo + n] = from_f32<OutT>(0.f);
              }
            }
          }
        }
        if (warp == 2 && lane == 0) bulk_wait_group_read<0>();  // the copies out have read the partial
      }
    }
  }

  __syncwarp();
  if (!waited) cluster_wait();  // the same value for every lane of a warp
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
template <int MP, bool W_MN, int EPI, typename OutT, typename T16>
cudaError_t run_rows(const T16* x, const T16* w, const RowsArgs<OutT, T16>& ea, cudaStream_t stream) {
  using Cfg = RowsCfg<MP>;
  auto kern = gemm_rows<MP, W_MN, EPI, OutT, T16>;
  static int configured[64] = {0};
  static int cluster_ok[64][kRMaxCluster + 1] = {{0}};  // resident clusters per cluster size (-1: none)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         std::max(Cfg::SMEM_BYTES, Cfg::SMEM_BYTES_PERSIST));
    if (e != cudaSuccess) return e;
    // clusters beyond the portable 8 CTAs (all 16 in one GPC)
    if (kRClusterCap > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    configured[dev] = 1;
  }
  constexpr CUtensorMapDataType dt = Type16<T16>::kTma;
  const int M = ea.M, N = ea.N, K = ea.K;
  CUtensorMap tw, tx;
  const bool okw = W_MN ? encode_tma_2d(&tw, dt, w, N, K, static_cast<uint64_t>(N) * 2, 64, kRK)
                        : encode_tma_2d(&tw, dt, w, K, N, static_cast<uint64_t>(K) * 2, kRK, kRF);
  if (!okw || !encode_tma_2d(&tx, dt, x, K, M, static_cast<uint64_t>(K) * 2, kRK, MP)) return cudaErrorInvalidValue;

  const int sms = num_sms();
  const int tiles = (N + kRF - 1) / kRF;
  const int KB = K / kRK;
  // CTAs resident per SM with this shared memory (at least 1)
  const int per_sm = std::max(1, std::min(2, 232448 / (Cfg::SMEM_BYTES + 1024)));
  int S = 1;
  if (2 * tiles < sms && !ea.cand) {  // argmax candidates are made by the single-CTA epilogue
    S = std::min(kRClusterCap, std::min(KB, std::max(1, per_sm * sms / tiles)));
    // the largest cluster size whose clusters all fit at once
    for (; S > 1; --S) {
      int& known = cluster_ok[dev][S];
      if (known == 0) {
        cudaLaunchConfig_t qc = {};
        qc.gridDim = dim3(S * tiles, 1, 1);
        qc.blockDim = dim3(kRThreads, 1, 1);
        qc.dynamicSmemBytes = Cfg::SMEM_BYTES;
        cudaLaunchAttribute qa;
        qa.id = cudaLaunchAttributeClusterDimension;
        qa.val.clusterDim.x = S;
        qa.val.clusterDim.y = 1;
        qa.val.clusterDim.z = 1;
        qc.attrs = &qa;
        qc.numAttrs = 1;
        int n = 0;
        known = (cudaOccupancyMaxActiveClusters(&n, kern, &qc) == cudaSuccess && n > 0) ? n : -1;
      }
      if (known >= tiles) break;
    }
  }
  const unsigned grid = S > 1 ? S * tiles : std::min(tiles, sms);
  const int smem = S > 1 ? Cfg::SMEM_BYTES : Cfg::SMEM_BYTES_PERSIST;
  return launch_pdl(kern, grid, kRThreads, smem, stream, static_cast<unsigned>(S), tw, tx, ea);
}

template <int MP, bool W_MN, typename T16>
cudaError_t rows_dispatch_epi(const T16* x, const T16* w, const T16* bias, const float* residual, void* y, int M,
                              int N, int K, long long ldy, int epi, gpt2_dtype y_t, float2* cand, cudaStream_t s) {
  unsigned* err = device_error_word();
  if (cand) {  // argmax candidates: no epilogue, fp32 output (optional)
    RowsArgs<float, T16> ea{nullptr, nullptr, static_cast<float*>(y), ldy, M, N, K, err, cand};
    return run_rows<MP, W_MN, R_NONE, float, T16>(x, w, ea, s);
  }
  if (epi == R_RES) {
    RowsArgs<float, T16> ea{bias, residual, static_cast<float*>(y), ldy, M, N, K, err, nullptr};
    return run_rows<MP, W_MN, R_RES, float, T16>(x, w, ea, s);
  }
  if (y_t != GPT2_F32) {
    RowsArgs<T16, T16> ea{bias, residual, static_cast<T16*>(y), ldy, M, N, K, err, nullptr};
    ea.gelu_exact = epi == GPT2_EPI_BIAS_GELU_EXACT;
    switch (epi) {
      case R_NONE: return run_rows<MP, W_MN, R_NONE, T16, T16>(x, w, ea, s);
      case R_BIAS: return run_rows<MP, W_MN, R_BIAS, T16, T16>(x, w, ea, s);
      default: return run_rows<MP, W_MN, R_GELU, T16, T16>(x, w, ea, s);
    }
  }
  RowsArgs<float, T16> ea{bias, residual, static_cast<float*>(y), ldy, M, N, K, err, nullptr};
  ea.gelu_exact = epi == GPT2_EPI_BIAS_GELU_EXACT;
  switch (epi) {
    case R_NONE: return run_rows<MP, W_MN, R_NONE, float, T16>(x, w, ea, s);
    case R_BIAS: return run_rows<MP, W_MN, R_BIAS, float, T16>(x, w, ea, s);
    default: return run_rows<MP, W_MN, R_GELU, float, T16>(x, w, ea, s);
  }
}

template <bool W_MN, typename T16>
cudaError_t rows_dispatch(const void* x, const void* w, const void* bias, const float* residual, void* y, int M, int N,
                          int K, long long ldy, int epi, gpt2_dtype y_t, float2* cand, cudaStream_t s) {
  const T16* X = static_cast<const T16*>(x);
  const T16* W = static_cast<const T16*>(w);
  const T16* Bv = static_cast<const T16*>(bias);
  if (M <= 16) return rows_dispatch_epi<16, W_MN, T16>(X, W, Bv, residual, y, M, N, K, ldy, epi, y_t, cand, s);
  if (M <= 32) return rows_dispatch_epi<32, W_MN, T16>(X, W, Bv, residual, y, M, N, K, ldy, epi, y_t, cand, s);
  if (M <= 64) return rows_dispatch_epi<64, W_MN, T16>(X, W, Bv, residual, y, M, N, K, ldy, epi, y_t, cand, s);
  return rows_dispatch_epi<128, W_MN, T16>(X, W, Bv, residual, y, M, N, K, ldy, epi, y_t, cand, s);
}

}  // namespace

cudaError_t launch_gemm_rows_16(gpt2_dtype dt, const void* x, const void* w, const void* bias, const float* residual,
                                void* y, int64_t M, int N, int K, int64_t ldy, bool w_out_in, int epilogue,
                                gpt2_dtype y_t, cudaStream_t stream, float2* argmax_cand) {
  if (M <= 0) return cudaSuccess;
  if (M > kMaxRowsGemm) return cudaErrorInvalidValue;
  const int m = static_cast<int>(M);
  float2* c = argmax_cand;
  if (dt == GPT2_F16)
    return w_out_in ? rows_dispatch<false, __half>(x, w, bias, residual, y, m, N, K, ldy, epilogue, y_t, c, stream)
                    : rows_dispatch<true, __half>(x, w, bias, residual, y, m, N, K, ldy, epilogue, y_t, c, stream);
  return w_out_in
             ? rows_dispatch<false, __nv_bfloat16>(x, w, bias, residual, y, m, N, K, ldy, epilogue, y_t, c, stream)
             : rows_dispatch<true, __nv_bfloat16>(x, w, bias, residual, y, m, N, K, ldy, epilogue, y_t, c, stream);
}

}  // namespace gpt2
