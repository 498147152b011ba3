// Causal multi-head self-attention on the 5th-generation tensor cores.
//
//   out[b, i, h*64 + d] = sum_{j <= i} softmax_j(q_i . k_j / sqrt(64)) v_j[d]
//
// ("逐行拆GPT-2源码", GPT2Attention ``_split_heads`` / ``_attn`` /
// ``_merge_heads``; llm.c notes 2.2-2.3: scale 1/sqrt(d_k), future positions
// masked before the softmax, row maximum subtracted.)
//
// Persistent CTAs, four per SM, so that the softmax of some CTAs overlaps
// the tensor-core work of the others; each walks a list of (batch, head,
// tile of 128 queries) items, heaviest first, keeping its tensor memory and
// barriers.  Per key tile of 64:
//   S = Q K^T          tcgen05.mma M=128 N=64 K=64 -> tensor memory (fp32)
//   softmax            4 warps, thread = query row = tensor-memory lane: the
//                      row maximum and sum need no cross-thread exchange;
//                      P = exp2(S * log2(e)/8 - m) written as 16-bit values
//                      over the S columns already read (tcgen05.st)
//   O += P V           tcgen05.mma M=128 N=64 K=64 with A = P read from
//                      tensor memory and V from shared memory (MN-major)
// Tensor memory: S (and P over its first 32 columns) 0-63, O 64-127: 128
// columns per CTA, so four CTAs share an SM's 512.  P.V of a tile is issued
// once its softmax has published P, and the S of the next tile only after
// that P.V has completed (S overwrites P; MMAs into different accumulators
// are not ordered among themselves), so a CTA runs S -> softmax -> P.V in
// turn and the four CTAs of an SM fill each other's gaps.  Q sits in one
// slot, K and V in separate two-slot rings: a K slot is refilled as soon as
// its S has been computed, a V slot once its P.V has.
// The running maximum m is only raised (and O, l rescaled) when a row's new
// maximum exceeds it by more than 8 in the log2 domain; otherwise P may reach
// 2^8, harmless in fp32 sums and 16-bit P.  Key tiles entirely above the
// diagonal or past T are never loaded; 32-key chunks of the diagonal tiles
// are skipped or masked by index.  Q, K, V tiles are read by TMA straight
// from the packed [B*T, 3D] c_attn output (the Q|K|V split and head split are
// the TMA coordinates); the head merge is the store into [B, T, D].
//
// Waits are bounded (common.cuh): a timeout records GPT2_ERR_TIMEOUT and the
// roles unwind; tensor memory is freed on every path.
#include "common.cuh"
#include "internal.h"

namespace gpt2 {

namespace {

constexpr int kHd = 64;
constexpr int kTq = 128;  // queries per item
constexpr int kTk = 64;   // keys per tile
constexpr int kAttnThreads = 192;
constexpr int kAttnCtasPerSm = 4;
constexpr int kRowBytes = kHd * 2;              // one 128-byte swizzled row
constexpr int kQBytes = kTq * kRowBytes;        // 16 KB
constexpr int kKVBytes = kTk * kRowBytes;       // 8 KB (one TMA box)
constexpr int kSmemBytes = 1024 + kQBytes + 4 * kKVBytes + 256;  // Q, K x2, V x2, barriers
constexpr uint32_t kTmemCols = 128;  // S (P over its first 32 columns): 64, O: 64
constexpr uint32_t kSCol = 0;
constexpr uint32_t kPCol = 0;
constexpr uint32_t kOCol = 64;
constexpr float kRescaleLog2 = 8.f;

// Key tiles of query tile qt: those below or on the diagonal, and holding
// at least one key < T.
__device__ __forceinline__ int attn_key_tiles(int qt, int T) {
  const int diag = 2 * qt + 2;
  const int valid = (T + kTk - 1) / kTk;
  return diag < valid ? diag : valid;
}

// Position of the 32-key chunk c of key tile j against the 32 rows of warp
// quadrant `quad` of query tile qt: d = first key - first row.  d <= -32:
// every key is at or before every row (no mask); d == 0: key i of the chunk
// is visible to lane L iff i <= L; d >= 32: no key is visible.
__device__ __forceinline__ int attn_chunk_offset(int j, int c, int qt, int quad) {
  return kTk * j + 32 * c - kTq * qt - 32 * quad;
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Work item w of a launch (heaviest first): query tile n_qt - 1 - w / BH of
// (batch, head) w % BH.  CTA c takes items c, then 2G - 1 - c, 2G + c, ...
// (G CTAs; a snake order, so that the CTAs that took the heaviest items of
// one round take the lightest of the next).
__device__ __forceinline__ int attn_item(int k, int c, int G) {
  return k * G + ((k & 1) ? G - 1 - c : c);
}

template <typename T16>
__global__ void __launch_bounds__(kAttnThreads, kAttnCtasPerSm)
    attn_causal_tc(const __grid_constant__ CUtensorMap tm_qkv, T16* __restrict__ out, float* __restrict__ lse_out,
                   int B, int T, int H, float scale_log2, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem);          // Q (one item)
  const uint32_t sK0 = sQ + kQBytes;           // K slots 0, 1 (key tiles)
  const uint32_t sV0 = sK0 + 2 * kKVBytes;     // V slots 0, 1 (key tiles)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQBytes + 4 * kKVBytes);
  const uint32_t q_full = smem_u32(bars + 0);
  const uint32_t q_empty = smem_u32(bars + 1);
  auto k_full = [&](int s) { return smem_u32(bars + 2 + s); };
  auto k_empty = [&](int s) { return smem_u32(bars + 4 + s); };
  auto v_full = [&](int s) { return smem_u32(bars + 6 + s); };
  auto v_empty = [&](int s) { return smem_u32(bars + 8 + s); };
  const uint32_t s_full = smem_u32(bars + 10);
  const uint32_t p_ready = smem_u32(bars + 11);
  const uint32_t pv_done = smem_u32(bars + 12);
  const uint32_t drain = smem_u32(bars + 13);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int D = H * kHd;
  const int BH = B * H;
  const int n_qt = (T + kTq - 1) / kTq;
  const int n_items = BH * n_qt;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_qkv);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_ready, 4);  // one arrival per softmax warp
    mbar_init(pv_done, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  griddep_wait();  // qkv comes from the kernel before; tensor memory only after it completed
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

  // Barrier phases run on across items: key tile g (counted over all items
  // of this CTA) uses K and V slot g & 1 in its (g >> 1)-th round and the
  // g-th phase of s_full / p_ready / pv_done; item i uses the Q slot in its
  // i-th round.  The producer issues each tile's K ahead of the V of the
  // tile before.
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      struct Item {
        int qt, nkt, row_base, h;
      };
      auto get_item = [&](int kk, Item& it) {
        const int w = attn_item(kk, cta, G);
        if (w >= n_items) return false;
        const int bh = w % BH;
        it.qt = n_qt - 1 - w / BH;
        it.nkt = attn_key_tiles(it.qt, T);
        it.row_base = (bh / H) * T;
        it.h = bh % H;
        return true;
      };
      long long nq = 0, nk = 0, nv = 0;  // loads issued
      auto load_q = [&](int kk, const Item& it) {
        if (!mbar_wait(q_empty, static_cast<uint32_t>(kk & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(q_full, kQBytes);
        const int r0 = it.row_base + it.qt * kTq;
        tma_load_2d(sQ, &tm_qkv, q_full, it.h * kHd, r0);
        tma_load_2d(sQ + kKVBytes, &tm_qkv, q_full, it.h * kHd, r0 + kTk);
        ++nq;
        return true;
      };
      auto load_k = [&](long long gg, const Item& it, int jj) {
        const int sl = static_cast<int>(gg & 1);
        if (!mbar_wait(k_empty(sl), static_cast<uint32_t>((gg >> 1) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(k_full(sl), kKVBytes);
        tma_load_2d(sK0 + sl * kKVBytes, &tm_qkv, k_full(sl), D + it.h * kHd, it.row_base + jj * kTk);
        ++nk;
        return true;
      };
      auto load_v = [&](long long gg, const Item& it, int jj) {
        const int sl = static_cast<int>(gg & 1);
        if (!mbar_wait(v_empty(sl), static_cast<uint32_t>((gg >> 1) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(v_full(sl), kKVBytes);
        tma_load_2d(sV0 + sl * kKVBytes, &tm_qkv, v_full(sl), 2 * D + it.h * kHd, it.row_base + jj * kTk);
        ++nv;
        return true;
      };
      bool ok = true;
      Item cur;
      if (get_item(0, cur)) {
        int k = 0, j = 0;
        long long g = 0;
        ok = load_q(0, cur) && load_k(0, cur, 0);
        while (ok) {
          // the key tile after g: (k, j + 1), or the first of item k + 1
          Item nx = cur;
          int nk_i = k, nj = j + 1;
          bool has_next = true;
          if (nj >= cur.nkt) {
            nk_i = k + 1;
            nj = 0;
            has_next = get_item(nk_i, nx);
          }
          if (has_next) {
            if (nj == 0 && !load_q(nk_i, nx)) {
              ok = false;
              break;
            }
            if (!load_k(g + 1, nx, nj)) {
              ok = false;
              break;
            }
          }
          if (!load_v(g, cur, j)) {
            ok = false;
            break;
          }
          if (!has_next) break;
          cur = nx;
          k = nk_i;
          j = nj;
          ++g;
        }
      }
      if (!ok) record_error(err, kErrTimeout, kSiteAttnProducer);
      // copies still in flight: the last Q and the last (up to two) K and V
      bool drained = true;
      if (nq > 0) drained = mbar_wait(q_full, static_cast<uint32_t>((nq - 1) & 1));
      for (long long x = nk > 2 ? nk - 2 : 0; x < nk && drained; ++x)
        drained = mbar_wait(k_full(static_cast<int>(x & 1)), static_cast<uint32_t>((x >> 1) & 1));
      for (long long x = nv > 2 ? nv - 2 : 0; x < nv && drained; ++x)
        drained = mbar_wait(v_full(static_cast<int>(x & 1)), static_cast<uint32_t>((x >> 1) & 1));
      if (!drained) record_error(err, kErrTimeout, kSiteAttnProducer);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_s = idesc_f16kind_f32(kTq, kTk, false, false, Type16<T16>::kFormat);
      constexpr uint32_t idesc_pv = idesc_f16kind_f32(kTq, kHd, false, true, Type16<T16>::kFormat);
      // Per key tile g: P.V of tile g - 1 once its softmax has published P,
      // then (after that P.V has read P) S of tile g into the same columns.
      bool ok = true;
      bool any = false;
      long long g = 0;
      int prev_j = 0;   // tile index within its item of tile g - 1
      auto pv = [&](long long gp, int jj) {
        const int st = static_cast<int>(gp & 1);
        const uint32_t ph = static_cast<uint32_t>((gp >> 1) & 1);
        if (!mbar_wait(p_ready, static_cast<uint32_t>(gp & 1)) || !mbar_wait(v_full(st), ph)) return false;
        tc_fence_after();
        const uint32_t vb = sV0 + st * kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kTk / 16; ++kk)  // P: 8 tensor-memory columns (16 keys) per K=16
          umma_bf16_ts(tmem + kOCol, tmem + kPCol + kk * 8, sdesc_sw128(vb + kk * 2048, 8192, 1024), idesc_pv,
                       (jj | kk) != 0 ? 1u : 0u);
        umma_commit(pv_done);
        umma_commit(v_empty(st));
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int w = attn_item(k, cta, G);
        if (w >= n_items) break;
        const int qt = n_qt - 1 - w / BH;
        const int nkt = attn_key_tiles(qt, T);
        for (int j = 0; j < nkt && ok; ++j, ++g) {
          if (g > 0) {
            if (!pv(g - 1, prev_j) || !mbar_wait(pv_done, static_cast<uint32_t>((g - 1) & 1))) {
              ok = false;
              break;
            }
          }
          const int st = static_cast<int>(g & 1);
          if (j == 0 && !mbar_wait(q_full, static_cast<uint32_t>(k & 1))) {
            ok = false;
            break;
          }
          if (!mbar_wait(k_full(st), static_cast<uint32_t>((g >> 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kb = sK0 + st * kKVBytes;
#pragma unroll
          for (int kk = 0; kk < kHd / 16; ++kk)
            umma_bf16(tmem + kSCol, sdesc_sw128(sQ + kk * 32, 16, 1024), sdesc_sw128(kb + kk * 32, 16, 1024),
                      idesc_s, kk > 0 ? 1u : 0u);
          umma_commit(s_full);
          umma_commit(k_empty(st));
          if (j == nkt - 1) umma_commit(q_empty);  // the item's last read of its Q
          any = true;
          prev_j = j;
        }
      }
      // the last tile's P.V
      if (ok && g > 0 && !pv(g - 1, prev_j)) ok = false;
      if (!ok) record_error(err, kErrTimeout, kSiteAttnMma);
      if (any) {
        umma_commit(drain);
        if (!mbar_wait(drain, 0)) record_error(err, kErrTimeout, kSiteAttnMma);
      }
    }
  } else {
    // ------------------------------------------------ softmax (warps 2..5)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + kSCol;
    const uint32_t tO = tmem + lane_off + kOCol;
    const uint32_t tP = tmem + lane_off + kPCol;
    const float scale = scale_log2;  // log2(e) times the score scale (1/sqrt(64) for GPT-2)
    bool ok = true;
    long long g = 0;
    for (int k = 0; ok; ++k) {
      const int w = attn_item(k, cta, G);
      if (w >= n_items) break;
      const int qt = n_qt - 1 - w / BH, bh = w % BH;
      const int b = bh / H, h = bh % H;
      const int q = qt * kTq + r;
      const int nkt = attn_key_tiles(qt, T);
      float m_run = -INFINITY;
      float l = 0.f;
      for (int j = 0; j < nkt; ++j, ++g) {
        // S of tile g; the P.V of tile g - 1 completed before it was issued,
        // and this commit covers it, so O is settled too
        const bool got = mbar_wait(s_full, static_cast<uint32_t>(g & 1));
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // One pass per 32-key chunk, each score read once from tensor
        // memory: the chunk's row maximum (masked on the diagonal; the scale
        // is positive, so it is applied once to the maximum), then
        // P = exp2(s * scale - m_run) as 16-bit values written over S
        // columns this thread has already read (chunk c's P lands in columns
        // 16c .. 16c + 15 < 32c + 32), paired fp32 arithmetic, 4 independent
        // pair sums; chunks wholly above the diagonal are written as zeros.
        // m_run is raised only when a chunk's maximum exceeds it by more
        // than 8 (log2 units); then O (from earlier tiles of the item), l,
        // this tile's sums so far and the P already written for chunk 0 are
        // brought to the new maximum first.
        float2 ps[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) ps[e] = make_float2(0.f, 0.f);
        const float2 scale2 = make_float2(scale, scale);
#pragma unroll
        for (int c = 0; c < kTk / 32; ++c) {
          const int d = attn_chunk_offset(j, c, qt, quad);
          uint32_t pk[16];
          if (d > 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = 0u;
          } else {
            uint32_t raw[32];
            tmem_ld_32x32b_x32(tS + c * 32, raw);
            tmem_ld_wait();
            float pm[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pm[e] = -INFINITY;
            if (d == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i <= lane) pm[i & 3] = fmaxf(pm[i & 3], __uint_as_float(raw[i]));
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pm[i & 3] = max3f(pm[i & 3], __uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1]));
            }
            const float mx = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])) * scale;
            const bool raise = mx > m_run + kRescaleLog2;
            // tcgen05.ld / tcgen05.st are warp-collective: the whole warp
            // takes the rescale branch if any of its rows needs it (alpha = 1
            // for the others; alpha = 0 for a row's first keys, m_run = -inf)
            if (__any_sync(0xffffffffu, raise)) {
              const float alpha = raise ? ex2_approx(m_run - mx) : 1.f;
              const float2 alpha2 = make_float2(alpha, alpha);
              l *= alpha;
#pragma unroll
              for (int e = 0; e < 4; ++e) ps[e] = mul_f32x2(ps[e], alpha2);
              if (j > 0) {  // (the item's first P.V overwrites O)
#pragma unroll 1
                for (int h = 0; h < kHd / 16; ++h) {  // 16 columns at a time (the scores stay in registers)
                  uint32_t o[16];
                  tmem_ld_32x32b_x16(tO + h * 16, o);
                  tmem_ld_wait();
#pragma unroll
                  for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st_32x32b_x16(tO + h * 16, o);
                }
              }
              if (c > 0) {  // chunk 0's P, written against the old maximum
                uint32_t p0[16];
                tmem_st_wait();
                tmem_ld_32x32b_x16(tP, p0);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float2 q = Type16<T16>::unpack2(p0[i]);
                  p0[i] = Type16<T16>::pack2(q.x * alpha, q.y * alpha);
                }
                tmem_st_32x32b_x16(tP, p0);
              }
              if (raise) m_run = mx;
            }
            const float2 neg_m2 = make_float2(-m_run, -m_run);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = fma_f32x2(make_float2(__uint_as_float(raw[2 * i]), __uint_as_float(raw[2 * i + 1])),
                                         scale2, neg_m2);
              float2 p2 = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              if (d == 0) {
                if (2 * i > lane) p2.x = 0.f;
                if (2 * i + 1 > lane) p2.y = 0.f;
              }
              ps[i & 3] = add_f32x2(ps[i & 3], p2);
              pk[i] = Type16<T16>::pack2(p2.x, p2.y);
            }
          }
          tmem_st_32x32b_x16(tP + c * 16, pk);
        }
        l += ((ps[0].x + ps[0].y) + (ps[1].x + ps[1].y)) + ((ps[2].x + ps[2].y) + (ps[3].x + ps[3].y));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_ready);
      }
      if (!ok) break;
      // the item's last P.V has completed when pv_done reaches phase g - 1
      if (!__all_sync(0xffffffffu, mbar_wait(pv_done, static_cast<uint32_t>((g - 1) & 1)))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = 1.f / l;
      // the row's log-sum-exp of the scaled scores, in log2 units (for the
      // backward): log2 sum_j 2^(s_j * scale) = m_run + log2 l
      if (lse_out && q < T) lse_out[(static_cast<long long>(b) * H + h) * T + q] = m_run + log2f(l);
      T16* orow = out + (static_cast<long long>(b) * T + q) * D + h * kHd;
#pragma unroll
      for (int c = 0; c < kHd / 32; ++c) {
        uint32_t raw[32];
        tmem_ld_32x32b_x32(tO + c * 32, raw);
        tmem_ld_wait();
        if (q < T) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wv[e] = Type16<T16>::pack2(__uint_as_float(raw[v * 8 + 2 * e]) * inv,
                                         __uint_as_float(raw[v * 8 + 2 * e + 1]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + v * 8) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
      }
      // O is read out before the next item's first P.V (which waits for
      // this warp's first P of that item) overwrites it
      tc_fence_before();
    }
    if (!ok && lane == 0) record_error(err, kErrTimeout, kSiteAttnSoftmax);
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

template <typename T16>
cudaError_t launch_t(const void* qkv, void* out, float* lse, int B, int T, int n_head, float score_scale,
                     cudaStream_t stream) {
  if (B == 0 || T == 0) return cudaSuccess;
  const uint64_t D = static_cast<uint64_t>(n_head) * kHd;
  CUtensorMap map;
  if (!encode_tma_2d(&map, Type16<T16>::kTma, qkv, 3 * D, static_cast<uint64_t>(B) * T, 3 * D * 2, kHd, kTk))
    return cudaErrorInvalidValue;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_causal_tc<T16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  // persistent: four CTAs per SM (the launch bounds, ~50 KB of shared
  // memory and 128 tensor-memory columns each are sized for that), each
  // walking its share of the (batch, head, query tile) items
  const long long items = static_cast<long long>(B) * n_head * ((T + kTq - 1) / kTq);
  const long long resident = static_cast<long long>(kAttnCtasPerSm) * num_sms();
  const int grid = static_cast<int>(items < resident ? items : resident);
  return launch_pdl(attn_causal_tc<T16>, dim3(grid), kAttnThreads, kSmemBytes, stream, 0, map,
                    static_cast<T16*>(out), lse, B, T, n_head, 1.4426950408889634f * score_scale, device_error_word());
}

}  // namespace

cudaError_t launch_attention_tc(gpt2_dtype dt, const void* qkv, void* out, int B, int T, int n_head, float score_scale,
                                cudaStream_t stream, float* lse) {
  if (dt == GPT2_F16) return launch_t<__half>(qkv, out, lse, B, T, n_head, score_scale, stream);
  return launch_t<__nv_bfloat16>(qkv, out, lse, B, T, n_head, score_scale, stream);
}

}  // namespace gpt2
