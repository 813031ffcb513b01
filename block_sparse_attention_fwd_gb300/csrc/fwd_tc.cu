// Attention forward with per-(query row, key tile) LSE statistics on tcgen05
// tensor cores (sm_103a), head dim 64 or 128.  The MMA tiles are 128 query
// rows x 128 keys whatever the statistics' tile sizes: with 64-key tiles the
// two halves of each S row are summed separately, one statistic each, and
// with 64-row query tiles the statistics rows are simply stored as rows.
//
// Math: "Introducing BackLite", Backpropagation for attention (S = s Q K^T,
// P = softmax_row(S), O = P V, computed exactly, Using Sparsity); "BackLite"
// README, How It Works, Phase 1: the forward also records, for every query
// row and key tile j, LSE_{r,j} = log sum_{c in tile j} exp(S_rc).  The row
// softmax runs online over the key tiles (Flash Attention explainer, Online
// Softmax): a reference max m and a running sum l; the accumulator is
// rescaled when m moves.  Here m moves only when a tile's max exceeds it by
// more than 2^8 (in base-2 units), so the rescale of O in TMEM is rare; the
// exponentials stay below 2^8 and the result is the same softmax.
//
// One CTA per (pair of 128-row query tiles A and B, head, batch).  TMEM:
// S_A [0,128), S_B [128,256), O_A [256,256+d), O_B [256+d,256+2d).  P (bf16)
// is written over the first 64 columns of its S and read from TMEM by the
// P V product, so P never passes through shared memory.  Warp roles:
//   warp 0     TMA producer: Q_A, Q_B once; K_j into a 3-stage ring and V_j
//              into a 2-stage ring (V one key tile behind K).
//   warp 1     MMA issuer (one thread), TMEM owner.  For key tile j and each
//              query tile t: O_t += P_t(j) V_j, then S_t(j+1) = Q_t K_{j+1}^T,
//              so while one softmax warpgroup works on its tile the tensor
//              core runs the other tile's products.
//   warps 4-7  softmax warpgroup of tile A, warps 8-11 of tile B; thread =
//              query row: S row from TMEM, tile statistic (coalesced 512 B
//              per key tile), P back into TMEM; at the end O = acc / l, LSE.
// Causal and sliding-window attention (the BackLite blog's Nanochat runs,
// "Introducing BackLite", Training Nanochat): a pair visits only the key
// tiles [lo, hi] that hold an attending pair for one of its two query
// tiles; scores of keys a row does not attend are -inf before the max, and
// the statistics of the key tiles outside [lo, hi] are written as -inf.  The
// heaviest pairs (latest query tiles) are launched first.
// Every mbarrier wait is bounded (tc.cuh).
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace bl {

namespace {

using namespace tc;

template <int D>
struct FCfg {
  static constexpr int NK = 3, NV = 2;                  // K and V ring stages
  static constexpr int CHK = D / 64;
  static constexpr int CHUNK = 128 * 128;               // [128 rows][128 B]
  static constexpr int TILE_BYTES = CHUNK * CHK;        // one 128 x d bf16 tile
  static constexpr int OFF_Q = 0;                       // Q_A, Q_B
  static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NK * TILE_BYTES;
  static constexpr int BYTES = OFF_V + NV * TILE_BYTES;
  static constexpr uint32_t T_S = 0, T_O = 256, T_COLS = 512;
  static constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t ID_O = idesc_bf16(128, D, false, true);
  static constexpr float kRescale = 8.f;  // base-2 headroom before O is rescaled
};

struct FBars {
  // done[u % 3] completes when every product up to S(u) has: K_u (read by
  // S(u)) and V_(u-1) (read by PV(u-1)) are free.  One commit per key tile
  // releases both rings.
  uint64_t q, k_full[3], v_full[2], done[3];
  uint64_t s_full[2], p_ready[2], o_done[2];
};

__device__ __forceinline__ bool failed(const int* f) { return *(volatile const int*)f != 0; }

// max that propagates NaN (one operation carries the maximum and the "some
// term is NaN" flag of a reduction)
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Scratch for the tile weights without a statistics output: `nslots` slots
// of [T_c][kRowStride] floats (the two query tiles' 256 rows of every key
// tile, then 4 floats of padding), one per CTA that can be resident at once,
// each claimed with a lock word.  Slots are slot_floats apart (T_c *
// kRowStride for one call; the largest T_c when the launches of a packed
// batch share the slots).
constexpr int kRowStride = 260;
struct RowScratch {
  float* slots;
  int32_t* locks;
  int nslots;
  int64_t slot_floats;
};

// SUB: statistics per 128-key MMA tile (1 for 128-key tiles, 2 for 64-key
// tiles, whose two halves of the S row are summed separately).
// WL: the launch runs under a non-default wait limit (bl_set_wait_limit).
template <int D, int SUB, bool WL>
__global__ void __launch_bounds__(384, 1) fwd_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o,
    float* __restrict__ lse, float* __restrict__ stats, float* __restrict__ logw,
    RowScratch scr, Shape sh, float scale_log2, uint64_t wait_ns) {
  using C = FCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) FBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  __shared__ uint64_t s_wait;      // the launch's wait limit (ns)
  __shared__ int s_loads[2];       // K and V visits whose loads the producer issued
  __shared__ int s_slot;
  __shared__ __align__(16) float s_lse[256];   // the pair's final LSE rows (tile weights)
  __shared__ __align__(8) uint64_t s_wbar[2];   // statistics staging buffers (tile weights)
  __shared__ int s_wissued;                      // the staging copies were requested

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // under causal structure later pairs visit more key tiles: start them first
  const int pair = (sh.causal ? gridDim.x - 1 - blockIdx.x : blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (sh.H / sh.Hk);
  const int Tc = sh.T_c;                  // statistics key tiles (block_k wide)
  const int Tq = (sh.n + 127) / 128;      // 128-row query tiles (the MMA's rows)
  // the second tile of the last pair may lie wholly past the last query tile
  const int ntile = min(2, Tq - 2 * pair);
  // 128-key tiles [j_lo, j_hi] hold an attending pair for tile A or tile B;
  // the rings and barrier phases count visits jj = j - j_lo.  Causal and
  // window structure come with 128 x 128 tiles only.
  int j_lo = 0, j_hi = (sh.n + 127) / 128 - 1;
  if (sh.causal || sh.window) {
    int lo_b, hi_b;
    key_tile_range(sh, 2 * pair, j_lo, j_hi);
    key_tile_range(sh, 2 * pair + ntile - 1, lo_b, hi_b);
    j_hi = hi_b;
  }
  const int nj = j_hi - j_lo + 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars.q, 1);
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.done[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) mbar_init(&bars.v_full[s], 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_ready[t], 128);
      mbar_init(&bars.o_done[t], 1);
    }
    mbar_init(&s_wbar[0], 1);
    mbar_init(&s_wbar[1], 1);
    s_fail = 0;
    s_wait = wait_ns;
    s_loads[0] = s_loads[1] = 0;
    // without a statistics output the rows go to a scratch slot of this CTA's
    // own (claimed from a lock word; at most nslots CTAs are resident at once)
    s_slot = -1;
    if (!stats && logw && scr.slots) {
      // start at this SM's own slot: the CTA that ran here before released it
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      const uint64_t t0 = globaltimer();
      for (int tries = 0;; ++tries) {
        const int sl = (int)((smid + tries) % scr.nslots);
        if (atomicCAS(&scr.locks[sl], 0, 1) == 0) {
          __threadfence();
          s_slot = sl;
          break;
        }
        if (tries % scr.nslots == scr.nslots - 1 && globaltimer() - t0 > kWaitLimitNs) break;
      }
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s_tmem, C::T_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;

  auto fail = [&]() { atomicOr(&s_fail, 1); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_expect_tx(&bars.q, ntile * C::TILE_BYTES);
      for (int t = 0; t < ntile; ++t)
        for (int c = 0; c < C::CHK; ++c)
          tma_load_4d(sm + C::OFF_Q + t * C::TILE_BYTES + c * C::CHUNK, &tm_q, &bars.q, c * 64,
                      h, (2 * pair + t) * 128, b);
      auto load_v = [&](int jv) -> bool {   // jv counts visits
        const int sv = jv % C::NV;
        // V_(jv-2), the slot's previous tile, is free once done for u = jv - 1
        if (jv >= C::NV && !wait_phase<WL>(&bars.done[(jv - 1) % 3], ((jv - 1) / 3) & 1, &s_wait))
          return false;
        mbar_expect_tx(&bars.v_full[sv], C::TILE_BYTES);
        for (int c = 0; c < C::CHK; ++c)
          tma_load_4d(sm + C::OFF_V + sv * C::TILE_BYTES + c * C::CHUNK, &tm_v, &bars.v_full[sv],
                      c * 64, hk, (j_lo + jv) * 128, b);
        return true;
      };
      int k_loads = 0, v_loads = 0;   // visits whose K / V load was issued
      bool ok = true;
      for (int jj = 0; ok && jj <= nj; ++jj) {
        if (jj < nj) {
          const int sk = jj % C::NK;
          // K_(jj-3), the slot's previous tile, is free once done for u = jj - 3
          ok = !failed(&s_fail) &&
               (jj < C::NK || wait_phase<WL>(&bars.done[sk], ((jj - C::NK) / 3) & 1, &s_wait));
          if (!ok) break;
          mbar_expect_tx(&bars.k_full[sk], C::TILE_BYTES);
          for (int c = 0; c < C::CHK; ++c)
            tma_load_4d(sm + C::OFF_K + sk * C::TILE_BYTES + c * C::CHUNK, &tm_k,
                        &bars.k_full[sk], c * 64, hk, (j_lo + jj) * 128, b);
          k_loads = jj + 1;
        }
        if (jj >= 1) {                       // V stays one key tile behind K
          ok = load_v(jj - 1);
          if (ok) v_loads = jj;
        }
      }
      if (!ok) fail();
      s_loads[0] = k_loads;
      s_loads[1] = v_loads;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sQ = saddr(sm + C::OFF_Q), sK = saddr(sm + C::OFF_K);
      const uint32_t sV = saddr(sm + C::OFF_V);
      auto issue_s = [&](int t, int jj) {   // S_t = Q_t K^T of visit jj into S_t
        const uint32_t qb = sQ + t * C::TILE_BYTES, kb = sK + (jj % C::NK) * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          mma_ss(tmem + C::T_S + t * 128, sdesc_sw128(qb + off, 16, 1024),
                 sdesc_sw128(kb + off, 16, 1024), C::ID_S, kk > 0 ? 1u : 0u);
        }
        // S_B's completion is signalled by the key tile's done commit, which
        // follows it: one commit fewer per key tile for the issuing thread
        if (t == 0) mma_commit(&bars.s_full[0]);
      };
      auto issue_pv = [&](int t, int jj) {  // O_t += P_t V of visit jj, P_t read from TMEM
        const uint32_t vb = sV + (jj % C::NV) * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + C::T_O + t * D, tmem + C::T_S + t * 128 + kk * 8,
                 sdesc_sw128(vb + kk * 2048, C::CHUNK, 1024), C::ID_O,
                 (jj > 0 || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_phase<WL>(&bars.q, 0, &s_wait) && wait_phase<WL>(&bars.k_full[0], 0, &s_wait);
      if (ok) {
        fence_after_sync();
        for (int t = 0; t < ntile; ++t) issue_s(t, 0);
        mma_commit(&bars.done[0]);
      }
      for (int jj = 0; ok && jj < nj; ++jj) {
        const bool more = jj + 1 < nj;
        // the three phases the next group needs, tested together so that
        // their shared-memory round trips overlap; a blocking wait only for
        // one that has not completed yet
        const uint32_t kp = ((jj + 1) / C::NK) & 1, vp = (jj / C::NV) & 1;
        const uint32_t rd =
            mbar_test3(saddr(&bars.k_full[(jj + 1) % C::NK]), kp,
                       saddr(&bars.v_full[jj % C::NV]), vp, saddr(&bars.p_ready[0]), jj & 1);
        if (more && !(rd & 1))
          ok = !failed(&s_fail) && wait_phase<WL>(&bars.k_full[(jj + 1) % C::NK], kp, &s_wait);
        if (ok && !(rd & 2)) ok = wait_phase<WL>(&bars.v_full[jj % C::NV], vp, &s_wait);
        for (int t = 0; ok && t < ntile; ++t) {
          ok = (t == 0 && (rd & 4)) || wait_phase<WL>(&bars.p_ready[t], jj & 1, &s_wait);
          if (!ok) break;
          fence_after_sync();
          issue_pv(t, jj);
          // S_t(jj+1) overwrites P_t(jj) in TMEM; it is queued after PV_t(jj)
          if (more) issue_s(t, jj + 1);
        }
        if (!ok) break;
        if (more) mma_commit(&bars.done[(jj + 1) % 3]);   // K_(jj+1) and V_jj are free
      }
      if (!ok) fail();
      for (int t = 0; t < 2; ++t) mma_commit(&bars.o_done[t]);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;                 // tile A (warps 4-7) or B (8-11)
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int row = (2 * pair + t) * 128 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t s_col = lane_base + C::T_S + t * 128;
    const uint32_t o_col = lane_base + C::T_O + t * D;
    const int64_t bh = (int64_t)b * sh.H + h;
    const bool valid_tile = t < ntile;
    // this row's statistic of key tile j lives at st_row[j * st_stride]: in the
    // statistics output, else in the CTA's scratch slot (tile weights only)
    float* st_row = nullptr;
    int st_stride = 0;
    if (stats) {
      st_row = stats + bh * sh.T_c * sh.n_pad + row;
      st_stride = (int)sh.n_pad;
    } else if (s_slot >= 0) {
      st_row = scr.slots + (int64_t)s_slot * scr.slot_floats + t * 128 + r;
      st_stride = kRowStride;
    }
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = valid_tile;
    for (int jj = 0; ok && jj < nj; ++jj) {
      const int j = j_lo + jj;
      // S_A(jj) signals s_full[0]; S_B(jj) the done commit of visit jj
      ok = __all_sync(0xffffffffu,
                      !failed(&s_fail) &&
                          (t == 0 ? wait_phase<WL>(&bars.s_full[0], jj & 1, &s_wait)
                                  : wait_phase<WL>(&bars.done[jj % 3], (jj / 3) & 1, &s_wait)));
      if (!ok) break;
      fence_after_sync();
      uint32_t x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld32(s_col + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]));
      tmem_ld_wait();
      // this row attends keys c_lo..c_hi of the tile: keys that exist, c <= row
      // (causal), c > row - window (window)
      int c_hi = sh.n - j * 128 - 1, c_lo = 0;
      if (sh.causal) c_hi = min(c_hi, row - j * 128);
      if (sh.window) c_lo = row - sh.window + 1 - j * 128;
      if (__any_sync(0xffffffffu, c_hi < 127 || c_lo > 0)) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > c_hi || c < c_lo) x[c] = __float_as_uint(-INFINITY);
      }
      // max over the raw scores (the scale is positive), in base-2 units
      float mr = fmaxf(__uint_as_float(x[0]), __uint_as_float(x[1]));
#pragma unroll
      for (int c = 2; c < 128; c += 2)
        mr = fmax3(mr, __uint_as_float(x[c]), __uint_as_float(x[c + 1]));
      const float mt = mr * scale_log2;
      const bool grow = mt > m_ref + C::kRescale;
      const float m_new = grow ? mt : m_ref;
      const float alpha = grow ? fast_exp2(m_ref - m_new) : 1.f;
      // a row that has attended no key yet keeps m = -inf: its p are 0
      const float m_sub = m_new == -INFINITY ? 0.f : m_new;
      // p = 2^(x s log2 e - m); bf16 pairs packed in place (entry c from 2c,
      // 2c+1).  Arguments and row sums go two columns per instruction: the
      // even and the odd columns' p are summed separately.
      const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-m_sub, -m_sub);
      uint64_t ts2 = f2_pack(0.f, 0.f), ts2_lo = ts2;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float a0, a1;
        f2_unpack(ffma2(f2_pack(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1])), sc2,
                        nm2),
                  a0, a1);
        const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
        if (SUB == 2 && c == 32) {   // keys 0-63 and 64-127: two 64-key tiles
          ts2_lo = ts2;
          ts2 = f2_pack(0.f, 0.f);
        }
        ts2 = fadd2(ts2, f2_pack(p0, p1));
        x[c] = pack_bf16(p0, p1);
      }
      float ts, ts_lo;
      {
        float u0, u1;
        f2_unpack(ts2, u0, u1);
        ts = u0 + u1;
        f2_unpack(ts2_lo, u0, u1);
        ts_lo = u0 + u1;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_st16(s_col + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&x[c * 16]));
      // rows past the statistics' T_r * block_q rows are not stored (with
      // 64-row query tiles and an odd T_r the last 128-row MMA tile reaches
      // 64 rows past them)
      if constexpr (SUB == 1) {
        if (st_row && row < sh.n_pad)
          st_row[(int64_t)j * st_stride] = row < sh.n ? (m_new + __log2f(ts)) * kLn2 : -INFINITY;
      } else {
        if (st_row && row < sh.n_pad) {
          st_row[(int64_t)(2 * j) * st_stride] =
              row < sh.n ? (m_new + __log2f(ts_lo)) * kLn2 : -INFINITY;
          if (2 * j + 1 < Tc)
            st_row[(int64_t)(2 * j + 1) * st_stride] =
                row < sh.n ? (m_new + __log2f(ts)) * kLn2 : -INFINITY;
        }
        ts += ts_lo;
      }
      l_run = l_run * alpha + ts;
      m_ref = m_new;
      // rescale O in TMEM (rare).  S_t(jj) has completed, hence so has
      // PV_t(jj-1): the MMA issuer queues S_t(jj) behind it; PV_t(jj) waits
      // for p_ready.
      if (jj > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t ov[16];
          tmem_ld16(o_col + c0, ov);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st16(o_col + c0, ov);
        }
      }
      tmem_st_wait();
      fence_before_sync();
      mbar_arrive(&bars.p_ready[t]);
    }
    if (valid_tile) {
      if (!ok && lane == 0) fail();
      // key tiles this pair never visits carry no weight for this row
      if (SUB == 1 && stats) {
        for (int j = 0; j < j_lo; ++j) st_row[(int64_t)j * sh.n_pad] = -INFINITY;
        for (int j = j_hi + 1; j < Tc; ++j) st_row[(int64_t)j * sh.n_pad] = -INFINITY;
      }
    }
    // Tile weights of the pair's query tiles: d_ij = max over the tile's rows
    // r < n of fp32(LSE_{r,j} - LSE_r) (NaN if any term is NaN), clamped to
    // <= 0 with -0 -> +0; key tiles outside tile i's attending range enter
    // with LSE_{r,j} = -inf.  Once every MMA has completed the dynamic shared
    // memory is free: the pair's statistics rows (1 KB per key tile: 128 rows
    // of each query tile) come in with bulk copies, in chunks of JB key tiles
    // into two alternating buffers (rows of consecutive key tiles kRowStride
    // floats apart).  The first two chunks are requested before the O rows
    // are written out; the eight softmax warps then reduce chunk by chunk
    // while the next one arrives.  One lane per key tile: a lane runs over the
    // tile's rows with float4 loads (the 16-byte padding per key tile spreads
    // the 32 lanes over all banks) and keeps its own maximum, so nothing
    // waits on another lane.
    const int ww = warp - 4;                         // 0..7
    constexpr int JB = (C::BYTES / 2 / (kRowStride * 4)) / 32 * 32;   // key tiles per buffer
    const int nchunks = (Tc + JB - 1) / JB;
    int lo0 = 0, hi0 = -1, lo1 = 0, hi1 = -1;
    const float* gsrc = nullptr;                     // row block of key tile j: gsrc + j * gstride
    int64_t gstride = 0;
    uint32_t rowbytes = 0;
    bool issuer = false;
    auto issue = [&](int c) {
      const int j0 = c * JB, jn = min(JB, Tc - j0);
      uint8_t* dst = sm + (c & 1) * JB * (kRowStride * 4);
      if (!stats) {   // the slot already has the buffer's layout: one copy
        mbar_expect_tx(&s_wbar[c & 1], (uint32_t)jn * kRowStride * 4u);
        bulk_load(dst, gsrc + (int64_t)j0 * kRowStride, (uint32_t)jn * kRowStride * 4u,
                  &s_wbar[c & 1]);
      } else {
        mbar_expect_tx(&s_wbar[c & 1], (uint32_t)jn * rowbytes);
        for (int jj = 0; jj < jn; ++jj)
          bulk_load(dst + jj * (kRowStride * 4), gsrc + (int64_t)(j0 + jj) * gstride, rowbytes,
                    &s_wbar[c & 1]);
      }
    };
    if (logw) {
      key_tile_range(sh, 2 * pair, lo0, hi0);
      if (ntile == 2) key_tile_range(sh, 2 * pair + 1, lo1, hi1);
      gsrc = stats ? stats + bh * sh.T_c * sh.n_pad + pair * 256
                   : (s_slot >= 0 ? scr.slots + (int64_t)s_slot * scr.slot_floats : nullptr);
      gstride = stats ? sh.n_pad : kRowStride;
      // the pair's rows of a key tile: 256, fewer in the last pair
      rowbytes = (uint32_t)min(256, (int)(sh.n_pad - pair * 256)) * 4u;
      issuer = ww == 0 && lane == 0 && gsrc != nullptr;
      fence_proxy_async_global();   // this thread's statistics, for the copies
      named_sync(1, 256);           // every row's statistics are written
      if (ww == 0 && lane == 0) {
        s_wissued = issuer && mbar_wait(&bars.o_done[0], 0);
        if (s_wissued) {
          issue(0);
          if (nchunks > 1) issue(1);
        }
      }
    }
    if (valid_tile) {
      // epilogue: O = acc / l, LSE = ln 2 (m + log2 l), once the last PV landed
      const bool done = __all_sync(0xffffffffu, ok && wait_phase<WL>(&bars.o_done[t], 0, &s_wait));
      fence_after_sync();
      const float inv = 1.f / l_run;
      __nv_bfloat16* orow = o + bshd(sh.os, b, row, h);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t ov[32];
        if (done) {
          tmem_ld32(o_col + c0, ov);
          tmem_ld_wait();
        }
        if (done && row < sh.n) {
#pragma unroll
          for (int x8 = 0; x8 < 32; x8 += 8) {
            uint4 w = make_uint4(
                pack_bf16(__uint_as_float(ov[x8]) * inv, __uint_as_float(ov[x8 + 1]) * inv),
                pack_bf16(__uint_as_float(ov[x8 + 2]) * inv, __uint_as_float(ov[x8 + 3]) * inv),
                pack_bf16(__uint_as_float(ov[x8 + 4]) * inv, __uint_as_float(ov[x8 + 5]) * inv),
                pack_bf16(__uint_as_float(ov[x8 + 6]) * inv, __uint_as_float(ov[x8 + 7]) * inv));
            *reinterpret_cast<uint4*>(orow + c0 + x8) = w;
          }
        }
      }
      // a forward that gave up on a bounded wait marks its rows' LSE with NaN
      const float lse_v = done ? (m_ref + __log2f(l_run)) * kLn2 : __uint_as_float(0x7fc00000u);
      if (row < sh.n) lse[bh * sh.n + row] = lse_v;
      if (!done && lane == 0) fail();
      if (logw) s_lse[t * 128 + r] = lse_v;
    }
    if (logw) {
      named_sync(1, 256);            // every row's final LSE is in s_lse
      const int qr = sh.block_q;                        // rows per query tile
      const int qt0 = pair * (256 / qr);                // the pair's first query tile
      const int nq = min(256 / qr, sh.T_r - qt0);       // and how many it holds
      const bool ranged = sh.causal || sh.window;       // (128 x 128 tiles only)
      for (int c = 0; c < nchunks; ++c) {
        const int j0 = c * JB, jn = min(JB, Tc - j0);
        const bool have = s_wissued && mbar_wait(&s_wbar[c & 1], (c >> 1) & 1);
        const float* buf = reinterpret_cast<const float*>(sm + (c & 1) * JB * (kRowStride * 4));
        // tasks: (query tile, 32 consecutive key tiles of the chunk); the
        // pair's 256 rows hold 2 query tiles of 128 rows or 4 of 64
        const int ngrp = (jn + 31) / 32;
        for (int task = ww; task < nq * ngrp; task += 8) {
          const int tt = task / ngrp, jl = (task - tt * ngrp) * 32 + lane;
          const int j = j0 + jl;
          const int nv = min(qr, sh.n - (qt0 + tt) * qr);   // valid rows
          const bool in = jl < jn && (!ranged || (j >= (tt ? lo1 : lo0) && j <= (tt ? hi1 : hi0)));
          const float* src = buf + jl * kRowStride + tt * qr;
          const float* lp = s_lse + tt * qr;
          const float ninf = -INFINITY, qnan = __uint_as_float(0x7fc00000u);
          const float4 fill = have ? make_float4(ninf, ninf, ninf, ninf)
                                   : make_float4(qnan, qnan, qnan, qnan);
          float m0 = ninf, m1 = ninf, m2 = ninf, m3 = ninf;
          if (nv == qr) {            // a whole tile: no row checks
#pragma unroll 8
            for (int r4 = 0; r4 < qr; r4 += 4) {
              const float4 v = (in && have) ? *reinterpret_cast<const float4*>(src + r4)
                                            : (in ? fill : make_float4(ninf, ninf, ninf, ninf));
              const float4 l = *reinterpret_cast<const float4*>(lp + r4);
              m0 = max_nan(m0, __fsub_rn(v.x, l.x));
              m1 = max_nan(m1, __fsub_rn(v.y, l.y));
              m2 = max_nan(m2, __fsub_rn(v.z, l.z));
              m3 = max_nan(m3, __fsub_rn(v.w, l.w));
            }
          } else {
            for (int r4 = 0; r4 < nv; r4 += 4) {
              const float4 v = (in && have) ? *reinterpret_cast<const float4*>(src + r4)
                                            : (in ? fill : make_float4(ninf, ninf, ninf, ninf));
              const float4 l = *reinterpret_cast<const float4*>(lp + r4);
              m0 = max_nan(m0, __fsub_rn(v.x, l.x));
              if (r4 + 1 < nv) m1 = max_nan(m1, __fsub_rn(v.y, l.y));
              if (r4 + 2 < nv) m2 = max_nan(m2, __fsub_rn(v.z, l.z));
              if (r4 + 3 < nv) m3 = max_nan(m3, __fsub_rn(v.w, l.w));
            }
          }
          if (jl < jn) {
            const float mx = max_nan(max_nan(m0, m1), max_nan(m2, m3));
            float dv = isnan(mx) ? qnan : fminf(mx, 0.f);
            if (dv == 0.f) dv = 0.f;   // -0 -> +0
            logw[(bh * sh.T_r + qt0 + tt) * (int64_t)Tc + j] = dv;
          }
        }
        named_sync(1, 256);          // every warp is done with this buffer
        if (issuer && s_wissued && c + 2 < nchunks) issue(c + 2);
      }
    }
  }

  fence_before_sync();
  __syncthreads();
  if (failed(&s_fail)) {
    // A role gave up on a wait, so loads and MMAs it meant to consume may still
    // be in flight: the producer waits for the last load of every barrier it
    // armed, the MMA issuer for the commit behind its last MMA, before the
    // tensor memory is freed and the CTA exits.  (Without a failure every
    // load and MMA has been consumed by then.)
    if (warp == 0 && lane == 0) {
      mbar_wait_poll(&bars.q, 0);
      for (int u = s_loads[0] - 1; u >= 0 && u >= s_loads[0] - C::NK; --u)
        mbar_wait_poll(&bars.k_full[u % C::NK], (u / C::NK) & 1);
      for (int u = s_loads[1] - 1; u >= 0 && u >= s_loads[1] - C::NV; --u)
        mbar_wait_poll(&bars.v_full[u % C::NV], (u / C::NV) & 1);
    }
    if (warp == 1 && lane == 0) mbar_wait_poll(&bars.o_done[0], 0);
    fence_before_sync();
    __syncthreads();
  }
  if (warp == 1) tmem_free(tmem, C::T_COLS);
  if (threadIdx.x == 0 && s_slot >= 0) {   // the slot's rows have all been read
    __threadfence();
    atomicExch(&scr.locks[s_slot], 0);
  }
}

template <int D, int SUB, bool WL>
cudaError_t launch_t(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                     float* lse, float* stats, float* logw, RowScratch scr, float scale,
                     bool zero_locks, cudaStream_t st) {
  using C = FCfg<D>;
  CUtensorMap mq, mk, mv;
  if (!make_bshd_map(&mq, q, sh.B, sh.n, sh.H, D, 128, sh.qs) ||
      !make_bshd_map(&mk, k, sh.B, sh.n, sh.Hk, D, 128, sh.ks) ||
      !make_bshd_map(&mv, v, sh.B, sh.n, sh.Hk, D, 128, sh.vs))
    return cudaErrorInvalidValue;
  const int smem = C::BYTES + 1024;
  auto kern = fwd_tc_kernel<D, SUB, WL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (scr.locks && zero_locks) {
    e = cudaMemsetAsync(scr.locks, 0, (size_t)scr.nslots * sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(((sh.n + 127) / 128 + 1) / 2, sh.H, sh.B);
  kern<<<grid, 384, smem, st>>>(mq, mk, mv, (__nv_bfloat16*)o, lse, stats, logw, scr, sh,
                                scale * kLog2e, wait_limit_ns());
  return cudaGetLastError();
}

// CTAs of the forward that can be resident on the current device at once.
template <int D>
int resident_ctas() {
  using C = FCfg<D>;
  const int smem = C::BYTES + 1024;
  auto kern = fwd_tc_kernel<D, 1, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 0;
  int occ = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 384, smem) != cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return occ * sms;
}

}  // namespace

bool fwd_tc_supported(const Shape& sh) {
  return (sh.block_q == 64 || sh.block_q == 128) && (sh.block_k == 64 || sh.block_k == 128) &&
         (sh.d == 64 || sh.d == 128);
}

bool fwd_tile_weights_supported(const Shape& sh) {
  return (sh.block_q == 64 || sh.block_q == 128) && (sh.block_k == 64 || sh.block_k == 128) &&
         (sh.d == 64 || sh.d == 128) && sh.T_c <= 2048;
}

size_t fwd_scratch_bytes(int d, int T_c) {
  const int ns = d == 128 ? resident_ctas<128>() : resident_ctas<64>();
  if (ns <= 0) return 0;
  const size_t locks = ((size_t)ns * sizeof(int32_t) + 255) & ~(size_t)255;
  return locks + (size_t)ns * T_c * kRowStride * sizeof(float);
}

size_t fwd_scratch_bytes(const Shape& sh) { return fwd_scratch_bytes(sh.d, sh.T_c); }

cudaError_t fwd_scratch_clear(int d, void* scratch, cudaStream_t st) {
  const int ns = d == 128 ? resident_ctas<128>() : resident_ctas<64>();
  if (ns <= 0 || !scratch) return cudaErrorInvalidValue;
  return cudaMemsetAsync(scratch, 0, (size_t)ns * sizeof(int32_t), st);
}

cudaError_t launch_fwd_tc(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                          float* lse, float* stats, float* logw, void* scratch, float scale,
                          cudaStream_t st, int slot_tc, bool zero_locks) {
  RowScratch scr{nullptr, nullptr, 0, 0};
  if (logw && !stats) {
    const int ns = sh.d == 128 ? resident_ctas<128>() : resident_ctas<64>();
    if (ns <= 0 || !scratch) return cudaErrorInvalidValue;
    const size_t locks = ((size_t)ns * sizeof(int32_t) + 255) & ~(size_t)255;
    scr.locks = static_cast<int32_t*>(scratch);
    scr.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + locks);
    scr.nslots = ns;
    if (slot_tc <= 0) slot_tc = sh.T_c;
    if (slot_tc < sh.T_c) return cudaErrorInvalidValue;
    scr.slot_floats = (int64_t)slot_tc * kRowStride;
  }
  auto go = [&](auto d_c, auto sub_c, auto wl_c) {
    return launch_t<decltype(d_c)::value, decltype(sub_c)::value, decltype(wl_c)::value>(
        sh, q, k, v, o, lse, stats, logw, scr, scale, zero_locks, st);
  };
  using I64 = std::integral_constant<int, 64>;
  using I128 = std::integral_constant<int, 128>;
  using S1 = std::integral_constant<int, 1>;
  using S2 = std::integral_constant<int, 2>;
  if (wait_limit_ns() != tc::kWaitLimitNs) {
    using W = std::true_type;
    if (sh.block_k == 64) return sh.d == 128 ? go(I128{}, S2{}, W{}) : go(I64{}, S2{}, W{});
    return sh.d == 128 ? go(I128{}, S1{}, W{}) : go(I64{}, S1{}, W{});
  }
  using N = std::false_type;
  if (sh.block_k == 64) return sh.d == 128 ? go(I128{}, S2{}, N{}) : go(I64{}, S2{}, N{});
  return sh.d == 128 ? go(I128{}, S1{}, N{}) : go(I64{}, S1{}, N{});
}

cudaError_t launch_fwd(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                       float* lse, float* stats, float scale, cudaStream_t st) {
  if (!fwd_tc_supported(sh)) return cudaErrorInvalidValue;
  return launch_fwd_tc(sh, q, k, v, o, lse, stats, nullptr, nullptr, scale, st);
}

}  // namespace bl
