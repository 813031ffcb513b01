// Block-sparse attention backward on tcgen05 tensor cores (sm_103a), 128 x
// 128 tiles, head dim 64 or 128.
//
// Math ("Introducing BackLite", Backpropagation for attention; Using
// Sparsity): for every kept tile pair (query tile i, key tile j)
//   S^T = K_j Q_i^T,  P^T = exp(s S^T - LSE_i),  dP^T = V_j dO_i^T,
//   dS^T = P^T (.) (dP^T - D_i),  dV_j += P^T dO_i,  dK_j += dS^T Q_i,
//   dQ_i += dS K_j,
// with D = rowsum(dO (.) O) from the preprocessing pass; dK and dQ take the
// softmax scale s at the end.  Skipped tiles are never loaded.
//
// One CTA per (key tile j, kv head, batch) walks, for each query head of its
// GQA group, the ascending list of query tiles the mask keeps for j.  Every
// product is a 128 x 128 (x d) tcgen05.mma, the shape whose instructions keep
// the tensor core busiest for M = 128.  TMEM (512 columns):
//   R_S  [0,128)        S^T; after the softmax, P^T (bf16 pairs) in its
//                       columns [0,32) and [64,96), read as the TMEM A operand
//                       of dV += P^T dO
//   R_dP [128,256)      dP^T; after the softmax, the dQ tile dS K
//   dV   [256,256+d)    dK [256+d,256+2d)
// Per tile the issuer queues dV as soon as the softmax has written P^T
// (first phase) and the next tile's S^T right behind it, so S^T runs while
// the softmax forms dS^T (second phase); then dK and dQ once dS^T is in
// shared memory, and the next tile's dP^T once the dQ tile has been drained
// from R_dP.  The tensor core runs them in issue order, which makes every
// reuse safe: S^T of the next tile (into R_S) is queued behind dV, which
// reads P^T from R_S, and dS^T is rewritten only after the next dP^T, hence
// after dK and dQ, have completed.
// Warp roles (16 warps):
//   warp 0      TMA producer: K_j, V_j once; then Q_i into two alternating
//               slots and dO_i into a third (4-D tensor maps, 128-byte
//               swizzle, rows past n read as 0), plus the tile's LSE and D
//               rows; dO's slot frees once dV has read it, so the next dO
//               loads while dK, S^T and dQ run.
//   warp 1      MMA issuer (one thread) and TMEM owner.
//   warps 2-3   at start: copy this CTA's tile lists into shared memory.
//   warps 4-7   softmax, query columns 0-63; warps 8-11 columns 64-127.
//               Thread = key row: S^T, dP^T rows from TMEM -> P^T (TMEM) and
//               dS^T (bf16, swizzled shared memory); at the end they write dV
//               (warps 4-7) and dK (warps 8-11).
//   warps 12-15 dQ drain: thread = query row; the dQ tile goes from TMEM
//               through a 128-byte-swizzled staging buffer into the fp32
//               accumulator with TMA bulk reduce-adds (whole-line L2 adds).
// Registers: the block starts at 128 per thread; warps 0-3 give some back
// (setmaxnreg.dec to 64) so the drain warpgroup can hold a whole 128-column
// dQ row (setmaxnreg.inc to 192): 128*64 + 256*128 + 128*192 = 65536.
// Causal and sliding-window attention ("Introducing BackLite", Training
// Nanochat): P^T entries of (key, query) pairs that do not attend are 0, so
// they add nothing to any gradient; the mask never keeps a tile without an
// attending pair and, without lists, the walk skips such tiles.
// All hand-offs are mbarriers; every wait is bounded (tc.cuh).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace bl {

namespace {

using namespace tc;

template <int D>
struct Cfg {
  static constexpr int NS = 3;                    // tile slots: Q_t in slot t % 2, dO in slot 2
  static constexpr int CHK = D / 64;              // 64-element chunks along d
  static constexpr int CHUNK = 128 * 128;         // [128 rows][128 B]
  static constexpr int TILE = CHUNK * CHK;        // one 128 x d bf16 tile
  static constexpr int DS_BYTES = 2 * CHUNK;      // dS^T [128 keys][128 q] bf16
  static constexpr int STAGE_BYTES = 128 * 128;   // dQ staging: [128 rows][32 fp32]
  static constexpr int LIST_CAP = 2048;           // cached list entries per CTA
  static constexpr int GMAX = 32;                 // heads per GQA group with cached lists
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_RING = OFF_V + TILE;
  static constexpr int OFF_DS = OFF_RING + NS * TILE;
  static constexpr int OFF_STAGE = OFF_DS + DS_BYTES;
  static constexpr int OFF_L = OFF_STAGE + STAGE_BYTES;   // NS x 128 floats: lse*log2e
  static constexpr int OFF_D = OFF_L + NS * 128 * 4;      // NS x 128 floats: D
  static constexpr int OFF_LIST = OFF_D + NS * 128 * 4;   // LIST_CAP ints
  static constexpr int OFF_LCNT = OFF_LIST + LIST_CAP * 4;
  static constexpr int OFF_LBASE = OFF_LCNT + GMAX * 4;
  static constexpr int BYTES = OFF_LBASE + GMAX * 4;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  static constexpr uint32_t T_COLS = 512;
  static constexpr uint32_t ID_SS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
  static constexpr uint32_t ID_G = idesc_bf16(128, D, false, true);      // dV, dK
  static constexpr uint32_t ID_Q = idesc_bf16(128, D, true, true);       // dQ
};

struct Bars {
  uint64_t kv, full[3], empty[3], s_full, dp_full, p1_ready, p2_ready, dq_ready, dq_free, acc;
};

// Load x = 2t brings Q_t, x = 2t + 1 brings dO_t.  Q_t alternates between
// slots 0 and 1 (its last reader, dK_t, frees it); every dO uses slot 2,
// which frees as soon as dV_t (its last reader) completes, so the next dO
// loads while dK_t, S^T and dQ run.
__device__ __forceinline__ int slot_of(int x) { return (x & 1) ? 2 : ((x >> 1) & 1); }
__device__ __forceinline__ uint32_t phase_of(int x) {
  return (uint32_t)(((x & 1) ? (x >> 1) : (x >> 2)) & 1);
}

// Iterates the kept query tiles of key tile j over the heads of one GQA group,
// identically in every role.  Reads the lists from shared memory when they
// were cached there (s_list/s_cnt/s_base), else from global memory.
struct Walk {
  const int32_t* q_idx;
  const int32_t* q_cnt;
  const Shape* sh;
  int j, b, hk, G;
  const int32_t* s_list;   // nullptr: not cached
  const int32_t* s_cnt;
  const int32_t* s_base;
  int gi = 0, li = 0, cnt = -1;
  int h = 0, i = 0;
  bool corrupt = false;
  __device__ bool next() {
    for (;;) {
      if (gi >= G) return false;
      h = hk * G + gi;
      const int64_t bh = (int64_t)b * sh->H + h;
      if (cnt < 0) {
        if (s_list) {
          cnt = s_cnt[gi];
        } else {
          cnt = q_cnt ? q_cnt[bh * sh->T_c + j] : sh->T_r;
          if (cnt < 0 || cnt > sh->T_r) {
            corrupt = true;
            cnt = 0;
          }
        }
        li = 0;
      }
      if (li >= cnt) {
        ++gi;
        cnt = -1;
        continue;
      }
      if (s_list)
        i = s_list[s_base[gi] + li];
      else
        i = q_idx ? q_idx[(bh * sh->T_c + j) * (int64_t)sh->T_r + li] : li;
      ++li;
      if (i < 0 || i >= sh->T_r) {
        corrupt = true;
        continue;
      }
      if (!q_idx && tile_empty(*sh, i, j)) continue;   // dense walk: nothing attends
      return true;
    }
  }
};

__device__ __forceinline__ bool failed(const int* f) { return *(volatile const int*)f != 0; }

// MASKED: causal / sliding-window element masks are compiled in.
template <int D, bool MASKED>
__global__ void __launch_bounds__(512, 1) bwd_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_gk,
    const __grid_constant__ CUtensorMap tm_gv, const float* __restrict__ lse,
    const float* __restrict__ Dv, const int32_t* __restrict__ q_idx,
    const int32_t* __restrict__ q_cnt, __nv_bfloat16* __restrict__ g_k,
    __nv_bfloat16* __restrict__ g_v, int32_t* __restrict__ status, Shape sh, float scale,
    float scale_log2) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail, s_cached;
  __shared__ int s_drain_ok[4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int G = sh.H / sh.Hk;

  if (threadIdx.x == 0) {
    mbar_init(&bars.kv, 1);
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&bars.full[s], 33);   // 32 producer lanes + the expect_tx arrival
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.p1_ready, 256);
    mbar_init(&bars.p2_ready, 256);
    mbar_init(&bars.dq_ready, 1);
    mbar_init(&bars.dq_free, 128);
    mbar_init(&bars.acc, 1);
    s_fail = 0;
    fence_mbar_init();
    // K_j, V_j start loading before the lists are copied and TMEM allocated
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_g);
    mbar_expect_tx(&bars.kv, 2 * C::TILE);
    for (int c = 0; c < C::CHK; ++c) {
      tma_load_4d(sm + C::OFF_K + c * C::CHUNK, &tm_k, &bars.kv, c * 64, hk, j * 128, b);
      tma_load_4d(sm + C::OFF_V + c * C::CHUNK, &tm_v, &bars.kv, c * 64, hk, j * 128, b);
    }
  }
  if (warp == 1) tmem_alloc(&s_tmem, C::T_COLS);
  int32_t* s_list = reinterpret_cast<int32_t*>(sm + C::OFF_LIST);
  int32_t* s_lcnt = reinterpret_cast<int32_t*>(sm + C::OFF_LCNT);
  int32_t* s_lbase = reinterpret_cast<int32_t*>(sm + C::OFF_LBASE);
  if (warp == 2 || warp == 3) {
    // copy this CTA's lists (all heads of the GQA group) into shared memory
    const int t = threadIdx.x - 64;
    const bool can = q_idx != nullptr && G <= C::GMAX;
    if (can) {
      for (int g = t; g < G; g += 64) {
        int c = q_cnt[((int64_t)b * sh.H + hk * G + g) * sh.T_c + j];
        if (c < 0 || c > sh.T_r) {
          c = 0;
          atomicOr(status, kStatusCorrupt);
        }
        s_lcnt[g] = c;
      }
    }
    named_sync(2, 64);
    if (t == 0) {
      int tot = 0;
      if (can)
        for (int g = 0; g < G; ++g) {
          s_lbase[g] = tot;
          tot += s_lcnt[g];
        }
      s_cached = can && tot <= C::LIST_CAP;
    }
    named_sync(2, 64);
    if (s_cached) {
      for (int g = 0; g < G; ++g) {
        const int32_t* src =
            q_idx + (((int64_t)b * sh.H + hk * G + g) * sh.T_c + j) * (int64_t)sh.T_r;
        for (int li = t; li < s_lcnt[g]; li += 64) s_list[s_lbase[g] + li] = src[li];
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;

  auto fail = [&]() {
    atomicOr(&s_fail, 1);
    atomicOr(status, kStatusTimeout);
  };
  const bool cached = s_cached != 0;
  Walk walk{q_idx, q_cnt, &sh, j, b, hk, G, cached ? s_list : nullptr, s_lcnt, s_lbase};
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    int x = 0;   // load index: 2t for Q of tile t, 2t+1 for its dO
    bool ok = true;
    while (ok && walk.next()) {
      const int64_t bh = (int64_t)b * sh.H + walk.h;
      const int r0 = walk.i * 128;
      for (int which = 0; which < 2 && ok; ++which, ++x) {
        const int s = slot_of(x);
        float lv[4], dv[4];
        if (which == 0) {   // this tile's LSE and D travel with its Q slot
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = r0 + lane + 32 * e;
            const bool in = r < sh.n;
            lv[e] = in ? lse[bh * sh.n + r] * kLog2e : INFINITY;
            dv[e] = in ? Dv[bh * sh.n + r] : 0.f;
          }
        }
        ok = !failed(&s_fail) && mbar_wait(&bars.empty[s], phase_of(x) ^ 1);
        if (!ok) break;
        if (lane == 0) {
          mbar_expect_tx(&bars.full[s], C::TILE);
          for (int c = 0; c < C::CHK; ++c)
            tma_load_4d(sm + C::OFF_RING + s * C::TILE + c * C::CHUNK, which ? &tm_g : &tm_q,
                        &bars.full[s], c * 64, walk.h, r0, b);
        }
        if (which == 0) {
          float* sl = reinterpret_cast<float*>(sm + C::OFF_L) + s * 128;
          float* sd = reinterpret_cast<float*>(sm + C::OFF_D) + s * 128;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sl[lane + 32 * e] = lv[e];
            sd[lane + 32 * e] = dv[e];
          }
        }
        mbar_arrive(&bars.full[s]);
      }
    }
    if (!ok && lane == 0) fail();
    if (lane == 0 && walk.corrupt) atomicOr(status, kStatusCorrupt);
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sK = saddr(sm + C::OFF_K), sV = saddr(sm + C::OFF_V);
      const uint32_t sR = saddr(sm + C::OFF_RING), sDS = saddr(sm + C::OFF_DS);
      auto slot_addr = [&](int xx) { return sR + slot_of(xx) * C::TILE; };
      auto issue_s = [&](int t) {      // S^T = K Q_t^T  -> R_S
        const uint32_t qb = slot_addr(2 * t);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          mma_ss(tmem + C::T_S, sdesc_sw128(sK + off, 16, 1024),
                 sdesc_sw128(qb + off, 16, 1024), C::ID_SS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full);
      };
      auto issue_dp = [&](int t) {     // dP^T = V dO_t^T -> R_dP
        const uint32_t gb = slot_addr(2 * t + 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          mma_ss(tmem + C::T_DP, sdesc_sw128(sV + off, 16, 1024),
                 sdesc_sw128(gb + off, 16, 1024), C::ID_SS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.dp_full);
      };
      auto wait_slot = [&](int xx) {
        return mbar_wait(&bars.full[slot_of(xx)], phase_of(xx));
      };
      bool ok = mbar_wait(&bars.kv, 0);
      int t = 0;
      bool have = ok && walk.next();
      if (have) {
        ok = wait_slot(0);
        if (ok) {
          fence_after_sync();
          issue_s(0);
          ok = wait_slot(1);
          if (ok) {
            fence_after_sync();
            issue_dp(0);
          }
        }
      }
      while (ok && have) {
        // dV_t as soon as the first softmax phase has written P^T; it runs
        // while the second phase forms dS^T
        ok = !failed(&s_fail) && mbar_wait(&bars.p1_ready, t & 1);
        if (!ok) break;
        fence_after_sync();
        const uint32_t qb = slot_addr(2 * t), gb = slot_addr(2 * t + 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {      // dV += P^T dO  (P^T from TMEM)
          const uint32_t pcol = C::T_S + (kk >> 2) * 64 + (kk & 3) * 8;
          mma_ts(tmem + C::T_DV, tmem + pcol, sdesc_sw128(gb + kk * 2048, C::CHUNK, 1024),
                 C::ID_G, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars.empty[2]);           // dO_t's slot: dP^T and dV have read it
        // S^T of the next tile right behind dV (which read P^T from R_S): it
        // runs while the softmax forms dS^T, so the first softmax phase of the
        // next tile can start as soon as the second phase of this one ends
        have = walk.next();
        if (have) {
          ok = wait_slot(2 * (t + 1));
          if (!ok) break;
          fence_after_sync();
          issue_s(t + 1);
        }
        // dK_t once dS^T is in shared memory
        ok = mbar_wait(&bars.p2_ready, t & 1);
        if (!ok) break;
        fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)        // dK += dS^T Q
          mma_ss(tmem + C::T_DK,
                 sdesc_sw128(sDS + (kk >> 2) * C::CHUNK + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(qb + kk * 2048, C::CHUNK, 1024), C::ID_G,
                 (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.empty[t & 1]);       // Q_t's slot
        // dQ = dS K into R_dP (dP^T was consumed by the softmax)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + C::T_DP, sdesc_sw128(sDS + kk * 2048, C::CHUNK, 1024),
                 sdesc_sw128(sK + kk * 2048, C::CHUNK, 1024), C::ID_Q, kk > 0 ? 1u : 0u);
        mma_commit(&bars.dq_ready);
        if (have) {
          // dP^T of the next tile once the dQ tile has left R_dP; the dS^T
          // buffer is rewritten only after dP^T completes, hence after dQ
          ok = mbar_wait(&bars.dq_free, t & 1) && wait_slot(2 * (t + 1) + 1);
          if (!ok) break;
          fence_after_sync();
          issue_dp(t + 1);
        }
        ++t;
      }
      if (!ok) fail();
      mma_commit(&bars.acc);
    }
   }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax
    const int half = (warp - 4) >> 2;           // query columns [64 half, 64 half + 64)
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;               // key row within the tile
    const bool key_ok = j * 128 + r < sh.n;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    uint8_t* ds_row = sm + C::OFF_DS + half * C::CHUNK + r * 128;
    int t = 0;
    bool ok = true;
    while (ok && walk.next()) {
      const int s = t & 1;                      // Q_t's slot: its LSE and D rows
      // phase 1: P^T from S^T (needs only S^T), written back over S^T
      ok = __all_sync(0xffffffffu, !failed(&s_fail) &&
                                       mbar_wait(&bars.full[s], (t >> 1) & 1) &&
                                       mbar_wait(&bars.s_full, t & 1));
      if (!ok) break;
      fence_after_sync();
      const float* sl = reinterpret_cast<const float*>(sm + C::OFF_L) + s * 128 + half * 64;
      const float* sd = reinterpret_cast<const float*>(sm + C::OFF_D) + s * 128 + half * 64;
      // this key row attends query columns q_lo..q_hi of the warpgroup's 64:
      // query >= key (causal) and query < key + window (window)
      const int kq = j * 128 + r - walk.i * 128 - half * 64;
      const int q_lo = MASKED && sh.causal ? kq : 0;
      const int q_hi = MASKED && sh.window ? kq + sh.window - 1 : 63;
      const bool diag = MASKED && __any_sync(0xffffffffu, q_lo > 0 || q_hi < 63);
      float pf[64];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {          // 32 query columns -> 16 packed
        uint32_t pk[16];
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {     // 16 query columns per load
          const int c0 = h2 * 32 + sub * 16;
          uint32_t sv[16];
          tmem_ld16(lane_base + C::T_S + half * 64 + c0, sv);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 l4 = reinterpret_cast<const float4*>(sl + c0)[c4];
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              const int c = 4 * c4 + y;
              pf[c0 + c] =
                  key_ok ? fast_exp2(fmaf(__uint_as_float(sv[c]), scale_log2, -lv[y])) : 0.f;
            }
          }
          if (diag) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              if (c0 + c < q_lo || c0 + c > q_hi) pf[c0 + c] = 0.f;
          }
#pragma unroll
          for (int c2 = 0; c2 < 8; ++c2)
            pk[sub * 8 + c2] = pack_bf16(pf[c0 + 2 * c2], pf[c0 + 2 * c2 + 1]);
        }
        // P^T pairs over this warpgroup's own S^T columns (already read)
        tmem_st16(lane_base + C::T_S + half * 64 + h2 * 16, pk);
      }
      tmem_st_wait();
      fence_before_sync();
      mbar_arrive(&bars.p1_ready);               // dV_t may read P^T now
      // phase 2: dS^T = P^T (dP^T - D) once dP^T has landed
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.dp_full, t & 1));
      if (!ok) break;
      fence_after_sync();
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {    // 16 query columns per pass
        uint32_t pv[16];
        tmem_ld16(lane_base + C::T_DP + half * 64 + pass * 16, pv);
        tmem_ld_wait();
        uint32_t dk[8];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const float4 d4 = reinterpret_cast<const float4*>(sd + pass * 16)[c4];
          const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
          float ds[4];
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const int c = 4 * c4 + y;
            ds[y] = pf[pass * 16 + c] * (__uint_as_float(pv[c]) - dv[y]);
          }
          dk[2 * c4] = pack_bf16(ds[0], ds[1]);
          dk[2 * c4 + 1] = pack_bf16(ds[2], ds[3]);
        }
        // dS^T, K-major [key][q] with the 128-byte swizzle, 2 x 16 B chunks
#pragma unroll
        for (int c16 = 0; c16 < 2; ++c16) {
          const int chunk = pass * 2 + c16;
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(dk[4 * c16], dk[4 * c16 + 1], dk[4 * c16 + 2], dk[4 * c16 + 3]);
        }
      }
      fence_async_smem();
      fence_before_sync();
      mbar_arrive(&bars.p2_ready);               // dK_t and dQ_t may read dS^T
      ++t;
    }
    if (!ok && lane == 0) fail();
    // epilogue: warps 4-7 write dV, warps 8-11 dK (scaled), rows of this key tile
    const bool acc_ok = mbar_wait(&bars.acc, 0);
    fence_after_sync();
    const bool have = __all_sync(0xffffffffu, ok && acc_ok) && t > 0;
    // Stage the bf16 rows in ring slot `half` (free: every load has been
    // consumed by the finished MMAs) with the 128-byte swizzle and store them
    // with TMA, which drops rows past n.
    const float mul = half == 0 ? 1.f : scale;
    const uint32_t col = half == 0 ? C::T_DV : C::T_DK;
    uint8_t* stg = sm + C::OFF_RING + half * C::TILE;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t a[32];
      if (have) {  // warp-uniform: the TMEM loads are warp-collective
        tmem_ld32(lane_base + col + c0, a);
        tmem_ld_wait();
      }
      uint8_t* row_base = stg + (c0 >> 6) * C::CHUNK + r * 128;
#pragma unroll
      for (int x8 = 0; x8 < 32; x8 += 8) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (have)
          w = make_uint4(
              pack_bf16(__uint_as_float(a[x8]) * mul, __uint_as_float(a[x8 + 1]) * mul),
              pack_bf16(__uint_as_float(a[x8 + 2]) * mul, __uint_as_float(a[x8 + 3]) * mul),
              pack_bf16(__uint_as_float(a[x8 + 4]) * mul, __uint_as_float(a[x8 + 5]) * mul),
              pack_bf16(__uint_as_float(a[x8 + 6]) * mul, __uint_as_float(a[x8 + 7]) * mul));
        const int piece = ((c0 & 63) + x8) >> 3;     // 16-byte chunk within the 128-byte row
        *reinterpret_cast<uint4*>(row_base + ((piece ^ (r & 7)) << 4)) = w;
      }
    }
    fence_async_smem();
    named_sync(3 + half, 128);
    if (q4 == 0 && lane == 0) {
      for (int c = 0; c < C::CHK; ++c)
        tma_store_4d(half == 0 ? &tm_gv : &tm_gk, stg + c * C::CHUNK, c * 64, hk, j * 128, b);
      bulk_commit();
      bulk_wait_read0();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // ------------------------------------------------------------ dQ drain
    const int q4 = warp & 3;
    const int dt = threadIdx.x - 384;              // 0..127, = query row within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    uint8_t* stage = sm + C::OFF_STAGE;
    uint8_t* srow = stage + dt * 128;
    int u = 0;
    bool ok = true;
    while (ok && walk.next()) {
      // the four drain warps agree on success before any named barrier
      const bool w_ok =
          __all_sync(0xffffffffu, !failed(&s_fail) && mbar_wait(&bars.dq_ready, u & 1));
      if (lane == 0) s_drain_ok[q4] = w_ok;
      named_sync(1, 128);
      ok = s_drain_ok[0] && s_drain_ok[1] && s_drain_ok[2] && s_drain_ok[3];
      named_sync(1, 128);
      if (!ok) break;
      fence_after_sync();
      uint32_t a[D];
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32)
        tmem_ld32(lane_base + C::T_DP + c0, *reinterpret_cast<uint32_t(*)[32]>(&a[c0]));
      tmem_ld_wait();
      fence_before_sync();
      mbar_arrive(&bars.dq_free);    // R_dP is free for the next dP^T
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        if (dt == 0) bulk_wait_read0();   // previous reduce has read the staging rows
        named_sync(1, 128);
#pragma unroll
        for (int y = 0; y < 8; ++y)
          *reinterpret_cast<uint4*>(srow + ((y ^ (dt & 7)) << 4)) =
              make_uint4(a[c0 + 4 * y], a[c0 + 4 * y + 1], a[c0 + 4 * y + 2], a[c0 + 4 * y + 3]);
        fence_async_smem();
        named_sync(1, 128);
        if (dt == 0) {
          tma_reduce_add_4d(&tm_dq, stage, c0, walk.h, walk.i * 128, b);
          bulk_commit();
        }
      }
      ++u;
    }
    if (dt == 0) bulk_wait_read0();   // the staging rows must outlive the reads
    if (!ok && lane == 0) fail();
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_free(tmem, C::T_COLS);
}

template <int D, bool MASKED>
cudaError_t launch_t(const Shape& sh, const void* q, const void* k, const void* v, const void* g_o,
                     const float* lse, const float* Dv, const int32_t* q_idx,
                     const int32_t* q_cnt, void* g_k, void* g_v, float* dq_acc, int32_t* status,
                     float scale, cudaStream_t st) {
  using C = Cfg<D>;
  CUtensorMap mq, mk, mv, mg, md, mgk, mgv;
  if (!make_bshd_map(&mq, q, sh.B, sh.n, sh.H, D, 128) ||
      !make_bshd_map(&mg, g_o, sh.B, sh.n, sh.H, D, 128) ||
      !make_bshd_map(&mk, k, sh.B, sh.n, sh.Hk, D, 128) ||
      !make_bshd_map(&mv, v, sh.B, sh.n, sh.Hk, D, 128) ||
      !make_bshd_map_f32(&md, dq_acc, sh.B, sh.n, sh.H, D, 128) ||
      !make_bshd_map(&mgk, g_k, sh.B, sh.n, sh.Hk, D, 128) ||
      !make_bshd_map(&mgv, g_v, sh.B, sh.n, sh.Hk, D, 128))
    return cudaErrorInvalidValue;
  const int smem = C::BYTES + 1024;
  auto kern = bwd_tc_kernel<D, MASKED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(sh.T_c, sh.Hk, sh.B);
  kern<<<grid, 512, smem, st>>>(mq, mk, mv, mg, md, mgk, mgv, lse, Dv, q_idx, q_cnt, (__nv_bfloat16*)g_k,
                                (__nv_bfloat16*)g_v, status, sh, scale, scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace

bool bwd_tc_supported(const Shape& sh) {
  return sh.block_q == 128 && sh.block_k == 128 && (sh.d == 64 || sh.d == 128);
}

cudaError_t launch_bwd_tc(const Shape& sh, const void* q, const void* k, const void* v,
                          const void* g_o, const float* lse, const float* Dv,
                          const int32_t* q_idx, const int32_t* q_cnt, void* g_k, void* g_v,
                          float* dq_acc, int32_t* status, float scale, cudaStream_t st) {
  const bool masked = sh.causal || sh.window;
  if (sh.d == 128)
    return masked ? launch_t<128, true>(sh, q, k, v, g_o, lse, Dv, q_idx, q_cnt, g_k, g_v, dq_acc,
                                        status, scale, st)
                  : launch_t<128, false>(sh, q, k, v, g_o, lse, Dv, q_idx, q_cnt, g_k, g_v, dq_acc,
                                         status, scale, st);
  return masked ? launch_t<64, true>(sh, q, k, v, g_o, lse, Dv, q_idx, q_cnt, g_k, g_v, dq_acc,
                                     status, scale, st)
                : launch_t<64, false>(sh, q, k, v, g_o, lse, Dv, q_idx, q_cnt, g_k, g_v, dq_acc,
                                      status, scale, st);
}

}  // namespace bl
