// Block-sparse attention backward on tcgen05 tensor cores (sm_103a), head dim
// 64 or 128.  The products run on 128 x 128 tiles; a mask of 64-wide tiles is
// regrouped into lists of 128 x 128 tiles whose entries carry which 64 x 64
// quarters are kept (sub_lists_kernel), and a dropped quarter's P^T is 0, so
// it adds nothing to any gradient: the same result as skipping it.
//
// Math ("Introducing BackLite", Backpropagation for attention; Using
// Sparsity): for every kept tile pair (query tile i, key tile j)
//   S^T = K_j Q_i^T,  P^T = exp(s S^T - LSE_i),  dP^T = V_j dO_i^T,
//   dS^T = P^T (.) (dP^T - D_i),  dV_j += P^T dO_i,  dK_j += dS^T Q_i,
//   dQ_i += dS K_j,
// with D = rowsum(dO (.) O) from the preprocessing pass; dK and dQ take the
// softmax scale s at the end.  Skipped tiles are never loaded.
//
// Work item = (key tile j, kv head, batch): walk, for each query head of the
// GQA group, the ascending list of query tiles the mask keeps for j, and
// write dK_j, dV_j.  The kernel is persistent: one CTA per SM takes items in
// order from a global counter (so the CTAs running at one time work on
// neighbouring key tiles and share the query tiles they load through L2),
// and its barrier phases count tiles over all its items, so the pipeline
// runs on across item boundaries: the next item's K and V load as soon as
// the last dQ of the current one has read K, and the dK/dV epilogue of one
// item overlaps the first products of the next.
// Every product is a 128 x 128 (x d) tcgen05.mma.  TMEM (512 columns):
//   R_S  [0,128)        S^T; after the softmax, P^T (bf16 pairs) in its
//                       columns [0,32) and [64,96), read as the TMEM A operand
//                       of dV += P^T dO
//   R_dP [128,256)      dP^T; after the softmax, dS^T (bf16 pairs) in its
//                       columns [0,32) and [64,96), the TMEM A operand of
//                       dK += dS^T Q; then the dQ tile dS K (issued after dK)
//   dV   [256,256+d)    dK [256+d,256+2d)
// The issuer queues, per tile t: dK_t and dQ_t once the softmax has put
// dS^T_t in shared memory (second phase); then, for the next tile, dV_{t+1}
// once the first phase has written P^T_{t+1}, which runs while the drain
// empties R_dP of dQ_t; dP^T_{t+1} once R_dP is drained; and S^T_{t+2}
// right behind it, which runs while the softmax forms dS^T_{t+1}.  The
// tensor core runs them in issue order, which makes every reuse safe: S^T
// (into R_S) is queued behind the dV that reads P^T from R_S, and dS^T is
// rewritten only after the next dP^T, hence after dK and dQ, have completed.
// The first dV and dK of an item overwrite the accumulators: they are issued
// after the softmax warps, which read the previous item's accumulators in
// their epilogue, have signalled the item's first tile.
// Warp roles (16 warps):
//   warp 0      TMA producer: per item K_j, V_j; per tile Q_i into two
//               alternating slots and dO_i into a third (4-D tensor maps,
//               128-byte swizzle, rows past n read as 0), plus the tile's
//               LSE and D rows; dO's slot frees once dV and dP^T have read
//               it, so the next dO loads while S^T, dK and dQ run.
//   warp 1      MMA issuer (one thread) and TMEM owner.
//   warps 2-3   take the next item from the global counter and copy its
//               tile lists into one of two shared-memory list buffers, one
//               item ahead of the other roles.
//   warps 4-7   softmax, query columns 0-63; warps 8-11 columns 64-127.
//               Thread = key row: S^T, dP^T rows from TMEM -> P^T (TMEM) and
//               dS^T (TMEM for dK, and bf16 swizzled shared memory, where dQ
//               reads it transposed); after an item's last tile they write
//               dV (warps 4-7) and s dK (warps 8-11).
//   warps 12-15 dQ drain: thread = query row; the dQ tile goes from TMEM
//               through 128-byte-swizzled staging rows into the fp32
//               accumulator with TMA bulk reduce-adds (whole-line L2 adds),
//               each warp its own 32 rows, 32 columns per reduce.
// Registers: the block starts at 128 per thread; warps 0-3 give some back
// (setmaxnreg.dec to 80) so the drain warpgroup can hold a whole 128-column
// dQ row (setmaxnreg.inc to 176): 128*80 + 256*128 + 128*176 = 65536.  The
// issuer forms its shared-memory descriptors next to each MMA (from bases
// the compiler cannot hoist), which keeps them within that budget.
// Causal and sliding-window attention ("Introducing BackLite", Training
// Nanochat): P^T entries of (key, query) pairs that do not attend are 0, so
// they add nothing to any gradient; the mask never keeps a tile without an
// attending pair and, without lists, the walk skips such tiles.
// All hand-offs are mbarriers; every wait is bounded (tc.cuh).
#include <type_traits>

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
  static constexpr int STAGE_BYTES = 128 * 128;   // dQ staging: 4 warps x [32 rows][32 fp32]
  static constexpr int LIST_CAP = 1536;           // cached list entries per buffer
  static constexpr int GMAX = 32;                 // heads per GQA group with cached lists
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_RING = OFF_V + TILE;
  static constexpr int OFF_DS = OFF_RING + NS * TILE;
  static constexpr int OFF_STAGE = OFF_DS + DS_BYTES;
  static constexpr int OFF_L = OFF_STAGE + STAGE_BYTES;   // NS x 128 floats: -lse*log2e
  static constexpr int OFF_D = OFF_L + NS * 128 * 4;      // NS x 128 floats: D
  static constexpr int OFF_LIST = OFF_D + NS * 128 * 4;   // 2 x LIST_CAP ints
  static constexpr int OFF_LCNT = OFF_LIST + 2 * LIST_CAP * 4;
  static constexpr int OFF_LBASE = OFF_LCNT + 2 * GMAX * 4;
  static constexpr int BYTES = OFF_LBASE + 2 * GMAX * 4;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
  static constexpr uint32_t T_COLS = 512;
  static constexpr uint32_t ID_SS = idesc_bf16(128, 128, false, false);  // S^T, dP^T
  static constexpr uint32_t ID_G = idesc_bf16(128, D, false, true);      // dV, dK
  static constexpr uint32_t ID_Q = idesc_bf16(128, D, true, true);       // dQ
};

// Arrivals that release a list buffer: the producer warp, the MMA thread, the
// eight softmax warps and the four drain warps (one elected lane each).
constexpr int kListUsers = 14;

struct Bars {
  uint64_t kv_full, kv_empty, full[3], empty[3], s_full, dp_full, p1_ready, p2_ready;
  uint64_t dq_ready, dq_free, acc_full, list_full[2], list_empty[2];
  uint64_t quiesce;   // the MMA issuer's last commit, waited for before TMEM is freed
};

// Load x = 2t brings Q_t, x = 2t + 1 brings dO_t.  Q_t alternates between
// slots 0 and 1 (its last reader, dK_t, frees it); every dO uses slot 2,
// which frees as soon as dP^T_t (its last reader) completes, so the next dO
// loads while S^T, dK_t and dQ_t run.
__device__ __forceinline__ int slot_of(int x) { return (x & 1) ? 2 : ((x >> 1) & 1); }
__device__ __forceinline__ uint32_t phase_of(int x) {
  return (uint32_t)(((x & 1) ? (x >> 1) : (x >> 2)) & 1);
}

// Work item m (key tile fastest, so consecutive items share query tiles).
struct Item {
  int j, hk, b;
};
__device__ __forceinline__ Item item_of(const Shape& sh, int m) {
  Item it;
  it.j = m % sh.T_c;
  const int r = m / sh.T_c;
  it.hk = r % sh.Hk;
  it.b = r / sh.Hk;
  return it;
}

// Iterates the kept query tiles of key tile j over the heads of one GQA group,
// identically in every role.  Reads the lists from the item's shared-memory
// list buffer when they were cached there, else from global memory.  The
// pointers are passed to next() (kernel parameters and a shared-memory base)
// rather than held, so a walk keeps only its counters in registers.
// With SUB, list entries carry a 64 x 64 sub-tile mask in bits 24-27 (bit
// 2 * query half + key half set = that quarter of the 128 x 128 tile is kept);
// the walk returns it in `sub`.  Without SUB every quarter is kept.
template <bool SUB>
struct Walk {
  int j, b, hk;
  bool cached;
  int gi = 0, li = 0, cnt = -1;
  int h = 0, i = 0, sub = 15;
  bool corrupt = false;
  __device__ bool next(const Shape& sh, int G, const int32_t* q_idx, const int32_t* q_cnt,
                       const int32_t* s_list, const int32_t* s_cnt, const int32_t* s_base) {
    for (;;) {
      if (gi >= G) return false;
      h = hk * G + gi;
      const int64_t bh = (int64_t)b * sh.H + h;
      if (cnt < 0) {
        if (cached) {
          cnt = s_cnt[gi];
        } else {
          cnt = q_cnt ? q_cnt[bh * sh.T_c + j] : sh.T_r;
          if (cnt < 0 || cnt > sh.T_r) {
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
      if (cached)
        i = s_list[s_base[gi] + li];
      else
        i = q_idx ? q_idx[(bh * sh.T_c + j) * (int64_t)sh.T_r + li] : li;
      if (SUB) {
        sub = (i >> 24) & 15;
        i &= 0xFFFFFF;
      }
      ++li;
      if (i < 0 || i >= sh.T_r) {
        corrupt = true;
        continue;
      }
      if (!q_idx && tile_empty(sh, i, j)) continue;   // dense walk: nothing attends
      return true;
    }
  }
};

__device__ __forceinline__ bool failed(const int* f) { return *(volatile const int*)f != 0; }

// MASKED: causal / sliding-window element masks; SUB: sub-tile lists (64-wide
// tiles of the mask, computed as 128 x 128 tiles with the dropped quarters'
// P^T set to 0).
// WL: the launch runs under a non-default wait limit (bl_set_wait_limit).
template <int D, bool MASKED, bool SUB, bool WL>
__global__ void __launch_bounds__(512, 1) bwd_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
    const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_gk,
    const __grid_constant__ CUtensorMap tm_gv, const float* __restrict__ lse,
    const float* __restrict__ Dv, const int32_t* __restrict__ q_idx,
    const int32_t* __restrict__ q_cnt, __nv_bfloat16* __restrict__ g_k,
    __nv_bfloat16* __restrict__ g_v, int32_t* __restrict__ status, Shape sh, float scale,
    float scale_log2, uint64_t wait_ns) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;
  __shared__ uint64_t s_wait;      // the launch's wait limit (ns)
  // parity of the last load armed on full[0..2] and on kv_full (-1: none)
  __shared__ int s_par[4];
  __shared__ int s_cached[2];
  __shared__ int s_item[2];        // item of each list buffer, -1: no more items
  __shared__ int s_drain_ok[4];
  __shared__ int s_copy_ok[2];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = sh.H / sh.Hk;
  const int n_items = sh.T_c * sh.Hk * sh.B;
  int32_t* item_counter = status + 1;   // zeroed by the preprocessing pass

  if (threadIdx.x == 0) {
    mbar_init(&bars.kv_full, 1);
    mbar_init(&bars.kv_empty, 1);
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
    mbar_init(&bars.acc_full, 1);
    mbar_init(&bars.quiesce, 1);
    for (int u = 0; u < 2; ++u) {
      mbar_init(&bars.list_full[u], 64);
      mbar_init(&bars.list_empty[u], kListUsers);
    }
    s_fail = 0;
    s_wait = wait_ns;
    s_par[0] = s_par[1] = s_par[2] = s_par[3] = -1;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_g);
    prefetch_tmap(&tm_dq);
    prefetch_tmap(&tm_gk);
    prefetch_tmap(&tm_gv);
  }
  if (warp == 1) tmem_alloc(&s_tmem, C::T_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;


  auto fail = [&]() {
    atomicOr(&s_fail, 1);
    atomicOr(status, kStatusTimeout);
  };
  int32_t* s_list0 = reinterpret_cast<int32_t*>(sm + C::OFF_LIST);
  int32_t* s_lcnt0 = reinterpret_cast<int32_t*>(sm + C::OFF_LCNT);
  int32_t* s_lbase0 = reinterpret_cast<int32_t*>(sm + C::OFF_LBASE);
  // the walk of an item over list buffer buf (filled by warps 2-3)
  auto make_walk = [&](const Item& it, int buf) {
    Walk<SUB> w;
    w.j = it.j;
    w.b = it.b;
    w.hk = it.hk;
    w.cached = s_cached[buf] != 0;
    return w;
  };
  auto step = [&](Walk<SUB>& w, int buf) {
    return w.next(sh, G, q_idx, q_cnt, s_list0 + buf * C::LIST_CAP, s_lcnt0 + buf * C::GMAX,
                  s_lbase0 + buf * C::GMAX);
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    int x = 0;    // load index over all items: 2t for Q of tile t, 2t+1 for its dO
    int kk = 0;   // items with at least one tile so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int buf = k & 1;
      ok = !failed(&s_fail) && wait_phase<WL>(&bars.list_full[buf], (k >> 1) & 1, &s_wait);
      if (!ok) break;
      const int m = s_item[buf];
      if (m < 0) break;
      const Item it = item_of(sh, m);
      Walk<SUB> walk = make_walk(it, buf);
      bool first = true;
      while (ok && step(walk, buf)) {
        const int64_t bh = (int64_t)it.b * sh.H + walk.h;
        const int r0 = walk.i * 128;
        for (int which = 0; which < 2 && ok; ++which, ++x) {
          const int s = slot_of(x);
          float lv[4], dv[4];
          if (which == 0) {   // this tile's -LSE log2(e) and D travel with its Q slot
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int r = r0 + lane + 32 * e;
              const bool in = r < sh.n;
              lv[e] = in ? -(lse[bh * sh.n + r] * kLog2e) : -INFINITY;
              dv[e] = in ? Dv[bh * sh.n + r] : 0.f;
            }
          }
          ok = !failed(&s_fail) && wait_phase<WL>(&bars.empty[s], phase_of(x) ^ 1, &s_wait);
          if (!ok) break;
          if (lane == 0) {
            mbar_expect_tx(&bars.full[s], C::TILE);
            for (int c = 0; c < C::CHK; ++c)
              tma_load_4d(sm + C::OFF_RING + s * C::TILE + c * C::CHUNK, which ? &tm_g : &tm_q,
                          &bars.full[s], c * 64, walk.h, r0, it.b);
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
          if (lane == 0) s_par[s] = (int)phase_of(x);
          if (which == 0 && first) {
            // this item's K_j and V_j, once the previous item's last dQ has read K
            ok = wait_phase<WL>(&bars.kv_empty, (kk & 1) ^ 1, &s_wait);
            if (!ok) break;
            if (lane == 0) {
              mbar_expect_tx(&bars.kv_full, 2 * C::TILE);
              for (int c = 0; c < C::CHK; ++c) {
                tma_load_4d(sm + C::OFF_K + c * C::CHUNK, &tm_k, &bars.kv_full, c * 64, it.hk,
                            it.j * 128, it.b);
                tma_load_4d(sm + C::OFF_V + c * C::CHUNK, &tm_v, &bars.kv_full, c * 64, it.hk,
                            it.j * 128, it.b);
              }
            }
            if (lane == 0) s_par[3] = kk & 1;
            first = false;
          }
        }
      }
      if (!first) ++kk;
      if (lane == 0 && walk.corrupt) atomicOr(status, kStatusCorrupt);
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&bars.list_empty[buf]);
    }
    if (!ok && lane == 0) fail();
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sK = saddr(sm + C::OFF_K), sV = saddr(sm + C::OFF_V);
      const uint32_t sR = saddr(sm + C::OFF_RING), sDS = saddr(sm + C::OFF_DS);
      // Descriptors: one per operand and tile, from a shared-memory base the
      // compiler cannot hoist out of the tile loop (which keeps the issuer
      // within its registers); a K step advances the descriptor's address
      // field (address / 16, shared addresses stay below 2^18) by off / 16.
      auto opaque = [](uint32_t v) {
        asm volatile("" : "+r"(v));
        return v;
      };
      auto slot_addr = [&](int xx) { return opaque(sR) + slot_of(xx) * C::TILE; };
      auto issue_s = [&](int t) {      // S^T = K Q_t^T  -> R_S
        const uint64_t kd = sdesc_sw128(opaque(sK), 16, 1024);
        const uint64_t qd = sdesc_sw128(slot_addr(2 * t), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::T_S, kd + off, qd + off, C::ID_SS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full);
      };
      auto issue_dp = [&](int t) {     // dP^T = V dO_t^T -> R_dP
        const uint64_t vd = sdesc_sw128(opaque(sV), 16, 1024);
        const uint64_t gd = sdesc_sw128(slot_addr(2 * t + 1), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4;
          mma_ss(tmem + C::T_DP, vd + off, gd + off, C::ID_SS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.dp_full);
      };
      auto wait_slot = [&](int xx) {
        return wait_phase<WL>(&bars.full[slot_of(xx)], phase_of(xx), &s_wait);
      };
      int t = 0;     // tile index over all items
      int kk = 0;    // items with at least one tile so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int buf = k & 1;
        ok = !failed(&s_fail) && wait_phase<WL>(&bars.list_full[buf], (k >> 1) & 1, &s_wait);
        if (!ok) break;
        const int m = s_item[buf];
        if (m < 0) break;
        const Item it = item_of(sh, m);
        Walk<SUB> walk = make_walk(it, buf);
        // dV_u = P^T dO_u (P^T from TMEM); the item's first one overwrites
        auto issue_dv = [&](int u, bool fst) {
          const uint64_t gmn = sdesc_sw128(slot_addr(2 * u + 1), C::CHUNK, 1024);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t pcol = C::T_S + (ks >> 2) * 64 + (ks & 3) * 8;
            mma_ts(tmem + C::T_DV, tmem + pcol, gmn + ks * (2048 >> 4), C::ID_G,
                   (!fst || ks > 0) ? 1u : 0u);
          }
        };
        bool have = step(walk, buf);
        bool next = false;
        if (have) {
          // the item's first tile: S^T needs its K; dV the first softmax phase;
          // dP^T its V and a drained R_dP
          ok = wait_phase<WL>(&bars.kv_full, kk & 1, &s_wait) && wait_slot(2 * t);
          if (!ok) break;
          fence_after_sync();
          issue_s(t);
          ok = !failed(&s_fail) && wait_phase<WL>(&bars.p1_ready, t & 1, &s_wait) &&
               wait_slot(2 * t + 1);
          if (!ok) break;
          fence_after_sync();
          issue_dv(t, true);
          ok = t == 0 || wait_phase<WL>(&bars.dq_free, (t - 1) & 1, &s_wait);
          if (!ok) break;
          fence_after_sync();
          issue_dp(t);
          mma_commit(&bars.empty[2]);           // dO_t's slot: dV and dP^T have read it
          // S^T of the next tile right behind dP^T: it runs while the softmax
          // forms dS^T
          next = step(walk, buf);
          if (next) {
            ok = wait_slot(2 * (t + 1));
            if (!ok) break;
            fence_after_sync();
            issue_s(t + 1);
          }
        }
        bool first = true;
        while (ok && have) {
          // dK_t and dQ_t once dS^T is in shared memory
          ok = !failed(&s_fail) && wait_phase<WL>(&bars.p2_ready, t & 1, &s_wait);
          if (!ok) break;
          fence_after_sync();
          const uint32_t dsb = opaque(sDS);
          const uint64_t qmn = sdesc_sw128(slot_addr(2 * t), C::CHUNK, 1024);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {      // dK += dS^T Q  (dS^T from TMEM)
            const uint32_t dcol = C::T_DP + (ks >> 2) * 64 + (ks & 3) * 8;
            mma_ts(tmem + C::T_DK, tmem + dcol, qmn + ks * (2048 >> 4), C::ID_G,
                   (!first || ks > 0) ? 1u : 0u);
          }
          mma_commit(&bars.empty[t & 1]);       // Q_t's slot
          if (!next) mma_commit(&bars.acc_full);  // dV, dK of this item are final
          // dQ = dS K into R_dP (dP^T was consumed by the softmax)
          const uint64_t dsm = sdesc_sw128(dsb, C::CHUNK, 1024);  // dS, MN-major
          const uint64_t kmn = sdesc_sw128(opaque(sK), C::CHUNK, 1024);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_ss(tmem + C::T_DP, dsm + ks * (2048 >> 4), kmn + ks * (2048 >> 4), C::ID_Q,
                   ks > 0 ? 1u : 0u);
          mma_commit(&bars.dq_ready);
          if (!next) mma_commit(&bars.kv_empty);  // K and V of this item are read
          bool next2 = false;
          if (next) {
            // dV of the next tile runs while the drain empties R_dP; then its
            // dP^T.  The dS^T buffer is rewritten only after that dP^T
            // completes, hence after dQ_t.
            ok = wait_phase<WL>(&bars.p1_ready, (t + 1) & 1, &s_wait) &&
                 wait_slot(2 * (t + 1) + 1);
            if (!ok) break;
            fence_after_sync();
            issue_dv(t + 1, false);
            ok = wait_phase<WL>(&bars.dq_free, t & 1, &s_wait);
            if (!ok) break;
            fence_after_sync();
            issue_dp(t + 1);
            mma_commit(&bars.empty[2]);         // dO_{t+1}'s slot
            next2 = step(walk, buf);
            if (next2) {
              ok = wait_slot(2 * (t + 2));
              if (!ok) break;
              fence_after_sync();
              issue_s(t + 2);
            }
          }
          first = false;
          have = next;
          next = next2;
          ++t;
        }
        if (!ok) break;
        if (!first) ++kk;
        mbar_arrive(&bars.list_empty[buf]);
      }
      if (!ok) fail();
    }
   } else {
    // ------------------------------------------------------------ list copy
    // warps 2-3: item k's lists (all heads of the GQA group) into buffer k % 2
    // once every role has finished item k - 2
    const int tt = threadIdx.x - 64;
    const bool can = q_idx != nullptr && G <= C::GMAX;
    // the two warps agree on success before any named barrier
    auto agree = [&](bool mine) {
      const bool w_ok = __all_sync(0xffffffffu, mine);
      if (lane == 0) s_copy_ok[warp - 2] = w_ok;
      named_sync(2, 64);
      const bool all = s_copy_ok[0] && s_copy_ok[1];
      named_sync(2, 64);
      return all;
    };
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int buf = k & 1;
      ok = agree(!failed(&s_fail) &&
                 wait_phase<WL>(&bars.list_empty[buf], ((k >> 1) & 1) ^ 1, &s_wait));
      if (!ok) break;
      if (tt == 0) {
        const int mm = atomicAdd(item_counter, 1);
        s_item[buf] = mm < n_items ? mm : -1;
      }
      named_sync(2, 64);
      const int m = s_item[buf];
      if (m < 0) {   // no more items: release the roles, which stop here
        mbar_arrive(&bars.list_full[buf]);
        break;
      }
      const Item it = item_of(sh, m);
      int32_t* lcnt = s_lcnt0 + buf * C::GMAX;
      int32_t* lbase = s_lbase0 + buf * C::GMAX;
      int32_t* list = s_list0 + buf * C::LIST_CAP;
      if (can) {
        for (int g = tt; g < G; g += 64) {
          int c = q_cnt[((int64_t)it.b * sh.H + it.hk * G + g) * sh.T_c + it.j];
          if (c < 0 || c > sh.T_r) {
            c = 0;
            atomicOr(status, kStatusCorrupt);
          }
          lcnt[g] = c;
        }
      }
      named_sync(2, 64);
      if (tt == 0) {
        int tot = 0;
        if (can)
          for (int g = 0; g < G; ++g) {
            lbase[g] = tot;
            tot += lcnt[g];
          }
        s_cached[buf] = can && tot <= C::LIST_CAP;
      }
      named_sync(2, 64);
      if (s_cached[buf]) {
        for (int g = 0; g < G; ++g) {
          const int32_t* src =
              q_idx + (((int64_t)it.b * sh.H + it.hk * G + g) * sh.T_c + it.j) * (int64_t)sh.T_r;
          for (int li = tt; li < lcnt[g]; li += 64) list[lbase[g] + li] = src[li];
        }
      }
      mbar_arrive(&bars.list_full[buf]);
    }
    if (!ok && lane == 0) fail();
   }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax
    const int half = (warp - 4) >> 2;           // query columns [64 half, 64 half + 64)
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;               // key row within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    uint8_t* ds_row = sm + C::OFF_DS + half * C::CHUNK + r * 128;
    const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
    int t = 0, kk = 0;
    bool ok = true;
    bool store_pending = false;   // this warp's dK/dV rows may still be read from ds_row
    for (int k = 0; ok; ++k) {
      const int buf = k & 1;
      ok = __all_sync(0xffffffffu, !failed(&s_fail) &&
                                       wait_phase<WL>(&bars.list_full[buf], (k >> 1) & 1, &s_wait));
      if (!ok) break;
      const int m = s_item[buf];
      if (m < 0) break;
      const Item it = item_of(sh, m);
      Walk<SUB> walk = make_walk(it, buf);
      const int j = it.j;
      const bool key_ok = j * 128 + r < sh.n;
      int nt = 0;
      while (ok && step(walk, buf)) {
        const int s = t & 1;                      // Q_t's slot: its LSE and D rows
        // phase 1: P^T from S^T (needs only S^T), written back over S^T
        ok = __all_sync(0xffffffffu, !failed(&s_fail) &&
                                         wait_phase<WL>(&bars.full[s], (t >> 1) & 1, &s_wait) &&
                                         wait_phase<WL>(&bars.s_full, t & 1, &s_wait));
        if (!ok) break;
        fence_after_sync();
        // a dropped 64 x 64 quarter (SUB) contributes P^T = 0, like a key past n
        const bool key_on = key_ok && (!SUB || ((walk.sub >> (2 * half + (r >> 6))) & 1));
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
            // two columns per fma: s S^T log2(e) - LSE log2(e) (sl holds the negation)
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const float4 l4 = reinterpret_cast<const float4*>(sl + c0)[c4];
#pragma unroll
              for (int y = 0; y < 4; y += 2) {
                const int c = 4 * c4 + y;
                float a0, a1;
                f2_unpack(ffma2(f2_pack(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2,
                                y == 0 ? f2_pack(l4.x, l4.y) : f2_pack(l4.z, l4.w)),
                          a0, a1);
                pf[c0 + c] = key_on ? fast_exp2(a0) : 0.f;
                pf[c0 + c + 1] = key_on ? fast_exp2(a1) : 0.f;
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
        ok = __all_sync(0xffffffffu, wait_phase<WL>(&bars.dp_full, t & 1, &s_wait));
        if (!ok) break;
        fence_after_sync();
        if (store_pending) {                       // the rows are about to be overwritten
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          store_pending = false;
        }
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {    // 16 query columns per pass
          uint32_t pv[16];
          tmem_ld16(lane_base + C::T_DP + half * 64 + pass * 16, pv);
          tmem_ld_wait();
          uint32_t dk[8];
          // dS^T = P^T (dP^T - D), two columns per instruction
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 d4 = reinterpret_cast<const float4*>(sd + pass * 16)[c4];
#pragma unroll
            for (int y = 0; y < 4; y += 2) {
              const int c = 4 * c4 + y;
              float s0, s1;
              f2_unpack(fmul2(f2_pack(pf[pass * 16 + c], pf[pass * 16 + c + 1]),
                              fsub2(f2_pack(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])),
                                    y == 0 ? f2_pack(d4.x, d4.y) : f2_pack(d4.z, d4.w))),
                        s0, s1);
              dk[2 * c4 + y / 2] = pack_bf16(s0, s1);
            }
          }
          // dS^T, K-major [key][q] with the 128-byte swizzle, 2 x 16 B chunks
#pragma unroll
          for (int c16 = 0; c16 < 2; ++c16) {
            const int chunk = pass * 2 + c16;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) << 4)) =
                make_uint4(dk[4 * c16], dk[4 * c16 + 1], dk[4 * c16 + 2], dk[4 * c16 + 3]);
          }
          // and as bf16 pairs over dP^T columns already read, the TMEM A
          // operand of dK += dS^T Q
          tmem_st8(lane_base + C::T_DP + half * 64 + pass * 8, dk);
        }
        tmem_st_wait();
        fence_async_smem();
        fence_before_sync();
        mbar_arrive(&bars.p2_ready);               // dK_t and dQ_t may read dS^T
        ++t;
        ++nt;
      }
      if (!ok) break;
      // epilogue: warps 4-7 write dV, warps 8-11 s dK, this key tile's rows (0
      // for an item without tiles).  The accumulators are read before this
      // warpgroup's first arrival of the next item, which gates the next
      // item's first dV and dK (they overwrite).  Each warp stages its 32 rows
      // in its part of the warpgroup's half of the dS^T buffer and writes them
      // with one TMA store per 64 columns: row-per-thread global stores would
      // touch 32 rows 10 KB apart per warp instruction and hold the SM's
      // load/store path for thousands of cycles.  The buffer is free once the
      // item's last dQ has completed (dq_ready); the warp waits for its
      // stores to have read it only before it next writes dS^T there.
      const Item ie = item_of(sh, s_item[buf]);
      if (nt > 0) {
        ok = __all_sync(0xffffffffu, !failed(&s_fail) && wait_phase<WL>(&bars.acc_full, kk & 1, &s_wait) &&
                                         wait_phase<WL>(&bars.dq_ready, (t - 1) & 1, &s_wait));
        if (!ok) break;
        fence_after_sync();
        ++kk;
        const float mul = half == 0 ? 1.f : scale;
        const uint32_t col = half == 0 ? C::T_DV : C::T_DK;
        uint8_t* wstage = sm + C::OFF_DS + half * C::CHUNK + q4 * 32 * 128;   // 1024-aligned
        uint8_t* srow = wstage + lane * 128;
        const int row0 = ie.j * 128 + q4 * 32;
#pragma unroll
        for (int hc = 0; hc < C::CHK; ++hc) {       // 64 columns = one 128-byte row
          if (hc > 0) {                               // the previous store has read the rows
            if (lane == 0) bulk_wait_read0();
            __syncwarp();
          }
#pragma unroll
          for (int c32 = 0; c32 < 2; ++c32) {
            uint32_t a[32];
            tmem_ld32(lane_base + col + hc * 64 + c32 * 32, a);
            tmem_ld_wait();
#pragma unroll
            for (int x8 = 0; x8 < 4; ++x8) {
              const int chunk = c32 * 4 + x8;
              *reinterpret_cast<uint4*>(srow + ((chunk ^ (lane & 7)) << 4)) = make_uint4(
                  pack_bf16(__uint_as_float(a[8 * x8]) * mul, __uint_as_float(a[8 * x8 + 1]) * mul),
                  pack_bf16(__uint_as_float(a[8 * x8 + 2]) * mul,
                            __uint_as_float(a[8 * x8 + 3]) * mul),
                  pack_bf16(__uint_as_float(a[8 * x8 + 4]) * mul,
                            __uint_as_float(a[8 * x8 + 5]) * mul),
                  pack_bf16(__uint_as_float(a[8 * x8 + 6]) * mul,
                            __uint_as_float(a[8 * x8 + 7]) * mul));
            }
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < sh.n) {
            tma_store_4d(half == 0 ? &tm_gv : &tm_gk, wstage, hc * 64, ie.hk, row0, ie.b);
            bulk_commit();
          }
        }
        store_pending = true;
      } else {
        const int row = ie.j * 128 + r;
        uint4* dst = reinterpret_cast<uint4*>(
            half == 0 ? g_v + bshd(sh.vs, ie.b, row, ie.hk) : g_k + bshd(sh.ks, ie.b, row, ie.hk));
        if (row < sh.n) {
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.list_empty[buf]);
    }
    if (lane == 0) bulk_wait0();   // the rows of the last item have been written
    if (!ok && lane == 0) fail();
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
    // ------------------------------------------------------------ dQ drain
    const int q4 = warp & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    // each warp stages its own 32 rows and issues its own reduce-adds, so the
    // four drain warps never wait for one another between chunks
    uint8_t* wst = sm + C::OFF_STAGE + q4 * 4096;
    uint8_t* wrow = wst + lane * 128;
    // the four drain warps agree on success before any named barrier
    auto agree = [&](bool mine) {
      const bool w_ok = __all_sync(0xffffffffu, mine);
      if (lane == 0) s_drain_ok[q4] = w_ok;
      named_sync(1, 128);
      const bool all = s_drain_ok[0] && s_drain_ok[1] && s_drain_ok[2] && s_drain_ok[3];
      named_sync(1, 128);
      return all;
    };
    int u = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int buf = k & 1;
      ok = agree(!failed(&s_fail) && wait_phase<WL>(&bars.list_full[buf], (k >> 1) & 1, &s_wait));
      if (!ok) break;
      const int m = s_item[buf];
      if (m < 0) break;
      const Item it = item_of(sh, m);
      Walk<SUB> walk = make_walk(it, buf);
      while (ok && step(walk, buf)) {
        ok = agree(!failed(&s_fail) && wait_phase<WL>(&bars.dq_ready, u & 1, &s_wait));
        if (!ok) break;
        fence_after_sync();
        uint32_t a[D];
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32)
          tmem_ld32(lane_base + C::T_DP + c0, *reinterpret_cast<uint32_t(*)[32]>(&a[c0]));
        tmem_ld_wait();
        fence_before_sync();
        mbar_arrive(&bars.dq_free);    // R_dP is free for the next dP^T
        const int z0 = walk.i * 128 + q4 * 32;   // this warp's first query row
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          if (lane == 0) bulk_wait_read0();   // the warp's previous reduce has read its rows
          __syncwarp();
#pragma unroll
          for (int y = 0; y < 8; ++y)
            *reinterpret_cast<uint4*>(wrow + ((y ^ (lane & 7)) << 4)) =
                make_uint4(a[c0 + 4 * y], a[c0 + 4 * y + 1], a[c0 + 4 * y + 2], a[c0 + 4 * y + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0 && z0 < sh.n) {   // rows past n are dropped by the TMA unit
            tma_reduce_add_4d(&tm_dq, wst, c0, walk.h, z0, it.b);
            bulk_commit();
          }
        }
        ++u;
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.list_empty[buf]);
    }
    if (lane == 0) bulk_wait_read0();   // the staging rows must outlive the reads
    if (!ok && lane == 0) fail();
  }

  fence_before_sync();
  __syncthreads();
  if (failed(&s_fail)) {
    // A role gave up on a wait, so loads and MMAs it meant to consume may still
    // be in flight: the producer waits for the last load of every barrier it
    // armed (its phase parity recorded in s_par as it was issued), the MMA
    // issuer for a commit behind its last MMA, before the tensor memory is
    // freed and the CTA exits.  (Without a failure every load and MMA has been
    // consumed by then.)
    if (warp == 0 && lane == 0) {
#pragma unroll
      for (int sl = 0; sl < 3; ++sl)
        if (s_par[sl] >= 0) mbar_wait_poll(&bars.full[sl], (uint32_t)s_par[sl]);
      if (s_par[3] >= 0) mbar_wait_poll(&bars.kv_full, (uint32_t)s_par[3]);
    }
    if (warp == 1 && lane == 0) {
      mma_commit(&bars.quiesce);
      mbar_wait_poll(&bars.quiesce, 0);
    }
    fence_before_sync();
    __syncthreads();
  }
  if (warp == 1) tmem_free(tmem, C::T_COLS);
}

int sm_count() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (count[dev] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
      c = 148;
    count[dev] = c;
  }
  return count[dev];
}

template <int D, bool MASKED, bool SUB, bool WL>
cudaError_t launch_t(const Shape& sh, const void* q, const void* k, const void* v, const void* g_o,
                     const float* lse, const float* Dv, const int32_t* q_idx,
                     const int32_t* q_cnt, void* g_k, void* g_v, float* dq_acc, int32_t* status,
                     float scale, cudaStream_t st) {
  using C = Cfg<D>;
  CUtensorMap mq, mk, mv, mg, md, mgk, mgv;
  if (!make_bshd_map(&mq, q, sh.B, sh.n, sh.H, D, 128, sh.qs) ||
      !make_bshd_map(&mg, g_o, sh.B, sh.n, sh.H, D, 128, sh.os) ||
      !make_bshd_map(&mk, k, sh.B, sh.n, sh.Hk, D, 128, sh.ks) ||
      !make_bshd_map(&mv, v, sh.B, sh.n, sh.Hk, D, 128, sh.vs) ||
      !make_bshd_map(&mgk, g_k, sh.B, sh.n, sh.Hk, D, 32, sh.ks) ||
      !make_bshd_map(&mgv, g_v, sh.B, sh.n, sh.Hk, D, 32, sh.vs) ||
      !make_bshd_map_f32(&md, dq_acc, sh.B, sh.n, sh.H, D, 32))
    return cudaErrorInvalidValue;
  const int smem = C::BYTES + 1024;
  auto kern = bwd_tc_kernel<D, MASKED, SUB, WL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)sh.T_c * sh.Hk * sh.B;
  const int grid = (int)(items < sm_count() ? items : sm_count());
  kern<<<grid, 512, smem, st>>>(mq, mk, mv, mg, md, mgk, mgv, lse, Dv, q_idx, q_cnt,
                                (__nv_bfloat16*)g_k, (__nv_bfloat16*)g_v, status, sh, scale,
                                scale * kLog2e, wait_limit_ns());
  return cudaGetLastError();
}

// Lists of 64-wide tiles as lists of 128 x 128 tiles: for every (batch,
// head, 128-key tile) the ascending 128-row query tiles that hold a kept
// 64 x 64 quarter, each entry carrying the quarter mask in bits 24-27 (bit
// 2 * query half + key half).  A 128-wide side keeps both of its halves
// together.  Entries and counts out of range are skipped and recorded in the
// status word, as the walk does.  One CTA of 128 threads per (128-key tile,
// head, batch); `bits` in dynamic shared memory, one word per 128-row tile.
__global__ void __launch_bounds__(128) sub_lists_kernel(const int32_t* __restrict__ q_idx,
                                                        const int32_t* __restrict__ q_cnt,
                                                        Shape sh, Shape sh128,
                                                        int32_t* __restrict__ out_idx,
                                                        int32_t* __restrict__ out_cnt,
                                                        int32_t* __restrict__ status) {
  extern __shared__ uint32_t bits[];
  __shared__ int s_wcnt[4];
  const int J = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bh = (int64_t)blockIdx.z * sh.H + blockIdx.y;
  const int R = sh128.T_r;
  for (int x = tid; x < R; x += 128) bits[x] = 0;
  __syncthreads();
  const int nsrc = sh.block_k == 64 ? 2 : 1;
  bool bad = false;
  for (int e = 0; e < nsrc; ++e) {
    const int j = nsrc == 2 ? 2 * J + e : J;
    if (j >= sh.T_c) break;
    const uint32_t kmask = sh.block_k == 64 ? (1u << e) : 3u;   // key halves of this tile
    int cnt = q_cnt[bh * sh.T_c + j];
    if (cnt < 0 || cnt > sh.T_r) {
      bad = true;
      cnt = 0;
    }
    const int32_t* list = q_idx + (bh * sh.T_c + j) * (int64_t)sh.T_r;
    for (int li = tid; li < cnt; li += 128) {
      const int i = list[li];
      if (i < 0 || i >= sh.T_r) {
        bad = true;
        continue;
      }
      const int I = sh.block_q == 64 ? i >> 1 : i;
      const uint32_t qmask = sh.block_q == 64 ? (1u << (i & 1)) : 3u;   // query halves
      uint32_t m = 0;
      for (int qh = 0; qh < 2; ++qh)
        if (qmask & (1u << qh)) m |= kmask << (2 * qh);
      atomicOr(&bits[I], m);
    }
  }
  if (bad) atomicOr(status, tc::kStatusCorrupt);
  __syncthreads();
  // compact the non-empty 128-row tiles in ascending order
  int32_t* orow = out_idx + (bh * sh128.T_c + J) * (int64_t)R;
  int run = 0;
  for (int x0 = 0; x0 < R; x0 += 128) {
    const int x = x0 + tid;
    const uint32_t m = x < R ? bits[x] : 0u;
    const unsigned bal = __ballot_sync(0xffffffffu, m != 0);
    if (lane == 0) s_wcnt[warp] = __popc(bal);
    __syncthreads();
    int off = run;
    for (int w = 0; w < warp; ++w) off += s_wcnt[w];
    if (m) orow[off + __popc(bal & ((1u << lane) - 1u))] = x | (int)(m << 24);
    run += s_wcnt[0] + s_wcnt[1] + s_wcnt[2] + s_wcnt[3];
    __syncthreads();
  }
  if (tid == 0) out_cnt[bh * sh128.T_c + J] = run;
}

}  // namespace

bool bwd_tc_supported(const Shape& sh) { return sh.d == 64 || sh.d == 128; }

// The 128 x 128 view of a shape with 64-wide tiles.
Shape tiles128(const Shape& sh) {
  Shape t = sh;
  t.block_q = t.block_k = 128;
  t.T_r = t.T_c = (sh.n + 127) / 128;
  t.n_pad = (int64_t)t.T_r * 128;
  return t;
}

size_t bwd_sub_lists_bytes(const Shape& sh) {
  if (sh.block_q == 128 && sh.block_k == 128) return 0;
  const Shape t = tiles128(sh);
  const size_t e = (size_t)sh.B * sh.H * t.T_c * ((size_t)t.T_r + 1);
  return (e * sizeof(int32_t) + 255) & ~(size_t)255;
}

cudaError_t launch_bwd_tc(const Shape& sh, const void* q, const void* k, const void* v,
                          const void* g_o, const float* lse, const float* Dv,
                          const int32_t* q_idx, const int32_t* q_cnt, void* g_k, void* g_v,
                          float* dq_acc, int32_t* sub_ws, int32_t* status, float scale,
                          cudaStream_t st) {
  const bool masked = sh.causal || sh.window;
  const bool sub = !(sh.block_q == 128 && sh.block_k == 128);
  const Shape s128 = tiles128(sh);
  if (sub && q_idx) {   // 64-wide tiles: lists of 128 x 128 tiles with quarter masks
    if ((size_t)s128.T_r * sizeof(uint32_t) > 48 * 1024) return cudaErrorInvalidValue;
    int32_t* idx = sub_ws;
    int32_t* cnt = sub_ws + (size_t)sh.B * sh.H * s128.T_c * s128.T_r;
    dim3 g(s128.T_c, sh.H, sh.B);
    sub_lists_kernel<<<g, 128, (size_t)s128.T_r * sizeof(uint32_t), st>>>(q_idx, q_cnt, sh, s128,
                                                                          idx, cnt, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    q_idx = idx;
    q_cnt = cnt;
  }
  auto run = [&](auto wl_c) {
    auto go = [&](auto d_c, auto m_c, auto s_c) {
      return launch_t<decltype(d_c)::value, decltype(m_c)::value, decltype(s_c)::value,
                      decltype(wl_c)::value>(s128, q, k, v, g_o, lse, Dv, q_idx, q_cnt, g_k, g_v,
                                             dq_acc, status, scale, st);
    };
    using I64 = std::integral_constant<int, 64>;
    using I128 = std::integral_constant<int, 128>;
    using T = std::true_type;
    using F = std::false_type;
    if (sub && q_idx) return sh.d == 128 ? go(I128{}, F{}, T{}) : go(I64{}, F{}, T{});
    if (sh.d == 128) return masked ? go(I128{}, T{}, F{}) : go(I128{}, F{}, F{});
    return masked ? go(I64{}, T{}, F{}) : go(I64{}, F{}, F{});
  };
  return wait_limit_ns() != kWaitLimitNs ? run(std::true_type{}) : run(std::false_type{});
}

}  // namespace bl
