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
// GQA group, the ascending list of query tiles the mask keeps for j.  Each
// query tile is handled as two halves of 64 rows so that every accumulator
// fits the 512 TMEM columns of the SM:
//   [0,64) S^T half   [64,128) dP^T half   [128,128+d) dQ (one query tile)
//   [128+d,128+2d) dV   [128+2d,128+3d) dK
// Warp roles (12 warps):
//   warp 0      TMA producer: K_j, V_j once; then per half Q and dO (4-D
//               tensor maps, 128-byte swizzle, out-of-range rows read as 0)
//               into a 2-slot ring, plus the half's LSE and D rows.
//   warp 1      MMA issuer (one thread) and TMEM owner.  Per half h it issues
//               S^T_h, dP^T_h, then the gradient MMAs of half h-1 (dV, dK and,
//               after the second half of a tile, dQ), so the softmax of h
//               overlaps the tensor-core work of h-1.
//   warps 4-7   softmax warpgroup: thread = key row; reads S^T/dP^T rows from
//               TMEM, writes P^T and dS^T (bf16, swizzled) to shared memory;
//               at the end writes dK, dV.
//   warps 2-3   at start: copy this CTA's tile lists into shared memory.
//   warps 8-11  dQ warpgroup: thread = query row; drains the dQ tile from
//               TMEM through a 128-byte-swizzled staging buffer (32 columns at
//               a time) into the fp32 accumulator with TMA bulk reduce-adds,
//               which the L2 applies as whole-line reductions.
// All hand-offs are mbarriers; every wait is bounded (tc.cuh).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace bl {

namespace {

using namespace tc;

template <int D>
struct Cfg {
  static constexpr int BK = 128, HQ = 64, NS = 2;
  static constexpr int CHK = D / 64;              // 64-element chunks along d
  static constexpr int KV_CHUNK = BK * 128;       // [128 rows][128 B]
  static constexpr int QH_CHUNK = HQ * 128;       // [64 rows][128 B]
  static constexpr int KV_BYTES = KV_CHUNK * CHK;
  static constexpr int QH_BYTES = QH_CHUNK * CHK;
  static constexpr int P_BYTES = BK * HQ * 2;     // [128 keys][64 q] bf16
  static constexpr int STAGE_BYTES = 128 * 128;   // dQ staging: [128 rows][32 fp32]
  static constexpr int LIST_CAP = 2048;           // cached list entries per CTA
  static constexpr int GMAX = 32;                 // heads per GQA group with cached lists
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;
  static constexpr int OFF_G = OFF_Q + NS * QH_BYTES;
  static constexpr int OFF_P = OFF_G + NS * QH_BYTES;
  static constexpr int OFF_S = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_STAGE = OFF_S + 2 * P_BYTES;
  static constexpr int OFF_L = OFF_STAGE + STAGE_BYTES;   // NS x 64 floats: lse*log2e
  static constexpr int OFF_D = OFF_L + NS * HQ * 4;       // NS x 64 floats: D
  static constexpr int OFF_LIST = OFF_D + NS * HQ * 4;    // LIST_CAP ints
  static constexpr int OFF_LCNT = OFF_LIST + LIST_CAP * 4;  // GMAX ints
  static constexpr int OFF_LBASE = OFF_LCNT + GMAX * 4;     // GMAX ints
  static constexpr int BYTES = OFF_LBASE + GMAX * 4;
  static constexpr uint32_t T_S = 0, T_DP = 64, T_DQ = 128, T_DV = 128 + D, T_DK = 128 + 2 * D;
  static constexpr uint32_t T_COLS = 512;
  static constexpr uint32_t ID_S = idesc_bf16(128, 64, false, false);
  static constexpr uint32_t ID_G = idesc_bf16(128, D, false, true);
  static constexpr uint32_t ID_Q = idesc_bf16(128, D, true, true);
};

struct Bars {
  uint64_t kv, full[2], empty[2], s, p, pfree[2], dsfree, dqready, dqfree, acc;
};

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
      return true;
    }
  }
};

__device__ __forceinline__ bool failed(const int* f) { return *(volatile const int*)f != 0; }

template <int D>
__global__ void __launch_bounds__(384, 1) bwd_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
    const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ lse, const float* __restrict__ Dv, const int32_t* __restrict__ q_idx,
    const int32_t* __restrict__ q_cnt, __nv_bfloat16* __restrict__ g_k,
    __nv_bfloat16* __restrict__ g_v, float* __restrict__ dq_acc, int32_t* __restrict__ status,
    Shape sh, float scale, float scale_log2) {
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
      mbar_init(&bars.full[s], 33);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.s, 1);
    mbar_init(&bars.p, 128);
    mbar_init(&bars.pfree[0], 1);
    mbar_init(&bars.pfree[1], 1);
    mbar_init(&bars.dsfree, 1);
    mbar_init(&bars.dqready, 1);
    mbar_init(&bars.dqfree, 128);
    mbar_init(&bars.acc, 1);
    s_fail = 0;
    fence_mbar_init();
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_g);
      mbar_expect_tx(&bars.kv, 2 * C::KV_BYTES);
      for (int c = 0; c < C::CHK; ++c) {
        tma_load_4d(sm + C::OFF_K + c * C::KV_CHUNK, &tm_k, &bars.kv, c * 64, hk, j * 128, b);
        tma_load_4d(sm + C::OFF_V + c * C::KV_CHUNK, &tm_v, &bars.kv, c * 64, hk, j * 128, b);
      }
    }
    int hc = 0;
    while (walk.next()) {
      const int64_t bh = (int64_t)b * sh.H + walk.h;
      for (int half = 0; half < 2; ++half, ++hc) {
        const int s = hc % C::NS;
        const int r0 = walk.i * 128 + half * 64;
        // start the LSE and D loads of this half before waiting for its slot
        float lv[2], dv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = r0 + lane + 32 * e;
          const bool ok = r < sh.n;
          lv[e] = ok ? lse[bh * sh.n + r] * kLog2e : INFINITY;
          dv[e] = ok ? Dv[bh * sh.n + r] : 0.f;
        }
        if (failed(&s_fail) || !mbar_wait(&bars.empty[s], ((hc / C::NS) & 1) ^ 1)) {
          if (lane == 0) fail();
          goto producer_done;
        }
        if (lane == 0) {
          mbar_expect_tx(&bars.full[s], 2 * C::QH_BYTES);
          for (int c = 0; c < C::CHK; ++c) {
            tma_load_4d(sm + C::OFF_Q + s * C::QH_BYTES + c * C::QH_CHUNK, &tm_q, &bars.full[s],
                        c * 64, walk.h, r0, b);
            tma_load_4d(sm + C::OFF_G + s * C::QH_BYTES + c * C::QH_CHUNK, &tm_g, &bars.full[s],
                        c * 64, walk.h, r0, b);
          }
        }
        float* sl = reinterpret_cast<float*>(sm + C::OFF_L) + s * 64;
        float* sd = reinterpret_cast<float*>(sm + C::OFF_D) + s * 64;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sl[lane + 32 * e] = lv[e];
          sd[lane + 32 * e] = dv[e];
        }
        mbar_arrive(&bars.full[s]);   // with lane 0's expect_tx arrival: 33 per phase
      }
    }
    if (lane == 0 && walk.corrupt) atomicOr(status, kStatusCorrupt);
  producer_done:;
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sK = saddr(sm + C::OFF_K), sV = saddr(sm + C::OFF_V);
      const uint32_t sQ = saddr(sm + C::OFF_Q), sG = saddr(sm + C::OFF_G);
      const uint32_t sP = saddr(sm + C::OFF_P), sS = saddr(sm + C::OFF_S);
      bool ok = mbar_wait(&bars.kv, 0);
      int hc = 0;
      // gradient MMAs of half g (slot g % NS, P/dS buffer g % 2)
      auto grads = [&](int g) -> bool {
        const int slot = g % C::NS, pb = g & 1;
        const uint32_t q_half = sQ + slot * C::QH_BYTES, g_half = sG + slot * C::QH_BYTES;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (g > 0 || kk > 0) ? 1u : 0u;
          mma_ss(tmem + C::T_DV, sdesc_sw128(sP + pb * C::P_BYTES + kk * 32, 16, 1024),
                 sdesc_sw128(g_half + kk * 2048, C::QH_CHUNK, 1024), C::ID_G, acc);
          mma_ss(tmem + C::T_DK, sdesc_sw128(sS + pb * C::P_BYTES + kk * 32, 16, 1024),
                 sdesc_sw128(q_half + kk * 2048, C::QH_CHUNK, 1024), C::ID_G, acc);
        }
        mma_commit(&bars.pfree[pb]);
        mma_commit(&bars.empty[slot]);
        if (pb == 1) {
          const int u = g >> 1;
          if (!mbar_wait(&bars.dqfree, (u & 1) ^ 1)) return false;
          fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + C::T_DQ, sdesc_sw128(sS + kk * 2048, C::P_BYTES, 1024),
                   sdesc_sw128(sK + kk * 2048, C::KV_CHUNK, 1024), C::ID_Q, kk > 0 ? 1u : 0u);
          mma_commit(&bars.dqready);
          mma_commit(&bars.dsfree);
        }
        return true;
      };
      while (ok && walk.next()) {
        for (int half = 0; half < 2 && ok; ++half, ++hc) {
          const int s = hc % C::NS;
          ok = !failed(&s_fail) && mbar_wait(&bars.full[s], (hc / C::NS) & 1);
          if (ok && hc > 0) ok = mbar_wait(&bars.p, (hc - 1) & 1);
          if (!ok) break;
          fence_after_sync();
          const uint32_t q_half = sQ + s * C::QH_BYTES, g_half = sG + s * C::QH_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
            const uint32_t qo = (kk >> 2) * C::QH_CHUNK + (kk & 3) * 32;
            mma_ss(tmem + C::T_S, sdesc_sw128(sK + ko, 16, 1024),
                   sdesc_sw128(q_half + qo, 16, 1024), C::ID_S, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32;
            const uint32_t qo = (kk >> 2) * C::QH_CHUNK + (kk & 3) * 32;
            mma_ss(tmem + C::T_DP, sdesc_sw128(sV + ko, 16, 1024),
                   sdesc_sw128(g_half + qo, 16, 1024), C::ID_S, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars.s);
          if (hc > 0) ok = grads(hc - 1);
        }
      }
      if (ok && hc > 0) {
        ok = mbar_wait(&bars.p, (hc - 1) & 1);
        if (ok) {
          fence_after_sync();
          ok = grads(hc - 1);
        }
      }
      if (!ok) fail();
      mma_commit(&bars.acc);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                  // key row within the tile
    const bool key_ok = j * 128 + r < sh.n;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    uint8_t* sP = sm + C::OFF_P;
    uint8_t* sS = sm + C::OFF_S;
    int hc = 0;
    bool ok = true;
    while (ok && walk.next()) {
      for (int half = 0; half < 2; ++half, ++hc) {
        const int s = hc % C::NS, pb = hc & 1, u = hc >> 1;
        ok = __all_sync(0xffffffffu, !failed(&s_fail) &&
                                         mbar_wait(&bars.full[s], (hc / C::NS) & 1) &&
                                         mbar_wait(&bars.s, hc & 1));
        if (!ok) break;
        fence_after_sync();
        uint32_t sv[2][32], pv[2][32];
        tmem_ld32(lane_base + C::T_S, sv[0]);
        tmem_ld32(lane_base + C::T_S + 32, sv[1]);
        tmem_ld32(lane_base + C::T_DP, pv[0]);
        tmem_ld32(lane_base + C::T_DP + 32, pv[1]);
        tmem_ld_wait();
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.pfree[pb], ((hc >> 1) & 1) ^ 1) &&
                                         mbar_wait(&bars.dsfree, (u & 1) ^ 1));
        if (!ok) break;
        const float* sl = reinterpret_cast<const float*>(sm + C::OFF_L) + s * 64;
        const float* sd = reinterpret_cast<const float*>(sm + C::OFF_D) + s * 64;
        uint8_t* prow = sP + pb * C::P_BYTES + r * 128;
        uint8_t* srow = sS + pb * C::P_BYTES + r * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {      // 8 columns (16 bytes) at a time
          uint32_t pk[4], dk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float p2[2], d2[2];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              const int c = c8 * 8 + e * 2 + x;
              const float sc = __uint_as_float(sv[c >> 5][c & 31]);
              const float dp = __uint_as_float(pv[c >> 5][c & 31]);
              const float p = key_ok ? fast_exp2(fmaf(sc, scale_log2, -sl[c])) : 0.f;
              p2[x] = p;
              d2[x] = p * (dp - sd[c]);
            }
            pk[e] = pack_bf16(p2[0], p2[1]);
            dk[e] = pack_bf16(d2[0], d2[1]);
          }
          const int phys = (c8 ^ (r & 7)) * 16;
          *reinterpret_cast<uint4*>(prow + phys) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(srow + phys) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
        }
        fence_async_smem();
        fence_before_sync();
        mbar_arrive(&bars.p);
      }
    }
    if (!ok && lane == 0) fail();
    // epilogue: dV, dK rows of this key tile (accumulators complete at bars.acc)
    const bool acc_ok = mbar_wait(&bars.acc, 0);
    fence_after_sync();
    const bool have = __all_sync(0xffffffffu, ok && acc_ok) && hc > 0;
    const int key = j * 128 + r;
    __nv_bfloat16* vr = g_v + (((int64_t)b * sh.n + key) * sh.Hk + hk) * D;
    __nv_bfloat16* kr = g_k + (((int64_t)b * sh.n + key) * sh.Hk + hk) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t a[32], k2[32];
      if (have) {  // warp-uniform: the TMEM loads are warp-collective
        tmem_ld32(lane_base + C::T_DV + c0, a);
        tmem_ld32(lane_base + C::T_DK + c0, k2);
        tmem_ld_wait();
      }
      if (key < sh.n) {
#pragma unroll
        for (int x = 0; x < 32; x += 8) {
          uint4 wv = make_uint4(0u, 0u, 0u, 0u), wk = make_uint4(0u, 0u, 0u, 0u);
          if (have) {
            wv = make_uint4(pack_bf16(__uint_as_float(a[x]), __uint_as_float(a[x + 1])),
                            pack_bf16(__uint_as_float(a[x + 2]), __uint_as_float(a[x + 3])),
                            pack_bf16(__uint_as_float(a[x + 4]), __uint_as_float(a[x + 5])),
                            pack_bf16(__uint_as_float(a[x + 6]), __uint_as_float(a[x + 7])));
            wk = make_uint4(
                pack_bf16(__uint_as_float(k2[x]) * scale, __uint_as_float(k2[x + 1]) * scale),
                pack_bf16(__uint_as_float(k2[x + 2]) * scale, __uint_as_float(k2[x + 3]) * scale),
                pack_bf16(__uint_as_float(k2[x + 4]) * scale, __uint_as_float(k2[x + 5]) * scale),
                pack_bf16(__uint_as_float(k2[x + 6]) * scale, __uint_as_float(k2[x + 7]) * scale));
          }
          *reinterpret_cast<uint4*>(vr + c0 + x) = wv;
          *reinterpret_cast<uint4*>(kr + c0 + x) = wk;
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ drain
    const int q4 = warp & 3;
    const int dt = threadIdx.x - 256;              // 0..127, = row within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    uint8_t* stage = sm + C::OFF_STAGE;
    uint8_t* srow = stage + dt * 128;
    int u = 0;
    bool ok = true;
    while (ok && walk.next()) {
      // the four drain warps agree on success before any named barrier
      const bool w_ok =
          __all_sync(0xffffffffu, !failed(&s_fail) && mbar_wait(&bars.dqready, u & 1));
      if (lane == 0) s_drain_ok[q4] = w_ok;
      named_sync(1, 128);
      ok = s_drain_ok[0] && s_drain_ok[1] && s_drain_ok[2] && s_drain_ok[3];
      named_sync(1, 128);
      if (!ok) break;
      fence_after_sync();
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(lane_base + C::T_DQ + c0, a);
        tmem_ld_wait();
        if (c0 + 32 == D) {          // the dQ columns of TMEM are free again
          fence_before_sync();
          mbar_arrive(&bars.dqfree);
        }
        if (dt == 0) bulk_wait_read0();   // previous reduce has read the staging rows
        named_sync(1, 128);
#pragma unroll
        for (int x = 0; x < 8; ++x)
          *reinterpret_cast<uint4*>(srow + ((x ^ (dt & 7)) << 4)) =
              make_uint4(a[4 * x], a[4 * x + 1], a[4 * x + 2], a[4 * x + 3]);
        fence_async_smem();
        named_sync(1, 128);
        if (dt == 0) {
          tma_reduce_add_4d(&tm_dq, stage, c0, walk.h, walk.i * 128, b);
          bulk_commit();
        }
      }
      ++u;
    }
    if (dt == 0) bulk_wait0();
    if (!ok && lane == 0) fail();
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_free(tmem, C::T_COLS);
}

template <int D>
cudaError_t launch_t(const Shape& sh, const void* q, const void* k, const void* v, const void* g_o,
                     const float* lse, const float* Dv, const int32_t* q_idx,
                     const int32_t* q_cnt, void* g_k, void* g_v, float* dq_acc, int32_t* status,
                     float scale, cudaStream_t st) {
  using C = Cfg<D>;
  CUtensorMap mq, mk, mv, mg, md;
  if (!make_bshd_map(&mq, q, sh.B, sh.n, sh.H, D, 64) || !make_bshd_map(&mg, g_o, sh.B, sh.n, sh.H, D, 64) ||
      !make_bshd_map(&mk, k, sh.B, sh.n, sh.Hk, D, 128) || !make_bshd_map(&mv, v, sh.B, sh.n, sh.Hk, D, 128) ||
      !make_bshd_map_f32(&md, dq_acc, sh.B, sh.n, sh.H, D, 128))
    return cudaErrorInvalidValue;
  const int smem = C::BYTES + 1024;
  auto kern = bwd_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(sh.T_c, sh.Hk, sh.B);
  kern<<<grid, 384, smem, st>>>(mq, mk, mv, mg, md, lse, Dv, q_idx, q_cnt, (__nv_bfloat16*)g_k,
                                (__nv_bfloat16*)g_v, dq_acc, status, sh, scale, scale * kLog2e);
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
  if (sh.d == 128)
    return launch_t<128>(sh, q, k, v, g_o, lse, Dv, q_idx, q_cnt, g_k, g_v, dq_acc, status, scale, st);
  return launch_t<64>(sh, q, k, v, g_o, lse, Dv, q_idx, q_cnt, g_k, g_v, dq_acc, status, scale, st);
}

}  // namespace bl
