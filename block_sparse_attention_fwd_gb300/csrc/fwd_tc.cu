// Attention forward with per-(query row, key tile) LSE statistics on tcgen05
// tensor cores (sm_103a), 128 x 128 tiles, head dim 64 or 128.
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
// One CTA per (128-row query tile, head, batch).  TMEM: S double buffer
// [0,128) and [128,256), O [256,256+d).  Warp roles (8 warps):
//   warp 0     TMA producer: Q once, then K_j, V_j into a 2-stage ring.
//   warp 1     MMA issuer (one thread), TMEM owner: S_j = Q K_j^T, then
//              O += P_{j-1} V_{j-1}, so the softmax of tile j overlaps the PV
//              product of tile j-1.
//   warps 4-7  softmax warpgroup, thread = query row: reads S_j from TMEM,
//              writes the tile statistic (one coalesced 512-byte row per key
//              tile), P_j (bf16, 128-byte swizzled) to shared memory; at the
//              end writes O = acc / l and LSE.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace bl {

namespace {

using namespace tc;

template <int D>
struct FCfg {
  static constexpr int NS = 2;
  static constexpr int CHK = D / 64;
  static constexpr int CHUNK = 128 * 128;               // [128 rows][128 B]
  static constexpr int Q_BYTES = CHUNK * CHK;
  static constexpr int KV_BYTES = CHUNK * CHK;
  static constexpr int P_BYTES = 2 * CHUNK;             // [128 q][128 keys] bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NS * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NS * KV_BYTES;
  static constexpr int BYTES = OFF_P + 2 * P_BYTES;
  static constexpr uint32_t T_S = 0, T_O = 256, T_COLS = 512;
  static constexpr uint32_t ID_S = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t ID_O = idesc_bf16(128, D, false, true);
  static constexpr float kRescale = 8.f;  // base-2 headroom before O is rescaled
};

struct FBars {
  uint64_t q, kv_full[2], kv_empty[2], s_full[2], p_ready[2], p_free[2], o_step, o_done;
};

__device__ __forceinline__ bool failed(const int* f) { return *(volatile const int*)f != 0; }

template <int D>
__global__ void __launch_bounds__(256, 1) fwd_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ o,
    float* __restrict__ lse, float* __restrict__ stats, int32_t* __restrict__ status, Shape sh,
    float scale_log2) {
  using C = FCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) FBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ int s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (sh.H / sh.Hk);
  const int Tc = sh.T_c;

  if (threadIdx.x == 0) {
    mbar_init(&bars.q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.p_ready[s], 128);
      mbar_init(&bars.p_free[s], 1);
    }
    mbar_init(&bars.o_step, 1);
    mbar_init(&bars.o_done, 1);
    s_fail = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&s_tmem, C::T_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;
  auto fail = [&]() {
    atomicOr(&s_fail, 1);
    if (status) atomicOr(status, kStatusTimeout);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_expect_tx(&bars.q, C::Q_BYTES);
      for (int c = 0; c < C::CHK; ++c)
        tma_load_4d(sm + C::OFF_Q + c * C::CHUNK, &tm_q, &bars.q, c * 64, h, qt * 128, b);
      for (int j = 0; j < Tc; ++j) {
        const int s = j & 1;
        if (failed(&s_fail) || !mbar_wait(&bars.kv_empty[s], ((j >> 1) & 1) ^ 1)) {
          fail();
          break;
        }
        mbar_expect_tx(&bars.kv_full[s], 2 * C::KV_BYTES);
        for (int c = 0; c < C::CHK; ++c) {
          tma_load_4d(sm + C::OFF_K + s * C::KV_BYTES + c * C::CHUNK, &tm_k, &bars.kv_full[s],
                      c * 64, hk, j * 128, b);
          tma_load_4d(sm + C::OFF_V + s * C::KV_BYTES + c * C::CHUNK, &tm_v, &bars.kv_full[s],
                      c * 64, hk, j * 128, b);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sQ = saddr(sm + C::OFF_Q), sK = saddr(sm + C::OFF_K);
      const uint32_t sV = saddr(sm + C::OFF_V), sP = saddr(sm + C::OFF_P);
      bool ok = mbar_wait(&bars.q, 0);
      auto pv = [&](int jj) -> bool {   // O += P_jj V_jj
        const int s = jj & 1;
        if (!mbar_wait(&bars.p_ready[s], (jj >> 1) & 1)) return false;
        fence_after_sync();
        const uint32_t pbase = sP + s * C::P_BYTES, vbase = sV + s * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + C::T_O, sdesc_sw128(pbase + (kk >> 2) * C::CHUNK + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(vbase + kk * 2048, C::CHUNK, 1024), C::ID_O,
                 (jj > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.kv_empty[s]);
        mma_commit(&bars.p_free[s]);
        mma_commit(&bars.o_step);
        return true;
      };
      for (int j = 0; ok && j < Tc; ++j) {
        const int s = j & 1;
        ok = !failed(&s_fail) && mbar_wait(&bars.kv_full[s], (j >> 1) & 1);
        // S buffer s was last read by the softmax of tile j-2
        if (ok && j >= 2) ok = mbar_wait(&bars.p_ready[s], ((j - 2) >> 1) & 1);
        if (!ok) break;
        fence_after_sync();
        const uint32_t kbase = sK + s * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK + (kk & 3) * 32;
          mma_ss(tmem + C::T_S + s * 128, sdesc_sw128(sQ + off, 16, 1024),
                 sdesc_sw128(kbase + off, 16, 1024), C::ID_S, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_full[s]);
        if (j >= 1) ok = pv(j - 1);
      }
      if (ok && Tc >= 1) ok = pv(Tc - 1);
      if (!ok) fail();
      mma_commit(&bars.o_done);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int row = qt * 128 + r;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const int64_t bh = (int64_t)b * sh.H + h;
    float* st_row = stats ? stats + bh * sh.T_c * sh.n_pad + row : nullptr;
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < Tc; ++j) {
      const int s = j & 1;
      ok = __all_sync(0xffffffffu, !failed(&s_fail) && mbar_wait(&bars.s_full[s], (j >> 1) & 1));
      if (!ok) break;
      fence_after_sync();
      uint32_t x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t (&xc)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[c * 32]);
        tmem_ld32(lane_base + C::T_S + s * 128 + c * 32, xc);
      }
      tmem_ld_wait();
      const int valid = min(128, sh.n - j * 128);   // keys of this tile that exist
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        float v = __uint_as_float(x[c]) * scale_log2;
        v = c < valid ? v : -INFINITY;
        x[c] = __float_as_uint(v);
        mt = fmaxf(mt, v);
      }
      const bool grow = mt > m_ref + C::kRescale;
      const float m_new = grow ? mt : m_ref;
      const float alpha = grow ? fast_exp2(m_ref - m_new) : 1.f;
      // P (bf16) into shared memory once the buffer's previous PV product is done
      ok = __all_sync(0xffffffffu, mbar_wait(&bars.p_free[s], ((j >> 1) & 1) ^ 1));
      if (!ok) break;
      uint8_t* prow = sm + C::OFF_P + s * C::P_BYTES + r * 128;
      float ts = 0.f;
#pragma unroll
      for (int k8 = 0; k8 < 16; ++k8) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = fast_exp2(__uint_as_float(x[k8 * 8 + 2 * e]) - m_new);
          const float p1 = fast_exp2(__uint_as_float(x[k8 * 8 + 2 * e + 1]) - m_new);
          ts += p0 + p1;
          pk[e] = pack_bf16(p0, p1);
        }
        const int chunk = k8 >> 3, piece = k8 & 7;
        *reinterpret_cast<uint4*>(prow + chunk * C::CHUNK + ((piece ^ (r & 7)) << 4)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      if (st_row) st_row[(int64_t)j * sh.n_pad] = row < sh.n ? (m_new + __log2f(ts)) * kLn2 : -INFINITY;
      l_run = l_run * alpha + ts;
      m_ref = m_new;
      // rescale O in TMEM (rare): PV_{j-1} must have landed first
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars.o_step, (j - 1) & 1));
        if (!ok) break;
        fence_after_sync();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t ov[16];
          tmem_ld16(lane_base + C::T_O + c0, ov);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
          tmem_st16(lane_base + C::T_O + c0, ov);
        }
        tmem_st_wait();
      }
      fence_async_smem();
      fence_before_sync();
      mbar_arrive(&bars.p_ready[s]);
    }
    if (!ok && lane == 0) fail();
    // epilogue: O = acc / l, LSE = ln 2 (m + log2 l), once the last PV product landed
    const bool done = __all_sync(0xffffffffu, ok && mbar_wait(&bars.o_done, 0));
    fence_after_sync();
    const float inv = 1.f / l_run;
    __nv_bfloat16* orow = o + (((int64_t)b * sh.n + row) * sh.H + h) * D;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t ov[32];
      if (done) {
        tmem_ld32(lane_base + C::T_O + c0, ov);
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
    if (row < sh.n)
      lse[bh * sh.n + row] = done ? (m_ref + __log2f(l_run)) * kLn2 : __uint_as_float(0x7fc00000u);
    if (!done && lane == 0) fail();
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_free(tmem, C::T_COLS);
}

template <int D>
cudaError_t launch_t(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                     float* lse, float* stats, int32_t* status, float scale, cudaStream_t st) {
  using C = FCfg<D>;
  CUtensorMap mq, mk, mv;
  if (!make_bshd_map(&mq, q, sh.B, sh.n, sh.H, D, 128) ||
      !make_bshd_map(&mk, k, sh.B, sh.n, sh.Hk, D, 128) ||
      !make_bshd_map(&mv, v, sh.B, sh.n, sh.Hk, D, 128))
    return cudaErrorInvalidValue;
  const int smem = C::BYTES + 1024;
  auto kern = fwd_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(sh.T_r, sh.H, sh.B);
  kern<<<grid, 256, smem, st>>>(mq, mk, mv, (__nv_bfloat16*)o, lse, stats, status, sh,
                                scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace

bool fwd_tc_supported(const Shape& sh) {
  return sh.block_q == 128 && sh.block_k == 128 && (sh.d == 64 || sh.d == 128);
}

cudaError_t launch_fwd_tc(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                          float* lse, float* stats, int32_t* status, float scale,
                          cudaStream_t st) {
  if (sh.d == 128) return launch_t<128>(sh, q, k, v, o, lse, stats, status, scale, st);
  return launch_t<64>(sh, q, k, v, o, lse, stats, status, scale, st);
}

}  // namespace bl
