// Attention forward with per-(query row, key tile) LSE statistics.
//
// "Introducing BackLite", Backpropagation for attention: S = s Q K^T,
// P = softmax_row(S), O = P V, computed exactly (Using Sparsity).  "BackLite"
// README, How It Works, Phase 1: the forward also records the log-sum-exp of
// every (query row, key tile).  The row softmax is evaluated online, one key
// tile at a time (Flash Attention explainer, Online Softmax and Flash
// Attention: running max m and running sum l, with the accumulator rescaled
// by exp(m_old - m_new) whenever the max grows).
//
// Work split: one CTA of 4 warps per (64-row query block, head, batch); each
// warp owns 16 query rows and runs the whole key loop on m16n8k16 bf16 tensor
// core MMAs with fp32 accumulation.  Scores are kept in base 2
// (x * s * log2 e) so every exponential is one ex2.
#include "common.cuh"
#include "kernels.h"

namespace bl {

namespace {

template <int D, int BK>
__global__ void __launch_bounds__(128) fwd_mma_kernel(const __nv_bfloat16* __restrict__ q,
                                                      const __nv_bfloat16* __restrict__ k,
                                                      const __nv_bfloat16* __restrict__ v,
                                                      __nv_bfloat16* __restrict__ o,
                                                      float* __restrict__ lse,
                                                      float* __restrict__ stats, Shape sh,
                                                      float scale_log2) {
  constexpr int BQ = 64;
  constexpr int CH = D / 8;
  constexpr int NB = BK / 8;   // n8 blocks of S per warp
  constexpr int ND = D / 8;    // n8 blocks of O per warp
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + BQ * D * 2;
  uint8_t* sV = sK + BK * D * 2;

  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (sh.H / sh.Hk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * BQ;
  const int64_t qs = (int64_t)sh.H * D, ks = (int64_t)sh.Hk * D;
  const __nv_bfloat16* qb = q + ((int64_t)b * sh.n * sh.H + h) * D;
  const __nv_bfloat16* kb = k + ((int64_t)b * sh.n * sh.Hk + hk) * D;
  const __nv_bfloat16* vb = v + ((int64_t)b * sh.n * sh.Hk + hk) * D;
  float* st_bh = stats ? stats + ((int64_t)b * sh.H + h) * sh.T_c * sh.n_pad : nullptr;

  if (row0 >= sh.n) {
    // padding rows of the last statistics tile: no query exists there
    if (st_bh)
      for (int idx = tid; idx < sh.T_c * BQ; idx += blockDim.x)
        st_bh[(int64_t)(idx / BQ) * sh.n_pad + row0 + idx % BQ] = -INFINITY;
    return;
  }

  for (int idx = tid; idx < BQ * CH; idx += blockDim.x) {
    int r = idx / CH, c = idx % CH, gr = row0 + r;
    bool ok = gr < sh.n;
    cp_async16(smem_u32(sQ) + swz<CH>(r, c), qb + (int64_t)(ok ? gr : 0) * qs + c * 8, ok ? 16 : 0);
  }
  cp_async_commit();

  float acc[ND][4];
#pragma unroll
  for (int i = 0; i < ND; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};

  for (int j = 0; j < sh.T_c; ++j) {
    const int col0 = j * BK;
    for (int idx = tid; idx < BK * CH; idx += blockDim.x) {
      int r = idx / CH, c = idx % CH, gr = col0 + r;
      bool ok = gr < sh.n;
      int64_t off = (int64_t)(ok ? gr : 0) * ks + c * 8;
      cp_async16(smem_u32(sK) + swz<CH>(r, c), kb + off, ok ? 16 : 0);
      cp_async16(smem_u32(sV) + swz<CH>(r, c), vb + off, ok ? 16 : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    float s[NB][4];
#pragma unroll
    for (int i = 0; i < NB; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4];
      ldsm_x4(smem_u32(sQ) + swz<CH>(warp * 16 + (lane & 15), kk * 2 + (lane >> 4)), a[0], a[1],
              a[2], a[3]);
#pragma unroll
      for (int nb2 = 0; nb2 < BK / 16; ++nb2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(sK) + swz<CH>(nb2 * 16 + (lane & 7) + ((lane >> 4) << 3),
                                       kk * 2 + ((lane >> 3) & 1)),
                b0, b1, b2, b3);
        mma_bf16(s[2 * nb2], a, b0, b1);
        mma_bf16(s[2 * nb2 + 1], a, b2, b3);
      }
    }

    // scale to base 2, drop key columns past n, tile max per row
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int col = col0 + nb * 8 + 2 * t + (e & 1);
        float x = col < sh.n ? s[nb][e] * scale_log2 : -INFINITY;
        s[nb][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    }
    float m_new[2], alpha[2], ts[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      m_new[r] = fmaxf(m_run[r], mx[r]);
      alpha[r] = fast_exp2(m_run[r] - m_new[r]);
    }
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float p = fast_exp2(s[nb][e] - m_new[e >> 1]);
        s[nb][e] = p;
        ts[e >> 1] += p;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      ts[r] += __shfl_xor_sync(0xffffffffu, ts[r], 1);
      ts[r] += __shfl_xor_sync(0xffffffffu, ts[r], 2);
      l_run[r] = l_run[r] * alpha[r] + ts[r];
      m_run[r] = m_new[r];
    }
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      acc[nd][0] *= alpha[0];
      acc[nd][1] *= alpha[0];
      acc[nd][2] *= alpha[1];
      acc[nd][3] *= alpha[1];
    }
    // tile statistic: LSE_{r,j} = ln 2 * (m_new + log2(sum of this tile's p))
    if (st_bh && t == 0) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        int row = row0 + warp * 16 + g + 8 * r;
        st_bh[(int64_t)j * sh.n_pad + row] =
            row < sh.n ? (m_new[r] + __log2f(ts[r])) * kLn2 : -INFINITY;
      }
    }

    // O += P V
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < D / 16; ++nd2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(sV) + swz<CH>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                         nd2 * 2 + (lane >> 4)),
                  b0, b1, b2, b3);
        mma_bf16(acc[2 * nd2], a, b0, b1);
        mma_bf16(acc[2 * nd2 + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }

  // epilogue: O = acc / l, LSE = ln 2 * (m + log2 l)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    int row = row0 + warp * 16 + g + 8 * r;
    if (row >= sh.n) continue;
    float inv = 1.f / l_run[r];
    __nv_bfloat16* orow = o + (((int64_t)b * sh.n + row) * sh.H + h) * D;
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      uint32_t pk = pack_bf16(acc[nd][2 * r] * inv, acc[nd][2 * r + 1] * inv);
      *reinterpret_cast<uint32_t*>(orow + nd * 8 + 2 * t) = pk;
    }
    if (t == 0) lse[((int64_t)b * sh.H + h) * sh.n + row] = (m_run[r] + __log2f(l_run[r])) * kLn2;
  }
}

template <int D, int BK>
cudaError_t launch_fwd_t(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                         float* lse, float* stats, float scale, cudaStream_t st) {
  constexpr int BQ = 64;
  size_t smem = (size_t)(BQ + 2 * BK) * D * 2;
  auto kern = fwd_mma_kernel<D, BK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(sh.n_pad / BQ), sh.H, sh.B);
  kern<<<grid, 128, smem, st>>>((const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                (const __nv_bfloat16*)v, (__nv_bfloat16*)o, lse, stats, sh,
                                scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                       float* lse, float* stats, float scale, cudaStream_t st) {
  if (fwd_tc_supported(sh))
    return launch_fwd_tc(sh, q, k, v, o, lse, stats, nullptr, nullptr, scale, st);
  if (sh.d == 64 && sh.block_k == 64) return launch_fwd_t<64, 64>(sh, q, k, v, o, lse, stats, scale, st);
  if (sh.d == 64 && sh.block_k == 128) return launch_fwd_t<64, 128>(sh, q, k, v, o, lse, stats, scale, st);
  if (sh.d == 128 && sh.block_k == 64) return launch_fwd_t<128, 64>(sh, q, k, v, o, lse, stats, scale, st);
  if (sh.d == 128 && sh.block_k == 128) return launch_fwd_t<128, 128>(sh, q, k, v, o, lse, stats, scale, st);
  return cudaErrorInvalidValue;
}

}  // namespace bl
