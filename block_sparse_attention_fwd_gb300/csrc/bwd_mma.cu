// Block-sparse attention backward.
//
// "Introducing BackLite", Backpropagation for attention:
//   G_V = P^T G_O, G_P = G_O V^T, D = diag(G_O O^T), G_S = G_P (.) P - diag(D) P,
//   G_Q = G_S K s, G_K = G_S^T Q s    (s = softmax scale).
// Using Sparsity: P is masked by the tile mask recorded from the forward and
// the same mask serves G_V, G_S and both products with Q and K; a skipped
// tile is neither loaded nor computed.  The tiled split follows the Flash
// Attention explainer, Flash Attention Backward Pass: a preprocessing pass
// computes D_i = rowsum(dO_i (.) O_i); the main pass fixes a key tile j,
// keeps K_j, V_j and the dK_j, dV_j accumulators on chip, and streams the
// query tiles i that the mask keeps for (i, j).  dQ_i receives the partial
// products dS_ij K_j through fp32 atomic adds into a workspace accumulator,
// which a final pass scales and rounds to bf16.
//
// Main pass work split: one CTA per (key tile, kv head, batch) with one warp
// per 16 keys.  For GQA the CTA walks every query head of its group, each
// with that head's own list of kept query tiles.  Query tiles are processed
// in chunks of 64 rows.  Each warp holds S^T = K_w Q^T (16 x 64) on
// m16n8k16 bf16 MMAs with fp32 accumulators, so rows are keys and the
// per-query LSE and D enter as column vectors.
#include "common.cuh"
#include "kernels.h"

namespace bl {

namespace {

constexpr int QC = 64;  // query rows per chunk

// D[b,h,r] = sum_d G_O[b,r,h,d] * O[b,r,h,d]: one warp per (b, r, h) row.
// The same warp zeroes that row of the fp32 dQ accumulator, and block 0 the
// status word and the word after it (the tcgen05 backward's work-item
// counter), so no separate memset pass is needed.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ g_o,
                                                      float* __restrict__ Dv,
                                                      float* __restrict__ dq_acc,
                                                      int32_t* __restrict__ status, Shape sh) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t total = (int64_t)sh.B * sh.n * sh.H;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    status[0] = 0;
    status[1] = 0;
  }
  if (row >= total) return;
  {
    float* z = dq_acc + row * D + lane * (D / 32);
    if constexpr (D == 128)
      *reinterpret_cast<float4*>(z) = make_float4(0.f, 0.f, 0.f, 0.f);
    else
      *reinterpret_cast<float2*>(z) = make_float2(0.f, 0.f);
  }
  constexpr int E = D / 32;  // elements per lane (2 or 4)
  const int rh = (int)(row % sh.H);
  const int64_t rbr = row / sh.H;
  const int64_t ro = bshd(sh.os, (int)(rbr / sh.n), (int)(rbr % sh.n), rh);
  const __nv_bfloat16* op = o + ro + lane * E;
  const __nv_bfloat16* gp = g_o + ro + lane * E;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(op + e));
    float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(gp + e));
    acc += a.x * c.x + a.y * c.y;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    int h = (int)(row % sh.H);
    int64_t br = row / sh.H;
    int r = (int)(br % sh.n);
    int b = (int)(br / sh.n);
    Dv[((int64_t)b * sh.H + h) * sh.n + r] = acc;
  }
}

template <int D, int BK>
__global__ void __launch_bounds__(BK * 2) bwd_dkdv_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g_o,
    const float* __restrict__ lse, const float* __restrict__ Dv, const int32_t* __restrict__ q_idx,
    const int32_t* __restrict__ q_cnt, __nv_bfloat16* __restrict__ g_k,
    __nv_bfloat16* __restrict__ g_v, float* __restrict__ dq_acc, int32_t* __restrict__ status,
    Shape sh, float scale, float scale_log2) {
  constexpr int NW = BK / 16;
  constexpr int CH = D / 8;
  constexpr int ND = D / 8;
  constexpr int NQ = QC / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem;
  uint8_t* sV = sK + BK * D * 2;
  uint8_t* sQ = sV + BK * D * 2;
  uint8_t* sG = sQ + QC * D * 2;
  uint8_t* sS = sG + QC * D * 2;                       // dS^T [BK][QC] bf16
  float* sL = reinterpret_cast<float*>(sS + BK * QC * 2);  // lse * log2 e
  float* sDv = sL + QC;

  const int j = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = sh.H / sh.Hk;
  const int key0 = j * BK;
  const int64_t ks = (int64_t)sh.Hk * D, qs = (int64_t)sh.H * D;
  const __nv_bfloat16* kb = k + ((int64_t)b * sh.n * sh.Hk + hk) * D;
  const __nv_bfloat16* vb = v + ((int64_t)b * sh.n * sh.Hk + hk) * D;

  for (int idx = tid; idx < BK * CH; idx += blockDim.x) {
    int r = idx / CH, c = idx % CH, gr = key0 + r;
    bool ok = gr < sh.n;
    int64_t off = (int64_t)(ok ? gr : 0) * ks + c * 8;
    cp_async16(smem_u32(sK) + swz<CH>(r, c), kb + off, ok ? 16 : 0);
    cp_async16(smem_u32(sV) + swz<CH>(r, c), vb + off, ok ? 16 : 0);
  }
  cp_async_commit();

  float dk[ND][4], dv[ND][4];
#pragma unroll
  for (int i = 0; i < ND; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

  const bool key_ok[2] = {key0 + warp * 16 + g < sh.n, key0 + warp * 16 + g + 8 < sh.n};

  for (int gi = 0; gi < G; ++gi) {
    const int h = hk * G + gi;
    const int64_t bh = (int64_t)b * sh.H + h;
    int cnt = sh.T_r;
    const int32_t* list = nullptr;
    if (q_idx) {
      cnt = q_cnt[bh * sh.T_c + j];
      list = q_idx + (bh * sh.T_c + j) * (int64_t)sh.T_r;
      if (cnt < 0 || cnt > sh.T_r) {
        if (tid == 0) atomicOr(status, 1);
        cnt = 0;
      }
    }
    const __nv_bfloat16* qb = q + ((int64_t)b * sh.n * sh.H + h) * D;
    const __nv_bfloat16* gb = g_o + ((int64_t)b * sh.n * sh.H + h) * D;
    for (int li = 0; li < cnt; ++li) {
      const int i = list ? list[li] : li;
      if (i < 0 || i >= sh.T_r) {
        if (tid == 0) atomicOr(status, 1);
        continue;
      }
      for (int r0 = i * sh.block_q; r0 < (i + 1) * sh.block_q && r0 < sh.n; r0 += QC) {
        for (int idx = tid; idx < QC * CH; idx += blockDim.x) {
          int r = idx / CH, c = idx % CH, gr = r0 + r;
          bool ok = gr < sh.n;
          int64_t off = (int64_t)(ok ? gr : 0) * qs + c * 8;
          cp_async16(smem_u32(sQ) + swz<CH>(r, c), qb + off, ok ? 16 : 0);
          cp_async16(smem_u32(sG) + swz<CH>(r, c), gb + off, ok ? 16 : 0);
        }
        cp_async_commit();
        for (int r = tid; r < QC; r += blockDim.x) {
          int gr = r0 + r;
          bool ok = gr < sh.n;
          sL[r] = ok ? lse[bh * sh.n + gr] * kLog2e : INFINITY;
          sDv[r] = ok ? Dv[bh * sh.n + gr] : 0.f;
        }
        cp_async_wait<0>();
        __syncthreads();

        // S^T = K_w Q^T and dP^T = V_w G_O^T, both 16 x QC per warp
        float st[NQ][4], dp[NQ][4];
#pragma unroll
        for (int x = 0; x < NQ; ++x)
#pragma unroll
          for (int e = 0; e < 4; ++e) st[x][e] = dp[x][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t ak[4], av[4];
          uint32_t aoff = swz<CH>(warp * 16 + (lane & 15), kk * 2 + (lane >> 4));
          ldsm_x4(smem_u32(sK) + aoff, ak[0], ak[1], ak[2], ak[3]);
          ldsm_x4(smem_u32(sV) + aoff, av[0], av[1], av[2], av[3]);
#pragma unroll
          for (int nb2 = 0; nb2 < QC / 16; ++nb2) {
            uint32_t boff = swz<CH>(nb2 * 16 + (lane & 7) + ((lane >> 4) << 3),
                                    kk * 2 + ((lane >> 3) & 1));
            uint32_t b0, b1, b2, b3;
            ldsm_x4(smem_u32(sQ) + boff, b0, b1, b2, b3);
            mma_bf16(st[2 * nb2], ak, b0, b1);
            mma_bf16(st[2 * nb2 + 1], ak, b2, b3);
            ldsm_x4(smem_u32(sG) + boff, b0, b1, b2, b3);
            mma_bf16(dp[2 * nb2], av, b0, b1);
            mma_bf16(dp[2 * nb2 + 1], av, b2, b3);
          }
        }
        // P^T = exp2(S^T s log2e - lse log2e); dS^T = P^T (dP^T - D)
#pragma unroll
        for (int x = 0; x < NQ; ++x) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            int c = x * 8 + 2 * t + (e & 1);
            float p = key_ok[e >> 1] ? fast_exp2(st[x][e] * scale_log2 - sL[c]) : 0.f;
            st[x][e] = p;
            dp[x][e] = p * (dp[x][e] - sDv[c]);
          }
          // dS^T to shared memory as bf16 [key][q] for the dQ product
          *reinterpret_cast<uint32_t*>(sS + swz<QC / 8>(warp * 16 + g, x) + 4 * t) =
              pack_bf16(dp[x][0], dp[x][1]);
          *reinterpret_cast<uint32_t*>(sS + swz<QC / 8>(warp * 16 + g + 8, x) + 4 * t) =
              pack_bf16(dp[x][2], dp[x][3]);
        }
        // dV += P^T G_O and dK += dS^T Q (A from registers, B = [q][d] tiles, transposed loads)
#pragma unroll
        for (int kk = 0; kk < QC / 16; ++kk) {
          uint32_t ap[4], as[4];
          ap[0] = pack_bf16(st[2 * kk][0], st[2 * kk][1]);
          ap[1] = pack_bf16(st[2 * kk][2], st[2 * kk][3]);
          ap[2] = pack_bf16(st[2 * kk + 1][0], st[2 * kk + 1][1]);
          ap[3] = pack_bf16(st[2 * kk + 1][2], st[2 * kk + 1][3]);
          as[0] = pack_bf16(dp[2 * kk][0], dp[2 * kk][1]);
          as[1] = pack_bf16(dp[2 * kk][2], dp[2 * kk][3]);
          as[2] = pack_bf16(dp[2 * kk + 1][0], dp[2 * kk + 1][1]);
          as[3] = pack_bf16(dp[2 * kk + 1][2], dp[2 * kk + 1][3]);
#pragma unroll
          for (int nd2 = 0; nd2 < D / 16; ++nd2) {
            uint32_t boff = swz<CH>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                    nd2 * 2 + (lane >> 4));
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(smem_u32(sG) + boff, b0, b1, b2, b3);
            mma_bf16(dv[2 * nd2], ap, b0, b1);
            mma_bf16(dv[2 * nd2 + 1], ap, b2, b3);
            ldsm_x4_t(smem_u32(sQ) + boff, b0, b1, b2, b3);
            mma_bf16(dk[2 * nd2], as, b0, b1);
            mma_bf16(dk[2 * nd2 + 1], as, b2, b3);
          }
        }
        __syncthreads();

        // dQ partial (QC x D) = dS K: units of 16 query rows x 16 dims over the warps
        constexpr int UNITS = (QC / 16) * (D / 16);
        for (int u = warp; u < UNITS; u += NW) {
          const int mb = u / (D / 16), nb2 = u % (D / 16);
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            uint32_t a[4], b0, b1, b2, b3;
            ldsm_x4_t(smem_u32(sS) + swz<QC / 8>(kk * 16 + (lane & 7) + ((lane >> 4) << 3),
                                                 mb * 2 + ((lane >> 3) & 1)),
                      a[0], a[1], a[2], a[3]);
            ldsm_x4_t(smem_u32(sK) + swz<CH>(kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3),
                                             nb2 * 2 + (lane >> 4)),
                      b0, b1, b2, b3);
            mma_bf16(acc[0], a, b0, b1);
            mma_bf16(acc[1], a, b2, b3);
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            int r = r0 + mb * 16 + g + 8 * hh;
            if (r >= sh.n) continue;
            float* dst = dq_acc + (((int64_t)b * sh.n + r) * sh.H + h) * D + nb2 * 16 + 2 * t;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              atomicAdd(dst + x * 8, acc[x][2 * hh]);
              atomicAdd(dst + x * 8 + 1, acc[x][2 * hh + 1]);
            }
          }
        }
        __syncthreads();
      }
    }
  }

  cp_async_wait<0>();  // K/V copies are still in flight when no tile was kept

  // write dK (scaled) and dV rows of the key tile
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    if (!key_ok[hh]) continue;
    int key = key0 + warp * 16 + g + 8 * hh;
    __nv_bfloat16* kr = g_k + (((int64_t)b * sh.n + key) * sh.Hk + hk) * D;
    __nv_bfloat16* vr = g_v + (((int64_t)b * sh.n + key) * sh.Hk + hk) * D;
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      *reinterpret_cast<uint32_t*>(kr + nd * 8 + 2 * t) =
          pack_bf16(dk[nd][2 * hh] * scale, dk[nd][2 * hh + 1] * scale);
      *reinterpret_cast<uint32_t*>(vr + nd * 8 + 2 * t) =
          pack_bf16(dv[nd][2 * hh], dv[nd][2 * hh + 1]);
    }
  }
}

// G_Q = bf16(s * dq_acc); with STRIDED, G_Q has the strides sh.qs (the
// accumulator is contiguous [B,n,H,d]).
template <bool STRIDED>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ acc,
                                                         uint2* __restrict__ g_q, int64_t n4,
                                                         float scale, Shape sh) {
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n4;
       x += (int64_t)gridDim.x * blockDim.x) {
    float4 a = acc[x];
    uint2 r;
    r.x = pack_bf16(a.x * scale, a.y * scale);
    r.y = pack_bf16(a.z * scale, a.w * scale);
    if constexpr (STRIDED) {
      const int64_t e = x * 4, row = e / sh.d, br = row / sh.H;
      const int64_t off = bshd(sh.qs, (int)(br / sh.n), (int)(br % sh.n), (int)(row % sh.H)) +
                          e % sh.d;
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(g_q) + off) = r;
    } else {
      g_q[x] = r;
    }
  }
}

template <int D, int BK>
cudaError_t launch_dkdv_t(const Shape& sh, const void* q, const void* k, const void* v,
                          const void* g_o, const float* lse, const float* Dv,
                          const int32_t* q_idx, const int32_t* q_cnt, void* g_k, void* g_v,
                          float* dq_acc, int32_t* status, float scale, cudaStream_t st) {
  size_t smem = (size_t)(2 * BK + 2 * QC) * D * 2 + (size_t)BK * QC * 2 + 2 * QC * 4;
  auto kern = bwd_dkdv_kernel<D, BK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(sh.T_c, sh.Hk, sh.B);
  kern<<<grid, BK * 2, smem, st>>>((const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                   (const __nv_bfloat16*)v, (const __nv_bfloat16*)g_o, lse, Dv,
                                   q_idx, q_cnt, (__nv_bfloat16*)g_k, (__nv_bfloat16*)g_v, dq_acc,
                                   status, sh, scale, scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(const Shape& sh, const void* q, const void* k, const void* v,
                       const void* o, const void* g_o, const float* lse, float scale,
                       const int32_t* q_idx, const int32_t* q_cnt, void* g_q, void* g_k,
                       void* g_v, float* ws_D, float* ws_dq, int32_t* ws_status,
                       cudaStream_t st) {
  const int64_t rows = (int64_t)sh.B * sh.n * sh.H;
  unsigned pre_blocks = (unsigned)((rows + 7) / 8);
  if (sh.d == 64)
    bwd_pre_kernel<64><<<pre_blocks, 256, 0, st>>>((const __nv_bfloat16*)o,
                                                   (const __nv_bfloat16*)g_o, ws_D, ws_dq,
                                                   ws_status, sh);
  else
    bwd_pre_kernel<128><<<pre_blocks, 256, 0, st>>>((const __nv_bfloat16*)o,
                                                    (const __nv_bfloat16*)g_o, ws_D, ws_dq,
                                                    ws_status, sh);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (bwd_tc_supported(sh))
    e = launch_bwd_tc(sh, q, k, v, g_o, lse, ws_D, q_idx, q_cnt, g_k, g_v, ws_dq, ws_status,
                      scale, st);
  else if (sh.d == 64 && sh.block_k == 64)
    e = launch_dkdv_t<64, 64>(sh, q, k, v, g_o, lse, ws_D, q_idx, q_cnt, g_k, g_v, ws_dq, ws_status, scale, st);
  else if (sh.d == 64 && sh.block_k == 128)
    e = launch_dkdv_t<64, 128>(sh, q, k, v, g_o, lse, ws_D, q_idx, q_cnt, g_k, g_v, ws_dq, ws_status, scale, st);
  else if (sh.d == 128 && sh.block_k == 64)
    e = launch_dkdv_t<128, 64>(sh, q, k, v, g_o, lse, ws_D, q_idx, q_cnt, g_k, g_v, ws_dq, ws_status, scale, st);
  else if (sh.d == 128 && sh.block_k == 128)
    e = launch_dkdv_t<128, 128>(sh, q, k, v, g_o, lse, ws_D, q_idx, q_cnt, g_k, g_v, ws_dq, ws_status, scale, st);
  else
    return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  const int64_t n4 = rows * sh.d / 4;
  unsigned cblocks = (unsigned)((n4 + 255) / 256);
  if (cblocks > 152u * 16u) cblocks = 152u * 16u;
  if (sh.strided)
    dq_convert_kernel<true><<<cblocks, 256, 0, st>>>((const float4*)ws_dq, (uint2*)g_q, n4, scale,
                                                     sh);
  else
    dq_convert_kernel<false><<<cblocks, 256, 0, st>>>((const float4*)ws_dq, (uint2*)g_q, n4,
                                                      scale, sh);
  return cudaGetLastError();
}

}  // namespace bl
