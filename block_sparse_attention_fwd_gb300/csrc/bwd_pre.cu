// Block-sparse attention backward: the passes around the tcgen05 kernel.
//
// "Introducing BackLite", Backpropagation for attention:
//   G_V = P^T G_O, G_P = G_O V^T, D = diag(G_O O^T), G_S = G_P (.) P - diag(D) P,
//   G_Q = G_S K s, G_K = G_S^T Q s    (s = softmax scale).
// The tiled split follows the Flash Attention explainer, Flash Attention
// Backward Pass: a preprocessing pass computes D_i = rowsum(dO_i (.) O_i);
// the main pass (bwd_tc.cu) fixes a key tile and streams the query tiles the
// mask keeps for it; dQ receives the partial products dS K through fp32
// reduce-adds into a workspace accumulator, which a final pass scales and
// rounds to bf16.
#include "common.cuh"
#include "kernels.h"

namespace bl {

namespace {

// D[b,h,r] = sum_d G_O[b,r,h,d] * O[b,r,h,d].  One warp per (b, block of 32
// rows r, h), h fastest, so the eight warps of a block read neighbouring
// heads of the same rows.  D / 8 lanes share a row (16 bytes of O and of G_O
// each), and 32 / (D / 8) rows go per step; the loads of four steps are in
// flight together.  Lane l keeps D of row r0 + l, so the warp writes its 32
// values with one coalesced store.  The warp also zeroes its rows of the fp32
// dQ accumulator, and block 0 the status word and the word after it (the
// tcgen05 backward's work-item counter), so no separate memset pass is needed.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ g_o,
                                                      float* __restrict__ Dv,
                                                      float* __restrict__ dq_acc,
                                                      int32_t* __restrict__ status, Shape sh) {
  constexpr int LPR = D / 8;        // lanes per row
  constexpr int RPS = 32 / LPR;     // rows per step
  constexpr int STEPS = 32 / RPS;
  constexpr int U = 4;              // steps whose loads are in flight together
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    status[0] = 0;
    status[1] = 0;
  }
  const int nblk = (sh.n + 31) / 32;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= (int64_t)sh.B * nblk * sh.H) return;
  const int h = (int)(w % sh.H);
  const int64_t br = w / sh.H;
  const int b = (int)(br / nblk);
  const int r0 = (int)(br % nblk) * 32;
  const int sub = lane / LPR, c8 = (lane % LPR) * 8;
  float d_mine = 0.f;
#pragma unroll
  for (int s0 = 0; s0 < STEPS; s0 += U) {
    uint4 ov[U], gv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + (s0 + u) * RPS + sub;
      ov[u] = make_uint4(0u, 0u, 0u, 0u);
      gv[u] = ov[u];
      if (r < sh.n) {
        const int64_t off = bshd(sh.os, b, r, h) + c8;
        ov[u] = *reinterpret_cast<const uint4*>(o + off);
        gv[u] = *reinterpret_cast<const uint4*>(g_o + off);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t* a = reinterpret_cast<const uint32_t*>(&ov[u]);
      const uint32_t* c = reinterpret_cast<const uint32_t*>(&gv[u]);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[e]));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&c[e]));
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      // row (s0 + u) * RPS + i sits in lanes i * LPR ...; lane l takes row l
      const float v = __shfl_sync(0xffffffffu, acc, (lane % RPS) * LPR);
      if (lane / RPS == s0 + u) d_mine = v;
    }
  }
  if (r0 + lane < sh.n) Dv[((int64_t)b * sh.H + h) * sh.n + r0 + lane] = d_mine;
  // zero the accumulator rows (b, r0..r0+31, h): D fp32 = D / 4 float4 per row
  constexpr int F4 = D / 4;
#pragma unroll 4
  for (int x = lane; x < 32 * F4; x += 32) {
    const int r = r0 + x / F4;
    if (r < sh.n)
      reinterpret_cast<float4*>(dq_acc + (((int64_t)b * sh.n + r) * sh.H + h) * D)[x % F4] =
          make_float4(0.f, 0.f, 0.f, 0.f);
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

}  // namespace

cudaError_t launch_bwd(const Shape& sh, const void* q, const void* k, const void* v,
                       const void* o, const void* g_o, const float* lse, float scale,
                       const int32_t* q_idx, const int32_t* q_cnt, void* g_q, void* g_k,
                       void* g_v, float* ws_D, float* ws_dq, int32_t* ws_sub,
                       int32_t* ws_status, cudaStream_t st) {
  const int64_t rows = (int64_t)sh.B * sh.n * sh.H;
  const int64_t pre_warps = (int64_t)sh.B * ((sh.n + 31) / 32) * sh.H;
  unsigned pre_blocks = (unsigned)((pre_warps + 7) / 8);
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
  e = launch_bwd_tc(sh, q, k, v, g_o, lse, ws_D, q_idx, q_cnt, g_k, g_v, ws_dq, ws_sub, ws_status,
                    scale, st);
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
