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
