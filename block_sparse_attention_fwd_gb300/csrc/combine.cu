// LSE-combine: merge partial attention results over disjoint key sets
// ("BackLite" README, Key properties: the LSE output serves to combine partial
// attention results).  For every (batch, row, head):
//   LSE = log sum_p exp(LSE_p),  O = sum_p exp(LSE_p - LSE) O_p,
// parts with LSE_p = -inf carry no weight; a row with no finite part gets
// O = 0 and LSE = -inf.
//
// One warp per (b, r, h) row: lane p < parts holds LSE_p, the warp reduces the
// max and the weight sum with shuffles, then every lane accumulates d/32
// elements of every part in fp32 (coalesced 128/256-byte row reads).  The
// pass is bound by HBM: parts*(2d+4) bytes in, 2d+4 bytes out per row.
#include "common.cuh"
#include "kernels.h"

namespace bl {

namespace {

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ o_parts,
                                                      const float* __restrict__ lse_parts,
                                                      __nv_bfloat16* __restrict__ o,
                                                      float* __restrict__ lse, int parts, int B,
                                                      int n, int H) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)B * n * H;
  if (row >= rows) return;
  const int h = (int)(row % H);
  const int64_t br = row / H;
  const int r = (int)(br % n);
  const int b = (int)(br / n);
  const int64_t lse_off = ((int64_t)b * H + h) * n + r;
  const int64_t lse_stride = (int64_t)B * H * n;
  const float lp = lane < parts ? lse_parts[lane * lse_stride + lse_off] : -INFINITY;
  float m = lp;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  constexpr int E = D / 32;   // elements per lane
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  if (isinf(m)) {   // no part saw a key for this row
    if (lane == 0) lse[lse_off] = -INFINITY;
  } else {
    const float w_l = isinf(lp) ? 0.f : __expf(lp - m);
    float tot = w_l;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    const float inv = 1.f / tot;
    for (int p = 0; p < parts; ++p) {
      const float w = __shfl_sync(0xffffffffu, w_l, p) * inv;
      const __nv_bfloat16* src = o_parts + ((int64_t)p * rows + row) * D + lane * E;
      if constexpr (E == 4) {
        uint2 raw = *reinterpret_cast<const uint2*>(src);
        float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.x));
        float2 c = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&raw.y));
        acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * c.x; acc[3] += w * c.y;
      } else {
        float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src));
        acc[0] += w * a.x; acc[1] += w * a.y;
      }
    }
    if (lane == 0) lse[lse_off] = m + __logf(tot);
  }
  __nv_bfloat16* dst = o + row * D + lane * E;
  if constexpr (E == 4) {
    uint2 w2;
    w2.x = pack_bf16(acc[0], acc[1]);
    w2.y = pack_bf16(acc[2], acc[3]);
    *reinterpret_cast<uint2*>(dst) = w2;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0], acc[1]);
  }
}

}  // namespace

cudaError_t launch_combine(int parts, int B, int n, int H, int d, const void* o_parts,
                           const float* lse_parts, void* o, float* lse, cudaStream_t st) {
  const int64_t rows = (int64_t)B * n * H;
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  if (d == 128)
    combine_kernel<128><<<blocks, 256, 0, st>>>((const __nv_bfloat16*)o_parts, lse_parts,
                                                (__nv_bfloat16*)o, lse, parts, B, n, H);
  else
    combine_kernel<64><<<blocks, 256, 0, st>>>((const __nv_bfloat16*)o_parts, lse_parts,
                                               (__nv_bfloat16*)o, lse, parts, B, n, H);
  return cudaGetLastError();
}

}  // namespace bl
