// LSE-combine: merge partial attention results over disjoint key sets
// ("BackLite" README, Key properties: the LSE output serves to combine partial
// attention results).  For every (batch, row, head):
//   LSE = log sum_p exp(LSE_p),  O = sum_p exp(LSE_p - LSE) O_p,
// parts with LSE_p = -inf carry no weight; a row with no finite part gets
// O = 0 and LSE = -inf.
//
// The pass is bound by HBM: parts*(2d+4) bytes in, 2d+4 bytes out per row.
// Thread = EPT consecutive elements (EPT/8 16-byte loads per part) of one
// row; rows are numbered in the LSE's [B, H, n] order, so the threads of a
// warp read LSE values of consecutive rows and whole 2d-byte output rows.
// Every thread of a row forms the same weights from the parts' LSEs (a
// broadcast read).  The parts are taken GP at a time and all loads of a group
// are issued before any is used: (EPT, GP) = (16, 2) for up to two parts,
// (8, 4) otherwise, which keeps 64 B per thread in flight at a register count
// that leaves the SM well occupied.
#include "common.cuh"
#include "kernels.h"

namespace bl {

namespace {

__device__ __forceinline__ void fma_bf16x8(float* acc, const uint4& raw, float w) {
  const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[e]));
    acc[2 * e] = fmaf(w, f.x, acc[2 * e]);
    acc[2 * e + 1] = fmaf(w, f.y, acc[2 * e + 1]);
  }
}

template <int D, int EPT, int GP>
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ o_parts,
                                                      const float* __restrict__ lse_parts,
                                                      __nv_bfloat16* __restrict__ o,
                                                      float* __restrict__ lse, int parts, int B,
                                                      int n, int H) {
  constexpr int TPR = D / EPT;   // threads per row
  constexpr int NV = EPT / 8;    // 16-byte vectors per part
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t rows = (int64_t)B * n * H;
  const int64_t lrow = gid / TPR;          // row in [B, H, n] order
  const int chunk = (int)(gid % TPR);
  if (lrow >= rows) return;
  const int r = (int)(lrow % n);
  const int64_t bh = lrow / n;
  const int h = (int)(bh % H);
  const int b = (int)(bh / H);
  const int64_t orow = ((int64_t)b * n + r) * H + h;   // row of the BSHD tensors
  float m = -INFINITY;
  for (int p = 0; p < parts; ++p) m = fmaxf(m, lse_parts[p * rows + lrow]);
  float acc[EPT];
#pragma unroll
  for (int e = 0; e < EPT; ++e) acc[e] = 0.f;
  float out_lse = -INFINITY;
  if (!isinf(m)) {
    float tot = 0.f;
    for (int p = 0; p < parts; ++p) {
      const float lp = lse_parts[p * rows + lrow];
      tot += isinf(lp) ? 0.f : __expf(lp - m);
    }
    const float inv = 1.f / tot;
    const __nv_bfloat16* src = o_parts + orow * D + chunk * EPT;
    const int64_t pstride = rows * D;
    for (int p = 0; p < parts; p += GP) {
      uint4 raw[GP][NV];
      float w[GP];
#pragma unroll
      for (int u = 0; u < GP; ++u) {
        const bool in = p + u < parts;
        const uint4* s4 = reinterpret_cast<const uint4*>(src + (int64_t)(p + u) * pstride);
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) raw[u][vv] = in ? s4[vv] : make_uint4(0u, 0u, 0u, 0u);
        const float lp = in ? lse_parts[(p + u) * rows + lrow] : -INFINITY;
        w[u] = isinf(lp) ? 0.f : __expf(lp - m) * inv;
      }
#pragma unroll
      for (int u = 0; u < GP; ++u)
#pragma unroll
        for (int vv = 0; vv < NV; ++vv) fma_bf16x8(acc + 8 * vv, raw[u][vv], w[u]);
    }
    out_lse = m + __logf(tot);
  }
  if (chunk == 0) lse[lrow] = out_lse;
  uint4* dst = reinterpret_cast<uint4*>(o + orow * D + chunk * EPT);
#pragma unroll
  for (int vv = 0; vv < NV; ++vv) {
    const float* a = acc + 8 * vv;
    dst[vv] = make_uint4(pack_bf16(a[0], a[1]), pack_bf16(a[2], a[3]), pack_bf16(a[4], a[5]),
                         pack_bf16(a[6], a[7]));
  }
}

template <int D>
void launch_d(int parts, int B, int n, int H, const void* o_parts, const float* lse_parts,
              void* o, float* lse, cudaStream_t st) {
  const int64_t rows = (int64_t)B * n * H;
  const auto* op = (const __nv_bfloat16*)o_parts;
  auto* out = (__nv_bfloat16*)o;
  if (parts <= 2) {
    const unsigned blocks = (unsigned)((rows * (D / 16) + 255) / 256);
    combine_kernel<D, 16, 2><<<blocks, 256, 0, st>>>(op, lse_parts, out, lse, parts, B, n, H);
  } else {
    const unsigned blocks = (unsigned)((rows * (D / 8) + 255) / 256);
    combine_kernel<D, 8, 4><<<blocks, 256, 0, st>>>(op, lse_parts, out, lse, parts, B, n, H);
  }
}

}  // namespace

cudaError_t launch_combine(int parts, int B, int n, int H, int d, const void* o_parts,
                           const float* lse_parts, void* o, float* lse, cudaStream_t st) {
  if (d == 128)
    launch_d<128>(parts, B, n, H, o_parts, lse_parts, o, lse, st);
  else
    launch_d<64>(parts, B, n, H, o_parts, lse_parts, o, lse, st);
  return cudaGetLastError();
}

}  // namespace bl
