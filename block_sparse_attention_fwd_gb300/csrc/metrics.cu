// Error statistics of a bf16 gradient against a bf16 reference, for choosing
// negl_prob ("Introducing BackLite", Using Sparsity: the sparse backward is
// judged by the cosine similarity and relative L2 error of its gradients
// against the dense backward; the post proposes tuning negl_prob to a target
// on them).  For n elements:
//   out[0] = sum (a - b)^2,  out[1] = sum b^2,  out[2] = sum a b,  out[3] = sum a^2
// so rel-L2 = sqrt(out[0] / out[1]) and cos = out[2] / sqrt(out[1] out[3]).
//
// The pass is bound by HBM (4 bytes read per element).  Thread = 8 elements
// per step (one 16-byte load from each array); each step's sums are formed in
// fp32 and added into per-thread fp64 accumulators, then the block reduces
// in fp64 and adds its four sums into out with fp64 atomics.
#include "common.cuh"
#include "kernels.h"

namespace bl {

namespace {

__device__ __forceinline__ void acc8(const uint4& ra, const uint4& rb, double* s) {
  const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w};
  const uint32_t wb[4] = {rb.x, rb.y, rb.z, rb.w};
  float d2 = 0.f, b2 = 0.f, ab = 0.f, a2 = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
    const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[e]));
    const float dx = fa.x - fb.x, dy = fa.y - fb.y;
    d2 += dx * dx + dy * dy;
    b2 += fb.x * fb.x + fb.y * fb.y;
    ab += fa.x * fb.x + fa.y * fb.y;
    a2 += fa.x * fa.x + fa.y * fa.y;
  }
  s[0] += d2;
  s[1] += b2;
  s[2] += ab;
  s[3] += a2;
}

__global__ void __launch_bounds__(256) grad_error_kernel(const __nv_bfloat16* __restrict__ a,
                                                         const __nv_bfloat16* __restrict__ b,
                                                         int64_t n, double* __restrict__ out) {
  __shared__ double red[4][8];
  double s[4] = {0.0, 0.0, 0.0, 0.0};
  const int64_t nv = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const uint4* a4 = reinterpret_cast<const uint4*>(a);
  const uint4* b4 = reinterpret_cast<const uint4*>(b);
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + stride < nv; i += 2 * stride) {   // two independent loads in flight
    const uint4 ra0 = a4[i], rb0 = b4[i], ra1 = a4[i + stride], rb1 = b4[i + stride];
    acc8(ra0, rb0, s);
    acc8(ra1, rb1, s);
  }
  if (i < nv) acc8(a4[i], b4[i], s);
  if (blockIdx.x == 0) {   // the n % 8 tail
    for (int64_t t = nv * 8 + threadIdx.x; t < n; t += blockDim.x) {
      const float x = __bfloat162float(a[t]), y = __bfloat162float(b[t]);
      s[0] += (double)(x - y) * (x - y);
      s[1] += (double)y * y;
      s[2] += (double)x * y;
      s[3] += (double)x * x;
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    double v = s[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) red[c][warp] = v;
  }
  __syncthreads();
  if (threadIdx.x < 4) {
    double v = 0.0;
    for (int w = 0; w < 8; ++w) v += red[threadIdx.x][w];
    atomicAdd(out + threadIdx.x, v);
  }
}

}  // namespace

cudaError_t launch_grad_error(const void* a, const void* b, int64_t n, double* out,
                              cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, 4 * sizeof(double), st);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n / 8 + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  const unsigned blocks = (unsigned)(want < 1 ? 1 : (want < cap ? want : cap));
  grad_error_kernel<<<blocks, 256, 0, st>>>((const __nv_bfloat16*)a, (const __nv_bfloat16*)b, n,
                                            out);
  return cudaGetLastError();
}

}  // namespace bl
