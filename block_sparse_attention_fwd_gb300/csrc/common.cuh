// Shared device helpers for the bl_attn kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bl {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Shape {
  int B, n, H, Hk, d, block_q, block_k;
  int T_r, T_c;
  int64_t n_pad;  // T_r * block_q
  int causal, window;
  // element strides of the batch, sequence and head dims (the d stride is 1)
  // of q and g_q (qs), k and g_k (ks), v and g_v (vs), o and g_o (os)
  int64_t qs[3], ks[3], vs[3], os[3];
  bool strided;   // some tensor is not contiguous BSHD
};

// Element offset of (batch b, row r, head h) in a BSHD tensor with strides s.
__host__ __device__ __forceinline__ int64_t bshd(const int64_t (&s)[3], int b, int r, int h) {
  return (int64_t)b * s[0] + (int64_t)r * s[1] + (int64_t)h * s[2];
}

// Key tiles [lo, hi] of query tile i that hold at least one attending
// (query, key) pair under the causal / sliding-window structure: causal keeps
// keys c <= r, so the last such tile holds the tile's last row; a window W
// keeps keys c >= r - W + 1, so the first holds key r0 - W + 1 of the tile's
// first row r0.  Without structure the range is every key tile.
__host__ __device__ __forceinline__ void key_tile_range(const Shape& sh, int i, int& lo, int& hi) {
  lo = 0;
  hi = sh.T_c - 1;
  const int r0 = i * sh.block_q;
  const int r1 = min(sh.n, (i + 1) * sh.block_q) - 1;
  if (sh.causal) hi = min(hi, r1 / sh.block_k);
  if (sh.window) {
    const int x = r0 - sh.window + 1;
    if (x > 0) lo = x / sh.block_k;
  }
}

// True when no (query, key) pair of tile (i, j) attends.
__host__ __device__ __forceinline__ bool tile_empty(const Shape& sh, int i, int j) {
  if (!sh.causal && !sh.window) return false;
  int lo, hi;
  key_tile_range(sh, i, lo, hi);
  return j < lo || j > hi;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100 family): one instruction does the round-to-nearest
// fma / add of two independent lanes, which halves the issue slots of
// elementwise softmax arithmetic.  A pair lives in a 64-bit register (low
// word first).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (NaN inputs ignored, as fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace bl
