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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async global->shared copy; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D (fp32)
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

// Byte offset of 16-byte chunk `c` of row `r` in a tile whose rows hold
// `CH` chunks (CH >= 8), XOR-swizzled so that any 8 consecutive rows read at
// the same logical chunk hit 8 distinct bank groups (conflict-free ldmatrix).
template <int CH>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  static_assert(CH >= 8, "rows must span at least 128 bytes");
  return static_cast<uint32_t>((r * CH + (c ^ (r & 7))) * 16);
}

}  // namespace bl
