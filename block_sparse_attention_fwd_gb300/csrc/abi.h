// Host-side helpers shared by the C entry points of libbl_attn.so: shape
// validation and the backward workspace layout.
#pragma once

#include <math.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/bl_attn.h"
#include "common.cuh"
#include "kernels.h"

namespace bl {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates a public shape and fills the internal one (tile counts included).
bl_status check_shape(const bl_shape* s, Shape* out);

// Backward workspace: D [B,H,n] fp32 (rounded up to 256 bytes), then the fp32
// dQ accumulator [B,n,H,d], then (64-wide tiles only) the lists of 128 x 128
// tiles with quarter masks, then 256 bytes for the status word and the
// work-item counter.
inline size_t ws_D_bytes(const Shape& sh) {
  size_t b = (size_t)sh.B * sh.H * sh.n * sizeof(float);
  return (b + 255) & ~(size_t)255;
}
inline size_t ws_dq_bytes(const Shape& sh) {
  return (size_t)sh.B * sh.n * sh.H * sh.d * sizeof(float);
}
inline size_t ws_sub_bytes(const Shape& sh) { return bwd_sub_lists_bytes(sh); }
// Byte offset of the status word.
inline size_t ws_status_off(const Shape& sh) {
  return ws_D_bytes(sh) + ws_dq_bytes(sh) + ws_sub_bytes(sh);
}
constexpr size_t kWsStatusBytes = 256;

// Integer skip threshold of the mask pass, T = ceil(negl_prob * 2^40); the
// product is exact in fp64.  negl_prob must lie in [0, 1).
inline unsigned long long mask_threshold(double negl_prob) {
  return (unsigned long long)ceil(negl_prob * 1099511627776.0);
}

}  // namespace bl
