// C ABI of libbl_attn.so: argument validation, workspace layout, launches.
// The operations and layouts are documented in include/bl_attn.h.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "../../include/bl_attn.h"
#include "abi.h"
#include "common.cuh"
#include "kernels.h"

namespace bl {

namespace {
constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // 2 s
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
}  // namespace

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

bl_status check_shape(const bl_shape* s, Shape* out) {
  if (!s) return BL_ERR_INVALID_ARG;
  if (s->B < 1 || s->n < 1 || s->H < 1 || s->Hk < 1 || s->H % s->Hk != 0)
    return BL_ERR_INVALID_ARG;
  if (s->B > 65535 || s->H > 65535) return BL_ERR_UNSUPPORTED;
  if (s->d != 64 && s->d != 128) return BL_ERR_UNSUPPORTED;
  if ((s->block_q != 64 && s->block_q != 128) || (s->block_k != 64 && s->block_k != 128))
    return BL_ERR_UNSUPPORTED;
  if (s->causal != 0 && s->causal != 1) return BL_ERR_INVALID_ARG;
  if (s->window < 0 || (s->window > 0 && !s->causal)) return BL_ERR_INVALID_ARG;
  if ((s->causal || s->window) && (s->block_q != 128 || s->block_k != 128))
    return BL_ERR_UNSUPPORTED;
  Shape sh;
  sh.B = s->B; sh.n = s->n; sh.H = s->H; sh.Hk = s->Hk; sh.d = s->d;
  sh.block_q = s->block_q; sh.block_k = s->block_k;
  sh.causal = s->causal; sh.window = s->window;
  sh.T_r = (s->n + s->block_q - 1) / s->block_q;
  sh.T_c = (s->n + s->block_k - 1) / s->block_k;
  sh.n_pad = (int64_t)sh.T_r * s->block_q;
  // strides: all zero means contiguous BSHD; otherwise the d stride is 1 and
  // the others are positive multiples of 8 elements (16 bytes, for TMA)
  sh.strided = false;
  const int64_t* in[4] = {s->q_strides, s->k_strides, s->v_strides, s->o_strides};
  int64_t* dst[4] = {sh.qs, sh.ks, sh.vs, sh.os};
  const int heads[4] = {s->H, s->Hk, s->Hk, s->H};
  for (int t = 0; t < 4; ++t) {
    const int64_t* st = in[t];
    if (st[0] == 0 && st[1] == 0 && st[2] == 0 && st[3] == 0) {
      dst[t][2] = s->d;
      dst[t][1] = (int64_t)heads[t] * s->d;
      dst[t][0] = (int64_t)s->n * heads[t] * s->d;
      continue;
    }
    if (st[3] != 1) return BL_ERR_INVALID_ARG;
    for (int k = 0; k < 3; ++k) {
      if (st[k] <= 0 || st[k] % 8 != 0) return BL_ERR_INVALID_ARG;
      dst[t][k] = st[k];
    }
    if (dst[t][2] < s->d) return BL_ERR_INVALID_ARG;   // rows of one head may not overlap
    if (dst[t][2] != s->d || dst[t][1] != (int64_t)heads[t] * s->d ||
        dst[t][0] != (int64_t)s->n * heads[t] * s->d)
      sh.strided = true;
  }
  *out = sh;
  return BL_OK;
}

}  // namespace bl

namespace {

using bl::aligned16;
using bl::check_shape;
using bl::ws_D_bytes;
using bl::ws_dq_bytes;

bl_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BL_OK : BL_ERR_CUDA; }

}  // namespace

extern "C" {

size_t bl_tile_stats_elems(const bl_shape* shape) {
  bl::Shape sh;
  if (check_shape(shape, &sh) != BL_OK) return 0;
  return (size_t)sh.B * sh.H * sh.T_c * (size_t)sh.n_pad;
}

size_t bl_lists_elems(const bl_shape* shape, size_t out[5]) {
  bl::Shape sh;
  if (!out || check_shape(shape, &sh) != BL_OK) return 0;
  const size_t bh = (size_t)sh.B * sh.H;
  out[0] = out[1] = bh * sh.T_r * sh.T_c;
  out[2] = bh * sh.T_r;
  out[3] = bh * sh.T_c * sh.T_r;
  out[4] = bh * sh.T_c;
  return out[0] + 4 * (out[1] + out[2] + out[3] + out[4]);
}

size_t bl_bwd_workspace_bytes(const bl_shape* shape) {
  bl::Shape sh;
  if (check_shape(shape, &sh) != BL_OK) return 0;
  return bl::ws_status_off(sh) + bl::kWsStatusBytes;
}

bl_status bl_attn_fwd(const bl_shape* shape, const void* q, const void* k, const void* v,
                      float scale, void* o, float* lse, float* tile_stats, void* stream) {
  bl::Shape sh;
  bl_status s = check_shape(shape, &sh);
  if (s != BL_OK) return s;
  if (!q || !k || !v || !o || !lse) return BL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (tile_stats && !aligned16(tile_stats)))
    return BL_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return BL_ERR_INVALID_ARG;
  return cuda_status(bl::launch_fwd(sh, q, k, v, o, lse, tile_stats, scale, (cudaStream_t)stream));
}

bl_status bl_mask_from_stats(const bl_shape* shape, const float* tile_stats, const float* lse,
                             double negl_prob, const bl_lists* lists, void* stream) {
  bl::Shape sh;
  bl_status s = check_shape(shape, &sh);
  if (s != BL_OK) return s;
  if (!tile_stats || !lse || !lists) return BL_ERR_INVALID_ARG;
  if (!lists->mask || !lists->kv_idx || !lists->kv_cnt || !lists->q_idx || !lists->q_cnt)
    return BL_ERR_INVALID_ARG;
  if (!aligned16(tile_stats) || !aligned16(lse)) return BL_ERR_INVALID_ARG;
  if (!(negl_prob >= 0.0) || !(negl_prob < 1.0)) return BL_ERR_INVALID_ARG;
  if (sh.T_c > 2048) return BL_ERR_UNSUPPORTED;
  return cuda_status(bl::launch_mask(sh, tile_stats, lse, nullptr, bl::mask_threshold(negl_prob),
                                     lists->mask, lists->kv_idx, lists->kv_cnt, lists->q_idx,
                                     lists->q_cnt, lists->nan_count, (cudaStream_t)stream));
}

size_t bl_fwd_workspace_bytes(const bl_shape* shape) {
  bl::Shape sh;
  if (check_shape(shape, &sh) != BL_OK || !bl::fwd_tile_weights_supported(sh)) return 0;
  return bl::fwd_scratch_bytes(sh);
}

bl_status bl_attn_fwd_tile_weights(const bl_shape* shape, const void* q, const void* k,
                                   const void* v, float scale, void* o, float* lse,
                                   float* tile_stats, float* tile_logw, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  bl::Shape sh;
  bl_status s = check_shape(shape, &sh);
  if (s != BL_OK) return s;
  if (!q || !k || !v || !o || !lse || !tile_logw) return BL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(tile_logw) || (tile_stats && !aligned16(tile_stats)))
    return BL_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return BL_ERR_INVALID_ARG;
  if (!bl::fwd_tile_weights_supported(sh)) return BL_ERR_UNSUPPORTED;
  if (!tile_stats) {
    const size_t need = bl::fwd_scratch_bytes(sh);
    if (need == 0) return BL_ERR_CUDA;
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return BL_ERR_WORKSPACE;
  }
  return cuda_status(bl::launch_fwd_tc(sh, q, k, v, o, lse, tile_stats, tile_logw,
                                       tile_stats ? nullptr : workspace, scale,
                                       (cudaStream_t)stream));
}

bl_status bl_mask_from_tile_weights(const bl_shape* shape, const float* tile_logw,
                                    double negl_prob, const bl_lists* lists, void* stream) {
  bl::Shape sh;
  bl_status s = check_shape(shape, &sh);
  if (s != BL_OK) return s;
  if (!tile_logw || !lists) return BL_ERR_INVALID_ARG;
  if (!lists->mask || !lists->kv_idx || !lists->kv_cnt || !lists->q_idx || !lists->q_cnt)
    return BL_ERR_INVALID_ARG;
  if (!aligned16(tile_logw)) return BL_ERR_INVALID_ARG;
  if (!(negl_prob >= 0.0) || !(negl_prob < 1.0)) return BL_ERR_INVALID_ARG;
  if (sh.T_c > 2048) return BL_ERR_UNSUPPORTED;
  return cuda_status(bl::launch_mask(sh, nullptr, nullptr, tile_logw,
                                     bl::mask_threshold(negl_prob), lists->mask, lists->kv_idx,
                                     lists->kv_cnt, lists->q_idx, lists->q_cnt, lists->nan_count,
                                     (cudaStream_t)stream));
}

bl_status bl_attn_bwd(const bl_shape* shape, const void* q, const void* k, const void* v,
                      const void* o, const void* g_o, const float* lse, float scale,
                      const bl_lists* lists, void* g_q, void* g_k, void* g_v, void* workspace,
                      size_t workspace_bytes, void* stream) {
  bl::Shape sh;
  bl_status s = check_shape(shape, &sh);
  if (s != BL_OK) return s;
  const void* ptrs[] = {q, k, v, o, g_o, lse, g_q, g_k, g_v};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return BL_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return BL_ERR_INVALID_ARG;
  if (lists && (!lists->q_idx || !lists->q_cnt)) return BL_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return BL_ERR_WORKSPACE;
  if (workspace_bytes < bl_bwd_workspace_bytes(shape)) return BL_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* ws_D = reinterpret_cast<float*>(ws);
  float* ws_dq = reinterpret_cast<float*>(ws + ws_D_bytes(sh));
  int32_t* ws_sub = reinterpret_cast<int32_t*>(ws + ws_D_bytes(sh) + ws_dq_bytes(sh));
  int32_t* ws_status = reinterpret_cast<int32_t*>(ws + bl::ws_status_off(sh));
  return cuda_status(bl::launch_bwd(sh, q, k, v, o, g_o, lse, scale,
                                    lists ? lists->q_idx : nullptr, lists ? lists->q_cnt : nullptr,
                                    g_q, g_k, g_v, ws_D, ws_dq, ws_sub, ws_status,
                                    (cudaStream_t)stream));
}

bl_status bl_bwd_check_status(const bl_shape* shape, const void* workspace, void* stream) {
  bl::Shape sh;
  bl_status s = check_shape(shape, &sh);
  if (s != BL_OK) return s;
  if (!workspace) return BL_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const int32_t* st = reinterpret_cast<const int32_t*>(ws + bl::ws_status_off(sh));
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, st, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return BL_ERR_CUDA;
  if (host & 2) return BL_ERR_TIMEOUT;
  return (host & 1) ? BL_ERR_CORRUPT_LISTS : BL_OK;
}

bl_status bl_lse_combine(int parts, int B, int n, int H, int d, const void* o_parts,
                         const float* lse_parts, void* o, float* lse, void* stream) {
  if (parts < 1 || parts > 32 || B < 1 || n < 1 || H < 1) return BL_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return BL_ERR_UNSUPPORTED;
  if (!o_parts || !lse_parts || !o || !lse) return BL_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o) || !aligned16(lse))
    return BL_ERR_INVALID_ARG;
  return cuda_status(bl::launch_combine(parts, B, n, H, d, o_parts, lse_parts, o, lse,
                                        (cudaStream_t)stream));
}

bl_status bl_grad_error(const void* a, const void* b, size_t n, double* out, void* stream) {
  if (!a || !b || !out || n == 0) return BL_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b) || (reinterpret_cast<uintptr_t>(out) & 7u))
    return BL_ERR_INVALID_ARG;
  return cuda_status(bl::launch_grad_error(a, b, (int64_t)n, out, (cudaStream_t)stream));
}

double bl_set_wait_limit(double seconds) {
  uint64_t v = bl::kDefaultWaitNs;
  if (seconds >= 0.0 && seconds < 2.0) v = (uint64_t)(seconds * 1e9);
  return (double)bl::g_wait_ns.exchange(v) * 1e-9;
}

const char* bl_status_string(bl_status status) {
  switch (status) {
    case BL_OK: return "ok";
    case BL_ERR_INVALID_ARG: return "invalid argument";
    case BL_ERR_UNSUPPORTED: return "unsupported configuration";
    case BL_ERR_CUDA: return "CUDA error";
    case BL_ERR_WORKSPACE: return "workspace missing or too small";
    case BL_ERR_CORRUPT_LISTS: return "tile list entry out of range";
    case BL_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

}  // extern "C"
