// Packed variable-length batches (declared in include/bl_attn.h).
//
// The sequences are walked on the host, and the fixed-length kernels run once
// per run of consecutive sequences of equal length, on that run's slice of
// every buffer.  Token for token, a run of `count` sequences of length n is a
// [count, n, heads, d] batch, and the packed layout stores each per-sequence
// array exactly as the fixed-length call lays it out for that batch, so every
// result equals the fixed-length call on each sequence alone.  No host wait
// separates the launches.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "../../include/bl_attn.h"
#include "abi.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// One run of equal-length sequences and its offsets into the packed buffers.
struct Run {
  bl::Shape sh;                                   // B = sequences of the run, n = their length
  int64_t tok;                                    // first token row of q/k/v/o and gradients
  size_t lse, stats, mask, kv_cnt, q_idx, q_cnt;  // element offsets of the run's blocks
};

// Status words of the varlen backward: one 16-byte slot per run (flags word,
// work-item counter), after the shared D and dQ areas.
constexpr size_t kSlotBytes = 16;

struct Plan {
  std::vector<Run> runs;
  bl_varlen_sizes sz;
  size_t ws_D, ws_dq;  // largest D and dQ areas over the runs
  int max_T_c;         // most key tiles of any sequence
};

bl_status make_plan(const bl_varlen* v, Plan* p) {
  if (!v || !v->cu_seqlens || v->nseq < 1) return BL_ERR_INVALID_ARG;
  const int32_t* cu = v->cu_seqlens;
  if (cu[0] != 0) return BL_ERR_INVALID_ARG;
  for (int s = 0; s < v->nseq; ++s)
    if (cu[s + 1] < cu[s]) return BL_ERR_INVALID_ARG;
  if (cu[v->nseq] < 1) return BL_ERR_INVALID_ARG;
  // The head and tile fields follow the fixed-length rules whatever the lengths.
  const bl_shape probe = {1, 1, v->H, v->Hk, v->d, v->block_q, v->block_k, v->causal, v->window};
  bl::Shape sh;
  bl_status st = bl::check_shape(&probe, &sh);
  if (st != BL_OK) return st;

  p->runs.clear();
  memset(&p->sz, 0, sizeof(p->sz));
  p->ws_D = p->ws_dq = 0;
  p->max_T_c = 0;
  bl_varlen_sizes& z = p->sz;
  z.total = (size_t)cu[v->nseq];
  z.lse = (size_t)v->H * z.total;
  for (int s = 0; s < v->nseq;) {
    const int n = cu[s + 1] - cu[s];
    if (n == 0) {
      ++s;
      continue;
    }
    int e = s + 1;
    while (e < v->nseq && cu[e + 1] - cu[e] == n && e - s < 65535) ++e;
    const bl_shape run_shape = {e - s, n, v->H, v->Hk, v->d, v->block_q, v->block_k,
                                v->causal, v->window};
    Run r;
    st = bl::check_shape(&run_shape, &r.sh);
    if (st != BL_OK) return st;
    p->max_T_c = std::max(p->max_T_c, r.sh.T_c);
    const size_t BH = (size_t)r.sh.B * r.sh.H;
    r.tok = cu[s];
    r.lse = (size_t)v->H * cu[s];
    r.stats = z.tile_stats;
    r.mask = z.mask;
    r.kv_cnt = z.kv_cnt;
    r.q_idx = z.q_idx;
    r.q_cnt = z.q_cnt;
    z.tile_stats += BH * r.sh.T_c * (size_t)r.sh.n_pad;
    z.mask += BH * r.sh.T_r * r.sh.T_c;
    z.kv_cnt += BH * r.sh.T_r;
    z.q_idx += BH * r.sh.T_c * r.sh.T_r;
    z.q_cnt += BH * r.sh.T_c;
    p->ws_D = std::max(p->ws_D, bl::ws_D_bytes(r.sh));
    p->ws_dq = std::max(p->ws_dq, bl::ws_dq_bytes(r.sh));
    p->runs.push_back(r);
    s = e;
  }
  z.groups = (int)p->runs.size();
  z.bwd_workspace_bytes = p->ws_D + p->ws_dq + p->runs.size() * kSlotBytes;
  return BL_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

template <typename T>
T* at(T* base, size_t elems) {
  return base ? base + elems : nullptr;
}

const __nv_bfloat16* rows(const void* base, int64_t tok, int heads, int d) {
  return static_cast<const __nv_bfloat16*>(base) + tok * heads * d;
}
__nv_bfloat16* rows(void* base, int64_t tok, int heads, int d) {
  return static_cast<__nv_bfloat16*>(base) + tok * heads * d;
}

int32_t* status_slot(void* workspace, const Plan& p, size_t run) {
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + p.ws_D + p.ws_dq +
                                    run * kSlotBytes);
}

}  // namespace

extern "C" {

bl_status bl_varlen_layout(const bl_varlen* varlen, bl_varlen_sizes* sizes) {
  if (!sizes) return BL_ERR_INVALID_ARG;
  Plan p;
  bl_status st = make_plan(varlen, &p);
  if (st == BL_OK) *sizes = p.sz;
  return st;
}

bl_status bl_attn_fwd_varlen(const bl_varlen* varlen, const void* q, const void* k,
                             const void* v, float scale, void* o, float* lse, float* tile_stats,
                             void* stream) {
  Plan p;
  bl_status st = make_plan(varlen, &p);
  if (st != BL_OK) return st;
  if (!q || !k || !v || !o || !lse) return BL_ERR_INVALID_ARG;
  if (!bl::aligned16(q) || !bl::aligned16(k) || !bl::aligned16(v) || !bl::aligned16(o) ||
      !aligned4(lse) || (tile_stats && !bl::aligned16(tile_stats)))
    return BL_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return BL_ERR_INVALID_ARG;
  const int H = varlen->H, Hk = varlen->Hk, d = varlen->d;
  for (const Run& r : p.runs) {
    cudaError_t e = bl::launch_fwd(r.sh, rows(q, r.tok, H, d), rows(k, r.tok, Hk, d),
                                   rows(v, r.tok, Hk, d), rows(o, r.tok, H, d), lse + r.lse,
                                   at(tile_stats, r.stats), scale, (cudaStream_t)stream);
    if (e != cudaSuccess) return BL_ERR_CUDA;
  }
  return BL_OK;
}

bl_status bl_mask_from_stats_varlen(const bl_varlen* varlen, const float* tile_stats,
                                    const float* lse, double negl_prob, const bl_lists* lists,
                                    void* stream) {
  Plan p;
  bl_status st = make_plan(varlen, &p);
  if (st != BL_OK) return st;
  if (!tile_stats || !lse || !lists) return BL_ERR_INVALID_ARG;
  if (!lists->mask || !lists->kv_idx || !lists->kv_cnt || !lists->q_idx || !lists->q_cnt)
    return BL_ERR_INVALID_ARG;
  if (!bl::aligned16(tile_stats) || !aligned4(lse)) return BL_ERR_INVALID_ARG;
  if (!(negl_prob >= 0.0) || !(negl_prob < 1.0)) return BL_ERR_INVALID_ARG;
  if (p.max_T_c > 2048) return BL_ERR_UNSUPPORTED;
  const unsigned long long T = bl::mask_threshold(negl_prob);
  for (const Run& r : p.runs) {
    cudaError_t e = bl::launch_mask(r.sh, tile_stats + r.stats, lse + r.lse, T,
                                    lists->mask + r.mask, lists->kv_idx + r.mask,
                                    lists->kv_cnt + r.kv_cnt, lists->q_idx + r.q_idx,
                                    lists->q_cnt + r.q_cnt, lists->nan_count,
                                    (cudaStream_t)stream);
    if (e != cudaSuccess) return BL_ERR_CUDA;
  }
  return BL_OK;
}

bl_status bl_attn_bwd_varlen(const bl_varlen* varlen, const void* q, const void* k,
                             const void* v, const void* o, const void* g_o, const float* lse,
                             float scale, const bl_lists* lists, void* g_q, void* g_k,
                             void* g_v, void* workspace, size_t workspace_bytes, void* stream) {
  Plan p;
  bl_status st = make_plan(varlen, &p);
  if (st != BL_OK) return st;
  const void* ptrs[] = {q, k, v, o, g_o, g_q, g_k, g_v};
  for (const void* ptr : ptrs)
    if (!ptr || !bl::aligned16(ptr)) return BL_ERR_INVALID_ARG;
  if (!lse || !aligned4(lse)) return BL_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return BL_ERR_INVALID_ARG;
  if (lists && (!lists->q_idx || !lists->q_cnt)) return BL_ERR_INVALID_ARG;
  if (!workspace || !bl::aligned16(workspace)) return BL_ERR_WORKSPACE;
  if (workspace_bytes < p.sz.bwd_workspace_bytes) return BL_ERR_WORKSPACE;
  const int H = varlen->H, Hk = varlen->Hk, d = varlen->d;
  float* ws_D = static_cast<float*>(workspace);
  float* ws_dq = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + p.ws_D);
  for (size_t i = 0; i < p.runs.size(); ++i) {
    const Run& r = p.runs[i];
    cudaError_t e = bl::launch_bwd(
        r.sh, rows(q, r.tok, H, d), rows(k, r.tok, Hk, d), rows(v, r.tok, Hk, d),
        rows(o, r.tok, H, d), rows(g_o, r.tok, H, d), lse + r.lse, scale,
        lists ? lists->q_idx + r.q_idx : nullptr, lists ? lists->q_cnt + r.q_cnt : nullptr,
        rows(g_q, r.tok, H, d), rows(g_k, r.tok, Hk, d), rows(g_v, r.tok, Hk, d), ws_D, ws_dq,
        status_slot(workspace, p, i), (cudaStream_t)stream);
    if (e != cudaSuccess) return BL_ERR_CUDA;
  }
  return BL_OK;
}

bl_status bl_varlen_bwd_check_status(const bl_varlen* varlen, const void* workspace,
                                     void* stream) {
  Plan p;
  bl_status st = make_plan(varlen, &p);
  if (st != BL_OK) return st;
  if (!workspace) return BL_ERR_WORKSPACE;
  std::vector<int32_t> host(p.runs.size() * (kSlotBytes / sizeof(int32_t)));
  cudaError_t e = cudaMemcpyAsync(host.data(), status_slot(const_cast<void*>(workspace), p, 0),
                                  host.size() * sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return BL_ERR_CUDA;
  int32_t flags = 0;
  for (size_t i = 0; i < p.runs.size(); ++i) flags |= host[i * (kSlotBytes / sizeof(int32_t))];
  if (flags & 2) return BL_ERR_TIMEOUT;
  return (flags & 1) ? BL_ERR_CORRUPT_LISTS : BL_OK;
}

}  // extern "C"
