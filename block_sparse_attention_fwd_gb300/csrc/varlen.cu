// Packed variable-length batches (declared in include/bl_attn.h).
//
// The sequences are walked on the host, and the fixed-length kernels run once
// per run of consecutive sequences of equal length, on that run's slice of
// every buffer.  Token for token, a run of `count` sequences of length n is a
// [count, n, heads, d] batch, and the packed layout stores each per-sequence
// array exactly as the fixed-length call lays it out for that batch, so every
// result equals the fixed-length call on each sequence alone.
//
// A short sequence's launch fills only part of the 152 SMs, so the runs go
// to a few side streams that the GPU runs side by side: largest run first,
// each to the stream with the least work so far.  The side streams wait on
// an event recorded on the caller's stream and the caller's stream waits on
// one event per side stream, so the work stays ordered with the caller's and
// the calls can be captured in a CUDA graph.  No host wait separates the
// launches.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <numeric>
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
  size_t ws;                                      // byte offset of its D and dQ areas
  double work;                                    // attending tile pairs, for scheduling
};

// Status words of the varlen backward: one 16-byte slot per run (flags word,
// work-item counter), after the runs' D and dQ areas.
constexpr size_t kSlotBytes = 16;
constexpr int kMaxStreams = 8;
constexpr int kDefaultStreams = 8;

struct Plan {
  std::vector<Run> runs;
  bl_varlen_sizes sz;
  size_t ws_areas;     // bytes of all runs' D and dQ areas
  int max_T_c;         // most key tiles of any sequence
  int streams;         // side streams to spread the runs over (1: the caller's only)
};

// (query tile, key tile) pairs of one sequence that hold an attending pair.
double attending_tiles(const bl::Shape& sh) {
  if (!sh.causal && !sh.window) return (double)sh.T_r * sh.T_c;
  double t = 0;
  for (int i = 0; i < sh.T_r; ++i) {
    int lo, hi;
    bl::key_tile_range(sh, i, lo, hi);
    t += hi - lo + 1;
  }
  return t;
}

bl_status make_plan(const bl_varlen* v, Plan* p) {
  if (!v || !v->cu_seqlens || v->nseq < 1) return BL_ERR_INVALID_ARG;
  const int32_t* cu = v->cu_seqlens;
  if (cu[0] != 0) return BL_ERR_INVALID_ARG;
  for (int s = 0; s < v->nseq; ++s)
    if (cu[s + 1] < cu[s]) return BL_ERR_INVALID_ARG;
  if (cu[v->nseq] < 1) return BL_ERR_INVALID_ARG;
  if (v->streams < 0 || v->streams > kMaxStreams) return BL_ERR_INVALID_ARG;
  // The head and tile fields follow the fixed-length rules whatever the lengths.
  const bl_shape probe = {1, 1, v->H, v->Hk, v->d, v->block_q, v->block_k, v->causal, v->window};
  bl::Shape sh;
  bl_status st = bl::check_shape(&probe, &sh);
  if (st != BL_OK) return st;

  p->runs.clear();
  memset(&p->sz, 0, sizeof(p->sz));
  p->ws_areas = 0;
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
    r.ws = p->ws_areas;
    p->ws_areas += bl::ws_D_bytes(r.sh) + bl::ws_dq_bytes(r.sh) + bl::ws_sub_bytes(r.sh);
    r.work = r.sh.B * (double)r.sh.H * attending_tiles(r.sh);
    p->runs.push_back(r);
    s = e;
  }
  z.groups = (int)p->runs.size();
  z.bwd_workspace_bytes = p->ws_areas + p->runs.size() * kSlotBytes;
  p->streams = std::min<int>(v->streams ? v->streams : kDefaultStreams, (int)p->runs.size());
  return BL_OK;
}

// Side streams and events of one device, created on first use and kept for
// the life of the process.  `mu` serialises the fork/launch/join sequence of
// a call, because the events are reused from call to call.
struct Pool {
  std::mutex mu;
  bool ready = false;
  cudaStream_t side[kMaxStreams] = {};
  cudaEvent_t fork = nullptr, join[kMaxStreams] = {};
};
constexpr int kMaxDevices = 64;
Pool g_pool[kMaxDevices];

cudaError_t pool_init(Pool& pl) {
  if (pl.ready) return cudaSuccess;
  cudaError_t e = cudaEventCreateWithFlags(&pl.fork, cudaEventDisableTiming);
  for (int i = 0; i < kMaxStreams && e == cudaSuccess; ++i) {
    e = cudaStreamCreateWithFlags(&pl.side[i], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pl.join[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) pl.ready = true;
  return e;
}

// Runs launch(run, stream) for every run of the plan: all on the caller's
// stream when the plan uses one stream, else spread over the side streams
// between a fork and a join on the caller's stream.  The join is enqueued
// even when a launch fails, so the caller's stream never runs ahead of work
// already enqueued.
template <typename F>
bl_status run_all(const Plan& p, cudaStream_t caller, F&& launch) {
  if (p.streams <= 1) {
    for (const Run& r : p.runs)
      if (launch(r, caller) != cudaSuccess) return BL_ERR_CUDA;
    return BL_OK;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return BL_ERR_CUDA;
  Pool& pl = g_pool[dev];
  std::lock_guard<std::mutex> lock(pl.mu);
  if (pool_init(pl) != cudaSuccess) return BL_ERR_CUDA;

  std::vector<size_t> order(p.runs.size());
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](size_t a, size_t b) { return p.runs[a].work > p.runs[b].work; });
  double load[kMaxStreams] = {};

  cudaError_t e = cudaEventRecord(pl.fork, caller);
  if (e != cudaSuccess) return BL_ERR_CUDA;
  for (int i = 0; i < p.streams; ++i)
    if (cudaStreamWaitEvent(pl.side[i], pl.fork, 0) != cudaSuccess) e = cudaErrorUnknown;
  if (e == cudaSuccess) {
    for (size_t idx : order) {
      const int i = (int)(std::min_element(load, load + p.streams) - load);
      load[i] += p.runs[idx].work;
      if ((e = launch(p.runs[idx], pl.side[i])) != cudaSuccess) break;
    }
  }
  bl_status st = e == cudaSuccess ? BL_OK : BL_ERR_CUDA;
  for (int i = 0; i < p.streams; ++i) {
    if (cudaEventRecord(pl.join[i], pl.side[i]) != cudaSuccess ||
        cudaStreamWaitEvent(caller, pl.join[i], 0) != cudaSuccess)
      st = BL_ERR_CUDA;
  }
  return st;
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
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + p.ws_areas +
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
  return run_all(p, (cudaStream_t)stream, [&](const Run& r, cudaStream_t st) {
    return bl::launch_fwd(r.sh, rows(q, r.tok, H, d), rows(k, r.tok, Hk, d),
                          rows(v, r.tok, Hk, d), rows(o, r.tok, H, d), lse + r.lse,
                          at(tile_stats, r.stats), scale, st);
  });
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
  return run_all(p, (cudaStream_t)stream, [&](const Run& r, cudaStream_t st) {
    return bl::launch_mask(r.sh, tile_stats + r.stats, lse + r.lse, nullptr, T,
                           lists->mask + r.mask,
                           lists->kv_idx + r.mask, lists->kv_cnt + r.kv_cnt,
                           lists->q_idx + r.q_idx, lists->q_cnt + r.q_cnt, lists->nan_count,
                           st);
  });
}

size_t bl_fwd_workspace_bytes_varlen(const bl_varlen* varlen) {
  Plan p;
  if (make_plan(varlen, &p) != BL_OK) return 0;
  for (const Run& r : p.runs)
    if (!bl::fwd_tile_weights_supported(r.sh)) return 0;
  return bl::fwd_scratch_bytes(varlen->d, p.max_T_c);
}

bl_status bl_attn_fwd_tile_weights_varlen(const bl_varlen* varlen, const void* q, const void* k,
                                          const void* v, float scale, void* o, float* lse,
                                          float* tile_stats, float* tile_logw, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  Plan p;
  bl_status st = make_plan(varlen, &p);
  if (st != BL_OK) return st;
  if (!q || !k || !v || !o || !lse || !tile_logw) return BL_ERR_INVALID_ARG;
  if (!bl::aligned16(q) || !bl::aligned16(k) || !bl::aligned16(v) || !bl::aligned16(o) ||
      !aligned4(lse) || !aligned4(tile_logw) || (tile_stats && !bl::aligned16(tile_stats)))
    return BL_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return BL_ERR_INVALID_ARG;
  for (const Run& r : p.runs)
    if (!bl::fwd_tile_weights_supported(r.sh)) return BL_ERR_UNSUPPORTED;
  if (!tile_stats) {
    const size_t need = bl::fwd_scratch_bytes(varlen->d, p.max_T_c);
    if (need == 0) return BL_ERR_CUDA;
    if (!workspace || !bl::aligned16(workspace) || workspace_bytes < need)
      return BL_ERR_WORKSPACE;
    // every launch group claims slots of the one scratch (sized for the
    // longest sequence): its locks are cleared once, on the caller's stream
    // before the groups fork
    if (bl::fwd_scratch_clear(varlen->d, workspace, (cudaStream_t)stream) != cudaSuccess)
      return BL_ERR_CUDA;
  }
  const int H = varlen->H, Hk = varlen->Hk, d = varlen->d;
  return run_all(p, (cudaStream_t)stream, [&](const Run& r, cudaStream_t st) {
    return bl::launch_fwd_tc(r.sh, rows(q, r.tok, H, d), rows(k, r.tok, Hk, d),
                             rows(v, r.tok, Hk, d), rows(o, r.tok, H, d), lse + r.lse,
                             at(tile_stats, r.stats), tile_logw + r.mask,
                             tile_stats ? nullptr : workspace, scale, st, p.max_T_c,
                             /*zero_locks=*/false);
  });
}

bl_status bl_mask_from_tile_weights_varlen(const bl_varlen* varlen, const float* tile_logw,
                                           double negl_prob, const bl_lists* lists,
                                           void* stream) {
  Plan p;
  bl_status st = make_plan(varlen, &p);
  if (st != BL_OK) return st;
  if (!tile_logw || !lists) return BL_ERR_INVALID_ARG;
  if (!lists->mask || !lists->kv_idx || !lists->kv_cnt || !lists->q_idx || !lists->q_cnt)
    return BL_ERR_INVALID_ARG;
  if (!aligned4(tile_logw)) return BL_ERR_INVALID_ARG;
  if (!(negl_prob >= 0.0) || !(negl_prob < 1.0)) return BL_ERR_INVALID_ARG;
  if (p.max_T_c > 2048) return BL_ERR_UNSUPPORTED;
  const unsigned long long T = bl::mask_threshold(negl_prob);
  return run_all(p, (cudaStream_t)stream, [&](const Run& r, cudaStream_t st) {
    return bl::launch_mask(r.sh, nullptr, nullptr, tile_logw + r.mask, T, lists->mask + r.mask,
                           lists->kv_idx + r.mask, lists->kv_cnt + r.kv_cnt,
                           lists->q_idx + r.q_idx, lists->q_cnt + r.q_cnt, lists->nan_count,
                           st);
  });
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
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return run_all(p, (cudaStream_t)stream, [&](const Run& r, cudaStream_t st) {
    float* ws_D = reinterpret_cast<float*>(ws + r.ws);
    float* ws_dq = reinterpret_cast<float*>(ws + r.ws + bl::ws_D_bytes(r.sh));
    int32_t* ws_sub =
        reinterpret_cast<int32_t*>(ws + r.ws + bl::ws_D_bytes(r.sh) + bl::ws_dq_bytes(r.sh));
    const size_t idx = (size_t)(&r - p.runs.data());
    return bl::launch_bwd(
        r.sh, rows(q, r.tok, H, d), rows(k, r.tok, Hk, d), rows(v, r.tok, Hk, d),
        rows(o, r.tok, H, d), rows(g_o, r.tok, H, d), lse + r.lse, scale,
        lists ? lists->q_idx + r.q_idx : nullptr, lists ? lists->q_cnt + r.q_cnt : nullptr,
        rows(g_q, r.tok, H, d), rows(g_k, r.tok, Hk, d), rows(g_v, r.tok, Hk, d), ws_D, ws_dq,
        ws_sub, status_slot(workspace, p, idx), st);
  });
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
