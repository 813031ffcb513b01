// bl_attn_bwd_noalloc: the block-sparse backward without a caller-supplied
// workspace, for callers that cannot call cudaMalloc themselves -- for
// example a host runtime that owns all device memory through its own pool
// and lets no library allocate behind its back, or a latency-critical caller
// that cannot accept the implicit device synchronisation of cudaMalloc.
//
// The scratch the backward needs (D = rowsum(G_O * O), the fp32 dQ
// accumulator and the status word) lives in one fixed array in device
// global memory, BL_NOALLOC_SCRATCH_BYTES long, that every GPU loading this
// library holds until the process exits.  The call itself allocates
// nothing: no cudaMalloc, no cudaFree, no allocating library routine.
#include <math.h>

#include <mutex>

#include "../../include/bl_attn.h"
#include "abi.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// The scratch array.  In host code this name is only a host-side stand-in
// for the symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[BL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).  nullptr on failure.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" bl_status bl_attn_bwd_noalloc(const bl_shape* shape, const void* q, const void* k,
                                         const void* v, const void* o, const void* g_o,
                                         const float* lse, float scale, const bl_lists* lists,
                                         void* g_q, void* g_k, void* g_v, void* stream) {
  if (!shape) return BL_ERR_INVALID_ARG;
  const size_t need = bl_bwd_workspace_bytes(shape);
  if (need == 0)  // invalid shape: bl_attn_bwd returns its shape error before any launch
    return bl_attn_bwd(shape, q, k, v, o, g_o, lse, scale, lists, g_q, g_k, g_v, nullptr, 0,
                       stream);
  if (need > (size_t)BL_NOALLOC_SCRATCH_BYTES) return BL_ERR_WORKSPACE;
  const void* ptrs[] = {q, k, v, o, g_o, lse, g_q, g_k, g_v};
  for (const void* p : ptrs)
    if (!p || !bl::aligned16(p)) return BL_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return BL_ERR_INVALID_ARG;
  if (lists && (!lists->q_idx || !lists->q_cnt)) return BL_ERR_INVALID_ARG;
  unsigned char* ws = static_cast<unsigned char*>(scratch_address());
  if (!ws) return BL_ERR_CUDA;

  bl::Shape sh;
  if (bl::check_shape(shape, &sh) != BL_OK) return BL_ERR_INVALID_ARG;  // unreachable: need > 0
  // Same layout as the workspace of bl_attn_bwd.  The preprocessing kernel
  // that launch_bwd runs first writes every D entry and zeroes the dQ
  // accumulator and the status word, so nothing left by an earlier call leaks
  // into this one.
  float* ws_D = reinterpret_cast<float*>(ws);
  float* ws_dq = reinterpret_cast<float*>(ws + bl::ws_D_bytes(sh));
  int32_t* ws_sub = reinterpret_cast<int32_t*>(ws + bl::ws_D_bytes(sh) + bl::ws_dq_bytes(sh));
  int32_t* ws_status = reinterpret_cast<int32_t*>(ws + bl::ws_status_off(sh));
  cudaError_t e = bl::launch_bwd(sh, q, k, v, o, g_o, lse, scale, lists ? lists->q_idx : nullptr,
                                 lists ? lists->q_cnt : nullptr, g_q, g_k, g_v, ws_D, ws_dq,
                                 ws_sub, ws_status, (cudaStream_t)stream);
  return e == cudaSuccess ? BL_OK : BL_ERR_CUDA;
}

// The status word of the last bl_attn_bwd_noalloc call on this device with
// this shape: it sits in the scratch array where the workspace layout of that
// shape puts it.  Reading it allocates nothing either.
extern "C" bl_status bl_bwd_noalloc_check_status(const bl_shape* shape, void* stream) {
  bl::Shape sh;
  bl_status s = bl::check_shape(shape, &sh);
  if (s != BL_OK) return s;
  if (bl_bwd_workspace_bytes(shape) > (size_t)BL_NOALLOC_SCRATCH_BYTES) return BL_ERR_WORKSPACE;
  const unsigned char* ws = static_cast<const unsigned char*>(scratch_address());
  if (!ws) return BL_ERR_CUDA;
  const int32_t* st =
      reinterpret_cast<const int32_t*>(ws + bl::ws_status_off(sh));
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, st, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return BL_ERR_CUDA;
  if (host & 2) return BL_ERR_TIMEOUT;
  return (host & 1) ? BL_ERR_CORRUPT_LISTS : BL_OK;
}
