// Host-side launchers of the bl_attn kernels (internal to libbl_attn.so).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bl {

struct Shape;

// Limit (ns of global time) the kernels launched now give every bounded
// device-side wait (bl_set_wait_limit; 2 s by default).
uint64_t wait_limit_ns();

// Forward + optional tile statistics (stats == nullptr skips them).
cudaError_t launch_fwd(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                       float* lse, float* stats, float scale, cudaStream_t st);

// Tile selection: per-query-tile mask row, kv list and count, then the
// transposed per-key-tile q list and count.  From the statistics and the
// LSE, or (stats == nullptr) from the tile weights logw [B,H,T_r,T_c].
cudaError_t launch_mask(const Shape& sh, const float* stats, const float* lse,
                        const float* logw, unsigned long long threshold, uint8_t* mask,
                        int32_t* kv_idx, int32_t* kv_cnt, int32_t* q_idx, int32_t* q_cnt,
                        int32_t* nan_count, cudaStream_t st);

// Backward.  q_idx/q_cnt == nullptr runs every tile.  ws_D [B,H,n] fp32,
// ws_dq [B,n,H,d] fp32, ws_sub bwd_sub_lists_bytes(sh) (64-wide tiles),
// ws_status two int32.
cudaError_t launch_bwd(const Shape& sh, const void* q, const void* k, const void* v,
                       const void* o, const void* g_o, const float* lse, float scale,
                       const int32_t* q_idx, const int32_t* q_cnt, void* g_q, void* g_k,
                       void* g_v, float* ws_D, float* ws_dq, int32_t* ws_sub,
                       int32_t* ws_status, cudaStream_t st);

// tcgen05 dK/dV/dQ pass (head dim 64 or 128).  Shapes with 64-wide tiles run
// as 128 x 128 tiles whose lists (built in sub_ws) carry 64 x 64 quarter masks.
bool bwd_tc_supported(const Shape& sh);
size_t bwd_sub_lists_bytes(const Shape& sh);
cudaError_t launch_bwd_tc(const Shape& sh, const void* q, const void* k, const void* v,
                          const void* g_o, const float* lse, const float* Dv,
                          const int32_t* q_idx, const int32_t* q_cnt, void* g_k, void* g_v,
                          float* dq_acc, int32_t* sub_ws, int32_t* status, float scale,
                          cudaStream_t st);

// tcgen05 forward with tile statistics for 128 x 128 tiles (head dim 64 or
// 128).  logw != nullptr also writes the tile weights [B,H,T_r,T_c]; with
// stats == nullptr their rows go through `scratch` (fwd_scratch_bytes).
bool fwd_tc_supported(const Shape& sh);
bool fwd_tile_weights_supported(const Shape& sh);
size_t fwd_scratch_bytes(const Shape& sh);
size_t fwd_scratch_bytes(int d, int T_c);
// Clears the slot locks of a forward scratch (the first bytes of it).
cudaError_t fwd_scratch_clear(int d, void* scratch, cudaStream_t st);
// slot_tc: key tiles a scratch slot holds (0: sh.T_c); zero_locks: clear the
// slot locks on st first (launches that share a scratch clear it once, before
// any of them).
cudaError_t launch_fwd_tc(const Shape& sh, const void* q, const void* k, const void* v, void* o,
                          float* lse, float* stats, float* logw, void* scratch, float scale,
                          cudaStream_t st, int slot_tc = 0, bool zero_locks = true);

// LSE-combine of `parts` partial results (layouts in include/bl_attn.h).
// Error sums of bf16 a against bf16 b (n elements) into out[4] (fp64).
cudaError_t launch_grad_error(const void* a, const void* b, int64_t n, double* out,
                              cudaStream_t st);
cudaError_t launch_combine(int parts, int B, int n, int H, int d, const void* o_parts,
                           const float* lse_parts, void* o, float* lse, cudaStream_t st);

// 4-D TMA map of a BSHD bf16 tensor [B][n][heads][d] with element strides
// st = {batch, seq, head} (d contiguous): box of 64 elements of d x 1 head x
// `rows` tokens x 1 batch, 128-byte swizzle, out-of-range reads 0.
bool make_bshd_map(CUtensorMap* m, const void* base, int B, int n, int heads, int d, int rows,
                   const int64_t* st);

// The same for an fp32 BSHD tensor, box of 32 elements of d (128 bytes) x 1
// head x `rows` tokens, 128-byte swizzle: the target of dQ reduce-adds.
bool make_bshd_map_f32(CUtensorMap* m, const void* base, int B, int n, int heads, int d,
                       int rows);

}  // namespace bl
