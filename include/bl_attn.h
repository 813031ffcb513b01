/*
 * bl_attn.h -- C ABI of libbl_attn.so: BackLite-style attention on GB300.
 *
 * Three calls make up the hot path, in this order:
 *
 *   bl_attn_fwd         exact attention forward that also records, for every
 *                       (query row, key tile), the log-sum-exp of that row's
 *                       scores over the tile ("BackLite" README, How It Works,
 *                       Phase 1; "Introducing BackLite", Using Sparsity).
 *   bl_mask_from_stats  turns those statistics into a block-sparse mask and
 *                       compacted tile lists (README, How It Works, Phase 2).
 *   bl_attn_bwd         attention backward that reads and computes nothing
 *                       for masked tiles ("Introducing BackLite",
 *                       Backpropagation for attention, and Using Sparsity).
 *
 * Tensors
 *   q, o, g_o, g_q : [B, n, H,  d] bf16 (batch, seq, head, dim), contiguous
 *                    unless bl_shape gives strides
 *   k, v, g_k, g_v : [B, n, Hk, d] bf16, likewise; query head h reads kv
 *                    head h / (H / Hk) (grouped-query attention, README,
 *                    Forward signature: key/value carry heads_k heads).
 *   lse            : [B, H, n] fp32, natural log: LSE_r = log sum_c exp(s q_r.k_c)
 *   tile_stats     : [B, H, T_c, T_r*block_q] fp32, key-tile major:
 *                    tile_stats[b,h,j,r] = log sum_{c in key tile j} exp(s q_r.k_c);
 *                    -inf where the tile's terms underflow and for rows r >= n.
 *   T_r = ceil(n / block_q), T_c = ceil(n / block_k).
 *
 * Every pointer is device memory owned by the caller; the library allocates
 * nothing and frees nothing.  Calls are asynchronous on the given stream
 * (a cudaStream_t passed as void*; NULL is the legacy default stream).
 * Arguments are validated on the host before any launch: a failing check
 * launches nothing and returns an error code.  Device pointers must be
 * 16-byte aligned.
 */
#ifndef BL_ATTN_H
#define BL_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BL_OK = 0,
  BL_ERR_INVALID_ARG = 1,    /* bad shape, pointer, alignment or parameter   */
  BL_ERR_UNSUPPORTED = 2,    /* valid but not built (e.g. head_dim 96)       */
  BL_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed         */
  BL_ERR_WORKSPACE = 4,      /* workspace missing or too small               */
  BL_ERR_CORRUPT_LISTS = 5,  /* a tile list held an out-of-range entry       */
  BL_ERR_TIMEOUT = 6         /* a bounded device-side wait ran out           */
} bl_status;

/* Problem shape.  d in {64, 128}; block_q, block_k in {64, 128}; H % Hk == 0;
 * n >= 1.  One shape describes the forward, the mask and the backward: the
 * statistics, the mask and the backward all use the same block_q x block_k
 * tiles.
 *   causal  0: every query attends to every key; 1: query r attends to keys
 *           c <= r.
 *   window  0: no limit; W > 0 (needs causal = 1): query r attends to keys
 *           r - W < c <= r, the sliding windows the BackLite blog trains
 *           Nanochat with ("Introducing BackLite", Training Nanochat).
 * causal/window need 128 x 128 tiles.  A tile with no attending (query, key)
 * pair has tile statistic -inf and is never kept by the mask. */
typedef struct {
  int B, n, H, Hk, d;
  int block_q, block_k;
  int causal, window;
  /* Element strides of the four BSHD dims [batch, seq, head, dim], for
   * tensors that are views of larger ones (a kv-head slice of a batch, a
   * fused QKV projection): q_strides for q and g_q, k_strides for k and g_k,
   * v_strides for v and g_v, o_strides for o and g_o.  All four entries 0
   * (what a zero-initialised struct holds) means contiguous BSHD.  Otherwise
   * the dim stride is 1, the others positive multiples of 8 (16 bytes), and
   * the head stride at least d.  The packed (varlen) calls take contiguous
   * tensors. */
  int64_t q_strides[4], k_strides[4], v_strides[4], o_strides[4];
} bl_shape;

/* Block-sparse tile lists of one backward, all device memory.
 *   mask   [B,H,T_r,T_c] uint8   1 = compute tile (i, j), 0 = skip
 *   kv_idx [B,H,T_r,T_c] int32   per query tile: active key tiles, ascending,
 *                                then -1 up to T_c
 *   kv_cnt [B,H,T_r]     int32   number of active key tiles per query tile
 *   q_idx  [B,H,T_c,T_r] int32   per key tile: active query tiles, ascending,
 *                                then -1 up to T_r
 *   q_cnt  [B,H,T_c]     int32   number of active query tiles per key tile
 *   nan_count            int32*  optional (may be NULL): the mask pass adds
 *                                the number of NaN tile weights it met (such
 *                                tiles are kept).  The caller zeroes it.
 * The mask is per query head: the heads of one GQA group each have their own
 * lists ("BackLite" README, Key properties: sparsity per sample, per head). */
typedef struct {
  uint8_t* mask;
  int32_t* kv_idx;
  int32_t* kv_cnt;
  int32_t* q_idx;
  int32_t* q_cnt;
  int32_t* nan_count;
} bl_lists;

/* Number of fp32 elements of tile_stats: B*H*T_c*T_r*block_q. */
size_t bl_tile_stats_elems(const bl_shape* shape);

/* Element counts of the five list arrays of bl_lists, written to out[0..4]
 * in field order: mask and kv_idx B*H*T_r*T_c each, kv_cnt B*H*T_r, q_idx
 * B*H*T_c*T_r, q_cnt B*H*T_c.  Returns the total bytes of the five arrays
 * (uint8 mask, int32 others), or 0 for an invalid shape (out untouched). */
size_t bl_lists_elems(const bl_shape* shape, size_t out[5]);

/* Bytes of device workspace bl_attn_bwd needs (16-byte aligned base):
 * D = rowsum(G_O * O) [B,H,n] fp32, the fp32 dQ accumulator [B,n,H,d], with
 * 64-wide tiles the tile lists regrouped into 128 x 128 tiles, a device
 * status word and the backward kernel's work-item counter.  The call
 * initialises all of it, so the workspace needs no clearing between calls;
 * two calls in flight at the same time must not share one. */
size_t bl_bwd_workspace_bytes(const bl_shape* shape);

/* Exact attention forward ("Introducing BackLite", Backpropagation for
 * attention: S = s Q K^T, P = softmax_row(S), O = P V; the forward is not
 * approximated, Using Sparsity).
 *   scale       softmax scale s (finite, > 0); 1/sqrt(d) is the usual value.
 *   o, lse      outputs (layouts above).
 *   tile_stats  output, or NULL to skip recording the statistics (the
 *               negl_prob = 0 path: README, Key properties, zero forward
 *               overhead when nothing will be skipped).
 * Errors: BL_ERR_INVALID_ARG (shape, pointers, alignment, scale),
 *         BL_ERR_UNSUPPORTED (d or tile size), BL_ERR_CUDA (launch). */
bl_status bl_attn_fwd(const bl_shape* shape, const void* q, const void* k,
                      const void* v, float scale, void* o, float* lse,
                      float* tile_stats, void* stream);

/* Tile selection (README, How It Works, Phase 2; Key properties).  For
 * every (b, h, query tile i) and key tile j:
 *   d_ij = max over rows r < n of tile i of fp32(tile_stats[b,h,j,r] - lse[b,h,r]),
 *          clamped to <= 0, so w_ij = exp(d_ij) bounds the weight any row of
 *          the tile puts on key tile j;
 *   E_ij = ceil(detexp(d_ij) * 2^40), a 40-bit fixed-point weight (detexp is
 *          an exp evaluated by a fixed sequence of round-to-nearest fp32
 *          operations, so every implementation gets the same integers);
 *   the key tiles are ordered by (d ascending, j ascending) and the longest
 *   prefix whose integer running sum stays below ceil(negl_prob * 2^40) is
 *   skipped.  negl_prob = 0 skips nothing.
 * Writes every field of *lists (layouts above).
 * Errors: BL_ERR_INVALID_ARG (negl_prob outside [0, 1), null pointers),
 *         BL_ERR_UNSUPPORTED (T_c > 2048), BL_ERR_CUDA. */
bl_status bl_mask_from_stats(const bl_shape* shape, const float* tile_stats,
                             const float* lse, double negl_prob,
                             const bl_lists* lists, void* stream);

/* ---------------------------------------------------------------------------
 * Tile weights reduced in the forward.
 *
 * The statistics hold n * T_c floats per head (17 GB at n = 131072 with 32
 * heads), and the mask pass reads all of them.  The forward can instead
 * reduce them itself, right after a query tile's last key tile, into the
 * per-(query tile, key tile) log-weights the selection rule starts from
 * ("BackLite" README, How It Works, Phase 2: p_tile = exp(LSE_tile - LSE_row);
 * "Introducing BackLite", Training Nanochat, reports the stored statistics at
 * about 1% of peak memory):
 *   tile_logw : [B, H, T_r, T_c] fp32,
 *               tile_logw[b,h,i,j] = d_ij = max over rows r < n of query tile
 *               i of fp32(tile_stats[b,h,j,r] - lse[b,h,r]) (NaN if any term
 *               is NaN), clamped to <= 0 with -0 stored as +0; key tiles that
 *               no row of the tile attends (causal / window) enter with
 *               tile_stats = -inf.  This is exactly the d_ij of
 *               bl_mask_from_stats, bit for bit.
 * Tiles of 64 or 128 on either side, T_c <= 2048.
 * ------------------------------------------------------------------------- */

/* Bytes of scratch bl_attn_fwd_tile_weights needs when tile_stats is NULL:
 * one slot of 260 * T_c floats for every forward CTA that can be resident on
 * the CURRENT device at once (about 152 * 260 * T_c * 4 bytes on a GB300:
 * 40 MB at T_c = 256, 162 MB at T_c = 1024), plus one lock word per slot.
 * 0 for an invalid or unsupported shape. */
size_t bl_fwd_workspace_bytes(const bl_shape* shape);

/* bl_attn_fwd that also writes tile_logw (above).
 *   tile_stats  the statistics output as in bl_attn_fwd, or NULL: then the
 *               statistics rows live only in `workspace` (at least
 *               bl_fwd_workspace_bytes, 16-byte aligned), one slot per
 *               resident CTA, and are not returned.  Two calls in flight at
 *               the same time must not share a workspace.  workspace may be
 *               NULL when tile_stats is given.
 * O, LSE and tile_stats are the same as bl_attn_fwd's, and tile_logw does not
 * depend on whether tile_stats is given.
 * Errors: as bl_attn_fwd; BL_ERR_UNSUPPORTED (T_c > 2048);
 *         BL_ERR_WORKSPACE (tile_stats NULL and the workspace missing or
 *         too small). */
bl_status bl_attn_fwd_tile_weights(const bl_shape* shape, const void* q, const void* k,
                                   const void* v, float scale, void* o, float* lse,
                                   float* tile_stats, float* tile_logw, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* bl_mask_from_stats from the tile weights: the same lists, bit for bit, as
 * bl_mask_from_stats on the statistics and LSE the weights were reduced from,
 * reading T_r * T_c floats per head instead of n * T_c.
 * Errors: as bl_mask_from_stats. */
bl_status bl_mask_from_tile_weights(const bl_shape* shape, const float* tile_logw,
                                    double negl_prob, const bl_lists* lists, void* stream);

/* Masked attention backward ("Introducing BackLite", Backpropagation for
 * attention and Using Sparsity), with M the element mask expanded from
 * lists->mask and P recomputed from the full-row lse:
 *   D = rowsum(G_O * O), P^ = P * M, G_V = P^T G_O, G_P = G_O V^T,
 *   G_S = P^ * (G_P - D), G_Q = s G_S K, G_K = s G_S^T Q
 * (kv-head gradients sum over the query heads of their group).  Tiles not
 * in the lists are neither loaded nor computed.  lists == NULL runs the
 * dense backward (every tile).  Only q_idx/q_cnt of the lists are read.
 *   workspace  device buffer of at least bl_bwd_workspace_bytes(shape).
 * Errors: BL_ERR_INVALID_ARG, BL_ERR_UNSUPPORTED, BL_ERR_WORKSPACE,
 *         BL_ERR_CUDA.  A list entry outside [0, T_r) (or a count outside
 *         [0, T_r]) is skipped on the device and recorded in the status word;
 *         bl_bwd_check_status reports it as BL_ERR_CORRUPT_LISTS. */
bl_status bl_attn_bwd(const bl_shape* shape, const void* q, const void* k,
                      const void* v, const void* o, const void* g_o,
                      const float* lse, float scale, const bl_lists* lists,
                      void* g_q, void* g_k, void* g_v, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Synchronises the stream and reads the status word a previous bl_attn_bwd
 * left in this workspace: BL_OK, BL_ERR_CORRUPT_LISTS, or BL_ERR_TIMEOUT (a
 * bounded device-side wait gave up; the outputs of that call are invalid). */
bl_status bl_bwd_check_status(const bl_shape* shape, const void* workspace,
                              void* stream);

/* LSE-combine ("BackLite" README, Key properties: the LSE output serves to
 * combine partial attention results).  Given `parts` results of the same
 * queries over disjoint key sets,
 *   o_parts   [parts, B, n, H, d] bf16   (each part laid out like o)
 *   lse_parts [parts, B, H, n]    fp32   (each part laid out like lse)
 * writes LSE = log sum_p exp(LSE_p) and O = sum_p exp(LSE_p - LSE) O_p into
 * o [B, n, H, d] bf16 and lse [B, H, n] fp32.  A part whose LSE is -inf (it
 * saw no key) carries no weight; a row with no finite part gets O = 0 and
 * LSE = -inf.  parts in [1, 32], d in {64, 128}.
 * Errors: BL_ERR_INVALID_ARG, BL_ERR_UNSUPPORTED, BL_ERR_CUDA. */
bl_status bl_lse_combine(int parts, int B, int n, int H, int d, const void* o_parts,
                         const float* lse_parts, void* o, float* lse, void* stream);

/* Error statistics of a gradient against a reference, for choosing negl_prob
 * ("Introducing BackLite", Using Sparsity: the sparse backward is judged by
 * the cosine similarity and relative L2 error of its gradients against the
 * dense backward, and the post proposes tuning negl_prob to a target on
 * them).  a and b: n bf16 values each (device, 16-byte aligned), b the
 * reference.  out: 4 doubles of device memory (8-byte aligned), overwritten
 * with
 *   out[0] = sum (a - b)^2,  out[1] = sum b^2,  out[2] = sum a*b,  out[3] = sum a^2
 * so rel-L2 = sqrt(out[0] / out[1]) and cos = out[2] / sqrt(out[1] * out[3]).
 * Asynchronous on the stream.  Errors: BL_ERR_INVALID_ARG, BL_ERR_CUDA. */
bl_status bl_grad_error(const void* a, const void* b, size_t n, double* out, void* stream);

/* Size of the fixed device scratch array behind bl_attn_bwd_noalloc: 32 MiB
 * on every GPU that loads the library, held until the process exits. */
#define BL_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* bl_attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory themselves (for instance a host runtime that owns every byte
 * of device memory through its own pool, or a latency-critical caller that
 * cannot afford cudaMalloc's implicit synchronisation).  The BackLite pages
 * have no counterpart: this is a deployment convenience of this library.
 *
 * Same arguments, results and errors as bl_attn_bwd, except that the
 * scratch (D, the fp32 dQ accumulator, the status word) lives in a fixed
 * file-scope device array of BL_NOALLOC_SCRATCH_BYTES.  The call allocates
 * nothing.  A shape whose bl_bwd_workspace_bytes exceeds that size is
 * rejected with BL_ERR_WORKSPACE before any launch.  The first call on each
 * device looks the array's device address up (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  All calls
 * share the one array and it keeps the last call's contents (each call
 * clears what must start at zero), so calls that overlap on the GPU -- on
 * different streams, or from different threads -- race and must be
 * serialised by the caller.  List entries out of range are skipped exactly
 * as in bl_attn_bwd and recorded in a status word inside the array, which
 * bl_bwd_noalloc_check_status reads back. */
bl_status bl_attn_bwd_noalloc(const bl_shape* shape, const void* q, const void* k,
                              const void* v, const void* o, const void* g_o,
                              const float* lse, float scale, const bl_lists* lists,
                              void* g_q, void* g_k, void* g_v, void* stream);

/* bl_bwd_check_status for bl_attn_bwd_noalloc: synchronises the stream and
 * reads the status word the last bl_attn_bwd_noalloc call with this shape
 * left in the fixed scratch array of the current device: BL_OK,
 * BL_ERR_CORRUPT_LISTS, or BL_ERR_TIMEOUT (a bounded device-side wait gave
 * up; that call's outputs are invalid).  Allocates nothing.  A later call
 * with another shape moves the word, so read it before the next call. */
bl_status bl_bwd_noalloc_check_status(const bl_shape* shape, void* stream);

/* ---------------------------------------------------------------------------
 * Packed variable-length batches.
 *
 * nseq sequences of lengths n_s = cu_seqlens[s+1] - cu_seqlens[s] are packed
 * back to back along the token axis; a query attends only to keys of its own
 * sequence.  The BackLite pages train on fixed-length batches and say
 * nothing about packing; this is the plain reading of packing: the result
 * for every sequence is exactly the result of the fixed-length call with
 * B = 1, n = n_s on that sequence alone, and every per-sequence array is
 * that call's array, stored one sequence after another.
 *
 * Tensors (total = cu_seqlens[nseq])
 *   q, o, g_o, g_q : [total, H,  d] bf16, contiguous
 *   k, v, g_k, g_v : [total, Hk, d] bf16, contiguous
 *   lse            : per sequence a [H, n_s] fp32 block, at element offset
 *                    H * cu_seqlens[s]
 *   tile_stats     : per sequence a [H, T_c(s), T_r(s)*block_q] fp32 block,
 *                    blocks back to back in sequence order
 *   lists          : each field per sequence a block laid out as the
 *                    fixed-length field with B = 1, blocks back to back;
 *                    nan_count is one counter for the whole batch
 * with T_r(s) = ceil(n_s / block_q), T_c(s) = ceil(n_s / block_k).
 * bl_varlen_layout gives every size.  A sequence of length 0 owns nothing
 * and launches nothing.
 *
 * Execution: the calls walk the sequences on the host and run the
 * fixed-length kernels once per run of consecutive sequences of equal
 * length (such a run is exactly a [count, n_s, ...] batch).  The runs are
 * spread over up to `streams` side streams of the library (largest run
 * first, each to the least-loaded stream), forked from and joined back to
 * the caller's stream with events, so that short sequences fill the GPU
 * together; the call returns with all its work ordered before anything the
 * caller enqueues next on its stream.  Nothing waits on the host, so the
 * calls can be captured in a CUDA graph.  The side streams belong to the
 * library, one set per device shared by every caller: packed calls on
 * different caller streams are serialised through them, and a packed call
 * made while another thread captures a packed call on the same device would
 * be recorded into that capture, so callers serialise packed calls that may
 * overlap a capture on one device.  lse only needs 4-byte alignment here;
 * the other device pointers need 16 bytes, as in the fixed-length calls.
 * ------------------------------------------------------------------------- */

/* cu_seqlens: HOST array of nseq + 1 int32, cu_seqlens[0] = 0,
 * non-decreasing, cu_seqlens[nseq] >= 1.  streams: most runs in flight at
 * once, 1..8, or 0 for the default of 8; 1 runs them one after another on
 * the caller's stream.  The other fields mean what they mean in bl_shape and
 * obey the same limits. */
typedef struct {
  int nseq;
  const int32_t* cu_seqlens;
  int H, Hk, d;
  int block_q, block_k;
  int causal, window;
  int streams;
} bl_varlen;

/* Element counts (bytes for bwd_workspace_bytes) of a packed batch. */
typedef struct {
  size_t total;                /* packed tokens                                  */
  size_t lse;                  /* fp32: H * total                                */
  size_t tile_stats;           /* fp32: sum_s H * T_c(s) * T_r(s) * block_q      */
  size_t mask;                 /* uint8 mask and int32 kv_idx: sum_s H*T_r*T_c   */
  size_t kv_cnt;               /* int32: sum_s H * T_r(s)                        */
  size_t q_idx;                /* int32: sum_s H * T_c(s) * T_r(s)               */
  size_t q_cnt;                /* int32: sum_s H * T_c(s)                        */
  size_t bwd_workspace_bytes;  /* workspace of bl_attn_bwd_varlen                */
  int groups;                  /* launches of each kernel per call               */
} bl_varlen_sizes;

/* Validates *varlen and fills *sizes.  Errors: BL_ERR_INVALID_ARG (bad
 * cu_seqlens or shape fields), BL_ERR_UNSUPPORTED (d or tile size). */
bl_status bl_varlen_layout(const bl_varlen* varlen, bl_varlen_sizes* sizes);

/* bl_attn_fwd over a packed batch (layouts above; tile_stats may be NULL). */
bl_status bl_attn_fwd_varlen(const bl_varlen* varlen, const void* q, const void* k,
                             const void* v, float scale, void* o, float* lse,
                             float* tile_stats, void* stream);

/* bl_mask_from_stats over a packed batch: the selection of every sequence
 * uses only that sequence's statistics.  BL_ERR_UNSUPPORTED when a sequence
 * has more than 2048 key tiles. */
bl_status bl_mask_from_stats_varlen(const bl_varlen* varlen, const float* tile_stats,
                                    const float* lse, double negl_prob,
                                    const bl_lists* lists, void* stream);

/* Tile weights over a packed batch: bl_attn_fwd_tile_weights on every
 * sequence.  tile_logw holds sizes.mask floats, each sequence's
 * [H, T_r, T_c] block where its mask block is (at the same element offset).
 * At most 2048 key tiles per sequence.  Without
 * tile_stats the statistics rows live in `workspace` (at least
 * bl_fwd_workspace_bytes_varlen, 16-byte aligned), whose slots every launch
 * group of the call shares.  Two calls in flight at the same time must not
 * share a workspace.
 * Errors: as bl_attn_fwd_varlen; BL_ERR_UNSUPPORTED (more than 2048 key
 *         tiles); BL_ERR_WORKSPACE. */
size_t bl_fwd_workspace_bytes_varlen(const bl_varlen* varlen);
bl_status bl_attn_fwd_tile_weights_varlen(const bl_varlen* varlen, const void* q, const void* k,
                                          const void* v, float scale, void* o, float* lse,
                                          float* tile_stats, float* tile_logw, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* bl_mask_from_stats_varlen from the tile weights: the same lists, bit for
 * bit, as from the statistics the weights were reduced from. */
bl_status bl_mask_from_tile_weights_varlen(const bl_varlen* varlen, const float* tile_logw,
                                           double negl_prob, const bl_lists* lists,
                                           void* stream);

/* bl_attn_bwd over a packed batch.  workspace: at least
 * sizes.bwd_workspace_bytes; every run has its own D and dQ areas and status
 * word in it. */
bl_status bl_attn_bwd_varlen(const bl_varlen* varlen, const void* q, const void* k,
                             const void* v, const void* o, const void* g_o,
                             const float* lse, float scale, const bl_lists* lists,
                             void* g_q, void* g_k, void* g_v, void* workspace,
                             size_t workspace_bytes, void* stream);

/* bl_bwd_check_status for bl_attn_bwd_varlen: synchronises the stream and
 * reports the worst status word of the call's runs (BL_ERR_TIMEOUT before
 * BL_ERR_CORRUPT_LISTS before BL_OK). */
bl_status bl_varlen_bwd_check_status(const bl_varlen* varlen, const void* workspace,
                                     void* stream);

/* Every device-side wait of the tcgen05 kernels (an mbarrier phase, a peer
 * warp's hand-off) is bounded: when one runs out the kernel records it (the
 * backward's status word: BL_ERR_TIMEOUT; the forward: NaN in the LSE rows it
 * could not finish), skips the rest of its work, waits with a fixed 2 s
 * limit for the copies and MMAs it already issued, frees its tensor memory
 * and ends, so the context stays usable.  This sets the limit for kernels
 * launched from now on, process-wide: seconds in [0, 2) (0 gives up on any
 * wait that is not already satisfied), anything else restores the default of
 * 2 s.  Returns the previous limit in seconds.  A diagnostic knob for testing
 * the failure path; calls racing with launches in other threads see either
 * value. */
double bl_set_wait_limit(double seconds);

/* Static description of a status code. */
const char* bl_status_string(bl_status status);

#ifdef __cplusplus
}
#endif

#endif /* BL_ATTN_H */
