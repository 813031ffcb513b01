// mask_from_stats: tile statistics -> block-sparse mask and tile lists.
//
// "BackLite" README, How It Works, Phase 2: per tile pair the weight is
// p_tile = exp(LSE_tile - LSE_row), and the smallest-weight tiles whose
// cumulative weight stays below negl_prob are skipped.  Key properties:
// "cumulative weight < negl_prob" (strict) and negl_prob = 0 keeps every
// tile.  "Introducing BackLite", Using Sparsity: a skipped tile costs no
// loads and no FLOPs in the backward.
//
// The rule as implemented (the pages leave the reduction, tie-break and
// arithmetic open):
//   d_ij = max over rows r < n of query tile i of fp32(stats[j][r] - lse[r]),
//          NaN if any term is NaN, then clamped to <= 0 with -0 -> +0;
//   E_ij = ceil(detexp(d_ij) * 2^40) as a 64-bit integer;
//   per query tile, order the non-NaN key tiles by (d asc, j asc) and skip
//   the longest prefix whose integer running sum is < ceil(negl_prob*2^40).
// detexp is a fixed sequence of round-to-nearest fp32 operations (no FMA):
//   t = d*log2(e); t < -48 -> E = 1; k = rint(t); f = t - k;
//   p = Horner over the degree-7 Taylor polynomial of 2^f = exp(f ln 2);
//   e = p * 2^k.  Integer sums make the result independent of the order in
//   which a parallel scan adds them.
//
// Kernel 1: one CTA per (query tile, head, batch).  Warps stream the
// statistics of the tile's rows (coalesced 256/512-byte rows per key tile,
// four key tiles in flight per warp) and reduce d_ij; then the CTA sorts
// (key, E) pairs with a bitonic network, scans E, and writes the mask row
// plus the compacted kv list.  With several CTAs per SM, one CTA's loads
// overlap another's sort.  The shared arrays are sized by a capacity CAP (the
// smallest power of two >= T_c, at least 256); at CAP = 256 each thread holds
// one element and the network's stages closer than a warp run on shuffles.
// From the tile weights the forward reduced (bl_mask_from_tile_weights) the
// d_ij come ready-made and mask_rows_warp_kernel (below) takes one warp per
// query tile instead.
// Kernel 2: one warp per (key tile, head, batch) compacts the mask column
// into the ascending q list with ballots.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace bl {

namespace {

constexpr int kMaskThreads = 256;
constexpr int kMaxTc = 2048;

// fp32 nearest to log2(e) and to (ln 2)^m / m!, m = 0..7 (Taylor series of 2^f).
__device__ __forceinline__ uint64_t detexp_fixed40(float d) {
  if (isinf(d)) return 0ull;  // d == -inf: the tile has no weight
  const float log2e = __uint_as_float(0x3fb8aa3bu);
  const float c0 = __uint_as_float(0x3f800000u), c1 = __uint_as_float(0x3f317218u),
              c2 = __uint_as_float(0x3e75fdf0u), c3 = __uint_as_float(0x3d635847u),
              c4 = __uint_as_float(0x3c1d955bu), c5 = __uint_as_float(0x3aaec3ffu),
              c6 = __uint_as_float(0x39218489u), c7 = __uint_as_float(0x377fe5feu);
  float t = __fmul_rn(d, log2e);
  if (t < -48.f) return 1ull;
  float kf = rintf(t);
  float f = __fsub_rn(t, kf);
  float p = c7;
  p = __fadd_rn(__fmul_rn(p, f), c6);
  p = __fadd_rn(__fmul_rn(p, f), c5);
  p = __fadd_rn(__fmul_rn(p, f), c4);
  p = __fadd_rn(__fmul_rn(p, f), c3);
  p = __fadd_rn(__fmul_rn(p, f), c2);
  p = __fadd_rn(__fmul_rn(p, f), c1);
  p = __fadd_rn(__fmul_rn(p, f), c0);
  int ki = (int)kf;                                   // -48 <= ki <= 0
  float e = __fmul_rn(p, __uint_as_float((uint32_t)(ki + 127) << 23));
  float s = __fmul_rn(e, 1099511627776.0f);           // * 2^40, exact
  return (uint64_t)__float2ull_rn(ceilf(s));
}

// max that propagates NaN: one operation carries both the maximum and the
// "some term is NaN" flag of the reduction
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ uint32_t order_key(float d) {
  uint32_t u = __float_as_uint(d);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int RPL, int CAP>  // rows per lane: block_q / 32; capacity >= T_c
__global__ void __launch_bounds__(kMaskThreads) mask_rows_kernel(
    const float* __restrict__ stats, const float* __restrict__ lse, Shape sh,
    unsigned long long T, uint8_t* __restrict__ mask,
    int32_t* __restrict__ kv_idx, int32_t* __restrict__ kv_cnt,
    int32_t* __restrict__ nan_count) {
  __shared__ float s_d[CAP];
  __shared__ unsigned long long s_key[CAP];
  __shared__ unsigned long long s_E[CAP];
  __shared__ unsigned long long s_wsum[kMaskThreads / 32];
  __shared__ int s_wcnt[kMaskThreads / 32];
  __shared__ uint8_t s_act[CAP];

  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Tc = sh.T_c;
  const int64_t bh = (int64_t)b * sh.H + h;
  int k_lo, k_hi;
  key_tile_range(sh, i, k_lo, k_hi);
  {
    const int r0 = i * sh.block_q + lane * RPL;
    float lrow[RPL];
    bool valid[RPL];
#pragma unroll
    for (int e = 0; e < RPL; ++e) {
      valid[e] = (r0 + e) < sh.n;
      lrow[e] = valid[e] ? lse[bh * sh.n + r0 + e] : 0.f;
    }
    const float* st = stats + bh * sh.T_c * sh.n_pad + r0;
    constexpr int NW = kMaskThreads / 32;
    constexpr int UNR = 4;   // key tiles in flight per warp
    for (int j0 = warp; j0 < Tc; j0 += NW * UNR) {
      float vals[UNR][RPL];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int j = j0 + u * NW;
        if (j >= Tc || j < k_lo || j > k_hi) {
#pragma unroll
          for (int e = 0; e < RPL; ++e) vals[u][e] = -INFINITY;
          continue;
        }
        if constexpr (RPL == 4) {
          const float4 x = *reinterpret_cast<const float4*>(st + (int64_t)j * sh.n_pad);
          vals[u][0] = x.x; vals[u][1] = x.y; vals[u][2] = x.z; vals[u][3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(st + (int64_t)j * sh.n_pad);
          vals[u][0] = x.x; vals[u][1] = x.y;
        }
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int j = j0 + u * NW;
        if (j >= Tc) continue;   // warp-uniform
        // max over the tile's rows of fl32(stat - lse), NaN if any term is
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < RPL; ++e)
          if (valid[e]) mx = max_nan(mx, __fsub_rn(vals[u][e], lrow[e]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          mx = max_nan(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) {
          float dv = isnan(mx) ? __uint_as_float(0x7fc00000u) : fminf(mx, 0.f);
          if (dv == 0.f) dv = 0.f;  // -0 -> +0
          s_d[j] = dv;
        }
      }
    }
  }
  __syncthreads();

  int P2 = 1;
  while (P2 < Tc) P2 <<= 1;
  if (CAP == kMaskThreads) P2 = CAP;   // the register network sorts all CAP entries
  int local_nan = 0;
  for (int m = tid; m < P2; m += kMaskThreads) {
    unsigned long long key = ~0ull;
    if (m < Tc) {
      float dv = s_d[m];
      if (isnan(dv)) {
        key = (0xffffffffull << 32) | (unsigned)m;
        ++local_nan;
      } else {
        key = ((unsigned long long)order_key(dv) << 32) | (unsigned)m;
      }
      s_act[m] = 1;
    }
    s_key[m] = key;
  }
  if (nan_count) {
    local_nan = __reduce_add_sync(0xffffffffu, local_nan);
    if (lane == 0 && local_nan) atomicAdd(nan_count, local_nan);
  }
  __syncthreads();

  // bitonic sort of the keys ascending (unique but for the padding, which is
  // equal and last); E follows from d once the order is known
  if constexpr (CAP == kMaskThreads) {
    // one element per thread: partners closer than a warp swap through
    // shuffles, the six stages with stride >= 32 through shared memory
    unsigned long long key = s_key[tid];
    for (int kk = 2; kk <= CAP; kk <<= 1) {
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        unsigned long long pk;
        if (jj >= 32) {
          __syncthreads();
          s_key[tid] = key;
          __syncthreads();
          pk = s_key[tid ^ jj];
        } else {
          pk = __shfl_xor_sync(0xffffffffu, key, jj);
        }
        // the lower element of an ascending pair keeps the smaller key
        const bool up = (tid & kk) == 0, lower = (tid & jj) == 0;
        if ((lower == up) ? (pk < key) : (pk > key)) key = pk;
      }
    }
    __syncthreads();
    s_key[tid] = key;
  } else {
    for (int kk = 2; kk <= P2; kk <<= 1) {
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        for (int tt = tid; tt < (P2 >> 1); tt += kMaskThreads) {
          const int a = 2 * tt - (tt & (jj - 1));   // pair (a, a + jj), jj a power of two
          const int c = a + jj;
          const bool up = (a & kk) == 0;
          const unsigned long long ka = s_key[a], kc = s_key[c];
          if ((ka > kc) == up) {
            s_key[a] = kc;
            s_key[c] = ka;
          }
        }
        __syncthreads();
      }
    }
  }
  // E in sorted order (0 for NaN and padding keys, which sort last)
  for (int m = tid; m < P2; m += kMaskThreads) {
    const unsigned long long key = s_key[m];
    s_E[m] = (key >> 32) != 0xffffffffull ? detexp_fixed40(s_d[(int)(key & 0xffffffffull)]) : 0ull;
  }
  __syncthreads();

  // inclusive scan of E in sorted order; count positions with prefix < T
  // among the non-NaN entries (NaN and padding keys sort last).
  constexpr int PER = CAP / kMaskThreads;  // <= 8 elements per thread
  int per = (P2 + kMaskThreads - 1) / kMaskThreads;
  int base = tid * per;
  unsigned long long run = 0ull;
  for (int e = 0; e < per && e < PER; ++e) {
    int m = base + e;
    if (m < P2) run += s_E[m];
  }
  // exclusive scan of per-thread totals
  unsigned long long incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  unsigned long long woff = 0ull;
  for (int w = 0; w < warp; ++w) woff += s_wsum[w];
  unsigned long long pre = woff + incl - run;
  int nskip = 0;
  for (int e = 0; e < per && e < PER; ++e) {
    int m = base + e;
    if (m >= P2) break;
    unsigned long long key = s_key[m];
    pre += s_E[m];
    if ((key >> 32) != 0xffffffffull && pre < T) ++nskip;
  }
  __syncthreads();
  // the skipped entries form a prefix of the sorted order: mark them
  for (int e = 0; e < per && e < PER; ++e) {
    int m = base + e;
    if (m < P2 && e < nskip) s_act[(int)(s_key[m] & 0xffffffffull)] = 0;
  }
  __syncthreads();

  // write the mask row and the ascending kv list
  uint8_t* mrow = mask + (bh * sh.T_r + i) * (int64_t)Tc;
  int32_t* krow = kv_idx + (bh * sh.T_r + i) * (int64_t)Tc;
  int cnt_run = 0;
  for (int j0 = 0; j0 < Tc; j0 += kMaskThreads) {
    int j = j0 + tid;
    int f = (j < Tc && j >= k_lo && j <= k_hi) ? s_act[j] : 0;
    if (j < Tc) mrow[j] = (uint8_t)f;
    unsigned bal = __ballot_sync(0xffffffffu, f);
    int wpos = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) s_wcnt[warp] = __popc(bal);
    __syncthreads();
    int off = cnt_run;
    for (int w = 0; w < warp; ++w) off += s_wcnt[w];
    if (f) krow[off + wpos] = j;
    int tot = 0;
    for (int w = 0; w < kMaskThreads / 32; ++w) tot += s_wcnt[w];
    __syncthreads();
    cnt_run += tot;
  }
  for (int j = cnt_run + tid; j < Tc; j += kMaskThreads) krow[j] = -1;
  if (tid == 0) kv_cnt[bh * sh.T_r + i] = cnt_run;
}

// The same rule from the tile weights, one warp per query tile: lane l holds
// entries PER l .. PER l + PER - 1 of the row (entry = key tile j; PER =
// 8, 16, 32 or 64 for T_c up to 256, 512, 1024, 2048).  Only the 32-bit
// order keys of d are sorted (bitonic network: strides below PER swap within
// a lane, the others through shuffles), which fixes the position nskip where
// the skipped prefix ends and the key K* of its last entry.  Ties in d carry
// equal E, so the prefix sums, hence nskip, do not depend on how the network
// orders them; the skipped entries in (d asc, j asc) order are then every j
// with key < K* and, of the j with key == K*, the lowest r = nskip -
// #(key < K*), ranked by j with a warp scan.  No shared memory, no block
// barrier.
__device__ __forceinline__ float key_to_d(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// k[idx] for a register array through a select tree (a loop of conditional
// moves would let the compiler move the array to local memory)
template <int LO, int HI>
__device__ __forceinline__ uint32_t pick(const uint32_t* k, int idx) {
  if constexpr (HI - LO == 1) {
    return k[LO];
  } else {
    constexpr int MID = (LO + HI) / 2;
    return idx < MID ? pick<LO, MID>(k, idx) : pick<MID, HI>(k, idx);
  }
}

// rows (warps) per block: eight for the small rows; two where a warp holds
// many registers, so that more of them fit on an SM
template <int PER>
constexpr int kWarpRows = PER <= 8 ? 8 : 2;
// rows that keep more tiles than this are sorted
constexpr int kMaxTop = 32;

template <int PER>
__global__ void __launch_bounds__(32 * kWarpRows<PER>) mask_rows_warp_kernel(
    const float* __restrict__ logw, Shape sh, unsigned long long T, uint8_t* __restrict__ mask,
    int32_t* __restrict__ kv_idx, int32_t* __restrict__ kv_cnt,
    int32_t* __restrict__ nan_count) {
  constexpr int N = 32 * PER;               // sorted entries (padding past T_c)
  constexpr uint32_t kLast = 0xffffffffu;   // NaN weights and padding: sorted last, E = 0
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpRows<PER> + warp;
  if (row >= (int64_t)sh.B * sh.H * sh.T_r) return;
  const int i = (int)(row % sh.T_r);
  const int Tc = sh.T_c;
  int k_lo, k_hi;
  key_tile_range(sh, i, k_lo, k_hi);
  const float* wrow = logw + row * (int64_t)Tc;
  // the unsorted key of entry e: kept in registers up to PER = 16, re-read
  // (from L1) above, so that more warps fit on an SM
  constexpr bool kKeep = PER <= 16;
  uint32_t orig[kKeep ? PER : 1], key[PER];
  auto load_key = [&](int e) -> uint32_t {
    const int m = lane * PER + e;
    if (m >= Tc) return kLast;
    const float dv = wrow[m];
    return isnan(dv) ? kLast : order_key(dv);
  };
  auto unsorted = [&](int e) -> uint32_t {
    if constexpr (kKeep) return orig[e];
    else return load_key(e);
  };
  int local_nan = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int m = lane * PER + e;
    key[e] = load_key(e);
    if (m < Tc && key[e] == kLast) ++local_nan;
    if constexpr (kKeep) orig[e] = key[e];
  }
  if (nan_count) {
    local_nan = __reduce_add_sync(0xffffffffu, local_nan);
    if (lane == 0 && local_nan) atomicAdd(nan_count, local_nan);
  }
  uint64_t fbits = 0ull;   // bit e: entry PER lane + e is kept (mask row)
  // Few kept tiles, the usual case: the kept entries are the top K in (d
  // desc, j desc) order, K the least count whose removal leaves a sum of E
  // below T -- the complement of the longest prefix in (d asc, j asc) order
  // whose sum stays below T.  They are taken one at a time with a warp-wide
  // max of (key, j); a row that keeps more than kMaxTop is sorted instead.
  // At 8 entries per lane the sort is cheaper than the extraction and always
  // runs.
  bool sort_row = true;
  if constexpr (PER > 8) {
    unsigned long long S = 0ull;
    int nn = 0;
#pragma unroll
    for (int e = 0; e < PER; ++e)
      if (key[e] != kLast) {
        S += detexp_fixed40(key_to_d(key[e]));
        ++nn;
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    nn = __reduce_add_sync(0xffffffffu, nn);
    uint64_t kept = 0ull;
    auto lane_best = [&]() {   // 0: none (every valid (key, j) is above 0)
      unsigned long long bst = 0ull;
#pragma unroll
      for (int e = 0; e < PER; ++e)
        if (!((kept >> e) & 1ull) && key[e] != kLast)
          bst = max(bst, ((unsigned long long)key[e] << 32) | (unsigned)(lane * PER + e));
      return bst;
    };
    unsigned long long best = lane_best(), taken = 0ull;
    for (int k = 0;; ++k) {
      if (k >= nn || S - taken < T) {
        sort_row = false;
        break;
      }
      if (k >= kMaxTop) break;
      unsigned long long w = best;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) w = max(w, __shfl_xor_sync(0xffffffffu, w, o));
      const int j = (int)(w & 0xffffffffull), owner = j / PER;
      unsigned long long ew = 0ull;
      if (lane == owner) {
        kept |= 1ull << (j - lane * PER);
        ew = detexp_fixed40(key_to_d((uint32_t)(w >> 32)));
        best = lane_best();
      }
      taken += __shfl_sync(0xffffffffu, ew, owner);
    }
    if (!sort_row) {
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const int m = lane * PER + e;
        // NaN weights are never skipped
        if (m < Tc && (key[e] == kLast || ((kept >> e) & 1ull)) && m >= k_lo && m <= k_hi)
          fbits |= 1ull << e;
      }
    }
  }
  if (sort_row) {
  #pragma unroll
    for (int kk = 2; kk <= N; kk <<= 1) {
  #pragma unroll
      for (int jj = kk >> 1; jj > 0; jj >>= 1) {
        if (jj < PER) {
  #pragma unroll
          for (int e = 0; e < PER; ++e) {
            if (e & jj) continue;
            const bool up = ((lane * PER + e) & kk) == 0;
            const uint32_t lo = min(key[e], key[e | jj]), hi = max(key[e], key[e | jj]);
            key[e] = up ? lo : hi;
            key[e | jj] = up ? hi : lo;
          }
        } else {
          const int lj = jj / PER;
          const bool lower = (lane & lj) == 0;
  #pragma unroll
          for (int e = 0; e < PER; ++e) {
            const uint32_t pk = __shfl_xor_sync(0xffffffffu, key[e], lj);
            const bool up = ((lane * PER + e) & kk) == 0;
            // the lower element of an ascending pair keeps the smaller key
            key[e] = (lower == up) ? min(key[e], pk) : max(key[e], pk);
          }
        }
      }
    }
    // inclusive prefix of E in sorted order: nskip = the non-NaN positions whose
    // prefix stays below T (a prefix of the order)
    unsigned long long tot = 0ull;
  #pragma unroll
    for (int e = 0; e < PER; ++e)
      tot += key[e] != kLast ? detexp_fixed40(key_to_d(key[e])) : 0ull;
    unsigned long long incl = tot;
  #pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    unsigned long long pre = incl - tot;
    int nskip = 0;
  #pragma unroll
    for (int e = 0; e < PER; ++e) {
      pre += key[e] != kLast ? detexp_fixed40(key_to_d(key[e])) : 0ull;
      nskip += (key[e] != kLast && pre < T);
    }
    nskip = __reduce_add_sync(0xffffffffu, nskip);
    // K*: the sorted key at position nskip - 1; r of its ties are skipped
    uint32_t kstar = 0u;
    int r = 0;
    if (nskip > 0) {
      const int p = nskip - 1;
      kstar = __shfl_sync(0xffffffffu, pick<0, PER>(key, p % PER), p / PER);
      int less = 0;
  #pragma unroll
      for (int e = 0; e < PER; ++e) less += unsorted(e) < kstar;
      r = nskip - __reduce_add_sync(0xffffffffu, less);
    }
    // rank of each tie (key == K*) by j: warp exclusive scan of the per-lane counts
    int ties = 0;
  #pragma unroll
    for (int e = 0; e < PER; ++e) ties += (nskip > 0 && unsorted(e) == kstar);
    int tie_off = ties;
  #pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, tie_off, o);
      if (lane >= o) tie_off += y;
    }
    tie_off -= ties;
    // the mask row
  #pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int m = lane * PER + e;
      bool skip = false;
      if (nskip > 0) {
        const uint32_t ke = unsorted(e);
        if (ke < kstar) {
          skip = true;
        } else if (ke == kstar) {
          skip = tie_off < r;
          ++tie_off;
        }
      }
      if (m < Tc && !skip && m >= k_lo && m <= k_hi) fbits |= 1ull << e;
    }
  }
  const int mine = __popcll(fbits);
  uint8_t* mrow = mask + row * (int64_t)Tc;
  int32_t* krow = kv_idx + row * (int64_t)Tc;
  int off = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, off, o);
    if (lane >= o) off += y;
  }
  const int cnt = __shfl_sync(0xffffffffu, off, 31);
  off -= mine;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int m = lane * PER + e;
    const uint32_t fe = (uint32_t)(fbits >> e) & 1u;
    if (m < Tc) mrow[m] = (uint8_t)fe;
    if (fe) krow[off++] = m;
  }
  for (int j = cnt + lane; j < Tc; j += 32) krow[j] = -1;
  if (lane == 0) kv_cnt[row] = cnt;
}

__global__ void __launch_bounds__(256) q_lists_kernel(const uint8_t* __restrict__ mask, Shape sh,
                                                      int32_t* __restrict__ q_idx,
                                                      int32_t* __restrict__ q_cnt) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * 8 + warp;
  const int h = blockIdx.y, b = blockIdx.z;
  if (j >= sh.T_c) return;
  const int64_t bh = (int64_t)b * sh.H + h;
  const uint8_t* mcol = mask + bh * sh.T_r * (int64_t)sh.T_c + j;
  int32_t* qrow = q_idx + (bh * sh.T_c + j) * (int64_t)sh.T_r;
  int cnt = 0;
  for (int i0 = 0; i0 < sh.T_r; i0 += 32) {
    int i = i0 + lane;
    int f = (i < sh.T_r) ? mcol[(int64_t)i * sh.T_c] : 0;
    unsigned bal = __ballot_sync(0xffffffffu, f);
    if (f) qrow[cnt + __popc(bal & ((1u << lane) - 1u))] = i;
    cnt += __popc(bal);
  }
  for (int i = cnt + lane; i < sh.T_r; i += 32) qrow[i] = -1;
  if (lane == 0) q_cnt[bh * sh.T_c + j] = cnt;
}

}  // namespace

cudaError_t launch_mask(const Shape& sh, const float* stats, const float* lse,
                        const float* logw, unsigned long long threshold, uint8_t* mask,
                        int32_t* kv_idx, int32_t* kv_cnt, int32_t* q_idx, int32_t* q_cnt,
                        int32_t* nan_count, cudaStream_t st) {
  if (sh.T_c > kMaxTc) return cudaErrorInvalidValue;
  dim3 g1(sh.T_r, sh.H, sh.B);
  if (!stats) {   // from the tile weights: one warp per query tile
    auto warp_rows = [&](auto per) {
      constexpr int R = kWarpRows<decltype(per)::value>;
      const unsigned blocks = (unsigned)(((int64_t)sh.B * sh.H * sh.T_r + R - 1) / R);
      mask_rows_warp_kernel<decltype(per)::value><<<blocks, 32 * R, 0, st>>>(
          logw, sh, threshold, mask, kv_idx, kv_cnt, nan_count);
    };
    if (sh.T_c <= 256) warp_rows(std::integral_constant<int, 8>{});
    else if (sh.T_c <= 512) warp_rows(std::integral_constant<int, 16>{});
    else if (sh.T_c <= 1024) warp_rows(std::integral_constant<int, 32>{});
    else warp_rows(std::integral_constant<int, 64>{});
  } else {
    auto rows = [&](auto rpl, auto cap) {
      mask_rows_kernel<decltype(rpl)::value, decltype(cap)::value>
          <<<g1, kMaskThreads, 0, st>>>(stats, lse, sh, threshold, mask, kv_idx, kv_cnt,
                                        nan_count);
    };
    auto by_cap = [&](auto rpl) {
      if (sh.T_c <= 256) rows(rpl, std::integral_constant<int, 256>{});
      else if (sh.T_c <= 512) rows(rpl, std::integral_constant<int, 512>{});
      else if (sh.T_c <= 1024) rows(rpl, std::integral_constant<int, 1024>{});
      else rows(rpl, std::integral_constant<int, 2048>{});
    };
    if (sh.block_q == 128)
      by_cap(std::integral_constant<int, 4>{});
    else
      by_cap(std::integral_constant<int, 2>{});
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 g2((sh.T_c + 7) / 8, sh.H, sh.B);
  q_lists_kernel<<<g2, 256, 0, st>>>(mask, sh, q_idx, q_cnt);
  return cudaGetLastError();
}

}  // namespace bl
