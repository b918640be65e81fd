// select.cuh -- exact top-k / top-p cut of one logit row by one block of
// kSelThreads threads (shared by the dense row pass and the tree walk).
//
// The kept set is the top-k set in the order (logit desc, index asc), then the
// shortest prefix of it whose renormalised mass reaches top_p ("LLM speculative
// decoding: EAGLE", jingming.pro, section 1 note on sampling transforms).  The
// cut key K* is the largest order key whose "at or above" tally (count for
// top-k, exact 42-bit fixed-point mass for top-p) still reaches the target; it is
// found by an 8-way split of the key range per pass over the row; ties inside K*
// are cut in index order.  `Sync` names the barrier over the block's threads.
//
// Several blocks can share one row, each covering a contiguous slice of its units
// [u_begin, u_end): `Red` then combines the blocks' tallies (integer counts and
// fixed-point masses, so the totals are exact and every block takes the same
// steps), the exclusive base of the tie count, and the tie index.  A row held by
// one block uses NoReduce.
#pragma once

#include "common.cuh"

namespace svk {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

struct SelShared {
  unsigned warp_cnt[kSelWarps];
  unsigned long long warp_mass[kSelWarps];
  unsigned red_cnt[8];
  unsigned long long red_mass[8];
  unsigned red_min;
  int tie_idx;
};

// The combination step of a row held by a single block: nothing to combine.
struct NoReduce {
  __device__ void tally(SelShared&) {}
  __device__ void base(unsigned mine, unsigned& base, unsigned& total) {
    base = 0;
    total = mine;
  }
  __device__ int max_int(int v) { return v; }
};

// Block-wide exclusive scan of (count, mass) pairs; also returns the totals.
template <class Sync>
__device__ void block_exscan(unsigned c, unsigned long long w, unsigned& base_c,
                             unsigned long long& base_w, unsigned& tot_c,
                             unsigned long long& tot_w, SelShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned ic = c;
  unsigned long long iw = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned tc = __shfl_up_sync(kFull, ic, o);
    unsigned long long tw = __shfl_up_sync(kFull, iw, o);
    if (lane >= o) { ic += tc; iw += tw; }
  }
  Sync::sync();
  if (lane == 31) { sh.warp_cnt[warp] = ic; sh.warp_mass[warp] = iw; }
  Sync::sync();
  unsigned bc = 0, tc = 0;
  unsigned long long bw = 0, tw = 0;
  for (int i = 0; i < kSelWarps; ++i) {
    if (i < warp) { bc += sh.warp_cnt[i]; bw += sh.warp_mass[i]; }
    tc += sh.warp_cnt[i];
    tw += sh.warp_mass[i];
  }
  base_c = bc + ic - c;
  base_w = bw + iw - w;
  tot_c = tc;
  tot_w = tw;
}

// ---------------------------------------------------------------------------
// Exact full-row selection (fallback, or forced by SPEC_FLAG_EXACT_SELECT).
// The cut key K* is the largest key whose "at or above" tally (count for top-k,
// fixed-point mass for top-p) still reaches the target; it is found by 4-way
// bisection, three thresholds per pass over the row, each tally accumulated in
// registers and reduced across the block.  Ties inside K* are cut in index order.
// ---------------------------------------------------------------------------
struct Eligible {
  bool active;  // restrict to the top-k set
  uint32_t key;
  int idx;
  __device__ __forceinline__ bool operator()(uint32_t k, int i) const {
    return !active || k > key || (k == key && i <= idx);
  }
};

struct SelOut {
  uint32_t key;
  int idx;
  unsigned kept;          // eligible tokens up to and including the cut
  uint64_t mass_kept;     // their fixed-point mass
};

// Tallies over eligible tokens whose shifted key s = key >> ks lies in [th[0], hi]:
// for each t, the count and fixed-point mass of those with s >= th[t]; plus the
// minimum eligible shifted key.  Weights are computed only inside the range.
// Results land in sh.red_cnt / sh.red_mass / sh.red_min.
constexpr int kSplit = 7;  // thresholds per pass: an 8-way split of the key range

template <typename T, class Sync, class Red>
__device__ void tally_range(const void* row, int V, float m, float c, int ks,
                            const uint32_t (&th)[kSplit], uint32_t hi, const Eligible& elig,
                            SelShared& sh, int u_begin, int u_end, Red& red) {
  constexpr int E = Elt<T>::kPerUnit;
  const int lane = threadIdx.x & 31;
  unsigned cnt[kSplit];
  unsigned long long mass[kSplit];
#pragma unroll
  for (int t = 0; t < kSplit; ++t) { cnt[t] = 0; mass[t] = 0; }
  unsigned kmin = 0xffffffffu;
  for (int u = u_begin + (int)threadIdx.x; u < u_end; u += kSelThreads) {
    float f[E];
    load_unit<T>(row, V, u, f);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = u * E + e;
      if (i >= V) break;
      const uint32_t k = order_key(f[e]);
      if (!elig(k, i)) continue;
      const uint32_t sk = k >> ks;
      kmin = min(kmin, sk);
      if (sk >= th[0] && sk <= hi) {
        const unsigned long long w = to_fixed(tempered_weight(f[e], m, c));
#pragma unroll
        for (int t = 0; t < kSplit; ++t)
          if (sk >= th[t]) { cnt[t] += 1; mass[t] += w; }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kSplit; ++t) {
    cnt[t] = (unsigned)warp_sum_u64(cnt[t]);
    mass[t] = warp_sum_u64(mass[t]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
  Sync::sync();
  if (threadIdx.x == 0) {
    for (int t = 0; t < kSplit; ++t) { sh.red_cnt[t] = 0; sh.red_mass[t] = 0; }
    sh.red_min = 0xffffffffu;
  }
  Sync::sync();
  if (lane == 0) {
    for (int t = 0; t < kSplit; ++t) {
      atomicAdd(&sh.red_cnt[t], cnt[t]);
      atomicAdd(&sh.red_mass[t], mass[t]);
    }
    atomicMin(&sh.red_min, kmin);
  }
  Sync::sync();
  red.tally(sh);
}

// The j-th (1-based) eligible token with order key `key`, in index order.
template <typename T, class Sync, class Red>
__device__ int tie_cut(const void* row, int V, uint32_t key, unsigned j, const Eligible& elig,
                       SelShared& sh, int u_begin, int u_end, Red& red) {
  constexpr int E = Elt<T>::kPerUnit;
  const int per = (u_end - u_begin + kSelThreads - 1) / kSelThreads;
  const int u_lo = min(u_end, u_begin + (int)threadIdx.x * per), u_hi = min(u_end, u_lo + per);
  unsigned mine = 0;
  for (int u = u_lo; u < u_hi; ++u) {
    float f[E];
    load_unit<T>(row, V, u, f);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = u * E + e;
      if (i < V) {
        const uint32_t k = order_key(f[e]);
        mine += (k == key && elig(k, i));
      }
    }
  }
  unsigned base, tot;
  unsigned long long bw, tw;
  block_exscan<Sync>(mine, 0ull, base, bw, tot, tw, sh);
  unsigned cbase, ctot;
  red.base(tot, cbase, ctot);  // tokens of the blocks before this one
  base += cbase;
  if (threadIdx.x == 0) sh.tie_idx = -1;
  Sync::sync();
  if (base < j && base + mine >= j) {
    unsigned want = j - base;
    for (int u = u_lo; u < u_hi && want; ++u) {
      float f[E];
      load_unit<T>(row, V, u, f);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = u * E + e;
        if (i < V && want) {
          const uint32_t k = order_key(f[e]);
          if (k == key && elig(k, i) && --want == 0) sh.tie_idx = i;
        }
      }
    }
  }
  Sync::sync();
  return red.max_int(sh.tie_idx);
}

template <typename T, class Sync, class Red>
__device__ SelOut exact_select(const void* row, int V, float m, float c, bool by_mass,
                               unsigned need_count, uint64_t need_mass, Eligible elig,
                               SelShared& sh, int u_begin, int u_end, Red& red) {
  const int ks = (sizeof(T) == 2) ? 16 : 0;  // bf16 keys carry 16 constant low bits
  const uint32_t kmax = order_key(m) >> ks;
  auto reaches = [&](unsigned cnt, unsigned long long mass) {
    return by_mass ? (mass >= need_mass) : (cnt >= need_count);
  };
  // first pass: eligible totals and the smallest eligible key
  uint32_t th[kSplit];
  for (int t = 0; t < kSplit; ++t) th[t] = 0u;
  tally_range<T, Sync, Red>(row, V, m, c, ks, th, 0xffffffffu, elig, sh, u_begin, u_end, red);
  uint64_t lo = sh.red_min, hi = kmax;
  // tokens with a key above hi: their count and mass, carried from pass to pass
  unsigned above_c = 0;
  unsigned long long above_m = 0;
  const unsigned total_c = sh.red_cnt[0];
  const unsigned long long total_m = sh.red_mass[0];
  const bool short_all = !reaches(total_c, total_m);
  if (short_all) hi = lo;  // eligible mass short of the target (rounding): keep them all
  while (lo < hi) {
    const uint64_t span = hi - lo;
    for (int t = 0; t < kSplit; ++t)
      th[t] = (uint32_t)(lo + (span * (uint64_t)(t + 1) + kSplit) / (kSplit + 1));
    tally_range<T, Sync, Red>(row, V, m, c, ks, th, (uint32_t)hi, elig, sh, u_begin, u_end, red);
    int pick = -1;
    for (int t = kSplit - 1; t >= 0; --t)
      if (reaches(above_c + sh.red_cnt[t], above_m + sh.red_mass[t])) { pick = t; break; }
    if (pick < 0) {
      hi = (uint64_t)th[0] - 1;
      above_c += sh.red_cnt[0];
      above_m += sh.red_mass[0];
    } else {
      lo = th[pick];
      if (pick < kSplit - 1) {
        hi = (uint64_t)th[pick + 1] - 1;
        above_c += sh.red_cnt[pick + 1];
        above_m += sh.red_mass[pick + 1];
      }
    }
  }
  // the tokens carrying the cut key
  const uint32_t kstar = (uint32_t)lo;
  for (int t = 0; t < kSplit; ++t) th[t] = kstar;
  tally_range<T, Sync, Red>(row, V, m, c, ks, th, kstar, elig, sh, u_begin, u_end, red);
  const unsigned cnt_eq = sh.red_cnt[0];
  const unsigned long long w_eq = cnt_eq ? sh.red_mass[0] / cnt_eq : 0ull;
  unsigned j;
  if (short_all) {
    // every eligible token is kept; the cut is the last one, in the lowest key
    above_c = total_c - cnt_eq;
    above_m = total_m - sh.red_mass[0];
    j = cnt_eq;
  } else if (!by_mass) {
    j = need_count - above_c;
  } else if (w_eq == 0) {
    j = cnt_eq;
  } else {
    const unsigned long long jj = (need_mass - above_m + w_eq - 1) / w_eq;
    j = (unsigned)(jj < 1 ? 1 : (jj > cnt_eq ? cnt_eq : jj));
  }
  const uint32_t key = ks ? key_from16(kstar) : kstar;
  SelOut r;
  r.key = key;
  r.idx = tie_cut<T, Sync, Red>(row, V, key, j, elig, sh, u_begin, u_end, red);
  r.kept = above_c + j;
  r.mass_kept = above_m + w_eq * j;
  return r;
}

}  // namespace svk
