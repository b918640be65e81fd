// rows.cu -- the dense row pass: per logit row, the maximum and its lowest index,
// the tempered normaliser, and the top-k / top-p cut ("LLM speculative decoding:
// EAGLE", section 1 note: p and q are compared after temperature, top-k, top-p or
// argmax processing).
//
// One block of kRowThreads threads owns one row at a time (persistent grid-stride
// over rows).  A single streaming pass over the row computes
//   * each warp's running maximum and the sum of 2^((z - M_warp) c), rescaled
//     whenever the warp maximum grows (online softmax), Kahan-summed;
//   * the argmax (lowest index of the maximum);
//   * when top-k / top-p is active, a candidate window: every token within
//     kWindowNats nats of the block's running maximum is appended to shared memory.
// The cut is then found inside the window.  bf16 windows are resolved with an
// exact histogram over their (few hundred) distinct keys -- equal logits carry
// equal weights, so a bin's mass is its count times one weight; fp32 windows are
// sorted.  Masses are 42-bit fixed point, so every sum is exact and independent
// of order.  When the window overflows or provably misses the cut, the row falls
// back to an exact full-row selection by 4-way bisection on the order key; both
// routes produce bit-identical statistics.
#include <climits>

#include "common.cuh"

namespace svk {

namespace {

constexpr int NT = kRowThreads;
constexpr int NW = NT / 32;
constexpr int kUnroll = 4;
constexpr int kBinsPerThread = kHistBins / NT;
constexpr size_t kDynSmem = (size_t)kCandCap * 8 + (size_t)kSortCap * 8;

struct RowShared {
  float warp_m[NW];
  double warp_s[NW];
  float warp_best[NW];
  int warp_best_idx[NW];
  int warp_bad[NW];
  unsigned warp_cnt[NW];
  unsigned long long warp_mass[NW];
  unsigned run_key;
  unsigned n_cand;
  unsigned n_keep;
  int first;
  int ok;
  unsigned tie_n;
  int tie_idx;
  unsigned sel_j;
  unsigned red_cnt[4];
  unsigned long long red_mass[4];
  unsigned red_min;
  unsigned long long tau;
  // results broadcast by thread 0
  float m;
  double s_total;
  int argmax;
  int bad;
};

__device__ __forceinline__ const void* row_ptr(const void* base, int64_t elems, int bytes) {
  return static_cast<const void*>(static_cast<const char*>(base) + elems * bytes);
}

// Block-wide exclusive scan of (count, mass) pairs; also returns the totals.
__device__ void block_exscan(unsigned c, unsigned long long w, unsigned& base_c,
                             unsigned long long& base_w, unsigned& tot_c,
                             unsigned long long& tot_w, RowShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned ic = c;
  unsigned long long iw = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned tc = __shfl_up_sync(kFull, ic, o);
    unsigned long long tw = __shfl_up_sync(kFull, iw, o);
    if (lane >= o) { ic += tc; iw += tw; }
  }
  __syncthreads();
  if (lane == 31) { sh.warp_cnt[warp] = ic; sh.warp_mass[warp] = iw; }
  __syncthreads();
  unsigned bc = 0, tc = 0;
  unsigned long long bw = 0, tw = 0;
  for (int i = 0; i < NW; ++i) {
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

// Tallies of eligible tokens with (key >> ks) >= th[t], t < 3, plus the minimum
// eligible shifted key.  Results land in sh.red_cnt / sh.red_mass / sh.red_min.
template <typename T>
__device__ void tally3(const void* row, int V, float m, float c, int ks, const uint32_t (&th)[3],
                       const Eligible& elig, RowShared& sh) {
  constexpr int E = Elt<T>::kPerUnit;
  const int nunits = (V + E - 1) / E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned cnt[3] = {0, 0, 0};
  unsigned long long mass[3] = {0, 0, 0};
  unsigned kmin = 0xffffffffu;
  for (int u = threadIdx.x; u < nunits; u += NT) {
    float f[E];
    load_unit<T>(row, V, u, f);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = u * E + e;
      if (i >= V) break;
      const uint32_t k = order_key(f[e]);
      if (!elig(k, i)) continue;
      const uint32_t s = k >> ks;
      kmin = min(kmin, s);
      if (s >= th[0]) {
        const unsigned long long w = to_fixed(tempered_weight(f[e], m, c));
#pragma unroll
        for (int t = 0; t < 3; ++t)
          if (s >= th[t]) { cnt[t] += 1; mass[t] += w; }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    cnt[t] = (unsigned)warp_sum_u64(cnt[t]);
    mass[t] = warp_sum_u64(mass[t]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int t = 0; t < 3; ++t) { sh.red_cnt[t] = 0; sh.red_mass[t] = 0; }
    sh.red_min = 0xffffffffu;
  }
  __syncthreads();
  if (lane == 0) {
    for (int t = 0; t < 3; ++t) {
      atomicAdd(&sh.red_cnt[t], cnt[t]);
      atomicAdd(&sh.red_mass[t], mass[t]);
    }
    atomicMin(&sh.red_min, kmin);
  }
  __syncthreads();
}

// The j-th (1-based) eligible token with order key `key`, in index order.
template <typename T>
__device__ int tie_cut(const void* row, int V, uint32_t key, unsigned j, const Eligible& elig,
                       RowShared& sh) {
  constexpr int E = Elt<T>::kPerUnit;
  const int nunits = (V + E - 1) / E;
  const int per = (nunits + NT - 1) / NT;
  const int u_lo = threadIdx.x * per, u_hi = min(nunits, u_lo + per);
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
  block_exscan(mine, 0ull, base, bw, tot, tw, sh);
  if (threadIdx.x == 0) sh.tie_idx = -1;
  __syncthreads();
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
  __syncthreads();
  return sh.tie_idx;
}

template <typename T>
__device__ SelOut exact_select(const void* row, int V, float m, float c, bool by_mass,
                               unsigned need_count, uint64_t need_mass, Eligible elig,
                               RowShared& sh) {
  const int ks = (sizeof(T) == 2) ? 16 : 0;  // bf16 keys carry 16 zero low bits
  const uint32_t kmax = order_key(m) >> ks;
  auto reaches = [&](unsigned cnt, unsigned long long mass) {
    return by_mass ? (mass >= need_mass) : (cnt >= need_count);
  };
  // first pass: the eligible totals and the smallest eligible key
  uint32_t th0[3] = {0u, 0u, 0u};
  tally3<T>(row, V, m, c, ks, th0, elig, sh);
  uint64_t lo = sh.red_min, hi = kmax;
  bool short_all = !reaches(sh.red_cnt[0], sh.red_mass[0]);
  if (short_all) {
    hi = lo;  // eligible mass short of the target (rounding): keep every eligible token
  }
  while (lo < hi) {
    // three thresholds split (lo, hi] into four parts; keep the highest reaching part
    uint64_t span = hi - lo;
    uint32_t th[3];
    for (int t = 0; t < 3; ++t) th[t] = (uint32_t)(lo + (span * (uint64_t)(t + 1) + 3) / 4);
    tally3<T>(row, V, m, c, ks, th, elig, sh);
    uint64_t nlo = lo, nhi = hi;
    for (int t = 2; t >= 0; --t) {
      if (reaches(sh.red_cnt[t], sh.red_mass[t])) { nlo = th[t]; break; }
      nhi = (uint64_t)th[t] - 1;
    }
    lo = nlo;
    hi = nhi;
  }
  const uint32_t ks_key = (uint32_t)lo;
  // tallies at and above the cut key
  uint32_t th1[3] = {ks_key, ks_key + 1u, ks_key + 1u};
  tally3<T>(row, V, m, c, ks, th1, elig, sh);
  const unsigned cnt_ge = sh.red_cnt[0], cnt_gt = sh.red_cnt[1];
  const unsigned long long mass_ge = sh.red_mass[0], mass_gt = sh.red_mass[1];
  const unsigned cnt_eq = cnt_ge - cnt_gt;
  const unsigned long long w_eq = cnt_eq ? (mass_ge - mass_gt) / cnt_eq : 0ull;
  unsigned j;
  if (short_all) {
    j = cnt_eq;
  } else if (!by_mass) {
    j = need_count - cnt_gt;
  } else if (w_eq == 0) {
    j = cnt_eq;
  } else {
    unsigned long long jj = (need_mass - mass_gt + w_eq - 1) / w_eq;
    j = (unsigned)(jj < 1 ? 1 : (jj > cnt_eq ? cnt_eq : jj));
  }
  const uint32_t key = ks ? key_from16(ks_key) : ks_key;
  SelOut r;
  r.key = key;
  r.idx = tie_cut<T>(row, V, key, j, elig, sh);
  r.kept = cnt_gt + j;
  r.mass_kept = mass_gt + w_eq * j;
  return r;
}

// ---------------------------------------------------------------------------
// The row pass kernel.  MODE 0: greedy (max + argmax only).  MODE 1: sampling
// without truncation.  MODE 2: sampling with top-k and/or top-p.
// ---------------------------------------------------------------------------
template <typename T, int MODE>
__global__ void __launch_bounds__(NT, kRowBlocksPerSm) row_pass_kernel(RowJob job) {
  constexpr int E = Elt<T>::kPerUnit;
  __shared__ RowShared sh;
  extern __shared__ __align__(16) unsigned char dyn[];
  uint2* cand = reinterpret_cast<uint2*>(dyn);  // (index, logit bits)
  unsigned long long* pre = reinterpret_cast<unsigned long long*>(dyn);  // reuses cand
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(dyn + (size_t)kCandCap * 8);
  unsigned* hist = reinterpret_cast<unsigned*>(dyn + (size_t)kCandCap * 8);  // aliases keys
  unsigned* ties = hist + kHistBins;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int V = job.V;
  const int nunits = (V + E - 1) / E;
  const int full_units = V / E;
  const float c = job.c;
  const int BN = job.B * job.N;
  const int total = (job.mode == kRowsList) ? job.R : (job.with_q ? 2 * BN : BN);
  const bool topk_on = job.top_k > 0 && job.top_k < V;
  const bool topp_on = job.top_p < 1.0f;

  for (int v = blockIdx.x; v < total; v += gridDim.x) {
    const void* row;
    spec_row_stats* out;
    if (job.mode == kRowsList) {
      row = row_ptr(job.base_p, (int64_t)v * job.row_pitch, Elt<T>::kBytes);
      out = job.stats_p + v;
    } else {
      const bool is_q = v >= BN;
      const int r = is_q ? v - BN : v;
      if (is_q && !job.need_q[r]) continue;
      const int b = r / job.N, n = r - b * job.N;
      const int64_t off = (int64_t)b * job.batch_stride + (int64_t)n * job.row_pitch;
      row = row_ptr(is_q ? job.base_q : job.base_p, off, Elt<T>::kBytes);
      out = (is_q ? job.stats_q : job.stats_p) + r;
    }
    if (threadIdx.x == 0) {
      sh.n_cand = 0;
      sh.run_key = 0u;
    }
    __syncthreads();

    // ---------------- streaming pass ----------------
    float Mw = -CUDART_INF_F;
    Kahan S;
    float best = -CUDART_INF_F;
    int best_idx = INT_MAX;
    int bad = 0;
    const uint4* row4 = reinterpret_cast<const uint4*>(row);
    for (int u0 = 0; u0 < nunits; u0 += NT * kUnroll) {
      float f[kUnroll][E];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int u = u0 + k * NT + threadIdx.x;
        if (u < full_units) {
          uint4 raw = __ldg(row4 + u);
          Elt<T>::unpack(raw, f[k]);
        } else if (u < nunits) {
          load_unit<T>(row, V, u, f[k]);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) f[k][e] = -CUDART_INF_F;
        }
      }
      float tmax = -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < kUnroll; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) tmax = fmaxf(tmax, f[k][e]);
      if (tmax > best) {
        int idx = INT_MAX;
#pragma unroll
        for (int k = kUnroll - 1; k >= 0; --k)
#pragma unroll
          for (int e = E - 1; e >= 0; --e)
            if (f[k][e] == tmax) idx = (u0 + k * NT + threadIdx.x) * E + e;
        best = tmax;
        best_idx = idx;
      }
      if (MODE == 0) {
#pragma unroll
        for (int k = 0; k < kUnroll; ++k)
#pragma unroll
          for (int e = 0; e < E; ++e) bad |= (f[k][e] != f[k][e]);
        continue;
      }
      const float wm = warp_max(tmax);
      if (MODE == 2) {
        // publish the warp maximum; the first iteration waits for every warp so that
        // the window starts from a block-wide maximum
        if (lane == 0 && wm > -CUDART_INF_F) atomicMax(&sh.run_key, order_key(wm));
        if (u0 == 0) __syncthreads();
      }
      if (wm > Mw) {
        if (Mw != -CUDART_INF_F) {
          const float scale = ex2_approx((Mw - wm) * c);
          S.s *= scale;
          S.c *= scale;
        }
        Mw = wm;
      }
      if (Mw == -CUDART_INF_F) {  // nothing finite yet: only NaN can hide here
#pragma unroll
        for (int k = 0; k < kUnroll; ++k)
#pragma unroll
          for (int e = 0; e < E; ++e) bad |= (f[k][e] != f[k][e]);
        continue;
      }
      const float negMc = -Mw * c;
      float part = 0.f;
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        float pk = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) pk += ex2_approx(fmaf(f[k][e], c, negMc));
        part += pk;
      }
      S.add(part);
      if (MODE == 2) {
        const unsigned rk = *((volatile unsigned*)&sh.run_key);
        const float bmax = rk ? fmaxf(Mw, key_value(rk)) : Mw;
        const float thr = bmax - job.delta_z;
        int mine = 0;
#pragma unroll
        for (int k = 0; k < kUnroll; ++k)
#pragma unroll
          for (int e = 0; e < E; ++e) mine += (f[k][e] >= thr);
        if (__any_sync(kFull, mine > 0)) {
          int incl = mine;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
          }
          unsigned base = 0;
          if (lane == 31) base = atomicAdd(&sh.n_cand, (unsigned)incl);
          base = __shfl_sync(kFull, base, 31);
          unsigned pos = base + incl - mine;
#pragma unroll
          for (int k = 0; k < kUnroll; ++k)
#pragma unroll
            for (int e = 0; e < E; ++e)
              if (f[k][e] >= thr) {
                if (pos < (unsigned)kCandCap)
                  cand[pos] = make_uint2((unsigned)((u0 + k * NT + threadIdx.x) * E + e),
                                         __float_as_uint(f[k][e]));
                ++pos;
              }
        }
      }
    }

    // ---------------- block combine ----------------
    {
      const double ws = warp_sum_d(S.value());
      const float wb = warp_max(best);
      const int wi = warp_min_i(best == wb ? best_idx : INT_MAX);
      const int wbad = __any_sync(kFull, bad);
      if (lane == 0) {
        sh.warp_m[warp] = Mw;
        sh.warp_s[warp] = ws;
        sh.warp_best[warp] = wb;
        sh.warp_best_idx[warp] = wi;
        sh.warp_bad[warp] = wbad;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = -CUDART_INF_F;
      int am = INT_MAX, anybad = 0;
      for (int w = 0; w < NW; ++w) {
        const float b = sh.warp_best[w];
        if (b > m) { m = b; am = sh.warp_best_idx[w]; }
        else if (b == m) am = min(am, sh.warp_best_idx[w]);
        anybad |= sh.warp_bad[w];
      }
      double s = 0.0;
      if (MODE != 0) {
        for (int w = 0; w < NW; ++w)
          if (sh.warp_m[w] != -CUDART_INF_F)
            s += sh.warp_s[w] * exp2(((double)sh.warp_m[w] - (double)m) * (double)c);
      }
      const bool finite = !anybad && m != CUDART_INF_F && m != -CUDART_INF_F && !(m != m) &&
                          (MODE == 0 || (s == s && s != CUDART_INF));
      sh.m = m;
      sh.s_total = s;
      sh.argmax = (am == INT_MAX) ? 0 : am;
      sh.bad = !finite;
      if (job.counters) {
        atomicAdd(&job.counters[0], 1ull);
        atomicAdd(&job.counters[1], (unsigned long long)V * Elt<T>::kBytes);
      }
    }
    __syncthreads();
    const float m = sh.m;
    const int argmax = sh.argmax;

    if (sh.bad) {
      if (threadIdx.x == 0) {
        spec_row_stats st;
        st.m = m; st.status = SPEC_ROW_NONFINITE; st.s_f = 0.0; st.cut_key = 0;
        st.cut_idx = -1; st.argmax = argmax; st.kept = 0;
        *out = st;
      }
      __syncthreads();
      continue;
    }
    if (MODE == 0 || MODE == 1) {
      if (threadIdx.x == 0) {
        spec_row_stats st;
        st.m = m;
        st.status = SPEC_TREE_OK;
        st.argmax = argmax;
        if (MODE == 0) {
          st.s_f = 1.0; st.cut_key = order_key(m); st.cut_idx = argmax; st.kept = 1;
        } else {
          st.s_f = sh.s_total; st.cut_key = 0u; st.cut_idx = V - 1; st.kept = V;
        }
        *out = st;
      }
      __syncthreads();
      continue;
    }

    // ---------------- MODE 2: the cut ----------------
    const double s_total = sh.s_total;
    const unsigned K = topk_on ? (unsigned)job.top_k : (unsigned)V;
    const double tau_scale = 4398046511104.0;  // 2^42
    bool done = false;
    uint32_t cut_key = 0;
    int cut_idx = 0;
    unsigned kept = 0;
    uint64_t sf_fixed = 0;
    const unsigned n_buf = sh.n_cand;
    const float thr = m - job.delta_z;
    const uint32_t K16m = order_key(m) >> 16;
    const uint32_t K16thr = order_key(thr) >> 16;
    const bool use_hist = (sizeof(T) == 2) && (K16m - K16thr < (uint32_t)kHistBins);
    if (!(job.flags & SPEC_FLAG_EXACT_SELECT) && n_buf <= (unsigned)kCandCap && use_hist) {
      // ---- bf16 window: one bin per key below the maximum ----
      const int nb = (int)(K16m - K16thr) + 1;
      for (int i = threadIdx.x; i < nb; i += NT) hist[i] = 0u;
      if (threadIdx.x == 0) { sh.first = INT_MAX; sh.ok = 1; sh.tie_n = 0; sh.tie_idx = -1; }
      __syncthreads();
      for (unsigned i = threadIdx.x; i < n_buf; i += NT) {
        const float z = __uint_as_float(cand[i].y);
        if (z >= thr) atomicAdd(&hist[K16m - (order_key(z) >> 16)], 1u);
      }
      __syncthreads();
      // per-thread chunk of bins; bin b holds the key b steps below the maximum, and
      // its weight is the weight of that key
      const int b_lo = threadIdx.x * kBinsPerThread;
      auto bin_w = [&](int bin) -> unsigned long long {
        return to_fixed(tempered_weight(key_value(key_from16(K16m - (uint32_t)bin)), m, c));
      };
      unsigned lc = 0;
      unsigned long long lw = 0;
      for (int t = 0; t < kBinsPerThread; ++t) {
        const int bin = b_lo + t;
        if (bin < nb && hist[bin]) { lc += hist[bin]; lw += (unsigned long long)hist[bin] * bin_w(bin); }
      }
      unsigned base_c, tot_c;
      unsigned long long base_w, tot_w;
      block_exscan(lc, lw, base_c, base_w, tot_c, tot_w, sh);
      // top-k: the bin holding the K-th token
      int b_k = nb;  // "no top-k": past the last bin
      unsigned jk = 0;
      unsigned long long s_k_fixed = 0;
      if (topk_on) {
        if (tot_c < K) {
          if (threadIdx.x == 0) sh.ok = 0;
        } else {
          unsigned rc = base_c;
          for (int t = 0; t < kBinsPerThread; ++t) {
            const int bin = b_lo + t;
            if (bin >= nb) break;
            if (rc + hist[bin] >= K) { atomicMin(&sh.first, bin); break; }
            rc += hist[bin];
          }
        }
        __syncthreads();
        if (sh.ok) {
          b_k = sh.first;
          // counts / masses before b_k, owned by the thread whose chunk holds b_k
          if (b_k >= b_lo && b_k < b_lo + kBinsPerThread) {
            unsigned rc = base_c;
            unsigned long long rw = base_w;
            for (int bin = b_lo; bin < b_k; ++bin) { rc += hist[bin]; rw += (unsigned long long)hist[bin] * bin_w(bin); }
            const unsigned j = K - rc;
            sh.sel_j = j;
            sh.tau = rw + (unsigned long long)j * bin_w(b_k);  // mass of the top-k set
            sh.n_keep = rc;
            sh.warp_mass[0] = rw;
          }
          __syncthreads();
          jk = sh.sel_j;
          s_k_fixed = sh.tau;
          if (!topp_on) {
            cut_key = key_from16(K16m - (uint32_t)b_k);
            kept = sh.n_keep + jk;
            sf_fixed = s_k_fixed;
          }
        }
      }
      __syncthreads();
      int b_cut = b_k;
      unsigned j_cut = jk;
      if (sh.ok && topp_on) {
        const unsigned long long tau = (unsigned long long)ceil(
            (double)job.top_p * (topk_on ? (double)s_k_fixed : s_total * tau_scale));
        if (threadIdx.x == 0) sh.first = INT_MAX;
        __syncthreads();
        // masses up to b_k (bin b_k only counts its first jk tokens)
        unsigned long long rw = base_w;
        for (int t = 0; t < kBinsPerThread; ++t) {
          const int bin = b_lo + t;
          if (bin >= nb || bin > b_k) break;
          const unsigned cnt = (bin == b_k) ? jk : hist[bin];
          const unsigned long long w = (unsigned long long)cnt * bin_w(bin);
          if (cnt && rw + w >= tau) { atomicMin(&sh.first, bin); break; }
          rw += w;
        }
        __syncthreads();
        if (sh.first == INT_MAX) {
          if (threadIdx.x == 0) sh.ok = 0;  // the window holds too little mass
        } else {
          const int b_p = sh.first;
          if (b_p >= b_lo && b_p < b_lo + kBinsPerThread) {
            unsigned rc = base_c;
            unsigned long long rw2 = base_w;
            for (int bin = b_lo; bin < b_p; ++bin) { rc += hist[bin]; rw2 += (unsigned long long)hist[bin] * bin_w(bin); }
            const unsigned avail = (b_p == b_k) ? jk : hist[b_p];
            const unsigned long long w1 = bin_w(b_p);
            unsigned j = avail;
            if (w1 > 0) {
              const unsigned long long jj = (tau - rw2 + w1 - 1) / w1;
              j = (unsigned)(jj < 1 ? 1 : (jj > avail ? avail : jj));
            }
            sh.sel_j = j;
            sh.n_keep = rc;
            sh.warp_mass[0] = rw2 + (unsigned long long)j * w1;
          }
          __syncthreads();
          b_cut = b_p;
          j_cut = sh.sel_j;
          cut_key = key_from16(K16m - (uint32_t)b_p);
          kept = sh.n_keep + j_cut;
          sf_fixed = sh.warp_mass[0];
        }
        __syncthreads();
      }
      if (sh.ok) {
        // the j_cut-th token of the cut key in index order: rank its members
        if (hist[b_cut] > (unsigned)kTieCap) {
          if (threadIdx.x == 0) sh.ok = 0;
        } else {
          for (unsigned i = threadIdx.x; i < n_buf; i += NT) {
            const uint2 e = cand[i];
            if (order_key(__uint_as_float(e.y)) == cut_key) ties[atomicAdd(&sh.tie_n, 1u)] = e.x;
          }
          __syncthreads();
          const unsigned nt = sh.tie_n;
          for (unsigned i = threadIdx.x; i < nt; i += NT) {
            const unsigned me = ties[i];
            unsigned rank = 0;
            for (unsigned t = 0; t < nt; ++t) rank += (ties[t] < me);
            if (rank + 1 == j_cut) sh.tie_idx = (int)me;
          }
        }
        __syncthreads();
        cut_idx = sh.tie_idx;
      }
      __syncthreads();
      done = sh.ok;
      __syncthreads();
    } else if (!(job.flags & SPEC_FLAG_EXACT_SELECT) && n_buf <= (unsigned)kCandCap) {
      // ---- sorted window (fp32 logits, or a bf16 window spanning many keys) ----
      if (threadIdx.x == 0) sh.n_keep = 0;
      __syncthreads();
      for (unsigned i = threadIdx.x; i < n_buf; i += NT) {
        const uint2 e = cand[i];
        const float z = __uint_as_float(e.y);
        if (z >= thr) {
          const unsigned pos = atomicAdd(&sh.n_keep, 1u);
          if (pos < (unsigned)kSortCap)
            keys[pos] = ((unsigned long long)order_key(z) << 32) | (unsigned long long)(~e.x);
        }
      }
      __syncthreads();
      const unsigned n_c = sh.n_keep;
      if (n_c >= 1 && n_c <= (unsigned)kSortCap && (!topk_on || n_c >= K)) {
        unsigned n_pad = 2;
        while (n_pad < n_c) n_pad <<= 1;
        for (unsigned i = n_c + threadIdx.x; i < n_pad; i += NT) keys[i] = 0ull;
        __syncthreads();
        for (unsigned k = 2; k <= n_pad; k <<= 1) {  // bitonic sort, descending
          for (unsigned jj = k >> 1; jj > 0; jj >>= 1) {
            for (unsigned i = threadIdx.x; i < n_pad; i += NT) {
              const unsigned ixj = i ^ jj;
              if (ixj > i) {
                const unsigned long long a = keys[i], b = keys[ixj];
                const bool swap = ((i & k) == 0) ? (a < b) : (a > b);
                if (swap) { keys[i] = b; keys[ixj] = a; }
              }
            }
            __syncthreads();
          }
        }
        // inclusive prefix of fixed-point masses over the sorted window
        constexpr int C = kSortCap / NT;
        const unsigned lo = threadIdx.x * C;
        unsigned long long run = 0;
#pragma unroll
        for (int t = 0; t < C; ++t) {
          const unsigned i = lo + t;
          if (i < n_c) run += to_fixed(tempered_weight(key_value((uint32_t)(keys[i] >> 32)), m, c));
          pre[i] = run;
        }
        unsigned bc, tc;
        unsigned long long bw, tw;
        block_exscan(0u, run, bc, bw, tc, tw, sh);
#pragma unroll
        for (int t = 0; t < C; ++t) pre[lo + t] += bw;
        if (threadIdx.x == 0) sh.first = INT_MAX;
        __syncthreads();
        const unsigned K_eff = topk_on ? K : n_c;
        bool ok = true;
        unsigned cut_pos = K_eff - 1;
        if (topp_on) {
          const unsigned long long tau = (unsigned long long)ceil(
              (double)job.top_p * (topk_on ? (double)pre[K - 1] : s_total * tau_scale));
          int fj = INT_MAX;
          for (int t = 0; t < C; ++t) {
            const unsigned i = lo + t;
            if (i < K_eff && pre[i] >= tau) { fj = (int)i; break; }
          }
          fj = warp_min_i(fj);
          if (lane == 0 && fj != INT_MAX) atomicMin(&sh.first, fj);
          __syncthreads();
          if (sh.first == INT_MAX) ok = false;  // the window holds too little mass
          else cut_pos = (unsigned)sh.first;
        }
        if (ok) {
          const unsigned long long kk = keys[cut_pos];
          cut_key = (uint32_t)(kk >> 32);
          cut_idx = (int)(~(uint32_t)kk);
          kept = cut_pos + 1;
          sf_fixed = pre[cut_pos];
          done = true;
        }
      }
      __syncthreads();
    }
    if (!done) {
      // exact full-row selection
      SelOut rk{};
      const Eligible all{false, 0u, 0};
      if (topk_on) rk = exact_select<T>(row, V, m, c, false, K, 0ull, all, sh);
      if (topp_on) {
        const Eligible in_k{topk_on, rk.key, rk.idx};
        const unsigned long long tau = (unsigned long long)ceil(
            (double)job.top_p * (topk_on ? (double)rk.mass_kept : s_total * tau_scale));
        const SelOut rp = exact_select<T>(row, V, m, c, true, 0u, tau, in_k, sh);
        cut_key = rp.key; cut_idx = rp.idx; kept = rp.kept; sf_fixed = rp.mass_kept;
      } else {
        cut_key = rk.key; cut_idx = rk.idx; kept = rk.kept; sf_fixed = rk.mass_kept;
      }
      if (threadIdx.x == 0 && job.counters) atomicAdd(&job.counters[5], 1ull);
    }
    if (threadIdx.x == 0) {
      spec_row_stats st;
      st.m = m;
      st.status = SPEC_TREE_OK;
      st.s_f = fixed_to_double(sf_fixed);
      st.cut_key = cut_key;
      st.cut_idx = cut_idx;
      st.argmax = argmax;
      st.kept = (int)kept;
      *out = st;
    }
    __syncthreads();
  }
}

template <typename T, int MODE>
cudaError_t launch_mode(const RowJob& job, int num_rows, cudaStream_t s) {
  const size_t dyn = (MODE == 2) ? kDynSmem : 0;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(row_pass_kernel<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dyn);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  int grid = device_sm_count() * kRowBlocksPerSm;
  if (grid > num_rows) grid = num_rows;
  if (grid < 1) grid = 1;
  row_pass_kernel<T, MODE><<<grid, NT, dyn, s>>>(job);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_row_pass(const RowJob& job, spec_dtype dtype, int num_rows, cudaStream_t s) {
  const bool greedy = job.temperature == 0.0f;
  const bool filt = !greedy && ((job.top_k > 0 && job.top_k < job.V) || job.top_p < 1.0f);
  const int mode = greedy ? 0 : (filt ? 2 : 1);
  if (dtype == SPEC_BF16) {
    if (mode == 0) return launch_mode<uint16_t, 0>(job, num_rows, s);
    if (mode == 1) return launch_mode<uint16_t, 1>(job, num_rows, s);
    return launch_mode<uint16_t, 2>(job, num_rows, s);
  }
  if (mode == 0) return launch_mode<float, 0>(job, num_rows, s);
  if (mode == 1) return launch_mode<float, 1>(job, num_rows, s);
  return launch_mode<float, 2>(job, num_rows, s);
}

}  // namespace svk
