// walk.cu -- tree preparation and the per-tree accept walk.
//
// Multi-round speculative sampling on a tree (EAGLE / EAGLE-2 translation,
// modelers.csdn.net, sections 1.3.2 and 1.7; "LLM speculative decoding: EAGLE",
// jingming.pro, section 2.3 steps 3-5): at the current node u the children are
// tried in increasing node index against the draft row q_u; a child with token x
// is accepted with probability min(1, p(x)/q(x)); after a rejection p becomes
// norm(max(0, p - q)) and the next sibling is tried; when every child is
// rejected, or u is a leaf, the final token is drawn from the current p by
// inverse CDF.  At temperature 0 the first child whose token is the target
// argmax is accepted and the final token is the argmax ("EAGLE close reading",
// edgeai1.github.io, sections 3 and 5).
#include <climits>

#include "common.cuh"

namespace svk {

namespace {

constexpr int WT = kWalkThreads;
constexpr int WW = WT / 32;

__device__ __forceinline__ const void* row_at(const void* base, const TreeJob& j, int b, int n,
                                              int bytes) {
  int64_t off = (int64_t)b * j.batch_stride + (int64_t)n * j.row_pitch;
  return static_cast<const void*>(static_cast<const char*>(base) + off * bytes);
}

// ---------------------------------------------------------------------------
// Tree preparation: one thread per tree validates parent_idx / draft_tokens,
// builds the children lists in node order (CSR) and flags the q rows the walk
// may need (nodes with at least one child).
// ---------------------------------------------------------------------------
__global__ void tree_prep_kernel(TreeJob job, int greedy) {
  if (blockIdx.x == 0 && threadIdx.x < 8 && job.counters) job.counters[threadIdx.x] = 0ull;
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= job.B) return;
  const int N = job.N;
  const int32_t* par = job.parents + (int64_t)b * N;
  const int32_t* tok = job.tokens + (int64_t)b * N;
  int32_t* cs = job.child_start + (int64_t)b * (N + 1);
  int32_t* cl = job.child_list + (int64_t)b * N;
  uint8_t* nq = job.need_q + (int64_t)b * N;
  if (job.out_alpha)
    for (int n = 0; n < N; ++n) job.out_alpha[(int64_t)b * N + n] = __int_as_float(0x7fc00000);
  for (int n = 0; n < N; ++n) nq[n] = 0;

  int status = SPEC_TREE_OK;
  if (par[0] != -1) status = SPEC_TREE_INVALID;
  // depth of each node, kept in the child list until the lists are built
  cl[0] = 0;
  for (int n = 1; n < N && status == SPEC_TREE_OK; ++n) {
    int p = par[n], t = tok[n];
    if (p < 0 || p >= n || t < 0 || t >= job.V) { status = SPEC_TREE_INVALID; break; }
    int d = cl[p] + 1;
    if (d > job.W - 1) { status = SPEC_TREE_INVALID; break; }
    cl[n] = d;
  }
  job.tree_info[b] = status;
  if (status != SPEC_TREE_OK) return;
  for (int u = 0; u <= N; ++u) cs[u] = 0;
  for (int n = 1; n < N; ++n) cs[par[n] + 1] += 1;
  for (int u = 1; u <= N; ++u) cs[u] += cs[u - 1];  // cs[u] = first slot of u's children
  for (int n = 1; n < N; ++n) cl[cs[par[n]]++] = n; // children land in node order
  for (int u = N; u >= 1; --u) cs[u] = cs[u - 1];
  cs[0] = 0;
  if (!greedy)
    for (int u = 0; u < N; ++u) nq[u] = (cs[u + 1] > cs[u]);
}

// ---------------------------------------------------------------------------
// Walk helpers.
// ---------------------------------------------------------------------------
struct WalkShared {
  double red[WW];
  double wtot[WW];
  double target;
  int target_warp;
  int accept;
  int final_tok;
};

// Is token x (logit z) inside the kept set of a filtered row?
__device__ __forceinline__ bool kept_tok(float z, int x, const spec_row_stats& st) {
  uint32_t k = order_key(z);
  return k > st.cut_key || (k == st.cut_key && x <= st.cut_idx);
}

// Filtered probability of one token in fp64 (for the acceptance test).
template <typename T>
__device__ double prob64(const void* row, int x, const spec_row_stats& st, double T_) {
  float z = Elt<T>::at(row, x);
  if (!kept_tok(z, x, st)) return 0.0;
  return exp(((double)z - (double)st.m) / T_) / st.s_f;
}

// Filtered probability in fp32 for the elementwise passes.
__device__ __forceinline__ float prob32(float z, int x, const spec_row_stats& st, float c,
                                        float inv_s) {
  return kept_tok(z, x, st) ? tempered_weight(z, st.m, c) * inv_s : 0.f;
}

// p after j renormalised residual steps: p <- max(0, p - q) / Z_r (unchanged when Z_r == 0).
__device__ __forceinline__ float residual_chain(float p, float q, int j, const float* invz) {
  for (int r = 0; r < j; ++r) {
    float iz = invz[r];
    if (iz > 0.f) p = fmaxf(0.f, p - q) * iz;
  }
  return p;
}

__device__ double block_sum_d(double v, WalkShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_d(v);
  __syncthreads();
  if (lane == 0) sh.red[warp] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < WW; ++w) t += sh.red[w];
  return t;
}

// Values of the current distribution over one unit of E tokens.
template <typename T>
__device__ __forceinline__ void unit_values(const void* prow, const void* qrow, int V, int u,
                                            const spec_row_stats& sp, const spec_row_stats& sq,
                                            float c, float inv_sp, float inv_sq, int j,
                                            const float* invz,
                                            float (&val)[Elt<T>::kPerUnit]) {
  constexpr int E = Elt<T>::kPerUnit;
  float zp[E];
  load_unit<T>(prow, V, u, zp);
  if (j == 0) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      int x = u * E + e;
      val[e] = (x < V) ? prob32(zp[e], x, sp, c, inv_sp) : 0.f;
    }
    return;
  }
  float zq[E];
  load_unit<T>(qrow, V, u, zq);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    int x = u * E + e;
    if (x < V) {
      float p = prob32(zp[e], x, sp, c, inv_sp);
      float q = prob32(zq[e], x, sq, c, inv_sq);
      val[e] = residual_chain(p, q, j, invz);
    } else {
      val[e] = 0.f;
    }
  }
}

// Z = sum_x max(0, p^(j)(x) - q(x)) over the row pair (block-wide, fp64 result).
// Each thread issues the loads of kWalkUnroll units of both rows before using them.
constexpr int kWalkUnroll = 2;

template <typename T>
__device__ double residual_mass(const void* prow, const void* qrow, int V,
                                const spec_row_stats& sp, const spec_row_stats& sq, float c,
                                float inv_sp, float inv_sq, int j, const float* invz,
                                WalkShared& sh) {
  constexpr int E = Elt<T>::kPerUnit;
  const int nunits = (V + E - 1) / E;
  Kahan acc;
  for (int u0 = threadIdx.x; u0 < nunits; u0 += WT * kWalkUnroll) {
    float zp[kWalkUnroll][E], zq[kWalkUnroll][E];
#pragma unroll
    for (int k = 0; k < kWalkUnroll; ++k) {
      const int u = u0 + k * WT;
      if (u < nunits) {
        load_unit<T>(prow, V, u, zp[k]);
        load_unit<T>(qrow, V, u, zq[k]);
      }
    }
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < kWalkUnroll; ++k) {
      const int u = u0 + k * WT;
      if (u >= nunits) break;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int x = u * E + e;
        if (x < V) {
          float p = prob32(zp[k][e], x, sp, c, inv_sp);
          const float q = prob32(zq[k][e], x, sq, c, inv_sq);
          p = residual_chain(p, q, j, invz);
          part += fmaxf(0.f, p - q);
        }
      }
    }
    acc.add(part);
  }
  return block_sum_d(acc.value(), sh);
}

// Inverse-CDF draw in index order: the smallest x with C_x >= r * C_V, where C is the
// inclusive prefix sum of the current distribution.  Warps own contiguous ranges of
// units; a warp step covers 32 consecutive units (one per lane) and its total is a
// butterfly sum.  The owning warp retraces its step totals in the same order in the
// second phase, so its running sum reproduces the first phase exactly.
template <typename T>
__device__ __forceinline__ float unit_sum(const void* prow, const void* qrow, int V, int u,
                                          const spec_row_stats& sp, const spec_row_stats& sq,
                                          float c, float inv_sp, float inv_sq, int j,
                                          const float* invz, float (&val)[Elt<T>::kPerUnit]) {
  unit_values<T>(prow, qrow, V, u, sp, sq, c, inv_sp, inv_sq, j, invz, val);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < Elt<T>::kPerUnit; ++e) s += val[e];
  return s;
}

template <typename T>
__device__ int inverse_cdf(const void* prow, const void* qrow, int V, const spec_row_stats& sp,
                           const spec_row_stats& sq, float c, float inv_sp, float inv_sq, int j,
                           const float* invz, double r, WalkShared& sh) {
  constexpr int E = Elt<T>::kPerUnit;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nunits = (V + E - 1) / E;
  const int per_warp = (nunits + WW - 1) / WW;
  const int u_lo = warp * per_warp, u_hi = min(nunits, u_lo + per_warp);
  double wt = 0.0;
  for (int ub = u_lo; ub < u_hi; ub += 64) {
    float val0[E], val1[E];
    const int ua = ub + lane, ubb = ub + 32 + lane;
    const float s0 = (ua < u_hi) ? unit_sum<T>(prow, qrow, V, ua, sp, sq, c, inv_sp, inv_sq, j, invz, val0) : 0.f;
    const float s1 = (ubb < u_hi) ? unit_sum<T>(prow, qrow, V, ubb, sp, sq, c, inv_sp, inv_sq, j, invz, val1) : 0.f;
    wt += warp_sum_d((double)s0);
    wt += warp_sum_d((double)s1);
  }
  if (lane == 0) sh.wtot[warp] = wt;
  __syncthreads();
  if (threadIdx.x == 0) {
    double total = 0.0;
    for (int w = 0; w < WW; ++w) total += sh.wtot[w];
    double t = r * total, cum = 0.0;
    int tw = -1, last = -1;
    double tw_base = 0.0, last_base = 0.0;
    for (int w = 0; w < WW; ++w) {
      if (sh.wtot[w] > 0.0) {
        last = w;
        last_base = cum;
        if (tw < 0 && cum + sh.wtot[w] >= t) { tw = w; tw_base = cum; }
      }
      cum += sh.wtot[w];
    }
    if (tw < 0) { tw = last; tw_base = last_base; t = last_base + sh.wtot[last]; }
    sh.target_warp = tw;
    sh.target = fmin(t - tw_base, sh.wtot[tw]);
    sh.final_tok = -1;
  }
  __syncthreads();
  if (warp == sh.target_warp) {
    const double target = sh.target;
    double cum = 0.0;
    bool found = false;
    for (int ub = u_lo; ub < u_hi && !found; ub += 32) {
      // same unit order and butterfly totals as the first phase (two 32-unit steps per 64)
      const int u = ub + lane;
      float val[E];
      const float s = (u < u_hi) ? unit_sum<T>(prow, qrow, V, u, sp, sq, c, inv_sp, inv_sq, j, invz, val) : 0.f;
      const double it = warp_sum_d((double)s);
      if (it > 0.0 && cum + it >= target) {
        double incl = (double)s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double t = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t;
        }
        const double before = cum + incl - (double)s;
        const unsigned hit = __ballot_sync(kFull, s > 0.f && cum + incl >= target);
        const unsigned pos = __ballot_sync(kFull, s > 0.f);
        const int L = hit ? (__ffs(hit) - 1) : (31 - __clz(pos));
        int tok = -1;
        if (lane == L) {
          double acc = before;
          int lastpos = -1;
#pragma unroll
          for (int e = 0; e < E; ++e) {
            if (val[e] > 0.f) {
              lastpos = u * E + e;
              acc += (double)val[e];
              if (acc >= target) { tok = u * E + e; break; }
            }
          }
          if (tok < 0) tok = lastpos;
        }
        tok = __shfl_sync(kFull, tok, L);
        if (lane == 0) sh.final_tok = tok;
        found = true;
      }
      cum += it;
    }
  }
  __syncthreads();
  return sh.final_tok;
}

// ---------------------------------------------------------------------------
// The walk: one block per tree.
// ---------------------------------------------------------------------------
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(WT) tree_walk_kernel(TreeJob job) {
  __shared__ WalkShared sh;
  const int b = blockIdx.x;
  const int N = job.N, V = job.V, W = job.W;
  int32_t* out_tok = job.out_tokens + (int64_t)b * W;
  int32_t* out_path = job.out_path + (int64_t)b * W;
  int status = job.tree_info[b];
  double* Z = job.resid_z + (int64_t)b * N;
  float* invz = job.resid_invz + (int64_t)b * N;
  const int32_t* cs = job.child_start + (int64_t)b * (N + 1);
  const int32_t* cl = job.child_list + (int64_t)b * N;
  const int32_t* tok = job.tokens + (int64_t)b * N;
  const double Td = (double)job.temperature;
  const float c = job.c;

  int u = 0, n_acc = 0, final_tok = -1;
  while (status == SPEC_TREE_OK) {
    const spec_row_stats sp = job.stats_p[(int64_t)b * N + u];
    if (sp.status != SPEC_TREE_OK) { status = SPEC_ROW_NONFINITE; break; }
    const int c0 = cs[u], c1 = cs[u + 1];
    if (GREEDY) {
      int next = -1;
      for (int i = c0; i < c1; ++i) {
        int ch = cl[i];
        bool ok = tok[ch] == sp.argmax;
        if (threadIdx.x == 0 && job.out_alpha) job.out_alpha[(int64_t)b * N + ch] = ok ? 1.f : 0.f;
        if (ok) { next = ch; break; }
      }
      if (next >= 0) {
        if (threadIdx.x == 0) {
          out_tok[n_acc] = tok[next];
          out_path[n_acc + 1] = next;
        }
        ++n_acc;
        u = next;
        continue;
      }
      final_tok = sp.argmax;
      break;
    }
    const void* prow = row_at(job.base_p, job, b, u, Elt<T>::kBytes);
    const void* qrow = row_at(job.base_q, job, b, u, Elt<T>::kBytes);
    spec_row_stats sq = sp;
    if (c1 > c0) {
      sq = job.stats_q[(int64_t)b * N + u];
      if (sq.status != SPEC_TREE_OK) { status = SPEC_ROW_NONFINITE; break; }
    }
    const float inv_sp = (float)(1.0 / sp.s_f);
    const float inv_sq = (float)(1.0 / sq.s_f);
    int j = 0, next = -1;
    for (int i = c0; i < c1; ++i) {
      const int ch = cl[i];
      if (threadIdx.x == 0) {
        const int x = tok[ch];
        double P = prob64<T>(prow, x, sp, Td);
        double Q = prob64<T>(qrow, x, sq, Td);
        for (int r = 0; r < j; ++r)
          if (Z[r] > 0.0) P = fmax(0.0, P - Q) / Z[r];
        double alpha = (Q > 0.0) ? fmin(1.0, P / Q) : (P > 0.0 ? 1.0 : 0.0);
        uint4 w = philox_words(job.seed, job.offset, b, ch);
        double r = unit_uniform(w.x);
        if (job.out_alpha) job.out_alpha[(int64_t)b * N + ch] = (float)alpha;
        sh.accept = (r <= alpha);
      }
      __syncthreads();
      const int acc = sh.accept;
      __syncthreads();
      if (acc) { next = ch; break; }
      double z = residual_mass<T>(prow, qrow, V, sp, sq, c, inv_sp, inv_sq, j, invz, sh);
      if (threadIdx.x == 0) {
        Z[j] = z;
        invz[j] = (z > 0.0) ? (float)(1.0 / z) : -1.f;
        if (job.counters) {
          atomicAdd(&job.counters[2], 2ull * (unsigned long long)V * Elt<T>::kBytes);
          atomicAdd(&job.counters[3], 1ull);
        }
      }
      __syncthreads();
      ++j;
    }
    if (next >= 0) {
      if (threadIdx.x == 0) {
        out_tok[n_acc] = tok[next];
        out_path[n_acc + 1] = next;
      }
      ++n_acc;
      u = next;
      continue;
    }
    uint4 w = philox_words(job.seed, job.offset, b, u);
    double r = unit_uniform(w.y);
    final_tok = inverse_cdf<T>(prow, qrow, V, sp, sq, c, inv_sp, inv_sq, j, invz, r, sh);
    if (threadIdx.x == 0 && job.counters) {
      atomicAdd(&job.counters[2], (unsigned long long)(j > 0 ? 2 : 1) * V * Elt<T>::kBytes);
      atomicAdd(&job.counters[4], 1ull);
    }
    break;
  }
  if (threadIdx.x == 0) {
    if (status != SPEC_TREE_OK) {
      job.out_accept_len[b] = -1;
      for (int k = 0; k < W; ++k) { out_tok[k] = -1; out_path[k] = -1; }
    } else {
      job.out_accept_len[b] = n_acc;
      out_path[0] = 0;
      out_tok[n_acc] = final_tok;
      for (int k = n_acc + 1; k < W; ++k) { out_tok[k] = -1; out_path[k] = -1; }
    }
    if (job.out_status) job.out_status[b] = status;
  }
}

__global__ void philox_words_kernel(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                                    const int32_t* node_idx, int32_t n, uint32_t* out) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  uint4 w = philox_words(seed, offset, b_idx[i], node_idx[i]);
  reinterpret_cast<uint4*>(out)[i] = w;
}

}  // namespace

cudaError_t launch_tree_prep(const TreeJob& job, bool greedy, cudaStream_t s) {
  const int threads = 64;
  int blocks = (job.B + threads - 1) / threads;
  if (blocks < 1) blocks = 1;
  tree_prep_kernel<<<blocks, threads, 0, s>>>(job, greedy ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_tree_walk(const TreeJob& job, spec_dtype dtype, bool greedy, cudaStream_t s) {
  dim3 grid(job.B);
  if (dtype == SPEC_BF16) {
    if (greedy) tree_walk_kernel<uint16_t, true><<<grid, WT, 0, s>>>(job);
    else tree_walk_kernel<uint16_t, false><<<grid, WT, 0, s>>>(job);
  } else {
    if (greedy) tree_walk_kernel<float, true><<<grid, WT, 0, s>>>(job);
    else tree_walk_kernel<float, false><<<grid, WT, 0, s>>>(job);
  }
  return cudaGetLastError();
}

cudaError_t launch_philox_words(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                                const int32_t* node_idx, int32_t n, uint32_t* out,
                                cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  philox_words_kernel<<<(n + 255) / 256, 256, 0, s>>>(seed, offset, b_idx, node_idx, n, out);
  return cudaGetLastError();
}

}  // namespace svk
