// walk.cu -- the per-tree accept walk.
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
//
// One block per tree.  The block first checks the tree and builds its child
// lists in shared memory; the walk itself is sequential, and every rejection or
// final draw is one block-wide pass over the (p_u, q_u) row pair.
#include <climits>

#include "common.cuh"

namespace svk {

namespace {

constexpr int WT = kWalkThreads;
constexpr int WW = WT / 32;
constexpr int kWalkUnroll = 4;

__device__ __forceinline__ const void* row_at(const void* base, const TreeJob& j, int b, int n,
                                              int bytes) {
  const int64_t off = (int64_t)b * j.batch_stride + (int64_t)n * j.row_pitch;
  return static_cast<const void*>(static_cast<const char*>(base) + off * bytes);
}

struct WalkShared {
  double red[WW];
  double wtot[WW];
  double target;
  int target_warp;
  int accept;
  int final_tok;
  int status;
  float inv_sp, inv_sq;
};

// Is token x (logit z) inside the kept set of a filtered row?
__device__ __forceinline__ bool kept_tok(float z, int x, const spec_row_stats& st) {
  const uint32_t k = order_key(z);
  return k > st.cut_key || (k == st.cut_key && x <= st.cut_idx);
}

// Filtered probability of one token in fp64 (for the acceptance test).
template <typename T>
__device__ double prob64(const void* row, int x, const spec_row_stats& st, double T_) {
  const float z = Elt<T>::at(row, x);
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
    const float iz = invz[r];
    if (iz > 0.f) p = fmaxf(0.f, p - q) * iz;
  }
  return p;
}

// Block sum of per-thread Kahan accumulators (float-float within warps, fp64 across).
__device__ double block_sum(const Kahan& k, WalkShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const FF v = warp_sum_ff(k.ff());
  __syncthreads();
  if (lane == 0) sh.red[warp] = v.value();
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
      const int x = u * E + e;
      val[e] = (x < V) ? prob32(zp[e], x, sp, c, inv_sp) : 0.f;
    }
    return;
  }
  float zq[E];
  load_unit<T>(qrow, V, u, zq);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int x = u * E + e;
    if (x < V) {
      const float p = prob32(zp[e], x, sp, c, inv_sp);
      const float q = prob32(zq[e], x, sq, c, inv_sq);
      val[e] = residual_chain(p, q, j, invz);
    } else {
      val[e] = 0.f;
    }
  }
}

// Z = sum_x max(0, p^(j)(x) - q(x)) over the row pair (block-wide).  Each thread
// issues the loads of kWalkUnroll units of both rows before using them.
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
  return block_sum(acc, sh);
}

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

// Inverse-CDF draw in index order: the smallest x with C_x >= r * C_V, where C is the
// inclusive prefix sum of the current distribution.  Warps own contiguous ranges of
// units; a warp step covers 32 consecutive units (one per lane) and its total is an
// fp32 butterfly sum, accumulated in float-float.  The owning warp retraces its step
// totals in the same order in the second phase, so its running sum reproduces the
// first phase exactly.
template <typename T>
__device__ int inverse_cdf(const void* prow, const void* qrow, int V, const spec_row_stats& sp,
                           const spec_row_stats& sq, float c, float inv_sp, float inv_sq, int j,
                           const float* invz, double r, WalkShared& sh) {
  constexpr int E = Elt<T>::kPerUnit;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nunits = (V + E - 1) / E;
  const int per_warp = (nunits + WW - 1) / WW;
  const int u_lo = warp * per_warp, u_hi = min(nunits, u_lo + per_warp);
  FF wt;
  for (int ub = u_lo; ub < u_hi; ub += 64) {
    float val0[E], val1[E];
    const int ua = ub + lane, uc = ub + 32 + lane;
    const float s0 = (ua < u_hi) ? unit_sum<T>(prow, qrow, V, ua, sp, sq, c, inv_sp, inv_sq, j, invz, val0) : 0.f;
    const float s1 = (uc < u_hi) ? unit_sum<T>(prow, qrow, V, uc, sp, sq, c, inv_sp, inv_sq, j, invz, val1) : 0.f;
    wt.add(warp_sum_f(s0));
    wt.add(warp_sum_f(s1));
  }
  if (lane == 0) sh.wtot[warp] = wt.value();
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
    if (tw < 0 && last >= 0) { tw = last; tw_base = last_base; t = last_base + sh.wtot[last]; }
    // an all-zero distribution (not reachable from a valid row) draws nothing: the
    // caller falls back to the row's argmax
    sh.target_warp = tw;
    sh.target = tw >= 0 ? fmin(t - tw_base, sh.wtot[tw]) : 0.0;
    sh.final_tok = -1;
  }
  __syncthreads();
  if (warp == sh.target_warp) {
    const double target = sh.target;
    FF cum;
    bool found = false;
    for (int ub = u_lo; ub < u_hi && !found; ub += 32) {
      const int u = ub + lane;
      float val[E];
      const float s = (u < u_hi) ? unit_sum<T>(prow, qrow, V, u, sp, sq, c, inv_sp, inv_sq, j, invz, val) : 0.f;
      const float it = warp_sum_f(s);
      FF next = cum;
      next.add(it);
      // the crossing test is made once (lane 0) in fp64 and broadcast
      int cross = 0;
      if (lane == 0) cross = (it > 0.f && next.value() >= target);
      cross = __shfl_sync(kFull, cross, 0);
      if (cross) {
        float incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += t;
        }
        const double base = cum.value();
        const double before = base + (double)(incl - s);
        const unsigned hit = __ballot_sync(kFull, s > 0.f && base + (double)incl >= target);
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
      cum = next;
    }
  }
  __syncthreads();
  return sh.final_tok;
}

// ---------------------------------------------------------------------------
// The walk: one block per tree.
// ---------------------------------------------------------------------------
template <typename T, bool GREEDY>
__global__ void __launch_bounds__(WT, 1) tree_walk_kernel(TreeJob job) {
  __shared__ WalkShared sh;
  // parents [N], tokens [N], child_start [N+1], children [N], then Z [N] (fp64) and 1/Z [N]
  extern __shared__ __align__(16) int32_t tsm[];
  const int b = blockIdx.x;
  const int N = job.N, V = job.V, W = job.W;
  int32_t* par = tsm;
  int32_t* tok = tsm + N;
  int32_t* cs = tsm + 2 * N;
  int32_t* cl = tsm + 3 * N + 1;
  int32_t* out_tok = job.out_tokens + (int64_t)b * W;
  int32_t* out_path = job.out_path + (int64_t)b * W;
  double* Z = reinterpret_cast<double*>(tsm + ((4 * N + 1 + 1) & ~1));
  float* invz = reinterpret_cast<float*>(Z + N);
  const double Td = (double)job.temperature;
  const float c = job.c;

  // ---- tree checks and child lists ----
  for (int n = threadIdx.x; n < N; n += WT) {
    par[n] = job.parents[(int64_t)b * N + n];
    tok[n] = job.tokens[(int64_t)b * N + n];
    if (job.out_alpha) job.out_alpha[(int64_t)b * N + n] = __int_as_float(0x7fc00000);
  }
  __syncthreads();
  int bad = 0;
  for (int n = threadIdx.x; n < N; n += WT) {
    if (n == 0) bad |= (par[0] != -1);
    else bad |= (par[n] < 0 || par[n] >= n || tok[n] < 0 || tok[n] >= V);
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    int status = bad ? SPEC_TREE_INVALID : SPEC_TREE_OK;
    if (!bad) {
      // depths (kept in the child array until the lists are built) and the depth limit
      cl[0] = 0;
      for (int n = 1; n < N; ++n) {
        cl[n] = cl[par[n]] + 1;
        if (cl[n] > W - 1) { status = SPEC_TREE_INVALID; break; }
      }
    }
    if (status == SPEC_TREE_OK) {
      for (int u = 0; u <= N; ++u) cs[u] = 0;
      for (int n = 1; n < N; ++n) cs[par[n] + 1] += 1;
      for (int u = 1; u <= N; ++u) cs[u] += cs[u - 1];
      for (int n = 1; n < N; ++n) cl[cs[par[n]]++] = n;  // children land in node order
      for (int u = N; u >= 1; --u) cs[u] = cs[u - 1];
      cs[0] = 0;
    }
    sh.status = status;
  }
  __syncthreads();
  int status = sh.status;

  int u = 0, n_acc = 0, final_tok = -1;
  while (status == SPEC_TREE_OK) {
    const spec_row_stats sp = job.stats_p[(int64_t)b * N + u];
    if (sp.status != SPEC_TREE_OK) { status = sp.status; break; }
    const int c0 = cs[u], c1 = cs[u + 1];
    if (GREEDY) {
      int next = -1;
      for (int i = c0; i < c1; ++i) {
        const int ch = cl[i];
        const bool ok = tok[ch] == sp.argmax;
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
      if (sq.status != SPEC_TREE_OK) { status = sq.status; break; }
    }
    if (threadIdx.x == 0) {
      sh.inv_sp = (float)(1.0 / sp.s_f);
      sh.inv_sq = (float)(1.0 / sq.s_f);
    }
    __syncthreads();
    const float inv_sp = sh.inv_sp, inv_sq = sh.inv_sq;
    int j = 0, next = -1;
    for (int i = c0; i < c1; ++i) {
      const int ch = cl[i];
      if (threadIdx.x == 0) {
        const int x = tok[ch];
        double P = prob64<T>(prow, x, sp, Td);
        const double Q = prob64<T>(qrow, x, sq, Td);
        for (int r = 0; r < j; ++r)
          if (Z[r] > 0.0) P = fmax(0.0, P - Q) / Z[r];
        const double alpha = (Q > 0.0) ? fmin(1.0, P / Q) : (P > 0.0 ? 1.0 : 0.0);
        const uint4 w = philox_words(job.seed, job.offset, b, ch);
        const double rr = unit_uniform(w.x);
        if (job.out_alpha) job.out_alpha[(int64_t)b * N + ch] = (float)alpha;
        sh.accept = (rr <= alpha);
      }
      __syncthreads();
      const int acc = sh.accept;
      __syncthreads();
      if (acc) { next = ch; break; }
      const double z = residual_mass<T>(prow, qrow, V, sp, sq, c, inv_sp, inv_sq, j, invz, sh);
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
    const uint4 w = philox_words(job.seed, job.offset, b, u);
    const double rr = unit_uniform(w.y);
    final_tok = inverse_cdf<T>(prow, qrow, V, sp, sq, c, inv_sp, inv_sq, j, invz, rr, sh);
    if (final_tok < 0) final_tok = sp.argmax;
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
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 w = philox_words(seed, offset, b_idx[i], node_idx[i]);
  reinterpret_cast<uint4*>(out)[i] = w;
}

template <typename T, bool GREEDY>
cudaError_t launch_walk_t(const TreeJob& job, cudaStream_t s) {
  const size_t dyn = (size_t)((4 * job.N + 1 + 1) & ~1) * sizeof(int32_t) +
                     (size_t)job.N * (sizeof(double) + sizeof(float));
  if (dyn > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        tree_walk_kernel<T, GREEDY>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
  }
  tree_walk_kernel<T, GREEDY><<<job.B, WT, dyn, s>>>(job);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tree_walk(const TreeJob& job, spec_dtype dtype, bool greedy, cudaStream_t s) {
  if (dtype == SPEC_BF16)
    return greedy ? launch_walk_t<uint16_t, true>(job, s) : launch_walk_t<uint16_t, false>(job, s);
  return greedy ? launch_walk_t<float, true>(job, s) : launch_walk_t<float, false>(job, s);
}

cudaError_t launch_philox_words(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                                const int32_t* node_idx, int32_t n, uint32_t* out,
                                cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  philox_words_kernel<<<(n + 255) / 256, 256, 0, s>>>(seed, offset, b_idx, node_idx, n, out);
  return cudaGetLastError();
}

}  // namespace svk
