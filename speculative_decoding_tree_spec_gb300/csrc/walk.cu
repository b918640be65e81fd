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
// Greedy trees need only the row statistics: one small block per tree follows
// the argmax.  Sampling trees run on a thread-block cluster of C CTAs per tree.
// Every CTA owns a contiguous slice of the vocabulary, all CTAs take the same
// walk decisions, and each rejection or final draw is one pass over the slices of
// the (p_u, q_u) row pair whose partial sums are exchanged through distributed
// shared memory: every CTA pushes its partial into every CTA's slot array and
// arrives on that CTA's mbarrier, then sums the C slots in rank order, so all CTAs
// hold bit-identical totals.  Every mbarrier wait is bounded in time.
#include <climits>

#include <cuda_bf16.h>

#include "common.cuh"

namespace svk {

namespace {

constexpr int GT = kWalkThreads;          // greedy walk block
constexpr int CT = kClusterWalkThreads;   // sampling walk CTA
constexpr int CW = CT / 32;
constexpr int kMaxC = kMaxWalkCluster;
constexpr int kUnitsInFlight = 2;          // units of each row a thread loads before using them
constexpr uint64_t kExchangeLimitNs = 2000000000ull;

__device__ __forceinline__ const void* row_at(const void* base, const TreeJob& j, int b, int n,
                                              int bytes) {
  const int64_t off = (int64_t)b * j.batch_stride + (int64_t)n * j.row_pitch;
  return static_cast<const void*>(static_cast<const char*>(base) + off * bytes);
}

// ---------------------------------------------------------------------------
// Tree checks and child lists (both walks).  par/tok/cs/cl live in shared
// memory: parents, tokens, child-list offsets [N+1] and child lists [N].
// Children of a node land in increasing node order.  Returns the tree status,
// uniform over the block.
// ---------------------------------------------------------------------------
__device__ int load_tree(const TreeJob& job, int b, int32_t* par, int32_t* tok, int32_t* cs,
                         int32_t* cl, bool init_alpha, int* s_status) {
  const int N = job.N, V = job.V, W = job.W;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    par[n] = job.parents[(int64_t)b * N + n];
    tok[n] = job.tokens[(int64_t)b * N + n];
    if (init_alpha && job.out_alpha) job.out_alpha[(int64_t)b * N + n] = __int_as_float(0x7fc00000);
  }
  __syncthreads();
  int bad = 0;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
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
      for (int n = 1; n < N; ++n) cl[cs[par[n]]++] = n;
      for (int u = N; u >= 1; --u) cs[u] = cs[u - 1];
      cs[0] = 0;
    }
    *s_status = status;
  }
  __syncthreads();
  return *s_status;
}

// Final writes of one tree (one thread): accepted length, the final token unless
// another CTA wrote it, the padding, the status.
__device__ void finish_tree(const TreeJob& job, int b, int status, int n_acc, int final_tok,
                            bool write_final) {
  const int W = job.W;
  int32_t* out_tok = job.out_tokens + (int64_t)b * W;
  int32_t* out_path = job.out_path + (int64_t)b * W;
  if (status != SPEC_TREE_OK) {
    job.out_accept_len[b] = -1;
    for (int k = 0; k < W; ++k) { out_tok[k] = -1; out_path[k] = -1; }
  } else {
    job.out_accept_len[b] = n_acc;
    out_path[0] = 0;
    if (write_final) out_tok[n_acc] = final_tok;
    for (int k = n_acc + 1; k < W; ++k) { out_tok[k] = -1; out_path[k] = -1; }
  }
  if (job.out_status) job.out_status[b] = status;
}

// ---------------------------------------------------------------------------
// Greedy walk: one block per tree; decisions come from the row argmax alone.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(GT) greedy_walk_kernel(TreeJob job) {
  __shared__ int s_status;
  extern __shared__ __align__(16) int32_t tsm[];
  const int b = blockIdx.x;
  const int N = job.N;
  int32_t *par = tsm, *tok = tsm + N, *cs = tsm + 2 * N, *cl = tsm + 3 * N + 1;
  int status = load_tree(job, b, par, tok, cs, cl, true, &s_status);
  if (threadIdx.x != 0) return;
  int32_t* out_tok = job.out_tokens + (int64_t)b * job.W;
  int32_t* out_path = job.out_path + (int64_t)b * job.W;
  int u = 0, n_acc = 0, final_tok = -1;
  while (status == SPEC_TREE_OK) {
    const spec_row_stats sp = job.stats_p[(int64_t)b * N + u];
    if (sp.status != SPEC_TREE_OK) { status = sp.status; break; }
    int next = -1;
    for (int i = cs[u]; i < cs[u + 1]; ++i) {
      const int ch = cl[i];
      const bool ok = tok[ch] == sp.argmax;
      if (job.out_alpha) job.out_alpha[(int64_t)b * N + ch] = ok ? 1.f : 0.f;
      if (ok) { next = ch; break; }
    }
    if (next < 0) { final_tok = sp.argmax; break; }
    out_tok[n_acc] = tok[next];
    out_path[n_acc + 1] = next;
    ++n_acc;
    u = next;
  }
  finish_tree(job, b, status, n_acc, final_tok, true);
}

// ---------------------------------------------------------------------------
// Sampling walk: elementwise filtered probabilities.
// ---------------------------------------------------------------------------

// One filtered row: token x (logit z) is kept iff z > zc, or z == zc and x <= ci
// (the order-key rule of spec_row_stats written on values; the no-truncation
// sentinel keeps everything).  Its probability is 2^((z - m) c) * inv_s.
struct RowF {
  float m, c, inv_s, zc;
  int ci;
  uint32_t zc2;  // zc as a pair of bf16 (bf16 rows: zc is exactly representable)
};

__device__ __forceinline__ RowF make_rowf(const spec_row_stats& st, float c, float inv_s) {
  RowF f;
  f.m = st.m;
  f.c = c;
  f.inv_s = inv_s;
  if (st.cut_key == 0u) {
    f.zc = -CUDART_INF_F;
    f.ci = INT_MAX;
  } else {
    f.zc = key_value(st.cut_key);
    f.ci = st.cut_idx;
  }
  const uint32_t h = __float_as_uint(f.zc) >> 16;
  f.zc2 = h | (h << 16);
  return f;
}

constexpr uint32_t kNegInfBf16x2 = 0xff80ff80u;
constexpr uint32_t kNegInfF32 = 0xff800000u;

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}

// Raw bits of unit u (16 bytes); positions at or beyond V read as -inf.
template <typename T>
__device__ __forceinline__ uint4 load_raw(const void* row, int V, int u) {
  constexpr int E = Elt<T>::kPerUnit;
  const int x0 = u * E;
  if (x0 + E <= V) return __ldg(reinterpret_cast<const uint4*>(row) + u);
  uint32_t w[4];
  if (E == 8) {
    const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t lo = (x0 + 2 * q < V) ? (uint32_t)__ldg(r + x0 + 2 * q) : 0xff80u;
      const uint32_t hi = (x0 + 2 * q + 1 < V) ? (uint32_t)__ldg(r + x0 + 2 * q + 1) : 0xff80u;
      w[q] = lo | (hi << 16);
    }
  } else {
    const uint32_t* r = reinterpret_cast<const uint32_t*>(row);
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = (x0 + q < V) ? __ldg(r + x0 + q) : kNegInfF32;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Tokens of the unit outside the kept set become -inf (weight 0).
__device__ __forceinline__ void filter_unit(uint4& raw, int x0, const RowF& f, uint16_t) {
  const __nv_bfloat162 t = as_bf2(f.zc2);
  uint32_t r[4] = {raw.x, raw.y, raw.z, raw.w};
  if (x0 + 7 <= f.ci) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t m = __hge2_mask(as_bf2(r[q]), t);
      r[q] = (r[q] & m) | (kNegInfBf16x2 & ~m);
    }
  } else if (x0 > f.ci) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t m = __hgt2_mask(as_bf2(r[q]), t);
      r[q] = (r[q] & m) | (kNegInfBf16x2 & ~m);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t sel = ((x0 + 2 * q <= f.ci) ? 0x0000ffffu : 0u) |
                           ((x0 + 2 * q + 1 <= f.ci) ? 0xffff0000u : 0u);
      const uint32_t m = (__hge2_mask(as_bf2(r[q]), t) & sel) |
                         (__hgt2_mask(as_bf2(r[q]), t) & ~sel);
      r[q] = (r[q] & m) | (kNegInfBf16x2 & ~m);
    }
  }
  raw = make_uint4(r[0], r[1], r[2], r[3]);
}
__device__ __forceinline__ void filter_unit(uint4& raw, int x0, const RowF& f, float) {
  uint32_t r[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float z = __uint_as_float(r[q]);
    const bool kept = (x0 + q <= f.ci) ? (z >= f.zc) : (z > f.zc);
    r[q] = kept ? r[q] : kNegInfF32;
  }
  raw = make_uint4(r[0], r[1], r[2], r[3]);
}

// Filtered probabilities of one unit: 2^((z - m) c) * inv_s, evaluated with the
// same roundings as the dense row pass's weights.
template <typename T>
__device__ __forceinline__ void unit_probs(uint4 raw, int x0, const RowF& f,
                                           float (&w)[Elt<T>::kPerUnit]) {
  constexpr int E = Elt<T>::kPerUnit;
  filter_unit(raw, x0, f, T());
  float z[E];
  Elt<T>::unpack(raw, z);
  const float2 nm = make_float2(-f.m, -f.m), c2 = make_float2(f.c, f.c);
  const float2 s2 = make_float2(f.inv_s, f.inv_s);
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float2 d = __fmul2_rn(__fadd2_rn(make_float2(z[e], z[e + 1]), nm), c2);
    const float2 v = __fmul2_rn(make_float2(ex2_approx(d.x), ex2_approx(d.y)), s2);
    w[e] = v.x;
    w[e + 1] = v.y;
  }
}

// p after j renormalised residual steps: p <- max(0, p - q) / Z_r for every r < j
// with Z_r > 0 (a zero residual mass leaves p unchanged).
template <int E>
__device__ __forceinline__ void residual_chain(float (&p)[E], const float (&q)[E], int j,
                                               const float* invz) {
  for (int r = 0; r < j; ++r) {
    const float iz = invz[r];
    if (iz > 0.f) {
#pragma unroll
      for (int e = 0; e < E; ++e) p[e] = __fmul_rn(fmaxf(0.f, __fsub_rn(p[e], q[e])), iz);
    }
  }
}

// Values of the current distribution on unit u (p after j residual steps) and
// their sum in element order.  Both inverse-CDF phases call this, so a unit
// always yields the same values and sum.
template <typename T>
__device__ __forceinline__ float dist_unit(const void* prow, const void* qrow, int V, int u,
                                           const RowF& fp, const RowF& fq, int j,
                                           const float* invz, float (&val)[Elt<T>::kPerUnit]) {
  constexpr int E = Elt<T>::kPerUnit;
  unit_probs<T>(load_raw<T>(prow, V, u), u * E, fp, val);
  if (j > 0) {
    float q[E];
    unit_probs<T>(load_raw<T>(qrow, V, u), u * E, fq, q);
    residual_chain<E>(val, q, j, invz);
  }
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) s = __fadd_rn(s, val[e]);
  return s;
}

// Filtered probability of one token in fp64 (for the acceptance test).
template <typename T>
__device__ double prob64(const void* row, int x, const spec_row_stats& st, double T_) {
  const float z = Elt<T>::at(row, x);
  const uint32_t k = order_key(z);
  if (!(k > st.cut_key || (k == st.cut_key && x <= st.cut_idx))) return 0.0;
  return exp(((double)z - (double)st.m) / T_) / st.s_f;
}

// ---------------------------------------------------------------------------
// Cluster plumbing.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;\n" ::
                   : "memory");
}
// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_peer_f64(uint32_t addr, double v) {
  asm volatile("st.shared::cluster.f64 [%0], %1;\n" ::"r"(addr), "d"(v) : "memory");
}
__device__ __forceinline__ void arrive_peer(uint32_t bar_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(bar_addr)
               : "memory");
}
__device__ __forceinline__ void or_peer_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.or.b32 [%0], %1;\n" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ bool mbar_try_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int k = 0; k < 32; ++k)
      if (mbar_try_cluster(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

struct CShared {
  double slot[2][kMaxC];  // partials pushed by every CTA, two alternating sets
  uint64_t xbar[2];       // one mbarrier per slot set, C arrivals per phase
  double wred[CW];
  double wtot[CW];
  double target;
  int accept, status, target_warp, final_tok;
  unsigned err;           // rank 0: timeouts reported by any CTA of the cluster
  float inv_sp, inv_sq;
};

// Cluster-wide sum of one value per CTA (`v` is read from thread 0).  Every CTA
// pushes v into slot[set][rank] of every CTA and arrives on that CTA's mbarrier;
// after the local mbarrier completes, each thread sums the C slots in rank order.
// Returns false (uniformly over the CTA) if the wait gave up.  A slot set is
// written again two exchanges later, which no CTA can start before every CTA has
// pushed the exchange in between -- after its threads read this one.
__device__ bool cluster_sum(double v, CShared& sh, int C, uint32_t rank, uint32_t& n_ex,
                            double& total, const double** slots) {
  const int set = n_ex & 1;
  const uint32_t parity = (n_ex >> 1) & 1u;
  ++n_ex;
  if (threadIdx.x == 0) {
    for (int c = 0; c < C; ++c) {
      st_peer_f64(peer_addr(&sh.slot[set][rank], c), v);
      arrive_peer(peer_addr(&sh.xbar[set], c));
    }
  }
  const bool ok = __syncthreads_and(mbar_wait_cluster(&sh.xbar[set], parity, kExchangeLimitNs));
  double t = 0.0;
  for (int c = 0; c < C; ++c) t += sh.slot[set][c];
  total = t;
  if (slots) *slots = sh.slot[set];
  return ok;
}

// Block sum of per-thread float-float partials in fixed order (result in thread 0).
__device__ double block_sum_ff(FF v, CShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_ff(v);
  if (lane == 0) sh.wred[warp] = v.value();
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < CW; ++w) t += sh.wred[w];
  return t;
}

// Partial residual mass of this CTA's slice: sum over its tokens of
// max(0, p^(j) - q).
template <typename T>
__device__ FF residual_partial(const void* prow, const void* qrow, int V, int ua, int ub,
                               const RowF& fp, const RowF& fq, int j, const float* invz) {
  constexpr int E = Elt<T>::kPerUnit;
  FF acc;
  for (int u0 = ua + threadIdx.x; u0 < ub; u0 += CT * kUnitsInFlight) {
    uint4 rp[kUnitsInFlight], rq[kUnitsInFlight];
#pragma unroll
    for (int k = 0; k < kUnitsInFlight; ++k) {
      const int u = u0 + k * CT;
      if (u < ub) {
        rp[k] = load_raw<T>(prow, V, u);
        rq[k] = load_raw<T>(qrow, V, u);
      }
    }
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < kUnitsInFlight; ++k) {
      const int u = u0 + k * CT;
      if (u < ub) {
        float p[E], q[E];
        unit_probs<T>(rp[k], u * E, fp, p);
        unit_probs<T>(rq[k], u * E, fq, q);
        residual_chain<E>(p, q, j, invz);
#pragma unroll
        for (int e = 0; e < E; ++e) part += fmaxf(0.f, __fsub_rn(p[e], q[e]));
      }
    }
    acc.add(part);
  }
  return acc;
}

// First index whose running total reaches `t` among n non-negative totals (fixed
// order, fp64); the last positive one when rounding leaves the target just above
// the sum.  Returns -1 when every total is zero; `base` gets the sum before the
// chosen index and `t_in` the target inside it, clamped to its total.
__device__ __forceinline__ int pick_crossing(const double* tot, int n, double t, double& base,
                                             double& t_in) {
  double cum = 0.0, last_base = 0.0;
  int hit = -1, last = -1;
  for (int i = 0; i < n; ++i) {
    if (tot[i] > 0.0) {
      last = i;
      last_base = cum;
      if (hit < 0 && cum + tot[i] >= t) { hit = i; base = cum; }
    }
    cum += tot[i];
  }
  if (hit < 0 && last >= 0) { hit = last; base = last_base; t = last_base + tot[last]; }
  if (hit >= 0) t_in = fmin(t - base, tot[hit]);
  return hit;
}

// Inverse-CDF draw over the cluster: the smallest token x with C_x >= r * C_V,
// C the inclusive prefix sum of the current distribution in vocabulary order.
// Phase 1: every warp of every CTA sums its contiguous range in 32-unit steps
// (fp32 butterfly per step, float-float across steps) and keeps each step total in
// shared memory; CTA totals are exchanged.  Phase 2: the CTA whose slice holds the
// crossing picks the warp, replays that warp's step totals in the same order to
// find the step, recomputes that one step and resolves the lane and the token.
// Returns the token in the owning CTA (-1 elsewhere); `owner` is the owning rank
// for every CTA, -1 when the distribution is all zero.
template <typename T>
__device__ int cluster_inverse_cdf(const void* prow, const void* qrow, int V, int ua, int ub,
                                   const RowF& fp, const RowF& fq, int j, const float* invz,
                                   double r, float* steps, int max_steps, CShared& sh, int C,
                                   uint32_t rank, uint32_t& n_ex, bool& ok, int& owner) {
  constexpr int E = Elt<T>::kPerUnit;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per_warp = (ub - ua + CW - 1) / CW;
  const int lo = min(ub, ua + warp * per_warp), hi = min(ub, lo + per_warp);
  float* st = steps + warp * max_steps;
  FF wt;
  int ns = 0;
  for (int base_u = lo; base_u < hi; base_u += 32, ++ns) {
    const int u = base_u + lane;
    float val[E];
    const float s = (u < hi) ? dist_unit<T>(prow, qrow, V, u, fp, fq, j, invz, val) : 0.f;
    const float it = warp_sum_f(s);
    if (lane == 0) st[ns] = it;
    wt.add(it);
  }
  if (lane == 0) sh.wtot[warp] = wt.value();
  __syncthreads();
  double v = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < CW; ++w) v += sh.wtot[w];
  double total;
  const double* cta_tot = nullptr;
  ok = cluster_sum(v, sh, C, rank, n_ex, total, &cta_tot);
  owner = -1;
  if (!ok) return -1;
  double base_c = 0.0, t_c = 0.0;
  owner = pick_crossing(cta_tot, C, r * total, base_c, t_c);
  if (owner != (int)rank) return -1;
  if (threadIdx.x == 0) {
    double base_w = 0.0, t_w = 0.0;
    sh.target_warp = pick_crossing(sh.wtot, CW, t_c, base_w, t_w);
    sh.target = t_w;
    sh.final_tok = -1;
  }
  __syncthreads();
  if (warp == sh.target_warp) {
    const double target = sh.target;
    // the crossing step, found by replaying phase 1's accumulation
    int s_hit = -1;
    double base = 0.0;
    if (lane == 0) {
      FF cum;
      int s_last = -1;
      double last_base = 0.0;
      for (int s = 0; s < ns; ++s) {
        const float it = st[s];
        FF next = cum;
        next.add(it);
        if (it > 0.f) {
          s_last = s;
          last_base = cum.value();
          if (next.value() >= target) { s_hit = s; base = cum.value(); break; }
        }
        cum = next;
      }
      if (s_hit < 0) { s_hit = s_last; base = last_base; }
    }
    s_hit = __shfl_sync(kFull, s_hit, 0);
    base = __shfl_sync(kFull, base, 0);
    if (s_hit >= 0) {
      const int u = lo + 32 * s_hit + lane;
      float val[E];
      const float s = (u < hi) ? dist_unit<T>(prow, qrow, V, u, fp, fq, j, invz, val) : 0.f;
      float incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
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
    }
  }
  __syncthreads();
  return sh.final_tok;
}

// ---------------------------------------------------------------------------
// Sampling walk: one cluster of C CTAs per tree.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(CT, 3) cluster_walk_kernel(TreeJob job, int C, int max_steps) {
  __shared__ CShared sh;
  // parents [N], tokens [N], child offsets [N+1], children [N]; then Z [N] (fp64),
  // 1/Z [N] and the per-warp step totals [CW][max_steps]
  extern __shared__ __align__(16) int32_t tsm[];
  constexpr int E = Elt<T>::kPerUnit;
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / C;
  const int N = job.N, V = job.V, W = job.W;
  int32_t *par = tsm, *tok = tsm + N, *cs = tsm + 2 * N, *cl = tsm + 3 * N + 1;
  double* Z = reinterpret_cast<double*>(tsm + ((4 * N + 1 + 1) & ~1));
  float* invz = reinterpret_cast<float*>(Z + N);
  float* steps = invz + N;
  const double Td = (double)job.temperature;
  const float c = job.c;
  const bool lead = (rank == 0);

  if (threadIdx.x == 0) {
    mbar_init(&sh.xbar[0], (uint32_t)C);
    mbar_init(&sh.xbar[1], (uint32_t)C);
    sh.err = 0u;
    fence_barrier_init();
  }
  cluster_sync_all();

  int status = load_tree(job, b, par, tok, cs, cl, lead, &sh.status);
  const int nunits = (V + E - 1) / E;
  const int ua = (int)((int64_t)nunits * rank / C), ub = (int)((int64_t)nunits * (rank + 1) / C);
  int32_t* out_tok = job.out_tokens + (int64_t)b * W;
  int32_t* out_path = job.out_path + (int64_t)b * W;
  uint32_t n_ex = 0;
  bool timed_out = false;
  int u = 0, n_acc = 0, final_tok = -1, owner = -1;

  while (status == SPEC_TREE_OK) {
    const spec_row_stats sp = job.stats_p[(int64_t)b * N + u];
    if (sp.status != SPEC_TREE_OK) { status = sp.status; break; }
    const int c0 = cs[u], c1 = cs[u + 1];
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
    const RowF fp = make_rowf(sp, c, sh.inv_sp), fq = make_rowf(sq, c, sh.inv_sq);
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
        if (lead && job.out_alpha) job.out_alpha[(int64_t)b * N + ch] = (float)alpha;
        sh.accept = (unit_uniform(w.x) <= alpha);
      }
      __syncthreads();
      const int acc = sh.accept;
      __syncthreads();
      if (acc) { next = ch; break; }
      const double part = block_sum_ff(
          residual_partial<T>(prow, qrow, V, ua, ub, fp, fq, j, invz), sh);
      double z;
      if (!cluster_sum(part, sh, C, rank, n_ex, z, nullptr)) { timed_out = true; break; }
      if (threadIdx.x == 0) {
        Z[j] = z;
        invz[j] = (z > 0.0) ? (float)(1.0 / z) : -1.f;
        if (lead && job.counters) {
          atomicAdd(&job.counters[2], 2ull * (unsigned long long)V * Elt<T>::kBytes);
          atomicAdd(&job.counters[3], 1ull);
        }
      }
      __syncthreads();
      ++j;
    }
    if (timed_out) { status = SPEC_ROW_TIMEOUT; break; }
    if (next >= 0) {
      if (lead && threadIdx.x == 0) {
        out_tok[n_acc] = tok[next];
        out_path[n_acc + 1] = next;
      }
      ++n_acc;
      u = next;
      continue;
    }
    const uint4 w = philox_words(job.seed, job.offset, b, u);
    bool ok = true;
    const int t = cluster_inverse_cdf<T>(prow, qrow, V, ua, ub, fp, fq, j, invz,
                                         unit_uniform(w.y), steps, max_steps, sh, C, rank, n_ex,
                                         ok, owner);
    if (!ok) { status = SPEC_ROW_TIMEOUT; timed_out = true; break; }
    // the owning CTA writes the drawn token; an all-zero distribution (not
    // reachable from a valid row) falls back to the row's argmax
    if (owner < 0) final_tok = sp.argmax;
    else if (owner == (int)rank && threadIdx.x == 0) out_tok[n_acc] = (t >= 0) ? t : sp.argmax;
    if (lead && threadIdx.x == 0 && job.counters) {
      atomicAdd(&job.counters[2], (unsigned long long)(j > 0 ? 2 : 1) * V * Elt<T>::kBytes);
      atomicAdd(&job.counters[4], 1ull);
    }
    break;
  }
  // timeouts of any CTA reach the lead CTA before the last cluster barrier, after
  // which no CTA touches another's shared memory
  if (threadIdx.x == 0 && timed_out) or_peer_u32(peer_addr(&sh.err, 0), 1u);
  cluster_sync_all();
  if (lead && threadIdx.x == 0) {
    if (status == SPEC_TREE_OK && sh.err) status = SPEC_ROW_TIMEOUT;
    finish_tree(job, b, status, n_acc, final_tok, owner < 0);
  }
}

__global__ void philox_words_kernel(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                                    const int32_t* node_idx, int32_t n, uint32_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 w = philox_words(seed, offset, b_idx[i], node_idx[i]);
  reinterpret_cast<uint4*>(out)[i] = w;
}

size_t tree_smem_bytes(int N) { return (size_t)((4 * N + 1 + 1) & ~1) * sizeof(int32_t); }

cudaError_t launch_greedy(const TreeJob& job, cudaStream_t s) {
  const size_t dyn = tree_smem_bytes(job.N);
  if (dyn > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        greedy_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
  }
  greedy_walk_kernel<<<job.B, GT, dyn, s>>>(job);
  return cudaGetLastError();
}

int floor_pow2(int x) {
  int p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}

// CTAs per tree: enough to give about four CTAs per SM over all trees, at most
// kMaxC, and at least two 256-thread rounds of units per CTA.
int cluster_size(int B, int V, int E) {
  const int units = (V + E - 1) / E;
  int C = floor_pow2(max(1, 4 * device_sm_count() / max(B, 1)));
  C = min(C, floor_pow2(max(1, units / (2 * CT))));
  return max(1, min(C, kMaxC));
}

template <typename T>
cudaError_t launch_sampling(const TreeJob& job, cudaStream_t s) {
  constexpr int E = Elt<T>::kPerUnit;
  const int C = cluster_size(job.B, job.V, E);
  const int units = (job.V + E - 1) / E;
  const int slice = (units + C - 1) / C;
  const int max_steps = max(1, ((slice + CW - 1) / CW + 31) / 32);
  const size_t dyn = tree_smem_bytes(job.N) + (size_t)job.N * (sizeof(double) + sizeof(float)) +
                     (size_t)CW * max_steps * sizeof(float);
  if (dyn > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        cluster_walk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)job.B * (unsigned)C);
  cfg.blockDim = dim3(CT);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, cluster_walk_kernel<T>, job, C, max_steps);
}

}  // namespace

cudaError_t launch_tree_walk(const TreeJob& job, spec_dtype dtype, bool greedy, cudaStream_t s) {
  if (greedy) return launch_greedy(job, s);
  if (dtype == SPEC_BF16) return launch_sampling<uint16_t>(job, s);
  return launch_sampling<float>(job, s);
}

cudaError_t launch_philox_words(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                                const int32_t* node_idx, int32_t n, uint32_t* out,
                                cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  philox_words_kernel<<<(n + 255) / 256, 256, 0, s>>>(seed, offset, b_idx, node_idx, n, out);
  return cudaGetLastError();
}

}  // namespace svk
