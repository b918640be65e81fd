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
#include "select.cuh"

namespace svk {

namespace {

constexpr int GT = kWalkThreads;          // greedy walk block
constexpr int CT = kClusterWalkThreads;   // sampling walk CTA
constexpr int CW = CT / 32;
constexpr int kMaxC = kMaxWalkCluster;
constexpr uint64_t kExchangeLimitNs = 2000000000ull;
constexpr int kSlotW = 16;     // 64-bit words one CTA can push in one exchange
constexpr int kCandCTA = 512;  // window candidates one CTA keeps per row
constexpr int kSortW = 2048;   // largest window (per row) the walk resolves by sorting
constexpr int kSortPer = kSortW / CT;
constexpr int kWalkBins = 1024;
constexpr int kWalkCtasPerSm = 2;  // resident sampling-walk CTAs per SM (register budget)
constexpr int kPreKids = 16;   // children whose accept-test inputs are prepared in parallel
static_assert(CT == kSelThreads, "the exact selection runs on one walk CTA");

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
  for (int u = threadIdx.x; u <= N; u += blockDim.x) cs[u] = 0;
  __syncthreads();
  int bad = 0;
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    if (n == 0) {
      bad |= (par[0] != -1);
    } else {
      bad |= (par[n] < 0 || par[n] >= n || tok[n] < 0 || tok[n] >= V);
    }
  }
  bad = __syncthreads_or(bad);
  if (!bad) {
    // depth of every node (its ancestor chain reaches the root within W - 1 steps) and
    // the number of children of every node
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
      int x = n, d = 0;
      while (x != 0 && d < W) { x = par[x]; ++d; }
      bad |= (x != 0 || d > W - 1);  // deeper than max_depth
      if (n > 0) atomicAdd(&cs[par[n] + 1], 1);
    }
  }
  bad = __syncthreads_or(bad);
  if (!bad) {
    // child-list offsets: inclusive scan of the counts (one warp)
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const int per = (N + 1 + 31) / 32;
      const int lo = min(N + 1, lane * per), hi = min(N + 1, lo + per);
      int run = 0;
      for (int i = lo; i < hi; ++i) { run += cs[i]; cs[i] = run; }
      int incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      const int base = incl - run;
      for (int i = lo; i < hi; ++i) cs[i] += base;
    }
    __syncthreads();
    // node n goes after its earlier siblings, so every list is in increasing node order
    for (int n = threadIdx.x + 1; n < N; n += blockDim.x) {
      const int u = par[n];
      int before = 0;
      for (int m = u + 1; m < n; ++m) before += (par[m] == u);
      cl[cs[u] + before] = n;
    }
  }
  if (threadIdx.x == 0) *s_status = bad ? SPEC_TREE_INVALID : SPEC_TREE_OK;
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
// Argmax of one row by the whole block (visited-rows-only schedule): the lowest index
// of the maximum, and whether the row is not finite (NaN, +inf, or all -inf).
template <typename T>
__device__ void block_argmax(const void* row, int V, int& arg, int& status, float* red_m,
                             int* red_i) {
  constexpr int E = Elt<T>::kPerUnit;
  const int nunits = (V + E - 1) / E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float m = -CUDART_INF_F;
  int idx = INT_MAX, bad = 0;
  for (int u = threadIdx.x; u < nunits; u += blockDim.x) {
    float z[E];
    load_unit<T>(row, V, u, z);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      bad |= (z[e] != z[e]);
      if (z[e] > m) { m = z[e]; idx = u * E + e; }
    }
  }
  const float wm = warp_max(m);
  const int wi = warp_min_i(m == wm ? idx : INT_MAX);
  bad = __syncthreads_or(bad);
  if (lane == 0) { red_m[warp] = wm; red_i[warp] = wi; }
  __syncthreads();
  float bm = -CUDART_INF_F;
  int bi = INT_MAX;
  for (int q = 0; q < (int)(blockDim.x >> 5); ++q) bm = fmaxf(bm, red_m[q]);
  for (int q = 0; q < (int)(blockDim.x >> 5); ++q)
    if (red_m[q] == bm) bi = min(bi, red_i[q]);
  __syncthreads();
  arg = (bi == INT_MAX) ? 0 : bi;
  status = (bad || bm == CUDART_INF_F || bm == -CUDART_INF_F) ? SPEC_ROW_NONFINITE : SPEC_TREE_OK;
}

template <typename T>
__global__ void __launch_bounds__(GT) greedy_walk_kernel(TreeJob job) {
  __shared__ int s_status;
  __shared__ float red_m[GT / 32];
  __shared__ int red_i[GT / 32];
  extern __shared__ __align__(16) int32_t tsm[];
  const int b = blockIdx.x;
  const int N = job.N;
  int32_t *par = tsm, *tok = tsm + N, *cs = tsm + 2 * N, *cl = tsm + 3 * N + 1;
  int status = load_tree(job, b, par, tok, cs, cl, true, &s_status);
  int32_t* out_tok = job.out_tokens + (int64_t)b * job.W;
  int32_t* out_path = job.out_path + (int64_t)b * job.W;
  int u = 0, n_acc = 0, final_tok = -1;
  while (status == SPEC_TREE_OK) {
    int argmax, st;
    if (job.visited_only) {
      block_argmax<T>(row_at(job.base_p, job, b, u, Elt<T>::kBytes), job.V, argmax, st, red_m,
                      red_i);
      if (threadIdx.x == 0 && job.counters)
        atomicAdd(&job.counters[2], (unsigned long long)job.V * Elt<T>::kBytes);
    } else {
      const spec_row_stats sp = job.stats_p[(int64_t)b * N + u];
      argmax = sp.argmax;
      st = sp.status;
    }
    if (st != SPEC_TREE_OK) { status = st; break; }
    int next = -1;
    for (int i = cs[u]; i < cs[u + 1]; ++i) {
      const int ch = cl[i];
      const bool ok = tok[ch] == argmax;
      if (threadIdx.x == 0 && job.out_alpha) job.out_alpha[(int64_t)b * N + ch] = ok ? 1.f : 0.f;
      if (ok) { next = ch; break; }
    }
    if (next < 0) { final_tok = argmax; break; }
    if (threadIdx.x == 0) {
      out_tok[n_acc] = tok[next];
      out_path[n_acc + 1] = next;
    }
    ++n_acc;
    u = next;
  }
  if (threadIdx.x == 0) finish_tree(job, b, status, n_acc, final_tok, true);
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

// True when every token of the unit lies strictly below the cut value, so that none
// is kept and its filtered probabilities are all exactly 0 (NaN never counts as
// below).  With top-k / top-p most units of a row are skipped this way.
__device__ __forceinline__ bool unit_below(const uint4& raw, const RowF& f, uint16_t) {
  const __nv_bfloat162 m2 = __hmax2(__hmax2(as_bf2(raw.x), as_bf2(raw.y)),
                                    __hmax2(as_bf2(raw.z), as_bf2(raw.w)));
  return __hlt2_mask(m2, as_bf2(f.zc2)) == 0xffffffffu;
}
__device__ __forceinline__ bool unit_below(const uint4& raw, const RowF& f, float) {
  const float m = fmaxf(fmaxf(__uint_as_float(raw.x), __uint_as_float(raw.y)),
                        fmaxf(__uint_as_float(raw.z), __uint_as_float(raw.w)));
  return m < f.zc;
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
__device__ __forceinline__ float dist_from_raw(uint4 rp, uint4 rq, int u, const RowF& fp,
                                               const RowF& fq, int j, const float* invz,
                                               float (&val)[Elt<T>::kPerUnit]) {
  constexpr int E = Elt<T>::kPerUnit;
  if (unit_below(rp, fp, T())) {  // p (and so every residual of it) is 0 here
#pragma unroll
    for (int e = 0; e < E; ++e) val[e] = 0.f;
    return 0.f;
  }
  unit_probs<T>(rp, u * E, fp, val);
  if (j > 0) {
    float q[E];
    unit_probs<T>(rq, u * E, fq, q);
    residual_chain<E>(val, q, j, invz);
  }
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) s = __fadd_rn(s, val[e]);
  return s;
}

// Is the token x with order key k inside the kept set of a filtered row?
__device__ __forceinline__ bool kept_key(uint32_t k, int x, const spec_row_stats& st) {
  return k > st.cut_key || (k == st.cut_key && x <= st.cut_idx);
}

// Filtered probability of one token in fp64 (for the acceptance test).
template <typename T>
__device__ double prob64(const void* row, int x, const spec_row_stats& st, double T_) {
  const float z = Elt<T>::at(row, x);
  if (!kept_key(order_key(z), x, st)) return 0.0;
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
__device__ __forceinline__ void st_peer_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;\n" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_peer_u64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];\n" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
  return v;
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

// Slots for n items per lane from a shared counter, one atomic per warp (every lane
// of the warp calls it): the first of this lane's slots.
// Shared-memory add with no result (a reduction on a shared-window address).
__device__ __forceinline__ void red_add_shared(unsigned* p, unsigned v) {
  asm volatile("red.shared.add.u32 [%0], %1;\n" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// Bits e (0..7) of a unit's bf16 logits that are >= t, t a bf16 pair of one value:
// two logits per compare (for bf16 z and fp32 thr, z >= thr iff z >= thr rounded up
// to bf16; -0 and +0 compare equal, as their order keys do).
__device__ __forceinline__ uint32_t unit_ge_bits(const uint4& v, __nv_bfloat162 t) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t mk = __hge2_mask(as_bf2(w[q]), t);
    m |= ((mk & 1u) | ((mk >> 15) & 2u)) << (2 * q);
  }
  return m;
}
// Order key of element e (a runtime index, 0..7) of a unit of bf16 logits, selected
// from the packed words (no array indexed at run time).
__device__ __forceinline__ uint32_t unit_key(const uint4& v, int e) {
  const uint32_t w = (e & 4) ? ((e & 2) ? v.w : v.z) : ((e & 2) ? v.y : v.x);
  const uint32_t b = (e & 1) ? (w >> 16) : (w & 0xffffu);
  return order_key(__uint_as_float(b << 16));
}

__device__ __forceinline__ unsigned warp_reserve(unsigned* ctr, unsigned n) {
  const int lane = threadIdx.x & 31;
  unsigned incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned tot = __shfl_sync(kFull, incl, 31);
  unsigned base = 0;
  if (lane == 31 && tot) base = atomicAdd(ctr, tot);
  return __shfl_sync(kFull, base, 31) + incl - n;
}

typedef uint64_t SlotRow[kSlotW];

struct CShared {
  SlotRow slot[2][kMaxC];  // words pushed by every CTA, two alternating sets
  uint64_t xbar[2];        // one mbarrier per slot set, C arrivals per phase
  double wred[CW];
  double wtot[CW];
  double target;
  int accept, status, target_warp, final_tok;
  Samp smp;  // the tree's sampling parameters
  unsigned err;            // rank 0: timeouts reported by any CTA of the cluster
  float inv_sp, inv_sq;
  unsigned ncand[2];       // window candidates of this CTA's slice, per row
  int first;
  unsigned long long massk;
  unsigned long long cut_w[4];
  // bf16 window scan results, per row
  int sc_ok[2], sc_bin[2];
  unsigned sc_j[2], sc_kept[2], sc_ncut[2];
  unsigned long long sc_sf[2];
  unsigned mem_n[2];
  // accept-test inputs of the first kPreKids children of the current node: the
  // unnormalised fp64 weights of the drafted token under p and q, its order keys,
  // and its accept uniform
  double kid_e[2][kPreKids];
  uint32_t kid_k[2][kPreKids];
  double kid_u[kPreKids];
  int tie_idx[2];
  // visited-rows-only schedule: per-warp row statistics of the cluster's stats pass
  float st_m[2][CW];
  double st_s[2][CW];
  int st_arg[2][CW];
  int st_bad[2];
  SelShared sel;
  uint4* ring;      // the slice-streaming ring (dynamic shared memory)
  int ring_stages;  // its depth: 4, or 2 where shared memory is short
  unsigned kp_n;    // this CTA's kept tokens of p (kept-set mode)
  unsigned long long ured[CW];
  int kp_tok;
  // fp64 reciprocals (GB300's fp64 divide is slow: each is taken once): 1 / T of the
  // tree, 1 / s_f of the node's p and q rows
  double inv_td, inv_s64[2];
  // window-pass staging: the two stages' barriers, rounds staged so far
  uint64_t wbar[2];
  uint32_t win_g;
  // top-k route: per row, the list threshold (an order key) and the selection digits
  uint32_t tk_thr[2];
  int tk_d1[2];
  unsigned tk_above[2];
};

struct BSync {
  __device__ static void sync() { __syncthreads(); }
};

// Slice streaming: each thread copies its own units of one or two rows into its own
// slots of a shared-memory ring with cp.async (kRingUnits units of each row per stage,
// S stages in flight) and reads back only those slots, so no block barrier is needed
// and the copies in flight cost no registers.  body(u, valid, raw0, raw1) is called by
// every thread the same number of times (so a body may use warp collectives); with
// valid set it sees unit u of both rows (raw1 repeats raw0 when nrows is 1), every unit
// of [ua, ub) once, in increasing u per thread.
constexpr int kRingUnits = 2;
constexpr size_t ring_bytes(int stages) { return (size_t)stages * kRingUnits * 2 * CT * 16; }

template <typename T, int S, typename Body>
__device__ __forceinline__ void stream_slice_s(const void* const (&rows)[2], int nrows, int V,
                                               int ua, int ub, uint4* ring, Body&& body) {
  constexpr int E = Elt<T>::kPerUnit;
  const int span = CT * kRingUnits;
  const int niter = (ub - ua + span - 1) / span;  // the same for every thread
  auto slot = [&](int st, int k, int r) {
    return ring + ((st * kRingUnits + k) * 2 + r) * CT + threadIdx.x;
  };
  auto issue = [&](int it) {
    if (it < niter) {
      const int st = it % S;
#pragma unroll
      for (int k = 0; k < kRingUnits; ++k) {
        const int u = ua + (int)threadIdx.x + it * span + k * CT;
        if (u >= ub) continue;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (r >= nrows) break;
          if ((u + 1) * E <= V) cp_async16(slot(st, k, r), reinterpret_cast<const uint4*>(rows[r]) + u);
          else *slot(st, k, r) = load_raw<T>(rows[r], V, u);  // the partial last unit
        }
      }
    }
    cp_async_commit();  // every thread commits every group: the counts stay aligned
  };
#pragma unroll
  for (int it = 0; it < S - 1; ++it) issue(it);
  for (int it = 0; it < niter; ++it) {
    issue(it + S - 1);
    cp_async_wait<S - 1>();
    const int st = it % S;
#pragma unroll
    for (int k = 0; k < kRingUnits; ++k) {
      const int u = ua + (int)threadIdx.x + it * span + k * CT;
      const bool valid = u < ub;
      uint4 r0 = make_uint4(0u, 0u, 0u, 0u), r1 = r0;
      if (valid) {
        r0 = *slot(st, k, 0);
        r1 = nrows > 1 ? *slot(st, k, 1) : r0;
      }
      body(u, valid, r0, r1);
    }
  }
  cp_async_wait<0>();
}

template <typename T, typename Body>
__device__ __forceinline__ void stream_slice(const void* const (&rows)[2], int nrows, int V,
                                             int ua, int ub, const CShared& sh, Body&& body) {
  if (sh.ring_stages == 4) stream_slice_s<T, 4>(rows, nrows, V, ua, ub, sh.ring, body);
  else stream_slice_s<T, 2>(rows, nrows, V, ua, ub, sh.ring, body);
}

// Cluster exchange: every CTA pushes nv words (thread 0's v) into slot[set][rank]
// of every CTA and arrives on that CTA's mbarrier; once the local mbarrier
// completes, slot[set][c] holds CTA c's words in every CTA.  Returns the slot set,
// or nullptr (uniformly over the CTA) if the wait gave up.  Shared-memory writes
// a CTA made before the call are visible to the other CTAs after it.  A slot set
// is written again two exchanges later, which no CTA can start before every CTA
// has pushed the exchange in between -- after its threads read this one.
__device__ const SlotRow* cluster_share(const uint64_t* v, int nv, CShared& sh, int C,
                                        uint32_t rank, uint32_t& n_ex) {
  const int set = n_ex & 1;
  const uint32_t parity = (n_ex >> 1) & 1u;
  ++n_ex;
  __syncthreads();  // the CTA's earlier writes happen before the releasing arrives below
  if (threadIdx.x < 32) {
    // thread t pushes thread 0's words to CTA t (all targets at once)
    uint64_t w[kSlotW];
#pragma unroll
    for (int k = 0; k < kSlotW; ++k)
      w[k] = __shfl_sync(kFull, (threadIdx.x == 0 && k < nv) ? v[k] : 0ull, 0);
    if ((int)threadIdx.x < C) {
      const uint32_t t = threadIdx.x;
#pragma unroll
      for (int k = 0; k < kSlotW; ++k)
        if (k < nv) st_peer_u64(peer_addr(&sh.slot[set][rank][k], t), w[k]);
      arrive_peer(peer_addr(&sh.xbar[set], t));
    }
  }
  // one thread waits (a spinning CTA would take issue slots from the other tree on
  // its SM); the barrier then orders its acquire before every thread's reads
  bool got = true;
  if (threadIdx.x == 0) got = mbar_wait_cluster(&sh.xbar[set], parity, kExchangeLimitNs);
  const bool ok = __syncthreads_and(got);
  return ok ? sh.slot[set] : nullptr;
}

// Cluster-wide sum of one fp64 value per CTA (read from thread 0), added in rank
// order so that every CTA holds the same bits.
__device__ bool cluster_sum(double v, CShared& sh, int C, uint32_t rank, uint32_t& n_ex,
                            double& total, double* per_cta) {
  const uint64_t w = (uint64_t)__double_as_longlong(v);
  const SlotRow* sl = cluster_share(&w, 1, sh, C, rank, n_ex);
  if (!sl) return false;
  double t = 0.0;
  for (int c = 0; c < C; ++c) {
    const double x = __longlong_as_double((long long)sl[c][0]);
    if (per_cta) per_cta[c] = x;
    t += x;
  }
  total = t;
  return true;
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
                               const RowF& fp, const RowF& fq, int j, const float* invz,
                               const CShared& sh) {
  constexpr int E = Elt<T>::kPerUnit;
  FF acc;
  const void* const rows[2] = {prow, qrow};
  stream_slice<T>(rows, 2, V, ua, ub, sh, [&](int u, bool valid, const uint4& rp, const uint4& rq) {
    if (!valid || unit_below(rp, fp, T())) return;  // p is 0 on the unit: max(0, p - q) too
    float p[E], q[E];
    unit_probs<T>(rp, u * E, fp, p);
    unit_probs<T>(rq, u * E, fq, q);
    residual_chain<E>(p, q, j, invz);
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) part += fmaxf(0.f, __fsub_rn(p[e], q[e]));
    acc.add(part);
  });
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
  constexpr int kSteps = 4;  // 32-unit steps whose loads are issued before any is used
  for (int base_u = lo; base_u < hi; base_u += 32 * kSteps) {
    uint4 rp[kSteps], rq[kSteps];
#pragma unroll
    for (int h = 0; h < kSteps; ++h) {
      const int u = base_u + 32 * h + lane;
      if (u < hi) {
        rp[h] = load_raw<T>(prow, V, u);
        if (j > 0) rq[h] = load_raw<T>(qrow, V, u);
      }
    }
#pragma unroll
    for (int h = 0; h < kSteps; ++h) {
      if (base_u + 32 * h >= hi) break;
      const int u = base_u + 32 * h + lane;
      float val[E];
      const float s = (u < hi) ? dist_from_raw<T>(rp[h], rq[h], u, fp, fq, j, invz, val) : 0.f;
      const float it = warp_sum_f(s);
      if (lane == 0) st[ns] = it;
      wt.add(it);
      ++ns;
    }
  }
  if (lane == 0) sh.wtot[warp] = wt.value();
  __syncthreads();
  double v = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < CW; ++w) v += sh.wtot[w];
  double total;
  double cta_tot[kMaxC];
  ok = cluster_sum(v, sh, C, rank, n_ex, total, cta_tot);
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
      float s = 0.f;
      if (u < hi) {
        const uint4 rp = load_raw<T>(prow, V, u);
        const uint4 rq = (j > 0) ? load_raw<T>(qrow, V, u) : rp;
        s = dist_from_raw<T>(rp, rq, u, fp, fq, j, invz, val);
      }
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
// Top-k / top-p cut of the rows the walk visits ("LLM speculative decoding:
// EAGLE", jingming.pro, section 1 note: p and q are compared after the sampling
// transforms).  The row pass supplies each row's maximum m and full sum; here the
// cluster finds (cut key, cut index, kept count, filtered sum) exactly:
//   1. every CTA collects the tokens of its slice with logit >= m - delta_z (the
//      candidate window) as (order key << 32 | ~index), so that a descending
//      sort orders them by (logit desc, index asc);
//   2. the CTAs exchange their counts, every CTA gathers all candidates through
//      distributed shared memory, sorts them (bitonic, the same input in every
//      CTA) and scans their exact 42-bit fixed-point masses for the top-k and
//      top-p crossings;
//   3. when the window cannot decide the cut (too few candidates for top-k, too
//      little mass for top-p, or more candidates than fit), CTA 0 runs the exact
//      full-row selection and shares its result.
// Both routes give the same statistics the dense row pass computes for a row.
// ---------------------------------------------------------------------------
struct RowCut {
  uint32_t key;
  int idx;
  unsigned kept;
  uint64_t mass;  // fixed point, 2^-42
};

// Step 1 for up to two rows: candidates of units [ua, ub) go to cand[r][...];
// with bf16 rows also one count per key in hist[r][K16m[r] - key16].
template <typename T>
__device__ void window_collect(const void* const (&rows)[2], int nrows, int V, int ua, int ub,
                               const float (&thr)[2], uint64_t* const (&cand)[2],
                               unsigned* const (&hist)[2], const uint32_t (&k16m)[2],
                               CShared& sh) {
  constexpr int E = Elt<T>::kPerUnit;
  const int lane = threadIdx.x & 31;
  stream_slice<T>(rows, nrows, V, ua, ub, sh,
                  [&](int u, bool valid, const uint4& raw0, const uint4& raw1) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nrows) break;
      float z[E];
      Elt<T>::unpack(r ? raw1 : raw0, z);
      unsigned bits = 0u;  // window members of this lane's unit
      if (valid) {
#pragma unroll
        for (int e = 0; e < E; ++e) bits |= (unsigned)(z[e] >= thr[r]) << e;
      }
      if (!__any_sync(kFull, bits != 0u)) continue;
      // one list reservation per warp: offsets from a warp scan of the lanes' counts
      const unsigned mine = __popc(bits);
      unsigned incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned total = __shfl_sync(kFull, incl, 31);
      unsigned base = 0u;
      if (lane == 0) base = atomicAdd(&sh.ncand[r], total);
      base = __shfl_sync(kFull, base, 0) + incl - mine;
      // elements by compile-time index (a runtime index would put z in local memory)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (!((bits >> e) & 1u)) continue;
        const uint32_t k = order_key(z[e]);
        if (base < (unsigned)kCandCTA)
          cand[r][base] = ((uint64_t)k << 32) | (uint64_t)(~(uint32_t)(u * E + e));
        ++base;
        if (hist[r]) {
          const uint32_t bin = k16m[r] - (k >> 16);
          if (bin < (uint32_t)kWalkBins) red_add_shared(&hist[r][bin], 1u);
        }
      }
    }
  });
}

constexpr int kWinUnits = 4;  // units of each row per thread and round of a window pass

// Window-pass staging.  A bf16 window pass reads its slice of one or two rows in
// rounds of CT * kWinUnits whole units per row.  With a 64 KB streaming ring the
// rounds arrive by bulk copy in two 32 KB stages, thread 0 issuing each round two
// rounds ahead: one round is filtered while the next two are in flight (twice the
// bytes in flight of loads into registers).  Rounds are counted over the kernel
// (sh.win_g): round g uses stage g & 1 and completes that stage's barrier phase
// (g >> 1) & 1.
struct WinStage {
  const uint4* src[2];
  int nrows, ua, ubf, nfull;  // nfull: rounds of whole units
  uint32_t g0;
  bool on;
  __device__ uint4* slot(CShared& sh, int rd, int r) const {
    return sh.ring + ((size_t)((g0 + (uint32_t)rd) & 1u) * 2 + (size_t)r) * (CT * kWinUnits);
  }
  // thread 0: the bulk copies of round rd
  __device__ void issue(CShared& sh, int rd) const {
    const uint32_t st = (g0 + (uint32_t)rd) & 1u;
    const int base = ua + rd * CT * kWinUnits;
    const uint32_t bytes = (uint32_t)min(CT * kWinUnits, ubf - base) * 16u;
    mbar_arrive_expect_tx(&sh.wbar[st], bytes * (uint32_t)nrows);
    for (int r = 0; r < nrows; ++r) bulk_copy_g2s(slot(sh, rd, r), src[r] + base, bytes, &sh.wbar[st]);
  }
  __device__ bool wait(CShared& sh, int rd) const {
    const uint32_t g = g0 + (uint32_t)rd;
    return mbar_wait(&sh.wbar[g & 1u], (g >> 1) & 1u, kExchangeLimitNs);
  }
};

// Every thread: the staging of a pass over whole units [ua, ubf) of `nrows` rows;
// issues its first two rounds.
__device__ WinStage win_stage_begin(const void* const (&rows)[2], int nrows, int ua, int ubf,
                                    CShared& sh) {
  WinStage w;
  w.src[0] = reinterpret_cast<const uint4*>(rows[0]);
  w.src[1] = reinterpret_cast<const uint4*>(nrows > 1 ? rows[1] : rows[0]);
  w.nrows = nrows;
  w.ua = ua;
  w.ubf = ubf;
  w.nfull = ubf > ua ? (ubf - ua + CT * kWinUnits - 1) / (CT * kWinUnits) : 0;
  w.on = sh.ring_stages == 4 && w.nfull > 0;
  w.g0 = sh.win_g;
  if (w.on) {
    // the ring's earlier contents were written and read through the generic proxy
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
      w.issue(sh, 0);
      if (w.nfull > 1) w.issue(sh, 1);
    }
  }
  return w;
}

// Every thread, after the pass (or when a stage's wait gave up at round `stop`):
// the rounds staged so far are recorded; after a failed wait thread 0 first waits,
// bounded, for the copies still in flight.
__device__ void win_stage_end(const WinStage& w, CShared& sh, int stop) {
  if (!w.on) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (stop < w.nfull)
      for (int rd = stop; rd < min(w.nfull, stop + 2); ++rd) w.wait(sh, rd);
    sh.win_g = w.g0 + (uint32_t)w.nfull;
  }
  __syncthreads();
}

// bf16 rows, the window pass: units [ua, ub) of one or two rows are read with
// vector loads straight into registers, kWinUnits units of each row per thread in
// flight (a CTA's slice in a few rounds); a unit is unpacked only when its packed
// bf16 maximum reaches the window threshold.  Tokens z >= thr[r] go to cand[r] (slots
// reserved once per warp and round; sh.ncand[r] counts all of them, cand[r] keeps
// the first kCandCTA) and are counted per key in hist[r] (when not null).

__device__ bool window_collect_fast(const void* const (&rows)[2], int nrows, int V, int ua,
                                    int ub, const float (&thr)[2], uint64_t* const (&cand)[2],
                                    unsigned* const (&hist)[2], const uint32_t (&k16m)[2],
                                    CShared& sh) {
  const int full = V / 8;  // units wholly inside the row
  const int ubf = min(ub, full);
  const uint4* const r0 = reinterpret_cast<const uint4*>(rows[0]);
  const uint4* const r1 = reinterpret_cast<const uint4*>(nrows > 1 ? rows[1] : rows[0]);
  const WinStage stg = win_stage_begin(rows, nrows, ua, ubf, sh);
  int stop = INT_MAX;
  const __nv_bfloat162 t2[2] = {__bfloat162bfloat162(__float2bfloat16_ru(thr[0])),
                                __bfloat162bfloat162(__float2bfloat16_ru(thr[1]))};
  // the rounds cover the whole units; the partial last unit (if this slice has it) is
  // one more round of its own, read with element loads
  const int nround = (ubf > ua ? (ubf - ua + CT * kWinUnits - 1) / (CT * kWinUnits) : 0) +
                     (ub > full ? 1 : 0);
  for (int rd = 0; rd < nround; ++rd) {  // the same rounds in every thread
    const bool tail = ub > full && rd == nround - 1;
    const int base = tail ? full : ua + rd * CT * kWinUnits;
    uint4 raw[2][kWinUnits];
    if (!tail && stg.on) {
      // this round's stage (bounded wait; every thread gives up together)
      if (!__syncthreads_and(stg.wait(sh, rd))) { stop = rd; break; }
      const uint4* s0 = stg.slot(sh, rd, 0);
      const uint4* s1 = stg.slot(sh, rd, 1);
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h) {
        const int u = base + h * CT + (int)threadIdx.x;
        const bool in = u < ubf;
        raw[0][h] = in ? s0[h * CT + threadIdx.x]
                       : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
        raw[1][h] = (in && nrows > 1)
                        ? s1[h * CT + threadIdx.x]
                        : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
      }
      // every thread has read the stage: it takes round rd + 2
      __syncthreads();
      if (threadIdx.x == 0 && rd + 2 < stg.nfull) {
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        stg.issue(sh, rd + 2);
      }
    } else if (!tail) {
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h) {
        const int u = base + h * CT + (int)threadIdx.x;
        const bool in = u < ubf;
        raw[0][h] = in ? __ldg(r0 + u)
                       : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
        raw[1][h] = (in && nrows > 1)
                        ? __ldg(r1 + u)
                        : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
      }
    } else {
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          raw[r][h] = (h == 0 && threadIdx.x == 0 && r < nrows)
                          ? load_raw<uint16_t>(rows[r], V, full)
                          : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
    }
    uint32_t mb[2][kWinUnits];
    unsigned cnt[2] = {0u, 0u};
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h) {
        const uint32_t m = unit_ge_bits(raw[r][h], t2[r]);
        mb[r][h] = m;
        cnt[r] += __popc(m);
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!cnt[r]) continue;
      // one shared atomic per lane with members (their order in the list is free: every
      // reader of a list treats it as a set)
      unsigned pos = atomicAdd(&sh.ncand[r], cnt[r]);
      // the lane's members over all its units in one loop (bit 8 h + e), so the warp
      // iterates as often as its busiest lane has members, not once per unit
      static_assert(kWinUnits * 8 <= 32, "a lane's window bits fit one word");
      uint32_t bits = 0u;
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h) bits |= mb[r][h] << (8 * h);
      while (bits) {
        const int t = __ffs(bits) - 1;
        bits &= bits - 1u;
        const int h = t >> 3, e = t & 7;
        const uint4 v = h == 0 ? raw[r][0] : h == 1 ? raw[r][1] : h == 2 ? raw[r][2] : raw[r][3];
        const int u = tail ? full : base + h * CT + (int)threadIdx.x;
        const uint32_t k = unit_key(v, e);
        if (pos < (unsigned)kCandCTA) {
          cand[r][pos] = ((uint64_t)k << 32) | (uint64_t)(~(uint32_t)(u * 8 + e));
        } else if (hist[r]) {
          // a member past the list is counted here; listed ones after the pass
          const uint32_t bin = k16m[r] - (k >> 16);
          if (bin < (uint32_t)kWalkBins) red_add_shared(&hist[r][bin], 1u);
        }
        ++pos;
      }
    }
  }
  win_stage_end(stg, sh, stop);  // ends with a barrier: the lists are complete
  if (stop != INT_MAX) return false;
  // the listed members' key counts, every thread over its share of the lists
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows || !hist[r]) continue;
    const unsigned n = min(sh.ncand[r], (unsigned)kCandCTA);
    for (unsigned i = threadIdx.x; i < n; i += CT) {
      const uint32_t bin = k16m[r] - (uint32_t)(cand[r][i] >> 48);
      if (bin < (uint32_t)kWalkBins) red_add_shared(&hist[r][bin], 1u);
    }
  }
  return true;
}

// Step 2 after the sort: the cut from n sorted candidates (descending, padded to
// n_pad with zeros), or false when the window cannot decide it.  Same rule as the
// dense row pass's sorted window.
__device__ bool window_cut(const uint64_t* keys, unsigned n, unsigned n_pad, float m, float c,
                           double s_all, const Samp& smp, CShared& sh, RowCut& out) {
  const bool topk_on = smp.top_k > 0, topp_on = smp.top_p < 1.0f;
  const unsigned K = topk_on ? (unsigned)smp.top_k : n;
  const int lane = threadIdx.x & 31;
  const unsigned lo = threadIdx.x * (unsigned)kSortPer;
  if (threadIdx.x == 0) sh.first = INT_MAX;
  unsigned long long pre[kSortPer];
  unsigned long long run = 0;
#pragma unroll
  for (int t = 0; t < kSortPer; ++t) {
    const unsigned i = lo + t;
    if (i < n) run += to_fixed(tempered_weight(key_value((uint32_t)(keys[i] >> 32)), m, c));
    pre[t] = run;
  }
  unsigned bc, tc;
  unsigned long long bw, tw;
  block_exscan<BSync>(0u, run, bc, bw, tc, tw, sh.sel);
#pragma unroll
  for (int t = 0; t < kSortPer; ++t) pre[t] += bw;
  unsigned cut_pos = K - 1;
  if (topp_on) {
    if (topk_on && K - 1 >= lo && K - 1 < lo + kSortPer) {
#pragma unroll
      for (int t = 0; t < kSortPer; ++t)
        if (lo + t == K - 1) sh.massk = pre[t];
    }
    __syncthreads();
    const unsigned long long tau = (unsigned long long)ceil(
        (double)smp.top_p * (topk_on ? (double)sh.massk : s_all * 4398046511104.0));
    int fj = INT_MAX;
#pragma unroll
    for (int t = 0; t < kSortPer; ++t) {
      const unsigned i = lo + t;
      if (fj == INT_MAX && i < K && pre[t] >= tau) fj = (int)i;
    }
    fj = warp_min_i(fj);
    if (lane == 0 && fj != INT_MAX) atomicMin(&sh.first, fj);
    __syncthreads();
    if (sh.first == INT_MAX) return false;  // the window holds too little mass
    cut_pos = (unsigned)sh.first;
  }
  if (cut_pos >= lo && cut_pos < lo + kSortPer) {
#pragma unroll
    for (int t = 0; t < kSortPer; ++t)
      if (lo + t == cut_pos) {
        sh.cut_w[0] = keys[cut_pos];
        sh.cut_w[1] = pre[t];
      }
  }
  __syncthreads();
  out.key = (uint32_t)(sh.cut_w[0] >> 32);
  out.idx = (int)(~(uint32_t)sh.cut_w[0]);
  out.kept = cut_pos + 1;
  out.mass = sh.cut_w[1];
  __syncthreads();
  return true;
}


__device__ __forceinline__ void set_cut(spec_row_stats& s, const RowCut& rc) {
  s.cut_key = rc.key;
  s.cut_idx = rc.idx;
  s.kept = (int)rc.kept;
  s.s_f = fixed_to_double(rc.mass);
}

// The exact selection's combination step over a cluster: every CTA tallies its own
// slice and the tallies are exchanged and summed in rank order (integers: the same
// totals everywhere).  `ok` drops when an exchange gives up.
struct ClusterReduce {
  CShared* sh;
  int C;
  uint32_t rank;
  uint32_t* n_ex;
  bool ok;
  __device__ void tally(SelShared& s) {
    uint64_t w[2 * kSplit + 1];
    for (int t = 0; t < kSplit; ++t) {
      w[t] = s.red_cnt[t];
      w[kSplit + t] = s.red_mass[t];
    }
    w[2 * kSplit] = s.red_min;
    const SlotRow* sl = cluster_share(w, 2 * kSplit + 1, *sh, C, rank, *n_ex);
    if (!sl) {
      ok = false;
      return;
    }
    unsigned cnt[kSplit];
    unsigned long long mass[kSplit];
    unsigned mn = 0xffffffffu;
    for (int t = 0; t < kSplit; ++t) { cnt[t] = 0u; mass[t] = 0ull; }
    for (int q = 0; q < C; ++q) {
      for (int t = 0; t < kSplit; ++t) {
        cnt[t] += (unsigned)sl[q][t];
        mass[t] += sl[q][kSplit + t];
      }
      mn = min(mn, (unsigned)sl[q][2 * kSplit]);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int t = 0; t < kSplit; ++t) { s.red_cnt[t] = cnt[t]; s.red_mass[t] = mass[t]; }
      s.red_min = mn;
    }
    __syncthreads();
  }
  __device__ void base(unsigned mine, unsigned& b, unsigned& total) {
    const uint64_t w = mine;
    const SlotRow* sl = cluster_share(&w, 1, *sh, C, rank, *n_ex);
    b = 0u;
    total = mine;
    if (!sl) {
      ok = false;
      return;
    }
    total = 0u;
    for (int q = 0; q < C; ++q) {
      if (q < (int)rank) b += (unsigned)sl[q][0];
      total += (unsigned)sl[q][0];
    }
  }
  __device__ int max_int(int v) {
    const uint64_t w = (uint64_t)(uint32_t)(v + 1);  // -1 (not found here) -> 0
    const SlotRow* sl = cluster_share(&w, 1, *sh, C, rank, *n_ex);
    if (!sl) {
      ok = false;
      return v;
    }
    int mx = 0;
    for (int q = 0; q < C; ++q) mx = max(mx, (int)(uint32_t)sl[q][0]);
    return mx - 1;
  }
};

// The exact selection of one row by the whole cluster (each CTA over its slice of
// units [ua, ub)): the dense row pass's rule, the same result.
template <typename T>
__device__ bool cluster_exact_cut(const TreeJob& job, const void* row, const spec_row_stats& s,
                                  int ua, int ub, CShared& sh, int C, uint32_t rank,
                                  uint32_t& n_ex, const Samp& smp, RowCut& out) {
  const float c = smp.c;
  const bool topk_on = smp.top_k > 0, topp_on = smp.top_p < 1.0f;
  const int V = job.V;
  ClusterReduce red{&sh, C, rank, &n_ex, true};
  SelOut rk{};
  const Eligible all{false, 0u, 0};
  if (topk_on)
    rk = exact_select<T, BSync>(row, V, s.m, c, false, (unsigned)smp.top_k, 0ull, all, sh.sel,
                                ua, ub, red);
  if (topp_on) {
    const Eligible in_k{topk_on, rk.key, rk.idx};
    const unsigned long long tau = (unsigned long long)ceil(
        (double)smp.top_p * (topk_on ? (double)rk.mass_kept : s.s_f * 4398046511104.0));
    const SelOut rp = exact_select<T, BSync>(row, V, s.m, c, true, 0u, tau, in_k, sh.sel, ua,
                                             ub, red);
    out.key = rp.key; out.idx = rp.idx; out.kept = rp.kept; out.mass = rp.mass_kept;
  } else {
    out.key = rk.key; out.idx = rk.idx; out.kept = rk.kept; out.mass = rk.mass_kept;
  }
  if (rank == 0 && threadIdx.x == 0 && job.counters) atomicAdd(&job.counters[5], 1ull);
  return red.ok;
}

// The cut of the p row (and of the q row when with_q) of node u, written into the
// statistics every CTA holds (rows of any dtype: gathered window, sorted).  `cand` holds this node's two candidate lists (the
// caller alternates between two sets from node to node, so a list is rewritten
// only after an exchange that every CTA reaches after reading it); `sortb` the two
// sort buffers.  Returns false if an exchange gave up.
template <typename T>
__device__ bool cluster_cut_sorted(const TreeJob& job, const void* prow, const void* qrow,
                                   bool with_q, spec_row_stats& sp, spec_row_stats& sq, int ua,
                                   int ub, uint64_t* cand, uint64_t* sortb, CShared& sh, int C,
                                   uint32_t rank, uint32_t& n_ex, const Samp& smp) {
  const float c = smp.c;
  const int V = job.V;
  const int nrows = with_q ? 2 : 1;
  spec_row_stats* st[2] = {&sp, &sq};
  const void* const rows[2] = {prow, qrow};
  const float thr[2] = {sp.m - smp.delta_z, sq.m - smp.delta_z};
  uint64_t* const cl[2] = {cand, cand + kCandCTA};
  unsigned* const no_hist[2] = {nullptr, nullptr};
  const uint32_t no_k16[2] = {0u, 0u};
  if (threadIdx.x == 0) { sh.ncand[0] = 0u; sh.ncand[1] = 0u; }
  __syncthreads();
  if (!job.exact) window_collect<T>(rows, nrows, V, ua, ub, thr, cl, no_hist, no_k16, sh);
  __syncthreads();
  const uint64_t counts = (uint64_t)sh.ncand[0] | ((uint64_t)sh.ncand[1] << 32);
  const SlotRow* sl = cluster_share(&counts, 1, sh, C, rank, n_ex);
  if (!sl) return false;
  unsigned cnt[2][kMaxC], total[2] = {0u, 0u}, n_pad[2] = {2u, 2u};
  bool fast[2] = {false, false};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    bool over = false;
    for (int q = 0; q < C; ++q) {
      cnt[r][q] = (unsigned)(sl[q][0] >> (32 * r));
      over |= cnt[r][q] > (unsigned)kCandCTA;
      total[r] += min(cnt[r][q], (unsigned)kCandCTA);
    }
    const bool topk_on = smp.top_k > 0;
    fast[r] = !job.exact && !over && total[r] >= 1u && total[r] <= (unsigned)kSortW &&
              (!topk_on || total[r] >= (unsigned)smp.top_k);
    while (n_pad[r] < total[r]) n_pad[r] <<= 1;
  }
  // gather every CTA's candidates (remote shared memory) into the sort buffers
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    if (!fast[r]) continue;
    uint64_t* keys = sortb + r * kSortW;
    for (unsigned i = threadIdx.x; i < n_pad[r]; i += CT) {
      uint64_t v = 0ull;
      if (i < total[r]) {
        unsigned off = 0, q = 0;
        while (q + 1 < (unsigned)C && i >= off + cnt[r][q]) { off += cnt[r][q]; ++q; }
        unsigned li = i - off;
        SPEC_CHECK_INDEX(li, kCandCTA, 0);
        SPEC_CHECK_INDEX(q, C, 0);
        v = ld_peer_u64(peer_addr(cl[r] + li, q));
      }
      unsigned ki = i;
      SPEC_CHECK_INDEX(ki, kSortW, 1);
      keys[ki] = v;
    }
  }
  __syncthreads();
  const unsigned pad_max = max(fast[0] ? n_pad[0] : 0u, fast[1] ? n_pad[1] : 0u);
  for (unsigned k = 2; k <= pad_max; k <<= 1) {  // bitonic sort, descending
    for (unsigned jj = k >> 1; jj > 0; jj >>= 1) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r >= nrows) break;
        if (!fast[r] || k > n_pad[r]) continue;
        uint64_t* keys = sortb + r * kSortW;
        for (unsigned i = threadIdx.x; i < n_pad[r]; i += CT) {
          const unsigned ixj = i ^ jj;
          if (ixj > i) {
            const uint64_t a = keys[i], b = keys[ixj];
            const bool swap = ((i & k) == 0) ? (a < b) : (a > b);
            if (swap) { keys[i] = b; keys[ixj] = a; }
          }
        }
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    spec_row_stats& s = *st[r];
    RowCut rc{};
    bool ok = fast[r] && window_cut(sortb + r * kSortW, total[r], n_pad[r], s.m, c, s.s_f, smp,
                                    sh, rc);
    if (!ok && !cluster_exact_cut<T>(job, rows[r], s, ua, ub, sh, C, rank, n_ex, smp, rc))
      return false;
    set_cut(s, rc);
  }
  return true;
}


// bf16 rows: the window's cut from the cluster's merged counts per 16-bit key
// (bin = K16m - key) and the keys' fixed-point weights (wbin, filled beforehand),
// scanned by one warp with the dense row pass's crossing rules (top-k count, then
// the top-p mass target over exact fixed-point weights).
// Results in sh.sc_*[r]; sh.sc_ok[r] = 0 when the window cannot decide the cut.
__device__ void bf16_window_scan(const unsigned* hist, unsigned long long* wbin, int nb,
                                 uint32_t K16m, float m, float c, double s_all,
                                 const Samp& smp, CShared& sh, int r) {
  const int lane = threadIdx.x & 31;
  const bool topk_on = smp.top_k > 0, topp_on = smp.top_p < 1.0f;
  const unsigned K = topk_on ? (unsigned)smp.top_k : 0u;
  const int Cb = (nb + 31) / 32;
  const int b_lo = min(nb, lane * Cb), b_hi = min(nb, b_lo + Cb);
  unsigned lc = 0;
  unsigned long long lw = 0;
  for (int bin = b_lo; bin < b_hi; ++bin) {
    const unsigned long long wgt = wbin[bin];  // filled with the merge, every thread a bin
    lc += hist[bin];
    lw += (unsigned long long)hist[bin] * wgt;
  }
  __syncwarp();
  unsigned ic = lc;
  unsigned long long iw = lw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned tc = __shfl_up_sync(kFull, ic, o);
    const unsigned long long tw = __shfl_up_sync(kFull, iw, o);
    if (lane >= o) { ic += tc; iw += tw; }
  }
  const unsigned base_c = ic - lc, tot_c = __shfl_sync(kFull, ic, 31);
  const unsigned long long base_w = iw - lw;
  int ok = 1;
  int b_k = nb;  // no top-k: past the last bin
  unsigned jk = 0;
  unsigned long long s_k = 0;
  int bcut = 0;
  unsigned j = 0, kept = 0;
  unsigned long long sf = 0;
  if (topk_on) {
    if (tot_c < K) {
      ok = 0;
    } else {
      int hitbin = INT_MAX;
      unsigned rc = base_c;
      for (int bin = b_lo; bin < b_hi; ++bin) {
        if (rc + hist[bin] >= K) { hitbin = bin; break; }
        rc += hist[bin];
      }
      b_k = warp_min_i(hitbin);
      if (b_k >= nb) b_k = 0;  // cannot happen when tot_c >= K; keeps indices in range
      const int owner = __ffs(__ballot_sync(kFull, hitbin == b_k)) - 1;
      unsigned long long rw = base_w;
      unsigned rc2 = base_c;
      if (lane == owner)
        for (int bin = b_lo; bin < min(b_k, b_hi); ++bin) {
          rc2 += hist[bin];
          rw += (unsigned long long)hist[bin] * wbin[bin];
        }
      rc2 = __shfl_sync(kFull, rc2, owner);
      rw = __shfl_sync(kFull, rw, owner);
      jk = K - rc2;
      s_k = rw + (unsigned long long)jk * wbin[b_k];
      bcut = b_k; j = jk; kept = K; sf = s_k;
    }
  }
  if (ok && topp_on) {
    const unsigned long long tau = (unsigned long long)ceil(
        (double)smp.top_p * (topk_on ? (double)s_k : s_all * 4398046511104.0));
    int hitbin = INT_MAX;
    unsigned long long rw = base_w;
    for (int bin = b_lo; bin < b_hi && bin <= b_k; ++bin) {
      const unsigned cnt = (bin == b_k) ? jk : hist[bin];
      const unsigned long long wsum = (unsigned long long)cnt * wbin[bin];
      if (cnt && rw + wsum >= tau) { hitbin = bin; break; }
      rw += wsum;
    }
    const int b_p = warp_min_i(hitbin);
    if (b_p == INT_MAX) {
      ok = 0;  // the window holds too little mass
    } else {
      const int owner = __ffs(__ballot_sync(kFull, hitbin == b_p)) - 1;
      unsigned rc = base_c;
      unsigned long long rw2 = base_w;
      if (lane == owner)
        for (int bin = b_lo; bin < min(b_p, b_hi); ++bin) {
          rc += hist[bin];
          rw2 += (unsigned long long)hist[bin] * wbin[bin];
        }
      rc = __shfl_sync(kFull, rc, owner);
      rw2 = __shfl_sync(kFull, rw2, owner);
      const unsigned avail = (b_p == b_k) ? jk : hist[b_p];
      const unsigned long long w1 = wbin[b_p];
      unsigned jj2 = avail;
      if (w1 > 0) {
        const unsigned long long jj = (tau - rw2 + w1 - 1) / w1;
        jj2 = (unsigned)(jj < 1 ? 1 : (jj > avail ? avail : jj));
      }
      bcut = b_p; j = jj2; kept = rc + jj2; sf = rw2 + (unsigned long long)jj2 * w1;
    }
  }
  if (lane == 0) {
    sh.sc_ok[r] = ok;
    sh.sc_bin[r] = bcut;
    sh.sc_j[r] = j;
    sh.sc_kept[r] = kept;
    sh.sc_sf[r] = sf;
    sh.sc_ncut[r] = ok ? hist[bcut] : 0u;
  }
}

// Layout of the bf16 cut's buffers in `smem`: the per-CTA key counts of both rows
// [2][kWalkBins], the merged counts [2][kWalkBins], the bin weights [2][kWalkBins]
// (u64), then the CTA's lists of window tokens [2][kCandCTA] (u64 words).
__device__ __forceinline__ uint64_t* bf16_cand_list(unsigned char* smem, int r) {
  unsigned long long* wbin = reinterpret_cast<unsigned long long*>(
      reinterpret_cast<unsigned*>(smem) + 4 * kWalkBins);
  return reinterpret_cast<uint64_t*>(wbin + 2 * kWalkBins) + (size_t)r * kCandCTA;
}

// bf16 rows: the cut of the p row (and of the q row when with_q) of node u, from
// per-CTA key histograms merged through distributed shared memory; the cut key's
// ties are resolved by index from the CTAs' own candidate lists.  A histogram is
// read by the other CTAs only between the count exchange and the tie exchange.
__device__ bool cluster_cut_bf16(const TreeJob& job, const void* prow, const void* qrow,
                                 bool with_q, spec_row_stats& sp, spec_row_stats& sq, int ua,
                                 int ub, unsigned char* smem, CShared& sh, int C, uint32_t rank,
                                 uint32_t& n_ex, const Samp& smp, bool& p_listed) {
  p_listed = false;
  const float c = smp.c;
  const int V = job.V;
  const int nrows = with_q ? 2 : 1;
  spec_row_stats* st[2] = {&sp, &sq};
  const void* const rows[2] = {prow, qrow};
  unsigned* hist[2] = {reinterpret_cast<unsigned*>(smem),
                       reinterpret_cast<unsigned*>(smem) + kWalkBins};
  unsigned* merged[2] = {hist[1] + kWalkBins, hist[1] + 2 * kWalkBins};
  unsigned long long* wbin[2] = {reinterpret_cast<unsigned long long*>(merged[1] + kWalkBins),
                                 reinterpret_cast<unsigned long long*>(merged[1] + kWalkBins) +
                                     kWalkBins};
  uint64_t* const cl[2] = {bf16_cand_list(smem, 0), bf16_cand_list(smem, 1)};
  float thr[2];
  uint32_t k16m[2];
  int nb[2];
  bool fits[2];
  unsigned* hp[2] = {nullptr, nullptr};
  for (int r = 0; r < 2; ++r) {
    thr[r] = st[r]->m - smp.delta_z;
    k16m[r] = order_key(st[r]->m) >> 16;
    uint32_t k16t = order_key(thr[r]) >> 16;  // lowest key the window can hold
    if (k16m[r] - k16t >= (uint32_t)kWalkBins) {
      // clip the window to the kWalkBins keys below the maximum; the scan checks that
      // it still holds the cut (else the exact selection decides)
      k16t = k16m[r] - (uint32_t)(kWalkBins - 1);
      thr[r] = key_value(key_from16(k16t));
    }
    fits[r] = r < nrows;
    nb[r] = fits[r] ? (int)(k16m[r] - k16t) + 1 : 0;
    if (fits[r]) hp[r] = hist[r];
    for (int i = threadIdx.x; i < nb[r]; i += CT) hist[r][i] = 0u;
  }
  if (threadIdx.x == 0) { sh.ncand[0] = 0u; sh.ncand[1] = 0u; }
  __syncthreads();
  if (!job.exact && !window_collect_fast(rows, nrows, V, ua, ub, thr, cl, hp, k16m, sh))
    return false;
  __syncthreads();
  const unsigned own_n[2] = {min(sh.ncand[0], (unsigned)kCandCTA), min(sh.ncand[1], (unsigned)kCandCTA)};
  // a CTA whose list overflowed finds the cut key's members by a pass over its slice
  const bool own_over[2] = {sh.ncand[0] > (unsigned)kCandCTA, sh.ncand[1] > (unsigned)kCandCTA};
  const uint64_t counts = (uint64_t)sh.ncand[0] | ((uint64_t)sh.ncand[1] << 32);
  const SlotRow* sl = cluster_share(&counts, 1, sh, C, rank, n_ex);
  if (!sl) return false;
  // every CTA's list of p's window tokens is complete (no CTA overflowed)
  bool p_all_listed = !job.exact;
  for (int q = 0; q < C; ++q) p_all_listed &= (unsigned)sl[q][0] <= (unsigned)kCandCTA;
  bool win[2] = {false, false};
#pragma unroll
  for (int r = 0; r < 2; ++r)
    if (r < nrows) win[r] = !job.exact && fits[r];
  // merge the key counts of every CTA (same order, integer sums: identical everywhere)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    if (!win[r]) continue;
    for (int i = threadIdx.x; i < nb[r]; i += CT) {
      // every peer's count is requested before any is added (the loads overlap)
      unsigned v[kMaxC];
#pragma unroll
      for (int q = 0; q < kMaxC; ++q) v[q] = q < C ? ld_peer_u32(peer_addr(hist[r] + i, q)) : 0u;
      unsigned t = 0;
#pragma unroll
      for (int q = 0; q < kMaxC; ++q) t += v[q];
      merged[r][i] = t;
      // the key's weight, for the scan (every thread its bins, not one warp all)
      wbin[r][i] = to_fixed(tempered_weight(key_value(key_from16(k16m[r] - (uint32_t)i)),
                                            st[r]->m, c));
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if (warp < nrows) {
    if (win[warp])
      bf16_window_scan(merged[warp], wbin[warp], nb[warp], k16m[warp], st[warp]->m, c,
                       st[warp]->s_f, smp, sh, warp);
    else if ((threadIdx.x & 31) == 0)
      sh.sc_ok[warp] = 0;
  }
  __syncthreads();
  bool ok[2] = {false, false};
#pragma unroll
  for (int r = 0; r < 2; ++r)
    if (r < nrows) ok[r] = sh.sc_ok[r] != 0;
  uint32_t cut32[2] = {0u, 0u};
  if (ok[0] || ok[1]) {
    // Each CTA's number of members of the cut key is its own count of that key, read
    // from its histogram through distributed shared memory (every histogram stays as
    // it is until all CTAs have passed the exchange below).  The cut index is the
    // largest member when the whole group is kept, else the j-th member in index
    // order; either way one CTA (the owner) holds it.
    int owner[2] = {-1, -1};
    unsigned jr[2] = {0u, 0u};
    bool want_max[2] = {false, false};
    int cut_idx[2] = {0, 0};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nrows) break;
      if (!ok[r]) continue;
      cut32[r] = key_from16(k16m[r] - (uint32_t)sh.sc_bin[r]);
      unsigned cnt[kMaxC];
#pragma unroll
      for (int q = 0; q < kMaxC; ++q)
        cnt[q] = q < C ? ld_peer_u32(peer_addr(hist[r] + sh.sc_bin[r], q)) : 0u;
      if (sh.sc_j[r] == sh.sc_ncut[r]) {
        want_max[r] = true;
#pragma unroll
        for (int q = 0; q < kMaxC; ++q)
          if (q < C && cnt[q]) owner[r] = q;  // the last CTA with a member
      } else {
        unsigned before = 0;
#pragma unroll
        for (int q = 0; q < kMaxC; ++q) {
          if (q < C && owner[r] < 0 && before + cnt[q] >= sh.sc_j[r]) {
            owner[r] = q;
            jr[r] = sh.sc_j[r] - before;
          }
          before += cnt[q];
        }
      }
    }
    const bool need = owner[0] >= 0 || owner[1] >= 0;
    if (need) {
      // the merged counts are no longer needed and hold the owner's member indices
      if (threadIdx.x < 2) { sh.mem_n[threadIdx.x] = 0u; sh.tie_idx[threadIdx.x] = -1; }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r >= nrows) break;
        if (owner[r] != (int)rank) continue;
        // gather this CTA's members of the cut key (at most kWalkBins of them;
        // more leaves the row to the exact selection)
        if (own_over[r]) {
          for (int u = ua + threadIdx.x; u < ub; u += CT) {
            float z[8];
            Elt<uint16_t>::unpack(load_raw<uint16_t>(rows[r], V, u), z);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (order_key(z[e]) == cut32[r]) {
                const unsigned pos = atomicAdd(&sh.mem_n[r], 1u);
                if (pos < (unsigned)kWalkBins) merged[r][pos] = (unsigned)(u * 8 + e);
              }
          }
        } else {
          for (unsigned i = threadIdx.x; i < own_n[r]; i += CT) {
            const uint64_t e = cl[r][i];
            if ((uint32_t)(e >> 32) == cut32[r]) {
              unsigned pos = atomicAdd(&sh.mem_n[r], 1u);
              SPEC_CHECK_INDEX(pos, kWalkBins, 8);
              merged[r][pos] = ~(uint32_t)e;
            }
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r >= nrows) break;
        if (owner[r] != (int)rank) continue;
        const unsigned nm = sh.mem_n[r];
        if (nm > (unsigned)kWalkBins) continue;  // tie_idx stays -1: the exact selection decides
        if (want_max[r]) {
          for (unsigned i = threadIdx.x; i < nm; i += CT) atomicMax(&sh.tie_idx[r], (int)merged[r][i]);
          continue;
        }
        for (unsigned i = threadIdx.x; i < nm; i += CT) {
          const unsigned me = merged[r][i];
          unsigned rk = 0;
          for (unsigned t = 0; t < nm; ++t) rk += (merged[r][t] < me);
          if (rk + 1 == jr[r]) sh.tie_idx[r] = (int)me;
        }
      }
      __syncthreads();
      uint64_t iw[2] = {0ull, 0ull};
      for (int r = 0; r < 2; ++r)
        if (owner[r] == (int)rank) iw[r] = (uint64_t)(uint32_t)sh.tie_idx[r];
      const SlotRow* xs = cluster_share(iw, 2, sh, C, rank, n_ex);
      if (!xs) return false;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r >= nrows) break;
        if (!ok[r] || owner[r] < 0) continue;
        cut_idx[r] = (int)(uint32_t)xs[owner[r]][r];
        if (cut_idx[r] < 0) ok[r] = false;  // too many tied members: exact selection
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (r < nrows && ok[r] && owner[r] < 0) ok[r] = false;  // no member found: exact selection
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nrows) break;
      if (!ok[r]) continue;
      RowCut rc;
      rc.key = cut32[r];
      rc.idx = cut_idx[r];
      rc.kept = sh.sc_kept[r];
      rc.mass = sh.sc_sf[r];
      set_cut(*st[r], rc);
    }
  }
  // p's kept set lies in the window (its cut came from it) and in the CTAs' lists
  p_listed = ok[0] && p_all_listed;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    if (ok[r]) continue;
    RowCut rc;
    if (!cluster_exact_cut<uint16_t>(job, rows[r], *st[r], ua, ub, sh, C, rank, n_ex, smp, rc))
      return false;
    set_cut(*st[r], rc);
  }
  return true;
}

// ---------------------------------------------------------------------------
// bf16 rows under top-k (1 <= k <= kTopkList).  The window's key histogram cannot
// span a window that crosses zero (bf16 keys are dense there), and a window of
// thousands of tokens overflows the lists; but only the row's k largest tokens
// matter.  So each CTA keeps the list of its slice's tokens at or above a
// threshold that starts at m - delta_z and, whenever the list fills, rises to the
// k-th largest 16-bit key the list holds: the CTA's own k largest tokens never
// fall below it.  The union of the CTAs' lists holds the row's k largest tokens;
// sorted (logit desc, index asc) they give the cut by the dense row pass's rule
// (top-k, then the top-p crossing within it), and p's kept set is in the lists.
// ---------------------------------------------------------------------------
constexpr int kTopkList = 128;  // largest k this route takes
constexpr int kTkSort = 1024;   // merged list entries it sorts, per row
constexpr int kTkRetry = 8;     // threshold raises one round of loads may take

// Its buffers inside the cut's shared memory: two sets of this CTA's lists
// [2 sets][2 rows][kCandCTA] (the sets alternate from node to node, so a list the
// other CTAs read is rewritten only after an exchange that each of them reaches
// after reading it), the sort buffers [2][kTkSort], the digit counts [2][256].
__device__ __forceinline__ uint64_t* tk_list(unsigned char* smem, uint32_t set, int r) {
  return reinterpret_cast<uint64_t*>(smem) + ((size_t)(set & 1u) * 2 + r) * kCandCTA;
}
__device__ __forceinline__ uint64_t* tk_sortb(unsigned char* smem, int r) {
  return reinterpret_cast<uint64_t*>(smem) + 4 * kCandCTA + (size_t)r * kTkSort;
}
__device__ __forceinline__ unsigned* tk_hist(unsigned char* smem, int r) {
  return reinterpret_cast<unsigned*>(reinterpret_cast<uint64_t*>(smem) + 4 * kCandCTA +
                                     2 * kTkSort) + r * 256;
}
constexpr size_t kTkSmemBytes = (4 * (size_t)kCandCTA + 2 * (size_t)kTkSort) * 8 + 2 * 256 * 4;

// One warp: the digit (0..255) at which the counts, taken from digit 255 down,
// reach `need` (1 <= need <= their total); `above` = the count of the digits above it.
__device__ void tk_digit(const unsigned* hist, unsigned need, int& digit, unsigned& above) {
  const int lane = threadIdx.x & 31;
  unsigned s = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) s += hist[255 - (8 * lane + t)];
  unsigned incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  const unsigned base = incl - s;
  int d = INT_MAX;
  unsigned ab = 0;
  if (base < need && need <= incl) {
    unsigned run = base;
    for (int t = 0; t < 8; ++t) {
      const unsigned h = hist[255 - (8 * lane + t)];
      if (run + h >= need) { d = 255 - (8 * lane + t); ab = run; break; }
      run += h;
    }
  }
  const unsigned who = __ballot_sync(kFull, d != INT_MAX);
  const int src = who ? __ffs(who) - 1 : 0;
  digit = __shfl_sync(kFull, d, src);
  above = __shfl_sync(kFull, ab, src);
}

// Raises row r's threshold to the K-th largest 16-bit key among this CTA's n list
// entries (K <= n <= kCandCTA) and keeps the entries at or above it (at least K).
// Every thread calls it.
__device__ __noinline__ void tk_compact(uint64_t* list, unsigned n, unsigned K, unsigned* hist, CShared& sh,
                           int r) {
  constexpr int PER = kCandCTA / CT;
  uint64_t mine[PER];
#pragma unroll
  for (int t = 0; t < PER; ++t) {
    const unsigned i = threadIdx.x + t * CT;
    mine[t] = i < n ? list[i] : 0ull;
  }
  for (int i = threadIdx.x; i < 256; i += CT) hist[i] = 0u;
  __syncthreads();
#pragma unroll
  for (int t = 0; t < PER; ++t)
    if (threadIdx.x + t * CT < n) atomicAdd(&hist[(unsigned)(mine[t] >> 56)], 1u);
  __syncthreads();
  if (threadIdx.x < 32) {
    int d;
    unsigned ab;
    tk_digit(hist, K, d, ab);
    if (threadIdx.x == 0) { sh.tk_d1[r] = d; sh.tk_above[r] = ab; }
  }
  __syncthreads();
  const unsigned d1 = (unsigned)sh.tk_d1[r];
  for (int i = threadIdx.x; i < 256; i += CT) hist[i] = 0u;
  __syncthreads();
#pragma unroll
  for (int t = 0; t < PER; ++t)
    if (threadIdx.x + t * CT < n && (unsigned)(mine[t] >> 56) == d1)
      atomicAdd(&hist[(unsigned)(mine[t] >> 48) & 255u], 1u);
  __syncthreads();
  if (threadIdx.x < 32) {
    int d;
    unsigned ab;
    tk_digit(hist, K - sh.tk_above[r], d, ab);
    if (threadIdx.x == 0) {
      sh.tk_thr[r] = key_from16((d1 << 8) | (unsigned)d);
      sh.ncand[r] = 0u;
    }
  }
  __syncthreads();
  const uint32_t thr = sh.tk_thr[r];
  unsigned keep = 0;
#pragma unroll
  for (int t = 0; t < PER; ++t)
    keep += (threadIdx.x + t * CT < n && (uint32_t)(mine[t] >> 32) >= thr) ? 1u : 0u;
  unsigned pos = warp_reserve(&sh.ncand[r], keep);
#pragma unroll
  for (int t = 0; t < PER; ++t)
    if (threadIdx.x + t * CT < n && (uint32_t)(mine[t] >> 32) >= thr) {
      unsigned at = pos++;
      SPEC_CHECK_INDEX(at, n, 9);
      list[at] = mine[t];
    }
  __syncthreads();
}

// The pass over units [ua, ub) of one or two rows (loads as in window_collect_fast):
// tokens whose order key reaches sh.tk_thr[r] go to list[r] (sh.ncand[r] entries).
// A round whose tokens overflow a list raises the threshold and re-inserts them
// from registers; a list past half full is compacted between rounds.  fail[r] is
// set when kTkRetry raises do not make room (ties at one key).
__device__ bool tk_collect(const void* const (&rows)[2], int nrows, int V, int ua, int ub,
                           uint64_t* const (&list)[2], unsigned K, unsigned* const (&hist)[2],
                           CShared& sh, bool (&fail)[2]) {
  const int full = V / 8;
  const int ubf = min(ub, full);
  const uint4* const r0 = reinterpret_cast<const uint4*>(rows[0]);
  const uint4* const r1 = reinterpret_cast<const uint4*>(nrows > 1 ? rows[1] : rows[0]);
  const WinStage stg = win_stage_begin(rows, nrows, ua, ubf, sh);
  int stop = INT_MAX;
  const int nround = (ubf > ua ? (ubf - ua + CT * kWinUnits - 1) / (CT * kWinUnits) : 0) +
                     (ub > full ? 1 : 0);
  for (int rd = 0; rd < nround; ++rd) {  // the same rounds in every thread
    const bool tail = ub > full && rd == nround - 1;
    const int base = tail ? full : ua + rd * CT * kWinUnits;
    uint4 raw[2][kWinUnits];
    if (!tail && stg.on) {
      // this round's stage (bounded wait; every thread gives up together)
      if (!__syncthreads_and(stg.wait(sh, rd))) { stop = rd; break; }
      const uint4* s0 = stg.slot(sh, rd, 0);
      const uint4* s1 = stg.slot(sh, rd, 1);
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h) {
        const int u = base + h * CT + (int)threadIdx.x;
        const bool in = u < ubf;
        raw[0][h] = in ? s0[h * CT + threadIdx.x]
                       : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
        raw[1][h] = (in && nrows > 1)
                        ? s1[h * CT + threadIdx.x]
                        : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
      }
      // every thread has read the stage: it takes round rd + 2
      __syncthreads();
      if (threadIdx.x == 0 && rd + 2 < stg.nfull) {
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        stg.issue(sh, rd + 2);
      }
    } else if (!tail) {
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h) {
        const int u = base + h * CT + (int)threadIdx.x;
        const bool in = u < ubf;
        raw[0][h] = in ? __ldg(r0 + u)
                       : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
        raw[1][h] = (in && nrows > 1)
                        ? __ldg(r1 + u)
                        : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
      }
    } else {
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h)
#pragma unroll
        for (int r = 0; r < 2; ++r)
          raw[r][h] = (h == 0 && threadIdx.x == 0 && r < nrows)
                          ? load_raw<uint16_t>(rows[r], V, full)
                          : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
    }
    // members at or above the threshold, inserted; those past the list's end kept
    // in drop[r] (bit 8 h + e of unit h's element e) for after the threshold rises;
    // end[r]: the end of this thread's slots (0 if it took none)
    uint32_t drop[2] = {0u, 0u};
    unsigned end[2] = {0u, 0u};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      // the threshold key's value rounded up to bf16: a bf16 logit reaches the key
      // exactly when it reaches that value
      const uint32_t thr = sh.tk_thr[r];
      const __nv_bfloat162 t2 = __bfloat162bfloat162(__float2bfloat16_ru(key_value(thr)));
      uint32_t mb[kWinUnits];
      unsigned cnt = 0;
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h) {
        const uint32_t m = (r < nrows && !fail[r]) ? unit_ge_bits(raw[r][h], t2) : 0u;
        mb[h] = m;
        cnt += __popc(m);
      }
      if (!cnt) continue;
      unsigned pos = atomicAdd(&sh.ncand[r], cnt);
      end[r] = pos + cnt;
      uint32_t bits = 0u;
#pragma unroll
      for (int h = 0; h < kWinUnits; ++h) bits |= mb[h] << (8 * h);
      while (bits) {
        const int t = __ffs(bits) - 1;
        bits &= bits - 1u;
        const int h = t >> 3, e = t & 7;
        const uint4 v = h == 0 ? raw[r][0] : h == 1 ? raw[r][1] : h == 2 ? raw[r][2] : raw[r][3];
        const int u = tail ? full : base + h * CT + (int)threadIdx.x;
        if (pos < (unsigned)kCandCTA)
          list[r][pos] = ((uint64_t)unit_key(v, e) << 32) | (uint64_t)(~(uint32_t)(u * 8 + e));
        else
          drop[r] |= 1u << t;
        ++pos;
      }
    }
    // whether a list passed half full: the largest slot end any thread took is the list
    // size, so one barrier reduction decides it for the block; only then is the size
    // read (nothing changes it before the compaction's own barriers)
    const int busy = __syncthreads_or((end[0] > (unsigned)kCandCTA / 2) ||
                                      (end[1] > (unsigned)kCandCTA / 2));
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (!busy || r >= nrows || fail[r]) continue;
      unsigned n = sh.ncand[r];
      if (n <= (unsigned)kCandCTA) {
        if (n > (unsigned)kCandCTA / 2) tk_compact(list[r], n, K, hist[r], sh, r);
        continue;
      }
      for (int it = 0;; ++it) {
        if (it == kTkRetry) { fail[r] = true; break; }
        // the list is full: raise the threshold on what it holds, then re-insert the
        // round's tokens that did not fit and still reach it
        tk_compact(list[r], (unsigned)kCandCTA, K, hist[r], sh, r);
        const uint32_t thr = sh.tk_thr[r];
        unsigned cnt = 0;
        // the units are read again (from cache) rather than held in registers
        auto unit = [&](int h) {
          const int u = tail ? full : base + h * CT + (int)threadIdx.x;
          if (tail) return load_raw<uint16_t>(rows[r], V, full);
          return u < ubf ? __ldg(reinterpret_cast<const uint4*>(rows[r]) + u)
                         : make_uint4(kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2, kNegInfBf16x2);
        };
        uint32_t keep = 0u;
        for (uint32_t bits = drop[r]; bits; bits &= bits - 1u) {
          const int t = __ffs(bits) - 1;
          if (unit_key(unit(t >> 3), t & 7) >= thr) keep |= 1u << t;
        }
        drop[r] = keep;
        cnt = __popc(keep);
        unsigned pos = cnt ? atomicAdd(&sh.ncand[r], cnt) : 0u;
        uint32_t left = 0u;
        for (uint32_t bits = drop[r]; bits; bits &= bits - 1u) {
          const int t = __ffs(bits) - 1;
          const int h = t >> 3, e = t & 7;
          const int u = tail ? full : base + h * CT + (int)threadIdx.x;
          if (pos < (unsigned)kCandCTA)
            list[r][pos] = ((uint64_t)unit_key(unit(h), e) << 32) | (uint64_t)(~(uint32_t)(u * 8 + e));
          else
            left |= 1u << t;
          ++pos;
        }
        drop[r] = left;
        __syncthreads();
        n = sh.ncand[r];
        if (n <= (unsigned)kCandCTA) break;
      }
      if (fail[r] && threadIdx.x == 0) sh.ncand[r] = 0u;
      __syncthreads();
    }
    // every thread has read the sizes before the next round reserves slots
    if (busy) __syncthreads();
  }
  win_stage_end(stg, sh, stop);
  return stop == INT_MAX;
}

// The cut of the p row (and of the q row when with_q) under top-k by the route
// above; rows it cannot decide go to the exact selection.  p_list receives this
// CTA's list of p (sh.ncand[0] entries), which holds its slice's part of p's kept
// set when p_listed.
__device__ bool cluster_cut_topk(const TreeJob& job, const void* prow, const void* qrow,
                                 bool with_q, spec_row_stats& sp, spec_row_stats& sq, int ua,
                                 int ub, unsigned char* smem, uint32_t n_visit, CShared& sh,
                                 int C, uint32_t rank, uint32_t& n_ex, const Samp& smp,
                                 bool& p_listed, const uint64_t*& p_list) {
  p_listed = false;
  const float c = smp.c;
  const int V = job.V;
  const int nrows = with_q ? 2 : 1;
  const unsigned K = (unsigned)smp.top_k;
  spec_row_stats* st[2] = {&sp, &sq};
  const void* const rows[2] = {prow, qrow};
  uint64_t* const list[2] = {tk_list(smem, n_visit, 0), tk_list(smem, n_visit, 1)};
  unsigned* const hist[2] = {tk_hist(smem, 0), tk_hist(smem, 1)};
  p_list = list[0];
  if (threadIdx.x < 2) {
    const int r = threadIdx.x;
    sh.ncand[r] = 0u;
    sh.tk_thr[r] = order_key(st[r]->m - smp.delta_z);
  }
  __syncthreads();
  bool fail[2] = {false, nrows < 2};
  if (!tk_collect(rows, nrows, V, ua, ub, list, K, hist, sh, fail)) return false;
  // every CTA's list sizes (all ones: the row failed somewhere)
  auto exchange = [&](unsigned (&total)[2], bool (&bad)[2], unsigned (&cnt)[2][kMaxC]) -> bool {
    uint64_t w = 0;
    for (int r = 0; r < 2; ++r)
      w |= (uint64_t)(fail[r] ? 0xffffffffu : sh.ncand[r]) << (32 * r);
    const SlotRow* sl = cluster_share(&w, 1, sh, C, rank, n_ex);
    if (!sl) return false;
    for (int r = 0; r < 2; ++r) {
      total[r] = 0u;
      bad[r] = false;
      for (int q = 0; q < C; ++q) {
        const unsigned v = (unsigned)(sl[q][0] >> (32 * r));
        bad[r] |= v == 0xffffffffu;
        cnt[r][q] = v;
        total[r] += bad[r] ? 0u : v;
      }
    }
    return true;
  };
  unsigned total[2], cnt[2][kMaxC];
  bool bad[2];
  if (!exchange(total, bad, cnt)) return false;
  // a row whose window held fewer than K tokens (its K-th largest lies more than
  // delta_z below the maximum) is collected again with no floor
  const bool redo[2] = {!bad[0] && total[0] < K, nrows > 1 && !bad[1] && total[1] < K};
  if (redo[0] || redo[1]) {
    if (threadIdx.x < 2 && redo[threadIdx.x]) {
      sh.ncand[threadIdx.x] = 0u;
      // the lowest finite key: -inf tokens (and the -inf padding of units past the
      // slice) never enter a list
      sh.tk_thr[threadIdx.x] = order_key(-3.402823466e38f);
    }
    __syncthreads();
    bool again[2] = {!redo[0], !redo[1]};  // rows set here are skipped
    if (!tk_collect(rows, nrows, V, ua, ub, list, K, hist, sh, again)) return false;
    for (int r = 0; r < 2; ++r)
      if (redo[r]) fail[r] = again[r];
    if (!exchange(total, bad, cnt)) return false;
  }
  bool ok[2];
  for (int r = 0; r < 2; ++r) ok[r] = r < nrows && !bad[r] && total[r] >= K;
  if ((ok[0] && total[0] > (unsigned)kTkSort) || (ok[1] && total[1] > (unsigned)kTkSort)) {
    // too many to sort: each CTA keeps its own K largest (the lists were final at
    // the exchange; they change only now, and are read after the next one)
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (r < nrows && ok[r] && sh.ncand[r] > K) tk_compact(list[r], sh.ncand[r], K, hist[r], sh, r);
    if (!exchange(total, bad, cnt)) return false;
    for (int r = 0; r < 2; ++r) ok[r] = ok[r] && !bad[r] && total[r] >= K;
  }
  unsigned n_pad[2] = {2u, 2u};
  for (int r = 0; r < 2; ++r) {
    ok[r] = ok[r] && total[r] <= (unsigned)kTkSort;
    while (n_pad[r] < total[r]) n_pad[r] <<= 1;
  }
  // gather every CTA's list (remote shared memory) into the sort buffers
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    if (!ok[r]) continue;
    uint64_t* keys = tk_sortb(smem, r);
    for (unsigned i = threadIdx.x; i < n_pad[r]; i += CT) {
      uint64_t v = 0ull;
      if (i < total[r]) {
        unsigned off = 0, q = 0;
        while (q + 1 < (unsigned)C && i >= off + cnt[r][q]) { off += cnt[r][q]; ++q; }
        unsigned li = i - off;
        SPEC_CHECK_INDEX(li, kCandCTA, 2);
        SPEC_CHECK_INDEX(q, C, 2);
        v = ld_peer_u64(peer_addr(list[r] + li, q));
      }
      unsigned ki = i;
      SPEC_CHECK_INDEX(ki, kTkSort, 3);
      keys[ki] = v;
    }
  }
  __syncthreads();
  const unsigned pad_max = max(ok[0] ? n_pad[0] : 0u, ok[1] ? n_pad[1] : 0u);
  for (unsigned k = 2; k <= pad_max; k <<= 1) {  // bitonic sort, descending
    for (unsigned jj = k >> 1; jj > 0; jj >>= 1) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r >= nrows) break;
        if (!ok[r] || k > n_pad[r]) continue;
        uint64_t* keys = tk_sortb(smem, r);
        for (unsigned i = threadIdx.x; i < n_pad[r]; i += CT) {
          const unsigned ixj = i ^ jj;
          if (ixj > i) {
            const uint64_t a = keys[i], b = keys[ixj];
            const bool swap = ((i & k) == 0) ? (a < b) : (a > b);
            if (swap) { keys[i] = b; keys[ixj] = a; }
          }
        }
      }
      __syncthreads();
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    RowCut rc{};
    if (ok[r])
      ok[r] = window_cut(tk_sortb(smem, r), total[r], n_pad[r], st[r]->m, c, st[r]->s_f, smp, sh,
                         rc);
    if (ok[r]) set_cut(*st[r], rc);
  }
  // p's kept set is among its K largest tokens, all in the CTAs' lists
  p_listed = ok[0];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    if (ok[r]) continue;
    RowCut rc;
    if (!cluster_exact_cut<uint16_t>(job, rows[r], *st[r], ua, ub, sh, C, rank, n_ex, smp, rc))
      return false;
    set_cut(*st[r], rc);
  }
  return true;
}

// Visited-rows-only schedule: the statistics the dense row pass would have written
// for the p row (and the q row when with_q) of a node the walk visits, computed by
// the cluster.  Every CTA covers its slice with a running maximum (its first index)
// and the Kahan sum of 2^((z - max) c), referred to the warp's maximum, then to the
// CTA's; the CTAs' (maximum, sum, argmax, NaN) are exchanged and combined in rank
// order, so every CTA holds the same statistics.
template <typename T>
__device__ bool cluster_row_stats(const TreeJob& job, const void* prow, const void* qrow,
                                  bool with_q, spec_row_stats& sp, spec_row_stats& sq, int ua,
                                  int ub, CShared& sh, int C, uint32_t rank, uint32_t& n_ex,
                                  float c) {
  constexpr int E = Elt<T>::kPerUnit;
  const int V = job.V;
  const int nrows = with_q ? 2 : 1;
  const void* const rows[2] = {prow, qrow};
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float tm[2] = {-CUDART_INF_F, -CUDART_INF_F};
  int targ[2] = {INT_MAX, INT_MAX};
  Kahan ks[2];
  int bad[2] = {0, 0};
  if (threadIdx.x < 2) sh.st_bad[threadIdx.x] = 0;
  __syncthreads();
  // the slices stream through the ring; a thread meets its units in increasing order,
  // so the first index of a strictly larger maximum is its first occurrence
  stream_slice<T>(rows, nrows, V, ua, ub, sh, [&](int u, bool valid, const uint4& raw0,
                                                   const uint4& raw1) {
    if (!valid) return;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nrows) break;
      float z[E];
      Elt<T>::unpack(r ? raw1 : raw0, z);
      float um = z[0];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        bad[r] |= (z[e] != z[e]);
        um = fmaxf(um, z[e]);
      }
      if (um > tm[r]) {
        int first = E - 1;
#pragma unroll
        for (int e = E - 1; e >= 0; --e)
          if (z[e] == um) first = e;
        targ[r] = u * E + first;
        if (tm[r] != -CUDART_INF_F) {
          const float scale = ex2_approx((tm[r] - um) * c);
          ks[r].s *= scale;
          ks[r].c *= scale;
        }
        tm[r] = um;
      }
      if (tm[r] != -CUDART_INF_F) {
        float part = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) part += tempered_weight(z[e], tm[r], c);
        ks[r].add(part);
      }
    }
  });
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    const float wm = warp_max(tm[r]);
    FF sv = ks[r].ff();
    if (tm[r] != -CUDART_INF_F && tm[r] != wm) {
      const float scale = ex2_approx((tm[r] - wm) * c);
      sv.hi *= scale;
      sv.lo *= scale;
    }
    const FF ws = warp_sum_ff(sv);
    const int warg = warp_min_i(tm[r] == wm ? targ[r] : INT_MAX);
    const int wbad = __any_sync(kFull, bad[r]);
    if (lane == 0) {
      sh.st_m[r][warp] = wm;
      sh.st_s[r][warp] = ws.value();
      sh.st_arg[r][warp] = warg;
      if (wbad) atomicOr(&sh.st_bad[r], 1);
    }
  }
  __syncthreads();
  uint64_t w[8] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull};
  if (threadIdx.x == 0) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nrows) break;
      float m = -CUDART_INF_F;
      for (int q = 0; q < CW; ++q) m = fmaxf(m, sh.st_m[r][q]);
      double s = 0.0;
      int arg = INT_MAX;
      for (int q = 0; q < CW; ++q) {
        if (sh.st_m[r][q] != -CUDART_INF_F)
          s += sh.st_s[r][q] * (double)exp2f((sh.st_m[r][q] - m) * c);
        if (sh.st_m[r][q] == m) arg = min(arg, sh.st_arg[r][q]);
      }
      w[4 * r + 0] = (uint64_t)__float_as_uint(m);
      w[4 * r + 1] = (uint64_t)__double_as_longlong(s);
      w[4 * r + 2] = (uint64_t)(uint32_t)arg;
      w[4 * r + 3] = (uint64_t)sh.st_bad[r];
    }
  }
  const SlotRow* sl = cluster_share(w, 4 * nrows, sh, C, rank, n_ex);
  if (!sl) return false;
  spec_row_stats* st[2] = {&sp, &sq};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r >= nrows) break;
    float m = -CUDART_INF_F;
    int any_bad = 0;
    for (int q = 0; q < C; ++q) {
      m = fmaxf(m, __uint_as_float((uint32_t)sl[q][4 * r]));
      any_bad |= (int)sl[q][4 * r + 3];
    }
    double s = 0.0;
    int arg = INT_MAX;
    for (int q = 0; q < C; ++q) {
      const float mq = __uint_as_float((uint32_t)sl[q][4 * r]);
      if (mq != -CUDART_INF_F)
        s += __longlong_as_double((long long)sl[q][4 * r + 1]) * (double)exp2f((mq - m) * c);
      if (mq == m) arg = min(arg, (int)(uint32_t)sl[q][4 * r + 2]);
    }
    const bool finite = !any_bad && m != CUDART_INF_F && m != -CUDART_INF_F && s == s &&
                        s != CUDART_INF;
    spec_row_stats& o = *st[r];
    o.m = m;
    o.status = finite ? SPEC_TREE_OK : SPEC_ROW_NONFINITE;
    o.s_f = s;
    o.cut_key = 0u;
    o.cut_idx = V - 1;
    o.argmax = (arg == INT_MAX) ? 0 : arg;
    o.kept = V;
  }
  if (rank == 0 && threadIdx.x == 0 && job.counters)
    atomicAdd(&job.counters[2], (unsigned long long)nrows * V * Elt<T>::kBytes);
  return true;
}

template <typename T>
__device__ bool cluster_cut(const TreeJob& job, const void* prow, const void* qrow, bool with_q,
                            spec_row_stats& sp, spec_row_stats& sq, int ua, int ub,
                            unsigned char* smem, uint32_t n_visit, CShared& sh, int C,
                            uint32_t rank, uint32_t& n_ex, const Samp& smp, bool& p_listed,
                            const uint64_t*& p_list) {
  p_listed = false;
  p_list = nullptr;
  if constexpr (sizeof(T) == 2) {
    if (!job.exact && smp.top_k > 0 && smp.top_k <= kTopkList)
      return cluster_cut_topk(job, prow, qrow, with_q, sp, sq, ua, ub, smem, n_visit, sh, C, rank,
                              n_ex, smp, p_listed, p_list);
    p_list = bf16_cand_list(smem, 0);
    return cluster_cut_bf16(job, prow, qrow, with_q, sp, sq, ua, ub, smem, sh, C, rank, n_ex, smp,
                            p_listed);
  } else {
    // candidate lists alternate between two sets from node to node (they are read
    // by the other CTAs); then the two sort buffers
    uint64_t* cand = reinterpret_cast<uint64_t*>(smem) + (size_t)(n_visit & 1) * 2 * kCandCTA;
    uint64_t* sortb = reinterpret_cast<uint64_t*>(smem) + 4 * kCandCTA;
    return cluster_cut_sorted<T>(job, prow, qrow, with_q, sp, sq, ua, ub, cand, sortb, sh, C,
                                 rank, n_ex, smp);
  }
}

// ---------------------------------------------------------------------------
// Kept-set mode.  When a node's p cut came from the window and every CTA's list
// of p's window tokens is complete, the kept tokens of p -- the support of p and
// of every residual p^(j) -- are already in the CTAs' shared memory: each CTA holds
// those of its vocabulary slice.  Each CTA keeps them with their filtered p and q
// probabilities; a residual mass is the sum over the cluster of each CTA's exact
// fixed-point sum of max(0, p - q), and the final draw finds the owning CTA from
// the CTAs' fixed-point totals (slices are in rank order = vocabulary order), which
// then ranks its own tokens by index.  No row is read again for the node.
// ---------------------------------------------------------------------------
constexpr int kKeptCTA = kCandCTA;  // kept tokens of one CTA's slice (a subset of its list)

struct KeptSet {
  uint32_t* idx;
  float* p;
  float* q;
  __device__ static KeptSet in_ring(uint4* ring) {
    KeptSet k;
    k.idx = reinterpret_cast<uint32_t*>(ring);
    k.p = reinterpret_cast<float*>(k.idx + kKeptCTA);
    k.q = k.p + kKeptCTA;
    return k;
  }
};

// Block sum of one u64 per thread (the total in every thread).
__device__ unsigned long long block_sum_u64(unsigned long long v, CShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u64(v);
  if (lane == 0) sh.ured[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < CW; ++w) t += sh.ured[w];
  __syncthreads();
  return t;
}

// This CTA's kept tokens of p: the members of its list of p's window (words
// (order key << 32 | ~index)) at or above the cut's word, with their filtered
// probabilities under p and q (0 where q does not keep the token, or when the node
// has no q row), computed with the roundings of unit_probs.
template <typename T>
__device__ void build_kept(const TreeJob& job, const uint64_t* list_p, unsigned n,
                           const void* qrow, bool with_q, const spec_row_stats& sp,
                           const spec_row_stats& sq, const RowF& fp, const RowF& fq,
                           const KeptSet& ks, CShared& sh) {
  const int lane = threadIdx.x & 31;
  const uint64_t cutw = ((uint64_t)sp.cut_key << 32) | (uint64_t)(~(uint32_t)sp.cut_idx);
  if (threadIdx.x == 0) sh.kp_n = 0u;
  __syncthreads();
  for (unsigned i0 = threadIdx.x - lane; i0 < n; i0 += CT) {
    const unsigned i = i0 + lane;
    const uint64_t w = i < n ? list_p[i] : 0ull;
    const bool in = i < n && w >= cutw;
    unsigned pos = warp_reserve(&sh.kp_n, in ? 1u : 0u);
    if (in) {
      SPEC_CHECK_INDEX(pos, kKeptCTA, 4);
      ks.idx[pos] = ~(uint32_t)w;
      ks.p[pos] = key_value((uint32_t)(w >> 32));
    }
  }
  __syncthreads();
  const unsigned nk = sh.kp_n;
  for (unsigned i = threadIdx.x; i < nk; i += CT) {
    const uint32_t id = ks.idx[i];
    const float z = ks.p[i];
    ks.p[i] = __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(z, fp.m), fp.c)), fp.inv_s);
    float qv = 0.f;
    if (with_q) {
      const float zq = Elt<T>::at(qrow, id);
      if (kept_key(order_key(zq), (int)id, sq))
        qv = __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(zq, fq.m), fq.c)), fq.inv_s);
    }
    ks.q[i] = qv;
  }
  if (with_q && threadIdx.x == 0 && job.counters)
    atomicAdd(&job.counters[2], (unsigned long long)nk * Elt<T>::kBytes);
  __syncthreads();
}

// Residual mass over the kept set: every CTA's exact fixed-point sum of
// max(0, p - q) over its tokens, summed over the cluster in rank order; then
// p <- max(0, p - q) / Z where Z > 0 (the step residual_chain applies per token).
// rz[j] receives 1 / Z in fp64 (0 when Z == 0), invz[j] the same in fp32 (-1).
// Returns false if the exchange gave up.
__device__ bool kept_residual(const KeptSet& ks, unsigned nk, double* rz, float* invz, int j,
                              CShared& sh, int C, uint32_t rank, uint32_t& n_ex) {
  unsigned long long part = 0;
  for (unsigned i = threadIdx.x; i < nk; i += CT)
    part += to_fixed(fmaxf(0.f, __fsub_rn(ks.p[i], ks.q[i])));
  part = block_sum_u64(part, sh);
  double tot;
  if (!cluster_sum((double)part, sh, C, rank, n_ex, tot, nullptr)) return false;
  const double z = tot * (1.0 / 4398046511104.0);
  if (threadIdx.x == 0) {
    const double r = z > 0.0 ? 1.0 / z : 0.0;
    rz[j] = r;  // j < N: one residual per child of the node at most
    invz[j] = z > 0.0 ? (float)r : -1.f;
  }
  __syncthreads();
  const float iz = invz[j];
  if (iz > 0.f)
    for (unsigned i = threadIdx.x; i < nk; i += CT)
      ks.p[i] = __fmul_rn(fmaxf(0.f, __fsub_rn(ks.p[i], ks.q[i])), iz);
  __syncthreads();
  return true;
}

// Inverse-CDF draw over the kept set: the smallest token x with C_x >= r * C_V, C the
// inclusive prefix sum in vocabulary order of the fixed-point values of the current
// distribution.  The CTA totals are exchanged; the owning CTA ranks its tokens by
// index and walks them.  Returns the token in the owning CTA (-1 elsewhere); `owner`
// is the owning rank for every CTA, -1 when the distribution is all zero.
__device__ int kept_draw(const KeptSet& ks, unsigned nk, double r, CShared& sh, int C,
                         uint32_t rank, uint32_t& n_ex, bool& ok, int& owner) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long part = 0;
  for (unsigned i = threadIdx.x; i < nk; i += CT) part += to_fixed(ks.p[i]);
  part = block_sum_u64(part, sh);
  double total;
  double cta_tot[kMaxC];
  ok = cluster_sum((double)part, sh, C, rank, n_ex, total, cta_tot);
  owner = -1;
  if (!ok || !(total > 0.0)) return -1;
  double base_c = 0.0, t_c = 0.0;
  owner = pick_crossing(cta_tot, C, r * total, base_c, t_c);
  if (owner != (int)rank) return -1;
  // rank this CTA's tokens by index (all distinct); warp 0's lane 0 then walks them
  uint32_t* order = reinterpret_cast<uint32_t*>(ks.q);  // q is not needed any more
  for (unsigned i = threadIdx.x; i < nk; i += CT) {
    const uint32_t me = ks.idx[i];
    unsigned rk = 0;
    for (unsigned t = 0; t < nk; ++t) rk += (ks.idx[t] < me);
    SPEC_CHECK_INDEX(rk, kKeptCTA, 5);
    order[rk] = i;
  }
  __syncthreads();
  if (warp == 0 && lane == 0) {
    unsigned long long cum = 0;
    int tok = -1;
    for (unsigned t = 0; t < nk; ++t) {
      const uint32_t i = order[t];
      const unsigned long long f = to_fixed(ks.p[i]);
      if (!f) continue;
      cum += f;
      tok = (int)ks.idx[i];
      if ((double)cum >= t_c) break;
    }
    sh.kp_tok = tok;
  }
  __syncthreads();
  return sh.kp_tok;
}

// Shared-memory bytes of the cut's buffers.
template <typename T>
constexpr size_t cut_smem_bytes() {
  return sizeof(T) == 2
             ? (size_t)kWalkBins * (4 * sizeof(unsigned) + 2 * sizeof(unsigned long long)) +
                   2 * (size_t)kCandCTA * sizeof(uint64_t)
             : (4 * (size_t)kCandCTA + 2 * (size_t)kSortW) * sizeof(uint64_t);
}
static_assert(kTkSmemBytes <= cut_smem_bytes<uint16_t>(),
              "the top-k route's buffers fit in the bf16 cut's shared memory");
static_assert(kTopkList <= kCandCTA / 2, "a compacted list keeps room for a round");

// ---------------------------------------------------------------------------
// Sampling walk: one cluster of C CTAs per tree.
// ---------------------------------------------------------------------------
// The sampling parameters of tree b: the launch's, or the tree's own from the
// per-request arrays (the same normalisation as the host applies to the launch's:
// top_k >= V or 0 is off, top_p >= 1 is off).  Invalid values (a temperature that is
// negative, infinite or NaN, top_p <= 0 or NaN, top_k < 0) set `status` to
// SPEC_TREE_INVALID.
__device__ Samp tree_samp(const TreeJob& job, int b, int& status) {
  Samp s{job.temperature, job.c, job.delta_z, job.top_p, job.top_k, job.trunc};
  if (!job.req_temperature) return s;
  const float T = job.req_temperature[b];
  const int k = job.req_top_k ? job.req_top_k[b] : 0;
  const float p = job.req_top_p ? job.req_top_p[b] : 1.0f;
  if (!(T >= 0.0f && T <= 3.402823466e38f) || !(p > 0.0f) || k < 0) {
    status = SPEC_TREE_INVALID;
    s.temperature = 1.0f;
    s.c = 1.0f;
    s.trunc = 0;
    return s;
  }
  s.temperature = T;
  s.c = T > 0.0f ? (float)(1.4426950408889634 / (double)T) : 0.0f;
  s.delta_z = kWindowNats * T;
  s.top_k = (k > 0 && k < job.V) ? k : 0;
  s.top_p = p >= 1.0f ? 1.0f : p;
  s.trunc = (T > 0.0f && (s.top_k > 0 || s.top_p < 1.0f)) ? 1 : 0;
  return s;
}

template <typename T>
__global__ void __launch_bounds__(CT, kWalkCtasPerSm) cluster_walk_kernel(TreeJob job, int C, int max_steps, int ring_stages) {
  __shared__ CShared sh;
  // parents [N], tokens [N], child offsets [N+1], children [N]; then Z [N] (fp64),
  // 1/Z [N] and the per-warp step totals [CW][max_steps]
  extern __shared__ __align__(16) int32_t tsm[];
  constexpr int E = Elt<T>::kPerUnit;
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / C;
  const int N = job.N, V = job.V, W = job.W;
  int32_t *par = tsm, *tok = tsm + N, *cs = tsm + 2 * N, *cl = tsm + 3 * N + 1;
  // per residual step j: 1 / Z_j in fp64 (0 when Z_j == 0) and in fp32 (-1 then)
  double* rz = reinterpret_cast<double*>(tsm + ((4 * N + 1 + 1) & ~1));
  float* invz = reinterpret_cast<float*>(rz + N);
  float* steps = invz + N;
  // the top-k / top-p cut's buffers (16-byte aligned)
  unsigned char* cut_smem = reinterpret_cast<unsigned char*>(
      reinterpret_cast<uintptr_t>(steps + CW * max_steps + 3) & ~(uintptr_t)15);
  // the streaming ring follows the cut's buffers (16-byte aligned: both sizes are)
  uint4* ring = reinterpret_cast<uint4*>(cut_smem + (job.trunc ? cut_smem_bytes<T>() : 0));
  int status = SPEC_TREE_OK;
  {
    const Samp s0 = tree_samp(job, b, status);
    if (threadIdx.x == 0) {
      sh.smp = s0;
      sh.inv_td = s0.temperature > 0.0f ? 1.0 / (double)s0.temperature : 0.0;
    }
  }
  // read from shared memory where used (kept out of the registers)
  const Samp& smp = sh.smp;
  const bool lead = (rank == 0);

  if (threadIdx.x == 0) {
    mbar_init(&sh.xbar[0], (uint32_t)C);
    mbar_init(&sh.xbar[1], (uint32_t)C);
    mbar_init(&sh.wbar[0], 1u);
    mbar_init(&sh.wbar[1], 1u);
    sh.win_g = 0u;
    sh.err = 0u;
    sh.ring = ring;
    sh.ring_stages = ring_stages;
    fence_barrier_init();
  }
  cluster_sync_all();
  const double Td = (double)smp.temperature;
  const float c = smp.c;

  {
    const int st = load_tree(job, b, par, tok, cs, cl, lead, &sh.status);
    if (status == SPEC_TREE_OK) status = st;
  }
  // the kernel launched before this one in the stream (the dense pass) has completed
  // and its writes are visible after this point (returns at once without one)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int nunits = (V + E - 1) / E;
  const int ua = (int)((int64_t)nunits * rank / C), ub = (int)((int64_t)nunits * (rank + 1) / C);
  int32_t* out_tok = job.out_tokens + (int64_t)b * W;
  int32_t* out_path = job.out_path + (int64_t)b * W;
  uint32_t n_ex = 0;
  uint32_t n_visit = 0;
  bool timed_out = false;
  int u = 0, n_acc = 0, final_tok = -1, owner = -1;

  // a greedy tree of a per-request batch: the target's argmax chain
  while (status == SPEC_TREE_OK && smp.temperature == 0.0f) {
    const void* prow = row_at(job.base_p, job, b, u, Elt<T>::kBytes);
    spec_row_stats sp, sq;
    if (job.visited_only) {
      if (!cluster_row_stats<T>(job, prow, prow, false, sp, sq, ua, ub, sh, C, rank, n_ex, 1.0f)) {
        timed_out = true;
        status = SPEC_ROW_TIMEOUT;
        break;
      }
    } else {
      sp = job.stats_p[(int64_t)b * N + u];
    }
    if (sp.status != SPEC_TREE_OK) { status = sp.status; break; }
    int next = -1;
    for (int i = cs[u]; i < cs[u + 1]; ++i) {
      const int ch = cl[i];
      const bool hit = tok[ch] == sp.argmax;
      if (lead && threadIdx.x == 0 && job.out_alpha)
        job.out_alpha[(int64_t)b * N + ch] = hit ? 1.f : 0.f;
      if (hit) { next = ch; break; }
    }
    if (next < 0) { final_tok = sp.argmax; break; }
    if (lead && threadIdx.x == 0) {
      out_tok[n_acc] = tok[next];
      out_path[n_acc + 1] = next;
    }
    ++n_acc;
    u = next;
  }

  while (status == SPEC_TREE_OK && smp.temperature != 0.0f) {
    const int c0 = cs[u], c1 = cs[u + 1];
    const void* prow = row_at(job.base_p, job, b, u, Elt<T>::kBytes);
    const void* qrow = row_at(job.base_q, job, b, u, Elt<T>::kBytes);
    spec_row_stats sp, sq;
    if (job.visited_only) {
      // no dense pass: the statistics of this node's rows come from the cluster
      if (!cluster_row_stats<T>(job, prow, qrow, c1 > c0, sp, sq, ua, ub, sh, C, rank, n_ex, c)) {
        timed_out = true;
        status = SPEC_ROW_TIMEOUT;
        break;
      }
      if (c1 == c0) sq = sp;
    } else {
      sp = job.stats_p[(int64_t)b * N + u];
      sq = sp;
      if (c1 > c0 && sp.status == SPEC_TREE_OK) sq = job.stats_q[(int64_t)b * N + u];
    }
    if (sp.status != SPEC_TREE_OK) { status = sp.status; break; }
    if (c1 > c0 && sq.status != SPEC_TREE_OK) { status = sq.status; break; }
    // the first children's accept-test inputs, one lane per (child, row) of warp 0;
    // they do not depend on the cut and overlap the rest of the block's work
    const int n_pre = min(c1 - c0, kPreKids);
    if (threadIdx.x < 2 * n_pre) {
      const int i = (int)threadIdx.x % n_pre, r = (int)threadIdx.x / n_pre;
      const int ch = cl[c0 + i];
      const float z = Elt<T>::at(r ? qrow : prow, tok[ch]);
      sh.kid_e[r][i] = exp(((double)z - (double)(r ? sq.m : sp.m)) * sh.inv_td);
      sh.kid_k[r][i] = order_key(z);
      if (r == 0) sh.kid_u[i] = unit_uniform(philox_words(job.seed, job.offset, b, ch).x);
    }
    bool p_listed = false;  // kept-set mode for this node
    const uint64_t* p_list = nullptr;  // this CTA's list of p's window tokens
    if (smp.trunc) {
      // cut the visited rows
      if (!cluster_cut<T>(job, prow, qrow, c1 > c0, sp, sq, ua, ub, cut_smem, n_visit++, sh, C,
                          rank, n_ex, smp, p_listed, p_list)) {
        timed_out = true;
        status = SPEC_ROW_TIMEOUT;
        break;
      }
    }
    if (threadIdx.x == 0) {
      sh.inv_s64[0] = 1.0 / sp.s_f;
      sh.inv_s64[1] = c1 > c0 ? 1.0 / sq.s_f : 0.0;
      sh.inv_sp = (float)sh.inv_s64[0];
      sh.inv_sq = (float)sh.inv_s64[1];
    }
    __syncthreads();
    const RowF fp = make_rowf(sp, c, sh.inv_sp), fq = make_rowf(sq, c, sh.inv_sq);
    // p's kept set is in the CTAs' lists: each keeps its slice's part (the ring is idle:
    // this node streams no row again)
    const KeptSet ks = KeptSet::in_ring(ring);
    if (p_listed)
      build_kept<T>(job, p_list, min(sh.ncand[0], (unsigned)kCandCTA), qrow,
                    c1 > c0, sp, sq, fp, fq, ks, sh);
    int j = 0, next = -1;
    for (int i = c0; i < c1; ++i) {
      const int ch = cl[i];
      if (threadIdx.x == 0) {
        const int x = tok[ch];
        double P, Q, uu;
        if (i - c0 < kPreKids) {
          const int k = i - c0;
          P = kept_key(sh.kid_k[0][k], x, sp) ? sh.kid_e[0][k] * sh.inv_s64[0] : 0.0;
          Q = kept_key(sh.kid_k[1][k], x, sq) ? sh.kid_e[1][k] * sh.inv_s64[1] : 0.0;
          uu = sh.kid_u[k];
        } else {
          P = prob64<T>(prow, x, sp, Td);
          Q = prob64<T>(qrow, x, sq, Td);
          uu = unit_uniform(philox_words(job.seed, job.offset, b, ch).x);
        }
        for (int r = 0; r < j; ++r)
          if (rz[r] > 0.0) P = fmax(0.0, P - Q) * rz[r];
        // accept iff uu <= min(1, P / Q), tested as uu * Q <= P (no fp64 divide); the
        // reported alpha is divided in fp32 where both lie in its normal range
        bool accept;
        if (Q > 0.0) {
          accept = P >= Q || uu * Q <= P;
          if (lead && job.out_alpha) {
            float a = 1.0f;
            if (P < Q)
              a = (P > 1e-30 && Q > 1e-30) ? (float)P / (float)Q : (float)(P / Q);
            job.out_alpha[(int64_t)b * N + ch] = a;
          }
        } else {
          accept = P > 0.0;
          if (lead && job.out_alpha) job.out_alpha[(int64_t)b * N + ch] = accept ? 1.0f : 0.0f;
        }
        sh.accept = accept;
      }
      __syncthreads();
      const int acc = sh.accept;
      __syncthreads();
      if (acc) { next = ch; break; }
      if (p_listed) {
        if (!kept_residual(ks, sh.kp_n, rz, invz, j, sh, C, rank, n_ex)) { timed_out = true; break; }
        if (lead && threadIdx.x == 0 && job.counters) atomicAdd(&job.counters[3], 1ull);
        ++j;
        continue;
      }
      const double part = block_sum_ff(
          residual_partial<T>(prow, qrow, V, ua, ub, fp, fq, j, invz, sh), sh);
      double z;
      if (!cluster_sum(part, sh, C, rank, n_ex, z, nullptr)) { timed_out = true; break; }
      if (threadIdx.x == 0) {
        const double r = z > 0.0 ? 1.0 / z : 0.0;
        int jj = j;
        SPEC_CHECK_INDEX(jj, N, 7);
        rz[jj] = r;
        invz[jj] = z > 0.0 ? (float)r : -1.f;
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
        int at = n_acc;
        SPEC_CHECK_INDEX(at, W - 1, 6);
        out_tok[at] = tok[next];
        out_path[at + 1] = next;
      }
      ++n_acc;
      u = next;
      continue;
    }
    const uint4 w = philox_words(job.seed, job.offset, b, u);
    if (p_listed) {
      bool ok = true;
      const int t = kept_draw(ks, sh.kp_n, unit_uniform(w.y), sh, C, rank, n_ex, ok, owner);
      if (!ok) { status = SPEC_ROW_TIMEOUT; timed_out = true; break; }
      // the owning CTA writes the drawn token; an all-zero distribution (not
      // reachable from a valid row) falls back to the row's argmax
      if (owner < 0) final_tok = sp.argmax;
      else if (owner == (int)rank && threadIdx.x == 0) out_tok[n_acc] = (t >= 0) ? t : sp.argmax;
      if (lead && threadIdx.x == 0 && job.counters) atomicAdd(&job.counters[4], 1ull);
      break;
    }
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

template <typename T>
cudaError_t launch_greedy(const TreeJob& job, cudaStream_t s) {
  const size_t dyn = tree_smem_bytes(job.N);
  if (dyn > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        greedy_walk_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
  }
  greedy_walk_kernel<T><<<job.B, GT, dyn, s>>>(job);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Small vocabularies (V <= kSmallMaxV) without a top-k / top-p cut: one warp per
// tree computes everything itself.  A row is eight logits per lane at most, so the
// statistics, the accept tests, the residuals and the final draw are warp
// reductions over registers, and no dense pass precedes the walk (a tree reads only
// the rows it visits).  The rules are the cluster walk's: children in node order,
// accept iff u <= min(1, P/Q) (Q = 0: iff P > 0), p <- max(0, p - q) / Z after a
// rejection (unchanged when Z = 0), the final token the smallest index whose
// inclusive prefix reaches r times the total; probabilities in fp64 (a row is at
// most kSmallPer values per lane).
// ---------------------------------------------------------------------------
constexpr int kSmallMaxV = 256;
constexpr int kSmallPer = kSmallMaxV / 32;  // logits per lane
constexpr int kSmallMaxN = 64;
constexpr int kSmallWarps = 4;              // trees per block

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Tempered probabilities of one row into pr[] (fp64, as the oracle takes them; slots
// past V hold 0); status of the row (SPEC_ROW_NONFINITE for NaN, +inf or all -inf)
// and its argmax.
template <typename T>
__device__ int small_row(const void* row, int V, double inv_t, double (&pr)[kSmallPer],
                         int& argmax) {
  const int lane = threadIdx.x & 31;
  float z[kSmallPer];
  int bad = 0;
  float m = -CUDART_INF_F;
#pragma unroll
  for (int k = 0; k < kSmallPer; ++k) {
    const int i = k * 32 + lane;
    z[k] = i < V ? Elt<T>::at(row, i) : -CUDART_INF_F;
    bad |= (z[k] != z[k]) || (z[k] == CUDART_INF_F);
    m = fmaxf(m, z[k]);
  }
  m = warp_max(m);
  bad = __any_sync(kFull, bad) || m == -CUDART_INF_F;
  int idx = INT_MAX;
#pragma unroll
  for (int k = kSmallPer - 1; k >= 0; --k)
    if (z[k] == m && k * 32 + lane < V) idx = k * 32 + lane;
  argmax = warp_min_i(idx);
  if (bad) return SPEC_ROW_NONFINITE;
  double s = 0.0;
#pragma unroll
  for (int k = 0; k < kSmallPer; ++k) {
    pr[k] = 0.0;
    if (k * 32 < V && z[k] != -CUDART_INF_F) pr[k] = exp(((double)z[k] - (double)m) * inv_t);
    s += pr[k];
  }
  const double inv_s = 1.0 / warp_sum_d(s);
#pragma unroll
  for (int k = 0; k < kSmallPer; ++k) pr[k] *= inv_s;
  return SPEC_TREE_OK;
}

// Element x of a lane-strided fp64 row held in registers (lane x % 32, slot x / 32).
__device__ __forceinline__ double small_at(const double (&a)[kSmallPer], int x) {
  double v = 0.0;
#pragma unroll
  for (int k = 0; k < kSmallPer; ++k)
    if (k == (x >> 5)) v = a[k];
  return __shfl_sync(kFull, v, x & 31);
}

template <typename T>
__global__ void __launch_bounds__(32 * kSmallWarps) small_walk_kernel(TreeJob job) {
  __shared__ int32_t s_par[kSmallWarps][kSmallMaxN];
  __shared__ int32_t s_tok[kSmallWarps][kSmallMaxN];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kSmallWarps + w;
  if (b >= job.B) return;  // the whole warp: nothing below synchronises the block
  const int N = job.N, V = job.V, W = job.W;
  int32_t* par = s_par[w];
  int32_t* tok = s_tok[w];
  int n_max = N;
  SPEC_CHECK_INDEX(n_max, kSmallMaxN + 1, 10);  // the dispatch admits N <= kSmallMaxN
  if (n_max != N) return;
  for (int n = lane; n < N; n += 32) {
    par[n] = job.parents[(int64_t)b * N + n];
    tok[n] = job.tokens[(int64_t)b * N + n];
    if (job.out_alpha) job.out_alpha[(int64_t)b * N + n] = __int_as_float(0x7fc00000);
  }
  __syncwarp();
  // the tree checks of load_tree: root first, parents before children, tokens in the
  // vocabulary, no node deeper than max_depth
  int bad = 0;
  for (int n = lane; n < N; n += 32)
    bad |= n == 0 ? (par[0] != -1) : (par[n] < 0 || par[n] >= n || tok[n] < 0 || tok[n] >= V);
  bad = __any_sync(kFull, bad);
  if (!bad) {
    for (int n = lane; n < N; n += 32) {
      int x = n, d = 0;
      while (x != 0 && d < W) { x = par[x]; ++d; }
      bad |= (x != 0 || d > W - 1);
    }
    bad = __any_sync(kFull, bad);
  }
  int status = bad ? SPEC_TREE_INVALID : SPEC_TREE_OK;
  int32_t* out_tok = job.out_tokens + (int64_t)b * W;
  int32_t* out_path = job.out_path + (int64_t)b * W;
  const double inv_t = 1.0 / (double)job.temperature;
  const size_t eb = Elt<T>::kBytes;
  int u = 0, n_acc = 0, final_tok = -1;
  double P[kSmallPer], Q[kSmallPer];
  while (status == SPEC_TREE_OK) {
    int argmax_p = 0, argmax_q = 0;
    status = small_row<T>(row_at(job.base_p, job, b, u, eb), V, inv_t, P, argmax_p);
    if (status != SPEC_TREE_OK) break;
    bool has_child = false;
    for (int n = u + 1 + lane; n < N; n += 32) has_child |= (par[n] == u);
    has_child = __any_sync(kFull, has_child);
    if (has_child) {
      status = small_row<T>(row_at(job.base_q, job, b, u, eb), V, inv_t, Q, argmax_q);
      if (status != SPEC_TREE_OK) break;
    }
    if (lane == 0 && job.counters)
      atomicAdd(&job.counters[2], (unsigned long long)(has_child ? 2 : 1) * V * eb);
    int next = -1;
    for (int ch = u + 1; has_child && ch < N; ++ch) {
      if (par[ch] != u) continue;
      const int x = tok[ch];
      const double px = small_at(P, x), qx = small_at(Q, x);
      const double uu = unit_uniform(philox_words(job.seed, job.offset, b, ch).x);
      bool accept;
      float alpha;
      if (qx > 0.0) {
        accept = px >= qx || uu * qx <= px;
        alpha = px >= qx ? 1.0f
                         : ((px > 1e-30 && qx > 1e-30) ? (float)px / (float)qx : (float)(px / qx));
      } else {
        accept = px > 0.0;
        alpha = accept ? 1.0f : 0.0f;
      }
      if (lane == 0 && job.out_alpha) job.out_alpha[(int64_t)b * N + ch] = alpha;
      if (accept) { next = ch; break; }
      // rejected: p <- max(0, p - q) / Z (unchanged when Z == 0)
      double part = 0.0;
#pragma unroll
      for (int k = 0; k < kSmallPer; ++k) part += fmax(0.0, P[k] - Q[k]);
      const double z = warp_sum_d(part);
      if (z > 0.0) {
        const double iz = 1.0 / z;
#pragma unroll
        for (int k = 0; k < kSmallPer; ++k) P[k] = fmax(0.0, P[k] - Q[k]) * iz;
      }
      if (lane == 0 && job.counters) atomicAdd(&job.counters[3], 1ull);
    }
    if (next >= 0) {
      if (lane == 0) {
        int at = n_acc;
        SPEC_CHECK_INDEX(at, W - 1, 11);
        out_tok[at] = tok[next];
        out_path[at + 1] = next;
      }
      ++n_acc;
      u = next;
      continue;
    }
    // the final draw from p: the smallest index whose inclusive prefix reaches r times
    // the total (index order: slot-major, lanes within a slot)
    const double r = unit_uniform(philox_words(job.seed, job.offset, b, u).y);
    double mine = 0.0;
#pragma unroll
    for (int k = 0; k < kSmallPer; ++k) mine += P[k];
    const double total = warp_sum_d(mine);
    int tokx = -1, last = -1;
    if (total > 0.0) {
      const double t = r * total;
      double run = 0.0;
#pragma unroll
      for (int k = 0; k < kSmallPer; ++k) {
        if (k * 32 >= V) break;
        double incl = P[k];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double v = __shfl_up_sync(kFull, incl, o);
          if (lane >= o) incl += v;
        }
        incl += run;
        const unsigned hit = __ballot_sync(kFull, P[k] > 0.0 && incl >= t);
        const unsigned any = __ballot_sync(kFull, P[k] > 0.0);
        if (any) last = k * 32 + 31 - __clz(any);
        if (hit && tokx < 0) tokx = k * 32 + __ffs(hit) - 1;
        run = __shfl_sync(kFull, incl, 31);
      }
      if (tokx < 0) tokx = last;  // r == 1 under rounding: the last token with mass
    }
    final_tok = tokx >= 0 ? tokx : argmax_p;
    if (lane == 0 && job.counters) atomicAdd(&job.counters[4], 1ull);
    break;
  }
  if (lane == 0) finish_tree(job, b, status, n_acc, final_tok, true);
}

template <typename T>
cudaError_t launch_small(const TreeJob& job, cudaStream_t s) {
  const int grid = (job.B + kSmallWarps - 1) / kSmallWarps;
  small_walk_kernel<T><<<grid, 32 * kSmallWarps, 0, s>>>(job);
  return cudaGetLastError();
}

int floor_pow2(int x) {
  int p = 1;
  while (p * 2 <= x) p *= 2;
  return p;
}

// CTAs per tree: as many as keep every tree's cluster resident at once (the SMs
// hold kWalkCtasPerSm CTAs each), at most kMaxC, and at least two 256-thread
// rounds of units per CTA.
int cluster_size(int B, int V, int E) {
  const int units = (V + E - 1) / E;
  int C = floor_pow2(max(1, kWalkCtasPerSm * device_sm_count() / max(B, 1)));
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
  size_t dyn = tree_smem_bytes(job.N) + (size_t)job.N * (sizeof(double) + sizeof(float)) +
               (size_t)CW * max_steps * sizeof(float);
  dyn += 16;                                       // 16-byte alignment of what follows
  if (job.trunc) dyn += cut_smem_bytes<T>();       // the cut's buffers
  // the streaming ring: 4 stages where two CTAs per SM still fit, else 2
  static int static_bytes = -1;
  if (static_bytes < 0) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, cluster_walk_kernel<T>) != cudaSuccess) return cudaErrorInvalidValue;
    static_bytes = (int)fa.sharedSizeBytes;
  }
  const size_t two_per_sm = 233472 / kWalkCtasPerSm - 1024;
  const int ring_stages = (dyn + ring_bytes(4) + (size_t)static_bytes <= two_per_sm) ? 4 : 2;
  dyn += ring_bytes(ring_stages);
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
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the walk's CTAs may start (and load their trees)
  // while the dense pass before it in the stream finishes; they wait for its
  // results with griddepcontrol.wait before reading any row statistics
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, cluster_walk_kernel<T>, job, C, max_steps, ring_stages);
}

}  // namespace

bool small_walk_applies(const TreeJob& job, bool greedy, uint32_t flags) {
  return !greedy && !job.trunc && !job.req_temperature && job.V <= kSmallMaxV &&
         job.N <= kSmallMaxN && !(flags & SPEC_FLAG_TEST_STALL);
}

cudaError_t launch_tree_walk(const TreeJob& job, spec_dtype dtype, bool greedy, bool small,
                             cudaStream_t s) {
  if (small)
    return dtype == SPEC_BF16 ? launch_small<uint16_t>(job, s) : launch_small<float>(job, s);
  if (greedy)
    return dtype == SPEC_BF16 ? launch_greedy<uint16_t>(job, s) : launch_greedy<float>(job, s);
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

// Checked builds: this translation unit's error word, read and cleared (0 in other
// builds).  Synchronous: it waits for the device.
uint32_t check_word_walk() {
#ifdef SPEC_CHECK
  unsigned v = 0u;
  const unsigned zero = 0u;
  if (cudaMemcpyFromSymbol(&v, g_spec_check, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (cudaMemcpyToSymbol(g_spec_check, &zero, sizeof(zero)) != cudaSuccess) return 0xffffffffu;
  return v;
#else
  return 0u;
#endif
}

}  // namespace svk
