// dyntree.cu -- the EAGLE-2 dynamic draft tree on the device (EAGLE / EAGLE-2 paper
// translation, modelers.csdn.net, sections 2.3.1 and 2.3.2; "LLM speculative
// decoding: EAGLE", jingming.pro, section 4.2.1).
//
// The draft model's candidates of a tree arrive in creation order (layer by layer):
// candidate i has a parent candidate (or -1: a child of the root), a token and the
// draft model's confidence p_i.  Its value -- the estimated global acceptance rate --
// is the product of the confidences from the root, taken root-first in fp32,
// v_i = v_parent * p_i (v_root = 1).
//   - expansion: the top-k candidates of the newest layer by value (ties to the lower
//     candidate number) are the ones the draft model expands next;
//   - reranking: the top-m candidates of all layers by value, a shallower candidate
//     winning a tie (then the lower number), form the draft; since a value never
//     exceeds its parent's, they are a connected tree;
//   - flattening: the root, then the kept candidates breadth-first (by depth, then
//     candidate number); the parent of each position, its position id (depth), the
//     candidate it came from, and the attention mask that lets a position see only
//     its ancestors and itself.
// One CTA per tree.  A candidate's 64-bit key orders (value desc, depth asc, number
// asc) as an unsigned integer; the rerank is a radix select of the m largest keys
// (8-bit digits, most significant first, stopping at the first digit whose bin is
// taken whole), the orders within a list are counts of the keys above (short lists)
// or bitonic sorts (long ones).
#include <type_traits>

#include "common.cuh"

namespace svk {

namespace {

constexpr int kTreeThreads = 256;
constexpr int kMaxCand = 4096;   // candidates per tree
constexpr int kMaxDepth = 255;   // of a candidate

// Value and depth of candidate i (walk up to the root, multiply root-first).  Returns
// false for a malformed chain (a parent not before its child, too deep, a confidence
// outside [0, 1]).
__device__ bool cand_value(const int32_t* par, const float* prob, int i, float& v, int& depth) {
  int chain[64];
  int d = 0, x = i;
  while (x >= 0) {
    if (d == 64) return false;
    chain[d++] = x;
    const float q = prob[x];
    if (!(q >= 0.0f && q <= 1.0f)) return false;
    const int p = par[x];
    if (p >= x || p < -1) return false;
    x = p;
  }
  float val = 1.0f;
  for (int j = d - 1; j >= 0; --j) val = __fmul_rn(val, prob[chain[j]]);
  v = __fadd_rn(val, 0.0f);  // -0 counts as +0
  depth = d;
  return true;
}

__device__ __forceinline__ uint64_t rank_key(float v, int depth, int i) {
  return ((uint64_t)__float_as_uint(v) << 32) | ((uint64_t)(kMaxDepth - depth) << 24) |
         (uint64_t)(0xFFFFFF - i);
}

__device__ void bitonic_desc(uint64_t* keys, int n_pad) {
  for (int k = 2; k <= n_pad; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < n_pad; i += blockDim.x) {
        const int ixj = i ^ jj;
        if (ixj > i) {
          const uint64_t a = keys[i], b = keys[ixj];
          const bool swap = ((i & k) == 0) ? (a < b) : (a > b);
          if (swap) { keys[i] = b; keys[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
}

// Lists up to kRankMax long are ordered by counting (one pass over the list per
// member, no barriers); longer ones by a bitonic sort.
constexpr int kRankMax = 1024;

// r[q] = the number of keys[0, cnt) that come before the key of member
// threadIdx.x + q * blockDim (Desc: larger keys first; else smaller first).  A warp
// with no member in a round skips it.
template <int R, bool Desc, typename K>
__device__ __forceinline__ void count_before(const K* keys, int cnt, int (&r)[R]) {
  const int warp_base = threadIdx.x & ~31;
#pragma unroll
  for (int q = 0; q < R; ++q) {
    r[q] = 0;
    if (warp_base + q * kTreeThreads >= cnt) continue;
    const int i = threadIdx.x + q * kTreeThreads;
    const K mine = i < cnt ? keys[i] : K(0);
    int c = 0;
#pragma unroll 8
    for (int j = 0; j < cnt; ++j) c += Desc ? (keys[j] > mine) : (keys[j] < mine);
    r[q] = c;
  }
}

struct RadixState {
  unsigned long long prefix;
  int digit, need, bin, taken;
};

// The m largest of the distinct keys[0, n), into lst[0, m) in no particular order.
// Invariant of a pass: every key above `prefix` on the bits in `mask` is taken, and
// `need` more are to come from the keys equal to it there.
__device__ void radix_select_top(const uint64_t* keys, int n, int m, int* lst, unsigned* hist,
                                 RadixState* st) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t prefix = 0ull, mask = 0ull;
  int need = m;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int d = threadIdx.x; d < 256; d += blockDim.x) hist[d] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint64_t k = keys[i];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds digits 255 - 8l down to 248 - 8l
      unsigned c[8], sum = 0u;
#pragma unroll
      for (int t = 0; t < 8; ++t) { c[t] = hist[255 - 8 * lane - t]; sum += c[t]; }
      unsigned incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      unsigned above = incl - sum;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (above < (unsigned)need && above + c[t] >= (unsigned)need) {
          st->digit = 255 - 8 * lane - t;
          st->need = need - (int)above;
          st->bin = (int)c[t];
        }
        above += c[t];
      }
    }
    __syncthreads();
    prefix |= (uint64_t)st->digit << shift;
    mask |= 0xFFull << shift;
    need = st->need;
    if (st->bin == need) break;  // the whole bin is taken (the same for every thread)
  }
  if (threadIdx.x == 0) st->taken = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x)
    if ((keys[i] & mask) >= prefix) lst[atomicAdd(&st->taken, 1)] = i;
}

struct TreeBuildJob {
  const int32_t* par;    // [B, n]
  const int32_t* tok;    // [B, n]
  const float* prob;     // [B, n]
  const int32_t* root;   // [B]
  int B, n, m;
  int32_t* out_tok;      // [B, m + 1]
  int32_t* out_par;
  int32_t* out_pos;
  int32_t* out_src;
  uint8_t* out_mask;     // [B, m + 1, m + 1]
  int32_t* out_status;   // [B]
};

__global__ void __launch_bounds__(kTreeThreads) tree_build_kernel(TreeBuildJob job) {
  extern __shared__ __align__(16) unsigned char tb_smem[];
  const int b = blockIdx.x;
  const int n = job.n, m = job.m, M = m + 1;
  int n_pad = 2;
  while (n_pad < n) n_pad <<= 1;
  uint64_t* keys = reinterpret_cast<uint64_t*>(tb_smem);  // [n_pad]
  int* pos_of = reinterpret_cast<int*>(keys + n_pad);     // [n]
  int* depth_of = pos_of + n;                             // [n]
  int* flat_par = depth_of + n;                           // [M]
  int32_t* par = flat_par + M;                            // [n] staged parents
  float* prob = reinterpret_cast<float*>(par + n);        // [n] staged confidences
  int* bfs = reinterpret_cast<int*>(prob + n);            // [m] kept, breadth-first
  int* lst = bfs + m;                                     // [m] kept, by value
  uint32_t* k2 = reinterpret_cast<uint32_t*>(lst + m);    // [m]
  __shared__ unsigned hist[256];
  __shared__ RadixState rst;
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    par[i] = job.par[(int64_t)b * n + i];
    prob[i] = job.prob[(int64_t)b * n + i];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n_pad; i += blockDim.x) {
    uint64_t key = 0ull;
    if (i < n) {
      float v;
      int d;
      if (!cand_value(par, prob, i, v, d)) {
        atomicExch(&bad, 1);
      } else {
        key = rank_key(v, d, i);
        depth_of[i] = d;
      }
      pos_of[i] = -1;
    }
    keys[i] = key;
  }
  __syncthreads();
  int32_t* otok = job.out_tok + (int64_t)b * M;
  int32_t* opar = job.out_par + (int64_t)b * M;
  int32_t* opos = job.out_pos + (int64_t)b * M;
  int32_t* osrc = job.out_src + (int64_t)b * M;
  uint8_t* omask = job.out_mask + (int64_t)b * M * M;
  if (bad) {
    for (int j = threadIdx.x; j < M; j += blockDim.x) {
      otok[j] = -1; opar[j] = -1; opos[j] = -1; osrc[j] = -1;
    }
    for (int j = threadIdx.x; j < M * M; j += blockDim.x) omask[j] = 0;
    if (threadIdx.x == 0 && job.out_status) job.out_status[b] = SPEC_TREE_INVALID;
    return;
  }
  // rerank: the m largest keys
  radix_select_top(keys, n, m, lst, hist, &rst);
  __syncthreads();
  // flatten: breadth-first, i.e. ascending (depth, number)
  if (m <= kRankMax) {
    for (int t = threadIdx.x; t < m; t += blockDim.x) {
      const int i = lst[t];
      k2[t] = ((uint32_t)depth_of[i] << 24) | (uint32_t)i;
    }
    __syncthreads();
    auto place = [&](auto rr) {
      constexpr int R = decltype(rr)::value;
      int r[R];
      count_before<R, false>(k2, m, r);
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int t = threadIdx.x + q * kTreeThreads;
        if (t < m) bfs[r[q]] = lst[t];
      }
    };
    if (m <= kTreeThreads) place(std::integral_constant<int, 1>());
    else if (m <= 2 * kTreeThreads) place(std::integral_constant<int, 2>());
    else place(std::integral_constant<int, 4>());
  } else {
    // descending on the complement of (depth, number); the other entries sort last
    for (int j = threadIdx.x; j < n_pad; j += blockDim.x) {
      uint64_t key2 = 0ull;
      if (j < m) {
        const int i = lst[j];
        key2 = ((uint64_t)(kMaxDepth - depth_of[i]) << 32) | (uint64_t)(0xFFFFFF - i);
      }
      keys[j] = key2;
    }
    __syncthreads();
    bitonic_desc(keys, n_pad);
    for (int j = threadIdx.x; j < m; j += blockDim.x)
      bfs[j] = 0xFFFFFF - (int)(keys[j] & 0xFFFFFFu);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < m; j += blockDim.x) pos_of[bfs[j]] = j + 1;
  __syncthreads();
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    if (j == 0) {
      otok[0] = job.root[b];
      opar[0] = -1;
      opos[0] = 0;
      osrc[0] = -1;
      flat_par[0] = -1;
    } else {
      const int i = bfs[j - 1];
      const int p = par[i];
      const int pp = (p < 0) ? 0 : pos_of[p];
      otok[j] = job.tok[(int64_t)b * n + i];
      opar[j] = pp;
      opos[j] = depth_of[i];
      osrc[j] = i;
      flat_par[j] = pp;
    }
  }
  __syncthreads();
  // ancestor mask: zeros with coalesced stores, then each thread marks the ancestors
  // of its rows (the barrier orders the block's global stores)
  for (int e = threadIdx.x; e < M * M; e += blockDim.x) omask[e] = 0;
  __syncthreads();
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    uint8_t* row = omask + (int64_t)j * M;
    int a = j, guard = 0;
    while (a >= 0 && guard++ <= M) {
      row[a] = 1;
      a = flat_par[a];
    }
  }
  if (threadIdx.x == 0 && job.out_status) job.out_status[b] = SPEC_TREE_OK;
}

// Expansion: the k candidates of [lo, hi) with the largest values (ties to the lower
// number), in that order.
__global__ void __launch_bounds__(kTreeThreads)
    tree_expand_kernel(const int32_t* par_all, const float* prob_all, int n, int lo, int hi, int k,
                       int32_t* out_idx) {
  extern __shared__ __align__(16) unsigned char te_smem[];
  const int b = blockIdx.x;
  const int cnt = hi - lo;
  int n_pad = 2;
  while (n_pad < cnt) n_pad <<= 1;
  uint64_t* keys = reinterpret_cast<uint64_t*>(te_smem);   // [n_pad]
  int32_t* par = reinterpret_cast<int32_t*>(keys + n_pad);  // [hi]: the chains stay below hi
  float* prob = reinterpret_cast<float*>(par + hi);         // [hi]
  for (int i = threadIdx.x; i < hi; i += blockDim.x) {
    par[i] = par_all[(int64_t)b * n + i];
    prob[i] = prob_all[(int64_t)b * n + i];
  }
  __syncthreads();
  for (int j = threadIdx.x; j < n_pad; j += blockDim.x) {
    uint64_t key = 0ull;
    if (j < cnt) {
      float v;
      int d;
      if (cand_value(par, prob, lo + j, v, d))
        key = ((uint64_t)__float_as_uint(v) << 32) | (uint64_t)(0xFFFFFF - (lo + j));
    }
    keys[j] = key;
  }
  __syncthreads();
  int32_t* out = out_idx + (int64_t)b * k;
  if (cnt <= kRankMax) {
    // place = the number of keys above; malformed candidates (key 0) take no place
    auto place = [&](auto rr) {
      constexpr int R = decltype(rr)::value;
      int r[R];
      count_before<R, true>(keys, cnt, r);
      int valid = 0;
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int j = threadIdx.x + q * kTreeThreads;
        const bool ok = j < cnt && keys[j] != 0ull;
        if (ok && r[q] < k) out[r[q]] = lo + j;
        valid += __syncthreads_count(ok);
      }
      for (int j = valid + threadIdx.x; j < k; j += blockDim.x) out[j] = -1;
    };
    if (cnt <= kTreeThreads) place(std::integral_constant<int, 1>());
    else if (cnt <= 2 * kTreeThreads) place(std::integral_constant<int, 2>());
    else place(std::integral_constant<int, 4>());
    return;
  }
  bitonic_desc(keys, n_pad);
  for (int j = threadIdx.x; j < k; j += blockDim.x)
    out[j] = (j < cnt && keys[j] != 0ull) ? 0xFFFFFF - (int)(keys[j] & 0xFFFFFFu) : -1;
}

}  // namespace

}  // namespace svk

using namespace svk;

extern "C" int spec_tree_expand_topk(const int32_t* cand_parent, const float* cand_prob,
                                     int32_t B, int32_t n, int32_t layer_begin,
                                     int32_t layer_end, int32_t k, int32_t* out_idx,
                                     spec_stream_t stream) {
  if (B < 0 || n < 1 || n > kMaxCand || k < 1 || layer_begin < 0 || layer_end > n ||
      layer_begin > layer_end)
    return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!cand_parent || !cand_prob || !out_idx) return SPEC_ERR_INVALID_ARG;
  int n_pad = 2;
  while (n_pad < layer_end - layer_begin) n_pad <<= 1;
  const size_t smem = (size_t)n_pad * sizeof(uint64_t) + (size_t)layer_end * 8;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(tree_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  tree_expand_kernel<<<B, kTreeThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(
      cand_parent, cand_prob, n, layer_begin, layer_end, k, out_idx);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" int spec_tree_build(const int32_t* cand_parent, const int32_t* cand_token,
                               const float* cand_prob, const int32_t* root_token, int32_t B,
                               int32_t n, int32_t m, int32_t* out_tokens, int32_t* out_parent_idx,
                               int32_t* out_position_ids, int32_t* out_src, uint8_t* out_mask,
                               int32_t* out_status, spec_stream_t stream) {
  if (B < 0 || n < 1 || n > kMaxCand || m < 1 || m > n || m + 1 > SPEC_MAX_NODES)
    return SPEC_ERR_INVALID_ARG;
  if (B == 0) return SPEC_OK;
  if (!cand_parent || !cand_token || !cand_prob || !root_token || !out_tokens ||
      !out_parent_idx || !out_position_ids || !out_src || !out_mask)
    return SPEC_ERR_INVALID_ARG;
  int n_pad = 2;
  while (n_pad < n) n_pad <<= 1;
  const size_t smem = (size_t)n_pad * sizeof(uint64_t) + (size_t)(4 * n + 4 * m + 1) * sizeof(int);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(tree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  TreeBuildJob job{cand_parent, cand_token, cand_prob, root_token, B, n, m, out_tokens,
                   out_parent_idx, out_position_ids, out_src, out_mask, out_status};
  tree_build_kernel<<<B, kTreeThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(job);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
