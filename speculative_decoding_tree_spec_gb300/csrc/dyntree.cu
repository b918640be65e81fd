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
// One CTA per tree; the orders are bitonic sorts of 64-bit keys built so that a
// descending sort is (value desc, depth asc, number asc).
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
  bitonic_desc(keys, n_pad);
  // flatten the kept candidates breadth-first: ascending (depth, number) is descending
  // on its complement
  // (each entry is rewritten by the one thread that reads it)
  for (int j = threadIdx.x; j < n_pad; j += blockDim.x) {
    uint64_t k2 = 0ull;
    if (j < m) {
      const int i = 0xFFFFFF - (int)(keys[j] & 0xFFFFFFu);
      k2 = ((uint64_t)(kMaxDepth - depth_of[i]) << 32) | (uint64_t)(0xFFFFFF - i);
    }
    keys[j] = k2;
  }
  __syncthreads();
  bitonic_desc(keys, n_pad);
  for (int j = threadIdx.x; j < m; j += blockDim.x) {
    const int i = 0xFFFFFF - (int)(keys[j] & 0xFFFFFFu);
    pos_of[i] = j + 1;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < M; j += blockDim.x) {
    if (j == 0) {
      otok[0] = job.root[b];
      opar[0] = -1;
      opos[0] = 0;
      osrc[0] = -1;
      flat_par[0] = -1;
    } else {
      const int i = 0xFFFFFF - (int)(keys[j - 1] & 0xFFFFFFu);
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
  bitonic_desc(keys, n_pad);
  for (int j = threadIdx.x; j < k; j += blockDim.x)
    out_idx[(int64_t)b * k + j] =
        (j < cnt && keys[j] != 0ull) ? 0xFFFFFF - (int)(keys[j] & 0xFFFFFFu) : -1;
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
  const size_t smem = (size_t)n_pad * sizeof(uint64_t) + (size_t)(4 * n + m + 1) * sizeof(int);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(tree_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return SPEC_ERR_CUDA;
  TreeBuildJob job{cand_parent, cand_token, cand_prob, root_token, B, n, m, out_tokens,
                   out_parent_idx, out_position_ids, out_src, out_mask, out_status};
  tree_build_kernel<<<B, kTreeThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(job);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
