// draft.cu -- the draft-side top-k drafting step (EAGLE / EAGLE-2 paper translation,
// modelers.csdn.net, sections 2.3.1-2.3.2; "LLM speculative decoding: EAGLE",
// jingming.pro, section 4.2.1): at every node the draft model expands, its row of draft
// logits proposes the k largest tokens as children, each with the draft model's
// confidence -- its softmax probability at temperature T over the whole row -- which
// the dynamic tree multiplies along a path.
//
// One 256-thread CTA per row.  Each lane takes kDraftUnroll 16-byte units of the row
// per round (one load each, all in flight) and keeps the running maximum and the Kahan
// sum of 2^((z - max) c), c = log2(e)/T, rescaled when the maximum grows (the row
// pass's normaliser; the weights by packed fp32 FMAs).  Each warp keeps the K largest
// order keys it has seen (logit order bits, then the complement of the index: a larger
// key is a larger logit or, on a tie, a lower index), lane j holding the j-th.  Per
// round one ballot asks which lanes' units reach the list's last logit (packed bf16
// maxima); only their elements are offered to the list, one at a time by shuffles,
// so after the first few rounds almost no round inserts anything.  The 8 warp lists
// are merged by counting, for each key, the keys above it.
#include <cuda_bf16.h>

#include "common.cuh"

namespace svk {

namespace {

constexpr int kDraftThreads = 256;
constexpr int kDraftWarps = kDraftThreads / 32;
constexpr int kDraftUnroll = 4;
constexpr int kDraftMaxK = 32;

struct DraftJob {
  const void* base;
  int64_t pitch_bytes;
  int R, V, k;
  float c;       // log2(e) / T
  double inv_t;  // 1 / T
  int32_t* out_tok;
  float* out_prob;
  int32_t* out_status;
  const int* err;  // the producing GEMM's error flag, or null
};

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}

// A unit past the full ones: its elements below V, the rest -inf, as raw words.
template <typename T>
__device__ __forceinline__ uint4 tail_unit(const void* row, int V, int u) {
  constexpr int E = Elt<T>::kPerUnit;
  uint32_t w[4];
  if constexpr (sizeof(T) == 2) {
    const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i0 = u * E + 2 * q, i1 = i0 + 1;
      const uint32_t lo = i0 < V ? r[i0] : 0xFF80u, hi = i1 < V ? r[i1] : 0xFF80u;
      w[q] = lo | (hi << 16);
    }
  } else {
    const uint32_t* r = reinterpret_cast<const uint32_t*>(row);
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = (u * E + q) < V ? r[u * E + q] : 0xFF800000u;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// NaN-propagating maximum of a lane's units.
template <typename T>
__device__ __forceinline__ float units_max(const uint4 (&raw)[kDraftUnroll]) {
  if constexpr (sizeof(T) == 2) {
    __nv_bfloat162 m2 = as_bf2(raw[0].x);
#pragma unroll
    for (int k = 0; k < kDraftUnroll; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = (k == 0 ? 1 : 0); q < 4; ++q) m2 = __hmax2_nan(m2, as_bf2(w[q]));
    }
    const float lo = __low2float(m2), hi = __high2float(m2);
    return (lo != lo || hi != hi) ? CUDART_NAN_F : fmaxf(lo, hi);
  } else {
    float m = -CUDART_INF_F;
    int nan = 0;
#pragma unroll
    for (int k = 0; k < kDraftUnroll; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float v = __uint_as_float(w[q]);
        m = fmaxf(m, v);
        nan |= (v != v);
      }
    }
    return nan ? CUDART_NAN_F : m;
  }
}

// Candidate bits of a lane's units: element e of unit k (bit k E + e) is not below
// thr.  bf16: two logits per compare, against thr (a bf16 value, exact).
template <typename T>
__device__ __forceinline__ uint32_t candidate_bits(const uint4 (&raw)[kDraftUnroll], float thr) {
  uint32_t bits = 0u;
  if constexpr (sizeof(T) == 2) {
    const __nv_bfloat162 t2 = __bfloat162bfloat162(__float2bfloat16_rn(thr));
#pragma unroll
    for (int k = 0; k < kDraftUnroll; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const unsigned m = __hge2_mask(as_bf2(w[q]), t2);
        bits |= ((m & 1u) | ((m >> 15) & 2u)) << (k * 8 + 2 * q);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kDraftUnroll; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) bits |= (uint32_t)(!(__uint_as_float(w[q]) < thr)) << (k * 4 + q);
    }
  }
  return bits;
}

// A lane's U units of the round starting at unit u0 (padding past V is -inf).
template <typename T>
__device__ __forceinline__ void load_round(const void* row, int V, int nunits, int full_units,
                                           int u0, int lane, uint4 (&raw)[kDraftUnroll]) {
  constexpr uint32_t kNegInf = sizeof(T) == 2 ? 0xFF80FF80u : 0xFF800000u;
  if (u0 + 31 + (kDraftUnroll - 1) * kDraftThreads < full_units) {  // no tail (warp-uniform)
#pragma unroll
    for (int k = 0; k < kDraftUnroll; ++k)
      raw[k] = __ldg(reinterpret_cast<const uint4*>(row) + u0 + lane + k * kDraftThreads);
    return;
  }
#pragma unroll
  for (int k = 0; k < kDraftUnroll; ++k) {
    const int u = u0 + lane + k * kDraftThreads;
    if (u < full_units) raw[k] = __ldg(reinterpret_cast<const uint4*>(row) + u);
    else if (u < nunits) raw[k] = tail_unit<T>(row, V, u);
    else raw[k] = make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
  }
}

template <typename T, int K>
__global__ void __launch_bounds__(kDraftThreads) draft_topk_kernel(DraftJob job) {
  constexpr int E = Elt<T>::kPerUnit;
  constexpr int U = kDraftUnroll;
  __shared__ uint64_t wlist[kDraftWarps * K];
  __shared__ uint64_t fin[K];
  __shared__ float wmax[kDraftWarps];
  __shared__ double wsum[kDraftWarps];
  __shared__ float s_m;
  __shared__ unsigned s_cut;  // order key of the largest warp threshold published so far
  __shared__ __align__(16) uint4 stage[kDraftWarps][U][32];  // a round's units, for candidates
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x;
  const void* row = static_cast<const char*>(job.base) + (int64_t)r * job.pitch_bytes;
  const int V = job.V, k_out = job.k;
  const int nunits = (V + E - 1) / E, full_units = V / E;
  const float c = job.c;
  const float2 c2 = make_float2(c, c);

  // the warp's list: lane j < k holds its j-th largest key (0 = empty); only the first
  // k places matter (the row's k largest are among every warp's k largest)
  uint64_t wkey = 0ull;
  bool full = false;           // warp-uniform: the list holds k keys
  float thr = -CUDART_INF_F;   // warp-uniform: the logit of its k-th key once full
  float lo = -CUDART_INF_F;    // warp-uniform: a floor below which nothing can place
  float m = -CUDART_INF_F;
  Kahan s;
  int bad = 0;
  const int step = kDraftThreads * U;
  // a warp whose list is full holds k elements at or above its threshold, so nothing
  // below the largest threshold of any warp can place: the warps share it
  if (threadIdx.x == 0) s_cut = order_key(-CUDART_INF_F);
  __syncthreads();
  uint4 raw[U], nxt[U];
  int u0 = warp * 32;
  if (u0 < nunits) load_round<T>(row, V, nunits, full_units, u0, lane, nxt);
  // every lane runs the same number of rounds (the ballots below need the whole warp);
  // the next round's loads are issued before this round's arithmetic
  for (; u0 < nunits; u0 += step) {
#pragma unroll
    for (int k = 0; k < U; ++k) raw[k] = nxt[k];
    if (u0 + step < nunits) load_round<T>(row, V, nunits, full_units, u0 + step, lane, nxt);
    const float um = units_max<T>(raw);
    bad |= (um != um);
    if (um > m) {
      if (m != -CUDART_INF_F) {
        const float scale = ex2_approx((m - um) * c);
        s.s *= scale;
        s.c *= scale;
      }
      m = um;
    }
    if (m != -CUDART_INF_F) {
      // 2^((z - m) c) for pairs of logits: packed fp32 FMAs and adds
      const float nmc = -m * c;
      const float2 n2 = make_float2(nmc, nmc);
      float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int k = 0; k < U; ++k) {
        float f[E];
        Elt<T>::unpack(raw[k], f);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 a = __ffma2_rn(make_float2(f[e], f[e + 1]), c2, n2);
          acc[(e >> 1) & 1] = __fadd2_rn(acc[(e >> 1) & 1], make_float2(ex2_approx(a.x), ex2_approx(a.y)));
        }
      }
      const float2 tot = __fadd2_rn(acc[0], acc[1]);
      s.add(tot.x + tot.y);
    }

    if (!full) {
      // until the list is full: a floor from this round, the k-th largest lane maximum
      // (k lanes hold an element at least this large, so nothing below it can place)
      const float v = (um != um) ? -CUDART_INF_F : um;
      int above = 0;
#pragma unroll 8
      for (int j = 0; j < 32; ++j) {
        const float o = __shfl_sync(kFull, v, j);
        above += (o > v) || (o == v && j < lane);
      }
      const unsigned at = __ballot_sync(kFull, above == k_out - 1);
      if (at) lo = fmaxf(lo, __shfl_sync(kFull, v, __ffs(at) - 1));
    }
    // offer the elements that reach the list's last logit (padding past V never)
    const float cut = fmaxf(full ? fmaxf(thr, lo) : lo, key_value(*(volatile unsigned*)&s_cut));
    if (!__any_sync(kFull, !(um < cut))) continue;
    uint32_t cand = 0u;
    if (!(um < cut)) {
      uint32_t valid = 0xFFFFFFFFu;
      if (u0 + 32 + (U - 1) * kDraftThreads > full_units) {
        valid = 0u;
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int u = u0 + lane + k * kDraftThreads;
          const int n_in = min(max(V - u * E, 0), E);  // elements of this unit below V
          valid |= (uint32_t)((1ull << n_in) - 1ull) << (k * E);
        }
      }
      cand = candidate_bits<T>(raw, cut) & valid;
    }
#pragma unroll
    for (int k = 0; k < U; ++k) stage[warp][k][lane] = raw[k];
    __syncwarp();
    unsigned bal = __ballot_sync(kFull, cand != 0u);
    while (bal) {
      const int src = __ffs(bal) - 1;
      bal &= bal - 1;
      uint32_t bits = __shfl_sync(kFull, cand, src);
      while (bits) {
        const int bit = __ffs(bits) - 1;
        bits &= bits - 1;
        const int k = bit / E, e = bit % E;
        const float z = sizeof(T) == 2
            ? __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(&stage[warp][k][src])[e] << 16)
            : reinterpret_cast<const float*>(&stage[warp][k][src])[e];
        if (full && z < thr) continue;  // the list moved on meanwhile (warp-uniform)
        const int idx = (u0 + src + k * kDraftThreads) * E + e;
        const uint64_t x =
            ((uint64_t)order_key(z) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
        // the lanes holding larger keys are a prefix of the list
        const int pos = __popc(__ballot_sync(kFull, lane < k_out && wkey > x));
        if (pos < k_out) {
          const uint64_t up = __shfl_up_sync(kFull, wkey, 1);
          if (lane > pos && lane < k_out) wkey = up;
          if (lane == pos) wkey = x;
          const uint64_t last = __shfl_sync(kFull, wkey, k_out - 1);
          full = last != 0ull;
          thr = key_value((uint32_t)(last >> 32));
        }
      }
    }
    if (full && lane == 0) atomicMax(&s_cut, order_key(thr));
    __syncwarp();
  }

  // the row's maximum and normaliser
  bad = __syncthreads_or(bad);
  const float wm = warp_max(m);
  if (lane == 0) wmax[warp] = wm;
  if (lane < K) wlist[warp * K + lane] = lane < k_out ? wkey : 0ull;
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -CUDART_INF_F;
    for (int w = 0; w < kDraftWarps; ++w) M = fmaxf(M, wmax[w]);
    s_m = M;
  }
  // the k largest of the warps' keys: a key's place is the number of keys above it
  if ((int)threadIdx.x < kDraftWarps * K) {
    const uint64_t mine = wlist[threadIdx.x];
    int above = 0;
    for (int j = 0; j < kDraftWarps * K; ++j) above += wlist[j] > mine;
    if (mine != 0ull && above < k_out) fin[above] = mine;
  }
  __syncthreads();
  const float M = s_m;
  FF sv = s.ff();
  if (m != -CUDART_INF_F && M != CUDART_INF_F) {
    const float scale = ex2_approx((m - M) * c);
    sv.hi *= scale;
    sv.lo *= scale;
  } else {
    sv.hi = sv.lo = 0.f;
  }
  const FF ws = warp_sum_ff(sv);
  if (lane == 0) wsum[warp] = ws.value();
  __syncthreads();
  const bool finite = !bad && M != CUDART_INF_F && M != -CUDART_INF_F;
  if ((int)threadIdx.x < k_out) {
    double S = 0.0;
    for (int w = 0; w < kDraftWarps; ++w) S += wsum[w];
    const int t = threadIdx.x;
    const uint64_t key = fin[t];
    int32_t tok = -1;
    float p = 0.f;
    if (finite) {
      tok = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
      const float z = key_value((uint32_t)(key >> 32));
      p = (float)(exp(((double)z - (double)M) * job.inv_t) / S);
    }
    job.out_tok[(int64_t)r * k_out + t] = tok;
    job.out_prob[(int64_t)r * k_out + t] = p;
  }
  if (threadIdx.x == 0 && job.out_status)
    job.out_status[r] = (job.err && *job.err) ? SPEC_ROW_TIMEOUT
                                              : (finite ? SPEC_TREE_OK : SPEC_ROW_NONFINITE);
}

template <typename T>
cudaError_t launch_draft(const DraftJob& job, cudaStream_t s) {
  if (job.k <= 8) draft_topk_kernel<T, 8><<<job.R, kDraftThreads, 0, s>>>(job);
  else if (job.k <= 16) draft_topk_kernel<T, 16><<<job.R, kDraftThreads, 0, s>>>(job);
  else draft_topk_kernel<T, 32><<<job.R, kDraftThreads, 0, s>>>(job);
  return cudaGetLastError();
}

}  // namespace

}  // namespace svk

using namespace svk;

namespace {

int draft_topk_impl(const void* logits, spec_dtype dtype, int32_t R, int32_t V, int64_t row_pitch,
                    int32_t k, float temperature, int32_t* out_tokens, float* out_probs,
                    int32_t* out_status, const int* err, spec_stream_t stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if (R < 0 || V < 1 || k < 1 || k > kDraftMaxK || k > V) return SPEC_ERR_INVALID_ARG;
  if (V > SPEC_MAX_VOCAB) return SPEC_ERR_TOO_LARGE;
  if (!(temperature > 0.0f) || !(temperature <= 3.402823466e38f)) return SPEC_ERR_INVALID_ARG;
  if (row_pitch < V) return SPEC_ERR_INVALID_ARG;
  if (R == 0) return SPEC_OK;
  if (!logits || !out_tokens || !out_probs) return SPEC_ERR_INVALID_ARG;
  const int64_t es = dtype == SPEC_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) || (row_pitch * es) % 16 != 0)
    return SPEC_ERR_MISALIGNED;
  DraftJob job{};
  job.base = logits;
  job.pitch_bytes = row_pitch * es;
  job.R = R;
  job.V = V;
  job.k = k;
  job.c = (float)(1.4426950408889634 / (double)temperature);
  job.inv_t = 1.0 / (double)temperature;
  job.out_tok = out_tokens;
  job.out_prob = out_probs;
  job.out_status = out_status;
  job.err = err;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      dtype == SPEC_BF16 ? launch_draft<uint16_t>(job, s) : launch_draft<float>(job, s);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

extern "C" int spec_draft_topk(const void* logits, spec_dtype dtype, int32_t R, int32_t V,
                               int64_t row_pitch, int32_t k, float temperature,
                               int32_t* out_tokens, float* out_probs, int32_t* out_status,
                               spec_stream_t stream) {
  return draft_topk_impl(logits, dtype, R, V, row_pitch, k, temperature, out_tokens, out_probs,
                         out_status, nullptr, stream);
}

// ---------------------------------------------------------------------------------------
// Draft LM head + top-k in one call: the draft logits F W^T of the expanded nodes are
// formed on the tensor cores (the LM-head GEMM of lmhead.cu, bf16 rows written once)
// and ranked by the kernel above.  Ranking inside the GEMM's epilogue (one row per
// epilogue thread, a register list per row and tile) was measured 2.2x slower than
// this pair: the list upkeep outlasted the tile's MMAs.
// ---------------------------------------------------------------------------------------
namespace {

struct DraftFusedLayout {
  size_t part, err, logits, total;
  int64_t pitch;  // of the logits rows kept in the workspace
};

DraftFusedLayout draft_fused_layout(int32_t R, int32_t V) {
  DraftFusedLayout L{};
  L.pitch = ((int64_t)V + 7) / 8 * 8;  // 16-byte aligned rows
  L.part = 0;
  L.err = align_up(lmhead_part_bytes(R, V), 256);
  L.logits = align_up(L.err + sizeof(int), 256);
  L.total = align_up(L.logits + (size_t)R * (size_t)L.pitch * 2, 256);
  return L;
}

constexpr int kDraftFusedMaxK = 32;

}  // namespace

extern "C" size_t spec_draft_fused_workspace_size(int32_t R, int32_t V, int32_t k) {
  if (R < 1 || V < 1 || k < 1 || k > kDraftFusedMaxK || V > SPEC_MAX_VOCAB) return 0;
  return draft_fused_layout(R, V).total;
}

extern "C" int spec_draft_topk_fused_lmhead(const void* features, const void* lm_head_w,
                                            int32_t d, int32_t R, int32_t V, int32_t k,
                                            float temperature, void* out_logits,
                                            int64_t logits_pitch, int32_t* out_tokens,
                                            float* out_probs, int32_t* out_status,
                                            void* workspace, size_t workspace_bytes,
                                            spec_stream_t stream) {
  if (R < 0 || V < 1 || d < 1 || k < 1 || k > kDraftFusedMaxK || k > V) return SPEC_ERR_INVALID_ARG;
  if (V > SPEC_MAX_VOCAB) return SPEC_ERR_TOO_LARGE;
  if (!(temperature > 0.0f) || !(temperature <= 3.402823466e38f)) return SPEC_ERR_INVALID_ARG;
  if (R == 0) return SPEC_OK;
  if (!features || !lm_head_w || !out_tokens || !out_probs || !workspace) return SPEC_ERR_INVALID_ARG;
  // the tensor maps need 16-byte aligned bases and rows (d a multiple of 8)
  if ((reinterpret_cast<uintptr_t>(features) & 15u) || (reinterpret_cast<uintptr_t>(lm_head_w) & 15u) ||
      d % 8 != 0)
    return SPEC_ERR_MISALIGNED;
  if (out_logits) {
    if (logits_pitch < V) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out_logits) & 15u) || (logits_pitch * 2) % 16 != 0)
      return SPEC_ERR_MISALIGNED;
  }
  const DraftFusedLayout L = draft_fused_layout(R, V);
  if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPEC_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int* err = reinterpret_cast<int*>(ws + L.err);
  void* logits = out_logits ? out_logits : static_cast<void*>(ws + L.logits);
  const int64_t pitch = out_logits ? logits_pitch : L.pitch;
  if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (launch_lmhead_logits(features, lm_head_w, R, V, d, logits, pitch, ws + L.part, err, s) !=
      cudaSuccess)
    return SPEC_ERR_CUDA;
  return draft_topk_impl(logits, SPEC_BF16, R, V, pitch, k, temperature, out_tokens, out_probs,
                         out_status, err, stream);
}
