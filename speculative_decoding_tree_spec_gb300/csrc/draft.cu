// draft.cu -- the draft-side top-k drafting step (EAGLE / EAGLE-2 paper translation,
// modelers.csdn.net, sections 2.3.1-2.3.2; "LLM speculative decoding: EAGLE",
// jingming.pro, section 4.2.1): at every node the draft model expands, its row of draft
// logits proposes the k largest tokens as children, each with the draft model's
// confidence -- its softmax probability at temperature T over the whole row -- which
// the dynamic tree multiplies along a path.
//
// One 192-thread CTA per row, five per SM (so 640 rows of the full vocabulary fit in one
// wave of 152 SMs).  Each lane takes kDraftUnroll 16-byte units of the row per round
// (one load each, all in flight, the next round's issued before this round's
// arithmetic) and keeps the running maximum and the Kahan sum of 2^((z - max) c),
// c = log2(e)/T, rescaled when the maximum grows (the row pass's normaliser; the
// weights by packed fp32 FMAs).  The CTA keeps one list of the row's largest order keys
// (logit order bits, then the complement of the index: a larger key is a larger logit
// or, on a tie, a lower index) in shared memory.  A round covers a contiguous block of
// units, so every element of a later round has a larger index than every listed key and
// only elements strictly above the list's k-th logit can place: a lane offers those
// (packed bf16 compares against the threshold) to a candidate buffer shared by a group
// of kDraftGroup rounds (one barrier per group), and one warp, a different one each
// group, merges that buffer into the list while the next group streams (bitonic merges
// across the warp's lanes).  The first round is seeded with a floor (the k-th largest
// lane maximum) and merged before the second starts.  A group that offers more
// candidates than the buffer holds merges it at once and offers the rest again against
// the raised list.
#include <cuda_bf16.h>

#include "common.cuh"

namespace svk {

namespace {

constexpr int kDraftThreads = 192;
constexpr int kDraftWarps = kDraftThreads / 32;
constexpr int kDraftUnroll = 4;
constexpr int kDraftMaxK = 32;
constexpr int kDraftCap = 512;  // candidate keys a group's buffer holds
constexpr int kDraftGroup = 2;  // rounds between two barriers

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

// Candidate bits of a lane's units: bit k E + e is set when element e of unit k is
// above thr (kStrict) or not below it.  bf16: two logits per compare, against thr (a
// bf16 value, exact).
template <typename T, bool kStrict>
__device__ __forceinline__ uint32_t candidate_bits(const uint4 (&raw)[kDraftUnroll], float thr) {
  uint32_t bits = 0u;
  if constexpr (sizeof(T) == 2) {
    const __nv_bfloat162 t2 = __bfloat162bfloat162(__float2bfloat16_rn(thr));
#pragma unroll
    for (int k = 0; k < kDraftUnroll; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const unsigned m = kStrict ? __hgt2_mask(as_bf2(w[q]), t2) : __hge2_mask(as_bf2(w[q]), t2);
        bits |= ((m & 1u) | ((m >> 15) & 2u)) << (k * 8 + 2 * q);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kDraftUnroll; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float v = __uint_as_float(w[q]);
        bits |= (uint32_t)(kStrict ? (v > thr) : !(v < thr)) << (k * 4 + q);
      }
    }
  }
  return bits;
}

// 64-bit keys held one per lane, sorted descending by a bitonic network (blocks of
// size s alternate direction so that each pair forms a bitonic sequence; size 32 is
// descending).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t x, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t y = __shfl_xor_sync(kFull, x, stride);
      const bool desc = (lane & size) == 0, low = (lane & stride) == 0;
      x = (low == desc) ? (x > y ? x : y) : (x < y ? x : y);
    }
  }
  return x;
}

// The row's list (32 keys, descending, lane j holding the j-th) merged with n keys of a
// candidate buffer by one whole warp.  A chunk of up to 32 keys is sorted, reversed
// against the list (the lane-wise larger of the list and the reversed chunk holds the
// 32 largest of both, as a bitonic sequence) and merged; a chunk of a few keys is
// inserted one key at a time instead.  Returns the merged list.
__device__ uint64_t merge_into_list(uint64_t L, const uint64_t* buf, int n, int k_out, int lane) {
  for (int c = 0; c < n; c += 32) {
    const int m = min(32, n - c);
    if (m <= 6) {
      for (int i = 0; i < m; ++i) {
        const uint64_t x = buf[c + i];
        const int pos = __popc(__ballot_sync(kFull, L > x));
        if (pos < k_out) {
          const uint64_t up = __shfl_up_sync(kFull, L, 1);
          if (lane > pos) L = up;
          if (lane == pos) L = x;
        }
      }
    } else {
      uint64_t x = lane < m ? buf[c + lane] : 0ull;
      x = warp_sort_desc(x, lane);
      const uint64_t y = __shfl_sync(kFull, x, 31 - lane);
      L = L > y ? L : y;
#pragma unroll
      for (int stride = 16; stride > 0; stride >>= 1) {
        const uint64_t o = __shfl_xor_sync(kFull, L, stride);
        L = ((lane & stride) == 0) == (L > o) ? L : o;
      }
    }
  }
  return L;
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

// The key of element idx of a row: its logit's order bits, then the complement of idx.
template <typename T>
__device__ __forceinline__ uint64_t element_key(const void* row, int idx) {
  const float z = Elt<T>::at(row, idx);
  return ((uint64_t)order_key(z) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)idx);
}

// A lane's candidates (bits of its units in the round at u0) into the round's buffer;
// those past its capacity are returned as still pending.  With lk != 0 only keys above
// lk (the list's k-th key) are kept.
template <typename T>
__device__ __forceinline__ uint32_t append_candidates(const void* row, uint32_t bits, int u0, int lane,
                                                      uint64_t lk, uint64_t* buf, int* cnt) {
  constexpr int E = Elt<T>::kPerUnit;
  uint32_t keep = bits;
  if (lk != 0ull) {
    uint32_t b = bits;
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      const int idx = (u0 + lane + (bit / E) * kDraftThreads) * E + bit % E;
      if (!(element_key<T>(row, idx) > lk)) keep &= ~(1u << bit);
    }
  }
  if (!keep) return 0u;
  int slot = atomicAdd(cnt, __popc(keep));
  uint32_t pend = 0u;
  while (keep) {
    const int bit = __ffs(keep) - 1;
    keep &= keep - 1;
    if (slot < kDraftCap) {
      const int idx = (u0 + lane + (bit / E) * kDraftThreads) * E + bit % E;
      buf[slot] = element_key<T>(row, idx);
    } else {
      pend |= 1u << bit;
    }
    ++slot;
  }
  return pend;
}

template <typename T>
__global__ void __launch_bounds__(kDraftThreads, 5) draft_topk_kernel(DraftJob job) {
  constexpr int E = Elt<T>::kPerUnit;
  constexpr int U = kDraftUnroll;
  __shared__ uint64_t s_list[32];               // the row's largest keys so far, descending
  __shared__ uint64_t s_buf[2][kDraftCap];      // candidates of a group of rounds, by its parity
  __shared__ int s_cnt[2];
  __shared__ unsigned s_thr;  // order key of a logit that nothing later at or below it can beat
  __shared__ float wmax[kDraftWarps];
  __shared__ double wsum[kDraftWarps];
  __shared__ float s_m;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x;
  const void* row = static_cast<const char*>(job.base) + (int64_t)r * job.pitch_bytes;
  const int V = job.V, k_out = job.k;
  const int nunits = (V + E - 1) / E, full_units = V / E;
  const float c = job.c;
  const float2 c2 = make_float2(c, c);
  const int step = kDraftThreads * U;  // units of one round: round q covers [q step, (q+1) step)
  const int nrounds = (nunits + step - 1) / step;

  if (threadIdx.x < 32) s_list[threadIdx.x] = 0ull;  // 0 is below every key
  if (threadIdx.x < 2) s_cnt[threadIdx.x] = 0;
  if (threadIdx.x == 0) s_thr = order_key(-CUDART_INF_F);
  __syncthreads();

  float m = -CUDART_INF_F;
  Kahan s;
  int bad = 0;
  uint4 raw[U], nxt[U];

  // round q: the units loaded last round become this round's, the next round's loads go
  // out, then the running maximum and normaliser; returns the lane's maximum
  auto stream = [&](int q) -> float {
#pragma unroll
    for (int k = 0; k < U; ++k) raw[k] = nxt[k];
    if (q + 1 < nrounds) load_round<T>(row, V, nunits, full_units, (q + 1) * step + warp * 32, lane, nxt);
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
    return um;
  };
  // buffer bb joins the list (a whole warp); its count is cleared and the threshold raised
  auto merge_buffer = [&](int bb, int n) {
    const uint64_t L = merge_into_list(s_list[lane], s_buf[bb], n, k_out, lane);
    s_list[lane] = L;
    const uint64_t lk = __shfl_sync(kFull, L, k_out - 1);
    if (lane == 0) {
      s_cnt[bb] = 0;
      if (lk != 0ull) atomicMax(&s_thr, (unsigned)(lk >> 32));
    }
  };
  // a group that offered more candidates than buffer bb holds: the buffer joins the list,
  // then the pending ones above the list's k-th key are offered again (every pass takes in
  // a full buffer or clears every pending element, so the pass count is bounded by the
  // group's elements over the capacity).  Every thread calls it after a barrier.
  auto drain_overflow = [&](int bb, uint32_t (&pend)[kDraftGroup], int q0, int ng) {
    int n = s_cnt[bb];
    for (int pass = 0; n > kDraftCap && pass <= kDraftGroup * step * E / kDraftCap; ++pass) {
      __syncthreads();  // every thread has read n
      if (warp == 0) merge_buffer(bb, kDraftCap);
      __syncthreads();
      const uint64_t lk = s_list[k_out - 1];
#pragma unroll
      for (int j = 0; j < kDraftGroup; ++j)
        if (j < ng)
          pend[j] = append_candidates<T>(row, pend[j], (q0 + j) * step + warp * 32, lane, lk, s_buf[bb],
                                         &s_cnt[bb]);
      __syncthreads();
      n = s_cnt[bb];
    }
  };

  load_round<T>(row, V, nunits, full_units, warp * 32, lane, nxt);
  {
    // the first round: a floor, per warp the k-th largest lane maximum (k lanes hold an
    // element at least this large), the largest over the warps; every element at or
    // above it is offered, and the list takes them in before the next round starts
    const int u0 = warp * 32;
    const float um = stream(0);
    const float v = (um != um) ? -CUDART_INF_F : um;
    int above = 0;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) {
      const float o = __shfl_sync(kFull, v, j);
      above += (o > v) || (o == v && j < lane);
    }
    if (above == k_out - 1) atomicMax(&s_thr, order_key(v));
    __syncthreads();
    const float fl = key_value(s_thr);
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
    uint32_t pend[kDraftGroup];
#pragma unroll
    for (int j = 0; j < kDraftGroup; ++j) pend[j] = 0u;
    const uint32_t cand = (um != um || um < fl) ? 0u : candidate_bits<T, false>(raw, fl) & valid;
    pend[0] = append_candidates<T>(row, cand, u0, lane, 0ull, s_buf[0], &s_cnt[0]);
    __syncthreads();
    drain_overflow(0, pend, 0, 1);
    if (warp == 0) merge_buffer(0, min(s_cnt[0], kDraftCap));
    __syncthreads();
  }
  // later rounds, kDraftGroup to a barrier: their elements hold larger indices than every
  // listed key, so an element must lie strictly above the threshold to place (the
  // threshold may lag the list); group g offers into buffer g & 1, which one warp, a
  // different one each group, merges into the list while the next group streams
  for (int g = 0, q0 = 1; q0 < nrounds; ++g, q0 += kDraftGroup) {
    const int b = g & 1;
    if (warp == g % kDraftWarps) {
      const int n = min(s_cnt[b ^ 1], kDraftCap);
      if (n > 0) merge_buffer(b ^ 1, n);
    }
    uint32_t pend[kDraftGroup];
#pragma unroll
    for (int j = 0; j < kDraftGroup; ++j) {
      pend[j] = 0u;
      const int q = q0 + j;
      if (q < nrounds) {
        const float um = stream(q);
        const float thr = key_value(*(volatile unsigned*)&s_thr);
        if (__any_sync(kFull, um > thr)) {
          const uint32_t cand = um > thr ? candidate_bits<T, true>(raw, thr) : 0u;
          pend[j] = append_candidates<T>(row, cand, q * step + warp * 32, lane, 0ull, s_buf[b], &s_cnt[b]);
        }
      }
    }
    __syncthreads();
    drain_overflow(b, pend, q0, min(kDraftGroup, nrounds - q0));
  }
  // the last group's candidates
  if (nrounds > 1 && warp == 0) {
    const int b = ((nrounds - 2) / kDraftGroup) & 1;
    const int n = min(s_cnt[b], kDraftCap);
    if (n > 0) s_list[lane] = merge_into_list(s_list[lane], s_buf[b], n, k_out, lane);
  }

  // the row's maximum and normaliser
  bad = __syncthreads_or(bad);
  const float wm = warp_max(m);
  if (lane == 0) wmax[warp] = wm;
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -CUDART_INF_F;
    for (int w = 0; w < kDraftWarps; ++w) M = fmaxf(M, wmax[w]);
    s_m = M;
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
    const uint64_t key = s_list[t];
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
  draft_topk_kernel<T><<<job.R, kDraftThreads, 0, s>>>(job);
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
