// rows.cu -- the dense row pass: per logit row, the maximum and its lowest index,
// the tempered normaliser, and the top-k / top-p cut ("LLM speculative decoding:
// EAGLE", section 1 note: p and q are compared after temperature, top-k, top-p or
// argmax processing).
//
// One persistent block per SM, warp-specialised: one producer warp streams the
// block's rows, chunk after chunk, into a ring of kRingStages shared-memory stages
// with bulk (TMA) copies, running ahead across row boundaries; kRowThreads
// consumer threads own one row at a time.  A single pass over each chunk computes
//   * each warp's running maximum and the sum of 2^((z - M_warp) c), rescaled
//     whenever the warp maximum grows (online softmax), Kahan-summed;
//   * the maximum (its lowest index is recovered at the end of the row);
//   * when top-k / top-p is active, a candidate window: every token within
//     kWindowNats nats of the block's running maximum is appended to its warp's
//     region of shared memory.
// The cut is then found inside the window.  bf16 windows are resolved with an
// exact histogram over their (few hundred) distinct keys -- equal logits carry
// equal weights, so a bin's mass is its count times one weight; fp32 windows are
// sorted.  Masses are 42-bit fixed point, so every sum is exact and independent
// of order.  When the window overflows or provably misses the cut, the row falls
// back to an exact full-row selection by 4-way bisection on the order key; both
// routes produce bit-identical statistics.  Consumer-only synchronisation uses a
// named barrier, so the producer keeps streaming while a row is being selected.
#include <cuda_bf16.h>

#include <climits>

#include "common.cuh"
#include "select.cuh"

namespace svk {

namespace {

constexpr int NT = kRowThreads;        // consumer threads
constexpr int NW = NT / 32;            // consumer warps
constexpr int kBlockThreads = NT + 32; // + the producer warp
constexpr int kStageBytes = kRingUnits * NT * 16;

// barrier over the consumer threads only
__device__ __forceinline__ void csync() { named_sync(NT); }
struct CSync {
  __device__ static void sync() { named_sync(NT); }
};
static_assert(NT == kSelThreads, "the exact selection runs on the consumer threads");

struct RowShared {
  unsigned wcnt[NW];     // candidates appended by each warp (may exceed its region)
  int woverflow[NW];
  int tmo;              // a bounded wait gave up in this block (sticky)
  int sel_ok, sel_bcut;
  unsigned sel_jcut, sel_kept, sel_ncut;
  unsigned long long sel_sf;
  uint32_t sel_cutkey;
  float warp_m[NW];
  double warp_s[NW];
  float warp_best[NW];
  int warp_best_idx[NW];
  int warp_bad[NW];
  unsigned run_key;
  unsigned n_cand;
  unsigned n_keep;
  int first;
  int ok;
  unsigned tie_n;
  int tie_idx;
  unsigned sel_j;
  SelShared sel;         // the exact selection's scratch
  unsigned long long tau;
  // results broadcast by thread 0
  float m;
  double s_total;
  int argmax;
  int bad;
};

__device__ __forceinline__ __nv_bfloat162 bf2(uint32_t w) {
  return *reinterpret_cast<const __nv_bfloat162*>(&w);
}

__device__ __forceinline__ const void* row_ptr(const void* base, int64_t elems, int bytes) {
  return static_cast<const void*>(static_cast<const char*>(base) + elems * bytes);
}

// ---------------------------------------------------------------------------
// The row pass kernel.  MODE 0: greedy (max + argmax only).  MODE 1: sampling
// without truncation.  MODE 2: sampling with top-k and/or top-p.
// ---------------------------------------------------------------------------
// Candidate entries.  bf16: one 32-bit word, the vocabulary index above the key's
// offset from the row's floor key (fixed after the first iteration; every later
// window threshold is higher, so offsets are never negative).  fp32: (index, bits).
template <typename T> struct Cand;
template <> struct Cand<uint16_t> {
  static constexpr int kCap = kCandCapBf16;
  using entry_t = uint32_t;
  __device__ __forceinline__ static uint4 neg_inf() {
    return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
  }
  __device__ __forceinline__ static uint4 partial(const void* row, int V, int u) {
    uint32_t w[4];
    const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i0 = u * 8 + 2 * q, i1 = i0 + 1;
      const uint32_t lo = i0 < V ? (uint32_t)__ldg(r + i0) : 0xff80u;
      const uint32_t hi = i1 < V ? (uint32_t)__ldg(r + i1) : 0xff80u;
      w[q] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <> struct Cand<float> {
  static constexpr int kCap = kCandCapF32;
  using entry_t = uint2;
  __device__ __forceinline__ static uint4 neg_inf() {
    return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
  }
  __device__ __forceinline__ static uint4 partial(const void* row, int V, int u) {
    uint32_t w[4];
    const float* r = reinterpret_cast<const float*>(row);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = u * 4 + q;
      w[q] = i < V ? __float_as_uint(__ldg(r + i)) : 0xff800000u;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Dynamic shared memory: the ring, its full / empty barriers, the candidate
// regions, and the selection scratch (histogram, bin weights, ties; or the sort
// keys of an fp32 window).
// The streaming modes (0, 1) need no candidate regions or selection scratch: their
// blocks are small enough for 4 per SM (3 ring stages each, 56 registers), twice the
// warps of the cutting mode's 2 blocks to cover the latency of the stages in flight.
constexpr int kRingStagesStream = 3;
constexpr int kRowBlocksStream = 4;  // resident blocks per SM in the streaming modes
template <int MODE>
__host__ __device__ constexpr int ring_stages() { return MODE == 2 ? kRingStages : kRingStagesStream; }
template <int MODE>
__host__ __device__ constexpr int row_blocks() { return MODE == 2 ? kRowBlocksPerSm : kRowBlocksStream; }
template <int MODE>
__host__ __device__ constexpr size_t ring_bytes() { return (size_t)ring_stages<MODE>() * kStageBytes; }
template <int MODE>
__host__ __device__ constexpr size_t bar_bytes() { return (size_t)ring_stages<MODE>() * 16; }

// Balanced schedule of a tree launch's rows (sampling without a cut, the verify
// step's dense pass): the draft row of a node without children is never read, so
// every G-th virtual row would give the blocks unequal numbers of real rows.  Each
// block instead lists the rows it streams: every G-th of the needed rows, in virtual
// order, from its own index.  Its buffers (small: four blocks per SM must still fit):
// the needed-draft-row bit mask, the words' exclusive population prefix (+ the
// total), and the block's list of rows.
constexpr int kSchedMaxNodes = 16384;  // B * N the schedule covers
constexpr int kSchedWords = kSchedMaxNodes / 32;
constexpr int kSchedRows = 64;         // rows of one block
constexpr int kSchedBatch = 8;         // parent entries one thread loads at once
template <int MODE>
__host__ __device__ constexpr size_t sched_bytes() {
  return MODE == 1 ? (size_t)kSchedWords * 4 + (size_t)(kSchedWords + 2) * 2 + kSchedRows * 4 : 0;
}
constexpr size_t kScratchBytes = (size_t)kHistBins * 12 + (size_t)kTieCap * 4 > (size_t)kSortCap * 8
                                     ? (size_t)kHistBins * 12 + (size_t)kTieCap * 4
                                     : (size_t)kSortCap * 8;
template <typename T>
__host__ __device__ constexpr size_t cand_bytes() {
  return (size_t)Cand<T>::kCap * sizeof(typename Cand<T>::entry_t);
}
template <typename T, int MODE>
__host__ __device__ constexpr size_t row_dyn_smem() {
  return ring_bytes<MODE>() + bar_bytes<MODE>() + (MODE == 2 ? cand_bytes<T>() + kScratchBytes : 0) +
         sched_bytes<MODE>();
}

// 16-bit order key of the bf16 logit with raw bits b.
__device__ __forceinline__ uint32_t key16_bits(uint32_t b) {
  return order_key(__uint_as_float(b << 16)) >> 16;
}

// Maximum of a thread's U units: packed bf16x2 maxima for bf16 logits (NaN-propagating
// when asked), fmaxf for fp32.
template <typename T, bool PROPAGATE_NAN>
__device__ __forceinline__ float packed_max(const uint4 (&raw)[kRingUnits]) {
  if constexpr (sizeof(T) == 2) {
    __nv_bfloat162 m2 = bf2(raw[0].x);
#pragma unroll
    for (int k = 0; k < kRingUnits; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = (k == 0 ? 1 : 0); q < 4; ++q)
        m2 = PROPAGATE_NAN ? __hmax2_nan(m2, bf2(w[q])) : __hmax2(m2, bf2(w[q]));
    }
    const float lo = __low2float(m2), hi = __high2float(m2);
    return PROPAGATE_NAN ? ((lo != lo || hi != hi) ? CUDART_NAN_F : fmaxf(lo, hi)) : fmaxf(lo, hi);
  } else {
    float m = -CUDART_INF_F;
    int nan = 0;
#pragma unroll
    for (int k = 0; k < kRingUnits; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float v = __uint_as_float(w[q]);
        m = fmaxf(m, v);
        if (PROPAGATE_NAN) nan |= (v != v);
      }
    }
    return (PROPAGATE_NAN && nan) ? CUDART_NAN_F : m;
  }
}

// Window membership bits of a thread's units (a superset is fine: the final window
// is re-filtered exactly).  bf16: compares against the threshold rounded down to
// bf16, two logits per instruction; bit p = low half of word p, bit p + 16 = high
// half.  fp32: bit p = word p.
template <typename T>
__device__ __forceinline__ unsigned window_mask(const uint4 (&raw)[kRingUnits],
                                                const float (&f)[kRingUnits][Elt<T>::kPerUnit],
                                                __nv_bfloat162 t2, float thr) {
  unsigned mask = 0;
  if constexpr (sizeof(T) == 2) {
#pragma unroll
    for (int k = 0; k < kRingUnits; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int p = k * 4 + q;
        mask |= __hge2_mask(bf2(w[q]), t2) & ((1u << p) | (1u << (p + 16)));
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kRingUnits; ++k)
#pragma unroll
      for (int e = 0; e < 4; ++e) mask |= (f[k][e] >= thr) ? (1u << (k * 4 + e)) : 0u;
  }
  return mask;
}

// Unit k, element e and the shared-memory byte offset (within the stage) of the
// logit named by a window bit.
template <typename T>
__device__ __forceinline__ uint32_t window_slot(int bit, int& k, int& e) {
  static_assert(kRingUnits * 4 <= 16, "window bits are laid out for up to 16 words per thread");
  if constexpr (sizeof(T) == 2) {
    const int p = bit & 15, half = bit >> 4;
    k = p >> 2;
    const int q = p & 3;
    e = 2 * q + half;
    return (uint32_t)((k * NT + (int)threadIdx.x) * 16 + q * 4 + half * 2);
  } else {
    k = bit >> 2;
    e = bit & 3;
    return (uint32_t)((k * NT + (int)threadIdx.x) * 16 + e * 4);
  }
}

__device__ __forceinline__ bool use_schedule(const RowJob& job, int MODE, int G) {
  if (MODE != 1 || job.mode != kRowsTree || !job.with_q) return false;
  const int BN = job.B * job.N;
  return BN <= kSchedMaxNodes && (2 * BN + G - 1) / G <= kSchedRows;
}

// Every thread of the block: the rows this block streams, in order, into rows[];
// returns their number.  A draft row is needed when its node has a child (a later
// node naming it as parent) and the tree is sampled.
__device__ int build_schedule(const RowJob& job, uint32_t* mask, uint16_t* pre, int* rows) {
  const int lane = threadIdx.x & 31;
  const int BN = job.B * job.N;
  const int nwords = (BN + 31) >> 5;
  const int p_lo = min(job.first_row, BN);   // first target row of the launch
  const int P = BN - p_lo;                    // its target rows
  const int q_lo = max(job.first_row - BN, 0);  // first draft row (as a node index)
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) mask[w] = 0u;
  __syncthreads();
  // the parent entries are loaded kSchedBatch at a time (independent loads in flight)
  for (int i0 = 0; i0 < BN; i0 += kSchedBatch * (int)blockDim.x) {
    int par[kSchedBatch];
    float temp[kSchedBatch];
#pragma unroll
    for (int k = 0; k < kSchedBatch; ++k) {
      const int i = i0 + k * (int)blockDim.x + (int)threadIdx.x;
      par[k] = i < BN ? job.parents[i] : -1;
      temp[k] = (i < BN && job.req_temperature) ? job.req_temperature[i / job.N] : 1.0f;
    }
#pragma unroll
    for (int k = 0; k < kSchedBatch; ++k) {
      const int i = i0 + k * (int)blockDim.x + (int)threadIdx.x;
      if (i >= BN) continue;
      const int b = i / job.N, ch = i - b * job.N;
      // a child (a node after its parent) of a sampled tree
      if (ch == 0 || par[k] < 0 || par[k] >= ch || !(temp[k] > 0.0f)) continue;
      const int r = b * job.N + par[k];
      int word = r >> 5;
      SPEC_CHECK_INDEX(word, kSchedWords, 16);
      if (r >= q_lo) atomicOr(&mask[word], 1u << (r & 31));
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t run = 0;
    for (int w0 = 0; w0 < nwords; w0 += 32) {
      const int w = w0 + lane;
      const uint32_t c = w < nwords ? (uint32_t)__popc(mask[w]) : 0u;
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += t;
      }
      if (w < nwords) pre[w] = (uint16_t)(run + incl - c);
      run += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) pre[nwords] = (uint16_t)run;
  }
  __syncthreads();
  const int total = P + (int)pre[nwords];
  const int G = (int)gridDim.x;
  const int n_mine = total > (int)blockIdx.x ? (total - 1 - (int)blockIdx.x) / G + 1 : 0;
  for (int i = threadIdx.x; i < n_mine; i += blockDim.x) {
    const int j = (int)blockIdx.x + i * G;
    int v;
    if (j < P) {
      v = p_lo + j;
    } else {
      // the word holding the t-th needed draft row: the last word whose prefix is <= t
      const uint32_t t = (uint32_t)(j - P);
      int lo = 0, hi = nwords - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= t) lo = mid; else hi = mid - 1;
      }
      uint32_t m = mask[lo];
      for (uint32_t k = t - pre[lo]; k > 0 && m; --k) m &= m - 1u;  // drop the lower bits
      v = BN + lo * 32 + (m ? __ffs(m) - 1 : 0);
    }
    int at = i;
    SPEC_CHECK_INDEX(at, kSchedRows, 17);
    rows[at] = v;
  }
  __syncthreads();
  return n_mine;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kBlockThreads, row_blocks<MODE>()) row_pass_kernel(RowJob job) {
  constexpr int E = Elt<T>::kPerUnit;
  constexpr int U = kRingUnits;
  constexpr int S = ring_stages<MODE>();
  constexpr int CAP = Cand<T>::kCap;
  constexpr int CAPW = CAP / NW;  // candidate region of one warp
  using entry_t = typename Cand<T>::entry_t;
  __shared__ RowShared sh;
  extern __shared__ __align__(128) unsigned char dyn[];
  uint4* ring = reinterpret_cast<uint4*>(dyn);
  // (modes 0 and 1 allocate no candidate regions or scratch: those pointers are formed
  // but never used there)
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(dyn + ring_bytes<MODE>());
  uint64_t* empty_bar = full_bar + S;
  entry_t* cand = reinterpret_cast<entry_t*>(dyn + ring_bytes<MODE>() + bar_bytes<MODE>());
  unsigned char* scratch = dyn + ring_bytes<MODE>() + bar_bytes<MODE>() + cand_bytes<T>();
  unsigned* hist = reinterpret_cast<unsigned*>(scratch);
  unsigned long long* wbin = reinterpret_cast<unsigned long long*>(scratch + (size_t)kHistBins * 4);
  unsigned* ties = reinterpret_cast<unsigned*>(scratch + (size_t)kHistBins * 12);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(scratch);
  unsigned long long* pre = reinterpret_cast<unsigned long long*>(cand);  // after compaction

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int V = job.V;
  const int nunits = (V + E - 1) / E;
  const int full_units = V / E;
  const int per_iter = NT * U;
  const int niter = (nunits + per_iter - 1) / per_iter;
  const float c_launch = job.c;
  const int BN = job.B * job.N;
  const int total = (job.mode == kRowsList) ? job.R : (job.with_q ? 2 * BN : BN);
  const bool topk_on = job.top_k > 0 && job.top_k < V;
  const bool topp_on = job.top_p < 1.0f;
  entry_t* region = cand + (warp < NW ? warp : 0) * CAPW;
  const uint64_t limit = job.wait_limit_ns;
  const uint32_t row_bytes = (uint32_t)V * Elt<T>::kBytes;
  const uint32_t row_bytes16 = row_bytes & ~15u;   // the part the bulk copies move
  const int nchunks = (int)((row_bytes + kStageBytes - 1) / kStageBytes);

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full_bar[i], 1);       // the producer's arrive + the copy's bytes
      mbar_init(&empty_bar[i], NW);     // one arrive per consumer warp
    }
    sh.tmo = 0;
    sh.run_key = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  // a kernel launched after this one with programmatic stream serialization (the tree
  // walk) may be scheduled now; it waits for this grid's completion before reading
  // anything this grid writes
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  // the balanced schedule (modes 0 and 2 and list launches: every G-th virtual row)
  const bool sched = use_schedule(job, MODE, (int)gridDim.x);
  int* const sched_rows = reinterpret_cast<int*>(
      dyn + row_dyn_smem<T, MODE>() - (size_t)kSchedRows * 4);
  int n_mine = 0;
  if (sched) {
    uint32_t* const mask = reinterpret_cast<uint32_t*>(dyn + row_dyn_smem<T, MODE>() -
                                                       sched_bytes<MODE>());
    n_mine = build_schedule(job, mask, reinterpret_cast<uint16_t*>(mask + kSchedWords), sched_rows);
  }

  if (warp == NW) {
    // ---------------- producer warp ----------------
    uint32_t g = 0;  // chunks issued so far (the same count the consumers walk)
    bool stop = false;
    for (int i = 0, v0 = job.first_row + (int)blockIdx.x; !stop; ++i, v0 += gridDim.x) {
      int v = v0;
      if (sched) {
        if (i >= n_mine) break;
        v = sched_rows[i];
      } else if (v0 >= total) {
        break;
      }
      const char* row;
      if (job.mode == kRowsList) {
        row = static_cast<const char*>(row_ptr(job.base_p, (int64_t)v * job.row_pitch, Elt<T>::kBytes));
      } else {
        const bool is_q = v >= BN;
        const int r = is_q ? v - BN : v;
        const int b = r / job.N, n = r - b * job.N;
        if (!sched && is_q && job.req_temperature && !(job.req_temperature[b] > 0.0f)) continue;
        if (is_q && !sched) {
          int has_child = 0;
          for (int ch = n + 1 + lane; ch < job.N; ch += 32)
            has_child |= (job.parents[(int64_t)b * job.N + ch] == n);
          if (!__any_sync(kFull, has_child)) continue;
        }
        const int64_t off = (int64_t)b * job.batch_stride + (int64_t)n * job.row_pitch;
        row = static_cast<const char*>(row_ptr(is_q ? job.base_q : job.base_p, off, Elt<T>::kBytes));
      }
      for (int ck = 0; ck < nchunks; ++ck, ++g) {
        // lane 0 waits and issues; the warp follows its decision
        int go = 0;
        if (lane == 0) {
          const int st = (int)(g % S);
          const uint32_t use = g / S;
          if (!*((volatile int*)&sh.tmo)) {
            if (mbar_wait(&empty_bar[st], (use & 1u) ^ 1u, limit)) {
              const uint32_t off = (uint32_t)ck * kStageBytes;
              const uint32_t bytes =
                  off < row_bytes16 ? min((uint32_t)kStageBytes, row_bytes16 - off) : 0u;
              // the stall self-test announces 16 bytes more than the copy delivers, so
              // this phase never completes and the consumers' bounded wait runs out;
              // nothing more is issued after it
              const bool stall = (job.flags & SPEC_FLAG_TEST_STALL) && g == 1;
              mbar_arrive_expect_tx(&full_bar[st], bytes + (stall ? 16u : 0u));
              if (bytes) bulk_copy_g2s(ring + (size_t)st * U * NT, row + off, bytes, &full_bar[st]);
              go = stall ? 2 : 1;
            } else {
              atomicExch(&sh.tmo, 1);
            }
          }
        }
        go = __shfl_sync(kFull, go, 0);
        if (go != 1) {
          if (go == 2) ++g;  // the withheld chunk was issued
          stop = true;
          break;
        }
      }
    }
    // no copy may still be landing when the block exits: wait (bounded) for the
    // last stages issued
    if (lane == 0) {
      const uint32_t first = g > (uint32_t)S ? g - S : 0u;
      for (uint32_t h = first; h < g; ++h) mbar_wait(&full_bar[h % S], (h / S) & 1u, limit);
    }
    return;
  }

  // ---------------- consumer threads ----------------
  uint32_t g = 0;
  for (int i = 0, v0 = job.first_row + (int)blockIdx.x;; ++i, v0 += gridDim.x) {
    int v = v0;
    if (sched) {
      if (i >= n_mine) break;
      v = sched_rows[i];
    } else if (v0 >= total) {
      break;
    }
    const void* row;
    spec_row_stats* out;
    float c = c_launch;
    if (job.mode == kRowsList) {
      row = row_ptr(job.base_p, (int64_t)v * job.row_pitch, Elt<T>::kBytes);
      out = job.stats_p + v;
    } else {
      const bool is_q = v >= BN;
      const int r = is_q ? v - BN : v;
      const int b = r / job.N, n = r - b * job.N;
      if (job.req_temperature) {
        // the tree's own temperature; a greedy tree (or one with an invalid
        // temperature, which the walk reports) needs only its target rows' argmax
        const float temp = job.req_temperature[b];
        const bool sampled = temp > 0.0f && temp <= 3.402823466e38f;
        if (is_q && !(temp > 0.0f)) continue;
        c = sampled ? (float)(1.4426950408889634 / (double)temp) : 1.0f;
      }
      if (is_q && !sched) {
        // the draft row of node n is read only if some node has n as its parent
        // (every warp decides for itself, identically)
        int has_child = 0;
        for (int ch = n + 1 + lane; ch < job.N; ch += 32)
          has_child |= (job.parents[(int64_t)b * job.N + ch] == n);
        if (!__any_sync(kFull, has_child)) continue;
      }
      const int64_t off = (int64_t)b * job.batch_stride + (int64_t)n * job.row_pitch;
      row = row_ptr(is_q ? job.base_q : job.base_p, off, Elt<T>::kBytes);
      int ro = r;
      SPEC_CHECK_INDEX(ro, BN, 18);
      out = (is_q ? job.stats_q : job.stats_p) + ro;
    }
    // the block-wide running maximum starts afresh for every row (all reads of the
    // previous row's value happened before that row's last barrier)
    if (threadIdx.x == 0) sh.run_key = 0u;
    csync();

    // ---------------- streaming pass ----------------
    float Mw = -CUDART_INF_F;
    Kahan Sk;
    float best = -CUDART_INF_F;  // warp-uniform: the warp's maximum so far
    int best_idx = INT_MAX;      // and its lowest vocabulary index
    int bad = 0;
    unsigned wcount = 0;     // warp-uniform: entries this warp appended
    int overflow = 0;
    uint32_t floor16 = 0;    // bf16: key of the first window threshold
    const int full_iters = full_units / per_iter;  // iterations with no partial unit
    for (int it = 0; it < niter; ++it, ++g) {
      const int sidx = (int)(g % S);
      if (!*((volatile int*)&sh.tmo) && !mbar_wait(&full_bar[sidx], (g / S) & 1u, limit))
        atomicExch(&sh.tmo, 1);
      uint4* st = ring + (size_t)sidx * U * NT;
      uint4 raw[U];
      if (it < full_iters) {
#pragma unroll
        for (int k = 0; k < U; ++k) raw[k] = st[k * NT + threadIdx.x];
      } else {
        // the last chunk: units past the bulk copy are loaded here and parked in this
        // thread's own slots of the stage, so the window can read them back
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int u = it * per_iter + k * NT + threadIdx.x;
          if (u < full_units) {
            raw[k] = st[k * NT + threadIdx.x];
          } else {
            raw[k] = u < nunits ? Cand<T>::partial(row, V, u) : Cand<T>::neg_inf();
            st[k * NT + threadIdx.x] = raw[k];
          }
        }
      }
      const float tmax = packed_max<T, MODE == 0>(raw);
      const float wm = warp_max(tmax);
      if (wm > best) {
        // the warp maximum improved (a warp-uniform branch): every lane holding it
        // finds its first position (increasing unit, then element, is increasing
        // vocabulary index within a lane) and the warp keeps the lowest index
        int idx = INT_MAX;
        if (tmax == wm) {
#pragma unroll
          for (int k = U - 1; k >= 0; --k) {
            float fk[E];
            Elt<T>::unpack(raw[k], fk);
#pragma unroll
            for (int e = E - 1; e >= 0; --e)
              if (fk[e] == wm) idx = (it * per_iter + k * NT + threadIdx.x) * E + e;
          }
        }
        best = wm;
        best_idx = warp_min_i(idx);
      }
      if (MODE == 0) {
        bad |= (tmax != tmax);  // the NaN-propagating maximum flags a NaN
      } else {
        if (MODE == 2) {
          // publish the warp maximum; the first iteration waits for every warp so that
          // the window starts from a block-wide maximum
          if (lane == 0 && wm > -CUDART_INF_F) atomicMax(&sh.run_key, order_key(wm));
          if (it == 0) {
            csync();
            const unsigned rk0 = sh.run_key;
            if (sizeof(T) == 2 && rk0)
              floor16 = order_key(__bfloat162float(
                            __float2bfloat16_rd(key_value(rk0) - job.delta_z))) >> 16;
          }
        }
        if (wm > Mw) {
          if (Mw != -CUDART_INF_F) {
            const float scale = ex2_approx((Mw - wm) * c);
            Sk.s *= scale;
            Sk.c *= scale;
          }
          Mw = wm;
        }
        float f[U][E];
#pragma unroll
        for (int k = 0; k < U; ++k) Elt<T>::unpack(raw[k], f[k]);
        if (Mw == -CUDART_INF_F) {  // nothing finite yet: only NaN can hide here
#pragma unroll
          for (int k = 0; k < U; ++k)
#pragma unroll
            for (int e = 0; e < E; ++e) bad |= (f[k][e] != f[k][e]);
        } else {
          // 2^((z - Mw) c) for pairs of logits: packed fp32 FMAs and adds
          const float negMc = -Mw * c;
          const float2 c2 = make_float2(c, c), n2 = make_float2(negMc, negMc);
          float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int k = 0; k < U; ++k)
#pragma unroll
            for (int e = 0; e < E; e += 2) {
              const float2 a = __ffma2_rn(make_float2(f[k][e], f[k][e + 1]), c2, n2);
              acc[(e >> 1) & 1] = __fadd2_rn(acc[(e >> 1) & 1], make_float2(ex2_approx(a.x), ex2_approx(a.y)));
            }
          const float2 tot = __fadd2_rn(acc[0], acc[1]);
          Sk.add(tot.x + tot.y);
          if (MODE == 2) {
            const unsigned rk = *((volatile unsigned*)&sh.run_key);
            const float bmax = rk ? fmaxf(Mw, key_value(rk)) : Mw;
            const float thr = bmax - job.delta_z;
            const __nv_bfloat162 t2 = __bfloat162bfloat162(__float2bfloat16_rd(thr));
            unsigned mask = window_mask<T>(raw, f, t2, thr);
            if (__any_sync(kFull, mask != 0)) {
              // append to this warp's region; no atomics: offsets from a warp scan
              const unsigned mine = __popc(mask);
              unsigned incl = mine;
#pragma unroll
              for (int o = 1; o < 32; o <<= 1) {
                const unsigned t = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += t;
              }
              unsigned pos = wcount + incl - mine;
              wcount += __shfl_sync(kFull, incl, 31);
              const unsigned char* stb = reinterpret_cast<const unsigned char*>(st);
              while (mask) {
                const int bit = __ffs(mask) - 1;
                mask &= mask - 1;
                int k, e;
                const uint32_t off = window_slot<T>(bit, k, e);
                const uint32_t idx = (uint32_t)((it * per_iter + k * NT + threadIdx.x) * E + e);
                if constexpr (sizeof(T) == 2) {
                  const uint32_t zb = *reinterpret_cast<const unsigned short*>(stb + off);
                  const uint32_t rel = key16_bits(zb) - floor16;
                  if (pos < (unsigned)CAPW && rel < (uint32_t)kHistBins)
                    region[pos] = (idx << kKeySpanBits) | rel;
                  else
                    overflow = 1;
                } else {
                  const uint32_t zb = *reinterpret_cast<const uint32_t*>(stb + off);
                  if (pos < (unsigned)CAPW) region[pos] = make_uint2(idx, zb);
                  else overflow = 1;
                }
                ++pos;
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[sidx]);  // this warp is done with the stage
    }
    // ---------------- block combine ----------------
    {
      const FF ws = warp_sum_ff(Sk.ff());
      const float wb = best;
      const int wbad = __any_sync(kFull, bad);
      const int wof = __any_sync(kFull, overflow);
      if (lane == 0) {
        sh.warp_m[warp] = Mw;
        sh.warp_s[warp] = ws.value();
        sh.warp_best[warp] = wb;
        sh.warp_bad[warp] = wbad;
        sh.wcnt[warp] = wcount;
        sh.woverflow[warp] = wof || wcount > (unsigned)CAPW;
      }
    }
    csync();
    if (threadIdx.x == 0) {
      float m = -CUDART_INF_F;
      int anybad = 0;
      for (int w = 0; w < NW; ++w) {
        m = fmaxf(m, sh.warp_best[w]);
        anybad |= sh.warp_bad[w];
      }
      double s = 0.0;
      if (MODE != 0) {
        for (int w = 0; w < NW; ++w)
          if (sh.warp_m[w] != -CUDART_INF_F) s += sh.warp_s[w] * (double)exp2f((sh.warp_m[w] - m) * c);
      }
      const bool finite = !anybad && m != CUDART_INF_F && m != -CUDART_INF_F && !(m != m) &&
                          (MODE == 0 || (s == s && s != CUDART_INF));
      sh.m = m;
      sh.s_total = s;
      sh.argmax = INT_MAX;
      // a timed-out wait leaves the row's data unknown
      sh.bad = *((volatile int*)&sh.tmo) ? SPEC_ROW_TIMEOUT : (finite ? 0 : SPEC_ROW_NONFINITE);
      if (job.counters) {
        atomicAdd(&job.counters[0], 1ull);
        atomicAdd(&job.counters[1], (unsigned long long)V * Elt<T>::kBytes);
      }
    }
    csync();
    // argmax: the lowest index among the warps holding the maximum
    if (lane == 0 && best == sh.m && best_idx != INT_MAX) atomicMin(&sh.argmax, best_idx);
    csync();
    if (threadIdx.x == 0 && sh.argmax == INT_MAX) sh.argmax = 0;
    csync();
    const float m = sh.m;
    const int argmax = sh.argmax;

    if (sh.bad) {
      if (threadIdx.x == 0) {
        spec_row_stats st;
        st.m = m; st.status = sh.bad; st.s_f = 0.0; st.cut_key = 0;
        st.cut_idx = -1; st.argmax = argmax; st.kept = 0;
        *out = st;
      }
      csync();
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
      csync();
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
    const float thr = m - job.delta_z;
    int any_overflow = 0;
    for (int w = 0; w < NW; ++w) any_overflow |= sh.woverflow[w];
    const bool window_ok = !(job.flags & SPEC_FLAG_EXACT_SELECT) && !any_overflow;
    if constexpr (sizeof(T) == 2) {
      const uint32_t K16m = order_key(m) >> 16;
      const uint32_t K16thr = order_key(thr) >> 16;  // lowest key the window can hold
      // a stored maximum bounds the window by kHistBins keys; check it regardless and
      // leave any wider window to the exact selection
      const bool fits = K16m - K16thr < (uint32_t)kHistBins;
      if (window_ok && fits) {
        // ---- bf16 window: one bin per key below the maximum ----
        const int nb = (int)(K16m - K16thr) + 1;
        for (int i = threadIdx.x; i < nb; i += NT) hist[i] = 0u;
        csync();
        {
          const int n_own = min((int)sh.wcnt[warp], CAPW);  // each warp reads its own region
          for (int i = lane; i < n_own; i += 32) {
            const uint32_t k16 = floor16 + (region[i] & (kHistBins - 1));
            const uint32_t bin = K16m - k16;
            if (bin < (uint32_t)nb && key_value(key_from16(k16)) >= thr) atomicAdd(&hist[bin], 1u);
          }
        }
        csync();
        if (warp == 0) {
          // one warp scans the bins in key order: lane l owns bins [l*C, (l+1)*C)
          const int C = (nb + 31) / 32;
          const int b_lo = lane * C, b_hi = min(nb, b_lo + C);
          unsigned lc = 0;
          unsigned long long lw = 0;
          for (int bin = b_lo; bin < b_hi; ++bin) {
            const unsigned long long wgt =
                to_fixed(tempered_weight(key_value(key_from16(K16m - (uint32_t)bin)), m, c));
            wbin[bin] = wgt;
            lc += hist[bin];
            lw += (unsigned long long)hist[bin] * wgt;
          }
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
              if (lane == 0) {
                sh.sel_bcut = b_k;
                sh.sel_jcut = jk;
                sh.sel_kept = K;
                sh.sel_sf = s_k;
              }
            }
          }
          if (ok && topp_on) {
            const unsigned long long tau = (unsigned long long)ceil(
                (double)job.top_p * (topk_on ? (double)s_k : s_total * tau_scale));
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
              unsigned j = avail;
              if (w1 > 0) {
                const unsigned long long jj = (tau - rw2 + w1 - 1) / w1;
                j = (unsigned)(jj < 1 ? 1 : (jj > avail ? avail : jj));
              }
              if (lane == 0) {
                sh.sel_bcut = b_p;
                sh.sel_jcut = j;
                sh.sel_kept = rc + j;
                sh.sel_sf = rw2 + (unsigned long long)j * w1;
              }
            }
          }
          if (lane == 0) {
            sh.sel_ok = ok;
            if (ok) {
              sh.sel_ncut = hist[sh.sel_bcut];
              sh.sel_cutkey = key_from16(K16m - (uint32_t)sh.sel_bcut);
            }
            sh.tie_n = 0;
            sh.tie_idx = (sh.sel_ok && sh.sel_jcut == sh.sel_ncut) ? -1 : INT_MAX;
          }
        }
        csync();
        if (sh.sel_ok) {
          const uint32_t ck16 = sh.sel_cutkey >> 16;
          const unsigned jc = sh.sel_jcut, nc = sh.sel_ncut;
          if (jc == nc) {
            // the whole group of the cut key is kept: the cut is its largest index
            const int n_own = min((int)sh.wcnt[warp], CAPW);
            for (int i = lane; i < n_own; i += 32) {
              const uint32_t e = region[i];
              if (floor16 + (e & (kHistBins - 1)) == ck16) atomicMax(&sh.tie_idx, (int)(e >> kKeySpanBits));
            }
            csync();
          } else if (nc <= (unsigned)kTieCap) {
            // the jc-th member of the cut key in index order: rank the members
            const int n_own = min((int)sh.wcnt[warp], CAPW);
            for (int i = lane; i < n_own; i += 32) {
              const uint32_t e = region[i];
              if (floor16 + (e & (kHistBins - 1)) == ck16) {
                const unsigned pos = atomicAdd(&sh.tie_n, 1u);
                if (pos < (unsigned)kTieCap) ties[pos] = e >> kKeySpanBits;
              }
            }
            csync();
            const unsigned nt = min(sh.tie_n, (unsigned)kTieCap);
            for (unsigned i = threadIdx.x; i < nt; i += NT) {
              const unsigned me = ties[i];
              unsigned rank = 0;
              for (unsigned t = 0; t < nt; ++t) rank += (ties[t] < me);
              if (rank + 1 == jc) sh.tie_idx = (int)me;
            }
            csync();
          } else if (threadIdx.x == 0) {
            sh.sel_ok = 0;
          }
          csync();
          if (sh.sel_ok) {
            done = true;
            cut_key = sh.sel_cutkey;
            cut_idx = sh.tie_idx;
            kept = sh.sel_kept;
            sf_fixed = sh.sel_sf;
          }
        }
        csync();
      }
    } else {
      if (window_ok) {
        // ---- fp32 window: sorted by (key desc, index asc) ----
        if (threadIdx.x == 0) sh.n_keep = 0;
        csync();
        {
          const int n_own = min((int)sh.wcnt[warp], CAPW);
          for (int i = lane; i < n_own; i += 32) {
            const uint2 e = region[i];
            const float z = __uint_as_float(e.y);
            if (z >= thr) {
              const unsigned pos = atomicAdd(&sh.n_keep, 1u);
              if (pos < (unsigned)kSortCap)
                keys[pos] = ((unsigned long long)order_key(z) << 32) | (unsigned long long)(~e.x);
            }
          }
        }
        csync();
        const unsigned n_c = sh.n_keep;
        if (n_c >= 1 && n_c <= (unsigned)kSortCap && (!topk_on || n_c >= K)) {
          unsigned n_pad = 2;
          while (n_pad < n_c) n_pad <<= 1;
          for (unsigned i = n_c + threadIdx.x; i < n_pad; i += NT) keys[i] = 0ull;
          csync();
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
              csync();
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
          block_exscan<CSync>(0u, run, bc, bw, tc, tw, sh.sel);
#pragma unroll
          for (int t = 0; t < C; ++t) pre[lo + t] += bw;
          if (threadIdx.x == 0) sh.first = INT_MAX;
          csync();
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
            csync();
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
        csync();
      }
    }
    if (!done) {
      // exact full-row selection
      SelOut rk{};
      const Eligible all{false, 0u, 0};
      NoReduce one;
      if (topk_on)
        rk = exact_select<T, CSync>(row, V, m, c, false, K, 0ull, all, sh.sel, 0, nunits, one);
      if (topp_on) {
        const Eligible in_k{topk_on, rk.key, rk.idx};
        const unsigned long long tau = (unsigned long long)ceil(
            (double)job.top_p * (topk_on ? (double)rk.mass_kept : s_total * tau_scale));
        const SelOut rp =
            exact_select<T, CSync>(row, V, m, c, true, 0u, tau, in_k, sh.sel, 0, nunits, one);
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
    csync();
  }
}

template <typename T, int MODE>
cudaError_t launch_mode(const RowJob& job, int num_rows, cudaStream_t s) {
  const size_t dyn = row_dyn_smem<T, MODE>();
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
  int grid = device_sm_count() * row_blocks<MODE>();  // persistent blocks
  if (grid > num_rows) grid = num_rows;
  if (grid < 1) grid = 1;
  row_pass_kernel<T, MODE><<<grid, kBlockThreads, dyn, s>>>(job);
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

// Checked builds: this translation unit's error word, read and cleared (0 in other
// builds).  Synchronous: it waits for the device.
uint32_t check_word_rows() {
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
