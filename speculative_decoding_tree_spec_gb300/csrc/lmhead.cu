// lmhead.cu -- the fused LM head of the verify step: the target logits
// p = F W^T (F [M, d] node features, W [V, d] LM-head weight, both bf16) computed on
// the fifth-generation tensor cores, and in the same kernel the per-(row, column
// tile) statistics the verify step needs from every target row (maximum, its first
// index, sum of tempered weights).  A combine kernel turns them into row
// statistics; the draft rows take the dense row pass and the walk runs as for
// given logits.  (EAGLE computes the target's next-token distribution of every tree
// node from its features with the LM head: "EAGLE close reading", edgeai1.github.io,
// section 3; the verify step then follows the pages cited in walk.cu.)
//
// GEMM: persistent, one CTA per SM, 128 x 256 output tiles, K in steps of 64.
//   warp 0      TMA producer: A (128 x 64) and B (256 x 64) bf16 tiles with the
//               128-byte swizzle into a 4-stage shared-memory ring (mbarrier
//               complete_tx)
//   warp 1      TMEM owner; one lane issues tcgen05.mma kind::f16 (M 128, N 256,
//               K 16) into two 256-column fp32 accumulators; tcgen05.commit frees a
//               stage once its MMAs are done and publishes a finished accumulator
//   warps 2-5   epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (one output row
//               per thread) with tcgen05.ld, rounds to bf16, writes the logits once,
//               and keeps the row's running maximum, first argmax and sum of
//               2^((z - max) log2(e) / T) over the tile's columns
// Every mbarrier wait is bounded by %globaltimer: on a timeout the error flag is set,
// every role stops, and the kernel waits (bounded) for its own copies and MMAs
// before it frees the TMEM.
#include <cuda.h>

#include <climits>

#include <cuda_bf16.h>

#include "common.cuh"

namespace svk {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, UK = 16;
constexpr int kStages = 4;
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;  // 32 KB
constexpr int kEpiWarps = 4;
constexpr int kLmThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 2 * BN;  // two accumulators
constexpr size_t kLmSmem = 1024 + (size_t)kStages * (kABytes + kBBytes);

// tcgen05 instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

struct LmShared {
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], done;
  uint32_t tmem;
};

// Shared-memory matrix descriptor of a K-major tile written by TMA with the 128-byte
// swizzle: rows of 128 bytes in 1024-byte groups of 8 (stride byte offset 1024),
// descriptor version 1, layout "128-byte swizzle".  The tile base is 1024-aligned.
__device__ __forceinline__ uint64_t sw128_desc(const void* p) {
  const uint32_t a = smem_u32(p);
  uint64_t d = (uint64_t)((a >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;               // leading byte offset (unused by this layout)
  d |= (uint64_t)(1024u >> 4) << 32;     // stride byte offset
  d |= (uint64_t)1u << 46;               // version
  d |= (uint64_t)2u << 61;               // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 16 consecutive fp32 accumulator columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Statistics of one row over one 256-column tile.
struct TilePart {
  float m;      // maximum of the bf16 logits (-inf: no column)
  float s_hi;   // sum of 2^((z - m) c) as a float-float pair
  float s_lo;
  int arg;      // lowest column holding m
};

struct LmJob {
  int M, V, K;
  int m_tiles, n_tiles;
  float c;          // log2(e) / T (0 at T = 0: no sums)
  uint16_t* p;      // [M] rows of the bf16 logits, row r at p + r * pitch
  int64_t pitch;
  TilePart* part;   // [n_tiles][M]
  int* err;
  uint64_t wait_limit_ns;
};

__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  LmJob job) {
  __shared__ LmShared sh;
  extern __shared__ unsigned char lm_dyn[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(lm_dyn) + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = base;
  unsigned char* sB = base + (size_t)kStages * kABytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = job.m_tiles * job.n_tiles;
  const int KB = (job.K + BK - 1) / BK;
  const uint64_t limit = job.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.tfull[a], 1);
      mbar_init(&sh.tempty[a], kEpiWarps);
    }
    mbar_init(&sh.done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(&sh.tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < tiles && !stop; t += gridDim.x) {
        const int mt = t % job.m_tiles, nt = t / job.m_tiles;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = (int)(it % kStages);
          const uint32_t ph = (it / kStages) & 1u;
          if (*((volatile int*)job.err) || !mbar_wait(&sh.empty[s], ph ^ 1u, limit)) {
            atomicExch(job.err, 1);
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(&sh.full[s], kABytes + kBBytes);
          tma_load_2d(sA + (size_t)s * kABytes, &tmA, kb * BK, mt * BM, &sh.full[s]);
          tma_load_2d(sB + (size_t)s * kBBytes, &tmB, kb * BK, nt * BN, &sh.full[s]);
        }
      }
      // no copy may still be landing when the CTA exits: wait (bounded) for the
      // last stages issued
      const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0u;
      for (uint32_t h = first; h < it; ++h)
        mbar_wait(&sh.full[h % kStages], (h / kStages) & 1u, limit);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, lt = 0;
      bool stop = false;
      for (int t = blockIdx.x; t < tiles && !stop; t += gridDim.x, ++lt) {
        const int acc = (int)(lt & 1u);
        const uint32_t aph = (lt >> 1) & 1u;
        if (!mbar_wait(&sh.tempty[acc], aph ^ 1u, limit)) {
          atomicExch(job.err, 1);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = (int)(it % kStages);
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait(&sh.full[s], ph, limit)) {
            atomicExch(job.err, 1);
            stop = true;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sw128_desc(sA + (size_t)s * kABytes);
          const uint64_t bdesc = sw128_desc(sB + (size_t)s * kBBytes);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k) {
            // the next 16 K-elements are 32 bytes further along the swizzled rows
            const uint64_t koff = (uint64_t)((k * UK * 2) >> 4);
            tc_mma(d_tmem, adesc + koff, bdesc + koff, kIdesc, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(&sh.empty[s]);  // the stage is free once these MMAs are done
        }
        if (stop) break;
        tc_commit(&sh.tfull[acc]);  // the accumulator is complete
      }
      // every MMA issued has finished before the TMEM is freed
      tc_commit(&sh.done);
      mbar_wait(&sh.done, 0u, limit);
    }
  } else {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;  // this warp's TMEM lanes: 32 quarter .. +31
    const float c = job.c;
    uint32_t lt = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++lt) {
      const int acc = (int)(lt & 1u);
      const uint32_t aph = (lt >> 1) & 1u;
      // the whole warp takes one decision (the TMEM loads below are warp-collective)
      const bool ready = __all_sync(kFull, !*((volatile int*)job.err) &&
                                               mbar_wait(&sh.tfull[acc], aph, limit));
      if (!ready) {
        if (lane == 0) atomicExch(job.err, 1);
        break;
      }
      tc_fence_after();
      const int mt = t % job.m_tiles, nt = t / job.m_tiles;
      const int row = mt * BM + quarter * 32 + lane;
      const int n0 = nt * BN;
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      uint16_t* prow = job.p + (int64_t)row * job.pitch;
      float m = -CUDART_INF_F;
      int arg = 0;
      Kahan Sk;
#pragma unroll 1
      for (int ch = 0; ch < BN / 16; ++ch) {
        float v[16];
        tmem_ld16(taddr + (uint32_t)(ch * 16), v);
        const int col0 = n0 + ch * 16;
        uint32_t packed[8];
        float z[16];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(v[i], v[i + 1]);
          packed[i / 2] = *reinterpret_cast<const uint32_t*>(&h);
          z[i] = __low2float(h);
          z[i + 1] = __high2float(h);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (col0 + i >= job.V) z[i] = -CUDART_INF_F;
        if (row < job.M) {
          if (col0 + 16 <= job.V) {
            uint4* dst = reinterpret_cast<uint4*>(prow + col0);
            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
          } else {
            for (int i = 0; i < 16 && col0 + i < job.V; ++i)
              prow[col0 + i] = (uint16_t)(packed[i / 2] >> (16 * (i & 1)));
          }
        }
        // running maximum (first index), then the sum referred to it
        float cm = z[0];
#pragma unroll
        for (int i = 1; i < 16; ++i) cm = fmaxf(cm, z[i]);
        if (cm > m) {
          int first = 15;
#pragma unroll
          for (int i = 15; i >= 0; --i)
            if (z[i] == cm) first = i;
          arg = col0 + first;
          if (c > 0.f && m != -CUDART_INF_F) {
            const float scale = ex2_approx((m - cm) * c);
            Sk.s *= scale;
            Sk.c *= scale;
          }
          m = cm;
        }
        if (c > 0.f && m != -CUDART_INF_F) {
          float part = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) part += tempered_weight(z[i], m, c);
          Sk.add(part);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.tempty[acc]);  // the accumulator may be reused
      if (row < job.M) {
        const FF f = Sk.ff();
        TilePart tp;
        tp.m = m;
        tp.s_hi = f.hi;
        tp.s_lo = f.lo;
        tp.arg = arg;
        job.part[(int64_t)nt * job.M + row] = tp;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  __syncwarp();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// Row statistics from the tiles' statistics (one warp per row), in the form the
// dense row pass writes them (no truncation recorded; T = 0: one-hot argmax).
__global__ void lmhead_combine_kernel(const TilePart* part, int M, int n_tiles, float c,
                                      int greedy, const int* err, spec_row_stats* stats,
                                      unsigned long long* counters, int V) {
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= M) return;
  float m = -CUDART_INF_F;
  for (int t = lane; t < n_tiles; t += 32) m = fmaxf(m, part[(int64_t)t * M + warp].m);
  m = warp_max(m);
  FF s;
  int arg = INT_MAX;
  int bad = 0;
  for (int t = lane; t < n_tiles; t += 32) {
    const TilePart tp = part[(int64_t)t * M + warp];
    bad |= (tp.m != tp.m);
    if (tp.m == m && tp.arg < arg) arg = tp.arg;
    if (!greedy && tp.m != -CUDART_INF_F) {
      const float scale = exp2f((tp.m - m) * c);
      s.add(tp.s_hi * scale);
      s.add(tp.s_lo * scale);
    }
  }
  s = warp_sum_ff(s);
  arg = warp_min_i(arg);
  bad = __any_sync(kFull, bad);
  if (lane == 0) {
    const double st = s.value();
    const bool finite = !bad && m != CUDART_INF_F && m != -CUDART_INF_F &&
                        (greedy || (st == st && st != CUDART_INF));
    spec_row_stats r;
    r.m = m;
    r.status = *err ? SPEC_ROW_TIMEOUT : (finite ? SPEC_TREE_OK : SPEC_ROW_NONFINITE);
    r.argmax = (arg == INT_MAX) ? 0 : arg;
    if (greedy) {
      r.s_f = 1.0;
      r.cut_key = order_key(m);
      r.cut_idx = r.argmax;
      r.kept = 1;
    } else {
      r.s_f = st;
      r.cut_key = 0u;
      r.cut_idx = V - 1;
      r.kept = V;
    }
    stats[warp] = r;
    if (counters) atomicAdd(&counters[0], 1ull);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D tensor map of a row-major [rows, K] bf16 matrix, box [box_rows, 64], 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, int rows, int K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t lmhead_part_bytes(int M, int V) {
  const int n_tiles = (V + BN - 1) / BN;
  return (size_t)n_tiles * (size_t)M * sizeof(TilePart);
}

cudaError_t launch_lmhead(const void* features, const void* weight, int M, int V, int K,
                          float temperature, void* p, int64_t pitch, void* part, int* err,
                          spec_row_stats* stats, unsigned long long* counters, cudaStream_t s) {
  CUtensorMap tmA, tmB;
  if (!make_map(&tmA, features, M, K, BM) || !make_map(&tmB, weight, V, K, BN))
    return cudaErrorInvalidValue;
  LmJob job{};
  job.M = M;
  job.V = V;
  job.K = K;
  job.m_tiles = (M + BM - 1) / BM;
  job.n_tiles = (V + BN - 1) / BN;
  job.c = temperature > 0.f ? (float)(1.4426950408889634 / (double)temperature) : 0.f;
  job.p = static_cast<uint16_t*>(p);
  job.pitch = pitch;
  job.part = static_cast<TilePart*>(part);
  job.err = err;
  job.wait_limit_ns = 2000000000ull;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kLmSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const int tiles = job.m_tiles * job.n_tiles;
  int grid = device_sm_count();
  if (grid > tiles) grid = tiles;
  lmhead_kernel<<<grid, kLmThreads, kLmSmem, s>>>(tmA, tmB, job);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int threads = 256;
  const int blocks = (M * 32 + threads - 1) / threads;
  lmhead_combine_kernel<<<blocks, threads, 0, s>>>(job.part, M, job.n_tiles, job.c,
                                                   temperature == 0.f ? 1 : 0, err, stats,
                                                   counters, V);
  return cudaGetLastError();
}

cudaError_t launch_lmhead_logits(const void* features, const void* weight, int M, int V, int K,
                                 void* p, int64_t pitch, void* part, int* err, cudaStream_t s) {
  CUtensorMap tmA, tmB;
  if (!make_map(&tmA, features, M, K, BM) || !make_map(&tmB, weight, V, K, BN))
    return cudaErrorInvalidValue;
  LmJob job{};
  job.M = M;
  job.V = V;
  job.K = K;
  job.m_tiles = (M + BM - 1) / BM;
  job.n_tiles = (V + BN - 1) / BN;
  job.c = 0.f;  // no sums: the caller ranks the written rows itself
  job.p = static_cast<uint16_t*>(p);
  job.pitch = pitch;
  job.part = static_cast<TilePart*>(part);
  job.err = err;
  job.wait_limit_ns = 2000000000ull;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kLmSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const int tiles = job.m_tiles * job.n_tiles;
  int grid = device_sm_count();
  if (grid > tiles) grid = tiles;
  lmhead_kernel<<<grid, kLmThreads, kLmSmem, s>>>(tmA, tmB, job);
  return cudaGetLastError();
}

}  // namespace svk
