// commit.cu -- accepted-path commit: after a verify step, move the cache entries of
// each tree's accepted path to consecutive positions after its prefix, in every
// plane of a strided cache (target or draft KV cache, or the features), so the
// caches continue the accepted sequence ("EAGLE close reading", edgeai1.github.io,
// section 5: both caches are trimmed to what was accepted).
//
// Node n of tree b sits at position prefix_len[b] + n; position prefix_len[b] + k
// receives node path[b][k] for k = 1 .. accept_len[b] (k = 0 is the root, already in
// place).  A path increases strictly (parents precede children), so path[b][k] >= k;
// one thread owns each 16-byte column of a (plane, tree) and no other thread touches
// its bytes.
#include "common.cuh"

namespace svk {

namespace {

constexpr int kCommitThreads = 256;

struct CommitJob {
  unsigned char* cache;
  int B, n_planes, n_pos, W;
  int64_t plane_stride, batch_stride, pos_stride;  // bytes
  int64_t row_bytes;                               // multiple of 16
  const int32_t* prefix_len;
  const int32_t* path;
  const int32_t* accept_len;
};

constexpr int kBatchMoves = 8;  // moves whose sources one thread loads before storing

// One thread per (plane, tree, 16-byte column) item, grid-stride.  The moves of a tree
// are taken in batches of kBatchMoves in increasing k: a batch loads all its sources,
// then stores all its destinations.  Sources of later batches lie above every
// destination of earlier ones (path[k] >= k), so nothing is read after it is
// overwritten.
__global__ void __launch_bounds__(kCommitThreads) commit_kernel(CommitJob job) {
  const int64_t nvec = job.row_bytes / 16;
  const int64_t total = (int64_t)job.B * job.n_planes * nvec;
  for (int64_t item = (int64_t)blockIdx.x * kCommitThreads + threadIdx.x; item < total;
       item += (int64_t)gridDim.x * kCommitThreads) {
    const int64_t pair = item / nvec, v = item - pair * nvec;
    const int b = (int)(pair % job.B);
    const int plane = (int)(pair / job.B);
    const int a = min(job.accept_len[b], job.W - 1);
    if (a <= 0) continue;
    const int base = job.prefix_len[b];
    const int32_t* path = job.path + (int64_t)b * job.W;
    unsigned char* col = job.cache + plane * job.plane_stride + (int64_t)b * job.batch_stride + v * 16;
    for (int k0 = 1; k0 <= a; k0 += kBatchMoves) {
      uint4 x[kBatchMoves];
      int dst[kBatchMoves];
#pragma unroll
      for (int i = 0; i < kBatchMoves; ++i) {
        const int k = k0 + i;
        dst[i] = -1;
        if (k <= a) {
          const int src = base + path[k], d = base + k;
          if (src != d && src >= 0 && src < job.n_pos && d < job.n_pos) {
            x[i] = *reinterpret_cast<const uint4*>(col + src * job.pos_stride);
            dst[i] = d;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kBatchMoves; ++i)
        if (dst[i] >= 0) *reinterpret_cast<uint4*>(col + dst[i] * job.pos_stride) = x[i];
    }
  }
}

}  // namespace

}  // namespace svk

using namespace svk;

extern "C" int spec_commit_accepted_path(void* cache, int32_t B, int32_t n_planes, int32_t n_pos,
                                         int64_t plane_stride, int64_t batch_stride,
                                         int64_t pos_stride, int64_t row_bytes,
                                         const int32_t* prefix_len,
                                         const int32_t* accepted_path,
                                         const int32_t* accept_len, int32_t W,
                                         spec_stream_t stream) {
  if (B < 0 || n_planes < 0 || n_pos < 0 || W < 1 || row_bytes < 0) return SPEC_ERR_INVALID_ARG;
  if (B == 0 || n_planes == 0 || row_bytes == 0) return SPEC_OK;
  if (!cache || !prefix_len || !accepted_path || !accept_len) return SPEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(cache) & 15u) || (plane_stride & 15) || (batch_stride & 15) ||
      (pos_stride & 15) || (row_bytes & 15))
    return SPEC_ERR_MISALIGNED;
  if (row_bytes > pos_stride && n_pos > 1) return SPEC_ERR_INVALID_ARG;  // rows may not overlap
  const int64_t pairs = (int64_t)B * n_planes;
  if (pairs > 0x7fffffff) return SPEC_ERR_TOO_LARGE;
  CommitJob job{};
  job.cache = static_cast<unsigned char*>(cache);
  job.B = B;
  job.n_planes = n_planes;
  job.n_pos = n_pos;
  job.W = W;
  job.plane_stride = plane_stride;
  job.batch_stride = batch_stride;
  job.pos_stride = pos_stride;
  job.row_bytes = row_bytes;
  job.prefix_len = prefix_len;
  job.path = accepted_path;
  job.accept_len = accept_len;
  const int64_t items = pairs * (row_bytes / 16);
  int64_t blocks = (items + kCommitThreads - 1) / kCommitThreads;
  const int64_t cap = (int64_t)device_sm_count() * 16;  // grid-stride beyond this
  if (blocks > cap) blocks = cap;
  commit_kernel<<<(unsigned)blocks, kCommitThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(job);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
