// internal.h -- launch descriptors and the workspace layout shared by the
// translation units of the verify library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/spec_verify.h"

namespace svk {

constexpr int kRowThreads = 512;   // threads of one row-pass block
constexpr int kRowBlocksPerSm = 2; // resident row-pass blocks per SM
constexpr int kCandCap = 8192;     // candidate-window capacity, (index, logit) entries
constexpr int kSortCap = 4096;     // largest window resolved by sorting (fp32 / wide windows)
constexpr int kHistBins = 4096;    // one bin per bf16 key below the row maximum
constexpr int kTieCap = 1024;      // largest group of equal logits cut by index ranking
constexpr int kWalkThreads = 1024; // threads of one tree-walk block
// Width of the single-pass candidate window below the running row maximum, in
// nats of the tempered distribution (tokens further below carry < e^-9 of the top
// token's weight each).  When the window misses the top-k / top-p cut, or holds
// more tokens than fit, the row falls back to the exact full-row selection.
constexpr float kWindowNats = 9.0f;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t stats_p, stats_q, child_start, child_list, need_q, tree_info, resid_z, resid_invz,
      counters, total;
};

// Workspace sections for B trees of N nodes: row statistics of every p row and of
// every q row, the children of each node in index order (CSR), a per-node flag
// "q row needed", per-tree status, the residual masses Z_1..Z_j of the node the
// walk is at (at most N - 1 per tree) with their fp32 reciprocals, and the work
// counters.
inline WsLayout ws_layout(int32_t B, int32_t N) {
  WsLayout L{};
  size_t bn = (size_t)B * (size_t)N;
  size_t off = 0;
  L.stats_p = off;     off = align_up(off + bn * sizeof(spec_row_stats), 256);
  L.stats_q = off;     off = align_up(off + bn * sizeof(spec_row_stats), 256);
  L.child_start = off; off = align_up(off + (size_t)B * (N + 1) * sizeof(int32_t), 256);
  L.child_list = off;  off = align_up(off + bn * sizeof(int32_t), 256);
  L.need_q = off;      off = align_up(off + bn * sizeof(uint8_t), 256);
  L.tree_info = off;   off = align_up(off + (size_t)B * sizeof(int32_t), 256);
  L.resid_z = off;     off = align_up(off + bn * sizeof(double), 256);
  L.resid_invz = off;  off = align_up(off + bn * sizeof(float), 256);
  L.counters = off;    off = align_up(off + sizeof(spec_verify_counters), 256);
  L.total = off;
  return L;
}

// One dense row pass launch.  Mode kRowsList: row r at base_p + r * row_pitch
// (spec_filter_rows).  Mode kRowsTree: virtual rows [0, B*N) are the p rows
// (b, n), and when q is needed [B*N, 2*B*N) the q rows, skipped unless need_q.
enum RowMode { kRowsList = 0, kRowsTree = 1 };

struct RowJob {
  const void* base_p;
  const void* base_q;
  int64_t row_pitch;
  int64_t batch_stride;
  int32_t V, N, B, R;
  int32_t mode;
  int32_t with_q;
  const uint8_t* need_q;
  spec_row_stats* stats_p;
  spec_row_stats* stats_q;
  float temperature;
  float c;        // log2(e) / T
  float delta_z;  // candidate window in logit units (kWindowNats * T)
  int32_t top_k;  // 0: off
  float top_p;    // >= 1: off
  uint32_t flags;
  unsigned long long* counters;  // spec_verify_counters as an array of 8 u64, or null
};

struct TreeJob {
  const void* base_p;
  const void* base_q;
  int64_t row_pitch;
  int64_t batch_stride;
  int32_t V, N, B, W;
  const int32_t* tokens;
  const int32_t* parents;
  int32_t* child_start;
  int32_t* child_list;
  uint8_t* need_q;
  int32_t* tree_info;
  const spec_row_stats* stats_p;
  const spec_row_stats* stats_q;
  double* resid_z;
  float* resid_invz;
  float temperature;
  float c;
  uint64_t seed, offset;
  int32_t* out_accept_len;
  int32_t* out_tokens;
  int32_t* out_path;
  float* out_alpha;
  int32_t* out_status;
  unsigned long long* counters;
};

// Launchers (each returns cudaGetLastError() of its launch).
cudaError_t launch_row_pass(const RowJob& job, spec_dtype dtype, int num_rows, cudaStream_t s);
cudaError_t launch_tree_prep(const TreeJob& job, bool greedy, cudaStream_t s);
cudaError_t launch_tree_walk(const TreeJob& job, spec_dtype dtype, bool greedy, cudaStream_t s);
cudaError_t launch_philox_words(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                                const int32_t* node_idx, int32_t n, uint32_t* out,
                                cudaStream_t s);
int device_sm_count();

}  // namespace svk
