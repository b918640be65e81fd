// internal.h -- launch descriptors and the workspace layout shared by the
// translation units of the verify library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

namespace svk {

constexpr int kRowThreads = 256;   // consumer threads of one row-pass block (+ 1 producer warp)
constexpr int kRowBlocksPerSm = 2; // resident row-pass blocks per SM
constexpr int kRingStages = 3;     // bulk-copy stages of the row pass's shared-memory ring
constexpr int kRingUnits = 4;      // 16-byte units per consumer thread per stage
constexpr int kCandCapBf16 = 8192; // candidate-window capacity for bf16 rows (32-bit entries)
constexpr int kCandCapF32 = 4096;  // candidate-window capacity for fp32 rows (index + logit)
constexpr int kKeySpanBits = 11;   // bf16 entries: key offset above the row's floor key
constexpr int kSortCap = 2048;     // largest window resolved by sorting (fp32 rows)
constexpr int kHistBins = 1 << kKeySpanBits;  // one bin per bf16 key below the row maximum
constexpr int kTieCap = 1024;      // largest group of equal logits cut by index ranking
constexpr int kWalkThreads = 128;         // threads of one greedy tree-walk block
constexpr int kClusterWalkThreads = 256;  // threads of one CTA of a sampling tree-walk cluster
constexpr int kMaxWalkCluster = 8;        // CTAs that share one tree in the sampling walk
// Width of the single-pass candidate window below the running row maximum, in
// nats of the tempered distribution (tokens further below carry < e^-9 of the top
// token's weight each).  When the window misses the top-k / top-p cut, or holds
// more tokens than fit, the row falls back to the exact full-row selection.
constexpr float kWindowNats = 9.0f;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t stats_p, stats_q, counters, total;
};

// Workspace sections for B trees of N nodes: row statistics of every p row and of
// every q row, and the work counters.
inline WsLayout ws_layout(int32_t B, int32_t N) {
  WsLayout L{};
  size_t bn = (size_t)B * (size_t)N;
  size_t off = 0;
  L.stats_p = off;     off = align_up(off + bn * sizeof(spec_row_stats), 256);
  L.stats_q = off;     off = align_up(off + bn * sizeof(spec_row_stats), 256);
  L.counters = off;    off = align_up(off + sizeof(spec_verify_counters), 256);
  L.total = off;
  return L;
}

// One dense row pass launch.  Mode kRowsList: row r at base_p + r * row_pitch
// (spec_filter_rows).  Mode kRowsTree: virtual rows [0, B*N) are the p rows
// (b, n), and when q is needed [B*N, 2*B*N) the q rows, skipped for leaves.
enum RowMode { kRowsList = 0, kRowsTree = 1 };

struct RowJob {
  const void* base_p;
  const void* base_q;
  int64_t row_pitch;
  int64_t batch_stride;
  int32_t V, N, B, R;
  int32_t mode;
  int32_t with_q;
  int32_t first_row;       // first virtual row of the launch (kRowsTree: B*N = q rows only)
  const int32_t* parents;  // [B, N]: a q row is needed only for nodes with a child
  spec_row_stats* stats_p;
  spec_row_stats* stats_q;
  float temperature;
  float c;        // log2(e) / T
  float delta_z;  // candidate window in logit units (kWindowNats * T)
  int32_t top_k;  // 0: off
  float top_p;    // >= 1: off
  uint32_t flags;
  const float* req_temperature;  // [B] per-tree temperatures (kRowsTree), or null
  uint64_t wait_limit_ns;        // bound of every device-side wait
  unsigned long long* counters;  // spec_verify_counters as an array of 8 u64, or null
};

// The sampling parameters one tree is verified under (the launch's, or the tree's own
// when per-request arrays are given): c = log2(e) / T, delta_z = the candidate window
// below the row maximum in logit units, trunc = a top-k / top-p cut is needed.
struct Samp {
  float temperature, c, delta_z, top_p;
  int32_t top_k, trunc;
};

struct TreeJob {
  const void* base_p;
  const void* base_q;
  int64_t row_pitch;
  int64_t batch_stride;
  int32_t V, N, B, W;
  const int32_t* tokens;
  const int32_t* parents;
  const spec_row_stats* stats_p;
  const spec_row_stats* stats_q;
  float temperature;
  float c;
  // top-k / top-p cut, computed by the walk for the rows it visits (the row pass
  // then supplies only max, sum and argmax): trunc = a cut is needed
  int32_t trunc;
  int32_t top_k;      // 0 = off
  float top_p;        // 1 = off
  float delta_z;      // candidate window below the row maximum (logit units)
  int32_t exact;      // always take the full-row exact selection
  int32_t visited_only;  // no dense pass: the walk computes the statistics of the rows it visits
  // per-request sampling parameters, [B] each (null: the launch's values above);
  // trunc is then 1 (a tree may cut) and each tree reads its own
  const float* req_temperature;
  const int32_t* req_top_k;
  const float* req_top_p;
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
// Checked builds (-DSPEC_CHECK): each file's device error word, read and cleared.
uint32_t check_word_rows();
uint32_t check_word_walk();
// Small vocabularies without a cut: one warp per tree computes its visited rows'
// statistics itself (no dense pass precedes it).
bool small_walk_applies(const TreeJob& job, bool greedy, uint32_t flags);
cudaError_t launch_tree_walk(const TreeJob& job, spec_dtype dtype, bool greedy, bool small,
                             cudaStream_t s);
cudaError_t launch_philox_words(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                                const int32_t* node_idx, int32_t n, uint32_t* out,
                                cudaStream_t s);
int device_sm_count();

// Fused LM head (lmhead.cu): bytes of the per-(row, column tile) statistics, and the
// launch of the GEMM + statistics kernel and of the combine kernel that writes the
// row statistics of the M target rows.
size_t lmhead_part_bytes(int M, int V);
// The LM-head GEMM alone: bf16 logits F W^T into p (rows of pitch elements), no row
// statistics (the draft-side top-k ranks the rows itself).
cudaError_t launch_lmhead_logits(const void* features, const void* weight, int M, int V, int K,
                                 void* p, int64_t pitch, void* part, int* err, cudaStream_t s);
cudaError_t launch_lmhead(const void* features, const void* weight, int M, int V, int K,
                          float temperature, void* p, int64_t pitch, void* part, int* err,
                          spec_row_stats* stats, unsigned long long* counters, cudaStream_t s);

}  // namespace svk
