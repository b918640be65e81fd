// api.cu -- the extern "C" entry points: host-side argument checks, workspace
// carving and the launches of one verify call on the caller's stream: (prepare)
// zero the work counters when they are requested, (rows) the dense row pass,
// (walk) the per-tree accept walk.
#include <climits>
#include <cmath>

#include "internal.h"

namespace svk {

int device_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

namespace {

int elem_bytes(spec_dtype dt) { return dt == SPEC_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_params(const spec_sampling_params& prm) {
  if (!std::isfinite(prm.temperature) || prm.temperature < 0.0f) return SPEC_ERR_INVALID_ARG;
  if (!(prm.top_p > 0.0f)) return SPEC_ERR_INVALID_ARG;  // also rejects NaN
  if (prm.flags & ~(SPEC_FLAG_EXACT_SELECT | SPEC_FLAG_TEST_STALL | SPEC_FLAG_VISITED_ONLY))
    return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

int check_layout(const void* base, spec_dtype dt, int64_t row_pitch, int64_t batch_stride,
                 int32_t V) {
  if (row_pitch < V || batch_stride < 0) return SPEC_ERR_INVALID_ARG;
  const int64_t s = elem_bytes(dt);
  if (!aligned16(base) || (row_pitch * s) % 16 != 0 || (batch_stride * s) % 16 != 0)
    return SPEC_ERR_MISALIGNED;
  return SPEC_OK;
}

RowJob make_row_job(spec_dtype, int32_t V, const spec_sampling_params& prm) {
  RowJob j{};
  j.V = V;
  j.temperature = prm.temperature;
  j.c = prm.temperature > 0.0f ? (float)(1.4426950408889634 / (double)prm.temperature) : 0.0f;
  j.delta_z = kWindowNats * prm.temperature;
  j.top_k = (prm.top_k > 0 && prm.top_k < V) ? prm.top_k : 0;
  j.top_p = prm.top_p >= 1.0f ? 1.0f : prm.top_p;
  j.flags = prm.flags;
  // a healthy wait lasts microseconds; the stall self-test uses a short limit
  j.wait_limit_ns = (prm.flags & SPEC_FLAG_TEST_STALL) ? 20000000ull : 2000000000ull;
  return j;
}

}  // namespace
}  // namespace svk

using namespace svk;

extern "C" size_t spec_verify_workspace_size(int32_t B, int32_t N, int32_t V, spec_dtype dtype) {
  if (B < 0 || N < 1 || V < 1 || N > SPEC_MAX_NODES || V > SPEC_MAX_VOCAB) return 0;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return 0;
  return ws_layout(B > 0 ? B : 1, N).total;
}

namespace {

// One verify call; req_* are the per-request arrays (null: the launch's params).
int verify_impl(uint32_t phases, const void* logits_p, const void* logits_q, spec_dtype dtype,
                int32_t B, int32_t N, int32_t V, int64_t row_pitch, int64_t batch_stride,
                const int32_t* draft_tokens, const int32_t* parent_idx, int32_t max_depth,
                spec_sampling_params params, const float* req_temperature,
                const int32_t* req_top_k, const float* req_top_p, uint64_t rng_seed,
                uint64_t rng_offset, int32_t* out_accept_len, int32_t* out_tokens,
                int32_t* out_accepted_path, float* out_alpha, int32_t* out_status,
                spec_verify_counters* out_counters, void* workspace, size_t workspace_bytes,
                spec_stream_t stream) {
  if (phases == 0 || (phases & ~SPEC_PHASE_ALL)) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if (B < 0 || N < 1 || V < 1 || max_depth < 0) return SPEC_ERR_INVALID_ARG;
  if (N > SPEC_MAX_NODES || V > SPEC_MAX_VOCAB || max_depth >= SPEC_MAX_NODES)
    return SPEC_ERR_TOO_LARGE;
  int rc = check_params(params);
  if (rc != SPEC_OK) return rc;
  const bool per_request = req_temperature != nullptr;
  const bool greedy = !per_request && params.temperature == 0.0f;
  if (!logits_p || (!greedy && !logits_q) || !draft_tokens || !parent_idx || !out_accept_len ||
      !out_tokens || !out_accepted_path || !workspace)
    return SPEC_ERR_INVALID_ARG;
  rc = check_layout(logits_p, dtype, row_pitch, batch_stride, V);
  if (rc != SPEC_OK) return rc;
  if (!greedy) {
    rc = check_layout(logits_q, dtype, row_pitch, batch_stride, V);
    if (rc != SPEC_OK) return rc;
  }
  const WsLayout L = ws_layout(B > 0 ? B : 1, N);
  if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPEC_ERR_WORKSPACE;
  if (B == 0) return SPEC_OK;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  spec_row_stats* stats_p = reinterpret_cast<spec_row_stats*>(ws + L.stats_p);
  spec_row_stats* stats_q = reinterpret_cast<spec_row_stats*>(ws + L.stats_q);
  unsigned long long* counters = reinterpret_cast<unsigned long long*>(ws + L.counters);

  TreeJob tj{};
  tj.base_p = logits_p;
  tj.base_q = logits_q;
  tj.row_pitch = row_pitch;
  tj.batch_stride = batch_stride;
  tj.V = V;
  tj.N = N;
  tj.B = B;
  tj.W = max_depth + 1;
  tj.tokens = draft_tokens;
  tj.parents = parent_idx;
  tj.stats_p = stats_p;
  tj.stats_q = stats_q;
  tj.temperature = params.temperature;
  tj.c = greedy ? 0.0f : (float)(1.4426950408889634 / (double)params.temperature);
  tj.top_k = (params.top_k > 0 && params.top_k < V) ? params.top_k : 0;
  tj.top_p = params.top_p >= 1.0f ? 1.0f : params.top_p;
  tj.trunc = (!greedy && (tj.top_k > 0 || tj.top_p < 1.0f)) ? 1 : 0;
  tj.delta_z = kWindowNats * params.temperature;
  tj.exact = (params.flags & SPEC_FLAG_EXACT_SELECT) ? 1 : 0;
  tj.visited_only = (params.flags & SPEC_FLAG_VISITED_ONLY) ? 1 : 0;
  if (per_request) {
    tj.req_temperature = req_temperature;
    tj.req_top_k = req_top_k;
    tj.req_top_p = req_top_p;
    tj.trunc = 1;  // any tree may cut: the walk reserves the cut's buffers
  }
  tj.seed = rng_seed;
  tj.offset = rng_offset;
  tj.out_accept_len = out_accept_len;
  tj.out_tokens = out_tokens;
  tj.out_path = out_accepted_path;
  tj.out_alpha = out_alpha;
  tj.out_status = out_status;
  // work counters are kept only when the caller asks for them
  tj.counters = out_counters ? counters : nullptr;

  if ((phases & SPEC_PHASE_PREPARE) && out_counters &&
      cudaMemsetAsync(counters, 0, sizeof(spec_verify_counters), s) != cudaSuccess)
    return SPEC_ERR_CUDA;

  RowJob rj = make_row_job(dtype, V, params);
  rj.base_p = logits_p;
  rj.base_q = logits_q;
  rj.row_pitch = row_pitch;
  rj.batch_stride = batch_stride;
  rj.N = N;
  rj.B = B;
  rj.mode = kRowsTree;
  rj.with_q = greedy ? 0 : 1;
  // the row pass supplies max, sum and argmax only; the walk cuts the rows it visits
  rj.top_k = 0;
  rj.top_p = 1.0f;
  rj.parents = parent_idx;
  rj.stats_p = stats_p;
  rj.stats_q = stats_q;
  rj.counters = tj.counters;
  rj.req_temperature = req_temperature;
  const int virtual_rows = B * N * (greedy ? 1 : 2);
  // small vocabularies without a cut: one warp per tree reads the rows it visits
  const bool small = small_walk_applies(tj, greedy, params.flags);
  // the visited-rows-only schedule and the small-vocabulary walk have no dense pass
  if ((phases & SPEC_PHASE_ROWS) && !tj.visited_only && !small &&
      launch_row_pass(rj, dtype, virtual_rows, s) != cudaSuccess)
    return SPEC_ERR_CUDA;

  if (phases & SPEC_PHASE_WALK) {
    if (launch_tree_walk(tj, dtype, greedy, small, s) != cudaSuccess) return SPEC_ERR_CUDA;
    if (out_counters &&
        cudaMemcpyAsync(out_counters, counters, sizeof(spec_verify_counters),
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_tree_phases(uint32_t phases, const void* logits_p,
                                       const void* logits_q, spec_dtype dtype, int32_t B,
                                       int32_t N, int32_t V, int64_t row_pitch,
                                       int64_t batch_stride, const int32_t* draft_tokens,
                                       const int32_t* parent_idx, int32_t max_depth,
                                       spec_sampling_params params, uint64_t rng_seed,
                                       uint64_t rng_offset, int32_t* out_accept_len,
                                       int32_t* out_tokens, int32_t* out_accepted_path,
                                       float* out_alpha, int32_t* out_status,
                                       spec_verify_counters* out_counters, void* workspace,
                                       size_t workspace_bytes, spec_stream_t stream) {
  return verify_impl(phases, logits_p, logits_q, dtype, B, N, V, row_pitch, batch_stride,
                     draft_tokens, parent_idx, max_depth, params, nullptr, nullptr, nullptr,
                     rng_seed, rng_offset, out_accept_len, out_tokens, out_accepted_path,
                     out_alpha, out_status, out_counters, workspace, workspace_bytes, stream);
}

extern "C" int spec_verify_tree_per_request(
    uint32_t phases, const void* logits_p, const void* logits_q, spec_dtype dtype, int32_t B,
    int32_t N, int32_t V, int64_t row_pitch, int64_t batch_stride, const int32_t* draft_tokens,
    const int32_t* parent_idx, int32_t max_depth, const float* temperature, const int32_t* top_k,
    const float* top_p, uint32_t flags, uint64_t rng_seed, uint64_t rng_offset,
    int32_t* out_accept_len, int32_t* out_tokens, int32_t* out_accepted_path, float* out_alpha,
    int32_t* out_status, spec_verify_counters* out_counters, void* workspace,
    size_t workspace_bytes, spec_stream_t stream) {
  if (!temperature) return SPEC_ERR_INVALID_ARG;
  // the launch-wide values only select the sampling row pass; each tree reads its own
  spec_sampling_params prm{1.0f, 0, 1.0f, flags};
  return verify_impl(phases, logits_p, logits_q, dtype, B, N, V, row_pitch, batch_stride,
                     draft_tokens, parent_idx, max_depth, prm, temperature, top_k, top_p,
                     rng_seed, rng_offset, out_accept_len, out_tokens, out_accepted_path,
                     out_alpha, out_status, out_counters, workspace, workspace_bytes, stream);
}

extern "C" int spec_verify_tree(const void* logits_p, const void* logits_q, spec_dtype dtype,
                                int32_t B, int32_t N, int32_t V, int64_t row_pitch,
                                int64_t batch_stride, const int32_t* draft_tokens,
                                const int32_t* parent_idx, int32_t max_depth,
                                spec_sampling_params params, uint64_t rng_seed,
                                uint64_t rng_offset, int32_t* out_accept_len,
                                int32_t* out_tokens, int32_t* out_accepted_path,
                                float* out_alpha, int32_t* out_status,
                                spec_verify_counters* out_counters, void* workspace,
                                size_t workspace_bytes, spec_stream_t stream) {
  return spec_verify_tree_phases(SPEC_PHASE_ALL, logits_p, logits_q, dtype, B, N, V, row_pitch,
                                 batch_stride, draft_tokens, parent_idx, max_depth, params,
                                 rng_seed, rng_offset, out_accept_len, out_tokens,
                                 out_accepted_path, out_alpha, out_status, out_counters,
                                 workspace, workspace_bytes, stream);
}

namespace {
// Workspace of the fused call: the verify workspace, then the LM head's tile
// statistics and its error flag (256-byte aligned sections).
struct FusedLayout {
  WsLayout base;
  size_t part, err, total;
};
FusedLayout fused_layout(int32_t B, int32_t N, int32_t V) {
  FusedLayout L{};
  L.base = ws_layout(B, N);
  L.part = L.base.total;
  L.err = align_up(L.part + lmhead_part_bytes(B * N, V), 256);
  L.total = align_up(L.err + sizeof(int), 256);
  return L;
}
}  // namespace

extern "C" size_t spec_fused_lmhead_workspace_size(int32_t B, int32_t N, int32_t V) {
  if (B < 1 || N < 1 || V < 1 || N > SPEC_MAX_NODES || V > SPEC_MAX_VOCAB) return 0;
  if ((int64_t)B * N > (int64_t)INT32_MAX / 2) return 0;
  return fused_layout(B, N, V).total;
}

extern "C" int spec_verify_tree_fused_lmhead_phases(
    uint32_t phases, const void* features, const void* lm_head_w, int32_t d, const void* logits_q, int32_t B,
    int32_t N, int32_t V, int64_t row_pitch, const int32_t* draft_tokens,
    const int32_t* parent_idx, int32_t max_depth, spec_sampling_params params,
    uint64_t rng_seed, uint64_t rng_offset, void* out_logits_p, int32_t* out_accept_len,
    int32_t* out_tokens, int32_t* out_accepted_path, float* out_alpha, int32_t* out_status,
    spec_verify_counters* out_counters, void* workspace, size_t workspace_bytes,
    spec_stream_t stream) {
  if (phases == 0 || (phases & ~SPEC_PHASE_ALL_FUSED)) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || N < 1 || V < 1 || max_depth < 0 || d < 1) return SPEC_ERR_INVALID_ARG;
  if (N > SPEC_MAX_NODES || V > SPEC_MAX_VOCAB || max_depth >= SPEC_MAX_NODES)
    return SPEC_ERR_TOO_LARGE;
  if ((int64_t)B * N > (int64_t)INT32_MAX / 2) return SPEC_ERR_TOO_LARGE;
  int rc = check_params(params);
  if (rc != SPEC_OK) return rc;
  const bool greedy = params.temperature == 0.0f;
  if (!features || !lm_head_w || (!greedy && !logits_q) || !draft_tokens || !parent_idx ||
      !out_logits_p || !out_accept_len || !out_tokens || !out_accepted_path || !workspace)
    return SPEC_ERR_INVALID_ARG;
  // the tensor maps need 16-byte aligned bases and rows (d a multiple of 8)
  if (!aligned16(features) || !aligned16(lm_head_w) || d % 8 != 0) return SPEC_ERR_MISALIGNED;
  const int64_t batch_stride = (int64_t)N * row_pitch;
  rc = check_layout(out_logits_p, SPEC_BF16, row_pitch, batch_stride, V);
  if (rc != SPEC_OK) return rc;
  if (!greedy) {
    rc = check_layout(logits_q, SPEC_BF16, row_pitch, batch_stride, V);
    if (rc != SPEC_OK) return rc;
  }
  if (B == 0) return SPEC_OK;
  const FusedLayout L = fused_layout(B, N, V);
  if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SPEC_ERR_WORKSPACE;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  spec_row_stats* stats_p = reinterpret_cast<spec_row_stats*>(ws + L.base.stats_p);
  spec_row_stats* stats_q = reinterpret_cast<spec_row_stats*>(ws + L.base.stats_q);
  unsigned long long* counters = reinterpret_cast<unsigned long long*>(ws + L.base.counters);
  int* err = reinterpret_cast<int*>(ws + L.err);
  unsigned long long* cnt = out_counters ? counters : nullptr;

  if (phases & SPEC_PHASE_PREPARE) {
    if (out_counters &&
        cudaMemsetAsync(counters, 0, sizeof(spec_verify_counters), s) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess) return SPEC_ERR_CUDA;
  }
  // target rows: logits and their statistics from the tensor-core GEMM
  if ((phases & SPEC_PHASE_LMHEAD) &&
      launch_lmhead(features, lm_head_w, B * N, V, d, params.temperature, out_logits_p,
                    row_pitch, ws + L.part, err, stats_p, cnt, s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  // draft rows of nodes with children: the dense row pass
  if (!greedy && (phases & SPEC_PHASE_ROWS)) {
    RowJob rj = make_row_job(SPEC_BF16, V, params);
    rj.base_p = out_logits_p;
    rj.base_q = logits_q;
    rj.row_pitch = row_pitch;
    rj.batch_stride = batch_stride;
    rj.N = N;
    rj.B = B;
    rj.mode = kRowsTree;
    rj.with_q = 1;
    rj.first_row = B * N;
    rj.top_k = 0;
    rj.top_p = 1.0f;
    rj.parents = parent_idx;
    rj.stats_p = stats_p;
    rj.stats_q = stats_q;
    rj.counters = cnt;
    if (launch_row_pass(rj, SPEC_BF16, B * N, s) != cudaSuccess) return SPEC_ERR_CUDA;
  }
  TreeJob tj{};
  tj.base_p = out_logits_p;
  tj.base_q = logits_q;
  tj.row_pitch = row_pitch;
  tj.batch_stride = batch_stride;
  tj.V = V;
  tj.N = N;
  tj.B = B;
  tj.W = max_depth + 1;
  tj.tokens = draft_tokens;
  tj.parents = parent_idx;
  tj.stats_p = stats_p;
  tj.stats_q = stats_q;
  tj.temperature = params.temperature;
  tj.c = greedy ? 0.0f : (float)(1.4426950408889634 / (double)params.temperature);
  tj.top_k = (params.top_k > 0 && params.top_k < V) ? params.top_k : 0;
  tj.top_p = params.top_p >= 1.0f ? 1.0f : params.top_p;
  tj.trunc = (!greedy && (tj.top_k > 0 || tj.top_p < 1.0f)) ? 1 : 0;
  tj.delta_z = kWindowNats * params.temperature;
  tj.exact = (params.flags & SPEC_FLAG_EXACT_SELECT) ? 1 : 0;
  tj.seed = rng_seed;
  tj.offset = rng_offset;
  tj.out_accept_len = out_accept_len;
  tj.out_tokens = out_tokens;
  tj.out_path = out_accepted_path;
  tj.out_alpha = out_alpha;
  tj.out_status = out_status;
  tj.counters = cnt;
  if (phases & SPEC_PHASE_WALK) {
    if (launch_tree_walk(tj, SPEC_BF16, greedy, false, s) != cudaSuccess) return SPEC_ERR_CUDA;
    if (out_counters && cudaMemcpyAsync(out_counters, counters, sizeof(spec_verify_counters),
                                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

extern "C" int spec_verify_tree_fused_lmhead(
    const void* features, const void* lm_head_w, int32_t d, const void* logits_q, int32_t B,
    int32_t N, int32_t V, int64_t row_pitch, const int32_t* draft_tokens,
    const int32_t* parent_idx, int32_t max_depth, spec_sampling_params params,
    uint64_t rng_seed, uint64_t rng_offset, void* out_logits_p, int32_t* out_accept_len,
    int32_t* out_tokens, int32_t* out_accepted_path, float* out_alpha, int32_t* out_status,
    spec_verify_counters* out_counters, void* workspace, size_t workspace_bytes,
    spec_stream_t stream) {
  return spec_verify_tree_fused_lmhead_phases(
      SPEC_PHASE_ALL_FUSED, features, lm_head_w, d, logits_q, B, N, V, row_pitch, draft_tokens,
      parent_idx, max_depth, params, rng_seed, rng_offset, out_logits_p, out_accept_len,
      out_tokens, out_accepted_path, out_alpha, out_status, out_counters, workspace,
      workspace_bytes, stream);
}

extern "C" int spec_filter_rows(const void* logits, spec_dtype dtype, int32_t R, int32_t V,
                                int64_t row_pitch, spec_sampling_params params,
                                spec_row_stats* out_stats, spec_stream_t stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if (R < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (V > SPEC_MAX_VOCAB) return SPEC_ERR_TOO_LARGE;
  int rc = check_params(params);
  if (rc != SPEC_OK) return rc;
  if (!logits || !out_stats) return SPEC_ERR_INVALID_ARG;
  rc = check_layout(logits, dtype, row_pitch, 0, V);
  if (rc != SPEC_OK) return rc;
  if (R == 0) return SPEC_OK;
  RowJob rj = make_row_job(dtype, V, params);
  rj.base_p = logits;
  rj.row_pitch = row_pitch;
  rj.R = R;
  rj.mode = kRowsList;
  rj.stats_p = out_stats;
  if (launch_row_pass(rj, dtype, R, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

extern "C" int spec_philox_words(uint64_t seed, uint64_t offset, const int32_t* b_idx,
                                 const int32_t* node_idx, int32_t n, uint32_t* out_words,
                                 spec_stream_t stream) {
  if (n < 0) return SPEC_ERR_INVALID_ARG;
  if (n == 0) return SPEC_OK;
  if (!b_idx || !node_idx || !out_words) return SPEC_ERR_INVALID_ARG;
  if (!aligned16(out_words)) return SPEC_ERR_MISALIGNED;
  if (launch_philox_words(seed, offset, b_idx, node_idx, n, out_words,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

extern "C" const char* spec_error_string(int code) {
  switch (code) {
    case SPEC_OK: return "success";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case SPEC_ERR_MISALIGNED: return "misaligned pointer or stride (16-byte alignment required)";
    case SPEC_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case SPEC_ERR_CUDA: return "CUDA launch failed";
    case SPEC_ERR_TOO_LARGE: return "size above the library limits";
    default: return "unknown error code";
  }
}

extern "C" int spec_check_errors(uint32_t* out_words) {
  if (!out_words) return SPEC_ERR_INVALID_ARG;
  out_words[0] = check_word_rows();
  out_words[1] = check_word_walk();
  if (out_words[0] == 0xffffffffu || out_words[1] == 0xffffffffu) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

extern "C" int spec_check_build(void) {
#ifdef SPEC_CHECK
  return 1;
#else
  return 0;
#endif
}
