// noalloc.cu -- spec_verify_tree_noalloc: the verify call without a caller
// workspace.  The scratch it needs (the row statistics of every p and q row and
// the work counters) lives in one file-scope __device__ array of this library,
// sized for at most SPEC_STATIC_WORKSPACE_BYTES; nothing is allocated per call.
//
// Some callers cannot hand over a workspace: cudaMalloc and cudaFree may
// synchronise the whole device and stall other streams, which a decode loop
// under a latency budget cannot afford, and a host program whose memory pool owns
// all device memory may forbid any allocation it did not make.  Those callers use
// this entry point instead of spec_verify_tree.
#include <atomic>
#include <mutex>

#include "internal.h"

namespace svk {
namespace {

// Scratch of the no-allocation entry point: one copy per device, part of this
// library's module image, so it is reserved when the module loads.
static __device__ __align__(256) unsigned char g_static_workspace[SPEC_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_static_ptr[kMaxDevices];
std::mutex g_static_mutex;

// Device address of g_static_workspace on the current device, resolved once per
// device (with that device current) and cached; nullptr on a CUDA error.
void* static_workspace_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* ptr = g_static_ptr[dev].load(std::memory_order_acquire);
  if (ptr) return ptr;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  ptr = g_static_ptr[dev].load(std::memory_order_relaxed);
  if (ptr) return ptr;
  if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) return nullptr;
  g_static_ptr[dev].store(ptr, std::memory_order_release);
  return ptr;
}

}  // namespace
}  // namespace svk

using namespace svk;

extern "C" int spec_verify_tree_noalloc(const void* logits_p, const void* logits_q,
                                        spec_dtype dtype, int32_t B, int32_t N, int32_t V,
                                        int64_t row_pitch, int64_t batch_stride,
                                        const int32_t* draft_tokens, const int32_t* parent_idx,
                                        int32_t max_depth, spec_sampling_params params,
                                        uint64_t rng_seed, uint64_t rng_offset,
                                        int32_t* out_accept_len, int32_t* out_tokens,
                                        int32_t* out_accepted_path, float* out_alpha,
                                        int32_t* out_status, spec_verify_counters* out_counters,
                                        spec_stream_t stream) {
  // the size limit is checked before anything touches the device
  if (B > 0 && N >= 1 && N <= SPEC_MAX_NODES &&
      ws_layout(B, N).total > (size_t)SPEC_STATIC_WORKSPACE_BYTES)
    return SPEC_ERR_TOO_LARGE;
  void* ws = static_workspace_on_current_device();
  if (!ws) return SPEC_ERR_CUDA;
  // Nothing in the scratch has to start at zero: the row pass writes every
  // statistics record the walk reads, and the work counters are reset on the
  // stream (cudaMemsetAsync, no allocation) when out_counters is requested.
  return spec_verify_tree_phases(SPEC_PHASE_ALL, logits_p, logits_q, dtype, B, N, V, row_pitch,
                                 batch_stride, draft_tokens, parent_idx, max_depth, params,
                                 rng_seed, rng_offset, out_accept_len, out_tokens,
                                 out_accepted_path, out_alpha, out_status, out_counters, ws,
                                 (size_t)SPEC_STATIC_WORKSPACE_BYTES, stream);
}
