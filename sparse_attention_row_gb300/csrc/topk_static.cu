// topk_ragged_static: the same selection as topk_ragged, for callers that
// cannot allocate device memory.
//
// Some callers have no allocator to hand: plugins and runtimes that may only
// enqueue work on streams they are given, code running where cudaMalloc is
// forbidden or would synchronise the device (for example inside a captured or
// latency-critical region), or hosts that budget every allocation themselves.
// They still pass the input and output buffers, but cannot provide the
// workspace that topk_ragged needs. This entry point uses a scratch area that
// lives in a fixed device array instead, loaded with the library.
//
// The scratch holds the status word and kStaticGroups row-group areas: every
// plan that splits rows across CTAs on a GPU with up to 2 * kStaticGroups SMs
// fits. A plan needing more row groups is rejected with
// TOPK_ERR_WORKSPACE_TOO_SMALL.
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <mutex>

#include "libtopk.h"
#include "topk_internal.h"

namespace {

constexpr int kStaticGroups = 76;
constexpr size_t kStaticBytes = ltk::kWsHeaderBytes + sizeof(ltk::GroupWs) * kStaticGroups;
constexpr int kMaxDevices = 64;

// One copy per GPU that loads the library; it stays allocated until the
// process exits. Every call on a device uses this same area.
static __device__ __align__(256) unsigned char g_topk_scratch[kStaticBytes];

struct StaticDevice {
  bool ready = false;
  void* scratch = nullptr;  // device address of g_topk_scratch on that device
};

std::mutex g_static_mu;
StaticDevice g_static_dev[kMaxDevices];

}  // namespace

extern "C" int topk_ragged_static(const float* logits, int64_t row_stride, const int32_t* lengths,
                                  int64_t num_rows, int next_n, int topk, int32_t* out_idx,
                                  void* stream) {
  // the host-side checks come first, as in topk_ragged: nothing is set up or
  // enqueued for a call that returns an error
  if (num_rows < 0 || row_stride < 1 || next_n < 1 || (num_rows % next_n) != 0)
    return TOPK_ERR_INVALID_ARG;
  if (topk < 1 || topk > ltk::kWideMaxTopK) return TOPK_ERR_UNSUPPORTED_TOPK;
  if (num_rows == 0) return TOPK_OK;
  if (logits == nullptr || lengths == nullptr || out_idx == nullptr) return TOPK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || (reinterpret_cast<uintptr_t>(lengths) & 3u) ||
      (reinterpret_cast<uintptr_t>(out_idx) & 3u))
    return TOPK_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    // First call on this device (the device is current here): look up the
    // array's device address and zero it once, in stream order. Later calls
    // reuse it; every completed launch leaves it zeroed again.
    std::lock_guard<std::mutex> lk(g_static_mu);
    StaticDevice& d = g_static_dev[dev];
    if (!d.ready) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_topk_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
      }
      if (cudaMemsetAsync(ptr, 0, kStaticBytes, s) != cudaSuccess) {
        cudaGetLastError();
        return TOPK_ERR_CUDA;
      }
      d.scratch = ptr;
      d.ready = true;
    }
    scratch = d.scratch;
  }
  // the same checks, planning (LIBTOPK_* knobs included) and launch as
  // topk_ragged, on the fixed array; a plan needing more row groups than the
  // array holds is refused
  const int64_t max_len = row_stride < INT32_MAX ? row_stride : INT32_MAX;  // lengths are int32
  const ltk::Call c{logits, row_stride, 1, max_len, lengths, num_rows, next_n, topk, out_idx};
  return ltk::run_selection(c, scratch, kStaticGroups, s, nullptr);
}
