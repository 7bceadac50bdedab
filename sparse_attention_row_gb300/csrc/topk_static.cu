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
  topk_device_props props{};
  int rc = topk_query_device(dev, &props);
  if (rc != TOPK_OK) return rc;

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

  topk_plan plan{};
  rc = topk_make_plan(&props, num_rows, row_stride, next_n, topk, nullptr, &plan);
  if (rc != TOPK_OK) return rc;
  if (plan.grid < 1) return TOPK_OK;
  if (plan.ctas_per_group > 1 && plan.num_groups > kStaticGroups) return TOPK_ERR_WORKSPACE_TOO_SMALL;

  ltk::Params p{};
  p.logits = logits;
  p.stride = row_stride;
  p.col_stride = 1;
  p.max_len = row_stride;
  p.lengths = lengths;
  p.num_rows = num_rows;
  p.out = out_idx;
  p.topk = topk;
  p.G = plan.ctas_per_group;
  p.num_groups = plan.num_groups;
  p.status = static_cast<uint32_t*>(scratch);
  p.groups = reinterpret_cast<ltk::GroupWs*>(static_cast<char*>(scratch) + ltk::kWsHeaderBytes);
  p.timeout_ns = ltk::kDefaultTimeoutNs;
  p.inject = 0;
  p.cluster = plan.cluster;
  if (ltk::launch_shape(plan.shape, p, plan.grid, plan.cooperative != 0, s) != cudaSuccess) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  return TOPK_OK;
}
