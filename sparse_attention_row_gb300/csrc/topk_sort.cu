// Values and order for selected rows: gathers the value of every selected
// index and, on request, orders each row by (value desc, index asc) with -1
// padding last. The pages' consumer receives a set of indices; callers that
// want the values or a ranking (vLLM PR #54110 page, the int32 index output of
// the top-k launcher) get them here in one extra launch.
//
// One CTA handles one row at a time: the row's (value, index) pairs become
// 64-bit keys (inverted order-preserving value key in the high half, index in
// the low half), so one ascending sort gives value descending, then index
// ascending; padding is the largest key. A bitonic network over the next power
// of two at or above TopK (at most 4096 keys, 32 KB of shared memory) sorts
// them; each of its stages is one pass of compare-exchanges and a barrier.
#include <cuda_runtime.h>
#include <stdint.h>

#include "libtopk.h"
#include "topk_internal.h"

namespace ltk {
namespace sortk {

constexpr int kThreads = 1024;

struct SortParams {
  const float* logits;
  int64_t row_stride, col_stride, max_len;
  int64_t num_rows;
  int topk;
  int width;  // power of two >= topk
  int32_t* idx;
  float* val;
  int sort;
};

__device__ __forceinline__ uint32_t value_key(float x) {
  uint32_t u = __float_as_uint(x);
  u = (u == 0x80000000u) ? 0u : u;  // -0.0 ranks as +0.0
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads) topk_sort_kernel(const SortParams p) {
  extern __shared__ unsigned long long keys[];
  const int tid = threadIdx.x;
  const int K = p.topk;
  const int P = p.width;
  // programmatic dependent launch: wait for the kernel before this one on the
  // stream (typically the selection that wrote the indices) to complete, then
  // let the next one start early in the same way
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int64_t r = blockIdx.x; r < p.num_rows; r += gridDim.x) {
    int32_t* row_idx = p.idx + r * K;
    float* row_val = p.val ? p.val + r * K : nullptr;
    const float* row = p.logits + r * p.row_stride;
    for (int i = tid; i < P; i += kThreads) {
      unsigned long long k = ~0ull;
      if (i < K) {
        const int32_t x = row_idx[i];
        if (x >= 0 && x < p.max_len) {
          const uint32_t vk = value_key(__ldg(row + static_cast<int64_t>(x) * p.col_stride));
          k = (static_cast<unsigned long long>(~vk) << 32) | static_cast<uint32_t>(x);
        }
      }
      keys[i] = k;
    }
    __syncthreads();
    if (p.sort) {
      for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int t = tid; t < (P >> 1); t += kThreads) {
            const int lo = 2 * t - (t & (stride - 1));
            const int hi = lo + stride;
            const bool ascending = (lo & size) == 0;
            const unsigned long long a = keys[lo];
            const unsigned long long b = keys[hi];
            if ((a > b) == ascending) {
              keys[lo] = b;
              keys[hi] = a;
            }
          }
          __syncthreads();
        }
      }
    }
    for (int i = tid; i < K; i += kThreads) {
      const unsigned long long k = keys[i];
      const int32_t x = (k == ~0ull) ? -1 : static_cast<int32_t>(k & 0xFFFFFFFFull);
      if (p.sort) row_idx[i] = x;
      if (row_val) row_val[i] = (x >= 0) ? __ldg(row + static_cast<int64_t>(x) * p.col_stride)
                                         : -__int_as_float(0x7F800000);
    }
    __syncthreads();  // the next row reuses the keys
  }
}

}  // namespace sortk
}  // namespace ltk

extern "C" int topk_gather_sort(const float* logits, int64_t row_stride, int64_t col_stride, int64_t max_len,
                                int64_t num_rows, int topk, int32_t* out_idx, float* out_val, int sort,
                                void* stream) {
  if (num_rows < 0 || row_stride < 0 || col_stride < 1 || max_len < 1) return TOPK_ERR_INVALID_ARG;
  if (topk < 1 || topk > ltk::kWideMaxTopK) return TOPK_ERR_UNSUPPORTED_TOPK;
  if (num_rows == 0 || (!sort && out_val == nullptr)) return TOPK_OK;
  if (logits == nullptr || out_idx == nullptr) return TOPK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) || (reinterpret_cast<uintptr_t>(out_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(out_val) & 3u))
    return TOPK_ERR_MISALIGNED;
  int width = 1;
  while (width < topk) width <<= 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  ltk::sortk::SortParams p{};
  p.logits = logits;
  p.row_stride = row_stride;
  p.col_stride = col_stride;
  p.max_len = max_len;
  p.num_rows = num_rows;
  p.topk = topk;
  p.width = width;
  p.idx = out_idx;
  p.val = out_val;
  p.sort = sort ? 1 : 0;
  const int64_t grid = num_rows < 2ll * sms ? num_rows : 2ll * sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(ltk::sortk::kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(width) * sizeof(unsigned long long);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = ltk::dependent_launch_default() ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, ltk::sortk::topk_sort_kernel, p) != cudaSuccess) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  return TOPK_OK;
}
