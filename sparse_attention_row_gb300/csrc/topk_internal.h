// Internal declarations shared by the kernel and the C-ABI translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "libtopk.h"

namespace ltk {

// Shared by both CTA shapes of the kernel (see topk_kernel.cu for the shapes).
constexpr int kBins = 4096;            // 12-bit radix digits
constexpr int kListCap = 2048;         // entries of the threshold bin listed by the row finish
constexpr int kWideMaxTopK = 4096;     // largest TopK of the wide shape (buffer: TopK + a chunk)
constexpr int kPairMaxTopK = 2048;     // largest TopK of the paired shape
constexpr int kSmallMaxTopK = 2048;    // largest TopK of the small shape
constexpr int kMaxGroup = 16;          // CTAs that may split one row
constexpr int kMaxCluster = 8;         // CTAs of a group that may form one thread-block cluster
constexpr int kLenCache = 64;          // row lengths cached in shared memory
constexpr int kSmallSet = 64;          // candidate sets up to this size are ranked by one warp
constexpr uint64_t kDefaultTimeoutNs = 1000ull * 1000ull * 1000ull;  // 1 s

// CTA shapes. kShapeWide: one CTA of 24 consumer warps per SM (any row split).
// kShapePair: two CTAs of 12 consumer warps per SM, whole rows only; with many
// rows per SM one CTA's row finish overlaps the other's streaming.
// kShapeSmall: 8 consumer warps in about 83 KB of shared memory, whole rows
// only, for devices or partitions with less shared memory per block.
// kShapeShort: the short-row kernel (topk_short.cu), one CTA of 32 warps per
// SM; a row of at most 32768 elements (16 pieces) stays resident in its 128 KB
// ring, a longer one streams through it. kShapeShort16: the same kernel with 16
// warps per CTA (topk_short16.cu).
constexpr int kShapeWide = 1;
constexpr int kShapePair = 2;
constexpr int kShapeSmall = 3;
constexpr int kShapeShort = 4;
constexpr int kShapeShort16 = 5;
constexpr int kWideCtaThreads = 800;   // 24 consumer warps + the copy warp
constexpr int kPairCtaThreads = 416;   // 12 consumer warps + the copy warp
constexpr int kSmallCtaThreads = 288;  // 8 consumer warps + the copy warp
constexpr int kShortCtaThreads = 1024;
constexpr int kShort16CtaThreads = 512;

// Per row group exchange area. Everything but the status word returns to zero
// at the end of every launch that completes.
struct __align__(256) GroupWs {
  uint32_t bar_count;              // barrier arrivals, counted up during a launch
  uint32_t exit_count;             // CTAs of the group that have finished
  uint32_t pad_[62];
  uint32_t h1[kBins];              // merged histogram, bits 31..20 of the keys
  uint32_t h2[kBins];              // merged histogram, bits 19..8
  uint32_t h3[kMaxGroup][256];     // per-CTA histograms, bits 7..0
  uint32_t cnt[kMaxGroup][4];      // per-CTA counts selected in the first two passes
};

constexpr size_t kWsHeaderBytes = 256;  // status word + reserved

inline size_t workspace_bytes_for(int num_sms) {
  return kWsHeaderBytes + sizeof(GroupWs) * (size_t)(num_sms > 0 ? num_sms : 1);
}

struct Params {
  const float* logits;
  int64_t stride;      // elements between row starts
  int64_t col_stride;  // elements between consecutive columns (1: contiguous rows, bulk copies)
  int64_t max_len;     // columns of every row; lengths are clamped into [0, max_len]
  const int32_t* lengths;
  int64_t num_rows;
  int32_t* out;
  int topk;
  int G;             // CTAs per row group
  int num_groups;
  uint32_t* status;  // sticky device status word
  GroupWs* groups;
  uint64_t timeout_ns;
  int inject;
  int cluster;       // 1: the G CTAs of a group are one cluster and merge through its shared memory
  int dependent_launch;  // host side: 1 = launch with programmatic stream serialisation (short-row kernel)
};

// Programmatic dependent launch unless LIBTOPK_DEPENDENT_LAUNCH=2 (read once).
bool dependent_launch_default();

// Host side of one compiled kernel shape (ltk::wide, ltk::pair, ltk::small, ltk::shortrow, ltk::short16).
#define LTK_DECLARE_SHAPE(NS)                                                                  \
  namespace NS {                                                                               \
  int kernel_threads();                                                                        \
  size_t kernel_smem_bytes();                                                                  \
  cudaError_t kernel_configure();                  /* shared-memory opt-in (current device) */ \
  cudaError_t kernel_occupancy(int* ctas_per_sm);  /* occupancy of the exact kernel */         \
  cudaError_t kernel_max_clusters(int cluster_size, int* clusters);                            \
  cudaError_t launch_topk(const Params& p, int grid, bool cooperative, cudaStream_t stream);   \
  }
LTK_DECLARE_SHAPE(wide)
LTK_DECLARE_SHAPE(pair)
LTK_DECLARE_SHAPE(small)
LTK_DECLARE_SHAPE(shortrow)
LTK_DECLARE_SHAPE(short16)
#undef LTK_DECLARE_SHAPE

// One selection as the entry points receive it (device pointers, caller-owned).
struct Call {
  const float* logits;
  int64_t row_stride;
  int64_t col_stride;
  int64_t max_len;
  const int32_t* lengths;
  int64_t num_rows;
  int next_n;
  int topk;
  int32_t* out;
};


// Checks the arguments, plans and enqueues one selection on `stream`, with
// `scratch` laid out as a workspace (status word, then row-group areas) that
// holds `max_groups` row groups; a plan needing more returns
// TOPK_ERR_WORKSPACE_TOO_SMALL. `options` may be null; the LIBTOPK_*
// environment knobs fill the fields it leaves at zero. Used by every entry
// point that selects (topk_api.cu, topk_static.cu).
int run_selection(const Call& c, void* scratch, int max_groups, cudaStream_t stream, const topk_options* options);

inline cudaError_t launch_shape(int shape, const Params& p, int grid, bool cooperative, cudaStream_t stream) {
  if (shape == kShapePair) return pair::launch_topk(p, grid, cooperative, stream);
  if (shape == kShapeSmall) return small::launch_topk(p, grid, cooperative, stream);
  if (shape == kShapeShort) return shortrow::launch_topk(p, grid, cooperative, stream);
  if (shape == kShapeShort16) return short16::launch_topk(p, grid, cooperative, stream);
  return wide::launch_topk(p, grid, cooperative, stream);
}

}  // namespace ltk
