// Internal declarations shared by the kernel and the C-ABI translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ltk {

// CTA shape and shared-memory staging.
constexpr int kThreads = 768;          // consumer threads per CTA (24 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kCtaThreads = kThreads + 32;  // plus one copy-issuing warp
constexpr int kChunk = 6144;           // fp32 elements per staging slot (24 KB)
constexpr int kStages = 4;             // staging slots in flight per CTA (96 KB)
constexpr int kBins = 4096;            // 12-bit radix digits
constexpr int kBufCap = 12288;         // candidate (key, index) pairs kept per CTA
constexpr int kMaxTopK = 2048;
constexpr int kMaxGroup = 16;          // CTAs that may split one row
constexpr int kMaxCluster = 8;         // CTAs of a group that may form one thread-block cluster
constexpr int kLenCache = 64;          // row lengths cached in shared memory
constexpr int kSmallSet = 64;          // candidate sets up to this size are ranked by one warp
constexpr int kMinSpan = 8192;         // fewest elements per CTA when a row is split
constexpr int64_t kDefaultLongRowThreshold = 32768;
constexpr int64_t kSplitGain = 90000;         // elements a workspace-merged split must save per CTA (measured)
constexpr int64_t kSplitGainCluster = 24000;  // elements a cluster-merged split must save per CTA
constexpr uint64_t kDefaultTimeoutNs = 1000ull * 1000ull * 1000ull;  // 1 s

static_assert(kMaxTopK + kChunk <= kBufCap, "a chunk must fit next to topk kept candidates");
static_assert(kChunk % (4 * kThreads) == 0, "a chunk is a whole number of float4 per thread");

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
  int64_t stride;
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
};

size_t kernel_smem_bytes();
cudaError_t kernel_configure();                 // sets the shared-memory opt-in (current device)
cudaError_t kernel_occupancy(int* ctas_per_sm);  // occupancy of the exact kernel
cudaError_t kernel_max_clusters(int cluster_size, int* clusters);  // co-resident clusters of that size
cudaError_t launch_topk(const Params& p, int grid, bool cooperative, cudaStream_t stream);

}  // namespace ltk
