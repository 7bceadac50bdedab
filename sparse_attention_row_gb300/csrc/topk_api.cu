// C ABI of libtopk: argument checks, per-device property cache, planning and
// the single launch per call. Every entry point returns a topk_status code and
// never throws.
#include <cuda_runtime.h>
#include <stdint.h>
#include <climits>
#include <stdlib.h>

#include <mutex>

#include "libtopk.h"
#include "topk_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceEntry {
  bool ready = false;
  topk_device_props props{};
};

std::mutex g_mu;
DeviceEntry g_dev[kMaxDevices];

// Environment overrides, read once.
struct EnvKnobs {
  int64_t long_row_threshold = 0;
  int force_ctas_per_group = 0;
  uint32_t timeout_us = 0;
  int merge = 0;
  int dependent_launch = 0;
};

EnvKnobs read_env() {
  EnvKnobs e;
  if (const char* v = getenv("LIBTOPK_LONG_ROW_THRESHOLD")) e.long_row_threshold = atoll(v);
  if (const char* v = getenv("LIBTOPK_FORCE_CTAS_PER_GROUP")) e.force_ctas_per_group = atoi(v);
  if (const char* v = getenv("LIBTOPK_BARRIER_TIMEOUT_US")) e.timeout_us = static_cast<uint32_t>(atoll(v));
  if (const char* v = getenv("LIBTOPK_MERGE")) e.merge = atoi(v);
  if (const char* v = getenv("LIBTOPK_DEPENDENT_LAUNCH")) e.dependent_launch = atoi(v);
  return e;
}

const EnvKnobs& env_knobs() {
  static const EnvKnobs e = read_env();
  return e;
}

int query_device_locked(int device, topk_device_props* out) {
  if (device < 0 || device >= kMaxDevices) return TOPK_ERR_INVALID_ARG;
  DeviceEntry& d = g_dev[device];
  if (!d.ready) {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return TOPK_ERR_CUDA;
    topk_device_props p{};
    int rc = TOPK_OK;
    if (cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&p.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess) {
      rc = TOPK_ERR_CUDA;
    }
    p.smem_per_cta = static_cast<int>(ltk::wide::kernel_smem_bytes());
    p.pair_smem_per_cta = static_cast<int>(ltk::pair::kernel_smem_bytes());
    if (rc == TOPK_OK && p.smem_per_cta <= p.max_smem_optin) {
      if (ltk::wide::kernel_configure() != cudaSuccess ||
          ltk::wide::kernel_occupancy(&p.ctas_per_sm) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
      for (int c = 2; rc == TOPK_OK && c <= ltk::kMaxCluster; ++c) {
        if (ltk::wide::kernel_max_clusters(c, &p.cluster_groups[c]) != cudaSuccess) {
          cudaGetLastError();  // a device without clusters: no cluster merge is planned
          p.cluster_groups[c] = 0;
        }
      }
    } else if (rc == TOPK_OK) {
      p.ctas_per_sm = 0;  // the kernel cannot be resident; planning reports TOPK_ERR_PLAN
    }
    if (rc == TOPK_OK && p.pair_smem_per_cta <= p.max_smem_optin) {
      if (ltk::pair::kernel_configure() != cudaSuccess ||
          ltk::pair::kernel_occupancy(&p.pair_ctas_per_sm) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
    }
    p.small_smem_per_cta = static_cast<int>(ltk::small::kernel_smem_bytes());
    if (rc == TOPK_OK && p.small_smem_per_cta <= p.max_smem_optin) {
      if (ltk::small::kernel_configure() != cudaSuccess ||
          ltk::small::kernel_occupancy(&p.small_ctas_per_sm) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
    }
    p.short_smem_per_cta = static_cast<int>(ltk::shortrow::kernel_smem_bytes());
    if (rc == TOPK_OK && p.short_smem_per_cta <= p.max_smem_optin) {
      if (ltk::shortrow::kernel_configure() != cudaSuccess ||
          ltk::shortrow::kernel_occupancy(&p.short_ctas_per_sm) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
      for (int c = 2; rc == TOPK_OK && c <= ltk::kMaxCluster; ++c) {
        if (ltk::shortrow::kernel_max_clusters(c, &p.short_cluster_groups[c]) != cudaSuccess) {
          cudaGetLastError();  // no clusters of this size: the row split is not planned
          p.short_cluster_groups[c] = 0;
        }
      }
    }
    p.short16_smem_per_cta = static_cast<int>(ltk::short16::kernel_smem_bytes());
    if (rc == TOPK_OK && p.short16_smem_per_cta <= p.max_smem_optin) {
      if (ltk::short16::kernel_configure() != cudaSuccess ||
          ltk::short16::kernel_occupancy(&p.short16_ctas_per_sm) != cudaSuccess)
        rc = TOPK_ERR_CUDA;
      for (int c = 2; rc == TOPK_OK && c <= ltk::kMaxCluster; ++c) {
        if (ltk::short16::kernel_max_clusters(c, &p.short16_cluster_groups[c]) != cudaSuccess) {
          cudaGetLastError();
          p.short16_cluster_groups[c] = 0;
        }
      }
    }
    if (prev != device) cudaSetDevice(prev);
    if (rc != TOPK_OK) {
      cudaGetLastError();
      return rc;
    }
    d.props = p;
    d.ready = true;
  }
  *out = d.props;
  return TOPK_OK;
}

int current_props(topk_device_props* out, int* device) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  if (device) *device = dev;
  std::lock_guard<std::mutex> lk(g_mu);
  return query_device_locked(dev, out);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

namespace ltk {

bool dependent_launch_default() { return env_knobs().dependent_launch != 2; }

int run_selection(const Call& c, void* scratch, int max_groups, cudaStream_t stream, const topk_options* options) {
  if (c.num_rows < 0 || c.row_stride < 0 || c.col_stride < 1 || c.max_len < 1 || c.max_len > INT32_MAX ||
      c.next_n < 1 || (c.num_rows % c.next_n) != 0)
    return TOPK_ERR_INVALID_ARG;
  if (c.topk < 1 || c.topk > kWideMaxTopK) return TOPK_ERR_UNSUPPORTED_TOPK;
  if (c.num_rows == 0) return TOPK_OK;
  if (c.logits == nullptr || c.lengths == nullptr || c.out == nullptr || scratch == nullptr)
    return TOPK_ERR_INVALID_ARG;
  if (!aligned(c.logits, 4) || !aligned(c.lengths, 4) || !aligned(c.out, 4) || !aligned(scratch, 16))
    return TOPK_ERR_MISALIGNED;

  topk_device_props props{};
  int rc = current_props(&props, nullptr);
  if (rc != TOPK_OK) return rc;
  if (options != nullptr && options->workspace_bytes != 0 &&
      options->workspace_bytes < workspace_bytes_for(props.num_sms))
    return TOPK_ERR_WORKSPACE_TOO_SMALL;

  const EnvKnobs& env = env_knobs();
  topk_options opt{};
  if (options != nullptr) opt = *options;
  if (opt.long_row_threshold == 0) opt.long_row_threshold = env.long_row_threshold;
  if (opt.force_ctas_per_group == 0) opt.force_ctas_per_group = env.force_ctas_per_group;
  if (opt.barrier_timeout_us == 0) opt.barrier_timeout_us = env.timeout_us;
  if (opt.merge == 0) opt.merge = env.merge;
  if (opt.dependent_launch == 0) opt.dependent_launch = env.dependent_launch;
  if (opt.dependent_launch < 0 || opt.dependent_launch > 2) return TOPK_ERR_INVALID_ARG;

  topk_plan plan{};
  rc = topk_make_plan(&props, c.num_rows, c.max_len, c.next_n, c.topk, &opt, &plan);
  if (rc != TOPK_OK) return rc;
  // the short-row kernel splits only contiguous rows over a cluster; strided
  // ones stay whole
  const bool short_shape = plan.shape == kShapeShort || plan.shape == kShapeShort16;
  if (short_shape && plan.ctas_per_group > 1 && c.col_stride != 1) {
    opt.force_ctas_per_group = 1;
    rc = topk_make_plan(&props, c.num_rows, c.max_len, c.next_n, c.topk, &opt, &plan);
    if (rc != TOPK_OK) return rc;
  }
  if (plan.grid < 1) return TOPK_OK;
  // a caller-provided workspace holds num_sms row groups, as many as the planner
  // ever uses (the short-row kernel's cluster split uses none)
  if (max_groups >= 0 && plan.ctas_per_group > 1 && plan.shape != kShapeShort && plan.shape != kShapeShort16 &&
      plan.num_groups > max_groups)
    return TOPK_ERR_WORKSPACE_TOO_SMALL;

  Params p{};
  p.logits = c.logits;
  p.stride = c.row_stride;
  p.col_stride = c.col_stride;
  p.max_len = c.max_len;
  p.lengths = c.lengths;
  p.num_rows = c.num_rows;
  p.out = c.out;
  p.topk = c.topk;
  p.G = plan.ctas_per_group;
  p.num_groups = plan.num_groups;
  p.status = static_cast<uint32_t*>(scratch);
  p.groups = reinterpret_cast<GroupWs*>(static_cast<char*>(scratch) + kWsHeaderBytes);
  p.timeout_ns = opt.barrier_timeout_us ? static_cast<uint64_t>(opt.barrier_timeout_us) * 1000ull : kDefaultTimeoutNs;
  p.inject = opt.inject_skip_arrival;
  p.cluster = plan.cluster;
  p.dependent_launch = opt.dependent_launch != 2 ? 1 : 0;
  if (launch_shape(plan.shape, p, plan.grid, plan.cooperative != 0, stream) != cudaSuccess) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  return TOPK_OK;
}

}  // namespace ltk

extern "C" {

const char* topk_status_string(int code) {
  switch (code) {
    case TOPK_OK: return "ok";
    case TOPK_ERR_INVALID_ARG: return "invalid argument";
    case TOPK_ERR_UNSUPPORTED_TOPK: return "topk must be between 1 and 4096 (2048 for the paired shape)";
    case TOPK_ERR_MISALIGNED: return "misaligned pointer";
    case TOPK_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case TOPK_ERR_CUDA: return "CUDA runtime error";
    case TOPK_ERR_BARRIER_TIMEOUT: return "a device-side wait timed out";
    case TOPK_ERR_LENGTH_CLAMPED: return "a row length was outside [0, row_stride]";
    case TOPK_ERR_PLAN: return "no launch configuration fits the device";
    default: return "unknown status";
  }
}

int topk_query_device(int device, topk_device_props* props) {
  if (props == nullptr) return TOPK_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  return query_device_locked(device, props);
}

size_t topk_workspace_size(int device, int64_t num_rows, int64_t row_stride, int next_n, int topk) {
  (void)num_rows;
  (void)row_stride;
  (void)next_n;
  (void)topk;
  topk_device_props p{};
  if (topk_query_device(device, &p) != TOPK_OK) return 0;
  return ltk::workspace_bytes_for(p.num_sms);
}

int topk_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (workspace == nullptr || bytes < ltk::kWsHeaderBytes) return TOPK_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return TOPK_ERR_MISALIGNED;
  if (cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  return TOPK_OK;
}

int topk_get_status(const void* workspace, void* stream, uint32_t* device_status) {
  if (workspace == nullptr || device_status == nullptr) return TOPK_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return TOPK_ERR_CUDA;
  }
  *device_status = word;
  return TOPK_OK;
}

int topk_ragged_strided(const float* logits, int64_t row_stride, int64_t col_stride, int64_t max_len,
                        const int32_t* lengths, int64_t num_rows, int next_n, int topk, int32_t* out_idx,
                        void* workspace, void* stream, const topk_options* options) {
  const ltk::Call c{logits, row_stride, col_stride, max_len, lengths, num_rows, next_n, topk, out_idx};
  return ltk::run_selection(c, workspace, -1, static_cast<cudaStream_t>(stream), options);
}

int topk_ragged_ex(const float* logits, int64_t row_stride, const int32_t* lengths, int64_t num_rows,
                   int next_n, int topk, int32_t* out_idx, void* workspace, void* stream,
                   const topk_options* options) {
  if (row_stride < 1) return TOPK_ERR_INVALID_ARG;
  const int64_t max_len = row_stride < INT32_MAX ? row_stride : INT32_MAX;  // lengths are int32
  return topk_ragged_strided(logits, row_stride, 1, max_len, lengths, num_rows, next_n, topk, out_idx,
                             workspace, stream, options);
}

int topk_ragged(const float* logits, int64_t row_stride, const int32_t* lengths, int64_t num_rows,
                int next_n, int topk, int32_t* out_idx, void* workspace, void* stream) {
  return topk_ragged_ex(logits, row_stride, lengths, num_rows, next_n, topk, out_idx, workspace,
                        stream, nullptr);
}

}  // extern "C"
