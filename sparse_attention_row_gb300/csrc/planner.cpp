// Host planner: picks the launch shape from the device's measured occupancy.
//
// The persistent_topk launcher on the vLLM PR #41189 page ("Implementation
// breakdown") derives the number of row groups from num_sms x occupancy and
// must stay below it whenever CTAs wait on one another; an oversized
// cooperative grid deadlocks (same page, "Feature and motivation": TopK=1024,
// MTP=1). Here the plan is a pure function of the device properties, so the
// bound can be checked on made-up devices, and the launch that waits across
// CTAs is a cooperative launch, which the CUDA driver refuses rather than hangs if
// the grid cannot be resident.
//
// Shape rules:
//   - one CTA owns whole rows (G = 1) unless the rows are long (row_stride
//     above the long-row threshold) and too few to fill the GPU; then G CTAs
//     may split each row, G = min(16, capacity / num_rows, row_stride / 8192);
//   - a split is kept only if it takes at least kSplitGain elements off the
//     longest share a CTA streams (row_stride * (G - 1) / G >= kSplitGain).
//     Measured on a GB300: a CTA filters about 6144 elements per 1.1 us, and
//     merging a row across a group costs about 16 us more than finishing it in
//     one CTA, so smaller savings lose (64 rows of 163840 run faster whole,
//     16 rows of 131072 faster split nine ways);
//   - where the device runs thread-block clusters of G CTAs (G <= 8), the CTAs
//     of a group form one cluster and merge in its distributed shared memory;
//     the split is then the largest size up to 8 whose clusters can all be
//     resident with one per row, and kept if it saves at least
//     kSplitGainCluster elements per CTA; otherwise they merge through the
//     workspace with a grid-level barrier;
//   - rows of at least 65536 elements, fewer than half the SMs, are split over
//     thread-block clusters of the short-row kernel: the largest size up to 8
//     with rows x size <= num_sms whose clusters can all be resident, one row
//     per cluster, if each CTA's expected filter candidates stay within
//     kShortMaxCandidates; whole rows take that kernel only under the same
//     bound and up to kShortMaxWholeStride elements, and longer rows that it
//     cannot split take the wide shape;
//   - G = 1 launches min(num_rows, capacity) persistent CTAs, no waiting;
//     with at least kPairRowsPerSm rows per SM of at most kPairMaxStride
//     elements it uses the paired shape (two CTAs of 12 consumer warps per
//     SM); otherwise the short-row kernel (one CTA of 32 warps per SM, rows
//     resident in or streamed through its 128 KB ring) where the device holds
//     it and TopK is below half the row stride; otherwise the wide shape;
//   - a device whose shared memory per block cannot hold the wide shape gets
//     whole rows on the paired shape if it fits, else on the small shape
//     (about 83 KB), else TOPK_ERR_PLAN;
//   - a workspace merge launches num_groups = min(capacity / G, num_rows,
//     num_sms) groups cooperatively, so grid = num_groups * G <= num_sms *
//     ctas_per_sm always; a cluster merge launches at most cluster_groups[G]
//     groups, and its CTAs wait only on CTAs of their own cluster.
#include <stdint.h>

#include <algorithm>
#include <cmath>

#include "libtopk.h"
#include "topk_internal.h"

namespace ltk {

// The planner's rules, from sweeps on a GB300 (bench.py --sweep; the tables
// behind them are in profiles/planner_sweep.md).
constexpr int kMinSpan = 8192;                      // fewest elements per CTA when a row is split
constexpr int64_t kDefaultLongRowThreshold = 32768;  // rows longer than this may be split (wide shape)
constexpr int64_t kSplitGain = 90000;         // elements a workspace-merged split must save per CTA (measured)
constexpr int64_t kSplitGainCluster = 24000;  // elements a cluster-merged split must save per CTA
constexpr int64_t kPairRowsPerSm = 4;         // rows per SM from which the paired shape is planned
constexpr int64_t kPairMaxStride = 16384;     // ... for rows up to this long (longer: the short-row kernel)
constexpr int64_t kShortMaxLen = 32768;       // longest row the short-row kernel holds resident in its ring
constexpr int64_t kShortSeedLen = 2048;       // elements it samples for its threshold (rows this short: all)
// Rows at least this long, too few to give every SM its own, are split over a
// thread-block cluster of the short-row kernel (16 warps per CTA): clusters of
// 2 .. 8 CTAs finish 32768-element rows in 12.3 us against 14.1 to 14.3 us
// whole (1 to 16 rows; 64 rows tie), 65536-element rows in 12.3 against 16.4
// us, 2^20 in 20.6 against 41.2 us for the other kernel's split; on shorter
// rows they gain nothing (8192, 16384: 12.3 either way).
constexpr int64_t kShortClusterStride = 32768;
// The short-row kernel samples 2048 elements for its threshold, so on long
// rows the threshold keeps many more candidates than TopK (expected count:
// short_row_candidates). A CTA that streams its row is planned at most this
// many: more overflow its candidate regions now and then, and the exact
// fallback that follows reads the row from global memory several times (TopK
// 2048, four rows of 2^20 elements whole, about 6100 candidates each, 654 us,
// split over clusters of 8 CTAs 22 us; TopK 4096, 64 rows of 65536, about 5200
// each, 73.7 us whole, 16.6 us over clusters of 2).
constexpr double kShortMaxCandidates = 4096.0;
// Longest row the short-row kernel is planned to select whole: beyond it the
// 2048-element sample holds so few of the row's TopK best that its threshold
// scatters widely (TopK 512, rows of 2^20: 706 us whole against 476 us on the
// wide shape; TopK 2048, 2^19: 354 us against 66 us), while 2^18 still wins
// (TopK 2048, 152 rows: 36.9 us against 45.1 us).
constexpr int64_t kShortMaxWholeStride = 1 << 18;
// Longest rows planned whole on the 16-warp instance of the short-row kernel,
// at any TopK and at TopK up to kShort16LongTopK (TopK 512 of 4096-element
// rows 10.2 against 11.8 us, of 16384 10.2 to 12.3 against 10.3 to 12.3; TopK
// 2048 of 16384 14.3 against 12.3 us).
constexpr int64_t kShort16MaxStride = 4096;
constexpr int64_t kShort16MaxLongStride = 16384;
constexpr int kShort16LongTopK = 512;
// Largest share of a row (elements per CTA) planned on the 16-warp instance
// when rows are split over clusters; larger shares stream faster on 32 warps
// (81920 per CTA, mtp, 19.1 against 20.8 us on 16 warps; 131072 per CTA, one
// row of 2^20 over 8 CTAs, 22.1 against 20.5 us).
constexpr int64_t kShort16MaxShare = 98304;

}  // namespace ltk

namespace {

bool topk_supported(int topk) { return topk >= 1 && topk <= ltk::kWideMaxTopK; }

// The two instances of the short-row kernel (32 and 16 warps per CTA).
bool is_short(int shape) { return shape == ltk::kShapeShort || shape == ltk::kShapeShort16; }

// Candidates the short-row kernel's filter is expected to keep on a row of
// `stride` elements: its threshold keeps mu + 3 sqrt(mu) + 2 keys of the
// kShortSeedLen-element sample (mu = topk * kShortSeedLen / stride, the
// sample's expected share of the row's TopK best), projected over the row.
double short_row_candidates(int64_t stride, int topk) {
  const double rho = static_cast<double>(stride) / static_cast<double>(ltk::kShortSeedLen);
  if (rho <= 1.0) return topk;
  return topk + 3.0 * std::sqrt(topk * rho) + 2.0 * rho;
}

}  // namespace

extern "C" int topk_make_plan(const topk_device_props* props, int64_t num_rows, int64_t row_stride,
                              int next_n, int topk, const topk_options* options, topk_plan* plan) {
  if (props == nullptr || plan == nullptr) return TOPK_ERR_INVALID_ARG;
  if (num_rows < 0 || row_stride < 1 || next_n < 1 || (num_rows % next_n) != 0)
    return TOPK_ERR_INVALID_ARG;
  if (!topk_supported(topk)) return TOPK_ERR_UNSUPPORTED_TOPK;
  *plan = topk_plan{};
  const int merge = (options != nullptr) ? options->merge : 0;
  if (merge < 0 || merge > 2) return TOPK_ERR_INVALID_ARG;
  const int shape = (options != nullptr) ? options->shape : 0;
  if (shape < 0 || shape > ltk::kShapeShort16) return TOPK_ERR_INVALID_ARG;
  const int force = (options != nullptr) ? options->force_ctas_per_group : 0;
  if (force < 0 || force > ltk::kMaxGroup) return TOPK_ERR_INVALID_ARG;
  // the paired and small shapes split no row; the short-row kernel splits one
  // over a thread-block cluster of up to 8 CTAs
  if (shape > ltk::kShapeWide && force > 1 && (!is_short(shape) || force > ltk::kMaxCluster))
    return TOPK_ERR_INVALID_ARG;
  if (props->num_sms < 1) return TOPK_ERR_PLAN;
  const bool wide_ok = props->ctas_per_sm >= 1 && props->smem_per_cta <= props->max_smem_optin;
  const bool pair_ok = props->pair_ctas_per_sm >= 1 && props->pair_smem_per_cta <= props->max_smem_optin;
  const bool small_ok = props->small_ctas_per_sm >= 1 && props->small_smem_per_cta <= props->max_smem_optin;
  const bool short_ok = props->short_ctas_per_sm >= 1 && props->short_smem_per_cta <= props->max_smem_optin;
  const bool short16_ok = props->short16_ctas_per_sm >= 1 && props->short16_smem_per_cta <= props->max_smem_optin;

  // the CTA shape when it is not the planner's to choose, or when the wide
  // shape does not fit the device (then the largest whole-row shape that fits)
  int chosen = shape;
  if (chosen == 0 && !wide_ok) chosen = pair_ok ? ltk::kShapePair : ltk::kShapeSmall;
  if (chosen == ltk::kShapeWide && !wide_ok) return TOPK_ERR_PLAN;
  if (chosen == ltk::kShapePair && !pair_ok) return TOPK_ERR_PLAN;
  if (chosen == ltk::kShapeSmall && !small_ok) return TOPK_ERR_PLAN;
  if (chosen == ltk::kShapeShort && !short_ok) return TOPK_ERR_PLAN;
  if (chosen == ltk::kShapeShort16 && !short16_ok) return TOPK_ERR_PLAN;
  if (chosen == ltk::kShapePair && topk > ltk::kPairMaxTopK) return TOPK_ERR_UNSUPPORTED_TOPK;
  if (chosen == ltk::kShapeSmall && topk > ltk::kSmallMaxTopK) return TOPK_ERR_UNSUPPORTED_TOPK;

  int64_t cap = static_cast<int64_t>(props->num_sms) * props->ctas_per_sm;
  if (options != nullptr && options->max_ctas > 0) cap = std::min<int64_t>(cap, options->max_ctas);
  const int64_t threshold = (options != nullptr && options->long_row_threshold > 0)
                                ? options->long_row_threshold
                                : ltk::kDefaultLongRowThreshold;
  auto clusters_of = [&](int64_t c) -> int64_t {
    return (c >= 2 && c <= ltk::kMaxCluster) ? props->cluster_groups[c] : 0;
  };
  // the short-row kernel's cluster split of each row: the largest size up to
  // 8 with rows x size within the SMs whose clusters are all resident at once,
  // if its CTAs' expected candidates stay within kShortMaxCandidates (0: none)
  const double candidates = short_row_candidates(row_stride, topk);
  // resident clusters of each size for an instance of the short-row kernel
  auto short_groups = [&](int s) -> const int* {
    return s == ltk::kShapeShort16 ? props->short16_cluster_groups : props->short_cluster_groups;
  };
  auto short_cluster_size = [&](int s) -> int64_t {
    const bool ok = s == ltk::kShapeShort16 ? short16_ok : short_ok;
    if (!ok || force != 0 || merge == 1 || num_rows < 1 || row_stride < ltk::kShortClusterStride ||
        2 * static_cast<int64_t>(topk) >= row_stride)
      return 0;
    int64_t sms = props->num_sms;
    if (options != nullptr && options->max_ctas > 0) sms = std::min<int64_t>(sms, options->max_ctas);
    int64_t g = std::min<int64_t>(ltk::kMaxCluster, sms / num_rows);
    while (g >= 2 && short_groups(s)[g] < num_rows) --g;
    return (g >= 2 && candidates / static_cast<double>(g) <= ltk::kShortMaxCandidates) ? g : 0;
  };
  // the split runs on the 16-warp instance where the device holds it (faster:
  // mtp 19.1 against 20.8 us, long_coop 15.0 against 15.5 us on a GB300),
  // unless each CTA's share of the row is large
  int split_shape = short16_ok ? ltk::kShapeShort16 : ltk::kShapeShort;
  if (split_shape == ltk::kShapeShort16 && short_ok) {
    const int64_t g16 = short_cluster_size(ltk::kShapeShort16);
    if (g16 >= 2 && row_stride > ltk::kShort16MaxShare * g16) split_shape = ltk::kShapeShort;
  }
  // whole rows: resident in the short-row kernel's ring (an overflow of its
  // candidate regions then costs an exact pass over the ring: TopK 4096 of
  // 32768, 16.4 us against 22.5 us on the wide shape), or streamed with their
  // candidates within the regions and their threshold sample adequate
  const bool short_whole =
      short_ok && (row_stride <= ltk::kShortMaxLen ||
                   (candidates <= ltk::kShortMaxCandidates && row_stride <= ltk::kShortMaxWholeStride));
  int64_t G = 1;
  bool cluster = false;
  if (chosen == 0 && short_cluster_size(split_shape) >= 2) {
    chosen = split_shape;  // few long rows: split over clusters of the short-row kernel
  } else if (chosen <= ltk::kShapeWide) {  // the wide shape, given or still open
    if (force != 0) {
      G = force;
      if (G > 1) {
        if (merge == 2 && clusters_of(G) < 1) return TOPK_ERR_PLAN;
        cluster = merge == 2 || (merge == 0 && clusters_of(G) >= 1);
      }
    } else if (num_rows > 0 && row_stride > threshold && num_rows < cap && (!short_whole || shape == ltk::kShapeWide)) {
      G = cap / num_rows;
      G = std::min<int64_t>(G, ltk::kMaxGroup);
      G = std::min<int64_t>(G, std::max<int64_t>(1, row_stride / ltk::kMinSpan));
      // the largest cluster size whose clusters hold every row at once
      int64_t gc = (merge != 1 && G >= 2) ? std::min<int64_t>(G, ltk::kMaxCluster) : 0;
      while (gc >= 2 && clusters_of(gc) < num_rows) --gc;
      if (gc >= 2) {
        G = gc;
        cluster = true;
      } else if (merge == 2) {
        G = 1;
      }
      const int64_t gain = cluster ? ltk::kSplitGainCluster : ltk::kSplitGain;
      if (G < 2 || row_stride * (G - 1) / G < gain) {
        G = 1;
        cluster = false;
      }
    }
    // whole rows: the paired shape (two narrower CTAs per SM, one CTA's row
    // finish overlapping the other's streaming) when every SM gets several
    // short rows; else the short-row kernel, unless TopK is half the row or
    // more on rows longer than its sample (its sampled threshold then rarely
    // brackets the K-th key) or its expected candidates overflow; else the wide
    // shape. Measured on a GB300 (bench.py --sweep, TopK 512 to 2048): the
    // paired shape wins from 608 rows of up to 16384 elements, the short-row
    // kernel at 32768 and beyond and for fewer rows, the wide shape for TopK
    // 2048 of 4096-element rows
    if (chosen == 0) {
      const bool many = num_rows >= ltk::kPairRowsPerSm * props->num_sms;
      const bool pair = G == 1 && topk <= ltk::kPairMaxTopK && pair_ok && props->pair_ctas_per_sm >= 2 && many &&
                        (row_stride <= ltk::kPairMaxStride || !short_ok);
      const bool shrt = G == 1 && short_whole &&
                        (row_stride <= ltk::kShortSeedLen || 2 * static_cast<int64_t>(topk) < row_stride);
      // short rows on the 16-warp instance, whose block-wide phases cost half
      // the instructions; longer ones on the 32-warp one, whose filter keeps up
      const bool shrt16 = short16_ok && (row_stride <= ltk::kShort16MaxStride ||
                                         (row_stride <= ltk::kShort16MaxLongStride && topk <= ltk::kShort16LongTopK));
      chosen = pair ? ltk::kShapePair : shrt ? (shrt16 ? ltk::kShapeShort16 : ltk::kShapeShort) : ltk::kShapeWide;
    }
  }
  if (is_short(chosen) && force > 1) {
    // a row split over a cluster of the short-row kernel: one row per cluster,
    // merged in its shared memory only
    if (merge == 1 || short_groups(chosen)[force] < 1) return TOPK_ERR_PLAN;
    G = force;
    cluster = true;
  } else if (is_short(chosen) && G == 1) {
    const int64_t g = short_cluster_size(chosen);  // also when the short-row kernel was asked for
    if (g >= 2) {
      G = g;
      cluster = true;
    }
  }
  plan->shape = chosen;
  if (chosen == ltk::kShapeWide) {
    plan->threads = ltk::kWideCtaThreads;
    plan->smem_bytes = props->smem_per_cta;
  } else {
    const int per_sm = chosen == ltk::kShapePair    ? props->pair_ctas_per_sm
                       : chosen == ltk::kShapeSmall ? props->small_ctas_per_sm
                       : chosen == ltk::kShapeShort ? props->short_ctas_per_sm
                                                    : props->short16_ctas_per_sm;
    plan->threads = chosen == ltk::kShapePair    ? ltk::kPairCtaThreads
                    : chosen == ltk::kShapeSmall ? ltk::kSmallCtaThreads
                    : chosen == ltk::kShapeShort ? ltk::kShortCtaThreads
                                                 : ltk::kShort16CtaThreads;
    plan->smem_bytes = chosen == ltk::kShapePair    ? props->pair_smem_per_cta
                       : chosen == ltk::kShapeSmall ? props->small_smem_per_cta
                       : chosen == ltk::kShapeShort ? props->short_smem_per_cta
                                                    : props->short16_smem_per_cta;
    cap = static_cast<int64_t>(props->num_sms) * per_sm;
    if (options != nullptr && options->max_ctas > 0) cap = std::min<int64_t>(cap, options->max_ctas);
  }
  plan->ctas_per_group = static_cast<int>(G);
  plan->cluster = cluster ? 1 : 0;
  if (num_rows == 0) {
    plan->num_groups = 0;
    plan->grid = 0;
    plan->cooperative = (G > 1 && !cluster) ? 1 : 0;
    return TOPK_OK;
  }
  int64_t groups;
  if (is_short(chosen) && G > 1) {
    // one row per cluster; clusters that are not resident wait for a free slot
    if (num_rows > INT32_MAX / G) return TOPK_ERR_PLAN;
    groups = num_rows;
    plan->cooperative = 0;
  } else if (G == 1) {
    groups = std::min<int64_t>(num_rows, cap);
    plan->cooperative = 0;
  } else if (cluster) {
    // clusters never wait on one another; the hardware co-schedules each one
    groups = std::min<int64_t>(num_rows, clusters_of(G));
    groups = std::min<int64_t>(groups, cap / G);
    groups = std::min<int64_t>(groups, props->num_sms);  // workspace holds num_sms groups
    if (groups < 1) return TOPK_ERR_PLAN;
    plan->cooperative = 0;
  } else {
    groups = std::min<int64_t>(cap / G, num_rows);
    groups = std::min<int64_t>(groups, props->num_sms);  // workspace holds num_sms groups
    if (groups < 1) return TOPK_ERR_PLAN;
    plan->cooperative = 1;
  }
  plan->num_groups = static_cast<int>(groups);
  plan->grid = static_cast<int>(groups * G);
  return TOPK_OK;
}
