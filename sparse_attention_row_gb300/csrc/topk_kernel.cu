// Ragged per-row top-K for sm_103a: seeded streaming filter + exact radix select.
//
// One kernel serves every row length. A CTA (or a group of G CTAs that split
// one row) streams its part of the row from HBM through a ring of shared-memory
// slots. A dedicated copy warp keeps the ring full with bulk asynchronous
// copies (cp.async.bulk, completion counted on "full" mbarriers; consumers free
// slots through "empty" mbarriers), so each logit crosses HBM exactly once.
//
// Filtering: the first staged chunk of a row is histogrammed on the top 12 bits
// of the keys and seeds a threshold aimed at about 1.25 K survivors over the
// whole row. Every later element costs one fp32 compare against that threshold;
// only survivors become (key, index) candidates in shared memory. The consumer
// warps form groups that own ring slots, and each group filters the chunks of
// its slots on its own, with no CTA-wide barrier between chunks. At the end of the
// row the seed is verified: if fewer than K elements reached it, or the
// candidates outgrew the buffer (heavy ties at the seed's bin), the row is
// streamed again in index order with no seed (exact whatever the data); there a
// buffer that runs full is shrunk, first to the current threshold bin, then if
// needed to exactly the K best, raising the threshold each time.
//
// Selection: an exact radix select on the composite key (value bits, then index)
// finds the K-th candidate (T, I); the output is {key > T} + {key == T, index <=
// I}, so equal values go to the smaller index.
//
// Split rows (G > 1 CTAs per row) merge in one of two ways. Where the G CTAs
// form a thread-block cluster, each reads the others' bin counts through
// distributed shared memory, all find the same threshold bin, and the members
// append their candidates to the leader's buffer, which then finishes the row
// as a whole-row CTA would (cluster_merge). Otherwise, or when that union
// would not fit, the CTAs merge their histograms through a workspace in global
// memory, meeting at a group barrier after each radix pass (finish_group);
// this replaces the per-row RadixRowState of the persistent_topk kernel (vLLM
// PR #41444 page, "Executive summary": arrival counter plus histogram per row
// group). Every workspace word a launch touches is returned to zero before the
// launch ends, with the fencing that the vLLM PR #41748 page's review asks for
// ("Code Review": zero in parallel, reset the arrival counter only after the
// zeros are visible), so no per-call memset is needed and graph replays start
// from a clean workspace.
//
// Strided logits (a column stride above 1) have no contiguous run to copy: the
// consumers then read each row from global memory element by element through
// the unseeded streaming path, and the copy warp stays idle.
//
// Keys: an fp32 value x maps to a uint32 whose unsigned order is the order of
// the values: -0.0 is first mapped to +0.0, then positive values get the sign
// bit set and negative values are bit-inverted.
//
// Code size: a decode-sized launch runs every phase once per SM, right after
// other kernels have evicted this one's code from L2, so each instruction line
// it executes is a cold fetch (ncu shows "no instruction" as the second stall
// reason there). Phases run once per row (radix finds, ranking) and the rare
// paths (buffer shrinking, re-streaming, the group merge, the radix fallback)
// are therefore out of line, and the row finish uses short rolled loops.

#include <cuda_runtime.h>
#include <stdint.h>

#include "topk_internal.h"

// This file is compiled three times: as is (the wide CTA shape, namespace
// ltk::wide), from topk_kernel_pair.cu with LTK_SHAPE_PAIR set (two narrower
// CTAs per SM, ltk::pair) and from topk_kernel_small.cu with LTK_SHAPE_SMALL
// set (a CTA that fits in about 83 KB of shared memory, ltk::small).
#ifndef LTK_SHAPE_PAIR
#define LTK_SHAPE_PAIR 0
#endif
#ifndef LTK_SHAPE_SMALL
#define LTK_SHAPE_SMALL 0
#endif
#if LTK_SHAPE_PAIR
#define LTK_SHAPE_NS pair
#elif LTK_SHAPE_SMALL
#define LTK_SHAPE_NS small
#else
#define LTK_SHAPE_NS wide
#endif

namespace ltk {
namespace LTK_SHAPE_NS {

#if LTK_SHAPE_PAIR
constexpr int kTopKMax = kPairMaxTopK;
constexpr int kThreads = 384;   // consumer threads per CTA (12 warps)
constexpr int kChunk = 3072;    // fp32 elements per staging slot (12 KB)
constexpr int kStages = 3;      // staging slots per CTA (36 KB)
constexpr int kBufCap = 6144;   // candidate (key, index) pairs kept per CTA
constexpr int kMinBlocks = 2;   // CTAs per SM the shape is built for
#elif LTK_SHAPE_SMALL
constexpr int kTopKMax = kSmallMaxTopK;
constexpr int kThreads = 256;   // consumer threads per CTA (8 warps)
constexpr int kChunk = 2048;    // fp32 elements per staging slot (8 KB)
constexpr int kStages = 3;      // staging slots per CTA (24 KB)
constexpr int kBufCap = 4096;   // candidate (key, index) pairs kept per CTA
constexpr int kMinBlocks = 1;
#else
constexpr int kTopKMax = kWideMaxTopK;
constexpr int kThreads = 768;   // consumer threads per CTA (24 warps)
constexpr int kChunk = 6144;    // fp32 elements per staging slot (24 KB)
constexpr int kStages = 4;      // staging slots per CTA (96 KB)
constexpr int kBufCap = 12288;  // candidate (key, index) pairs kept per CTA
constexpr int kMinBlocks = 1;
#endif
constexpr int kWarps = kThreads / 32;
// Warp groups of the streaming loop: group g filters exactly the chunks staged
// in the ring slots s with s % kGroups == g, so each group waits on its own
// slots' phases in order and a warp filters a whole chunk's share of
// kChunk / (4 * kGroupThreads) float4 per lane (every warp still reads the
// seed chunk of a row for its histogram).
// Paired shape: 3 groups of 4 warps, one slot each. Wide shape: 2 groups of
// 12 warps, two slots each, so a group's next chunk is in flight while it
// filters one (measured faster than 4 groups of 6 on split rows). Small
// shape: one group (8 warps do not divide into its 3 slots).
constexpr int kGroups = LTK_SHAPE_PAIR ? kStages : (LTK_SHAPE_SMALL ? 1 : 2);
static_assert(kStages % kGroups == 0 && kWarps % kGroups == 0, "groups own whole slots and whole warps");
constexpr int kGroupWarps = kWarps / kGroups;
constexpr int kGroupThreads = kGroupWarps * 32;
static_assert(kChunk % (4 * kGroupThreads) == 0 && kChunk / (4 * kGroupThreads) <= 8,
              "a group's share of a chunk fits one 32-bit survivor mask per lane");
constexpr int kCtaThreads = kThreads + 32;  // plus one copy-issuing warp
static_assert(kCtaThreads == (LTK_SHAPE_PAIR ? kPairCtaThreads : LTK_SHAPE_SMALL ? kSmallCtaThreads : kWideCtaThreads),
              "shape constants agree");
static_assert(kThreads - 32 >= kSmallSet, "close_window pads the ranking slots with all but warp 0");

static_assert(kTopKMax + kChunk <= kBufCap, "a chunk must fit next to topk kept candidates");
static_assert(kChunk % (4 * kThreads) == 0, "a chunk is a whole number of float4 per thread");

struct __align__(128) Smem {
  float stage[kStages][kChunk];   // staging ring (bulk-copy destination)
  uint32_t hist[kBins];           // histogram of kept keys (also radix scratch)
  uint32_t bkey[kBufCap];         // candidate keys
  int32_t bidx[kBufCap];          // candidate indices (row-relative)
  int32_t emit[kListCap];         // bin-t entries of the row being finished; staged survivors
  int32_t small[kSmallSet];       // candidate positions ranked by rank_small
  alignas(16) uint32_t rk[kSmallSet];  // their keys, copied for ranking
  alignas(16) int32_t ri[kSmallSet];   // their indices
  alignas(16) uint32_t sub[256];  // 8-bit sub-histogram of the threshold bin
  uint32_t bsum[kBins / 32];      // 32-bin block sums used by block_find
  unsigned long long full[kStages];
  unsigned long long empty[kStages];
  unsigned long long xbar[2];     // cluster merge barriers (one arrival per member CTA)
  int32_t lens[kLenCache];
  uint32_t wtot[kWarps];
  int g_e[kMaxGroup];
  int g_tot[kMaxGroup];
  int buf_n, buf_mark, n_emit, n_small;
  int t, cnt_ge;
  uint32_t thr_lo;
  float thr_f;
  int find_b, find_gt;
  int abort, last, off, take;
  int full_row;  // the buffer reached its mark: this row is streamed again at its end
  int n_list;
  uint32_t red;
  uint32_t sel_T;
  int sel_I;
  uint32_t run_kmin, run_kmax;  // tied_run's extremes
  int run_imin, run_imax;
  int x_t, x_in;                  // cluster merge: t_max, then the count in bin t*
  int x_n0;                       // cluster merge: this CTA's buffer size when the merge began
  int x_ln;                       // cluster merge: the leader's buffer size, as read here
  int x_push;                     // cluster merge: entries the other members appended (leader only)
  int x_hi;                       // cluster merge: highest occupied bin of this CTA (-1: none)
  int x_top;                      // cluster merge: highest occupied bin of any member
};

// ---------------------------------------------------------------- primitives

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Barrier among the consumer warps only (the copy warp never joins it).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"r"(kThreads) : "memory"); }

// Consumer barrier that also ORs a predicate over the consumer threads: every
// thread gets the same answer, so a decision taken from it is uniform even when
// the state it was computed from changes right after the barrier.
__device__ __forceinline__ bool csync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(kThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for an mbarrier phase, giving up after timeout_ns or when *abort is set.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity,
                                                  uint64_t timeout_ns, const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (global_timer() - t0 > timeout_ns) return false;
  }
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Distributed shared memory of a thread-block cluster: the address of the same
// shared variable in the CTA of cluster rank `rank`, and accesses through it.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}

__device__ __forceinline__ uint32_t dsmem_ld(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void dsmem_st(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t dsmem_atom_add(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

// Arrives on an mbarrier of another CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The hardware cluster barrier, split: every thread of every CTA arrives once
// at kernel start (after the merge barriers are initialised); a thread that
// will touch another CTA's shared memory waits first, which completes once
// every thread of the cluster has arrived (threads that exited count as
// arrived). Warp-uniform in both halves.
__device__ __forceinline__ void cluster_arrive_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_all() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// The CTA's abort flag. It is set by this CTA's own threads and, in a cluster
// launch, by a member CTA that gave up, at any time: every CTA-wide decision
// taken from it goes through a reducing barrier (csync_or), so that all
// consumer warps take the same branch.
__device__ __forceinline__ bool abort_set(const int* flag) { return *reinterpret_cast<const volatile int*>(flag) != 0; }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Order-preserving key of an fp32 value (see the file comment).
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t u = __float_as_uint(x);
  u = (u == 0x80000000u) ? 0u : u;
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// fp32 value whose ">=" test is equivalent to "key >= k" for every non-NaN input.
__device__ __forceinline__ float key_floor_value(uint32_t k) {
  if (k <= 0x007FFFFFu) return -__int_as_float(0x7F800000);  // at or below key(-inf): all pass
  if (k > 0xFF800000u) return __int_as_float(0x7FC00000);     // above key(+inf): NaN, none pass
  const uint32_t u = (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k;
  return __uint_as_float(u);
}

// Appends `val` to list[] (capacity `cap`) for every lane with `pred`, one
// shared atomic per warp. Entries past the capacity are dropped (never written).
template <typename T>
__device__ __forceinline__ void warp_push(T* list, int* counter, int cap, bool pred, T val) {
  const uint32_t m = __ballot_sync(0xFFFFFFFFu, pred);
  if (m == 0) return;
  int base = 0;
  if (lane_id() == 0) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  const int o = base + __popc(m & lanemask_lt());
  if (pred && o < cap) list[o] = val;
}

// ----------------------------------------------------------------- radix find

// Over hist[0, nb) (nb a power of two, 32..4096): with from_top, finds the
// largest bin b whose suffix sum (bins >= b) reaches `need`; otherwise the
// smallest bin b whose prefix sum (bins <= b) reaches `need`. Writes b to
// s.find_b and the count strictly beyond b (above it, or below it) to
// s.find_gt. Requires need >= 1 and a total of at least need.
// Short dependency chains: every warp sums whole 32-bin blocks with one warp
// reduction each; one warp then scans the block sums (4 per lane) and the one
// block holding the crossing. Consumer-wide; starts and ends with a barrier.
__device__ __noinline__ void block_find(Smem& s, const uint32_t* hist, int nb, int need, bool from_top) {
  const int tid = threadIdx.x;
  const int lane = static_cast<int>(lane_id());
  const int warp = tid >> 5;
  const int nblk = nb >> 5;
  csync();
  for (int q = warp; q < nblk; q += kWarps) {
    const int pos = 32 * q + lane;  // scan position: bin nb-1-pos from the top, bin pos from the bottom
    const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, hist[from_top ? nb - 1 - pos : pos]);
    if (lane == 0) s.bsum[q] = sum;
  }
  csync();
  if (warp == 0) {
    uint32_t b4[4];
    uint32_t own = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int q = 4 * lane + k;
      b4[k] = (q < nblk) ? s.bsum[q] : 0u;
      own += b4[k];
    }
    uint32_t incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl >= static_cast<uint32_t>(need));
    const int L = hit ? __ffs(hit) - 1 : 31;
    uint32_t run = incl - own;
    int qsel = 0;
    if (lane == L) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (run + b4[k] >= static_cast<uint32_t>(need)) {
          qsel = 4 * lane + k;
          break;
        }
        run += b4[k];
      }
    }
    qsel = __shfl_sync(0xFFFFFFFFu, qsel, L);
    run = __shfl_sync(0xFFFFFFFFu, run, L);
    const int pos = 32 * qsel + lane;
    const int bin = from_top ? nb - 1 - pos : pos;
    const uint32_t h = hist[bin];
    uint32_t in2 = h;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, in2, o);
      if (lane >= o) in2 += v;
    }
    const uint32_t hit2 = __ballot_sync(0xFFFFFFFFu, run + in2 >= static_cast<uint32_t>(need));
    const int L2 = hit2 ? __ffs(hit2) - 1 : 0;
    if (lane == L2) {
      s.find_b = bin;
      s.find_gt = static_cast<int>(run + in2 - h);
    }
  }
  csync();
}

// hist[(key >> shift) & mask] counts buffer entries with (key >> pshift) == prefix.
__device__ void hist_keys(Smem& s, int nb, uint32_t prefix, int pshift, int shift, uint32_t mask) {
  const int tid = threadIdx.x;
  csync();
  for (int b = tid; b < nb; b += kThreads) s.hist[b] = 0;
  csync();
  const int n = s.buf_n;
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t k = s.bkey[i];
    if ((k >> pshift) == prefix) atomicAdd(&s.hist[(k >> shift) & mask], 1u);
  }
  csync();
}

// hist[(idx >> shift) & mask] counts entries with key == T and (idx >> pshift) == prefix.
__device__ void hist_tied_indices(Smem& s, int nb, uint32_t T, uint32_t prefix, int pshift, int shift,
                                  uint32_t mask) {
  const int tid = threadIdx.x;
  csync();
  for (int b = tid; b < nb; b += kThreads) s.hist[b] = 0;
  csync();
  const int n = s.buf_n;
  for (int i = tid; i < n; i += kThreads) {
    if (s.bkey[i] != T) continue;
    const uint32_t x = static_cast<uint32_t>(s.bidx[i]);
    if ((x >> pshift) == prefix) atomicAdd(&s.hist[(x >> shift) & mask], 1u);
  }
  csync();
}

// Smallest key among buffer entries with (key >> pshift) == prefix.
__device__ uint32_t block_min_key(Smem& s, uint32_t prefix, int pshift) {
  csync();
  if (threadIdx.x == 0) s.red = 0xFFFFFFFFu;
  csync();
  uint32_t mn = 0xFFFFFFFFu;
  const int n = s.buf_n;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint32_t k = s.bkey[i];
    if ((k >> pshift) == prefix) mn = min(mn, k);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
  if (lane_id() == 0 && mn != 0xFFFFFFFFu) atomicMin(&s.red, mn);
  csync();
  return s.red;
}

// Largest index among entries with key == T and (idx >> pshift) == prefix.
__device__ int block_max_tied_index(Smem& s, uint32_t T, uint32_t prefix, int pshift) {
  csync();
  if (threadIdx.x == 0) s.red = 0u;
  csync();
  uint32_t mx = 0u;
  const int n = s.buf_n;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    if (s.bkey[i] != T) continue;
    const uint32_t x = static_cast<uint32_t>(s.bidx[i]);
    if ((x >> pshift) == prefix) mx = max(mx, x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  if (lane_id() == 0 && mx != 0u) atomicMax(&s.red, mx);
  csync();
  return static_cast<int>(s.red);
}

// Number of buffer entries for which pred(key, idx) holds.
template <class Pred>
__device__ int block_count(Smem& s, Pred pred) {
  csync();
  if (threadIdx.x == 0) s.red = 0u;
  csync();
  const int warp = threadIdx.x >> 5;
  const int n = s.buf_n;
  for (int base = warp * 32; base < n; base += kThreads) {
    const int i = base + static_cast<int>(lane_id());
    const bool p = i < n && pred(s.bkey[i], s.bidx[i]);
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, p);
    if (lane_id() == 0 && m) atomicAdd(&s.red, static_cast<uint32_t>(__popc(m)));
  }
  csync();
  return static_cast<int>(s.red);
}

// Collects the positions of the entries for which pred holds into s.small
// (the caller knows there are at most kSmallSet of them); returns the count.
template <class Pred>
__device__ int gather_small(Smem& s, Pred pred) {
  csync();
  if (threadIdx.x == 0) s.n_small = 0;
  csync();
  const int warp = threadIdx.x >> 5;
  const int n = s.buf_n;
  for (int base = warp * 32; base < n; base += kThreads) {
    const int i = base + static_cast<int>(lane_id());
    const bool p = i < n && pred(s.bkey[i], s.bidx[i]);
    warp_push<int32_t>(s.small, &s.n_small, kSmallSet, p, i);
  }
  csync();
  return min(s.n_small, kSmallSet);
}

// Ranks the m <= kSmallSet candidates listed (as buffer positions) in s.small
// by (key desc, index asc): thread j < m counts the candidates that beat
// candidate j, reading four at a time so the loads overlap. The need-th best
// (1 <= need <= m) goes to s.sel_T / s.sel_I. Returns this thread's rank
// (kSmallSet for threads without a candidate). Consumer-wide; ends with a barrier.
__device__ __noinline__ int rank_small(Smem& s, int m, int need) {
  const int j = threadIdx.x;
  if (j < kSmallSet) {
    uint32_t k = 0u;
    int32_t x = 0x7FFFFFFF;
    if (j < m) {
      const int pos = s.small[j];
      k = s.bkey[pos];
      x = s.bidx[pos];
    }
    s.rk[j] = k;  // padding entries (key 0, largest index) never beat a real candidate
    s.ri[j] = x;
  }
  csync();
  int rank = kSmallSet;
  if (j < m) {
    const uint32_t kj = s.rk[j];
    const int32_t ij = s.ri[j];
    int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
    for (int i0 = 0; i0 < m; i0 += 4) {
      const uint4 k4 = *reinterpret_cast<const uint4*>(&s.rk[i0]);
      const int4 x4 = *reinterpret_cast<const int4*>(&s.ri[i0]);
      r0 += (k4.x > kj || (k4.x == kj && x4.x < ij)) ? 1 : 0;
      r1 += (k4.y > kj || (k4.y == kj && x4.y < ij)) ? 1 : 0;
      r2 += (k4.z > kj || (k4.z == kj && x4.z < ij)) ? 1 : 0;
      r3 += (k4.w > kj || (k4.w == kj && x4.w < ij)) ? 1 : 0;
    }
    rank = r0 + r1 + r2 + r3;
    if (rank == need - 1) {
      s.sel_T = kj;
      s.sel_I = ij;
    }
  }
  csync();
  return rank;
}

// Among entries with key == T, the need-th smallest index (1 <= need <= count).
// Radix on the index from the top bit down: 11, 10, 10 bits.
__device__ int select_tied_indices(Smem& s, uint32_t T, int need) {
  uint32_t prefix = 0;
  int pshift = 31;
#pragma unroll 1
  for (int l = 0; l < 3; ++l) {
    const int bits = (l == 0) ? 11 : 10;
    const int shift = (l == 0) ? 20 : (l == 1) ? 10 : 0;
    const int nb = 1 << bits;
    hist_tied_indices(s, nb, T, prefix, pshift, shift, static_cast<uint32_t>(nb - 1));
    block_find(s, s.hist, nb, need, false);
    const uint32_t b = static_cast<uint32_t>(s.find_b);
    need -= s.find_gt;
    const int c = static_cast<int>(s.hist[b]);
    prefix = (prefix << bits) | b;
    pshift = shift;
    if (need == c) return block_max_tied_index(s, T, prefix, pshift);
  }
  return static_cast<int>(prefix);
}

// The selection of exactly K in-play entries (bits 31..20 >= t) expressed as a
// composite threshold: the set {key > T} + {key == T and idx <= I}. Small
// candidate sets are ranked by one warp, larger ones go through radix levels.
// Uses hist as scratch.
__device__ __noinline__ void select_threshold(Smem& s, int K, uint32_t& T, int& I) {
  csync();
  const uint32_t t = static_cast<uint32_t>(s.t);
  const int inbin = static_cast<int>(s.hist[t]);
  int need = K - (s.cnt_ge - inbin);
  I = 0x7FFFFFFF;
  if (need >= inbin) {
    T = block_min_key(s, t, 20);
    return;
  }
  if (inbin <= kSmallSet) {
    const int m = gather_small(s, [=](uint32_t k, int32_t) { return (k >> 20) == t; });
    rank_small(s, m, need);
    T = s.sel_T;
    I = s.sel_I;
    return;
  }
  hist_keys(s, kBins, t, 20, 8, 0xFFFu);
  block_find(s, s.hist, kBins, need, true);
  const uint32_t b1 = static_cast<uint32_t>(s.find_b);
  need -= s.find_gt;
  const int c1 = static_cast<int>(s.hist[b1]);
  const uint32_t p1 = (t << 12) | b1;
  if (need >= c1) {
    T = block_min_key(s, p1, 8);
    return;
  }
  if (c1 <= kSmallSet) {
    const int m = gather_small(s, [=](uint32_t k, int32_t) { return (k >> 8) == p1; });
    rank_small(s, m, need);
    T = s.sel_T;
    I = s.sel_I;
    return;
  }
  hist_keys(s, 256, p1, 8, 0, 0xFFu);
  block_find(s, s.hist, 256, need, true);
  const uint32_t b2 = static_cast<uint32_t>(s.find_b);
  need -= s.find_gt;
  const int c2 = static_cast<int>(s.hist[b2]);
  T = (p1 << 8) | b2;
  if (need >= c2) return;
  if (c2 <= kSmallSet) {
    const uint32_t TT = T;
    const int m = gather_small(s, [=](uint32_t k, int32_t) { return k == TT; });
    rank_small(s, m, need);
    I = s.sel_I;
    return;
  }
  I = select_tied_indices(s, T, need);
}

// Writes the indices of the selected entries ({key > T} + {key == T, idx <= I})
// to dst[0, cap) (one shared reservation per warp; entries past cap are
// dropped); returns how many were selected. Consumer-wide; ends with a barrier.
__device__ __noinline__ int emit_selected(Smem& s, uint32_t T, int I, int32_t* dst, int cap) {
  csync();
  if (threadIdx.x == 0) s.n_emit = 0;
  csync();
  const int warp = threadIdx.x >> 5;
  const int n = s.buf_n;
  for (int base = warp * 32; base < n; base += kThreads) {
    const int i = base + static_cast<int>(lane_id());
    bool sel = false;
    int32_t x = 0;
    if (i < n) {
      const uint32_t k = s.bkey[i];
      x = s.bidx[i];
      sel = k > T || (k == T && x <= I);
    }
    warp_push<int32_t>(dst, &s.n_emit, cap, sel, x);
  }
  csync();
  return s.n_emit;
}

// ------------------------------------------------------------ streaming state

__device__ void reset_row_state(Smem& s) {
  for (int b = threadIdx.x; b < kBins; b += kThreads) s.hist[b] = 0;
  if (threadIdx.x == 0) {
    s.buf_n = 0;
    s.buf_mark = 0;
    s.t = 0;
    s.cnt_ge = 0;
    s.thr_lo = 0;
    s.thr_f = key_floor_value(0u);
    s.n_emit = 0;
    s.x_push = 0;  // other members append to a leader only after the next merge's first sync
    s.full_row = 0;
    s.x_hi = -1;
  }
}

__device__ __forceinline__ void set_threshold(Smem& s, uint32_t lo) {
  if (lo > s.thr_lo) {
    s.thr_lo = lo;
    s.thr_f = key_floor_value(lo);
  }
}

// One warp: moves the threshold bin t up as far as the kept counts allow.
// cnt_ge counts buffered keys with bits 31..20 >= t (all of them are in play);
// after the move, at least K of them still sit at or above t and fewer than K
// above it. Raises the filter to the lower edge of bin t.
__device__ void advance_threshold(Smem& s, int K) {
  const int lane = static_cast<int>(lane_id());
  int cnt = s.cnt_ge + (s.buf_n - s.buf_mark);
  int t = s.t;
  if (cnt >= K) {
    auto fine = [&]() -> int {
      const int b = t + lane;
      int q = (b < kBins) ? static_cast<int>(s.hist[b]) : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, q, o);
        if (lane >= o) q += v;
      }
      const int f = __popc(__ballot_sync(0xFFFFFFFFu, cnt - q >= K));
      if (f > 0) {
        cnt -= __shfl_sync(0xFFFFFFFFu, q, f - 1);
        t += f;
      }
      return f;
    };
    if (fine() == 32) {
      // coarse steps over blocks of 32 bins; lanes read skewed to avoid bank conflicts
      while (true) {
        const int b0 = t + 32 * lane;
        int sum = 0;
#pragma unroll 8
        for (int j = 0; j < 32; ++j) {
          const int b = b0 + ((j + lane) & 31);
          sum += (b < kBins) ? static_cast<int>(s.hist[b]) : 0;
        }
        int p = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xFFFFFFFFu, p, o);
          if (lane >= o) p += v;
        }
        const int c = __popc(__ballot_sync(0xFFFFFFFFu, cnt - p >= K));
        if (c > 0) {
          cnt -= __shfl_sync(0xFFFFFFFFu, p, c - 1);
          t += 32 * c;
        }
        if (c < 32 || t >= kBins) break;
      }
      if (t < kBins) fine();
      if (t >= kBins) t = kBins - 1;  // unreachable with consistent counts; keeps t in range
    }
  }
  if (lane == 0) {
    s.cnt_ge = cnt;
    s.t = t;
    s.buf_mark = s.buf_n;
    set_threshold(s, static_cast<uint32_t>(t) << 20);
  }
}

// Keeps the buffer entries for which keep(key, idx) holds. In place, in rounds
// of 4 entries per thread: every round reads before it writes, and the write
// cursor never passes the start of the next round.
template <class Keep>
__device__ void compact_buffer(Smem& s, Keep keep) {
  constexpr int kPer = 4;
  constexpr int kRound = kPer * kThreads;
  const int tid = threadIdx.x;
  csync();
  const int n = s.buf_n;
  csync();
  if (tid == 0) s.buf_n = 0;
  const uint32_t lt = lanemask_lt();
  for (int r0 = 0; r0 < n; r0 += kRound) {
    uint32_t kk[kPer];
    int32_t ii[kPer];
    bool kp[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int e = r0 + j * kThreads + tid;
      kk[j] = 0u;
      ii[j] = 0;
      kp[j] = false;
      if (e < n) {
        kk[j] = s.bkey[e];
        ii[j] = s.bidx[e];
        kp[j] = keep(kk[j], ii[j]);
      }
    }
    csync();
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, kp[j]);
      if (m == 0) continue;
      int base = 0;
      if (lane_id() == 0) base = atomicAdd(&s.buf_n, __popc(m));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (kp[j]) {
        const int o = min(base + __popc(m & lt), kBufCap - 1);
        s.bkey[o] = kk[j];
        s.bidx[o] = ii[j];
      }
    }
    csync();
  }
  csync();
  if (tid == 0) s.buf_mark = s.buf_n;
  csync();
}

// Keeps exactly the K best buffered candidates and raises the filter to
// (K-th key) + 1: a later element equal to that key has a larger index than
// every kept one, so it can never be selected.
// A buffer whose keys are all equal and whose n indices form the contiguous run
// [i0, i0 + n) (n distinct indices spanning n values) holds ties only, and by
// the tie rule its K best are i0 .. i0 + K - 1. One pass finds the key and
// index extremes; returns whether that holds (then T, I describe the K best).
// Consumer-wide; every thread gets the same answer.
__device__ bool tied_run(Smem& s, int K, uint32_t& T, int& I) {
  const int tid = threadIdx.x;
  csync();
  if (tid == 0) {
    s.run_kmin = 0xFFFFFFFFu;
    s.run_kmax = 0u;
    s.run_imin = 0x7FFFFFFF;
    s.run_imax = -1;
  }
  csync();
  const int n = s.buf_n;
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  int imin = 0x7FFFFFFF, imax = -1;
  for (int i = tid; i < n; i += kThreads) {
    const uint32_t k = s.bkey[i];
    const int x = s.bidx[i];
    kmin = min(kmin, k);
    kmax = max(kmax, k);
    imin = min(imin, x);
    imax = max(imax, x);
  }
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  imin = __reduce_min_sync(0xFFFFFFFFu, imin);
  imax = __reduce_max_sync(0xFFFFFFFFu, imax);
  if (lane_id() == 0) {
    atomicMin(&s.run_kmin, kmin);
    atomicMax(&s.run_kmax, kmax);
    atomicMin(&s.run_imin, imin);
    atomicMax(&s.run_imax, imax);
  }
  csync();
  T = s.run_kmin;
  I = s.run_imin + K - 1;
  return n >= K && s.run_kmin == s.run_kmax &&
         static_cast<int64_t>(s.run_imax) - static_cast<int64_t>(s.run_imin) + 1 == n;
}

__device__ __noinline__ void compact_exact(Smem& s, int K) {
  uint32_t T;
  int I;
  const bool run = tied_run(s, K, T, I);
  if (!run) select_threshold(s, K, T, I);
  compact_buffer(s, [=](uint32_t k, int32_t i) { return k > T || (k == T && i <= I); });
  for (int b = threadIdx.x; b < kBins; b += kThreads) s.hist[b] = 0;
  csync();
  const int n = s.buf_n;
  if (run) {
    if (threadIdx.x == 0) s.hist[T >> 20] = static_cast<uint32_t>(n);  // all kept keys are T
  } else {
    for (int i = threadIdx.x; i < n; i += kThreads) atomicAdd(&s.hist[s.bkey[i] >> 20], 1u);
  }
  csync();
  if (threadIdx.x == 0) {
    s.buf_mark = n;
    s.cnt_ge = n;
    s.t = static_cast<int>(T >> 20);
    set_threshold(s, T + 1u);
  }
  csync();
}

// Frees buffer space: raise the threshold bin, drop what fell below it, and if
// that is not enough keep exactly the K best.
__device__ __noinline__ void make_room(Smem& s, int K) {
  csync();
  if (threadIdx.x < 32) advance_threshold(s, K);
  csync();
  const uint32_t t = static_cast<uint32_t>(s.t);
  compact_buffer(s, [=](uint32_t k, int32_t) { return (k >> 20) >= t; });
  if (csync_or(threadIdx.x == 0 && s.buf_n + kChunk > kBufCap)) compact_exact(s, K);
}

// ----------------------------------------------------------------- row plans

struct RowWin {
  int64_t r;
  const float* rowp;
  int len, lo, hi, wstart, wend, nch;
};

__device__ __forceinline__ int clamp_len(const Params& p, int32_t raw) {
  if (raw < 0 || static_cast<int64_t>(raw) > p.max_len) {
    atomicOr(p.status, 0x1u);
    return raw < 0 ? 0 : static_cast<int>(p.max_len);
  }
  return raw;
}

__device__ __forceinline__ int row_len(const Params& p, const Smem& s, int64_t k, int64_t r) {
  if (k < kLenCache) return s.lens[k];
  return clamp_len(p, __ldg(p.lengths + r));
}

// Part of row r (length len) that member m of a group streams, and its copy
// windows.
__device__ __forceinline__ void row_window(const Params& p, int64_t r, int len, int m, RowWin& w) {
  w.r = r;
  w.len = len;
  w.rowp = p.logits + w.r * p.stride;
  w.nch = 0;
  w.lo = w.hi = w.wstart = w.wend = 0;
  if (w.len > p.topk) {
    const int64_t span = ((static_cast<int64_t>(w.len) + p.G - 1) / p.G + 3) & ~static_cast<int64_t>(3);
    const int64_t lo = min(static_cast<int64_t>(m) * span, static_cast<int64_t>(w.len));
    const int64_t hi = min(lo + span, static_cast<int64_t>(w.len));
    w.lo = static_cast<int>(lo);
    w.hi = static_cast<int>(hi);
    if (w.hi > w.lo) {
      // copies start on the 16-byte boundary at or below element lo and end on
      // the one at or above element hi; every 16-byte granule copied holds at
      // least one element of [lo, hi), so no copy leaves the row's pages.
      // Strided rows are read element by element from lo on.
      const int mis = (p.col_stride != 1) ? 0
                          : static_cast<int>((reinterpret_cast<uintptr_t>(w.rowp + w.lo) & 15u) >> 2);
      w.wstart = w.lo - mis;
      w.wend = w.wstart + ((w.hi - w.wstart + 3) & ~3);
      w.nch = (w.wend - w.wstart + kChunk - 1) / kChunk;
    }
  }
}

// Row k of this CTA's group, and this CTA's part of it.
__device__ __forceinline__ bool get_row(const Params& p, const Smem& s, int64_t k, int g, int m,
                                        RowWin& w) {
  const int64_t r = g + k * p.num_groups;
  if (r >= p.num_rows) return false;
  row_window(p, r, row_len(p, s, k, r), m, w);
  return true;
}

// The copy warp issues the first chunk of the CTA's first row early. With whole
// rows per CTA it does so at kernel start, before the length cache is filled:
// the copy window is sized by the row stride, which covers the first chunk of
// any length; it becomes that row's chunk 0, or a chunk the consumers discard
// if the row needs no streaming.
__device__ __noinline__ void producer_first_whole(const Params& p, Smem& s, int g) {
  const float* rowp = p.logits + static_cast<int64_t>(g) * p.stride;
  const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(rowp) & 15u) >> 2);
  const int64_t ws = -mis;
  const int64_t wend = ws + ((p.max_len - ws + 3) & ~static_cast<int64_t>(3));
  const int64_t we = min(ws + kChunk, wend);
  const uint32_t bytes = static_cast<uint32_t>(we - ws) * 4u;
  fence_proxy_async();
  mbar_expect_tx(&s.full[0], bytes);
  bulk_copy_g2s(s.stage[0], rowp + ws, bytes, &s.full[0]);
}

// When rows are split, the copy thread reads the first row's length itself
// (the read is in flight across the start-up barriers) and issues chunk 0 of
// its part, if it has one. Returns whether a copy was issued.
__device__ __noinline__ bool producer_first_split(const Params& p, Smem& s, int g, int m, int32_t raw_len) {
  if (g >= p.num_rows) return false;
  RowWin w;
  row_window(p, g, clamp_len(p, raw_len), m, w);
  if (w.nch == 0) return false;
  const int we = min(w.wstart + kChunk, w.wend);
  const uint32_t bytes = static_cast<uint32_t>(we - w.wstart) * 4u;
  fence_proxy_async();
  mbar_expect_tx(&s.full[0], bytes);
  bulk_copy_g2s(s.stage[0], w.rowp + w.wstart, bytes, &s.full[0]);
  return true;
}

// The copy warp's loop (one lane): issues every chunk this CTA will consume,
// in consumption order, into the ring slot freed by the consumers. `first`:
// producer_first issued chunk 0 of the first row.
__device__ __noinline__ void producer_loop(const Params& p, Smem& s, int g, int m, bool first) {
  const bool spec = first;
  uint32_t q = spec ? 1u : 0u;
  RowWin w;
  bool stop = false;
  for (int64_t k = 0; !stop && get_row(p, s, k, g, m, w); ++k) {
    int j0 = 0;
    if (k == 0 && spec) {
      if (w.nch == 0) continue;  // the early chunk is discarded by the consumers
      j0 = 1;
    }
    for (int j = j0; j < w.nch; ++j, ++q) {
      const int slot = static_cast<int>(q % kStages);
      if (q >= kStages &&
          !mbar_wait_bounded(&s.empty[slot], ((q / kStages) - 1u) & 1u, p.timeout_ns, &s.abort)) {
        stop = true;
        break;
      }
      const int ws = w.wstart + j * kChunk;
      const int we = min(ws + kChunk, w.wend);
      const uint32_t bytes = static_cast<uint32_t>(we - ws) * 4u;
      fence_proxy_async();
      mbar_expect_tx(&s.full[slot], bytes);
      bulk_copy_g2s(s.stage[slot], w.rowp + ws, bytes, &s.full[slot]);
    }
  }
  // every issued copy must land before the CTA may exit
  const uint32_t oldest = q > kStages ? q - kStages : 0u;
  for (uint32_t i = oldest; i < q; ++i)
    mbar_wait_bounded(&s.full[i % kStages], (i / kStages) & 1u, p.timeout_ns, nullptr);
}

// A consumer's wait for a staged chunk ended without the chunk: flag a
// time-out unless the CTA was already giving up (then the cause is elsewhere).
__device__ __noinline__ void stage_gave_up(Smem& s, const Params& p) {
  if (!abort_set(&s.abort)) atomicOr(p.status, 0x4u);
  *reinterpret_cast<volatile int*>(&s.abort) = 1;
}

// ------------------------------------------------------------- chunk filter

// Bits of the elements of f (window elements i0 .. i0 + 3) at or above thr,
// elements outside [lo, hi) cleared unless the whole chunk is inside.
__device__ __forceinline__ uint32_t quad_bits(const float4 f, float thr, bool interior, int i0, int lo, int hi) {
  uint32_t b = (f.x >= thr ? 1u : 0u) | (f.y >= thr ? 2u : 0u) | (f.z >= thr ? 4u : 0u) | (f.w >= thr ? 8u : 0u);
  if (!interior) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (i0 + e < lo || i0 + e >= hi) b &= ~(1u << e);
  }
  return b;
}

template <bool kCount, bool kGlobal, int kT>
__device__ __forceinline__ bool append_survivors(Smem& s, uint32_t m, const float* src, int ws, int tid);

// Filters one chunk of a row window against the running threshold: one fp32
// compare per element; a warp reserves buffer space once; only survivors are
// converted to keys, stored and (with kCount) counted in the histogram.
// src holds the window's elements [ws, ws + 4*nvec) (shared or global memory);
// thread tid of kT takes float4 tid, tid + kT, ... Returns whether the warp
// appended (or tried to append) any.
template <bool kCount, bool kGlobal, int kT = kThreads>
__device__ __forceinline__ bool filter_chunk(Smem& s, const float* src, int ws, int nvec, int lo, int hi,
                                             int tid = threadIdx.x) {
  const float thr = s.thr_f;
  const float4* s4 = reinterpret_cast<const float4*>(src);
  const bool interior = ws >= lo && ws + 4 * nvec <= hi;
  uint32_t m = 0;
#pragma unroll
  for (int v = 0; v < kChunk / (4 * kT); ++v) {
    const int vi = tid + v * kT;
    if (vi < nvec)
      m |= quad_bits(kGlobal ? __ldg(s4 + vi) : s4[vi], thr, interior, ws + 4 * vi, lo, hi) << (4 * v);
  }
  return append_survivors<kCount, kGlobal, kT>(s, m, src, ws, tid);
}

// Appends the elements of a thread's share marked in m (bit 4v + e: element e
// of float4 tid + v * kT) to the buffer.
template <bool kCount, bool kGlobal, int kT>
__device__ __forceinline__ bool append_survivors(Smem& s, uint32_t m, const float* src, int ws, int tid) {
  constexpr int V = kChunk / (4 * kT);
  // bits of a lane's survivor count (at most 4 V)
  constexpr int kCB = (4 * V >= 32) ? 6 : (4 * V >= 16) ? 5 : (4 * V >= 8) ? 4 : (4 * V >= 4) ? 3 : 2;
  const int lane = static_cast<int>(lane_id());
  const int c = __popc(m);
  const uint32_t lt = lanemask_lt();
  uint32_t qb[kCB];
#pragma unroll
  for (int b = 0; b < kCB; ++b) qb[b] = __ballot_sync(0xFFFFFFFFu, (c >> b) & 1);
  int tot = 0;
#pragma unroll
  for (int b = 0; b < kCB; ++b) tot += __popc(qb[b]) << b;
  if (tot == 0) return false;
  int base = 0;
  if (lane == 0) base = atomicAdd(&s.buf_n, tot);
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  if (base + tot > kBufCap) {
    // no room: nothing of this reservation is stored and the row is marked
    // to be streamed again at its end (the warps of a row filter unsynchronised)
    if (lane == 0) *reinterpret_cast<volatile int*>(&s.full_row) = 1;
    return true;
  }
  int o = 0;
#pragma unroll
  for (int b = 0; b < kCB; ++b) o += __popc(qb[b] & lt) << b;
  constexpr int kStaged = (2 * kListCap) / kWarps;  // 16-bit slots per warp in s.emit
  if (tot <= kStaged) {
    // each lane only notes where its survivors are (a short divergent loop);
    // the whole warp then converts and stores them, 32 at a time. s.emit is
    // idle while a row streams, so it holds the per-warp lists.
    uint16_t* stg = reinterpret_cast<uint16_t*>(s.emit) + (threadIdx.x >> 5) * kStaged;
    while (m) {
      const int j = __ffs(m) - 1;
      m &= m - 1;
      stg[o++] = static_cast<uint16_t>(4 * (tid + (j >> 2) * kT) + (j & 3));
    }
    __syncwarp();
    for (int e = lane; e < tot; e += 32) {
      const int off = stg[e];
      const uint32_t k = fkey(kGlobal ? __ldg(src + off) : src[off]);
      const int oo = min(base + e, kBufCap - 1);
      s.bkey[oo] = k;
      s.bidx[oo] = ws + off;
      if (kCount) atomicAdd(&s.hist[k >> 20], 1u);
    }
    __syncwarp();
    return true;
  }
  o += base;
  while (m) {
    const int j = __ffs(m) - 1;
    m &= m - 1;
    const int off = 4 * (tid + (j >> 2) * kT) + (j & 3);
    const uint32_t k = fkey(kGlobal ? __ldg(src + off) : src[off]);
    const int oo = min(o, kBufCap - 1);
    s.bkey[oo] = k;
    s.bidx[oo] = ws + off;
    if (kCount) atomicAdd(&s.hist[k >> 20], 1u);
    ++o;
  }
  return true;
}

// filter_chunk for strided rows read straight from global memory: element e
// of the window is rowp[e * col_stride], loaded only inside [lo, hi).
__device__ __forceinline__ bool filter_chunk_strided(Smem& s, const float* rowp, int64_t cs, int ws, int nvec,
                                                     int lo, int hi) {
  constexpr int V = kChunk / (4 * kThreads);
  const int tid = threadIdx.x;
  const int lane = static_cast<int>(lane_id());
  const float thr = s.thr_f;
  uint32_t m = 0;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int vi = tid + v * kThreads;
    if (vi < nvec) {
      const int i0 = ws + 4 * vi;
      uint32_t b = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = i0 + e;
        if (i >= lo && i < hi && __ldg(rowp + static_cast<int64_t>(i) * cs) >= thr) b |= 1u << e;
      }
      m |= b << (4 * v);
    }
  }
  const uint32_t lt = lanemask_lt();
  const int c = __popc(m);
  const uint32_t q0 = __ballot_sync(0xFFFFFFFFu, c & 1);
  const uint32_t q1 = __ballot_sync(0xFFFFFFFFu, c & 2);
  const uint32_t q2 = __ballot_sync(0xFFFFFFFFu, c & 4);
  const uint32_t q3 = __ballot_sync(0xFFFFFFFFu, c & 8);
  const int tot = __popc(q0) + 2 * __popc(q1) + 4 * __popc(q2) + 8 * __popc(q3);
  if (tot == 0) return false;
  int base = 0;
  if (lane == 0) base = atomicAdd(&s.buf_n, tot);
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  int o = base + __popc(q0 & lt) + 2 * __popc(q1 & lt) + 4 * __popc(q2 & lt) + 8 * __popc(q3 & lt);
  while (m) {
    const int j = __ffs(m) - 1;
    m &= m - 1;
    const int idx = ws + 4 * (tid + (j >> 2) * kThreads) + (j & 3);
    const uint32_t k = fkey(__ldg(rowp + static_cast<int64_t>(idx) * cs));
    const int oo = min(o, kBufCap - 1);
    s.bkey[oo] = k;
    s.bidx[oo] = idx;
    atomicAdd(&s.hist[k >> 20], 1u);
    ++o;
  }
  return true;
}

// Histograms the keys of one staged chunk (elements inside [lo, hi)).
__device__ __forceinline__ void hist_chunk(Smem& s, const float* src, int ws, int nvec, int lo, int hi) {
  constexpr int V = kChunk / (4 * kThreads);
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int vi = threadIdx.x + v * kThreads;
    if (vi < nvec) {
      const float4 f = s4[vi];
      const int i0 = ws + 4 * vi;
      if (i0 >= lo && i0 < hi) atomicAdd(&s.hist[fkey(f.x) >> 20], 1u);
      if (i0 + 1 >= lo && i0 + 1 < hi) atomicAdd(&s.hist[fkey(f.y) >> 20], 1u);
      if (i0 + 2 >= lo && i0 + 2 < hi) atomicAdd(&s.hist[fkey(f.z) >> 20], 1u);
      if (i0 + 3 >= lo && i0 + 3 < hi) atomicAdd(&s.hist[fkey(f.w) >> 20], 1u);
    }
  }
}

// Streams the window [lo, hi) of row w straight from global memory with no
// seed: every element starts eligible and the threshold rises as candidates
// accumulate. Used when a seeded pass kept fewer than K elements, and for
// every row of strided logits (no bulk copies there).
// The threshold moves only after a chunk that added candidates, and once at
// the end.
__device__ __noinline__ void restream_row(Smem& s, const Params& p, const RowWin w) {
  csync();
  reset_row_state(s);
  csync();
  // Every chunk starts with room for a whole chunk (make_room keeps at most
  // TopK + what a compaction leaves, and TopK + a chunk fits the buffer).
  for (int j = 0; j < w.nch; ++j) {
    const int ws = w.wstart + j * kChunk;
    const int we = min(ws + kChunk, w.wend);
    const bool added = p.col_stride == 1
                           ? filter_chunk<true, true>(s, w.rowp + ws, ws, (we - ws) >> 2, w.lo, w.hi)
                           : filter_chunk_strided(s, w.rowp, p.col_stride, ws, (we - ws) >> 2, w.lo, w.hi);
    if (csync_or(added) || j + 1 == w.nch) {
      if (threadIdx.x < 32) advance_threshold(s, p.topk);
      // thread 0 reads the count while every other thread waits at the barrier
      if (csync_or(threadIdx.x == 0 && s.buf_n + kChunk > kBufCap) && j + 1 < w.nch) make_room(s, p.topk);
    }
  }
}

// ------------------------------------------------------------ row finishing

__device__ void write_trivial_row(const Params& p, int64_t r, int len) {
  int32_t* o = p.out + r * static_cast<int64_t>(p.topk);
  for (int j = threadIdx.x; j < p.topk; j += kThreads) o[j] = (j < len) ? j : -1;
}

// Clears what the row finish accumulates into (the sub-histogram, the list
// counters) and pads the ranking slots; thread u of `nthreads` takes its share.
__device__ __forceinline__ void prepare_finish(Smem& s, int u, int nthreads) {
  for (int b = u; b < 256; b += nthreads) s.sub[b] = 0;
  if (u < kSmallSet) {
    s.rk[u] = 0u;  // padding never beats a real candidate
    s.ri[u] = 0x7FFFFFFF;
  }
  if (u == 0) {
    s.n_emit = 0;
    s.n_list = 0;
    s.n_small = 0;
  }
}

// Highest bin with a buffered key, into s.x_hi (which starts at -1): thread
// u of `nthreads` scans its share of the histogram. Bins below the threshold
// may hold stale counts, but the highest occupied bin is the top key's bin.
__device__ __forceinline__ void note_highest_bin(Smem& s, int u, int nthreads) {
  int hi = -1;
  for (int b = u; b < kBins; b += nthreads)
    if (s.hist[b] != 0u) hi = b;
  hi = __reduce_max_sync(0xFFFFFFFFu, hi);
  if (lane_id() == 0 && hi >= 0) atomicMax(&s.x_hi, hi);
}

// After the last chunk: settle the threshold bin and re-stream the window if
// the seed kept fewer than K elements. While warp 0 moves the threshold, the
// other warps prepare the finish (and, in a cluster, note the highest occupied
// bin for the merge). Consumer-wide; ends with a barrier.
__device__ void close_window(Smem& s, const Params& p, const RowWin& w) {
  csync();
  const int tid = threadIdx.x;
  if (tid < 32) {
    advance_threshold(s, p.topk);
  } else {
    prepare_finish(s, tid - 32, kThreads - 32);
    if (p.cluster) note_highest_bin(s, tid - 32, kThreads - 32);
  }
  csync();
  if (s.full_row || (s.thr_lo != 0u && s.cnt_ge < p.topk)) {
    restream_row(s, p, w);  // may use the ranking slots; prepare again
    prepare_finish(s, tid, kThreads);
    if (p.cluster) note_highest_bin(s, tid, kThreads);
    csync();
  }
}

// One warp, over h[0, 256): the largest bin b whose suffix sum (bins >= b)
// reaches need (1 <= need <= total). Lane l sums bins 255-8l down to 248-8l;
// a scan over the lanes finds the lane holding the crossing, which walks its
// eight bins. Writes b to s.find_b and the count above b to s.find_gt.
__device__ __forceinline__ void warp_find_top256(Smem& s, const uint32_t* h, int need) {
  const int lane = static_cast<int>(lane_id());
  const uint4 lo4 = *reinterpret_cast<const uint4*>(h + 248 - 8 * lane);
  const uint4 hi4 = *reinterpret_cast<const uint4*>(h + 252 - 8 * lane);
  const uint32_t v[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};  // bins 255-8l, 254-8l, ...
  uint32_t own = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) own += v[k];
  uint32_t incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl >= static_cast<uint32_t>(need));
  const int L = hit ? __ffs(hit) - 1 : 31;
  if (lane == L) {
    uint32_t run = incl - own;
    int b = 255 - 8 * lane - 7;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (run + v[k] >= static_cast<uint32_t>(need)) {
        b = 255 - 8 * lane - k;
        break;
      }
      run += v[k];
    }
    s.find_b = b;
    s.find_gt = static_cast<int>(run);
  }
}

// G == 1: the CTA holds every candidate of the row. One pass over the buffer
// writes the sure winners (keys above the threshold bin t) to the output,
// lists the entries of bin t and histograms their key bits 19..12; one warp
// picks the sub-bin holding the K-th key, a pass over the short list writes
// the sub-bins above it and stages that sub-bin's few entries for ranking, and
// they are ranked directly. Output slots come from one shared atomic per warp.
// Starts right after close_window's barrier; five barriers in all.
__device__ void finish_local(Smem& s, const Params& p, int64_t r) {
  constexpr int kListIt = (kListCap + kThreads - 1) / kThreads;
  const int K = p.topk;
  const int tid = threadIdx.x;
  const int lane = static_cast<int>(lane_id());
  const uint32_t lt = lanemask_lt();
  int32_t* o = p.out + r * static_cast<int64_t>(K);
  const uint32_t t = static_cast<uint32_t>(s.t);
  const int inbin = static_cast<int>(s.hist[t]);
  const int need = K - (s.cnt_ge - inbin);
  const int n = s.buf_n;
  bool done = false;
  if (inbin <= kListCap) {
    // pass 1 over the buffer, in two short loops (counts, then writes) so the
    // code stays small: one reservation per warp for winners and for the list
    int tw = 0, tc = 0;
#pragma unroll 1
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t k = s.bkey[i];
      const uint32_t d = k >> 20;
      tw += (d > t) ? 1 : 0;
      if (d == t) {
        ++tc;
        atomicAdd(&s.sub[(k >> 12) & 0xFFu], 1u);
      }
    }
    tw = __reduce_add_sync(0xFFFFFFFFu, tw);
    tc = __reduce_add_sync(0xFFFFFFFFu, tc);
    int ow = 0, oc = 0;
    if (lane == 0) {
      if (tw) ow = atomicAdd(&s.n_emit, tw);
      if (tc) oc = atomicAdd(&s.n_list, tc);
    }
    ow = __shfl_sync(0xFFFFFFFFu, ow, 0);
    oc = __shfl_sync(0xFFFFFFFFu, oc, 0);
    const int jmax = (n + kThreads - 1) / kThreads;  // the same trips for the whole warp
#pragma unroll 1
    for (int j = 0; j < jmax; ++j) {
      const int i = tid + j * kThreads;
      const uint32_t d = (i < n) ? (s.bkey[i] >> 20) : 0u;
      const uint32_t bw = __ballot_sync(0xFFFFFFFFu, i < n && d > t);
      const uint32_t bc = __ballot_sync(0xFFFFFFFFu, i < n && d == t);
      if ((bw >> lane) & 1u) {
        const int q = ow + __popc(bw & lt);
        if (q < K) o[q] = s.bidx[i];
      }
      if ((bc >> lane) & 1u) s.emit[min(oc + __popc(bc & lt), kListCap - 1)] = i;
      ow += __popc(bw);
      oc += __popc(bc);
    }
    csync();
    const int nL = min(s.n_list, kListCap);
    if (need >= nL) {
      const int base = s.n_emit;
      for (int j = tid; j < nL; j += kThreads)
        if (base + j < K) o[base + j] = s.bidx[s.emit[j]];
      done = true;
    } else {
      if (tid < 32) warp_find_top256(s, s.sub, need);
      csync();
      const uint32_t b1 = static_cast<uint32_t>(s.find_b);
      const int need1 = need - s.find_gt;
      const int c1 = static_cast<int>(s.sub[b1]);
      if (c1 <= kSmallSet) {
        // list pass: sub-bins above b1 are winners; the entries of sub-bin b1
        // go straight into the ranking slots
        uint32_t lw[kListIt], lk[kListIt];
        int pw = 0, pk = 0;
        int pos[kListIt];
#pragma unroll
        for (int j = 0; j < kListIt; ++j) {
          const int e = tid + j * kThreads;
          pos[j] = (e < nL) ? s.emit[e] : 0;
          const uint32_t dg = (e < nL) ? ((s.bkey[pos[j]] >> 12) & 0xFFu) : 0u;
          lw[j] = __ballot_sync(0xFFFFFFFFu, e < nL && dg > b1);
          lk[j] = __ballot_sync(0xFFFFFFFFu, e < nL && dg == b1);
          pw += __popc(lw[j]);
          pk += __popc(lk[j]);
        }
        int qw = 0, qk = 0;
        if (lane == 0) {
          if (pw) qw = atomicAdd(&s.n_emit, pw);
          if (pk) qk = atomicAdd(&s.n_small, pk);
        }
        qw = __shfl_sync(0xFFFFFFFFu, qw, 0);
        qk = __shfl_sync(0xFFFFFFFFu, qk, 0);
#pragma unroll
        for (int j = 0; j < kListIt; ++j) {
          if ((lw[j] >> lane) & 1u) {
            const int q = qw + __popc(lw[j] & lt);
            if (q < K) o[q] = s.bidx[pos[j]];
          }
          if ((lk[j] >> lane) & 1u) {
            const int slot = min(qk + __popc(lk[j] & lt), kSmallSet - 1);
            s.rk[slot] = s.bkey[pos[j]];
            s.ri[slot] = s.bidx[pos[j]];
          }
          qw += __popc(lw[j]);
          qk += __popc(lk[j]);
        }
        csync();
        // rank the staged entries by (key desc, index asc); the need1 best are
        // selected. Slots past m hold padding that beats nothing.
        const int base = s.n_emit;
        const int m = min(s.n_small, kSmallSet);
        if (tid < m) {
          const uint32_t kj = s.rk[tid];
          const int32_t ij = s.ri[tid];
          int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
          for (int i0 = 0; i0 < m; i0 += 4) {
            const uint4 k4 = *reinterpret_cast<const uint4*>(&s.rk[i0]);
            const int4 x4 = *reinterpret_cast<const int4*>(&s.ri[i0]);
            r0 += (k4.x > kj || (k4.x == kj && x4.x < ij)) ? 1 : 0;
            r1 += (k4.y > kj || (k4.y == kj && x4.y < ij)) ? 1 : 0;
            r2 += (k4.z > kj || (k4.z == kj && x4.z < ij)) ? 1 : 0;
            r3 += (k4.w > kj || (k4.w == kj && x4.w < ij)) ? 1 : 0;
          }
          const int rank = r0 + r1 + r2 + r3;
          if (rank < need1 && base + rank < K) o[base + rank] = ij;
        }
        done = true;
      }
    }
  }
  if (!done) {
    // crowded threshold bin (heavy ties): radix select over the whole buffer;
    // rewrites the full output row
    uint32_t T;
    int I;
    select_threshold(s, K, T, I);
    emit_selected(s, T, I, o, K);
  }
  csync();
  reset_row_state(s);
  csync();
}

// Group barrier over the workspace: arrive (release), then wait (acquire)
// until `target` arrivals, at most timeout_ns. Returns false if this CTA must
// abandon the launch (time-out, or the test-only injected departure).
__device__ bool group_sync(Smem& s, uint32_t* ctr, uint32_t target, const Params& p, bool skip) {
  csync();
  if (threadIdx.x == 0) {
    if (skip) {
      *reinterpret_cast<volatile int*>(&s.abort) = 1;
    } else {
      __threadfence();
      atom_add_release_gpu(ctr, 1u);
      const uint64_t t0 = global_timer();
      uint32_t spins = 0;
      while (ld_acquire_gpu(ctr) < target) {
        if ((++spins & 63u) != 0) continue;
        if (abort_set(&s.abort)) break;  // a member of this cluster gave up
        if (global_timer() - t0 > p.timeout_ns) {
          *reinterpret_cast<volatile int*>(&s.abort) = 1;
          atomicOr(p.status, 0x2u);
          break;
        }
      }
      __threadfence();
    }
  }
  return !csync_or(abort_set(&s.abort));
}

__device__ __forceinline__ void clear_slice(uint32_t* a, int n, int m, int G) {
  for (int i = m * kThreads + static_cast<int>(threadIdx.x); i < n; i += G * kThreads) __stcg(a + i, 0u);
}

// G > 1: three radix passes whose histograms are merged across the group.
__device__ __noinline__ bool finish_group(Smem& s, const Params& p, int64_t r, int g, int m, uint32_t& epoch,
                             bool& first_barrier) {
  const int tid = threadIdx.x;
  const int K = p.topk;
  const int G = p.G;
  GroupWs* gw = p.groups + g;
  const bool skip = (p.inject == 1) && g == 0 && m == 1 && first_barrier;
  first_barrier = false;

  // pass A: bits 31..20 of every member's candidates still in play
  csync();
  for (int b = s.t + tid; b < kBins; b += kThreads) {
    const uint32_t h = s.hist[b];
    if (h) atomicAdd(&gw->h1[b], h);
  }
  epoch += G;
  if (!group_sync(s, &gw->bar_count, epoch, p, skip)) return false;
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = __ldcg(&gw->h1[b]);
  block_find(s, s.hist, kBins, K, true);
  const uint32_t T1 = static_cast<uint32_t>(s.find_b);
  const int needA = K - s.find_gt;
  const int gtA = block_count(s, [=](uint32_t k, int32_t) { return (k >> 20) > T1; });

  // pass B: bits 19..8 of the candidates in bin T1
  hist_keys(s, kBins, T1, 20, 8, 0xFFFu);
  for (int b = tid; b < kBins; b += kThreads) {
    const uint32_t h = s.hist[b];
    if (h) atomicAdd(&gw->h2[b], h);
  }
  epoch += G;
  if (!group_sync(s, &gw->bar_count, epoch, p, false)) return false;
  clear_slice(gw->h1, kBins, m, G);  // every member read h1 before arriving here
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = __ldcg(&gw->h2[b]);
  block_find(s, s.hist, kBins, needA, true);
  const uint32_t T2 = static_cast<uint32_t>(s.find_b);
  const int needB = needA - s.find_gt;
  const uint32_t P2 = (T1 << 12) | T2;
  const int gtB = block_count(s, [=](uint32_t k, int32_t) { return (k >> 20) == T1 && ((k >> 8) & 0xFFFu) > T2; });

  // pass C: bits 7..0, histogram kept per member so ties can be ranked by member
  hist_keys(s, 256, P2, 8, 0, 0xFFu);
  for (int b = tid; b < 256; b += kThreads) __stcg(&gw->h3[m][b], s.hist[b]);
  if (tid == 0) {
    __stcg(&gw->cnt[m][0], static_cast<uint32_t>(gtA));
    __stcg(&gw->cnt[m][1], static_cast<uint32_t>(gtB));
  }
  epoch += G;
  if (!group_sync(s, &gw->bar_count, epoch, p, false)) return false;
  clear_slice(gw->h2, kBins, m, G);  // every member read h2 before arriving here
  for (int b = tid; b < 256; b += kThreads) {
    uint32_t sum = 0;
    for (int mm = 0; mm < G; ++mm) sum += __ldcg(&gw->h3[mm][b]);
    s.hist[b] = sum;
  }
  block_find(s, s.hist, 256, needB, true);
  const uint32_t T3 = static_cast<uint32_t>(s.find_b) & 0xFFu;
  const int needC = needB - s.find_gt;
  const uint32_t T = (P2 << 8) | T3;
  if (tid < G) {
    const int mm = tid;
    uint32_t gtc = 0;
    for (int b = static_cast<int>(T3) + 1; b < 256; ++b) gtc += __ldcg(&gw->h3[mm][b]);
    s.g_e[mm] = static_cast<int>(__ldcg(&gw->h3[mm][T3]));
    s.g_tot[mm] = static_cast<int>(__ldcg(&gw->cnt[mm][0]) + __ldcg(&gw->cnt[mm][1]) + gtc);
  }
  csync();
  if (tid == 0) {
    // ties at the exact threshold key go to the smaller indices: members hold
    // consecutive index ranges, so the members before this one take theirs first
    int pre = 0, off = 0;
    for (int mm = 0; mm < G; ++mm) {
      const int take = max(0, min(needC - pre, s.g_e[mm]));
      if (mm == m) {
        s.off = off;
        s.take = take;
      }
      off += s.g_tot[mm] + take;
      pre += s.g_e[mm];
    }
  }
  csync();
  const int take = s.take;
  const int off = s.off;
  const int mine = s.g_e[m];
  int I = -1;
  if (take >= mine) {
    I = 0x7FFFFFFF;
  } else if (take > 0) {
    if (mine <= kSmallSet) {
      const int cnt = gather_small(s, [=](uint32_t k, int32_t) { return k == T; });
      rank_small(s, cnt, take);
      I = s.sel_I;
    } else {
      I = select_tied_indices(s, T, take);
    }
  }
  int32_t* o = p.out + r * static_cast<int64_t>(K);
  emit_selected(s, T, I, o + off, max(0, K - off));
  reset_row_state(s);
  csync();
  return true;
}

// ------------------------------------------------------------- cluster merge

// Barrier among the consumer warps of every CTA of the cluster, with a bounded
// wait: threads 0..G-1 of each CTA arrive on the merge barrier of CTA `tid`,
// then every consumer thread waits until its own CTA's barrier has collected
// G arrivals. Two barriers alternate, so a CTA that has passed one sync cannot
// land its next arrival on a phase another CTA is still waiting for. The copy
// warp takes no part (a hardware cluster barrier would wait for it). Returns
// false, with TOPK_DEV_BARRIER_TIMEOUT set, if the wait ran out. Consumer-wide.
__device__ bool cluster_sync(Smem& s, const Params& p, uint32_t& xph, int g, int m) {
  csync();  // this CTA's writes, local and remote, come before its arrivals
  const int b = static_cast<int>(xph & 1u);
  const uint32_t parity = (xph >> 1) & 1u;
  // test only: CTA 1 of cluster 0 withholds its arrivals at the launch's first merge sync
  const bool skip = p.inject == 2 && g == 0 && m == 1 && xph == 0;
  ++xph;
  if (!skip && threadIdx.x < static_cast<unsigned>(p.G)) mbar_arrive_remote(dsmem_addr(&s.xbar[b], threadIdx.x));
  bool ok = mbar_try_wait_cluster(&s.xbar[b], parity);
  if (!ok) {
    const uint64_t t0 = global_timer();
    bool gave_up = false;
    while (!ok) {
#pragma unroll 1
      for (int i = 0; i < 32 && !ok; ++i) ok = mbar_try_wait_cluster(&s.xbar[b], parity);
      if (ok || abort_set(&s.abort)) break;  // a member gave up: it will not arrive
      if (global_timer() - t0 > p.timeout_ns) {
        gave_up = true;
        break;
      }
    }
    if (gave_up) {
      atomicOr(p.status, 0x2u);
      *reinterpret_cast<volatile int*>(&s.abort) = 1;
    }
  }
  return !csync_or(abort_set(&s.abort));
}

// Count of bin b over the members of the cluster: this CTA's own count plus
// the other members' (read from their shared memory).
__device__ __forceinline__ uint32_t merged_count(Smem& s, int b, int m, int G) {
  uint32_t c = s.hist[b];
  for (int r = 0; r < G; ++r)
    if (r != m) c += dsmem_ld(dsmem_addr(&s.hist[b], static_cast<uint32_t>(r)));
  return c;
}

// block_find from the top over the members' merged counts of bins in
// [tmax, top], top the highest occupied bin of any member (those counts are
// exact; bins below tmax are never reached because the suffix at tmax already
// holds need). Writes the bin to s.find_b, the count above it to s.find_gt and
// its own count to s.x_in. Consumer-wide; ends with a barrier.
__device__ void cluster_find(Smem& s, int tmax, int top, int need, int m, int G) {
  const int lane = static_cast<int>(lane_id());
  const int warp = threadIdx.x >> 5;
  const int nblk = (top - tmax + 32) >> 5;
  for (int q = warp; q < nblk; q += kWarps) {
    const int b = top - (32 * q + lane);
    const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, (b >= tmax) ? merged_count(s, b, m, G) : 0u);
    if (lane == 0) s.bsum[q] = sum;
  }
  csync();
  if (warp == 0) {
    uint32_t b4[4];
    uint32_t own = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int q = 4 * lane + k;
      b4[k] = (q < nblk) ? s.bsum[q] : 0u;
      own += b4[k];
    }
    uint32_t incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl >= static_cast<uint32_t>(need));
    const int L = hit ? __ffs(hit) - 1 : 31;
    uint32_t run = incl - own;
    int qsel = 0;
    if (lane == L) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (run + b4[k] >= static_cast<uint32_t>(need)) {
          qsel = 4 * lane + k;
          break;
        }
        run += b4[k];
      }
    }
    qsel = __shfl_sync(0xFFFFFFFFu, qsel, L);
    run = __shfl_sync(0xFFFFFFFFu, run, L);
    const int bin = top - (32 * qsel + lane);
    const uint32_t h = (bin >= tmax) ? merged_count(s, bin, m, G) : 0u;
    uint32_t in2 = h;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, in2, o);
      if (lane >= o) in2 += v;
    }
    const uint32_t hit2 = __ballot_sync(0xFFFFFFFFu, run + in2 >= static_cast<uint32_t>(need));
    const int L2 = hit2 ? __ffs(hit2) - 1 : 0;
    if (lane == L2) {
      s.find_b = bin;
      s.find_gt = static_cast<int>(run + in2 - h);
      s.x_in = static_cast<int>(h);
    }
  }
  csync();
}

// This member's buffered entries in bins >= ts, appended to the leader's
// buffer from position n0 on (one remote reservation per warp).
__device__ void push_to_leader(Smem& s, uint32_t ts, int n0) {
  const int tid = threadIdx.x;
  const int lane = static_cast<int>(lane_id());
  const int n = s.buf_n;
  int c = 0;
#pragma unroll 1
  for (int i = tid; i < n; i += kThreads) c += ((s.bkey[i] >> 20) >= ts) ? 1 : 0;
  c = __reduce_add_sync(0xFFFFFFFFu, c);
  int base = 0;
  if (lane == 0 && c) base = static_cast<int>(dsmem_atom_add(dsmem_addr(&s.x_push, 0u), static_cast<uint32_t>(c)));
  base = n0 + __shfl_sync(0xFFFFFFFFu, base, 0);
  const uint32_t kaddr = dsmem_addr(&s.bkey[0], 0u);
  const uint32_t iaddr = dsmem_addr(&s.bidx[0], 0u);
  const uint32_t lt = lanemask_lt();
  const int jmax = (n + kThreads - 1) / kThreads;
#pragma unroll 1
  for (int j = 0; j < jmax; ++j) {
    const int i = tid + j * kThreads;
    const uint32_t k = (i < n) ? s.bkey[i] : 0u;
    const bool sel = i < n && (k >> 20) >= ts;
    const uint32_t bm = __ballot_sync(0xFFFFFFFFu, sel);
    const int q = base + __popc(bm & lt);
    if (sel && q < kBufCap) {
      dsmem_st(kaddr + 4u * static_cast<uint32_t>(q), k);
      dsmem_st(iaddr + 4u * static_cast<uint32_t>(q), static_cast<uint32_t>(s.bidx[i]));
    }
    base += __popc(bm);
  }
}

// Merge of one split row inside a cluster, after every member closed its
// window. Every member's buffer holds at least the best K of its own part, so
// the union holds the row's best K, and each member with threshold bin t_m > 0
// keeps at least K keys in bins >= t_m: the K-th key of the row lies in a bin
// >= t_max, the largest t_m. From X1 to X3 no member changes its counts,
// threshold or buffer size, so every member reads the others' counts of bins
// >= t_max and finds the same bin t* of the K-th key; the members then append
// their entries of bins >= t* to the leader's (rank 0) buffer, and the leader
// finishes the row like a whole-row CTA, its own entries below t* ignored.
// If the leader's buffer cannot take them as it is, it first keeps only its
// bins >= t* (one more sync); if even the union does not fit, every member
// goes to the workspace merge. Returns 1 on the leader, 0 on the members, 2
// for the workspace merge (everywhere), -1 on a time-out.
__device__ __noinline__ int cluster_merge(Smem& s, const Params& p, int g, int m, uint32_t& xph) {
  const int tid = threadIdx.x;
  const int G = p.G;
  if (tid == 0) s.x_n0 = s.buf_n;  // what the others read as this CTA's size until X3
  if (!cluster_sync(s, p, xph, g, m)) return -1;  // X1: every window is closed
  if (tid < 32) {
    uint32_t tm = 0;
    int hi = -1;
    if (tid < G) {
      tm = (tid == m) ? static_cast<uint32_t>(s.t) : dsmem_ld(dsmem_addr(&s.t, static_cast<uint32_t>(tid)));
      hi = (tid == m) ? s.x_hi : static_cast<int>(dsmem_ld(dsmem_addr(&s.x_hi, static_cast<uint32_t>(tid))));
    }
    tm = __reduce_max_sync(0xFFFFFFFFu, tm);
    hi = __reduce_max_sync(0xFFFFFFFFu, hi);
    if (tid == 0) {
      s.x_top = max(hi, static_cast<int>(tm));
      s.x_t = static_cast<int>(tm);
      s.x_ln = (m == 0) ? s.x_n0 : static_cast<int>(dsmem_ld(dsmem_addr(&s.x_n0, 0u)));
    }
  }
  csync();
  cluster_find(s, s.x_t, s.x_top, p.topk, m, G);
  const int ts = s.find_b;
  const int inbin = s.x_in;
  const int tot = s.find_gt + inbin;
  int n0 = s.x_ln;
  if (n0 + tot > kBufCap) {
    if (tot > kBufCap) return 2;  // heavy ties at t*: same decision in every member
    if (m == 0) compact_buffer(s, [=](uint32_t k, int32_t) { return (k >> 20) >= static_cast<uint32_t>(ts); });
    if (!cluster_sync(s, p, xph, g, m)) return -1;  // X2: the leader kept only its bins >= t*
    if (tid == 0) s.x_ln = (m == 0) ? s.buf_n : static_cast<int>(dsmem_ld(dsmem_addr(&s.buf_n, 0u)));
    csync();
    n0 = s.x_ln;
  }
  if (m != 0) push_to_leader(s, static_cast<uint32_t>(ts), n0);
  if (!cluster_sync(s, p, xph, g, m)) return -1;  // X3: the union is in the leader's buffer
  if (m != 0) return 0;
  if (tid == 0) {
    s.t = ts;
    s.cnt_ge = tot;
    s.hist[ts] = static_cast<uint32_t>(inbin);
    int n = n0 + s.x_push;
    if (n > kBufCap) {  // cannot happen when the counts agree; never read past the buffer
      atomicOr(p.status, 0x4u);
      n = kBufCap;
    }
    s.buf_n = n;
    s.x_push = 0;
  }
  csync();
  return 1;
}

// ------------------------------------------------------------------- kernel

__global__ void __launch_bounds__(kCtaThreads, kMinBlocks) topk_ragged_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  const int g = static_cast<int>(blockIdx.x) / p.G;
  const int m = static_cast<int>(blockIdx.x) % p.G;

  int32_t len0 = 0;     // copy thread, split rows: the first row's length
  bool first = false;   // copy thread: chunk 0 of the first row is issued
  if (tid == kThreads) {
    // the copy thread sets up the ring and, with whole rows per CTA, issues
    // the first copy right away; everyone else meets it at the barrier below
    if (p.G > 1 && g < p.num_rows) len0 = __ldg(p.lengths + g);
    s.abort = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1u);
      mbar_init(&s.empty[i], kGroupWarps);
    }
    if (p.cluster) {
      mbar_init(&s.xbar[0], static_cast<uint32_t>(p.G));
      mbar_init(&s.xbar[1], static_cast<uint32_t>(p.G));
    }
    fence_mbar_init();
    if (p.G == 1 && p.col_stride == 1) {
      producer_first_whole(p, s, g);
      first = true;
    }
  }
  uint32_t status0 = 0;  // split rows: the status word as this launch found it
  if (tid < kThreads) {
    if (p.G > 1 && tid == 0) status0 = *reinterpret_cast<const volatile uint32_t*>(p.status);
    reset_row_state(s);
    for (int k = tid; k < kLenCache; k += kThreads) {
      const int64_t r = g + static_cast<int64_t>(k) * p.num_groups;
      s.lens[k] = (r < p.num_rows) ? clamp_len(p, p.lengths[r]) : 0;
    }
  }
  // the other CTAs of the cluster may reach into this one's shared memory only
  // after every thread has arrived here (their wait comes before their first
  // merge); the copies fill this CTA's own shared memory and need no wait.
  // The barrier is .aligned: the copy warp, whose lane 0 alone ran the set-up
  // above, reconverges first.
  __syncwarp();
  if (p.cluster) cluster_arrive_all();
  __syncthreads();
  if (tid >= kThreads) {
    if (tid == kThreads && p.col_stride == 1) {  // strided rows are read by the consumers
      if (p.G > 1) first = producer_first_split(p, s, g, m, len0);
      producer_loop(p, s, g, m, first);
    }
    if (p.cluster) {
      // the copy warp also meets the rest of the cluster before leaving: it
      // waits out the start-up phase, then arrives at the exit phase
      __syncwarp();
      cluster_wait_all();
      cluster_arrive_all();
      cluster_wait_all();
    }
    return;
  }

  const int K = p.topk;
  const int grp = (tid >> 5) / kGroupWarps;  // this warp's group: it filters the slots s with s % kGroups == grp
  const int gtid = tid - grp * kGroupThreads;
  uint32_t q = 0;  // chunks consumed
  uint32_t epoch = 0;
  uint32_t xph = 0;       // cluster merge syncs passed
  bool cluster_ready = false;  // this thread passed the start-up cluster barrier
  bool used_ws = false;   // some row of a split group went through the workspace merge
  bool first_barrier = true;
  bool aborted = false;
  if (p.G > 1 && csync_or(tid == 0 && (status0 & (0x2u | 0x4u)) != 0)) {
    // An earlier launch on this workspace timed out and left its group words
    // as they were; merging through them could give wrong rows. Write rows of
    // -1 instead, flag the refusal, and let topk_workspace_init restore service.
    if (tid == 0) {
      atomicOr(p.status, 0x8u);
      *reinterpret_cast<volatile int*>(&s.abort) = 1;  // the copy warp stops issuing
    }
    if (m == 0)
      for (int64_t r = g; r < p.num_rows; r += p.num_groups) write_trivial_row(p, r, 0);
    aborted = true;
  }
  RowWin w;
  for (int64_t k = 0; !aborted && get_row(p, s, k, g, m, w); ++k) {
    if (w.len <= K) {
      if (m == 0) write_trivial_row(p, w.r, w.len);
      if (p.G == 1 && k == 0 && p.col_stride == 1) {
        // slot 0's group discards the early copy the copy warp issued for this row
        if (grp == 0) {
          if (!mbar_wait_bounded(&s.full[0], 0u, p.timeout_ns, &s.abort) && lane_id() == 0) stage_gave_up(s, p);
          __syncwarp();
          if (lane_id() == 0) mbar_arrive(&s.empty[0]);
        }
        q = 1;
      }
      continue;
    }
    const int span = w.hi - w.lo;
    if (p.col_stride != 1) restream_row(s, p, w);  // strided rows: no staging ring
    // The warps walk the chunks on their own, each group the chunks of its
    // ring slot. The only CTA-wide barriers of a row are the seed's (first
    // chunk, read by every warp) and the row end's, and every warp reaches all
    // of them whatever its waits returned. A warp waits on another group's
    // slot only for a seed chunk, after the barrier that ended the previous
    // row, when that slot's earlier phases have all completed. A reservation
    // that would pass the end of the buffer stores nothing and marks the row
    // full; the warps then skip its remaining chunks and the row is streamed
    // again, exactly, at its end (the seed aims at 1.25 K survivors and the
    // buffer holds at least 2 K, so mostly rows of heavy ties get there).
    bool release_late = false;
    if (p.col_stride == 1 && w.nch > 0) {
      const uint32_t q0 = q;  // ring position of the window's chunk 0
      int j = 0;
      if (span > K) {
        // seed: every warp histograms the first chunk, and the threshold aims at
        // ~1.25 K survivors over the window (exactly K when it is this one chunk)
        const int slot = static_cast<int>(q0 % kStages);
        const bool mine = slot % kGroups == grp;
        bool ok = mbar_wait_bounded(&s.full[slot], (q0 / kStages) & 1u, p.timeout_ns, &s.abort);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok && lane_id() == 0) stage_gave_up(s, p);
        const int ws = w.wstart;
        const int we = min(ws + kChunk, w.wend);
        const int nvec = (we - ws) >> 2;
        hist_chunk(s, s.stage[slot], ws, nvec, w.lo, w.hi);
        const int in_chunk = min(w.hi, we) - max(w.lo, ws);
        int target = K;
        if (w.nch > 1) {
          const int64_t tt = (5ll * K * in_chunk + 4ll * span - 1) / (4ll * span);
          target = static_cast<int>(tt < 1 ? 1 : tt);
        }
        target = min(target, in_chunk);
        block_find(s, s.hist, kBins, target, true);
        if (tid == 0) {
          // the histogram now counts every element of this chunk; the ones at or
          // above bin t are exactly those the filter below appends, which the
          // next threshold update counts through buf_n - buf_mark
          s.t = s.find_b;
          s.cnt_ge = 0;
          s.buf_mark = 0;
          set_threshold(s, static_cast<uint32_t>(s.find_b) << 20);
        }
        // Crowded seed bin (heavy ties, e.g. a constant row): the chunk holds
        // at least K elements at or above it and the projection overflows the
        // buffer. Then the chunk's own K best (by value, then index) are
        // kept and the filter rises to their K-th key + 1: every later element
        // of this window has a larger index than all of them, so one equal to
        // that key can never be selected (exact for any data).
        const int at_or_above = s.find_gt + static_cast<int>(s.hist[s.find_b]);
        const bool crowded = w.nch > 1 && at_or_above >= K &&
                             static_cast<int64_t>(at_or_above) * span > static_cast<int64_t>(kBufCap) * in_chunk;
        csync();
        if (crowded) {
          const bool staged = !csync_or(!ok);  // the same answer in every warp
          if (staged) {
            filter_chunk<false, false>(s, s.stage[slot], ws, nvec, w.lo, w.hi);
            csync();
          }
          if (mine) {
            __syncwarp();
            if (lane_id() == 0) mbar_arrive(&s.empty[slot]);
          }
          if (staged) {
            if (tid < 32) advance_threshold(s, K);
            csync();
            compact_exact(s, K);
          }
        } else if (w.nch == 1) {
          // a one-chunk window: every warp filters it and the slot is released
          // after the row-end barrier
          if (ok) filter_chunk<false, false>(s, s.stage[slot], ws, nvec, w.lo, w.hi);
          release_late = mine;
        } else if (mine) {
          if (ok) filter_chunk<false, false, kGroupThreads>(s, s.stage[slot], ws, nvec, w.lo, w.hi, gtid);
          __syncwarp();
          if (lane_id() == 0) mbar_arrive(&s.empty[slot]);
        }
        j = 1;
      }
      // then the group's own chunks: ring positions q0 + j stepping by kGroups
      // (slot % kGroups == grp; kGroups divides kStages)
      if (kGroups > 1)
        j += static_cast<int>((static_cast<uint32_t>(grp) + kGroups - (q0 + j) % kGroups) % kGroups);
      int slot = static_cast<int>((q0 + j) % kStages);
      uint32_t par = ((q0 + j) / kStages) & 1u;
      for (; j < w.nch; j += kGroups) {
        bool ok = mbar_wait_bounded(&s.full[slot], par, p.timeout_ns, &s.abort);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok && lane_id() == 0) stage_gave_up(s, p);
        // warp-uniform: the filter's ballots need every lane
        if (ok && !__any_sync(0xFFFFFFFFu, *reinterpret_cast<volatile int*>(&s.full_row) != 0)) {
          const int ws = w.wstart + j * kChunk;
          const int we = min(ws + kChunk, w.wend);
          filter_chunk<true, false, kGroupThreads>(s, s.stage[slot], ws, (we - ws) >> 2, w.lo, w.hi, gtid);
        }
        __syncwarp();
        if (lane_id() == 0) mbar_arrive(&s.empty[slot]);
        slot += kGroups;  // the next own chunk; past the last slot it is the next lap
        if (slot >= kStages) {
          slot -= kStages;
          par ^= 1u;
        }
      }
      q = q0 + static_cast<uint32_t>(w.nch);
    }
    const bool abort_row = csync_or(abort_set(&s.abort));  // the same answer in every warp
    if (release_late) {
      if (lane_id() == 0) mbar_arrive(&s.empty[static_cast<int>((q - 1) % kStages)]);
      release_late = false;
    }
    if (abort_row) {
      aborted = true;
      break;
    }
    if (aborted) break;
    close_window(s, p, w);
    if (p.G == 1) {
      finish_local(s, p, w.r);
    } else if (p.cluster) {
      if (!cluster_ready) {
        cluster_wait_all();
        cluster_ready = true;
      }
      const int mode = cluster_merge(s, p, g, m, xph);
      if (mode == 1) {
        finish_local(s, p, w.r);
      } else if (mode == 0) {
        reset_row_state(s);
        csync();
      } else if (mode == 2) {
        used_ws = true;
        if (!finish_group(s, p, w.r, g, m, epoch, first_barrier)) aborted = true;
      } else {
        aborted = true;
      }
    } else if (!finish_group(s, p, w.r, g, m, epoch, first_barrier)) {
      aborted = true;
    }
  }

  if (aborted) *reinterpret_cast<volatile int*>(&s.abort) = 1;  // the copy warp stops issuing
  if (p.cluster) {
    // No CTA leaves while another may still reach into its shared memory:
    // every thread of the cluster, the copy warps included, meets at the exit
    // phase of the hardware cluster barrier. Every wait before it is bounded,
    // so every thread gets there. A CTA that gave up first tells the others,
    // whose bounded waits then end at once instead of at their own limits.
    if (!cluster_ready) cluster_wait_all();
    if (aborted && tid < p.G) dsmem_st(dsmem_addr(&s.abort, static_cast<uint32_t>(tid)), 1u);
    __syncwarp();
    cluster_arrive_all();
    cluster_wait_all();
  }
  if (aborted) return;
  if (p.G > 1 && (!p.cluster || used_ws)) {
    // last CTA of the group to finish clears the per-member words and counters
    GroupWs* gw = p.groups + g;
    csync();
    if (tid == 0) {
      __threadfence();
      const uint32_t old = atom_add_acq_rel_gpu(&gw->exit_count, 1u);
      s.last = (old == static_cast<uint32_t>(p.G - 1)) ? 1 : 0;
    }
    csync();
    if (s.last) {
      uint32_t* h3 = &gw->h3[0][0];
      for (int i = tid; i < kMaxGroup * 256; i += kThreads) __stcg(h3 + i, 0u);
      uint32_t* c = &gw->cnt[0][0];
      for (int i = tid; i < kMaxGroup * 4; i += kThreads) __stcg(c + i, 0u);
      csync();
      if (tid == 0) {
        __threadfence();
        __stcg(&gw->bar_count, 0u);
        __stcg(&gw->exit_count, 0u);
      }
    }
  }
}

// ---------------------------------------------------------------- host side

int kernel_threads() { return kCtaThreads; }

size_t kernel_smem_bytes() { return sizeof(Smem); }

cudaError_t kernel_configure() {
  return cudaFuncSetAttribute(topk_ragged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(Smem)));
}

cudaError_t kernel_occupancy(int* ctas_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, topk_ragged_kernel, kCtaThreads,
                                                       sizeof(Smem));
}

cudaError_t kernel_max_clusters(int cluster_size, int* clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster_size));
  cfg.blockDim = dim3(kCtaThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, topk_ragged_kernel, &cfg);
}

cudaError_t launch_topk(const Params& p, int grid, bool cooperative, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kCtaThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (p.cluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.G);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  } else if (cooperative) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, topk_ragged_kernel, p);
}

}  // namespace LTK_SHAPE_NS
}  // namespace ltk
