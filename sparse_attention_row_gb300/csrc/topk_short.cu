// The short-row kernel: one CTA of 32 warps per SM owns whole rows (any
// length), held in or streamed through a shared-memory ring; in its cluster
// form (topk_short_cluster_kernel, further down) the CTAs of a thread-block
// cluster share one row.
//
// This is the single-CTA path of the method: a shared-memory histogram seeds a
// threshold, a filter keeps the elements at or above it as candidates with
// warp-level compaction, and a radix select on the candidates finishes the row
// (the "decode / medium" path that rows below the cooperative radix threshold
// take in the persistent_topk launcher of the vLLM PR #41189 page,
// "Implementation breakdown"; the single-CTA FilteredTopK there keeps rows in
// at least 128 KB of shared memory, vLLM PR #54110 page, "Feature and
// motivation"). Here one CTA also streams rows longer than its ring, and a
// launch with too few long rows for the GPU splits each over a cluster.
//
// Per row:
//   - lanes of warp 0 issue the row's window as 8 KB bulk copies
//     (cp.async.bulk), one mbarrier per ring slot; a row of up to 16 pieces
//     stays resident, a longer one streams (each piece's slot goes to piece
//     j + 16, and the last pieces' slots to the next row's first pieces);
//   - piece 0 is histogrammed on the top 12 key bits and one warp picks the
//     seed bin for about three standard deviations more than the row's K best
//     that the sample should hold (split on 8 more bits when it is wide);
//   - every warp filters tasks of up to 8 float4 per lane as their pieces land,
//     one fp32 compare per element; survivors go to the warp's own candidate
//     region and its own fine-bin counters, (key - threshold) >> 17: no
//     contended atomics;
//   - one warp finds the K-th key's fine bin t from the folded counters; the
//     warps write the winners above t through shared output counters, and t's
//     entries are ranked by (key desc, index asc), split first on 8 more key
//     bits when there are many.
// Anything outside that shape (fewer than K survivors, a full region, the K-th
// key in a crowded bin) falls back to an exact radix select over the row (from
// the ring when resident, from global memory when streamed), whose ties are
// taken in index order by a block-wide scan. A K-th key above the counted bins
// only recounts the candidates with wider bins.
//
// Strided logits (a column stride above 1) are loaded into the ring by every
// thread with plain loads (rows up to the ring's size) or selected by the exact
// path straight from global memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include "topk_internal.h"

// Two instances are built from this source: ltk::shortrow, 32 warps (the
// default below), and ltk::short16, 16 warps with twice the candidate slots
// per warp (topk_short16.cu), whose block-wide phases cost half the
// instructions: faster on short rows and split rows, slower where the filter
// sets the pace.
#ifndef LTK_SHORT_NS
#define LTK_SHORT_NS shortrow
#define LTK_SHORT_THREADS kShortCtaThreads
#define LTK_SHORT_REGION 256
#endif

namespace ltk {
namespace LTK_SHORT_NS {

constexpr int kThreads = LTK_SHORT_THREADS;
constexpr int kWarps = kThreads / 32;
constexpr int kPiece = 2048;                        // elements per bulk copy (8 KB), one mbarrier each
constexpr int kRing = 16;                           // ring slots of one piece (128 KB): a row of up to 16
                                                    // pieces is resident; longer rows stream through it
constexpr int kTask = 512;                          // window elements a warp filters at a time (4 float4 per lane)
constexpr int kSeed = kPiece;                       // window elements histogrammed for the seed (piece 0)
constexpr int kRegion = LTK_SHORT_REGION;           // candidate slots per warp
constexpr int kCand = kWarps * kRegion;
constexpr int kFine = 17;                           // fine bins: (key - threshold) >> 17, or coarser
constexpr int kTrack = 64;                          // fine bins counted during the filter, from the seed bin's edge
constexpr int kRank = 512;                          // entries of the K-th key's fine bin at most (fast path)
static_assert(kRank <= kThreads, "one thread per ranked entry at least");
constexpr int kRankDirect = 192;                    // up to this many are ranked at once; more are first
                                                    // split on 8 more key bits
constexpr int kBlind = 4;                           // pieces of a CTA's first window issued before its
                                                    // length is known (the rest follow once it is)
constexpr int kTaskSurvivors = 128;                 // expected survivors a filter task may take
constexpr int kMinTasks = 8;                        // filter tasks a window is split into at least
constexpr int kRefineExcess = 256;                  // a resident row refines its seed bin only when that
                                                    // keeps more than this many extra survivors out
constexpr int kClusterRefineExcess = 2048;          // ... a split row only when it keeps more than this
                                                    // many out of each CTA (a refined, tighter threshold
                                                    // falls short of K survivors more often, and the
                                                    // exact path then reads the row from global memory)
static_assert(kRing <= 32, "slot phases fit one 32-bit mask");
constexpr int kRingF4 = kRing * kPiece / 4;        // float4s in the ring
static_assert(kWarps <= 32, "one lane of warp 0 per warp when counts are gathered");
static_assert(kPiece % (2 * kTask) == 0 && kTask == 4 * 4 * 32, "tasks of up to 8 float4 per lane tile a piece");

struct __align__(128) Smem {
  float row[kRing * kPiece];      // the ring: slot q holds pieces q, q + kRing, ... of the window
  uint32_t ckey[kCand];           // candidate keys, warp w in [w * kRegion, (w + 1) * kRegion)
  int32_t cidx[kCand];            // candidate indices (first the survivors' task positions)
  uint32_t hseed[kBins];          // seed histogram; scratch of the fallback
  uint32_t bsum[kBins / 32];      // 32-bin block sums (find_top, in the fallback)
  alignas(16) uint32_t hsub[256]; // the seed bin's 8-bit sub-histogram (key bits 19..12)
  alignas(16) uint32_t rk[kRank];  // bin t's entries, ranked
  alignas(16) int32_t ri[kRank];
  alignas(16) int wbin[kWarps][kTrack + 4];  // per warp: candidates in fine bin j, (key - thr) >> shift (thr: the
                                             // edge); rows padded by 16 bytes so a lane per row reads no bank twice
  alignas(16) int ftot[kTrack];   // fine-bin counts summed over the warps
  int n_win, n_bt;                // winners above bin t written, bin t's entries held (emission)
  int wcnt[kWarps];               // survivors per warp (may exceed kRegion: overflow)
  int tcnt[2][kWarps];            // tie counts per warp (block scans; two buffers, one barrier each)
  unsigned long long bar[kRing];
  int pdone[kRing];               // warps done with the piece in a slot (streaming rows)
  int slot_issues[kRing];         // copies issued into each slot since the launch began
  int abort;
  int len_next;
  int fb, fgt;                    // find_top result (fallback)
  int n_out;
  uint32_t key_max;
  int t0, t, need, in_t, sel_ok;  // seed bin, the K-th key's fine bin, its entries taken and held, fast path ok
  int target;                     // the sample's best that the seed threshold keeps
  int sub_b, sub_above;           // a large K-th fine bin: the sub-bin holding the K-th, the count above it
  int wide;                       // the K-th key lies above the counted fine bins: count again, coarser
  uint32_t cmax;                  // the largest candidate key of the row
  int crowded;                    // the seed bin of a streamed row is crowded (heavy ties)
  int refine, need_in;            // the seed bin is wide: refine the threshold inside it, to `need_in` of its entries
  uint32_t thr_key;               // the filter keeps keys >= thr_key
};

// ---------------------------------------------------------------- primitives

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(unsigned long long* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, unsigned long long* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
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

// Waits for a piece, at most timeout_ns; false if it gave up (or, with an
// abort flag given, once the CTA is giving up).
__device__ __noinline__ bool wait_piece(unsigned long long* bar, uint32_t parity, uint64_t timeout_ns,
                                        const int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *reinterpret_cast<const volatile int*>(abort)) return false;
    if (global_timer() - t0 > timeout_ns) return false;
  }
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the kernel before it on the stream is still
// running. Every thread waits here, before its first access to global memory,
// until that kernel has completed and its writes are visible (at once when
// there is none, or when the launch did not allow the early start). The signal
// that follows lets the next kernel on the stream start early in the same way:
// that kernel waits for this one's completion before it reads its output.
__device__ __forceinline__ void wait_previous_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Block barrier that ORs a predicate: every thread gets the same answer.
__device__ __forceinline__ bool sync_or(bool pred) { return __syncthreads_or(pred ? 1 : 0) != 0; }

__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t u = __float_as_uint(x);
  u = (u == 0x80000000u) ? 0u : u;
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

// fp32 value whose ">=" test is equivalent to "key >= k" for every non-NaN input.
__device__ __forceinline__ float key_floor_value(uint32_t k) {
  if (k <= 0x007FFFFFu) return -__int_as_float(0x7F800000);
  if (k > 0xFF800000u) return __int_as_float(0x7FC00000);
  const uint32_t u = (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ float pick(const float4 f, int j) {
  return j == 0 ? f.x : j == 1 ? f.y : j == 2 ? f.z : f.w;
}

// Appends val at out[*counter ...] for every lane with pred: one shared atomic
// per warp (the fallback's emission; the fast path reserves nothing).
__device__ __forceinline__ void warp_emit(int32_t* out, int* counter, int cap, bool pred, int32_t val) {
  const uint32_t m = __ballot_sync(0xFFFFFFFFu, pred);
  if (m == 0) return;
  int base = 0;
  if (lane_id() == 0) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  const int o = base + __popc(m & lanemask_lt());
  if (pred && o < cap) out[o] = val;
}

// Over h[0, kBins): the largest bin b whose suffix sum (bins >= b) reaches
// need, into s.fb, and the count above b into s.fgt. Requires 1 <= need <=
// total. Every warp sums whole 32-bin blocks; warp 0 scans the block sums and
// then the block holding the crossing. Two barriers.
__device__ __noinline__ void find_top(Smem& s, const uint32_t* h, int need) {
  const int lane = static_cast<int>(lane_id());
  const int warp = threadIdx.x >> 5;
  for (int q = warp; q < kBins / 32; q += kWarps)  // block q: bins kBins-1-32q down to kBins-32-32q
    s.bsum[q] = __reduce_add_sync(0xFFFFFFFFu, h[kBins - 1 - (32 * q + lane)]);
  __syncthreads();
  if (warp == 0) {
    uint32_t b4[4], own = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      b4[k] = s.bsum[4 * lane + k];
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
    int qsel = 4 * L + 3;
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
    const int bin = kBins - 1 - (32 * qsel + lane);
    const uint32_t hv = h[bin];
    uint32_t in2 = hv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, in2, o);
      if (lane >= o) in2 += v;
    }
    const uint32_t hit2 = __ballot_sync(0xFFFFFFFFu, run + in2 >= static_cast<uint32_t>(need));
    const int L2 = hit2 ? __ffs(hit2) - 1 : 31;
    if (lane == L2) {
      s.fb = bin;
      s.fgt = static_cast<int>(run + in2 - hv);
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ copies

struct Win {
  const float* rowp;  // element 0 of the row
  int len;            // valid length (clamped)
  int mis;            // window elements before element 0 (16-byte alignment of the copies)
  int nwin;           // window elements, a multiple of 4 (0: nothing to read)
  int np;             // pieces of the window
};

__device__ __forceinline__ int clamp_len(const Params& p, int32_t raw, bool flag) {
  if (raw < 0 || static_cast<int64_t>(raw) > p.max_len) {
    if (flag) atomicOr(p.status, 0x1u);
    return raw < 0 ? 0 : static_cast<int>(p.max_len);
  }
  return raw;
}

// The window of row r for a length of n elements (n = max_len: the blind window).
__device__ __forceinline__ Win make_win(const Params& p, int64_t r, int n) {
  Win w;
  w.rowp = p.logits + r * p.stride;
  w.len = n;
  w.mis = (p.col_stride == 1) ? static_cast<int>((reinterpret_cast<uintptr_t>(w.rowp) & 15u) >> 2) : 0;
  w.nwin = (n > p.topk) ? ((n + w.mis + 3) & ~3) : 0;
  w.np = (w.nwin + kPiece - 1) / kPiece;
  return w;
}

// Issues the bulk copy of window piece j into ring slot q. Each 16-byte
// granule copied holds at least one element of the row, so no copy leaves the
// row's pages.
__device__ __forceinline__ void issue_piece(Smem& s, const Win& w, int j, int q, bool after_use) {
  if (after_use) fence_proxy_async();  // the slot was read through the generic proxy
  const int e0 = j * kPiece;
  const int e1 = min(e0 + kPiece, w.nwin);
  s.slot_issues[q] += 1;
  bulk_copy(&s.row[q * kPiece], w.rowp - w.mis + e0, static_cast<uint32_t>(e1 - e0) * 4u, &s.bar[q]);
}

// Pieces [i0, i1) of window w (i1 - i0 <= 32), piece i into slot (s0 + i) %
// kRing: lane l of the calling warp issues piece i0 + l, so the copies leave
// together.
__device__ __forceinline__ void issue_pieces(Smem& s, const Win& w, int i0, int i1, int s0, bool after_use) {
  const int i = i0 + static_cast<int>(lane_id());
  if (i < i1) issue_piece(s, w, i, (s0 + i) % kRing, after_use);
}

// Parity flips of the slots over the ring positions [s0, s0 + span) of one row.
__device__ __forceinline__ uint32_t slot_flips(int s0, int span) {
  // positions s0 .. s0 + span - 1 round the ring: every slot takes span / kRing
  // of them, and the span % kRing slots from s0 on one more
  constexpr uint32_t kAll = (1u << kRing) - 1u;
  const uint32_t extra = (1u << (span % kRing)) - 1u;
  const uint32_t m = ((span / kRing) & 1) ? kAll : 0u;
  return m ^ (((extra << s0) | (extra >> (kRing - s0))) & kAll);
}

// A row's window as 16-byte groups: group v holds window elements 4v .. 4v + 3
// (window element i is row element i - mis). The window sits in the ring (from
// float4 `ring0` on, wrapping round it), or in global memory: contiguous float4s
// from a 16-byte aligned base, or a row with a column stride (mis = 0; elements
// at or past the length are not read).
struct Src {
  const float* g;  // global memory: the window's base, or the strided row
  int64_t cs;      // global memory: the column stride (1: float4 loads)
  int ring0;       // the window's first float4 in the ring; -1: global memory
  int len;         // the row's length
};

__device__ __forceinline__ float4 load_group(const Smem& s, const Src& src, int v) {
  if (src.ring0 >= 0) return reinterpret_cast<const float4*>(s.row)[(src.ring0 + v) % kRingF4];
  if (src.cs == 1) return __ldg(reinterpret_cast<const float4*>(src.g) + v);
  float f[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = 4 * v + j;
    f[j] = (e < src.len) ? __ldg(src.g + static_cast<int64_t>(e) * src.cs) : 0.0f;
  }
  return make_float4(f[0], f[1], f[2], f[3]);
}

// ---------------------------------------------------------------- fallback

// The K-th key of the window elements [lo, lo + n), exactly, whatever the
// data: three radix levels over the full key (12, 12 and 8 bits). Returns the
// key T; `need` is how many of the keys equal to T are among the K best (the
// first ones in index order) and `equal` how many keys equal T. Thread t reads
// groups t, t + kThreads, ... (coalesced in global memory, free of bank
// conflicts in the ring); a thread counts each run of equal digits with one
// atomic, so tie-heavy rows cost few atomics. Uses s.hseed and clears s.n_out.
// Block-wide; every thread gets the answer.
__device__ __noinline__ uint32_t exact_kth(Smem& s, const Src src, int lo, int n, int K, int& need,
                                          int& equal) {
  const int tid = threadIdx.x;
  const int hi = lo + n;
  const int nv = (hi + 3) >> 2;
  uint32_t prefix = 0;
  need = K;
  if (tid == 0) s.n_out = 0;
  // levels: bits 31..20, 19..8 (within prefix), 7..0 (within prefix)
#pragma unroll 1
  for (int lv = 0; lv < 3; ++lv) {
    const int shift = lv == 0 ? 20 : lv == 1 ? 8 : 0;
    const int pshift = lv == 0 ? 32 : lv == 1 ? 20 : 8;
    const uint32_t mask = lv == 2 ? 0xFFu : 0xFFFu;
    for (int b = tid; b < kBins; b += kThreads) s.hseed[b] = 0;
    __syncthreads();
    uint32_t cur = 0xFFFFFFFFu, run = 0;
#pragma unroll 4
    for (int v = tid; v < nv; v += kThreads) {
      const float4 f = load_group(s, src, v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * v + j;
        if (i < lo || i >= hi) continue;
        const uint32_t k = fkey(pick(f, j));
        if (pshift < 32 && (k >> pshift) != prefix) continue;
        const uint32_t d = (k >> shift) & mask;
        if (d != cur) {
          if (run) atomicAdd(&s.hseed[cur], run);
          cur = d;
          run = 0;
        }
        ++run;
      }
    }
    if (run) atomicAdd(&s.hseed[cur], run);
    __syncthreads();
    find_top(s, s.hseed, need);  // digits above 255 stay empty at level 2
    need -= s.fgt;
    prefix = (prefix << (lv == 2 ? 8 : 12)) | static_cast<uint32_t>(s.fb);
  }
  equal = static_cast<int>(s.hseed[s.fb]);  // the last level's bin holds exactly the keys equal to T
  return prefix;
}

// Exact selection over a whole row, whatever the data (the fallback of the
// fast path, and the path of strided rows longer than the ring): the K-th key
// T from exact_kth, then one pass writes the keys above T and the keys equal
// to T, the first `need` of them in index order when not all are taken (a
// block-wide scan ranks the ties of every kThreads groups). Rewrites the whole
// output row.
__device__ __noinline__ void fallback_select(Smem& s, const Params& p, int64_t r, const Win& w, const Src src) {
  const int tid = threadIdx.x;
  const int lane = static_cast<int>(lane_id());
  const int warp = tid >> 5;
  const int K = p.topk;
  int need, equal;
  const uint32_t T = exact_kth(s, src, w.mis, w.len, K, need, equal);
  const bool ranked = equal > need;  // keys equal to T are left out: take the first ones
  int32_t* o = p.out + r * static_cast<int64_t>(K);
  const int lo = w.mis, hi = w.mis + w.len;
  const int nv = (hi + 3) >> 2;
  int before = 0;  // keys equal to T in the groups already passed
#pragma unroll 1
  for (int c = 0; c * kThreads < nv; ++c) {
    const int v = c * kThreads + tid;
    uint32_t above = 0, tie = 0;  // bit j: window element 4v + j
    if (v < nv) {
      const float4 f = load_group(s, src, v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = 4 * v + j;
        if (i >= lo && i < hi) {
          const uint32_t k = fkey(pick(f, j));
          above |= (k > T ? 1u : 0u) << j;
          tie |= (k == T ? 1u : 0u) << j;
        }
      }
    }
    if (ranked) {
      const int nt = __popc(tie);
      int incl = nt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += x;
      }
      if (lane == 31) s.tcnt[c & 1][warp] = incl;
      __syncthreads();
      const int wt = lane < kWarps ? s.tcnt[c & 1][lane] : 0;
      int wincl = wt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int x = __shfl_up_sync(0xFFFFFFFFu, wincl, d);
        if (lane >= d) wincl += x;
      }
      int rank = before + __shfl_sync(0xFFFFFFFFu, wincl - wt, warp) + incl - nt;
      before += __shfl_sync(0xFFFFFFFFu, wincl, 31);
      uint32_t keep = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if ((tie >> j) & 1u) {
          if (rank < need) keep |= 1u << j;
          ++rank;
        }
      }
      tie = keep;
    }
    const uint32_t sel = above | tie;
#pragma unroll
    for (int j = 0; j < 4; ++j) warp_emit(o, &s.n_out, K, (sel >> j) & 1u, 4 * v + j - lo);
  }
  __syncthreads();
}

// ------------------------------------------------------------------ kernel

// Waits for an mbarrier phase, the thread suspended (not spinning) until it
// completes or the hint runs out.
__device__ __forceinline__ bool mbar_wait_sleep(unsigned long long* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Waits (bounded) for piece q's phase `parity`. Warp-uniform answer.
__device__ __forceinline__ bool piece_ready(Smem& s, int q, uint32_t parity, uint64_t timeout_ns) {
  bool ok = mbar_try_wait(&s.bar[q], parity);
  if (!__all_sync(0xFFFFFFFFu, ok)) {
    const uint64_t t0 = global_timer();
    while (!ok) {
      ok = mbar_wait_sleep(&s.bar[q], parity);
      if (!ok && global_timer() - t0 > timeout_ns) break;
    }
  }
  return __all_sync(0xFFFFFFFFu, ok);
}

// One warp, every lane with the same answer: over h[0, kBins), with no counts
// above bin `top`, the bin b where the suffix sum (bins >= b) reaches need;
// `above` = the count in bins > b. Requires 1 <= need <= total. Up to two
// steps of 128 bins down from top (lane l: four bins, one 16-byte load); a
// crossing lower down is found at once (lane l sums 128 bins), then within
// that lane's stretch, four bins a lane.
__device__ __forceinline__ void warp_scan_down(const uint32_t* h, int top, int need, int& bin, int& above) {
  const int lane = static_cast<int>(lane_id());
  const uint32_t u_need = static_cast<uint32_t>(need);
  uint32_t carry = 0;  // the count in bins above the current step
  // one step over bins hi - 127 .. hi (hi = 4 k + 3): lane l holds hi - 4l - 3 .. hi - 4l
  auto step4 = [&](int hi) -> bool {
    const int lo4 = hi - 4 * lane - 3;
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    if (lo4 >= 0) q = *reinterpret_cast<const uint4*>(h + lo4);
    const uint32_t own = q.x + q.y + q.z + q.w;
    uint32_t incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += x;
    }
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, carry + incl >= u_need);
    if (hit == 0) {
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
      return false;
    }
    const int L = __ffs(hit) - 1;
    uint32_t run = carry + __shfl_sync(0xFFFFFFFFu, incl - own, L);
    const uint32_t v3 = __shfl_sync(0xFFFFFFFFu, q.w, L), v2 = __shfl_sync(0xFFFFFFFFu, q.z, L);
    const uint32_t v1 = __shfl_sync(0xFFFFFFFFu, q.y, L);
    const int base = hi - 4 * L - 3;
    if (run + v3 >= u_need) {
      bin = base + 3;
    } else if (run += v3, run + v2 >= u_need) {
      bin = base + 2;
    } else if (run += v2, run + v1 >= u_need) {
      bin = base + 1;
    } else {
      run += v1;
      bin = base;
    }
    above = static_cast<int>(run);
    return true;
  };
  int b0 = top | 3;
#pragma unroll 1
  for (int st = 0; st < 2 && b0 >= 0; ++st, b0 -= 128)
    if (step4(b0)) return;
  bin = 0;
  above = static_cast<int>(carry);
  if (b0 < 0) return;  // unreachable when the total reaches need
  // the rest at once: lane l sums bins b0 - 128 l - 127 .. b0 - 128 l
  uint32_t own = 0;
#pragma unroll 8
  for (int k = 0; k < 32; ++k) {
    const int lo4 = b0 - 128 * lane - 4 * k - 3;
    if (lo4 >= 0) {
      const uint4 q = *reinterpret_cast<const uint4*>(h + lo4);
      own += q.x + q.y + q.z + q.w;
    }
  }
  uint32_t incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  const uint32_t hit = __ballot_sync(0xFFFFFFFFu, carry + incl >= u_need);
  if (hit == 0) return;  // unreachable when the total reaches need
  const int L = __ffs(hit) - 1;
  carry += __shfl_sync(0xFFFFFFFFu, incl - own, L);
  step4(b0 - 128 * L);
}

// One warp, every lane with the same answer: over h[0, 256), the largest bin b
// whose suffix sum reaches need (1 <= need <= total); `above` = the count in
// bins > b.
__device__ __forceinline__ int warp_find256(const uint32_t* h, int need, int& above) {
  const int lane = static_cast<int>(lane_id());
  const uint4 lo4 = *reinterpret_cast<const uint4*>(h + 248 - 8 * lane);
  const uint4 hi4 = *reinterpret_cast<const uint4*>(h + 252 - 8 * lane);
  const uint32_t v[8] = {hi4.w, hi4.z, hi4.y, hi4.x, lo4.w, lo4.z, lo4.y, lo4.x};  // bins 255-8l down
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
  uint32_t run = __shfl_sync(0xFFFFFFFFu, incl - own, L);
  int b = 255 - 8 * L - 7;
  bool found = false;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t vk = __shfl_sync(0xFFFFFFFFu, v[k], L);
    if (!found && run + vk >= static_cast<uint32_t>(need)) {
      b = 255 - 8 * L - k;
      found = true;
    }
    if (!found) run += vk;
  }
  above = static_cast<int>(run);
  return b;
}

// Ranks entries [0, n) of (kk, ii) by key descending, then index ascending
// (entries [n, c4) hold padding that never beats a real entry), and writes the
// index of every entry of rank < need at out[rank]. Groups of 2^lg lanes (the
// most that fit the block, at most a warp) share an entry: lane `sub` of a
// group compares it with entries 4 sub .. 4 sub + 3, then every 4 * 2^lg-th
// on. Needs n <= kThreads. Block-wide (no barrier).
__device__ __forceinline__ void rank_out(const uint32_t* kk, const int32_t* ii, int n, int c4, int need,
                                         int32_t* out) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  int lg = 5;
  while ((n << lg) > kThreads) --lg;
  const int e = tid >> lg;
  const int sub = tid & ((1 << lg) - 1);
  if (((warp << 5) >> lg) >= n) return;  // no entry's group in this warp (groups never straddle warps)
  const bool act = e < n;
  const uint32_t kj = act ? kk[e] : 0u;
  const int32_t ij = act ? ii[e] : 0;
  int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
  for (int i0 = 4 * sub; i0 < c4; i0 += 4 << lg) {
    const uint4 k4 = *reinterpret_cast<const uint4*>(&kk[i0]);
    const int4 x4 = *reinterpret_cast<const int4*>(&ii[i0]);
    r0 += (k4.x > kj || (k4.x == kj && x4.x < ij)) ? 1 : 0;
    r1 += (k4.y > kj || (k4.y == kj && x4.y < ij)) ? 1 : 0;
    r2 += (k4.z > kj || (k4.z == kj && x4.z < ij)) ? 1 : 0;
    r3 += (k4.w > kj || (k4.w == kj && x4.w < ij)) ? 1 : 0;
  }
  int rank = r0 + r1 + r2 + r3;
  for (int o2 = 1; o2 < (1 << lg); o2 <<= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o2);
  if (act && sub == 0 && rank < need) out[rank] = ij;
}

// Exclusive prefix over the lanes of a warp.
__device__ __forceinline__ int warp_excl(int v) {
  const int lane = static_cast<int>(lane_id());
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  return incl - v;
}

__device__ __forceinline__ int atom_add_acq_rel_cta(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}

// A crowded seed bin on a streamed row (heavy ties): the seed piece's own K
// best, that is its K-th key T and the first `need` of its elements equal to T
// in index order, go into the candidate regions (warp w's at most 64 into its
// own). Every later element of the row has a larger index than all of them,
// so one equal to T can never be selected: the filter then keeps key > T only,
// which is exact for any data. Returns T; `wc` = this warp's candidates, also
// counted in its fine bin 0 (T's). Block-wide.
__device__ __noinline__ uint32_t crowded_seed(Smem& s, int S, int mis, int n_seed, int len, int K, int& wc) {
  const int tid = threadIdx.x;
  const int lane = static_cast<int>(lane_id());
  const int warp = tid >> 5;
  const float* seed = s.row + S * kPiece;
  int need_t, equal_t;
  const uint32_t T = exact_kth(s, Src{nullptr, 1, S * (kPiece / 4), len}, mis, n_seed, K, need_t, equal_t);
  // thread i owns seed elements E i .. E i + E - 1; a block scan ranks the ties
  constexpr int E = kSeed / kThreads;
  static_assert(E * kThreads == kSeed && 32 * E <= kRegion, "the seed's ties fit the warps' regions");
  const int e0 = E * tid;
  uint32_t tie = 0;
#pragma unroll
  for (int j = 0; j < E; ++j)
    if (e0 + j < n_seed && fkey(seed[mis + e0 + j]) == T) tie |= 1u << j;
  const int mine = __popc(tie);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) s.tcnt[0][warp] = incl;
  __syncthreads();
  int rank = incl - mine;
  for (int q = 0; q < warp; ++q) rank += s.tcnt[0][q];
  uint32_t keep = 0;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    if ((tie >> j) & 1u) {
      if (rank < need_t) keep |= 1u << j;
      ++rank;
    }
  }
  const int sel = __popc(keep);
  int at = warp * kRegion + warp_excl(sel);  // at most 32 E per warp: inside its region
#pragma unroll
  for (int j = 0; j < E; ++j) {
    if ((keep >> j) & 1u) {
      s.ckey[at] = T;
      s.cidx[at] = e0 + j;
      ++at;
    }
  }
  wc = static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, static_cast<uint32_t>(sel)));
  if (lane == 0 && wc) atomicAdd(&s.wbin[warp][0], wc);  // T's fine bin: 0
  __syncthreads();
  return T;
}

__global__ void __launch_bounds__(kThreads, 1) topk_short_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  const int lane = static_cast<int>(lane_id());
  const int warp = tid >> 5;
  const uint32_t lt = lanemask_lt();
  const int K = p.topk;
  const bool bulk = p.col_stride == 1;
  int64_t r = blockIdx.x;
  if (r >= p.num_rows) return;
  wait_previous_grid();

  // Set-up: warp 0's lanes initialise the slot barriers and, with contiguous
  // rows, lane 0 issues piece 0 of the first row's blind window (sized by
  // max_len, up to kBlind pieces) before anything else; after the barrier,
  // when the first length is in, warp 1 issues the rest of the blind pieces
  // and then the row's own window up to a ring's worth, so the seed's piece is
  // queued behind none of them and few pieces are fetched past the row.
  const int32_t len_raw0 = __ldg(p.lengths + r);
  // thread 0 holds the raw length of the next row, loaded a row ahead of its use
  int32_t nl_raw = (tid == 0 && r + gridDim.x < p.num_rows) ? __ldg(p.lengths + r + gridDim.x) : 0;
  int blind = 0;  // pieces of the first row in flight before its length is known
  if (bulk) blind = min(make_win(p, r, static_cast<int>(p.max_len)).np, kBlind);  // the same in every thread
  if (warp == 0) {
    if (lane < kRing) {
      mbar_init(&s.bar[lane], 1u);
      fence_mbar_init();
      s.pdone[lane] = 0;
      s.slot_issues[lane] = 0;
    }
    if (lane == 0) {
      s.abort = 0;
      s.key_max = 0;
    }
    if (bulk) issue_pieces(s, make_win(p, r, static_cast<int>(p.max_len)), 0, min(blind, 1), 0, false);
  }
  for (int b = tid; b < kBins; b += kThreads) s.hseed[b] = 0;
  for (int i = tid; i < kWarps * kTrack; i += kThreads) s.wbin[i / kTrack][i % kTrack] = 0;
  if (tid < 256) s.hsub[tid] = 0;
  if (tid < kTrack) s.ftot[tid] = 0;
  if (tid == 0) {
    s.n_win = 0;
    s.n_bt = 0;
    s.cmax = 0;
  }
  __syncthreads();
  int len = clamp_len(p, len_raw0, tid == 0);
  if (warp == 1 && bulk) {
    issue_pieces(s, make_win(p, r, static_cast<int>(p.max_len)), 1, blind, 0, false);
    const Win w0 = make_win(p, r, len);
    issue_pieces(s, w0, blind, min(w0.np, kRing), 0, false);
  }

  uint32_t par = 0;  // bit q: parity of the next phase of slot q's barrier
  int S = 0;         // ring slot of the current row's piece 0 (rows follow one another round the ring)
  bool aborted = false;
#pragma unroll 1
  for (int64_t k = 0; r < p.num_rows; ++k) {
    const int64_t rn = r + gridDim.x;
    if (tid == 0) {
      s.len_next = (rn < p.num_rows) ? clamp_len(p, nl_raw, true) : 0;
      const int64_t rnn = rn + gridDim.x;
      nl_raw = (rnn < p.num_rows) ? __ldg(p.lengths + rnn) : 0;
    }
    const Win w = make_win(p, r, len);
    int32_t* o = p.out + r * static_cast<int64_t>(K);
    const int dead = (k == 0) ? blind : 0;     // the first row's blind pieces (those past its window are dead)
    const bool stream = bulk && w.np > kRing;  // the row streams through the ring
    // ring positions the row takes (its pieces, and the first row's dead blind ones)
    const int span = bulk ? max(w.np, dead) : 0;
    const int S_next = (S + span) % kRing;
    // cross-row prefetch: the next row's first pieces go into the ring while this
    // row is still being filtered, as slots come free (not after a row of dead
    // blind pieces, whose slots free up only at its end, nor after a trivial row)
    const bool cross = bulk && rn < p.num_rows && w.nwin > 0 && dead <= w.np;
    Win wn{};
    int np_next = 0;  // the next row's pieces that this row hands slots to
    if (w.nwin == 0) {
      for (int j = tid; j < K; j += kThreads) o[j] = (j < len) ? j : -1;
    } else if (!bulk && w.nwin > kRing * kPiece) {
      // a strided row longer than the ring: exact selection straight from global memory
      fallback_select(s, p, r, w, Src{w.rowp, p.col_stride, -1, len});
    } else {
      if (!bulk) {
        // strided rows: every thread loads its elements into the window
        const int64_t cs = p.col_stride;
        for (int e = tid; e < len; e += kThreads) s.row[e] = __ldg(w.rowp + static_cast<int64_t>(e) * cs);
        __syncthreads();
      }
      // ---- seed: the top 12 key bits of piece 0 (slot S) and its largest key. Warp 0
      // first works out how many of the sample's best the threshold should keep
      // (it needs no data)
      const int n_seed = min(len, kSeed - w.mis);
      int target = K;
      if (warp == 0 && n_seed < len) {
        // mu = the expected count of the row's K best in the sample; aim three
        // standard deviations above it (mu is small on long rows), so a sample
        // that runs short of it still leaves K survivors
        const float mu = static_cast<float>(K) * static_cast<float>(n_seed) / static_cast<float>(len);
        target = max(1, static_cast<int>(ceilf(mu + 3.0f * sqrtf(mu) + 2.0f)));
      }
      target = min(target, n_seed);
      bool ok = !bulk || piece_ready(s, S, (par >> S) & 1u, p.timeout_ns);
      const int seed_hi = min(kSeed, w.nwin);
      const float* seed = s.row + S * kPiece;  // a piece never wraps round the ring
      uint32_t kmax = 0;
      for (int i = tid; i < seed_hi; i += kThreads) {
        const int e = i - w.mis;
        if (e >= 0 && e < len) {
          const uint32_t key = fkey(seed[i]);
          kmax = max(kmax, key);
          atomicAdd(&s.hseed[key >> 20], 1u);
        }
      }
      kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
      if (lane == 0 && kmax) atomicMax(&s.key_max, kmax);
      if (sync_or(!ok)) {
        aborted = true;
      } else {
        if (cross) {
          // the next row's length is in (thread 0 wrote it before the barrier); its
          // first pieces whose slots this row never takes go into the ring now
          wn = make_win(p, rn, s.len_next);
          np_next = min(wn.np, kRing);
          if (warp == 0) issue_pieces(s, wn, 0, min(np_next, kRing - span), S_next, true);
        }
        if (warp == 0) {
          int t0, above0;
          warp_scan_down(s.hseed, static_cast<int>(s.key_max >> 20), target, t0, above0);
          const int c0 = static_cast<int>(s.hseed[t0]);
          const int need_in = target - above0;  // of bin t0's sample entries, 1 .. c0
          // a crowded seed bin on a streamed row (heavy ties): the seed piece holds
          // K or more elements at or above t0, and the projection over the row
          // overflows the candidate regions
          const int at_or_above = above0 + static_cast<int>(s.hseed[t0]);
          const bool crowded = stream && n_seed >= K && at_or_above >= K &&
                               static_cast<int64_t>(at_or_above) * len > (3ll * kCand / 4) * n_seed;
          // a wide seed bin (its sample count well beyond what the target needs from
          // it) is split on the next 8 key bits, so the threshold lands close to it
          const bool refine = !crowded && c0 - need_in > max(target / 4, 16) &&
                              (stream || static_cast<int64_t>(c0 - need_in) * len > static_cast<int64_t>(kRefineExcess) * n_seed);
          if (lane == 0) {
            s.target = target;
            s.t0 = t0;
            s.crowded = crowded ? 1 : 0;
            s.refine = refine ? 1 : 0;
            s.need_in = need_in;
            s.thr_key = static_cast<uint32_t>(t0) << 20;
          }
        }
        __syncthreads();
        if (s.refine) {
          const uint32_t t0 = static_cast<uint32_t>(s.t0);
          for (int i = tid; i < seed_hi; i += kThreads) {
            const int e = i - w.mis;
            if (e >= 0 && e < len) {
              const uint32_t key = fkey(seed[i]);
              if ((key >> 20) == t0) atomicAdd(&s.hsub[(key >> 12) & 0xFFu], 1u);
            }
          }
          __syncthreads();
          if (warp == 0) {
            int above_b;
            const int b = warp_find256(s.hsub, s.need_in, above_b);
            if (lane == 0) s.thr_key = (t0 << 20) | (static_cast<uint32_t>(b) << 12);
          }
          __syncthreads();
          if (tid < 256) s.hsub[tid] = 0;  // clear again for the selection (read after later barriers)
        }
        // ---- filter: warp tasks of 128 F window elements (F = 1, 2, 4 or 8); lane l of a task takes
        // float4s l, l + 32, ... of it. Piece j sits in slot j % kRing; on a
        // streamed row the last of its tasks hands the slot to piece j + kRing.
        uint32_t thr_key = s.thr_key;  // the filter keeps keys >= thr_key
        float thr = key_floor_value(thr_key);
        const int base = warp * kRegion;
        int wc = 0;
        int* my_bins = s.wbin[warp];  // this warp's own counters: no other warp touches them
        if (s.crowded) {
          const uint32_t T = crowded_seed(s, S, w.mis, n_seed, len, K, wc);
          thr_key = T;                    // the fine bins count from T's (the ties are candidates)
          thr = key_floor_value(T + 1u);  // T is at most the key of +inf, so T + 1 does not wrap
        }
        const int nvec = w.nwin >> 2;
        // float4s per lane in a task: the most (up to 8, which spreads the per-task
        // work over the most elements) that keep a task's expected survivors (the
        // seed's share of the row) within kTaskSurvivors, and the window in at least
        // kMinTasks tasks
        int F = 8;
        while (F > 1 && (static_cast<int64_t>(128 * F) * s.target > static_cast<int64_t>(kTaskSurvivors) * n_seed ||
                         w.nwin < kMinTasks * 128 * F))
          F >>= 1;
        const int tsz = 128 * F;  // window elements per task
        const int ntask = (w.nwin + tsz - 1) / tsz;
#pragma unroll 1
        for (int task = warp; task < ntask; task += kWarps) {
          const int j = (task * tsz) / kPiece;    // window piece
          const int q = (S + j) % kRing;          // its slot
          if (bulk && j >= 1 && !piece_ready(s, q, ((par >> q) ^ static_cast<uint32_t>(j / kRing)) & 1u, p.timeout_ns)) {
            ok = false;  // the whole warp leaves the filter; the barrier below decides for the CTA
            break;
          }
          const int sb = q * kPiece + (task * tsz) % kPiece;  // the task's first element in the ring
          const int v0 = task * (tsz / 4);                    // and its first float4 in the window
          uint32_t m = 0;
          if (v0 + 32 * F <= nvec && 4 * v0 - w.mis >= 0 && 4 * v0 + tsz - w.mis <= len) {
            // a task inside the row: no element needs a bounds check (the common
            // F = 8 spelt out, so that its eight loads go out unconditionally)
            if (F == 8) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 f = *reinterpret_cast<const float4*>(&s.row[sb + 4 * (lane + 32 * i)]);
                m |= ((f.x >= thr ? 1u : 0u) | (f.y >= thr ? 2u : 0u) | (f.z >= thr ? 4u : 0u) |
                      (f.w >= thr ? 8u : 0u)) << (4 * i);
              }
            } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (i < F) {
                const float4 f = *reinterpret_cast<const float4*>(&s.row[sb + 4 * (lane + 32 * i)]);
                m |= ((f.x >= thr ? 1u : 0u) | (f.y >= thr ? 2u : 0u) | (f.z >= thr ? 4u : 0u) |
                      (f.w >= thr ? 8u : 0u)) << (4 * i);
              }
            }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int v = v0 + lane + 32 * i;
              if (i < F && v < nvec) {
                const float4 f = *reinterpret_cast<const float4*>(&s.row[sb + 4 * (lane + 32 * i)]);
                uint32_t b = (f.x >= thr ? 1u : 0u) | (f.y >= thr ? 2u : 0u) | (f.z >= thr ? 4u : 0u) |
                             (f.w >= thr ? 8u : 0u);
                const int e0 = 4 * v - w.mis;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  if (e0 + c < 0 || e0 + c >= len) b &= ~(1u << c);
                m |= b << (4 * i);
              }
            }
          }
          const int c = __popc(m);  // at most 32
          // the warp's survivors and this lane's exclusive prefix, one ballot per bit of
          // the lanes' counts: bits 0..2 always, bits 3..5 only when a lane has 8 or
          // more (rare: the threshold keeps a few percent of the elements)
          int tot = 0, pre = 0;
#pragma unroll
          for (int bit = 0; bit < 3; ++bit) {
            const uint32_t qb = __ballot_sync(0xFFFFFFFFu, (c >> bit) & 1);
            tot += __popc(qb) << bit;
            pre += __popc(qb & lt) << bit;
          }
          if (__any_sync(0xFFFFFFFFu, c >= 8)) {
#pragma unroll
            for (int bit = 3; bit < 6; ++bit) {
              const uint32_t qb = __ballot_sync(0xFFFFFFFFu, (c >> bit) & 1);
              tot += __popc(qb) << bit;
              pre += __popc(qb & lt) << bit;
            }
          }
          if (tot > 0) {
            if (wc + tot <= kRegion) {
              // each lane notes where its survivors are (task positions) in the
              // region, then the warp converts them 32 at a time
              int at = base + wc + pre;
              while (m) {
                const int jb = __ffs(m) - 1;
                m &= m - 1;
                s.cidx[at++] = 4 * (lane + 32 * (jb >> 2)) + (jb & 3);
              }
              __syncwarp();
#pragma unroll 1
              for (int e0 = 0; e0 < tot; e0 += 32) {
                const int e = e0 + lane;
                if (e < tot) {
                  const int pos = s.cidx[base + wc + e];
                  const uint32_t key = fkey(s.row[sb + pos]);
                  s.ckey[base + wc + e] = key;
                  s.cidx[base + wc + e] = task * tsz + pos - w.mis;
                  const uint32_t d = (key - thr_key) >> kFine;
                  if (d < kTrack) atomicAdd(&my_bins[d], 1);
                }
              }
              __syncwarp();
            }
            wc += tot;
          }
          // once every task of piece j is done, its slot goes to piece j + kRing of
          // this row, or, on a streamed row, on to the next row's piece j + kRing -
          // np (a resident row keeps its slots until it is selected: its exact
          // fallback reads them)
          const bool same = bulk && j + kRing < w.np;
          const bool onto_next = cross && stream && !same && j + kRing - w.np < np_next;
          if (same || onto_next) {
            const int tasks_j = min(kPiece / tsz, ntask - j * (kPiece / tsz));  // a last piece may be short
            __syncwarp();  // every lane's reads of the slot come before the hand-over
            if (lane == 0 && atom_add_acq_rel_cta(&s.pdone[q], 1) == tasks_j - 1) {
              s.pdone[q] = 0;
              if (same)
                issue_piece(s, w, j + kRing, q, true);
              else
                issue_piece(s, wn, j + kRing - w.np, q, true);
            }
          }
        }
        if (lane == 0) s.wcnt[warp] = wc;
        if (wc > 0) {
          // this warp's fine-bin counts into the totals over the warps
          const int2 v2 = *reinterpret_cast<const int2*>(&my_bins[2 * lane]);
          if (v2.x) atomicAdd(&s.ftot[2 * lane], v2.x);
          if (v2.y) atomicAdd(&s.ftot[2 * lane + 1], v2.y);
        }
        if (sync_or(!ok)) {
          aborted = true;
        } else {
          // ---- the K-th key's fine bin t (warp 0; lane l reads warp l's survivor
          // count and the totals of fine bins 2l and 2l + 1). When the K-th key lies
          // above the 64 bins counted, the candidates are counted once more in bins
          // wide enough to hold them all, and the search repeats.
          int fsh = kFine;  // fine bin of a candidate: (key - thr_key) >> fsh
#pragma unroll 1
          for (;;) {
          if (warp == 0) {
            const int n_l = lane < kWarps ? s.wcnt[lane] : 0;
            const int2 c2 = *reinterpret_cast<const int2*>(&s.ftot[2 * lane]);
            const int c0 = c2.x, c1 = c2.y;
            const bool over = __any_sync(0xFFFFFFFFu, n_l > kRegion);
            const int n_c = static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, static_cast<uint32_t>(n_l)));
            const int skip = n_c - K;  // the K-th key's bin: the first whose prefix (from f0) passes skip
            const int pair = c0 + c1;
            int incl = pair;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
              if (lane >= o) incl += x;
            }
            const int p0 = incl - pair + c0;  // prefix through bin 2 lane
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl > skip);
            const int L = hit ? __ffs(hit) - 1 : 0;
            const bool first = __shfl_sync(0xFFFFFFFFu, p0, L) > skip;
            const int jt = 2 * L + (first ? 0 : 1);
            const int cum = first ? __shfl_sync(0xFFFFFFFFu, p0, L) : __shfl_sync(0xFFFFFFFFu, incl, L);
            const int in_t = first ? __shfl_sync(0xFFFFFFFFu, c0, L) : __shfl_sync(0xFFFFFFFFu, c1, L);
            const int need = K - (n_c - cum);
            const bool all_t = need == in_t;
            const bool sel_ok = !over && n_c >= K && hit != 0 && (all_t || in_t <= kRank);
            if (lane == 0) {
              s.wide = (!over && n_c >= K && hit == 0 && fsh == kFine) ? 1 : 0;
              s.sel_ok = sel_ok ? 1 : 0;
              s.t = jt;
              s.need = all_t ? 0 : need;  // 0: bin t is taken whole
              s.in_t = in_t;
            }
          }
          __syncthreads();
          if (!s.wide) break;
          // count again: the smallest shift that puts every candidate in the 64 bins
          const int cnt_w = s.wcnt[warp];  // at most kRegion: no overflow here
          uint32_t cmax = thr_key;
          for (int e = lane; e < cnt_w; e += 32) cmax = max(cmax, s.ckey[base + e]);
          cmax = __reduce_max_sync(0xFFFFFFFFu, cmax);
          if (lane == 0) atomicMax(&s.cmax, cmax);
          *reinterpret_cast<int2*>(&my_bins[2 * lane]) = make_int2(0, 0);
          if (tid < kTrack) s.ftot[tid] = 0;
          __syncthreads();
          const uint32_t span = s.cmax - thr_key;
          while ((span >> fsh) >= static_cast<uint32_t>(kTrack)) ++fsh;
          for (int e = lane; e < cnt_w; e += 32) atomicAdd(&my_bins[(s.ckey[base + e] - thr_key) >> fsh], 1);
          __syncwarp();
          if (cnt_w > 0) {
            const int2 v2 = *reinterpret_cast<const int2*>(&my_bins[2 * lane]);
            if (v2.x) atomicAdd(&s.ftot[2 * lane], v2.x);
            if (v2.y) atomicAdd(&s.ftot[2 * lane + 1], v2.y);
          }
          __syncthreads();
          }
          bool done = false;
          if (s.sel_ok) {
            // ---- winners above bin t out; bin t's entries into the ranking slots
            const int jt = s.t;
            const int need = s.need;
            const bool all_t = need == 0;
            const int cnt = s.wcnt[warp];  // at most kRegion here
            // this warp's candidates above bin t and in it, from its own fine bins;
            // its output range and ranking slots come from two shared counters (the
            // order of a row's indices is free)
            const int2 b2 = *reinterpret_cast<const int2*>(&my_bins[2 * lane]);
            const int below = static_cast<int>(__reduce_add_sync(
                0xFFFFFFFFu, static_cast<uint32_t>((2 * lane <= jt ? b2.x : 0) + (2 * lane + 1 <= jt ? b2.y : 0))));
            int bt = my_bins[jt];
            int nw = cnt - below;
            if (all_t) {
              nw += bt;
              bt = 0;
            }
            int ow = 0, os = 0;
            if (lane == 0) {
              if (nw) ow = atomicAdd(&s.n_win, nw);
              if (bt) os = atomicAdd(&s.n_bt, bt);
            }
            ow = __shfl_sync(0xFFFFFFFFu, ow, 0);
            os = __shfl_sync(0xFFFFFFFFu, os, 0);
#pragma unroll 1
            for (int e0 = 0; e0 < cnt; e0 += 32) {
              const int e = e0 + lane;
              uint32_t key = 0;
              int32_t idx = 0;
              int d = -1;
              if (e < cnt) {
                key = s.ckey[base + e];
                idx = s.cidx[base + e];
                d = static_cast<int>((key - thr_key) >> fsh);
              }
              const bool win = d > jt || (all_t && d == jt);
              const bool inb = !all_t && d == jt;
              const uint32_t bw = __ballot_sync(0xFFFFFFFFu, win);
              if (win) o[ow + __popc(bw & lt)] = idx;
              ow += __popc(bw);
              const uint32_t bb = __ballot_sync(0xFFFFFFFFu, inb);
              if (inb) {
                const int at = os + __popc(bb & lt);
                s.rk[at] = key;
                s.ri[at] = idx;
              }
              os += __popc(bb);
            }
            if (!all_t) {
              const int in_t = s.in_t;
              const int c4 = (in_t + 3) & ~3;
              if (tid >= in_t && tid < c4) {  // padding never beats a real entry
                s.rk[tid] = 0u;
                s.ri[tid] = 0x7FFFFFFF;
              }
              __syncthreads();
              if (in_t <= kRankDirect) {
                rank_out(s.rk, s.ri, in_t, c4, need, o + (K - need));
              } else {
                // a large bin t: its entries split on the next 8 bits of key -
                // thr_key; entries above the sub-bin b that holds the need-th are
                // taken, those in it ranked
                if (tid < in_t) atomicAdd(&s.hsub[((s.rk[tid] - thr_key) >> (fsh - 8)) & 0xFFu], 1u);
                __syncthreads();
                if (warp == 0) {
                  int above_b;
                  const int b = warp_find256(s.hsub, need, above_b);
                  if (lane == 0) {
                    s.sub_b = b;
                    s.sub_above = above_b;
                    s.n_win = 0;  // the counters place the taken entries and gather sub-bin b's
                    s.n_bt = 0;
                  }
                }
                __syncthreads();
                const int b = s.sub_b;
                const int sab = s.sub_above;
                const int in_b = static_cast<int>(s.hsub[b]);
                if (tid < in_t) {
                  const uint32_t kj = s.rk[tid];
                  const int32_t ij = s.ri[tid];
                  const int d = static_cast<int>(((kj - thr_key) >> (fsh - 8)) & 0xFFu);
                  if (d > b) {
                    o[K - need + atomicAdd(&s.n_win, 1)] = ij;
                  } else if (d == b) {
                    const int at = atomicAdd(&s.n_bt, 1);
                    s.ckey[at] = kj;  // the candidate slots are free once emitted
                    s.cidx[at] = ij;
                  }
                }
                const int c4b = (in_b + 3) & ~3;
                if (tid >= in_b && tid < c4b) {
                  s.ckey[tid] = 0u;
                  s.cidx[tid] = 0x7FFFFFFF;
                }
                __syncthreads();
                rank_out(s.ckey, s.cidx, in_b, c4b, need - sab, o + (K - need + sab));
              }
            }
            done = true;
          }
          // a streamed row is read again from global memory; a resident one (strided rows
          // included: they were loaded contiguously) from the ring
          if (!done) {
            if (stream)
              fallback_select(s, p, r, w, Src{w.rowp - w.mis, 1, -1, len});
            else
              fallback_select(s, p, r, w, Src{nullptr, 1, bulk ? S * (kPiece / 4) : 0, len});
          }
        }
      }
    }
    // the row's end: clear the seed histogram, learn the next length, issue its window
    if (aborted) break;
    if (rn >= p.num_rows) {
      // the CTA's last row: nothing to clear; only the first row's dead blind
      // pieces may still be landing (lane q waits for slot q)
      if (warp == 0 && lane < kRing && lane >= w.np && lane < dead)
        wait_piece(&s.bar[lane], (par >> lane) & 1u, p.timeout_ns, &s.abort);
      break;
    }
    __syncthreads();
    // read here, between two barriers: thread 0 writes the one after it at the next row's start
    const int len_next = s.len_next;
    static_assert(kBins % (4 * kThreads) == 0, "16-byte stores clear the seed histogram");
#pragma unroll
    for (int b = tid; b < kBins / 4; b += kThreads) reinterpret_cast<uint4*>(s.hseed)[b] = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<int2*>(&s.wbin[warp][2 * lane]) = make_int2(0, 0);
    if (tid < 256) s.hsub[tid] = 0;
    if (tid < kTrack) s.ftot[tid] = 0;
    if (tid == 0) {
      s.n_win = 0;
      s.n_bt = 0;
      s.cmax = 0;
    }
    if (warp == 0) {
      // the first row's blind pieces past its window may still be landing:
      // wait for them before the ring takes the next window (lane q, slot q;
      // the first row starts at slot 0)
      if (lane < kRing && lane >= w.np && lane < dead)
        wait_piece(&s.bar[lane], (par >> lane) & 1u, p.timeout_ns, &s.abort);
      __syncwarp();
      if (lane == 0) s.key_max = 0;
      // the next row's first pieces not yet in the ring: all of them without
      // cross-row prefetch, else those whose slots a resident row kept
      if (rn < p.num_rows && bulk && !(cross && stream)) {
        const Win wn2 = make_win(p, rn, len_next);
        const int i0 = cross ? max(0, kRing - span) : 0;
        issue_pieces(s, wn2, i0, min(wn2.np, kRing), S_next, true);
      }
    }
    par ^= slot_flips(S, span);
    S = S_next;
    __syncthreads();
    r = rn;
    len = len_next;
  }
  if (aborted && tid == 0) {
    // a piece did not land in time: flag it, and wait (bounded) for the last
    // copy issued into every slot before the CTA leaves
    atomicOr(p.status, 0x4u);
    for (int q = 0; q < kRing; ++q) {
      const int n = s.slot_issues[q];
      if (n > 0) wait_piece(&s.bar[q], static_cast<uint32_t>(n - 1) & 1u, p.timeout_ns, nullptr);
    }
  }
}

// ------------------------------------------------------- cluster row split
//
// A row split over the C CTAs (C = 2 .. 8) of a thread-block cluster, one row
// per cluster, for launches with too few rows to fill the GPU (the same
// single-pass shape; the merge takes the place of the pages' cross-CTA radix
// histograms). CTA c takes window pieces c, c + C, c + 2 C, ..., a balanced
// share whatever the length, so each issues its first pieces before the
// length is read. Every CTA fetches piece 0 too and seeds the threshold from
// it as one CTA does, so all find the same one without waiting for each
// other; every CTA filters its pieces into its own candidate regions and
// stores its fine-bin counts into every CTA, so each finds the K-th key's fine
// bin t on its own, with the same answer, and knows where its winners and bin
// t entries go; it writes its winners and sends bin t's entries to CTA 0,
// which ranks them. Two cluster barriers a row after a start barrier (two more
// when the K-th key lies above the counted bins), taken by every thread of
// every CTA whatever happened before them, so a CTA that gave up still
// arrives; no CTA touches another's shared memory after the last one. The
// exact fallback runs in CTA 0, over the row in global memory.

// Every CTA of the cluster holds every CTA's counts (each CTA stores its own
// into all of them), so each takes the same decision on its own.
struct SmemC : Smem {
  alignas(16) int c_fc[kMaxCluster][kTrack];  // fine-bin counts of each CTA
  int c_nc[kMaxCluster];             // each CTA's count word: candidates, region overflow, gave up
  uint32_t c_mx[kMaxCluster];        // each CTA's largest candidate key
  int c_dec[7];                      // mode, fine bin t, need (0: bin t whole), bin t's entries, bin shift,
                                     // this CTA's first output slot and first ranking slot
};
static_assert(sizeof(SmemC) <= 227 * 1024, "the cluster kernel's shared memory fits one SM");

// The fine-bin counts of CTA c.
__device__ __forceinline__ int* cluster_fc(SmemC& s, int c) { return s.c_fc[c]; }

constexpr int kModeSelect = 1;  // bin t found: winners out, bin t's entries ranked in rank 0
constexpr int kModeWide = 2;    // the K-th key lies above the counted bins: count again, coarser
constexpr int kModeExact = 3;   // the exact fallback in rank 0
constexpr int kModeAbort = 4;   // a CTA gave up (a copy did not land in time)

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(v));
  return v;
}

// The address of the same shared variable in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* ptr, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(ptr)), "r"(rank));
  return a;
}

__device__ __forceinline__ void dsmem_st(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// The hardware cluster barrier: completes once every thread of every CTA of
// the cluster has arrived; shared-memory writes before it (this CTA's own and
// remote ones) are seen by every thread after it. Warp-uniform.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Warp 0 of each CTA: the K-th key's fine bin from the counts of all C CTAs of
// the cluster (bins of (key - thr_key) >> fsh), into c_dec; every
// CTA reads the same counts and takes the same decision. A K-th key above the
// counted bins asks for a recount (when `may_widen`) with the smallest shift
// that holds the cluster's largest candidate. With bin t found, CTA me's first
// output slot and first ranking slot follow the winners and bin t entries of
// CTAs 0 .. me - 1.
__device__ __forceinline__ void cluster_decide(SmemC& s, int K, int C, int me, int fsh, bool may_widen,
                                               uint32_t thr_key) {
  const int lane = static_cast<int>(lane_id());
  int c0 = 0, c1 = 0;  // bins 2 lane and 2 lane + 1, over the cluster
  int below = 0;       // packed: the earlier CTAs' candidates in bins up to t (low 16 bits) and in t (high)
  for (int c = 0; c < C; ++c) {
    const int2 v = *reinterpret_cast<const int2*>(cluster_fc(s, c) + 2 * lane);
    c0 += v.x;
    c1 += v.y;
  }
  // lane c < C: CTA c's packed count word (see cluster_push_counts); the sum
  // carries the candidates and how many CTAs overflowed or gave up
  const uint32_t word_l = lane < C ? static_cast<uint32_t>(s.c_nc[lane]) : 0u;
  const uint32_t sum = __reduce_add_sync(0xFFFFFFFFu, word_l);
  const int n_c = static_cast<int>(sum & 0xFFFFFFu);
  const uint32_t flags = ((sum >> 24) & 0xFu ? 1u : 0u) | ((sum >> 28) ? 2u : 0u);
  const int skip = n_c - K;  // the K-th key's bin: the first whose prefix (from bin 0) passes skip
  const int pair = c0 + c1;
  int incl = pair;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += x;
  }
  const int p0 = incl - pair + c0;
  const uint32_t hit = __ballot_sync(0xFFFFFFFFu, incl > skip);
  const int L = hit ? __ffs(hit) - 1 : 0;
  const bool first = __shfl_sync(0xFFFFFFFFu, p0, L) > skip;
  const int jt = 2 * L + (first ? 0 : 1);
  const int cum = first ? __shfl_sync(0xFFFFFFFFu, p0, L) : __shfl_sync(0xFFFFFFFFu, incl, L);
  const int in_t = first ? __shfl_sync(0xFFFFFFFFu, c0, L) : __shfl_sync(0xFFFFFFFFu, c1, L);
  const int need = K - (n_c - cum);
  const bool all_t = need == in_t;
  const bool base = flags == 0u && n_c >= K;
  int mode = kModeExact;
  if (flags & 2u)
    mode = kModeAbort;
  else if (base && hit != 0 && (all_t || in_t <= kRank))
    mode = kModeSelect;
  else if (base && hit == 0 && may_widen)
    mode = kModeWide;
  int fsh2 = fsh;
  if (mode == kModeWide) {
    const uint32_t cmax = __reduce_max_sync(0xFFFFFFFFu, lane < C ? s.c_mx[lane] : 0u);
    const uint32_t span = cmax - thr_key;
    while ((span >> fsh2) >= static_cast<uint32_t>(kTrack)) ++fsh2;
  }
  // the winners (bins above t, and t when taken whole) and bin t entries of the
  // CTAs before this one: one packed sum of their bins up to t and in t, and one
  // of their candidates
  int ow = 0, os = 0;
  if (mode == kModeSelect) {
    for (int c = 0; c < me; ++c) {
      const int2 v = *reinterpret_cast<const int2*>(cluster_fc(s, c) + 2 * lane);
      below += (2 * lane <= jt ? v.x : 0) + (2 * lane + 1 <= jt ? v.y : 0) +
               (((2 * lane == jt ? v.x : 0) + (2 * lane + 1 == jt ? v.y : 0)) << 16);
    }
    const uint32_t bsum = __reduce_add_sync(0xFFFFFFFFu, static_cast<uint32_t>(below));
    const int n_before = static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, lane < me ? word_l & 0xFFFFFFu : 0u));
    const int bt = static_cast<int>(bsum >> 16);
    ow = n_before - static_cast<int>(bsum & 0xFFFFu) + (all_t ? bt : 0);
    os = all_t ? 0 : bt;
  }
  if (lane == 0) {
    s.c_dec[0] = mode;
    s.c_dec[1] = jt;
    s.c_dec[2] = all_t ? 0 : need;
    s.c_dec[3] = in_t;
    s.c_dec[4] = fsh2;
    s.c_dec[5] = ow;
    s.c_dec[6] = os;
  }
}

// Warp 0: this CTA's fine-bin counts (s.ftot) into every CTA of
// the cluster, and with `all` its candidate count, flags and largest key.
__device__ __forceinline__ void cluster_push_counts(SmemC& s, int C, int me, bool all, int n_c, int flags,
                                                    uint32_t cmax) {
  const int lane = static_cast<int>(lane_id());
  const int2 v = *reinterpret_cast<const int2*>(&s.ftot[2 * lane]);
  // the count word: candidates (saturated at 2^20: more overflow the regions
  // anyway) in bits 0..23, 1 in bit 24 for an overflow and in bit 28 for a CTA
  // that gave up, so that a sum over 8 CTAs keeps every field apart
  const uint32_t word = static_cast<uint32_t>(min(n_c, 1 << 20)) | ((flags & 1) ? 1u << 24 : 0u) |
                        ((flags & 2) ? 1u << 28 : 0u);
  for (int c = 0; c < C; ++c) {
    const uint32_t a = dsmem_addr(cluster_fc(s, me) + 2 * lane, static_cast<uint32_t>(c));
    dsmem_st(a, static_cast<uint32_t>(v.x));
    dsmem_st(a + 4u, static_cast<uint32_t>(v.y));
    if (all && lane == 0) {
      dsmem_st(dsmem_addr(&s.c_nc[me], static_cast<uint32_t>(c)), word);
      dsmem_st(dsmem_addr(&s.c_mx[me], static_cast<uint32_t>(c)), cmax);
    }
  }
}

// Ranks bin t's in_t entries (s.rk, s.ri) and writes the first `need` of them
// at o[K - need ...]: at once up to kRankDirect entries; more are first split
// on the next 8 bits of key - thr_key (shift fsh - 8), the sub-bins above the
// one holding the need-th taken whole and that one ranked. Block-wide; uses
// s.hsub (zero on entry), s.n_win, s.n_bt and the candidate slots.
__device__ __forceinline__ void finish_bin_t(Smem& s, int in_t, int need, uint32_t thr_key, int fsh, int32_t* o,
                                             int K) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = static_cast<int>(lane_id());
  const int c4 = (in_t + 3) & ~3;
  if (tid >= in_t && tid < c4) {  // padding never beats a real entry
    s.rk[tid] = 0u;
    s.ri[tid] = 0x7FFFFFFF;
  }
  __syncthreads();
  if (in_t <= kRankDirect) {
    rank_out(s.rk, s.ri, in_t, c4, need, o + (K - need));
    return;
  }
  if (tid < in_t) atomicAdd(&s.hsub[((s.rk[tid] - thr_key) >> (fsh - 8)) & 0xFFu], 1u);
  __syncthreads();
  if (warp == 0) {
    int above_b;
    const int b = warp_find256(s.hsub, need, above_b);
    if (lane == 0) {
      s.sub_b = b;
      s.sub_above = above_b;
      s.n_win = 0;
      s.n_bt = 0;
    }
  }
  __syncthreads();
  const int b = s.sub_b;
  const int sab = s.sub_above;
  const int in_b = static_cast<int>(s.hsub[b]);
  if (tid < in_t) {
    const uint32_t kj = s.rk[tid];
    const int32_t ij = s.ri[tid];
    const int d = static_cast<int>(((kj - thr_key) >> (fsh - 8)) & 0xFFu);
    if (d > b) {
      o[K - need + atomicAdd(&s.n_win, 1)] = ij;
    } else if (d == b) {
      const int at = atomicAdd(&s.n_bt, 1);
      s.ckey[at] = kj;
      s.cidx[at] = ij;
    }
  }
  const int c4b = (in_b + 3) & ~3;
  if (tid >= in_b && tid < c4b) {
    s.ckey[tid] = 0u;
    s.cidx[tid] = 0x7FFFFFFF;
  }
  __syncthreads();
  rank_out(s.ckey, s.cidx, in_b, c4b, need - sab, o + (K - need + sab));
}

__global__ void __launch_bounds__(kThreads, 1) topk_short_cluster_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  SmemC& s = *reinterpret_cast<SmemC*>(smem_raw);
  const int tid = threadIdx.x;
  const int lane = static_cast<int>(lane_id());
  const int warp = tid >> 5;
  const uint32_t lt = lanemask_lt();
  const int K = p.topk;
  const int C = p.G;
  const int me = static_cast<int>(cluster_rank());
  const int64_t r = blockIdx.x / C;
  if (r >= p.num_rows) return;  // the whole cluster: its CTAs share the row
  wait_previous_grid();

  // Set-up: this CTA's first kBlind pieces of the blind window (sized by
  // max_len) go out before the length is read, local piece 0 first and the
  // rest (by warp 1) after the barrier, followed by the row's own pieces up to a
  // ring's worth; local piece i (window piece me + C i) sits in slot i % kRing.
  // A CTA other than 0 also fetches window piece 0 (the seed sample) into its
  // last slot, so that every CTA finds the same threshold from the same bytes
  // without waiting for CTA 0; its own piece kRing - 1 follows once the seed
  // is read.
  const int32_t len_raw = __ldg(p.lengths + r);
  const Win wmax = make_win(p, r, static_cast<int>(p.max_len));
  const int blind = min(wmax.np > me ? (wmax.np - me + C - 1) / C : 0, kBlind);
  const int S = me == 0 ? 0 : kRing - 1;  // the seed sample's slot
  if (warp == 0) {
    if (lane < kRing) {
      mbar_init(&s.bar[lane], 1u);
      fence_mbar_init();
      s.pdone[lane] = 0;
      s.slot_issues[lane] = 0;
    }
    if (lane == 0) s.key_max = 0;
    if (lane == 0 && blind > 0) issue_piece(s, wmax, me, 0, false);
    if (lane == kRing - 1 && me != 0 && wmax.np > 0) issue_piece(s, wmax, 0, kRing - 1, false);
  }
  for (int b = tid; b < kBins; b += kThreads) s.hseed[b] = 0;
  for (int i = tid; i < kWarps * kTrack; i += kThreads) s.wbin[i / kTrack][i % kTrack] = 0;
  if (tid < 256) s.hsub[tid] = 0;
  if (tid < kTrack) s.ftot[tid] = 0;
  if (tid == 0) {
    s.n_win = 0;
    s.n_bt = 0;
    s.cmax = 0;
  }
  __syncthreads();
  const int len = clamp_len(p, len_raw, tid == 0 && me == 0);
  if (warp == 1 && lane >= 1 && lane < blind) issue_piece(s, wmax, me + C * lane, lane, false);
  const Win w = make_win(p, r, len);
  int32_t* o = p.out + r * static_cast<int64_t>(K);
  const int npl = w.np > me ? (w.np - me + C - 1) / C : 0;  // this CTA's pieces of the window
  const int first_slots = me == 0 ? kRing : kRing - 1;      // slots free before the seed is read
  if (warp == 1 && lane >= blind && lane < min(npl, first_slots)) issue_piece(s, w, me + C * lane, lane, false);
  bool aborted = false;
  bool drain = false;  // pieces may still be in flight at the end: wait for every slot's last copy
  if (w.nwin == 0) {
    // every CTA of the cluster reads the same length: none takes a cluster barrier
    if (me == 0)
      for (int j = tid; j < K; j += kThreads) o[j] = (j < len) ? j : -1;
    drain = me != 0 && wmax.np > 0;  // the seed sample's copy
  } else {
    // every CTA of the cluster is running once this barrier's phase completes:
    // a CTA waits on it before its first access to another CTA's shared memory
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // ---- seed (every CTA, from the same piece 0): its top 12 key bits, as one
    // CTA seeds a row
    const int n_seed = min(len, kSeed - w.mis);
    const float* seed = s.row + S * kPiece;
    int wc = 0;  // this warp's candidates
    int target = K;
    if (warp == 0 && n_seed < len) {
      const float mu = static_cast<float>(K) * static_cast<float>(n_seed) / static_cast<float>(len);
      target = max(1, static_cast<int>(ceilf(mu + 3.0f * sqrtf(mu) + 2.0f)));
    }
    target = min(target, n_seed);
    bool ok = piece_ready(s, S, 0u, p.timeout_ns);
    if (p.inject == 3 && blockIdx.x == 1) ok = false;  // test: CTA 1 of cluster 0 gives up
    const int seed_hi = min(kSeed, w.nwin);
    uint32_t kmax = 0;
    for (int i = tid; i < seed_hi; i += kThreads) {
      const int e = i - w.mis;
      if (e >= 0 && e < len) {
        const uint32_t key = fkey(seed[i]);
        kmax = max(kmax, key);
        atomicAdd(&s.hseed[key >> 20], 1u);
      }
    }
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
    if (lane == 0 && kmax) atomicMax(&s.key_max, kmax);
    uint32_t thr_key = 0;
    bool strict = false;  // crowded: the filter keeps keys above thr_key only
    if (sync_or(!ok)) {
      aborted = true;
    } else {
      if (warp == 0) {
        int t0, above0;
        warp_scan_down(s.hseed, static_cast<int>(s.key_max >> 20), target, t0, above0);
        const int c0 = static_cast<int>(s.hseed[t0]);
        const int need_in = target - above0;
        // crowded: the seed's projection over the row overflows the cluster's
        // candidate regions (heavy ties); wide: refine inside the seed bin when
        // its extra entries would crowd the CTAs' regions
        const int at_or_above = above0 + c0;
        const bool crowded = n_seed >= K && at_or_above >= K &&
                             static_cast<int64_t>(at_or_above) * len > (3ll * kCand / 4) * C * n_seed;
        const bool refine = !crowded && c0 - need_in > max(target / 4, 16) &&
                            static_cast<int64_t>(c0 - need_in) * len >
                                static_cast<int64_t>(kClusterRefineExcess) * C * n_seed;
        if (lane == 0) {
          s.target = target;
          s.t0 = t0;
          s.crowded = crowded ? 1 : 0;
          s.refine = refine ? 1 : 0;
          s.need_in = need_in;
          s.thr_key = static_cast<uint32_t>(t0) << 20;
        }
      }
      __syncthreads();
      if (s.refine) {
        const uint32_t t0 = static_cast<uint32_t>(s.t0);
        for (int i = tid; i < seed_hi; i += kThreads) {
          const int e = i - w.mis;
          if (e >= 0 && e < len) {
            const uint32_t key = fkey(seed[i]);
            if ((key >> 20) == t0) atomicAdd(&s.hsub[(key >> 12) & 0xFFu], 1u);
          }
        }
        __syncthreads();
        if (warp == 0) {
          int above_b;
          const int b = warp_find256(s.hsub, s.need_in, above_b);
          if (lane == 0) s.thr_key = (t0 << 20) | (static_cast<uint32_t>(b) << 12);
        }
        __syncthreads();
        if (tid < 256) s.hsub[tid] = 0;  // clear again for the ranking (read after later barriers)
      }
      thr_key = s.thr_key;
      target = s.target;
      strict = s.crowded != 0;
      if (strict) {
        // the seed's K-th key T, exactly (every thread gets it); CTA 0, which
        // owns piece 0, also takes the seed's ties as its candidates
        if (me == 0) {
          thr_key = crowded_seed(s, 0, w.mis, n_seed, len, K, wc);
        } else {
          int need_t, equal_t;
          thr_key = exact_kth(s, Src{nullptr, 1, S * (kPiece / 4), len}, w.mis, n_seed, K, need_t, equal_t);
        }
      }
      __syncthreads();  // the seed sample is read: its slot takes the CTA's own piece kRing - 1
      if (me != 0 && tid == 0 && npl > kRing - 1) issue_piece(s, w, me + C * (kRing - 1), kRing - 1, true);
    }
    const bool seed_ok = !aborted;
    const float thr = key_floor_value(strict ? thr_key + 1u : thr_key);
    const int base = warp * kRegion;
    int* my_bins = s.wbin[warp];
    uint32_t kmx = 0;  // this lane's largest candidate key
    if (seed_ok) {
      // ---- filter this CTA's pieces: tasks of 128 F window elements, F chosen as
      // one CTA chooses it for its share; lane l takes float4s l, l + 32, ... of a
      // task. Local piece i hands its slot to local piece i + kRing once its
      // tasks are done. The task body is the whole-row kernel's, written out
      // again: one inline helper for both measured 0.9% slower on prefill (the
      // 32-warp whole-row kernel sits at its 64-register limit).
      const int nvec = w.nwin >> 2;
      int F = 8;
      while (F > 1 && (static_cast<int64_t>(128 * F) * target > static_cast<int64_t>(kTaskSurvivors) * n_seed ||
                       npl * kPiece < kMinTasks * 128 * F))
        F >>= 1;
      const int tsz = 128 * F;
      const int tpp = kPiece / tsz;  // tasks per piece
      int ntask = 0;
      if (npl > 0) {
        const int j_last = me + C * (npl - 1);
        const int size_last = min(kPiece, w.nwin - j_last * kPiece);  // only the window's last piece is short
        ntask = (npl - 1) * tpp + (size_last + tsz - 1) / tsz;
      }
#pragma unroll 1
      for (int task = warp; task < ntask; task += kWarps) {
        const int jl = task / tpp;             // local piece
        const int j = me + C * jl;             // window piece
        const int q = jl % kRing;              // its slot
        // the slot's copies so far: earlier local pieces in it, and (CTAs other
        // than 0, last slot) the seed sample before them
        const uint32_t phase = static_cast<uint32_t>(jl / kRing + ((me != 0 && q == kRing - 1) ? 1 : 0));
        if (!piece_ready(s, q, phase & 1u, p.timeout_ns)) {
          ok = false;
          break;
        }
        const int off = (task % tpp) * tsz;  // the task's first element in the piece
        const int sb = q * kPiece + off;
        const int v0 = (j * kPiece + off) >> 2;  // its first float4 in the window
        uint32_t m = 0;
        if (v0 + 32 * F <= nvec && 4 * v0 - w.mis >= 0 && 4 * v0 + tsz - w.mis <= len) {
          if (F == 8) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 f = *reinterpret_cast<const float4*>(&s.row[sb + 4 * (lane + 32 * i)]);
              m |= ((f.x >= thr ? 1u : 0u) | (f.y >= thr ? 2u : 0u) | (f.z >= thr ? 4u : 0u) |
                    (f.w >= thr ? 8u : 0u)) << (4 * i);
            }
          } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (i < F) {
              const float4 f = *reinterpret_cast<const float4*>(&s.row[sb + 4 * (lane + 32 * i)]);
              m |= ((f.x >= thr ? 1u : 0u) | (f.y >= thr ? 2u : 0u) | (f.z >= thr ? 4u : 0u) |
                    (f.w >= thr ? 8u : 0u)) << (4 * i);
            }
          }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int v = v0 + lane + 32 * i;
            if (i < F && v < nvec) {
              const float4 f = *reinterpret_cast<const float4*>(&s.row[sb + 4 * (lane + 32 * i)]);
              uint32_t b = (f.x >= thr ? 1u : 0u) | (f.y >= thr ? 2u : 0u) | (f.z >= thr ? 4u : 0u) |
                           (f.w >= thr ? 8u : 0u);
              const int e0 = 4 * v - w.mis;
#pragma unroll
              for (int c = 0; c < 4; ++c)
                if (e0 + c < 0 || e0 + c >= len) b &= ~(1u << c);
              m |= b << (4 * i);
            }
          }
        }
        const int c = __popc(m);
        // the warp's survivors and this lane's exclusive prefix, one ballot per bit of
        // the lanes' counts: bits 0..2 always, bits 3..5 only when a lane has 8 or
        // more (rare: the threshold keeps a few percent of the elements)
        int tot = 0, pre = 0;
#pragma unroll
        for (int bit = 0; bit < 3; ++bit) {
          const uint32_t qb = __ballot_sync(0xFFFFFFFFu, (c >> bit) & 1);
          tot += __popc(qb) << bit;
          pre += __popc(qb & lt) << bit;
        }
        if (__any_sync(0xFFFFFFFFu, c >= 8)) {
#pragma unroll
          for (int bit = 3; bit < 6; ++bit) {
            const uint32_t qb = __ballot_sync(0xFFFFFFFFu, (c >> bit) & 1);
            tot += __popc(qb) << bit;
            pre += __popc(qb & lt) << bit;
          }
        }
        if (tot > 0) {
          if (wc + tot <= kRegion) {
            int at = base + wc + pre;
            while (m) {
              const int jb = __ffs(m) - 1;
              m &= m - 1;
              s.cidx[at++] = 4 * (lane + 32 * (jb >> 2)) + (jb & 3);
            }
            __syncwarp();
#pragma unroll 1
            for (int e0 = 0; e0 < tot; e0 += 32) {
              const int e = e0 + lane;
              if (e < tot) {
                const int pos = s.cidx[base + wc + e];
                const uint32_t key = fkey(s.row[sb + pos]);
                kmx = max(kmx, key);
                s.ckey[base + wc + e] = key;
                s.cidx[base + wc + e] = j * kPiece + off + pos - w.mis;
                const uint32_t d = (key - thr_key) >> kFine;
                if (d < kTrack) atomicAdd(&my_bins[d], 1);
              }
            }
            __syncwarp();
          }
          wc += tot;
        }
        if (jl + kRing < npl) {
          __syncwarp();  // every lane's reads of the slot come before the hand-over
          if (lane == 0 && atom_add_acq_rel_cta(&s.pdone[q], 1) == tpp - 1) {
            s.pdone[q] = 0;
            issue_piece(s, w, me + C * (jl + kRing), q, true);
          }
        }
      }
    }
    if (lane == 0) s.wcnt[warp] = wc;
    if (wc > 0) {
      const int2 v2 = *reinterpret_cast<const int2*>(&my_bins[2 * lane]);
      if (v2.x) atomicAdd(&s.ftot[2 * lane], v2.x);
      if (v2.y) atomicAdd(&s.ftot[2 * lane + 1], v2.y);
    }
    kmx = __reduce_max_sync(0xFFFFFFFFu, kmx);
    if (lane == 0 && kmx) atomicMax(&s.cmax, kmx);
    if (sync_or(!ok)) aborted = true;
    // ---- this CTA's counts into every CTA of the cluster (warp 0; lane l: warp l's
    // count, fine bins 2l and 2l + 1); then each CTA finds bin t on its own. The
    // start-up phase of the cluster barrier completes first: every CTA runs.
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (warp == 0) {
      const int n_l = lane < kWarps ? s.wcnt[lane] : 0;
      const bool over = __any_sync(0xFFFFFFFFu, n_l > kRegion);
      const int n_c = static_cast<int>(__reduce_add_sync(0xFFFFFFFFu, static_cast<uint32_t>(n_l)));
      cluster_push_counts(s, C, me, true, n_c, (over ? 1 : 0) | (aborted ? 2 : 0), s.cmax);
    }
    cluster_sync_all();  // every CTA's counts are in every CTA
    if (warp == 0) cluster_decide(s, K, C, me, kFine, true, thr_key);
    __syncthreads();
    int mode = s.c_dec[0];
    int fsh = kFine;  // fine bin of a candidate: (key - thr_key) >> fsh
    if (mode == kModeWide) {
      // the K-th key lies above the 64 bins counted: every CTA counts its
      // candidates again in bins wide enough for the cluster's largest key
      fsh = s.c_dec[4];
      const int cnt_w = s.wcnt[warp];  // at most kRegion: no overflow here
      *reinterpret_cast<int2*>(&my_bins[2 * lane]) = make_int2(0, 0);
      if (tid < kTrack) s.ftot[tid] = 0;
      __syncthreads();
      for (int e = lane; e < cnt_w; e += 32) atomicAdd(&my_bins[(s.ckey[base + e] - thr_key) >> fsh], 1);
      __syncwarp();
      if (cnt_w > 0) {
        const int2 v2 = *reinterpret_cast<const int2*>(&my_bins[2 * lane]);
        if (v2.x) atomicAdd(&s.ftot[2 * lane], v2.x);
        if (v2.y) atomicAdd(&s.ftot[2 * lane + 1], v2.y);
      }
      cluster_sync_all();  // every CTA has read the first counts: they may be overwritten
      if (warp == 0) cluster_push_counts(s, C, me, false, 0, 0, 0u);
      cluster_sync_all();  // every CTA's recount is in every CTA
      if (warp == 0) cluster_decide(s, K, C, me, fsh, false, thr_key);
      __syncthreads();
      mode = s.c_dec[0];
    }
    const int jt = s.c_dec[1];
    const int need = s.c_dec[2];
    const bool all_t = need == 0;
    if (mode == kModeSelect) {
      // ---- winners above bin t out, bin t's entries into rank 0's ranking slots,
      // each CTA from the first slots the decision gave it
      const int cnt = s.wcnt[warp];  // at most kRegion here
      const int2 b2 = *reinterpret_cast<const int2*>(&my_bins[2 * lane]);
      const int below = static_cast<int>(__reduce_add_sync(
          0xFFFFFFFFu, static_cast<uint32_t>((2 * lane <= jt ? b2.x : 0) + (2 * lane + 1 <= jt ? b2.y : 0))));
      int bt = my_bins[jt];
      int nw = cnt - below;
      if (all_t) {
        nw += bt;
        bt = 0;
      }
      // this CTA's output range and ranking slots start where the decision put them
      int ow = 0, os = 0;
      if (lane == 0) {
        if (nw) ow = atomicAdd(&s.n_win, nw);
        if (bt) os = atomicAdd(&s.n_bt, bt);
      }
      ow = s.c_dec[5] + __shfl_sync(0xFFFFFFFFu, ow, 0);
      os = s.c_dec[6] + __shfl_sync(0xFFFFFFFFu, os, 0);
      const uint32_t rk0 = dsmem_addr(&s.rk[0], 0u);
      const uint32_t ri0 = dsmem_addr(&s.ri[0], 0u);
#pragma unroll 1
      for (int e0 = 0; e0 < cnt; e0 += 32) {
        const int e = e0 + lane;
        uint32_t key = 0;
        int32_t idx = 0;
        int d = -1;
        if (e < cnt) {
          key = s.ckey[base + e];
          idx = s.cidx[base + e];
          d = static_cast<int>((key - thr_key) >> fsh);
        }
        const bool win = d > jt || (all_t && d == jt);
        const bool inb = !all_t && d == jt;
        const uint32_t bw = __ballot_sync(0xFFFFFFFFu, win);
        if (win) o[ow + __popc(bw & lt)] = idx;
        ow += __popc(bw);
        const uint32_t bb = __ballot_sync(0xFFFFFFFFu, inb);
        if (inb) {
          const uint32_t at = static_cast<uint32_t>(os + __popc(bb & lt));
          dsmem_st(rk0 + 4u * at, key);
          dsmem_st(ri0 + 4u * at, static_cast<uint32_t>(idx));
        }
        os += __popc(bb);
      }
    }
    cluster_sync_all();  // B4: bin t's entries are in rank 0; no CTA touches another's memory from here on
    if (me == 0) {
      if (mode == kModeSelect && !all_t)
        finish_bin_t(s, s.c_dec[3], need, thr_key, fsh, o, K);
      else if (mode == kModeExact)
        fallback_select(s, p, r, w, Src{w.rowp - w.mis, 1, -1, len});
    }
  }
  // the blind pieces past this CTA's share land before it leaves (lane q: slot q)
  drain = drain || aborted;
  if (!drain && warp == 0 && lane >= npl && lane < blind) wait_piece(&s.bar[lane], 0u, p.timeout_ns, nullptr);
  if (drain && tid == 0) {
    // a piece did not land in time (flagged), or the seed's did not: wait
    // (bounded) for the last copy issued into every slot before the CTA leaves
    if (aborted) atomicOr(p.status, 0x4u);
    for (int q = 0; q < kRing; ++q) {
      const int n = s.slot_issues[q];
      if (n > 0) wait_piece(&s.bar[q], static_cast<uint32_t>(n - 1) & 1u, p.timeout_ns, nullptr);
    }
  }
}

// ---------------------------------------------------------------- host side

int kernel_threads() { return kThreads; }

size_t kernel_smem_bytes() { return sizeof(Smem); }

cudaError_t kernel_configure() {
  const cudaError_t e = cudaFuncSetAttribute(topk_short_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(sizeof(Smem)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(topk_short_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(SmemC)));
}

cudaError_t kernel_occupancy(int* ctas_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, topk_short_kernel, kThreads, sizeof(Smem));
}

// Clusters of `cluster_size` CTAs of the cluster kernel that can be resident at once.
cudaError_t kernel_max_clusters(int cluster_size, int* clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster_size));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(SmemC);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_size);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, topk_short_cluster_kernel, &cfg);
}

// G = 1: the whole-row kernel over `grid` persistent CTAs. G > 1 (contiguous
// rows only): the cluster kernel, clusters of G CTAs, one row each (grid =
// num_rows * G).
cudaError_t launch_topk(const Params& p, int grid, bool, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (p.dependent_launch) {
    // may start while the previous kernel on the stream finishes (the kernel
    // waits for it before touching global memory)
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
  if (p.G <= 1) {
    cfg.dynamicSmemBytes = sizeof(Smem);
    return cudaLaunchKernelEx(&cfg, topk_short_kernel, p);
  }
  if (p.G > kMaxCluster || p.col_stride != 1 || grid % p.G != 0) return cudaErrorInvalidValue;
  cfg.dynamicSmemBytes = sizeof(SmemC);
  attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
  attr[cfg.numAttrs].val.clusterDim.x = static_cast<unsigned>(p.G);
  attr[cfg.numAttrs].val.clusterDim.y = 1;
  attr[cfg.numAttrs].val.clusterDim.z = 1;
  ++cfg.numAttrs;
  return cudaLaunchKernelEx(&cfg, topk_short_cluster_kernel, p);
}

}  // namespace LTK_SHORT_NS
}  // namespace ltk
