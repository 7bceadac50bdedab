// Ragged per-row top-K for sm_103a: streaming filter + radix select.
//
// One kernel serves every row length. A CTA (or a group of G CTAs that split
// one row) streams its part of the row from HBM through a ring of shared-memory
// slots filled by bulk asynchronous copies (cp.async.bulk, completion counted
// on an mbarrier). While streaming it keeps a 12-bit histogram of the keys it
// has kept and a running threshold bin: once K kept keys sit at or above a bin,
// every later key below that bin can never be selected and is dropped at once.
// Only the survivors are written to a shared-memory candidate buffer, so each
// logit is read from HBM exactly once and most of them cost a compare.
//
// At the end of the row the candidates go through an exact radix select on the
// composite key (value bits, then inverted index bits), which settles ties by
// the smaller index. When G > 1 the CTAs of a group merge their histograms
// through a workspace in global memory, meeting at a group barrier after each
// radix pass; this replaces the per-row RadixRowState of the persistent_topk
// kernel (vLLM PR #41444 page, "Executive summary": arrival counter plus
// histogram per row group). Every workspace word a launch touches is returned
// to zero before the launch ends, with the fencing that the vLLM PR #41748
// page's review asks for ("Code Review": zero in parallel, and reset the
// arrival counter only after the zeros are visible), so no per-call memset is
// needed and graph replays start from a clean workspace.
//
// Keys: an fp32 value x maps to a uint32 whose unsigned order is the order of
// the values: -0.0 is first mapped to +0.0, then positive values get the sign
// bit set and negative values are bit-inverted.

#include <cuda_runtime.h>
#include <stdint.h>

#include "topk_internal.h"

namespace ltk {

struct __align__(128) Smem {
  float stage[kStages][kChunk];   // staging ring (bulk-copy destination)
  uint32_t hist[kBins];           // histogram of kept keys (also radix scratch)
  uint32_t bkey[kBufCap];         // candidate keys
  int32_t bidx[kBufCap];          // candidate indices (row-relative)
  uint16_t listA[kBufCap];        // candidate positions, ping
  uint16_t listB[kBufCap];        // candidate positions, pong
  uint16_t emit[kMaxTopK];        // positions selected for output
  unsigned long long full[kStages];
  int32_t lens[kLenCache];
  uint32_t wtot[kWarps];
  int g_e[kMaxGroup];
  int g_tot[kMaxGroup];
  int buf_n, buf_mark, n_emit, nA, nB;
  int t, cnt_ge;
  uint32_t thr_lo;
  int find_b, find_gt;
  int abort, last, off, take;
  uint32_t min_key;
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

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              unsigned long long* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
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

// Waits for an mbarrier phase, giving up after timeout_ns.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long* bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
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

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

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

// Radix digit of the composite key (key, ~index) at a level:
// 0: key 31..20, 1: key 19..8, 2: key 7..0, 3: ~idx 31..20, 4: ~idx 19..8, 5: ~idx 7..0.
__device__ __forceinline__ uint32_t digit_of(int level, uint32_t key, int32_t idx) {
  const uint32_t v = (level < 3) ? key : ~static_cast<uint32_t>(idx);
  const int l = (level < 3) ? level : level - 3;
  return (l == 0) ? (v >> 20) : (l == 1) ? ((v >> 8) & 0xFFFu) : (v & 0xFFu);
}

__device__ __forceinline__ int level_bins(int level) { return (level == 2 || level == 5) ? 256 : kBins; }

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

// Finds the largest bin b of s.hist[0, nb) with sum(hist[b:]) >= need (need >= 1
// and the total must reach need). Writes b to s.find_b and sum(hist[b+1:]) to
// s.find_gt. Block-wide; ends with a barrier.
__device__ void block_find(Smem& s, int nb, int need) {
  const int tid = threadIdx.x;
  const int per = (nb + kThreads - 1) / kThreads;
  const int nact = nb / per;
  const int lo = tid * per;
  if (tid == 0) {
    s.find_b = 0;
    s.find_gt = 0;
  }
  uint32_t sum = 0;
  if (tid < nact)
    for (int j = 0; j < per; ++j) sum += s.hist[lo + j];
  uint32_t suf = sum;  // suffix sum within the warp (lanes at and above this one)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xFFFFFFFFu, suf, o);
    if (lane_id() + o < 32) suf += v;
  }
  const int warp = tid >> 5;
  if (lane_id() == 0) s.wtot[warp] = suf;
  __syncthreads();
  uint32_t above = 0;
  for (int w = warp + 1; w < kWarps; ++w) above += s.wtot[w];
  const uint32_t incl = suf + above;  // sum of bins >= lo
  const uint32_t excl = incl - sum;   // sum of bins >= lo + per
  if (tid < nact && incl >= static_cast<uint32_t>(need) && excl < static_cast<uint32_t>(need)) {
    uint32_t run = excl;
    for (int j = per - 1; j >= 0; --j) {
      const uint32_t h = s.hist[lo + j];
      if (run + h >= static_cast<uint32_t>(need)) {
        s.find_b = lo + j;
        s.find_gt = static_cast<int>(run);
        break;
      }
      run += h;
    }
  }
  __syncthreads();
}

// Candidates at s.listX positions: emits those whose digit is above b and moves
// those equal to b into dst. Warp-uniform loop; no barrier.
__device__ void partition_list(Smem& s, const uint16_t* src, int n, int level, uint32_t b,
                               uint16_t* dst, int* dst_n) {
  const int warp = threadIdx.x >> 5;
  for (int base = warp * 32; base < n; base += kThreads) {
    const int i = base + static_cast<int>(lane_id());
    const bool in = i < n;
    const uint16_t pos = in ? src[i] : static_cast<uint16_t>(0);
    const uint32_t d = in ? digit_of(level, s.bkey[pos], s.bidx[pos]) : 0u;
    warp_push<uint16_t>(s.emit, &s.n_emit, kMaxTopK, in && d > b, pos);
    warp_push<uint16_t>(dst, dst_n, kBufCap, in && d == b, pos);
  }
}

// Buffer entries: emits those with key bits 31..20 above b, lists those equal to b.
__device__ void partition_buffer(Smem& s, uint32_t b) {
  const int warp = threadIdx.x >> 5;
  const int n = s.buf_n;
  for (int base = warp * 32; base < n; base += kThreads) {
    const int i = base + static_cast<int>(lane_id());
    const bool in = i < n;
    const uint32_t d = in ? (s.bkey[i] >> 20) : 0u;
    warp_push<uint16_t>(s.emit, &s.n_emit, kMaxTopK, in && d > b, static_cast<uint16_t>(i));
    warp_push<uint16_t>(s.listA, &s.nA, kBufCap, in && d == b, static_cast<uint16_t>(i));
  }
}

// Emits exactly `need` positions of A (all sharing the digits of the levels
// before `level`): the best ones under (key desc, index asc). Uses s.hist as
// scratch. Block-wide; ends with a barrier.
__device__ void select_exact(Smem& s, uint16_t* A, uint16_t* B, int nA, int need, int level) {
  const int tid = threadIdx.x;
  while (need > 0) {
    if (need >= nA) {
      for (int base = (tid >> 5) * 32; base < nA; base += kThreads) {
        const int i = base + static_cast<int>(lane_id());
        warp_push<uint16_t>(s.emit, &s.n_emit, kMaxTopK, i < nA, i < nA ? A[i] : static_cast<uint16_t>(0));
      }
      break;
    }
    if (nA <= 32 || level > 5) {
      // Direct ranking inside one warp; composite keys are distinct, so exactly
      // `need` lanes have rank < need. (level > 5 cannot happen with distinct
      // composite keys; it is kept as a terminating case.)
      if (tid < 32) {
        const int lane = static_cast<int>(lane_id());
        const bool in = lane < nA;
        const uint16_t pos = in ? A[lane] : static_cast<uint16_t>(0);
        const uint32_t hi = in ? s.bkey[pos] : 0u;
        const uint32_t lo = in ? ~static_cast<uint32_t>(s.bidx[pos]) : 0u;
        int rank = 0;
        const int lim = nA < 32 ? nA : 32;
        for (int j = 0; j < lim; ++j) {
          const uint32_t h2 = __shfl_sync(0xFFFFFFFFu, hi, j);
          const uint32_t l2 = __shfl_sync(0xFFFFFFFFu, lo, j);
          rank += (h2 > hi || (h2 == hi && l2 > lo)) ? 1 : 0;
        }
        warp_push<uint16_t>(s.emit, &s.n_emit, kMaxTopK, in && rank < need, pos);
      }
      break;
    }
    const int nb = level_bins(level);
    for (int b = tid; b < nb; b += kThreads) s.hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < nA; i += kThreads) {
      const uint16_t pos = A[i];
      atomicAdd(&s.hist[digit_of(level, s.bkey[pos], s.bidx[pos])], 1u);
    }
    if (tid == 0) s.nB = 0;
    __syncthreads();
    block_find(s, nb, need);
    const uint32_t b = static_cast<uint32_t>(s.find_b);
    const int gt = s.find_gt;
    partition_list(s, A, nA, level, b, B, &s.nB);
    __syncthreads();
    need -= gt;
    nA = s.nB;
    uint16_t* tmp = A;
    A = B;
    B = tmp;
    ++level;
  }
  __syncthreads();
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
    s.n_emit = 0;
    s.nA = 0;
    s.nB = 0;
  }
}

// One warp: moves the threshold bin t up as far as the kept counts allow.
// cnt_ge counts buffered keys with bits 31..20 >= t (all of them are in play);
// after the move, at least K of them still sit at or above t and fewer than K
// above it.
__device__ void advance_threshold(Smem& s, int K) {
  const int lane = static_cast<int>(lane_id());
  int cnt = s.cnt_ge + (s.buf_n - s.buf_mark);
  int t = s.t;
  if (cnt >= K) {
    // fine step over 32 bins
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
    const uint32_t lo = static_cast<uint32_t>(t) << 20;
    if (lo > s.thr_lo) s.thr_lo = lo;
  }
}

// Drops buffered keys below bin t (they can no longer be selected).
__device__ void compact_to_bin(Smem& s) {
  constexpr int kPer = kBufCap / kThreads;
  const int tid = threadIdx.x;
  const int n = s.buf_n;
  const uint32_t tmin = static_cast<uint32_t>(s.t);
  uint32_t kk[kPer];
  int32_t ii[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = tid + j * kThreads;
    kk[j] = 0u;
    ii[j] = 0;
    if (e < n) {
      kk[j] = s.bkey[e];
      ii[j] = s.bidx[e];
    }
  }
  __syncthreads();
  if (tid == 0) s.buf_n = 0;
  __syncthreads();
  const uint32_t lt = lanemask_lt();
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = tid + j * kThreads;
    const bool keep = e < n && (kk[j] >> 20) >= tmin;
    const uint32_t m = __ballot_sync(0xFFFFFFFFu, keep);
    if (m) {
      int base = 0;
      if (lane_id() == 0) base = atomicAdd(&s.buf_n, __popc(m));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (keep) {
        const int o = base + __popc(m & lt);
        s.bkey[o] = kk[j];
        s.bidx[o] = ii[j];
      }
    }
  }
  __syncthreads();
  if (tid == 0) s.buf_mark = s.buf_n;
  __syncthreads();
}

// Keeps exactly the K best buffered candidates and raises the filter to
// (K-th key) + 1: a later element equal to that key has a larger index than
// every kept one, so it can never be selected.
__device__ void compact_exact(Smem& s, int K) {
  const int tid = threadIdx.x;
  const int t = s.t;
  const int need = K - (s.cnt_ge - static_cast<int>(s.hist[t]));
  if (tid == 0) {
    s.n_emit = 0;
    s.nA = 0;
    s.min_key = 0xFFFFFFFFu;
  }
  __syncthreads();
  partition_buffer(s, static_cast<uint32_t>(t));
  __syncthreads();
  select_exact(s, s.listA, s.listB, s.nA, need, 1);
  constexpr int kPer = kMaxTopK / kThreads;
  uint32_t kk[kPer];
  int32_t ii[kPer];
  uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = tid + j * kThreads;
    kk[j] = 0u;
    ii[j] = 0;
    if (e < K) {
      const int pos = s.emit[e] & (kBufCap - 1);
      kk[j] = s.bkey[pos];
      ii[j] = s.bidx[pos];
      mn = min(mn, kk[j]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
  if (lane_id() == 0) atomicMin(&s.min_key, mn);
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int e = tid + j * kThreads;
    if (e < K) {
      s.bkey[e] = kk[j];
      s.bidx[e] = ii[j];
      atomicAdd(&s.hist[kk[j] >> 20], 1u);
    }
  }
  if (tid == 0) {
    const uint32_t T = s.min_key;
    s.buf_n = K;
    s.buf_mark = K;
    s.cnt_ge = K;
    s.t = static_cast<int>(T >> 20);
    s.thr_lo = T + 1u;
    s.n_emit = 0;
  }
  __syncthreads();
}

// ----------------------------------------------------------------- row plans

struct RowWin {
  int64_t r;
  const float* rowp;
  int len, lo, hi, wstart, wend, nch;
};

__device__ __forceinline__ int clamp_len(const Params& p, int32_t raw) {
  if (raw < 0 || static_cast<int64_t>(raw) > p.stride) {
    atomicOr(p.status, 0x1u);
    return raw < 0 ? 0 : static_cast<int>(p.stride);
  }
  return raw;
}

__device__ __forceinline__ int row_len(const Params& p, const Smem& s, int64_t k, int64_t r) {
  if (k < kLenCache) return s.lens[k];
  return clamp_len(p, __ldg(p.lengths + r));
}

// Part of row k (of this CTA's group) that this CTA streams, and its copy windows.
__device__ __forceinline__ bool get_row(const Params& p, const Smem& s, int64_t k, int g, int m,
                                        RowWin& w) {
  w.r = g + k * p.num_groups;
  if (w.r >= p.num_rows) return false;
  w.len = row_len(p, s, k, w.r);
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
      // least one element of [lo, hi), so no copy leaves the row's pages
      const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(w.rowp + w.lo) & 15u) >> 2);
      w.wstart = w.lo - mis;
      w.wend = w.wstart + ((w.hi - w.wstart + 3) & ~3);
      w.nch = (w.wend - w.wstart + kChunk - 1) / kChunk;
    }
  }
  return true;
}

// Copy issuer state, held by thread 0.
struct Producer {
  int64_t k;
  RowWin w;
  int j;
  uint32_t q;  // sequence number of the next chunk to issue
  bool done;
};

__device__ void producer_seek(const Params& p, const Smem& s, Producer& P, int g, int m) {
  while (true) {
    if (!get_row(p, s, P.k, g, m, P.w)) {
      P.done = true;
      return;
    }
    if (P.w.nch > 0) {
      P.j = 0;
      return;
    }
    ++P.k;
  }
}

__device__ void producer_issue(const Params& p, Smem& s, Producer& P, int g, int m) {
  if (P.done) return;
  const int ws = P.w.wstart + P.j * kChunk;
  const int we = min(ws + kChunk, P.w.wend);
  const uint32_t bytes = static_cast<uint32_t>(we - ws) * 4u;
  const int slot = static_cast<int>(P.q % kStages);
  fence_proxy_async();
  mbar_expect_tx(&s.full[slot], bytes);
  bulk_copy_g2s(s.stage[slot], P.w.rowp + ws, bytes, &s.full[slot]);
  ++P.q;
  if (++P.j == P.w.nch) {
    ++P.k;
    producer_seek(p, s, P, g, m);
  }
}

// Waits (bounded) for every copy issued but not consumed, so that none lands
// after the CTA has left.
__device__ void drain_copies(Smem& s, const Producer& P, uint32_t consumed, uint64_t timeout_ns) {
  for (uint32_t q = consumed; q < P.q; ++q)
    mbar_wait_bounded(&s.full[q % kStages], (q / kStages) & 1u, timeout_ns);
}

// ------------------------------------------------------------- chunk filter

// Filters one staged chunk: keys at or above the running threshold are kept
// (appended to the candidate buffer and counted in the histogram).
__device__ __forceinline__ void filter_chunk(Smem& s, const float* stage, int ws, int nvec, int lo,
                                             int hi) {
  const int warp = threadIdx.x >> 5;
  const int lane = static_cast<int>(lane_id());
  const uint32_t thr = s.thr_lo;
  const bool interior = ws >= lo && ws + 4 * nvec <= hi;
  const float4* st4 = reinterpret_cast<const float4*>(stage);
  const uint32_t lt = lanemask_lt();
  for (int vb = warp * 32; vb < nvec; vb += kThreads) {
    const int v = vb + lane;
    const bool in = v < nvec;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (in) f = st4[v];
    const int i0 = ws + 4 * v;
    const uint32_t k0 = fkey(f.x), k1 = fkey(f.y), k2 = fkey(f.z), k3 = fkey(f.w);
    bool p0 = in && k0 >= thr, p1 = in && k1 >= thr, p2 = in && k2 >= thr, p3 = in && k3 >= thr;
    if (!interior) {
      p0 = p0 && i0 >= lo && i0 < hi;
      p1 = p1 && i0 + 1 >= lo && i0 + 1 < hi;
      p2 = p2 && i0 + 2 >= lo && i0 + 2 < hi;
      p3 = p3 && i0 + 3 >= lo && i0 + 3 < hi;
    }
    const uint32_t m0 = __ballot_sync(0xFFFFFFFFu, p0);
    const uint32_t m1 = __ballot_sync(0xFFFFFFFFu, p1);
    const uint32_t m2 = __ballot_sync(0xFFFFFFFFu, p2);
    const uint32_t m3 = __ballot_sync(0xFFFFFFFFu, p3);
    const int c0 = __popc(m0), c1 = __popc(m1), c2 = __popc(m2), c3 = __popc(m3);
    const int tot = c0 + c1 + c2 + c3;
    if (tot == 0) continue;
    int base = 0;
    if (lane == 0) base = atomicAdd(&s.buf_n, tot);
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (p0) {
      const int o = min(base + __popc(m0 & lt), kBufCap - 1);
      s.bkey[o] = k0;
      s.bidx[o] = i0;
      atomicAdd(&s.hist[k0 >> 20], 1u);
    }
    if (p1) {
      const int o = min(base + c0 + __popc(m1 & lt), kBufCap - 1);
      s.bkey[o] = k1;
      s.bidx[o] = i0 + 1;
      atomicAdd(&s.hist[k1 >> 20], 1u);
    }
    if (p2) {
      const int o = min(base + c0 + c1 + __popc(m2 & lt), kBufCap - 1);
      s.bkey[o] = k2;
      s.bidx[o] = i0 + 2;
      atomicAdd(&s.hist[k2 >> 20], 1u);
    }
    if (p3) {
      const int o = min(base + c0 + c1 + c2 + __popc(m3 & lt), kBufCap - 1);
      s.bkey[o] = k3;
      s.bidx[o] = i0 + 3;
      atomicAdd(&s.hist[k3 >> 20], 1u);
    }
  }
}

// ------------------------------------------------------------ row finishing

__device__ void write_trivial_row(const Params& p, int64_t r, int len) {
  int32_t* o = p.out + r * static_cast<int64_t>(p.topk);
  for (int j = threadIdx.x; j < p.topk; j += kThreads) o[j] = (j < len) ? j : -1;
}

// G == 1: the CTA holds every candidate of the row.
__device__ void finish_local(Smem& s, const Params& p, int64_t r) {
  const int K = p.topk;
  const int t = s.t;
  const int need = K - (s.cnt_ge - static_cast<int>(s.hist[t]));
  if (threadIdx.x == 0) {
    s.n_emit = 0;
    s.nA = 0;
  }
  __syncthreads();
  partition_buffer(s, static_cast<uint32_t>(t));
  __syncthreads();
  select_exact(s, s.listA, s.listB, s.nA, need, 1);
  int32_t* o = p.out + r * static_cast<int64_t>(K);
  for (int j = threadIdx.x; j < K; j += kThreads) o[j] = s.bidx[s.emit[j] & (kBufCap - 1)];
  __syncthreads();
  reset_row_state(s);
  __syncthreads();
}

// Group barrier over the workspace: arrive (release), then wait (acquire)
// until `target` arrivals, at most timeout_ns. Returns false if this CTA must
// abandon the launch (time-out, or the test-only injected departure).
__device__ bool group_sync(Smem& s, uint32_t* ctr, uint32_t target, const Params& p, bool skip) {
  __syncthreads();
  if (threadIdx.x == 0) {
    if (skip) {
      s.abort = 1;
    } else {
      __threadfence();
      atom_add_release_gpu(ctr, 1u);
      const uint64_t t0 = global_timer();
      uint32_t spins = 0;
      while (ld_acquire_gpu(ctr) < target) {
        if ((++spins & 63u) == 0 && global_timer() - t0 > p.timeout_ns) {
          s.abort = 1;
          atomicOr(p.status, 0x2u);
          break;
        }
      }
      __threadfence();
    }
  }
  __syncthreads();
  return s.abort == 0;
}

__device__ __forceinline__ void clear_slice(uint32_t* a, int n, int m, int G) {
  for (int i = m * kThreads + static_cast<int>(threadIdx.x); i < n; i += G * kThreads) __stcg(a + i, 0u);
}

// G > 1: three radix passes whose histograms are merged across the group.
__device__ bool finish_group(Smem& s, const Params& p, int64_t r, int g, int m, uint32_t& epoch,
                             bool& first_barrier) {
  const int tid = threadIdx.x;
  const int K = p.topk;
  const int G = p.G;
  GroupWs* gw = p.groups + g;
  const bool skip = (p.inject == 1) && g == 0 && m == 1 && first_barrier;
  first_barrier = false;

  // pass A: bits 31..20 of every member's candidates still in play
  for (int b = s.t + tid; b < kBins; b += kThreads) {
    const uint32_t h = s.hist[b];
    if (h) atomicAdd(&gw->h1[b], h);
  }
  epoch += G;
  if (!group_sync(s, &gw->bar_count, epoch, p, skip)) return false;
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = __ldcg(&gw->h1[b]);
  if (tid == 0) {
    s.n_emit = 0;
    s.nA = 0;
  }
  __syncthreads();
  block_find(s, kBins, K);
  const uint32_t T1 = static_cast<uint32_t>(s.find_b);
  const int needA = K - s.find_gt;
  partition_buffer(s, T1);
  __syncthreads();
  const int gtA = s.n_emit;
  const int nA = s.nA;

  // pass B: bits 19..8 of the candidates in bin T1
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = 0;
  __syncthreads();
  for (int i = tid; i < nA; i += kThreads) {
    const uint16_t pos = s.listA[i];
    atomicAdd(&s.hist[digit_of(1, s.bkey[pos], 0)], 1u);
  }
  __syncthreads();
  for (int b = tid; b < kBins; b += kThreads) {
    const uint32_t h = s.hist[b];
    if (h) atomicAdd(&gw->h2[b], h);
  }
  epoch += G;
  if (!group_sync(s, &gw->bar_count, epoch, p, false)) return false;
  clear_slice(gw->h1, kBins, m, G);  // every member read h1 before arriving here
  for (int b = tid; b < kBins; b += kThreads) s.hist[b] = __ldcg(&gw->h2[b]);
  if (tid == 0) s.nB = 0;
  __syncthreads();
  block_find(s, kBins, needA);
  const uint32_t T2 = static_cast<uint32_t>(s.find_b);
  const int needB = needA - s.find_gt;
  partition_list(s, s.listA, nA, 1, T2, s.listB, &s.nB);
  __syncthreads();
  const int gtB = s.n_emit - gtA;
  const int nB = s.nB;

  // pass C: bits 7..0, histogram kept per member so ties can be ranked by member
  for (int b = tid; b < 256; b += kThreads) s.hist[b] = 0;
  __syncthreads();
  for (int i = tid; i < nB; i += kThreads) {
    const uint16_t pos = s.listB[i];
    atomicAdd(&s.hist[s.bkey[pos] & 0xFFu], 1u);
  }
  __syncthreads();
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
  __syncthreads();
  block_find(s, 256, needB);
  const uint32_t T3 = static_cast<uint32_t>(s.find_b) & 0xFFu;
  const int needC = needB - s.find_gt;
  if (tid < G) {
    const int mm = tid;
    uint32_t gtc = 0;
    for (int b = static_cast<int>(T3) + 1; b < 256; ++b) gtc += __ldcg(&gw->h3[mm][b]);
    s.g_e[mm] = static_cast<int>(__ldcg(&gw->h3[mm][T3]));
    s.g_tot[mm] = static_cast<int>(__ldcg(&gw->cnt[mm][0]) + __ldcg(&gw->cnt[mm][1]) + gtc);
  }
  __syncthreads();
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
    s.nA = 0;
  }
  __syncthreads();
  partition_list(s, s.listB, nB, 2, T3, s.listA, &s.nA);
  __syncthreads();
  select_exact(s, s.listA, s.listB, s.nA, s.take, 3);
  const int off = s.off;
  const int ne = min(s.n_emit, kMaxTopK);
  int32_t* o = p.out + r * static_cast<int64_t>(K);
  for (int j = tid; j < ne; j += kThreads)
    if (off + j < K) o[off + j] = s.bidx[s.emit[j] & (kBufCap - 1)];
  __syncthreads();
  reset_row_state(s);
  __syncthreads();
  return true;
}

// ------------------------------------------------------------------- kernel

__global__ void __launch_bounds__(kThreads, 1) topk_ragged_kernel(const Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x;
  const int g = static_cast<int>(blockIdx.x) / p.G;
  const int m = static_cast<int>(blockIdx.x) % p.G;

  reset_row_state(s);
  if (tid == 0) {
    s.abort = 0;
    for (int i = 0; i < kStages; ++i) mbar_init(&s.full[i], 1u);
    fence_mbar_init();
  }
  for (int k = tid; k < kLenCache; k += kThreads) {
    const int64_t r = g + static_cast<int64_t>(k) * p.num_groups;
    s.lens[k] = (r < p.num_rows) ? clamp_len(p, p.lengths[r]) : 0;
  }
  __syncthreads();

  Producer P;
  P.k = 0;
  P.q = 0;
  P.j = 0;
  P.done = false;
  if (tid == 0) {
    producer_seek(p, s, P, g, m);
    for (int i = 0; i < kStages; ++i) producer_issue(p, s, P, g, m);
  }

  uint32_t q = 0;  // chunks consumed
  uint32_t epoch = 0;
  bool first_barrier = true;
  bool aborted = false;
  RowWin w;
  for (int64_t k = 0; !aborted && get_row(p, s, k, g, m, w); ++k) {
    if (w.len <= p.topk) {
      if (m == 0) write_trivial_row(p, w.r, w.len);
      continue;
    }
    for (int j = 0; j < w.nch; ++j) {
      if (s.buf_n + kChunk > kBufCap) {
        compact_to_bin(s);
        if (s.cnt_ge + kChunk > kBufCap) compact_exact(s, p.topk);
      }
      const int slot = static_cast<int>(q % kStages);
      const bool ok = mbar_wait_bounded(&s.full[slot], (q / kStages) & 1u, p.timeout_ns);
      if (!ok) {
        s.abort = 1;
        atomicOr(p.status, 0x4u);
      } else {
        const int ws = w.wstart + j * kChunk;
        const int we = min(ws + kChunk, w.wend);
        filter_chunk(s, s.stage[slot], ws, (we - ws) >> 2, w.lo, w.hi);
      }
      __syncthreads();
      if (s.abort) {
        aborted = true;
        break;
      }
      if (tid < 32) {
        advance_threshold(s, p.topk);
        if (tid == 0) producer_issue(p, s, P, g, m);
      }
      ++q;
      __syncthreads();
    }
    if (aborted) break;
    if (p.G == 1) {
      finish_local(s, p, w.r);
    } else if (!finish_group(s, p, w.r, g, m, epoch, first_barrier)) {
      aborted = true;
    }
  }

  if (aborted) {
    if (tid == 0) drain_copies(s, P, q, p.timeout_ns);
    return;
  }
  if (p.G > 1) {
    // last CTA of the group to finish clears the per-member words and counters
    GroupWs* gw = p.groups + g;
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const uint32_t old = atom_add_acq_rel_gpu(&gw->exit_count, 1u);
      s.last = (old == static_cast<uint32_t>(p.G - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (s.last) {
      uint32_t* h3 = &gw->h3[0][0];
      for (int i = tid; i < kMaxGroup * 256; i += kThreads) __stcg(h3 + i, 0u);
      uint32_t* c = &gw->cnt[0][0];
      for (int i = tid; i < kMaxGroup * 4; i += kThreads) __stcg(c + i, 0u);
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        __stcg(&gw->bar_count, 0u);
        __stcg(&gw->exit_count, 0u);
      }
    }
  }
}

// ---------------------------------------------------------------- host side

size_t kernel_smem_bytes() { return sizeof(Smem); }

cudaError_t kernel_configure() {
  return cudaFuncSetAttribute(topk_ragged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(Smem)));
}

cudaError_t kernel_occupancy(int* ctas_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, topk_ragged_kernel, kThreads,
                                                       sizeof(Smem));
}

cudaError_t launch_topk(const Params& p, int grid, bool cooperative, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, topk_ragged_kernel, p);
}

}  // namespace ltk
