/*
 * CPU oracle for the ragged per-row top-K selection.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do. It shares no code, header or table with the CUDA path.
 *
 * What it computes (the plain definition the GPU path must reproduce exactly):
 *   For every row r, with the valid length len_r taken from a per-row int32
 *   lengths vector (vLLM PR #54110 page, "Implementation breakdown" item 2:
 *   next_n comes from the second dimension of a 2-D lengths tensor, so every
 *   MTP row carries its own length), take the fp32 logits
 *   x[r*row_stride + i] for 0 <= i < len_r, order the pairs (x_i, i) by value
 *   descending and, for equal values, by index ascending, and keep the first
 *   min(len_r, topk) indices. The rest of the int32 output row (topk entries,
 *   the TopK template of the persistent_topk kernel on the vLLM PR #41189 page,
 *   "Implementation breakdown" code excerpt) is filled with -1.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - equal values are ordered by index (IEEE equality, so -0.0 == +0.0);
 *   - values are compared exactly (no flush of denormals to zero);
 *   - +inf / -inf inside the valid prefix are ordinary values;
 *   - NaN is outside the contract and never generated;
 *   - a length below 0 is treated as 0 and a length above row_stride as
 *     row_stride; either sets bit 0 of the returned status word;
 *   - next_n only describes the layout (rows of one request are adjacent); it
 *     must divide num_rows.
 *
 * The output row is written in selection order (value desc, index asc), which
 * is also the order the parity tests sort the GPU result into.
 *
 * Deliberate mistakes for the pin tests: compiling with -DORACLE_MUTANT=<n>
 * plants one plausible bug (see the switch below); the pin tests must reject
 * every such build.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

typedef struct {
  float v;
  int32_t i;
} entry_t;

/* Total order: larger value first; on equal values the smaller index first. */
static int cmp_entry(const void* pa, const void* pb) {
  const entry_t* a = (const entry_t*)pa;
  const entry_t* b = (const entry_t*)pb;
#if ORACLE_MUTANT == 6
  /* mutant: smallest values first */
  if (a->v < b->v) return -1;
  if (a->v > b->v) return 1;
#elif ORACLE_MUTANT == 4
  /* mutant: orders -0.0 below +0.0 by comparing sign bits first */
  if (a->v == b->v && a->v == 0.0f) {
    int sa = signbit(a->v) != 0, sb = signbit(b->v) != 0;
    if (sa != sb) return sa ? 1 : -1;
  }
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
#else
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
#endif
#if ORACLE_MUTANT == 1
  /* mutant: ties go to the larger index */
  return (a->i > b->i) ? -1 : (a->i < b->i);
#else
  return (a->i < b->i) ? -1 : (a->i > b->i);
#endif
}

typedef struct {
  const float* logits;
  int64_t row_stride;
  const int32_t* lengths;
  int64_t num_rows;
  int next_n;
  int topk;
  int32_t* out;
  int tid;
  int nthreads;
  unsigned status;
} job_t;

static void* run_rows(void* arg) {
  job_t* jb = (job_t*)arg;
  entry_t* scratch = NULL;
  int64_t cap = 0;
  for (int64_t r = jb->tid; r < jb->num_rows; r += jb->nthreads) {
#if ORACLE_MUTANT == 11
    /* mutant: one length per request instead of one per row */
    int64_t len = jb->lengths[(r / jb->next_n) * jb->next_n];
#else
    int64_t len = jb->lengths[r];
#endif
    if (len < 0) {
      len = 0;
      jb->status |= 1u;
    }
    if (len > jb->row_stride) {
      len = jb->row_stride;
      jb->status |= 1u;
    }
#if ORACLE_MUTANT == 3
    /* mutant: drops the last valid element */
    if (len > 0) len -= 1;
#endif
#if ORACLE_MUTANT == 10
    /* mutant: rows addressed by length instead of by stride */
    const float* x = jb->logits + r * (int64_t)jb->lengths[0];
#else
    const float* x = jb->logits + r * jb->row_stride;
#endif
    if (len > cap) {
      free(scratch);
      cap = len;
      scratch = (entry_t*)malloc((size_t)cap * sizeof(entry_t));
      if (!scratch) {
        jb->status |= 0x80000000u;
        return NULL;
      }
    }
    for (int64_t i = 0; i < len; ++i) {
      scratch[i].v = x[i];
      scratch[i].i = (int32_t)i;
    }
    qsort(scratch, (size_t)len, sizeof(entry_t), cmp_entry);
    int32_t* o = jb->out + r * (int64_t)jb->topk;
    int64_t take = len < jb->topk ? len : jb->topk;
#if ORACLE_MUTANT == 7
    /* mutant: off by one at the topk boundary for long rows */
    if (len >= jb->topk) take = jb->topk - 1;
#endif
    for (int64_t j = 0; j < take; ++j) o[j] = scratch[j].i;
#if ORACLE_MUTANT == 2
    /* mutant: pads with 0 instead of -1 */
    for (int64_t j = take; j < jb->topk; ++j) o[j] = 0;
#else
    for (int64_t j = take; j < jb->topk; ++j) o[j] = -1;
#endif
  }
  free(scratch);
  return NULL;
}

/*
 * Selects, for every row, the indices described in the header comment.
 * logits:  host pointer, num_rows * row_stride fp32 values (row-major).
 * lengths: host pointer, num_rows int32 valid lengths.
 * out_idx: host pointer, num_rows * topk int32 results (written).
 * nthreads: worker threads (rows are dealt round-robin); values < 1 mean 1.
 * Returns a status word: bit 0 = some length was clamped into [0, row_stride];
 * bit 31 = out of host memory; 0xFFFFFFFE = invalid arguments.
 */
unsigned oracle_topk_ragged(const float* logits, int64_t row_stride,
                            const int32_t* lengths, int64_t num_rows,
                            int next_n, int topk, int32_t* out_idx,
                            int nthreads) {
  if (num_rows < 0 || row_stride < 1 || topk < 1 || next_n < 1 ||
      (num_rows % next_n) != 0)
    return 0xFFFFFFFEu;
  if (num_rows == 0) return 0;
  if (!logits || !lengths || !out_idx) return 0xFFFFFFFEu;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > num_rows) nthreads = (int)num_rows;
  job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return 0x80000000u;
  }
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].logits = logits;
    jobs[t].row_stride = row_stride;
    jobs[t].lengths = lengths;
    jobs[t].num_rows = num_rows;
    jobs[t].next_n = next_n;
    jobs[t].topk = topk;
    jobs[t].out = out_idx;
    jobs[t].tid = t;
    jobs[t].nthreads = nthreads;
    jobs[t].status = 0;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, run_rows, &jobs[t]) != 0) break;
    started = t;
  }
  run_rows(&jobs[0]);
  /* rows of threads that failed to start are done here, serially */
  for (int t = started + 1; t < nthreads; ++t) run_rows(&jobs[t]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  unsigned status = 0;
  for (int t = 0; t < nthreads; ++t) status |= jobs[t].status;
  free(jobs);
  free(th);
  return status;
}
