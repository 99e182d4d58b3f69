/*
 * topk_oracle.c — CPU oracle for batched row-wise TopK.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header or table with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *   For each row, decode every element of [0, len) to a real number in double
 *   precision (bf16: the 16 stored bits are the upper half of a binary32, which
 *   converts to double exactly; fp32: exact conversion). Sort all (value, index)
 *   pairs of the row with one comparator — value descending, then index
 *   ascending on equal values — and keep the first k pairs. Emit their indices
 *   in ascending index order, and the input bit patterns at those indices.
 *
 * Where this comes from:
 *   - deepseek.csdn.net, "DeepSeek 一次开源三个仓库", section 三 (算子层): TopK of
 *     each row, topk <= 4096, int32 indices, the sorted_index option. The page's
 *     scheme (threshold filter, compaction to K, threshold raised to the
 *     compacted minimum) never drops a true top-K element, so it reaches exactly
 *     this set; the oracle computes the set by its definition instead.
 *   - github-research.aiutil.com, "deepseek-ai/DeepSelect", section 关键技术亮点:
 *     TopK does no floating-point math, so the values are copies of the input.
 *   - deepseek-v4-pro.uk (zh-tw), section "DeepSelect：快速且刻意狹義的 TopK": the
 *     NaN check is always on. Here: a row containing a NaN in [0, len) raises the
 *     flag and gets no selection (its outputs are filled with -1 / zero bits).
 *
 * Readings where the pages are silent (the same ones the library documents):
 *   ties at the k-th value resolve to the lowest indices; -0.0 equals +0.0; +inf
 *   and -inf are ordinary values; subnormals compare as their exact values
 *   (build without -ffast-math); padding [len, row_stride) is never read.
 *
 * Build: gcc -O2 -fPIC -shared -pthread (no fast-math). Rows run in parallel
 * over POSIX threads only so that the CPU baseline can use every host core; each
 * row is handled by the same plain code.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
  double value;
  int32_t index;
} oracle_pair;

/* The total order: value descending, then index ascending. */
static int by_value_desc_index_asc(const void* pa, const void* pb) {
  const oracle_pair* a = (const oracle_pair*)pa;
  const oracle_pair* b = (const oracle_pair*)pb;
  if (a->value > b->value) return -1;
  if (a->value < b->value) return 1;
  if (a->index < b->index) return -1;
  if (a->index > b->index) return 1;
  return 0;
}

static int by_index_asc(const void* pa, const void* pb) {
  const oracle_pair* a = (const oracle_pair*)pa;
  const oracle_pair* b = (const oracle_pair*)pb;
  return (a->index > b->index) - (a->index < b->index);
}

/* Decode element `i` of a row to double. dtype 0 = bf16, 1 = fp32. */
static double decode(const void* row, int dtype, int64_t i) {
  if (dtype == 0) {
    uint16_t h = ((const uint16_t*)row)[i];
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  float f = ((const float*)row)[i];
  return (double)f;
}

typedef struct {
  const void* x;
  int dtype;
  int64_t len, row_stride;
  int k;
  int return_value;
  void* out_values;
  int32_t* out_indices;
  uint8_t* row_nan;
  int64_t row_begin, row_end;
  int by_value; /* 1: keep the first k pairs in the total order (value order) */
  int any_nan;
  int failed;
} oracle_job;

static void select_rows(oracle_job* job) {
  const size_t esize = job->dtype == 0 ? 2 : 4;
  oracle_pair* pairs = (oracle_pair*)malloc(sizeof(oracle_pair) * (size_t)job->len);
  if (!pairs) {
    job->failed = 1;
    return;
  }
  for (int64_t b = job->row_begin; b < job->row_end; ++b) {
    const char* row = (const char*)job->x + (size_t)b * (size_t)job->row_stride * esize;
    int has_nan = 0;
    for (int64_t i = 0; i < job->len; ++i) {
      pairs[i].value = decode(row, job->dtype, i);
      pairs[i].index = (int32_t)i;
      if (isnan(pairs[i].value)) has_nan = 1;
    }
    if (job->row_nan) job->row_nan[b] = (uint8_t)has_nan;
    int32_t* oi = job->out_indices + (size_t)b * (size_t)job->k;
    if (has_nan) {
      /* No order exists with a NaN in the row: no selection, sentinel outputs. */
      job->any_nan = 1;
      for (int j = 0; j < job->k; ++j) oi[j] = -1;
      if (job->return_value)
        memset((char*)job->out_values + (size_t)b * (size_t)job->k * esize, 0,
               (size_t)job->k * esize);
      continue;
    }
    qsort(pairs, (size_t)job->len, sizeof(oracle_pair), by_value_desc_index_asc);
    if (!job->by_value) qsort(pairs, (size_t)job->k, sizeof(oracle_pair), by_index_asc);
    for (int j = 0; j < job->k; ++j) {
      oi[j] = pairs[j].index;
      if (job->return_value) {
        char* ov = (char*)job->out_values + ((size_t)b * (size_t)job->k + (size_t)j) * esize;
        memcpy(ov, row + (size_t)pairs[j].index * esize, esize);
      }
    }
  }
  free(pairs);
}

static void* run_job(void* arg) {
  select_rows((oracle_job*)arg);
  return NULL;
}

/*
 * oracle_topk — same argument meaning as the library's ds_topk, on HOST memory.
 * row_nan (optional, may be NULL) receives 1 for rows that hold a NaN.
 * nthreads <= 0 uses every online core. Returns 0, 1 on a bad argument, 2 on an
 * allocation or thread failure. *nan_flag gets bit 0 set if any row had a NaN
 * (never cleared). The output order is ascending index for sorted_index 0 and 1;
 * for sorted_index 2 it is the total order itself (value descending, equal values
 * by ascending index), as the first k pairs of the full sort come out
 * (github-research.aiutil.com, "deepseek-ai/DeepSelect", section 关键技术亮点,
 * item 2: outputs ordered by index or by value).
 */
int oracle_topk(const void* x, int dtype, int64_t batch, int64_t len, int64_t row_stride,
                int k, int sorted_index, int return_value, void* out_values,
                int32_t* out_indices, int32_t* nan_flag, uint8_t* row_nan, int nthreads) {
  if (dtype != 0 && dtype != 1) return 1;
  if (sorted_index < 0 || sorted_index > 2) return 1;
  if (batch < 0 || len < 1 || len > INT32_MAX || row_stride < len) return 1;
  if (k < 1 || k > 4096 || (int64_t)k > len) return 1;
  if (batch == 0) return 0;
  if (!x || !out_indices || !nan_flag || (return_value && !out_values)) return 1;

  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if ((int64_t)nthreads > batch) nthreads = (int)batch;

  oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  char* live = (char*)calloc((size_t)nthreads, 1);
  if (!jobs || !tids || !live) {
    free(jobs);
    free(tids);
    free(live);
    return 2;
  }
  int rc = 0;
  for (int t = 0; t < nthreads; ++t) {
    oracle_job* j = &jobs[t];
    j->x = x;
    j->dtype = dtype;
    j->len = len;
    j->row_stride = row_stride;
    j->k = k;
    j->return_value = return_value;
    j->out_values = out_values;
    j->out_indices = out_indices;
    j->row_nan = row_nan;
    j->by_value = sorted_index == 2;
    j->row_begin = batch * t / nthreads;
    j->row_end = batch * (t + 1) / nthreads;
    if (nthreads == 1) {
      select_rows(j);
    } else if (pthread_create(&tids[t], NULL, run_job, j) == 0) {
      live[t] = 1;
    } else {
      select_rows(j); /* run inline if a thread cannot be started */
    }
  }
  for (int t = 0; t < nthreads; ++t)
    if (live[t]) pthread_join(tids[t], NULL);
  int any_nan = 0;
  for (int t = 0; t < nthreads; ++t) {
    any_nan |= jobs[t].any_nan;
    if (jobs[t].failed) rc = 2;
  }
  if (any_nan) *nan_flag |= 1;
  free(jobs);
  free(tids);
  free(live);
  return rc;
}

/* Number of online host cores (what nthreads <= 0 uses). */
int oracle_cores(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }
