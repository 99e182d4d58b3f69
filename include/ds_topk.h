/*
 * ds_topk.h — C ABI of the batched row-wise TopK library (libds_topk.so).
 *
 * What the operation is
 * ---------------------
 * For every row b of a row-major matrix x, select the k largest elements of
 * x[b, 0:len) under the TOTAL order "value descending, then column index
 * ascending on equal values", and write their int32 column indices (and,
 * optionally, the input bit patterns at those columns).
 *
 * Sources (web pages about DeepSeek's DeepSelect TopK kernel):
 *  - deepseek.csdn.net, "DeepSeek 一次开源三个仓库：模型厂开始把'部署栈'也开源了",
 *    section 三 (算子层): the call deep_select.topk(x, topk, sorted_index=...,
 *    indices_type=torch.int32), the limit topk <= 4096, and the selection scheme
 *    (block scan, threshold filter into a candidate buffer, compaction to K in
 *    shared memory, threshold raised to the compacted minimum).
 *  - deepseek-v4-pro.uk (zh-tw), "深入 DeepSeek V4.1 全新開放推論工具包",
 *    section "DeepSelect：快速且刻意狹義的 TopK": bf16 Lightning-Indexer path and
 *    fp32 sampler path, topk <= 4096, rows need a specific alignment (callers may
 *    pad; here such rows take a slower path instead of being refused),
 *    return_value=False skips the values output, the NaN check is always on.
 *  - github-research.aiutil.com, "deepseek-ai/DeepSelect", section 关键技术亮点:
 *    TopK does no floating-point math, so values are copied, never computed.
 *
 * The pages give only the Python surface; this C signature, the error codes,
 * the alignment rule and the NaN flag (instead of a trap) are this library's
 * readings of it.
 */
#ifndef DS_TOPK_H_
#define DS_TOPK_H_

#include <stdint.h>
#include <cuda_runtime_api.h>

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define DS_TOPK_API __attribute__((visibility("default")))
#else
#define DS_TOPK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of x (and of out_values). */
typedef enum {
  DS_TOPK_BF16 = 0, /* bfloat16 bit patterns, 2 bytes: the Lightning-Indexer scores   */
  DS_TOPK_FP32 = 1  /* IEEE binary32, 4 bytes: the sampler logits                       */
} ds_topk_dtype;

/* Return codes of every entry point. */
typedef enum {
  DS_TOPK_OK = 0,       /* launched (or nothing to do: batch == 0)                      */
  DS_TOPK_EINVAL = 1,   /* bad argument; nothing was launched                            */
  DS_TOPK_EALIGN = 2,   /* x or an output pointer misaligned; nothing launched           */
  DS_TOPK_ECUDA = 3,    /* a CUDA runtime call failed (device query or launch)           */
  DS_TOPK_ETIMEOUT = 4  /* reserved: a bounded device-side wait expired (see flag bits)  */
} ds_topk_status;

/* Bits the kernels OR into *nan_flag (the device status word). */
#define DS_TOPK_FLAG_NAN 1     /* some row held a NaN in [0, len)                        */
#define DS_TOPK_FLAG_TIMEOUT 2 /* a bounded device-side wait gave up (never expected);
                                  every output of the call is then undefined          */

/* Hard limit on k, from the pages ("topk <= 4096"). */
#define DS_TOPK_MAX_K 4096

/* Index type of out_indices (the index_type argument of ds_topk_ex). */
#define DS_TOPK_INDEX_INT32 0
#define DS_TOPK_INDEX_INT64 1

/* Output order (the sorted_index argument). */
#define DS_TOPK_SORT_NONE 0  /* unspecified order                                  */
#define DS_TOPK_SORT_INDEX 1 /* ascending index                                    */
#define DS_TOPK_SORT_VALUE 2 /* value descending, equal values by ascending index  */

/*
 * ds_topk — batched row-wise TopK, enqueued on `stream`.
 *
 * Arguments (all sizes in ELEMENTS unless stated):
 *   x            device pointer, row-major [batch, row_stride] of `dtype`.
 *                Row b starts at element b*row_stride; elements [0, len) of it
 *                are the row. Only those elements are inspected (padding
 *                [len, row_stride) is never selected nor checked for NaN).
 *                Must be aligned to sizeof(dtype); rows need not start on a
 *                16-byte boundary. Every kernel reads a row as the 16-byte
 *                aligned blocks that overlap [0, len): the elements of those
 *                blocks outside the row are masked before any compare (never
 *                selected nor checked for NaN), and no block without a row
 *                element is read. Rows off 16-byte boundaries (x not 16-byte
 *                aligned, or row_stride * sizeof(dtype) not a multiple of 16)
 *                give the same result; on the one-CTA/cluster-per-row paths
 *                they forgo the next-row prefetch.
 *   dtype        DS_TOPK_BF16 or DS_TOPK_FP32.
 *   batch        number of rows, >= 0. batch == 0 returns DS_TOPK_OK at once
 *                (pointers may then be NULL).
 *   len          row length, 1 <= len <= INT32_MAX.
 *   row_stride   elements between row starts, >= len. Any value (see x); the
 *                pages' kernel requires 16-byte aligned rows and leaves the
 *                padding to callers, this library does not.
 *   k            1 <= k <= min(len, DS_TOPK_MAX_K).
 *   sorted_index DS_TOPK_SORT_NONE (0), DS_TOPK_SORT_INDEX (1) or
 *                DS_TOPK_SORT_VALUE (2). 1: each output row lists its k indices
 *                in ascending index order. 0: the order within a row is
 *                unspecified (the one-CTA/cluster paths emit ascending index
 *                order anyway; the one-warp-per-row path writes the elements
 *                above the k-th value first and the ties at it last).
 *                2: value descending, equal values by ascending index (the
 *                selection's total order); this costs one more kernel launch on
 *                the same stream, a per-row sort of the k outputs
 *                (github-research.aiutil.com, "deepseek-ai/DeepSelect", section
 *                关键技术亮点, item 2: outputs ordered by index or by value, either
 *                at a cost in speed).
 *   return_value 0 or 1. 1: out_values[b*k + j] = the input bit pattern at
 *                column out_indices[b*k + j] (bitwise copy, -0.0 stays -0.0).
 *                0: out_values is not touched and may be NULL.
 *   out_values   device pointer [batch, k] of `dtype`, contiguous, aligned to
 *                sizeof(dtype); required iff return_value == 1.
 *   out_indices  device pointer [batch, k] int32, contiguous, 4-byte aligned.
 *   nan_flag     device pointer to one int32 status word, 4-byte aligned. The
 *                kernels OR DS_TOPK_FLAG_NAN into it if any element of any
 *                row's [0, len) is NaN; the word is never cleared by the
 *                library (the caller zeroes it). A row holding a NaN gets
 *                unspecified (but in-range, in-bounds) outputs; every other
 *                row is exact. There is no trap: the pages' kernel aborts on
 *                NaN by default, which a shared GPU cannot afford.
 *   stream       CUDA stream the work is enqueued on (0 = legacy default).
 *
 * Selected set: with v_i the value of column i (bf16 decodes exactly to fp32;
 * -0.0 == +0.0; +inf largest, -inf smallest), the row's pairs (v_i, i) are
 * ordered by value descending, then index ascending, and the first k pairs are
 * selected. The result is a pure function of the input.
 *
 * Ownership and memory: the caller owns every buffer and the stream. The call
 * allocates no device or host memory and uses no global scratch memory: a row
 * split over several CTAs is reduced through thread-block-cluster distributed
 * shared memory.
 *
 * Errors: arguments are validated before anything is enqueued; a bad argument
 * returns DS_TOPK_EINVAL or DS_TOPK_EALIGN and launches nothing. A failed
 * device query or launch returns DS_TOPK_ECUDA. The call does not synchronize;
 * device-side conditions are reported only through *nan_flag.
 *
 * Threading: reentrant; concurrent calls on different streams are safe (no
 * shared mutable state besides a per-device cache of launch attributes that is
 * filled under a lock).
 */
DS_TOPK_API int ds_topk(const void* x, int dtype, int64_t batch, int64_t len, int64_t row_stride,
            int k, int sorted_index, int return_value, void* out_values,
            int32_t* out_indices, int32_t* nan_flag, cudaStream_t stream);

/*
 * ds_topk_ex — ds_topk with a selectable index type (deepseek.csdn.net,
 * "DeepSeek 一次开源三个仓库", section 三: the call's indices_type argument).
 * index_type DS_TOPK_INDEX_INT32: out_indices is int32 [batch, k] (4-byte
 * aligned), exactly ds_topk; DS_TOPK_INDEX_INT64: out_indices is int64
 * [batch, k], 8-byte aligned. Everything else as ds_topk; any other index_type
 * returns DS_TOPK_EINVAL with nothing enqueued.
 */
DS_TOPK_API int ds_topk_ex(const void* x, int dtype, int64_t batch, int64_t len, int64_t row_stride,
               int k, int sorted_index, int return_value, int index_type, void* out_values,
               void* out_indices, int32_t* nan_flag, cudaStream_t stream);

/*
 * ds_topk_sample — the sampler tail after TopK: for each row, select the k
 * largest logits in value order (as ds_topk with sorted_index =
 * DS_TOPK_SORT_VALUE and return_value = 1, into out_values / out_indices), then
 * draw one column from them:
 *   w_j = exp((v_j - v_0) / temperature)  over the k survivors in value order
 *         (v_0 the largest; if v_0 is +inf, the +inf values weigh 1, the rest 0),
 *   C_j = w_0 + ... + w_j, the nucleus is the shortest prefix [0, m] with
 *   C_m >= top_p * C_{k-1}, and the token is the column at the first j <= m with
 *   C_j > u[b] * C_m (inverse CDF).
 * github-research.aiutil.com, "deepseek-ai/DeepSelect", section 关键技术亮点: the
 * sampler path of TopK, whose survivors the next token is drawn from;
 * deepseek.csdn.net, "DeepSeek 一次开源三个仓库": temperature and top_p as the
 * request's sampling parameters. Readings where the pages are silent: the
 * softmax runs over the k survivors only; top-p keeps the shortest prefix that
 * reaches the mass; the draw takes the caller's uniform number.
 *
 * Arguments: x, dtype, batch, len, row_stride, k, nan_flag and stream as for
 * ds_topk.
 *   temperature  finite, > 0.
 *   top_p        0 < top_p <= 1.
 *   u            device pointer [batch] float, each in [0, 1), 4-byte aligned:
 *                one uniform random number per row (the caller draws them).
 *   out_values   device pointer [batch, k] of `dtype` (required): the k
 *                selected values in value order.
 *   out_indices  device pointer [batch, k] int32: their columns.
 *   out_tokens   device pointer [batch] int32, 4-byte aligned: the drawn column.
 * The arithmetic is fp32 (expf and sums over the k survivors); a draw can
 * differ from an exact (float64) computation only when u * C_m or
 * top_p * C_{k-1} lies within (k + 40) * 2^-22 * C_{k-1} of a step of C (expf
 * within 2 ulp, the rounded argument, a block scan of depth at most 40 and the
 * two products; the tests check the draws against exactly this bound).
 * A row holding a NaN gets an unspecified but in-range token.
 * Returns DS_TOPK_OK, DS_TOPK_EINVAL (also for a bad temperature or top_p),
 * DS_TOPK_EALIGN or DS_TOPK_ECUDA, like ds_topk; nothing is enqueued on an
 * argument error. Kernel launches on `stream`: two when the value order sorts
 * one row per CTA (that sort draws the tokens too), three after the
 * one-warp-per-row sort (many bf16 rows); no allocation.
 */
DS_TOPK_API int ds_topk_sample(const void* x, int dtype, int64_t batch, int64_t len, int64_t row_stride,
                   int k, float temperature, float top_p, const float* u, void* out_values,
                   int32_t* out_indices, int32_t* out_tokens, int32_t* nan_flag, cudaStream_t stream);

/* Which kernel family a call runs. */
typedef enum {
  DS_TOPK_PATH_ROW = 0,      /* one CTA per row                                     */
  DS_TOPK_PATH_CLUSTER = 1,  /* one thread-block cluster per row (row split in slices) */
  DS_TOPK_PATH_WARP_ROWS = 2  /* one warp per row, several rows per CTA: many rows of at
                                 most 65536 elements with k <= 1024                  */
} ds_topk_path;

/* Launch plan of one ds_topk call, as chosen by the host dispatcher. */
typedef struct {
  int32_t path;                /* ds_topk_path                                         */
  int32_t cluster_size;        /* CTAs cooperating on one row (1 for DS_TOPK_PATH_ROW) */
  int32_t threads_per_cta;
  int32_t vectors_per_granule; /* 16-byte vectors summarised by one granule maximum
                                  (1 on DS_TOPK_PATH_WARP_ROWS: vectors are tested one
                                  by one)                                              */
  int64_t grid_ctas;           /* CTAs if every row had its own cluster (warp rows: if
                                  every 8 rows had their own CTA), capped at INT32_MAX
                                  on the warp-rows path; ds_topk
                                  launches at most as many as can be co-resident, and
                                  each persistent cluster (warp) then walks rows with
                                  a stride                                             */
  int64_t granules_per_cta;    /* size of the per-CTA granule-maximum array; on
                                  DS_TOPK_PATH_WARP_ROWS the candidate slots per warp  */
  int32_t smem_bytes;          /* dynamic shared memory per CTA                        */
  int32_t launches;            /* kernel launches per call with sorted_index 0 or 1
                                  (DS_TOPK_SORT_VALUE adds one)                        */
} ds_topk_plan_t;

/*
 * ds_topk_plan — fill *plan with the launch plan ds_topk would use for these
 * sizes on a GPU with `sm_count` SMs, without touching the GPU (pure host logic;
 * runs without a device). Same validation as ds_topk for the size arguments
 * (x/output pointers are not involved: x is taken to be 16-byte aligned; for an
 * x that is not, the row/cluster plans may hold one 16-byte block more per row
 * and no next-row prefetch, the path is the same).
 * Returns DS_TOPK_OK or DS_TOPK_EINVAL; plan must be non-NULL and
 * sm_count >= 1.
 */
DS_TOPK_API int ds_topk_plan(int dtype, int64_t batch, int64_t len, int64_t row_stride, int k,
                 int sm_count, ds_topk_plan_t* plan);

/* Short static description of a status code ("ok", "invalid argument", ...). */
DS_TOPK_API const char* ds_topk_status_string(int status);

/* Library version, e.g. 100 for 0.1.0. */
DS_TOPK_API int ds_topk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DS_TOPK_H_ */
