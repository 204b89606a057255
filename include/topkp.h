/*
 * topkp.h -- C ABI of libtopkp.so, the fused top-k / top-p logit filter for
 * NVIDIA GB300 (sm_103a).
 *
 * What it computes.  The operation is the one defined in section 2
 * (计算流程与公式) of the web page "CANN ops-nn 算子实战：
 * ApplyTopKTopPWithSorted 的 top-k/top-p 采样过滤原理与 aclnn 调用指南":
 * per row of a [B, V] logits matrix,
 *   1. order the row ascending with a stable sort (equal values keep their
 *      index order; -0 equals +0);
 *   2. if top-k is on, every value strictly below the k-th largest becomes
 *      -inf (values equal to the k-th largest survive);
 *   3. softmax in fp32 over the surviving values;
 *   4. ascending cumulative sum C_j of those probabilities;
 *   5. if top-p is on, every sorted position with C_j <= round_D(1 - p)
 *      becomes -inf, except the last (largest) position, which always stays;
 *   6. results go back to the original order: each output element is either
 *      the input element, bit for bit, or the dtype's -inf
 *      (fp32 0xFF800000, fp16 0xFC00, bf16 0xFF80).
 * Top-k is on for row b iff k != NULL and 1 <= k[b] <= V-1 (section 4,
 * 约束说明: k <= 0 or k >= V means no top-k).  Top-p is on iff p != NULL.
 * round_D(1 - p) is 1 - p evaluated in fp32 and rounded to the logits dtype,
 * because p has the logits dtype (section 3, 参数说明).
 *
 * Results.  Top-k decisions are exact.  A top-p decision can differ from the
 * exact fp32 definition only at positions whose cumulative probability lies
 * within 1e-5 of round_D(1 - p): the library sums probability mass exactly
 * in 64-bit fixed point, from fp32 exponentials whose relative error is
 * about 2e-6, and 1e-5 is the bound the tests hold it to.  Results are
 * deterministic: the same inputs give the same bits on every call.
 *
 * Conventions shared by every entry point.
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never frees or retains them past the call, and allocates no device
 *     memory per call.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous: the function returns after the launch is enqueued, and
 *     no argument check synchronises the device.
 *   - Row-major layout; V is the fastest-varying dimension.
 *   - The calling thread's current CUDA device must own the pointers.
 *   - Value ranges are not checked (the page's CheckParams checks null
 *     pointers, dtypes and shapes only): p outside [0, 1], NaN or +inf
 *     logits, an unsorted sorted_value or a sorted_indices that is not a
 *     permutation give unspecified output; sorted_indices entries outside
 *     [0, V) are skipped, never written through.
 *   - On any non-zero status nothing was launched; topkp_last_error_string()
 *     gives a one-line reason (thread-local, like aclGetRecentErrMsg in
 *     section 8 of the page).
 */
#ifndef TOPKP_H
#define TOPKP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of logits, p, sorted_value and out (section 3: FLOAT,
 * FLOAT16, BFLOAT16; p has the same dtype as the logits). */
typedef enum {
  TOPKP_F32 = 0,
  TOPKP_F16 = 1,
  TOPKP_BF16 = 2
} topkp_dtype;

typedef int topkp_status;

/* Status codes.  The two parameter errors reuse the page's aclnn codes
 * (section 5.3 返回码与异常场景). */
#define TOPKP_SUCCESS 0
/* logits / sorted_value / sorted_indices / out is NULL on a non-empty
 * problem, or p and k are both NULL. */
#define TOPKP_ERR_PARAM_NULLPTR 161001
/* unknown dtype, B or V negative, V above TOPKP_MAX_V, a row stride below V,
 * or out overlapping an input without being identical to it. */
#define TOPKP_ERR_PARAM_INVALID 161002
/* the CUDA launch failed (including: no CUDA device). */
#define TOPKP_ERR_LAUNCH 561000
/* a kernel gave up a bounded wait on its own copy-completion barrier; it
 * skipped its writes for the affected rows.  Reported by
 * topkp_device_status(). */
#define TOPKP_ERR_DEVICE_TIMEOUT 561001
/* topkp_sort_static only: the device had no room for the library's static
 * scratch when the sort's module was first loaded on it. */
#define TOPKP_ERR_NO_MEMORY 561002

/* Largest supported row length: probability mass is summed in unsigned
 * 64-bit fixed point with 2^40 per unit, so a row may hold at most 2^23
 * elements. */
#define TOPKP_MAX_V (1LL << 23)

/*
 * topkp_apply -- aclnnApplyTopKTopP (section 5 of the page): filter raw
 * logits; the ordering is found internally, without a full sort.
 *
 *   logits     device, [B, V] of dtype, row stride ld_logits elements (>= V).
 *   B, V       rows and row length (>= 0).  B == 0 or V == 0 returns
 *              TOPKP_SUCCESS without a launch.  V == 1 copies the row.
 *   ld_logits  row stride of logits in elements.
 *   dtype      TOPKP_F32, TOPKP_F16 or TOPKP_BF16.
 *   p          device, [B] of dtype, or NULL (top-p off).
 *   k          device, [B] int32, or NULL (top-k off).  p and k must not both
 *              be NULL.
 *   out        device, [B, V] of dtype, row stride ld_out elements (>= V).
 *              out == logits with ld_out == ld_logits (in place) is allowed;
 *              any other overlap with logits, p or k is rejected.
 *   stream     cudaStream_t to launch on.
 * Rows of at most 4096 elements, and 16-bit rows of at most 32768, run on a
 * kernel that holds each row on chip (one block per row); longer rows on the
 * main filter kernel.  Both give the same bits.  One kernel launch per
 * 2^31 - 1 blocks.
 */
topkp_status topkp_apply(const void* logits, int64_t B, int64_t V, int64_t ld_logits,
                         topkp_dtype dtype, const void* p, const int32_t* k,
                         void* out, int64_t ld_out, void* stream);

/*
 * topkp_apply_sample -- topkp_apply and topkp_sample in one pass: the filter
 * of section 2 of the page, then, on its survivors, the min-p step and the
 * sample of the web page "aclnnTopKTopPSampleV2" (Formula / minP sampling,
 * Formula / Subsequent processing).  The result equals topkp_sample run on
 * topkp_apply's output with the same min_p, q and eps (same arithmetic, so
 * the same bits), but no filtered row is read back, and with out == NULL
 * nothing is written but the token.
 *
 *   logits, B, V, ld_logits, dtype, p, k   as for topkp_apply.
 *   min_p      device, [B] float, or NULL (no min-p).
 *   q          device, [B, V] float, row stride ldq (>= V), or NULL (the
 *              token is the largest element, of equals the largest index).
 *   eps        added to every q, >= 0.
 *   out        device, [B, V] of dtype, row stride ld_out (>= V), or NULL:
 *              the rows after the filter and min-p.  out == logits with
 *              ld_out == ld_logits (in place) is allowed.
 *   token      device, [B] int32, or NULL.  out and token must not both be
 *              NULL; neither may overlap another argument.
 * Results: as topkp_apply and topkp_sample.  One kernel launch.
 */
topkp_status topkp_apply_sample(const void* logits, int64_t B, int64_t V, int64_t ld_logits, topkp_dtype dtype,
                                const void* p, const int32_t* k, const float* min_p, const float* q, int64_t ldq,
                                float eps, void* out, int64_t ld_out, int32_t* token, void* stream);

/*
 * topkp_apply_sorted -- the graph op ApplyTopKTopPWithSorted (section 3 of
 * the page): the caller supplies each row already sorted.
 *
 *   sorted_value    device, [B, V] contiguous, dtype; each row ascending, and
 *                   equal values in increasing original-index order (the
 *                   stable sort of section 6.1).
 *   sorted_indices  device, [B, V] contiguous int32: sorted_value[b][j] came
 *                   from column sorted_indices[b][j] of the logits.
 *   B, V, dtype     as for topkp_apply.
 *   p, k            as for topkp_apply (same top-k disable rule).
 *   logits          device, [B, V] contiguous, dtype, or NULL.  When given,
 *                   kept outputs are read from it in original order and only
 *                   the elements tied with the cut value go through
 *                   sorted_indices (the page's CompareSelectOnLogits +
 *                   ScatterBoundary); when NULL, every output is scattered
 *                   through sorted_indices.
 *   out             device, [B, V] contiguous, dtype; must not overlap any
 *                   input.
 */
topkp_status topkp_apply_sorted(const void* sorted_value, const int32_t* sorted_indices,
                                int64_t B, int64_t V, topkp_dtype dtype,
                                const void* p, const int32_t* k, const void* logits,
                                void* out, void* stream);

/*
 * topkp_sample -- the last two steps of the web page "aclnnTopKTopPSampleV2"
 * (CANN API reference; Formula / minP sampling and Formula / Subsequent
 * processing, its None and QSample modes), run on the output of
 * topkp_apply or topkp_apply_sorted: original order, filtered elements -inf.
 * Per row, with probs the softmax over the elements that are not -inf:
 *   1. min-p (min_p != NULL and min_p[b] > 0): every element whose
 *      probability is below min_p[b] times the largest probability becomes
 *      -inf; with min_p[b] >= 1 only the largest element stays (of equal
 *      largest values, the one with the largest index);
 *   2. the token: with q == NULL, the index of the largest element (ties:
 *      the largest index); otherwise the index of the largest
 *      probs / (q + eps) among the elements step 1 kept (ties: the largest
 *      index).  With q drawn i.i.d. from Exp(1), that index is a draw from
 *      probs.
 * The page forms probs over the top-k survivors and indexes q by sorted
 * position; here probs are over the filter's survivors and q follows the
 * original order.  Both decisions compare ratios of probabilities, so the
 * normaliser changes none of them.
 *
 *   filtered  device, [B, V] of dtype, row stride ld elements (>= V).  A row
 *             must hold at least one element that is not -inf; a row without
 *             one is copied unchanged and gets token -1.
 *   B, V      rows and row length (>= 0); B == 0 or V == 0 returns
 *             TOPKP_SUCCESS without a launch.
 *   dtype     TOPKP_F32, TOPKP_F16 or TOPKP_BF16.
 *   min_p     device, [B] float, or NULL (step 1 off).
 *   q         device, [B, V] float, row stride ldq (>= V), or NULL (None
 *             mode).  Values are expected >= 0.
 *   eps       added to every q (the page names it without a value), >= 0.
 *   out       device, [B, V] of dtype, row stride ld_out (>= V), or NULL:
 *             the rows after step 1 (input bits or -inf).  out == filtered
 *             with ld_out == ld is allowed; other overlaps are rejected.
 *   token     device, [B] int32, or NULL.  out and token must not both be
 *             NULL.
 *   stream    cudaStream_t to launch on.
 * Results.  The kernel compares base-2 logarithms of the ratios in fp32
 * ((x - max) log2 e against log2(min_p[b]); (x - max) log2 e - log2(q + eps)
 * for the race), so a min-p decision can differ from exact arithmetic only
 * where exp(x - max) lies within about 1e-5 (relative) of min_p[b], and the
 * token only where another kept element's probs / (q + eps) lies within
 * about 1e-5 (relative) of the largest.  Deterministic.
 */
topkp_status topkp_sample(const void* filtered, int64_t B, int64_t V, int64_t ld, topkp_dtype dtype,
                          const float* min_p, const float* q, int64_t ldq, float eps,
                          void* out, int64_t ld_out, int32_t* token, void* stream);

/*
 * topkp_sample_v2 -- the TopKTopPSampleV2 semantics of the web page
 * "aclnnTopKTopPSampleV2" (CANN API reference; Formula / TopK sampling,
 * TopP sampling, minP sampling, Optional output, Subsequent processing, and
 * Constraints).  Per row, on the row ordered from the largest value down
 * (equal values in increasing original index):
 *   1. top-k runs iff top_k != NULL and 1 <= top_k[b] <= min(V, ks_max
 *      rounded up to a multiple of 8); it keeps exactly the first top_k[b]
 *      positions (ties with the k-th value beyond them are removed);
 *   2. the probabilities: with input_is_logits, the softmax over the
 *      positions left; otherwise the input values themselves;
 *   3. top-p runs iff top_p != NULL and top_p[b] < 1.  After a top-k stage a
 *      position stays iff the probabilities before it sum to <= top_p[b];
 *      when top-k was skipped, iff its own and every later probability sum
 *      to > fp32(1 - top_p[b]).  The first position always stays;
 *   4. min-p (min_p != NULL and min_p[b] > 0): positions whose probability
 *      is below prob[0] * min_p[b] go; min_p[b] >= 1 keeps position 0 alone;
 *   5. the token: without q, the original index of position 0; with q, of
 *      the kept position with the largest prob / (q[b][j] + eps), where q is
 *      read by sorted position j (first on ties).
 * The kept positions form a prefix of the order.
 *
 *   logits       device, [B, V] of dtype, row stride ld_logits (>= V).
 *   B, V         rows and row length; 0 <= V <= 2^20 ([V2] Constraints).
 *                B == 0 or V == 0 returns TOPKP_SUCCESS without a launch.
 *   top_k        device, [B] int32, or NULL (top-k skipped on every row).
 *   top_p        device, [B] float, or NULL (top-p skipped).
 *   min_p        device, [B] float, or NULL (min-p skipped).
 *   q            device, [B, V] float, row stride ldq (>= V), or NULL (the
 *                token is position 0).
 *   eps          added to every q (>= 0; the page gives it no value).
 *   ks_max       in [1, 1024]; the page's default is lost, so it is an
 *                argument.
 *   input_is_logits  nonzero: logits, softmax them, removed outputs -inf;
 *                zero: the input already holds probabilities, removed
 *                outputs 0 (the page's defLogit).
 * Outputs (each may be NULL, not all; none may overlap an input, the
 * workspace or another output):
 *   select       device, [B, V] of dtype, row stride ld_select (>= V): the
 *                input element where its position was kept, defLogit
 *                elsewhere (logitsTopKPSelect).
 *   token        device, [B] int32: the sampled original index
 *                (logitsSelectIdx).
 *   logits_idx   device, [B, V] int32, contiguous: the original index of
 *                sorted position j for j < n (n = top_k[b] after a top-k
 *                stage, V otherwise), -1 past n (logitsIdx).
 *   sort_masked  device, [B, V] float, contiguous: the fp32 probability of
 *                each kept sorted position; a position not kept holds 0 when
 *                min-p ran or the input is probabilities, -inf otherwise
 *                (logitsSortMasked).
 *   workspace    device, at least topkp_sample_v2_workspace_size(B, V,
 *                dtype) bytes, 256-byte aligned, owned by the caller (the
 *                rows whose top-k is skipped are sorted into it; the page's
 *                two-stage form).
 * Results.  Probabilities are fp32 from fp32 exponentials; a top-p or min-p
 * decision can differ from exact arithmetic only where the cumulative
 * probability lies within 1e-5 of its threshold (or the probability within
 * 1e-5, relative, of prob[0] * min_p), and the token only where another
 * kept position's prob / (q + eps) lies within 1e-5 (relative) of the
 * largest.  Deterministic.  Three kernel launches.
 */
size_t topkp_sample_v2_workspace_size(int64_t B, int64_t V, topkp_dtype dtype);
topkp_status topkp_sample_v2(const void* logits, int64_t B, int64_t V, int64_t ld_logits, topkp_dtype dtype,
                             const int32_t* top_k, const float* top_p, const float* min_p, const float* q,
                             int64_t ldq, float eps, int32_t ks_max, int32_t input_is_logits, void* select,
                             int64_t ld_select, int32_t* token, int32_t* logits_idx, float* sort_masked,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * topkp_sort -- the sort that aclnnApplyTopKTopP runs before the filter
 * (section 6.1 of the page: l0op::Sort with descending = false and stable =
 * true), producing the inputs of topkp_apply_sorted.  Per row:
 * sorted_value holds the row's elements in ascending order (bits kept, -0
 * and +0 equal), equal values in increasing original index, and
 * sorted_indices[b][j] is the column sorted_value[b][j] came from.
 *
 *   logits          device, [B, V] of dtype, row stride ld_logits (>= V).
 *   B, V, dtype     as for topkp_apply; B == 0 or V == 0 returns
 *                   TOPKP_SUCCESS without a launch.
 *   sorted_value    device, [B, V] contiguous, dtype.
 *   sorted_indices  device, [B, V] contiguous int32.
 *   workspace       device, at least topkp_sort_workspace_size(B, V, dtype)
 *                   bytes, 256-byte aligned, owned by the caller; its contents
 *                   on entry do not matter and are clobbered.  The page's
 *                   two-stage form: ask for the size, then run.
 *   No output may overlap the logits, another output or the workspace.
 * Results are exact (a permutation and its values; no arithmetic).
 */
size_t topkp_sort_workspace_size(int64_t B, int64_t V, topkp_dtype dtype);
topkp_status topkp_sort(const void* logits, int64_t B, int64_t V, int64_t ld_logits, topkp_dtype dtype,
                        void* sorted_value, int32_t* sorted_indices, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * topkp_sort_static -- topkp_sort for callers that cannot allocate device
 * memory when they sort (they run inside a memory pool they do not own, are
 * handed only the tensors they work on, or find the GPU's memory already
 * reserved): the scratch is a fixed 16 MiB array of the library's own device
 * memory, held until the process exits.  The source pages have no
 * counterpart to this call.
 *
 *   logits, B, V, ld_logits, dtype, sorted_value, sorted_indices, stream
 *                   as for topkp_sort.
 *   A problem whose topkp_sort_workspace_size exceeds 16 MiB (for example
 *   more than 18 rows of V = 152064 bf16) is rejected with
 *   TOPKP_ERR_PARAM_INVALID and nothing is launched.
 *   When the array is reserved: the sort's code is a module of its own, and
 *   a GPU reserves the module's 16 MiB when it loads that module.  Under
 *   CUDA's default lazy module loading that happens at the first
 *   topkp_sort or topkp_sort_static call on that device, not when the
 *   library is loaded.  So make one topkp_sort_static call on every device
 *   you will use before handing the rest of its memory to a pool, and before
 *   any stream capture: that first call also looks up the array's device
 *   address (a host call that touches no stream) and keeps it for the
 *   device.  If the device has no 16 MiB left at that point, the call
 *   returns TOPKP_ERR_NO_MEMORY and launches nothing.  The kept address
 *   belongs to the device's context as it was then: after cudaDeviceReset
 *   this entry point must not be called again in the same process.
 *   Every call shares the one array: calls that can overlap on the GPU
 *   (other streams, other host threads) race on it and must be ordered by
 *   the caller.  Nothing of an earlier call's scratch is read.
 */
topkp_status topkp_sort_static(const void* logits, int64_t B, int64_t V, int64_t ld_logits, topkp_dtype dtype,
                               void* sorted_value, int32_t* sorted_indices, void* stream);

/* One-line description of the last non-zero status returned on the calling
 * thread ("" if none).  The pointer stays valid until the thread's next call
 * into the library. */
const char* topkp_last_error_string(void);

/* Waits for all work on stream, then reports (and clears) the device-side
 * error word on the current device: TOPKP_SUCCESS, TOPKP_ERR_DEVICE_TIMEOUT,
 * or TOPKP_ERR_LAUNCH if the stream itself reported a CUDA error. */
topkp_status topkp_device_status(void* stream);

/* Number of kernel launches the most recent successful topkp_apply /
 * topkp_apply_sorted / topkp_sample / topkp_sample_v2 / topkp_sort call on
 * this thread enqueued (0 for an empty problem). */
int topkp_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TOPKP_H */
