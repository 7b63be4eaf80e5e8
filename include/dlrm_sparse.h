/*
 * dlrm_sparse.h -- C ABI of the GB300 (sm_103a) DLRM sparse hot path.
 *
 * The path, as the Deep Learning Recommendation Model is described in
 * "Notes/DLRM" (vault-aram.pages.dev) and in "Terabyte Embedding Tables and
 * Compute-Bound Neural Layers Force Meta's DLRM to Split Training"
 * (factlen.com):
 *   1. embedding-bag forward   (sum-pooled lookups, one table per feature)
 *   2. interaction forward     (pairwise dot products, concatenated with e0)
 *   3. interaction backward
 *   4. embedding-bag backward  (coalescing of duplicate rows + row-wise SGD)
 *
 * Conventions shared by every call:
 *  - Tensor pointers are DEVICE pointers owned by the caller unless a
 *    parameter says "host".  The library never allocates device memory;
 *    scratch space comes from a caller-provided workspace.
 *  - Every compute call is asynchronous on the given stream (a cudaStream_t
 *    passed as void*; NULL is the legacy default stream) and never
 *    synchronizes with the host.
 *  - Host-detectable errors (bad sizes, null pointers, misalignment the call
 *    cannot handle, short workspace) are returned synchronously before
 *    anything is launched.  Data-dependent errors (an index outside its
 *    table, inconsistent offsets) are raised as bits in an optional device
 *    int32 flag; the offending lookup is skipped (it contributes zero), no
 *    kernel faults or traps.  Read the flag with dlrm_read_error().
 *  - Lookups are table-major CSR: bag (t, b) of table t and sample b is
 *    indices[offsets[t*B + b] .. offsets[t*B + b + 1]), offsets has T*B + 1
 *    int64 entries with offsets[0] == 0 and offsets[T*B] == nnz, indices has
 *    nnz int64 row numbers.
 *  - Tables are row-major [rows_t][d] in fp32, fp16 or bf16; pooled values,
 *    interaction values and all gradients are fp32; all accumulation is fp32.
 *  - Return value: DLRM_OK (0) or a negative dlrm_status.
 */
#ifndef DLRM_SPARSE_H
#define DLRM_SPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *dlrm_stream_t; /* a cudaStream_t */

enum dlrm_dtype { DLRM_F32 = 0, DLRM_F16 = 1, DLRM_BF16 = 2, DLRM_INT4 = 3 };

enum dlrm_status {
    DLRM_OK = 0,
    DLRM_ERR_INVALID_ARG = -1,
    DLRM_ERR_UNSUPPORTED = -2,
    DLRM_ERR_WORKSPACE_TOO_SMALL = -3,
    DLRM_ERR_INDEX_OOB = -4,
    DLRM_ERR_BAD_OFFSETS = -5,
    DLRM_ERR_CAPACITY = -6,
    DLRM_ERR_CUDA = -7,
    DLRM_ERR_WAIT_TIMEOUT = -8
};

/* Bits of the device error flag. */
#define DLRM_FLAG_INDEX_OOB 1   /* an index was < 0 or >= rows of its table */
#define DLRM_FLAG_BAD_OFFSETS 2 /* offsets not monotone, or not 0 .. nnz */
#define DLRM_FLAG_CAPACITY 4    /* more unique rows than grad_rows can hold */
#define DLRM_FLAG_WAIT_TIMEOUT 8 /* a kernel gave up waiting on another CTA's result
                                    (every such wait is bounded); outputs invalid */

#define DLRM_MAX_TABLES 256

/*
 * Embedding-bag forward ("Notes/DLRM", section 2: one embedding table per
 * categorical feature, each ID looked up as a learned vector; section 9:
 * multi-valued features are aggregated -- here by summation).
 *
 *   out[b*out_sample_stride + t*out_table_stride + e]
 *       = sum_{k in bag (t,b)} tables[t][indices[k]*d + e]      (fp32 sum)
 *
 * tables    host array of T device pointers, each 16-byte aligned for the
 *           vectorised path (any alignment of the element size works).
 * rows      host array of T row counts (1 .. 2^32-2).
 * T, d      number of tables (1 .. DLRM_MAX_TABLES), embedding dimension.
 * dtype     storage type of all tables (dlrm_dtype).
 * offsets   device int64 [T*B + 1];  indices  device int64 [nnz].
 * out       device fp32, strides in elements; with out_table_stride = d and
 *           out_sample_stride = T*d it is the [B][T][d] pooled block.
 * err_flag  optional device int32 (NULL: no flag); bits are OR-ed in.
 * An empty bag pools to zero.  An out-of-range index contributes zero and
 * sets DLRM_FLAG_INDEX_OOB; a bag with bad offsets pools to zero and sets
 * DLRM_FLAG_BAD_OFFSETS.
 */
int dlrm_emb_bag_fwd(const void *const *tables, const int64_t *rows, int T, int d, int dtype,
                     const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                     float *out, int64_t out_sample_stride, int64_t out_table_stride,
                     int32_t *err_flag, dlrm_stream_t stream);

/*
 * Row-wise int4 tables (DLRM_INT4).  The factlen.com page ("Terabyte Embedding
 * Tables and Compute-Bound Neural Layers Force Meta's DLRM to Split
 * Training", section "Scaling limits and the reality of production") reports
 * 4-bit integer quantization of the vectors; the format here is the row-wise
 * affine codec.
 * A row of d values (d % 8 == 0, d <= 512) takes dlrm_int4_row_bytes(d)
 * bytes: d codes q of 4 bits (element 2j in the low nibble of byte j, 2j+1 in
 * the high nibble), then the row's fp32 scale s and fp32 bias b, then zero
 * padding to a multiple of 16 bytes.  Element e of the row has the value
 * b + s q[e].  An int4 table pointer is 16-byte aligned and holds rows[t]
 * such rows.  dlrm_emb_bag_fwd and dlrm_emb_bag_interact_fwd (two-kernel
 * path) read int4 tables, with the output 16-byte aligned and its strides
 * multiples of 4 (DLRM_ERR_UNSUPPORTED otherwise); the backward calls
 * return DLRM_ERR_UNSUPPORTED for them (4-bit tables are served, not
 * trained).  The pooled sum is fp32: per element the sum of s q, plus the
 * sum of the biases.
 */
int64_t dlrm_int4_row_bytes(int d);  /* -1 for d <= 0 or odd d */

/*
 * Encodes rows x d values (src: device, dtype DLRM_F32/F16/BF16, row stride
 * d, element-aligned) into the int4 layout at dst (device, 16-byte aligned,
 * rows * dlrm_int4_row_bytes(d) bytes).  Per row, in fp32: lo and hi the
 * minimum and maximum (a zero stored as +0), s = (hi - lo) / 15, b = lo, and
 * q = round-half-to-even((w - lo) / s) kept in 0 .. 15 (all 0 when s == 0);
 * the subtraction and the divisions are IEEE-rounded, so the codes are
 * reproducible bit for bit.  Rows are expected to be finite.
 */
int dlrm_quantize_int4(const void *src, int src_dtype, int64_t rows, int d, void *dst, dlrm_stream_t stream);

/*
 * Number of interaction terms over F = N + 1 vectors (e0 and N pooled
 * embeddings): F(F-1)/2 strict pairs, F(F+1)/2 with self pairs
 * ("Notes/DLRM", section 3; N(N+1)/2 there counts the strict pairs of
 * e0..eN).  Bit 0 of include_self selects self pairs (a mode below may be
 * passed).  Returns -1 if N < 0.
 */
int64_t dlrm_num_pairs(int N, int include_self);

/*
 * Interaction modes (bits of the `mode` argument of the interaction calls).
 * DLRM_INTERACT_SELF: self pairs z_i . z_i are included.
 * DLRM_INTERACT_ALONGSIDE: the original embeddings are concatenated
 *   alongside the interaction vector ("Notes/DLRM", section 3 names this
 *   variant; its order is not given there): an output row is
 *   [e0 | e_1 .. e_N | pairs] instead of [e0 | pairs].
 */
#define DLRM_INTERACT_SELF 1
#define DLRM_INTERACT_ALONGSIDE 2

/* Width of an interaction output row: d (or d (N + 1) alongside) plus the
 * pairs.  Returns -1 for N < 0, d <= 0 or unknown mode bits. */
int64_t dlrm_interact_width(int N, int d, int mode);

/*
 * Interaction forward ("Notes/DLRM", section 3, and the architecture figure
 * of section 2).  With z_0 = e0[b] and z_i = emb[b][i-1] (i = 1..N):
 *
 *   y[b][0 .. d)       = e0[b]                    (the concatenated e0)
 *   y[b][i*d .. i*d+d) = z_i, i = 1..N             (DLRM_INTERACT_ALONGSIDE only)
 *   y[b][o + p(i,j)]   = z_i . z_j  for j < i, or j <= i with DLRM_INTERACT_SELF
 *   p(i,j)             = i(i-1)/2 + j (strict),  i(i+1)/2 + j (self pairs)
 *   o                  = d, or (N + 1) d alongside
 *
 * mode  bits DLRM_INTERACT_SELF | DLRM_INTERACT_ALONGSIDE (0: strict pairs
 *       after e0; 1 selects self pairs as a boolean did before).
 * e0    device fp32 rows of d, row stride e0_stride (elements).
 * emb   device fp32; pooled embedding i of sample b at
 *       emb[b*emb_sample_stride + i*d] (the [B][N][d] block of
 *       dlrm_emb_bag_fwd with out_table_stride = d).
 * y     device fp32 rows of dlrm_interact_width(N, d, mode), row stride
 *       y_stride.  N may be 0 .. 127.
 * The kernels that stage operands through mbarrier-tracked copies wait only
 * on their own CTA's copies and MMAs, and every such wait is bounded; should
 * one run out, the samples of that CTA get NaN outputs (this call has no
 * error flag), so a failure is visible rather than silent.
 */
int dlrm_interact_fwd(const float *e0, int64_t e0_stride, const float *emb,
                      int64_t emb_sample_stride, int N, int d, int64_t B, int mode,
                      float *y, int64_t y_stride, dlrm_stream_t stream);

/*
 * Interaction backward: the gradient of the forward above by the product
 * rule.  With G the F x F matrix holding dy[b][o + p(i,j)] at (i, j), j <= i,
 * and zero above the diagonal:
 *
 *   dZ        = (G + G^T) Z        (a self term contributes 2 g_ii z_i)
 *   de0[b]    = dy[b][0 .. d) + dZ[0]
 *   demb[b*demb_sample_stride + (i-1)*d + e] = dZ[i][e]     (i = 1..N)
 *               + dy[b][i*d + e]   (alongside: the gradient of the copy)
 *
 * Inputs as in dlrm_interact_fwd; dy has row stride dy_stride, de0 row
 * stride de0_stride.  Outputs are overwritten (not accumulated).  Bounded
 * waits as in dlrm_interact_fwd (NaN outputs if one runs out).
 */
int dlrm_interact_bwd(const float *e0, int64_t e0_stride, const float *emb,
                      int64_t emb_sample_stride, int N, int d, int64_t B, int mode,
                      const float *dy, int64_t dy_stride, float *de0, int64_t de0_stride,
                      float *demb, int64_t demb_sample_stride, dlrm_stream_t stream);

/*
 * Kernel family of dlrm_interact_fwd and dlrm_interact_bwd (a process-wide
 * setting, for benchmarking and testing the alternatives).
 * DLRM_INTERACT_KERNEL_AUTO (the default): the tensor-core kernels where they
 * apply -- 16-byte aligned operands, d and the row strides multiples of 4 --
 * else the CUDA-core kernels.  The tensor-core kernels run TF32 MMAs on a
 * hi + lo split of every fp32 operand, which carries each product z_i.z_j to
 * about 2^-21 of |z_i||z_j|, with fp32 accumulation.
 * DLRM_INTERACT_KERNEL_CUDA_CORE: always the CUDA-core kernels (fp32 FMAs).
 * dlrm_set_interact_kernel returns DLRM_OK, or DLRM_ERR_INVALID_ARG for an
 * unknown value (the setting is then unchanged); calls already enqueued are
 * not affected.  dlrm_get_interact_kernel returns the setting.
 */
#define DLRM_INTERACT_KERNEL_AUTO 0
#define DLRM_INTERACT_KERNEL_CUDA_CORE 1
int dlrm_set_interact_kernel(int kind);
int dlrm_get_interact_kernel(void);

/*
 * Embedding-bag forward and interaction forward in one call ("Notes/DLRM",
 * section 3: the interaction directly follows the lookups).  Computes what
 * dlrm_emb_bag_fwd followed by dlrm_interact_fwd with N = T computes:
 *
 *   pooled[b][t] = sum_{k in bag (t,b)} tables[t][indices[k]]      (fp32)
 *   y[b]         = [ e0[b] | z_i . z_j over the pairs (i, j) ]     (z_0 = e0[b],
 *                                                                   z_i = pooled[b][i-1])
 *
 * without writing the pooled block unless `pooled` is given (the backward
 * needs it; inference does not).  Arguments as in those two calls; pooled is
 * optional (NULL: not written), with strides in elements.  The pooled values
 * equal dlrm_emb_bag_fwd's bit for bit; y equals dlrm_interact_fwd's within
 * the accuracy of the two (fp32 dot products summed in another order, or the
 * tensor-core split's 2^-20 of |z_i||z_j| per product).  When `pooled` is
 * given (pooled_table_stride == d) and the tensor-core interaction takes the
 * operands, the call runs the lookup into `pooled` and then that interaction:
 * in training the pooled block is written anyway, and the tensor-core
 * interaction is faster than the single kernel's CUDA-core dot products.
 * T may be 1 .. 127.  The single-kernel path needs rows of a whole number of
 * 16-byte chunks up to 1 KB, 16-byte aligned tables (and pooled, with
 * strides that are multiples of 4), and a Z block of each sample that fits
 * on chip (about (T + 1) <= 32 with d <= 256); otherwise the call runs the
 * two kernels through `pooled`, which must then be given with
 * pooled_table_stride == d, else DLRM_ERR_UNSUPPORTED.  Errors are flagged
 * as in dlrm_emb_bag_fwd.
 */
int dlrm_emb_bag_interact_fwd(const void *const *tables, const int64_t *rows, int T, int d, int dtype,
                              const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                              const float *e0, int64_t e0_stride, int mode, float *y,
                              int64_t y_stride, float *pooled, int64_t pooled_sample_stride,
                              int64_t pooled_table_stride, int32_t *err_flag, dlrm_stream_t stream);

/*
 * Device pointers into the workspace of the last dlrm_emb_bag_bwd_sgd call,
 * valid once the stream has passed that call and until the workspace is
 * reused.  The coalescing is a stable sort of lookup positions by
 * (table, row) followed by run-length encoding; U = *num_unique.
 */
typedef struct dlrm_coalesced_view {
    const uint32_t *sorted_pos; /* [nnz] positions k, sorted; ties keep position order */
    const uint32_t *sorted_row; /* [nnz] indices[sorted_pos[j]] */
    const int32_t *uniq_table;  /* [U] table of each unique key, ascending */
    const uint32_t *uniq_row;   /* [U] row of each unique key, ascending within a table */
    const uint32_t *seg_off;    /* [U + 1] first sorted position of each key; [U] = nnz */
    const int64_t *num_unique;  /* [1] U */
} dlrm_coalesced_view;

/*
 * Bytes of workspace dlrm_emb_bag_bwd_sgd needs for these sizes (a bound
 * that does not depend on the data).  Returns 0 for invalid sizes.
 */
size_t dlrm_emb_bag_bwd_workspace_size(int T, int64_t B, int64_t nnz, int d);

/*
 * The coalescing's sort for these sizes (host only, no device work): into
 * *passes the number of LSD radix passes over the row bits (1 to 4, digits of
 * at most 8 bits), into *msd 1 when the sort instead orders the keys by the
 * top 8 row bits in one pass and then sorts each table's 256 buckets in
 * shared memory (rows of 17 bits or more, every table above half the
 * largest power of two, and 256 to 2560 keys per bucket on average), else 0.
 * The LSD passes are launched either way: when the digit counts show a bucket
 * of more than 4096 keys the first launch sorts by the lowest digit and the
 * LSD passes run, else they return at once.  Both orders are the same stable
 * sort.  rows: host array of T row counts.  Returns DLRM_OK, or
 * DLRM_ERR_INVALID_ARG for invalid sizes or null pointers.
 */
int dlrm_emb_bag_sort_plan(const int64_t *rows, int T, int64_t nnz, int *passes, int *msd);

/*
 * Embedding-bag backward with row-wise SGD ("Notes/DLRM", section 5: the
 * tables are trained by an optimizer; plain SGD on the touched rows here).
 * Duplicate lookups are coalesced first (stable radix sort by (table, row),
 * run-length encoding), then for every unique key u = (t, r):
 *
 *   g_u = sum over the lookups k of r in table t, in sorted order, of
 *         dpooled[b(k)*dp_sample_stride + t*dp_table_stride + 0 .. d)
 *   tables[t][r] <- tables[t][r] - lr * g_u
 *
 * Rounding of the update: fp32 and fp16 tables receive the step -lr * g_u
 * (computed in fp32, rounded to the table type, nearest even) as one
 * reduction performed in L2, which rounds the sum once more; bf16 tables are
 * read, updated in fp32 (one fused multiply-add) and written back with one
 * rounding.  Every unique row is updated exactly once per call, so results
 * are reproducible bit for bit from run to run.
 *
 * Rows no lookup touches are not written.  lr == 0 leaves the tables
 * untouched (the coalesced gradient only).
 * grad_rows      optional device fp32 [grad_rows_cap][d]: receives g_u in
 *                row u; if U > grad_rows_cap the rows past the cap are not
 *                written and DLRM_FLAG_CAPACITY is raised.
 * workspace      device memory of at least
 *                dlrm_emb_bag_bwd_workspace_size(T, B, nnz, d) bytes,
 *                256-byte aligned; its content need not be initialised.
 * view           optional host struct, filled with device pointers to the
 *                integer results of the coalescing (see above).
 * nnz may be at most 2^31 and B at most 2^31 - 1 (DLRM_ERR_UNSUPPORTED
 * beyond); B == 0 requires nnz == 0.  The sort's CTAs wait on the results of
 * earlier CTAs of the same launch, each wait bounded; one that runs out
 * raises DLRM_FLAG_WAIT_TIMEOUT (results then invalid, all writes still
 * inside the workspace and the tables' touched rows).  The vectorised path needs d % 4 == 0,
 * 16-byte aligned tables, dpooled and grad_rows, and dpooled strides that are
 * multiples of 4; other layouts take a scalar path.
 */
int dlrm_emb_bag_bwd_sgd(void *const *tables, const int64_t *rows, int T, int d, int dtype,
                         const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                         const float *dpooled, int64_t dp_sample_stride, int64_t dp_table_stride,
                         float lr, float *grad_rows, int64_t grad_rows_cap, void *workspace,
                         size_t workspace_bytes, dlrm_coalesced_view *view, int32_t *err_flag,
                         dlrm_stream_t stream);

/*
 * Embedding-bag backward with row-wise SGD applied by atomic reductions, for
 * fp32 tables ("Notes/DLRM", section 5: the tables are trained by an
 * optimizer; the same plain SGD on the touched rows as dlrm_emb_bag_bwd_sgd,
 * without coalescing the duplicate lookups first):
 *
 *   tables[t][r] += -lr * dpooled[b][t]   for every lookup of row r in bag (t, b)
 *
 * Each bag's pooled gradient is read once; lookups of one row within a group
 * of a bag's indices are merged, and every (bag, row) pair adds its share to
 * the row with fp32 vector reductions performed in L2.  No sort, no
 * workspace, no coalesced gradient (no grad_rows, no view).
 *  - dtype must be DLRM_F32 (DLRM_ERR_UNSUPPORTED otherwise): a half-precision
 *    table would be rounded at every reduction.
 *  - A row touched by k bags receives k fp32 additions in an unspecified
 *    order: the result is not reproducible bit for bit from run to run, and
 *    its rounding error grows with k (about k * 2^-24 of |w| + |lr| * sum |g|
 *    at worst), against one rounding in dlrm_emb_bag_bwd_sgd.  It suits index
 *    streams spread over large tables (few lookups per row, as uniform
 *    indices over tables much larger than the batch's lookups); skewed
 *    streams, whose hot rows collect thousands of additions, are better served
 *    by dlrm_emb_bag_bwd_sgd.  The reductions flush subnormal values to zero.
 *  - lr == 0 or B == 0: nothing is launched.  Errors are flagged as in
 *    dlrm_emb_bag_fwd (an out-of-range lookup is skipped; a bag with bad
 *    offsets adds nothing); arguments otherwise as in dlrm_emb_bag_bwd_sgd.
 * The vectorised path needs d % 4 == 0, 16-byte aligned tables and dpooled,
 * and dpooled strides that are multiples of 4; other layouts take a scalar
 * path.
 */
int dlrm_emb_bag_bwd_sgd_atomic(void *const *tables, const int64_t *rows, int T, int d, int dtype,
                                const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                                const float *dpooled, int64_t dp_sample_stride, int64_t dp_table_stride,
                                float lr, int32_t *err_flag, dlrm_stream_t stream);

/*
 * The two halves of dlrm_emb_bag_bwd_sgd, for callers that overlap them with
 * other work.  dlrm_emb_bag_coalesce does the coalescing (the stable sort by
 * (table, row) and the run-length encoding) into the workspace; it reads only
 * rows, offsets and indices -- not the tables or the gradients -- so it can
 * run on a second stream while the forward and interaction kernels run, or
 * one step ahead.  dlrm_emb_bag_reduce_sgd then sums the pooled gradients of
 * each run and applies the update, exactly as dlrm_emb_bag_bwd_sgd would.
 *  - Both calls take the same T, d, nnz and B, and the same workspace
 *    (dlrm_emb_bag_bwd_workspace_size bytes, 256-byte aligned); the reduce
 *    must be given the rows the coalescing was given and be ordered after it
 *    on the GPU (same stream, or an event).  None of this is checked.
 *  - The workspace holds one coalescing at a time: a second coalesce into it
 *    before the reduce has run replaces the first.
 *  - The view (optional) is filled by the coalesce call, as in
 *    dlrm_emb_bag_bwd_sgd.
 */
int dlrm_emb_bag_coalesce(const int64_t *rows, int T, int d, const int64_t *offsets, const int64_t *indices,
                          int64_t nnz, int64_t B, void *workspace, size_t workspace_bytes,
                          dlrm_coalesced_view *view, int32_t *err_flag, dlrm_stream_t stream);
int dlrm_emb_bag_reduce_sgd(void *const *tables, const int64_t *rows, int T, int d, int dtype, int64_t nnz,
                            int64_t B, const float *dpooled, int64_t dp_sample_stride,
                            int64_t dp_table_stride, float lr, float *grad_rows, int64_t grad_rows_cap,
                            void *workspace, size_t workspace_bytes, int32_t *err_flag,
                            dlrm_stream_t stream);

/*
 * Embedding-bag backward with row-wise AdaGrad ("Notes/DLRM", section 5: the
 * optimizer is typically adaptive, Adam or AdaGrad; the notes give no
 * formula, and this is AdaGrad with one accumulator per row).  The coalescing
 * and the coalesced gradient g_u are those of dlrm_emb_bag_bwd_sgd; then, for
 * every unique key u = (t, r), in fp32:
 *
 *   state[t][r] <- s' = state[t][r] + (1/d) sum_e g_u[e]^2
 *   tables[t][r][e] <- tables[t][r][e] - lr * g_u[e] / (sqrt(s') + eps)
 *
 * The row update rounds as dlrm_emb_bag_bwd_sgd's does, with the step
 * lr / (sqrt(s') + eps) in place of lr: fp32 and fp16 rows by one L2
 * reduction of the rounded step (two roundings), bf16 rows by one fused
 * multiply-add and one rounding.  The accumulator is rounded once (fp32).
 *
 * state   host array of T device pointers, each fp32 [rows[t]], 4-byte
 *         aligned: the accumulators, updated in place for touched rows only
 *         (start them at 0 for plain AdaGrad).
 * eps     > 0 and finite (it keeps the step of an all-zero gradient at 0).
 * lr == 0 leaves tables and accumulators untouched.  d may be at most 256
 * (DLRM_ERR_UNSUPPORTED beyond): the update needs a row's whole gradient in
 * registers.  The other arguments are those of dlrm_emb_bag_bwd_sgd;
 * dlrm_emb_bag_reduce_adagrad is the reduce half, used after
 * dlrm_emb_bag_coalesce exactly as dlrm_emb_bag_reduce_sgd is.
 */
int dlrm_emb_bag_bwd_adagrad(void *const *tables, float *const *state, const int64_t *rows, int T, int d,
                             int dtype, const int64_t *offsets, const int64_t *indices, int64_t nnz,
                             int64_t B, const float *dpooled, int64_t dp_sample_stride,
                             int64_t dp_table_stride, float lr, float eps, float *grad_rows,
                             int64_t grad_rows_cap, void *workspace, size_t workspace_bytes,
                             dlrm_coalesced_view *view, int32_t *err_flag, dlrm_stream_t stream);
int dlrm_emb_bag_reduce_adagrad(void *const *tables, float *const *state, const int64_t *rows, int T, int d,
                                int dtype, int64_t nnz, int64_t B, const float *dpooled,
                                int64_t dp_sample_stride, int64_t dp_table_stride, float lr, float eps,
                                float *grad_rows, int64_t grad_rows_cap, void *workspace,
                                size_t workspace_bytes, int32_t *err_flag, dlrm_stream_t stream);

/*
 * dlrm_emb_bag_bwd_sgd for callers that cannot allocate device memory (the
 * pages have no counterpart to this; it is a deployment aid).  Some callers
 * can neither call cudaMalloc nor hand the library a workspace -- a plugin
 * whose host framework passes it only its input and output tensors and owns
 * every device allocation, or a service that must not touch the device
 * allocator once it runs.  This variant computes exactly what
 * dlrm_emb_bag_bwd_sgd computes, with the same arguments minus the workspace,
 * and allocates nothing: its scratch is a fixed array of
 * DLRM_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.
 *  - The status of every refused call is the one dlrm_emb_bag_bwd_sgd returns
 *    for the same arguments and a workspace of DLRM_NOALLOC_SCRATCH_BYTES:
 *    sizes whose scratch would not fit (dlrm_emb_bag_bwd_workspace_size(T, B,
 *    nnz, d) > DLRM_NOALLOC_SCRATCH_BYTES; about 1.7M lookups at d = 128) are
 *    refused with DLRM_ERR_WORKSPACE_TOO_SMALL, before the device is touched.
 *  - Each call looks up the array's device address (a CUDA runtime query,
 *    made with the calling device current).  With lazily loaded modules (the
 *    CUDA default) the first call on a device is the one that loads the
 *    module and makes the array resident there, so it can fail with
 *    DLRM_ERR_CUDA when the device has no memory left.  A service that must
 *    not claim device memory once it runs should make one small call at
 *    start-up (nnz = 0 is enough) and before any stream capture.
 *  - All calls share the array and it keeps the last call's contents; the
 *    call re-initialises what it needs.  Calls that may run at the same time
 *    on the GPU (different streams with no ordering between them) race on it
 *    and must not be issued.  The view, if requested, points into the array
 *    and is valid until the next call.
 */
#define DLRM_NOALLOC_SCRATCH_BYTES (64 * 1024 * 1024)
int dlrm_emb_bag_bwd_sgd_noalloc(void *const *tables, const int64_t *rows, int T, int d, int dtype,
                                 const int64_t *offsets, const int64_t *indices, int64_t nnz,
                                 int64_t B, const float *dpooled, int64_t dp_sample_stride,
                                 int64_t dp_table_stride, float lr, float *grad_rows,
                                 int64_t grad_rows_cap, dlrm_coalesced_view *view,
                                 int32_t *err_flag, dlrm_stream_t stream);

/*
 * Testing aid (the pages have no counterpart): makes the kernels' bounded
 * waits run out on purpose, so that a test can check what a wait that gives
 * up does.  A process-wide setting, read when a call launches its kernels;
 * calls already enqueued are not affected.  Results of calls made while a
 * hook is set are invalid; set all three back to their defaults (-1, 0, -1)
 * afterwards.
 *  sort_wait_polls   polls of one look-back word by the radix sort's passes
 *                    before the wait gives up (negative: the default, about
 *                    a second; at most the default).
 *  sort_first_tile   the first tile the passes claim (0: normal).  k > 0
 *                    leaves tiles 0 .. k-1 unclaimed, so the pass's tile k
 *                    waits for counts that never come and gives up:
 *                    DLRM_FLAG_WAIT_TIMEOUT is raised, every write stays in
 *                    the workspace, and the reduce that follows updates no
 *                    table row (it checks the coalescing's failure word).
 *  copy_wait_polls   polls of a stage barrier in the main loop of the
 *                    bulk-copy (CUDA-core) interaction forward (negative: the
 *                    default; 0: give up at once).  A CTA that gives up waits,
 *                    with the default limit, for its copies in flight, writes
 *                    NaN into its samples' pair outputs and returns.
 * Returns DLRM_OK, or DLRM_ERR_INVALID_ARG for a negative sort_first_tile.
 */
int dlrm_set_wait_test_hooks(int64_t sort_wait_polls, int sort_first_tile, int64_t copy_wait_polls);

/* Synchronizes the stream, reads the flag and maps its bits to a status
 * (DLRM_OK if no bit is set).  A CUDA failure returns DLRM_ERR_CUDA. */
int dlrm_read_error(const int32_t *err_flag, dlrm_stream_t stream);

/* Clears the flag asynchronously on the stream. */
int dlrm_clear_error(int32_t *err_flag, dlrm_stream_t stream);

/* Static, human-readable name of a status code. */
const char *dlrm_status_string(int status);

/* Number of kernels this library has launched in this process so far. */
uint64_t dlrm_kernel_launch_count(void);

/*
 * Profiling aid (the pages have no counterpart): registers n cudaEvent_t
 * handles (passed as void*) for the calling host thread.  After each of the
 * next n kernel launches the library makes on this thread, it records the
 * next event on that launch's stream, so a caller can time every kernel of a
 * multi-kernel call with events of its own.  n = 0 unregisters.  The events
 * stay owned by the caller; at most DLRM_MAX_PROFILE_EVENTS.
 */
#define DLRM_MAX_PROFILE_EVENTS 64
int dlrm_profile_events(void *const *events, int n);

#ifdef __cplusplus
}
#endif

#endif /* DLRM_SPARSE_H */
