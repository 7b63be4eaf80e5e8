// C ABI of the DLRM sparse path: argument checks and dispatch.
//
// Every check here runs on the host before anything is launched, so a call
// with bad sizes or pointers returns an error without touching the GPU.
#include <atomic>
#include <cstring>

#include "common.cuh"

namespace dlrm {

static std::atomic<uint64_t> g_launches{0};

// Profiling events registered by the calling host thread.
static thread_local cudaEvent_t g_prof_events[DLRM_MAX_PROFILE_EVENTS];
static thread_local int g_prof_n = 0, g_prof_next = 0;

void count_launch(cudaStream_t st)
{
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (g_prof_next < g_prof_n)
        cudaEventRecord(g_prof_events[g_prof_next++], st);
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? DLRM_OK : DLRM_ERR_CUDA; }

int allow_dynamic_smem(const void *kernel, int bytes, std::atomic<unsigned long long> *done)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DLRM_ERR_CUDA;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;  // devices past 64: set every time
    if (bit && (done->load(std::memory_order_acquire) & bit))
        return DLRM_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return DLRM_ERR_CUDA;
    done->fetch_or(bit, std::memory_order_release);
    return DLRM_OK;
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 1;
    return n;
}

static std::atomic<int> g_interact_kernel{DLRM_INTERACT_KERNEL_AUTO};

// testing hook of the bounded waits (negative: the kernel's default)
static std::atomic<int64_t> g_hook_sort_polls{-1}, g_hook_copy_polls{-1};
static std::atomic<uint32_t> g_hook_first_tile{0};

WaitHooks wait_hooks(int default_sort_polls, int default_copy_polls)
{
    WaitHooks h;
    const int64_t sp = g_hook_sort_polls.load(std::memory_order_relaxed);
    const int64_t cp = g_hook_copy_polls.load(std::memory_order_relaxed);
    h.sort_polls = sp < 0 ? default_sort_polls : (int)(sp < default_sort_polls ? sp : default_sort_polls);
    h.copy_polls = cp < 0 ? default_copy_polls : (int)(cp < default_copy_polls ? cp : default_copy_polls);
    h.sort_first_tile = g_hook_first_tile.load(std::memory_order_relaxed);
    return h;
}

bool interact_tensor_cores() { return g_interact_kernel.load(std::memory_order_relaxed) == DLRM_INTERACT_KERNEL_AUTO; }

// kernels (defined in the other translation units)
bool emb_bag_fwd_vectorisable(const TableSet &, int, int, int, const float *, int64_t, int64_t);
int64_t int4_row_bytes(int);
int launch_emb_bag_fwd_int4(const TableSet &, int, int, const int64_t *, const int64_t *, int64_t, int64_t, float *,
                            int64_t, int64_t, int32_t *, cudaStream_t);
int launch_quantize_int4(const void *, int, int64_t, int, void *, cudaStream_t);
int launch_emb_bag_fwd(const TableSet &, int, int, int, bool, const int64_t *, const int64_t *, int64_t,
                       int64_t, float *, int64_t, int64_t, int32_t *, cudaStream_t);
int launch_interact_fwd(const float *, int64_t, const float *, int64_t, int, int, int64_t, int, float *,
                        int64_t, cudaStream_t);
int launch_interact_bwd(const float *, int64_t, const float *, int64_t, int, int, int64_t, int,
                        const float *, int64_t, float *, int64_t, float *, int64_t, cudaStream_t);
struct FusedShape {
    int S, KS, threads;
    size_t smem;
};
bool emb_bag_interact_shape(int, int, int, int64_t, FusedShape &);
bool interact_fwd_tc_applies(const float *, int64_t, const float *, int64_t, int, int, int64_t);
int launch_emb_bag_interact_fwd(const TableSet &, int, int, int, const int64_t *, const int64_t *, int64_t,
                                int64_t, const float *, int64_t, int, float *, int64_t, float *, int64_t, int64_t,
                                const FusedShape &, int32_t *, cudaStream_t);
bool emb_bag_bwd_vectorisable(const TableSet &, int, int, const float *, int64_t, int64_t, const float *);
size_t emb_bag_bwd_workspace(int, int64_t, int);
void coalesce_plan(const int64_t *, int, int64_t, int &, bool &);
int launch_emb_bag_bwd(const TableSet &, int, int, int, const int64_t *, const int64_t *, int64_t, int64_t,
                       const float *, int64_t, int64_t, float, float *, int64_t, void *, bool,
                       dlrm_coalesced_view *, int32_t *, cudaStream_t);
int launch_coalesce(const TableSet &, int, int, const int64_t *, const int64_t *, int64_t, int64_t, void *,
                    dlrm_coalesced_view *, int32_t *, cudaStream_t);
int launch_reduce_sgd(const TableSet &, int, int, int, int64_t, int64_t, const float *, int64_t, int64_t, float,
                      float *, int64_t, void *, bool, int32_t *, cudaStream_t, float, float *const *);
int launch_emb_bag_bwd_atomic(const TableSet &, int, int, const int64_t *, const int64_t *, int64_t, int64_t,
                              const float *, int64_t, int64_t, float, bool, int32_t *, cudaStream_t);

// Lookup positions are 32-bit in the backward's sort and scans; the bound
// leaves headroom for tile and chunk arithmetic.
static const int64_t kMaxLookups = (int64_t)1 << 31;

static int elem_bytes(int dtype) { return dtype == DLRM_F32 ? 4 : 2; }  // of the float table types

static const int kInt4MaxD = 512;  // 32 lanes of 16 codes

static bool aligned(const void *p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// Common checks of the table arguments; fills the kernel-parameter view.
int make_tables(const void *const *tables, const int64_t *rows, int T, int d, int dtype, TableSet &ts)
{
    if (!tables || !rows || T <= 0 || d <= 0)
        return DLRM_ERR_INVALID_ARG;
    if (dtype != DLRM_F32 && dtype != DLRM_F16 && dtype != DLRM_BF16 && dtype != DLRM_INT4)
        return DLRM_ERR_INVALID_ARG;
    if (dtype == DLRM_INT4 && d % 2 != 0)
        return DLRM_ERR_INVALID_ARG;
    if (T > DLRM_MAX_TABLES || (dtype == DLRM_INT4 && (d % 8 != 0 || d > kInt4MaxD)))
        return DLRM_ERR_UNSUPPORTED;
    std::memset(&ts, 0, sizeof ts);
    for (int t = 0; t < T; t++) {
        if (!tables[t] || rows[t] <= 0)
            return DLRM_ERR_INVALID_ARG;
        if (rows[t] > (int64_t)0xfffffffeLL)
            return DLRM_ERR_UNSUPPORTED;
        if (!aligned(tables[t], dtype == DLRM_INT4 ? 16 : (size_t)elem_bytes(dtype)))
            return DLRM_ERR_INVALID_ARG;
        ts.ptr[t] = tables[t];
        ts.rows[t] = rows[t];
    }
    return DLRM_OK;
}

// The pooled lookup into out, for every table type.
static int launch_lookup(const TableSet &ts, int T, int d, int dtype, const int64_t *offsets, const int64_t *indices,
                         int64_t nnz, int64_t B, float *out, int64_t oss, int64_t ots, int32_t *err, cudaStream_t st)
{
    if (dtype == DLRM_INT4) {
        if (!aligned(out, 16) || oss % 4 != 0 || ots % 4 != 0)
            return DLRM_ERR_UNSUPPORTED;
        return launch_emb_bag_fwd_int4(ts, T, d, offsets, indices, nnz, B, out, oss, ots, err, st);
    }
    const bool vec = emb_bag_fwd_vectorisable(ts, T, d, elem_bytes(dtype), out, oss, ots);
    return launch_emb_bag_fwd(ts, T, d, dtype, vec, offsets, indices, nnz, B, out, oss, ots, err, st);
}

}  // namespace dlrm

using namespace dlrm;

extern "C" {

int dlrm_emb_bag_fwd(const void *const *tables, const int64_t *rows, int T, int d, int dtype,
                     const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                     float *out, int64_t out_sample_stride, int64_t out_table_stride,
                     int32_t *err_flag, dlrm_stream_t stream)
{
    TableSet ts;
    int s = make_tables(tables, rows, T, d, dtype, ts);
    if (s != DLRM_OK)
        return s;
    if (B < 0 || nnz < 0 || out_sample_stride < 0 || out_table_stride < 0)
        return DLRM_ERR_INVALID_ARG;
    if (B == 0)
        return DLRM_OK;
    if (!offsets || !out || (nnz > 0 && !indices) || !aligned(out, 4))
        return DLRM_ERR_INVALID_ARG;
    if (!aligned(offsets, 8) || (indices && !aligned(indices, 8)))
        return DLRM_ERR_INVALID_ARG;
    return launch_lookup(ts, T, d, dtype, offsets, indices, nnz, B, out, out_sample_stride, out_table_stride,
                         err_flag, static_cast<cudaStream_t>(stream));
}

int64_t dlrm_int4_row_bytes(int d)
{
    if (d <= 0 || d % 2 != 0)
        return -1;
    return int4_row_bytes(d);
}

int dlrm_quantize_int4(const void *src, int src_dtype, int64_t rows, int d, void *dst, dlrm_stream_t stream)
{
    if (rows < 0 || d <= 0 || d % 2 != 0)
        return DLRM_ERR_INVALID_ARG;
    if (src_dtype != DLRM_F32 && src_dtype != DLRM_F16 && src_dtype != DLRM_BF16)
        return DLRM_ERR_INVALID_ARG;
    if (d % 8 != 0 || d > kInt4MaxD)
        return DLRM_ERR_UNSUPPORTED;
    if (rows == 0)
        return DLRM_OK;
    if (!src || !dst || !aligned(src, (size_t)elem_bytes(src_dtype)) || !aligned(dst, 16))
        return DLRM_ERR_INVALID_ARG;
    return launch_quantize_int4(src, src_dtype, rows, d, dst, static_cast<cudaStream_t>(stream));
}

int64_t dlrm_num_pairs(int N, int include_self)
{
    if (N < 0)
        return -1;
    const int64_t F = (int64_t)N + 1;
    return (include_self & DLRM_INTERACT_SELF) ? F * (F + 1) / 2 : F * (F - 1) / 2;
}

static int check_interact(const float *e0, int64_t e0_stride, const float *emb, int64_t emb_sample_stride,
                          int N, int d, int64_t B)
{
    if (N < 0 || d <= 0 || B < 0 || e0_stride < d || (N > 0 && emb_sample_stride < (int64_t)N * d))
        return DLRM_ERR_INVALID_ARG;
    if (N > 127 || B > (int64_t)1 << 31)
        return DLRM_ERR_UNSUPPORTED;
    if (B > 0 && (!e0 || (N > 0 && !emb)))
        return DLRM_ERR_INVALID_ARG;
    if (!aligned(e0, 4) || !aligned(emb, 4))
        return DLRM_ERR_INVALID_ARG;
    return DLRM_OK;
}

int64_t dlrm_interact_width(int N, int d, int mode)
{
    if (N < 0 || d <= 0 || (mode & ~(DLRM_INTERACT_SELF | DLRM_INTERACT_ALONGSIDE)))
        return -1;
    return (int64_t)d * ((mode & DLRM_INTERACT_ALONGSIDE) ? (int64_t)N + 1 : 1) +
           dlrm_num_pairs(N, mode & DLRM_INTERACT_SELF);
}

int dlrm_set_interact_kernel(int kind)
{
    if (kind != DLRM_INTERACT_KERNEL_AUTO && kind != DLRM_INTERACT_KERNEL_CUDA_CORE)
        return DLRM_ERR_INVALID_ARG;
    dlrm::g_interact_kernel.store(kind, std::memory_order_relaxed);
    return DLRM_OK;
}

int dlrm_get_interact_kernel(void) { return dlrm::g_interact_kernel.load(std::memory_order_relaxed); }

int dlrm_set_wait_test_hooks(int64_t sort_wait_polls, int sort_first_tile, int64_t copy_wait_polls)
{
    if (sort_first_tile < 0)
        return DLRM_ERR_INVALID_ARG;
    dlrm::g_hook_sort_polls.store(sort_wait_polls < 0 ? -1 : sort_wait_polls, std::memory_order_relaxed);
    dlrm::g_hook_copy_polls.store(copy_wait_polls < 0 ? -1 : copy_wait_polls, std::memory_order_relaxed);
    dlrm::g_hook_first_tile.store((uint32_t)sort_first_tile, std::memory_order_relaxed);
    return DLRM_OK;
}

int dlrm_interact_fwd(const float *e0, int64_t e0_stride, const float *emb, int64_t emb_sample_stride,
                      int N, int d, int64_t B, int mode, float *y, int64_t y_stride,
                      dlrm_stream_t stream)
{
    int s = check_interact(e0, e0_stride, emb, emb_sample_stride, N, d, B);
    if (s != DLRM_OK)
        return s;
    const int64_t width = dlrm_interact_width(N, d, mode);
    if (width < 0 || y_stride < width || (B > 0 && !y) || !aligned(y, 4))
        return DLRM_ERR_INVALID_ARG;
    if (B == 0)
        return DLRM_OK;
    return launch_interact_fwd(e0, e0_stride, emb, emb_sample_stride, N, d, B, mode, y, y_stride,
                               static_cast<cudaStream_t>(stream));
}

int dlrm_interact_bwd(const float *e0, int64_t e0_stride, const float *emb, int64_t emb_sample_stride,
                      int N, int d, int64_t B, int mode, const float *dy, int64_t dy_stride,
                      float *de0, int64_t de0_stride, float *demb, int64_t demb_sample_stride,
                      dlrm_stream_t stream)
{
    int s = check_interact(e0, e0_stride, emb, emb_sample_stride, N, d, B);
    if (s != DLRM_OK)
        return s;
    const int64_t width = dlrm_interact_width(N, d, mode);
    if (width < 0 || dy_stride < width || de0_stride < d ||
        (N > 0 && demb_sample_stride < (int64_t)N * d))
        return DLRM_ERR_INVALID_ARG;
    if (B > 0 && (!dy || !de0 || (N > 0 && !demb)))
        return DLRM_ERR_INVALID_ARG;
    if (!aligned(dy, 4) || !aligned(de0, 4) || !aligned(demb, 4))
        return DLRM_ERR_INVALID_ARG;
    if (B == 0)
        return DLRM_OK;
    return launch_interact_bwd(e0, e0_stride, emb, emb_sample_stride, N, d, B, mode, dy,
                               dy_stride, de0, de0_stride, demb, demb_sample_stride,
                               static_cast<cudaStream_t>(stream));
}

int dlrm_emb_bag_interact_fwd(const void *const *tables, const int64_t *rows, int T, int d, int dtype,
                              const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                              const float *e0, int64_t e0_stride, int mode, float *y, int64_t y_stride,
                              float *pooled, int64_t pooled_sample_stride, int64_t pooled_table_stride,
                              int32_t *err_flag, dlrm_stream_t stream)
{
    TableSet ts;
    int s = make_tables(tables, rows, T, d, dtype, ts);
    if (s != DLRM_OK)
        return s;
    const int64_t width = dlrm_interact_width(T, d, mode);
    if (B < 0 || nnz < 0 || e0_stride < d || width < 0 || y_stride < width)
        return DLRM_ERR_INVALID_ARG;
    if (pooled && (pooled_sample_stride < 0 || pooled_table_stride < 0))
        return DLRM_ERR_INVALID_ARG;
    if (T > 127 || B > (int64_t)1 << 31)
        return DLRM_ERR_UNSUPPORTED;
    if (B == 0)
        return DLRM_OK;
    if (!offsets || !e0 || !y || (nnz > 0 && !indices))
        return DLRM_ERR_INVALID_ARG;
    if (!aligned(offsets, 8) || (indices && !aligned(indices, 8)) || !aligned(e0, 4) || !aligned(y, 4) ||
        (pooled && !aligned(pooled, 4)))
        return DLRM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t row_bytes = (int64_t)d * elem_bytes(dtype);
    bool fused = dtype != DLRM_INT4 && row_bytes % 16 == 0 && row_bytes <= 1024;
    for (int t = 0; t < T && fused; t++)
        fused = aligned(tables[t], 16);
    if (pooled)
        fused = fused && aligned(pooled, 16) && pooled_sample_stride % 4 == 0 && pooled_table_stride % 4 == 0;
    // With the pooled block requested (training: the backward reads it) the
    // lookup followed by the tensor-core interaction is the faster path: the
    // single kernel's Gram runs on the CUDA cores, and the pooled write it
    // saves is needed anyway (multi-hot training step 4.65 ms against 5.10).
    // The single kernel serves inference, where no pooled block is written.
    if (pooled && pooled_table_stride == d &&
        interact_fwd_tc_applies(e0, e0_stride, pooled, pooled_sample_stride, T, d, B))
        fused = false;
    FusedShape fs;
    if (fused && emb_bag_interact_shape(T, d, mode & DLRM_INTERACT_SELF, B, fs))
        return launch_emb_bag_interact_fwd(ts, T, d, dtype, offsets, indices, nnz, B, e0, e0_stride, mode, y,
                                           y_stride, pooled, pooled_sample_stride, pooled_table_stride, fs,
                                           err_flag, st);
    // the two calls it fuses, through the caller's pooled block
    if (!pooled || pooled_table_stride != d)
        return DLRM_ERR_UNSUPPORTED;
    s = launch_lookup(ts, T, d, dtype, offsets, indices, nnz, B, pooled, pooled_sample_stride,
                      pooled_table_stride, err_flag, st);
    if (s != DLRM_OK)
        return s;
    return launch_interact_fwd(e0, e0_stride, pooled, pooled_sample_stride, T, d, B, mode, y, y_stride, st);
}

size_t dlrm_emb_bag_bwd_workspace_size(int T, int64_t B, int64_t nnz, int d)
{
    if (T <= 0 || T > DLRM_MAX_TABLES || B < 0 || nnz < 0 || nnz > kMaxLookups || d <= 0)
        return 0;
    return emb_bag_bwd_workspace(T, nnz, d);
}

int dlrm_emb_bag_sort_plan(const int64_t *rows, int T, int64_t nnz, int *passes, int *msd)
{
    if (!rows || !passes || !msd || T <= 0 || T > DLRM_MAX_TABLES || nnz < 0 || nnz > kMaxLookups)
        return DLRM_ERR_INVALID_ARG;
    for (int t = 0; t < T; t++)
        if (rows[t] <= 0)
            return DLRM_ERR_INVALID_ARG;
    bool m = false;
    coalesce_plan(rows, T, nnz, *passes, m);
    *msd = m ? 1 : 0;
    return DLRM_OK;
}

}  // extern "C"

namespace dlrm {

// Checks shared by the backward's calls: the sizes and the coalescing inputs.
int check_coalesce_args(int T, int d, const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                        const void *workspace, size_t workspace_bytes)
{
    if (B < 0 || nnz < 0)
        return DLRM_ERR_INVALID_ARG;
    if (nnz > kMaxLookups || B > (int64_t)0x7fffffffLL)
        return DLRM_ERR_UNSUPPORTED;
    if (B == 0 && nnz != 0)  // no bags cannot hold lookups
        return DLRM_ERR_INVALID_ARG;
    if (!offsets || !workspace || !aligned(workspace, 256) || !aligned(offsets, 8))
        return DLRM_ERR_INVALID_ARG;
    if (nnz > 0 && (!indices || !aligned(indices, 8)))
        return DLRM_ERR_INVALID_ARG;
    if (workspace_bytes < emb_bag_bwd_workspace(T, nnz, d))
        return DLRM_ERR_WORKSPACE_TOO_SMALL;
    return DLRM_OK;
}

// Checks of the reduce's inputs: pooled gradients, learning rate, outputs.
int check_reduce_args(int64_t nnz, const float *dpooled, int64_t dp_sample_stride, int64_t dp_table_stride,
                      float lr, const float *grad_rows, int64_t grad_rows_cap)
{
    if (dp_sample_stride < 0 || dp_table_stride < 0 || grad_rows_cap < 0)
        return DLRM_ERR_INVALID_ARG;
    if (dp_sample_stride > ((int64_t)1 << 29))  // the reduce addresses pooled rows with 32-bit byte strides
        return DLRM_ERR_UNSUPPORTED;
    if (!(lr == lr))  // NaN learning rate
        return DLRM_ERR_INVALID_ARG;
    if (nnz > 0 && (!dpooled || !aligned(dpooled, 4)))
        return DLRM_ERR_INVALID_ARG;
    if (grad_rows && !aligned(grad_rows, 4))
        return DLRM_ERR_INVALID_ARG;
    return DLRM_OK;
}

// Every host check of dlrm_emb_bag_bwd_sgd, in its order; also used by the
// call without a workspace (with its fixed scratch as the workspace).
int check_bwd_sgd_args(void *const *tables, const int64_t *rows, int T, int d, int dtype, const int64_t *offsets,
                       const int64_t *indices, int64_t nnz, int64_t B, const float *dpooled, int64_t dpss,
                       int64_t dpts, float lr, const float *grad_rows, int64_t grad_rows_cap, const void *workspace,
                       size_t workspace_bytes, TableSet &ts)
{
    int s = make_tables(const_cast<const void *const *>(tables), rows, T, d, dtype, ts);
    if (s != DLRM_OK)
        return s;
    if (dtype == DLRM_INT4)  // 4-bit tables are looked up, not trained
        return DLRM_ERR_UNSUPPORTED;
    if ((s = check_reduce_args(nnz, dpooled, dpss, dpts, lr, grad_rows, grad_rows_cap)) != DLRM_OK)
        return s;
    return check_coalesce_args(T, d, offsets, indices, nnz, B, workspace, workspace_bytes);
}

}  // namespace dlrm

extern "C" {

int dlrm_emb_bag_bwd_sgd(void *const *tables, const int64_t *rows, int T, int d, int dtype,
                         const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                         const float *dpooled, int64_t dp_sample_stride, int64_t dp_table_stride,
                         float lr, float *grad_rows, int64_t grad_rows_cap, void *workspace,
                         size_t workspace_bytes, dlrm_coalesced_view *view, int32_t *err_flag,
                         dlrm_stream_t stream)
{
    TableSet ts;
    const int s = check_bwd_sgd_args(tables, rows, T, d, dtype, offsets, indices, nnz, B, dpooled, dp_sample_stride,
                                     dp_table_stride, lr, grad_rows, grad_rows_cap, workspace, workspace_bytes, ts);
    if (s != DLRM_OK)
        return s;
    const bool vec = emb_bag_bwd_vectorisable(ts, T, d, dpooled, dp_sample_stride, dp_table_stride, grad_rows);
    return launch_emb_bag_bwd(ts, T, d, dtype, offsets, indices, nnz, B, dpooled, dp_sample_stride,
                              dp_table_stride, lr, grad_rows, grad_rows ? grad_rows_cap : 0, workspace, vec,
                              view, err_flag, static_cast<cudaStream_t>(stream));
}

int dlrm_emb_bag_bwd_sgd_atomic(void *const *tables, const int64_t *rows, int T, int d, int dtype,
                                const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                                const float *dpooled, int64_t dp_sample_stride, int64_t dp_table_stride,
                                float lr, int32_t *err_flag, dlrm_stream_t stream)
{
    TableSet ts;
    int s = make_tables(const_cast<const void *const *>(tables), rows, T, d, dtype, ts);
    if (s != DLRM_OK)
        return s;
    if (dtype != DLRM_F32)  // one fp32 reduction per lookup: half tables would round at every one
        return DLRM_ERR_UNSUPPORTED;
    if ((s = check_reduce_args(nnz, dpooled, dp_sample_stride, dp_table_stride, lr, nullptr, 0)) != DLRM_OK)
        return s;
    if (B < 0 || nnz < 0 || (B == 0 && nnz != 0))
        return DLRM_ERR_INVALID_ARG;
    if (nnz > kMaxLookups || B > (int64_t)0x7fffffffLL)
        return DLRM_ERR_UNSUPPORTED;
    if (!offsets || !aligned(offsets, 8) || (nnz > 0 && (!indices || !aligned(indices, 8))))
        return DLRM_ERR_INVALID_ARG;
    if (B == 0 || lr == 0.f)
        return DLRM_OK;
    const bool vec = emb_bag_bwd_vectorisable(ts, T, d, dpooled, dp_sample_stride, dp_table_stride, nullptr);
    return launch_emb_bag_bwd_atomic(ts, T, d, offsets, indices, nnz, B, dpooled, dp_sample_stride, dp_table_stride,
                                     lr, vec, err_flag, static_cast<cudaStream_t>(stream));
}

int dlrm_emb_bag_coalesce(const int64_t *rows, int T, int d, const int64_t *offsets, const int64_t *indices,
                          int64_t nnz, int64_t B, void *workspace, size_t workspace_bytes,
                          dlrm_coalesced_view *view, int32_t *err_flag, dlrm_stream_t stream)
{
    if (!rows || T <= 0 || d <= 0)
        return DLRM_ERR_INVALID_ARG;
    if (T > DLRM_MAX_TABLES)
        return DLRM_ERR_UNSUPPORTED;
    TableSet ts;
    std::memset(&ts, 0, sizeof ts);
    for (int t = 0; t < T; t++) {
        if (rows[t] <= 0)
            return DLRM_ERR_INVALID_ARG;
        if (rows[t] > (int64_t)0xfffffffeLL)
            return DLRM_ERR_UNSUPPORTED;
        ts.rows[t] = rows[t];
    }
    int s = check_coalesce_args(T, d, offsets, indices, nnz, B, workspace, workspace_bytes);
    if (s != DLRM_OK)
        return s;
    return launch_coalesce(ts, T, d, offsets, indices, nnz, B, workspace, view, err_flag,
                           static_cast<cudaStream_t>(stream));
}

int dlrm_emb_bag_reduce_sgd(void *const *tables, const int64_t *rows, int T, int d, int dtype, int64_t nnz,
                            int64_t B, const float *dpooled, int64_t dp_sample_stride, int64_t dp_table_stride,
                            float lr, float *grad_rows, int64_t grad_rows_cap, void *workspace,
                            size_t workspace_bytes, int32_t *err_flag, dlrm_stream_t stream)
{
    TableSet ts;
    int s = make_tables(const_cast<const void *const *>(tables), rows, T, d, dtype, ts);
    if (s != DLRM_OK)
        return s;
    if (dtype == DLRM_INT4)  // 4-bit tables are looked up, not trained
        return DLRM_ERR_UNSUPPORTED;
    if ((s = check_reduce_args(nnz, dpooled, dp_sample_stride, dp_table_stride, lr, grad_rows, grad_rows_cap)) !=
        DLRM_OK)
        return s;
    if (B < 0 || nnz < 0 || (B == 0 && nnz != 0))
        return DLRM_ERR_INVALID_ARG;
    if (nnz > kMaxLookups || B > (int64_t)0x7fffffffLL)
        return DLRM_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256))
        return DLRM_ERR_INVALID_ARG;
    if (workspace_bytes < emb_bag_bwd_workspace(T, nnz, d))
        return DLRM_ERR_WORKSPACE_TOO_SMALL;
    const bool vec = emb_bag_bwd_vectorisable(ts, T, d, dpooled, dp_sample_stride, dp_table_stride, grad_rows);
    return launch_reduce_sgd(ts, T, d, dtype, nnz, B, dpooled, dp_sample_stride, dp_table_stride, lr, grad_rows,
                             grad_rows ? grad_rows_cap : 0, workspace, vec, err_flag,
                             static_cast<cudaStream_t>(stream), 0.f, nullptr);
}

// Checks of the AdaGrad arguments: one fp32 accumulator array per table,
// a positive finite eps, rows short enough to be held whole.
static int check_adagrad(float *const *state, int T, int d, float lr, float eps)
{
    if (!state || !(eps > 0.f) || !(eps <= 3.0e38f) || !(lr == lr) || lr > 3.0e38f || lr < -3.0e38f)
        return DLRM_ERR_INVALID_ARG;
    for (int t = 0; t < T; t++)
        if (!state[t] || !aligned(state[t], 4))
            return DLRM_ERR_INVALID_ARG;
    if (d > 256)
        return DLRM_ERR_UNSUPPORTED;
    return DLRM_OK;
}

int dlrm_emb_bag_bwd_adagrad(void *const *tables, float *const *state, const int64_t *rows, int T, int d, int dtype,
                             const int64_t *offsets, const int64_t *indices, int64_t nnz, int64_t B,
                             const float *dpooled, int64_t dp_sample_stride, int64_t dp_table_stride, float lr,
                             float eps, float *grad_rows, int64_t grad_rows_cap, void *workspace,
                             size_t workspace_bytes, dlrm_coalesced_view *view, int32_t *err_flag,
                             dlrm_stream_t stream)
{
    TableSet ts;
    int s = make_tables(const_cast<const void *const *>(tables), rows, T, d, dtype, ts);
    if (s != DLRM_OK)
        return s;
    if (dtype == DLRM_INT4)  // 4-bit tables are looked up, not trained
        return DLRM_ERR_UNSUPPORTED;
    if ((s = check_adagrad(state, T, d, lr, eps)) != DLRM_OK)
        return s;
    if ((s = check_reduce_args(nnz, dpooled, dp_sample_stride, dp_table_stride, lr, grad_rows, grad_rows_cap)) !=
        DLRM_OK)
        return s;
    if ((s = check_coalesce_args(T, d, offsets, indices, nnz, B, workspace, workspace_bytes)) != DLRM_OK)
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = launch_coalesce(ts, T, d, offsets, indices, nnz, B, workspace, view, err_flag, st)) != DLRM_OK)
        return s;
    const bool vec = emb_bag_bwd_vectorisable(ts, T, d, dpooled, dp_sample_stride, dp_table_stride, grad_rows);
    return launch_reduce_sgd(ts, T, d, dtype, nnz, B, dpooled, dp_sample_stride, dp_table_stride, lr, grad_rows,
                             grad_rows ? grad_rows_cap : 0, workspace, vec, err_flag, st, eps, state);
}

int dlrm_emb_bag_reduce_adagrad(void *const *tables, float *const *state, const int64_t *rows, int T, int d,
                                int dtype, int64_t nnz, int64_t B, const float *dpooled, int64_t dp_sample_stride,
                                int64_t dp_table_stride, float lr, float eps, float *grad_rows,
                                int64_t grad_rows_cap, void *workspace, size_t workspace_bytes, int32_t *err_flag,
                                dlrm_stream_t stream)
{
    TableSet ts;
    int s = make_tables(const_cast<const void *const *>(tables), rows, T, d, dtype, ts);
    if (s != DLRM_OK)
        return s;
    if (dtype == DLRM_INT4)  // 4-bit tables are looked up, not trained
        return DLRM_ERR_UNSUPPORTED;
    if ((s = check_adagrad(state, T, d, lr, eps)) != DLRM_OK)
        return s;
    if ((s = check_reduce_args(nnz, dpooled, dp_sample_stride, dp_table_stride, lr, grad_rows, grad_rows_cap)) !=
        DLRM_OK)
        return s;
    if (B < 0 || nnz < 0 || (B == 0 && nnz != 0))
        return DLRM_ERR_INVALID_ARG;
    if (nnz > kMaxLookups || B > (int64_t)0x7fffffffLL)
        return DLRM_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256))
        return DLRM_ERR_INVALID_ARG;
    if (workspace_bytes < emb_bag_bwd_workspace(T, nnz, d))
        return DLRM_ERR_WORKSPACE_TOO_SMALL;
    const bool vec = emb_bag_bwd_vectorisable(ts, T, d, dpooled, dp_sample_stride, dp_table_stride, grad_rows);
    return launch_reduce_sgd(ts, T, d, dtype, nnz, B, dpooled, dp_sample_stride, dp_table_stride, lr, grad_rows,
                             grad_rows ? grad_rows_cap : 0, workspace, vec, err_flag,
                             static_cast<cudaStream_t>(stream), eps, state);
}

int dlrm_read_error(const int32_t *err_flag, dlrm_stream_t stream)
{
    if (!err_flag)
        return DLRM_ERR_INVALID_ARG;
    int32_t h = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaMemcpy(&h, err_flag, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
        return DLRM_ERR_CUDA;
    if (h & DLRM_FLAG_INDEX_OOB)
        return DLRM_ERR_INDEX_OOB;
    if (h & DLRM_FLAG_BAD_OFFSETS)
        return DLRM_ERR_BAD_OFFSETS;
    if (h & DLRM_FLAG_CAPACITY)
        return DLRM_ERR_CAPACITY;
    if (h & DLRM_FLAG_WAIT_TIMEOUT)
        return DLRM_ERR_WAIT_TIMEOUT;
    return DLRM_OK;
}

int dlrm_clear_error(int32_t *err_flag, dlrm_stream_t stream)
{
    if (!err_flag)
        return DLRM_ERR_INVALID_ARG;
    return cudaMemsetAsync(err_flag, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DLRM_OK
               : DLRM_ERR_CUDA;
}

const char *dlrm_status_string(int status)
{
    switch (status) {
    case DLRM_OK:
        return "ok";
    case DLRM_ERR_INVALID_ARG:
        return "invalid argument";
    case DLRM_ERR_UNSUPPORTED:
        return "unsupported size or layout";
    case DLRM_ERR_WORKSPACE_TOO_SMALL:
        return "workspace too small";
    case DLRM_ERR_INDEX_OOB:
        return "index out of range of its table";
    case DLRM_ERR_BAD_OFFSETS:
        return "offsets not monotone or not spanning 0..nnz";
    case DLRM_ERR_CAPACITY:
        return "more unique rows than grad_rows can hold";
    case DLRM_ERR_CUDA:
        return "CUDA error";
    case DLRM_ERR_WAIT_TIMEOUT:
        return "a kernel's bounded wait on another CTA ran out";
    default:
        return "unknown status";
    }
}

uint64_t dlrm_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int dlrm_profile_events(void *const *events, int n)
{
    if (n < 0 || n > DLRM_MAX_PROFILE_EVENTS || (n > 0 && !events))
        return DLRM_ERR_INVALID_ARG;
    for (int i = 0; i < n; i++) {
        if (!events[i])
            return DLRM_ERR_INVALID_ARG;
        g_prof_events[i] = static_cast<cudaEvent_t>(events[i]);
    }
    g_prof_n = n;
    g_prof_next = 0;
    return DLRM_OK;
}

}  // extern "C"
