// Embedding-bag backward + row-wise SGD for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: for
// example a plugin whose host framework passes it only the input and output
// tensors and owns every device allocation, or a service that must not touch
// the device allocator once it is running.  This entry point runs the same
// pipeline as dlrm_emb_bag_bwd_sgd, with its scratch in a fixed-size array in
// this file instead of a caller workspace, and allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library's module holds its DLRM_NOALLOC_SCRATCH_BYTES until the process
// exits.  All calls share it, and it keeps the last call's contents: the
// pipeline re-initialises everything it reads (counters, flags, offsets), and
// two calls that overlap on the GPU (different streams, no ordering between
// them) race on it.
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace dlrm {

size_t emb_bag_bwd_workspace(int, int64_t, int);
bool emb_bag_bwd_vectorisable(const TableSet &, int, int, const float *, int64_t, int64_t, const float *);
int launch_emb_bag_bwd(const TableSet &, int, int, int, const int64_t *, const int64_t *, int64_t, int64_t,
                       const float *, int64_t, int64_t, float, float *, int64_t, void *, bool,
                       dlrm_coalesced_view *, int32_t *, cudaStream_t);

static __device__ __align__(256) unsigned char g_noalloc_scratch[DLRM_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current, and cached.
static int scratch_address(void **out)
{
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return DLRM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return DLRM_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return DLRM_OK;
}

}  // namespace dlrm

using namespace dlrm;

extern "C" int dlrm_emb_bag_bwd_sgd_noalloc(void *const *tables, const int64_t *rows, int T, int d, int dtype,
                                            const int64_t *offsets, const int64_t *indices, int64_t nnz,
                                            int64_t B, const float *dpooled, int64_t dp_sample_stride,
                                            int64_t dp_table_stride, float lr, float *grad_rows,
                                            int64_t grad_rows_cap, dlrm_coalesced_view *view,
                                            int32_t *err_flag, dlrm_stream_t stream)
{
    // Argument checks identical to dlrm_emb_bag_bwd_sgd's, all on the host.
    if (!tables || !rows || T <= 0 || d <= 0)
        return DLRM_ERR_INVALID_ARG;
    if (dtype != DLRM_F32 && dtype != DLRM_F16 && dtype != DLRM_BF16)
        return DLRM_ERR_INVALID_ARG;
    if (T > DLRM_MAX_TABLES)
        return DLRM_ERR_UNSUPPORTED;
    const size_t es = dtype == DLRM_F32 ? 4 : 2;
    TableSet ts;
    std::memset(&ts, 0, sizeof ts);
    for (int t = 0; t < T; t++) {
        if (!tables[t] || rows[t] <= 0)
            return DLRM_ERR_INVALID_ARG;
        if (rows[t] > (int64_t)0xfffffffeLL)
            return DLRM_ERR_UNSUPPORTED;
        if (reinterpret_cast<uintptr_t>(tables[t]) % es != 0)
            return DLRM_ERR_INVALID_ARG;
        ts.ptr[t] = tables[t];
        ts.rows[t] = rows[t];
    }
    if (B < 0 || nnz < 0 || dp_sample_stride < 0 || dp_table_stride < 0 || grad_rows_cap < 0)
        return DLRM_ERR_INVALID_ARG;
    if (nnz > ((int64_t)1 << 31) || B > (int64_t)0x7fffffffLL)
        return DLRM_ERR_UNSUPPORTED;
    if (B == 0 && nnz != 0)
        return DLRM_ERR_INVALID_ARG;
    if (dp_sample_stride > ((int64_t)1 << 29))  // the reduce addresses pooled rows with 32-bit byte strides
        return DLRM_ERR_UNSUPPORTED;
    if (!(lr == lr))
        return DLRM_ERR_INVALID_ARG;
    if (!offsets || reinterpret_cast<uintptr_t>(offsets) % 8 != 0)
        return DLRM_ERR_INVALID_ARG;
    if (nnz > 0 && (!indices || reinterpret_cast<uintptr_t>(indices) % 8 != 0 || !dpooled ||
                    reinterpret_cast<uintptr_t>(dpooled) % 4 != 0))
        return DLRM_ERR_INVALID_ARG;
    if (grad_rows && reinterpret_cast<uintptr_t>(grad_rows) % 4 != 0)
        return DLRM_ERR_INVALID_ARG;
    // Sizes whose scratch does not fit the fixed array are refused.
    if (emb_bag_bwd_workspace(T, nnz, d) > (size_t)DLRM_NOALLOC_SCRATCH_BYTES)
        return DLRM_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    int s = scratch_address(&scratch);
    if (s != DLRM_OK)
        return s;
    const bool vec = emb_bag_bwd_vectorisable(ts, T, d, dpooled, dp_sample_stride, dp_table_stride, grad_rows);
    return launch_emb_bag_bwd(ts, T, d, dtype, offsets, indices, nnz, B, dpooled, dp_sample_stride,
                              dp_table_stride, lr, grad_rows, grad_rows ? grad_rows_cap : 0, scratch, vec, view,
                              err_flag, static_cast<cudaStream_t>(stream));
}
