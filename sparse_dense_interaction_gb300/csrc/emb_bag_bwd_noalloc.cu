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
#include "common.cuh"

namespace dlrm {

bool emb_bag_bwd_vectorisable(const TableSet &, int, int, const float *, int64_t, int64_t, const float *);
int launch_emb_bag_bwd(const TableSet &, int, int, int, const int64_t *, const int64_t *, int64_t, int64_t,
                       const float *, int64_t, int64_t, float, float *, int64_t, void *, bool,
                       dlrm_coalesced_view *, int32_t *, cudaStream_t);

static __device__ __align__(256) unsigned char g_noalloc_scratch[DLRM_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is asked of
// the runtime, with the device current, at every call (a host-side lookup; no
// address is kept that could outlive the context it belongs to).  With lazily
// loaded modules the first lookup on a device loads the module and makes the
// array resident there; if that fails (no memory left) the runtime's error is
// cleared, so that later calls do not report it, and DLRM_ERR_CUDA returned.
static int scratch_address(void **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        (void)cudaGetLastError();
        return DLRM_ERR_CUDA;
    }
    *out = p;
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
    // dlrm_emb_bag_bwd_sgd's own checks, with the array in place of the
    // workspace: sizes whose scratch does not fit it are refused with
    // DLRM_ERR_WORKSPACE_TOO_SMALL.  The checks only need the workspace's size
    // and that its address is non-null and 256-byte aligned, which the array's
    // is; its device address is looked up once they have passed, so a refused
    // call never touches the device.
    const void *const array_stand_in = reinterpret_cast<const void *>(static_cast<uintptr_t>(256));
    TableSet ts;
    int s = check_bwd_sgd_args(tables, rows, T, d, dtype, offsets, indices, nnz, B, dpooled, dp_sample_stride,
                               dp_table_stride, lr, grad_rows, grad_rows_cap, array_stand_in,
                               DLRM_NOALLOC_SCRATCH_BYTES, ts);
    if (s != DLRM_OK)
        return s;
    void *scratch = nullptr;
    if ((s = scratch_address(&scratch)) != DLRM_OK)
        return s;
    const bool vec = emb_bag_bwd_vectorisable(ts, T, d, dpooled, dp_sample_stride, dp_table_stride, grad_rows);
    return launch_emb_bag_bwd(ts, T, d, dtype, offsets, indices, nnz, B, dpooled, dp_sample_stride,
                              dp_table_stride, lr, grad_rows, grad_rows ? grad_rows_cap : 0, scratch, vec, view,
                              err_flag, static_cast<cudaStream_t>(stream));
}
