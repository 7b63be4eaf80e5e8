// Shared device helpers of the sm_103a DLRM sparse path.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "dlrm_sparse.h"

namespace dlrm {

// Kernel-parameter view of the caller's tables (4 KB at 256 tables, well
// inside the 32 KB parameter space of sm_70+ kernels).
struct TableSet {
    const void *ptr[DLRM_MAX_TABLES];
    int64_t rows[DLRM_MAX_TABLES];
};

// Called after every kernel launch: counts it and, when the calling thread
// has registered profiling events, records the next one on the stream.
void count_launch(cudaStream_t st);
// cudaGetLastError mapped to a status, for use right after a launch.
int launch_status();
// Streaming multiprocessor count of the current device.
int sm_count();
// Raises a kernel's dynamic shared-memory limit on the current device, once
// per device and kernel (`done` is the kernel's bit mask of devices already
// set; concurrent callers may both set it, which is harmless).
int allow_dynamic_smem(const void *kernel, int bytes, std::atomic<unsigned long long> *done);
// Whether the interaction calls may take the tensor-core kernels (the
// process-wide setting of dlrm_set_interact_kernel).
bool interact_tensor_cores();
// Limits of the kernels' bounded waits for the next launches, as the testing
// hook dlrm_set_wait_test_hooks left them (defaults when unset): polls of a
// radix pass's look-back word, the first tile the passes claim, polls of a
// stage barrier in the main loop of the bulk-copy interaction forward.
struct WaitHooks {
    int sort_polls;
    uint32_t sort_first_tile;
    int copy_polls;
};
WaitHooks wait_hooks(int default_sort_polls, int default_copy_polls);
// Host checks shared by the entry points (api.cu): the table arguments (fills
// the kernel-parameter view), and the whole argument list of the backward with
// SGD (the call without a workspace passes its fixed scratch as workspace).
int make_tables(const void *const *tables, const int64_t *rows, int T, int d, int dtype, TableSet &ts);
int check_bwd_sgd_args(void *const *tables, const int64_t *rows, int T, int d, int dtype, const int64_t *offsets,
                       const int64_t *indices, int64_t nnz, int64_t B, const float *dpooled, int64_t dpss,
                       int64_t dpts, float lr, const float *grad_rows, int64_t grad_rows_cap, const void *workspace,
                       size_t workspace_bytes, TableSet &ts);

// Table t and sample b of bag `bag` (table-major: bag = t * B + b), by a 32-bit
// division when every bag index fits in 32 bits (`small`, fixed per launch), as
// it does for all but gigantic batches; 64 bits otherwise.
__device__ __forceinline__ void bag_table_sample(int64_t bag, int64_t B, bool small, int &t, int64_t &b)
{
    if (small) {
        const uint32_t q = (uint32_t)bag / (uint32_t)B;
        t = (int)q;
        b = bag - (int64_t)q * B;
    } else {
        t = (int)(bag / B);
        b = bag - (int64_t)t * B;
    }
}

__device__ __forceinline__ void raise_flag(int32_t *flag, int bits)
{
    if (flag)
        atomicOr(flag, bits);
}

// 16-byte table chunk added into fp32 accumulators (kElems/2 float2 pairs).
// fp32 chunks use packed fp32 adds.
template <typename TT>
struct Chunk16;

template <>
struct Chunk16<float> {
    static constexpr int kElems = 4;
    __device__ __forceinline__ static void add(float2 *acc, const uint4 &v)
    {
        acc[0] = __fadd2_rn(acc[0], make_float2(__uint_as_float(v.x), __uint_as_float(v.y)));
        acc[1] = __fadd2_rn(acc[1], make_float2(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
};

// Half-precision chunks use mixed-precision adds (the 16-bit operand is
// widened exactly inside the add), one instruction per element.
template <>
struct Chunk16<__half> {
    static constexpr int kElems = 8;
    __device__ __forceinline__ static void add(float2 *acc, const uint4 &v)
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; i++)
            asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.f16 %0, lo, %0; add.rn.f32.f16 %1, hi, %1; }"
                : "+f"(acc[i].x), "+f"(acc[i].y) : "r"(w[i]));
    }
};

template <>
struct Chunk16<__nv_bfloat16> {
    static constexpr int kElems = 8;
    __device__ __forceinline__ static void add(float2 *acc, const uint4 &v)
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; i++)
            asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; add.rn.f32.bf16 %0, lo, %0; add.rn.f32.bf16 %1, hi, %1; }"
                : "+f"(acc[i].x), "+f"(acc[i].y) : "r"(w[i]));
    }
};

template <typename TT>
__device__ __forceinline__ float to_f32(TT v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename TT>
__device__ __forceinline__ TT from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Loads that should not displace hot table rows from L2.
__device__ __forceinline__ int64_t load_stream(const int64_t *p) { return __ldcs(p); }
__device__ __forceinline__ uint4 load_table(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }

}  // namespace dlrm
