// Device-side table initialisation for the synthetic workloads.
//
// Input generation only: this library holds none of the DLRM path's
// arithmetic and is not part of the path's C ABI.  It fills a table with the
// same values as the host generator in workloads.py, element by element:
// element n = row*d + col of table t is SplitMix64's output for state
// s_t + (n+1)*gamma (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014), whose top 24 bits m give the exact fp32
// value v = (2m - 2^24) * 2^-24; the element is fp32(v * scale) rounded once
// more, to nearest even, into the table's storage type.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t splitmix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

template <typename TT>
__device__ __forceinline__ TT cast_out(float v);
template <>
__device__ __forceinline__ float cast_out<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half cast_out<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 cast_out<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

template <typename TT>
__global__ void fill_kernel(TT *table, uint64_t n_elems, uint64_t seed, float scale)
{
    for (uint64_t n = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; n < n_elems;
         n += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t z = splitmix64(seed + (n + 1) * 0x9E3779B97F4A7C15ull);
        const int64_t m = (int64_t)(z >> 40);
        const float v = __fmul_rn((float)(2 * m - (1LL << 24)), 5.9604644775390625e-08f);  // * 2^-24, exact
        table[n] = cast_out<TT>(__fmul_rn(v, scale));
    }
}

}  // namespace

extern "C" int dlrm_workload_fill_table(void *table, int dtype, int64_t rows, int d, uint64_t seed,
                                        float scale, void *stream)
{
    if (!table || rows <= 0 || d <= 0)
        return -1;
    const uint64_t n = (uint64_t)rows * (uint64_t)d;
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned grid = (unsigned)(sms * 8);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == 0)
        fill_kernel<float><<<grid, 256, 0, st>>>(static_cast<float *>(table), n, seed, scale);
    else if (dtype == 1)
        fill_kernel<__half><<<grid, 256, 0, st>>>(static_cast<__half *>(table), n, seed, scale);
    else
        fill_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<__nv_bfloat16 *>(table), n, seed, scale);
    return cudaGetLastError() == cudaSuccess ? 0 : -7;
}
