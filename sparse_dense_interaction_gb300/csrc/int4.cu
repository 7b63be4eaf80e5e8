// Row-wise int4 tables: the encoder and the pooled lookup over them.
//
// The factlen.com page ("Terabyte Embedding Tables and Compute-Bound Neural
// Layers Force Meta's DLRM to Split Training", section "The limits of
// scale") reports 4-bit integer quantization of the vectors, without a
// format.  The codec here is the row-wise affine one: a row of d values is
// stored as d 4-bit codes q (element 2j in the low nibble of byte j, 2j+1 in
// the high nibble), then its fp32 scale s and bias b, padded to a multiple of
// 16 bytes; an element's value is b + s q.  A 128-wide row takes 80 bytes
// instead of 256 (fp16) or 512 (fp32).
//
// Encoder: one warp per row; the codes are decided in fp32 with IEEE
// subtraction and division and round-half-even, so that every code is
// reproducible.  Lookup: as the 16-bit lookup, a group of G lanes sums one
// bag; each lane owns 16 codes (8 bytes) of the row, reads the row's scale
// and bias (one 8-byte load when d % 16 == 0), and adds s q per element (q
// made a float by a byte permute into the low mantissa byte of 2^23 and a
// subtraction of 2^23); the biases are summed once per row.
#include "common.cuh"

namespace dlrm {

int64_t int4_row_bytes(int d) { return ((int64_t)d / 2 + 8 + 15) / 16 * 16; }

template <typename TT>
__global__ void __launch_bounds__(256)
quantize_int4_kernel(const TT *__restrict__ src, int64_t R, int d, uint8_t *__restrict__ dst, int64_t rb)
{
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < R; r += nwarps) {
        const TT *w = src + r * d;
        float lo = INFINITY, hi = -INFINITY;
        for (int e = lane; e < d; e += 32) {
            const float v = to_f32(w[e]);
            lo = fminf(lo, v);
            hi = fmaxf(hi, v);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        lo = __fadd_rn(lo, 0.f);  // -0 becomes +0: the stored bias and scale are unique
        hi = __fadd_rn(hi, 0.f);
        const float scale = __fdiv_rn(__fsub_rn(hi, lo), 15.f);
        uint8_t *row = dst + r * rb;
        for (int j = lane; j < d / 2; j += 32) {
            int q[2] = {0, 0};
            if (scale > 0.f) {
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int v = __float2int_rn(__fdiv_rn(__fsub_rn(to_f32(w[2 * j + h]), lo), scale));
                    q[h] = v < 0 ? 0 : (v > 15 ? 15 : v);
                }
            }
            row[j] = (uint8_t)(q[0] | (q[1] << 4));
        }
        if (lane == 0) {
            *reinterpret_cast<float *>(row + d / 2) = scale;
            *reinterpret_cast<float *>(row + d / 2 + 4) = lo;
        }
        for (int64_t i = d / 2 + 8 + lane; i < rb; i += 32)
            row[i] = 0;
    }
}

// The float values of the 8 codes of a word: the low and the high nibbles of
// its bytes are masked out, and each is moved by a byte permute into the low
// byte of 2^23 (0x4B000000), whose value minus 2^23 is the code.
__device__ __forceinline__ void codes_f32(uint32_t word, float *v)
{
    const uint32_t lo = word & 0x0F0F0F0Fu, hi = (word >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        // bytes: [lo or hi byte i, 0, 0, 0x4B] taken from (x, 0x0000004B)
        const uint32_t sel = (uint32_t)i | (5u << 4) | (5u << 8) | (4u << 12);
        v[2 * i] = __int_as_float(__byte_perm(lo, 0x4Bu, sel)) - 8388608.f;
        v[2 * i + 1] = __int_as_float(__byte_perm(hi, 0x4Bu, sel)) - 8388608.f;
    }
}

template <int G, int U>
__global__ void __launch_bounds__(256, 4)
emb_bag_fwd_int4_kernel(TableSet ts, int T, int d, int64_t rb, const int64_t *__restrict__ offsets,
                        const int64_t *__restrict__ indices, int64_t nnz, int64_t B, float *__restrict__ out,
                        int64_t oss, int64_t ots, int32_t *err)
{
    constexpr int GPW = 32 / G;             // bags per warp
    constexpr uint32_t kBad = 0xffffffffu;  // row slot without a valid lookup
    static_assert(U <= G && G % U == 0, "a group walks its G indices in steps of U");
    const int lane = threadIdx.x & 31;
    const int gl = lane % G;
    const int grp = lane / G;
    const unsigned gmask = (G == 32) ? 0xffffffffu : (((1u << G) - 1u) << (grp * G));
    const int64_t nbags = (int64_t)T * B;
    const bool small = nbags <= 0xffffffffll;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const bool on = 16 * gl < d;  // this lane owns codes 16 gl .. 16 gl + 15
    const bool pair_params = d % 16 == 0;  // scale and bias 8-byte aligned: one load

    for (int64_t bag = warp * GPW + grp; bag < nbags; bag += nwarps * GPW) {
        int t;
        int64_t b;
        bag_table_sample(bag, B, small, t, b);
        int64_t k0 = offsets[bag];
        int64_t k1 = offsets[bag + 1];
        if (k0 < 0 || k1 < k0 || k1 > nnz) {
            if (gl == 0)
                raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
            k0 = k1 = 0;
        }
        const uint8_t *tab = static_cast<const uint8_t *>(ts.ptr[t]);
        const int64_t R = ts.rows[t];
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; k++)
            acc[k] = 0.f;
        float bsum = 0.f;
        for (int64_t kb = k0; kb < k1; kb += G) {
            const int n = (k1 - kb < G) ? (int)(k1 - kb) : G;
            uint32_t row = kBad;
            if (gl < n) {
                const int64_t r = load_stream(indices + kb + gl);
                if (r >= 0 && r < R)
                    row = (uint32_t)r;
                else
                    raise_flag(err, DLRM_FLAG_INDEX_OOB);
            }
            for (int q = 0; q < n; q += U) {
                uint2 c[U];
                float2 sb[U];  // scale, bias
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const uint32_t r = __shfl_sync(gmask, row, q + u, G);
                    const uint8_t *p = tab + (int64_t)r * rb;
                    const bool ok = r != kBad;
                    c[u] = (ok && on) ? __ldg(reinterpret_cast<const uint2 *>(p + 8 * gl)) : make_uint2(0u, 0u);
                    if (!ok)
                        sb[u] = make_float2(0.f, 0.f);
                    else if (pair_params)
                        sb[u] = __ldg(reinterpret_cast<const float2 *>(p + d / 2));
                    else
                        sb[u] = make_float2(__ldg(reinterpret_cast<const float *>(p + d / 2)),
                                            __ldg(reinterpret_cast<const float *>(p + d / 2 + 4)));
                }
#pragma unroll
                for (int u = 0; u < U; u++) {
                    bsum += sb[u].y;
                    float v[8];
                    codes_f32(c[u].x, v);
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        acc[k] = fmaf(sb[u].x, v[k], acc[k]);
                    codes_f32(c[u].y, v);
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        acc[8 + k] = fmaf(sb[u].x, v[k], acc[8 + k]);
                }
            }
        }
        if (on) {
            float *o = out + b * oss + (int64_t)t * ots + 16 * gl;
            if (16 * gl + 16 <= d) {
#pragma unroll
                for (int k = 0; k < 16; k += 4)
                    __stcs(reinterpret_cast<float4 *>(o + k),
                           make_float4(acc[k] + bsum, acc[k + 1] + bsum, acc[k + 2] + bsum, acc[k + 3] + bsum));
            } else {
#pragma unroll
                for (int k = 0; k < 8; k++)  // d % 16 == 8: half a chunk
                    o[k] = acc[k] + bsum;
            }
        }
    }
}

template <typename K>
static int resident_grid(K kernel, int64_t work_blocks)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t resident = (int64_t)per_sm * sm_count();
    return (int)(work_blocks < resident ? (work_blocks < 1 ? 1 : work_blocks) : resident);
}

template <int G>
static int launch_int4(const TableSet &ts, int T, int d, const int64_t *offsets, const int64_t *indices, int64_t nnz,
                       int64_t B, float *out, int64_t oss, int64_t ots, int32_t *err, cudaStream_t st)
{
    constexpr int U = G < 4 ? G : 4;
    auto kernel = emb_bag_fwd_int4_kernel<G, U>;
    const int64_t bags_per_block = 8 * (32 / G);
    const int grid = resident_grid(kernel, ((int64_t)T * B + bags_per_block - 1) / bags_per_block);
    kernel<<<grid, 256, 0, st>>>(ts, T, d, int4_row_bytes(d), offsets, indices, nnz, B, out, oss, ots, err);
    count_launch(st);
    return launch_status();
}

// d % 8 == 0 and d <= 512; out 16-byte aligned with strides that are multiples of 4.
int launch_emb_bag_fwd_int4(const TableSet &ts, int T, int d, const int64_t *offsets, const int64_t *indices,
                            int64_t nnz, int64_t B, float *out, int64_t oss, int64_t ots, int32_t *err,
                            cudaStream_t st)
{
    const int lanes = (d + 15) / 16;
    if (lanes <= 4)
        return launch_int4<4>(ts, T, d, offsets, indices, nnz, B, out, oss, ots, err, st);
    if (lanes <= 8)
        return launch_int4<8>(ts, T, d, offsets, indices, nnz, B, out, oss, ots, err, st);
    if (lanes <= 16)
        return launch_int4<16>(ts, T, d, offsets, indices, nnz, B, out, oss, ots, err, st);
    return launch_int4<32>(ts, T, d, offsets, indices, nnz, B, out, oss, ots, err, st);
}

int launch_quantize_int4(const void *src, int dtype, int64_t R, int d, void *dst, cudaStream_t st)
{
    const int64_t rb = int4_row_bytes(d);
    const int64_t blocks = (R + 7) / 8;
    const int grid = (int)(blocks < (int64_t)sm_count() * 16 ? (blocks < 1 ? 1 : blocks) : (int64_t)sm_count() * 16);
    uint8_t *o = static_cast<uint8_t *>(dst);
    switch (dtype) {
    case DLRM_F32:
        quantize_int4_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float *>(src), R, d, o, rb);
        break;
    case DLRM_F16:
        quantize_int4_kernel<__half><<<grid, 256, 0, st>>>(static_cast<const __half *>(src), R, d, o, rb);
        break;
    default:
        quantize_int4_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(src), R, d,
                                                                   o, rb);
        break;
    }
    count_launch(st);
    return launch_status();
}

}  // namespace dlrm
