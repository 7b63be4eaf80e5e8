// Embedding-bag forward: sum-pooled gathers of table rows.
//
// Follows "Notes/DLRM" (vault-aram.pages.dev), section 2 (one table per
// categorical feature, each ID looked up as a learned vector) and section 9
// (multi-valued features are aggregated; here, summed).
//
// Design: a group of G lanes (G = 4..32) owns one bag at a time; each lane
// owns one or more 16-byte chunks of the row, so a row is read as one fully
// coalesced burst of 16-byte loads.  The group loads up to G indices of its
// bag at once (one per lane, streaming) and each lane checks its own index
// against the table, so the walk over the bag only broadcasts 32-bit rows
// (one shuffle per lookup) and keeps 8 rows in flight per lane; the fp32 sums
// use packed adds.  The kernel stays within 64 registers, so 32 warps share
// an SM and hide the gather latency.  Bags are visited in table-major order,
// so at any moment the warps of the GPU touch the same few tables and hot
// (Zipf) rows stay in L2.  The pooled vector is written once with streaming
// stores.  Grid: persistent, resident blocks only.
#include "common.cuh"

namespace dlrm {

template <typename TT, int G, int C, int U>
__global__ void __launch_bounds__(256, 4)
emb_bag_fwd_vec_kernel(TableSet ts, int T, int nchunks, const int64_t *__restrict__ offsets,
                       const int64_t *__restrict__ indices, int64_t nnz, int64_t B,
                       float *__restrict__ out, int64_t oss, int64_t ots, int32_t *err)
{
    constexpr int EPC = Chunk16<TT>::kElems;  // elements per 16-byte chunk
    constexpr int GPW = 32 / G;               // bags per warp
    constexpr uint32_t kBad = 0xffffffffu;    // row slot without a valid lookup
    static_assert(U <= G && G % U == 0, "a group walks its G indices in steps of U");
    const int lane = threadIdx.x & 31;
    const int gl = lane % G;
    const int grp = lane / G;
    const unsigned gmask = (G == 32) ? 0xffffffffu : (((1u << G) - 1u) << (grp * G));
    const int64_t nbags = (int64_t)T * B;
    const bool small = nbags <= 0xffffffffll;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    bool chunk_on[C];
#pragma unroll
    for (int c = 0; c < C; c++)
        chunk_on[c] = c * G + gl < nchunks;
    const uint32_t row_bytes = (uint32_t)nchunks * 16;

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
        const char *tab = static_cast<const char *>(ts.ptr[t]) + gl * 16;  // this lane's first piece
        const int64_t R = ts.rows[t];

        float2 acc[C][EPC / 2];
#pragma unroll
        for (int c = 0; c < C; c++)
#pragma unroll
            for (int e = 0; e < EPC / 2; e++)
                acc[c][e] = make_float2(0.f, 0.f);

        for (int64_t kb = k0; kb < k1; kb += G) {
            const int n = (k1 - kb < G) ? (int)(k1 - kb) : G;
            // each lane checks one index; invalid ones and the slots past the
            // bag's end read nothing
            uint32_t row = kBad;
            if (gl < n) {
                const int64_t r = load_stream(indices + kb + gl);
                if (r >= 0 && r < R)
                    row = (uint32_t)r;
                else
                    raise_flag(err, DLRM_FLAG_INDEX_OOB);
            }
            for (int q = 0; q < n; q += U) {
                uint4 v[U][C];
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const uint32_t r = __shfl_sync(gmask, row, q + u, G);
                    const char *p = tab + (size_t)r * row_bytes;
#pragma unroll
                    for (int c = 0; c < C; c++)
                        v[u][c] = (r != kBad && chunk_on[c]) ? load_table(p + c * G * 16) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < U; u++)
#pragma unroll
                    for (int c = 0; c < C; c++)
                        Chunk16<TT>::add(acc[c], v[u][c]);
            }
        }

        float *o = out + b * oss + (int64_t)t * ots;
#pragma unroll
        for (int c = 0; c < C; c++) {
            if (chunk_on[c]) {
                float4 *dst = reinterpret_cast<float4 *>(o + (int64_t)(c * G + gl) * EPC);
#pragma unroll
                for (int e = 0; e < EPC / 4; e++)
                    __stcs(dst + e, make_float4(acc[c][2 * e].x, acc[c][2 * e].y, acc[c][2 * e + 1].x, acc[c][2 * e + 1].y));
            }
        }
    }
}

// Any d, any alignment: one warp per bag, one element per lane per step.
template <typename TT>
__global__ void __launch_bounds__(256)
emb_bag_fwd_scalar_kernel(TableSet ts, int T, int d, const int64_t *__restrict__ offsets,
                          const int64_t *__restrict__ indices, int64_t nnz, int64_t B,
                          float *__restrict__ out, int64_t oss, int64_t ots, int32_t *err)
{
    const int lane = threadIdx.x & 31;
    const int64_t nbags = (int64_t)T * B;
    const bool small = nbags <= 0xffffffffll;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t bag = warp; bag < nbags; bag += nwarps) {
        int t;
        int64_t b;
        bag_table_sample(bag, B, small, t, b);
        int64_t k0 = offsets[bag], k1 = offsets[bag + 1];
        if (k0 < 0 || k1 < k0 || k1 > nnz) {
            if (lane == 0)
                raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
            k0 = k1 = 0;
        }
        const TT *tab = static_cast<const TT *>(ts.ptr[t]);
        const int64_t R = ts.rows[t];
        float *o = out + b * oss + (int64_t)t * ots;
        for (int e0 = 0; e0 < d; e0 += 32) {
            const int e = e0 + lane;
            float acc = 0.f;
            for (int64_t k = k0; k < k1; k++) {
                const int64_t r = indices[k];
                if (r < 0 || r >= R) {
                    if (lane == 0 && e0 == 0)
                        raise_flag(err, DLRM_FLAG_INDEX_OOB);
                    continue;
                }
                if (e < d)
                    acc += to_f32(tab[r * d + e]);
            }
            if (e < d)
                o[e] = acc;
        }
    }
}

template <typename K>
static int grid_for(K kernel, int64_t work_blocks)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t resident = (int64_t)per_sm * sm_count();
    return (int)(work_blocks < resident ? (work_blocks < 1 ? 1 : work_blocks) : resident);
}

template <typename TT, int G, int C, int UF = 0>
static int launch_vec(const TableSet &ts, int T, int nchunks, const int64_t *offsets,
                      const int64_t *indices, int64_t nnz, int64_t B, float *out, int64_t oss,
                      int64_t ots, int32_t *err, cudaStream_t st)
{
    // 8 x 16 bytes in flight per lane; half-precision rows need twice the
    // accumulators, so wide half rows keep fewer in flight (UF > 0 sets it)
    constexpr int U0 = UF > 0 ? UF : (C == 1 ? 8 : (C == 2 ? 4 : 2)) / ((Chunk16<TT>::kElems == 8 && C > 1) ? 2 : 1);
    constexpr int U = U0 < G ? U0 : G;
    auto kernel = emb_bag_fwd_vec_kernel<TT, G, C, U>;
    const int64_t bags_per_block = 8 * (32 / G);
    const int grid = grid_for(kernel, ((int64_t)T * B + bags_per_block - 1) / bags_per_block);
    kernel<<<grid, 256, 0, st>>>(ts, T, nchunks, offsets, indices, nnz, B, out, oss, ots, err);
    count_launch(st);
    return launch_status();
}

template <typename TT>
static int launch_typed(const TableSet &ts, int T, int d, bool vec, const int64_t *offsets,
                        const int64_t *indices, int64_t nnz, int64_t B, float *out, int64_t oss,
                        int64_t ots, int32_t *err, cudaStream_t st)
{
    if (vec) {
        const int nchunks = (int)((int64_t)d * sizeof(TT) / 16);
        if (nchunks <= 4)
            return launch_vec<TT, 4, 1>(ts, T, nchunks, offsets, indices, nnz, B, out, oss, ots, err, st);
        if (nchunks <= 8)
            return launch_vec<TT, 8, 1>(ts, T, nchunks, offsets, indices, nnz, B, out, oss, ots, err, st);
        // half rows of 9 to 16 chunks (d = 72 .. 128): 8 lanes of two chunks each, 4 rows in
        // flight -- half the lanes' per-lookup work per byte, where the walk over L2-resident
        // rows is bound by issue (measured 6 % faster on Zipf indices, 4 % slower on uniform
        // ones, whose lookup stays at 0.74 of HBM)
        if (Chunk16<TT>::kElems == 8 && nchunks > 8 && nchunks <= 16 && nchunks % 2 == 0)
            return launch_vec<TT, 8, 2, 4>(ts, T, nchunks, offsets, indices, nnz, B, out, oss, ots, err, st);
        if (nchunks <= 16)
            return launch_vec<TT, 16, 1>(ts, T, nchunks, offsets, indices, nnz, B, out, oss, ots, err, st);
        if (nchunks <= 32)
            return launch_vec<TT, 32, 1>(ts, T, nchunks, offsets, indices, nnz, B, out, oss, ots, err, st);
        if (nchunks <= 64)
            return launch_vec<TT, 32, 2>(ts, T, nchunks, offsets, indices, nnz, B, out, oss, ots, err, st);
        if (nchunks <= 128)
            return launch_vec<TT, 32, 4>(ts, T, nchunks, offsets, indices, nnz, B, out, oss, ots, err, st);
    }
    auto kernel = emb_bag_fwd_scalar_kernel<TT>;
    const int grid = grid_for(kernel, ((int64_t)T * B + 7) / 8);
    kernel<<<grid, 256, 0, st>>>(ts, T, d, offsets, indices, nnz, B, out, oss, ots, err);
    count_launch(st);
    return launch_status();
}

// True when every row starts on a 16-byte boundary and rows are a whole
// number of 16-byte chunks no longer than 2 KB, and the output chunks are
// 16-byte aligned: the vectorised kernel's preconditions.
bool emb_bag_fwd_vectorisable(const TableSet &ts, int T, int d, int elem_bytes, const float *out,
                              int64_t oss, int64_t ots)
{
    const int64_t row_bytes = (int64_t)d * elem_bytes;
    if (row_bytes % 16 != 0 || row_bytes > 2048)
        return false;
    if (reinterpret_cast<uintptr_t>(out) % 16 != 0 || oss % 4 != 0 || ots % 4 != 0)
        return false;
    for (int t = 0; t < T; t++)
        if (reinterpret_cast<uintptr_t>(ts.ptr[t]) % 16 != 0)
            return false;
    return true;
}

int launch_emb_bag_fwd(const TableSet &ts, int T, int d, int dtype, bool vec, const int64_t *offsets,
                       const int64_t *indices, int64_t nnz, int64_t B, float *out, int64_t oss,
                       int64_t ots, int32_t *err, cudaStream_t st)
{
    switch (dtype) {
    case DLRM_F32:
        return launch_typed<float>(ts, T, d, vec, offsets, indices, nnz, B, out, oss, ots, err, st);
    case DLRM_F16:
        return launch_typed<__half>(ts, T, d, vec, offsets, indices, nnz, B, out, oss, ots, err, st);
    default:
        return launch_typed<__nv_bfloat16>(ts, T, d, vec, offsets, indices, nnz, B, out, oss, ots, err, st);
    }
}

}  // namespace dlrm
