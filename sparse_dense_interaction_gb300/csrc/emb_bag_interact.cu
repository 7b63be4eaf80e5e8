// Fused embedding-bag forward + interaction forward.
//
// "Notes/DLRM" (vault-aram.pages.dev), section 3: the pairwise interaction
// directly follows the embedding lookups, and its inputs are the pooled
// vectors of section 2 (summed per section 9) together with the bottom-MLP
// output e0.  Computed one after the other, the pooled [B][T][d] block is
// written by the lookup and read back by the interaction; here a CTA keeps
// the whole F x d block Z of each of its samples in shared memory, so the
// pooled vectors go to global memory only when the caller asks for them (the
// backward needs them; inference does not).
//
// Design: a CTA takes S samples.
//  1. Gather: a group of G lanes sums one bag at a time with the lane layout
//     and add order of the standalone lookup (each lane owns C 16-byte row
//     chunks, U rows in flight), so the pooled values are bit-identical to
//     dlrm_emb_bag_fwd's.  The sums are stored transposed, Zt[k][i] with the
//     column groups XOR-swizzled by k, next to e0 in column 0.
//  2. Gram triangle: each 4 x 4 tile of the lower triangle of Z Z^T is
//     shared by KS adjacent lanes, lane ks summing the 8-column blocks with
//     (k / 8) % KS == ks (16 FMAs per two 16-byte shared loads); the KS
//     partial tiles are added by butterfly shuffles.  Splitting the columns
//     keeps S small, so several CTAs fit an SM and the gathers of some
//     overlap the arithmetic of others.
//  3. The triangle is staged in shared memory and written as one contiguous
//     row per sample; e0 is copied while Z is built.
#include "interact.cuh"

namespace dlrm {

template <typename TT, int G, int C, int U>
__global__ void __launch_bounds__(256, 4)
emb_bag_interact_fwd_kernel(TableSet ts, int T, int d, int nchunks, const int64_t *__restrict__ offsets,
                            const int64_t *__restrict__ indices, int64_t nnz, int64_t B,
                            const float *__restrict__ e0, int64_t e0s, int mode, float *__restrict__ y,
                            int64_t ys, float *__restrict__ pooled, int64_t pss, int64_t pts, int S, int KS,
                            int32_t *err)
{
    extern __shared__ __align__(16) float smem[];
    constexpr int EPC = Chunk16<TT>::kElems;  // elements per 16-byte chunk
    constexpr uint32_t kBad = 0xffffffffu;    // row slot without a valid lookup
    static_assert(U <= G && G % U == 0, "a group walks its G indices in steps of U");
    const int inc = mode & kInteractSelf;
    const bool along = (mode & kInteractAlongside) != 0;
    const int F = T + 1;
    const int Fp = (F + 3) & ~3;
    const int TS = (Fp + 31) & ~31;  // staged row of Zt: Fp columns, swizzled
    const int nTR = Fp / 4;
    const int ntiles = nTR * (nTR + 1) / 2;
    const int dpad = (d + 8 * KS - 1) / (8 * KS) * (8 * KS);  // rows of Zt; rows d.. are zero
    const int64_t P = num_pairs_of(F, inc);
    float *Zt = smem;                             // [S][dpad][TS]
    float *ybuf = Zt + (size_t)S * dpad * TS;     // [S][P]
    uint8_t *tileI = reinterpret_cast<uint8_t *>(ybuf + (size_t)S * P);
    uint8_t *tileJ = tileI + ntiles;
    const int tid = threadIdx.x;
    const int64_t b0 = (int64_t)blockIdx.x * S;
    const int nS = (int)(B - b0 < S ? B - b0 : S);  // samples of this CTA

    fill_tile_tables(ntiles, tileI, tileJ);
    // e0 into column 0 and the output; zero rows past d
    for (int idx = tid; idx < nS * d; idx += blockDim.x) {
        const int ss = idx / d, k = idx - ss * d;
        const float v = e0[(b0 + ss) * e0s + k];
        Zt[((size_t)ss * dpad + k) * TS + zt_col(k, 0)] = v;
        __stcs(y + (b0 + ss) * ys + k, v);
    }
    for (int idx = tid; idx < nS * (dpad - d) * TS; idx += blockDim.x) {
        const int ss = idx / ((dpad - d) * TS), r = idx - ss * (dpad - d) * TS;
        Zt[((size_t)ss * dpad + d) * TS + r] = 0.f;
    }

    // 1. gather: group grp sums bags grp, grp + ngrp, ... of the CTA's nS*T
    {
        const int lane = tid & 31;
        const int gl = lane % G;
        const int grp = tid / G;
        const int ngrp = blockDim.x / G;
        const unsigned gmask = (G == 32) ? 0xffffffffu : (((1u << G) - 1u) << ((lane / G) * G));
        bool chunk_on[C];
#pragma unroll
        for (int c = 0; c < C; c++)
            chunk_on[c] = c * G + gl < nchunks;
        const uint32_t row_bytes = (uint32_t)nchunks * 16;
        for (int bi = grp; bi < nS * T; bi += ngrp) {
            const int ss = bi / T, t = bi - ss * T;
            const int64_t b = b0 + ss;
            const int64_t bag = (int64_t)t * B + b;
            int64_t k0 = offsets[bag];
            int64_t k1 = offsets[bag + 1];
            if (k0 < 0 || k1 < k0 || k1 > nnz) {
                if (gl == 0)
                    raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
                k0 = k1 = 0;
            }
            const char *tab = static_cast<const char *>(ts.ptr[t]) + gl * 16;
            const int64_t R = ts.rows[t];
            float2 acc[C][EPC / 2];
#pragma unroll
            for (int c = 0; c < C; c++)
#pragma unroll
                for (int e = 0; e < EPC / 2; e++)
                    acc[c][e] = make_float2(0.f, 0.f);
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
                    uint4 v[U][C];
#pragma unroll
                    for (int u = 0; u < U; u++) {
                        const uint32_t r = __shfl_sync(gmask, row, q + u, G);
                        const char *p = tab + (size_t)r * row_bytes;
#pragma unroll
                        for (int c = 0; c < C; c++)
                            v[u][c] = (r != kBad && chunk_on[c]) ? load_table(p + c * G * 16)
                                                                 : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < U; u++)
#pragma unroll
                        for (int c = 0; c < C; c++)
                            Chunk16<TT>::add(acc[c], v[u][c]);
                }
            }
            float *zs = Zt + (size_t)ss * dpad * TS;
#pragma unroll
            for (int c = 0; c < C; c++) {
                if (!chunk_on[c])
                    continue;
                const int e = (c * G + gl) * EPC;
#pragma unroll
                for (int m = 0; m < EPC / 2; m++) {
                    zs[(size_t)(e + 2 * m) * TS + zt_col(e + 2 * m, t + 1)] = acc[c][m].x;
                    zs[(size_t)(e + 2 * m + 1) * TS + zt_col(e + 2 * m + 1, t + 1)] = acc[c][m].y;
                }
                if (pooled) {
                    float4 *dst = reinterpret_cast<float4 *>(pooled + b * pss + (int64_t)t * pts + e);
#pragma unroll
                    for (int q = 0; q < EPC / 4; q++)
                        __stcs(dst + q, make_float4(acc[c][2 * q].x, acc[c][2 * q].y, acc[c][2 * q + 1].x,
                                                    acc[c][2 * q + 1].y));
                }
                if (along) {  // the pooled vector alongside, in column block t + 1 of y
                    float *dst = y + b * ys + (int64_t)(t + 1) * d + e;
#pragma unroll
                    for (int m = 0; m < EPC / 2; m++) {
                        __stcs(dst + 2 * m, acc[c][m].x);
                        __stcs(dst + 2 * m + 1, acc[c][m].y);
                    }
                }
            }
        }
    }
    __syncthreads();

    // 2. Gram triangle, KS lanes per 4 x 4 tile; the trip count is the same
    // for every thread, so the shuffles below always see full warps
    const int work = S * ntiles * KS;
    for (int w0 = 0; w0 < work; w0 += blockDim.x) {
        const int wi = w0 + tid;
        const int ks = wi % KS;
        const int tt = wi / KS;
        const int s = tt / ntiles, tile = tt - s * ntiles;
        const bool active = wi < work && s < nS;
        float acc[4][4];
#pragma unroll
        for (int r = 0; r < 4; r++)
#pragma unroll
            for (int c = 0; c < 4; c++)
                acc[r][c] = 0.f;
        int I = 0, J = 0;
        if (active) {
            I = tileI[tile];
            J = tileJ[tile];
            const float *zs = Zt + (size_t)s * dpad * TS;
            for (int kb = 8 * ks; kb < dpad; kb += 8 * KS) {
#pragma unroll
                for (int m = 0; m < 8; m++) {
                    const int k = kb + m;
                    const float4 a = *reinterpret_cast<const float4 *>(zs + (size_t)k * TS + zt_col(k, 4 * I));
                    const float4 bb = *reinterpret_cast<const float4 *>(zs + (size_t)k * TS + zt_col(k, 4 * J));
                    const float av[4] = {a.x, a.y, a.z, a.w};
                    const float bv[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                    for (int r = 0; r < 4; r++)
#pragma unroll
                        for (int c = 0; c < 4; c++)
                            acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
                }
            }
        }
        for (int o = 1; o < KS; o <<= 1)
#pragma unroll
            for (int r = 0; r < 4; r++)
#pragma unroll
                for (int c = 0; c < 4; c++)
                    acc[r][c] += __shfl_xor_sync(0xffffffffu, acc[r][c], o);
        if (active) {
            // lane ks of the tile writes rows r with r % KS == ks
#pragma unroll
            for (int r = 0; r < 4; r++) {
                const int i = 4 * I + r;
                if (r % KS != ks || i >= F)
                    continue;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int j = 4 * J + c;
                    if (inc ? j <= i : j < i)
                        ybuf[(size_t)s * P + pair_pos(i, j, inc)] = acc[r][c];
                }
            }
        }
    }
    __syncthreads();

    // 3. the triangle rows, contiguous per sample
    for (int64_t li = tid; li < (int64_t)nS * P; li += blockDim.x) {
        const int ss = (int)(li / P);
        const int64_t p = li - (int64_t)ss * P;
        __stcs(y + (b0 + ss) * ys + (along ? (int64_t)F * d : d) + p, ybuf[li]);
    }
}

// Shape of a launch: samples per CTA, lanes per tile, threads and shared
// memory (the same struct is declared where the C ABI dispatches).
struct FusedShape {
    int S, KS, threads;
    size_t smem;
};

static size_t fused_smem(int S, int KS, int F, int d, int inc)
{
    const int Fp = (F + 3) & ~3, TS = (Fp + 31) & ~31, nTR = Fp / 4, ntiles = nTR * (nTR + 1) / 2;
    const int dpad = (d + 8 * KS - 1) / (8 * KS) * (8 * KS);
    return (size_t)S * ((size_t)dpad * TS + (size_t)num_pairs_of(F, inc)) * sizeof(float) + 2 * (size_t)ntiles;
}

// Largest shared memory the fused kernel is given per CTA; beyond it (about
// F > 32 with d > 256) the two-kernel path is used.
static const size_t kFusedSmemMax = 100 * 1024;

bool emb_bag_interact_shape(int T, int d, int inc, int64_t B, FusedShape &fs)
{
    const int F = T + 1, Fp = (F + 3) & ~3, nTR = Fp / 4, ntiles = nTR * (nTR + 1) / 2;
    fs.threads = 256;
    // four lanes per tile for two or more samples if they fit, else fewer
    fs.KS = ntiles * 4 * 2 <= fs.threads ? 4 : (ntiles * 2 * 2 <= fs.threads ? 2 : 1);
    fs.S = fs.threads / (ntiles * fs.KS);
    if (fs.S < 1)
        fs.S = 1;
    if (fs.S > 4)
        fs.S = 4;
    if (fs.S > B)
        fs.S = (int)(B < 1 ? 1 : B);
    while (fs.S > 1 && fused_smem(fs.S, fs.KS, F, d, inc) > kFusedSmemMax)
        fs.S--;
    fs.smem = fused_smem(fs.S, fs.KS, F, d, inc);
    return fs.smem <= kFusedSmemMax;
}

template <typename TT, int G, int C>
static int launch_fused(const TableSet &ts, int T, int d, int nchunks, const int64_t *offsets,
                        const int64_t *indices, int64_t nnz, int64_t B, const float *e0, int64_t e0s, int mode,
                        float *y, int64_t ys, float *pooled, int64_t pss, int64_t pts, const FusedShape &fs,
                        int32_t *err, cudaStream_t st)
{
    constexpr int U0 = (C == 1 ? 8 : (C == 2 ? 4 : 2)) / ((Chunk16<TT>::kElems == 8 && C > 1) ? 2 : 1);
    constexpr int U = U0 < G ? U0 : G;
    auto kernel = emb_bag_interact_fwd_kernel<TT, G, C, U>;
    static std::atomic<unsigned long long> smem_set{0};  // devices whose limit has been raised
    if (allow_dynamic_smem(reinterpret_cast<const void *>(kernel), (int)kFusedSmemMax, &smem_set) != DLRM_OK)
        return DLRM_ERR_CUDA;
    const int64_t grid = (B + fs.S - 1) / fs.S;
    kernel<<<(unsigned)grid, fs.threads, fs.smem, st>>>(ts, T, d, nchunks, offsets, indices, nnz, B, e0, e0s,
                                                        mode, y, ys, pooled, pss, pts, fs.S, fs.KS, err);
    count_launch(st);
    return launch_status();
}

template <typename TT>
static int fused_typed(const TableSet &ts, int T, int d, const int64_t *offsets, const int64_t *indices,
                       int64_t nnz, int64_t B, const float *e0, int64_t e0s, int mode, float *y, int64_t ys,
                       float *pooled, int64_t pss, int64_t pts, const FusedShape &fs, int32_t *err,
                       cudaStream_t st)
{
    const int nchunks = (int)((int64_t)d * sizeof(TT) / 16);
    if (nchunks <= 4)
        return launch_fused<TT, 4, 1>(ts, T, d, nchunks, offsets, indices, nnz, B, e0, e0s, mode, y, ys, pooled,
                                      pss, pts, fs, err, st);
    if (nchunks <= 8)
        return launch_fused<TT, 8, 1>(ts, T, d, nchunks, offsets, indices, nnz, B, e0, e0s, mode, y, ys, pooled,
                                      pss, pts, fs, err, st);
    if (nchunks <= 16)
        return launch_fused<TT, 16, 1>(ts, T, d, nchunks, offsets, indices, nnz, B, e0, e0s, mode, y, ys, pooled,
                                       pss, pts, fs, err, st);
    if (nchunks <= 32)
        return launch_fused<TT, 32, 1>(ts, T, d, nchunks, offsets, indices, nnz, B, e0, e0s, mode, y, ys, pooled,
                                       pss, pts, fs, err, st);
    return launch_fused<TT, 32, 2>(ts, T, d, nchunks, offsets, indices, nnz, B, e0, e0s, mode, y, ys, pooled, pss,
                                   pts, fs, err, st);
}

int launch_emb_bag_interact_fwd(const TableSet &ts, int T, int d, int dtype, const int64_t *offsets,
                                const int64_t *indices, int64_t nnz, int64_t B, const float *e0, int64_t e0s,
                                int mode, float *y, int64_t ys, float *pooled, int64_t pss, int64_t pts,
                                const FusedShape &fs, int32_t *err, cudaStream_t st)
{
    switch (dtype) {
    case DLRM_F32:
        return fused_typed<float>(ts, T, d, offsets, indices, nnz, B, e0, e0s, mode, y, ys, pooled, pss, pts, fs,
                                  err, st);
    case DLRM_F16:
        return fused_typed<__half>(ts, T, d, offsets, indices, nnz, B, e0, e0s, mode, y, ys, pooled, pss, pts, fs,
                                   err, st);
    default:
        return fused_typed<__nv_bfloat16>(ts, T, d, offsets, indices, nnz, B, e0, e0s, mode, y, ys, pooled, pss,
                                          pts, fs, err, st);
    }
}

}  // namespace dlrm
