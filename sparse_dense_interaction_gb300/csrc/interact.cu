// Pairwise dot-product interaction, forward and backward, on the CUDA cores
// (fp32 FMAs), and the dispatch between the kernel families.
//
// Follows "Notes/DLRM" (vault-aram.pages.dev), section 3 "The Pairwise
// Interaction Layer": one dot product per pair of the vectors
// {e0, e_1 .. e_N}, self pairs optional, the terms concatenated with e0.
//
// Dispatch: the tensor-core kernels (interact_tc.cu) where they apply, else
// for the forward the bulk-tensor-copy kernel (interact_tma.cu) where the
// copy engine can describe the operands, else the kernels below; all compute
// the same values within the fp32 tolerance.
//
// Forward design (operands neither of the others takes): a CTA takes S samples.  The F x d
// block Z of each sample
// (row 0 = e0, rows 1..N = pooled embeddings) is staged through shared memory
// in chunks of KC = 32 columns: each row chunk is one coalesced 128-byte read
// (4 lanes x 32 bytes), transposed to [k][i] (column groups XOR-swizzled by k
// so the transposing stores are conflict-free) so that four consecutive rows
// of one column are one 16-byte load.  Each thread owns one 4 x 4 tile of
// the lower triangle of Z Z^T and accumulates it in registers over all
// chunks (16 FMAs per two 16-byte shared loads; lanes of a warp share tile
// rows and columns, so those loads are broadcasts).  The triangle is staged
// in shared memory and written out as one contiguous, coalesced row per
// sample; the e0 copy (and, in the alongside layout, each pooled row) is
// written while Z is loaded.
//
// Backward design: dZ = (G + G^T) Z with G the lower-triangular matrix of
// upstream gradients.  A CTA takes S samples, expands dy into the symmetric
// matrix (G + G^T) in shared memory once, then streams Z in chunks of KC
// columns; each thread owns a 4-row x 4-column tile of dZ and loops over the
// F rows of the chunk (a broadcast 16-byte load of four G entries and a
// conflict-free 16-byte load of four Z entries per 16 FMAs).  dZ rows go
// straight to de0 (plus the e0 part of dy) and to the pooled gradients (plus
// their copies' part of dy in the alongside layout).
#include "interact.cuh"

namespace dlrm {

// 8 consecutive fp32 values of a row, zero past the end (d) or past B.
__device__ __forceinline__ void load8(const float *src, int k, int d, bool vec, float *v)
{
    if (vec && k + 8 <= d) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(src + k));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(src + k + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int m = 0; m < 8; m++)
            v[m] = (k + m < d) ? __ldg(src + k + m) : 0.f;
    }
}

// TS: staged row of Zt, Fp columns rounded up to a multiple of 32 (32, 64 or
// 128); a compile-time row width makes every shared-memory address of the
// inner loops an immediate offset.
template <int TS>
__global__ void __launch_bounds__(1024)
interact_fwd_kernel(const float *__restrict__ e0, int64_t e0s, const float *__restrict__ emb,
                    int64_t embs, int N, int d, int64_t B, int mode, float *__restrict__ y,
                    int64_t ys, int S, int vec_in, int vec_out)
{
    extern __shared__ __align__(16) float smem[];
    const int inc = mode & kInteractSelf;
    const bool along = (mode & kInteractAlongside) != 0;
    const int F = N + 1;
    const int64_t poff = along ? (int64_t)F * d : d;  // first pair column
    const int Fp = (F + 3) & ~3;
    const int nTR = Fp / 4;
    const int ntiles = nTR * (nTR + 1) / 2;
    const int64_t P = inc ? (int64_t)F * (F + 1) / 2 : (int64_t)F * (F - 1) / 2;
    float *Zt = smem;                                   // [S][kKC][TS], transposed chunk of Z
    float *ybuf = Zt + (size_t)S * kKC * TS;            // [S][P]
    uint8_t *tileI = reinterpret_cast<uint8_t *>(ybuf + (size_t)S * P);
    uint8_t *tileJ = tileI + ntiles;
    const int tid = threadIdx.x;
    const int64_t b0 = (int64_t)blockIdx.x * S;

    fill_tile_tables(ntiles, tileI, tileJ);

    const int s = tid / ntiles;
    const int tile = tid - s * ntiles;
    const bool active = s < S && b0 + s < B;
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < 4; c++)
            acc[r][c] = 0.f;

    const bool vec_y = vec_out != 0;
    const int rblocks = (F + 7) / 8;
    // staging work items: (sample, block of 8 rows) per warp, stepped by the
    // warp count without dividing in the loop
    const int lane = tid & 31, nwarps = blockDim.x >> 5;
    const int items = S * rblocks;
    const int wi0 = tid >> 5;
    const int ss0 = wi0 / rblocks, ib0 = wi0 - ss0 * rblocks;
    const int dss = nwarps / rblocks, dib = nwarps - dss * rblocks;
    const int q = lane >> 3;  // column octet of the lane
    for (int kc = 0; kc < d; kc += kKC) {
        // stage: a warp reads 8 rows x 4 column octets (32 bytes per lane, so
        // each row chunk is one coalesced 128-byte read) and transposes them
        int ss = ss0, ib = ib0;
        for (int wi = wi0; wi < items; wi += nwarps) {
            const int i = ib * 8 + (lane & 7);
            const int cur_ss = ss;
            ss += dss;
            ib += dib;
            if (ib >= rblocks) {
                ib -= rblocks;
                ss++;
            }
            if (i >= F)
                continue;
            const int64_t b = b0 + cur_ss;
            const int k = kc + 8 * q;
            float v[8];
            if (b < B && k < d) {
                const float *src = (i == 0) ? e0 + b * e0s : emb + b * embs + (int64_t)(i - 1) * d;
                load8(src, k, d, vec_in != 0, v);
                if (i == 0 || along) {  // e0, and the embeddings when they go alongside
                    float *dst = y + b * ys + (int64_t)i * d + k;
                    if (vec_y && k + 8 <= d) {
                        __stcs(reinterpret_cast<float4 *>(dst), make_float4(v[0], v[1], v[2], v[3]));
                        __stcs(reinterpret_cast<float4 *>(dst + 4), make_float4(v[4], v[5], v[6], v[7]));
                    } else {
                        for (int m = 0; m < 8; m++)
                            if (k + m < d)
                                dst[m] = v[m];
                    }
                }
            } else {
#pragma unroll
                for (int m = 0; m < 8; m++)
                    v[m] = 0.f;  // rows past d (or past B) are zero: the inner loop runs whole chunks
            }
            // the 8 rows of an octet share one swizzle: (8q + m) >> 3 == q
            float *zt = Zt + (size_t)cur_ss * kKC * TS + 8 * q * TS + zt_col(8 * q, i);
#pragma unroll
            for (int m = 0; m < 8; m++)
                zt[m * TS] = v[m];
        }
        __syncthreads();
        if (active) {
            const int I = tileI[tile], J = tileJ[tile];
            const float *zs = Zt + (size_t)s * kKC * TS;
#pragma unroll
            for (int kb = 0; kb < kKC / 8; kb++) {
                // within 8 consecutive rows the swizzle of a column group is fixed
                const float *pa = zs + kb * 8 * TS + ((I ^ (kb << 1)) << 2);
                const float *pb = zs + kb * 8 * TS + ((J ^ (kb << 1)) << 2);
#pragma unroll
                for (int m = 0; m < 8; m++) {
                    const float4 a = *reinterpret_cast<const float4 *>(pa + m * TS);
                    const float4 bb = *reinterpret_cast<const float4 *>(pb + m * TS);
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
        __syncthreads();
    }

    if (active) {
        const int I = tileI[tile], J = tileJ[tile];
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int i = 4 * I + r;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int j = 4 * J + c;
                if (i < F && (inc ? j <= i : j < i))
                    ybuf[(size_t)s * P + pair_pos(i, j, inc)] = acc[r][c];
            }
        }
    }
    __syncthreads();
    for (int64_t li = tid; li < (int64_t)S * P; li += blockDim.x) {
        const int ss = (int)(li / P);
        const int64_t p = li - (int64_t)ss * P;
        const int64_t b = b0 + ss;
        if (b < B)
            __stcs(y + b * ys + poff + p, ybuf[li]);
    }
}

__global__ void __launch_bounds__(1024)
interact_bwd_kernel(const float *__restrict__ e0, int64_t e0s, const float *__restrict__ emb,
                    int64_t embs, int N, int d, int64_t B, int mode, const float *__restrict__ dy,
                    int64_t dys, float *__restrict__ de0, int64_t de0s, float *__restrict__ demb,
                    int64_t dembs, int S, int vec_in, int vec_out)
{
    extern __shared__ __align__(16) float smem[];
    const int inc = mode & kInteractSelf;
    const bool along = (mode & kInteractAlongside) != 0;
    const int F = N + 1;
    const int64_t poff = along ? (int64_t)F * d : d;  // first pair column of dy
    const int Fp = (F + 3) & ~3;
    const int nTR = Fp / 4;
    constexpr int KQ = kKC / 4;
    const int items = nTR * KQ;
    float *Gs = smem;                            // [S][Fp][Fp], symmetric (G + G^T)
    float *Zc = Gs + (size_t)S * Fp * Fp;        // [S][F][kKC]
    const int tid = threadIdx.x;
    const int64_t b0 = (int64_t)blockIdx.x * S;

    for (int li = tid; li < S * Fp * Fp; li += blockDim.x) {
        const int ss = li / (Fp * Fp);
        const int rem = li - ss * Fp * Fp;
        const int i = rem / Fp, j = rem - (rem / Fp) * Fp;
        const int64_t b = b0 + ss;
        float g = 0.f;
        if (b < B && i < F && j < F) {
            const float *row = dy + b * dys + poff;
            if (i > j)
                g = row[pair_pos(i, j, inc)];
            else if (i < j)
                g = row[pair_pos(j, i, inc)];
            else if (inc)
                g = 2.f * row[pair_pos(i, i, inc)];
        }
        Gs[li] = g;
    }

    const int s = tid / items;
    const int rem = tid - s * items;
    const int I = rem / KQ, kq = rem - (rem / KQ) * KQ;
    const int64_t b = b0 + s;
    const bool active = s < S && b < B;

    for (int kc = 0; kc < d; kc += kKC) {
        for (int li = tid; li < S * F * (kKC / 8); li += blockDim.x) {
            const int q = li % (kKC / 8);
            const int r2 = li / (kKC / 8);
            const int j = r2 % F;
            const int ss = r2 / F;
            const int64_t bb = b0 + ss;
            const int k = kc + 8 * q;
            float v[8];
            if (bb < B && k < d) {
                const float *src = (j == 0) ? e0 + bb * e0s : emb + bb * embs + (int64_t)(j - 1) * d;
                load8(src, k, d, vec_in != 0, v);
            } else {
#pragma unroll
                for (int m = 0; m < 8; m++)
                    v[m] = 0.f;
            }
            float4 *dst = reinterpret_cast<float4 *>(Zc + ((size_t)ss * F + j) * kKC + 8 * q);
            dst[0] = make_float4(v[0], v[1], v[2], v[3]);
            dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
        __syncthreads();
        if (active) {
            float acc[4][4];
#pragma unroll
            for (int r = 0; r < 4; r++)
#pragma unroll
                for (int c = 0; c < 4; c++)
                    acc[r][c] = 0.f;
            const float *gs = Gs + (size_t)s * Fp * Fp + 4 * I;
            const float *zc = Zc + (size_t)s * F * kKC + 4 * kq;
#pragma unroll 4
            for (int j = 0; j < F; j++) {
                const float4 g4 = *reinterpret_cast<const float4 *>(gs + (size_t)j * Fp);
                const float4 z4 = *reinterpret_cast<const float4 *>(zc + (size_t)j * kKC);
                const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
                const float zv[4] = {z4.x, z4.y, z4.z, z4.w};
#pragma unroll
                for (int r = 0; r < 4; r++)
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        acc[r][c] = fmaf(gv[r], zv[c], acc[r][c]);
            }
            const int k = kc + 4 * kq;
            if (k < d) {
                const bool full = vec_out && k + 4 <= d;
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    const int i = 4 * I + r;
                    if (i >= F)
                        continue;
                    float out[4] = {acc[r][0], acc[r][1], acc[r][2], acc[r][3]};
                    float *dst;
                    if (i == 0 || along) {  // the gradient of the copy in the output
                        const float *dyr = dy + b * dys + (int64_t)i * d + k;
                        for (int c = 0; c < 4; c++)
                            if (k + c < d)
                                out[c] += __ldg(dyr + c);
                    }
                    if (i == 0)
                        dst = de0 + b * de0s + k;
                    else
                        dst = demb + b * dembs + (int64_t)(i - 1) * d + k;
                    if (full) {
                        __stcs(reinterpret_cast<float4 *>(dst), make_float4(out[0], out[1], out[2], out[3]));
                    } else {
                        for (int c = 0; c < 4; c++)
                            if (k + c < d)
                                dst[c] = out[c];
                    }
                }
            }
        }
        __syncthreads();
    }
}

static bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

int launch_interact_fwd_tma(const float *, int64_t, const float *, int64_t, int, int, int64_t, int, float *,
                            int64_t, cudaStream_t);
int launch_interact_fwd_tc(const float *, int64_t, const float *, int64_t, int, int, int64_t, int, float *,
                           int64_t, cudaStream_t);
int launch_interact_bwd_tc(const float *, int64_t, const float *, int64_t, int, int, int64_t, int, const float *,
                           int64_t, float *, int64_t, float *, int64_t, cudaStream_t);

int launch_interact_fwd(const float *e0, int64_t e0s, const float *emb, int64_t embs, int N, int d,
                        int64_t B, int mode, float *y, int64_t ys, cudaStream_t st)
{
    // the tensor-core kernel where it applies, else the bulk-tensor-copy
    // kernel when the copy engine can describe the operands
    if (interact_tensor_cores()) {
        const int r = launch_interact_fwd_tc(e0, e0s, emb, embs, N, d, B, mode, y, ys, st);
        if (r != 1)
            return r;
    }
    const int r = launch_interact_fwd_tma(e0, e0s, emb, embs, N, d, B, mode, y, ys, st);
    if (r != 1)
        return r;
    const int inc = mode & kInteractSelf;
    const int F = N + 1;
    const int Fp = (F + 3) & ~3;
    const int nTR = Fp / 4;
    const int ntiles = nTR * (nTR + 1) / 2;
    const int64_t P = num_pairs_of(F, inc);
    const int TS = (Fp + 31) & ~31;
    const size_t per_sample = ((size_t)kKC * TS + (size_t)P) * sizeof(float);
    int S = ntiles >= 256 ? 1 : 256 / ntiles;
    while (S > 1 && (size_t)S * per_sample > 96 * 1024)
        S--;
    if (S > B)
        S = (int)B;
    const int threads = ((S * ntiles + 31) / 32) * 32;
    const size_t smem = (size_t)S * per_sample + 2 * (size_t)ntiles;
    const int vec_in = d % 4 == 0 && aligned16(e0) && aligned16(emb) && e0s % 4 == 0 && embs % 4 == 0;
    const int vec_out = aligned16(y) && ys % 4 == 0;
    const int64_t grid = (B + S - 1) / S;
    auto kernel = TS == 32 ? interact_fwd_kernel<32> : (TS == 64 ? interact_fwd_kernel<64> : interact_fwd_kernel<128>);
    static std::atomic<unsigned long long> smem_set[3];  // per row width: devices whose limit has been raised
    if (allow_dynamic_smem(reinterpret_cast<const void *>(kernel), 200 * 1024,
                           &smem_set[TS == 32 ? 0 : (TS == 64 ? 1 : 2)]) != DLRM_OK)
        return DLRM_ERR_CUDA;
    kernel<<<(unsigned)grid, threads, smem, st>>>(e0, e0s, emb, embs, N, d, B, mode, y, ys, S, vec_in, vec_out);
    count_launch(st);
    return launch_status();
}

int launch_interact_bwd(const float *e0, int64_t e0s, const float *emb, int64_t embs, int N, int d,
                        int64_t B, int mode, const float *dy, int64_t dys, float *de0, int64_t de0s,
                        float *demb, int64_t dembs, cudaStream_t st)
{
    if (interact_tensor_cores()) {
        const int r = launch_interact_bwd_tc(e0, e0s, emb, embs, N, d, B, mode, dy, dys, de0, de0s, demb, dembs, st);
        if (r != 1)
            return r;
    }
    const int F = N + 1;
    const int Fp = (F + 3) & ~3;
    const int nTR = Fp / 4;
    const int items = nTR * (kKC / 4);
    const size_t per_sample = ((size_t)Fp * Fp + (size_t)F * kKC) * sizeof(float);
    int S = items >= 256 ? 1 : 256 / items;
    while (S > 1 && (size_t)S * per_sample > 96 * 1024)
        S--;
    if (S > B)
        S = (int)B;
    const int threads = ((S * items + 31) / 32) * 32;
    const size_t smem = (size_t)S * per_sample;
    static std::atomic<unsigned long long> smem_set{0};  // devices whose limit has been raised
    if (allow_dynamic_smem(reinterpret_cast<const void *>(interact_bwd_kernel), 200 * 1024, &smem_set) != DLRM_OK)
        return DLRM_ERR_CUDA;
    const int vec_in = d % 4 == 0 && aligned16(e0) && aligned16(emb) && e0s % 4 == 0 && embs % 4 == 0;
    const int vec_out = d % 4 == 0 && aligned16(de0) && aligned16(demb) && de0s % 4 == 0 && dembs % 4 == 0;
    const int64_t grid = (B + S - 1) / S;
    interact_bwd_kernel<<<(unsigned)grid, threads, smem, st>>>(e0, e0s, emb, embs, N, d, B, mode, dy, dys,
                                                               de0, de0s, demb, dembs, S, vec_in, vec_out);
    count_launch(st);
    return launch_status();
}

}  // namespace dlrm
