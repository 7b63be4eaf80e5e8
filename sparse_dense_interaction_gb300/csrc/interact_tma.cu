// Interaction forward on the CUDA cores, fed by the tensor memory accelerator
// (taken where the tensor-core kernel of interact_tc.cu does not apply, e.g.
// d < 32 or more than 128 vectors per sample).
//
// Same arithmetic as interact_fwd_kernel ("Notes/DLRM", vault-aram.pages.dev,
// section 3: one dot product per pair of {e0, e_1 .. e_N}, concatenated with
// e0): a CTA takes S samples; each 4 x 4 tile of the lower triangle of Z Z^T is
// owned by two adjacent lanes, each summing every other 16-byte column group
// of the 32-column chunks, and a butterfly shuffle adds the halves.  What
// differs is how the chunks reach shared memory: one thread issues, per
// sample, one 3-D bulk tensor copy of the 32-column slice of its N pooled rows
// and one of e0 into a stage, completing on the stage's mbarrier, while all
// threads compute on the other stage.  No thread waits on a global load; the
// copies use the 128-byte swizzle (the 16-byte chunk index of a 128-byte row
// XOR-ed with the row index mod 8), so the loads of four consecutive columns
// of eight different rows hit distinct banks.
//
// Layout of a sample's slot in a stage (1024-byte aligned): R8 = N rounded up
// to 8 rows of 128 bytes (pooled row i-1 holds z_i), then e0 at the start of
// its own 1024-byte block, i.e. as row R8, where the swizzle is the identity:
// element k of slot row r is at r*128 + ((k/4 ^ (r % 8)) * 16) + (k % 4) * 4.
//
// Waits on the mbarriers are bounded.  A CTA whose wait runs out waits again,
// bounded, for its copies still in flight, writes NaN into its samples'
// outputs (the call has no error flag; a poisoned output is visible) and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "interact.cuh"

namespace dlrm {

namespace {

constexpr int kSpinLimitTma = 1 << 22;  // polls of a stage barrier (far beyond any copy's latency)
constexpr int kTmaLanesPerTile = 2;     // lanes sharing a 4 x 4 tile (each sums every other column group)

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// true once the phase of the given parity has completed; gives up after
// `polls` polls
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int polls = kSpinLimitTma)
{
    uint32_t done = 0;
    for (int it = 0; it < polls && !done; it++)
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(done)
                     : "r"(smem_u32(bar)), "r"(parity)
                     : "memory");
    return done != 0;
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace

template <int KS>  // lanes per tile
__global__ void __launch_bounds__(512, 2)
interact_fwd_tma_kernel(const __grid_constant__ CUtensorMap map_emb, const __grid_constant__ CUtensorMap map_e0,
                        int N, int d, int64_t B, int mode, float *__restrict__ y, int64_t ys, int S, int R8,
                        int wait_polls)
{
    extern __shared__ unsigned char smem_raw[];
    const int inc = mode & kInteractSelf;
    const bool along = (mode & kInteractAlongside) != 0;
    const int F = N + 1;
    const int64_t poff = along ? (int64_t)F * d : d;
    const int Fp = (F + 3) & ~3;
    const int nTR = Fp / 4;
    const int ntiles = nTR * (nTR + 1) / 2;
    const int64_t P = num_pairs_of(F, inc);
    const int slot = R8 * 128 + 1024;  // bytes per sample and stage
    // 1024-byte aligned start of the stages
    unsigned char *base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const size_t stage_bytes = (size_t)S * slot;  // stage st starts at base + st * stage_bytes
    float *ybuf = reinterpret_cast<float *>(base + 2 * stage_bytes);  // [S][P]
    uint64_t *bar = reinterpret_cast<uint64_t *>(ybuf + (size_t)S * P + ((S * P) & 1));
    uint8_t *tileI = reinterpret_cast<uint8_t *>(bar + 2);
    uint8_t *tileJ = tileI + ntiles;
    __shared__ int failed;

    const int tid = threadIdx.x;
    const int64_t b0 = (int64_t)blockIdx.x * S;
    const int nS = (int)(B - b0 < S ? B - b0 : S);
    const int nchunks = (d + kKC - 1) / kKC;
    const uint32_t bytes = (uint32_t)nS * 128u * (uint32_t)(N + 1);

    fill_tile_tables(ntiles, tileI, tileJ);
    if (tid == 0) {
        failed = 0;
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    auto issue = [&](int c) {  // chunk c into stage c % 2 (thread 0)
        const int st = c & 1;
        mbar_expect_tx(&bar[st], bytes);
        for (int s = 0; s < nS; s++) {
            unsigned char *dst = base + st * stage_bytes + (size_t)s * slot;
            tma_load_3d(dst, &map_emb, c * kKC, 0, (int)(b0 + s), &bar[st]);
            tma_load_2d(dst + R8 * 128, &map_e0, c * kKC, (int)(b0 + s), &bar[st]);
        }
    };
    if (tid == 0) {
        issue(0);
        if (nchunks > 1)
            issue(1);
    }

    // KS adjacent lanes per tile: lane ks takes the 16-byte column groups
    // k4 = ks, ks + KS, ... of each chunk
    const int s = tid / (KS * ntiles);
    const int rem = tid - s * KS * ntiles;
    const int tile = rem / KS, ks = rem % KS;
    const bool active = s < nS;
    int I = 0, J = 0;
    // row words: slot offset of the row OR its swizzle (bits 4..6); the
    // address of 16-byte group k4 is then slot + (word ^ (k4 << 4))
    uint32_t rw[8];
#pragma unroll
    for (int q = 0; q < 8; q++)
        rw[q] = 0;
    if (active) {
        I = tileI[tile];
        J = tileJ[tile];
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int i = q < 4 ? 4 * I + q : 4 * J + (q - 4);
            const uint32_t sr = i == 0 ? (uint32_t)R8 : (uint32_t)(i - 1);  // e0 sits at row R8
            rw[q] = (sr << 7) | ((sr & 7u) << 4);
        }
    }
    float acc[4][4];
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < 4; c++)
            acc[r][c] = 0.f;

    const bool vec_y = (reinterpret_cast<uintptr_t>(y) % 16 == 0) && ys % 4 == 0;
    int waited = 0;  // chunks whose stage this CTA has seen complete
    for (int c = 0; c < nchunks; c++) {
        const int st = c & 1;
        if (!mbar_wait(&bar[st], (uint32_t)((c >> 1) & 1), wait_polls))
            failed = 1;
        __syncthreads();
        if (failed)
            break;
        waited = c + 1;
        const unsigned char *stg = base + st * stage_bytes;
        const int kc = c * kKC;
        // e0 (and the pooled rows when they go alongside) into the output, 16 bytes at a time
        const int rows_out = along ? F : 1;
        for (int li = tid; li < nS * rows_out * (kKC / 4); li += blockDim.x) {
            const int k4 = li & (kKC / 4 - 1);
            const int rr = li >> 3;
            const int ss = rr / rows_out, i = rr - ss * rows_out;
            const int k = kc + 4 * k4;
            if (k >= d)
                continue;  // d % 4 == 0: a group is whole or past the end
            const uint32_t sr = i == 0 ? (uint32_t)R8 : (uint32_t)(i - 1);
            const float4 v = *reinterpret_cast<const float4 *>(stg + (size_t)ss * slot + (sr << 7) +
                                                               ((((uint32_t)k4) ^ (sr & 7u)) << 4));
            float *dst = y + (b0 + ss) * ys + (int64_t)i * d + k;
            if (vec_y) {
                __stcs(reinterpret_cast<float4 *>(dst), v);
            } else {
                dst[0] = v.x;
                dst[1] = v.y;
                dst[2] = v.z;
                dst[3] = v.w;
            }
        }
        if (active) {
            const unsigned char *sl = stg + (size_t)s * slot;
#pragma unroll
            for (int h = 0; h < kKC / 4 / KS; h++) {
                const uint32_t kx = (uint32_t)(KS * h + ks) << 4;
                float4 bv[4];
#pragma unroll
                for (int q = 0; q < 4; q++)
                    bv[q] = *reinterpret_cast<const float4 *>(sl + (rw[4 + q] ^ kx));
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    const float4 av = *reinterpret_cast<const float4 *>(sl + (rw[r] ^ kx));
#pragma unroll
                    for (int cc = 0; cc < 4; cc++) {
                        acc[r][cc] = fmaf(av.x, bv[cc].x, acc[r][cc]);
                        acc[r][cc] = fmaf(av.y, bv[cc].y, acc[r][cc]);
                        acc[r][cc] = fmaf(av.z, bv[cc].z, acc[r][cc]);
                        acc[r][cc] = fmaf(av.w, bv[cc].w, acc[r][cc]);
                    }
                }
            }
        }
        __syncthreads();  // the stage has been read
        if (tid == 0 && c + 2 < nchunks) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(c + 2);
        }
    }
    // the lanes of a tile add their parts (all lanes of the warp take part)
#pragma unroll
    for (int o = 1; o < KS; o <<= 1)
#pragma unroll
        for (int r = 0; r < 4; r++)
#pragma unroll
            for (int cc = 0; cc < 4; cc++)
                acc[r][cc] += __shfl_xor_sync(0xffffffffu, acc[r][cc], o);

    if (failed) {
        // copies still in flight target this CTA's shared memory: wait for
        // them (bounded by the default limit, whatever the main loop's) before
        // leaving, and poison the outputs
        for (int c = waited; c < nchunks && c < waited + 2; c++)
            mbar_wait(&bar[c & 1], (uint32_t)((c >> 1) & 1), kSpinLimitTma);
        __syncthreads();
        for (int64_t li = tid; li < (int64_t)nS * P; li += blockDim.x) {
            const int ss = (int)(li / P);
            y[(b0 + ss) * ys + poff + (li - (int64_t)ss * P)] = __int_as_float(0x7fc00000);
        }
        return;
    }

    if (active) {
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const int i = 4 * I + r;
            if (r % KS != ks)
                continue;  // lane ks writes rows r with r % KS == ks
#pragma unroll
            for (int cc = 0; cc < 4; cc++) {
                const int j = 4 * J + cc;
                if (i < F && (inc ? j <= i : j < i))
                    ybuf[(size_t)s * P + pair_pos(i, j, inc)] = acc[r][cc];
            }
        }
    }
    __syncthreads();
    for (int64_t li = tid; li < (int64_t)nS * P; li += blockDim.x) {
        const int ss = (int)(li / P);
        __stcs(y + (b0 + ss) * ys + poff + (li - (int64_t)ss * P), ybuf[li]);
    }
}

// cuTensorMapEncodeTiled from the driver, looked up through the runtime (no
// link against the driver library); null if the driver has none.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    // looked up once (a function-local static is initialised thread-safely)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        return nullptr;
    }();
    return fn;
}

// Returns 1 (not launched) when the copy engine cannot describe these
// operands: rows not of whole 16-byte chunks, unaligned bases or strides,
// no pooled rows, or no encoder.  Otherwise launches and returns the status.
int launch_interact_fwd_tma(const float *e0, int64_t e0s, const float *emb, int64_t embs, int N, int d, int64_t B,
                            int mode, float *y, int64_t ys, cudaStream_t st)
{
    auto al16 = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    if (N < 1 || d % 4 != 0 || e0s % 4 != 0 || embs % 4 != 0 || !al16(e0) || !al16(emb) || B > 0x7fffffff)
        return 1;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return 1;
    CUtensorMap map_emb, map_e0;
    std::memset(&map_emb, 0, sizeof map_emb);
    std::memset(&map_e0, 0, sizeof map_e0);
    const cuuint64_t dims3[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides3[2] = {(cuuint64_t)d * 4, (cuuint64_t)embs * 4};
    const cuuint32_t box3[3] = {(cuuint32_t)kKC, (cuuint32_t)N, 1};
    const cuuint32_t one3[3] = {1, 1, 1};
    if (enc(&map_emb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(emb), dims3, strides3, box3, one3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const cuuint64_t dims2[2] = {(cuuint64_t)d, (cuuint64_t)B};
    const cuuint64_t strides2[1] = {(cuuint64_t)e0s * 4};
    const cuuint32_t box2[2] = {(cuuint32_t)kKC, 1};
    const cuuint32_t one2[2] = {1, 1};
    if (enc(&map_e0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(e0), dims2, strides2, box2, one2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;

    const int F = N + 1, Fp = (F + 3) & ~3, nTR = Fp / 4, ntiles = nTR * (nTR + 1) / 2;
    const int64_t P = num_pairs_of(F, mode & kInteractSelf);
    const int R8 = (N + 7) / 8 * 8;
    const size_t slot = (size_t)R8 * 128 + 1024;
    auto smem_for = [&](int S) {
        return 1024 + 2 * (size_t)S * slot + ((size_t)S * P + 1) * 4 + 16 + 2 * (size_t)ntiles;
    };
    constexpr int KS = kTmaLanesPerTile;
    int S = KS * ntiles >= 512 ? 1 : 512 / (KS * ntiles);
    if (S > 8)
        S = 8;
    while (S > 1 && smem_for(S) > 112 * 1024)
        S--;
    if (S > B)
        S = (int)B;
    const size_t smem = smem_for(S);
    if (smem > 112 * 1024 || (int64_t)S * KS * ntiles > 512)  // two CTAs of up to 512 threads per SM
        return 1;
    const int threads = ((S * KS * ntiles + 31) / 32) * 32;
    static std::atomic<unsigned long long> smem_set{0};  // devices whose limit has been raised
    if (allow_dynamic_smem(reinterpret_cast<const void *>(interact_fwd_tma_kernel<KS>), 200 * 1024, &smem_set) !=
        DLRM_OK)
        return DLRM_ERR_CUDA;
    const int64_t grid = (B + S - 1) / S;
    const int wait_polls = wait_hooks(0, kSpinLimitTma).copy_polls;  // the default unless a test shortens it
    interact_fwd_tma_kernel<KS><<<(unsigned)grid, threads, smem, st>>>(map_emb, map_e0, N, d, B, mode, y, ys, S, R8,
                                                                       wait_polls);
    count_launch(st);
    return launch_status();
}

}  // namespace dlrm
