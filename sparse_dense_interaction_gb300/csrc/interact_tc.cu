// Interaction forward and backward on the fifth-generation tensor cores
// (tcgen05, TF32 MMAs, accumulators in tensor memory).
//
// Computes what "Notes/DLRM" (vault-aram.pages.dev), section 3 "The Pairwise
// Interaction Layer", defines: one dot product per pair of the vectors
// {e0, e_1 .. e_N} (strict or self-inclusive pairs), concatenated with e0 and
// optionally with the pooled embeddings; the backward by the product rule.
// Per sample Z is the F x d block of those vectors (row 0 = e0); the pairs
// are the lower triangle of Z Z^T, and dZ = (G + G^T) Z with G the pair
// gradients in the lower triangle.
//
// Precision: fp32 through TF32 MMAs on a split of the operands into a TF32
// part and a TF32-rounded remainder; the products keep about 20 bits (the
// dropped remainder.remainder term is below 2^-20 of |x||x'|), accumulated in
// fp32.
//
// The kernels are persistent (one CTA per SM) and warp-specialised over 14
// warps; every hand-off is an mbarrier:
//   epilogue      tensor-memory lanes 32 (w % 4) .. + 31 of a finished
//                 accumulator -> global memory (forward: warps 0..3;
//                 backward: two groups, warps 0..3 and 4..7, alternate units);
//   converters    raw rows (landed in shared memory by bulk tensor copies) ->
//                 the split A operand, written straight into tensor memory
//                 (forward: two groups, warps 4..7 and 8..11, alternate
//                 chunks; backward: warps 8..11);
//   warp 12       the copies (one lane issues the bulk tensor copies);
//   warp 13       allocates tensor memory; one lane issues the MMAs and
//                 commits operand slots and accumulators back.
// Shared memory that the tensor core reads is written by the bulk copies
// (forward) or, for the small Gs operand of the backward, by the converters
// behind a proxy fence.  Every wait is bounded; a CTA whose wait runs out
// stops all its roles, waits (bounded) for its copies and MMAs in flight,
// frees its tensor memory and writes NaN into its outputs (the calls have no
// error flag; a poisoned output is visible).
#include <cstring>

#include "interact.cuh"
#include "tc.cuh"

namespace dlrm {

namespace {

constexpr int kEpiThreads = 128;               // warps 0..3
constexpr int kEpiBarrier = 1;                 // named barrier of the epilogue warps
constexpr size_t kMaxSmem = 227 * 1024 - 256;  // the opt-in limit less the static variables

// true on every participating thread iff pred holds on all of them
__device__ __forceinline__ bool all_of(bool pred, int id, int threads)
{
    uint32_t r;
    asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.red.and.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(id), "r"(threads)
                 : "memory");
    return r != 0;
}

// byte offset of 16-byte unit q of row r in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(int r, int q) { return (uint32_t)r * 128u + ((uint32_t)(q ^ (r & 7)) << 4); }

// Waits for the tensor core to finish what this thread issued, and for the
// barrier arrivals of its earlier commits, before the CTA frees its tensor
// memory and leaves: no commit may arrive on the shared memory of a CTA that
// has exited, whether it left normally (nobody waits on the last phases of
// the slot-free barriers) or gave up.  Bounded.
__device__ __forceinline__ void drain_mmas(uint64_t *bar)
{
    tc::mma_commit(bar);
    for (int k = 0; k < tc::kSpinLimit && !tc::mbar_try_wait(bar, 0); k++) {
    }
}

}  // namespace

// ----------------------------------------------------------------- forward
//
// Tiles: the F rows of a sample are padded to Fb = 32, 64 or 128 and
// SPT = 128 / Fb samples share one 128-row tile.  The MMA computes
// D = A . B^T, M = 128, N = 144, K = 8 per instruction, per 32-column chunk
// of d:
//   B (shared memory, raw fp32 as the bulk tensor copies leave it; the MMA
//     reads each value truncated to TF32, t = trunc(x)): rows s Fb .. s Fb +
//     N - 1 = the pooled rows of sample s, rows 128 .. 128 + SPT - 1 = the
//     tile's e0 rows (one box, so every box starts on a 1024-byte boundary);
//   A (tensor memory, written by the converters): lane s Fb + i - 1 = pooled
//     row i, lane s Fb + N = e0 of sample s, as [t | 2 lo] along K with
//     lo = x - t exactly (the MMA reads 2 lo truncated to TF32), so
//     D = t t'^T + 2 lo t'^T.
// For two vectors u, v of a sample with lanes a, b and B rows a', b',
// (D[a][b'] + D[b][a']) / 2 = t_u.t_v + lo_u.t_v + t_u.lo_v: the product to
// about 2^-20 of |u||v| (lo.lo', below 2^-20, is dropped).  e0's B row is
// 128 + s.  The epilogue gathers each lane's sample block (its e0 column from
// D[.][128 + s]) into shared memory and writes the pairs, averaged over both
// orders, as one contiguous row per sample.
//
// Roles (14 warps): 0..3 epilogue, 4..7 and 8..11 two groups of converters
// taking alternate chunks (raw rows -> A in tensor memory, and the copies of
// e0 / the pooled rows into y), 12 the bulk-copy issuer, 13 tensor-memory
// allocation and MMA issue.  No thread writes shared memory that the tensor
// core reads, so no proxy fence is needed.

namespace {

constexpr int kFwdConvWarp0 = 4, kFwdConvGroups = 2, kFwdTmaWarp = 12, kFwdMmaWarp = 13;
constexpr int kFwdThreads = 448;
constexpr int kFwdRows = 144;                  // B rows per slot (and N of the MMA)
constexpr int kFwdSlotBytes = kFwdRows * 128;  // 18 KB, a multiple of 1024
constexpr uint32_t kFwdDCol1 = 160;            // accumulators at columns 0 and 160 (144 wide)
constexpr uint32_t kFwdACol = 320;             // A slots at 320 + 64 a: t at +0, 2 lo at +32
constexpr int kFwdAS = 3;

}  // namespace

__global__ void __launch_bounds__(kFwdThreads, 1)
interact_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_emb, const __grid_constant__ CUtensorMap map_e0,
                       int N, int d, int64_t B, int mode, float *__restrict__ y, int64_t ys, int fb_log2, int NS)
{
    constexpr int kTmemCols = 512;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ int aborted_s;
    __shared__ __align__(8) uint64_t drain_bar;
    volatile int *aborted = &aborted_s;

    const int inc = mode & kInteractSelf;
    const bool along = (mode & kInteractAlongside) != 0;
    const int F = N + 1;
    const int Fb = 1 << fb_log2, SPT = 128 >> fb_log2;  // rows per sample block, samples per tile
    const int SR = Fb + 1;                               // row stride of the staged blocks
    const int64_t poff = along ? (int64_t)F * d : d;     // first pair column of y
    const int P = (int)num_pairs_of(F, inc);
    const int64_t ntiles = (B + SPT - 1) / SPT;
    const int nch = (d + 31) / 32;

    unsigned char *ring = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);  // [NS] B slots
    float *gram = reinterpret_cast<float *>(ring + (size_t)NS * kFwdSlotBytes);           // [128][SR]
    uint16_t *ptab = reinterpret_cast<uint16_t *>(gram + 128 * SR);  // pair -> block positions pi << 8 | pj
    uint64_t *full = reinterpret_cast<uint64_t *>(ptab + ((P + 3) & ~3));  // [NS] bulk copies landed
    uint64_t *empty = full + NS;                                           // [NS] MMAs done with the slot
    uint64_t *afull = empty + NS;                                          // [kFwdAS] A written
    uint64_t *tfull = afull + kFwdAS;                                      // [2]
    uint64_t *tempty = tfull + 2;                                          // [2]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int p = tid; p < P; p += blockDim.x) {
        // pair p = (i, j): row i starts at i(i-1)/2 (strict pairs) or i(i+1)/2 (self pairs);
        // vector i sits at block position i - 1, e0 (i = 0) at N
        const float rt = sqrtf(8.f * (float)p + 1.f);
        int i = inc ? (int)((rt - 1.f) * 0.5f) : (int)((rt + 1.f) * 0.5f);
        while (pair_pos(i + 1, 0, inc) <= p)
            i++;
        while (pair_pos(i, 0, inc) > p)
            i--;
        const int j = p - (int)pair_pos(i, 0, inc);
        const int pi = i == 0 ? N : i - 1, pj = j == 0 ? N : j - 1;
        ptab[p] = (uint16_t)((pi << 8) | pj);
    }
    if (tid == 0) {
        for (int s = 0; s < NS; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < kFwdAS; s++)
            tc::mbar_init(&afull[s], 128);
        for (int b = 0; b < 2; b++) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 128);
        }
        tc::mbar_init(&drain_bar, 1);
        aborted_s = 0;
        tc::mbar_init_fence();
    }
    if (warp == kFwdMmaWarp)
        tc::tmem_alloc<kTmemCols>(&tmem_slot);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;

    if (warp == kFwdTmaWarp) {
        // ---- bulk copies of the chunks into the B slots (one lane)
        if (lane == 0) {
            uint32_t it = 0;
            bool stop = false;
            for (int64_t t = blockIdx.x; t < ntiles && !stop; t += gridDim.x) {
                const int nS = (int)(B - t * SPT < SPT ? B - t * SPT : SPT);
                const uint32_t bytes = (uint32_t)(nS * N + SPT) * 128u;
                for (int c = 0; c < nch; c++, it++) {
                    const uint32_t slot = it % (uint32_t)NS, u = it / (uint32_t)NS;
                    if (u > 0 && !tc::mbar_wait(&empty[slot], (u - 1) & 1, aborted)) {
                        stop = true;
                        break;
                    }
                    unsigned char *dst = ring + (size_t)slot * kFwdSlotBytes;
                    tc::mbar_expect_tx(&full[slot], bytes);
                    for (int s = 0; s < nS; s++)
                        tc::tma_load_3d(dst + (size_t)s * Fb * 128, &map_emb, c * 32, 0, (int)(t * SPT + s), &full[slot]);
                    tc::tma_load_2d(dst + 128 * 128, &map_e0, c * 32, (int)(t * SPT), &full[slot]);
                }
            }
            if (*aborted) {
                // copies in flight target this CTA's shared memory: wait for them before leaving
                for (uint32_t i = it > (uint32_t)NS ? it - NS : 0; i < it; i++)
                    for (int k = 0; k < tc::kSpinLimit && !tc::mbar_try_wait(&full[i % NS], (i / NS) & 1); k++) {
                    }
            }
        }
        __syncwarp();
    } else if (warp >= kFwdConvWarp0 && warp < kFwdConvWarp0 + 4 * kFwdConvGroups) {
        // ---- converters: group g = chunks it with it % 2 == g; thread a of a group writes A lane a
        // (its warp's lane quarter is a / 32)
        const int g = (tid - kFwdConvWarp0 * 32) >> 7;
        const int a = (tid - kFwdConvWarp0 * 32) & 127;
        const int s = a >> fb_log2, x = a & (Fb - 1);
        const int sr = x < N ? a : (x == N ? 128 + s : -1);  // source row in the slot
        const int f = x == N ? 0 : x + 1;                     // the vector's index in the sample
        const bool vec_y = (reinterpret_cast<uintptr_t>(y) & 15) == 0 && (ys & 3) == 0;
        const uint32_t lane_base = (uint32_t)(warp & 3) * 32 << 16;
        uint32_t it = 0;
        bool stop = false;
        for (int64_t t = blockIdx.x; t < ntiles && !stop; t += gridDim.x) {
            const int64_t b = t * SPT + s;
            const bool valid = sr >= 0 && b < B;
            for (int c = 0; c < nch; c++, it++) {
                if ((int)(it & 1) != g)
                    continue;
                const uint32_t slot = it % (uint32_t)NS, u = it / (uint32_t)NS;
                const uint32_t as = it % kFwdAS, av = it / kFwdAS;
                if (!tc::mbar_wait(&full[slot], u & 1, aborted)) {
                    stop = true;
                    break;
                }
                float v[32];
                if (valid) {
                    const unsigned char *row = ring + (size_t)slot * kFwdSlotBytes + (size_t)sr * 128;
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        const float4 w = *reinterpret_cast<const float4 *>(row + ((q ^ (sr & 7)) << 4));
                        v[4 * q] = w.x;
                        v[4 * q + 1] = w.y;
                        v[4 * q + 2] = w.z;
                        v[4 * q + 3] = w.w;
                    }
                    if (f == 0 || along) {  // e0 (and the pooled rows alongside) into y
                        float *dst = y + b * ys + (int64_t)f * d + c * 32;
#pragma unroll
                        for (int q = 0; q < 8; q++) {
                            if (c * 32 + 4 * q < d) {
                                if (vec_y) {
                                    __stcs(reinterpret_cast<float4 *>(dst + 4 * q),
                                           make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
                                } else {
                                    dst[4 * q] = v[4 * q];
                                    dst[4 * q + 1] = v[4 * q + 1];
                                    dst[4 * q + 2] = v[4 * q + 2];
                                    dst[4 * q + 3] = v[4 * q + 3];
                                }
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 32; k++)
                        v[k] = 0.f;
                }
                float tv[32], lv[32];
#pragma unroll
                for (int k = 0; k < 32; k++) {
                    tv[k] = tc::tf32_trunc(v[k]);
                    lv[k] = 2.f * (v[k] - tv[k]);  // exact; the MMA reads it truncated to TF32
                }
                // A slot `as` is free once the MMAs of item it - kFwdAS are done, which the B slot
                // of that item signals (NS > kFwdAS, so that phase cannot have been passed)
                if (av > 0) {
                    const uint32_t j = it - kFwdAS;
                    if (!tc::mbar_wait(&empty[j % (uint32_t)NS], (j / (uint32_t)NS) & 1, aborted)) {
                        stop = true;
                        break;
                    }
                }
                tc::fence_after_sync();
                const uint32_t ta = tmem + lane_base + kFwdACol + 64 * as;
                tc::tmem_st32(ta, tv);
                tc::tmem_st32(ta + 32, lv);
                tc::tmem_st_wait();
                tc::fence_before_sync();
                tc::mbar_arrive(&afull[as]);
            }
        }
    } else if (warp == kFwdMmaWarp) {
        // ---- MMA issue (one lane)
        if (lane == 0) {
            constexpr uint32_t idesc = tc::tf32_idesc(128, kFwdRows);
            uint32_t it = 0, lt = 0;
            bool issued = false;
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, lt++) {
                const uint32_t buf = lt & 1, v = lt >> 1;
                if (v > 0 && !tc::mbar_wait(&tempty[buf], (v - 1) & 1, aborted))
                    break;
                tc::fence_after_sync();
                const uint32_t dt = tmem + (buf ? kFwdDCol1 : 0u);
                bool ok = true;
                for (int c = 0; c < nch; c++, it++) {
                    const uint32_t slot = it % (uint32_t)NS;
                    const uint32_t as = it % kFwdAS, av = it / kFwdAS;
                    // the converters arrive on afull only after they have seen the chunk's bulk
                    // copies land (full), so afull orders the B slot too
                    if (!tc::mbar_wait(&afull[as], av & 1, aborted)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t bs = tc::smem_u32(ring + (size_t)slot * kFwdSlotBytes);
                    const uint32_t ta = tmem + kFwdACol + 64 * as;
                    const int ksteps = min(4, (d - 32 * c + 7) / 8);
                    for (int kk = 0; kk < ksteps; kk++) {
                        const uint64_t bd = tc::sw128_desc(bs + 32u * kk);
                        tc::mma_tf32_ta(dt, ta + 8 * kk, bd, idesc, c > 0 || kk > 0);
                        tc::mma_tf32_ta(dt, ta + 32 + 8 * kk, bd, idesc, true);
                    }
                    issued = true;
                    tc::mma_commit(&empty[slot]);  // frees the B slot and, kFwdAS items on, the A slot
                }
                if (!ok)
                    break;
                tc::mma_commit(&tfull[buf]);
            }
            if (issued)
                drain_mmas(&drain_bar);
        }
        __syncwarp();
    } else {
        // ---- epilogue: tile row r = tensor-memory lane r
        const int r = tid;
        const int sb = r >> fb_log2;  // sample of the row within the tile
        uint32_t lt = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, lt++) {
            const uint32_t buf = lt & 1;
            const bool ok = tc::mbar_wait(&tfull[buf], (lt >> 1) & 1, aborted);
            if (!all_of(ok, kEpiBarrier, kEpiThreads))
                break;
            tc::fence_after_sync();
            const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + (buf ? kFwdDCol1 : 0u);
            float *row = gram + (size_t)r * SR;
            for (int cb = 0; cb < Fb / 32; cb++) {
                float v[32];
                tc::tmem_ld32(ta + (uint32_t)(sb * Fb + 32 * cb), v);
#pragma unroll
                for (int k = 0; k < 32; k++)
                    row[32 * cb + k] = v[k];
            }
            row[N] = tc::tmem_ld1(ta + 128 + (uint32_t)sb);  // the e0 column of the sample
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[buf]);
            tc::named_sync(kEpiBarrier, kEpiThreads);
            for (int s = 0; s < SPT; s++) {
                const int64_t b = t * SPT + s;
                if (b >= B)
                    break;
                const float *blk = gram + (size_t)s * Fb * SR;
                float *yo = y + b * ys + poff;
                for (int p = r; p < P; p += kEpiThreads) {
                    const int ij = ptab[p], pi = ij >> 8, pj = ij & 255;
                    __stcs(yo + p, 0.5f * (blk[pi * SR + pj] + blk[pj * SR + pi]));
                }
            }
            tc::named_sync(kEpiBarrier, kEpiThreads);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kFwdMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_free<kTmemCols>(tmem);
    }
    if (*aborted) {
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x)
            for (int s = 0; s < SPT && t * SPT + s < B; s++)
                for (int p = tid; p < P; p += blockDim.x)
                    y[(t * SPT + s) * ys + poff + p] = __int_as_float(0x7fc00000);
    }
}

// ---------------------------------------------------------------- backward
//
// One unit = one sample and one tile of up to 128 columns of d.  The MMA
// computes dZ transposed, M = 128, N = Np (F rounded up to 16), K = 8 per
// instruction:
//   D (tensor memory, lane m = column m of the tile) = Z^T . Gs,
//   A = Z^T in tensor memory (lane m holds z_k[m], k = 0 .. F-1, e0 first),
//   B = Gs = G + G^T in shared memory (row n holds Gs[n][k]; a self pair
//     counts twice),
// split hi + lo on both sides (hi = x truncated to TF32, lo = x - hi exactly,
// which the MMA reads truncated in turn: what the three MMAs per K step,
// hi.hi + lo.hi + hi.lo, leave out stays below 3 * 2^-20 of |z||g|).  F <= 32: one K tile.  Bulk tensor copies bring the unit's raw rows
// of Z (unswizzled, one row per vector), 4-byte asynchronous copies its pair
// gradients (a row of dy need not be 16-byte aligned); the converters write A
// into tensor memory (no shared-memory write) and Gs into shared memory
// (published to the tensor core by a proxy fence).
// Four 32-column accumulators drained by two epilogue groups (warps 0..3 and
// 4..7, alternate units: the writes of dZ, row i as 32 consecutive floats per
// warp, are the slow part); each loads the e0 part of dy (and the alongside
// parts) of its next unit ahead.  One converter group (warps 8..11).

namespace {

constexpr int kBwdEpiGroups = 2, kBwdConvWarp0 = 8, kBwdTmaWarp = 12, kBwdMmaWarp = 13;
constexpr int kBwdThreads = 448;
constexpr int kBwdAcc = 4;                 // accumulators of 32 columns at 0, 32, 64, 96
constexpr int kBwdAS = 4;                  // operand slots: A at 128 + 64 a (hi +0, lo +32), B in shared memory
constexpr uint32_t kBwdACol = 128;

}  // namespace

__global__ void __launch_bounds__(kBwdThreads, 1)
interact_bwd_tc_kernel(const __grid_constant__ CUtensorMap map_emb, const __grid_constant__ CUtensorMap map_e0, int N,
                       int d, int64_t B, int mode, const float *__restrict__ dy, int64_t dys,
                       float *__restrict__ de0, int64_t de0s, float *__restrict__ demb, int64_t dembs, int Np, int bx,
                       int NS)
{
    constexpr int kTmemCols = 512;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ int aborted_s;
    __shared__ __align__(8) uint64_t drain_bar;
    volatile int *aborted = &aborted_s;

    const int inc = mode & kInteractSelf;
    const bool along = (mode & kInteractAlongside) != 0;
    const int F = N + 1;
    const int P = (int)num_pairs_of(F, inc);
    const int nd = (d + 127) / 128;                  // d tiles
    const int64_t nunits = B * nd;
    const int ksteps = (F + 7) / 8;
    // raw slot: N pooled rows of bx floats, e0, the pair gradients (128-byte aligned parts)
    const uint32_t rs = (uint32_t)bx * 4u;
    const uint32_t e0off = ((uint32_t)N * rs + 127u) & ~127u;
    const uint32_t dyoff = (e0off + rs + 127u) & ~127u;
    const uint32_t slot_bytes = (dyoff + (uint32_t)P * 4u + 1023u) & ~1023u;
    const uint32_t bbytes = (uint32_t)Np * 128u;  // one B half (hi or lo)

    unsigned char *ring = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);  // [NS] raw slots
    unsigned char *bring = ring + (size_t)NS * slot_bytes;                                 // [kBwdAS] B hi, B lo
    uint64_t *full = reinterpret_cast<uint64_t *>(bring + (size_t)kBwdAS * 2 * bbytes);     // [NS]
    uint64_t *empty = full + NS;                                                           // [NS]
    uint64_t *afull = empty + NS;                                                          // [kBwdAS]
    uint64_t *aempty = afull + kBwdAS;                                                     // [kBwdAS]
    uint64_t *tfull = aempty + kBwdAS;                                                     // [kBwdAcc]
    uint64_t *tempty = tfull + kBwdAcc;                                                    // [kBwdAcc]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < NS; s++) {
            tc::mbar_init(&full[s], 1 + 32);  // the bulk copies' expect_tx, one copy arrival per lane
            tc::mbar_init(&empty[s], 128);
        }
        for (int s = 0; s < kBwdAS; s++) {
            tc::mbar_init(&afull[s], 128);
            tc::mbar_init(&aempty[s], 1);
        }
        for (int b = 0; b < kBwdAcc; b++) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 128);
        }
        tc::mbar_init(&drain_bar, 1);
        aborted_s = 0;
        tc::mbar_init_fence();
    }
    if (warp == kBwdMmaWarp)
        tc::tmem_alloc<kTmemCols>(&tmem_slot);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    const int64_t poff = along ? (int64_t)F * d : d;  // first pair column of dy

    if (warp == kBwdTmaWarp) {
        // ---- copies of the units' raw rows: bulk tensor copies of Z (lane 0), 4-byte asynchronous
        // copies of the pair gradients (all lanes), all completing on the slot's mbarrier
        const uint32_t bytes = (uint32_t)(N + 1) * rs;
        uint32_t it = 0;
        for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x, it++) {
            const uint32_t slot = it % (uint32_t)NS, ph = it / (uint32_t)NS;
            if (ph > 0 && !tc::mbar_wait(&empty[slot], (ph - 1) & 1, aborted))
                break;
            const int64_t b = u / nd;
            const int x = (int)(u - b * nd) * 128;
            unsigned char *dst = ring + (size_t)slot * slot_bytes;
            if (lane == 0) {
                tc::mbar_expect_tx(&full[slot], bytes);
                tc::tma_load_3d(dst, &map_emb, x, 0, (int)b, &full[slot]);
                tc::tma_load_2d(dst + e0off, &map_e0, x, (int)b, &full[slot]);
            }
            const float *src = dy + b * dys + poff;
            for (int p = lane; p < P; p += 32)
                tc::cp_async4(dst + dyoff + p * 4, src + p, true);
            tc::cp_async_arrive(&full[slot]);
        }
        tc::cp_async_wait_all();
        if (*aborted && lane == 0)
            for (uint32_t i = it > (uint32_t)NS ? it - NS : 0; i < it; i++)
                for (int k = 0; k < tc::kSpinLimit && !tc::mbar_try_wait(&full[i % NS], (i / NS) & 1); k++) {
                }
        __syncwarp();
    } else if (warp >= kBwdConvWarp0 && warp < kBwdTmaWarp) {
        // ---- converters: thread a writes A lane a and the Gs entries (n = a / 4, k = 8 (a % 4) .. + 7)
        const int a = tid - kBwdConvWarp0 * 32;
        const uint32_t lane_base = (uint32_t)(warp & 3) * 32 << 16;
        const int n = a >> 2, k0 = 8 * (a & 3);
        int gidx[8];  // pair position of each Gs entry (-1: zero), and whether it is a self pair
        bool gself[8];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int k = k0 + e;
            gself[e] = n == k;
            gidx[e] = (n < F && k < F && (n != k || inc)) ? (int)(n > k ? pair_pos(n, k, inc) : pair_pos(k, n, inc))
                                                           : -1;
        }
        uint32_t it = 0;
        for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x, it++) {
            const uint32_t slot = it % (uint32_t)NS, ph = it / (uint32_t)NS;
            const uint32_t as = it % kBwdAS, av = it / kBwdAS;
            if (!tc::mbar_wait(&full[slot], ph & 1, aborted))
                break;
            const unsigned char *raw = ring + (size_t)slot * slot_bytes;
            float zh[32], zl[32], gh[8], gl[8];
#pragma unroll
            for (int k = 0; k < 32; k++) {
                float z = 0.f;
                if (k < F && a < bx)
                    z = *reinterpret_cast<const float *>(raw + (k == 0 ? e0off : (uint32_t)(k - 1) * rs) + a * 4);
                zh[k] = tc::tf32_trunc(z);
                zl[k] = z - zh[k];  // exact; the MMA reads it truncated to TF32
            }
            const float *dyp = reinterpret_cast<const float *>(raw + dyoff);
#pragma unroll
            for (int e = 0; e < 8; e++) {
                float v = gidx[e] >= 0 ? dyp[gidx[e]] : 0.f;
                if (gself[e])
                    v *= 2.f;  // a self pair counts in G and in G^T
                gh[e] = tc::tf32_trunc(v);
                gl[e] = v - gh[e];
            }
            tc::mbar_arrive(&empty[slot]);  // the raw slot has been read
            if (av > 0 && !tc::mbar_wait(&aempty[as], (av - 1) & 1, aborted))
                break;
            tc::fence_after_sync();
            if (n < Np) {
                unsigned char *bh = bring + (size_t)as * 2 * bbytes;
                const int q0 = 2 * (a & 3);
                *reinterpret_cast<float4 *>(bh + sw128(n, q0)) = make_float4(gh[0], gh[1], gh[2], gh[3]);
                *reinterpret_cast<float4 *>(bh + sw128(n, q0 + 1)) = make_float4(gh[4], gh[5], gh[6], gh[7]);
                *reinterpret_cast<float4 *>(bh + bbytes + sw128(n, q0)) = make_float4(gl[0], gl[1], gl[2], gl[3]);
                *reinterpret_cast<float4 *>(bh + bbytes + sw128(n, q0 + 1)) = make_float4(gl[4], gl[5], gl[6], gl[7]);
            }
            const uint32_t ta = tmem + lane_base + kBwdACol + 64 * as;
            tc::tmem_st32(ta, zh);
            tc::tmem_st32(ta + 32, zl);
            tc::fence_async_smem();
            tc::tmem_st_wait();
            tc::fence_before_sync();
            tc::mbar_arrive(&afull[as]);
        }
    } else if (warp == kBwdMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc = tc::tf32_idesc(128, Np);
            uint32_t it = 0;
            bool issued = false;
            for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x, it++) {
                const uint32_t buf = it % kBwdAcc, v = it / kBwdAcc;
                const uint32_t as = it % kBwdAS, av = it / kBwdAS;
                if (v > 0 && !tc::mbar_wait(&tempty[buf], (v - 1) & 1, aborted))
                    break;
                if (!tc::mbar_wait(&afull[as], av & 1, aborted))
                    break;
                tc::fence_after_sync();
                const uint32_t dt = tmem + buf * 32;
                const uint32_t ta = tmem + kBwdACol + 64 * as;
                const uint32_t bh = tc::smem_u32(bring + (size_t)as * 2 * bbytes), bl = bh + bbytes;
                for (int kk = 0; kk < ksteps; kk++) {
                    const uint64_t bhd = tc::sw128_desc(bh + 32u * kk), bld = tc::sw128_desc(bl + 32u * kk);
                    tc::mma_tf32_ta(dt, ta + 8 * kk, bhd, idesc, kk > 0);
                    tc::mma_tf32_ta(dt, ta + 32 + 8 * kk, bhd, idesc, true);
                    tc::mma_tf32_ta(dt, ta + 8 * kk, bld, idesc, true);
                }
                issued = true;
                tc::mma_commit(&aempty[as]);
                tc::mma_commit(&tfull[buf]);
            }
            if (issued)
                drain_mmas(&drain_bar);
        }
        __syncwarp();
    } else {
        // ---- epilogue: group g (warps 4g .. 4g + 3) takes units it with it % 2 == g; lane m of the
        // accumulator = column m of the unit's d tile.  The dy parts of the group's next unit are
        // loaded while this one is waited for and written.
        const int g = warp >> 2, et = tid & 127;
        float g0n = 0.f, gan[32];
        auto load_dy = [&](int64_t u) {
            const int64_t b = u / nd;
            const int m = (int)(u - b * nd) * 128 + et;
            const bool act = u < nunits && m < d;
            const float *dyb = dy + b * dys;
            g0n = act ? __ldg(dyb + m) : 0.f;
#pragma unroll
            for (int i = 1; i < 32; i++)
                gan[i] = (along && act && i < F) ? __ldg(dyb + (int64_t)i * d + m) : 0.f;
        };
        load_dy(blockIdx.x + (int64_t)g * gridDim.x);
        uint32_t it = g;
        for (int64_t u = blockIdx.x + (int64_t)g * gridDim.x; u < nunits;
             u += kBwdEpiGroups * (int64_t)gridDim.x, it += kBwdEpiGroups) {
            const int64_t b = u / nd;
            const int m = (int)(u - b * nd) * 128 + et;
            const bool act = m < d;
            float ga[32];
            const float g0 = g0n;
#pragma unroll
            for (int i = 1; i < 32; i++)
                ga[i] = gan[i];
            load_dy(u + kBwdEpiGroups * (int64_t)gridDim.x);
            const uint32_t buf = it % kBwdAcc;
            const bool ok = tc::mbar_wait(&tfull[buf], (it / kBwdAcc) & 1, aborted);
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc::fence_after_sync();
            float v[32];
            tc::tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + buf * 32, v);
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[buf]);
            if (act) {
                __stcs(de0 + b * de0s + m, v[0] + g0);
                float *dz = demb + b * dembs + m;
#pragma unroll
                for (int i = 1; i < 32; i++)
                    if (i < F)
                        __stcs(dz + (int64_t)(i - 1) * d, v[i] + ga[i]);
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kBwdMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_free<kTmemCols>(tmem);
    }
    if (*aborted) {
        const float nan = __int_as_float(0x7fc00000);
        for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
            const int64_t b = u / nd;
            const int m0 = (int)(u - b * nd) * 128;
            for (int m = m0 + tid; m < d && m < m0 + 128; m += blockDim.x) {
                de0[b * de0s + m] = nan;
                for (int i = 1; i < F; i++)
                    demb[b * dembs + (int64_t)(i - 1) * d + m] = nan;
            }
        }
    }
}

// ------------------------------------------------- backward, 33 to 128 vectors
//
// One unit = one sample and one tile of up to 128 columns of d.  The MMA
// computes dZ transposed, M = 128, N = Np (F rounded up to 16), K = 8 per
// instruction:
//   D (tensor memory, lane m = column m of the tile) = Z^T . Gs,
//   A = Z^T in tensor memory (lane m holds z_k[m], k = 0 .. F-1, e0 first),
//   B = Gs = G + G^T in shared memory (row n holds Gs[n][k]; a self pair
//     counts twice),
// split hi + lo on both sides (hi = x truncated to TF32, lo = x - hi exactly,
// which the MMA reads truncated in turn: what the three MMAs per K step,
// hi.hi + lo.hi + hi.lo, leave out stays below 3 * 2^-20 of |z||g|).  K runs in chunks of 32 vectors: a bulk tensor copy brings the
// chunk's 32 raw rows of Z (unswizzled; the box starts one row before the
// chunk, so for the first chunk its row 0 reads as zero and e0 comes in a row
// of its own), 4-byte asynchronous copies bring the unit's pair gradients
// once (a row of dy need not be 16-byte aligned).  The converters write the
// chunk's A into tensor memory (no shared-memory write) and its columns of Gs
// into shared memory (published to the tensor core by a proxy fence).  Gs
// depends on the sample only: a CTA takes the d tiles of each of its samples
// one after the other and builds the sample's Gs once, into one shared-memory
// slot per chunk that the MMAs of all its tiles read.
// Accumulators of Np rounded up to 32 columns fill tensor-memory columns
// 0 .. 255 (8, 4 or 2 of them), drained by two epilogue groups (warps 0..3
// and 4..7, alternate units: the writes of dZ, row i as 32 consecutive floats
// per warp, are the slow part); each loads the e0 part of dy of its next unit
// ahead.  Two converter groups (warps 8..11 and 12..15) take the chunks in
// turn; with an odd number of raw slots a slot's fills alternate between them,
// so a group waits for the slot's previous fill to be released before it waits
// for its own (a parity wait cannot tell a fill from the one two phases on).
// The tensor pipe bounds the kernel: 3 x ceil(F / 8) MMAs per unit of about
// 160 to 200 cycles each (M = 128, N = 112, K = 8, A in tensor memory).
// (For F <= 32 the one-chunk kernel above is faster: measured 0.50 vs 0.83 ms
// on the multi-hot shape.)

namespace {

constexpr int kBwcEpiGroups = 2, kBwcConvGroups = 2, kBwcConvWarp0 = 8, kBwcTmaWarp = 16, kBwcMmaWarp = 17;
constexpr int kBwcThreads = 576;
constexpr uint32_t kBwcACol = 256;  // A chunk slots at 256 + 64 a (hi at +0, lo at +32); accumulators below
constexpr int kBwcMaxAS = 4;
constexpr int kBwcMaxDS = 8;        // pair-gradient slots (units)
constexpr int kBwcMaxAcc = 8;       // accumulators of W = Np rounded up to 32 columns in columns 0 .. 255
constexpr int kBwcMaxChunks = 4;    // K chunks of 32 vectors (F <= 128): one Gs slot each
// each A slot belongs to one converter group (slot ic % AS, group ic % 2), which takes its uses in order
static_assert(kBwcMaxAS % kBwcConvGroups == 0, "A slots must not alternate between converter groups");

}  // namespace

__global__ void __launch_bounds__(kBwcThreads, 1)
interact_bwd_tc_chunked_kernel(const __grid_constant__ CUtensorMap map_emb,
                               const __grid_constant__ CUtensorMap map_e0, int N, int d, int64_t B, int mode,
                               const float *__restrict__ dy, int64_t dys, float *__restrict__ de0, int64_t de0s,
                               float *__restrict__ demb, int64_t dembs, int Np, int bx, int NR, int AS, int DS)
{
    constexpr int kTmemCols = 512;
    extern __shared__ unsigned char smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ int aborted_s;
    __shared__ __align__(8) uint64_t drain_bar;
    volatile int *aborted = &aborted_s;

    const int inc = mode & kInteractSelf;
    const bool along = (mode & kInteractAlongside) != 0;
    const int F = N + 1;
    const int P = (int)num_pairs_of(F, inc);
    const int nd = (d + 127) / 128;  // d tiles
    const int nkc = (F + 31) / 32;   // K chunks of 32 vectors
    const int64_t poff = along ? (int64_t)F * d : d;  // first pair column of dy
    const uint32_t rs = (uint32_t)bx * 4u;             // bytes of a raw row
    const uint32_t zslot = (33u * rs + 1023u) & ~1023u;           // 32 chunk rows, then e0
    const uint32_t dslot = ((uint32_t)P * 4u + 127u) & ~127u;     // the unit's pair gradients
    const uint32_t bbytes = (uint32_t)Np * 128u;                  // one B half (hi or lo)
    const uint32_t W = ((uint32_t)Np + 31u) & ~31u;               // accumulator width
    const uint32_t nacc = 256u / W;                               // accumulators: 8, 4 or 2

    unsigned char *zring = smem_raw + ((1024 - (tc::smem_u32(smem_raw) & 1023)) & 1023);  // [NR]
    unsigned char *bring = zring + (size_t)NR * zslot;                                     // [nkc] B hi, B lo
    unsigned char *dring = bring + (size_t)nkc * 2 * bbytes;                               // [DS]
    uint64_t *zfull = reinterpret_cast<uint64_t *>(dring + (size_t)DS * dslot);             // [NR]
    uint64_t *zempty = zfull + NR;                                                         // [NR]
    uint64_t *dfull = zempty + NR;                                                         // [DS]
    uint64_t *dempty = dfull + DS;                                                         // [DS]
    uint64_t *afull = dempty + DS;                                                         // [AS]
    uint64_t *aempty = afull + AS;                                                         // [AS]
    uint64_t *tfull = aempty + AS;                                                         // [nacc]
    uint64_t *tempty = tfull + kBwcMaxAcc;                                                 // [nacc]
    uint64_t *bfull = tempty + kBwcMaxAcc;                                                 // [nkc]
    uint64_t *bempty = bfull + kBwcMaxChunks;                                              // [nkc]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < NR; s++) {
            tc::mbar_init(&zfull[s], 1);
            tc::mbar_init(&zempty[s], 128);
        }
        for (int s = 0; s < DS; s++) {
            tc::mbar_init(&dfull[s], 32);  // one copy arrival per lane of the copy warp
            tc::mbar_init(&dempty[s], 128 * kBwcConvGroups);
        }
        for (int s = 0; s < AS; s++) {
            tc::mbar_init(&afull[s], 128);
            tc::mbar_init(&aempty[s], 1);
        }
        for (uint32_t b = 0; b < nacc; b++) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 128);
        }
        for (int c = 0; c < nkc; c++) {
            tc::mbar_init(&bfull[c], 128);
            tc::mbar_init(&bempty[c], 1);
        }
        tc::mbar_init(&drain_bar, 1);
        aborted_s = 0;
        tc::mbar_init_fence();
    }
    // the Gs slots start zero: their padding (rows and columns from F on, and the
    // diagonal for strict pairs) is never written again
    for (uint32_t o = (uint32_t)tid * 16u; o < (uint32_t)nkc * 2u * bbytes; o += kBwcThreads * 16u)
        *reinterpret_cast<float4 *>(bring + o) = make_float4(0.f, 0.f, 0.f, 0.f);
    tc::fence_async_smem();
    if (warp == kBwcMmaWarp)
        tc::tmem_alloc<kTmemCols>(&tmem_slot);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_slot;
    // this CTA's units: its samples b = blockIdx.x + i gridDim.x, the d tiles of each in turn
    const uint32_t nsamp = blockIdx.x < B ? (uint32_t)((B - 1 - blockIdx.x) / gridDim.x + 1) : 0u;
    const uint32_t ncta = nsamp * (uint32_t)nd;
    auto sample_of = [&](uint32_t iu) { return (int64_t)blockIdx.x + (int64_t)(iu / (uint32_t)nd) * gridDim.x; };

    if (warp == kBwcTmaWarp) {
        // ---- copies: per unit the pair gradients (all lanes, 4-byte asynchronous copies), per
        // chunk the raw rows of Z (lane 0, bulk tensor copies)
        uint32_t ic = 0;
        bool stop = false;
        for (uint32_t iu = 0; iu < ncta && !stop; iu++) {
            const int64_t b = sample_of(iu);
            const int tile = (int)(iu % (uint32_t)nd), x = tile * 128;
            const uint32_t ds = iu % (uint32_t)DS, dph = iu / (uint32_t)DS;
            if (dph > 0 && !tc::mbar_wait(&dempty[ds], (dph - 1) & 1, aborted))
                break;
            if (tile == 0) {  // the sample's pair gradients (its other tiles reuse its Gs)
                unsigned char *dd = dring + (size_t)ds * dslot;
                const float *src = dy + b * dys + poff;
                for (int p = lane; p < P; p += 32)
                    tc::cp_async4(dd + p * 4, src + p, true);
            }
            tc::cp_async_arrive(&dfull[ds]);
            for (int c = 0; c < nkc; c++, ic++) {
                const uint32_t zs = ic % (uint32_t)NR, zph = ic / (uint32_t)NR;
                if (zph > 0 && !tc::mbar_wait(&zempty[zs], (zph - 1) & 1, aborted)) {
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    unsigned char *zd = zring + (size_t)zs * zslot;
                    tc::mbar_expect_tx(&zfull[zs], (c == 0 ? 33u : 32u) * rs);
                    // rows 32c - 1 .. 32c + 30 of the pooled block = vectors 32c .. 32c + 31
                    tc::tma_load_3d(zd, &map_emb, x, 32 * c - 1, (int)b, &zfull[zs]);
                    if (c == 0)
                        tc::tma_load_2d(zd + 32 * rs, &map_e0, x, (int)b, &zfull[zs]);
                }
            }
        }
        tc::cp_async_wait_all();
        if (*aborted && lane == 0)
            for (uint32_t i = ic > (uint32_t)NR ? ic - NR : 0; i < ic; i++)
                for (int k = 0; k < tc::kSpinLimit && !tc::mbar_try_wait(&zfull[i % NR], (i / NR) & 1); k++) {
                }
        __syncwarp();
    } else if (warp >= kBwcConvWarp0 && warp < kBwcTmaWarp) {
        // ---- converters, two groups taking the chunks in turn (group cg the chunks ic with
        // ic % 2 == cg, counted over all units): thread a writes A lane a
        const int a = (tid - kBwcConvWarp0 * 32) & 127, cg = (warp - kBwcConvWarp0) >> 2;
        const uint32_t lane_base = (uint32_t)(warp & 3) * 32 << 16;
        uint32_t ic = 0;
        bool stop = false;
        for (uint32_t iu = 0; iu < ncta && !stop; iu++) {
            const int tile = (int)(iu % (uint32_t)nd);
            const uint32_t sc = iu / (uint32_t)nd;  // the sample's index among this CTA's
            const uint32_t ds = iu % (uint32_t)DS, dph = iu / (uint32_t)DS;
            if (!tc::mbar_wait(&dfull[ds], dph & 1, aborted))
                break;
            const float *dyp = reinterpret_cast<const float *>(dring + (size_t)ds * dslot);
            // the last of the unit's chunks that this group takes (each takes one at least: nkc >= 2)
            const int clast = nkc - 1 - (int)(((ic + (uint32_t)nkc - 1u) & 1u) != (uint32_t)cg);
            for (int c = 0; c < nkc; c++, ic++) {
                if ((ic & 1u) != (uint32_t)cg)
                    continue;
                const uint32_t zs = ic % (uint32_t)NR, zph = ic / (uint32_t)NR;
                const uint32_t as = ic % (uint32_t)AS, av = ic / (uint32_t)AS;
                // With an odd number of raw slots, consecutive fills of a slot go to alternate groups: a
                // group must see the slot's previous fill released before it waits for this one, or the
                // parity wait below would take the phase of the fill before (still in flight) for it.
                if ((zph > 0 && !tc::mbar_wait(&zempty[zs], (zph - 1) & 1, aborted)) ||
                    !tc::mbar_wait(&zfull[zs], zph & 1, aborted)) {
                    stop = true;
                    break;
                }
                const unsigned char *raw = zring + (size_t)zs * zslot;
                float zh[32], zl[32];
#pragma unroll
                for (int r = 0; r < 32; r++) {
                    float z = 0.f;
                    if (a < bx && 32 * c + r < F)
                        z = *reinterpret_cast<const float *>(raw + (c == 0 && r == 0 ? 32 * rs : (uint32_t)r * rs) +
                                                             a * 4);
                    zh[r] = tc::tf32_trunc(z);
                    zl[r] = z - zh[r];  // exact; the MMA reads it truncated to TF32
                }
                tc::mbar_arrive(&zempty[zs]);
                if (av > 0 && !tc::mbar_wait(&aempty[as], (av - 1) & 1, aborted)) {
                    stop = true;
                    break;
                }
                if (tile == 0 && sc > 0 && !tc::mbar_wait(&bempty[c], (sc - 1) & 1, aborted)) {
                    stop = true;
                    break;
                }
                tc::fence_after_sync();
                unsigned char *bh = bring + (size_t)c * 2 * bbytes;
                // Gs of rows n < F and the chunk's columns k < F, 4 columns (one 16-byte unit) per
                // item; the rest of the slot stays zero.  Pair (i, j), j <= i, sits at T(i) + j with
                // T(i) = i (i + sh) / 2, so T(i + 1) = T(i) + i + inc.
                const int sh = inc ? 1 : -1;
                const int kc = min(32, F - 32 * c);
                const int lq = kc > 16 ? 3 : (kc > 8 ? 2 : (kc > 4 ? 1 : 0));  // items per row: 1 << lq
                for (int e = a; e < (F << lq) && tile == 0; e += 128) {
                    const int n = e >> lq, k0 = 32 * c + 4 * (e & ((1 << lq) - 1));
                    float v[4];
                    if (n >= k0 + 4) {  // below the diagonal: four consecutive pairs of row n
                        const float *s = dyp + ((n * (n + sh)) >> 1) + k0;
#pragma unroll
                        for (int j = 0; j < 4; j++)
                            v[j] = s[j];
                    } else if (n < k0) {  // above it: entry n of rows k0 .. k0 + 3
                        int t = (k0 * (k0 + sh)) >> 1;
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            v[j] = k0 + j < F ? dyp[t + n] : 0.f;
                            t += k0 + j + inc;
                        }
                    } else {  // the 4 x 4 block on the diagonal
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            const int k = k0 + j, hi = n > k ? n : k, lo = n > k ? k : n;
                            v[j] = (k < F && (n != k || inc)) ? dyp[((hi * (hi + sh)) >> 1) + lo] : 0.f;
                            if (n == k)
                                v[j] *= 2.f;  // a self pair counts in G and in G^T
                        }
                    }
                    float h[4], l[4];
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        h[j] = tc::tf32_trunc(v[j]);
                        l[j] = v[j] - h[j];
                    }
                    const uint32_t o = sw128(n, (k0 & 31) >> 2);
                    *reinterpret_cast<float4 *>(bh + o) = make_float4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<float4 *>(bh + bbytes + o) = make_float4(l[0], l[1], l[2], l[3]);
                }
                const uint32_t ta = tmem + lane_base + kBwcACol + 64 * as;
                tc::tmem_st32(ta, zh);
                tc::tmem_st32(ta + 32, zl);
                if (tile == 0)
                    tc::fence_async_smem();  // the Gs stores, for the tensor core (A is in tensor memory)
                tc::tmem_st_wait();
                tc::fence_before_sync();
                if (tile == 0)
                    tc::mbar_arrive(&bfull[c]);
                tc::mbar_arrive(&afull[as]);
                if (c == clast)
                    tc::mbar_arrive(&dempty[ds]);  // this group has read the unit's pair gradients
            }
        }
    } else if (warp == kBwcMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc = tc::tf32_idesc(128, Np);
            uint32_t ic = 0;
            bool issued = false, ok = true;
            for (uint32_t iu = 0; iu < ncta && ok; iu++) {
                const int tile = (int)(iu % (uint32_t)nd);
                const uint32_t sc = iu / (uint32_t)nd;
                const uint32_t buf = iu % nacc, v = iu / nacc;
                if (v > 0 && !tc::mbar_wait(&tempty[buf], (v - 1) & 1, aborted))
                    break;
                tc::fence_after_sync();
                const uint32_t dt = tmem + buf * W;
                for (int c = 0; c < nkc; c++, ic++) {
                    const uint32_t as = ic % (uint32_t)AS, av = ic / (uint32_t)AS;
                    if (!tc::mbar_wait(&afull[as], av & 1, aborted) ||
                        (tile == 0 && !tc::mbar_wait(&bfull[c], sc & 1, aborted))) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t ta = tmem + kBwcACol + 64 * as;
                    const uint32_t bh = tc::smem_u32(bring + (size_t)c * 2 * bbytes), bl = bh + bbytes;
                    const int ksteps = min(4, (F - 32 * c + 7) / 8);
                    for (int kk = 0; kk < ksteps; kk++) {
                        const uint64_t bhd = tc::sw128_desc(bh + 32u * kk), bld = tc::sw128_desc(bl + 32u * kk);
                        const bool acc = c > 0 || kk > 0;
                        tc::mma_tf32_ta(dt, ta + 8 * kk, bhd, idesc, acc);
                        tc::mma_tf32_ta(dt, ta + 32 + 8 * kk, bhd, idesc, true);
                        tc::mma_tf32_ta(dt, ta + 8 * kk, bld, idesc, true);
                    }
                    issued = true;
                    tc::mma_commit(&aempty[as]);
                    if (tile == nd - 1)
                        tc::mma_commit(&bempty[c]);  // the sample's last tile has read its Gs chunk
                }
                if (!ok)
                    break;
                tc::mma_commit(&tfull[buf]);
            }
            if (issued)
                drain_mmas(&drain_bar);
        }
        __syncwarp();
    } else {
        // ---- epilogue: group g (warps 4g .. 4g + 3) takes units iu with iu % 2 == g; lane m of the
        // accumulator = column m of the unit's d tile
        const int g = warp >> 2, et = tid & 127;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        auto load_g0 = [&](uint32_t iu) -> float {
            const int64_t b = sample_of(iu);
            const int m = (int)(iu % (uint32_t)nd) * 128 + et;
            return (iu < ncta && m < d) ? __ldg(dy + b * dys + m) : 0.f;
        };
        float g0n = load_g0((uint32_t)g);
        for (uint32_t iu = (uint32_t)g; iu < ncta; iu += kBwcEpiGroups) {
            const int64_t b = sample_of(iu);
            const int m = (int)(iu % (uint32_t)nd) * 128 + et;
            const bool act = m < d;
            const float g0 = g0n;
            g0n = load_g0(iu + kBwcEpiGroups);
            const uint32_t buf = iu % nacc;
            const bool okw = tc::mbar_wait(&tfull[buf], (iu / nacc) & 1, aborted);
            if (!__all_sync(0xffffffffu, okw))
                break;
            tc::fence_after_sync();
            const uint32_t ta = tmem + lane_base + buf * W;
            const float *dyb = dy + b * dys;
            for (int c = 0; c < nkc; c++) {
                float ga[32];
#pragma unroll
                for (int r = 0; r < 32; r++) {
                    const int i = 32 * c + r;
                    ga[r] = (along && act && i > 0 && i < F) ? __ldg(dyb + (int64_t)i * d + m) : 0.f;
                }
                float v[32];
                tc::tmem_ld32(ta + 32 * c, v);
                if (act) {
#pragma unroll
                    for (int r = 0; r < 32; r++) {
                        const int i = 32 * c + r;
                        if (i == 0)
                            __stcs(de0 + b * de0s + m, v[0] + g0);
                        else if (i < F)
                            __stcs(demb + b * dembs + (int64_t)(i - 1) * d + m, v[r] + ga[r]);
                    }
                }
            }
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[buf]);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kBwcMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_free<kTmemCols>(tmem);
    }
    if (*aborted) {
        const float nan = __int_as_float(0x7fc00000);
        for (uint32_t iu = 0; iu < ncta; iu++) {
            const int64_t b = sample_of(iu);
            const int m0 = (int)(iu % (uint32_t)nd) * 128;
            for (int m = m0 + tid; m < d && m < m0 + 128; m += blockDim.x) {
                de0[b * de0s + m] = nan;
                for (int i = 1; i < F; i++)
                    demb[b * dembs + (int64_t)(i - 1) * d + m] = nan;
            }
        }
    }
}

// ------------------------------------------------------------------ launch
//
// Both return 1 (not launched) when the operands do not suit the kernels:
// rows not of whole 16-byte chunks, unaligned bases or strides, no pooled
// rows, more than 128 vectors per sample, rows
// too short to fill the tiles (d < 32 forward, d < 64 backward), or too few
// units to fill the backward's pipeline.  Otherwise they launch and return
// the status.

static bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

// Whether the tensor-core forward takes these operands (d < 32 leaves most of a
// 32-column chunk empty: the CUDA-core kernels are faster there).
bool interact_fwd_tc_applies(const float *e0, int64_t e0s, const float *emb, int64_t embs, int N, int d, int64_t B)
{
    return interact_tensor_cores() && N >= 1 && N + 1 <= 128 && d >= 32 && d % 4 == 0 && e0s % 4 == 0 &&
           embs % 4 == 0 && aligned16(e0) && aligned16(emb) && B <= 0x7fffffff;
}

int launch_interact_fwd_tc(const float *e0, int64_t e0s, const float *emb, int64_t embs, int N, int d, int64_t B,
                           int mode, float *y, int64_t ys, cudaStream_t st)
{
    const int F = N + 1;
    if (!interact_fwd_tc_applies(e0, e0s, emb, embs, N, d, B))
        return 1;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return 1;
    const int fb_log2 = F <= 32 ? 5 : (F <= 64 ? 6 : 7);
    const int Fb = 1 << fb_log2, SPT = 128 / Fb;
    CUtensorMap map_emb, map_e0;
    std::memset(&map_emb, 0, sizeof map_emb);
    std::memset(&map_e0, 0, sizeof map_e0);
    const cuuint64_t dims3[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides3[2] = {(cuuint64_t)d * 4, (cuuint64_t)embs * 4};
    const cuuint32_t box3[3] = {32, (cuuint32_t)N, 1};
    const cuuint32_t one3[3] = {1, 1, 1};
    if (enc(&map_emb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(emb), dims3, strides3, box3, one3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const cuuint64_t dims2[2] = {(cuuint64_t)d, (cuuint64_t)B};
    const cuuint64_t strides2[1] = {(cuuint64_t)e0s * 4};
    const cuuint32_t box2[2] = {32, (cuuint32_t)SPT};
    const cuuint32_t one2[2] = {1, 1};
    if (enc(&map_e0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(e0), dims2, strides2, box2, one2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const int P = (int)num_pairs_of(F, mode & kInteractSelf);
    const size_t fixed = 1024 + (size_t)128 * (Fb + 1) * 4 + (size_t)((P + 3) & ~3) * 2 + (kFwdAS + 4) * 8;
    int NS = kFwdAS + 1;  // B slots (18 KB): as many as fit, up to 8, more than the A slots
    while (NS < 8 && fixed + (size_t)(NS + 1) * (kFwdSlotBytes + 16) <= kMaxSmem)
        NS++;
    const size_t smem = fixed + (size_t)NS * (kFwdSlotBytes + 16);
    if (smem > kMaxSmem)
        return 1;
    static std::atomic<unsigned long long> smem_set{0};  // devices whose limit has been raised
    if (allow_dynamic_smem(reinterpret_cast<const void *>(interact_fwd_tc_kernel), (int)kMaxSmem, &smem_set) !=
        DLRM_OK)
        return DLRM_ERR_CUDA;
    const int64_t ntiles = (B + SPT - 1) / SPT;
    const int64_t grid = ntiles < sm_count() ? ntiles : sm_count();
    interact_fwd_tc_kernel<<<(unsigned)grid, kFwdThreads, smem, st>>>(map_emb, map_e0, N, d, B, mode, y, ys, fb_log2,
                                                                       NS);
    count_launch(st);
    return launch_status();
}

static int launch_interact_bwd_tc_chunked(const float *e0, int64_t e0s, const float *emb, int64_t embs, int N,
                                          int d, int64_t B, int mode, const float *dy, int64_t dys, float *de0,
                                          int64_t de0s, float *demb, int64_t dembs, cudaStream_t st)
{
    const int F = N + 1;
    const int64_t nunits = B * ((d + 127) / 128);
    // d < 64 leaves most of a 128-lane tile idle, and with fewer than 32 units per SM the
    // pipeline does not fill: the CUDA-core kernel is faster there
    if (N < 1 || F > 128 || d < 64 || nunits < 32 * (int64_t)sm_count() || d % 4 != 0 || e0s % 4 != 0 ||
        embs % 4 != 0 || !aligned16(e0) || !aligned16(emb) || B > 0x7fffffff)
        return 1;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return 1;
    const int P = (int)num_pairs_of(F, mode & kInteractSelf);
    const int Np = (F + 15) & ~15;
    const int bx = d < 128 ? d : 128;  // columns of a d tile
    CUtensorMap map_emb, map_e0;
    std::memset(&map_emb, 0, sizeof map_emb);
    std::memset(&map_e0, 0, sizeof map_e0);
    const cuuint64_t dims3[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides3[2] = {(cuuint64_t)d * 4, (cuuint64_t)embs * 4};
    const cuuint32_t box3[3] = {(cuuint32_t)bx, 32, 1};  // 32 rows, zero-filled past the sample's N
    const cuuint32_t one3[3] = {1, 1, 1};
    const cuuint32_t one2[2] = {1, 1};
    if (enc(&map_emb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(emb), dims3, strides3, box3, one3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const cuuint64_t dims_e0[2] = {(cuuint64_t)d, (cuuint64_t)B};
    const cuuint64_t strides_e0[1] = {(cuuint64_t)e0s * 4};
    const cuuint32_t box_e0[2] = {(cuuint32_t)bx, 1};
    if (enc(&map_e0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(e0), dims_e0, strides_e0, box_e0, one2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const size_t zslot = (33 * (size_t)bx * 4 + 1023) & ~(size_t)1023;
    const size_t dslot = ((size_t)P * 4 + 127) & ~(size_t)127;
    const size_t bslot = 2 * (size_t)Np * 128;
    const int nkc = (F + 31) / 32;  // one Gs slot per K chunk, reused by the sample's d tiles
    const size_t fixed = 1024 + (size_t)kBwcMaxAcc * 16 + (size_t)kBwcMaxChunks * 16 + (size_t)nkc * bslot;
    // A operand slots: 4 (tensor memory); pair-gradient slots and raw chunks: as many as fit, up to 8
    int AS = kBwcMaxAS, NR = 2, DS = 2;
    auto total = [&](int as, int nr, int ds) {
        return fixed + (size_t)as * 16 + (size_t)nr * (zslot + 16) + (size_t)ds * (dslot + 16);
    };
    for (bool grew = true; grew;) {
        grew = false;
        if (NR < 8 && total(AS, NR + 1, DS) <= kMaxSmem) {
            NR++;
            grew = true;
        }
        if (DS < kBwcMaxDS && total(AS, NR, DS + 1) <= kMaxSmem) {
            DS++;
            grew = true;
        }
    }
    const size_t smem = total(AS, NR, DS);
    if (smem > kMaxSmem)
        return 1;
    static std::atomic<unsigned long long> smem_set{0};
    if (allow_dynamic_smem(reinterpret_cast<const void *>(interact_bwd_tc_chunked_kernel), (int)kMaxSmem, &smem_set) !=
        DLRM_OK)
        return DLRM_ERR_CUDA;
    const int64_t grid = nunits < sm_count() ? nunits : sm_count();
    interact_bwd_tc_chunked_kernel<<<(unsigned)grid, kBwcThreads, smem, st>>>(map_emb, map_e0, N, d, B, mode, dy, dys, de0,
                                                                       de0s, demb, dembs, Np, bx, NR, AS, DS);
    count_launch(st);
    return launch_status();
}

int launch_interact_bwd_tc(const float *e0, int64_t e0s, const float *emb, int64_t embs, int N, int d, int64_t B,
                           int mode, const float *dy, int64_t dys, float *de0, int64_t de0s, float *demb,
                           int64_t dembs, cudaStream_t st)
{
    const int F = N + 1;
    if (F > 32)
        return launch_interact_bwd_tc_chunked(e0, e0s, emb, embs, N, d, B, mode, dy, dys, de0, de0s, demb, dembs,
                                              st);
    const int64_t nunits = B * ((d + 127) / 128);
    // d < 64 leaves most of a 128-lane tile idle, and with fewer than 32 units per SM the
    // pipeline does not fill: the CUDA-core kernel is faster there
    if (N < 1 || F > 32 || d < 64 || nunits < 32 * (int64_t)sm_count() || d % 4 != 0 || e0s % 4 != 0 ||
        embs % 4 != 0 || !aligned16(e0) || !aligned16(emb) || B > 0x7fffffff)
        return 1;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return 1;
    const int P = (int)num_pairs_of(F, mode & kInteractSelf);
    const int Np = F <= 16 ? 16 : 32;
    const int bx = d < 128 ? d : 128;  // columns of a d tile
    CUtensorMap map_emb, map_e0;
    std::memset(&map_emb, 0, sizeof map_emb);
    std::memset(&map_e0, 0, sizeof map_e0);
    const cuuint64_t dims3[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides3[2] = {(cuuint64_t)d * 4, (cuuint64_t)embs * 4};
    const cuuint32_t box3[3] = {(cuuint32_t)bx, (cuuint32_t)N, 1};
    const cuuint32_t one3[3] = {1, 1, 1};
    const cuuint32_t one2[2] = {1, 1};
    if (enc(&map_emb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(emb), dims3, strides3, box3, one3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const cuuint64_t dims_e0[2] = {(cuuint64_t)d, (cuuint64_t)B};
    const cuuint64_t strides_e0[1] = {(cuuint64_t)e0s * 4};
    const cuuint32_t box_e0[2] = {(cuuint32_t)bx, 1};
    if (enc(&map_e0, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(e0), dims_e0, strides_e0, box_e0, one2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return 1;
    const size_t rs = (size_t)bx * 4;
    const size_t e0off = ((size_t)N * rs + 127) & ~(size_t)127;
    const size_t dyoff = (e0off + rs + 127) & ~(size_t)127;
    const size_t slot = (dyoff + (size_t)P * 4 + 1023) & ~(size_t)1023;
    const size_t fixed = 1024 + (size_t)kBwdAS * 2 * Np * 128 + (2 * kBwdAS + 2 * kBwdAcc) * 8;
    int NS = 2;  // raw slots: as many as fit, up to 8
    while (NS < 8 && fixed + (size_t)(NS + 1) * (slot + 16) <= kMaxSmem)
        NS++;
    const size_t smem = fixed + (size_t)NS * (slot + 16);
    if (smem > kMaxSmem)
        return 1;
    static std::atomic<unsigned long long> smem_set{0};
    if (allow_dynamic_smem(reinterpret_cast<const void *>(interact_bwd_tc_kernel), (int)kMaxSmem, &smem_set) !=
        DLRM_OK)
        return DLRM_ERR_CUDA;
    const int64_t grid = nunits < sm_count() ? nunits : sm_count();
    interact_bwd_tc_kernel<<<(unsigned)grid, kBwdThreads, smem, st>>>(map_emb, map_e0, N, d, B, mode, dy, dys, de0,
                                                                       de0s, demb, dembs, Np, bx, NS);
    count_launch(st);
    return launch_status();
}

}  // namespace dlrm
