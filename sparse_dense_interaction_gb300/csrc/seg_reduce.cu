// Segmented reduce of pooled-vector gradients over runs of equal rows, and
// the row-wise update of each unique row (the embedding-bag backward of
// "Notes/DLRM", vault-aram.pages.dev: section 2's per-feature lookups are
// summed, so every lookup of a row receives its bag's pooled gradient;
// section 5: the rows are then trained by an optimizer -- plain SGD, or
// row-wise AdaGrad).
//
// Design.  One CTA per sort tile (4096 sorted lookups of one table):
//  A. the CTA stages the tile's sorted rows and, through the position of each
//     lookup, its bag id in shared memory, marks where runs of equal rows
//     start, counts the starts of every chunk and numbers the runs;
//  B. a stream of G lanes walks one chunk of sorted lookups (for d >= 128: 16
//     streams of 16 lanes, 256 lookups each; a lane owns two 16-byte pieces
//     of each pooled-gradient row), 2 rows in flight, fp32 sums with packed
//     adds; the table rows of runs starting a step ahead are prefetched into
//     L2.  The kernel is kept lean (at most 64 registers, so 4 CTAs of 8
//     warps share an SM and hide the latency of the row gathers); when a run
//     ends its table row is updated once (SGD: w - lr*g; AdaGrad: the row's
//     sum of squares reduced over the stream, the accumulator updated once,
//     w - lr*g/(sqrt(s')+eps)): fp32 and fp16 rows by an L2 reduction of the
//     rounded step, bf16 rows read, updated and written back.  Runs that
//     cross a chunk boundary leave partial sums, which two small kernels
//     combine in chunk order (block sums of 32 chunks, then the run's owner),
//     so results are deterministic.
#include <type_traits>

#include "emb_bag_bwd.cuh"

namespace dlrm {

// VEC fp32 gradient values of one lane, added with packed fp32 adds.
template <int VEC>
struct Vec;
template <>
struct Vec<4> {
    using F = float4;
    __device__ __forceinline__ static F zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ static F load(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
    __device__ __forceinline__ static void store(float *p, const F &v) { *reinterpret_cast<float4 *>(p) = v; }
    __device__ __forceinline__ static void add(F &a, const F &b)
    {
        const float2 lo = __fadd2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y));
        const float2 hi = __fadd2_rn(make_float2(a.z, a.w), make_float2(b.z, b.w));
        a = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    __device__ __forceinline__ static float get(const F &v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
    // s + the squares of the four values
    __device__ __forceinline__ static float sumsq(const F &v, float s)
    {
        return fmaf(v.w, v.w, fmaf(v.z, v.z, fmaf(v.y, v.y, fmaf(v.x, v.x, s))));
    }
};
template <>
struct Vec<1> {
    using F = float;
    __device__ __forceinline__ static F zero() { return 0.f; }
    __device__ __forceinline__ static F load(const float *p) { return __ldg(p); }
    __device__ __forceinline__ static void store(float *p, const F &v) { *p = v; }
    __device__ __forceinline__ static void add(F &a, const F &b) { a += b; }
    __device__ __forceinline__ static float get(const F &v, int) { return v; }
    __device__ __forceinline__ static float sumsq(const F &v, float s) { return fmaf(v, v, s); }
};

// VEC consecutive table elements of one lane.
template <typename TT, int VEC>
struct RowChunk {
    static constexpr int kBytes = (int)sizeof(TT) * VEC;
    using R = typename std::conditional<
        kBytes == 16, uint4,
        typename std::conditional<kBytes == 8, uint2,
                                  typename std::conditional<kBytes == 4, uint32_t, uint16_t>::type>::type>::type;
    __device__ __forceinline__ static R load(const TT *p) { return *reinterpret_cast<const R *>(p); }
    __device__ __forceinline__ static void store(TT *p, const R &r) { *reinterpret_cast<R *>(p) = r; }
    // w <- w - lr * g in fp32 (one fused multiply-add), rounded once to TT
    __device__ __forceinline__ static R sgd(R r, const typename Vec<VEC>::F &g, float lr)
    {
        TT *h = reinterpret_cast<TT *>(&r);
#pragma unroll
        for (int i = 0; i < VEC; i++)
            h[i] = from_f32<TT>(fmaf(-lr, Vec<VEC>::get(g, i), to_f32<TT>(h[i])));
        return r;
    }
};

// The update of fp32 and fp16 rows as one reduction performed in L2: the
// step -lr*g (AdaGrad: lr / (sqrt(s') + eps) in place of lr) is computed in
// fp32, rounded to the table type and added to the row (rounded again);
// nothing waits for the row.  Each unique row receives
// one such update per launch (its run's whole sum), so the result does not
// depend on timing.  bf16 rows keep the read-modify-write (one rounding):
// their 8-bit significand leaves too little room for two.
template <typename TT, int VEC>
struct RedUpdate {
    static constexpr bool kUse = false;
    __device__ __forceinline__ static void apply(TT *, const typename Vec<VEC>::F &, float) {}
};
template <>
struct RedUpdate<float, 4> {
    static constexpr bool kUse = true;
    __device__ __forceinline__ static void apply(float *p, const float4 &g, float lr)
    {
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(-lr * g.x), "f"(-lr * g.y),
                     "f"(-lr * g.z), "f"(-lr * g.w)
                     : "memory");
    }
};
template <>
struct RedUpdate<float, 1> {
    static constexpr bool kUse = true;
    __device__ __forceinline__ static void apply(float *p, float g, float lr)
    {
        asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(-lr * g) : "memory");
    }
};
template <>
struct RedUpdate<__half, 4> {
    static constexpr bool kUse = true;
    __device__ __forceinline__ static void apply(__half *p, const float4 &g, float lr)
    {
        const __half2 a = __floats2half2_rn(-lr * g.x, -lr * g.y), b = __floats2half2_rn(-lr * g.z, -lr * g.w);
        asm volatile("red.global.add.noftz.v2.f16x2 [%0], {%1, %2};" ::"l"(p),
                     "r"(*reinterpret_cast<const uint32_t *>(&a)), "r"(*reinterpret_cast<const uint32_t *>(&b))
                     : "memory");
    }
};
template <>
struct RedUpdate<__half, 1> {
    static constexpr bool kUse = true;
    __device__ __forceinline__ static void apply(__half *p, float g, float lr)
    {
        const __half h = __float2half_rn(-lr * g);
        asm volatile("red.global.add.noftz.f16 [%0], %1;" ::"l"(p), "h"(*reinterpret_cast<const unsigned short *>(&h))
                     : "memory");
    }
};

// Asks L2 to fetch the line holding p (no register result, never faults the
// caller: only called on rows inside the table).
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// G lanes form a stream that walks one chunk; each lane owns C pieces of VEC
// fp32 values of every gradient row (piece c of lane l covers elements
// (c*G + l)*VEC ..), U lookups in flight per stream.  With the update on, the
// table rows of runs that start PD steps ahead are prefetched into L2, so the
// read-modify-write at a run's end finds its row there.  FULL: d is a whole
// number of passes of G*C*VEC elements, so every piece lies inside the row and
// the gathers test only that the lookup has a bag.
template <typename TT, int VEC, int G, int C, int U, int PD, bool FULL>
__global__ void __launch_bounds__(kReduceThreads, 4)
seg_reduce_kernel(ReduceArgs a, BwdPtrs w)
{
    using V = Vec<VEC>;
    using F = typename V::F;
    using RC = RowChunk<TT, VEC>;
    constexpr int S = 32 / G;                      // streams per warp
    constexpr int NS = (kReduceThreads / 32) * S;  // chunks per tile, one stream each
    constexpr int CW = kTile / NS;                 // sorted lookups per chunk
    constexpr int EB = G * C * VEC;                // row elements per pass
    constexpr int PER = kTile / kReduceThreads;    // staged lookups per thread
    constexpr uint32_t kStart = 0x80000000u;       // bag word: a run starts here
    constexpr uint32_t kNoBag = 0x7fffffffu;       // bag word: no valid bag
    static_assert(NS <= 32 && CW % 32 == 0, "chunk geometry");

    // sorted row, bag of the lookup | kStart at run starts; lookup i at sk(i): one spare entry
    // after each chunk, so the two 16-lane streams of a warp read different banks
    __shared__ uint2 skb[kTile + NS];
    auto sk = [](uint32_t i) { return i + i / CW; };
    __shared__ uint32_t cbase[NS];
    __shared__ TileInfo ti;
    __shared__ uint32_t key_before, key_after;
    if (*w.sort_failed)  // the coalescing gave up a wait: its results are invalid, update nothing
        return;
    const bool ids = *w.ids_ready != 0u;  // the unique keys are numbered: write the view's arrays
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 32)
        find_tile_warp(blockIdx.x, a.T, w.tile_base, w.tstart, ti);
    if (tid < NS)
        cbase[tid] = 0;
    __syncthreads();
    if (!ti.valid)
        return;
    const int t = ti.t;
    const uint32_t lo = ti.lo, n = ti.hi - ti.lo;
    const uint32_t ts = w.tstart[t], te = w.tstart[t + 1];
    const uint32_t *skey = w.keys[a.final_buf];
    const uint32_t *sval = w.vals[a.final_buf];
    if (tid == 0) {
        key_before = lo > ts ? skey[lo - 1] : 0u;
        key_after = ti.hi < te ? skey[ti.hi] : 0u;
    }
    const bool update = a.lr != 0.f;
    const bool adagrad = a.opt == kOptAdagrad;
    TT *wtab = static_cast<TT *>(const_cast<void *>(a.tables.ptr[t]));
    const int64_t rows_t = a.tables.rows[t];

    // A. stage rows and bag ids (8 lookups per thread in flight); the sort carried the bag ids
    // unless the coalescing was asked for its view (then the positions, whose bags are looked up)
    const bool vals_bags = *w.vals_bags != 0u;
    for (int r0 = 0; r0 < PER; r0 += 8) {
        uint32_t pos[8];
#pragma unroll
        for (int r = 0; r < 8; r++) {
            const uint32_t i = (uint32_t)(r0 + r) * kReduceThreads + tid;
            pos[r] = 0;
            if (i < n) {
                skb[sk(i)].x = skey[lo + i];
                pos[r] = sval[lo + i];
            }
        }
#pragma unroll
        for (int r = 0; r < 8; r++) {
            const uint32_t i = (uint32_t)(r0 + r) * kReduceThreads + tid;
            if (i < n) {
                uint32_t b = vals_bags ? pos[r] : w.bag_of[pos[r]];
                if ((int64_t)b >= a.B) {
                    raise_flag(a.err, DLRM_FLAG_BAD_OFFSETS);
                    b = kNoBag;
                }
                skb[sk(i)].y = b;
            }
        }
    }
    __syncthreads();
    // run starts, counted per chunk (each warp step covers 32 consecutive lookups)
    for (int r = 0; r < PER; r++) {
        const uint32_t i = (uint32_t)r * kReduceThreads + tid;
        bool st = false;
        if (i < n) {
            st = lo + i == ts || skb[sk(i)].x != (i == 0 ? key_before : skb[sk(i - 1)].x);
            if (st)
                skb[sk(i)].y |= kStart;
        }
        const unsigned bal = __ballot_sync(0xffffffffu, st);
        if (lane == 0 && bal)
            atomicAdd(&cbase[((uint32_t)r * kReduceThreads + warp * 32) / CW], (uint32_t)__popc(bal));
    }
    // pad the tile to a whole number of steps with lookups that contribute
    // nothing and start no run, so the walk below needs no bounds checks
    if (tid < (int)((U - n % U) % U))  // n is then below kTile, a multiple of U
        skb[sk(n + tid)] = make_uint2(0u, kNoBag);
    __syncthreads();
    if (warp == 0) {
        const uint32_t v = lane < NS ? cbase[lane] : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += x;
        }
        if (lane < NS)
            cbase[lane] = (ids ? w.tile_ubase[blockIdx.x] : 0u) + incl - v;
    }
    __syncthreads();

    // B. one stream of G lanes per chunk
    const int sidx = warp * S + lane / G;
    const int gl = lane % G;
    const unsigned smask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (lane / G * G));  // this stream's lanes
    const size_t ch = (size_t)blockIdx.x * NS + sidx;
    const uint32_t c0 = (uint32_t)sidx * CW;
    const uint32_t c1 = c0 + CW < n ? c0 + CW : n;
    if (c0 >= c1) {
        if (gl == 0)
            w.chunk_flags[ch] = 0;
        return;
    }
    const bool carry_in = !(skb[sk(c0)].y & kStart);
    const bool carry_out = c1 < n ? !(skb[sk(c1)].y & kStart) : (ti.hi < te && key_after == skb[sk(n - 1)].x);
    const uint2 *skc = skb + sidx;  // this chunk's lookups: skc[p] is lookup p (p in c0 .. c1e)
    const uint32_t ub = cbase[sidx];
    uint32_t flags = 0;

    for (int eb = 0; eb < a.d; eb += EB) {
        bool on[C];
#pragma unroll
        for (int c = 0; c < C; c++)
            on[c] = eb + (c * G + gl) * VEC < a.d;
        const char *dpt_bytes = reinterpret_cast<const char *>(a.dpooled + (int64_t)t * a.dpts + eb + gl * VEC);
        const uint32_t dpss_bytes = (uint32_t)a.dpss * 4u;
        F acc[C];
#pragma unroll
        for (int c = 0; c < C; c++)
            acc[c] = V::zero();
        bool cur_carry = carry_in;
        uint32_t cur_row = 0, cur_u = 0, cur_start = lo + c0, nseg = 0;

        auto flush = [&](bool last) {
            if (cur_carry) {
#pragma unroll
                for (int c = 0; c < C; c++)
                    if (on[c])
                        V::store(w.head + ch * a.d + eb + (c * G + gl) * VEC, acc[c]);
                flags |= kHasHead | ((last && carry_out) ? 0u : kHeadEnds);
            } else {
                if (ids && eb == 0 && gl == 0) {
                    w.uniq_table[cur_u] = t;
                    w.uniq_row[cur_u] = cur_row;
                    w.seg_off[cur_u] = cur_start;
                }
                if (last && carry_out) {
#pragma unroll
                    for (int c = 0; c < C; c++)
                        if (on[c])
                            V::store(w.tail + ch * a.d + eb + (c * G + gl) * VEC, acc[c]);
                    flags |= kHasTail;
                    if (eb == 0 && gl == 0) {
                        w.chunk_tail_row[ch] = cur_row;
                        w.chunk_tail_t[ch] = t;
                        w.chunk_tail_u[ch] = cur_u;  // meaningful when the keys are numbered
                    }
                } else {
                    if (a.grad_rows) {
                        if ((int64_t)cur_u < a.grad_cap) {
#pragma unroll
                            for (int c = 0; c < C; c++)
                                if (on[c])
                                    V::store(a.grad_rows + (int64_t)cur_u * a.d + eb + (c * G + gl) * VEC, acc[c]);
                        } else if (gl == 0 && eb == 0) {
                            raise_flag(a.err, DLRM_FLAG_CAPACITY);
                        }
                    }
                    if (update && (int64_t)cur_row < rows_t) {
                        float step = a.lr;
                        if (adagrad) {
                            // the whole row is in this stream's registers (d <= EB)
                            float ss = 0.f;
#pragma unroll
                            for (int c = 0; c < C; c++)
                                if (on[c])
                                    ss = V::sumsq(acc[c], ss);
#pragma unroll
                            for (int o = G / 2; o > 0; o >>= 1)
                                ss += __shfl_xor_sync(smask, ss, o);
                            float *sp = a.state.ptr[t] + cur_row;
                            const float s1 = *sp + ss / (float)a.d;
                            step = a.lr / (sqrtf(s1) + a.eps);
                            if (gl == 0)
                                *sp = s1;
                        }
#pragma unroll
                        for (int c = 0; c < C; c++)
                            if (on[c]) {
                                TT *wp = wtab + (int64_t)cur_row * a.d + eb + (c * G + gl) * VEC;
                                if (RedUpdate<TT, VEC>::kUse)
                                    RedUpdate<TT, VEC>::apply(wp, acc[c], step);
                                else
                                    RC::store(wp, RC::sgd(RC::load(wp), acc[c], step));
                            }
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < C; c++)
                acc[c] = V::zero();
        };

        const uint32_t c1e = c1 + (U - c1 % U) % U;  // padded end of the walk
        for (uint32_t p0 = c0; p0 < c1e; p0 += U) {
            if (PD > 0 && update && (adagrad || !RedUpdate<TT, VEC>::kUse)) {
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const uint32_t q = p0 + PD * U + u;
                    if (q < c1) {
                        const uint2 kb = skc[q];
                        if ((kb.y & kStart) && (int64_t)kb.x < rows_t) {
                            if (!RedUpdate<TT, VEC>::kUse) {  // rows updated in L2 are not read here
                                const TT *wr = wtab + (int64_t)kb.x * a.d + eb + gl * VEC;
#pragma unroll
                                for (int c = 0; c < C; c++)
                                    if (on[c])
                                        prefetch_l2(wr + c * G * VEC);
                            }
                            if (adagrad && gl == 0)
                                prefetch_l2(a.state.ptr[t] + kb.x);
                        }
                    }
                }
            }
            F g[U][C];
            uint32_t starts = 0;  // bit u: a run starts at p0 + u
#pragma unroll
            for (int u = 0; u < U; u++) {
                const uint32_t by = skc[p0 + u].y;
                starts |= (by >> 31) << u;
                const uint32_t b = by & ~kStart;
                const float *src = reinterpret_cast<const float *>(dpt_bytes + (uint64_t)b * dpss_bytes);
#pragma unroll
                for (int c = 0; c < C; c++) {
                    g[u][c] = V::zero();
                    if (b != kNoBag && (FULL || on[c]))
                        g[u][c] = V::load(src + c * G * VEC);
                }
            }
#pragma unroll
            for (int u = 0; u < U; u++) {
                if ((starts >> u) & 1u) {
                    if (p0 + u > c0)
                        flush(false);
                    cur_carry = false;
                    cur_row = skc[p0 + u].x;
                    cur_start = lo + p0 + u;
                    cur_u = ub + nseg;
                    nseg++;
                }
#pragma unroll
                for (int c = 0; c < C; c++)
                    V::add(acc[c], g[u][c]);
            }
        }
        flush(true);
    }
    if (gl == 0)
        w.chunk_flags[ch] = flags;
}

// Runs that cross chunk boundaries are combined in two levels, all sums in
// chunk order (deterministic).  Level 1: one warp per block of 32 chunks sums
// the partials of the run that enters the block at its first chunk, up to that
// run's end or the block's end.  Level 2: the warp of the chunk where a run
// starts adds the partials of the following chunks up to the next block
// boundary, then one block sum per block, and applies the update.
constexpr uint32_t kBlockEnters = 1u, kBlockEnds = 2u;

// Sums chunk partials head[c0 .. c0 + count) into acc, 8 loads in flight.
template <int VEC>
__device__ __forceinline__ void add_heads(typename Vec<VEC>::F &acc, const float *head, size_t c0, int count,
                                          int d, int e)
{
    using V = Vec<VEC>;
    for (int i0 = 0; i0 < count; i0 += 8) {
        typename V::F g[8];
#pragma unroll
        for (int i = 0; i < 8; i++)
            g[i] = (i0 + i < count && e < d) ? V::load(head + (c0 + i0 + i) * d + e) : V::zero();
#pragma unroll
        for (int i = 0; i < 8; i++)
            V::add(acc, g[i]);
    }
}

// Number of chunk flags from c (at most `limit`) to add for a run that
// continues into chunk c: up to and including the first chunk where it ends.
// Sets ends when the run ends within them; flags a chunk without a partial.
__device__ __forceinline__ int run_extent(const uint32_t *flags, size_t c, int limit, bool &ends, int lane,
                                          int32_t *err)
{
    const uint32_t f = lane < limit ? flags[c + lane] : kHasHead;
    const unsigned endm = __ballot_sync(0xffffffffu, lane < limit && (f & kHeadEnds));
    const unsigned bad = __ballot_sync(0xffffffffu, lane < limit && !(f & kHasHead));
    int count = endm ? __ffs(endm) : limit;
    ends = endm != 0;
    if (bad && __ffs(bad) - 1 < count) {
        if (lane == 0)
            raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
        count = __ffs(bad) - 1;
        ends = true;
    }
    return count;
}

template <int VEC>
__global__ void __launch_bounds__(256)
seg_block_sum_kernel(ReduceArgs a, BwdPtrs w, int NS)
{
    if (*w.sort_failed)
        return;
    using V = Vec<VEC>;
    using F = typename V::F;
    constexpr int EB = 32 * VEC;
    const int lane = threadIdx.x & 31;
    const size_t nch = (size_t)w.tile_base[a.T] * NS;
    const size_t nblk = (nch + kFinalizeBlock - 1) / kFinalizeBlock;
    const size_t nwarps = (size_t)gridDim.x * (blockDim.x / 32);
    for (size_t blk = (size_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); blk < nblk; blk += nwarps) {
        const size_t c0 = blk * kFinalizeBlock;
        if (!(w.chunk_flags[c0] & kHasHead)) {
            if (lane == 0)
                w.block_flags[blk] = 0;
            continue;
        }
        const int limit = (int)(nch - c0 < (size_t)kFinalizeBlock ? nch - c0 : kFinalizeBlock);
        bool ends;
        const int count = run_extent(w.chunk_flags, c0, limit, ends, lane, a.err);
        for (int eb = 0; eb < a.d; eb += EB) {
            const int e = eb + lane * VEC;
            F acc = V::zero();
            add_heads<VEC>(acc, w.head, c0, count, a.d, e);
            if (e < a.d)
                V::store(w.block_sum + blk * a.d + e, acc);
        }
        if (lane == 0)
            w.block_flags[blk] = kBlockEnters | (ends ? kBlockEnds : 0u);
    }
}

template <typename TT, int VEC, int NB>
__global__ void __launch_bounds__(256)
seg_finalize_kernel(ReduceArgs a, BwdPtrs w, int NS)
{
    if (*w.sort_failed)
        return;
    using V = Vec<VEC>;
    using F = typename V::F;
    constexpr int EB = 32 * VEC;
    const int lane = threadIdx.x & 31;
    const size_t nch = (size_t)w.tile_base[a.T] * NS;
    const size_t nblk = (nch + kFinalizeBlock - 1) / kFinalizeBlock;
    const size_t nwarps = (size_t)gridDim.x * (blockDim.x / 32);
    for (size_t ch = (size_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); ch < nch; ch += nwarps) {
        if (!(w.chunk_flags[ch] & kHasTail))
            continue;
        const uint32_t row = w.chunk_tail_row[ch];
        const int t = w.chunk_tail_t[ch];
        const uint32_t u = a.grad_rows ? w.chunk_tail_u[ch] : 0u;  // gradient rows: the keys are numbered
        // chunks up to the next block boundary, one by one
        const size_t c1 = ch + 1;
        const size_t bound = ((c1 + kFinalizeBlock - 1) / kFinalizeBlock) * kFinalizeBlock;
        const size_t stop = bound < nch ? bound : nch;
        bool ends = c1 >= nch;
        int count = 0;
        if (!ends && stop > c1)
            count = run_extent(w.chunk_flags, c1, (int)(stop - c1), ends, lane, a.err);
        // then whole blocks: their flags 32 at a time
        size_t first_blk = stop / kFinalizeBlock, nblocks_run = 0;
        for (size_t blk = first_blk; !ends && blk < nblk; blk += 32) {
            const uint32_t bf = blk + lane < nblk ? w.block_flags[blk + lane] : (kBlockEnters | kBlockEnds);
            const unsigned endm = __ballot_sync(0xffffffffu, (bf & kBlockEnds) != 0);
            const unsigned bad = __ballot_sync(0xffffffffu, (bf & kBlockEnters) == 0);
            int n = endm ? __ffs(endm) : 32;
            if (bad && __ffs(bad) - 1 < n) {
                if (lane == 0)
                    raise_flag(a.err, DLRM_FLAG_BAD_OFFSETS);
                n = __ffs(bad) - 1;
                ends = true;
            }
            nblocks_run += n;
            if (endm)
                ends = true;
        }
        if (a.opt == kOptAdagrad) {
            // the whole row (d <= NB * EB), then its sum of squares over the warp
            F acc[NB];
            float ss = 0.f;
#pragma unroll
            for (int nb = 0; nb < NB; nb++) {
                const int e = nb * EB + lane * VEC;
                acc[nb] = e < a.d ? V::load(w.tail + ch * a.d + e) : V::zero();
                add_heads<VEC>(acc[nb], w.head, c1, count, a.d, e);
                add_heads<VEC>(acc[nb], w.block_sum, first_blk, (int)nblocks_run, a.d, e);
                ss = V::sumsq(acc[nb], ss);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const bool in_table = (int64_t)row < a.tables.rows[t];
            float step = 0.f;
            if (in_table && a.lr != 0.f) {
                float *sp = a.state.ptr[t] + row;
                const float s1 = *sp + ss / (float)a.d;
                step = a.lr / (sqrtf(s1) + a.eps);
                if (lane == 0)
                    *sp = s1;
            }
#pragma unroll
            for (int nb = 0; nb < NB; nb++) {
                const int e = nb * EB + lane * VEC;
                if (e >= a.d)
                    continue;
                if (a.grad_rows) {
                    if ((int64_t)u < a.grad_cap)
                        V::store(a.grad_rows + (int64_t)u * a.d + e, acc[nb]);
                    else if (lane == 0 && nb == 0)
                        raise_flag(a.err, DLRM_FLAG_CAPACITY);
                }
                if (in_table && a.lr != 0.f) {
                    TT *wp = static_cast<TT *>(const_cast<void *>(a.tables.ptr[t])) + (int64_t)row * a.d + e;
                    if (RedUpdate<TT, VEC>::kUse)
                        RedUpdate<TT, VEC>::apply(wp, acc[nb], step);
                    else
                        RowChunk<TT, VEC>::store(wp, RowChunk<TT, VEC>::sgd(RowChunk<TT, VEC>::load(wp), acc[nb], step));
                }
            }
            continue;
        }
        for (int eb = 0; eb < a.d; eb += EB) {
            const int e = eb + lane * VEC;
            F acc = e < a.d ? V::load(w.tail + ch * a.d + e) : V::zero();
            add_heads<VEC>(acc, w.head, c1, count, a.d, e);
            add_heads<VEC>(acc, w.block_sum, first_blk, (int)nblocks_run, a.d, e);
            if (e < a.d) {
                if (a.grad_rows) {
                    if ((int64_t)u < a.grad_cap)
                        V::store(a.grad_rows + (int64_t)u * a.d + e, acc);
                    else if (lane == 0 && eb == 0)
                        raise_flag(a.err, DLRM_FLAG_CAPACITY);
                }
                if (a.lr != 0.f && (int64_t)row < a.tables.rows[t]) {
                    TT *wp = static_cast<TT *>(const_cast<void *>(a.tables.ptr[t])) + (int64_t)row * a.d + e;
                    if (RedUpdate<TT, VEC>::kUse)
                        RedUpdate<TT, VEC>::apply(wp, acc, a.lr);
                    else
                        RowChunk<TT, VEC>::store(wp, RowChunk<TT, VEC>::sgd(RowChunk<TT, VEC>::load(wp), acc, a.lr));
                }
            }
        }
    }
}

template <typename TT, int VEC, int G, int C, int U, int PD>
static int run_reduce(const ReduceArgs &a, const BwdPtrs &w, int64_t grid, cudaStream_t st)
{
    if (a.d % (G * C * VEC) == 0)
        seg_reduce_kernel<TT, VEC, G, C, U, PD, true><<<(unsigned)grid, kReduceThreads, 0, st>>>(a, w);
    else
        seg_reduce_kernel<TT, VEC, G, C, U, PD, false><<<(unsigned)grid, kReduceThreads, 0, st>>>(a, w);
    count_launch(st);
    int s = launch_status();
    if (s != DLRM_OK)
        return s;
    constexpr int NS = (kReduceThreads / 32) * (32 / G);
    const int64_t chunks = grid * NS;
    const int64_t blocks = (chunks + kFinalizeBlock - 1) / kFinalizeBlock;  // one warp per block of chunks
    seg_block_sum_kernel<VEC><<<(unsigned)((blocks + 7) / 8), 256, 0, st>>>(a, w, NS);
    count_launch(st);
    if ((s = launch_status()) != DLRM_OK)
        return s;
    // AdaGrad holds whole rows: 2 x 128 (vectorised) or 8 x 32 (scalar) elements
    seg_finalize_kernel<TT, VEC, kAdagradMaxD / (32 * VEC)><<<(unsigned)((chunks + 7) / 8), 256, 0, st>>>(a, w, NS);
    count_launch(st);
    return launch_status();
}

template <typename TT>
static int reduce_typed(const ReduceArgs &a, const BwdPtrs &w, int64_t grid, bool vec, cudaStream_t st)
{
    if (a.opt == kOptAdagrad) {
        // a stream holds the whole row: up to 128 (16 x 2 x 4), 256 (32 x 2 x 4)
        // or 256 (32 x 8 x 1, scalar) elements
        if (!vec)
            return run_reduce<TT, 1, 32, 8, 2, 0>(a, w, grid, st);
        if (a.d > 128)
            return run_reduce<TT, 4, 32, 2, 2, 1>(a, w, grid, st);
        return run_reduce<TT, 4, 16, 2, 2, 1>(a, w, grid, st);
    }
    if (!vec)
        return run_reduce<TT, 1, 32, 1, 8, 0>(a, w, grid, st);
    // 16-lane streams (more chunks per tile, shorter serial walks): two
    // 16-byte pieces per lane for rows of 128+ values, one for rows of up to
    // 64; rows in between keep one 32-lane stream per chunk (a single walk)
    // (the rows of fp32 and fp16 tables are updated by L2 reductions and never
    // read here: nothing to prefetch)
    constexpr int PD = RedUpdate<TT, 4>::kUse ? 0 : 1;
    if (a.d >= 128)
        return run_reduce<TT, 4, 16, 2, 2, PD>(a, w, grid, st);
    if (a.d <= 64)
        return run_reduce<TT, 4, 16, 1, 2, PD>(a, w, grid, st);
    return run_reduce<TT, 4, 32, 1, 4, PD>(a, w, grid, st);
}

int launch_seg_reduce(int dtype, const ReduceArgs &a, const BwdPtrs &w, int64_t grid, bool vec, cudaStream_t st)
{
    switch (dtype) {
    case DLRM_F32:
        return reduce_typed<float>(a, w, grid, vec, st);
    case DLRM_F16:
        return reduce_typed<__half>(a, w, grid, vec, st);
    default:
        return reduce_typed<__nv_bfloat16>(a, w, grid, vec, st);
    }
}

}  // namespace dlrm
