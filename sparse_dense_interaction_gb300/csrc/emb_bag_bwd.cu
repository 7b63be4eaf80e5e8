// Embedding-bag backward with row-wise SGD.
//
// The gradient of a table row is the sum of the pooled-vector gradients of
// every bag that looked it up ("Notes/DLRM", vault-aram.pages.dev, sections 2
// and 9: the lookups are summed into one vector per feature); the rows are
// then trained by the optimizer (section 5; plain SGD on the touched rows).
//
// Pipeline (all on the caller's stream, no host synchronisation):
//  1. prep       table start positions from the CSR offsets, tiles per table
//  2. bag ids    bag number of every lookup position (4 bytes per lookup)
//  3. sort       stable LSD radix sort of (row, position) pairs, segmented by
//                table: the CSR input is already grouped by table, so tiles
//                never straddle a table and only the row bits are sorted
//                (ceil(log2 max_rows) bits, <= 8 per pass).  Per pass:
//                tile histograms -> per-(table,digit) scan across tiles ->
//                stable local ranking in shared memory (warp match + per-warp
//                histograms) and a coalesced scatter.
//  4. count      segment starts per 512-position chunk of the sorted order
//  5. scan       exclusive scan of the per-tile counts: unique ids
//  6. reduce     one warp per chunk: walks its 512 sorted lookups, gathers
//                the pooled gradient rows (16-byte loads, 8 rows in flight
//                per lane), accumulates each run of equal rows in fp32 and
//                applies SGD to the run's row in place, one read-modify-write
//                per unique row.  Runs that cross chunk boundaries leave
//                partial sums.  Work per warp is fixed (512 lookups) however
//                skewed the row distribution is.
//  7. finalize   the warp whose chunk holds the start of a crossing run sums
//                the partials in chunk order and applies the update, so every
//                result is deterministic.
#include "common.cuh"

namespace dlrm {

constexpr int kTile = 4096;          // sorted positions per CTA
constexpr int kSortThreads = 256;    // 8 warps
constexpr int kItems = kTile / kSortThreads;  // 16 per thread
constexpr int kChunk = kTile / 8;    // 512 positions per warp in count/reduce
constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kMaxPasses = 4;
constexpr uint32_t kSentinel = 0xffffffffu;
constexpr uint32_t kHasHead = 1u, kHeadEnds = 2u, kHasTail = 4u;

struct BwdLayout {
    size_t keys[2], vals[2], bag_of, uniq_table, uniq_row, seg_off, hist, counts, tstart, tile_base,
        tile_count, tile_ubase, chunk_count, chunk_flags, chunk_tail_u, head, tail, num_unique, total;
    int64_t ntiles_max, nchunks_max;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

BwdLayout bwd_layout(int T, int64_t nnz, int d)
{
    BwdLayout L{};
    L.ntiles_max = (nnz + kTile - 1) / kTile + T;
    L.nchunks_max = L.ntiles_max * 8;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align256(off + bytes);
        return at;
    };
    const size_t n4 = (size_t)nnz * 4;
    L.keys[0] = take(n4);
    L.vals[0] = take(n4);
    L.keys[1] = take(n4);
    L.vals[1] = take(n4);
    L.bag_of = take(n4);
    L.uniq_table = take(n4);
    L.uniq_row = take(n4);
    L.seg_off = take(n4 + 4);
    L.hist = take((size_t)kRadix * L.ntiles_max * 4);
    L.counts = take((size_t)kMaxPasses * T * kRadix * 4);
    L.tstart = take(((size_t)T + 1) * 4);
    L.tile_base = take(((size_t)T + 1) * 4);
    L.tile_count = take((size_t)L.ntiles_max * 4);
    L.tile_ubase = take((size_t)L.ntiles_max * 4);
    L.chunk_count = take((size_t)L.nchunks_max * 4);
    L.chunk_flags = take((size_t)L.nchunks_max * 4);
    L.chunk_tail_u = take((size_t)L.nchunks_max * 4);
    L.head = take((size_t)L.nchunks_max * d * 4);
    L.tail = take((size_t)L.nchunks_max * d * 4);
    L.num_unique = take(8);
    L.total = off;
    return L;
}

struct BwdPtrs {
    uint32_t *keys[2], *vals[2], *bag_of, *uniq_row, *seg_off, *hist, *counts, *tstart, *tile_base,
        *tile_count, *tile_ubase, *chunk_count, *chunk_flags, *chunk_tail_u;
    int32_t *uniq_table;
    float *head, *tail;
    int64_t *num_unique;
    int64_t ntiles_max;
};

struct TileInfo {
    int t;
    uint32_t lo, hi;
    int valid;
};

// Table and position range of sort tile tau (thread 0; broadcast via smem).
__device__ __forceinline__ void find_tile(int64_t tau, int T, const uint32_t *tile_base,
                                          const uint32_t *tstart, TileInfo &ti)
{
    if (tau >= tile_base[T]) {
        ti.valid = 0;
        return;
    }
    int lo = 0, hi = T;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (tile_base[mid] <= tau)
            lo = mid;
        else
            hi = mid;
    }
    ti.t = lo;
    ti.lo = tstart[lo] + (uint32_t)(tau - tile_base[lo]) * kTile;
    const uint32_t end = tstart[lo + 1];
    ti.hi = ti.lo + kTile < end ? ti.lo + kTile : end;
    ti.valid = 1;
}

// ---------------------------------------------------------------- prep ---

__global__ void __launch_bounds__(256)
bwd_prep_kernel(const int64_t *__restrict__ offsets, int T, int64_t B, int64_t nnz, BwdPtrs w,
                int32_t *err)
{
    __shared__ int64_t start[DLRM_MAX_TABLES + 1];
    for (int t = threadIdx.x; t <= T; t += blockDim.x)
        start[t] = offsets[(int64_t)t * B];
    __syncthreads();
    if (threadIdx.x == 0) {
        bool bad = start[0] != 0 || start[T] != nnz;
        int64_t prev = 0;
        for (int t = 0; t <= T; t++) {
            int64_t v = start[t];
            v = v < prev ? prev : (v > nnz ? nnz : v);
            if (t == T)
                v = nnz;
            if (v != start[t])
                bad = true;
            start[t] = v;
            prev = v;
        }
        if (bad)
            raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
        uint32_t tb = 0;
        for (int t = 0; t < T; t++) {
            w.tile_base[t] = tb;
            tb += (uint32_t)((start[t + 1] - start[t] + kTile - 1) / kTile);
        }
        w.tile_base[T] = tb;
        *w.num_unique = 0;
    }
    __syncthreads();
    for (int t = threadIdx.x; t <= T; t += blockDim.x)
        w.tstart[t] = (uint32_t)start[t];
    for (int i = threadIdx.x; i < kMaxPasses * T * kRadix; i += blockDim.x)
        w.counts[i] = 0;
}

// ------------------------------------------------------------- bag ids ---

__global__ void __launch_bounds__(256)
bag_ids_kernel(const int64_t *__restrict__ offsets, int T, int64_t B, int64_t nnz,
               uint32_t *__restrict__ bag_of, int32_t *err)
{
    const int64_t nbags = (int64_t)T * B;
    for (int64_t bag = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; bag < nbags;
         bag += (int64_t)gridDim.x * blockDim.x) {
        const int64_t k0 = offsets[bag], k1 = offsets[bag + 1];
        if (k0 < 0 || k1 < k0 || k1 > nnz) {
            raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
            continue;
        }
        const uint32_t b = (uint32_t)(bag % B);
        for (int64_t k = k0; k < k1; k++)
            bag_of[k] = b;
    }
}

// ---------------------------------------------------------------- sort ---

// Sort key of position j: its row in pass 0 (read from the int64 indices and
// checked against the table), the carried key afterwards.
__device__ __forceinline__ uint32_t pass0_key(const int64_t *indices, uint32_t j, int64_t R)
{
    const int64_t r = indices[j];
    return (r >= 0 && r < R) ? (uint32_t)r : kSentinel;
}

__global__ void __launch_bounds__(kSortThreads)
sort_upsweep_kernel(int pass, int shift, int nbits, const int64_t *__restrict__ indices,
                    TableSet ts, int T, BwdPtrs w, int32_t *err)
{
    __shared__ uint32_t hist[kRadix];
    __shared__ TileInfo ti;
    if (threadIdx.x == 0)
        find_tile(blockIdx.x, T, w.tile_base, w.tstart, ti);
    for (int i = threadIdx.x; i < kRadix; i += blockDim.x)
        hist[i] = 0;
    __syncthreads();
    if (!ti.valid)
        return;
    const uint32_t mask = (1u << nbits) - 1u;
    // pass p reads buffer (p+1)&1 (written by pass p-1) and writes buffer p&1
    const uint32_t *keys = w.keys[(pass + 1) & 1];
    const int64_t R = ts.rows[ti.t];
    bool oob = false;
    const int lane = threadIdx.x & 31;
    for (uint32_t base = ti.lo; base < ti.hi; base += kSortThreads) {
        const uint32_t j = base + threadIdx.x;
        const bool valid = j < ti.hi;
        uint32_t digit = kRadix;  // never matches a real digit
        if (valid) {
            uint32_t key;
            if (pass == 0) {
                key = pass0_key(indices, j, R);
                oob |= key == kSentinel;
            } else {
                key = keys[j];
            }
            digit = (key >> shift) & mask;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        if (valid && lane == __ffs(peers) - 1)
            atomicAdd(&hist[digit], __popc(peers));
    }
    if (oob)
        raise_flag(err, DLRM_FLAG_INDEX_OOB);
    __syncthreads();
    uint32_t *counts = w.counts + ((size_t)pass * T + ti.t) * kRadix;
    for (int dg = threadIdx.x; dg <= (int)mask; dg += blockDim.x) {
        const uint32_t c = hist[dg];
        w.hist[(size_t)dg * w.ntiles_max + blockIdx.x] = c;
        if (c)
            atomicAdd(&counts[dg], c);
    }
}

// One warp per (table, digit): global start of the digit's run in the table
// plus the exclusive prefix over the table's tiles, written in place.
__global__ void __launch_bounds__(256)
sort_scan_kernel(int pass, int nbits, int T, BwdPtrs w)
{
    const int radix = 1 << nbits;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= (int64_t)T * radix)
        return;
    const int t = (int)(gw / radix);
    const int dg = (int)(gw % radix);
    const uint32_t *counts = w.counts + ((size_t)pass * T + t) * kRadix;
    uint32_t below = 0;
    for (int i = lane; i < dg; i += 32)
        below += counts[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        below += __shfl_xor_sync(0xffffffffu, below, o);
    uint32_t run = w.tstart[t] + below;
    const uint32_t t0 = w.tile_base[t], t1 = w.tile_base[t + 1];
    uint32_t *h = w.hist + (size_t)dg * w.ntiles_max;
    for (uint32_t tb = t0; tb < t1; tb += 32) {
        const uint32_t tau = tb + lane;
        const uint32_t v = tau < t1 ? h[tau] : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += n;
        }
        if (tau < t1)
            h[tau] = run + incl - v;
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
}

__global__ void __launch_bounds__(kSortThreads)
sort_downsweep_kernel(int pass, int shift, int nbits, const int64_t *__restrict__ indices,
                      TableSet ts, int T, BwdPtrs w)
{
    __shared__ uint32_t skey[kTile];
    __shared__ uint32_t sval[kTile];
    __shared__ uint32_t whist[8][kRadix];
    __shared__ uint32_t tdig[kRadix];  // exclusive prefix of the tile's digit counts
    __shared__ uint32_t gbase[kRadix];
    __shared__ uint32_t wsum[8];
    __shared__ TileInfo ti;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        find_tile(blockIdx.x, T, w.tile_base, w.tstart, ti);
    for (int i = tid; i < 8 * kRadix; i += kSortThreads)
        (&whist[0][0])[i] = 0;
    __syncthreads();
    if (!ti.valid)
        return;
    const uint32_t mask = (1u << nbits) - 1u;
    const int radix = 1 << nbits;
    for (int dg = tid; dg < radix; dg += kSortThreads)
        gbase[dg] = w.hist[(size_t)dg * w.ntiles_max + blockIdx.x];
    const uint32_t *keys_in = w.keys[(pass + 1) & 1];
    const uint32_t *vals_in = w.vals[(pass + 1) & 1];
    uint32_t *keys_out = w.keys[pass & 1];
    uint32_t *vals_out = w.vals[pass & 1];
    const int64_t R = ts.rows[ti.t];

    uint32_t key[kItems], val[kItems], rank[kItems];
    const uint32_t wbase = ti.lo + warp * (kTile / 8);
#pragma unroll
    for (int i = 0; i < kItems; i++) {
        const uint32_t j = wbase + i * 32 + lane;
        const bool valid = j < ti.hi;
        if (pass == 0) {
            key[i] = valid ? pass0_key(indices, j, R) : 0u;
            val[i] = j;
        } else {
            key[i] = valid ? keys_in[j] : 0u;
            val[i] = valid ? vals_in[j] : 0u;
        }
    }
    // stable rank within the warp: items in position order (i, then lane)
#pragma unroll
    for (int i = 0; i < kItems; i++) {
        const uint32_t j = wbase + i * 32 + lane;
        const bool valid = j < ti.hi;
        const uint32_t digit = valid ? (key[i] >> shift) & mask : (uint32_t)kRadix;
        const unsigned peers = __match_any_sync(0xffffffffu, digit);
        const uint32_t before = __popc(peers & ((1u << lane) - 1u));
        uint32_t r = 0;
        if (valid)
            r = whist[warp][digit] + before;
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1)
            whist[warp][digit] += __popc(peers);
        __syncwarp();
        rank[i] = r;
    }
    __syncthreads();
    // per digit: exclusive prefix across warps, then across digits
    uint32_t total = 0;
    if (tid < radix) {
        for (int wi = 0; wi < 8; wi++) {
            const uint32_t c = whist[wi][tid];
            whist[wi][tid] = total;
            total += c;
        }
    }
    // block-wide exclusive scan of the digit totals (radix <= 256 threads)
    uint32_t incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += n;
    }
    if (lane == 31)
        wsum[warp] = incl;
    __syncthreads();
    uint32_t wprefix = 0;
    for (int wi = 0; wi < warp; wi++)
        wprefix += wsum[wi];
    if (tid < radix)
        tdig[tid] = wprefix + incl - total;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kItems; i++) {
        const uint32_t j = wbase + i * 32 + lane;
        if (j < ti.hi) {
            const uint32_t digit = (key[i] >> shift) & mask;
            const uint32_t lp = tdig[digit] + whist[warp][digit] + rank[i];
            skey[lp] = key[i];
            sval[lp] = val[i];
        }
    }
    __syncthreads();
    const uint32_t n = ti.hi - ti.lo;
    for (uint32_t j = tid; j < n; j += kSortThreads) {
        const uint32_t k = skey[j];
        const uint32_t digit = (k >> shift) & mask;
        const uint32_t dest = gbase[digit] + (j - tdig[digit]);
        keys_out[dest] = k;
        vals_out[dest] = sval[j];
    }
}

// ------------------------------------------------------ segment count ---

__global__ void __launch_bounds__(256)
seg_count_kernel(int T, int final_buf, BwdPtrs w)
{
    __shared__ TileInfo ti;
    __shared__ uint32_t wc[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        find_tile(blockIdx.x, T, w.tile_base, w.tstart, ti);
    __syncthreads();
    if (!ti.valid)
        return;
    const uint32_t *skey = w.keys[final_buf];
    const uint32_t ts = w.tstart[ti.t];
    const uint32_t c0 = ti.lo + warp * kChunk;
    const uint32_t c1 = c0 + kChunk < ti.hi ? c0 + kChunk : ti.hi;
    uint32_t count = 0;
    for (uint32_t jb = c0; jb < c1; jb += 32) {
        const uint32_t j = jb + lane;
        const bool start = j < c1 && (j == ts || skey[j] != skey[j - 1]);
        count += __popc(__ballot_sync(0xffffffffu, start));
    }
    if (lane == 0) {
        w.chunk_count[(size_t)blockIdx.x * 8 + warp] = count;
        wc[warp] = count;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t s = 0;
        for (int i = 0; i < 8; i++)
            s += wc[i];
        w.tile_count[blockIdx.x] = s;
    }
}

// Exclusive scan of the per-tile segment counts (one CTA of 1024 threads).
__global__ void __launch_bounds__(1024)
seg_scan_kernel(int T, int64_t nnz, BwdPtrs w)
{
    __shared__ uint32_t wsum[32];
    __shared__ uint32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t n = w.tile_base[T];
    if (tid == 0)
        carry = 0;
    __syncthreads();
    constexpr int PER = 8;
    for (uint32_t base = 0; base < n; base += 1024 * PER) {
        uint32_t v[PER], s = 0;
#pragma unroll
        for (int i = 0; i < PER; i++) {
            const uint32_t idx = base + tid * PER + i;
            v[i] = idx < n ? w.tile_count[idx] : 0u;
            s += v[i];
        }
        uint32_t incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += x;
        }
        if (lane == 31)
            wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            uint32_t ws = wsum[lane];
            uint32_t wi = ws;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t x = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o)
                    wi += x;
            }
            wsum[lane] = wi - ws;
        }
        __syncthreads();
        uint32_t run = carry + wsum[warp] + incl - s;
#pragma unroll
        for (int i = 0; i < PER; i++) {
            const uint32_t idx = base + tid * PER + i;
            if (idx < n)
                w.tile_ubase[idx] = run;
            run += v[i];
        }
        __syncthreads();
        if (tid == 1023)
            carry = run;
        __syncthreads();
    }
    if (tid == 0) {
        *w.num_unique = carry;
        w.seg_off[carry] = (uint32_t)nnz;
    }
}

// ------------------------------------------------ reduce + row update ---

struct ReduceArgs {
    TableSet tables;  // written in place when lr != 0
    int T, d;
    int64_t B;
    const float *dpooled;
    int64_t dpss, dpts;
    float lr;
    float *grad_rows;
    int64_t grad_cap;
    int final_buf;
    int32_t *err;
};

template <int VEC>
struct Vec;
template <>
struct Vec<4> {
    using F = float4;
    __device__ __forceinline__ static F zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ static F load(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
    __device__ __forceinline__ static void store(float *p, const F &v) { *reinterpret_cast<float4 *>(p) = v; }
    __device__ __forceinline__ static void add(F &a, const F &b) { a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w; }
    __device__ __forceinline__ static float get(const F &v, int i) { return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w; }
};
template <>
struct Vec<1> {
    using F = float;
    __device__ __forceinline__ static F zero() { return 0.f; }
    __device__ __forceinline__ static F load(const float *p) { return __ldg(p); }
    __device__ __forceinline__ static void store(float *p, const F &v) { *p = v; }
    __device__ __forceinline__ static void add(F &a, const F &b) { a += b; }
    __device__ __forceinline__ static float get(const F &v, int) { return v; }
};

// SGD on VEC consecutive elements of one row: w <- w - lr * g, computed in
// fp32 with one fused multiply-add and one rounding to the table type.
template <typename TT, int VEC>
__device__ __forceinline__ void sgd_update(TT *wrow, const typename Vec<VEC>::F &g, float lr)
{
    if constexpr (VEC == 4 && sizeof(TT) == 4) {
        float4 wv = *reinterpret_cast<float4 *>(wrow);
        wv.x = fmaf(-lr, g.x, wv.x);
        wv.y = fmaf(-lr, g.y, wv.y);
        wv.z = fmaf(-lr, g.z, wv.z);
        wv.w = fmaf(-lr, g.w, wv.w);
        *reinterpret_cast<float4 *>(wrow) = wv;
    } else if constexpr (VEC == 4) {
        uint2 raw = *reinterpret_cast<uint2 *>(wrow);
        TT *h = reinterpret_cast<TT *>(&raw);
#pragma unroll
        for (int i = 0; i < 4; i++)
            h[i] = from_f32<TT>(fmaf(-lr, Vec<4>::get(g, i), to_f32<TT>(h[i])));
        *reinterpret_cast<uint2 *>(wrow) = raw;
    } else {
        wrow[0] = from_f32<TT>(fmaf(-lr, g, to_f32<TT>(wrow[0])));
    }
}

template <typename TT, int VEC, int NV>
__device__ __forceinline__ void apply_row(const ReduceArgs &a, int t, uint32_t u, uint32_t row,
                                          int eb, int lane, const typename Vec<VEC>::F (&acc)[NV])
{
    if (a.grad_rows) {
        if ((int64_t)u < a.grad_cap) {
#pragma unroll
            for (int v = 0; v < NV; v++) {
                const int e = eb + (lane + 32 * v) * VEC;
                if (e < a.d)
                    Vec<VEC>::store(a.grad_rows + (int64_t)u * a.d + e, acc[v]);
            }
        } else if (lane == 0 && eb == 0) {
            raise_flag(a.err, DLRM_FLAG_CAPACITY);
        }
    }
    if (a.lr != 0.f && (int64_t)row < a.tables.rows[t]) {
        TT *wrow = static_cast<TT *>(const_cast<void *>(a.tables.ptr[t])) + (int64_t)row * a.d;
#pragma unroll
        for (int v = 0; v < NV; v++) {
            const int e = eb + (lane + 32 * v) * VEC;
            if (e < a.d)
                sgd_update<TT, VEC>(wrow + e, acc[v], a.lr);
        }
    }
}

template <typename TT, int VEC, int NV>
__global__ void __launch_bounds__(256)
seg_reduce_kernel(ReduceArgs a, BwdPtrs w)
{
    using V = Vec<VEC>;
    using F = typename V::F;
    constexpr int EB = 32 * VEC * NV;  // elements per pass over the chunk
    constexpr int U = 8;               // gradient rows in flight per lane
    __shared__ TileInfo ti;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        find_tile(blockIdx.x, a.T, w.tile_base, w.tstart, ti);
    __syncthreads();
    if (!ti.valid)
        return;
    const int t = ti.t;
    const size_t ch = (size_t)blockIdx.x * 8 + warp;
    const uint32_t c0 = ti.lo + warp * kChunk;
    const uint32_t c1 = c0 + kChunk < ti.hi ? c0 + kChunk : ti.hi;
    if (c0 >= c1) {
        if (lane == 0)
            w.chunk_flags[ch] = 0;
        return;
    }
    const uint32_t *skey = w.keys[a.final_buf];
    const uint32_t *sval = w.vals[a.final_buf];
    const uint32_t ts = w.tstart[t], te = w.tstart[t + 1];
    uint32_t ub = lane < warp ? w.chunk_count[(size_t)blockIdx.x * 8 + lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        ub += __shfl_xor_sync(0xffffffffu, ub, o);
    ub += w.tile_ubase[blockIdx.x];
    const bool carry_in = c0 > ts && skey[c0] == skey[c0 - 1];
    const bool carry_out = c1 < te && skey[c1] == skey[c1 - 1];
    const float *dpt = a.dpooled + (int64_t)t * a.dpts;
    uint32_t flags = 0;

    for (int eb = 0; eb < a.d; eb += EB) {
        F acc[NV];
#pragma unroll
        for (int v = 0; v < NV; v++)
            acc[v] = V::zero();
        bool cur_carry = carry_in;
        uint32_t cur_row = skey[c0], cur_u = 0, cur_start = c0, nseg = 0;

        auto flush = [&](bool last) {
            if (cur_carry) {
#pragma unroll
                for (int v = 0; v < NV; v++) {
                    const int e = eb + (lane + 32 * v) * VEC;
                    if (e < a.d)
                        V::store(w.head + ch * a.d + e, acc[v]);
                }
                flags |= kHasHead | ((last && carry_out) ? 0u : kHeadEnds);
            } else {
                if (eb == 0 && lane == 0) {
                    w.uniq_table[cur_u] = t;
                    w.uniq_row[cur_u] = cur_row;
                    w.seg_off[cur_u] = cur_start;
                }
                if (last && carry_out) {
#pragma unroll
                    for (int v = 0; v < NV; v++) {
                        const int e = eb + (lane + 32 * v) * VEC;
                        if (e < a.d)
                            V::store(w.tail + ch * a.d + e, acc[v]);
                    }
                    flags |= kHasTail;
                    if (eb == 0 && lane == 0)
                        w.chunk_tail_u[ch] = cur_u;
                } else {
                    apply_row<TT, VEC, NV>(a, t, cur_u, cur_row, eb, lane, acc);
                }
            }
#pragma unroll
            for (int v = 0; v < NV; v++)
                acc[v] = V::zero();
        };

        for (uint32_t jb = c0; jb < c1; jb += 32) {
            const uint32_t j = jb + lane;
            const bool valid = j < c1;
            const uint32_t key_l = valid ? skey[j] : 0u;
            const uint32_t pos_l = valid ? sval[j] : 0u;
            const bool start_l = valid && (j == ts || key_l != skey[j - 1]);
            uint32_t b_l = valid ? w.bag_of[pos_l] : 0u;
            if (valid && (int64_t)b_l >= a.B) {
                raise_flag(a.err, DLRM_FLAG_BAD_OFFSETS);
                b_l = 0xffffffffu;
            }
            const unsigned startmask = __ballot_sync(0xffffffffu, start_l);
            const int n = (int)(c1 - jb < 32 ? c1 - jb : 32);
            for (int q = 0; q < n; q += U) {
                F g[U][NV];
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const uint32_t bq = __shfl_sync(0xffffffffu, b_l, (q + u) & 31);
                    const bool ok = (q + u) < n && bq != 0xffffffffu;
                    const float *src = dpt + (int64_t)bq * a.dpss;
#pragma unroll
                    for (int v = 0; v < NV; v++) {
                        const int e = eb + (lane + 32 * v) * VEC;
                        g[u][v] = (ok && e < a.d) ? V::load(src + e) : V::zero();
                    }
                }
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const int src = q + u;
                    if (src < n) {
                        if ((startmask >> src) & 1u) {
                            if (jb + src > c0)
                                flush(false);
                            cur_carry = false;
                            cur_row = __shfl_sync(0xffffffffu, key_l, src);
                            cur_start = jb + src;
                            cur_u = ub + nseg;
                            nseg++;
                        }
#pragma unroll
                        for (int v = 0; v < NV; v++)
                            V::add(acc[v], g[u][v]);
                    }
                }
            }
        }
        flush(true);
    }
    if (lane == 0)
        w.chunk_flags[ch] = flags;
}

// Runs that cross chunk boundaries: the owner (the chunk where the run
// starts) adds the partial sums of the following chunks in order.
template <typename TT, int VEC, int NV>
__global__ void __launch_bounds__(256)
seg_finalize_kernel(ReduceArgs a, BwdPtrs w)
{
    using V = Vec<VEC>;
    using F = typename V::F;
    constexpr int EB = 32 * VEC * NV;
    const int lane = threadIdx.x & 31;
    const size_t ch = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const size_t nch = (size_t)w.tile_base[a.T] * 8;
    if (ch >= nch || !(w.chunk_flags[ch] & kHasTail))
        return;
    const uint32_t u = w.chunk_tail_u[ch];
    const uint32_t row = w.uniq_row[u];
    const int t = w.uniq_table[u];
    for (int eb = 0; eb < a.d; eb += EB) {
        F acc[NV];
#pragma unroll
        for (int v = 0; v < NV; v++) {
            const int e = eb + (lane + 32 * v) * VEC;
            acc[v] = e < a.d ? V::load(w.tail + ch * a.d + e) : V::zero();
        }
        bool done = false;
        for (size_t c = ch + 1; !done && c < nch; c += 32) {
            const size_t cc = c + lane;
            const uint32_t f = cc < nch ? w.chunk_flags[cc] : (kHasHead | kHeadEnds);
            const unsigned ends = __ballot_sync(0xffffffffu, (f & kHeadEnds) != 0);
            const unsigned bad = __ballot_sync(0xffffffffu, (f & kHasHead) == 0);
            int count = ends ? __ffs(ends) : 32;
            if (bad) {
                const int first_bad = __ffs(bad) - 1;
                if (first_bad < count) {
                    if (lane == 0)
                        raise_flag(a.err, DLRM_FLAG_BAD_OFFSETS);
                    count = first_bad;
                    done = true;
                }
            }
            for (int i0 = 0; i0 < count; i0 += 8) {
                F g[8][NV];
#pragma unroll
                for (int i = 0; i < 8; i++)
#pragma unroll
                    for (int v = 0; v < NV; v++) {
                        const int e = eb + (lane + 32 * v) * VEC;
                        g[i][v] = (i0 + i < count && e < a.d) ? V::load(w.head + (c + i0 + i) * a.d + e)
                                                               : V::zero();
                    }
#pragma unroll
                for (int i = 0; i < 8; i++)
#pragma unroll
                    for (int v = 0; v < NV; v++)
                        V::add(acc[v], g[i][v]);
            }
            if (ends)
                done = true;
        }
        apply_row<TT, VEC, NV>(a, t, u, row, eb, lane, acc);
    }
}

// ---------------------------------------------------------------- host ---

static int row_bits(const TableSet &ts, int T)
{
    int64_t maxr = 1;
    for (int t = 0; t < T; t++)
        maxr = ts.rows[t] > maxr ? ts.rows[t] : maxr;
    int bits = 1;
    while (bits < 32 && ((int64_t)1 << bits) < maxr)
        bits++;
    return bits;
}

template <typename TT, int VEC, int NV>
static int launch_reduce(const ReduceArgs &a, const BwdPtrs &w, int64_t grid, cudaStream_t st)
{
    seg_reduce_kernel<TT, VEC, NV><<<(unsigned)grid, 256, 0, st>>>(a, w);
    count_launch(st);
    int s = launch_status();
    if (s != DLRM_OK)
        return s;
    seg_finalize_kernel<TT, VEC, NV><<<(unsigned)grid, 256, 0, st>>>(a, w);
    count_launch(st);
    return launch_status();
}

template <typename TT>
static int launch_reduce_typed(const ReduceArgs &a, const BwdPtrs &w, int64_t grid, bool vec,
                               cudaStream_t st)
{
    if (vec)
        return a.d <= 128 ? launch_reduce<TT, 4, 1>(a, w, grid, st) : launch_reduce<TT, 4, 2>(a, w, grid, st);
    return launch_reduce<TT, 1, 4>(a, w, grid, st);
}

bool emb_bag_bwd_vectorisable(const TableSet &ts, int T, int d, const float *dpooled, int64_t dpss,
                              int64_t dpts, const float *grad_rows)
{
    auto al = [](const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    if (d % 4 != 0 || !al(dpooled) || dpss % 4 != 0 || dpts % 4 != 0)
        return false;
    if (grad_rows && !al(grad_rows))
        return false;
    for (int t = 0; t < T; t++)
        if (!al(ts.ptr[t]))
            return false;
    return true;
}

size_t emb_bag_bwd_workspace(int T, int64_t nnz, int d) { return bwd_layout(T, nnz, d).total; }

int launch_emb_bag_bwd(const TableSet &ts, int T, int d, int dtype, const int64_t *offsets,
                       const int64_t *indices, int64_t nnz, int64_t B, const float *dpooled,
                       int64_t dpss, int64_t dpts, float lr, float *grad_rows, int64_t grad_cap,
                       void *workspace, bool vec, dlrm_coalesced_view *view, int32_t *err,
                       cudaStream_t st)
{
    const BwdLayout L = bwd_layout(T, nnz, d);
    char *base = static_cast<char *>(workspace);
    BwdPtrs w;
    for (int i = 0; i < 2; i++) {
        w.keys[i] = reinterpret_cast<uint32_t *>(base + L.keys[i]);
        w.vals[i] = reinterpret_cast<uint32_t *>(base + L.vals[i]);
    }
    w.bag_of = reinterpret_cast<uint32_t *>(base + L.bag_of);
    w.uniq_table = reinterpret_cast<int32_t *>(base + L.uniq_table);
    w.uniq_row = reinterpret_cast<uint32_t *>(base + L.uniq_row);
    w.seg_off = reinterpret_cast<uint32_t *>(base + L.seg_off);
    w.hist = reinterpret_cast<uint32_t *>(base + L.hist);
    w.counts = reinterpret_cast<uint32_t *>(base + L.counts);
    w.tstart = reinterpret_cast<uint32_t *>(base + L.tstart);
    w.tile_base = reinterpret_cast<uint32_t *>(base + L.tile_base);
    w.tile_count = reinterpret_cast<uint32_t *>(base + L.tile_count);
    w.tile_ubase = reinterpret_cast<uint32_t *>(base + L.tile_ubase);
    w.chunk_count = reinterpret_cast<uint32_t *>(base + L.chunk_count);
    w.chunk_flags = reinterpret_cast<uint32_t *>(base + L.chunk_flags);
    w.chunk_tail_u = reinterpret_cast<uint32_t *>(base + L.chunk_tail_u);
    w.head = reinterpret_cast<float *>(base + L.head);
    w.tail = reinterpret_cast<float *>(base + L.tail);
    w.num_unique = reinterpret_cast<int64_t *>(base + L.num_unique);
    w.ntiles_max = L.ntiles_max;

    const int bits = row_bits(ts, T);
    const int passes = (bits + kRadixBits - 1) / kRadixBits;
    const int final_buf = (passes - 1) & 1;
    if (view) {
        view->sorted_pos = w.vals[final_buf];
        view->sorted_row = w.keys[final_buf];
        view->uniq_table = w.uniq_table;
        view->uniq_row = w.uniq_row;
        view->seg_off = w.seg_off;
        view->num_unique = w.num_unique;
    }

    int s;
    bwd_prep_kernel<<<1, 256, 0, st>>>(offsets, T, B, nnz, w, err);
    count_launch(st);
    if ((s = launch_status()) != DLRM_OK)
        return s;
    if (nnz == 0) {
        cudaMemsetAsync(w.seg_off, 0, 4, st);
        return launch_status();
    }
    {
        const int64_t nbags = (int64_t)T * B;
        int64_t grid = (nbags + 255) / 256;
        const int64_t cap = (int64_t)sm_count() * 8;
        bag_ids_kernel<<<(unsigned)(grid < cap ? grid : cap), 256, 0, st>>>(offsets, T, B, nnz, w.bag_of, err);
        count_launch(st);
        if ((s = launch_status()) != DLRM_OK)
            return s;
    }
    const int64_t grid = L.ntiles_max;
    int shift = 0;
    for (int p = 0; p < passes; p++) {
        const int nb = bits / passes + (p < bits % passes ? 1 : 0);
        sort_upsweep_kernel<<<(unsigned)grid, kSortThreads, 0, st>>>(p, shift, nb, indices, ts, T, w, err);
        count_launch(st);
        if ((s = launch_status()) != DLRM_OK)
            return s;
        const int64_t warps = (int64_t)T << nb;
        sort_scan_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, st>>>(p, nb, T, w);
        count_launch(st);
        if ((s = launch_status()) != DLRM_OK)
            return s;
        sort_downsweep_kernel<<<(unsigned)grid, kSortThreads, 0, st>>>(p, shift, nb, indices, ts, T, w);
        count_launch(st);
        if ((s = launch_status()) != DLRM_OK)
            return s;
        shift += nb;
    }
    seg_count_kernel<<<(unsigned)grid, 256, 0, st>>>(T, final_buf, w);
    count_launch(st);
    if ((s = launch_status()) != DLRM_OK)
        return s;
    seg_scan_kernel<<<1, 1024, 0, st>>>(T, nnz, w);
    count_launch(st);
    if ((s = launch_status()) != DLRM_OK)
        return s;

    ReduceArgs a;
    a.tables = ts;
    a.T = T;
    a.d = d;
    a.B = B;
    a.dpooled = dpooled;
    a.dpss = dpss;
    a.dpts = dpts;
    a.lr = lr;
    a.grad_rows = grad_rows;
    a.grad_cap = grad_cap;
    a.final_buf = final_buf;
    a.err = err;
    switch (dtype) {
    case DLRM_F32:
        return launch_reduce_typed<float>(a, w, grid, vec, st);
    case DLRM_F16:
        return launch_reduce_typed<__half>(a, w, grid, vec, st);
    default:
        return launch_reduce_typed<__nv_bfloat16>(a, w, grid, vec, st);
    }
}

}  // namespace dlrm
