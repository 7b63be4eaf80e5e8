// Embedding-bag backward with row-wise SGD.
//
// The gradient of a table row is the sum of the pooled-vector gradients of
// every bag that looked it up ("Notes/DLRM", vault-aram.pages.dev, sections 2
// and 9: the lookups are summed into one vector per feature); the rows are
// then trained by the optimizer (section 5; plain SGD on the touched rows).
//
// Pipeline (all on the caller's stream, no host synchronisation):
//  1. prep       table start positions from the CSR offsets, tiles per table
//  2. bag ids    bag number of every lookup position (4 bytes per lookup,
//                written coalesced)
//  3. sort       stable LSD radix sort of (row, position) pairs, segmented by
//                table: the CSR input is already grouped by table, so tiles
//                never straddle a table and only the row bits are sorted
//                (ceil(log2 max_rows) bits, <= 8 per pass).  One kernel
//                counts the digits of every pass per table; then one kernel
//                per pass ranks each tile in shared memory (warp match +
//                per-warp histograms), finds the counts of the tiles before
//                it by decoupled look-back, and scatters coalesced.  For
//                uniform lookups into large tables the first pass sorts by
//                the top 8 row bits instead and one CTA per bucket finishes
//                the sort in shared memory, unless the digit counts show a
//                bucket larger than a tile.
//  4. count      run starts (a new row, or a table's first lookup) per tile
//  5. scan       exclusive scan of the per-tile counts: the runs' unique ids
//  6. reduce     per tile, the summed pooled gradient of every run of equal
//                rows and the SGD update of its row (seg_reduce.cu)
//  7. finalize   runs that cross chunk boundaries (seg_reduce.cu)
#include <cstring>

#include "emb_bag_bwd.cuh"

namespace dlrm {

struct BwdLayout {
    size_t keys[2], vals[2], bag_of, uniq_table, uniq_row, seg_off, status[2], tile_ctr, tile_hist, counts, tstart, tile_base,
        tile_count, tile_ubase, chunk_flags, chunk_tail_u, chunk_tail_row, chunk_tail_t, head, tail, block_flags,
        block_sum, num_unique, total;
    int64_t ntiles_max, nchunks_max;
};

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

BwdLayout bwd_layout(int T, int64_t nnz, int d)
{
    BwdLayout L{};
    L.ntiles_max = (nnz + kTile - 1) / kTile + T;
    L.nchunks_max = L.ntiles_max * reduce_chunks_per_tile(d);
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
    L.status[0] = take((size_t)kRadix * L.ntiles_max * 8);
    L.status[1] = take((size_t)kRadix * L.ntiles_max * 8);
    // the LSD passes' and the MSD pass's tile counters, sort failed, value kind, ids ready, MSD state
    L.tile_ctr = take(((size_t)kMaxPasses + 5) * 4);
    L.tile_hist = take((size_t)L.ntiles_max * kSortRows * kRadix * 4);
    L.counts = take((size_t)kSortRows * T * kRadix * 4);
    L.tstart = take(((size_t)T + 1) * 4);
    L.tile_base = take(((size_t)T + 1) * 4);
    L.tile_count = take((size_t)L.ntiles_max * 4);
    L.tile_ubase = take((size_t)L.ntiles_max * 4);
    L.chunk_flags = take((size_t)L.nchunks_max * 4);
    L.chunk_tail_u = take((size_t)L.nchunks_max * 4);
    L.chunk_tail_row = take((size_t)L.nchunks_max * 4);
    L.chunk_tail_t = take((size_t)L.nchunks_max * 4);
    L.head = take((size_t)L.nchunks_max * d * 4);
    L.tail = take((size_t)L.nchunks_max * d * 4);
    const int64_t nblocks = L.nchunks_max / kFinalizeBlock + 1;
    L.block_flags = take((size_t)nblocks * 4);
    L.block_sum = take((size_t)nblocks * d * 4);
    L.num_unique = take(8);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------- prep ---

__global__ void __launch_bounds__(256)
bwd_prep_kernel(const int64_t *__restrict__ offsets, int T, int64_t B, int64_t nnz, BwdPtrs w,
                uint32_t first_tile, uint32_t vals_bags, uint32_t msd, int32_t *err)
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
    if (threadIdx.x <= kMaxPasses)
        w.tile_ctr[threadIdx.x] = first_tile;  // 0 unless a test leaves the first tiles unclaimed
    if (threadIdx.x == kMaxPasses + 1)
        *w.sort_failed = 0;
    if (threadIdx.x == kMaxPasses + 2)
        *w.vals_bags = vals_bags;
    if (threadIdx.x == kMaxPasses + 3)
        *w.ids_ready = 0;  // until the unique keys are numbered
    if (threadIdx.x == kMaxPasses + 4)
        *w.msd_state = msd ? kMsdPlanned : 0u;
}

// ------------------------------------------------------------- bag ids ---

// A warp takes 32 consecutive bags; each lane finds the bag of a lookup
// position by binary search over the 33 offsets held in the warp's lanes, so
// the bag ids are written as coalesced 128-byte rows.
__global__ void __launch_bounds__(256)
bag_ids_kernel(const int64_t *__restrict__ offsets, int T, int64_t B, int64_t nnz,
               uint32_t *__restrict__ bag_of, int32_t *err)
{
    const int lane = threadIdx.x & 31;
    const int64_t nbags = (int64_t)T * B;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t g0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * 32; g0 < nbags; g0 += nwarps * 32) {
        const int64_t bag = g0 + lane;
        // start of this lane's bag; lanes past the last bag never match
        int64_t o = bag <= nbags ? offsets[bag] : nnz + 1;
        const int64_t last = g0 + 32 < nbags ? g0 + 32 : nbags;
        const int64_t end = offsets[last];
        const int64_t next = __shfl_down_sync(0xffffffffu, o, 1);
        const bool bad = bag < last && (o < 0 || o > nnz || (lane < 31 ? next : end) < o);
        if (__any_sync(0xffffffffu, bad)) {
            if (lane == 0)
                raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
            continue;
        }
        if (bag > last)
            o = nnz + 1;
        const int64_t start = __shfl_sync(0xffffffffu, o, 0);
        const uint32_t bid = (uint32_t)((g0 + lane) % B);  // this lane's bag within its table, once per group
        // positions relative to the group's first one fit in 32 bits (nnz <= 2^31): 32-bit shuffles
        // and compares in the search (lanes past the last bag never match)
        const uint32_t orel = o <= nnz ? (uint32_t)(o - start) : 0xffffffffu;
        const uint32_t n = (uint32_t)(end - start);
        // warp-uniform trip count: every lane takes part in every shuffle
        for (uint32_t q0 = 0; q0 < n; q0 += 32) {
            const uint32_t q = q0 + lane;
            int l = 0;
#pragma unroll
            for (int step = 16; step > 0; step >>= 1) {  // l + step <= 31
                if (__shfl_sync(0xffffffffu, orel, l + step) <= q)
                    l += step;
            }
            const uint32_t b = __shfl_sync(0xffffffffu, bid, l);
            if (q < n)
                bag_of[start + q] = b;
        }
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

// Digit width and shift of pass p when `bits` key bits are split over
// `passes` passes as evenly as possible (wider passes first).
__host__ __device__ __forceinline__ int pass_bits(int bits, int passes, int p)
{
    return bits / passes + (p < bits % passes ? 1 : 0);
}

// Digit counts of every pass from one read of the indices, one CTA of 512
// threads per tile (8 indices per thread in flight), written to the tile's row
// of counts.  A table's digit
// histogram does not depend on the order of its keys, so all passes are
// counted here; the digit scan below sums the rows of the table's tiles, and
// each pass finds the counts of the tiles before its own by looking back.
// With msd_shift >= 0 row `passes` counts the top digit (key >> msd_shift)
// for the pass that sorts by it first.  Also clears the look-back words of
// pass 1 (the first pass needs none) and flags indices out of range.
__global__ void __launch_bounds__(2 * kSortThreads)
sort_hist_kernel(int bits, int passes, int msd_shift, const int64_t *__restrict__ indices, TableSet ts, int T,
                 BwdPtrs w, int32_t *err)
{
    constexpr int kThreads = 2 * kSortThreads;  // 512: one CTA per tile, 8 indices per thread in flight
    __shared__ uint32_t h[kSortRows][kRadix];
    __shared__ TileInfo ti;
    const int tid = threadIdx.x;
    const int64_t tau = blockIdx.x;
    if (tid < 32)
        find_tile_warp(tau, T, w.tile_base, w.tstart, ti);
    for (int i = tid; i < kSortRows * kRadix; i += kThreads)
        (&h[0][0])[i] = 0;
    __syncthreads();
    if (!ti.valid)
        return;
    if (tid < kRadix)
        w.status[1][(size_t)tau * kRadix + tid] = 0;
    const int64_t R = ts.rows[ti.t];
    const uint32_t lo = ti.lo;
    uint32_t key[kTile / kThreads];
#pragma unroll
    for (int i = 0; i < kTile / kThreads; i++) {
        const uint32_t j = lo + i * kThreads + tid;
        key[i] = j < ti.hi ? pass0_key(indices, j, R) : 0u;
    }
    bool oob = false;
#pragma unroll
    for (int i = 0; i < kTile / kThreads; i++) {
        if (lo + i * kThreads + tid < ti.hi) {
            oob |= key[i] == kSentinel;
            int shift = 0;
            for (int p = 0; p < passes; p++) {
                const int nb = pass_bits(bits, passes, p);
                atomicAdd(&h[p][(key[i] >> shift) & ((1u << nb) - 1u)], 1u);
                shift += nb;
            }
            if (msd_shift >= 0)
                atomicAdd(&h[passes][(key[i] >> msd_shift) & (kRadix - 1u)], 1u);
        }
    }
    if (oob)
        raise_flag(err, DLRM_FLAG_INDEX_OOB);
    __syncthreads();
    uint32_t *row = w.tile_hist + ((size_t)blockIdx.x * kSortRows) * kRadix;
    const int rows = passes + (msd_shift >= 0 ? 1 : 0);
    for (int i = tid; i < rows * kRadix; i += kThreads)
        row[i] = (&h[0][0])[i];
}

// One CTA per (pass, table): sums the digit counts of the table's tiles
// (four groups of kRadix threads, one thread per digit) and scans them into
// the start position of each digit's keys in the table's sorted range.  For
// the rows in `prefix_rows` (the first pass's: its tiles hold the keys in the
// order the histogram counted them) the groups take consecutive quarters of
// the tiles and replace each tile's counts by the exclusive prefix over the
// table's earlier tiles, so the first pass finds its offsets without looking
// back.  For the MSD digit's row (`msd_row`) a bucket of more than kTile keys
// sets kMsdOverflow before any pass runs.
constexpr int kScanGroups = 4;
__global__ void __launch_bounds__(kScanGroups * kRadix)
sort_digit_scan_kernel(int msd_row, unsigned prefix_rows, int T, BwdPtrs w)
{
    __shared__ uint32_t part[kScanGroups][kRadix];
    __shared__ uint32_t wsum[kRadix / 32];
    const int p = blockIdx.x / T, t = blockIdx.x % T;
    const int tid = threadIdx.x, dg = tid % kRadix, g = tid / kRadix, lane = tid & 31, warp = tid >> 5;
    const uint32_t h0 = w.tile_base[t], h1 = w.tile_base[t + 1];
    uint32_t *col = w.tile_hist + (size_t)p * kRadix + dg;
    constexpr size_t kRow = (size_t)kSortRows * kRadix;  // words per tile
    const bool prefix = (prefix_rows >> p) & 1u;
    uint32_t c = 0, r0 = 0, r1 = 0;
    if (prefix) {
        const uint32_t n = h1 - h0, q = (n + kScanGroups - 1) / kScanGroups;
        r0 = h0 + min((uint32_t)g * q, n);
        r1 = h0 + min((uint32_t)(g + 1) * q, n);
        uint32_t hb = r0;
        for (; hb + 8 <= r1; hb += 8) {
            uint32_t a[8];
#pragma unroll
            for (int k = 0; k < 8; k++)
                a[k] = col[(hb + k) * kRow];
#pragma unroll
            for (int k = 0; k < 8; k++)
                c += a[k];
        }
        for (; hb < r1; hb++)
            c += col[hb * kRow];
    } else {
        uint32_t hb = h0 + g;
        for (; hb + 3 * kScanGroups < h1; hb += 4 * kScanGroups) {
            const uint32_t a0 = col[hb * kRow], a1 = col[(hb + kScanGroups) * kRow];
            const uint32_t a2 = col[(hb + 2 * kScanGroups) * kRow], a3 = col[(hb + 3 * kScanGroups) * kRow];
            c += (a0 + a1) + (a2 + a3);
        }
        for (; hb < h1; hb += kScanGroups)
            c += col[hb * kRow];
    }
    part[g][dg] = c;
    __syncthreads();
    if (prefix) {  // each group rewrites its own quarter: counts -> exclusive prefixes
        uint32_t run = 0;
        for (int gi = 0; gi < g; gi++)
            run += part[gi][dg];
        uint32_t hb = r0;
        for (; hb + 8 <= r1; hb += 8) {
            uint32_t v[8];
#pragma unroll
            for (int k = 0; k < 8; k++)
                v[k] = col[(hb + k) * kRow];
#pragma unroll
            for (int k = 0; k < 8; k++) {
                col[(hb + k) * kRow] = run;
                run += v[k];
            }
        }
        for (; hb < r1; hb++) {
            const uint32_t v = col[hb * kRow];
            col[hb * kRow] = run;
            run += v;
        }
    }
    if (tid >= kRadix)
        return;
    c = 0;
#pragma unroll
    for (int gi = 0; gi < kScanGroups; gi++)
        c += part[gi][dg];
    if (p == msd_row && c > (uint32_t)kTile)
        atomicExch(w.msd_state, kMsdOverflow);
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += x;
    }
    if (lane == 31)
        wsum[warp] = incl;
    // named barrier over the first kRadix threads only (the rest have left)
    asm volatile("bar.sync 1, %0;" ::"n"(kRadix));
    uint32_t before = 0;
    for (int wi = 0; wi < warp; wi++)
        before += wsum[wi];
    w.counts[((size_t)p * T + t) * kRadix + dg] = w.tstart[t] + before + incl - c;
}

// Look-back words: kind in the high half (0 = not yet written), count in the
// low half.  Each word is written whole, so a reader sees a kind with its own
// count and needs no other ordering.
constexpr uint32_t kAggregate = 1u;  // the tile's own count of the digit
constexpr uint32_t kInclusive = 2u;  // count of the digit in this and all earlier tiles of the table
constexpr int kSpinLimit = 1 << 20;  // default polls of one word before a wait gives up (about a second)
constexpr int kFewDigits = 16;       // distinct digits among a warp's items below which a match is cheaper

__device__ __forceinline__ void store_status(uint64_t *p, uint32_t kind, uint32_t count)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(((uint64_t)kind << 32) | count) : "memory");
}

__device__ __forceinline__ uint64_t load_status(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// One radix pass in a single launch.  Tiles are taken in order from a
// counter, so every tile before a CTA's own is held by a CTA that is running
// or done; the CTA ranks its keys in shared memory, publishes its digit
// counts, sums the counts of the tiles before it in the same table (decoupled
// look-back), and scatters its keys, in stable order, to the digit ranges
// found by the histogram kernel.  The first pass needs no look-back: its
// tiles hold the keys in the order the histogram kernel counted them, and the
// digit scan has turned those counts into each tile's offsets.  A wait that runs out raises
// DLRM_FLAG_WAIT_TIMEOUT and writes stay inside the table's range.
// The first pass (pass 0, which reads the indices) sorts by the top 8 row
// bits when the MSD sort is planned and no bucket is too large (`msd_d`), by
// the lowest digit otherwise (`lsd_d`); the later LSD passes leave at once
// after an MSD pass.  A digit names its shift and width, the tile counter and
// the row of digit counts it uses.
struct PassDigit {
    int shift, nbits, ctr, crow;
};
constexpr int kRoleFirst = 1, kRoleLsd = 0;
__global__ void __launch_bounds__(kSortThreads, 4)
sort_onesweep_kernel(int pass, PassDigit lsd_d, PassDigit msd_d, int role, const int64_t *__restrict__ indices,
                     TableSet ts, int T, BwdPtrs w, int spin_limit, int32_t *err)
{
    __shared__ uint32_t skey[kTile];
    __shared__ uint32_t sval[kTile];
    __shared__ uint32_t whist[8][kRadix];
    __shared__ uint32_t tdig[kRadix];  // exclusive prefix of the tile's digit counts
    __shared__ uint32_t gbase[kRadix];
    __shared__ uint32_t wsum[8];
    __shared__ uint16_t srank[kItems][kSortThreads];  // each key's rank among its warp's keys of its digit
    __shared__ TileInfo ti;
    __shared__ uint32_t tau_s;
    __shared__ int timed_out;
    const bool msd = *w.msd_state == kMsdPlanned;
    if (role == kRoleLsd && msd)
        return;
    const PassDigit pd = role == kRoleFirst && msd ? msd_d : lsd_d;
    const int shift = pd.shift, nbits = pd.nbits, ctr = pd.ctr, crow = pd.crow;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 32) {
        uint32_t tau = 0;
        if (lane == 0)
            tau = atomicAdd(&w.tile_ctr[ctr], 1u);
        tau = __shfl_sync(0xffffffffu, tau, 0);
        find_tile_warp(tau, T, w.tile_base, w.tstart, ti);
        if (lane == 0) {
            tau_s = tau;
            timed_out = 0;
        }
    }
    for (int i = tid; i < 8 * kRadix; i += kSortThreads)
        (&whist[0][0])[i] = 0;
    __syncthreads();
    if (!ti.valid)
        return;
    const uint32_t tau = tau_s;
    // the next pass reuses the other buffer of look-back words: clear this tile's
    // (pass 1's were cleared by the histogram kernel, for every tile)
    if (pass != 0)
        w.status[(pass + 1) & 1][(size_t)tau * kRadix + tid] = 0;
    const uint32_t mask = (1u << nbits) - 1u;
    const int radix = 1 << nbits;
    const bool first_vals_bags = pass == 0 && *w.vals_bags != 0u;  // the first pass's values: bags or positions
    const uint32_t *keys_in = w.keys[(pass + 1) & 1];
    const uint32_t *vals_in = w.vals[(pass + 1) & 1];
    uint32_t *keys_out = w.keys[pass & 1];
    uint32_t *vals_out = w.vals[pass & 1];
    const int64_t R = ts.rows[ti.t];

    uint32_t key[kItems];  // values are read at the local scatter
    const uint32_t wbase = ti.lo + warp * (kTile / 8);
#pragma unroll
    for (int i = 0; i < kItems; i++) {
        const uint32_t j = wbase + i * 32 + lane;
        const bool valid = j < ti.hi;
        if (pass == 0)
            key[i] = valid ? pass0_key(indices, j, R) : 0u;
        else
            key[i] = valid ? keys_in[j] : 0u;
    }
    // stable rank within the warp: items in position order (i, then lane)
    bool few = false;
#pragma unroll
    for (int i = 0; i < kItems; i++) {
        const uint32_t j = wbase + i * 32 + lane;
        const bool valid = j < ti.hi;
        const uint32_t digit = valid ? (key[i] >> shift) & mask : (uint32_t)kRadix;
        // lanes with the same digit: a match instruction, whose cost grows with the number
        // of distinct digits among the lanes, while the previous item had few of them, else
        // one ballot per digit bit (a constant cost; the lanes past the end of a table's
        // last tile match none of the others)
        unsigned peers;
        if (few) {
            peers = __match_any_sync(0xffffffffu, digit);
        } else {
            peers = __ballot_sync(0xffffffffu, valid);
            if (!valid)
                peers = ~peers;
#pragma unroll
            for (int b = 0; b < kRadixBits; b++) {
                const bool bit = (digit >> b) & 1u;
                const unsigned m = __ballot_sync(0xffffffffu, bit);
                peers &= bit ? m : ~m;
            }
        }
        few = __popc(__ballot_sync(0xffffffffu, lane == __ffs(peers) - 1)) <= kFewDigits;
        const uint32_t before = __popc(peers & ((1u << lane) - 1u));
        uint32_t r = 0;
        if (valid)
            r = whist[warp][digit] + before;
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1)
            whist[warp][digit] += __popc(peers);
        __syncwarp();
        srank[i][tid] = (uint16_t)r;
    }
    __syncthreads();
    // per digit: exclusive prefix across warps and the tile's total
    uint32_t total = 0;
    if (tid < radix) {
        for (int wi = 0; wi < 8; wi++) {
            const uint32_t c = whist[wi][tid];
            whist[wi][tid] = total;
            total += c;
        }
    }
    const uint32_t t0 = w.tile_base[ti.t];  // the table's first tile
    const bool first = tau == t0;
    // the first pass reads its tile's offsets from the digit scan; the later ones look back
    const bool look_back = pass != 0;
    uint64_t *stat = w.status[pass & 1];
    if (look_back && tid < radix)
        store_status(stat + (size_t)tau * kRadix + tid, first ? kInclusive : kAggregate, total);
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
            const uint32_t lp = tdig[digit] + whist[warp][digit] + srank[i][tid];
            skey[lp] = key[i];
            sval[lp] = pass == 0 ? (first_vals_bags ? w.bag_of[j] : j) : vals_in[j];
        }
    }
    // the first pass: the digit scan's prefix of this tile.  Later passes
    // look back over the tiles before this one in the table (after the local
    // scatter, so that they have had the longest time to publish): the words
    // of up to 4 tiles k, k - 1, .. (none before the table's first) are read
    // at once and taken in order, down to an inclusive count; a word not yet
    // written is read again, with those before it
    if (tid < radix) {
        uint32_t excl = 0;
        if (!look_back) {
            excl = w.tile_hist[((size_t)tau * kSortRows + crow) * kRadix + tid];
        } else if (!first) {
            uint32_t k = tau - 1;
            int spins = 0;
            for (;;) {
                const uint32_t m = k - t0 + 1 < 4u ? k - t0 + 1 : 4u;
                uint64_t v[4];
#pragma unroll
                for (int q = 0; q < 4; q++)
                    v[q] = (uint32_t)q < m ? load_status(stat + (size_t)(k - q) * kRadix + tid) : 0ull;
                bool done = false, stalled = false;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    if (done || stalled || (uint32_t)q >= m)
                        continue;
                    const uint32_t kind = (uint32_t)(v[q] >> 32);
                    if (kind == 0u) {
                        stalled = true;
                        continue;
                    }
                    excl += (uint32_t)v[q];
                    if (kind == kInclusive || k == t0)
                        done = true;
                    else
                        k--;
                }
                if (done)
                    break;
                if (stalled && ++spins > spin_limit) {
                    timed_out = 1;
                    break;
                }
            }
            store_status(stat + (size_t)tau * kRadix + tid, kInclusive, excl + total);
        }
        gbase[tid] = w.counts[((size_t)crow * T + ti.t) * kRadix + tid] + excl;
    }
    __syncthreads();
    if (tid == 0 && timed_out) {
        raise_flag(err, DLRM_FLAG_WAIT_TIMEOUT);
        atomicOr(w.sort_failed, 1u);
    }
    const uint32_t n = ti.hi - ti.lo;
    const uint32_t tbeg = w.tstart[ti.t], tlen = w.tstart[ti.t + 1] - tbeg;
    for (uint32_t j = tid; j < n; j += kSortThreads) {
        const uint32_t k = skey[j];
        const uint32_t digit = (k >> shift) & mask;
        const uint32_t dest = gbase[digit] + (j - tdig[digit]);
        if (dest - tbeg < tlen) {
            keys_out[dest] = k;
            vals_out[dest] = sval[j];
        }
    }
}

// ------------------------------------------------------- bucket sort ---

// After the pass on the top 8 row bits a table's keys lie in 256 buckets, each
// in position order.  One CTA per (table, bucket) sorts the bucket's keys by
// the remaining `lbits` low bits in shared memory, stably (LSD passes of at
// most 9 bits: ranks within each warp's run of positions from ballots over the
// digit bits, then a scan over digits and warps), and writes them to the
// buffer the LSD passes would have ended in: the result is the full stable
// sort.  The digit scan has checked that no bucket holds more than kTile keys
// (else the first pass sorted by the lowest digit and this kernel does
// nothing); a bucket's size is its count from that scan, so a larger one
// means counts that disagree with the keys: the sort is then marked failed
// (nothing is updated) and DLRM_FLAG_BAD_OFFSETS raised.
constexpr int kBucketThreads = 256;  // 8 warps, at most 16 keys per thread
constexpr int kBucketBits = 9;       // widest digit of the local passes
constexpr int kBucketRadix = 1 << kBucketBits;
__global__ void __launch_bounds__(kBucketThreads, 4)
bucket_sort_kernel(int lbits, int lpasses, int crow, int out_buf, int T, BwdPtrs w, int32_t *err)
{
    __shared__ uint32_t skey[kTile];
    __shared__ uint32_t sval[kTile];
    __shared__ uint16_t whist[8][kBucketRadix];  // per warp and digit: count, then exclusive prefix (<= kTile)
    __shared__ uint32_t tdig[kBucketRadix];
    __shared__ uint32_t wsum[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the MSD pass gave up a wait (its order is invalid, and so the result), or did not run
    if (*w.sort_failed || *w.msd_state != kMsdPlanned)
        return;
    const int t = blockIdx.x / kRadix, v = blockIdx.x % kRadix;
    const uint32_t *cnt = w.counts + ((size_t)crow * T + t) * kRadix;
    const uint32_t s = cnt[v], e = v + 1 < kRadix ? cnt[v + 1] : w.tstart[t + 1];
    const uint32_t n = e - s;
    if (n == 0)
        return;
    if (n > (uint32_t)kTile) {
        if (tid == 0) {
            atomicOr(w.sort_failed, 1u);
            raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
        }
        return;
    }
    // warp `warp` holds positions warp*span .. +span, item i at warp*span + 32 i + lane
    const int nit = (int)((n + 8 * 32 - 1) / (8 * 32));  // items per thread, 1 .. 16
    const uint32_t wb = (uint32_t)warp * (uint32_t)nit * 32u;
    const uint32_t *kin = w.keys[0] + s, *vin = w.vals[0] + s;
    uint32_t key[kItems], val[kItems];
#pragma unroll
    for (int i = 0; i < kItems; i++) {
        const uint32_t j = wb + i * 32 + lane;
        key[i] = 0u;
        val[i] = 0u;
        if (i < nit && j < n) {
            key[i] = kin[j];
            val[i] = vin[j];
        }
    }
    int shift = 0;
    for (int p = 0; p < lpasses; p++) {
        const int nb = pass_bits(lbits, lpasses, p);
        const uint32_t mask = (1u << nb) - 1u;
        const int radix = 1 << nb;
        for (int i = tid; i < 8 * kBucketRadix / 2; i += kBucketThreads)
            reinterpret_cast<uint32_t *>(&whist[0][0])[i] = 0u;
        __syncthreads();
        uint32_t rank[kItems];
#pragma unroll
        for (int i = 0; i < kItems; i++) {
            rank[i] = 0u;
            if (i < nit) {  // uniform over the block
                const bool valid = wb + i * 32 + lane < n;
                const uint32_t digit = valid ? (key[i] >> shift) & mask : 0xffffffffu;
                unsigned peers = __ballot_sync(0xffffffffu, valid);
                if (!valid)
                    peers = ~peers;
                for (int b = 0; b < nb; b++) {  // a loop: unrolled and predicated it ran 35 % slower
                    const bool bit = (digit >> b) & 1u;
                    const unsigned m = __ballot_sync(0xffffffffu, bit);
                    peers &= bit ? m : ~m;
                }
                if (valid)
                    rank[i] = whist[warp][digit] + __popc(peers & ((1u << lane) - 1u));
                __syncwarp();
                if (valid && lane == __ffs(peers) - 1)
                    whist[warp][digit] = (uint16_t)(whist[warp][digit] + __popc(peers));
                __syncwarp();
            }
        }
        __syncthreads();
        // digits 2 tid and 2 tid + 1: exclusive prefix over the warps and the
        // digits' totals; then the exclusive scan of the totals over the digits
        uint32_t tot[2] = {0u, 0u};
#pragma unroll
        for (int k = 0; k < 2; k++) {
            const int dg = 2 * tid + k;
            if (dg < radix) {
                for (int wi = 0; wi < 8; wi++) {
                    const uint32_t c = whist[wi][dg];
                    whist[wi][dg] = (uint16_t)tot[k];
                    tot[k] += c;
                }
            }
        }
        const uint32_t mine = tot[0] + tot[1];
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += x;
        }
        if (lane == 31)
            wsum[warp] = incl;
        __syncthreads();
        uint32_t before = incl - mine;
        for (int wi = 0; wi < warp; wi++)
            before += wsum[wi];
        if (2 * tid < radix)
            tdig[2 * tid] = before;
        if (2 * tid + 1 < radix)
            tdig[2 * tid + 1] = before + tot[0];
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kItems; i++) {
            if (i < nit && wb + i * 32 + lane < n) {
                const uint32_t digit = (key[i] >> shift) & mask;
                const uint32_t dest = tdig[digit] + whist[warp][digit] + rank[i];
                skey[dest] = key[i];
                sval[dest] = val[i];
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kItems; i++) {
            const uint32_t j = wb + i * 32 + lane;
            if (i < nit && j < n) {
                key[i] = skey[j];
                val[i] = sval[j];
            }
        }
        __syncthreads();  // before the next pass clears the counts and overwrites the keys
        shift += nb;
    }
    uint32_t *kout = w.keys[out_buf] + s, *vout = w.vals[out_buf] + s;
#pragma unroll
    for (int i = 0; i < kItems; i++) {
        const uint32_t j = wb + i * 32 + lane;
        if (i < nit && j < n) {
            kout[j] = key[i];
            vout[j] = val[i];
        }
    }
}

// ------------------------------------------------------ segment count ---

// Number of run starts in each tile (the reduce numbers the runs of a tile
// from the exclusive scan of these counts).
__global__ void __launch_bounds__(256)
seg_count_kernel(int T, int final_buf, BwdPtrs w)
{
    __shared__ TileInfo ti;
    __shared__ uint32_t wc[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 32)
        find_tile_warp(blockIdx.x, T, w.tile_base, w.tstart, ti);
    __syncthreads();
    if (!ti.valid)
        return;
    const uint32_t *skey = w.keys[final_buf];
    const uint32_t ts = w.tstart[ti.t];
    // a sorted position starts a run when it is its table's first or its row differs from
    // the previous sorted row; all of the thread's keys are in flight at once, and a key's
    // predecessor comes from the lane before (lane 0 reads its own)
    constexpr int PER = kTile / 256;
    uint32_t k[PER], kp[PER];
#pragma unroll
    for (int i = 0; i < PER; i++) {
        const uint32_t j = ti.lo + (uint32_t)i * 256 + tid;
        const bool in = j < ti.hi;
        k[i] = in ? skey[j] : 0u;
        kp[i] = (in && lane == 0 && j != ts) ? skey[j - 1] : 0u;
    }
    uint32_t count = 0;
#pragma unroll
    for (int i = 0; i < PER; i++) {
        const uint32_t j = ti.lo + (uint32_t)i * 256 + tid;
        const uint32_t up = __shfl_up_sync(0xffffffffu, k[i], 1);
        const uint32_t prev = lane == 0 ? kp[i] : up;
        const bool start = j < ti.hi && (j == ts || k[i] != prev);
        count += __popc(__ballot_sync(0xffffffffu, start));
    }
    if (lane == 0)
        wc[warp] = count;
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
        *w.ids_ready = 1;
    }
}

// ---------------------------------------------------------------- host ---

static int row_bits(const int64_t *rows, int T)
{
    int64_t maxr = 1;
    for (int t = 0; t < T; t++)
        maxr = rows[t] > maxr ? rows[t] : maxr;
    int bits = 1;
    while (bits < 32 && ((int64_t)1 << bits) < maxr)
        bits++;
    return bits;
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

// Device pointers of the workspace's regions.
static BwdPtrs bind_workspace(int T, int64_t nnz, int d, void *workspace)
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
    w.status[0] = reinterpret_cast<uint64_t *>(base + L.status[0]);
    w.status[1] = reinterpret_cast<uint64_t *>(base + L.status[1]);
    w.tile_ctr = reinterpret_cast<uint32_t *>(base + L.tile_ctr);
    w.sort_failed = w.tile_ctr + kMaxPasses + 1;
    w.vals_bags = w.tile_ctr + kMaxPasses + 2;
    w.ids_ready = w.tile_ctr + kMaxPasses + 3;
    w.msd_state = w.tile_ctr + kMaxPasses + 4;
    w.tile_hist = reinterpret_cast<uint32_t *>(base + L.tile_hist);
    w.counts = reinterpret_cast<uint32_t *>(base + L.counts);
    w.tstart = reinterpret_cast<uint32_t *>(base + L.tstart);
    w.tile_base = reinterpret_cast<uint32_t *>(base + L.tile_base);
    w.tile_count = reinterpret_cast<uint32_t *>(base + L.tile_count);
    w.tile_ubase = reinterpret_cast<uint32_t *>(base + L.tile_ubase);
    w.chunk_flags = reinterpret_cast<uint32_t *>(base + L.chunk_flags);
    w.chunk_tail_u = reinterpret_cast<uint32_t *>(base + L.chunk_tail_u);
    w.chunk_tail_row = reinterpret_cast<uint32_t *>(base + L.chunk_tail_row);
    w.chunk_tail_t = reinterpret_cast<int32_t *>(base + L.chunk_tail_t);
    w.head = reinterpret_cast<float *>(base + L.head);
    w.tail = reinterpret_cast<float *>(base + L.tail);
    w.block_flags = reinterpret_cast<uint32_t *>(base + L.block_flags);
    w.block_sum = reinterpret_cast<float *>(base + L.block_sum);
    w.num_unique = reinterpret_cast<int64_t *>(base + L.num_unique);
    w.ntiles_max = L.ntiles_max;

    return w;
}

// Passes of the radix sort for these tables and the buffer that ends up
// holding the sorted keys (both halves of the backward derive them alike).
static void sort_plan(const TableSet &ts, int T, int &bits, int &passes, int &final_buf)
{
    bits = row_bits(ts.rows, T);
    passes = (bits + kRadixBits - 1) / kRadixBits;
    final_buf = (passes - 1) & 1;
}

// Whether the coalescing sorts by the top 8 row bits first and then each
// bucket in shared memory, one pass over all keys instead of three or four:
// for rows of 17 bits or more, every table above half the largest power of
// two (so that its keys spread over the buckets) and buckets of 256 to 2560
// keys on average (the shape of uniform lookups into large tables).  Lookups
// skewed enough that a bucket outgrows a tile fall back to the LSD passes on
// the device.
constexpr int64_t kMsdMinAvg = 256, kMsdMaxAvg = 2560;
static bool use_msd(const int64_t *rows, int bits, int T, int64_t nnz)
{
    const int64_t buckets = (int64_t)T * kRadix;
    if (bits < 17 || nnz < buckets * kMsdMinAvg || nnz > buckets * kMsdMaxAvg)
        return false;
    for (int t = 0; t < T; t++)
        if (rows[t] <= ((int64_t)1 << (bits - 1)))
            return false;
    return true;
}

void coalesce_plan(const int64_t *rows, int T, int64_t nnz, int &passes, bool &msd)
{
    const int bits = row_bits(rows, T);
    passes = (bits + kRadixBits - 1) / kRadixBits;
    msd = use_msd(rows, bits, T, nnz);
}

// Numbers the unique keys of a coalescing (their runs' starts counted per
// tile, then scanned): the view's arrays and the gradient rows are indexed by
// these numbers; the update itself does not need them.
static int launch_number_keys(int T, int64_t nnz, int final_buf, int64_t grid, BwdPtrs w, cudaStream_t st)
{
    seg_count_kernel<<<(unsigned)grid, 256, 0, st>>>(T, final_buf, w);
    count_launch(st);
    int s = launch_status();
    if (s != DLRM_OK)
        return s;
    seg_scan_kernel<<<1, 1024, 0, st>>>(T, nnz, w);
    count_launch(st);
    return launch_status();
}

int launch_coalesce(const TableSet &ts, int T, int d, const int64_t *offsets, const int64_t *indices,
                    int64_t nnz, int64_t B, void *workspace, dlrm_coalesced_view *view, int32_t *err,
                    cudaStream_t st)
{
    const BwdLayout L = bwd_layout(T, nnz, d);
    BwdPtrs w = bind_workspace(T, nnz, d, workspace);
    int bits, passes, final_buf;
    sort_plan(ts, T, bits, passes, final_buf);
    if (view) {
        view->sorted_pos = w.vals[final_buf];
        view->sorted_row = w.keys[final_buf];
        view->uniq_table = w.uniq_table;
        view->uniq_row = w.uniq_row;
        view->seg_off = w.seg_off;
        view->num_unique = w.num_unique;
    }

    const WaitHooks hooks = wait_hooks(kSpinLimit, 0);
    int s;
    // without a view the sort carries each lookup's bag (read in position order in the first pass),
    // so the reduce need not gather it by position; the view keeps the positions
    const uint32_t vals_bags = view ? 0u : 1u;
    const bool msd = use_msd(ts.rows, bits, T, nnz);
    bwd_prep_kernel<<<1, 256, 0, st>>>(offsets, T, B, nnz, w, hooks.sort_first_tile, vals_bags, msd ? 1u : 0u,
                                       err);
    count_launch(st);
    if ((s = launch_status()) != DLRM_OK)
        return s;
    if (nnz == 0) {
        cudaMemsetAsync(w.seg_off, 0, 4, st);
        return launch_status();
    }
    {
        const int64_t nbags = (int64_t)T * B;
        int64_t grid = (nbags + 255) / 256;  // 8 warps of 32 bags per block
        const int64_t cap = (int64_t)sm_count() * 8;
        bag_ids_kernel<<<(unsigned)(grid < cap ? grid : cap), 256, 0, st>>>(offsets, T, B, nnz, w.bag_of, err);
        count_launch(st);
        if ((s = launch_status()) != DLRM_OK)
            return s;
    }
    const int64_t grid = L.ntiles_max;
    const int lbits = bits - kRadixBits;  // below the MSD digit
    sort_hist_kernel<<<(unsigned)grid, 2 * kSortThreads, 0, st>>>(bits, passes, msd ? lbits : -1, indices, ts, T,
                                                                   w, err);
    count_launch(st);
    if ((s = launch_status()) != DLRM_OK)
        return s;
    const int rows = passes + (msd ? 1 : 0);  // the MSD digit's counts are row `passes`
    const unsigned prefix_rows = 1u | (msd ? 1u << passes : 0u);  // the rows the first pass may sort by
    sort_digit_scan_kernel<<<(unsigned)(rows * T), kScanGroups * kRadix, 0, st>>>(msd ? passes : -1, prefix_rows,
                                                                                   T, w);
    count_launch(st);
    if ((s = launch_status()) != DLRM_OK)
        return s;
    // with the MSD sort: the first launch sorts by the top digit (unless the digit scan found a
    // bucket too large), the bucket sort follows, and the later LSD passes leave at once
    const PassDigit msd_d{lbits, kRadixBits, kMaxPasses, passes};
    int shift = 0;
    for (int p = 0; p < passes; p++) {
        const int nb = pass_bits(bits, passes, p);
        const PassDigit lsd_d{shift, nb, p, p};
        sort_onesweep_kernel<<<(unsigned)grid, kSortThreads, 0, st>>>(p, lsd_d, msd_d, p == 0 ? kRoleFirst : kRoleLsd,
                                                                      indices, ts, T, w, hooks.sort_polls, err);
        count_launch(st);
        if ((s = launch_status()) != DLRM_OK)
            return s;
        if (p == 0 && msd) {
            bucket_sort_kernel<<<(unsigned)(T * kRadix), kBucketThreads, 0, st>>>(
                lbits, (lbits + kBucketBits - 1) / kBucketBits, passes, final_buf, T, w, err);
            count_launch(st);
            if ((s = launch_status()) != DLRM_OK)
                return s;
        }
        shift += nb;
    }
    if (!view)  // the unique keys are numbered for a view, or by the reduce for gradient rows
        return DLRM_OK;
    return launch_number_keys(T, nnz, final_buf, grid, w, st);
}

int launch_reduce_sgd(const TableSet &ts, int T, int d, int dtype, int64_t nnz, int64_t B, const float *dpooled,
                      int64_t dpss, int64_t dpts, float lr, float *grad_rows, int64_t grad_cap, void *workspace,
                      bool vec, int32_t *err, cudaStream_t st, float eps, float *const *state)
{
    if (nnz == 0)
        return DLRM_OK;
    const BwdLayout L = bwd_layout(T, nnz, d);
    BwdPtrs w = bind_workspace(T, nnz, d, workspace);
    int bits, passes, final_buf;
    sort_plan(ts, T, bits, passes, final_buf);
    if (grad_rows) {  // gradient rows are indexed by the unique keys' numbers
        const int s = launch_number_keys(T, nnz, final_buf, L.ntiles_max, w, st);
        if (s != DLRM_OK)
            return s;
    }
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
    a.opt = state ? kOptAdagrad : kOptSgd;
    a.eps = eps;
    std::memset(&a.state, 0, sizeof a.state);
    if (state)
        for (int t = 0; t < T; t++)
            a.state.ptr[t] = state[t];
    return launch_seg_reduce(dtype, a, w, L.ntiles_max, vec, st);
}

int launch_emb_bag_bwd(const TableSet &ts, int T, int d, int dtype, const int64_t *offsets,
                       const int64_t *indices, int64_t nnz, int64_t B, const float *dpooled,
                       int64_t dpss, int64_t dpts, float lr, float *grad_rows, int64_t grad_cap,
                       void *workspace, bool vec, dlrm_coalesced_view *view, int32_t *err,
                       cudaStream_t st)
{
    const int s = launch_coalesce(ts, T, d, offsets, indices, nnz, B, workspace, view, err, st);
    if (s != DLRM_OK)
        return s;
    return launch_reduce_sgd(ts, T, d, dtype, nnz, B, dpooled, dpss, dpts, lr, grad_rows, grad_cap, workspace,
                             vec, err, st, 0.f, nullptr);
}

}  // namespace dlrm
