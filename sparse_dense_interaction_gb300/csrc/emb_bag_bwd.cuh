// Shared definitions of the embedding-bag backward (coalescing sort, segmented
// reduce, row-wise SGD).
#pragma once

#include "common.cuh"

namespace dlrm {

constexpr int kTile = 4096;                   // sorted positions per tile
constexpr int kSortThreads = 256;             // 8 warps
constexpr int kItems = kTile / kSortThreads;  // 16 per thread
constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kMaxPasses = 4;                 // LSD passes of up to 8 bits over 32-bit rows
constexpr int kSortRows = kMaxPasses + 1;     // digit-count rows: the LSD passes' and the MSD digit's
constexpr uint32_t kMsdPlanned = 1u;          // sorted by the top 8 row bits, then per bucket
constexpr uint32_t kMsdOverflow = 2u;         // a bucket exceeded a tile: the LSD passes sort instead
constexpr uint32_t kSentinel = 0xffffffffu;   // sort key of an out-of-range index
constexpr uint32_t kHasHead = 1u, kHeadEnds = 2u, kHasTail = 4u;
constexpr int kReduceThreads = 256;           // 8 warps per tile in the reduce, one or two chunks each
constexpr int kFinalizeBlock = 32;            // chunks summed per block in the finalize's first level

// Reduce chunks per tile (the layout of the partial sums is sized for it):
// one per stream of 16 or 32 lanes.
inline int reduce_chunks_per_tile(int) { return (kReduceThreads / 32) * 2; }

struct BwdPtrs {
    uint32_t *keys[2], *vals[2], *bag_of, *uniq_row, *seg_off, *tile_ctr, *tile_hist, *counts, *tstart, *tile_base,
        *tile_count, *tile_ubase, *chunk_flags, *chunk_tail_u, *block_flags;
    uint32_t *sort_failed;  // set by a radix pass whose wait ran out: the reduce then updates nothing
    uint32_t *vals_bags;    // 1: the sort carried each lookup's bag (no view asked for); 0: its position
    uint32_t *ids_ready;    // 1: the unique keys are numbered (tile_ubase, num_unique): a view or gradient rows
    uint32_t *msd_state;    // kMsdPlanned: sorted by the top digit and per bucket; kMsdOverflow: LSD passes
    uint32_t *chunk_tail_row;  // row and table of the run that leaves each chunk (read by the finalize)
    int32_t *chunk_tail_t;
    int32_t *uniq_table;
    uint64_t *status[2];  // look-back words of the radix passes, by tile and digit
    float *head, *tail, *block_sum;
    int64_t *num_unique;
    int64_t ntiles_max;
};

struct TileInfo {
    int t;
    uint32_t lo, hi;
    int valid;
};

// Table and position range of tile tau (tiles never straddle a table).
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

// The same by the 32 lanes of one warp (all of them call it; lane 0 writes
// ti).  For fewer than 32 tables every lane loads one table's first tile and
// first position at once, and a ballot counts the tables that start at or
// before tau (the tile's table is the last of them): one round trip to
// memory instead of a binary search's chain of loads.
__device__ __forceinline__ void find_tile_warp(int64_t tau, int T, const uint32_t *tile_base,
                                               const uint32_t *tstart, TileInfo &ti)
{
    const int lane = threadIdx.x & 31;
    if (T >= 32) {
        if (lane == 0)
            find_tile(tau, T, tile_base, tstart, ti);
        return;
    }
    const uint32_t tb = lane <= T ? tile_base[lane] : 0xffffffffu;
    const uint32_t ts = lane <= T ? tstart[lane] : 0u;
    const int n = __popc(__ballot_sync(0xffffffffu, lane < T && (int64_t)tb <= tau));
    const int t = n > 0 ? n - 1 : 0;
    const uint32_t total = __shfl_sync(0xffffffffu, tb, T);
    const uint32_t tbt = __shfl_sync(0xffffffffu, tb, t);
    const uint32_t lo = __shfl_sync(0xffffffffu, ts, t);
    const uint32_t end = __shfl_sync(0xffffffffu, ts, t + 1);
    if (lane == 0) {
        if (tau >= (int64_t)total) {
            ti.valid = 0;
            return;
        }
        ti.t = t;
        ti.lo = lo + (uint32_t)(tau - tbt) * kTile;
        ti.hi = ti.lo + kTile < end ? ti.lo + kTile : end;
        ti.valid = 1;
    }
}

// Optimizers of the update: plain SGD, or row-wise AdaGrad (one fp32
// accumulator per row: s' = s + mean(g^2), w' = w - lr g / (sqrt(s') + eps)).
constexpr int kOptSgd = 0, kOptAdagrad = 1;
constexpr int kAdagradMaxD = 256;  // rows the AdaGrad update holds whole in registers

struct StateSet {
    float *ptr[DLRM_MAX_TABLES];  // accumulator of each row, per table (AdaGrad)
};

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
    int opt;        // kOptSgd or kOptAdagrad
    float eps;      // AdaGrad
    StateSet state; // AdaGrad
};

// Segmented reduce + SGD and the combine of cross-chunk runs (seg_reduce.cu).
int launch_seg_reduce(int dtype, const ReduceArgs &a, const BwdPtrs &w, int64_t grid, bool vec,
                      cudaStream_t st);

}  // namespace dlrm
