// Shared pieces of the interaction kernels (interact.cu, emb_bag_interact.cu).
#pragma once

#include "common.cuh"

namespace dlrm {

constexpr int kKC = 32;  // columns of Z per shared-memory chunk

// Bits of the interaction mode: self pairs; the original embeddings
// concatenated alongside, [e0 | e_1 .. e_N | pairs] (else [e0 | pairs]).
constexpr int kInteractSelf = 1, kInteractAlongside = 2;

// Output position of the pair (i, j), j < i (strict) or j <= i (self pairs):
// rows of the lower triangle in order, i ascending, then j ascending.
__device__ __forceinline__ int64_t pair_pos(int i, int j, int inc)
{
    return inc ? (int64_t)i * (i + 1) / 2 + j : (int64_t)i * (i - 1) / 2 + j;
}

// Position of element (k, i) in a staged row of TS columns (TS a multiple
// of 32): 4-column groups are XOR-swizzled by bits 3..4 of k, so the
// transposing stores of 8 rows x 4 column octets from one warp hit 32
// distinct banks, while 4 consecutive columns stay one aligned 16-byte word.
__device__ __forceinline__ int zt_col(int k, int i)
{
    return ((((i >> 2) ^ (((k >> 3) & 3) << 1))) << 2) | (i & 3);
}

// The lower-triangle 4 x 4 tiles (I, J), J <= I, of a row of nTR tiles, in
// row order: tile number idx -> (I, J), written to two byte tables.
__device__ __forceinline__ void fill_tile_tables(int ntiles, uint8_t *tileI, uint8_t *tileJ)
{
    for (int idx = threadIdx.x; idx < ntiles; idx += blockDim.x) {
        int I = 0;
        while ((I + 1) * (I + 2) / 2 <= idx)
            I++;
        tileI[idx] = (uint8_t)I;
        tileJ[idx] = (uint8_t)(idx - I * (I + 1) / 2);
    }
}

__host__ __device__ inline int64_t num_pairs_of(int F, int inc)
{
    return inc ? (int64_t)F * (F + 1) / 2 : (int64_t)F * (F - 1) / 2;
}

}  // namespace dlrm
