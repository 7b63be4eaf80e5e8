// Embedding-bag backward with row-wise SGD applied by atomic reductions, for
// fp32 tables, without coalescing the duplicate lookups first.
//
// The update is the one of "Notes/DLRM" (vault-aram.pages.dev), section 5
// (the tables are trained by an optimizer; plain SGD on the touched rows):
// every row receives -lr times the sum of the pooled gradients of the bags
// that looked it up.  Sum pooling (section 9: multi-valued features are
// aggregated) makes each lookup's share the gradient of its bag.
//
// Design: bags are walked in table-major order, a group of G lanes per bag
// (one 16-byte piece of the row per lane and pass).  The group reads the
// bag's pooled gradient once, scales it by -lr, then loads up to G of the
// bag's indices at a time; lookups of the same row among them are merged
// (the first lane of the row adds count x the scaled gradient) and each
// distinct row receives one vector reduction (red.global.add.v4.f32) per
// 16-byte piece, performed in L2.  Nothing waits on a table row, so the
// kernel streams: its traffic is the pooled gradients and indices once plus
// the reductions' read-modify-writes of the touched rows.
//
// Rows touched by several bags receive one reduction per bag in an
// unspecified order: the result is the update of the coalesced path up to the
// rounding of one fp32 add per reduction (not bit-reproducible from run to
// run).  The fp32 reductions flush subnormal inputs and results to zero.
#include "common.cuh"

namespace dlrm {

__device__ __forceinline__ void red_add(float *p, const float4 &v)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void red_add(float *p, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

__device__ __forceinline__ float4 scaled(const float4 &v, float s)
{
    return make_float4(s * v.x, s * v.y, s * v.z, s * v.w);
}
__device__ __forceinline__ float scaled(float v, float s) { return s * v; }

template <int VEC>
struct Piece;
template <>
struct Piece<4> {
    using F = float4;
    __device__ __forceinline__ static F zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ static F load(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
};
template <>
struct Piece<1> {
    using F = float;
    __device__ __forceinline__ static F zero() { return 0.f; }
    __device__ __forceinline__ static F load(const float *p) { return __ldg(p); }
};

// G lanes per bag, C pieces of VEC values per lane (piece c of lane l covers
// elements (c*G + l)*VEC ..); rows wider than C*G*VEC are taken in passes.
template <int G, int C, int VEC>
__global__ void __launch_bounds__(256)
emb_bag_bwd_atomic_kernel(TableSet ts, int T, int d, const int64_t *__restrict__ offsets,
                          const int64_t *__restrict__ indices, int64_t nnz, int64_t B,
                          const float *__restrict__ dpooled, int64_t dpss, int64_t dpts, float lr, int32_t *err)
{
    using P = Piece<VEC>;
    using F = typename P::F;
    constexpr int GPW = 32 / G;  // bags per warp
    constexpr int EB = C * G * VEC;
    const int lane = threadIdx.x & 31;
    const int gl = lane % G, grp = lane / G;
    const unsigned gmask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (grp * G));
    const int64_t nbags = (int64_t)T * B;
    const bool small = nbags <= 0xffffffffll;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const float step = -lr;

    for (int64_t bag = warp * GPW + grp; bag < nbags; bag += nwarps * GPW) {
        int t;
        int64_t b;
        bag_table_sample(bag, B, small, t, b);
        int64_t k0 = offsets[bag];
        int64_t k1 = offsets[bag + 1];
        if (k0 < 0 || k1 < k0 || k1 > nnz) {
            if (gl == 0)
                raise_flag(err, DLRM_FLAG_BAD_OFFSETS);
            continue;
        }
        if (k0 == k1)
            continue;
        float *tab = static_cast<float *>(const_cast<void *>(ts.ptr[t]));
        const int64_t R = ts.rows[t];
        const float *dp = dpooled + b * dpss + (int64_t)t * dpts;
        for (int eb = 0; eb < d; eb += EB) {
            F v[C];
#pragma unroll
            for (int c = 0; c < C; c++) {
                const int e = eb + (c * G + gl) * VEC;
                v[c] = e < d ? scaled(P::load(dp + e), step) : P::zero();
            }
            for (int64_t kb = k0; kb < k1; kb += G) {
                const int n = k1 - kb < G ? (int)(k1 - kb) : G;
                int64_t r = -1;
                if (gl < n) {
                    r = load_stream(indices + kb + gl);
                    if (r < 0 || r >= R) {
                        if (eb == 0)
                            raise_flag(err, DLRM_FLAG_INDEX_OOB);
                        r = -1;
                    }
                }
                // lookups of one row among these: the lowest lane adds them all
                const unsigned peers = __match_any_sync(gmask, r);
                const float cnt = (r >= 0 && __ffs(peers) - 1 == lane) ? (float)__popc(peers) : 0.f;
                for (int j = 0; j < n; j++) {
                    const float cj = __shfl_sync(gmask, cnt, grp * G + j);
                    const int64_t rj = __shfl_sync(gmask, r, grp * G + j);
                    if (cj == 0.f)
                        continue;
                    float *row = tab + rj * d;
#pragma unroll
                    for (int c = 0; c < C; c++) {
                        const int e = eb + (c * G + gl) * VEC;
                        if (e < d)
                            red_add(row + e, cj == 1.f ? v[c] : scaled(v[c], cj));
                    }
                }
            }
        }
    }
}

template <int G, int C, int VEC>
static int launch(const TableSet &ts, int T, int d, const int64_t *offsets, const int64_t *indices, int64_t nnz,
                  int64_t B, const float *dpooled, int64_t dpss, int64_t dpts, float lr, int32_t *err,
                  cudaStream_t st)
{
    const int64_t groups = (int64_t)T * B;
    int64_t grid = (groups + (256 / G) - 1) / (256 / G);
    const int64_t cap = (int64_t)sm_count() * 8;  // resident blocks of 256 threads
    if (grid > cap)
        grid = cap;
    emb_bag_bwd_atomic_kernel<G, C, VEC><<<(unsigned)grid, 256, 0, st>>>(ts, T, d, offsets, indices, nnz, B,
                                                                       dpooled, dpss, dpts, lr, err);
    count_launch(st);
    return launch_status();
}

int launch_emb_bag_bwd_atomic(const TableSet &ts, int T, int d, const int64_t *offsets, const int64_t *indices,
                              int64_t nnz, int64_t B, const float *dpooled, int64_t dpss, int64_t dpts, float lr,
                              bool vec, int32_t *err, cudaStream_t st)
{
    if (!vec)
        return launch<32, 1, 1>(ts, T, d, offsets, indices, nnz, B, dpooled, dpss, dpts, lr, err, st);
    // one 16-byte piece per lane and pass: groups of 8, 16 or 32 lanes
    if (d <= 32)
        return launch<8, 1, 4>(ts, T, d, offsets, indices, nnz, B, dpooled, dpss, dpts, lr, err, st);
    if (d <= 64)
        return launch<16, 1, 4>(ts, T, d, offsets, indices, nnz, B, dpooled, dpss, dpts, lr, err, st);
    if (d <= 128)
        return launch<32, 1, 4>(ts, T, d, offsets, indices, nnz, B, dpooled, dpss, dpts, lr, err, st);
    return launch<32, 2, 4>(ts, T, d, offsets, indices, nnz, B, dpooled, dpss, dpts, lr, err, st);
}

}  // namespace dlrm
