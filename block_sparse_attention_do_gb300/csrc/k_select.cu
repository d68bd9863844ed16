// k_select.cu -- the step that produces the index: the compressed keys'
// mean-pooling stand-in and the top-S selection from block scores (the
// scores themselves come from the tensor-core kernel in k_gtc.cu).
//
// NSA's selection (the pages take the index as given; plainest reading):
// block j of a sequence is complete at row t when (j + 1) * bs - 1 <= t; a
// row's index is its own block t / bs, then the S - 1 blocks other than it
// that are complete at t with the largest scores, in decreasing order of
// score (equal scores: the smaller block id first; NaN ranks as -infinity),
// then -1.
#include <math.h>

#include "launch.h"

namespace nsa {

namespace {

constexpr int kThreads = 256;

int grid_of(int64_t n, int per_block, int cap)
{
    int64_t b = (n + per_block - 1) / per_block;
    return (int)(b < 1 ? 1 : b > cap ? cap : b);
}

// 16-byte vectors of the element type (8 bf16 or 4 fp32), added into fp32 sums
template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void add(const uint4 &w, float *acc)
    {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] += __uint_as_float(u[i] << 16);
            acc[2 * i + 1] += __uint_as_float(u[i] & 0xffff0000u);
        }
    }
};
template <> struct Vec<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void add(const uint4 &w, float *acc)
    {
        acc[0] += __uint_as_float(w.x);
        acc[1] += __uint_as_float(w.y);
        acc[2] += __uint_as_float(w.z);
        acc[3] += __uint_as_float(w.w);
    }
};

// kc[b, g, j, :] = the mean of keys j*bs .. j*bs + bs - 1 of sequence b, kv
// head g, for blocks complete in the sequence; zero rows for the others.  One
// CTA per block: thread (group, v) sums 16-byte vector v of the rows group,
// group + groups, ... (all its loads in flight), then the groups' partial
// sums meet in shared memory.
template <typename T> __global__ void __launch_bounds__(kThreads) compress_mean_kernel(const Geo g, const T *k, T *kc)
{
    constexpr int N = Vec<T>::N;
    __shared__ float part[kThreads * N];
    const int nv = g.D / N, groups = kThreads / nv;  // nv divides kThreads (D / N is 4 .. 32)
    const int v = threadIdx.x % nv, grp = threadIdx.x / nv;
    const int nb = g.nbmax;
    const int64_t nrows = (int64_t)g.B * g.Hkv * nb;
    const float inv = 1.0f / (float)g.bs;  // bs is a power of two: exact
    for (int64_t row = blockIdx.x; row < nrows; row += gridDim.x) {  // row = (b * Hkv + kvh) * nb + j
        const int j = (int)(row % nb), bg = (int)(row / nb), b = bg / g.Hkv, kvh = bg % g.Hkv;
        const bool complete = (int64_t)(j + 1) * g.bs <= seq_len(g, b);
        float acc[N];
#pragma unroll
        for (int i = 0; i < N; ++i)
            acc[i] = 0.f;
        if (complete) {
#pragma unroll 4
            for (int i = grp; i < g.bs; i += groups)
                Vec<T>::add(__ldg((const uint4 *)(k + kv_off(g, b, kvh, j * g.bs + i) + v * N)), acc);
        }
#pragma unroll
        for (int i = 0; i < N; ++i)
            part[(grp * nv + v) * N + i] = acc[i];
        __syncthreads();
        if (threadIdx.x < g.D) {  // element d: vector d / N, lane d % N of it
            const int d = threadIdx.x;
            float sum = 0.f;
            for (int q = 0; q < groups; ++q)
                sum += part[(q * nv + d / N) * N + d % N];
            kc[row * g.D + d] = (T)(sum * inv);
        }
        __syncthreads();
    }
}

// The selection order as one unsigned key: a larger score gives a larger
// key; NaN counts as -infinity and -0 as +0 (they compare equal); every key
// is above 0, which stands for "no block".
__device__ __forceinline__ uint32_t order_key(float x)
{
    x = isnan(x) ? -INFINITY : x + 0.0f;  // -0 + 0 = +0
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp per index row R (the index's own row order: BHTD (b*Hkv + kvh)*T
// + t, THD token*Hkv + kvh; the scores use the same rows, nb = nbmax each).
// Round s takes the best complete block left (largest key, then smallest
// id): a warp max of the lanes' best keys and a warp min of the ids among
// the lanes holding that key.  Rows of up to 32 * REGS blocks keep their
// keys in registers (REGS per lane, block lane + 32 i; a taken block's key
// is cleared); REGS = 0 reads every round's keys from memory and takes the
// best block that ranks after the previous round's pick (a strict total
// order, so no block is taken twice).
template <int REGS> __global__ void __launch_bounds__(kThreads) select_topk_kernel(const Geo g, const float *scores, int *idx)
{
    constexpr int R = REGS > 0 ? REGS : 1;
    const int lane = threadIdx.x & 31;
    const int64_t nrows = (int64_t)g.ntok * g.Hkv;
    const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nb = g.nbmax, S = g.S;
    for (int64_t row = warp0; row < nrows; row += nwarps) {
        int t;
        if (g.thd) {
            const int tok = (int)(row / g.Hkv);
            int lo = 0, hi = g.B - 1;  // the sequence holding token tok: the last b with cu[b] <= tok
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (g.cu[mid] <= tok)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            t = tok - g.cu[lo];
        } else {
            t = (int)(row % g.T);
        }
        const float *sc = scores + row * nb;
        int *out = idx + row * S;
        const int own = t / g.bs, nc = (t + 1) / g.bs;
        uint32_t key[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int j = lane + 32 * i;
            key[i] = (REGS > 0 && j < nc && j != own) ? order_key(__ldg(sc + j)) : 0u;
        }
        if (lane == 0)
            out[0] = own;
        int filled = 1;
        if constexpr (REGS > 0) {
            // each lane's best remaining key (ids ascend with i, so the first
            // of equal keys -- the smallest id -- wins); only the lane whose
            // block was taken looks again
            uint32_t bk = 0u;
            int bj = 0x7fffffff;
            auto lane_best = [&]() {
                bk = 0u;
                bj = 0x7fffffff;
#pragma unroll
                for (int i = 0; i < R; ++i)
                    if (key[i] > bk) {
                        bk = key[i];
                        bj = lane + 32 * i;
                    }
            };
            lane_best();
            for (int s = 1; s < S; ++s) {
                const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
                if (wk == 0u)  // no complete block left (warp-uniform)
                    break;
                const int wj = (int)__reduce_min_sync(0xffffffffu, (unsigned)(bk == wk ? bj : 0x7fffffff));
                if (lane == 0)
                    out[s] = wj;
                filled = s + 1;
                if (lane == (wj & 31)) {
#pragma unroll
                    for (int i = 0; i < R; ++i)
                        if (i == (wj >> 5))
                            key[i] = 0u;
                    lane_best();
                }
            }
        } else {
            uint32_t pk = 0xffffffffu;  // the previous pick: above every key
            int pj = -1;
            for (int s = 1; s < S; ++s) {
                uint32_t bk = 0u;
                int bj = 0x7fffffff;
                for (int j = lane; j < nc; j += 32) {
                    if (j == own)
                        continue;
                    const uint32_t kk = order_key(__ldg(sc + j));
                    if (kk > bk && (kk < pk || (kk == pk && j > pj))) {
                        bk = kk;
                        bj = j;
                    }
                }
                const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
                if (wk == 0u)
                    break;
                const int wj = (int)__reduce_min_sync(0xffffffffu, (unsigned)(bk == wk ? bj : 0x7fffffff));
                if (lane == 0)
                    out[s] = wj;
                pk = wk;
                pj = wj;
                filled = s + 1;
            }
        }
        for (int s = filled + lane; s < S; s += 32)
            out[s] = -1;
    }
}

}  // namespace

cudaError_t launch_compress_mean(const Geo &g, const void *k, void *kc, int dtype, cudaStream_t st)
{
    const int grid = grid_of((int64_t)g.B * g.Hkv * g.nbmax, 1, 152 * 8);
    if (dtype == NSA_DTYPE_BF16)
        compress_mean_kernel<__nv_bfloat16>
            <<<grid, kThreads, 0, st>>>(g, (const __nv_bfloat16 *)k, (__nv_bfloat16 *)kc);
    else
        compress_mean_kernel<float><<<grid, kThreads, 0, st>>>(g, (const float *)k, (float *)kc);
    return cudaGetLastError();
}

cudaError_t launch_select_topk(const Geo &g, const float *scores, int *idx, cudaStream_t st)
{
    const int64_t rows = (int64_t)g.ntok * g.Hkv;
    const int grid = grid_of(rows, kThreads / 32, 152 * 16);
    // a row's complete blocks number at most nbmax: the smallest register set that holds them
    const int nb = g.nbmax;
    if (nb <= 32)
        select_topk_kernel<1><<<grid, kThreads, 0, st>>>(g, scores, idx);
    else if (nb <= 64)
        select_topk_kernel<2><<<grid, kThreads, 0, st>>>(g, scores, idx);
    else if (nb <= 128)
        select_topk_kernel<4><<<grid, kThreads, 0, st>>>(g, scores, idx);
    else if (nb <= 256)
        select_topk_kernel<8><<<grid, kThreads, 0, st>>>(g, scores, idx);
    else
        select_topk_kernel<0><<<grid, kThreads, 0, st>>>(g, scores, idx);
    return cudaGetLastError();
}

}  // namespace nsa
