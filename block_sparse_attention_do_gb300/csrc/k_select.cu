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

// 16-byte vectors of the element type: 8 bf16 or 4 fp32
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
    static __device__ __forceinline__ uint4 pack(const float *x)
    {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            u[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        return make_uint4(u[0], u[1], u[2], u[3]);
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
    static __device__ __forceinline__ uint4 pack(const float *x)
    {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
};

// kc[b, g, j, :] = the mean of keys j*bs .. j*bs + bs - 1 of sequence b, kv
// head g, for blocks complete in the sequence; zero rows for the others.  One
// thread per 16-byte vector of kc (consecutive threads: consecutive vectors
// of a row, so a warp reads whole key rows).
template <typename T> __global__ void __launch_bounds__(kThreads) compress_mean_kernel(const Geo g, const T *k, T *kc)
{
    constexpr int N = Vec<T>::N;
    const int nv = g.D / N, nb = g.nbmax;
    const int64_t total = (int64_t)g.B * g.Hkv * nb * nv;
    const float inv = 1.0f / (float)g.bs;  // bs is a power of two: exact
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int v = (int)(e % nv);
        const int64_t row = e / nv;  // (b * Hkv + kvh) * nb + j
        const int j = (int)(row % nb), bg = (int)(row / nb), b = bg / g.Hkv, kvh = bg % g.Hkv;
        float acc[N];
#pragma unroll
        for (int i = 0; i < N; ++i)
            acc[i] = 0.f;
        if ((int64_t)(j + 1) * g.bs <= seq_len(g, b)) {
            for (int i = 0; i < g.bs; ++i)
                Vec<T>::add(__ldg((const uint4 *)(k + kv_off(g, b, kvh, j * g.bs + i) + v * N)), acc);
#pragma unroll
            for (int i = 0; i < N; ++i)
                acc[i] *= inv;
        }
        *(uint4 *)(kc + row * g.D + v * N) = Vec<T>::pack(acc);
    }
}

// (x, i) ranks before (y, j): larger score first, then smaller block id;
// NaN scores were mapped to -infinity by the caller
__device__ __forceinline__ bool ranks_before(float x, int i, float y, int j) { return x > y || (x == y && i < j); }

__device__ __forceinline__ float rank_key(float x) { return isnan(x) ? -INFINITY : x; }

// One warp per index row R (the index's own row order: BHTD (b*Hkv + kvh)*T
// + t, THD token*Hkv + kvh; the scores use the same rows, nb = nbmax each).
// Each of the S - 1 rounds takes the best complete block that ranks after
// the previous round's pick (a strict total order, so no block is taken
// twice): every lane scans its blocks j = lane, lane + 32, ..., then a
// butterfly of shuffles keeps the best.
__global__ void __launch_bounds__(kThreads) select_topk_kernel(const Geo g, const float *scores, int *idx)
{
    const int lane = threadIdx.x & 31;
    const int64_t nrows = (int64_t)g.ntok * g.Hkv;
    const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nb = g.nbmax, S = g.S;
    for (int64_t R = warp0; R < nrows; R += nwarps) {
        int t;
        if (g.thd) {
            const int tok = (int)(R / g.Hkv);
            int lo = 0, hi = g.B - 1;  // the sequence holding token tok: cu[lo] <= tok < cu[lo + 1]
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (g.cu[mid] <= tok)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            t = tok - g.cu[lo];
        } else {
            t = (int)(R % g.T);
        }
        const float *sc = scores + R * nb;
        int *out = idx + R * S;
        const int own = t / g.bs, nc = (t + 1) / g.bs;
        if (lane == 0)
            out[0] = own;
        float pv = INFINITY;  // the previous pick; (+inf, -1) ranks before every block
        int pj = -1, filled = 1;
        for (int s = 1; s < S; ++s) {
            float bv = -INFINITY;
            int bj = -1;
            for (int j = lane; j < nc; j += 32) {
                if (j == own)
                    continue;
                const float v = rank_key(__ldg(sc + j));
                if (ranks_before(pv, pj, v, j) && (bj < 0 || ranks_before(v, j, bv, bj))) {
                    bv = v;
                    bj = j;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oj = __shfl_xor_sync(0xffffffffu, bj, off);
                if (oj >= 0 && (bj < 0 || ranks_before(ov, oj, bv, bj))) {
                    bv = ov;
                    bj = oj;
                }
            }
            if (bj < 0)  // warp-uniform after the butterfly: no complete block left
                break;
            if (lane == 0)
                out[s] = bj;
            pv = bv;
            pj = bj;
            filled = s + 1;
        }
        for (int s = filled + lane; s < S; s += 32)
            out[s] = -1;
    }
}

}  // namespace

cudaError_t launch_compress_mean(const Geo &g, const void *k, void *kc, int dtype, cudaStream_t st)
{
    const int64_t total = (int64_t)g.B * g.Hkv * g.nbmax * (g.D / (dtype == NSA_DTYPE_BF16 ? 8 : 4));
    const int grid = grid_of(total, kThreads, 152 * 16);
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
    select_topk_kernel<<<grid, kThreads, 0, st>>>(g, scores, idx);
    return cudaGetLastError();
}

}  // namespace nsa
