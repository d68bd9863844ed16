// k_simt.cu -- CUDA-core (FFMA) kernels for every supported shape, fp32 or
// bf16 storage with fp32 arithmetic.  They carry the fp32 problems (the
// tensor-core path would round operands to bf16 or tf32 and miss the fp32
// gate) and the bf16 shapes the tensor-core kernels do not cover.
//
// One warp owns one output row (a query row for the forward and dQ, a key
// for dK/dV); lane l holds elements d = l + 32 i of the D-vector, so each
// dot product is a per-lane partial plus a warp butterfly reduction.
#include "launch.h"

namespace nsa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// decode a linear query-row number (lse order) into (b, h, t)
__device__ __forceinline__ void decode_qrow(const Geo &g, int64_t r, int &b, int &h, int &t)
{
    if (g.thd) {
        h = (int)(r % g.Hq);
        const int tok = (int)(r / g.Hq);
        b = seq_of_token(g, tok);
        t = tok - g.cu[b];
    } else {
        t = (int)(r % g.T);
        const int64_t bh = r / g.T;
        h = (int)(bh % g.Hq);
        b = (int)(bh / g.Hq);
    }
}

// decode a linear key-row number (k order) into (b, kvh, key)
__device__ __forceinline__ void decode_krow(const Geo &g, int64_t r, int &b, int &kvh, int &t)
{
    if (g.thd) {
        kvh = (int)(r % g.Hkv);
        const int tok = (int)(r / g.Hkv);
        b = seq_of_key(g, tok);
        t = tok - g.cuk[b];
    } else {
        t = (int)(r % g.Tk);
        const int64_t bh = r / g.Tk;
        kvh = (int)(bh % g.Hkv);
        b = (int)(bh / g.Hkv);
    }
}

// j-th selected block of a row, or -1.  Invalid entries (out of range, in
// the future) are skipped here and reported by the index validation.
__device__ __forceinline__ int slot_block(const Geo &g, const int *row, int s, int t)
{
    if (g.dense)
        return s;
    const int j = row[s];
    return (j >= 0 && j <= t / g.bs) ? j : -1;
}

// slots to walk for a row whose last attended key is `hi` (dense: blocks 0 .. hi / bs)
__device__ __forceinline__ int n_slots(const Geo &g, int hi) { return g.dense ? (hi >= 0 ? hi / g.bs + 1 : 0) : g.S; }

template <typename T, int DPL>
__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(Geo g, const T *__restrict__ q,
                                                            const T *__restrict__ k,
                                                            const T *__restrict__ v,
                                                            const int *__restrict__ idx,
                                                            T *__restrict__ o, float *__restrict__ lse)
{
    const int lane = threadIdx.x & 31;
    const int64_t nrows = (int64_t)g.ntok * g.Hq;
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < nrows;
         r += (int64_t)gridDim.x * kWarps) {
        int b, h, t;
        decode_qrow(g, r, b, h, t);
        const int kvh = h / g.G;
        const T *qp = q + q_off(g, b, h, t);
        float qv[DPL], acc[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            qv[i] = to_f(qp[lane + 32 * i]);
            acc[i] = 0.f;
        }
        float m = -INFINITY, l = 0.f;
        const int *row = g.dense ? nullptr : idx_row(g, idx, b, kvh, t);
        // keys klo .. khi: the window's left edge up to the diagonal (and the keys' end)
        const int c = kdiag(g, b, t), khi = min(c, seq_len_k(g, b) - 1);
        const int klo = key_lo(g, c);
        const int ns = n_slots(g, khi);
        for (int s = 0; s < ns; ++s) {
            const int j = slot_block(g, row, s, t);
            if (j < 0)
                continue;
            const int kend = min((j + 1) * g.bs, khi + 1);
            for (int kk = max(j * g.bs, klo); kk < kend; ++kk) {
                const int64_t ko = kv_off(g, b, kvh, kk);
                float part = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i)
                    part = fmaf(qv[i], to_f(k[ko + lane + 32 * i]), part);
                const float sc = warp_sum(part) * g.scale;
                const float mn = fmaxf(m, sc);
                const float corr = __expf(m - mn);  // 0 while m = -inf
                const float p = __expf(sc - mn);
                l = l * corr + p;
#pragma unroll
                for (int i = 0; i < DPL; ++i)
                    acc[i] = fmaf(p, to_f(v[ko + lane + 32 * i]), acc[i] * corr);
                m = mn;
            }
        }
        T *op = o + o_off(g, b, h, t);
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i)
            op[lane + 32 * i] = from_f<T>(acc[i] * inv);
        if (lane == 0)
            lse[stat_off(g, b, h, t)] = l > 0.f ? m + logf(l) : -INFINITY;
    }
}

template <typename T, int DPL>
__global__ void __launch_bounds__(kThreads) dq_simt_kernel(Geo g, const T *__restrict__ q,
                                                           const T *__restrict__ k,
                                                           const T *__restrict__ v,
                                                           const T *__restrict__ dO,
                                                           const float *__restrict__ lse,
                                                           const float *__restrict__ delta,
                                                           const int *__restrict__ idx,
                                                           T *__restrict__ dq)
{
    const int lane = threadIdx.x & 31;
    const int64_t nrows = (int64_t)g.ntok * g.Hq;
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < nrows;
         r += (int64_t)gridDim.x * kWarps) {
        int b, h, t;
        decode_qrow(g, r, b, h, t);
        const int kvh = h / g.G;
        const int64_t qo = q_off(g, b, h, t), oo = o_off(g, b, h, t);
        const int64_t so = stat_off(g, b, h, t);
        const float L = lse[so], Dt = delta[so];
        float qv[DPL], ov[DPL], acc[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            qv[i] = to_f(q[qo + lane + 32 * i]);
            ov[i] = to_f(dO[oo + lane + 32 * i]);
            acc[i] = 0.f;
        }
        if (L != -INFINITY) {
            const int *row = g.dense ? nullptr : idx_row(g, idx, b, kvh, t);
            const int c = kdiag(g, b, t), khi = min(c, seq_len_k(g, b) - 1);
            const int klo = key_lo(g, c);
            const int ns = n_slots(g, khi);
            for (int s = 0; s < ns; ++s) {
                const int j = slot_block(g, row, s, t);
                if (j < 0)
                    continue;
                const int kend = min((j + 1) * g.bs, khi + 1);
                for (int kk = max(j * g.bs, klo); kk < kend; ++kk) {
                    const int64_t ko = kv_off(g, b, kvh, kk);
                    float ps = 0.f, pd = 0.f;
                    float kv[DPL];
#pragma unroll
                    for (int i = 0; i < DPL; ++i) {
                        kv[i] = to_f(k[ko + lane + 32 * i]);
                        ps = fmaf(qv[i], kv[i], ps);
                        pd = fmaf(ov[i], to_f(v[ko + lane + 32 * i]), pd);
                    }
                    ps = warp_sum(ps);
                    pd = warp_sum(pd);
                    const float p = __expf(ps * g.scale - L);
                    const float ds = p * (pd - Dt);
#pragma unroll
                    for (int i = 0; i < DPL; ++i)
                        acc[i] = fmaf(ds, kv[i], acc[i]);
                }
            }
        }
        const int64_t dqo = dq_off(g, b, h, t);
#pragma unroll
        for (int i = 0; i < DPL; ++i)
            dq[dqo + lane + 32 * i] = from_f<T>(acc[i] * g.scale);
    }
}

// one warp per key: sum over the group's heads and the tokens that select
// the key's block (the inverse index), in ascending token order
template <typename T, int DPL>
__global__ void __launch_bounds__(kThreads) dkdv_simt_kernel(Geo g, const T *__restrict__ q,
                                                             const T *__restrict__ k,
                                                             const T *__restrict__ v,
                                                             const T *__restrict__ dO,
                                                             const float *__restrict__ lse,
                                                             const float *__restrict__ delta,
                                                             const int *__restrict__ offsets,
                                                             const int *__restrict__ rows,
                                                             T *__restrict__ dk, T *__restrict__ dv)
{
    const int lane = threadIdx.x & 31;
    const int64_t nkeys = (int64_t)g.ntok_k * g.Hkv;
    for (int64_t r = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); r < nkeys;
         r += (int64_t)gridDim.x * kWarps) {
        int b, kvh, kk;
        decode_krow(g, r, b, kvh, kk);
        const int j = kk / g.bs;
        const int64_t ko = kv_off(g, b, kvh, kk);
        float kv[DPL], vv[DPL], ak[DPL], av[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            kv[i] = to_f(k[ko + lane + 32 * i]);
            vv[i] = to_f(v[ko + lane + 32 * i]);
            ak[i] = 0.f;
            av[i] = 0.f;
        }
        int n, beg;
        if (j >= g.nbmax) {  // sequence longer than the declared bound
            n = 0;
            beg = 0;
        } else if (g.dense) {
            beg = dense_first(g, b, j);
            n = dense_count(g, b, j);
        } else {
            const int bgj = ((b * g.Hkv) + kvh) * g.nbmax + j;
            beg = offsets[bgj];
            n = offsets[bgj + 1] - beg;
        }
        for (int e = 0; e < n; ++e) {
            const int t = g.dense ? beg + e : rows[beg + e];
            const int c = kdiag(g, b, t);
            if (c < kk)
                continue;
            if (g.window > 0 && c - kk >= g.window)
                break;  // tokens ascend: the rest are past the window too
            for (int h = kvh * g.G; h < (kvh + 1) * g.G; ++h) {
                const int64_t qo = q_off(g, b, h, t), oo = o_off(g, b, h, t);
                const int64_t so = stat_off(g, b, h, t);
                float qv[DPL], ov[DPL], ps = 0.f, pd = 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i) {
                    qv[i] = to_f(q[qo + lane + 32 * i]);
                    ov[i] = to_f(dO[oo + lane + 32 * i]);
                    ps = fmaf(qv[i], kv[i], ps);
                    pd = fmaf(ov[i], vv[i], pd);
                }
                ps = warp_sum(ps);
                pd = warp_sum(pd);
                const float p = __expf(ps * g.scale - lse[so]);
                const float ds = p * (pd - delta[so]);
#pragma unroll
                for (int i = 0; i < DPL; ++i) {
                    ak[i] = fmaf(ds, qv[i], ak[i]);
                    av[i] = fmaf(p, ov[i], av[i]);
                }
            }
        }
        const int64_t dko = dkv_off(g, b, kvh, kk);
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
            dk[dko + lane + 32 * i] = from_f<T>(ak[i] * g.scale);
            dv[dko + lane + 32 * i] = from_f<T>(av[i]);
        }
    }
}

inline int rows_grid(int64_t nrows)
{
    int64_t b = (nrows + kWarps - 1) / kWarps;
    return (int)(b < 1 ? 1 : (b > 152 * 64 ? 152 * 64 : b));
}

}  // namespace

#define NSA_DISPATCH_D(D, BODY)                 \
    switch (D) {                                \
    case 32: { constexpr int DPL = 1; BODY; } break; \
    case 64: { constexpr int DPL = 2; BODY; } break; \
    case 128: { constexpr int DPL = 4; BODY; } break; \
    default: return cudaErrorInvalidValue;      \
    }

cudaError_t launch_fwd_simt(const Geo &g, const void *q, const void *k, const void *v,
                            const int *idx, void *o, float *lse, int dtype, cudaStream_t st)
{
    const int grid = rows_grid((int64_t)g.ntok * g.Hq);
    if (dtype == NSA_DTYPE_BF16) {
        using T = __nv_bfloat16;
        NSA_DISPATCH_D(g.D, (fwd_simt_kernel<T, DPL><<<grid, kThreads, 0, st>>>(
                                g, (const T *)q, (const T *)k, (const T *)v, idx, (T *)o, lse)));
    } else {
        using T = float;
        NSA_DISPATCH_D(g.D, (fwd_simt_kernel<T, DPL><<<grid, kThreads, 0, st>>>(
                                g, (const T *)q, (const T *)k, (const T *)v, idx, (T *)o, lse)));
    }
    return cudaGetLastError();
}

cudaError_t launch_dq_simt(const Geo &g, const void *q, const void *k, const void *v,
                           const void *dO, const float *lse, const float *delta, const int *idx,
                           void *dq, int dtype, cudaStream_t st)
{
    const int grid = rows_grid((int64_t)g.ntok * g.Hq);
    if (dtype == NSA_DTYPE_BF16) {
        using T = __nv_bfloat16;
        NSA_DISPATCH_D(g.D, (dq_simt_kernel<T, DPL><<<grid, kThreads, 0, st>>>(
                                g, (const T *)q, (const T *)k, (const T *)v, (const T *)dO, lse,
                                delta, idx, (T *)dq)));
    } else {
        using T = float;
        NSA_DISPATCH_D(g.D, (dq_simt_kernel<T, DPL><<<grid, kThreads, 0, st>>>(
                                g, (const T *)q, (const T *)k, (const T *)v, (const T *)dO, lse,
                                delta, idx, (T *)dq)));
    }
    return cudaGetLastError();
}

cudaError_t launch_dkdv_simt(const Geo &g, const void *q, const void *k, const void *v,
                             const void *dO, const float *lse, const float *delta,
                             const int *offsets, const int *rows, void *dk, void *dv, int dtype,
                             cudaStream_t st)
{
    const int grid = rows_grid((int64_t)g.ntok_k * g.Hkv);
    if (dtype == NSA_DTYPE_BF16) {
        using T = __nv_bfloat16;
        NSA_DISPATCH_D(g.D, (dkdv_simt_kernel<T, DPL><<<grid, kThreads, 0, st>>>(
                                g, (const T *)q, (const T *)k, (const T *)v, (const T *)dO, lse,
                                delta, offsets, rows, (T *)dk, (T *)dv)));
    } else {
        using T = float;
        NSA_DISPATCH_D(g.D, (dkdv_simt_kernel<T, DPL><<<grid, kThreads, 0, st>>>(
                                g, (const T *)q, (const T *)k, (const T *)v, (const T *)dO, lse,
                                delta, offsets, rows, (T *)dk, (T *)dv)));
    }
    return cudaGetLastError();
}

}  // namespace nsa
