// nsa_common.cuh -- problem geometry, addressing and the device error word,
// shared by every kernel of libnsa.
//
// Addressing follows the two layouts of the C ABI (include/nsa.h): BHTD
// (fixed length) and THD (packed variable length with cu_seqlens).  A query
// or key row is named by (sequence b, head h, sequence-local token t).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nsa.h"

namespace nsa {

// Element strides of (batch, head, token) of one tensor; the head dimension
// is contiguous.  THD: `b` is unused and `t` steps one packed row.
struct Strides {
    int64_t b, h, t;
};

// Device-side view of an nsa_problem plus derived quantities.
struct Geo {
    int B, Hq, Hkv, G, T, D, bs, S;
    int nbmax;       // ceil(T / bs): blocks of the longest sequence
    int ntok;        // B*T (BHTD) or total_tokens (THD)
    int thd;         // 1 for the packed layout
    int dense;       // 1: every row selects blocks 0..t/bs (no index read)
    int window;      // > 0: keys k with t - k < window only (sliding window); 0: none
    float scale;     // softmax scale
    float scale_l2;  // scale * log2(e)
    const int *cu;   // cu_seqlens (THD) or nullptr
    Strides sq;      // q
    Strides skv;     // k and v
    Strides so;      // o and dO
    Strides sdq;     // dq
    Strides sdkv;    // dk and dv
    int q_bt, o_bt;  // BHTD q / o: batch and token fold into one row index (b*T + t) for the row-gather maps
    int o_lin;       // o and dO are dense: query row r's vector sits at r * D
    // keys (the causal entries may give them their own lengths; elsewhere
    // they equal the queries'): BHTD key length, packed key count, cu_seqlens
    // of the keys (THD), and the alignment of the causal diagonal
    int Tk, ntok_k;
    const int *cuk;
    int br;          // 1: row t sits at key position t + Lk - Lq (bottom-right); 0: at t
};

__device__ __forceinline__ int seq_len(const Geo &g, int b) { return g.thd ? g.cu[b + 1] - g.cu[b] : g.T; }

// keys of sequence b
__device__ __forceinline__ int seq_len_k(const Geo &g, int b) { return g.thd ? g.cuk[b + 1] - g.cuk[b] : g.Tk; }

// the key position of row t's diagonal: keys k <= kdiag (and k < Lk) are causal
__device__ __forceinline__ int kdiag(const Geo &g, int b, int t)
{
    return g.br ? t + seq_len_k(g, b) - seq_len(g, b) : t;
}

// first key a row whose diagonal sits at key position c may attend (the
// sliding window's left edge; 0 without one)
__host__ __device__ __forceinline__ int key_lo(const Geo &g, int c)
{
    return (g.window > 0 && c - g.window + 1 > 0) ? c - g.window + 1 : 0;
}

// element offset of the D-vector of (b, head h, token t) in a tensor with strides s
__device__ __forceinline__ int64_t vec_off(const Geo &g, const Strides &s, int b, int h, int t)
{
    if (g.thd)
        return (int64_t)(g.cu[b] + t) * s.t + (int64_t)h * s.h;
    return (int64_t)b * s.b + (int64_t)h * s.h + (int64_t)t * s.t;
}
__device__ __forceinline__ int64_t q_off(const Geo &g, int b, int h, int t) { return vec_off(g, g.sq, b, h, t); }
__device__ __forceinline__ int64_t o_off(const Geo &g, int b, int h, int t) { return vec_off(g, g.so, b, h, t); }
__device__ __forceinline__ int64_t dq_off(const Geo &g, int b, int h, int t) { return vec_off(g, g.sdq, b, h, t); }
// the same for key rows (packed by the keys' cu_seqlens)
__device__ __forceinline__ int64_t vec_off_k(const Geo &g, const Strides &s, int b, int h, int k)
{
    if (g.thd)
        return (int64_t)(g.cuk[b] + k) * s.t + (int64_t)h * s.h;
    return (int64_t)b * s.b + (int64_t)h * s.h + (int64_t)k * s.t;
}
__device__ __forceinline__ int64_t kv_off(const Geo &g, int b, int h, int k) { return vec_off_k(g, g.skv, b, h, k); }
__device__ __forceinline__ int64_t dkv_off(const Geo &g, int b, int h, int k) { return vec_off_k(g, g.sdkv, b, h, k); }

// the D-vector of query row number r (the row order of lse and delta: BHTD
// (b*Hq + h)*T + t, THD token*Hq + h) in a tensor with strides s
__device__ __forceinline__ int64_t qrow_off(const Geo &g, const Strides &s, int64_t r)
{
    if (g.thd)
        return (r / g.Hq) * s.t + (r % g.Hq) * s.h;
    const int64_t bh = r / g.T;
    return (bh / g.Hq) * s.b + (bh % g.Hq) * s.h + (r % g.T) * s.t;
}

// offset of a per-row scalar (lse, delta) of (b, query head h, t)
__device__ __forceinline__ int64_t stat_off(const Geo &g, int b, int h, int t)
{
    if (g.thd)
        return (int64_t)(g.cu[b] + t) * g.Hq + h;
    return ((int64_t)b * g.Hq + h) * g.T + t;
}

// the number of index row (b, kvh, t): BHTD (b*Hkv + kvh)*T + t, THD token*Hkv + kvh
// (the block scores of the selection step use the same rows)
__device__ __forceinline__ int64_t index_row(const Geo &g, int b, int kvh, int t)
{
    if (g.thd)
        return (int64_t)(g.cu[b] + t) * g.Hkv + kvh;
    return ((int64_t)b * g.Hkv + kvh) * g.T + t;
}

__device__ __forceinline__ const int *idx_row(const Geo &g, const int *idx, int b, int kvh, int t)
{
    if (g.thd)
        return idx + ((int64_t)(g.cu[b] + t) * g.Hkv + kvh) * g.S;
    return idx + (((int64_t)b * g.Hkv + kvh) * g.T + t) * g.S;
}

// sequence holding packed token `tok` (THD); binary search over cu_seqlens
__device__ __forceinline__ int seq_of_token(const Geo &g, int tok)
{
    int lo = 0, hi = g.B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (g.cu[mid] <= tok)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// sequence holding packed key `tok` (THD); binary search over the keys' cu_seqlens
__device__ __forceinline__ int seq_of_key(const Geo &g, int tok)
{
    int lo = 0, hi = g.B - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (g.cuk[mid] <= tok)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// does row (b, kvh, t) select block j?  (dense: every block holding a key
// between the window's left edge and the diagonal)
__device__ __forceinline__ bool row_selects(const Geo &g, const int *idx, int b, int kvh, int t, int j)
{
    if (g.dense) {
        const int c = kdiag(g, b, t), hi = min(c, seq_len_k(g, b) - 1);
        const int lo = key_lo(g, c);
        return lo <= hi && j <= hi / g.bs && j >= lo / g.bs;
    }
    const int *r = idx_row(g, idx, b, kvh, t);
    for (int s = 0; s < g.S; ++s)
        if (r[s] == j)
            return true;
    return false;
}

// Dense entries: the tokens of sequence b that attend a key of block j form
// one range, from dense_first (the first row whose diagonal reaches the
// block) for dense_count tokens (up to the last row, or with a window the
// last row whose window still reaches the block's last key).  0 for a block
// past the keys' end.
__device__ __forceinline__ int dense_first(const Geo &g, int b, int j)
{
    const int shift = g.br ? seq_len_k(g, b) - seq_len(g, b) : 0;
    return max(0, j * g.bs - shift);
}
__device__ __forceinline__ int dense_count(const Geo &g, int b, int j)
{
    const int Lq = seq_len(g, b), Lk = seq_len_k(g, b);
    if (j * g.bs >= Lk)
        return 0;
    const int shift = g.br ? Lk - Lq : 0;
    int end = Lq;
    if (g.window > 0)
        end = min(end, (j + 1) * g.bs + g.window - 1 - shift);
    return max(0, end - dense_first(g, b, j));
}

// The first error recorded wins; later ones are dropped.
__device__ __forceinline__ void set_error(int *err, int code)
{
    if (err)
        atomicCAS(err, 0, code);
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// A dK/dV work unit: rows [begin, begin + count) of the token list of
// (bg = b*Hkv + kvh, block j); slot >= 0 names the fp32 partial buffer the
// unit writes when the block is split into several units, -1 = write the
// final dK/dV directly.
struct Unit {
    int bg, j, begin, count, slot, pad0, pad1, pad2;
};

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
    int err;        // nsa_status recorded by the device
    int n_units;    // number of dK/dV units built for the current call
    int tile_next;  // the query-tile kernels' work counter (zeroed with the header)
    int pad[61];
};

}  // namespace nsa
