// k_gtc.cu -- the forward, dQ and dK/dV on the tcgen05 tensor cores for the
// shapes the specialised kernels (bf16, D = 128, 64-key blocks) do not take:
// head dims 32, 64 and 128 with blocks of 16, 32 or 64 keys in bf16, and head
// dims 32 and 64 in fp32.
//
// fp32 runs in split precision on the bf16 tensor cores: every fp32 operand x
// is held as a bf16 high part h = bf16(x) and a bf16 low part l = bf16(x - h)
// (|x - h - l| <= 2^-18 |x|), and every product A B^T is issued as three MMAs,
// Ah Bh^T + Ah Bl^T + Al Bh^T, accumulated in fp32 (the dropped Al Bl^T and the
// parts' rounding leave about 2^-16 of |A||B|).
//
// One CTA of 256 threads per work item -- a query tile (Tq tokens x the G
// heads of a kv head) for the forward and dQ, a dK/dV unit of the inverse
// index -- and two threads own each tile row r (TMEM lane r), each taking
// half of the row's keys and output columns.  Thread 0 issues the MMAs and
// commits them to one mbarrier, on which all threads wait (bounded).  Every
// tile is stored once, K-major in 128-byte-swizzled shared memory, as the
// threads that load or compute it write it; a product that needs the tile
// transposed (V and K in P V and dS K, dO and Q in dV^T and dK^T, P and dS)
// reads it by columns, as an MN-major operand.  Head dims below 64 are
// zero-padded to 64; with them dV^T and dK^T are one M = 128 product:
// [dO^T; Q^T] times [P dS], whose diagonal blocks are the two results.
//
// The forward takes two passes over the tile's blocks: the first finds each
// row's maximum and sum (its LSE), the second forms P = exp(S - LSE) and
// accumulates P V, so no accumulator is rescaled.
#include <string.h>

#include "tc_common.cuh"

namespace nsa {

namespace {

using namespace tc;

constexpr int kThr = 128;    // threads per CTA = tile rows
constexpr int kKeyPad = 64;  // key-dimension width of P, dS, K^T, V^T tiles

struct GParams {
    Geo g;
    const void *q, *k, *v, *dO;
    const float *lse, *delta;
    const int *idx;
    const int *offsets, *rows;
    const Unit *units;
    const WsHeader *hdr;
    float *partials;
    void *o, *dq, *dk, *dv;
    float *lse_out;
    float *scores;  // block scores (selection step)
    int *err;
    int Dp;       // head dim padded to 64 or 128
    int ntiles;   // query tiles (forward / dQ)
    int wait_us;  // bounded-wait limit in microseconds (0: the default)
};

// byte offset of element (r, c) of a K-major tile with R rows (a multiple of
// 8) and 64-column chunks of 128-byte rows, 128-byte swizzle
__device__ __forceinline__ uint32_t swz(int r, int c, int R)
{
    return (uint32_t)((c >> 6) * (R * 128) + (r >> 3) * 1024 + (r & 7) * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                      ((c & 7) << 1));
}

// descriptor of K-step kk (16 elements) of such a tile
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int R, int kk)
{
    return sdesc_sw128(tile + (kk >> 2) * (R * 128) + (kk & 3) * 32, 16, 1024);
}

__device__ __forceinline__ uint16_t bf16_bits(float x)
{
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t *>(&b);
}

// An operand value as stored: its high part, and (SPLIT) its low part
template <bool SPLIT> struct Parts {
    uint16_t hi, lo;
};
template <bool SPLIT> __device__ __forceinline__ Parts<SPLIT> split_of(float x)
{
    Parts<SPLIT> p;
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    p.hi = *reinterpret_cast<uint16_t *>(&h);
    p.lo = SPLIT ? bf16_bits(x - __bfloat162float(h)) : (uint16_t)0;
    return p;
}

// descriptor of K-step kk (16 rows) of such a tile read as an MN-major
// operand: its rows are the K index and its columns the N index (64-column
// chunks R * 128 bytes apart)
__device__ __forceinline__ uint64_t mndesc(uint32_t tile, int R, int kk)
{
    return sdesc_sw128(tile + kk * 2048, R * 128, 1024);
}

// writes elements (r, c .. c+7) of a tile (c a multiple of 8: one 16-byte
// chunk), and of its low-part copy lo_off bytes on
template <bool SPLIT>
__device__ __forceinline__ void put8(uint32_t tile, int R, uint32_t lo_off, int r, int c, const float *x)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const Parts<SPLIT> p0 = split_of<SPLIT>(x[2 * i]), p1 = split_of<SPLIT>(x[2 * i + 1]);
        h[i] = (uint32_t)p0.hi | ((uint32_t)p1.hi << 16);
        l[i] = (uint32_t)p0.lo | ((uint32_t)p1.lo << 16);
    }
    const uint32_t a = tile + swz(r, c, R);
    st_shared_v4(a, h[0], h[1], h[2], h[3]);
    if (SPLIT)
        st_shared_v4(a + lo_off, l[0], l[1], l[2], l[3]);
}

// D (+)= A B^T over nk K-steps; SPLIT: three products of the parts.  A and B
// are K-major tiles (A with Ra rows, B with Rb rows) whose low parts sit
// alo / blo bytes after them.
template <bool SPLIT>
__device__ __forceinline__ void product(uint32_t d, uint32_t a, int Ra, uint32_t alo, uint32_t b, int Rb, uint32_t blo,
                                        uint32_t idesc, int nk, bool acc)
{
    for (int kk = 0; kk < nk; ++kk) {
        const uint32_t on = (acc || kk > 0) ? 1u : 0u;
        mma_bf16(d, kdesc(a, Ra, kk), kdesc(b, Rb, kk), idesc, on);
        if (SPLIT) {
            mma_bf16(d, kdesc(a, Ra, kk), kdesc(b + blo, Rb, kk), idesc, 1u);
            mma_bf16(d, kdesc(a + alo, Ra, kk), kdesc(b, Rb, kk), idesc, 1u);
        }
    }
}

// D (+)= A B over nk K-steps, B MN-major: a K-major tile of Rb rows (the K
// index) read by columns (the N index), as mndesc; otherwise as product
template <bool SPLIT>
__device__ __forceinline__ void product_bmn(uint32_t d, uint32_t a, int Ra, uint32_t alo, uint32_t b, int Rb,
                                            uint32_t blo, uint32_t idesc, int nk, bool acc)
{
    for (int kk = 0; kk < nk; ++kk) {
        const uint32_t on = (acc || kk > 0) ? 1u : 0u;
        mma_bf16(d, kdesc(a, Ra, kk), mndesc(b, Rb, kk), idesc, on);
        if (SPLIT) {
            mma_bf16(d, kdesc(a, Ra, kk), mndesc(b + blo, Rb, kk), idesc, 1u);
            mma_bf16(d, kdesc(a + alo, Ra, kk), mndesc(b, Rb, kk), idesc, 1u);
        }
    }
}

// D (+)= A B over nk K-steps, both operands MN-major: A a K-major tile read
// by columns whose 64-column chunks (the M index) lie a_lbo bytes apart
// (within one tile, or two tiles placed that far apart), B as product_bmn
template <bool SPLIT>
__device__ __forceinline__ void product_mn(uint32_t d, uint32_t a, uint32_t a_lbo, uint32_t alo, uint32_t b, int Rb,
                                           uint32_t blo, uint32_t idesc, int nk, bool acc)
{
    for (int kk = 0; kk < nk; ++kk) {
        const uint32_t on = (acc || kk > 0) ? 1u : 0u;
        const uint64_t ad = sdesc_sw128(a + kk * 2048, a_lbo, 1024);
        mma_bf16(d, ad, mndesc(b, Rb, kk), idesc, on);
        if (SPLIT) {
            mma_bf16(d, ad, mndesc(b + blo, Rb, kk), idesc, 1u);
            mma_bf16(d, sdesc_sw128(a + alo + kk * 2048, a_lbo, 1024), mndesc(b, Rb, kk), idesc, 1u);
        }
    }
}

// output element (bf16 or fp32 by SPLIT)
template <bool SPLIT> __device__ __forceinline__ void out_at(void *base, int64_t off, float x)
{
    if (SPLIT)
        ((float *)base)[off] = x;
    else
        ((__nv_bfloat16 *)base)[off] = __float2bfloat16_rn(x);
}

// 16 consecutive output elements x[i] * mul (zeros without `any`) as 16-byte
// stores: rows start 16-byte aligned and off is a multiple of 16 from a row's
// start (D is a multiple of 16)
template <bool SPLIT>
__device__ __forceinline__ void out16(void *base, int64_t off, const float *x, float mul, bool any)
{
    uint32_t w[SPLIT ? 16 : 8];
#pragma unroll
    for (int i = 0; i < (SPLIT ? 16 : 8); ++i)
        w[i] = SPLIT ? __float_as_uint(any ? x[i] * mul : 0.f)
                     : (uint32_t)bf16_bits(any ? x[2 * i] * mul : 0.f) |
                           ((uint32_t)bf16_bits(any ? x[2 * i + 1] * mul : 0.f) << 16);
    uint4 *d = SPLIT ? (uint4 *)((float *)base + off) : (uint4 *)((__nv_bfloat16 *)base + off);
#pragma unroll
    for (int i = 0; i < (SPLIT ? 4 : 2); ++i)
        d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// Shared synchronisation of the CTA: the MMA barrier's phase and the wait
// context (abort flag, limit).  issue_wait: thread 0 commits every MMA it
// issued so far to the barrier, everyone waits for it; false (on every
// thread) once a wait gave up.
// A second MMA-issuing thread (warp 1's lane 0): one thread issues a tcgen05
// MMA only every ~120 cycles, so S and dP go out from two threads at once.
// Every commit_wait takes a commit from both (a commit with nothing
// outstanding arrives at once).
constexpr int kIssuer2 = 32;

struct Sync {
    uint64_t *bar;
    volatile int *ctx;
    uint32_t phase;
};

__device__ __forceinline__ bool commit_wait(Sync &s)
{
    if (threadIdx.x == 0 || threadIdx.x == 32)  // both issuing threads (see kIssuer2)
        mma_commit(s.bar);
    bool ok = mbar_wait(s.bar, s.phase, s.ctx);
    s.phase ^= 1;
    ok = __syncthreads_and(ok) != 0;
    tc_fence_after();
    return ok;
}

// every thread's shared-memory writes are visible to the tensor cores, and
// every thread's TMEM reads are done, before thread 0 issues the next MMAs
__device__ __forceinline__ void to_mma()
{
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// The kernels' common start: the wait context, the MMA barrier and 256 TMEM
// columns; the end: every MMA done, TMEM freed, a timeout reported.
__device__ __forceinline__ uint32_t g_start(uint8_t *misc, const GParams &p, Sync &s, uint32_t cols = 256)
{
    uint64_t *bar = (uint64_t *)misc;
    volatile int *ctx = (volatile int *)(misc + 16);
    uint32_t *slot = (uint32_t *)(misc + 32);
    if (threadIdx.x == 0) {
        ctx[0] = 0;
        ctx[1] = p.wait_us;
        mbar_init(bar, 2);  // commits from threads 0 and kIssuer2
        fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(slot, cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    s.bar = bar;
    s.ctx = ctx;
    s.phase = 0;
    return *slot;
}

__device__ __forceinline__ void g_end(uint32_t tmem, Sync &s, const GParams &p, uint32_t cols = 256)
{
    // MMAs still in flight (after a timeout) complete before TMEM is freed
    if (threadIdx.x == 0 || threadIdx.x == 32)
        mma_commit(s.bar);
    if (threadIdx.x == 0) {
        volatile int never[2] = {0, s.ctx[1]};
        mbar_wait(s.bar, s.phase, never);
    }
    tc_fence_before();
    __syncthreads();
    if (s.ctx[0] && threadIdx.x == 0)
        set_error(p.err, NSA_ERR_DEVICE_TIMEOUT);
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, cols);
    }
}

// 16-byte vectors of the input: 8 bf16 or 4 fp32 elements
template <bool SPLIT> struct In {
    static constexpr int VEC = SPLIT ? 4 : 8;
    static constexpr int ES = SPLIT ? 4 : 2;
};

// a vector's VEC elements into row r, columns c .. c+VEC-1 of a tile (c a
// multiple of VEC): one 16-byte store (bf16), or 8 bytes of high parts and 8
// of low parts (SPLIT)
template <bool SPLIT>
__device__ __forceinline__ void put_vec(uint32_t tile, int R, uint32_t lo_off, int r, int c, const uint4 &w)
{
    const uint32_t a = tile + swz(r, c, R);
    if (!SPLIT) {
        st_shared_v4(a, w.x, w.y, w.z, w.w);
        return;
    }
    const float x[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w)};
    uint32_t h[2], l[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const Parts<true> p0 = split_of<true>(x[2 * i]), p1 = split_of<true>(x[2 * i + 1]);
        h[i] = (uint32_t)p0.hi | ((uint32_t)p1.hi << 16);
        l[i] = (uint32_t)p0.lo | ((uint32_t)p1.lo << 16);
    }
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a), "r"(h[0]), "r"(h[1]) : "memory");
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(a + lo_off), "r"(l[0]), "r"(l[1]) : "memory");
}

// A key block of a kv-shaped tensor in registers: this thread's vector i is
// vector e = (threadIdx.x % kThr) + i * kThr of the block (each 128 threads
// of a larger CTA cover the whole block) (key e / (D / VEC), columns
// from (e % (D / VEC)) * VEC); keys past the sequence's end read as zeros.
constexpr int kBlkVec = 8;  // bs * D / VEC <= 1024 vectors per block
struct BlockRegs {
    uint4 v[kBlkVec];
};

template <bool SPLIT>
__device__ __forceinline__ void fetch_block(const Geo &g, const void *src, int b, int kvh, int k0, BlockRegs &R)
{
    constexpr int VEC = In<SPLIT>::VEC;
    // vectors per key row: D / VEC, a power of two (D is 32, 64 or 128)
    const int nv = g.D / VEC, lnv = __ffs(nv) - 1, n = g.bs * nv, nk = min(g.bs, seq_len_k(g, b) - k0);
#pragma unroll
    for (int i = 0; i < kBlkVec; ++i) {
        const int e = (threadIdx.x & (kThr - 1)) + i * kThr, key = e >> lnv, c = (e & (nv - 1)) * VEC;
        R.v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (e < n && key < nk)
            R.v[i] = __ldg((const uint4 *)((const uint8_t *)src + (kv_off(g, b, kvh, k0 + key) + c) * In<SPLIT>::ES));
    }
}

// the block into a [bs][Dp] tile
template <bool SPLIT>
__device__ __forceinline__ void store_block(const Geo &g, const BlockRegs &R, uint32_t tile, uint32_t lo_off)
{
    constexpr int VEC = In<SPLIT>::VEC;
    const int nv = g.D / VEC, lnv = __ffs(nv) - 1, n = g.bs * nv;
#pragma unroll
    for (int i = 0; i < kBlkVec; ++i) {
        const int e = (threadIdx.x & (kThr - 1)) + i * kThr;
        if (e < n)
            put_vec<SPLIT>(tile, g.bs, lo_off, e >> lnv, (e & (nv - 1)) * VEC, R.v[i]);
    }
}

// A group of 64 keys: the 64 / BS union blocks list[i0 ..] (fewer at the
// list's end), block list[i0 + r / BS]'s key r % BS in row r.  The query-tile
// kernels walk their blocks a group at a time, so that each step's fixed
// costs (stores, barriers, MMA latencies) are paid once per 64 keys.
constexpr int kGroupKeys = 64;

template <bool SPLIT, int BS, int NT = kThr>
__device__ __forceinline__ void fetch_group(const Geo &g, const void *src, int b, int kvh, const int *list, int i0,
                                            int U, BlockRegs &R)
{
    constexpr int VEC = In<SPLIT>::VEC;
    const int nv = g.D / VEC, lnv = __ffs(nv) - 1, n = kGroupKeys * nv, Lk = seq_len_k(g, b);
#pragma unroll
    for (int i = 0; i < kBlkVec * kThr / NT; ++i) {
        const int e = threadIdx.x + i * NT, row = e >> lnv, c = (e & (nv - 1)) * VEC, gi = i0 + row / BS;
        R.v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (e < n && gi < U) {
            const int key = list[gi] * BS + row % BS;
            if (key < Lk)
                R.v[i] = __ldg((const uint4 *)((const uint8_t *)src + (kv_off(g, b, kvh, key) + c) * In<SPLIT>::ES));
        }
    }
}

// the group into a [64][Dp] tile
template <bool SPLIT, int NT = kThr>
__device__ __forceinline__ void store_group(const Geo &g, const BlockRegs &R, uint32_t tile, uint32_t lo_off)
{
    constexpr int VEC = In<SPLIT>::VEC;
    const int nv = g.D / VEC, lnv = __ffs(nv) - 1, n = kGroupKeys * nv;
#pragma unroll
    for (int i = 0; i < kBlkVec * kThr / NT; ++i) {
        const int e = threadIdx.x + i * NT;
        if (e < n)
            put_vec<SPLIT>(tile, kGroupKeys, lo_off, e >> lnv, (e & (nv - 1)) * VEC, R.v[i]);
    }
}

// One row of a q-shaped tensor (this thread's) in registers
constexpr int kRowVec = 16;  // D * element bytes / 16 <= 16
struct RowRegs {
    uint4 v[kRowVec];
};

template <bool SPLIT>
__device__ __forceinline__ void fetch_row(const Geo &g, const void *src, int64_t off, bool valid, RowRegs &R)
{
    constexpr int VEC = In<SPLIT>::VEC;
#pragma unroll
    for (int i = 0; i < kRowVec; ++i) {
        R.v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (valid && i * VEC < g.D)
            R.v[i] = __ldg((const uint4 *)((const uint8_t *)src + (off + i * VEC) * In<SPLIT>::ES));
    }
}

// the row into row r of a [128][Dp] tile
template <bool SPLIT>
__device__ __forceinline__ void store_row(const Geo &g, const RowRegs &R, uint32_t tile, uint32_t lo_off, int r)
{
    constexpr int VEC = In<SPLIT>::VEC;
#pragma unroll
    for (int i = 0; i < kRowVec; ++i) {
        if (i * VEC >= g.D)
            break;
        put_vec<SPLIT>(tile, 128, lo_off, r, i * VEC, R.v[i]);
    }
}

// The query tile's union (as qtile_union_warp builds it) from the whole CTA:
// every thread reads its share of the tile's index entries at once (one
// round of loads for a tile of up to 4 entries a thread), then one warp
// compacts the list.  Holds three CTA-wide barriers; nvalid > 0.
__device__ __forceinline__ void qtile_union_cta(const Geo &g, const int *idx, const UnionBuf &u, int *buf, int b,
                                                int kvh, int t0, int nvalid)
{
    const int words = (g.nbmax + 31) / 32, tid = threadIdx.x, nt = blockDim.x;
    uint32_t *mask = union_mask(buf), *ubits = mask + u.mask_words;
    for (int x = tid; x < u.mask_words + words; x += nt)  // the tokens' bitmaps, then the union's
        mask[x] = 0u;
    __syncthreads();
    if (g.dense) {
        const int hi = min(kdiag(g, b, t0 + nvalid - 1), seq_len_k(g, b) - 1);
        const int jmin = key_lo(g, kdiag(g, b, t0)) / g.bs, jmax = hi >= 0 ? hi / g.bs : -1;
        for (int j = jmin + tid; j <= jmax; j += nt)
            atomicOr(&ubits[j >> 5], 1u << (j & 31));
    } else {
        const int n = nvalid * g.S;
        for (int x0 = 0; x0 < n; x0 += 4 * nt) {
            int jv[4];
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                const int x = x0 + u4 * nt + tid;
                jv[u4] = x < n ? idx_row(g, idx, b, kvh, t0 + x / g.S)[x % g.S] : -1;
            }
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                const int x = x0 + u4 * nt + tid;
                const int tl = x / g.S, t = t0 + tl, j = jv[u4];
                if (x < n && j >= 0 && j <= t / g.bs && j < g.nbmax) {
                    atomicOr(&mask[tl * words + (j >> 5)], 1u << (j & 31));
                    atomicOr(&ubits[j >> 5], 1u << (j & 31));
                }
            }
        }
    }
    __syncthreads();
    if (tid < 32) {  // ordered compaction
        const int lane = tid;
        int *list = union_list(buf, u);
        int base = 0;
        for (int w0 = 0; w0 < words; w0 += 32) {
            const uint32_t bits = (w0 + lane < words) ? ubits[w0 + lane] : 0u;
            const int cnt = __popc(bits);
            int incl = cnt;
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off)
                    incl += y;
            }
            int pos = base + incl - cnt;
            for (uint32_t bb = bits; bb; bb &= bb - 1)
                list[pos++] = (w0 + lane) * 32 + __ffs(bb) - 1;
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            buf[UH_B] = b;
            buf[UH_KVH] = kvh;
            buf[UH_T0] = t0;
            buf[UH_NVALID] = nvalid;
            buf[UH_GROUPED] = 0;
            buf[UH_COUNT] = base;
        }
    }
    __syncthreads();
}

// row r of a query tile: token tl of the tile (rows token-major), head hh of the group
__device__ __forceinline__ void qrow(int G, int r, int &tl, int &hh)
{
    tl = r / G;
    hh = r % G;
}

// N consecutive TMEM columns (a multiple of 16) of this thread's lane (row)
// as floats, from col_a into a and (NB = N) from col_b into b: every load
// goes out before the one wait
template <int N, int NB = 0>
__device__ __forceinline__ void ld_cols(uint32_t tmem, int col_a, float *a, int col_b = 0, float *b = nullptr)
{
    static_assert(N % 16 == 0 && (NB == 0 || NB == N), "whole 16-column loads");
    const uint32_t base = tmem + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16);  // warp w: lanes 32*(w%4)..
    uint32_t va[N / 16][16], vb[NB ? N / 16 : 1][16];
#pragma unroll
    for (int c = 0; c < N / 16; ++c) {
        tmem_ld16(base + col_a + c * 16, va[c]);
        if (NB)
            tmem_ld16(base + col_b + c * 16, vb[c]);
    }
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < N / 16; ++c)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            a[c * 16 + i] = __uint_as_float(va[c][i]);
            if (NB)
                b[c * 16 + i] = __uint_as_float(vb[c][i]);
        }
}

constexpr uint32_t TM_S = 0, TM_DP = 64, TM_ACC = 128, TM_ACC2 = 192;

// zeroes n bytes of shared memory from p (16-byte multiples)
__device__ __forceinline__ void zero_smem(uint8_t *p, int n)
{
    for (int i = threadIdx.x; i < n / 16; i += blockDim.x)
        ((uint4 *)p)[i] = make_uint4(0, 0, 0, 0);
}

// The query-tile kernels (forward, dQ) run two threads per tile row (256
// threads): thread r + 128 hc takes key columns 32 hc .. 32 hc + 31 of row
// r's S, P and dS, and output columns 16 hc + 32 i.  MINB = 1 gives each
// thread the registers of one CTA per SM (grids of at most one tile per SM);
// MINB = 2 caps them for two resident CTAs (larger grids).
constexpr int kRowThr = 2 * kThr;

// ---------------------------------------------------------------- forward
template <bool SPLIT, int BS, int MINB>
__global__ void __launch_bounds__(kRowThr, MINB) fwd_gtc_kernel(const GParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Geo &g = p.g;
    constexpr int bs = BS;                     // keys per block (the launch picks the instance for g.bs)
    constexpr int GB = kGroupKeys / BS;        // blocks per group
    constexpr int NK = kGroupKeys;             // keys per group: the products' N (S) and K (P V)
    const int Dp = p.Dp, G = g.G, Tq = tile_tokens(G), nrows = Tq * G, parts = SPLIT ? 2 : 1;
    const UnionBuf up = union_buf(g);
    // plan: Q [128][Dp] | K [64][Dp] | V [64][Dp] (read MN-major by P V) |
    // P [128][64] (each with its low part right after it) | union buffer |
    // barrier, wait context, TMEM slot | the halves' row statistics
    const uint32_t QB = 128 * Dp * 2, KB = NK * Dp * 2, VB = KB, PB = 128 * kKeyPad * 2;
    uint8_t *q_t = sm, *k_t = q_t + parts * QB, *v_t = k_t + parts * KB, *p_t = v_t + parts * VB;
    int *ubuf = (int *)(p_t + parts * PB);
    uint8_t *misc = (uint8_t *)ubuf + up.bytes;
    Sync sy;
    float *xchg = (float *)(misc + 64);  // [2 halves][m, l][128 rows]
    const uint32_t tmem = g_start(misc, p, sy);
    const int r = threadIdx.x & (kThr - 1), hc = threadIdx.x >> 7;
    int b = 0, kvh = 0, t0 = 0, nvalid = 0;
    qtile_of(g, blockIdx.x, b, kvh, t0, nvalid);
    zero_smem(sm, parts * (QB + KB + VB + PB));
    if (nvalid > 0)
        qtile_union_cta(g, p.idx, up, ubuf, b, kvh, t0, nvalid);
    __syncthreads();
    const int U = nvalid > 0 ? ubuf[UH_COUNT] : 0, NG = (U + GB - 1) / GB;
    const int *list = union_list(ubuf, up);
    int tl, hh;
    qrow(G, r, tl, hh);
    const bool rvalid = r < nrows && tl < nvalid;
    const int t = t0 + tl, words = (g.nbmax + 31) / 32;
    const int cdiag = rvalid ? kdiag(g, b, t) : -1;
    const int khi = rvalid ? min(cdiag, seq_len_k(g, b) - 1) : -1, klo = key_lo(g, cdiag);
    const uint32_t *my_mask = union_mask(ubuf) + (rvalid ? tl : 0) * words;
    const uint32_t qs = smem_u32(q_t), ks = smem_u32(k_t), vs = smem_u32(v_t), ps = smem_u32(p_t);
    // the row's q (zero for rows past the tile's tokens)
    if (hc == 0) {
        RowRegs qr;
        fetch_row<SPLIT>(g, p.q, rvalid ? q_off(g, b, kvh * G + hh, t) : 0, rvalid, qr);
        store_row<SPLIT>(g, qr, qs, QB, r);
    }
    const uint32_t idS = idesc_bf16(128, NK, false, false), idO = idesc_bf16(128, Dp, false, true);
    // the first key of each block of group gi (-1 past the list's end) and
    // whether the row takes that block
    auto group_blocks = [&](int gi, int *k0s, bool *sel) {
#pragma unroll
        for (int e = 0; e < GB; ++e) {
            const int li = gi * GB + e;
            const int j = li < U ? list[li] : -1;
            k0s[e] = j * bs;
            sel[e] = j >= 0 && rvalid && qtile_selects(g, my_mask, klo, khi, j);
        }
    };
    bool ok = true;
    // pass 1: the maximum m and sum l of exp2(scale_l2 * s) over the row's
    // keys in this thread's columns, then the two halves' combined
    float m = -INFINITY, l = 0.f;
    BlockRegs kr, vr;  // the next group's K (and V), fetched while the MMAs run
    if (NG > 0)
        fetch_group<SPLIT, BS, kRowThr>(g, p.k, b, kvh, list, 0, U, kr);
    for (int gi = 0; gi < NG && ok; ++gi) {
        store_group<SPLIT, kRowThr>(g, kr, ks, KB);
        to_mma();
        if (threadIdx.x == 0)
            product<SPLIT>(tmem + TM_S, qs, 128, QB, ks, NK, KB, idS, Dp / 16, false);
        if (gi + 1 < NG)
            fetch_group<SPLIT, BS, kRowThr>(g, p.k, b, kvh, list, (gi + 1) * GB, U, kr);
        if (!(ok = commit_wait(sy)))
            break;
        int k0s[GB];
        bool sel[GB];
        group_blocks(gi, k0s, sel);
        constexpr int NH = NK / 2;
        const int c1 = hc * NH;
        float sc[NH];
        ld_cols<NH>(tmem, TM_S + c1, sc);
        // the group's maximum first, then its terms against the new maximum
        float bm = -INFINITY;
#pragma unroll
        for (int x = 0; x < NH; ++x) {
            const int c = c1 + x, key = k0s[c / bs] + c % bs;
            sc[x] = (sel[c / bs] && key >= klo && key <= khi) ? sc[x] * g.scale_l2 : -INFINITY;
            bm = fmaxf(bm, sc[x]);
        }
        if (bm != -INFINITY) {
            const float mn = fmaxf(m, bm);
            float sum = 0.f;
#pragma unroll
            for (int x = 0; x < NH; ++x)
                sum += ex2(sc[x] - mn);  // exp2(-inf) = 0 off the row's keys
            l = l * ex2(m - mn) + sum;
            m = mn;
        }
    }
    xchg[(hc * 2) * kThr + r] = m;
    xchg[(hc * 2 + 1) * kThr + r] = l;
    __syncthreads();
    {  // both halves combine the same two pairs in the same order
        const float m0 = xchg[r], l0 = xchg[kThr + r], m1 = xchg[2 * kThr + r], l1 = xchg[3 * kThr + r];
        m = fmaxf(m0, m1);
        l = m == -INFINITY ? 0.f : l0 * ex2(m0 - m) + l1 * ex2(m1 - m);
    }
    const float lse2 = l > 0.f ? m + log2f(l) : -INFINITY;
    // pass 2: P = exp2(scale_l2 s - lse2) on the row's keys, O += P V
    if (NG > 0 && ok) {
        fetch_group<SPLIT, BS, kRowThr>(g, p.k, b, kvh, list, 0, U, kr);
        fetch_group<SPLIT, BS, kRowThr>(g, p.v, b, kvh, list, 0, U, vr);
    }
    for (int gi = 0; gi < NG && ok; ++gi) {
        store_group<SPLIT, kRowThr>(g, kr, ks, KB);
        store_group<SPLIT, kRowThr>(g, vr, vs, VB);
        to_mma();
        if (threadIdx.x == 0)
            product<SPLIT>(tmem + TM_S, qs, 128, QB, ks, NK, KB, idS, Dp / 16, false);
        if (gi + 1 < NG) {
            fetch_group<SPLIT, BS, kRowThr>(g, p.k, b, kvh, list, (gi + 1) * GB, U, kr);
            fetch_group<SPLIT, BS, kRowThr>(g, p.v, b, kvh, list, (gi + 1) * GB, U, vr);
        }
        if (!(ok = commit_wait(sy)))
            break;
        int k0s[GB];
        bool sel[GB];
        group_blocks(gi, k0s, sel);
        {
            const int c1 = hc * 32;
            float sc[32];
            ld_cols<32>(tmem, TM_S + c1, sc);
#pragma unroll
            for (int c0 = 0; c0 < 32; c0 += 8) {
                float pv[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int c = c1 + c0 + x, key = k0s[c / bs] + c % bs;
                    pv[x] = (sel[c / bs] && lse2 != -INFINITY && key >= klo && key <= khi)
                                ? ex2(sc[c0 + x] * g.scale_l2 - lse2)
                                : 0.f;
                }
                put8<SPLIT>(ps, 128, PB, r, c1 + c0, pv);
            }
        }
        to_mma();
        if (threadIdx.x == 0)  // O += P V, V read MN-major from its plain tile
            product_bmn<SPLIT>(tmem + TM_ACC, ps, 128, PB, vs, NK, VB, idO, NK / 16, gi > 0);
        ok = commit_wait(sy);
    }
    // epilogue: O (already normalised) and the natural-log LSE.  Every lane
    // runs the TMEM loads (warp-wide .sync.aligned); valid rows store.
    if (ok) {
        const int64_t oo = rvalid ? o_off(g, b, kvh * G + hh, t) : 0;
        float acc[16];
        for (int c0 = hc * 16; c0 < g.D; c0 += 32) {
            if (U > 0)
                ld_cols<16>(tmem, TM_ACC + c0, acc);
            if (rvalid)
                out16<SPLIT>(p.o, oo + c0, acc, 1.f, U > 0 && lse2 != -INFINITY);
        }
        if (rvalid && hc == 0)
            p.lse_out[stat_off(g, b, kvh * G + hh, t)] = lse2 == -INFINITY ? -INFINITY : lse2 * 0.6931471805599453f;
    }
    g_end(tmem, sy, p);
}

// --------------------------------------------------------------------- dQ
template <bool SPLIT, int BS, int MINB>
__global__ void __launch_bounds__(kRowThr, MINB) dq_gtc_kernel(const GParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Geo &g = p.g;
    constexpr int bs = BS;
    constexpr int GB = kGroupKeys / BS;  // blocks per group
    constexpr int NK = kGroupKeys;       // keys per group: the products' N (S, dP) and K (dS K)
    const int Dp = p.Dp, G = g.G, Tq = tile_tokens(G), nrows = Tq * G, parts = SPLIT ? 2 : 1;
    const UnionBuf up = union_buf(g);
    // plan: Q, dO [128][Dp] | K, V [64][Dp] (K also read MN-major by dS K) |
    // dS [128][64] | union | misc
    const uint32_t QB = 128 * Dp * 2, KB = NK * Dp * 2, PB = 128 * kKeyPad * 2;
    uint8_t *q_t = sm, *do_t = q_t + parts * QB, *k_t = do_t + parts * QB, *v_t = k_t + parts * KB;
    uint8_t *ds_t = v_t + parts * KB;
    int *ubuf = (int *)(ds_t + parts * PB);
    uint8_t *misc = (uint8_t *)ubuf + up.bytes;
    Sync sy;
    const uint32_t tmem = g_start(misc, p, sy);
    const int r = threadIdx.x & (kThr - 1), hc = threadIdx.x >> 7;
    int b = 0, kvh = 0, t0 = 0, nvalid = 0;
    qtile_of(g, blockIdx.x, b, kvh, t0, nvalid);
    zero_smem(sm, parts * (2 * QB + 2 * KB + PB));
    if (nvalid > 0)
        qtile_union_cta(g, p.idx, up, ubuf, b, kvh, t0, nvalid);
    __syncthreads();
    const int U = nvalid > 0 ? ubuf[UH_COUNT] : 0, NG = (U + GB - 1) / GB;
    const int *list = union_list(ubuf, up);
    int tl, hh;
    qrow(G, r, tl, hh);
    const bool rvalid = r < nrows && tl < nvalid;
    const int t = t0 + tl, words = (g.nbmax + 31) / 32;
    const int cdiag = rvalid ? kdiag(g, b, t) : -1;
    const int khi = rvalid ? min(cdiag, seq_len_k(g, b) - 1) : -1, klo = key_lo(g, cdiag);
    const uint32_t *my_mask = union_mask(ubuf) + (rvalid ? tl : 0) * words;
    const uint32_t qs = smem_u32(q_t), dos = smem_u32(do_t), ks = smem_u32(k_t), vs = smem_u32(v_t);
    const uint32_t dss = smem_u32(ds_t);
    float l2 = -INFINITY, dl = 0.f;
    {
        const int h = kvh * G + hh;
        RowRegs rr;  // the row of Q (hc = 0) or of dO (hc = 1)
        fetch_row<SPLIT>(g, hc ? p.dO : p.q, !rvalid ? 0 : hc ? o_off(g, b, h, t) : q_off(g, b, h, t), rvalid, rr);
        store_row<SPLIT>(g, rr, hc ? dos : qs, QB, r);
        if (rvalid) {
            const int64_t so = stat_off(g, b, h, t);
            l2 = p.lse[so] * 1.4426950408889634f;
            dl = p.delta[so];
        }
    }
    const uint32_t idS = idesc_bf16(128, NK, false, false), idQ = idesc_bf16(128, Dp, false, true);
    bool ok = true;
    BlockRegs kr, vr;  // the next group's K and V, fetched while the MMAs run
    if (NG > 0) {
        fetch_group<SPLIT, BS, kRowThr>(g, p.k, b, kvh, list, 0, U, kr);
        fetch_group<SPLIT, BS, kRowThr>(g, p.v, b, kvh, list, 0, U, vr);
    }
    for (int gi = 0; gi < NG && ok; ++gi) {
        store_group<SPLIT, kRowThr>(g, kr, ks, KB);
        store_group<SPLIT, kRowThr>(g, vr, vs, KB);
        to_mma();
        if (threadIdx.x == 0)
            product<SPLIT>(tmem + TM_S, qs, 128, QB, ks, NK, KB, idS, Dp / 16, false);
        else if (threadIdx.x == kIssuer2)
            product<SPLIT>(tmem + TM_DP, dos, 128, QB, vs, NK, KB, idS, Dp / 16, false);
        if (gi + 1 < NG) {
            fetch_group<SPLIT, BS, kRowThr>(g, p.k, b, kvh, list, (gi + 1) * GB, U, kr);
            fetch_group<SPLIT, BS, kRowThr>(g, p.v, b, kvh, list, (gi + 1) * GB, U, vr);
        }
        if (!(ok = commit_wait(sy)))
            break;
        // the first key of each block of the group, and whether the row takes it
        int k0s[GB];
        bool sel[GB];
#pragma unroll
        for (int e = 0; e < GB; ++e) {
            const int li = gi * GB + e;
            const int j = li < U ? list[li] : -1;
            k0s[e] = j * bs;
            sel[e] = j >= 0 && rvalid && l2 != -INFINITY && qtile_selects(g, my_mask, klo, khi, j);
        }
        {
            const int c1 = hc * 32;
            float sc[32], dp[32];
            ld_cols<32, 32>(tmem, TM_S + c1, sc, TM_DP + c1, dp);
#pragma unroll
            for (int c0 = 0; c0 < 32; c0 += 8) {
                float dsv[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const int c = c1 + c0 + x, key = k0s[c / bs] + c % bs;
                    const float pv =
                        (sel[c / bs] && key >= klo && key <= khi) ? ex2(sc[c0 + x] * g.scale_l2 - l2) : 0.f;
                    dsv[x] = pv * (dp[c0 + x] - dl);
                }
                put8<SPLIT>(dss, 128, PB, r, c1 + c0, dsv);
            }
        }
        to_mma();
        if (threadIdx.x == 0)  // dQ += dS K, K read MN-major from its plain tile
            product_bmn<SPLIT>(tmem + TM_ACC, dss, 128, PB, ks, NK, KB, idQ, NK / 16, gi > 0);
        ok = commit_wait(sy);
    }
    if (ok) {
        float acc[16];
        const int64_t qo = rvalid ? dq_off(g, b, kvh * G + hh, t) : 0;
        for (int c0 = hc * 16; c0 < g.D; c0 += 32) {
            if (U > 0)
                ld_cols<16>(tmem, TM_ACC + c0, acc);
            if (rvalid)
                out16<SPLIT>(p.dq, qo + c0, acc, g.scale, U > 0);
        }
    }
    g_end(tmem, sy, p);
}

// ------------------------------------------------------------------ dK/dV
// width (columns) of the stacked P / dS tile for blocks of bs keys
constexpr int stacked_pw(int bs) { return 2 * bs <= 64 ? 64 : 2 * bs; }

// One work unit (b, kv head, block j, a run of the block's token list) per
// CTA of two threads per tile row, two CTAs per SM.  Per tile of Tt tokens x
// G heads (128 rows):
//   S = Q K_j^T, dP = dO V_j^T, P and dS per row, then
//   Dp = 64:  [dV^T; dK^T-ish] += [dO^T; Q^T] [P^T; dS^T]^T  (one M = 128 product
//             whose diagonal blocks are dV^T (lanes 0..63, columns 0..bs-1) and
//             dK^T (lanes 64..127, columns bs..2bs-1))
//   Dp = 128: dV^T += dO^T P, dK^T += Q^T dS (two M = 128 products)
// accumulated in TMEM over the unit's tiles; then written out (a whole block)
// or as fp32 partials of a split block.
template <bool SPLIT, int BS>
__global__ void __launch_bounds__(kRowThr, 2) dkdv_gtc_kernel(const GParams p)
{
    const int ui = blockIdx.x;
    if (ui >= p.hdr->n_units)
        return;  // uniform over the CTA: nothing allocated yet
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Geo &g = p.g;
    constexpr int bs = BS;
    // two threads per tile row: thread r + 128 hc forms P and dS for keys
    // hc bs/2 .. hc bs/2 + bs/2 - 1 of row r, reading 16 columns of S and dP
    // at a time (with 16-key blocks both threads read the block's 16)
    constexpr int NH = bs / 2, kCh = NH < 16 ? 16 : NH;
    const int Dp = p.Dp, G = g.G, parts = SPLIT ? 2 : 1;
    const int Tt = tile_tokens(G), nrows = Tt * G;
    const bool stacked = Dp == 64;
    // plan: K, V [bs][Dp] | dO, Q [128][Dp] | P and dS: stacked one [128][PW]
    // tile (row r: P's bs keys, then dS's), else a [128][64] tile each (low
    // parts right after each) | misc.  dO and Q are the K-major A operands of
    // S and dP and, read by columns (MN-major), the A operands of dV^T and
    // dK^T; P and dS are read by columns as their B operands.  Stacked, Q
    // sits right after dO, so [dO^T; Q^T] is one M = 128 operand of two
    // 64-dim chunks parts * QB bytes apart.
    constexpr int PW = stacked_pw(BS);  // stacked P / dS tile width: 2 bs columns, padded to a 64-column chunk
    const uint32_t KB = bs * Dp * 2, QB = 128 * Dp * 2, PB = 128 * (stacked ? PW : kKeyPad) * 2;
    uint8_t *k_t = sm, *v_t = k_t + parts * KB, *do_t = v_t + parts * KB, *q_t = do_t + parts * QB;
    uint8_t *p_t = q_t + parts * QB;                       // P (stacked: P and dS)
    uint8_t *ds_t = p_t + (stacked ? 0 : parts * PB);      // dS (separate)
    uint8_t *misc = p_t + parts * PB * (stacked ? 1 : 2);
    Sync sy;
    const uint32_t tmem = g_start(misc, p, sy);
    const int r = threadIdx.x & (kThr - 1), hc = threadIdx.x >> 7, wq = r >> 5;
    const Unit u = p.units[ui];
    const int b = u.bg / g.Hkv, kvh = u.bg % g.Hkv, j = u.j, k0 = j * bs;
    const int Lk = seq_len_k(g, b), nk = min(bs, Lk - k0);
    zero_smem(sm, (int)(misc - sm));
    __syncthreads();
    const uint32_t ks = smem_u32(k_t), vs = smem_u32(v_t), qs = smem_u32(q_t), dos = smem_u32(do_t);
    const uint32_t ps = smem_u32(p_t), dss = smem_u32(ds_t);
    {  // K (hc = 0) or V (hc = 1)
        BlockRegs kr;
        fetch_block<SPLIT>(g, hc ? p.v : p.k, b, kvh, k0, kr);
        store_block<SPLIT>(g, kr, hc ? vs : ks, KB);
    }
    // Launched (selection) as a programmatic dependent of the kernel before
    // it (the inverse index's fill, or delta with a prebuilt plan): the
    // set-up above read only the unit list, which a launch before that kernel
    // wrote; the token rows and delta are read after this wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the split-block sum launched next may start (it waits for this kernel)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int tl, hh;
    qrow(G, r, tl, hh);
    const int csr0 = g.dense ? dense_first(g, b, j) + u.begin : p.offsets[u.bg * g.nbmax + j] + u.begin;
    const uint32_t idS = idesc_bf16(128, bs, false, false);
    const uint32_t idA = idesc_bf16(128, stacked ? 2 * bs : bs, true, true);
    const int ntiles = (u.count + Tt - 1) / Tt;
    const int h = kvh * G + hh;
    // The row's token in tile ti (-1 past the list), and its dO (hc = 0) or
    // q (hc = 1) row with its LSE and delta: tile ti + 1's token is read
    // while tile ti's S and dP products run, its row while the dV and dK
    // products run, so the loads' latency stays off the tile's chain.  (With
    // 64-key blocks the row is read at the tile's start instead: held across
    // the tile, its registers would spill.)
    constexpr bool kRowAhead = BS < 64;
    auto token_of = [&](int ti) -> int {
        const int pos = ti * Tt + tl;
        return (r < nrows && pos < u.count) ? (g.dense ? csr0 + pos : p.rows[csr0 + pos]) : -1;
    };
    RowRegs rr;
    float lse_raw = 0.f, dl = 0.f;
    auto fetch_row_of = [&](int tk) {
        const bool v = tk >= 0;
        if (hc == 0)
            fetch_row<SPLIT>(g, p.dO, v ? o_off(g, b, h, tk) : 0, v, rr);
        else
            fetch_row<SPLIT>(g, p.q, v ? q_off(g, b, h, tk) : 0, v, rr);
    };
    auto fetch_tile = [&](int tk) {
        const bool v = tk >= 0;
        if (kRowAhead)
            fetch_row_of(tk);
        lse_raw = 0.f;
        dl = 0.f;
        if (v) {
            const int64_t so = stat_off(g, b, h, tk);
            lse_raw = p.lse[so];
            dl = p.delta[so];
        }
    };
    int t = ntiles > 0 ? token_of(0) : -1;
    if (ntiles > 0)
        fetch_tile(t);
    bool ok = true;
    for (int ti = 0; ti < ntiles && ok; ++ti) {
        const bool rvalid = t >= 0;
        const float l2 = rvalid ? lse_raw * 1.4426950408889634f : 0.f;
        // the rows (zeros for rows past the list)
        if (!kRowAhead)
            fetch_row_of(t);
        store_row<SPLIT>(g, rr, hc == 0 ? dos : qs, QB, r);
        to_mma();
        if (threadIdx.x == 0)
            product<SPLIT>(tmem + TM_S, qs, 128, QB, ks, bs, KB, idS, Dp / 16, false);
        else if (threadIdx.x == kIssuer2)
            product<SPLIT>(tmem + TM_DP, dos, 128, QB, vs, bs, KB, idS, Dp / 16, false);
        const int tn = ti + 1 < ntiles ? token_of(ti + 1) : -1;
        if (!(ok = commit_wait(sy)))
            break;
        // the row's keys: from the window's left edge to its diagonal
        const int cdiag = rvalid ? kdiag(g, b, t) : -1;
        const int khi = rvalid ? min(cdiag, Lk - 1) : -1, klo = key_lo(g, cdiag);
        const bool live = rvalid && l2 != -INFINITY;
        {
            const int c1 = NH < 16 ? 0 : hc * NH;
            float sc[kCh], dp[kCh];
            ld_cols<kCh, kCh>(tmem, TM_S + c1, sc, TM_DP + c1, dp);
            // P and dS of this thread's keys, 8 columns per 16-byte store
#pragma unroll
            for (int x0 = 0; x0 < kCh; x0 += 8) {
                if (NH < 16 && x0 / NH != hc)  // x stays a compile-time register index
                    continue;
                float pv[8], dsv[8];
#pragma unroll
                for (int z = 0; z < 8; ++z) {
                    const int x = x0 + z, key = k0 + c1 + x;
                    pv[z] = (live && key >= klo && key <= khi) ? ex2(sc[x] * g.scale_l2 - l2) : 0.f;
                    dsv[z] = pv[z] * (dp[x] - dl);
                }
                put8<SPLIT>(ps, 128, PB, r, c1 + x0, pv);
                put8<SPLIT>(stacked ? ps : dss, 128, PB, r, (stacked ? bs : 0) + c1 + x0, dsv);
            }
        }
        to_mma();
        // [dV^T; dK^T] += [dO^T; Q^T] [P dS] (stacked), else dV^T += dO^T P
        // and dK^T += Q^T dS; K = the tile's 128 rows
        if (threadIdx.x == 0)
            product_mn<SPLIT>(tmem + TM_ACC, dos, stacked ? parts * QB : 128 * 128, QB, ps, 128, PB, idA, 128 / 16,
                              ti > 0);
        else if (threadIdx.x == kIssuer2 && !stacked)
            product_mn<SPLIT>(tmem + TM_ACC2, qs, 128 * 128, QB, dss, 128, PB, idA, 128 / 16, ti > 0);
        if (ti + 1 < ntiles)
            fetch_tile(tn);
        t = tn;
        ok = commit_wait(sy);
    }
    // epilogue: lane r holds dim r of dV^T (stacked: lanes 0..63) and of dK^T
    // (stacked: lanes 64..127, columns bs..2bs-1; else the second accumulator);
    // the two threads of a lane take alternate 16-column pieces of (dV, dK)
    if (ok) {
        const bool direct = u.slot < 0;
        for (int which = 0; which < 2; ++which) {  // 0 dV, 1 dK
            // warp-uniform columns: stacked lane quarters 0-1 read dV's, 2-3 dK's
            int col, d;
            bool mine;
            if (stacked) {
                col = TM_ACC + (wq >= 2 ? bs : 0);
                d = r & 63;
                mine = (which == 0) == (wq < 2);
            } else {
                col = which == 0 ? TM_ACC : TM_ACC2;
                d = r;
                mine = true;
            }
            const float mul = which == 1 ? g.scale : 1.f;
            for (int c1 = 0; c1 < bs; c1 += 16) {
                if (((which * (bs / 16) + c1 / 16) & 1) != hc)
                    continue;
                float ac[16];
                ld_cols<16>(tmem, col + c1, ac);  // every lane: a warp-wide load
                if (!mine || d >= g.D)
                    continue;
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int c = c1 + x;
                    if (c >= nk)
                        break;
                    const float v = ac[x] * mul;
                    if (direct)
                        out_at<SPLIT>(which == 1 ? p.dk : p.dv, dkv_off(g, b, kvh, k0 + c) + d, v);
                    else  // a split block's partial: dK first, then dV (the reduction's order)
                        p.partials[((int64_t)u.slot * 2 + (which == 1 ? 0 : 1)) * bs * g.D + c * g.D + d] = v;
                }
            }
        }
    }
    g_end(tmem, sy, p);
}

// ------------------------------------------------------------ block scores
// The selection step's scores: for row (b, query head h, t) and block j
// complete at t ((j + 1) bs - 1 <= t), p = exp(scale <q, kc_j>) normalised
// over the row's complete blocks; a token's score of block j is the sum of
// p over the G heads of its kv head (0 for blocks not complete at t).
// One CTA of two threads per tile row (each takes 32 of a chunk's 64
// columns) per query tile (Tq tokens x G heads).  The compressed keys of the
// blocks complete at the tile's last row are read in chunks of 64 (the MMA's
// N).  Up to 4 chunks (256 blocks) are resident: the q tile and every chunk
// are loaded at once -- by TMA (bf16 with D a multiple of 64: the q tile as
// boxes of G heads x Tq tokens, head-major rows for BHTD and token-major for
// THD), else by per-thread copies -- all S products go out from two threads
// and stay in TMEM; pass 1 takes each row's maximum and sum, pass 2 forms
// p, stages it in shared memory (row stride 65 floats: writes by rows and
// reads by columns are both conflict-free) and sums each token's G rows.
// Longer rows walk the chunks one at a time and recompute S in pass 2.
constexpr int kScoreThr = 256;  // two threads per tile row
constexpr int kScoreCh = 64;   // compressed keys per chunk
constexpr int kScoreBufs = 4;  // resident chunks at most
constexpr int kPStride = 65;   // floats per staged row

__host__ __device__ inline int score_bufs(int nb)
{
    const int n = (nb + kScoreCh - 1) / kScoreCh;
    return n < 1 ? 1 : n > kScoreBufs ? kScoreBufs : n;
}

// Shared-memory offsets and TMEM columns of the scores kernel.  With every
// tile's chunks resident (nb <= 4 * 64) the staged p goes over the q and
// chunk tiles, and the TMEM holds just the resident chunks' S.
struct ScorePlan {
    uint32_t pbuf_off, misc_off, tmem_cols;
};
__host__ __device__ inline ScorePlan score_plan(int nb, int parts, int Dp)
{
    const int nbuf = score_bufs(nb);
    const bool all_resident = (nb + kScoreCh - 1) / kScoreCh <= nbuf;
    const uint32_t tiles = (uint32_t)parts * (128 + nbuf * kScoreCh) * Dp * 2, pb = 128 * kPStride * 4;
    ScorePlan s;
    s.pbuf_off = all_resident && tiles >= pb ? 0u : tiles;
    s.misc_off = s.pbuf_off + (s.pbuf_off ? pb : tiles);
    s.tmem_cols = all_resident ? (uint32_t)(nbuf == 3 ? 256 : nbuf * kScoreCh) : (uint32_t)kScoreCh;
    return s;
}

template <bool SPLIT, bool TMA>
__global__ void __launch_bounds__(kScoreThr, 3)
    scores_gtc_kernel(const GParams p, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kcmap)
{
    static_assert(!(SPLIT && TMA), "the TMA path moves bf16 tiles");
    extern __shared__ uint8_t smem_raw[];
    // aligned by an offset into the shared array, so that plain accesses
    // through these pointers stay shared-memory accesses
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const Geo &g = p.g;
    constexpr int VEC = In<SPLIT>::VEC, ES = In<SPLIT>::ES;
    const int Dp = p.Dp, G = g.G, Tq = tile_tokens(G), nrows = Tq * G, parts = SPLIT ? 2 : 1, nb = g.nbmax;
    const int nbuf = score_bufs(nb);
    // plan: Q [128][Dp] | nbuf chunk tiles [64][Dp] (each with its low part
    // after it) | staged p [128][kPStride] fp32 -- over the tiles when every
    // tile's chunks are resident (their products are done before p is
    // staged) | misc (+48: the TMA barrier)
    const uint32_t QB = 128 * Dp * 2, CB = kScoreCh * Dp * 2;
    const ScorePlan plan = score_plan(nb, parts, Dp);
    uint8_t *q_t = sm, *c_t = q_t + parts * QB;
    float *pbuf = (float *)(sm + plan.pbuf_off);
    uint8_t *misc = sm + plan.misc_off;
    uint64_t *tbar = (uint64_t *)(misc + 48);
    float *xchg = (float *)(misc + 64);  // [2 halves][2 (m, l)][128 rows]: the rows' statistics
    Sync sy;
    if (TMA && threadIdx.x == 0) {
        mbar_init(tbar, 1);
        prefetch_tmap(&qmap);
        prefetch_tmap(&kcmap);
    }
    const uint32_t tmem = g_start(misc, p, sy, plan.tmem_cols);  // (its barrier-init fence and sync cover tbar too)
    uint32_t tphase = 0;
    // two threads per row: thread (hc, r) takes columns hc*32 .. hc*32+31 of
    // every chunk; warp w reads TMEM lanes 32*(w%4) ..
    const int r = threadIdx.x & (kThr - 1), hc = threadIdx.x >> 7, colh = hc * 32;
    const uint32_t lane_base = tmem + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16);
    int b = 0, kvh = 0, t0 = 0, nvalid = 0;
    qtile_of(g, blockIdx.x, b, kvh, t0, nvalid);
    if (g.D < Dp)  // zero padding columns (every other byte is written below)
        zero_smem(sm, (int)(nbuf * parts * CB + parts * QB));
    __syncthreads();
    // the tile's rows: head-major (row = head * Tq + token) where the BHTD
    // TMA box puts them, else token-major
    const bool head_major = TMA && !g.thd;
    int tl, hh;
    if (head_major) {
        tl = r % Tq;
        hh = r / Tq;
    } else {
        qrow(G, r, tl, hh);
    }
    const bool rvalid = r < nrows && tl < nvalid;
    const int t = t0 + tl;
    const int nc = rvalid ? (t + 1) / g.bs : 0;               // the row's complete blocks
    const int ncmax = nvalid > 0 ? (t0 + nvalid) / g.bs : 0;  // ... of the tile's last row
    const int nch = (ncmax + kScoreCh - 1) / kScoreCh;
    const bool resident = nch <= nbuf;
    const uint32_t qs = smem_u32(q_t), cs = smem_u32(c_t);
    const int nv = g.D / VEC, lnv = __ffs(nv) - 1, nvec = kScoreCh * nv;
    const int halves = g.D / 64;  // TMA boxes per row (64 columns each)
    const uint8_t *kc_bg = (const uint8_t *)p.k + (int64_t)(b * g.Hkv + kvh) * nb * g.D * ES;
    // chunk c of the compressed keys into chunk tile `buf` (rows past nb read as zeros)
    auto fetch_chunk = [&](int c, int buf) {
        const uint32_t dst = cs + buf * parts * CB;
        if constexpr (TMA) {
            if (threadIdx.x == 0)
                for (int h = 0; h < halves; ++h)
                    tma_load_3d(c_t + buf * CB + h * (kScoreCh * 128), &kcmap, tbar, h * 64, c * kScoreCh,
                                b * g.Hkv + kvh);
        } else if constexpr (!SPLIT) {
            for (int e = threadIdx.x; e < nvec; e += kScoreThr) {
                const int row = e >> lnv, j = c * kScoreCh + row, col = (e & (nv - 1)) * VEC;
                cp_async_16(dst + swz(row, col, kScoreCh), kc_bg + ((int64_t)(j < nb ? j : 0) * g.D + col) * ES,
                            j < nb ? 16u : 0u);
            }
        } else {
            for (int e0 = 0; e0 < nvec; e0 += kBlkVec * kScoreThr) {
                uint4 v[kBlkVec];
#pragma unroll
                for (int i = 0; i < kBlkVec; ++i) {
                    const int e = e0 + threadIdx.x + i * kScoreThr, j = c * kScoreCh + (e >> lnv);
                    v[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (e < nvec && j < nb)
                        v[i] = __ldg((const uint4 *)(kc_bg + ((int64_t)j * g.D + (e & (nv - 1)) * VEC) * ES));
                }
#pragma unroll
                for (int i = 0; i < kBlkVec; ++i) {
                    const int e = e0 + threadIdx.x + i * kScoreThr;
                    if (e < nvec)
                        put_vec<SPLIT>(dst, kScoreCh, CB, e >> lnv, (e & (nv - 1)) * VEC, v[i]);
                }
            }
        }
    };
    // thread 0 announces the bytes the TMA loads that follow will bring
    bool tma_pending = false;  // (thread 0) loads announced and not yet seen landing
    auto tma_expect = [&](int chunks, bool with_q) {
        if (TMA && threadIdx.x == 0) {
            mbar_arrive_expect_tx(tbar, (uint32_t)(halves * (chunks * kScoreCh * 128 + (with_q ? nrows * 128 : 0))));
            tma_pending = true;
        }
    };
    // every load issued so far has landed (bounded wait on the TMA barrier)
    auto loads_done = [&]() -> bool {
        if constexpr (TMA) {
            const bool got = mbar_wait(tbar, tphase, sy.ctx);
            if (got) {
                tphase ^= 1;
                tma_pending = false;
            }
            return __syncthreads_and(got) != 0;
        } else {
            if constexpr (!SPLIT) {
                cp_async_commit();
                cp_async_wait<0>();
            }
            return true;
        }
    };
    bool ok = true;
    // the q tile (rows past the tile's tokens are zeros or unused)
    if (resident)
        tma_expect(nch, true);
    else
        tma_expect(1, true);
    if constexpr (TMA) {
        if (threadIdx.x == 0)
            for (int h = 0; h < halves; ++h) {
                if (g.thd)
                    tma_load_3d(q_t + h * (128 * 128), &qmap, tbar, h * 64, kvh * G, g.cu[b] + t0);
                else
                    tma_load_4d(q_t + h * (128 * 128), &qmap, tbar, h * 64, t0, kvh * G, b);
            }
    } else if (hc == 0) {
        const int64_t qo = rvalid ? q_off(g, b, kvh * G + hh, t) : 0;
        if constexpr (!SPLIT) {
            for (int c = 0; c < g.D; c += VEC)
                cp_async_16(qs + swz(r, c, 128), (const uint8_t *)p.q + (qo + c) * ES, rvalid ? 16u : 0u);
        } else {
            for (int i0 = 0; i0 * VEC < g.D; i0 += kRowVec) {
                uint4 v[kRowVec];
#pragma unroll
                for (int i = 0; i < kRowVec; ++i) {
                    const int c = (i0 + i) * VEC;
                    v[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (rvalid && c < g.D)
                        v[i] = __ldg((const uint4 *)((const uint8_t *)p.q + (qo + c) * ES));
                }
#pragma unroll
                for (int i = 0; i < kRowVec; ++i)
                    if ((i0 + i) * VEC < g.D)
                        put_vec<SPLIT>(qs, 128, QB, r, (i0 + i) * VEC, v[i]);
            }
        }
    }
    const uint32_t idS = idesc_bf16(128, kScoreCh, false, false);
    float m = -INFINITY, l = 0.f;
    // pass 1 on columns [col, col + 64) of TMEM holding chunk c: the row's
    // running maximum m and sum l of exp2(scale_l2 s) over its complete blocks
    // this thread's 32 columns of TMEM column block col, as floats
    auto ld32 = [&](uint32_t col, float *out) {
        uint32_t v[32];
        tmem_ld32(lane_base + col + colh, v);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x)
            out[x] = __uint_as_float(v[x]);
    };
    auto stats = [&](int c, uint32_t col) {
        {
            float s[32];
            ld32(col, s);
            float bm = -INFINITY;
#pragma unroll
            for (int x = 0; x < 32; ++x) {
                s[x] = c * kScoreCh + colh + x < nc ? s[x] * g.scale_l2 : -INFINITY;
                bm = fmaxf(bm, s[x]);
            }
            if (bm != -INFINITY) {
                const float mn = fmaxf(m, bm);
                float sum = 0.f;
#pragma unroll
                for (int x = 0; x < 32; ++x)
                    sum += ex2(s[x] - mn);
                l = l * ex2(m - mn) + sum;
                m = mn;
            }
        }
    };
    // S of chunk c from chunk tile `buf` into TMEM columns [col, col + 64)
    auto s_product = [&](int c, int buf, uint32_t col) {
        product<SPLIT>(tmem + col, qs, 128, QB, cs + buf * parts * CB, kScoreCh, CB, idS, Dp / 16, false);
    };
    if (resident) {
        for (int c = 0; c < nch; ++c)
            fetch_chunk(c, c);
        ok = loads_done();
        to_mma();
        if (ok && (threadIdx.x == 0 || threadIdx.x == kIssuer2))  // chunks split between the two issuing threads
            for (int c = threadIdx.x == 0 ? 0 : 1; c < nch; c += 2)
                s_product(c, c, c * kScoreCh);
        ok = commit_wait(sy) && ok;
        for (int c = 0; c < nch && ok; ++c)
            stats(c, c * kScoreCh);
    } else {
        for (int c = 0; c < nch && ok; ++c) {
            if (c > 0)
                tma_expect(1, false);
            fetch_chunk(c, 0);
            ok = loads_done();
            if (!ok)
                break;
            to_mma();
            if (threadIdx.x == 0)
                s_product(c, 0, 0);
            ok = commit_wait(sy);
            if (ok)
                stats(c, 0);
        }
    }
    // the row's statistics over both halves of its columns
    xchg[(hc * 2) * kThr + r] = m;
    xchg[(hc * 2 + 1) * kThr + r] = l;
    __syncthreads();
    {
        const float mo = xchg[((1 - hc) * 2) * kThr + r], lo = xchg[((1 - hc) * 2 + 1) * kThr + r];
        const float mn = fmaxf(m, mo);
        if (mn != -INFINITY) {
            l = (m != -INFINITY ? l * ex2(m - mn) : 0.f) + (mo != -INFINITY ? lo * ex2(mo - mn) : 0.f);
            m = mn;
        }
    }
    const float lse2 = l > 0.f ? m + log2f(l) : INFINITY;  // +inf: no complete block, p = 0
    // pass 2: p per row, staged; each token's G rows summed into its scores
    for (int c = 0; c < nch && ok; ++c) {
        uint32_t col = c * kScoreCh;
        if (!resident) {
            col = 0;
            tma_expect(1, false);
            fetch_chunk(c, 0);
            ok = loads_done();
            if (!ok)
                break;
            to_mma();
            if (threadIdx.x == 0)
                s_product(c, 0, 0);
            ok = commit_wait(sy);
            if (!ok)
                break;
        }
        {
            float s[32];
            ld32(col, s);
#pragma unroll
            for (int x = 0; x < 32; ++x)
                pbuf[r * kPStride + colh + x] = c * kScoreCh + colh + x < nc ? ex2(s[x] * g.scale_l2 - lse2) : 0.f;
        }
        __syncthreads();
        {
            // thread: column jj, tokens tk0, tk0 + 2, ...
            const int jj = threadIdx.x % kScoreCh, j = c * kScoreCh + jj;
            const int rs = head_major ? Tq : 1, ts = head_major ? 1 : G;  // row steps per head / token
            if (j < nb)
                for (int tk = threadIdx.x / kScoreCh; tk < nvalid; tk += kScoreThr / kScoreCh) {
                    const float *col = pbuf + tk * ts * kPStride + jj;
                    float sum = 0.f;
                    for (int h2 = 0; h2 < G; ++h2)
                        sum += col[h2 * rs * kPStride];
                    p.scores[index_row(g, b, kvh, t0 + tk) * nb + j] = sum;
                }
        }
        tc_fence_before();  // this chunk's TMEM reads and staged rows are done before the next
        __syncthreads();
        tc_fence_after();
    }
    // zeros for the blocks past the tile's chunks
    if (ok) {
        const int j0 = nch * kScoreCh, rest = nb - j0;
        for (int o = threadIdx.x; rest > 0 && o < nvalid * rest; o += kScoreThr)
            p.scores[index_row(g, b, kvh, t0 + o / rest) * nb + j0 + o % rest] = 0.f;
    }
    if constexpr (!TMA && !SPLIT)
        cp_async_wait<0>();  // nothing left in flight after an early exit
    if (TMA && tma_pending) {
        // (thread 0, after a wait gave up) the TMA loads already issued land
        // before the CTA exits, within the wait limit again
        volatile int never[2] = {0, sy.ctx[1]};
        mbar_wait(tbar, tphase, never);
    }
    g_end(tmem, sy, p, plan.tmem_cols);
}

constexpr int kSmemLimit = 232448;

template <typename K> bool smem_ok(K kernel, size_t bytes)
{
    if (bytes > (size_t)kSmemLimit)
        return false;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
}

size_t union_bytes(const Geo &g) { return union_buf(g).bytes; }

// the instance of a kernel for the element type and the block size (16, 32 or 64)
using GKernel = void (*)(const GParams);
template <template <bool, int> class K> GKernel pick(int dtype, int bs)
{
    if (dtype == NSA_DTYPE_F32)
        return bs == 16 ? K<true, 16>::fn : bs == 32 ? K<true, 32>::fn : K<true, 64>::fn;
    return bs == 16 ? K<false, 16>::fn : bs == 32 ? K<false, 32>::fn : K<false, 64>::fn;
}
template <bool S, int B> struct FwdK1 {
    static constexpr GKernel fn = fwd_gtc_kernel<S, B, 1>;
};
template <bool S, int B> struct FwdK2 {
    static constexpr GKernel fn = fwd_gtc_kernel<S, B, 2>;
};
template <bool S, int B> struct DqK1 {
    static constexpr GKernel fn = dq_gtc_kernel<S, B, 1>;
};
template <bool S, int B> struct DqK2 {
    static constexpr GKernel fn = dq_gtc_kernel<S, B, 2>;
};
template <bool S, int B> struct DkdvK {
    static constexpr GKernel fn = dkdv_gtc_kernel<S, B>;
};

cudaError_t launch_g(GKernel k, int grid, size_t smem, const GParams &p, cudaStream_t st, int threads = kThr,
                     bool dependent = false)
{
    if (!smem_ok(k, smem))
        return cudaErrorInvalidValue;
    if (dependent)
        return launch_dependent(k, dim3(grid), dim3(threads), smem, st, p);
    k<<<grid, threads, smem, st>>>(p);
    return cudaGetLastError();
}

GParams base_params(const Geo &g, int dtype)
{
    GParams p;
    memset(&p, 0, sizeof(p));
    p.g = g;
    p.Dp = g.D <= 64 ? 64 : 128;
    p.wait_us = wait_test().wait_us;
    (void)dtype;
    return p;
}

}  // namespace

bool gtc_supported(const Geo &g, int dtype)
{
    if (g.G < 1 || g.G > kRows || !qtile_shape_ok(g))
        return false;
    if (g.bs != 16 && g.bs != 32 && g.bs != 64)
        return false;
    if (dtype == NSA_DTYPE_BF16)
        return g.D == 32 || g.D == 64 || g.D == 128;
    return g.D == 32 || g.D == 64;  // fp32: split precision
}

bool scores_gtc_supported(const Geo &g, int dtype)
{
    return g.G >= 1 && g.G <= kRows && (g.D == 32 || g.D == 64 || g.D == 128) &&
           (dtype == NSA_DTYPE_BF16 || dtype == NSA_DTYPE_F32);
}

cudaError_t launch_scores_gtc(const Geo &g, const void *q, const void *kc, float *scores, int dtype, int *err,
                              cudaStream_t st)
{
    GParams p = base_params(g, dtype);
    p.q = q;
    p.k = kc;
    p.scores = scores;
    p.err = err;
    const int Tq = tile_tokens(g.G);
    p.ntiles = ((g.T + Tq - 1) / Tq) * g.B * g.Hkv;
    const int parts = dtype == NSA_DTYPE_F32 ? 2 : 1;
    const size_t smem = 1024 + (size_t)score_plan(g.nbmax, parts, p.Dp).misc_off + 64 + 4 * kThr * 4;
    if (p.ntiles < 1)
        return cudaSuccess;
    CUtensorMap qmap, kcmap;
    memset(&qmap, 0, sizeof(qmap));
    memset(&kcmap, 0, sizeof(kcmap));
    // TMA tiles for bf16 with D a multiple of 64: the q tile as one box of
    // G heads x Tq tokens per 64 columns, a chunk of 64 compressed keys
    bool tma = dtype == NSA_DTYPE_BF16 && g.D % 64 == 0;
    if (tma) {
        const uint64_t dims[3] = {(uint64_t)g.D, (uint64_t)g.nbmax, (uint64_t)g.B * g.Hkv};
        const uint64_t strides[2] = {(uint64_t)g.D * 2, (uint64_t)g.nbmax * g.D * 2};
        const uint32_t box[3] = {64, (uint32_t)kScoreCh, 1};
        tma = make_tmap(&qmap, q, g, g.Hq, Tq, g.G, g.sq) && make_tmap_3d(&kcmap, kc, dims, strides, box);
    }
    void (*k)(const GParams, const CUtensorMap, const CUtensorMap) =
        dtype == NSA_DTYPE_F32 ? scores_gtc_kernel<true, false>
        : tma                  ? scores_gtc_kernel<false, true>
                               : scores_gtc_kernel<false, false>;
    if (!smem_ok(k, smem))
        return cudaErrorInvalidValue;
    k<<<p.ntiles, kScoreThr, smem, st>>>(p, qmap, kcmap);
    return cudaGetLastError();
}

cudaError_t launch_fwd_gtc(const Geo &g, const void *q, const void *k, const void *v, const int *idx, void *o,
                           float *lse, int dtype, int *err, cudaStream_t st)
{
    GParams p = base_params(g, dtype);
    p.q = q;
    p.k = k;
    p.v = v;
    p.idx = idx;
    p.o = o;
    p.lse_out = lse;
    p.err = err;
    const int Tq = tile_tokens(g.G);
    p.ntiles = ((g.T + Tq - 1) / Tq) * g.B * g.Hkv;
    const int parts = dtype == NSA_DTYPE_F32 ? 2 : 1;
    const size_t smem = 1024 + parts * (size_t)(128 * p.Dp * 2 + 2 * kGroupKeys * p.Dp * 2 + 128 * kKeyPad * 2) +
                        union_bytes(g) + 64 + 4 * kThr * 4;
    if (p.ntiles < 1)
        return cudaSuccess;
    // two CTAs per SM once the grid has more tiles than SMs (measured: T = 8192
    // bf16 D = 64 forward 1.16 -> 0.75 ms; at one tile per SM the full
    // register budget is the faster)
    const GKernel kern = p.ntiles > num_sms() ? pick<FwdK2>(dtype, g.bs) : pick<FwdK1>(dtype, g.bs);
    return launch_g(kern, p.ntiles, smem, p, st, kRowThr);
}

cudaError_t launch_dq_gtc(const Geo &g, const void *q, const void *k, const void *v, const void *dO,
                          const float *lse, const float *delta, const int *idx, void *dq, int dtype, int *err,
                          cudaStream_t st)
{
    GParams p = base_params(g, dtype);
    p.q = q;
    p.k = k;
    p.v = v;
    p.dO = dO;
    p.lse = lse;
    p.delta = delta;
    p.idx = idx;
    p.dq = dq;
    p.err = err;
    const int Tq = tile_tokens(g.G);
    p.ntiles = ((g.T + Tq - 1) / Tq) * g.B * g.Hkv;
    const int parts = dtype == NSA_DTYPE_F32 ? 2 : 1;
    const size_t smem = 1024 +
                        parts * (size_t)(2 * 128 * p.Dp * 2 + 2 * kGroupKeys * p.Dp * 2 + 128 * kKeyPad * 2) +
                        union_bytes(g) + 64;
    if (p.ntiles < 1)
        return cudaSuccess;
    // as the forward, but split precision keeps one CTA per SM: its register
    // cap for two spills and measured slower at every size
    const bool two = dtype == NSA_DTYPE_BF16 && p.ntiles > num_sms();
    const GKernel kern = two ? pick<DqK2>(dtype, g.bs) : pick<DqK1>(dtype, g.bs);
    return launch_g(kern, p.ntiles, smem, p, st, kRowThr);
}

cudaError_t launch_dkdv_gtc(const Geo &g, const void *q, const void *k, const void *v, const void *dO,
                            const float *lse, const float *delta, const int *offsets, const int *rows,
                            const Unit *units, const WsHeader *hdr, int max_units, float *partials, void *dk,
                            void *dv, int dtype, int *err, cudaStream_t st)
{
    GParams p = base_params(g, dtype);
    p.q = q;
    p.k = k;
    p.v = v;
    p.dO = dO;
    p.lse = lse;
    p.delta = delta;
    p.offsets = offsets;
    p.rows = rows;
    p.units = units;
    p.hdr = hdr;
    p.partials = partials;
    p.dk = dk;
    p.dv = dv;
    p.err = err;
    const int parts = dtype == NSA_DTYPE_F32 ? 2 : 1;
    const bool stacked = p.Dp == 64;
    const size_t tiles = (size_t)2 * g.bs * p.Dp * 2 + 2 * 128 * p.Dp * 2 +
                         (stacked ? (size_t)128 * stacked_pw(g.bs) * 2 : (size_t)2 * 128 * kKeyPad * 2);
    const size_t smem = 1024 + parts * tiles + 64;
    if (max_units < 1)
        return cudaSuccess;
    // a programmatic dependent of the inverse index's fill (or, with a plan,
    // of delta); the dense entry's unit list comes from the kernel just
    // before (the scan), so that launch waits for it in full
    return launch_g(pick<DkdvK>(dtype, g.bs), max_units, smem, p, st, kRowThr, !g.dense);
}

}  // namespace nsa
