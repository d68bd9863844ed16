// k_prep.cu -- the memory-bound steps around the attention kernels:
//   * do_dot: delta_t = sum_d dO_td * O_td (the do_dot kernel of the backward
//     chain on the cuDNN-frontend pull-request page);
//   * index validation;
//   * the block -> token inverse index (count, scan, ordered fill) that lets
//     dK/dV accumulate per kv block without atomics on data;
//   * the fixed-order reduction of split dK/dV blocks;
//   * the (query row, key) pair count used for effective-FLOP reporting.
#include "launch.h"
#include "tc_common.cuh"

namespace nsa {

namespace {

constexpr int kThreads = 256;

inline int grid_for(int64_t n, int per_block, int cap = 152 * 32)
{
    int64_t b = (n + per_block - 1) / per_block;
    if (b < 1)
        b = 1;
    if (b > cap)
        b = cap;
    return (int)b;
}

// ---------------------------------------------------------------- do_dot
// delta uses the row order of lse (BHTD (b*Hq + h)*T + t, THD token*Hq + h);
// each row's D-vector of o and dO sits where the strides of o put it, so the
// kernel is a segmented dot product over rows.
// blocks blk of nblk (grid-stride); each warp takes kDotU row groups per
// step, so that 2 * kDotU 16-byte loads per thread are in flight
constexpr int kDotU = 4;
// blocks of the dot (16 per SM of 152: warps loop over several row groups;
// a grid of one short-lived block per 64 rows measured ~6% slower)
constexpr int kDotBlocks = 152 * 16;
template <typename T, bool LIN>
__device__ __forceinline__ void do_dot_rows(const Geo &g, const T *__restrict__ o, const T *__restrict__ dO,
                                            float *__restrict__ out, int64_t nrows, int D, int blk, int nblk)
{
    constexpr int VEC = 16 / sizeof(T);
    const int tpr = D / VEC;  // threads per row (power of two, <= 32)
    const int lane = threadIdx.x & 31;
    const int sub = lane / tpr, part = lane % tpr, rpw = 32 / tpr;
    const int64_t warp = ((int64_t)blk * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)nblk * blockDim.x) >> 5;
    for (int64_t r0 = warp * kDotU * rpw; r0 < nrows; r0 += nwarps * kDotU * rpw) {
        uint4 a[kDotU], b[kDotU];
#pragma unroll
        for (int u = 0; u < kDotU; ++u) {
            const int64_t r = r0 + u * rpw + sub;
            a[u] = b[u] = make_uint4(0, 0, 0, 0);
            if (r < nrows) {
                const int64_t off = (LIN ? r * D : qrow_off(g, g.so, r)) + part * VEC;
                a[u] = __ldcs(reinterpret_cast<const uint4 *>(o + off));
                b[u] = __ldcs(reinterpret_cast<const uint4 *>(dO + off));
            }
        }
#pragma unroll
        for (int u = 0; u < kDotU; ++u) {
            const int64_t r = r0 + u * rpw + sub;
            const T *ea = reinterpret_cast<const T *>(&a[u]);
            const T *eb = reinterpret_cast<const T *>(&b[u]);
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < VEC; ++i)
                acc = fmaf(to_f(ea[i]), to_f(eb[i]), acc);
            for (int off = tpr >> 1; off > 0; off >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (r < nrows && part == 0)
                out[r] = acc;
        }
    }
}

// LIN: dense o/dO (row r at r * D), chosen on the host so that each kernel
// holds one addressing scheme (the strided one's divisions would raise the
// dense kernel's register count and cut the loads it keeps in flight)
template <typename T, bool LIN>
__global__ void __launch_bounds__(kThreads) do_dot_kernel(Geo g, const T *__restrict__ o, const T *__restrict__ dO,
                                                          float *__restrict__ out, int64_t nrows, int D)
{
    do_dot_rows<T, LIN>(g, o, dO, out, nrows, D, blockIdx.x, gridDim.x);
}

// decode a linear index-row number into (b, kvh, t)
__device__ __forceinline__ void decode_idx_row(const Geo &g, int64_t lin, int &b, int &kvh, int &t)
{
    if (g.thd) {
        kvh = (int)(lin % g.Hkv);
        int tok = (int)(lin / g.Hkv);
        b = seq_of_token(g, tok);
        t = tok - g.cu[b];
    } else {
        t = (int)(lin % g.T);
        int64_t bk = lin / g.T;
        kvh = (int)(bk % g.Hkv);
        b = (int)(bk / g.Hkv);
    }
}

// 0 = use, 1 = padding, 2 = invalid (reported), 3 = repeat (reported)
// slot s of an index row: 0 use it, 1 padding (-1), 2 out of range or in the
// future, 3 a repeat of an earlier slot
__device__ __forceinline__ int classify(const int *row, int s, int t, int bs, int nbmax)
{
    const int j = row[s];
    if (j == -1)
        return 1;
    if (j < -1 || j > t / bs || j >= nbmax)
        return 2;
    for (int s2 = 0; s2 < s; ++s2)
        if (row[s2] == j)
            return 3;
    return 0;
}

// The slots of one index row that name a block to use (bit s set), each
// block once; `bad` reports a slot that is out of range, in the future or a
// repeat of an earlier slot (-1 is padding).  The row is read into registers
// once (S <= 32).
__device__ __forceinline__ unsigned row_slots(const int *row, int S, int t, int bs, int nbmax, bool &bad)
{
    int v[32];
#pragma unroll
    for (int s = 0; s < 32; ++s)
        v[s] = s < S ? row[s] : -1;
    const int jmax = min(t / bs, nbmax - 1);
    unsigned m = 0u;
    bool b = false;
#pragma unroll
    for (int s = 0; s < 32; ++s) {
        if (s >= S)
            break;
        const int j = v[s];
        if (j == -1)
            continue;
        bool dup = false;
#pragma unroll
        for (int s2 = 0; s2 < s; ++s2)
            dup |= v[s2] == j;
        if (j < 0 || j > jmax || dup)
            b = true;
        else
            m |= 1u << s;
    }
    bad = b;
    return m;
}

__global__ void __launch_bounds__(kThreads) validate_kernel(Geo g, const int *__restrict__ idx,
                                                            int *err)
{
    // the forward kernel launched next does not wait for this check
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t n = (int64_t)g.ntok * g.Hkv;
    for (int64_t lin = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; lin < n;
         lin += (int64_t)gridDim.x * blockDim.x) {
        int b, kvh, t;
        decode_idx_row(g, lin, b, kvh, t);
        const int *row = idx_row(g, idx, b, kvh, t);
        bool bad = false;
        if (g.S <= 32)
            row_slots(row, g.S, t, g.bs, g.nbmax, bad);
        else
            for (int s = 0; s < g.S; ++s)
                bad |= classify(row, s, t, g.bs, g.nbmax) >= 2;
        if (bad)
            set_error(err, NSA_ERR_BAD_INDEX);
    }
}

__global__ void __launch_bounds__(kThreads) csr_count_kernel(Geo g, const int *__restrict__ idx,
                                                             int *__restrict__ counts, int *err)
{
    const int64_t n = (int64_t)g.ntok * g.Hkv;
    for (int64_t lin = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; lin < n;
         lin += (int64_t)gridDim.x * blockDim.x) {
        int b, kvh, t;
        decode_idx_row(g, lin, b, kvh, t);
        const int *row = idx_row(g, idx, b, kvh, t);
        int *cnt = counts + ((int64_t)b * g.Hkv + kvh) * g.nbmax;
        bool bad = false;
        if (g.S <= 32) {
            for (unsigned m = row_slots(row, g.S, t, g.bs, g.nbmax, bad); m; m &= m - 1u)
                atomicAdd(&cnt[row[__ffs(m) - 1]], 1);
        } else {
            for (int s = 0; s < g.S; ++s) {
                const int c = classify(row, s, t, g.bs, g.nbmax);
                if (c == 0)
                    atomicAdd(&cnt[row[s]], 1);
                bad |= c >= 2;
            }
        }
        if (bad)
            set_error(err, NSA_ERR_BAD_INDEX);
    }
}

// exclusive scan of one int per thread over a 1024-thread block
__device__ __forceinline__ int block_scan_excl(int v, int &total, int *sm)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        sm[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = sm[lane];
        int z = s;
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, z, off);
            if (lane >= off)
                z += y;
        }
        sm[32 + lane] = z - s;  // exclusive prefix of warp totals
        if (lane == 31)
            sm[64] = z;
    }
    __syncthreads();
    const int r = sm[32 + w] + x - v;
    total = sm[64];
    __syncthreads();
    return r;
}

// One block of 1024 threads: offsets, the unit list (full-size chunks
// first, then the shorter tails, longest first, so that the dK/dV kernel's
// snake schedule of units over CTAs starts with the longest work and ends
// balanced) and the per-block chunk/partial-slot table.
__global__ void __launch_bounds__(1024) csr_scan_kernel(Geo g, const int *__restrict__ counts,
                                                        int *__restrict__ offsets,
                                                        Unit *__restrict__ units,
                                                        int *__restrict__ blk_nchunk,
                                                        int *__restrict__ blk_slot, WsHeader *hdr,
                                                        int chunk)
{
    // The index-build kernels (count, prefix, scan, fill) launch as
    // programmatic dependents of the kernel before each and let the next one
    // launch at once: each waits here, before reading anything, for the one
    // before it to complete, so only the launches overlap.  The dense
    // entries follow the scan with the persistent dK/dV kernel, whose CTA on
    // this kernel's SM would then start late and end the last: there the next
    // kernel launches when this one ends.
    if (!g.dense)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Tails (each block's last, partial chunk) go after the full chunks,
    // longest first by kTailBins bins (stable within a bin), so that the
    // dK/dV kernel's snake assignment of units to CTAs balances their work.
    constexpr int kTailBins = 16;
    __shared__ int sm[80];
    __shared__ int wbin[32][kTailBins];
    __shared__ int binbase[kTailBins];
    const int n = g.B * g.Hkv * g.nbmax;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    auto block_count = [&](int i) {
        if (i >= n)
            return 0;
        if (g.dense) {
            const int b = i / (g.Hkv * g.nbmax), j = i % g.nbmax;
            return dense_count(g, b, j);
        }
        return counts[i];
    };
    auto tail_bin = [&](int cnt) {
        const int r = cnt % chunk;  // tail length, 1 .. chunk-1
        return r ? (kTailBins - 1) - (int)(((int64_t)(r - 1) * kTailBins) / chunk) : -1;
    };
    // pass 1: totals of full chunks (to place the tails after them) and the
    // tails' bin sizes
    if (threadIdx.x < kTailBins)
        binbase[threadIdx.x] = 0;
    __syncthreads();
    int full_total = 0;
    for (int base = 0; base < n; base += 1024) {
        const int cnt = block_count(base + threadIdx.x);
        const int bin = tail_bin(cnt);
        if (bin >= 0)
            atomicAdd(&binbase[bin], 1);
        int tot;
        block_scan_excl(cnt / chunk, tot, sm);
        full_total += tot;
    }
    __syncthreads();
    if (threadIdx.x == 0) {  // bin sizes -> first position of each bin
        int run = 0;
        for (int k = 0; k < kTailBins; ++k) {
            const int c = binbase[k];
            binbase[k] = run;
            run += c;
        }
    }
    __syncthreads();
    int c_off = 0, c_full = 0, c_tail = 0, c_slot = 0;
    for (int base = 0; base < n; base += 1024) {
        const int i = base + threadIdx.x;
        int b = 0, kvh = 0, j = 0;
        const int cnt = block_count(i);
        if (i < n) {
            j = i % g.nbmax;
            kvh = (i / g.nbmax) % g.Hkv;
            b = i / (g.Hkv * g.nbmax);
        }
        const int nfull = cnt / chunk, tail = (cnt % chunk) ? 1 : 0, nch = nfull + tail;
        int t_off, t_full, t_tail, t_slot;
        const int p_off = block_scan_excl(cnt, t_off, sm);
        const int p_full = block_scan_excl(nfull, t_full, sm);
        block_scan_excl(tail, t_tail, sm);
        const int p_slot = block_scan_excl(nch >= 2 ? nch : 0, t_slot, sm);
        // rank of this tail among the tails of its bin, in block order
        const int bin = tail_bin(cnt);
        for (int x = threadIdx.x; x < 32 * kTailBins; x += blockDim.x)
            (&wbin[0][0])[x] = 0;
        __syncthreads();
        const unsigned same = __match_any_sync(0xffffffffu, bin);
        const int rank_w = __popc(same & ((1u << lane) - 1u));
        if (bin >= 0 && rank_w == 0)
            wbin[w][bin] = __popc(same);
        __syncthreads();
        if (w < kTailBins) {  // warp k: exclusive scan of bin k over the 32 warps
            const int v = wbin[lane][w];
            int x = v;
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off)
                    x += y;
            }
            wbin[lane][w] = binbase[w] + x - v;
            __syncwarp();
            if (lane == 31)
                binbase[w] += x;
        }
        __syncthreads();
        if (i < n) {
            offsets[i] = c_off + p_off;
            blk_nchunk[i] = nch;
            const int slot0 = nch >= 2 ? c_slot + p_slot : -1;
            blk_slot[i] = slot0;
            const int bg = b * g.Hkv + kvh;
            for (int c = 0; c < nfull; ++c) {
                Unit u;
                u.bg = bg;
                u.j = j;
                u.begin = c * chunk;
                u.count = chunk;
                u.slot = slot0 >= 0 ? slot0 + c : -1;
                u.pad0 = u.pad1 = u.pad2 = 0;
                units[c_full + p_full + c] = u;
            }
            if (tail) {
                Unit u;
                u.bg = bg;
                u.j = j;
                u.begin = nfull * chunk;
                u.count = cnt - nfull * chunk;
                u.slot = slot0 >= 0 ? slot0 + nfull : -1;
                u.pad0 = u.pad1 = u.pad2 = 0;
                units[full_total + wbin[w][bin] + rank_w] = u;
            }
        }
        c_off += t_off;
        c_full += t_full;
        c_tail += t_tail;
        c_slot += t_slot;
        __syncthreads();  // wbin is cleared for the next round
    }
    if (threadIdx.x == 0) {
        offsets[n] = c_off;
        hdr->n_units = full_total + c_tail;
    }
}

// One block per (b, kvh, j): walk the tokens that may select block j in
// ascending order and append those that do.  Ascending order comes from the
// block-wide ballot prefix, so the list is the same on every run.
__global__ void __launch_bounds__(kThreads) csr_fill_kernel(Geo g, const int *__restrict__ idx,
                                                            const int *__restrict__ offsets,
                                                            int *__restrict__ rows)
{
    __shared__ int warp_tot[kThreads / 32];
    __shared__ int carry;
    const int i = blockIdx.x;
    const int j = i % g.nbmax, kvh = (i / g.nbmax) % g.Hkv, b = i / (g.Hkv * g.nbmax);
    const int begin = offsets[i], cnt = offsets[i + 1] - begin;
    if (cnt == 0)
        return;
    const int L = seq_len(g, b);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (threadIdx.x == 0)
        carry = 0;
    __syncthreads();
    for (int t0 = j * g.bs; t0 < L; t0 += kThreads) {
        const int t = t0 + threadIdx.x;
        const bool sel = t < L && row_selects(g, idx, b, kvh, t, j);
        const unsigned m = __ballot_sync(0xffffffffu, sel);
        if (lane == 0)
            warp_tot[w] = __popc(m);
        __syncthreads();
        int before = carry;
        for (int x = 0; x < w; ++x)
            before += warp_tot[x];
        if (sel) {
            const int pos = before + __popc(m & ((1u << lane) - 1u));
            if (pos < cnt)
                rows[begin + pos] = t;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int s = 0;
            for (int x = 0; x < kThreads / 32; ++x)
                s += warp_tot[x];
            carry += s;
        }
        __syncthreads();
    }
}

// dK/dV of blocks whose token list was split over several units: the sum of
// the units' fp32 partials in unit order (deterministic); blocks nobody
// selected get zeros.  One CTA per (b, kv head, block, quarter of its keys);
// a thread takes 4 consecutive dims of one key.
template <typename T>
__global__ void __launch_bounds__(kThreads) dkdv_reduce_kernel(Geo g, const int *__restrict__ nchunk,
                                                               const int *__restrict__ slot,
                                                               const float *__restrict__ partials,
                                                               T *__restrict__ dk, T *__restrict__ dv)
{
    // (other shapes) a programmatic dependent of the dK/dV kernel: nothing is
    // read before it completes
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int i = blockIdx.x >> 2, quarter = blockIdx.x & 3;
    const int nch = nchunk[i];
    if (nch == 1)
        return;  // written directly by the dK/dV kernel
    const int j = i % g.nbmax, kvh = (i / g.nbmax) % g.Hkv, b = i / (g.Hkv * g.nbmax);
    const int L = seq_len_k(g, b);
    const int k0 = j * g.bs;
    if (k0 >= L)
        return;
    const int nkeys = min(g.bs, L - k0);
    const int64_t per = (int64_t)g.bs * g.D;
    const int kq = g.bs / 4, d4 = g.D / 4;
    const float *base = partials + (nch >= 2 ? (int64_t)slot[i] * 2 * per : 0);
    for (int e = threadIdx.x; e < kq * d4; e += blockDim.x) {
        const int kk = quarter * kq + e / d4, d = (e % d4) * 4;
        if (kk >= nkeys)
            continue;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), c = a;
        const float *p = base + kk * g.D + d;
        int s = 0;
        for (; s + 2 <= nch; s += 2) {  // fixed order: deterministic
            const float4 a0 = *reinterpret_cast<const float4 *>(p + (int64_t)s * 2 * per);
            const float4 c0 = *reinterpret_cast<const float4 *>(p + (int64_t)s * 2 * per + per);
            const float4 a1 = *reinterpret_cast<const float4 *>(p + (int64_t)(s + 1) * 2 * per);
            const float4 c1 = *reinterpret_cast<const float4 *>(p + (int64_t)(s + 1) * 2 * per + per);
            a.x += a0.x; a.y += a0.y; a.z += a0.z; a.w += a0.w;
            c.x += c0.x; c.y += c0.y; c.z += c0.z; c.w += c0.w;
            a.x += a1.x; a.y += a1.y; a.z += a1.z; a.w += a1.w;
            c.x += c1.x; c.y += c1.y; c.z += c1.z; c.w += c1.w;
        }
        if (s < nch) {
            const float4 a0 = *reinterpret_cast<const float4 *>(p + (int64_t)s * 2 * per);
            const float4 c0 = *reinterpret_cast<const float4 *>(p + (int64_t)s * 2 * per + per);
            a.x += a0.x; a.y += a0.y; a.z += a0.z; a.w += a0.w;
            c.x += c0.x; c.y += c0.y; c.z += c0.z; c.w += c0.w;
        }
        const int64_t off = dkv_off(g, b, kvh, k0 + kk) + d;
        dk[off] = from_f<T>(a.x);
        dk[off + 1] = from_f<T>(a.y);
        dk[off + 2] = from_f<T>(a.z);
        dk[off + 3] = from_f<T>(a.w);
        dv[off] = from_f<T>(c.x);
        dv[off + 1] = from_f<T>(c.y);
        dv[off + 2] = from_f<T>(c.z);
        dv[off + 3] = from_f<T>(c.w);
    }
}

__global__ void __launch_bounds__(kThreads) count_pairs_kernel(Geo g, const int *__restrict__ idx,
                                                               unsigned long long *out)
{
    const int64_t n = (int64_t)g.ntok * g.Hkv;
    unsigned long long local = 0;
    for (int64_t lin = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; lin < n;
         lin += (int64_t)gridDim.x * blockDim.x) {
        int b, kvh, t;
        decode_idx_row(g, lin, b, kvh, t);
        const int *row = idx_row(g, idx, b, kvh, t);
        auto add = [&](int j) { local += (unsigned long long)g.G * (min((j + 1) * g.bs - 1, t) - j * g.bs + 1); };
        if (g.S <= 32) {
            bool bad;
            for (unsigned m = row_slots(row, g.S, t, g.bs, g.nbmax, bad); m; m &= m - 1u)
                add(row[__ffs(m) - 1]);
        } else {
            for (int s = 0; s < g.S; ++s)
                if (classify(row, s, t, g.bs, g.nbmax) == 0)
                    add(row[s]);
        }
    }
    for (int off = 16; off > 0; off >>= 1)
        local += __shfl_xor_sync(0xffffffffu, local, off);
    if ((threadIdx.x & 31) == 0 && local)
        atomicAdd(out, local);
}

// ---- inverse index by 32-token chunks ------------------------------------
// chunk_counts[(bg * nbmax + j) * nchunks + c] = tokens of chunk c (tokens
// 32c .. 32c+31) selecting block j, turned in place into an exclusive prefix
// over c.  The fill gives each (token, block) its rank among the chunk's
// earlier tokens with a per-block lane mask, so every list comes out in
// ascending token order (deterministic, no ordering by atomics).
constexpr int kChunkTok = 32;
constexpr int kFillWarps = 4;

// valid slots of a row, each block counted once (bit s set = use slot s)
__device__ __forceinline__ unsigned valid_slots(const int *row, int S, int t, int bs, int nbmax, int *err)
{
    bool bad;
    const unsigned m = row_slots(row, S, t, bs, nbmax, bad);
    if (bad && err)
        set_error(err, NSA_ERR_BAD_INDEX);
    return m;
}

__device__ __forceinline__ void chunk_count_body(const Geo &g, const int *__restrict__ idx, int *__restrict__ chunk_counts,
                                                 int nchunks, int *err, int blk, int nblk)
{
    const int64_t n = (int64_t)g.ntok * g.Hkv;
    for (int64_t lin = (int64_t)blk * blockDim.x + threadIdx.x; lin < n; lin += (int64_t)nblk * blockDim.x) {
        int b, kvh, t;
        decode_idx_row(g, lin, b, kvh, t);
        const int *row = idx_row(g, idx, b, kvh, t);
        unsigned m = valid_slots(row, g.S, t, g.bs, g.nbmax, err);
        const int64_t base = ((int64_t)b * g.Hkv + kvh) * g.nbmax;
        while (m) {
            const int s = __ffs(m) - 1;
            m &= m - 1u;
            atomicAdd(&chunk_counts[(base + row[s]) * nchunks + t / kChunkTok], 1);
        }
    }
}

__global__ void __launch_bounds__(kThreads) csr_chunk_count_kernel(Geo g, const int *__restrict__ idx,
                                                                   int *__restrict__ chunk_counts, int nchunks,
                                                                   int *err)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the prefix may launch (it waits)
    chunk_count_body(g, idx, chunk_counts, nchunks, err, blockIdx.x, gridDim.x);
}

// The chunk count and delta = rowsum(dO * O) in one launch: they are
// independent, the first latency-bound and the second bandwidth-bound, so
// the count's blocks (the first count_blocks) run under the dot's.
template <typename T, bool LIN>
__global__ void __launch_bounds__(kThreads) chunk_count_dot_kernel(Geo g, const int *__restrict__ idx,
                                                                   int *__restrict__ chunk_counts, int nchunks,
                                                                   int *err, int count_blocks, const T *__restrict__ o,
                                                                   const T *__restrict__ dO, float *__restrict__ out,
                                                                   int64_t nrows)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // the prefix may launch (it waits)
    if ((int)blockIdx.x < count_blocks)
        chunk_count_body(g, idx, chunk_counts, nchunks, err, blockIdx.x, count_blocks);
    else
        do_dot_rows<T, LIN>(g, o, dO, out, nrows, g.D, blockIdx.x - count_blocks, gridDim.x - count_blocks);
}

// one warp per (bg, j): exclusive prefix over chunks, list length in counts
__global__ void __launch_bounds__(kThreads) csr_chunk_prefix_kernel(Geo g, int *__restrict__ chunk_counts,
                                                                    int nchunks, int *__restrict__ counts)
{
    // a programmatic dependent of the count, and the scan's primary (see csr_scan_kernel)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int n = g.B * g.Hkv * g.nbmax;
    for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += (gridDim.x * blockDim.x) >> 5) {
        int *p = chunk_counts + (int64_t)i * nchunks;
        int carry = 0;
        for (int c0 = 0; c0 < nchunks; c0 += 32) {
            const int c = c0 + lane;
            const int v = c < nchunks ? p[c] : 0;
            int x = v;
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off)
                    x += y;
            }
            if (c < nchunks)
                p[c] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0)
            counts[i] = carry;
    }
}

// one warp per (bg, chunk): lane = token
__global__ void __launch_bounds__(kFillWarps * 32) csr_chunk_fill_kernel(Geo g, const int *__restrict__ idx,
                                                                         const int *__restrict__ chunk_prefix,
                                                                         int nchunks, const int *__restrict__ offsets,
                                                                         int *__restrict__ rows)
{
    // this kernel waits for the scan (see csr_scan_kernel); then the kernel
    // launched next may start its set-up, which reads the scan's unit list
    // but not this kernel's lists (it waits for this kernel before those)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ unsigned mask_all[];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned *mask = mask_all + w * g.nbmax;  // lanes selecting block j
    for (int j = lane; j < g.nbmax; j += 32)
        mask[j] = 0u;
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    const int total = g.B * g.Hkv * nchunks;
    for (int item = blockIdx.x * kFillWarps + w; item < total; item += gridDim.x * kFillWarps) {
        const int bg = item / nchunks, c = item % nchunks;
        const int b = bg / g.Hkv, kvh = bg % g.Hkv;
        const int t = c * kChunkTok + lane;
        const int *row = nullptr;
        unsigned m = 0u;
        if (t < seq_len(g, b)) {
            row = idx_row(g, idx, b, kvh, t);
            m = valid_slots(row, g.S, t, g.bs, g.nbmax, nullptr);
        }
        for (unsigned mm = m; mm; mm &= mm - 1u)
            atomicOr(&mask[row[__ffs(mm) - 1]], 1u << lane);
        __syncwarp();
        for (unsigned mm = m; mm; mm &= mm - 1u) {
            const int j = row[__ffs(mm) - 1];
            const int64_t bgj = (int64_t)bg * g.nbmax + j;
            rows[offsets[bgj] + chunk_prefix[bgj * nchunks + c] + __popc(mask[j] & lt)] = t;
        }
        __syncwarp();
        for (unsigned mm = m; mm; mm &= mm - 1u)
            mask[row[__ffs(mm) - 1]] = 0u;
        __syncwarp();
    }
}

// ---- attention sinks
// Row i of o / lse (the same linear row order in both layouts) belongs to
// query head (i / T) % Hq (BHTD) or i % Hq (THD).
__device__ __forceinline__ int row_head(const Geo &g, int64_t i)
{
    return g.thd ? (int)(i % g.Hq) : (int)((i / g.T) % g.Hq);
}

// Folds each head's sink into the forward's rows, one warp per row:
// LSE' = log(e^LSE + e^sink), O' = O e^(LSE - LSE') (an empty row, LSE =
// -inf, becomes LSE' = sink, O' = 0).
template <typename T>
__global__ void __launch_bounds__(kThreads) sink_fwd_kernel(Geo g, const float *__restrict__ sinks, T *__restrict__ o,
                                                            float *__restrict__ lse, int64_t nrows)
{
    const int lane = threadIdx.x & 31;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < nrows;
         i += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const float sk = sinks[row_head(g, i)], L = lse[i];
        float Ln, f;
        if (L == -INFINITY) {
            Ln = sk;
            f = 0.f;
        } else {
            const float m = fmaxf(L, sk);
            Ln = m + log1pf(expf(-fabsf(L - sk)));
            f = expf(L - Ln);
        }
        T *row = o + (g.o_lin ? i * g.D : qrow_off(g, g.so, i));
        for (int d = lane; d < g.D; d += 32)
            row[d] = from_f<T>(to_f(row[d]) * f);
        if (lane == 0)
            lse[i] = Ln;
    }
}

// dsinks[h] = - sum over the head's rows of exp(sink - LSE) * delta: one
// block per head, a fixed split over threads and a fixed tree (deterministic).
__global__ void __launch_bounds__(kThreads) sink_bwd_kernel(Geo g, const float *__restrict__ sinks,
                                                            const float *__restrict__ lse,
                                                            const float *__restrict__ delta, float *__restrict__ dsinks)
{
    __shared__ double part[kThreads];
    const int h = blockIdx.x;
    const float sk = sinks[h];
    const int64_t per_head = g.thd ? (int64_t)g.ntok : (int64_t)g.B * g.T;
    double acc = 0.0;
    for (int64_t x = threadIdx.x; x < per_head; x += blockDim.x) {
        // the x-th row of head h: token x (THD) or (b, t) = (x / T, x % T)
        const int64_t i = g.thd ? x * g.Hq + h : ((x / g.T) * g.Hq + h) * g.T + x % g.T;
        acc -= (double)expf(sk - lse[i]) * (double)delta[i];
    }
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w)
            part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0)
        dsinks[h] = (float)part[0];
}

}  // namespace

cudaError_t launch_do_dot(const Geo &g, const void *o, const void *dO, float *delta, int dtype,
                          cudaStream_t st)
{
    const int64_t nrows = (int64_t)g.ntok * g.Hq;
    const int elems = dtype == NSA_DTYPE_BF16 ? 8 : 4;
    const int rpw = 32 / (g.D / elems);
    const int grid = grid_for(nrows, (kThreads / 32) * kDotU * rpw, kDotBlocks);
    using B16 = __nv_bfloat16;
    if (dtype == NSA_DTYPE_BF16) {
        if (g.o_lin)
            do_dot_kernel<B16, true><<<grid, kThreads, 0, st>>>(g, (const B16 *)o, (const B16 *)dO, delta, nrows, g.D);
        else
            do_dot_kernel<B16, false><<<grid, kThreads, 0, st>>>(g, (const B16 *)o, (const B16 *)dO, delta, nrows, g.D);
    } else {
        if (g.o_lin)
            do_dot_kernel<float, true><<<grid, kThreads, 0, st>>>(g, (const float *)o, (const float *)dO, delta, nrows,
                                                                  g.D);
        else
            do_dot_kernel<float, false><<<grid, kThreads, 0, st>>>(g, (const float *)o, (const float *)dO, delta,
                                                                   nrows, g.D);
    }
    return cudaGetLastError();
}

cudaError_t launch_validate_index(const Geo &g, const int *idx, int *err, cudaStream_t st)
{
    const int64_t n = (int64_t)g.ntok * g.Hkv;
    validate_kernel<<<grid_for(n, kThreads), kThreads, 0, st>>>(g, idx, err);
    return cudaGetLastError();
}

cudaError_t launch_csr_count(const Geo &g, const int *idx, int *counts, int *err, cudaStream_t st)
{
    const int64_t n = (int64_t)g.ntok * g.Hkv;
    csr_count_kernel<<<grid_for(n, kThreads), kThreads, 0, st>>>(g, idx, counts, err);
    return cudaGetLastError();
}

cudaError_t launch_csr_scan(const Geo &g, const int *counts, int *offsets, Unit *units,
                            int *blk_nchunk, int *blk_slot, WsHeader *hdr, int chunk,
                            cudaStream_t st)
{
    return launch_dependent(csr_scan_kernel, dim3(1), dim3(1024), 0, st, g, counts, offsets, units, blk_nchunk,
                            blk_slot, hdr, chunk);
}

int csr_nchunks(const Geo &g) { return (g.T + kChunkTok - 1) / kChunkTok; }

bool csr_chunked_ok(const Geo &g)
{
    return g.S <= 32 && g.nbmax <= 2048 && (int64_t)g.B * g.Hkv * g.nbmax * csr_nchunks(g) <= ((int64_t)1 << 24);
}

cudaError_t launch_csr_chunk_count(const Geo &g, const int *idx, int *chunk_counts, int *counts, int *err,
                                   cudaStream_t st, const DotArgs *dot)
{
    const int nchunks = csr_nchunks(g);
    const int64_t nbgj = (int64_t)g.B * g.Hkv * g.nbmax;
    cudaError_t e = cudaMemsetAsync(chunk_counts, 0, sizeof(int) * nbgj * nchunks, st);
    if (e != cudaSuccess)
        return e;
    const int64_t n = (int64_t)g.ntok * g.Hkv;
    const int cblocks = grid_for(n, kThreads);
    if (dot) {
        const int64_t nrows = (int64_t)g.ntok * g.Hq;
        const int elems = dot->dtype == NSA_DTYPE_BF16 ? 8 : 4;
        const int rpw = 32 / (g.D / elems);
        const int grid = cblocks + grid_for(nrows, (kThreads / 32) * kDotU * rpw, kDotBlocks);
        using B16 = __nv_bfloat16;
        auto go = [&](auto kernel, const auto *o, const auto *dO) {
            kernel<<<grid, kThreads, 0, st>>>(g, idx, chunk_counts, nchunks, err, cblocks, o, dO, dot->delta, nrows);
        };
        if (dot->dtype == NSA_DTYPE_BF16) {
            if (g.o_lin)
                go(chunk_count_dot_kernel<B16, true>, (const B16 *)dot->o, (const B16 *)dot->dO);
            else
                go(chunk_count_dot_kernel<B16, false>, (const B16 *)dot->o, (const B16 *)dot->dO);
        } else {
            if (g.o_lin)
                go(chunk_count_dot_kernel<float, true>, (const float *)dot->o, (const float *)dot->dO);
            else
                go(chunk_count_dot_kernel<float, false>, (const float *)dot->o, (const float *)dot->dO);
        }
    } else {
        csr_chunk_count_kernel<<<cblocks, kThreads, 0, st>>>(g, idx, chunk_counts, nchunks, err);
    }
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    return launch_dependent(csr_chunk_prefix_kernel, dim3(grid_for(nbgj * 32, kThreads)), dim3(kThreads), 0, st, g,
                            chunk_counts, nchunks, counts);
}

cudaError_t launch_csr_chunk_fill(const Geo &g, const int *idx, const int *chunk_prefix, const int *offsets,
                                  int *rows, cudaStream_t st)
{
    const int nchunks = csr_nchunks(g);
    const int items = g.B * g.Hkv * nchunks;
    const int grid = grid_for(items, kFillWarps);
    const size_t smem = sizeof(unsigned) * kFillWarps * g.nbmax;
    return launch_dependent(csr_chunk_fill_kernel, dim3(grid), dim3(kFillWarps * 32), smem, st, g, idx, chunk_prefix,
                            nchunks, offsets, rows);
}

cudaError_t launch_csr_fill(const Geo &g, const int *idx, const int *offsets, int *rows,
                            cudaStream_t st)
{
    const int n = g.B * g.Hkv * g.nbmax;
    if (n == 0)
        return cudaSuccess;
    csr_fill_kernel<<<n, kThreads, 0, st>>>(g, idx, offsets, rows);
    return cudaGetLastError();
}

cudaError_t launch_dkdv_reduce(const Geo &g, const int *blk_nchunk, const int *blk_slot,
                               const float *partials, void *dk, void *dv, int dtype,
                               cudaStream_t st, bool dependent)
{
    const int n = g.B * g.Hkv * g.nbmax;
    if (n == 0)
        return cudaSuccess;
    auto go = [&](auto kernel, auto *k_out, auto *v_out) -> cudaError_t {
        if (dependent)
            return launch_dependent(kernel, dim3(4 * n), dim3(kThreads), 0, st, g, blk_nchunk, blk_slot, partials,
                                    k_out, v_out);
        kernel<<<4 * n, kThreads, 0, st>>>(g, blk_nchunk, blk_slot, partials, k_out, v_out);
        return cudaGetLastError();
    };
    if (dtype == NSA_DTYPE_BF16)
        return go(dkdv_reduce_kernel<__nv_bfloat16>, (__nv_bfloat16 *)dk, (__nv_bfloat16 *)dv);
    return go(dkdv_reduce_kernel<float>, (float *)dk, (float *)dv);
}

cudaError_t launch_count_pairs(const Geo &g, const int *idx, long long *out, cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(long long), st);
    if (e != cudaSuccess)
        return e;
    const int64_t n = (int64_t)g.ntok * g.Hkv;
    count_pairs_kernel<<<grid_for(n, kThreads), kThreads, 0, st>>>(g, idx,
                                                                   (unsigned long long *)out);
    return cudaGetLastError();
}

cudaError_t launch_sink_fwd(const Geo &g, const float *sinks, void *o, float *lse, int dtype, cudaStream_t st)
{
    const int64_t nrows = (int64_t)g.ntok * g.Hq;
    const int grid = grid_for(nrows, kThreads / 32);
    if (dtype == NSA_DTYPE_BF16)
        sink_fwd_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(g, sinks, (__nv_bfloat16 *)o, lse, nrows);
    else
        sink_fwd_kernel<float><<<grid, kThreads, 0, st>>>(g, sinks, (float *)o, lse, nrows);
    return cudaGetLastError();
}

cudaError_t launch_sink_bwd(const Geo &g, const float *sinks, const float *lse, const float *delta, float *dsinks,
                            cudaStream_t st)
{
    sink_bwd_kernel<<<g.Hq, kThreads, 0, st>>>(g, sinks, lse, delta, dsinks);
    return cudaGetLastError();
}

}  // namespace nsa
