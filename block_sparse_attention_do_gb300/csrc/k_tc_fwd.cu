// k_tc_fwd.cu -- selection forward (O, LSE) on the tcgen05 tensor cores
// (bf16, D = 128, block_size = 64).
//
// Same query tile as the dQ kernel (Tq tokens x G heads = 128 rows) walking
// the ascending union of the tile's selected blocks two at a time.  For a
// pair (j_a, j_b), step i:
//   S_i = Q [K_a; K_b]^T                          (M=128 rows, N=128 keys, K=128)
//   P_i = exp(S_i - m) on the row's attended keys, l += rowsum(P_i)
//   O  += P_i [V_a; V_b]   accumulated in TMEM    (M=128 rows, N=128 dims, K=128 keys)
// m is a running reference that a row raises only when a pair's maximum
// exceeds it by more than 2^8; then that row's O (in TMEM) and l are scaled
// by exp(m_old - m_new) before the pair's P.V is issued.  Every term of O
// and l carries the same reference, so O / l at the end is exact; P stays
// below 2^8.  LSE = m + log l.  Warps whose rows all skip a pair write zero P
// without computing it.  P is written into the pair's K slot, free once S is
// computed.
//
// Roles (8 warps): warp 0 issues the TMA copies (the Q tile once, then the
// K/V pairs, one box per lane); warp 2 issues the S MMAs and warp 3 the P.V
// MMAs (one thread each); warps 4-7 build the block union, then run the
// online softmax one row per thread and the epilogue.
#include "tc_common.cuh"

namespace nsa {

namespace {

using namespace tc;

constexpr int NS = 2;                       // K/V pair stages
constexpr int kPairBytes = 2 * kTileBytes;  // K pair (32 KB, later P) | V pair (32 KB)
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + kTileBytes;
constexpr int OFF_MASK = OFF_KV + NS * kPairBytes;
constexpr int OFF_LIST = OFF_MASK + MASK_WORDS * 4;
constexpr int OFF_UBITS = OFF_LIST + MAX_BLOCKS * 4;
constexpr int OFF_BAR = OFF_UBITS + (MAX_BLOCKS / 32) * 4;
constexpr int NUM_BARS = 20;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;

enum {
    B_QFULL = 0, B_LIST, B_DONE, B_PVFULL, B_SFULL0, B_SFULL1, B_SFREE0, B_SFREE1,
    B_KVF0, B_KVF1, B_KVE0, B_KVE1, B_PF0, B_PF1, B_DONES, B_VF0, B_VF1, B_COUNT  // B_KVF*: the pair's K (its V: B_VF*)
};
static_assert(B_COUNT <= NUM_BARS, "barrier slots");

constexpr uint32_t TM_S = 0;    // buffer b at b*128 (keys of the pair)
constexpr uint32_t TM_O = 256;  // 128 lanes (rows) x 128 columns (dims)
constexpr uint32_t TM_COLS = 512;
constexpr float kRescaleLog2 = 8.f;  // raise the reference only past a 2^8 growth

struct Params {
    Geo g;
    const int *idx;
    __nv_bfloat16 *o;
    float *lse;
    int *err;
};

__global__ void __launch_bounds__(256, 1) fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                        const __grid_constant__ CUtensorMap tm_k,
                                                        const __grid_constant__ CUtensorMap tm_v,
                                                        const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(sm + OFF_BAR);
    volatile int *abort_flag = (volatile int *)(sm + OFF_MISC);
    uint32_t *tmem_slot = (uint32_t *)(sm + OFF_MISC + 16);
    volatile int *n_list = (volatile int *)(sm + OFF_MISC + 32);
    uint32_t *mask = (uint32_t *)(sm + OFF_MASK);
    int *list = (int *)(sm + OFF_LIST);
    uint32_t *ubits = (uint32_t *)(sm + OFF_UBITS);

    const Geo &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = g.G;
    const int Tq = tile_tokens(G);
    const int nrows = Tq * G;
    const int ntiles_seq = (g.T + Tq - 1) / Tq;
    const int tile = ntiles_seq - 1 - (int)blockIdx.x;  // heavier (later) tiles first
    const int kvh = blockIdx.y, b = blockIdx.z;
    const int L = seq_len(g, b);
    const int t0 = tile * Tq;
    if (t0 >= L)
        return;
    const int nvalid = min(Tq, L - t0);
    const int words = (g.nbmax + 31) / 32;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(&bars[B_QFULL], 1);
        mbar_init(&bars[B_LIST], kRows);
        mbar_init(&bars[B_DONE], 1);
        mbar_init(&bars[B_DONES], 1);
        mbar_init(&bars[B_PVFULL], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_SFULL0 + s], 1);
            mbar_init(&bars[B_SFREE0 + s], kRows);
            mbar_init(&bars[B_KVF0 + s], 1);
            mbar_init(&bars[B_VF0 + s], 1);
            mbar_init(&bars[B_KVE0 + s], 1);
            mbar_init(&bars[B_PF0 + s], kRows);
        }
        fence_barrier_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    // Tile rows past Tq * G receive no data; they meet P = 0 but must be
    // finite.  (A pair's missing second block is loaded as a copy of its first.)
    // With G % 8 == 0 in BHTD the tile is in the row-group layout (one TMA
    // box per token: its G heads, both halves), else rows of 128 bytes per half.
    const bool rg = !g.thd && (G % 8) == 0;
    if (nrows < kRows)
        for (int i = threadIdx.x; i < 2 * (kRows - nrows) * 8; i += blockDim.x) {
            const int half = i / ((kRows - nrows) * 8), rem = i % ((kRows - nrows) * 8);
            const int row = nrows + (rem >> 3);
            *(uint4 *)(sm + OFF_Q + (rg ? rg_off(row, half) : half * kHalfBytes + row * 128) + (rem & 7) * 16) =
                make_uint4(0, 0, 0, 0);
        }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------- TMA
        // One TMA box per lane: issuing them from a single thread serialises
        // about a hundred cycles per box.
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(&bars[B_QFULL], 2 * nrows * 128);
        }
        __syncwarp();
        {
            const int nbox = rg ? Tq : 2;
            for (int box = lane; box < nbox; box += 32) {
                if (rg) {  // token box: G heads x both halves, contiguous in the row-group layout
                    tma_load_5d(sm + OFF_Q + box * G * 256, &tm_q, &bars[B_QFULL], 0, 0, 0, (b * g.Hq + kvh * G) / 8,
                                t0 + box);
                } else {
                    uint8_t *dst = sm + OFF_Q + box * kHalfBytes;
                    if (g.thd)
                        tma_load_3d(dst, &tm_q, &bars[B_QFULL], box * 64, kvh * G, g.cu[b] + t0);
                    else
                        tma_load_4d(dst, &tm_q, &bars[B_QFULL], box * 64, t0, kvh * G, b);
                }
            }
        }
        bool ok = mbar_wait_warp(&bars[B_LIST], 0, abort_flag);
        const int U = ok ? *n_list : 0;
        const int npairs = (U + 1) >> 1;
        int last = -1;
        for (int i = 0; i < npairs && ok; ++i) {
            const int s = i % NS;
            if (!mbar_wait_warp(&bars[B_KVE0 + s], ((i / NS) & 1) ^ 1, abort_flag))
                break;
            uint8_t *kd = sm + OFF_KV + s * kPairBytes, *vd = kd + kTileBytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[B_KVF0 + s], 2 * kKvBytes);
                mbar_arrive_expect_tx(&bars[B_VF0 + s], 2 * kKvBytes);
            }
            __syncwarp();
            last = i;
            // lane -> (K or V, block e of the pair, 64-column half h), the K
            // boxes first (S needs K only; V is read by the later P.V).  A
            // missing second block repeats the first (finite data, P = 0).
            if (lane < 8) {
                const int isv = lane >> 2, e = (lane >> 1) & 1, h = lane & 1;
                const int j = list[min(2 * i + e, U - 1)];
                uint8_t *dst = (isv ? vd : kd) + h * kHalfBytes + e * kKvHalfBytes;
                const CUtensorMap *map = isv ? &tm_v : &tm_k;
                uint64_t *bar = &bars[(isv ? B_VF0 : B_KVF0) + s];
                if (g.thd)
                    tma_load_3d(dst, map, bar, h * 64, kvh, g.cu[b] + j * kKeys);
                else
                    tma_load_4d(dst, map, bar, h * 64, j * kKeys, kvh, b);
            }
        }
        // copies in flight must land before the CTA may exit
        if (lane == 0) {
            volatile int never = 0;
            mbar_wait(&bars[B_QFULL], 0, &never);
            if (*abort_flag && last >= 0) {
                mbar_wait(&bars[B_KVF0 + last % NS], (last / NS) & 1, &never);
                mbar_wait(&bars[B_VF0 + last % NS], (last / NS) & 1, &never);
            }
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------------- MMA
        // Two issuing threads: warp 2 issues S of each pair, warp 3 the P.V
        // products (whose completion frees a K/V stage), so a ready P.V never
        // queues behind the next pair's S issue.  TMEM columns are disjoint
        // (S buffers vs O); each commit covers its own thread's MMAs.
        if (lane == 0) {
            const uint32_t kv_s = smem_u32(sm + OFF_KV);
            bool ok = mbar_wait(&bars[B_LIST], 0, abort_flag) && mbar_wait(&bars[B_QFULL], 0, abort_flag);
            const int U = ok ? *n_list : 0;
            const int npairs = (U + 1) >> 1;
            if (warp == 2) {
                const uint32_t idS = idesc_bf16(128, 128, false, false);
                const uint32_t q_s = smem_u32(sm + OFF_Q);
                // Q tile: 64-column halves and 8-row groups apart by these
                const uint32_t qhalf = rg ? kRgHalf : kHalfBytes, qsbo = rg ? kRgStride : 1024;
                for (int si = 0; si < npairs && ok; ++si) {
                    // the pair's K/V have landed; the softmax has taken S of
                    // pair si - 2 out of this TMEM buffer
                    if (!mbar_wait(&bars[B_KVF0 + si % NS], (si / NS) & 1, abort_flag) ||
                        !mbar_wait(&bars[B_SFREE0 + (si & 1)], ((si >> 1) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k_s = kv_s + (si % NS) * kPairBytes;
                    for (int kk = 0; kk < kHead / 16; ++kk) {
                        const uint32_t o = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                        const uint32_t oq = (kk >> 2) * qhalf + (kk & 3) * 32;
                        mma_bf16(tmem + TM_S + (si & 1) * 128, sdesc_sw128(q_s + oq, 16, qsbo),
                                 sdesc_sw128(k_s + o, 16, 1024), idS, kk > 0);
                    }
                    mma_commit(&bars[B_SFULL0 + (si & 1)]);
                }
                mma_commit(&bars[B_DONES]);
                volatile int never = 0;
                mbar_wait(&bars[B_DONES], 0, &never);
            } else {
                const uint32_t idO = idesc_bf16(128, 128, false, true);
                for (int oi = 0; oi < npairs && ok; ++oi) {
                    if (!mbar_wait(&bars[B_PF0 + oi % NS], (oi / NS) & 1, abort_flag) ||
                        !mbar_wait(&bars[B_VF0 + oi % NS], (oi / NS) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int s = oi % NS;
                    const uint32_t p_s = kv_s + s * kPairBytes, v_s = p_s + kTileBytes;
                    for (int kk = 0; kk < 8; ++kk)  // 128 keys: P (K-major, 2 halves) x V pair (MN-major)
                        mma_bf16(tmem + TM_O, sdesc_sw128(p_s + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024),
                                 sdesc_sw128(v_s + kk * 2048, kHalfBytes, 1024), idO, (oi > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bars[B_PVFULL]);
                    mma_commit(&bars[B_KVE0 + s]);
                }
                // O is final once this commit completes
                mma_commit(&bars[B_DONE]);
                volatile int never = 0;
                mbar_wait(&bars[B_DONE], 0, &never);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------- union, softmax, epilogue
        const int tid = threadIdx.x - 128;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const int U = qtile_union(g, p.idx, b, kvh, t0, nvalid, mask, ubits, list, tid, lane, wq);
        if (tid == 0)
            *n_list = U;
        mbar_arrive(&bars[B_LIST]);
        const int npairs = (U + 1) >> 1;

        int tl, hh;
        qtile_row(g, Tq, r, tl, hh);
        const bool rvalid = r < nrows && tl < nvalid;
        const int t = t0 + tl;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const uint32_t *my_mask = mask + (rvalid ? tl : 0) * words;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < npairs; ++i) {
            const int s = i & 1;
            if (!mbar_wait_warp(&bars[B_SFULL0 + s], (i >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[128];
            tmem_ld64(lane_base + TM_S + s * 128, *reinterpret_cast<uint32_t(*)[64]>(&sv[0]));
            tmem_ld64(lane_base + TM_S + s * 128 + 64, *reinterpret_cast<uint32_t(*)[64]>(&sv[64]));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&bars[B_SFREE0 + s]);
            // block e: the row attends keys j*64 + c, lo[e] <= c <= lim[e]
            int lim[2], lo[2];
            bool anysel = false;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = (2 * i + e < U) ? list[2 * i + e] : -1;
                const bool sel = rvalid && j >= 0 && qtile_selects(g, my_mask, t, j);
                lim[e] = sel ? t - j * kKeys : -1;
                lo[e] = key_lo(g, t) - j * kKeys;
                anysel |= sel;
            }
            uint32_t pk[64];
            if (__any_sync(0xffffffffu, anysel)) {
                // no row of the warp ends inside either block: a row attends a
                // whole block or none of it; none gets a -inf bias
                const bool whole = __all_sync(0xffffffffu, (lim[0] < 0 || (lim[0] >= kKeys - 1 && lo[0] <= 0)) &&
                                                               (lim[1] < 0 || (lim[1] >= kKeys - 1 && lo[1] <= 0)));
                float mb = -INFINITY;
                if (whole) {
                    const float b0 = lim[0] >= 0 ? 0.f : -INFINITY, b1 = lim[1] >= 0 ? 0.f : -INFINITY;
                    const uint64_t sc2 = f2(g.scale_l2, g.scale_l2), bb0 = f2(b0, b0), bb1 = f2(b1, b1);
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        float x0, x1;
                        f2_split(f2_fma(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, c < 64 ? bb0 : bb1),
                                 x0, x1);
                        sv[c] = __float_as_uint(x0);
                        sv[c + 1] = __float_as_uint(x1);
                        mb = fmaxf(mb, fmaxf(x0, x1));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const float x = __uint_as_float(sv[c]) * g.scale_l2;
                        sv[c] = __float_as_uint(x);
                        if ((c & 63) <= lim[c >> 6] && (c & 63) >= lo[c >> 6])
                            mb = fmaxf(mb, x);
                    }
                }
                const bool raise = mb > m + kRescaleLog2;
                if (__any_sync(0xffffffffu, raise)) {
                    // O must hold every earlier pair before it is rescaled
                    if (i > 0 && !mbar_wait_warp(&bars[B_PVFULL], (i - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float alpha = raise ? ex2(m - mb) : 1.f;  // 0 when m = -inf
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t a[16];
                        tmem_ld16(lane_base + TM_O + c * 16, a);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            a[e] = __float_as_uint(__uint_as_float(a[e]) * alpha);
                        tmem_st16(lane_base + TM_O + c * 16, a);
                    }
                    tmem_wait_st();
                    if (raise) {
                        l *= alpha;
                        m = mb;
                    }
                }
                float rs = 0.f;
                if (whole) {
                    // a row with nothing attended so far has m = -inf and only
                    // -inf scores: subtract 0 there so that exp2 gives 0, not NaN
                    const float ms = m == -INFINITY ? 0.f : m;
                    const uint64_t nms2 = f2(-ms, -ms);
                    uint64_t rs2 = f2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        float x0, x1;
                        f2_split(f2_add(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), nms2), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        rs2 = f2_add(rs2, f2(p0, p1));
                        pk[c >> 1] = pack_bf16(p0, p1);
                    }
                    float r0, r1;
                    f2_split(rs2, r0, r1);
                    rs = r0 + r1;
                } else {
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        const int lm = lim[c >> 6], lw = lo[c >> 6];
                        const float p0 = ((c & 63) <= lm && (c & 63) >= lw) ? ex2(__uint_as_float(sv[c]) - m) : 0.f;
                        const float p1 = (((c + 1) & 63) <= lm && ((c + 1) & 63) >= lw)
                                             ? ex2(__uint_as_float(sv[c + 1]) - m)
                                             : 0.f;
                        rs += p0 + p1;
                        pk[c >> 1] = pack_bf16(p0, p1);
                    }
                }
                l += rs;
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    pk[c] = 0u;
            }
            // P goes into this pair's K slot (S is already computed)
            const uint32_t p_row = smem_u32(sm + OFF_KV + (i % NS) * kPairBytes) + r * 128;
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(p_row + e * kHalfBytes + ((c ^ (r & 7)) << 4), pk[32 * e + 4 * c],
                                 pk[32 * e + 4 * c + 1], pk[32 * e + 4 * c + 2], pk[32 * e + 4 * c + 3]);
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&bars[B_PF0 + i % NS]);
        }
        float o[128];
        if (ok && npairs > 0) {
            // The last two P.V products may both still be running here, which
            // a parity wait on PVFULL cannot tell apart; DONE is committed
            // once, after the final MMA.
            if (!mbar_wait_warp(&bars[B_DONE], 0, abort_flag)) {
                ok = false;
            } else {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t a[16];
                    tmem_ld16(lane_base + TM_O + c * 16, a);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[c * 16 + e] = __uint_as_float(a[e]);
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < 128; ++e)
                o[e] = 0.f;
        }
        if (ok && rvalid) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *dst = p.o + row_off(g, g.Hq, b, kvh * G + hh, t);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16(o[c * 8 + 2 * e] * inv, o[c * 8 + 2 * e + 1] * inv);
                *(uint4 *)(dst + c * 8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            p.lse[stat_off(g, b, kvh * G + hh, t)] = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
        tc_fence_before();
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 0)
        set_error(p.err, NSA_ERR_DEVICE_TIMEOUT);
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace

cudaError_t launch_fwd_tc(const Geo &g, const void *q, const void *k, const void *v, const int *idx,
                          void *o, float *lse, int *err, cudaStream_t st)
{
    if (!qtile_shape_ok(g))
        return launch_fwd_simt(g, q, k, v, idx, o, lse, NSA_DTYPE_BF16, st);
    const int Tq = tile_tokens(g.G);
    CUtensorMap tq, tk, tv;
    const bool rg = !g.thd && (g.G % 8) == 0;  // row-group Q tile, one box per token
    const bool qmap = rg ? make_tmap_rows(&tq, q, g, g.Hq, g.G) : make_tmap(&tq, q, g, g.Hq, Tq, g.G);
    if (!qmap || !make_tmap(&tk, k, g, g.Hkv, kKeys, 1) || !make_tmap(&tv, v, g, g.Hkv, kKeys, 1))
        return cudaErrorInvalidValue;
    Params p;
    p.g = g;
    p.idx = idx;
    p.o = (__nv_bfloat16 *)o;
    p.lse = lse;
    p.err = err;
    dim3 grid((g.T + Tq - 1) / Tq, g.Hkv, g.B);
    cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    fwd_tc_kernel<<<grid, 256, SMEM_BYTES, st>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace nsa
