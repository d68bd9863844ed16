// k_tc_fwd.cu -- selection forward (O, LSE) on the tcgen05 tensor cores
// (bf16, D = 128, block_size = 64).
//
// Same query tiles as the dQ kernel (Tq tokens x G heads = 128 rows), each
// walking the ascending union of its tokens' selected blocks two at a time.
// For a pair (j_0, j_1), step i:
//   S_i = Q [K_0; K_1]^T                  (M=128 rows, N=128 keys, K=128)
// and block e of the pair (keys e*64 .. e*64+63 of S_i) goes to softmax
// warpgroup e, which keeps its own running reference m_e and sum l_e per row
// and its own accumulator:
//   P_e = exp(S_i[:, block e] - m_e) on the row's attended keys, l_e += rowsum(P_e)
//   O_e += P_e V_{j_e}                    (M=128 rows, N=128 dims, K=64 keys)
// A warpgroup raises a row's m_e only when a pair's maximum exceeds it by
// more than 2^8; then that row of O_e (in TMEM) and l_e are scaled by
// exp(m_old - m_new) first.  Every term of O_e and l_e carries the same
// reference, and the epilogue merges the two halves exactly:
//   m = max(m_0, m_1),  a_e = exp(m_e - m),  l = a_0 l_0 + a_1 l_1,
//   O = (a_0 O_0 + a_1 O_1) / l,  LSE = m + log l.
// Warps whose rows all skip a block write zero P without computing it.
//
// P_e stays in TMEM: it is written (bf16 pairs) over the first 32 columns of
// its S block and read from there as the A operand of O_e += P_e V.  So a
// pair's K is free as soon as S is computed, and K and V have rings of their
// own: K is held only from its load to S, V from its load to P.V.
//
// The kernel is persistent like the dQ kernel: one CTA per SM, tiles taken
// heaviest first from a launch-wide counter (each claimed a tile ahead), a
// selection tile's union copied from the table qtile_union_kernel built
// (a dense tile's built here), the next tile's union and Q load overlapping
// the current tile; S (with P) is double-buffered in TMEM and the K and V
// rings carry across tiles.
//
// Roles (12 warps): warp 0 deals the tiles, copies in (or builds) each
// tile's block union and issues the TMA copies (the tile's Q, then per pair its K boxes and its
// V boxes, one box per lane); one thread of warp 2 (which owns TMEM) issues
// S, one thread each of warps 1 and 3 the P.V products of blocks 0 and 1;
// warps 4-7 and 8-11 are softmax warpgroups 0 and 1, one row per thread,
// and split the epilogue's columns.
#include "tc_common.cuh"

namespace nsa {

namespace {

using namespace tc;

constexpr int NK = 2;  // K pair stages (32 KB each)
constexpr int NV = 3;  // V pair stages (32 KB each)
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + kTileBytes;
constexpr int OFF_V = OFF_K + NK * kTileBytes;
constexpr int OFF_UNION = OFF_V + NV * kTileBytes;  // union buffers, sized at launch
constexpr int kXchgBytes = 2 * 2 * kRows * 8;       // row (m, l) of both warpgroups, two tiles
constexpr int NUM_BARS = 40;
constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per block

enum {
    B_QFULL = 0, B_QEMPTY, B_ACCFULL, B_ACCEMPTY, B_DONE0, B_DONE1, B_DONE2, B_SFULL0, B_SFULL1, B_SFREE0, B_SFREE1,
    B_PF00, B_PF01, B_PF10, B_PF11, B_PVFULL00, B_PVFULL01, B_PVFULL10, B_PVFULL11,  // [warpgroup][buffer]
    B_UFULL0, B_UFULL1, B_UEMPTY0, B_UEMPTY1, B_XCHG0, B_XCHG1,
    B_KF0, B_KE0 = B_KF0 + NK, B_VF0 = B_KE0 + NK, B_VE0 = B_VF0 + NV, B_COUNT = B_VE0 + NV
};
static_assert(B_COUNT <= NUM_BARS, "barrier slots");
// threads releasing a tile's union: the loader warp, the three MMA threads
// and the 256 softmax threads
constexpr int kUnionUsers = 32 + 3 + 2 * kRows;

constexpr uint32_t TM_S = 0;    // S buffer x at x*128 (the pair's 128 keys); P_e over its columns e*64 .. +31
constexpr uint32_t TM_O = 256;  // O_e at 256 + e*128: 128 lanes (rows) x 128 columns (dims)
constexpr uint32_t TM_COLS = 512;
constexpr float kRescaleLog2 = 8.f;  // raise the reference only past a 2^8 growth

struct Params {
    Geo g;
    const int *idx;
    const int *utable;  // every tile's union buffer, built by the union kernel (null: built here)
    __nv_bfloat16 *o;
    float *lse;
    int *err;
    int ntiles;      // query tiles over all (b, kv head)
    int *tile_next;  // work counter, zero at launch
    int nub;     // union buffers (1 or 2)
    int v8;      // o is 32-byte aligned: the epilogue stores 32 bytes at a time
    int wait_us;  // bounded-wait limit in microseconds (0: the default)
    int stall;    // self-test: the S-product issuer stays idle (see wait_test)
};

// GROUPED: the union table's tiles are grouped by shared blocks (each row's
// token is read from the tile's record); else a tile's row tl has token T0 + tl
template <bool GROUPED>
__global__ void __launch_bounds__(384, 1) fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                        const __grid_constant__ CUtensorMap tm_k,
                                                        const __grid_constant__ CUtensorMap tm_v,
                                                        const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Geo &g = p.g;
    const UnionBuf up = union_buf(g);
    const int nub = p.nub;
    const int off_x = OFF_UNION + nub * up.bytes;
    const int off_bar = off_x + kXchgBytes;
    float2 *xchg = (float2 *)(sm + off_x);  // [tile parity][warpgroup][row]
    uint64_t *bars = (uint64_t *)(sm + off_bar);
    volatile int *abort_flag = (volatile int *)(sm + off_bar + NUM_BARS * 8);
    uint32_t *tmem_slot = (uint32_t *)(sm + off_bar + NUM_BARS * 8 + 16);
    // union buffer of this CTA's k-th tile, and the parity of its phase
    auto u_buf = [&](int k) { return (int *)(sm + OFF_UNION + (k % nub) * up.bytes); };
    auto u_hdr = [&](int k) { return (volatile int *)u_buf(k); };
    auto u_par = [&](int k) { return (uint32_t)((k / nub) & 1); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = g.G;
    const int Tq = tile_tokens(G);
    const int nrows = Tq * G;
    const int words = (g.nbmax + 31) / 32;

    if (threadIdx.x == 0) {
        abort_flag[0] = 0;
        abort_flag[1] = p.wait_us;  // the wait limit (0: the default)
        mbar_init(&bars[B_QFULL], 1);
        mbar_init(&bars[B_QEMPTY], 1);
        mbar_init(&bars[B_ACCFULL], 2);
        mbar_init(&bars[B_ACCEMPTY], 2 * kRows);
        for (int x = 0; x < 3; ++x)
            mbar_init(&bars[B_DONE0 + x], 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars[B_SFULL0 + x], 1);
            mbar_init(&bars[B_SFREE0 + x], 2);
            mbar_init(&bars[B_PF00 + x], kRows);
            mbar_init(&bars[B_PF10 + x], kRows);
            mbar_init(&bars[B_PVFULL00 + x], 1);
            mbar_init(&bars[B_PVFULL10 + x], 1);
            mbar_init(&bars[B_UFULL0 + x], 32);
            mbar_init(&bars[B_UEMPTY0 + x], kUnionUsers);
            mbar_init(&bars[B_XCHG0 + x], 2 * kRows);
        }
        for (int s = 0; s < NK; ++s) {
            mbar_init(&bars[B_KF0 + s], 1);
            mbar_init(&bars[B_KE0 + s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&bars[B_VF0 + s], 1);
            mbar_init(&bars[B_VE0 + s], 2);
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
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
        int lastq = -1, last = -1, lastv = -1, gi = 0;
        // The union table is written by the kernel this one depends on.
        if (p.utable)
            asm volatile("griddepcontrol.wait;" ::: "memory");
        int claimed = qtile_claim(p.tile_next, lane);
        for (int k = 0;; ++k) {
            // The tile and its block union: this warp deals the tiles (each
            // claimed a tile ahead) and takes each union from the table (or
            // builds it) after issuing the previous tile's copies, while the
            // K/V rings still hold several of that tile's pairs; after the last
            // tile a header with a negative count tells the other roles to stop.
            int b = 0, kvh = 0, t0 = 0, nvalid = 0, L = 0;
            const bool more = qtile_take(g, p.ntiles, p.tile_next, lane, claimed, b, kvh, t0, nvalid, &L);
            if (!mbar_wait_warp(&bars[B_UEMPTY0 + k % nub], u_par(k) ^ 1, abort_flag))
                break;
            if (more && p.utable) {
                // copy the tile's union buffer in, 16 bytes per lane and step
                const uint4 *src = (const uint4 *)(p.utable + (int64_t)L * (up.bytes / 4));
                uint4 *dst = (uint4 *)u_buf(k);
                for (int x = lane; x < up.bytes / 16; x += 32)
                    dst[x] = src[x];
                __syncwarp();
            } else if (more) {
                qtile_union_warp(g, p.idx, up, u_buf(k), b, kvh, t0, nvalid, lane);
            } else {
                if (lane == 0)
                    u_hdr(k)[UH_COUNT] = -1;
                __syncwarp();
            }
            mbar_arrive(&bars[B_UFULL0 + k % nub]);
            if (!more)
                break;
            claimed = qtile_claim(p.tile_next, lane);
            const int U = u_hdr(k)[UH_COUNT];
            const int *list = union_list(u_buf(k), up);
            // the tile's Q, once the previous tile's last S has run
            if (!mbar_wait_warp(&bars[B_QEMPTY], (k & 1) ^ 1, abort_flag))
                break;
            if (lane == 0)
                mbar_arrive_expect_tx(&bars[B_QFULL], nrows * 128 * 2);
            __syncwarp();
            lastq = k;
            if (rg) {  // token box: G heads x both halves, contiguous in the row-group layout
                for (int tl = lane; tl < Tq; tl += 32) {
                    if (g.q_bt)  // batch folded into the token index
                        tma_load_5d(sm + OFF_Q + tl * G * 256, &tm_q, &bars[B_QFULL], 0, 0, 0, kvh * G / 8,
                                    b * g.T + (GROUPED ? qtile_token(u_hdr(k), tl) : t0 + tl));
                    else
                        tma_load_5d(sm + OFF_Q + tl * G * 256, &tm_q, &bars[B_QFULL], 0, 0, 0, (b * g.Hq + kvh * G) / 8,
                                    GROUPED ? qtile_token(u_hdr(k), tl) : t0 + tl);
                }
            } else if (lane < 2) {
                const int h = lane;
                if (g.thd)
                    tma_load_3d(sm + OFF_Q + h * kHalfBytes, &tm_q, &bars[B_QFULL], h * 64, kvh * G, g.cu[b] + t0);
                else
                    tma_load_4d(sm + OFF_Q + h * kHalfBytes, &tm_q, &bars[B_QFULL], h * 64, t0, kvh * G, b);
            }
            bool ok = true;
            for (int i = 0; i < (U + 1) >> 1; ++i, ++gi) {
                // lane -> (block e of the pair, 64-column half h); K first (S
                // needs K only), then V once its stage is free.  A missing
                // second block repeats the first (finite data, P = 0).
                const int e = lane >> 1, h = lane & 1;
                const int j = list[min(2 * i + (e & 1), U - 1)];
                for (int isv = 0; isv < 2; ++isv) {
                    const int ns = isv ? NV : NK, st = gi % ns;
                    uint64_t *full = &bars[(isv ? B_VF0 : B_KF0) + st];
                    if (!mbar_wait_warp(&bars[(isv ? B_VE0 : B_KE0) + st], ((gi / ns) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0)
                        mbar_arrive_expect_tx(full, 2 * kKvBytes);
                    __syncwarp();
                    (isv ? lastv : last) = gi;
                    if (lane < 4) {
                        uint8_t *dst = sm + (isv ? OFF_V : OFF_K) + st * kTileBytes + h * kHalfBytes + e * kKvHalfBytes;
                        const CUtensorMap *map = isv ? &tm_v : &tm_k;
                        if (g.thd)
                            tma_load_3d(dst, map, full, h * 64, kvh, g.cuk[b] + j * kKeys);
                        else
                            tma_load_4d(dst, map, full, h * 64, j * kKeys, kvh, b);
                    }
                }
                if (!ok)
                    break;
            }
            if (!ok)
                break;
            mbar_arrive(&bars[B_UEMPTY0 + k % nub]);
        }
        // copies in flight must land before the CTA may exit
        if (lane == 0 && *abort_flag) {
            volatile int never[2] = {0, abort_flag[1]};  // own limit, no abort
            if (lastq >= 0)
                mbar_wait(&bars[B_QFULL], lastq & 1, never);
            if (last >= 0)
                mbar_wait(&bars[B_KF0 + last % NK], (last / NK) & 1, never);
            if (lastv >= 0)
                mbar_wait(&bars[B_VF0 + lastv % NV], (lastv / NV) & 1, never);
        }
        __syncwarp();
    } else if (warp <= 3) {
        // ---------------------------------------------------------------- MMA
        // Three issuing threads in three warps (one thread issues a tcgen05 MMA
        // only every ~150 cycles): warp 2 issues S of each pair (whose
        // completion frees its K stage), warps 1 and 3 the P.V products of
        // blocks 0 and 1 (O_0 and O_1; both completions free the V stage and
        // the S buffer holding P), so a ready product never queues behind
        // another's issue.  Each commit covers its own thread's MMAs.
        if (lane == 0) {
            const int e = warp == 3 ? 1 : 0;  // the P.V threads' block
            const uint32_t idS = idesc_bf16(128, 128, false, false), idO = idesc_bf16(128, 128, false, true);
            const uint32_t q_s = smem_u32(sm + OFF_Q);
            // Q tile: 64-column halves and 8-row groups apart by these
            const uint32_t qhalf = rg ? kRgHalf : kHalfBytes, qsbo = rg ? kRgStride : 1024;
            int gi = 0;
            // (self-test of the bounded waits: an idle S issuer makes the
            // softmax's first wait run out)
            bool ok = !(p.stall && warp == 2);
            for (int k = 0; ok; ++k) {
                if (!mbar_wait(&bars[B_UFULL0 + k % nub], u_par(k), abort_flag))
                    break;
                const int U = u_hdr(k)[UH_COUNT];
                if (U < 0)
                    break;
                mbar_arrive(&bars[B_UEMPTY0 + k % nub]);
                const int npairs = (U + 1) >> 1;
                if (warp == 2) {
                    if (!mbar_wait(&bars[B_QFULL], k & 1, abort_flag))
                        break;
                    for (int i = 0; i < npairs; ++i, ++gi) {
                        // the pair's K has landed; P.V of pair gi - 2 has read
                        // its P out of this TMEM buffer
                        if (!mbar_wait(&bars[B_KF0 + gi % NK], (gi / NK) & 1, abort_flag) ||
                            !mbar_wait(&bars[B_SFREE0 + (gi & 1)], ((gi >> 1) & 1) ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t k_s = smem_u32(sm + OFF_K) + (gi % NK) * kTileBytes;
                        for (int kk = 0; kk < kHead / 16; ++kk) {
                            const uint32_t o = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                            const uint32_t oq = (kk >> 2) * qhalf + (kk & 3) * 32;
                            mma_bf16(tmem + TM_S + (gi & 1) * 128, sdesc_sw128(q_s + oq, 16, qsbo),
                                     sdesc_sw128(k_s + o, 16, 1024), idS, kk > 0);
                        }
                        mma_commit(&bars[B_SFULL0 + (gi & 1)]);
                        mma_commit(&bars[B_KE0 + gi % NK]);
                    }
                    if (!ok)
                        break;
                    mma_commit(&bars[B_QEMPTY]);  // the next tile's Q may land
                } else {
                    // the epilogue has read the previous tile's O_e
                    if (!mbar_wait(&bars[B_ACCEMPTY], (k & 1) ^ 1, abort_flag))
                        break;
                    tc_fence_after();
                    for (int i = 0; i < npairs; ++i, ++gi) {
                        const int sb = gi & 1, sv = gi % NV;
                        if (!mbar_wait(&bars[B_PF00 + e * 2 + sb], (gi >> 1) & 1, abort_flag) ||
                            !mbar_wait(&bars[B_VF0 + sv], (gi / NV) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t v_s = smem_u32(sm + OFF_V) + sv * kTileBytes;
                        // O_e += P_e V_e: 64 keys, P from TMEM x the block's V (MN-major)
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16_ts(tmem + TM_O + e * 128, tmem + TM_S + sb * 128 + e * 64 + kk * 8,
                                        sdesc_sw128(v_s + (e * 4 + kk) * 2048, kHalfBytes, 1024), idO,
                                        (i > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&bars[B_PVFULL00 + e * 2 + sb]);
                        mma_commit(&bars[B_VE0 + sv]);
                        mma_commit(&bars[B_SFREE0 + sb]);
                    }
                    if (!ok)
                        break;
                    mma_commit(&bars[B_ACCFULL]);
                }
            }
            // every MMA of this thread completes before TMEM is freed
            uint64_t *done = &bars[B_DONE0 + warp - 1];
            mma_commit(done);
            volatile int never[2] = {0, abort_flag[1]};  // own limit, no abort
            mbar_wait(done, 0, never);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ----------------------------------------------------- softmax, epilogue
        // Warpgroup e (warps 4-7: e = 0, warps 8-11: e = 1) takes block e of
        // every pair (S columns e*64 .. e*64+63) into its accumulator O_e, and
        // output columns e*64 .. e*64+63 in the epilogue; warp w reads TMEM
        // lanes 32*(w%4) .. 32*(w%4)+31, so row r = 32*(w%4) + lane in both.
        const int e = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        int tl, hh;
        qtile_row(g, Tq, r, tl, hh);
        int gi = 0;
        for (int k = 0;; ++k) {
            if (!mbar_wait_warp(&bars[B_UFULL0 + k % nub], u_par(k), abort_flag))
                break;
            const volatile int *hdr = u_hdr(k);
            const int U = hdr[UH_COUNT];
            if (U < 0)
                break;
            const int b = hdr[UH_B], kvh = hdr[UH_KVH], t0 = hdr[UH_T0], nvalid = hdr[UH_NVALID];
            const int *list = union_list(u_buf(k), up);
            const int npairs = (U + 1) >> 1;
            const bool rvalid = r < nrows && tl < nvalid;
            const int t = GROUPED ? qtile_token(hdr, tl) : t0 + tl;  // the row's token
            // the row's keys: from the window's left edge to its diagonal
            const int cdiag = rvalid ? kdiag(g, b, t) : -1;
            const int khi = rvalid ? min(cdiag, seq_len_k(g, b) - 1) : -1, klo = key_lo(g, cdiag);
            const uint32_t *my_mask = union_mask(u_buf(k)) + (rvalid ? tl : 0) * words;
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int i = 0; i < npairs; ++i, ++gi) {
                const int sb = gi & 1;
                const int j = (2 * i + e < U) ? list[2 * i + e] : -1;
                const bool sel = rvalid && j >= 0 && qtile_selects(g, my_mask, klo, khi, j);
                // the row attends keys j*64 + c, lo <= c <= lim (lim < 0: none)
                const int lim = sel ? khi - j * kKeys : -1;
                const int lo = klo - j * kKeys;
                const bool any = __any_sync(0xffffffffu, sel);
                // no row of the warp ends or starts inside the block: a row attends
                // all of it or none; none gets a -inf bias
                const bool whole = __all_sync(0xffffffffu, lim < 0 || (lim >= kKeys - 1 && lo <= 0));
                if (!mbar_wait_warp(&bars[B_SFULL0 + sb], (gi >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sv[64];
                if (any) {
                    tmem_ld64(lane_base + TM_S + sb * 128 + e * 64, sv);
                    tmem_wait_ld();
                }
                uint32_t pk[32];
                if (any) {
                    float mb = -INFINITY;
                    if (whole) {
                        const float bias = sel ? 0.f : -INFINITY;
                        const uint64_t sc2 = f2(g.scale_l2, g.scale_l2), bb = f2(bias, bias);
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            float x0, x1;
                            f2_split(f2_fma(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2, bb), x0, x1);
                            sv[c] = __float_as_uint(x0);
                            sv[c + 1] = __float_as_uint(x1);
                            mb = fmaxf(mb, fmaxf(x0, x1));
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            const float x = __uint_as_float(sv[c]) * g.scale_l2;
                            sv[c] = __float_as_uint(x);
                            if (c <= lim && c >= lo)
                                mb = fmaxf(mb, x);
                        }
                    }
                    const bool raise = mb > m + kRescaleLog2;
                    if (__any_sync(0xffffffffu, raise)) {
                        const float alpha = raise ? ex2(m - mb) : 1.f;  // 0 when m = -inf
                        if (i > 0) {
                            // O_e must hold every earlier pair of the tile before it is rescaled
                            if (!mbar_wait_warp(&bars[B_PVFULL00 + e * 2 + ((gi - 1) & 1)], ((gi - 1) >> 1) & 1,
                                                abort_flag)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                uint32_t a[16];
                                tmem_ld16(lane_base + TM_O + e * 128 + c * 16, a);
                                tmem_wait_ld();
#pragma unroll
                                for (int x = 0; x < 16; ++x)
                                    a[x] = __float_as_uint(__uint_as_float(a[x]) * alpha);
                                tmem_st16(lane_base + TM_O + e * 128 + c * 16, a);
                            }
                            tmem_wait_st();
                        }
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
                        for (int c = 0; c < 64; c += 2) {
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
                        for (int c = 0; c < 64; c += 2) {
                            const float p0 = (c <= lim && c >= lo) ? ex2(__uint_as_float(sv[c]) - m) : 0.f;
                            const float p1 = (c + 1 <= lim && c + 1 >= lo) ? ex2(__uint_as_float(sv[c + 1]) - m) : 0.f;
                            rs += p0 + p1;
                            pk[c >> 1] = pack_bf16(p0, p1);
                        }
                    }
                    l += rs;
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        pk[c] = 0u;
                }
                // P_e over the first half of this block's S columns
                tmem_st32(lane_base + TM_S + sb * 128 + e * 64, pk);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[B_PF00 + e * 2 + sb]);
            }
            if (!ok)
                break;
            mbar_arrive(&bars[B_UEMPTY0 + k % nub]);  // the union buffer may be rebuilt
            // epilogue: merge the two warpgroups' row statistics, then output
            // columns e*64 .. e*64+63 = (a_0 O_0 + a_1 O_1) / l
            float2 *xk = xchg + (k & 1) * 2 * kRows;
            xk[e * kRows + r] = make_float2(m, l);
            mbar_arrive(&bars[B_XCHG0 + (k & 1)]);
            if (!mbar_wait_warp(&bars[B_XCHG0 + (k & 1)], (k >> 1) & 1, abort_flag))
                break;
            const float2 other = xk[(e ^ 1) * kRows + r];
            const float mx = fmaxf(m, other.x);
            const float a_me = m == -INFINITY ? 0.f : ex2(m - mx);
            const float a_ot = other.x == -INFINITY ? 0.f : ex2(other.x - mx);
            const float lsum = l * a_me + other.y * a_ot;
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            const float c0 = (e == 0 ? a_me : a_ot) * inv, c1 = (e == 0 ? a_ot : a_me) * inv;
            if (!mbar_wait_warp(&bars[B_ACCFULL], k & 1, abort_flag))
                break;
            tc_fence_after();
            __nv_bfloat16 *dst = rvalid ? p.o + o_off(g, b, kvh * G + hh, t) + e * 64 : nullptr;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t o0[32], o1[32];
                tmem_ld32(lane_base + TM_O + e * 64 + h * 32, o0);
                tmem_ld32(lane_base + TM_O + 128 + e * 64 + h * 32, o1);
                tmem_wait_ld();
                if (h == 1) {
                    // the accumulators are read: free for the next tile before the stores
                    tc_fence_before();
                    mbar_arrive(&bars[B_ACCEMPTY]);
                }
                uint32_t w[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float v0 = __uint_as_float(o0[2 * x]) * c0 + __uint_as_float(o1[2 * x]) * c1;
                    const float v1 = __uint_as_float(o0[2 * x + 1]) * c0 + __uint_as_float(o1[2 * x + 1]) * c1;
                    w[x] = npairs > 0 ? pack_bf16(v0, v1) : 0u;
                }
                if (rvalid) {
                    if (p.v8) {
                        st_global_v8(dst + h * 32, w);
                        st_global_v8(dst + h * 32 + 16, w + 8);
                    } else {
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            *(uint4 *)(dst + h * 32 + x * 8) =
                                make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
                    }
                }
            }
            if (e == 0 && rvalid)
                p.lse[stat_off(g, b, kvh * G + hh, t)] =
                    lsum > 0.f ? (mx + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
        }
    }

    __syncthreads();
    if (*abort_flag && threadIdx.x == 0)
        set_error(p.err, NSA_ERR_DEVICE_TIMEOUT);
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
    // As a programmatic dependent this kernel may have started before
    // the index validation ended: its completion implies that one's (a no-op otherwise).
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_fwd_tc(const Geo &g, const void *q, const void *k, const void *v, const int *idx,
                          const int *utable, bool grouped, void *o, float *lse, int *err, int *tile_next,
                          bool after_kernel, cudaStream_t st)
{
    if (!qtile_shape_ok(g))
        return launch_fwd_simt(g, q, k, v, idx, o, lse, NSA_DTYPE_BF16, st);
    const int Tq = tile_tokens(g.G);
    const UnionBuf up = union_buf(g);
    const int fixed = OFF_UNION + kXchgBytes + NUM_BARS * 8 + 64 + 1024;  // + alignment slack
    const int nub = fixed + 2 * up.bytes <= kSmemLimit ? 2 : 1;
    const int smem = fixed + nub * up.bytes;
    if (smem > kSmemLimit)
        return launch_fwd_simt(g, q, k, v, idx, o, lse, NSA_DTYPE_BF16, st);
    CUtensorMap tq, tk, tv;
    const bool rg = !g.thd && (g.G % 8) == 0;  // row-group Q tile, one box per token
    const bool qmap = rg ? make_tmap_rows(&tq, q, g, g.Hq, g.G, g.sq, g.q_bt) : make_tmap(&tq, q, g, g.Hq, Tq, g.G, g.sq);
    if (!qmap || !make_tmap(&tk, k, g, g.Hkv, kKeys, 1, g.skv, true) || !make_tmap(&tv, v, g, g.Hkv, kKeys, 1, g.skv, true))
        return cudaErrorInvalidValue;
    Params p;
    p.g = g;
    p.idx = idx;
    p.utable = utable;
    p.o = (__nv_bfloat16 *)o;
    p.lse = lse;
    p.err = err;
    p.ntiles = ((g.T + Tq - 1) / Tq) * g.B * g.Hkv;
    p.nub = nub;
    // 32-byte stores when every row of o starts on a 32-byte boundary
    p.v8 = ((uintptr_t)o & 31) == 0 && (g.so.h % 16) == 0 && (g.so.t % 16) == 0 && (g.so.b % 16) == 0;
    p.tile_next = tile_next;
    p.wait_us = wait_test().wait_us;
    p.stall = wait_test().kernel == WAIT_TEST_FWD;
    int grid = num_sms();
    if (grid > p.ntiles)
        grid = p.ntiles;
    if (grid < 1)
        return cudaSuccess;
    auto fwd_tc = grouped && utable ? fwd_tc_kernel<true> : fwd_tc_kernel<false>;
    cudaFuncSetAttribute(fwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    // After the index validation, a programmatic dependent of it (the check
    // only reports errors; this kernel skips invalid entries by itself).
    if (after_kernel)
        return launch_dependent(fwd_tc, dim3(grid), dim3(384), smem, st, tq, tk, tv, p);
    fwd_tc<<<grid, 384, smem, st>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace nsa
