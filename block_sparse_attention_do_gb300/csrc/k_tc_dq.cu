// k_tc_dq.cu -- dQ on the tcgen05 tensor cores (bf16, D = 128, block_size
// = 64).
//
// Work is cut into query tiles: Tq consecutive tokens of one sequence times
// the G query heads of one kv head (Tq * G <= 128 rows, Tq = 128 / G).  A
// tile walks, two at a time, the ascending union U of the blocks its tokens
// select.  For a pair (j_a, j_b) of U (128 keys):
//   S = Q [K_a; K_b]^T,  dP = dO [V_a; V_b]^T           (M=128 rows, N=128 keys, K=128)
//   P = exp(scale S - LSE) where the row's token selects the key's block and
//   key <= token,  dS = P (dP - delta)
//   dQ += dS [K_a; K_b]                                 (M=128 rows, N=128 dims, K=128 keys)
// and writes dQ * scale once at the end.  Rows of a token that did not select
// a block get P = dS = 0 there, so the sum over U is exactly the sum over the
// token's own blocks.  Pairing keeps every MMA at N = 128: a tcgen05 MMA with
// M = 128 costs about the same for N = 64 as for N = 128.
//
// The kernel is persistent: one CTA per SM takes tiles from a launch-wide
// counter, heaviest (latest tokens) first, each claimed a tile ahead.  A
// selection tile's block union comes from a table built before the kernel
// (qtile_union_kernel, below); a dense tile's is a block range built here.
// The next tile's union, its Q/dO load and its first K/V pairs overlap the
// current tile's last pairs and epilogue: the union sits in one of two
// shared-memory buffers (one when two do not fit).
//
// dP has two TMEM buffers, so dP of the next pair runs while the softmax
// works on this one; dS (bf16 pairs) is written over the first 32 columns
// of its dP block and read from there as the A operand of dQ += dS K.  So K
// and V have rings of their own, carried across tiles: V is held from its
// load to dP, K from its load to the dQ product (three stages when they
// fit, else two).
//
// Roles (12 warps): warp 0 deals the tiles, copies in (or builds) each
// tile's block union and issues the TMA copies (the tile's Q and dO, then per pair its K boxes
// and its V boxes, one box per lane); one thread each of warps 2, 1 and 3
// issues the S, dP and dQ MMAs (warp 2 owns TMEM); warps 4-7 form dS of each
// pair's first block and warps 8-11 of its second, one row per thread (P
// from S while dP still runs), and split the epilogue's columns the same way.
#include "tc_common.cuh"

namespace nsa {

namespace {

using namespace tc;

constexpr int kMaxNK = 3;  // K pair stages (32 KB each)
constexpr int NV = 2;      // V pair stages (32 KB each)
constexpr int OFF_Q = 0;
constexpr int OFF_DO = OFF_Q + kTileBytes;
constexpr int OFF_K = OFF_DO + kTileBytes;  // then the V ring, then the union buffers (sized at launch)
constexpr int NUM_BARS = 32;
constexpr int kSmemLimit = 232448;  // opt-in dynamic shared memory per block

enum {
    B_QFULL = 0, B_QEMPTY, B_DOFULL, B_DOEMPTY, B_SFULL, B_SFREE, B_DPFULL0, B_DPFULL1, B_DPFREE0, B_DPFREE1,
    B_UFULL0, B_UFULL1, B_UEMPTY0, B_UEMPTY1, B_ACCFULL, B_ACCEMPTY, B_DONE0, B_DONE1, B_DONE2, B_DSF0, B_DSF1,
    B_KF0, B_KE0 = B_KF0 + kMaxNK, B_VF0 = B_KE0 + kMaxNK, B_VE0 = B_VF0 + NV, B_COUNT = B_VE0 + NV
};
static_assert(B_COUNT <= NUM_BARS, "barrier slots");
// threads releasing a tile's union: the loader warp, the three MMA threads
// and the 256 softmax threads
constexpr int kUnionUsers = 32 + 3 + 2 * kRows;

constexpr uint32_t TM_S = 0;     // S: 128 columns (keys)
constexpr uint32_t TM_DP = 128;  // dP buffer x at 128 + x*128 (keys); dS of block e over its columns e*64 .. +31
constexpr uint32_t TM_DQ = 384;  // dQ: 128 lanes (rows) x 128 columns (dims)
constexpr uint32_t TM_COLS = 512;

struct Params {
    Geo g;
    const int *idx;
    const int *utable;  // every tile's union buffer, built by qtile_union_kernel (null: built here)
    const float *lse, *delta;
    __nv_bfloat16 *dq;
    int *err;
    int ntiles;      // query tiles over all (b, kv head)
    int *tile_next;  // work counter, zero at launch
    int nub;     // union buffers (1 or 2)
    int v8;      // dq is 32-byte aligned: the epilogue stores 32 bytes at a time
    int nk;      // K pair stages (2 or 3)
    int wait_us;  // bounded-wait limit in microseconds (0: the default)
    int stall;    // self-test: the S-product issuer stays idle (see wait_test)
};

// GROUPED: the union table's tiles are grouped by shared blocks (each row's
// token is read from the tile's record); else a tile's row tl has token T0 + tl
template <bool GROUPED>
__global__ void __launch_bounds__(384, 1) dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                       const __grid_constant__ CUtensorMap tm_do,
                                                       const __grid_constant__ CUtensorMap tm_k,
                                                       const __grid_constant__ CUtensorMap tm_v,
                                                       const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Geo &g = p.g;
    const UnionBuf up = union_buf(g);
    const int nub = p.nub, NK = p.nk;
    const int OFF_V = OFF_K + NK * kTileBytes, OFF_UNION = OFF_V + NV * kTileBytes;
    const int off_bar = OFF_UNION + nub * up.bytes;
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
        mbar_init(&bars[B_DOFULL], 1);
        mbar_init(&bars[B_DOEMPTY], 1);
        mbar_init(&bars[B_SFULL], 1);
        mbar_init(&bars[B_SFREE], 2 * kRows);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars[B_DPFULL0 + x], 1);
            mbar_init(&bars[B_DPFREE0 + x], 1);
        }
        for (int x = 0; x < 3; ++x)
            mbar_init(&bars[B_DONE0 + x], 1);
        mbar_init(&bars[B_ACCFULL], 1);
        mbar_init(&bars[B_ACCEMPTY], 2 * kRows);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars[B_UFULL0 + x], 32);
            mbar_init(&bars[B_UEMPTY0 + x], kUnionUsers);
            mbar_init(&bars[B_DSF0 + x], 2 * kRows);
        }
        for (int s = 0; s < NK; ++s) {
            mbar_init(&bars[B_KF0 + s], 1);
            mbar_init(&bars[B_KE0 + s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&bars[B_VF0 + s], 1);
            mbar_init(&bars[B_VE0 + s], 1);
        }
        fence_barrier_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    // Tile rows past Tq * G receive no data; they meet P = dS = 0 but must be
    // finite.  (A pair's missing second block is loaded as a copy of its first.)
    // With G % 8 == 0 in BHTD the Q and dO tiles are in the row-group layout
    // (one TMA box per token: its G heads, both halves), else rows of 128
    // bytes per half.
    const bool rg = !g.thd && (G % 8) == 0;
    if (nrows < kRows)
        for (int i = threadIdx.x; i < 4 * (kRows - nrows) * 8; i += blockDim.x) {
            const int part = i / ((kRows - nrows) * 8), rem = i % ((kRows - nrows) * 8);
            const int row = nrows + (rem >> 3), half = part & 1, tensor = part >> 1;
            *(uint4 *)(sm + OFF_Q + tensor * kTileBytes + (rg ? rg_off(row, half) : half * kHalfBytes + row * 128) +
                       (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // registers: the role warps (warpgroup 0) need few, the softmax warps many
    // (launch: 384 x 168 = 64512; after: 128 x 96 + 256 x 200 = 63488)
    if (warp < 4)
        setmaxnreg_dec<96>();
    else
        setmaxnreg_inc<200>();

    if (warp == 0) {
        // ------------------------------------------------------------- TMA
        // One TMA box per lane: issuing them from a single thread serialises
        // about a hundred cycles per box.
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_do);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
        int lastq = -1, lastd = -1, last = -1, lastv = -1, gi = 0;
        int claimed = qtile_claim(p.tile_next, lane);
        for (int k = 0;; ++k) {
            // The tile and its block union: this warp deals the tiles (each
            // claimed a tile ahead) and copies in (or builds) each union after
            // issuing the previous tile's copies, while the K/V rings still
            // hold several of that tile's pairs; after the last tile a header
            // with a negative count tells the other roles to stop.
            int b = 0, kvh = 0, t0 = 0, nvalid = 0, L = 0;
            const bool more = qtile_take(g, p.ntiles, p.tile_next, lane, claimed, b, kvh, t0, nvalid, &L);
            if (!mbar_wait_warp(&bars[B_UEMPTY0 + k % nub], u_par(k) ^ 1, abort_flag))
                break;
            if (more && p.utable) {
                // the union was built before this kernel (qtile_union_kernel):
                // copy its buffer in, 16 bytes per lane and step
                const uint4 *src = (const uint4 *)(p.utable + (int64_t)L * (up.bytes / 4));
                uint4 *dst = (uint4 *)u_buf(k);
                for (int x = lane; x < up.bytes / 16; x += 32)
                    dst[x] = src[x];
                __syncwarp();
            } else if (more) {
                // a dense entry's union is a block range: cheap to build here
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
            // Q once the previous tile's last S has run, dO once its last dP has
            bool ok = true;
            for (int tensor = 0; tensor < 2 && ok; ++tensor) {
                if (!mbar_wait_warp(&bars[tensor ? B_DOEMPTY : B_QEMPTY], (k & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                uint64_t *bar = &bars[tensor ? B_DOFULL : B_QFULL];
                if (lane == 0)
                    mbar_arrive_expect_tx(bar, nrows * 128 * 2);
                __syncwarp();
                (tensor ? lastd : lastq) = k;
                const CUtensorMap *map = tensor ? &tm_do : &tm_q;
                uint8_t *base = sm + (tensor ? OFF_DO : OFF_Q);
                if (rg) {  // token box: G heads x both halves, contiguous in the row-group layout
                    for (int tl = lane; tl < Tq; tl += 32)
                        if (tensor ? g.o_bt : g.q_bt)  // batch folded into the token index
                            tma_load_5d(base + tl * G * 256, map, bar, 0, 0, 0, kvh * G / 8,
                                        b * g.T + (GROUPED ? qtile_token(u_hdr(k), tl) : t0 + tl));
                        else
                            tma_load_5d(base + tl * G * 256, map, bar, 0, 0, 0, (b * g.Hq + kvh * G) / 8,
                                        GROUPED ? qtile_token(u_hdr(k), tl) : t0 + tl);
                } else if (lane < 2) {
                    const int h = lane;
                    if (g.thd)
                        tma_load_3d(base + h * kHalfBytes, map, bar, h * 64, kvh * G, g.cu[b] + t0);
                    else
                        tma_load_4d(base + h * kHalfBytes, map, bar, h * 64, t0, kvh * G, b);
                }
            }
            if (!ok)
                break;
            for (int i = 0; i < (U + 1) >> 1; ++i, ++gi) {
                // lane -> (block e of the pair, 64-column half h); K first (S
                // needs K only), then V once its stage is free.  A missing
                // second block repeats the first (finite data, P = dS = 0).
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
            if (lastd >= 0)
                mbar_wait(&bars[B_DOFULL], lastd & 1, never);
            if (last >= 0)
                mbar_wait(&bars[B_KF0 + last % NK], (last / NK) & 1, never);
            if (lastv >= 0)
                mbar_wait(&bars[B_VF0 + lastv % NV], (lastv / NV) & 1, never);
        }
        __syncwarp();
    } else if (warp <= 3) {
        // ---------------------------------------------------------------- MMA
        // Three issuing threads in three warps (one thread issues a tcgen05 MMA
        // only every ~150 cycles): warp 2 issues S, warp 1 dP (whose completion
        // frees the V stage), warp 3 dQ (whose completion frees the K stage
        // and the dP buffer holding dS), so a ready product never queues behind
        // another's issue.  Each commit covers its own thread's MMAs.
        if (lane == 0) {
            const uint32_t q_s = smem_u32(sm + OFF_Q), do_s = smem_u32(sm + OFF_DO);
            const uint32_t k_ring = smem_u32(sm + OFF_K), v_ring = smem_u32(sm + OFF_V);
            // Q/dO tiles: 64-column halves and 8-row groups apart by these
            const uint32_t qhalf = rg ? kRgHalf : kHalfBytes, qsbo = rg ? kRgStride : 1024;
            const uint32_t idS = idesc_bf16(128, 128, false, false), idQ = idesc_bf16(128, 128, false, true);
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
                    // S = Q K^T, once the tile's Q has landed
                    if (!mbar_wait(&bars[B_QFULL], k & 1, abort_flag))
                        break;
                    for (int i = 0; i < npairs; ++i, ++gi) {
                        // the pair's K has landed; the softmax has taken the previous S
                        if (!mbar_wait(&bars[B_KF0 + gi % NK], (gi / NK) & 1, abort_flag) ||
                            !mbar_wait(&bars[B_SFREE], (gi & 1) ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t k_s = k_ring + (gi % NK) * kTileBytes;
                        for (int kk = 0; kk < kHead / 16; ++kk) {
                            const uint32_t o = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                            const uint32_t oq = (kk >> 2) * qhalf + (kk & 3) * 32;
                            mma_bf16(tmem + TM_S, sdesc_sw128(q_s + oq, 16, qsbo), sdesc_sw128(k_s + o, 16, 1024),
                                     idS, kk > 0);
                        }
                        mma_commit(&bars[B_SFULL]);
                    }
                    if (!ok)
                        break;
                    mma_commit(&bars[B_QEMPTY]);  // the next tile's Q may land
                } else if (warp == 1) {
                    // dP = dO V^T, once the tile's dO has landed
                    if (!mbar_wait(&bars[B_DOFULL], k & 1, abort_flag))
                        break;
                    for (int i = 0; i < npairs; ++i, ++gi) {
                        // the V has landed; dQ of pair gi - 2 has read its dS out
                        // of this dP buffer
                        if (!mbar_wait(&bars[B_VF0 + gi % NV], (gi / NV) & 1, abort_flag) ||
                            !mbar_wait(&bars[B_DPFREE0 + (gi & 1)], ((gi >> 1) & 1) ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t v_s = v_ring + (gi % NV) * kTileBytes;
                        for (int kk = 0; kk < kHead / 16; ++kk) {
                            const uint32_t o = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                            const uint32_t oq = (kk >> 2) * qhalf + (kk & 3) * 32;
                            mma_bf16(tmem + TM_DP + (gi & 1) * 128, sdesc_sw128(do_s + oq, 16, qsbo),
                                     sdesc_sw128(v_s + o, 16, 1024), idS, kk > 0);
                        }
                        mma_commit(&bars[B_DPFULL0 + (gi & 1)]);
                        mma_commit(&bars[B_VE0 + gi % NV]);
                    }
                    if (!ok)
                        break;
                    mma_commit(&bars[B_DOEMPTY]);  // the next tile's dO may land
                } else {
                    // the epilogue has read the previous tile's dQ
                    if (!mbar_wait(&bars[B_ACCEMPTY], (k & 1) ^ 1, abort_flag))
                        break;
                    tc_fence_after();
                    for (int i = 0; i < npairs; ++i, ++gi) {
                        // dQ += dS K once the pair's dS is in TMEM; the commits free
                        // the K stage and the dP buffer
                        const int db = gi & 1, sk = gi % NK;
                        if (!mbar_wait(&bars[B_DSF0 + db], (gi >> 1) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t k_s = k_ring + sk * kTileBytes;
                        for (int kk = 0; kk < 8; ++kk)  // 128 keys: dS (TMEM) x K pair (MN-major)
                            mma_bf16_ts(tmem + TM_DQ, tmem + TM_DP + db * 128 + (kk >> 2) * 64 + (kk & 3) * 8,
                                        sdesc_sw128(k_s + kk * 2048, kHalfBytes, 1024), idQ,
                                        (i > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&bars[B_KE0 + sk]);
                        mma_commit(&bars[B_DPFREE0 + db]);
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
        // Two warpgroups: warpgroup e (warps 4-7: e = 0, warps 8-11: e = 1)
        // takes block e of every pair (S/dP columns e*64 .. e*64+63) and dQ
        // columns e*64 .. e*64+63 in the epilogue; warp w reads TMEM lanes
        // 32*(w%4) .. 32*(w%4)+31, so row r = 32*(w%4) + lane in both.
        const int e = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        int tl, hh;
        qtile_row(g, Tq, r, tl, hh);
        int gi = 0;
        // A tile's header and this row's LSE / delta, fetched while the
        // previous tile's dQ products complete (the first tile's here); the
        // header stays in the union buffer until the tile releases it.
        int nU = -1;
        float nl2 = 0.f, ndl = 0.f;
        auto fetch = [&](int k) {
            nU = -1;
            if (!mbar_wait_warp(&bars[B_UFULL0 + k % nub], u_par(k), abort_flag))
                return;
            const volatile int *hdr = u_hdr(k);
            nU = hdr[UH_COUNT];
            if (nU >= 0 && r < nrows && tl < hdr[UH_NVALID]) {
                const int64_t so =
                    stat_off(g, hdr[UH_B], hdr[UH_KVH] * G + hh, GROUPED ? qtile_token(hdr, tl) : hdr[UH_T0] + tl);
                nl2 = p.lse[so];  // scaled by log2(e) at use, so the load does not stall here
                ndl = p.delta[so];
            }
        };
        fetch(0);
        for (int k = 0; nU >= 0; ++k) {
            const volatile int *hdr = u_hdr(k);
            const int U = nU, b = hdr[UH_B], kvh = hdr[UH_KVH], t0 = hdr[UH_T0], nvalid = hdr[UH_NVALID];
            const float l2 = nl2 * 1.4426950408889634f, dl = ndl;
            const int *list = union_list(u_buf(k), up);
            const int npairs = (U + 1) >> 1;
            const bool rvalid = r < nrows && tl < nvalid;
            const int t = GROUPED ? qtile_token(hdr, tl) : t0 + tl;  // the row's token
            // the row's keys: from the window's left edge to its diagonal
            const int cdiag = rvalid ? kdiag(g, b, t) : -1;
            const int khi = rvalid ? min(cdiag, seq_len_k(g, b) - 1) : -1, klo = key_lo(g, cdiag);
            // the row's dQ columns e*64 .. e*64+63
            __nv_bfloat16 *dst = rvalid ? p.dq + dq_off(g, b, kvh * G + hh, t) + e * 64 : nullptr;
            const uint32_t *my_mask = union_mask(u_buf(k)) + (rvalid ? tl : 0) * words;
            bool ok = true;
            for (int i = 0; i < npairs; ++i, ++gi) {
                const int db = gi & 1;  // dP buffer
                const int j = (2 * i + e < U) ? list[2 * i + e] : -1;
                const bool sel = rvalid && j >= 0 && qtile_selects(g, my_mask, klo, khi, j);
                // the row attends keys j*64 + c, lo <= c <= lim (lim < 0: none)
                const int lim = sel ? khi - j * kKeys : -1;
                const int lo = klo - j * kKeys;
                // no row of the warp ends or starts inside the block: a row attends
                // all of it or none; none gets a +inf bias (exp2(-inf) = 0)
                const bool whole = __all_sync(0xffffffffu, lim < 0 || (lim >= kKeys - 1 && lo <= 0));
                const bool any = __any_sync(0xffffffffu, sel);
                // P = exp2(scale S - LSE) on the attended keys, while dP is still running
                if (!mbar_wait_warp(&bars[B_SFULL], gi & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t pv[64];
                tmem_ld64(lane_base + TM_S + e * 64, pv);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bars[B_SFREE]);
                if (any) {
                    if (whole) {
                        const float bias = sel ? l2 : __int_as_float(0x7f800000);
                        const uint64_t sc2 = f2(g.scale_l2, g.scale_l2), nb2 = f2(-bias, -bias);
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            float x0, x1;
                            f2_split(f2_fma(f2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])), sc2, nb2), x0,
                                     x1);
                            pv[c] = __float_as_uint(ex2(x0));
                            pv[c + 1] = __float_as_uint(ex2(x1));
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            pv[c] = __float_as_uint(
                                (c <= lim && c >= lo) ? ex2(__uint_as_float(pv[c]) * g.scale_l2 - l2) : 0.f);
                    }
                }
                // dS = P (dP - delta)
                if (!mbar_wait_warp(&bars[B_DPFULL0 + db], (gi >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t dv_[64];
                tmem_ld64(lane_base + TM_DP + db * 128 + e * 64, dv_);
                tmem_wait_ld();
                uint32_t dk_[32];
                if (any) {
                    const uint64_t nd2 = f2(-dl, -dl);
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        float d0, d1;
                        f2_split(f2_mul(f2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])),
                                        f2_add(f2(__uint_as_float(dv_[c]), __uint_as_float(dv_[c + 1])), nd2)),
                                 d0, d1);
                        dk_[c >> 1] = pack_bf16(d0, d1);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        dk_[c] = 0u;
                }
                // dS over the first half of this block's dP columns
                tmem_st32(lane_base + TM_DP + db * 128 + e * 64, dk_);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars[B_DSF0 + db]);
            }
            if (!ok)
                break;
            mbar_arrive(&bars[B_UEMPTY0 + k % nub]);  // the union buffer may be rebuilt
            fetch(k + 1);
            // epilogue: dQ row r, columns e*64 .. e*64+63 = scale * TMEM.  Every
            // lane of the warp runs the TMEM loads (.sync.aligned); only valid
            // rows store.
            if (!mbar_wait_warp(&bars[B_ACCFULL], k & 1, abort_flag))
                break;
            tc_fence_after();
            // all 64 columns in one go; the accumulator is free for the next
            // tile's dQ products before the stores
            uint32_t acc[64];
            tmem_ld64(lane_base + TM_DQ + e * 64, acc);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&bars[B_ACCEMPTY]);
            uint32_t w[32];
#pragma unroll
            for (int x = 0; x < 32; ++x)
                w[x] = npairs > 0 ? pack_bf16(__uint_as_float(acc[2 * x]) * g.scale,
                                              __uint_as_float(acc[2 * x + 1]) * g.scale)
                                  : 0u;
            if (rvalid) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (p.v8) {
                        st_global_v8(dst + c * 16, w + 8 * c);
                    } else {
                        *(uint4 *)(dst + c * 16) = make_uint4(w[8 * c], w[8 * c + 1], w[8 * c + 2], w[8 * c + 3]);
                        *(uint4 *)(dst + c * 16 + 8) =
                            make_uint4(w[8 * c + 4], w[8 * c + 5], w[8 * c + 6], w[8 * c + 7]);
                    }
                }
            }
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
    // the dK/dV kernel ended: its completion implies that one's (a no-op otherwise).
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

namespace {

// Every query tile's union buffer, one warp per tile (built in shared memory,
// then copied out whole).  A programmatic dependent of the kernel before it:
// it reads only the index, so it runs alongside that kernel, and waits for
// it at the end so that its own completion implies that kernel's.
__global__ void __launch_bounds__(256) qtile_union_kernel(Geo g, const int *__restrict__ idx, int ntiles,
                                                          UnionBuf up, int *__restrict__ utable)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ int ubuf_all[];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int *buf = ubuf_all + w * (up.bytes / 4);
    for (int L = blockIdx.x * (blockDim.x >> 5) + w; L < ntiles; L += gridDim.x * (blockDim.x >> 5)) {
        int b, kvh, t0, nvalid;
        if (!qtile_of(g, L, b, kvh, t0, nvalid))
            continue;  // never taken
        qtile_union_warp(g, idx, up, buf, b, kvh, t0, nvalid, lane);
        uint4 *dst = (uint4 *)(utable + (int64_t)L * (up.bytes / 4));
        for (int x = lane; x < up.bytes / 16; x += 32)
            dst[x] = ((const uint4 *)buf)[x];
        __syncwarp();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Tiles grouped by shared blocks.  The tokens of Wt consecutive tiles (a
// window of W = Wt * Tq <= 64 or 128 tokens of one (b, kv head)) are dealt
// into the same number of tiles greedily: a tile starts with the window's first
// free token and takes, Tq - 1 times, the free token that adds the fewest
// blocks to its union (ties to the lower token).  A tile need not hold
// consecutive tokens, and tokens that share blocks make smaller unions: on
// uniformly drawn selections the block pairs a tile walks drop by ~13%
// (64-token windows) or ~16% (128); on selections that cluster, by more.
// One warp per window: lane l holds the block bitmaps of tokens l + 32 q in
// registers (every index entry read at once), and a pick is one warp-wide
// minimum of (cost, token).
// The union records go where qtile_union_kernel puts them, with UH_GROUPED
// set and the tokens as offsets from the window's start.  For tiles of
// 2 .. kGroupMaxTq tokens whose Q (and dO) rows the kernels load by token
// (row-group layout).
constexpr int kGroupWords = 8;  // block bitmap words a grouped window may need (nbmax <= 256)

// WORDS: the block bitmap's words, (nbmax + 31) / 32 rounded up to 1, 2, 4 or
// 8; TPL: tokens a lane holds, so a window holds up to 32 TPL tokens (64 or
// 128: the larger groups better and takes about twice as long)
template <int WORDS, int TPL>
__global__ void __launch_bounds__(128) qtile_group_kernel(Geo g, const int *__restrict__ idx, UnionBuf up,
                                                          int *__restrict__ utable)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int words = (g.nbmax + 31) / 32;
    const int Tq = tile_tokens(g.G), Wt = 32 * TPL / Tq, W = Wt * Tq;
    const int nbg = g.B * g.Hkv, per_seq = (g.T + Tq - 1) / Tq, nwin = (per_seq + Wt - 1) / Wt;
    const bool vec = (g.S & 3) == 0 && ((uintptr_t)idx & 15) == 0;  // index rows in 16-byte pieces
    for (int item = blockIdx.x * (blockDim.x >> 5) + w; item < nbg * nwin; item += gridDim.x * (blockDim.x >> 5)) {
        const int bg = item % nbg, win = item / nbg;
        const int b = bg / g.Hkv, kvh = bg % g.Hkv;
        const int t0 = win * W, ntok = min(W, g.T - t0);
        // lane l holds window tokens l + 32 q (q < TPL): their block bitmaps,
        // and bit q of avail while the token is free
        uint32_t m[TPL][WORDS];
        uint32_t avail = 0u;
        int tq[TPL];
#pragma unroll
        for (int q = 0; q < TPL; ++q) {
#pragma unroll
            for (int x = 0; x < WORDS; ++x)
                m[q][x] = 0u;
            if (lane + 32 * q < ntok)
                avail |= 1u << q;
            tq[q] = t0 + min(lane + 32 * q, ntok - 1);  // a token past the window reads a valid row, unused
        }
        // the tokens' index entries: every load of a round issued before any is used
        for (int s0 = 0; s0 < g.S; s0 += 8) {
            int jv[TPL][8];
#pragma unroll
            for (int q = 0; q < TPL; ++q) {
                const int *row = idx_row(g, idx, b, kvh, tq[q]);
                if (vec) {
#pragma unroll
                    for (int u = 0; u < 8; u += 4) {
                        const int4 v4 = __ldg((const int4 *)(row + min(s0 + u, g.S - 4)));
                        jv[q][u] = v4.x;
                        jv[q][u + 1] = v4.y;
                        jv[q][u + 2] = v4.z;
                        jv[q][u + 3] = v4.w;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        jv[q][u] = __ldg(row + min(s0 + u, g.S - 1));
                }
            }
#pragma unroll
            for (int q = 0; q < TPL; ++q) {
                const int t = tq[q];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = jv[q][u];
                    const bool use = s0 + u < g.S && j >= 0 && j <= t / g.bs && j < g.nbmax;
                    const uint32_t bit = use ? 1u << (j & 31) : 0u;
#pragma unroll
                    for (int x = 0; x < WORDS; ++x)
                        m[q][x] |= (j >> 5) == x ? bit : 0u;
                }
            }
        }
        const int ntiles_w = (ntok + Tq - 1) / Tq;
        for (int k = 0; k < ntiles_w; ++k) {
            const int nk = min(Tq, ntok - k * Tq);
            const int tile = win * Wt + k;
            int *dst = utable + (int64_t)((per_seq - 1 - tile) * nbg + bg) * (up.bytes / 4);
            uint32_t *mask = (uint32_t *)(dst + UH_INTS), *ubits = mask + up.mask_words;
            int *list = dst + UH_INTS + up.mask_words + up.ubits_words;
            uint32_t cur[WORDS];
#pragma unroll
            for (int x = 0; x < WORDS; ++x)
                cur[x] = 0u;
            int slot[TPL];  // the tile row each of this lane's tokens took
#pragma unroll
            for (int q = 0; q < TPL; ++q)
                slot[q] = -1;
            for (int pick = 0; pick < nk; ++pick) {
                // key = cost << 8 | token: the free token adding the fewest
                // blocks (for the first pick every cost is 0: the lowest token)
                unsigned key = 0xffffffffu;
#pragma unroll
                for (int q = 0; q < TPL; ++q) {
                    unsigned cost = 0u;
#pragma unroll
                    for (int x = 0; x < WORDS; ++x)
                        cost += __popc(m[q][x] & ~cur[x]);
                    if ((avail >> q) & 1u)
                        key = min(key, (cost << 8) | (unsigned)(lane + 32 * q));
                }
                key = __reduce_min_sync(0xffffffffu, key);
                if (key == 0xffffffffu)
                    break;  // (never: a window's tiles take exactly its tokens)
                const int best = (int)(key & 0xffu), owner = best & 31, qb = best >> 5;
                // the token's bitmap from its lane into the union
#pragma unroll
                for (int x = 0; x < WORDS; ++x) {
                    uint32_t v = m[0][x];
#pragma unroll
                    for (int q = 1; q < TPL; ++q)
                        v = qb == q ? m[q][x] : v;
                    cur[x] |= __shfl_sync(0xffffffffu, v, owner);
                }
                // the owner's bookkeeping as selects: no divergent branch on the chain
                const bool mine = lane == owner;
                avail &= mine ? ~(1u << qb) : 0xffffffffu;
#pragma unroll
                for (int q = 0; q < TPL; ++q)
                    slot[q] = mine && qb == q ? pick : slot[q];
            }
            // the tile's rows: each token's bitmap by its lane, then empty
            // bitmaps for rows past the tile's tokens
#pragma unroll
            for (int q = 0; q < TPL; ++q) {
                const int sl = slot[q];
                if (sl >= 0)
#pragma unroll
                    for (int x = 0; x < WORDS; ++x)
                        if (x < words)
                            mask[sl * words + x] = m[q][x];
            }
            for (int x = nk * words + lane; x < up.mask_words; x += 32)
                mask[x] = 0u;
            // the union bitmap, and its blocks in ascending order (lane x <
            // words takes word x)
            uint32_t bits = 0u;
#pragma unroll
            for (int x = 0; x < WORDS; ++x)
                if (lane == x)
                    bits = cur[x];
            for (int x = lane; x < up.ubits_words; x += 32)
                ubits[x] = x < words ? bits : 0u;
            const int cnt = __popc(bits);
            int incl = cnt;
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off)
                    incl += y;
            }
            int pos = incl - cnt;
            for (uint32_t bb = bits; bb; bb &= bb - 1u)
                list[pos++] = lane * 32 + __ffs(bb) - 1;
            const int total = __shfl_sync(0xffffffffu, incl, 31);  // every lane takes part
            // the tile's tokens, byte r of the words = row r's offset in the window
#pragma unroll
            for (int x = 0; x < kGroupMaxTq / 4; ++x) {
                uint32_t part = 0u;
#pragma unroll
                for (int q = 0; q < TPL; ++q)
                    if (slot[q] >= 0 && (slot[q] >> 2) == x)
                        part |= (uint32_t)(lane + 32 * q) << ((slot[q] & 3) * 8);
                part = __reduce_or_sync(0xffffffffu, part);
                if (lane == x)
                    dst[UH_TOK + x] = (int)part;
            }
            if (lane == 0) {
                dst[UH_B] = b;
                dst[UH_KVH] = kvh;
                dst[UH_T0] = t0;
                dst[UH_NVALID] = nk;
                dst[UH_COUNT] = total;
                dst[UH_GROUPED] = 1;
            }
            __syncwarp();
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

bool qtile_groupable(const Geo &g)
{
    const int Tq = tile_tokens(g.G);
    return !g.dense && !g.thd && g.G % 8 == 0 && Tq >= 2 && Tq <= kGroupMaxTq && g.nbmax <= 32 * kGroupWords &&
           qtile_shape_ok(g);
}

size_t qtile_union_table_bytes(const Geo &g)
{
    if (g.dense || !qtile_shape_ok(g))
        return 0;
    const int Tq = tile_tokens(g.G);
    return (size_t)((g.T + Tq - 1) / Tq) * g.B * g.Hkv * union_buf(g).bytes;
}

cudaError_t launch_qtile_unions(const Geo &g, const int *idx, int *utable, cudaStream_t st, bool group, int tpl)
{
    if (qtile_union_table_bytes(g) == 0)
        return cudaSuccess;
    const int Tq = tile_tokens(g.G);
    const int ntiles = ((g.T + Tq - 1) / Tq) * g.B * g.Hkv;
    const UnionBuf up = union_buf(g);
    if (group && qtile_groupable(g)) {
        tpl = tpl < 2 ? 2 : tpl > 4 ? 4 : tpl;
        const int Wt = 32 * tpl / Tq, nwin = ((g.T + Tq - 1) / Tq + Wt - 1) / Wt;
        const int items = g.B * g.Hkv * nwin, grid = (items + 3) / 4;
        if (grid < 1)
            return cudaSuccess;
        const int words = (g.nbmax + 31) / 32;
        auto pick = [&](auto tpl) {
            constexpr int T_ = decltype(tpl)::value;
            return words <= 1 ? qtile_group_kernel<1, T_> : words <= 2 ? qtile_group_kernel<2, T_>
                 : words <= 4 ? qtile_group_kernel<4, T_> : qtile_group_kernel<8, T_>;
        };
        auto kern = tpl == 4 ? pick(std::integral_constant<int, 4>())
                  : tpl == 3 ? pick(std::integral_constant<int, 3>()) : pick(std::integral_constant<int, 2>());
        return launch_dependent(kern, dim3(grid), dim3(128), 0, st, g, idx, up, utable);
    }
    const int grid = (ntiles + 7) / 8;
    if (grid < 1)
        return cudaSuccess;
    const size_t smem = (size_t)8 * up.bytes;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(qtile_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_dependent(qtile_union_kernel, dim3(grid), dim3(256), smem, st, g, idx, ntiles, up, utable);
}

cudaError_t launch_dq_tc(const Geo &g, const void *q, const void *k, const void *v, const void *dO,
                         const float *lse, const float *delta, const int *idx, const int *utable, bool grouped,
                         void *dq, int *err, int *tile_next, cudaStream_t st)
{
    if (!qtile_shape_ok(g))
        return launch_dq_simt(g, q, k, v, dO, lse, delta, idx, dq, NSA_DTYPE_BF16, st);
    const int Tq = tile_tokens(g.G);
    const UnionBuf up = union_buf(g);
    // three K stages and two union buffers when they fit, else fewer
    const int base = OFF_K + NV * kTileBytes + NUM_BARS * 8 + 64 + 1024;  // + alignment slack
    int nk = 0, nub = 0;
    for (int c = 0; c < 4 && !nk; ++c) {
        const int k_ = c < 2 ? 3 : 2, u_ = 2 - (c & 1);
        if (base + k_ * kTileBytes + u_ * up.bytes <= kSmemLimit) {
            nk = k_;
            nub = u_;
        }
    }
    if (!nk)
        return launch_dq_simt(g, q, k, v, dO, lse, delta, idx, dq, NSA_DTYPE_BF16, st);
    const int smem = base + nk * kTileBytes + nub * up.bytes;
    CUtensorMap tq, tdo, tk, tv;
    const bool rg = !g.thd && (g.G % 8) == 0;  // row-group Q/dO tiles, one box per token and tensor
    const bool qmaps = rg ? make_tmap_rows(&tq, q, g, g.Hq, g.G, g.sq, g.q_bt) &&
                                make_tmap_rows(&tdo, dO, g, g.Hq, g.G, g.so, g.o_bt)
                          : make_tmap(&tq, q, g, g.Hq, Tq, g.G, g.sq) && make_tmap(&tdo, dO, g, g.Hq, Tq, g.G, g.so);
    if (!qmaps || !make_tmap(&tk, k, g, g.Hkv, kKeys, 1, g.skv, true) || !make_tmap(&tv, v, g, g.Hkv, kKeys, 1, g.skv, true))
        return cudaErrorInvalidValue;
    Params p;
    p.g = g;
    p.idx = idx;
    p.utable = utable;
    p.lse = lse;
    p.delta = delta;
    p.dq = (__nv_bfloat16 *)dq;
    p.err = err;
    p.ntiles = ((g.T + Tq - 1) / Tq) * g.B * g.Hkv;
    p.nub = nub;
    p.nk = nk;
    // 32-byte stores when every row of dq starts on a 32-byte boundary
    p.v8 = ((uintptr_t)dq & 31) == 0 && (g.sdq.h % 16) == 0 && (g.sdq.t % 16) == 0 && (g.sdq.b % 16) == 0;
    p.tile_next = tile_next;
    p.wait_us = wait_test().wait_us;
    p.stall = wait_test().kernel == WAIT_TEST_DQ;
    int grid = num_sms();
    if (grid > p.ntiles)
        grid = p.ntiles;
    if (grid < 1)
        return cudaSuccess;
    auto kernel = grouped && utable ? dq_tc_kernel<true> : dq_tc_kernel<false>;
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    // a programmatic dependent of the kernel before it on the stream (the dK/dV
    // kernel, whose outputs it does not read): its CTAs start as that kernel's
    // CTAs end; everything it reads was written by earlier, completed launches
    return launch_dependent(kernel, dim3(grid), dim3(384), smem, st, tq, tdo, tk, tv, p);
}

}  // namespace nsa
