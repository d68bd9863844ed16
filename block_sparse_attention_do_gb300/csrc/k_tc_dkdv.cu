// k_tc_dkdv.cu -- dK/dV on the tcgen05 tensor cores (bf16, D = 128,
// block_size = 64).
//
// One work unit is (sequence b, kv head g, kv block j, a run of the block's
// token list from the inverse index).  Its rows are (token, query head) pairs
// for the G query heads of the group, 128 rows per tile.  For every tile:
//   S   = Q K_j^T,  dP = dO V_j^T                     (M=128 rows, N=64 keys, K=128)
//   P   = exp(scale S - LSE) on the rows' attended keys, dS = P (dP - delta)
//   dV_j^T += dO^T P,  dK_j^T += Q^T dS               (M=128 dims, N=64 keys, K=128 rows)
// so the sum over the G heads (the GQA reduction) and over the tokens happens
// inside the accumulator, in a fixed order.  A block whose list is split over
// several units writes fp32 partials that a separate kernel adds in unit
// order; a block held by one unit writes dK/dV directly.
//
// Roles (15 warps; 16 with the third cp.async gather warp):  warps 0 and 3 load (TMA for K_j/V_j; Q rows from warp 0
// and dO rows from warp 3 by one TMA box per token -- its G heads, both
// halves -- when G % 8 == 0; else by 16-byte cp.async, two whole rows per
// warp instruction with the swizzle applied by hand, each lane's copies
// arriving on the tile's barrier as they land); warp 1 resolves each tile's token ids a tile
// ahead; warp 2 owns TMEM; one thread each of warps 2, 8, 9 and 10 issues the
// S, dP, dV^T and dK^T MMAs; two softmax warpgroups (warps 4-7 and 11-14, or
// 12-15 where warp 11 gathers) compute P/dS for one row each, keys 0..31 and
// 32..63 of the block (reading the row's LSE and delta themselves), and split
// the epilogue's columns the same way.  Q has three
// stages and dO two (row-group layout, so that a token's box is contiguous):
// a tile's Q is held from its load until dK^T has read it, its dO only from
// its load until dV^T has, so the dO ring refills later and needs fewer
// slots.  Three S/dP TMEM buffers (so S and dP run up to two tiles ahead of
// the softmax), one P and one dS buffer.
#include "tc_common.cuh"

namespace nsa {

namespace {

using namespace tc;

// shared-memory plan (bytes from a 1024-aligned base)
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + kKvBytes;
constexpr int NQ = 3;                            // Q stages
constexpr int NDO = 2;                           // dO stages
constexpr int NSB = 3;                           // S/dP TMEM buffers
constexpr int OFF_Q = OFF_V + kKvBytes;
constexpr int OFF_DO = OFF_Q + NQ * kTileBytes;
constexpr int NPB = 1;                           // P and dS shared-memory buffers (a second one measured slower: it costs a Q stage)
constexpr int OFF_P = OFF_DO + NDO * kTileBytes; // P buffer x at OFF_P + x * kRows * 128
constexpr int OFF_DS = OFF_P + NPB * kRows * 128;
constexpr int OFF_TOK = OFF_DS + NPB * kRows * 128;  // int [NQ][128]: a tile's token ids, one slot per Q stage
constexpr int OFF_BAR = OFF_TOK + NQ * kRows * 4;
constexpr int NUM_BARS = 40;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack

// barrier slots (QFULL/QEMPTY/IDX per Q stage, DOFULL/DOEMPTY per dO stage,
// SFULL/SFREE/DPFULL per S/dP buffer)
enum {
    B_QFULL0 = 0, B_QEMPTY0 = B_QFULL0 + NQ, B_IDX0 = B_QEMPTY0 + NQ, B_DOFULL0 = B_IDX0 + NQ,
    B_DOEMPTY0 = B_DOFULL0 + NDO, B_KVFULL = B_DOEMPTY0 + NDO, B_KVEMPTY, B_SFULL0,
    B_SFREE0 = B_SFULL0 + NSB, B_DPFULL0 = B_SFREE0 + NSB, B_PFULL0 = B_DPFULL0 + NSB, B_PFREE0 = B_PFULL0 + NPB,
    B_DSFULL0 = B_PFREE0 + NPB, B_DSFREE0 = B_DSFULL0 + NPB, B_ACCFULL = B_DSFREE0 + NPB, B_ACCEMPTY, B_DONE0,
    B_DONE1, B_DONE2, B_DONE3, B_STAGED, B_COPIED, B_COUNT
};
static_assert(B_COUNT <= NUM_BARS, "barrier slots");
static_assert(OFF_MISC + 64 + 1024 <= 232448, "shared memory");

// TMEM columns
constexpr uint32_t TM_S = 0;                // S of buffer b at b*128, dP at b*128 + 64
constexpr uint32_t TM_DV = NSB * 128;       // dV^T: 128 lanes (d) x 64 columns (keys)
constexpr uint32_t TM_DK = TM_DV + 64;      // dK^T
constexpr uint32_t TM_COLS = 512;

struct Params {
    Geo g;
    const __nv_bfloat16 *q, *dO;
    const float *lse, *delta;
    const int *offsets, *rows;
    const Unit *units;
    const WsHeader *hdr;
    float *partials;
    __nv_bfloat16 *dk, *dv;
    int *err;
    int wait_us;  // bounded-wait limit in microseconds (0: the default)
    int stall;    // self-test: the S-product issuer stays idle (see wait_test)
};

// The CTA's k-th work unit, or -1 past the end.  Units are dealt to the CTAs
// in a snake (row k left to right for even k, right to left for odd k);
// with the unit list's longest-first order this balances the CTAs' work.
__device__ __forceinline__ int unit_of(int k, int n_units)
{
    const int G = gridDim.x, c = blockIdx.x;
    const int64_t ui = (int64_t)k * G + ((k & 1) ? G - 1 - c : c);
    return ui < n_units ? (int)ui : -1;
}

// How a tile's Q and dO rows arrive: one TMA box per token (its G heads,
// both halves; G % 8 == 0), two TMA tile boxes per tensor (the dense
// entries' units hold consecutive tokens; G % 8 != 0), or 16-byte cp.async
// (selection, G % 8 != 0).  ROWS and CPASYNC fill the row-group layout
// (rg_off); TILE fills one 64-column half after the other (rows head-major
// for BHTD, token-major for THD).  (Token boxes for one tensor and cp.async
// for the other measured three times slower than token boxes for both.)
enum { LOAD_ROWS = 0, LOAD_TILE = 1, LOAD_CPASYNC = 2 };

// Warps: 11, plus a third gather warp (warp 11) in the cp.async mode: one
// warp's cp.async gather of a 32 KB tile takes ~6,300 cycles (about 100 cycles
// per warp instruction), so three warps share both tensors' rows.  12 warps at
// 168 registers still fit (3 warps per SM sub-partition).
template <int MODE> constexpr int dkdv_threads() { return MODE == LOAD_CPASYNC ? 512 : 480; }
constexpr int kGatherWarps = 3;  // warps 0, 3 and 11 in the cp.async mode
// the second softmax warpgroup (keys 32..63 of every tile; the first, warps
// 4-7, takes keys 0..31): warps 11-14, or 12-15 in the cp.async mode
template <int MODE> constexpr int softmax1_warp0() { return MODE == LOAD_CPASYNC ? 12 : 11; }

template <int MODE>
__global__ void __launch_bounds__(dkdv_threads<MODE>(), 1) dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                         const __grid_constant__ CUtensorMap tm_do,
                                                         const __grid_constant__ CUtensorMap tm_k,
                                                         const __grid_constant__ CUtensorMap tm_v,
                                                         const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = (uint64_t *)(sm + OFF_BAR);
    volatile int *abort_flag = (volatile int *)(sm + OFF_MISC);
    uint32_t *tmem_slot = (uint32_t *)(sm + OFF_MISC + 16);
    int *tok_s = (int *)(sm + OFF_TOK);

    const Geo &g = p.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = g.G;
    const int Tt = G >= kRows ? 1 : kRows / G;  // tokens per tile
    const int nrows = Tt * G;                  // used rows per tile

    if (threadIdx.x == 0) {
        abort_flag[0] = 0;
        abort_flag[1] = p.wait_us;  // the wait limit (0: the default)
        for (int x = 0; x < NQ; ++x) {
            mbar_init(&bars[B_QFULL0 + x], MODE == LOAD_CPASYNC ? 32 * kGatherWarps : 1);
            mbar_init(&bars[B_QEMPTY0 + x], 1);  // dK^T's commit
            mbar_init(&bars[B_IDX0 + x], 32);
        }
        for (int x = 0; x < NDO; ++x) {
            mbar_init(&bars[B_DOFULL0 + x], MODE == LOAD_CPASYNC ? 32 * kGatherWarps : 1);
            mbar_init(&bars[B_DOEMPTY0 + x], 2);  // dP's and dV^T's commits
        }
        mbar_init(&bars[B_KVFULL], 1);
        mbar_init(&bars[B_KVEMPTY], 2);
        for (int x = 0; x < NSB; ++x) {
            mbar_init(&bars[B_SFULL0 + x], 1);
            mbar_init(&bars[B_DPFULL0 + x], 1);
            mbar_init(&bars[B_SFREE0 + x], 2 * kRows);  // both softmax warpgroups
        }
        for (int x = 0; x < NPB; ++x) {
            mbar_init(&bars[B_PFULL0 + x], 2 * kRows);
            mbar_init(&bars[B_PFREE0 + x], 1);
            mbar_init(&bars[B_DSFULL0 + x], 2 * kRows);
            mbar_init(&bars[B_DSFREE0 + x], 1);
        }
        mbar_init(&bars[B_ACCFULL], 2);
        mbar_init(&bars[B_ACCEMPTY], 2 * kRows);
        mbar_init(&bars[B_STAGED], 2 * kRows);
        mbar_init(&bars[B_COPIED], 2 * kRows);
        for (int x = 0; x < 4; ++x)
            mbar_init(&bars[B_DONE0 + x], 1);
        fence_barrier_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    // rows a tile never fills must hold finite values (they meet P = 0)
    for (int i = threadIdx.x; i < ((NQ + NDO) * kTileBytes) / 16; i += blockDim.x)
        *(uint4 *)(sm + OFF_Q + i * 16) = make_uint4(0, 0, 0, 0);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the kernel before it (the
    // query-tile unions, whose completion implies the index build's; or the
    // index build or delta): everything above overlapped that kernel; nothing
    // it or an earlier launch writes is read before this wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_units = p.hdr->n_units;
    // The dQ kernel, launched next as a programmatic dependent, reads nothing
    // this kernel writes: let it take each SM as this kernel's CTA there ends.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0 || warp == 3 || (MODE == LOAD_CPASYNC && warp == 11)) {
        // ------------------------------------------------------- tile loader
        // K_j / V_j once per unit (warp 0); per tile, once the indexer has
        // published the tile's tokens (it does so when the tile's Q stage is
        // free), the Q and dO rows: by TMA when G % 8 == 0, one box per token
        // (its G heads, both halves), warp 0 the Q boxes and warp 3 the dO
        // boxes once the tile's dO stage is free (a box takes ~85 cycles to
        // issue, so two warps halve the time to the tile's last one); else by
        // 16-byte cp.async with the swizzle applied by hand, warps 0, 3 and
        // 11 each taking every third 8-row group of Q and then of dO.
        const int tensor = warp == 3 ? 1 : 0;
        const int gw = warp == 0 ? 0 : warp == 3 ? 1 : 2;  // cp.async: this warp's share of the row groups
        constexpr bool cpa = MODE == LOAD_CPASYNC;
        const uint32_t q_s = smem_u32(sm + OFF_Q), do_s = smem_u32(sm + OFF_DO);
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_do);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
        }
        int it = 0, uc = 0, qs = 0, qph = 0;  // tile count; its Q stage and that stage's phase
        int last_tile = -1, last_kv = -1;     // newest TMA batches (for the abort path)
        // cp.async gather: the swizzled destination of this lane's chunk in row
        // 2u + (lane >> 4) of an 8-row group, and ceil(2^16 / G) for r / G
        uint32_t dsto[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int rr = 2 * u + (lane >> 4), c = lane & 15;
            dsto[u] = (c >> 3) * kRgHalf + rr * 128 + (((c & 7) ^ rr) << 4);
        }
        const int recipG = (65536 + G - 1) / G;
        bool okl = true;
        for (int ui; (ui = unit_of(uc, n_units)) >= 0 && okl; ++uc) {
            const Unit u = p.units[ui];
            const int b = u.bg / g.Hkv, kvh = u.bg % g.Hkv;
            const int ntiles = (u.count + Tt - 1) / Tt;
            // the K/V stage frees once the previous unit's last S and dP have run
            if (warp == 0 && !mbar_wait_warp(&bars[B_KVEMPTY], (uc & 1) ^ 1, abort_flag)) {
                okl = false;
                break;
            }
            if (warp == 0 && lane == 0) {
                last_kv = uc;
                mbar_arrive_expect_tx(&bars[B_KVFULL], 2 * kKvBytes);
                for (int h = 0; h < 2; ++h) {
                    if (g.thd) {
                        const int t0 = g.cuk[b] + u.j * kKeys;
                        tma_load_3d(sm + OFF_K + h * kKvHalfBytes, &tm_k, &bars[B_KVFULL], h * 64, kvh, t0);
                        tma_load_3d(sm + OFF_V + h * kKvHalfBytes, &tm_v, &bars[B_KVFULL], h * 64, kvh, t0);
                    } else {
                        tma_load_4d(sm + OFF_K + h * kKvHalfBytes, &tm_k, &bars[B_KVFULL], h * 64, u.j * kKeys,
                                    kvh, b);
                        tma_load_4d(sm + OFF_V + h * kKvHalfBytes, &tm_v, &bars[B_KVFULL], h * 64, u.j * kKeys,
                                    kvh, b);
                    }
                }
            }
            for (int ti = 0; ti < ntiles; ++ti, ++it) {
                const int ds = it & 1;  // dO stage
                if (!mbar_wait_warp(&bars[B_IDX0 + qs], qph, abort_flag) ||
                    (!cpa && tensor == 1 && !mbar_wait_warp(&bars[B_DOEMPTY0 + ds], ((it >> 1) & 1) ^ 1, abort_flag))) {
                    okl = false;
                    break;
                }
                const int ntok = min(Tt, u.count - ti * Tt);
                const int *tok = tok_s + qs * kRows;
                if (MODE == LOAD_TILE) {
                    // the tile's tokens are consecutive: one box per 64-column half
                    uint64_t *full = tensor ? &bars[B_DOFULL0 + ds] : &bars[B_QFULL0 + qs];
                    if (lane == 0) {
                        last_tile = it;
                        mbar_arrive_expect_tx(full, nrows * 256);
                    }
                    __syncwarp();
                    if (lane < 2) {
                        const int h = lane, t0 = tok[0];
                        uint8_t *dst = sm + (tensor ? OFF_DO + ds * kTileBytes : OFF_Q + qs * kTileBytes) + h * kHalfBytes;
                        const CUtensorMap *map = tensor ? &tm_do : &tm_q;
                        if (g.thd)
                            tma_load_3d(dst, map, full, h * 64, kvh * G, g.cu[b] + t0);
                        else
                            tma_load_4d(dst, map, full, h * 64, t0, kvh * G, b);
                    }
                } else if (!cpa) {
                    uint64_t *full = tensor ? &bars[B_DOFULL0 + ds] : &bars[B_QFULL0 + qs];
                    if (lane == 0) {
                        last_tile = it;
                        mbar_arrive_expect_tx(full, nrows * 256);
                    }
                    __syncwarp();
                    for (int tl = lane; tl < Tt; tl += 32) {
                        // rows past the list repeat the last token (finite data, P = 0)
                        const int t = tok[min(tl, ntok - 1)];
                        uint8_t *dst = sm + (tensor ? OFF_DO + ds * kTileBytes : OFF_Q + qs * kTileBytes) + tl * G * 256;
                        const CUtensorMap *map = tensor ? &tm_do : &tm_q;
                        if (g.thd)
                            tma_load_5d(dst, map, full, 0, 0, 0, kvh * G / 8, g.cu[b] + t);
                        else if (tensor ? g.o_bt : g.q_bt)  // batch folded into the token index
                            tma_load_5d(dst, map, full, 0, 0, 0, kvh * G / 8, b * g.T + t);
                        else
                            tma_load_5d(dst, map, full, 0, 0, 0, (b * g.Hq + kvh * G) / 8, t);
                    }
                } else {
                    // cp.async: Q, then (once the tile's dO stage is free) dO; per
                    // tensor 128 rows x 16 chunks of 16 bytes, two whole rows
                    // (256 contiguous bytes each) per warp instruction, this warp
                    // taking 8-row groups gw, gw + 3, ...; rows past the tile's
                    // tokens are zero-filled.  Each lane's arrival on the
                    // tile's barrier lands once its copies have; the consumers
                    // fence them for the tensor cores after their wait.
                    const int c = lane & 15, hi = lane >> 4;
                    for (int tn = 0; tn < 2; ++tn) {
                        if (tn == 1 && !mbar_wait_warp(&bars[B_DOEMPTY0 + ds], ((it >> 1) & 1) ^ 1, abort_flag)) {
                            okl = false;
                            break;
                        }
                        const __nv_bfloat16 *base = tn ? p.dO : p.q;
                        const Strides &str = tn ? g.so : g.sq;
                        const uint32_t tile_s = tn ? do_s + ds * kTileBytes : q_s + qs * kTileBytes;
                        // lane: chunk c of rows 8*grp + 2u + hi; its head 0 of the
                        // group and its column, then per row token * stride_t + head * stride_h
                        const __nv_bfloat16 *rowbase = base + (int64_t)(kvh * G) * str.h + c * 8 +
                                                       (g.thd ? (int64_t)g.cu[b] * str.t : (int64_t)b * str.b);
                        for (int grp = gw; grp < kRows / 8; grp += kGatherWarps) {
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int r = grp * 8 + 2 * u + hi;
                                const int tl = (r * recipG) >> 16, hh = r - tl * G;  // r / G, r % G (r < 128)
                                const bool valid = r < nrows && tl < ntok;
                                const __nv_bfloat16 *src =
                                    valid ? rowbase + (int64_t)tok[tl] * str.t + (int64_t)hh * str.h : base;
                                cp_async_16(tile_s + grp * kRgStride + dsto[u], src, valid ? 16u : 0u);
                            }
                        }
                        cp_async_mbar_arrive(tn ? &bars[B_DOFULL0 + ds] : &bars[B_QFULL0 + qs]);
                    }
                    if (!okl)
                        break;
                }
                if (++qs == NQ) {
                    qs = 0;
                    qph ^= 1;
                }
            }
        }
        if (cpa)
            cp_async_wait<0>();  // every copy lands before the CTA may exit
        if (*abort_flag && lane == 0) {
            // let TMA copies still in flight land before the CTA exits
            volatile int never[2] = {0, abort_flag[1]};  // own limit, no abort
            if (last_tile >= 0) {
                if (tensor)
                    mbar_wait(&bars[B_DOFULL0 + (last_tile & 1)], (last_tile >> 1) & 1, never);
                else
                    mbar_wait(&bars[B_QFULL0 + last_tile % NQ], (last_tile / NQ) & 1, never);
            }
            if (last_kv >= 0)
                mbar_wait(&bars[B_KVFULL], last_kv & 1, never);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ indexer
        // Resolves each tile's token ids from the inverse index one tile
        // ahead, into registers, while the Q stage it will fill is still
        // busy; publishes them when that stage frees.  Lane l owns the
        // tile's tokens l, l + 32, l + 64, l + 96.
        int qs = 0, qph = 0;
        int ku = 0, ti = 0;
        int ui = unit_of(0, n_units);
        Unit u;
        int csr0 = 0, ntiles = 0;
        auto load_unit = [&]() {
            u = p.units[ui];
            // dense: the block's tokens are one range from its first attending row
            csr0 = g.dense ? dense_first(g, u.bg / g.Hkv, u.j) + u.begin : p.offsets[u.bg * g.nbmax + u.j] + u.begin;
            ntiles = (u.count + Tt - 1) / Tt;
        };
        int tok_r[4];
        auto fetch = [&]() {
            const int ntok = min(Tt, u.count - ti * Tt);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const int tl = lane + k4 * 32;
                tok_r[k4] = -1;
                if (tl < ntok) {
                    const int pos = ti * Tt + tl;
                    tok_r[k4] = g.dense ? csr0 + pos : p.rows[csr0 + pos];
                }
            }
        };
        if (ui >= 0) {
            load_unit();
            fetch();
        }
        while (ui >= 0) {
            if (!mbar_wait_warp(&bars[B_QEMPTY0 + qs], qph ^ 1, abort_flag))
                break;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
                if (lane + k4 * 32 < Tt)
                    tok_s[qs * kRows + lane + k4 * 32] = tok_r[k4];
            mbar_arrive(&bars[B_IDX0 + qs]);
            // next tile (possibly of the next unit): resolve its tokens now
            if (++qs == NQ) {
                qs = 0;
                qph ^= 1;
            }
            if (++ti == ntiles) {
                ti = 0;
                ui = unit_of(++ku, n_units);
                if (ui >= 0)
                    load_unit();
            }
            if (ui >= 0)
                fetch();
        }
    } else if (warp == 2 || (warp >= 8 && warp <= 10)) {
        // -------------------------------------------------------------- MMA
        // Four issuing threads in four warps (one thread issues a tcgen05 MMA
        // only every ~150 cycles): warp 2 issues S, warp 8 dP, warp 9 dV^T (as
        // soon as P is in shared memory) and warp 10 dK^T (once dS is); each
        // walks every (unit, tile).  KVEMPTY counts the S and dP commits,
        // ACCFULL the dV and dK ones; a Q stage is free once dK^T of its tile
        // is done, a dO stage once dP and dV^T of its tile are.
        if (lane == 0) {
            const int role = warp == 2 ? 0 : warp - 7;  // 0 S, 1 dP, 2 dV, 3 dK
            const uint32_t idS = idesc_bf16(128, 64, false, false);
            const uint32_t idV = idesc_bf16(128, 64, true, true);
            const uint32_t q_s = smem_u32(sm + OFF_Q), do_s = smem_u32(sm + OFF_DO);
            const uint32_t k_s = smem_u32(sm + OFF_K), v_s = smem_u32(sm + OFF_V);
            // Q/dO tiles: 64-column halves and 8-row groups apart by these
            const uint32_t qhalf = MODE == LOAD_TILE ? kHalfBytes : kRgHalf;
            const uint32_t qsbo = MODE == LOAD_TILE ? 1024 : kRgStride;
            const uint32_t p_s = smem_u32(sm + OFF_P), ds_s = smem_u32(sm + OFF_DS);
            // S / dP: A = Q / dO (row-group tile), B = K_j / V_j
            const bool on_do = role == 1 || role == 2;
            const uint32_t b_s = role == 1 ? v_s : k_s;
            int it = 0, uc = 0, qs = 0, qph = 0, tb = 0, tph = 0;  // (tb, tph): S/dP buffer and its phase
            // (self-test of the bounded waits: an idle S issuer makes the
            // softmax's first wait run out)
            bool ok = !(p.stall && role == 0);
            for (int ui; ok && (ui = unit_of(uc, n_units)) >= 0; ++uc) {
                const int ntiles = (p.units[ui].count + Tt - 1) / Tt;
                for (int ti = 0; ti < ntiles; ++ti, ++it) {
                    const int st = it & 1;  // dO stage
                    const uint32_t a_s = on_do ? do_s + st * kTileBytes : q_s + qs * kTileBytes;
                    if (role <= 1) {
                        // the tile's Q (S) or dO (dP) rows, and at a unit's start
                        // K_j / V_j, have landed; the softmax has loaded S/dP of
                        // tile it - NSB
                        if (!(role == 0 ? mbar_wait(&bars[B_QFULL0 + qs], qph, abort_flag)
                                        : mbar_wait(&bars[B_DOFULL0 + st], (it >> 1) & 1, abort_flag)) ||
                            !mbar_wait(&bars[B_SFREE0 + tb], tph ^ 1, abort_flag) ||
                            (ti == 0 && !mbar_wait(&bars[B_KVFULL], uc & 1, abort_flag))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (MODE == LOAD_CPASYNC)  // rows written by cp.async: order them for the tensor cores
                            fence_async_smem();
                        const uint32_t col = tmem + TM_S + tb * 128 + role * 64;
                        for (int kk = 0; kk < kHead / 16; ++kk) {
                            const uint32_t ao = (kk >> 2) * qhalf + (kk & 3) * 32;
                            const uint32_t bo = (kk >> 2) * kKvHalfBytes + (kk & 3) * 32;
                            mma_bf16(col, sdesc_sw128(a_s + ao, 16, qsbo), sdesc_sw128(b_s + bo, 16, 1024), idS,
                                     kk > 0);
                        }
                        mma_commit(&bars[(role == 0 ? B_SFULL0 : B_DPFULL0) + tb]);
                        if (role == 1)
                            mma_commit(&bars[B_DOEMPTY0 + st]);
                        if (ti + 1 == ntiles)
                            mma_commit(&bars[B_KVEMPTY]);
                    } else {
                        // P (dV) or dS (dK) of the tile is in shared memory (and
                        // for dV the tile's dO rows have landed); at a unit's
                        // start the epilogue has read the accumulators
                        const int pbuf = it % NPB;  // the tile's P / dS buffer
                        if (!mbar_wait(&bars[(role == 2 ? B_PFULL0 : B_DSFULL0) + pbuf], (it / NPB) & 1, abort_flag) ||
                            (role == 2 && !mbar_wait(&bars[B_DOFULL0 + st], (it >> 1) & 1, abort_flag)) ||
                            (ti == 0 && !mbar_wait(&bars[B_ACCEMPTY], (uc & 1) ^ 1, abort_flag))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (MODE == LOAD_CPASYNC)  // dO (dV^T) or Q (dK^T) written by cp.async
                            fence_async_smem();
                        const uint32_t col = tmem + (role == 2 ? TM_DV : TM_DK);
                        const uint32_t pb = (role == 2 ? p_s : ds_s) + pbuf * (kRows * 128);
                        for (int kr = 0; kr < kRows / 16; ++kr)
                            // 16 rows = two row groups; LBO steps the 64-dim halves (M)
                            mma_bf16(col, sdesc_sw128(a_s + kr * 2 * qsbo, qhalf, qsbo),
                                     sdesc_sw128(pb + kr * 2048, 8192, 1024), idV, (ti > 0 || kr > 0) ? 1u : 0u);
                        mma_commit(&bars[(role == 2 ? B_PFREE0 : B_DSFREE0) + pbuf]);
                        mma_commit(&bars[role == 2 ? B_DOEMPTY0 + st : B_QEMPTY0 + qs]);
                        if (ti + 1 == ntiles)
                            mma_commit(&bars[B_ACCFULL]);
                    }
                    if (++qs == NQ) {
                        qs = 0;
                        qph ^= 1;
                    }
                    if (++tb == NSB) {
                        tb = 0;
                        tph ^= 1;
                    }
                }
            }
            // every MMA issued must finish before TMEM is released
            mma_commit(&bars[B_DONE0 + role]);
            volatile int never[2] = {0, abort_flag[1]};  // own limit, no abort
            mbar_wait(&bars[B_DONE0 + role], 0, never);
        }
        __syncwarp();
    } else if ((warp >= 4 && warp < 8) || (warp >= softmax1_warp0<MODE>() && warp < softmax1_warp0<MODE>() + 4)) {
        // ------------------------------------------------- softmax / epilogue
        // two warpgroups, one row per thread each: keys (and, in the
        // epilogue, dK/dV columns) cb .. cb + 31
        const int half = warp >= 8 ? 1 : 0, cb = half * 32;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // tile row = TMEM lane
        // the row's token within the tile and head within the group
        // (head-major rows for a BHTD tile box, token-major otherwise)
        const bool head_major = MODE == LOAD_TILE && !g.thd;
        const int my_tl = head_major ? r % Tt : r / G, my_hh = head_major ? r / Tt : r % G;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const uint32_t p_row = smem_u32(sm + OFF_P) + r * 128;
        const uint32_t ds_row = smem_u32(sm + OFF_DS) + r * 128;
        // The next tile's token and raw LSE / delta for this thread's row,
        // read halfway through the tile before, so that the loads' latency
        // stays off the softmax's path.  (pq, pph): the next tile's Q stage
        // and phase; (pu, pti, p_ui): its unit and tile within the unit.
        int pq = 0, pph = 0, pu = 0, pti = 0;
        int p_ui = unit_of(0, n_units);
        int ptok = -1;
        float plse = 0.f, pdlt = 0.f;
        // The next tile's unit (its kv group and token count) stays in
        // registers, read again only when the unit changes: reading it for
        // every tile put a global load's latency on every tile's path.
        int nu_bg = 0, nu_cnt = 0;
        if (p_ui >= 0) {
            nu_bg = p.units[p_ui].bg;
            nu_cnt = p.units[p_ui].count;
        }
        auto prefetch = [&]() -> bool {
            if (p_ui < 0)
                return true;
            if (!mbar_wait_warp(&bars[B_IDX0 + pq], pph, abort_flag))
                return false;
            ptok = r < nrows ? tok_s[pq * kRows + my_tl] : -1;
            plse = 0.f;
            pdlt = 0.f;
            if (ptok >= 0) {
                const int64_t so = stat_off(g, nu_bg / g.Hkv, (nu_bg % g.Hkv) * G + my_hh, ptok);
                plse = p.lse[so];
                pdlt = p.delta[so];
            }
            if (++pq == NQ) {
                pq = 0;
                pph ^= 1;
            }
            if (++pti == (nu_cnt + Tt - 1) / Tt) {
                pti = 0;
                p_ui = unit_of(++pu, n_units);
                if (p_ui >= 0) {
                    nu_bg = p.units[p_ui].bg;
                    nu_cnt = p.units[p_ui].count;
                }
            }
            return true;
        };
        int it = 0, uc = 0, tb = 0, tph = 0;  // (tb, tph): S/dP buffer and its phase
        int ep = 0;                           // staged (direct) epilogues so far
        bool ok = prefetch();
        for (int ui; ok && (ui = unit_of(uc, n_units)) >= 0; ++uc) {
            const Unit u = p.units[ui];
            const int b = u.bg / g.Hkv, kvh = u.bg % g.Hkv;
            const int L = seq_len_k(g, b);  // keys of the sequence
            const int k0 = u.j * kKeys;
            const int ntiles = (u.count + Tt - 1) / Tt;
            for (int ti = 0; ti < ntiles; ++ti, ++it) {
                const int tok = ptok;
                const float l2 = plse * 1.4426950408889634f, dl = pdlt;
                if (!mbar_wait_warp(&bars[B_SFULL0 + tb], tph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // keys k0 + c with lo <= c <= lim are attended (the token selected block j):
                // from the window's left edge to the row's diagonal and the keys' end
                const int cdiag = tok < 0 ? -1 : kdiag(g, b, tok);
                const int lim = tok < 0 ? -1 : min(cdiag, L - 1) - k0;
                const int lo = tok < 0 ? 0 : key_lo(g, cdiag) - k0;  // window's left edge
                // P from S while dP is still running (this warpgroup's 32 keys)
                uint32_t pv[32];
                tmem_ld32(lane_base + TM_S + tb * 128 + cb, pv);
                tmem_wait_ld();
                if (__all_sync(0xffffffffu, lim < 0 || (lim >= kKeys - 1 && lo <= 0))) {
                    // no row of the warp ends or starts inside the block: a row
                    // attends all of it or none; none gets a +inf bias (exp2(-inf) = 0)
                    const float bias = lim >= 0 ? l2 : __int_as_float(0x7f800000);
                    const uint64_t sc2 = f2(g.scale_l2, g.scale_l2), nb2 = f2(-bias, -bias);
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        float x0, x1;
                        f2_split(f2_fma(f2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])), sc2, nb2), x0, x1);
                        pv[c] = __float_as_uint(ex2(x0));
                        pv[c + 1] = __float_as_uint(ex2(x1));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        pv[c] = __float_as_uint((cb + c <= lim && cb + c >= lo)
                                                    ? ex2(__uint_as_float(pv[c]) * g.scale_l2 - l2)
                                                    : 0.f);
                }
                // P (bf16) to shared memory as soon as the dV product of the
                // previous tile has read it: dV^T += dO^T P starts while dS forms
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2)
                    pk[c >> 1] = pack_bf16(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1]));
                const int pbuf = it % NPB;  // this tile's P / dS buffer
                if (!mbar_wait_warp(&bars[B_PFREE0 + pbuf], ((it / NPB) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_shared_v4(p_row + pbuf * (kRows * 128) + (((cb / 8 + c) ^ (r & 7)) << 4), pk[4 * c],
                                 pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                fence_async_smem();
                mbar_arrive(&bars[B_PFULL0 + pbuf]);
                if (!prefetch()) {
                    ok = false;
                    break;
                }
                // dS = P (dP - delta)
                if (!mbar_wait_warp(&bars[B_DPFULL0 + tb], tph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t dv_[32];
                tmem_ld32(lane_base + TM_S + tb * 128 + 64 + cb, dv_);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bars[B_SFREE0 + tb]);
                if (++tb == NSB) {
                    tb = 0;
                    tph ^= 1;
                }
                uint32_t dk_[16];
                const uint64_t nd2 = f2(-dl, -dl);
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float d0, d1;
                    const uint64_t pp = f2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1]));
                    f2_split(f2_mul(pp, f2_add(f2(__uint_as_float(dv_[c]), __uint_as_float(dv_[c + 1])), nd2)), d0, d1);
                    dk_[c >> 1] = pack_bf16(d0, d1);
                }
                if (!mbar_wait_warp(&bars[B_DSFREE0 + pbuf], ((it / NPB) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    st_shared_v4(ds_row + pbuf * (kRows * 128) + (((cb / 8 + c) ^ (r & 7)) << 4), dk_[4 * c],
                                 dk_[4 * c + 1], dk_[4 * c + 2], dk_[4 * c + 3]);
                fence_async_smem();
                mbar_arrive(&bars[B_DSFULL0 + pbuf]);
            }
            if (!ok)
                break;
            // ---- epilogue: lane = head dimension d, columns = keys.  A split
            // block's fp32 partials go out directly (each warp store covers
            // 128 contiguous bytes); a whole block's bf16 dK/dV rows are first
            // staged in the idle dS / P buffers (thread d writes column d) and
            // then written as whole 256-byte rows with 16-byte stores, since
            // 2-byte stores, 64 bytes per warp, drain many times slower.
            if (!mbar_wait_warp(&bars[B_ACCFULL], uc & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int d = r;
            const int nk = min(kKeys, L - k0);
            const bool direct = u.slot < 0;
            for (int which = 0; which < 2; ++which) {  // this warpgroup's keys cb .. cb + 31
                const uint32_t col = (which == 0 ? TM_DK : TM_DV) + cb;
                const float mul = which == 0 ? g.scale : 1.f;
                uint32_t a[32];
                tmem_ld32(lane_base + col, a);
                tmem_wait_ld();
                if (!direct) {
                    float *dst = p.partials + ((int64_t)u.slot * 2 + which) * kKeys * kHead + cb * kHead + d;
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        dst[c * kHead] = __uint_as_float(a[c]) * mul;
                } else {
                    // dS buffer holds dK, P buffer dV: [64 keys][128 dims] bf16
                    __nv_bfloat16 *stage = (__nv_bfloat16 *)(sm + (which == 0 ? OFF_DS : OFF_P)) + cb * kHead + d;
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        stage[c * kHead] = __float2bfloat16_rn(__uint_as_float(a[c]) * mul);
                }
            }
            if (direct) {
                // every row staged: copy both tensors out, 16 bytes per thread and step
                mbar_arrive(&bars[B_STAGED]);
                if (!mbar_wait_warp(&bars[B_STAGED], ep & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                // distance between consecutive keys (elements)
                const int64_t kstride = g.sdkv.t;
#pragma unroll 4
                for (int q = r + half * kRows; q < 2 * kKeys * 16; q += 2 * kRows) {
                    const int which = q / (kKeys * 16), c = (q >> 4) & (kKeys - 1), ch = q & 15;
                    if (c < nk) {
                        __nv_bfloat16 *out = (which == 0 ? p.dk : p.dv) + dkv_off(g, b, kvh, k0) + c * kstride;
                        *(uint4 *)(out + ch * 8) =
                            *(const uint4 *)(sm + (which == 0 ? OFF_DS : OFF_P) + c * (kHead * 2) + ch * 16);
                    }
                }
                // the buffers take the next unit's P and dS only after every thread's copy
                mbar_arrive(&bars[B_COPIED]);
                if (!mbar_wait_warp(&bars[B_COPIED], ep & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                ++ep;
            }
            tc_fence_before();
            mbar_arrive(&bars[B_ACCEMPTY]);
        }
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

cudaError_t launch_dkdv_tc(const Geo &g, const void *q, const void *k, const void *v,
                           const void *dO, const float *lse, const float *delta,
                           const int *offsets, const int *rows, const Unit *units,
                           const WsHeader *hdr, int max_units, float *partials, void *dk, void *dv,
                           int *err, cudaStream_t st)
{
    CUtensorMap tq, tdo, tk, tv;
    const int mode = g.G % 8 == 0 ? LOAD_ROWS : g.dense ? LOAD_TILE : LOAD_CPASYNC;
    const int Tt = g.G >= kRows ? 1 : kRows / g.G;
    bool qmaps;
    if (mode == LOAD_ROWS)
        qmaps = make_tmap_rows(&tq, q, g, g.Hq, g.G, g.sq, g.q_bt) && make_tmap_rows(&tdo, dO, g, g.Hq, g.G, g.so, g.o_bt);
    else if (mode == LOAD_TILE)
        qmaps = make_tmap(&tq, q, g, g.Hq, Tt, g.G, g.sq) && make_tmap(&tdo, dO, g, g.Hq, Tt, g.G, g.so);
    else
        qmaps = make_tmap(&tq, q, g, g.Hq, 1, 1, g.sq) && make_tmap(&tdo, dO, g, g.Hq, 1, 1, g.so);
    if (!qmaps || !make_tmap(&tk, k, g, g.Hkv, kKeys, 1, g.skv, true) || !make_tmap(&tv, v, g, g.Hkv, kKeys, 1, g.skv, true))
        return cudaErrorInvalidValue;
    Params p;
    p.g = g;
    p.q = (const __nv_bfloat16 *)q;
    p.dO = (const __nv_bfloat16 *)dO;
    p.lse = lse;
    p.delta = delta;
    p.offsets = offsets;
    p.rows = rows;
    p.units = units;
    p.hdr = hdr;
    p.partials = partials;
    p.dk = (__nv_bfloat16 *)dk;
    p.dv = (__nv_bfloat16 *)dv;
    p.err = err;
    p.wait_us = wait_test().wait_us;
    p.stall = wait_test().kernel == WAIT_TEST_DKDV;
    int grid = num_sms();
    if (grid > max_units)
        grid = max_units;
    if (grid < 1)
        grid = 1;
    // a programmatic dependent of the kernel before it (see the kernel's wait)
    auto go = [&](auto kernel, int threads) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        return launch_dependent(kernel, dim3(grid), dim3(threads), SMEM_BYTES, st, tq, tdo, tk, tv, p);
    };
    if (mode == LOAD_ROWS)
        return go(dkdv_tc_kernel<LOAD_ROWS>, dkdv_threads<LOAD_ROWS>());
    if (mode == LOAD_TILE)
        return go(dkdv_tc_kernel<LOAD_TILE>, dkdv_threads<LOAD_TILE>());
    return go(dkdv_tc_kernel<LOAD_CPASYNC>, dkdv_threads<LOAD_CPASYNC>());
}

}  // namespace nsa
