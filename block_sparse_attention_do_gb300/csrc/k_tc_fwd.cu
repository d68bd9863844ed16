// k_tc_fwd.cu -- selection forward (O, LSE) on the tcgen05 tensor cores
// (bf16, D = 128, block_size = 64).
//
// Same query tile as the dQ kernel (Tq tokens x G heads = 128 rows) walking
// the ascending union of the tile's selected blocks.  For block j (step i):
//   S_i = Q K_j^T                                (M=128 rows, N=64 keys, K=128)
//   P_i = exp(S_i - m) on the row's attended keys, l += rowsum(P_i)
//   O  += P_i V_j   accumulated in TMEM          (M=128 rows, N=128 dims, K=64)
// m is a running reference that a row raises only when a block's maximum
// exceeds it by more than 2^8; then that row's O (in TMEM) and l are scaled
// by exp(m_old - m_new) before the block's P.V is issued.  Every term of O
// and l carries the same reference, so O / l at the end is exact; P stays
// below 2^8.  LSE = m + log l.  Warps whose rows all skip block j write
// zero P without computing it.
#include "tc_common.cuh"

namespace nsa {

namespace {

using namespace tc;

constexpr int NS = 4;  // K/V stages
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + kTileBytes;          // NS stages x (K | V)
constexpr int OFF_P = OFF_KV + NS * 2 * kKvBytes;     // 2 buffers of [128 rows][64 keys]
constexpr int OFF_MASK = OFF_P + 2 * kRows * 128;
constexpr int OFF_LIST = OFF_MASK + MASK_WORDS * 4;
constexpr int OFF_UBITS = OFF_LIST + MAX_BLOCKS * 4;
constexpr int OFF_BAR = OFF_UBITS + (MAX_BLOCKS / 32) * 4;
constexpr int KVF = 16, KVE = 16 + NS;  // barrier slots of the K/V ring
constexpr int NUM_BARS = 16 + 2 * NS;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;

enum {
    B_QFULL = 0, B_KVFULL0, B_KVFULL1, B_KVEMPTY0, B_KVEMPTY1, B_SFULL0, B_SFULL1, B_SFREE0, B_SFREE1,
    B_PFULL0, B_PFULL1, B_PVFULL0, B_PVFULL1, B_OFREE0, B_OFREE1, B_LIST
};

constexpr uint32_t TM_S = 0;    // buffer b at b*64
constexpr uint32_t TM_O = 128;  // 128 lanes (rows) x 128 columns (dims)
constexpr uint32_t TM_COLS = 256;
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
    uint64_t *done_bar = (uint64_t *)(sm + OFF_MISC + 48);
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
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars[B_SFULL0 + s], 1);
            mbar_init(&bars[B_SFREE0 + s], kRows);
            mbar_init(&bars[B_PFULL0 + s], kRows);
            mbar_init(&bars[B_PVFULL0 + s], 1);
        }
        mbar_init(&bars[B_LIST], kRows);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars[KVF + s], 1);
            mbar_init(&bars[KVE + s], 1);
        }
        mbar_init(done_bar, 1);
        fence_barrier_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    if (nrows < kRows) {
        for (int i = threadIdx.x; i < kTileBytes / 16; i += blockDim.x) {
            const int r = (i * 16 % kHalfBytes) / 128;
            if (r >= nrows)
                *(uint4 *)(sm + OFF_Q + i * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------- TMA
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(&bars[B_QFULL], 2 * nrows * 128);
            for (int h = 0; h < 2; ++h) {
                if (g.thd)
                    tma_load_3d(sm + OFF_Q + h * kHalfBytes, &tm_q, &bars[B_QFULL], h * 64, kvh * G, g.cu[b] + t0);
                else if (qtile_token_major(g))
                    for (int tl = 0; tl < Tq; ++tl)
                        tma_load_4d(sm + OFF_Q + h * kHalfBytes + tl * G * 128, &tm_q, &bars[B_QFULL], h * 64,
                                    t0 + tl, kvh * G, b);
                else
                    tma_load_4d(sm + OFF_Q + h * kHalfBytes, &tm_q, &bars[B_QFULL], h * 64, t0, kvh * G, b);
            }
            bool ok = mbar_wait(&bars[B_LIST], 0, abort_flag);
            const int U = ok ? *n_list : 0;
            int last = -1;
            for (int i = 0; i < U && ok; ++i) {
                const int s = i % NS;
                if (!mbar_wait(&bars[KVE + s], ((i / NS) & 1) ^ 1, abort_flag))
                    break;
                const int j = list[i];
                uint8_t *kd = sm + OFF_KV + s * 2 * kKvBytes;
                uint8_t *vd = kd + kKvBytes;
                mbar_arrive_expect_tx(&bars[KVF + s], 2 * kKvBytes);
                last = i;
                for (int h = 0; h < 2; ++h) {
                    if (g.thd) {
                        tma_load_3d(kd + h * kKvHalfBytes, &tm_k, &bars[KVF + s], h * 64, kvh,
                                    g.cu[b] + j * kKeys);
                        tma_load_3d(vd + h * kKvHalfBytes, &tm_v, &bars[KVF + s], h * 64, kvh,
                                    g.cu[b] + j * kKeys);
                    } else {
                        tma_load_4d(kd + h * kKvHalfBytes, &tm_k, &bars[KVF + s], h * 64, j * kKeys, kvh, b);
                        tma_load_4d(vd + h * kKvHalfBytes, &tm_v, &bars[KVF + s], h * 64, j * kKeys, kvh, b);
                    }
                }
            }
            volatile int never = 0;
            mbar_wait(&bars[B_QFULL], 0, &never);
            if (*abort_flag && last >= 0)
                mbar_wait(&bars[KVF + last % NS], (last / NS) & 1, &never);
        }
        __syncwarp();
    } else if (warp == 2) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, 64, false, false);
            const uint32_t idO = idesc_bf16(128, 128, false, true);
            const uint32_t q_s = smem_u32(sm + OFF_Q), kv_s = smem_u32(sm + OFF_KV), p_s = smem_u32(sm + OFF_P);
            bool ok = mbar_wait(&bars[B_LIST], 0, abort_flag) && mbar_wait(&bars[B_QFULL], 0, abort_flag);
            const int U = ok ? *n_list : 0;
            int si = 0, oi = 0;
            uint64_t t_last = globaltimer();
            while (ok && oi < U && !*abort_flag) {
                bool progressed = false;
                if (oi < si && mbar_try_wait(&bars[B_PFULL0 + (oi & 1)], (oi >> 1) & 1)) {
                    tc_fence_after();
                    const int s = oi & 1, ks = oi % NS;
                    const uint32_t v_s = kv_s + ks * 2 * kKvBytes + kKvBytes;
                    for (int kk = 0; kk < kKeys / 16; ++kk)
                        mma_bf16(tmem + TM_O, sdesc_sw128(p_s + s * kRows * 128 + kk * 32, 16, 1024),
                                 sdesc_sw128(v_s + kk * 2048, kKvHalfBytes, 1024), idO, (oi > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&bars[B_PVFULL0 + s]);
                    mma_commit(&bars[KVE + ks]);
                    ++oi;
                    progressed = true;
                }
                if (si < U && si < oi + 2 && mbar_try_wait(&bars[KVF + si % NS], (si / NS) & 1) &&
                    mbar_try_wait(&bars[B_SFREE0 + (si & 1)], ((si >> 1) & 1) ^ 1)) {
                    tc_fence_after();
                    const int s = si & 1;
                    const uint32_t k_s = kv_s + (si % NS) * 2 * kKvBytes;
                    for (int kk = 0; kk < kHead / 16; ++kk) {
                        const uint32_t ao = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                        const uint32_t bo = (kk >> 2) * kKvHalfBytes + (kk & 3) * 32;
                        mma_bf16(tmem + TM_S + s * 64, sdesc_sw128(q_s + ao, 16, 1024),
                                 sdesc_sw128(k_s + bo, 16, 1024), idS, kk > 0);
                    }
                    mma_commit(&bars[B_SFULL0 + s]);
                    ++si;
                    progressed = true;
                }
                if (progressed)
                    t_last = globaltimer();
                else if (globaltimer() - t_last > kWaitLimitNs)
                    *abort_flag = 1;
            }
            mma_commit(done_bar);
            volatile int never = 0;
            mbar_wait(done_bar, 0, &never);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------- union, softmax, epilogue
        const int tid = threadIdx.x - 128;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const int Un = qtile_union(g, p.idx, b, kvh, t0, nvalid, mask, ubits, list, tid, lane, wq);
        if (tid == 0)
            *n_list = Un;
        mbar_arrive(&bars[B_LIST]);
        const int U = Un;

        int tl, hh;
        qtile_row(g, Tq, r, tl, hh);
        const bool rvalid = r < nrows && tl < nvalid;
        const int t = t0 + tl;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const uint32_t p_row = smem_u32(sm + OFF_P) + r * 128;
        const uint32_t *my_mask = mask + (rvalid ? tl : 0) * words;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < U; ++i) {
            const int s = i & 1;
            if (!mbar_wait_warp(&bars[B_SFULL0 + s], (i >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[64];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld16(lane_base + TM_S + s * 64 + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[c * 16]));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&bars[B_SFREE0 + s]);
            const int j = list[i];
            const bool sel = rvalid && qtile_selects(g, my_mask, t, j);
            const int lim = sel ? t - j * kKeys : -1;
            uint32_t pk[32];
            if (__any_sync(0xffffffffu, sel)) {
                float mb = -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const float x = __uint_as_float(sv[c]) * g.scale_l2;
                    sv[c] = __float_as_uint(x);
                    if (c <= lim)
                        mb = fmaxf(mb, x);
                }
                const bool raise = mb > m + kRescaleLog2;
                if (__any_sync(0xffffffffu, raise)) {
                    // O must hold every earlier block before it is rescaled
                    if (i > 0 && !mbar_wait_warp(&bars[B_PVFULL0 + ((i - 1) & 1)], ((i - 1) >> 1) & 1, abort_flag)) {
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
#pragma unroll
                for (int c = 0; c < 64; c += 2) {
                    const float p0 = (c <= lim) ? ex2(__uint_as_float(sv[c]) - m) : 0.f;
                    const float p1 = (c + 1 <= lim) ? ex2(__uint_as_float(sv[c + 1]) - m) : 0.f;
                    rs += p0 + p1;
                    pk[c >> 1] = pack_bf16(p0, p1);
                }
                l += rs;
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    pk[c] = 0u;
            }
            // P buffer s was last read by the P.V of block i - 2
            if (i >= 2 && !mbar_wait_warp(&bars[B_PVFULL0 + s], ((i >> 1) & 1) ^ 1, abort_flag)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(p_row + s * kRows * 128 + ((c ^ (r & 7)) << 4), pk[4 * c], pk[4 * c + 1],
                             pk[4 * c + 2], pk[4 * c + 3]);
            fence_async_smem();
            tc_fence_before();
            mbar_arrive(&bars[B_PFULL0 + s]);
        }
        float o[128];
        if (ok && U > 0) {
            const int sp = (U - 1) & 1;
            if (!mbar_wait_warp(&bars[B_PVFULL0 + sp], ((U - 1) >> 1) & 1, abort_flag)) {
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
    const int box_tok = (!g.thd && qtile_token_major(g)) ? 1 : Tq;
    if (!make_tmap(&tq, q, g, g.Hq, box_tok, g.G) || !make_tmap(&tk, k, g, g.Hkv, kKeys, 1) ||
        !make_tmap(&tv, v, g, g.Hkv, kKeys, 1))
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
