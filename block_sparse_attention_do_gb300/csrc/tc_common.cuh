// tc_common.cuh -- pieces shared by the tensor-core kernels: tensor-map
// construction on the host and the row <-> (token, head) mapping of a
// 128-row tile.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "launch.h"
#include "tc_ptx.cuh"

namespace nsa {

// Tile shape of every tensor-core kernel: 128 query rows (tokens x the G
// heads of one kv group), kv blocks of 64 keys, head dimension 128 split in
// two 64-element (128-byte) halves.
constexpr int kRows = 128;
constexpr int kKeys = 64;
constexpr int kHead = 128;
constexpr int kHalfBytes = kRows * 128;    // one 64-column half of a 128-row tile
constexpr int kTileBytes = 2 * kHalfBytes; // a 128 x 128 bf16 tile
constexpr int kKvHalfBytes = kKeys * 128;  // one half of a 64-key block
constexpr int kKvBytes = 2 * kKvHalfBytes;

// Tensor maps of one operand: `rows` maps a box of `box_tok` tokens x
// `box_heads` heads x 64 columns; the smem result is box_tok*box_heads rows
// of 128 bytes, 128B-swizzled, in (token-major for THD, head-major for BHTD)
// order.
bool make_tmap(CUtensorMap *map, const void *base, const Geo &g, int H, int box_tok, int box_heads);

// Row-group tile layout (gathered rows of the dK/dV kernel): the tile's
// rows go in groups of 8; group R/8 occupies 2048 bytes, its 64-column half h
// the 1024 bytes at h * 1024, row R at (R % 8) * 128 inside it, 128B-swizzled.
// Both halves of a group sit in one 2 KB span, so a TMA box covering a
// token's G heads (G % 8 == 0) and both halves lands as one contiguous run.
constexpr int kRgStride = 2048;
constexpr int kRgHalf = 1024;
__host__ __device__ inline int rg_off(int r, int half) { return (r >> 3) * kRgStride + half * kRgHalf + (r & 7) * 128; }

// Tensor map whose box is one token's G consecutive query heads (G % 8 == 0,
// H % 8 == 0), both 64-column halves, in the row-group layout above:
// box {64 columns, 8 heads, 2 halves, G/8 head octets, 1 token}.
// Coordinates: (0, 0, 0, octet, token) with octet = (b*H + head0)/8 (BHTD)
// or head0/8 (THD, token = packed row).
bool make_tmap_rows(CUtensorMap *map, const void *base, const Geo &g, int H, int G);

// the host launcher's view of the device: SM count (cached)
int num_sms();

// ---- query-tile kernels (forward, dQ): a tile is Tq consecutive tokens of
// one sequence times the G query heads of one kv head.
constexpr int MAX_BLOCKS = 2048;  // nbmax limit (union list and bitmap)
constexpr int MASK_WORDS = 4096;  // per-token block bitmaps: Tq * ceil(nbmax/32) words

__host__ __device__ inline int tile_tokens(int G) { return G >= kRows ? 1 : kRows / G; }

inline bool qtile_shape_ok(const Geo &g)
{
    return g.nbmax <= MAX_BLOCKS && tile_tokens(g.G) * ((g.nbmax + 31) / 32) <= MASK_WORDS;
}

// Rows of a tile are token-major (row = token * G + head) for THD and, when
// G % 8 == 0, for BHTD too (one TMA box of G heads per token, 1024-byte
// aligned); otherwise BHTD rows are head-major (one box {64, Tq, G}).
// Token-major rows let a whole warp skip a block none of its tokens chose.
__host__ __device__ inline bool qtile_token_major(const Geo &g) { return g.thd || (g.G % 8) == 0; }

// tile row -> (token within tile, head within group)
__device__ __forceinline__ void qtile_row(const Geo &g, int Tq, int r, int &tl, int &hh)
{
    if (qtile_token_major(g)) {
        tl = r / g.G;
        hh = r % g.G;
    } else {
        hh = r / Tq;
        tl = r % Tq;
    }
}

// Builds, with the 128 threads of warps 4-7 (named barrier 1), the ascending
// list of blocks selected by any of the tile's tokens and one bitmap per
// token.  Entries that are -1, out of range or in the future are skipped.
// Returns the list length.
__device__ __forceinline__ int qtile_union(const Geo &g, const int *idx, int b, int kvh, int t0, int nvalid,
                                           uint32_t *mask, uint32_t *ubits, int *list, int tid, int lane,
                                           int wq)
{
    const int words = (g.nbmax + 31) / 32;
    for (int i = tid; i < tile_tokens(g.G) * words; i += 128)
        mask[i] = 0;
    for (int i = tid; i < words; i += 128)
        ubits[i] = 0;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (g.dense) {
        const int jmin = key_lo(g, t0) / g.bs, jmax = (t0 + nvalid - 1) / g.bs;
        for (int j = jmin + tid; j <= jmax; j += 128)
            atomicOr(&ubits[j >> 5], 1u << (j & 31));
    } else {
        for (int i = tid; i < nvalid * g.S; i += 128) {
            const int tl = i / g.S, s = i % g.S;
            const int t = t0 + tl;
            const int j = idx_row(g, idx, b, kvh, t)[s];
            if (j >= 0 && j <= t / g.bs && j < g.nbmax) {
                atomicOr(&mask[tl * words + (j >> 5)], 1u << (j & 31));
                atomicOr(&ubits[j >> 5], 1u << (j & 31));
            }
        }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    __shared__ int n_out;
    if (wq == 0) {  // ordered compaction by one warp
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
            uint32_t bb = bits;
            while (bb) {
                const int bit = __ffs(bb) - 1;
                bb &= bb - 1;
                list[pos++] = (w0 + lane) * 32 + bit;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            n_out = base;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    return n_out;
}

// does the row's token select block j?  (valid rows only)
__device__ __forceinline__ bool qtile_selects(const Geo &g, const uint32_t *my_mask, int t, int j)
{
    return g.dense ? (j <= t / g.bs && j >= key_lo(g, t) / g.bs) : (((my_mask[j >> 5] >> (j & 31)) & 1u) != 0);
}

}  // namespace nsa
