// tc_common.cuh -- pieces shared by the tensor-core kernels: tensor-map
// construction on the host and the row <-> (token, head) mapping of a
// 128-row tile.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <utility>

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
// keys = true maps a key-side tensor (k, v): the key length / key count.
bool make_tmap(CUtensorMap *map, const void *base, const Geo &g, int H, int box_tok, int box_heads, const Strides &s,
               bool keys = false);

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
// Coordinates: (0, 0, 0, octet, token) with octet = (b*H + head0)/8 (BHTD,
// batch and head folded into one index: needs s.b = H * s.h or B = 1), or
// octet = head0/8 and token = b*T + t (BHTD with bt set: batch and token
// folded, needs s.b = T * s.t) or the packed row (THD).
bool make_tmap_rows(CUtensorMap *map, const void *base, const Geo &g, int H, int G, const Strides &s, int bt);

// A plain 3-D bf16 tensor map, 128B-swizzled (dims and box innermost first,
// byte strides of dims 1 and 2); rows past an end read as zeros.
bool make_tmap_3d(CUtensorMap *map, const void *base, const uint64_t dims[3], const uint64_t strides_bytes[2],
                  const uint32_t box[3]);

// Whether the row-gather map of a BHTD tensor with these strides can be
// built, and in which form (bt: batch folded into the token index).
inline bool rows_map_form(const Geo &g, int H, const Strides &s, int &bt)
{
    bt = 0;
    if (g.thd || g.B == 1 || s.b == (int64_t)H * s.h)
        return true;
    if (s.b == (int64_t)g.T * s.t) {
        bt = 1;
        return true;
    }
    return false;
}

// the host launcher's view of the device: SM count (cached)
int num_sms();

// Launches kernel as a programmatic dependent of the previous kernel on st:
// it may start before that kernel completes (once that kernel's CTAs have
// executed griddepcontrol.launch_dependents and resources free up), so it
// must not read what that kernel writes.  Later launches on st still wait
// for both.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

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

// ---- persistent query-tile kernels: tiles are taken from a launch-wide
// counter, heaviest (latest tokens) first, and one warp per CTA puts each
// tile's block union (copied from the table qtile_union_kernel built, or
// built in place) a tile ahead of its use into one of (up to) two buffers.

// A union buffer: UH_INTS header ints (the tile's coordinates and the list
// length; a negative length ends the walk), the per-token block bitmaps, the
// union bitmap and the ascending list.  The tile's token tl is T0 + tl, or
// with UH_GROUPED set T0 + byte tl of the words from UH_TOK (a tile of at
// most 16 tokens grouped from a window that starts at T0; see
// qtile_group_kernel).
enum { UH_B = 0, UH_KVH, UH_T0, UH_NVALID, UH_COUNT, UH_GROUPED, UH_TOK = 8, UH_INTS = 12 };
constexpr int kGroupMaxTq = 16;  // tokens a grouped tile names (4 words of bytes)

// the tile's token tl (sequence-local)
__device__ __forceinline__ int qtile_token(const volatile int *hdr, int tl)
{
    return hdr[UH_T0] + (hdr[UH_GROUPED] ? (hdr[UH_TOK + (tl >> 2)] >> ((tl & 3) * 8)) & 0xff : tl);
}
struct UnionBuf {
    int mask_words, ubits_words, list_ints, bytes;
};
__host__ __device__ inline UnionBuf union_buf(const Geo &g)
{
    UnionBuf u;
    const int words = (g.nbmax + 31) / 32;
    u.mask_words = tile_tokens(g.G) * words;
    u.ubits_words = (words + 3) & ~3;
    u.list_ints = (g.nbmax + 3) & ~3;
    u.bytes = ((UH_INTS + u.mask_words + u.ubits_words + u.list_ints) * 4 + 127) & ~127;
    return u;
}
__device__ __forceinline__ uint32_t *union_mask(int *buf) { return (uint32_t *)(buf + UH_INTS); }
__device__ __forceinline__ int *union_list(int *buf, const UnionBuf &u)
{
    return buf + UH_INTS + u.mask_words + u.ubits_words;
}

// The next tile for the calling warp's CTA from the launch-wide counter
// *next (zero at launch): tile L covers (b, kv head) = L % (B*Hkv) and is the
// (L / (B*Hkv))-th from the end of the sequence, so the heaviest tiles (the
// latest tokens) go first and a CTA that finishes early takes more.  Tiles
// past a sequence's end are skipped.  False once the counter passes the tile
// count.  Called by all lanes of one warp.
// Claims a tile index from the launch-wide counter *next: lane 0's value,
// 0 on the other lanes.  A claim issued early keeps the counter's round trip
// off the path; qtile_take turns it into a tile.
__device__ __forceinline__ int qtile_claim(int *next, int lane) { return lane == 0 ? atomicAdd(next, 1) : 0; }

// Tile L's coordinates: (b, kv head) = L % (B*Hkv), tokens t0 .. t0+nvalid-1
// counted from the sequence's end; false for a tile past a shorter
// sequence's end (nothing to do).
__device__ __forceinline__ bool qtile_of(const Geo &g, int L, int &b, int &kvh, int &t0, int &nvalid)
{
    const int Tq = tile_tokens(g.G), per_seq = (g.T + Tq - 1) / Tq, nbg = g.B * g.Hkv;
    const int bg = L % nbg, tile = per_seq - 1 - L / nbg;
    b = bg / g.Hkv;
    kvh = bg % g.Hkv;
    t0 = tile * Tq;
    const int len = seq_len(g, b);
    nvalid = t0 < len ? min(Tq, len - t0) : 0;
    return nvalid > 0;
}

// The tile of a claim (lane 0's `claimed`), claiming again past tiles that
// lie beyond a shorter sequence's end; false once the tiles are used up.
// *Lout (if given) receives the tile's index.
__device__ __forceinline__ bool qtile_take(const Geo &g, int ntiles, int *next, int lane, int claimed, int &b,
                                           int &kvh, int &t0, int &nvalid, int *Lout = nullptr)
{
    for (;;) {
        const int L = __shfl_sync(0xffffffffu, claimed, 0);
        if (L >= ntiles)
            return false;
        if (qtile_of(g, L, b, kvh, t0, nvalid)) {
            if (Lout)
                *Lout = L;
            return true;
        }
        claimed = qtile_claim(next, lane);
    }
}

__device__ __forceinline__ bool qtile_next(const Geo &g, int ntiles, int *next, int lane, int &b, int &kvh,
                                           int &t0, int &nvalid)
{
    return qtile_take(g, ntiles, next, lane, qtile_claim(next, lane), b, kvh, t0, nvalid);
}

// One warp fills buf for a tile: each token's block bitmap, the ascending
// list of blocks selected by any of its tokens, then the header (written
// last, with the list length).  Entries that are -1, out of range or in the
// future are skipped.  The caller orders the writes before its release.
__device__ __forceinline__ void qtile_union_warp(const Geo &g, const int *idx, const UnionBuf &u, int *buf, int b,
                                                 int kvh, int t0, int nvalid, int lane)
{
    const int words = (g.nbmax + 31) / 32;
    uint32_t *mask = union_mask(buf), *ubits = mask + u.mask_words;
    int *list = union_list(buf, u);
    if (!g.dense)
        for (int x = lane; x < u.mask_words; x += 32)
            mask[x] = 0u;
    for (int x = lane; x < words; x += 32)
        ubits[x] = 0u;
    __syncwarp();
    if (g.dense) {
        // from the first row's window edge to the last row's diagonal
        const int hi = min(kdiag(g, b, t0 + nvalid - 1), seq_len_k(g, b) - 1);
        const int jmin = key_lo(g, kdiag(g, b, t0)) / g.bs, jmax = hi >= 0 ? hi / g.bs : -1;
        for (int j = jmin + lane; j <= jmax; j += 32)
            atomicOr(&ubits[j >> 5], 1u << (j & 31));
    } else {
        // four index entries per lane read at a time, all loads in flight
        // together, then recorded
        const int n = nvalid * g.S;
        for (int x0 = 0; x0 < n; x0 += 128) {
            int jv[4];
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                const int x = x0 + u4 * 32 + lane;
                jv[u4] = x < n ? idx_row(g, idx, b, kvh, t0 + x / g.S)[x % g.S] : -1;
            }
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                const int x = x0 + u4 * 32 + lane;
                const int tl = x / g.S, t = t0 + tl, j = jv[u4];
                if (x < n && j >= 0 && j <= t / g.bs && j < g.nbmax) {
                    atomicOr(&mask[tl * words + (j >> 5)], 1u << (j & 31));
                    atomicOr(&ubits[j >> 5], 1u << (j & 31));
                }
            }
        }
    }
    __syncwarp();
    // ordered compaction
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
    if (lane == 0) {
        buf[UH_B] = b;
        buf[UH_KVH] = kvh;
        buf[UH_T0] = t0;
        buf[UH_NVALID] = nvalid;
        buf[UH_GROUPED] = 0;
        buf[UH_COUNT] = base;
    }
    __syncwarp();
}

// does the row's token select block j?  (valid rows only; klo .. khi: the
// row's attended key range, which decides for the dense entries)
__device__ __forceinline__ bool qtile_selects(const Geo &g, const uint32_t *my_mask, int klo, int khi, int j)
{
    return g.dense ? (klo <= khi && j <= khi / g.bs && j >= klo / g.bs) : (((my_mask[j >> 5] >> (j & 31)) & 1u) != 0);
}

}  // namespace nsa
