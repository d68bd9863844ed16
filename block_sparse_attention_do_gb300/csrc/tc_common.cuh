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

// the host launcher's view of the device: SM count (cached)
int num_sms();

}  // namespace nsa
