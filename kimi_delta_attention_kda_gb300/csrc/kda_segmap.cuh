// kda_segmap.cuh -- layouts of the segment maps of the segmented scan.
#pragma once

#include <cstdint>

namespace kda {

// Segment maps of the segmented scan in the warp MMA's fragment order, so the
// segment chain loads its operands with one coalesced 16- or 8-byte load per
// lane and no shared-memory staging.  Both are BF16, 32 KB per (segment,
// head).
//  - The transition F (S -> S F, F 128 x 128 keys x keys) as the A operand
//    F^T of m16n8k16 (m = column of F, k = row of F): 64 tiles of 16 x 16,
//    tile (mt, kt) at byte 512 (8 mt + kt), lane L's four registers (rows
//    g, g + 8 and columns 2 t, 2 t + 8 of the tile, g = L / 4, t = L % 4) at
//    16 L within it.
//  - The zero-start state Z (128 value rows x 128 keys) as the C operand Z^T
//    (m = key, n = value row): 128 tiles of 16 x 8, tile (nt, mt) at byte
//    256 (8 nt + mt), lane L's two BF16 pairs (rows g and g + 8, columns
//    2 t, 2 t + 1) at 8 L within it.
// A 16 x 16 A tile is two 16 x 8 C tiles side by side, so the fragment of F^T
// for k tile kt is the pair of C fragments of value tiles 2 kt and 2 kt + 1.
__host__ __device__ __forceinline__ uint32_t fmap_frag_off(uint32_t mt, uint32_t kt, uint32_t lane) {
    return ((8 * mt + kt) * 32 + lane) * 16;
}
__host__ __device__ __forceinline__ uint32_t zmap_frag_off(uint32_t nt, uint32_t mt, uint32_t lane) {
    return ((8 * nt + mt) * 32 + lane) * 8;
}

}  // namespace kda
