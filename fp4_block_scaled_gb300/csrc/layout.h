// layout.h -- packed expert layout shared by the packer and the kernels.
//
// An expert is three row-major matrices, each stored as "mma tiles" of 16
// rows.  In the gate/up section tile t holds gate rows 8t..8t+7 followed by up
// rows 8t..8t+7 (so one mma tile yields both SwiGLU inputs of 8 outputs); in
// the down section tile t holds down rows 16t..16t+15.  Along K a tile is cut
// into k-groups of 128 elements (4 scale blocks of 32) plus, when K % 128 == 64,
// one half group of 64 elements at the end.
//
// Codes of one full k-group (1024 bytes) are ordered [lane 0..31][half 0..1]
// [block 0..3][4 bytes]: lane (g = lane/4, c = lane%4) finds, for mma row
// g + 8*half, bytes 4c..4c+3 of each of the 4 blocks, i.e. exactly the E2M1
// pairs its mma.m16n8k16 A fragments need, in two 16-byte loads.  A half group
// (512 bytes) is [lane][half][block 0..1][4 bytes].  Scales of a full group
// (64 bytes) are [g 0..7][half][block 0..3], of a half group (32 bytes)
// [g][half][block 0..1].  Tiles are stored one after another, codes and scales
// in two separate arrays, so a tile (and any run of k-groups in it) is one
// contiguous span.  The packing is a pure permutation: sizes equal the
// published layout's.
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace moe {

struct MatLayout {
    int rows;      // matrix rows (mma rows)
    int k;         // reduction length (multiple of 64)
    int tiles;     // rows / 16
    int kg_full;   // k / 128
    int kg_half;   // 1 if k % 128 == 64
    __host__ __device__ size_t tile_code_bytes() const { return (size_t)16 * k / 2; }
    __host__ __device__ size_t tile_scale_bytes() const { return (size_t)16 * k / 32; }
};

__host__ __device__ inline MatLayout make_layout(int rows, int k)
{
    MatLayout m;
    m.rows = rows;
    m.k = k;
    m.tiles = rows / 16;
    m.kg_full = k / 128;
    m.kg_half = (k % 128) ? 1 : 0;
    return m;
}

struct ExpertLayout {
    MatLayout gu;   // 2*I rows (gate and up interleaved per 8), K = H
    MatLayout dn;   // H rows, K = I
    size_t gu_code_off, dn_code_off, code_bytes;
    size_t gu_scale_off, dn_scale_off, scale_bytes;
};

__host__ __device__ inline ExpertLayout make_expert_layout(int hidden, int inter)
{
    ExpertLayout L;
    L.gu = make_layout(2 * inter, hidden);
    L.dn = make_layout(hidden, inter);
    L.gu_code_off = 0;
    L.dn_code_off = (size_t)L.gu.tiles * L.gu.tile_code_bytes();
    L.code_bytes = L.dn_code_off + (size_t)L.dn.tiles * L.dn.tile_code_bytes();
    L.gu_scale_off = 0;
    L.dn_scale_off = (size_t)L.gu.tiles * L.gu.tile_scale_bytes();
    L.scale_bytes = L.dn_scale_off + (size_t)L.dn.tiles * L.dn.tile_scale_bytes();
    return L;
}

}  // namespace moe
