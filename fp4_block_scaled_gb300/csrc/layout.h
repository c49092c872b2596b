// layout.h -- packed expert layout shared by the packer and the kernels.
//
// An expert is three row-major matrices, each cut into "mma tiles" of 16
// rows.  In the gate/up section tile t holds gate rows 8t..8t+7 followed by up
// rows 8t..8t+7 (so one mma tile yields both SwiGLU inputs of 8 outputs); in
// the down section tile t holds down rows 16t..16t+15.  Along K a tile is cut
// into k-groups of 128 elements (4 scale blocks of 32) plus, when K % 128 == 64,
// one half group of 64 elements at the end.
//
// Four consecutive tiles form a tile group (64 rows: 32 SwiGLU outputs in the
// gate/up section, 64 output rows in the down section).  A tile group is
// stored k-group by k-group, and within a k-group tile by tile, so one
// "unit" = (tile group, k-group) is a contiguous 4 KB span of codes (2 KB for
// the half group) and 256 B of scales (128 B), and consecutive units of a tile
// group are adjacent.  The kernels stream units with bulk copies.
//
// Codes of one tile's full k-group (1024 bytes) are ordered [half 0..1]
// [lane 0..31][block 0..3][4 bytes]: lane (g = lane/4, c = lane%4) finds, for
// mma row g + 8*half, bytes 4c..4c+3 of each of the 4 blocks -- exactly the
// E2M1 pairs its mma.m16n8k16 A fragments need -- in two conflict-free 16-byte
// shared-memory reads.  A half group (512 bytes) is [half][lane][block 0..1]
// [4 bytes].  Scales of a tile's full group (64 bytes) are [g 0..7][half]
// [block 0..3], of a half group (32 bytes) [g][half][block 0..1].  The packing
// is a pure permutation: sizes equal the published layout's.
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kTilesPerGroup = 4;
constexpr int kUnitCodeBytes = 4096;   // full k-group of a tile group
constexpr int kUnitScaleBytes = 256;

struct MatLayout {
    int rows;      // matrix rows (mma rows)
    int k;         // reduction length (multiple of 64)
    int tiles;     // rows / 16
    int groups;    // tiles / 4
    int kg_full;   // k / 128
    int kg_half;   // 1 if k % 128 == 64
    __host__ __device__ int kgt() const { return kg_full + kg_half; }
    __host__ __device__ size_t tile_code_bytes() const { return (size_t)16 * k / 2; }
    __host__ __device__ size_t tile_scale_bytes() const { return (size_t)16 * k / 32; }
    __host__ __device__ size_t group_code_bytes() const { return kTilesPerGroup * tile_code_bytes(); }
    __host__ __device__ size_t group_scale_bytes() const { return kTilesPerGroup * tile_scale_bytes(); }
    // offset of unit (tile group, k-group) inside the section
    __host__ __device__ size_t unit_code_off(int grp, int kg) const
    {
        return (size_t)grp * group_code_bytes() + (size_t)kg * kUnitCodeBytes;
    }
    __host__ __device__ size_t unit_scale_off(int grp, int kg) const
    {
        return (size_t)grp * group_scale_bytes() + (size_t)kg * kUnitScaleBytes;
    }
};

__host__ __device__ inline MatLayout make_layout(int rows, int k)
{
    MatLayout m;
    m.rows = rows;
    m.k = k;
    m.tiles = rows / 16;
    m.groups = m.tiles / kTilesPerGroup;
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
