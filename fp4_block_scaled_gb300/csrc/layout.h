// layout.h -- packed expert layout shared by the packer and the kernels.
//
// Each expert matrix is cut into tiles of 128 rows, the M of one tensor-core
// MMA: a gate/up tile t holds gate rows 64t..64t+63 followed by up rows
// 64t..64t+63 (so one accumulator holds both SwiGLU inputs of 64 outputs); a
// down tile t holds down rows 128t..128t+127.  Along K a tile is cut into
// units of 128 elements (two MMAs of K = 64, four ue8m0 blocks of 32), plus one
// half unit of 64 when K % 128 == 64.
//
// A unit is its codes followed by its scale atom, so that one bulk copy moves
// any run of units, codes and scales together:
//   codes (8 KB; 4 KB for a half unit), stored as the MMA reads them from
//   shared memory: per MMA m (4 KB), 16 row groups of 8 rows, each holding two
//   "core matrices" of 8 rows x 16 bytes (the two 32-element blocks of that
//   MMA's K range), i.e. offset = m*4096 + (row/8)*256 + c*128 + (row%8)*16
//   for block 2m+c of the unit;
//   then one 512-byte scale atom: byte (row%32)*16 + (row/32)*4 + kb holds the
//   scale of block kb of row `row` -- the order in which tcgen05.cp moves 32
//   lanes x 128 bits into the tensor memory for 128 rows.  A half unit's atom
//   leaves bytes kb = 2, 3 at 127 (scale 1, never read).
// Tiles are stored one after another, gate/up tiles first, in one blob per
// expert.  The blob holds every code and scale byte of the published layout
// once (a permutation), plus 256 padding bytes per half-unit atom.
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kTileRows = 128;
constexpr int kUnitCodeBytes = 8192;   // 128 rows x 128 E2M1 codes
constexpr int kMmaCodeBytes = 4096;    // one MMA (K = 64)
constexpr int kUnitSfBytes = 512;      // scale atom of a unit
constexpr int kUnitBytes = kUnitCodeBytes + kUnitSfBytes;       // a full unit in the blob
constexpr int kHalfUnitBytes = kMmaCodeBytes + kUnitSfBytes;    // a half unit in the blob

struct MatLayout {
    int rows;      // matrix rows
    int k;         // reduction length
    int tiles;     // rows / 128
    int kg_full;   // k / 128
    int kg_half;   // 1 if k % 128 == 64
    __host__ __device__ int kgt() const { return kg_full + kg_half; }
    __host__ __device__ size_t tile_bytes() const
    {
        return (size_t)kg_full * kUnitBytes + (size_t)kg_half * kHalfUnitBytes;
    }
};

__host__ __device__ inline MatLayout make_layout(int rows, int k)
{
    MatLayout m;
    m.rows = rows;
    m.k = k;
    m.tiles = rows / kTileRows;
    m.kg_full = k / 128;
    m.kg_half = (k % 128) ? 1 : 0;
    return m;
}

struct ExpertLayout {
    MatLayout gu;   // 2*I rows (gate / up halves per tile), K = H
    MatLayout dn;   // H rows, K = I
    size_t gu_off, dn_off, bytes;
};

__host__ __device__ inline ExpertLayout make_expert_layout(int hidden, int inter)
{
    ExpertLayout L;
    L.gu = make_layout(2 * inter, hidden);
    L.dn = make_layout(hidden, inter);
    L.gu_off = 0;
    L.dn_off = (size_t)L.gu.tiles * L.gu.tile_bytes();
    L.bytes = L.dn_off + (size_t)L.dn.tiles * L.dn.tile_bytes();
    return L;
}

// Activation operand ("pieces"): a vector v of length K is carried as 16
// E2M1 vectors p_0..p_15 with one ue8m0 scale per (piece, 32-block), so that
// v = sum_p p_p * scale_p; p_0 is v rounded to E2M1 under its block scale and
// each next piece encodes what is left.  As the MMA's B operand the pieces are
// its N = 16 rows: per MMA m, 512 bytes laid out like the A codes (2 row groups
// x 2 core matrices x 8 rows x 16 bytes), and a 512-byte scale atom per unit
// (rows 0..15 used).
constexpr int kPieces = 16;
constexpr int kBRows = 16;
constexpr int kMmaBBytes = 512;
constexpr int kUnitBBytes = 1024;

__host__ __device__ inline size_t act_bytes(int k)       // B codes of one vector
{
    return (size_t)(k / 128) * kUnitBBytes + (size_t)((k % 128) ? kMmaBBytes : 0);
}
__host__ __device__ inline size_t act_sf_bytes(int k)    // B scale atoms of one vector
{
    return (size_t)((k + 127) / 128) * kUnitSfBytes;
}

}  // namespace moe
