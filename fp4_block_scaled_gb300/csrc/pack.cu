// pack.cu -- load-time re-layout of one expert.
//
// Reorders the published layout (gate | up | down, row-major, two E2M1 codes
// per byte, one ue8m0 byte per 32 weights) into the tile / unit / MMA / core-
// matrix order of layout.h, so that the decode kernels stream contiguous units
// with bulk copies straight into the shared-memory layout the tensor-core MMA
// reads, and the scale atoms straight into the form tcgen05.cp moves to the
// tensor memory; each unit's atom follows its codes in the one blob.
#include "internal.h"

namespace moe {
namespace {

struct SectionMap {
    const uint8_t* codes;   // canonical section base (codes)
    const uint8_t* scales;  // canonical section base (scales)
    int gate_up;            // 1: tile = 64 gate rows then 64 up rows
    size_t up_code_off, up_scale_off;
};

__device__ inline void canon_row(const SectionMap& s, int tile, int r, int k, const uint8_t*& crow,
                                 const uint8_t*& srow)
{
    size_t row, cbase = 0, sbase = 0;
    if (s.gate_up) {
        row = (size_t)tile * 64 + (r & 63);
        if (r >= 64) {
            cbase = s.up_code_off;
            sbase = s.up_scale_off;
        }
    } else {
        row = (size_t)tile * kTileRows + r;
    }
    crow = s.codes + cbase + row * (k / 2);
    srow = s.scales + sbase + row * (k / 32);
}

// One thread per 16-byte chunk of codes (one row x one 32-element block).
__global__ void pack_codes_kernel(SectionMap s, MatLayout L, uint8_t* out)
{
    const size_t per_tile = ((size_t)L.kg_full * kUnitCodeBytes + (size_t)L.kg_half * kMmaCodeBytes) / 16;
    const size_t total = per_tile * L.tiles;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t qi = (size_t)blockIdx.x * blockDim.x + threadIdx.x; qi < total; qi += stride) {
        const int tile = (int)(qi / per_tile);
        const int q = (int)(qi % per_tile);
        const int kg = q / 512, r = q % 512;
        const int m = r / 256, r2 = r % 256;
        const int row = (r2 / 16) * 8 + (r2 % 8);
        const int c = (r2 % 16) / 8;
        const int block = kg * 4 + m * 2 + c;
        const uint8_t *crow, *srow;
        canon_row(s, tile, row, L.k, crow, srow);
        uint8_t* dst = out + (size_t)tile * L.tile_bytes() + (size_t)kg * kUnitBytes + (size_t)r * 16;
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(crow + (size_t)block * 16);
    }
}

// One thread per scale-atom byte; a unit's atom follows its codes.
__global__ void pack_scales_kernel(SectionMap s, MatLayout L, uint8_t* out)
{
    const size_t per_tile = (size_t)L.kgt() * kUnitSfBytes;
    const size_t total = per_tile * L.tiles;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t bi = (size_t)blockIdx.x * blockDim.x + threadIdx.x; bi < total; bi += stride) {
        const int tile = (int)(bi / per_tile);
        const int q = (int)(bi % per_tile);
        const int kg = q / kUnitSfBytes, b = q % kUnitSfBytes;
        const int row = b / 16 + 32 * ((b % 16) / 4);
        const int kb = b % 4;
        const bool half = kg == L.kg_full;
        uint8_t* dst = out + (size_t)tile * L.tile_bytes() + (size_t)kg * kUnitBytes +
                       (half ? kMmaCodeBytes : kUnitCodeBytes) + b;
        if (half && kb >= 2) {      // padding of a half unit
            *dst = 127;
            continue;
        }
        const uint8_t *crow, *srow;
        canon_row(s, tile, row, L.k, crow, srow);
        *dst = srow[kg * 4 + kb];
    }
}

int grid_for(size_t n)
{
    size_t g = (n + 255) / 256;
    return (int)(g > 4096 ? 4096 : (g ? g : 1));
}

}  // namespace

cudaError_t launch_pack_expert(const uint8_t* cc, const uint8_t* cs, uint8_t* packed, int H, int I,
                               cudaStream_t st)
{
    ExpertLayout E = make_expert_layout(H, I);
    const size_t gu_c = (size_t)I * H / 2, gu_s = (size_t)I * H / 32;
    SectionMap gu{cc, cs, 1, gu_c, gu_s};
    SectionMap dn{cc + 2 * gu_c, cs + 2 * gu_s, 0, 0, 0};
    size_t n;
    n = (size_t)E.gu.tiles * E.gu.kg_full * 512 + (size_t)E.gu.tiles * E.gu.kg_half * 256;
    pack_codes_kernel<<<grid_for(n), 256, 0, st>>>(gu, E.gu, packed + E.gu_off);
    n = (size_t)E.dn.tiles * E.dn.kg_full * 512 + (size_t)E.dn.tiles * E.dn.kg_half * 256;
    pack_codes_kernel<<<grid_for(n), 256, 0, st>>>(dn, E.dn, packed + E.dn_off);
    n = (size_t)E.gu.tiles * E.gu.kgt() * kUnitSfBytes;
    pack_scales_kernel<<<grid_for(n), 256, 0, st>>>(gu, E.gu, packed + E.gu_off);
    n = (size_t)E.dn.tiles * E.dn.kgt() * kUnitSfBytes;
    pack_scales_kernel<<<grid_for(n), 256, 0, st>>>(dn, E.dn, packed + E.dn_off);
    return cudaGetLastError();
}

}  // namespace moe
