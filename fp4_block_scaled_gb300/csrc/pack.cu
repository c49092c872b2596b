// pack.cu -- load-time re-layout of one expert (a pure byte permutation).
//
// Reorders the published layout (gate | up | down, row-major, two E2M1 codes
// per byte, one ue8m0 byte per 32 weights) into the tile-group / k-group /
// tile / lane order of layout.h, so that the decode kernels stream contiguous
// units with bulk copies and find every mma fragment already in place.
#include "internal.h"

namespace moe {
namespace {

// Canonical row of mma row m in tile t of a section.
struct SectionMap {
    const uint8_t* codes;   // canonical section base (codes)
    const uint8_t* scales;  // canonical section base (scales)
    int interleave;         // 1: gate/up interleave per 8 rows, 0: plain
    size_t up_code_off, up_scale_off;
};

__device__ inline void canon_row(const SectionMap& s, int tile, int m, int k, const uint8_t*& crow,
                                 const uint8_t*& srow)
{
    size_t r;
    size_t cbase = 0, sbase = 0;
    if (s.interleave) {
        r = (size_t)tile * 8 + (m & 7);
        if (m >= 8) {
            cbase = s.up_code_off;
            sbase = s.up_scale_off;
        }
    } else {
        r = (size_t)tile * 16 + m;
    }
    crow = s.codes + cbase + r * (k / 2);
    srow = s.scales + sbase + r * (k / 32);
}

// One thread per packed 4-byte code word.
__global__ void pack_codes_kernel(SectionMap s, MatLayout L, uint8_t* out)
{
    size_t words_per_group = L.group_code_bytes() / 4;
    size_t total = words_per_group * L.groups;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t wi = (size_t)blockIdx.x * blockDim.x + threadIdx.x; wi < total; wi += stride) {
        int grp = (int)(wi / words_per_group);
        int wg = (int)(wi % words_per_group);
        int kg = wg / 1024;
        int q, half, lane, j, block;
        if (kg < L.kg_full) {          // [tile q][half][lane][block 0..3][4 B]
            int r = wg % 1024;
            q = r / 256;
            r %= 256;
            half = r / 128;
            lane = (r % 128) / 4;
            j = r % 4;
            block = kg * 4 + j;
        } else {                       // half k-group: [tile q][half][lane][block 0..1][4 B]
            int r = wg - L.kg_full * 1024;
            q = r / 128;
            r %= 128;
            half = r / 64;
            lane = (r % 64) / 2;
            j = r % 2;
            block = L.kg_full * 4 + j;
        }
        int g = lane >> 2, c = lane & 3;
        const uint8_t *crow, *srow;
        canon_row(s, grp * kTilesPerGroup + q, g + 8 * half, L.k, crow, srow);
        uint32_t v = *reinterpret_cast<const uint32_t*>(crow + block * 16 + 4 * c);
        reinterpret_cast<uint32_t*>(out)[wi] = v;
    }
}

// One thread per packed scale byte.
__global__ void pack_scales_kernel(SectionMap s, MatLayout L, uint8_t* out)
{
    size_t per_group = L.group_scale_bytes();
    size_t total = per_group * L.groups;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t bi = (size_t)blockIdx.x * blockDim.x + threadIdx.x; bi < total; bi += stride) {
        int grp = (int)(bi / per_group);
        int sg = (int)(bi % per_group);
        int kg = sg / 256;
        int q, g, half, block;
        if (kg < L.kg_full) {          // [tile q][g][half][block 0..3]
            int r = sg % 256;
            q = r / 64;
            r %= 64;
            g = r / 8;
            half = (r / 4) & 1;
            block = kg * 4 + (r & 3);
        } else {                       // half k-group: [tile q][g][half][block 0..1]
            int r = sg - L.kg_full * 256;
            q = r / 32;
            r %= 32;
            g = r / 4;
            half = (r / 2) & 1;
            block = L.kg_full * 4 + (r & 1);
        }
        const uint8_t *crow, *srow;
        canon_row(s, grp * kTilesPerGroup + q, g + 8 * half, L.k, crow, srow);
        out[bi] = srow[block];
    }
}

int grid_for(size_t n)
{
    size_t g = (n + 255) / 256;
    return (int)(g > 4096 ? 4096 : (g ? g : 1));
}

}  // namespace

cudaError_t launch_pack_expert(const uint8_t* cc, const uint8_t* cs, uint8_t* pc, uint8_t* ps,
                               int H, int I, cudaStream_t st)
{
    ExpertLayout E = make_expert_layout(H, I);
    size_t gu_c = (size_t)I * H / 2, gu_s = (size_t)I * H / 32;
    SectionMap gu{cc, cs, 1, gu_c, gu_s};
    SectionMap dn{cc + 2 * gu_c, cs + 2 * gu_s, 0, 0, 0};
    size_t n;
    n = E.gu.groups * E.gu.group_code_bytes() / 4;
    pack_codes_kernel<<<grid_for(n), 256, 0, st>>>(gu, E.gu, pc + E.gu_code_off);
    n = E.dn.groups * E.dn.group_code_bytes() / 4;
    pack_codes_kernel<<<grid_for(n), 256, 0, st>>>(dn, E.dn, pc + E.dn_code_off);
    n = E.gu.groups * E.gu.group_scale_bytes();
    pack_scales_kernel<<<grid_for(n), 256, 0, st>>>(gu, E.gu, ps + E.gu_scale_off);
    n = E.dn.groups * E.dn.group_scale_bytes();
    pack_scales_kernel<<<grid_for(n), 256, 0, st>>>(dn, E.dn, ps + E.dn_scale_off);
    return cudaGetLastError();
}

}  // namespace moe
