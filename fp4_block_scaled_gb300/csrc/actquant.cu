// actquant.cu -- E4M3 activation quantizer with one ue8m0 scale per 128.
//
// One warp per (row, 128-element block); lane l holds elements 4l..4l+3.  The
// block maximum is exact (a max of bf16 values); the scale exponent k is the
// least integer with amax <= 448 * 2^k, read off amax's bits: with
// amax = m * 2^E, m in [1, 2), k = E - 8 if m <= 1.75 and E - 7 otherwise
// (448 = 1.75 * 2^8).  Codes are round-to-nearest-even conversions of
// x * 2^-k (an exact scaling) with saturation to +-448.  A block whose
// maximum is zero gets k = 0; a non-finite maximum gives the NaN scale byte 255
// and NaN codes.  The computation is per element and fixed, so it is
// bit-exact and identical from run to run.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

// x: [rows][n] bf16, codes [rows][n], scales [rows][nb]; optional row gather
// (src_row[r] selects the input row of output row r; -1 writes zeros).
__global__ void __launch_bounds__(256) k_act_quant(ActQuantArgs a)
{
    const int nb = (a.n + 127) / 128;
    const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    pdl_wait();
    if (wid < (long long)a.rows * nb) {
        const int r = (int)(wid / nb), b = (int)(wid % nb);
        const int src = a.src_row ? a.src_row[r] : r;
        const int c0 = b * 128 + lane * 4;
        const bool in = c0 < a.n;                 // n is a multiple of 32, so 4 | (n - c0)
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (in && src >= 0) {
            const uint2 u = *reinterpret_cast<const uint2*>(a.x + (size_t)src * a.n + c0);
            v[0] = __uint_as_float(u.x << 16);
            v[1] = __uint_as_float(u.x & 0xFFFF0000u);
            v[2] = __uint_as_float(u.y << 16);
            v[3] = __uint_as_float(u.y & 0xFFFF0000u);
        }
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
        // a NaN element makes the block maximum NaN
        bool nan = (v[0] != v[0]) || (v[1] != v[1]) || (v[2] != v[2]) || (v[3] != v[3]);
        nan = __any_sync(0xFFFFFFFFu, nan);
        amax = warp_max(amax);
        const int s = nan ? 255 : ue8m0_for_amax_bits(amax);
        if (in) {
            uint32_t out;
            if (s == 255) {
                out = 0x7F7F7F7Fu;
            } else {
                const float down = __uint_as_float((uint32_t)(254 - s) << 23);   // 2^-(s-127)
                out = (uint32_t)e4m3_rn_sat(v[0] * down) | ((uint32_t)e4m3_rn_sat(v[1] * down) << 8) |
                      ((uint32_t)e4m3_rn_sat(v[2] * down) << 16) |
                      ((uint32_t)e4m3_rn_sat(v[3] * down) << 24);
            }
            *reinterpret_cast<uint32_t*>(a.codes + (size_t)r * a.n + c0) = out;
        }
        if (lane == 0) a.scales[(size_t)r * nb + b] = (uint8_t)s;
    }
    pdl_trigger();
}

cudaError_t launch_act_quant(const ActQuantArgs& a0, cudaStream_t s, bool pdl)
{
    ActQuantArgs a = a0;
    const long long warps = (long long)a.rows * ((a.n + 127) / 128);
    if (warps == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[] = {&a};
    return cudaLaunchKernelExC(&cfg, (const void*)k_act_quant, args);
}

}  // namespace moe
