// gemv.cu -- batch-1 / small-batch path of one routed FP4 MoE layer.
//
// Three launches per layer, chained with programmatic dependent launch:
//   k_prep     x (bf16, or the fp32 residual through a fused RMSNorm) -> f16
//              with one power-of-two scale per 32 elements (exact for bf16).
//   k_gate_up  per (slot, block of 32 outputs, K chunk): stream the packed
//              gate/up tiles, decode E2M1 pairs to f16 in registers, multiply
//              on the tensor cores (mma.m16n8k16, fp32 accumulate) one 32-weight
//              block at a time and apply the ue8m0 scale of each (row, block);
//              the last K chunk to finish a block sums the chunks in fixed
//              order, applies SwiGLU and the routing weight, and stores h as
//              f16 hi + lo words with a per-32 scale (about 22 bits).
//   k_down     per (token, 16 output rows, slot): the same stream over the down
//              tiles against h; the last slot to finish sums the k slot
//              partials in fixed order into y (or adds them to the residual).
// Every sum has a fixed order, so results are bitwise reproducible.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kWarps = 4;   // warps per CTA in both GEMV kernels

// -------------------------------------------------------------- k_prep

__global__ void __launch_bounds__(256) k_prep(GemvArgs a)
{
    const int t = blockIdx.x;
    const int H = a.H;
    __shared__ float s_red[8];
    __shared__ float s_inv;

    float inv = 1.0f;
    if (a.x_resid) {
        // RMSNorm with unit weight: sum of squares in a fixed tree order
        pdl_wait();
        const float* xr = a.x_resid + (size_t)t * H;
        float ss = 0.0f;
        for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.0f;
            for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += s_red[w];
            s_inv = sqrtf(tot / (float)H + a.eps);
        }
        __syncthreads();
        inv = s_inv;
    } else {
        pdl_wait();
    }
    pdl_trigger();

    // one thread per 32-element block
    for (int b = threadIdx.x; b < H / 32; b += blockDim.x) {
        float v[32];
        if (a.x_resid) {
            const float4* src = reinterpret_cast<const float4*>(a.x_resid + (size_t)t * H + b * 32);
#pragma unroll
            for (int q = 0; q < 8; q++) {
                float4 f = src[q];
                v[4 * q + 0] = f.x;
                v[4 * q + 1] = f.y;
                v[4 * q + 2] = f.z;
                v[4 * q + 3] = f.w;
            }
#pragma unroll
            for (int i = 0; i < 32; i++)  // the MoE input is the bf16 rounding of the norm
                v[i] = __bfloat162float(__float2bfloat16_rn(v[i] / inv));
        } else {
            const uint4* src = reinterpret_cast<const uint4*>(a.x_bf16 + (size_t)t * H + b * 32);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                uint4 u = src[q];
                uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    v[8 * q + 2 * r] = __uint_as_float(w4[r] << 16);
                    v[8 * q + 2 * r + 1] = __uint_as_float(w4[r] & 0xFFFF0000u);
                }
            }
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; i++) amax = fmaxf(amax, fabsf(v[i]));
        int e = f16_block_exponent(amax);
        float down = exp2i(-e);
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 16; i++) {
            __half2 hv = __floats2half2_rn(v[2 * i] * down, v[2 * i + 1] * down);
            packed[i] = *reinterpret_cast<uint32_t*>(&hv);
        }
        uint4* dst = reinterpret_cast<uint4*>(a.xh + (size_t)t * H + b * 32);
#pragma unroll
        for (int q = 0; q < 4; q++)
            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
        a.xs[(size_t)t * a.xs_stride + b] = exp2i(e);
    }
}

// One 32-weight block of a 16-row mma tile against one 8-column B fragment.
// w0 / w1: bytes 4c..4c+3 of the block for rows g and g+8; bx: f16 B values
// k-ordered for this lane (zero where the column is unused).
__device__ __forceinline__ void block_mma(float (&d)[4], uint32_t w0, uint32_t w1, uint4 bx)
{
    uint32_t p0[4], p1[4];
    e2m1x8_to_f16x2(w0, p0);
    e2m1x8_to_f16x2(w1, p1);
    d[0] = d[1] = d[2] = d[3] = 0.0f;
    mma_16816(d, p0[0], p1[0], p0[1], p1[1], bx.x, bx.y);
    mma_16816(d, p0[2], p1[2], p0[3], p1[3], bx.z, bx.w);
}

// -------------------------------------------------------------- k_gate_up

__global__ void __launch_bounds__(kWarps * 32) k_gate_up(GemvArgs a)
{
    const int KC = a.kc_gu;
    const int NHB = a.I / 32;
    int unit = blockIdx.x;
    const int kc = unit % KC;
    unit /= KC;
    const int hb = unit % NHB;
    const int j = unit / NHB;          // slot = t * topk + kk
    const int t = j / a.topk;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const MatLayout L = make_layout(2 * a.I, a.H);
    const int kgt = L.kg_full + L.kg_half;
    const int per = (kgt + KC - 1) / KC;
    const int kg0 = kc * per, kg1 = min(kgt, kg0 + per);

    const int e = a.idx[j];
    const uint8_t* cbase = nullptr;
    const uint8_t* sbase = nullptr;
    bool ok = (e >= 0 && e < a.E);
    if (ok) {
        cbase = a.codes[e];
        sbase = a.scales[e];
        ok = cbase && sbase && ((reinterpret_cast<uintptr_t>(cbase) | reinterpret_cast<uintptr_t>(sbase)) & 15) == 0;
    }
    const int tile = hb * 4 + warp;
    const uint8_t* tc = ok ? cbase + (size_t)tile * L.tile_code_bytes() : nullptr;
    const uint8_t* ts = ok ? sbase + (size_t)tile * L.tile_scale_bytes() : nullptr;
    if (ok && kg1 > kg0) {
        // weights do not depend on the previous kernel: start their HBM reads now
        int kf = min(kg1, L.kg_full);
        uint32_t bytes = (uint32_t)(kf - kg0) * 1024u + (kg1 > L.kg_full ? 512u : 0u);
        if (lane == 0) prefetch_l2_bulk(tc + (size_t)kg0 * 1024, bytes);
    }
    pdl_wait();
    pdl_trigger();

    float acc_g = 0.0f, acc_u = 0.0f;
    if (ok) {
        const uint16_t* xt = a.xh + (size_t)t * a.H;
        const float* xst = a.xs + (size_t)t * a.xs_stride;
        int kg = kg0;
        for (; kg < min(kg1, L.kg_full); kg++) {
            const uint8_t* p = tc + (size_t)kg * 1024 + lane * 32;
            uint4 A0 = ldg_stream_v4(p);
            uint4 A1 = ldg_stream_v4(p + 16);
            uint2 S = ldg_stream_v2(ts + (size_t)kg * 64 + g * 8);
            float4 xs4 = *reinterpret_cast<const float4*>(xst + kg * 4);
            uint4 X[4];
#pragma unroll
            for (int jb = 0; jb < 4; jb++)
                X[jb] = (g == 0) ? *reinterpret_cast<const uint4*>(xt + kg * 128 + jb * 32 + 8 * c)
                                 : make_uint4(0, 0, 0, 0);
            const uint32_t r0[4] = {A0.x, A0.y, A0.z, A0.w};
            const uint32_t r1[4] = {A1.x, A1.y, A1.z, A1.w};
            const float xsv[4] = {xs4.x, xs4.y, xs4.z, xs4.w};
#pragma unroll
            for (int jb = 0; jb < 4; jb++) {
                float d[4];
                block_mma(d, r0[jb], r1[jb], X[jb]);
                acc_g = fmaf(d[0] * xsv[jb], ue8m0_f32(byte_of(S.x, jb)), acc_g);
                acc_u = fmaf(d[2] * xsv[jb], ue8m0_f32(byte_of(S.y, jb)), acc_u);
            }
        }
        if (kg < kg1) {  // half k-group (K % 128 == 64)
            const uint8_t* p = tc + (size_t)kg * 1024 + lane * 16;
            uint2 A0 = ldg_stream_v2(p);
            uint2 A1 = ldg_stream_v2(p + 8);
            uint32_t S = ldg_stream_u32(ts + (size_t)kg * 64 + g * 4);
#pragma unroll
            for (int jb = 0; jb < 2; jb++) {
                uint4 X = (g == 0) ? *reinterpret_cast<const uint4*>(xt + kg * 128 + jb * 32 + 8 * c)
                                   : make_uint4(0, 0, 0, 0);
                float xsv = xst[kg * 4 + jb];
                float d[4];
                block_mma(d, jb ? A0.y : A0.x, jb ? A1.y : A1.x, X);
                acc_g = fmaf(d[0] * xsv, ue8m0_f32(byte_of(S, jb)), acc_g);
                acc_u = fmaf(d[2] * xsv, ue8m0_f32(byte_of(S, 2 + jb)), acc_u);
            }
        }
    } else if (threadIdx.x == 0 && kc == 0 && hb == 0) {
        atomicOr(a.status, kStatusBadIndex);
    }

    // this chunk's partial sums: 64 rows = 4 tiles x (8 gate + 8 up)
    float* part = a.part_gu + (((size_t)j * NHB + hb) * KC) * 64;
    if (c == 0) {
        part[kc * 64 + warp * 16 + g] = acc_g;
        part[kc * 64 + warp * 16 + 8 + g] = acc_u;
    }
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        int prev = atomicAdd(a.cnt_gu + (size_t)j * NHB + hb, 1);
        s_last = (prev == KC - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (warp == 0) {
        // lane i owns h index 32*hb + i: tile (i / 8), row (i % 8)
        const int q = lane >> 3, r = lane & 7;
        float gs = 0.0f, us = 0.0f;
        for (int k = 0; k < KC; k++) {
            gs += __ldcg(part + k * 64 + q * 16 + r);
            us += __ldcg(part + k * 64 + q * 16 + 8 + r);
        }
        float h = ok ? silu(gs) * us * a.w[j] : 0.0f;
        float amax = warp_max(fabsf(h));
        int ex = f16_block_exponent(amax);
        float hsd = h * exp2i(-ex);
        __half hi = __float2half_rn(hsd);
        __half lo = __float2half_rn(hsd - __half2float(hi));
        uint16_t* hh = a.hh + ((size_t)j * NHB + hb) * 64;
        hh[lane] = __half_as_ushort(hi);
        hh[32 + lane] = __half_as_ushort(lo);
        if (lane == 0) {
            a.hs[(size_t)j * a.hs_stride + hb] = exp2i(ex);
            a.cnt_gu[(size_t)j * NHB + hb] = 0;   // ready for the next launch
        }
    }
}

// -------------------------------------------------------------- k_down

__global__ void __launch_bounds__(kWarps * 32) k_down(GemvArgs a)
{
    const int NT = a.H / 16;
    const int NHB = a.I / 32;
    int unit = blockIdx.x;
    const int kk = unit % a.topk;
    unit /= a.topk;
    const int tile = unit % NT;
    const int t = unit / NT;
    const int j = t * a.topk + kk;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const MatLayout L = make_layout(a.H, a.I);
    const ExpertLayout EL = make_expert_layout(a.H, a.I);
    const int kgt = L.kg_full + L.kg_half;

    const int e = a.idx[j];
    bool ok = (e >= 0 && e < a.E);
    const uint8_t *tc = nullptr, *ts = nullptr;
    if (ok) {
        const uint8_t* cb = a.codes[e];
        const uint8_t* sb = a.scales[e];
        ok = cb && sb && ((reinterpret_cast<uintptr_t>(cb) | reinterpret_cast<uintptr_t>(sb)) & 15) == 0;
        if (ok) {
            tc = cb + EL.dn_code_off + (size_t)tile * L.tile_code_bytes();
            ts = sb + EL.dn_scale_off + (size_t)tile * L.tile_scale_bytes();
        }
    }
    if (ok && threadIdx.x == 0) prefetch_l2_bulk(tc, (uint32_t)L.tile_code_bytes());
    pdl_wait();
    pdl_trigger();

    float acc0 = 0.0f, acc1 = 0.0f;
    if (ok) {
        const uint16_t* hh = a.hh + (size_t)j * NHB * 64;
        const float* hs = a.hs + (size_t)j * a.hs_stride;
        for (int kg = warp; kg < kgt; kg += kWarps) {
            if (kg < L.kg_full) {
                const uint8_t* p = tc + (size_t)kg * 1024 + lane * 32;
                uint4 A0 = ldg_stream_v4(p);
                uint4 A1 = ldg_stream_v4(p + 16);
                uint2 S = ldg_stream_v2(ts + (size_t)kg * 64 + g * 8);
                float4 hs4 = __ldcg(reinterpret_cast<const float4*>(hs + kg * 4));
                uint4 X[4];
#pragma unroll
                for (int jb = 0; jb < 4; jb++)
                    X[jb] = (g < 2) ? __ldcg(reinterpret_cast<const uint4*>(hh + (size_t)(kg * 4 + jb) * 64 + g * 32 + 8 * c))
                                    : make_uint4(0, 0, 0, 0);
                const uint32_t r0[4] = {A0.x, A0.y, A0.z, A0.w};
                const uint32_t r1[4] = {A1.x, A1.y, A1.z, A1.w};
                const float hsv[4] = {hs4.x, hs4.y, hs4.z, hs4.w};
#pragma unroll
                for (int jb = 0; jb < 4; jb++) {
                    float d[4];
                    block_mma(d, r0[jb], r1[jb], X[jb]);
                    acc0 = fmaf((d[0] + d[1]) * hsv[jb], ue8m0_f32(byte_of(S.x, jb)), acc0);
                    acc1 = fmaf((d[2] + d[3]) * hsv[jb], ue8m0_f32(byte_of(S.y, jb)), acc1);
                }
            } else {
                const uint8_t* p = tc + (size_t)kg * 1024 + lane * 16;
                uint2 A0 = ldg_stream_v2(p);
                uint2 A1 = ldg_stream_v2(p + 8);
                uint32_t S = ldg_stream_u32(ts + (size_t)kg * 64 + g * 4);
#pragma unroll
                for (int jb = 0; jb < 2; jb++) {
                    uint4 X = (g < 2) ? __ldcg(reinterpret_cast<const uint4*>(hh + (size_t)(kg * 4 + jb) * 64 + g * 32 + 8 * c))
                                      : make_uint4(0, 0, 0, 0);
                    float hsv = __ldcg(hs + kg * 4 + jb);
                    float d[4];
                    block_mma(d, jb ? A0.y : A0.x, jb ? A1.y : A1.x, X);
                    acc0 = fmaf((d[0] + d[1]) * hsv, ue8m0_f32(byte_of(S, jb)), acc0);
                    acc1 = fmaf((d[2] + d[3]) * hsv, ue8m0_f32(byte_of(S, 2 + jb)), acc1);
                }
            }
        }
    } else if (threadIdx.x == 0 && tile == 0) {
        atomicOr(a.status, kStatusBadIndex);
    }

    __shared__ float s_red[kWarps][16];
    if (c == 0) {
        s_red[warp][g] = acc0;
        s_red[warp][8 + g] = acc1;
    }
    __syncthreads();
    float* part = a.part_dn + ((size_t)t * NT + tile) * a.topk * 16;
    if (threadIdx.x < 16) {
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; w++) v += s_red[w][threadIdx.x];
        part[kk * 16 + threadIdx.x] = v;
    }
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        int prev = atomicAdd(a.cnt_dn + (size_t)t * NT + tile, 1);
        s_last = (prev == a.topk - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < 16) {
        float v = 0.0f;
        for (int k = 0; k < a.topk; k++) v += __ldcg(part + k * 16 + threadIdx.x);
        size_t o = (size_t)t * a.H + tile * 16 + threadIdx.x;
        if (a.x_resid) {
            a.x_resid[o] += v;
        } else if (a.out_f32) {
            reinterpret_cast<float*>(a.y)[o] = v;
        } else {
            reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(v);
        }
    }
    if (threadIdx.x == 0) a.cnt_dn[(size_t)t * NT + tile] = 0;
}

cudaError_t launch(const void* fn, dim3 grid, dim3 block, cudaStream_t s, bool pdl, GemvArgs* a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[] = {a};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

int gemv_default_kc(int H)
{
    MatLayout L = make_layout(32, H);
    int kgt = L.kg_full + L.kg_half;
    return kgt >= 16 ? 4 : (kgt >= 4 ? 2 : 1);
}

GemvWorkspaceSizes gemv_workspace_sizes(int T, int topk, int H, int I, int kc)
{
    GemvWorkspaceSizes s;
    size_t slots = (size_t)T * topk, nhb = I / 32;
    s.xh = (size_t)T * H;
    s.xs = (size_t)T * ((H / 32 + 3) / 4 * 4);
    s.part_gu = slots * nhb * kc * 64;
    s.cnt_gu = slots * nhb;
    s.hh = slots * nhb * 64;
    s.hs = slots * ((nhb + 3) / 4 * 4);
    s.part_dn = (size_t)T * (H / 16) * topk * 16;
    s.cnt_dn = (size_t)T * (H / 16);
    return s;
}

cudaError_t launch_gemv_layer(const GemvArgs& a0, cudaStream_t s, bool pdl, Profiler* prof)
{
    GemvArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    cudaError_t err;
    struct Step { const void* fn; unsigned grid; int phase; };
    const Step steps[3] = {
        {(const void*)k_prep, (unsigned)a.T, kPhasePrep},
        {(const void*)k_gate_up, (unsigned)(a.T * a.topk * (a.I / 32) * a.kc_gu), kPhaseGateUp},
        {(const void*)k_down, (unsigned)(a.T * (a.H / 16) * a.topk), kPhaseDown},
    };
    for (const Step& st : steps) {
        if (prof) prof->begin(st.phase, s);
        unsigned threads = st.phase == kPhasePrep ? 128u : (unsigned)(kWarps * 32);
        err = launch(st.fn, dim3(st.grid), dim3(threads), s, pdl && !prof, &a);
        if (prof) prof->end(s);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace moe
