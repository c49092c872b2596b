// gemv.cu -- batch-1 / small-batch path of one routed FP4 MoE layer.
//
// Three launches per layer, chained with programmatic dependent launch (PDL):
//   k_prep    x (bf16, or the fp32 residual through a fused RMSNorm) -> f16
//             with one power-of-two scale per 32 elements (exact for bf16).
//   k_stream<gate/up>  h = w_k * silu(Wg x) (.) (Wu x) for every slot (t, k).
//   k_stream<down>     y[t] = sum_k Wd_k h_(t,k), or x += that in a stack.
//
// k_stream is a persistent, one-CTA-per-SM kernel.  The work of a projection
// is a sequence of units -- one k-group (128 K) of one tile group (64 rows) of
// one expert matrix, 4 KB of E2M1 codes + 256 B of ue8m0 scales -- and every
// CTA takes an equal contiguous range of it (stream-K split), so all SMs
// stream the same number of bytes.  One producer thread moves chunks of up to
// 4 units, together with the matching activation slice, from HBM into a ring
// of shared-memory stages with cp.async.bulk and mbarrier transaction counts.
// Consumer warps (one per tile of the group, one or two sets taking alternate
// stages) decode E2M1 pairs to f16 in registers (hardware cvt), multiply on the
// tensor cores (mma.m16n8k16, fp32 accumulate) one 32-weight block at a time,
// and apply the ue8m0 scale of each (row, block) and the activation block
// scale in fp32.  At the end of a reduction group (64 outputs) the warps'
// sums are combined in a fixed order; a group split between CTAs is finished
// by the last contributor, which adds the contributors' partial sums in CTA
// order.  Results are therefore bitwise reproducible on a given GPU.
// Every mbarrier wait is bounded (2 s); on expiry the kernel records the
// "device timeout" status, stops issuing copies and drains what is in flight
// before it exits.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kCU = 4;                                   // units per chunk (stage)
constexpr int kStageCodes = kCU * kUnitCodeBytes;        // 16 KB
constexpr int kStageScales = kCU * kUnitScaleBytes;      // 1 KB
constexpr int kStageB = kCU * 512;                       // activation slice
constexpr int kStageBs = kCU * 16;                       // activation block scales
constexpr int kStageBytes = kStageCodes + kStageScales + kStageB + kStageBs;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

static_assert(kStageBytes % 16 == 0, "stage alignment");

struct JobInfo {
    const uint8_t* code;    // unit k-group 0 of this job's tile group
    const uint8_t* scale;
    const uint8_t* B;       // activation slice at k-group 0
    const uint8_t* Bs;      // activation block scales at k-group 0
    int j, t, tg;
    bool ok;
};

constexpr int kJobWindow = 32;

template <int NSETS, int S>
struct StreamSmem {
    uint8_t stage[S][kStageBytes];
    uint64_t full[S];
    uint64_t empty[S];
    float flush[2][NSETS][kTilesPerGroup][16];
    float comb[2][64];
    JobInfo jobs[kJobWindow];   // the CTA's first jobs, resolved once
    int abort;
};

// Host-computed description of one projection's unit stream.
struct StreamPlan {
    long long U;            // total units
    int G;                  // CTAs
    int kgt, kg_half;       // k-groups per tile (incl. half group), half flag
    int group_units;        // units per reduction group
    int ntg;                // tile groups per expert matrix
    int Bsz, Bblk, ncolB;   // activation bytes per unit, per block; B columns used
    size_t code_off, scale_off, group_code_bytes, group_scale_bytes;
};

// -------------------------------------------------------------- k_prep

__global__ void __launch_bounds__(256) k_prep(GemvArgs a)
{
    const int t = blockIdx.x;
    const int H = a.H;
    __shared__ float s_red[8];
    __shared__ float s_den;

    pdl_wait();
    float den = 1.0f;
    if (a.x_resid) {
        // RMSNorm with unit weight: sum of squares in a fixed tree order
        const float* xr = a.x_resid + (size_t)t * H;
        float ss = 0.0f;
        for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
        ss = warp_sum(ss);
        if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.0f;
            for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += s_red[w];
            s_den = sqrtf(tot / (float)H + a.eps);
        }
        __syncthreads();
        den = s_den;
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
                v[i] = __bfloat162float(__float2bfloat16_rn(v[i] / den));
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

// -------------------------------------------------------------- k_stream

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


template <int PHASE>
__device__ __forceinline__ JobInfo job_info(const GemvArgs& a, const StreamPlan& p, long long job)
{
    JobInfo ji;
    if (PHASE == 0) {        // job = (slot, h-block); B = x of the slot's token
        ji.j = (int)(job / p.ntg);
        ji.tg = (int)(job % p.ntg);
        ji.t = ji.j / a.topk;
        ji.B = reinterpret_cast<const uint8_t*>(a.xh + (size_t)ji.t * a.H);
        ji.Bs = reinterpret_cast<const uint8_t*>(a.xs + (size_t)ji.t * a.xs_stride);
    } else {                 // job = ((t, tile group), slot); B = h of the slot
        const long long grp = job / a.topk;
        const int kk = (int)(job % a.topk);
        ji.t = (int)(grp / p.ntg);
        ji.tg = (int)(grp % p.ntg);
        ji.j = ji.t * a.topk + kk;
        ji.B = reinterpret_cast<const uint8_t*>(a.hh + (size_t)ji.j * (a.I / 32) * 64);
        ji.Bs = reinterpret_cast<const uint8_t*>(a.hs + (size_t)ji.j * a.hs_stride);
    }
    const int e = a.idx[ji.j];
    ji.ok = e >= 0 && e < a.E;
    ji.code = nullptr;
    ji.scale = nullptr;
    if (ji.ok) {
        const uint8_t* cb = a.codes[e];
        const uint8_t* sb = a.scales[e];
        ji.ok = cb && sb && ((reinterpret_cast<uintptr_t>(cb) | reinterpret_cast<uintptr_t>(sb)) & 15) == 0;
        if (ji.ok) {
            ji.code = cb + p.code_off + (size_t)ji.tg * p.group_code_bytes;
            ji.scale = sb + p.scale_off + (size_t)ji.tg * p.group_scale_bytes;
        }
    }
    return ji;
}

__device__ __forceinline__ long long range_start(const StreamPlan& p, int c)
{
    return (long long)c * p.U / p.G;
}

__device__ __forceinline__ int cta_of_unit(const StreamPlan& p, long long x)
{
    return (int)(((x + 1) * p.G - 1) / p.U);
}

// Consume one unit (one k-group of the 4-tile group) from a stage: warp q
// handles tile q.
__device__ __forceinline__ void consume_unit(const uint8_t* stg, int i, bool half, int q, int lane,
                                             const StreamPlan& p, float& acc0, float& acc1)
{
    const int g = lane >> 2, c = lane & 3;
    const uint8_t* codes = stg + i * kUnitCodeBytes;
    const uint8_t* scales = stg + kStageCodes + i * kUnitScaleBytes;
    const uint8_t* B = stg + kStageCodes + kStageScales + i * p.Bsz;
    const float4 bs = *reinterpret_cast<const float4*>(stg + kStageCodes + kStageScales + kStageB + i * 16);
    const bool bcol = g < p.ncolB;
    if (!half) {
        const uint4 A0 = *reinterpret_cast<const uint4*>(codes + q * 1024 + lane * 16);
        const uint4 A1 = *reinterpret_cast<const uint4*>(codes + q * 1024 + 512 + lane * 16);
        const uint2 S = *reinterpret_cast<const uint2*>(scales + q * 64 + g * 8);
        uint4 X[4];
#pragma unroll
        for (int jb = 0; jb < 4; jb++)
            X[jb] = bcol ? *reinterpret_cast<const uint4*>(B + jb * p.Bblk + g * 64 + c * 16)
                         : make_uint4(0, 0, 0, 0);
        const uint32_t r0[4] = {A0.x, A0.y, A0.z, A0.w};
        const uint32_t r1[4] = {A1.x, A1.y, A1.z, A1.w};
        const float bsv[4] = {bs.x, bs.y, bs.z, bs.w};
#pragma unroll
        for (int jb = 0; jb < 4; jb++) {
            float d[4];
            block_mma(d, r0[jb], r1[jb], X[jb]);
            acc0 = fmaf((d[0] + d[1]) * bsv[jb], ue8m0_f32(byte_of(S.x, jb)), acc0);
            acc1 = fmaf((d[2] + d[3]) * bsv[jb], ue8m0_f32(byte_of(S.y, jb)), acc1);
        }
    } else {
        const uint2 A0 = *reinterpret_cast<const uint2*>(codes + q * 512 + lane * 8);
        const uint2 A1 = *reinterpret_cast<const uint2*>(codes + q * 512 + 256 + lane * 8);
        const uint32_t S = *reinterpret_cast<const uint32_t*>(scales + q * 32 + g * 4);
        const float bsv[2] = {bs.x, bs.y};
        const uint32_t r0[2] = {A0.x, A0.y};
        const uint32_t r1[2] = {A1.x, A1.y};
#pragma unroll
        for (int jb = 0; jb < 2; jb++) {
            const uint4 X = bcol ? *reinterpret_cast<const uint4*>(B + jb * p.Bblk + g * 64 + c * 16)
                                 : make_uint4(0, 0, 0, 0);
            float d[4];
            block_mma(d, r0[jb], r1[jb], X);
            acc0 = fmaf((d[0] + d[1]) * bsv[jb], ue8m0_f32(byte_of(S, jb)), acc0);
            acc1 = fmaf((d[2] + d[3]) * bsv[jb], ue8m0_f32(byte_of(S, 2 + jb)), acc1);
        }
    }
}

// Finish a reduction group from its 64 combined sums (smem), by one warp.
template <int PHASE>
__device__ __forceinline__ void finalize_group(const GemvArgs& a, const StreamPlan& p, long long group,
                                               const float* v, int lane)
{
    if (PHASE == 0) {
        // group = (slot j, h-block hb): lane i owns h index 32*hb + i, whose gate
        // and up sums are rows (i%8) and 8+(i%8) of tile i/8
        const int j = (int)(group / p.ntg), hb = (int)(group % p.ntg);
        const int e = a.idx[j];
        const bool ok = e >= 0 && e < a.E;
        const int q = lane >> 3, r = lane & 7;
        const float gs = v[q * 16 + r], us = v[q * 16 + 8 + r];
        const float h = ok ? silu(gs) * us * a.w[j] : 0.0f;
        const float amax = warp_max(fabsf(h));
        const int ex = f16_block_exponent(amax);
        const float hsd = h * exp2i(-ex);
        const __half hi = __float2half_rn(hsd);
        const __half lo = __float2half_rn(hsd - __half2float(hi));
        uint16_t* hh = a.hh + ((size_t)j * p.ntg + hb) * 64;
        hh[lane] = __half_as_ushort(hi);
        hh[32 + lane] = __half_as_ushort(lo);
        if (lane == 0) a.hs[(size_t)j * a.hs_stride + hb] = exp2i(ex);
    } else {
        // group = (token t, tile group tg): 64 output rows, two per lane
        const int t = (int)(group / p.ntg), tg = (int)(group % p.ntg);
#pragma unroll
        for (int h2 = 0; h2 < 2; h2++) {
            const int r = lane + 32 * h2;
            const size_t o = (size_t)t * a.H + (size_t)tg * 64 + r;
            const float val = v[r];
            if (a.x_resid) a.x_resid[o] += val;
            else if (a.out_f32) reinterpret_cast<float*>(a.y)[o] = val;
            else reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(val);
        }
    }
}

template <int PHASE, int NSETS, int S>
__global__ void __launch_bounds__((4 * NSETS + 1) * 32, 1) k_stream(GemvArgs a, StreamPlan p)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    auto& sm = *reinterpret_cast<StreamSmem<NSETS, S>*>(smem_raw);
    constexpr int NCW = 4 * NSETS;          // consumer warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t kgt = (uint32_t)p.kgt;
    const uint32_t u0 = (uint32_t)range_start(p, blockIdx.x);
    const uint32_t u1 = (uint32_t)range_start(p, blockIdx.x + 1);
    const uint32_t j0 = u0 / kgt, jlast = (u1 - 1) / kgt;
    float* part = PHASE == 0 ? a.part_gu : a.part_dn;
    int* cnt = PHASE == 0 ? a.cnt_gu : a.cnt_dn;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 4);
        }
        sm.abort = 0;
        mbar_fence_init();
    }
    if (warp == NCW && j0 + lane <= jlast) {
        // the producer warp resolves the CTA's first jobs (expert pointers) in parallel
        const JobInfo ji = job_info<PHASE>(a, p, j0 + lane);
        sm.jobs[lane] = ji;
        if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
    }
    __syncthreads();
    pdl_trigger();
    auto job_at = [&](uint32_t job) -> JobInfo {
        const uint32_t d = job - j0;
        if (d < (uint32_t)kJobWindow) return sm.jobs[d];
        const JobInfo ji = job_info<PHASE>(a, p, job);
        if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
        return ji;
    };

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        struct Pend { int s; const uint8_t *B, *Bs; uint32_t nb, nbs; };
        Pend pend[S];
        int npend = 0;
        bool pdl_done = false;
        uint32_t u = u0, job = j0, kg = u0 - j0 * kgt;
        JobInfo ji = job_at(job);
        int n = 0;
        while (u < u1) {
            const uint32_t nun = min(min(kgt - kg, u1 - u), (uint32_t)kCU);
            const bool has_half = p.kg_half && (kg + nun == kgt);
            const uint32_t nfull = nun - (has_half ? 1u : 0u);
            const uint32_t cb = nfull * kUnitCodeBytes + (has_half ? kUnitCodeBytes / 2 : 0);
            const uint32_t sb = nfull * kUnitScaleBytes + (has_half ? kUnitScaleBytes / 2 : 0);
            const uint32_t bb = nfull * p.Bsz + (has_half ? p.Bsz / 2 : 0);
            const uint32_t bsb = nun * 16;
            const int s = n % S;
            if (n >= S) {
                if (!pdl_done) {
                    pdl_wait();
                    for (int i = 0; i < npend; i++) {
                        uint8_t* st = sm.stage[pend[i].s];
                        bulk_g2s(st + kStageCodes + kStageScales, pend[i].B, pend[i].nb, &sm.full[pend[i].s]);
                        bulk_g2s(st + kStageCodes + kStageScales + kStageB, pend[i].Bs, pend[i].nbs,
                                 &sm.full[pend[i].s]);
                    }
                    npend = 0;
                    pdl_done = true;
                }
                if (*(volatile int*)&sm.abort ||
                    !mbar_wait_bounded(&sm.empty[s], ((n / S) & 1) ^ 1, kWaitLimitNs)) {
                    atomicOr(a.status, kStatusTimeout);
                    sm.abort = 1;
                    break;
                }
            }
            uint8_t* st = sm.stage[s];
            if (ji.ok) {
                mbar_arrive_expect_tx(&sm.full[s], cb + sb + bb + bsb);
                bulk_g2s(st, ji.code + (size_t)kg * kUnitCodeBytes, cb, &sm.full[s]);
                bulk_g2s(st + kStageCodes, ji.scale + (size_t)kg * kUnitScaleBytes, sb, &sm.full[s]);
                const uint8_t* Bsrc = ji.B + (size_t)kg * p.Bsz;
                const uint8_t* Bssrc = ji.Bs + (size_t)kg * 16;
                if (pdl_done) {
                    bulk_g2s(st + kStageCodes + kStageScales, Bsrc, bb, &sm.full[s]);
                    bulk_g2s(st + kStageCodes + kStageScales + kStageB, Bssrc, bsb, &sm.full[s]);
                } else {
                    pend[npend++] = Pend{s, Bsrc, Bssrc, bb, bsb};
                }
            } else {
                mbar_arrive(&sm.full[s]);      // an empty stage: the consumers skip it
            }
            u += nun;
            kg += nun;
            n++;
            if (kg == kgt && u < u1) {
                kg = 0;
                job++;
                ji = job_at(job);
            }
        }
        if (!pdl_done) {
            pdl_wait();
            for (int i = 0; i < npend; i++) {
                uint8_t* st = sm.stage[pend[i].s];
                bulk_g2s(st + kStageCodes + kStageScales, pend[i].B, pend[i].nb, &sm.full[pend[i].s]);
                bulk_g2s(st + kStageCodes + kStageScales + kStageB, pend[i].Bs, pend[i].nbs,
                         &sm.full[pend[i].s]);
            }
        }
        // drain: no copy may still be in flight into this CTA's memory at exit
        for (int m = n > S ? n - S : 0; m < n; m++)
            mbar_wait_bounded(&sm.full[m % S], (m / S) & 1, kWaitLimitNs);
        return;
    }

    // ---------------------------------------------------------------- consumers
    pdl_wait();
    const int set = warp / 4, q = warp % 4;
    const uint32_t jpg = PHASE == 0 ? 1u : (uint32_t)a.topk;     // jobs per reduction group
    const uint32_t gu = (uint32_t)p.group_units;
    float acc0 = 0.0f, acc1 = 0.0f;
    uint32_t u = u0, job = j0, kg = u0 - j0 * kgt, jg = j0 % jpg, group = j0 / jpg, gstart = u0;
    bool ok = job_at(job).ok;
    int n = 0, fb = 0;
    while (u < u1) {
        const uint32_t nun = min(min(kgt - kg, u1 - u), (uint32_t)kCU);
        if (n % NSETS == set) {
            const int s = n % S;
            bool have = !*(volatile int*)&sm.abort;
            if (have && !mbar_wait_bounded(&sm.full[s], (n / S) & 1, kWaitLimitNs)) {
                if (lane == 0) {
                    atomicOr(a.status, kStatusTimeout);
                    sm.abort = 1;
                }
                have = false;
            }
            if (have && ok) {
                for (uint32_t i = 0; i < nun; i++) {
                    const bool half = p.kg_half && (kg + i == kgt - 1);
                    consume_unit(sm.stage[s], (int)i, half, q, lane, p, acc0, acc1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
        u += nun;
        kg += nun;
        n++;
        bool group_end = (u == u1);
        bool next_group = false;
        if (kg == kgt) {
            kg = 0;
            job++;
            if (++jg == jpg) {
                jg = 0;
                group_end = true;
                next_group = true;
            }
            if (u < u1) ok = job_at(job).ok;
        }
        if (!group_end) continue;

        // ------------------------------------------------ end of a reduction group
        if ((lane & 3) == 0) {
            sm.flush[fb][set][q][lane >> 2] = acc0;
            sm.flush[fb][set][q][8 + (lane >> 2)] = acc1;
        }
        named_sync(1, NCW * 32);
        if (warp == 0) {
            float v0 = 0.0f, v1 = 0.0f;
#pragma unroll
            for (int st = 0; st < NSETS; st++) {
                v0 += sm.flush[fb][st][lane >> 4][lane & 15];
                v1 += sm.flush[fb][st][2 + (lane >> 4)][lane & 15];
            }
            const bool complete = group * gu >= u0 && (group + 1) * gu <= u1;
            bool fin = complete;
            if (!complete) {
                const int slot = (group == u0 / gu) ? 0 : 1;
                float* mine = part + ((size_t)blockIdx.x * 2 + slot) * 64;
                mine[lane] = v0;
                mine[lane + 32] = v1;
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    const int add = (int)(u - gstart);
                    const int old = atomicAdd(cnt + group, add);
                    last = (old + add == (int)gu);
                }
                last = __shfl_sync(0xFFFFFFFFu, last, 0);
                if (last) {
                    __threadfence();
                    const long long gs = (long long)group * gu, ge = gs + gu;
                    const int c0 = cta_of_unit(p, gs), c1 = cta_of_unit(p, ge - 1);
                    v0 = v1 = 0.0f;
                    for (int c = c0; c <= c1; c++) {
                        const int sl = (group == (uint32_t)(range_start(p, c) / gu)) ? 0 : 1;
                        const float* pc = part + ((size_t)c * 2 + sl) * 64;
                        v0 += __ldcg(pc + lane);
                        v1 += __ldcg(pc + lane + 32);
                    }
                    if (lane == 0) cnt[group] = 0;   // ready for the next launch
                    fin = true;
                }
            }
            if (fin) {
                sm.comb[fb][lane] = v0;
                sm.comb[fb][lane + 32] = v1;
                __syncwarp();
                finalize_group<PHASE>(a, p, group, sm.comb[fb], lane);
            }
        }
        acc0 = acc1 = 0.0f;
        fb ^= 1;
        gstart = u;
        if (next_group) group++;
    }
}

cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      void** args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// consumer warp sets (4 warps each) and ring stages; overridable at build time
#ifndef MOE_GEMV_SETS
#define MOE_GEMV_SETS 4
#endif
#ifndef MOE_GEMV_STAGES
#define MOE_GEMV_STAGES 8
#endif
constexpr int kSets = MOE_GEMV_SETS;
constexpr int kStages = MOE_GEMV_STAGES;

StreamPlan make_plan(const GemvArgs& a, int phase, int sms)
{
    StreamPlan p{};
    ExpertLayout E = make_expert_layout(a.H, a.I);
    const MatLayout& L = phase == 0 ? E.gu : E.dn;
    p.kgt = L.kgt();
    p.kg_half = L.kg_half;
    p.ntg = L.groups;
    p.group_code_bytes = L.group_code_bytes();
    p.group_scale_bytes = L.group_scale_bytes();
    if (phase == 0) {
        p.U = (long long)a.T * a.topk * L.groups * p.kgt;
        p.group_units = p.kgt;
        p.Bsz = 256;
        p.Bblk = 64;
        p.ncolB = 1;
        p.code_off = E.gu_code_off;
        p.scale_off = E.gu_scale_off;
    } else {
        p.U = (long long)a.T * L.groups * a.topk * p.kgt;
        p.group_units = a.topk * p.kgt;
        p.Bsz = 512;
        p.Bblk = 128;
        p.ncolB = 2;
        p.code_off = E.dn_code_off;
        p.scale_off = E.dn_scale_off;
    }
    p.G = (int)(p.U < sms ? p.U : sms);
    return p;
}

}  // namespace

size_t gemv_stream_smem() { return sizeof(StreamSmem<kSets, kStages>); }

GemvWorkspaceSizes gemv_workspace_sizes(int T, int topk, int H, int I, int sms)
{
    GemvWorkspaceSizes s;
    size_t slots = (size_t)T * topk, nhb = I / 32;
    s.xh = (size_t)T * H;
    s.xs = (size_t)T * ((H / 32 + 3) / 4 * 4);
    s.part_gu = (size_t)sms * 2 * 64;
    s.cnt_gu = slots * nhb;
    s.hh = slots * nhb * 64;
    s.hs = slots * ((nhb + 3) / 4 * 4);
    s.part_dn = (size_t)sms * 2 * 64;
    s.cnt_dn = (size_t)T * (H / 64);
    return s;
}

cudaError_t gemv_init_device()
{
    const int smem = (int)sizeof(StreamSmem<kSets, kStages>);
    cudaError_t e = cudaFuncSetAttribute((const void*)k_stream<0, kSets, kStages>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute((const void*)k_stream<1, kSets, kStages>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return e;
}

cudaError_t launch_gemv_layer(const GemvArgs& a0, cudaStream_t s, bool pdl, Profiler* prof)
{
    GemvArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    cudaError_t err;
    {
        void* args[] = {&a};
        if (prof) prof->begin(kPhasePrep, s);
        err = launch_ex((const void*)k_prep, dim3(a.T), dim3(128), 0, s, pdl && !prof, args);
        if (prof) prof->end(s);
        if (err != cudaSuccess) return err;
    }
    const size_t smem = sizeof(StreamSmem<kSets, kStages>);
    const dim3 block((4 * kSets + 1) * 32);
    for (int phase = 0; phase < 2; phase++) {
        StreamPlan p = make_plan(a, phase, a.sms);
        void* args[] = {&a, &p};
        const void* fn = phase == 0 ? (const void*)k_stream<0, kSets, kStages>
                                    : (const void*)k_stream<1, kSets, kStages>;
        if (prof) prof->begin(phase == 0 ? kPhaseGateUp : kPhaseDown, s);
        err = launch_ex(fn, dim3(p.G), block, smem, s, pdl && !prof, args);
        if (prof) prof->end(s);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace moe
