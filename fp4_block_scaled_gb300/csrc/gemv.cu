// gemv.cu -- batch-1 / small-batch path of one routed FP4 MoE layer on the
// fifth-generation tensor cores (tcgen05, block-scaled E2M1 MMA).
//
// Three launches per layer, chained with programmatic dependent launch (PDL):
//   k_prep        x (bf16, or the fp32 residual through a fused RMSNorm) ->
//                 8 E2M1 "pieces" per element with one ue8m0 scale per
//                 (piece, 32-block): the MMA's B operand (see layout.h).
//   k_tc<gate/up> per slot (t, k): Wg x and Wu x for 64 outputs per tile,
//                 then h = w_k * silu(g) * u, written back as pieces.
//   k_tc<down>    y[t] = sum_k Wd_k h_(t,k), or x += that in a stack.
//
// k_tc is persistent, one CTA per SM.  A projection is a sequence of units --
// one 128-K slice of one 128-row tile of one expert matrix: 8 KB of E2M1
// codes + a 512 B scale atom -- and each CTA takes an equal contiguous range
// of it (stream-K split), so every SM streams the same number of bytes.
//   warp 0 (one thread)  bulk-copies chunks of 4 units, with the matching
//                        activation pieces, from HBM into a ring of shared-
//                        memory stages (cp.async.bulk, mbarrier tx counts);
//   warps 1-4            one MMA-issuing thread each (tcgen05 issue from a
//                        single thread is serial; from several it overlaps):
//                        issuer i moves the scale atoms of unit i of every
//                        stage to tensor memory (tcgen05.cp) and issues its
//                        block-scaled MMAs (kind::mxf4, M = 128, N = 16, K = 64,
//                        scale_vec 2X) into its own TMEM accumulator;
//                        tcgen05.commit releases its part of the stage;
//   warps 5-8            at the end of each reduction group read the issuers'
//                        accumulators (tcgen05.ld), add the 8 piece columns
//                        and the issuers in a fixed order, and finish the
//                        group: directly when the CTA covered all of it, else
//                        by the last contributor, which adds the CTAs' partial
//                        sums in CTA order.
// The tensor core does the E2M1 decoding, the per-(row, 32-block) scaling and
// the fp32 accumulation; the CUDA cores only touch 128 values per group.
// Results are bitwise reproducible on a given GPU.  Every wait is bounded
// (2 s); on expiry the kernel records the "device timeout" status, stops
// issuing work, waits (bounded) for what is in flight and frees its TMEM.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

// units per chunk (stage) = MMA-issuing warps, and ring stages; build-time tunables
#ifndef MOE_TC_CU
#define MOE_TC_CU 4
#endif
#ifndef MOE_TC_STAGES
#define MOE_TC_STAGES 5
#endif
constexpr int kCU = MOE_TC_CU;
constexpr int kStageCodes = kCU * kUnitCodeBytes;            // 16 KB
constexpr int kStageSfa = kCU * kUnitSfBytes;                // 1 KB
constexpr int kStageB = kCU * kUnitBBytes;                   // 2 KB
constexpr int kStageSfb = kCU * kUnitSfBytes;                // 1 KB
constexpr int kOffSfa = kStageCodes;
constexpr int kOffB = kOffSfa + kStageSfa;
constexpr int kOffSfb = kOffB + kStageB;
constexpr int kStageBytes = kOffSfb + kStageSfb;
constexpr int kStages = MOE_TC_STAGES;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 16;                                 // N = 16 fp32 columns
constexpr int kIssuers = kCU;                                // MMA-issuing warps, one unit of a stage each
constexpr int kSfCol0 = kIssuers * 2 * 16;                  // scale atoms after the accumulators
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kThreads = (1 + kIssuers + 4) * 32;     // producer, issuers, epilogue
constexpr int kJobWindow = 32;

#ifdef MOE_TC_TRACE
// debug builds only: per-event timestamps of CTA 0 ([role][event], ns)
}  // namespace
__device__ long long g_tc_trace[2][4][4096];
__device__ long long g_tc_cta[2][2][1024];   // per-CTA start / end
namespace {
#define TC_TRACE(role, idx)                                                         \
    do {                                                                            \
        if (blockIdx.x == 0 && (idx) < 4096) g_tc_trace[PHASE][role][idx] = (long long)globaltimer_ns(); \
    } while (0)
#else
#define TC_TRACE(role, idx) \
    do {                    \
    } while (0)
#endif

static_assert(kStageBytes % 1024 == 0, "stage alignment");
static_assert(kSfCol0 + kStages * kCU * 8 <= kTmemCols, "tensor memory budget");

struct JobInfo {
    const uint8_t* code;    // unit 0 of this job's tile
    const uint8_t* sf;
    const uint8_t* B;       // activation pieces at unit 0
    const uint8_t* Bsf;
    bool ok;
};

struct TcSmem {
    uint8_t stage[kStages][kStageBytes];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    float comb[kTileRows];
    JobInfo jobs[kJobWindow];
    uint32_t tmem;
    int abort;
    int last;
};

// Host-computed description of one projection's unit stream.
struct StreamPlan {
    long long U;            // total units
    int G;                  // CTAs
    int kgt, kg_half;       // units per tile (incl. half unit), half flag
    int jobs_per_group;     // gate/up: 1 (slot, tile); down: topk slots of (token, tile)
    int ntiles;             // tiles per expert matrix
    size_t code_off, sf_off, tile_code_bytes, tile_sf_bytes;
    size_t act_bytes, act_sf_bytes;    // per B vector
};

// ----------------------------------------------------------------- pieces

// Write the 8 E2M1 pieces of one 32-element block held one value per lane:
// piece p = round(r_p / 2^e_p) with e_p the smallest exponent such that
// max|r_p| <= 6 * 2^e_p, and r_{p+1} = r_p - piece_p * 2^e_p (exact in fp32).
// Bunit: the unit's B codes, Bsf: its scale atom, bu: block index in the unit.
__device__ __forceinline__ void write_pieces(float v, int lane, uint8_t* Bunit, uint8_t* Bsf, int bu)
{
    const int m = bu >> 1, c = bu & 1;
    uint8_t* rows = Bunit + m * kMmaBBytes + c * 128;
    float r = v;
#pragma unroll 1
    for (int p = 0; p < kPieces; p++) {
        const float amax = warp_max(fabsf(r));
        const int s = e2m1_scale_byte(amax);
        const float down = exp2i(127 - s), up = exp2i(s - 127);
        const float q = r * down;
        const float qn = __shfl_xor_sync(0xFFFFFFFFu, q, 1);
        const bool even = (lane & 1) == 0;
        const uint32_t byte = f32x2_to_e2m1x2(even ? q : qn, even ? qn : q);
        const float2 dec = e2m1x2_to_f32x2(byte);
        r -= (even ? dec.x : dec.y) * up;
        if (even) rows[p * 16 + (lane >> 1)] = (uint8_t)byte;
        if (lane == 0) Bsf[p * 16 + bu] = (uint8_t)s;
    }
    // rows 8..15 of the operand are zero, with a finite scale
    reinterpret_cast<uint32_t*>(rows + 256)[lane] = 0u;
    if (lane < 8) Bsf[(kPieces + lane) * 16 + bu] = 127;
}

// ------------------------------------------------------------------ k_prep

// grid (T, ceil(H/32 / 8)), 256 threads: one warp per 32-element block.
__global__ void __launch_bounds__(256) k_prep(GemvArgs a)
{
    const int t = blockIdx.x;
    const int H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
        if (lane == 0) s_red[warp] = ss;
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
    const int b = blockIdx.y * (blockDim.x >> 5) + warp;      // 32-element block
    if (b >= H / 32) return;
    const int i = b * 32 + lane;
    float v;
    if (a.x_resid)  // the MoE input is the bf16 rounding of the norm
        v = __bfloat162float(__float2bfloat16_rn(a.x_resid[(size_t)t * H + i] / den));
    else
        v = __uint_as_float((uint32_t)a.x_bf16[(size_t)t * H + i] << 16);
    const size_t ab = act_bytes(H), asb = act_sf_bytes(H);
    uint8_t* Bunit = a.xq + (size_t)t * ab + (size_t)(b / 4) * kUnitBBytes;
    uint8_t* Bsf = a.xsf + (size_t)t * asb + (size_t)(b / 4) * kUnitSfBytes;
    write_pieces(v, lane, Bunit, Bsf, b % 4);
}

// ------------------------------------------------------------------- k_tc

template <int PHASE>
__device__ __forceinline__ JobInfo job_info(const GemvArgs& a, const StreamPlan& p, long long job)
{
    JobInfo ji;
    int j, t, tile;
    if (PHASE == 0) {        // job = (slot, tile); B = pieces of the slot's token
        j = (int)(job / p.ntiles);
        tile = (int)(job % p.ntiles);
        t = j / a.topk;
        ji.B = a.xq + (size_t)t * p.act_bytes;
        ji.Bsf = a.xsf + (size_t)t * p.act_sf_bytes;
    } else {                 // job = ((token, tile), slot); B = pieces of the slot's h
        const long long grp = job / a.topk;
        const int kk = (int)(job % a.topk);
        t = (int)(grp / p.ntiles);
        tile = (int)(grp % p.ntiles);
        j = t * a.topk + kk;
        ji.B = a.hq + (size_t)j * p.act_bytes;
        ji.Bsf = a.hsf + (size_t)j * p.act_sf_bytes;
    }
    const int e = a.idx[j];
    ji.ok = e >= 0 && e < a.E;
    ji.code = nullptr;
    ji.sf = nullptr;
    if (ji.ok) {
        const uint8_t* cb = a.codes[e];
        const uint8_t* sb = a.scales[e];
        ji.ok = cb && sb && ((reinterpret_cast<uintptr_t>(cb) | reinterpret_cast<uintptr_t>(sb)) & 15) == 0;
        if (ji.ok) {
            ji.code = cb + p.code_off + (size_t)tile * p.tile_code_bytes;
            ji.sf = sb + p.sf_off + (size_t)tile * p.tile_sf_bytes;
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

// Walks a CTA's unit range in chunks (never crossing a job), as every role
// must see the same sequence.
struct Walk {
    uint32_t u, u1, kgt, job, kg, jg, jpg, group;
    __device__ uint32_t chunk() const { return min(min(kgt - kg, u1 - u), (uint32_t)kCU); }
    // advance past a chunk of n units; returns true when a group ended
    __device__ bool advance(uint32_t n, bool& next_job)
    {
        u += n;
        kg += n;
        next_job = false;
        bool gend = (u == u1);
        if (kg == kgt) {
            kg = 0;
            job++;
            next_job = true;
            if (++jg == jpg) {
                jg = 0;
                group++;
                gend = true;
            }
        }
        return gend;
    }
};

template <int PHASE>
__device__ __forceinline__ void finalize_group(const GemvArgs& a, const StreamPlan& p, uint32_t group,
                                               const float* comb, int row, int lane, TcSmem& sm)
{
    if (PHASE == 0) {
        // group = (slot j, tile): rows 0..63 gate, 64..127 up of h indices 64*tile + i;
        // the two warps holding rows 0..63 each turn one 32-block of h into pieces
        if (row >= 64) return;
        const int j = (int)(group / p.ntiles), tile = (int)(group % p.ntiles);
        const int e = a.idx[j];
        const bool ok = e >= 0 && e < a.E;
        const float h = ok ? silu(comb[row]) * comb[64 + row] * a.w[j] : 0.0f;
        const int hb = tile * 2 + (row >> 5);                 // 32-block of h
        uint8_t* Bunit = a.hq + (size_t)j * act_bytes(a.I) + (size_t)(hb / 4) * kUnitBBytes;
        uint8_t* Bsf = a.hsf + (size_t)j * act_sf_bytes(a.I) + (size_t)(hb / 4) * kUnitSfBytes;
        write_pieces(h, lane, Bunit, Bsf, hb % 4);
    } else {
        // group = (token t, tile): 128 output rows, one per thread
        const int t = (int)(group / p.ntiles), tile = (int)(group % p.ntiles);
        const size_t o = (size_t)t * a.H + (size_t)tile * kTileRows + row;
        const float val = comb[row];
        if (a.x_resid) a.x_resid[o] += val;
        else if (a.out_f32) reinterpret_cast<float*>(a.y)[o] = val;
        else reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(val);
    }
}

template <int PHASE>
__global__ void __launch_bounds__(kThreads, 1) k_tc(GemvArgs a, StreamPlan p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t kgt = (uint32_t)p.kgt;
    const uint32_t u0 = (uint32_t)range_start(p, blockIdx.x);
    const uint32_t u1 = (uint32_t)range_start(p, blockIdx.x + 1);
    const uint32_t j0 = u0 / kgt, jlast = (u1 - 1) / kgt;
    const uint32_t jpg = (uint32_t)p.jobs_per_group;
    const uint32_t gunits = kgt * jpg;
    float* part = PHASE == 0 ? a.part_gu : a.part_dn;
    int* cnt = PHASE == 0 ? a.cnt_gu : a.cnt_dn;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kIssuers);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&sm.acc_full[b], kIssuers);
            mbar_init(&sm.acc_empty[b], 4);
        }
        sm.abort = 0;
        mbar_fence_init();
    }
    if (warp == 0 && j0 + lane <= jlast && lane < kJobWindow) {
        // resolve the CTA's first jobs (expert pointers) in parallel
        const JobInfo ji = job_info<PHASE>(a, p, j0 + lane);
        sm.jobs[lane] = ji;
        if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
    }
    if (warp == 1) tmem_alloc(&sm.tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = sm.tmem;
    if (threadIdx.x == 0) TC_TRACE(0, 4095);
#ifdef MOE_TC_TRACE
    if (threadIdx.x == 0) g_tc_cta[PHASE][0][blockIdx.x] = (long long)globaltimer_ns();
#endif
    auto job_at = [&](uint32_t job) -> JobInfo {
        const uint32_t d = job - j0;
        if (d < (uint32_t)kJobWindow) return sm.jobs[d];
        const JobInfo ji = job_info<PHASE>(a, p, job);
        if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
        return ji;
    };
    Walk w0{u0, u1, kgt, j0, u0 - j0 * kgt, j0 % jpg, jpg, j0 / jpg};

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane != 0) return;
        struct Pend { int s; const uint8_t *B, *Bsf; uint32_t nb, nsf; };
        Pend pend[kStages];
        int npend = 0, n = 0;
        bool pdl_done = false;
        Walk wk = w0;
        JobInfo ji = job_at(wk.job);
        while (wk.u < wk.u1) {
            const uint32_t nun = wk.chunk();
            const bool has_half = p.kg_half && (wk.kg + nun == kgt);
            const uint32_t nfull = nun - (has_half ? 1u : 0u);
            const uint32_t cb = nfull * kUnitCodeBytes + (has_half ? kMmaCodeBytes : 0);
            const uint32_t sb = nun * kUnitSfBytes;
            const uint32_t bb = nfull * kUnitBBytes + (has_half ? kMmaBBytes : 0);
            const uint32_t bsb = nun * kUnitSfBytes;
            const int s = n % kStages;
            if (n >= kStages) {
                if (!pdl_done) {
                    pdl_wait();
                    for (int i = 0; i < npend; i++) {
                        uint8_t* st = sm.stage[pend[i].s];
                        bulk_g2s(st + kOffB, pend[i].B, pend[i].nb, &sm.full[pend[i].s]);
                        bulk_g2s(st + kOffSfb, pend[i].Bsf, pend[i].nsf, &sm.full[pend[i].s]);
                    }
                    npend = 0;
                    pdl_done = true;
                }
                if (*(volatile int*)&sm.abort ||
                    !mbar_wait_bounded(&sm.empty[s], ((n / kStages) & 1) ^ 1, kWaitLimitNs)) {
                    atomicOr(a.status, kStatusTimeout);
                    sm.abort = 1;
                    break;
                }
            }
            uint8_t* st = sm.stage[s];
            if (ji.ok) {
                mbar_arrive_expect_tx(&sm.full[s], cb + sb + bb + bsb);
                bulk_g2s(st, ji.code + (size_t)wk.kg * kUnitCodeBytes, cb, &sm.full[s]);
                bulk_g2s(st + kOffSfa, ji.sf + (size_t)wk.kg * kUnitSfBytes, sb, &sm.full[s]);
                const uint8_t* Bsrc = ji.B + (size_t)wk.kg * kUnitBBytes;
                const uint8_t* Bsfsrc = ji.Bsf + (size_t)wk.kg * kUnitSfBytes;
                if (pdl_done) {
                    bulk_g2s(st + kOffB, Bsrc, bb, &sm.full[s]);
                    bulk_g2s(st + kOffSfb, Bsfsrc, bsb, &sm.full[s]);
                } else {
                    pend[npend++] = Pend{s, Bsrc, Bsfsrc, bb, bsb};
                }
            } else {
                mbar_arrive(&sm.full[s]);      // an empty stage: nothing to multiply
            }
            TC_TRACE(0, n);
            bool nj;
            wk.advance(nun, nj);
            n++;
            if (nj && wk.u < wk.u1) ji = job_at(wk.job);
        }
        if (!pdl_done) {
            pdl_wait();
            for (int i = 0; i < npend; i++) {
                uint8_t* st = sm.stage[pend[i].s];
                bulk_g2s(st + kOffB, pend[i].B, pend[i].nb, &sm.full[pend[i].s]);
                bulk_g2s(st + kOffSfb, pend[i].Bsf, pend[i].nsf, &sm.full[pend[i].s]);
            }
        }
        // no copy may still be in flight into this CTA's memory at exit
        for (int m = n > kStages ? n - kStages : 0; m < n; m++)
            mbar_wait_bounded(&sm.full[m % kStages], (m / kStages) & 1, kWaitLimitNs);
        return;
    }

    if (warp >= 1 && warp <= kIssuers) {
        // ------------------------------------------------------------ MMA issue
        // Issuer ii takes unit ii of every stage into its own accumulator:
        // tcgen05 issue from one thread is serial, from several it overlaps.
        if (lane == 0) {
            const int ii = warp - 1;
            const uint32_t idesc = mxf4_idesc(kTileRows, kBRows);
            Walk wk = w0;
            bool ok = job_at(wk.job).ok;
            bool any = false;               // this issuer wrote its accumulator in this group
            int n = 0, buf = 0;
            uint32_t use[2] = {0, 0};
            bool abort = false, group_start = true;
            while (wk.u < wk.u1) {
                const uint32_t nun = wk.chunk();
                const int s = n % kStages;
                if (group_start) {
                    // the epilogue must have read this accumulator's previous group
                    if (!abort && use[buf] > 0 &&
                        !mbar_wait_bounded(&sm.acc_empty[buf], (use[buf] - 1) & 1, kWaitLimitNs)) {
                        atomicOr(a.status, kStatusTimeout);
                        sm.abort = 1;
                        abort = true;
                    }
                    group_start = false;
                }
                if (!abort && (*(volatile int*)&sm.abort ||
                               !mbar_wait_bounded(&sm.full[s], (n / kStages) & 1, kWaitLimitNs))) {
                    atomicOr(a.status, kStatusTimeout);
                    sm.abort = 1;
                    abort = true;
                }
                if (ii == 0) TC_TRACE(1, n);
                if (!abort && ok && (uint32_t)ii < nun) {
                    tc_fence_after();
                    const uint8_t* st = sm.stage[s];
                    const uint32_t col = tmem + kSfCol0 + (uint32_t)(s * kCU + ii) * 8;
                    tc_cp_sf(col, umma_desc(smem_u32(st + kOffSfa + ii * kUnitSfBytes), 16, 128));
                    tc_cp_sf(col + 4, umma_desc(smem_u32(st + kOffSfb + ii * kUnitSfBytes), 16, 128));
                    const bool half = p.kg_half && (wk.kg + (uint32_t)ii == kgt - 1);
                    for (int m = 0; m < (half ? 1 : 2); m++) {
                        const uint64_t ad = umma_desc(smem_u32(st + ii * kUnitCodeBytes + m * kMmaCodeBytes), 128, 256);
                        const uint64_t bd = umma_desc(smem_u32(st + kOffB + ii * kUnitBBytes + m * kMmaBBytes), 128, 256);
                        tc_mma_mxf4(tmem + (uint32_t)(ii * 2 + buf) * kAccCols, ad, bd, mxf4_idesc_sf(idesc, 2 * m),
                                    col, col + 4, any ? 1u : 0u);
                        any = true;
                    }
                }
                tc_commit(&sm.empty[s]);       // this issuer's part of the stage is consumed
                if (ii == 0) TC_TRACE(2, n);
                bool nj;
                const bool gend = wk.advance(nun, nj);
                n++;
                if (nj && wk.u < wk.u1) ok = job_at(wk.job).ok;
                if (gend) {
                    tc_commit(&sm.acc_full[buf]);  // this issuer's accumulator is final
                    use[buf]++;
                    buf ^= 1;
                    any = false;
                    group_start = true;
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        pdl_wait();
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;          // accumulator row of this thread
        const int et = threadIdx.x - (kIssuers + 1) * 32;   // 0..127 among the epilogue threads
        Walk wk = w0;
        uint32_t mask = 0;                         // issuers that accumulated into this group
        bool cur_ok = job_at(wk.job).ok;
        int buf = 0;
        uint32_t use[2] = {0, 0};
        uint32_t gstart = u0;
        while (wk.u < wk.u1) {
            bool nj;
            const uint32_t group = wk.group;
            const uint32_t nun = wk.chunk();
            if (cur_ok) mask |= (1u << nun) - 1u;
            const bool gend = wk.advance(nun, nj);
            if (nj && wk.u < wk.u1) cur_ok = job_at(wk.job).ok;
            if (!gend) continue;

            // ------------------------------------------- end of a reduction group
            const bool ready = mbar_wait_bounded(&sm.acc_full[buf], use[buf] & 1, kWaitLimitNs);
            if (et == 0) TC_TRACE(3, use[0] + use[1]);
            use[buf]++;
            if (!ready) {
                atomicOr(a.status, kStatusTimeout);
                sm.abort = 1;
            }
            tc_fence_after();
            float v = 0.0f;
            if (ready && !*(volatile int*)&sm.abort) {
#pragma unroll
                for (int ii = 0; ii < kIssuers; ii++) {
                    if (!((mask >> ii) & 1u)) continue;
                    float acc[16];
                    tc_ld16(tmem + (uint32_t)(ii * 2 + buf) * kAccCols + ((uint32_t)(quad * 32) << 16), acc);
#pragma unroll
                    for (int c = 0; c < kPieces; c++) v += acc[c];
                }
            }
            mask = 0;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
            buf ^= 1;

            const bool complete = group * gunits >= u0 && (group + 1) * gunits <= u1;
            if (!complete) {
                const int slot = (group == u0 / gunits) ? 0 : 1;
                float* mine = part + ((size_t)blockIdx.x * 2 + slot) * kTileRows;
                mine[row] = v;
                __threadfence();
                named_sync(1, 128);
                if (et == 0) {
                    const int add = (int)(wk.u - gstart);
                    const int old = atomicAdd(cnt + group, add);
                    sm.last = (old + add == (int)gunits);
                }
                named_sync(1, 128);
                const bool last = sm.last;
                if (last) {
                    __threadfence();
                    const long long gs = (long long)group * gunits, ge = gs + gunits;
                    const int c0 = cta_of_unit(p, gs), c1 = cta_of_unit(p, ge - 1);
                    v = 0.0f;
                    for (int c = c0; c <= c1; c++) {
                        const int sl = (group == (uint32_t)(range_start(p, c) / gunits)) ? 0 : 1;
                        v += __ldcg(part + ((size_t)c * 2 + sl) * kTileRows + row);
                    }
                    if (et == 0) cnt[group] = 0;       // ready for the next launch
                }
                if (last) {
                    sm.comb[row] = v;
                    named_sync(1, 128);
                    finalize_group<PHASE>(a, p, group, sm.comb, row, lane, sm);
                }
                named_sync(1, 128);
            } else {
                sm.comb[row] = v;
                named_sync(1, 128);
                finalize_group<PHASE>(a, p, group, sm.comb, row, lane, sm);
                named_sync(1, 128);
            }
            gstart = wk.u;
        }
    }
    // the issuer and epilogue warps meet here before the tensor memory is released
    tc_fence_before();
    named_sync(2, (kIssuers + 4) * 32);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
#ifdef MOE_TC_TRACE
    if (threadIdx.x == 32) g_tc_cta[PHASE][1][blockIdx.x] = (long long)globaltimer_ns();
#endif
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

StreamPlan make_plan(const GemvArgs& a, int phase, int sms)
{
    StreamPlan p{};
    ExpertLayout E = make_expert_layout(a.H, a.I);
    const MatLayout& L = phase == 0 ? E.gu : E.dn;
    p.kgt = L.kgt();
    p.kg_half = L.kg_half;
    p.ntiles = L.tiles;
    p.tile_code_bytes = L.tile_code_bytes();
    p.tile_sf_bytes = L.tile_sf_bytes();
    if (phase == 0) {
        p.U = (long long)a.T * a.topk * L.tiles * p.kgt;
        p.jobs_per_group = 1;
        p.code_off = E.gu_code_off;
        p.sf_off = E.gu_sf_off;
        p.act_bytes = act_bytes(a.H);
        p.act_sf_bytes = act_sf_bytes(a.H);
    } else {
        p.U = (long long)a.T * L.tiles * a.topk * p.kgt;
        p.jobs_per_group = a.topk;
        p.code_off = E.dn_code_off;
        p.sf_off = E.dn_sf_off;
        p.act_bytes = act_bytes(a.I);
        p.act_sf_bytes = act_sf_bytes(a.I);
    }
    p.G = (int)(p.U < sms ? p.U : sms);
    return p;
}

}  // namespace

GemvWorkspaceSizes gemv_workspace_sizes(int T, int topk, int H, int I, int sms)
{
    GemvWorkspaceSizes s;
    const size_t slots = (size_t)T * topk;
    s.xq = (size_t)T * act_bytes(H);
    s.xsf = (size_t)T * act_sf_bytes(H);
    s.hq = slots * act_bytes(I);
    s.hsf = slots * act_sf_bytes(I);
    s.part_gu = (size_t)sms * 2 * kTileRows;
    s.part_dn = (size_t)sms * 2 * kTileRows;
    s.cnt_gu = slots * (size_t)(I / 64);
    s.cnt_dn = (size_t)T * (size_t)(H / kTileRows);
    return s;
}

cudaError_t gemv_init_device()
{
    const int smem = (int)sizeof(TcSmem);
    cudaError_t e = cudaFuncSetAttribute((const void*)k_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute((const void*)k_tc<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return e;
}

size_t gemv_stream_smem() { return sizeof(TcSmem); }

cudaError_t launch_gemv_layer(const GemvArgs& a0, cudaStream_t s, bool pdl, Profiler* prof)
{
    GemvArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    cudaError_t err;
    {
        void* args[] = {&a};
        if (prof) prof->begin(kPhasePrep, s);
        err = launch_ex((const void*)k_prep, dim3(a.T, (a.H / 32 + 7) / 8), dim3(256), 0, s, pdl && !prof, args);
        if (prof) prof->end(s);
        if (err != cudaSuccess) return err;
    }
    for (int phase = 0; phase < 2; phase++) {
        StreamPlan p = make_plan(a, phase, a.sms);
        void* args[] = {&a, &p};
        const void* fn = phase == 0 ? (const void*)k_tc<0> : (const void*)k_tc<1>;
        if (prof) prof->begin(phase == 0 ? kPhaseGateUp : kPhaseDown, s);
        err = launch_ex(fn, dim3(p.G), dim3(kThreads), sizeof(TcSmem), s, pdl && !prof, args);
        if (prof) prof->end(s);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace moe
