// gemv.cu -- batch-1 / small-batch path of one routed FP4 MoE layer on the
// fifth-generation tensor cores (tcgen05, block-scaled E2M1 MMA).
//
// Two launches per layer, chained with programmatic dependent launch (PDL):
//   k_prep   x (bf16, or the fp32 residual through a fused RMSNorm) -> 16
//            E2M1 "pieces" per element with one ue8m0 scale per (piece,
//            32-block): the MMA's B operand (see layout.h).
//   k_layer  both projections in one persistent grid, one CTA per SM:
//            gate/up: per slot (t, k), Wg x and Wu x for 64 outputs per tile,
//                     then h = w_k * silu(g) * u, written back as pieces;
//            down:    y[t] = sum_k Wd_k h_(t,k), or x += that in a stack.
//
// A projection is a sequence of units -- one 128-K slice of one 128-row tile
// of one expert matrix: 8 KB of E2M1 codes + a 512 B scale atom -- and each
// CTA takes an equal contiguous range of it (stream-K split), so every SM
// streams the same number of bytes.  Per CTA (kCU = 5 units per stage, 4
// stages):
//   warp 0 (one thread)  streams the weights: bulk-copies chunks of kCU units
//                        (codes + scale atoms) from HBM into a ring of
//                        shared-memory stages (cp.async.bulk, mbarrier tx
//                        counts), gate/up then down without a pause; nothing
//                        is prefetched beyond the ring, so the gate/up tail and
//                        the h hand-off do not queue behind down weights;
//   last warp            copies the matching activation pieces into each
//                        stage: x's once the previous kernel is done (PDL),
//                        h's once every gate/up group of the grid has been
//                        finalized (a grid-wide counter, bounded wait); before
//                        that wait it makes its own CTA's finished groups
//                        grid-visible (the finalizing warps hand them over at
//                        CTA scope and go on);
//   warps 1..kCU         one MMA-issuing thread each (one thread issues a
//                        tcgen05 instruction per ~150 cycles; several overlap):
//                        issuer i moves the scale atoms of unit i of every
//                        stage to tensor memory (tcgen05.cp) and issues its
//                        block-scaled MMAs (kind::mxf4, M = 128, N = 16, K = 64,
//                        scale_vec 2X) into its own TMEM accumulator;
//                        tcgen05.commit releases its part of the stage;
//   4 epilogue warps     at the end of each reduction group read the issuers'
//                        accumulators (tcgen05.ld), add the 16 piece columns
//                        and the issuers in a fixed order, and finish the
//                        group.  A group split over several CTAs is finished
//                        by the one holding its first unit, which reaches it
//                        last; the others leave launch-tagged partial sums
//                        that it adds in CTA order (no fences or counters on
//                        the way, and mostly read before its own sum is done).
//                        The owned gate/up groups' h go to the four warps in
//                        turn.
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
#define MOE_TC_CU 5
#endif
#ifndef MOE_TC_STAGES
#define MOE_TC_STAGES 4
#endif
constexpr int kCU = MOE_TC_CU;
constexpr int kStageA = kCU * kUnitBytes;                    // kCU units of weights: codes + scale atom each
constexpr int kStageB = kCU * kUnitBBytes;                   // their activation pieces
constexpr int kStageSfb = kCU * kUnitSfBytes;                // and the pieces' scale atoms
constexpr int kOffB = kStageA;
constexpr int kOffSfb = kOffB + kStageB;
constexpr int kStageBytes = (kOffSfb + kStageSfb + 1023) / 1024 * 1024;
constexpr int kStages = MOE_TC_STAGES;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 16;                                 // N = 16 fp32 columns
constexpr int kIssuers = kCU;                                // MMA-issuing warps, one unit of a stage each
constexpr int kSfCol0 = kIssuers * 2 * kAccCols;             // scale atoms after the accumulators
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
constexpr int kWarpEpi0 = 1 + kIssuers;                      // first of the 4 epilogue warps
constexpr int kWarpLoader = kWarpEpi0 + 4;                   // activation copies
constexpr int kThreads = (kWarpLoader + 1) * 32;
constexpr int kJobWindow = 32;
constexpr int kSlotCache = 256;                              // routing weights kept in shared memory

#ifdef MOE_TC_TRACE
// debug builds only: per-event timestamps of CTA 0 ([phase][role][idx], ns)
// and per-CTA milestones
}  // namespace
__device__ long long g_tc_trace[2][4][4096];
__device__ long long g_tc_cta[12][1024];
__device__ long long g_tc_grp[5][1024];   // per gate/up group: acc ready, folded, barrier, fin start, fin end
__device__ long long g_tc_fin[4][64];
namespace {
#define TC_FIN(step, idx)                                                                       \
    do {                                                                                        \
        if (blockIdx.x == 0 && lane == 0 && (idx) < 64) g_tc_fin[step][idx] = (long long)globaltimer_ns(); \
    } while (0)
#define TC_TRACE(ph, role, idx)                                                     \
    do {                                                                            \
        if (blockIdx.x == 0 && (idx) < 4096) g_tc_trace[ph][role][idx] = (long long)globaltimer_ns(); \
    } while (0)
#define TC_CTA(slot) (g_tc_cta[slot][blockIdx.x] = (long long)globaltimer_ns())
#define TC_GRP(k, g) (g_tc_grp[k][(g) & 1023] = (long long)globaltimer_ns())
#else
#define TC_TRACE(ph, role, idx) \
    do {                        \
    } while (0)
#define TC_CTA(slot) \
    do {             \
    } while (0)
#define TC_FIN(step, idx) \
    do {                  \
    } while (0)
#define TC_GRP(k, g) \
    do {             \
    } while (0)
#endif

static_assert(kStageBytes % 1024 == 0, "stage alignment");
static_assert(kSfCol0 + kStages * kCU * 8 <= kTmemCols, "tensor memory budget");
static_assert(kPieces == kAccCols && kBRows == kAccCols, "one accumulator column per piece");
// k_layer's CTAs wait on one another (the down projection needs every h), so
// two of them must never share an SM, where the second would block in the
// tensor-memory allocation: the dynamic shared memory asked for is at least
// more than half of an SM's.
constexpr size_t kOneCtaPerSmSmem = 116 * 1024;
// activation numerics, one instance of the layer kernel each (each instance
// holds only its own mode's code, which keeps the kernel small: its code
// competes for the instruction caches with the weight stream)
enum : int { kModeBf16 = 0, kModeE4m3 = 1, kModeE2m1 = 2 };

struct JobInfo {
    const uint8_t* w;       // unit 0 of this job's weight tile (codes + scale atom per unit)
    const uint8_t* B;       // activation pieces at unit 0
    const uint8_t* Bsf;
    bool ok;
};

// Activation copy of one stage, posted by the weight producer.
struct BSrc {
    const uint8_t* B;       // nullptr: the stage multiplies nothing
    const uint8_t* Bsf;
    uint32_t nb, nsf;
    int phase;
};

struct TcSmem {
    uint8_t stage[kStages][kStageBytes];
    uint64_t full[kStages];      // weights + activations of the stage landed
    uint64_t empty[kStages];     // the issuers are done with the stage
    uint64_t posted[kStages];    // the producer issued the stage's weights and posted bsrc
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain[kIssuers];    // the issuers' last MMAs are done
    BSrc bsrc[kStages];
    float comb[4][kTileRows];    // gate/up sums of the last four owned groups
    uint4 tr[4][32];             // per epilogue warp: the pieces' byte transpose
    float slot_w[kSlotCache];    // w of each slot, 0 where its expert index is invalid
    JobInfo jobs[2][kJobWindow]; // first jobs of the gate/up and down streams
    uint32_t tmem;
    int abort;
    int last;
    // finished gate/up groups of this CTA: (count << 32) | h tiles written,
    // added at CTA scope by the finalizing warps; the loader thread makes them
    // grid-visible (it alone waits for the release at GPU scope)
    unsigned long long fin_word;
};

// Host-computed description of one projection's unit stream.
struct StreamPlan {
    long long U;            // total units
    int G;                  // CTAs
    int kgt, kg_half;       // units per tile (incl. half unit), half flag
    int jobs_per_group;     // gate/up: 1 (slot, tile); down: topk slots of (token, tile)
    int ntiles;             // tiles per expert matrix
    size_t off, tile_bytes; // the matrix in the expert blob, one tile
    size_t act_bytes, act_sf_bytes;    // per B vector
};

// ----------------------------------------------------------------- pieces

// Pieces of 64 consecutive elements of a vector -- the 32-blocks blk0 and
// blk0 + 1, blk0 even, so both lie in one MMA's K range -- held two per lane
// (lane l: elements 2l and 2l + 1 of the span).  With e_0 the smallest
// exponent such that the block's max|v| <= 6 * 2^e_0, piece p is the E2M1
// rounding of the residual r_p at the scale 2^(e_0 - 2p), and r_(p+1) = r_p -
// piece_p * 2^(e_0 - 2p), exact in fp32.  Rounding to E2M1 leaves at most
// 2^(e_0 - 2p) of residual, inside the next piece's range 6 * 2^(e_0 - 2p - 2),
// so the 16 pieces carry every element to within 2^(e_0 - 30) while only the
// first scale needs a reduction across lanes.
// Bunit: the unit's B codes, Bsf: its scale atom.
// The half-warp's 16 x 16 bytes (lane: its byte of each piece) are transposed
// through `scratch` (32 x 16 bytes, this warp's) so that each lane stores one
// 16-byte row -- piece i of its block -- and one scale byte.
__device__ __forceinline__ void write_pieces64(float v0, float v1, int lane, uint8_t* Bunit, uint8_t* Bsf,
                                               int blk0, uint4* scratch)
{
    const int bu = (blk0 & 3) + (lane >> 4);       // block within the unit
    const int i = lane & 15;                       // byte within the block's row
    float amax = fmaxf(fabsf(v0), fabsf(v1));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int s0 = e2m1_scale_byte(amax);
    float r0 = v0, r1 = v1;
    uint32_t w[4] = {0u, 0u, 0u, 0u};              // byte p: this lane's pair of piece p
#pragma unroll
    for (int p = 0; p < kPieces; p++) {
        const int s = max(s0 - 2 * p, 1);
        const float down = exp2i(127 - s), up = exp2i(s - 127);
        const uint32_t byte = f32x2_to_e2m1x2(r0 * down, r1 * down);
        const float2 d = e2m1x2_to_f32x2(byte);
        r0 = fmaf(-d.x, up, r0);
        r1 = fmaf(-d.y, up, r1);
        w[p >> 2] |= (byte & 0xFFu) << (8 * (p & 3));
    }
    scratch[lane] = make_uint4(w[0], w[1], w[2], w[3]);
    __syncwarp();
    const uint8_t* sb = reinterpret_cast<const uint8_t*>(scratch + (lane & 16));   // this half-warp's lanes
    uint32_t row[4];
#pragma unroll
    for (int q = 0; q < 4; q++)
        row[q] = (uint32_t)sb[(4 * q) * 16 + i] | ((uint32_t)sb[(4 * q + 1) * 16 + i] << 8) |
                 ((uint32_t)sb[(4 * q + 2) * 16 + i] << 16) | ((uint32_t)sb[(4 * q + 3) * 16 + i] << 24);
    __syncwarp();                                  // scratch free again
    uint8_t* dst = Bunit + (bu >> 1) * kMmaBBytes + (bu & 1) * 128 + (i >> 3) * 256 + (i & 7) * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(row[0], row[1], row[2], row[3]);
    Bsf[i * 16 + bu] = (uint8_t)max(s0 - 2 * i, 1);
}

// write_pieces64 with the piece loop rolled: the layer kernel's copy has to
// stay small, since its code competes for the instruction caches with the
// weight stream (each piece byte goes to the transpose buffer as it comes).
__device__ __forceinline__ void write_pieces64_small(float v0, float v1, int lane, uint8_t* Bunit, uint8_t* Bsf,
                                                     int blk0, uint4* scratch)
{
    const int bu = (blk0 & 3) + (lane >> 4);
    const int i = lane & 15;
    float amax = fmaxf(fabsf(v0), fabsf(v1));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int s0 = e2m1_scale_byte(amax);
    float r0 = v0, r1 = v1;
    uint8_t* mine = reinterpret_cast<uint8_t*>(scratch + lane);
#pragma unroll 1
    for (int p = 0; p < kPieces; p++) {
        const int s = max(s0 - 2 * p, 1);
        const float down = exp2i(127 - s), up = exp2i(s - 127);
        const uint32_t byte = f32x2_to_e2m1x2(r0 * down, r1 * down);
        const float2 d = e2m1x2_to_f32x2(byte);
        r0 = fmaf(-d.x, up, r0);
        r1 = fmaf(-d.y, up, r1);
        mine[p] = (uint8_t)byte;
    }
    __syncwarp();
    const uint8_t* sb = reinterpret_cast<const uint8_t*>(scratch + (lane & 16));   // this half-warp's lanes
    uint32_t row[4];
#pragma unroll
    for (int q = 0; q < 4; q++)
        row[q] = (uint32_t)sb[(4 * q) * 16 + i] | ((uint32_t)sb[(4 * q + 1) * 16 + i] << 8) |
                 ((uint32_t)sb[(4 * q + 2) * 16 + i] << 16) | ((uint32_t)sb[(4 * q + 3) * 16 + i] << 24);
    __syncwarp();                                  // scratch free again
    uint8_t* dst = Bunit + (bu >> 1) * kMmaBBytes + (bu & 1) * 128 + (i >> 3) * 256 + (i & 7) * 16;
    *reinterpret_cast<uint4*>(dst) = make_uint4(row[0], row[1], row[2], row[3]);
    Bsf[i * 16 + bu] = (uint8_t)max(s0 - 2 * i, 1);
}

// ------------------------------------------------------------------ k_prep

constexpr int kPrepParts = 1024;

// grid (T, ceil(H/64 / 8)), 256 threads: one warp per 64 elements.
__global__ void __launch_bounds__(256) k_prep(GemvArgs a)
{
    const int t = blockIdx.x;
    const int H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_part[kPrepParts];   // the RMSNorm's partial sums of squares, per 32 rows
    __shared__ uint4 s_tr[8][32];          // per warp: the pieces' byte transpose

    // k_layer reads nothing this kernel or the previous layer writes before its
    // own wait, so it may start (on the SMs the previous layer frees) right away
    pdl_trigger();
    pdl_wait();
    // this warp's elements of the residual, loaded before the sum of squares
    // so that the two reads overlap (E4M3: a 128-element block, 4 per lane;
    // otherwise a 64-element span, 2 per lane)
    const int wb = blockIdx.y * (blockDim.x >> 5) + warp;
    float xv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (a.x_resid && wb < (a.act_e4m3 ? H / 128 : H / 64)) {
        const float* xr = a.x_resid + (size_t)t * H;
        if (a.act_e4m3) {
#pragma unroll
            for (int hh = 0; hh < 2; hh++)
#pragma unroll
                for (int e = 0; e < 2; e++) xv[2 * hh + e] = __ldcg(xr + wb * 128 + hh * 64 + 2 * lane + e);
        } else {
            xv[0] = __ldcg(xr + wb * 64 + 2 * lane);
            xv[1] = __ldcg(xr + wb * 64 + 2 * lane + 1);
        }
    }
    float den = 1.0f;
    if (a.x_resid) {
        // RMSNorm with unit weight.  The sum of squares in one fixed order: per
        // 32 rows a butterfly sum of the squares (lane l: row 32 g + l), then the
        // H / 32 partials added lane-strided in index order and a butterfly sum
        // -- the order in which a stack's layer leaves them for the next one
        // (ssq_in: read instead of the row, 128 floats instead of 4096)
        const int ng = H / 32, nw = (int)(blockDim.x >> 5);
        float ss = 0.0f;
        if (a.ssq_in) {
            const float* part = a.ssq + (size_t)t * ng;
            for (int q = lane; q < ng; q += 32) ss += __ldcg(part + q);
        } else {
            const float* xr = a.x_resid + (size_t)t * H;
            for (int g0 = 0; g0 < ng; g0 += kPrepParts) {
                const int gn = min(kPrepParts, ng - g0);
                // warp w: groups w, w + nw, ..., eight loads in flight
                for (int q0 = warp; q0 < gn; q0 += 8 * nw) {
                    float v[8];
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        const int q = q0 + nw * k;
                        v[k] = q < gn ? __ldcg(xr + (size_t)(g0 + q) * 32 + lane) : 0.0f;
                    }
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        const float p = warp_sum(__fmul_rn(v[k], v[k]));
                        if (q0 + nw * k < gn && lane == 0) s_part[q0 + nw * k] = p;
                    }
                }
                __syncthreads();
                for (int q = lane; q < gn; q += 32) ss += s_part[q];
                __syncthreads();
            }
        }
        den = sqrtf(warp_sum(ss) / (float)H + a.eps);
    }
    if (a.act_e4m3) {
        // x quantized to E4M3 under one ue8m0 scale per 128 elements (lane l holds
        // elements 2l, 2l + 1 of each half), and the dequantized values as pieces
        const int b = wb;                                      // 128-element block
        if (b >= H / 128) return;
        float v[4];
        for (int hh = 0; hh < 2; hh++)
            for (int e = 0; e < 2; e++) {
                const int i = b * 128 + hh * 64 + 2 * lane + e;
                v[2 * hh + e] = a.x_resid ? __bfloat162float(__float2bfloat16_rn(xv[2 * hh + e] / den))
                                          : __uint_as_float((uint32_t)a.x_bf16[(size_t)t * H + i] << 16);
            }
        const float amax = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
        const int s = ue8m0_for_amax_bits(amax);
        for (int hh = 0; hh < 2; hh++) {
            uint8_t* Bunit = a.xq + (size_t)t * act_bytes(H) + (size_t)b * kUnitBBytes;
            uint8_t* Bsf = a.xsf + (size_t)t * act_sf_bytes(H) + (size_t)b * kUnitSfBytes;
            write_pieces64(e4m3_quant_dequant(v[2 * hh], s), e4m3_quant_dequant(v[2 * hh + 1], s), lane, Bunit,
                           Bsf, 2 * hh, s_tr[warp]);
        }
        return;
    }
    const int b = wb;                                          // 64-element span
    if (b >= H / 64) return;
    const int i = b * 64 + 2 * lane;
    float v0, v1;
    if (a.x_resid) {  // the MoE input is the bf16 rounding of the norm
        v0 = __bfloat162float(__float2bfloat16_rn(xv[0] / den));
        v1 = __bfloat162float(__float2bfloat16_rn(xv[1] / den));
    } else {
        const uint16_t* xb = a.x_bf16 + (size_t)t * H + i;   // only 2-byte alignment is assumed
        v0 = __uint_as_float((uint32_t)xb[0] << 16);
        v1 = __uint_as_float((uint32_t)xb[1] << 16);
    }
    if (a.act_e2m1) {      // x quantized to E2M1 per 32 (carried exactly by the pieces)
        const float2 q = e2m1_block_quant_dequant(v0, v1);
        v0 = q.x;
        v1 = q.y;
    }
    uint8_t* Bunit = a.xq + (size_t)t * act_bytes(H) + (size_t)(b / 2) * kUnitBBytes;
    uint8_t* Bsf = a.xsf + (size_t)t * act_sf_bytes(H) + (size_t)(b / 2) * kUnitSfBytes;
    write_pieces64(v0, v1, lane, Bunit, Bsf, 2 * b, s_tr[warp]);
}

// ----------------------------------------------------------------- k_layer

// Limit of every bounded wait of the launch.
__device__ __forceinline__ uint64_t wait_limit(const GemvArgs& a) { return a.wait_ns ? a.wait_ns : kDefaultWaitNs; }

// The slot j and weight tile of a job.
template <int PHASE>
__device__ __forceinline__ void job_slot(const GemvArgs& a, const StreamPlan& p, long long job, int& j, int& tile)
{
    if (PHASE == 0) {        // job = (slot, tile)
        j = (int)(job / p.ntiles);
        tile = (int)(job % p.ntiles);
    } else {                 // job = ((token, tile), slot)
        const long long grp = job / a.topk;
        const int kk = (int)(job % a.topk);
        const int t = (int)(grp / p.ntiles);
        tile = (int)(grp % p.ntiles);
        j = t * a.topk + kk;
    }
}

// A job's weight and activation sources, given its slot's expert id e and that
// expert's blob (read only when e is in range).
template <int PHASE>
__device__ __forceinline__ JobInfo job_info_e(const GemvArgs& a, const StreamPlan& p, int j, int tile, int e,
                                              const uint8_t* blob)
{
    JobInfo ji;
    if (PHASE == 0) {        // B = pieces of the slot's token
        const int t = j / a.topk;
        ji.B = a.xq + (size_t)t * p.act_bytes;
        ji.Bsf = a.xsf + (size_t)t * p.act_sf_bytes;
    } else {                 // B = pieces of the slot's h
        ji.B = a.hq + (size_t)j * p.act_bytes;
        ji.Bsf = a.hsf + (size_t)j * p.act_sf_bytes;
    }
    ji.ok = e >= 0 && e < a.E && blob && (reinterpret_cast<uintptr_t>(blob) & 15) == 0;
    ji.w = ji.ok ? blob + p.off + (size_t)tile * p.tile_bytes : nullptr;
    return ji;
}

template <int PHASE>
__device__ __forceinline__ JobInfo job_info(const GemvArgs& a, const StreamPlan& p, long long job)
{
    int j, tile;
    job_slot<PHASE>(a, p, job, j, tile);
    const int e = a.idx[j];
    const bool in = e >= 0 && e < a.E;
    return job_info_e<PHASE>(a, p, j, tile, e, in ? a.experts[e] : nullptr);
}

__device__ __forceinline__ long long range_start(const StreamPlan& p, int c)
{
    return (long long)c * p.U / p.G;
}

__device__ __forceinline__ int cta_of_unit(const StreamPlan& p, long long x)
{
    return (int)(((x + 1) * p.G - 1) / p.U);
}

// A CTA's unit range of one projection.
struct Range {
    uint32_t u0, u1, j0, jlast;
};

__device__ __forceinline__ Range cta_range(const StreamPlan& p)
{
    Range r;
    r.u0 = (uint32_t)range_start(p, blockIdx.x);
    r.u1 = (uint32_t)range_start(p, blockIdx.x + 1);
    r.j0 = r.u0 / (uint32_t)p.kgt;
    r.jlast = (r.u1 - 1) / (uint32_t)p.kgt;
    return r;
}

// Walks a CTA's unit range in chunks (never crossing a job), as every role
// must see the same sequence.
struct Walk {
    uint32_t u, u1, kgt, job, kg, jg, jpg, group;
    __device__ Walk(const StreamPlan& p, const Range& r)
    {
        u = r.u0;
        u1 = r.u1;
        kgt = (uint32_t)p.kgt;
        job = r.j0;
        kg = r.u0 - r.j0 * kgt;
        jpg = (uint32_t)p.jobs_per_group;
        jg = r.j0 % jpg;
        group = r.j0 / jpg;
    }
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

__device__ __forceinline__ int count_chunks(const StreamPlan& p, const Range& r)
{
    Walk wk(p, r);
    int n = 0;
    while (wk.u < wk.u1) {
        bool nj;
        wk.advance(wk.chunk(), nj);
        n++;
    }
    return n;
}

template <int PHASE>
__device__ __forceinline__ JobInfo job_at(const GemvArgs& a, const StreamPlan& p, const Range& r, TcSmem& sm,
                                          uint32_t job)
{
    const uint32_t d = job - r.j0;
    if (d < (uint32_t)kJobWindow) return sm.jobs[PHASE][d];
    const JobInfo ji = job_info<PHASE>(a, p, job);
    if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
    return ji;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const int* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void set_abort(const GemvArgs& a, TcSmem& sm)
{
    atomicOr(a.status, kStatusTimeout);
    sm.abort = 1;
}

// ------------------------------------------------------------------ producer

// Streams the weights of one projection's range into the ring and posts each
// stage's activation source to the loader.  n: chunks so far (both phases).
template <int PHASE>
__device__ bool produce(const GemvArgs& a, const StreamPlan& p, const Range& r, TcSmem& sm, int& n)
{
    Walk wk(p, r);
    const uint32_t kgt = wk.kgt;
    JobInfo ji = job_at<PHASE>(a, p, r, sm, wk.job);
    while (wk.u < wk.u1) {
        const uint32_t nun = wk.chunk();
        const bool has_half = p.kg_half && (wk.kg + nun == kgt);
        const uint32_t nfull = nun - (has_half ? 1u : 0u);
        const uint32_t wb = nfull * kUnitBytes + (has_half ? kHalfUnitBytes : 0);   // one copy
        const uint32_t bb = nfull * kUnitBBytes + (has_half ? kMmaBBytes : 0);
        const uint32_t bsb = nun * kUnitSfBytes;
        const int s = n % kStages;
        if (n >= kStages && !mbar_wait_or_abort(&sm.empty[s], ((n / kStages) & 1) ^ 1, &sm.abort, wait_limit(a))) {
            set_abort(a, sm);
            return false;
        }
        uint8_t* stg = sm.stage[s];
        if (ji.ok) {
            mbar_arrive_expect_tx(&sm.full[s], wb + bb + bsb);
            bulk_g2s(stg, ji.w + (size_t)wk.kg * kUnitBytes, wb, &sm.full[s]);
            sm.bsrc[s] = BSrc{ji.B + (size_t)wk.kg * kUnitBBytes, ji.Bsf + (size_t)wk.kg * kUnitSfBytes, bb, bsb,
                              PHASE};
        } else {
            mbar_arrive(&sm.full[s]);      // an empty stage: nothing to multiply
            sm.bsrc[s] = BSrc{nullptr, nullptr, 0, 0, PHASE};
        }
        mbar_arrive(&sm.posted[s]);        // release: bsrc is visible to the loader
        TC_TRACE(PHASE, 0, n);
        bool nj;
        wk.advance(nun, nj);
        n++;
        if (nj && wk.u < wk.u1) ji = job_at<PHASE>(a, p, r, sm, wk.job);
    }
    return true;
}

// ------------------------------------------------------------------ loader

// Issues the activation copies of every stage the producer posted, in order.
// x's pieces wait for the previous kernel (PDL); h's for the grid-wide count
// of finalized gate/up groups.  Once a stage is posted its copies are always
// issued, even after a timeout, so that every transaction count completes.
__device__ __forceinline__ unsigned long long ld_acquire_cta_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.cta.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

// Makes this CTA's `owned` finished gate/up groups grid-visible, as they come:
// each increment of the CTA-scope word is added to the grid-wide count with a
// GPU-scope release (cumulative over the finalizing warps' stores, which it
// acquired).  Bounded; false on timeout or abort.
__device__ bool publish_own_groups(const GemvArgs& a, TcSmem& sm, uint32_t owned)
{
    uint32_t cnt = 0, pub = 0;
    uint64_t t0 = 0;
    // test hook: the first CTA keeps its groups back, so the others' waits run out
    const bool withhold = a.debug_withhold && blockIdx.x == 0;
    while (cnt < owned) {
        const unsigned long long w = ld_acquire_cta_u64(&sm.fin_word);
        const uint32_t c = (uint32_t)(w >> 32), d = (uint32_t)w;
        if (d > pub && !withhold) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(a.sync), "r"(d - pub) : "memory");
            pub = d;
        }
        if (c > cnt) {
            cnt = c;
            t0 = 0;
            continue;
        }
        if (*(volatile int*)&sm.abort) return false;
        if (t0 == 0) t0 = wait_clock();
        else if (wait_clock() - t0 > wait_cycles(wait_limit(a))) return false;
    }
    return true;
}

__device__ void load_b(const GemvArgs& a, int nchunks, uint32_t gu_groups, uint32_t owned, TcSmem& sm)
{
    bool pdl_done = false, h_done = false, published = false;
    for (int n = 0; n < nchunks; n++) {
        const int s = n % kStages;
        if (!mbar_wait_or_abort(&sm.posted[s], (n / kStages) & 1, &sm.abort, wait_limit(a))) {
            set_abort(a, sm);
            return;
        }
        const BSrc q = sm.bsrc[s];
        if (q.phase == 1 && !published) {
            // every CTA's finished gate/up groups must reach the grid-wide count,
            // also when its own down stages multiply nothing
            if (!publish_own_groups(a, sm, owned)) set_abort(a, sm);
            published = true;
        }
        if (!q.B) continue;
        if (!pdl_done) {
            pdl_wait();
            pdl_done = true;
        }
        if (q.phase == 1 && !h_done) {
            bool ok = ld_acquire_u32(a.sync) >= gu_groups;
            if (!ok) {
                const uint64_t t0 = wait_clock();
                while (!(ok = ld_acquire_u32(a.sync) >= gu_groups))
                    if (*(volatile int*)&sm.abort || wait_clock() - t0 > wait_cycles(wait_limit(a))) break;
            }
            TC_CTA(3);
            // h was written with generic stores; the copies read it through the async proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
            if (!ok) set_abort(a, sm);
            h_done = true;
        }
        uint8_t* stg = sm.stage[s];
        bulk_g2s(stg + kOffB, q.B, q.nb, &sm.full[s]);
        bulk_g2s(stg + kOffSfb, q.Bsf, q.nsf, &sm.full[s]);
    }
    if (!published && !publish_own_groups(a, sm, owned)) set_abort(a, sm);
}

// ------------------------------------------------------------------ MMA issue

struct IssState {
    int n, buf;
    uint32_t use[2];
    bool abort;
};

// Issuer ii takes unit ii of every stage into its own accumulator.
template <int PHASE>
__device__ void issue(const GemvArgs& a, const StreamPlan& p, const Range& r, TcSmem& sm, uint32_t tmem, int ii,
                      IssState& is)
{
    const uint32_t idesc = mxf4_idesc(kTileRows, kBRows);
    Walk wk(p, r);
    const uint32_t kgt = wk.kgt;
    bool ok = job_at<PHASE>(a, p, r, sm, wk.job).ok;
    bool any = false;               // this issuer wrote its accumulator in this group
    bool group_start = true;
    while (wk.u < wk.u1) {
        const uint32_t nun = wk.chunk();
        const int s = is.n % kStages;
        if (group_start) {
            // the epilogue must have read this accumulator's previous group
            if (!is.abort && is.use[is.buf] > 0 &&
                !mbar_wait_or_abort(&sm.acc_empty[is.buf], (is.use[is.buf] - 1) & 1, &sm.abort, wait_limit(a))) {
                set_abort(a, sm);
                is.abort = true;
            }
            group_start = false;
        }
        if (!is.abort && !mbar_wait_or_abort(&sm.full[s], (is.n / kStages) & 1, &sm.abort, wait_limit(a))) {
            set_abort(a, sm);
            is.abort = true;
        }
        if (ii == 0) TC_TRACE(PHASE, 1, is.n);
        if (!is.abort && ok && (uint32_t)ii < nun) {
            tc_fence_after();
            const uint8_t* st = sm.stage[s];
            const uint32_t col = tmem + kSfCol0 + (uint32_t)(s * kCU + ii) * 8;
            const bool half = p.kg_half && (wk.kg + (uint32_t)ii == kgt - 1);
            const uint8_t* unit = st + ii * kUnitBytes;            // codes, then the scale atom
            tc_cp_sf(col, umma_desc(smem_u32(unit + (half ? kMmaCodeBytes : kUnitCodeBytes)), 16, 128));
            tc_cp_sf(col + 4, umma_desc(smem_u32(st + kOffSfb + ii * kUnitSfBytes), 16, 128));
            for (int m = 0; m < (half ? 1 : 2); m++) {
                const uint64_t ad = umma_desc(smem_u32(unit + m * kMmaCodeBytes), 128, 256);
                const uint64_t bd = umma_desc(smem_u32(st + kOffB + ii * kUnitBBytes + m * kMmaBBytes), 128, 256);
                tc_mma_mxf4(tmem + (uint32_t)(ii * 2 + is.buf) * kAccCols, ad, bd, mxf4_idesc_sf(idesc, 2 * m), col,
                            col + 4, any ? 1u : 0u);
                any = true;
            }
        }
        tc_commit(&sm.empty[s]);           // this issuer's part of the stage is consumed
        if (ii == 0) TC_TRACE(PHASE, 2, is.n);
        bool nj;
        const bool gend = wk.advance(nun, nj);
        is.n++;
        if (nj && wk.u < wk.u1) ok = job_at<PHASE>(a, p, r, sm, wk.job).ok;
        if (gend) {
            tc_commit(&sm.acc_full[is.buf]);   // this issuer's accumulator is final
            is.use[is.buf]++;
            is.buf ^= 1;
            any = false;
            group_start = true;
        }
    }
}

// ------------------------------------------------------------------ epilogue

__device__ __forceinline__ float slot_weight(const GemvArgs& a, const TcSmem& sm, int j)
{
    if (j < kSlotCache) return sm.slot_w[j];
    const int e = a.idx[j];
    return (e >= 0 && e < a.E) ? a.w[j] : 0.0f;
}

// Gate/up group (slot j, tile) -> the 64 values h = w_j * silu(g) * u, as
// pieces, by one warp; then the group goes to the loader thread, which adds it
// to the grid-wide count.
__device__ __forceinline__ void fin_signal(TcSmem& sm, int lane, uint32_t done)
{
    if (lane == 0)
        asm volatile("red.release.cta.shared::cta.add.u64 [%0], %1;" ::"r"(smem_u32(&sm.fin_word)),
                     "l"((1ull << 32) | (unsigned long long)done)
                     : "memory");
}

template <int MODE>
__device__ __forceinline__ void finalize_gate_up(const GemvArgs& a, const StreamPlan& p, TcSmem& sm,
                                                 uint32_t group, const float* comb, int lane, int tr_warp)
{
    const int j = (int)(group / p.ntiles), tile = (int)(group % p.ntiles);
    TC_FIN(0, group % 64);
    if (lane == 0) TC_CTA(8);
    if (lane == 0) TC_GRP(3, group);
    const float w = slot_weight(a, sm, j);
    const float2 g = *reinterpret_cast<const float2*>(comb + 2 * lane);
    const float2 u = *reinterpret_cast<const float2*>(comb + 64 + 2 * lane);
    float h0 = silu(g.x) * u.x, h1 = silu(g.y) * u.y;
    int done = 1;                         // tiles of h whose pieces this call writes
    if (MODE == kModeE2m1) {                     // h quantized to E2M1 per 32 along I, before w
        const float2 q = e2m1_block_quant_dequant(h0, h1);
        h0 = q.x;
        h1 = q.y;
    }
    if (MODE == kModeE4m3) {
        // h is quantized to E4M3 per 128 along I (tiles 2b, 2b + 1; a last block
        // of 64 is one tile), before w.  The second tile of a block to finish
        // quantizes both, from the first one's raw h.
        const int blk = tile / 2, nblk = (p.ntiles + 1) / 2;
        const bool pair = (tile | 1) < p.ntiles;
        float o0 = 0.0f, o1 = 0.0f;
        if (pair) {
            float* mine = a.hraw + (size_t)j * a.I + (size_t)tile * 64 + 2 * lane;
            mine[0] = h0;
            mine[1] = h1;
            __threadfence();
            __syncwarp();
            int old = 0;
            if (lane == 0) old = atomicAdd(a.hpair + (size_t)j * nblk + blk, 1);
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == 0) {               // the other tile finishes the block
                fin_signal(sm, lane, 0);
                return;
            }
            __threadfence();
            const float* other = a.hraw + (size_t)j * a.I + (size_t)(tile ^ 1) * 64 + 2 * lane;
            o0 = __ldcg(other);
            o1 = __ldcg(other + 1);
            if (lane == 0) a.hpair[(size_t)j * nblk + blk] = 0;     // ready for the next launch
            done = 2;
        }
        const float amax = warp_max(fmaxf(fmaxf(fabsf(h0), fabsf(h1)), fmaxf(fabsf(o0), fabsf(o1))));
        const int s = ue8m0_for_amax_bits(amax);
        h0 = e4m3_quant_dequant(h0, s);
        h1 = e4m3_quant_dequant(h1, s);
        if (pair) {
            const int ot = tile ^ 1;
            uint8_t* Bunit = a.hq + (size_t)j * act_bytes(a.I) + (size_t)(ot / 2) * kUnitBBytes;
            uint8_t* Bsf = a.hsf + (size_t)j * act_sf_bytes(a.I) + (size_t)(ot / 2) * kUnitSfBytes;
            write_pieces64_small(e4m3_quant_dequant(o0, s) * w, e4m3_quant_dequant(o1, s) * w, lane, Bunit, Bsf, 2 * ot,
                           sm.tr[tr_warp]);
        }
    }
    uint8_t* Bunit = a.hq + (size_t)j * act_bytes(a.I) + (size_t)(tile / 2) * kUnitBBytes;
    uint8_t* Bsf = a.hsf + (size_t)j * act_sf_bytes(a.I) + (size_t)(tile / 2) * kUnitSfBytes;
    write_pieces64_small(h0 * w, h1 * w, lane, Bunit, Bsf, 2 * tile, sm.tr[tr_warp]);
    TC_FIN(1, group % 64);
    // the down projection reads these with bulk copies (async proxy), in other CTAs
    asm volatile("fence.proxy.async.global;" ::: "memory");
    TC_FIN(2, group % 64);
    __syncwarp();
    // the pieces (this warp's stores, ordered by the warp barrier) go to the
    // loader thread with a CTA-scope release; its GPU-scope release of the
    // count covers them, and this warp goes back to the epilogue at once
    fin_signal(sm, lane, (uint32_t)done);
    TC_FIN(3, group % 64);
    if (lane == 0) TC_CTA(9);
    if (lane == 0) TC_GRP(4, group);
}

struct EpiState {
    int buf, cb;
    uint32_t use[2];
    uint32_t tag;               // this launch's tag of the partial sums
};

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Partial sums of a split group from the CTAs after its owner, added in CTA
// order into *acc; returns the first CTA not yet folded in.  With spin, waits
// (bounded) for each; without, stops at the first that is not there yet.
__device__ __forceinline__ int fold_partials(const uint64_t* part, int c, int c1, int row, uint32_t tag,
                                             bool spin, float* acc, bool* timed_out, uint64_t limit)
{
    uint64_t t0 = 0;
    while (c <= c1) {
        const uint64_t e = ld_relaxed_u64(part + (size_t)c * kTileRows + row);
        if ((uint32_t)(e >> 32) == tag) {
            *acc += __uint_as_float((uint32_t)e);
            c++;
            continue;
        }
        if (!spin) break;
        if (t0 == 0) t0 = wait_clock();
        else if (wait_clock() - t0 > wait_cycles(limit)) {
            *timed_out = true;
            break;
        }
    }
    return c;
}

template <int PHASE, int MODE>
__device__ void epilogue(const GemvArgs& a, const StreamPlan& p, const Range& r, TcSmem& sm, uint32_t tmem,
                         int quad, int lane, int et, EpiState& es)
{
    uint64_t* part = PHASE == 0 ? a.part_gu : a.part_dn;
    const int row = quad * 32 + lane;                      // accumulator row of this thread
    const uint32_t gunits = (uint32_t)p.kgt * (uint32_t)p.jobs_per_group;
    Walk wk(p, r);
    uint32_t mask = 0;                                     // issuers that accumulated into this group
    bool cur_ok = job_at<PHASE>(a, p, r, sm, wk.job).ok;
    while (wk.u < wk.u1) {
        bool nj;
        const uint32_t group = wk.group;
        const uint32_t nun = wk.chunk();
        if (cur_ok) mask |= (1u << nun) - 1u;
        const bool gend = wk.advance(nun, nj);
        if (nj && wk.u < wk.u1) cur_ok = job_at<PHASE>(a, p, r, sm, wk.job).ok;
        if (!gend) continue;

        // ------------------------------------------- end of a reduction group
        // A group split over CTAs c0..c1 is finished by c0, the CTA holding its
        // first unit, which reaches it last (at the end of its range); the others
        // leave their sums, tagged with the launch, in their partial vector.
        const long long gs = (long long)group * gunits, ge = gs + gunits;
        const bool owner = gs >= r.u0;
        const int c1 = owner && ge > r.u1 ? cta_of_unit(p, ge - 1) : (int)blockIdx.x;
        float pacc = 0.0f;
        bool late = false;
        int cnext = blockIdx.x + 1;
        if (c1 > (int)blockIdx.x)   // while the last MMAs run: the partials that are there already
            cnext = fold_partials(part, cnext, c1, row, es.tag, false, &pacc, &late, wait_limit(a));

        const int buf = es.buf;
        const bool ready = !*(volatile int*)&sm.abort &&
                           mbar_wait_or_abort(&sm.acc_full[buf], es.use[buf] & 1, &sm.abort, wait_limit(a));
        if (et == 0) TC_TRACE(PHASE, 3, es.use[0] + es.use[1]);
        if (PHASE == 0 && et == 0) TC_CTA(10);
        if (PHASE == 0 && et == 0 && owner) TC_GRP(0, group);
        es.use[buf]++;
        if (!ready) set_abort(a, sm);
        tc_fence_after();
        float v = 0.0f;
        if (ready) {
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
        es.buf ^= 1;

        if (!owner) {
            // a later part of a group owned by an earlier CTA
            st_relaxed_u64(part + (size_t)blockIdx.x * kTileRows + row,
                           ((uint64_t)es.tag << 32) | __float_as_uint(v));
            continue;
        }
        if (cnext <= c1) {
            const bool abort = *(volatile int*)&sm.abort;
            fold_partials(part, cnext, c1, row, es.tag, !abort, &pacc, &late, wait_limit(a));
            if (late) set_abort(a, sm);
        }
        if (PHASE == 0 && et == 0) TC_CTA(11);
        if (PHASE == 0 && et == 0) TC_GRP(1, group);
        v += pacc;
        if (PHASE == 0) {
            // the owned groups' h go to the four epilogue warps in turn: the
            // others only arrive at the group's barrier, so one warp's finalize
            // overlaps the next groups' accumulator reads and finalizes.  Buffer
            // and barrier cb are reused four groups later, when that warp has
            // long finished (the issuers cannot pass it by more than the two
            // accumulator buffers).
            float* comb = sm.comb[es.cb];
            comb[row] = v;
            if (quad == es.cb) {
                named_sync(3 + es.cb, 128);
                if (lane == 0) TC_GRP(2, group);
                finalize_gate_up<MODE>(a, p, sm, group, comb, lane, quad);
            } else {
                named_arrive(3 + es.cb, 128);
            }
            es.cb = (es.cb + 1) & 3;
        } else {
            // group = (token t, tile): 128 output rows, one per thread
            const int t = (int)(group / p.ntiles), tile = (int)(group % p.ntiles);
            const size_t o = (size_t)t * a.H + (size_t)tile * kTileRows + row;
            if (a.x_resid) {
                const float xn = a.x_resid[o] + v;
                a.x_resid[o] = xn;
                // the next layer's RMSNorm: this warp's 32 rows' sum of squares
                const float ss = warp_sum(__fmul_rn(xn, xn));
                if (lane == 0) a.ssq[(size_t)t * (a.H / 32) + tile * 4 + quad] = ss;
            } else if (a.out_f32) reinterpret_cast<float*>(a.y)[o] = v;
            else reinterpret_cast<__nv_bfloat16*>(a.y)[o] = __float2bfloat16_rn(v);
        }
    }
}

// ------------------------------------------------------------------ kernel

// One MoE layer: the gate/up projection then the down projection, in one
// persistent grid.  The producer streams the down weights right after the
// gate/up weights; only the copies of h wait until the last h piece is
// written.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) k_layer(GemvArgs a, StreamPlan p0, StreamPlan p1)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) TC_CTA(7);
    const Range r0 = cta_range(p0), r1 = cta_range(p1);
    const uint32_t gu_groups = (uint32_t)(p0.U / ((long long)p0.kgt * p0.jobs_per_group));

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kIssuers);
            mbar_init(&sm.posted[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&sm.acc_full[b], kIssuers);
            mbar_init(&sm.acc_empty[b], 4);
        }
        for (int i = 0; i < kIssuers; i++) mbar_init(&sm.drain[i], 1);
        sm.abort = 0;
        sm.fin_word = 0;
        mbar_fence_init();
    }
    // a caller whose routing comes from a kernel that releases its dependents
    // early asks for the routing to be read after the dependency wait
    if (a.routing_after_wait) pdl_wait();
    if (warp == 0) {
        // resolve the CTA's first jobs of both projections (expert pointers), one
        // per lane and projection, the two projections' loads in flight together
        const bool h0 = r0.j0 + lane <= r0.jlast && lane < kJobWindow;
        const bool h1 = r1.j0 + lane <= r1.jlast && lane < kJobWindow;
        int j0 = 0, t0 = 0, j1 = 0, t1 = 0;
        if (h0) job_slot<0>(a, p0, r0.j0 + lane, j0, t0);
        if (h1) job_slot<1>(a, p1, r1.j0 + lane, j1, t1);
        const int e0 = h0 ? a.idx[j0] : -1, e1 = h1 ? a.idx[j1] : -1;
        const bool in0 = e0 >= 0 && e0 < a.E, in1 = e1 >= 0 && e1 < a.E;
        const uint8_t* b0 = in0 ? a.experts[e0] : nullptr;
        const uint8_t* b1 = in1 ? a.experts[e1] : nullptr;
        if (h0) {
            const JobInfo ji = job_info_e<0>(a, p0, j0, t0, e0, b0);
            sm.jobs[0][lane] = ji;
            if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
        }
        if (h1) {
            const JobInfo ji = job_info_e<1>(a, p1, j1, t1, e1, b1);
            sm.jobs[1][lane] = ji;
            if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
        }
    } else {
        // routing weights of the slots: inputs of the call, complete before its
        // first kernel may start (their producers let dependents launch only at
        // completion), so they are read before griddepcontrol.wait
        const int slots = min(a.T * a.topk, kSlotCache);
        for (int j = threadIdx.x - 32; j < slots; j += kThreads - 32) {
            const int e = a.idx[j];
            sm.slot_w[j] = (e >= 0 && e < a.E) ? a.w[j] : 0.0f;
        }
    }
    if (warp == 1) tmem_alloc(&sm.tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = sm.tmem;
    if (threadIdx.x == 0) TC_CTA(0);

    if (warp == 0) {
        if (lane == 0) {
            int n = 0;
            const bool ok = produce<0>(a, p0, r0, sm, n);
            TC_CTA(2);
            // the down weights follow at once into the ring; nothing more is
            // prefetched, so that the gate/up tail and the h hand-off (the
            // critical path) do not queue behind them in the memory system
            if (ok) produce<1>(a, p1, r1, sm, n);
            // no copy may still be in flight into this CTA's memory at exit
            for (int m = n > kStages ? n - kStages : 0; m < n; m++)
                mbar_wait_bounded(&sm.full[m % kStages], (m / kStages) & 1, wait_limit(a));
        }
        return;
    }
    if (warp == kWarpLoader) {
        // gate/up groups whose first unit is in this CTA's range: it finalizes them
        const uint32_t owned = (r0.u1 + p0.kgt - 1) / (uint32_t)p0.kgt - (r0.u0 + p0.kgt - 1) / (uint32_t)p0.kgt;
        if (lane == 0) load_b(a, count_chunks(p0, r0) + count_chunks(p1, r1), gu_groups, owned, sm);
        return;
    }
    if (warp < kWarpEpi0) {
        if (lane == 0) {
            IssState is;
            is.n = 0;
            is.buf = 0;
            is.use[0] = is.use[1] = 0;
            is.abort = false;
            issue<0>(a, p0, r0, sm, tmem, warp - 1, is);
            if (warp == 1) TC_CTA(4);
            issue<1>(a, p1, r1, sm, tmem, warp - 1, is);
            // none of this thread's MMAs may be in flight when TMEM is freed (after
            // an abort the epilogue no longer waits for the accumulators)
            tc_commit(&sm.drain[warp - 1]);
            mbar_wait_bounded(&sm.drain[warp - 1], 0, wait_limit(a));
        }
        __syncwarp();
    } else {
        pdl_wait();
        const int et = threadIdx.x - kWarpEpi0 * 32;     // 0..127 among the epilogue threads
        EpiState es;
        es.buf = 0;
        es.cb = 0;
        es.use[0] = es.use[1] = 0;
        es.tag = 1u + (ld_acquire_u32(a.sync + 2) & 0x3FFFFFFFu);   // never 0, the cleared value
        epilogue<0, MODE>(a, p0, r0, sm, tmem, warp & 3, lane, et, es);
        if (et == 0) TC_CTA(5);
        epilogue<1, MODE>(a, p1, r1, sm, tmem, warp & 3, lane, et, es);
        if (et == 0) TC_CTA(6);
        if (et == 0) {
            // the last CTA to finish resets the layer's counters for the next launch
            __threadfence();
            const int done = atomicAdd(a.sync + 1, 1);
            if (done == (int)gridDim.x - 1) {
                a.sync[0] = 0;
                a.sync[1] = 0;
                a.sync[2] += 1;      // the next launch tags its partial sums differently
                __threadfence();
            }
        }
    }
    // the issuer and epilogue warps meet here before the tensor memory is released
    tc_fence_before();
    named_sync(2, (kIssuers + 4) * 32);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    if (threadIdx.x == 32) TC_CTA(1);
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

StreamPlan make_plan(const GemvArgs& a, int phase)
{
    StreamPlan p{};
    ExpertLayout E = make_expert_layout(a.H, a.I);
    const MatLayout& L = phase == 0 ? E.gu : E.dn;
    p.kgt = L.kgt();
    p.kg_half = L.kg_half;
    p.ntiles = L.tiles;
    p.tile_bytes = L.tile_bytes();
    if (phase == 0) {
        p.U = (long long)a.T * a.topk * L.tiles * p.kgt;
        p.jobs_per_group = 1;
        p.off = E.gu_off;
        p.act_bytes = act_bytes(a.H);
        p.act_sf_bytes = act_sf_bytes(a.H);
    } else {
        p.U = (long long)a.T * L.tiles * a.topk * p.kgt;
        p.jobs_per_group = a.topk;
        p.off = E.dn_off;
        p.act_bytes = act_bytes(a.I);
        p.act_sf_bytes = act_sf_bytes(a.I);
    }
    return p;
}

size_t layer_smem() { return sizeof(TcSmem) > kOneCtaPerSmSmem ? sizeof(TcSmem) : kOneCtaPerSmSmem; }

}  // namespace

GemvWorkspaceSizes gemv_workspace_sizes(int T, int topk, int H, int I, int sms, bool e4m3)
{
    GemvWorkspaceSizes s;
    const size_t slots = (size_t)T * topk;
    s.xq = (size_t)T * act_bytes(H);
    s.xsf = (size_t)T * act_sf_bytes(H);
    s.hq = slots * act_bytes(I);
    s.hsf = slots * act_sf_bytes(I);
    s.part_gu = (size_t)sms * kTileRows;
    s.part_dn = (size_t)sms * kTileRows;
    s.hraw = e4m3 ? slots * I * sizeof(float) : 0;
    s.hpair = e4m3 ? slots * (size_t)((I + 127) / 128) * sizeof(int) : 0;
    s.ssq = (size_t)T * (H / 32) * sizeof(float);
    return s;
}

cudaError_t gemv_init_device()
{
    cudaError_t e = cudaSuccess;
    for (const void* fn : {(const void*)k_layer<kModeBf16>, (const void*)k_layer<kModeE4m3>,
                           (const void*)k_layer<kModeE2m1>})
        if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)layer_smem());
    // k_prep asks for the same shared-memory carveout as k_layer, so that the
    // SMs need no reconfiguration between the two kernels of a layer
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute((const void*)k_prep, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    return e;
}

size_t gemv_stream_smem() { return layer_smem(); }

cudaError_t launch_gemv_layer(const GemvArgs& a0, cudaStream_t s, bool pdl, Profiler* prof)
{
    GemvArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    cudaError_t err;
    if (!a.skip_prep) {
        void* args[] = {&a};
        if (prof) prof->begin(kPhasePrep, s);
        const int spans = a.act_e4m3 ? a.H / 128 : a.H / 64;      // one warp each
        err = launch_ex((const void*)k_prep, dim3(a.T, (spans + 7) / 8), dim3(256), 0, s, pdl && !prof, args);
        if (prof) prof->end(s);
        if (err != cudaSuccess) return err;
    }
    StreamPlan p0 = make_plan(a, 0), p1 = make_plan(a, 1);
    long long G = a.sms;
    if (p0.U < G) G = p0.U;
    if (p1.U < G) G = p1.U;
    p0.G = p1.G = (int)G;     // every CTA has units of both projections
    void* args[] = {&a, &p0, &p1};
    if (prof) prof->begin(kPhaseGateUp, s);
    const void* fn = a.act_e4m3 ? (const void*)k_layer<kModeE4m3>
                     : a.act_e2m1 ? (const void*)k_layer<kModeE2m1> : (const void*)k_layer<kModeBf16>;
    err = launch_ex(fn, dim3((unsigned)G), dim3(kThreads), layer_smem(), s, pdl && !prof, args);
    if (prof) prof->end(s);
    return err;
}

}  // namespace moe

#ifdef MOE_TC_TRACE
// debug builds only: the per-CTA milestones of the last layer launch (ns,
// globaltimer), cleared after the read
extern "C" int moe_debug_layer_trace(long long* dst, size_t bytes)
{
    const size_t n = bytes < sizeof(moe::g_tc_cta) ? bytes : sizeof(moe::g_tc_cta);
    if (cudaMemcpyFromSymbol(dst, moe::g_tc_cta, n) != cudaSuccess) return 1;
    static long long zero[12][1024];
    return cudaMemcpyToSymbol(moe::g_tc_cta, zero, sizeof(zero)) == cudaSuccess ? 0 : 1;
}
#endif
