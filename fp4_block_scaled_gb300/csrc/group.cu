// group.cu -- expert-major ("grouped") path of one routed FP4 MoE layer, for
// decode batches in which tokens share experts.
//
// Four launches per layer, chained with programmatic dependent launch (PDL):
//   k_route    (route.cu) stable counting sort of the T*k slots by expert and
//              the group table: each expert's sorted slots are cut into groups
//              of up to S slots (S = 8 in the E4M3 mode, 4 in the bf16 mode);
//   k_gprep    x (bf16, or RMSNorm of the fp32 residual; in the E4M3 mode
//              quantized per 128 first) -> P E2M1 pieces per element (P = 8
//              in the E4M3 mode, 16 in the bf16 mode; see below), written once
//              per slot into its group's B operand;
//   k_glayer   both projections in one persistent grid, one CTA per SM.  A job
//              is (group, tile): 128 weight rows against the group's nt slots,
//              block-scaled MMAs (kind::mxf4, M = 128, N = P nt <= 64, K = 64),
//              the nt slots' pieces being the N columns.  Jobs are ordered
//              (expert, tile, group), so a weight tile leaves HBM once per
//              expert and its further groups re-read it from L2 right away;
//   k_gcombine y[t] = sum_k o[t, k] over the token's slots in k order (or
//              x += that on a residual stream).
//
// Pieces: v is carried as P E2M1 vectors with one ue8m0 scale per (piece,
// 32-block), p_0 at the least scale 2^e0 with max|v| <= 6 2^e0, each next
// piece encoding the remainder 4x finer, so an element is carried to within
// 2^(e0 - 2P + 2): 2^-30 of the block scale 2^e0 for P = 16, 2^-14 for P = 8
// (the E4M3 values have 4 significant bits; those within 2^10 of the block's
// largest are carried exactly).
//
// B operand layout (group order): a slot at sorted position P keeps its pieces
// at P * pb(K), pb(K) = 64 P bytes per 128-K unit (32 P for a last half unit);
// a group's slots are consecutive positions, and inside the group, unit u of
// K holds, per MMA m, the nt slots' (32 P)-byte piece blocks side by side --
// byte offset  u nt 64P + m nt 32P + i 32P  for slot i -- so the B rows of one
// MMA (P per slot) are one contiguous run with 256-byte row-group stride, and
// a run of units of one group is one contiguous copy.  Scale atoms are per
// (group, unit): 512 bytes in the order tcgen05.cp moves them, row n = P i + p
// (slot i, piece p) at byte (n % 32) * 16 + (n / 32) * 4 + block.
//
// Roles of k_glayer (as in the slot-major layer kernel of gemv.cu): a weight
// producer thread fills a ring of shared-memory stages (kGCU units each) with
// cp.async.bulk; an activation loader thread fills a second, shallower ring
// with the matching pieces; three MMA-issuing warps (one thread each issues at
// most one tcgen05 instruction per ~150 cycles, several overlap) take one unit
// of each stage into their own double-buffered accumulators; four epilogue
// warps read them with tcgen05.ld, add the P piece columns of each slot and
// the issuers in a fixed order, and finish a job: gate/up -> h = w silu(g) u
// as pieces into the down projection's B operand; down -> o of each slot.  A
// job split over several CTAs is finished by the CTA holding its first unit,
// which adds the others' launch-tagged partial sums in CTA order, so results
// are bitwise reproducible.  Every wait is bounded (2 s); on expiry the kernel
// records the device-timeout status, stops issuing, waits (bounded) for its
// copies in flight and frees its TMEM.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kNT = kGroupTokens;                            // slots per group, at most (shared memory, partials)
constexpr int kGIssuers = 3;
constexpr int kGCU = kGIssuers;                              // units per stage: one per issuer
constexpr int kGStagesA = 5;                                 // weights (HBM): the deep ring
constexpr int kGStagesB = 4;                                 // pieces (L2, issued later)
constexpr int kGUnitB = 2 * kGroupN * 32;                    // B bytes of a unit at N = 64
constexpr int kGStageA = 26 * 1024;                          // kGCU units of weights (codes + scale atom each)
constexpr int kGOffSfb = kGCU * kGUnitB;                     // 12 KB of pieces, then their scale atoms
constexpr int kGStageB = 14 * 1024;
constexpr int kGTmemCols = 512;
constexpr int kGAccCols = kGroupN;                           // 64 fp32 columns per accumulator
constexpr int kGSfCol0 = kGIssuers * 2 * kGAccCols;          // scale atoms after the accumulators
constexpr uint64_t kGWaitLimitNs = 2000000000ull;
constexpr int kGWarpEpi0 = 1 + kGIssuers;                    // epilogue warps 4..7
constexpr int kGWarpLoader = kGWarpEpi0 + 4;
constexpr int kGThreads = (kGWarpLoader + 1) * 32;

#ifdef MOE_G_TRACE
// debug builds only: event timestamps of one CTA ([role][idx], ns) and per-CTA milestones
}  // namespace
__device__ long long g_gtrace[4][8192];
__device__ long long g_gcta[16][1024];
__device__ int g_gtrace_cta;
namespace {
#define G_TRACE(role, idx)                                                                               \
    do {                                                                                                 \
        if ((int)blockIdx.x == g_gtrace_cta && (idx) < 8192) g_gtrace[role][idx] = (long long)globaltimer_ns(); \
    } while (0)
#define G_CTA(slot) (g_gcta[slot][blockIdx.x] = (long long)globaltimer_ns())
#define G_ACC(var, t0) ((var) += globaltimer_ns() - (t0))
#define G_ADD(slot, var) (g_gcta[slot][blockIdx.x] += (long long)(var))
#define G_NOW() globaltimer_ns()
#else
#define G_TRACE(role, idx) \
    do {                   \
    } while (0)
#define G_CTA(slot) \
    do {            \
    } while (0)
#define G_ACC(var, t0) \
    do {               \
    } while (0)
#define G_ADD(slot, var) \
    do {                 \
    } while (0)
#define G_NOW() 0ull
#endif

static_assert(kGCU * kUnitBytes <= kGStageA && kGOffSfb + kGCU * kUnitSfBytes <= kGStageB, "stage sizes");
static_assert(kGStageA % 1024 == 0 && kGStageB % 1024 == 0, "stage alignment");
static_assert(kGSfCol0 + kGStagesA * kGCU * 8 <= kGTmemCols, "tensor memory budget");
static_assert(kGStagesB <= kGStagesA, "the activation ring is the shallower one");
static_assert(kGroupN % 16 == 0 && kGroupN <= 256, "MMA N");
// CTAs of k_glayer wait on one another (the down projection needs every h):
// two must never share an SM, so the shared memory asked for is more than
// half of an SM's.
constexpr size_t kGOneCtaPerSmSmem = 116 * 1024;

struct GJob {
    const uint8_t* w;       // weight tile, unit 0 (codes + scale atom per unit)
    const uint8_t* B;       // the group's pieces, unit 0
    const uint8_t* Bsf;     // the group's scale atoms, unit 0
    int nt, p0, tile, g;    // slots, first sorted position, weight tile, group
    bool ok;
};

struct GBSrc {
    const uint8_t* B;       // nullptr: the stage multiplies nothing
    const uint8_t* Bsf;
    uint32_t nb, nsf;
    int phase;
};

struct GSmem {
    uint8_t stageA[kGStagesA][kGStageA];
    uint8_t stageB[kGStagesB][kGStageB];
    uint64_t fullA[kGStagesA];   // the stage's weights landed
    uint64_t emptyA[kGStagesA];  // the issuers are done with them
    uint64_t posted[kGStagesA];  // the producer issued them and posted bsrc
    uint64_t fullB[kGStagesB];   // the stage's pieces landed (the slot is free again once
                                 // the weight stage of the chunk it held is empty)
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain[kGIssuers];
    GBSrc bsrc[kGStagesA];
    float comb[2][kNT][kTileRows];
    float hstash[kNT][64];       // raw h of the first tile of a pair, per slot
    uint4 tr[4][32];             // per epilogue warp: the pieces' byte transpose
    uint32_t tmem;
    int abort;
};
static_assert(sizeof(GSmem) <= 227 * 1024, "shared memory per CTA");

// One projection's unit stream (host part; the job count is read on the device).
struct GPlan {
    int kgt, kg_half, ntiles;
    size_t off, tile_bytes; // the matrix in the expert blob, one tile
    size_t act_bytes;       // piece bytes of one slot over K
    int gs, np;             // slots per group (at most), pieces per slot
    int phase;
};

// Piece bytes of one slot over K with P pieces: 64 P per 128-K unit, 32 P for
// a last half unit.
__host__ __device__ inline size_t g_act_bytes(int K, int P)
{
    return (size_t)(K / 128) * 64 * P + (size_t)((K % 128) ? 32 * P : 0);
}

// B bytes of one 128-K unit of a group of nt slots of P pieces: per MMA
// (K = 64) whole 8-row groups of 256 bytes, P nt rows (64 P nt bytes when 8
// divides P; one row group for the one-piece E2M1 mode).
__host__ __device__ inline uint32_t g_unit_b(int P, int nt) { return (uint32_t)((P * nt + 7) / 8) * 512u; }

// The pieces of a group (first sorted position p0, group g; pact = piece
// bytes of one slot over K): slot-proportional when 8 divides P, else a region
// per group sized for a full group (its units are whole 8-row groups), which
// is at most the 16-piece bytes of a slot, so the buffers sized per slot hold
// it (there are no more groups than slots).
__host__ __device__ inline uint8_t* g_group_b(uint8_t* base, int P, int p0, int g, size_t pact)
{
    const int S = kGroupN / P < kGroupTokens ? kGroupN / P : kGroupTokens;
    return P >= 8 ? base + (size_t)p0 * pact : base + (size_t)g * pact * S;
}

// ----------------------------------------------------------------- pieces

// P pieces of 64 consecutive elements (32-blocks blk0, blk0 + 1 of a unit;
// lane l holds elements 2l, 2l + 1), computed once: byte[p] = the lane's E2M1
// pair of piece p, sc[p] = the piece's scale byte.  The first scale is the
// least e with max|v| <= 6 * 2^e over the 32-block (a half-warp), each next
// piece encodes the remainder 4x finer; the remainders are exact in fp32.
template <int P>
struct Pieces64 {
    uint8_t byte[P];
    uint8_t sc[P];
};

template <int P>
__device__ __forceinline__ void make_pieces64(float v0, float v1, Pieces64<P>& pc)
{
    float amax = fmaxf(fabsf(v0), fabsf(v1));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int s0 = e2m1_scale_byte(amax);
    float r0 = v0, r1 = v1;
#pragma unroll
    for (int p = 0; p < P; p++) {
        const int s = max(s0 - 2 * p, 1);
        const float down = exp2i(127 - s), up = exp2i(s - 127);
        const uint32_t byte = f32x2_to_e2m1x2(r0 * down, r1 * down);
        const float2 d = e2m1x2_to_f32x2(byte);
        r0 = fmaf(-d.x, up, r0);
        r1 = fmaf(-d.y, up, r1);
        pc.byte[p] = (uint8_t)byte;
        pc.sc[p] = (uint8_t)s;
    }
}

// Stores the pieces of slot i of a group: unit points at the group's unit
// (codes), mstride = nt * 32P (distance between the unit's two MMAs), atom =
// the group's scale atom of that unit; blk0 = the span's first 32-block
// within the unit (0 or 2).  Rows n = P i + p: row group n / 8, row n % 8 of
// a core matrix (16 bytes = one 32-block of two-element bytes).
template <int P>
__device__ __forceinline__ void store_pieces64(const Pieces64<P>& pc, int lane, uint8_t* unit, int mstride,
                                               uint8_t* atom, int i, int blk0)
{
    const int bu = blk0 + (lane >> 4);             // 32-block within the unit
    const int ib = lane & 15;                      // byte within the block's row
    uint8_t* rows = unit + (bu >> 1) * mstride + (bu & 1) * 128 + ib;
#pragma unroll
    for (int p = 0; p < P; p++) {
        const int n = P * i + p;
        rows[(n >> 3) * 256 + (n & 7) * 16] = pc.byte[p];
    }
    if (ib == 0) {
#pragma unroll
        for (int p = 0; p < P; p++) {
            const int n = P * i + p;
            atom[(n & 31) * 16 + (n >> 5) * 4 + bu] = pc.sc[p];
        }
    }
}

// A lane's share of its half-warp's pieces after a transpose through shared
// memory (P = 8 or 16): with 16 pieces row ib (16 bytes: piece ib of the
// half-warp's 16 lanes), with 8 half `ib % 2` of row ib / 2 (8 bytes).
template <int P>
struct PieceRow {
    uint32_t w[P / 4];
    int s0;                 // the first piece's scale byte
};

template <int P>
__device__ __forceinline__ PieceRow<P> transpose_pieces(const Pieces64<P>& pc, int lane, uint4* scratch)
{
    static_assert(P == 8 || P == 16, "row transpose for 8 or 16 pieces");
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int p = 0; p < P; p++) w[p >> 2] |= (uint32_t)pc.byte[p] << (8 * (p & 3));
    scratch[lane] = make_uint4(w[0], w[1], w[2], w[3]);
    __syncwarp();
    const uint8_t* sb = reinterpret_cast<const uint8_t*>(scratch + (lane & 16));
    const int ib = lane & 15;
    const int p = P == 16 ? ib : ib >> 1, k0 = P == 16 ? 0 : 8 * (ib & 1);
    PieceRow<P> r;
#pragma unroll
    for (int q = 0; q < P / 4; q++)
        r.w[q] = (uint32_t)sb[(k0 + 4 * q) * 16 + p] | ((uint32_t)sb[(k0 + 4 * q + 1) * 16 + p] << 8) |
                 ((uint32_t)sb[(k0 + 4 * q + 2) * 16 + p] << 16) | ((uint32_t)sb[(k0 + 4 * q + 3) * 16 + p] << 24);
    r.s0 = pc.sc[0];
    __syncwarp();
    return r;
}

// The transposed pieces of slot i of a group (as store_pieces64): one 16- or
// 8-byte store and at most one scale byte per lane.
template <int P>
__device__ __forceinline__ void store_piece_rows(const PieceRow<P>& r, int lane, uint8_t* unit, int mstride,
                                                 uint8_t* atom, int i, int blk0)
{
    const int bu = blk0 + (lane >> 4);
    const int ib = lane & 15;
    uint8_t* rows = unit + (bu >> 1) * mstride + (bu & 1) * 128;
    if (P == 16) {
        const int n = 16 * i + ib;
        *reinterpret_cast<uint4*>(rows + (n >> 3) * 256 + (n & 7) * 16) = make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]);
    } else {
        const int n = 8 * i + (ib >> 1);
        *reinterpret_cast<uint2*>(rows + (n >> 3) * 256 + (n & 7) * 16 + 8 * (ib & 1)) = make_uint2(r.w[0], r.w[1]);
    }
    if (ib < P) {
        const int n = P * i + ib;
        atom[(n & 31) * 16 + (n >> 5) * 4 + bu] = (uint8_t)max(r.s0 - 2 * ib, 1);
    }
}

// Where slot position P's pieces of unit u (of a K with kgt units) go, with
// groups of up to S = min(kGroupN / NP, kGroupTokens) slots of NP pieces.
struct GDst {
    uint8_t* unit;
    uint8_t* atom;
    int mstride, i;
};

template <int NP>
__device__ __forceinline__ GDst group_dst(int off, int gbase, int count, int P, int u, int kgt, size_t abytes,
                                          uint8_t* codes, uint8_t* atoms)
{
    constexpr int S = kGroupN / NP < kGroupTokens ? kGroupN / NP : kGroupTokens;
    const int rel = P - off;              // off, gbase, count: the expert's offsets / gbase / counts
    const int q = rel / S;
    const int g = gbase + q;
    const int p0 = off + q * S;
    const int nt = min(S, count - q * S);
    GDst d;
    d.i = rel - q * S;
    d.mstride = (int)g_unit_b(NP, nt) / 2;
    d.unit = g_group_b(codes, NP, p0, g, abytes) + (size_t)u * g_unit_b(NP, nt);
    d.atom = atoms + ((size_t)g * kgt + u) * kUnitSfBytes;
    return d;
}

// ------------------------------------------------------------------ k_gprep

// grid (T, ceil(spans / 8)), 256 threads: one warp per 64 elements (bf16
// mode, 16 pieces) or per 128-element block (E4M3 mode, 8 pieces); the
// pieces are made once and stored for each of the token's slots.
__global__ void __launch_bounds__(256) k_gprep(GroupArgs a)
{
    const int t = blockIdx.x;
    const int H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_red[33];
    __shared__ int s_e[16], s_P[16], s_off[16], s_gb[16], s_cnt[16];
    __shared__ uint4 s_tr[8][32];          // per warp: the pieces' byte transpose

    pdl_wait();
    pdl_trigger();
    if (threadIdx.x < a.topk) {
        // the token's slots: their sorted positions and experts, then each
        // expert's group table entries (two round trips, not one per slot later)
        const int j = t * a.topk + threadIdx.x;
        const int P = a.inv[j];
        const int e = a.idx[j];
        const bool ok = P >= 0 && e >= 0 && e < a.E;
        s_P[threadIdx.x] = ok ? P : -1;
        s_e[threadIdx.x] = ok ? e : -1;
        s_off[threadIdx.x] = ok ? a.offsets[e] : 0;
        s_gb[threadIdx.x] = ok ? a.gbase[e] : 0;
        s_cnt[threadIdx.x] = ok ? a.counts[e] : 0;
    }
    const float den = a.x_resid ? block_rms_den(a.x_resid + (size_t)t * H, H, a.eps, s_red) : 1.0f;
    __syncthreads();
    const int kgt = H / 128;
    auto xval = [&](int i) {
        return a.x_resid ? __bfloat162float(__float2bfloat16_rn(a.x_resid[(size_t)t * H + i] / den))
                         : __uint_as_float((uint32_t)a.x_bf16[(size_t)t * H + i] << 16);
    };
    if (a.act_e4m3) {
        // x quantized to E4M3 under one ue8m0 scale per 128 elements, then the
        // dequantized values as 8 pieces
        const int b = blockIdx.y * (blockDim.x >> 5) + warp;      // 128-element block = unit
        if (b >= H / 128) return;
        const size_t abytes = g_act_bytes(H, 8);
        float v[4];
        for (int hh = 0; hh < 2; hh++)
            for (int e = 0; e < 2; e++) v[2 * hh + e] = xval(b * 128 + hh * 64 + 2 * lane + e);
        const float amax = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
        const int s = ue8m0_for_amax_bits(amax);
        for (int hh = 0; hh < 2; hh++) {
            Pieces64<8> pc;
            make_pieces64<8>(e4m3_quant_dequant(v[2 * hh], s), e4m3_quant_dequant(v[2 * hh + 1], s), pc);
            const PieceRow<8> pr = transpose_pieces<8>(pc, lane, s_tr[warp]);
            for (int kk = 0; kk < a.topk; kk++) {
                if (s_P[kk] < 0) continue;
                const GDst d = group_dst<8>(s_off[kk], s_gb[kk], s_cnt[kk], s_P[kk], b, kgt, abytes, a.xg, a.xgsf);
                store_piece_rows<8>(pr, lane, d.unit, d.mstride, d.atom, d.i, 2 * hh);
            }
        }
        return;
    }
    const int b = blockIdx.y * (blockDim.x >> 5) + warp;          // 64-element span
    if (b >= H / 64) return;
    if (a.act_e2m1) {
        // the one piece of a 32-block is its E2M1 quantization: the scale is
        // the least 2^e with max|x| <= 6 * 2^e, codes round to nearest even
        const size_t abytes = g_act_bytes(H, 1);
        Pieces64<1> pc;
        make_pieces64<1>(xval(b * 64 + 2 * lane), xval(b * 64 + 2 * lane + 1), pc);
        for (int kk = 0; kk < a.topk; kk++) {
            if (s_P[kk] < 0) continue;
            const GDst d = group_dst<1>(s_off[kk], s_gb[kk], s_cnt[kk], s_P[kk], b / 2, kgt, abytes, a.xg, a.xgsf);
            store_pieces64<1>(pc, lane, d.unit, d.mstride, d.atom, d.i, 2 * (b & 1));
        }
        return;
    }
    const size_t abytes = g_act_bytes(H, 16);
    Pieces64<16> pc;
    make_pieces64<16>(xval(b * 64 + 2 * lane), xval(b * 64 + 2 * lane + 1), pc);
    const PieceRow<16> pr = transpose_pieces<16>(pc, lane, s_tr[warp]);
    for (int kk = 0; kk < a.topk; kk++) {
        if (s_P[kk] < 0) continue;
        const GDst d = group_dst<16>(s_off[kk], s_gb[kk], s_cnt[kk], s_P[kk], b / 2, kgt, abytes, a.xg, a.xgsf);
        store_piece_rows<16>(pr, lane, d.unit, d.mstride, d.atom, d.i, 2 * (b & 1));
    }
}

// ----------------------------------------------------------------- k_glayer

// A CTA's part of one projection's unit stream: U units over the first
// G = min(grid, U) CTAs (CTA c < G takes [c U / G, (c + 1) U / G), at least
// one unit; the others none), so the CTAs between a split job's first and
// last all hold part of it.
struct GRange {
    uint32_t u0, u1, j0, jlast;
    int G;                  // CTAs that take part in this projection
    int ngroups;            // groups of the layer (from the route kernel)
    bool empty;
};

__device__ __forceinline__ long long g_range_start(long long U, int G, int c) { return (long long)c * U / G; }

__device__ __forceinline__ int g_cta_of_unit(long long U, int G, long long x)
{
    return (int)(((x + 1) * G - 1) / U);
}

__device__ __forceinline__ GRange g_cta_range(long long U, int grid, int kgt, int ngroups)
{
    GRange r;
    r.ngroups = ngroups;
    const int G = (int)(U < grid ? U : grid);
    const int c = (int)blockIdx.x < G ? (int)blockIdx.x : G;
    r.G = G;
    r.u0 = (uint32_t)(G > 0 ? g_range_start(U, G, c) : 0);
    r.u1 = (uint32_t)(G > 0 ? g_range_start(U, G, c < G ? c + 1 : c) : 0);
    r.empty = r.u1 == r.u0;
    r.j0 = r.u0 / (uint32_t)kgt;
    r.jlast = r.empty ? r.j0 : (r.u1 - 1) / (uint32_t)kgt;
    return r;
}

// Walks a CTA's range in chunks of at most kGCU units that never cross a job;
// every role sees the same sequence.
struct GWalk {
    uint32_t u, u1, kgt, job, kg;
    __device__ GWalk(int kgt_, const GRange& r)
    {
        u = r.u0;
        u1 = r.u1;
        kgt = (uint32_t)kgt_;
        job = r.j0;
        kg = r.u0 - r.j0 * kgt;
    }
    __device__ uint32_t chunk() const { return min(min(kgt - kg, u1 - u), (uint32_t)kGCU); }
    // advance past a chunk of n units; true at the end of a job or of the range
    __device__ bool advance(uint32_t n, bool& next_job)
    {
        u += n;
        kg += n;
        next_job = false;
        bool jend = (u == u1);
        if (kg == kgt) {
            kg = 0;
            job++;
            next_job = true;
            jend = true;
        }
        return jend;
    }
};

// Chunks of a CTA's range (as GWalk cuts it: never across a job, at most
// kGCU units), in closed form.
__device__ __forceinline__ int g_count_chunks(int kgt, const GRange& r)
{
    if (r.empty) return 0;
    const uint32_t K = (uint32_t)kgt, CU = (uint32_t)kGCU;
    const uint32_t fj = (r.u0 / K + 1) * K;            // end of the first job
    if (r.u1 <= fj) return (int)((r.u1 - r.u0 + CU - 1) / CU);
    const uint32_t whole = (r.u1 - fj) / K, rest = (r.u1 - fj) % K;
    return (int)((fj - r.u0 + CU - 1) / CU + whole * ((K + CU - 1) / CU) + (rest + CU - 1) / CU);
}

// Walks the jobs of one projection in order.  Jobs are ordered (expert, tile
// pair, group of the expert, tile of the pair): the two tiles 2b, 2b + 1 of a
// group are adjacent jobs (the E4M3 mode quantizes h per 128 = two gate/up
// tiles, so both halves usually meet in one CTA), and the groups of an expert
// re-read a tile from L2 within two jobs.  Expert e's jobs are [ntiles gb,
// ntiles (gb + ng)), so job / ntiles is one of its groups.  Moving to the next
// job is arithmetic; only an expert boundary reads the next expert's group
// record and weight pointers.
struct GCursor {
    int b, c, t;                 // tile pair, group within the expert, tile of the pair
    int gb, ng, cnt, p0e;        // the expert's first group, groups, slots, first sorted position
    int ngroups, gs;
    const uint8_t* blob;         // the expert's packed blob
    bool ok;

    __device__ void enter(const GroupArgs& a, int gl)
    {
        const GroupInfo gi = a.groups[gl];
        gb = gi.gb;
        ng = gi.ng;
        cnt = gi.cnt;
        p0e = gi.p0 - (gl - gi.gb) * gs;
        blob = a.experts[gi.e];
        ok = blob && (reinterpret_cast<uintptr_t>(blob) & 15) == 0;
    }
    __device__ void init(const GroupArgs& a, const GPlan& p, uint32_t job, int ngroups_)
    {
        ngroups = ngroups_;
        gs = p.gs;
        enter(a, (int)(job / (uint32_t)p.ntiles));
        const uint32_t local = job - (uint32_t)gb * (uint32_t)p.ntiles;
        const uint32_t paired = (uint32_t)(p.ntiles / 2) * 2u * (uint32_t)ng;   // jobs in full pairs
        if (local < paired) {
            b = (int)(local / (2u * (uint32_t)ng));
            const uint32_t r = local % (2u * (uint32_t)ng);
            c = (int)(r / 2);
            t = (int)(r % 2);
        } else {               // the last, single tile (odd tile count)
            b = p.ntiles / 2;
            c = (int)(local - paired);
            t = 0;
        }
    }
    __device__ void next(const GroupArgs& a, const GPlan& p)
    {
        if (t == 0 && 2 * b + 1 < p.ntiles) {
            t = 1;
            return;
        }
        t = 0;
        if (++c < ng) return;
        c = 0;
        if (++b < (p.ntiles + 1) / 2) return;
        b = 0;
        if (gb + ng < ngroups) enter(a, gb + ng);
    }
    template <int PHASE>
    __device__ GJob job(const GroupArgs& a, const GPlan& p) const
    {
        GJob j;
        j.tile = 2 * b + t;
        j.g = gb + c;
        j.p0 = p0e + c * gs;
        j.nt = min(gs, cnt - c * gs);
        j.B = g_group_b(PHASE == 0 ? a.xg : a.hg, p.np, j.p0, j.g, p.act_bytes);
        j.Bsf = (PHASE == 0 ? a.xgsf : a.hgsf) + (size_t)j.g * p.kgt * kUnitSfBytes;
        j.ok = ok;
        j.w = ok ? blob + p.off + (size_t)j.tile * p.tile_bytes : nullptr;
        return j;
    }
};

__device__ __forceinline__ uint32_t g_ld_acquire_u32(const int* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t g_ld_relaxed_u64(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void g_st_relaxed_u64(uint64_t* p, uint64_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void g_set_abort(const GroupArgs& a, GSmem& sm)
{
    atomicOr(a.status, kStatusTimeout);
    sm.abort = 1;
}

// Streams the weights of one projection's range into the ring and posts each
// stage's activation source to the loader.  n: chunks so far (both phases).
template <int PHASE>
__device__ bool gproduce(const GroupArgs& a, const GPlan& p, const GRange& r, GSmem& sm, int& n)
{
    if (r.empty) return true;
    GWalk wk(p.kgt, r);
    GCursor cur;
    cur.init(a, p, wk.job, r.ngroups);
    GJob ji = cur.job<PHASE>(a, p);
    if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
    uint64_t w_e = 0;                          // debug builds: time spent waiting
    while (wk.u < wk.u1) {
        const uint32_t nun = wk.chunk();
        const bool has_half = p.kg_half && (wk.kg + nun == wk.kgt);
        const uint32_t nfull = nun - (has_half ? 1u : 0u);
        const uint32_t wb = nfull * kUnitBytes + (has_half ? kHalfUnitBytes : 0);   // one copy
        const uint32_t gub = g_unit_b(p.np, ji.nt);               // piece bytes of the group per unit
        const uint32_t bb = nfull * gub + (has_half ? gub / 2 : 0);
        const uint32_t bsb = nun * kUnitSfBytes;
        const int s = n % kGStagesA;
        const uint64_t tw = G_NOW();
        if (n >= kGStagesA &&
            !mbar_wait_or_abort(&sm.emptyA[s], ((n / kGStagesA) & 1) ^ 1, &sm.abort, kGWaitLimitNs)) {
            g_set_abort(a, sm);
            return false;
        }
        G_ACC(w_e, tw);
        uint8_t* stg = sm.stageA[s];
        if (ji.ok) {
            mbar_arrive_expect_tx(&sm.fullA[s], wb);
            bulk_g2s(stg, ji.w + (size_t)wk.kg * kUnitBytes, wb, &sm.fullA[s]);
            sm.bsrc[s] = GBSrc{ji.B + (size_t)wk.kg * gub, ji.Bsf + (size_t)wk.kg * kUnitSfBytes, bb, bsb, PHASE};
        } else {
            mbar_arrive(&sm.fullA[s]);     // an empty stage: nothing to multiply
            sm.bsrc[s].B = nullptr;
        }
        mbar_arrive(&sm.posted[s]);        // release: bsrc is visible to the loader
        G_TRACE(0, n);
        bool nj;
        wk.advance(nun, nj);
        n++;
        if (nj && wk.u < wk.u1) {
            cur.next(a, p);
            ji = cur.job<PHASE>(a, p);
            if (!ji.ok) atomicOr(a.status, kStatusBadIndex);
        }
    }
    G_ADD(11, w_e);
    (void)w_e;
    return true;
}

// Issues the activation copies of every posted stage, in order, into the
// activation ring: x's pieces after the previous kernel (PDL), h's once the
// grid-wide count of finished h tiles reaches h_target.  Before exiting it
// waits (bounded) for its own copies in flight.
__device__ void gload_b(const GroupArgs& a, int nchunks, uint32_t h_target, GSmem& sm)
{
    bool pdl_done = false, h_done = false;
    int n = 0;
    for (; n < nchunks; n++) {
        const int s = n % kGStagesA, sb = n % kGStagesB;
        // slot sb last held chunk n - kGStagesB: it is free once that chunk's
        // weight stage is empty (all issuers committed it).  That barrier cannot
        // be two phases ahead here: chunk n - kGStagesB + kGStagesA needs pieces
        // this loop has not issued yet (kGStagesB <= kGStagesA).
        const int m = n - kGStagesB;
        if (!mbar_wait_or_abort(&sm.posted[s], (n / kGStagesA) & 1, &sm.abort, kGWaitLimitNs) ||
            (m >= 0 &&
             !mbar_wait_or_abort(&sm.emptyA[m % kGStagesA], (m / kGStagesA) & 1, &sm.abort, kGWaitLimitNs))) {
            g_set_abort(a, sm);
            break;
        }
        const GBSrc q = sm.bsrc[s];
        if (!q.B) {
            mbar_arrive(&sm.fullB[sb]);    // nothing to multiply in this stage
            continue;
        }
        if (!pdl_done) {
            pdl_wait();
            pdl_done = true;
        }
        if (q.phase == 1 && !h_done) {
            bool ok = g_ld_acquire_u32(a.sync) >= h_target;
            if (!ok) {
                const uint64_t t0 = wait_clock();
                while (!(ok = g_ld_acquire_u32(a.sync) >= h_target))
                    if (*(volatile int*)&sm.abort || wait_clock() - t0 > wait_cycles(kGWaitLimitNs)) break;
            }
            G_CTA(7);
            // h was written with generic stores; the copies read it through the async proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
            if (!ok) g_set_abort(a, sm);
            h_done = true;
        }
        uint8_t* stg = sm.stageB[sb];
        mbar_arrive_expect_tx(&sm.fullB[sb], q.nb + q.nsf);
        bulk_g2s(stg, q.B, q.nb, &sm.fullB[sb]);
        bulk_g2s(stg + kGOffSfb, q.Bsf, q.nsf, &sm.fullB[sb]);
    }
    // no copy may still be in flight into this CTA's memory at exit
    for (int m = n > kGStagesB ? n - kGStagesB : 0; m < n; m++)
        mbar_wait_bounded(&sm.fullB[m % kGStagesB], (m / kGStagesB) & 1, kGWaitLimitNs);
}

struct GIss {
    int n, buf;
    uint32_t use[2];
    bool abort;
};

// Issuer ii takes unit ii of every stage: its two scale atoms to TMEM, then
// one MMA per 64-K step (two per unit, one for a half unit) of N = np nt
// (rounded up to a multiple of 16; the extra columns are never read) into its
// own double-buffered accumulator.
template <int PHASE>
__device__ void gissue(const GroupArgs& a, const GPlan& p, const GRange& r, GSmem& sm, uint32_t tmem, int ii,
                       GIss& is)
{
    if (r.empty) return;
    GWalk wk(p.kgt, r);
    GCursor cur;
    cur.init(a, p, wk.job, r.ngroups);
    GJob ji = cur.job<PHASE>(a, p);
    bool any = false;               // this issuer's accumulator holds part of this job
    bool job_start = true;
    uint64_t w_acc = 0, w_a = 0, w_b = 0, w_is = 0, w_all = 0;   // debug builds: time spent waiting / issuing
    const uint64_t t_begin = G_NOW();
    while (wk.u < wk.u1) {
        const uint32_t nun = wk.chunk();
        const int s = is.n % kGStagesA, sbi = is.n % kGStagesB;
        if (job_start) {
            // the epilogue must have read this accumulator's previous job
            const uint64_t tw = G_NOW();
            if (!is.abort && is.use[is.buf] > 0 &&
                !mbar_wait_or_abort(&sm.acc_empty[is.buf], (is.use[is.buf] - 1) & 1, &sm.abort, kGWaitLimitNs)) {
                g_set_abort(a, sm);
                is.abort = true;
            }
            G_ACC(w_acc, tw);
            job_start = false;
        }
        const uint64_t tw1 = G_NOW();
        bool okA = is.abort || mbar_wait_or_abort(&sm.fullA[s], (is.n / kGStagesA) & 1, &sm.abort, kGWaitLimitNs);
        G_ACC(w_a, tw1);
        const uint64_t tw2 = G_NOW();
        bool okB = is.abort || !okA ||
                   mbar_wait_or_abort(&sm.fullB[sbi], (is.n / kGStagesB) & 1, &sm.abort, kGWaitLimitNs);
        G_ACC(w_b, tw2);
        if (!is.abort && (!okA || !okB)) {
            g_set_abort(a, sm);
            is.abort = true;
        }
        if (ii == 0) G_TRACE(1, is.n);
        const uint64_t tis = G_NOW();
        if (!is.abort && ji.ok && (uint32_t)ii < nun) {
            tc_fence_after();
            const uint8_t* st = sm.stageA[s];
            const uint8_t* sbs = sm.stageB[sbi];
            const uint32_t nt = (uint32_t)ji.nt;
            const uint32_t idesc = mxf4_idesc(kTileRows, ((uint32_t)p.np * nt + 15u) & ~15u);
            const uint32_t col = tmem + kGSfCol0 + (uint32_t)(s * kGCU + ii) * 8;
            const bool half = p.kg_half && (wk.kg + (uint32_t)ii == wk.kgt - 1);
            const uint8_t* unit = st + ii * kUnitBytes;            // codes, then the scale atom
            tc_cp_sf(col, umma_desc(smem_u32(unit + (half ? kMmaCodeBytes : kUnitCodeBytes)), 16, 128));
            tc_cp_sf(col + 4, umma_desc(smem_u32(sbs + kGOffSfb + ii * kUnitSfBytes), 16, 128));
            for (uint32_t m = 0; m < (half ? 1u : 2u); m++) {
                const uint64_t ad = umma_desc(smem_u32(unit + m * kMmaCodeBytes), 128, 256);
                const uint32_t gub = g_unit_b(p.np, (int)nt);
                const uint64_t bd = umma_desc(smem_u32(sbs + ii * gub + m * (gub / 2)), 128, 256);
                tc_mma_mxf4(tmem + (uint32_t)(ii * 2 + is.buf) * kGAccCols, ad, bd, mxf4_idesc_sf(idesc, 2 * m),
                            col, col + 4, any ? 1u : 0u);
                any = true;
            }
        }
        tc_commit(&sm.emptyA[s]);          // this issuer's part of the stage (weights and pieces) is consumed
        G_ACC(w_is, tis);
        bool nj;
        const bool jend = wk.advance(nun, nj);
        is.n++;
        if (nj && wk.u < wk.u1) {
            cur.next(a, p);
            ji = cur.job<PHASE>(a, p);
        }
        if (jend) {
            tc_commit(&sm.acc_full[is.buf]);   // this issuer's accumulator is final
            is.use[is.buf]++;
            is.buf ^= 1;
            any = false;
            job_start = true;
        }
    }
    G_ACC(w_all, t_begin);
    if (ii == 0) {
        G_ADD(8, w_acc);
        G_ADD(9, w_a);
        G_ADD(10, w_b);
        G_ADD(12, w_is);
        G_ADD(13, w_all);
    }
    (void)w_acc;
    (void)w_a;
    (void)w_b;
    (void)w_is;
    (void)w_all;
    (void)t_begin;
}

// ------------------------------------------------------------------ epilogue

// Gate/up job (group, tile), slot i -> the 64 values h = w * silu(g) * u of
// that slot as NP pieces into the down projection's B operand, by one warp;
// then the grid-wide count of finished h tiles grows by the tiles written.
// In the E4M3 mode h is quantized per 128 (two tiles): local = 1 for the first
// tile of a pair whose second tile this CTA finishes next (raw h goes to the
// warp's stash), 2 for that second tile (the first one's h is in the stash),
// 0 for a pair split between CTAs (met through global memory).
// The pieces of one slot: transposed into 16- or 8-byte rows (8, 16 pieces) or
// stored as they are (one piece: a byte per lane, already contiguous).
template <int NP>
__device__ __forceinline__ void put_pieces(const Pieces64<NP>& pc, int lane, uint8_t* unit, int mstride,
                                           uint8_t* atom, int i, int blk0, uint4* scratch)
{
    if constexpr (NP == 1) {
        store_pieces64<1>(pc, lane, unit, mstride, atom, i, blk0);
    } else {
        const PieceRow<NP> pr = transpose_pieces<NP>(pc, lane, scratch);
        store_piece_rows<NP>(pr, lane, unit, mstride, atom, i, blk0);
    }
}

template <int NP>
__device__ void gfinalize_gate_up(const GroupArgs& a, const GPlan& p, const GJob& jb, int i, const float* comb,
                                  int lane, float* stash, int local, uint4* scratch)
{
    const int P = jb.p0 + i, tile = jb.tile;
    const float2 g = *reinterpret_cast<const float2*>(comb + 2 * lane);
    const float2 u = *reinterpret_cast<const float2*>(comb + 64 + 2 * lane);
    float h0 = silu(g.x) * u.x, h1 = silu(g.y) * u.y;
    const size_t abytes = g_act_bytes(a.I, NP);
    const int kgt = (a.I + 127) / 128;
    uint8_t* unit = g_group_b(a.hg, NP, jb.p0, jb.g, abytes) + (size_t)(tile / 2) * g_unit_b(NP, jb.nt);
    uint8_t* atom = a.hgsf + ((size_t)jb.g * kgt + tile / 2) * kUnitSfBytes;
    const int mstride = (int)g_unit_b(NP, jb.nt) / 2;
    int done = 1;                         // h tiles whose pieces this call writes
    if (a.act_e4m3) {
        // h is quantized to E4M3 per 128 along I (tiles 2b, 2b + 1; a last block
        // of 64 is one tile) before w; the second tile of a block to finish
        // quantizes both, from the first one's raw h
        const int blk = tile / 2, nblk = (p.ntiles + 1) / 2;
        const bool pair = (tile | 1) < p.ntiles;
        float o0 = 0.0f, o1 = 0.0f;
        if (pair && local == 1) {
            stash[2 * lane] = h0;
            stash[2 * lane + 1] = h1;
            return;
        }
        if (pair && local == 2) {
            o0 = stash[2 * lane];
            o1 = stash[2 * lane + 1];
            done = 2;
        } else if (pair) {
            float* mine = a.hraw + (size_t)P * a.I + (size_t)tile * 64 + 2 * lane;
            mine[0] = h0;
            mine[1] = h1;
            __threadfence();
            __syncwarp();
            int old = 0;
            if (lane == 0) old = atomicAdd(a.hpair + (size_t)P * nblk + blk, 1);
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == 0) return;         // the other tile finishes the block
            __threadfence();
            const float* other = a.hraw + (size_t)P * a.I + (size_t)(tile ^ 1) * 64 + 2 * lane;
            o0 = __ldcg(other);
            o1 = __ldcg(other + 1);
            if (lane == 0) a.hpair[(size_t)P * nblk + blk] = 0;     // ready for the next launch
            done = 2;
        }
        const float amax = warp_max(fmaxf(fmaxf(fabsf(h0), fabsf(h1)), fmaxf(fabsf(o0), fabsf(o1))));
        const int s = ue8m0_for_amax_bits(amax);
        h0 = e4m3_quant_dequant(h0, s);
        h1 = e4m3_quant_dequant(h1, s);
        if (pair) {
            const float w = a.w[a.perm[P]];
            Pieces64<NP> po;
            make_pieces64<NP>(e4m3_quant_dequant(o0, s) * w, e4m3_quant_dequant(o1, s) * w, po);
            put_pieces<NP>(po, lane, unit, mstride, atom, i, 2 * ((tile ^ 1) & 1), scratch);
        }
    }
    // E2M1 mode: the one piece is h quantized per 32 (w scales the down output);
    // otherwise w * h as pieces
    const float w = a.act_e2m1 ? 1.0f : a.w[a.perm[P]];
    Pieces64<NP> pc;
    make_pieces64<NP>(h0 * w, h1 * w, pc);
    put_pieces<NP>(pc, lane, unit, mstride, atom, i, 2 * (tile & 1), scratch);
    // the down projection reads these with bulk copies (async proxy), in other CTAs
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    // release: the pieces (this warp's stores, ordered by the warp barrier) are
    // visible before the count; the thread does not wait for the add
    if (lane == 0) asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(a.sync), "r"(done) : "memory");
}

struct GEpi {
    int buf, cb;
    uint32_t use[2];
    uint32_t tag;               // this launch's tag of the partial sums
};

// Partial sums (nt per row) of a split job from CTAs c..c1, added in CTA
// order into acc; returns the first CTA not yet folded in.  With spin, waits
// (bounded) for each; without, stops at the first whose entries are not all
// there yet.
template <int NT>
__device__ __forceinline__ int gfold(const uint64_t* part, int c, int c1, int row, int nt, uint32_t tag, bool spin,
                                     float (&acc)[NT], bool* timed_out)
{
    uint64_t t0 = 0;
    while (c <= c1) {
        float v[NT];
        bool all = true;
#pragma unroll
        for (int i = 0; i < NT; i++) {
            v[i] = 0.0f;
            if (i < nt && all) {
                const uint64_t e = g_ld_relaxed_u64(part + ((size_t)c * NT + i) * kTileRows + row);
                if ((uint32_t)(e >> 32) == tag) v[i] = __uint_as_float((uint32_t)e);
                else all = false;
            }
        }
        if (all) {
#pragma unroll
            for (int i = 0; i < NT; i++) acc[i] += v[i];
            c++;
            continue;
        }
        if (!spin) break;
        if (t0 == 0) t0 = wait_clock();
        else if (wait_clock() - t0 > wait_cycles(kGWaitLimitNs)) {
            *timed_out = true;
            break;
        }
    }
    return c;
}

template <int PHASE, int NT>
__device__ void gepilogue(const GroupArgs& a, const GPlan& p, const GRange& r, GSmem& sm, uint32_t tmem, long long U,
                          int quad, int lane, GEpi& es)
{
    if (r.empty) return;
    uint64_t* part = PHASE == 0 ? a.part_gu : a.part_dn;
    const int row = quad * 32 + lane;                      // accumulator row of this thread
    const int G = r.G;
    GWalk wk(p.kgt, r);
    GCursor cs;
    cs.init(a, p, wk.job, r.ngroups);
    GJob ji = cs.job<PHASE>(a, p);
    uint32_t mask = 0;                                     // issuers that accumulated into this job
    while (wk.u < wk.u1) {
        const uint32_t job = wk.job;
        const GJob cur = ji;
        const uint32_t nun = wk.chunk();
        if (cur.ok) mask |= (1u << nun) - 1u;
        bool nj;
        const bool jend = wk.advance(nun, nj);
        if (nj && wk.u < wk.u1) {
            cs.next(a, p);
            ji = cs.job<PHASE>(a, p);
        }
        if (!jend) continue;

        // --------------------------------------------- end of (this CTA's part of) a job
        const long long js = (long long)job * p.kgt, je = js + p.kgt;
        const bool owner = js >= r.u0;
        const int c1 = owner && je > r.u1 ? g_cta_of_unit(U, G, je - 1) : (int)blockIdx.x;
        const int nt = cur.nt;
        float pacc[NT];
#pragma unroll
        for (int i = 0; i < NT; i++) pacc[i] = 0.0f;
        bool late = false;
        int cnext = blockIdx.x + 1;
        if (c1 > (int)blockIdx.x)   // while the last MMAs run: the partials that are there already
            cnext = gfold<NT>(part, cnext, c1, row, nt, es.tag, false, pacc, &late);

        const int buf = es.buf;
        const bool ready = !*(volatile int*)&sm.abort &&
                           mbar_wait_or_abort(&sm.acc_full[buf], es.use[buf] & 1, &sm.abort, kGWaitLimitNs);
        es.use[buf]++;
        if (!ready) g_set_abort(a, sm);
        tc_fence_after();
        float v[NT];
#pragma unroll
        for (int i = 0; i < NT; i++) v[i] = 0.0f;
        if (ready) {
            // slot i: the sum of its np piece columns, issuers in order
#pragma unroll
            for (int ii = 0; ii < kGIssuers; ii++) {
                if (!((mask >> ii) & 1u)) continue;
                const uint32_t acc0 = tmem + (uint32_t)(ii * 2 + buf) * kGAccCols + ((uint32_t)(quad * 32) << 16);
#pragma unroll
                if (p.np == 1) {            // one column per slot
                    float acc[16];
                    tc_ld16(acc0, acc);
#pragma unroll
                    for (int i = 0; i < NT; i++) v[i] += acc[i];
                    continue;
                }
#pragma unroll
                for (int i = 0; i < NT; i++) {
                    if (i >= nt) break;
                    if (p.np == 8) {
                        float acc[8];
                        tc_ld8(acc0 + (uint32_t)(i * 8), acc);
#pragma unroll
                        for (int c = 0; c < 8; c++) v[i] += acc[c];
                    } else {
                        float acc[16];
                        tc_ld16(acc0 + (uint32_t)(i * 16), acc);
#pragma unroll
                        for (int c = 0; c < 16; c++) v[i] += acc[c];
                    }
                }
            }
        }
        mask = 0;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
        es.buf ^= 1;

        if (!owner) {
            // a later part of a job owned by an earlier CTA
#pragma unroll
            for (int i = 0; i < NT; i++)
                if (i < nt)
                    g_st_relaxed_u64(part + ((size_t)blockIdx.x * NT + i) * kTileRows + row,
                                     ((uint64_t)es.tag << 32) | __float_as_uint(v[i]));
            continue;
        }
        if (cnext <= c1) {
            const bool abort = *(volatile int*)&sm.abort;
            gfold<NT>(part, cnext, c1, row, nt, es.tag, !abort, pacc, &late);
            if (late) g_set_abort(a, sm);
        }
#pragma unroll
        for (int i = 0; i < NT; i++) v[i] += pacc[i];
        if (quad == 0 && lane == 0) G_TRACE(2, es.use[0] + es.use[1]);
        if (PHASE == 0) {
            float(*comb)[kTileRows] = sm.comb[es.cb];
#pragma unroll
            for (int i = 0; i < NT; i++)
                if (i < nt) comb[i][row] = v[i];
            named_sync(1, 128);
            int local = 0;      // E4M3 pair of tiles finished in this CTA (see gfinalize_gate_up)
            if (a.act_e4m3 && (cur.tile | 1) < p.ntiles) {
                const long long partner = (cur.tile & 1) ? (long long)job - 1 : (long long)job + 1;
                if (g_cta_of_unit(U, G, partner * p.kgt) == (int)blockIdx.x) local = (cur.tile & 1) ? 2 : 1;
            }
            for (int i = quad; i < nt; i += 4) {
                if (p.np == 8) gfinalize_gate_up<8>(a, p, cur, i, comb[i], lane, sm.hstash[i], local, sm.tr[quad]);
                else if (p.np == 1)
                    gfinalize_gate_up<1>(a, p, cur, i, comb[i], lane, sm.hstash[i], local, sm.tr[quad]);
                else gfinalize_gate_up<16>(a, p, cur, i, comb[i], lane, sm.hstash[i], local, sm.tr[quad]);
            }
            if (quad == 0 && lane == 0) G_TRACE(3, es.use[0] + es.use[1]);
            es.cb ^= 1;
        } else {
            // o of each slot: rows tile*128 .. +127 of the down output
#pragma unroll
            for (int i = 0; i < NT; i++)
                if (i < nt) a.obuf[(size_t)(cur.p0 + i) * a.H + (size_t)cur.tile * kTileRows + row] = v[i];
        }
    }
}

// ------------------------------------------------------------------ kernel

// One MoE layer on the expert-major path: the gate/up projection then the
// down projection, in one persistent grid.  The job count comes from the
// route kernel, finished before this grid starts (k_gprep lets it start only
// after waiting for the route kernel).
template <int NT>
__global__ void __launch_bounds__(kGThreads, 1) k_glayer(GroupArgs a, GPlan p0, GPlan p1)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    GSmem& sm = *reinterpret_cast<GSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const long long ngroups = a.gbase[a.E];
    const long long U0 = ngroups * p0.ntiles * p0.kgt, U1 = ngroups * p1.ntiles * p1.kgt;
    const GRange r0 = g_cta_range(U0, G, p0.kgt, (int)ngroups), r1 = g_cta_range(U1, G, p1.kgt, (int)ngroups);
    const uint32_t h_target = (uint32_t)a.offsets[a.E] * (uint32_t)p0.ntiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStagesA; s++) {
            mbar_init(&sm.fullA[s], 1);
            mbar_init(&sm.emptyA[s], kGIssuers);
            mbar_init(&sm.posted[s], 1);
        }
        for (int s = 0; s < kGStagesB; s++) mbar_init(&sm.fullB[s], 1);
        for (int b = 0; b < 2; b++) {
            mbar_init(&sm.acc_full[b], kGIssuers);
            mbar_init(&sm.acc_empty[b], 4);
        }
        for (int i = 0; i < kGIssuers; i++) mbar_init(&sm.drain[i], 1);
        sm.abort = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(&sm.tmem, kGTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = sm.tmem;

    if (warp == 0) {
        if (lane == 0) {
            int n = 0;
            G_CTA(0);
            const bool ok0 = gproduce<0>(a, p0, r0, sm, n);
            G_CTA(1);
            if (ok0) gproduce<1>(a, p1, r1, sm, n);
            G_CTA(2);
            // no copy may still be in flight into this CTA's memory at exit
            for (int m = n > kGStagesA ? n - kGStagesA : 0; m < n; m++)
                mbar_wait_bounded(&sm.fullA[m % kGStagesA], (m / kGStagesA) & 1, kGWaitLimitNs);
        }
        return;
    }
    if (warp == kGWarpLoader) {
        if (lane == 0) gload_b(a, g_count_chunks(p0.kgt, r0) + g_count_chunks(p1.kgt, r1), h_target, sm);
        return;
    }
    if (warp < kGWarpEpi0) {
        if (lane == 0) {
            GIss is;
            is.n = 0;
            is.buf = 0;
            is.use[0] = is.use[1] = 0;
            is.abort = false;
            gissue<0>(a, p0, r0, sm, tmem, warp - 1, is);
            if (warp == 1) G_CTA(3);
            gissue<1>(a, p1, r1, sm, tmem, warp - 1, is);
            if (warp == 1) G_CTA(4);
            // none of this thread's MMAs may be in flight when TMEM is freed
            tc_commit(&sm.drain[warp - 1]);
            mbar_wait_bounded(&sm.drain[warp - 1], 0, kGWaitLimitNs);
        }
        __syncwarp();
    } else {
        pdl_wait();
        GEpi es;
        es.buf = 0;
        es.cb = 0;
        es.use[0] = es.use[1] = 0;
        es.tag = 1u + (g_ld_acquire_u32(a.sync + 2) & 0x3FFFFFFFu);   // never 0, the cleared value
        gepilogue<0, NT>(a, p0, r0, sm, tmem, U0, warp & 3, lane, es);
        if (warp == kGWarpEpi0 && lane == 0) G_CTA(5);
        gepilogue<1, NT>(a, p1, r1, sm, tmem, U1, warp & 3, lane, es);
        if (warp == kGWarpEpi0 && lane == 0) G_CTA(6);
        if (warp == kGWarpEpi0 && lane == 0) {
            // the last CTA to finish resets the layer's counters for the next launch
            __threadfence();
            const int done = atomicAdd(a.sync + 1, 1);
            if (done == G - 1) {
                a.sync[0] = 0;
                a.sync[1] = 0;
                a.sync[2] += 1;      // the next launch tags its partial sums differently
                __threadfence();
            }
        }
    }
    // the issuer and epilogue warps meet here before the tensor memory is released
    tc_fence_before();
    named_sync(2, (kGIssuers + 4) * 32);
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kGTmemCols);
}

// --------------------------------------------------------------- k_gcombine

// grid (T), 256 threads: y[t] = sum over the token's slots, in k order, of the
// down outputs (or x[t] += that).
__global__ void __launch_bounds__(256) k_gcombine(GroupArgs a)
{
    const int t = blockIdx.x, H = a.H;
    __shared__ int s_P[16];
    __shared__ float s_w[16];
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x < a.topk) {
        s_P[threadIdx.x] = a.inv[t * a.topk + threadIdx.x];
        // the E2M1 mode and the kind::mxf8f6f4 path apply the routing weight
        // here (the piece modes fold it into h)
        s_w[threadIdx.x] = (a.act_e2m1 || a.o_unweighted) ? a.w[t * a.topk + threadIdx.x] : 1.0f;
    }
    __syncthreads();
    for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
        // every slot's output (and the residual) loaded first (topk <= 16),
        // then added in k order
        const size_t o = (size_t)t * H + c;
        float4 ov[16];
#pragma unroll
        for (int kk = 0; kk < 16; kk++) {
            const int P = kk < a.topk ? s_P[kk] : -1;
            ov[kk] = P >= 0 ? __ldcg(reinterpret_cast<const float4*>(a.obuf + (size_t)P * H + c))
                            : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (a.x_resid) x = *reinterpret_cast<const float4*>(a.x_resid + o);
        float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int kk = 0; kk < 16; kk++) {
            if (kk >= a.topk || s_P[kk] < 0) continue;
            const float w = s_w[kk];
            s.x = fmaf(w, ov[kk].x, s.x);
            s.y = fmaf(w, ov[kk].y, s.y);
            s.z = fmaf(w, ov[kk].z, s.z);
            s.w = fmaf(w, ov[kk].w, s.w);
        }
        if (a.x_resid) {
            x.x += s.x;
            x.y += s.y;
            x.z += s.z;
            x.w += s.w;
            *reinterpret_cast<float4*>(a.x_resid + o) = x;
        } else if (a.out_f32) {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.y) + o) = s;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y), hi = __floats2bfloat162_rn(s.z, s.w);
            uint2 v;
            v.x = *reinterpret_cast<uint32_t*>(&lo);
            v.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.y) + o) = v;
        }
    }
}

cudaError_t glaunch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void** args)
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

GPlan gplan(const GroupArgs& a, int phase)
{
    GPlan p{};
    const ExpertLayout E = make_expert_layout(a.H, a.I);
    const MatLayout& L = phase == 0 ? E.gu : E.dn;
    p.kgt = L.kgt();
    p.kg_half = L.kg_half;
    p.ntiles = L.tiles;
    p.tile_bytes = L.tile_bytes();
    p.off = phase == 0 ? E.gu_off : E.dn_off;
    p.np = group_pieces(a.act_e4m3 != 0, a.act_e2m1 != 0);
    p.gs = group_slots(a.act_e4m3 != 0, a.act_e2m1 != 0);
    p.act_bytes = g_act_bytes(phase == 0 ? a.H : a.I, p.np);
    p.phase = phase;
    return p;
}

size_t glayer_smem() { return sizeof(GSmem) > kGOneCtaPerSmSmem ? sizeof(GSmem) : kGOneCtaPerSmSmem; }

}  // namespace

GroupWorkspaceSizes group_workspace_sizes(int T, int topk, int E, int H, int I, int sms, bool e4m3)
{
    GroupWorkspaceSizes s{};
    const size_t n = (size_t)T * topk;
    const size_t G = (size_t)max_groups((int)n, E, group_slots(false));
    s.counts = (size_t)E * 4;
    s.offsets = (size_t)(E + 1) * 4;
    s.perm = n * 4;
    s.inv = n * 4;
    s.gbase = (size_t)(E + 1) * 4;
    s.groups = G * sizeof(GroupInfo);
    s.xg = n * act_bytes(H);
    s.xgsf = G * (size_t)((H + 127) / 128) * kUnitSfBytes;
    s.hg = n * act_bytes(I);
    s.hgsf = G * (size_t)((I + 127) / 128) * kUnitSfBytes;
    s.obuf = n * (size_t)H * 4;
    s.part_gu = (size_t)sms * kNT * kTileRows * 8;
    s.part_dn = s.part_gu;
    s.hraw = e4m3 ? n * (size_t)I * 4 : 0;
    s.hpair = e4m3 ? n * (size_t)((I + 127) / 128) * 4 : 0;
    return s;
}

cudaError_t group_init_device()
{
    cudaError_t e = cudaFuncSetAttribute((const void*)k_glayer<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)glayer_smem());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute((const void*)k_glayer<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)glayer_smem());
    return e;
}

cudaError_t launch_group_layer(const GroupArgs& a0, cudaStream_t s, bool pdl, Profiler* prof)
{
    GroupArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    const bool chain = pdl && !prof;
    cudaError_t err;
    RouteArgs ra{a.idx,     a.T * a.topk, a.E,       a.counts, a.offsets,
                 a.perm,    a.inv,        a.status,  a.gbase,  a.groups,
                 group_slots(a.act_e4m3 != 0, a.act_e2m1 != 0)};
    if (prof) prof->begin(kPhaseRoute, s);
    err = launch_route(ra, s, chain);
    if (prof) prof->end(s);
    if (err != cudaSuccess) return err;
    void* args1[] = {&a};
    {
        const int spans = a.act_e4m3 ? a.H / 128 : a.H / 64;     // one warp each
        if (prof) prof->begin(kPhasePrep, s);
        err = glaunch((const void*)k_gprep, dim3(a.T, (spans + 7) / 8), dim3(256), 0, s, chain, args1);
        if (prof) prof->end(s);
        if (err != cudaSuccess) return err;
    }
    GPlan p0 = gplan(a, 0), p1 = gplan(a, 1);
    void* args[] = {&a, &p0, &p1};
    if (prof) prof->begin(kPhaseGateUp, s);
    // the epilogue is compiled for the mode's group size: 16 slots (E2M1) or at most 8
    const void* fn = p0.gs > 8 ? (const void*)k_glayer<16> : (const void*)k_glayer<8>;
    err = glaunch(fn, dim3((unsigned)a.sms), dim3(kGThreads), glayer_smem(), s, chain, args);
    if (prof) prof->end(s);
    if (err != cudaSuccess) return err;
    if (prof) prof->begin(kPhaseDown, s);
    err = launch_group_combine(a, s, chain);
    if (prof) prof->end(s);
    return err;
}

cudaError_t launch_group_combine(const GroupArgs& a0, cudaStream_t s, bool pdl)
{
    GroupArgs a = a0;
    void* args[] = {&a};
    return glaunch((const void*)k_gcombine, dim3(a.T), dim3(256), 0, s, pdl, args);
}

}  // namespace moe
