// gemm8.cu -- expert-major path of one routed FP4 MoE layer with E4M3
// activations fed to the tensor core as they are: block-scaled
// tcgen05.mma kind::mxf8f6f4, the E2M1 weights as operand A and the E4M3
// activation rows as operand B, one ue8m0 scale per 32 along K on both sides
// (the activations' per-128 scale repeated in each of its four 32-blocks).
// A slot is one MMA column, so a group holds up to kF8GroupSlots slots of one
// expert and a weight tile leaves HBM once per group of up to 224 tokens.
//
// Launches, chained with programmatic dependent launch:
//   k_route    (route.cu) the T*k slots sorted by expert, cut into groups of
//              up to kF8GroupSlots consecutive slots of one expert;
//   k_f8prep   x (bf16, or RMSNorm of the fp32 residual) -> E4M3 codes with a
//              ue8m0 scale per 128, written once per slot into its group's B
//              operand;
//   k_f8gemm<0> gate/up: per job (group, tile of 64 gate + 64 up rows) the
//              128 x nb accumulator over K = H, then h = silu(g) * u (fp32)
//              into hraw [sorted slot][I];
//   k_f8hquant h -> E4M3 with a ue8m0 scale per 128 along I (the same rule as
//              x), into the down projection's B operand;
//   k_f8gemm<1> down: per job (group, tile of 128 rows of H) the accumulator
//              over K = I, stored per slot into obuf [sorted slot][H];
//   k_gcombine (group.cu) y[t] = sum_k w_k o[t, k], or x += that.
//
// B operand of a group g (first sorted slot p0, nt slots, nb = nt rounded up
// to 16 rows) over a reduction of K elements: nb x K bytes at
// (p0 + 16 g) * K (a group's rows never reach the next group's start), in
// 128-K units of nb x 128 bytes (a last half unit of nb x 64); inside a unit,
// per 32-K step kb, the no-swizzle K-major layout of the MMA:
//   kb * nb * 32 + (row / 8) * 256 + half * 128 + (row % 8) * 16
// (16 codes per 16-byte row, half 0/1 = codes 0-15 / 16-31 of the step).
// Scale atoms per (group, unit): two of 512 bytes (rows 0-127, 128-255) in
// the order tcgen05.cp moves them, byte (row % 32) * 16 + (row % 128 / 32) * 4
// + kb.
//
// Shared memory: a ring of units -- per unit its packed weights (a blob unit,
// layout.h: codes + scale atom, one bulk copy) followed by the group's
// activation rows of that unit and their scale atoms -- in which each unit
// takes a contiguous span sized to its group (a few KB of rows for a group of
// a few slots, 28 KB for 224), so that small groups keep many units in flight
// while HBM latency is covered; and four stages of expanded weights: four
// warps rewrite each unit's codes into the form kind::mxf8f6f4 reads E2M1 in
// (16 codes in 8 bytes, then 8 bytes of padding, per 16-byte row of a core
// matrix; K = 32 per MMA, so a blob core-matrix row of 32 codes becomes two)
// with the unit's scale atom beside them.
//
// Roles of k_f8gemm (one CTA per SM, jobs j = CTA, CTA + grid, ...; jobs are
// ordered (expert, tile, group) so that the groups of one expert read a tile
// at about the same time, one of them from HBM and the rest from L2):
//   warp 0  weight producer: each unit's packed weights into its span;
//   warp 1  activation producer: the unit's rows and scale atoms beside them
//           (both producers replay the same span order and wait for the
//           spans they overwrite to be consumed);
//   warps 2-4  wide form: warp 2 the MMA issuer (one thread; per unit one
//           MMA per 32-K step over all the group's rows, into the job's
//           double-buffered accumulator) and warp 4 the scale stager (one
//           thread; per unit the scale atoms to TMEM by tcgen05.cp, committed
//           to the issuer's barrier), since one thread issues a tcgen05
//           instruction only every ~120 cycles; narrow form: three issuers,
//           one thread each, taking alternate units of every job, each with
//           its own scale copies and accumulators;
//   warps 5-8  expanders (kind::mxf8f6f4): packed weights -> an
//           expanded-weight stage;
//   warps 9-12 epilogue: tcgen05.ld of the job's accumulator (the narrow
//           form: the issuers' accumulators, added in issuer order), then
//           SwiGLU or the per-slot store.
// Every wait is bounded (2 s): on expiry the kernel records the device-timeout
// status, stops, waits (bounded) for its copies and MMAs in flight and frees
// its TMEM.
#include "common.cuh"
#include "internal.h"

namespace moe {

#ifdef MOE_F8_TRACE
// debug builds only: per CTA, the issuers' cycles spent waiting for each
// dependency and issuing ([0] expanded weights, [1] activation rows, [2] scale
// slot, [3] accumulator, [4] issuing, [5] units), and the first epilogue
// warp's cycles waiting for a finished accumulator [6], reading it out [7],
// and within that: TMEM loads [8], gate/up exchange, SwiGLU and stores [11],
// the pair's closing barrier [12], down stores [13]; the wide form's scale
// stager waiting for the expanded weights [14] and the activation rows [15],
// and issuing [16]; the first expander thread waiting for the packed weights
// [17] and for the stage to be free [18], and expanding [19]
__device__ unsigned long long g_f8_trace[20][1024];
#define F8_ACC(k, t0) atomicAdd(&g_f8_trace[k][blockIdx.x], (unsigned long long)(clock64() - (t0)))
#define F8_NOW() clock64()
#else
#define F8_NOW() 0ll
#define F8_ACC(k, t0) \
    do {              \
    } while (0)
#endif

namespace {

constexpr int kF8Cap = 150 * 1024;                    // the unit ring: packed weights + activation rows
constexpr int kF8D = 32;                               // units in the ring, at most
constexpr int kF8Pad = 4;                              // stages of expanded weights
constexpr int kF8PadBytes = 4 * 4096;                  // a unit's weights, padded: 4 steps x 128 rows x 32 B
constexpr int kF8PadStage = kF8PadBytes + kUnitSfBytes; // ... and its scale atom
constexpr int kF8TmemCols = 512;
constexpr uint64_t kF8WaitNs = 2000000000ull;
constexpr int kF8MaxIssuers = 3;
constexpr int kF8WarpProdA = 0, kF8WarpProdB = 1, kF8WarpMma0 = 2;
constexpr int kF8WarpExp0 = kF8WarpMma0 + kF8MaxIssuers, kF8WarpEpi0 = kF8WarpExp0 + 4;
constexpr int kF8Threads = (kF8WarpEpi0 + 4) * 32;

static_assert(kF8GroupSlots % 16 == 0 && kF8GroupSlots <= 224 && kF8GroupSlotsNarrow <= 64, "MMA N and TMEM");
static_assert(kF8Cap % 128 == 0 && kF8PadStage % 128 == 0, "alignment");
static_assert(kUnitBytes + kF8GroupSlots * 128 + 2 * kUnitSfBytes <= kF8Cap, "a unit fits the ring");

// Tensor memory of the two forms (NI = MMA-issuing threads):
//   NI = 1 (groups of up to kF8GroupSlots = 224 slots): the accumulator of a
//     job at column 256 b (b = 0, 1: double-buffered); the scale slot of unit
//     c, s = c % 4 (the unit's expanded-weight stage), at
//     256 (s % 2) + 224 + 12 (s / 2) (A 4, B 8), filled by the scale stager;
//   NI = 3 (groups of up to 64): issuer i takes the units c with c % 3 == i
//     of every job into accumulators of its own, b = 0, 1 at 64 (2 i + b),
//     columns 0-383, added by the epilogue in issuer order; its scale slots
//     s = 0..4 at 384 + 8 (5 i + s) (A 4, B 4), which it fills itself.
// A scale slot is reused once the unit it held has been multiplied.
template <int NI>
struct F8Tm {
    static_assert(NI == 1 || NI == 3, "the two forms");
    static constexpr bool kWide = NI == 1;
    static constexpr int kSlots = kWide ? 4 : 5;
    static constexpr int kAccs = kWide ? 1 : NI;         // accumulators the epilogue adds
    __device__ static uint32_t acc(int i, uint32_t b) { return kWide ? 256u * b : 64u * (2u * (uint32_t)i + b); }
    __device__ static uint32_t sf(int i, uint32_t c)
    {
        if (kWide) {
            const uint32_t s = c % kSlots;
            return 256u * (s & 1u) + (uint32_t)kF8GroupSlots + 12u * (s >> 1);
        }
        return 384u + 8u * (uint32_t)(kSlots * i) + 8u * ((c / NI) % kSlots);
    }
};
static_assert(384 + 8 * 5 * kF8MaxIssuers <= kF8TmemCols && kF8GroupSlots + 2 * 12 <= 256, "TMEM budget");
static_assert(kF8Pad == 4, "the wide form's scale slots follow the expanded-weight stages");

// A unit's place in the ring: its packed weights (codes + scale atom, one
// bulk copy from the blob) at the start, then the group's activation rows of
// the unit and their scale atoms.  Units take contiguous spans in order; a unit
// that would cross the ring's end starts again at its beginning.
struct F8Smem {
    uint8_t ring[kF8Cap];
    uint8_t pad[kF8Pad][kF8PadStage];   // expanded weights, then the unit's A atom
    float xch[2][32][32];               // epilogue: up values of 32 rows x 32 slots, per warp pair
    uint64_t full_a[kF8D], full_b[kF8D], unit_free[kF8D];
    uint64_t pad_ready[kF8Pad], sf_ready[kF8Pad];
    uint64_t acc_full[2], acc_empty[2], drain[kF8MaxIssuers];
    uint32_t tmem;
    int abort;
};

// One projection's shape, from the host.
struct F8Plan {
    int ntiles;           // 128-row weight tiles
    int kgt;              // 128-K units (a last half unit included)
    int half;             // 1: the last unit is a half unit (K % 128 == 64)
    int K;                // reduction length
    int bunit;            // bytes of one B row per 128-K unit: 128 (E4M3), 64 (E2M1)
    size_t tile_bytes;    // bytes of a tile in the blob
    size_t mat_off;       // the projection's offset in the blob
};

struct F8Job {
    const uint8_t* a;     // weight tile, unit 0
    const uint8_t* b;     // the group's activation rows, unit 0
    const uint8_t* bsf;   // the group's scale atoms, unit 0
    int p0, nt, nb, tile;
    bool ok;              // the expert's blob is present and 16-byte aligned
};

__host__ __device__ inline size_t f8_group_rows(int p0, int g) { return (size_t)p0 + 16 * (size_t)g; }

// Job j of a projection: expert e's jobs are [ntiles gb, ntiles (gb + ng)),
// (tile, group) in that order, so j / ntiles is one of e's groups.
template <int PHASE>
__device__ __forceinline__ F8Job f8_job(const GroupArgs& a, const F8Plan& p, int j)
{
    const int ge = __ldcg(&a.groups[j / p.ntiles].gb), ng = __ldcg(&a.groups[j / p.ntiles].ng);
    const int local = j - p.ntiles * ge;
    const int g = ge + local % ng;
    const int e = __ldcg(&a.groups[g].e), p0 = __ldcg(&a.groups[g].p0), nt = __ldcg(&a.groups[g].nt);
    F8Job J;
    J.tile = local / ng;
    J.p0 = p0;
    J.nt = nt;
    J.nb = (nt + 15) & ~15;
    const uint8_t* blob = a.experts[e];
    J.ok = blob != nullptr && (reinterpret_cast<uintptr_t>(blob) & 15) == 0;
    J.a = blob + p.mat_off + (size_t)J.tile * p.tile_bytes;
    J.b = (PHASE == 0 ? a.xb8 : a.hb8) + f8_group_rows(p0, g) * (size_t)p.K * p.bunit / 128;
    J.bsf = (PHASE == 0 ? a.xb8sf : a.hb8sf) + (size_t)g * p.kgt * (2 * kUnitSfBytes);
    return J;
}

// Sizes of unit u of a job in the ring (the same whether or not the job's
// blob is usable, so that every role places the units alike).
struct F8Unit {
    uint32_t abytes, bbytes, sbytes, size;
    bool half;
};

__device__ __forceinline__ F8Unit f8_unit(const F8Plan& p, const F8Job& jb, int u)
{
    F8Unit U;
    U.half = p.half && u == p.kgt - 1;
    U.abytes = U.half ? kHalfUnitBytes : kUnitBytes;
    U.bbytes = (uint32_t)jb.nb * (uint32_t)(U.half ? p.bunit / 2 : p.bunit);
    U.sbytes = jb.nb > 128 ? 2 * kUnitSfBytes : kUnitSfBytes;
    U.size = (U.abytes + U.bbytes + U.sbytes + 127u) & ~127u;
    return U;
}

// The ring's allocation order, replayed by every role: absolute byte
// positions, a unit starting at the ring's beginning when it would cross the end.
struct F8Ring {
    uint64_t head = 0;
    __device__ __forceinline__ uint64_t take(uint32_t size)
    {
        uint64_t st = head;
        if (st % kF8Cap + size > kF8Cap) st = (st / kF8Cap + 1) * kF8Cap;
        head = st + size;
        return st;
    }
};

// Producers: before unit c (absolute span [st, end)) is written, the units
// still in the ring that it would overlap, and unit c - kF8D (whose barriers
// it reuses), must have been consumed (their MMAs done).
struct F8Space {
    uint64_t starts[kF8D];
    uint32_t oldest = 0;
    __device__ __forceinline__ bool make_room(F8Smem& sm, uint32_t c, uint64_t st, uint64_t end)
    {
        while (oldest < c && (c - oldest >= (uint32_t)kF8D || starts[oldest % kF8D] + kF8Cap < end)) {
            if (!mbar_wait_or_abort(&sm.unit_free[oldest % kF8D], (oldest / kF8D) & 1, &sm.abort, kF8WaitNs))
                return false;
            oldest++;
        }
        starts[c % kF8D] = st;
        return true;
    }
};

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A E2M1 (5),
// B E4M3 (0), ue8m0 scales, fp32 accumulate, both K-major; the scale byte
// of step kb of a unit is byte kb of the TMEM word, for A and for B.
__device__ __forceinline__ uint32_t f8_idesc(uint32_t N, uint32_t kb)
{
    return (5u << 7) | (0u << 10) | ((N >> 3) << 17) | (1u << 23) | ((uint32_t)(kTileRows >> 4) << 24) |
           (kb << 29) | (kb << 4);
}

__device__ __forceinline__ void tc_mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::
            "r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

__device__ __forceinline__ void tc_ld32_nowait(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void f8_set_abort(const GroupArgs& a, F8Smem& sm)
{
    atomicOr(a.status, kStatusTimeout);
    sm.abort = 1;
}

// ------------------------------------------------------------ the E4M3 rows

// E4M3 codes of four consecutive elements under the ue8m0 byte s (255: NaN
// codes), round to nearest even, saturating at +-448 -- the rule of the
// activation quantizer (actquant.cu).
__device__ __forceinline__ uint32_t f8_codes4(const float (&v)[4], int s)
{
    if (s == 255) return 0x7F7F7F7Fu;
    const float down = __uint_as_float((uint32_t)(254 - s) << 23);     // 2^-(s-127)
    return (uint32_t)e4m3_rn_sat(v[0] * down) | ((uint32_t)e4m3_rn_sat(v[1] * down) << 8) |
           ((uint32_t)e4m3_rn_sat(v[2] * down) << 16) | ((uint32_t)e4m3_rn_sat(v[3] * down) << 24);
}

// The block's scale byte from a warp's four elements per lane (elements
// 4 lane .. 4 lane + 3; lanes past the block hold zeros).
__device__ __forceinline__ int f8_block_scale(const float (&v)[4])
{
    const bool nan = __any_sync(0xFFFFFFFFu, (v[0] != v[0]) || (v[1] != v[1]) || (v[2] != v[2]) || (v[3] != v[3]));
    const float amax = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    return nan ? 255 : ue8m0_for_amax_bits(amax);
}

// Stores a lane's four codes of row i of a group's unit (nb rows) and, from
// lane 0, the row's scale bytes into the unit's atoms.
__device__ __forceinline__ void f8_store_row(uint8_t* unit, uint8_t* atoms, int nb, int i, int lane, bool in,
                                             uint32_t codes, int s)
{
    if (in) {
        const int kb = lane >> 3, half = (lane >> 2) & 1;
        *reinterpret_cast<uint32_t*>(unit + (size_t)kb * nb * 32 + (i >> 3) * 256 + half * 128 + (i & 7) * 16 +
                                     (lane & 3) * 4) = codes;
    }
    if (lane == 0)
        *reinterpret_cast<uint32_t*>(atoms + (i >> 7) * kUnitSfBytes + (i & 31) * 16 + ((i & 127) >> 5) * 4) =
            (uint32_t)s * 0x01010101u;
}

// E2M1 rows (the E2M1 activation mode; kind::mxf4): a lane's four elements
// 4 lane .. 4 lane + 3 of a 128-element unit (lanes 8 b .. 8 b + 7 hold its
// 32-block b) under the block's ue8m0 byte -- the least 2^e with max |v| <=
// 6 * 2^e, the E2M1 activation rule -- rounded to nearest even, as two bytes
// (element 2i in the low nibble of byte i); s: the block's scale byte.
__device__ __forceinline__ uint32_t f4_codes4(const float (&v)[4], int& s)
{
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    s = e2m1_scale_byte(amax);
    const float down = exp2i(127 - s);
    return f32x2_to_e2m1x2(v[0] * down, v[1] * down) | (f32x2_to_e2m1x2(v[2] * down, v[3] * down) << 8);
}

// Stores a lane's two code bytes of row i of a group's unit (nb rows; per
// 64-K MMA m, the kind::mxf4 K-major layout: core matrices of 8 rows x 16 B)
// and, from lane 0, the row's four block scale bytes into the unit's atoms.
// Every lane of the warp takes part.
__device__ __forceinline__ void f4_store_row(uint8_t* unit, uint8_t* atoms, int nb, int i, int lane, bool in,
                                             uint32_t codes, int s)
{
    const int kb = lane >> 3;
    if (in)
        *reinterpret_cast<uint16_t*>(unit + (size_t)(kb >> 1) * nb * 32 + (i >> 3) * 256 + (kb & 1) * 128 +
                                     (i & 7) * 16 + (lane & 7) * 2) = (uint16_t)codes;
    const uint32_t s0 = (uint32_t)__shfl_sync(0xFFFFFFFFu, s, 0), s1 = (uint32_t)__shfl_sync(0xFFFFFFFFu, s, 8);
    const uint32_t s2 = (uint32_t)__shfl_sync(0xFFFFFFFFu, s, 16), s3 = (uint32_t)__shfl_sync(0xFFFFFFFFu, s, 24);
    if (lane == 0)
        *reinterpret_cast<uint32_t*>(atoms + (i >> 7) * kUnitSfBytes + (i & 31) * 16 + ((i & 127) >> 5) * 4) =
            s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// Where sorted slot P's rows go: its group, its row in the group, the
// group's first slot and rows of the MMA (from the route kernel's output).
struct F8Slot {
    int g, i, p0, nb;
};

__device__ __forceinline__ F8Slot f8_slot(const GroupArgs& a, int e, int P)
{
    const int off = a.offsets[e], gb = a.gbase[e], cnt = a.counts[e];
    const int gs = a.f8_gs;
    const int q = (P - off) / gs;
    F8Slot s;
    s.g = gb + q;
    s.i = P - off - q * gs;
    s.p0 = off + q * gs;
    s.nb = (min(gs, cnt - q * gs) + 15) & ~15;
    return s;
}

// grid (T, ceil(H / 1024)), 256 threads: warp w of CTA (t, y) quantizes the
// 128-block 8y + w of token t's row and stores it into each of the token's
// slots' groups.
__global__ void __launch_bounds__(256) k_f8prep(GroupArgs a)
{
    const int t = blockIdx.x, H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_red[33];
    __shared__ F8Slot s_sl[16];
    __shared__ int s_ok[16];

    pdl_wait();
    pdl_trigger();
    if (threadIdx.x < a.topk) {
        const int j = t * a.topk + threadIdx.x;
        const int P = a.inv[j], e = a.idx[j];
        const bool ok = P >= 0 && e >= 0 && e < a.E;
        s_ok[threadIdx.x] = ok;
        if (ok) s_sl[threadIdx.x] = f8_slot(a, e, P);
    }
    const float den = a.x_resid ? block_rms_den(a.x_resid + (size_t)t * H, H, a.eps, s_red) : 1.0f;
    __syncthreads();
    const int b = blockIdx.y * 8 + warp;
    if (b >= H / 128) return;
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const size_t i = (size_t)t * H + b * 128 + 4 * lane + q;
        v[q] = a.x_resid ? __bfloat162float(__float2bfloat16_rn(a.x_resid[i] / den))
                         : __uint_as_float((uint32_t)a.x_bf16[i] << 16);
    }
    if (a.act_e2m1) {
        int s;
        const uint32_t codes = f4_codes4(v, s);
        for (int kk = 0; kk < a.topk; kk++) {
            if (!s_ok[kk]) continue;
            const F8Slot sl = s_sl[kk];
            uint8_t* unit = a.xb8 + f8_group_rows(sl.p0, sl.g) * (H / 2) + (size_t)b * sl.nb * 64;
            uint8_t* atoms = a.xb8sf + ((size_t)sl.g * (H / 128) + b) * (2 * kUnitSfBytes);
            f4_store_row(unit, atoms, sl.nb, sl.i, lane, true, codes, s);
        }
        return;
    }
    const int s = f8_block_scale(v);
    const uint32_t codes = f8_codes4(v, s);
    for (int kk = 0; kk < a.topk; kk++) {
        if (!s_ok[kk]) continue;
        const F8Slot sl = s_sl[kk];
        uint8_t* unit = a.xb8 + f8_group_rows(sl.p0, sl.g) * H + (size_t)b * sl.nb * 128;
        uint8_t* atoms = a.xb8sf + ((size_t)sl.g * (H / 128) + b) * (2 * kUnitSfBytes);
        f8_store_row(unit, atoms, sl.nb, sl.i, lane, true, codes, s);
    }
}

// One warp per (sorted slot, 128-block of I): h of the slot quantized like x,
// into the down projection's B operand.
__global__ void __launch_bounds__(256) k_f8hquant(GroupArgs a)
{
    const int I = a.I, kgt = (I + 127) / 128;
    const int lane = threadIdx.x & 31;
    const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    pdl_wait();
    pdl_trigger();
    const int nvalid = a.offsets[a.E];
    if (wid >= (long long)nvalid * kgt) return;
    const int P = (int)(wid / kgt), u = (int)(wid % kgt);
    const int e = a.idx[a.perm[P]];
    const F8Slot sl = f8_slot(a, e, P);
    const int len = (u == kgt - 1 && (I & 127)) ? 64 : 128;
    const bool in = 4 * lane < len;
    float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (in) {
        const float4 h = __ldcg(reinterpret_cast<const float4*>(a.hraw + (size_t)P * I + (size_t)u * 128 + 4 * lane));
        v[0] = h.x;
        v[1] = h.y;
        v[2] = h.z;
        v[3] = h.w;
    }
    uint8_t* atoms = a.hb8sf + ((size_t)sl.g * kgt + u) * (2 * kUnitSfBytes);
    if (a.act_e2m1) {
        int s;
        const uint32_t codes = f4_codes4(v, s);
        uint8_t* unit = a.hb8 + f8_group_rows(sl.p0, sl.g) * (I / 2) + (size_t)u * sl.nb * 64;
        f4_store_row(unit, atoms, sl.nb, sl.i, lane, in, codes, s);
        return;
    }
    const int s = f8_block_scale(v);
    const uint32_t codes = f8_codes4(v, s);
    uint8_t* unit = a.hb8 + f8_group_rows(sl.p0, sl.g) * I + (size_t)u * sl.nb * 128;
    f8_store_row(unit, atoms, sl.nb, sl.i, lane, in, codes, s);
}

// ------------------------------------------------------------------ k_f8gemm

// Weight producer: every unit's packed weights into its span of the ring.
template <int PHASE>
__device__ void f8_produce_a(const GroupArgs& a, const F8Plan& p, F8Smem& sm, int njobs)
{
    F8Ring ring;
    F8Space sp;
    uint32_t c = 0;
    bool ok = true;
    for (int j = blockIdx.x; ok && j < njobs && !*(volatile int*)&sm.abort; j += gridDim.x) {
        const F8Job jb = f8_job<PHASE>(a, p, j);
        for (int u = 0; u < p.kgt; u++, c++) {
            const F8Unit U = f8_unit(p, jb, u);
            const uint64_t st = ring.take(U.size);
            if (!sp.make_room(sm, c, st, st + U.size)) {
                f8_set_abort(a, sm);
                ok = false;
                break;
            }
            uint64_t* bar = &sm.full_a[c % kF8D];
            if (jb.ok) {
                mbar_arrive_expect_tx(bar, U.abytes);
                bulk_g2s(sm.ring + st % kF8Cap, jb.a + (size_t)u * kUnitBytes, U.abytes, bar);
            } else {
                mbar_arrive(bar);                  // nothing to expand
            }
        }
    }
    // no copy may still be in flight into this CTA's memory at exit
    for (uint32_t m = c > (uint32_t)kF8D ? c - kF8D : 0; m < c; m++)
        if (!mbar_wait_bounded(&sm.full_a[m % kF8D], (m / kF8D) & 1, kF8WaitNs)) break;
}

// Activation producer: each unit's rows and scale atoms of the job's group
// beside its weights (once the previous kernel's stores are complete).
template <int PHASE>
__device__ void f8_produce_b(const GroupArgs& a, const F8Plan& p, F8Smem& sm, int njobs)
{
    pdl_wait();
    F8Ring ring;
    F8Space sp;
    uint32_t c = 0;
    bool ok = true;
    for (int j = blockIdx.x; ok && j < njobs && !*(volatile int*)&sm.abort; j += gridDim.x) {
        const F8Job jb = f8_job<PHASE>(a, p, j);
        for (int u = 0; u < p.kgt; u++, c++) {
            const F8Unit U = f8_unit(p, jb, u);
            const uint64_t st = ring.take(U.size);
            if (!sp.make_room(sm, c, st, st + U.size)) {
                f8_set_abort(a, sm);
                ok = false;
                break;
            }
            uint64_t* bar = &sm.full_b[c % kF8D];
            if (jb.ok) {
                uint8_t* dst = sm.ring + st % kF8Cap + U.abytes;
                mbar_arrive_expect_tx(bar, U.bbytes + U.sbytes);
                bulk_g2s(dst, jb.b + (size_t)u * jb.nb * p.bunit, U.bbytes, bar);
                bulk_g2s(dst + U.bbytes, jb.bsf + (size_t)u * (2 * kUnitSfBytes), U.sbytes, bar);
            } else {
                mbar_arrive(bar);
            }
        }
    }
    for (uint32_t m = c > (uint32_t)kF8D ? c - kF8D : 0; m < c; m++)
        if (!mbar_wait_bounded(&sm.full_b[m % kF8D], (m / kF8D) & 1, kF8WaitNs)) break;
}

// Expanders (128 threads): each unit's packed codes into the padded layout of
// a stage of expanded weights -- blob chunk (step m, row group, core matrix c,
// row) of 32 codes becomes rows of 16 codes in step kb = 2m + c, halves 0 and
// 1 -- and its scale atom beside them.
template <int PHASE>
__device__ void f8_expand(const GroupArgs& a, const F8Plan& p, F8Smem& sm, int njobs, int et)
{
    F8Ring ring;
    uint32_t c = 0;
    const int lane = et & 31;
    for (int j = blockIdx.x; j < njobs && !*(volatile int*)&sm.abort; j += gridDim.x) {
        const F8Job jb = f8_job<PHASE>(a, p, j);
        for (int u = 0; u < p.kgt; u++, c++) {
            const F8Unit U = f8_unit(p, jb, u);
            const uint64_t st = ring.take(U.size);
            const uint32_t sp = c % kF8Pad;
            // the stage's previous unit (c - kF8Pad) must have been multiplied
            const uint32_t prev = c - kF8Pad;
            long long tw = F8_NOW();
            bool ok = mbar_wait_or_abort(&sm.full_a[c % kF8D], (c / kF8D) & 1, &sm.abort, kF8WaitNs);
            if (et == 0) F8_ACC(17, tw);
            tw = F8_NOW();
            ok = ok && (c < (uint32_t)kF8Pad ||
                        mbar_wait_or_abort(&sm.unit_free[prev % kF8D], (prev / kF8D) & 1, &sm.abort, kF8WaitNs));
            if (et == 0) F8_ACC(18, tw);
            tw = F8_NOW();
            if (!ok) {
                f8_set_abort(a, sm);
                return;
            }
            if (jb.ok) {
                const uint8_t* src = sm.ring + st % kF8Cap;
                uint8_t* dst = sm.pad[sp];
                const int nchunks = U.half ? 256 : 512;
#pragma unroll 4
                for (int q = et; q < nchunks; q += 128) {
                    const uint4 v = *reinterpret_cast<const uint4*>(src + q * 16);
                    const int kb = 2 * (q >> 8) + ((q >> 3) & 1), rg = (q >> 4) & 15, r8 = q & 7;
                    uint8_t* d = dst + kb * 4096 + rg * 256 + r8 * 16;
                    *reinterpret_cast<uint4*>(d) = make_uint4(v.x, v.y, 0u, 0u);
                    *reinterpret_cast<uint4*>(d + 128) = make_uint4(v.z, v.w, 0u, 0u);
                }
                const uint8_t* atom = src + (U.half ? kMmaCodeBytes : kUnitCodeBytes);
                reinterpret_cast<uint32_t*>(dst + kF8PadBytes)[et] = reinterpret_cast<const uint32_t*>(atom)[et];
                // the tensor core reads these through the async proxy
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.pad_ready[sp]);
            if (et == 0) F8_ACC(19, tw);
        }
    }
}

// Scale stager of the wide form (one thread): per unit, once its weights are
// expanded (kind::mxf8f6f4) or have landed (kind::mxf4; the scale slot's
// previous unit multiplied) and its activation rows are in, the unit's A
// scale atom and the group's B atoms to the unit's scale slot (tcgen05.cp),
// committed to sf_ready: the issuers then wait once per unit and only issue
// MMAs (one thread issues a tcgen05 instruction every ~110 cycles).
template <int PHASE, int KIND>
__device__ void f8_stage_sf(const GroupArgs& a, const F8Plan& p, F8Smem& sm, int njobs, uint32_t tmem)
{
    using Tm = F8Tm<1>;
    F8Ring ring;
    uint32_t c = 0;
    bool ok = true;
    for (int j = blockIdx.x; ok && j < njobs; j += gridDim.x) {
        const F8Job jb = f8_job<PHASE>(a, p, j);
        for (int u = 0; u < p.kgt; u++, c++) {
            const F8Unit U = f8_unit(p, jb, u);
            const uint64_t st = ring.take(U.size);
            const uint32_t sp = c % kF8Pad;
            long long tw = F8_NOW();
            if (KIND == 0) {
                ok = mbar_wait_or_abort(&sm.pad_ready[sp], (c / kF8Pad) & 1, &sm.abort, kF8WaitNs);
            } else {
                ok = mbar_wait_or_abort(&sm.full_a[c % kF8D], (c / kF8D) & 1, &sm.abort, kF8WaitNs);
                const uint32_t prev = c - kF8Pad;
                if (ok && c >= (uint32_t)kF8Pad)
                    ok = mbar_wait_or_abort(&sm.unit_free[prev % kF8D], (prev / kF8D) & 1, &sm.abort, kF8WaitNs);
            }
            F8_ACC(14, tw);
            tw = F8_NOW();
            ok = ok && mbar_wait_or_abort(&sm.full_b[c % kF8D], (c / kF8D) & 1, &sm.abort, kF8WaitNs);
            F8_ACC(15, tw);
            tw = F8_NOW();
            if (!ok) break;
            tc_fence_after();
            if (jb.ok) {
                const uint8_t* ring_u = sm.ring + st % kF8Cap;
                const uint8_t* pb = ring_u + U.abytes;
                const uint8_t* atom_a = KIND == 0 ? sm.pad[sp] + kF8PadBytes
                                                  : ring_u + (U.half ? kMmaCodeBytes : kUnitCodeBytes);
                const uint32_t sf = tmem + Tm::sf(0, c);
                tc_cp_sf(sf, umma_desc(smem_u32(atom_a), 16, 128));
                tc_cp_sf(sf + 4, umma_desc(smem_u32(pb + U.bbytes), 16, 128));
                if (jb.nb > 128) tc_cp_sf(sf + 8, umma_desc(smem_u32(pb + U.bbytes + kUnitSfBytes), 16, 128));
            }
            tc_commit(&sm.sf_ready[sp]);
            F8_ACC(16, tw);
        }
    }
    if (!ok) f8_set_abort(a, sm);
    tc_commit(&sm.drain[2]);
    mbar_wait_bounded(&sm.drain[2], 0, kF8WaitNs);
}

// MMA issuer of the wide form (one thread): per unit, once its scale slot is
// filled, one MMA per 32-K step (kind::mxf8f6f4; 64-K steps for kind::mxf4)
// over all the group's rows of B into the job's accumulator; the unit's span
// of the ring, its expanded-weight stage and its scale slot are freed by the
// commit after them, the accumulator handed to the epilogue after the job's
// last unit.
template <int PHASE, int KIND>
__device__ void f8_issue_wide(const GroupArgs& a, const F8Plan& p, F8Smem& sm, int njobs, uint32_t tmem)
{
    using Tm = F8Tm<1>;
    F8Ring ring;
    uint32_t c = 0, jl = 0;
    bool abort = false;
    for (int j = blockIdx.x; j < njobs && !abort; j += gridDim.x, jl++) {
        const F8Job jb = f8_job<PHASE>(a, p, j);
        const uint32_t buf = jl & 1;
        long long tw = F8_NOW();
        if (!mbar_wait_or_abort(&sm.acc_empty[buf], ((jl >> 1) & 1) ^ 1, &sm.abort, kF8WaitNs)) {
            abort = true;
            break;
        }
        F8_ACC(3, tw);
        const int n = jb.nb;
        const uint32_t acc = tmem + Tm::acc(0, buf);
        bool first = true;
        for (int u = 0; u < p.kgt; u++, c++) {
            const F8Unit U = f8_unit(p, jb, u);
            const uint64_t st = ring.take(U.size);
            const uint32_t sp = c % kF8Pad;
            tw = F8_NOW();
            if (!mbar_wait_or_abort(&sm.sf_ready[sp], (c / kF8Pad) & 1, &sm.abort, kF8WaitNs)) {
                abort = true;
                break;
            }
            F8_ACC(0, tw);
            tw = F8_NOW();
            tc_fence_after();
            if (jb.ok) {
                const uint8_t* pb = sm.ring + st % kF8Cap + U.abytes;
                // B's scale atoms: rows 0-127 at sf + 4, rows 128- at sf + 8 (the MMA
                // over all the rows reads both)
                const uint32_t sf = tmem + Tm::sf(0, c), sfb = sf + 4;
                if (KIND == 0) {
                    // E2M1 weights (expanded) x E4M3 rows: K = 32 per MMA, scale byte kb
                    const uint8_t* pa = sm.pad[sp];
                    const int steps = U.half ? 2 : 4;
                    for (int kb = 0; kb < steps; kb++) {
                        const uint64_t ad = umma_desc(smem_u32(pa + kb * 4096), 128, 256);
                        const uint64_t bd = umma_desc(smem_u32(pb + kb * jb.nb * 32), 128, 256);
                        tc_mma_mxf8f6f4(acc, ad, bd, f8_idesc((uint32_t)n, (uint32_t)kb), sf, sfb,
                                        (!first || kb) ? 1u : 0u);
                    }
                } else {
                    // E2M1 weights (packed, as the blob holds them) x E2M1 rows: K = 64
                    // per MMA, scale bytes 2m, 2m + 1
                    const uint8_t* pa = sm.ring + st % kF8Cap;
                    const uint32_t idesc = mxf4_idesc(kTileRows, (uint32_t)n);
                    const int steps = U.half ? 1 : 2;
                    for (int m = 0; m < steps; m++) {
                        const uint64_t ad = umma_desc(smem_u32(pa + m * kMmaCodeBytes), 128, 256);
                        const uint64_t bd = umma_desc(smem_u32(pb + m * jb.nb * 32), 128, 256);
                        tc_mma_mxf4(acc, ad, bd, mxf4_idesc_sf(idesc, 2u * (uint32_t)m), sf, sfb,
                                    (!first || m) ? 1u : 0u);
                    }
                }
                first = false;
            }
            tc_commit(&sm.unit_free[c % kF8D]);
            F8_ACC(4, tw);
#ifdef MOE_F8_TRACE
            atomicAdd(&g_f8_trace[5][blockIdx.x], 1ull);
#endif
        }
        if (abort) break;
        tc_commit(&sm.acc_full[buf]);
    }
    if (abort) f8_set_abort(a, sm);
    // none of this thread's tensor-core operations may be in flight when the
    // TMEM is freed or the CTA exits
    tc_commit(&sm.drain[0]);
    mbar_wait_bounded(&sm.drain[0], 0, kF8WaitNs);
}

// MMA issuer i of the narrow form (one thread of three): per unit c with
// c % 3 == i, the scale sets of A and B to its own scale slot, then one MMA
// per 32-K step into its accumulator; a unit's span of the ring and its
// expanded-weight stage are freed by the commit after them, the accumulator
// handed to the epilogue (count 3) after the job's last unit.
template <int PHASE, int KIND>
__device__ void f8_issue_narrow(const GroupArgs& a, const F8Plan& p, F8Smem& sm, int njobs, uint32_t tmem, int ii)
{
    constexpr int NI = 3;
    using Tm = F8Tm<NI>;
    F8Ring ring;
    uint32_t c = 0, jl = 0;
    bool abort = false;
    for (int j = blockIdx.x; j < njobs && !abort; j += gridDim.x, jl++) {
        const F8Job jb = f8_job<PHASE>(a, p, j);
        const uint32_t buf = jl & 1;
        // the epilogue has read this accumulator's previous job (every issuer
        // waits, also one without units in this job, so that none can arrive
        // for a later job before this one's phase is complete)
        long long tw = F8_NOW();
        if (!mbar_wait_or_abort(&sm.acc_empty[buf], ((jl >> 1) & 1) ^ 1, &sm.abort, kF8WaitNs)) {
            abort = true;
            break;
        }
        F8_ACC(3, tw);
        bool first = true;
        for (int u = 0; u < p.kgt; u++, c++) {
            const F8Unit U = f8_unit(p, jb, u);
            const uint64_t st = ring.take(U.size);
            if ((int)(c % NI) != ii) continue;
            const uint32_t sp = c % kF8Pad;
            const uint32_t reuse = (uint32_t)(NI * Tm::kSlots);      // the scale slot's previous unit
            tw = F8_NOW();
            // kind::mxf8f6f4: the expanded weights; kind::mxf4: the packed ones in the ring
            bool ok = KIND == 0 ? mbar_wait_or_abort(&sm.pad_ready[sp], (c / kF8Pad) & 1, &sm.abort, kF8WaitNs)
                                : mbar_wait_or_abort(&sm.full_a[c % kF8D], (c / kF8D) & 1, &sm.abort, kF8WaitNs);
            F8_ACC(0, tw);
            tw = F8_NOW();
            ok = ok && mbar_wait_or_abort(&sm.full_b[c % kF8D], (c / kF8D) & 1, &sm.abort, kF8WaitNs);
            F8_ACC(1, tw);
            tw = F8_NOW();
            if (ok && c >= reuse)
                ok = mbar_wait_or_abort(&sm.unit_free[(c - reuse) % kF8D], ((c - reuse) / kF8D) & 1, &sm.abort,
                                        kF8WaitNs);
            F8_ACC(2, tw);
            tw = F8_NOW();
            if (!ok) {
                abort = true;
                break;
            }
            tc_fence_after();
            if (jb.ok) {
                const uint8_t* pb = sm.ring + st % kF8Cap + U.abytes;
                const uint32_t sf = tmem + Tm::sf(ii, c);
                const uint32_t acc = tmem + Tm::acc(ii, buf);
                if (KIND == 0) {
                    const uint8_t* pa = sm.pad[sp];
                    tc_cp_sf(sf, umma_desc(smem_u32(pa + kF8PadBytes), 16, 128));
                    tc_cp_sf(sf + 4, umma_desc(smem_u32(pb + U.bbytes), 16, 128));
                    const int steps = U.half ? 2 : 4;
                    for (int kb = 0; kb < steps; kb++) {
                        const uint64_t ad = umma_desc(smem_u32(pa + kb * 4096), 128, 256);
                        const uint64_t bd = umma_desc(smem_u32(pb + kb * jb.nb * 32), 128, 256);
                        tc_mma_mxf8f6f4(acc, ad, bd, f8_idesc((uint32_t)jb.nb, (uint32_t)kb), sf, sf + 4,
                                        (!first || kb) ? 1u : 0u);
                    }
                } else {
                    const uint8_t* pa = sm.ring + st % kF8Cap;
                    tc_cp_sf(sf, umma_desc(smem_u32(pa + (U.half ? kMmaCodeBytes : kUnitCodeBytes)), 16, 128));
                    tc_cp_sf(sf + 4, umma_desc(smem_u32(pb + U.bbytes), 16, 128));
                    const uint32_t idesc = mxf4_idesc(kTileRows, (uint32_t)jb.nb);
                    const int steps = U.half ? 1 : 2;
                    for (int m = 0; m < steps; m++) {
                        const uint64_t ad = umma_desc(smem_u32(pa + m * kMmaCodeBytes), 128, 256);
                        const uint64_t bd = umma_desc(smem_u32(pb + m * jb.nb * 32), 128, 256);
                        tc_mma_mxf4(acc, ad, bd, mxf4_idesc_sf(idesc, 2u * (uint32_t)m), sf, sf + 4,
                                    (!first || m) ? 1u : 0u);
                    }
                }
                first = false;
            }
            tc_commit(&sm.unit_free[c % kF8D]);
            F8_ACC(4, tw);
#ifdef MOE_F8_TRACE
            atomicAdd(&g_f8_trace[5][blockIdx.x], 1ull);
#endif
        }
        if (abort) break;
        tc_commit(&sm.acc_full[buf]);
    }
    if (abort) f8_set_abort(a, sm);
    tc_commit(&sm.drain[ii]);
    mbar_wait_bounded(&sm.drain[ii], 0, kF8WaitNs);
}

// Epilogue (four warps; warp q of the TMEM lane quadrants holds rows 32q..):
// the issuers' accumulators of the job added in issuer order, then gate/up ->
// h = silu(g) u of the tile's 64 outputs per slot (the up rows reach the gate
// rows' warps through shared memory); down -> the tile's 128 outputs per slot.
// 32 slots at a time.
template <int PHASE, int NI>
__device__ void f8_epilogue(const GroupArgs& a, const F8Plan& p, F8Smem& sm, int njobs, uint32_t tmem, int q,
                            int lane)
{
    using Tm = F8Tm<NI>;
    pdl_wait();
    uint32_t jl = 0;
    for (int j = blockIdx.x; j < njobs; j += gridDim.x, jl++) {
        const F8Job jb = f8_job<PHASE>(a, p, j);
        const uint32_t buf = jl & 1;
        long long tw = F8_NOW();
        if (!mbar_wait_or_abort(&sm.acc_full[buf], (jl >> 1) & 1, &sm.abort, kF8WaitNs)) {
            f8_set_abort(a, sm);
            return;
        }
        if (q == 0 && lane == 0) F8_ACC(6, tw);
        tw = F8_NOW();
        tc_fence_after();
        // issuer i holds part of this job if one of its units c = jl kgt + u has c % NI == i
        const uint32_t c0 = jl * (uint32_t)p.kgt;
        const uint32_t lq = (uint32_t)(32 * q) << 16;
        auto holds = [&](int ii) {
            return !((uint32_t)p.kgt < (uint32_t)NI && (uint32_t)((ii - (int)(c0 % NI) + NI) % NI) >= (uint32_t)p.kgt);
        };
        for (int n0 = 0; n0 < jb.nt; n0 += 32) {
            const int ncol = min(32, jb.nt - n0);
            float v[32];
            long long tc = F8_NOW();
#pragma unroll
            for (int i = 0; i < 32; i++) v[i] = 0.0f;
            if (jb.ok && Tm::kAccs == 1) {
                uint32_t r[32];
                tc_ld32_nowait(tmem + lq + Tm::acc(0, buf) + (uint32_t)n0, r);
                tc_wait_ld();
                tc_ld_fence_regs<32>(r);
#pragma unroll
                for (int i = 0; i < 32; i++) v[i] += __uint_as_float(r[i]);
            } else if (jb.ok) {
#pragma unroll
                for (int ii = 0; ii < NI; ii++) {
                    if (!holds(ii)) continue;
                    uint32_t r[32];
                    tc_ld32_nowait(tmem + lq + Tm::acc(ii, buf) + (uint32_t)n0, r);
                    tc_wait_ld();
                    tc_ld_fence_regs<32>(r);
#pragma unroll
                    for (int i = 0; i < 32; i++) v[i] += __uint_as_float(r[i]);
                }
            }
            if (q == 0 && lane == 0) F8_ACC(8, tc);
            tc = F8_NOW();
            if (PHASE == 0) {
                // gate warp q and up warp q + 2 hold the same 32 outputs: the gate
                // warp hands over its slots 16-31, the up warp its slots 0-15, and
                // each makes h for 16 slots (all 16 products first, so that their
                // exponentials and quotients overlap, then the stores)
                const int pair = q & 1, base = q >= 2 ? 16 : 0;
                float* hrow = a.hraw + (size_t)(jb.p0 + n0 + base) * a.I + (size_t)jb.tile * 64 + 32 * pair + lane;
                float hv[16];
                if (q >= 2) {
#pragma unroll
                    for (int i = 0; i < 16; i++) sm.xch[pair][i][lane] = v[i];
                    named_sync(2 + pair, 64);
#pragma unroll
                    for (int i = 0; i < 16; i++) hv[i] = silu(sm.xch[pair][16 + i][lane]) * v[16 + i];
                } else {
#pragma unroll
                    for (int i = 16; i < 32; i++) sm.xch[pair][i][lane] = v[i];
                    named_sync(2 + pair, 64);
#pragma unroll
                    for (int i = 0; i < 16; i++) hv[i] = silu(v[i]) * sm.xch[pair][i][lane];
                }
#pragma unroll
                for (int i = 0; i < 16; i++)
                    if (base + i < ncol) hrow[(size_t)i * a.I] = hv[i];
                if (q == 0 && lane == 0) F8_ACC(11, tc);
                tc = F8_NOW();
                named_sync(2 + pair, 64);
                if (q == 0 && lane == 0) F8_ACC(12, tc);
            } else {
                float* orow = a.obuf + (size_t)(jb.p0 + n0) * a.H + (size_t)jb.tile * kTileRows + 32 * q + lane;
#pragma unroll
                for (int i = 0; i < 32; i++)
                    if (i < ncol) orow[(size_t)i * a.H] = v[i];
                if (q == 0 && lane == 0) F8_ACC(13, tc);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
        if (q == 0 && lane == 0) F8_ACC(7, tw);
    }
}

template <int PHASE, int NI, int KIND>
__global__ void __launch_bounds__(kF8Threads, 1) k_f8gemm(GroupArgs a, F8Plan p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    F8Smem& sm = *reinterpret_cast<F8Smem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kF8D; s++) {
            mbar_init(&sm.full_a[s], 1);
            mbar_init(&sm.full_b[s], 1);
            mbar_init(&sm.unit_free[s], 1);
        }
        for (int s = 0; s < kF8Pad; s++) {
            mbar_init(&sm.pad_ready[s], 4);
            mbar_init(&sm.sf_ready[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&sm.acc_full[b], NI);
            mbar_init(&sm.acc_empty[b], 4);
        }
        for (int i = 0; i < kF8MaxIssuers; i++) mbar_init(&sm.drain[i], 1);
        sm.abort = 0;
        mbar_fence_init();
    }
    if (warp == kF8WarpMma0) tmem_alloc(&sm.tmem, kF8TmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    const uint32_t tmem = sm.tmem;
    // the group table was written by the route kernel, which completed before
    // the kernel ahead of this one passed its own dependency wait
    const int njobs = p.ntiles * __ldcg(&a.gbase[a.E]);

    if (warp == kF8WarpProdA) {
        if (lane == 0) f8_produce_a<PHASE>(a, p, sm, njobs);
        return;
    }
    if (warp == kF8WarpProdB) {
        if (lane == 0) f8_produce_b<PHASE>(a, p, sm, njobs);
        return;
    }
    if (warp >= kF8WarpExp0 && warp < kF8WarpEpi0) {
        // kind::mxf4 multiplies the packed weights where they landed
        if (KIND == 0) f8_expand<PHASE>(a, p, sm, njobs, threadIdx.x - kF8WarpExp0 * 32);
        return;
    }
    if (warp < kF8WarpExp0) {
        const int ii = warp - kF8WarpMma0;
        if (lane == 0) {
            if (NI == 1) {
                if (ii == 0) f8_issue_wide<PHASE, KIND>(a, p, sm, njobs, tmem);
                else if (ii == 2) f8_stage_sf<PHASE, KIND>(a, p, sm, njobs, tmem);
            } else {
                f8_issue_narrow<PHASE, KIND>(a, p, sm, njobs, tmem, ii);
            }
        }
        __syncwarp();
    } else {
        f8_epilogue<PHASE, NI>(a, p, sm, njobs, tmem, warp & 3, lane);
    }
    // the issuer and epilogue warps meet here before the tensor memory is released
    tc_fence_before();
    named_sync(1, (kF8MaxIssuers + 4) * 32);
    tc_fence_after();
    if (warp == kF8WarpMma0) tmem_dealloc(tmem, kF8TmemCols);
}

F8Plan f8plan(const GroupArgs& a, int phase)
{
    const ExpertLayout L = make_expert_layout(a.H, a.I);
    const MatLayout& m = phase ? L.dn : L.gu;
    F8Plan p;
    p.ntiles = m.tiles;
    p.kgt = m.kgt();
    p.half = m.kg_half;
    p.K = m.k;
    p.bunit = a.act_e2m1 ? 64 : 128;
    p.tile_bytes = m.tile_bytes();
    p.mat_off = phase ? L.dn_off : L.gu_off;
    return p;
}

cudaError_t f8launch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void** args)
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

constexpr size_t f8_smem() { return sizeof(F8Smem); }

}  // namespace

F8WorkspaceSizes f8_workspace_sizes(int T, int topk, int E, int H, int I)
{
    F8WorkspaceSizes s{};
    const size_t n = (size_t)T * topk;
    const size_t G = (size_t)max_groups((int)n, E, kF8GroupSlotsNarrow);   // the smaller groups: more of them
    s.xb8 = (n + 16 * G) * (size_t)H;
    s.xb8sf = G * (size_t)(H / 128) * 2 * kUnitSfBytes;
    s.hb8 = (n + 16 * G) * (size_t)I;
    s.hb8sf = G * (size_t)((I + 127) / 128) * 2 * kUnitSfBytes;
    return s;
}

cudaError_t f8_init_device()
{
    cudaError_t e = cudaSuccess;
    for (const void* fn : {(const void*)k_f8gemm<0, 1, 0>, (const void*)k_f8gemm<1, 1, 0>,
                           (const void*)k_f8gemm<0, 3, 0>, (const void*)k_f8gemm<1, 3, 0>,
                           (const void*)k_f8gemm<0, 1, 1>, (const void*)k_f8gemm<1, 1, 1>})
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f8_smem());
    return e;
}

cudaError_t launch_f8_layer(const GroupArgs& a0, cudaStream_t s, bool pdl, Profiler* prof)
{
    GroupArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    a.o_unweighted = 1;                       // the combine applies the routing weights
    // the form: groups of up to 224 slots, one issuer and a scale stager where
    // experts hold many slots on average (the MMAs are large: tensor-bound
    // shapes), else groups of up to 64 and three issuers (HBM-bound decode
    // batches, where one thread could not issue the small MMAs as fast as the
    // weights arrive)
    // (the E2M1 mode, kind::mxf4, has the wide form only)
    const bool wide = a.act_e2m1 || (long long)a.T * a.topk >= 128LL * a.E;
    a.f8_gs = wide ? kF8GroupSlots : kF8GroupSlotsNarrow;
    const bool chain = pdl && !prof;
    cudaError_t err;
    RouteArgs ra{a.idx, a.T * a.topk, a.E, a.counts, a.offsets, a.perm, a.inv, a.status, a.gbase, a.groups,
                 a.f8_gs};
    if (prof) prof->begin(kPhaseRoute, s);
    err = launch_route(ra, s, chain);
    if (prof) prof->end(s);
    if (err != cudaSuccess) return err;
    void* args1[] = {&a};
    if (prof) prof->begin(kPhasePrep, s);
    err = f8launch((const void*)k_f8prep, dim3(a.T, (a.H / 128 + 7) / 8), dim3(256), 0, s, chain, args1);
    if (prof) prof->end(s);
    if (err != cudaSuccess) return err;
    F8Plan p0 = f8plan(a, 0), p1 = f8plan(a, 1);
    void* args_gu[] = {&a, &p0};
    if (prof) prof->begin(kPhaseGateUp, s);
    const void* gu = a.act_e2m1 ? (const void*)k_f8gemm<0, 1, 1>
                     : wide        ? (const void*)k_f8gemm<0, 1, 0>
                                   : (const void*)k_f8gemm<0, 3, 0>;
    const void* dn = a.act_e2m1 ? (const void*)k_f8gemm<1, 1, 1>
                     : wide        ? (const void*)k_f8gemm<1, 1, 0>
                                   : (const void*)k_f8gemm<1, 3, 0>;
    err = f8launch(gu, dim3((unsigned)a.sms), dim3(kF8Threads), f8_smem(), s, chain, args_gu);
    if (prof) prof->end(s);
    if (err != cudaSuccess) return err;
    const long long hw = (long long)a.T * a.topk * ((a.I + 127) / 128);
    if (prof) prof->begin(kPhaseActQuant, s);
    err = f8launch((const void*)k_f8hquant, dim3((unsigned)((hw + 7) / 8)), dim3(256), 0, s, chain, args1);
    if (prof) prof->end(s);
    if (err != cudaSuccess) return err;
    void* args_dn[] = {&a, &p1};
    if (prof) prof->begin(kPhaseGateUp, s);     // the layer's MMA kernels, both projections
    err = f8launch(dn, dim3((unsigned)a.sms), dim3(kF8Threads), f8_smem(), s, chain, args_dn);
    if (prof) prof->end(s);
    if (err != cudaSuccess) return err;
    if (prof) prof->begin(kPhaseDown, s);
    err = launch_group_combine(a, s, chain);
    if (prof) prof->end(s);
    return err;
}

}  // namespace moe

#ifdef MOE_F8_TRACE
// debug builds only: the issuer's wait and issue cycles per CTA (cleared after the read)
extern "C" int moe_debug_f8_trace(unsigned long long* dst, size_t bytes)
{
    const size_t n = bytes < sizeof(moe::g_f8_trace) ? bytes : sizeof(moe::g_f8_trace);
    if (cudaMemcpyFromSymbol(dst, moe::g_f8_trace, n) != cudaSuccess) return 1;
    static unsigned long long zero[20][1024];
    return cudaMemcpyToSymbol(moe::g_f8_trace, zero, sizeof(zero)) == cudaSuccess ? 0 : 1;
}
#endif
