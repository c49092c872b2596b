// common.cuh -- small device helpers (inline PTX for sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// Streaming read-only loads: weights are read once per call, so keep them out of L1.
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 2^e as fp32 for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Programmatic dependent launch: let the next grid start its prologue, and wait
// for the previous grid's results.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// silu(g) = g / (1 + e^-g).  The quotient by __fdividef: within 2 ulp while the
// divisor is below 2^126, and 0 beyond (g < -87: silu(g) is below 1e-36 in
// magnitude there), where an IEEE division would take its slow path for the
// huge or infinite divisor, at hundreds of cycles per value.
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + expf(-g)); }

// RMSNorm (unit weight) denominator sqrt(mean(x^2) + eps) of one row of H
// floats, by the whole CTA (every thread calls it; at most 32 warps): the sum
// of squares in a fixed order -- eight loads in flight per thread, added as
// one element at a time (i = tid, tid + blockDim, ...), then the warps' sums
// in warp order.  s_red: 33 floats of shared memory.
__device__ __forceinline__ float block_rms_den(const float* xr, int H, float eps, float* s_red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float ss = 0.0f;
    for (int i0 = threadIdx.x; i0 < H; i0 += 8 * (int)blockDim.x) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int i = i0 + q * (int)blockDim.x;
            v[q] = i < H ? __ldcg(xr + i) : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < 8; q++)
            if (i0 + q * (int)blockDim.x < H) ss = fmaf(v[q], v[q], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) s_red[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += s_red[w];
        s_red[32] = sqrtf(tot / (float)H + eps);
    }
    __syncthreads();
    return s_red[32];
}

// ---------------------------------------------------------------- mbarrier / bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Deadlines of the bounded waits count SM clock cycles (a per-SM counter that
// costs nothing to read), at 2 cycles per nanosecond: a wait gives up after
// its limit at 2 GHz and proportionally later at lower clocks.
__device__ __forceinline__ uint64_t wait_clock() { return (uint64_t)clock64(); }
__device__ __forceinline__ uint64_t wait_cycles(uint64_t ns) { return 2 * ns; }

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Adds tx bytes to the current phase of `bar` without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended in hardware for up to
// hint_ns while the phase is not complete (it resumes as soon as it
// completes), so that waiting threads leave the issue slots to working warps.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

constexpr uint32_t kWaitSleepNs = 2000;   // suspend-time hint of one try in the bounded waits

// Wait for the phase of `bar` with the given parity to complete, for at most
// limit_ns of wall time.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = wait_clock(), lim = wait_cycles(limit_ns);
#ifdef MOE_WAIT_BACKOFF
    while (!mbar_try_wait(bar, parity)) {
        __nanosleep(64);
        if (wait_clock() - t0 > lim) return false;
    }
#else
    while (!mbar_try_wait_sleep(bar, parity, kWaitSleepNs))
        if (wait_clock() - t0 > lim) return false;
#endif
    return true;
}

// As mbar_wait_bounded, but also gives up as soon as *abort is set.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, const int* abort,
                                                   uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = wait_clock(), lim = wait_cycles(limit_ns);
#ifdef MOE_WAIT_BACKOFF
    while (!mbar_try_wait(bar, parity)) {
        __nanosleep(64);
        if (*(const volatile int*)abort || wait_clock() - t0 > lim) return false;
    }
#else
    while (!mbar_try_wait_sleep(bar, parity, kWaitSleepNs))
        if (*(const volatile int*)abort || wait_clock() - t0 > lim) return false;
#endif
    return true;
}

// Bulk copy global -> this CTA's shared memory, completing tx bytes on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of 8
// rows x 16 bytes stored contiguously (128 B); lbo = byte distance between
// core matrices adjacent along K, sbo = between adjacent 8-row groups.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;     // descriptor version of this MMA generation
    return d;                   // base offset 0, no swizzle
}

// Instruction descriptor of kind::mxf4 block-scaled MMA: E2M1 x E2M1, ue8m0
// scales, fp32 accumulate, both operands K-major.
__host__ __device__ constexpr uint32_t mxf4_idesc(uint32_t M, uint32_t N)
{
    return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

// scale-factor byte selectors (which two bytes of the 32-bit TMEM word)
__device__ __forceinline__ uint32_t mxf4_idesc_sf(uint32_t idesc, uint32_t sf_id)
{
    return idesc | (sf_id << 29) | (sf_id << 4);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 128 bits from shared memory (a 512-byte scale-factor atom) to
// TMEM, replicated to all four lane quadrants.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Warp-collective: 16 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// Warp-collective, without waiting: 64 / 16 consecutive 32-bit TMEM columns
// of this warp's 32 lanes into raw registers; tc_wait_ld() completes every
// load issued so far (the registers may not be read before it).
__device__ __forceinline__ void tc_ld64_nowait(uint32_t taddr, uint32_t (&r)[64])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,"
        "%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
}

__device__ __forceinline__ void tc_ld16_nowait(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Marks registers a non-waiting TMEM load wrote as read only after
// tc_wait_ld(): each passes through an empty volatile asm placed after it, so
// the compiler cannot move a use above the wait.
template <int N>
__device__ __forceinline__ void tc_ld_fence_regs(uint32_t (&r)[N])
{
#pragma unroll
    for (int i = 0; i < N; i++) asm volatile("" : "+r"(r[i]));
}

// Warp-collective: one 32-bit TMEM column of this warp's 32 lanes from r;
// tc_wait_st() completes the stores issued so far.
__device__ __forceinline__ void tc_st1(uint32_t taddr, float v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(__float_as_uint(v)) : "memory");
}

__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Warp-collective: 8 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = __uint_as_float(r[i]);
}

// Two fp32 values to one byte of two E2M1 codes (lo -> low nibble),
// round to nearest even, saturating at +-6.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi)
{
    uint16_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// E2M1 pair (low byte of w) back to two fp32 values.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t w)
{
    uint32_t h;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
        : "=r"(h)
        : "r"(w));
    __half2 hv = *reinterpret_cast<__half2*>(&h);
    return __half22float2(hv);
}

// The ue8m0 scale byte of an E4M3 block: k + 127 with k the least integer
// such that amax <= 448 * 2^k, read off amax's bits (amax = m * 2^E, m in
// [1, 2): k = E - 8 if m <= 1.75, else E - 7; 448 = 1.75 * 2^8).  A zero
// maximum gives k = 0, a non-finite one the NaN byte 255.
__device__ __forceinline__ int ue8m0_for_amax_bits(float amax)
{
    if (amax == 0.0f) return 127;
    const uint32_t b = __float_as_uint(amax);
    const int ef = (int)((b >> 23) & 0xFF);
    if (ef == 0xFF) return 255;
    int E;
    uint32_t mant;
    if (ef == 0) {                       // subnormal: amax = m * 2^-149
        const uint32_t m = b & 0x7FFFFF;
        const int p = 31 - __clz(m);     // leading one
        E = p - 149;
        mant = (m << (23 - p)) & 0x7FFFFF;
    } else {
        E = ef - 127;
        mant = b & 0x7FFFFF;
    }
    int k = (mant <= 0x600000u) ? E - 8 : E - 7;
    k = k < -127 ? -127 : (k > 127 ? 127 : k);
    return k + 127;
}

// E4M3, round to nearest even, saturating at +-448.
__device__ __forceinline__ uint8_t e4m3_rn_sat(float v)
{
    return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// v quantized to E4M3 under the scale byte s (1 <= s <= 254) and taken back:
// code(v * 2^(127 - s)) * 2^(s - 127), both scalings exact.
__device__ __forceinline__ float e4m3_quant_dequant(float v, int s)
{
    const float down = __uint_as_float((uint32_t)(254 - s) << 23);     // 2^(127 - s)
    const __half_raw hr = __nv_cvt_fp8_to_halfraw(e4m3_rn_sat(v * down), __NV_E4M3);
    const float up = s > 0 ? __uint_as_float((uint32_t)s << 23) : __uint_as_float(0x00400000u);  // 2^(s-127)
    return __half2float(__half(hr)) * up;
}

// Smallest e with amax <= 6 * 2^e (the ue8m0 scale of an E2M1 piece),
// returned as the scale byte e + 127, clamped to [1, 254].  amax = m * 2^E,
// m in [1, 2): e = E - 2 if m <= 1.5, else E - 1.
__device__ __forceinline__ int e2m1_scale_byte(float amax)
{
    const uint32_t b = __float_as_uint(amax);
    int ef = (int)((b >> 23) & 0xFF);
    if (amax == 0.0f || ef == 0xFF) return 127;
    int E;
    uint32_t mant;
    if (ef == 0) {
        const uint32_t m = b & 0x7FFFFF;
        const int p = 31 - __clz(m);
        E = p - 149;
        mant = (m << (23 - p)) & 0x7FFFFF;
    } else {
        E = ef - 127;
        mant = b & 0x7FFFFF;
    }
    int e = (mant <= 0x400000u) ? E - 2 : E - 1;
    int s = e + 127;
    return s < 1 ? 1 : (s > 254 ? 254 : s);
}

// Two elements of a 32-block held by the 16 lanes of a half-warp (lane l:
// elements 2l, 2l + 1 of the block) quantized to E2M1 under the block's
// ue8m0 scale -- the least 2^e with max|v| <= 6 * 2^e -- and taken back: a
// round-to-nearest-even conversion of an exact scaling.  Every lane of the
// warp takes part.
__device__ __forceinline__ float2 e2m1_block_quant_dequant(float v0, float v1)
{
    float amax = fmaxf(fabsf(v0), fabsf(v1));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int s = e2m1_scale_byte(amax);
    const float down = exp2i(127 - s), up = exp2i(s - 127);
    const float2 d = e2m1x2_to_f32x2(f32x2_to_e2m1x2(v0 * down, v1 * down));
    return make_float2(d.x * up, d.y * up);
}

// Arrive at named barrier `id` without waiting (the waiting side uses
// named_sync with the same id and thread count).
__device__ __forceinline__ void named_arrive(int id, int threads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier over the first `threads` threads of the CTA (id 1..15).
__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace moe
