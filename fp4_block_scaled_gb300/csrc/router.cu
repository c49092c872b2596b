// router.cu -- the router ahead of the routed FFN: logits = W x for every
// token, then each token's top-k experts and the softmax of their logits.
//
//   k_router_logits  grid (ceil(E / nw), ceil(T / tpc)), nw = 4 or 8 warps:
//                    warp w owns expert row e = nw blockIdx.x + w; the CTA's
//                    tpc <= 8 tokens sit in shared memory (bf16, fp32 for 8); each
//                    lane loads its 16 chunks of 16 bytes of the row (8
//                    weights each; a warp covers 4096 of H per pass) at once,
//                    so a pass keeps the whole row in flight, and accumulates
//                    the tpc dot products in fp32 (bf16 products are exact),
//                    then a butterfly warp sum, so the result is
//                    reproducible.  Given a ticket counter per token tile,
//                    the last CTA of the tile to finish also runs the
//                    selection below for its tokens: one launch per call.
// A kernel that writes topk_idx / topk_w never lets its dependents launch early
// (no griddepcontrol.launch_dependents): the layer's kernels resolve expert
// pointers from topk_idx before their own griddepcontrol.wait.
//   k_router_select  one warp per token: the logits as order keys in
//                    registers, k rounds of a warp arg-max under the order
//                    "larger logit first, NaN after every number, ties to the
//                    lower expert id" over the lanes' running bests, then the
//                    softmax of the selected logits in fp32.
// The token tile of k_router_logits is a template parameter (1..8) so that a
// small batch runs small code (a fully unrolled 16-token body stalled on
// instruction fetch).
#include <math_constants.h>

#include "common.cuh"
#include "internal.h"
#include "rsel.cuh"

namespace moe {
using namespace rsel;
namespace {

constexpr int kRPerLane = 32;       // most logits per lane in k_router_select (E <= 1024)
// grid ceil(T / 8), 256 threads: one warp per token.
template <int R>
__global__ void __launch_bounds__(256) k_router_select(RouterArgs a)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    pdl_wait();
    // no early launch_dependents (unless the handle's layer reads the routing
    // after its own wait): the next kernel may read topk_idx / topk_w before its
    // griddepcontrol.wait, so it starts only once they are written
    if (a.release_early) pdl_trigger();
    if (t >= a.T) return;
    select_token<R>(a, t, lane);
}

template <int TPC, int NW>
__global__ void __launch_bounds__(NW * 32) k_router_logits(RouterArgs a)
{
    extern __shared__ __align__(16) uint4 s_x[];      // [TPC][H / 8]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H8 = a.H / 8;
    const int t0 = blockIdx.y * TPC;
    const int nt = min(TPC, a.T - t0);
    const int e = blockIdx.x * NW + warp;
    const uint4* wrow = reinterpret_cast<const uint4*>(a.w + (size_t)min(e, a.E - 1) * a.H);
    float acc[TPC];
#pragma unroll
    for (int t = 0; t < TPC; t++) acc[t] = 0.0f;
    auto dot = [&](const uint4 wq, int c) {
        float wf[8];
        bf16x8_to_f32(wq, wf);
#pragma unroll
        for (int t = 0; t < TPC; t++) {
            if (t < nt) {
                float xf[8];
                bf16x8_to_f32(s_x[t * H8 + c], xf);
#pragma unroll
                for (int q = 0; q < 8; q++) acc[t] = fmaf(wf[q], xf[q], acc[t]);
            }
        }
    };
    if constexpr (TPC <= 4) {
        // small batches are latency-bound: a whole pass of the row (a warp covers
        // 4096 of H) in flight at once, issued before the wait for the previous
        // kernel (the router weights are not written by earlier kernels)
        uint4 wv[kRChunks];
#pragma unroll
        for (int i = 0; i < kRChunks; i++) {
            const int c = lane + 32 * i;
            wv[i] = c < H8 ? ldg_stream_v4(wrow + c) : make_uint4(0, 0, 0, 0);
        }
        pdl_wait();
        if (!a.tickets || a.release_early) pdl_trigger();     // selecting here: dependents start at completion
        stage_x(reinterpret_cast<const uint4*>(a.x + (size_t)t0 * a.H), nt * H8,
                [&](int i, const uint4 v) { s_x[i] = v; });
        __syncthreads();
        const bool live = e < a.E;     // warps past E stay for the selection below
        for (int c0 = 0; live && c0 < H8; c0 += 32 * kRChunks) {
            if (c0 > 0) {
#pragma unroll
                for (int i = 0; i < kRChunks; i++) {
                    const int c = c0 + lane + 32 * i;
                    wv[i] = c < H8 ? ldg_stream_v4(wrow + c) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int i = 0; i < kRChunks; i++) {
                const int c = c0 + lane + 32 * i;
                if (c < H8) dot(wv[i], c);
            }
        }
    } else {
        // larger batches reuse each weight chunk for TPC tokens: x is staged as
        // fp32 once per CTA ([TPC][H]) and the weights stream
        float4* s_xf = reinterpret_cast<float4*>(s_x);
        pdl_wait();
        if (!a.tickets || a.release_early) pdl_trigger();     // selecting here: dependents start at completion
        stage_x(reinterpret_cast<const uint4*>(a.x + (size_t)t0 * a.H), nt * H8, [&](int i, const uint4 v) {
            float f[8];
            bf16x8_to_f32(v, f);
            s_xf[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
            s_xf[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
        });
        __syncthreads();
        const bool live = e < a.E;     // warps past E stay for the selection below
        constexpr int kDepth = 8;                 // weight chunks in flight per lane
        for (int c0 = lane; live && c0 < H8; c0 += 32 * kDepth) {
            uint4 wq[kDepth];
#pragma unroll
            for (int q = 0; q < kDepth; q++) {
                const int c = c0 + 32 * q;
                wq[q] = c < H8 ? ldg_stream_v4(wrow + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < kDepth; q++) {
            const int c = c0 + 32 * q;
            if (c >= H8) break;
            float wf[8];
            bf16x8_to_f32(wq[q], wf);
#pragma unroll
            for (int t = 0; t < TPC; t++) {
                if (t < nt) {
                    const float4 x0 = s_xf[(t * H8 + c) * 2], x1 = s_xf[(t * H8 + c) * 2 + 1];
                    acc[t] = fmaf(wf[0], x0.x, acc[t]);
                    acc[t] = fmaf(wf[1], x0.y, acc[t]);
                    acc[t] = fmaf(wf[2], x0.z, acc[t]);
                    acc[t] = fmaf(wf[3], x0.w, acc[t]);
                    acc[t] = fmaf(wf[4], x1.x, acc[t]);
                    acc[t] = fmaf(wf[5], x1.y, acc[t]);
                    acc[t] = fmaf(wf[6], x1.z, acc[t]);
                    acc[t] = fmaf(wf[7], x1.w, acc[t]);
                }
            }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < TPC; t++) {
        if (t < nt) {
            const float v = warp_sum(acc[t]);
            if (lane == 0 && e < a.E) a.logits[(size_t)(t0 + t) * a.E + e] = v;
        }
    }
    if (!a.tickets) return;
    // the last CTA of this token tile to finish selects its tokens' top-k: the
    // logits are made visible before the ticket is taken, and the counter is
    // cleared for the next launch (whose CTAs take tickets only after this
    // grid has completed, behind their griddepcontrol.wait)
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.tickets + blockIdx.y, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (warp < nt) select_token_any(a, t0 + warp, lane);
    if (threadIdx.x == 0) a.tickets[blockIdx.y] = 0;
}

// ------------------------------------------------ one token, one cluster

// grid = one cluster of C CTAs, NW warps each, for one token: warp w of CTA
// r owns expert row e = NW r + w and computes its logit exactly as
// k_router_logits does for a one-token tile (the lane's whole share of the row
// loaded before the wait for the previous kernel, the same order of products
// and the same butterfly sum); each logit goes to global memory and into the
// first CTA's shared memory, and after one cluster barrier that CTA's first
// warp selects -- no ticket, fence or global round trip between the logits and
// the selection.
template <int NW>
__global__ void __launch_bounds__(NW * 32) k_router_cluster(RouterArgs a)
{
    extern __shared__ __align__(16) uint4 s_x[];      // [H / 8] x (bf16), then [E] logits (the first CTA's)
    float* s_logit = reinterpret_cast<float*>(s_x + a.H / 8);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int e = (int)rank * NW + warp;
    uint4 wv[kRChunks];
    row_load(a, e, lane, wv);
    if (a.release_early) pdl_trigger();
    pdl_wait();
    stage_x(reinterpret_cast<const uint4*>(a.x), a.H / 8, [&](int i, const uint4 v) { s_x[i] = v; });
    __syncthreads();
    if (e < a.E) {
        const float v = row_dot(a, e, lane, wv, s_x);
        if (lane == 0) {
            a.logits[e] = v;
            st_cluster_f32(&s_logit[e], 0, v);
        }
    }
    cluster_barrier();
    if (rank == 0 && warp == 0) {
        if (a.E <= 128) select_token<4>(a, 0, lane, s_logit);
        else select_token<8>(a, 0, lane, s_logit);
    }
}

// ------------------------------------------------ tensor-core batch path

constexpr uint64_t kRWaitLimitNs = 2000000000ull;

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulate,
// both operands K-major.
__host__ __device__ constexpr uint32_t f16_bf16_idesc(uint32_t M, uint32_t N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 bytes global -> shared, asynchronously; valid = false fills zeros (the
// source address is then not read).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

// grid (ceil(E / 128), ceil(T / N), H / kr), 256 threads: the logits of 128
// experts x N tokens over one K slice of kr, as kr / 16 tcgen05 MMAs (M = 128,
// N, K = 16, bf16 in, fp32 in tensor memory) by one thread.  Both operands
// are staged K-major without swizzle (per MMA: 8-row groups of 256 bytes, two
// 8 x 16-byte core matrices along K), rows past E or T as zeros; the
// accumulator goes to part[split][t][e].
template <int N>
__global__ void __launch_bounds__(256) k_router_mma(RouterArgs a, int kr)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    constexpr uint32_t kCols = N < 32 ? 32 : N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * 128, t0 = blockIdx.y * N, sp = blockIdx.z, k0 = sp * kr;
    const int nm = kr / 16, cpr = kr / 8;          // MMAs; 16-byte chunks per row
    uint8_t* sA = smem;
    uint8_t* sB = smem + (size_t)nm * 4096;
    if (warp == 0) tmem_alloc(&tbase, kCols);
    if (threadIdx.x == 32) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    // A warp copies 8 rows x 4 chunks at a time (lane: row lane % 8, chunk
    // lane / 8): each quarter-warp writes 8 rows of one core matrix, 8
    // different bank groups, and each row's 4 chunks are 64 contiguous bytes.
    const int q4 = cpr / 4;                        // power of two
    // the router weights are no previous kernel's output: staged before the wait
    for (int it = warp; it < 16 * q4; it += 8) {
        const int r = (it / q4) * 8 + (lane & 7), q = (it % q4) * 4 + (lane >> 3), e = e0 + r;
        const bool ok = e < a.E;
        cp_async16(sA + (q >> 1) * 4096 + (r >> 3) * 256 + (q & 1) * 128 + (r & 7) * 16,
                   a.w + (size_t)(ok ? e : 0) * a.H + k0 + 8 * q, ok);
    }
    pdl_wait();
    pdl_trigger();
    for (int it = warp; it < (N / 8) * q4; it += 8) {
        const int r = (it / q4) * 8 + (lane & 7), q = (it % q4) * 4 + (lane >> 3), t = t0 + r;
        const bool ok = t < a.T;
        cp_async16(sB + (q >> 1) * (N * 32) + (r >> 3) * 256 + (q & 1) * 128 + (r & 7) * 16,
                   a.x + (size_t)(ok ? t : 0) * a.H + k0 + 8 * q, ok);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    // the copies wrote through the generic proxy; the tensor core reads through the async one
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tbase;
    if (threadIdx.x == 0) {
        const uint32_t idesc = f16_bf16_idesc(128, N);
        for (int m = 0; m < nm; m++)
            tc_mma_f16(tmem, umma_desc(smem_u32(sA + m * 4096), 128, 256),
                       umma_desc(smem_u32(sB + (size_t)m * N * 32), 128, 256), idesc, m > 0 ? 1u : 0u);
        tc_commit(&bar);
    }
    bool done = mbar_wait_bounded(&bar, 0, kRWaitLimitNs);
    if (!done) {
        if (threadIdx.x == 0 && a.status) atomicOr(a.status, kStatusTimeout);
        done = mbar_wait_bounded(&bar, 0, kRWaitLimitNs);     // the MMAs must be over before the free
    }
    tc_fence_after();
    if (warp < 4 && done) {
        const int e = e0 + warp * 32 + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tc_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int t = t0 + c0 + j;
                if (t < a.T && e < a.E) a.part[((size_t)sp * a.T + t) * a.E + e] = v[j];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kCols);
}

cudaError_t rlaunch(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, void** args)
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

constexpr size_t kRSmemMax = 200 * 1024;

// CTAs per cluster of k_router_cluster on this device (0: not available),
// set by router_init_device
int g_cluster_ctas = 0;

}  // namespace

int router_max_experts() { return 32 * kRPerLane; }

// Largest token tile the logits kernel can hold for width H: tiles of up to 4
// tokens keep x in bf16, of 8 in fp32.
int router_tokens_per_cta(int H)
{
    if ((size_t)8 * H * 4 <= kRSmemMax) return 8;
    if ((size_t)4 * H * 2 <= kRSmemMax) return 4;
    if ((size_t)2 * H * 2 <= kRSmemMax) return 2;
    return (size_t)H * 2 <= kRSmemMax ? 1 : 0;
}

namespace {

int mma_tile_n(int T)
{
    int n = 16;
    while (n < T && n < 256) n *= 2;
    return n;
}

size_t mma_smem(int N, int kr) { return (size_t)(kr / 16) * (4096 + (size_t)N * 32); }

}  // namespace

int router_max_splits(int H) { return H % 128 == 0 ? H / 128 : 0; }

int router_mma_splits(int T, int H, int E)
{
    if (T <= 8 || H % 128 != 0 || E <= 0) return 0;
    const int N = mma_tile_n(T);
    const long long tiles = (long long)((E + 127) / 128) * ((T + N - 1) / N);
    // K slices of 256 where that still gives about 96 CTAs (fewer partials to
    // add), else of 128
    const int kr = (H % 256 == 0 && tiles * (H / 256) >= 96 && mma_smem(N, 256) <= kRSmemMax) ? 256 : 128;
    return H / kr;
}

cudaError_t router_init_device()
{
    const void* fns[] = {(const void*)k_router_logits<1, 4>, (const void*)k_router_logits<2, 4>,
                         (const void*)k_router_logits<4, 4>, (const void*)k_router_logits<8, 8>};
    cudaError_t e = cudaSuccess;
    for (const void* f : fns) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmemMax);
        // the same shared-memory carveout as the layer kernels: no SM reconfiguration between them
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
    }
    const void* sel[] = {(const void*)k_router_select<4>, (const void*)k_router_select<8>,
                         (const void*)k_router_select<12>, (const void*)k_router_select<16>,
                         (const void*)k_router_select<32>};
    for (const void* f : sel)
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
    // the one-token cluster kernel: 16 CTAs where the device allows that size, else 8
    g_cluster_ctas = 0;
    const void* clu[] = {(const void*)k_router_cluster<4>, (const void*)k_router_cluster<8>,
                         (const void*)k_router_cluster<16>};
    bool allow16 = true;
    for (const void* f : clu) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        if (cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            (void)cudaGetLastError();
            allow16 = false;
        }
    }
    if (e == cudaSuccess) {
        for (int cs : {16, 8}) {
            if (cs == 16 && !allow16) continue;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(cs);
            cfg.blockDim = dim3(16 * 32);
            cfg.dynamicSmemBytes = 64 * 1024;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = cs;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, (const void*)k_router_cluster<16>, &cfg) == cudaSuccess && n > 0) {
                g_cluster_ctas = cs;
                break;
            }
            (void)cudaGetLastError();
        }
    }
    const void* mma[] = {(const void*)k_router_mma<16>, (const void*)k_router_mma<32>, (const void*)k_router_mma<64>,
                         (const void*)k_router_mma<128>, (const void*)k_router_mma<256>};
    for (const void* f : mma) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRSmemMax);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
    }
    return e;
}

// The logits of T > 8 tokens on the tensor cores, as a.nsplit K slices of
// partial sums in a.part (router_mma_splits(T, H, E) of them).
cudaError_t launch_router_mma(const RouterArgs& a0, cudaStream_t s, bool pdl)
{
    RouterArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    if (a.nsplit <= 0 || a.H % a.nsplit != 0 || !a.part) return cudaErrorInvalidValue;
    const int N = mma_tile_n(a.T), kr = a.H / a.nsplit;
    if (kr % 128 != 0 || mma_smem(N, kr) > kRSmemMax) return cudaErrorInvalidValue;
    int krv = kr;
    void* args[] = {&a, &krv};
    const dim3 grid((a.E + 127) / 128, (a.T + N - 1) / N, a.nsplit);
    const void* fn = N == 16    ? (const void*)k_router_mma<16>
                     : N == 32  ? (const void*)k_router_mma<32>
                     : N == 64  ? (const void*)k_router_mma<64>
                     : N == 128 ? (const void*)k_router_mma<128>
                                : (const void*)k_router_mma<256>;
    return rlaunch(fn, grid, dim3(256), mma_smem(N, kr), s, pdl, args);
}

cudaError_t launch_router_logits(const RouterArgs& a0, cudaStream_t s, bool pdl)
{
    RouterArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    const int cap = router_tokens_per_cta(a.H);
    int tpc = 8;
    while (tpc > 1 && (tpc > cap || tpc / 2 >= a.T)) tpc /= 2;     // the smallest tile that holds T, within cap
    a.tpc = tpc;
    void* args[] = {&a};
    const int nw = tpc <= 4 ? 4 : 8;          // small tiles: more CTAs pull the weights
    const dim3 grid((a.E + nw - 1) / nw, (a.T + tpc - 1) / tpc);
    const size_t smem = (size_t)tpc * a.H * (tpc > 4 ? 4 : 2);
    const void* fn = tpc == 1   ? (const void*)k_router_logits<1, 4>
                     : tpc == 2 ? (const void*)k_router_logits<2, 4>
                     : tpc == 4 ? (const void*)k_router_logits<4, 4>
                                : (const void*)k_router_logits<8, 8>;
    return rlaunch(fn, grid, dim3(nw * 32), smem, s, pdl, args);
}

bool router_cluster_fits(int T, int E, int H)
{
    return T == 1 && g_cluster_ctas > 0 && E >= 1 && E <= g_cluster_ctas * 16 && E <= 256 && H % 8 == 0 &&
           (size_t)H * 2 + (size_t)E * 4 <= 64 * 1024;
}

cudaError_t launch_router_cluster(const RouterArgs& a0, cudaStream_t s, bool pdl)
{
    RouterArgs a = a0;
    if (!router_cluster_fits(a.T, a.E, a.H)) return cudaErrorInvalidValue;
    const int cs = g_cluster_ctas;
    const int per = (a.E + cs - 1) / cs;                 // rows per CTA
    const int nw = per <= 4 ? 4 : per <= 8 ? 8 : 16;
    const void* fn = nw == 4 ? (const void*)k_router_cluster<4>
                     : nw == 8 ? (const void*)k_router_cluster<8> : (const void*)k_router_cluster<16>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs);
    cfg.blockDim = dim3((unsigned)nw * 32);
    cfg.dynamicSmemBytes = (size_t)a.H * 2 + (size_t)a.E * 4;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    void* args[] = {&a};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_router_select(const RouterArgs& a0, cudaStream_t s, bool pdl)
{
    RouterArgs a = a0;
    if (a.T == 0) return cudaSuccess;
    void* args[] = {&a};
    const void* fn = a.E <= 128   ? (const void*)k_router_select<4>
                     : a.E <= 256 ? (const void*)k_router_select<8>
                     : a.E <= 384 ? (const void*)k_router_select<12>
                     : a.E <= 512 ? (const void*)k_router_select<16>
                                  : (const void*)k_router_select<32>;
    return rlaunch(fn, dim3((a.T + 7) / 8), dim3(256), 0, s, pdl, args);
}

}  // namespace moe
