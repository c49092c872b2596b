// route.cu -- token -> expert grouping on the device (no host round trip).
//
// A stable counting sort of the T*k routing slots by expert id, in one CTA:
//   1. histogram of expert ids in shared memory (order-free integer counts);
//   2. exclusive prefix sum over the E counts (offsets);
//   3. one warp walks the slots in order, 32 at a time: lanes that carry the
//      same expert find each other with match.any, the lowest of them reserves
//      a run of positions from that expert's cursor, and each lane takes
//      cursor + (rank among the earlier equal lanes).  Slot order is kept
//      within an expert, so perm is unique and the result bit-exact.
// Out-of-range ids are left out (inv = -1, status "bad index"); perm entries
// past the number of valid slots are -1.
// When asked for, the same pass also cuts each expert's sorted slots into
// groups of up to group_size slots (the expert-major path's MMA columns): a
// second exclusive scan, over ceil(count / group_size), numbers the groups.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kRouteThreads = 1024;
constexpr size_t kRouteSplitSmem = 200 * 1024;

// Exclusive prefix sum of v over the CTA (thread order); *total = the sum.
// s_warp: one int per warp.  Every thread must call it.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    __syncthreads();                        // s_warp is free (earlier scans done)
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w += u;
        }
        if (lane < nw) s_warp[lane] = w;    // inclusive warp totals
    }
    __syncthreads();
    *total = s_warp[nw - 1];
    return incl - v + (warp ? s_warp[warp - 1] : 0);
}

__global__ void __launch_bounds__(kRouteThreads) k_route(RouteArgs a)
{
    extern __shared__ int s_cur[];          // E counters, then cursors
    __shared__ int s_warp[kRouteThreads / 32];
    __shared__ int s_bad;
    const int n = a.n, E = a.E;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    pdl_wait();
    for (int e = tid; e < E; e += blockDim.x) s_cur[e] = 0;
    if (tid == 0) s_bad = 0;
    __syncthreads();
#pragma unroll 4
    for (int j = tid; j < n; j += blockDim.x) {
        const int e = a.idx[j];
        if (e >= 0 && e < E) atomicAdd(&s_cur[e], 1);
        else s_bad = 1;
    }
    __syncthreads();

    // exclusive scans over E of the counts and of the group counts: each thread
    // owns a contiguous run of experts
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    const int gs = a.groups ? a.group_size : 1;
    int local = 0, lgrp = 0;
    for (int e = e0; e < e1; e++) {
        local += s_cur[e];
        lgrp += (s_cur[e] + gs - 1) / gs;
    }
    int total = 0, gtotal = 0;
    int run = block_exclusive_scan(local, s_warp, &total);
    int grun = block_exclusive_scan(lgrp, s_warp, &gtotal);
    for (int e = e0; e < e1; e++) {
        const int c = s_cur[e];
        const int ng = (c + gs - 1) / gs;
        a.counts[e] = c;
        a.offsets[e] = run;
        if (a.groups) {
            a.gbase[e] = grun;
            for (int q = 0; q < ng; q++) {
                GroupInfo gi = {};
                gi.e = e;
                gi.p0 = run + q * gs;
                gi.nt = min(gs, c - q * gs);
                gi.gb = grun;
                gi.ng = ng;
                gi.cnt = c;
                a.groups[grun + q] = gi;
            }
        }
        s_cur[e] = run;                     // becomes the placement cursor
        run += c;
        grun += ng;
    }
    if (tid == 0) {
        a.offsets[E] = total;
        if (a.groups) a.gbase[E] = gtotal;
        if (s_bad) atomicOr(a.status, kStatusBadIndex);
    }
    __syncthreads();

    // stable placement: pos(j) = offsets[e_j] + (slots before j with expert
    // e_j).  With room for 32 x E counters in shared memory, warp w takes the
    // w-th contiguous segment of the slots: it counts its segment per expert,
    // an exclusive scan over the warps per expert gives its start cursors,
    // then it places its segment in order (32 slots at a time, ranks within a
    // chunk by match).  Otherwise one warp walks all slots.
    const int nw = blockDim.x >> 5;
    const bool split = a.split != 0;
    int* s_seg = s_cur + E;                                      // [32][E] when split
    const int seg = split ? (n + nw - 1) / nw : n;
    const int w_lo = split ? min(n, warp * seg) : 0, w_hi = split ? min(n, w_lo + seg) : n;
    int* cur = split ? s_seg + (size_t)warp * E : s_cur;     // this warp's cursors
    if (split) {
        for (int i = tid; i < nw * E; i += blockDim.x) s_seg[i] = 0;
        __syncthreads();
        for (int j = w_lo + lane; j < w_hi; j += 32) {
            const int e = a.idx[j];
            if (e >= 0 && e < E) atomicAdd(&cur[e], 1);
        }
        __syncthreads();
        for (int e = tid; e < E; e += blockDim.x) {
            int c = s_cur[e];                                   // the expert's offset
            for (int w = 0; w < nw; w++) {
                int* pw = s_seg + (size_t)w * E + e;
                const int cnt = *pw;
                *pw = c;
                c += cnt;
            }
        }
        __syncthreads();
    }
    if (split || warp == 0) {
        constexpr int kBatch = 8;                               // ids of 8 chunks per round trip
        int ev[kBatch];
        for (int base = w_lo; base < w_hi; base += 32) {
            const int q = ((base - w_lo) >> 5) % kBatch;
            if (q == 0) {
#pragma unroll
                for (int b = 0; b < kBatch; b++) {
                    const int jj = base + 32 * b + lane;
                    ev[b] = jj < w_hi ? a.idx[jj] : -1;
                }
            }
            const int j = base + lane;
            int e = -1;
#pragma unroll
            for (int b = 0; b < kBatch; b++)
                if (b == q) e = ev[b];
            const bool valid = j < w_hi && e >= 0 && e < E;
            const int key = valid ? e : E + lane;          // invalid lanes match nobody
            const unsigned mask = __match_any_sync(0xFFFFFFFFu, key);
            const int leader = __ffs(mask) - 1;
            const int rank = __popc(mask & ((1u << lane) - 1u));
            int start = 0;
            if (valid && lane == leader) {
                start = cur[e];
                cur[e] = start + __popc(mask);
            }
            start = __shfl_sync(0xFFFFFFFFu, start, leader);
            if (valid) {
                const int pos = start + rank;
                a.perm[pos] = j;
                a.inv[j] = pos;
            } else if (j < w_hi) {
                a.inv[j] = -1;
            }
            __syncwarp();
        }
    }
    for (int p = total + tid; p < n; p += blockDim.x) a.perm[p] = -1;
    pdl_trigger();
}

}  // namespace

int route_max_experts() { return 32768; }

cudaError_t route_init_device()
{
    const size_t need = (size_t)route_max_experts() * sizeof(int);
    return cudaFuncSetAttribute((const void*)k_route, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(need > kRouteSplitSmem ? need : kRouteSplitSmem));
}

cudaError_t launch_route(const RouteArgs& a0, cudaStream_t s, bool pdl)
{
    RouteArgs a = a0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kRouteThreads);
    // E cursors, and 32 x E per-warp counters for the parallel placement when
    // they fit
    a.split = (size_t)33 * a.E * sizeof(int) <= kRouteSplitSmem ? 1 : 0;
    cfg.dynamicSmemBytes = (size_t)(a.split ? 33 : 1) * a.E * sizeof(int);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    void* args[] = {&a};
    return cudaLaunchKernelExC(&cfg, (const void*)k_route, args);
}

}  // namespace moe
