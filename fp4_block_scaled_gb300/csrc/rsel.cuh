// rsel.cuh -- device helpers of the router's kernels (router.cu): the staging
// of a token, one warp's logit of one expert row, the order keys and the
// one-warp top-k selection with its softmax, and the thread-block-cluster
// primitives.
#pragma once
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace rsel {

constexpr int kRChunks = 16;        // 16-byte weight chunks per lane per pass

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// dst[i] = f(src[i]) for i < n by the CTA's threads, eight loads in flight per
// thread before the stores (a load-store pair per iteration would wait a full
// memory round trip each).
template <class F>
__device__ __forceinline__ void stage_x(const uint4* src, int n, F store)
{
    for (int i0 = threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int i = i0 + q * blockDim.x;
            v[q] = i < n ? src[i] : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int i = i0 + q * blockDim.x;
            if (i < n) store(i, v[q]);
        }
    }
}

// Order key of a logit: larger keys rank first; -0 and +0 tie; NaN ranks after
// every number (key 1); key 0 is "taken" or "no expert".
__device__ __forceinline__ uint32_t order_key(float v)
{
    if (isnan(v)) return 1u;
    const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp selects token t's top-k.  Lane l holds the order keys of experts
// l, l + 32, ... (R of them) in registers and its best untaken one; a round
// takes the warp's best with two redux.sync (the largest key, then the lowest
// id holding it), and only the winning lane picks its next best.  Lane i keeps
// pick i for the softmax.  The logits are read through L2 (other CTAs of the
// same grid may have written them).
template <int R>
__device__ __forceinline__ void select_token(const RouterArgs& a, int t, int lane, const float* srow = nullptr)
{
    float v[R];
    uint32_t key[R];
    if (srow) {
        // the logits in this CTA's shared memory (the cluster path)
#pragma unroll
        for (int j = 0; j < R; j++) {
            const int e = lane + 32 * j;
            v[j] = e < a.E ? srow[e] : 0.0f;
        }
    } else if (a.nsplit == 0) {
        const float* row = a.logits + (size_t)t * a.E;
#pragma unroll
        for (int j = 0; j < R; j++) {
            const int e = lane + 32 * j;
            v[j] = e < a.E ? __ldcg(row + e) : 0.0f;
        }
    } else {
        // the tensor-core path's split-K partials, added in split order; the
        // sums are the logits
#pragma unroll
        for (int j = 0; j < R; j++) v[j] = 0.0f;
        // four splits' loads in flight at once, added in split order
        constexpr int kQ = R <= 16 ? 4 : 2;
        for (int sp0 = 0; sp0 < a.nsplit; sp0 += kQ) {
            float q[kQ][R];
#pragma unroll
            for (int u = 0; u < kQ; u++) {
                const float* row = a.part + ((size_t)(sp0 + u) * a.T + t) * a.E;
#pragma unroll
                for (int j = 0; j < R; j++) {
                    const int e = lane + 32 * j;
                    q[u][j] = (sp0 + u < a.nsplit && e < a.E) ? __ldcg(row + e) : 0.0f;
                }
            }
#pragma unroll
            for (int u = 0; u < kQ; u++)
#pragma unroll
                for (int j = 0; j < R; j++)
                    if (sp0 + u < a.nsplit) v[j] += q[u][j];
        }
        float* out = a.logits + (size_t)t * a.E;
#pragma unroll
        for (int j = 0; j < R; j++) {
            const int e = lane + 32 * j;
            if (e < a.E) out[e] = v[j];
        }
    }
#pragma unroll
    for (int j = 0; j < R; j++) key[j] = lane + 32 * j < a.E ? order_key(v[j]) : 0u;
    uint32_t bk = 0;                                   // this lane's best: key, slot, value
    int bj = 0;
    float bv = 0.0f;
    auto lane_best = [&]() {
        bk = 0;
        bj = 0;
#pragma unroll
        for (int j = 0; j < R; j++)                    // strict >: the lower id on equal keys
            if (key[j] > bk) {
                bk = key[j];
                bj = j;
                bv = v[j];
            }
    };
    lane_best();
    float mine = 0.0f;
    int mine_e = 0;
    for (int i = 0; i < a.topk; i++) {
        const uint32_t gk = __reduce_max_sync(0xFFFFFFFFu, bk);
        const int ge = (int)__reduce_min_sync(0xFFFFFFFFu, bk == gk ? (uint32_t)(lane + 32 * bj) : 0xFFFFFFFFu);
        const float gv = __shfl_sync(0xFFFFFFFFu, bv, ge & 31);
        if (lane == i) {
            mine = gv;
            mine_e = ge;
        }
        if ((ge & 31) == lane) {
#pragma unroll
            for (int j = 0; j < R; j++)
                if (j == (ge >> 5)) key[j] = 0u;
            lane_best();
        }
    }
    const float m = __shfl_sync(0xFFFFFFFFu, mine, 0);
    const float p = lane < a.topk ? expf(mine - m) : 0.0f;
    float sum = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane < a.topk) {
        a.idx[(size_t)t * a.topk + lane] = mine_e;
        a.wout[(size_t)t * a.topk + lane] = p / sum;
    }
}

__device__ __forceinline__ void select_token_any(const RouterArgs& a, int t, int lane)
{
    if (a.E <= 128) select_token<4>(a, t, lane);
    else if (a.E <= 256) select_token<8>(a, t, lane);
    else if (a.E <= 384) select_token<12>(a, t, lane);
    else if (a.E <= 512) select_token<16>(a, t, lane);
    else select_token<32>(a, t, lane);
}


__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// v into the float at `local`'s offset in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ void st_cluster_f32(const float* local, uint32_t rank, float v)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Every thread of every CTA of the cluster; the writes before it (shared
// memory of any CTA of the cluster included) are visible after it.
__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}


// One warp's logit of expert row e (a bf16 row of H) against the token staged
// in shared memory (s_x: H / 8 chunks of 8 bf16): the lane's first pass of
// kRChunks 16-byte weight chunks (wv) is loaded by row_load, before the wait
// for the previous kernel; row_dot loads any further passes, multiplies in
// chunk order and returns the butterfly sum of the lanes (fp32; the bf16
// products are exact), the same for every caller, so every path gives the same
// logits.
__device__ __forceinline__ void row_load(const RouterArgs& a, int e, int lane, uint4 (&wv)[kRChunks])
{
    const uint4* wrow = reinterpret_cast<const uint4*>(a.w + (size_t)min(e, a.E - 1) * a.H);
    const int H8 = a.H / 8;
#pragma unroll
    for (int i = 0; i < kRChunks; i++) {
        const int c = lane + 32 * i;
        wv[i] = c < H8 ? ldg_stream_v4(wrow + c) : make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ float row_dot(const RouterArgs& a, int e, int lane, uint4 (&wv)[kRChunks], const uint4* s_x)
{
    const uint4* wrow = reinterpret_cast<const uint4*>(a.w + (size_t)min(e, a.E - 1) * a.H);
    const int H8 = a.H / 8;
    float acc = 0.0f;
    for (int c0 = 0; c0 < H8; c0 += 32 * kRChunks) {
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
            if (c < H8) {
                float wf[8], xf[8];
                bf16x8_to_f32(wv[i], wf);
                bf16x8_to_f32(s_x[c], xf);
#pragma unroll
                for (int q = 0; q < 8; q++) acc = fmaf(wf[q], xf[q], acc);
            }
        }
    }
    return warp_sum(acc);
}

}  // namespace rsel
}  // namespace moe
