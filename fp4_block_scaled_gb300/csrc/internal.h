// internal.h -- interfaces between the C ABI (api.cu) and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/moe_ffn.h"
#include "layout.h"

namespace moe {

// bits of the sticky device status word
enum : int { kStatusBadIndex = 1, kStatusTimeout = 2 };

// Arguments of one MoE layer on the GEMV (slot-major) path.
struct GemvArgs {
    int T, topk, E, H, I;
    int sms;                            // CTAs of the streaming kernels (SM count)
    // inputs: bf16 x (forward) or fp32 residual x (stack, rmsnorm fused)
    const uint16_t* x_bf16;
    float* x_resid;
    float eps;
    const int32_t* idx;
    const float* w;
    const uint8_t* const* experts;      // per expert: the packed blob (layout.h)
    // workspace
    uint8_t* xq;                        // [T][act_bytes(H)] activation pieces (B operand)
    uint8_t* xsf;                       // [T][act_sf_bytes(H)] their scale atoms
    uint8_t* hq;                        // [T*k][act_bytes(I)] pieces of w_k * h
    uint8_t* hsf;                       // [T*k][act_sf_bytes(I)]
    // partial sums of split reduction groups, one 128-row vector per CTA and
    // projection: entries are (fp32 bits | tag << 32), the tag naming the launch
    uint64_t* part_gu;                  // [sms][128]
    uint64_t* part_dn;                  // [sms][128]
    // E4M3 activation mode (x and h quantized to E4M3, one ue8m0 scale per 128)
    int act_e4m3;
    // E2M1 activation mode (x and h quantized to E2M1, one ue8m0 scale per 32)
    int act_e2m1;
    float* hraw;                        // [T*k][I] h before quantization
    int* hpair;                         // [T*k][ceil(I/128)] tiles of each 128-block of h done
    int* sync;                          // [3]: gate/up groups finished, CTAs finished (both
                                        // zero between launches: the last CTA resets them),
                                        // launches so far (the partials' tag)
    int* status;
    unsigned long long wait_ns;         // limit of every bounded wait in the kernels (0: 2 s)
    int debug_withhold;                 // test hook: CTA 0 never reports its finished gate/up groups
    int skip_prep;                      // measurement mode: launch the layer kernel alone (the
                                        // activation pieces of the previous call are reused)
    int routing_after_wait;             // read idx, w and the expert table only after the
                                        // dependency wait (their writer may release early)
    // residual stream: per token, the sum of squares of each 32 rows of x that
    // the layer's down projection wrote ([T][H / 32]); ssq_in: the previous
    // layer left them for this layer's x (its RMSNorm reads them, not x)
    float* ssq;
    int ssq_in;
    // output (forward): y [T][H] fp32 or bf16
    void* y;
    int out_f32;
};

// Workspace of the GEMV path for up to T tokens: bytes for xq, xsf, hq, hsf;
// entry counts for part_* (uint64); the sync words are kGemvSyncInts ints.
struct GemvWorkspaceSizes {
    size_t xq, xsf, hq, hsf, part_gu, part_dn;
    size_t hraw, hpair;                 // bytes, E4M3 activation mode only
    size_t ssq;                         // bytes
};
constexpr int kGemvSyncInts = 3;
GemvWorkspaceSizes gemv_workspace_sizes(int T, int topk, int H, int I, int sms, bool e4m3);
cudaError_t gemv_init_device();   // per device, before the first launch

// Every device and page-locked allocation of the library goes through these,
// so that a test can make them fail (moe_ffn_test_fail_allocs).
cudaError_t lib_malloc(void** p, size_t bytes);
cudaError_t lib_host_alloc(void** p, size_t bytes, unsigned flags);
size_t gemv_stream_smem();

// Optional per-phase event recorder (moe_ffn_profile_*); nullptr = off.
struct Profiler {
    struct Rec { int phase; cudaEvent_t a, b; };
    std::vector<Rec> recs;
    std::vector<cudaEvent_t> pool;
    cudaEvent_t get()
    {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
    void begin(int phase, cudaStream_t s)
    {
        Rec r{phase, get(), get()};
        cudaEventRecord(r.a, s);
        recs.push_back(r);
    }
    void end(cudaStream_t s) { cudaEventRecord(recs.back().b, s); }
    ~Profiler()
    {
        for (auto& r : recs) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
        for (auto e : pool) cudaEventDestroy(e);
    }
};

enum { kPhasePrep = 0, kPhaseGateUp = 1, kPhaseDown = 2, kPhaseRoute = 3, kPhaseActQuant = 4,
       kPhaseRouter = 5, kNumPhases = 8 };

cudaError_t launch_gemv_layer(const GemvArgs& a, cudaStream_t s, bool pdl, Profiler* prof);

// Slots per group of the expert-major path, at most: a group is up to this
// many consecutive sorted slots of one expert, multiplied as the N = pieces x
// slots columns of one block-scaled MMA (N <= 64: 8 slots of 8 pieces in the
// E4M3 mode, 4 slots of 16 pieces in the bf16 mode, 16 slots of one piece in
// the E2M1 mode).
constexpr int kGroupTokens = 16;
constexpr int kGroupN = 64;
// pieces per slot of the expert-major path's activations, by mode (E2M1: the
// quantized vector itself), and slots per group (at most kGroupTokens)
__host__ __device__ inline int group_pieces(bool e4m3, bool e2m1 = false) { return e2m1 ? 1 : (e4m3 ? 8 : 16); }
__host__ __device__ inline int group_slots(bool e4m3, bool e2m1 = false)
{
    const int s = kGroupN / group_pieces(e4m3, e2m1);
    return s < kGroupTokens ? s : kGroupTokens;
}

// One group of the expert-major path.
struct __align__(16) GroupInfo {
    int e;          // expert
    int p0;         // first sorted position (perm index) of its slots
    int nt;         // slots, 1..group size
    int gb, ng;     // first group of the expert, groups of the expert
    int cnt;        // slots of the expert
    int pad[2];
};

// Token -> expert grouping (route.cu).
struct RouteArgs {
    const int32_t* idx;     // [n] expert ids of the slots
    int n, E;
    int32_t *counts, *offsets, *perm, *inv;
    int* status;
    // optional (nullptr: not made): group table of the expert-major path
    int32_t* gbase;         // [E+1] first group of each expert; gbase[E] = groups
    GroupInfo* groups;      // [max groups]
    int group_size;         // slots per group, at most
    int split;              // set by the launcher: parallel placement (32 x E counters fit)
};
// Upper bound on the groups of n slots over E experts (groups of >= gs slots).
inline int max_groups(int n, int E, int gs)
{
    const int used = n < E ? n : E;
    const int g = (n + gs - 1) / gs + used;
    return g < n ? g : n;
}

// Arguments of one MoE layer on the expert-major (grouped) path (group.cu).
struct GroupArgs {
    int T, topk, E, H, I;
    int sms;
    const uint16_t* x_bf16;
    float* x_resid;
    float eps;
    const int32_t* idx;
    const float* w;
    const uint8_t* const* experts;      // per expert: the packed blob (layout.h)
    // routing workspace (filled by the route kernel of the layer)
    int32_t *counts, *offsets, *perm, *inv, *gbase;
    GroupInfo* groups;
    // B operands in group order: the pieces of slot at sorted position P start
    // at P * (bytes of one slot's pieces over K) (units of a group hold its nt
    // slots side by side); scale atoms per (group, unit)
    uint8_t* xg;            // [n][act_bytes(H)]
    uint8_t* xgsf;          // [max groups][H/128][512]
    uint8_t* hg;            // [n][act_bytes(I)]
    uint8_t* hgsf;          // [max groups][ceil(I/128)][512]
    float* obuf;            // [n][H] down-projection output per sorted slot
    uint64_t* part_gu;      // [sms][kGroupTokens][128] tagged partial sums
    uint64_t* part_dn;
    int act_e4m3;
    int act_e2m1;           // one E2M1 piece per slot; w scales the down output
    float* hraw;            // [n][I]
    int* hpair;             // [n][ceil(I/128)]
    int* sync;              // [3], as on the slot-major path (its own words)
    int* status;
    void* y;
    int out_f32;
    // kind::mxf8f6f4 path (gemm8.cu): E4M3 rows of x and h per group, and
    // their scale atoms (two per group and 128-K unit)
    uint8_t* xb8;
    uint8_t* xb8sf;
    uint8_t* hb8;
    uint8_t* hb8sf;
    int o_unweighted;       // obuf holds unweighted down outputs: the combine applies w
    int f8_gs;              // slots per group of the kind::mxf8f6f4 launch (set by its launcher)
};

struct GroupWorkspaceSizes {
    size_t counts, offsets, perm, inv, gbase, groups;    // bytes
    size_t xg, xgsf, hg, hgsf, obuf, part_gu, part_dn, hraw, hpair;
};
GroupWorkspaceSizes group_workspace_sizes(int T, int topk, int E, int H, int I, int sms, bool e4m3);
cudaError_t group_init_device();
cudaError_t launch_group_layer(const GroupArgs& a, cudaStream_t s, bool pdl, Profiler* prof);
// y[t] = sum over the token's slots of w * obuf (or x += that), group.cu
cudaError_t launch_group_combine(const GroupArgs& a, cudaStream_t s, bool pdl);

// The expert-major path with E4M3 activations multiplied directly
// (tcgen05.mma kind::mxf8f6f4, gemm8.cu): groups of up to kF8GroupSlots slots
// of one expert, one MMA column per slot.
constexpr int kF8GroupSlots = 224;         // groups of the form for tensor-bound shapes
constexpr int kF8GroupSlotsNarrow = 64;    // ... and for HBM-bound decode batches
struct F8WorkspaceSizes {
    size_t xb8, xb8sf, hb8, hb8sf;      // bytes
};
F8WorkspaceSizes f8_workspace_sizes(int T, int topk, int E, int H, int I);
cudaError_t f8_init_device();
cudaError_t launch_f8_layer(const GroupArgs& a, cudaStream_t s, bool pdl, Profiler* prof);
// library default of moe_ffn_config.gemm_min_tokens
constexpr int kDefaultGemmMinTokens = MOE_DEFAULT_GEMM_MIN_TOKENS;
int route_max_experts();
cudaError_t route_init_device();
cudaError_t launch_route(const RouteArgs& a, cudaStream_t s, bool pdl = false);

// Router ahead of the path (router.cu).
struct RouterArgs {
    const uint16_t* x;      // bf16 [T][H]
    const uint16_t* w;      // bf16 [E][H] router weights
    float* logits;          // fp32 [T][E]
    int32_t* idx;           // [T][topk]
    float* wout;            // [T][topk]
    int T, H, E, topk;
    int tpc;                // tokens per CTA of the logits kernel (set by the launcher)
    // tensor-core batch path: split-K partial logits [nsplit][T][E], summed in
    // split order by the selection (nsplit = 0: the logits are in `logits`)
    float* part;
    int nsplit;
    int* status;
    // non-null: k_router_logits also selects (the last CTA of each token tile,
    // counted here; [ceil(T / tpc)] ints, zero between launches)
    int* tickets;
    // the handle's layer kernels read the routing only after their dependency
    // wait, so the router kernels may let the next launch start at once
    int release_early;
};
int router_max_experts();
int router_tokens_per_cta(int H);     // 0: H too large for the logits kernel
// Splits of the tensor-core batch path for T tokens (0: the path does not
// apply: T <= 8, or H not a multiple of 128); its partials need
// router_max_splits(H) * T * E floats.
int router_mma_splits(int T, int H, int E);
int router_max_splits(int H);
cudaError_t router_init_device();
cudaError_t launch_router_logits(const RouterArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_router_mma(const RouterArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_router_select(const RouterArgs& a, cudaStream_t s, bool pdl);
// one token on one thread-block cluster (logits and selection in one launch,
// no global round trip between them), where the device and the shape allow it
bool router_cluster_fits(int T, int E, int H);
cudaError_t launch_router_cluster(const RouterArgs& a, cudaStream_t s, bool pdl);

// E4M3 / ue8m0-per-128 activation quantizer (actquant.cu).
struct ActQuantArgs {
    const uint16_t* x;      // bf16 [src rows][n]
    const int32_t* src_row; // optional gather: output row r reads x row src_row[r] (-1: zeros)
    int rows, n;            // output rows; n % 32 == 0
    uint8_t* codes;         // [rows][n]
    uint8_t* scales;        // [rows][ceil(n/128)]
};
cudaError_t launch_act_quant(const ActQuantArgs& a, cudaStream_t s, bool pdl);

// Host-side config validation shared by the entry points (api.cu).
int check_config(const moe_ffn_config* cfg);

cudaError_t launch_pack_expert(const uint8_t* canon_codes, const uint8_t* canon_scales, uint8_t* packed,
                               int H, int I, cudaStream_t s);

}  // namespace moe
