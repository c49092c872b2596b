// api.cu -- the C ABI: validation, workspace, launches, graphs, status.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <new>
#include <vector>

#include "../../include/moe_ffn.h"
#include "internal.h"

using namespace moe;

namespace {

struct StackGraph {
    float* x;
    const int32_t* idx;
    const float* w;
    int L, T;
    std::vector<const void*> tables;  // expert table array pointer per layer
    cudaGraphExec_t exec;
    unsigned long long last_use;
};

// The layer's kernels of one small-batch moe_ffn_forward_host call as a graph,
// reading their inputs from and writing y to the handle's mapped page-locked
// staging buffer.
struct HostGraph {
    int T;
    const void* experts;
    cudaGraphExec_t exec;
    unsigned long long last_use;
};

// A handle keeps at most this many cached graphs of each kind; the least
// recently used one makes room for a new one.
constexpr size_t kMaxGraphs = 8;

template <class G>
void evict_lru_graph(std::vector<G>& graphs)
{
    if (graphs.size() < kMaxGraphs) return;
    size_t v = 0;
    for (size_t i = 1; i < graphs.size(); i++)
        if (graphs[i].last_use < graphs[v].last_use) v = i;
    cudaGraphExecDestroy(graphs[v].exec);
    graphs.erase(graphs.begin() + (long)v);
}

}  // namespace

// n 16-byte words from src to dst (the host-buffer stack call's staging copies,
// mapped host memory <-> device memory)
__global__ void k_stage_copy(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

static cudaError_t launch_stage_copy(const void* src, void* dst, size_t bytes, cudaStream_t s)
{
    const size_t n = bytes / 16;
    const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, 64);
    k_stage_copy<<<blocks, 256, 0, s>>>((const uint4*)src, (uint4*)dst, n);
    return cudaGetLastError();
}

struct moe_ffn {
    moe_ffn_config cfg;
    int device;
    int sms;
    void* ws;
    size_t ws_bytes;
    GemvArgs base;              // workspace pointers, problem sizes (slot-major path)
    GroupArgs gbase;            // the same for the expert-major path
    int gemm_min_tokens;        // T >= this takes the expert-major path
    int mma_kind;               // MOE_MMA_*: the expert-major path's MMA in the E4M3 mode
    int* status;
    uint8_t* in_stage;          // device staging for moe_ffn_forward_host: x | idx | w, packed per T
    void* y_stage;
    uint8_t* host_stage;        // page-locked, mapped: the packed inputs, then y (allocated on first use)
    uint8_t* host_stage_dev;    // its device address
    std::vector<HostGraph> hgraphs;
    cudaStream_t cap_stream;    // private stream used only for graph capture
    std::vector<StackGraph> graphs;
    // moe_stack_forward_host: page-locked mapped staging (x | idx | w) and its
    // device copy, grown on demand, and the graphs of the whole call
    uint8_t* sstage;
    uint8_t* sstage_dev;
    uint8_t* sdev;
    size_t scap;
    std::vector<StackGraph> sgraphs;
    unsigned long long use_clock;
    Profiler* prof;             // non-null while moe_ffn_profile_enable(h, 1)
    float* rlogits;             // router logits scratch [max_tokens][E]
    float* rpart;               // router split-K partials [max splits][max_tokens][E] (batches above 8)
    int* rtickets;              // router: finished CTAs per token tile [max_tokens], zero between calls
};

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Packed inputs of moe_ffn_forward_host for T tokens: x (bf16 [T][H]) at 0,
// topk_idx at idx_off(T), topk_w at w_off(T), each 16-byte aligned.
size_t host_idx_off(int T, int H) { return align_up((size_t)T * H * 2, 16); }
size_t host_w_off(int T, int H, int k) { return host_idx_off(T, H) + align_up((size_t)T * k * 4, 16); }
size_t host_in_bytes(int T, int H, int k) { return host_w_off(T, H, k) + (size_t)T * k * 4; }
// Above this many bytes of x and y, moe_ffn_forward_host copies straight from
// and to the caller's buffers instead of through its page-locked staging.
constexpr size_t kHostStageMax = 128 * 1024;

int check_cfg(const moe_ffn_config* c)
{
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->num_experts <= 0 || c->hidden <= 0 || c->inter <= 0 || c->topk <= 0 ||
        c->max_tokens < 0)
        return MOE_ERR_INVALID_ARG;
    if (c->topk > 16 || c->topk > c->num_experts) return MOE_ERR_INVALID_ARG;
    if (c->act_mode != MOE_ACT_BF16 && c->act_mode != MOE_ACT_E4M3_UE8M0_128 &&
        c->act_mode != MOE_ACT_E2M1_UE8M0_32)
        return MOE_ERR_INVALID_ARG;
    if (c->out_dtype != MOE_OUT_BF16 && c->out_dtype != MOE_OUT_F32) return MOE_ERR_INVALID_ARG;
    if (c->hidden % 128 || c->inter % 64) return MOE_ERR_UNSUPPORTED;
    if ((long long)c->hidden * c->inter > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    if (c->max_tokens > (1 << 16)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard()
    {
        int cur;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

GemvArgs layer_args(const moe_ffn* h, int T, const int32_t* idx, const float* w,
                    const moe_expert_table* tbl)
{
    GemvArgs a = h->base;
    a.T = T;
    a.idx = idx;
    a.w = w;
    a.experts = tbl->experts;
    return a;
}

int check_forward(const moe_ffn* h, const void* x, const int32_t* idx, const float* w,
                  const moe_expert_table* tbl, const void* y, int T)
{
    if (!h) return MOE_ERR_INVALID_ARG;
    if (T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !idx || !w || !y || !tbl || !tbl->experts) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(idx, 4) || !aligned(w, 4) ||
        !aligned(tbl->experts, 8))
        return MOE_ERR_INVALID_ARG;
    if (x == y) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

GroupArgs group_args(const moe_ffn* h, int T, const int32_t* idx, const float* w,
                     const moe_expert_table* tbl)
{
    GroupArgs a = h->gbase;
    a.T = T;
    a.idx = idx;
    a.w = w;
    a.experts = tbl->experts;
    return a;
}

// One layer, on the path the config selects for T tokens: x_bf16 -> y, or
// (x_bf16 == nullptr) the residual x_resid += moe(rmsnorm(x_resid)).
cudaError_t launch_layer(const moe_ffn* h, const uint16_t* x_bf16, float* x_resid, const int32_t* idx,
                         const float* w, const moe_expert_table* tbl, void* y, int T, cudaStream_t s,
                         Profiler* prof, bool ssq_in = false)
{
    if (T >= h->gemm_min_tokens) {
        GroupArgs a = group_args(h, T, idx, w, tbl);
        a.x_bf16 = x_bf16;
        a.x_resid = x_resid;
        a.y = y;
        // E4M3: kind::mxf8f6f4 where asked for, and by default where experts hold
        // many slots on average (the tensor-bound shapes; on HBM-bound decode
        // batches the pieces path streams the weights faster)
        // (the E2M1 mode likewise: its activation rows as they are, kind::mxf4)
        if ((a.act_e4m3 || a.act_e2m1) &&
            (h->mma_kind == MOE_MMA_MXF8F6F4 ||
             (h->mma_kind == MOE_MMA_AUTO && (long long)T * a.topk >= 128LL * a.E)))
            return launch_f8_layer(a, s, true, prof);
        return launch_group_layer(a, s, true, prof);
    }
    GemvArgs a = layer_args(h, T, idx, w, tbl);
    a.x_bf16 = x_bf16;
    a.x_resid = x_resid;
    a.ssq_in = ssq_in ? 1 : 0;
    a.y = y;
    return launch_gemv_layer(a, s, true, prof);
}

int run_forward(moe_ffn* h, const void* x, const int32_t* idx, const float* w,
                const moe_expert_table* tbl, void* y, int T, cudaStream_t s)
{
    return cuda_rc(launch_layer(h, (const uint16_t*)x, nullptr, idx, w, tbl, y, T, s, h->prof));
}

}  // namespace

int moe::check_config(const moe_ffn_config* cfg) { return check_cfg(cfg); }

namespace {
std::atomic<int> g_fail_allocs{0};    // test hook: this many allocations still to fail

bool fail_this_alloc()
{
    int n = g_fail_allocs.load();
    while (n > 0)
        if (g_fail_allocs.compare_exchange_weak(n, n - 1)) return true;
    return false;
}
}  // namespace

cudaError_t moe::lib_malloc(void** p, size_t bytes)
{
    if (fail_this_alloc()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}

cudaError_t moe::lib_host_alloc(void** p, size_t bytes, unsigned flags)
{
    if (fail_this_alloc()) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaHostAlloc(p, bytes, flags);
}

extern "C" {

size_t moe_ffn_packed_expert_bytes(const moe_ffn_config* cfg)
{
    if (check_cfg(cfg) != MOE_OK) return 0;
    return make_expert_layout(cfg->hidden, cfg->inter).bytes;
}

int moe_ffn_create(moe_ffn_t* out, const moe_ffn_config* cfg, int device)
{
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    int rc = check_cfg(cfg);
    if (rc) return rc;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
        return ndev ? MOE_ERR_INVALID_ARG : MOE_ERR_CUDA;
    DeviceGuard guard(device);

    moe_ffn* h = new (std::nothrow) moe_ffn();
    if (!h) return MOE_ERR_OOM;
    h->cfg = *cfg;
    h->device = device;
    if (cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        gemv_init_device() != cudaSuccess || route_init_device() != cudaSuccess ||
        group_init_device() != cudaSuccess || f8_init_device() != cudaSuccess ||
        router_init_device() != cudaSuccess) {
        delete h;
        return MOE_ERR_CUDA;
    }
    const int T = cfg->max_tokens > 0 ? cfg->max_tokens : 1;
    const int H = cfg->hidden, I = cfg->inter, k = cfg->topk;
    const bool e4m3 = cfg->act_mode == MOE_ACT_E4M3_UE8M0_128;
    GemvWorkspaceSizes g = gemv_workspace_sizes(T, k, H, I, h->sms, e4m3);
    h->gemm_min_tokens = cfg->gemm_min_tokens > 0 ? cfg->gemm_min_tokens : kDefaultGemmMinTokens;
    const bool grouped = T >= h->gemm_min_tokens;      // the expert-major path can be taken
    GroupWorkspaceSizes gw{};
    if (grouped) gw = group_workspace_sizes(T, k, cfg->num_experts, H, I, h->sms, e4m3);
    const bool e2m1 = cfg->act_mode == MOE_ACT_E2M1_UE8M0_32;
    F8WorkspaceSizes fw{};
    if (grouped && (e4m3 || e2m1)) fw = f8_workspace_sizes(T, k, cfg->num_experts, H, I);
    const size_t f4_hraw = grouped && e2m1 ? (size_t)T * k * I * sizeof(float) : 0;   // h of the direct form
    h->mma_kind = MOE_MMA_AUTO;

    // one allocation, carved into aligned pieces
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, kAlign);
        return o;
    };
    size_t o_status = take(sizeof(int)), o_sync = take(kGemvSyncInts * sizeof(int));
    size_t o_xq = take(g.xq), o_xsf = take(g.xsf), o_hq = take(g.hq), o_hsf = take(g.hsf);
    size_t o_pgu = take(g.part_gu * 8), o_pdn = take(g.part_dn * 8);
    size_t o_hraw = take(g.hraw), o_hpair = take(g.hpair), o_ssq = take(g.ssq);
    size_t o_gsync = take(kGemvSyncInts * sizeof(int));
    size_t o_gcnt = take(gw.counts), o_goff = take(gw.offsets), o_gperm = take(gw.perm);
    size_t o_ginv = take(gw.inv), o_gbase = take(gw.gbase), o_ggrp = take(gw.groups);
    size_t o_gxg = take(gw.xg), o_gxgsf = take(gw.xgsf), o_ghg = take(gw.hg), o_ghgsf = take(gw.hgsf);
    size_t o_gobuf = take(gw.obuf), o_gpgu = take(gw.part_gu), o_gpdn = take(gw.part_dn);
    size_t o_ghraw = take(gw.hraw), o_ghpair = take(gw.hpair);
    size_t o_fxb = take(fw.xb8), o_fxbsf = take(fw.xb8sf), o_fhb = take(fw.hb8), o_fhbsf = take(fw.hb8sf);
    size_t o_f4hraw = take(f4_hraw);
    size_t o_rlog = take((size_t)T * cfg->num_experts * 4), o_rtk = take((size_t)T * sizeof(int));
    const size_t rpart_bytes = T > 8 ? (size_t)router_max_splits(H) * T * cfg->num_experts * 4 : 0;
    size_t o_rpart = take(rpart_bytes);
    size_t o_inst = take(host_in_bytes(T, H, k)), o_yst = take((size_t)T * H * 4);
    h->ws_bytes = off;
    if (lib_malloc(&h->ws, h->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return MOE_ERR_OOM;
    }
    if (cudaMemset(h->ws, 0, h->ws_bytes) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
        cudaFree(h->ws);
        delete h;
        return MOE_ERR_CUDA;
    }
    char* b = (char*)h->ws;
    h->status = (int*)(b + o_status);
    GemvArgs& a = h->base;
    memset(&a, 0, sizeof(a));
    a.topk = k;
    a.E = cfg->num_experts;
    a.H = H;
    a.I = I;
    a.sms = h->sms;
    a.eps = 1e-6f;
    a.xq = (uint8_t*)(b + o_xq);
    a.xsf = (uint8_t*)(b + o_xsf);
    a.hq = (uint8_t*)(b + o_hq);
    a.hsf = (uint8_t*)(b + o_hsf);
    a.part_gu = (uint64_t*)(b + o_pgu);
    a.part_dn = (uint64_t*)(b + o_pdn);
    a.sync = (int*)(b + o_sync);
    a.status = h->status;
    a.out_f32 = cfg->out_dtype == MOE_OUT_F32;
    a.act_e4m3 = e4m3;
    a.act_e2m1 = cfg->act_mode == MOE_ACT_E2M1_UE8M0_32;
    a.hraw = e4m3 ? (float*)(b + o_hraw) : nullptr;
    a.hpair = e4m3 ? (int*)(b + o_hpair) : nullptr;
    a.ssq = (float*)(b + o_ssq);
    GroupArgs& ga = h->gbase;
    memset(&ga, 0, sizeof(ga));
    ga.topk = k;
    ga.E = cfg->num_experts;
    ga.H = H;
    ga.I = I;
    ga.sms = h->sms;
    ga.eps = 1e-6f;
    ga.status = h->status;
    ga.out_f32 = a.out_f32;
    ga.act_e4m3 = e4m3;
    ga.act_e2m1 = a.act_e2m1;
    if (grouped) {
        ga.sync = (int*)(b + o_gsync);
        ga.counts = (int32_t*)(b + o_gcnt);
        ga.offsets = (int32_t*)(b + o_goff);
        ga.perm = (int32_t*)(b + o_gperm);
        ga.inv = (int32_t*)(b + o_ginv);
        ga.gbase = (int32_t*)(b + o_gbase);
        ga.groups = (GroupInfo*)(b + o_ggrp);
        ga.xg = (uint8_t*)(b + o_gxg);
        ga.xgsf = (uint8_t*)(b + o_gxgsf);
        ga.hg = (uint8_t*)(b + o_ghg);
        ga.hgsf = (uint8_t*)(b + o_ghgsf);
        ga.obuf = (float*)(b + o_gobuf);
        ga.part_gu = (uint64_t*)(b + o_gpgu);
        ga.part_dn = (uint64_t*)(b + o_gpdn);
        ga.hraw = e4m3 ? (float*)(b + o_ghraw) : nullptr;
        ga.hpair = e4m3 ? (int*)(b + o_ghpair) : nullptr;
        if (e4m3 || e2m1) {
            ga.xb8 = (uint8_t*)(b + o_fxb);
            ga.xb8sf = (uint8_t*)(b + o_fxbsf);
            ga.hb8 = (uint8_t*)(b + o_fhb);
            ga.hb8sf = (uint8_t*)(b + o_fhbsf);
        }
        if (e2m1) ga.hraw = (float*)(b + o_f4hraw);
    }
    h->rlogits = (float*)(b + o_rlog);
    h->rtickets = (int*)(b + o_rtk);
    h->rpart = rpart_bytes ? (float*)(b + o_rpart) : nullptr;
    h->in_stage = (uint8_t*)(b + o_inst);
    h->y_stage = (void*)(b + o_yst);
    *out = h;
    return MOE_OK;
}

int moe_ffn_pack_expert(moe_ffn_t h, const void* canon_codes, const void* canon_scales, void* packed,
                        void* stream)
{
    if (!h || !canon_codes || !canon_scales || !packed) return MOE_ERR_INVALID_ARG;
    if (!aligned(canon_codes, 16) || !aligned(packed, 16)) return MOE_ERR_INVALID_ARG;
    const ExpertLayout L = make_expert_layout(h->cfg.hidden, h->cfg.inter);
    const size_t nc = (size_t)3 * h->cfg.hidden * h->cfg.inter / 2, ns = nc / 16;
    const char* pk = (const char*)packed;
    const char* cc = (const char*)canon_codes;
    const char* cs = (const char*)canon_scales;
    if ((cc < pk + L.bytes && pk < cc + nc) || (cs < pk + L.bytes && pk < cs + ns)) return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    return cuda_rc(launch_pack_expert((const uint8_t*)canon_codes, (const uint8_t*)canon_scales, (uint8_t*)packed,
                                      h->cfg.hidden, h->cfg.inter, (cudaStream_t)stream));
}

int moe_ffn_forward(moe_ffn_t h, const void* x, const int32_t* topk_idx, const float* topk_w,
                    const moe_expert_table* tbl, void* y, int T, void* stream)
{
    int rc = check_forward(h, x, topk_idx, topk_w, tbl, y, T);
    if (rc || T == 0) return rc;
    DeviceGuard guard(h->device);
    return run_forward(h, x, topk_idx, topk_w, tbl, y, T, (cudaStream_t)stream);
}

int moe_ffn_forward_host(moe_ffn_t h, const void* x_host, const int32_t* idx_host,
                         const float* w_host, const moe_expert_table* tbl, void* y_host, int T,
                         void* stream)
{
    if (!h) return MOE_ERR_INVALID_ARG;
    if (T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x_host || !idx_host || !w_host || !y_host || !tbl || !tbl->experts)
        return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    cudaStream_t s = (cudaStream_t)stream;
    const int H = h->cfg.hidden, k = h->cfg.topk, Tmax = h->cfg.max_tokens;
    const size_t ybytes = (size_t)T * H * (h->cfg.out_dtype == MOE_OUT_F32 ? 4 : 2);
    const size_t io = host_idx_off(T, H), wo = host_w_off(T, H, k);
    const size_t ytok = (size_t)H * (h->cfg.out_dtype == MOE_OUT_F32 ? 4 : 2);
    const int Tst = (int)std::min<size_t>((size_t)Tmax, kHostStageMax / ((size_t)H * 2 + ytok));  // largest staged T
    const size_t yo = align_up(host_in_bytes(Tst, H, k), 256);
    const int32_t* idx_d = (const int32_t*)(h->in_stage + io);
    const float* w_d = (const float*)(h->in_stage + wo);
    cudaError_t e = cudaSuccess;
    if ((size_t)T * H * 2 + ybytes > kHostStageMax) {
        // large batches: three copies straight from the caller's buffers and one
        // back (host-side staging copies would cost more than the launches saved)
        e = cudaMemcpyAsync(h->in_stage, x_host, (size_t)T * H * 2, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaMemcpyAsync((void*)idx_d, idx_host, (size_t)T * k * 4, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaMemcpyAsync((void*)w_d, w_host, (size_t)T * k * 4, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        int rc = run_forward(h, h->in_stage, idx_d, w_d, tbl, h->y_stage, T, s);
        if (rc) return rc;
        e = cudaMemcpyAsync(y_host, h->y_stage, ybytes, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        return cuda_rc(e);
    }
    if (!h->host_stage) {
        void* p = nullptr;
        void* d = nullptr;
        if (lib_host_alloc(&p, yo + (size_t)Tst * ytok, cudaHostAllocMapped) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_OOM;
        }
        if (cudaHostGetDevicePointer(&d, p, 0) != cudaSuccess) {
            cudaGetLastError();
            cudaFreeHost(p);
            return MOE_ERR_CUDA;
        }
        h->host_stage = (uint8_t*)p;
        h->host_stage_dev = (uint8_t*)d;
    }
    uint8_t* hs = h->host_stage;
    uint8_t* hd = h->host_stage_dev;
    // the previous call waited for its stream, so the staging buffer is free
    memcpy(hs, x_host, (size_t)T * H * 2);
    memcpy(hs + io, idx_host, (size_t)T * k * 4);
    memcpy(hs + wo, w_host, (size_t)T * k * 4);
    // the kernels read x, topk_idx, topk_w from the mapped staging buffer and
    // write y into it: the bytes cross the host link inside the kernels' own
    // loads and stores, with no copy of their own
    const int32_t* idx_m = (const int32_t*)(hd + io);
    const float* w_m = (const float*)(hd + wo);
    if (h->prof) {  // profiling times each launch on its own: no graph
        int rc = run_forward(h, hd, idx_m, w_m, tbl, hd + yo, T, s);
        if (rc) return rc;
    } else {
        h->use_clock++;
        HostGraph* g = nullptr;
        for (auto& c : h->hgraphs)
            if (c.T == T && c.experts == tbl->experts) g = &c;
        if (!g) {
            cudaGraph_t graph = nullptr;
            e = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
            const int rc = run_forward(h, hd, idx_m, w_m, tbl, hd + yo, T, h->cap_stream);
            e = cudaStreamEndCapture(h->cap_stream, &graph);
            if (rc != MOE_OK || e != cudaSuccess) {
                if (graph) cudaGraphDestroy(graph);
                cudaGetLastError();
                return rc != MOE_OK ? rc : MOE_ERR_CUDA;
            }
            cudaGraphExec_t exec = nullptr;
            e = cudaGraphInstantiate(&exec, graph, 0);
            cudaGraphDestroy(graph);
            if (e != cudaSuccess) return MOE_ERR_CUDA;
            evict_lru_graph(h->hgraphs);
            h->hgraphs.push_back(HostGraph{T, tbl->experts, exec, 0});
            g = &h->hgraphs.back();
        }
        g->last_use = h->use_clock;
        e = cudaGraphLaunch(g->exec, s);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    memcpy(y_host, hs + yo, ybytes);
    return MOE_OK;
}

int moe_ffn_route(moe_ffn_t h, const int32_t* topk_idx, int T, int32_t* counts, int32_t* offsets,
                  int32_t* perm, int32_t* inv, void* stream)
{
    if (!h || T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !perm || !inv)) return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 4) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(perm, 4) ||
        !aligned(inv, 4))
        return MOE_ERR_INVALID_ARG;
    if (h->cfg.num_experts > route_max_experts()) return MOE_ERR_UNSUPPORTED;
    DeviceGuard guard(h->device);
    RouteArgs a{topk_idx, T * h->cfg.topk, h->cfg.num_experts, counts, offsets, perm, inv, h->status, nullptr, nullptr, 1};
    cudaStream_t s = (cudaStream_t)stream;
    if (h->prof) h->prof->begin(kPhaseRoute, s);
    cudaError_t e = launch_route(a, s);
    if (h->prof) h->prof->end(s);
    return cuda_rc(e);
}

int moe_ffn_act_quant(moe_ffn_t h, const void* x, int rows, int n, uint8_t* codes,
                      uint8_t* scales, void* stream)
{
    if (!h || rows < 0 || n <= 0 || n % 32) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 4)) return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    ActQuantArgs a{(const uint16_t*)x, nullptr, rows, n, codes, scales};
    cudaStream_t s = (cudaStream_t)stream;
    if (h->prof) h->prof->begin(kPhaseActQuant, s);
    cudaError_t e = launch_act_quant(a, s, false);
    if (h->prof) h->prof->end(s);
    return cuda_rc(e);
}

int moe_router_topk(moe_ffn_t h, const void* x, const void* router_w, int T, float* logits,
                    int32_t* topk_idx, float* topk_w, void* stream)
{
    if (!h || T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !router_w || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(router_w, 16) || !aligned(logits, 4) || !aligned(topk_idx, 4) ||
        !aligned(topk_w, 4))
        return MOE_ERR_INVALID_ARG;
    if (h->cfg.num_experts > router_max_experts() || router_tokens_per_cta(h->cfg.hidden) == 0)
        return MOE_ERR_UNSUPPORTED;
    DeviceGuard guard(h->device);
    RouterArgs a{(const uint16_t*)x, (const uint16_t*)router_w, logits ? logits : h->rlogits, topk_idx, topk_w,
                 T, h->cfg.hidden, h->cfg.num_experts, h->cfg.topk, 0};
    a.status = h->status;
    a.release_early = h->base.routing_after_wait;
    // batches above 8 tokens: the tensor cores, in split-K partials that the
    // selection adds up; smaller ones stream the weights on the CUDA cores
    a.part = h->rpart;
    a.nsplit = h->rpart ? router_mma_splits(T, h->cfg.hidden, h->cfg.num_experts) : 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (h->prof) h->prof->begin(kPhaseRouter, s);
    cudaError_t e;
    if (a.nsplit) {
        e = launch_router_mma(a, s, !h->prof);
        if (e == cudaSuccess) e = launch_router_select(a, s, !h->prof);
    } else if (router_cluster_fits(T, h->cfg.num_experts, h->cfg.hidden)) {
        // one token: one cluster computes the logits and selects
        e = launch_router_cluster(a, s, !h->prof);
    } else {  // one launch: the logits kernel's last CTA per token tile selects
        a.tickets = h->rtickets;
        e = launch_router_logits(a, s, !h->prof);
    }
    if (h->prof) h->prof->end(s);
    return cuda_rc(e);
}

int moe_router_select(moe_ffn_t h, const float* logits, int T, int32_t* topk_idx, float* topk_w, void* stream)
{
    if (!h || T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_idx || !topk_w || !aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4))
        return MOE_ERR_INVALID_ARG;
    if (h->cfg.num_experts > router_max_experts()) return MOE_ERR_UNSUPPORTED;
    DeviceGuard guard(h->device);
    RouterArgs a{nullptr, nullptr, const_cast<float*>(logits), topk_idx, topk_w, T, h->cfg.hidden,
                 h->cfg.num_experts, h->cfg.topk, 0};
    return cuda_rc(launch_router_select(a, (cudaStream_t)stream, false));
}

int moe_stack_forward(moe_ffn_t h, float* x, const moe_expert_table* tbls,
                      const int32_t* topk_idx, const float* topk_w, int L, int T, void* stream)
{
    if (!h || L < 0 || T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (L == 0 || T == 0) return MOE_OK;
    if (!x || !tbls || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4)) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < L; l++)
        if (!tbls[l].experts) return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    cudaStream_t s = (cudaStream_t)stream;

    std::vector<const void*> key((size_t)L);
    for (int l = 0; l < L; l++) key[l] = tbls[l].experts;
    h->use_clock++;
    for (auto& gph : h->graphs) {
        if (gph.x == x && gph.idx == topk_idx && gph.w == topk_w && gph.L == L && gph.T == T &&
            gph.tables == key) {
            gph.last_use = h->use_clock;
            return cuda_rc(cudaGraphLaunch(gph.exec, s));
        }
    }
    // capture the L layers on the private stream, then replay on the caller's
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    cudaError_t le = cudaSuccess;
    for (int l = 0; l < L && le == cudaSuccess; l++)
        le = launch_layer(h, nullptr, x, topk_idx + (size_t)l * T * h->cfg.topk,
                          topk_w + (size_t)l * T * h->cfg.topk, &tbls[l], nullptr, T, h->cap_stream,
                          nullptr, l > 0);     // each layer leaves the next one its RMSNorm partials
    e = cudaStreamEndCapture(h->cap_stream, &graph);
    if (le != cudaSuccess || e != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    evict_lru_graph(h->graphs);
    h->graphs.push_back(StackGraph{x, topk_idx, topk_w, L, T, key, exec, h->use_clock});
    return cuda_rc(cudaGraphLaunch(exec, s));
}

int moe_stack_forward_host(moe_ffn_t h, float* x_host, const moe_expert_table* tbls,
                           const int32_t* topk_idx_host, const float* topk_w_host, int L, int T, void* stream)
{
    if (!h || L < 0 || T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
    if (L == 0 || T == 0) return MOE_OK;
    if (!x_host || !tbls || !topk_idx_host || !topk_w_host) return MOE_ERR_INVALID_ARG;
    for (int l = 0; l < L; l++)
        if (!tbls[l].experts) return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    cudaStream_t s = (cudaStream_t)stream;
    const int H = h->cfg.hidden, k = h->cfg.topk;
    const size_t xb = (size_t)T * H * 4, rb = (size_t)L * T * k * 4;
    const size_t io = align_up(xb, 256), wo = io + align_up(rb, 256), total = wo + align_up(rb, 256);
    if (total > h->scap) {
        // grow: the previous call waited for its stream, so the old buffers are idle;
        // graphs that name them go with them
        for (auto& g : h->sgraphs) cudaGraphExecDestroy(g.exec);
        h->sgraphs.clear();
        if (h->sstage) cudaFreeHost(h->sstage);
        if (h->sdev) cudaFree(h->sdev);
        h->sstage = h->sstage_dev = h->sdev = nullptr;
        h->scap = 0;
        void* p = nullptr;
        void* d = nullptr;
        void* dv = nullptr;
        if (lib_host_alloc(&p, total, cudaHostAllocMapped) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_OOM;
        }
        if (lib_malloc(&dv, total) != cudaSuccess) {
            cudaGetLastError();
            cudaFreeHost(p);
            return MOE_ERR_OOM;
        }
        if (cudaHostGetDevicePointer(&d, p, 0) != cudaSuccess) {
            cudaGetLastError();
            cudaFreeHost(p);
            cudaFree(dv);
            return MOE_ERR_CUDA;
        }
        h->sstage = (uint8_t*)p;
        h->sstage_dev = (uint8_t*)d;
        h->sdev = (uint8_t*)dv;
        h->scap = total;
    }
    memcpy(h->sstage, x_host, xb);
    memcpy(h->sstage + io, topk_idx_host, rb);
    memcpy(h->sstage + wo, topk_w_host, rb);
    float* xd = (float*)h->sdev;
    const int32_t* id = (const int32_t*)(h->sdev + io);
    const float* wd = (const float*)(h->sdev + wo);
    std::vector<const void*> key((size_t)L);
    for (int l = 0; l < L; l++) key[l] = tbls[l].experts;
    h->use_clock++;
    StackGraph* g = nullptr;
    for (auto& c : h->sgraphs)
        if (c.L == L && c.T == T && c.tables == key) g = &c;
    cudaError_t e = cudaSuccess;
    if (!g) {
        // one graph for the whole call: the inputs from the mapped staging buffer
        // into device memory (one copy kernel), the L layers, x back
        cudaGraph_t graph = nullptr;
        e = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        cudaError_t le = launch_stage_copy(h->sstage_dev, h->sdev, total, h->cap_stream);
        for (int l = 0; l < L && le == cudaSuccess; l++)
            le = launch_layer(h, nullptr, xd, id + (size_t)l * T * k, wd + (size_t)l * T * k, &tbls[l], nullptr, T,
                              h->cap_stream, nullptr, l > 0);
        if (le == cudaSuccess) le = launch_stage_copy(h->sdev, h->sstage_dev, align_up(xb, 16), h->cap_stream);
        e = cudaStreamEndCapture(h->cap_stream, &graph);
        if (le != cudaSuccess || e != cudaSuccess) {
            if (graph) cudaGraphDestroy(graph);
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        cudaGraphExec_t exec = nullptr;
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        evict_lru_graph(h->sgraphs);
        h->sgraphs.push_back(StackGraph{xd, id, wd, L, T, key, exec, 0});
        g = &h->sgraphs.back();
    }
    g->last_use = h->use_clock;
    e = cudaGraphLaunch(g->exec, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    memcpy(x_host, h->sstage, xb);
    return MOE_OK;
}

int moe_ffn_profile_layer_only(moe_ffn_t h, int on)
{
    if (!h) return MOE_ERR_INVALID_ARG;
    h->base.skip_prep = on ? 1 : 0;
    return MOE_OK;
}

// The cached graphs hold the kernel arguments of the settings they were
// captured with: a settings change drops them (after the device is done with
// them), and the next calls capture new ones.
static int drop_graphs(moe_ffn* h)
{
    if (h->graphs.empty() && h->hgraphs.empty() && h->sgraphs.empty()) return MOE_OK;
    DeviceGuard guard(h->device);
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);
    for (auto& g : h->hgraphs) cudaGraphExecDestroy(g.exec);
    for (auto& g : h->sgraphs) cudaGraphExecDestroy(g.exec);
    h->graphs.clear();
    h->hgraphs.clear();
    h->sgraphs.clear();
    return MOE_OK;
}

int moe_ffn_set_routing_wait(moe_ffn_t h, int on)
{
    if (!h || (on != 0 && on != 1)) return MOE_ERR_INVALID_ARG;
    if (h->base.routing_after_wait == on) return MOE_OK;
    h->base.routing_after_wait = on;
    return drop_graphs(h);
}

int moe_ffn_set_mma_kind(moe_ffn_t h, int kind)
{
    if (!h || (kind != MOE_MMA_AUTO && kind != MOE_MMA_MXF4_PIECES && kind != MOE_MMA_MXF8F6F4))
        return MOE_ERR_INVALID_ARG;
    if (h->mma_kind == kind) return MOE_OK;
    h->mma_kind = kind;
    return drop_graphs(h);
}

void moe_ffn_test_fail_allocs(int n) { g_fail_allocs.store(n > 0 ? n : 0); }

int moe_ffn_test_copy_h(moe_ffn_t h, float* h_dst, int32_t* perm_dst, int n, void* stream)
{
    if (!h || !h->gbase.hraw || !h->gbase.xb8 || !h_dst || !perm_dst || n < 0 ||
        (long long)n > (long long)h->cfg.max_tokens * h->cfg.topk)
        return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t hb = (size_t)n * h->cfg.inter * sizeof(float);
    if (cudaMemcpyAsync(h_dst, h->gbase.hraw, hb, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(perm_dst, h->gbase.perm, (size_t)n * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_ffn_test_set_wait(moe_ffn_t h, unsigned long long wait_ns, int withhold)
{
    if (!h) return MOE_ERR_INVALID_ARG;
    h->base.wait_ns = wait_ns;
    h->base.debug_withhold = withhold ? 1 : 0;
    return MOE_OK;
}

int moe_ffn_status(moe_ffn_t h, void* stream)
{
    if (!h) return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    cudaStream_t s = (cudaStream_t)stream;
    int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (v && cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    if (v & kStatusTimeout) return MOE_ERR_DEVICE_TIMEOUT;
    if (v & kStatusBadIndex) return MOE_ERR_BAD_INDEX;
    return MOE_OK;
}

int moe_ffn_profile_enable(moe_ffn_t h, int on)
{
    if (!h) return MOE_ERR_INVALID_ARG;
    DeviceGuard guard(h->device);
    if (on && !h->prof) {
        h->prof = new (std::nothrow) Profiler();
        if (!h->prof) return MOE_ERR_OOM;
    } else if (!on && h->prof) {
        if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
        delete h->prof;
        h->prof = nullptr;
    }
    return MOE_OK;
}

int moe_ffn_profile_read(moe_ffn_t h, double* ms, int* launches)
{
    if (!h || !ms || !launches) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < MOE_NUM_PHASES; i++) {
        ms[i] = 0.0;
        launches[i] = 0;
    }
    if (!h->prof) return MOE_OK;
    DeviceGuard guard(h->device);
    Profiler* p = h->prof;
    int rc = MOE_OK;
    for (auto& r : p->recs) {
        float t = 0.0f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
            rc = MOE_ERR_CUDA;
        if (r.phase >= 0 && r.phase < MOE_NUM_PHASES) {
            ms[r.phase] += t;
            launches[r.phase] += 1;
        }
        p->pool.push_back(r.a);
        p->pool.push_back(r.b);
    }
    p->recs.clear();
    return rc;
}

const char* moe_ffn_strerror(int code)
{
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_OOM: return "out of device memory";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_BAD_INDEX: return "expert index out of range (slot contributed zero)";
        case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        default: return "unknown error code";
    }
}

void moe_ffn_destroy(moe_ffn_t h)
{
    if (!h) return;
    DeviceGuard guard(h->device);
    for (auto& g : h->graphs) cudaGraphExecDestroy(g.exec);
    for (auto& g : h->hgraphs) cudaGraphExecDestroy(g.exec);
    for (auto& g : h->sgraphs) cudaGraphExecDestroy(g.exec);
    if (h->host_stage) cudaFreeHost(h->host_stage);
    if (h->sstage) cudaFreeHost(h->sstage);
    if (h->sdev) cudaFree(h->sdev);
    delete h->prof;
    if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
    cudaFree(h->ws);
    delete h;
}

}  // extern "C"
