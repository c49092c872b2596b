// noalloc.cu -- moe_ffn_forward_noalloc: the batch-1 / small-batch layer
// with its scratch memory in a fixed, file-scope device array.
//
// For callers that may not allocate device memory on their call path: hosts
// that own every device allocation and give a library no allocator of its own
// (embedded inference runtimes, plugin hosts with a fixed memory budget, code
// that must never fail on an out-of-memory at call time).  moe_ffn_create
// needs cudaMalloc for its workspace; this entry point needs no handle and
// calls no cudaMalloc, cudaFree or allocating library routine.  It runs the
// same kernels as moe_ffn_forward; their scratch (activation pieces, h, split-K
// partial sums and counters) lives in g_scratch below.
//
// g_scratch is a static __device__ array: every GPU that loads this library
// holds its kNoAllocScratchBytes until the process exits, and all calls share
// it.  In host code the name g_scratch is only a host-side stand-in for the
// symbol, not a device address; its device address is obtained with
// cudaGetSymbolAddress, with the device current, and passed to the kernels.
// The first call on a device also sets the kernels' shared-memory limits, so
// it should come before any stream capture; later calls look the address up
// again and redo that set-up if it changed (a device reset makes a new
// context, with a new copy of the array).  Each call clears the counters that
// must start at zero (cudaMemsetAsync on the call's stream); the rest keeps
// the previous call's contents, and two calls whose work overlaps on the GPU
// (different streams, or different threads without ordering) race on it.  The
// launch-tagged partial sums sit at fixed offsets, in areas sized for the
// largest SM count, so they only ever hold tagged words (whose tags, counting
// launches, never repeat) or the array's initial zeros, whatever the shapes of
// earlier calls.
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

#include "internal.h"

using namespace moe;

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;   // 4 MiB in all:
constexpr size_t kSyncBytes = 256;                      // status word and counters
constexpr int kMaxSms = 256;
constexpr size_t kPartBytes = (size_t)kMaxSms * 128 * 8; // one area of tagged partial sums
constexpr size_t kOffPartGu = kSyncBytes;
constexpr size_t kOffPartDn = kOffPartGu + kPartBytes;
constexpr size_t kOffRest = kOffPartDn + kPartBytes;    // then the activation and h pieces
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

struct DeviceScratch {
    void* ptr = nullptr;   // device address of g_scratch in that device's current context
    int sms = 0;
};

DeviceScratch g_devices[kMaxDevices];
std::mutex g_setup_mutex;

// With the device current: g_scratch's address, and (first call, or a new
// context since) the kernels' shared-memory limits.
int setup_device(int device, DeviceScratch* out)
{
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceScratch& d = g_devices[device];
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) return MOE_ERR_CUDA;
    if (ptr != d.ptr) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (gemv_init_device() != cudaSuccess) return MOE_ERR_CUDA;
        d.ptr = ptr;
        d.sms = sms;
    }
    *out = d;
    return MOE_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

extern "C" int moe_ffn_forward_noalloc(const moe_ffn_config* cfg, int device, const void* x,
                                       const int32_t* topk_idx, const float* topk_w,
                                       const moe_expert_table* tbl, void* y, int T,
                                       int* status, void* stream)
{
    int rc = check_config(cfg);
    if (rc) return rc;
    if (cfg->act_mode != MOE_ACT_BF16) return MOE_ERR_UNSUPPORTED;
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !topk_idx || !topk_w || !y || !tbl || !tbl->experts || x == y)
        return MOE_ERR_INVALID_ARG;
    if (((uintptr_t)x | (uintptr_t)y) % 16 || ((uintptr_t)topk_idx | (uintptr_t)topk_w) % 4 ||
        ((uintptr_t)status) % 4)
        return MOE_ERR_INVALID_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) return MOE_ERR_CUDA;
    if (device < 0 || device >= ndev || device >= kMaxDevices) return MOE_ERR_INVALID_ARG;

    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return MOE_ERR_CUDA;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
    struct Restore {
        int prev, dev;
        ~Restore() { if (prev >= 0 && prev != dev) cudaSetDevice(prev); }
    } restore{prev, device};

    DeviceScratch d;
    rc = setup_device(device, &d);
    if (rc) return rc;
    if (d.sms > kMaxSms) return MOE_ERR_UNSUPPORTED;

    // fixed areas first (status and counters, cleared every call except the
    // launch count that tags the partial sums; the two areas of tagged partial
    // sums), then the activation and h pieces
    const int H = cfg->hidden, I = cfg->inter, k = cfg->topk;
    const GemvWorkspaceSizes g = gemv_workspace_sizes(T, k, H, I, d.sms, false);
    size_t off = kOffRest;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_xq = take(g.xq), o_xsf = take(g.xsf), o_hq = take(g.hq), o_hsf = take(g.hsf);
    if (off > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;   // problem too large for the array

    cudaStream_t s = (cudaStream_t)stream;
    char* b = (char*)d.ptr;
    int* status_w = (int*)b;
    int* sync_w = status_w + 1;
    if (cudaMemsetAsync(b, 0, 3 * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;   // status, sync[0..1]

    GemvArgs a;
    memset(&a, 0, sizeof(a));
    a.T = T;
    a.topk = k;
    a.E = cfg->num_experts;
    a.H = H;
    a.I = I;
    a.sms = d.sms;
    a.eps = 1e-6f;
    a.x_bf16 = (const uint16_t*)x;
    a.idx = topk_idx;
    a.w = topk_w;
    a.experts = tbl->experts;
    a.xq = (uint8_t*)(b + o_xq);
    a.xsf = (uint8_t*)(b + o_xsf);
    a.hq = (uint8_t*)(b + o_hq);
    a.hsf = (uint8_t*)(b + o_hsf);
    a.part_gu = (uint64_t*)(b + kOffPartGu);
    a.part_dn = (uint64_t*)(b + kOffPartDn);
    a.sync = sync_w;
    a.status = status ? status : status_w;
    a.y = y;
    a.out_f32 = cfg->out_dtype == MOE_OUT_F32;
    return launch_gemv_layer(a, s, true, nullptr) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
