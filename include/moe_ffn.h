/*
 * moe_ffn.h -- C ABI of the GB300 (sm_103a) routed FP4 MoE expert-FFN library.
 *
 * The operation is the routed expert FFN of an LLM decode step as described by
 *   [8GB]  "在 8 GB 显卡上运行 510 GB 的 DeepSeek-V4.1-Flash——以及三个从不抛错的 Bug"
 *   [A100] "把不支持 FP4 的 A100 拉到 673 tok/s，回过神来发现比官方 API 还快"
 * Each token chooses top-k experts of a layer ([8GB] §每 token 字节数决定一切:
 * 6 of 384); each expert is a SwiGLU block o = Wd (silu(Wg x) (.) (Wu x)) whose
 * weights are FP4 E2M1 codes with one ue8m0 power-of-two scale per 32 weights
 * ([A100] §质疑「不支持 FP4」这句话 for E2M1; [8GB] §RTX 50xx 上的三个从不抛错的
 * Bug for ue8m0); the token's output is y = sum_k w_k o_k.
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must be CUDA device (or managed)
 *    memory of the handle's device; host pointers are plain host memory.
 *  - Tensors are C-contiguous, with the shapes given, and their base addresses
 *    16-byte aligned; no strides are accepted.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *    except the *_host variants and moe_ffn_status is asynchronous: it only
 *    enqueues work and never waits for the device.
 *  - The caller owns every buffer it passes and must keep it alive until the
 *    stream has executed the call.  The handle owns its workspace.
 *  - Calls on one handle must be ordered (one stream, or externally
 *    synchronized): they share the handle's workspace.
 *  - Return value: MOE_OK (0) or a negative MOE_ERR_* code.  Argument errors
 *    are found on the host before anything is enqueued.  Errors that only the
 *    device can see (an expert id out of range, a NULL expert pointer) do not
 *    trap: the affected slot contributes zero and a sticky status word is set,
 *    read and cleared by moe_ffn_status().
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK                   0
#define MOE_ERR_INVALID_ARG     (-1)  /* bad pointer, size, alignment or config   */
#define MOE_ERR_CUDA            (-2)  /* a CUDA runtime call failed               */
#define MOE_ERR_OOM             (-3)  /* workspace allocation failed              */
#define MOE_ERR_UNSUPPORTED     (-4)  /* valid request this build does not serve  */
#define MOE_ERR_BAD_INDEX       (-5)  /* device saw an expert id outside [0, E)   */
#define MOE_ERR_DEVICE_TIMEOUT  (-6)  /* a bounded device-side wait gave up       */

/* Activation numerics (chosen explicitly; no hidden heuristic). */
enum {
    /* x (bf16) and the SwiGLU output h are carried at (better than) fp32
     * accuracy: products of exact E2M1 weights and activations, fp32 sums. */
    MOE_ACT_BF16 = 0,
    /* x and h are quantized to FP8 E4M3 with one ue8m0 scale per 128
     * consecutive elements (the last block of h may be shorter) before each
     * projection; the scale is 2^k with k the least integer such that
     * amax <= 448 * 2^k, and codes round to nearest even, saturating. */
    MOE_ACT_E4M3_UE8M0_128 = 1,
    /* x and h are quantized to FP4 E2M1 with one ue8m0 scale per 32
     * consecutive elements (MXFP4) before each projection; the scale is 2^k
     * with k the least integer such that amax <= 6 * 2^k, and codes round to
     * nearest even, saturating.  On the expert-major path a slot's activation
     * is then one E2M1 vector (the MMA's B operand is 4-bit, like the
     * weights) and the routing weight scales the slot's down output. */
    MOE_ACT_E2M1_UE8M0_32 = 2
};

enum { MOE_OUT_BF16 = 0, MOE_OUT_F32 = 1 };

typedef struct moe_ffn* moe_ffn_t;

typedef struct {
    int num_experts;      /* E, experts of one layer                         */
    int hidden;           /* H, model width; multiple of 64                  */
    int inter;            /* I, expert intermediate width; multiple of 64    */
    int topk;             /* k, experts per token, 1..16                     */
    int max_tokens;       /* largest T passed to forward calls               */
    int act_mode;         /* MOE_ACT_*                                       */
    int out_dtype;        /* MOE_OUT_*                                       */
    int gemm_min_tokens;  /* T >= this uses the grouped (expert-major) path;
                             0 selects MOE_DEFAULT_GEMM_MIN_TOKENS           */
} moe_ffn_config;

/* Below this many tokens a layer runs slot-major: each (token, expert) slot
 * streams its expert's weights (batch 1 reads every chosen expert once; two
 * launches per layer).  From it on, the layer runs expert-major: the slots are
 * sorted by expert ([8GB] §提速之路：v1 到 v4, the per-expert token grouping)
 * and each expert's weights are multiplied against up to 8 of its slots per
 * tensor-core MMA, so an expert chosen by many tokens is streamed from HBM
 * once per layer (four launches: route, prep, layer, combine).  Both paths
 * compute the same function within the float tolerance. */
#define MOE_DEFAULT_GEMM_MIN_TOKENS 16

/* One layer's experts.  experts is a DEVICE array of E DEVICE pointers, each
 * to one expert's packed blob (moe_ffn_packed_expert_bytes bytes, 16-byte
 * aligned) made by moe_ffn_pack_expert.  A NULL entry is allowed for an expert
 * that is never routed to. */
typedef struct {
    const uint8_t* const* experts;
} moe_expert_table;

/* Bytes of one expert's packed blob: every code and scale byte of the
 * published layout ([8GB] §方案：不重写模型，只迁移其存储: 3*I*H/2 = 17.7 MB of
 * codes and 3*I*H/32 = 1.1 MB of scales at H = 4096, I = 2880), re-laid out,
 * plus 256 padding bytes per half-unit scale atom (H/128 of them when
 * I % 128 == 64): 18,808,832 bytes at H = 4096, I = 2880.  Returns 0 for an
 * invalid config. */
size_t moe_ffn_packed_expert_bytes(const moe_ffn_config* cfg);

/* Validate cfg, select `device`, allocate the workspace (sized from
 * max_tokens) and return a handle in *out.  Errors: INVALID_ARG (config),
 * UNSUPPORTED (shape outside what the kernels serve), OOM, CUDA. */
int moe_ffn_create(moe_ffn_t* out, const moe_ffn_config* cfg, int device);

/* Re-lay one expert once, at load time, into the order the kernels stream
 * ([A100] §但 CPU 也没那么快: reorder weights at load time into the order the
 * compute unit consumes).  Input: the published layout, device memory:
 *   canon_codes : gate [I][H/2] | up [I][H/2] | down [H][I/2]   (low nibble =
 *                 even element), canon_scales: gate [I][H/32] | up [I][H/32] |
 *                 down [H][I/32] (one ue8m0 byte per 32 weights of a row).
 * Output: packed (moe_ffn_packed_expert_bytes), device memory, 16-byte
 * aligned, not overlapping the inputs: tiles of 128 rows, each a run of
 * 128-wide K units, each unit its codes in the tensor-core operand order
 * followed by its 512-byte scale atom, so that the kernels move a run of
 * units, codes and scales together, with one bulk copy. */
int moe_ffn_pack_expert(moe_ffn_t h, const void* canon_codes, const void* canon_scales, void* packed,
                        void* stream);

/* One MoE layer for T tokens (0 <= T <= max_tokens):
 *   x        device bf16 [T][H]
 *   topk_idx device int32 [T][k]   expert ids (repeats in a row are allowed)
 *   topk_w   device fp32  [T][k]   combine weights, used as given
 *   tbl      host struct of device pointer arrays (see moe_expert_table)
 *   y        device [T][H], bf16 or fp32 per cfg.out_dtype; y must not alias x
 * y[t] = sum_{k} topk_w[t,k] * FFN_{topk_idx[t,k]}(x[t]).  Deterministic:
 * repeated calls give bitwise identical y.  The layer's first kernels read
 * topk_idx, topk_w and the expert table before they wait for the stream's
 * previous kernel (programmatic dependent launch), so these must be written by
 * stream work that completes before a dependent launch may begin: an ordinary
 * kernel or copy, or moe_router_topk / moe_router_select (which let the next
 * launch start only once their outputs are written) -- not by a kernel that
 * lets dependents launch early, unless moe_ffn_set_routing_wait(h, 1) is set. */
int moe_ffn_forward(moe_ffn_t h, const void* x, const int32_t* topk_idx, const float* topk_w,
                    const moe_expert_table* tbl, void* y, int T, void* stream);

/* on = 1: the layer's kernels read topk_idx, topk_w and the expert table only
 * after they have waited for the stream's previous kernel, so those inputs may
 * come from a kernel that lets its dependents launch early (programmatic
 * dependent launch) and writes them afterwards.  The weight stream then starts
 * only once that kernel has completed (at batch 1 the layer loses the overlap
 * with the previous kernel's tail).  on = 0 (the default): as documented at
 * moe_ffn_forward.  Applies to moe_ffn_forward, moe_ffn_forward_host and
 * moe_stack_forward on this handle; results are identical either way.  With
 * it on, moe_router_topk on this handle lets the next launch start at once
 * (before its outputs are written): only kernels that wait before reading them
 * may follow it.  A change drops the handle's cached graphs (after waiting for
 * the device), so the next calls capture new ones.  Errors: INVALID_ARG, CUDA. */
int moe_ffn_set_routing_wait(moe_ffn_t h, int on);

/* moe_ffn_forward with HOST x / topk_idx / topk_w / y (any host memory; the
 * call waits for `stream` before it returns).  Small batches (x and y
 * together at most 128 KB): the inputs are packed into a page-locked staging
 * buffer of the handle that is mapped into the device's address space
 * (allocated on the first such call); the layer's kernels read x, topk_idx and
 * topk_w from it and write y into it over the host link, with no copy
 * operations, run as one CUDA graph on `stream` (captured on the first call
 * for each (T, tbl->experts) pair, at most 8 kept; launched one by one while
 * profiling is enabled); then y is copied out on the host.  Larger batches:
 * x, topk_idx and topk_w are copied straight from the caller's buffers into
 * device memory (pinned memory makes these copies DMA-only) and y straight
 * back.  The expert table stays in device memory.  Returns MOE_ERR_OOM if the
 * staging buffer cannot be allocated. */
int moe_ffn_forward_host(moe_ffn_t h, const void* x_host, const int32_t* topk_idx_host,
                         const float* topk_w_host, const moe_expert_table* tbl, void* y_host,
                         int T, void* stream);

/* Token -> expert grouping on the device ([8GB] §提速之路：v1 到 v4: the
 * per-expert token search, done without a host round trip).  Device outputs:
 *   counts  int32 [E]      slots routed to each expert
 *   offsets int32 [E+1]    exclusive prefix sum of counts
 *   perm    int32 [T*k]    slot ids j = t*k + kk ordered by (expert, t, kk)
 *   inv     int32 [T*k]    inv[perm[p]] = p
 * Bit-exact and deterministic.  Out-of-range ids set MOE_ERR_BAD_INDEX in the
 * status word and are left out of every output (their inv entry is -1). */
int moe_ffn_route(moe_ffn_t h, const int32_t* topk_idx, int T, int32_t* counts,
                  int32_t* offsets, int32_t* perm, int32_t* inv, void* stream);

/* Activation quantizer of the MOE_ACT_E4M3_UE8M0_128 mode ([8GB] §RTX 50xx
 * 上的三个从不抛错的 Bug, item 2: the ue8m0 act_quant step).  Device in/out:
 *   x       bf16 [rows][n]
 *   codes   uint8 [rows][n]          E4M3 codes
 *   scales  uint8 [rows][ceil(n/128)] ue8m0 bytes (2^(s-127))
 * Bit-exact and deterministic. n must be a multiple of 32. */
int moe_ffn_act_quant(moe_ffn_t h, const void* x, int rows, int n, uint8_t* codes,
                      uint8_t* scales, void* stream);

/* The router ahead of the path (the pages pick each token's top-6 experts of a
 * layer with that layer's router, [8GB] §提速之路：v1 到 v4, v4; the gating
 * function is not on the pages).  Reading: for each token t,
 *   logits[t][e] = sum_h router_w[e][h] * x[t][h]      (fp32 accumulation)
 * the k = cfg.topk experts with the largest logits, in descending order (ties
 * to the lower expert id; a NaN logit ranks after every number), and
 *   topk_w[t][i] = exp(l_i - l_0) / sum_j exp(l_j - l_0)  over the selected.
 *   x        device bf16 [T][H];  router_w device bf16 [E][H]
 *   logits   optional device fp32 [T][E] output (NULL: kept in the workspace)
 *   topk_idx device int32 [T][k], topk_w device fp32 [T][k] -- the routing
 *            inputs of moe_ffn_forward.
 * Deterministic.  One token with E <= 256: one launch of one thread-block
 * cluster (a warp per expert row; the selection in the cluster's first CTA,
 * from the logits gathered in its shared memory), where the device runs
 * clusters of 8 or 16 CTAs.  Up to 8 tokens otherwise: one launch, the logits
 * streaming the weights on the CUDA cores and the last CTA of each token tile
 * selecting.  Above 8 tokens (H a multiple of 128): tcgen05 bf16 MMAs in
 * split-K partial sums, then a selection launch that adds them in a fixed
 * order.  Every path gives the same logits for a one-token call.
 * UNSUPPORTED beyond 1024 experts or H above 102,400. */
int moe_router_topk(moe_ffn_t h, const void* x, const void* router_w, int T, float* logits,
                    int32_t* topk_idx, float* topk_w, void* stream);

/* The selection and softmax of moe_router_topk alone, from given device fp32
 * logits [T][E] (bit-exact selection for given logits). */
int moe_router_select(moe_ffn_t h, const float* logits, int T, int32_t* topk_idx, float* topk_w,
                      void* stream);

/* Expert-sharing batch planner (host code; needs no GPU and no handle).
 * Alike prompts route to alike experts, so batching alike sequences cuts the
 * distinct experts a layer streams ([A100] §批处理不是「同时处理几个人」: 216 ->
 * 156 in one layer; the pages give no algorithm).  Reading: a greedy cover --
 * a batch starts from the lowest-numbered unplaced sequence and grows, until
 * it holds B, by the unplaced sequence adding the fewest experts not yet in
 * the batch summed over the layers (ties to the lower number).
 *   sig    host int32 [N][L][topk]: each sequence's signature, its recent
 *          top-k expert ids per layer (-1: none); ids in [-1, E)
 *   order  host int32 [N] output: the sequences in batch order (batch b is
 *          order[bB .. min((b+1)B, N)))
 * Deterministic; O(N^2 L topk).  INVALID_ARG on a bad size or id. */
int moe_batch_plan(const int32_t* sig, int N, int L, int topk, int E, int B, int32_t* order);

/* The metric of the planner: the distinct experts each (batch, layer) touches
 * when the sequences, in `order`, are cut into batches of B.
 *   routing   host int32 [N][L][topk] (e.g. the next step's routing)
 *   order     host int32 [N], a permutation of 0..N-1 (else INVALID_ARG)
 *   distinct  host int32 [ceil(N/B)][L] output */
int moe_batch_distinct(const int32_t* routing, const int32_t* order, int N, int L, int topk, int E, int B,
                       int32_t* distinct);

/* Host-resident experts with an HBM cache and prefetch ([8GB] §提速之路：v1 到
 * v4 and [A100] §但 CPU 也没那么快 stream experts that do not fit on the GPU
 * and hide the copies; here host memory sits behind NVLink-C2C).  Host code.
 *   create   cfg: the layer's sizes; host_blobs: host array [E] of HOST
 *            pointers (16-byte aligned, page-locked for asynchronous copies)
 *            to packed expert blobs (moe_ffn_pack_expert's layout); slots:
 *            expert-sized slots of device memory.  OOM if they do not fit.
 *   fetch    ids: host int32 [n] expert ids (-1 ignored).  Makes them
 *            resident: a miss takes the least recently used slot that the
 *            request does not use (lowest slot on ties) and is copied there
 *            on one of four internal copy streams (round-robin); `stream` then waits for the
 *            copies and receives the layer's table in *tbl (a device array of
 *            E pointers, NULL for experts not resident) for launches on
 *            `stream` until the next fetch.  INVALID_ARG if the request holds
 *            more distinct experts than there are slots.
 *   prefetch the same copies for experts expected next, without waiting;
 *            slots the previous fetch returned stay intact until the work
 *            enqueued on `stream` before this call is done.
 * All calls of one cache must use one stream.  A slot is never overwritten
 * while work enqueued before the call that evicts it may read it. */
typedef struct moe_expert_cache_s* moe_expert_cache_t;
int moe_expert_cache_create(const moe_ffn_config* cfg, int device, const void* const* host_blobs, int slots,
                            moe_expert_cache_t* out);
int moe_expert_cache_fetch(moe_expert_cache_t c, const int32_t* ids, int n, void* stream, moe_expert_table* tbl);
int moe_expert_cache_prefetch(moe_expert_cache_t c, const int32_t* ids, int n, void* stream);
/* The slot holding expert e, or -1. */
int moe_expert_cache_slot(moe_expert_cache_t c, int expert);
/* Fetch hits and misses so far, and bytes copied by fetches and prefetches. */
int moe_expert_cache_stats(moe_expert_cache_t c, long long* hits, long long* misses, long long* bytes);
/* Waits for the copies in flight and frees the cache. */
void moe_expert_cache_destroy(moe_expert_cache_t c);

/* L-layer decode step on a residual stream ([A100] §然后又发现每 token 启动
 * 2000 次内核: RMSNorm and the MoE per layer, launched as a handful of
 * dispatches): for l = 0..L-1,
 *   u = bf16(x / sqrt(mean(x^2) + 1e-6))   (unit norm weight)
 *   x = x + moe_l(u)
 *   x        device fp32 [T][H], updated in place
 *   tbls     host array [L] of expert tables (one per layer)
 *   topk_idx device int32 [L][T][k];  topk_w device fp32 [L][T][k]
 * The whole step is captured once into a CUDA graph per (T, L, pointer set)
 * and replayed; later calls with the same pointers only replay it. */
int moe_stack_forward(moe_ffn_t h, float* x, const moe_expert_table* tbls,
                      const int32_t* topk_idx, const float* topk_w, int L, int T,
                      void* stream);

/* moe_stack_forward with HOST x (fp32 [T][H], updated in place), topk_idx and
 * topk_w (int32 / fp32 [L][T][k]); the call waits for `stream` before it
 * returns.  The inputs are packed into a page-locked staging buffer of the
 * handle that is mapped into the device's address space (grown on demand),
 * and one CUDA graph per (T, L, expert tables) copies them into device memory
 * with one kernel, runs the L layers and copies x back into the staging
 * buffer, from which it is copied out on the host.  Results equal
 * moe_stack_forward's bit for bit.  Returns MOE_ERR_OOM if the staging
 * buffers cannot be allocated. */
int moe_stack_forward_host(moe_ffn_t h, float* x_host, const moe_expert_table* tbls,
                           const int32_t* topk_idx_host, const float* topk_w_host, int L, int T, void* stream);

/* Per-kernel timing, a tracing aid.  While enabled, forward calls record a
 * CUDA event pair around each of their kernel launches on the call's stream
 * (this also stops a kernel's prologue from overlapping the previous kernel).
 * moe_ffn_profile_read waits for the recorded events, writes the summed
 * milliseconds and launch counts per phase (MOE_PHASE_*; arrays of
 * MOE_NUM_PHASES entries, host memory) and resets the record.  The stack
 * entry point is not traced.  Errors: INVALID_ARG, CUDA. */
enum {
    MOE_PHASE_PREP = 0,      /* activation prep (and fused RMSNorm)         */
    MOE_PHASE_GATE_UP = 1,   /* the layer kernel: gate/up + SwiGLU + down
                                (+ the combine on the slot-major path); on
                                the kind::mxf8f6f4 expert-major path its two
                                launches, gate/up and down                  */
    MOE_PHASE_DOWN = 2,      /* the combine kernel (expert-major path)      */
    MOE_PHASE_ROUTE = 3,     /* token -> expert grouping (moe_ffn_route and
                                the expert-major path's first kernel)       */
    MOE_PHASE_ACT_QUANT = 4, /* E4M3 activation quantizer (and h's, on the
                                kind::mxf8f6f4 expert-major path)           */
    MOE_PHASE_ROUTER = 5,    /* router logits + top-k + softmax (moe_router_topk) */
    MOE_NUM_PHASES = 8
};
int moe_ffn_profile_enable(moe_ffn_t h, int on);
int moe_ffn_profile_read(moe_ffn_t h, double* ms, int* launches);

/* The tensor-core operation of the expert-major path for quantized
 * activations.
 *   MOE_MMA_MXF8F6F4 ("direct"): the activations as they are, one slot per MMA
 *     column -- E4M3 mode (MOE_ACT_E4M3_UE8M0_128): tcgen05.mma
 *     kind::mxf8f6f4, the E2M1 weights times the E4M3 rows, groups of up to
 *     224 slots of an expert (one MMA issuer and a scale-copy thread) where
 *     T * topk >= 128 * E, else up to 64 (three issuers); E2M1 mode
 *     (MOE_ACT_E2M1_UE8M0_32): kind::mxf4, the E2M1 weights as the blob holds
 *     them times the E2M1 rows (FP4 on both sides), groups of up to 224.  Six
 *     launches (route, prep, gate/up, h quantizer, down, combine).
 *   MOE_MMA_MXF4_PIECES: kind::mxf4 with the activations carried as E2M1
 *     pieces (8 per E4M3 value, groups of up to 8 slots; 1 per E2M1 value,
 *     groups of up to 16).
 *   MOE_MMA_AUTO (the default): direct where T * topk >= 128 * E
 *     (tensor-bound shapes, where it is several times faster), else pieces
 *     (HBM-bound decode batches, where that streams the weights faster).
 * All compute the same function within the float tolerance ([8GB] §三个从不抛错的
 * Bug, item 2, fixes the E4M3 + ue8m0-per-128 activation format; the pages
 * leave the MMA to the build).  The bf16 mode and the slot-major path are not
 * affected.  A change drops the handle's cached graphs (after waiting for the
 * device).  Errors: INVALID_ARG, CUDA. */
enum { MOE_MMA_AUTO = 0, MOE_MMA_MXF4_PIECES = 1, MOE_MMA_MXF8F6F4 = 2 };
int moe_ffn_set_mma_kind(moe_ffn_t h, int kind);

/* Measurement mode of the slot-major path (the sources have no counterpart;
 * it serves timing): while on, moe_ffn_forward calls that take the
 * slot-major path launch only the layer kernel, which reuses the activation
 * pieces that the last full call left in the handle's workspace -- its
 * output is the layer applied to that call's x with this call's routing and
 * experts.  A CUDA graph of such calls, back to back, measures the layer
 * kernel's duration as it runs inside a step (each launch overlapping the
 * previous one's tail, as programmatic dependent launch allows), which the
 * profiling events above cannot (they separate the launches).  The expert-
 * major path and moe_stack_forward are not affected.  Errors: INVALID_ARG. */
int moe_ffn_profile_layer_only(moe_ffn_t h, int on);

/* moe_ffn_forward without a handle and without allocating.  The sources have
 * no counterpart of this call; it serves callers that may not allocate device
 * memory on their call path -- hosts that own every device allocation and give
 * a library no allocator of its own (embedded inference runtimes, plugin hosts
 * with a fixed memory budget), where moe_ffn_create's cudaMalloc is not
 * allowed.  It calls no cudaMalloc, cudaFree or allocating library routine.
 *
 * Same arguments and result as moe_ffn_forward (x, topk_idx, topk_w, y are
 * device pointers; cfg is read on the host; only MOE_ACT_BF16), plus:
 *   device  the CUDA device to run on (made current for the call)
 *   status  optional DEVICE int; when non-NULL the kernels OR the device-side
 *           status bits into it (1 = expert id out of range, 2 = a bounded
 *           wait timed out); the caller clears it.  NULL: not reported.
 * Scratch memory is one fixed 4 MiB array in this library's device code,
 * present on every GPU that loads the library until the process exits and
 * shared by all calls.  A call whose scratch need (for T tokens: activations,
 * h, split-K partial sums and counters; about 240 KB per token at H = 4096,
 * I = 2880, top-6) exceeds it returns MOE_ERR_UNSUPPORTED before enqueuing
 * anything.  Each call clears the counters that must start at zero on
 * `stream`; the array otherwise keeps the previous call's contents, and calls
 * whose work overlaps on the GPU race on it, so calls must be ordered on one
 * stream.  The first call on a device resolves the array's device address and
 * sets kernel attributes; make that first call before any stream capture.
 * Calls look the address up again and redo that set-up when it changed (a
 * device reset made a new context). */
int moe_ffn_forward_noalloc(const moe_ffn_config* cfg, int device, const void* x,
                            const int32_t* topk_idx, const float* topk_w,
                            const moe_expert_table* tbl, void* y, int T, int* status,
                            void* stream);

/* Test hooks for the failure paths.  The sources have no counterpart of
 * these; they exist so that tests can drive the error handling without a GPU
 * fault, trap or hang.
 *
 * moe_ffn_test_set_wait: later calls on h run the slot-major layer kernel
 * with every bounded device-side wait giving up after wait_ns nanoseconds
 * (at 2 GHz SM clock; 0: the default, 2 s), and with withhold != 0 its first
 * CTA never reports its finished gate/up groups, so that the other CTAs' waits
 * for the whole of h run out: the call completes, y is incomplete, and
 * moe_ffn_status returns MOE_ERR_DEVICE_TIMEOUT.  Graphs the handle captured earlier keep the
 * settings they were captured with.  Errors: INVALID_ARG.
 *
 * moe_ffn_test_fail_allocs: the next n device or page-locked allocations the
 * library makes (any handle, cache or staging buffer) fail as if out of
 * memory; n = 0 clears.  The calls that make them return MOE_ERR_OOM.
 *
 * moe_ffn_test_copy_h: after an expert-major call in the E4M3 mode on the
 * kind::mxf8f6f4 path, copies (enqueued on `stream`, device to device) the
 * fp32 h = silu(g) u of each of the call's first n sorted slots, before its
 * E4M3 quantization, into h_dst ([n][inter] floats) and the slot order into
 * perm_dst ([n] int32: sorted position -> slot t * topk + k), so that a test
 * can check h itself and the down projection on the GPU's own quantized h.
 * Errors: INVALID_ARG (no such workspace on this handle, n out of range). */
int moe_ffn_test_set_wait(moe_ffn_t h, unsigned long long wait_ns, int withhold);
int moe_ffn_test_copy_h(moe_ffn_t h, float* h_dst, int32_t* perm_dst, int n, void* stream);
void moe_ffn_test_fail_allocs(int n);

/* Wait for `stream`, then return and clear the sticky device status:
 * MOE_OK, MOE_ERR_BAD_INDEX or MOE_ERR_DEVICE_TIMEOUT (or MOE_ERR_CUDA if the
 * read itself failed). */
int moe_ffn_status(moe_ffn_t h, void* stream);

/* Static message for a MOE_* code. */
const char* moe_ffn_strerror(int code);

/* Free the workspace and cached graphs.  The caller must first make sure no
 * enqueued call on the handle is still pending.  NULL is a no-op. */
void moe_ffn_destroy(moe_ffn_t h);

#ifdef __cplusplus
}
#endif
#endif /* MOE_FFN_H */
