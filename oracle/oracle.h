/*
 * oracle.h -- CPU reference of the routed FP4 MoE expert FFN (decode step).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg load liboracle.so.  It shares no code, table or constant with
 * the CUDA path.
 *
 * Everything is computed in fp64 by the plain definitions, in the order the
 * sources give them.  Sources (page title, section):
 *   [A100]  "把不支持 FP4 的 A100 拉到 673 tok/s，回过神来发现比官方 API 还快"
 *           and its Japanese original "DeepSeek v4.1 Flashを動かしたくて
 *           FP4に対応していないA100を…"
 *   [8GB]   "在 8 GB 显卡上运行 510 GB 的 DeepSeek-V4.1-Flash——以及三个从不抛错的 Bug"
 * Readings where the sources are silent are stated at each function.
 *
 * Canonical expert layout (the layout the weights are published in, [8GB]
 * §方案：不重写模型，只迁移其存储: the three matrices of an expert sit next to
 * each other, its scales are a separate block).  Reading: order gate, up, down;
 * each matrix row-major [out][in]; two E2M1 codes per byte, element 2i in the
 * low nibble; one ue8m0 scale byte per 32 consecutive weights of a row.
 *   codes : gate [I][H/2] | up [I][H/2] | down [H][I/2]     (3*I*H/2 bytes)
 *   scales: gate [I][H/32] | up [I][H/32] | down [H][I/32]  (3*I*H/32 bytes)
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_ACT_BF16 = 0, ORC_ACT_E4M3_UE8M0_128 = 1, ORC_ACT_E2M1_UE8M0_32 = 2 };

/* One layer's expert set: codes[e] / scales[e] point to the canonical blobs of
 * expert e (NULL allowed for experts that the routing never selects; selecting
 * one is an error). */
typedef struct {
    int num_experts, hidden, inter;
    const uint8_t* const* codes;
    const uint8_t* const* scales;
} orc_layer;

double orc_e2m1_value(int code);
double orc_ue8m0_value(int s);
double orc_bf16_value(uint16_t bits);
uint16_t orc_bf16_rne(double v);
double orc_e4m3_value(uint8_t code);
uint8_t orc_e4m3_rne(double v);
int orc_ue8m0_for_amax(double amax);
void orc_act_quant_e4m3(const double* v, int n, int block, uint8_t* codes, uint8_t* scale_bytes);
int orc_e2m1_rne(double v);
int orc_ue8m0_for_amax_e2m1(double amax);
void orc_act_quant_e2m1(const double* v, int n, int block, uint8_t* codes, uint8_t* scale_bytes);
double orc_silu(double g);

int orc_matvec(const uint8_t* codes, const uint8_t* scales, int rows, int k,
               const double* v, double* out);
int orc_expert_ffn(const uint8_t* codes, const uint8_t* scales, int hidden, int inter,
                   const double* x, int act_mode, double* o);
int orc_moe_ffn(const orc_layer* layer, const uint16_t* x_bf16, int T, int topk,
                const int32_t* topk_idx, const float* topk_w, int act_mode,
                double* y, int nthreads);
int orc_route(const int32_t* topk_idx, int T, int topk, int num_experts,
              int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv);
void orc_rmsnorm_bf16(const double* x, int n, double eps, uint16_t* out);
int orc_moe_stack(const orc_layer* layers, int L, double* x, int T, int topk,
                  const int32_t* topk_idx, const float* topk_w, int act_mode,
                  double eps, int nthreads);

/* Router ahead of the path (the pages use a layer's router to pick its top-6
 * experts, [8GB] §提速之路：v1 到 v4, v4; the gating function itself is not on
 * the pages).  Reading: logits[t][e] = sum_h W[e][h] x[t][h] with W [E][H] and
 * x [T][H] in bf16; the k experts with the largest logits are selected in
 * descending order, ties to the lower expert id, a NaN logit below every
 * number; their weights are the softmax of the selected logits. */
void orc_router_logits(const uint16_t* x_bf16, const uint16_t* w_bf16, int T, int H, int E, double* logits);
int orc_topk_softmax(const double* logits, int T, int E, int k, int32_t* idx, double* w);

#ifdef __cplusplus
}
#endif
#endif
