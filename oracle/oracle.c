/*
 * oracle.c -- plain, slow CPU reference of the routed FP4 MoE expert FFN.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product library.  It shares no
 * code with the CUDA path.  All arithmetic is fp64; every weight is decoded
 * from the 16-entry E2M1 table and its ue8m0 scale one element at a time.
 * Source titles ([A100], [8GB]) are spelled out in oracle.h.
 */
#define _GNU_SOURCE
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- formats */

/* E2M1: 1 sign, 2 exponent, 1 mantissa bit.  The eight magnitudes, doubled,
 * are the integers 0,1,2,3,4,6,8,12 ([A100] §质疑「不支持 FP4」这句话; the
 * Japanese original lists them in §「FP4非対応」という言葉を疑う).  Codes 8..15
 * are the negatives of codes 0..7 (code 8 is -0). */
static const double E2M1_MAGNITUDE[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code)
{
    double m = E2M1_MAGNITUDE[code & 7];
    return (code & 8) ? -m : m;
}

/* ue8m0: exponent-only scale byte, value 2^(s-127) ([8GB] §RTX 50xx 上的三个
 * 从不抛错的 Bug names the format).  Reading: s = 255 is NaN, as in the OCP MX
 * scale type; s = 0 is 2^-127, computed exactly. */
double orc_ue8m0_value(int s)
{
    if (s == 255) return NAN;
    return ldexp(1.0, s - 127);
}

double orc_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Nearest bf16 (8 significant bits) to v, ties to even, computed directly from
 * the fp64 value so that there is no double rounding through fp32. */
uint16_t orc_bf16_rne(double v)
{
    if (isnan(v)) return 0x7FC0;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else if (a < ldexp(1.0, -126)) {
        r = ldexp(nearbyint(ldexp(a, 133)), -133);     /* subnormal grid 2^-133 */
    } else {
        int e;
        frexp(a, &e);                                   /* a in [2^(e-1), 2^e) */
        r = ldexp(nearbyint(ldexp(a, 8 - e)), e - 8);
    }
    float f = (float)r;                                 /* exact, or inf on overflow */
    if (isinf(f) || r >= ldexp(1.0, 128)) f = INFINITY;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)((u >> 16) | (neg ? 0x8000u : 0u));
}

/* E4M3 (bias 7, no infinities, S.1111.111 is NaN, largest finite 448). */
double orc_e4m3_value(uint8_t code)
{
    int e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);               /* subnormal: m/8 * 2^-6 */
    else        v = ldexp((double)(8 + m), e - 10);     /* (1 + m/8) * 2^(e-7)   */
    return (code & 0x80) ? -v : v;
}

/* Round v to the nearest E4M3 value, ties to even mantissa, saturating to
 * +-448.  The sign of v is kept (a negative value that rounds to zero gives
 * the -0 code 0x80). */
uint8_t orc_e4m3_rne(double v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    int code;
    if (a >= 448.0) {
        code = 0x7E;
    } else if (a < ldexp(1.0, -6)) {
        code = (int)nearbyint(ldexp(a, 9));              /* 0..8; 8 is 2^-6, the first normal */
    } else {
        int e;
        frexp(a, &e);
        int E = e - 1;                                  /* a in [2^E, 2^(E+1)) */
        int m = (int)nearbyint(ldexp(a, 3 - E));        /* 8..16 */
        code = ((E + 7) << 3) + (m - 8);                /* m = 16 carries into the exponent */
        if (code > 0x7E) code = 0x7E;
    }
    return (uint8_t)(code | sign);
}

/* Scale byte of an activation block: 2^k with k the least integer such that
 * amax <= 448 * 2^k, found by exact comparisons.  Reading (the sources only
 * name the ue8m0 act_quant kernel): amax = 0 gives k = 0; k is clamped to
 * [-127, 127]; a non-finite amax gives the NaN byte 255. */
int orc_ue8m0_for_amax(double amax)
{
    if (!(amax == amax) || isinf(amax)) return 255;
    if (amax == 0.0) return 127;
    int e;
    frexp(amax, &e);
    int k = e - 9;
    while (amax > ldexp(448.0, k)) k++;
    while (amax <= ldexp(448.0, k - 1)) k--;
    if (k < -127) k = -127;
    if (k > 127) k = 127;
    return k + 127;
}

/* Quantize v[0..n) in consecutive blocks of `block` elements (the last block
 * may be shorter) to E4M3 codes with one ue8m0 scale byte per block. */
void orc_act_quant_e4m3(const double* v, int n, int block, uint8_t* codes, uint8_t* scale_bytes)
{
    for (int b0 = 0, b = 0; b0 < n; b0 += block, b++) {
        int nb = (n - b0 < block) ? n - b0 : block;
        double amax = 0.0;
        for (int i = 0; i < nb; i++) {
            double a = fabs(v[b0 + i]);
            if (a > amax || a != a) amax = a;
        }
        int s = orc_ue8m0_for_amax(amax);
        scale_bytes[b] = (uint8_t)s;
        for (int i = 0; i < nb; i++)
            codes[b0 + i] = (s == 255) ? 0x7F : orc_e4m3_rne(ldexp(v[b0 + i], 127 - s));
    }
}

/* ------------------------------------------------ E2M1 activations (MXFP4) */

/* Nearest E2M1 value to v (the grid 0, 0.5, 1, 1.5, 2, 3, 4, 6 and
 * negatives), ties to the even mantissa bit, saturating to +-6; returned as
 * the 4-bit code (sign in bit 3).  Reading (the sources give FP4 weights,
 * [A100] §FP4の正体, not FP4 activations): activations are rounded the way a
 * float is rounded to a narrower float, round-to-nearest-even. */
int orc_e2m1_rne(double v)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs(v);
    if (!(a == a)) return 0;
    if (a >= 6.0) return 7 | sign;                              /* saturate */
    int best = 0;
    for (int c = 1; c < 8; c++) {
        double d = fabs(orc_e2m1_value(c) - a), db = fabs(orc_e2m1_value(best) - a);
        if (d < db || (d == db && (c & 1) == 0)) best = c;     /* tie: even mantissa (code bit 0) */
    }
    return best | sign;
}

/* Scale byte of an E2M1 activation block: 2^k with k the least integer such
 * that amax <= 6 * 2^k (6 is E2M1's largest value), found by exact
 * comparisons -- the ue8m0 convention of the model's activation quantizer
 * ([8GB] §三个从不抛错的 Bug, 2: scales are ue8m0) with E2M1's range.
 * Readings: amax = 0 gives k = 0; k is clamped to [-126, 127]; a non-finite
 * amax gives the NaN byte 255. */
int orc_ue8m0_for_amax_e2m1(double amax)
{
    if (!(amax == amax) || isinf(amax)) return 255;
    if (amax == 0.0) return 127;
    int e;
    frexp(amax, &e);
    int k = e - 3;
    while (amax > ldexp(6.0, k)) k++;
    while (amax <= ldexp(6.0, k - 1)) k--;
    if (k < -126) k = -126;
    if (k > 127) k = 127;
    return k + 127;
}

/* Quantize v[0..n) in consecutive blocks of `block` elements (the last block
 * may be shorter) to E2M1 codes (one per byte here) with one ue8m0 scale byte
 * per block: code = nearest E2M1 to v * 2^-k. */
void orc_act_quant_e2m1(const double* v, int n, int block, uint8_t* codes, uint8_t* scale_bytes)
{
    for (int b0 = 0, b = 0; b0 < n; b0 += block, b++) {
        int nb = (n - b0 < block) ? n - b0 : block;
        double amax = 0.0;
        for (int i = 0; i < nb; i++) {
            double a = fabs(v[b0 + i]);
            if (a > amax || a != a) amax = a;
        }
        int s = orc_ue8m0_for_amax_e2m1(amax);
        scale_bytes[b] = (uint8_t)s;
        for (int i = 0; i < nb; i++)
            codes[b0 + i] = (uint8_t)((s == 255) ? 0 : orc_e2m1_rne(ldexp(v[b0 + i], 127 - s)));
    }
}

/* silu(g) = g * sigmoid(g) = g / (1 + e^-g). */
double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* ------------------------------------------------------------ arithmetic */

/* out[r] = sum_i W[r][i] * v[i], W given as E2M1 codes (two per byte, element
 * 2i in the low nibble) and one ue8m0 byte per 32 weights of a row. */
int orc_matvec(const uint8_t* codes, const uint8_t* scales, int rows, int k,
               const double* v, double* out)
{
    if (k % 32 != 0) return -1;
    for (int r = 0; r < rows; r++) {
        const uint8_t* crow = codes + (size_t)r * (k / 2);
        const uint8_t* srow = scales + (size_t)r * (k / 32);
        double acc = 0.0;
        for (int i = 0; i < k; i++) {
            int byte = crow[i / 2];
            int nib = (i & 1) ? (byte >> 4) : (byte & 15);
            double w = orc_e2m1_value(nib) * orc_ue8m0_value(srow[i / 32]);
            acc += w * v[i];
        }
        out[r] = acc;
    }
    return 0;
}

static void quant_dequant_e2m1(double* v, int n, int block)
{
    uint8_t* c = (uint8_t*)malloc((size_t)n);
    uint8_t* s = (uint8_t*)malloc((size_t)(n + block - 1) / block);
    orc_act_quant_e2m1(v, n, block, c, s);
    for (int i = 0; i < n; i++)
        v[i] = (s[i / block] == 255) ? NAN : orc_e2m1_value(c[i]) * orc_ue8m0_value(s[i / block]);
    free(c);
    free(s);
}

static void quant_dequant(double* v, int n, int block)
{
    uint8_t* c = (uint8_t*)malloc((size_t)n);
    uint8_t* s = (uint8_t*)malloc((size_t)(n + block - 1) / block);
    orc_act_quant_e4m3(v, n, block, c, s);
    for (int i = 0; i < n; i++)
        v[i] = orc_e4m3_value(c[i]) * orc_ue8m0_value(s[i / block]);
    free(c);
    free(s);
}

/* One expert: o = Wd * (silu(Wg*x) (.) (Wu*x)).  In the E4M3 activation mode
 * x and h are first replaced by their per-128 E4M3/ue8m0 quantized values, in
 * the E2M1 mode by their per-32 E2M1/ue8m0 (MXFP4) quantized values. */
int orc_expert_ffn(const uint8_t* codes, const uint8_t* scales, int hidden, int inter,
                   const double* x, int act_mode, double* o)
{
    int H = hidden, I = inter;
    if (H % 32 || I % 32) return -1;
    double* xin = (double*)malloc(sizeof(double) * H);
    double* g = (double*)malloc(sizeof(double) * I);
    double* u = (double*)malloc(sizeof(double) * I);
    memcpy(xin, x, sizeof(double) * H);
    if (act_mode == ORC_ACT_E4M3_UE8M0_128) quant_dequant(xin, H, 128);
    if (act_mode == ORC_ACT_E2M1_UE8M0_32) quant_dequant_e2m1(xin, H, 32);

    size_t gu_codes = (size_t)I * H / 2, gu_scales = (size_t)I * H / 32;
    orc_matvec(codes, scales, I, H, xin, g);
    orc_matvec(codes + gu_codes, scales + gu_scales, I, H, xin, u);
    for (int i = 0; i < I; i++) g[i] = orc_silu(g[i]) * u[i];      /* g now holds h */
    if (act_mode == ORC_ACT_E4M3_UE8M0_128) quant_dequant(g, I, 128);
    if (act_mode == ORC_ACT_E2M1_UE8M0_32) quant_dequant_e2m1(g, I, 32);
    orc_matvec(codes + 2 * gu_codes, scales + 2 * gu_scales, H, I, g, o);
    free(xin);
    free(g);
    free(u);
    return 0;
}

/* ------------------------------------------------------------- the layer */

typedef struct {
    const orc_layer* layer;
    const uint16_t* x_bf16;
    int topk, act_mode, nslots, stride, first;
    const int32_t* idx;
    double* o;                 /* [nslots][H] */
    int err;
} ffn_job;

static void* ffn_worker(void* arg)
{
    ffn_job* j = (ffn_job*)arg;
    const orc_layer* L = j->layer;
    int H = L->hidden;
    double* x = (double*)malloc(sizeof(double) * H);
    for (int s = j->first; s < j->nslots; s += j->stride) {
        int t = s / j->topk, e = j->idx[s];
        if (e < 0 || e >= L->num_experts || !L->codes[e] || !L->scales[e]) { j->err = -2; break; }
        for (int i = 0; i < H; i++) x[i] = orc_bf16_value(j->x_bf16[(size_t)t * H + i]);
        if (orc_expert_ffn(L->codes[e], L->scales[e], H, L->inter, x, j->act_mode,
                           j->o + (size_t)s * H)) { j->err = -1; break; }
    }
    free(x);
    return NULL;
}

/* y[t] = sum_{k=0..topk-1} w[t,k] * FFN_{idx[t,k]}(x[t]), summed in the fixed
 * order k = 0..topk-1 ([8GB] §每 token 字节数决定一切: each token uses 6 of
 * the 384 experts of a layer; the weighted sum is the plain MoE combine).
 * topk_w is used as given.  Slots run in parallel on `nthreads` threads. */
int orc_moe_ffn(const orc_layer* layer, const uint16_t* x_bf16, int T, int topk,
                const int32_t* topk_idx, const float* topk_w, int act_mode,
                double* y, int nthreads)
{
    int H = layer->hidden, nslots = T * topk;
    if (T < 0 || topk <= 0) return -1;
    if (T == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nslots) nthreads = nslots;
    double* o = (double*)calloc((size_t)nslots * H, sizeof(double));
    if (!o) return -3;
    ffn_job* jobs = (ffn_job*)calloc((size_t)nthreads, sizeof(ffn_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; i++) {
        jobs[i] = (ffn_job){layer, x_bf16, topk, act_mode, nslots, nthreads, i, topk_idx, o, 0};
        if (i > 0) pthread_create(&th[i], NULL, ffn_worker, &jobs[i]);
    }
    ffn_worker(&jobs[0]);
    int err = jobs[0].err;
    for (int i = 1; i < nthreads; i++) {
        pthread_join(th[i], NULL);
        if (jobs[i].err) err = jobs[i].err;
    }
    if (!err) {
        for (int t = 0; t < T; t++)
            for (int i = 0; i < H; i++) {
                double acc = 0.0;
                for (int k = 0; k < topk; k++)
                    acc += (double)topk_w[t * topk + k] * o[((size_t)t * topk + k) * H + i];
                y[(size_t)t * H + i] = acc;
            }
    }
    free(o);
    free(jobs);
    free(th);
    return err;
}

/* Token -> expert grouping by counting sort ([8GB] §提速之路：v1 到 v4 finds
 * each expert's tokens with a per-expert search; this is the same grouping
 * written as a sort).  counts[e] = number of slots j = t*topk+k with
 * idx[j] = e; offsets = exclusive prefix sum (E+1 entries); perm lists the slot
 * ids ordered by (expert, t, k); inv[j] is the position of slot j in perm.
 * Reading: ties between slots of one expert keep slot order. */
int orc_route(const int32_t* topk_idx, int T, int topk, int num_experts,
              int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv)
{
    int n = T * topk;
    for (int e = 0; e < num_experts; e++) counts[e] = 0;
    for (int j = 0; j < n; j++) {
        int e = topk_idx[j];
        if (e < 0 || e >= num_experts) return -2;
        counts[e]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < num_experts; e++) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (num_experts > 0 ? num_experts : 1));
    for (int e = 0; e < num_experts; e++) cursor[e] = offsets[e];
    for (int j = 0; j < n; j++) {
        int pos = cursor[topk_idx[j]]++;
        perm[pos] = j;
        inv[j] = pos;
    }
    free(cursor);
    return 0;
}

/* RMSNorm with unit weight, rounded to bf16 as the MoE input:
 * out_i = bf16(x_i / sqrt(mean(x^2) + eps)). */
void orc_rmsnorm_bf16(const double* x, int n, double eps, uint16_t* out)
{
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += x[i] * x[i];
    double d = sqrt(ss / n + eps);
    for (int i = 0; i < n; i++) out[i] = orc_bf16_rne(x[i] / d);
}

/* L-layer decode step: x_{l+1} = x_l + moe_l(rmsnorm(x_l)), residual in fp64
 * ([A100] §然后又发现每 token 启动 2000 次内核 lists RMSNorm among the per-layer
 * steps of the decode loop).  topk_idx / topk_w are [L][T][topk]. */
int orc_moe_stack(const orc_layer* layers, int L, double* x, int T, int topk,
                  const int32_t* topk_idx, const float* topk_w, int act_mode,
                  double eps, int nthreads)
{
    if (L <= 0 || T <= 0) return (L < 0 || T < 0) ? -1 : 0;
    int H = layers[0].hidden;
    uint16_t* u = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)T * H);
    double* y = (double*)malloc(sizeof(double) * (size_t)T * H);
    int err = 0;
    for (int l = 0; l < L && !err; l++) {
        for (int t = 0; t < T; t++) orc_rmsnorm_bf16(x + (size_t)t * H, H, eps, u + (size_t)t * H);
        err = orc_moe_ffn(&layers[l], u, T, topk, topk_idx + (size_t)l * T * topk,
                          topk_w + (size_t)l * T * topk, act_mode, y, nthreads);
        if (!err)
            for (size_t i = 0; i < (size_t)T * H; i++) x[i] += y[i];
    }
    free(u);
    free(y);
    return err;
}

/* ---------------------------------------------------------------- router */

/* logits[t][e] = sum over h of W[e][h] * x[t][h], every product and sum in
 * fp64 (a bf16 x bf16 product is exact in fp64). */
void orc_router_logits(const uint16_t* x_bf16, const uint16_t* w_bf16, int T, int H, int E, double* logits)
{
    for (int t = 0; t < T; t++)
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int h = 0; h < H; h++)
                acc += orc_bf16_value(w_bf16[(size_t)e * H + h]) * orc_bf16_value(x_bf16[(size_t)t * H + h]);
            logits[(size_t)t * E + e] = acc;
        }
}

/* a ranks before b: larger logit first, NaN after every number, ties (and
 * two NaNs) to the lower expert id */
static int ranks_before(double va, int a, double vb, int b)
{
    const int na = isnan(va), nb = isnan(vb);
    if (na != nb) return nb;
    if (!na && va != vb) return va > vb;
    return a < b;
}

/* Selection by k passes of "best remaining expert", then the softmax of the
 * selected logits: w_i = exp(l_i - l_max) / sum_j exp(l_j - l_max). */
int orc_topk_softmax(const double* logits, int T, int E, int k, int32_t* idx, double* w)
{
    if (k < 1 || k > E) return -1;
    char* taken = (char*)malloc((size_t)E);
    if (!taken) return -1;
    for (int t = 0; t < T; t++) {
        const double* l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int i = 0; i < k; i++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || ranks_before(l[e], e, l[best], best))) best = e;
            taken[best] = 1;
            idx[(size_t)t * k + i] = best;
        }
        const double lmax = l[idx[(size_t)t * k]];
        double sum = 0.0;
        for (int i = 0; i < k; i++) sum += exp(l[idx[(size_t)t * k + i]] - lmax);
        for (int i = 0; i < k; i++) w[(size_t)t * k + i] = exp(l[idx[(size_t)t * k + i]] - lmax) / sum;
    }
    free(taken);
    return 0;
}
