/*
 * oracle.c -- plain, slow, f64 CPU oracle for the weight-only group-quantized
 * GEMV, the fused gate/up, and the routed-expert MLP.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package entry's smoke check and
 * the bench's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library: every definition below is
 * written out here from the pages' statement of the method.
 *
 * Sources (page title, section):
 *  [GUIDE]  "colibri Vulkan 计算后端完全指南" (xdnf.cn): section
 *           "着色器层面的实现细节" (shader-level details: int8, int4 two per
 *           byte decoded nibble-8, int3-g64 one group per 64 inputs in two
 *           planes, one f32 scale per group, MXFP4 e2m1 nibbles with bit 3 the
 *           sign, its scale turned into one f32 per 32 inputs on the host);
 *           section "API 契约" (coli_vk_matmul: one quantized GEMV;
 *           coli_vk_gate_up: silu(gate(x))*up(x); coli_vk_expert_group: the
 *           fused MLP of a batch of experts); section "正确性如何在两个实现之间
 *           建立信任" item 3 (int4 is offset binary, nibble - 8).
 *  [VULKAN] colibri "docs/vulkan.md": the expert tier's paragraph on the sum
 *           (each row adds its experts' outputs in routing (rank) order),
 *           and the cooperative-matrix paragraph (int8, int4, int3-g64 and
 *           MXFP4 weights decode exactly to fp16, i.e. to small integers and
 *           e2m1 values).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - int4 and MXFP4: the low nibble of byte b holds element 2b, the high
 *    nibble element 2b+1.
 *  - int3-g64: plane A holds the low two bits of four codes per byte, plane B
 *    the high bit of eight codes per byte, least significant bits first; the
 *    whole plane A [O][I/4] comes first in the buffer, then plane B [O][I/8];
 *    value = code - 4.
 *  - e2m1 is the OCP microscaling FP4 element: sign bit 3, two exponent bits
 *    (bias 1), one mantissa bit; exponent 0 is subnormal (0 or 0.5).
 *  - Groups run along i inside a row: element (o, i) takes scale
 *    [o][i / gs], scales stored row-major [O][I/gs].  int8 per row: gs = I.
 *  - silu(z) = z / (1 + exp(-z)); the activation is silu(g) * u, or with a
 *    limit L (clamped SwiGLU) silu(min(g, L)) * min(max(u, -L), L).
 *  - out[t] = sum over rank r of w[t][r] * down_e (act(gate_e x_t, up_e x_t))
 *    with e = ids[t][r], summed in rank order.
 *
 * Everything is evaluated in double from the f32 inputs, in index order, with
 * no intermediate rounding to f32.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define ORACLE_INT8_ROW 1
#define ORACLE_INT4_ROW 2
#define ORACLE_INT4_G 4
#define ORACLE_INT3_G64 5
#define ORACLE_MXFP4_G32 7
#define ORACLE_MXFP4_E8M0 8
#define ORACLE_INT8_G 13

/* Bytes of one packed O x I matrix in format fmt ([GUIDE] shader details). */
long oracle_packed_bytes(int fmt, long O, long I)
{
    switch (fmt) {
    case ORACLE_INT8_ROW:
    case ORACLE_INT8_G: return O * I;              /* one byte per code */
    case ORACLE_INT4_ROW:
    case ORACLE_INT4_G:
    case ORACLE_MXFP4_G32:
    case ORACLE_MXFP4_E8M0: return O * I / 2;      /* two codes per byte */
    case ORACLE_INT3_G64: return O * I / 4 + O * I / 8; /* plane A + plane B */
    default: return -1;
    }
}

/* Step a1 (unpack): the raw code of element (o, i) of a packed O x I matrix. */
int oracle_code(int fmt, const uint8_t *w, long O, long I, long o, long i)
{
    switch (fmt) {
    case ORACLE_INT8_ROW:
    case ORACLE_INT8_G:
        /* one signed byte per code */
        return (int)(int8_t)w[o * I + i];
    case ORACLE_INT4_ROW:
    case ORACLE_INT4_G:
    case ORACLE_MXFP4_G32:
    case ORACLE_MXFP4_E8M0: {
        /* two codes per byte: even i in the low nibble, odd i in the high one */
        uint8_t b = w[o * (I / 2) + i / 2];
        return (i % 2 == 0) ? (b & 0x0F) : ((b >> 4) & 0x0F);
    }
    case ORACLE_INT3_G64: {
        /* dual plane: low two bits from plane A, high bit from plane B */
        const uint8_t *A = w;
        const uint8_t *B = w + O * (I / 4);
        int lo = (A[o * (I / 4) + i / 4] >> (2 * (i % 4))) & 3;
        int hi = (B[o * (I / 8) + i / 8] >> (i % 8)) & 1;
        return lo | (hi << 2);
    }
    default:
        return 0;
    }
}

/* e2m1 (FP4): bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa. */
double oracle_e2m1(int c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* Step a2, first half: the value a code stands for, before its scale. */
double oracle_code_value(int fmt, int code)
{
    switch (fmt) {
    case ORACLE_INT8_ROW:
    case ORACLE_INT8_G: return (double)code;            /* int8 as is */
    case ORACLE_INT4_ROW:
    case ORACLE_INT4_G: return (double)(code - 8);      /* offset binary, nibble - 8 */
    case ORACLE_INT3_G64: return (double)(code - 4);    /* 3-bit code - 4 */
    case ORACLE_MXFP4_G32:
    case ORACLE_MXFP4_E8M0: return oracle_e2m1(code);   /* e2m1 element */
    default: return 0.0;
    }
}

/* Group size of a format: int8 and int4 per row have one group per row;
 * int3-g64 groups 64 inputs and MXFP4 32 ([GUIDE] shader details); grouped
 * int4 and int8 take gs. */
static long group_of(int fmt, long I, long gs)
{
    switch (fmt) {
    case ORACLE_INT8_ROW:
    case ORACLE_INT4_ROW: return I;
    case ORACLE_INT3_G64: return 64;
    case ORACLE_MXFP4_G32:
    case ORACLE_MXFP4_E8M0: return 32;
    default: return gs;
    }
}

/* ue8m0 scale byte (OCP microscaling): 2^(e - 127); e = 255 is NaN. */
double oracle_e8m0(int e)
{
    return e == 255 ? NAN : ldexp(1.0, e - 127);
}

/* The scale of element (o, i): one per group of gs inputs along the row,
 * stored row-major [O][I/gs]: f32, or for MXFP4_E8M0 one ue8m0 byte
 * ([VULKAN] model table: the checkpoints store MXFP4 with ue8m0 scales). */
static double scale_of(int fmt, const float *scales, long I, long gs, long o, long i)
{
    gs = group_of(fmt, I, gs);
    if (fmt == ORACLE_MXFP4_E8M0)
        return oracle_e8m0(((const uint8_t *)scales)[o * (I / gs) + i / gs]);
    return (double)scales[o * (I / gs) + i / gs];
}

/* Step a2: dequantized weight (o, i) = value(code) * scale, exact in double. */
double oracle_weight(int fmt, long gs, const uint8_t *w, const float *scales,
                     long O, long I, long o, long i)
{
    return oracle_code_value(fmt, oracle_code(fmt, w, O, I, o, i)) * scale_of(fmt, scales, I, gs, o, i);
}

/* Step a2 as f32: the exact double product rounded once to f32 (IEEE f32
 * multiplication of the f32 value by the f32 scale gives the same bits). */
void oracle_dequant_f32(int fmt, long gs, const uint8_t *w, const float *scales,
                        long O, long I, float *out)
{
    for (long o = 0; o < O; o++)
        for (long i = 0; i < I; i++)
            out[o * I + i] = (float)oracle_weight(fmt, gs, w, scales, O, I, o, i);
}

/* Step a3 for one output row: y = sum_i W(o, i) * x[i], double, index order. */
static double row_dot(int fmt, long gs, const uint8_t *w, const float *scales,
                      long O, long I, long o, const float *x)
{
    double acc = 0.0;
    for (long i = 0; i < I; i++)
        acc += oracle_weight(fmt, gs, w, scales, O, I, o, i) * (double)x[i];
    return acc;
}

/* Step a3 ([GUIDE] API contract, coli_vk_matmul): y[t][o] = sum_i W[o][i] x[t][i]
 * for t < s.  x is f32 [s][I]; y is double [s][O]. */
void oracle_qgemv(int fmt, long gs, const uint8_t *w, const float *scales,
                  const float *x, long O, long I, long s, double *y)
{
#pragma omp parallel for schedule(static)
    for (long o = 0; o < O; o++)
        for (long t = 0; t < s; t++)
            y[t * O + o] = row_dot(fmt, gs, w, scales, O, I, o, x + t * I);
}

/* Step a3 on a sample of rows: y[t][j] for row rows[j]. */
void oracle_qgemv_rows(int fmt, long gs, const uint8_t *w, const float *scales,
                       const float *x, long O, long I, long s,
                       const long *rows, long nrows, double *y)
{
#pragma omp parallel for schedule(static)
    for (long j = 0; j < nrows; j++)
        for (long t = 0; t < s; t++)
            y[t * nrows + j] = row_dot(fmt, gs, w, scales, O, I, rows[j], x + t * I);
}

/* silu(z) = z / (1 + e^-z). */
double oracle_silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* The gate/up activation.  act 0: silu(g) * u (SwiGLU).  act 1: SwiGLU with
 * a limit L (the pages' swiglu_limit, [VULKAN] expert-tier paragraph on
 * GLM-5.3 Flash): the gate is capped at L and the up value clamped to
 * [-L, L] before the product, so that L = 0 zeroes the output (the page's
 * swiglu_clamped clamps at every limit, 0 included). */
double oracle_glu(int act, double limit, double g, double u)
{
    if (act == 1) {
        if (g > limit) g = limit;
        if (u > limit) u = limit;
        if (u < -limit) u = -limit;
    }
    return oracle_silu(g) * u;
}

/* Step a4 ([GUIDE] API contract, coli_vk_gate_up): h[t][f] = silu(g) * u with
 * g = gate[f] . x[t] and u = up[f] . x[t]; gate and up are F x D. */
void oracle_qgate_up_act(int fmt, long gs, const uint8_t *wg, const float *sg,
                         const uint8_t *wu, const float *su, const float *x,
                         long F, long D, long s, int act, double limit, double *h)
{
#pragma omp parallel for schedule(static)
    for (long f = 0; f < F; f++)
        for (long t = 0; t < s; t++) {
            double g = row_dot(fmt, gs, wg, sg, F, D, f, x + t * D);
            double u = row_dot(fmt, gs, wu, su, F, D, f, x + t * D);
            h[t * F + f] = oracle_glu(act, limit, g, u);
        }
}

void oracle_qgate_up(int fmt, long gs, const uint8_t *wg, const float *sg,
                     const uint8_t *wu, const float *su, const float *x,
                     long F, long D, long s, double *h)
{
    oracle_qgate_up_act(fmt, gs, wg, sg, wu, su, x, F, D, s, 0, 0.0, h);
}

/* Step a4 on a sample of rows f = rows[j]. */
void oracle_qgate_up_rows_act(int fmt, long gs, const uint8_t *wg, const float *sg,
                              const uint8_t *wu, const float *su, const float *x,
                              long F, long D, long s, const long *rows, long nrows, int act, double limit,
                              double *h)
{
#pragma omp parallel for schedule(static)
    for (long j = 0; j < nrows; j++)
        for (long t = 0; t < s; t++) {
            double g = row_dot(fmt, gs, wg, sg, F, D, rows[j], x + t * D);
            double u = row_dot(fmt, gs, wu, su, F, D, rows[j], x + t * D);
            h[t * nrows + j] = oracle_glu(act, limit, g, u);
        }
}

void oracle_qgate_up_rows(int fmt, long gs, const uint8_t *wg, const float *sg,
                          const uint8_t *wu, const float *su, const float *x,
                          long F, long D, long s, const long *rows, long nrows, double *h)
{
    oracle_qgate_up_rows_act(fmt, gs, wg, sg, wu, su, x, F, D, s, rows, nrows, 0, 0.0, h);
}

/* Steps a4 + a5 ([GUIDE] API contract, coli_vk_expert_group; [VULKAN] the sum
 * in routing order).  Experts are stored back to back: gate and up [E][F][D]
 * packed with scales [E][F][D/gs]; down [E][D][F] packed with scales
 * [E][D][F/gs].  For each token t and rank r (e = ids[t][r]):
 *     h = silu(gate_e x_t) * (up_e x_t)          (length F)
 *     out[t][d] += w[t][r] * (down_e[d] . h)      (rank order r = 0..k-1)
 * Only the output columns cols[0..ncols) are formed (all of them when
 * cols == NULL, then ncols must be D); out is double [s][ncols]. */
void oracle_expert_group_act_cols(int fmt, long gs,
                                  const uint8_t *gate, const float *gate_s,
                                  const uint8_t *up, const float *up_s,
                                  const uint8_t *down, const float *down_s,
                                  long E, long D, long F,
                                  const float *x, long s, long k,
                                  const int32_t *ids, const float *wts, int act, double limit,
                                  const long *cols, long ncols, double *out, double *h_scratch)
{
    long gu_bytes = oracle_packed_bytes(fmt, F, D);
    long gu_scales = F * (D / group_of(fmt, D, gs));
    long dn_bytes = oracle_packed_bytes(fmt, D, F);
    long dn_scales = D * (F / group_of(fmt, F, gs));
    (void)E;
    for (long t = 0; t < s; t++) {
        for (long j = 0; j < ncols; j++)
            out[t * ncols + j] = 0.0;
        for (long r = 0; r < k; r++) {
            long e = ids[t * k + r];
            const uint8_t *ge = gate + e * gu_bytes;
            const uint8_t *ue = up + e * gu_bytes;
            const uint8_t *de = down + e * dn_bytes;
            /* expert e's scales: e * (scales per matrix) elements of f32, or of one byte for ue8m0 */
            long ssz = fmt == ORACLE_MXFP4_E8M0 ? 1 : (long)sizeof(float);
            const float *gse = (const float *)((const uint8_t *)gate_s + e * gu_scales * ssz);
            const float *use = (const float *)((const uint8_t *)up_s + e * gu_scales * ssz);
            const float *dse = (const float *)((const uint8_t *)down_s + e * dn_scales * ssz);
            double wr = (double)wts[t * k + r];
#pragma omp parallel for schedule(static)
            for (long f = 0; f < F; f++) {
                double g = row_dot(fmt, gs, ge, gse, F, D, f, x + t * D);
                double u = row_dot(fmt, gs, ue, use, F, D, f, x + t * D);
                h_scratch[f] = oracle_glu(act, limit, g, u);
            }
#pragma omp parallel for schedule(static)
            for (long j = 0; j < ncols; j++) {
                long d = cols ? cols[j] : j;
                double z = 0.0;
                for (long f = 0; f < F; f++)
                    z += oracle_weight(fmt, gs, de, dse, D, F, d, f) * h_scratch[f];
                out[t * ncols + j] += wr * z;
            }
        }
    }
}

/* The same with SwiGLU (act 0). */
void oracle_expert_group_cols(int fmt, long gs,
                              const uint8_t *gate, const float *gate_s,
                              const uint8_t *up, const float *up_s,
                              const uint8_t *down, const float *down_s,
                              long E, long D, long F,
                              const float *x, long s, long k,
                              const int32_t *ids, const float *wts,
                              const long *cols, long ncols, double *out, double *h_scratch)
{
    oracle_expert_group_act_cols(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids, wts, 0,
                                 0.0, cols, ncols, out, h_scratch);
}

/* ------------------------------------------------------------------------
 * The router ([VULKAN] the per-engine host steps: a softmax followed by a
 * top-k for the softmax models; for the sigmoid-router models, sigmoid scores
 * whose top-k is picked with a correction bias and then renormalized).  Per token t, over its
 * E logits l[t][e]:
 *   kind 0 (softmax): score p_e = exp(l_e) / sum_j exp(l_j); the k largest
 *          p_e are chosen; weight = p_e, or with renorm p_e / sum over the
 *          chosen of p.
 *   kind 1 (sigmoid with correction bias): score s_e = 1 / (1 + exp(-l_e));
 *          the k largest s_e + bias_e are chosen; weight = s_e, or with
 *          renorm s_e / sum over the chosen of s.
 * Every weight is then multiplied by `scale` (the models' routed scaling
 * factor; 1 for none).  Readings where the pages are silent: ranks are in
 * decreasing selection key, equal keys rank the lower expert index first.
 * Selection for kind 0 compares the logits themselves (exp is increasing, so
 * that is the same choice as comparing p); kind 1 compares s_e + bias_e in
 * double.  Outputs ids[t][r], wts[t][r] for rank r < k.
 * ------------------------------------------------------------------------ */
double oracle_sigmoid(double z)
{
    return 1.0 / (1.0 + exp(-z));
}

void oracle_route(int kind, const float *logits, const float *bias, long s, long E, long k, int renorm,
                  double scale, int32_t *ids, double *wts, double *key_scratch, unsigned char *taken)
{
    for (long t = 0; t < s; t++) {
        const float *l = logits + t * E;
        for (long e = 0; e < E; e++) {
            key_scratch[e] = kind == 0 ? (double)l[e] : oracle_sigmoid((double)l[e]) + (double)bias[e];
            taken[e] = 0;
        }
        /* top k: repeatedly the largest remaining key, lowest index on ties */
        for (long r = 0; r < k; r++) {
            long best = -1;
            for (long e = 0; e < E; e++) {
                if (taken[e]) continue;
                if (best < 0 || key_scratch[e] > key_scratch[best]) best = e;
            }
            taken[best] = 1;
            ids[t * k + r] = (int32_t)best;
        }
        /* weights */
        double denom = 0.0;
        if (kind == 0) {
            double mx = -INFINITY;
            for (long e = 0; e < E; e++) mx = l[e] > mx ? l[e] : mx;
            if (renorm) {
                for (long r = 0; r < k; r++) denom += exp((double)l[ids[t * k + r]] - mx);
            } else {
                for (long e = 0; e < E; e++) denom += exp((double)l[e] - mx);
            }
            for (long r = 0; r < k; r++)
                wts[t * k + r] = scale * exp((double)l[ids[t * k + r]] - mx) / denom;
        } else {
            if (renorm)
                for (long r = 0; r < k; r++) denom += oracle_sigmoid((double)l[ids[t * k + r]]);
            for (long r = 0; r < k; r++) {
                const double sg = oracle_sigmoid((double)l[ids[t * k + r]]);
                wts[t * k + r] = scale * (renorm ? sg / denom : sg);
            }
        }
    }
}

/* Number of threads the OpenMP loops above use (1 when built without it). */
int oracle_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the number of threads the OpenMP loops use (n >= 1; ignored when built
 * without OpenMP).  Only the timing of the oracle depends on it: each output
 * row is computed by one thread in the same order whatever the count. */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
