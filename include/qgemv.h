/*
 * qgemv.h -- C ABI of the GB300 (sm_103a) weight-only quantized GEMV library.
 *
 * The operations are the decode-time primitives of colibri's GPU backends:
 *   qgemv          one quantized GEMV                 ("colibri Vulkan 计算后端完全指南",
 *                                                      xdnf.cn, section "API 契约":
 *                                                      coli_vk_matmul)
 *   qgate_up       silu(gate x) * (up x), x read once (same section: coli_vk_gate_up)
 *   qexpert_group  the fused gate/up -> down MLP of a batch of routed experts,
 *                  summed with router weights in routing order
 *                                                     (same section:
 *                                                      coli_vk_expert_group; colibri
 *                                                      docs/vulkan.md, the expert tier:
 *                                                      each row adds its experts'
 *                                                      outputs in rank order)
 *   qdequant       the dequantized weights as f32, for checking the decoders
 *   qgemm          the same product as qgemv for many activation rows, on the
 *                  tensor cores (prefill)   (colibri docs/vulkan.md, the
 *                                            tiled-GEMM / cooperative-matrix
 *                                            paragraph)
 *   qroute         the router's top-k and weights on the device, and
 *   qexpert_group_routed  the router chained ahead of the expert group
 *                                           (docs/vulkan.md, the per-engine
 *                                            host-step tables)
 * The formats are those of the same guide's section "着色器层面的实现细节":
 * int8, int4 decoded nibble - 8 with one f32 scale per group, int3-g64 in two
 * bit planes with one f32 scale per 64 inputs, and MXFP4 (e2m1 nibbles, bit 3
 * the sign) whose scale the host has expanded to f32 per 32 inputs.
 *
 * Conventions for every call:
 *  - All array pointers are DEVICE pointers, owned by the caller.  The library
 *    allocates no device memory and keeps no state between calls; scratch
 *    that a call needs (qexpert_group, qgemm) is a caller-provided workspace.
 *  - Calls are asynchronous on the given CUDA stream (`stream` is a
 *    cudaStream_t; NULL is the legacy default stream).  They return once the
 *    work is enqueued; the caller synchronizes before reading results.
 *  - Kernels are launched with programmatic dependent launch: when the kernel
 *    before a call in the stream allows it (this library's kernels do), the
 *    call starts reading its packed weights and scales before that kernel has
 *    finished; activations, ids, router weights and the workspace are read,
 *    and outputs written, only after it completed.  So weights and scales
 *    must not be written by a kernel that allows early starts of the next.
 *  - Every call returns a status: QSTATUS_OK (0) or a negative code.  On a
 *    negative return nothing was enqueued, except QSTATUS_LAUNCH (a CUDA error
 *    at launch; qlast_cuda_error() has its text).  There is no CPU fallback.
 *  - Matrices are row-major, O rows of I inputs.  Element (o, i) takes the scale
 *    scales[o * (I / gs) + i / gs] (groups run along a row).  Packed layouts:
 *      QFMT_INT8_ROW   int8 codes [O][I], value = code; one scale per row
 *                      (gs must be 0 or I).
 *      QFMT_INT4_G     [O][I/2] bytes, the low nibble holds the even input i,
 *                      value = nibble - 8; gs a power of two in [32, 1024].
 *      QFMT_INT3_G64   plane A [O][I/4] (the low two bits of four codes per
 *                      byte, least significant first) followed in the same
 *                      buffer by plane B [O][I/8] (the high bit of eight codes
 *                      per byte); value = code - 4; gs must be 0 or 64.
 *      QFMT_MXFP4_G32  [O][I/2] bytes of e2m1 nibbles, the low nibble holds the
 *                      even input; gs must be 0 or 32.
 *    Variants that share those decoders (colibri's other storage ids):
 *      QFMT_INT4_ROW   the int4 layout with one scale per row (gs 0 or I).
 *      QFMT_INT8_G     the int8 layout with one scale per group; gs a power of
 *                      two in [16, 512].
 *      QFMT_MXFP4_E8M0 the MXFP4 layout with the checkpoint's scale bytes as
 *                      stored: `scales` points to uint8 ue8m0 bytes [O][I/32]
 *                      (value 2^(e - 127); e = 255 is NaN), read in place of
 *                      the host-expanded f32; gs must be 0 or 32.
 *  - Alignment: packed weights and activation/hidden vectors (x, h) 16-byte
 *    aligned; workspaces 256-byte aligned; scales and outputs 4-byte aligned
 *    (ue8m0 scale bytes too); else QSTATUS_MISALIGNED.
 *  - Sizes: I % 16 == 0 (int8), I % 32 == 0 (int4 per row), I % 128 == 0
 *    (MXFP4 with ue8m0 bytes), I % gs == 0 (grouped formats), O, I, s >= 1.
 *    The activation rows of one launch share shared memory with the weight
 *    copy rings, so a row of I f32 must fit what the rings leave: I up to
 *    about 37,000 (int8, int4, MXFP4; qgate_up and qexpert_group too) or
 *    43,000 (int3); longer rows return QSTATUS_BAD_DIM.
 */
#ifndef QGEMV_GB300_H
#define QGEMV_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Weight formats (colibri's storage ids). */
enum {
    QFMT_INT8_ROW = 1,
    QFMT_INT4_ROW = 2,
    QFMT_INT4_G = 4,
    QFMT_INT3_G64 = 5,
    QFMT_MXFP4_G32 = 7,
    QFMT_MXFP4_E8M0 = 8,
    QFMT_INT8_G = 13
};

/* Status codes. */
enum {
    QSTATUS_OK = 0,
    QSTATUS_BAD_FMT = -1,        /* unknown format id, or gs not allowed for it */
    QSTATUS_BAD_DIM = -2,        /* a size out of range or not a multiple it must be */
    QSTATUS_MISALIGNED = -3,     /* a pointer without the alignment stated above */
    QSTATUS_NULL = -4,           /* a required pointer is NULL */
    QSTATUS_WORKSPACE = -5,      /* workspace smaller than the call's *_workspace() size */
    QSTATUS_LAUNCH = -6,         /* CUDA reported an error at launch */
    QSTATUS_DEVICE_TIMEOUT = -7, /* a bounded device-side wait ran out */
    QSTATUS_BAD_EXPERT_ID = -8,  /* an expert id outside [0, E) (reported on the device) */
    QSTATUS_BAD_ACT = -9,        /* unknown activation, or a limit that is negative or NaN */
    QSTATUS_BAD_ROUTE = -10      /* unknown router kind, or a NaN router scale */
};

/*
 * Activations of the gate/up product (h = act(g, u), g = gate x, u = up x):
 *   QACT_SWIGLU          silu(g) * u, silu(z) = z / (1 + e^-z)
 *   QACT_SWIGLU_CLAMPED  silu(min(g, L)) * min(max(u, -L), L) for a limit
 *                        L >= 0 -- the swiglu_limit of the models in colibri
 *                        docs/vulkan.md (expert-tier paragraph on GLM-5.3
 *                        Flash); L = 0 gives zeros, L = +inf is SwiGLU.
 */
#define QACT_SWIGLU 0
#define QACT_SWIGLU_CLAMPED 1

/*
 * y[t][o] = sum_i value(W[o][i]) * scales[o][i/gs] * x[t][i],  t < s, o < O.
 *   w       packed weights (layout above)
 *   scales  f32 [O][I/gs] (QFMT_MXFP4_E8M0: uint8 [O][I/32])
 *   x       f32 [s][I]
 *   y       f32 [s][O], written
 * Weights are streamed once per group of up to 8 activation rows; larger s is
 * processed in groups of 8.
 */
int qgemv(int fmt, int gs, const void* w, const float* scales,
          const float* x, int O, int I, int s, float* y, void* stream);

/*
 * h[t][f] = silu(g) * u with g = gate[f] . x[t], u = up[f] . x[t], and
 * silu(z) = z / (1 + e^-z); gate and up are F x D matrices of one format.
 *   x  f32 [s][D];  h  f32 [s][F], written.
 */
int qgate_up(int fmt, int gs, const void* wg, const float* sg,
             const void* wu, const float* su,
             const float* x, int F, int D, int s, float* h, void* stream);

/* qgate_up with the activation act (QACT_*) and its limit (read only for
 * QACT_SWIGLU_CLAMPED).  QSTATUS_BAD_ACT for an unknown act or a negative or
 * NaN limit of the clamped one. */
int qgate_up_act(int fmt, int gs, const void* wg, const float* sg,
                 const void* wu, const float* su,
                 const float* x, int F, int D, int s, int act, float limit, float* h, void* stream);

/* Bytes of workspace qexpert_group needs for these sizes.  The workspace
 * must hold zeros before its first use (cudaMemset it once after allocating
 * it); every call leaves the words that must be zero that way -- its first
 * words are the one-launch expert group's counters (per-batch readiness and
 * its closing barrier). */
size_t qexpert_group_workspace(int E, int D, int F, int s, int k);

/*
 * The routed-expert MLP of s tokens, each routed to k experts:
 *   out[t] = sum_{r=0}^{k-1} w[t][r] * down_e (silu(gate_e x_t) * (up_e x_t)),
 *   e = ids[t][r], summed in rank order r for every t.
 *   gate, up  packed [E][F][D] (expert e's F x D matrix at e * its size),
 *             scales f32 [E][F][D/gs]
 *   down      packed [E][D][F], scales f32 [E][D][F/gs]   (row formats: one per row;
 *             QFMT_MXFP4_E8M0: the scales are ue8m0 bytes of the same counts)
 *   x         f32 [s][D];  ids int32 [s][k];  wts f32 [s][k]
 *   out       f32 [s][D], written
 *   workspace device scratch of ws_bytes >= qexpert_group_workspace(E, D, F, s, k)
 *             bytes, 256-byte aligned, zeroed before its first use (see
 *             qexpert_group_workspace); calls leave it zeroed.
 *   status_dev optional device int32: set to QSTATUS_OK, or to
 *             QSTATUS_BAD_EXPERT_ID when an id is outside [0, E) -- then out is
 *             all zeros -- or to QSTATUS_DEVICE_TIMEOUT when a bounded wait of
 *             the launch ran out.  The host-side return cannot see device-side
 *             checks.
 * Up to 256 (token, rank) pairs the call is one persistent launch (gate/up,
 * act, down and the rank-order sum; its CTAs, one per SM, wait on one another
 * -- the down rows of an expert batch for that batch's gate/up rows, the sums
 * for every down row -- so the launch needs every SM of the device at once;
 * qexpert_group_launches tells which path a call takes); past that,
 * and under QKERNEL_RING or QKERNEL_TILE, four launches that stream each
 * expert's weights once for all the pairs routed to it.  Repeated ids in a row
 * are allowed and summed.  s * k <= 4096.
 */
int qexpert_group(int fmt, int gs,
                  const void* gate, const float* gate_s,
                  const void* up, const float* up_s,
                  const void* down, const float* down_s,
                  int E, int D, int F,
                  const float* x, int s, int k,
                  const int32_t* ids, const float* wts,
                  float* out, void* workspace, size_t ws_bytes,
                  int32_t* status_dev, void* stream);

/*
 * How many kernel launches qexpert_group (routed = 0) or qexpert_group_routed
 * (routed != 0) makes for these sizes on the current device under the
 * current qkernel_policy: 1 when the call runs as the one fused launch, 4
 * for the four-launch path (pair sort, gate/up, down, rank-order sum), plus
 * 1 for the router kernel of a routed call with E > 256.  Nothing is
 * enqueued.  Negative QSTATUS_* for sizes or a format the call rejects, or
 * when no device is usable.
 */
int qexpert_group_launches(int fmt, int gs, int E, int D, int F, int s, int k, int routed);

/* qexpert_group with the activation act (QACT_*) and its limit in place of
 * silu(g) * u; QSTATUS_BAD_ACT as for qgate_up_act. */
int qexpert_group_act(int fmt, int gs,
                      const void* gate, const float* gate_s,
                      const void* up, const float* up_s,
                      const void* down, const float* down_s,
                      int E, int D, int F,
                      const float* x, int s, int k,
                      const int32_t* ids, const float* wts, int act, float limit,
                      float* out, void* workspace, size_t ws_bytes,
                      int32_t* status_dev, void* stream);

/*
 * qexpert_group for callers that cannot allocate device memory -- for
 * example a plugin inside a host application that owns all of the GPU's
 * memory through its own allocator and gives plugins no way to allocate, or a
 * decode loop that must never allocate.  The pages have no counterpart: their
 * backends allocate their own device buffers.
 *
 * Same arguments, result and status word as qexpert_group, without the
 * workspace: the scratch is a fixed array of QEXPERT_NOALLOC_SCRATCH_BYTES
 * compiled into the library, which every GPU that loads the library holds
 * until the process exits.  Sizes whose qexpert_group_workspace() exceeds it
 * are rejected with QSTATUS_WORKSPACE before anything is enqueued.  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress); make that first call before any
 * stream capture.  Every call on a device shares the one array: it starts
 * zeroed when the library loads, and each call leaves the words that must be
 * zero (the grid-barrier counters) zeroed and writes every other scratch word
 * before it reads it.  Calls that overlap on the GPU (other streams, other
 * host threads) race on the array: serialize them.
 */
#define QEXPERT_NOALLOC_SCRATCH_BYTES (4u << 20)

int qexpert_group_noalloc(int fmt, int gs,
                          const void* gate, const float* gate_s,
                          const void* up, const float* up_s,
                          const void* down, const float* down_s,
                          int E, int D, int F,
                          const float* x, int s, int k,
                          const int32_t* ids, const float* wts,
                          float* out, int32_t* status_dev, void* stream);

/*
 * out[o][i] = value(W[o][i]) * scales[o][i/gs] as f32 (one IEEE f32
 * multiplication of the exact code value by the scale).  For checking the
 * decoders bit for bit; out f32 [O][I].
 */
int qdequant(int fmt, int gs, const void* w, const float* scales,
             int O, int I, float* out, void* stream);

/*
 * The prefill GEMM: y[t][o] = sum_i value(W[o][i]) * scales[o][i/gs] * x[t][i]
 * for many activation rows t < s, on the tensor cores -- the tiled GEMM that
 * colibri's docs/vulkan.md (the tiled-GEMM and cooperative-matrix paragraph)
 * takes instead of the per-row GEMV from two rows on.  Weight codes are
 * decoded exactly to f16; every activation row is scaled by a power of two
 * and split into two f16 parts (22 significand bits; written to the
 * workspace), the MMA runs on both, and each group of gs inputs (at most 128
 * at a time) sums into a fresh f32 partial that is added to the row's sum
 * times the group scale.  The result meets the f32 GEMV's error bound, not
 * its bits.  Range: the power of two is limited to 2^-126 .. 2^126, so every
 * finite activation row fits, and the split's error stays within 2^-22 of
 * each element plus 2^-151 absolute (below f32's resolution) for every row.
 *   w, scales, x, y as for qgemv;  workspace of ws_bytes >= qgemm_workspace(I,
 *   s) device bytes, 256-byte aligned, contents on entry irrelevant.
 * Every format, with I % 64 == 0 and groups of at least 32 inputs
 * (QFMT_INT8_G with gs 16: QSTATUS_BAD_FMT).  Intended for s >= 16; any s >= 1
 * works.  I <= 2^20, s <= 65536; O, I or s below 1 or past these limits, or I
 * not a multiple of 64: QSTATUS_BAD_DIM.  A workspace smaller than
 * qgemm_workspace(I, s): QSTATUS_WORKSPACE; one not 256-byte aligned:
 * QSTATUS_MISALIGNED.  qgemm_workspace returns 0 for I or s below 1.
 */
size_t qgemm_workspace(int I, int s);
int qgemm(int fmt, int gs, const void* w, const float* scales,
          const float* x, int O, int I, int s, float* y,
          void* workspace, size_t ws_bytes, void* stream);

/*
 * The router on the device: for each token t < s, the k of E experts with the
 * largest keys and their weights, from the router logits -- the step
 * colibri's engines run on the host (docs/vulkan.md, the per-engine host-step
 * tables: a softmax followed by a top-k for the softmax routers; sigmoid
 * scores, a top-k picked with a correction bias and renormalized for the
 * sigmoid routers).
 *   QROUTE_SOFTMAX       key = logit (the same order as the softmax
 *                        probability); weight = the probability
 *                        exp(l_e) / sum_j exp(l_j) over all E experts, or with
 *                        renorm != 0 over the k chosen.
 *   QROUTE_SIGMOID_BIAS  key = sigmoid(logit) + bias[e]; weight = sigmoid(logit),
 *                        divided by the sum over the k chosen if renorm != 0.
 * Every weight is multiplied by `scale` (a routed scaling factor; 1 for none).
 * Ranks run in decreasing key; equal keys rank the lower expert index first; a
 * NaN key ranks below every number.
 *   logits f32 [s][E];  bias f32 [E] (QROUTE_SIGMOID_BIAS only, else may be
 *   NULL);  ids int32 [s][k] and wts f32 [s][k], written in rank order.
 * s >= 1, 1 <= k <= 32, k <= E <= 1024, else QSTATUS_BAD_DIM.
 * QSTATUS_BAD_ROUTE for an unknown kind or a NaN scale; QSTATUS_NULL for a
 * missing logits, ids or wts pointer, or a missing bias with
 * QROUTE_SIGMOID_BIAS; QSTATUS_MISALIGNED for a pointer not 4-byte aligned.
 */
#define QROUTE_SOFTMAX 0
#define QROUTE_SIGMOID_BIAS 1
int qroute(int kind, const float* logits, const float* bias, int s, int E, int k, int renorm, float scale,
           int32_t* ids, float* wts, void* stream);

/*
 * qroute followed by qexpert_group_act in one call: the routing is written to
 * ids_out / wts_out (device int32 / f32 [s][k], caller-owned) and the expert
 * group reads it from there; the expert launches wait for the router on the
 * device (no host round trip).  Arguments and statuses as for the two calls.
 */
int qexpert_group_routed(int fmt, int gs,
                         const void* gate, const float* gate_s,
                         const void* up, const float* up_s,
                         const void* down, const float* down_s,
                         int E, int D, int F,
                         const float* x, int s, int k,
                         int route_kind, const float* logits, const float* bias, int renorm, float route_scale,
                         int act, float limit,
                         float* out, int32_t* ids_out, float* wts_out,
                         void* workspace, size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * Test hook (no counterpart in the pages, whose backends inject their faults
 * through environment switches): arms one fault for the next one-launch
 * expert group of this process.  QDEBUG_WITHHOLD_SIGNAL makes one CTA of that
 * launch skip counting its finished gate/up rows, so the waits of the CTAs
 * that need them run out after wait_ns nanoseconds (every wait of that launch
 * is bounded by wait_ns): the launch records QSTATUS_DEVICE_TIMEOUT (in
 * qdevice_error and in the call's status word), its results are undefined, it
 * returns, and it leaves the workspace ready for the next call.  Nothing
 * faults or waits without bound.  QDEBUG_NONE disarms.  Returns QSTATUS_OK,
 * or QSTATUS_BAD_DIM for an unknown kind or wait_ns below 1.
 */
#define QDEBUG_NONE 0
#define QDEBUG_WITHHOLD_SIGNAL 1
int qdebug_inject(int kind, long long wait_ns);

/* A static description of a status code. */
const char* qstatus_string(int status);

/* Text of the CUDA error behind the calling thread's last QSTATUS_LAUNCH. */
const char* qlast_cuda_error(void);

/*
 * QSTATUS_DEVICE_TIMEOUT when a bounded device-side wait in one of this
 * library's kernels ran out on the current device since the last clear (the
 * results of that launch are undefined; qexpert_group also reports it in its
 * status word), else QSTATUS_OK.  Reads a device word, so it synchronizes with
 * the device; clear != 0 resets the word.
 */
int qdevice_error(int clear);

/*
 * Kernel choice for the streaming launches of this process (a tuning and
 * testing knob; the pages have no counterpart).  QKERNEL_AUTO picks
 * per shape; QKERNEL_RING forces the per-lane copy kernel; QKERNEL_TILE the
 * tensor-copy tile kernel wherever its plan fits (else the ring kernel);
 * QKERNEL_ROW the row-team kernel wherever its plan fits (one activation
 * row, rows a whole number of 32-chunk warp steps; else the automatic
 * choice).  The ring and tile kernels give the same bits; the
 * row-team kernel sums each row in another (fixed) order.  For the expert
 * group, QKERNEL_AUTO and QKERNEL_ROW take the one-launch path where it
 * applies, QKERNEL_RING and QKERNEL_TILE the four launches (the same bits
 * as the one launch under QKERNEL_TILE).  Returns the
 * previous policy, or QSTATUS_BAD_FMT for an unknown one (the policy is then
 * unchanged).  Not synchronized with launches in flight on other threads.
 */
#define QKERNEL_AUTO 0
#define QKERNEL_RING 1
#define QKERNEL_TILE 2
#define QKERNEL_ROW 3
int qkernel_policy(int policy);

#ifdef __cplusplus
}
#endif

#endif /* QGEMV_GB300_H */
