// qg_abi.cu -- the C entry points: argument checks, launch set-up, and the
// format-independent kernels of the routed-expert group (grouping the
// (token, rank) pairs by expert, and the rank-order weighted sum).
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "qg_internal.h"
#include "qg_route.cuh"

namespace qg {

static thread_local const char* g_last_cuda_error = "no error";

static std::atomic<int> g_kernel_policy{QKERNEL_AUTO};
int kernel_policy() { return g_kernel_policy.load(std::memory_order_relaxed); }

// The armed test fault (qdebug_inject) and its wait bound, consumed by the
// next fused expert-group launch.
static std::atomic<int> g_inject{QDEBUG_NONE};
static std::atomic<long long> g_inject_ns{0};

static int launch_status(cudaError_t e)
{
    if (e == cudaSuccess) return QSTATUS_OK;
    g_last_cuda_error = cudaGetErrorString(e);
    return QSTATUS_LAUNCH;
}

// Number of SMs of the current device (read once per device).
static int sm_count(int* status)
{
    static int cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { *status = launch_status(e); return 0; }
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || n <= 0) { *status = launch_status(e == cudaSuccess ? cudaErrorInvalidDevice : e); return 0; }
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Resolves and checks the group size of an O x I matrix in format fmt.
static int check_fmt(int fmt, int gs, int I, int* gs_out)
{
    switch (fmt) {
    case QFMT_INT8_ROW:
        if (gs != 0 && gs != I) return QSTATUS_BAD_FMT;
        if (I % 16) return QSTATUS_BAD_DIM;
        *gs_out = I;
        return QSTATUS_OK;
    case QFMT_INT8_G:   // a warp step covers 512 codes: at most one group per step
        if (gs < 16 || gs > 512 || (gs & (gs - 1))) return QSTATUS_BAD_FMT;
        if (I % gs) return QSTATUS_BAD_DIM;
        *gs_out = gs;
        return QSTATUS_OK;
    case QFMT_INT4_ROW:
        if (gs != 0 && gs != I) return QSTATUS_BAD_FMT;
        if (I % 32) return QSTATUS_BAD_DIM;
        *gs_out = I;
        return QSTATUS_OK;
    case QFMT_INT4_G:
        if (gs < 32 || gs > 1024 || (gs & (gs - 1))) return QSTATUS_BAD_FMT;
        if (I % gs) return QSTATUS_BAD_DIM;
        *gs_out = gs;
        return QSTATUS_OK;
    case QFMT_INT3_G64:
        if (gs != 0 && gs != 64) return QSTATUS_BAD_FMT;
        if (I % 64) return QSTATUS_BAD_DIM;
        *gs_out = 64;
        return QSTATUS_OK;
    case QFMT_MXFP4_G32:
        if (gs != 0 && gs != 32) return QSTATUS_BAD_FMT;
        if (I % 32) return QSTATUS_BAD_DIM;
        *gs_out = 32;
        return QSTATUS_OK;
    case QFMT_MXFP4_E8M0:   // four lanes read their scale bytes as one aligned word
        if (gs != 0 && gs != 32) return QSTATUS_BAD_FMT;
        if (I % 128) return QSTATUS_BAD_DIM;
        *gs_out = 32;
        return QSTATUS_OK;
    default:
        return QSTATUS_BAD_FMT;
    }
}

constexpr int kMaxI = 51200;   // an upper bound; the shared-memory budget below decides
constexpr int kGemmMaxI = 1 << 20;   // qgemm: tensor-map and index ranges
constexpr int kGemmMaxS = 1 << 16;

// Shared memory left for activation rows once the copy rings of a launch of
// format fmt with nm matrices per row tile are placed.
// QSTATUS_BAD_ACT unless act is a QACT_* and, for the clamped one, the limit
// is a number >= 0 (+inf allowed).
static int check_act(int act, float limit)
{
    if (act == QACT_SWIGLU) return QSTATUS_OK;
    if (act == QACT_SWIGLU_CLAMPED) return (limit >= 0.0f) ? QSTATUS_OK : QSTATUS_BAD_ACT;   // NaN fails too
    return QSTATUS_BAD_ACT;
}

static size_t ring_bytes(int fmt, int nm)
{
    switch (fmt) {
    case QFMT_INT8_ROW: return ring_bytes_int8(nm);
    case QFMT_INT8_G: return ring_bytes_int8g(nm);
    case QFMT_INT4_ROW: return ring_bytes_int4r(nm);
    case QFMT_INT4_G: return ring_bytes_int4(nm);
    case QFMT_INT3_G64: return ring_bytes_int3(nm);
    case QFMT_MXFP4_E8M0: return ring_bytes_mxfp4e(nm);
    default: return ring_bytes_mxfp4(nm);
    }
}

// Activation rows of length I one launch can stage (0: I is too long).
static int rows_per_launch(int fmt, int nm, int I)
{
    const long long budget = (long long)kSmemMax - (long long)ring_bytes(fmt, nm) - 16;
    long long s = budget > 0 ? budget / ((long long)I * (long long)sizeof(float)) : 0;
    return (int)(s < kSmax ? s : kSmax);
}

#define QG_FMT_SWITCH(fmt, CALL)                                 \
    switch (fmt) {                                               \
    case QFMT_INT8_ROW: e = CALL(int8); break;                   \
    case QFMT_INT8_G: e = CALL(int8g); break;                    \
    case QFMT_INT4_ROW: e = CALL(int4r); break;                  \
    case QFMT_INT4_G: e = CALL(int4); break;                     \
    case QFMT_INT3_G64: e = CALL(int3); break;                   \
    case QFMT_MXFP4_E8M0: e = CALL(mxfp4e); break;               \
    default: e = CALL(mxfp4); break;                             \
    }

// ---------------------------------------------------------------------------
// Expert group: (token, rank) pairs sorted by (expert, pair index), split into
// batches of at most smax pairs of one expert.
// ---------------------------------------------------------------------------
// It also splits the row tiles of each streaming phase over the G CTAs by
// cost: a row tile of a batch of n pairs costs n (one pass of arithmetic per
// pair), and CTA c starts at the tile where the cost so far reaches
// total * c / G.  Tiles stay in order, so results do not change.
// With route_kind >= 0 it first routes the tokens itself (one warp per token,
// route_token), writing ids and wts (which are then outputs) -- the router
// fused ahead of the expert group, one launch fewer.
__global__ void __launch_bounds__(1024) k_expert_prep(int32_t* __restrict__ ids, int P, int k, int E, int smax,
                                                      int G, int tpb_up, int tpb_down, unsigned char* ws,
                                                      WsLayout L, int32_t* status_dev, int route_kind,
                                                      const float* __restrict__ logits,
                                                      const float* __restrict__ bias, int renorm, float route_scale,
                                                      float* __restrict__ wts_out)
{
    __shared__ int s_ids[kMaxPairs + 1];
    __shared__ int s_sorted[kMaxPairs];
    __shared__ int s_bad;
    pdl_wait_prev();              // ids may come from the kernel before; the workspace may still be read
    pdl_allow_next();
    int32_t* hdr = reinterpret_cast<int32_t*>(ws + L.hdr);
    int4* batches = reinterpret_cast<int4*>(ws + L.batches);
    int32_t* pair_tok = reinterpret_cast<int32_t*>(ws + L.pair_tok);
    int32_t* pair_of = reinterpret_cast<int32_t*>(ws + L.pair_of);
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    if (route_kind >= 0) {
        const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
        for (int t = threadIdx.x >> 5; t < P / k; t += nw) {
            int id;
            float w;
            route_token<kFusedRouteMaxE / 32>(route_kind, logits + (long long)t * E, bias, E, k, renorm, route_scale,
                                              lane, id, w);
            if (lane < k) {
                s_ids[t * k + lane] = id;
                ids[t * k + lane] = id;
                wts_out[t * k + lane] = w;
            }
        }
    } else {
        for (int p = threadIdx.x; p < P; p += blockDim.x) {
            const int e = ids[p];
            s_ids[p] = e;
            if (e < 0 || e >= E) s_bad = 1;
        }
    }
    __syncthreads();
    if (s_bad) {
        if (threadIdx.x == 0) {
            hdr[0] = QSTATUS_BAD_EXPERT_ID;
            hdr[1] = 0;
            hdr[2] = P;
            if (status_dev) *status_dev = QSTATUS_BAD_EXPERT_ID;
        }
        return;
    }
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int e = s_ids[p];
        int pos = 0;
        for (int q = 0; q < P; q++) {
            const int eq = s_ids[q];
            pos += (eq < e) || (eq == e && q < p);
        }
        s_sorted[pos] = e;
        pair_tok[pos] = p / k;
        pair_of[p] = pos;
    }
    __syncthreads();
    __shared__ int s_nb;
    if (threadIdx.x == 0) {
        int nb = 0;
        for (int pos = 0; pos < P;) {
            const int e = s_sorted[pos];
            int n = 1;
            while (pos + n < P && s_sorted[pos + n] == e && n < smax) n++;
            batches[nb] = make_int4(e, pos, n, 0);
            s_ids[nb] = pos;                       // pairs before batch nb (ids are no longer needed)
            nb++;
            pos += n;
        }
        s_ids[nb] = P;
        s_nb = nb;
        hdr[0] = QSTATUS_OK;
        hdr[1] = nb;
        hdr[2] = P;
        if (status_dev) *status_dev = QSTATUS_OK;
    }
    __syncthreads();
    const int nb = s_nb;
    int32_t* bounds = reinterpret_cast<int32_t*>(ws + L.bounds);
    for (int i = threadIdx.x; i < 2 * (G + 1); i += blockDim.x) {
        const int phase = i / (G + 1), c = i - phase * (G + 1);
        const long long tpb = phase ? tpb_down : tpb_up;
        long long tile = (long long)nb * tpb;
        if (c < G && tpb > 0) {
            const long long x = (long long)P * tpb * c / G;     // cost before CTA c
            int lo = 0, hi = nb - 1;                            // last batch starting at or before x
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if ((long long)s_ids[mid] * tpb <= x) lo = mid;
                else hi = mid - 1;
            }
            const long long n = s_ids[lo + 1] - s_ids[lo];
            tile = (long long)lo * tpb + (x - (long long)s_ids[lo] * tpb) / n;
        } else if (c < G) {
            tile = 0;
        }
        bounds[phase * (kMaxGrid + 1) + c] = (int32_t)tile;   // the layout's two rows of kMaxGrid + 1
    }
}

// out[t][d] = sum_{r < k} w[t][r] * z[pair_of[t k + r]][d], in rank order.
__global__ void k_expert_combine(const float* __restrict__ wts, int k, int D, const unsigned char* ws, WsLayout L,
                                 float* __restrict__ out)
{
    pdl_allow_next();
    pdl_wait_prev();              // z comes from the down phase
    const int t = blockIdx.y;
    const int d = blockIdx.x * blockDim.x + threadIdx.x;
    if (d >= D) return;
    const int32_t* hdr = reinterpret_cast<const int32_t*>(ws + L.hdr);
    const int32_t* pair_of = reinterpret_cast<const int32_t*>(ws + L.pair_of);
    const float* z = reinterpret_cast<const float*>(ws + L.z);
    float acc = 0.0f;
    if (hdr[0] == QSTATUS_OK) {
        for (int r = 0; r < k; r++)
            acc = fmaf(wts[t * k + r], z[(long long)pair_of[t * k + r] * D + d], acc);
    }
    out[(long long)t * D + d] = acc;
}

cudaError_t expert_prep(const ExpertArgs& a, cudaStream_t st)
{
    const WsLayout L = ws_layout(a.D, a.F, a.s, a.k);
    return launch_pdl(k_expert_prep, dim3(1), dim3(1024), 0, st, const_cast<int32_t*>(a.ids), a.s * a.k, a.k, a.E,
                      a.smax, a.grid, a.tpb_up, a.tpb_down, a.ws, L, a.status_dev, a.route_kind, a.logits, a.bias,
                      a.renorm, a.route_scale, const_cast<float*>(a.wts));
}

cudaError_t expert_combine(const ExpertArgs& a, cudaStream_t st)
{
    const WsLayout L = ws_layout(a.D, a.F, a.s, a.k);
    dim3 grid((a.D + 255) / 256, a.s);
    return launch_pdl(k_expert_combine, grid, dim3(256), 0, st, a.wts, a.k, a.D,
                      static_cast<const unsigned char*>(a.ws), L, a.out);
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against
// the driver library).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled_fn()
{
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

bool encode_rows_map(CUtensorMap* map, const void* base, long long rows, long long row_bytes, int box_bytes,
                     int box_rows, bool f32)
{
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn || rows <= 0 || row_bytes <= 0 || row_bytes % 16 || box_bytes % 16 || box_bytes > 1024 ||
        box_rows < 1 || box_rows > 256 || !aligned(base, 16))
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(box_bytes / 4), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT32, 2,
              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_x_map(CUtensorMap* map, const void* base, long long rows, long long cols, int box_rows)
{
    const EncodeTiledFn fn = encode_tiled_fn();
    if (!fn || rows < box_rows || cols <= 0 || cols % 64 || box_rows < 1 || box_rows > 256 || !aligned(base, 16))
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qg

using namespace qg;

extern "C" {

const char* qstatus_string(int status)
{
    switch (status) {
    case QSTATUS_OK: return "ok";
    case QSTATUS_BAD_FMT: return "unknown weight format, or a group size that format does not allow";
    case QSTATUS_BAD_DIM: return "a size is out of range or not the multiple its format needs";
    case QSTATUS_MISALIGNED: return "a pointer lacks the required alignment (16 B for packed weights and "
                                    "activations, 256 B for workspaces, 4 B for scales and outputs)";
    case QSTATUS_NULL: return "a required pointer is NULL";
    case QSTATUS_WORKSPACE: return "workspace smaller than the call's *_workspace() size";
    case QSTATUS_LAUNCH: return "CUDA reported an error at launch (see qlast_cuda_error)";
    case QSTATUS_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case QSTATUS_BAD_EXPERT_ID: return "an expert id is outside [0, E)";
    case QSTATUS_BAD_ACT: return "unknown activation, or a clamp limit that is negative or NaN";
    case QSTATUS_BAD_ROUTE: return "unknown router kind, or a NaN router scale";
    default: return "unknown status";
    }
}

const char* qlast_cuda_error(void) { return g_last_cuda_error; }

int qdebug_inject(int kind, long long wait_ns)
{
    if (kind == QDEBUG_NONE) {
        g_inject.store(QDEBUG_NONE);
        return QSTATUS_OK;
    }
    if (kind != QDEBUG_WITHHOLD_SIGNAL || wait_ns < 1) return QSTATUS_BAD_DIM;
    g_inject_ns.store(wait_ns);
    g_inject.store(kind);
    return QSTATUS_OK;
}

int qkernel_policy(int policy)
{
    if (policy != QKERNEL_AUTO && policy != QKERNEL_RING && policy != QKERNEL_TILE && policy != QKERNEL_ROW)
        return QSTATUS_BAD_FMT;
    return g_kernel_policy.exchange(policy);
}

int qdevice_error(int clear)
{
    const int e[7] = {device_error_int8(clear),  device_error_int8g(clear), device_error_int4r(clear),
                      device_error_int4(clear),  device_error_int3(clear),  device_error_mxfp4(clear),
                      device_error_mxfp4e(clear)};
    for (int v : e)
        if (v != QSTATUS_OK) return v;
    return QSTATUS_OK;
}

int qgemv(int fmt, int gs, const void* w, const float* scales, const float* x, int O, int I, int s, float* y,
          void* stream)
{
    int g = 0;
    int st = check_fmt(fmt, gs, I, &g);
    if (st) return st;
    if (O < 1 || I < 1 || s < 1 || I > kMaxI) return QSTATUS_BAD_DIM;
    if (!w || !scales || !x || !y) return QSTATUS_NULL;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(scales, 4) || !aligned(y, 4)) return QSTATUS_MISALIGNED;
    int status = QSTATUS_OK;
    const int grid = sm_count(&status);
    if (status) return status;
    const HostMat m{w, scales, O, I, g};
    const int per = rows_per_launch(fmt, 1, I);
    if (per < 1) return QSTATUS_BAD_DIM;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    for (int s0 = 0; s0 < s; s0 += per) {
        const int n = s - s0 < per ? s - s0 : per;
        const float* xs = x + (size_t)s0 * I;
        float* ys = y + (size_t)s0 * O;
        cudaError_t e;
#define QG_CALL(name) gemv_##name(m, xs, n, ys, O, grid, cs)
        QG_FMT_SWITCH(fmt, QG_CALL)
#undef QG_CALL
        if (e != cudaSuccess) return launch_status(e);
    }
    return QSTATUS_OK;
}

int qgate_up(int fmt, int gs, const void* wg, const float* sg, const void* wu, const float* su, const float* x,
             int F, int D, int s, float* h, void* stream)
{
    return qgate_up_act(fmt, gs, wg, sg, wu, su, x, F, D, s, QACT_SWIGLU, 0.0f, h, stream);
}

int qgate_up_act(int fmt, int gs, const void* wg, const float* sg, const void* wu, const float* su,
                 const float* x, int F, int D, int s, int act, float limit, float* h, void* stream)
{
    int st = check_act(act, limit);
    if (st) return st;
    int g = 0;
    st = check_fmt(fmt, gs, D, &g);
    if (st) return st;
    if (F < 1 || D < 1 || s < 1 || D > kMaxI) return QSTATUS_BAD_DIM;
    if (!wg || !sg || !wu || !su || !x || !h) return QSTATUS_NULL;
    if (!aligned(wg, 16) || !aligned(wu, 16) || !aligned(x, 16) || !aligned(sg, 4) || !aligned(su, 4) ||
        !aligned(h, 4))
        return QSTATUS_MISALIGNED;
    int status = QSTATUS_OK;
    const int grid = sm_count(&status);
    if (status) return status;
    const HostMat mg{wg, sg, F, D, g}, mu{wu, su, F, D, g};
    const int per = rows_per_launch(fmt, 2, D);
    if (per < 1) return QSTATUS_BAD_DIM;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    for (int s0 = 0; s0 < s; s0 += per) {
        const int n = s - s0 < per ? s - s0 : per;
        cudaError_t e;
#define QG_CALL(name) gate_up_##name(mg, mu, x + (size_t)s0 * D, n, h + (size_t)s0 * F, F, act, limit, grid, cs)
        QG_FMT_SWITCH(fmt, QG_CALL)
#undef QG_CALL
        if (e != cudaSuccess) return launch_status(e);
    }
    return QSTATUS_OK;
}

size_t qexpert_group_workspace(int E, int D, int F, int s, int k)
{
    (void)E;
    if (D < 1 || F < 1 || s < 1 || k < 1) return 0;
    return ws_layout(D, F, s, k).total;
}

int qexpert_group(int fmt, int gs, const void* gate, const float* gate_s, const void* up, const float* up_s,
                  const void* down, const float* down_s, int E, int D, int F, const float* x, int s, int k,
                  const int32_t* ids, const float* wts, float* out, void* workspace, size_t ws_bytes,
                  int32_t* status_dev, void* stream)
{
    return qexpert_group_act(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids, wts,
                             QACT_SWIGLU, 0.0f, out, workspace, ws_bytes, status_dev, stream);
}

struct FusedRoute {
    int kind;
    const float* logits;
    const float* bias;
    int renorm;
    float scale;
};

static int expert_group_impl(int fmt, int gs, const void* gate, const float* gate_s, const void* up,
                             const float* up_s, const void* down, const float* down_s, int E, int D, int F,
                             const float* x, int s, int k, const int32_t* ids, const float* wts, int act, float limit,
                             float* out, void* workspace, size_t ws_bytes, int32_t* status_dev, void* stream,
                             const FusedRoute* route);

int qexpert_group_act(int fmt, int gs, const void* gate, const float* gate_s, const void* up, const float* up_s,
                      const void* down, const float* down_s, int E, int D, int F, const float* x, int s, int k,
                      const int32_t* ids, const float* wts, int act, float limit, float* out, void* workspace,
                      size_t ws_bytes, int32_t* status_dev, void* stream)
{
    return expert_group_impl(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids, wts, act, limit,
                             out, workspace, ws_bytes, status_dev, stream, nullptr);
}

}  // extern "C"

// Every host-side check of the expert group (the same for the routed call,
// which runs it before it enqueues the router).
static int expert_checks(int fmt, int gs, const void* gate, const float* gate_s, const void* up, const float* up_s,
                         const void* down, const float* down_s, int E, int D, int F, const float* x, int s, int k,
                         const int32_t* ids, const float* wts, int act, float limit, const float* out,
                         const void* workspace, size_t ws_bytes, const int32_t* status_dev, int* g_up, int* g_dn)
{
    int st = check_act(act, limit);
    if (st) return st;
    st = check_fmt(fmt, gs, D, g_up);
    if (st) return st;
    st = check_fmt(fmt, gs, F, g_dn);
    if (st) return st;
    if (E < 1 || D < 1 || F < 1 || s < 1 || k < 1 || D > kMaxI || F > kMaxI) return QSTATUS_BAD_DIM;
    if ((long long)s * k > kMaxPairs) return QSTATUS_BAD_DIM;
    if (!gate || !gate_s || !up || !up_s || !down || !down_s || !x || !ids || !wts || !out || !workspace)
        return QSTATUS_NULL;
    if (!aligned(gate, 16) || !aligned(up, 16) || !aligned(down, 16) || !aligned(x, 16) ||
        !aligned(workspace, 256) || !aligned(gate_s, 4) || !aligned(up_s, 4) || !aligned(down_s, 4) ||
        !aligned(ids, 4) || !aligned(wts, 4) || !aligned(out, 4) || (status_dev && !aligned(status_dev, 4)))
        return QSTATUS_MISALIGNED;
    if (ws_bytes < ws_layout(D, F, s, k).total) return QSTATUS_WORKSPACE;
    return QSTATUS_OK;
}

// Pairs per expert batch at most (a batch's weights are streamed once for all
// its pairs; each pair of a batch holds its own accumulators in the kernels).
// Measured on GB300 for 8 tokens x top 8 of 256 int4 experts: two pairs per
// batch 313 us, four 321 us, one 329 us (four-launch path; the one-launch
// path in the same order).
#ifndef QG_SMAX_CAP
#define QG_SMAX_CAP 2
#endif

// The launch shape of an expert group (no pointers): the grid, the batch
// size smax and the tile counts of the four-launch path.
static int expert_shape(int fmt, int gs_up, int E, int D, int F, int s, int k, ExpertArgs& a)
{
    int status = QSTATUS_OK;
    int grid = sm_count(&status);
    if (status) return status;
    if (grid > kMaxGrid) grid = kMaxGrid;
    a.grid = grid;
    int r_up = 1, r_dn = 1;
    switch (fmt) {
    case QFMT_INT8_ROW: r_up = tile_rows_int8(2); r_dn = tile_rows_int8(1); break;
    case QFMT_INT8_G: r_up = tile_rows_int8g(2); r_dn = tile_rows_int8g(1); break;
    case QFMT_INT4_ROW: r_up = tile_rows_int4r(2); r_dn = tile_rows_int4r(1); break;
    case QFMT_INT4_G: r_up = tile_rows_int4(2); r_dn = tile_rows_int4(1); break;
    case QFMT_INT3_G64: r_up = tile_rows_int3(2); r_dn = tile_rows_int3(1); break;
    case QFMT_MXFP4_E8M0: r_up = tile_rows_mxfp4e(2); r_dn = tile_rows_mxfp4e(1); break;
    default: r_up = tile_rows_mxfp4(2); r_dn = tile_rows_mxfp4(1); break;
    }
    a.tpb_up = (F + r_up - 1) / r_up;
    a.tpb_down = (D + r_dn - 1) / r_dn;
    a.gs = (fmt == QFMT_INT8_ROW || fmt == QFMT_INT4_ROW) ? 0 : gs_up;   // per-row formats: one scale per row
    a.E = E; a.D = D; a.F = F; a.s = s; a.k = k;
    const int up_rows = rows_per_launch(fmt, 2, D), down_rows = rows_per_launch(fmt, 1, F);
    a.smax = up_rows < down_rows ? up_rows : down_rows;
    if (a.smax > QG_SMAX_CAP) a.smax = QG_SMAX_CAP;
    if (a.smax > s) a.smax = s;   // a batch holds pairs of distinct tokens unless a token repeats an id
    if (a.smax < 1) return QSTATUS_BAD_DIM;
    return QSTATUS_OK;
}

// Whether the call runs as the one fused launch (the plan fits and the
// policy allows it).
static bool expert_fuses(int fmt, const ExpertArgs& a)
{
    const int pol = kernel_policy();
    if (!(pol == QKERNEL_AUTO || pol == QKERNEL_ROW) || (long long)a.s * a.k > kFusedMaxPairs) return false;
    bool fits = false;
    cudaError_t e = cudaSuccess;
#define QG_CALL(name) expert_fused_##name(a, a.grid, nullptr, &fits, true)
    QG_FMT_SWITCH(fmt, QG_CALL)
#undef QG_CALL
    return e == cudaSuccess && fits;
}

static int expert_group_impl(int fmt, int gs, const void* gate, const float* gate_s, const void* up,
                             const float* up_s, const void* down, const float* down_s, int E, int D, int F,
                             const float* x, int s, int k, const int32_t* ids, const float* wts, int act, float limit,
                             float* out, void* workspace, size_t ws_bytes, int32_t* status_dev, void* stream,
                             const FusedRoute* route)
{
    int g_up = 0, g_dn = 0;
    int st = expert_checks(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids, wts, act, limit, out,
                           workspace, ws_bytes, status_dev, &g_up, &g_dn);
    if (st) return st;
    ExpertArgs a;
    st = expert_shape(fmt, g_up, E, D, F, s, k, a);
    if (st) return st;
    const int grid = a.grid;
    a.act = act;
    a.limit = limit;
    a.gate = gate; a.up = up; a.down = down;
    a.gate_s = gate_s; a.up_s = up_s; a.down_s = down_s;
    a.x = x; a.ids = ids; a.wts = wts; a.out = out;
    a.ws = static_cast<unsigned char*>(workspace);
    a.status_dev = status_dev;
    if (route) {
        a.route_kind = route->kind;
        a.logits = route->logits;
        a.bias = route->bias;
        a.renorm = route->renorm;
        a.route_scale = route->scale;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    cudaError_t e = cudaSuccess;
    const int pol = kernel_policy();
    if ((pol == QKERNEL_AUTO || pol == QKERNEL_ROW) && (long long)s * k <= kFusedMaxPairs) {
        // one persistent launch: routing (optional), gate/up, down and the rank-order sum
        if (g_inject.exchange(QDEBUG_NONE) == QDEBUG_WITHHOLD_SIGNAL) {
            a.withhold = 1;
            a.wait_ns = (unsigned long long)g_inject_ns.load();
        }
        bool launched = false;
#define QG_CALL(name) expert_fused_##name(a, grid, cs, &launched, false)
        QG_FMT_SWITCH(fmt, QG_CALL)
#undef QG_CALL
        if (launched || e != cudaSuccess) return launch_status(e);
    }
    e = expert_prep(a, cs);
    if (e != cudaSuccess) return launch_status(e);
#define QG_CALL(name) expert_up_##name(a, grid, cs)
    QG_FMT_SWITCH(fmt, QG_CALL)
#undef QG_CALL
    if (e != cudaSuccess) return launch_status(e);
#define QG_CALL(name) expert_down_##name(a, grid, cs)
    QG_FMT_SWITCH(fmt, QG_CALL)
#undef QG_CALL
    if (e != cudaSuccess) return launch_status(e);
    e = expert_combine(a, cs);
    if (e != cudaSuccess) return launch_status(e);
    return QSTATUS_OK;
}

extern "C" {

int qroute(int kind, const float* logits, const float* bias, int s, int E, int k, int renorm, float scale,
           int32_t* ids, float* wts, void* stream)
{
    if ((kind != QROUTE_SOFTMAX && kind != QROUTE_SIGMOID_BIAS) || !(scale == scale)) return QSTATUS_BAD_ROUTE;
    if (s < 1 || E < 1 || E > 1024 || k < 1 || k > E || k > 32) return QSTATUS_BAD_DIM;
    if (!logits || !ids || !wts || (kind == QROUTE_SIGMOID_BIAS && !bias)) return QSTATUS_NULL;
    if (!aligned(logits, 4) || !aligned(ids, 4) || !aligned(wts, 4) || (bias && !aligned(bias, 4)))
        return QSTATUS_MISALIGNED;
    return launch_status(route_launch(kind, logits, kind == QROUTE_SIGMOID_BIAS ? bias : nullptr, s, E, k,
                                      renorm != 0, scale, ids, wts, static_cast<cudaStream_t>(stream)));
}

int qexpert_group_routed(int fmt, int gs, const void* gate, const float* gate_s, const void* up, const float* up_s,
                         const void* down, const float* down_s, int E, int D, int F, const float* x, int s, int k,
                         int route_kind, const float* logits, const float* bias, int renorm, float route_scale,
                         int act, float limit, float* out, int32_t* ids_out, float* wts_out, void* workspace,
                         size_t ws_bytes, int32_t* status_dev, void* stream)
{
    // every host-side check of the expert group first (with the routing outputs
    // as its ids and weights), so a rejected call enqueues nothing
    int g_up = 0, g_dn = 0;
    int st = expert_checks(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids_out, wts_out, act,
                           limit, out, workspace, ws_bytes, status_dev, &g_up, &g_dn);
    if (st) return st;
    if (E > kFusedRouteMaxE) {
        // more experts than the prep kernel's fused routing holds: the router
        // kernel first (qroute checks its own arguments before it enqueues)
        st = qroute(route_kind, logits, bias, s, E, k, renorm, route_scale, ids_out, wts_out, stream);
        if (st) return st;
        return qexpert_group_act(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids_out, wts_out,
                                 act, limit, out, workspace, ws_bytes, status_dev, stream);
    }
    // the routing inside the expert prep kernel: qroute's checks, then one launch fewer
    if ((route_kind != QROUTE_SOFTMAX && route_kind != QROUTE_SIGMOID_BIAS) || !(route_scale == route_scale))
        return QSTATUS_BAD_ROUTE;
    if (k > E || k > 32) return QSTATUS_BAD_DIM;
    if (!logits || (route_kind == QROUTE_SIGMOID_BIAS && !bias)) return QSTATUS_NULL;
    if (!aligned(logits, 4) || (bias && !aligned(bias, 4))) return QSTATUS_MISALIGNED;
    const FusedRoute fr{route_kind, logits, route_kind == QROUTE_SIGMOID_BIAS ? bias : nullptr, renorm != 0,
                        route_scale};
    return expert_group_impl(fmt, gs, gate, gate_s, up, up_s, down, down_s, E, D, F, x, s, k, ids_out, wts_out, act,
                             limit, out, workspace, ws_bytes, status_dev, stream, &fr);
}

int qexpert_group_launches(int fmt, int gs, int E, int D, int F, int s, int k, int routed)
{
    int g_up = 0, g_dn = 0;
    int st = check_fmt(fmt, gs, D, &g_up);
    if (st) return st;
    st = check_fmt(fmt, gs, F, &g_dn);
    if (st) return st;
    if (E < 1 || D < 1 || F < 1 || s < 1 || k < 1 || D > kMaxI || F > kMaxI) return QSTATUS_BAD_DIM;
    if ((long long)s * k > kMaxPairs) return QSTATUS_BAD_DIM;
    ExpertArgs a;
    st = expert_shape(fmt, g_up, E, D, F, s, k, a);
    if (st) return st;
    const int router = routed && E > kFusedRouteMaxE ? 1 : 0;   // the router kernel ahead of the group
    return router + (expert_fuses(fmt, a) ? 1 : 4);
}

size_t qgemm_workspace(int I, int s)
{
    if (I < 1 || s < 1) return 0;
    return gemm_ws_layout(I, s).total;
}

int qgemm(int fmt, int gs, const void* w, const float* scales, const float* x, int O, int I, int s, float* y,
          void* workspace, size_t ws_bytes, void* stream)
{
    int g = 0;
    int st = check_fmt(fmt, gs, I, &g);
    if (st) return st;
    if (g < 32) return QSTATUS_BAD_FMT;                     // partials of at least 32 inputs
    if (O < 1 || I < 1 || s < 1 || I % 64 || I > kGemmMaxI || s > kGemmMaxS) return QSTATUS_BAD_DIM;
    if (!w || !scales || !x || !y || !workspace) return QSTATUS_NULL;
    if (!aligned(w, 16) || !aligned(x, 16) || !aligned(scales, 4) || !aligned(y, 4) || !aligned(workspace, 256))
        return QSTATUS_MISALIGNED;
    const GemmWs L = gemm_ws_layout(I, s);
    if (ws_bytes < L.total) return QSTATUS_WORKSPACE;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    GemmArgs a;
    a.xh = ws + L.xh;
    a.xl = ws + L.xl;
    a.pexp = reinterpret_cast<const int32_t*>(ws + L.pexp);
    a.s = s;
    a.sp = gemm_rows(s);
    a.y = y;
    // the decoders' input order: int4 nibble pairs (q, q + 4), int3 (q, q + 8)
    const int perm = (fmt == QFMT_INT4_G || fmt == QFMT_INT4_ROW) ? 8 : (fmt == QFMT_INT3_G64 ? 16 : 0);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = gemm_split_x(x, s, a.sp, I, perm, ws + L.xh, ws + L.xl, reinterpret_cast<int32_t*>(ws + L.pexp),
                                 cs);
    if (e != cudaSuccess) return launch_status(e);
    const HostMat m{w, scales, O, I, g};
#define QG_CALL(name) gemm_##name(m, a, cs)
    QG_FMT_SWITCH(fmt, QG_CALL)
#undef QG_CALL
    return launch_status(e);
}

int qdequant(int fmt, int gs, const void* w, const float* scales, int O, int I, float* out, void* stream)
{
    int g = 0;
    int st = check_fmt(fmt, gs, I, &g);
    if (st) return st;
    if (O < 1 || I < 1) return QSTATUS_BAD_DIM;
    if (!w || !scales || !out) return QSTATUS_NULL;
    if (!aligned(w, 16) || !aligned(scales, 4) || !aligned(out, 4)) return QSTATUS_MISALIGNED;
    const HostMat m{w, scales, O, I, g};
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
#define QG_CALL(name) dequant_##name(m, out, cs)
    QG_FMT_SWITCH(fmt, QG_CALL)
#undef QG_CALL
    return launch_status(e);
}

}  // extern "C"
