// qg_fmt_impl.cuh -- the streaming kernels and their launchers for one weight
// format.  Included by qg_fmt_<format>.cu with QG_FMT (format id) and QG_NAME
// (launcher suffix) defined, so the four formats compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "qg_device.cuh"
#include "qg_internal.h"
#include "qg_route.cuh"

#ifndef QG_FMT
#error "define QG_FMT and QG_NAME before including qg_fmt_impl.cuh"
#endif

#define QG_CAT2(a, b) a##b
#define QG_CAT(a, b) QG_CAT2(a, b)

namespace qg {
namespace QG_CAT(fmt_, QG_NAME) {

constexpr int QF = QG_FMT;                 // the format of this translation unit
constexpr int FMT = decode_of(QF);         // its code decoding
constexpr int SK = scale_kind_of(QF);      // its scales: per row, f32 per group, ue8m0 per group
constexpr int EPL = Traits<FMT>::EPL;

// Ring kernels with shared scales (see RowStreamer): always for row scales and
// ue8m0 words; for the grouped int4/int8 formats when a group spans several
// chunks (gsh > 0), picked per launch.
constexpr bool kShareAlways = SK != SK_F32;
constexpr bool kShareMaybe = SK == SK_F32 && (QF == FMT_INT4_G || QF == FMT_INT8_G);

template <class F>
static cudaError_t with_share(int gsh, F&& f)
{
    if constexpr (kShareMaybe) {
        if (gsh > 0) return f(std::true_type{});
        return f(std::false_type{});
    } else {
        return f(std::integral_constant<bool, kShareAlways>{});
    }
}

// Rows per warp tile: up to 4 chunk rows (NM matrices x R rows) so each x
// quad read from shared memory serves several rows, and at most 8
// accumulators (S x NM x R) so everything stays in registers.
// int3 chunks take 7 registers instead of 5, so their budget is 4
// accumulators beyond the single-row-set case.
#ifndef QG_RMAX
#define QG_RMAX 4
#endif
template <int S, int NM>
__host__ __device__ constexpr int rows_per_tile()
{
    constexpr int acc_budget = FMT == FMT_INT3_G64 ? 4 : 8;
    constexpr int rmax = FMT == FMT_INT3_G64 ? 2 : QG_RMAX;
    constexpr int by_acc = acc_budget / (S * NM) > 0 ? acc_budget / (S * NM) : 1;
    constexpr int by_rows = rmax / NM > 0 ? rmax / NM : 1;
    return by_rows < by_acc ? by_rows : by_acc;
}

// Rows per tile of the tile kernel: up to QG_TILE_RMAX / NM rows of each
// matrix, at most 16 accumulators (S x NM x R), so that each x quad loaded
// from shared memory serves four rows up to four activation rows (shared
// memory bandwidth bounds the several-row case).  MXFP4 decodes with fewer live
// registers and measured faster with taller tiles.
#ifndef QG_TILE_RMAX
#define QG_TILE_RMAX (FMT == FMT_MXFP4_G32 ? 8 : 4)
#endif
#ifndef QG_TILE_ACC
#define QG_TILE_ACC 16
#endif
template <int S, int NM>
__host__ __device__ constexpr int tile_rows_per()
{
    constexpr int rmax = FMT == FMT_INT3_G64 ? (QG_TILE_RMAX < 4 ? QG_TILE_RMAX : 4) : QG_TILE_RMAX;
    constexpr int by_acc = QG_TILE_ACC / (S * NM) > 0 ? QG_TILE_ACC / (S * NM) : 1;
    constexpr int by_rows = rmax / NM > 0 ? rmax / NM : 1;
    return by_rows < by_acc ? by_rows : by_acc;
}

#ifndef QG_RING
#define QG_RING 2
#endif
constexpr int kRing = QG_RING;   // chunk-register ring depth

inline Mat to_mat(const HostMat& h)
{
    Mat m;
    m.w = static_cast<const uint8_t*>(h.w);
    m.sc = h.sc;
    m.O = h.O;
    m.I = h.I;
    m.ngrp = SK == SK_ROW ? 1 : h.I / h.gs;
    int sh = 0;                            // groups are whole chunks: chunk q is in group q >> sh
    if (SK != SK_ROW) while ((EPL << sh) < h.gs) sh++;
    m.gsh = sh;
    return m;
}

// ---------------------------------------------------------------------------
// Jobs: where rows, activations and results of a streaming launch live.
// ---------------------------------------------------------------------------

// One matrix (or a gate/up pair) against s <= 8 activation rows.
// Shared-memory layout of every streaming launch: the activation rows at
// offset 0, then one cp.async ring per warp at ring_off + warp * ring_stride.
struct RingLayout {
    int ring_off;
    int ring_stride;
};

// Ring bytes per warp: kRing slots sized for the tiles of S activation rows.
template <int NM, int S = 1>
__host__ __device__ constexpr int ring_stride_bytes()
{
    return kRing * ring_slot_bytes<FMT, NM * rows_per_tile<S, NM>()>();
}

// Tensor-copy sources of the tile kernel: per matrix m, tm[3m] codes (int3:
// plane A), tm[3m + 1] int3 plane B, tm[3m + 2] scales, each a tensor of rows;
// row r of expert e of piece p is tensor row e * row_mul[p] + row_add[p] + r.
template <int NM>
struct TileSource {
    TileLayout tile;
    CUtensorMap tm[3 * NM];
    long long row_mul[3], row_add[3];
    // Activation rows come from before the launch; no per-batch signals.
    static constexpr bool kFreshX = false;
    static constexpr bool kSignals = false;
    static constexpr bool kWaits = false;
    __device__ void warp_done(int, int) const {}
    __device__ void segment_poll(int) const {}
    __device__ bool segment_ready() const { return true; }
    __device__ const TileLayout& layout() const { return tile; }
    __device__ const CUtensorMap* tmap(int i) const { return &tm[i]; }
    __device__ long long rmul(int p) const { return row_mul[p]; }
    __device__ long long radd(int p) const { return row_add[p]; }
};

template <int NM>
struct DenseJob : RingLayout, TileSource<NM> {
    static constexpr bool kLoopS = false;     // activation rows share each decoded word
    // Reads nothing the previous kernel may write before the activations: the
    // weight stream may start before that kernel completes.
    static constexpr bool kWaitFirst = false;
    Mat m[NM];
    const float* x;      // [S][I]
    float* y;            // y[s * ldy + row]
    long long ldy;
    int S;
    int act;             // NM = 2: QACT_* of the gate/up product
    float limit;

    __device__ bool bad() const { return false; }
    __device__ int nbatch() const { return 1; }
    __device__ long long rows_per() const { return m[0].O; }
    __device__ int batch_S(int) const { return S; }
    __device__ void mats(int, Mat (&out)[NM]) const
    {
#pragma unroll
        for (int k = 0; k < NM; k++) out[k] = m[k];
    }
    __device__ const float* xrow(int, int s) const { return x + (long long)s * m[0].I; }
    __device__ void store(int, int s, long long row, float v) const { y[(long long)s * ldy + row] = v; }
    __device__ int width() const { return m[0].I; }
    __device__ int* status_word() const { return nullptr; }
    __device__ long long expert_of(int) const { return 0; }
    // row tiles [t0, t1) of CTA c of G (T tiles in all): an even split
    __device__ void cta_tiles(int c, int G, long long T, int& t0, int& t1) const
    {
        t0 = (int)(T * c / G);
        t1 = (int)(T * (c + 1) / G);
    }
};

// Expert phase A: the gate and up rows of every used expert, against the
// tokens routed to it; stores h = silu(g) * u per sorted pair.
struct ExpertUpJob : RingLayout, TileSource<2> {
    static constexpr bool kLoopS = true;      // one-pair tiles, one pass of arithmetic per pair
    // Its batches come from the prep kernel just before it: wait first.  (It
    // lets the down phase start only after that, so the down phase may read
    // the batches early.)
    static constexpr bool kWaitFirst = true;
    int* status;
    Mat gate0, up0;                 // expert 0's matrices (w, sc advanced per expert)
    long long mat_bytes, mat_scales;
    const float* x;
    const int32_t* hdr;
    const int4* batches;
    const int32_t* pair_tok;
    const int32_t* bounds;          // CTA tile bounds of this phase (G + 1 entries)
    float* h;
    int D, F;
    int act;                        // QACT_* of the gate/up product
    float limit;

    __device__ bool bad() const { return hdr[0] != 0; }
    __device__ int nbatch() const { return hdr[1]; }
    __device__ long long rows_per() const { return F; }
    __device__ int batch_S(int b) const { return batches[b].z; }
    __device__ void mats(int b, Mat (&out)[2]) const
    {
        const long long e = batches[b].x;
        out[0] = gate0;
        out[0].w += e * mat_bytes;
        out[0].sc = sc_ptr<SK>(out[0].sc, e * mat_scales);
        out[1] = up0;
        out[1].w += e * mat_bytes;
        out[1].sc = sc_ptr<SK>(out[1].sc, e * mat_scales);
    }
    __device__ const float* xrow(int b, int s) const { return x + (long long)pair_tok[batches[b].y + s] * D; }
    __device__ void store(int b, int s, long long row, float v) const
    {
        h[(long long)(batches[b].y + s) * F + row] = v;
    }
    __device__ int width() const { return D; }
    __device__ int* status_word() const { return status; }
    __device__ long long expert_of(int b) const { return batches[b].x; }
    // row tiles [t0, t1) of CTA c: the cost-balanced split the prep kernel wrote
    __device__ void cta_tiles(int c, int, long long T, int& t0, int& t1) const
    {
        t0 = bounds[c];
        t1 = bounds[c + 1];
        t0 = t0 < 0 ? 0 : (t0 > T ? (int)T : t0);         // never trust a workspace word with an index
        t1 = t1 < t0 ? t0 : (t1 > T ? (int)T : t1);
    }
};

// Expert phase B: the down rows of every used expert against the h vectors of
// its pairs; stores z = down h per sorted pair.
struct ExpertDownJob : RingLayout, TileSource<1> {
    static constexpr bool kLoopS = true;
    // The batches were complete before the up phase let this kernel start;
    // only h (the up phase's output) needs the wait.
    static constexpr bool kWaitFirst = false;
    int* status;
    Mat down0;
    long long mat_bytes, mat_scales;
    const int32_t* hdr;
    const int4* batches;
    const int32_t* bounds;
    const float* h;
    float* z;
    int D, F;

    __device__ bool bad() const { return hdr[0] != 0; }
    __device__ int nbatch() const { return hdr[1]; }
    __device__ long long rows_per() const { return D; }
    __device__ int batch_S(int b) const { return batches[b].z; }
    __device__ void mats(int b, Mat (&out)[1]) const
    {
        const long long e = batches[b].x;
        out[0] = down0;
        out[0].w += e * mat_bytes;
        out[0].sc = sc_ptr<SK>(out[0].sc, e * mat_scales);
    }
    __device__ const float* xrow(int b, int s) const { return h + (long long)(batches[b].y + s) * F; }
    __device__ void store(int b, int s, long long row, float v) const
    {
        z[(long long)(batches[b].y + s) * D + row] = v;
    }
    __device__ int width() const { return F; }
    __device__ int* status_word() const { return status; }
    __device__ long long expert_of(int b) const { return batches[b].x; }
    // row tiles [t0, t1) of CTA c: the cost-balanced split the prep kernel wrote
    __device__ void cta_tiles(int c, int, long long T, int& t0, int& t1) const
    {
        t0 = bounds[c];
        t1 = bounds[c + 1];
        t0 = t0 < 0 ? 0 : (t0 > T ? (int)T : t0);         // never trust a workspace word with an index
        t1 = t1 < t0 ? t0 : (t1 > T ? (int)T : t1);
    }
};

// Hands finished tiles to the job (NM = 2: h = silu(gate) * up).  A reduced
// value with index v = (s * R + r) * NM + m belongs to activation row s, tile
// row r, matrix m; V is the (power-of-two) count that was reduced.
template <class Job, int S, int R, int NM>
struct Sink {
    const Job& job;
    int b;
    int s_act;
    template <int V>
    __device__ __forceinline__ void put(float v, int idx, bool lane_ok, long long tile_row0, long long row_end) const
    {
        if constexpr (NM == 2) {
            float u = __shfl_xor_sync(0xffffffffu, v, V / 2);
            if (lane_ok && !(idx & 1) && idx < S * R * 2) {
                const int sr = idx >> 1, s = sr / R, r = sr - (sr / R) * R;
                const long long row = tile_row0 + r;
                float g = v;
                if (job.act == QACT_SWIGLU_CLAMPED) {    // clamped SwiGLU: gate capped, up clamped to [-L, L]
                    g = fminf(g, job.limit);
                    u = fminf(fmaxf(u, -job.limit), job.limit);
                }
                if (row < row_end && s < s_act) job.store(b, s, row, g / (1.0f + expf(-g)) * u);
            }
        } else {
            if (lane_ok && idx < S * R) {
                const int s = idx / R, r = idx - (idx / R) * R;
                const long long row = tile_row0 + r;
                if (row < row_end && s < s_act) job.store(b, s, row, v);
            }
        }
    }
};

// One segment: rows [l0, l1) of batch b, all warps of the CTA, with the
// batch's s_act <= S activation rows; warp w takes the row tiles w, w + W, ...
template <int NM, int S, class Job, int RF = 0, bool SH = false>
__device__ __forceinline__ void segment(const Job& job, int b, long long l0, long long l1, int s_act, float* xs,
                                        int& staged)
{
    constexpr int R = RF > 0 ? RF : rows_per_tile<Job::kLoopS ? 1 : S, NM>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Mat m[NM];
    job.mats(b, m);
    RowStreamer<QF, S, R, kRing, NM, Job::kLoopS, SH> st;
    const int ntiles = (int)((l1 - l0 + R - 1) / R);
    st.begin(m, l0, l1, warp, ntiles, (int)(blockDim.x >> 5), lane,
             (uint32_t)(job.ring_off + warp * job.ring_stride));   // copies in flight during staging
    const int I = m[0].I;
    if (b != staged) {
        if (!Job::kWaitFirst && staged < 0) pdl_wait_prev();   // before the first read of activations
        __syncthreads();
        const float* src[S];
#pragma unroll
        for (int s = 0; s < S; s++) src[s] = job.xrow(b, s < s_act ? s : 0);
        stage_rows<EPL>(xs, I, src, s_act, I);
        __syncthreads();
        staged = b;
    }
    uint32_t xsh[S];
#pragma unroll
    for (int s = 0; s < S; s++) xsh[s] = (uint32_t)(s * I) * 4u;   // byte offsets: x rows start at 0
    Sink<Job, S, R, NM> sink{job, b, s_act};
    st.run(xsh, s_act, sink);
}

// The streaming kernel: CTA c takes the rows [N c / G, N (c+1) / G) of the
// job's batches laid end to end (N = batches * rows per batch), so every SM
// gets the same number of weight rows; the range splits into segments where
// the batch (and so the staged activation set) changes.  S is the number of
// activation rows the code is built for; a batch may use fewer.  RF > 0
// forces RF rows per tile (single rows for matrices too short to give every
// warp a tile of the default height).
template <int NM, int S, class Job, int RF = 0, bool SH = false>
__global__ void __launch_bounds__(kThreads, 1) k_stream(const __grid_constant__ Job job)
{
    float* xs = reinterpret_cast<float*>(qg_smem4);
    if constexpr (Job::kWaitFirst) pdl_wait_prev();
    pdl_allow_next();
    if (job.bad()) return;
    const long long rows_per = job.rows_per();
    const long long N = (long long)job.nbatch() * rows_per;
    const long long r_begin = N * blockIdx.x / gridDim.x;
    const long long r_end = N * (blockIdx.x + 1) / gridDim.x;
    int staged = -1;
    long long r = r_begin;
    while (r < r_end) {
        const int b = (int)(r / rows_per);
        const long long base = (long long)b * rows_per;
        const long long l0 = r - base;
        const long long l1 = (r_end - base) < rows_per ? (r_end - base) : rows_per;
        segment<NM, S, Job, RF, SH>(job, b, l0, l1, job.batch_S(b), xs, staged);
        r = base + l1;
    }
}

#include "qg_tile.cuh"

// ---------------------------------------------------------------------------
// Dequantization: one thread per chunk, the same decoding arithmetic as the
// dot products, then one f32 multiplication by the scale.
// ---------------------------------------------------------------------------
template <int F_>
__device__ __forceinline__ void decode_chunk(const Chunk<F_>& c, float* v)
{
    if constexpr (F_ == FMT_INT4_G || F_ == FMT_MXFP4_G32) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float2 d[4];
            if constexpr (F_ == FMT_INT4_G) decode_int4_word(word(c.w, j), Int4Magic(), d);
            else decode_mxfp4_word(word(c.w, j), d);
#pragma unroll
            for (int k = 0; k < 4; k++) {
                v[8 * j + 2 * k] = d[k].x;
                v[8 * j + 2 * k + 1] = d[k].y;
            }
        }
    } else if constexpr (F_ == FMT_INT8_ROW) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float2 d[2];
            decode_int8_word(word(c.w, j), d);
            v[4 * j + 0] = d[0].x;
            v[4 * j + 1] = d[0].y;
            v[4 * j + 2] = d[1].x;
            v[4 * j + 3] = d[1].y;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            uint32_t cls[4];
            const uint32_t bh = ((j & 2) ? c.b.y : c.b.x) >> ((j & 1) * 16);
            int3_classes(word(c.a, j), bh, cls);
#pragma unroll
            for (int m = 0; m < 4; m++) {
                float2 d[2];
                decode_int3_quad(cls, m, d);
                v[16 * j + 4 * m + 0] = d[0].x;
                v[16 * j + 4 * m + 1] = d[0].y;
                v[16 * j + 4 * m + 2] = d[1].x;
                v[16 * j + 4 * m + 3] = d[1].y;
            }
        }
    }
}

__global__ void k_dequant(const Mat m, float* __restrict__ out)
{
    const long long nchunks = (long long)(m.I / EPL);
    const long long total = m.O * nchunks;
    for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const long long o = t / nchunks;
        const int q = (int)(t - o * nchunks);
        Chunk<FMT> c;
        float sc;
        load_chunk<QF>(m, o, q, c, sc);
        float v[EPL];
        decode_chunk<FMT>(c, v);
        float* dst = out + o * m.I + (long long)q * EPL;
#pragma unroll
        for (int i = 0; i < EPL; i++) dst[i] = v[i] * sc;
    }
}

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------
// Raises a kernel's dynamic shared-memory limit when a launch needs more than
// it was last given (per device), so repeated calls -- and launches captured
// into a CUDA graph after a first eager call -- make no attribute call.
// `granted` is the calling launcher's own per-device record for `kernel`.
template <class K>
static cudaError_t set_smem(K kernel, size_t bytes, int (&granted)[64])
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && granted[dev] >= (int)bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) granted[dev] = (int)bytes;
    return e;
}

#ifndef QG_TILE
#define QG_TILE 1
#endif
#ifndef QG_TILE_PMAX
#define QG_TILE_PMAX 2
#endif

static int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Plans the tile kernel's shared memory for NM matrices, R rows per tile, rows
// of I inputs in groups of gs and xrows staged activation rows.  False when
// the shapes do not suit it (a slice's scales under 16 bytes) or fewer than
// two slots per warp fit; the per-warp ring kernel then runs instead.
static bool plan_tile(int NM, int R, int I, int gs, int xrows, TileLayout& L)
{
    if (!QG_TILE) return false;
    constexpr int KS = 32 * EPL;
    L.nslices = (I + KS - 1) / KS;
    L.xstride = L.nslices * KS;
    // scale bytes per row per slice: none for one scale per row (read from global per tile)
    L.sbox = SK == SK_ROW ? 0 : (KS / gs) * (SK == SK_E8M0 ? 1 : 4);
    if (SK != SK_ROW && (KS % gs != 0 || L.sbox < 16)) return false;
    L.tx_bytes = NM * R * (512 + (FMT == FMT_INT3_G64 ? 256 : 0) + L.sbox);
    int off = 0;
    for (int m = 0; m < 2; m++) L.code_off[m] = L.b_off[m] = L.s_off[m] = 0;
    for (int m = 0; m < NM; m++) { L.code_off[m] = off; off = align_up(off + R * 512, 128); }
    if (FMT == FMT_INT3_G64)
        for (int m = 0; m < NM; m++) { L.b_off[m] = off; off = align_up(off + R * 256, 128); }
    if (SK != SK_ROW)
        for (int m = 0; m < NM; m++) { L.s_off[m] = off; off = align_up(off + R * L.sbox, 128); }
    L.slot_bytes = off;
    L.ring_off = align_up(xrows * L.xstride * 4, 128);
    const int per_p = kTileWarps * L.slot_bytes;
    int P = (kSmemMax - L.ring_off - 8 * (kTileWarps * QG_TILE_PMAX + 1)) / per_p;
    if (P > QG_TILE_PMAX) P = QG_TILE_PMAX;
    if (P < 2) return false;
    L.P = P;
    L.warp_bytes = P * L.slot_bytes;
    L.bar_off = L.ring_off + P * per_p;
    L.total = L.bar_off + 8 * (kTileWarps * P + 1);
    return true;
}

// Code-row bytes of a matrix with I inputs (int3: plane A).
static long long code_row_bytes(int I) { return FMT == FMT_INT8_ROW ? I : (FMT == FMT_INT3_G64 ? I / 4 : I / 2); }

// Tensor maps of NM matrices of E experts (E = 1: a plain matrix) of O rows
// and I inputs each, matrix bytes mat_bytes apart, R rows per tile.
template <int NM>
static bool tile_sources(TileSource<NM>& src, const void* const (&w)[NM], const float* const (&sc)[NM], long long E,
                         long long O, int I, int gs, long long mat_bytes, int R)
{
    const long long rb = code_row_bytes(I);
    const long long rbB = I / 8;
    const long long sb = (long long)(I / gs) * (SK == SK_E8M0 ? 1 : 4);   // scale bytes per row
    const long long total = E * mat_bytes;
    if (E * O >= (1ll << 31) || total / rb >= (1ll << 31) || (FMT == FMT_INT3_G64 && total / rbB >= (1ll << 31)))
        return false;     // tensor rows and tile indices are 32-bit in the kernel
    if (E > 1 && (mat_bytes % rb || (FMT == FMT_INT3_G64 && mat_bytes % rbB))) return false;
    for (int m = 0; m < NM; m++) {
        if (!encode_rows_map(&src.tm[3 * m], w[m], total / rb, rb, 512, R, false)) return false;
        if (FMT == FMT_INT3_G64 && !encode_rows_map(&src.tm[3 * m + 1], w[m], total / rbB, rbB, 256, R, false))
            return false;
        // ue8m0 scale rows are moved as 4-byte elements: only bytes count
        if (SK != SK_ROW &&
            !encode_rows_map(&src.tm[3 * m + 2], sc[m], E * O, sb, src.tile.sbox, R, SK == SK_F32))
            return false;
    }
    src.row_mul[0] = mat_bytes / rb;
    src.row_add[0] = 0;
    src.row_mul[1] = FMT == FMT_INT3_G64 ? mat_bytes / rbB : 0;
    src.row_add[1] = FMT == FMT_INT3_G64 ? 2 * O : 0;    // plane B follows O rows of plane A (2 O rows of I/8)
    src.row_mul[2] = O;
    src.row_add[2] = 0;
    return true;
}

template <int NM, int S, class Job>
static cudaError_t launch_tile(const Job& job, int grid, cudaStream_t st)
{
    auto kern = k_tile<NM, S, Job>;
    static int granted[64];
    cudaError_t e = set_smem(kern, (size_t)job.tile.total, granted);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kTileThreads), (size_t)job.tile.total, st, job);
}

#include "qg_row.cuh"

#include "qg_moe.cuh"

// Whether the automatic choice takes the row-team kernel for one activation row.
#ifndef QG_ROW_AUTO
#define QG_ROW_AUTO 0
#endif

template <int NM, int S>
static cudaError_t launch_dense(const DenseJob<NM>& job_in, int grid, size_t x_bytes, cudaStream_t st)
{
    DenseJob<NM> job = job_in;
    if constexpr (S == 1) {
        // the row-team kernel wherever its plan fits (one activation row, rows of whole warp steps)
        const int pol = kernel_policy();
        if ((QG_ROW_AUTO && pol == QKERNEL_AUTO) || pol == QKERNEL_ROW) {
            bool launched = false;
            const cudaError_t e = launch_row_dense<NM, S>(job, grid, st, launched);
            if (launched) return e;
        }
    }
    constexpr int R = tile_rows_per<S, NM>();
    const int I = job.m[0].I;
    const int gs = SK == SK_ROW ? I : I / job.m[0].ngrp;
    const void* w[NM];
    const float* sc[NM];
    for (int k = 0; k < NM; k++) {
        w[k] = job.m[k].w;
        sc[k] = job.m[k].sc;
    }
    const long long O = job.m[0].O;
    const long long mat_bytes = FMT == FMT_INT3_G64 ? O * (I / 4) + O * (I / 8) : O * code_row_bytes(I);
    // Measured on GB300: with one activation row and one scale per lane the
    // int8/int4/MXFP4 rows are cheap to decode and the per-lane copy kernel is
    // a little faster; int3, several activation rows, and -- on matrices with
    // enough rows per CTA for full tiles -- scales shared by several lanes
    // (rows, ue8m0 words, long groups) go to the tile kernel.
    const int policy = kernel_policy();
    const bool short_matrix = (O + grid - 1) / grid < (long long)kWarps * rows_per_tile<1, NM>();
    const bool shares = (kShareAlways || (kShareMaybe && job.m[0].gsh > 0)) && !short_matrix;
    const bool prefer_tile =
        policy == QKERNEL_TILE || (policy == QKERNEL_AUTO && (S > 1 || FMT == FMT_INT3_G64 || shares));
    if (prefer_tile && plan_tile(NM, R, I, gs, S, job.tile) &&
        tile_sources<NM>(job, w, sc, 1, O, I, gs, mat_bytes, R))
        return launch_tile<NM, S>(job, grid, st);
    return with_share(job.m[0].gsh, [&](auto sh) -> cudaError_t {
        constexpr bool SH = decltype(sh)::value;
        if constexpr (S == 1) {
            // fewer rows per CTA than warps x tile height: single-row tiles keep more warps busy
            if (short_matrix) {
                auto kern1 = k_stream<NM, 1, DenseJob<NM>, 1, SH>;
                job.ring_stride = kRing * ring_slot_bytes<FMT, NM>();
                const size_t smem1 = x_bytes + (size_t)kWarps * job.ring_stride;
                static int granted1[64];
                cudaError_t e = set_smem(kern1, smem1, granted1);
                if (e != cudaSuccess) return e;
                return launch_pdl(kern1, dim3(grid), dim3(kThreads), smem1, st, job);
            }
        }
        auto kern = k_stream<NM, S, DenseJob<NM>, 0, SH>;
        const size_t smem = x_bytes + (size_t)kWarps * job.ring_stride;
        static int granted[64];
        cudaError_t e = set_smem(kern, smem, granted);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, job);
    });
}

template <int NM>
static cudaError_t launch_dense_s(const DenseJob<NM>& job, int s, int grid, size_t x_bytes, cudaStream_t st)
{
    switch (s) {
    case 1: return launch_dense<NM, 1>(job, grid, x_bytes, st);
    case 2: return launch_dense<NM, 2>(job, grid, x_bytes, st);
    case 3: return launch_dense<NM, 3>(job, grid, x_bytes, st);
    case 4: return launch_dense<NM, 4>(job, grid, x_bytes, st);
    case 5: return launch_dense<NM, 5>(job, grid, x_bytes, st);
    case 6: return launch_dense<NM, 6>(job, grid, x_bytes, st);
    case 7: return launch_dense<NM, 7>(job, grid, x_bytes, st);
    case 8: return launch_dense<NM, 8>(job, grid, x_bytes, st);
    default: return cudaErrorInvalidValue;
    }
}

#include "qg_gemm.cuh"

}  // namespace fmt_<name>

using namespace QG_CAT(fmt_, QG_NAME);

cudaError_t QG_CAT(gemv_, QG_NAME)(const HostMat& hm, const float* x, int s, float* y, long long ldy, int grid,
                                   cudaStream_t st)
{
    DenseJob<1> job;
    job.act = QACT_SWIGLU;
    job.limit = 0.0f;
    job.m[0] = to_mat(hm);
    job.x = x;
    job.y = y;
    job.ldy = ldy;
    job.S = s;
    job.ring_off = (int)align16((size_t)s * hm.I * sizeof(float));
    job.ring_stride = ring_stride_bytes<1>();
    return launch_dense_s<1>(job, s, grid, job.ring_off, st);
}

cudaError_t QG_CAT(gate_up_, QG_NAME)(const HostMat& g, const HostMat& u, const float* x, int s, float* h,
                                      long long ldh, int act, float limit, int grid, cudaStream_t st)
{
    DenseJob<2> job;
    job.act = act;
    job.limit = limit;
    job.m[0] = to_mat(g);
    job.m[1] = to_mat(u);
    job.x = x;
    job.y = h;
    job.ldy = ldh;
    job.S = s;
    job.ring_off = (int)align16((size_t)s * g.I * sizeof(float));
    job.ring_stride = ring_stride_bytes<2>();
    return launch_dense_s<2>(job, s, grid, job.ring_off, st);
}

cudaError_t QG_CAT(expert_up_, QG_NAME)(const ExpertArgs& a, int grid, cudaStream_t st)
{
    const WsLayout L = ws_layout(a.D, a.F, a.s, a.k);
    const int gs = SK == SK_ROW ? a.D : a.gs;
    ExpertUpJob job;
    job.gate0 = to_mat(HostMat{a.gate, a.gate_s, a.F, a.D, gs});
    job.up0 = to_mat(HostMat{a.up, a.up_s, a.F, a.D, gs});
    job.mat_bytes = FMT == FMT_INT8_ROW ? (long long)a.F * a.D
                  : FMT == FMT_INT3_G64 ? (long long)a.F * a.D / 4 + (long long)a.F * a.D / 8
                                        : (long long)a.F * a.D / 2;
    job.mat_scales = (long long)a.F * (a.D / gs);
    job.x = a.x;
    job.hdr = reinterpret_cast<const int32_t*>(a.ws + L.hdr);
    job.batches = reinterpret_cast<const int4*>(a.ws + L.batches);
    job.pair_tok = reinterpret_cast<const int32_t*>(a.ws + L.pair_tok);
    job.h = reinterpret_cast<float*>(a.ws + L.h);
    job.bounds = reinterpret_cast<const int32_t*>(a.ws + L.bounds);
    job.act = a.act;
    job.limit = a.limit;
    job.D = a.D;
    job.F = a.F;
    job.ring_off = (int)align16((size_t)a.smax * a.D * sizeof(float));
    job.ring_stride = ring_stride_bytes<2, 1>();
    job.status = a.status_dev;
    {
        const void* w[2] = {a.gate, a.up};
        const float* sc[2] = {a.gate_s, a.up_s};
        constexpr int R = tile_rows_per<1, 2>();
        if (kernel_policy() != QKERNEL_RING && (long long)a.s * a.k * ((a.F + R - 1) / R) < (1ll << 31) &&
            plan_tile(2, R, a.D, gs, a.smax, job.tile) &&
            tile_sources<2>(job, w, sc, a.E, a.F, a.D, gs, job.mat_bytes, R))
        {
            if (a.smax <= 1) return launch_tile<2, 1>(job, grid, st);
            if (a.smax <= 2) return launch_tile<2, 2>(job, grid, st);
            return launch_tile<2, kExpertSmax>(job, grid, st);
        }
    }
    return with_share(job.gate0.gsh, [&](auto sh) -> cudaError_t {
        auto kern = k_stream<2, kExpertSmax, ExpertUpJob, 0, decltype(sh)::value>;
        const size_t smem = job.ring_off + (size_t)kWarps * job.ring_stride;
        static int granted[64];
        cudaError_t e = set_smem(kern, smem, granted);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, job);
    });
}

cudaError_t QG_CAT(expert_down_, QG_NAME)(const ExpertArgs& a, int grid, cudaStream_t st)
{
    const WsLayout L = ws_layout(a.D, a.F, a.s, a.k);
    const int gs = SK == SK_ROW ? a.F : a.gs;
    ExpertDownJob job;
    job.down0 = to_mat(HostMat{a.down, a.down_s, a.D, a.F, gs});
    job.mat_bytes = FMT == FMT_INT8_ROW ? (long long)a.D * a.F
                  : FMT == FMT_INT3_G64 ? (long long)a.D * a.F / 4 + (long long)a.D * a.F / 8
                                        : (long long)a.D * a.F / 2;
    job.mat_scales = (long long)a.D * (a.F / gs);
    job.hdr = reinterpret_cast<const int32_t*>(a.ws + L.hdr);
    job.batches = reinterpret_cast<const int4*>(a.ws + L.batches);
    job.h = reinterpret_cast<const float*>(a.ws + L.h);
    job.z = reinterpret_cast<float*>(a.ws + L.z);
    job.bounds = reinterpret_cast<const int32_t*>(a.ws + L.bounds) + (kMaxGrid + 1);
    job.D = a.D;
    job.F = a.F;
    job.ring_off = (int)align16((size_t)a.smax * a.F * sizeof(float));
    job.ring_stride = ring_stride_bytes<1, 1>();
    job.status = a.status_dev;
    {
        const void* w[1] = {a.down};
        const float* sc[1] = {a.down_s};
        constexpr int R = tile_rows_per<1, 1>();
        if (kernel_policy() != QKERNEL_RING && (long long)a.s * a.k * ((a.D + R - 1) / R) < (1ll << 31) &&
            plan_tile(1, R, a.F, gs, a.smax, job.tile) &&
            tile_sources<1>(job, w, sc, a.E, a.D, a.F, gs, job.mat_bytes, R))
        {
            if (a.smax <= 1) return launch_tile<1, 1>(job, grid, st);
            if (a.smax <= 2) return launch_tile<1, 2>(job, grid, st);
            return launch_tile<1, kExpertSmax>(job, grid, st);
        }
    }
    return with_share(job.down0.gsh, [&](auto sh) -> cudaError_t {
        auto kern = k_stream<1, kExpertSmax, ExpertDownJob, 0, decltype(sh)::value>;
        const size_t smem = job.ring_off + (size_t)kWarps * job.ring_stride;
        static int granted[64];
        cudaError_t e = set_smem(kern, smem, granted);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, job);
    });
}

cudaError_t QG_CAT(expert_fused_, QG_NAME)(const ExpertArgs& a, int grid, cudaStream_t st, bool* launched, bool dry)
{
    *launched = false;
    const int gs_up = SK == SK_ROW ? a.D : a.gs, gs_dn = SK == SK_ROW ? a.F : a.gs;
    MoeJob job;
    job.gate0 = to_mat(HostMat{a.gate, a.gate_s, a.F, a.D, gs_up});
    job.up0 = to_mat(HostMat{a.up, a.up_s, a.F, a.D, gs_up});
    job.down0 = to_mat(HostMat{a.down, a.down_s, a.D, a.F, gs_dn});
    if (!plan_moe(a.D, a.F, gs_up, gs_dn, a.smax, job)) return cudaSuccess;
    const long long D = a.D, F = a.F;
    job.up_bytes = FMT == FMT_INT8_ROW ? F * D : FMT == FMT_INT3_G64 ? F * D / 4 + F * D / 8 : F * D / 2;
    job.dn_bytes = FMT == FMT_INT8_ROW ? D * F : FMT == FMT_INT3_G64 ? D * F / 4 + D * F / 8 : D * F / 2;
    job.up_scales = F * (D / gs_up);
    job.dn_scales = D * (F / gs_dn);
    {
        constexpr int RA = TilePhase<2, 1, MoeUpView>::R;
        constexpr int RB = TilePhase<1, 1, MoeDownView>::R;
        TileSource<2> sa;
        TileSource<1> sb;
        sa.tile = job.la;
        sb.tile = job.lb;
        const void* wa[2] = {a.gate, a.up};
        const float* sca[2] = {a.gate_s, a.up_s};
        const void* wb[1] = {a.down};
        const float* scb[1] = {a.down_s};
        if ((long long)a.s * a.k * ((F + RA - 1) / RA) >= (1ll << 31) ||
            (long long)a.s * a.k * ((D + RB - 1) / RB) >= (1ll << 31))
            return cudaSuccess;
        if (dry) {                                 // the plan only: it would launch
            *launched = true;
            return cudaSuccess;
        }
        if (!tile_sources<2>(sa, wa, sca, a.E, a.F, a.D, gs_up, job.up_bytes, RA) ||
            !tile_sources<1>(sb, wb, scb, a.E, a.D, a.F, gs_dn, job.dn_bytes, RB))
            return cudaSuccess;
        for (int i = 0; i < 6; i++) job.tma[i] = sa.tm[i];
        for (int i = 0; i < 3; i++) job.tmb[i] = sb.tm[i];
        for (int p = 0; p < 3; p++) {
            job.rmA[p] = sa.row_mul[p];
            job.raA[p] = sa.row_add[p];
            job.rmB[p] = sb.row_mul[p];
            job.raB[p] = sb.row_add[p];
        }
    }
    const WsLayout L = ws_layout(a.D, a.F, a.s, a.k);
    job.x = a.x;
    job.ids = a.ids;
    job.wts = a.wts;
    // a routed call passes its routing outputs as ids / wts (the caller's writable buffers)
    job.ids_out = a.route_kind >= 0 ? const_cast<int32_t*>(a.ids) : nullptr;
    job.wts_out = a.route_kind >= 0 ? const_cast<float*>(a.wts) : nullptr;
    job.out = a.out;
    job.h = reinterpret_cast<float*>(a.ws + L.h);
    job.z = reinterpret_cast<float*>(a.ws + L.z);
    job.ctr = reinterpret_cast<unsigned*>(a.ws + L.hdr) + 4;
    job.done = reinterpret_cast<unsigned*>(a.ws + L.done);
    job.status = a.status_dev;
    job.E = a.E;
    job.D = a.D;
    job.F = a.F;
    job.s = a.s;
    job.k = a.k;
    job.P = a.s * a.k;
    job.smax = a.smax;
    job.act = a.act;
    job.limit = a.limit;
    job.wait_ns = a.wait_ns;
    job.withhold = a.withhold;
    job.route_kind = a.route_kind;
    job.logits = a.logits;
    job.bias = a.bias;
    job.renorm = a.renorm;
    job.route_scale = a.route_scale;
    *launched = true;
    return launch_moe(job, grid, st);
}

int QG_CAT(device_error_, QG_NAME)(int clear)
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(int)) != cudaSuccess) return QSTATUS_LAUNCH;
    if (clear && v) {
        const int zero = 0;
        cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(int));
    }
    return v;
}

int QG_CAT(tile_rows_, QG_NAME)(int nm)
{
    return nm == 2 ? tile_rows_per<1, 2>() : tile_rows_per<1, 1>();
}

size_t QG_CAT(ring_bytes_, QG_NAME)(int nm)
{
    return (size_t)kWarps * (nm == 2 ? ring_stride_bytes<2>() : ring_stride_bytes<1>());
}

cudaError_t QG_CAT(gemm_, QG_NAME)(const HostMat& hm, const GemmArgs& g, cudaStream_t st)
{
    switch (gemm_bn(g.s)) {
    case 32: return launch_gemm<32>(hm, g, st);
    case 64: return launch_gemm<64>(hm, g, st);
    default: return launch_gemm<128>(hm, g, st);
    }
}

cudaError_t QG_CAT(dequant_, QG_NAME)(const HostMat& hm, float* out, cudaStream_t st)
{
    const Mat m = to_mat(hm);
    const long long total = hm.O * (long long)(hm.I / EPL);
    long long blocks = (total + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    k_dequant<<<(int)blocks, 256, 0, st>>>(m, out);
    return cudaGetLastError();
}

}  // namespace qg
