// qg_internal.h -- host-side declarations shared by the library's translation
// units: launch functions per format and the expert-group workspace layout.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>            // CUtensorMap (the encoder is looked up at run time)
#include <cuda_runtime.h>

#include "qgemv.h"

namespace qg {

#ifndef QG_WARPS
#define QG_WARPS 16
#endif
constexpr int kWarps = QG_WARPS;            // warps per CTA of the streaming kernels
constexpr int kThreads = kWarps * 32;
#ifndef QG_TILE_WARPS
#define QG_TILE_WARPS 16
#endif
constexpr int kTileWarps = QG_TILE_WARPS;   // warps per CTA of the tile kernel
constexpr int kTileThreads = kTileWarps * 32;
constexpr int kSmax = 8;                    // activation rows per dense launch
constexpr int kExpertSmax = 4;              // (token, rank) pairs per expert batch
constexpr int kSmemMax = 227 * 1024;        // dynamic shared memory per CTA (sm_103a)
constexpr int kMaxPairs = 4096;             // s * k limit of qexpert_group

// Description of one packed matrix for the host launchers.
struct HostMat {
    const void* w;
    const float* sc;
    long long O;
    int I;
    int gs;       // resolved group size (int8: I)
};

// Workspace of qexpert_group (all offsets 256-byte aligned):
//   hdr      int32[8]     [0] status, [1] batches, [2] pairs (four-launch path);
//                         [4..7] the one-launch path's counters (zero between calls)
//   done     int32[kDoneWords]  one-launch path: phase-A row tiles finished per batch (zero between calls)
//   batches  int4[P]      (expert, first sorted pair, pairs in batch, 0)
//   pair_tok int32[P]     token of the sorted pair
//   pair_of  int32[P]     sorted position of pair t * k + r
//   bounds   int32[2][kMaxGrid + 1]  first row tile of each CTA (gate/up, down)
//   h        f32[P][F]    silu(gate x) * (up x) of each sorted pair
//   z        f32[P][D]    down h of each sorted pair
constexpr int kMaxGrid = 1024;              // CTAs of an expert launch
constexpr int kDoneWords = 256;             // per-batch counters of the one-launch path (its batches at most)
struct WsLayout {
    size_t hdr, done, batches, pair_tok, pair_of, bounds, h, z, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

inline WsLayout ws_layout(int D, int F, int s, int k)
{
    const size_t P = (size_t)s * (size_t)k;
    WsLayout L;
    size_t off = 0;
    L.hdr = off;      off = align256(off + 8 * sizeof(int32_t));
    L.done = off;     off = align256(off + kDoneWords * sizeof(int32_t));
    L.batches = off;  off = align256(off + P * 4 * sizeof(int32_t));
    L.pair_tok = off; off = align256(off + P * sizeof(int32_t));
    L.pair_of = off;  off = align256(off + P * sizeof(int32_t));
    L.bounds = off;   off = align256(off + 2 * (kMaxGrid + 1) * sizeof(int32_t));
    L.h = off;        off = align256(off + P * (size_t)F * sizeof(float));
    L.z = off;        off = align256(off + P * (size_t)D * sizeof(float));
    L.total = off;
    return L;
}

struct ExpertArgs {
    int gs;
    int act;           // QACT_* of the gate/up product
    float limit;       // its limit (QACT_SWIGLU_CLAMPED)
    const void *gate, *up, *down;
    const float *gate_s, *up_s, *down_s;
    int E, D, F, s, k;
    const float* x;
    const int32_t* ids;
    const float* wts;
    float* out;
    unsigned char* ws;
    int32_t* status_dev;
    int smax;          // pairs per batch
    int grid;               // CTAs of the streaming launches (<= kMaxGrid)
    int tpb_up, tpb_down;   // row tiles per batch of the tile kernel's two phases
    // routing fused into the prep kernel (route_kind >= 0, E <= kFusedRouteMaxE):
    // ids / wts above are then its outputs
    int route_kind = -1;
    const float* logits = nullptr;
    const float* bias = nullptr;
    int renorm = 0;
    float route_scale = 1.0f;
    // the fused launch: bound of its device waits, and the test hook that
    // withholds one CTA's phase-A signal
    unsigned long long wait_ns = 2000000000ull;
    int withhold = 0;
};

// Pairs (s * k) up to which qexpert_group runs as one fused launch.
constexpr int kFusedMaxPairs = 256;

constexpr int kFusedRouteMaxE = 256;   // experts the prep kernel's fused routing holds (8 per lane)

// Shared-memory plan of a tile-streaming launch (byte offsets from the start
// of dynamic shared memory).  The activation rows sit at offset 0, zero-padded
// to whole slices; then one ring of P slots per warp; then the mbarriers.
// A slot holds one slice (32 lanes x EPL inputs) of R rows of every matrix:
// their codes (512 B per row), int3 plane B (256 B per row) and scales
// (sbox bytes per row).
struct TileLayout {
    int P;             // slots per warp ring
    int slot_bytes;    // slot stride
    int tx_bytes;      // bytes the tensor copies of one slot deliver
    int ring_off;      // first ring
    int warp_bytes;    // ring stride from one warp to the next (>= P * slot_bytes)
    int bar_off;       // P full barriers per warp, then the CTA barrier
    int total;         // dynamic shared memory of the launch
    int nslices;       // slices per row
    int xstride;       // floats per staged activation row (nslices * slice)
    int sbox;          // scale bytes per row per slice
    int code_off[2], b_off[2], s_off[2];   // per matrix, inside a slot
};

// Tensor map over `rows` rows of `row_bytes` bytes (a multiple of 16) at
// `base` (16-byte aligned), read in boxes of `box_rows` rows x `box_bytes`
// bytes (a multiple of 16, at most 1024): 32-bit elements, no swizzle,
// out-of-range elements read as zero.  False when the driver refuses it.
bool encode_rows_map(CUtensorMap* map, const void* base, long long rows, long long row_bytes, int box_bytes,
                     int box_rows, bool f32);

// The prefill GEMM's activations (workspace of qgemm): x rows scaled by 2^pexp
// and split into f16 high and low parts, rows padded with zeros to a whole
// number of activation-row tiles.
struct GemmArgs {
    const void* xh;           // f16 [sp][I]
    const void* xl;           // f16 [sp][I]
    const int32_t* pexp;      // [sp]
    int s;                    // activation rows (y has s rows)
    int sp;                   // padded rows
    float* y;                 // [s][O]
};

// Activation rows per tile of the prefill GEMM for s rows, and the padded row
// count of its workspace.
inline int gemm_bn(int s) { return s <= 32 ? 32 : (s <= 64 ? 64 : 128); }
inline int gemm_rows(int s) { const int bn = gemm_bn(s); return (s + bn - 1) / bn * bn; }

struct GemmWs {
    size_t xh, xl, pexp, total;
};
inline GemmWs gemm_ws_layout(int I, int s)
{
    const size_t sp = (size_t)gemm_rows(s);
    GemmWs L;
    size_t off = 0;
    L.xh = off;   off = align256(off + sp * (size_t)I * 2);
    L.xl = off;   off = align256(off + sp * (size_t)I * 2);
    L.pexp = off; off = align256(off + sp * sizeof(int32_t));
    L.total = off;
    return L;
}

// Tensor map over an f16 [rows][cols] matrix (cols a multiple of 64) read in
// boxes of 64 columns x box_rows rows with the 128-byte swizzle.
bool encode_x_map(CUtensorMap* map, const void* base, long long rows, long long cols, int box_rows);

// Writes the prefill GEMM's activation parts (qg_gemm_x.cu); perm is the
// weight decoder's input order inside blocks of perm inputs (0: in order).
cudaError_t gemm_split_x(const float* x, int s, int sp, int I, int perm, void* xh, void* xl, int32_t* pexp,
                         cudaStream_t st);

// The router kernel (qg_route.cu).
cudaError_t route_launch(int kind, const float* logits, const float* bias, int s, int E, int k, int renorm,
                         float scale, int32_t* ids, float* wts, cudaStream_t st);

// Per-format launchers (defined in qg_fmt_<format>.cu).  Each returns a
// cudaError_t of the launch.
#define QG_DECLARE_FMT(name)                                                                            \
    cudaError_t gemv_##name(const HostMat& m, const float* x, int s, float* y, long long ldy,          \
                            int grid, cudaStream_t st);                                                \
    cudaError_t gate_up_##name(const HostMat& g, const HostMat& u, const float* x, int s, float* h,    \
                               long long ldh, int act, float limit, int grid, cudaStream_t st);        \
    cudaError_t expert_up_##name(const ExpertArgs& a, int grid, cudaStream_t st);                       \
    cudaError_t expert_down_##name(const ExpertArgs& a, int grid, cudaStream_t st);                     \
    cudaError_t expert_fused_##name(const ExpertArgs& a, int grid, cudaStream_t st, bool* launched,    \
                                   bool dry);                                                      \
    cudaError_t dequant_##name(const HostMat& m, float* out, cudaStream_t st);                         \
    cudaError_t gemm_##name(const HostMat& m, const GemmArgs& g, cudaStream_t st);                     \
    size_t ring_bytes_##name(int nm);                                                                 \
    int tile_rows_##name(int nm);                                                                     \
    int device_error_##name(int clear);

QG_DECLARE_FMT(int8)
QG_DECLARE_FMT(int8g)
QG_DECLARE_FMT(int4r)
QG_DECLARE_FMT(int4)
QG_DECLARE_FMT(int3)
QG_DECLARE_FMT(mxfp4)
QG_DECLARE_FMT(mxfp4e)

#undef QG_DECLARE_FMT

// The process's QKERNEL_* policy (qg_abi.cu).
int kernel_policy();

// Launches allowing programmatic dependent launch: the kernel may start while
// the previous kernel in the stream finishes, if that one lets it (each of
// this library's kernels does, early); the kernel itself waits for the
// previous one before it touches anything the previous one may write.
#ifndef QG_PDL
#define QG_PDL 1
#endif
// Device side: let the next kernel in the stream start (it waits for this one
// before touching what this one writes), and wait for the previous kernel to
// complete with its memory visible.
__device__ __forceinline__ void pdl_allow_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prev() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = QG_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Format-independent expert kernels (qg_abi.cu).
cudaError_t expert_prep(const ExpertArgs& a, cudaStream_t st);
cudaError_t expert_combine(const ExpertArgs& a, cudaStream_t st);

}  // namespace qg
