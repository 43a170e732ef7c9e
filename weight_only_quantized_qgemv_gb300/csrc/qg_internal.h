// qg_internal.h -- host-side declarations shared by the library's translation
// units: launch functions per format and the expert-group workspace layout.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "qgemv.h"

namespace qg {

#ifndef QG_WARPS
#define QG_WARPS 16
#endif
constexpr int kWarps = QG_WARPS;            // warps per CTA of the streaming kernels
constexpr int kThreads = kWarps * 32;
#ifndef QG_BULK_CONSUMERS
#define QG_BULK_CONSUMERS 16
#endif
constexpr int kBulkConsumers = QG_BULK_CONSUMERS;   // consumer warps of the bulk-copy kernels
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
//   hdr      int32[8]     [0] status, [1] batches, [2] pairs
//   batches  int4[P]      (expert, first sorted pair, pairs in batch, 0)
//   pair_tok int32[P]     token of the sorted pair
//   pair_of  int32[P]     sorted position of pair t * k + r
//   h        f32[P][F]    silu(gate x) * (up x) of each sorted pair
//   z        f32[P][D]    down h of each sorted pair
struct WsLayout {
    size_t hdr, batches, pair_tok, pair_of, h, z, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

inline WsLayout ws_layout(int D, int F, int s, int k)
{
    const size_t P = (size_t)s * (size_t)k;
    WsLayout L;
    size_t off = 0;
    L.hdr = off;      off = align256(off + 8 * sizeof(int32_t));
    L.batches = off;  off = align256(off + P * 4 * sizeof(int32_t));
    L.pair_tok = off; off = align256(off + P * sizeof(int32_t));
    L.pair_of = off;  off = align256(off + P * sizeof(int32_t));
    L.h = off;        off = align256(off + P * (size_t)F * sizeof(float));
    L.z = off;        off = align256(off + P * (size_t)D * sizeof(float));
    L.total = off;
    return L;
}

struct ExpertArgs {
    int gs;
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
};

// Shared-memory plan of a bulk-copy launch (byte offsets from the start of
// dynamic shared memory; the activation rows sit at offset 0).
struct BulkLayout {
    int rs;            // rows per stage
    int nstage;        // stages in the ring
    int kp;            // work units per row tile (K parts)
    int kpw;           // warp steps per work unit
    int stage_off, stage_bytes, part_off, cnt_off, bar_off, total;
    int w_off[2], b_off[2], s_off[2];   // per matrix, inside a stage
    int rb, rbB, sb;   // bytes per row: codes (int3: plane A), int3 plane B, scales (0: read from global)
};

// Per-format launchers (defined in qg_fmt_<format>.cu).  Each returns a
// cudaError_t of the launch.
#define QG_DECLARE_FMT(name)                                                                            \
    cudaError_t gemv_##name(const HostMat& m, const float* x, int s, float* y, long long ldy,          \
                            int grid, cudaStream_t st);                                                \
    cudaError_t gate_up_##name(const HostMat& g, const HostMat& u, const float* x, int s, float* h,    \
                               long long ldh, int grid, cudaStream_t st);                              \
    cudaError_t expert_up_##name(const ExpertArgs& a, int grid, cudaStream_t st);                       \
    cudaError_t expert_down_##name(const ExpertArgs& a, int grid, cudaStream_t st);                     \
    cudaError_t dequant_##name(const HostMat& m, float* out, cudaStream_t st);                         \
    size_t ring_bytes_##name(int nm);                                                                 \
    int device_error_##name(int clear);

QG_DECLARE_FMT(int8)
QG_DECLARE_FMT(int4)
QG_DECLARE_FMT(int3)
QG_DECLARE_FMT(mxfp4)

#undef QG_DECLARE_FMT

// Format-independent expert kernels (qg_abi.cu).
cudaError_t expert_prep(const ExpertArgs& a, cudaStream_t st);
cudaError_t expert_combine(const ExpertArgs& a, cudaStream_t st);

}  // namespace qg
