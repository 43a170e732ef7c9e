// qg_route.cuh -- one token's routing by one warp (the router kernel and the
// expert prep kernel's fused routing).
//
// colibri keeps this step on the host (docs/vulkan.md, the per-engine host
// steps: a softmax followed by a top-k for most models; for the sigmoid
// routers, sigmoid scores whose top-k is picked with a correction bias and
// then renormalized).  The warp holds
// the token's E logits in registers (J per lane, E <= 32 J) and runs k rounds
// of a warp argmax:
//   softmax:        key = logit (exp is increasing, so the k largest logits
//                   are the k largest probabilities); weight = softmax
//                   probability, over all E or renormalized over the k chosen;
//   sigmoid + bias: key = sigmoid(logit) + bias; weight = sigmoid(logit),
//                   renormalized over the k chosen if asked;
// every weight times `scale`.  Ranks run in decreasing key, equal keys lower
// expert index first; a NaN key ranks below every number.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qgemv.h"

namespace qg {

constexpr int kRouteMaxE = 1024;
constexpr int kRouteMaxK = 32;

// Routes token row l (E logits) with the calling warp; lane r < k returns
// rank r's expert in id and its weight in w (other lanes: undefined).
template <int J>
__device__ __forceinline__ void route_token(int kind, const float* __restrict__ l, const float* __restrict__ bias,
                                            int E, int k, int renorm, float scale, int lane, int& id, float& w)
{
    float lg[J], key[J];
    uint32_t taken = 0;                // bit j: expert lane + 32 j chosen
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < J; j++) {
        const int e = lane + 32 * j;
        lg[j] = e < E ? l[e] : -INFINITY;
        float kv = lg[j];
        if (kind == QROUTE_SIGMOID_BIAS && e < E) kv = 1.0f / (1.0f + expf(-lg[j])) + bias[e];
        key[j] = (e < E && kv == kv) ? kv : -INFINITY;     // NaN ranks last
        if (e >= E) taken |= 1u << j;                        // not an expert
        mx = fmaxf(mx, lg[j]);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));

    int my_id = 0;                     // lane r < k: the expert of rank r
    float my_logit = 0.f;
    for (int r = 0; r < k; r++) {
        // this lane's best untaken expert
        float bk = 0.f;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < J; j++) {
            if (!(taken >> j & 1u) && (be == 0x7FFFFFFF || key[j] > bk)) {
                bk = key[j];
                be = lane + 32 * j;
            }
        }
        // the warp's: larger key, then lower index
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, d);
            const int oe = __shfl_xor_sync(0xffffffffu, be, d);
            const bool other = oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ok > bk || (ok == bk && oe < be));
            if (other) {
                bk = ok;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        // its logit, from the owning lane
        float vl = 0.f;
#pragma unroll
        for (int j = 0; j < J; j++)
            if (lane + 32 * j == be) vl = lg[j];
        vl = __shfl_sync(0xffffffffu, vl, be & 31);
        if (lane == r) {
            my_id = be;
            my_logit = vl;
        }
    }
    // weights
    float wv = 0.f;
    if (kind == QROUTE_SOFTMAX) {
        wv = lane < k ? expf(my_logit - mx) : 0.f;
        float denom = 0.f;
        if (renorm) {
            denom = wv;
        } else {
#pragma unroll
            for (int j = 0; j < J; j++)
                if (lane + 32 * j < E) denom += expf(lg[j] - mx);
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, d);
        wv = scale * (wv / denom);
    } else {
        wv = lane < k ? 1.0f / (1.0f + expf(-my_logit)) : 0.f;
        float denom = wv;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, d);
        wv = scale * (renorm ? wv / denom : wv);
    }
    id = my_id;
    w = wv;
}

}  // namespace qg
