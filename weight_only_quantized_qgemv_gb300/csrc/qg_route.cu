// qg_route.cu -- the router on the device: per token, the top k of E experts
// and their weights from the router logits (one warp per token; the routing
// itself is route_token in qg_route.cuh).
#include <cuda_runtime.h>

#include "qg_internal.h"
#include "qg_route.cuh"

namespace qg {

__global__ void __launch_bounds__(256) k_route(int kind, const float* __restrict__ logits,
                                               const float* __restrict__ bias, int s, int E, int k, int renorm,
                                               float scale, int32_t* __restrict__ ids, float* __restrict__ wts)
{
    pdl_allow_next();
    pdl_wait_prev();                   // the logits may come from the kernel before
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= s) return;
    int id;
    float w;
    route_token<kRouteMaxE / 32>(kind, logits + (long long)t * E, bias, E, k, renorm, scale, lane, id, w);
    if (lane < k) {
        ids[(long long)t * k + lane] = id;
        wts[(long long)t * k + lane] = w;
    }
}

cudaError_t route_launch(int kind, const float* logits, const float* bias, int s, int E, int k, int renorm,
                         float scale, int32_t* ids, float* wts, cudaStream_t st)
{
    const int tokens_per_block = 8;
    const int grid = (s + tokens_per_block - 1) / tokens_per_block;
    return launch_pdl(k_route, dim3(grid), dim3(32 * tokens_per_block), 0, st, kind, logits, bias, s, E, k,
                      renorm, scale, ids, wts);
}

}  // namespace qg
