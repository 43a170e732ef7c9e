// qg_gemm_x.cu -- the activation side of the prefill GEMM.
//
// colibri's docs/vulkan.md (the cooperative-matrix paragraph) keeps the GEMM
// exact to f32 level by scaling each activation row by a power of two and
// splitting it into an f16 high part (the top 11 significand bits) and an f16
// low part, the MMA running on both.  Here one CTA per activation row finds
// the row's largest magnitude, picks p with max|x| * 2^p in [2^14, 2^15) (the
// high part never overflows f16), and writes hi = f16(x * 2^p) and
// lo = f16(x * 2^p - hi) -- the subtraction is exact in f32 -- in the order
// the weight decoder produces inputs, plus p.  Rows past s are zero.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qg_internal.h"

namespace qg {

__global__ void __launch_bounds__(256) k_gemm_split_x(const float* __restrict__ x, int s, int I, int perm,
                                                      __half* __restrict__ xh, __half* __restrict__ xl,
                                                      int32_t* __restrict__ pexp)
{
    const int n = blockIdx.x;
    __half* hrow = xh + (long long)n * I;
    __half* lrow = xl + (long long)n * I;
    if (n >= s) {                       // padding rows
        for (int j = threadIdx.x; j < I; j += blockDim.x) {
            hrow[j] = __float2half_rn(0.f);
            lrow[j] = __float2half_rn(0.f);
        }
        if (threadIdx.x == 0) pexp[n] = 0;
        return;
    }
    const float* xr = x + (long long)n * I;
    float amax = 0.f;
    for (int i = threadIdx.x; i < I; i += blockDim.x) amax = fmaxf(amax, fabsf(xr[i]));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); w++) amax = fmaxf(amax, red[w]);
    // amax in [2^(e-127), 2^(e-126)) for biased exponent e: p = 141 - e puts
    // it in [2^14, 2^15); zero, non-finite or subnormal maxima take p = 0 or
    // the clamp
    const uint32_t e = (__float_as_uint(amax) >> 23) & 0xFFu;
    int p = (amax == 0.f || e == 255u) ? 0 : (e == 0u ? 100 : 141 - (int)e);
    p = p < -100 ? -100 : (p > 100 ? 100 : p);
    const float scale = __uint_as_float((uint32_t)(127 + p) << 23);
    const int half = perm >> 1;
    for (int j = threadIdx.x; j < I; j += blockDim.x) {
        int i = j;
        if (perm) {                     // stored position 2q holds input q, 2q + 1 holds q + perm/2
            const int q = j & (perm - 1);
            i = (j - q) + ((q & 1) ? (q >> 1) + half : (q >> 1));
        }
        const float v = xr[i] * scale;
        const __half h = __float2half_rn(v);
        hrow[j] = h;
        lrow[j] = __float2half_rn(v - __half2float(h));
    }
    if (threadIdx.x == 0) pexp[n] = p;
}

cudaError_t gemm_split_x(const float* x, int s, int sp, int I, int perm, void* xh, void* xl, int32_t* pexp,
                         cudaStream_t st)
{
    k_gemm_split_x<<<sp, 256, 0, st>>>(x, s, I, perm, static_cast<__half*>(xh), static_cast<__half*>(xl), pexp);
    return cudaGetLastError();
}

}  // namespace qg
