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
    // blocks of 16 inputs per thread (I is a multiple of 64): four 16-byte
    // loads, two 16-byte stores per part
    const int n = blockIdx.x;
    uint4* hrow = reinterpret_cast<uint4*>(xh + (long long)n * I);
    uint4* lrow = reinterpret_cast<uint4*>(xl + (long long)n * I);
    const int nblk = I / 16;
    if (n >= s) {                       // padding rows
        for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
            hrow[2 * b] = hrow[2 * b + 1] = make_uint4(0, 0, 0, 0);
            lrow[2 * b] = lrow[2 * b + 1] = make_uint4(0, 0, 0, 0);
        }
        if (threadIdx.x == 0) pexp[n] = 0;
        return;
    }
    const float4* xr = reinterpret_cast<const float4*>(x + (long long)n * I);
    float amax = 0.f;
    for (int i = threadIdx.x; i < I / 4; i += blockDim.x) {
        const float4 v = xr[i];
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    __shared__ float red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); w++) amax = fmaxf(amax, red[w]);
    // amax in [2^(e-127), 2^(e-126)) for biased exponent e: p = 141 - e puts
    // it in [2^14, 2^15); zero, non-finite or subnormal maxima take p = 0 or
    // the clamp.  p stays in [-126, 126], where 2^p and 2^-p are both normal
    // f32: every finite row fits (FLT_MAX takes p = -113); rows below 2^-112
    // are scaled below 2^14, where the split's error is still at most 2^-22 of
    // each element plus 2^-25 absolute (2^-151 in x's units).
    const uint32_t e = (__float_as_uint(amax) >> 23) & 0xFFu;
    int p = (amax == 0.f || e == 255u) ? 0 : (e == 0u ? 126 : 141 - (int)e);
    p = p < -126 ? -126 : (p > 126 ? 126 : p);
    const float scale = __uint_as_float((uint32_t)(127 + p) << 23);
    for (int b = threadIdx.x; b < nblk; b += blockDim.x) {
        float v[16];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const float4 f = xr[4 * b + q];
            v[4 * q] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
        // stored position j holds input src(j): in order, or within blocks of
        // perm inputs position 2q holds q and 2q + 1 holds q + perm / 2
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            int s0 = j, s1 = j + 1;
            if (perm == 8) {
                const int base = j & ~7, q = (j & 7) >> 1;
                s0 = base + q;
                s1 = base + q + 4;
            } else if (perm == 16) {
                const int q = j >> 1;
                s0 = q;
                s1 = q + 8;
            }
            const float a0 = v[s0] * scale, a1 = v[s1] * scale;
            const __half h0 = __float2half_rn(a0), h1 = __float2half_rn(a1);
            const __half l0 = __float2half_rn(a0 - __half2float(h0)), l1 = __float2half_rn(a1 - __half2float(h1));
            hw[j >> 1] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
            lw[j >> 1] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
        }
        hrow[2 * b] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        hrow[2 * b + 1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        lrow[2 * b] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        lrow[2 * b + 1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
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
