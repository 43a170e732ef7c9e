// qg_gemm.cuh -- the prefill GEMM of one weight format on the tensor cores
// (included by qg_fmt_impl.cuh inside the format's namespace).
//
// y[n][o] = sum_i value(W[o][i]) * scale[o][i/gs] * x[n][i] for many
// activation rows n, the tiled GEMM with which colibri's docs/vulkan.md (the
// tiled-GEMM and cooperative-matrix paragraph) replaces the per-row GEMV from
// two rows on, built for the fifth-generation tensor cores:
//  * weight codes decode exactly to f16 (int8, int4, int3, e2m1 are small
//    integers or e2m1 values), so nothing of W is rounded;
//  * x is split into two f16 parts whose sum holds 22 of its 24 significand
//    bits, after scaling each activation row by a power of two (a separate
//    launch writes the parts to the workspace), and the MMA runs on both;
//  * every group of gs inputs (at most 128 at a time for longer groups and
//    per-row scales) sums into a fresh f32 partial in tensor memory, which the
//    threads read back and add to their running sums times the group scale --
//    the blocked summation the pages' GEMM uses to keep the GEMV's error.
//
// A CTA owns a tile of 128 weight rows x BN activation rows.  Per K step of 64
// inputs: every thread decodes its weight row's 64 codes into f16 (shared
// memory, the tensor cores' 128-byte swizzled K-major layout), one thread
// issues the MMAs (A = the decoded slab, B = the x parts, copied by the tensor
// copy engine with the same swizzle), and the threads fold the partials of the
// previous step into their sums while the tensor cores work.  The weight rows
// stream through a ring of per-thread asynchronous copies several steps deep.
#pragma once

namespace gemm {

constexpr int kBM = 128;       // weight rows per tile (tensor-memory lanes)
constexpr int kBK = 64;        // inputs per K step (one 128-byte row of f16)
constexpr int kFoldWarps = 8;     // fold partials: warp w reads tensor-memory lanes 32 (w % 4).., columns half w / 4
constexpr int kDecodeWarps = 4;   // decode the weights: one thread per weight row
constexpr int kThreads = 32 * (kFoldWarps + kDecodeWarps + 1);   // + one warp issuing tensor copies and MMAs
// 16-byte raw cells per row per K step: int8 64 B; int4 / e2m1 32 B; int3
// 16 B of plane A and 8 B of plane B.
constexpr int kCells = FMT == FMT_INT8_ROW ? 4 : 2;
constexpr uint32_t kABytes = kBM * 128;
constexpr uint32_t kRawBytes = kCells * kBM * 16;

// Shared memory of a CTA: two decoded weight slabs, kBStages x-part slots,
// kRawStages raw weight and scale slots -- as deep as 227 KB allows, since
// the copies have to run several K steps ahead of their use.
template <int BN>
struct Layout {
    static constexpr uint32_t kBBytes = 2 * BN * 128;     // x high part, then low part
    static constexpr int kBStages = BN == 128 ? 4 : 6;
    static constexpr uint32_t kFixed = 2 * kABytes + kBStages * kBBytes + 4 * kBM * 8 + 8 * (kBStages + 10) + 16 + 1024;
    static constexpr int kRawStages = kFixed + 8 * (kRawBytes + kBM * 8) <= 225 * 1024 ? 8 : 6;
    static constexpr uint32_t kA = 0;
    static constexpr uint32_t kB = kA + 2 * kABytes;
    static constexpr uint32_t kRaw = kB + kBStages * kBBytes;
    static constexpr uint32_t kScl = kRaw + kRawStages * kRawBytes;   // per step and row: 8 bytes of scales
    static constexpr uint32_t kPScale = kScl + kRawStages * kBM * 8;   // 4 steps x rows: the folding scales
    static constexpr uint32_t kBar = kPScale + 4 * kBM * 8;             // kBStages + 2 + 2 + 4 + 2 barriers
    static constexpr uint32_t kTmemSlot = kBar + 8 * (kBStages + 10);   // tensor-memory address, abort flag
    static constexpr uint32_t kBytes = kTmemSlot + 16 + 1024;          // + alignment of the base
};

}  // namespace gemm

// The job of one prefill GEMM launch.
struct GemmJob {
    CUtensorMap xh, xl;        // x parts, f16 [s][I], boxes of 64 inputs x BN rows, 128-byte swizzle
    Mat m;                     // the weights
    const int32_t* pexp;       // x row n was scaled by 2^pexp[n]
    float* y;                  // [s][O]
    int s;                     // activation rows
    int ntn;                   // activation-row tiles
    int pbl;                   // log2 of the inputs per partial (32, 64 or 128)
    int gsl;                   // log2 of the group size (grouped formats)
};

// Decodes the raw codes of one weight row's K step (cells at `raw`, `cstride`
// bytes apart) into eight 16-byte chunks of f16 in stored order: int8 and
// e2m1 in input order; int4 as (0,4,1,5,2,6,3,7) per 8 inputs and int3 as
// (0,8,1,9,...,7,15) per 16 (the x parts are written in the same order).
__device__ __forceinline__ void gemm_decode_step(uint32_t raw, uint32_t cstride, uint4 (&out)[8])
{
    constexpr uint32_t kMag = 0x64006400u;            // f16 1024 in both halves
    if constexpr (FMT == FMT_INT8_ROW) {
        constexpr uint32_t kSub = 0x64806480u;        // 1024 + 128
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint4 v = lds16(raw + c * cstride);
            const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint32_t a = w[2 * h], b = w[2 * h + 1];
                out[2 * c + h] = make_uint4(hsub2_u32(__byte_perm(a, 0x64646464u, 0x4140u), kSub),
                                            hsub2_u32(__byte_perm(a, 0x64646464u, 0x4342u), kSub),
                                            hsub2_u32(__byte_perm(b, 0x64646464u, 0x4140u), kSub),
                                            hsub2_u32(__byte_perm(b, 0x64646464u, 0x4342u), kSub));
            }
        }
    } else if constexpr (FMT == FMT_INT4_G) {
        constexpr uint32_t kSub = 0x64086408u;        // 1024 + 8
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const uint4 v = lds16(raw + c * cstride);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; q++)
                out[4 * c + q] = make_uint4(hsub2_u32(lop3_and_or(w[q], 0x000F000Fu, kMag), kSub),
                                            hsub2_u32(lop3_and_or(w[q] >> 4, 0x000F000Fu, kMag), kSub),
                                            hsub2_u32(lop3_and_or(w[q] >> 8, 0x000F000Fu, kMag), kSub),
                                            hsub2_u32(lop3_and_or(w[q] >> 12, 0x000F000Fu, kMag), kSub));
        }
    } else if constexpr (FMT == FMT_MXFP4_G32) {
#pragma unroll
        for (int c = 0; c < 2; c++) {
            const uint4 v = lds16(raw + c * cstride);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; q++)
                out[4 * c + q] = make_uint4(e2m1x2_to_h2(w[q]), e2m1x2_to_h2(w[q] >> 8), e2m1x2_to_h2(w[q] >> 16),
                                            e2m1x2_to_h2(w[q] >> 24));
        }
    } else {   // int3-g64: cell 0 = 16 B of plane A, cell 1 = 8 B of plane B
        constexpr uint32_t kSub = 0x64046404u;        // 1024 + 4
        const uint4 a = lds16(raw);
        const uint2 b = lds8(raw + cstride);
        const uint32_t A[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            uint32_t ce, co;
            const uint32_t B = (q >> 1) ? b.y : b.x;
            if (q & 1) int3_nibbles<0x4342u>(A[q], B, ce, co);
            else int3_nibbles<0x4140u>(A[q], B, ce, co);
            out[2 * q] = make_uint4(hsub2_u32(lop3_and_or(ce, 0x000F000Fu, kMag), kSub),
                                    hsub2_u32(lop3_and_or(co, 0x000F000Fu, kMag), kSub),
                                    hsub2_u32(lop3_and_or(ce >> 4, 0x000F000Fu, kMag), kSub),
                                    hsub2_u32(lop3_and_or(co >> 4, 0x000F000Fu, kMag), kSub));
            out[2 * q + 1] = make_uint4(hsub2_u32(lop3_and_or(ce >> 8, 0x000F000Fu, kMag), kSub),
                                        hsub2_u32(lop3_and_or(co >> 8, 0x000F000Fu, kMag), kSub),
                                        hsub2_u32(lop3_and_or(ce >> 12, 0x000F000Fu, kMag), kSub),
                                        hsub2_u32(lop3_and_or(co >> 12, 0x000F000Fu, kMag), kSub));
        }
    }
}

// Blocks (partials of 2^pbl inputs) that end inside K step t of T: n of
// them, the first with index b0 (a 128-input block ends early at the row's
// end when I is an odd multiple of 64).
__device__ __forceinline__ void gemm_blocks_ending(int t, int T, int pbl, int& n, int& b0)
{
    if (pbl <= 6) {
        n = gemm::kBK >> pbl;
        b0 = (t * gemm::kBK) >> pbl;
    } else {
        const int end = (t + 1) * gemm::kBK;
        n = ((end & ((1 << pbl) - 1)) == 0 || t == T - 1) ? 1 : 0;
        b0 = (t * gemm::kBK) >> pbl;
    }
}

template <int BN>
__global__ void __launch_bounds__(gemm::kThreads, 1) k_gemm(const __grid_constant__ GemmJob job)
{
    using L = gemm::Layout<BN>;
    constexpr int HN = BN / 2;                         // partial columns per folding thread
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x / job.ntn, nt = blockIdx.x - mt * job.ntn;
    const long long O = job.m.O;
    const long long o0 = (long long)mt * gemm::kBM;
    const int n0 = nt * BN;
    const int T = job.m.I / gemm::kBK;
    const int pbl = job.pbl;
    const int nbuf = pbl == 5 ? 4 : 2;                 // partial buffers in tensor memory
    const uint32_t ncols = (uint32_t)(nbuf * BN);

    // 1024-byte aligned base for the swizzled tiles
    const uint32_t sbase = smem_base();
    const uint32_t off0 = ((sbase + 1023u) & ~1023u) - sbase;
    const uint32_t oA = off0 + L::kA, oB = off0 + L::kB, oRaw = off0 + L::kRaw, oScl = off0 + L::kScl;
    const uint32_t oPs = off0 + L::kPScale;
    const uint32_t bfull = sbase + off0 + L::kBar;     // kBStages: x parts landed (tensor copies)
    const uint32_t afull = bfull + 8 * L::kBStages;     // 2: decoded weight slab written (decode warps)
    const uint32_t sdone = afull + 16;                  // 2: the MMAs of a step completed (commit)
    const uint32_t sfull = sdone + 16;                  // 4: a step's folding scales written (decode warps)
    const uint32_t tfree = sfull + 32;                  // 2: a step's partials read (folding warps)
    const uint32_t tslot = sbase + off0 + L::kTmemSlot;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(reinterpret_cast<char*>(qg_smem4) + off0 +
                                                               L::kTmemSlot + 4);

    if (warp == 0) tmem_alloc(tslot, ncols);
    if (tid == 0) {
        for (int i = 0; i < L::kBStages; i++) mbar_init(bfull + 8 * i, 1);
        for (int i = 0; i < 2; i++) mbar_init(afull + 8 * i, gemm::kDecodeWarps);
        for (int i = 0; i < 2; i++) mbar_init(sdone + 8 * i, 1);
        for (int i = 0; i < 4; i++) mbar_init(sfull + 8 * i, gemm::kDecodeWarps);
        for (int i = 0; i < 2; i++) mbar_init(tfree + 8 * i, gemm::kFoldWarps);
        *abort_flag = 0;
        mbar_init_fence();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = lds_u32(off0 + L::kTmemSlot);
    bool failed_here = false;

    if (warp >= gemm::kFoldWarps + gemm::kDecodeWarps) {
        // ---- issue warp, one thread: tensor copies of the x parts, the MMAs ----
        if (lane == 0) {
            auto issue_x = [&](int u) {
                const uint32_t slot = u % L::kBStages;
                const uint32_t bar = bfull + 8 * slot;
                const uint32_t dst = sbase + oB + slot * L::kBBytes;
                mbar_expect_tx(bar, L::kBBytes);
                tma_load_2d(dst, &job.xh, u * gemm::kBK, n0, bar);
                tma_load_2d(dst + BN * 128, &job.xl, u * gemm::kBK, n0, bar);
            };
            int issued_x = L::kBStages < T ? L::kBStages : T;
            for (int u = 0; u < issued_x; u++) issue_x(u);
            constexpr uint32_t idesc = tc_idesc_f16(gemm::kBM, BN);
            int t = 0;
            for (; t < T; t++) {
                if (*abort_flag) break;
                // the slab is decoded, the partial buffers of step t - 2 were read, x landed
                if (!mbar_wait(afull + 8 * (t & 1), (uint32_t)(t >> 1) & 1u) ||
                    (t >= 2 && !mbar_wait(tfree + 8 * (t & 1), (uint32_t)((t - 2) >> 1) & 1u)) ||
                    !mbar_wait(bfull + 8 * (t % L::kBStages), (uint32_t)(t / L::kBStages) & 1u)) {
                    failed_here = true;
                    break;
                }
                tc_fence_after();
                // descriptors of the step's slabs; a K step of 16 inputs is 32
                // bytes further along the rows (+2 in the address field)
                const uint64_t da = tc_desc_sw128(sbase + oA + (t & 1) * gemm::kABytes);
                const uint64_t dh = tc_desc_sw128(sbase + oB + (uint32_t)(t % L::kBStages) * L::kBBytes);
                const uint64_t dl = dh + (uint64_t)((BN * 128) >> 4);
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const int k = t * gemm::kBK + 16 * j;
                    const uint32_t d = tmem + (uint32_t)(((k >> pbl) % nbuf) * BN);
                    const uint32_t first = (k & ((1 << pbl) - 1)) == 0;
                    tc_mma_f16(d, da + 2 * j, dh + 2 * j, idesc, first ? 0u : 1u);
                    tc_mma_f16(d, da + 2 * j, dl + 2 * j, idesc, 1u);
                }
                tc_commit(sdone + 8 * (t & 1));
                // the x slot of step t - 1 is free once its MMAs are done: refill it
                if (t >= 1 && issued_x < T) {
                    if (!mbar_wait(sdone + 8 * ((t - 1) & 1), (uint32_t)((t - 1) >> 1) & 1u)) {
                        failed_here = true;
                        t++;
                        break;
                    }
                    issue_x(issued_x++);
                }
            }
            if (failed_here) {
                *abort_flag = 1;
                // leave no copy or MMA in flight: wait (bounded) for what was issued
                if (t > 0) mbar_wait(sdone + 8 * ((t - 1) & 1), (uint32_t)((t - 1) >> 1) & 1u);
                for (int u = t; u < issued_x; u++)
                    mbar_wait(bfull + 8 * (u % L::kBStages), (uint32_t)(u / L::kBStages) & 1u);
            }
        }
    } else if (warp >= gemm::kFoldWarps) {
        // ---- decode warps: weight row m; raw copies, scales, the f16 slab ----
        const int m = (warp - gemm::kFoldWarps) * 32 + lane;
        const long long o = o0 + m;
        const long long o_ld = o < O ? o : O - 1;      // rows past the end repeat the last one
        const long long srow = o_ld * job.m.ngrp;      // first scale of the row
        float row_scale = 0.f;
        if constexpr (SK == SK_ROW) row_scale = ldg_f32(job.m.sc + o_ld);
        const uint8_t* wrow;
        const uint8_t* brow = nullptr;
        if constexpr (FMT == FMT_INT8_ROW) wrow = job.m.w + o_ld * job.m.I;
        else if constexpr (FMT == FMT_INT3_G64) {
            wrow = job.m.w + o_ld * (long long)(job.m.I / 4);
            brow = job.m.w + O * (long long)(job.m.I / 4) + o_ld * (long long)(job.m.I / 8);
        } else wrow = job.m.w + o_ld * (long long)(job.m.I / 2);
        // raw weight copies of K step u into its slot, with the row's scales of
        // the step (one commit group per step)
        auto issue_raw = [&](int u) {
            if (u < T) {
                const uint32_t dst = sbase + oRaw + (uint32_t)(u % L::kRawStages) * gemm::kRawBytes + m * 16;
                if constexpr (FMT == FMT_INT8_ROW) {
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        cp_async16(dst + c * gemm::kBM * 16, wrow + (long long)u * 64 + c * 16);
                } else if constexpr (FMT == FMT_INT3_G64) {
                    cp_async16(dst, wrow + (long long)u * 16);
                    cp_async8(dst + gemm::kBM * 16, brow + (long long)u * 8);
                } else {
#pragma unroll
                    for (int c = 0; c < 2; c++)
                        cp_async16(dst + c * gemm::kBM * 16, wrow + (long long)u * 32 + c * 16);
                }
                if constexpr (SK != SK_ROW) {
                    const uint32_t sdst = sbase + oScl + (uint32_t)(u % L::kRawStages) * (gemm::kBM * 8) + m * 8;
                    if constexpr (SK == SK_E8M0) {
                        // groups 2u, 2u + 1: bytes of the aligned word that holds them
                        cp_async4(sdst, reinterpret_cast<const uint8_t*>(job.m.sc) + ((srow + 2ll * u) & ~3ll));
                    } else if (pbl == 5) {
                        cp_async4(sdst, job.m.sc + srow + 2ll * u);           // groups 2u, 2u + 1
                        cp_async4(sdst + 4, job.m.sc + srow + 2ll * u + 1);   // (scales are 4-byte aligned)
                    } else {
                        // the group of the step's (first) block
                        cp_async4(sdst, job.m.sc + srow + (((long long)u * gemm::kBK) >> job.gsl));
                    }
                }
            }
            cp_async_commit();
        };
        for (int u = 0; u < L::kRawStages - 1; u++) issue_raw(u);
        for (int t = 0; t < T; t++) {
            if (*abort_flag) break;
            // A slot t % 2 is free once the MMAs of step t - 2 completed (that
            // also bounds how far decoding runs ahead of the folding warps)
            if (t >= 2 && !mbar_wait(sdone + 8 * (t & 1), (uint32_t)((t - 2) >> 1) & 1u)) {
                failed_here = true;
                break;
            }
            cp_async_wait<L::kRawStages - 2>();
            // the scales of the blocks ending in step t, for the folding warps
            float sc0, sc1;
            if constexpr (SK == SK_ROW) {
                sc0 = sc1 = row_scale;
            } else {
                const uint32_t so = oScl + (uint32_t)(t % L::kRawStages) * (gemm::kBM * 8) + m * 8;
                if constexpr (SK == SK_E8M0) {
                    const uint32_t wd = lds_u32(so), sh = (uint32_t)((2 * t) & 3);
                    sc0 = e8m0_to_f32(__byte_perm(wd, 0u, 0x4440u + sh));
                    sc1 = e8m0_to_f32(__byte_perm(wd, 0u, 0x4440u + sh + 1));
                } else if (pbl == 5) {
                    const uint2 v = lds8(so);
                    sc0 = __uint_as_float(v.x);
                    sc1 = __uint_as_float(v.y);
                } else {
                    sc0 = sc1 = lds_f32(so);
                }
            }
            *reinterpret_cast<float2*>(reinterpret_cast<char*>(qg_smem4) + oPs + (t & 3) * (gemm::kBM * 8) + m * 8) =
                make_float2(sc0, sc1);
            {
                uint4 ch[8];
                gemm_decode_step(oRaw + (uint32_t)(t % L::kRawStages) * gemm::kRawBytes + m * 16, gemm::kBM * 16, ch);
                char* arow = reinterpret_cast<char*>(qg_smem4) + oA + (t & 1) * gemm::kABytes + (m >> 3) * 1024 +
                             (m & 7) * 128;
#pragma unroll
                for (int j = 0; j < 8; j++) *reinterpret_cast<uint4*>(arow + ((j ^ (m & 7)) << 4)) = ch[j];
            }
            issue_raw(t + L::kRawStages - 1);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(afull + 8 * (t & 1));
                mbar_arrive(sfull + 8 * (t & 3));
            }
        }
        if (failed_here) *abort_flag = 1;
        cp_async_wait<0>();
    } else {
        // ---- folding warps: lanes 32 q.. of tensor memory, column half hh ----
        const int q = warp & 3, hh = warp >> 2;
        const int m = q * 32 + lane;                   // weight row of this thread
        const long long o = o0 + m;
        float acc[HN];                                 // columns hh * HN .. hh * HN + HN - 1
#pragma unroll
        for (int n = 0; n < HN; n++) acc[n] = 0.f;
        // folds this thread's columns of the partial of block b (weight scale
        // sc) into its sums
        auto promote = [&](int b, float sc) {
            const uint32_t col = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((b % nbuf) * BN + hh * HN);
            if constexpr (HN == 16) {
                float v[16];
                tmem_ld16(col, v);
#pragma unroll
                for (int i = 0; i < 16; i++) acc[i] = fmaf(sc, v[i], acc[i]);
            } else {
#pragma unroll
                for (int c = 0; c < HN / 32; c++) {
                    float v[32];
                    tmem_ld32(col + 32 * c, v);
#pragma unroll
                    for (int i = 0; i < 32; i++) acc[32 * c + i] = fmaf(sc, v[i], acc[32 * c + i]);
                }
            }
        };
        int t = 0;
        for (; t < T; t++) {
            if (*abort_flag) break;
            if (!mbar_wait(sdone + 8 * (t & 1), (uint32_t)(t >> 1) & 1u) ||
                !mbar_wait(sfull + 8 * (t & 3), (uint32_t)(t >> 2) & 1u)) {
                failed_here = true;
                break;
            }
            tc_fence_after();
            int nend, bend;
            gemm_blocks_ending(t, T, pbl, nend, bend);
            const float2 sc = *reinterpret_cast<const float2*>(reinterpret_cast<const char*>(qg_smem4) + oPs +
                                                                (t & 3) * (gemm::kBM * 8) + m * 8);
            if (nend > 0) promote(bend, sc.x);
            if (nend > 1) promote(bend + 1, sc.y);
            tc_fence_before();         // the partial reads precede the arrival
            __syncwarp();
            if (lane == 0) mbar_arrive(tfree + 8 * (t & 1));
        }
        if (failed_here) *abort_flag = 1;
        // y[n][o] = sum * 2^-pexp[n]
        if (!failed_here && t == T && o < O) {
#pragma unroll
            for (int i = 0; i < HN; i++) {
                const int n = n0 + hh * HN + i;
                if (n < job.s) {
                    const int p = job.pexp[n];
                    job.y[(long long)n * O + o] = acc[i] * __uint_as_float((uint32_t)(127 - p) << 23);
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0 && *abort_flag) tile_fail(nullptr);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

template <int BN>
static cudaError_t launch_gemm(const HostMat& hm, const GemmArgs& g, cudaStream_t st)
{
    GemmJob job;
    job.m = to_mat(hm);
    if (!encode_x_map(&job.xh, g.xh, g.sp, hm.I, BN) || !encode_x_map(&job.xl, g.xl, g.sp, hm.I, BN))
        return cudaErrorInvalidValue;
    job.pexp = g.pexp;
    job.y = g.y;
    job.s = g.s;
    job.ntn = g.sp / BN;
    int gsl = 0;
    while ((1 << gsl) < hm.gs) gsl++;
    job.gsl = gsl;
    job.pbl = SK == SK_ROW ? 7 : (gsl < 7 ? gsl : 7);
    const long long mtiles = (hm.O + gemm::kBM - 1) / gemm::kBM;
    const long long grid = mtiles * job.ntn;
    if (grid > 0x7FFFFFFFll) return cudaErrorInvalidValue;
    auto kern = k_gemm<BN>;
    static int granted[64];
    cudaError_t e = set_smem(kern, gemm::Layout<BN>::kBytes, granted);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, gemm::kThreads, gemm::Layout<BN>::kBytes, st>>>(job);
    return cudaGetLastError();
}
