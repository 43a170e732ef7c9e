// qg_device.cuh -- device code shared by the quantized GEMV, the fused gate/up
// and the routed-expert kernels (sm_103a).
//
// What is computed (colibri Vulkan guide, xdnf.cn, section 着色器层面的实现细节,
// and its API section): y[s][o] = sum_i value(code[o][i]) * scale[o][i/gs] * x[s][i]
// for int8 per row, int4 (nibble - 8), int3-g64 in two bit planes (code - 4)
// and MXFP4 e2m1 nibbles, with f32 group scales.
//
// How (GB300-first):
//  * One lane owns one 16-byte "chunk" of a row per step (int3: 16 B of plane A
//    plus 8 B of plane B), loaded with 128-bit non-caching loads: a warp step
//    reads 512 contiguous bytes of a row, fully coalesced.  int4, MXFP4 and
//    int3 chunks are exactly one scale group, so a lane needs one scale per
//    chunk.
//  * x (or the expert hidden vectors) sits in shared memory once per CTA in a
//    swizzled order: lane l's x segment is 64-256 contiguous bytes, so plain
//    placement would make the 8 lanes of a 128-bit shared-memory wavefront hit
//    the same banks; XOR-ing the 16-byte quad index with low bits of the chunk
//    index spreads them over all 32 banks.
//  * Codes become f32 without integer-to-float conversions: a code OR-ed into
//    the mantissa of 2^23 is the float 2^23 + code (shifted left by 4k bits,
//    2^23 + code * 16^k), and one subtraction of 2^23 + offset * 16^k gives
//    (code - offset) * 16^k exactly.  Sums of each power-of-16 class go to
//    their own accumulator and are rescaled (exactly) at the end of the chunk.
//    MXFP4 uses the hardware e2m1x2 -> f16x2 conversion.
//  * Packed f32x2 FMA/ADD halve the issue slots of the arithmetic.
//  * Each warp streams R rows at a time through a P-deep ring of chunk
//    registers, so P*R 16-byte loads per lane are in flight; finished row
//    tiles are reduced across the warp with a transposed (reduce-scatter)
//    butterfly, one shuffle per value instead of five.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qg {

enum : int {
    FMT_INT8_ROW = 1, FMT_INT4_ROW = 2, FMT_INT4_G = 4, FMT_INT3_G64 = 5, FMT_MXFP4_G32 = 7, FMT_MXFP4_E8M0 = 8,
    FMT_INT8_G = 13
};

// A format is a code decoding (int8, int4, int3 or e2m1: the first four ids
// above) and a scale kind: one f32 per row, f32 per group, or one ue8m0 byte
// per group of 32.
enum : int { SK_ROW = 0, SK_F32 = 1, SK_E8M0 = 2 };
__host__ __device__ constexpr int decode_of(int f)
{
    return f == FMT_INT8_G ? FMT_INT8_ROW
         : f == FMT_INT4_ROW ? FMT_INT4_G
         : f == FMT_MXFP4_E8M0 ? FMT_MXFP4_G32 : f;
}
__host__ __device__ constexpr int scale_kind_of(int f)
{
    return (f == FMT_INT8_ROW || f == FMT_INT4_ROW) ? SK_ROW : (f == FMT_MXFP4_E8M0 ? SK_E8M0 : SK_F32);
}

// Elements a lane decodes per chunk.
template <int FMT> struct Traits;
template <> struct Traits<FMT_INT8_ROW>  { static constexpr int EPL = 16; };
template <> struct Traits<FMT_INT4_G>    { static constexpr int EPL = 32; };
template <> struct Traits<FMT_INT3_G64>  { static constexpr int EPL = 64; };
template <> struct Traits<FMT_MXFP4_G32> { static constexpr int EPL = 32; };

// ---------------------------------------------------------------------------
// Swizzled placement of an activation vector in shared memory.
// Element i lives in chunk q = i / EPL, quad j = (i % EPL) / 4.  The quad is
// stored at (j ^ swz(q)) inside the chunk's segment.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int x_swz(int EPL, int q) { return EPL == 16 ? ((q >> 1) & 3) : (q & 7); }

// Physical float4 index of logical quad qd (= i / 4).
__device__ __forceinline__ int x_quad_phys(int EPL, int qd)
{
    const int qpc = EPL / 4;       // quads per chunk
    const int q = qd / qpc;
    const int j = qd - q * qpc;
    return q * qpc + (j ^ x_swz(EPL, q));
}

// ---------------------------------------------------------------------------
// Packed f32x2 helpers (sm_100+ PTX).
// ---------------------------------------------------------------------------
#ifndef QG_F32X2_BUILTIN
#define QG_F32X2_BUILTIN 0
#endif
#if QG_F32X2_BUILTIN
// The compiler's own packed builtins: it sees the pairs and places them.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }
#else
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
#endif

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// ---------------------------------------------------------------------------
// Global loads of streamed weights: read once, keep out of L1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_stream16(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg_stream8(const void* p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ float ldg_f32(const float* p)
{
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// A weight matrix as the kernels see it.
// ---------------------------------------------------------------------------
struct Mat {
    const uint8_t* w;      // packed codes (int3: plane A, then plane B)
    const float* sc;       // scales [O][I/gs] (ue8m0: bytes, addressed through sc_ptr)
    long long O;           // rows
    int I;                 // inputs per row
    int ngrp;              // scale groups per row (I/gs; per-row formats: 1)
    int gsh;               // chunk -> group shift: log2(gs / inputs per chunk); per-row formats: 0
};

// Scale element n of a scale array: f32 elements, or bytes for ue8m0.
template <int SK>
__host__ __device__ __forceinline__ const float* sc_ptr(const float* base, long long n)
{
    if constexpr (SK == SK_E8M0) return reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(base) + n);
    else return base + n;
}

// ue8m0 byte -> f32: 2^(e - 127) is the byte in the exponent field; byte 0 is
// the subnormal 2^-127 and byte 255 NaN (both get mantissa bit 22).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e)
{
    return __uint_as_float((e << 23) | ((e == 0u || e == 255u) ? 0x00400000u : 0u));
}

template <int FMT> struct Chunk { uint4 w; };
template <> struct Chunk<FMT_INT3_G64> { uint4 a; uint2 b; };

// One chunk of row o and its scale, straight from global memory (the
// dequantization kernel).  QF is the full format.
template <int QF>
__device__ __forceinline__ void load_chunk(const Mat& m, long long o, int q, Chunk<decode_of(QF)>& c, float& sc)
{
    constexpr int FMT = decode_of(QF), SK = scale_kind_of(QF);
    if constexpr (FMT == FMT_INT8_ROW) {
        c.w = ldg_stream16(m.w + o * m.I + (long long)q * 16);
    } else if constexpr (FMT == FMT_INT3_G64) {
        const long long rowA = (long long)(m.I / 4), rowB = (long long)(m.I / 8);
        c.a = ldg_stream16(m.w + o * rowA + (long long)q * 16);
        c.b = ldg_stream8(m.w + m.O * rowA + o * rowB + (long long)q * 8);
    } else {
        c.w = ldg_stream16(m.w + o * (long long)(m.I / 2) + (long long)q * 16);
    }
    const long long n = o * m.ngrp + (SK == SK_ROW ? 0 : (q >> m.gsh));
    if constexpr (SK == SK_E8M0) sc = e8m0_to_f32(reinterpret_cast<const uint8_t*>(m.sc)[n]);
    else sc = ldg_f32(m.sc + n);
}

#ifndef QG_INT3_SPREAD
#define QG_INT3_SPREAD 1
#endif

#ifndef QG_CXX_LDS
#define QG_CXX_LDS 1
#endif

// The kernels' dynamic shared memory; every shared address below is a byte
// offset from its start.
extern __shared__ float4 qg_smem4[];

__device__ __forceinline__ uint32_t smem_base() { return (uint32_t)__cvta_generic_to_shared(qg_smem4); }

// Loads from shared memory at byte offset a.  Plain loads let the compiler
// schedule them; the cp.async waits (memory clobbers) still order them.
__device__ __forceinline__ float4 lds4s(uint32_t a)
{
#if QG_CXX_LDS
    return *reinterpret_cast<const float4*>(reinterpret_cast<const char*>(qg_smem4) + a);
#else
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a + smem_base()));
    return v;
#endif
}

// (a & MASK) | c in one logic instruction.
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}

// ---------------------------------------------------------------------------
// Decoding.  A code c OR-ed into the mantissa of a float whose exponent is
// chosen for the code's bit position gives 2^e + c exactly; subtracting
// 2^e + offset gives c - offset.  int4 nibble k of a 16-bit half sits at bits
// 4k..4k+3, so its float is ((150 - 4k) << 23) | (w & (0xF << 4k)) =
// 2^(23-4k) + c.  Bytes (int8, int3 codes gathered into bytes) are moved under
// 2^23 with one byte permute.
// ---------------------------------------------------------------------------
constexpr uint32_t kMag0 = 0x4B000000u;   // 2^23, code at bits 0..
constexpr uint32_t kMag1 = 0x49000000u;   // 2^19, code at bits 4..
constexpr uint32_t kMag2 = 0x47000000u;   // 2^15, code at bits 8..
constexpr uint32_t kMag3 = 0x45000000u;   // 2^11, code at bits 12..

// int4 word (elements 8j..8j+7: low nibble first) -> four value pairs.
// mg[k] holds the exponent for nibble position k of a 16-bit half.
struct Int4Magic {
    uint32_t m0, m1, m2, m3;
    float2 b01, b23;
    __device__ __forceinline__ Int4Magic()
        : m0(kMag0), m1(kMag1), m2(kMag2), m3(kMag3),
          b01(make_float2(-8388616.0f, -524296.0f)),   // -(2^23 + 8), -(2^19 + 8)
          b23(make_float2(-32776.0f, -2056.0f)) {}     // -(2^15 + 8), -(2^11 + 8)
};

__device__ __forceinline__ void decode_int4_word(uint32_t v, const Int4Magic& g, float2 (&d)[4])
{
    const uint32_t h = v >> 16;
    d[0] = fadd2(make_float2(u2f(and_or<0x000Fu>(v, g.m0)), u2f(and_or<0x00F0u>(v, g.m1))), g.b01);
    d[1] = fadd2(make_float2(u2f(and_or<0x0F00u>(v, g.m2)), u2f(and_or<0xF000u>(v, g.m3))), g.b23);
    d[2] = fadd2(make_float2(u2f(and_or<0x000Fu>(h, g.m0)), u2f(and_or<0x00F0u>(h, g.m1))), g.b01);
    d[3] = fadd2(make_float2(u2f(and_or<0x0F00u>(h, g.m2)), u2f(and_or<0xF000u>(h, g.m3))), g.b23);
}

// int8 word (elements 4j..4j+3) -> two value pairs.  b ^ 0x80 = b + 128.
__device__ __forceinline__ void decode_int8_word(uint32_t v, float2 (&d)[2])
{
    const float2 B = make_float2(-8388736.0f, -8388736.0f);    // -(2^23 + 128)
    v ^= 0x80808080u;
    d[0] = fadd2(make_float2(u2f(__byte_perm(v, kMag0, 0x7440)), u2f(__byte_perm(v, kMag0, 0x7441))), B);
    d[1] = fadd2(make_float2(u2f(__byte_perm(v, kMag0, 0x7442)), u2f(__byte_perm(v, kMag0, 0x7443))), B);
}

// MXFP4: one byte = two e2m1 codes (low nibble first) -> f32 pair, through the
// hardware e2m1x2 -> f16x2 conversion.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte_in_low_bits)
{
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\t.reg .b16 u;\n\tcvt.u16.u32 u, %1;\n\tcvt.u8.u16 t, u;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2) : "r"(byte_in_low_bits));
    float lo, hi;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(h2));
    return make_float2(lo, hi);
}

__device__ __forceinline__ void decode_mxfp4_word(uint32_t v, float2 (&d)[4])
{
    d[0] = e2m1x2_to_f32x2(v);
    d[1] = e2m1x2_to_f32x2(v >> 8);
    d[2] = e2m1x2_to_f32x2(v >> 16);
    d[3] = e2m1x2_to_f32x2(v >> 24);
}

// int3-g64: plane A word j holds the low two bits of elements 16j..16j+15
// (two bits each, least significant first); the matching 16 bits of plane B
// hold their high bits.  Elements 16j + 4m + r are gathered per class r into
// byte m of word c[r] as a clean 3-bit code.
__device__ __forceinline__ void int3_classes(uint32_t A, uint32_t bhalf, uint32_t (&c)[4])
{
    uint32_t t = bhalf & 0xFFFFu;
    t = (t | (t << 8)) & 0x00FF00FFu;       // nibble m -> byte m
    t = (t | (t << 4)) & 0x0F0F0F0Fu;
    c[0] = (A & 0x03030303u) | ((t << 2) & 0x04040404u);
    c[1] = ((A >> 2) & 0x03030303u) | ((t << 1) & 0x04040404u);
    c[2] = ((A >> 4) & 0x03030303u) | (t & 0x04040404u);
    c[3] = ((A >> 6) & 0x03030303u) | ((t >> 1) & 0x04040404u);
}

// Elements 16j + 4m + 0..3 (quad 4j + m) -> two value pairs (code - 4).
__device__ __forceinline__ void decode_int3_quad(const uint32_t (&c)[4], int m, float2 (&d)[2])
{
    const float2 B = make_float2(-8388612.0f, -8388612.0f);    // -(2^23 + 4)
    const uint32_t sel = 0x7440u + (uint32_t)m;
    d[0] = fadd2(make_float2(u2f(__byte_perm(c[0], kMag0, sel)), u2f(__byte_perm(c[1], kMag0, sel))), B);
    d[1] = fadd2(make_float2(u2f(__byte_perm(c[2], kMag0, sel)), u2f(__byte_perm(c[3], kMag0, sel))), B);
}

// int3, nibble form: the 16 elements 16j..16j+15 (plane A word A, plane B
// bits in bytes sel of B) become two words of eight clean 3-bit codes, one per
// nibble: ce holds the even elements (nibble k = element 16j + 2k), co the odd
// ones.  Plane B's bit e is spread to bit 2e (byte permute, then three
// shift-and-mask steps), which puts the high bit of element 2k at bit 4k + 2
// after a shift by two and that of element 2k + 1 at bit 4k + 2 directly.
template <uint32_t SEL>
__device__ __forceinline__ void int3_nibbles(uint32_t A, uint32_t B, uint32_t& ce, uint32_t& co)
{
    uint32_t t = __byte_perm(B, 0u, SEL);              // the two plane-B bytes at bits 0..7 and 16..23
    t = (t | (t << 4)) & 0x0F0F0F0Fu;
    t = (t | (t << 2)) & 0x33333333u;
    t = (t | (t << 1)) & 0x55555555u;                  // bit e of the 16 -> bit 2e
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, 0x33333333, 0xE4;" : "=r"(d) : "r"(A), "r"(t << 2));      // (a & m) | (b & ~m)
    ce = d;
    asm("lop3.b32 %0, %1, %2, 0x33333333, 0xE4;" : "=r"(d) : "r"(A >> 2), "r"(t));
    co = d;
}

// Elements 16j + 2k and 16j + 2k + 1 (k = 0..3 from the low halves of ce and
// co, k = 4..7 from the high halves) -> value pairs (code - 4).
__device__ __forceinline__ void decode_int3_pairs(uint32_t ce, uint32_t co, float2 (&d)[8])
{
    const float2 B0 = make_float2(-8388612.0f, -8388612.0f);   // -(2^23 + 4)
    const float2 B1 = make_float2(-524292.0f, -524292.0f);     // -(2^19 + 4)
    const float2 B2 = make_float2(-32772.0f, -32772.0f);       // -(2^15 + 4)
    const float2 B3 = make_float2(-2052.0f, -2052.0f);         // -(2^11 + 4)
    const uint32_t he = ce >> 16, ho = co >> 16;
    d[0] = fadd2(make_float2(u2f(and_or<0x000Fu>(ce, kMag0)), u2f(and_or<0x000Fu>(co, kMag0))), B0);
    d[1] = fadd2(make_float2(u2f(and_or<0x00F0u>(ce, kMag1)), u2f(and_or<0x00F0u>(co, kMag1))), B1);
    d[2] = fadd2(make_float2(u2f(and_or<0x0F00u>(ce, kMag2)), u2f(and_or<0x0F00u>(co, kMag2))), B2);
    d[3] = fadd2(make_float2(u2f(and_or<0xF000u>(ce, kMag3)), u2f(and_or<0xF000u>(co, kMag3))), B3);
    d[4] = fadd2(make_float2(u2f(and_or<0x000Fu>(he, kMag0)), u2f(and_or<0x000Fu>(ho, kMag0))), B0);
    d[5] = fadd2(make_float2(u2f(and_or<0x00F0u>(he, kMag1)), u2f(and_or<0x00F0u>(ho, kMag1))), B1);
    d[6] = fadd2(make_float2(u2f(and_or<0x0F00u>(he, kMag2)), u2f(and_or<0x0F00u>(ho, kMag2))), B2);
    d[7] = fadd2(make_float2(u2f(and_or<0xF000u>(he, kMag3)), u2f(and_or<0xF000u>(ho, kMag3))), B3);
}

__device__ __forceinline__ uint32_t word(const uint4& v, int j)
{
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// ---------------------------------------------------------------------------
// Chunk consumption: for NR chunk rows (one chunk each) and S activation rows,
// acc[rr][s] += scale[rr] * sum_chunk value(code) * x_s.
// xq[s] is the shared-memory address of the chunk's swizzled x segment of
// activation row s; xo[j] = 16 * (j ^ swz) is this lane's byte offset of quad j.
// With one activation row, decoding and multiplying go row by row, the x quads
// of a word shared by all NR rows; with several, a word is decoded once for
// all of them.
// ---------------------------------------------------------------------------
// Shared-memory address of quad qd (0 .. EPL/4 - 1) of a lane's x segment.
// Swizzled layout: the segment is contiguous from xq, quads placed by xo.
// Lane-interleaved layout (PERM): quad qd of the 32 lanes of a warp step are
// 32 consecutive float4, so xq is the lane's quad 0 and quad qd sits 512 bytes
// per quad further.
template <bool PERM>
__device__ __forceinline__ uint32_t x_quad(uint32_t xq, const uint32_t (&xo)[8], int qd)
{
    if constexpr (PERM) return xq + 512u * (uint32_t)qd;
    else return xq + ((uint32_t)(qd >> 3) << 7) + xo[qd & 7];
}

template <int FMT, int S, int NR, bool PERM = false>
__device__ __forceinline__ void consume(const Chunk<FMT> (&c)[NR], const float (&sc)[NR],
                                        const uint32_t (&xq)[S], const uint32_t (&xo)[8], float (&acc)[S][NR],
                                        int s_act)
{
    // Every (row, activation row) accumulates in the same order whatever S is,
    // so a row's bits do not depend on how many activation rows share its launch.
    float2 part[NR][S];
#pragma unroll
    for (int rr = 0; rr < NR; rr++)
#pragma unroll
        for (int s = 0; s < S; s++) part[rr][s] = make_float2(0.f, 0.f);

    if constexpr (FMT == FMT_INT4_G || FMT == FMT_MXFP4_G32) {
        [[maybe_unused]] const Int4Magic g;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            if constexpr (S == 1) {
                const float4 xa = lds4s(x_quad<PERM>(xq[0], xo, 2 * j));
                const float4 xc = lds4s(x_quad<PERM>(xq[0], xo, 2 * j + 1));
#pragma unroll
                for (int rr = 0; rr < NR; rr++) {
                    float2 d[4];
                    if constexpr (FMT == FMT_INT4_G) decode_int4_word(word(c[rr].w, j), g, d);
                    else decode_mxfp4_word(word(c[rr].w, j), d);
                    part[rr][0] = ffma2(d[0], make_float2(xa.x, xa.y), part[rr][0]);
                    part[rr][0] = ffma2(d[1], make_float2(xa.z, xa.w), part[rr][0]);
                    part[rr][0] = ffma2(d[2], make_float2(xc.x, xc.y), part[rr][0]);
                    part[rr][0] = ffma2(d[3], make_float2(xc.z, xc.w), part[rr][0]);
                }
            } else {
                float2 d[NR][4];
#pragma unroll
                for (int rr = 0; rr < NR; rr++) {
                    if constexpr (FMT == FMT_INT4_G) decode_int4_word(word(c[rr].w, j), g, d[rr]);
                    else decode_mxfp4_word(word(c[rr].w, j), d[rr]);
                }
#pragma unroll
                for (int s = 0; s < S; s++) {
                    if (s >= s_act) break;                       // warp-uniform: activation rows in use
                    const float4 xa = lds4s(x_quad<PERM>(xq[s], xo, 2 * j));
                    const float4 xc = lds4s(x_quad<PERM>(xq[s], xo, 2 * j + 1));
#pragma unroll
                    for (int rr = 0; rr < NR; rr++) {
                            part[rr][s] = ffma2(d[rr][0], make_float2(xa.x, xa.y), part[rr][s]);
                        part[rr][s] = ffma2(d[rr][1], make_float2(xa.z, xa.w), part[rr][s]);
                        part[rr][s] = ffma2(d[rr][2], make_float2(xc.x, xc.y), part[rr][s]);
                        part[rr][s] = ffma2(d[rr][3], make_float2(xc.z, xc.w), part[rr][s]);
                    }
                }
            }
        }
    } else if constexpr (FMT == FMT_INT8_ROW) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float2 d[NR][2];
#pragma unroll
            for (int rr = 0; rr < NR; rr++) {
                decode_int8_word(word(c[rr].w, j), d[rr]);
            }
#pragma unroll
            for (int s = 0; s < S; s++) {
                if (s >= s_act) break;
                const float4 xa = lds4s(x_quad<PERM>(xq[s], xo, j));
#pragma unroll
                for (int rr = 0; rr < NR; rr++) {
                    part[rr][s] = ffma2(d[rr][0], make_float2(xa.x, xa.y), part[rr][s]);
                    part[rr][s] = ffma2(d[rr][1], make_float2(xa.z, xa.w), part[rr][s]);
                }
            }
        }
    } else if constexpr (QG_INT3_SPREAD) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float2 d[NR][8];
#pragma unroll
            for (int rr = 0; rr < NR; rr++) {
                uint32_t ce, co;
                const uint32_t B = (j & 2) ? c[rr].b.y : c[rr].b.x;
                if (j & 1) int3_nibbles<0x4342u>(word(c[rr].a, j), B, ce, co);
                else int3_nibbles<0x4140u>(word(c[rr].a, j), B, ce, co);
                decode_int3_pairs(ce, co, d[rr]);
            }
#pragma unroll
            for (int m = 0; m < 4; m++) {
                const int qd = 4 * j + m;
#pragma unroll
                for (int s = 0; s < S; s++) {
                    if (s >= s_act) break;
                    const float4 xv = lds4s(x_quad<PERM>(xq[s], xo, qd));
#pragma unroll
                    for (int rr = 0; rr < NR; rr++) {
                        part[rr][s] = ffma2(d[rr][2 * m], make_float2(xv.x, xv.y), part[rr][s]);
                        part[rr][s] = ffma2(d[rr][2 * m + 1], make_float2(xv.z, xv.w), part[rr][s]);
                    }
                }
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            uint32_t cls[NR][4];
#pragma unroll
            for (int rr = 0; rr < NR; rr++) {
                const uint32_t bh = ((j & 2) ? c[rr].b.y : c[rr].b.x) >> ((j & 1) * 16);
                int3_classes(word(c[rr].a, j), bh, cls[rr]);
            }
#pragma unroll
            for (int m = 0; m < 4; m++) {
                float2 d[NR][2];
#pragma unroll
                for (int rr = 0; rr < NR; rr++) {
                    decode_int3_quad(cls[rr], m, d[rr]);
                }
                const int qd = 4 * j + m;
#pragma unroll
                for (int s = 0; s < S; s++) {
                    if (s >= s_act) break;
                    const float4 xv = lds4s(x_quad<PERM>(xq[s], xo, qd));
#pragma unroll
                    for (int rr = 0; rr < NR; rr++) {
                            part[rr][s] = ffma2(d[rr][0], make_float2(xv.x, xv.y), part[rr][s]);
                        part[rr][s] = ffma2(d[rr][1], make_float2(xv.z, xv.w), part[rr][s]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < NR; rr++)
#pragma unroll
        for (int s = 0; s < S; s++) acc[s][rr] = fmaf(part[rr][s].x + part[rr][s].y, sc[rr], acc[s][rr]);
}

// ---------------------------------------------------------------------------
// Stage activation rows into shared memory (swizzled, float4 granularity).
// src[s] are f32 rows of length I (16-byte aligned); all threads take part.
// ---------------------------------------------------------------------------
template <int EPL>
__device__ __forceinline__ void stage_rows(float* xs, int xstride, const float* const* src, int nrows, int I)
{
    const int nq = I / 4;
    for (int idx = threadIdx.x; idx < nrows * nq; idx += blockDim.x) {
        const int s = idx / nq;
        const int qd = idx - s * nq;
        const float4 v = *reinterpret_cast<const float4*>(src[s] + 4 * qd);
        *reinterpret_cast<float4*>(xs + (long long)s * xstride + 4 * x_quad_phys(EPL, qd)) = v;
    }
}

// One float4 of activations; FRESH: through L2 only (written in this launch).
template <bool FRESH>
__device__ __forceinline__ float4 load_x4(const float* p)
{
    if constexpr (FRESH) return __ldcg(reinterpret_cast<const float4*>(p));
    else return *reinterpret_cast<const float4*>(p);
}

// The same rows in the lane-interleaved layout, rows of xstride floats (a
// multiple of 32 * EPL) zero beyond I: element i of chunk q = i / EPL (lane
// l = q % 32 of warp step k = q / 32), quad j of the chunk, goes to float4
// (k * EPL / 4 + j) * 32 + l.  Threads t of [0, nthreads) take part.
// FRESH: the rows were written earlier in the same launch (by other CTAs):
// read them through L2 only.
template <int EPL, bool FRESH = false>
__device__ __forceinline__ void stage_rows_perm(float* xs, int xstride, const float* const* src, int nrows, int I,
                                                int t, int nthreads)
{
    constexpr int QPC = EPL / 4;              // quads per chunk
    const int iq = I / 4;
    if (nrows >= 2) {
        // Several rows (measured faster with this order): one thread per chunk;
        // it reads the chunk's contiguous quads and writes quad j where the warp
        // step's 32 chunks sit side by side, so the 32 threads of a warp store
        // consecutive float4 (no bank conflicts).
        const int nc = xstride / EPL;
        for (int idx = t; idx < nrows * nc; idx += nthreads) {
            const int s = idx / nc;
            const int q = idx - s * nc;
            const float* src_q = src[s] + 4 * q * QPC;
            float* dst = xs + (long long)s * xstride + 4 * ((q >> 5) * QPC * 32 + (q & 31));
#pragma unroll 4
            for (int j = 0; j < QPC; j++) {
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (q * QPC + j < iq) v = load_x4<FRESH>(src_q + 4 * j);
                *reinterpret_cast<float4*>(dst + 4 * 32 * j) = v;
            }
        }
        return;
    }
    // One row: one thread per quad (coalesced reads).
    const int nq = xstride / 4;
    for (int idx = t; idx < nrows * nq; idx += nthreads) {
        const int s = idx / nq;
        const int qd = idx - s * nq;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (qd < iq) v = load_x4<FRESH>(src[s] + 4 * qd);
        const int q = qd / QPC, j = qd - q * QPC;
        const int phys = ((q >> 5) * QPC + j) * 32 + (q & 31);
        *reinterpret_cast<float4*>(xs + (long long)s * xstride + 4 * phys) = v;
    }
}

__host__ __device__ constexpr int ilog2(int v) { int l = 0; while ((1 << l) < v) l++; return l; }

// ---------------------------------------------------------------------------
// Transposed warp reduction of V (power of two, <= 32) values: afterwards lane
// l < V holds the sum over the warp of value idx(l), with
// idx(l) = sum_k bit_k(l) * (V >> (k + 1)).
// ---------------------------------------------------------------------------
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V], int lane)
{
    static_assert((V & (V - 1)) == 0 && V <= 32, "V must be a power of two <= 32");
#pragma unroll
    for (int k = 0, n = V; n > 1; k++, n >>= 1) {
        const bool up = (lane >> k) & 1;
#pragma unroll
        for (int i = 0; i < n / 2; i++) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << k);
        }
    }
    float r = v[0];
    constexpr int logv = ilog2(V);
#pragma unroll
    for (int k = logv; k < 5; k++) r += __shfl_xor_sync(0xffffffffu, r, 1 << k);
    return r;
}

template <int V>
__device__ __forceinline__ int reduce_scatter_index(int lane)
{
    int idx = 0;
#pragma unroll
    for (int k = 0; (V >> (k + 1)) > 0; k++)
        if ((lane >> k) & 1) idx += V >> (k + 1);
    return idx;
}

__host__ __device__ constexpr int pow2_ceil(int v) { int p = 1; while (p < v) p <<= 1; return p; }

// ---------------------------------------------------------------------------
// Asynchronous copies of 16, 8 and 4 bytes global -> shared (L2 only for the
// 16-byte weight chunks).  Each lane copies, and later reads back, only its
// own chunks, so completion is per thread (cp.async groups) and no barrier or
// spin-wait is involved.
// ---------------------------------------------------------------------------
// dst: absolute shared-window address.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ uint4 lds16(uint32_t a)
{
#if QG_CXX_LDS
    return *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(qg_smem4) + a);
#else
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a + smem_base()));
    return v;
#endif
}
__device__ __forceinline__ uint2 lds8(uint32_t a)
{
#if QG_CXX_LDS
    return *reinterpret_cast<const uint2*>(reinterpret_cast<const char*>(qg_smem4) + a);
#else
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a + smem_base()));
    return v;
#endif
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a)
{
    return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(qg_smem4) + a);
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a)
{
    return *reinterpret_cast<const uint8_t*>(reinterpret_cast<const char*>(qg_smem4) + a);
}
__device__ __forceinline__ float lds_f32(uint32_t a)
{
#if QG_CXX_LDS
    return *reinterpret_cast<const float*>(reinterpret_cast<const char*>(qg_smem4) + a);
#else
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a + smem_base()));
    return v;
#endif
}

// ---------------------------------------------------------------------------
// mbarriers and tensor (TMA engine) copies.  Every wait is bounded in time: a
// wait that has not completed after kWaitNs returns false and the caller
// records QSTATUS_DEVICE_TIMEOUT and leaves.
// ---------------------------------------------------------------------------
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase of the given parity to complete; false after kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t n = 1;; n++) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 15u) == 0 && global_ns() - t0 > kWaitNs) return false;   // the clock every 16 tries
    }
}
// Every warp of the CTA arrives on `bar` (initialized for one arrival per
// warp: lane 0 arrives once the warp's lanes have met at __syncwarp, which
// orders their memory operations before the arrival) and every thread waits
// for the others; `parity` tracks the barrier's phase.  False after kWaitNs.
// One arrival per warp rather than per thread keeps the barrier's
// shared-memory updates to one per warp.
__device__ __forceinline__ bool cta_barrier(uint32_t bar, uint32_t& parity)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait(bar, parity);
    parity ^= 1u;
    return ok;
}
// Tensor copy of one 2-D box (inner coordinate c0 in 4-byte elements, row
// coordinate c1) of the tensor map at `map` into this CTA's shared memory at
// `dst`; completion is counted on mbarrier `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, int c0, int c1, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 :: "r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar) : "memory");
}

// ---------------------------------------------------------------------------
// Tensor cores (tcgen05) and tensor memory, for the prefill GEMM.
// ---------------------------------------------------------------------------
// One warp allocates `ncols` (a power of two >= 32) columns of tensor memory
// for the CTA and writes their address to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Makes this thread's shared-memory stores visible to the tensor cores and
// the tensor copies (the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A * B^T for one 128 x N x 16 step, f16 inputs, f32 sums;
// `acc` = 0 overwrites D.  Issued by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}
// The mbarrier at `bar` receives one arrival once every tensor-core operation
// this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
                 : "memory");
}
// Instruction descriptor of kind::f16: f16 A and B, both K-major, f32 D,
// M x N (M = 128, N a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t tc_idesc_f16(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Shared-memory matrix descriptor: K-major rows of 128 bytes in the 128-byte
// swizzle (16-byte chunk c of row r stored at chunk c ^ (r % 8); groups of 8
// rows 1024 bytes apart), starting at shared address `saddr` (the tile
// 1024-byte aligned; a K step inside the row adds its byte offset).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// 32 consecutive 32-bit columns of this warp's 32 lanes of tensor memory
// (lane = thread), waited for before return.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                 "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, "
                 "%31}, [%32];\n\ttcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit columns of this warp's 32 lanes, waited for.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\ttcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// f16x2 helpers for decoding codes exactly to f16.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c)   // (a & b) | c
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Two e2m1 codes (low byte of v: the low nibble is the even element) as f16x2.
__device__ __forceinline__ uint32_t e2m1x2_to_h2(uint32_t v)
{
    uint32_t h2;
    asm("{\n\t.reg .b8 t;\n\t.reg .b16 u;\n\tcvt.u16.u32 u, %1;\n\tcvt.u8.u16 t, u;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
        : "=r"(h2) : "r"(v));
    return h2;
}

// Bytes of one ring slot: NR chunk rows x 32 lanes (16 B of codes, int3 also
// 8 B of plane B) and their scales.
template <int FMT, int NR>
__host__ __device__ constexpr int ring_slot_bytes()
{
    return NR * 32 * (16 + (FMT == FMT_INT3_G64 ? 8 : 0) + 4);
}

// ---------------------------------------------------------------------------
// Row streaming.  A warp processes row tiles of R rows (of NM matrices sharing
// the same row index: NM = 2 for gate and up): tiles tile_first,
// tile_first + tile_step, ... below ntiles, rows row0 + tile * R + r < row_end;
// rows of the last tile past row_end are not copied (their arithmetic runs on
// stale ring data and the sink drops it, which keeps the rows interleaved).
// Work is the flattened sequence (tile, step); step c covers chunk c*32 + lane
// of each row.  Copies run P steps ahead of use through a ring of P slots in
// this warp's part of shared memory.  Each row's chunk and scale addresses are
// set once per tile and advance by a constant per step.  The sink is called
// once per finished tile from every lane: sink(value, index, lane_holds_it,
// first row of the tile, row_end) with index v = (s * R + r) * NM + m.
// ---------------------------------------------------------------------------
// SH: lanes share scales (one per row, ue8m0 words, or groups longer than a
// chunk): only the first lane of each sharing set copies a scale (word) and
// the others take it by shuffle -- many lanes copying one address are slow.
template <int QF, int S, int R, int P, int NM, bool LOOP_S = false, bool SH = false>
struct RowStreamer {
    static constexpr int FMT = decode_of(QF);       // how codes decode
    static constexpr int SK = scale_kind_of(QF);    // how scales are stored
    static constexpr int EPL = Traits<FMT>::EPL;
    static constexpr int NR = NM * R;
    static constexpr int V = pow2_ceil(S * R * NM);
    static constexpr int SLOT = ring_slot_bytes<FMT, NR>();
    static constexpr int B_OFF = NR * 32 * 16;                                  // plane B part of a slot
    static constexpr int S_OFF = NR * 32 * (16 + (FMT == FMT_INT3_G64 ? 8 : 0)); // scales part of a slot

    const uint8_t* wp[NR];    // this lane's next chunk of each row (int3: plane A)
    const uint8_t* bp[NR];    // int3 plane B
    const float* sp[NR];      // this lane's next scale of each row (ue8m0: the aligned word holding it)
    int sstep;                // scale advance per step
    uint32_t lead;            // SH: this lane minus the first lane sharing its scale (word), which copies it
    uint32_t ring;            // this lane's byte offset in slot 0 of the warp's ring
    uint32_t sbase;           // shared-window address of the dynamic shared memory

    Mat mats[NM];
    long long row0, row_end;
    int it_tile, it_c, ct_tile, ct_c;
    int it_valid;             // rows of the issuing tile below row_end
    int total, issued, nchunks, nsteps, ntiles, tile_step, lane;

    __device__ __forceinline__ int tile_rows(int tile) const
    {
        const long long first = row0 + (long long)tile * R;
        return (int)(row_end - first < R ? row_end - first : R);
    }

    __device__ __forceinline__ void set_tile(int tile)
    {
        const long long first = row0 + (long long)tile * R;
        it_valid = tile_rows(tile);
#pragma unroll
        for (int r = 0; r < R; r++) {
            long long o = first + r;
            o = o < row_end ? o : row_end - 1;       // rows past the end are never loaded
#pragma unroll
            for (int m = 0; m < NM; m++) {
                const Mat& M = mats[m];
                const int rr = m * R + r;
                if constexpr (FMT == FMT_INT8_ROW) {
                    wp[rr] = M.w + o * M.I + lane * 16;
                } else if constexpr (FMT == FMT_INT3_G64) {
                    wp[rr] = M.w + o * (long long)(M.I / 4) + lane * 16;
                    bp[rr] = M.w + M.O * (long long)(M.I / 4) + o * (long long)(M.I / 8) + lane * 8;
                } else {
                    wp[rr] = M.w + o * (long long)(M.I / 2) + lane * 16;
                }
                if constexpr (SK == SK_ROW) sp[rr] = M.sc + o;
                else if constexpr (SK == SK_E8M0) sp[rr] = sc_ptr<SK>(M.sc, o * M.ngrp + (lane & ~3));
                else sp[rr] = M.sc + o * M.ngrp + (lane >> M.gsh);
            }
        }
    }

    // Copies of the next step into slot p; one cp.async group per call, empty
    // past the end, so group counts stay aligned with steps.
    __device__ __forceinline__ void issue(int p)
    {
        if (issued < total) {
            const bool ok = it_c * 32 + lane < nchunks;
            const uint32_t slot = sbase + ring + (uint32_t)(p * SLOT);
#pragma unroll
            for (int rr = 0; rr < NR; rr++) {
                if (ok && (rr % R) < it_valid) {
                    cp_async16(slot + rr * 512, wp[rr]);
                    if constexpr (FMT == FMT_INT3_G64) cp_async8(slot + B_OFF + rr * 256 - lane * 8, bp[rr]);
                    // one copy per scale (word): many lanes copying one address are slow
                    if (!SH || lead == 0) cp_async4(slot + S_OFF + rr * 128 - lane * 12, sp[rr]);
                }
                wp[rr] += 512;
                if constexpr (FMT == FMT_INT3_G64) bp[rr] += 256;
                sp[rr] = sc_ptr<SK>(sp[rr], sstep);
            }
            ++issued;
            if (++it_c == nsteps) {
                it_c = 0;
                it_tile += tile_step;
                if (it_tile < ntiles) set_tile(it_tile);
            }
        }
        cp_async_commit();
    }

    // ring_warp: byte offset of this warp's ring (P slots of SLOT bytes).
    __device__ __forceinline__ void begin(const Mat* m, long long row0_, long long row_end_, int tile_first,
                                          int ntiles_, int tile_step_, int lane_, uint32_t ring_warp)
    {
#pragma unroll
        for (int k = 0; k < NM; k++) mats[k] = m[k];
        row0 = row0_;
        row_end = row_end_;
        lane = lane_;
        tile_step = tile_step_;
        ntiles = ntiles_;
        ring = ring_warp + (uint32_t)lane * 16;
        sbase = smem_base();
        nchunks = m[0].I / EPL;
        nsteps = (nchunks + 31) / 32;
        // one scale per row: none; else 32 chunks span 32 >> gsh groups (ue8m0: that many bytes)
        sstep = SK == SK_ROW ? 0 : (32 >> m[0].gsh);
        // lanes sharing a scale: all 32 (one per row), 2^gsh (a group spans 2^gsh chunks), 4 (ue8m0 word)
        lead = (uint32_t)lane & (SK == SK_ROW ? 31u : SK == SK_E8M0 ? 3u : ((1u << m[0].gsh) - 1u) & 31u);
        const int my_tiles = tile_first < ntiles ? (ntiles - tile_first + tile_step - 1) / tile_step : 0;
        total = my_tiles * nsteps;
        issued = 0;
        it_tile = ct_tile = tile_first;
        it_c = ct_c = 0;
        if (total > 0) set_tile(it_tile);
#pragma unroll
        for (int p = 0; p < P; p++) issue(p);
    }

    // xs[s]: shared-memory byte offsets of the swizzled activation rows; only
    // the first s_act (<= S) are in use.
    template <class Sink>
    __device__ __forceinline__ void run(const uint32_t (&xs)[S], int s_act, Sink& sink)
    {
        const uint32_t swz = (uint32_t)x_swz(EPL, lane);
        uint32_t xo[8];
#pragma unroll
        for (int j = 0; j < 8; j++) xo[j] = 16u * ((uint32_t)j ^ swz);
        uint32_t xl[S];                      // this lane's first chunk segment of each row
#pragma unroll
        for (int s = 0; s < S; s++) xl[s] = xs[s] + (uint32_t)lane * (EPL * 4);

        float acc[S][NR];
#pragma unroll
        for (int s = 0; s < S; s++)
#pragma unroll
            for (int rr = 0; rr < NR; rr++) acc[s][rr] = 0.f;

        for (int j0 = 0; j0 < total; j0 += P) {
#pragma unroll
            for (int p = 0; p < P; p++) {
                if (j0 + p < total) {
                    cp_async_wait<P - 1>();          // this step's copies have landed
                    if (ct_c * 32 + lane < nchunks) {
                        const uint32_t slot = ring + (uint32_t)(p * SLOT);
                        Chunk<FMT> c[NR];
                        uint32_t sw[NR];     // scale words, each read at this lane's own slot position
#pragma unroll
                        for (int rr = 0; rr < NR; rr++) {
                            if constexpr (FMT == FMT_INT3_G64) {
                                c[rr].a = lds16(slot + rr * 512);
                                c[rr].b = lds8(slot + B_OFF + rr * 256 - lane * 8);
                            } else {
                                c[rr].w = lds16(slot + rr * 512);
                            }
                            sw[rr] = lds_u32(slot + S_OFF + rr * 128 - lane * 12);
                        }
                        if constexpr (SH) {
                            // lanes sharing a scale take the word of the lane that
                            // copied it; the lanes here are a prefix of the warp
                            // holding every such lane
                            const int rem = nchunks - ct_c * 32;
                            const uint32_t act = rem >= 32 ? 0xffffffffu : ((1u << rem) - 1u);
#pragma unroll
                            for (int rr = 0; rr < NR; rr++) sw[rr] = __shfl_sync(act, sw[rr], lane - (int)lead);
                        }
                        float sc[NR];
#pragma unroll
                        for (int rr = 0; rr < NR; rr++) {
                            if constexpr (SK == SK_E8M0)   // byte lane & 3 of the word
                                sc[rr] = e8m0_to_f32(__byte_perm(sw[rr], 0u, 0x4440u + (uint32_t)(lane & 3)));
                            else
                                sc[rr] = __uint_as_float(sw[rr]);
                        }
                        uint32_t xq[S];
#pragma unroll
                        for (int s = 0; s < S; s++) xq[s] = xl[s] + (uint32_t)ct_c * (32 * EPL * 4);
                        if constexpr (LOOP_S) {
                            // one-row arithmetic per activation row in use, on the same ring data
#pragma unroll
                            for (int s = 0; s < S; s++) {
                                if (s < s_act) {
                                    const uint32_t x1[1] = {xq[s]};
                                    consume<FMT, 1, NR>(c, sc, x1, xo,
                                                        reinterpret_cast<float(&)[1][NR]>(acc[s]), 1);
                                }
                            }
                        } else {
                            consume<FMT, S, NR>(c, sc, xq, xo, acc, s_act);
                        }
                    }
                    issue(p);
                    if (++ct_c == nsteps) {
                        // finished tile ct_tile: reduce and hand to the sink
                        if (LOOP_S && s_act == 1) {
                            // one activation row in use: reduce only its NR values
                            constexpr int V1 = pow2_ceil(R * NM);
                            float v[V1];
#pragma unroll
                            for (int i = 0; i < V1; i++) v[i] = 0.f;
#pragma unroll
                            for (int r = 0; r < R; r++)
#pragma unroll
                                for (int m = 0; m < NM; m++) v[r * NM + m] = acc[0][m * R + r];
                            const float red = warp_reduce_scatter<V1>(v, lane);
                            const int idx = reduce_scatter_index<V1>(lane);
                            sink.template put<V1>(red, idx, lane < V1, row0 + (long long)ct_tile * R, row_end);
                        } else {
                            float v[V];
#pragma unroll
                            for (int i = 0; i < V; i++) v[i] = 0.f;
#pragma unroll
                            for (int s = 0; s < S; s++)
#pragma unroll
                                for (int r = 0; r < R; r++)
#pragma unroll
                                    for (int m = 0; m < NM; m++) v[(s * R + r) * NM + m] = acc[s][m * R + r];
                            const float red = warp_reduce_scatter<V>(v, lane);
                            const int idx = reduce_scatter_index<V>(lane);
                            sink.template put<V>(red, idx, lane < V, row0 + (long long)ct_tile * R, row_end);
                        }
#pragma unroll
                        for (int s = 0; s < S; s++)
#pragma unroll
                            for (int rr = 0; rr < NR; rr++) acc[s][rr] = 0.f;
                        ct_c = 0;
                        ct_tile += tile_step;
                    }
                }
            }
        }
        cp_async_wait<0>();
    }
};

}  // namespace qg
