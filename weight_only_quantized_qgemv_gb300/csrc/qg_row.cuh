// qg_row.cuh -- the row-team streaming kernel (one format; included by
// qg_fmt_impl.cuh inside its format namespace).
//
// What it computes is the same contraction as the other streaming kernels
// (colibri Vulkan guide, xdnf.cn, section 着色器层面的实现细节: one quantized
// row against the activations staged once, reduced across the lanes), laid
// out for GB300 as follows:
//  * A row of P 16-byte chunks (int3: 16 bytes of plane A plus 8 of plane B)
//    is owned by a team of P threads, thread p always taking chunk p.  The CTA
//    holds G = threads / P such teams; team g takes the CTA's rows g, g + G,
//    g + 2G, ... so the teams stream neighbouring rows side by side.
//  * Because a thread always sees the same inputs, its slice of every
//    activation row (EPL floats per row) lives in registers for the whole
//    launch (the expert phases reload it when their batch changes): x is
//    never read from shared memory in the inner loop.
//  * Each thread keeps its own ring of D slots in shared memory, filled by
//    cp.async of its own chunk, scale and plane-B bytes of the row D ahead; a
//    thread reads back only what it copied, so the ring needs no barrier.
//    The first D rows are requested before the kernel waits for the previous
//    one in the stream (programmatic dependent launch), so a call's weight
//    stream starts under the previous call's tail.
//  * Every V rows the team reduces: a transposed butterfly inside each warp
//    (one shuffle per value), then the team's W = P / 32 warp sums of each
//    row are added in warp order by one thread after a team barrier.
// The summation order of a row is fixed by (P, G): results are deterministic.
#pragma once

// Threads per CTA: 576 (teams of 64 or 192 threads fill it; a thread may use
// up to 96 registers), 512 for int3, whose activation slice alone takes 64.
#ifndef QG_ROW_THREADS
#define QG_ROW_THREADS (FMT == FMT_INT3_G64 ? 512 : 576)
#endif
constexpr int kRowThreads = QG_ROW_THREADS;
#ifndef QG_ROW_SMEM
#define QG_ROW_SMEM (196 * 1024)
#endif

// Bytes one ring slot takes per thread and matrix: code chunk, int3 plane B,
// and the chunk's scale (none for one scale per row: applied after the sum).
constexpr int kRowSlot = 16 + (FMT == FMT_INT3_G64 ? 8 : 0) + (SK == SK_ROW ? 0 : 4);

// Rows a thread takes per ring step (one step = one wait, one round of copy
// issue, one slot): 4 chunks per step so the step's fixed cost is shared.
#ifndef QG_ROW_RT
#define QG_ROW_RT 4
#endif
template <int NM>
__host__ __device__ constexpr int row_rt()
{
    return QG_ROW_RT / NM > 0 ? QG_ROW_RT / NM : 1;
}

// Ring depth in steps for NM matrices per row, sized for kRowThreads threads.
template <int NM>
__host__ __device__ constexpr int row_depth()
{
    constexpr int d = QG_ROW_SMEM / (kRowThreads * NM * row_rt<NM>() * kRowSlot);
    return d > 16 ? 16 : (d < 2 ? 2 : d);
}

// Steps per team reduction round: 16 values per warp butterfly (8 for int3,
// whose activation slice takes 64 registers).
#ifndef QG_ROW_VALS
#define QG_ROW_VALS (FMT == FMT_INT3_G64 ? 8 : 16)
#endif
template <int S, int NM>
__host__ __device__ constexpr int row_v()
{
    constexpr int vals = QG_ROW_VALS;
    constexpr int per_step = row_rt<NM>() * S * NM;
    return vals / per_step > 0 ? vals / per_step : 1;
}

// The dot product of one chunk with the thread's activation slice x2 (EPL / 2
// pairs of floats, kept as pairs so the packed FMAs take them as they are), in
// two packed accumulators.
template <int F_>
__device__ __forceinline__ float chunk_dot(const Chunk<F_>& c, const float2* x2)
{
    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
    if constexpr (F_ == FMT_INT4_G || F_ == FMT_MXFP4_G32) {
        [[maybe_unused]] const Int4Magic g;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float2 d[4];
            if constexpr (F_ == FMT_INT4_G) decode_int4_word(word(c.w, j), g, d);
            else decode_mxfp4_word(word(c.w, j), d);
            a = ffma2(d[0], x2[4 * j + 0], a);
            b = ffma2(d[1], x2[4 * j + 1], b);
            a = ffma2(d[2], x2[4 * j + 2], a);
            b = ffma2(d[3], x2[4 * j + 3], b);
        }
    } else if constexpr (F_ == FMT_INT8_ROW) {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            float2 d[2];
            decode_int8_word(word(c.w, j), d);
            a = ffma2(d[0], x2[2 * j + 0], a);
            b = ffma2(d[1], x2[2 * j + 1], b);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; j++) {
            uint32_t ce, co;
            const uint32_t B = (j & 2) ? c.b.y : c.b.x;
            if (j & 1) int3_nibbles<0x4342u>(word(c.a, j), B, ce, co);
            else int3_nibbles<0x4140u>(word(c.a, j), B, ce, co);
            float2 d[8];
            decode_int3_pairs(ce, co, d);
#pragma unroll
            for (int k = 0; k < 8; k += 2) {
                a = ffma2(d[k], x2[8 * j + k], a);
                b = ffma2(d[k + 1], x2[8 * j + k + 1], b);
            }
        }
    }
    a = fadd2(a, b);
    return a.x + a.y;
}

// Host-computed plan of a row-team launch.
struct RowPlan {
    int P;          // threads per row (chunks per row)
    int G;          // teams per CTA
    int T;          // active threads, P * G
    int W;          // warps per team, P / 32
    int code_off, b_off, sc_off, red_off;   // shared-memory regions (bytes)
    int total;      // dynamic shared memory
};

// One matrix or a gate/up pair against S activation rows; row o is item o.
template <int NM>
struct RowDenseJob {
    static constexpr bool kWaitFirst = false;
    RowPlan plan;
    Mat m[NM];
    const float* x;      // [S][I]
    float* y;            // y[s * ldy + row]
    long long ldy;
    int act;             // NM = 2: QACT_* of the gate/up product
    float limit;
    long long rb, rbB;   // code (int3: plane A) and plane-B bytes per row
    int sbytes;          // scale bytes per row (f32: 4 * groups; ue8m0: groups)

    __device__ void cta_items(int c, int G, long long& i0, long long& i1) const
    {
        i0 = m[0].O * c / G;
        i1 = m[0].O * (c + 1) / G;
    }
    // addresses of thread p's chunk, plane-B bytes and scale word of row o of matrix k
    __device__ void ptrs(int k, long long o, int p, const uint8_t*& cp, const uint8_t*& bp, const uint8_t*& sp) const
    {
        const Mat& M = m[k];
        cp = M.w + o * rb + (long long)p * 16;
        bp = M.w + M.O * rb + o * rbB + (long long)p * 8;
        if constexpr (SK == SK_E8M0)
            sp = reinterpret_cast<const uint8_t*>(M.sc) + o * M.ngrp + (((long long)p >> M.gsh) & ~3ll);
        else
            sp = reinterpret_cast<const uint8_t*>(M.sc + o * M.ngrp + (p >> M.gsh));
    }
    __device__ const float* xrow(int s) const { return x + (long long)s * m[0].I; }
    __device__ float row_scale(int k, long long o) const { return ldg_f32(m[k].sc + o); }
    __device__ void store(int s, long long o, float v) const { y[(long long)s * ldy + o] = v; }
};

template <int NM, int S, class Job>
__global__ void __launch_bounds__(kRowThreads, 1) k_row(const __grid_constant__ Job job)
{
    constexpr int RT = row_rt<NM>();                 // rows per step
    constexpr int D = row_depth<NM>();               // steps in flight
    constexpr int V = row_v<S, NM>();                // steps per reduction round
    constexpr int VS = pow2_ceil(V * RT * S * NM);   // values per warp butterfly
    constexpr int QS = RT * NM;                      // chunks per slot
    const RowPlan& L = job.plan;
    const int tid = threadIdx.x;
    const bool active = tid < L.T;
    const int g = tid / L.P, p = tid - g * L.P;
    const int lane = tid & 31;
    const uint32_t sbase = smem_base();

    pdl_allow_next();
    long long i0, i1;
    job.cta_items(blockIdx.x, gridDim.x, i0, i1);
    const long long G = L.G, GR = G * RT;
    // team g's step k covers the rows i0 + (k G + g) RT + r, r < RT (those below i1)
    const long long first = i0 + (long long)g * RT;
    const int n = (active && first < i1) ? (int)((i1 - first + GR - 1) / GR) : 0;

    // ---- the thread's copy stream ----
    const uint8_t* cp[NM];
    const uint8_t* bp[NM];
    const uint8_t* sp[NM];
#pragma unroll
    for (int k = 0; k < NM; k++) job.ptrs(k, first, p, cp[k], bp[k], sp[k]);
    const long long rb = job.rb, rbB = job.rbB, sb = job.sbytes;
    // ring chunk q (= (slot RT + r) NM + matrix) of this thread: codes at
    // c_s + q c_q, plane B at b_s + q b_q, scales at s_s + q s_q (byte offsets
    // from the dynamic shared memory; copies take the window address sbase + it)
    const uint32_t T = (uint32_t)L.T;
    const uint32_t c_s = (uint32_t)L.code_off + (uint32_t)tid * 16u, c_q = T * 16u;
    const uint32_t b_s = (uint32_t)L.b_off + (uint32_t)tid * 8u, b_q = T * 8u;
    const uint32_t s_s = (uint32_t)L.sc_off + (uint32_t)tid * 4u, s_q = T * 4u;
    int issued = 0;
    long long irow = first;                          // first row of the next step to issue
    auto issue = [&](uint32_t q0) {
        if (issued < n) {
            const long long left = i1 - irow;
#pragma unroll
            for (int k = 0; k < NM; k++) {
                const uint8_t* c = cp[k];
                [[maybe_unused]] const uint8_t* bq = bp[k];
                [[maybe_unused]] const uint8_t* sq = sp[k];
#pragma unroll
                for (int r = 0; r < RT; r++) {
                    const uint32_t q = q0 + (uint32_t)(r * NM + k);
                    if (r < left) {                   // rows past the CTA's range are not copied
                        cp_async16(sbase + c_s + q * c_q, c);
                        if constexpr (FMT == FMT_INT3_G64) cp_async8(sbase + b_s + q * b_q, bq);
                        if constexpr (SK != SK_ROW) cp_async4(sbase + s_s + q * s_q, sq);
                    }
                    c += rb;
                    if constexpr (FMT == FMT_INT3_G64) bq += rbB;
                    if constexpr (SK != SK_ROW) sq += sb;
                }
                cp[k] += GR * rb;
                if constexpr (FMT == FMT_INT3_G64) bp[k] += GR * rbB;
                if constexpr (SK != SK_ROW) sp[k] += GR * sb;
            }
            irow += GR;
        }
        issued++;
        cp_async_commit();
    };
#pragma unroll
    for (int k = 0; k < D; k++) issue((uint32_t)(k * QS));

    if constexpr (!Job::kWaitFirst) pdl_wait_prev();   // activations and outputs from here on

    // ---- the activation slice of this thread, in registers, as pairs ----
    float2 xr[S][EPL / 2];
#pragma unroll
    for (int s = 0; s < S; s++) {
        const float4* src = reinterpret_cast<const float4*>(job.xrow(s) + (long long)p * EPL);
#pragma unroll
        for (int q = 0; q < EPL / 4; q++) {
            const float4 v = active ? src[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            xr[s][2 * q + 0] = make_float2(v.x, v.y);
            xr[s][2 * q + 1] = make_float2(v.z, v.w);
        }
    }

    float* red = reinterpret_cast<float*>(reinterpret_cast<char*>(qg_smem4) + L.red_off);
    const int warp_global = tid >> 5;
    uint32_t slot = 0;                               // first chunk index of the current slot
    int buf = 0;
    for (int j0 = 0; j0 < n; j0 += V) {
        float vb[VS];
#pragma unroll
        for (int i = 0; i < VS; i++) vb[i] = 0.f;
#pragma unroll
        for (int v = 0; v < V; v++) {
            if (j0 + v < n) {
                cp_async_wait<D - 1>();      // this step's copies have landed
                Chunk<FMT> ch[RT][NM];
                [[maybe_unused]] float sc[RT][NM];
#pragma unroll
                for (int r = 0; r < RT; r++)
#pragma unroll
                    for (int k = 0; k < NM; k++) {
                        const uint32_t q = slot + (uint32_t)(r * NM + k);
                        if constexpr (FMT == FMT_INT3_G64) {
                            ch[r][k].a = lds16(c_s + q * c_q);
                            ch[r][k].b = lds8(b_s + q * b_q);
                        } else {
                            ch[r][k].w = lds16(c_s + q * c_q);
                        }
                        if constexpr (SK == SK_E8M0)
                            sc[r][k] = e8m0_to_f32(__byte_perm(lds_u32(s_s + q * s_q), 0u,
                                                               0x4440u + (uint32_t)(p & 3)));
                        else if constexpr (SK == SK_F32)
                            sc[r][k] = lds_f32(s_s + q * s_q);
                    }
                issue(slot);                 // the step D ahead goes into the slot just read
                slot = slot + QS == (uint32_t)(D * QS) ? 0u : slot + QS;
#pragma unroll
                for (int r = 0; r < RT; r++)
#pragma unroll
                    for (int s = 0; s < S; s++)
#pragma unroll
                        for (int k = 0; k < NM; k++) {
                            const float dsum = chunk_dot<FMT>(ch[r][k], xr[s]);
                            vb[((v * RT + r) * S + s) * NM + k] = SK == SK_ROW ? dsum : dsum * sc[r][k];
                        }
            }
        }
        if (!active) continue;
        // ---- team reduction of the round: warp butterfly, then W warp sums in order ----
        const float rv = warp_reduce_scatter<VS>(vb, lane);
        const int idx = reduce_scatter_index<VS>(lane);
        float* rbuf = red + (size_t)buf * (kRowThreads / 32) * VS;
        if (lane < VS) rbuf[warp_global * VS + idx] = rv;
        asm volatile("bar.sync %0, %1;" :: "r"(1 + g), "r"(L.P) : "memory");
        if (p < V * RT * S) {
            const int vr = p / S, s = p - vr * S;        // row vr of the round (step vr / RT, row vr % RT)
            const int v = vr / RT, r = vr - v * RT;
            const long long o = first + (long long)(j0 + v) * GR + r;
            if (j0 + v < n && o < i1) {
                float tot[NM];
#pragma unroll
                for (int k = 0; k < NM; k++) {
                    float t = 0.f;
                    for (int w = 0; w < L.W; w++) t += rbuf[(g * L.W + w) * VS + (vr * S + s) * NM + k];
                    tot[k] = SK == SK_ROW ? t * job.row_scale(k, o) : t;
                }
                if constexpr (NM == 2) {
                    float gv = tot[0], u = tot[1];
                    if (job.act == QACT_SWIGLU_CLAMPED) {    // clamped SwiGLU: gate capped, up clamped to [-L, L]
                        gv = fminf(gv, job.limit);
                        u = fminf(fmaxf(u, -job.limit), job.limit);
                    }
                    job.store(s, o, gv / (1.0f + expf(-gv)) * u);
                } else {
                    job.store(s, o, tot[0]);
                }
            }
        }
        buf ^= 1;
    }
    cp_async_wait<0>();
}

#ifndef QG_ROW
#define QG_ROW 1
#endif

// Plans a row-team launch of NM matrices of rows of I inputs; false when the
// shape does not suit it (rows not a whole number of warps of chunks, more
// chunks than threads, groups spanning more than four chunks).
template <int NM>
static bool plan_row(int I, int gsh, RowPlan& L)
{
    if (!QG_ROW) return false;
    if (I % (32 * EPL)) return false;
    L.P = I / EPL;
    if (L.P > kRowThreads) return false;
    if (SK == SK_F32 && gsh > 2) return false;           // many lanes would copy one scale
    L.G = kRowThreads / L.P;
    if (L.G > 15) L.G = 15;                              // named barriers 1 .. 15
    L.T = L.P * L.G;
    L.W = L.P / 32;
    constexpr int D = row_depth<NM>();
    constexpr int QS = row_rt<NM>() * NM;        // chunks per slot
    constexpr int VS = 16;                       // values per warp butterfly, at most
    int off = 0;
    L.code_off = off; off += D * QS * L.T * 16;
    L.b_off = off;    off += FMT == FMT_INT3_G64 ? D * QS * L.T * 8 : 0;
    L.sc_off = off;   off += SK == SK_ROW ? 0 : D * QS * L.T * 4;
    L.red_off = off;  off += 2 * (kRowThreads / 32) * VS * 4;
    L.total = off;
    return L.total <= kSmemMax;
}

// Launches the row-team kernel for a dense job when its plan fits; `launched`
// tells whether it did.
template <int NM, int S>
static cudaError_t launch_row_dense(const DenseJob<NM>& dj, int grid, cudaStream_t st, bool& launched)
{
    RowDenseJob<NM> job;
    launched = false;
    const int I = dj.m[0].I;
    if (!plan_row<NM>(I, dj.m[0].gsh, job.plan)) return cudaSuccess;
    launched = true;
    for (int k = 0; k < NM; k++) job.m[k] = dj.m[k];
    job.x = dj.x;
    job.y = dj.y;
    job.ldy = dj.ldy;
    job.act = dj.act;
    job.limit = dj.limit;
    job.rb = code_row_bytes(I);
    job.rbB = I / 8;
    job.sbytes = SK == SK_ROW ? 0 : (SK == SK_E8M0 ? dj.m[0].ngrp : 4 * dj.m[0].ngrp);
    auto kern = k_row<NM, S, RowDenseJob<NM>>;
    static int granted[64];
    cudaError_t e = set_smem(kern, (size_t)job.plan.total, granted);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kRowThreads), (size_t)job.plan.total, st, job);
}
