// qg_moe.cuh -- the routed-expert group as one persistent launch (one format;
// included by qg_fmt_impl.cuh inside its format namespace, after qg_row.cuh).
//
// What it computes (colibri Vulkan guide, xdnf.cn, section 这些开关背后是…API
// 契约: coli_vk_expert_group, a batch of experts' gate+up -> act -> down in one
// submit with the hidden vector kept on the device; colibri docs/vulkan.md, the
// expert tier: every row adds its experts' outputs in rank order, and the
// chain_moe_gv paragraph: one kernel for all of a decode step's experts):
//   out[t] = sum_{r<k} w[t][r] * down_e(act(gate_e x_t, up_e x_t)), e = ids[t][r].
//
// How (GB300-first), one CTA per SM, all of them resident at once:
//  * prologue, in every CTA (each gets the same result): the (token, rank)
//    pairs in the order of (expert, pair index) -- the pairs of one expert are
//    neighbours, so the CTAs that stream its rows for them do so at the same
//    time and the second read is served from L2;
//  * phase A: the gate and up rows of every pair in row blocks, the blocks
//    split evenly over the CTAs; as in the row-team kernel a team of threads
//    owns a row, a thread a fixed 16-byte chunk of it with its slice of x in
//    registers; h = act(g, u) of each (pair, row) goes to the workspace;
//  * a grid barrier: each CTA adds one to a counter once its h rows are
//    written and waits (bounded) until every CTA has;
//  * phase B: the down rows of every pair in row blocks, split the same way,
//    with the thread's slice of that pair's h in registers; z = down h of each
//    (pair, row) goes to the workspace;
//  * a second barrier, then each CTA sums its share of the output rows in
//    rank order, out[t][d] = sum_r w[t][r] z[pair(t, r)][d], and the last CTA
//    to finish clears the counters (the workspace holds zeros before the
//    first call and after every call).
// Each thread's copies run D steps ahead through its ring without a break at
// the phase boundary, so phase B's first rows are in flight while the barrier
// waits.  Every wait is bounded; one that runs out records
// QSTATUS_DEVICE_TIMEOUT, and the CTA still arrives at every later counter so
// the others finish and the counters are cleared.
#pragma once

#ifndef QG_MOE_THREADS
#define QG_MOE_THREADS 384
#endif
constexpr int kMoeThreads = QG_MOE_THREADS;     // a multiple of the rows' chunk counts (64, 192 at the workloads)
constexpr int kMoeMaxPairs = 256;               // s * k of the fused launch
static_assert(kMoeMaxPairs <= kMoeThreads, "the prologue gives each thread at most one pair");
constexpr int kMoeSlot = 4;                     // chunks per ring slot: 2 rows x gate/up, or 4 down rows
constexpr int kMoeRTA = 2, kMoeRTB = 4;         // rows per step of the two phases

// Ring depth in steps.
__host__ __device__ constexpr int moe_depth()
{
    constexpr int d = QG_ROW_SMEM / (kMoeThreads * kMoeSlot * kRowSlot);
    return d > 16 ? 16 : (d < 2 ? 2 : d);
}

// Steps per team round: kMoeVals values per warp butterfly, one per (row, matrix).
#ifndef QG_MOE_VALS
#define QG_MOE_VALS 8
#endif
constexpr int kMoeVals = QG_MOE_VALS;
constexpr int kMoeVA = kMoeVals / (kMoeRTA * 2), kMoeVB = kMoeVals / kMoeRTB;

struct MoePlan {
    int PA, GA, TA, WA;     // phase A: threads per row, teams, active threads, warps per team
    int PB, GB, TB, WB;     // phase B
    int nbA, nbB;           // row blocks per pair (a block: one step of every team)
    int code_off, b_off, sc_off, redA_off, redB_off, tab_off, total;
};

struct MoeJob {
    MoePlan plan;
    Mat gate0, up0, down0;          // expert 0's matrices (w, sc advanced per expert)
    long long up_bytes, up_scales;  // bytes and scale elements of one gate / up matrix
    long long dn_bytes, dn_scales;  // of one down matrix
    long long rbA, rbA_B, sbA;      // gate/up: code (int3: plane A) bytes, plane-B bytes, scale bytes per row
    long long rbB, rbB_B, sbB;      // down: the same
    const float* x;                 // [s][D]
    const int32_t* ids;             // [s][k] (outputs when routed here)
    const float* wts;
    float* out;                     // [s][D]
    float* h;                       // workspace [P][F]
    float* z;                       // workspace [P][D]
    unsigned* ctr;                  // workspace: [0] phase A arrivals, [1] phase B arrivals, [2] finished CTAs,
                                    // [3] a wait ran out
    int* status;                    // optional status word
    int E, D, F, s, k, P;
    int act;
    float limit;
    unsigned long long wait_ns;     // bound of every wait
    int withhold;                   // test hook: CTA 0 does not signal phase A
    // routing inside the prologue (route_kind >= 0): ids / wts are its outputs
    int route_kind;
    const float* logits;
    const float* bias;
    int renorm;
    float route_scale;
};

// Waits until *c >= target (acquire); false after wait_ns.
__device__ __forceinline__ bool wait_count(const unsigned* c, unsigned target, unsigned long long wait_ns)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
    if (v >= target) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t n = 1;; n++) {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
        if (v >= target) return true;
        if ((n & 15u) == 0 && global_ns() - t0 > wait_ns) return false;
        __nanosleep(64);
    }
}

// A wait of this launch ran out: the library's error word now, the call's
// status word from the last CTA (through ctr[3]).
__device__ __forceinline__ void moe_fail(unsigned* ctr)
{
    atomicExch(&g_dev_error, QSTATUS_DEVICE_TIMEOUT);
    atomicOr(&ctr[3], 1u);
}

template <int F_>
__global__ void __launch_bounds__(kMoeThreads, 1) k_moe(const __grid_constant__ MoeJob job)
{
    static_assert(F_ == FMT, "one format per translation unit");
    constexpr int D_ = moe_depth();
    constexpr int QS = kMoeSlot;
    const MoePlan& L = job.plan;
    const int tid = threadIdx.x, lane = tid & 31, warp_global = tid >> 5;
    const uint32_t sbase = smem_base();
    const int G = gridDim.x, c = blockIdx.x;
    const int P = job.P;
    int* s_pair = reinterpret_cast<int*>(reinterpret_cast<char*>(qg_smem4) + L.tab_off);   // pair at sorted position
    int* s_exp = s_pair + kMoeMaxPairs;            // its expert
    int* s_tok = s_exp + kMoeMaxPairs;             // its token
    int* s_pos = s_tok + kMoeMaxPairs;             // sorted position of pair p
    float* s_w = reinterpret_cast<float*>(s_pos + kMoeMaxPairs);   // router weight of pair p
    __shared__ int s_bad, s_ok;

    pdl_wait_prev();                               // ids, weights, x and the workspace come from before
    pdl_allow_next();

    // ---- prologue: routing (optional), ids checked, pairs sorted by (expert, pair) ----
    if (tid == 0) {
        s_bad = 0;
        s_ok = 1;
    }
    __syncthreads();
    if (job.route_kind >= 0) {
        for (int t = warp_global; t < job.s; t += kMoeThreads / 32) {
            int id;
            float w;
            route_token<kFusedRouteMaxE / 32>(job.route_kind, job.logits + (long long)t * job.E, job.bias, job.E,
                                              job.k, job.renorm, job.route_scale, lane, id, w);
            if (lane < job.k) {
                s_exp[t * job.k + lane] = id;
                s_w[t * job.k + lane] = w;
                if (c == 0) {                      // one CTA writes the routing out
                    const_cast<int32_t*>(job.ids)[t * job.k + lane] = id;
                    const_cast<float*>(job.wts)[t * job.k + lane] = w;
                }
            }
        }
    } else {
        for (int p = tid; p < P; p += kMoeThreads) {
            const int e = job.ids[p];
            s_exp[p] = e;
            s_w[p] = job.wts[p];
            if (e < 0 || e >= job.E) s_bad = 1;
        }
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    int e_mine = 0;
    if (!bad) {
        for (int p = tid; p < P; p += kMoeThreads) {
            const int e = s_exp[p];
            int pos = 0;
            for (int q = 0; q < P; q++) {
                const int eq = s_exp[q];
                pos += (eq < e) || (eq == e && q < p);
            }
            s_pos[p] = pos;
        }
    }
    __syncthreads();
    if (!bad) {
        for (int p = tid; p < P; p += kMoeThreads) e_mine = s_exp[p];   // keep before overwriting
    }
    __syncthreads();
    if (!bad) {
        for (int p = tid; p < P; p += kMoeThreads) {
            const int pos = s_pos[p];
            s_pair[pos] = p;
            s_tok[pos] = p / job.k;
        }
    }
    __syncthreads();
    if (!bad) {
        for (int p = tid; p < P; p += kMoeThreads) s_exp[s_pos[p]] = e_mine;   // expert of each sorted position
    }
    __syncthreads();
    if (bad) {
        // an id outside [0, E): out is zeros, the status word says so; no counter is touched
        if (c == 0 && tid == 0 && job.status) *job.status = QSTATUS_BAD_EXPERT_ID;
        const long long d0 = (long long)job.D * c / G, d1 = (long long)job.D * (c + 1) / G;
        for (int t = 0; t < job.s; t++)
            for (long long d = d0 + tid; d < d1; d += kMoeThreads) job.out[(long long)t * job.D + d] = 0.f;
        return;
    }

    // ---- the CTA's row blocks of the two phases ----
    const long long NA = (long long)P * L.nbA, NB = (long long)P * L.nbB;
    const long long a0 = NA * c / G, a1 = NA * (c + 1) / G;
    const long long b0 = NB * c / G, b1 = NB * (c + 1) / G;
    const int nA = (int)(a1 - a0), nB = (int)(b1 - b0), nS = nA + nB;
    // this thread in each phase
    const bool actA = tid < L.TA, actB = tid < L.TB;
    const int gA = tid / L.PA, pA = tid - gA * L.PA;
    const int gB = tid / L.PB, pB = tid - gB * L.PB;

    // ring chunk q of this thread: codes at c_s + q c_q, plane B at b_s + q b_q, scales at s_s + q s_q
    const uint32_t c_s = (uint32_t)L.code_off + (uint32_t)tid * 16u, c_q = kMoeThreads * 16u;
    const uint32_t b_s = (uint32_t)L.b_off + (uint32_t)tid * 8u, b_q = kMoeThreads * 8u;
    const uint32_t s_s = (uint32_t)L.sc_off + (uint32_t)tid * 4u, s_q = kMoeThreads * 4u;

    // A block index as (pair position, row block of that pair), advanced one
    // block at a time (no division in the loops).
    const int posA0 = (int)(a0 / L.nbA), rbA0 = (int)(a0 - (long long)posA0 * L.nbA);
    const int posB0 = (int)(b0 / L.nbB), rbB0 = (int)(b0 - (long long)posB0 * L.nbB);

    // ---- the copy stream: one step = one row block = kMoeSlot chunks of this
    // thread (phase A: rows r = 0, 1 of gate and up, chunk r * 2 + m; phase B:
    // down rows r = 0 .. 3).  The chunks' source addresses are set up once per
    // pair (and for a pair's last, partial block) and advance by a fixed
    // stride otherwise.
    const uint8_t* pc[kMoeSlot];                  // codes (int3: plane A)
    const uint8_t* pb[kMoeSlot];                  // int3 plane B
    const uint8_t* ps[kMoeSlot];                  // scale word
    long long st_c = 0, st_b = 0, st_s = 0;       // per-step advance of the current phase
    unsigned vmask = 0;                           // chunks of the step that hold rows inside the matrix
    int ppos = posA0, prb = rbA0;                 // block of the next step to issue
    int issued = 0;
    auto setup = [&](bool phaseA) {               // the pointers of block (ppos, prb)
        const long long e = s_exp[ppos];
        vmask = 0;
        if (phaseA) {
            const long long GR = (long long)L.GA * kMoeRTA;
            st_c = GR * job.rbA;
            st_b = GR * job.rbA_B;
            st_s = GR * job.sbA;
#pragma unroll
            for (int q = 0; q < kMoeSlot; q++) {
                const int r = q >> 1, m = q & 1;
                const Mat& M = m == 0 ? job.gate0 : job.up0;
                long long row = (long long)prb * GR + gA * kMoeRTA + r;
                if (actA && row < job.F) vmask |= 1u << q;
                if (row >= job.F) row = 0;        // never copied: any valid address
                const uint8_t* base = M.w + e * job.up_bytes;
                pc[q] = base + row * job.rbA + (long long)pA * 16;
                pb[q] = base + (long long)job.F * job.rbA + row * job.rbA_B + (long long)pA * 8;
                if constexpr (SK == SK_E8M0)
                    ps[q] = reinterpret_cast<const uint8_t*>(M.sc) + e * job.up_scales + row * M.ngrp +
                            (((long long)pA >> M.gsh) & ~3ll);
                else
                    ps[q] = reinterpret_cast<const uint8_t*>(M.sc + e * job.up_scales + row * M.ngrp + (pA >> M.gsh));
            }
        } else {
            const long long GR = (long long)L.GB * kMoeRTB;
            st_c = GR * job.rbB;
            st_b = GR * job.rbB_B;
            st_s = GR * job.sbB;
            const Mat& M = job.down0;
            const uint8_t* base = M.w + e * job.dn_bytes;
#pragma unroll
            for (int q = 0; q < kMoeSlot; q++) {
                long long row = (long long)prb * GR + gB * kMoeRTB + q;
                if (actB && row < job.D) vmask |= 1u << q;
                if (row >= job.D) row = 0;
                pc[q] = base + row * job.rbB + (long long)pB * 16;
                pb[q] = base + (long long)job.D * job.rbB + row * job.rbB_B + (long long)pB * 8;
                if constexpr (SK == SK_E8M0)
                    ps[q] = reinterpret_cast<const uint8_t*>(M.sc) + e * job.dn_scales + row * M.ngrp +
                            (((long long)pB >> M.gsh) & ~3ll);
                else
                    ps[q] = reinterpret_cast<const uint8_t*>(M.sc + e * job.dn_scales + row * M.ngrp + (pB >> M.gsh));
            }
        }
    };
    if (nA > 0) setup(true);
    else if (nB > 0) {
        ppos = posB0;
        prb = rbB0;
        setup(false);
    }
    // copies of the next step into the slot whose first chunk is q0
    auto issue = [&](uint32_t q0) {
        const int j = issued;
        if (j < nS) {
#pragma unroll
            for (int q = 0; q < kMoeSlot; q++) {
                const uint32_t qq = q0 + (uint32_t)q;
                if (vmask >> q & 1u) {
                    cp_async16(sbase + c_s + qq * c_q, pc[q]);
                    if constexpr (FMT == FMT_INT3_G64) cp_async8(sbase + b_s + qq * b_q, pb[q]);
                    if constexpr (SK != SK_ROW) cp_async4(sbase + s_s + qq * s_q, ps[q]);
                }
            }
            // the next block: the same pair (a fixed stride), or a new pair / phase / last block
            const bool inA = j < nA;
            const int nb = inA ? L.nbA : L.nbB;
            if (j + 1 == nA) {
                ppos = posB0;
                prb = rbB0;
                if (nB > 0) setup(false);
            } else if (++prb == nb || prb == nb - 1) {
                if (prb == nb) {
                    prb = 0;
                    ppos++;
                }
                if (j + 1 < nS) setup(inA);
            } else {
#pragma unroll
                for (int q = 0; q < kMoeSlot; q++) {
                    pc[q] += st_c;
                    if constexpr (FMT == FMT_INT3_G64) pb[q] += st_b;
                    if constexpr (SK != SK_ROW) ps[q] += st_s;
                }
            }
        }
        issued++;
        cp_async_commit();
    };
#pragma unroll 1
    for (int k = 0; k < D_; k++) issue((uint32_t)(k * QS));

    float* redA = reinterpret_cast<float*>(reinterpret_cast<char*>(qg_smem4) + L.redA_off);
    float* redB = reinterpret_cast<float*>(reinterpret_cast<char*>(qg_smem4) + L.redB_off);
    uint32_t slot = 0;
    bool ok = true;

    // ---- phase A: gate and up rows, h = act(g, u) ----
    {
        float2 xr[EPL / 2];
        int tok_loaded = -1;
        int buf = 0;
        int cpos = posA0, crb = rbA0;             // block of the next step to consume
        for (int j0 = 0; j0 < nA; j0 += kMoeVA) {
            const int rpos = cpos, rrb = crb;     // the round's first block
            float vb[kMoeVals];
#pragma unroll
            for (int i = 0; i < kMoeVals; i++) vb[i] = 0.f;
#pragma unroll
            for (int v = 0; v < kMoeVA; v++) {
                const int j = j0 + v;
                if (j < nA) {
                    cp_async_wait<D_ - 1>();
                    Chunk<F_> ch[kMoeRTA][2];
                    [[maybe_unused]] float sc[kMoeRTA][2];
#pragma unroll
                    for (int r = 0; r < kMoeRTA; r++)
#pragma unroll
                        for (int m = 0; m < 2; m++) {
                            const uint32_t q = slot + (uint32_t)(r * 2 + m);
                            if constexpr (FMT == FMT_INT3_G64) {
                                ch[r][m].a = lds16(c_s + q * c_q);
                                ch[r][m].b = lds8(b_s + q * b_q);
                            } else {
                                ch[r][m].w = lds16(c_s + q * c_q);
                            }
                            if constexpr (SK == SK_E8M0)
                                sc[r][m] = e8m0_to_f32(__byte_perm(lds_u32(s_s + q * s_q), 0u,
                                                                   0x4440u + (uint32_t)(pA & 3)));
                            else if constexpr (SK == SK_F32)
                                sc[r][m] = lds_f32(s_s + q * s_q);
                        }
                    issue(slot);
                    slot = slot + QS == (uint32_t)(D_ * QS) ? 0u : slot + QS;
                    const int pos = cpos;
                    if (++crb == L.nbA) {
                        crb = 0;
                        cpos++;
                    }
                    if (actA) {
                        const int tok = s_tok[pos];
                        if (tok != tok_loaded) {          // the pair's token: its x slice into registers
                            const float4* src = reinterpret_cast<const float4*>(job.x + (long long)tok * job.D +
                                                                                (long long)pA * EPL);
#pragma unroll
                            for (int q = 0; q < EPL / 4; q++) {
                                const float4 f = src[q];
                                xr[2 * q] = make_float2(f.x, f.y);
                                xr[2 * q + 1] = make_float2(f.z, f.w);
                            }
                            tok_loaded = tok;
                        }
#pragma unroll
                        for (int r = 0; r < kMoeRTA; r++)
#pragma unroll
                            for (int m = 0; m < 2; m++) {
                                const float dsum = chunk_dot<F_>(ch[r][m], xr);
                                vb[(v * kMoeRTA + r) * 2 + m] = SK == SK_ROW ? dsum : dsum * sc[r][m];
                            }
                    }
                }
            }
            if (!actA) continue;
            const float rv = warp_reduce_scatter<kMoeVals>(vb, lane);
            const int idx = reduce_scatter_index<kMoeVals>(lane);
            float* rb = redA + (size_t)buf * (kMoeThreads / 32) * 16;
            if (lane < kMoeVals) rb[warp_global * 16 + idx] = rv;
            asm volatile("bar.sync %0, %1;" :: "r"(1 + gA), "r"(L.PA) : "memory");
            if (pA < kMoeVA * kMoeRTA) {
                const int v = pA / kMoeRTA, r = pA - v * kMoeRTA;
                const int j = j0 + v;
                if (j < nA) {
                    int pos = rpos, rb_ = rrb + v;
                    while (rb_ >= L.nbA) {
                        rb_ -= L.nbA;
                        pos++;
                    }
                    const long long row = (long long)rb_ * (L.GA * kMoeRTA) + gA * kMoeRTA + r;
                    if (row < job.F) {
                        float tot[2];
#pragma unroll
                        for (int m = 0; m < 2; m++) {
                            float t = 0.f;
                            for (int w = 0; w < L.WA; w++) t += rb[(gA * L.WA + w) * 16 + pA * 2 + m];
                            if constexpr (SK == SK_ROW) {
                                const Mat& M = m == 0 ? job.gate0 : job.up0;
                                t *= ldg_f32(M.sc + (long long)s_exp[pos] * job.up_scales + row);
                            }
                            tot[m] = t;
                        }
                        float gv = tot[0], u = tot[1];
                        if (job.act == QACT_SWIGLU_CLAMPED) {
                            gv = fminf(gv, job.limit);
                            u = fminf(fmaxf(u, -job.limit), job.limit);
                        }
                        job.h[(long long)pos * job.F + row] = gv / (1.0f + expf(-gv)) * u;
                    }
                }
            }
            buf ^= 1;
        }
    }

    // ---- grid barrier: every CTA's h rows written ----
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        if (!(job.withhold && c == 0)) atomicAdd(&job.ctr[0], 1u);
        if (!wait_count(&job.ctr[0], (unsigned)G, job.wait_ns)) {
            moe_fail(job.ctr);
            s_ok = 0;
        }
        __threadfence();
    }
    __syncthreads();
    ok = s_ok != 0;

    // ---- phase B: down rows, z = down h ----
    {
        float2 xr[EPL / 2];
        int pos_loaded = -1;
        int buf = 0;
        int cpos = posB0, crb = rbB0;
        for (int j0 = nA; j0 < nS; j0 += kMoeVB) {
            const int rpos = cpos, rrb = crb;
            float vb[kMoeVals];
#pragma unroll
            for (int i = 0; i < kMoeVals; i++) vb[i] = 0.f;
#pragma unroll
            for (int v = 0; v < kMoeVB; v++) {
                const int j = j0 + v;
                if (j < nS) {
                    cp_async_wait<D_ - 1>();
                    Chunk<F_> ch[kMoeRTB];
                    [[maybe_unused]] float sc[kMoeRTB];
#pragma unroll
                    for (int r = 0; r < kMoeRTB; r++) {
                        const uint32_t q = slot + (uint32_t)r;
                        if constexpr (FMT == FMT_INT3_G64) {
                            ch[r].a = lds16(c_s + q * c_q);
                            ch[r].b = lds8(b_s + q * b_q);
                        } else {
                            ch[r].w = lds16(c_s + q * c_q);
                        }
                        if constexpr (SK == SK_E8M0)
                            sc[r] = e8m0_to_f32(__byte_perm(lds_u32(s_s + q * s_q), 0u, 0x4440u + (uint32_t)(pB & 3)));
                        else if constexpr (SK == SK_F32)
                            sc[r] = lds_f32(s_s + q * s_q);
                    }
                    issue(slot);
                    slot = slot + QS == (uint32_t)(D_ * QS) ? 0u : slot + QS;
                    const int pos = cpos;
                    if (++crb == L.nbB) {
                        crb = 0;
                        cpos++;
                    }
                    if (actB && ok) {
                        if (pos != pos_loaded) {          // the pair's h slice into registers
                            const float4* src = reinterpret_cast<const float4*>(job.h + (long long)pos * job.F +
                                                                                (long long)pB * EPL);
#pragma unroll
                            for (int q = 0; q < EPL / 4; q++) {
                                const float4 f = __ldcg(src + q);    // written by this launch: no read-only path
                                xr[2 * q] = make_float2(f.x, f.y);
                                xr[2 * q + 1] = make_float2(f.z, f.w);
                            }
                            pos_loaded = pos;
                        }
#pragma unroll
                        for (int r = 0; r < kMoeRTB; r++) {
                            const float dsum = chunk_dot<F_>(ch[r], xr);
                            vb[v * kMoeRTB + r] = SK == SK_ROW ? dsum : dsum * sc[r];
                        }
                    }
                }
            }
            if (!actB || !ok) continue;
            const float rv = warp_reduce_scatter<kMoeVals>(vb, lane);
            const int idx = reduce_scatter_index<kMoeVals>(lane);
            float* rb = redB + (size_t)buf * (kMoeThreads / 32) * 16;
            if (lane < kMoeVals) rb[warp_global * 16 + idx] = rv;
            asm volatile("bar.sync %0, %1;" :: "r"(1 + L.GA + gB), "r"(L.PB) : "memory");
            if (pB < kMoeVB * kMoeRTB) {
                const int v = pB / kMoeRTB, r = pB - v * kMoeRTB;
                const int j = j0 + v;
                if (j < nS) {
                    int pos = rpos, rb_ = rrb + v;
                    while (rb_ >= L.nbB) {
                        rb_ -= L.nbB;
                        pos++;
                    }
                    const long long row = (long long)rb_ * (L.GB * kMoeRTB) + gB * kMoeRTB + r;
                    if (row < job.D) {
                        float t = 0.f;
                        for (int w = 0; w < L.WB; w++) t += rb[(gB * L.WB + w) * 16 + pB];
                        if constexpr (SK == SK_ROW)
                            t *= ldg_f32(job.down0.sc + (long long)s_exp[pos] * job.dn_scales + row);
                        job.z[(long long)pos * job.D + row] = t;
                    }
                }
            }
            buf ^= 1;
        }
    }
    cp_async_wait<0>();

    // ---- second barrier: every z row written; then the rank-order sums ----
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        atomicAdd(&job.ctr[1], 1u);
        if (!wait_count(&job.ctr[1], (unsigned)G, job.wait_ns)) {
            moe_fail(job.ctr);
            s_ok = 0;
        }
        __threadfence();
    }
    __syncthreads();
    {
        const long long d0 = (long long)job.D * c / G, d1 = (long long)job.D * (c + 1) / G;
        const long long nd = d1 - d0;
        for (long long i = tid; i < (long long)job.s * nd; i += kMoeThreads) {
            const int t = (int)(i / nd);
            const long long d = d0 + (i - (long long)t * nd);
            float acc = 0.f;
            if (s_ok)
                for (int r = 0; r < job.k; r++) {
                    const int p = t * job.k + r;
                    acc = fmaf(s_w[p], __ldcg(job.z + (long long)s_pos[p] * job.D + d), acc);
                }
            job.out[(long long)t * job.D + d] = acc;
        }
    }

    // ---- the last CTA out writes the status word and clears the counters ----
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&job.ctr[2], 1u);
        if (prev == (unsigned)G - 1) {
            const unsigned failed = atomicExch(&job.ctr[3], 0u);
            if (job.status) *job.status = failed ? QSTATUS_DEVICE_TIMEOUT : QSTATUS_OK;
            job.ctr[0] = 0;
            job.ctr[1] = 0;
            job.ctr[2] = 0;
            __threadfence();
        }
    }
}

#ifndef QG_MOE
#define QG_MOE 1
#endif

// Plans the fused launch for rows of D (gate/up) and F (down) inputs; false
// when the shapes do not suit it (rows not whole warp steps of chunks, more
// chunks than threads, groups spanning more than four chunks).
static bool plan_moe(int D, int F, int gsh_up, int gsh_dn, MoePlan& L)
{
    if (!QG_MOE) return false;
    if (D % (32 * EPL) || F % (32 * EPL)) return false;
    L.PA = D / EPL;
    L.PB = F / EPL;
    if (L.PA > kMoeThreads || L.PB > kMoeThreads) return false;
    if (SK == SK_F32 && (gsh_up > 2 || gsh_dn > 2)) return false;
    L.GA = kMoeThreads / L.PA;
    L.GB = kMoeThreads / L.PB;
    if (L.GA > 7) L.GA = 7;                        // named barriers 1 .. GA, GA + 1 .. GA + GB (<= 15)
    if (L.GA + L.GB > 15) L.GB = 15 - L.GA;
    L.TA = L.PA * L.GA;
    L.TB = L.PB * L.GB;
    L.WA = L.PA / 32;
    L.WB = L.PB / 32;
    L.nbA = (F + L.GA * kMoeRTA - 1) / (L.GA * kMoeRTA);
    L.nbB = (D + L.GB * kMoeRTB - 1) / (L.GB * kMoeRTB);
    constexpr int D_ = moe_depth();
    int off = 0;
    L.code_off = off; off += D_ * kMoeSlot * kMoeThreads * 16;
    L.b_off = off;    off += FMT == FMT_INT3_G64 ? D_ * kMoeSlot * kMoeThreads * 8 : 0;
    L.sc_off = off;   off += SK == SK_ROW ? 0 : D_ * kMoeSlot * kMoeThreads * 4;
    L.redA_off = off; off += 2 * (kMoeThreads / 32) * 16 * 4;
    L.redB_off = off; off += 2 * (kMoeThreads / 32) * 16 * 4;
    L.tab_off = off;  off += 5 * kMoeMaxPairs * 4;
    L.total = off;
    return L.total <= kSmemMax;
}
