// qg_moe.cuh -- the routed-expert group as one persistent launch (one format;
// included by qg_fmt_impl.cuh inside its format namespace, after qg_tile.cuh).
//
// What it computes (colibri Vulkan guide, xdnf.cn, section 这些开关背后是…API
// 契约: coli_vk_expert_group, a batch of experts' gate+up -> act -> down in one
// submit with the hidden vector kept on the device; colibri docs/vulkan.md, the
// expert tier: every row adds its experts' outputs in rank order, and the
// chain_moe_gv paragraph: one kernel for all of a decode step's experts):
//   out[t] = sum_{r<k} w[t][r] * down_e(act(gate_e x_t, up_e x_t)), e = ids[t][r].
//
// How (GB300-first), one CTA per SM, all of them resident at once:
//  * prologue, in every CTA (each gets the same result, nothing is waited
//    for): routing (optional), the (token, rank) pairs sorted by (expert,
//    pair index), cut into batches of at most smax pairs of one expert, and
//    the CTA's share of each phase's row tiles (a tile of a batch of n pairs
//    costs n);
//  * phase A: the tile kernel's streaming pass over the gate and up rows of
//    the batches -- every warp streams its own row tiles through a ring of
//    tensor copies, the batch's activation rows staged once per CTA in shared
//    memory -- storing h = act(g, u) per (pair, row) in the workspace; each
//    warp then adds the number of row tiles it finished to its batch's
//    counter (a release reduction);
//  * each warp issues its first down-row slices into its ring as soon as its
//    phase-A slices are consumed (the down weights do not depend on h);
//  * phase B: the same pass over the down rows against the pairs' h rows,
//    staged from L2 once the batch's counter holds all its phase-A tiles
//    (thread 0 waits, bounded; a CTA thus waits only for the warps that
//    computed the batches it needs), storing z = down h per (pair, row);
//  * a second barrier, then each CTA sums its share of the output columns in
//    rank order, out[t][d] = sum_r w[t][r] z[pair(t, r)][d], and the last CTA
//    to finish clears the counters (the workspace holds zeros before the
//    first call and after every call).
// The passes are the tile kernel's own, so every h, z and out value has the
// bits of the four-launch path.  Every wait is bounded; one that runs out
// records QSTATUS_DEVICE_TIMEOUT, and the CTA still arrives at the closing
// counters so the others finish and the counters are cleared.
#pragma once

constexpr int kMoeMaxPairs = 256;               // s * k of the fused launch
static_assert(kMoeMaxPairs <= kTileThreads, "the prologue gives each thread at most one pair");
static_assert(kMoeMaxPairs <= kDoneWords, "one workspace counter per batch");
// pair tables: expert, weight, sorted position per pair; token, expert, batch
// size per sorted position; first position per batch (+1); batches; flags
constexpr int kMoeTabBytes = 6 * kMoeMaxPairs * 4 + (kMoeMaxPairs + 4) * 4 + kMoeMaxPairs * 16 + 64 * 4;

struct MoeJob {
    TileLayout la, lb;              // slot layouts of phase A (gate/up) and phase B (down)
    CUtensorMap tma[6];             // phase A: gate codes, plane B, scales; up codes, plane B, scales
    CUtensorMap tmb[3];             // phase B: down
    long long rmA[3], raA[3];       // tensor row of expert e's row r: e * rm + ra + r, per piece
    long long rmB[3], raB[3];
    Mat gate0, up0, down0;          // expert 0's matrices (w, sc advanced per expert)
    long long up_bytes, up_scales;  // bytes and scale elements of one gate / up matrix
    long long dn_bytes, dn_scales;  // of one down matrix
    const float* x;                 // [s][D]
    const int32_t* ids;             // [s][k] (unused when routed here)
    const float* wts;
    int32_t* ids_out;               // routed here: where CTA 0 writes the routing
    float* wts_out;
    float* out;                     // [s][D]
    float* h;                       // workspace [P][F], by sorted pair position
    float* z;                       // workspace [P][D]
    unsigned* ctr;                  // workspace: [1] phase B arrivals, [2] finished CTAs, [3] a wait ran out
    unsigned* done;                 // workspace: phase-A row tiles finished per batch
    int* status;                    // optional status word
    int E, D, F, s, k, P, smax;
    int tab_off;                    // shared offset of the pair tables
    int act;
    float limit;
    unsigned long long wait_ns;     // bound of every grid-barrier wait
    int withhold;                   // test hook: CTA 0 does not count its phase-A tiles
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

// The two passes' views of the launch: batches and tokens from the prologue's
// shared tables, tensor maps from the launch's parameters.  Phase A tells
// each batch's counter how many of its row tiles a warp has finished (h rows
// written); phase B stages a batch's h rows once its counter is complete, so
// a CTA waits only for the warps that computed the batches it needs.
struct MoeUpView {
    static constexpr bool kLoopS = true;       // one pass of arithmetic per pair of a batch
    static constexpr bool kWaitFirst = true;   // (the prologue waited)
    static constexpr bool kFreshX = false;     // x comes from before the launch
    static constexpr bool kSignals = true;
    static constexpr bool kWaits = false;
    const MoeJob& g;
    const int4* bt;                            // (expert, first sorted position, pairs, 0) per batch
    const int* tok;                            // token of each sorted position
    int act;
    float limit;
    // the warp's h rows of batch b are stored: lane 0 publishes its tile count
    // with a release reduction (after __syncwarp, the release covers every
    // lane's stores; phase B reads the counter with acquire loads)
    __device__ void warp_done(int b, int tiles) const
    {
        __syncwarp();
        if ((threadIdx.x & 31) == 0 && !(g.withhold && blockIdx.x == 0))
            asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(&g.done[b]), "r"((unsigned)tiles)
                         : "memory");
    }
    __device__ void segment_poll(int) const {}
    __device__ bool segment_ready() const { return true; }
    __device__ const TileLayout& layout() const { return g.la; }
    __device__ const CUtensorMap* tmap(int i) const { return &g.tma[i]; }
    __device__ long long rmul(int p) const { return g.rmA[p]; }
    __device__ long long radd(int p) const { return g.raA[p]; }
    __device__ long long rows_per() const { return g.F; }
    __device__ int batch_S(int b) const { return bt[b].z; }
    __device__ long long expert_of(int b) const { return bt[b].x; }
    __device__ void mats(int b, Mat (&out)[2]) const
    {
        const long long e = bt[b].x;
        out[0] = g.gate0;
        out[0].w += e * g.up_bytes;
        out[0].sc = sc_ptr<SK>(out[0].sc, e * g.up_scales);
        out[1] = g.up0;
        out[1].w += e * g.up_bytes;
        out[1].sc = sc_ptr<SK>(out[1].sc, e * g.up_scales);
    }
    __device__ const float* xrow(int b, int s) const { return g.x + (long long)tok[bt[b].y + s] * g.D; }
    __device__ void store(int b, int s, long long row, float v) const
    {
        g.h[(long long)(bt[b].y + s) * g.F + row] = v;
    }
    __device__ int width() const { return g.D; }
};

struct MoeDownView {
    static constexpr bool kLoopS = true;
    static constexpr bool kWaitFirst = true;
    static constexpr bool kFreshX = true;      // h was written by this launch's CTAs: read through L2
    static constexpr bool kSignals = false;
    static constexpr bool kWaits = true;
    const MoeJob& g;
    const int4* bt;
    int act;                                   // (unused: one matrix)
    float limit;
    unsigned need;                             // phase-A row tiles per batch
    int* flag;                                 // shared: the last wait's outcome
    __device__ void warp_done(int, int) const {}
    // thread 0 waits (bounded) until all of batch b's h rows are written (one
    // poller per CTA keeps the counters' L2 line cool)
    __device__ void segment_poll(int b) const
    {
        if (threadIdx.x == 0) *flag = wait_count(&g.done[b], need, g.wait_ns) ? 1 : 0;
    }
    __device__ bool segment_ready() const { return *flag != 0; }
    __device__ const TileLayout& layout() const { return g.lb; }
    __device__ const CUtensorMap* tmap(int i) const { return &g.tmb[i]; }
    __device__ long long rmul(int p) const { return g.rmB[p]; }
    __device__ long long radd(int p) const { return g.raB[p]; }
    __device__ long long rows_per() const { return g.D; }
    __device__ int batch_S(int b) const { return bt[b].z; }
    __device__ long long expert_of(int b) const { return bt[b].x; }
    __device__ void mats(int b, Mat (&out)[1]) const
    {
        const long long e = bt[b].x;
        out[0] = g.down0;
        out[0].w += e * g.dn_bytes;
        out[0].sc = sc_ptr<SK>(out[0].sc, e * g.dn_scales);
    }
    __device__ const float* xrow(int b, int s) const { return g.h + (long long)(bt[b].y + s) * g.F; }
    __device__ void store(int b, int s, long long row, float v) const
    {
        g.z[(long long)(bt[b].y + s) * g.D + row] = v;
    }
    __device__ int width() const { return g.F; }
};

// A wait of this launch ran out: the library's error word now, the call's
// status word from the last CTA (through ctr[3]).
__device__ __forceinline__ void moe_fail(unsigned* ctr)
{
    atomicExch(&g_dev_error, QSTATUS_DEVICE_TIMEOUT);
    atomicOr(&ctr[3], 1u);
}

// First row tile of CTA c of G over nb batches of tpb tiles (first[b]: pairs
// before batch b, first[nb] = P): where the cost so far reaches P tpb c / G,
// a tile of a batch of n pairs costing n.
__device__ __forceinline__ int moe_bound(const int* first, int nb, int P, int tpb, int c, int G)
{
    if (c >= G) return nb * tpb;
    const long long x = (long long)P * tpb * c / G;
    int lo = 0, hi = nb - 1;                       // last batch starting at or before x
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)first[mid] * tpb <= x) lo = mid;
        else hi = mid - 1;
    }
    const long long n = first[lo + 1] - first[lo];
    return (int)((long long)lo * tpb + (x - (long long)first[lo] * tpb) / n);
}

// SM: the most pairs a batch holds (job.smax <= SM): the passes keep SM
// accumulator sets, so a launch whose batches hold one pair carries one.
template <int F_, int SM>
__global__ void __launch_bounds__(kTileThreads, 1) k_moe(const __grid_constant__ MoeJob job)
{
    static_assert(F_ == FMT, "one format per translation unit");
    constexpr int NT = kTileThreads;
    using PhaseA = TilePhase<2, SM, MoeUpView>;
    using PhaseB = TilePhase<1, SM, MoeDownView>;
    const int tid = threadIdx.x, lane = tid & 31;
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const uint32_t sbase = smem_base();
    const int G = gridDim.x, c = blockIdx.x;
    const int P = job.P, k = job.k;
    char* tab = reinterpret_cast<char*>(qg_smem4) + job.tab_off;
    int* s_exp = reinterpret_cast<int*>(tab);          // [pair] expert
    float* s_w = reinterpret_cast<float*>(s_exp + kMoeMaxPairs);   // [pair] router weight
    int* s_pos = reinterpret_cast<int*>(s_w + kMoeMaxPairs);       // [pair] sorted position
    int* s_tok = s_pos + kMoeMaxPairs;                 // [position] token
    int* s_sexp = s_tok + kMoeMaxPairs;                // [position] expert
    int* s_nstart = s_sexp + kMoeMaxPairs;             // [position] pairs of the batch it starts, or 0
    int* s_first = s_nstart + kMoeMaxPairs;            // [batch] first position; [nb] = P
    int4* s_bt = reinterpret_cast<int4*>(s_first + kMoeMaxPairs + 4);
    int* s_misc = reinterpret_cast<int*>(s_bt + kMoeMaxPairs);
    // s_misc: [0] a bad id, [1] batches, [2] grid waits ok, [3] a wait of this CTA ran out, [4..7] tile
    // bounds, [8] phase B's batch wait, [16..32) starts per warp

    pdl_wait_prev();                               // ids, weights, x and the workspace come from before
    pdl_allow_next();
    if (sbase & 127u) {                            // tensor copies land on 128-byte boundaries (the same in
        if (c == 0 && tid == 0) {                  // every CTA: none touches a counter)
            atomicExch(&g_dev_error, QSTATUS_DEVICE_TIMEOUT);
            if (job.status) *job.status = QSTATUS_DEVICE_TIMEOUT;
        }
        return;
    }

    // ---- prologue: routing (optional), ids checked, pairs sorted by (expert, pair), batches ----
    if (tid == 0) {
        s_misc[0] = 0;
        s_misc[2] = 1;
        s_misc[3] = 0;
    }
    __syncthreads();
    if (job.route_kind >= 0) {
        for (int t = warp; t < job.s; t += NT / 32) {
            int id;
            float w;
            route_token<kFusedRouteMaxE / 32>(job.route_kind, job.logits + (long long)t * job.E, job.bias, job.E, k,
                                              job.renorm, job.route_scale, lane, id, w);
            if (lane < k) {
                s_exp[t * k + lane] = id;
                s_w[t * k + lane] = w;
                if (c == 0) {                      // one CTA writes the routing out
                    job.ids_out[t * k + lane] = id;
                    job.wts_out[t * k + lane] = w;
                }
            }
        }
    } else if (tid < P) {
        const int e = job.ids[tid];
        s_exp[tid] = e;
        s_w[tid] = job.wts[tid];
        if (e < 0 || e >= job.E) s_misc[0] = 1;
    }
    __syncthreads();
    if (s_misc[0]) {
        // an id outside [0, E): out is zeros, the status word says so; no counter is touched
        if (c == 0 && tid == 0 && job.status) *job.status = QSTATUS_BAD_EXPERT_ID;
        const long long d0 = (long long)job.D * c / G, d1 = (long long)job.D * (c + 1) / G;
        for (int t = 0; t < job.s; t++)
            for (long long d = d0 + tid; d < d1; d += NT) job.out[(long long)t * job.D + d] = 0.f;
        return;
    }
    if (tid < P) {
        // the pair's sorted position; the pairs of its expert before it start a
        // new batch every smax pairs
        const int e = s_exp[tid];
        int pos = 0, lo = 0, hi = 0;
        for (int q = 0; q < P; q++) {
            const int eq = s_exp[q];
            lo += eq < e;
            hi += eq <= e;
            pos += (eq < e) || (eq == e && q < tid);
        }
        s_pos[tid] = pos;
        s_tok[pos] = tid / k;
        s_sexp[pos] = e;
        const int n = hi - pos < job.smax ? hi - pos : job.smax;
        s_nstart[pos] = (pos - lo) % job.smax == 0 ? n : 0;
    }
    __syncthreads();
    {
        // batch index of each start: a scan over sorted positions
        const int n = tid < P ? s_nstart[tid] : 0;
        const unsigned m = __ballot_sync(0xffffffffu, n > 0);
        if (lane == 0) s_misc[16 + warp] = __popc(m);
        __syncthreads();
        int before = 0, all = 0;
        for (int w = 0; w < NT / 32; w++) {
            const int cw = s_misc[16 + w];
            before += w < warp ? cw : 0;
            all += cw;
        }
        if (n > 0) {
            const int bi = before + __popc(m & ((1u << lane) - 1u));
            s_bt[bi] = make_int4(s_sexp[tid], tid, n, 0);
            s_first[bi] = tid;
        }
        if (tid == 0) {
            s_first[all] = P;
            s_misc[1] = all;
        }
    }
    __syncthreads();
    const int nb = s_misc[1];
    const int tpbA = (int)((job.F + PhaseA::R - 1) / PhaseA::R);
    const int tpbB = (int)((job.D + PhaseB::R - 1) / PhaseB::R);
    if (tid < 4) {
        const int tpb = tid < 2 ? tpbA : tpbB;
        s_misc[4 + tid] = moe_bound(s_first, nb, P, tpb, c + (tid & 1), G);
    }
    __syncthreads();
    const int a0 = s_misc[4], a1 = s_misc[5], b0 = s_misc[6], b1 = s_misc[7];
    float* xs = reinterpret_cast<float*>(qg_smem4);

    // ---- phase A: gate and up rows, h = act(g, u) ----
    PhaseA::init_barriers(job.la, sbase, warp);    // both passes' barriers (separate words)
    PhaseB::init_barriers(job.lb, sbase, warp);
    __syncthreads();
    {
        const MoeUpView up{job, s_bt, s_tok, job.act, job.limit};
        PhaseA pa(up, sbase, warp, a0, a1, tpbA);
        pa.prime();
        if (!pa.run(xs)) {
            pa.drain();
            s_misc[3] = 1;                         // a wait of this CTA ran out
        }
    }
    // The warp's ring is idle now (every phase A slice it issued was
    // consumed), and each warp's ring region is the same in both passes: it
    // issues its first down slices at once (the down weights do not depend
    // on h); phase B then waits per batch for the h rows it stages.
    const MoeDownView dn{job, s_bt, job.act, job.limit, (unsigned)tpbA, s_misc + 8};
    PhaseB pb(dn, sbase, warp, b0, b1, tpbB);
    pb.prime();
    __syncthreads();                               // every warp is done with phase A's staged x

    // ---- phase B: down rows, z = down h (all warps of the CTA, or none) ----
    if (s_misc[3] == 0) {
        if (!pb.run(xs)) {
            pb.drain();
            s_misc[3] = 1;
        }
    } else {
        pb.drain();
    }
    __syncthreads();
    if (tid == 0 && (s_misc[2] == 0 || s_misc[3] != 0)) {
        moe_fail(job.ctr);
        s_misc[2] = 0;
    }

    // ---- second barrier: every z row written; then the rank-order sums ----
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        atomicAdd(&job.ctr[1], 1u);
        if (!wait_count(&job.ctr[1], (unsigned)G, job.wait_ns)) {
            moe_fail(job.ctr);
            s_misc[2] = 0;
        }
        __threadfence();
    }
    __syncthreads();
    {
        const bool all_ok = s_misc[2] != 0;
        const long long d0 = (long long)job.D * c / G, d1 = (long long)job.D * (c + 1) / G;
        const long long nd = d1 - d0;
        for (long long i = tid; i < (long long)job.s * nd; i += NT) {
            const int t = (int)(i / nd);
            const long long d = d0 + (i - (long long)t * nd);
            float acc = 0.f;
            if (all_ok)
                for (int r = 0; r < k; r++) {
                    const int p = t * k + r;
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
            for (int b = 0; b < nb; b++) job.done[b] = 0;
            job.ctr[1] = 0;
            job.ctr[2] = 0;
            __threadfence();
        }
    }
}

#ifndef QG_MOE
#define QG_MOE 1
#endif

// Launches k_moe<FMT, SM> (its own record of the shared memory granted).
template <int SM>
static cudaError_t launch_moe_sm(const MoeJob& job, int grid, cudaStream_t st)
{
    const size_t smem = (size_t)job.la.total;
    static int granted[64];
    cudaError_t e = set_smem(k_moe<FMT, SM>, smem, granted);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_moe<FMT, SM>, dim3(grid), dim3(kTileThreads), smem, st, job);
}

// Launches k_moe with the fewest accumulator sets that hold job.smax pairs.
static cudaError_t launch_moe(const MoeJob& job, int grid, cudaStream_t st)
{
    if (job.smax <= 1) return launch_moe_sm<1>(job, grid, st);
    if (job.smax <= 2) return launch_moe_sm<2>(job, grid, st);
    return launch_moe_sm<kExpertSmax>(job, grid, st);
}

// Plans the fused launch's shared memory: the staged activation rows (smax
// rows of max(D, F) inputs), one ring region that phase A's and then phase
// B's slots share, each phase's barriers, the pair tables.  False when the
// shapes do not suit the tile passes or fewer than two slots per warp fit.
static bool plan_moe(int D, int F, int gs_up, int gs_dn, int smax, MoeJob& j)
{
    if (!QG_MOE) return false;
    constexpr int RA = TilePhase<2, 1, MoeUpView>::R;     // (one-pair passes: the height does not depend on SM)
    constexpr int RB = TilePhase<1, 1, MoeDownView>::R;
    if (!plan_tile(2, RA, D, gs_up, smax, j.la) || !plan_tile(1, RB, F, gs_dn, smax, j.lb)) return false;
    const int NW = kTileWarps;
    const int ring_off = j.la.ring_off > j.lb.ring_off ? j.la.ring_off : j.lb.ring_off;
    const int bars = 8 * (NW * QG_TILE_PMAX + 1);
    const int avail = kSmemMax - ring_off - 2 * bars - kMoeTabBytes - 16;
    int PA = avail / (NW * j.la.slot_bytes), PB = avail / (NW * j.lb.slot_bytes);
    if (PA > QG_TILE_PMAX) PA = QG_TILE_PMAX;
    if (PB > QG_TILE_PMAX) PB = QG_TILE_PMAX;
    if (PA < 2 || PB < 2) return false;
    const int ring = NW * (PA * j.la.slot_bytes > PB * j.lb.slot_bytes ? PA * j.la.slot_bytes : PB * j.lb.slot_bytes);
    j.la.P = PA;
    j.lb.P = PB;
    j.la.warp_bytes = j.lb.warp_bytes = ring / NW;   // a warp's region is the same in both passes
    j.la.ring_off = j.lb.ring_off = ring_off;
    j.la.bar_off = ring_off + ring;
    j.lb.bar_off = j.la.bar_off + 8 * (NW * PA + 1);
    j.tab_off = align_up(j.lb.bar_off + 8 * (NW * PB + 1), 16);
    j.la.total = j.lb.total = j.tab_off + kMoeTabBytes;
    return j.la.total <= kSmemMax;
}
