// qg_tile.cuh -- the tile-streaming kernel (one format; included by
// qg_fmt_impl.cuh inside its format namespace).
//
// Every warp streams its own row tiles.  A tile is R rows of each of the
// job's NM matrices; it is read one slice at a time -- 32 lanes x EPL inputs,
// that is 512 bytes of codes per row, plus int3 plane B and the slice's
// scales -- by 2-D tensor copies into the warp's ring of P shared-memory
// slots.  Lane 0 keeps P slices in flight: as soon as the warp is done with a
// slot it issues the slice P ahead into it.  Each slot has its own mbarrier,
// so warps never wait for one another, except where the staged activation
// rows change (a new batch of an expert job).
//
// The CTA takes the tiles [T c / G, T (c+1) / G) of the job's batches laid end
// to end (T tiles in all, G CTAs); inside a batch its warps take the tiles
// round-robin.  A batch's last tile may reach past the batch's rows: those
// rows are read (zeros past the end of the tensor) and never stored.  Rows are
// zero-padded to whole slices by the tensor copies, and the staged activation
// rows are padded with zeros to match, so a lane never tests a bound.  The
// activation rows are staged lane-interleaved (quad j of the 32 lanes' chunks
// side by side), so every x load is conflict-free at a fixed offset.
//
// A row's slices are accumulated in order, lane by lane, exactly as in the
// per-warp ring kernel, so both kernels give the same bits.
#pragma once

// Error word of this format's kernels: QSTATUS_DEVICE_TIMEOUT after a wait
// ran out (the launch's results are then undefined).
static __device__ int g_dev_error;

__device__ __forceinline__ void tile_fail(int* status_dev)
{
    atomicExch(&g_dev_error, QSTATUS_DEVICE_TIMEOUT);
    if (status_dev) atomicExch(status_dev, QSTATUS_DEVICE_TIMEOUT);
}

// A warp's tiles in order: the batch segments of the CTA's tile range and,
// inside each, the tiles seg0 + warp, seg0 + warp + nw, ...  (tile indices
// fit in 32 bits; the launcher checks.)
struct TileWalk {
    int t, seg1, t1, tpb, b, warp, nw;
    bool valid;
    __device__ __forceinline__ void start(int t0_, int t1_, int tpb_, int warp_, int nw_)
    {
        t1 = t1_;
        tpb = tpb_;
        warp = warp_;
        nw = nw_;
        b = t0_ / tpb;
        seg1 = (b + 1) * tpb < t1 ? (b + 1) * tpb : t1;
        t = t0_ + warp;
        settle();
    }
    __device__ __forceinline__ void settle()
    {
        while (t >= seg1 && seg1 < t1) {
            b++;                               // seg1 is a batch start from here on
            t = seg1 + warp;
            seg1 = seg1 + tpb < t1 ? seg1 + tpb : t1;
        }
        valid = t < seg1;
    }
    __device__ __forceinline__ void next()
    {
        t += nw;
        settle();
    }
};

// One streaming pass of the tile kernel over a CTA's row tiles [t0, t1) of a
// job's batches: the warp's ring (P slots with one mbarrier each), its
// producer (lane 0 issues, every lane keeps the same state) and its consumer.
// The job supplies the slot layout (layout()), the tensor maps (tmap()), the
// tensor rows of each piece (rmul(), radd()), its batches and where results
// go; a job with kSignals also hears when a warp has stored its results of a
// batch (warp_done(batch, tiles), every lane of the warp calling), and one
// with kWaits holds each batch back until its activations are complete
// (thread 0 waits in segment_poll(batch); every thread then reads
// segment_ready()).  A launch may run several passes one after another, each with its own
// ring barriers; a pass may prime its ring (issue its first P slices) long
// before it consumes.
template <int NM, int S, class Job>
struct TilePhase {
    static constexpr bool LOOP = Job::kLoopS;
    static constexpr int R = tile_rows_per<LOOP ? 1 : S, NM>();
    static constexpr int NR = NM * R;
    static constexpr int V = pow2_ceil(S * R * NM);
    static constexpr int KS = 32 * EPL;                     // inputs per slice
    static constexpr int CODE_ROW = 512;                    // code bytes per row per slice
    static constexpr int PLANE_B_ROW = 256;                 // int3 plane B bytes per row per slice
    static constexpr int B_OFF = NM * R * CODE_ROW;         // plane B pieces follow the code pieces
    static constexpr int NW = kTileWarps;

    const Job& job;
    // the layout, in registers
    int P, ns, xstride, sbox;
    uint32_t slot_bytes, tx_bytes, s_off0, s_step;
    int rm0, rm1, rm2, ra0, ra1, ra2;
    int warp, lane;
    bool leader;
    uint32_t sbase, full0, ctabar, ring0;
    int tpb, t0, t1;
    // producer
    TileWalk pw;
    int pk;                                  // slice of pw's tile to issue next
    int pb, pe;                              // batch of the last tile looked up, its expert
    int prow0, prow1, prow2;                 // tensor rows of pw's tile (codes, plane B, scales)
    int issued, consumed;
    // consumer
    int slot;
    uint32_t so, phase;

    // Lane 0 of each warp initializes the warp's slot barriers of layout L,
    // thread 0 the CTA barrier; the caller makes that visible to the CTA
    // (__syncthreads) before the pass's first call.
    static __device__ __forceinline__ void init_barriers(const TileLayout& L, uint32_t sbase_, int warp_)
    {
        const uint32_t f0 = sbase_ + (uint32_t)L.bar_off + 8u * (uint32_t)(warp_ * L.P);
        if ((threadIdx.x & 31) == 0)
            for (int p = 0; p < L.P; p++) mbar_init(f0 + 8u * p, 1);
        if (threadIdx.x == 0) mbar_init(sbase_ + (uint32_t)L.bar_off + 8u * (uint32_t)(NW * L.P), NW);
        mbar_init_fence();
    }

    // The pass over tiles [t0_, t1_) of tpb_ tiles per batch (its barriers
    // initialized).
    __device__ __forceinline__ TilePhase(const Job& j, uint32_t sbase_, int warp_, int t0_, int t1_, int tpb_)
        : job(j)
    {
        const TileLayout& L = job.layout();
        P = L.P;
        ns = L.nslices;
        xstride = L.xstride;
        slot_bytes = (uint32_t)L.slot_bytes;
        tx_bytes = (uint32_t)L.tx_bytes;
        sbox = L.sbox;
        s_off0 = (uint32_t)L.s_off[0];
        s_step = (uint32_t)(L.s_off[1] - L.s_off[0]);
        rm0 = (int)job.rmul(0);
        rm1 = (int)job.rmul(1);
        rm2 = (int)job.rmul(2);
        ra0 = (int)job.radd(0);
        ra1 = (int)job.radd(1);
        ra2 = (int)job.radd(2);
        warp = warp_;
        lane = threadIdx.x & 31;
        leader = lane == 0;
        sbase = sbase_;
        full0 = sbase + (uint32_t)L.bar_off + 8u * (uint32_t)(warp * P);
        ctabar = sbase + (uint32_t)L.bar_off + 8u * (uint32_t)(NW * P);
        ring0 = (uint32_t)L.ring_off + (uint32_t)warp * (uint32_t)L.warp_bytes;
        t0 = t0_;
        t1 = t1_;
        tpb = tpb_;
        pk = 0;
        pb = -1;
        pe = 0;
        prow0 = prow1 = prow2 = 0;
        issued = consumed = 0;
        slot = 0;
        so = ring0;
        phase = 0;
        pw.start(t0, t1 > t0 ? t1 : t0, tpb, warp, NW);
        if (t0 >= t1) pw.valid = false;
        if (pw.valid) tile_rows();
    }

    __device__ __forceinline__ void tile_rows()
    {
        if (pw.b != pb) {
            pb = pw.b;
            pe = (int)job.expert_of(pb);
        }
        const int r = (pw.t - pw.b * tpb) * R;
        prow0 = pe * rm0 + ra0 + r;
        prow1 = pe * rm1 + ra1 + r;
        prow2 = pe * rm2 + ra2 + r;
    }

    // Issues the next slice into the slot at shared offset `at` with barrier `bar`.
    __device__ __forceinline__ void issue(uint32_t at, uint32_t bar)
    {
        if (!pw.valid) return;
        if (leader) {
            mbar_expect_tx(bar, tx_bytes);
            const uint32_t dst = sbase + at;
#pragma unroll
            for (int m = 0; m < NM; m++) {
                tma_load_2d(dst + m * R * CODE_ROW, job.tmap(3 * m), pk * (CODE_ROW / 4), prow0, bar);
                if constexpr (FMT == FMT_INT3_G64)
                    tma_load_2d(dst + B_OFF + m * R * PLANE_B_ROW, job.tmap(3 * m + 1), pk * (PLANE_B_ROW / 4), prow1,
                                bar);
                if constexpr (SK != SK_ROW)
                    tma_load_2d(dst + s_off0 + m * s_step, job.tmap(3 * m + 2), pk * (sbox / 4), prow2, bar);
            }
        }
        __syncwarp();
        issued++;
        if (++pk == ns) {
            pk = 0;
            pw.next();
            if (pw.valid) tile_rows();
        }
    }

    // The first P slices into the ring.
    __device__ __forceinline__ void prime()
    {
        for (int p = 0; p < P; p++) issue(ring0 + (uint32_t)p * slot_bytes, full0 + 8u * p);
    }

    // Consumes every tile of the pass, batch segment by batch segment, all
    // warps in step (the batch's activation rows are staged at xs after every
    // warp is done with the last ones).  False when a wait ran out.
    __device__ __forceinline__ bool run(float* xs)
    {
        if (t0 >= t1) return true;
        const uint32_t xo[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // unused with the lane-interleaved x layout
        uint32_t cta_phase = 0;
        bool ok = true;
        int seg0 = t0;
        int b = t0 / tpb;
        while (ok && seg0 < t1) {
            const int seg1 = (b + 1) * tpb < t1 ? (b + 1) * tpb : t1;
            const int s_act = job.batch_S(b);
            // stage the batch's activation rows (after everyone is done with the last)
            if (seg0 != t0 && !cta_barrier(ctabar, cta_phase)) { ok = false; break; }
            if constexpr (Job::kWaits) {
                // one thread waits until the batch's activations are complete and
                // posts the outcome; the CTA barrier hands it to every warp
                job.segment_poll(b);
                if (!cta_barrier(ctabar, cta_phase) || !job.segment_ready()) { ok = false; break; }
            }
            if (!Job::kWaitFirst && seg0 == t0) pdl_wait_prev();   // before the first read of activations
            {
                const float* src[S];
#pragma unroll
                for (int s = 0; s < S; s++) src[s] = job.xrow(b, s < s_act ? s : 0);
                stage_rows_perm<EPL, Job::kFreshX>(xs, xstride, src, s_act, job.width(), threadIdx.x, NW * 32);
            }
            if (!cta_barrier(ctabar, cta_phase)) { ok = false; break; }

            Mat mt[NM];
            job.mats(b, mt);
            const long long rows = job.rows_per();
            // this lane's scale offsets inside a slot, per chunk row
            [[maybe_unused]] uint32_t sso[NR];
            if constexpr (SK != SK_ROW) {
                // f32: 4 bytes per group; ue8m0: one byte per group (one group per lane)
                const uint32_t ls = s_off0 + (((uint32_t)lane >> mt[0].gsh) << (SK == SK_E8M0 ? 0 : 2));
#pragma unroll
                for (int m = 0; m < NM; m++)
#pragma unroll
                    for (int r = 0; r < R; r++) sso[m * R + r] = ls + m * s_step + (uint32_t)(r * sbox);
            }
            Sink<Job, S, R, NM> sink{job, b, s_act};
            int mine = 0;                             // tiles of the segment this warp finished
            for (int t = seg0 + warp; ok && t < seg1; t += NW, mine++) {
                const long long row0 = (long long)(t - b * tpb) * R;
                float acc[S][NR];
#pragma unroll
                for (int s = 0; s < S; s++)
#pragma unroll
                    for (int rr = 0; rr < NR; rr++) acc[s][rr] = 0.f;
                [[maybe_unused]] float rsc[NR];
                if constexpr (SK == SK_ROW) {
#pragma unroll
                    for (int m = 0; m < NM; m++)
#pragma unroll
                        for (int r = 0; r < R; r++)
                            rsc[m * R + r] = ldg_f32(mt[m].sc + (row0 + r < rows ? row0 + r : rows - 1));
                }
                uint32_t xk = (uint32_t)lane * 16u;
                for (int k = 0; k < ns; k++) {
                    if (!mbar_wait(full0 + 8u * (uint32_t)slot, phase)) { ok = false; break; }
                    consumed++;
                    Chunk<FMT> ch[NR];
                    float sc[NR];
                    const uint32_t sl = so + (uint32_t)lane * 16u;
#pragma unroll
                    for (int m = 0; m < NM; m++)
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            const int rr = m * R + r;
                            if constexpr (FMT == FMT_INT3_G64) {
                                ch[rr].a = lds16(sl + (m * R + r) * CODE_ROW);
                                ch[rr].b = lds8(so + (uint32_t)lane * 8u + B_OFF + (m * R + r) * PLANE_B_ROW);
                            } else {
                                ch[rr].w = lds16(sl + (m * R + r) * CODE_ROW);
                            }
                            if constexpr (SK == SK_ROW) sc[rr] = rsc[rr];
                            else if constexpr (SK == SK_E8M0) sc[rr] = e8m0_to_f32(lds_u8(so + sso[rr]));
                            else sc[rr] = lds_f32(so + sso[rr]);
                        }
                    uint32_t xq[S];
#pragma unroll
                    for (int s = 0; s < S; s++) xq[s] = (uint32_t)(s * xstride) * 4u + xk;
                    if constexpr (LOOP) {
#pragma unroll
                        for (int s = 0; s < S; s++) {
                            if (s < s_act) {
                                const uint32_t x1[1] = {xq[s]};
                                consume<FMT, 1, NR, true>(ch, sc, x1, xo, reinterpret_cast<float(&)[1][NR]>(acc[s]),
                                                          1);
                            }
                        }
                    } else {
                        consume<FMT, S, NR, true>(ch, sc, xq, xo, acc, s_act);
                    }
                    __syncwarp();
                    issue(so, full0 + 8u * (uint32_t)slot);     // the slice P ahead goes into the slot just read
                    xk += KS * 4u;
                    so += slot_bytes;
                    if (++slot == P) {
                        slot = 0;
                        so = ring0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                constexpr int V1 = pow2_ceil(R * NM);        // one activation row in use (the common expert batch)
                if (LOOP && V1 < V && s_act == 1) {
                    float v[V1];
#pragma unroll
                    for (int i = 0; i < V1; i++) v[i] = 0.f;
#pragma unroll
                    for (int r = 0; r < R; r++)
#pragma unroll
                        for (int m = 0; m < NM; m++) v[r * NM + m] = acc[0][m * R + r];
                    const float red = warp_reduce_scatter<V1>(v, lane);
                    sink.template put<V1>(red, reduce_scatter_index<V1>(lane), lane < V1, row0, rows);
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
                    sink.template put<V>(red, reduce_scatter_index<V>(lane), lane < V, row0, rows);
                }
            }
            if constexpr (Job::kSignals) {
                if (ok && mine > 0) job.warp_done(b, mine);   // the warp's results of batch b are stored
            }
            seg0 = seg1;
            b++;
        }
        return ok;
    }

    // Waits for every slice issued and not yet consumed (each wait bounded,
    // without stopping at one that runs out): the CTA must not retire, or
    // reuse the ring, while copies into it are in flight.
    __device__ __forceinline__ void drain()
    {
        for (; consumed < issued; consumed++) {
            (void)mbar_wait(full0 + 8u * (uint32_t)slot, phase);
            if (++slot == P) {
                slot = 0;
                phase ^= 1u;
            }
        }
    }
};

template <int NM, int S, class Job>
__global__ void __launch_bounds__(kTileThreads, 1) k_tile(const __grid_constant__ Job job)
{
    // the warp index through a shuffle, so the compiler knows it is warp-uniform
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
    const uint32_t sbase = smem_base();
    int* status = job.status_word();

    if constexpr (Job::kWaitFirst) pdl_wait_prev();
    pdl_allow_next();
    if (job.bad()) return;
    if (sbase & 127u) {                           // tensor copies land on 128-byte boundaries
        if (threadIdx.x == 0) tile_fail(status);
        return;
    }
    constexpr int R = TilePhase<NM, S, Job>::R;
    const int tpb = (int)((job.rows_per() + R - 1) / R);    // tiles per batch
    const long long T = (long long)job.nbatch() * tpb;
    int t0, t1;
    job.cta_tiles(blockIdx.x, gridDim.x, T, t0, t1);
    TilePhase<NM, S, Job>::init_barriers(job.layout(), sbase, warp);
    __syncthreads();
    if (t0 >= t1) return;
    TilePhase<NM, S, Job> ph(job, sbase, warp, t0, t1, tpb);
    ph.prime();
    if (!ph.run(reinterpret_cast<float*>(qg_smem4))) {
        tile_fail(status);
        ph.drain();
    }
}
