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

template <int NM, int S, class Job>
__global__ void __launch_bounds__(kTileThreads, 1) k_tile(const __grid_constant__ Job job)
{
    constexpr bool LOOP = Job::kLoopS;
    constexpr int R = tile_rows_per<LOOP ? 1 : S, NM>();
    constexpr int NR = NM * R;
    constexpr int V = pow2_ceil(S * R * NM);
    constexpr int KS = 32 * EPL;                     // inputs per slice
    constexpr int CODE_ROW = 512;                    // code bytes per row per slice
    constexpr int PLANE_B_ROW = 256;                 // int3 plane B bytes per row per slice
    constexpr int B_OFF = NM * R * CODE_ROW;         // plane B pieces follow the code pieces
    constexpr int NW = kTileWarps;

    // the launch's layout, once, in registers
    const int P = job.tile.P;
    const int ns = job.tile.nslices;
    const int xstride = job.tile.xstride;
    const uint32_t slot_bytes = (uint32_t)job.tile.slot_bytes;
    const uint32_t tx_bytes = (uint32_t)job.tile.tx_bytes;
    const int sbox = job.tile.sbox;
    const uint32_t s_off0 = (uint32_t)job.tile.s_off[0];
    const uint32_t s_step = (uint32_t)(job.tile.s_off[1] - job.tile.s_off[0]);
    const int rm0 = (int)job.row_mul[0], rm1 = (int)job.row_mul[1], rm2 = (int)job.row_mul[2];
    const int ra0 = (int)job.row_add[0], ra1 = (int)job.row_add[1], ra2 = (int)job.row_add[2];

    // the warp index through a shuffle, so the compiler knows it is warp-uniform
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0), lane = threadIdx.x & 31;
    const bool leader = lane == 0;
    const uint32_t sbase = smem_base();
    const uint32_t full0 = sbase + (uint32_t)job.tile.bar_off + 8u * (uint32_t)(warp * P);
    const uint32_t ctabar = sbase + (uint32_t)job.tile.bar_off + 8u * (uint32_t)(NW * P);
    const uint32_t ring0 = (uint32_t)job.tile.ring_off + (uint32_t)warp * (uint32_t)P * slot_bytes;
    float* xs = reinterpret_cast<float*>(qg_smem4);
    int* status = job.status_word();

    if constexpr (Job::kWaitFirst) pdl_wait_prev();
    pdl_allow_next();
    if (job.bad()) return;
    if (sbase & 127u) {                           // tensor copies land on 128-byte boundaries
        if (threadIdx.x == 0) tile_fail(status);
        return;
    }
    if (leader)
        for (int p = 0; p < P; p++) mbar_init(full0 + 8u * p, 1);
    if (threadIdx.x == 0) mbar_init(ctabar, NW * 32);
    mbar_init_fence();
    __syncthreads();

    const int tpb = (int)((job.rows_per() + R - 1) / R);    // tiles per batch
    const long long T = (long long)job.nbatch() * tpb;
    int t0, t1;
    job.cta_tiles(blockIdx.x, gridDim.x, T, t0, t1);
    if (t0 >= t1) return;

    // ---- producer: lane 0 issues, every lane keeps the same state ----
    TileWalk pw;
    pw.start(t0, t1, tpb, warp, NW);
    int pk = 0;                                   // slice of pw's tile to issue next
    int pb = -1, pe = 0;                          // batch of the last tile looked up, its expert
    int prow0 = 0, prow1 = 0, prow2 = 0;          // tensor rows of pw's tile (codes, plane B, scales)
    int issued = 0, consumed = 0;
    auto tile_rows = [&]() {
        if (pw.b != pb) {
            pb = pw.b;
            pe = (int)job.expert_of(pb);
        }
        const int r = (pw.t - pw.b * tpb) * R;
        prow0 = pe * rm0 + ra0 + r;
        prow1 = pe * rm1 + ra1 + r;
        prow2 = pe * rm2 + ra2 + r;
    };
    // issues the next slice into the slot at shared offset `so` with barrier `bar`
    auto issue = [&](uint32_t so, uint32_t bar) {
        if (!pw.valid) return;
        if (leader) {
            mbar_expect_tx(bar, tx_bytes);
            const uint32_t dst = sbase + so;
#pragma unroll
            for (int m = 0; m < NM; m++) {
                tma_load_2d(dst + m * R * CODE_ROW, &job.tm[3 * m], pk * (CODE_ROW / 4), prow0, bar);
                if constexpr (FMT == FMT_INT3_G64)
                    tma_load_2d(dst + B_OFF + m * R * PLANE_B_ROW, &job.tm[3 * m + 1], pk * (PLANE_B_ROW / 4), prow1,
                                bar);
                if constexpr (SK != SK_ROW)
                    tma_load_2d(dst + s_off0 + m * s_step, &job.tm[3 * m + 2], pk * (sbox / 4), prow2, bar);
            }
        }
        __syncwarp();
        issued++;
        if (++pk == ns) {
            pk = 0;
            pw.next();
            if (pw.valid) tile_rows();
        }
    };
    if (pw.valid) tile_rows();
    for (int p = 0; p < P; p++) issue(ring0 + (uint32_t)p * slot_bytes, full0 + 8u * p);

    // ---- consumer: batch segments of the CTA range, all warps in step ----
    const uint32_t xo[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // unused with the lane-interleaved x layout
    int slot = 0;
    uint32_t so = ring0;                          // shared offset of the current slot
    uint32_t phase = 0, cta_phase = 0;
    bool ok = true;
    int seg0 = t0;
    int b = t0 / tpb;
    while (ok && seg0 < t1) {
        const int seg1 = (b + 1) * tpb < t1 ? (b + 1) * tpb : t1;
        const int s_act = job.batch_S(b);
        // stage the batch's activation rows (after everyone is done with the last)
        if (seg0 != t0 && !cta_barrier(ctabar, cta_phase)) { ok = false; break; }
        if (!Job::kWaitFirst && seg0 == t0) pdl_wait_prev();   // before the first read of activations
        {
            const float* src[S];
#pragma unroll
            for (int s = 0; s < S; s++) src[s] = job.xrow(b, s < s_act ? s : 0);
            stage_rows_perm<EPL>(xs, xstride, src, s_act, job.width(), threadIdx.x, NW * 32);
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
        for (int t = seg0 + warp; ok && t < seg1; t += NW) {
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
                            consume<FMT, 1, NR, true>(ch, sc, x1, xo, reinterpret_cast<float(&)[1][NR]>(acc[s]), 1);
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
        seg0 = seg1;
        b++;
    }
    if (!ok) {
        tile_fail(status);
        // the CTA must not retire while copies into its shared memory are in
        // flight: wait for every slot issued and not yet consumed, each wait
        // bounded, without stopping at one that runs out
        for (; consumed < issued; consumed++) {
            (void)mbar_wait(full0 + 8u * (uint32_t)slot, phase);
            if (++slot == P) {
                slot = 0;
                phase ^= 1u;
            }
        }
    }
}
