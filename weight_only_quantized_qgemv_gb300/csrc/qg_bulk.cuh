// qg_bulk.cuh -- the warp-specialized streaming kernel (one format; included
// by qg_fmt_impl.cuh inside its format namespace).
//
// A CTA streams a contiguous range of weight rows (the job's batches laid end
// to end, split evenly over the CTAs).  Rows of one matrix are contiguous in
// memory, so one producer warp moves each stage -- rs consecutive rows of
// every matrix of the tile, their packed codes and their scales -- with a few
// large bulk copies (TMA engine) into a ring of nstage shared-memory stages,
// and nothing but decode-and-multiply is left to the consumer warps.
//
// Hand-off per stage slot: full[slot] (the producer's expect_tx plus the
// copies' byte count) and empty[slot] (one arrival per consumer warp once it
// is done with the stage).  Every consumer warp waits on and releases every
// stage in order, whether or not it has work in it, so no warp can fall a
// whole ring behind and mistake a later phase of a slot for the one it
// waits for.  A stage
// holds rs / R row tiles; a tile's warp steps are split into kp work units of
// kpw steps, dealt round-robin over the consumer warps across stages.  A unit
// reduces its partial sums across the warp and leaves them in shared memory;
// the last unit of a tile (counted with a shared-memory atomic) adds the kp
// partials in order, so results do not depend on timing, and hands the tile
// to the sink.  When the batch changes, the consumers restage the activation
// rows between two arrivals on xbar.  Every wait is bounded in time.
#pragma once

// Error word of this format's kernels: QSTATUS_DEVICE_TIMEOUT after a wait
// ran out (the launch's results are then undefined).
static __device__ int g_bulk_error;

__device__ __forceinline__ void bulk_fail(int* status_dev)
{
    atomicExch(&g_bulk_error, QSTATUS_DEVICE_TIMEOUT);
    if (status_dev) atomicExch(status_dev, QSTATUS_DEVICE_TIMEOUT);
}

// The CTA's sequence of stages: (batch b, batch-local first row, rows n),
// walked without divisions after the first.
struct StageIter {
    long long r, r_end, rows_per;
    long long nb, nrow;     // where the next stage starts
    int rs;
    int b;
    long long row0, n;
    __device__ __forceinline__ void start(long long r0, long long r1, long long rows, int rs_)
    {
        r = r0;
        r_end = r1;
        rows_per = rows;
        rs = rs_;
        nb = rows > 0 ? r0 / rows : 0;
        nrow = r0 - nb * rows;
    }
    __device__ __forceinline__ bool next()
    {
        if (r >= r_end) return false;
        b = (int)nb;
        row0 = nrow;
        n = rows_per - row0;
        if (r_end - r < n) n = r_end - r;
        if (rs < n) n = rs;
        r += n;
        nrow += n;
        if (nrow == rows_per) {
            nb++;
            nrow = 0;
        }
        return true;
    }
};

template <int NM, int S, class Job>
__global__ void __launch_bounds__((kBulkConsumers + 1) * 32, 1) k_bulk(const __grid_constant__ Job job)
{
    constexpr bool LOOP = Job::kLoopS;
    constexpr int R = rows_per_tile<LOOP ? 1 : S, NM>();
    constexpr int NR = NM * R;
    constexpr int V = pow2_ceil(S * R * NM);
    constexpr int NC = kBulkConsumers;
    const BulkLayout& L = job.bulk;

    float* xs = reinterpret_cast<float*>(qg_smem4);
    const uint32_t sbase = smem_base();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tps = L.rs / R;                   // row tiles per stage
    const int ups = tps * L.kp;                 // work units per stage
    const uint32_t full0 = sbase + L.bar_off;   // full[i] at full0 + 8 i, empty[i] after them, then xbar
    const uint32_t empty0 = full0 + 8u * L.nstage;
    const uint32_t xbar = empty0 + 8u * L.nstage;
    int* cnt = reinterpret_cast<int*>(reinterpret_cast<char*>(qg_smem4) + L.cnt_off);
    float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(qg_smem4) + L.part_off);

    if (job.bad()) return;
    if (threadIdx.x == 0) {
        for (int i = 0; i < L.nstage; i++) {
            mbar_init(full0 + 8u * i, 1);
            mbar_init(empty0 + 8u * i, (uint32_t)NC);
        }
        mbar_init(xbar, NC);
        mbar_init_fence();
    }
    for (int i = threadIdx.x; i < L.nstage * tps; i += blockDim.x) cnt[i] = 0;
    __syncthreads();

    const long long rows_per = job.rows_per();
    const long long N = (long long)job.nbatch() * rows_per;
    StageIter it;
    it.start(N * blockIdx.x / gridDim.x, N * (blockIdx.x + 1) / gridDim.x, rows_per, L.rs);

    if (warp == NC) {
        // ----------------------------- producer ------------------------------
        int k = 0;
        bool ok = true;
        while (ok && it.next()) {
            const int slot = k % L.nstage;
            const int use = k / L.nstage;
            if (use > 0 && !mbar_wait(empty0 + 8u * slot, (uint32_t)((use - 1) & 1))) {
                bulk_fail(job.status_word());
                ok = false;
                break;
            }
            if (lane == 0) {
                Mat m[NM];
                job.mats(it.b, m);
                const uint32_t n = (uint32_t)it.n;
                uint32_t bytes = 0;
#pragma unroll
                for (int j = 0; j < NM; j++) bytes += n * (uint32_t)(L.rb + L.rbB + L.sb);
                const uint32_t full = full0 + 8u * slot;
                mbar_expect_tx(full, bytes);
                const uint32_t stage = sbase + (uint32_t)(L.stage_off + slot * L.stage_bytes);
#pragma unroll
                for (int j = 0; j < NM; j++) {
                    const long long r0 = it.row0;
                    bulk_g2s(stage + L.w_off[j], m[j].w + r0 * L.rb, n * L.rb, full);
                    if (L.rbB) bulk_g2s(stage + L.b_off[j], m[j].w + m[j].O * L.rb + r0 * L.rbB, n * L.rbB, full);
                    if (L.sb) bulk_g2s(stage + L.s_off[j], reinterpret_cast<const char*>(m[j].sc) + r0 * L.sb,
                                       n * L.sb, full);
                }
            }
            __syncwarp();
            k++;
        }
        // the CTA must not retire while copies into its shared memory are in flight
        for (int j = (k > L.nstage ? k - L.nstage : 0); j < k; j++) {
            if (!mbar_wait(full0 + 8u * (j % L.nstage), (uint32_t)((j / L.nstage) & 1))) {
                bulk_fail(job.status_word());
                break;
            }
        }
        return;
    }

    // ------------------------------- consumers -------------------------------
    const uint32_t swz = (uint32_t)x_swz(EPL, lane);
    uint32_t xo[8];
#pragma unroll
    for (int j = 0; j < 8; j++) xo[j] = 16u * ((uint32_t)j ^ swz);
    const int nchunks = job.width() / EPL;
    const int nsteps = (nchunks + 31) / 32;
    const int I = job.width();
    int staged = -1, xuse = 0, k = 0;
    long long g = 0;                            // global unit index of the stage's first unit

    while (it.next()) {
        const int slot = k % L.nstage;
        const uint32_t full = full0 + 8u * slot;
        const uint32_t empty = empty0 + 8u * slot;
        const int s_act = job.batch_S(it.b);
        if (it.b != staged) {
            // restage the activation rows of batch it.b
            if (staged >= 0) {
                __syncwarp();
                if (lane == 0) mbar_arrive(xbar);
                if (!mbar_wait(xbar, (uint32_t)(xuse & 1))) { bulk_fail(job.status_word()); return; }
                xuse++;
            }
            const float* src[S];
#pragma unroll
            for (int s = 0; s < S; s++) src[s] = job.xrow(it.b, s < s_act ? s : 0);
            stage_rows_part<EPL>(xs, I, src, s_act, I, threadIdx.x, NC * 32);
            __syncwarp();
            if (lane == 0) mbar_arrive(xbar);
            if (!mbar_wait(xbar, (uint32_t)(xuse & 1))) { bulk_fail(job.status_word()); return; }
            xuse++;
            staged = it.b;
        }
        Mat mt[NM];
        job.mats(it.b, mt);
        const int gsh = mt[0].gsh;
        const uint32_t stage = (uint32_t)(L.stage_off + slot * L.stage_bytes);
        const int tiles = (int)((it.n + R - 1) / R);
        if (!mbar_wait(full, (uint32_t)((k / L.nstage) & 1))) { bulk_fail(job.status_word()); return; }
        // units u of this stage with (g + u) % NC == warp
        for (int u = (int)((warp - g % NC + NC) % NC); u < ups; u += NC) {
            const int t = u / L.kp, kp = u - t * L.kp;
            if (t < tiles) {
                float acc[S][NR];
#pragma unroll
                for (int s = 0; s < S; s++)
#pragma unroll
                    for (int rr = 0; rr < NR; rr++) acc[s][rr] = 0.f;
                const int c0 = kp * L.kpw;
                const int c1 = (c0 + L.kpw) < nsteps ? (c0 + L.kpw) : nsteps;
                for (int c = c0; c < c1; c++) {
                    const int q = c * 32 + lane;
                    if (q >= nchunks) continue;
                    Chunk<FMT> ch[NR];
                    float sc[NR];
#pragma unroll
                    for (int m = 0; m < NM; m++)
#pragma unroll
                        for (int r = 0; r < R; r++) {
                            const int rr = m * R + r, row = t * R + r;
                            if constexpr (FMT == FMT_INT3_G64) {
                                ch[rr].a = lds16(stage + L.w_off[m] + row * L.rb + q * 16);
                                ch[rr].b = lds8(stage + L.b_off[m] + row * L.rbB + q * 8);
                            } else {
                                ch[rr].w = lds16(stage + L.w_off[m] + row * L.rb + q * 16);
                            }
                            if constexpr (FMT == FMT_INT8_ROW) {
                                const long long grow = it.row0 + (row < it.n ? row : it.n - 1);
                                sc[rr] = ldg_f32(mt[m].sc + grow);
                            } else {
                                sc[rr] = lds_f32(stage + L.s_off[m] + row * L.sb + (q >> gsh) * 4);
                            }
                        }
                    uint32_t xq[S];
#pragma unroll
                    for (int s = 0; s < S; s++) xq[s] = (uint32_t)(s * I) * 4u + (uint32_t)q * (EPL * 4);
                    if constexpr (LOOP) {
#pragma unroll
                        for (int s = 0; s < S; s++) {
                            if (s < s_act) {
                                const uint32_t x1[1] = {xq[s]};
                                consume<FMT, 1, NR>(ch, sc, x1, xo, reinterpret_cast<float(&)[1][NR]>(acc[s]), 1);
                            }
                        }
                    } else {
                        consume<FMT, S, NR>(ch, sc, xq, xo, acc, s_act);
                    }
                }
                // reduce across the warp: lane l < V holds value reduce_scatter_index<V>(l)
                float v[V];
#pragma unroll
                for (int i = 0; i < V; i++) v[i] = 0.f;
#pragma unroll
                for (int s = 0; s < S; s++)
#pragma unroll
                    for (int r = 0; r < R; r++)
#pragma unroll
                        for (int m = 0; m < NM; m++) v[(s * R + r) * NM + m] = acc[s][m * R + r];
                float red = warp_reduce_scatter<V>(v, lane);
                const int idx = reduce_scatter_index<V>(lane);
                bool last = true;
                if (L.kp > 1) {
                    float* tp = part + ((size_t)(slot * tps + t) * L.kp) * 32;
                    tp[kp * 32 + lane] = red;
                    __threadfence_block();
                    __syncwarp();
                    int prev = 0;
                    if (lane == 0) prev = atomicAdd(&cnt[slot * tps + t], 1);
                    prev = __shfl_sync(0xffffffffu, prev, 0);
                    last = prev == L.kp - 1;
                    if (last) {
                        __threadfence_block();
                        red = 0.f;
                        for (int j = 0; j < L.kp; j++) red += tp[j * 32 + lane];
                        if (lane == 0) cnt[slot * tps + t] = 0;
                    }
                }
                if (last) {
                    Sink<Job, S, R, NM> sink{job, it.b, s_act};
                    sink.template put<V>(red, idx, lane < V, it.row0 + (long long)t * R, it.row0 + it.n);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty);
        g += ups;
        k++;
    }
}
