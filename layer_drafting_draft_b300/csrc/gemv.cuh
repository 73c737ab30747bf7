// Weight-streaming GEMV for decode rows (M <= 8 activation rows), sm_103a.
//
// One launch runs a list of ops over the same M input rows; for op o and
// output feature n < N_o:
//   r_set[m][n] = sum over the op's segments s with set(s) = set:
//                 W_s[n, :] . x_{xs(s)}[m, :]
// with K-concatenated segments (several matrices and inputs summed into one
// output) and up to two accumulator sets (SwiGLU: gate and up).  Epilogues:
//   STORE    y[m][n]  = r0
//   ACC      y[m][n] += r0                      (residual add)
//   ACC_ADD  y[m][n] += r0 + add[m][n]          (residual add of two deltas)
//   SWIGLU   y[m][n]  = silu(r0) * r1
// Activation sources are plain rows, or normalised rows
//   x[m] = (h[m*stride + off] + add[...]) * rinv[m] * gain
// whose reciprocal rms `rinv` was computed by the launch before: after its
// ops, a launch may run a "post-norm" in which its last CTA to finish writes
// rinv[r] = 1 / rms(h[r*stride + off] + add[...]) for the next weight pass.
// So a consumer normalises while it stages its inputs, in the same single
// pass over memory.
//
// Data movement.  A stage is 32 consecutive rows x 512 bytes of one matrix.
// Each warp owns 4 rows of the 32-row tile and every lane one 16-byte column
// vector of each, read with 128-bit non-allocating loads into registers, the
// next chunk always requested before the current one is multiplied (two
// chunks in flight per thread, two CTAs per SM).  An activation vector read
// from shared memory serves 4 weight rows.  The launch descriptor is copied
// into shared memory and the first chunk requested before
// griddepcontrol.wait -- neither depends on the previous kernel -- so both
// arrive while that kernel drains.  Measured alternatives on B300 for this
// shape (all slower): TMA tensor tiles (capped near 4.6 TB/s per GPU by the
// per-SM TMA rate), one-dimensional bulk copies of 512-byte row pieces
// (under 2 TB/s), cp.async rings, L2 prefetch, and register-fed warp MMA
// (its 64-byte row pieces per load halve DRAM efficiency).
//
// Work split (stream-K).  The launch's stages -- ops, then 32-row tiles,
// then segments, then 512-byte column chunks -- form one sequence that is cut
// into equal contiguous ranges, one per CTA, so every SM streams the same
// number of bytes whatever the shapes.  A tile cut between CTAs is finished
// by the last CTA to arrive: each contributor stores its partial sums in
// `scratch`, bumps the tile's counter, and the last one adds the partials in
// CTA order (deterministic) and applies the epilogue, then clears the
// counter for the next launch.
#pragma once
#include "common.cuh"

namespace es {

constexpr int GV_WARPS = 8;
constexpr int GV_THREADS = GV_WARPS * 32;
constexpr int GV_R = 4;                        // rows per warp
constexpr int GV_RT = GV_WARPS * GV_R;         // rows per tile (32)
constexpr int GV_ROW_BYTES = 512;              // bytes of one row per stage
constexpr int GV_MAXM = 8;
constexpr int GV_MAX_XS = 16;
constexpr int GV_MAX_SEGS = 64;                // segments per launch
constexpr int GV_MAX_SEG = 16;                 // segments per op
constexpr int GV_MAX_OPS = 32;
constexpr int GV_XSMEM_MAX = 26 * 1024;        // floats of staged activations (104 KB)
constexpr int GV_CTAS_PER_SM = 2;
constexpr int GV_U = 1;                        // chunks per load batch (two batches in flight)
constexpr int GV_SCRATCH_CTAS = 1024;          // partial-sum slots
constexpr int GV_COUNTERS = 65536;             // arrival counters (tiles per launch)
constexpr int GV_SCRATCH_FLOATS = GV_SCRATCH_CTAS * 2 * 2 * GV_THREADS;

enum { GEPI_STORE = 0, GEPI_ACC = 1, GEPI_ACC_ADD = 2, GEPI_SWIGLU = 3 };

enum { XS_RAW = 0, XS_NORM = 1 };
// Input row r (< M) of x source i is row r*row_stride + row_off of `src`
// (leading dimension ld).  XS_NORM: x = (src + add) * rinv[r] * gain with the
// same row mapping for `add`.
struct GvXSrc {
    const float* src; const float* add; const void* gain; const float* rinv;
    int K, ld, row_stride, row_off, kind;
    int smem_off;  // float offset in the staged region, or -1: read from global
    int item0;     // first staging item (4 columns of one row) of this source
    int pad_;
    // XS_NORM with ss_tiles > 0 (tensor-core kernel): `rinv` holds the
    // producing launch's sums of squares instead, ss_tiles partials per row
    // at rinv[t * ss_ld + row]; the consumer adds them and takes 1/rms.
    int ss_tiles, ss_ld;
    float eps;
    int pad2_;
};
struct GvSeg { const void* W; int K, xs, set, nck; };
struct GvOp {
    float* y; const float* add;
    int seg0, nseg, epi, N, ldy;
    int ntiles, spt;       // 32-row tiles, stages per tile
    int tile0, stage0;     // launch-wide tile / stage index of the op's first
    int tile64_0;          // (SIMT GEMM) first 64-row tile of the op
};
// rinv[r] = 1 / sqrt(mean over k < K of (h + add)[r*row_stride + row_off][k]^2
//                     + eps), h and add with leading dimension K.
struct GvPost {
    const float* h; const float* add; float* rinv;
    int rows, row_stride, row_off, K;
    float eps; int pad_;
    // tensor-core kernel: instead of a last-CTA pass, the epilogue of op
    // `op` stores sums of squares of (h + add) over each of its 16-column
    // tiles: ssp[tile * M + row] (M = the launch's rows)
    float* ssp;
    int op, pad2_;
};
struct GvLaunch {
    int nops, nxs, M, ntiles, nstages, q, x_smem_floats, ntiles64, x_items, pad_;
    GvXSrc xs[GV_MAX_XS];
    GvOp ops[GV_MAX_OPS];
    GvSeg segs[GV_MAX_SEGS];
    GvPost post;
    int pad2_[2];
};
static_assert(sizeof(GvLaunch) % 16 == 0, "the descriptor is copied in 16-byte pieces");

ES_DEV float silu_f(float g) { return g / (1.0f + expf(-g)); }

// ------------------------------------------------------------ stage walker
// Position in the launch's stage sequence: op, tile, segment, column chunk.
struct GvWalk {
    const GvLaunch* L;
    int op, tile, seg, kc;
    __host__ __device__ void seek(const GvLaunch* L_, int s) {
        L = L_;
        op = 0;
        while (op + 1 < L->nops && L->ops[op + 1].stage0 <= s) ++op;
        const GvOp& o = L->ops[op];
        const int r = s - o.stage0;
        tile = r / o.spt;
        int c = r % o.spt;
        seg = 0;
        while (c >= L->segs[o.seg0 + seg].nck) { c -= L->segs[o.seg0 + seg].nck; ++seg; }
        kc = c;
    }
    // advance by n chunks within the current segment (n <= chunks left in
    // it); true when that finished the tile
    __host__ __device__ bool advance(int n) {
        const GvOp& o = L->ops[op];
        kc += n;
        if (kc < L->segs[o.seg0 + seg].nck) return false;
        kc = 0;
        if (++seg < o.nseg) return false;
        seg = 0;
        if (++tile >= o.ntiles) { tile = 0; ++op; }
        return true;
    }
};

// ------------------------------------------------------------ reductions
// Sum each of NV per-lane values over the warp; afterwards lane l holds the
// total of value (l mod P), P = NV rounded up to a power of two.
template <int NV>
ES_DEV float warp_reduce_scatter(const float (&v)[NV], int lane) {
    constexpr int P = NV <= 1 ? 1 : NV <= 2 ? 2 : NV <= 4 ? 4 : NV <= 8 ? 8 : NV <= 16 ? 16 : 32;
    float a[P];
#pragma unroll
    for (int i = 0; i < P; ++i) a[i] = i < NV ? v[i] : 0.f;
#pragma unroll
    for (int off = 16; off >= P; off >>= 1)
#pragma unroll
        for (int i = 0; i < P; ++i) a[i] += __shfl_xor_sync(0xffffffffu, a[i], off);
#pragma unroll
    for (int h = P / 2; h >= 1; h >>= 1) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? a[i] : a[i + h];
            const float keep = upper ? a[i + h] : a[i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, h);
        }
    }
    return a[0];
}


// ------------------------------------------------------------ post-norm
// Executed by one whole CTA (GV_THREADS threads) once the rows it reads are
// final.  The CTA's threads stride over all rows at once so that every load
// of every row is in flight together (one L2 round trip instead of one per
// few columns), then reduce per row through shared memory.
ES_DEV void post_rinv(const GvPost& p) {
    constexpr int ROWS = GV_MAXM, NW = GV_THREADS / 32;
    __shared__ float red[NW][ROWS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K4 = p.K >> 2;
    for (int r0 = 0; r0 < p.rows; r0 += ROWS) {
        const int nr = min(ROWS, p.rows - r0);
        float ss[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) ss[r] = 0.f;
        for (int k4 = tid; k4 < K4; k4 += GV_THREADS) {
            float4 v[ROWS];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < nr) {
                    const size_t base = (size_t)((r0 + r) * p.row_stride + p.row_off) * p.K + 4 * k4;
                    v[r] = __ldcg(reinterpret_cast<const float4*>(p.h + base));
                    if (p.add) {
                        const float4 a = __ldcg(reinterpret_cast<const float4*>(p.add + base));
                        v[r].x += a.x; v[r].y += a.y; v[r].z += a.z; v[r].w += a.w;
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
                ss[r] += v[r].x * v[r].x + v[r].y * v[r].y + v[r].z * v[r].z + v[r].w * v[r].w;
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const float t = warp_sum(ss[r]);
            if (lane == 0) red[warp][r] = t;
        }
        __syncthreads();
        if (tid < nr) {
            float t = 0.f;
            for (int w = 0; w < NW; ++w) t += red[w][tid];
            p.rinv[r0 + tid] = 1.0f / sqrtf(t / (float)p.K + p.eps);
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------ kernel
// acc[r][m] += W-vector(r) . x-vector(m) for one 16-byte column vector; x in
// shared memory or in global memory (through L1: all warps of the CTA read
// the same activation vectors).
template <typename T, int M>
ES_DEV void gv_fma(const uint4 (&w)[GV_R], const float* __restrict__ x, int xst, float (&acc)[GV_R][M]) {
    constexpr int EPV = 16 / sizeof(T);
    float wf[GV_R][EPV];
#pragma unroll
    for (int r = 0; r < GV_R; ++r) unpack16(w[r], wf[r], T());
#pragma unroll
    for (int m = 0; m < M; ++m) {
        float xv[EPV];
#pragma unroll
        for (int e = 0; e < EPV; e += 4) {
            const float4 t = *reinterpret_cast<const float4*>(x + (size_t)m * xst + e);
            xv[e] = t.x; xv[e + 1] = t.y; xv[e + 2] = t.z; xv[e + 3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < GV_R; ++r)
#pragma unroll
            for (int e = 0; e < EPV; ++e) acc[r][m] = fmaf(wf[r][e], xv[e], acc[r][m]);
    }
}

// The CTA's stage range, walked in batches of up to GV_U chunks of one
// segment.
struct GvBatch {
    int op, tile, seg, kc, n;
    bool tile_end;   // the batch completes its tile
    bool range_end;  // the batch is the last of this CTA's range
};

// Copy a launch descriptor into shared memory (whole CTA; synchronises).
ES_DEV void gv_load_desc(GvLaunch& L, const GvLaunch* __restrict__ Lg) {
    const int4* src = reinterpret_cast<const int4*>(Lg);
    int4* dst = reinterpret_cast<int4*>(&L);
    for (int i = threadIdx.x; i < (int)(sizeof(GvLaunch) / 16); i += blockDim.x) dst[i] = src[i];
    __syncthreads();
}

// The 16-byte weight vectors of batch b for this thread's 4 rows.
template <typename T>
ES_DEV void gv_load_batch(const GvLaunch& L, const GvBatch& b, uint4 (&wv)[GV_U][GV_R]) {
    constexpr int EPV = 16 / sizeof(T);
    constexpr int SC = GV_ROW_BYTES / sizeof(T);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const GvOp& o = L.ops[b.op];
    const GvSeg& sg = L.segs[o.seg0 + b.seg];
#pragma unroll
    for (int r = 0; r < GV_R; ++r) {
        // rows past N read the last row; their sums are dropped
        const T* wr = (const T*)sg.W + (size_t)min(b.tile * GV_RT + warp * GV_R + r, o.N - 1) * sg.K;
#pragma unroll
        for (int u = 0; u < GV_U; ++u) {
            const int k = (b.kc + u) * SC + lane * EPV;
            wv[u][r] = (u < b.n && k < sg.K) ? ld_stream16(wr + k) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// Step the walker over the next batch of CTA range [.., s_end).
ES_DEV bool gv_next_batch(GvWalk& w, int& s_next, int s_end, GvBatch& b) {
    if (s_next >= s_end) return false;
    const GvLaunch& L = *w.L;
    const int nck = L.segs[L.ops[w.op].seg0 + w.seg].nck;
    b.op = w.op; b.tile = w.tile; b.seg = w.seg; b.kc = w.kc;
    b.n = min(GV_U, min(nck - w.kc, s_end - s_next));
    b.tile_end = w.advance(b.n);
    s_next += b.n;
    b.range_end = s_next == s_end;
    return true;
}

// The first batch of CTA `cta`'s range (weights never depend on earlier
// work, so this may be issued before the inputs are ready).
template <typename T>
ES_DEV void gv_prefetch(const GvLaunch& L, int cta, uint4 (&wv)[GV_U][GV_R]) {
    const int s_begin = cta * L.q;
    if (s_begin >= L.nstages) return;
    GvWalk w;
    w.seek(&L, s_begin);
    int s_next = s_begin;
    GvBatch b;
    gv_next_batch(w, s_next, L.nstages < s_begin + L.q ? L.nstages : s_begin + L.q, b);
    gv_load_batch<T>(L, b, wv);
}

// The ops of descriptor L (in shared memory) over CTA `cta`'s stage range,
// whose first chunk is already in `wpre` (gv_prefetch).  Whole CTA; `xsm` is
// the dynamic shared memory for the staged activations.
template <typename T, int M>
ES_DEV void gv_run(const GvLaunch& L, float* xsm, float* __restrict__ scratch, int* __restrict__ counters,
                   int cta, const uint4 (&wpre)[GV_U][GV_R]) {
    constexpr int EPV = 16 / sizeof(T);            // weights per 16-byte vector
    constexpr int SC = GV_ROW_BYTES / sizeof(T);   // columns per stage: one vector per lane
    constexpr int NV = GV_R * M;
    __shared__ const float* xs_base[GV_MAX_XS];
    __shared__ int xs_stride[GV_MAX_XS];
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Q = L.q;
    const int s_begin = cta * Q;
    const int s_end = min(L.nstages, s_begin + Q);
    if (s_begin >= s_end) return;  // (uniform per CTA)

    GvWalk w;
    w.seek(&L, s_begin);
    int s_next = s_begin;
    GvBatch cur, nxt;
    uint4 wc[GV_U][GV_R], wn[GV_U][GV_R];
    bool have = gv_next_batch(w, s_next, s_end, cur);
#pragma unroll
    for (int u = 0; u < GV_U; ++u)
#pragma unroll
        for (int r = 0; r < GV_R; ++r) wc[u][r] = wpre[u][r];

    const int nxs = L.nxs;
    if (tid < nxs) {
        const GvXSrc& x = L.xs[tid];
        if (x.smem_off >= 0) {
            xs_base[tid] = xsm + x.smem_off;
            xs_stride[tid] = x.K;
        } else {
            xs_base[tid] = x.src + (size_t)x.row_off * x.ld;
            xs_stride[tid] = x.row_stride * x.ld;
        }
    }
    // Stage the shared-memory sources: all (source, row, 4-column) items form
    // one list; every thread issues the loads of 8 items (activation, added
    // delta, gain, 1/rms) before using any.
    const int nitems = L.x_items;
    constexpr int SB = 8;
    for (int t0 = tid; t0 < nitems; t0 += SB * GV_THREADS) {
        float4 v[SB], gn[SB];
        float ri[SB];
        float* dst[SB];
#pragma unroll
        for (int u = 0; u < SB; ++u) {
            const int t = t0 + u * GV_THREADS;
            dst[u] = nullptr;
            ri[u] = 0.f;
            if (t < nitems) {
                int i = 0;
                while (i + 1 < nxs && L.xs[i + 1].item0 <= t) ++i;
                const GvXSrc& x = L.xs[i];
                const int K4 = x.K >> 2, r = t - x.item0, m = r / K4, k = (r - m * K4) * 4;
                const size_t g = (size_t)(m * x.row_stride + x.row_off) * x.ld + k;
                v[u] = __ldcg(reinterpret_cast<const float4*>(x.src + g));
                if (x.add) {
                    const float4 a = __ldcg(reinterpret_cast<const float4*>(x.add + g));
                    v[u].x += a.x; v[u].y += a.y; v[u].z += a.z; v[u].w += a.w;
                }
                if (x.kind == XS_NORM) {
                    const T* gp = (const T*)x.gain + k;
                    gn[u] = make_float4(to_f32(gp[0]), to_f32(gp[1]), to_f32(gp[2]), to_f32(gp[3]));
                    ri[u] = __ldcg(x.rinv + m);
                }
                dst[u] = xsm + x.smem_off + (size_t)m * x.K + k;
            }
        }
#pragma unroll
        for (int u = 0; u < SB; ++u) {
            if (!dst[u]) continue;
            float4 y = v[u];
            if (ri[u] != 0.f) {
                y.x = y.x * ri[u] * gn[u].x;
                y.y = y.y * ri[u] * gn[u].y;
                y.z = y.z * ri[u] * gn[u].z;
                y.w = y.w * ri[u] * gn[u].w;
            }
            *reinterpret_cast<float4*>(dst[u]) = y;
        }
    }
    __syncthreads();

    float acc[GV_R][M];
#pragma unroll
    for (int r = 0; r < GV_R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;
    float vset[2] = {0.f, 0.f};  // reduced sums of finished accumulator sets (lane-distributed)
    int cur_set = -1;
    int tile_first = s_begin - ((s_begin - L.ops[cur.op].stage0) % L.ops[cur.op].spt);

    while (have) {
        const bool have_n = gv_next_batch(w, s_next, s_end, nxt);
        if (have_n) gv_load_batch<T>(L, nxt, wn);  // in flight while this batch is multiplied

        const GvOp& o = L.ops[cur.op];
        const GvSeg& sg = L.segs[o.seg0 + cur.seg];
        if (sg.set != cur_set) {
            if (cur_set >= 0) {
                float t[NV];
#pragma unroll
                for (int r = 0; r < GV_R; ++r)
#pragma unroll
                    for (int m = 0; m < M; ++m) { t[r * M + m] = acc[r][m]; acc[r][m] = 0.f; }
                vset[cur_set] += warp_reduce_scatter<NV>(t, lane);
            }
            cur_set = sg.set;
        }
#pragma unroll
        for (int u = 0; u < GV_U; ++u) {
            const int k = (cur.kc + u) * SC + lane * EPV;
            if (u < cur.n && k < sg.K) gv_fma<T, M>(wc[u], xs_base[sg.xs] + k, xs_stride[sg.xs], acc);
        }
        if (cur.tile_end || cur.range_end) {
            // ------------ finish the tile (or this CTA's part of it)
            {
                float t[NV];
#pragma unroll
                for (int r = 0; r < GV_R; ++r)
#pragma unroll
                    for (int m = 0; m < M; ++m) { t[r * M + m] = acc[r][m]; acc[r][m] = 0.f; }
                vset[cur_set] += warp_reduce_scatter<NV>(t, lane);
            }
            float v0 = vset[0], v1 = vset[1];
            vset[0] = vset[1] = 0.f;
            cur_set = -1;
            const bool two = o.epi == GEPI_SWIGLU;
            const int tile_last = tile_first + o.spt - 1;
            const bool complete = tile_first >= s_begin && tile_last < s_end;
            const int gtile = o.tile0 + cur.tile;
            bool do_epi = complete;
            if (!complete) {
                const int sid = s_begin >= tile_first ? 0 : 1;
                float* part = scratch + ((size_t)(cta * 2 + sid) * 2) * GV_THREADS + tid;
                part[0] = v0;
                if (two) part[GV_THREADS] = v1;
                __threadfence();
                __syncthreads();
                const int c_first = tile_first / Q, c_last = tile_last / Q;
                if (tid == 0) s_last = atomicAdd(counters + gtile, 1) == c_last - c_first;
                __syncthreads();
                if (s_last) {
                    __threadfence();
                    v0 = 0.f; v1 = 0.f;
                    for (int cc = c_first; cc <= c_last; ++cc) {
                        const int sd = cc * Q >= tile_first ? 0 : 1;
                        const float* pp = scratch + ((size_t)(cc * 2 + sd) * 2) * GV_THREADS + tid;
                        v0 += __ldcg(pp);
                        if (two) v1 += __ldcg(pp + GV_THREADS);
                    }
                    if (tid == 0) counters[gtile] = 0;
                    do_epi = true;
                }
                // every thread has read s_last before a later tile changes it
                __syncthreads();
            }
            if (do_epi && lane < NV) {
                const int r = lane / M, m = lane % M;
                const int n = cur.tile * GV_RT + warp * GV_R + r;
                if (n < o.N) {
                    float* y = o.y + (size_t)m * o.ldy + n;
                    switch (o.epi) {
                        case GEPI_STORE: *y = v0; break;
                        case GEPI_ACC: *y = __ldcg(y) + v0; break;
                        case GEPI_ACC_ADD: *y = __ldcg(y) + v0 + __ldcg(o.add + (size_t)m * o.ldy + n); break;
                        default: *y = silu_f(v0) * v1; break;
                    }
                }
            }
            tile_first = tile_last + 1;
        }
        cur = nxt;
#pragma unroll
        for (int u = 0; u < GV_U; ++u)
#pragma unroll
            for (int r = 0; r < GV_R; ++r) wc[u][r] = wn[u][r];
        have = have_n;
    }
}

// One weight-streaming launch as its own kernel.  With programmatic
// dependent launch the descriptor copy and the first weight chunk overlap
// the previous kernel's drain.  `done` counts finished CTAs: the last runs
// the post-norm.
template <typename T, int M>
__global__ void __launch_bounds__(GV_THREADS, GV_CTAS_PER_SM)
gv_kernel(const GvLaunch* __restrict__ Lg, float* __restrict__ scratch, int* __restrict__ counters,
          int* __restrict__ done) {
    extern __shared__ __align__(16) float xsm[];
    __shared__ __align__(16) GvLaunch L;
    __shared__ int s_done;
    gv_load_desc(L, Lg);
    uint4 wpre[GV_U][GV_R];
    gv_prefetch<T>(L, blockIdx.x, wpre);
    grid_dep_wait();
    grid_dep_launch();
    gv_run<T, M>(L, xsm, scratch, counters, blockIdx.x, wpre);
    if (L.post.rows > 0) {
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_done = atomicAdd(done, 1) == (int)gridDim.x - 1;
        __syncthreads();
        if (s_done) {
            __threadfence();
            post_rinv(L.post);
            if (threadIdx.x == 0) *done = 0;
        }
    }
}

// ------------------------------------------------------------ bf16: warp MMA
// Tensor-core variant for bf16 weights (same descriptor; planned with
// 128-row blocks and 128-column chunks).  Each warp of a CTA owns 16 rows of
// the block -- the M side of mma.sync m16n8k16 -- and the (up to 8)
// activation rows are its N side, so one MMA does the work of 256 fused
// multiply-adds per activation row.
//
// Register-fed A operand.  In one k32 group lane (g = lane/4, c = lane%4)
// loads 16 bytes of weight rows g and g+8 at columns 8c..8c+7: the fragments
// of two k16 MMAs under a fixed permutation of k inside the group (a dot
// product does not depend on the order of its terms).  MMA 0 takes columns
// 8c+0..3 as its k = (2c, 2c+1, 2c+8, 2c+9), MMA 1 columns 8c+4..7.  The B
// operand -- activation row g at the same eight columns -- is then one
// 16-byte load as well.  Activations enter as two bf16 planes, hi = bf16(x)
// and lo = bf16(x - hi), both multiplied into the same float32 accumulator,
// so the products keep about 16 significant bits of x (float32-level
// accuracy) at bf16 tensor-core cost.
//
// Work split: stream-K over CTA stages (op, 128-row block, segment,
// 128-column chunk); all warps of a CTA walk the same stages, each over its
// own 16 rows of the block, keeping GVM_D stages of weight loads in flight.
// Blocks cut between CTAs are summed by the last CTA to arrive (partials in
// CTA order: deterministic).
// Activation windows: a CTA stages, as hi/lo planes in shared memory, only
// the chunks of each source that its stage range multiplies (up to
// GVM_NWIN windows while the budget lasts); anything else is read as
// float32 through L2 and split in registers.  The planner sizes each
// launch's shared memory to its largest window set: a larger request would
// shrink the L1 that the streaming loads pass through.
constexpr int GVM_ROWS = 16;                     // rows per warp
constexpr int GVM_BLOCK = GVM_ROWS * GV_WARPS;   // rows per stage (128) of the 8-warp variant
// The 16-warp variant (one 512-thread CTA per SM, 256-row stages) shares one
// activation window between twice the warps: for widths whose windows do
// not fit the 8-warp budget.
constexpr int GVM_WIDE_WARPS = 16;
constexpr int GVM_WIDE_XSMEM = 48 * 1024;        // 4-byte words (192 KB)
constexpr int GVM_COLS = 128;                    // columns per stage
constexpr int GVM_D = 2;                         // stages in flight per warp
constexpr int GVM_NWIN = 16;                     // activation windows per CTA
constexpr int GVM_PAD = 32;                      // plane padding (columns)
constexpr int GVM_SCRATCH_CTAS = 1024;
// partial sums [cta][cut][warp][set][lane x 4]
constexpr int GVM_SCRATCH_FLOATS = GVM_SCRATCH_CTAS * 2 * GV_WARPS * 2 * 128;

// chunks [klo, khi) of source src, hi/lo planes at word offset off of the
// staged region (-1: read from global memory); plane width pw columns
struct GvmWin { int src, klo, khi, off, pw, item0; };

ES_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                           uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

ES_DEV uint32_t bf2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }

// hi/lo bf16 pairs of two floats (element 0 in the low half)
ES_DEV void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = bf2_bits(h);
    lo = bf2_bits(__floats2bfloat162_rn(a - hf.x, b - hf.y));
}

// Four activations of source x, row m, columns k..k+3 (k + 3 < K): the raw
// row plus `add`, normalised for XS_NORM.
ES_DEV float4 gvm_x4(const GvXSrc& x, int m, int k, const float* srinv) {
    const size_t gi = (size_t)(m * x.row_stride + x.row_off) * x.ld + k;
    float4 v = __ldcg(reinterpret_cast<const float4*>(x.src + gi));
    if (x.add) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(x.add + gi));
        v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
    }
    if (x.kind == XS_NORM) {
        // four bf16 gains in one 8-byte load (k is a multiple of 4)
        const uint2 gb = *reinterpret_cast<const uint2*>((const bf16*)x.gain + k);
        // with partial sums, 1/rms is a per-row factor applied in the epilogue
        const float ri = x.ss_tiles > 0 ? 1.0f : __ldcg(x.rinv + m);
        v.x *= ri * __uint_as_float(gb.x << 16);
        v.y *= ri * __uint_as_float(gb.x & 0xffff0000u);
        v.z *= ri * __uint_as_float(gb.y << 16);
        v.w *= ri * __uint_as_float(gb.y & 0xffff0000u);
    }
    return v;
}

// The activation windows of CTA stage range [S0, S1) (one thread), staged
// greedily in order while `budget` words of shared memory last.  Returns the
// number of windows; *nitems = staging items (4 columns of one row) and
// *used = words of the staged ones.  The planner runs the same function on
// the host to size each launch's shared memory.
__host__ __device__ inline int gvm_windows(const GvLaunch& L, int S0, int S1, GvmWin* win, int budget, int* nitems,
                                           int* used_words) {
    int n = 0;
    GvWalk w;
    w.seek(&L, S0);
    for (int s = S0; s < S1;) {
        const GvSeg& sg = L.segs[L.ops[w.op].seg0 + w.seg];
        const int run = sg.nck - w.kc < S1 - s ? sg.nck - w.kc : S1 - s;
        const int a = w.kc, b = w.kc + run;
        int i = 0;
        for (; i < n; ++i)
            if (win[i].src == sg.xs && a <= win[i].khi && b >= win[i].klo) break;
        if (i < n) {
            if (a < win[i].klo) win[i].klo = a;
            if (b > win[i].khi) win[i].khi = b;
        } else if (n < GVM_NWIN) {
            win[n].src = sg.xs; win[n].klo = a; win[n].khi = b;
            ++n;
        }
        w.advance(run);
        s += run;
    }
    // a widened window may now touch another of its source: merge those
    for (bool again = true; again;) {
        again = false;
        for (int i = 0; i < n && !again; ++i)
            for (int j = i + 1; j < n && !again; ++j)
                if (win[i].src == win[j].src && win[j].klo <= win[i].khi && win[j].khi >= win[i].klo) {
                    if (win[j].klo < win[i].klo) win[i].klo = win[j].klo;
                    if (win[j].khi > win[i].khi) win[i].khi = win[j].khi;
                    win[j] = win[--n];
                    again = true;
                }
    }
    int used = 0, items = 0;
    for (int i = 0; i < n; ++i) {
        const int cols = (win[i].khi - win[i].klo) * GVM_COLS;
        win[i].pw = cols + GVM_PAD;
        const int words = L.M * win[i].pw;
        win[i].off = -1;
        win[i].item0 = items;
        if (used + words <= budget) {
            win[i].off = used;
            used += words;
            items += L.M * (cols / 4);
        }
    }
    *nitems = items;
    *used_words = used;
    return n;
}

// Float4 columns of the staged windows (off >= 0), numbered window by window.
__host__ __device__ inline int gvm_stage_columns(const GvmWin* win, int nwin) {
    int total = 0;
    for (int w = 0; w < nwin; ++w)
        if (win[w].off >= 0) total += (win[w].khi - win[w].klo) * (GVM_COLS / 4);
    return total;
}
// Moves the cursor (window w, whose first column is wbase) to the staged
// window holding column c < the total; c must not decrease between calls.
__host__ __device__ inline void gvm_stage_cursor(const GvmWin* win, int c, int& w, int& wbase) {
    while (win[w].off < 0 || c >= wbase + (win[w].khi - win[w].klo) * (GVM_COLS / 4)) {
        if (win[w].off >= 0) wbase += (win[w].khi - win[w].klo) * (GVM_COLS / 4);
        ++w;
    }
}
// Item t < M * total of the small-window staging: activation row m =
// t / total, and the window w and first element kr of flat column t % total.
__host__ __device__ inline void gvm_stage_item(const GvmWin* win, int total, int t, int& w, int& m, int& kr) {
    m = t / total;
    int c = t - m * total;
    w = 0;
    for (;; ++w) {
        if (win[w].off < 0) continue;
        const int C4 = (win[w].khi - win[w].klo) * (GVM_COLS / 4);
        if (c < C4) break;
        c -= C4;
    }
    kr = 4 * c;
}

// Stage the windows with off >= 0 as hi/lo planes (whole CTA; synchronises):
// float32 (normalised) activations split into hi/lo bf16.  A thread takes
// float4 columns c, c + NT, ... numbered across the staged windows and loads
// that column of every activation row at once; the window of a column is
// found by a cursor that only moves forward, so a column costs its loads,
// the splits and the stores.
template <int NT>
ES_DEV void gvm_stage(const GvLaunch& L, const GvmWin* win, int nwin, unsigned char* xsm, const float* srinv) {
    constexpr int RB = GV_MAXM;
    const int M = L.M;
    const int total = gvm_stage_columns(win, nwin);
    int w = 0, wbase = 0;  // window of the current column, flat index of its first column
    for (int c = threadIdx.x; c < total; c += NT) {
        gvm_stage_cursor(win, c, w, wbase);
        const GvmWin& wn = win[w];
        const GvXSrc& x = L.xs[wn.src];
        const int kr = (c - wbase) * 4, k = wn.klo * GVM_COLS + kr;
        bf16* hi = reinterpret_cast<bf16*>(xsm + (size_t)wn.off * 4) + kr;
        for (int m0 = 0; m0 < M; m0 += RB) {
            float4 v[RB];
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (m0 + u < M && k < x.K) v[u] = gvm_x4(x, m0 + u, k, srinv);
            }
#pragma unroll
            for (int u = 0; u < RB; ++u) {
                const int m = m0 + u;
                if (m >= M) break;
                uint2 h, l;
                split2(v[u].x, v[u].y, h.x, l.x);
                split2(v[u].z, v[u].w, h.y, l.y);
                *reinterpret_cast<uint2*>(hi + (size_t)m * wn.pw) = h;
                *reinterpret_cast<uint2*>(hi + (size_t)(M + m) * wn.pw) = l;
            }
        }
    }
    __syncthreads();
}

// The same for a CTA with few stages (small windows) that holds both ring
// stages while staging: (row, column) items spread over all threads, two
// per thread with their loads in flight together.
template <int NT>
ES_DEV void gvm_stage_small(const GvLaunch& L, const GvmWin* win, int nwin, unsigned char* xsm,
                            const float* srinv) {
    const int M = L.M;
    const int total = gvm_stage_columns(win, nwin);
    for (int t0 = threadIdx.x; t0 < M * total; t0 += 2 * NT) {
        float4 v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = t0 + u * NT;
            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < M * total) {
                int w, m, kr;
                gvm_stage_item(win, total, t, w, m, kr);
                const GvXSrc& x = L.xs[win[w].src];
                const int k = win[w].klo * GVM_COLS + kr;
                if (k < x.K) v[u] = gvm_x4(x, m, k, srinv);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = t0 + u * NT;
            if (t >= M * total) break;
            int w, m, kr;
            gvm_stage_item(win, total, t, w, m, kr);
            bf16* hi = reinterpret_cast<bf16*>(xsm + (size_t)win[w].off * 4) + (size_t)m * win[w].pw + kr;
            uint2 h, l;
            split2(v[u].x, v[u].y, h.x, l.x);
            split2(v[u].z, v[u].w, h.y, l.y);
            *reinterpret_cast<uint2*>(hi) = h;
            *reinterpret_cast<uint2*>(hi + (size_t)M * win[w].pw) = l;
        }
    }
    __syncthreads();
}

// weight fragments of one stage for this warp: rows g and g+8, four k32 groups
struct GvmStage { uint4 a[4], b[4]; };

// A run: chunks [kc, kc_end) of one segment of one tile.  The loops below
// read the descriptor once per run, so a stage costs only its loads and MMAs.
struct GvmRun { int op, tile, seg, kc, kc_end; };

// Position (op, tile, segment, chunk) in the stage sequence of L.
struct GvmPos { int op, tile, seg, kc; };

ES_DEV GvmPos gvm_seek(const GvLaunch& L, int s) {
    GvWalk w;
    w.seek(&L, s);
    return GvmPos{w.op, w.tile, w.seg, w.kc};
}

// The run starting at p, within stage range [.., s_end) (s: p's index);
// p and s move past it.
ES_DEV GvmRun gvm_next_run(const GvLaunch& L, GvmPos& p, int& s, int s_end) {
    GvmRun r;
    r.op = p.op; r.tile = p.tile; r.seg = p.seg; r.kc = p.kc;
    const GvOp& o = L.ops[p.op];
    const int nck = L.segs[o.seg0 + p.seg].nck;
    const int n = min(nck - p.kc, s_end - s);
    r.kc_end = p.kc + n;
    s += n;
    p.kc += n;
    if (p.kc == nck) {
        p.kc = 0;
        if (++p.seg == o.nseg) {
            p.seg = 0;
            if (++p.tile == o.ntiles) { p.tile = 0; ++p.op; }
        }
    }
    return r;
}

// Per-warp cursor state that only run boundaries touch (kept in shared
// memory to leave the registers to the weight ring).  Every lane of the warp
// writes the same values.
struct GvmWarp {
    GvmPos ip, cp;  // issue / consume positions after their current runs
    int is, cs;     // their stage indices
    int op, tile, src;  // the consume run's op, tile and activation source
};

// Issue side: this lane's weight row pointers in the current run.
struct GvmIssue {
    const bf16* ra;  // row g, from column 8c
    const bf16* rb;  // row g + 8, from column 8c
    int K;           // segment width (0 for a warp wholly past N)
    int kc, kc_end;
};

template <int NW>
ES_DEV void gvm_issue_begin(const GvLaunch& L, GvmWarp& ws, GvmIssue& I, int s_end) {
    const GvmRun r = gvm_next_run(L, ws.ip, ws.is, s_end);
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const GvOp& o = L.ops[r.op];
    const GvSeg& sg = L.segs[o.seg0 + r.seg];
    const int w0 = r.tile * (NW * GVM_ROWS) + (threadIdx.x >> 5) * GVM_ROWS;
    // rows past N read the last row (their sums are dropped); warps wholly
    // past N load nothing
    I.ra = (const bf16*)sg.W + (size_t)min(w0 + g, o.N - 1) * sg.K + 8 * c;
    I.rb = (const bf16*)sg.W + (size_t)min(w0 + g + 8, o.N - 1) * sg.K + 8 * c;
    I.K = w0 < o.N ? sg.K : 0;
    I.kc = r.kc;
    I.kc_end = r.kc_end;
}

// Request chunk I.kc into st and step (a stage must remain in the range).
// Whole chunks take unpredicated loads; only a segment's ragged last chunk
// (or a warp past N) checks columns.  (A bulk L2 prefetch of the chunk 4 or
// 8 stages ahead measured slower: 223 and 219 against 236 tok/s.)
template <int NW>
ES_DEV void gvm_issue_step(const GvLaunch& L, GvmWarp& ws, GvmIssue& I, GvmStage& st, int s_end) {
    const int kb = I.kc * GVM_COLS;
    const bf16* pa = I.ra + kb;
    const bf16* pb = I.rb + kb;
    if (kb + GVM_COLS <= I.K) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            st.a[j] = ld_stream16(pa + 32 * j);
            st.b[j] = ld_stream16(pb + 32 * j);
        }
    } else {
        const int kl = I.K - 8 * (threadIdx.x & 3) - kb;  // this lane's columns left in the segment
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool in = 32 * j < kl;
            st.a[j] = in ? ld_stream16(pa + 32 * j) : make_uint4(0u, 0u, 0u, 0u);
            st.b[j] = in ? ld_stream16(pb + 32 * j) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (++I.kc == I.kc_end && ws.is < s_end) gvm_issue_begin<NW>(L, ws, I, s_end);
}

// Consume side: the activation operand of the current run.
struct GvmCons {
    int kc, kc_end, set;
    bool tile_end;  // the run completes its tile
    bool glob;      // no staged window: read float32 through L2
    uint32_t sa;    // shared address of this lane's hi-plane fragment at column 0 of the window
    uint32_t lo;    // hi -> lo plane distance (bytes)
    int kbase;      // first column of the window
};

ES_DEV void gvm_cons_begin(const GvLaunch& L, GvmWarp& ws, GvmCons& C, const GvmWin* win, int nwin,
                           const unsigned char* xsm, int s_end) {
    const GvmRun r = gvm_next_run(L, ws.cp, ws.cs, s_end);
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const GvOp& o = L.ops[r.op];
    const GvSeg& sg = L.segs[o.seg0 + r.seg];
    ws.op = r.op; ws.tile = r.tile; ws.src = sg.xs;
    C.kc = r.kc; C.kc_end = r.kc_end;
    C.set = sg.set;
    C.tile_end = r.kc_end == sg.nck && r.seg == o.nseg - 1;
    C.glob = true;
    C.sa = 0; C.lo = 0; C.kbase = 0;
    for (int i = 0; i < nwin; ++i)
        if (win[i].src == sg.xs && r.kc >= win[i].klo && r.kc < win[i].khi) {
            if (win[i].off >= 0) {
                // lanes of activation rows >= M read row M-1: the MMA columns
                // they feed are never stored
                const int row = min(g, L.M - 1);
                C.glob = false;
                C.sa = (uint32_t)__cvta_generic_to_shared(xsm) + (uint32_t)win[i].off * 4u +
                       (uint32_t)(row * win[i].pw + 8 * c) * 2u;
                C.lo = (uint32_t)(L.M * win[i].pw) * 2u;
                C.kbase = win[i].klo * GVM_COLS;
            }
            break;
        }
}

ES_DEV uint4 lds16(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// B fragments (hi, lo) of group j of chunk C.kc read as float32 from
// global memory: the fallback for sources without a staged window.
ES_DEV void gvm_x_global(const GvLaunch& L, const GvmWarp& ws, const GvmCons& C, int j, uint4& bh, uint4& bl,
                         const float* srinv) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const GvXSrc& x = L.xs[ws.src];
    const int k = C.kc * GVM_COLS + 32 * j + 8 * c;
    bh = bl = make_uint4(0u, 0u, 0u, 0u);
    if (g < L.M && k < x.K) {
        const float4 f0 = gvm_x4(x, g, k, srinv), f1 = gvm_x4(x, g, k + 4, srinv);
        split2(f0.x, f0.y, bh.x, bl.x);
        split2(f0.z, f0.w, bh.y, bl.y);
        split2(f1.x, f1.y, bh.z, bl.z);
        split2(f1.z, f1.w, bh.w, bl.w);
    }
}

ES_DEV void gvm_mma_group(float (&acc)[4], const uint4& a, const uint4& b, const uint4& bh, const uint4& bl) {
    mma_bf16_16816(acc, a.x, b.x, a.y, b.y, bh.x, bh.y);
    mma_bf16_16816(acc, a.z, b.z, a.w, b.w, bh.z, bh.w);
    mma_bf16_16816(acc, a.x, b.x, a.y, b.y, bl.x, bl.y);
    mma_bf16_16816(acc, a.z, b.z, a.w, b.w, bl.z, bl.w);
}

// acc += W(chunk C.kc of this warp's rows) . x, and step.
ES_DEV void gvm_cons_step(const GvLaunch& L, const GvmWarp& ws, GvmCons& C, const GvmStage& st, float (&acc)[4],
                          const float* srinv) {
    if (!C.glob) {
        const uint32_t a0 = C.sa + (uint32_t)(C.kc * GVM_COLS - C.kbase) * 2u;
        uint4 bh[4], bl[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            bh[j] = lds16(a0 + 64 * j);
            bl[j] = lds16(a0 + C.lo + 64 * j);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) gvm_mma_group(acc, st.a[j], st.b[j], bh[j], bl[j]);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 bh, bl;
            gvm_x_global(L, ws, C, j, bh, bl, srinv);
            gvm_mma_group(acc, st.a[j], st.b[j], bh, bl);
        }
    }
    ++C.kc;
}

// The op reads normalised sources with partial sums: its sums get 1/rms of
// the activation row in the epilogue (all of an op's segments read the same
// kind of source).
ES_DEV bool gvm_op_scaled(const GvLaunch& L, const GvOp& o) {
    const GvXSrc& x = L.xs[L.segs[o.seg0].xs];
    return x.kind == XS_NORM && x.ss_tiles > 0;
}

// Epilogue of one 16-row tile from the D fragments: lane (g, c) holds rows
// (n0+g, n0+g+8) x activation rows (2c, 2c+1).  With `ss`, also the sums of
// squares of the post-norm's input (h + add) over these 16 columns, per
// activation row, for the next launch's normalisation (deterministic: a
// fixed shuffle order).
ES_DEV void gvm_epilogue(const GvLaunch& L, const GvOp& o, int n0, const float (&v0)[4], const float (&v1)[4],
                         bool ss, const float* srinv) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const bool scaled = gvm_op_scaled(L, o);
    float sq[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int m = 2 * c + (e & 1), n = n0 + g + (e >> 1) * 8;
        if (m >= L.M || n >= o.N) continue;
        float* y = o.y + (size_t)m * o.ldy + n;
        const float f = scaled ? srinv[m] : 1.0f;
        const float r0 = v0[e] * f, r1 = v1[e] * f;
        float out;
        switch (o.epi) {
            case GEPI_STORE: out = r0; break;
            case GEPI_ACC: out = __ldcg(y) + r0; break;
            case GEPI_ACC_ADD: out = __ldcg(y) + r0 + __ldcg(o.add + (size_t)m * o.ldy + n); break;
            default: out = silu_f(r0) * r1; break;
        }
        *y = out;
        if (ss) {
            const GvPost& p = L.post;
            const size_t i = (size_t)m * p.K + n;
            float t = o.y == p.h ? out : __ldcg(p.h + i);
            if (p.add) t += o.y == p.add ? out : __ldcg(p.add + i);
            sq[e & 1] += t * t;
        }
    }
    if (ss) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            sq[0] += __shfl_xor_sync(0xffffffffu, sq[0], off);
            sq[1] += __shfl_xor_sync(0xffffffffu, sq[1], off);
        }
        if (g == 0) {
            float* dst = L.post.ssp + (size_t)(n0 / GVM_ROWS) * L.M;
            if (2 * c < L.M) dst[2 * c] = sq[0];
            if (2 * c + 1 < L.M) dst[2 * c + 1] = sq[1];
        }
    }
}

// 1/rms of this launch's normalised rows from the producer's sums of squares
// (first XS_NORM source with partials; all of a launch's normalised sources
// share h, add and rows).  Warp m handles row m: gvm_rinv_issue requests up
// to 8 partials per lane before the staging, gvm_rinv_finish adds them (and
// any further ones) lane-strided, then in a fixed shuffle order, so every CTA
// gets the same value.
struct GvmRinv { float r[8]; int xi; };

ES_DEV void gvm_rinv_issue(const GvLaunch& L, GvmRinv& R) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    R.xi = -1;
    for (int i = 0; i < L.nxs; ++i)
        if (L.xs[i].kind == XS_NORM && L.xs[i].ss_tiles > 0) { R.xi = i; break; }
#pragma unroll
    for (int u = 0; u < 8; ++u) R.r[u] = 0.f;
    if (R.xi < 0 || warp >= L.M) return;
    const GvXSrc& x = L.xs[R.xi];
    const int pr = warp * x.row_stride + x.row_off;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int i = lane + 32 * u;
        if (i < x.ss_tiles) R.r[u] = __ldcg(x.rinv + (size_t)i * x.ss_ld + pr);
    }
}

ES_DEV void gvm_rinv_finish(const GvLaunch& L, const GvmRinv& R, float* srinv) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (R.xi < 0 || warp >= L.M) return;
    const GvXSrc& x = L.xs[R.xi];
    const int pr = warp * x.row_stride + x.row_off;
    float t = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) t += R.r[u];
    // further partials (more than 256 tiles) in batches of 8 loads in flight,
    // added in the same lane-strided order
    for (int i0 = lane + 256; i0 < x.ss_tiles; i0 += 256) {
        float r[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + 32 * u;
            r[u] = i < x.ss_tiles ? __ldcg(x.rinv + (size_t)i * x.ss_ld + pr) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (i0 + 32 * u < x.ss_tiles) t += r[u];
    }
    t = warp_sum(t);
    if (lane == 0) srinv[warp] = 1.0f / sqrtf(t / (float)x.K + x.eps);
}


template <int NW>
__global__ void __launch_bounds__(NW * 32, NW == GV_WARPS ? GV_CTAS_PER_SM : 1)
gvm_kernel(const GvLaunch* __restrict__ Lg, float* __restrict__ scratch, int* __restrict__ counters,
           int* __restrict__ done) {
    extern __shared__ __align__(16) unsigned char gvm_xsm[];
    __shared__ __align__(16) GvLaunch L;
    __shared__ GvmWin win[GVM_NWIN];
    __shared__ GvmWarp wstate[NW];
    __shared__ float srinv[GV_MAXM];
    __shared__ int s_nwin, s_items, s_last, s_done;
    gv_load_desc(L, Lg);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q = L.q, cta = blockIdx.x;
    const int S0 = cta * q, S1 = min(L.nstages, S0 + q);
    GvmWarp& ws = wstate[warp];
    // nothing here depends on the previous kernel: the windows and the first
    // GVM_D - 1 stages of weights are set up before waiting for it
    if (tid == 0) {
        int used;
        s_nwin = gvm_windows(L, S0, S1, win, L.x_smem_floats, &s_items, &used);
    }
    GvmStage ring[GVM_D];
    GvmIssue I;
    int s_issue = S0;
    ws.ip = ws.cp = gvm_seek(L, S0);
    ws.is = ws.cs = S0;
    gvm_issue_begin<NW>(L, ws, I, S1);
#pragma unroll
    for (int i = 0; i < GVM_D - 1; ++i)
        if (s_issue < S1) { gvm_issue_step<NW>(L, ws, I, ring[i], S1); ++s_issue; }
    __syncthreads();
    grid_dep_wait();
    grid_dep_launch();
    const int nwin = s_nwin;
    {
        GvmRinv R;
        gvm_rinv_issue(L, R);
        // The ring's other stage: with more stages to come it goes out once
        // the staging loads are done (issued earlier, its loads queue ahead
        // of them); a CTA whose stages all fit the ring issues it first, so
        // that its latency hides behind the staging.
        if (S1 - S0 <= GVM_D) {
            if (s_issue < S1) { gvm_issue_step<NW>(L, ws, I, ring[GVM_D - 1], S1); ++s_issue; }
            gvm_stage_small<NW * 32>(L, win, nwin, gvm_xsm, srinv);  // ends with a barrier
        } else {
            gvm_stage<NW * 32>(L, win, nwin, gvm_xsm, srinv);  // ends with a barrier
            if (s_issue < S1) { gvm_issue_step<NW>(L, ws, I, ring[GVM_D - 1], S1); ++s_issue; }
        }
        gvm_rinv_finish(L, R, srinv);
        __syncthreads();
    }

    GvmCons C;
    gvm_cons_begin(L, ws, C, win, nwin, gvm_xsm, S1);
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    int blk_first = S0 - (S0 - L.ops[ws.op].stage0) % L.ops[ws.op].spt;
    for (int s = S0; s < S1; s += GVM_D) {
#pragma unroll
        for (int i = 0; i < GVM_D; ++i) {
            const int si = s + i;
            if (si >= S1) break;
            if (C.set == 0) gvm_cons_step(L, ws, C, ring[i], acc0, srinv);
            else gvm_cons_step(L, ws, C, ring[i], acc1, srinv);
            // refill the slot just multiplied: GVM_D stages stay in flight
            if (s_issue < S1) {
                gvm_issue_step<NW>(L, ws, I, ring[i], S1);
                ++s_issue;
            }
            if (C.kc < C.kc_end) continue;
            if (C.tile_end || si + 1 == S1) {
                // ---- finish the block (or this CTA's part of it); CTA-uniform
                const GvOp& o = L.ops[ws.op];
                const bool two = o.epi == GEPI_SWIGLU;
                const int blk_last = blk_first + o.spt - 1;
                bool do_epi = blk_first >= S0 && blk_last < S1;
                if (!do_epi) {
                    const int sid = S0 >= blk_first ? 0 : 1;
                    float* part = scratch + ((size_t)((cta * 2 + sid) * NW + warp) * 2) * 128 + lane * 4;
                    *reinterpret_cast<float4*>(part) = make_float4(acc0[0], acc0[1], acc0[2], acc0[3]);
                    if (two) *reinterpret_cast<float4*>(part + 128) = make_float4(acc1[0], acc1[1], acc1[2], acc1[3]);
                    __syncthreads();
                    const int c_first = blk_first / q, c_last = blk_last / q;
                    const int gblk = o.tile0 + ws.tile;
                    const int old = cta_arrive(counters + gblk);
                    if (tid == 0) s_last = old == c_last - c_first;
                    __syncthreads();
                    if (s_last) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc0[e] = acc1[e] = 0.f;
                        // partials of CTAs c_first..c_last, summed in CTA order;
                        // the loads of a batch are all in flight together
                        constexpr int RB = 8;
                        for (int set = 0; set < (two ? 2 : 1); ++set) {
                            float v[4] = {0.f, 0.f, 0.f, 0.f};
                            for (int cb = c_first; cb <= c_last; cb += RB) {
                                float4 pv[RB];
#pragma unroll
                                for (int u = 0; u < RB; ++u) {
                                    const int cc = cb + u;
                                    pv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                                    if (cc <= c_last) {
                                        const int sd = cc * q >= blk_first ? 0 : 1;
                                        pv[u] = __ldcg(reinterpret_cast<const float4*>(
                                            scratch + ((size_t)((cc * 2 + sd) * NW + warp) * 2 + set) * 128 +
                                            lane * 4));
                                    }
                                }
#pragma unroll
                                for (int u = 0; u < RB; ++u) {
                                    v[0] += pv[u].x; v[1] += pv[u].y; v[2] += pv[u].z; v[3] += pv[u].w;
                                }
                            }
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                if (set == 0) acc0[e] = v[e];
                                else acc1[e] = v[e];
                            }
                        }
                        if (tid == 0) counters[gblk] = 0;
                        do_epi = true;
                    }
                    // every thread has read s_last before a later block changes it
                    __syncthreads();
                }
                if (do_epi)
                    gvm_epilogue(L, o, ws.tile * (NW * GVM_ROWS) + warp * GVM_ROWS, acc0, acc1,
                                 L.post.ssp != nullptr && ws.op == L.post.op, srinv);
#pragma unroll
                for (int e = 0; e < 4; ++e) acc0[e] = acc1[e] = 0.f;
                blk_first = blk_last + 1;
            }
            if (si + 1 < S1) gvm_cons_begin(L, ws, C, win, nwin, gvm_xsm, S1);
        }
    }
    // (the last-CTA norm pass is sized for 8-warp CTAs; bf16 launches pass
    // sums of squares instead)
    if (NW == GV_WARPS && L.post.rows > 0 && !L.post.ssp) {
        __syncthreads();
        const int old = cta_arrive(done);
        if (tid == 0) s_done = old == (int)gridDim.x - 1;
        __syncthreads();
        if (s_done) {
            post_rinv(L.post);
            if (tid == 0) *done = 0;
        }
    }
}

// ------------------------------------------------------------ SIMT GEMM
// The same launch descriptor for many rows (prompt prefill): 64x64 output
// tiles, float32 FMA.  grid.x = 64-row tiles over all ops, grid.y = 64-row
// blocks of the M input rows.  Every source is read from global memory.
constexpr int GB = 64, GK = 32;
template <typename T>
__global__ void __launch_bounds__(256) gemm_kernel(const GvLaunch* __restrict__ L) {
    __shared__ float xs[GK][GB + 4];
    __shared__ float ws[GK][GB + 4];
    grid_dep_wait();
    const int tile = blockIdx.x, M = L->M;
    int oi = 0;
    while (oi + 1 < L->nops && L->ops[oi + 1].tile64_0 <= tile) ++oi;
    const GvOp& op = L->ops[oi];
    const int n0 = (tile - op.tile64_0) * GB, m0 = blockIdx.y * GB;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[2][4][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jx = 0; jx < 4; ++jx) acc[u][i][jx] = 0.f;
    for (int s = 0; s < op.nseg; ++s) {
        const GvSeg sg = L->segs[op.seg0 + s];
        const GvXSrc& xd = L->xs[sg.xs];
        const float* X = xd.src + (size_t)xd.row_off * xd.ld;
        const size_t xst = (size_t)xd.row_stride * xd.ld;
        const T* W = (const T*)sg.W;
        const int u = sg.set;
        for (int k0 = 0; k0 < sg.K; k0 += GK) {
            for (int t = threadIdx.x; t < GB * GK; t += 256) {
                const int r = t / GK, c = t % GK;
                const int m = m0 + r, n = n0 + r, k = k0 + c;
                xs[c][r] = (m < M && k < sg.K) ? X[(size_t)m * xst + k] : 0.f;
                ws[c][r] = (n < op.N && k < sg.K) ? to_f32(W[(size_t)n * sg.K + k]) : 0.f;
            }
            __syncthreads();
#pragma unroll 8
            for (int c = 0; c < GK; ++c) {
                float av[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) av[i] = xs[c][ty * 4 + i];
#pragma unroll
                for (int jx = 0; jx < 4; ++jx) bv[jx] = ws[c][tx * 4 + jx];
                if (u == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int jx = 0; jx < 4; ++jx) acc[0][i][jx] = fmaf(av[i], bv[jx], acc[0][i][jx]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int jx = 0; jx < 4; ++jx) acc[1][i][jx] = fmaf(av[i], bv[jx], acc[1][i][jx]);
                }
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int jx = 0; jx < 4; ++jx) {
            const int n = n0 + tx * 4 + jx;
            if (n >= op.N) continue;
            float* y = op.y + (size_t)m * op.ldy + n;
            switch (op.epi) {
                case GEPI_STORE: *y = acc[0][i][jx]; break;
                case GEPI_ACC: *y += acc[0][i][jx]; break;
                case GEPI_ACC_ADD: *y += acc[0][i][jx] + op.add[(size_t)m * op.ldy + n]; break;
                default: *y = silu_f(acc[0][i][jx]) * acc[1][i][jx]; break;
            }
        }
    }
}

}  // namespace es
