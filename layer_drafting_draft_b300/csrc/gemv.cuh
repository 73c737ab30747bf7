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
    ES_DEV void seek(const GvLaunch* L_, int s) {
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
    ES_DEV bool advance(int n) {
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
// Executed by one whole CTA (blockDim.x a multiple of 32) once the rows it
// reads are final: a warp per row.
ES_DEV void post_rinv(const GvPost& p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int r = warp; r < p.rows; r += nw) {
        const size_t base = (size_t)(r * p.row_stride + p.row_off) * p.K;
        float ss = 0.f;
#pragma unroll 4
        for (int k = lane * 4; k < p.K; k += 128) {
            float4 v = __ldcg(reinterpret_cast<const float4*>(p.h + base + k));
            if (p.add) {
                const float4 a = __ldcg(reinterpret_cast<const float4*>(p.add + base + k));
                v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
            }
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = warp_sum(ss);
        if (lane == 0) p.rinv[r] = 1.0f / sqrtf(ss / (float)p.K + p.eps);
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
