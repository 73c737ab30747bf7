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
// Activation inputs ("x sources") are either raw float rows in global memory
// or RMSNorm(h [+ add]) * gain of a residual row, normalised on the fly while
// they are staged into shared memory (the norm is fused into the GEMV).
//
// Data movement.  A stage is 32 consecutive rows x 512 bytes of one matrix.
// Each consumer warp owns 4 rows of the 32-row tile and every lane one
// 16-byte column vector of each, read with 128-bit non-allocating loads
// straight into registers, several stages ahead (HBM latency is covered by
// the loads in flight of two resident CTAs per SM), so an activation vector
// read from shared memory is reused for 4 weight rows.  One-dimensional bulk
// copies (cp.async.bulk) of 512-byte row pieces into a shared-memory ring
// were measured on B300 at under 2 TB/s for this access shape, against about
// 7 TB/s for plain 16-byte loads, so the weights do not go through TMA.
// Before griddepcontrol.wait every thread prefetches its first weight
// vectors into L2: they never depend on the previous kernel, so they stream
// in while that kernel drains.
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

constexpr int GV_WARPS = 8;                    // consumer warps
constexpr int GV_THREADS = GV_WARPS * 32;
constexpr int GV_R = 4;                        // rows per consumer warp
constexpr int GV_RT = GV_WARPS * GV_R;         // rows per tile (32)
constexpr int GV_ROW_BYTES = 512;              // bytes of one row per stage
constexpr int GV_MAXM = 8;
constexpr int GV_MAX_XS = 16;
constexpr int GV_MAX_SEG = 16;
constexpr int GV_MAX_OPS = 32;
constexpr int GV_XSMEM_MAX = 24 * 1024;        // floats of staged activations (96 KB)
constexpr int GV_CTAS_PER_SM = 2;
constexpr int GV_SCRATCH_CTAS = 1024;          // partial-sum slots
constexpr int GV_COUNTERS = 65536;             // arrival counters (tiles per launch)
constexpr int GV_SCRATCH_FLOATS = GV_SCRATCH_CTAS * 2 * 2 * GV_THREADS;

enum { XS_RAW = 0, XS_NORM = 1 };
enum { GEPI_STORE = 0, GEPI_ACC = 1, GEPI_ACC_ADD = 2, GEPI_SWIGLU = 3 };

// Input row r (< M) of x source i is row r*row_stride + row_off of `src`
// (leading dimension ld).  NORM: x = (src + add) / rms(src + add) * gain,
// rms over the K columns; `add` uses the same row mapping and ld.
struct GvXSrc {
    const float* src; const float* add; const void* gain;
    int K, ld, row_stride, row_off, kind;
    int smem_off;  // float offset in the staged region, or -1: read from global
};
struct GvSeg { const void* W; int K, xs, set, nck; };
struct GvOp {
    GvSeg seg[GV_MAX_SEG];
    int nseg, epi, N, ldy;
    float* y; const float* add;
    int ntiles, spt;       // 32-row tiles, stages per tile
    int tile0, stage0;     // launch-wide tile / stage index of the op's first
    int tile64_0, pad_;    // (SIMT GEMM) first 64-row tile of the op
};
struct GvLaunch {
    int nops, nxs, M, ntiles, nstages, q, x_smem_floats, ntiles64;
    float eps; int pad_;
    GvXSrc xs[GV_MAX_XS];
    GvOp ops[GV_MAX_OPS];
};

// ------------------------------------------------------------ PTX helpers
ES_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
ES_DEV void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

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
        while (c >= o.seg[seg].nck) { c -= o.seg[seg].nck; ++seg; }
        kc = c;
    }
    // advance by n chunks within the current segment (n <= chunks left in
    // it); true when that finished the tile
    ES_DEV bool advance(int n) {
        const GvOp& o = L->ops[op];
        kc += n;
        if (kc < o.seg[seg].nck) return false;
        kc = 0;
        if (++seg < o.nseg) return false;
        seg = 0;
        if (++tile >= o.ntiles) { tile = 0; ++op; }
        return true;
    }
    // true when the step crossed into a new tile
    ES_DEV bool next() {
        const GvOp& o = L->ops[op];
        if (++kc < o.seg[seg].nck) return false;
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

// ------------------------------------------------------------ kernel
ES_DEV void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// acc[r][m] += W-vector(r) . x-vector(m) for one 16-byte column vector.
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

template <typename T, int M>
__global__ void __launch_bounds__(GV_THREADS, 2)
gv_kernel(const GvLaunch* __restrict__ L, float* __restrict__ scratch, int* __restrict__ counters) {
    constexpr int EPV = 16 / sizeof(T);            // weights per 16-byte vector
    constexpr int SC = GV_ROW_BYTES / sizeof(T);   // columns per stage: one vector per lane
    constexpr int NV = GV_R * M;
    constexpr int U = M <= 2 ? 4 : 2;              // stages whose loads are issued together
    extern __shared__ __align__(16) float xsm[];
    __shared__ const float* xs_base[GV_MAX_XS];
    __shared__ int xs_stride[GV_MAX_XS];
    __shared__ float xs_rinv[GV_MAX_XS * GV_MAXM];
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Q = L->q;
    const int s_begin = blockIdx.x * Q;
    const int s_end = min(L->nstages, s_begin + Q);

    // Weights never depend on the previous kernel: pull this CTA's first
    // stages into L2 while that kernel drains.
    {
        GvWalk w;
        w.seek(L, s_begin);
        const GvOp& o = L->ops[w.op];
        const GvSeg& sg = o.seg[w.seg];
        const int n = min(min(s_end - s_begin, 2 * U), sg.nck - w.kc);
#pragma unroll
        for (int r = 0; r < GV_R; ++r) {
            const int row = min(w.tile * GV_RT + warp * GV_R + r, o.N - 1);
            const T* base = (const T*)sg.W + (size_t)row * sg.K + lane * EPV;
            for (int u = 0; u < n; ++u)
                if ((w.kc + u) * SC + lane * EPV < sg.K) prefetch_l2(base + (size_t)(w.kc + u) * SC);
        }
    }
    grid_dep_wait();
    const int nxs = L->nxs;
    // rms of every normalised source row (warp per row)
    for (int p = warp; p < nxs * M; p += GV_WARPS) {
        const int i = p / M, m = p % M;
        const GvXSrc& x = L->xs[i];
        if (x.kind != XS_NORM) continue;
        const size_t r = (size_t)(m * x.row_stride + x.row_off) * x.ld;
        const float* hr = x.src + r;
        const float* ar = x.add ? x.add + r : nullptr;
        float ss = 0.f;
        for (int k = lane * 4; k < x.K; k += 128) {
            float4 v = *reinterpret_cast<const float4*>(hr + k);
            if (ar) {
                const float4 a = *reinterpret_cast<const float4*>(ar + k);
                v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
            }
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
        ss = warp_sum(ss);
        if (lane == 0) xs_rinv[p] = 1.0f / sqrtf(ss / (float)x.K + L->eps);
    }
    if (tid < nxs) {
        const GvXSrc& x = L->xs[tid];
        if (x.smem_off >= 0) {
            xs_base[tid] = xsm + x.smem_off;
            xs_stride[tid] = x.K;
        } else {
            xs_base[tid] = x.src + (size_t)x.row_off * x.ld;
            xs_stride[tid] = x.row_stride * x.ld;
        }
    }
    __syncthreads();
    // stage shared-memory sources (normalised ones scaled by rinv * gain)
    for (int i = 0; i < nxs; ++i) {
        const GvXSrc& x = L->xs[i];
        if (x.smem_off < 0) continue;
        float* dst = xsm + x.smem_off;
        const int K4 = x.K / 4;
        for (int t = tid; t < M * K4; t += GV_THREADS) {
            const int m = t / K4, k = (t % K4) * 4;
            const size_t r = (size_t)(m * x.row_stride + x.row_off) * x.ld + k;
            float4 v = *reinterpret_cast<const float4*>(x.src + r);
            if (x.kind == XS_NORM) {
                if (x.add) {
                    const float4 a = *reinterpret_cast<const float4*>(x.add + r);
                    v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
                }
                const float ri = xs_rinv[i * M + m];
                const T* g = (const T*)x.gain + k;
                v.x = v.x * ri * to_f32(g[0]);
                v.y = v.y * ri * to_f32(g[1]);
                v.z = v.z * ri * to_f32(g[2]);
                v.w = v.w * ri * to_f32(g[3]);
            }
            *reinterpret_cast<float4*>(dst + (size_t)m * x.K + k) = v;
        }
    }
    __syncthreads();
    grid_dep_launch();

    float acc[GV_R][M];
#pragma unroll
    for (int r = 0; r < GV_R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;
    float vset[2] = {0.f, 0.f};  // reduced sums of finished accumulator sets (lane-distributed)
    int cur_set = -1;

    GvWalk w;
    w.seek(L, s_begin);
    int tile_first = s_begin - ((s_begin - L->ops[w.op].stage0) % L->ops[w.op].spt);
    int s = s_begin;
    while (s < s_end) {
        // one run: consecutive column chunks of a single segment
        const int cur_op = w.op, cur_tile = w.tile;
        const GvOp& o = L->ops[cur_op];
        const GvSeg& sg = o.seg[w.seg];
        const int run = min(s_end - s, sg.nck - w.kc);
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
        {
            const int K = sg.K;
            const T* wr[GV_R];
#pragma unroll
            for (int r = 0; r < GV_R; ++r)  // rows past N read the last row; their sums are dropped
                wr[r] = (const T*)sg.W + (size_t)min(cur_tile * GV_RT + warp * GV_R + r, o.N - 1) * K + lane * EPV;
            const float* xb = xs_base[sg.xs] + lane * EPV;
            const int xst = xs_stride[sg.xs];
            int kc = w.kc;
            const int kc_end = kc + run;
            const int kc_full = min(kc_end, K / SC);  // chunks lying wholly inside K
            for (; kc + U <= kc_full; kc += U) {
                uint4 wv[U][GV_R];
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int r = 0; r < GV_R; ++r) wv[u][r] = ld_stream16(wr[r] + (size_t)(kc + u) * SC);
#pragma unroll
                for (int u = 0; u < U; ++u) gv_fma<T, M>(wv[u], xb + (size_t)(kc + u) * SC, xst, acc);
            }
            for (; kc < kc_full; ++kc) {
                uint4 wv[GV_R];
#pragma unroll
                for (int r = 0; r < GV_R; ++r) wv[r] = ld_stream16(wr[r] + (size_t)kc * SC);
                gv_fma<T, M>(wv, xb + (size_t)kc * SC, xst, acc);
            }
            if (kc < kc_end && kc * SC + lane * EPV < K) {  // ragged last chunk of the segment
                uint4 wv[GV_R];
#pragma unroll
                for (int r = 0; r < GV_R; ++r) wv[r] = ld_stream16(wr[r] + (size_t)kc * SC);
                gv_fma<T, M>(wv, xb + (size_t)kc * SC, xst, acc);
            }
        }
        const bool tile_end = w.advance(run);
        s += run;
        if (!(tile_end || s == s_end)) continue;

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
        const int gtile = o.tile0 + cur_tile;
        bool do_epi = complete;
        if (!complete) {
            const int sid = s_begin >= tile_first ? 0 : 1;
            float* part = scratch + ((size_t)(blockIdx.x * 2 + sid) * 2) * GV_THREADS + tid;
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
            const int n = cur_tile * GV_RT + warp * GV_R + r;
            if (n < o.N) {
                float* y = o.y + (size_t)m * o.ldy + n;
                switch (o.epi) {
                    case GEPI_STORE: *y = v0; break;
                    case GEPI_ACC: *y += v0; break;
                    case GEPI_ACC_ADD: *y += v0 + o.add[(size_t)m * o.ldy + n]; break;
                    default: *y = silu_f(v0) * v1; break;
                }
            }
        }
        tile_first = tile_last + 1;
    }
}

// ------------------------------------------------------------ SIMT GEMM
// The same launch descriptor for many rows (prompt prefill): 64x64 output
// tiles, float32 FMA.  Every x source must be RAW (normalised inputs are
// produced beforehand).  grid.x = 64-row tiles over all ops, grid.y = 64-row
// blocks of the M input rows.
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
        const GvSeg sg = op.seg[s];
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
