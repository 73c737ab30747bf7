// Kernels of the speculative-decoding hot path (sm_103a).
//
// Activations and accumulation are float32; weights and KV cache are T
// (float or bf16).  Rows of a forward pass are described by device arrays
// row_pos / row_seq / row_tok, so the same launches (and CUDA graphs) serve
// every phase; a row with row_pos < 0 is inactive (no KV write, no output).
#pragma once
#include "common.cuh"

namespace es {

constexpr int PAGE = 64;          // KV page: 64 positions
constexpr int MAX_SEG = 16;       // K-concatenated segments per GEMV op
constexpr int MAX_GROUP = 8;      // layers per fused set (q heads per kv head <= 16)
constexpr int GEMV_WARPS = 8;     // output rows per GEMV tile (one per warp)
constexpr int MAX_GQA = 16;
constexpr int STATUS_BAD_POS = 1; // device status bits
constexpr int STATUS_BAD_TOKEN = 2;

enum { KIND_HOST = 0, KIND_CALIB = 1, KIND_FUZZY = 2, KIND_VERIFY = 3 };
enum { EPI_STORE = 0, EPI_ACC = 1, EPI_SWIGLU = 2 };

// -------------------------------------------------------------------- rows
// KIND_CALIB : rows (b, i), i = 0..gamma: position n_b - gamma - 1 + i (the
//              last gamma+1 committed tokens; recomputing already-exact
//              positions reproduces their entries, so the window always covers
//              every pending token)
// KIND_FUZZY : rows b, position n_b + step - 1, token d[b][step-1]
// KIND_VERIFY: rows (b, j), j = 0..gamma: position n_b - 1 + j, token
//              x_{n_b-1} for j = 0, d[b][j-1] otherwise
// KIND_HOST  : row arrays already filled by the host
template <typename T>
__global__ void prep_embed_kernel(int kind, int step, int gamma, int M,
                                  const int* __restrict__ n_commit, const int* __restrict__ tokens,
                                  int max_seq, const int* __restrict__ dtok, int gmax,
                                  int* row_pos, int* row_seq, int* row_tok,
                                  const T* __restrict__ E, float* __restrict__ h, int d, int V,
                                  int* status) {
    grid_dep_wait();
    const int m = blockIdx.x;
    if (m >= M) return;
    int b, pos, tok;
    if (kind == KIND_HOST) {
        b = row_seq[m]; pos = row_pos[m]; tok = row_tok[m];
    } else if (kind == KIND_CALIB) {
        b = m / (gamma + 1);
        const int i = m % (gamma + 1);
        pos = n_commit[b] - (gamma + 1) + i;
        if (pos < 0) pos = -1;
        tok = (pos >= 0 && pos < max_seq) ? tokens[(size_t)b * max_seq + pos] : 0;
    } else if (kind == KIND_FUZZY) {
        b = m;
        pos = n_commit[b] + step - 1;
        tok = dtok[b * gmax + step - 1];
    } else {
        b = m / (gamma + 1);
        const int j = m % (gamma + 1);
        pos = n_commit[b] - 1 + j;
        tok = j > 0 ? dtok[b * gmax + j - 1] : (pos >= 0 && pos < max_seq) ? tokens[(size_t)b * max_seq + pos] : 0;
    }
    if (pos >= max_seq) { if (threadIdx.x == 0) atomicOr(status, STATUS_BAD_POS); pos = -1; }
    if (tok < 0 || tok >= V) { if (threadIdx.x == 0) atomicOr(status, STATUS_BAD_TOKEN); tok = 0; }
    if (threadIdx.x == 0 && kind != KIND_HOST) { row_pos[m] = pos; row_seq[m] = b; row_tok[m] = tok; }
    const T* e = E + (size_t)tok * d;
    for (int i = threadIdx.x; i < d; i += blockDim.x) h[(size_t)m * d + i] = to_f32(e[i]);
}

// -------------------------------------------------------------------- RMSNorm
// out_j[r] = RMSNorm(h[src], g_j) for every job j, with src = r*stride + off.
// If `add` is set, h[src] += add[src] first (written back).
struct NormArgs {
    float* h; const float* add; int d; float eps; int src_stride, src_off;
    int njobs; const void* g[2 * MAX_GROUP]; float* out[2 * MAX_GROUP]; int out_ld;
};
template <typename T>
__global__ void norm_kernel(NormArgs a) {
    __shared__ float red[32];
    grid_dep_wait();
    const int r = blockIdx.x;
    const size_t src = (size_t)r * a.src_stride + a.src_off;
    float* hr = a.h + src * a.d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < a.d; i += blockDim.x) {
        float v = hr[i];
        if (a.add) { v += a.add[src * a.d + i]; hr[i] = v; }
        ss += v * v;
    }
    ss = block_sum(ss, red);
    const float rinv = 1.0f / sqrtf(ss / (float)a.d + a.eps);
    for (int j = 0; j < a.njobs; ++j) {
        const T* g = (const T*)a.g[j];
        float* o = a.out[j] + (size_t)r * a.out_ld;
        for (int i = threadIdx.x; i < a.d; i += blockDim.x) o[i] = hr[i] * rinv * to_f32(g[i]);
    }
}

// -------------------------------------------------------------------- GEMV
// One op: for n < N and input row m < M
//   r[m][n] = sum_s  W_s[n, :] . x_s[m, :]        (K-concatenated segments)
//   EPI_STORE : y[m][n] = r;  EPI_ACC : y[m][n] += r
//   EPI_SWIGLU: y[m][n] = silu(W_0[n].x_0[m]) * (W_1[n].x_1[m])  (nseg == 2)
// A launch runs several ops ("wide" fusion over the layers of a set); op i
// owns tiles [tile0_i, tile0_{i+1}) of GEMV_WARPS rows.
struct GemvSeg { const void* W; const float* x; int K; int ldx; };
struct GemvOp {
    GemvSeg seg[MAX_SEG];
    int nseg, epi, N, ldy, tile0, pad_;
    float* y;
};

template <typename T, int M>
ES_DEV void dot_seg(const T* __restrict__ W, const float* __restrict__ x, int K, int ldx,
                    float (&acc)[M], int lane) {
    constexpr int EPV = Vec16<T>::N;
#pragma unroll 4
    for (int k = lane * EPV; k < K; k += 32 * EPV) {
        float w[EPV];
        unpack16(ld_stream16(W + k), w, T());
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const float4* xp = reinterpret_cast<const float4*>(x + (size_t)m * ldx + k);
#pragma unroll
            for (int e = 0; e < EPV / 4; ++e) {
                const float4 xv = __ldg(xp + e);
                acc[m] = fmaf(w[4 * e + 0], xv.x, acc[m]);
                acc[m] = fmaf(w[4 * e + 1], xv.y, acc[m]);
                acc[m] = fmaf(w[4 * e + 2], xv.z, acc[m]);
                acc[m] = fmaf(w[4 * e + 3], xv.w, acc[m]);
            }
        }
    }
}

ES_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

template <typename T, int M>
__global__ void __launch_bounds__(GEMV_WARPS * 32)
gemv_kernel(const GemvOp* __restrict__ ops, int nops, int ntiles) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dep_wait();
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        int oi = 0;
        while (oi + 1 < nops && ops[oi + 1].tile0 <= tile) ++oi;
        const GemvOp* op = ops + oi;
        const int row = (tile - op->tile0) * GEMV_WARPS + warp;
        if (row >= op->N) continue;
        float a0[M], a1[M];
#pragma unroll
        for (int m = 0; m < M; ++m) { a0[m] = 0.f; a1[m] = 0.f; }
        const int epi = op->epi;
        if (epi == EPI_SWIGLU) {
            dot_seg<T, M>((const T*)op->seg[0].W + (size_t)row * op->seg[0].K, op->seg[0].x,
                          op->seg[0].K, op->seg[0].ldx, a0, lane);
            dot_seg<T, M>((const T*)op->seg[1].W + (size_t)row * op->seg[1].K, op->seg[1].x,
                          op->seg[1].K, op->seg[1].ldx, a1, lane);
        } else {
            for (int s = 0; s < op->nseg; ++s)
                dot_seg<T, M>((const T*)op->seg[s].W + (size_t)row * op->seg[s].K, op->seg[s].x,
                              op->seg[s].K, op->seg[s].ldx, a0, lane);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) { a0[m] = warp_sum(a0[m]); a1[m] = warp_sum(a1[m]); }
        if (lane == 0) {
            float* y = op->y + row;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float* ym = y + (size_t)m * op->ldy;
                if (epi == EPI_STORE) *ym = a0[m];
                else if (epi == EPI_ACC) *ym += a0[m];
                else *ym = silu(a0[m]) * a1[m];
            }
        }
    }
}

// -------------------------------------------------------------------- GEMM
// Same ops for M > 8 rows (prefill chunks): 64x64 output tiles, K step 32,
// float32 SIMT.  grid.x = tiles of 64 output features over all ops,
// grid.y = tiles of 64 input rows.
constexpr int GB = 64, GK = 32;
template <typename T>
__global__ void __launch_bounds__(256)
gemm_kernel(const GemvOp* __restrict__ ops, int nops, int M) {
    __shared__ float xs[GK][GB + 4];
    __shared__ float ws[1][GK][GB + 4];
    grid_dep_wait();
    const int tile = blockIdx.x;
    int oi = 0;
    while (oi + 1 < nops && ops[oi + 1].tile0 <= tile) ++oi;
    const GemvOp* op = ops + oi;
    const int n0 = (tile - op->tile0) * GB, m0 = blockIdx.y * GB;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int epi = op->epi;
    float acc[2][4][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[u][i][j] = 0.f;
    const int nseg = op->nseg;
    for (int s = 0; s < nseg; ++s) {
        const GemvSeg sg = op->seg[s];
        const int u = (epi == EPI_SWIGLU && s == 1) ? 1 : 0;
        const T* W = (const T*)sg.W;
        for (int k0 = 0; k0 < sg.K; k0 += GK) {
            for (int t = threadIdx.x; t < GB * GK; t += 256) {
                const int r = t / GK, c = t % GK;
                const int m = m0 + r, n = n0 + r, k = k0 + c;
                xs[c][r] = (m < M && k < sg.K) ? sg.x[(size_t)m * sg.ldx + k] : 0.f;
                ws[0][c][r] = (n < op->N && k < sg.K) ? to_f32(W[(size_t)n * sg.K + k]) : 0.f;
            }
            __syncthreads();
#pragma unroll 8
            for (int c = 0; c < GK; ++c) {
                float av[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) av[i] = xs[c][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[j] = ws[0][c][tx * 4 + j];
                if (u == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[0][i][j] = fmaf(av[i], bv[j], acc[0][i][j]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[1][i][j] = fmaf(av[i], bv[j], acc[1][i][j]);
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
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= op->N) continue;
            float* y = op->y + (size_t)m * op->ldy + n;
            if (epi == EPI_STORE) *y = acc[0][i][j];
            else if (epi == EPI_ACC) *y += acc[0][i][j];
            else *y = silu(acc[0][i][j]) * acc[1][i][j];
        }
    }
}

// -------------------------------------------------------------------- RoPE + KV append
// Paged cache: element (page p, layer l, K|V, kv head h, slot s, e) at
// ((((p*L + l)*2 + kv)*Hkv + h)*PAGE + s)*hd + e.
struct KVGeom {
    void* kv; const int* page_table; int pages_per_seq, L, Hkv, hd, max_seq;
};
template <typename T>
ES_DEV T* kv_ptr(const KVGeom& g, int seq, int pos, int layer, int kv, int h) {
    const int page = g.page_table[seq * g.pages_per_seq + pos / PAGE];
    const size_t off = ((((size_t)page * g.L + layer) * 2 + kv) * g.Hkv + h) * PAGE + pos % PAGE;
    return (T*)g.kv + off * g.hd;
}

struct RopeArgs {
    KVGeom g; const float* rope; int H, M;
    int nl; int layer[MAX_GROUP]; float* q[MAX_GROUP]; const float* k[MAX_GROUP];
    const float* v[MAX_GROUP];
    const int* row_pos; const int* row_seq;
};
// grid (M, nl); rotates q in place, writes rotated k and raw v to the cache.
template <typename T>
__global__ void rope_kv_kernel(RopeArgs a) {
    grid_dep_wait();
    const int m = blockIdx.x, j = blockIdx.y;
    const int pos = a.row_pos[m];
    if (pos < 0) return;
    const int seq = a.row_seq[m], hd = a.g.hd, half = hd / 2, H = a.H, Hkv = a.g.Hkv;
    const float* cs = a.rope + (size_t)pos * half * 2;
    float* q = a.q[j] + (size_t)m * H * hd;
    const float* k = a.k[j] + (size_t)m * Hkv * hd;
    const float* v = a.v[j] + (size_t)m * Hkv * hd;
    for (int t = threadIdx.x; t < (H + Hkv) * half; t += blockDim.x) {
        const int h = t / half, i = t % half;
        const float c = cs[2 * i], s = cs[2 * i + 1];
        if (h < H) {
            float* x = q + h * hd;
            const float x0 = x[i], x1 = x[i + half];
            x[i] = x0 * c - x1 * s;
            x[i + half] = x1 * c + x0 * s;
        } else {
            const int hk = h - H;
            const float* x = k + hk * hd;
            const float x0 = x[i], x1 = x[i + half];
            T* dst = kv_ptr<T>(a.g, seq, pos, a.layer[j], 0, hk);
            dst[i] = from_f32<T>(x0 * c - x1 * s);
            dst[i + half] = from_f32<T>(x1 * c + x0 * s);
        }
    }
    for (int t = threadIdx.x; t < Hkv * hd; t += blockDim.x) {
        const int hk = t / hd, e = t % hd;
        kv_ptr<T>(a.g, seq, pos, a.layer[j], 1, hk)[e] = from_f32<T>(v[hk * hd + e]);
    }
}

// -------------------------------------------------------------------- attention
// Split by KV page: CTA (row m, layer slot j * Hkv + kv head, page p) attends
// the row's query heads of that kv head over positions [64p, min(64p+64, pos+1))
// and writes an unnormalised partial (acc[hd], max, sum) per query head.
struct AttnArgs {
    KVGeom g; int H, M, nsplit;
    int nl; int layer[MAX_GROUP]; const float* q[MAX_GROUP]; float* out[MAX_GROUP];
    float* part;  // [M][nl][H][nsplit][hd + 2]
    const int* row_pos; const int* row_seq;
};
template <typename T>
__global__ void __launch_bounds__(128) attn_split_kernel(AttnArgs a) {
    __shared__ float qs[MAX_GQA * 256];
    __shared__ float sc[MAX_GQA][PAGE];
    grid_dep_wait();
    const int m = blockIdx.x, j = blockIdx.y / a.g.Hkv, hk = blockIdx.y % a.g.Hkv, p = blockIdx.z;
    const int pos = a.row_pos[m];
    if (pos < 0 || p * PAGE > pos) return;
    const int hd = a.g.hd, G = a.H / a.g.Hkv, seq = a.row_seq[m];
    const int n = min(PAGE, pos + 1 - p * PAGE);
    const float scale = 1.0f / sqrtf((float)hd);
    const float* q = a.q[j] + ((size_t)m * a.H + hk * G) * hd;
    for (int t = threadIdx.x; t < G * hd; t += blockDim.x) qs[t] = q[t] * scale;
    __syncthreads();
    const T* Kp = kv_ptr<T>(a.g, seq, p * PAGE, a.layer[j], 0, hk);
    const T* Vp = kv_ptr<T>(a.g, seq, p * PAGE, a.layer[j], 1, hk);
    // scores: thread -> (position i, head parity)
    {
        const int i = threadIdx.x % PAGE, hp = threadIdx.x / PAGE;
        if (i < n) {
            const T* kr = Kp + (size_t)i * hd;
            for (int h = hp; h < G; h += 2) {
                float s = 0.f;
                const float* qh = qs + h * hd;
                for (int e = 0; e < hd; ++e) s = fmaf(qh[e], to_f32(kr[e]), s);
                sc[h][i] = s;
            }
        }
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = warp; h < G; h += 4) {
        const float s0 = lane < n ? sc[h][lane] : -INFINITY;
        const float s1 = lane + 32 < n ? sc[h][lane + 32] : -INFINITY;
        const float mx = warp_max(fmaxf(s0, s1));
        const float e0 = lane < n ? expf(s0 - mx) : 0.f;
        const float e1 = lane + 32 < n ? expf(s1 - mx) : 0.f;
        sc[h][lane] = e0;
        sc[h][lane + 32] = e1;
        const float l = warp_sum(e0 + e1);
        if (lane == 0) {
            float* pp = a.part + ((((size_t)m * a.nl + j) * a.H + hk * G + h) * a.nsplit + p) * (hd + 2);
            pp[hd] = mx;
            pp[hd + 1] = l;
        }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < G * hd; t += blockDim.x) {
        const int h = t / hd, e = t % hd;
        float acc = 0.f;
        for (int i = 0; i < n; ++i) acc = fmaf(sc[h][i], to_f32(Vp[(size_t)i * hd + e]), acc);
        a.part[((((size_t)m * a.nl + j) * a.H + hk * G + h) * a.nsplit + p) * (hd + 2) + e] = acc;
    }
}

// grid (M, nl, H), block hd: merge the page partials of one query head.
__global__ void attn_combine_kernel(AttnArgs a) {
    grid_dep_wait();
    const int m = blockIdx.x, j = blockIdx.y, h = blockIdx.z, e = threadIdx.x, hd = a.g.hd;
    const int pos = a.row_pos[m];
    float* o = a.out[j] + ((size_t)m * a.H + h) * hd;
    if (pos < 0) { if (e < hd) o[e] = 0.f; return; }
    const int np = pos / PAGE + 1;
    const float* pp = a.part + (((size_t)m * a.nl + j) * a.H + h) * a.nsplit * (hd + 2);
    float mx = -INFINITY;
    for (int p = 0; p < np; ++p) mx = fmaxf(mx, pp[p * (hd + 2) + hd]);
    float num = 0.f, den = 0.f;
    for (int p = 0; p < np; ++p) {
        const float w = expf(pp[p * (hd + 2) + hd] - mx);
        den = fmaf(w, pp[p * (hd + 2) + hd + 1], den);
        if (e < hd) num = fmaf(w, pp[p * (hd + 2) + e], num);
    }
    if (e < hd) o[e] = num / den;
}

// -------------------------------------------------------------------- sampling
// Integer-quantised inverse CDF: W_i = floor(w_i * 2^40) (w_i >= 0 float32),
// T = sum W_i, t = floor(u * T / 2^64); result = first i whose inclusive
// prefix sum exceeds t.  Integer sums make the result independent of the
// summation order.  Returns -1 if T == 0.  Whole block participates;
// blockDim.x == 1024.
ES_DEV uint64_t q40(float w) { return (uint64_t)(w * 1099511627776.0f); }

ES_DEV uint64_t warp_incl_scan_u64(uint64_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

template <typename F>
ES_DEV int block_sample_q40(F weight, int V, uint64_t u, uint64_t* sh /* >= 34 */) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nt = blockDim.x;
    const int chunk = (V + nt - 1) / nt;
    const int b0 = min(V, tid * chunk), b1 = min(V, b0 + chunk);
    uint64_t s = 0;
    for (int i = b0; i < b1; ++i) s += q40(weight(i));
    const uint64_t incl = warp_incl_scan_u64(s, lane);
    __syncthreads();
    if (lane == 31) sh[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const uint64_t w = lane < (nt >> 5) ? sh[lane] : 0;
        const uint64_t wi = warp_incl_scan_u64(w, lane);
        sh[lane] = wi - w;  // exclusive warp offsets
        if (lane == 31) sh[32] = wi;  // total
    }
    __syncthreads();
    const uint64_t total = sh[32];
    const uint64_t excl = sh[wid] + incl - s;
    __syncthreads();
    if (tid == 0) sh[33] = (uint64_t)-1;
    __syncthreads();
    if (total == 0) return -1;
    const uint64_t t = __umul64hi(u, total);
    if (s > 0 && excl <= t && t < excl + s) {
        uint64_t acc = excl;
        for (int i = b0; i < b1; ++i) {
            acc += q40(weight(i));
            if (acc > t) { sh[33] = (uint64_t)i; break; }
        }
    }
    __syncthreads();
    return (int)sh[33];
}

// Argmax over float32 values, lowest index on ties (block-wide).
template <typename F>
ES_DEV int block_argmax(F val, int V, float* shv, int* shi) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = tid; i < V; i += blockDim.x) {
        const float v = val(i);
        if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    __syncthreads();
    if (lane == 0) { shv[wid] = bv; shi[wid] = bi; }
    __syncthreads();
    if (wid == 0) {
        bv = lane < (int)(blockDim.x >> 5) ? shv[lane] : -INFINITY;
        bi = lane < (int)(blockDim.x >> 5) ? shi[lane] : 0x7fffffff;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) shi[0] = bi;
    }
    __syncthreads();
    const int r = shi[0];
    __syncthreads();
    return r;
}

struct RunParams { uint64_t seed; float temperature; int pad_; };

// Row r of this launch: sequence b = r / per_seq, slot i = r % per_seq + off;
// its logits/probs live at ((b * ld_rows) + i) * V.
// Writes probabilities softmax(z/T) (or the logits themselves when T == 0);
// when `dtok` is set, also draws the draft token d[b][i] from them (greedy:
// argmax of the logits) with the phase's slot-i draw.
__global__ void __launch_bounds__(1024)
softmax_sample_kernel(const float* __restrict__ logits, float* __restrict__ probs, int V,
                      int per_seq, int off, int ld_rows, const RunParams* __restrict__ prm,
                      const int64_t* __restrict__ phase, int gamma, int* dtok, int gmax) {
    __shared__ float red[32];
    __shared__ int redi[32];
    __shared__ uint64_t sh[34];
    grid_dep_wait();
    const int r = blockIdx.x, b = r / per_seq, i = r % per_seq + off;
    const size_t base = ((size_t)b * ld_rows + i) * V;
    const float* z = logits + base;
    float* p = probs + base;
    const float T = prm->temperature;
    if (T == 0.f) {
        for (int v = threadIdx.x; v < V; v += blockDim.x) p[v] = z[v];
        if (dtok) {
            const int am = block_argmax([&](int v) { return z[v]; }, V, red, redi);
            if (threadIdx.x == 0) dtok[b * gmax + i] = am;
        }
        return;
    }
    const float invT = 1.0f / T;
    float mx = -INFINITY;
    for (int v = threadIdx.x; v < V; v += blockDim.x) mx = fmaxf(mx, z[v] * invT);
    mx = block_max(mx, red);
    float s = 0.f;
    for (int v = threadIdx.x; v < V; v += blockDim.x) s += expf(z[v] * invT - mx);
    s = block_sum(s, red);
    const float inv = 1.0f / s;
    for (int v = threadIdx.x; v < V; v += blockDim.x) p[v] = expf(z[v] * invT - mx) * inv;
    if (!dtok) return;
    __syncthreads();
    const uint64_t u = es_draw(prm->seed, b, phase[b], i, gamma);
    const int d = block_sample_q40([&](int v) { return p[v]; }, V, u, sh);
    if (threadIdx.x == 0) dtok[b * gmax + i] = d < 0 ? 0 : d;
}

// -------------------------------------------------------------------- accept / resample
// One block per sequence.  p [B][gamma+1][V], q [B][gamma][V] (probabilities,
// or logits when greedy), d [B][gmax].  Draws: u_explicit [B][gamma+1] when
// given, else the phase's slots gamma..2gamma.  Commits tokens when `tokens`
// is set (tokens[b][n_b + t], n_b += n_acc + 1, phase[b] += 1).
struct AcceptArgs {
    const float* p; const float* q; const int* d; int gmax; int gamma, V, greedy;
    const uint64_t* u_explicit; const RunParams* prm; int64_t* phase;
    int* n_acc; int* out_tok;  // out_tok [B][gamma+1]
    int* tokens; int max_seq; int* n_commit;
    const int* n_limit;  // a sequence with n_commit >= n_limit is finished: no commit
};
__global__ void __launch_bounds__(1024) accept_kernel(AcceptArgs a) {
    __shared__ float red[32];
    __shared__ int redi[32];
    __shared__ uint64_t sh[34];
    __shared__ int s_j;
    grid_dep_wait();
    const int b = blockIdx.x, g = a.gamma, V = a.V;
    const float* P = a.p + (size_t)b * (g + 1) * V;
    const float* Q = a.q + (size_t)b * g * V;
    const int* d = a.d + b * a.gmax;
    // greedy < 0: decided by the run's temperature (0 = greedy)
    const int greedy = a.greedy >= 0 ? a.greedy : (a.prm->temperature == 0.f ? 1 : 0);
    uint64_t seed = 0;
    int64_t ph = 0;
    if (!a.u_explicit) { seed = a.prm->seed; ph = a.phase[b]; }
    auto draw = [&](int t) -> uint64_t {  // t = 0..gamma (accept tests, then residual)
        return a.u_explicit ? a.u_explicit[(size_t)b * (g + 1) + t] : es_draw(seed, b, ph, g + t, g);
    };
    int j = g;
    if (greedy) {
        for (int i = 0; i < g; ++i) {
            const float* Pi = P + (size_t)i * V;
            const int am = block_argmax([&](int v) { return Pi[v]; }, V, red, redi);
            if (am != d[i]) { j = i; break; }
        }
    } else if (threadIdx.x == 0) {
        for (int i = 0; i < g; ++i) {
            const int x = d[i];
            if (x < 0 || x >= V) { j = i; break; }  // not a token: rejected
            const float u = uniform24(draw(i));
            if (!(__fmul_rn(u, Q[(size_t)i * V + x]) < P[(size_t)i * V + x])) { j = i; break; }
        }
        s_j = j;
    }
    if (!greedy) { __syncthreads(); j = s_j; }
    const float* Pj = P + (size_t)j * V;
    int y;
    if (greedy) {
        y = block_argmax([&](int v) { return Pj[v]; }, V, red, redi);
    } else {
        const uint64_t u = draw(g);
        if (j < g) {
            const float* Qj = Q + (size_t)j * V;
            y = block_sample_q40([&](int v) { return fmaxf(0.f, __fsub_rn(Pj[v], Qj[v])); }, V, u, sh);
            if (y < 0) y = block_sample_q40([&](int v) { return Pj[v]; }, V, u, sh);
        } else {
            y = block_sample_q40([&](int v) { return Pj[v]; }, V, u, sh);
        }
        if (y < 0) y = 0;
    }
    if (threadIdx.x == 0) {
        a.n_acc[b] = j;
        int* ot = a.out_tok + (size_t)b * (g + 1);
        for (int t = 0; t <= g; ++t) ot[t] = t < j ? d[t] : (t == j ? y : -1);
        if (a.tokens && a.n_commit[b] < a.n_limit[b]) {
            const int n = a.n_commit[b];
            int* tk = a.tokens + (size_t)b * a.max_seq;
            for (int t = 0; t < j && n + t < a.max_seq; ++t) tk[n + t] = d[t];
            if (n + j < a.max_seq) tk[n + j] = y;
            a.n_commit[b] = n + j + 1;
            a.phase[b] += 1;
        }
    }
}

// Sampling hook: row b of unnormalised weights w [B][V] with draw u[b].
__global__ void __launch_bounds__(1024)
sample_rows_kernel(const float* __restrict__ w, const uint64_t* __restrict__ u, int V, int* idx) {
    __shared__ uint64_t sh[34];
    const int b = blockIdx.x;
    const float* wb = w + (size_t)b * V;
    const int r = block_sample_q40([&](int v) { return wb[v]; }, V, u[b], sh);
    if (threadIdx.x == 0) idx[b] = r;
}

}  // namespace es
