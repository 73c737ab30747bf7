// Kernels of the speculative-decoding hot path (sm_103a).
//
// Activations and accumulation are float32; weights and KV cache are T
// (float or bf16).  Rows of a forward pass are described by device arrays
// row_pos / row_seq / row_tok, so the same launches (and CUDA graphs) serve
// every phase; a row with row_pos < 0 is inactive (no KV write, no output).
#pragma once
#include "common.cuh"
#include "gemv.cuh"
#include "attn.cuh"
#include "sample.cuh"

namespace es {

constexpr int STATUS_BAD_POS = 1; // device status bits
constexpr int STATUS_BAD_TOKEN = 2;

enum { KIND_HOST = 0, KIND_CALIB = 1, KIND_FUZZY = 2, KIND_VERIFY = 3 };

// -------------------------------------------------------------------- rows
// KIND_CALIB : rows (b, i), i = 0..gamma: position n_b - gamma - 1 + i (the
//              last gamma+1 committed tokens; recomputing already-exact
//              positions reproduces their entries, so the window always covers
//              every pending token).  Under the calibration ablation
//              (prm->calib_off) rows before kv_from[b] are inactive: the
//              accepted drafts keep their layer-parallel entries and only the
//              positions without one are computed.
// KIND_FUZZY : rows b, position n_b + step - 1, token d[b][step-1]
// KIND_VERIFY: rows (b, j), j = 0..gamma: position n_b - 1 + j, token
//              x_{n_b-1} for j = 0, d[b][j-1] otherwise
// KIND_HOST  : row arrays already filled by the host
// row_base[m] is the first row of m's sequence block (consecutive rows at
// consecutive positions), which the attention kernel needs.
struct EmbedArgs {
    int kind, step, gamma, M;
    const int* n_commit; const int* tokens; int max_seq; const int* dtok; int gmax;
    int* row_pos; int* row_seq; int* row_tok; int* row_base;
    const int* kv_from; const RunParams* prm;  // calibration ablation (KIND_CALIB)
    const void* E; float* h; int d, V;
    int* status;
    GvPost post;  // 1/rms of the embedded rows (rows map one to one)
};

// Row m: describe it (sequence, position, token) and gather its embedding.
// Whole CTA.  Device state written by earlier work is read through L2.
template <typename T>
ES_DEV void embed_item(const EmbedArgs& a, int m) {
    __shared__ float red[32];
    __syncthreads();  // shared memory of the previous item
    int b, pos, tok, base = m;
    const int kind = a.kind, gamma = a.gamma, max_seq = a.max_seq;
    if (kind == KIND_HOST) {
        b = __ldcg(a.row_seq + m); pos = __ldcg(a.row_pos + m); tok = __ldcg(a.row_tok + m);
        base = __ldcg(a.row_base + m);
    } else if (kind == KIND_CALIB) {
        b = m / (gamma + 1);
        const int nb = __ldcg(a.n_commit + b);
        // first position the window computes: 0, or kv_from[b] without
        // calibration (never past the last committed token)
        int lo = 0;
        if (a.kv_from && a.prm->calib_off) lo = min(max(__ldcg(a.kv_from + b), 0), nb - 1);
        // first active row of the block (rows before it have no position
        // yet, or keep their entries)
        base = b * (gamma + 1) + max(gamma + 1 - nb, lo - (nb - gamma - 1));
        base = max(base, b * (gamma + 1));
        const int i = m % (gamma + 1);
        pos = nb - (gamma + 1) + i;
        if (pos < lo) pos = -1;
        tok = (pos >= 0 && pos < max_seq) ? __ldcg(a.tokens + (size_t)b * max_seq + pos) : 0;
    } else if (kind == KIND_FUZZY) {
        b = m;
        pos = __ldcg(a.n_commit + b) + a.step - 1;
        tok = __ldcg(a.dtok + b * a.gmax + a.step - 1);
    } else {
        b = m / (gamma + 1);
        base = b * (gamma + 1);
        const int j = m % (gamma + 1);
        pos = __ldcg(a.n_commit + b) - 1 + j;
        tok = j > 0 ? __ldcg(a.dtok + b * a.gmax + j - 1)
                    : (pos >= 0 && pos < max_seq) ? __ldcg(a.tokens + (size_t)b * max_seq + pos) : 0;
    }
    if (pos >= max_seq) { if (threadIdx.x == 0) atomicOr(a.status, STATUS_BAD_POS); pos = -1; }
    if (tok < 0 || tok >= a.V) { if (threadIdx.x == 0) atomicOr(a.status, STATUS_BAD_TOKEN); tok = 0; }
    if (threadIdx.x == 0 && kind != KIND_HOST) {
        a.row_pos[m] = pos; a.row_seq[m] = b; a.row_tok[m] = tok; a.row_base[m] = base;
    }
    const int d = a.d;
    const T* e = (const T*)a.E + (size_t)tok * d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        const float v = to_f32(e[i]);
        a.h[(size_t)m * d + i] = v;
        ss += v * v;
    }
    // 1/rms of the embedded rows for the first weight pass
    if (a.post.rows > 0) {
        ss = block_sum(ss, red);
        if (threadIdx.x == 0) {
            if (a.post.ssp) a.post.ssp[m] = ss;  // one partial per row
            else a.post.rinv[m] = 1.0f / sqrtf(ss / (float)d + a.post.eps);
        }
    }
}

template <typename T>
__global__ void prep_embed_kernel(EmbedArgs a) {
    grid_dep_wait();
    if (blockIdx.x < a.M) embed_item<T>(a, blockIdx.x);
}

// ------------------------------------------------------- many-row helpers
// Row m of a source (row m*rs + ro of src, leading dimension ld) split into
// bf16 hi/lo planes [M][K]: hi = bf16(x), lo = bf16(x - hi), so a bf16
// tensor-core GEMM of each plane, summed, keeps ~16 significant bits of x.
__global__ void split_hilo_kernel(const float* __restrict__ src, int ld, int rs, int ro, int M, int K,
                                  bf16* __restrict__ hi, bf16* __restrict__ lo) {
    grid_dep_wait();
    grid_dep_launch();
    const int K4 = K >> 2;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < M * K4; t += gridDim.x * blockDim.x) {
        const int m = t / K4, k = (t - m * K4) * 4;
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + (size_t)(m * rs + ro) * ld + k));
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
        const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
        const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
        const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
        __nv_bfloat162* ph = reinterpret_cast<__nv_bfloat162*>(hi + (size_t)m * K + k);
        __nv_bfloat162* pl = reinterpret_cast<__nv_bfloat162*>(lo + (size_t)m * K + k);
        ph[0] = h0; ph[1] = h1; pl[0] = l0; pl[1] = l1;
    }
}

// Epilogues of a many-row weight pass after its GEMMs: y += add
// (residual + delta) or y = silu(g) * u (SwiGLU); y [M][ldy], g/u [M][N].
// Epilogue of a many-row pass over output columns [0, Nc) of y (already
// offset to the chunk): the GEMM of the stacked planes [hi; lo] left the hi
// products in rows 0..M-1 of s and the lo products in rows M..2M-1 ([2M][Nc]),
// so row m of the result is s[m] + s[M + m] (s1 likewise for the up
// projection of a SwiGLU op).
__global__ void epi_hilo_kernel(float* __restrict__ y, int ldy, const float* __restrict__ add, int epi,
                                const float* __restrict__ s0, const float* __restrict__ s1, int M, int Nc) {
    grid_dep_wait();
    grid_dep_launch();
    const size_t half = (size_t)M * Nc;
    for (size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x; t < half; t += (size_t)gridDim.x * blockDim.x) {
        const int m = (int)(t / Nc), n = (int)(t - (size_t)m * Nc);
        float* yp = y + (size_t)m * ldy + n;
        const float a = s0[t] + s0[half + t];
        switch (epi) {
            case GEPI_SWIGLU: {
                const float b = s1[t] + s1[half + t];
                *yp = a / (1.0f + expf(-a)) * b;
                break;
            }
            case GEPI_STORE: *yp = a; break;
            case GEPI_ACC: *yp = *yp + a; break;
            default: *yp = *yp + a + add[(size_t)m * ldy + n]; break;
        }
    }
}

// -------------------------------------------------------------------- RMSNorm
// out_j[r] = RMSNorm(h[src], g_j) for every job j, with src = r*stride + off.
// If `add` is set, h[src] += add[src] first (written back).
struct NormArgs {
    float* h; const float* add; int d; float eps; int src_stride, src_off;
    int njobs; const void* g[2 * MAX_GROUP]; float* out[2 * MAX_GROUP]; int out_ld;
    // job j with planes[j] set writes bf16 hi/lo planes [2][planes_M][d] of
    // its rows there (the input of a tensor-core pass) instead of out[j]
    bf16* planes[2 * MAX_GROUP]; int planes_M;
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
        if (a.planes[j]) {
            bf16* hi = a.planes[j] + (size_t)r * a.d;
            bf16* lo = hi + (size_t)a.planes_M * a.d;
            for (int i = threadIdx.x; i < a.d; i += blockDim.x) {
                const float x = hr[i] * rinv * to_f32(g[i]);
                const bf16 hb = __float2bfloat16_rn(x);
                hi[i] = hb;
                lo[i] = __float2bfloat16_rn(x - __bfloat162float(hb));
            }
            continue;
        }
        float* o = a.out[j] + (size_t)r * a.out_ld;
        for (int i = threadIdx.x; i < a.d; i += blockDim.x) o[i] = hr[i] * rinv * to_f32(g[i]);
    }
}

// -------------------------------------------------------------------- sampling
// Integer-quantised inverse CDF: W_i = floor(w_i * 2^40) (w_i >= 0 float32),
// T = sum W_i, t = floor(u * T / 2^64); result = first i whose inclusive
// prefix sum exceeds t.  Integer sums make the result independent of the
// summation order.  Returns -1 if T == 0.  Whole block participates;
// blockDim.x == 1024.
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
