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
//              every pending token)
// KIND_FUZZY : rows b, position n_b + step - 1, token d[b][step-1]
// KIND_VERIFY: rows (b, j), j = 0..gamma: position n_b - 1 + j, token
//              x_{n_b-1} for j = 0, d[b][j-1] otherwise
// KIND_HOST  : row arrays already filled by the host
// row_base[m] is the first row of m's sequence block (consecutive rows at
// consecutive positions), which the attention kernel needs.
template <typename T>
__global__ void prep_embed_kernel(int kind, int step, int gamma, int M,
                                  const int* __restrict__ n_commit, const int* __restrict__ tokens,
                                  int max_seq, const int* __restrict__ dtok, int gmax,
                                  int* row_pos, int* row_seq, int* row_tok, int* row_base,
                                  const T* __restrict__ E, float* __restrict__ h, int d, int V,
                                  int* status) {
    grid_dep_wait();
    const int m = blockIdx.x;
    if (m >= M) return;
    int b, pos, tok, base = m;
    if (kind == KIND_HOST) {
        b = row_seq[m]; pos = row_pos[m]; tok = row_tok[m]; base = row_base[m];
    } else if (kind == KIND_CALIB) {
        b = m / (gamma + 1);
        // first active row of the block (rows before it have no position yet)
        base = b * (gamma + 1) + max(0, gamma + 1 - n_commit[b]);
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
        base = b * (gamma + 1);
        const int j = m % (gamma + 1);
        pos = n_commit[b] - 1 + j;
        tok = j > 0 ? dtok[b * gmax + j - 1] : (pos >= 0 && pos < max_seq) ? tokens[(size_t)b * max_seq + pos] : 0;
    }
    if (pos >= max_seq) { if (threadIdx.x == 0) atomicOr(status, STATUS_BAD_POS); pos = -1; }
    if (tok < 0 || tok >= V) { if (threadIdx.x == 0) atomicOr(status, STATUS_BAD_TOKEN); tok = 0; }
    if (threadIdx.x == 0 && kind != KIND_HOST) {
        row_pos[m] = pos; row_seq[m] = b; row_tok[m] = tok; row_base[m] = base;
    }
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
    // greedy decisions consume no draws: the run parameters and phase counter
    // are read only for sampled runs without caller-given draws
    if (!greedy && !a.u_explicit) { seed = a.prm->seed; ph = a.phase[b]; }
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
