// Vocabulary softmax and token draws spread over many CTAs (sm_103a).
//
// A row of V logits is cut into nb chunks, one CTA each.
//   softmax_part_kernel   per chunk: max of z/T and sum of exp(z/T - max)
//                         (greedy, T = 0: max and its lowest index)
//   softmax_finish_kernel per chunk: the row's max and normaliser from the
//                         nb partials (added in chunk order), the chunk's
//                         probabilities p = exp(z/T - max) / sum, and -- when
//                         a token is drawn -- the chunk's integer mass
//                         sum floor(p * 2^40).  The last CTA of the row to
//                         finish (arrival counter) turns the draw u into the
//                         target t = floor(u * total / 2^64), finds the chunk
//                         whose prefix holds t and scans it for the index.
// Integer masses make the drawn index independent of the order of summation:
// the same rule as the single-block sampler used by the accept kernel.
#pragma once
#include "common.cuh"

namespace es {

constexpr int SM_THREADS = 256;
constexpr int SM_COUNTERS = 4096;

// calib_off: 1 = calibration ablation (the next exact draft forward covers
// only the positions that hold no draft entry, see the row setup)
struct RunParams { uint64_t seed; float temperature; int calib_off; };

// Row r of a launch: sequence b = r / per_seq, slot i = r % per_seq + off;
// its logits / probabilities live at row (b * ld_rows + i) of z / p.
struct SampleArgs {
    const float* z; float* p; int V, nb, chunk;
    int per_seq, off, ld_rows;
    const RunParams* prm; const int64_t* phase; int gamma;
    int greedy;                // 1 / 0, or -1: greedy when prm->temperature == 0
    int* dtok; int gmax;       // draw d[b][i] when set
    float* part;               // [rows][nb][2]
    unsigned long long* mass;  // [rows][nb]
    int* counters;             // [rows]
};

ES_DEV uint64_t q40(float w) { return (uint64_t)(w * 1099511627776.0f); }

ES_DEV uint64_t warp_incl_scan_u64(uint64_t v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Smallest i in [0, n) whose inclusive prefix of q40(weight(i)) exceeds t
// (t < the total, so one exists).  Whole block; sh >= 34 entries.
template <typename F>
ES_DEV int block_find_q40(F weight, int n, uint64_t t, uint64_t* sh) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nt = blockDim.x;
    const int per = (n + nt - 1) / nt;
    const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
    uint64_t s = 0;
    for (int i = b0; i < b1; ++i) s += q40(weight(i));
    const uint64_t incl = warp_incl_scan_u64(s, lane);
    __syncthreads();
    if (lane == 31) sh[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const uint64_t w = lane < (nt >> 5) ? sh[lane] : 0;
        const uint64_t wi = warp_incl_scan_u64(w, lane);
        sh[lane] = wi - w;
    }
    __syncthreads();
    const uint64_t excl = sh[wid] + incl - s;
    __syncthreads();
    if (tid == 0) sh[33] = (uint64_t)(n - 1);
    __syncthreads();
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

// Block-wide inclusive prefix sum of one u64 per thread (blockDim.x a
// multiple of 32, <= 1024); sh >= 33 entries.  Also returns the total.
ES_DEV uint64_t block_incl_scan_u64(uint64_t v, uint64_t* sh, uint64_t* total) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
    const uint64_t incl = warp_incl_scan_u64(v, lane);
    __syncthreads();
    if (lane == 31) sh[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const uint64_t w = lane < nw ? sh[lane] : 0;
        const uint64_t wi = warp_incl_scan_u64(w, lane);
        sh[lane] = wi - w;
        if (lane == 31) sh[32] = wi;
    }
    __syncthreads();
    const uint64_t r = sh[wid] + incl;
    *total = sh[32];
    __syncthreads();
    return r;
}

// The chunk of a categorical draw from per-chunk integer masses (nb <=
// blockDim.x, read with __ldcg at stride `stride`): t = floor(u * total /
// 2^64), the chunk whose prefix range holds t and t relative to its start.
// Returns the total (0: no chunk).  Whole block.
ES_DEV uint64_t block_locate_chunk(const unsigned long long* mass, int stride, int nb, uint64_t u,
                                   int* chunk, uint64_t* t_rel, uint64_t* sh) {
    __shared__ int s_ck;
    __shared__ uint64_t s_tr;
    const int tid = threadIdx.x;
    const uint64_t w = tid < nb ? (uint64_t)__ldcg(mass + (size_t)tid * stride) : 0;
    uint64_t total;
    const uint64_t incl = block_incl_scan_u64(w, sh, &total);
    if (tid == 0) { s_ck = -1; s_tr = 0; }
    __syncthreads();
    if (total > 0) {
        const uint64_t t = __umul64hi(u, total);
        if (w > 0 && incl - w <= t && t < incl) { s_ck = tid; s_tr = t - (incl - w); }
    }
    __syncthreads();
    *chunk = s_ck;
    *t_rel = s_tr;
    __syncthreads();
    return total;
}

ES_DEV bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// Item (row r, chunk c) of the partial softmax.  Whole CTA.
ES_DEV void softmax_part_item(const SampleArgs& a, int r, int c) {
    __shared__ float rv[SM_THREADS / 32];
    __shared__ int ri[SM_THREADS / 32];
    __syncthreads();  // shared memory of the previous item
    const int b = r / a.per_seq, i = r % a.per_seq + a.off;
    const float* z = a.z + ((size_t)b * a.ld_rows + i) * a.V;
    const int v0 = c * a.chunk, v1 = min(a.V, v0 + a.chunk);
    const float T = a.greedy > 0 ? 0.f : a.prm->temperature;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    float* out = a.part + ((size_t)r * a.nb + c) * 2;
    if (a.greedy > 0 || (a.greedy < 0 && T == 0.f)) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int v = v0 + tid; v < v1; v += SM_THREADS)
            { const float zv = __ldcg(z + v); if (better(zv, v, bv, bi)) { bv = zv; bi = v; } }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { rv[wid] = bv; ri[wid] = bi; }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < SM_THREADS / 32; ++w)
                if (better(rv[w], ri[w], bv, bi)) { bv = rv[w]; bi = ri[w]; }
            out[0] = bv;
            out[1] = __int_as_float(bi);
        }
        return;
    }
    const float invT = 1.0f / T;
    float mx = -INFINITY;
    for (int v = v0 + tid; v < v1; v += SM_THREADS) mx = fmaxf(mx, __ldcg(z + v) * invT);
    mx = warp_max(mx);
    if (lane == 0) rv[wid] = mx;
    __syncthreads();
    mx = rv[0];
    for (int w = 1; w < SM_THREADS / 32; ++w) mx = fmaxf(mx, rv[w]);
    float s = 0.f;
    for (int v = v0 + tid; v < v1; v += SM_THREADS) s += expf(__ldcg(z + v) * invT - mx);
    s = warp_sum(s);
    __syncthreads();
    if (lane == 0) rv[wid] = s;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < SM_THREADS / 32; ++w) t += rv[w];
        out[0] = mx;
        out[1] = t;
    }
}

// Item (row r, chunk c) of the softmax completion and draw.  Whole CTA.
ES_DEV void softmax_finish_item(const SampleArgs& a, int r, int c) {
    __shared__ float s_max, s_inv;
    __shared__ unsigned long long rs[SM_THREADS / 32];
    __shared__ uint64_t sh[34];
    __shared__ int s_last;
    __syncthreads();  // shared memory of the previous item
    const int b = r / a.per_seq, i = r % a.per_seq + a.off;
    const size_t row = ((size_t)b * a.ld_rows + i) * a.V;
    const float* z = a.z + row;
    float* p = a.p + row;
    const int v0 = c * a.chunk, v1 = min(a.V, v0 + a.chunk);
    const float T = a.greedy > 0 ? 0.f : a.prm->temperature;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float* part = a.part + (size_t)r * a.nb * 2;
    if (a.greedy > 0 || (a.greedy < 0 && T == 0.f)) {
        // greedy: the logits themselves are kept; the draw is the argmax
        for (int v = v0 + tid; v < v1; v += SM_THREADS) p[v] = __ldcg(z + v);
        if (a.dtok && c == 0 && tid == 0) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int k = 0; k < a.nb; ++k) {
                const float v = __ldcg(part + 2 * k);
                const int vi = __float_as_int(__ldcg(part + 2 * k + 1));
                if (better(v, vi, bv, bi)) { bv = v; bi = vi; }
            }
            a.dtok[b * a.gmax + i] = bi;
        }
        return;
    }
    if (wid == 0) {
        // the row's max and normaliser: fixed lane assignment and shuffle
        // tree, so every chunk CTA (and every run) gets the same values
        float mx = -INFINITY;
        for (int k = lane; k < a.nb; k += 32) mx = fmaxf(mx, __ldcg(part + 2 * k));
        mx = warp_max(mx);
        float s = 0.f;
        for (int k = lane; k < a.nb; k += 32) s += __ldcg(part + 2 * k + 1) * expf(__ldcg(part + 2 * k) - mx);
        s = warp_sum(s);
        if (lane == 0) { s_max = mx; s_inv = 1.0f / s; }
    }
    __syncthreads();
    const float invT = 1.0f / T, mx = s_max, inv = s_inv;
    unsigned long long ms = 0;
    for (int v = v0 + tid; v < v1; v += SM_THREADS) {
        const float pv = expf(__ldcg(z + v) * invT - mx) * inv;
        p[v] = pv;
        ms += q40(pv);
    }
    if (!a.dtok) return;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ms += __shfl_xor_sync(0xffffffffu, ms, o);
    if (lane == 0) rs[wid] = ms;
    __threadfence();  // this CTA's probabilities before its arrival below
    __syncthreads();
    if (tid == 0) {
        unsigned long long t = 0;
        for (int w = 0; w < SM_THREADS / 32; ++w) t += rs[w];
        a.mass[(size_t)r * a.nb + c] = t;
        __threadfence();
        s_last = atomicAdd(a.counters + r, 1) == a.nb - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // last chunk CTA of the row: locate the draw
    if (tid == 0) a.counters[r] = 0;
    const uint64_t u = es_draw(a.prm->seed, b, __ldcg(a.phase + b), i, a.gamma);
    int ck;
    uint64_t t_rel;
    block_locate_chunk(a.mass + (size_t)r * a.nb, 1, a.nb, u, &ck, &t_rel, sh);
    if (ck < 0) {
        if (tid == 0) a.dtok[b * a.gmax + i] = 0;
        return;
    }
    const int c0 = ck * a.chunk, c1 = min(a.V, c0 + a.chunk);
    const int idx = block_find_q40([&](int k) { return __ldcg(p + c0 + k); }, c1 - c0, t_rel, sh);
    if (tid == 0) a.dtok[b * a.gmax + i] = c0 + idx;
}

// ------------------------------------------------------------ accept / resample
// Grid (B, nb), one CTA per vocabulary chunk of each sequence.  p [B][g+1][V]
// and q [B][g][V] are probabilities (greedy: logits), d [B][gmax] the draft
// tokens.  Every CTA finds the first rejected slot j (sampled: the accept
// test fl(u * q_i(d_i)) < p_i(d_i) with the draw of slot g+i; greedy:
// d_i == argmax p_i, from the per-chunk argmax partials `gpart` of the g+1
// p rows).  Sampled runs then draw y from max(0, p_j - q_j) (j < g; from p_j
// when that has no integer mass) or from p_g (every draft accepted): each
// CTA adds the integer masses of its chunk, the last one locates the draw.
// The deciding CTA writes n_acc and the tokens and, when `tokens` is set,
// commits them (n_commit += j + 1 unless the sequence reached n_limit;
// phase += 1; kv_from = n + min(j, g - 1), the first committed position
// with no draft K/V entry once the accepted drafts keep theirs).
struct AcceptArgs {
    const float* p; const float* q; const int* d; int gmax, gamma, V, nb, chunk;
    int greedy;                    // 1 / 0, or -1: greedy when prm->temperature == 0
    const uint64_t* u_explicit;    // [B][g+1] draws, or null: the phase's slots g..2g
    const RunParams* prm; int64_t* phase;
    const float* gpart;            // [B*(g+1)][nb][2] (greedy)
    unsigned long long* mass;      // [B][nb][2]
    int* counters;                 // [B]
    int* n_acc; int* out_tok;      // [B], [B][g+1] (-1 past n_acc+1)
    int* tokens; int max_seq; int* n_commit; const int* n_limit;
    int* kv_from;                  // [B] or null
};

// Item (sequence b, chunk c) of accept/resample.  Whole CTA.
ES_DEV void accept_item(const AcceptArgs& a, int b, int c) {
    __shared__ int s_j, s_y, s_last;
    __shared__ int s_am[17];
    __shared__ uint64_t sh[34];
    __shared__ unsigned long long rs[2][SM_THREADS / 32];
    __syncthreads();  // shared memory of the previous item
    const int g = a.gamma, V = a.V;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int greedy = a.greedy >= 0 ? a.greedy : (a.prm->temperature == 0.f ? 1 : 0);
    const float* P = a.p + (size_t)b * (g + 1) * V;
    const float* Q = a.q + (size_t)b * g * V;
    const int* d = a.d + b * a.gmax;
    if (greedy) {
        if (c != 0) return;
        // argmax of each p row from the chunk partials (warp per row)
        for (int i = wid; i <= g; i += SM_THREADS / 32) {
            const float* gp = a.gpart + ((size_t)b * (g + 1) + i) * a.nb * 2;
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int k = lane; k < a.nb; k += 32) {
                const float v = __ldcg(gp + 2 * k);
                const int vi = __float_as_int(__ldcg(gp + 2 * k + 1));
                if (better(v, vi, bv, bi)) { bv = v; bi = vi; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            if (lane == 0) s_am[i] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            int j = g;
            for (int i = 0; i < g; ++i)
                if (s_am[i] != __ldcg(d + i)) { j = i; break; }
            s_j = j;
            s_y = s_am[j];
        }
    } else {
        uint64_t seed = 0;
        int64_t ph = 0;
        if (!a.u_explicit) { seed = a.prm->seed; ph = __ldcg(a.phase + b); }
        auto draw = [&](int t) -> uint64_t {  // t = 0..g (accept tests, then the residual)
            return a.u_explicit ? a.u_explicit[(size_t)b * (g + 1) + t] : es_draw(seed, b, ph, g + t, g);
        };
        if (tid == 0) {
            int j = g;
            for (int i = 0; i < g; ++i) {
                const int x = __ldcg(d + i);
                if (x < 0 || x >= V) { j = i; break; }  // not a token: rejected
                const float u = uniform24(draw(i));
                if (!(__fmul_rn(u, __ldcg(Q + (size_t)i * V + x)) < __ldcg(P + (size_t)i * V + x))) { j = i; break; }
            }
            s_j = j;
        }
        __syncthreads();
        const int j = s_j;
        const float* Pj = P + (size_t)j * V;
        const float* Qj = Q + (size_t)j * V;
        const int v0 = c * a.chunk, v1 = min(V, v0 + a.chunk);
        unsigned long long mr = 0, mp = 0;
        for (int v = v0 + tid; v < v1; v += SM_THREADS) {
            const float pv = __ldcg(Pj + v);
            mp += q40(pv);
            mr += j < g ? q40(fmaxf(0.f, __fsub_rn(pv, __ldcg(Qj + v)))) : q40(pv);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mr += __shfl_xor_sync(0xffffffffu, mr, o);
            mp += __shfl_xor_sync(0xffffffffu, mp, o);
        }
        if (lane == 0) { rs[0][wid] = mr; rs[1][wid] = mp; }
        __syncthreads();
        if (tid == 0) {
            unsigned long long t0 = 0, t1 = 0;
            for (int w = 0; w < SM_THREADS / 32; ++w) { t0 += rs[0][w]; t1 += rs[1][w]; }
            unsigned long long* ms = a.mass + ((size_t)b * a.nb + c) * 2;
            ms[0] = t0;
            ms[1] = t1;
            __threadfence();
            s_last = atomicAdd(a.counters + b, 1) == a.nb - 1;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        if (tid == 0) a.counters[b] = 0;
        const uint64_t u = draw(g);
        int ck;
        uint64_t t_rel;
        // the residual; with no integer mass left, the base distribution p_j
        int use_p = 0;
        if (block_locate_chunk(a.mass + (size_t)b * a.nb * 2, 2, a.nb, u, &ck, &t_rel, sh) == 0) {
            use_p = 1;
            block_locate_chunk(a.mass + (size_t)b * a.nb * 2 + 1, 2, a.nb, u, &ck, &t_rel, sh);
        }
        int y = 0;
        if (ck >= 0) {
            const int c0 = ck * a.chunk, c1 = min(V, c0 + a.chunk);
            const bool resid = j < g && !use_p;
            y = c0 + block_find_q40(
                         [&](int k) {
                             const float pv = __ldcg(Pj + c0 + k);
                             return resid ? fmaxf(0.f, __fsub_rn(pv, __ldcg(Qj + c0 + k))) : pv;
                         },
                         c1 - c0, t_rel, sh);
        }
        if (tid == 0) s_y = y;
    }
    __syncthreads();
    if (tid == 0) {
        const int j = s_j, y = s_y;
        a.n_acc[b] = j;
        int* ot = a.out_tok + (size_t)b * (g + 1);
        for (int t = 0; t <= g; ++t) ot[t] = t < j ? __ldcg(d + t) : (t == j ? y : -1);
        if (a.tokens && __ldcg(a.n_commit + b) < __ldcg(a.n_limit + b)) {
            const int n = __ldcg(a.n_commit + b);
            int* tk = a.tokens + (size_t)b * a.max_seq;
            for (int t = 0; t < j && n + t < a.max_seq; ++t) tk[n + t] = __ldcg(d + t);
            if (n + j < a.max_seq) tk[n + j] = y;
            a.n_commit[b] = n + j + 1;
            a.phase[b] = __ldcg(a.phase + b) + 1;
            // d_1..d_{g-1} were draft inputs at positions n..n+g-2
            if (a.kv_from) a.kv_from[b] = n + min(j, g - 1);
        }
    }
}

__global__ void __launch_bounds__(SM_THREADS) softmax_part_kernel(SampleArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    softmax_part_item(a, blockIdx.x, blockIdx.y);
}
__global__ void __launch_bounds__(SM_THREADS) softmax_finish_kernel(SampleArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    softmax_finish_item(a, blockIdx.x, blockIdx.y);
}
__global__ void __launch_bounds__(SM_THREADS) accept_kernel(AcceptArgs a) {
    grid_dep_wait();
    accept_item(a, blockIdx.x, blockIdx.y);
}

}  // namespace es
