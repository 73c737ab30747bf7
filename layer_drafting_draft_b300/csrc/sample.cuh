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

struct RunParams { uint64_t seed; float temperature; int pad_; };

// Row r of a launch: sequence b = r / per_seq, slot i = r % per_seq + off;
// its logits / probabilities live at row (b * ld_rows + i) of z / p.
struct SampleArgs {
    const float* z; float* p; int V, nb, chunk;
    int per_seq, off, ld_rows;
    const RunParams* prm; const int64_t* phase; int gamma;
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

ES_DEV bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

__global__ void __launch_bounds__(SM_THREADS) softmax_part_kernel(SampleArgs a) {
    __shared__ float rv[SM_THREADS / 32];
    __shared__ int ri[SM_THREADS / 32];
    grid_dep_wait();
    grid_dep_launch();
    const int r = blockIdx.x, c = blockIdx.y, b = r / a.per_seq, i = r % a.per_seq + a.off;
    const float* z = a.z + ((size_t)b * a.ld_rows + i) * a.V;
    const int v0 = c * a.chunk, v1 = min(a.V, v0 + a.chunk);
    const float T = a.prm->temperature;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    float* out = a.part + ((size_t)r * a.nb + c) * 2;
    if (T == 0.f) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int v = v0 + tid; v < v1; v += SM_THREADS)
            if (better(z[v], v, bv, bi)) { bv = z[v]; bi = v; }
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
    for (int v = v0 + tid; v < v1; v += SM_THREADS) mx = fmaxf(mx, z[v] * invT);
    mx = warp_max(mx);
    if (lane == 0) rv[wid] = mx;
    __syncthreads();
    mx = rv[0];
    for (int w = 1; w < SM_THREADS / 32; ++w) mx = fmaxf(mx, rv[w]);
    float s = 0.f;
    for (int v = v0 + tid; v < v1; v += SM_THREADS) s += expf(z[v] * invT - mx);
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

__global__ void __launch_bounds__(SM_THREADS) softmax_finish_kernel(SampleArgs a) {
    __shared__ float s_max, s_inv;
    __shared__ unsigned long long rs[SM_THREADS / 32];
    __shared__ uint64_t sh[34];
    __shared__ int s_last;
    grid_dep_wait();
    grid_dep_launch();
    const int r = blockIdx.x, c = blockIdx.y, b = r / a.per_seq, i = r % a.per_seq + a.off;
    const size_t row = ((size_t)b * a.ld_rows + i) * a.V;
    const float* z = a.z + row;
    float* p = a.p + row;
    const int v0 = c * a.chunk, v1 = min(a.V, v0 + a.chunk);
    const float T = a.prm->temperature;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const float* part = a.part + (size_t)r * a.nb * 2;
    if (T == 0.f) {
        // greedy: the logits themselves are kept; the draw is the argmax
        for (int v = v0 + tid; v < v1; v += SM_THREADS) p[v] = z[v];
        if (a.dtok && c == 0 && tid == 0) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int k = 0; k < a.nb; ++k) {
                const float v = part[2 * k];
                const int vi = __float_as_int(part[2 * k + 1]);
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
        for (int k = lane; k < a.nb; k += 32) mx = fmaxf(mx, part[2 * k]);
        mx = warp_max(mx);
        float s = 0.f;
        for (int k = lane; k < a.nb; k += 32) s += part[2 * k + 1] * expf(part[2 * k] - mx);
        s = warp_sum(s);
        if (lane == 0) { s_max = mx; s_inv = 1.0f / s; }
    }
    __syncthreads();
    const float invT = 1.0f / T, mx = s_max, inv = s_inv;
    unsigned long long ms = 0;
    for (int v = v0 + tid; v < v1; v += SM_THREADS) {
        const float pv = expf(z[v] * invT - mx) * inv;
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
    __shared__ int s_chunk;
    __shared__ unsigned long long s_t;
    if (tid == 0) {
        const unsigned long long* mr = a.mass + (size_t)r * a.nb;
        unsigned long long total = 0;
        for (int k = 0; k < a.nb; ++k) total += __ldcg(mr + k);
        int ck = -1;
        unsigned long long tt = 0;
        if (total > 0) {
            const uint64_t u = es_draw(a.prm->seed, b, a.phase[b], i, a.gamma);
            const unsigned long long t = __umul64hi(u, total);
            unsigned long long pre = 0;
            for (int k = 0; k < a.nb; ++k) {
                const unsigned long long w = __ldcg(mr + k);
                if (t < pre + w) { ck = k; tt = t - pre; break; }
                pre += w;
            }
        }
        s_chunk = ck;
        s_t = tt;
        a.counters[r] = 0;
    }
    __syncthreads();
    const int ck = s_chunk;
    if (ck < 0) {
        if (tid == 0) a.dtok[b * a.gmax + i] = 0;
        return;
    }
    const int c0 = ck * a.chunk, c1 = min(a.V, c0 + a.chunk);
    const int idx = block_find_q40([&](int k) { return __ldcg(p + c0 + k); }, c1 - c0, s_t, sh);
    if (tid == 0) a.dtok[b * a.gmax + i] = c0 + idx;
}

}  // namespace es
