// Grouped-query decode attention over the paged KV cache, with the rotary
// embedding and the KV append fused in (sm_103a).
//
// Rows of a launch are tokens at known positions.  The rows of one sequence
// sit in a block of consecutive rows with consecutive positions; row_base[m]
// is the first row of m's block.  Positions before that block's first
// position are read from the cache; positions inside the block come from
// this launch's own raw (un-rotated) k and v rows, rotated here.  So no CTA
// reads a cache entry that this launch writes, and each row's own K/V entry
// is written by the one CTA whose position split holds it (for layer sets,
// these are the "fuzzy" entries of layers that all read the set input).
//
// CTA (row m, layer slot j x kv head, split s) handles positions
// [64 s, min(64 s + 64, pos_m + 1)) for the G = H / Hkv query heads of its kv
// head: scores, softmax and the weighted sum of V.  With several splits each
// CTA stores an unnormalised partial (acc, max, sum) and the last CTA of the
// (m, j, kv head) group -- found with an arrival counter, no waiting --
// merges them in split order and writes the head outputs.
#pragma once
#include "common.cuh"

namespace es {

constexpr int PAGE = 64;          // KV page: 64 positions
constexpr int MAX_GROUP = 8;      // layers per fused set
constexpr int MAX_GQA = 16;       // query heads per kv head
constexpr int ATT_THREADS = 128;
constexpr int ATT_COUNTERS = 16384;

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

struct AttnArgs {
    KVGeom g; const float* rope; int H, M, nl, nsplit;
    int layer[MAX_GROUP];
    const float* q[MAX_GROUP]; const float* k[MAX_GROUP]; const float* v[MAX_GROUP];  // raw rows
    float* out[MAX_GROUP];
    float* part;   // [M][nl][H][nsplit][hd + 2]
    int* counters; // [M][nl][Hkv]
    const int* row_pos; const int* row_seq; const int* row_base;
};

// dynamic shared memory (floats): qs G*(hd+4) | ks 64*(hd+4) | vs 64*(hd+4) | sc G*64
inline size_t attn_smem_bytes(int G, int hd) {
    return sizeof(float) * ((size_t)G * (hd + 4) + 2 * 64 * (hd + 4) + (size_t)G * 64);
}

template <typename T>
__global__ void __launch_bounds__(ATT_THREADS) attn_kernel(AttnArgs a) {
    extern __shared__ __align__(16) float asm_[];
    __shared__ int s_last;
    grid_dep_wait();
    grid_dep_launch();
    const int Hkv = a.g.Hkv, hd = a.g.hd, half = hd / 2, G = a.H / Hkv, ld = hd + 4;
    const int m = blockIdx.x, j = blockIdx.y / Hkv, hk = blockIdx.y % Hkv, sp = blockIdx.z;
    const int pos = a.row_pos[m];
    const int p0 = sp * PAGE;
    if (pos < 0 || p0 > pos) return;
    const int n = min(PAGE, pos + 1 - p0);
    const int rb = a.row_base[m], bpos = a.row_pos[rb], seq = a.row_seq[m];
    const int tid = threadIdx.x, layer = a.layer[j];
    float* qs = asm_;
    float* ks = qs + G * ld;
    float* vs = ks + PAGE * ld;
    float* sc = vs + PAGE * ld;
    const float scale = 1.0f / sqrtf((float)hd);
    const int kvd = Hkv * hd, qd = a.H * hd;

    // rotated, scaled queries of the G heads at this row's position
    {
        const float* q = a.q[j] + (size_t)m * qd + (size_t)hk * G * hd;
        const float* cs = a.rope + (size_t)pos * hd;
        for (int t = tid; t < G * half; t += ATT_THREADS) {
            const int h = t / half, i = t % half;
            const float c = cs[2 * i], s = cs[2 * i + 1];
            const float x0 = q[h * hd + i], x1 = q[h * hd + i + half];
            qs[h * ld + i] = (x0 * c - x1 * s) * scale;
            qs[h * ld + i + half] = (x1 * c + x0 * s) * scale;
        }
    }
    // keys and values of positions p0 .. p0+n-1
    if (p0 + n <= bpos) {
        // all from the cache: contiguous [n][hd] blocks of this page
        const T* Kp = kv_ptr<T>(a.g, seq, p0, layer, 0, hk);
        const T* Vp = kv_ptr<T>(a.g, seq, p0, layer, 1, hk);
        for (int t = tid; t < n * hd; t += ATT_THREADS) {
            const int i = t / hd, e = t % hd;
            ks[i * ld + e] = to_f32(Kp[t]);
            vs[i * ld + e] = to_f32(Vp[t]);
        }
    } else {
        for (int t = tid; t < n * half; t += ATT_THREADS) {
            const int i = t / half, e = t % half, p = p0 + i;
            float k0, k1, v0, v1;
            if (p < bpos) {
                const T* kr = kv_ptr<T>(a.g, seq, p, layer, 0, hk);
                const T* vr = kv_ptr<T>(a.g, seq, p, layer, 1, hk);
                k0 = to_f32(kr[e]); k1 = to_f32(kr[e + half]);
                v0 = to_f32(vr[e]); v1 = to_f32(vr[e + half]);
            } else {
                // this launch's own row for position p: rotate, then round
                // to the cache type exactly as a cached entry would be
                const size_t r = (size_t)(rb + (p - bpos)) * kvd + (size_t)hk * hd;
                const float* cs = a.rope + (size_t)p * hd;
                const float c = cs[2 * e], s = cs[2 * e + 1];
                const float x0 = a.k[j][r + e], x1 = a.k[j][r + e + half];
                k0 = to_f32(from_f32<T>(x0 * c - x1 * s));
                k1 = to_f32(from_f32<T>(x1 * c + x0 * s));
                v0 = to_f32(from_f32<T>(a.v[j][r + e]));
                v1 = to_f32(from_f32<T>(a.v[j][r + e + half]));
            }
            ks[i * ld + e] = k0; ks[i * ld + e + half] = k1;
            vs[i * ld + e] = v0; vs[i * ld + e + half] = v1;
        }
    }
    __syncthreads();
    // append this row's own entry (it lies in this split when p0 <= pos)
    if (pos < p0 + n && pos >= bpos) {
        const int i = pos - p0;
        T* kd = kv_ptr<T>(a.g, seq, pos, layer, 0, hk);
        T* vd = kv_ptr<T>(a.g, seq, pos, layer, 1, hk);
        for (int e = tid; e < hd; e += ATT_THREADS) {
            kd[e] = from_f32<T>(ks[i * ld + e]);
            vd[e] = from_f32<T>(vs[i * ld + e]);
        }
    }
    // scores: thread -> (position i, every other head)
    {
        const int i = tid % PAGE, hp = tid / PAGE;
        if (i < n) {
            const float* kr = ks + i * ld;
            for (int h = hp; h < G; h += 2) {
                const float* qh = qs + h * ld;
                float s = 0.f;
                for (int e = 0; e < hd; e += 4) {
                    const float4 kv4 = *reinterpret_cast<const float4*>(kr + e);
                    const float4 qv4 = *reinterpret_cast<const float4*>(qh + e);
                    s = fmaf(qv4.x, kv4.x, s); s = fmaf(qv4.y, kv4.y, s);
                    s = fmaf(qv4.z, kv4.z, s); s = fmaf(qv4.w, kv4.w, s);
                }
                sc[h * PAGE + i] = s;
            }
        }
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    const int nact = pos / PAGE + 1;   // splits of this row
    float* part_row = a.part + (((size_t)m * a.nl + j) * a.H + (size_t)hk * G) * a.nsplit * (hd + 2);
    for (int h = warp; h < G; h += ATT_THREADS / 32) {
        const float s0 = lane < n ? sc[h * PAGE + lane] : -INFINITY;
        const float s1 = lane + 32 < n ? sc[h * PAGE + lane + 32] : -INFINITY;
        const float mx = warp_max(fmaxf(s0, s1));
        const float e0 = lane < n ? expf(s0 - mx) : 0.f;
        const float e1 = lane + 32 < n ? expf(s1 - mx) : 0.f;
        sc[h * PAGE + lane] = e0;
        sc[h * PAGE + lane + 32] = e1;
        const float l = warp_sum(e0 + e1);
        if (lane == 0 && nact > 1) {
            float* pp = part_row + ((size_t)h * a.nsplit + sp) * (hd + 2);
            pp[hd] = mx;
            pp[hd + 1] = l;
        }
        if (lane == 0) qs[h * ld + hd] = l;      // stash the sum in the row padding
    }
    __syncthreads();
    float* outp = a.out[j] + (size_t)m * qd + (size_t)hk * G * hd;
    for (int t = tid; t < G * hd; t += ATT_THREADS) {
        const int h = t / hd, e = t % hd;
        float acc = 0.f;
        for (int i = 0; i < n; ++i) acc = fmaf(sc[h * PAGE + i], vs[i * ld + e], acc);
        if (nact == 1) outp[t] = acc / qs[h * ld + hd];
        else part_row[((size_t)h * a.nsplit + sp) * (hd + 2) + e] = acc;
    }
    if (nact == 1) return;
    // last arriving split of (m, j, kv head) merges the partials
    __threadfence();
    __syncthreads();
    int* ctr = a.counters + ((size_t)m * a.nl + j) * Hkv + hk;
    if (tid == 0) s_last = atomicAdd(ctr, 1) == nact - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int t = tid; t < G * hd; t += ATT_THREADS) {
        const int h = t / hd, e = t % hd;
        const float* pp = part_row + (size_t)h * a.nsplit * (hd + 2);
        float mx = -INFINITY;
        for (int p = 0; p < nact; ++p) mx = fmaxf(mx, __ldcg(pp + (size_t)p * (hd + 2) + hd));
        float num = 0.f, den = 0.f;
        for (int p = 0; p < nact; ++p) {
            const float* q = pp + (size_t)p * (hd + 2);
            const float w = expf(__ldcg(q + hd) - mx);
            den = fmaf(w, __ldcg(q + hd + 1), den);
            num = fmaf(w, __ldcg(q + e), num);
        }
        outp[t] = num / den;
    }
    if (tid == 0) *ctr = 0;
}

}  // namespace es
