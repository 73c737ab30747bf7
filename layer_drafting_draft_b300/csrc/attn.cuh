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
constexpr int ATT_THREADS = 256;
constexpr int ATT_COUNTERS = 16384;

// Paged cache: element (page p, layer l, K|V, kv head h, slot s, e) at
// ((((p*L + l)*2 + kv)*Hkv + h)*PAGE + s)*hd + e.
struct KVGeom {
    void* kv; const int* page_table; int pages_per_seq, L, Hkv, hd, max_seq;
};

struct AttnArgs {
    KVGeom g; const float* rope; int H, M, nl, nsplit;
    int layer[MAX_GROUP];
    const float* q[MAX_GROUP]; const float* k[MAX_GROUP]; const float* v[MAX_GROUP];  // raw rows
    float* out[MAX_GROUP];
    float* part;   // [M][nl][H][nsplit][hd + 2]
    int* counters; // [M][nl][Hkv]
    const int* row_pos; const int* row_seq; const int* row_base;
    int rps, rg, ppc;   // rows per sequence (0: no fixed layout); grouped-row kernel: rows per CTA group, pages per CTA
};

// dynamic shared memory (floats): qs G*(hd+4) | ks 64*(hd+4) | vs 64*(hd+4) |
// sc G*max(64, nsplit) (scores, then the split-merge weights)
inline size_t attn_smem_bytes(int G, int hd, int nsplit) {
    return sizeof(float) * ((size_t)G * (hd + 4) + 2 * 64 * (hd + 4) + (size_t)G * (nsplit > 64 ? nsplit : 64));
}


// One work item: row m, layer slot x kv head `jy`, position split `sp`.
// Whole CTA (ATT_THREADS threads).
template <typename T>
ES_DEV void attn_item(const AttnArgs& a, int m, int jy, int sp) {
    extern __shared__ __align__(16) float asm_[];
    __shared__ int s_last;
    const int Hkv = a.g.Hkv, hd = a.g.hd, half = hd / 2, G = a.H / Hkv, ld = hd + 4;
    const int j = jy / Hkv, hk = jy % Hkv, pps = a.g.pages_per_seq;
    // The row's descriptors in one round of loads.  With rps rows per
    // sequence laid out sequence by sequence the row's sequence is m / rps,
    // which gives the split's page at the same time (looked up again below if
    // row_seq says otherwise).
    const int guess = a.rps > 0 ? m / a.rps : -1;
    const int pos = __ldcg(a.row_pos + m), rb = __ldcg(a.row_base + m), seq = __ldcg(a.row_seq + m);
    const int pg_guess = guess >= 0 && sp < pps ? __ldcg(a.g.page_table + (size_t)guess * pps + sp) : -1;
    const int p0 = sp * PAGE;
    if (pos < 0 || p0 > pos) return;
    const int n = min(PAGE, pos + 1 - p0);
    // the rows of a block hold consecutive positions from its first row on
    const int bpos = pos - (m - rb);
    const int page = seq == guess ? pg_guess : a.g.page_table[(size_t)seq * pps + sp];
    const int tid = threadIdx.x, layer = a.layer[j];
    float* qs = asm_;
    float* ks = qs + G * ld;
    float* vs = ks + PAGE * ld;
    float* sc = vs + PAGE * ld;
    const float scale = 1.0f / sqrtf((float)hd);
    const int kvd = Hkv * hd, qd = a.H * hd;

    // positions of this split already in the cache (all but the launch's own)
    const int ncached = max(0, min(n, bpos - p0));
    // Issue the independent global loads together: the cached part of the
    // split's K/V page (16-byte vectors), the queries and their rotation
    // factors.
    constexpr int EPV = 16 / sizeof(T);
    constexpr int VPT = 8;  // vectors of K (and of V) per thread and pass
    const int nv = ncached * hd / EPV;
    const size_t kvoff = ((((size_t)page * a.g.L + layer) * 2) * Hkv + hk) * PAGE * hd;
    const T* Kp = (const T*)a.g.kv + kvoff;
    const T* Vp = Kp + (size_t)Hkv * PAGE * hd;
    const float* q = a.q[j] + (size_t)m * qd + (size_t)hk * G * hd;
    const float* csq = a.rope + (size_t)pos * hd;
    // A cached page was written by earlier launches, and the row
    // descriptors by the embedding kernel, which finished before the weight
    // pass that launched this kernel: the first pass of page loads is
    // issued before waiting for that weight pass (the queries are not).
    uint4 kv4[VPT], vv4[VPT];
    auto load_pass = [&](int base) {
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int t = base + u * ATT_THREADS + tid;
            if (t < nv) {
                kv4[u] = __ldcg(reinterpret_cast<const uint4*>(Kp + (size_t)t * EPV));
                vv4[u] = __ldcg(reinterpret_cast<const uint4*>(Vp + (size_t)t * EPV));
            }
        }
    };
    if (nv > 0) load_pass(0);
    grid_dep_wait();
    grid_dep_launch();
    for (int base = 0; base < nv || base == 0; base += VPT * ATT_THREADS) {
        if (base > 0) load_pass(base);
        if (base == 0) {
            for (int t = tid; t < G * half; t += ATT_THREADS) {
                const int h = t / half, i = t % half;
                const float c = csq[2 * i], sn = csq[2 * i + 1];
                const float x0 = __ldcg(q + h * hd + i), x1 = __ldcg(q + h * hd + i + half);
                qs[h * ld + i] = (x0 * c - x1 * sn) * scale;
                qs[h * ld + i + half] = (x1 * c + x0 * sn) * scale;
            }
        }
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int t = base + u * ATT_THREADS + tid;
            if (t < nv) {
                float kf[EPV], vf[EPV];
                unpack16(kv4[u], kf, T());
                unpack16(vv4[u], vf, T());
                const int i = t * EPV / hd, e = t * EPV % hd;
#pragma unroll
                for (int x = 0; x < EPV; ++x) { ks[i * ld + e + x] = kf[x]; vs[i * ld + e + x] = vf[x]; }
            }
        }
    }
    // the launch's own positions (from bpos on): its raw k/v rows, rotated
    // and rounded to the cache type as a cached entry would be
    for (int t = tid; t < (n - ncached) * half; t += ATT_THREADS) {
        const int i = ncached + t / half, e = t % half, p = p0 + i;
        const size_t r = (size_t)(rb + (p - bpos)) * kvd + (size_t)hk * hd;
        const float* cs = a.rope + (size_t)p * hd;
        const float c = cs[2 * e], sn = cs[2 * e + 1];
        const float x0 = __ldcg(a.k[j] + r + e), x1 = __ldcg(a.k[j] + r + e + half);
        ks[i * ld + e] = to_f32(from_f32<T>(x0 * c - x1 * sn));
        ks[i * ld + e + half] = to_f32(from_f32<T>(x1 * c + x0 * sn));
        vs[i * ld + e] = to_f32(from_f32<T>(__ldcg(a.v[j] + r + e)));
        vs[i * ld + e + half] = to_f32(from_f32<T>(__ldcg(a.v[j] + r + e + half)));
    }
    __syncthreads();
    // append this row's own entry (it lies in this split when p0 <= pos)
    if (pos < p0 + n && pos >= bpos) {
        const int i = pos - p0;
        T* kd = (T*)a.g.kv + kvoff + (size_t)i * hd;
        T* vd = kd + (size_t)Hkv * PAGE * hd;
        for (int e = tid; e < hd; e += ATT_THREADS) {
            kd[e] = from_f32<T>(ks[i * ld + e]);
            vd[e] = from_f32<T>(vs[i * ld + e]);
        }
    }
    // scores: thread -> (position i, every fourth head)
    {
        const int i = tid % PAGE, hp = tid / PAGE;
        if (i < n) {
            const float* kr = ks + i * ld;
            for (int h = hp; h < G; h += ATT_THREADS / PAGE) {
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
    // last arriving split of (m, j, kv head) merges the partials (one
    // acquire-release arrival per CTA after the barrier)
    __syncthreads();
    int* ctr = a.counters + ((size_t)m * a.nl + j) * Hkv + hk;
    const int old = cta_arrive(ctr);
    if (tid == 0) s_last = old == nact - 1;
    __syncthreads();
    if (!s_last) return;
    // merge weights w[h][p] = exp(m_p - max) / sum_p' exp(m_p' - max) l_p'
    // (reusing the score buffer: nact <= nsplit splits per head)
    float* wsm = sc;
    for (int t = tid; t < G * nact; t += ATT_THREADS) {
        const int h = t / nact, p = t % nact;
        wsm[h * a.nsplit + p] = __ldcg(part_row + ((size_t)h * a.nsplit + p) * (hd + 2) + hd);
    }
    __syncthreads();
    for (int h = warp; h < G; h += ATT_THREADS / 32) {
        float mx = -INFINITY;
        for (int p = lane; p < nact; p += 32) mx = fmaxf(mx, wsm[h * a.nsplit + p]);
        mx = warp_max(mx);
        float den = 0.f;
        for (int p = lane; p < nact; p += 32) {
            const float w = expf(wsm[h * a.nsplit + p] - mx);
            wsm[h * a.nsplit + p] = w;
            den = fmaf(w, __ldcg(part_row + ((size_t)h * a.nsplit + p) * (hd + 2) + hd + 1), den);
        }
        den = warp_sum(den);
        const float inv = 1.0f / den;
        for (int p = lane; p < nact; p += 32) wsm[h * a.nsplit + p] *= inv;
    }
    __syncthreads();
    for (int t = tid; t < G * hd; t += ATT_THREADS) {
        const int h = t / hd, e = t % hd;
        const float* pp = part_row + (size_t)h * a.nsplit * (hd + 2) + e;
        const float* wh = wsm + h * a.nsplit;
        float num = 0.f;
#pragma unroll 4
        for (int p = 0; p < nact; ++p) num = fmaf(wh[p], __ldcg(pp + (size_t)p * (hd + 2)), num);
        outp[t] = num;
    }
    if (tid == 0) *ctr = 0;
}

// One CTA per work item; attn_item waits for the preceding kernel itself
// (after requesting the cached K/V page).
template <typename T>
__global__ void __launch_bounds__(ATT_THREADS) attn_kernel(AttnArgs a) {
    attn_item<T>(a, blockIdx.x, blockIdx.y, blockIdx.z);
}

}  // namespace es
