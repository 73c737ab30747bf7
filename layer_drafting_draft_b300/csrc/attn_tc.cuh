// Grouped-query attention for several consecutive rows of one sequence on
// tensor cores (sm_103a, bf16 K/V cache).
//
// The verify forward (gamma+1 rows per sequence), the calibration forward
// and the prompt prefill (a chunk of rows per sequence) all present rows of
// one sequence at consecutive positions.  The one-row kernel (attn.cuh)
// reads every cached K/V page once per row; here one CTA takes a group of
// up to 64 / G rows of one sequence -- all G query heads of one kv head, at
// most 64 query vectors -- against one 64-position page, so a page is read
// once per group.  Scores S = Q K^T and outputs O = P V run as
// mma.sync.m16n8k16 bf16 products with float32 accumulators: K and V are
// the cache's bf16 values (exact), and the float32 operands Q (rotated,
// scaled) and P (softmax weights) enter as hi/lo bf16 pairs, hi = bf16(x),
// lo = bf16(x - hi), both multiplied into the same accumulator (about 16
// significant bits, as in the weight passes).
//
// The rest follows the one-row kernel: positions before the sequence's
// first row in this launch come from the cache, later ones from the
// launch's own raw k/v rows (rotated and rounded to bf16 here), so no CTA
// reads an entry that the launch writes; each row's own entry is written by
// the CTA whose page holds its position; every row sees positions up to its
// own.  A CTA covers a chunk of pages with a running softmax; with several
// chunks, attn_merge_kernel combines the chunks' partials (unnormalised
// output, max, sum) in chunk order.
#pragma once
#include "attn.cuh"
#include "gemv.cuh"

namespace es {

constexpr int ATC_THREADS = 128;   // 4 warps: one 16-vector tile of queries each
constexpr int ATC_QV = 64;         // query vectors per CTA (rows x heads)

// dynamic shared memory (bytes) for head size hd
inline size_t attn_tc_smem_bytes(int hd) {
    const size_t ld = hd + 8;                       // bf16 row stride of Q and K
    return 2 * sizeof(bf16) * ATC_QV * ld           // Q hi, lo
           + sizeof(bf16) * PAGE * ld               // K [position][dim]
           + sizeof(bf16) * hd * (PAGE + 8);        // V transposed [dim][position]
}

ES_DEV void mma16816(float (&d)[4], const uint32_t* a, uint32_t b0, uint32_t b1) {
    mma_bf16_16816(d, a[0], a[1], a[2], a[3], b0, b1);
}

// Grid: (sequences x groups per sequence, layer slots x kv heads, chunks of
// a.ppc pages).  a.rps rows per sequence in this launch, groups of a.rg rows.
// A CTA walks the pages of its chunk with a running (online) softmax; when
// the group's pages span several chunks it stores its unnormalised output,
// max and sum per query vector at the chunk's slot, and attn_merge_kernel
// combines the chunks.
template <int HD>
__global__ void __launch_bounds__(ATC_THREADS) attn_tc_kernel(AttnArgs a) {
    extern __shared__ __align__(16) unsigned char atc_smem[];
    __shared__ int s_pos[ATC_QV];   // position of each query vector's row (-1: none)
    __shared__ int s_rp[ATC_QV];    // positions of the group's rows
    __shared__ int s_meta[3];       // the block's first row, the sequence, the chunk's first page
    constexpr int LD = HD + 8, LDV = PAGE + 8, HALF = HD / 2;
    constexpr int VPR = HD / 8;                    // 16-byte vectors of a K or V row
    constexpr int NV = PAGE * VPR / ATC_THREADS;   // of a page, per thread
    constexpr int QV4 = HALF / 4;                  // items (4 dimensions and their partners) per vector
    constexpr int QB = 4;                          // items per thread whose loads are in flight together
    bf16* qhi = reinterpret_cast<bf16*>(atc_smem);
    bf16* qlo = qhi + ATC_QV * LD;
    bf16* ks = qlo + ATC_QV * LD;
    bf16* vt = ks + PAGE * LD;

    const int Hkv = a.g.Hkv, G = a.H / Hkv, pps = a.g.pages_per_seq;
    const int gps = (a.rps + a.rg - 1) / a.rg;
    const int sq = blockIdx.x / gps, gi = blockIdx.x % gps;
    const int m0 = sq * a.rps + gi * a.rg, nr = min(a.rg, a.rps - gi * a.rg);
    const int j = blockIdx.y / Hkv, hk = blockIdx.y % Hkv, ch = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int layer = a.layer[j];
    const int kvd = Hkv * HD, qd = a.H * HD;
    const int nq = nr * G;                       // query vectors (row-major: r * G + h)
    // The descriptors in one round of independent loads: the rows' positions
    // (-1: inactive row), the block's first row and the sequence.  Rows are
    // laid out sequence by sequence, so the group's sequence is the launch's
    // sq-th and the chunk's first page can be looked up at the same time
    // (again below if row_seq says otherwise).
    if (tid < nr) s_rp[tid] = __ldcg(a.row_pos + m0 + tid);
    if (tid == ATC_THREADS - 1) s_meta[0] = __ldcg(a.row_base + m0);
    if (tid == ATC_THREADS - 2) s_meta[1] = __ldcg(a.row_seq + m0);
    if (tid == ATC_THREADS - 3)
        s_meta[2] = ch * a.ppc < pps ? __ldcg(a.g.page_table + (size_t)sq * pps + ch * a.ppc) : -1;
    __syncthreads();
    int maxpos = -1, ra = -1;
    for (int r = 0; r < nr; ++r) {
        const int p = s_rp[r];
        maxpos = max(maxpos, p);
        if (ra < 0 && p >= 0) ra = r;
    }
    const int npg = maxpos / PAGE + 1;           // pages of the group
    const int pg0 = ch * a.ppc, pg1 = min(npg, pg0 + a.ppc);
    if (maxpos < 0 || pg0 >= npg) return;
    const int nch = (npg + a.ppc - 1) / a.ppc;   // chunks of the group
    const int rb = s_meta[0], seq = s_meta[1];
    // the rows of a block hold consecutive positions from its first row on
    const int bpos = s_rp[ra] - (m0 + ra - rb);
    int page = seq == sq ? s_meta[2] : a.g.page_table[(size_t)seq * pps + pg0];
    if (tid < ATC_QV) s_pos[tid] = tid < nq ? s_rp[tid / G] : -1;

    // K and V of (page, this layer, this kv head)
    auto page_kv = [&](int pid, int kv) {
        return reinterpret_cast<bf16*>(a.g.kv) + ((((size_t)pid * a.g.L + layer) * 2 + kv) * Hkv + hk) * PAGE * HD;
    };
    // cached part of a page (written by earlier launches): 16-byte loads
    // into registers, then K row-major and V transposed into shared memory
    uint4 kk[NV], vv[NV];
    auto issue_cached = [&](int pid, int ncached) {
        const uint4* Kp = reinterpret_cast<const uint4*>(page_kv(pid, 0));
        const uint4* Vp = reinterpret_cast<const uint4*>(page_kv(pid, 1));
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int t = u * ATC_THREADS + tid;
            if (t < ncached * VPR) {
                kk[u] = __ldcg(Kp + t);
                vv[u] = __ldcg(Vp + t);
            }
        }
    };
    auto store_cached = [&](int ncached) {
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int t = u * ATC_THREADS + tid;
            if (t < ncached * VPR) {
                const int i = t / VPR, e = (t % VPR) * 8;
                *reinterpret_cast<uint4*>(ks + i * LD + e) = kk[u];
                const bf16* vb = reinterpret_cast<const bf16*>(&vv[u]);
#pragma unroll
                for (int x = 0; x < 8; ++x) vt[(e + x) * LDV + i] = vb[x];
            }
        }
    };
    // the first page's cached part is requested before waiting for the
    // preceding kernel
    {
        const int p0 = pg0 * PAGE, n = min(PAGE, maxpos + 1 - p0);
        issue_cached(page, max(0, min(n, bpos - p0)));
    }
    grid_dep_wait();
    grid_dep_launch();
    // queries: rotated to their row's position, scaled, split hi/lo
    const float scale = 1.0f / sqrtf((float)HD);
#pragma unroll 1
    for (int t0 = 0; t0 < ATC_QV * QV4; t0 += QB * ATC_THREADS) {
        float4 x0[QB], x1[QB], cA[QB], cB[QB];
#pragma unroll
        for (int u = 0; u < QB; ++u) {
            const int t = t0 + u * ATC_THREADS + tid, v = t / QV4, e = (t % QV4) * 4;
            const int pos = v < nq ? s_rp[v / G] : -1;
            x0[u] = x1[u] = cA[u] = cB[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (pos >= 0) {
                const float* q = a.q[j] + (size_t)(m0 + v / G) * qd + (size_t)(hk * G + v % G) * HD;
                const float* cs = a.rope + (size_t)pos * HD;
                x0[u] = __ldcg(reinterpret_cast<const float4*>(q + e));
                x1[u] = __ldcg(reinterpret_cast<const float4*>(q + e + HALF));
                cA[u] = __ldg(reinterpret_cast<const float4*>(cs + 2 * e));
                cB[u] = __ldg(reinterpret_cast<const float4*>(cs + 2 * e + 4));
            }
        }
        if (t0 == 0) {   // the cached page has arrived meanwhile
            const int p0 = pg0 * PAGE, n = min(PAGE, maxpos + 1 - p0);
            store_cached(max(0, min(n, bpos - p0)));
        }
#pragma unroll
        for (int u = 0; u < QB; ++u) {
            const int t = t0 + u * ATC_THREADS + tid, v = t / QV4, e = (t % QV4) * 4;
            const float xa[4] = {x0[u].x, x0[u].y, x0[u].z, x0[u].w};
            const float xb[4] = {x1[u].x, x1[u].y, x1[u].z, x1[u].w};
            const float c[4] = {cA[u].x, cA[u].z, cB[u].x, cB[u].z};
            const float sn[4] = {cA[u].y, cA[u].w, cB[u].y, cB[u].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float y0 = (xa[k] * c[k] - xb[k] * sn[k]) * scale;
                const float y1 = (xb[k] * c[k] + xa[k] * sn[k]) * scale;
                const bf16 h0 = __float2bfloat16_rn(y0), h1 = __float2bfloat16_rn(y1);
                qhi[v * LD + e + k] = h0;
                qhi[v * LD + e + k + HALF] = h1;
                qlo[v * LD + e + k] = __float2bfloat16_rn(y0 - __bfloat162float(h0));
                qlo[v * LD + e + k + HALF] = __float2bfloat16_rn(y1 - __bfloat162float(h1));
            }
        }
    }

    const int g = lane >> 2, cq = lane & 3;
    const int v0 = warp * 16;
    const bool active = v0 < nq;
    float o[HD / 8][4];
#pragma unroll
    for (int t = 0; t < HD / 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
    for (int pg = pg0; pg < pg1; ++pg) {
        const int p0 = pg * PAGE, n = min(PAGE, maxpos + 1 - p0);
        const int ncached = max(0, min(n, bpos - p0));
        if (pg > pg0) {
            __syncthreads();   // every warp is done with the previous page
            page = a.g.page_table[(size_t)seq * pps + pg];
            // later pages of a multi-page chunk: copied without the register
            // staging, which would compete with the running output here
            const uint4* Kp = reinterpret_cast<const uint4*>(page_kv(page, 0));
            const uint4* Vp = reinterpret_cast<const uint4*>(page_kv(page, 1));
            for (int t = tid; t < ncached * VPR; t += ATC_THREADS) {
                const int i = t / VPR, e = (t % VPR) * 8;
                const uint4 kv = __ldcg(Kp + t), vv1 = __ldcg(Vp + t);
                *reinterpret_cast<uint4*>(ks + i * LD + e) = kv;
                const bf16* vb = reinterpret_cast<const bf16*>(&vv1);
#pragma unroll
                for (int x = 0; x < 8; ++x) vt[(e + x) * LDV + i] = vb[x];
            }
        }
        // the launch's own positions (>= bpos): rotate and round the raw rows
#pragma unroll 1
        for (int t0 = 0; t0 < (n - ncached) * QV4; t0 += 2 * ATC_THREADS) {
            float4 k0[2], k1[2], w0[2], w1[2], cA[2], cB[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = t0 + u * ATC_THREADS + tid, i = ncached + t / QV4, e = (t % QV4) * 4, p = p0 + i;
                if (t < (n - ncached) * QV4) {
                    const size_t r = (size_t)(rb + (p - bpos)) * kvd + (size_t)hk * HD + e;
                    const float* cs = a.rope + (size_t)p * HD + 2 * e;
                    k0[u] = __ldcg(reinterpret_cast<const float4*>(a.k[j] + r));
                    k1[u] = __ldcg(reinterpret_cast<const float4*>(a.k[j] + r + HALF));
                    w0[u] = __ldcg(reinterpret_cast<const float4*>(a.v[j] + r));
                    w1[u] = __ldcg(reinterpret_cast<const float4*>(a.v[j] + r + HALF));
                    cA[u] = __ldg(reinterpret_cast<const float4*>(cs));
                    cB[u] = __ldg(reinterpret_cast<const float4*>(cs + 4));
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = t0 + u * ATC_THREADS + tid, i = ncached + t / QV4, e = (t % QV4) * 4;
                if (t >= (n - ncached) * QV4) continue;
                const float xa[4] = {k0[u].x, k0[u].y, k0[u].z, k0[u].w};
                const float xb[4] = {k1[u].x, k1[u].y, k1[u].z, k1[u].w};
                const float va[4] = {w0[u].x, w0[u].y, w0[u].z, w0[u].w};
                const float vb[4] = {w1[u].x, w1[u].y, w1[u].z, w1[u].w};
                const float c[4] = {cA[u].x, cA[u].z, cB[u].x, cB[u].z};
                const float sn[4] = {cA[u].y, cA[u].w, cB[u].y, cB[u].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    ks[i * LD + e + k] = __float2bfloat16_rn(xa[k] * c[k] - xb[k] * sn[k]);
                    ks[i * LD + e + k + HALF] = __float2bfloat16_rn(xb[k] * c[k] + xa[k] * sn[k]);
                    vt[(e + k) * LDV + i] = __float2bfloat16_rn(va[k]);
                    vt[(e + k + HALF) * LDV + i] = __float2bfloat16_rn(vb[k]);
                }
            }
        }
        // zero the tail of the page so the k16 steps read finite values
        for (int t = tid; t < (PAGE - n) * HD; t += ATC_THREADS) {
            const int i = n + t / HD, e = t % HD;
            ks[i * LD + e] = __float2bfloat16_rn(0.f);
            vt[e * LDV + i] = __float2bfloat16_rn(0.f);
        }
        __syncthreads();
        // each row's own entry, when this page holds its position (16 bytes
        // of K and of V per item)
        for (int t = tid; t < nr * VPR; t += ATC_THREADS) {
            const int r = t / VPR, e = (t % VPR) * 8, pos = s_rp[r];
            if (pos < bpos || pos < p0 || pos >= p0 + n) continue;
            const int i = pos - p0;
            *reinterpret_cast<uint4*>(page_kv(page, 0) + (size_t)i * HD + e) =
                *reinterpret_cast<const uint4*>(ks + i * LD + e);
            uint32_t w[4];
#pragma unroll
            for (int x = 0; x < 4; ++x)
                w[x] = (uint32_t)__bfloat16_as_ushort(vt[(e + 2 * x) * LDV + i]) |
                       ((uint32_t)__bfloat16_as_ushort(vt[(e + 2 * x + 1) * LDV + i]) << 16);
            *reinterpret_cast<uint4*>(page_kv(page, 1) + (size_t)i * HD + e) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (!active) continue;
        // S = Q K^T for this page (one 16-vector tile per warp)
        float s[PAGE / 8][4];
#pragma unroll
        for (int t = 0; t < PAGE / 8; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
        for (int k0 = 0; k0 < HD; k0 += 16) {
            uint32_t ah[4], al[4];
            const bf16* qa = qhi + (v0 + g) * LD + k0 + 2 * cq;
            const bf16* qb = qlo + (v0 + g) * LD + k0 + 2 * cq;
            ah[0] = *reinterpret_cast<const uint32_t*>(qa);
            ah[1] = *reinterpret_cast<const uint32_t*>(qa + 8 * LD);
            ah[2] = *reinterpret_cast<const uint32_t*>(qa + 8);
            ah[3] = *reinterpret_cast<const uint32_t*>(qa + 8 * LD + 8);
            al[0] = *reinterpret_cast<const uint32_t*>(qb);
            al[1] = *reinterpret_cast<const uint32_t*>(qb + 8 * LD);
            al[2] = *reinterpret_cast<const uint32_t*>(qb + 8);
            al[3] = *reinterpret_cast<const uint32_t*>(qb + 8 * LD + 8);
#pragma unroll
            for (int t = 0; t < PAGE / 8; ++t) {
                const bf16* kb = ks + (t * 8 + g) * LD + k0 + 2 * cq;
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(kb);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(kb + 8);
                mma16816(s[t], ah, b0, b1);
                mma16816(s[t], al, b0, b1);
            }
        }
        // causal mask and the page's valid positions; running max and sum
        const int pa = s_pos[v0 + g], pb = s_pos[v0 + g + 8];
        float mpg[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int t = 0; t < PAGE / 8; ++t)
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const int i = t * 8 + 2 * cq + x, p = p0 + i;
                if (i >= n || p > pa) s[t][x] = -INFINITY;
                if (i >= n || p > pb) s[t][2 + x] = -INFINITY;
                mpg[0] = fmaxf(mpg[0], s[t][x]);
                mpg[1] = fmaxf(mpg[1], s[t][2 + x]);
            }
        float mnew[2], keep[2], lpg[2] = {0.f, 0.f};
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            mpg[x] = fmaxf(mpg[x], __shfl_xor_sync(0xffffffffu, mpg[x], 1));
            mpg[x] = fmaxf(mpg[x], __shfl_xor_sync(0xffffffffu, mpg[x], 2));
            mnew[x] = fmaxf(mrun[x], mpg[x]);
            keep[x] = mrun[x] == -INFINITY ? 0.f : expf(mrun[x] - mnew[x]);
        }
#pragma unroll
        for (int t = 0; t < PAGE / 8; ++t)
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float mx = mnew[x >> 1];
                const float e = mx == -INFINITY ? 0.f : expf(s[t][x] - mx);
                s[t][x] = e;
                lpg[x >> 1] += e;
            }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            lpg[x] += __shfl_xor_sync(0xffffffffu, lpg[x], 1);
            lpg[x] += __shfl_xor_sync(0xffffffffu, lpg[x], 2);
            lrun[x] = lrun[x] * keep[x] + lpg[x];
            mrun[x] = mnew[x];
        }
#pragma unroll
        for (int t = 0; t < HD / 8; ++t) {
            o[t][0] *= keep[0]; o[t][1] *= keep[0];
            o[t][2] *= keep[1]; o[t][3] *= keep[1];
        }
        // O += P V: two score tiles (16 positions) form one A operand
#pragma unroll
        for (int kt = 0; kt < PAGE / 16; ++kt) {
            uint32_t ph[4], pl[4];
            split2(s[2 * kt][0], s[2 * kt][1], ph[0], pl[0]);
            split2(s[2 * kt][2], s[2 * kt][3], ph[1], pl[1]);
            split2(s[2 * kt + 1][0], s[2 * kt + 1][1], ph[2], pl[2]);
            split2(s[2 * kt + 1][2], s[2 * kt + 1][3], ph[3], pl[3]);
#pragma unroll
            for (int t = 0; t < HD / 8; ++t) {
                const bf16* vb = vt + (t * 8 + g) * LDV + kt * 16 + 2 * cq;
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(vb);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(vb + 8);
                mma16816(o[t], ph, b0, b1);
                mma16816(o[t], pl, b0, b1);
            }
        }
    }
    // ---- results: rows of vectors v0+g and v0+g+8
    if (!active) return;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int v = v0 + g + 8 * x;
        if (v >= nq || s_pos[v] < 0) continue;
        const int r = v / G, h = v % G;
        if (nch == 1) {
            float* out = a.out[j] + (size_t)(m0 + r) * qd + (size_t)(hk * G + h) * HD;
            const float inv = 1.0f / lrun[x];
#pragma unroll
            for (int t = 0; t < HD / 8; ++t) {
                out[t * 8 + 2 * cq] = o[t][2 * x] * inv;
                out[t * 8 + 2 * cq + 1] = o[t][2 * x + 1] * inv;
            }
        } else {
            float* pp = a.part + ((((size_t)(m0 + r) * a.nl + j) * a.H + (size_t)hk * G + h) * a.nsplit + ch) *
                                     (HD + 2);
#pragma unroll
            for (int t = 0; t < HD / 8; ++t) {
                pp[t * 8 + 2 * cq] = o[t][2 * x];
                pp[t * 8 + 2 * cq + 1] = o[t][2 * x + 1];
            }
            if (cq == 0) {
                pp[HD] = mrun[x];
                pp[HD + 1] = lrun[x];
            }
        }
    }
}

// Combines the chunks of attn_tc_kernel when a group's pages span several:
// one CTA of HD threads per (group, layer slot x kv head, query vector);
// out = sum_c w_c o_c / sum_c w_c l_c with w_c = exp(m_c - max_c m_c), in
// chunk order.  Groups that fit one chunk were finished by attn_tc_kernel.
template <int HD>
__global__ void __launch_bounds__(HD) attn_merge_kernel(AttnArgs a) {
    __shared__ float s_m[256], s_l[256];   // the chunks' max and sum (at most 256 chunks)
    const int Hkv = a.g.Hkv, G = a.H / Hkv;
    const int gps = (a.rps + a.rg - 1) / a.rg;
    const int sq = blockIdx.x / gps, gi = blockIdx.x % gps;
    const int m0 = sq * a.rps + gi * a.rg, nr = min(a.rg, a.rps - gi * a.rg);
    const int j = blockIdx.y / Hkv, hk = blockIdx.y % Hkv, v = blockIdx.z;
    grid_dep_wait();
    grid_dep_launch();
    if (v >= nr * G) return;
    // the group's row positions, loaded together (nr <= 64 <= HD)
    __shared__ int s_rp[ATC_QV];
    if (threadIdx.x < nr) s_rp[threadIdx.x] = __ldcg(a.row_pos + m0 + threadIdx.x);
    __syncthreads();
    int maxpos = -1;
    for (int r = 0; r < nr; ++r) maxpos = max(maxpos, s_rp[r]);
    const int nch = maxpos < 0 ? 0 : (maxpos / PAGE + 1 + a.ppc - 1) / a.ppc;
    const int r = v / G, h = v % G, pos = s_rp[r];
    if (nch <= 1 || pos < 0) return;
    const int na = (pos / PAGE + 1 + a.ppc - 1) / a.ppc;   // chunks this row sees
    const float* pp = a.part + (((size_t)(m0 + r) * a.nl + j) * a.H + (size_t)hk * G + h) * a.nsplit * (HD + 2);
    const int tid = threadIdx.x;
    // every chunk's max and sum, and this thread's output element of the
    // first NB chunks, in one round of loads
    constexpr int NB = 16;
    for (int c = tid; c < na; c += HD) {
        s_m[c] = __ldcg(pp + (size_t)c * (HD + 2) + HD);
        s_l[c] = __ldcg(pp + (size_t)c * (HD + 2) + HD + 1);
    }
    float oc[NB];
#pragma unroll
    for (int c = 0; c < NB; ++c) oc[c] = c < na ? __ldcg(pp + (size_t)c * (HD + 2) + tid) : 0.f;
    __syncthreads();
    float mx = -INFINITY;
    for (int c = 0; c < na; ++c) mx = fmaxf(mx, s_m[c]);
    // weights w_c = exp(m_c - max), summed with the outputs in chunk order
    float den = 0.f, num = 0.f;
#pragma unroll
    for (int c = 0; c < NB; ++c) {
        if (c >= na) break;
        const float wc = s_m[c] == -INFINITY ? 0.f : expf(s_m[c] - mx);
        den = fmaf(wc, s_l[c], den);
        num = fmaf(wc, oc[c], num);
    }
    for (int c = NB; c < na; ++c) {
        const float wc = s_m[c] == -INFINITY ? 0.f : expf(s_m[c] - mx);
        den = fmaf(wc, s_l[c], den);
        num = fmaf(wc, __ldcg(pp + (size_t)c * (HD + 2) + tid), num);
    }
    a.out[j][(size_t)(m0 + r) * (a.H * HD) + (size_t)(hk * G + h) * HD + tid] = num / den;
}

}  // namespace es
