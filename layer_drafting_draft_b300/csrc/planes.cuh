// Activation planes for the tensor-core weight pass (sm_103a): the hi/lo
// bf16 split of float32 activation rows (split_planes_kernel), and the
// normalised planes of a decode-size pass's input (norm_planes_kernel), which
// the pass then loads by TMA.
#pragma once
#include "common.cuh"
#include "tcgemm.cuh"

namespace es {

// Activation planes: for source i, rows r*row_stride + row_off of src
// (leading dimension ld, K columns) become hi/lo bf16 planes
// dst[0][r][k], dst[1][r][k] ([2][M][K]).
struct SplitArgs {
    const float* src[TC_MAX_SRCS];
    bf16* dst[TC_MAX_SRCS];
    int ld[TC_MAX_SRCS], rs[TC_MAX_SRCS], ro[TC_MAX_SRCS], K[TC_MAX_SRCS];
    int item0[TC_MAX_SRCS + 1];  // prefix of M*K/4 items per source
    int nsrc, M;
};

__global__ void split_planes_kernel(SplitArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    const int total = a.item0[a.nsrc];
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
        int i = 0;
        while (t >= a.item0[i + 1]) ++i;
        const int K4 = a.K[i] >> 2, u = t - a.item0[i];
        const int m = u / K4, k = (u - m * K4) * 4;
        const float4 v = __ldcg(reinterpret_cast<const float4*>(
            a.src[i] + (size_t)(m * a.rs[i] + a.ro[i]) * a.ld[i] + k));
        const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
        const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
        const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
        const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
        const size_t plane = (size_t)a.M * a.K[i];
        __nv_bfloat162* ph = reinterpret_cast<__nv_bfloat162*>(a.dst[i] + (size_t)m * a.K[i] + k);
        __nv_bfloat162* pl = reinterpret_cast<__nv_bfloat162*>(a.dst[i] + plane + (size_t)m * a.K[i] + k);
        ph[0] = h0; ph[1] = h1; pl[0] = l0; pl[1] = l1;
    }
}

// Normalised activation planes for a tensor-core pass that follows a
// decode-size weight pass: row r reads h[src] (src = r*stride + off; if `add`
// is set, h[src] += add[src] first, written back), takes
// rinv = 1 / sqrt(mean(h^2) + eps) and writes the hi/lo planes of
// h * rinv * gain to dst[0][r][.], dst[1][r][.] ([2][M][d]), the values the
// RMSNorm kernel would store in float32.  Grid (rows, column chunks of
// NPL_COLS): the mean comes from the producing pass's per-tile sums of
// squares (ss_tiles partials of the source row at ssp[t * ss_ld + src],
// added by one warp lane-strided and then in a fixed shuffle order, so every
// chunk of a row gets the same value), or, without them, from the row
// itself.
constexpr int NPL_COLS = 1024;
struct NormPlanesArgs {
    float* h; const float* add; const bf16* g; bf16* dst;
    const float* ssp; int ss_tiles, ss_ld;
    int d, M, src_stride, src_off;
    float eps;
};
__global__ void norm_planes_kernel(NormPlanesArgs a) {
    __shared__ float red[32];
    __shared__ float s_rinv;
    static_assert(NPL_COLS == 4 * 256, "four columns per thread of a 256-thread CTA");
    const int r = blockIdx.x, tid = threadIdx.x;
    const size_t src = (size_t)r * a.src_stride + a.src_off;
    float* hr = a.h + src * a.d;
    // this thread's four columns (the row width is a multiple of 4)
    const int i = blockIdx.y * NPL_COLS + 4 * tid;
    const bool mine = i < a.d;
    uint2 gb = make_uint2(0u, 0u);
    if (mine) gb = *reinterpret_cast<const uint2*>(a.g + i);  // gains: weights, before the wait
    grid_dep_wait();
    // the columns and the norm's partial sums are requested together
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f), av = v;
    if (mine) {
        v = __ldcg(reinterpret_cast<const float4*>(hr + i));
        if (a.add) av = __ldcg(reinterpret_cast<const float4*>(a.add + src * a.d + i));
    }
    if (a.ssp) {
        if (tid < 32) {
            // lane-strided partials, 8 loads per lane in flight, added in index order
            float t = 0.f;
            for (int i0 = tid; i0 < a.ss_tiles; i0 += 256) {
                float pr[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int k = i0 + 32 * u;
                    pr[u] = k < a.ss_tiles ? __ldcg(a.ssp + (size_t)k * a.ss_ld + src) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (i0 + 32 * u < a.ss_tiles) t += pr[u];
            }
            t = warp_sum(t);
            if (tid == 0) s_rinv = 1.0f / sqrtf(t / (float)a.d + a.eps);
        }
        __syncthreads();
    } else {
        // the whole row (the planner sends no addend here: other CTAs write
        // h + add back while this one reads)
        float ss = 0.f;
        for (int k = tid; k < a.d; k += blockDim.x) {
            float x = hr[k];
            if (a.add) x += a.add[src * a.d + k];
            ss += x * x;
        }
        ss = block_sum(ss, red);
        if (tid == 0) s_rinv = 1.0f / sqrtf(ss / (float)a.d + a.eps);
        __syncthreads();
    }
    grid_dep_launch();
    if (!mine) return;
    const float rinv = s_rinv;
    if (a.add) {
        v.x += av.x; v.y += av.y; v.z += av.z; v.w += av.w;
        *reinterpret_cast<float4*>(hr + i) = v;
    }
    const float vx[4] = {v.x, v.y, v.z, v.w};
    const float gx[4] = {__uint_as_float(gb.x << 16), __uint_as_float(gb.x & 0xffff0000u),
                         __uint_as_float(gb.y << 16), __uint_as_float(gb.y & 0xffff0000u)};
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float x0 = vx[2 * k] * rinv * gx[2 * k], x1 = vx[2 * k + 1] * rinv * gx[2 * k + 1];
        const bf16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
        const bf16 l0 = __float2bfloat16_rn(x0 - __bfloat162float(h0));
        const bf16 l1 = __float2bfloat16_rn(x1 - __bfloat162float(h1));
        hw[k] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        lw[k] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    bf16* hi = a.dst + (size_t)r * a.d + i;
    *reinterpret_cast<uint2*>(hi) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(hi + (size_t)a.M * a.d) = make_uint2(lw[0], lw[1]);
}

}  // namespace es
