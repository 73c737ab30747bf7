// Shared device helpers for libeasyspec (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define ES_DEV __device__ __forceinline__

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- conversions
ES_DEV float to_f32(float v) { return v; }
ES_DEV float to_f32(bf16 v) { return __bfloat162float(v); }
template <typename T> ES_DEV T from_f32(float v);
template <> ES_DEV float from_f32<float>(float v) { return v; }
template <> ES_DEV bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vector of weights -> floats.  Elements per vector: 4 (f32), 8 (bf16).
template <typename T> struct Vec16 { static constexpr int N = 16 / sizeof(T); };

ES_DEV uint4 ld_stream16(const void* p) {
    // weights are read exactly once per pass: bypass L1
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

ES_DEV void unpack16(const uint4& v, float* out, float) {
    out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
}
ES_DEV void unpack16(const uint4& v, float* out, bf16) {
    // bf16 -> f32 is a 16-bit left shift of the bit pattern
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Arrival of a whole CTA at a counter shared by several CTAs: after the
// barrier, one release-acquire atomic by thread 0 publishes every thread's
// earlier writes (the barrier orders them before the release) and, for the
// last arriver, makes the other CTAs' writes visible to it (its threads read
// them after the barrier that follows).  Returns the counter's old value to
// thread 0 (undefined elsewhere).
ES_DEV int cta_arrive(int* ctr) {
    int old = 0;
    if (threadIdx.x == 0)
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(ctr) : "memory");
    return old;
}

// ---------------------------------------------------------------- reductions
ES_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
ES_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block-wide sum/max for blockDim.x a multiple of 32 (<= 1024); `red` holds
// >= 32 floats of shared memory.  All threads receive the result.
ES_DEV float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float t = lane < nw ? red[lane] : 0.f;
    return warp_sum(t);
}
ES_DEV float block_max(float v, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float t = lane < nw ? red[lane] : -INFINITY;
    return warp_max(t);
}

// ---------------------------------------------------------------- PDL
// Programmatic dependent launch: a kernel may start while its predecessor
// drains; everything before grid_dep_wait() must not read the predecessor's
// outputs (weights and other constant inputs are fine).
ES_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
ES_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// ---------------------------------------------------------------- SplitMix64
// G. L. Steele Jr., D. Lea, C. H. Flood, "Fast Splittable Pseudorandom Number
// Generators" (OOPSLA 2014): state advanced by the golden gamma, 64-bit
// finaliser (xor-shift 30, multiply, xor-shift 27, multiply, xor-shift 31).
ES_DEV uint64_t sm64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
// Draw for (row, phase, slot) with 2*gamma+1 slots per phase.
ES_DEV uint64_t es_draw(uint64_t seed, int row, int64_t phase, int slot, int gamma) {
    const uint64_t ctr = ((uint64_t)(uint32_t)row << 32) +
                         (uint64_t)phase * (uint64_t)(2 * gamma + 1) + (uint64_t)slot;
    return sm64(seed ^ sm64(ctr));
}
ES_DEV float uniform24(uint64_t u) { return (float)(u >> 40) * 5.9604644775390625e-8f; }
