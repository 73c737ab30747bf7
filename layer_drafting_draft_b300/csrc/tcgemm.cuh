// Many-row weight passes on the fifth-generation tensor cores (sm_103a):
// tcgen05.mma with operands staged in shared memory by TMA and the
// accumulator in tensor memory.
//
// A pass with more than 8 activation rows (prompt prefill, the verify of
// gamma+1 rows per sequence for a batch, calibration of a batch) computes,
// for every op o of the launch and every output feature n < N_o and
// activation row r < M,
//   acc_set[n][r] = sum over the op's segments s of set `set`:
//                   W_s[n, :] . x_s[r, :]
// and applies the op's epilogue (STORE, ACC, ACC_ADD, SWIGLU as in the
// decode weight pass).  Activations arrive as bf16 planes hi = bf16(x),
// lo = bf16(x - hi) of the float32 rows (written by split_planes_kernel);
// both planes are multiplied into the same float32 accumulator, so the
// products keep ~16 significant bits of x with bf16 weights.
//
// Swapped operands: the weights are the MMA's A operand (M = 128 weight rows
// per tile) and the activation rows its B operand (N = the rows, padded to a
// multiple of 16, at most 256 per row chunk).  The accumulator D[n][r] sits
// in tensor memory with lane = weight row and column = activation row, so
// the epilogue thread of lane n writes y[r][n] for consecutive n across a
// warp: coalesced rows of the row-major output.
//
// CTA roles (256 threads): thread 0 issues the TMA loads (weights before
// griddepcontrol.wait -- they do not depend on the previous kernel --
// activations after), thread 32 issues the MMAs and commits each stage back
// to its "empty" barrier, and afterwards all 8 warps read the accumulator
// (warp w: lanes 32*(w%4).., column half w/4) and run the epilogue.
//
// Work split.  A unit is (op, 128-row weight tile, row chunk, k-range).  When
// the tiles alone cannot fill the SMs, every tile's 64-column k-blocks are
// cut into `cs` equal ranges, and the cs CTAs of one tile form a thread-block
// cluster.  After the main loop each CTA copies its accumulator to its own
// shared memory; after a cluster barrier, CTA s of the cluster adds the cs
// partials of its share of the tile's columns, reading them from the other
// CTAs' shared memory (distributed shared memory), in rank order -- the
// result does not depend on timing -- and applies the epilogue.  A second
// cluster barrier keeps every CTA's partial alive until all have been read.
// Cluster CTAs are scheduled together, so the barriers need no spin loop.
//
// Every wait on an mbarrier is bounded (TC_WAIT_NS of the global timer).  A
// wait that runs out sets bit 0 of `err`, the CTA stops issuing work, waits
// (bounded again) for the copies it still has in flight, frees its tensor
// memory and returns; the host reports ES_ERR_TIMEOUT.
#pragma once
#include <cooperative_groups.h>

#include "common.cuh"
#include "gemv.cuh"

namespace es {

constexpr int TC_BM = 128;            // weight rows per tile (MMA M)
constexpr int TC_BK = 64;             // k per stage: one 128-byte swizzle row of bf16
constexpr int TC_MAXN = 256;          // activation rows per chunk (MMA N)
constexpr int TC_THREADS = 256;
constexpr int TC_MAX_OPS = 32;
constexpr int TC_MAX_SEGS = 64;
constexpr int TC_MAX_SRCS = 16;
constexpr int TC_MAX_CLUSTER = 8;     // k-ranges per tile (portable cluster size)
constexpr unsigned long long TC_WAIT_NS = 2000000000ull;  // 2 s

// A CUtensorMap (128 bytes, 64-byte aligned), filled on the host.
struct alignas(64) TcMap { unsigned long long w[16]; };

struct TcSeg {
    int wmap;      // tensor map of the weights W_s [N, K] (box 64 x 128)
    int src;       // activation source (its planes' tensor map)
    int K, nkb;    // columns, 64-column k-blocks
    int kb0;       // first k-block of this segment within its op
    int pad_[3];
};
struct TcOp {
    float* y; const float* add;
    bf16* yp;                  // STORE / SWIGLU results as hi/lo planes [2][M][N] (the
                               // next tensor-core pass's input) instead of y, when set
    int N, ldy, epi, pair;     // pair: SwiGLU, segment seg0 = gate, seg0+1 = up
    int seg0, nseg, nkb;       // k-blocks over all segments (pair: of one)
    int ntiles, kbps;          // tiles, k-blocks per range
    int cl0;                   // first cluster (tile x row chunk) of this op
    int pad_[1];
};
struct TcLaunch {
    TcMap maps[TC_MAX_SEGS + TC_MAX_SRCS];  // weights, then activation planes
    TcSeg segs[TC_MAX_SEGS];
    TcOp ops[TC_MAX_OPS];
    int nops, nclusters, cs, M, rc, npad, stages, stage_bytes, tmem_cols, any_pair, pad_[6];
};
static_assert(sizeof(TcLaunch) % 64 == 0, "descriptor keeps its maps 64-byte aligned");

// Dynamic shared memory of one CTA alone on an SM (227 KB per CTA, less
// the kernel's 1 KB of static shared memory), and of each of two CTAs on
// one SM.  The second is kept to about the footprint of the decode weight
// passes (two CTAs with windows up to 72 KB, 164 KB of the SM's memory as
// shared memory): a pass that needs the largest carve-out forces the SM to
// switch configurations against its neighbours.  Measured in the CUDA graph
// of a verify step at the Llama-3-70B widths, with the gate/up pass on this
// kernel: 3.50 ms with two 36 KB stages per CTA against 4.37 ms with three.
constexpr int TC_SMEM_ONE = 226 * 1024;
constexpr int TC_SMEM_TWO = 80 * 1024;

// Layout of a launch whose rows (M) and ops (N, pair, nkb per op) are set:
// row chunks of at most TC_MAXN rows padded to a multiple of 16; stages
// (two CTAs per SM when two stages fit in TC_SMEM_TWO, else one CTA with up
// to 8 stages); tensor-memory columns; and, when the tiles fill less than
// half the CTA slots, cs k-ranges per tile run by a cluster of cs CTAs (a
// power of two up to TC_MAX_CLUSTER, each range at least 4 k-blocks long
// for the op with the most, and the partials fit in the CTA's shared
// memory).  Returns the CTAs per SM, or 0 when a stage does not fit twice.
inline int tc_layout(TcLaunch& L, int num_sms) {
    L.rc = (L.M + TC_MAXN - 1) / TC_MAXN;
    L.npad = ((L.M + L.rc - 1) / L.rc + 15) / 16 * 16;
    L.any_pair = 0;
    int tiles_all = 0, nkb_max = 0;
    for (int oi = 0; oi < L.nops; ++oi) {
        TcOp& o = L.ops[oi];
        L.any_pair |= o.pair;
        o.ntiles = (o.N + TC_BM - 1) / TC_BM;
        tiles_all += o.ntiles * L.rc;
        nkb_max = o.nkb > nkb_max ? o.nkb : nkb_max;
    }
    L.stage_bytes = TC_BM * TC_BK * 2 * (L.any_pair ? 2 : 1) + 2 * L.npad * TC_BK * 2;
    int ctas_per_sm = 1;
    if (2 * L.stage_bytes + 1024 <= TC_SMEM_TWO) {
        ctas_per_sm = 2;
        L.stages = (TC_SMEM_TWO - 1024) / L.stage_bytes;
    } else {
        L.stages = (TC_SMEM_ONE - 1024) / L.stage_bytes;
    }
    L.stages = L.stages < 8 ? L.stages : 8;
    if (L.stages < 2) return 0;
    const int cols = L.npad * (L.any_pair ? 2 : 1);
    L.tmem_cols = 32;
    while (L.tmem_cols < cols) L.tmem_cols *= 2;
    const int slots = num_sms * ctas_per_sm;
    L.cs = 1;
    if (2 * tiles_all <= slots) {
        const int want = slots / tiles_all < TC_MAX_CLUSTER ? slots / tiles_all : TC_MAX_CLUSTER;
        while (L.cs * 2 <= want) L.cs *= 2;
        while (L.cs > 1 && nkb_max / L.cs < 4) L.cs /= 2;
        const size_t red_bytes = (size_t)(L.any_pair ? 2 : 1) * L.npad * TC_BM * 4;
        if (red_bytes > (size_t)L.stages * L.stage_bytes) L.cs = 1;
    }
    int cl = 0;
    for (int oi = 0; oi < L.nops; ++oi) {
        TcOp& o = L.ops[oi];
        o.kbps = (o.nkb + L.cs - 1) / L.cs;
        o.cl0 = cl;
        cl += o.ntiles * L.rc;
    }
    L.nclusters = cl;
    return ctas_per_sm;
}

// The work of CTA `block`: its cluster is (op, tile, row chunk); its rank in
// the cluster is its k-range [kb_begin, kb_end) of the op's k-blocks
// (possibly empty).
struct TcUnit { int op, tile, chunk, split, kb_begin, kb_end; };
__host__ __device__ inline TcUnit tc_unit(const TcLaunch& L, int block) {
    TcUnit u;
    const int cl = block / L.cs;
    u.split = block % L.cs;
    u.op = 0;
    while (u.op + 1 < L.nops && L.ops[u.op + 1].cl0 <= cl) ++u.op;
    const TcOp& o = L.ops[u.op];
    const int tc = cl - o.cl0;
    u.chunk = tc % L.rc;
    u.tile = tc / L.rc;
    u.kb_begin = u.split * o.kbps < o.nkb ? u.split * o.kbps : o.nkb;
    u.kb_end = u.kb_begin + o.kbps < o.nkb ? u.kb_begin + o.kbps : o.nkb;
    return u;
}

// ------------------------------------------------------------ PTX wrappers
ES_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

ES_DEV unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

ES_DEV void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
ES_DEV void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
ES_DEV bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
// Wait for the phase of `parity` to complete, at most TC_WAIT_NS; false
// (and bit 0 of *err set) when the limit ran out, or when another thread of
// the CTA gave up (*abort) and `stop_on_abort` is set.
ES_DEV bool mbar_wait(uint32_t bar, uint32_t parity, int* err, volatile int* abort, bool stop_on_abort = true,
                      unsigned long long limit_ns = TC_WAIT_NS) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (stop_on_abort && *abort) return false;
            if (global_ns() - t0 > limit_ns) {
                atomicOr(err, 1);
                *abort = 1;
                return false;
            }
        }
    }
}

// The bounded wait on its own: thread 0 waits at most limit_ns for an
// mbarrier that thread 32 arrives at after arrive_ns (never when
// arrive_ns < 0; at most 1 s).  err[0] is set when the wait gives up.
__global__ void wait_selftest_kernel(long long limit_ns, long long arrive_ns, int* err) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_wait(smem_u32(&bar), 0, err, &abort, false, (unsigned long long)limit_ns);
    } else if (threadIdx.x == 32 && arrive_ns >= 0) {
        const unsigned long long t0 = global_ns();
        const unsigned long long d = arrive_ns < 1000000000ll ? (unsigned long long)arrive_ns : 1000000000ull;
        while (global_ns() - t0 < d) {
        }
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar)) : "memory");
    }
    __syncthreads();
}

ES_DEV void tma_load_2d(uint32_t dst, const TcMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar) : "memory");
}
ES_DEV void tma_load_3d(uint32_t dst, const TcMap* map, int c0, int c1, int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar) : "memory");
}

ES_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
ES_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// 128 bytes (64 bf16) in the 128-byte swizzle: 8-row groups 1024 bytes
// apart (stride byte offset), descriptor version 1, layout SWIZZLE_128B.
// The tile starts on a 1024-byte boundary; a k16 step inside it advances the
// start address by 32 bytes.
ES_DEV uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: float32 accumulator, bf16 A and B, both
// K-major, M = 128, N = n.
ES_DEV uint32_t mma_idesc(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(TC_BM >> 4) << 24);
}
ES_DEV void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, int accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        ::"r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
ES_DEV void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// 8 consecutive accumulator columns of this thread's lane, issued without
// waiting: the registers are valid after tmem_wait().
ES_DEV void tmem_ld8(uint32_t taddr, uint32_t* r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
}
ES_DEV void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

ES_DEV float tc_epi(int epi, float a, float b, const float* yp, const float* ap) {
    switch (epi) {
        case GEPI_SWIGLU: return silu_f(a) * b;
        case GEPI_STORE: return a;
        case GEPI_ACC: return __ldcg(yp) + a;
        default: return __ldcg(yp) + a + __ldcg(ap);
    }
}

// ------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(TC_THREADS, 1)
tc_gemm_kernel(const TcLaunch* __restrict__ Lg, int* __restrict__ err) {
    extern __shared__ __align__(1024) unsigned char tsm_raw[];
    __shared__ __align__(8) unsigned long long bars[2 * 8 + 1];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    namespace cg = cooperative_groups;
    // the dynamic region is aligned to 1024 bytes by hand
    unsigned char* tsm = tsm_raw + ((1024 - (smem_u32(tsm_raw) & 1023)) & 1023);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TcLaunch& L = *Lg;
    const int S = L.stages, npad = L.npad, cs = L.cs;
    // ---- which unit: cluster = (op, tile, row chunk), rank in it = k-range
    const TcUnit U = tc_unit(L, blockIdx.x);
    const TcOp& op = L.ops[U.op];
    const int split = U.split, chunk = U.chunk, tile = U.tile;
    const int kb_begin = U.kb_begin, nkb = U.kb_end - U.kb_begin;
    const int pair = op.pair;
    const uint32_t w_bytes = TC_BM * TC_BK * 2;
    const uint32_t x_bytes = 2u * npad * TC_BK * 2;   // both planes
    const uint32_t tx_bytes = w_bytes * (pair ? 2 : 1) + x_bytes;

    auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
    auto empty_bar = [&](int s) { return smem_u32(&bars[8 + s]); };
    const uint32_t acc_bar = smem_u32(&bars[16]);
    auto st_w0 = [&](int s) { return smem_u32(tsm + (size_t)s * L.stage_bytes); };
    auto st_w1 = [&](int s) { return st_w0(s) + w_bytes; };
    auto st_x = [&](int s) { return st_w0(s) + w_bytes * (L.any_pair ? 2 : 1); };

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(L.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort = &s_abort;

    // k-block j of this unit -> segment and its local k-block
    auto locate = [&](int kb, int* seg) {
        int s = op.seg0;
        if (!pair)
            while (s + 1 < op.seg0 + op.nseg && L.segs[s + 1].kb0 <= kb) ++s;
        *seg = s;
        return kb - L.segs[s].kb0;
    };

    if (tid == 0) {
        // ---- TMA producer.  The weight tiles of the first stages go out
        // before the dependency wait; their activation planes after it.
        const int pre = min(S, nkb);
        for (int j = 0; j < pre; ++j) {
            int sg;
            const int kl = locate(kb_begin + j, &sg);
            mbar_arrive_tx(full_bar(j), tx_bytes);
            tma_load_2d(st_w0(j), &L.maps[L.segs[sg].wmap], kl * TC_BK, tile * TC_BM, full_bar(j));
            if (pair) tma_load_2d(st_w1(j), &L.maps[L.segs[sg + 1].wmap], kl * TC_BK, tile * TC_BM, full_bar(j));
        }
        grid_dep_wait();
        for (int j = 0; j < pre; ++j) {
            int sg;
            const int kl = locate(kb_begin + j, &sg);
            tma_load_3d(st_x(j), &L.maps[TC_MAX_SEGS + L.segs[sg].src], kl * TC_BK, chunk * npad, 0, full_bar(j));
        }
        int issued = pre;
        for (int j = pre; j < nkb; ++j) {
            const int s = j % S;
            if (!mbar_wait(empty_bar(s), ((j / S) - 1) & 1, err, abort)) break;
            int sg;
            const int kl = locate(kb_begin + j, &sg);
            mbar_arrive_tx(full_bar(s), tx_bytes);
            tma_load_2d(st_w0(s), &L.maps[L.segs[sg].wmap], kl * TC_BK, tile * TC_BM, full_bar(s));
            if (pair) tma_load_2d(st_w1(s), &L.maps[L.segs[sg + 1].wmap], kl * TC_BK, tile * TC_BM, full_bar(s));
            tma_load_3d(st_x(s), &L.maps[TC_MAX_SEGS + L.segs[sg].src], kl * TC_BK, chunk * npad, 0, full_bar(s));
            issued = j + 1;
        }
        if (*abort) {
            // let the copies still in flight land before the CTA leaves
            for (int j = max(0, issued - S); j < issued; ++j) {
                const unsigned long long t0 = global_ns();
                while (!mbar_test(full_bar(j % S), (j / S) & 1) && global_ns() - t0 < TC_WAIT_NS) {
                }
            }
        }
    } else if (tid == 32) {
        // ---- MMA issuer
        const uint32_t idesc = mma_idesc(npad);
        for (int j = 0; j < nkb; ++j) {
            const int s = j % S;
            if (!mbar_wait(full_bar(s), (j / S) & 1, err, abort)) break;
            tc_fence_after();
            const uint32_t xa = st_x(s), xb = xa + npad * TC_BK * 2;
#pragma unroll
            for (int ks = 0; ks < TC_BK / 16; ++ks) {
                const uint64_t bh = sw128_desc(xa + ks * 32), bl = sw128_desc(xb + ks * 32);
                const uint64_t a0 = sw128_desc(st_w0(s) + ks * 32);
                mma_bf16(tmem, a0, bh, idesc, j > 0 || ks > 0);
                mma_bf16(tmem, a0, bl, idesc, 1);
                if (pair) {
                    const uint64_t a1 = sw128_desc(st_w1(s) + ks * 32);
                    mma_bf16(tmem + npad, a1, bh, idesc, j > 0 || ks > 0);
                    mma_bf16(tmem + npad, a1, bl, idesc, 1);
                }
            }
            mma_commit(empty_bar(s));
        }
        mma_commit(acc_bar);
    }
    __syncwarp();
    grid_dep_wait();

    // ---- epilogue: all warps.  The accumulator barrier completes once every
    // MMA issued has finished (also after an abort), so neither the tensor
    // memory nor the stage buffers are reused under a running MMA.
    bool ok = mbar_wait(acc_bar, 0, err, abort, false);
    ok = __all_sync(0xffffffffu, ok);
    __syncthreads();
    ok = ok && !*abort;            // uniform over the CTA
    const bool have = ok && nkb > 0;  // this CTA's accumulator holds its k-range
    tc_fence_after();
    const int lq = warp & 3, half = warp >> 2;
    const int nl = lq * 32 + lane;              // accumulator lane = weight row in the tile
    const int cw = npad / 2;                    // columns per warp half (multiple of 8)
    const uint32_t tl = tmem + ((uint32_t)(lq * 32) << 16);
    const int r0 = chunk * npad;
    const int nbase = tile * TC_BM;
    auto put = [&](int r, int n, float v) {
        if (op.yp) {
            const bf16 hb = __float2bfloat16_rn(v);
            op.yp[(size_t)r * op.N + n] = hb;
            op.yp[(size_t)L.M * op.N + (size_t)r * op.N + n] = __float2bfloat16_rn(v - __bfloat162float(hb));
        } else {
            op.y[(size_t)r * op.ldy + n] = v;
        }
    };
    auto store = [&](int r, int n, float a, float b) {
        const float* yp = op.y + (size_t)r * op.ldy + n;
        put(r, n, tc_epi(op.epi, a, b, yp, op.add ? op.add + (size_t)r * op.ldy + n : nullptr));
    };
    if (cs == 1) {
        // accumulator -> registers -> y: 16 columns (and the up projection's
        // 16) requested before one wait; for residual epilogues y is read
        // while the tensor-memory loads are in flight
        const int n = nbase + nl;
        if (have) {
            for (int c = half * cw; c < half * cw + cw; c += 16) {
                const int nc = min(16, half * cw + cw - c);  // 16 or 8
                uint32_t ra[16], rb[16];
                float yv[16];
                const bool rmw = op.epi == GEPI_ACC || op.epi == GEPI_ACC_ADD;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int r = r0 + c + i;
                    yv[i] = 0.f;
                    if (rmw && i < nc && r < L.M && n < op.N) {
                        yv[i] = __ldcg(op.y + (size_t)r * op.ldy + n);
                        if (op.epi == GEPI_ACC_ADD) yv[i] += __ldcg(op.add + (size_t)r * op.ldy + n);
                    }
                }
                tmem_ld8(tl + c, ra);
                if (nc == 16) tmem_ld8(tl + c + 8, ra + 8);
                if (pair) {
                    tmem_ld8(tl + npad + c, rb);
                    if (nc == 16) tmem_ld8(tl + npad + c + 8, rb + 8);
                }
                tmem_wait();
                if (n < op.N) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int r = r0 + c + i;
                        if (i >= nc || r >= L.M) continue;
                        const float a = __uint_as_float(ra[i]);
                        float v;
                        if (op.epi == GEPI_SWIGLU) v = silu_f(a) * __uint_as_float(rb[i]);
                        else if (op.epi == GEPI_STORE) v = a;
                        else v = yv[i] + a;
                        put(r, n, v);
                    }
                }
            }
        }
    } else {
        // split tile: partial accumulators meet in distributed shared memory
        // (the stage buffers are free: every load was consumed by an MMA
        // that has completed).  red[acc][column][lane], float32.
        cg::cluster_group cluster = cg::this_cluster();
        float* red = reinterpret_cast<float*>(tsm);
        for (int c = half * cw; c < half * cw + cw; c += 8) {
            uint32_t ra[8], rb[8];
            if (have) {
                tmem_ld8(tl + c, ra);
                if (pair) tmem_ld8(tl + npad + c, rb);
                tmem_wait();
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                red[(size_t)(c + i) * TC_BM + nl] = have ? __uint_as_float(ra[i]) : 0.f;
                if (pair) red[(size_t)(npad + c + i) * TC_BM + nl] = have ? __uint_as_float(rb[i]) : 0.f;
            }
        }
        cluster.sync();
        // this CTA's share: columns [c0, c1) of the tile, 4 lanes per item
        const int cper = (npad + cs - 1) / cs;
        const int c0 = split * cper, c1 = min(npad, c0 + cper);
        const int items = max(0, c1 - c0) * (TC_BM / 4);
        for (int it = tid; it < items; it += TC_THREADS) {
            const int c = c0 + it / (TC_BM / 4), l4 = (it % (TC_BM / 4)) * 4;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            float4 va[TC_MAX_CLUSTER], vb[TC_MAX_CLUSTER];
            float* ea = red + (size_t)c * TC_BM + l4;
            float* eb = red + (size_t)(npad + c) * TC_BM + l4;
#pragma unroll
            for (int q = 0; q < TC_MAX_CLUSTER; ++q) {
                if (q < cs) {
                    va[q] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(ea, q));
                    if (pair) vb[q] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(eb, q));
                }
            }
#pragma unroll
            for (int q = 0; q < TC_MAX_CLUSTER; ++q) {
                if (q < cs) {
                    a.x += va[q].x; a.y += va[q].y; a.z += va[q].z; a.w += va[q].w;
                    if (pair) { b.x += vb[q].x; b.y += vb[q].y; b.z += vb[q].z; b.w += vb[q].w; }
                }
            }
            const int r = r0 + c;
            if (!ok || r >= L.M) continue;
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (nbase + l4 + i < op.N) store(r, nbase + l4 + i, av[i], bv[i]);
        }
        cluster.sync();  // peers may still be reading this CTA's partial
    }
    // dependents launch once every CTA is past its epilogue: a weight-pass
    // CTA that started on an SM still holding this kernel's shared memory
    // would stream through a small L1
    grid_dep_launch();
    tc_fence_before();
    __syncthreads();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L.tmem_cols) : "memory");
}

}  // namespace es
