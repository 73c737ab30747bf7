// libeasyspec: host runtime and C ABI for EasySpec layer-parallel
// speculative decoding on one B300.  See include/easyspec.h for the contract.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/easyspec.h"
#include "kernels.cuh"

using namespace es;

namespace {

struct CudaError { cudaError_t e; const char* what; int line; };
struct ArgError { std::string msg; es_status st; };

#define CK(x)                                                        \
    do {                                                             \
        cudaError_t e_ = (x);                                        \
        if (e_ != cudaSuccess) throw CudaError{e_, #x, __LINE__};   \
    } while (0)

[[noreturn]] void arg_fail(es_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    throw ArgError{buf, st};
}

struct Layer { const void *an, *wq, *wk, *wv, *wo, *mn, *wg, *wu, *wd; };

struct GemvLaunch {
    const GemvOp* ops = nullptr;
    int nops = 0, gemv_tiles = 0, gemm_tiles = 0;
    // algorithmic bytes of one launch over M rows: wbytes + M * rowbytes
    // (weights once; per input row its activations read and outputs written)
    double wbytes = 0, rowbytes = 0;
    double bytes(int M) const { return wbytes + (double)M * rowbytes; }
};

struct ProfRec { const char* name; double bytes; cudaEvent_t a, b; };
struct ProfAgg { double ms = 0, bytes = 0; int64_t launches = 0; };

// One layer set of a forward plan.
struct GroupPlan {
    int first = 0, n = 1;
    bool fuzzy = false;
    NormArgs norm_in{};
    GemvLaunch wide;
    RopeArgs rope{};
    AttnArgs attn{};
    GemvLaunch o;                      // exact: o (acc into h); ATTN_ONLY set: A_j (store)
    int n_mlp = 0;                     // sequential MLPs (exact: 1, ATTN_ONLY set: n)
    NormArgs norm_mlp[MAX_GROUP]{};
    GemvLaunch swi[MAX_GROUP], down[MAX_GROUP];
    GemvLaunch kcat;                   // FULL_LAYER set: o (+) down, acc into h
};

struct Model {
    int L = 0, d = 0, H = 0, Hkv = 0, hd = 0, F = 0, V = 0, qd = 0, kvd = 0, dtype = 0;
    float theta = 0, eps = 0;
    size_t esz = 4;
    const void *embed = nullptr, *lm = nullptr, *fnorm = nullptr;
    std::vector<Layer> ly;
    KVGeom g{};
    float* rope = nullptr;
    int slots = 1, Mw = 0, nsplit = 0;
    float *h = nullptr, *xf = nullptr, *part = nullptr;
    std::vector<float*> xb, mb, q, k, v, a, s, A;
    int *row_pos = nullptr, *row_seq = nullptr, *row_tok = nullptr;
    NormArgs head_norm{};
};

struct Graph { cudaGraphExec_t exec = nullptr; int64_t kernels = 0; };

}  // namespace

struct es_ctx {
    es_config cfg{};
    Model md, mb;
    cudaStream_t st = nullptr;
    bool own_stream = false;
    int dev = 0, num_sms = 148;
    bool poisoned = false;
    std::string err;
    std::vector<void*> allocs;

    // device state
    int* tokens = nullptr;   // [Bmax][max_seq]
    int* n_commit = nullptr; // [Bmax]
    int* n_limit = nullptr;  // [Bmax] commit limit (generate: P + max_new)
    int64_t* phase = nullptr;
    int* dtok = nullptr;     // [Bmax][gmax]
    int* n_acc = nullptr;    // [Bmax]
    int* out_tok = nullptr;  // [Bmax][gmax+1]
    float *q_logits = nullptr, *q_probs = nullptr, *p_logits = nullptr, *p_probs = nullptr;
    RunParams* prm = nullptr;
    int* status = nullptr;
    // pinned host mirrors
    RunParams* h_prm = nullptr;
    int* h_small = nullptr;  // n_acc | out_tok | n_commit | status

    GemvOp* arena = nullptr;
    int arena_cap = 0, arena_used = 0;
    size_t cur_esz = 2;  // weight element size of the model being planned

    // session state
    int B = 0;
    std::vector<int> n_host;  // committed count per sequence (host copy)
    int cur_gamma = 0, cur_k = -1;
    bool calibrated = false, drafted = false;
    float cur_T = 0.f;
    uint64_t cur_seed = 0;

    // launch accounting and optional per-launch event timing
    int64_t launches = 0;
    bool profiling = false;
    std::vector<ProfRec> prof_pending;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> prof_pool;
    size_t prof_pool_used = 0;
    std::map<std::string, ProfAgg> prof;

    std::map<int, std::vector<GroupPlan>> plans;  // key: k (0 = explicit sets)
    std::map<std::tuple<int, int, int>, GemvLaunch> heads;  // (gamma, kind, step)
    std::map<std::tuple<int, int, int, int>, Graph> graphs;  // (part, gamma, k, B)

    template <typename T>
    T* dalloc(size_t n) {
        void* p = nullptr;
        if (n == 0) n = 1;
        cudaError_t e = cudaMalloc(&p, n * sizeof(T));
        if (e != cudaSuccess) { cudaGetLastError(); arg_fail(ES_ERR_OOM, "cudaMalloc of %zu bytes failed", n * sizeof(T)); }
        allocs.push_back(p);
        CK(cudaMemset(p, 0, n * sizeof(T)));
        return (T*)p;
    }
};

namespace {

// ------------------------------------------------------------------ launch helper
template <typename... KArgs, typename... Args>
void launch(es_ctx* c, const char* name, double bytes, void (*kern)(KArgs...), dim3 grid,
            dim3 block, Args... args) {
    if (grid.x == 0 || grid.y == 0 || grid.z == 0) return;
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    if (c->profiling) {
        if (c->prof_pool_used == c->prof_pool.size()) {
            cudaEvent_t x, y;
            CK(cudaEventCreate(&x));
            CK(cudaEventCreate(&y));
            c->prof_pool.emplace_back(x, y);
        }
        ev0 = c->prof_pool[c->prof_pool_used].first;
        ev1 = c->prof_pool[c->prof_pool_used].second;
        c->prof_pool_used++;
        CK(cudaEventRecord(ev0, c->st));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = c->st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CK(cudaLaunchKernelEx(&cfg, kern, args...));
    c->launches++;
    if (c->profiling) {
        CK(cudaEventRecord(ev1, c->st));
        c->prof_pending.push_back(ProfRec{name, bytes, ev0, ev1});
    }
}

// Fold finished event pairs into the per-kernel totals (after a sync).
void prof_collect(es_ctx* c) {
    for (const auto& r : c->prof_pending) {
        float ms = 0.f;
        CK(cudaEventElapsedTime(&ms, r.a, r.b));
        ProfAgg& g = c->prof[r.name];
        g.ms += ms;
        g.bytes += r.bytes;
        g.launches += 1;
    }
    c->prof_pending.clear();
    c->prof_pool_used = 0;
}

// ------------------------------------------------------------------ model setup
void check_shape(const es_model_shape& s, const char* which) {
    if (s.n_layers < 1 || s.d < 8 || s.n_heads < 1 || s.n_kv_heads < 1 || s.head_dim < 2 ||
        s.ffn < 8 || s.vocab < 2)
        arg_fail(ES_ERR_ARG, "%s: non-positive shape field", which);
    if (s.d % 8 || s.ffn % 8 || (s.n_heads * s.head_dim) % 8)
        arg_fail(ES_ERR_ARG, "%s: d, ffn and n_heads*head_dim must be multiples of 8", which);
    if (s.head_dim % 2 || s.head_dim > 256)
        arg_fail(ES_ERR_ARG, "%s: head_dim must be even and <= 256", which);
    if (s.n_heads % s.n_kv_heads || s.n_heads / s.n_kv_heads > MAX_GQA)
        arg_fail(ES_ERR_ARG, "%s: n_heads must be a multiple of n_kv_heads (ratio <= %d)", which, MAX_GQA);
    if (s.dtype != ES_DTYPE_F32 && s.dtype != ES_DTYPE_BF16)
        arg_fail(ES_ERR_ARG, "%s: dtype must be ES_DTYPE_F32 or ES_DTYPE_BF16", which);
    if (!(s.eps > 0) || !(s.rope_theta > 1))
        arg_fail(ES_ERR_ARG, "%s: eps must be > 0 and rope_theta > 1", which);
}

void check_ptr(const void* p, const char* what) {
    if (!p) arg_fail(ES_ERR_ARG, "null weight pointer: %s", what);
    if ((uintptr_t)p % 16) arg_fail(ES_ERR_ARG, "weight pointer not 16-byte aligned: %s", what);
}

void setup_model(es_ctx* c, Model& m, const es_model_shape& s, const es_weights* w,
                 int slots, const char* which) {
    check_shape(s, which);
    if (!w) arg_fail(ES_ERR_ARG, "%s: null weights", which);
    m.L = s.n_layers; m.d = s.d; m.H = s.n_heads; m.Hkv = s.n_kv_heads; m.hd = s.head_dim;
    m.F = s.ffn; m.V = s.vocab; m.qd = m.H * m.hd; m.kvd = m.Hkv * m.hd; m.dtype = s.dtype;
    m.theta = s.rope_theta; m.eps = s.eps; m.esz = s.dtype == ES_DTYPE_BF16 ? 2 : 4;
    check_ptr(w->embed, "embed"); check_ptr(w->lm_head, "lm_head"); check_ptr(w->final_norm, "final_norm");
    m.embed = w->embed; m.lm = w->lm_head; m.fnorm = w->final_norm;
    if (!w->attn_norm || !w->wq || !w->wk || !w->wv || !w->wo || !w->mlp_norm || !w->wgate ||
        !w->wup || !w->wdown)
        arg_fail(ES_ERR_ARG, "%s: null per-layer pointer array", which);
    m.ly.resize(m.L);
    for (int l = 0; l < m.L; ++l) {
        Layer& y = m.ly[l];
        y.an = w->attn_norm[l]; y.wq = w->wq[l]; y.wk = w->wk[l]; y.wv = w->wv[l]; y.wo = w->wo[l];
        y.mn = w->mlp_norm[l]; y.wg = w->wgate[l]; y.wu = w->wup[l]; y.wd = w->wdown[l];
        const void* ps[9] = {y.an, y.wq, y.wk, y.wv, y.wo, y.mn, y.wg, y.wu, y.wd};
        for (const void* p : ps) check_ptr(p, which);
    }
    const int Bmax = c->cfg.max_batch, S = c->cfg.max_seq;
    // paged KV: each sequence owns ceil(S/64) pages, listed in its page table
    const int pps = (S + PAGE - 1) / PAGE;
    m.g.pages_per_seq = pps; m.g.L = m.L; m.g.Hkv = m.Hkv; m.g.hd = m.hd; m.g.max_seq = S;
    const size_t page_elems = (size_t)m.L * 2 * m.Hkv * PAGE * m.hd;
    m.g.kv = c->dalloc<char>((size_t)Bmax * pps * page_elems * m.esz);
    std::vector<int> pt((size_t)Bmax * pps);
    for (size_t i = 0; i < pt.size(); ++i) pt[i] = (int)i;
    int* ptd = c->dalloc<int>(pt.size());
    CK(cudaMemcpy(ptd, pt.data(), pt.size() * sizeof(int), cudaMemcpyHostToDevice));
    m.g.page_table = ptd;
    // rotary table [pos][i][cos, sin], angle pos * theta^(-2i/hd), in double
    const int half = m.hd / 2;
    std::vector<float> rt((size_t)S * half * 2);
    for (int p = 0; p < S; ++p)
        for (int i = 0; i < half; ++i) {
            const double ang = (double)p * std::pow((double)m.theta, -2.0 * i / m.hd);
            rt[((size_t)p * half + i) * 2] = (float)std::cos(ang);
            rt[((size_t)p * half + i) * 2 + 1] = (float)std::sin(ang);
        }
    m.rope = c->dalloc<float>(rt.size());
    CK(cudaMemcpy(m.rope, rt.data(), rt.size() * sizeof(float), cudaMemcpyHostToDevice));
    // workspace rows: decode batches and prefill chunks
    m.Mw = std::max(Bmax * (c->cfg.max_gamma + 1), 256);
    m.slots = slots;
    const size_t Mw = m.Mw;
    m.h = c->dalloc<float>(Mw * m.d);
    m.xf = c->dalloc<float>(Mw * m.d);
    for (int j = 0; j < slots; ++j) {
        m.xb.push_back(c->dalloc<float>(Mw * m.d));
        m.mb.push_back(c->dalloc<float>(Mw * m.d));
        m.q.push_back(c->dalloc<float>(Mw * m.qd));
        m.k.push_back(c->dalloc<float>(Mw * m.kvd));
        m.v.push_back(c->dalloc<float>(Mw * m.kvd));
        m.a.push_back(c->dalloc<float>(Mw * m.qd));
        m.s.push_back(c->dalloc<float>(Mw * m.F));
        m.A.push_back(c->dalloc<float>(Mw * m.d));
    }
    m.nsplit = pps;
    m.part = c->dalloc<float>(Mw * slots * m.H * (size_t)pps * (m.hd + 2));
    m.row_pos = c->dalloc<int>(Mw);
    m.row_seq = c->dalloc<int>(Mw);
    m.row_tok = c->dalloc<int>(Mw);
}

// ------------------------------------------------------------------ op descriptors
GemvLaunch upload_ops(es_ctx* c, std::vector<GemvOp> ops) {
    GemvLaunch gl;
    int t8 = 0, t64 = 0;
    for (auto& op : ops) { op.tile0 = t8; t8 += (op.N + GEMV_WARPS - 1) / GEMV_WARPS; }
    // gemm tiles are derived from the same ops with a 64-row tile: store a
    // second copy with tile0 in 64-row units right after the first
    std::vector<GemvOp> ops64 = ops;
    for (auto& op : ops64) { op.tile0 = t64; t64 += (op.N + GB - 1) / GB; }
    const int n = (int)ops.size();
    if (c->arena_used + 2 * n > c->arena_cap) arg_fail(ES_ERR_OOM, "op descriptor arena exhausted");
    GemvOp* dst = c->arena + c->arena_used;
    CK(cudaMemcpy(dst, ops.data(), n * sizeof(GemvOp), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dst + n, ops64.data(), n * sizeof(GemvOp), cudaMemcpyHostToDevice));
    c->arena_used += 2 * n;
    gl.ops = dst; gl.nops = n; gl.gemv_tiles = t8; gl.gemm_tiles = t64;
    for (const auto& op : ops) {
        for (int s = 0; s < op.nseg; ++s) {
            gl.wbytes += (double)op.N * op.seg[s].K * c->cur_esz;
            gl.rowbytes += (double)op.seg[s].K * 4.0;
        }
        gl.rowbytes += (double)op.N * 4.0 * (op.epi == EPI_ACC ? 2 : 1);
    }
    return gl;
}

GemvOp make_op(int N, float* y, int ldy, int epi) {
    GemvOp op;
    memset(&op, 0, sizeof op);
    op.N = N; op.y = y; op.ldy = ldy; op.epi = epi;
    return op;
}
void add_seg(GemvOp& op, const void* W, const float* x, int K, int ldx) {
    if (op.nseg >= MAX_SEG) arg_fail(ES_ERR_ARG, "too many K-concatenated segments");
    op.seg[op.nseg++] = GemvSeg{W, x, K, ldx};
}

NormArgs norm_args(Model& m, float* h, const float* add) {
    NormArgs a;
    memset(&a, 0, sizeof a);
    a.h = h; a.add = add; a.d = m.d; a.eps = m.eps; a.src_stride = 1; a.src_off = 0;
    a.out_ld = m.d;
    return a;
}
void add_job(NormArgs& a, const void* g, float* out) {
    a.g[a.njobs] = g;
    a.out[a.njobs] = out;
    a.njobs++;
}

RopeArgs rope_args(Model& m) {
    RopeArgs r;
    memset(&r, 0, sizeof r);
    r.g = m.g; r.rope = m.rope; r.H = m.H; r.row_pos = m.row_pos; r.row_seq = m.row_seq;
    return r;
}
AttnArgs attn_args(Model& m) {
    AttnArgs a;
    memset(&a, 0, sizeof a);
    a.g = m.g; a.H = m.H; a.nsplit = m.nsplit; a.part = m.part; a.row_pos = m.row_pos;
    a.row_seq = m.row_seq;
    return a;
}

// Plan of one forward pass for the layer sets `groups` (sets of one layer are
// exact layers).
std::vector<GroupPlan> build_plan(es_ctx* c, Model& m, const std::vector<std::vector<int>>& groups,
                                  int mode) {
    std::vector<GroupPlan> plan;
    for (const auto& gl : groups) {
        GroupPlan gp;
        gp.first = gl.front();
        gp.n = (int)gl.size();
        gp.fuzzy = gp.n > 1;
        if (gp.n > m.slots || gp.n > MAX_GROUP) arg_fail(ES_ERR_ARG, "layer set larger than %d", MAX_GROUP);
        const int n = gp.n;
        const bool full = gp.fuzzy && mode == ES_FULL_LAYER;
        // input norms from the set input h
        gp.norm_in = norm_args(m, m.h, nullptr);
        for (int j = 0; j < n; ++j) add_job(gp.norm_in, m.ly[gp.first + j].an, m.xb[j]);
        if (full)
            for (int j = 0; j < n; ++j) add_job(gp.norm_in, m.ly[gp.first + j].mn, m.mb[j]);
        // wide pass: q,k,v of every layer (+ SwiGLU of every layer for FULL_LAYER)
        std::vector<GemvOp> wide;
        for (int j = 0; j < n; ++j) {
            const Layer& y = m.ly[gp.first + j];
            GemvOp oq = make_op(m.qd, m.q[j], m.qd, EPI_STORE); add_seg(oq, y.wq, m.xb[j], m.d, m.d);
            GemvOp ok = make_op(m.kvd, m.k[j], m.kvd, EPI_STORE); add_seg(ok, y.wk, m.xb[j], m.d, m.d);
            GemvOp ov = make_op(m.kvd, m.v[j], m.kvd, EPI_STORE); add_seg(ov, y.wv, m.xb[j], m.d, m.d);
            wide.push_back(oq); wide.push_back(ok); wide.push_back(ov);
        }
        if (full)
            for (int j = 0; j < n; ++j) {
                const Layer& y = m.ly[gp.first + j];
                GemvOp os = make_op(m.F, m.s[j], m.F, EPI_SWIGLU);
                add_seg(os, y.wg, m.mb[j], m.d, m.d);
                add_seg(os, y.wu, m.mb[j], m.d, m.d);
                wide.push_back(os);
            }
        gp.wide = upload_ops(c, wide);
        gp.rope = rope_args(m);
        gp.attn = attn_args(m);
        gp.rope.nl = gp.attn.nl = n;
        for (int j = 0; j < n; ++j) {
            gp.rope.layer[j] = gp.attn.layer[j] = gp.first + j;
            gp.rope.q[j] = m.q[j]; gp.rope.k[j] = m.k[j]; gp.rope.v[j] = m.v[j];
            gp.attn.q[j] = m.q[j]; gp.attn.out[j] = m.a[j];
        }
        if (full) {
            // K-concatenated [Wo_1 .. Wo_n, Wdown_1 .. Wdown_n] . [a_1..a_n, s_1..s_n]
            GemvOp kc = make_op(m.d, m.h, m.d, EPI_ACC);
            for (int j = 0; j < n; ++j) add_seg(kc, m.ly[gp.first + j].wo, m.a[j], m.qd, m.qd);
            for (int j = 0; j < n; ++j) add_seg(kc, m.ly[gp.first + j].wd, m.s[j], m.F, m.F);
            gp.kcat = upload_ops(c, {kc});
            gp.n_mlp = 0;
        } else {
            std::vector<GemvOp> os;
            for (int j = 0; j < n; ++j) {
                // exact layer: o accumulates into h; ATTN_ONLY set: A_j stored
                GemvOp o = gp.fuzzy ? make_op(m.d, m.A[j], m.d, EPI_STORE) : make_op(m.d, m.h, m.d, EPI_ACC);
                add_seg(o, m.ly[gp.first + j].wo, m.a[j], m.qd, m.qd);
                os.push_back(o);
            }
            gp.o = upload_ops(c, os);
            gp.n_mlp = n;
            for (int j = 0; j < n; ++j) {
                const Layer& y = m.ly[gp.first + j];
                gp.norm_mlp[j] = norm_args(m, m.h, gp.fuzzy ? m.A[j] : nullptr);
                add_job(gp.norm_mlp[j], y.mn, m.mb[0]);
                GemvOp sw = make_op(m.F, m.s[0], m.F, EPI_SWIGLU);
                add_seg(sw, y.wg, m.mb[0], m.d, m.d);
                add_seg(sw, y.wu, m.mb[0], m.d, m.d);
                gp.swi[j] = upload_ops(c, {sw});
                GemvOp dn = make_op(m.d, m.h, m.d, EPI_ACC);
                add_seg(dn, y.wd, m.s[0], m.F, m.F);
                gp.down[j] = upload_ops(c, {dn});
            }
        }
        plan.push_back(gp);
    }
    return plan;
}

std::vector<std::vector<int>> default_sets(int L, int k) {
    std::vector<std::vector<int>> g;
    if (k <= 1 || L <= 2) {
        for (int l = 0; l < L; ++l) g.push_back({l});
        return g;
    }
    g.push_back({0});
    for (int start = 0; start < L; start += k) {
        std::vector<int> blk;
        for (int l = start; l < start + k; ++l)
            if (l >= 1 && l <= L - 2) blk.push_back(l);
        if (!blk.empty()) g.push_back(blk);
    }
    g.push_back({L - 1});
    return g;
}

// ------------------------------------------------------------------ launches
template <typename T>
void run_gemv(es_ctx* c, const GemvLaunch& gl, int M) {
    if (gl.nops == 0 || M <= 0) return;
    const int block = GEMV_WARPS * 32;
    if (M <= 8) {
        const int grid = std::min(gl.gemv_tiles, c->num_sms * 6);
        switch (M) {
#define ES_GEMV_CASE(MM) \
    case MM: launch(c, "gemv_m" #MM, gl.bytes(M), gemv_kernel<T, MM>, dim3(grid), dim3(block), gl.ops, gl.nops, gl.gemv_tiles); break;
            ES_GEMV_CASE(1) ES_GEMV_CASE(2) ES_GEMV_CASE(3) ES_GEMV_CASE(4)
            ES_GEMV_CASE(5) ES_GEMV_CASE(6) ES_GEMV_CASE(7) ES_GEMV_CASE(8)
#undef ES_GEMV_CASE
        }
    } else {
        launch(c, "gemm_simt", gl.bytes(M), gemm_kernel<T>, dim3(gl.gemm_tiles, (M + GB - 1) / GB), dim3(256),
               gl.ops + gl.nops, gl.nops, M);
    }
}

template <typename T>
void run_norm(es_ctx* c, const NormArgs& a, int rows) {
    launch(c, "rmsnorm", 0.0, norm_kernel<T>, dim3(rows), dim3(256), a);
}

template <typename T>
void run_group(es_ctx* c, Model& m, const GroupPlan& gp, int M) {
    run_norm<T>(c, gp.norm_in, M);
    run_gemv<T>(c, gp.wide, M);
    RopeArgs r = gp.rope; r.M = M;
    launch(c, "rope_kv", 0.0, rope_kv_kernel<T>, dim3(M, gp.n), dim3(128), r);
    AttnArgs a = gp.attn; a.M = M;
    launch(c, "attn_split", 0.0, attn_split_kernel<T>, dim3(M, gp.n * m.Hkv, m.nsplit), dim3(128), a);
    launch(c, "attn_combine", 0.0, attn_combine_kernel, dim3(M, gp.n, m.H), dim3(std::max(32, (m.hd + 31) / 32 * 32)), a);
    if (gp.kcat.nops) {
        run_gemv<T>(c, gp.kcat, M);
        return;
    }
    run_gemv<T>(c, gp.o, M);
    for (int j = 0; j < gp.n_mlp; ++j) {
        run_norm<T>(c, gp.norm_mlp[j], M);
        run_gemv<T>(c, gp.swi[j], M);
        run_gemv<T>(c, gp.down[j], M);
    }
}

// Body of one forward pass over M rows already described by the row arrays
// (or described by `kind` on the device).
template <typename T>
void run_forward(es_ctx* c, Model& m, const std::vector<GroupPlan>& plan, int kind, int step,
                 int gamma, int M) {
    launch(c, "prep_embed", 0.0, prep_embed_kernel<T>, dim3(M), dim3(256), kind, step, gamma, M,
           (const int*)c->n_commit, (const int*)c->tokens, c->cfg.max_seq, (const int*)c->dtok,
           c->cfg.max_gamma, m.row_pos, m.row_seq, m.row_tok, (const T*)m.embed, m.h, m.d, m.V,
           c->status);
    for (const auto& gp : plan) run_group<T>(c, m, gp, M);
}

// Head: final norm of the selected rows and the output projection.
template <typename T>
void run_head(es_ctx* c, Model& m, int rows, int src_stride, int src_off, const GemvLaunch& lm) {
    NormArgs a = norm_args(m, m.h, nullptr);
    a.src_stride = src_stride; a.src_off = src_off;
    add_job(a, m.fnorm, m.xf);
    run_norm<T>(c, a, rows);
    run_gemv<T>(c, lm, rows);
}

const GemvLaunch& head_desc(es_ctx* c, Model& m, int gamma, int kind, int step) {
    auto key = std::make_tuple(gamma, kind, step);
    auto it = c->heads.find(key);
    if (it != c->heads.end()) return it->second;
    GemvOp op;
    if (kind == KIND_VERIFY) op = make_op(m.V, c->p_logits, m.V, EPI_STORE);
    else op = make_op(m.V, c->q_logits + (size_t)step * m.V, gamma * m.V, EPI_STORE);
    add_seg(op, m.lm, m.xf, m.d, m.d);
    c->cur_esz = m.esz;
    return c->heads[key] = upload_ops(c, {op});
}

// ------------------------------------------------------------------ phase parts
template <typename TD>
void enqueue_calibrate(es_ctx* c, const std::vector<GroupPlan>& exact_d, int gamma) {
    Model& m = c->md;
    const int B = c->B;
    const GemvLaunch& lm = head_desc(c, m, gamma, KIND_CALIB, 0);
    run_forward<TD>(c, m, exact_d, KIND_CALIB, 0, gamma, B * (gamma + 1));
    run_head<TD>(c, m, B, gamma + 1, gamma, lm);
    launch(c, "softmax_sample", 0.0, softmax_sample_kernel, dim3(B), dim3(1024), (const float*)c->q_logits, c->q_probs, m.V,
           1, 0, gamma, (const RunParams*)c->prm, (const int64_t*)c->phase, gamma, c->dtok,
           c->cfg.max_gamma);
}

template <typename TD>
void enqueue_fuzzy(es_ctx* c, const std::vector<GroupPlan>& plan, int gamma) {
    Model& m = c->md;
    const int B = c->B;
    for (int i = 1; i < gamma; ++i) {
        const GemvLaunch& lm = head_desc(c, m, gamma, KIND_FUZZY, i);
        run_forward<TD>(c, m, plan, KIND_FUZZY, i, gamma, B);
        run_head<TD>(c, m, B, 1, 0, lm);
        launch(c, "softmax_sample", 0.0, softmax_sample_kernel, dim3(B), dim3(1024), (const float*)c->q_logits, c->q_probs,
               m.V, 1, i, gamma, (const RunParams*)c->prm, (const int64_t*)c->phase, gamma, c->dtok,
               c->cfg.max_gamma);
    }
}

template <typename TB>
void enqueue_verify(es_ctx* c, const std::vector<GroupPlan>& exact_b, int gamma) {
    Model& m = c->mb;
    const int B = c->B, M = B * (gamma + 1);
    const GemvLaunch& lm = head_desc(c, m, gamma, KIND_VERIFY, 0);
    run_forward<TB>(c, m, exact_b, KIND_VERIFY, 0, gamma, M);
    run_head<TB>(c, m, M, 1, 0, lm);
    launch(c, "softmax", 0.0, softmax_sample_kernel, dim3(M), dim3(1024), (const float*)c->p_logits, c->p_probs, m.V,
           gamma + 1, 0, gamma + 1, (const RunParams*)c->prm, (const int64_t*)c->phase, gamma,
           (int*)nullptr, c->cfg.max_gamma);
    AcceptArgs a;
    memset(&a, 0, sizeof a);
    a.p = c->p_probs; a.q = c->q_probs; a.d = c->dtok; a.gmax = c->cfg.max_gamma; a.gamma = gamma;
    a.V = m.V; a.greedy = -1; a.u_explicit = nullptr; a.prm = c->prm; a.phase = c->phase;
    a.n_acc = c->n_acc; a.out_tok = c->out_tok; a.tokens = c->tokens; a.max_seq = c->cfg.max_seq;
    a.n_commit = c->n_commit; a.n_limit = c->n_limit;
    launch(c, "accept_resample", 0.0, accept_kernel, dim3(B), dim3(1024), a);
}

}  // namespace

namespace {

void set_error(es_ctx* c, const std::string& s) { if (c) c->err = s; }

template <typename F>
es_status guarded(es_ctx* c, F&& f) {
    if (c && c->poisoned) return ES_ERR_STATE;
    try {
        f();
        return ES_OK;
    } catch (const ArgError& e) {
        set_error(c, e.msg);
        return e.st;
    } catch (const CudaError& e) {
        char buf[512];
        snprintf(buf, sizeof buf, "CUDA error %d (%s) at easyspec.cu:%d in %s", (int)e.e,
                 cudaGetErrorString(e.e), e.line, e.what);
        set_error(c, buf);
        if (c) c->poisoned = true;
        return ES_ERR_CUDA;
    } catch (const std::exception& e) {
        set_error(c, e.what());
        if (c) c->poisoned = true;
        return ES_ERR_CUDA;
    }
}

void prof_collect(es_ctx* c);
void check_status(es_ctx* c) {
    // reads the device status word (call after a stream sync)
    if (c->profiling) prof_collect(c);
    int s = 0;
    CK(cudaMemcpy(&s, c->status, sizeof(int), cudaMemcpyDeviceToHost));
    if (s) {
        CK(cudaMemset(c->status, 0, sizeof(int)));
        arg_fail(ES_ERR_STATE, "device reported invalid rows (status 0x%x): position past max_seq or token out of range", s);
    }
}

const std::vector<GroupPlan>& get_plan(es_ctx* c, int key) {
    auto it = c->plans.find(key);
    if (it != c->plans.end()) return it->second;
    std::vector<std::vector<int>> sets;
    Model& m = (key == -1) ? c->mb : c->md;
    if (key == -1 || key == 1) {
        sets = default_sets(m.L, 1);
    } else if (key == 0) {
        for (int i = 0; i < c->cfg.n_groups; ++i) {
            const int s0 = c->cfg.group_starts[i];
            const int s1 = i + 1 < c->cfg.n_groups ? c->cfg.group_starts[i + 1] : m.L;
            std::vector<int> g;
            for (int l = s0; l < s1; ++l) g.push_back(l);
            sets.push_back(g);
        }
    } else {
        sets = default_sets(m.L, key);
    }
    c->cur_esz = m.esz;
    return c->plans[key] = build_plan(c, m, sets, c->cfg.parallel_mode);
}

void set_params(es_ctx* c, float T, uint64_t seed) {
    c->h_prm->seed = seed;
    c->h_prm->temperature = T;
    CK(cudaMemcpyAsync(c->prm, c->h_prm, sizeof(RunParams), cudaMemcpyHostToDevice, c->st));
}

template <typename TD, typename TB>
void enqueue_part(es_ctx* c, int part, int gamma, int k) {
    if (part == 0) {
        enqueue_calibrate<TD>(c, get_plan(c, 1), gamma);
        enqueue_fuzzy<TD>(c, get_plan(c, k), gamma);
    } else if (part == 1) {
        enqueue_verify<TB>(c, get_plan(c, -1), gamma);
    } else if (part == 2) {
        enqueue_calibrate<TD>(c, get_plan(c, 1), gamma);
    } else {
        enqueue_fuzzy<TD>(c, get_plan(c, k), gamma);
    }
}

void dispatch_part(es_ctx* c, int part, int gamma, int k) {
    const bool dbf = c->md.dtype == ES_DTYPE_BF16, bbf = c->mb.dtype == ES_DTYPE_BF16;
    if (dbf && bbf) enqueue_part<bf16, bf16>(c, part, gamma, k);
    else if (dbf) enqueue_part<bf16, float>(c, part, gamma, k);
    else if (bbf) enqueue_part<float, bf16>(c, part, gamma, k);
    else enqueue_part<float, float>(c, part, gamma, k);
}

// Parts: 0 = calibration + fuzzy drafts, 1 = verify + accept,
// 2 = calibration only, 3 = fuzzy drafts only.  Captured once per
// (part, gamma, k, B) as a CUDA graph and replayed.
void run_part(es_ctx* c, int part, int gamma, int k) {
    // build every descriptor before capture (uploads are synchronous)
    if (part != 1) { get_plan(c, 1); get_plan(c, k); }
    else get_plan(c, -1);
    for (int i = 0; i < gamma; ++i) head_desc(c, c->md, gamma, i == 0 ? KIND_CALIB : KIND_FUZZY, i);
    head_desc(c, c->mb, gamma, KIND_VERIFY, 0);
    if (c->profiling) {  // eager launches, each bracketed by events
        dispatch_part(c, part, gamma, k);
        return;
    }
    auto key = std::make_tuple(part, gamma, k, c->B);
    auto it = c->graphs.find(key);
    if (it == c->graphs.end()) {
        cudaGraph_t g;
        const int64_t l0 = c->launches;
        CK(cudaStreamBeginCapture(c->st, cudaStreamCaptureModeThreadLocal));
        try {
            dispatch_part(c, part, gamma, k);
        } catch (...) {
            cudaGraph_t junk;
            cudaStreamEndCapture(c->st, &junk);
            if (junk) cudaGraphDestroy(junk);
            cudaGetLastError();
            throw;
        }
        CK(cudaStreamEndCapture(c->st, &g));
        Graph gr;
        gr.kernels = c->launches - l0;
        c->launches = l0;
        CK(cudaGraphInstantiate(&gr.exec, g, 0));
        CK(cudaGraphDestroy(g));
        it = c->graphs.emplace(key, gr).first;
    }
    CK(cudaGraphLaunch(it->second.exec, c->st));
    c->launches += it->second.kernels;
}

template <typename T>
void prefill_model(es_ctx* c, Model& m, const int32_t* prompts, int B, int P) {
    // exact forward over positions 0..P-2 of every sequence, in chunks of
    // positions (rows of a chunk only attend to earlier positions)
    const auto& plan = (&m == &c->mb) ? get_plan(c, -1) : get_plan(c, 1);
    const int npos = P - 1;
    if (npos <= 0) return;
    const int chunk = std::max(1, m.Mw / B);
    std::vector<int> pos, seq, tok;
    for (int p0 = 0; p0 < npos; p0 += chunk) {
        const int p1 = std::min(npos, p0 + chunk);
        pos.clear(); seq.clear(); tok.clear();
        for (int b = 0; b < B; ++b)
            for (int p = p0; p < p1; ++p) {
                pos.push_back(p); seq.push_back(b); tok.push_back(prompts[(size_t)b * P + p]);
            }
        const int M = (int)pos.size();
        CK(cudaMemcpyAsync(m.row_pos, pos.data(), M * sizeof(int), cudaMemcpyHostToDevice, c->st));
        CK(cudaMemcpyAsync(m.row_seq, seq.data(), M * sizeof(int), cudaMemcpyHostToDevice, c->st));
        CK(cudaMemcpyAsync(m.row_tok, tok.data(), M * sizeof(int), cudaMemcpyHostToDevice, c->st));
        run_forward<T>(c, m, plan, KIND_HOST, 0, 0, M);
        CK(cudaStreamSynchronize(c->st));  // host row buffers are reused
    }
}

void do_prefill(es_ctx* c, const int32_t* prompts, int B, int P) {
    if (!prompts || B < 1 || P < 1) arg_fail(ES_ERR_ARG, "prefill: need prompts, B >= 1, P >= 1");
    if (B > c->cfg.max_batch) arg_fail(ES_ERR_ARG, "prefill: B=%d exceeds max_batch=%d", B, c->cfg.max_batch);
    if (P + 2 > c->cfg.max_seq) arg_fail(ES_ERR_CAPACITY, "prefill: prompt length %d too long for max_seq %d", P, c->cfg.max_seq);
    for (size_t i = 0; i < (size_t)B * P; ++i)
        if (prompts[i] < 0 || prompts[i] >= c->md.V) arg_fail(ES_ERR_ARG, "prefill: token id out of range");
    c->B = B;
    for (int b = 0; b < B; ++b)
        CK(cudaMemcpyAsync(c->tokens + (size_t)b * c->cfg.max_seq, prompts + (size_t)b * P,
                           P * sizeof(int), cudaMemcpyHostToDevice, c->st));
    std::vector<int> n(B, P), lim(B, 0x7fffffff);
    CK(cudaMemcpyAsync(c->n_commit, n.data(), B * sizeof(int), cudaMemcpyHostToDevice, c->st));
    CK(cudaMemcpyAsync(c->n_limit, lim.data(), B * sizeof(int), cudaMemcpyHostToDevice, c->st));
    CK(cudaMemsetAsync(c->phase, 0, sizeof(int64_t) * c->cfg.max_batch, c->st));
    c->n_host.assign(B, P);
    if (c->mb.dtype == ES_DTYPE_BF16) prefill_model<bf16>(c, c->mb, prompts, B, P);
    else prefill_model<float>(c, c->mb, prompts, B, P);
    if (c->md.dtype == ES_DTYPE_BF16) prefill_model<bf16>(c, c->md, prompts, B, P);
    else prefill_model<float>(c, c->md, prompts, B, P);
    CK(cudaStreamSynchronize(c->st));
    check_status(c);
    c->calibrated = c->drafted = false;
    c->cur_gamma = 0;
}

void check_phase_args(es_ctx* c, int gamma, float T) {
    if (c->B < 1) arg_fail(ES_ERR_STATE, "no prompts loaded (call easyspec_prefill or generate)");
    if (gamma < 1 || gamma > c->cfg.max_gamma) arg_fail(ES_ERR_ARG, "gamma=%d outside 1..max_gamma=%d", gamma, c->cfg.max_gamma);
    if (!(T >= 0.f) || std::isinf(T)) arg_fail(ES_ERR_ARG, "temperature must be finite and >= 0");
    for (int b = 0; b < c->B; ++b)
        if (c->n_host[b] + gamma + 1 > c->cfg.max_seq)
            arg_fail(ES_ERR_CAPACITY, "sequence %d would exceed max_seq=%d", b, c->cfg.max_seq);
}

int resolve_k(es_ctx* c, int k) {
    if (c->cfg.group_starts) {
        if (k != 0) arg_fail(ES_ERR_ARG, "explicit layer sets configured: k must be 0");
        return 0;
    }
    if (k < 1 || k > MAX_GROUP) arg_fail(ES_ERR_ARG, "k=%d outside 1..%d", k, MAX_GROUP);
    return k;
}

void read_phase_result(es_ctx* c, int gamma, int32_t* n_accepted, int32_t* tokens_out) {
    const int B = c->B;
    int* hs = c->h_small;
    CK(cudaMemcpyAsync(hs, c->n_acc, B * sizeof(int), cudaMemcpyDeviceToHost, c->st));
    CK(cudaMemcpyAsync(hs + 64, c->out_tok, (size_t)B * (gamma + 1) * sizeof(int), cudaMemcpyDeviceToHost, c->st));
    CK(cudaMemcpyAsync(hs + 64 + 64 * 17, c->n_commit, B * sizeof(int), cudaMemcpyDeviceToHost, c->st));
    CK(cudaStreamSynchronize(c->st));
    check_status(c);
    for (int b = 0; b < B; ++b) c->n_host[b] = hs[64 + 64 * 17 + b];
    if (n_accepted) memcpy(n_accepted, hs, B * sizeof(int));
    if (tokens_out) memcpy(tokens_out, hs + 64, (size_t)B * (gamma + 1) * sizeof(int));
}

es_stats do_decode(es_ctx* c, int max_new, int gamma, int k, float temperature, uint64_t seed) {
    const int kk = resolve_k(c, k);
    check_phase_args(c, gamma, temperature);
    const int B = c->B;
    auto t0 = std::chrono::steady_clock::now();
    const int64_t l0 = c->launches;
    set_params(c, temperature, seed);
    // a sequence stops committing once it has max_new more tokens; its rows
    // idle until the whole batch is done
    std::vector<int> start(c->n_host), lim(B);
    for (int b = 0; b < B; ++b) lim[b] = start[b] + max_new;
    CK(cudaMemcpyAsync(c->n_limit, lim.data(), B * sizeof(int), cudaMemcpyHostToDevice, c->st));
    std::vector<int64_t> ph0(B), ph1(B);
    CK(cudaMemcpyAsync(ph0.data(), c->phase, B * sizeof(int64_t), cudaMemcpyDeviceToHost, c->st));
    es_stats s{};
    // batches of phases that the least advanced sequence needs in any case
    // (a phase commits at most gamma+1 tokens), then read back the counts
    while (true) {
        int rem = 0;
        for (int b = 0; b < B; ++b) rem = std::max(rem, max_new - (c->n_host[b] - start[b]));
        if (rem <= 0) break;
        const int nph = (rem + gamma) / (gamma + 1);
        for (int i = 0; i < nph; ++i) {
            run_part(c, 0, gamma, kk);
            run_part(c, 1, gamma, kk);
        }
        s.phases += nph;
        read_phase_result(c, gamma, nullptr, nullptr);
    }
    // per-sequence phase counters advance only on commits
    CK(cudaMemcpy(ph1.data(), c->phase, B * sizeof(int64_t), cudaMemcpyDeviceToHost));
    int64_t active = 0;
    for (int b = 0; b < B; ++b) {
        s.emitted += c->n_host[b] - start[b];
        active += ph1[b] - ph0[b];
    }
    s.drafted = active * gamma;
    s.accepted = s.emitted - active;
    s.kernel_launches = c->launches - l0;
    s.decode_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    c->calibrated = c->drafted = false;
    return s;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

es_status easyspec_init(const es_config* cfg, const es_weights* draft, const es_weights* base,
                        es_ctx** out) {
    if (!out) return ES_ERR_ARG;
    *out = nullptr;
    if (!cfg) return ES_ERR_ARG;
    auto c = std::make_unique<es_ctx>();
    es_status st = guarded(c.get(), [&] {
        c->cfg = *cfg;
        c->cfg.group_starts = nullptr;  // replaced by a private copy below
        if (cfg->draft.vocab != cfg->base.vocab)
            arg_fail(ES_ERR_ARG, "draft and base vocabularies differ (%d vs %d): token ids must be shared",
                     cfg->draft.vocab, cfg->base.vocab);
        if (cfg->max_batch < 1 || cfg->max_batch > 64) arg_fail(ES_ERR_ARG, "max_batch must be 1..64");
        if (cfg->max_gamma < 1 || cfg->max_gamma > 16) arg_fail(ES_ERR_ARG, "max_gamma must be 1..16");
        if (cfg->max_seq < 8) arg_fail(ES_ERR_ARG, "max_seq must be >= 8");
        if (cfg->parallel_mode != ES_ATTN_ONLY && cfg->parallel_mode != ES_FULL_LAYER)
            arg_fail(ES_ERR_ARG, "parallel_mode must be ES_ATTN_ONLY or ES_FULL_LAYER");
        if (cfg->group_starts) {
            if (cfg->n_groups < 1 || cfg->group_starts[0] != 0) arg_fail(ES_ERR_ARG, "group_starts must begin at 0");
            for (int i = 1; i < cfg->n_groups; ++i)
                if (cfg->group_starts[i] <= cfg->group_starts[i - 1] || cfg->group_starts[i] >= cfg->draft.n_layers)
                    arg_fail(ES_ERR_ARG, "group_starts must increase within 0..n_layers-1");
            for (int i = 0; i < cfg->n_groups; ++i) {
                const int e = i + 1 < cfg->n_groups ? cfg->group_starts[i + 1] : cfg->draft.n_layers;
                if (e - cfg->group_starts[i] > MAX_GROUP) arg_fail(ES_ERR_ARG, "layer set larger than %d", MAX_GROUP);
            }
            // keep a private copy of the list (the accept kernel's greedy flag
            // and every other per-run choice are read at run time)
            int* gs = new int[cfg->n_groups];
            memcpy(gs, cfg->group_starts, sizeof(int) * cfg->n_groups);
            c->cfg.group_starts = gs;
        }
        CK(cudaGetDevice(&c->dev));
        CK(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->dev));
        // CUDA graphs cannot be captured on the legacy default stream: without
        // a caller stream, work goes to a private stream that still orders
        // with the legacy stream (created blocking)
        c->st = (cudaStream_t)cfg->cuda_stream;
        if (!c->st) {
            CK(cudaStreamCreate(&c->st));
            c->own_stream = true;
        }
        setup_model(c.get(), c->md, cfg->draft, draft, MAX_GROUP, "draft");
        setup_model(c.get(), c->mb, cfg->base, base, 1, "base");
        const int Bm = cfg->max_batch, S = cfg->max_seq, G = cfg->max_gamma, V = cfg->draft.vocab;
        c->tokens = c->dalloc<int>((size_t)Bm * S);
        c->n_commit = c->dalloc<int>(Bm);
        c->n_limit = c->dalloc<int>(Bm);
        c->phase = c->dalloc<int64_t>(Bm);
        c->dtok = c->dalloc<int>((size_t)Bm * G);
        c->n_acc = c->dalloc<int>(Bm);
        c->out_tok = c->dalloc<int>((size_t)Bm * (G + 1));
        c->q_logits = c->dalloc<float>((size_t)Bm * G * V);
        c->q_probs = c->dalloc<float>((size_t)Bm * G * V);
        c->p_logits = c->dalloc<float>((size_t)Bm * (G + 1) * V);
        c->p_probs = c->dalloc<float>((size_t)Bm * (G + 1) * V);
        c->prm = c->dalloc<RunParams>(1);
        c->status = c->dalloc<int>(1);
        c->arena_cap = 1 << 14;
        c->arena = c->dalloc<GemvOp>(c->arena_cap);
        CK(cudaMallocHost(&c->h_prm, sizeof(RunParams)));
        CK(cudaMallocHost(&c->h_small, sizeof(int) * (64 + 64 * 17 + 64)));
        CK(cudaDeviceSynchronize());
    });
    if (st != ES_OK) {
        fprintf(stderr, "easyspec_init: %s\n", c->err.c_str());
        easyspec_destroy(c.release());
        return st;
    }
    *out = c.release();
    return ES_OK;
}

es_status easyspec_prefill(es_ctx* c, const int32_t* prompts, int B, int P) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] { do_prefill(c, prompts, B, P); });
}

es_status calibrate_kv(es_ctx* c, int gamma, float temperature, uint64_t seed) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] {
        check_phase_args(c, gamma, temperature);
        set_params(c, temperature, seed);
        run_part(c, 2, gamma, 1);
        CK(cudaStreamSynchronize(c->st));
        check_status(c);
        c->calibrated = true; c->drafted = false;
        c->cur_gamma = gamma; c->cur_T = temperature; c->cur_seed = seed;
    });
}

es_status draft_step(es_ctx* c, int k, int gamma, float temperature, uint64_t seed, int32_t* draft_out) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] {
        const int kk = resolve_k(c, k);
        check_phase_args(c, gamma, temperature);
        if (c->calibrated && (gamma != c->cur_gamma || temperature != c->cur_T || seed != c->cur_seed))
            arg_fail(ES_ERR_STATE, "draft_step arguments differ from the preceding calibrate_kv");
        set_params(c, temperature, seed);
        run_part(c, c->calibrated ? 3 : 0, gamma, kk);
        if (draft_out) {
            std::vector<int> dt((size_t)c->B * c->cfg.max_gamma);
            CK(cudaMemcpyAsync(dt.data(), c->dtok, dt.size() * sizeof(int), cudaMemcpyDeviceToHost, c->st));
            CK(cudaStreamSynchronize(c->st));
            for (int b = 0; b < c->B; ++b)
                for (int i = 0; i < gamma; ++i) draft_out[b * gamma + i] = dt[(size_t)b * c->cfg.max_gamma + i];
        } else {
            CK(cudaStreamSynchronize(c->st));
        }
        check_status(c);
        c->calibrated = false; c->drafted = true;
        c->cur_gamma = gamma; c->cur_T = temperature; c->cur_seed = seed; c->cur_k = kk;
    });
}

es_status verify_step(es_ctx* c, float temperature, uint64_t seed, int32_t* n_accepted, int32_t* tokens_out) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] {
        if (!c->drafted) arg_fail(ES_ERR_STATE, "verify_step needs a preceding draft_step");
        if (temperature != c->cur_T || seed != c->cur_seed)
            arg_fail(ES_ERR_STATE, "verify_step temperature/seed differ from draft_step");
        run_part(c, 1, c->cur_gamma, c->cur_k);
        read_phase_result(c, c->cur_gamma, n_accepted, tokens_out);
        c->drafted = false;
    });
}

es_status generate(es_ctx* c, const int32_t* prompts, int B, int P, int max_new, int gamma, int k,
                   float temperature, uint64_t seed, int32_t* out, es_stats* stats) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] {
        if (!out || max_new < 1) arg_fail(ES_ERR_ARG, "generate: need out and max_new >= 1");
        if (gamma < 1 || gamma > c->cfg.max_gamma) arg_fail(ES_ERR_ARG, "gamma=%d outside 1..max_gamma", gamma);
        if ((int64_t)P + max_new + 2 * gamma + 2 > c->cfg.max_seq)
            arg_fail(ES_ERR_CAPACITY, "P + max_new + 2*gamma + 2 exceeds max_seq=%d", c->cfg.max_seq);
        resolve_k(c, k);
        auto t0 = std::chrono::steady_clock::now();
        do_prefill(c, prompts, B, P);
        auto t1 = std::chrono::steady_clock::now();
        es_stats s = do_decode(c, max_new, gamma, k, temperature, seed);
        // the new tokens: positions P .. P+max_new-1 of every sequence
        for (int b = 0; b < B; ++b)
            CK(cudaMemcpyAsync(out + (size_t)b * max_new, c->tokens + (size_t)b * c->cfg.max_seq + P,
                               max_new * sizeof(int), cudaMemcpyDeviceToHost, c->st));
        CK(cudaStreamSynchronize(c->st));
        s.prefill_ms = std::chrono::duration<double, std::milli>(t1 - t0).count();
        if (stats) *stats = s;
    });
}

es_status es_decode(es_ctx* c, int max_new, int gamma, int k, float temperature, uint64_t seed,
                    es_stats* stats) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] {
        if (max_new < 1) arg_fail(ES_ERR_ARG, "es_decode: max_new >= 1");
        if (c->B < 1) arg_fail(ES_ERR_STATE, "es_decode: no prompts loaded");
        if (gamma < 1 || gamma > c->cfg.max_gamma) arg_fail(ES_ERR_ARG, "gamma=%d outside 1..max_gamma", gamma);
        for (int b = 0; b < c->B; ++b)
            if ((int64_t)c->n_host[b] + max_new + 2 * gamma + 2 > c->cfg.max_seq)
                arg_fail(ES_ERR_CAPACITY, "sequence %d: n + max_new + 2*gamma + 2 exceeds max_seq", b);
        es_stats s = do_decode(c, max_new, gamma, k, temperature, seed);
        if (stats) *stats = s;
    });
}

es_status es_profile(es_ctx* c, int on) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] {
        CK(cudaStreamSynchronize(c->st));
        if (c->profiling) prof_collect(c);
        c->profiling = on != 0;
        c->prof.clear();
    });
}

es_status es_profile_read(es_ctx* c, int idx, char* name, int name_cap, double* ms,
                          int64_t* launches, double* bytes) {
    if (!c || !name || name_cap < 1) return ES_ERR_ARG;
    return guarded(c, [&] {
        if (c->profiling) {
            CK(cudaStreamSynchronize(c->st));
            prof_collect(c);
        }
        if (idx < 0 || idx >= (int)c->prof.size()) arg_fail(ES_ERR_ARG, "no profile entry %d", idx);
        auto it = c->prof.begin();
        std::advance(it, idx);
        snprintf(name, name_cap, "%s", it->first.c_str());
        if (ms) *ms = it->second.ms;
        if (launches) *launches = it->second.launches;
        if (bytes) *bytes = it->second.bytes;
    });
}

es_status es_accept_resample(const float* p, const float* q, const int32_t* d, const uint64_t* u,
                             int B, int gamma, int V, int greedy, int32_t* n_acc, int32_t* tok,
                             void* stream) {
    if (!p || !q || !d || !n_acc || !tok || B < 1 || gamma < 1 || gamma > 16 || V < 1) return ES_ERR_ARG;
    if (!greedy && !u) return ES_ERR_ARG;
    AcceptArgs a;
    memset(&a, 0, sizeof a);
    a.p = p; a.q = q; a.d = d; a.gmax = gamma; a.gamma = gamma; a.V = V; a.greedy = greedy ? 1 : 0;
    a.u_explicit = u; a.n_acc = n_acc; a.out_tok = tok;
    cudaStream_t st = (cudaStream_t)stream;
    accept_kernel<<<B, 1024, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return ES_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return ES_ERR_CUDA;
    return ES_OK;
}

es_status es_sample(const float* w, const uint64_t* u, int B, int V, int32_t* idx, void* stream) {
    if (!w || !u || !idx || B < 1 || V < 1) return ES_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    sample_rows_kernel<<<B, 1024, 0, st>>>(w, u, V, idx);
    if (cudaGetLastError() != cudaSuccess) return ES_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return ES_ERR_CUDA;
    return ES_OK;
}

es_status es_read_kv(es_ctx* c, int which, int layer, int seq, int n, float* k_out, float* v_out) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] {
        Model& m = which ? c->mb : c->md;
        if (layer < 0 || layer >= m.L || seq < 0 || seq >= c->cfg.max_batch || n < 0 || n > c->cfg.max_seq)
            arg_fail(ES_ERR_ARG, "es_read_kv: index out of range");
        std::vector<int> pt((size_t)c->cfg.max_batch * m.g.pages_per_seq);
        CK(cudaMemcpy(pt.data(), m.g.page_table, pt.size() * sizeof(int), cudaMemcpyDeviceToHost));
        std::vector<char> buf((size_t)PAGE * m.hd * m.esz);
        for (int kv = 0; kv < 2; ++kv) {
            float* dst = kv ? v_out : k_out;
            if (!dst) continue;
            for (int h = 0; h < m.Hkv; ++h)
                for (int p0 = 0; p0 < n; p0 += PAGE) {
                    const int page = pt[(size_t)seq * m.g.pages_per_seq + p0 / PAGE];
                    const size_t off = ((((size_t)page * m.L + layer) * 2 + kv) * m.Hkv + h) * PAGE * m.hd;
                    CK(cudaMemcpy(buf.data(), (char*)m.g.kv + off * m.esz, buf.size(), cudaMemcpyDeviceToHost));
                    for (int s = 0; s < PAGE && p0 + s < n; ++s)
                        for (int e = 0; e < m.hd; ++e) {
                            float v;
                            if (m.esz == 4) memcpy(&v, buf.data() + ((size_t)s * m.hd + e) * 4, 4);
                            else {
                                uint16_t b16;
                                memcpy(&b16, buf.data() + ((size_t)s * m.hd + e) * 2, 2);
                                uint32_t u32 = (uint32_t)b16 << 16;
                                memcpy(&v, &u32, 4);
                            }
                            dst[((size_t)(p0 + s) * m.Hkv + h) * m.hd + e] = v;
                        }
                }
        }
    });
}

es_status es_read_dist(es_ctx* c, int which, float* out) {
    if (!c || !out) return ES_ERR_ARG;
    return guarded(c, [&] {
        const int g = c->cur_gamma, B = c->B, V = c->md.V;
        if (g < 1 || B < 1) arg_fail(ES_ERR_STATE, "no phase has run");
        const float* src = which == 0 ? c->q_probs : which == 1 ? c->p_probs : which == 2 ? c->q_logits : c->p_logits;
        if (which < 0 || which > 3) arg_fail(ES_ERR_ARG, "which must be 0..3");
        const size_t rows = (size_t)B * (which == 0 || which == 2 ? g : g + 1);
        CK(cudaStreamSynchronize(c->st));
        CK(cudaMemcpy(out, src, rows * V * sizeof(float), cudaMemcpyDeviceToHost));
    });
}

es_status es_read_tokens(es_ctx* c, int seq, int32_t* out, int cap, int* n_committed) {
    if (!c || !n_committed) return ES_ERR_ARG;
    return guarded(c, [&] {
        if (seq < 0 || seq >= c->B) arg_fail(ES_ERR_ARG, "seq out of range");
        CK(cudaStreamSynchronize(c->st));
        int n = 0;
        CK(cudaMemcpy(&n, c->n_commit + seq, sizeof(int), cudaMemcpyDeviceToHost));
        *n_committed = n;
        if (out) CK(cudaMemcpy(out, c->tokens + (size_t)seq * c->cfg.max_seq, std::min(n, cap) * sizeof(int), cudaMemcpyDeviceToHost));
    });
}

const char* easyspec_last_error(const es_ctx* c) { return c ? c->err.c_str() : "null context"; }

void easyspec_destroy(es_ctx* c) {
    if (!c) return;
    cudaStreamSynchronize(c->st);
    for (auto& kv : c->graphs)
        if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    for (void* p : c->allocs) cudaFree(p);
    if (c->h_prm) cudaFreeHost(c->h_prm);
    if (c->h_small) cudaFreeHost(c->h_small);
    if (c->cfg.group_starts) delete[] c->cfg.group_starts;
    if (c->own_stream) cudaStreamDestroy(c->st);
    delete c;
}

}  // extern "C"
