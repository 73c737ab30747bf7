// libeasyspec: host runtime and C ABI for EasySpec layer-parallel
// speculative decoding on one B300.  See include/easyspec.h for the contract.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <set>
#include <string>
#include <type_traits>
#include <tuple>
#include <vector>

#include "../../include/easyspec.h"
#include "kernels.cuh"
#include "tcgemm.cuh"
#include "planes.cuh"
#include "attn_tc.cuh"

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

// One kernel launch of a planned forward pass.
enum RecKind { R_GV = 0, R_GEMM = 1, R_NORM = 2, R_ATTN = 3, R_TC = 4, R_NPL = 5 };
struct Rec {
    int kind = R_GV;
    const char* name = "";
    double bytes = 0;          // algorithmic bytes (weights + activations), 0 if not modelled
    const GvLaunch* gv = nullptr;           // device copy (after upload)
    std::shared_ptr<GvLaunch> host;         // host copy while the plan is built
    std::shared_ptr<TcLaunch> tc_host;      // many-row bf16 pass: tensor-core descriptor on the host
    const TcLaunch* tc = nullptr;           // its device copy
    SplitArgs split{};                      // the pass's activation planes
    int split_grid = 0, cluster = 1;        // split_grid 0: planes written by the launch before
    int attn_tc = 0;                        // attention: head size of the grouped-row kernel, or 0
    NormPlanesArgs npl{};                   // normalised planes for a tensor-core pass
    bool bf16 = false;                      // weights are bf16
    int nw = 8;                             // tensor-core weight pass: warps per CTA (8 or 16)
    int grid = 0, smem = 0, M = 0, ntiles64 = 0;
    NormArgs norm{};
    AttnArgs attn{};
    dim3 g3;
};

// A planned forward pass: the embedding kernel's normalisation jobs for the
// first weight pass, then the launches.
struct Plan {
    GvPost first{};
    std::vector<Rec> recs;
};

struct ProfRec { const char* name; double bytes; cudaEvent_t a, b; };
struct ProfAgg { double ms = 0, bytes = 0; int64_t launches = 0; };

struct Model {
    int L = 0, d = 0, H = 0, Hkv = 0, hd = 0, F = 0, V = 0, qd = 0, kvd = 0, dtype = 0;
    float theta = 0, eps = 0;
    size_t esz = 4;
    const char* tag = "";  // "draft" / "base": prefix of the profiling labels
    const void *embed = nullptr, *lm = nullptr, *fnorm = nullptr;
    std::vector<Layer> ly;
    KVGeom g{};
    float* rope = nullptr;
    float* ssp = nullptr;  // sums of squares for the next normalisation (bf16 fast path)
    int slots = 1, Mw = 0, nsplit = 0;
    float *h = nullptr, *xf = nullptr, *part = nullptr, *rinv = nullptr;
    std::vector<float*> xb, mb, q, k, v, a, s, A;
    int *row_pos = nullptr, *row_seq = nullptr, *row_tok = nullptr, *row_base = nullptr;
};

struct Graph { cudaGraphExec_t exec = nullptr; int64_t kernels = 0; };

}  // namespace

struct es_ctx {
    es_config cfg{};
    Model md, mb;
    // many-row bf16 passes (prompt prefill, batches past 8 rows): the
    // tcgen05 kernel on hi/lo activation planes
    bf16* tc_x = nullptr;          // planes of a pass's sources, [2][M][K] each
    size_t tc_x_elems = 0;
    cudaStream_t st = nullptr;
    bool own_stream = false;
    int dev = 0, num_sms = 148;
    bool poisoned = false;
    std::string err;
    std::vector<void*> allocs;

    // device state
    int* tokens = nullptr;   // [Bmax][max_seq]
    int* n_commit = nullptr; // [Bmax]
    int* kv_from = nullptr;  // [Bmax] first committed position without a draft K/V entry
    int* n_limit = nullptr;  // [Bmax] commit limit (generate: P + max_new)
    int64_t* phase = nullptr;
    int* dtok = nullptr;     // [Bmax][gmax]
    int* n_acc = nullptr;    // [Bmax]
    int* out_tok = nullptr;  // [Bmax][gmax+1]
    float *q_logits = nullptr, *q_probs = nullptr, *p_logits = nullptr, *p_probs = nullptr;
    RunParams* prm = nullptr;
    int* status = nullptr;
    // scratch of the split kernels (partials and arrival counters)
    float* gv_scratch = nullptr;
    int* gv_counters = nullptr;
    int* gv_done = nullptr;
    int* att_counters = nullptr;
    float* sm_part = nullptr;
    unsigned long long* sm_mass = nullptr;
    int* sm_counters = nullptr;
    int sm_rows_cap = 0, sm_nb_cap = 0;
    // pinned host mirrors
    RunParams* h_prm = nullptr;
    int* h_small = nullptr;  // n_acc | out_tok | n_commit | status

    // launch descriptors (GEMV launches) live in a device arena
    char* arena = nullptr;
    size_t arena_cap = 0, arena_used = 0;

    // session state
    int B = 0;
    std::vector<int> n_host;  // committed count per sequence (host copy)
    int cur_gamma = 0, cur_k = -1;
    bool calibrated = false, drafted = false;
    bool calib_off = false;  // calibration ablation
    float cur_T = 0.f;
    uint64_t cur_seed = 0;

    // launch accounting and optional per-launch event timing
    int64_t launches = 0;
    bool profiling = false;   // per-kernel timing: eager launches bracketed by events
    bool part_timing = false;  // per-part timing: graph launches bracketed by events
    std::vector<ProfRec> prof_pending;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> prof_pool;
    size_t prof_pool_used = 0;
    std::map<std::string, ProfAgg> prof;

    // planned forwards: key (model 0 draft / 1 base, set key, rows)
    std::map<std::tuple<int, int, int, int, int, int, int>, Plan> plans;
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
void launch_cl(es_ctx* c, const char* name, double bytes, int cluster, void (*kern)(KArgs...), dim3 grid,
               dim3 block, size_t smem, Args... args) {
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
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c->st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)cluster;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    CK(cudaLaunchKernelEx(&cfg, kern, args...));
    c->launches++;
    if (c->profiling) {
        CK(cudaEventRecord(ev1, c->st));
        c->prof_pending.push_back(ProfRec{name, bytes, ev0, ev1});
    }
}

template <typename... KArgs, typename... Args>
void launch(es_ctx* c, const char* name, double bytes, void (*kern)(KArgs...), dim3 grid, dim3 block,
            size_t smem, Args... args) {
    launch_cl(c, name, bytes, 1, kern, grid, block, smem, args...);
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
    if (s.n_layers < 1 || s.d < 8 || s.n_heads < 1 || s.n_kv_heads < 1 || s.head_dim < 8 ||
        s.ffn < 8 || s.vocab < 2)
        arg_fail(ES_ERR_ARG, "%s: non-positive shape field", which);
    if (s.d % 8 || s.ffn % 8 || (s.n_heads * s.head_dim) % 8)
        arg_fail(ES_ERR_ARG, "%s: d, ffn and n_heads*head_dim must be multiples of 8", which);
    if (s.head_dim % 8 || s.head_dim > 256)
        arg_fail(ES_ERR_ARG, "%s: head_dim must be a multiple of 8 and <= 256", which);
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
    m.tag = which;
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
    // workspace rows: decode batches and prefill chunks.  A prompt is
    // prefilled in chunks of Mw / B positions per sequence, each a full pass
    // over the weights: 1024 rows keep the tensor-core passes' row chunks
    // (256 rows each) several per tile, and stream the weights a quarter as
    // often as 256 rows did (long-context pair, batch 16, 4096-token
    // prompts: prefill 5.8 -> 3.9 s).
    m.Mw = std::max(Bmax * (c->cfg.max_gamma + 1), 1024);
    m.slots = slots;
    const size_t Mw = m.Mw;
    m.h = c->dalloc<float>(Mw * m.d);
    m.xf = c->dalloc<float>(Mw * m.d);
    m.rinv = c->dalloc<float>(Mw);
    // sums of squares per 16-column tile of h (tensor-core launches); a
    // 128-row block may end up to 7 tiles past d
    m.ssp = c->dalloc<float>((size_t)((m.d + GVM_ROWS - 1) / GVM_ROWS + 8) * Mw);
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
    m.row_base = c->dalloc<int>(Mw);
}

// Profiling label "<model>.<step>", interned so records can keep a pointer.
const char* label(const Model& m, const char* step) {
    static std::mutex mu;
    static std::set<std::string> names;
    std::lock_guard<std::mutex> lock(mu);
    return names.insert(std::string(m.tag) + "." + step).first->c_str();
}

// ------------------------------------------------------------------ GEMV launch building
// Collects the ops and activation sources of one weight-streaming launch.
struct GvBuild {
    std::shared_ptr<GvLaunch> L;
    size_t esz;
    int xfloats = 0;
    bool simt;  // many-row launch (SIMT GEMM): every source read from global memory
    bool mma;   // bf16 weights, few rows: tensor-core kernel (16-row tiles, hi/lo planes)
    GvBuild(int M, size_t esz_, bool simt_)
        : L(std::make_shared<GvLaunch>()), esz(esz_), simt(simt_), mma(esz_ == 2 && !simt_) {
        memset(L.get(), 0, sizeof(GvLaunch));
        L->M = M;
    }
    // An activation source: rows r*rs + ro of src (leading dimension ld).
    // SIMT-FMA kernel: staged in shared memory while room is left, else read
    // from global.  Tensor-core kernel: each CTA stages the windows it needs
    // while its budget lasts (decided on the device).
    int source(const float* src, int K, int ld, int rs = 1, int ro = 0) {
        if (L->nxs >= GV_MAX_XS) arg_fail(ES_ERR_ARG, "too many activation sources in one launch");
        const int need = L->M * K;
        int off = -1;
        if (mma) off = 0;
        else if (!simt && xfloats + need <= GV_XSMEM_MAX) { off = xfloats; xfloats += (need + 3) & ~3; }
        GvXSrc& x = L->xs[L->nxs];
        x.src = src; x.K = K; x.ld = ld; x.row_stride = rs; x.row_off = ro; x.smem_off = off; x.kind = XS_RAW;
        return L->nxs++;
    }
    // A normalised source (h + add) * rinv * gain, rows r*rs + ro of h; -1
    // when it does not fit in shared memory (the caller normalises it first).
    int norm_source(const float* h, const float* add, const void* gain, const float* rinv, int K, int rs, int ro) {
        if (simt || (!mma && xfloats + L->M * K > GV_XSMEM_MAX)) return -1;
        const int i = source(h, K, K, rs, ro);
        GvXSrc& x = L->xs[i];
        x.kind = XS_NORM; x.add = add; x.gain = gain; x.rinv = rinv;
        return i;
    }
    int op(int N, float* y, int ldy, int epi, const float* add = nullptr) {
        if (L->nops >= GV_MAX_OPS) arg_fail(ES_ERR_ARG, "too many ops in one launch");
        GvOp& o = L->ops[L->nops];
        o.N = N; o.y = y; o.ldy = ldy; o.epi = epi; o.add = add;
        o.seg0 = 0; o.nseg = 0;
        return L->nops++;
    }
    // segments of an op must be added right after the op, in order
    void seg(int oi, const void* W, int K, int xs, int set) {
        GvOp& o = L->ops[oi];
        int nsegs = 0;
        for (int i = 0; i < L->nops; ++i) nsegs += L->ops[i].nseg;
        if (o.nseg == 0) o.seg0 = nsegs;
        if (o.seg0 + o.nseg != nsegs) arg_fail(ES_ERR_ARG, "internal: segments out of order");
        if (o.nseg >= GV_MAX_SEG || nsegs >= GV_MAX_SEGS) arg_fail(ES_ERR_ARG, "too many K-concatenated segments");
        if (xs < 0 || L->xs[xs].K != K) arg_fail(ES_ERR_ARG, "segment / source width mismatch");
        if (mma && K % 8) arg_fail(ES_ERR_ARG, "bf16 weight rows must be a multiple of 8 elements (K = %d)", K);
        // an op's sums are scaled by the row's 1/rms when its sources are
        // normalised: all of its segments must then read normalised sources
        if (mma && o.nseg > 0) {
            const GvXSrc& x0 = L->xs[L->segs[o.seg0].xs];
            const GvXSrc& x1 = L->xs[xs];
            if ((x0.kind == XS_NORM) != (x1.kind == XS_NORM) || x0.rinv != x1.rinv)
                arg_fail(ES_ERR_ARG, "internal: an op mixes normalised and raw sources");
        }
        GvSeg& s = L->segs[nsegs];
        s.W = W; s.K = K; s.xs = xs; s.set = set;
        o.nseg++;
    }
};

// Stage bookkeeping; the descriptor stays on the host until upload_plan().
Rec finish_gv(es_ctx* c, GvBuild& b, const char* name) {
    GvLaunch& L = *b.L;
    // chunk columns and tile rows: 512-byte x 32-row stages (SIMT-FMA kernel)
    // or 128-column x (16 x warps)-row stages (tensor-core kernel)
    const int SC = b.mma ? GVM_COLS : GV_ROW_BYTES / (int)b.esz;
    double wbytes = 0, rowbytes = 0;
    for (int i = 0; i < L.nops; ++i) {
        GvOp& o = L.ops[i];
        o.spt = 0;
        for (int s = 0; s < o.nseg; ++s) {
            GvSeg& sg = L.segs[o.seg0 + s];
            sg.nck = (sg.K + SC - 1) / SC;
            o.spt += sg.nck;
            wbytes += (double)o.N * sg.K * b.esz;
        }
        rowbytes += (double)o.N * 4.0 * (o.epi == GEPI_STORE || o.epi == GEPI_SWIGLU ? 1 : o.epi == GEPI_ACC ? 2 : 3);
    }
    for (int i = 0; i < L.nxs; ++i) rowbytes += (double)L.xs[i].K * 4.0;
    // tiles and stages for a tile height; the CTA range per `ctas`
    auto layout = [&](int RT, int ctas) {
        int t = 0, st = 0, t64 = 0;
        for (int i = 0; i < L.nops; ++i) {
            GvOp& o = L.ops[i];
            o.ntiles = (o.N + RT - 1) / RT;
            o.tile0 = t; o.stage0 = st; o.tile64_0 = t64;
            t += o.ntiles; st += o.ntiles * o.spt; t64 += (o.N + GB - 1) / GB;
        }
        L.ntiles = t; L.nstages = st; L.ntiles64 = t64;
        L.q = std::max(1, (st + ctas - 1) / ctas);
        if (t > GV_COUNTERS) arg_fail(ES_ERR_ARG, "launch has %d tiles (> %d)", t, GV_COUNTERS);
    };
    // tensor-core kernel: the largest staged window set of any CTA within
    // `budget` words (the device repeats this computation with the result
    // as its budget); false if some window would go through L2
    auto windows_fit = [&](int budget, int* need) {
        const int grid = (L.nstages + L.q - 1) / L.q;
        bool all = true;
        *need = 0;
        for (int cta = 0; cta < grid; ++cta) {
            GvmWin win[GVM_NWIN];
            int items, used;
            const int n = gvm_windows(L, cta * L.q, std::min(L.nstages, (cta + 1) * L.q), win, budget, &items,
                                      &used);
            *need = std::max(*need, used);
            if (n == GVM_NWIN) all = false;  // windows may have been dropped
            for (int i = 0; i < n; ++i) all = all && win[i].off >= 0;
        }
        return all;
    };
    Rec r;
    r.nw = GV_WARPS;
    if (b.mma) {
        int need = 0;
        layout(GVM_BLOCK, c->num_sms * GV_CTAS_PER_SM);
        if (!windows_fit(GV_XSMEM_MAX, &need)) {
            // wide activations: one 16-warp CTA per SM shares a window twice
            // as large, if that makes every window fit
            int need_w = 0;
            layout(GVM_WIDE_WARPS * GVM_ROWS, c->num_sms);
            if (windows_fit(GVM_WIDE_XSMEM, &need_w)) {
                r.nw = GVM_WIDE_WARPS;
                need = need_w;
            } else {
                layout(GVM_BLOCK, c->num_sms * GV_CTAS_PER_SM);
                windows_fit(GV_XSMEM_MAX, &need);
            }
        }
        L.x_smem_floats = need;
    } else {
        layout(GV_RT, c->num_sms * GV_CTAS_PER_SM);
        L.x_smem_floats = b.xfloats;
    }
    int items = 0;  // staging items (4 columns of one row) of the shared-memory sources
    for (int i = 0; i < L.nxs; ++i) {
        L.xs[i].item0 = items;
        if (!b.mma && L.xs[i].smem_off >= 0) items += L.M * (L.xs[i].K / 4);
    }
    L.x_items = items;
    r.kind = b.simt ? R_GEMM : R_GV;
    r.name = name;
    r.M = L.M;
    r.grid = (L.nstages + L.q - 1) / L.q;
    r.smem = L.x_smem_floats * (int)sizeof(float);
    r.ntiles64 = L.ntiles64;
    r.bytes = wbytes + L.M * rowbytes;
    r.host = b.L;
    return r;
}

// ------------------------------------------------------------------ many-row tensor-core passes
// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        CK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q));
        if (q != cudaDriverEntryPointSuccess || !p) arg_fail(ES_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
        fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// Tiled bf16 tensor map with the 128-byte swizzle and zero fill outside the
// tensor: rank 2 or 3, dims[0] innermost (elements), strides in bytes of
// dims 1.., box in elements.
void encode_map(TcMap* out, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                const uint32_t* box) {
    static_assert(sizeof(TcMap) == sizeof(CUtensorMap), "tensor map size");
    cuuint64_t gd[3], gs[2];
    cuuint32_t bx[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; }
    for (int i = 0; i + 1 < rank; ++i) gs[i] = strides[i];
    const CUresult r = tensor_map_encoder()(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                            (cuuint32_t)rank, const_cast<void*>(base), gd, gs, bx, es,
                                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) arg_fail(ES_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
}



// A many-row bf16 weight pass: the ops of `b` become one tensor-core launch
// (tc_gemm_kernel) preceded by one launch that writes the hi/lo planes of
// its activation sources.
// Sources whose planes their producer writes directly skip the split:
// normalised inputs made by `pre` (the RMSNorm launch right before the
// pass), and SwiGLU outputs of an earlier tensor-core pass in `prior` (the
// plan so far) that nothing else reads.
Rec finish_tc(es_ctx* c, GvBuild& b, const char* name, bool planes_ready = false, NormArgs* pre = nullptr,
              std::vector<Rec>* prior = nullptr) {
    const GvLaunch& G = *b.L;
    auto T = std::make_shared<TcLaunch>();
    memset(T.get(), 0, sizeof(TcLaunch));
    TcLaunch& L = *T;
    const int M = G.M;
    L.M = M;
    L.rc = (M + TC_MAXN - 1) / TC_MAXN;                       // as tc_layout sets them:
    L.npad = ((M + L.rc - 1) / L.rc + 15) / 16 * 16;          // the activation maps' box needs npad
    Rec r;
    r.kind = R_TC;
    r.name = name;
    r.M = M;
    // activation sources -> planes in tc_x, one 3-D map each: [2][M][K].
    // Consecutive tensor-core passes of a plan take alternate halves of the
    // buffer, so a pass whose epilogue writes the next pass's planes never
    // overwrites the planes it is still reading.
    SplitArgs& sa = r.split;
    memset(&sa, 0, sizeof sa);
    sa.M = M;
    int src_of_xs[GV_MAX_XS];
    for (int i = 0; i < GV_MAX_XS; ++i) src_of_xs[i] = -1;
    int ntc = 0;
    if (prior)
        for (const Rec& q : *prior) ntc += q.kind == R_TC;
    const size_t half_elems = c->tc_x_elems / 2;
    bf16* const base = c->tc_x + (ntc % 2) * half_elems;
    size_t off = 0;
    double wbytes = 0, xbytes = 0, ybytes = 0;
    for (int si = 0; si < G.nops; ++si) {
        const GvOp& o = G.ops[si];
        for (int j = 0; j < o.nseg; ++j) {
            const int xs = G.segs[o.seg0 + j].xs;
            if (src_of_xs[xs] >= 0) continue;
            const GvXSrc& x = G.xs[xs];
            if (x.kind != XS_RAW) arg_fail(ES_ERR_ARG, "internal: many-row pass with a normalised source");
            if (x.K % 8) arg_fail(ES_ERR_ARG, "bf16 weight rows must be a multiple of 8 elements (K = %d)", x.K);
            const int i = sa.nsrc++;
            if (i >= TC_MAX_SRCS) arg_fail(ES_ERR_ARG, "too many activation sources in one pass");
            src_of_xs[xs] = i;
            off = (off + 127) & ~(size_t)127;  // 256-byte aligned planes
            if (off + 2 * (size_t)M * x.K > half_elems)
                arg_fail(ES_ERR_ARG, "internal: activation planes exceed their buffer");
            sa.src[i] = x.src; sa.dst[i] = base + off; sa.ld[i] = x.ld; sa.rs[i] = x.row_stride;
            sa.ro[i] = x.row_off; sa.K[i] = x.K;
            bool ready = planes_ready;
            const bool plain_rows = x.row_stride == 1 && x.row_off == 0 && x.ld == x.K;
            if (!ready && pre && plain_rows && pre->out_ld == x.K && pre->d == x.K)
                for (int j = 0; j < pre->njobs && !ready; ++j)
                    if (pre->out[j] == x.src) {
                        pre->planes[j] = sa.dst[i];
                        pre->planes_M = M;
                        ready = true;
                    }
            if (!ready && prior && plain_rows)
                for (auto it = prior->rbegin(); it != prior->rend() && !ready; ++it) {
                    if (it->kind != R_TC || !it->tc_host) continue;
                    TcLaunch& P = *it->tc_host;
                    bool writes = false;
                    for (int oi = 0; oi < P.nops; ++oi) {
                        TcOp& o = P.ops[oi];
                        if (o.y != x.src) continue;
                        writes = true;
                        if (o.epi == GEPI_SWIGLU && o.ldy == x.K && o.N == x.K && P.M == M && !o.yp) {
                            o.yp = sa.dst[i];
                            ready = true;
                        }
                    }
                    if (writes) break;  // the most recent writer decides
                }
            sa.item0[i + 1] = sa.item0[i] + (ready ? 0 : M * (x.K / 4));
            const uint64_t dims[3] = {(uint64_t)x.K, (uint64_t)M, 2};
            const uint64_t strides[2] = {(uint64_t)x.K * 2, (uint64_t)M * x.K * 2};
            const uint32_t box[3] = {TC_BK, (uint32_t)L.npad, 2};
            encode_map(&L.maps[TC_MAX_SEGS + i], sa.dst[i], 3, dims, strides, box);
            off += 2 * (size_t)M * x.K;
            xbytes += (double)M * x.K * 4;
        }
    }
    r.split_grid = sa.item0[sa.nsrc] == 0 ? 0 : std::max(1, std::min(4 * c->num_sms, (sa.item0[sa.nsrc] + 255) / 256));
    // ops and segments (one weight map per segment)
    int nseg = 0;
    for (int oi = 0; oi < G.nops; ++oi) {
        const GvOp& go = G.ops[oi];
        TcOp& o = L.ops[oi];
        o.y = go.y; o.add = go.add; o.N = go.N; o.ldy = go.ldy; o.epi = go.epi;
        o.pair = go.epi == GEPI_SWIGLU;
        if (o.pair && (go.nseg != 2 || G.segs[go.seg0].set != 0 || G.segs[go.seg0 + 1].set != 1 ||
                       G.segs[go.seg0].xs != G.segs[go.seg0 + 1].xs))
            arg_fail(ES_ERR_ARG, "internal: a SwiGLU op needs one gate and one up segment on one source");
        o.seg0 = nseg; o.nseg = go.nseg; o.nkb = 0;
        for (int j = 0; j < go.nseg; ++j) {
            const GvSeg& g = G.segs[go.seg0 + j];
            if (!o.pair && g.set != 0) arg_fail(ES_ERR_ARG, "internal: second accumulator outside SwiGLU");
            if (nseg >= TC_MAX_SEGS) arg_fail(ES_ERR_ARG, "too many weight segments in one pass");
            TcSeg& t = L.segs[nseg];
            t.wmap = nseg; t.src = src_of_xs[g.xs]; t.K = g.K; t.nkb = (g.K + TC_BK - 1) / TC_BK;
            t.kb0 = o.pair ? 0 : o.nkb;
            if (!o.pair || j == 0) o.nkb += t.nkb;
            const uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)go.N};
            const uint64_t strides[1] = {(uint64_t)g.K * 2};
            const uint32_t box[2] = {TC_BK, TC_BM};
            encode_map(&L.maps[nseg], g.W, 2, dims, strides, box);
            wbytes += (double)go.N * g.K * 2;
            ++nseg;
        }
        ybytes += (double)M * go.N * 4 * (go.epi == GEPI_ACC ? 2 : go.epi == GEPI_ACC_ADD ? 3 : 1);
    }
    L.nops = G.nops;
    if (tc_layout(L, c->num_sms) == 0)
        arg_fail(ES_ERR_ARG, "internal: tensor-core stage of %d bytes too large", L.stage_bytes);
    r.grid = L.nclusters * L.cs;
    r.cluster = L.cs;
    r.smem = L.stages * L.stage_bytes + 1024;
    r.bytes = wbytes + xbytes + ybytes;
    r.tc_host = T;
    return r;
}

void upload_plan(es_ctx* c, Plan& p) {
    for (Rec& r : p.recs) {
        if (r.tc_host) {
            const size_t bytes = sizeof(TcLaunch);
            const size_t at = (c->arena_used + 255) & ~(size_t)255;
            if (at + bytes > c->arena_cap) arg_fail(ES_ERR_OOM, "launch descriptor arena exhausted");
            CK(cudaMemcpy(c->arena + at, r.tc_host.get(), bytes, cudaMemcpyHostToDevice));
            c->arena_used = at + bytes;
            r.tc = reinterpret_cast<const TcLaunch*>(c->arena + at);
            r.tc_host.reset();
            continue;
        }
        if (!r.host) continue;
        const size_t bytes = sizeof(GvLaunch);
        const size_t at = (c->arena_used + 255) & ~(size_t)255;
        if (at + bytes > c->arena_cap) arg_fail(ES_ERR_OOM, "launch descriptor arena exhausted");
        CK(cudaMemcpy(c->arena + at, r.host.get(), bytes, cudaMemcpyHostToDevice));
        c->arena_used = at + bytes;
        r.gv = reinterpret_cast<const GvLaunch*>(c->arena + at);
        r.host.reset();
    }
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
Rec norm_rec(const NormArgs& a, int rows) {
    Rec r;
    r.kind = R_NORM; r.name = "rmsnorm"; r.norm = a; r.M = rows;
    return r;
}

// Normalised hi/lo planes of rows r*stride + off of h (h + add written
// back first when `add` is set) for the tensor-core pass that follows; ssp
// (or nullptr) holds ss_tiles sums of squares per source row from the pass
// before, ss_ld apart.
Rec norm_planes_rec(Model& m, const float* add, const void* gain, bf16* dst, int rows, int stride, int off,
                    const float* ssp, int ss_tiles, int ss_ld) {
    Rec r;
    r.kind = R_NPL; r.name = "norm_planes"; r.M = rows;
    NormPlanesArgs& a = r.npl;
    memset(&a, 0, sizeof a);
    a.h = m.h; a.add = add; a.g = (const bf16*)gain; a.dst = dst; a.d = m.d; a.M = rows;
    a.src_stride = stride; a.src_off = off; a.eps = m.eps;
    a.ssp = ssp; a.ss_tiles = ss_tiles; a.ss_ld = ss_ld;
    // the kernel moves 4 columns per thread (16-byte rows, 8-byte planes)
    if (m.d % 4 || (uintptr_t)dst % 16 || (uintptr_t)m.h % 16 || (add && (uintptr_t)add % 16))
        arg_fail(ES_ERR_ARG, "internal: normalised planes need 4-column aligned rows");
    // without partial sums every CTA sums the whole row of h + add, which
    // the CTAs also write back: only a row without `add` may take that path
    if (add && !ssp) arg_fail(ES_ERR_ARG, "internal: normalised planes with an addend need partial sums");
    r.g3 = dim3(rows, (m.d + NPL_COLS - 1) / NPL_COLS);
    return r;
}

// Weight bytes from which a decode-size (at most 8 rows) pass runs on the
// tensor-core kernel.  Pairs: the 7B- and 70B-shaped base gate/up (272 MB,
// 940 MB) gain; the 8B-shaped draft's (235 MB) measured no faster.
constexpr double TC_DECODE_PAIR_BYTES = 256e6;
constexpr double TC_DECODE_HEAD_BYTES = 1.5e9;

// Attention of the layers l0 .. l0+n-1 over M rows, `rps` consecutive rows
// per sequence.  bf16 caches with head size 64 or 128 and several rows per
// sequence take the grouped-row tensor-core kernel when it has at least 64
// (group, kv head, page) items: with fewer (one short sequence, few kv
// heads) the one-row kernel's wider grid is faster (measured: the
// Qwen2.5-0.5B/7B-shaped pair at batch 1, 2 and 4 kv heads over 5-6 pages).
Rec attn_rec(es_ctx* c, Model& m, int l0, int n, int M, int rps) {
    if ((size_t)M * n * m.Hkv > (size_t)ATT_COUNTERS) arg_fail(ES_ERR_ARG, "attention launch too large");
    Rec r;
    r.kind = R_ATTN; r.name = "attention";
    AttnArgs& a = r.attn;
    memset(&a, 0, sizeof a);
    a.g = m.g; a.rope = m.rope; a.H = m.H; a.M = M; a.nl = n; a.nsplit = m.nsplit;
    for (int j = 0; j < n; ++j) {
        a.layer[j] = l0 + j;
        a.q[j] = m.q[j]; a.k[j] = m.k[j]; a.v[j] = m.v[j]; a.out[j] = m.a[j];
    }
    a.part = m.part; a.counters = c->att_counters;
    a.row_pos = m.row_pos; a.row_seq = m.row_seq; a.row_base = m.row_base;
    r.g3 = dim3(M, n * m.Hkv, m.nsplit);
    r.bf16 = m.dtype == ES_DTYPE_BF16;
    r.smem = (int)attn_smem_bytes(m.H / m.Hkv, m.hd, m.nsplit);
    r.M = M;
    // rows laid out as M / rps sequences of rps rows: the kernels take row m's
    // sequence to be m / rps when they look up its first page (an index into
    // the max_batch sequences' page table)
    a.rps = rps >= 1 && M % rps == 0 && M / rps <= c->cfg.max_batch ? rps : 0;
    const int G = m.H / m.Hkv;
    const int rg = std::max(1, ATC_QV / G);
    const int groups = a.rps ? (M / rps) * ((rps + rg - 1) / rg) * n * m.Hkv : 0;
    if (r.bf16 && a.rps >= 2 && (m.hd == 64 || m.hd == 128) && groups * m.nsplit >= 64) {
        a.rg = rg;
        // pages per CTA: about four CTAs per SM over the cache's pages, and at
        // most 256 chunks (the merge kernel's weight buffer)
        a.ppc = std::max(1, std::min(m.nsplit, groups * m.nsplit / (4 * c->num_sms)));
        a.ppc = std::max(a.ppc, (m.nsplit + 255) / 256);
        r.attn_tc = m.hd;
        r.g3 = dim3((M / rps) * ((rps + a.rg - 1) / a.rg), n * m.Hkv, (m.nsplit + a.ppc - 1) / a.ppc);
        r.smem = (int)attn_tc_smem_bytes(m.hd);
    }
    if (r.smem > 200 * 1024) arg_fail(ES_ERR_ARG, "attention needs %d bytes of shared memory (max_seq too large)", r.smem);
    return r;
}

// Output head of a forward pass: logits of rows r*stride + off of h into
// y + r*ldy.
struct HeadSpec { int rows = 0, stride = 1, off = 0, ldy = 0; float* y = nullptr; };

// Plan of one forward pass over M rows for the layer sets `groups` (sets of
// one layer are exact layers), followed by the output head when
// head.rows > 0.  M <= GV_MAXM: fused weight-streaming launches; each
// launch's normalised inputs are produced by the launch before it (the
// embedding kernel for the first), RoPE and the KV append happen inside
// attention.  Larger M: explicit norm launches and the SIMT GEMM.
Plan build_forward(es_ctx* c, Model& m, const std::vector<std::vector<int>>& groups, int mode, int M, int rps,
                   const HeadSpec& head) {
    const bool fast = M <= GV_MAXM && head.rows <= GV_MAXM;
    // decode-size passes that stream faster on the tensor-core kernel than
    // on the register-fed one (measured: SwiGLU pairs of 256 MB and more,
    // output heads of 1.5 GB and more)
    const bool tc_pair = fast && m.esz == 2 && 2.0 * m.F * m.d * m.esz >= TC_DECODE_PAIR_BYTES;
    const bool tc_head = fast && m.esz == 2 && (double)m.V * m.d * m.esz >= TC_DECODE_HEAD_BYTES;
    Plan P;
    // -- fused path: attach a normalisation to the launch that runs just before
    //    its consumer
    int writer = -1;  // index in P.recs of the last weight launch (-1: embedding)
    // 1/rms of the rows the next launch normalises, computed at the end of
    // the launch before it
    // Tensor-core launches (bf16) pass sums of squares instead: the writer's
    // epilogue stores one partial per 16-column tile (the embedding kernel
    // one per row) and the consumer adds them while it stages.
    const bool ss_mode = fast && m.esz == 2;
    int ss_tiles = 0;
    auto request = [&](const float* add, int rows, int stride, int off) {
        GvPost& p = writer < 0 ? P.first : P.recs[writer].host->post;
        if (p.rows) arg_fail(ES_ERR_ARG, "internal: two normalisations after one launch");
        p.h = m.h; p.add = add; p.rinv = m.rinv; p.rows = rows; p.row_stride = stride; p.row_off = off;
        p.K = m.d; p.eps = m.eps;
        if (ss_mode) {
            p.ssp = m.ssp;
            p.op = 0;  // the writer's op 0 produces h (or, for attention-only sets, A_0)
            ss_tiles = writer < 0 ? 1 : (m.d + GVM_ROWS - 1) / GVM_ROWS;
        }
    };
    // whether the launch before can store sums of squares for the next
    // normalisation (a register-fed pass, or the embedding kernel)
    auto ss_writer = [&]() { return ss_mode && (writer < 0 || P.recs[writer].host); };
    // a normalised input of the launch being built: fused into its staging
    // when it fits, else written beforehand by a norm launch (which also
    // folds `add` into h) into `buf`
    auto norm_input = [&](GvBuild& b, NormArgs& pre, const void* gain, float* buf, const float* add,
                          int rs, int ro, bool* fused) -> int {
        if (fast) {
            const int xs = b.norm_source(m.h, add, gain, ss_mode ? m.ssp : m.rinv, m.d, rs, ro);
            if (xs >= 0) {
                if (ss_mode) {
                    GvXSrc& x = b.L->xs[xs];
                    x.ss_tiles = ss_tiles; x.ss_ld = M; x.eps = m.eps;
                }
                if (fused) *fused = true;
                return xs;
            }
        }
        if (fused) *fused = false;
        pre.add = add; pre.src_stride = rs; pre.src_off = ro;
        add_job(pre, gain, buf);
        return b.source(buf, m.d, m.d);
    };
    auto push_gv = [&](GvBuild& b, const char* name) {
        if (!fast && m.esz == 2) {
            NormArgs* pre = !P.recs.empty() && P.recs.back().kind == R_NORM ? &P.recs.back().norm : nullptr;
            Rec t = finish_tc(c, b, label(m, name), false, pre, &P.recs);
            P.recs.push_back(t);
        } else {
            P.recs.push_back(finish_gv(c, b, label(m, name)));
        }
        writer = (int)P.recs.size() - 1;
    };
    auto raw = [&](GvBuild& b, const float* p, int K) { return b.source(p, K, K); };
    for (const auto& gl : groups) {
        const int n = (int)gl.size(), l0 = gl.front();
        if (n > m.slots || n > MAX_GROUP) arg_fail(ES_ERR_ARG, "layer set larger than %d", MAX_GROUP);
        const bool fuzzy = n > 1, full = fuzzy && mode == ES_FULL_LAYER;
        // ---- wide pass: q, k, v of every layer (+ SwiGLU of every layer)
        {
            if (fast) request(nullptr, M, 1, 0);
            GvBuild b(M, m.esz, !fast);
            NormArgs pre = norm_args(m, m.h, nullptr);
            int xa[MAX_GROUP], xm[MAX_GROUP];
            for (int j = 0; j < n; ++j) xa[j] = norm_input(b, pre, m.ly[l0 + j].an, m.xb[j], nullptr, 1, 0, nullptr);
            if (full)
                for (int j = 0; j < n; ++j) xm[j] = norm_input(b, pre, m.ly[l0 + j].mn, m.mb[j], nullptr, 1, 0, nullptr);
            for (int j = 0; j < n; ++j) {
                const Layer& y = m.ly[l0 + j];
                b.seg(b.op(m.qd, m.q[j], m.qd, GEPI_STORE), y.wq, m.d, xa[j], 0);
                b.seg(b.op(m.kvd, m.k[j], m.kvd, GEPI_STORE), y.wk, m.d, xa[j], 0);
                b.seg(b.op(m.kvd, m.v[j], m.kvd, GEPI_STORE), y.wv, m.d, xa[j], 0);
            }
            if (full)
                for (int j = 0; j < n; ++j) {
                    const Layer& y = m.ly[l0 + j];
                    const int o = b.op(m.F, m.s[j], m.F, GEPI_SWIGLU);
                    b.seg(o, y.wg, m.d, xm[j], 0);
                    b.seg(o, y.wu, m.d, xm[j], 1);
                }
            if (pre.njobs) P.recs.push_back(norm_rec(pre, M));
            push_gv(b, full ? "gv_qkv_gateup" : "gv_qkv");
        }
        P.recs.push_back(attn_rec(c, m, l0, n, M, rps));
        P.recs.back().name = label(m, "attention");
        if (full) {
            // K-concatenated [Wo_1 .. Wo_n, Wdown_1 .. Wdown_n] . [a_1..a_n, s_1..s_n]
            GvBuild b(M, m.esz, !fast);
            int xa[MAX_GROUP], xs[MAX_GROUP];
            for (int j = 0; j < n; ++j) xa[j] = raw(b, m.a[j], m.qd);
            for (int j = 0; j < n; ++j) xs[j] = raw(b, m.s[j], m.F);
            const int o = b.op(m.d, m.h, m.d, GEPI_ACC);
            for (int j = 0; j < n; ++j) b.seg(o, m.ly[l0 + j].wo, m.qd, xa[j], 0);
            for (int j = 0; j < n; ++j) b.seg(o, m.ly[l0 + j].wd, m.F, xs[j], 0);
            push_gv(b, "gv_o_down_kcat");
            continue;
        }
        // output projections: an exact layer accumulates into h; an
        // attention-only set stores A_j for the sequential MLPs below
        {
            GvBuild b(M, m.esz, !fast);
            for (int j = 0; j < n; ++j) {
                const int xa = raw(b, m.a[j], m.qd);
                const int o = fuzzy ? b.op(m.d, m.A[j], m.d, GEPI_STORE) : b.op(m.d, m.h, m.d, GEPI_ACC);
                b.seg(o, m.ly[l0 + j].wo, m.qd, xa, 0);
            }
            push_gv(b, "gv_o");
        }
        for (int j = 0; j < n; ++j) {
            const Layer& y = m.ly[l0 + j];
            const float* add = fuzzy ? m.A[j] : nullptr;  // this MLP's input is h + A_j
            bool fused = false;
            if (tc_pair) {
                // a pair of this size streams faster through the tensor-core
                // pass: its normalised input goes to the pass's hi/lo planes
                // (h + A_j written back to h first)
                GvBuild b(M, m.esz, true);
                const int xm = b.source(m.mb[0], m.d, m.d);
                const int o = b.op(m.F, m.s[0], m.F, GEPI_SWIGLU);
                b.seg(o, y.wg, m.d, xm, 0);
                b.seg(o, y.wu, m.d, xm, 1);
                Rec t = finish_tc(c, b, label(m, "tc_gateup"), true, nullptr, &P.recs);
                const bool ss = ss_writer();
                if (ss) request(add, M, 1, 0);
                P.recs.push_back(norm_planes_rec(m, add, y.mn, t.split.dst[0], M, 1, 0, ss ? m.ssp : nullptr,
                                                 ss ? ss_tiles : 0, M));
                P.recs.push_back(t);
                writer = (int)P.recs.size() - 1;
            } else {
                if (fast) request(add, M, 1, 0);
                GvBuild b(M, m.esz, !fast);
                NormArgs pre = norm_args(m, m.h, nullptr);
                const int xm = norm_input(b, pre, y.mn, m.mb[0], add, 1, 0, &fused);
                const int o = b.op(m.F, m.s[0], m.F, GEPI_SWIGLU);
                b.seg(o, y.wg, m.d, xm, 0);
                b.seg(o, y.wu, m.d, xm, 1);
                if (pre.njobs) P.recs.push_back(norm_rec(pre, M));
                push_gv(b, "gv_gateup");
            }
            {
                GvBuild b(M, m.esz, !fast);
                const int xs = raw(b, m.s[0], m.F);
                // with the fused norm h does not hold A_j yet: add it here
                const int o = (add && fused) ? b.op(m.d, m.h, m.d, GEPI_ACC_ADD, add) : b.op(m.d, m.h, m.d, GEPI_ACC);
                b.seg(o, y.wd, m.F, xs, 0);
                push_gv(b, "gv_down");
            }
        }
    }
    if (head.rows > 0 && tc_head) {
        GvBuild b(head.rows, m.esz, true);
        const int xs = b.source(m.xf, m.d, m.d);
        b.seg(b.op(m.V, head.y, head.ldy, GEPI_STORE), m.lm, m.d, xs, 0);
        Rec t = finish_tc(c, b, label(m, "tc_lm_head"), true, nullptr, &P.recs);
        const bool ss = ss_writer();
        if (ss) request(nullptr, head.rows, head.stride, head.off);
        P.recs.push_back(norm_planes_rec(m, nullptr, m.fnorm, t.split.dst[0], head.rows, head.stride, head.off,
                                         ss ? m.ssp : nullptr, ss ? ss_tiles : 0, M));
        P.recs.push_back(t);
        writer = (int)P.recs.size() - 1;
    } else if (head.rows > 0) {
        if (fast) request(nullptr, head.rows, head.stride, head.off);
        GvBuild b(head.rows, m.esz, !fast);
        NormArgs pre = norm_args(m, m.h, nullptr);
        const int xs = norm_input(b, pre, m.fnorm, m.xf, nullptr, head.stride, head.off, nullptr);
        b.seg(b.op(m.V, head.y, head.ldy, GEPI_STORE), m.lm, m.d, xs, 0);
        if (pre.njobs) P.recs.push_back(norm_rec(pre, head.rows));
        push_gv(b, "gv_lm_head");
    }
    upload_plan(c, P);
    return P;
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
void run_rec(es_ctx* c, const Rec& r) {
    switch (r.kind) {
        case R_GV:
            if constexpr (std::is_same<T, bf16>::value) {
                if (r.nw == GVM_WIDE_WARPS)
                    launch(c, r.name, r.bytes, gvm_kernel<GVM_WIDE_WARPS>, dim3(r.grid), dim3(GVM_WIDE_WARPS * 32),
                           (size_t)r.smem, r.gv, c->gv_scratch, c->gv_counters, c->gv_done);
                else
                    launch(c, r.name, r.bytes, gvm_kernel<GV_WARPS>, dim3(r.grid), dim3(GV_THREADS), (size_t)r.smem,
                           r.gv, c->gv_scratch, c->gv_counters, c->gv_done);
            } else {
                switch (r.M) {
#define ES_GV_CASE(MM)                                                                              \
    case MM:                                                                                        \
        launch(c, r.name, r.bytes, gv_kernel<T, MM>, dim3(r.grid), dim3(GV_THREADS), (size_t)r.smem, \
               r.gv, c->gv_scratch, c->gv_counters, c->gv_done);                                    \
        break;
                    ES_GV_CASE(1) ES_GV_CASE(2) ES_GV_CASE(3) ES_GV_CASE(4)
                    ES_GV_CASE(5) ES_GV_CASE(6) ES_GV_CASE(7) ES_GV_CASE(8)
#undef ES_GV_CASE
                    default: arg_fail(ES_ERR_ARG, "internal: GEMV rows %d", r.M);
                }
            }
            break;
        case R_GEMM:
            launch(c, "gemm_simt", r.bytes, gemm_kernel<T>, dim3(r.ntiles64, (r.M + GB - 1) / GB),
                   dim3(256), (size_t)0, r.gv);
            break;
        case R_NPL:
            launch(c, "norm_planes", 0.0, norm_planes_kernel, r.g3, dim3(256), (size_t)0, r.npl);
            break;
        case R_TC:
            if (r.split_grid > 0)
                launch(c, "split_planes", 0.0, split_planes_kernel, dim3(r.split_grid), dim3(256), (size_t)0,
                       r.split);
            launch_cl(c, r.name, r.bytes, r.cluster, tc_gemm_kernel, dim3(r.grid), dim3(TC_THREADS),
                      (size_t)r.smem, r.tc, c->status + 1);
            break;
        case R_NORM:
            launch(c, r.name, 0.0, norm_kernel<T>, dim3(r.M), dim3(256), (size_t)0, r.norm);
            break;
        default:
            if (r.attn_tc == 64) {
                launch(c, r.name, 0.0, attn_tc_kernel<64>, r.g3, dim3(ATC_THREADS), (size_t)r.smem, r.attn);
                if (r.g3.z > 1)
                    launch(c, "attention_merge", 0.0, attn_merge_kernel<64>, dim3(r.g3.x, r.g3.y, ATC_QV), dim3(64),
                           (size_t)0, r.attn);
            } else if (r.attn_tc == 128) {
                launch(c, r.name, 0.0, attn_tc_kernel<128>, r.g3, dim3(ATC_THREADS), (size_t)r.smem, r.attn);
                if (r.g3.z > 1)
                    launch(c, "attention_merge", 0.0, attn_merge_kernel<128>, dim3(r.g3.x, r.g3.y, ATC_QV),
                           dim3(128), (size_t)0, r.attn);
            } else
                launch(c, r.name, 0.0, attn_kernel<T>, r.g3, dim3(ATT_THREADS), (size_t)r.smem, r.attn);
            break;
    }
}

EmbedArgs embed_args(es_ctx* c, Model& m, const Plan& plan, int kind, int step, int gamma, int M) {
    EmbedArgs e;
    memset(&e, 0, sizeof e);
    e.kind = kind; e.step = step; e.gamma = gamma; e.M = M;
    e.n_commit = c->n_commit; e.tokens = c->tokens; e.max_seq = c->cfg.max_seq; e.dtok = c->dtok;
    e.gmax = c->cfg.max_gamma; e.row_pos = m.row_pos; e.row_seq = m.row_seq; e.row_tok = m.row_tok;
    e.row_base = m.row_base; e.kv_from = c->kv_from; e.prm = c->prm; e.E = m.embed; e.h = m.h; e.d = m.d; e.V = m.V; e.status = c->status;
    e.post = plan.first;
    return e;
}

// Embedding of the rows described by `kind` (or by the host), then the
// planned forward (and its head, if planned).
template <typename T>
void run_forward(es_ctx* c, Model& m, const Plan& plan, int kind, int step, int gamma, int M) {
    launch(c, "prep_embed", 0.0, prep_embed_kernel<T>, dim3(M), dim3(256), (size_t)0,
           embed_args(c, m, plan, kind, step, gamma, M));
    for (const Rec& r : plan.recs) run_rec<T>(c, r);
}

// Vocabulary chunks of the softmax / draw / accept kernels: about one per SM.
void vocab_chunks(int V, int num_sms, int* chunk, int* nb) {
    *chunk = std::max(512, (V + num_sms - 1) / num_sms);
    *nb = (V + *chunk - 1) / *chunk;
}

// Softmax over rows of logits (and a draw per row when dtok is set).
void run_softmax(es_ctx* c, const float* z, float* p, int V, int rows, int per_seq, int off, int ld_rows,
                 int gamma, int* dtok) {
    SampleArgs a;
    memset(&a, 0, sizeof a);
    a.z = z; a.p = p; a.V = V; a.greedy = -1;
    vocab_chunks(V, c->num_sms, &a.chunk, &a.nb);
    a.per_seq = per_seq; a.off = off; a.ld_rows = ld_rows;
    a.prm = c->prm; a.phase = c->phase; a.gamma = gamma; a.dtok = dtok; a.gmax = c->cfg.max_gamma;
    a.part = c->sm_part; a.mass = c->sm_mass; a.counters = c->sm_counters;
    if (rows > c->sm_rows_cap || a.nb > c->sm_nb_cap) arg_fail(ES_ERR_ARG, "internal: softmax launch too large");
    launch(c, "softmax_part", 0.0, softmax_part_kernel, dim3(rows, a.nb), dim3(SM_THREADS), (size_t)0, a);
    launch(c, dtok ? "softmax_sample" : "softmax", 0.0, softmax_finish_kernel, dim3(rows, a.nb),
           dim3(SM_THREADS), (size_t)0, a);
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
    int st[2] = {0, 0};
    CK(cudaMemcpy(st, c->status, sizeof st, cudaMemcpyDeviceToHost));
    if (st[1]) {
        // a tensor-core pass gave up a bounded wait: its results are not
        // valid, and the context is not usable any more
        c->poisoned = true;
        arg_fail(ES_ERR_TIMEOUT, "a device-side wait of a tensor-core weight pass ran out of time (flag 0x%x)", st[1]);
    }
    if (st[0]) {
        CK(cudaMemset(c->status, 0, sizeof(int)));
        arg_fail(ES_ERR_STATE, "device reported invalid rows (status 0x%x): position past max_seq or token out of range", st[0]);
    }
}

// ------------------------------------------------------------------ plans
// Set keys: -1 base (exact), 1 draft exact, 0 draft explicit sets, k >= 2
// draft sets of size k by the default rule.  Heads: 0 none, 1 calibration
// (last row of each sequence -> q slot 0), 2 fuzzy step (-> q slot step),
// 3 verify (every row -> p).
enum { HEAD_NONE = 0, HEAD_CALIB = 1, HEAD_FUZZY = 2, HEAD_VERIFY = 3 };
const Plan& get_forward(es_ctx* c, int key, int M, int head_kind, int step, int gamma) {
    const int which = key == -1 ? 1 : 0;
    // rows per sequence: one for the layer-parallel drafts, gamma+1 for
    // calibration and verify, a chunk of positions for the prompt prefill
    const int rps = head_kind == HEAD_FUZZY ? 1 : head_kind == HEAD_NONE ? std::max(1, M / std::max(1, c->B))
                                                                          : gamma + 1;
    auto pk = std::make_tuple(which, key, M, head_kind, step, gamma, rps);
    auto it = c->plans.find(pk);
    if (it != c->plans.end()) return it->second;
    std::vector<std::vector<int>> sets;
    Model& m = which ? c->mb : c->md;
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
    HeadSpec h;
    const int B = c->B;
    if (head_kind == HEAD_CALIB) { h.rows = B; h.stride = gamma + 1; h.off = gamma; h.y = c->q_logits; h.ldy = gamma * m.V; }
    if (head_kind == HEAD_FUZZY) { h.rows = B; h.y = c->q_logits + (size_t)step * m.V; h.ldy = gamma * m.V; }
    if (head_kind == HEAD_VERIFY) { h.rows = M; h.y = c->p_logits; h.ldy = m.V; }
    return c->plans[pk] = build_forward(c, m, sets, c->cfg.parallel_mode, M, rps, h);
}

// ------------------------------------------------------------------ phase parts
template <typename TD>
void enqueue_calibrate(es_ctx* c, int gamma) {
    Model& m = c->md;
    const int B = c->B, M = B * (gamma + 1);
    run_forward<TD>(c, m, get_forward(c, 1, M, HEAD_CALIB, 0, gamma), KIND_CALIB, 0, gamma, M);
    run_softmax(c, c->q_logits, c->q_probs, m.V, B, 1, 0, gamma, gamma, c->dtok);
}

template <typename TD>
void enqueue_fuzzy(es_ctx* c, int key, int gamma) {
    Model& m = c->md;
    const int B = c->B;
    for (int i = 1; i < gamma; ++i) {
        run_forward<TD>(c, m, get_forward(c, key, B, HEAD_FUZZY, i, gamma), KIND_FUZZY, i, gamma, B);
        run_softmax(c, c->q_logits, c->q_probs, m.V, B, 1, i, gamma, gamma, c->dtok);
    }
}

template <typename TB>
void enqueue_verify(es_ctx* c, int gamma) {
    Model& m = c->mb;
    const int B = c->B, M = B * (gamma + 1);
    run_forward<TB>(c, m, get_forward(c, -1, M, HEAD_VERIFY, 0, gamma), KIND_VERIFY, 0, gamma, M);
    run_softmax(c, c->p_logits, c->p_probs, m.V, M, gamma + 1, 0, gamma + 1, gamma, nullptr);
    AcceptArgs a;
    memset(&a, 0, sizeof a);
    a.p = c->p_probs; a.q = c->q_probs; a.d = c->dtok; a.gmax = c->cfg.max_gamma; a.gamma = gamma;
    a.V = m.V; a.greedy = -1; a.u_explicit = nullptr; a.prm = c->prm; a.phase = c->phase;
    vocab_chunks(m.V, c->num_sms, &a.chunk, &a.nb);
    a.gpart = c->sm_part; a.mass = c->sm_mass; a.counters = c->sm_counters;
    a.n_acc = c->n_acc; a.out_tok = c->out_tok; a.tokens = c->tokens; a.max_seq = c->cfg.max_seq;
    a.n_commit = c->n_commit; a.n_limit = c->n_limit; a.kv_from = c->kv_from;
    launch(c, "accept_resample", 0.0, accept_kernel, dim3(B, a.nb), dim3(SM_THREADS), (size_t)0, a);
}

void set_params(es_ctx* c, float T, uint64_t seed) {
    c->h_prm->seed = seed;
    c->h_prm->temperature = T;
    c->h_prm->calib_off = c->calib_off ? 1 : 0;
    CK(cudaMemcpyAsync(c->prm, c->h_prm, sizeof(RunParams), cudaMemcpyHostToDevice, c->st));
}

template <typename TD, typename TB>
void enqueue_part(es_ctx* c, int part, int gamma, int k) {
    if (part == 0) {
        enqueue_calibrate<TD>(c, gamma);
        enqueue_fuzzy<TD>(c, k, gamma);
    } else if (part == 1) {
        enqueue_verify<TB>(c, gamma);
    } else if (part == 2) {
        enqueue_calibrate<TD>(c, gamma);
    } else {
        enqueue_fuzzy<TD>(c, k, gamma);
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
    // build every plan before capture (descriptor uploads are synchronous)
    const int B = c->B, M = B * (gamma + 1);
    if (part != 1) {
        get_forward(c, 1, M, HEAD_CALIB, 0, gamma);
        for (int i = 1; i < gamma; ++i) get_forward(c, k, B, HEAD_FUZZY, i, gamma);
    } else {
        get_forward(c, -1, M, HEAD_VERIFY, 0, gamma);
    }
    if (c->profiling) {  // eager launches, each bracketed by events
        dispatch_part(c, part, gamma, k);
        return;
    }
    auto key = std::make_tuple(part, gamma, k, B);
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
    if (c->part_timing) {
        static const char* const names[4] = {"phase.draft", "phase.verify", "phase.calibrate", "phase.fuzzy"};
        if (c->prof_pool_used == c->prof_pool.size()) {
            cudaEvent_t x, y;
            CK(cudaEventCreate(&x));
            CK(cudaEventCreate(&y));
            c->prof_pool.emplace_back(x, y);
        }
        const auto ev = c->prof_pool[c->prof_pool_used++];
        CK(cudaEventRecord(ev.first, c->st));
        CK(cudaGraphLaunch(it->second.exec, c->st));
        CK(cudaEventRecord(ev.second, c->st));
        c->prof_pending.push_back(ProfRec{names[part], 0.0, ev.first, ev.second});
    } else {
        CK(cudaGraphLaunch(it->second.exec, c->st));
    }
    c->launches += it->second.kernels;
}

template <typename T>
void prefill_model(es_ctx* c, Model& m, const int32_t* prompts, int B, int P) {
    // exact forward over positions 0..P-2 of every sequence, in chunks of
    // positions (rows of a chunk only attend to earlier positions)
    const int npos = P - 1;
    if (npos <= 0) return;
    const int key = (&m == &c->mb) ? -1 : 1;
    const int chunk = std::max(1, m.Mw / B);
    std::vector<int> pos, seq, tok, base;
    for (int p0 = 0; p0 < npos; p0 += chunk) {
        const int p1 = std::min(npos, p0 + chunk);
        pos.clear(); seq.clear(); tok.clear(); base.clear();
        for (int b = 0; b < B; ++b)
            for (int p = p0; p < p1; ++p) {
                pos.push_back(p); seq.push_back(b); tok.push_back(prompts[(size_t)b * P + p]);
                base.push_back(b * (p1 - p0));
            }
        const int M = (int)pos.size();
        const Plan& plan = get_forward(c, key, M, HEAD_NONE, 0, 0);
        CK(cudaMemcpyAsync(m.row_pos, pos.data(), M * sizeof(int), cudaMemcpyHostToDevice, c->st));
        CK(cudaMemcpyAsync(m.row_seq, seq.data(), M * sizeof(int), cudaMemcpyHostToDevice, c->st));
        CK(cudaMemcpyAsync(m.row_tok, tok.data(), M * sizeof(int), cudaMemcpyHostToDevice, c->st));
        CK(cudaMemcpyAsync(m.row_base, base.data(), M * sizeof(int), cudaMemcpyHostToDevice, c->st));
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
    std::vector<int> n(B, P), lim(B, 0x7fffffff), kv(B, P - 1);
    CK(cudaMemcpyAsync(c->n_commit, n.data(), B * sizeof(int), cudaMemcpyHostToDevice, c->st));
    // the draft's prompt prefill below computes positions 0..P-2 exactly
    CK(cudaMemcpyAsync(c->kv_from, kv.data(), B * sizeof(int), cudaMemcpyHostToDevice, c->st));
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
            if (c->part_timing) {  // the same kernels as part 0, timed as two graphs
                run_part(c, 2, gamma, 1);
                run_part(c, 3, gamma, kk);
            } else {
                run_part(c, 0, gamma, kk);
            }
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

// ------------------------------------------------------------------ fixed scratch
// Scratch of es_accept_resample_noalloc: a file-scope device array, so the
// entry point never allocates.  Every GPU that loads the library holds it
// until the process exits.  Three regions, each sized for the largest call
// (B = NOALLOC_MAX_B, gamma = NOALLOC_MAX_GAMMA, NOALLOC_MAX_NB chunks): greedy
// argmax partials (floats), chunk masses (u64) and arrival counters (int).  A
// call packs its data densely from the start of each region with its own
// row count and chunk count: partials [B*(gamma+1)][nb][2], masses [B][nb][2],
// counters [B].
constexpr int NOALLOC_MAX_B = 16;
constexpr int NOALLOC_MAX_GAMMA = 16;
constexpr int NOALLOC_MAX_NB = 160;
constexpr size_t NA_GPART_BYTES = (size_t)NOALLOC_MAX_B * (NOALLOC_MAX_GAMMA + 1) * NOALLOC_MAX_NB * 2 * sizeof(float);
constexpr size_t NA_MASS_BYTES = (size_t)NOALLOC_MAX_B * NOALLOC_MAX_NB * 2 * sizeof(unsigned long long);
constexpr size_t NA_CTR_BYTES = (size_t)NOALLOC_MAX_B * sizeof(int);
constexpr size_t NA_BYTES = NA_GPART_BYTES + NA_MASS_BYTES + NA_CTR_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_BYTES];

// Device address of the scratch array on the current device.  Host code
// cannot use the array's name as a device pointer; the address is looked up
// once per device (the first call on that device) and kept.
es_status noalloc_scratch(unsigned char** out) {
    constexpr int MAX_DEV = 64;
    static unsigned char* addr[MAX_DEV] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return ES_ERR_CUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return ES_ERR_CUDA;
        }
        addr[dev] = static_cast<unsigned char*>(p);
    }
    *out = addr[dev];
    return ES_OK;
}

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
        c->kv_from = c->dalloc<int>(Bm);
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
        c->status = c->dalloc<int>(2);  // [0] invalid rows, [1] a bounded device wait ran out
        c->arena_cap = (size_t)64 << 20;
        c->arena = c->dalloc<char>(c->arena_cap);
        c->gv_scratch = c->dalloc<float>(std::max(GV_SCRATCH_FLOATS, GVM_SCRATCH_FLOATS));
        if (c->md.dtype == ES_DTYPE_BF16 || c->mb.dtype == ES_DTYPE_BF16) {
            // many-row bf16 passes: activation planes of the widest pass
            // (a set's K-concatenated o/down sources, or its 2 x n
            // normalised inputs) and the partials of split tiles
            size_t per_row = 0, rows = 0;
            for (const Model* mm : {&c->md, &c->mb}) {
                rows = std::max(rows, (size_t)mm->Mw);
                const size_t n = (size_t)mm->slots;
                per_row = std::max({per_row, n * (size_t)(mm->qd + mm->F), 2 * n * (size_t)mm->d,
                                    (size_t)mm->F, (size_t)mm->qd, (size_t)mm->d});
            }
            c->tc_x_elems = 2 * (2 * rows * per_row + (size_t)128 * 2 * TC_MAX_SRCS);  // two halves
            c->tc_x = c->dalloc<bf16>(c->tc_x_elems);
            CK(cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM_ONE));
            tensor_map_encoder();
        }
        c->gv_counters = c->dalloc<int>(GV_COUNTERS);
        c->gv_done = c->dalloc<int>(1);
        c->att_counters = c->dalloc<int>(ATT_COUNTERS);
        c->sm_rows_cap = std::max(c->md.Mw, c->mb.Mw);
        c->sm_nb_cap = c->num_sms + 1;
        c->sm_part = c->dalloc<float>((size_t)c->sm_rows_cap * c->sm_nb_cap * 2);
        c->sm_mass = c->dalloc<unsigned long long>((size_t)c->sm_rows_cap * c->sm_nb_cap * 2);
        c->sm_counters = c->dalloc<int>(c->sm_rows_cap);
        // dynamic shared memory beyond 48 KB must be allowed per kernel
        const int gv_smem = GV_XSMEM_MAX * (int)sizeof(float);
#define ES_GV_ATTR(TT, MM) \
        CK(cudaFuncSetAttribute(gv_kernel<TT, MM>, cudaFuncAttributeMaxDynamicSharedMemorySize, gv_smem));
        ES_GV_ATTR(float, 1) ES_GV_ATTR(float, 2) ES_GV_ATTR(float, 3) ES_GV_ATTR(float, 4)
        ES_GV_ATTR(float, 5) ES_GV_ATTR(float, 6) ES_GV_ATTR(float, 7) ES_GV_ATTR(float, 8)
#undef ES_GV_ATTR
        CK(cudaFuncSetAttribute(gvm_kernel<GV_WARPS>, cudaFuncAttributeMaxDynamicSharedMemorySize, gv_smem));
        CK(cudaFuncSetAttribute(gvm_kernel<GVM_WIDE_WARPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GVM_WIDE_XSMEM * (int)sizeof(float)));
        const int att_smem = 200 * 1024;
        CK(cudaFuncSetAttribute(attn_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, att_smem));
        CK(cudaFuncSetAttribute(attn_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, att_smem));
        CK(cudaFuncSetAttribute(attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
        CK(cudaFuncSetAttribute(attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
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

es_status es_set_calibration(es_ctx* c, int on) {
    if (!c) return ES_ERR_ARG;
    return guarded(c, [&] {
        if (on != 0 && on != 1) arg_fail(ES_ERR_ARG, "es_set_calibration: on must be 0 or 1");
        if (c->calibrated || c->drafted)
            arg_fail(ES_ERR_STATE, "es_set_calibration: a phase is in progress (finish it with verify_step)");
        c->calib_off = on == 0;
    });
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
        if (c->profiling || c->part_timing) prof_collect(c);
        if (on < 0 || on > 2) arg_fail(ES_ERR_ARG, "es_profile: mode %d (0, 1 or 2)", on);
        c->profiling = on == 1;
        c->part_timing = on == 2;
        c->prof.clear();
    });
}

es_status es_profile_read(es_ctx* c, int idx, char* name, int name_cap, double* ms,
                          int64_t* launches, double* bytes) {
    if (!c || !name || name_cap < 1) return ES_ERR_ARG;
    return guarded(c, [&] {
        if (c->profiling || c->part_timing) {
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
    cudaStream_t st = (cudaStream_t)stream;
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ES_ERR_CUDA;
    AcceptArgs a;
    memset(&a, 0, sizeof a);
    a.p = p; a.q = q; a.d = d; a.gmax = gamma; a.gamma = gamma; a.V = V; a.greedy = greedy ? 1 : 0;
    a.u_explicit = u; a.n_acc = n_acc; a.out_tok = tok;
    vocab_chunks(V, nsm, &a.chunk, &a.nb);
    // scratch of the split kernels, owned by this call
    const size_t rows = (size_t)B * (gamma + 1);
    float* gpart = nullptr;
    unsigned long long* mass = nullptr;
    int* ctr = nullptr;
    es_status rc = ES_OK;
    if (cudaMalloc(&gpart, rows * a.nb * 2 * sizeof(float)) != cudaSuccess ||
        cudaMalloc(&mass, (size_t)B * a.nb * 2 * sizeof(unsigned long long)) != cudaSuccess ||
        cudaMalloc(&ctr, (size_t)B * sizeof(int)) != cudaSuccess ||
        cudaMemsetAsync(ctr, 0, (size_t)B * sizeof(int), st) != cudaSuccess) {
        rc = ES_ERR_OOM;
    } else {
        a.gpart = gpart; a.mass = mass; a.counters = ctr;
        if (greedy) {
            SampleArgs s;
            memset(&s, 0, sizeof s);
            s.z = p; s.V = V; s.chunk = a.chunk; s.nb = a.nb; s.per_seq = 1; s.off = 0; s.ld_rows = 1;
            s.greedy = 1; s.part = gpart;
            softmax_part_kernel<<<dim3((unsigned)rows, a.nb), SM_THREADS, 0, st>>>(s);
        }
        accept_kernel<<<dim3(B, a.nb), SM_THREADS, 0, st>>>(a);
        if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) rc = ES_ERR_CUDA;
    }
    cudaFree(gpart);
    cudaFree(mass);
    cudaFree(ctr);
    return rc;
}

es_status es_accept_resample_noalloc(const float* p, const float* q, const int32_t* d, const uint64_t* u,
                                     int B, int gamma, int V, int greedy, int32_t* n_acc, int32_t* tok,
                                     void* stream) {
    if (!p || !q || !d || !n_acc || !tok || B < 1 || gamma < 1 || V < 1) return ES_ERR_ARG;
    if (!greedy && !u) return ES_ERR_ARG;
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ES_ERR_CUDA;
    AcceptArgs a;
    memset(&a, 0, sizeof a);
    vocab_chunks(V, nsm, &a.chunk, &a.nb);
    if (B > NOALLOC_MAX_B || gamma > NOALLOC_MAX_GAMMA || a.nb > NOALLOC_MAX_NB) {
        fprintf(stderr, "es_accept_resample_noalloc: B=%d gamma=%d (%d vocabulary chunks) beyond the fixed "
                        "scratch (B <= %d, gamma <= %d, chunks <= %d)\n",
                B, gamma, a.nb, NOALLOC_MAX_B, NOALLOC_MAX_GAMMA, NOALLOC_MAX_NB);
        return ES_ERR_ARG;
    }
    unsigned char* base = nullptr;
    const es_status sst = noalloc_scratch(&base);
    if (sst != ES_OK) return sst;
    cudaStream_t st = (cudaStream_t)stream;
    a.p = p; a.q = q; a.d = d; a.gmax = gamma; a.gamma = gamma; a.V = V; a.greedy = greedy ? 1 : 0;
    a.u_explicit = u; a.n_acc = n_acc; a.out_tok = tok;
    float* gpart = reinterpret_cast<float*>(base);
    a.gpart = gpart;
    a.mass = reinterpret_cast<unsigned long long*>(base + NA_GPART_BYTES);
    a.counters = reinterpret_cast<int*>(base + NA_GPART_BYTES + NA_MASS_BYTES);
    // the arrival counters must start at zero (the array keeps the last
    // call's contents)
    if (cudaMemsetAsync(a.counters, 0, (size_t)B * sizeof(int), st) != cudaSuccess) return ES_ERR_CUDA;
    if (greedy) {
        SampleArgs s;
        memset(&s, 0, sizeof s);
        s.z = p; s.V = V; s.chunk = a.chunk; s.nb = a.nb; s.per_seq = 1; s.off = 0; s.ld_rows = 1;
        s.greedy = 1; s.part = gpart;
        softmax_part_kernel<<<dim3((unsigned)(B * (gamma + 1)), a.nb), SM_THREADS, 0, st>>>(s);
    }
    accept_kernel<<<dim3(B, a.nb), SM_THREADS, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess) return ES_ERR_CUDA;
    return ES_OK;
}

es_status es_wait_selftest(int64_t limit_ns, int64_t arrive_ns, void* stream) {
    if (limit_ns <= 0 || limit_ns > 2000000000ll || arrive_ns > 1000000000ll) return ES_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int* flag = nullptr;
    if (cudaMalloc(&flag, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return ES_ERR_OOM;
    }
    es_status rc = ES_OK;
    int h = 0;
    if (cudaMemsetAsync(flag, 0, sizeof(int), st) != cudaSuccess) rc = ES_ERR_CUDA;
    if (rc == ES_OK) {
        wait_selftest_kernel<<<1, 64, 0, st>>>((long long)limit_ns, (long long)arrive_ns, flag);
        if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess ||
            cudaMemcpy(&h, flag, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
            rc = ES_ERR_CUDA;
    }
    cudaFree(flag);
    if (rc == ES_OK && h) rc = ES_ERR_TIMEOUT;
    return rc;
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

es_status es_layer_sets(int n_layers, int k, int32_t* starts, int cap, int* n_sets) {
    if (n_layers < 1 || k < 1 || k > MAX_GROUP || !n_sets || cap < 0 || (cap > 0 && !starts)) return ES_ERR_ARG;
    const auto sets = default_sets(n_layers, k);
    *n_sets = (int)sets.size();
    for (int i = 0; i < (int)sets.size() && i < cap; ++i) starts[i] = sets[i].front();
    return ES_OK;
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
