// Host check of the tensor-core weight pass's stage walker and activation
// windows: the __host__ __device__ functions that the kernel itself runs
// (GvWalk, gvm_windows), driven here on the CPU over random launches.
//
// For every CTA range of stages it checks that
//  * the walker visits the stages in (op, tile, segment, column chunk) order,
//    each stage of the launch exactly once over all CTAs, and reports the end
//    of a tile exactly when the tile's last chunk is consumed;
//  * every chunk the CTA multiplies lies in one of its windows (unless the
//    window table is full, when the kernel reads the rest from global memory),
//    windows of one source neither overlap nor touch, and no window stages a
//    chunk the CTA does not multiply;
//  * staged windows sit back to back within the budget, with a plane row
//    stride of 64 mod 128 bytes (conflict-free fragment loads), and the
//    device's rerun with the host's computed size as its budget stages the
//    same windows at the same offsets;
//  * the staging loops (gvm_stage_cursor's column walk and gvm_stage_item's
//    item split, run here for every thread of a 256- and a 512-thread CTA)
//    visit every (staged window, float4 column, activation row) exactly once.
//
// Exit status 0 when every check holds; the first failures go to stderr.
#include <algorithm>
#include <cstdio>
#include <random>
#include <vector>

#include "gemv.cuh"

using namespace es;

static int g_fails = 0;
#define CHECK(cond, ...)                                                   \
    do {                                                                   \
        if (!(cond)) {                                                     \
            if (g_fails++ < 20) {                                          \
                fprintf(stderr, "check failed at line %d: ", __LINE__);    \
                fprintf(stderr, __VA_ARGS__);                              \
                fprintf(stderr, "\n");                                     \
            }                                                              \
        }                                                                  \
    } while (0)

struct Stage { int op, tile, seg, kc; };

// tiles of RT rows, chunks of GVM_COLS columns, equal stage ranges for `ctas`
static void lay_out(GvLaunch& L, int RT, int ctas) {
    int t = 0, st = 0;
    for (int i = 0; i < L.nops; ++i) {
        GvOp& o = L.ops[i];
        o.spt = 0;
        for (int s = 0; s < o.nseg; ++s) {
            GvSeg& g = L.segs[o.seg0 + s];
            g.nck = (g.K + GVM_COLS - 1) / GVM_COLS;
            o.spt += g.nck;
        }
        o.ntiles = (o.N + RT - 1) / RT;
        o.tile0 = t;
        o.stage0 = st;
        t += o.ntiles;
        st += o.ntiles * o.spt;
    }
    L.ntiles = t;
    L.nstages = st;
    L.q = std::max(1, (st + ctas - 1) / ctas);
}

static std::vector<Stage> enumerate(const GvLaunch& L) {
    std::vector<Stage> v;
    for (int op = 0; op < L.nops; ++op) {
        const GvOp& o = L.ops[op];
        for (int t = 0; t < o.ntiles; ++t)
            for (int s = 0; s < o.nseg; ++s)
                for (int c = 0; c < L.segs[o.seg0 + s].nck; ++c) v.push_back({op, t, s, c});
    }
    return v;
}

static void check_staging(const GvLaunch& L, const GvmWin* win, int n, int cta) {
    const int total = gvm_stage_columns(win, n), M = L.M;
    std::vector<int> base(n + 1, 0);  // first float4 column of each window (0 columns if not staged)
    for (int i = 0; i < n; ++i) base[i + 1] = base[i] + (win[i].off >= 0 ? (win[i].khi - win[i].klo) * (GVM_COLS / 4) : 0);
    CHECK(base[n] == total, "cta %d: %d staged columns, counted %d", cta, total, base[n]);
    std::vector<int> seen((size_t)total * M);
    auto visit = [&](int w, int kr, int m, const char* how) {
        const bool ok = w >= 0 && w < n && win[w].off >= 0 && kr % 4 == 0 && kr >= 0 &&
                        kr < (win[w].khi - win[w].klo) * GVM_COLS && m >= 0 && m < M;
        CHECK(ok, "cta %d (%s): window %d column %d row %d outside the staged windows", cta, how, w, kr, m);
        if (ok) ++seen[(size_t)(base[w] + kr / 4) * M + m];
    };
    auto all_once = [&](const char* how, int nt) {
        for (size_t i = 0; i < seen.size(); ++i)
            CHECK(seen[i] == 1, "cta %d (%s, %d threads): item %zu visited %d times", cta, how, nt, i, seen[i]);
        std::fill(seen.begin(), seen.end(), 0);
    };
    for (int nt : {256, 512}) {
        for (int tid = 0; tid < nt; ++tid) {
            int w = 0, wbase = 0;
            for (int c = tid; c < total; c += nt) {
                gvm_stage_cursor(win, c, w, wbase);
                for (int m = 0; m < M; ++m) visit(w, (c - wbase) * 4, m, "columns");
            }
        }
        all_once("columns", nt);
        for (int tid = 0; tid < nt; ++tid)
            for (int t0 = tid; t0 < M * total; t0 += 2 * nt)
                for (int u = 0; u < 2; ++u) {
                    const int t = t0 + u * nt;
                    if (t >= M * total) break;
                    int w, m, kr;
                    gvm_stage_item(win, total, t, w, m, kr);
                    visit(w, kr, m, "items");
                }
        all_once("items", nt);
    }
}

static void check_launch(const GvLaunch& L) {
    const std::vector<Stage> want = enumerate(L);
    CHECK((int)want.size() == L.nstages, "stage count %zu vs %d", want.size(), L.nstages);
    std::vector<int> seen(L.nstages, 0);
    const int grid = (L.nstages + L.q - 1) / L.q;
    std::vector<int> used_at_max(grid, 0);
    int need = 0;
    for (int cta = 0; cta < grid; ++cta) {
        const int S0 = cta * L.q, S1 = std::min(L.nstages, S0 + L.q);
        // walker
        std::vector<std::pair<int, int>> chunks;  // (source, chunk) multiplied by this CTA
        GvWalk w;
        w.seek(&L, S0);
        for (int s = S0; s < S1;) {
            const GvOp& o = L.ops[w.op];
            const GvSeg& sg = L.segs[o.seg0 + w.seg];
            const int run = std::min(sg.nck - w.kc, S1 - s);
            for (int j = 0; j < run; ++j) {
                const Stage& e = want[s + j];
                CHECK(e.op == w.op && e.tile == w.tile && e.seg == w.seg && e.kc == w.kc + j,
                      "stage %d: walker (%d,%d,%d,%d) expected (%d,%d,%d,%d)", s + j, w.op, w.tile, w.seg,
                      w.kc + j, e.op, e.tile, e.seg, e.kc);
                ++seen[s + j];
                chunks.push_back({sg.xs, w.kc + j});
            }
            const bool ends_tile = w.kc + run == sg.nck && w.seg == o.nseg - 1;
            const bool r = w.advance(run);
            CHECK(r == ends_tile, "stage %d: advance returned %d, tile end %d", s, (int)r, (int)ends_tile);
            s += run;
        }
        // windows, budget large enough for everything
        GvmWin win[GVM_NWIN];
        int items = 0, used = 0;
        const int n = gvm_windows(L, S0, S1, win, 1 << 30, &items, &used);
        CHECK(n >= 1 && n <= GVM_NWIN, "cta %d: %d windows", cta, n);
        for (const auto& ch : chunks) {
            bool in = false;
            for (int i = 0; i < n; ++i) in = in || (win[i].src == ch.first && win[i].klo <= ch.second && ch.second < win[i].khi);
            CHECK(in || n == GVM_NWIN, "cta %d: chunk %d of source %d outside every window", cta, ch.second, ch.first);
        }
        int off = 0, it = 0;
        for (int i = 0; i < n; ++i) {
            const int cols = (win[i].khi - win[i].klo) * GVM_COLS;
            CHECK(win[i].klo < win[i].khi, "cta %d: empty window", cta);
            CHECK(win[i].pw == cols + GVM_PAD && (win[i].pw * 2) % 128 == 64, "cta %d: plane stride %d", cta, win[i].pw);
            CHECK(win[i].off == off && win[i].item0 == it, "cta %d: window %d at %d (expected %d)", cta, i, win[i].off, off);
            off += L.M * win[i].pw;
            it += L.M * (cols / 4);
            for (int k = win[i].klo; k < win[i].khi; ++k)
                CHECK(std::find(chunks.begin(), chunks.end(), std::make_pair(win[i].src, k)) != chunks.end(),
                      "cta %d: window stages chunk %d of source %d that it never multiplies", cta, k, win[i].src);
            for (int j = i + 1; j < n; ++j)
                CHECK(win[i].src != win[j].src || win[i].khi < win[j].klo || win[j].khi < win[i].klo,
                      "cta %d: windows %d and %d of source %d overlap or touch", cta, i, j, win[i].src);
        }
        CHECK(used == off && items == it, "cta %d: used %d items %d", cta, used, items);
        // the 8-warp budget: greedy staging within it
        GvmWin wb[GVM_NWIN];
        int ib = 0, ub = 0;
        const int nb = gvm_windows(L, S0, S1, wb, GV_XSMEM_MAX, &ib, &ub);
        CHECK(nb == n && ub <= GV_XSMEM_MAX, "cta %d: budgeted windows %d used %d", cta, nb, ub);
        int acc = 0;
        for (int i = 0; i < nb; ++i) {
            const int words = L.M * wb[i].pw;
            if (acc + words <= GV_XSMEM_MAX) {
                CHECK(wb[i].off == acc, "cta %d: staged window %d at %d (expected %d)", cta, i, wb[i].off, acc);
                acc += words;
            } else {
                CHECK(wb[i].off == -1, "cta %d: window %d of %d words staged past the budget", cta, i, words);
            }
        }
        check_staging(L, wb, nb, cta);
        used_at_max[cta] = ub;
        need = std::max(need, ub);
    }
    for (int s = 0; s < L.nstages; ++s) CHECK(seen[s] == 1, "stage %d visited %d times", s, seen[s]);
    // the device reruns the window function with the host's size as budget
    for (int cta = 0; cta < grid; ++cta) {
        const int S0 = cta * L.q, S1 = std::min(L.nstages, S0 + L.q);
        GvmWin a[GVM_NWIN], b[GVM_NWIN];
        int ia = 0, ua = 0, ib = 0, ub = 0;
        const int na = gvm_windows(L, S0, S1, a, GV_XSMEM_MAX, &ia, &ua);
        const int nb = gvm_windows(L, S0, S1, b, need, &ib, &ub);
        CHECK(na == nb && ua == ub && ia == ib, "cta %d: rerun with budget %d differs", cta, need);
        for (int i = 0; i < std::min(na, nb); ++i)
            CHECK(a[i].off == b[i].off && a[i].klo == b[i].klo && a[i].khi == b[i].khi,
                  "cta %d: window %d differs on the rerun", cta, i);
    }
}

int main() {
    std::mt19937 rng(12345);
    auto uni = [&](int lo, int hi) { return std::uniform_int_distribution<int>(lo, hi)(rng); };
    static GvLaunch L;
    long stages = 0;
    int cases = 0;
    const int layouts[4][2] = {{GVM_BLOCK, 148 * GV_CTAS_PER_SM}, {GVM_WIDE_WARPS * GVM_ROWS, 148}, {GVM_BLOCK, 7},
                               {GVM_BLOCK, 1}};
    for (int trial = 0; trial < 400; ++trial) {
        memset(&L, 0, sizeof L);
        L.M = uni(1, 8);
        L.nxs = uni(1, 6);
        int Ks[GV_MAX_XS];
        for (int i = 0; i < L.nxs; ++i) {
            // ragged widths (multiples of 4, mostly not of 128) and the model widths
            const int pick = uni(0, 3);
            Ks[i] = pick == 0 ? 4 * uni(1, 1500) : pick == 1 ? 128 * uni(1, 40) : pick == 2 ? 896 : 3584;
            L.xs[i].K = Ks[i];
        }
        L.nops = uni(1, 8);
        int nseg = 0;
        for (int i = 0; i < L.nops; ++i) {
            GvOp& o = L.ops[i];
            o.N = uni(0, 3) == 0 ? uni(1, 300) : uni(1, 6000);
            o.seg0 = nseg;
            o.nseg = uni(1, 3);
            for (int s = 0; s < o.nseg; ++s) {
                GvSeg& g = L.segs[nseg++];
                g.xs = uni(0, L.nxs - 1);
                g.K = Ks[g.xs];
            }
        }
        const int* lo = layouts[trial % 4];
        lay_out(L, lo[0], lo[1]);
        check_launch(L);
        stages += L.nstages;
        ++cases;
    }
    printf("%d launches, %ld stages, %d failed checks\n", cases, stages, g_fails);
    return g_fails ? 1 : 0;
}
