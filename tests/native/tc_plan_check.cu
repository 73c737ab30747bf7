// Host check of the tensor-core weight pass's launch layout and unit decode:
// tc_layout (row chunks, stages, CTAs per SM, tensor-memory columns, cluster
// size, k-ranges) and tc_unit (what a CTA of the grid works on) -- the
// functions the planner and the kernel themselves use -- driven here on the
// CPU over random launches.
//
// For every launch it checks that
//  * row chunks cover the rows, none is empty, and each is padded to a
//    multiple of 16 of at most 256 rows (the MMA's N);
//  * stages are 1024-byte multiples, 2 to 8 of them, and the CTA's shared
//    memory fits one CTA per SM, or two when the layout says two;
//  * tensor-memory columns are a power of two from 32 to 512 that holds the
//    accumulators, and two CTAs on an SM fit the SM's 512 columns;
//  * the cluster size is 1, 2, 4 or 8; split tiles keep the grid within the
//    CTA slots, give every range at least 4 k-blocks of the largest op, and
//    the partials fit in a CTA's shared memory;
//  * over the grid, every (op, tile, row chunk) is one cluster whose ranks'
//    k-ranges partition [0, nkb) in rank order.
//
// Exit status 0 when every check holds; the first failures go to stderr.
#include <cstdio>
#include <cstring>
#include <random>
#include <vector>

#include "tcgemm.cuh"

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

int main() {
    std::mt19937 rng(2026);
    auto pick = [&](int lo, int hi) { return std::uniform_int_distribution<int>(lo, hi)(rng); };
    static TcLaunch L;
    long checks = 0;
    for (int it = 0; it < 3000; ++it) {
        memset(&L, 0, sizeof L);
        const int sms = pick(0, 2) == 0 ? 132 : 148;
        const int mkind = pick(0, 3);
        L.M = mkind == 0 ? pick(1, 8) : mkind == 1 ? pick(9, 96) : mkind == 2 ? pick(97, 300) : pick(300, 1100);
        L.nops = pick(1, 6);
        for (int oi = 0; oi < L.nops; ++oi) {
            TcOp& o = L.ops[oi];
            o.pair = pick(0, 3) == 0;
            o.N = pick(0, 1) ? pick(1, 1024) : pick(1024, 40000);
            const int K = 8 * pick(1, 4000);
            o.nkb = (K + TC_BK - 1) / TC_BK;
            if (!o.pair && pick(0, 2) == 0) o.nkb += (8 * pick(1, 3000) + TC_BK - 1) / TC_BK;  // K-concatenated
        }
        const int cps = tc_layout(L, sms);
        CHECK(cps == 1 || cps == 2, "CTAs per SM %d", cps);
        if (cps == 0) continue;
        // rows
        CHECK(L.npad % 16 == 0 && L.npad >= 16 && L.npad <= TC_MAXN, "npad %d", L.npad);
        CHECK(L.rc * L.npad >= L.M && (L.rc - 1) * L.npad < L.M, "M %d rc %d npad %d", L.M, L.rc, L.npad);
        // shared memory
        const int smem = L.stages * L.stage_bytes + 1024;
        CHECK(L.stage_bytes % 1024 == 0, "stage %d", L.stage_bytes);
        CHECK(L.stages >= 2 && L.stages <= 8, "stages %d", L.stages);
        CHECK(smem <= (cps == 2 ? TC_SMEM_TWO : TC_SMEM_ONE), "smem %d for %d CTAs", smem, cps);
        CHECK(L.stage_bytes == TC_BM * TC_BK * 2 * (L.any_pair ? 2 : 1) + 2 * L.npad * TC_BK * 2, "stage bytes");
        // tensor memory
        const int cols = L.npad * (L.any_pair ? 2 : 1);
        CHECK((L.tmem_cols & (L.tmem_cols - 1)) == 0 && L.tmem_cols >= 32 && L.tmem_cols <= 512, "tmem %d",
              L.tmem_cols);
        CHECK(L.tmem_cols >= cols && L.tmem_cols < 2 * cols + 32, "tmem %d for %d columns", L.tmem_cols, cols);
        CHECK(cps * L.tmem_cols <= 512, "tmem %d x %d CTAs", L.tmem_cols, cps);
        // clusters
        CHECK(L.cs == 1 || L.cs == 2 || L.cs == 4 || L.cs == 8, "cs %d", L.cs);
        if (L.cs > 1) {
            CHECK(L.nclusters * L.cs <= sms * cps, "grid %d over %d slots", L.nclusters * L.cs, sms * cps);
            int nkb_max = 0;
            for (int oi = 0; oi < L.nops; ++oi) nkb_max = L.ops[oi].nkb > nkb_max ? L.ops[oi].nkb : nkb_max;
            CHECK(nkb_max / L.cs >= 4, "ranges of %d k-blocks", nkb_max / L.cs);
            CHECK((L.any_pair ? 2 : 1) * L.npad * TC_BM * 4 <= L.stages * L.stage_bytes, "partials do not fit");
        }
        // the grid: every (op, tile, chunk) once, its ranks partition [0, nkb)
        int nclusters = 0;
        for (int oi = 0; oi < L.nops; ++oi) nclusters += L.ops[oi].ntiles * L.rc;
        CHECK(nclusters == L.nclusters, "clusters %d vs %d", L.nclusters, nclusters);
        std::vector<int> seen(nclusters, 0);
        for (int b = 0; b < L.nclusters * L.cs; ++b) {
            const TcUnit u = tc_unit(L, b);
            const TcOp& o = L.ops[u.op];
            CHECK(u.op >= 0 && u.op < L.nops, "op %d", u.op);
            CHECK(u.tile >= 0 && u.tile < o.ntiles && u.chunk >= 0 && u.chunk < L.rc, "tile %d chunk %d", u.tile,
                  u.chunk);
            CHECK(u.split == b % L.cs, "rank");
            const int cl = o.cl0 + u.tile * L.rc + u.chunk;
            CHECK(cl == b / L.cs, "cluster %d of block %d", cl, b);
            // rank r's range starts where rank r-1's ended (or at nkb)
            const int expect = u.split == 0 ? 0 : tc_unit(L, b - 1).kb_end;
            CHECK(u.kb_begin == expect, "range start %d vs %d", u.kb_begin, expect);
            CHECK(u.kb_end >= u.kb_begin && u.kb_end <= o.nkb, "range [%d, %d) of %d", u.kb_begin, u.kb_end, o.nkb);
            if (u.split == L.cs - 1) CHECK(u.kb_end == o.nkb, "last range ends at %d of %d", u.kb_end, o.nkb);
            seen[cl] += 1;
            ++checks;
        }
        for (int cl = 0; cl < nclusters; ++cl) CHECK(seen[cl] == L.cs, "cluster %d has %d CTAs", cl, seen[cl]);
    }
    printf("%ld units, %d failed checks\n", checks, g_fails);
    return g_fails ? 1 : 0;
}
