// planner_check.cu -- prints the dispatch plan for a grid of problems, one
// line per problem, for tests/test_planner_cpu.py.  Host code only: it runs
// without a GPU (make_plan is a pure function of its arguments).
//
// Output: the staged configuration table ("cfg index nt g v max_nv"), then
// per problem: mode esize D rows tier cfg nt g v max_nv stages tile_rows
// num_tiles grid smem stage_bytes max_ctas align shift cl cl_cols (align 1:
// rows on 16-byte boundaries, 2: rows at one shared offset from them; cl,
// cl_cols: the cluster tier's CTAs per row and columns per CTA)
#include <cstdio>

#include "planner.h"

int main() {
    using namespace rmsn;
    const int sm = 152;
    const int Ds[] = {8, 16, 64, 120, 128, 256, 264, 512, 520, 640, 768, 1000, 1024, 1032, 1536, 2048,
                      2056, 2560, 3072, 3584, 4096, 4104, 5120, 6144, 7168, 8192, 8200, 10240,
                      12288, 14336, 16384, 16392, 32768, 40000, 65536, 131072,
                      // rows off 16-byte boundaries (with align 2 every D is shifted)
                      7, 9, 63, 257, 1001, 1025, 2050, 3075, 4097, 4098, 4100, 6147, 8204,
                      12291, 16383};
    const long long rows_list[] = {1, 8, 9, 64, 300, 4096, 16384, 131072, 3000000000LL};
    for (int ci = 0; ci < N_STAGED_CFG; ++ci)
        std::printf("cfg %d %d %d %d %d\n", ci, STAGED_CFGS[ci].nt, STAGED_CFGS[ci].g,
                    STAGED_CFGS[ci].v, STAGED_CFGS[ci].max_nv);
    for (int align : {ALIGN_VEC, ALIGN_SHIFT})
    for (int mode = 0; mode < 4; ++mode)
        for (int esize : {2, 4})
            for (int D : Ds)
                for (long long rows : rows_list) {
                    // dense rows with aligned bases are shifted when D * esize % 16 != 0
                    const int a = align == ALIGN_VEC && (D * esize) % 16 != 0 ? ALIGN_SHIFT : align;
                    if (align == ALIGN_VEC && a != align) continue;
                    const Plan p = planner::make_plan(mode, rows, D, esize, a, sm);
                    int max_nv = 0, max_ctas = 0;
                    if (p.tier == TIER_STAGED) {
                        max_nv = STAGED_CFGS[p.cfg].max_nv;
                        max_ctas = staged_max_ctas_per_sm(mode, p.nt, p.g, p.v);
                    }
                    std::printf("%d %d %d %lld %d %d %d %d %d %d %d %d %lld %d %zu %u %d %d %d %d %d\n",
                                mode, esize, D, rows, p.tier, p.cfg, p.nt, p.g, p.v, max_nv,
                                p.stages, p.tile_rows, (long long)p.num_tiles, p.grid, p.smem,
                                p.stage_bytes, max_ctas, a, (int)p.shift, p.cl, p.cl_cols);
                }
    return 0;
}
