"""The dispatch table (csrc/planner.h) without a GPU: a host program prints
the plan for a grid of problems on a 152-SM device, and every plan is checked
against the limits the kernels rely on (tier boundaries, tightest-fitting
configuration, shared-memory and register budgets per SM, mbarrier byte
counts, TMA sizes, tile coverage)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "rmsnorm_fwd_bwd_add_gb300", "csrc")
NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"

pytestmark = pytest.mark.skipif(not os.path.exists(NVCC), reason="nvcc not available")

SM = 152
SMEM_PER_SM = 228 * 1024      # shared memory of one SM
SMEM_PER_CTA = 227 * 1024     # opt-in maximum of one CTA
RESERVED_PER_CTA = 1024
HEADER = 640
TX_LIMIT = (1 << 20) - 1      # mbarrier transaction count
WIDE = 10                     # the forward-only configuration the planner takes only when tuned


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("planner") / "planner_check")
    cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O1",
           "-I" + os.path.join(ROOT, "include"), "-I" + CSRC,
           os.path.join(ROOT, "tests", "planner_check.cu"), "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True)
    env = {k: v for k, v in os.environ.items() if k != "RMSNORM_TUNE"}
    out = subprocess.run([exe], check=True, capture_output=True, text=True, env=env).stdout
    cfgs, rows = {}, []
    for line in out.splitlines():
        f = line.split()
        if f[0] == "cfg":
            cfgs[int(f[1])] = tuple(int(x) for x in f[2:])
        else:
            rows.append([int(x) for x in f])
    return cfgs, rows


def _cluster_fits(mode, nv):
    """Whether a cluster of 2, 4 or 8 CTAs (slices of up to 2048 vectors)
    covers a row of nv vectors with three stages of its slices in one SM's
    shared memory."""
    ntens = 1 if mode == 1 else 3 if mode == 3 else 2
    for cl in (2, 4, 8):
        sl = -(-nv // cl)
        if sl <= 2048 and (225 * 1024) // (ntens * sl * 16) >= 3:
            return True
    return False


def test_tiers_and_configurations(plans):
    cfgs, rows = plans
    assert len(rows) > 1000
    for (mode, es, D, R, tier, cfg, nt, g, v, max_nv, stages, tr, ntiles, grid, smem, sb,
         max_ctas, align, shift, cl, cl_cols) in rows:
        if align == 2:
            continue  # shifted rows: test_shifted_plans
        nv = D * es // 16
        vjp = mode >= 2
        if R > 8 and nv <= 2048:
            assert tier == 0, (mode, es, D, R)
            # the configuration that fits the row most tightly
            fits = [c for c, (_, _, _, mx) in cfgs.items() if c != WIDE and nv <= mx]
            assert cfg == min(fits, key=lambda c: cfgs[c][3]), (D, es, cfg)
            assert (nt, g, v, max_nv) == cfgs[cfg]
        elif R > 8 and _cluster_fits(mode, nv):
            assert tier == 3, (mode, es, D, R)  # a cluster of CTAs per row
        elif R <= 8 and nv <= (2048 if vjp else 4096):
            assert tier == 1, (mode, es, D, R)
            # a decode VJP of 2-8 rows: one cluster of its rows sums gw itself
            if vjp and R >= 2:
                assert cl == R and smem == D * 4 and grid == R, (mode, es, D, R)
            else:
                assert cl == 0, (mode, es, D, R)
        else:
            assert tier == 2, (mode, es, D, R)


def test_staged_plans_fit_the_hardware(plans):
    _, rows = plans
    n = 0
    for (mode, es, D, R, tier, cfg, nt, g, v, max_nv, stages, tr, ntiles, grid, smem, sb,
         max_ctas, align, shift, cl, cl_cols) in rows:
        if tier != 0:
            continue
        n += 1
        ntens = 1 if mode == 1 else 3 if mode == 3 else 2
        where = (mode, es, D, R)
        assert 2 <= stages <= 8, where
        assert tr >= 1 and (g == nt and tr == 1 or tr % (nt // g) == 0), where
        if align == 1:
            assert not shift and sb == tr * D * es and sb % 16 == 0, where
        else:  # the aligned superset of the tile at the worst offset
            assert shift and sb % 16 == 0 and sb >= 16 - es + tr * D * es, where
        assert ntens * sb <= TX_LIMIT, where             # one tile's bytes on one mbarrier
        assert smem >= HEADER + stages * ntens * sb, where
        if mode >= 2 and g < nt:                          # the cross-group gw sum reuses the ring
            assert smem >= HEADER + (nt // g) * D * 4, where
        assert smem <= SMEM_PER_CTA, where
        assert ntiles == -(-R // tr) and 1 <= grid <= ntiles, where
        cps = -(-grid // SM)                              # CTAs per SM the grid implies
        if grid == ntiles:
            cps = min(cps, max_ctas)
        assert cps <= max_ctas, where
        assert cps * (smem + RESERVED_PER_CTA) <= SMEM_PER_SM, where
        assert cps * nt <= 2048, where                    # threads per SM
    assert n > 500


def test_plan_is_a_pure_function(plans, tmp_path):
    _, rows = plans
    again = {tuple(r[:4]) + (r[17],): r[4:] for r in rows}
    assert len(again) == len(rows)  # one plan per (mode, esize, D, rows)


def _smem_share(cps):
    """Shared memory one CTA may take when `cps` CTAs share an SM (the planner's budget)."""
    return {1: 225 * 1024, 2: 110 * 1024, 3: 72 * 1024}.get(cps, 224 * 1024 // max(cps, 1) - 2048)


def test_ring_depth_floor(plans):
    """CTA-per-row plans keep at least three stages where they fit when they run one CTA per
    SM or are VJPs: a stage is refilled only after the next row's barrier, so two leave nothing
    in flight while a row is read."""
    _, rows = plans
    n = 0
    for (mode, es, D, R, tier, cfg, nt, g, v, max_nv, stages, tr, ntiles, grid, smem, sb,
         max_ctas, align, shift, cl, cl_cols) in rows:
        if tier != 0 or g != nt or R < 16384:
            continue
        cps = grid // SM
        ntens = 1 if mode == 1 else 3 if mode == 3 else 2
        if (cps == 1 or mode >= 2) and _smem_share(cps) // (ntens * sb) >= 3:
            n += 1
            assert stages >= 3, (mode, es, D, R, cps, stages)
    assert n > 50


def test_reread_vjp_ctas_per_sm(plans):
    """The VJP instances that re-read their rows from the stage (384 and 448 threads) run two
    CTAs per SM; the 512-thread VJP, which holds its rows, runs one."""
    _, rows = plans
    seen = set()
    for (mode, es, D, R, tier, cfg, nt, g, v, max_nv, stages, tr, ntiles, grid, smem, sb,
         max_ctas, align, shift, cl, cl_cols) in rows:
        if tier != 0 or g != nt or mode < 2:
            continue
        if nt in (384, 448):
            assert max_ctas == 2, (mode, es, D, nt)
            seen.add(nt)
        if nt == 512:
            assert max_ctas == 1, (mode, es, D, nt)
            seen.add(nt)
    assert seen == {384, 448, 512}


def _period(D, es):
    """Rows after which a dense row's offset from a 16-byte boundary repeats."""
    rb = D * es % 16
    return 1 if rb == 0 else 2 if rb % 8 == 0 else 4 if rb % 4 == 0 else 8


def test_shifted_plans(plans):
    """Rows off 16-byte boundaries: the staged tier with the configuration an
    aligned row of the same D gets (its whole vectors; the edge elements are
    handled apart), stages that hold the superset of a tile at the worst
    offset, sub-warp tiles of a multiple of 8 rows, and CTAs that take
    several rows on a grid that is a multiple of the offset's period (so a
    CTA sees one offset on all of its rows)."""
    cfgs, rows = plans
    n = 0
    for (mode, es, D, R, tier, cfg, nt, g, v, max_nv, stages, tr, ntiles, grid, smem, sb,
         max_ctas, align, shift, cl, cl_cols) in rows:
        if align != 2:
            continue
        where = (mode, es, D, R)
        nv = D * es // 16  # whole vectors; the edge elements are handled apart
        if R > 8 and nv <= 2048:
            n += 1
            assert tier == 0 and shift, where
            fits = [c for c, (_, _, _, mx) in cfgs.items() if c != WIDE and nv <= mx]
            assert cfg == min(fits, key=lambda c: cfgs[c][3]), where
            assert g * v >= nv and g * 2 >= 14, where  # the edges: up to 14, 1-2 a lane
            if g < nt:
                assert tr % 8 == 0, where
            elif grid < ntiles:
                assert grid % _period(D, es) == 0, where
        else:
            assert tier != 0 and not shift, where
    assert n > 300


def test_cluster_plans(plans):
    """Rows of more than 2048 vectors (forward and VJP): clusters of 2, 4
    or 8 CTAs whose slices (whole 16-byte vectors) cover the row with no CTA
    left empty, each CTA sized to its slice (two vectors a thread up to 640
    threads, else four; threads rounded up to a warp), one CTA per SM, rings
    of at least three stages (four or more, for the pipelined loop, wherever
    they fit) in one SM's shared memory, and a grid of whole clusters
    (without a device query: SMs // cl clusters at most) of the size that
    keeps the most SMs busy, except that a forward whose busiest size leaves
    the ring three slices deep takes a size with four or more that keeps at
    least 94 % as many SMs busy and gives each cluster at least 32 rows."""
    _, rows = plans
    n = 0
    for (mode, es, D, R, tier, cfg, nt, g, v, max_nv, stages, tr, ntiles, grid, smem, sb,
         max_ctas, align, shift, cl, cl_cols) in rows:
        if tier != 3:
            continue
        n += 1
        where = (mode, es, D, R)
        nv = D * es // 16
        ntens = 1 if mode == 1 else 3 if mode == 3 else 2
        assert align == 1 and R > 8 and nv > 2048, where
        assert cl in (2, 4, 8) and v in (2, 4) and nt % 32 == 0, where
        assert cl_cols * es % 16 == 0, where
        slice_v = cl_cols * es // 16
        assert (v == 2) == (slice_v <= 1280) and nt <= (640 if v == 2 else 512), where
        assert slice_v <= v * nt < slice_v + 32 * v, where  # the CTA fits its slice
        assert cl * slice_v >= nv and (cl - 1) * slice_v < nv, where
        assert sb == cl_cols * es, where
        assert 3 <= stages <= 8 and smem == 1024 + stages * ntens * sb, where
        fits4 = (225 * 1024) // (ntens * sb) >= 4
        assert (stages >= 4) == fits4, where  # the pipelined loop wherever four fit
        assert smem + RESERVED_PER_CTA <= SMEM_PER_SM and smem <= SMEM_PER_CTA, where
        assert ntiles == R and grid % cl == 0 and grid // cl == min(R, SM // cl), where
        assert ntens * sb <= TX_LIMIT, where
        def depth(c):
            return (225 * 1024) // (ntens * -(-nv // c) * 16)

        def busy(c):
            return min(R, SM // c) * c

        fitting = [c for c in (2, 4, 8) if -(-nv // c) <= 2048 and depth(c) >= 3]
        want = max(fitting, key=lambda c: (busy(c), -c))
        if mode in (0, 1) and depth(want) < 4:
            deeper = [c for c in fitting if depth(c) >= 4 and busy(c) * 100 >= busy(want) * 94
                      and R >= 32 * (SM // c)]
            if deeper:
                want = max(deeper, key=lambda c: (busy(c), -c))
        assert cl == want, where
    assert n > 30
