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


def test_tiers_and_configurations(plans):
    cfgs, rows = plans
    assert len(rows) > 1000
    for (mode, es, D, R, tier, cfg, nt, g, v, max_nv, stages, tr, ntiles, grid, smem, sb,
         max_ctas) in rows:
        nv = D * es // 16
        vjp = mode >= 2
        if R > 8 and nv <= 2048:
            assert tier == 0, (mode, es, D, R)
            # the configuration that fits the row most tightly
            fits = [c for c, (_, _, _, mx) in cfgs.items() if c != WIDE and nv <= mx]
            assert cfg == min(fits, key=lambda c: cfgs[c][3]), (D, es, cfg)
            assert (nt, g, v, max_nv) == cfgs[cfg]
        elif R <= 8 and nv <= (2048 if vjp else 4096):
            assert tier == 1, (mode, es, D, R)
        elif nv > (2048 if vjp else 4096):
            assert tier == 2, (mode, es, D, R)


def test_staged_plans_fit_the_hardware(plans):
    _, rows = plans
    n = 0
    for (mode, es, D, R, tier, cfg, nt, g, v, max_nv, stages, tr, ntiles, grid, smem, sb,
         max_ctas) in rows:
        if tier != 0:
            continue
        n += 1
        ntens = 1 if mode == 1 else 3 if mode == 3 else 2
        where = (mode, es, D, R)
        assert 2 <= stages <= 8, where
        assert tr >= 1 and (g == nt and tr == 1 or tr % (nt // g) == 0), where
        assert sb == tr * D * es and sb % 16 == 0, where
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
    again = {tuple(r[:4]): r[4:] for r in rows}
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
         max_ctas) in rows:
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
         max_ctas) in rows:
        if tier != 0 or g != nt or mode < 2:
            continue
        if nt in (384, 448):
            assert max_ctas == 2, (mode, es, D, nt)
            seen.add(nt)
        if nt == 512:
            assert max_ctas == 1, (mode, es, D, nt)
            seen.add(nt)
    assert seen == {384, 448, 512}
