"""Rotary embedding of q and k with the KV-cache append against the fp64
oracle: decode and prefill token counts with Llama-like heads, both pair
layouts, a cos/sin table and on-the-fly angles at large positions, dense,
ring and paged slot patterns, skipped tokens and in-place q."""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_add_gb300 as rn
from parity import assert_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_add_gb300 import build
    build.build()
    rn.rmsnorm_device_status(clear=True)
    yield
    assert rn.rmsnorm_device_status(clear=True) == 0


def _inputs(T, Hq, Hkv, Dh, S, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(T, Hq, Dh, generator=gen).to(dtype)
    k = torch.randn(T, Hkv, Dh, generator=gen).to(dtype)
    v = torch.randn(T, Hkv, Dh, generator=gen).to(dtype)
    kc = torch.randn(S, Hkv, Dh, generator=gen).to(dtype)
    vc = torch.randn(S, Hkv, Dh, generator=gen).to(dtype)
    return q, k, v, kc, vc


def _table(max_pos, Dh, base):
    i = np.arange(Dh // 2)
    ang = np.arange(max_pos)[:, None] * np.power(float(np.float32(base)), -2.0 * i / Dh)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


def _run_and_check(q, k, v, kc, vc, pos, slots, base=10000.0, interleaved=False, table=None,
                   in_place=False):
    dev = lambda t: t.to(DEV)
    qd, kcd, vcd = dev(q), dev(kc), dev(vc)
    cs = None if table is None else torch.from_numpy(table).to(torch.float32).to(DEV)
    q_out = rn.rmsnorm_rope_kv_append(qd, dev(k), dev(v), dev(torch.tensor(pos)), dev(torch.tensor(slots)),
                                      kcd, vcd, rope_base=base, cos_sin=cs, interleaved=interleaved,
                                      q_out=qd if in_place else None)
    if in_place:
        assert q_out.data_ptr() == qd.data_ptr()
    cs64 = None if table is None else f64(torch.from_numpy(table).to(torch.float32))
    want_q, want_kc, want_vc = oracle.rope_kv_append(f64(q), f64(k), f64(v), pos, slots, f64(kc),
                                                     f64(vc), base, interleaved, cs64)
    assert_close("rope q", q_out, want_q)
    written = sorted({s for s in slots if s >= 0})
    untouched = [r for r in range(kc.shape[0]) if r not in written]
    got_kc, got_vc = kcd.cpu(), vcd.cpu()
    assert torch.equal(got_kc[untouched], kc[untouched]), "k rows no token names changed"
    assert torch.equal(got_vc[untouched], vc[untouched]), "v rows no token names changed"
    if written:
        assert_close("rope k cache", got_kc[written], want_kc[written])
        for t, s in enumerate(slots):
            if s >= 0:
                assert torch.equal(got_vc[s], v[t]), "v must be copied exactly"


@pytest.mark.parametrize("T", [1, 4, 8, 2048])
@pytest.mark.parametrize("interleaved", [False, True], ids=["half", "interleaved"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_rope_decode_and_prefill(T, interleaved, dtype):
    Hq, Hkv, Dh = 32, 8, 128
    S = T + 16
    q, k, v, kc, vc = _inputs(T, Hq, Hkv, Dh, S, dtype, T + interleaved)
    rng = np.random.default_rng(T)
    pos = (rng.integers(0, 120000, size=T) if T < 100 else np.arange(50000, 50000 + T)).tolist()
    slots = rng.permutation(S)[:T].tolist()
    _run_and_check(q, k, v, kc, vc, pos, slots, base=500000.0, interleaved=interleaved)


@pytest.mark.parametrize("interleaved", [False, True], ids=["half", "interleaved"])
def test_rope_far_positions(interleaved):
    """Computed angles at positions 10^6 - 1.6 * 10^7: the product p * base^(-2i/Dh) is formed
    as a double-float and reduced modulo 2 pi before the SFU sine and cosine, which are accurate
    only near [-pi, pi]; a plain float product would be off by up to 0.06 rad here."""
    T, Hq, Hkv, Dh = 64, 8, 2, 128
    S = T
    q, k, v, kc, vc = _inputs(T, Hq, Hkv, Dh, S, torch.float16, 77 + interleaved)
    rng = np.random.default_rng(5)
    pos = rng.integers(1_000_000, 16_000_000, size=T).tolist()
    slots = rng.permutation(S)[:T].tolist()
    _run_and_check(q, k, v, kc, vc, pos, slots, base=500000.0, interleaved=interleaved)


# Shapes of the warp-wide kernel (Dh % 16 == 0, up to 32 rotation units per
# head): units per head that do not divide 32 (Dh = 80: five), exactly 32
# (rotate-half Dh = 512, interleaved Dh = 256), past it (interleaved Dh = 512
# and Dh = 1024: the CTA-wide kernel), and token counts that spread a token
# over several warps (300, 40) or one warp (1000 with few heads).
@pytest.mark.parametrize("T,Hq,Hkv,Dh", [(300, 8, 2, 64), (1000, 4, 1, 80), (300, 6, 3, 128),
                                         (130, 2, 2, 256), (129, 3, 1, 512), (40, 2, 1, 1024)],
                         ids=["t300_d64", "t1000_d80", "t300_d128", "t130_d256", "t129_d512",
                              "t40_d1024"])
@pytest.mark.parametrize("interleaved", [False, True], ids=["half", "interleaved"])
@pytest.mark.parametrize("use_table", [False, True], ids=["computed", "table"])
def test_rope_warp_kernel_shapes(T, Hq, Hkv, Dh, interleaved, use_table):
    S = T + 5
    q, k, v, kc, vc = _inputs(T, Hq, Hkv, Dh, S, torch.bfloat16, T + Dh)
    rng = np.random.default_rng(Dh)
    max_pos = 5000
    pos = rng.integers(0, max_pos, size=T).tolist()
    slots = [(-1 if t % 7 == 3 else int(s)) for t, s in enumerate(rng.permutation(S)[:T])]
    table = _table(max_pos, Dh, 10000.0) if use_table else None
    _run_and_check(q, k, v, kc, vc, pos, slots, interleaved=interleaved, table=table,
                   in_place=(T % 2 == 0))


def test_rope_table_and_skipped_tokens():
    T, Hq, Hkv, Dh, S = 40, 8, 2, 64, 64
    q, k, v, kc, vc = _inputs(T, Hq, Hkv, Dh, S, torch.bfloat16, 3)
    table = _table(4096, Dh, 10000.0)
    rng = np.random.default_rng(4)
    pos = rng.integers(0, 4096, size=T).tolist()
    slots = [(-1 if t % 5 == 0 else int(s)) for t, s in enumerate(rng.permutation(S)[:T])]
    _run_and_check(q, k, v, kc, vc, pos, slots, table=table)
    _run_and_check(q, k, v, kc, vc, pos, slots, table=table, interleaved=True)


def test_rope_ring_and_paged_slots():
    T, Hq, Hkv, Dh = 12, 4, 2, 128
    # ring cache of 8 rows: slot = position mod 8 (the last 8 tokens survive)
    q, k, v, kc, vc = _inputs(8, Hq, Hkv, Dh, 8, torch.bfloat16, 5)
    pos = list(range(1000, 1008))
    _run_and_check(q, k, v, kc, vc, pos, [p % 8 for p in pos])
    # paged pool: 6 blocks of 4 rows, two sequences with scattered blocks
    q, k, v, kc, vc = _inputs(T, Hq, Hkv, Dh, 24, torch.bfloat16, 6)
    table = {0: [5, 2, 1], 1: [0, 4, 3]}
    pos, slots = [], []
    for t in range(T):
        seq, p = t % 2, 3 + t // 2
        pos.append(p)
        slots.append(table[seq][p // 4] * 4 + p % 4)
    _run_and_check(q, k, v, kc, vc, pos, slots)


def test_rope_in_place_and_element_path():
    q, k, v, kc, vc = _inputs(6, 3, 1, 128, 6, torch.float16, 7)
    _run_and_check(q, k, v, kc, vc, [0, 1, 2, 3, 4, 5], [0, 1, 2, 3, 4, 5], in_place=True)
    # Dh = 6: not a multiple of 16, the element-wise kernel
    q, k, v, kc, vc = _inputs(5, 2, 2, 6, 7, torch.bfloat16, 8)
    _run_and_check(q, k, v, kc, vc, [9, 8, 7, 6, 5], [6, 0, -1, 3, 2])
    _run_and_check(q, k, v, kc, vc, [9, 8, 7, 6, 5], [6, 0, -1, 3, 2], interleaved=True)


def test_rope_bad_indices_are_flagged_not_touched():
    """Positions past the table and slots past the cache are caught on the
    device: those tokens are skipped, the rest are right, the status says so."""
    T, Hq, Hkv, Dh, S = 6, 2, 1, 16, 4
    q, k, v, kc, vc = _inputs(T, Hq, Hkv, Dh, S, torch.bfloat16, 9)
    table = torch.from_numpy(_table(32, Dh, 10000.0)).to(torch.float32).to(DEV)
    pos = torch.tensor([1, 40, 3, 4, -2, 5], device=DEV)     # 40 >= 32 and -2 are bad
    slots = torch.tensor([0, 1, 9, 2, 3, -1], device=DEV)    # 9 >= 4 is bad
    qd, kcd, vcd = q.to(DEV), kc.to(DEV), vc.to(DEV)
    rn.rmsnorm_device_status(clear=True)
    q_out = torch.full_like(qd, float("nan"))
    rn.rmsnorm_rope_kv_append(qd, k.to(DEV), v.to(DEV), pos, slots, kcd, vcd, cos_sin=table,
                              q_out=q_out)
    bits = rn.rmsnorm_device_status(clear=True)
    assert bits & rn.DEVSTATUS_BAD_INDEX
    got = q_out.cpu()
    assert torch.isnan(got[1]).all() and torch.isnan(got[4]).all()  # skipped tokens
    want_q, want_kc, _ = oracle.rope_kv_append(f64(q), f64(k), f64(v), [1, 0, 3, 4, 0, 5],
                                               [0, -1, -1, 2, -1, -1], f64(kc), f64(vc),
                                               cos_sin=f64(table.cpu()))
    for t in (0, 2, 3, 5):  # token 2's q is rotated even though its slot is bad
        assert_close("q token %d" % t, got[t], want_q[t])
    assert torch.equal(kcd.cpu()[[1, 3]], kc[[1, 3]])  # rows only bad tokens named
    assert_close("k row 0", kcd.cpu()[0], want_kc[0])


def test_rope_argument_errors():
    q = torch.zeros(2, 2, 16, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(2, 1, 16, dtype=torch.bfloat16, device=DEV)
    pos = torch.zeros(2, dtype=torch.int64, device=DEV)
    lib = rn._native.lib()
    cache = torch.zeros(4, 1, 16, dtype=torch.bfloat16, device=DEV)
    vcache = torch.zeros(4, 1, 16, dtype=torch.bfloat16, device=DEV)
    args = [q.data_ptr(), k.data_ptr(), k.data_ptr(), pos.data_ptr(), pos.data_ptr(), q.data_ptr(),
            cache.data_ptr(), vcache.data_ptr(), None, 0, 10000.0, 0, 2, 2, 1, 16, 4, 1, None]
    bad = list(args)
    bad[13] = 15  # odd Dh
    assert lib.rmsnorm_rope_kv_append(*bad) == 1
    bad = list(args)
    bad[10] = -1.0  # no table and a negative base
    assert lib.rmsnorm_rope_kv_append(*bad) == 1
    bad = list(args)
    bad[7] = cache.data_ptr()  # v_cache overlapping k_cache
    assert lib.rmsnorm_rope_kv_append(*bad) == 1
