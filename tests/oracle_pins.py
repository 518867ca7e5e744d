"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, independent of the oracle's own code.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a mismatch.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on deliberately broken copies of the
oracle source and requires every copy to fail at least one pin.

What each pin rests on:
  * worked examples -- hand-derived exact values (tests/golden), from the
    definitions on "Fused residual-add RMSNorm and fused RoPE + KV-append
    decode kernels" (Background) and "RMSNormVJP backward writes a full
    {n_rows, D} gw_temp intermediate" (POC);
  * closed forms -- constant rows, D = 1, weight_bias = 1 with w = 0 against a
    library norm (numpy.linalg.norm), gw as a row sum written with einsum;
  * invariants -- scale invariance at eps = 0, the sum_j h_j gx_j identity,
    linearity in g, row-permutation equivariance, scaled weight;
  * central finite differences of L = sum(g * out) through the forward only.
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "worked_examples.json")


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, "%s: shape %s vs %s" % (what, a.shape, b.shape)
    ok = np.abs(a - b) <= atol + rtol * np.abs(b)
    assert ok.all(), "%s: max |diff| %.3e (rtol %.1e)" % (
        what, float(np.max(np.abs(a - b))), rtol)


def _rng(seed):
    return np.random.default_rng(seed)


def pin_worked_examples(orc):
    """Hand-derived exact values (tests/golden/worked_examples.json)."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x = np.array(c["x"], np.float64)
        res = None if c["residual"] is None else np.array(c["residual"], np.float64)
        w = np.array(c["w"], np.float64)
        out, new_res = orc.fwd(x, w, c["eps"], c["weight_bias"], res)
        _close(out, c["out"], 1e-14, 1e-15, c["name"] + " out")
        if res is not None:
            _close(new_res, c["new_residual"], 0, 0, c["name"] + " new_residual")
        h = x if res is None else x + res
        gx, gw = orc.vjp(h, w, np.array(c["g"], np.float64), c["eps"], c["weight_bias"])
        _close(gx, c["gx"], 1e-14, 1e-15, c["name"] + " gx")
        _close(gw, c["gw"], 1e-14, 1e-15, c["name"] + " gw")


def pin_constant_rows(orc):
    """A row of equal values c with w = 1, weight_bias = 0 normalises to
    c / sqrt(c^2 + eps): +-1 up to eps."""
    D = 37
    for c in (3.0, -0.5, 1e-3, 250.0):
        for eps in (0.0, 1e-6, 1e-2):
            x = np.full((2, D), c)
            out, _ = orc.fwd(x, np.ones(D), eps, 0.0)
            want = c / np.sqrt(c * c + orc.scalar(eps))
            _close(out, np.full((2, D), want), 1e-14, 0, "constant row c=%g eps=%g" % (c, eps))


def pin_d1(orc):
    """D = 1: out = h / sqrt(h^2 + eps) * (weight_bias + w)."""
    h = np.array([[-3.0], [0.25], [7.5]])
    for wb, w in ((0.0, 2.0), (1.0, -0.5)):
        out, _ = orc.fwd(h, np.array([w]), 0.5, wb)
        want = h / np.sqrt(h * h + 0.5) * (wb + w)
        _close(out, want, 1e-14, 0, "D=1")


def pin_unit_weight_bias_plain_norm(orc):
    """weight_bias = 1 with w = 0 is plain normalisation, written here with a
    library norm: h / sqrt(||h||^2 / D + eps)."""
    rng = _rng(11)
    for R, D in ((3, 16), (5, 129), (1, 1000)):
        h = rng.normal(size=(R, D)) * rng.uniform(0.1, 10, size=(R, 1))
        eps = 1e-3
        out, _ = orc.fwd(h, np.zeros(D), eps, 1.0)
        nrm = np.linalg.norm(h, axis=1, keepdims=True)
        want = h / np.sqrt(nrm ** 2 / D + orc.scalar(eps))
        _close(out, want, 1e-12, 0, "wb=1,w=0 R=%d D=%d" % (R, D))


def pin_residual_is_added(orc):
    """The fused forward equals the plain forward of x + residual, and
    new_residual is exactly x + residual."""
    rng = _rng(12)
    R, D = 4, 33
    x = rng.normal(size=(R, D))
    res = rng.normal(size=(R, D))
    w = rng.normal(1.0, 0.1, size=D)
    out_f, new_res = orc.fwd(x, w, 1e-5, 0.25, res)
    out_p, none = orc.fwd(x + res, w, 1e-5, 0.25)
    assert none is None
    _close(new_res, x + res, 0, 0, "new_residual")
    _close(out_f, out_p, 1e-14, 0, "fused vs plain on x + residual")
    # weight_bias enters as an additive bias on w
    out_b, _ = orc.fwd(x + res, w + 0.25, 1e-5, 0.0)
    _close(out_f, out_b, 1e-13, 0, "weight_bias shifts w")


def pin_scale_invariance(orc):
    """With eps = 0: out(a*h) = sign(a) * out(h), so by the chain rule
    gx(a*h) = gx(h) / |a| and gw(a*h) = sign(a) * gw(h)."""
    rng = _rng(13)
    R, D = 3, 20
    h = rng.normal(size=(R, D))
    w = rng.normal(1.0, 0.3, size=D)
    g = rng.normal(size=(R, D))
    out0, _ = orc.fwd(h, w, 0.0, 0.5)
    gx0, gw0 = orc.vjp(h, w, g, 0.0, 0.5)
    for a in (3.75, -0.25, 1e3):
        out1, _ = orc.fwd(a * h, w, 0.0, 0.5)
        gx1, gw1 = orc.vjp(a * h, w, g, 0.0, 0.5)
        _close(out1, np.sign(a) * out0, 1e-13, 1e-15, "out scale a=%g" % a)
        _close(gx1 * abs(a), gx0, 1e-12, 1e-14, "gx scale a=%g" % a)
        _close(gw1, np.sign(a) * gw0, 1e-12, 1e-14, "gw scale a=%g" % a)


def pin_gw_row_sum(orc):
    """gw_j = sum_i g_ij * h_ij * r_i with r_i from a library norm."""
    rng = _rng(14)
    R, D = 7, 24
    h = rng.normal(size=(R, D))
    w = rng.normal(size=D)
    g = rng.normal(size=(R, D))
    eps = 1e-4
    _, gw = orc.vjp(h, w, g, eps, 0.75)
    r = 1.0 / np.sqrt(np.linalg.norm(h, axis=1) ** 2 / D + orc.scalar(eps))
    want = np.einsum("ij,ij,i->j", g, h, r)
    _close(gw, want, 1e-12, 1e-14, "gw row sum")


def _loss(orc, x, w, g, eps, wb, res=None):
    out, _ = orc.fwd(x, w, eps, wb, res)
    return float(np.sum(g * out))


def pin_finite_differences(orc):
    """Central differences of L = sum(g * out) through the forward only match
    gx (with respect to x, and to residual in the fused op) and gw."""
    rng = _rng(15)
    for (R, D, eps, wb, with_res) in ((1, 1, 1e-2, 0.0, False), (2, 5, 1e-5, 0.0, True),
                                      (3, 9, 1e-3, 1.0, False), (3, 8, 0.0, 0.5, True)):
        x = rng.normal(size=(R, D))
        res = rng.normal(size=(R, D)) if with_res else None
        w = rng.normal(0.5, 0.5, size=D)
        g = rng.normal(size=(R, D))
        h = x if res is None else x + res
        gx, gw = orc.vjp(h, w, g, eps, wb)
        fd_x = np.zeros_like(x)
        fd_res = np.zeros_like(x)
        for i in range(R):
            for j in range(D):
                d = 1e-5 * (1.0 + abs(x[i, j]))
                xp = x.copy(); xp[i, j] += d
                xm = x.copy(); xm[i, j] -= d
                fd_x[i, j] = (_loss(orc, xp, w, g, eps, wb, res)
                              - _loss(orc, xm, w, g, eps, wb, res)) / (2 * d)
                if res is not None:
                    d = 1e-5 * (1.0 + abs(res[i, j]))
                    rp = res.copy(); rp[i, j] += d
                    rm = res.copy(); rm[i, j] -= d
                    fd_res[i, j] = (_loss(orc, x, w, g, eps, wb, rp)
                                    - _loss(orc, x, w, g, eps, wb, rm)) / (2 * d)
        fd_w = np.zeros(D)
        for j in range(D):
            d = 1e-5 * (1.0 + abs(w[j]))
            wp = w.copy(); wp[j] += d
            wm = w.copy(); wm[j] -= d
            fd_w[j] = (_loss(orc, x, wp, g, eps, wb, res)
                       - _loss(orc, x, wm, g, eps, wb, res)) / (2 * d)
        scale = max(1.0, float(np.max(np.abs(gx))))
        _close(gx, fd_x, 1e-6, 1e-6 * scale, "fd gx R=%d D=%d" % (R, D))
        if res is not None:
            _close(gx, fd_res, 1e-6, 1e-6 * scale, "fd g_residual R=%d D=%d" % (R, D))
        _close(gw, fd_w, 1e-6, 1e-6 * max(1.0, float(np.max(np.abs(gw)))),
               "fd gw R=%d D=%d" % (R, D))


def pin_h_dot_gx_identity(orc):
    """sum_j h_j gx_j = r * eps / (ms + eps) * dot for every row (zero when
    eps = 0: the output does not change under h -> (1 + t) h)."""
    rng = _rng(16)
    R, D = 5, 31
    h = rng.normal(size=(R, D))
    w = rng.normal(1.0, 0.2, size=D)
    g = rng.normal(size=(R, D))
    wb = orc.scalar(0.2)
    for eps in (0.0, 0.3):
        e = orc.scalar(eps)
        gx, _ = orc.vjp(h, w, g, eps, wb)
        ms = np.mean(h * h, axis=1)
        r = 1.0 / np.sqrt(ms + e)
        dot = np.sum(g * (wb + w) * h, axis=1)
        lhs = np.sum(h * gx, axis=1)
        _close(lhs, r * e / (ms + e) * dot, 1e-11, 1e-13, "identity eps=%g" % eps)


def pin_linearity_in_g(orc):
    """(gx, gw) is linear in g."""
    rng = _rng(17)
    R, D = 4, 12
    h = rng.normal(size=(R, D))
    w = rng.normal(size=D)
    g1 = rng.normal(size=(R, D))
    g2 = rng.normal(size=(R, D))
    a, b = 2.5, -0.75
    gx1, gw1 = orc.vjp(h, w, g1, 1e-3, 0.1)
    gx2, gw2 = orc.vjp(h, w, g2, 1e-3, 0.1)
    gx3, gw3 = orc.vjp(h, w, a * g1 + b * g2, 1e-3, 0.1)
    _close(gx3, a * gx1 + b * gx2, 1e-12, 1e-13, "gx linear")
    _close(gw3, a * gw1 + b * gw2, 1e-12, 1e-13, "gw linear")


def pin_row_permutation(orc):
    """Permuting rows permutes out and gx and leaves gw unchanged."""
    rng = _rng(18)
    R, D = 6, 10
    h = rng.normal(size=(R, D)) * rng.uniform(0.5, 3, size=(R, 1))
    w = rng.normal(size=D)
    g = rng.normal(size=(R, D))
    p = rng.permutation(R)
    out, _ = orc.fwd(h, w, 1e-4, 0.0)
    outp, _ = orc.fwd(h[p], w, 1e-4, 0.0)
    _close(outp, out[p], 0, 0, "out permuted")
    gx, gw = orc.vjp(h, w, g, 1e-4, 0.0)
    gxp, gwp = orc.vjp(h[p], w, g[p], 1e-4, 0.0)
    _close(gxp, gx[p], 0, 0, "gx permuted")
    _close(gwp, gw, 1e-13, 1e-15, "gw invariant")


def pin_scaled_weight(orc):
    """With weight_bias = 0, scaling w by a scales out and gx by a (the
    scaled-weight check of the regression-guard list)."""
    rng = _rng(19)
    R, D = 3, 14
    h = rng.normal(size=(R, D))
    w = rng.normal(1.0, 0.1, size=D)
    g = rng.normal(size=(R, D))
    a = 1.7
    out, _ = orc.fwd(h, w, 1e-5, 0.0)
    outa, _ = orc.fwd(h, a * w, 1e-5, 0.0)
    _close(outa, a * out, 1e-13, 1e-15, "out scaled weight")
    gx, gw = orc.vjp(h, w, g, 1e-5, 0.0)
    gxa, gwa = orc.vjp(h, a * w, g, 1e-5, 0.0)
    _close(gxa, a * gx, 1e-12, 1e-14, "gx scaled weight")
    _close(gwa, gw, 1e-13, 1e-15, "gw does not depend on w")


def _fused_loss(orc, x, res, w, g_out, g_res, eps, wb):
    out, new_res = orc.fwd(x, w, eps, wb, res)
    return float(np.sum(g_out * out) + np.sum(g_res * new_res))


def pin_fused_vjp_finite_differences(orc):
    """The two-output op's VJP: central differences of
    L = sum(g_out * out) + sum(g_res * new_residual) with respect to x, to
    residual and to w, through the forward only."""
    rng = _rng(20)
    for (R, D, eps, wb) in ((2, 6, 1e-4, 0.0), (3, 5, 1e-2, 1.0)):
        x = rng.normal(size=(R, D))
        res = rng.normal(size=(R, D))
        w = rng.normal(0.5, 0.5, size=D)
        g_out = rng.normal(size=(R, D))
        g_res = rng.normal(size=(R, D))
        g_h, gw = orc.fused_vjp(x + res, w, g_out, eps, wb, g_res)
        fd_x = np.zeros_like(x)
        fd_r = np.zeros_like(x)
        for i in range(R):
            for j in range(D):
                for arr, fd in ((x, fd_x), (res, fd_r)):
                    d = 1e-5 * (1.0 + abs(arr[i, j]))
                    keep = arr[i, j]
                    arr[i, j] = keep + d
                    lp = _fused_loss(orc, x, res, w, g_out, g_res, eps, wb)
                    arr[i, j] = keep - d
                    lm = _fused_loss(orc, x, res, w, g_out, g_res, eps, wb)
                    arr[i, j] = keep
                    fd[i, j] = (lp - lm) / (2 * d)
        fd_w = np.zeros(D)
        for j in range(D):
            d = 1e-5 * (1.0 + abs(w[j]))
            wp = w.copy(); wp[j] += d
            wm = w.copy(); wm[j] -= d
            fd_w[j] = (_fused_loss(orc, x, res, wp, g_out, g_res, eps, wb)
                       - _fused_loss(orc, x, res, wm, g_out, g_res, eps, wb)) / (2 * d)
        scale = max(1.0, float(np.max(np.abs(g_h))))
        _close(g_h, fd_x, 1e-6, 1e-6 * scale, "fused fd d/dx")
        _close(g_h, fd_r, 1e-6, 1e-6 * scale, "fused fd d/dresidual")
        _close(gw, fd_w, 1e-6, 1e-6 * max(1.0, float(np.max(np.abs(gw)))), "fused fd d/dw")
    # without a residual gradient it is the plain VJP
    h = rng.normal(size=(2, 7))
    w = rng.normal(size=7)
    g = rng.normal(size=(2, 7))
    a = orc.fused_vjp(h, w, g, 1e-3, 0.5)
    b = orc.vjp(h, w, g, 1e-3, 0.5)
    _close(a[0], b[0], 0, 0, "fused without g_res")
    _close(a[1], b[1], 0, 0, "fused gw without g_res")


def pin_gated_silu(orc):
    """Gated activation: silu(a) - silu(-a) = a (since sigmoid(a) +
    sigmoid(-a) = 1); silu(0) = 0; out is linear in the second half;
    sigmoid(ln k) = k / (k + 1) gives exact values at a = ln k (ln from the math
    library); silu(a) -> a for large a and -> 0 for very negative a."""
    import math
    rng = _rng(21)
    d = 9
    a = rng.normal(size=d) * 3
    b1 = np.ones(d)
    x = np.stack([np.concatenate([a, b1]), np.concatenate([-a, b1])])
    out = orc.gated_silu(x)
    _close(out[0] - out[1], a, 1e-13, 1e-14, "silu(a) - silu(-a) = a")
    b = rng.normal(size=d)
    z = orc.gated_silu(np.concatenate([np.zeros(d), b])[None, :])
    _close(z, np.zeros((1, d)), 0, 0, "silu(0) = 0")
    o1 = orc.gated_silu(np.concatenate([a, b])[None, :])
    o2 = orc.gated_silu(np.concatenate([a, 2.5 * b])[None, :])
    _close(o2, 2.5 * o1, 1e-14, 1e-15, "linear in the gate's second half")
    ks = np.array([1.0, 3.0, 7.0, 0.25, 1.0 / 3.0])
    av = np.array([math.log(k) for k in ks])
    bv = np.array([4.0, 4.0, 8.0, 5.0, 4.0])
    want = av * ks / (ks + 1.0) * bv
    got = orc.gated_silu(np.concatenate([av, bv])[None, :])
    _close(got, want[None, :], 1e-14, 1e-15, "silu(ln k) = ln k * k / (k + 1)")
    big = orc.gated_silu(np.array([[40.0, -40.0, 1.0, 1.0]]))
    _close(big[0, 0], 40.0, 1e-15, 0, "silu(40) ~ 40")
    assert abs(big[0, 1]) < 1e-15, "silu(-40) ~ 0"
    # rows are independent and the halves are taken per row
    xs = rng.normal(size=(3, 2 * d))
    _close(orc.gated_silu(xs)[1], orc.gated_silu(xs[1:2])[0], 0, 0, "row 1 alone")


def _rope(orc, x, positions, base=10000.0, interleaved=False, cos_sin=None):
    """rope of x (T, H, Dh) at the given positions through the oracle (q path)."""
    T, H, Dh = x.shape
    kc = np.zeros((1, 1, Dh))
    q_out, _, _ = orc.rope_kv_append(x, np.zeros((T, 1, Dh)), np.zeros((T, 1, Dh)), positions,
                                     -np.ones(T, np.int64), kc, kc, base, interleaved, cos_sin)
    return q_out


def pin_rope(orc):
    """Rotary embedding: position 0 is the identity; norms are kept; the
    score <rope(q, m), rope(k, n)> depends only on n - m; rope(rope(x, a), b)
    = rope(x, a + b); closed forms where theta is simple (Dh = 2: theta = p;
    Dh = 4, base 100: theta_1 = p / 10, with cos/sin from the math library);
    the interleaved layout is the rotate-half layout under the even/odd
    permutation; a table of the same cos/sin gives the same result."""
    import math
    rng = _rng(22)
    for inter in (False, True):
        x = rng.normal(size=(3, 2, 8))
        _close(_rope(orc, x, [0, 0, 0], interleaved=inter), x, 0, 0, "rope at 0")
        y = _rope(orc, x, [3, 1000, 123456], interleaved=inter)
        _close(np.linalg.norm(y, axis=2), np.linalg.norm(x, axis=2), 1e-13, 0, "norm kept")
        q = rng.normal(size=(1, 1, 16))
        k = rng.normal(size=(1, 1, 16))
        s1 = np.sum(_rope(orc, q, [7], interleaved=inter) * _rope(orc, k, [19], interleaved=inter))
        s2 = np.sum(_rope(orc, q, [1007], interleaved=inter) * _rope(orc, k, [1019], interleaved=inter))
        _close(s1, s2, 1e-11, 1e-12, "relative position")
        a = _rope(orc, _rope(orc, x, [5, 40, 7], interleaved=inter), [11, 2, 300], interleaved=inter)
        _close(a, _rope(orc, x, [16, 42, 307], interleaved=inter), 1e-12, 1e-13, "composition")
    # closed forms
    y = _rope(orc, np.array([[[1.0, 0.0]]]), [1])
    _close(y[0, 0], [math.cos(1.0), math.sin(1.0)], 1e-15, 1e-16, "Dh=2, p=1")
    y = _rope(orc, np.array([[[0.0, 2.0, 0.0, 0.0]]]), [5], base=100.0)
    # pair (1, 3): (x1, x3) = (2, 0) turns by theta_1 = 5 * 100^(-1/2) = 0.5
    _close(y[0, 0], [0.0, 2 * math.cos(0.5), 0.0, 2 * math.sin(0.5)], 1e-15, 1e-16, "Dh=4, base 100")
    # interleaved = rotate-half under the even/odd permutation
    x = rng.normal(size=(2, 3, 12))
    perm = np.concatenate([np.arange(0, 12, 2), np.arange(1, 12, 2)])
    half = _rope(orc, x[:, :, perm], [9, 77])
    inter = _rope(orc, x, [9, 77], interleaved=True)
    _close(inter[:, :, perm], half, 1e-14, 1e-15, "layouts")
    # table path
    Dh, base = 8, 500.0
    tab = np.zeros((64, Dh))
    for p in range(64):
        for i in range(Dh // 2):
            ang = p * math.pow(base, -2.0 * i / Dh)
            tab[p, i], tab[p, Dh // 2 + i] = math.cos(ang), math.sin(ang)
    x = rng.normal(size=(3, 2, Dh))
    _close(_rope(orc, x, [0, 17, 63], base=base, cos_sin=tab),
           _rope(orc, x, [0, 17, 63], base=base), 1e-13, 1e-14, "table = on the fly")


def pin_kv_append(orc):
    """The cache append: token t's rotated k and its v land in row slots[t];
    a negative slot writes nothing; rows no token names keep their contents;
    q's rotation does not depend on the slots; a ring cache (slot = position
    mod window) holds the same rows as the dense slab's last window."""
    rng = _rng(23)
    T, Hq, Hkv, Dh, S = 5, 4, 2, 8, 9
    q = rng.normal(size=(T, Hq, Dh))
    k = rng.normal(size=(T, Hkv, Dh))
    v = rng.normal(size=(T, Hkv, Dh))
    pos = np.array([3, 4, 5, 6, 7])
    slots = np.array([8, -1, 0, 2, 5])
    kc0 = rng.normal(size=(S, Hkv, Dh))
    vc0 = rng.normal(size=(S, Hkv, Dh))
    qo, kc, vc = orc.rope_kv_append(q, k, v, pos, slots, kc0, vc0)
    untouched = [r for r in range(S) if r not in slots]
    _close(kc[untouched], kc0[untouched], 0, 0, "untouched k rows")
    _close(vc[untouched], vc0[untouched], 0, 0, "untouched v rows")
    for t in range(T):
        if slots[t] >= 0:
            _close(vc[slots[t]], v[t], 0, 0, "v copied")
            # the cached k is k rotated like a q row at the same position
            _close(kc[slots[t]], _rope(orc, k[t:t + 1], [pos[t]])[0], 0, 0, "k rotated")
    qo2, _, _ = orc.rope_kv_append(q, k, v, pos, -np.ones(T, np.int64), kc0, vc0)
    _close(qo, qo2, 0, 0, "q independent of slots")
    # ring of window 4 vs dense slab
    T = 10
    k = rng.normal(size=(T, 1, Dh))
    v = rng.normal(size=(T, 1, Dh))
    pos = np.arange(100, 100 + T)
    z = np.zeros((T, 1, Dh))
    _, kd, vd = orc.rope_kv_append(z, k, v, pos, np.arange(T), np.zeros((T, 1, Dh)), np.zeros((T, 1, Dh)))
    _, kr, vr = orc.rope_kv_append(z, k, v, pos, pos % 4, np.zeros((4, 1, Dh)), np.zeros((4, 1, Dh)))
    for t in range(T - 4, T):
        _close(kr[pos[t] % 4], kd[t], 0, 0, "ring k")
        _close(vr[pos[t] % 4], vd[t], 0, 0, "ring v")


def pin_rstd(orc):
    """rstd is 1 / sqrt(||h||^2 / D + eps), written with a library norm, for
    h = x + residual and h = x; a constant row c gives 1 / sqrt(c^2 + eps);
    and the forward's out is exactly h * rstd * (weight_bias + w)."""
    rng = _rng(21)
    for R, D in ((4, 16), (3, 257), (1, 1)):
        x = rng.normal(size=(R, D)) * rng.uniform(0.1, 10, size=(R, 1))
        res = rng.normal(size=(R, D))
        eps = 1e-3
        for r in (None, res):
            h = x if r is None else x + r
            got = orc.rstd(x, eps, r)
            nrm = np.linalg.norm(h, axis=1)
            _close(got, 1.0 / np.sqrt(nrm ** 2 / D + orc.scalar(eps)), 1e-13, 0,
                   "rstd R=%d D=%d" % (R, D))
            w = rng.normal(1.0, 0.2, size=D)
            out, _ = orc.fwd(x, w, eps, 0.75, r)
            _close(out, h * got[:, None] * (0.75 + w), 1e-14, 1e-300, "out = h rstd w'")
    c = np.array([[2.5] * 6, [-0.125] * 6])
    _close(orc.rstd(c, 0.5), [1 / np.sqrt(6.25 + 0.5), 1 / np.sqrt(0.015625 + 0.5)], 1e-15, 0,
           "constant rows")


def pin_vjp_rstd(orc):
    """The VJP with a supplied per-row scale rho: a hand-worked two-row example
    (w' = [1, 2], rho = 0.5 and 2), D = 1's closed form
    gx = g w' rho (1 - rho^2 h^2), gw = g h rho, and the plain VJP when rho is
    the forward's rstd."""
    h = np.array([[1.0, 2.0], [0.0, 3.0]])
    g = np.array([[1.0, 0.0], [2.0, 1.0]])
    w = np.array([0.5, 1.5])  # w' = weight_bias + w = [1, 2] with weight_bias 0.5
    # row 0: dot = 1*1*1 = 1, rho^3/D = 1/16: gx = [1/2 - 1/16, -2/16]
    # row 1: dot = 1*2*3 = 6, rho^3/D = 4:    gx = [4, 4 - 72]
    # gw = [1*1*0.5 + 2*0*2, 0*2*0.5 + 1*3*2] = [0.5, 6]
    gx, gw = orc.vjp_rstd(h, w, g, [0.5, 2.0], 0.5)
    _close(gx, [[0.4375, -0.125], [4.0, -68.0]], 0, 0, "worked example gx")
    _close(gw, [0.5, 6.0], 0, 0, "worked example gw")
    a, gg, ww, rho = np.array([[-1.5], [0.75]]), np.array([[2.0], [-3.0]]), 0.25, np.array([0.3, 1.7])
    gx, gw = orc.vjp_rstd(a, np.array([ww]), gg, rho, 0.0)
    want = gg * ww * rho[:, None] * (1 - rho[:, None] ** 2 * a ** 2)
    _close(gx, want, 1e-14, 1e-16, "D=1 gx")
    _close(gw, [np.sum(gg[:, 0] * a[:, 0] * rho)], 1e-14, 0, "D=1 gw")
    rng = _rng(22)
    R, D = 5, 37
    x = rng.normal(size=(R, D)) * rng.uniform(0.5, 4, size=(R, 1))
    w = rng.normal(1.0, 0.2, size=D)
    g = rng.normal(size=(R, D))
    for eps, wb in ((1e-5, 0.0), (0.25, 1.0)):
        gx0, gw0 = orc.vjp(x, w, g, eps, wb)
        gx1, gw1 = orc.vjp_rstd(x, w, g, orc.rstd(x, eps), wb)
        _close(gx1, gx0, 1e-12, 1e-15, "vjp_rstd(rstd) = vjp gx")
        _close(gw1, gw0, 1e-12, 1e-15, "vjp_rstd(rstd) = vjp gw")


ALL_PINS = [
    pin_worked_examples,
    pin_constant_rows,
    pin_d1,
    pin_unit_weight_bias_plain_norm,
    pin_residual_is_added,
    pin_scale_invariance,
    pin_gw_row_sum,
    pin_finite_differences,
    pin_h_dot_gx_identity,
    pin_linearity_in_g,
    pin_row_permutation,
    pin_scaled_weight,
    pin_fused_vjp_finite_differences,
    pin_gated_silu,
    pin_rope,
    pin_kv_append,
    pin_rstd,
    pin_vjp_rstd,
]
