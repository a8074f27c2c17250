"""Pins of the oracle's pre-core and post-core steps (oracle/prepost.py) against closed forms
and the definitions on the pages (Kimi K3 wiki, "Notations mathématiques", table "Fonctions";
"Glossaire", entry "Décroissance bornée"; "Tableau des spécifications"). CPU only."""
import math

import numpy as np
import pytest

from oracle import prepost


def test_sigmoid_closed_forms():
    assert prepost.sigmoid(0.0) == 0.5
    assert prepost.sigmoid(math.log(3.0)) == pytest.approx(0.75, abs=1e-15)
    x = np.linspace(-30, 30, 61)
    assert np.allclose(prepost.sigmoid(x) + prepost.sigmoid(-x), 1.0, atol=1e-15)


def test_decay_gate_values_and_range():
    H, d = 3, 4
    z = np.zeros((2, H, d))
    A = np.zeros(H)
    b = np.zeros((H, d))
    assert np.all(prepost.decay_gate(z, A, b) == -2.5)  # g_min * sigma(0), g_min = -5
    # e^{A_h} scales the logit: A = ln 2, z = ln(3) / 2 gives sigma(ln 3) = 3/4
    A2 = np.array([0.0, math.log(2.0), 0.0])
    z2 = np.full((1, H, d), math.log(3.0) / 2)
    g = prepost.decay_gate(z2, A2, b)
    assert g[0, 1] == pytest.approx(np.full(d, -3.75), abs=1e-14)
    assert g[0, 0] == pytest.approx(np.full(d, -5.0 * prepost.sigmoid(math.log(3.0) / 2)), abs=1e-14)
    # the bias shifts the logit: z = 0, b = ln 3 -> -3.75
    b3 = np.full((H, d), math.log(3.0))
    assert np.allclose(prepost.decay_gate(z, A, b3), -3.75, atol=1e-14)
    # bounded decay: g in (g_min, 0) for any finite logit; the limits are g_min and 0
    zz = np.linspace(-30, 30, 7).reshape(1, 1, 7)
    gg = prepost.decay_gate(zz, np.zeros(1), np.zeros((1, 7)))
    assert np.all(gg < 0) and np.all(gg > -5.0)
    assert gg[0, 0, -1] == pytest.approx(-5.0, abs=1e-10) and gg[0, 0, 0] == pytest.approx(0.0, abs=1e-10)


def test_l2norm():
    assert np.allclose(prepost.l2norm(np.array([3.0, 4.0])), [0.6, 0.8], atol=1e-16)
    x = np.random.default_rng(0).normal(size=(5, 7, 128))
    n = prepost.l2norm(x)
    assert np.allclose(np.linalg.norm(n, axis=-1), 1.0, atol=1e-14)
    assert np.allclose(prepost.l2norm(3.5 * x), n, atol=1e-15)  # scale invariant


def test_rmsnorm_closed_forms():
    d = 8
    c = 0.3
    x = np.full(d, c)
    assert np.allclose(prepost.rmsnorm(x, np.ones(d), eps=1e-5), c / math.sqrt(c * c + 1e-5), atol=1e-15)
    assert np.allclose(prepost.rmsnorm(np.array([3.0, 4.0]), np.ones(2), eps=0.0),
                       np.array([3.0, 4.0]) / math.sqrt(12.5), atol=1e-15)
    w = np.arange(1, d + 1, dtype=float)
    y = prepost.rmsnorm(np.ones(d), w, eps=0.0)
    assert np.allclose(y, w, atol=1e-15)  # the weight scales channel by channel
    # with eps = 0 the mean square of the output (w = 1) is exactly 1
    r = np.random.default_rng(1).normal(size=(3, 128))
    assert np.allclose(np.mean(prepost.rmsnorm(r, np.ones(128), eps=0.0) ** 2, axis=-1), 1.0,
                       atol=1e-14)


def test_short_conv_impulse_causality_and_restart():
    B, T, H, d = 1, 12, 2, 3
    rng = np.random.default_rng(2)
    w = rng.normal(size=(H, d, 4))
    x = np.zeros((B, T, H, d))
    t0 = 5
    x[0, t0] = 1.0
    y = prepost.short_conv(x, w)
    for t in range(T):
        exp = w[..., t - t0] if 0 <= t - t0 <= 3 else np.zeros((H, d))
        assert np.allclose(y[0, t], exp, atol=0)
    # the identity filter gives x back; a zero filter gives zero
    xr = rng.normal(size=(B, T, H, d))
    ident = np.zeros((H, d, 4))
    ident[..., 0] = 1.0
    assert np.array_equal(prepost.short_conv(xr, ident), xr)
    assert not prepost.short_conv(xr, np.zeros((H, d, 4))).any()
    # causal: changing a token changes no earlier output
    x2 = xr.copy()
    x2[0, 7] += 10.0
    d2 = prepost.short_conv(x2, w) - prepost.short_conv(xr, w)
    assert not d2[0, :7].any() and d2[0, 7:11].any() and not d2[0, 11:].any()
    # packed batch: the convolution restarts at every sequence start
    cu = [0, 4, 12]
    yp = prepost.short_conv(xr, w, cu)
    y1 = prepost.short_conv(xr[:, :4], w)
    y2 = prepost.short_conv(xr[:, 4:], w)
    assert np.allclose(yp, np.concatenate([y1, y2], axis=1), atol=0)


def test_post_core_limits():
    rng = np.random.default_rng(3)
    o = rng.normal(size=(2, 5, 3, 16))
    w = rng.normal(size=16)
    n = prepost.rmsnorm(o, w)
    assert np.allclose(prepost.post_core(o, np.full(o.shape, 50.0), w), n, atol=1e-15)
    assert np.allclose(prepost.post_core(o, np.zeros(o.shape), w), 0.5 * n, atol=1e-15)
