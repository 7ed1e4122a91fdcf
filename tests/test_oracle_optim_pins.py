"""Pins of the optimizer oracle (clipping, AdamW, Muon / Newton-Schulz, the
learning-rate schedule) against closed forms, spectral identities and
invariants that do not come from the oracle's own code. CPU only.
"""

import json
import math
import os

import numpy as np

import oracle
from oracle import optim

HERE = os.path.dirname(os.path.abspath(__file__))


def golden():
    with open(os.path.join(HERE, "golden", "page_constants.json")) as f:
        return json.load(f)


def tiny_shape():
    return oracle.Shape(2, 128, 1, 256)


# ------------------------------------------------------------ groups, constants

def test_groups_cover_the_layout_once_and_follow_the_pages_split():
    g = golden()
    assert g["max_grad_norm"]["value"] == optim.Hyper().max_grad_norm
    assert g["weight_decay"]["value"] == optim.Hyper().weight_decay
    s = tiny_shape()
    a, m = optim.groups(s)
    assert [n for n, *_ in a] == g["optimizer_groups"]["value"]["adamw"]
    assert len(m) == 4 * s.depth
    covered = sorted((off, off + r * c) for _, off, r, c in a + m)
    assert covered[0][0] == 0 and covered[-1][1] == oracle.param_count(s)
    assert all(covered[i][1] == covered[i + 1][0] for i in range(len(covered) - 1))
    assert all(min(r, c) >= 2 for _, _, r, c in m)  # every Muon parameter is a 2-D matrix


# ------------------------------------------------------------ clipping

def test_clip_scale_on_a_pythagorean_triple_and_invariants():
    norm, k = optim.clip_scale(np.array([3.0, 4.0]), 1.0)
    assert norm == 5.0 and abs(k - 1.0 / (5.0 + 1e-6)) < 1e-15
    rng = np.random.default_rng(0)
    g = rng.standard_normal(1000)
    for max_norm in (0.5, 1.0, 1e3):
        norm, k = optim.clip_scale(g, max_norm)
        clipped = g * k
        assert abs(np.sqrt(np.sum(clipped ** 2)) - min(norm, max_norm)) <= 1e-5 * max_norm
        assert k <= 1.0
    assert optim.clip_scale(np.zeros(10), 1.0) == (0.0, 1.0)


# ------------------------------------------------------------ AdamW

def test_adamw_constant_gradient_closed_form():
    # with bias correction, a constant gradient gives m_hat = g and v_hat = g^2
    # exactly at every step, so p_k = c^k p0 - delta (1 - c^k) / (1 - c) with
    # c = 1 - lr wd and delta = lr g / (|g| + eps)
    rng = np.random.default_rng(1)
    p0 = rng.standard_normal(64)
    g = rng.standard_normal(64) * 1e-3
    lr, wd, eps = 1e-2, 0.1, 1e-8
    p, m, v = p0.copy(), np.zeros(64), np.zeros(64)
    for t in range(1, 6):
        p, m, v = optim.adamw(p, g, m, v, t, lr, 0.9, 0.999, eps, wd)
        c = 1.0 - lr * wd
        delta = lr * g / (np.abs(g) + eps)
        want = c ** t * p0 - delta * (1.0 - c ** t) / (1.0 - c)
        np.testing.assert_allclose(p, want, rtol=1e-9, atol=1e-12)


def test_adamw_two_steps_by_expanded_sums():
    rng = np.random.default_rng(2)
    p0, g1, g2 = rng.standard_normal((3, 32))
    b1, b2, lr, eps, wd = 0.8, 0.95, 0.1, 1e-8, 0.0
    p, m, v = optim.adamw(p0, g1, 0 * p0, 0 * p0, 1, lr, b1, b2, eps, wd)
    p, m, v = optim.adamw(p, g2, m, v, 2, lr, b1, b2, eps, wd)
    m2 = (b1 * (1 - b1) * g1 + (1 - b1) * g2) / (1 - b1 * b1)
    v2 = (b2 * (1 - b2) * g1 ** 2 + (1 - b2) * g2 ** 2) / (1 - b2 * b2)
    step1 = g1 / (np.abs(g1) + eps)
    np.testing.assert_allclose(p, p0 - lr * step1 - lr * m2 / (np.sqrt(v2) + eps), rtol=1e-12)


def test_adamw_zero_gradient_is_pure_decay():
    p0 = np.linspace(-1, 1, 9)
    p, _, _ = optim.adamw(p0, np.zeros(9), np.zeros(9), np.zeros(9), 1, 0.5, 0.9, 0.999, 1e-8, 0.1)
    np.testing.assert_allclose(p, p0 * (1 - 0.05), rtol=1e-15)


# ------------------------------------------------------------ Newton-Schulz

def _scalar_poly(x, steps, coeffs):
    a, b, c = coeffs
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def test_newton_schulz_acts_on_singular_values_only():
    # an odd matrix polynomial in X X^T maps U S V^T to U f(S) V^T: the
    # iteration equals the scalar polynomial applied to the normalised
    # singular values of an SVD, in either orientation
    rng = np.random.default_rng(3)
    for shape in ((16, 48), (48, 16), (24, 24)):
        G = rng.standard_normal(shape)
        U, S, Vt = np.linalg.svd(G, full_matrices=False)
        f = _scalar_poly(S / (np.sqrt(np.sum(S ** 2)) + optim.NS_EPS), 5, optim.NS_COEFFS)
        np.testing.assert_allclose(optim.newton_schulz(G), (U * f) @ Vt, atol=1e-10)


def test_newton_schulz_invariances_and_band():
    rng = np.random.default_rng(4)
    G = rng.standard_normal((32, 96))
    X = optim.newton_schulz(G)
    np.testing.assert_allclose(optim.newton_schulz(G.T), X.T, atol=1e-12)
    np.testing.assert_allclose(optim.newton_schulz(7.5 * G), X, atol=1e-8)
    # aspect ratio 3: every normalised singular value starts above 0.03, and
    # five quintic steps land them in the published band of roughly (0.7, 1.2)
    sv = np.linalg.svd(X, compute_uv=False)
    assert sv.min() > 0.68 and sv.max() < 1.2
    # exact rows of an orthogonal matrix: all singular values 1/sqrt(r) map to
    # the scalar iterate of 1/sqrt(r)
    Q, _ = np.linalg.qr(rng.standard_normal((96, 96)))
    Xq = optim.newton_schulz(Q[:32])
    want = _scalar_poly(1.0 / (math.sqrt(32) + optim.NS_EPS), 5, optim.NS_COEFFS)
    np.testing.assert_allclose(np.linalg.svd(Xq, compute_uv=False), want, rtol=1e-9)


def test_cubic_newton_schulz_converges_to_the_polar_factor():
    # with the classic cubic coefficients (1.5, -0.5, 0) the same iteration
    # converges to U V^T; checks the iteration's structure independently of
    # the quintic coefficients
    rng = np.random.default_rng(5)
    G = rng.standard_normal((12, 20)) + 3 * np.eye(12, 20)
    U, _, Vt = np.linalg.svd(G, full_matrices=False)
    X = optim.newton_schulz(G, steps=60, coeffs=(1.5, -0.5, 0.0))
    np.testing.assert_allclose(X, U @ Vt, atol=1e-9)


# ------------------------------------------------------------ Muon

def test_muon_constant_gradient_moves_along_the_orthogonalised_gradient():
    # buf_k = g (1 - mu^k) / (1 - mu) and u_k = g + mu buf_k are positive
    # multiples of g, so (NS being scale invariant) every step moves by
    # -lr sqrt(max(1, r/c)) NS(g) on top of the decay
    rng = np.random.default_rng(6)
    for r, c in ((48, 16), (16, 64)):
        p0 = rng.standard_normal((r, c))
        g = rng.standard_normal((r, c))
        mu, lr, wd = 0.95, 0.02, 0.1
        p, buf = p0.copy(), np.zeros((r, c))
        O = optim.newton_schulz(g)
        scale = math.sqrt(max(1.0, r / c))
        for k in range(1, 4):
            prev = p
            p, buf = optim.muon(p, g, buf, lr, mu, wd)
            np.testing.assert_allclose(buf, g * (1 - mu ** k) / (1 - mu), rtol=1e-12)
            np.testing.assert_allclose(p, prev * (1 - lr * wd) - lr * scale * O, atol=1e-7)


def test_muon_two_steps_use_the_nesterov_combination():
    # buf_2 = mu g1 + g2 and the Nesterov update direction is
    # u_2 = g2 + mu buf_2 = mu^2 g1 + (1 + mu) g2 (plain momentum would use buf_2)
    rng = np.random.default_rng(8)
    p0, g1, g2 = rng.standard_normal((3, 16, 40))
    mu, lr = 0.95, 0.05
    p, buf = optim.muon(p0, g1, np.zeros_like(p0), lr, mu, 0.0)
    p, buf = optim.muon(p, g2, buf, lr, mu, 0.0)
    np.testing.assert_allclose(buf, mu * g1 + g2, rtol=1e-14)
    want = p0 - lr * optim.newton_schulz(g1) - lr * optim.newton_schulz(mu * mu * g1 + (1 + mu) * g2)
    np.testing.assert_allclose(p, want, atol=1e-12)


# ------------------------------------------------------------ schedule

def test_lr_schedule_landmarks():
    peak, w, T, f = 0.02, 10, 110, 0.1
    assert optim.lr_at(0, w, T, peak, f) == peak / w
    assert optim.lr_at(w - 1, w, T, peak, f) == peak
    assert abs(optim.lr_at(w, w, T, peak, f) - peak) < 1e-15
    assert abs(optim.lr_at(w + 50, w, T, peak, f) - peak * (1 + f) / 2) < 1e-15
    assert abs(optim.lr_at(T, w, T, peak, f) - f * peak) < 1e-15
    assert abs(optim.lr_at(T + 5, w, T, peak, f) - f * peak) < 1e-15
    lrs = [optim.lr_at(t, w, T, peak, f) for t in range(w, T + 1)]
    assert all(a >= b for a, b in zip(lrs, lrs[1:]))


# ------------------------------------------------------------ whole step

def test_optimizer_step_routes_groups_and_clips_globally():
    s = tiny_shape()
    rng = np.random.default_rng(7)
    P = oracle.param_count(s)
    master = rng.standard_normal(P) * 0.02
    grads = rng.standard_normal(P) * 0.01  # norm ~ 20: clipped
    a, m = optim.groups(s)
    st0 = optim.init_state(master, s)
    # no Muon learning rate and no decay: the block matrices stay put
    h = optim.Hyper(lr_muon=0.0, weight_decay=0.0)
    out, st, norm, k = optim.optimizer_step(master, grads, st0, s, h)
    assert st["t"] == 1
    assert abs(norm - np.linalg.norm(grads)) < 1e-9 * norm and abs(k - 1.0 / (norm + 1e-6)) < 1e-15
    for name, off, r, c in m:
        assert np.array_equal(out[off:off + r * c], master[off:off + r * c])
        # the momentum saw the clipped gradient
        np.testing.assert_allclose(st["buf:" + name].reshape(-1), grads[off:off + r * c] * k, rtol=1e-12)
    for name, off, r, c in a:
        np.testing.assert_allclose(st["m:" + name].reshape(-1), 0.1 * k * grads[off:off + r * c], rtol=1e-12)
        assert not np.array_equal(out[off:off + r * c], master[off:off + r * c])
    # no AdamW learning rate and no decay: wte and lm_head stay put
    h = optim.Hyper(lr_adamw=0.0, weight_decay=0.0)
    out, *_ = optim.optimizer_step(master, grads, st0, s, h)
    for name, off, r, c in a:
        assert np.array_equal(out[off:off + r * c], master[off:off + r * c])
    for name, off, r, c in m:
        d = (out[off:off + r * c] - master[off:off + r * c]).reshape(r, c)
        want = -h.lr_muon * math.sqrt(max(1, r / c)) * optim.newton_schulz(grads[off:off + r * c].reshape(r, c))
        # first step: u = (1 + mu) k g, and NS is scale invariant up to its eps
        np.testing.assert_allclose(d, want, rtol=0, atol=1e-5 * np.abs(want).max())
