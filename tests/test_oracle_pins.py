"""Pins of the CPU oracle against facts that do not come from the oracle itself:
constants the pages print, closed forms, invariants, brute force on tiny
inputs and central finite differences. CPU only.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
import workload as W

HERE = os.path.dirname(os.path.abspath(__file__))


def golden():
    with open(os.path.join(HERE, "golden", "page_constants.json")) as f:
        return json.load(f)


def shape_of(w):
    return oracle.Shape(w.depth, w.d_model, w.n_head, w.vocab)


# ------------------------------------------------------------ layout / sizes

def test_dimension_rule_and_param_count():
    g = golden()
    for name in ("small", "gpt2_small", "d20", "d26"):
        w = W.WORKLOADS[name]
        assert w.d_model == g["d_model_per_depth"]["value"] * w.depth
        assert w.n_head == w.d_model // g["head_dim"]["value"]
        assert w.ffn == g["ffn_multiplier"]["value"] * w.d_model
        assert w.vocab == g["vocab"]["value"]
        s = shape_of(w)
        d, V, L = w.d_model, w.vocab, w.depth
        # two untied V x d tables + per layer 3d^2 + d^2 + 4d^2 + 4d^2
        assert oracle.param_count(s) == 2 * V * d + 12 * L * d * d
        assert oracle.param_count(s) == W.n_params(w)
    assert W.WORKLOADS["d20"].depth == g["speedrun_depth"]["value"]
    assert oracle.param_count(shape_of(W.WORKLOADS["d20"])) == 560_988_160


def test_layout_offsets_are_contiguous_and_ordered():
    s = shape_of(W.WORKLOADS["small"])
    lay = oracle.layout(s)
    names = [n for n, *_ in lay]
    assert names[0] == "wte" and names[-1] == "lm_head"
    assert names[1:5] == ["h0.w_qkv", "h0.w_o", "h0.w_fc", "h0.w_proj"]
    off = 0
    for _, o, r, c in lay:
        assert o == off and o % 128 == 0
        off += r * c


# ------------------------------------------------------------ RMSNorm

def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((7, 256)) * 3.0
    y, r = oracle.rmsnorm(z)
    ms = np.mean(z * z, axis=-1)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), ms / (ms + oracle.EPS), rtol=1e-12)
    y2, _ = oracle.rmsnorm(5.0 * z)
    np.testing.assert_allclose(y2, y, rtol=1e-6)
    # constant vector: y = c / sqrt(c^2 + eps)
    c = 0.25
    yc, _ = oracle.rmsnorm(np.full((1, 128), c))
    np.testing.assert_allclose(yc, c / math.sqrt(c * c + 1e-6), rtol=1e-14)
    # zero vector maps to zero (used by the attention closed form below)
    y0, _ = oracle.rmsnorm(np.zeros((1, 128)))
    assert np.all(y0 == 0)


def test_rmsnorm_backward_matches_finite_differences():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((3, 64))
    G = rng.standard_normal((3, 64))
    y, r = oracle.rmsnorm(z)
    an = oracle.rmsnorm_backward(G, y, r)
    h = 1e-6
    fd = np.zeros_like(z)
    for i in np.ndindex(z.shape):
        zp, zm = z.copy(), z.copy()
        zp[i] += h
        zm[i] -= h
        fd[i] = (np.sum(G * oracle.rmsnorm(zp)[0]) - np.sum(G * oracle.rmsnorm(zm)[0])) / (2 * h)
    np.testing.assert_allclose(an, fd, rtol=1e-6, atol=1e-9)


# ------------------------------------------------------------ RoPE

def test_rope_preserves_norm_and_is_identity_at_pos0():
    rng = np.random.default_rng(3)
    T, H, D = 50, 3, 128
    x = rng.standard_normal((T, H, D))
    cos, sin = oracle.rope_angles(T)
    y = oracle.rope(x, cos, sin)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    np.testing.assert_array_equal(y[0], x[0])


def test_rope_pairing_and_base():
    # dim 0 pairs with dim 64 and turns by exactly `pos` radians (theta_0 = 1);
    # dim 32 turns by pos * 10000^(-32/64) = pos / 100 radians.
    T = 301
    cos, sin = oracle.rope_angles(T)
    x = np.zeros((T, 1, 128))
    x[:, 0, 0] = 1.0
    x[:, 0, 32] = 1.0
    y = oracle.rope(x, cos, sin)
    pos = np.arange(T, dtype=np.float64)
    np.testing.assert_allclose(y[:, 0, 0], np.cos(pos), atol=1e-12)
    np.testing.assert_allclose(y[:, 0, 64], np.sin(pos), atol=1e-12)
    np.testing.assert_allclose(y[:, 0, 32], np.cos(pos / 100.0), atol=1e-12)
    np.testing.assert_allclose(y[:, 0, 96], np.sin(pos / 100.0), atol=1e-12)
    other = np.delete(np.arange(128), [0, 32, 64, 96])
    assert np.all(y[:, 0, other] == 0)


def test_rope_relative_position_property():
    # <R_m q, R_n k> depends only on n - m ("RoPE Intuition")
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    vals = []
    for shift in (0, 17, 900):
        cm, sm = oracle.rope_angles(1, offset=5 + shift)
        cn, sn = oracle.rope_angles(1, offset=12 + shift)
        vals.append(float(np.sum(oracle.rope(q, cm, sm) * oracle.rope(k, cn, sn))))
    np.testing.assert_allclose(vals, vals[0], rtol=1e-10)


def test_rope_backward_is_transpose():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((9, 2, 128))
    g = rng.standard_normal((9, 2, 128))
    cos, sin = oracle.rope_angles(9)
    lhs = np.sum(oracle.rope(x, cos, sin) * g)
    rhs = np.sum(x * oracle.rope_backward(g, cos, sin))
    assert abs(lhs - rhs) < 1e-10 * max(1.0, abs(lhs))


# ------------------------------------------------------------ attention

def brute_attention(q, k, v):
    """Scalar-loop causal attention on tiny inputs (math.exp, explicit sums)."""
    T, H, D = q.shape
    o = np.zeros_like(q)
    for h in range(H):
        for t in range(T):
            sc = [sum(q[t, h, e] * k[j, h, e] for e in range(D)) / math.sqrt(D) for j in range(t + 1)]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            z = sum(w)
            for e in range(D):
                o[t, h, e] = sum(w[j] * v[j, h, e] for j in range(t + 1)) / z
    return o


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(6)
    q, k, v = (rng.standard_normal((5, 2, 128)) for _ in range(3))
    o, _ = oracle.causal_attention(q, k, v)
    np.testing.assert_allclose(o, brute_attention(q, k, v), rtol=1e-10, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(7)
    T, H, D = 33, 2, 128
    v = rng.standard_normal((T, H, D))
    # T = 1: the only key is the query's own position -> o = v
    o1, lse1 = oracle.causal_attention(rng.standard_normal((1, H, D)), rng.standard_normal((1, H, D)), v[:1])
    np.testing.assert_allclose(o1, v[:1], rtol=1e-14)
    # q = 0: uniform weights -> o_t = mean(v_0..v_t), lse = log(t+1)
    o, lse = oracle.causal_attention(np.zeros((T, H, D)), rng.standard_normal((T, H, D)), v)
    prefix = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None, None]
    np.testing.assert_allclose(o, prefix, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.arange(1, T + 1))[None, :].repeat(H, 0), rtol=1e-12)
    # two keys k0 = q, k1 = -q: p0 = 1 / (1 + exp(-2 |q|^2 / sqrt(D))) pins the 1/sqrt(D) scale
    qv = rng.standard_normal(D) * 0.1
    q2 = np.zeros((2, 1, D))
    q2[1, 0] = qv
    k2 = np.stack([qv, -qv])[:, None, :]
    v2 = np.zeros((2, 1, D))
    v2[0, 0, 0] = 1.0
    o2, _ = oracle.causal_attention(q2, k2, v2)
    p0 = 1.0 / (1.0 + math.exp(-2.0 * float(qv @ qv) / math.sqrt(D)))
    assert abs(o2[1, 0, 0] - p0) < 1e-13


def test_attention_causality_bitwise():
    rng = np.random.default_rng(8)
    q, k, v = (rng.standard_normal((16, 2, 128)) for _ in range(3))
    o, _ = oracle.causal_attention(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[9:] += 3.0
    v2[9:] -= 1.0
    o2, _ = oracle.causal_attention(q, k2, v2)
    np.testing.assert_array_equal(o[:9], o2[:9])
    assert not np.allclose(o[9:], o2[9:])


def test_attention_backward_matches_finite_differences():
    rng = np.random.default_rng(9)
    T, H, D = 6, 2, 128
    q, k, v = (rng.standard_normal((T, H, D)) * 0.5 for _ in range(3))
    G = rng.standard_normal((T, H, D))
    dq, dk, dv = oracle.causal_attention_backward(q, k, v, G)

    def f(q_, k_, v_):
        return float(np.sum(oracle.causal_attention(q_, k_, v_)[0] * G))

    h = 1e-6
    for arr, an, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        idx = [tuple(rng.integers(0, s) for s in arr.shape) for _ in range(24)]
        for i in idx:
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][i] += h
            args_m[which][i] -= h
            fd = (f(*args_p) - f(*args_m)) / (2 * h)
            assert abs(fd - an[i]) <= 1e-5 * max(abs(fd), abs(an[i])) + 1e-9, (which, i, fd, an[i])


# ------------------------------------------------------------ ReLU^2, CE

def test_relu2_exact_zeros_and_values():
    u = np.array([-3.0, -1e-30, 0.0, 1e-3, 2.0, 7.5])
    a = oracle.relu2(u)
    assert np.all(a[:3] == 0.0)
    np.testing.assert_array_equal(a[3:], np.array([1e-6, 4.0, 56.25]))
    np.testing.assert_array_equal(oracle.relu2_backward(np.ones(6), u), np.array([0, 0, 0, 2e-3, 4.0, 15.0]))


def test_cross_entropy_uniform_and_ties():
    V, d, M = 4096, 16, 10
    rng = np.random.default_rng(10)
    hf = rng.standard_normal((M, d))
    tgt = rng.integers(0, V, M)
    lse, nll, amax = oracle.cross_entropy_rows(hf, np.zeros((V, d)), tgt)
    np.testing.assert_allclose(nll, math.log(V), rtol=1e-15)
    assert np.all(amax == 0)  # all logits tie -> lowest index
    # a row whose logits tie at two ids picks the lower one
    w = np.zeros((V, d))
    w[17, 0] = 1.0
    w[5, 0] = 1.0
    h1 = np.zeros((1, d))
    h1[0, 0] = 2.0
    _, _, am = oracle.cross_entropy_rows(h1, w, np.array([0]))
    assert am[0] == 5


# ------------------------------------------------------------ whole step

def tiny_case(vocab=None):
    w = W.WORKLOADS["tiny"]
    if vocab is not None:
        w = w.with_vocab(vocab)
    p = W.make_params(w).astype(np.float64)
    tok, tgt = W.make_tokens(w)
    return w, shape_of(w), p, tok, tgt


def test_zero_lm_head_gives_ln_vocab_and_closed_form_grads():
    g = golden()
    w, s, p, tok, tgt = tiny_case()
    off = oracle.layout(s)[-1][1]
    p[off:] = 0.0
    loss, grads, cache = oracle.step(p, tok, tgt, s, np.float64)
    assert abs(loss - g["ln_vocab"]["value"]) < 1e-12
    assert abs(math.log(w.vocab) - g["ln_vocab"]["value"]) < 1e-15
    # nothing upstream of lm_head receives gradient
    assert np.all(grads[:off] == 0.0)
    # dW_lm = (1/M) sum_t (1/V - onehot(tgt_t)) hf_t with hf from the forward
    M, d, V = w.tokens, w.d_model, w.vocab
    hf = cache["hf"].reshape(M, d)
    expect = np.tile(hf.sum(0) / (V * M), (V, 1))
    np.subtract.at(expect, tgt.reshape(M), hf / M)
    np.testing.assert_allclose(grads[off:].reshape(V, d), expect, rtol=1e-10, atol=1e-16)


def test_zero_blocks_reduce_to_softmax_regression():
    # with every block matrix zero the residual stream is the embedding, so
    # the model is softmax regression on rmsnorm(wte[tok]).
    from scipy.special import logsumexp
    w, s, p, tok, tgt = tiny_case(vocab=2048)
    lay = oracle.layout(s)
    for name, off, r, c in lay[1:-1]:
        p[off:off + r * c] = 0.0
    P = oracle.unpack(p, s)
    loss, grads, _ = oracle.step(p, tok, tgt, s, np.float64)
    e = P["wte"][tok.reshape(-1)]
    hf = e / np.sqrt(np.mean(e * e, axis=1, keepdims=True) + 1e-6)
    logits = hf @ P["lm_head"].T
    ref = np.mean(logsumexp(logits, axis=1) - logits[np.arange(len(logits)), tgt.reshape(-1)])
    assert abs(loss - ref) < 1e-12
    # every block gradient has a zero factor (o = 0, a = 0, and W_o = W_proj = 0
    # stop the gradient flowing into the blocks), so all of them are exactly 0
    for name, off, r, c in lay[1:-1]:
        assert np.all(grads[off:off + r * c] == 0.0), name
    assert np.any(grads[lay[0][1]:lay[1][1]] != 0.0)


def test_causality_of_whole_model():
    w, s, p, tok, tgt = tiny_case(vocab=4096)
    _, c1 = oracle.forward(p, tok, tgt, s, np.float64)
    tok2 = tok.copy()
    t = 37
    tok2[:, t] = (tok2[:, t] + 1000) % w.vocab
    _, c2 = oracle.forward(p, tok2, tgt, s, np.float64)
    B, T = tok.shape
    lse1, lse2 = c1["lse"].reshape(B, T), c2["lse"].reshape(B, T)
    np.testing.assert_array_equal(lse1[:, :t], lse2[:, :t])
    np.testing.assert_array_equal(c1["nll"].reshape(B, T)[:, :t], c2["nll"].reshape(B, T)[:, :t])
    assert np.all(lse1[:, t] != lse2[:, t])


def central(f, p, e, h):
    """Central difference of f at p along e, Richardson-extrapolated over
    steps h and h/2 so that the O(h^2) truncation term cancels."""
    d1 = (f(p + h * e) - f(p - h * e)) / (2 * h)
    h2 = h / 2
    d2 = (f(p + h2 * e) - f(p - h2 * e)) / (2 * h2)
    return (4 * d2 - d1) / 3


def _fd_check(w, s, p, tok, tgt, coords_per_tensor, seed, directional=True):
    loss, grads, _ = oracle.step(p, tok, tgt, s, np.float64)
    rng = np.random.default_rng(seed)

    def f(pp):
        return oracle.forward(pp, tok, tgt, s, np.float64, keep=False)[0]

    present = np.unique(tok)
    failures = []
    for name, off, r, c in oracle.layout(s):
        n = r * c
        if name == "wte":
            rows = np.concatenate([rng.choice(present, coords_per_tensor // 2),
                                   rng.integers(0, r, coords_per_tensor - coords_per_tensor // 2)])
            idx = rows * c + rng.integers(0, c, len(rows))
            absent = np.setdiff1d(np.arange(r), present)
            # rows no token uses get exactly zero gradient
            assert np.all(grads[off:off + n].reshape(r, c)[absent] == 0.0)
        else:
            idx = rng.integers(0, n, coords_per_tensor)
        for i in idx:
            j = off + int(i)
            e = np.zeros_like(p)
            e[j] = 1.0
            fd = central(f, p, e, 1e-4 * max(1.0, abs(p[j])))
            an = grads[j]
            if not abs(fd - an) <= 1e-3 * max(abs(fd), abs(an)) + 1e-12:
                failures.append((name, int(i), fd, an))
        if directional:
            dvec = np.zeros_like(p)
            dvec[off:off + n] = rng.standard_normal(n)
            fd = central(f, p, dvec, 1e-3 / math.sqrt(n))
            an = float(grads @ dvec)
            if not abs(fd - an) <= 1e-3 * max(abs(fd), abs(an)) + 1e-12:
                failures.append((name, "dir", fd, an))
    assert not failures, failures


def test_finite_differences_tiny_reduced_vocab():
    # the tiny workload's shapes with a 1024-id vocabulary: 32 coordinates
    # per parameter tensor plus one random direction per tensor
    w, s, p, tok, tgt = tiny_case(vocab=1024)
    _fd_check(w, s, p, tok, tgt, coords_per_tensor=32, seed=11)


def test_finite_differences_tiny_full_vocab():
    # the tiny workload exactly (65,536 ids): fewer coordinates, same criterion
    w, s, p, tok, tgt = tiny_case()
    _fd_check(w, s, p, tok, tgt, coords_per_tensor=2, seed=12)


def test_float32_oracle_tracks_float64():
    w, s, p, tok, tgt = tiny_case(vocab=4096)
    l64, g64, _ = oracle.step(p, tok, tgt, s, np.float64)
    l32, g32, _ = oracle.step(p.astype(np.float32), tok, tgt, s, np.float32)
    assert abs(l64 - l32) < 1e-5
    for name, off, r, c in oracle.layout(s):
        a, b = g64[off:off + r * c], g32[off:off + r * c].astype(np.float64)
        assert np.linalg.norm(a - b) <= 1e-4 * np.linalg.norm(a) + 1e-30, name


def test_inputs_are_deterministic_and_zipf_shaped():
    w = W.WORKLOADS["small"]
    t1, g1 = W.make_tokens(w)
    t2, g2 = W.make_tokens(w)
    np.testing.assert_array_equal(t1, t2)
    np.testing.assert_array_equal(t1[:, 1:], g1[:, :-1])  # targets are the next token
    assert t1.min() >= 0 and t1.max() < w.vocab
    # Zipf(1.1) over 65,536 ranks: P(id 0) = 1 / H_{65536,1.1}
    p0 = 1.0 / np.sum(np.arange(1, 65537, dtype=np.float64) ** -1.1)
    frac0 = np.mean(t1 == 0)
    assert abs(frac0 - p0) < 0.02
    p = W.make_params(w)
    assert np.all(W.round_bf16(p) == p)


# ------------------------------------------------------------ SFT: masked loss

def test_masked_loss_is_the_mean_over_response_positions():
    # explainer, "Supervised Fine-Tuning (SFT)": the same cross-entropy, only
    # on the response tokens. Masking changes nothing before the loss, so the
    # masked loss is the mean of the unmasked run's per-position losses over
    # the kept positions, and masked positions report nll 0.
    w, s, p, tok, tgt = tiny_case(vocab=1024)
    sft = W.make_sft_targets(tgt, seed=3, mean_turn=16)
    keep = sft != oracle.IGNORE
    assert 0 < keep.sum() < keep.size
    _, full = oracle.forward(p, tok, tgt, s, np.float64, keep=False)
    loss, masked = oracle.forward(p, tok, sft, s, np.float64, keep=False)
    assert abs(loss - float(np.mean(full["nll"][keep.reshape(-1)]))) < 1e-12
    assert np.all(masked["nll"][~keep.reshape(-1)] == 0.0)
    np.testing.assert_array_equal(masked["lse"], full["lse"])


def test_fully_masked_batch_has_zero_loss_and_zero_gradient():
    w, s, p, tok, tgt = tiny_case(vocab=1024)
    none = np.full_like(tgt, oracle.IGNORE)
    loss, grads, _ = oracle.step(p, tok, none, s, np.float64)
    assert loss == 0.0 and not np.any(grads)


def test_finite_differences_masked_loss():
    # the analytic backward of the masked mean, against central differences
    w, s, p, tok, tgt = tiny_case(vocab=1024)
    sft = W.make_sft_targets(tgt, seed=4, mean_turn=16)
    _fd_check(w, s, p, tok, sft, coords_per_tensor=8, seed=13)
