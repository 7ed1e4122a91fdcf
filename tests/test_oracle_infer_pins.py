"""Pins of the KV-cache generation oracle (oracle/infer.py) against the full
forward of oracle.model, which the other pins fix: a decode step must give
the logits the full forward gives at the same position of the extended
sequence. CPU only."""

import numpy as np

import oracle
import workload as W
from oracle import infer


def _case(vocab=512, depth=2, T0=12, B=2, seed=0):
    s = oracle.Shape(depth, 128, 1, vocab)
    rng = np.random.default_rng(seed)
    p = rng.standard_normal(oracle.param_count(s)) * 0.05
    tok = rng.integers(0, vocab, (B, T0))
    return s, p, tok


def _full_logits(p, tok, s):
    _, cache = oracle.forward(p, tok, np.zeros_like(tok), s, np.float64, keep=True)
    P = oracle.unpack(p, s)
    B, T = tok.shape
    return cache["hf"].reshape(B, T, -1) @ P["lm_head"].T     # [B, T, V]


def test_prefill_logits_equal_the_full_forward_at_the_last_position():
    s, p, tok = _case()
    cache, logits = infer.prefill(p, tok, s)
    np.testing.assert_allclose(logits, _full_logits(p, tok, s)[:, -1], rtol=1e-12, atol=1e-12)
    assert cache["pos"] == tok.shape[1] and len(cache["k"]) == s.depth
    assert cache["k"][0].shape == (tok.shape[0], tok.shape[1], s.n_head, 128)


def test_decode_step_equals_the_full_forward_of_the_extended_sequence():
    s, p, tok = _case(seed=1)
    cache, _ = infer.prefill(p, tok[:, :-1], s)
    _, logits = infer.decode_step(p, cache, tok[:, -1], s)
    np.testing.assert_allclose(logits, _full_logits(p, tok, s)[:, -1], rtol=1e-10, atol=1e-10)


def test_decode_from_a_one_token_prompt():
    # the shortest cache: the second position attends to exactly two keys
    s, p, tok = _case(T0=2, seed=2)
    cache, _ = infer.prefill(p, tok[:, :1], s)
    _, logits = infer.decode_step(p, cache, tok[:, 1], s)
    np.testing.assert_allclose(logits, _full_logits(p, tok, s)[:, -1], rtol=1e-10, atol=1e-10)


def test_greedy_generation_is_consistent_with_the_full_forward():
    # every generated id is the argmax the full forward assigns to the
    # previous position of the generated sequence, and the logits agree
    s, p, prompt = _case(T0=8, seed=3)
    ids, logits = infer.generate(p, prompt, 5, s)
    seq = np.concatenate([prompt, ids[:, :-1]], axis=1)
    full = _full_logits(p, seq, s)
    T0 = prompt.shape[1]
    for i in range(ids.shape[1]):
        np.testing.assert_allclose(logits[i], full[:, T0 - 1 + i], rtol=1e-10, atol=1e-10)
        np.testing.assert_array_equal(ids[:, i], np.argmax(full[:, T0 - 1 + i], axis=-1))


def test_decode_does_not_modify_the_cache_it_is_given():
    s, p, tok = _case(seed=4)
    cache, _ = infer.prefill(p, tok, s)
    k0 = [k.copy() for k in cache["k"]]
    new, _ = infer.decode_step(p, cache, tok[:, 0], s)
    assert all(np.array_equal(a, b) for a, b in zip(k0, cache["k"]))
    assert new["pos"] == cache["pos"] + 1 and new["k"][0].shape[1] == cache["k"][0].shape[1] + 1
