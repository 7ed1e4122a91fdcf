"""Pins of the oracle's token-row split and micro-batch averaging against
facts that do not come from the oracle's own arithmetic: brute-force
shifting of a small row, the workload generator's two views of one draw, and
the identity that the mean of per-micro-batch gradients of equal-size,
unmasked micro-batches is the gradient of the whole batch's mean loss (the
loss is a mean over positions, and positions of different sequences do not
interact)."""

import numpy as np
import pytest

import oracle
import workload as W


def test_split_packed_by_brute_force():
    packed = np.array([[5, 9, 2, 7], [0, 65535, 1, 3]], dtype=np.uint16)
    tok, tgt = oracle.split_packed(packed)
    for b in range(2):
        for t in range(3):
            assert tok[b, t] == int(packed[b, t])
            assert tgt[b, t] == int(packed[b, t + 1])
    assert tok.dtype == np.int32 and tgt.dtype == np.int32
    assert tgt[1, 0] == 65535  # the full 16-bit range survives the widening


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_packed_rows_and_token_pairs_are_one_draw(name):
    w = W.WORKLOADS[name]
    tok, tgt = W.make_tokens(w, seed=3)
    packed = W.make_packed_tokens(w, seed=3)
    assert packed.dtype == np.uint16 and packed.shape == (w.batch, w.seq_len + 1)
    t2, g2 = oracle.split_packed(packed)
    np.testing.assert_array_equal(t2, tok)
    np.testing.assert_array_equal(g2, tgt)


def test_one_micro_batch_is_the_plain_step():
    w = W.WORKLOADS["tiny"]
    s = oracle.Shape(w.depth, w.d_model, w.n_head, w.vocab)
    p = W.make_params(w).astype(np.float64)
    tok, tgt = W.make_tokens(w)
    loss, g, _ = oracle.step(p, tok, tgt, s)
    la, ga = oracle.step_accumulated(p, [(tok, tgt)], s)
    assert la == loss
    np.testing.assert_array_equal(ga, g)


def test_mean_of_micro_batch_gradients_is_the_whole_batch_gradient():
    w = W.WORKLOADS["tiny"]
    assert w.batch % 2 == 0
    s = oracle.Shape(w.depth, w.d_model, w.n_head, w.vocab)
    p = W.make_params(w).astype(np.float64)
    tok, tgt = W.make_tokens(w, seed=4)
    loss, g, _ = oracle.step(p, tok, tgt, s)
    h = w.batch // 2
    la, ga = oracle.step_accumulated(p, [(tok[:h], tgt[:h]), (tok[h:], tgt[h:])], s)
    assert abs(la - loss) <= 1e-12 * abs(loss)
    np.testing.assert_allclose(ga, g, rtol=1e-9, atol=1e-14 * np.abs(g).max())
    # and unequal halves are not the same thing: a wrong (sum, not mean) average fails
    assert not np.allclose(2 * ga, g)
