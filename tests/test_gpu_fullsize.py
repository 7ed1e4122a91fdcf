"""Parity at the full benchmark sizes, in the launch configuration the
benchmark times (bf16, batch 16 x seq 2048 for depth 20 and 26; batch 8 for
the GPT-2-small shape).

The oracle cannot run the whole batch, so the checks are ones it can make
one by one or that hold at any size:
* per-position lse / loss of sampled sequences: sequences are independent,
  and by causality the first 256 positions of a sequence depend on nothing
  after them, so the oracle runs just those positions of that sequence;
* the mean loss is the mean of the per-position losses the kernels report;
* the gradient of the full batch equals the mean of the gradients of its two
  halves (linearity of the mean loss), up to bf16 rounding;
* rows of wte that no token uses get exactly zero gradient, and every
  gradient is finite.
"""

import numpy as np
import pytest

import oracle
import workload as W
from gpu_util import load_nc, rel_l2, shape_of, to_device_i32, to_device_params

pytestmark = pytest.mark.gpu

PREFIX = 256


def _step(nc, st, dp, tok, tgt, grads):
    loss = st.forward_loss(dp, to_device_i32(tok), to_device_i32(tgt))
    lse, nll, am = st.token_outputs()
    st.backward(grads)
    nc.nc_sync(st.ctx)
    return loss, lse.cpu().numpy(), nll.cpu().numpy(), am.cpu().numpy()


@pytest.mark.parametrize("name,sampled", [("gpt2_small", (3,)), ("d20", (0, 11)), ("d26", (5,))])
def test_full_size_step(name, sampled):
    import torch
    nc = load_nc()
    w = W.WORKLOADS[name]
    p = W.make_params(w)
    tok, tgt = W.make_tokens(w)
    B, T = tok.shape
    dp = to_device_params(p, nc.NC_BF16)
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, B, nc.NC_BF16)
    try:
        g_full = torch.empty(st.n_params, dtype=torch.float32, device="cuda")
        loss, lse, nll, am = _step(nc, st, dp, tok, tgt, g_full)
    finally:
        st.close()
    assert np.isfinite(loss) and np.all(np.isfinite(lse))
    assert abs(loss - float(np.mean(nll.astype(np.float64)))) < 1e-4
    # sampled sequences against the oracle (first PREFIX positions)
    s = shape_of(w)
    for b in sampled:
        _, cache = oracle.forward(p, tok[b:b + 1, :PREFIX], tgt[b:b + 1, :PREFIX], s, np.float32, keep=False)
        g_lse = lse.reshape(B, T)[b, :PREFIX]
        g_nll = nll.reshape(B, T)[b, :PREFIX]
        assert np.abs(g_lse - cache["lse"]).max() <= 5e-2
        assert np.abs(g_nll - cache["nll"]).max() <= 1e-1
        assert abs(float(np.mean(g_nll)) - float(np.mean(cache["nll"]))) <= 2e-2
    # linearity: full-batch gradient = mean of the two half-batch gradients
    h = B // 2
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, h, nc.NC_BF16)
    try:
        g_a = torch.empty(st.n_params, dtype=torch.float32, device="cuda")
        g_b = torch.empty(st.n_params, dtype=torch.float32, device="cuda")
        _step(nc, st, dp, tok[:h], tgt[:h], g_a)
        _step(nc, st, dp, tok[h:], tgt[h:], g_b)
    finally:
        st.close()
    g_mean = ((g_a + g_b) * 0.5).cpu().numpy()
    g = g_full.cpu().numpy()
    assert np.all(np.isfinite(g))
    bad = []
    for tname, off, r, c in oracle.layout(s):
        e = rel_l2(g[off:off + r * c], g_mean[off:off + r * c])
        if not e <= 2e-2:
            bad.append((tname, e))
    assert not bad, bad
    V, d = w.vocab, w.d_model
    absent = np.setdiff1d(np.arange(V), np.unique(tok))
    assert np.all(g[:V * d].reshape(V, d)[absent] == 0.0)
