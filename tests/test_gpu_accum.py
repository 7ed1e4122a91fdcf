"""Gradient accumulation over micro-batches and the packed uint16 token input,
through the C ABI, against the oracle's whole-batch step (nanochat explainer,
"Distributed Training": gradients averaged over shards after the backward;
"Streaming Tokenization": packed 16-bit token ids; "Pretraining": targets are
the next tokens). Tolerances as for the plain step: fp32 debug within 1e-4,
bf16 within 2e-2 on the loss and 3e-2 relative L2 / cosine 0.999 per tensor.
"""

import numpy as np
import pytest

import oracle
import workload as W
from gpu_util import load_nc, per_tensor, run_gpu_step, shape_of, to_device_i32, to_device_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nc():
    return load_nc()


def _accumulate(nc, w, p, tok, tgt, prec, parts, g0=None):
    """Configure the micro-batch size, run forward + accumulating backward on
    each part with scale 1/parts into grads (zero, or g0), return (mean
    loss, grads)."""
    import torch
    mb = tok.shape[0] // parts
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, mb, prec)
    try:
        dp = to_device_params(p, prec)
        grads = (torch.zeros(st.n_params, dtype=torch.float32, device="cuda") if g0 is None
                 else torch.from_numpy(g0.astype(np.float32)).cuda())
        losses = []
        for i in range(parts):
            dt, dg = to_device_i32(tok[i * mb:(i + 1) * mb]), to_device_i32(tgt[i * mb:(i + 1) * mb])
            losses.append(st.forward_loss(dp, dt, dg))
            st.backward_accumulate(grads, 1.0 / parts)
        nc.nc_sync(st.ctx)
        return float(np.mean(losses)), grads.cpu().numpy().astype(np.float64)
    finally:
        st.close()


@pytest.mark.parametrize("name,prec", [("tiny", 1), ("small", 0)])
def test_two_micro_batches_match_the_whole_batch_oracle(nc, name, prec):
    w = W.WORKLOADS[name]
    if w.batch < 2:
        w = w.with_batch(2)
    p = W.make_params(w)
    tok, tgt = W.make_tokens(w, seed=7)
    loss_ref, g_ref, _ = oracle.step(p.astype(np.float64), tok, tgt, shape_of(w), np.float64)
    loss, g = _accumulate(nc, w, p, tok, tgt, prec, 2)
    if prec == 1:
        assert abs(loss - loss_ref) <= 1e-4 * abs(loss_ref)
        bad = [(n, r) for n, r, _ in per_tensor(w, g, g_ref) if not r <= 1e-4]
    else:
        assert abs(loss - loss_ref) <= 2e-2
        bad = [(n, r, c) for n, r, c in per_tensor(w, g, g_ref) if not (r <= 3e-2 and c >= 0.999)]
    assert not bad, bad


@pytest.mark.parametrize("name,prec", [("tiny", 1), ("small", 0)])
def test_accumulation_adds_onto_existing_gradients(nc, name, prec):
    """grads = g0 + s * grad: every gradient write (weight-gradient GEMMs with
    and without k-splits, lm_head, the embedding scatter) must add."""
    w = W.WORKLOADS[name]
    p = W.make_params(w)
    tok, tgt = W.make_tokens(w, seed=8)
    _, g_plain, *_ = run_gpu_step(nc, w, p, tok, tgt, prec)
    g0 = np.random.Generator(np.random.PCG64(9)).standard_normal(g_plain.size) * np.abs(g_plain).max()
    _, g = _accumulate(nc, w, p, tok, tgt, prec, 1, g0=g0)
    want = g0.astype(np.float32).astype(np.float64) + g_plain
    # atomics and reduce-adds make the two backward passes differ in the last bits
    for name_t, off, r, c in oracle.layout(shape_of(w)):
        a, b = g[off:off + r * c], want[off:off + r * c]
        err = np.linalg.norm(a - b) / max(np.linalg.norm(g_plain[off:off + r * c]), 1e-30)
        assert err <= 1e-3, (name_t, err)


def test_non_finite_scale_is_rejected(nc):
    import torch
    w = W.WORKLOADS["tiny"]
    p = W.make_params(w)
    tok, tgt = W.make_tokens(w)
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, w.batch, nc.NC_FP32_DEBUG)
    try:
        dp = to_device_params(p, 1)
        st.forward_loss(dp, to_device_i32(tok), to_device_i32(tgt))
        grads = torch.zeros(st.n_params, dtype=torch.float32, device="cuda")
        with pytest.raises(nc.NcError) as ei:
            st.backward_accumulate(grads, float("nan"))
        assert ei.value.status == 1  # NC_ERR_ARG
    finally:
        st.close()


@pytest.mark.parametrize("name,prec", [("tiny", 1), ("small", 0)])
def test_packed_u16_rows_give_the_int32_step(nc, name, prec):
    import torch
    w = W.WORKLOADS[name]
    p = W.make_params(w)
    packed = W.make_packed_tokens(w, seed=11)
    tok, tgt = oracle.split_packed(packed)
    loss_i, g_i, *_ = run_gpu_step(nc, w, p, tok, tgt, prec)
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, w.batch, prec)
    try:
        dp = to_device_params(p, prec)
        d_loss = torch.empty(1, dtype=torch.float32, device="cuda")
        dpk = torch.from_numpy(packed.view(np.int16)).cuda()  # 16-bit rows as they come
        st.forward_loss_u16(dp, dpk, d_loss)
        grads = torch.empty(st.n_params, dtype=torch.float32, device="cuda")
        st.backward(grads)
        nc.nc_sync(st.ctx)
        loss_u = float(d_loss.item())
        g_u = grads.cpu().numpy().astype(np.float64)
        # host rows through the end-to-end entry point
        h = torch.from_numpy(packed.view(np.int16)).pin_memory()
        g_h = torch.empty(st.n_params, dtype=torch.float32, device="cuda")
        loss_h = nc.nc_train_step_host_u16(st.ctx, dp.data_ptr(), h.data_ptr(), g_h.data_ptr())
    finally:
        st.close()
    assert loss_u == loss_i and loss_h == loss_i  # same ids, same deterministic forward
    for name_t, off, r, c in oracle.layout(shape_of(w)):
        ref = g_i[off:off + r * c]
        for got in (g_u, g_h.cpu().numpy().astype(np.float64)):
            err = np.linalg.norm(got[off:off + r * c] - ref) / max(np.linalg.norm(ref), 1e-30)
            assert err <= 1e-4, (name_t, err)
    loss_ref, g_ref, _ = oracle.step(p.astype(np.float64), tok, tgt, shape_of(w), np.float64)
    assert abs(loss_u - loss_ref) <= (1e-4 * abs(loss_ref) if prec == 1 else 2e-2)


def test_u16_ids_beyond_the_vocabulary_are_rejected(nc):
    import torch
    w = W.WORKLOADS["tiny"].with_vocab(4096)  # 16-bit ids can pass its end
    p = W.make_params(w)
    packed = W.make_packed_tokens(w, seed=12)
    packed[0, 3] = w.vocab  # one id past the end
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, w.batch, nc.NC_FP32_DEBUG)
    try:
        dp = to_device_params(p, 1)
        d_loss = torch.empty(1, dtype=torch.float32, device="cuda")
        st.forward_loss_u16(dp, torch.from_numpy(packed.view(np.int16)).cuda(), d_loss)
        with pytest.raises(nc.NcError) as ei:
            nc.nc_sync(st.ctx)
        assert ei.value.status == 5  # NC_ERR_DEVICE
    finally:
        st.close()
