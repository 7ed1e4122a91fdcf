"""Helpers shared by the GPU parity tests (device plumbing and metrics only)."""

from __future__ import annotations

import numpy as np

import oracle
import workload as W


def load_nc():
    from decoder_transformer_step_nanochat_b300 import build
    build.build()
    import decoder_transformer_step_nanochat_b300 as nc
    return nc


def shape_of(w: W.Workload) -> oracle.Shape:
    return oracle.Shape(w.depth, w.d_model, w.n_head, w.vocab)


def to_device_params(p: np.ndarray, precision: int):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(p, dtype=np.float32))
    if precision == 0:  # NC_BF16: the values are bf16-representable, so this is exact
        t = t.to(torch.bfloat16)
    return t.cuda()


def to_device_i32(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def run_gpu_step(nc, w: W.Workload, params: np.ndarray, tok: np.ndarray, tgt: np.ndarray, precision: int):
    """Forward + backward through the C ABI; returns loss, grads, lse, nll, argmax (numpy)."""
    import torch
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, tok.shape[0], precision)
    try:
        dp = to_device_params(params, precision)
        dt, dg = to_device_i32(tok), to_device_i32(tgt)
        grads = torch.empty(st.n_params, dtype=torch.float32, device="cuda")
        loss = st.forward_loss(dp, dt, dg)
        lse, nll, am = st.token_outputs()
        hf = st.hidden()
        st.backward(grads)
        nc.nc_sync(st.ctx)
        return (loss, grads.cpu().numpy(), lse.cpu().numpy(), nll.cpu().numpy(), am.cpu().numpy(),
                hf.float().cpu().numpy())
    finally:
        st.close()


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def per_tensor(w: W.Workload, g_gpu, g_ref):
    """[(name, rel_l2, cosine)] for every parameter tensor."""
    out = []
    for name, off, r, c in oracle.layout(shape_of(w)):
        a, b = g_gpu[off:off + r * c], g_ref[off:off + r * c]
        out.append((name, rel_l2(a, b), cosine(a, b)))
    return out


def logit_stats(hf_ref, hf_gpu, w_lm, chunk=2048):
    """Per position: oracle argmax and top-1/top-2 margin, the argmax and
    margin of the logits the GPU's own final hidden state gives (computed
    here in float64), the oracle logit gap of any id, and the largest
    |logit_gpu_hidden - logit_oracle| over all positions and ids."""
    w = np.asarray(w_lm, dtype=np.float64)
    M = hf_ref.shape[0]
    out = dict(am_ref=np.empty(M, np.int64), margin_ref=np.empty(M), am_g=np.empty(M, np.int64),
               margin_g=np.empty(M), max_dlogit=0.0, logits_ref=[])
    for i in range(0, M, chunk):
        lr = np.asarray(hf_ref[i:i + chunk], dtype=np.float64) @ w.T
        lg = np.asarray(hf_gpu[i:i + chunk], dtype=np.float64) @ w.T
        out["max_dlogit"] = max(out["max_dlogit"], float(np.abs(lr - lg).max()))
        for key, lgt in (("ref", lr), ("g", lg)):
            top2 = np.partition(lgt, -2, axis=1)[:, -2:]
            out["am_" + key][i:i + chunk] = np.argmax(lgt, axis=1)
            out["margin_" + key][i:i + chunk] = top2[:, 1] - top2[:, 0]
        out["logits_ref"].append(lr)
    return out


def check_bf16_step(w: W.Workload, loss, g, lse, nll, am, hf, loss_ref, g_ref, cache, report=None):
    """The bf16 tolerances of the step against the oracle: |dloss| <= 2e-2
    nats; every parameter tensor's gradient within rel-L2 3e-2 and cosine
    0.999; lse within 5e-2 and nll within 6e-2 at every position; argmax
    identical (a) to the argmax of the logits of the GPU's own final hidden
    state wherever their top-2 margin exceeds 1e-3 and (b) to the oracle's
    wherever the oracle margin exceeds 4 x the largest logit difference that
    the bf16 hidden state causes. `report`, a list, receives the measured
    figures."""
    pt = per_tensor(w, g, g_ref)
    dl = np.abs(lse - cache["lse"])
    dn = np.abs(nll - cache["nll"])
    M, d = w.tokens, w.d_model
    st = logit_stats(cache["hf"].reshape(M, d), hf, cache["P"]["lm_head"])
    own = st["margin_g"] > 1e-3
    sure = st["margin_ref"] > 4 * st["max_dlogit"]
    if report is not None:
        report.append(dict(loss=loss, loss_ref=loss_ref, max_rel_l2=max(r for _, r, _ in pt),
                           min_cos=min(c for _, _, c in pt), max_dlse=float(dl.max()), max_dnll=float(dn.max()),
                           argmax_checked=float(sure.mean()), max_dlogit=st["max_dlogit"]))
    assert abs(loss - loss_ref) <= 2e-2, (loss, loss_ref)
    bad = [(n, r, c) for n, r, c in pt if not (r <= 3e-2 and c >= 0.999)]
    assert not bad, bad
    assert dl.max() <= 5e-2, dl.max()
    assert dn.max() <= 6e-2, dn.max()
    np.testing.assert_array_equal(am[own], st["am_g"][own])
    assert sure.mean() > 0.3, (sure.mean(), st["max_dlogit"])
    np.testing.assert_array_equal(am[sure], cache["argmax"][sure])
