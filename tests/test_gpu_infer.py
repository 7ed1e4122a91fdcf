"""Generation with a KV cache (include/nc_infer.h) against the oracle
(oracle/infer.py): prefill of the workload's prompts, then decode steps fed
with the same seeded continuation tokens on both sides. fp32 debug mode
within 1e-4 relative on the logits, with the greedy token of every step equal
to the argmax of the oracle's logits; bf16 within the step's bar (logits
relative L2 <= 3e-2, lse within 5e-2 nats) with the greedy token equal
wherever the oracle's top-1/top-2 margin exceeds four times the largest
logit difference seen. The graph-replay test compares the device-position
steps with the host-position steps (no oracle)."""

import numpy as np
import pytest

import oracle
import workload as W
from gpu_util import load_nc, rel_l2, shape_of
from oracle import infer

pytestmark = pytest.mark.gpu


def _lse(x):
    m = x.max(-1, keepdims=True)
    return (m + np.log(np.exp(x - m).sum(-1, keepdims=True)))[:, 0]


def _generate_gpu(nc, w, params, prompt, steps, max_len, precision, feed=None):
    """Prefill + `steps` decode steps; step i is fed feed[:, i] when given,
    else the previous greedy token. Returns greedy tokens [B, steps+1] and
    the logits of every produced position."""
    import torch
    B, T = prompt.shape
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, B, precision)
    try:
        dt = torch.bfloat16 if precision == nc.NC_BF16 else torch.float32
        dp = torch.from_numpy(params).to(dt).cuda()
        kv = torch.empty(nc.nc_kv_cache_bytes(st.ctx, max_len) + 256, dtype=torch.uint8, device="cuda")
        kvp = (kv.data_ptr() + 255) // 256 * 256
        tok = torch.from_numpy(np.ascontiguousarray(prompt, dtype=np.int32)).cuda()
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        logits = torch.empty((B, w.vocab), dtype=torch.float32, device="cuda")
        nc.nc_prefill(st.ctx, dp.data_ptr(), tok.data_ptr(), kvp, max_len, nxt.data_ptr(), logits.data_ptr())
        ids, lg = [nxt.cpu().numpy().copy()], [logits.cpu().numpy().copy()]
        for i in range(steps):
            cur = nxt.clone() if feed is None else torch.from_numpy(np.ascontiguousarray(feed[:, i])).cuda()
            nc.nc_decode_step(st.ctx, dp.data_ptr(), cur.data_ptr(), T + i, kvp, max_len, nxt.data_ptr(),
                              logits.data_ptr())
            ids.append(nxt.cpu().numpy().copy())
            lg.append(logits.cpu().numpy().copy())
        nc.nc_sync(st.ctx)
        return np.stack(ids, 1), lg
    finally:
        st.close()


def _oracle_follow(w, params, prompt, feed, dtype):
    """Oracle logits of the prompt's last position and of each fed token."""
    s = shape_of(w)
    cache, logits = infer.prefill(params.astype(dtype), prompt, s, dtype)
    out = [logits]
    for i in range(feed.shape[1]):
        cache, logits = infer.decode_step(params.astype(dtype), cache, feed[:, i], s, dtype)
        out.append(logits)
    return out


def test_tiny_fp32_generation_matches_oracle():
    nc = load_nc()
    w = W.WORKLOADS["tiny"]
    p = W.make_params(w)
    tok, _ = W.make_tokens(w)
    feed = W.make_decode_tokens(w, 4)
    ids, lg = _generate_gpu(nc, w, p, tok, 4, w.seq_len + 8, nc.NC_FP32_DEBUG, feed)
    ref = _oracle_follow(w, p, tok, feed, np.float64)
    for i, (g, r) in enumerate(zip(lg, ref)):
        assert rel_l2(g, r) <= 1e-4, (i, rel_l2(g, r))
        np.testing.assert_array_equal(ids[:, i], np.argmax(r, -1))


@pytest.mark.parametrize("batch", [8, 1, 20], ids=["batch8", "batch1", "batch20"])
def test_small_bf16_generation_matches_oracle(batch):
    """Batches of up to 16 sequences take the weight-streaming decode products
    (one to sixteen rows), larger ones the tensor-core GEMM."""
    nc = load_nc()
    w = W.WORKLOADS["small"].with_batch(batch)
    p = W.make_params(w)
    tok, _ = W.make_tokens(w)
    feed = W.make_decode_tokens(w, 4)
    ids, lg = _generate_gpu(nc, w, p, tok, 4, w.seq_len + 64, nc.NC_BF16, feed)
    ref = _oracle_follow(w, p, tok, feed, np.float32)
    for i, (g, r) in enumerate(zip(lg, ref)):
        r = r.astype(np.float64)
        assert rel_l2(g, r) <= 3e-2, (i, rel_l2(g, r))
        assert np.abs(_lse(g.astype(np.float64)) - _lse(r)).max() <= 5e-2
        top2 = np.sort(r, -1)[:, -2:]
        sure = (top2[:, 1] - top2[:, 0]) > 4 * np.abs(g - r).max()
        np.testing.assert_array_equal(ids[sure, i], np.argmax(r, -1)[sure])


def test_generation_rejects_bad_arguments():
    import torch
    nc = load_nc()
    w = W.WORKLOADS["tiny"]
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, w.batch, nc.NC_FP32_DEBUG)
    try:
        buf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
        base = (buf.data_ptr() + 255) // 256 * 256
        ml = w.seq_len + 4
        for pos, kv, max_len in ((ml, base, ml), (0, base + 16, ml), (0, base, w.seq_len - 1)):
            with pytest.raises(nc.NcError) as ei:
                nc.nc_decode_step(st.ctx, base, base, pos, kv, max_len, base)
            assert ei.value.status == 1
        assert nc.nc_kv_cache_bytes(st.ctx, 0) == 0
    finally:
        st.close()


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_graph_replayed_decode_matches_host_position_steps(name):
    """nc_decode_step_dev reads and advances a device position, so one
    captured step replays for every position; its greedy tokens equal those
    of the host-position steps."""
    import torch
    nc = load_nc()
    w = W.WORKLOADS[name]
    prec = nc.NC_FP32_DEBUG if w.dtype == "fp32" else nc.NC_BF16
    p = W.make_params(w)
    prompt, _ = W.make_tokens(w)
    B, T = prompt.shape
    steps, max_len = 4, w.seq_len + 16
    ids_host, _ = _generate_gpu(nc, w, p, prompt, steps, max_len, prec)
    stream = torch.cuda.Stream()
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, B, prec, stream=stream)
    try:
        dt = torch.bfloat16 if prec == nc.NC_BF16 else torch.float32
        dp = torch.from_numpy(p).to(dt).cuda()
        kv = torch.empty(nc.nc_kv_cache_bytes(st.ctx, max_len) + 256, dtype=torch.uint8, device="cuda")
        kvp = (kv.data_ptr() + 255) // 256 * 256
        tok = torch.from_numpy(np.ascontiguousarray(prompt, dtype=np.int32)).cuda()
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        cur = torch.empty(B, dtype=torch.int32, device="cuda")
        pos = torch.full((1,), T, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            nc.nc_prefill(st.ctx, dp.data_ptr(), tok.data_ptr(), kvp, max_len, nxt.data_ptr())
            got = [nxt.clone()]
            cur.copy_(nxt)
            nc.nc_decode_step_dev(st.ctx, dp.data_ptr(), cur.data_ptr(), pos.data_ptr(), kvp, max_len, nxt.data_ptr())
            got.append(nxt.clone())
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            cur.copy_(nxt)
            nc.nc_decode_step_dev(st.ctx, dp.data_ptr(), cur.data_ptr(), pos.data_ptr(), kvp, max_len, nxt.data_ptr())
        for _ in range(steps - 1):
            g.replay()
            got.append(nxt.clone())
        torch.cuda.synchronize()
        nc.nc_sync(st.ctx)
        assert int(pos.item()) == T + steps
        ids_dev = torch.stack(got, 1).cpu().numpy()
    finally:
        st.close()
    np.testing.assert_array_equal(ids_dev, ids_host)
