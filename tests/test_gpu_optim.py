"""Parity of the optimizer step (include/nc_optim.h) and of the batched GEMM
that runs Muon's Newton-Schulz products, through the C ABI, against the
oracle (oracle/optim.py) on the same seeded inputs.

Tolerances: the fp32 debug mode follows the oracle to 1e-4 relative (per
tensor, on the update). In bf16 the AdamW group is fp32 arithmetic on fp32
state (1e-4 as well); Muon runs Newton-Schulz in bf16 with fp32 accumulation,
as the published Muon does, so its update is held to the bf16 gradient bar of
the step (relative L2 <= 3e-2, cosine >= 0.999). The bf16 parameters the step
writes must be the round-to-nearest-even image of the fp32 master weights,
bit for bit.
"""

import numpy as np
import pytest

import oracle
import workload as W
from gpu_util import load_nc, rel_l2, shape_of
from oracle import optim

pytestmark = pytest.mark.gpu


def _cos(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


# ------------------------------------------------------------ batched GEMM

def _bf16_dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).cuda()


# (name, M, N, K, a_kmajor, b_kmajor, epi): the four operand patterns of a
# Newton-Schulz step (gram of a wide / tall stack, the polynomial, the update
# of a wide / tall stack); s = 256 or 1664 (13 row blocks per problem and a
# ragged last column block)
NS_CASES = [
    ("gram_wide", 256, 256, 768, 1, 1, 0),
    ("gram_tall", 256, 256, 768, 0, 0, 0),
    ("poly", 256, 256, 256, 1, 0, 7),
    ("update_wide", 256, 768, 256, 1, 0, 7),
    ("update_tall", 768, 256, 256, 1, 1, 7),
    ("gram_wide_1664", 1664, 1664, 1664, 1, 1, 0),
    ("update_wide_1664", 1664, 1664, 1664, 1, 0, 7),
]


@pytest.mark.parametrize("name,M,N,K,ak,bk,epi", NS_CASES)
def test_batched_gemm_matches_per_problem_products(name, M, N, K, ak, bk, epi):
    import torch
    nc = load_nc()
    batch = 3 if M < 1024 else 2
    rng = np.random.default_rng(11)
    # stored operand shapes: A(m,k) = A[m,k] (k-major) or A[k,m]
    a_shape = (M, K) if ak else (K, M)
    b_shape = (N, K) if bk else (K, N)
    A = W.round_bf16(rng.standard_normal((batch,) + a_shape) * 0.1)
    B = W.round_bf16(rng.standard_normal((batch,) + b_shape) * 0.1)
    C2 = W.round_bf16(rng.standard_normal((batch, M, N)))
    alpha, beta = (2.0315, -4.775) if epi == 7 else (1.0, 0.0)
    st = nc.Step(1, 128, 1, 128, 128, 1, nc.NC_BF16)
    try:
        dA, dB, dC2 = _bf16_dev(A), _bf16_dev(B), _bf16_dev(C2)
        dC = torch.full((batch, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        nc.nc_op_gemm_batched(st.ctx, batch, M, N, K, dA.data_ptr(), a_shape[1], ak, a_shape[0],
                              dB.data_ptr(), b_shape[1], bk, b_shape[0], epi, alpha, beta,
                              dC.data_ptr(), N, dC2.data_ptr() if epi == 7 else None, N, M)
        nc.nc_sync(st.ctx)
        got = dC.float().cpu().numpy()
    finally:
        st.close()
    for i in range(batch):
        Am = A[i].astype(np.float64) if ak else A[i].astype(np.float64).T
        Bm = B[i].astype(np.float64) if bk else B[i].astype(np.float64).T
        want = alpha * (Am @ Bm.T) + (beta * C2[i] if epi == 7 else 0.0)
        assert np.all(np.isfinite(got[i])), (name, i)
        e = rel_l2(got[i], want)
        assert e <= 4e-3, (name, i, e)


# ------------------------------------------------------------ optimizer step

def _run(nc, w, params, grads_list, hypers, precision):
    """Steps t = 1.. with the given grads; returns per step (master, params,
    stats) read back from the device."""
    import torch
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, 1, precision)
    out = []
    try:
        dt = torch.bfloat16 if precision == nc.NC_BF16 else torch.float32
        dp = torch.from_numpy(params).to(dt).cuda()
        nbytes = nc.nc_optim_state_bytes(st.ctx)
        state = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
        stats = torch.zeros(2, dtype=torch.float32, device="cuda")
        nc.nc_optim_init(st.ctx, dp.data_ptr(), state.data_ptr())
        P = st.n_params
        for t, (g, h) in enumerate(zip(grads_list, hypers), start=1):
            dg = torch.from_numpy(g).cuda()
            nc.nc_optim_step(st.ctx, dp.data_ptr(), dg.data_ptr(), state.data_ptr(), t, h.lr_adamw, h.lr_muon,
                             h.weight_decay, h.max_grad_norm, stats.data_ptr())
            nc.nc_sync(st.ctx)
            out.append((state[:P].cpu().numpy().copy(), dp.float().cpu().numpy(), stats.cpu().numpy().copy()))
            assert np.array_equal(dg.cpu().numpy(), g)  # grads are read, never written
    finally:
        st.close()
    return out


def _oracle_run(w, params, grads_list, hypers):
    s = shape_of(w)
    master = params.astype(np.float64)
    state = optim.init_state(master, s)
    out = []
    for g, h in zip(grads_list, hypers):
        master, state, norm, k = optim.optimizer_step(master, g, state, s, h)
        out.append((master.copy(), norm, k))
    return out


def _compare(w, params, got, want, muon_tol, muon_cos):
    s = shape_of(w)
    adamw_g, muon_g = optim.groups(s)
    prev_g = params.astype(np.float64)
    prev_w = params.astype(np.float64)
    worst = {}
    for (mg, pg, stats), (mw, norm, k) in zip(got, want):
        assert abs(stats[0] - norm) <= 1e-5 * norm and abs(stats[1] - k) <= 1e-5 * k
        for group, tol, cmin in ((adamw_g, 1e-4, 0.99999999), (muon_g, muon_tol, muon_cos)):
            for name, off, r, c in group:
                sl = slice(off, off + r * c)
                du_g = mg[sl].astype(np.float64) - prev_g[sl]
                du_w = mw[sl] - prev_w[sl]
                e, cs = rel_l2(du_g, du_w), _cos(du_g, du_w)
                worst[name] = max(worst.get(name, 0.0), e)
                assert e <= tol and cs >= cmin, (name, e, cs)
        prev_g, prev_w = mg.astype(np.float64), mw
    return worst


def test_optimizer_step_fp32_debug_matches_oracle():
    nc = load_nc()
    w = W.WORKLOADS["tiny"]
    params = W.make_params(w)
    grads = [W.make_grads(w, seed=100), W.make_grads(w, seed=101, std=3e-4)]
    hypers = [optim.Hyper(), optim.Hyper(lr_adamw=1e-3, lr_muon=1e-2)]
    got = _run(nc, w, params, grads, hypers, nc.NC_FP32_DEBUG)
    want = _oracle_run(w, params, grads, hypers)
    _compare(w, params, got, want, 1e-4, 0.99999999)
    for mg, pg, _ in got:
        assert np.array_equal(mg, pg)  # fp32 params are the master weights


def test_optimizer_step_bf16_matches_oracle_and_rounds_master():
    nc = load_nc()
    w = W.WORKLOADS["small"]
    params = W.make_params(w)
    grads = [W.make_grads(w, seed=102), W.make_grads(w, seed=103, std=2e-3)]
    hypers = [optim.Hyper(), optim.Hyper(lr_adamw=1e-3, lr_muon=1e-2, max_grad_norm=0.5)]
    got = _run(nc, w, params, grads, hypers, nc.NC_BF16)
    want = _oracle_run(w, params, grads, hypers)
    worst = _compare(w, params, got, want, 3e-2, 0.999)
    print("worst update rel-L2 per tensor:", sorted(worst.items(), key=lambda kv: -kv[1])[:4])
    for mg, pg, _ in got:
        assert np.array_equal(W.bf16_bits(pg), W.bf16_bits(W.round_bf16(mg)))


def test_optimizer_step_is_deterministic():
    nc = load_nc()
    w = W.WORKLOADS["small"]
    params = W.make_params(w)
    grads = [W.make_grads(w, seed=104)]
    hypers = [optim.Hyper()]
    a = _run(nc, w, params, grads, hypers, nc.NC_BF16)
    b = _run(nc, w, params, grads, hypers, nc.NC_BF16)
    assert np.array_equal(a[0][0], b[0][0]) and np.array_equal(a[0][2], b[0][2])


def test_optimizer_rejects_bad_arguments():
    import torch
    nc = load_nc()
    w = W.WORKLOADS["tiny"]
    st = nc.Step(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab, 1, nc.NC_FP32_DEBUG)
    try:
        buf = torch.zeros(16, dtype=torch.float32, device="cuda")
        p = buf.data_ptr()
        for bad in (dict(t=0), dict(lr_adamw=-1.0), dict(max_grad_norm=0.0)):
            kw = dict(t=1, lr_adamw=1e-3, lr_muon=1e-2, weight_decay=0.1, max_grad_norm=1.0)
            kw.update(bad)
            with pytest.raises(nc.NcError) as ei:
                nc.nc_optim_step(st.ctx, p, p, p, kw["t"], kw["lr_adamw"], kw["lr_muon"], kw["weight_decay"],
                                 kw["max_grad_norm"])
            assert ei.value.status == 1
        with pytest.raises(nc.NcError):
            nc.nc_optim_step(st.ctx, p + 4, p, p, 1, 1e-3, 1e-2, 0.1, 1.0)  # misaligned params
    finally:
        st.close()


@pytest.mark.slow
def test_optimizer_step_full_size_d20_sampled():
    """d20 (561M parameters, bf16): one step on the whole model; the oracle
    checks the clip statistics over every gradient, AdamW on sampled rows of
    wte and lm_head, and Muon on three whole matrices of different kinds."""
    import torch
    nc = load_nc()
    w = W.WORKLOADS["d20"]
    s = shape_of(w)
    params = W.make_params(w)
    g = W.make_grads(w, seed=105)
    h = optim.Hyper()
    got = _run(nc, w, params, [g], [h], nc.NC_BF16)[0]
    mg, pg, stats = got
    norm, k = optim.clip_scale(g, h.max_grad_norm)
    assert abs(stats[0] - norm) <= 1e-5 * norm and abs(stats[1] - k) <= 1e-5 * k
    rng = np.random.default_rng(5)
    adamw_g, muon_g = optim.groups(s)
    for name, off, r, c in adamw_g:
        rows = rng.choice(r, 64, replace=False)
        idx = (off + rows[:, None] * c + np.arange(c)[None, :]).ravel()
        p0 = params[idx].astype(np.float64)
        gk = g[idx].astype(np.float64) * k
        pw, _, _ = optim.adamw(p0, gk, 0 * p0, 0 * p0, 1, h.lr_adamw, h.beta1, h.beta2, h.eps, h.weight_decay)
        assert rel_l2(mg[idx] - p0, pw - p0) <= 1e-4
    for name in ("h0.w_qkv", "h7.w_o", "h19.w_fc", "h12.w_proj"):
        (_, off, r, c), = [x for x in muon_g if x[0] == name]
        sl = slice(off, off + r * c)
        p0 = params[sl].astype(np.float64).reshape(r, c)
        gk = g[sl].astype(np.float64).reshape(r, c) * k
        pw, _ = optim.muon(p0, gk, np.zeros_like(p0), h.lr_muon, h.momentum, h.weight_decay, h.ns_steps)
        du_g = mg[sl].reshape(r, c) - p0
        e, cs = rel_l2(du_g, pw - p0), _cos(du_g, pw - p0)
        assert e <= 3e-2 and cs >= 0.999, (name, e, cs)
    sample = rng.choice(mg.size, 1 << 20, replace=False)
    assert np.array_equal(W.bf16_bits(pg[sample]), W.bf16_bits(W.round_bf16(mg[sample])))
    del torch
