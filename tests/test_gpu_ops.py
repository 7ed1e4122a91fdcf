"""Op-level parity: each step of the path through the C ABI against the
oracle's piece (or the textbook routine the oracle uses for it), on seeded
inputs that span several tiles and a ragged tail."""

import numpy as np
import pytest

import oracle
import workload as W
from gpu_util import load_nc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nc():
    return load_nc()


def torch_of(a, prec, nc):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return (t.to(torch.bfloat16) if prec == nc.NC_BF16 else t).cuda()


def host(t):
    import torch
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def rounded(a, prec):
    return W.round_bf16(a) if prec == 0 else np.asarray(a, dtype=np.float32)


class Ctx:
    def __init__(self, nc, depth, d, H, T, V, B, prec):
        self.step = nc.Step(depth, d, H, T, V, B, prec)
        self.ctx = self.step.ctx

    def close(self):
        self.step.close()


def close_enough(got, ref, prec, rel_bf16=8e-3, rel_f32=2e-5):
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.sqrt(np.mean(ref * ref)) + 1e-30
    rel = rel_bf16 if prec == 0 else rel_f32
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    return np.all(err <= rel * np.abs(ref) + rel * scale), float((err / scale).max())


# ---------------------------------------------------------------- GEMM

M_, N_, K_ = 304, 520, 200  # 2 full 128-row tiles + 48, 2 full 256-col tiles + 8, 3 k-slices + 8


@pytest.mark.parametrize("prec", [0, 1], ids=["bf16", "fp32"])
@pytest.mark.parametrize("ak,bk", [(1, 1), (1, 0), (0, 0), (0, 1)], ids=["TN", "NN_b", "MN_ab", "MN_a"])
@pytest.mark.parametrize("epi", [0, 1, 2, 3, 4, 8], ids=["store", "store_f32", "relu2", "relu2_bwd", "ce_bwd", "relu2a"])
def test_gemm_epilogues(nc, prec, ak, bk, epi):
    import torch
    rng = np.random.default_rng(100 + 10 * ak + bk + 3 * epi)
    A = rounded(rng.standard_normal((M_, K_)) * 0.5, prec)
    Bm = rounded(rng.standard_normal((N_, K_)) * 0.5, prec)
    acc = A.astype(np.float64) @ Bm.astype(np.float64).T
    alpha = 0.75
    a_st = A if ak else np.ascontiguousarray(A.T)
    b_st = Bm if bk else np.ascontiguousarray(Bm.T)
    lda = K_ if ak else M_
    ldb = K_ if bk else N_
    c = Ctx(nc, 1, 128, 1, 128, 1024, 1, prec)
    try:
        dA, dB = torch_of(a_st, prec, nc), torch_of(b_st, prec, nc)
        elem = torch.bfloat16 if prec == 0 else torch.float32
        C2 = None
        row_f = row_i = None
        beta = 0.0
        if epi == 1:
            C0 = rng.standard_normal((M_, N_)).astype(np.float32)
            C = torch.from_numpy(C0).cuda()
            beta = 0.5
            ref = alpha * acc + beta * C0
        else:
            C = torch.zeros((M_, N_), dtype=elem, device="cuda")
        if epi == 0:
            ref = alpha * acc
        elif epi == 2:
            C2 = torch.zeros((M_, N_), dtype=elem, device="cuda")
            u = alpha * acc
            ref = u
            ref2 = np.square(np.maximum(u, 0))  # the kernel squares the fp32 u, then rounds
        elif epi == 3:
            # C2 holds a = relu(u)^2 (what the forward keeps); relu(u) = sqrt(a)
            a_in = rounded(np.square(np.maximum(rng.standard_normal((M_, N_)), 0)), prec)
            C2 = torch_of(a_in, prec, nc)
            ref = alpha * acc * 2 * np.sqrt(a_in)
        elif epi == 8:
            ref = np.square(np.maximum(alpha * acc, 0))  # a only
        elif epi == 4:
            lse = np.log(np.sum(np.exp(alpha * acc), axis=1)).astype(np.float32)
            tgt = rng.integers(0, N_, M_).astype(np.int32)
            row_f = torch.from_numpy(lse).cuda()
            row_i = torch.from_numpy(tgt).cuda()
            ref = np.exp(alpha * acc - lse[:, None].astype(np.float64))
            ref[np.arange(M_), tgt] -= 1.0
        nc.nc_op_gemm(c.ctx, M_, N_, K_, dA.data_ptr(), lda, ak, dB.data_ptr(), ldb, bk, epi, alpha, beta,
                      C.data_ptr(), N_, C2.data_ptr() if C2 is not None else None, N_ if C2 is not None else 0,
                      row_f.data_ptr() if row_f is not None else None,
                      row_i.data_ptr() if row_i is not None else None)
        nc.nc_sync(c.ctx)
        ok, err = close_enough(host(C), ref, prec if epi != 1 else 1, rel_f32=5e-5 if prec == 0 else 2e-5)
        assert ok, err
        if epi == 2:
            ok, err = close_enough(host(C2), ref2, prec)
            assert ok, err
            assert np.all(host(C2)[host(C) <= 0] == 0.0)  # exact zeros of ReLU^2
        if epi == 8:
            assert np.all(host(C)[alpha * acc <= 0] == 0.0)
    finally:
        c.close()


@pytest.mark.parametrize("prec", [0, 1], ids=["bf16", "fp32"])
def test_gemm_degenerate_sizes(nc, prec):
    import torch
    c = Ctx(nc, 1, 128, 1, 128, 1024, 1, prec)
    try:
        elem = torch.bfloat16 if prec == 0 else torch.float32
        A = torch.ones((64, 64), dtype=elem, device="cuda")
        C = torch.full((64, 64), 7.0, dtype=torch.float32, device="cuda")
        # K = 0: the product is empty, C = alpha*0 + beta*C
        nc.nc_op_gemm(c.ctx, 64, 64, 0, A.data_ptr(), 64, 1, A.data_ptr(), 64, 1, 1, 1.0, 0.5, C.data_ptr(), 64)
        # M = 0 and N = 0: nothing is written
        nc.nc_op_gemm(c.ctx, 0, 64, 64, A.data_ptr(), 64, 1, A.data_ptr(), 64, 1, 1, 1.0, 0.0, C.data_ptr(), 64)
        nc.nc_op_gemm(c.ctx, 64, 0, 64, A.data_ptr(), 64, 1, A.data_ptr(), 64, 1, 1, 1.0, 0.0, C.data_ptr(), 64)
        nc.nc_sync(c.ctx)
        assert np.all(C.cpu().numpy() == 3.5)
    finally:
        c.close()


@pytest.mark.parametrize("beta", [0.5, 0.0, 1.0], ids=["beta_half", "beta0", "beta1"])
@pytest.mark.parametrize("ak,bk", [(0, 0), (1, 0)], ids=["MN_ab", "NN_b"])
def test_gemm_split_k_weight_gradient_shape(nc, ak, bk, beta):
    # few output tiles and a long K (the weight-gradient shape): the library
    # splits K into partial sums and adds them in a fixed order (with beta 0
    # or 1 inside the kernel, split after split; otherwise by a reduction
    # kernel over partial slabs)
    import torch
    M, N, K = 256, 264, 4160
    rng = np.random.default_rng(31 + ak)
    A = rounded(rng.standard_normal((M, K)) * 0.5, 0)
    Bm = rounded(rng.standard_normal((N, K)) * 0.5, 0)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    ref = 0.25 * (A.astype(np.float64) @ Bm.astype(np.float64).T) + beta * C0
    c = Ctx(nc, 1, 128, 1, 128, 1024, 1, 0)
    try:
        dA = torch_of(A if ak else np.ascontiguousarray(A.T), 0, nc)
        dB = torch_of(Bm if bk else np.ascontiguousarray(Bm.T), 0, nc)
        outs = []
        for _ in range(2):
            C = torch.from_numpy(C0.copy()).cuda()
            nc.nc_op_gemm(c.ctx, M, N, K, dA.data_ptr(), K if ak else M, ak, dB.data_ptr(), K if bk else N, bk,
                          1, 0.25, beta, C.data_ptr(), N)
            nc.nc_sync(c.ctx)
            outs.append(C.cpu().numpy())
        ok, err = close_enough(outs[0], ref, 1, rel_f32=5e-5)
        assert ok, err
        np.testing.assert_array_equal(outs[0], outs[1])  # fixed reduction order: bitwise repeatable
    finally:
        c.close()


def test_qkv_gemm_with_fused_qk_norm_rope(nc):
    # the QKV projection with QK-norm + RoPE in its epilogue, against the
    # oracle's rmsnorm and rotation applied to the float64 product
    import torch
    B, T, H = 2, 256, 3
    d, D = H * 128, 128
    M = B * T
    rng = np.random.default_rng(17)
    x = rounded(rng.standard_normal((M, d)), 0)
    w = rounded(rng.standard_normal((3 * d, d)) * 0.05, 0)
    c = Ctx(nc, 1, d, H, T, 1024, B, 0)
    try:
        qkv = torch.zeros((M, 3 * d), dtype=torch.bfloat16, device="cuda")
        rqk = torch.zeros((M, 2 * H), dtype=torch.float32, device="cuda")
        dx, dw = torch_of(x, 0, nc), torch_of(w, 0, nc)
        nc.nc_op_gemm(c.ctx, M, 3 * d, d, dx.data_ptr(), d, 1, dw.data_ptr(), d, 1, nc.NC_EPI_QKNORM_ROPE,
                      1.0, 0.0, qkv.data_ptr(), 3 * d, rqk.data_ptr(), 0)
        nc.nc_sync(c.ctx)
        acc = (x.astype(np.float64) @ w.astype(np.float64).T).reshape(B, T, 3, H, D)
        got = host(qkv).reshape(B, T, 3, H, D)
        cos, sin = oracle.rope_angles(T)
        for b in range(B):
            for which in (0, 1):
                n, rr = oracle.rmsnorm(acc[b, :, which])
                ok, err = close_enough(got[b, :, which], oracle.rope(n, cos, sin), 0)
                assert ok, err
                np.testing.assert_allclose(rqk.cpu().numpy().reshape(B, T, 2, H)[b, :, which], rr[..., 0], rtol=1e-4)
            ok, err = close_enough(got[b, :, 2], acc[b, :, 2], 0)
            assert ok, err
    finally:
        c.close()


# ---------------------------------------------------------------- attention

def _qkv(rng, B, T, H, prec):
    D = 128
    q = rng.standard_normal((B, T, H, D))
    k = rng.standard_normal((B, T, H, D))
    q = q / np.sqrt(np.mean(q * q, -1, keepdims=True))
    k = k / np.sqrt(np.mean(k * k, -1, keepdims=True))
    v = rng.standard_normal((B, T, H, D))
    qkv = np.concatenate([q.reshape(B, T, -1), k.reshape(B, T, -1), v.reshape(B, T, -1)], -1)
    return rounded(qkv, prec).reshape(B * T, 3 * H * D)


# Element-wise bounds of the attention kernels against the float64 oracle on
# the same bf16-exact inputs. In bf16 the bound follows the kernels' rounding
# points, each at most the unit roundoff u = 2^-8 (8 significant bits) of
# what it rounds:
#   forward: o = sum_j bf16(p_j) v_j / l with l summed from the unrounded p,
#     then o is rounded: |o_gpu - o| <= u * sum_j p_j |v_j| + u * |o|;
#   backward: dS = bf16(p (dP - D_gpu)) where D_gpu = rowsum(dO o_gpu) uses the
#     kernel's own o, so |dS_gpu - dS| <= u |dS| + p |dD| (dD = D_gpu - D, known
#     exactly here); dQ, dK sum those errors against |K|, |Q| (times 1/sqrt(128));
#     dV = sum_t bf16(p_t) dO_t, rounded: u * sum_t p_t |dO_t| + u |dV|.
# Each bound also carries fp32 accumulation (n * 2^-24 times the sum of the
# absolute terms) and is checked with a factor 2 of slack; a wrong tile (the
# diagonal, the last key tile of a ragged T) is off by O(1) of the terms and
# fails by far. The fp32 debug kernels round nowhere but in fp32 sums.
U_BF16 = 2.0 ** -8


def attention_bounds(q, k, v, do, o_ref, o_gpu, prec):
    """Per-element error bounds (o, dq, dk, dv) for one sequence, all heads.
    q, k, v, do: [T, H, D] float64; o_ref the oracle's output; o_gpu the
    kernel's (which the backward's row sums D use)."""
    T, H, D = q.shape
    u = U_BF16 if prec == 0 else 0.0
    gam = T * 2.0 ** -24
    sc = 1.0 / np.sqrt(D)
    mask = np.tril(np.ones((T, T), dtype=bool))
    bo, bdq, bdk, bdv = (np.empty((T, H, D)) for _ in range(4))
    for h in range(H):
        s = (q[:, h] @ k[:, h].T) * sc
        s = np.where(mask, s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        pv = p @ np.abs(v[:, h])
        bo[:, h] = (u + gam) * pv + u * np.abs(o_ref[:, h])
        dp = do[:, h] @ v[:, h].T
        dd_exact = np.sum(do[:, h] * o_ref[:, h], 1)
        dd_gpu = np.sum(do[:, h] * o_gpu[:, h], 1)
        ds = p * (dp - dd_exact[:, None])
        e_ds = u * np.abs(ds) + p * (np.abs(dd_gpu - dd_exact) + gam * np.sum(np.abs(do[:, h] * o_gpu[:, h]), 1))[:, None]
        a_ds = np.abs(ds) + e_ds
        bdq[:, h] = sc * (e_ds @ np.abs(k[:, h]) + gam * (a_ds @ np.abs(k[:, h])))
        bdk[:, h] = sc * (e_ds.T @ np.abs(q[:, h]) + gam * (a_ds.T @ np.abs(q[:, h])))
        dv = p.T @ do[:, h]
        bdv[:, h] = (u + gam) * (p.T @ np.abs(do[:, h])) + u * np.abs(dv)
    return bo, bdq, bdk, bdv


def within(got, ref, bound, slack=2.0):
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    lim = slack * bound + 1e-7 * (np.sqrt(np.mean(ref * ref)) + 1e-30)
    return bool(np.all(err <= lim)), float(np.max(err / lim))


@pytest.mark.parametrize("prec,T", [(0, 128), (0, 256), (0, 384), (0, 640), (0, 2048), (1, 100), (1, 200)],
                         ids=["bf16_T128", "bf16_T256", "bf16_T384", "bf16_T640", "bf16_T2048", "fp32_T100",
                              "fp32_T200"])
def test_attention_fwd_bwd(nc, prec, T):
    import torch
    B, H, D = 2, 2, 128
    d = H * D
    rng = np.random.default_rng(7)
    qkv = _qkv(rng, B, T, H, prec)
    dout = rounded(rng.standard_normal((B * T, d)), prec)
    c = Ctx(nc, 1, d, H, T, 1024, B, prec)
    try:
        elem = torch.bfloat16 if prec == 0 else torch.float32
        dq = torch_of(qkv, prec, nc)
        o = torch.zeros((B * T, d), dtype=elem, device="cuda")
        lse = torch.zeros((B, H, T), dtype=torch.float32, device="cuda")
        nc.nc_op_attention_fwd(c.ctx, dq.data_ptr(), o.data_ptr(), lse.data_ptr())
        ddo = torch_of(dout, prec, nc)
        dqk = torch.zeros((2, B * T, d), dtype=torch.float32, device="cuda")
        dqkv = torch.zeros((B * T, 3 * d), dtype=elem, device="cuda")
        nc.nc_op_attention_bwd(c.ctx, dq.data_ptr(), o.data_ptr(), ddo.data_ptr(), lse.data_ptr(),
                               dqk.data_ptr(), dqkv.data_ptr())
        nc.nc_sync(c.ctx)
        o_h, lse_h, dqk_h, dqkv_h = host(o), lse.cpu().numpy(), dqk.cpu().numpy(), host(dqkv)
        for b in range(B):
            x = qkv.reshape(B, T, 3, H, D)[b].astype(np.float64)
            q, k, v = x[:, 0], x[:, 1], x[:, 2]
            o_ref, lse_ref = oracle.causal_attention(q, k, v)
            ob = o_h.reshape(B, T, H, D)[b].astype(np.float64)
            g = dout.reshape(B, T, H, D)[b].astype(np.float64)
            bo, bdq, bdk, bdv = attention_bounds(q, k, v, g, o_ref, ob, prec)
            ok, worst = within(ob, o_ref, bo)
            assert ok, ("o", b, worst)
            # and in aggregate, where a small systematic error would show
            assert np.linalg.norm(ob - o_ref) <= (1e-2 if prec == 0 else 1e-5) * np.linalg.norm(o_ref)
            np.testing.assert_allclose(lse_h[b], lse_ref, atol=1e-3 if prec == 0 else 1e-5)
            dq_r, dk_r, dv_r = oracle.causal_attention_backward(q, k, v, g)
            got = dqk_h.reshape(2, B, T, H, D)[:, b]
            for name, gg, rr, bb in (("dq", got[0], dq_r, bdq), ("dk", got[1], dk_r, bdk),
                                     ("dv", dqkv_h.reshape(B, T, 3, H, D)[b][:, 2], dv_r, bdv)):
                ok, worst = within(gg, rr, bb)
                assert ok, (name, b, worst)
                assert np.linalg.norm(gg - rr) <= (2e-2 if prec == 0 else 2e-5) * np.linalg.norm(rr), name
        assert np.all(dqkv_h.reshape(B, T, 3, d)[:, :, :2] == 0)  # q,k columns untouched
    finally:
        c.close()


# ---------------------------------------------------------------- lm_head + CE

@pytest.mark.parametrize("prec", [0, 1], ids=["bf16", "fp32"])
def test_lmhead_cross_entropy(nc, prec):
    import torch
    d, H, T, B, V = 256, 2, 128, 3, 4224  # 16.5 vocabulary tiles of 256
    M = B * T
    rng = np.random.default_rng(11)
    hf = rng.standard_normal((M, d))
    hf = rounded(hf / np.sqrt(np.mean(hf * hf, -1, keepdims=True)), prec)
    wl = rounded(rng.standard_normal((V, d)) * 0.05, prec)
    tgt = rng.integers(0, V, M).astype(np.int32)
    c = Ctx(nc, 1, d, H, T, V, B, prec)
    try:
        dh, dw, dt = torch_of(hf, prec, nc), torch_of(wl, prec, nc), torch.from_numpy(tgt).cuda()
        lse = torch.zeros(M, dtype=torch.float32, device="cuda")
        nll = torch.zeros(M, dtype=torch.float32, device="cuda")
        am = torch.zeros(M, dtype=torch.int32, device="cuda")
        nc.nc_op_lmhead_ce_fwd(c.ctx, dh.data_ptr(), dw.data_ptr(), dt.data_ptr(), lse.data_ptr(),
                               nll.data_ptr(), am.data_ptr())
        dhf = torch.zeros((M, d), dtype=torch.float32, device="cuda")
        dwl = torch.full((V, d), 3.0, dtype=torch.float32, device="cuda")  # must be overwritten
        nc.nc_op_lmhead_ce_bwd(c.ctx, dh.data_ptr(), dw.data_ptr(), dt.data_ptr(), lse.data_ptr(),
                               dhf.data_ptr(), dwl.data_ptr())
        nc.nc_sync(c.ctx)
        h64, w64 = hf.astype(np.float64), wl.astype(np.float64)
        lse_r, nll_r, am_r = oracle.cross_entropy_rows(h64, w64, tgt)
        tol = 1e-3 if prec == 0 else 1e-5
        np.testing.assert_allclose(lse.cpu().numpy(), lse_r, atol=tol)
        np.testing.assert_allclose(nll.cpu().numpy(), nll_r, atol=tol)
        lg = h64 @ w64.T
        top2 = np.partition(lg, -2, axis=1)[:, -2:]
        sure = (top2[:, 1] - top2[:, 0]) > 1e-4
        np.testing.assert_array_equal(am.cpu().numpy()[sure], am_r[sure])
        dhf_r, dw_r = oracle.cross_entropy_backward(h64, w64, tgt, lse_r)
        # element-wise: g = softmax - onehot is rounded to bf16 (relative 2^-9)
        # before both products, whose sums then carry that rounding
        for name, got, ref in (("dhf", dhf.cpu().numpy(), dhf_r), ("dw_lm", dwl.cpu().numpy(), dw_r)):
            ok, err = close_enough(got, ref, prec, rel_bf16=2e-2, rel_f32=2e-5)
            assert ok, (name, err)
    finally:
        c.close()


# ---------------------------------------------------------------- norms

@pytest.mark.parametrize("prec", [0, 1], ids=["bf16", "fp32"])
def test_qk_norm_rope_and_rmsnorm(nc, prec):
    import torch
    B, T, H = 2, 256, 3
    d, D = H * 128, 128
    rng = np.random.default_rng(5)
    qkv = rounded(rng.standard_normal((B * T, 3 * d)) * 0.3, prec)
    x = rng.standard_normal((B * T, d)).astype(np.float32) * 2
    c = Ctx(nc, 1, d, H, T, 1024, B, prec)
    try:
        dq = torch_of(qkv, prec, nc)
        rqk = torch.zeros((B * T, 2 * H), dtype=torch.float32, device="cuda")
        nc.nc_op_qk_norm_rope_fwd(c.ctx, dq.data_ptr(), rqk.data_ptr())
        dx = torch.from_numpy(x).cuda()
        elem = torch.bfloat16 if prec == 0 else torch.float32
        y = torch.zeros((B * T, d), dtype=elem, device="cuda")
        r = torch.zeros(B * T, dtype=torch.float32, device="cuda")
        nc.nc_op_rmsnorm_fwd(c.ctx, dx.data_ptr(), y.data_ptr(), r.data_ptr())
        nc.nc_sync(c.ctx)
        cos, sin = oracle.rope_angles(T)
        got = host(dq).reshape(B, T, 3, H, D)
        src = qkv.reshape(B, T, 3, H, D).astype(np.float64)
        for which in (0, 1):
            for b in range(B):
                n, rr = oracle.rmsnorm(src[b, :, which])
                ref = oracle.rope(n, cos, sin)
                ok, err = close_enough(got[b, :, which], ref, prec)
                assert ok, err
                np.testing.assert_allclose(rqk.cpu().numpy().reshape(B, T, 2, H)[b, :, which], rr[..., 0], rtol=1e-5)
        np.testing.assert_array_equal(got[:, :, 2], qkv.reshape(B, T, 3, H, D)[:, :, 2])  # v untouched
        yn, rn = oracle.rmsnorm(x.astype(np.float64))
        ok, err = close_enough(host(y), yn, prec)
        assert ok, err
        np.testing.assert_allclose(r.cpu().numpy(), rn[:, 0], rtol=1e-5)
    finally:
        c.close()


# ---------------------------------------------------------------- embedding, RMSNorm and QK-norm/RoPE backward

@pytest.mark.parametrize("prec", [0, 1], ids=["bf16", "fp32"])
def test_embedding_forward_and_backward(nc, prec):
    """x = wte[tok] exactly (bf16 -> fp32 is exact); dwte[id] = sum of dx over
    the positions holding id (the oracle's np.add.at), absent ids exactly 0;
    an id out of range is reported as a device error, not trapped."""
    import torch
    B, T, H, V = 2, 256, 3, 1024
    d = H * 128
    M = B * T
    rng = np.random.default_rng(41)
    tok = np.minimum(rng.zipf(1.3, M) - 1, V - 1).astype(np.int32)  # repeated ids, a heavy first id
    wte = rounded(rng.standard_normal((V, d)) * 0.02, prec)
    dx = rng.standard_normal((M, d)).astype(np.float32)
    c = Ctx(nc, 1, d, H, T, V, B, prec)
    try:
        dtok, dw = torch.from_numpy(tok).cuda(), torch_of(wte, prec, nc)
        x = torch.full((M, d), np.nan, dtype=torch.float32, device="cuda")
        nc.nc_op_embed_fwd(c.ctx, dtok.data_ptr(), dw.data_ptr(), x.data_ptr())
        dwte = torch.full((V, d), 5.0, dtype=torch.float32, device="cuda")  # must be overwritten
        ddx = torch.from_numpy(dx).cuda()
        nc.nc_op_embed_bwd(c.ctx, dtok.data_ptr(), ddx.data_ptr(), dwte.data_ptr())
        nc.nc_sync(c.ctx)
        np.testing.assert_array_equal(x.cpu().numpy(), wte[tok])
        ref = np.zeros((V, d))
        np.add.at(ref, tok, dx.astype(np.float64))
        got = dwte.cpu().numpy()
        counts = np.bincount(tok, minlength=V)
        # fp32 sums of n terms: |err| <= n * 2^-24 * sum |terms| (a loose bound per row)
        bound = np.zeros((V, d))
        np.add.at(bound, tok, np.abs(dx.astype(np.float64)))
        assert np.all(np.abs(got - ref) <= counts[:, None] * 2.0 ** -23 * bound + 1e-30)
        assert np.all(got[counts == 0] == 0.0)
        bad = tok.copy()
        bad[5] = V
        nc.nc_op_embed_fwd(c.ctx, torch.from_numpy(bad).cuda().data_ptr(), dw.data_ptr(), x.data_ptr())
        with pytest.raises(nc.NcError) as ei:
            nc.nc_sync(c.ctx)
        assert ei.value.status == 5  # NC_ERR_DEVICE
        assert np.all(x.cpu().numpy()[5] == 0.0)
    finally:
        c.close()


def test_embedding_backward_is_deterministic_at_batch_size(nc):
    """At the d20 batch (32,768 positions, vocabulary 65,536, Zipf(1.1) ids:
    the heaviest id holds thousands of positions) the embedding gradient is
    the same bit for bit on every run, and within the fp32 summation bound
    of the float64 sum (nanochat explainer, "Pretraining": every position's
    gradient flows back into the row of its token)."""
    import torch
    B, T, H, V = 16, 2048, 2, 65536
    d = H * 128
    M = B * T
    rng = np.random.default_rng(7)
    tok = np.minimum(rng.zipf(1.1, M) - 1, V - 1).astype(np.int32)
    dx = rng.standard_normal((M, d)).astype(np.float32)
    c = Ctx(nc, 1, d, H, T, V, B, 0)
    try:
        dtok, ddx = torch.from_numpy(tok).cuda(), torch.from_numpy(dx).cuda()
        runs = []
        for _ in range(3):
            dwte = torch.full((V, d), 5.0, dtype=torch.float32, device="cuda")
            nc.nc_op_embed_bwd(c.ctx, dtok.data_ptr(), ddx.data_ptr(), dwte.data_ptr())
            nc.nc_sync(c.ctx)
            runs.append(dwte.cpu().numpy())
        for r in runs[1:]:
            assert np.array_equal(r.view(np.uint32), runs[0].view(np.uint32))
        counts = np.bincount(tok, minlength=V)
        assert counts.max() > 1000
        ref = np.zeros((V, d))
        np.add.at(ref, tok, dx.astype(np.float64))
        bound = np.zeros((V, d))
        np.add.at(bound, tok, np.abs(dx.astype(np.float64)))
        got = runs[0]
        assert np.all(np.abs(got - ref) <= counts[:, None] * 2.0 ** -23 * bound + 1e-30)
        assert np.all(got[counts == 0] == 0.0)
    finally:
        c.close()


@pytest.mark.parametrize("prec", [0, 1], ids=["bf16", "fp32"])
@pytest.mark.parametrize("accumulate", [0, 1], ids=["store", "accumulate"])
def test_rmsnorm_backward(nc, prec, accumulate):
    """dz = r (dy - y mean(dy y)) (+ dx when accumulating), element-wise
    against the oracle's rmsnorm_backward on the same rounded y and dy."""
    import torch
    B, T, H = 2, 256, 3
    d = H * 128
    M = B * T
    rng = np.random.default_rng(43 + accumulate)
    z = rng.standard_normal((M, d)) * 3
    y, r = oracle.rmsnorm(z)
    y = rounded(y, prec)
    dy = rounded(rng.standard_normal((M, d)) * 0.1, prec)
    dx0 = rng.standard_normal((M, d)).astype(np.float32)
    c = Ctx(nc, 1, d, H, T, 1024, B, prec)
    try:
        elem = torch.bfloat16 if prec == 0 else torch.float32
        ddy, dyv = torch_of(dy, prec, nc), torch_of(y, prec, nc)
        dr = torch.from_numpy(r[:, 0].astype(np.float32)).cuda()
        dx = torch.from_numpy(dx0.copy()).cuda()
        dxe = torch.zeros((M, d), dtype=elem, device="cuda")
        nc.nc_op_rmsnorm_bwd(c.ctx, ddy.data_ptr(), dyv.data_ptr(), dr.data_ptr(), dx.data_ptr(), dxe.data_ptr(),
                             accumulate)
        nc.nc_sync(c.ctx)
        ref = oracle.rmsnorm_backward(dy.astype(np.float64), y.astype(np.float64),
                                      r.astype(np.float32).astype(np.float64))
        if accumulate:
            ref = ref + dx0
        ok, err = close_enough(dx.cpu().numpy(), ref, 1, rel_f32=2e-5)
        assert ok, err
        ok, err = close_enough(host(dxe), ref, prec, rel_bf16=8e-3, rel_f32=2e-5)
        assert ok, err
    finally:
        c.close()


@pytest.mark.parametrize("prec", [0, 1], ids=["bf16", "fp32"])
def test_qk_norm_rope_backward(nc, prec):
    """dq = r (dq_n - q_n mean(dq_n q_n)) with dq_n, q_n the inverse rotation
    of dq_hat and of the stored q_hat, for q and k heads, element-wise against
    the oracle's rope_backward and rmsnorm_backward; v columns untouched."""
    import torch
    B, T, H = 2, 256, 3
    d, D = H * 128, 128
    M = B * T
    rng = np.random.default_rng(47)
    raw = rng.standard_normal((B, T, 3, H, D)) * 0.7
    cos, sin = oracle.rope_angles(T)
    qkv = raw.copy()
    rqk = np.empty((B, T, 2, H))
    for which in (0, 1):
        for b in range(B):
            n, rr = oracle.rmsnorm(raw[b, :, which])
            qkv[b, :, which] = oracle.rope(n, cos, sin)
            rqk[b, :, which] = rr[..., 0]
    qkv = rounded(qkv.reshape(M, 3 * d), prec)
    rqk = rqk.reshape(M, 2 * H).astype(np.float32)
    dqk = rng.standard_normal((2, M, d)).astype(np.float32)
    c = Ctx(nc, 1, d, H, T, 1024, B, prec)
    try:
        elem = torch.bfloat16 if prec == 0 else torch.float32
        dq_ = torch.from_numpy(dqk).cuda()
        dqkv = torch.full((M, 3 * d), 9.0, dtype=elem, device="cuda")
        nc.nc_op_qk_norm_rope_bwd(c.ctx, dq_.data_ptr(), torch_of(qkv, prec, nc).data_ptr(),
                                  torch.from_numpy(rqk).cuda().data_ptr(), dqkv.data_ptr())
        nc.nc_sync(c.ctx)
        got = host(dqkv).reshape(B, T, 3, H, D)
        src = qkv.reshape(B, T, 3, H, D).astype(np.float64)
        for which in (0, 1):
            for b in range(B):
                g = dqk[which].reshape(B, T, H, D)[b].astype(np.float64)
                gn = oracle.rope_backward(g, cos, sin)
                qn = oracle.rope_backward(src[b, :, which], cos, sin)
                rr = rqk.reshape(B, T, 2, H)[b, :, which].astype(np.float64)[..., None]
                ref = oracle.rmsnorm_backward(gn, qn, rr)
                ok, err = close_enough(got[b, :, which], ref, prec, rel_bf16=8e-3, rel_f32=2e-5)
                assert ok, (which, b, err)
        assert np.all(got[:, :, 2] == 9.0)
    finally:
        c.close()
