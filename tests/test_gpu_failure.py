"""The failure path of the tensor-core kernels on a GPU, in a form that
faults and hangs nothing: every pipeline wait of those kernels has a time
limit, after which the kernel records a timeout, waits (with the full limit)
for the copies and products it has in flight, frees its tensor memory and
returns. The test lowers the limit (nc_set_pipeline_wait_limit) so that the
waits give up at once, checks that the attention forward, the attention
backward and a single-CTA GEMM each report NC_ERR_TIMEOUT, restores the
limit, and checks that the same context then gives the oracle's results."""

import numpy as np
import pytest

import oracle
import workload as W
from gpu_util import load_nc, rel_l2

pytestmark = pytest.mark.gpu

NC_ERR_TIMEOUT = 4


def _attention_inputs(rng, B, T, H):
    D = 128
    q = rng.standard_normal((B, T, H, D))
    k = rng.standard_normal((B, T, H, D))
    q /= np.sqrt(np.mean(q * q, -1, keepdims=True))
    k /= np.sqrt(np.mean(k * k, -1, keepdims=True))
    v = rng.standard_normal((B, T, H, D))
    qkv = np.concatenate([q.reshape(B, T, -1), k.reshape(B, T, -1), v.reshape(B, T, -1)], -1)
    return W.round_bf16(qkv).reshape(B * T, 3 * H * D), W.round_bf16(rng.standard_normal((B * T, H * D)))


def test_short_wait_limit_reports_timeout_and_the_context_recovers():
    import torch
    nc = load_nc()
    B, T, H, V = 2, 256, 2, 1024
    d = H * 128
    M = B * T
    rng = np.random.default_rng(99)
    qkv_np, dout_np = _attention_inputs(rng, B, T, H)
    a_np = W.round_bf16(rng.standard_normal((128, 256)))
    b_np = W.round_bf16(rng.standard_normal((256, 256)) * 0.1)
    st = nc.Step(1, d, H, T, V, B, nc.NC_BF16)
    try:
        bf = torch.bfloat16
        qkv = torch.from_numpy(qkv_np).to(bf).cuda()
        dout = torch.from_numpy(dout_np).to(bf).cuda()
        o = torch.zeros((M, d), dtype=bf, device="cuda")
        lse = torch.zeros((B, H, T), dtype=torch.float32, device="cuda")
        dqk = torch.zeros((2, M, d), dtype=torch.float32, device="cuda")
        dqkv = torch.zeros((M, 3 * d), dtype=bf, device="cuda")
        ga = torch.from_numpy(a_np).to(bf).cuda()
        gb = torch.from_numpy(b_np).to(bf).cuda()
        gc = torch.zeros((128, 256), dtype=torch.float32, device="cuda")

        def fwd():
            nc.nc_op_attention_fwd(st.ctx, qkv.data_ptr(), o.data_ptr(), lse.data_ptr())

        def bwd():
            nc.nc_op_attention_bwd(st.ctx, qkv.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                                   dqk.data_ptr(), dqkv.data_ptr())

        def gemm():  # 128 rows: one CTA per tile, no CTA pairs
            nc.nc_op_gemm(st.ctx, 128, 256, 256, ga.data_ptr(), 256, 1, gb.data_ptr(), 256, 1,
                          nc.NC_EPI_STORE_F32, 1.0, 0.0, gc.data_ptr(), 256)

        for name, run in (("attention forward", fwd), ("attention backward", bwd), ("GEMM", gemm)):
            nc.nc_set_pipeline_wait_limit(1)
            try:
                run()
                with pytest.raises(nc.NcError) as ei:
                    nc.nc_sync(st.ctx)
                assert ei.value.status == NC_ERR_TIMEOUT, name
            finally:
                nc.nc_set_pipeline_wait_limit(0)
            nc.nc_sync(st.ctx)  # the status word was reset by the report: nothing pending

        # the same context with the default limit gives the oracle's results
        fwd()
        bwd()
        gemm()
        nc.nc_sync(st.ctx)
        o_h = o.float().cpu().numpy().reshape(B, T, H, 128)
        dq_h = dqk.cpu().numpy().reshape(2, B, T, H, 128)
        dv_h = dqkv.float().cpu().numpy().reshape(B, T, 3, H, 128)[:, :, 2]
        for b in range(B):
            x = qkv_np.reshape(B, T, 3, H, 128)[b].astype(np.float64)
            o_ref, lse_ref = oracle.causal_attention(x[:, 0], x[:, 1], x[:, 2])
            assert rel_l2(o_h[b], o_ref) <= 1e-2
            np.testing.assert_allclose(lse.cpu().numpy()[b], lse_ref, atol=1e-3)
            dq_r, dk_r, dv_r = oracle.causal_attention_backward(x[:, 0], x[:, 1], x[:, 2],
                                                                dout_np.reshape(B, T, H, 128)[b].astype(np.float64))
            assert rel_l2(dq_h[0, b], dq_r) <= 2e-2
            assert rel_l2(dq_h[1, b], dk_r) <= 2e-2
            assert rel_l2(dv_h[b], dv_r) <= 2e-2
        ref = a_np.astype(np.float64) @ b_np.astype(np.float64).T
        assert rel_l2(gc.cpu().numpy(), ref) <= 1e-5
    finally:
        nc.nc_set_pipeline_wait_limit(0)
        st.close()
