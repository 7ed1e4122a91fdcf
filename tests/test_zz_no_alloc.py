"""The allocation-free lm_head + cross-entropy forward (nc_lmhead_ce_fwd_static).

Callers that cannot call cudaMalloc at the point where they need the loss
(code inside another framework's memory pool or allocation budget) use this
entry point: its scratch lives in a static device array of the library. The
test checks it, through the C ABI, on two calls in a row with different
inputs (so a call that left stale scratch behind would show), against the
oracle's cross-entropy rows in float64 at row counts that take the
single-CTA path (100 rows), a ragged last row block (1000 rows) and the
largest request the static buffer holds at V = 65,536 (2,728 rows), and
against the workspace-based entry point nc_op_lmhead_ce_fwd at 2,048 rows.
It must pass in a fresh process and after the other tests.
"""

import numpy as np
import pytest

import oracle
import workload as W
from gpu_util import load_nc

pytestmark = pytest.mark.gpu


def _inputs(rng, M, d, V):
    hf = rng.standard_normal((M, d))
    hf = W.round_bf16(hf / np.sqrt(np.mean(hf * hf, -1, keepdims=True)))
    wl = W.round_bf16(rng.standard_normal((V, d)) * 0.05)
    tgt = rng.integers(0, V, M).astype(np.int32)
    return hf, wl, tgt


def _check_against_oracle(hf, wl, tgt, lse, nll, am):
    h64, w64 = hf.astype(np.float64), wl.astype(np.float64)
    lse_r, nll_r, am_r = oracle.cross_entropy_rows(h64, w64, tgt)
    np.testing.assert_allclose(lse, lse_r, atol=1e-3)
    np.testing.assert_allclose(nll, nll_r, atol=1e-3)
    lg = h64 @ w64.T
    top2 = np.partition(lg, -2, axis=1)[:, -2:]
    sure = (top2[:, 1] - top2[:, 0]) > 1e-4
    assert sure.mean() > 0.9
    np.testing.assert_array_equal(am[sure], am_r[sure])


def _static_call(nc, dh, dw, dt, M, d, V):
    import torch
    lse = torch.full((M,), np.nan, dtype=torch.float32, device="cuda")
    nll = torch.full((M,), np.nan, dtype=torch.float32, device="cuda")
    am = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    nc.nc_lmhead_ce_fwd_static(dh.data_ptr(), dw.data_ptr(), dt.data_ptr(), M, d, V, lse.data_ptr(),
                               nll.data_ptr(), am.data_ptr(), status.data_ptr(), None)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return lse.cpu().numpy(), nll.cpu().numpy(), am.cpu().numpy()


@pytest.mark.parametrize("M", [100, 1000, 2728])
def test_static_scratch_ce_matches_oracle_on_two_calls(M):
    import torch
    nc = load_nc()
    d, V = 256, 65536
    rng = np.random.default_rng(77 + M)
    for call in range(2):
        hf, wl, tgt = _inputs(rng, M, d, V)
        dh = torch.from_numpy(hf).to(torch.bfloat16).cuda()
        dw = torch.from_numpy(wl).to(torch.bfloat16).cuda()
        dt = torch.from_numpy(tgt).cuda()
        lse, nll, am = _static_call(nc, dh, dw, dt, M, d, V)
        assert np.all(np.isfinite(lse)) and np.all(np.isfinite(nll))
        _check_against_oracle(hf, wl, tgt, lse, nll, am)


def test_static_scratch_ce_matches_workspace_entry_point_on_two_calls():
    import torch
    nc = load_nc()
    d, H, T, B, V = 256, 2, 128, 16, 65536  # M = 2048 rows, 512 vocabulary tiles of 128
    M = B * T
    step = nc.Step(1, d, H, T, V, B, nc.NC_BF16)
    try:
        rng = np.random.default_rng(2024)
        for call in range(2):
            hf, wl, tgt = _inputs(rng, M, d, V)
            dh = torch.from_numpy(hf).to(torch.bfloat16).cuda()
            dw = torch.from_numpy(wl).to(torch.bfloat16).cuda()
            dt = torch.from_numpy(tgt).cuda()
            outs = []
            for which in ("workspace", "static"):
                lse = torch.full((M,), np.nan, dtype=torch.float32, device="cuda")
                nll = torch.full((M,), np.nan, dtype=torch.float32, device="cuda")
                am = torch.full((M,), -1, dtype=torch.int32, device="cuda")
                if which == "workspace":
                    nc.nc_op_lmhead_ce_fwd(step.ctx, dh.data_ptr(), dw.data_ptr(), dt.data_ptr(),
                                           lse.data_ptr(), nll.data_ptr(), am.data_ptr())
                    nc.nc_sync(step.ctx)
                else:
                    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
                    nc.nc_lmhead_ce_fwd_static(dh.data_ptr(), dw.data_ptr(), dt.data_ptr(), M, d, V,
                                               lse.data_ptr(), nll.data_ptr(), am.data_ptr(),
                                               status.data_ptr(), None)
                    torch.cuda.synchronize()
                    assert int(status.item()) == 0
                outs.append((lse.cpu().numpy(), nll.cpu().numpy(), am.cpu().numpy()))
            (l0, n0, a0), (l1, n1, a1) = outs
            assert np.all(np.isfinite(l1)) and np.all(np.isfinite(n1))
            np.testing.assert_allclose(l1, l0, atol=1e-3)
            np.testing.assert_allclose(n1, n0, atol=1e-3)
            lg = hf.astype(np.float64) @ wl.astype(np.float64).T
            top2 = np.partition(lg, -2, axis=1)[:, -2:]
            sure = (top2[:, 1] - top2[:, 0]) > 1e-4
            np.testing.assert_array_equal(a1[sure], a0[sure])
            _check_against_oracle(hf, wl, tgt, l1, n1, a1)
    finally:
        step.close()


def test_static_scratch_ce_rejects_sizes_beyond_its_buffer():
    nc = load_nc()
    # 2729 rows at V = 65536 need more than the 16 MiB static scratch; the
    # call is rejected on the host before any device work
    with pytest.raises(nc.NcError) as ei:
        nc.nc_lmhead_ce_fwd_static(256, 256, 256, 2729, 256, 65536, 256, 256, 256)
    assert ei.value.status == 6  # NC_ERR_UNSUPPORTED
    assert "16 MiB" in nc.nc_last_error()
