"""The supervised fine-tuning variant of the step (masked cross-entropy):
targets of -1 mark prompt positions that carry no loss (nanochat explainer,
"Supervised Fine-Tuning (SFT)"). Parity with the oracle through the C ABI on
seeded prompt/response turns, with the same tolerances as the full step."""

import numpy as np
import pytest

import oracle
import workload as W
from gpu_util import load_nc, per_tensor, run_gpu_step, shape_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nc():
    return load_nc()


def test_tiny_fp32_masked_step_matches_oracle(nc):
    w = W.WORKLOADS["tiny"]
    p = W.make_params(w)
    tok, tgt = W.make_tokens(w)
    sft = W.make_sft_targets(tgt, seed=5, mean_turn=16)
    keep = (sft != -1).reshape(-1)
    assert 0 < keep.sum() < keep.size
    loss_ref, g_ref, cache = oracle.step(p.astype(np.float64), tok, sft, shape_of(w), np.float64)
    loss, g, lse, nll, am, _ = run_gpu_step(nc, w, p, tok, sft, nc.NC_FP32_DEBUG)
    assert abs(loss - loss_ref) <= 1e-4 * abs(loss_ref)
    np.testing.assert_allclose(nll, cache["nll"], rtol=1e-4, atol=1e-4)
    assert np.all(nll[~keep] == 0.0)
    np.testing.assert_array_equal(am, cache["argmax"])
    bad = [(n, r) for n, r, _ in per_tensor(w, g, g_ref) if not r <= 1e-4]
    assert not bad, bad


def test_small_bf16_masked_step_matches_oracle(nc):
    w = W.WORKLOADS["small"]
    p = W.make_params(w)
    tok, tgt = W.make_tokens(w)
    sft = W.make_sft_targets(tgt, seed=6, mean_turn=128)
    keep = (sft != -1).reshape(-1)
    loss_ref, g_ref, cache = oracle.step(p.astype(np.float64), tok, sft, shape_of(w), np.float64)
    loss, g, lse, nll, am, _ = run_gpu_step(nc, w, p, tok, sft, nc.NC_BF16)
    assert abs(loss - loss_ref) <= 2e-2, (loss, loss_ref)
    bad = [(n, r, c) for n, r, c in per_tensor(w, g, g_ref) if not (r <= 3e-2 and c >= 0.999)]
    assert not bad, bad
    assert np.all(nll[~keep] == 0.0)
    np.testing.assert_allclose(nll[keep], cache["nll"][keep], atol=6e-2)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_fully_masked_batch_gives_zero_loss_and_gradient(nc, name):
    w = W.WORKLOADS[name]
    p = W.make_params(w)
    tok, tgt = W.make_tokens(w)
    none = np.full_like(tgt, -1)
    prec = nc.NC_FP32_DEBUG if w.dtype == "fp32" else nc.NC_BF16
    loss, g, lse, nll, am, _ = run_gpu_step(nc, w, p, tok, none, prec)
    assert loss == 0.0 and not np.any(g) and not np.any(nll)


def test_other_negative_targets_are_rejected(nc):
    w = W.WORKLOADS["tiny"]
    p = W.make_params(w)
    tok, tgt = W.make_tokens(w)
    tgt[0, 5] = -2
    with pytest.raises(nc.NcError) as ei:
        run_gpu_step(nc, w, p, tok, tgt, nc.NC_FP32_DEBUG)
    assert ei.value.status == 5  # NC_ERR_DEVICE
