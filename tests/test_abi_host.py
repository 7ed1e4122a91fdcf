"""Host-side checks of the C ABI: the library loads, exports every symbol the
public headers declare, and validates arguments without touching a GPU."""

import ctypes
import os
import re

import pytest

import oracle
import workload as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nc():
    from decoder_transformer_step_nanochat_b300 import build
    build.build()
    import decoder_transformer_step_nanochat_b300 as nc
    return nc


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        src = open(os.path.join(inc, f)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:[A-Za-z_]\w*[\s\*]+)+(nc_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(nc):
    names = declared_functions()
    assert "nc_create" in names and "nc_forward_loss" in names and "nc_backward" in names
    assert "nc_launch_count" in names and "nc_last_error" in names
    assert "nc_get_argmax" in names and "nc_get_token_outputs" in names
    L = ctypes.CDLL(nc.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # the binding mirrors every declared call under the same name
    assert not [n for n in names if not hasattr(nc, n)]


def test_create_validates_shapes(nc):
    bad = [
        (0, 128, 1, 64, 65536),       # depth < 1
        (2, 130, 1, 64, 65536),       # d_model != 128 * n_head
        (2, 256, 1, 64, 65536),
        (2, 128, 1, 64, 65537),       # vocab not a multiple of 128
        (2, 128, 1, 0, 65536),        # empty sequence
    ]
    for args in bad:
        with pytest.raises(nc.NcError) as ei:
            nc.nc_create(*args)
        assert ei.value.status == 1  # NC_ERR_ARG
        assert nc.nc_last_error()


def test_param_layout_matches_oracle(nc):
    for name in ("tiny", "small", "d20"):
        w = W.WORKLOADS[name]
        ctx = nc.nc_create(w.depth, w.d_model, w.n_head, w.seq_len, w.vocab)
        try:
            s = oracle.Shape(w.depth, w.d_model, w.n_head, w.vocab)
            assert nc.nc_param_count(ctx) == oracle.param_count(s) == W.n_params(w)
            for i, (_, off, r, c) in enumerate(oracle.layout(s)):
                assert nc.nc_param_offset(ctx, i) == (off, r, c)
            with pytest.raises(nc.NcError):
                nc.nc_param_offset(ctx, 2 + 4 * w.depth)
        finally:
            nc.nc_destroy(ctx)


def test_calls_before_configure_are_rejected(nc):
    ctx = nc.nc_create(2, 128, 1, 64, 65536)
    try:
        assert nc.nc_workspace_bytes(ctx) == 0
        with pytest.raises(nc.NcError) as ei:
            nc.nc_set_workspace(ctx, 1024, 1 << 20)
        assert ei.value.status == 2  # NC_ERR_STATE
        with pytest.raises(nc.NcError) as ei:
            nc.nc_backward(ctx, 1024)
        assert ei.value.status == 2
        with pytest.raises(nc.NcError):
            nc.nc_forward_loss(ctx, 1024, 1024, 1024)
        # bad arguments are rejected before any device work
        with pytest.raises(nc.NcError) as ei:
            nc.nc_configure(ctx, 0, nc.NC_FP32_DEBUG)
        assert ei.value.status == 1
        with pytest.raises(nc.NcError) as ei:
            nc.nc_configure(ctx, 4, 7)
        assert ei.value.status == 1
        # bf16 mode needs seq_len % 128 == 0; this model has seq 64
        with pytest.raises(nc.NcError) as ei:
            nc.nc_configure(ctx, 4, nc.NC_BF16)
        assert ei.value.status == 1
    finally:
        nc.nc_destroy(ctx)
    nc.nc_destroy(None)  # allowed


def test_configure_without_gpu_reports_cuda_error(nc):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    ctx = nc.nc_create(2, 128, 1, 64, 65536)
    try:
        with pytest.raises(nc.NcError) as ei:
            nc.nc_configure(ctx, 4, nc.NC_FP32_DEBUG)
        assert ei.value.status == 3  # NC_ERR_CUDA
    finally:
        nc.nc_destroy(ctx)


def test_accumulation_and_u16_entry_points_validate_before_device_work(nc):
    """Null pointers and a non-finite accumulation scale are argument errors;
    on an unconfigured context the calls report the state error, and nothing
    reaches a device."""
    ctx = nc.nc_create(2, 128, 1, 64, 65536)
    try:
        for bad in (lambda: nc.nc_backward_accumulate(ctx, None, 0.5),
                    lambda: nc.nc_backward_accumulate(ctx, 1024, float("nan")),
                    lambda: nc.nc_backward_accumulate(ctx, 1024, float("inf")),
                    lambda: nc.nc_forward_loss_u16(ctx, None, 1024, 1024),
                    lambda: nc.nc_forward_loss_u16(ctx, 1024, None, 1024),
                    lambda: nc.nc_forward_loss_u16(ctx, 1024, 1024, None)):
            with pytest.raises(nc.NcError) as ei:
                bad()
            assert ei.value.status == 1  # NC_ERR_ARG
        with pytest.raises(nc.NcError) as ei:
            nc.nc_backward_accumulate(ctx, 1024, 0.5)
        assert ei.value.status == 2  # NC_ERR_STATE: not configured
        with pytest.raises(nc.NcError) as ei:
            nc.nc_forward_loss_u16(ctx, 1024, 1024, 1024)
        assert ei.value.status == 2
    finally:
        nc.nc_destroy(ctx)


def test_argmax_query_validates_before_device_work(nc):
    """nc_get_argmax: a NULL destination is an argument error; on an
    unconfigured context (so with no forward to read) it is a state error."""
    ctx = nc.nc_create(2, 128, 1, 64, 65536)
    try:
        with pytest.raises(nc.NcError) as ei:
            nc.nc_get_argmax(ctx, None)
        assert ei.value.status == 1  # NC_ERR_ARG
        with pytest.raises(nc.NcError) as ei:
            nc.nc_get_argmax(ctx, 1024)
        assert ei.value.status == 2  # NC_ERR_STATE
    finally:
        nc.nc_destroy(ctx)
