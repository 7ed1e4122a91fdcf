"""Run one step of the path at the d20 shapes through the C ABI, for profiling.

  python -m decoder_transformer_step_nanochat_b300.profile_cases CASE [--reps N]

CASE: gemm_qkv (32768 x 3840 x 1280 forward GEMM), gemm_fc (32768 x 5120 x 1280
with the ReLU^2 epilogue), gemm_relu2_bwd (32768 x 5120 x 1280 with the ReLU^2
backward epilogue, which reads a), gemm_dw (1280 x 5120 x 32768 weight
gradient),
attn_fwd / attn_bwd (batch 16, seq 2048, 10 heads: 252 MB of qkv, larger
than L2), lmhead_ce (4096 rows x 65536 vocabulary x 1280). Inputs are random
and device-resident; every launch goes through the library.
"""

from __future__ import annotations

import argparse
import sys

import torch

import decoder_transformer_step_nanochat_b300 as nc


def _gemm(ctx, M, N, K, ak, bk, epi):
    A = torch.randn((M, K) if ak else (K, M), device="cuda").to(torch.bfloat16)
    B = (torch.randn((N, K) if bk else (K, N), device="cuda") * 0.05).to(torch.bfloat16)
    C = torch.empty((M, N), device="cuda", dtype=torch.float32 if epi == nc.NC_EPI_STORE_F32 else torch.bfloat16)
    C2 = None
    if epi == nc.NC_EPI_RELU2:
        C2 = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
    elif epi == nc.NC_EPI_RELU2_BWD:
        C2 = torch.rand((M, N), device="cuda").to(torch.bfloat16)   # a >= 0
    args = (ctx, M, N, K, A.data_ptr(), K if ak else M, ak, B.data_ptr(), K if bk else N, bk, epi, 1.0, 0.0,
            C.data_ptr(), N, C2.data_ptr() if C2 is not None else None, N if C2 is not None else 0)
    return lambda: nc.nc_op_gemm(*args), (A, B, C, C2)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["gemm_qkv", "gemm_fc", "gemm_relu2_bwd", "gemm_dw", "attn_fwd", "attn_bwd", "lmhead_ce"])
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args(argv)
    B, T, H, V = 16, 2048, 10, 65536
    d = H * 128
    if a.case == "lmhead_ce":
        B = 2
    st = nc.Step(1, d, H, T, V, B, nc.NC_BF16)
    ctx = st.ctx
    keep = None
    if a.case == "gemm_qkv":
        run, keep = _gemm(ctx, 32768, 3 * d, d, 1, 1, nc.NC_EPI_STORE)
    elif a.case == "gemm_fc":
        run, keep = _gemm(ctx, 32768, 4 * d, d, 1, 1, nc.NC_EPI_RELU2A)
    elif a.case == "gemm_relu2_bwd":
        run, keep = _gemm(ctx, 32768, 4 * d, d, 1, 0, nc.NC_EPI_RELU2_BWD)
    elif a.case == "gemm_dw":
        run, keep = _gemm(ctx, d, 4 * d, 32768, 0, 0, nc.NC_EPI_STORE_F32)
    elif a.case in ("attn_fwd", "attn_bwd"):
        M = B * T
        q = torch.randn((M, 3 * d), device="cuda")
        qkv = q.to(torch.bfloat16)
        o = torch.empty((M, d), device="cuda", dtype=torch.bfloat16)
        lse = torch.empty((B, H, T), device="cuda", dtype=torch.float32)
        dout = torch.randn((M, d), device="cuda").to(torch.bfloat16)
        dqk = torch.empty((2, M, d), device="cuda", dtype=torch.float32)
        dqkv = torch.empty((M, 3 * d), device="cuda", dtype=torch.bfloat16)
        nc.nc_op_attention_fwd(ctx, qkv.data_ptr(), o.data_ptr(), lse.data_ptr())
        if a.case == "attn_fwd":
            def run():
                nc.nc_op_attention_fwd(ctx, qkv.data_ptr(), o.data_ptr(), lse.data_ptr())
        else:
            def run():
                nc.nc_op_attention_bwd(ctx, qkv.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                                       dqk.data_ptr(), dqkv.data_ptr())
        keep = (qkv, o, lse, dout, dqk, dqkv)
    else:
        M = B * T
        hf = torch.randn((M, d), device="cuda").to(torch.bfloat16)
        w = (torch.randn((V, d), device="cuda") * 0.02).to(torch.bfloat16)
        tgt = torch.randint(0, V, (M,), device="cuda", dtype=torch.int32)
        lse = torch.empty(M, device="cuda")
        nll = torch.empty(M, device="cuda")
        am = torch.empty(M, device="cuda", dtype=torch.int32)

        def run():
            nc.nc_op_lmhead_ce_fwd(ctx, hf.data_ptr(), w.data_ptr(), tgt.data_ptr(), lse.data_ptr(),
                                   nll.data_ptr(), am.data_ptr())
        keep = (hf, w, tgt, lse, nll, am)
    torch.cuda.synchronize()
    for _ in range(a.reps):
        run()
    nc.nc_sync(ctx)
    del keep
    st.close()
    print(f"{a.case}: ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
