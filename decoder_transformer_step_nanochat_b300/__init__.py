"""Python binding of the nanochat pretraining-step library (libnc.so).

Argument marshalling only: every step of the forward, loss and backward runs
in the library's CUDA kernels. PyTorch is used by callers for device memory
and streams; this module takes raw device pointers (ints) and never computes
anything itself. Importing it loads libnc.so and fails loudly if it is
missing: there is no fallback implementation.

Names follow include/nc.h, include/nc_ops.h, include/nc_optim.h and
include/nc_infer.h.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnc.so")

NC_BF16 = 0
NC_FP32_DEBUG = 1

NC_FAM_GEMM = 0
NC_FAM_ATTN_FWD = 1
NC_FAM_ATTN_BWD = 2
NC_FAM_ROWS = 3
NC_FAM_OPT_NS = 4
NC_FAM_OPT_ELEM = 5
NC_FAM_DEC_GEMM = 6
NC_FAM_DEC_ATTN = 7
NC_FAM_DEC_ROWS = 8

NC_EPI_STORE = 0
NC_EPI_STORE_F32 = 1
NC_EPI_RELU2 = 2
NC_EPI_RELU2_BWD = 3
NC_EPI_CE_BWD = 4
NC_EPI_QKNORM_ROPE = 6
NC_EPI_AXPBY = 7
NC_EPI_RELU2A = 8

STATUS = {0: "NC_OK", 1: "NC_ERR_ARG", 2: "NC_ERR_STATE", 3: "NC_ERR_CUDA",
          4: "NC_ERR_TIMEOUT", 5: "NC_ERR_DEVICE", 6: "NC_ERR_UNSUPPORTED"}


class NcError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "nc_create": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_P)]),
    "nc_configure": (_I, [_P, _I, _I, _P]),
    "nc_param_count": (_SZ, [_P]),
    "nc_param_offset": (_I, [_P, _I, ctypes.POINTER(_SZ), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "nc_workspace_bytes": (_SZ, [_P]),
    "nc_set_workspace": (_I, [_P, _P, _SZ]),
    "nc_forward_loss": (_I, [_P, _P, _P, _P, ctypes.POINTER(_F)]),
    "nc_forward_loss_async": (_I, [_P, _P, _P, _P, _P]),
    "nc_backward": (_I, [_P, _P]),
    "nc_backward_accumulate": (_I, [_P, _P, _F]),
    "nc_forward_loss_u16": (_I, [_P, _P, _P, _P]),
    "nc_train_step_host_u16": (_I, [_P, _P, _P, _P, ctypes.POINTER(_F)]),
    "nc_train_step_host": (_I, [_P, _P, _P, _P, _P, ctypes.POINTER(_F)]),
    "nc_get_token_outputs": (_I, [_P, _P, _P, _P]),
    "nc_get_argmax": (_I, [_P, _P]),
    "nc_get_hidden": (_I, [_P, _P]),
    "nc_sync": (_I, [_P]),
    "nc_launch_count": (ctypes.c_ulonglong, [_P]),
    "nc_profile_enable": (_I, [_P, _I]),
    "nc_profile_read": (_I, [_P, _I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_LL),
                            ctypes.POINTER(ctypes.c_double)]),
    "nc_profile_reset": (_I, [_P]),
    "nc_set_pipeline_wait_limit": (_I, [ctypes.c_ulonglong]),
    "nc_last_error": (ctypes.c_char_p, [_P]),
    "nc_destroy": (None, [_P]),
    "nc_op_gemm": (_I, [_P, _I, _I, _I, _P, _LL, _I, _P, _LL, _I, _I, _F, _F, _P, _LL, _P, _LL, _P, _P]),
    "nc_op_lmhead_ce_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P]),
    "nc_op_lmhead_ce_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P]),
    "nc_op_attention_fwd": (_I, [_P, _P, _P, _P]),
    "nc_op_attention_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P]),
    "nc_op_qk_norm_rope_fwd": (_I, [_P, _P, _P]),
    "nc_op_rmsnorm_fwd": (_I, [_P, _P, _P, _P]),
    "nc_op_rmsnorm_bwd": (_I, [_P, _P, _P, _P, _P, _P, _I]),
    "nc_op_embed_fwd": (_I, [_P, _P, _P, _P]),
    "nc_op_embed_bwd": (_I, [_P, _P, _P, _P]),
    "nc_op_qk_norm_rope_bwd": (_I, [_P, _P, _P, _P, _P]),
    "nc_lmhead_ce_fwd_static": (_I, [_P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "nc_op_gemm_batched": (_I, [_P, _I, _I, _I, _I, _P, _LL, _I, _LL, _P, _LL, _I, _LL, _I, _F, _F, _P, _LL,
                                _P, _LL, _LL]),
    "nc_optim_state_bytes": (_SZ, [_P]),
    "nc_optim_init": (_I, [_P, _P, _P]),
    "nc_optim_set_hparams": (_I, [_P, _F, _F, _F, _F, _I]),
    "nc_optim_step": (_I, [_P, _P, _P, _P, _I, _F, _F, _F, _F, _P]),
    "nc_lr_at": (ctypes.c_double, [_LL, _LL, _LL, ctypes.c_double, ctypes.c_double]),
    "nc_kv_cache_bytes": (_SZ, [_P, _I]),
    "nc_prefill": (_I, [_P, _P, _P, _P, _I, _P, _P]),
    "nc_decode_step": (_I, [_P, _P, _P, _I, _P, _I, _P, _P]),
    "nc_decode_step_dev": (_I, [_P, _P, _P, _P, _P, _I, _P, _P]),
}


def lib() -> ctypes.CDLL:
    """Load libnc.so (built by `python -m decoder_transformer_step_nanochat_b300.build`)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m decoder_transformer_step_nanochat_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(st: int, ctx=None):
    if st != 0:
        msg = lib().nc_last_error(ctx)
        raise NcError(st, msg.decode() if msg else "")


# ------------------------------------------------------------------ C ABI mirror

def nc_create(depth, d_model, n_head, seq_len, vocab):
    h = _P()
    _check(lib().nc_create(depth, d_model, n_head, seq_len, vocab, ctypes.byref(h)))
    return h


def nc_configure(ctx, batch, precision, stream=0):
    _check(lib().nc_configure(ctx, batch, precision, stream or None), ctx)


def nc_param_count(ctx) -> int:
    return int(lib().nc_param_count(ctx))


def nc_param_offset(ctx, index):
    off, r, c = _SZ(), _I(), _I()
    _check(lib().nc_param_offset(ctx, index, ctypes.byref(off), ctypes.byref(r), ctypes.byref(c)), ctx)
    return int(off.value), int(r.value), int(c.value)


def nc_workspace_bytes(ctx) -> int:
    return int(lib().nc_workspace_bytes(ctx))


def nc_set_workspace(ctx, ptr, nbytes):
    _check(lib().nc_set_workspace(ctx, ptr, nbytes), ctx)


def nc_forward_loss(ctx, params, tokens, targets) -> float:
    out = _F()
    _check(lib().nc_forward_loss(ctx, params, tokens, targets, ctypes.byref(out)), ctx)
    return float(out.value)


def nc_forward_loss_async(ctx, params, tokens, targets, d_loss):
    _check(lib().nc_forward_loss_async(ctx, params, tokens, targets, d_loss), ctx)


def nc_backward(ctx, grads):
    _check(lib().nc_backward(ctx, grads), ctx)


def nc_backward_accumulate(ctx, grads, scale):
    _check(lib().nc_backward_accumulate(ctx, grads, scale), ctx)


def nc_forward_loss_u16(ctx, params, packed, d_loss):
    _check(lib().nc_forward_loss_u16(ctx, params, packed, d_loss), ctx)


def nc_train_step_host_u16(ctx, params, h_packed, grads) -> float:
    out = _F()
    _check(lib().nc_train_step_host_u16(ctx, params, h_packed, grads, ctypes.byref(out)), ctx)
    return float(out.value)


def nc_train_step_host(ctx, params, h_tokens, h_targets, grads) -> float:
    out = _F()
    _check(lib().nc_train_step_host(ctx, params, h_tokens, h_targets, grads, ctypes.byref(out)), ctx)
    return float(out.value)


def nc_get_token_outputs(ctx, d_lse=None, d_nll=None, d_argmax=None):
    _check(lib().nc_get_token_outputs(ctx, d_lse, d_nll, d_argmax), ctx)


def nc_get_argmax(ctx, d_argmax):
    _check(lib().nc_get_argmax(ctx, d_argmax), ctx)


def nc_get_hidden(ctx, d_hf):
    _check(lib().nc_get_hidden(ctx, d_hf), ctx)


def nc_sync(ctx):
    _check(lib().nc_sync(ctx), ctx)


def nc_launch_count(ctx) -> int:
    return int(lib().nc_launch_count(ctx))


def nc_profile_enable(ctx, enable):
    _check(lib().nc_profile_enable(ctx, 1 if enable else 0), ctx)


def nc_profile_read(ctx, family):
    """(device ms, launches, algorithmic work) summed over the recorded launches."""
    ms, n, w = ctypes.c_double(), _LL(), ctypes.c_double()
    _check(lib().nc_profile_read(ctx, family, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(w)), ctx)
    return float(ms.value), int(n.value), float(w.value)


def nc_profile_reset(ctx):
    _check(lib().nc_profile_reset(ctx), ctx)


def nc_set_pipeline_wait_limit(ns):
    _check(lib().nc_set_pipeline_wait_limit(ns))


def nc_last_error(ctx=None) -> str:
    m = lib().nc_last_error(ctx)
    return m.decode() if m else ""


def nc_destroy(ctx):
    lib().nc_destroy(ctx)


def nc_op_gemm(ctx, M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, epi, alpha, beta, C, ldc,
               C2=None, ldc2=0, row_f=None, row_i=None):
    _check(lib().nc_op_gemm(ctx, M, N, K, A, lda, a_kmajor, B, ldb, b_kmajor, epi, alpha, beta,
                            C, ldc, C2, ldc2, row_f, row_i), ctx)


def nc_op_lmhead_ce_fwd(ctx, hf, w_lm, tgt, lse, nll, argmax):
    _check(lib().nc_op_lmhead_ce_fwd(ctx, hf, w_lm, tgt, lse, nll, argmax), ctx)


def nc_op_lmhead_ce_bwd(ctx, hf, w_lm, tgt, lse, dhf, dw_lm):
    _check(lib().nc_op_lmhead_ce_bwd(ctx, hf, w_lm, tgt, lse, dhf, dw_lm), ctx)


def nc_op_attention_fwd(ctx, qkv, o, lse):
    _check(lib().nc_op_attention_fwd(ctx, qkv, o, lse), ctx)


def nc_op_attention_bwd(ctx, qkv, o, dout, lse, dqk, dqkv):
    _check(lib().nc_op_attention_bwd(ctx, qkv, o, dout, lse, dqk, dqkv), ctx)


def nc_op_qk_norm_rope_fwd(ctx, qkv, rqk):
    _check(lib().nc_op_qk_norm_rope_fwd(ctx, qkv, rqk), ctx)


def nc_op_rmsnorm_fwd(ctx, x, y, r):
    _check(lib().nc_op_rmsnorm_fwd(ctx, x, y, r), ctx)


def nc_op_rmsnorm_bwd(ctx, dy, y, r, dx, dx_e=None, accumulate=0):
    _check(lib().nc_op_rmsnorm_bwd(ctx, dy, y, r, dx, dx_e, 1 if accumulate else 0), ctx)


def nc_op_embed_fwd(ctx, tok, wte, x):
    _check(lib().nc_op_embed_fwd(ctx, tok, wte, x), ctx)


def nc_op_embed_bwd(ctx, tok, dx, dwte):
    _check(lib().nc_op_embed_bwd(ctx, tok, dx, dwte), ctx)


def nc_op_qk_norm_rope_bwd(ctx, dqk, qkv, rqk, dqkv):
    _check(lib().nc_op_qk_norm_rope_bwd(ctx, dqk, qkv, rqk, dqkv), ctx)


def nc_lmhead_ce_fwd_static(hf, w_lm, tgt, M, d, V, lse, nll, argmax, d_status=None, stream=None):
    """Allocation-free lm_head + cross-entropy forward (static device scratch)."""
    _check(lib().nc_lmhead_ce_fwd_static(hf, w_lm, tgt, M, d, V, lse, nll, argmax, d_status, stream))


def nc_op_gemm_batched(ctx, batch, M, N, K, A, lda, a_kmajor, a_brows, B, ldb, b_kmajor, b_brows, epi, alpha,
                       beta, C, ldc, C2=None, ldc2=0, c_brows=0):
    _check(lib().nc_op_gemm_batched(ctx, batch, M, N, K, A, lda, a_kmajor, a_brows, B, ldb, b_kmajor, b_brows,
                                    epi, alpha, beta, C, ldc, C2, ldc2, c_brows), ctx)


def nc_optim_state_bytes(ctx) -> int:
    return int(lib().nc_optim_state_bytes(ctx))


def nc_optim_init(ctx, params, state):
    _check(lib().nc_optim_init(ctx, params, state), ctx)


def nc_optim_set_hparams(ctx, beta1, beta2, eps, momentum, ns_steps):
    _check(lib().nc_optim_set_hparams(ctx, beta1, beta2, eps, momentum, ns_steps), ctx)


def nc_optim_step(ctx, params, grads, state, t, lr_adamw, lr_muon, weight_decay, max_grad_norm, stats=None):
    _check(lib().nc_optim_step(ctx, params, grads, state, t, lr_adamw, lr_muon, weight_decay, max_grad_norm,
                               stats), ctx)


def nc_lr_at(step, warmup, total, peak, final_frac=0.0) -> float:
    return float(lib().nc_lr_at(step, warmup, total, peak, final_frac))


def nc_kv_cache_bytes(ctx, max_len) -> int:
    return int(lib().nc_kv_cache_bytes(ctx, max_len))


def nc_prefill(ctx, params, tokens, kv_cache, max_len, next_tokens, last_logits=None):
    _check(lib().nc_prefill(ctx, params, tokens, kv_cache, max_len, next_tokens, last_logits), ctx)


def nc_decode_step(ctx, params, tokens, pos, kv_cache, max_len, next_tokens, logits=None):
    _check(lib().nc_decode_step(ctx, params, tokens, pos, kv_cache, max_len, next_tokens, logits), ctx)


def nc_decode_step_dev(ctx, params, tokens, d_pos, kv_cache, max_len, next_tokens, logits=None):
    _check(lib().nc_decode_step_dev(ctx, params, tokens, d_pos, kv_cache, max_len, next_tokens, logits), ctx)


# ------------------------------------------------------------------ convenience

class Step:
    """Owns one context plus a torch-allocated workspace on the current device.

    Memory plumbing only: the forward/backward run through the C ABI.
    """

    def __init__(self, depth, d_model, n_head, seq_len, vocab, batch, precision=NC_BF16, stream=None):
        import torch

        self.ctx = nc_create(depth, d_model, n_head, seq_len, vocab)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        nc_configure(self.ctx, batch, precision, self.stream.cuda_stream)
        nbytes = nc_workspace_bytes(self.ctx)
        # +1024 so the workspace can be aligned to 1024 bytes
        self._ws = torch.empty(nbytes + 1024, dtype=torch.uint8, device="cuda")
        base = self._ws.data_ptr()
        aligned = (base + 1023) // 1024 * 1024
        nc_set_workspace(self.ctx, aligned, nbytes)
        self.precision = precision
        self.batch, self.seq_len, self.vocab, self.d_model = batch, seq_len, vocab, d_model
        self.n_params = nc_param_count(self.ctx)

    def forward_loss(self, params, tokens, targets) -> float:
        return nc_forward_loss(self.ctx, params.data_ptr(), tokens.data_ptr(), targets.data_ptr())

    def forward_loss_async(self, params, tokens, targets, d_loss):
        nc_forward_loss_async(self.ctx, params.data_ptr(), tokens.data_ptr(), targets.data_ptr(),
                              d_loss.data_ptr())

    def backward(self, grads):
        nc_backward(self.ctx, grads.data_ptr())

    def backward_accumulate(self, grads, scale):
        nc_backward_accumulate(self.ctx, grads.data_ptr(), scale)

    def forward_loss_u16(self, params, packed, d_loss):
        nc_forward_loss_u16(self.ctx, params.data_ptr(), packed.data_ptr(), d_loss.data_ptr())

    def token_outputs(self):
        import torch

        M = self.batch * self.seq_len
        lse = torch.empty(M, dtype=torch.float32, device="cuda")
        nll = torch.empty(M, dtype=torch.float32, device="cuda")
        am = torch.empty(M, dtype=torch.int32, device="cuda")
        nc_get_token_outputs(self.ctx, lse.data_ptr(), nll.data_ptr(), am.data_ptr())
        return lse, nll, am

    def hidden(self):
        import torch

        dt = torch.bfloat16 if self.precision == NC_BF16 else torch.float32
        hf = torch.empty((self.batch * self.seq_len, self.d_model), dtype=dt, device="cuda")
        nc_get_hidden(self.ctx, hf.data_ptr())
        return hf

    def close(self):
        if self.ctx is not None:
            nc_destroy(self.ctx)
            self.ctx = None
        self._ws = None  # hand the workspace back to torch's allocator now

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
