"""CPU oracle of the nanochat pretraining step: forward, mean next-token
cross-entropy, and the analytic backward of every parameter.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module;
only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
It shares no code with the CUDA library.

Everything here is the plain textbook definition in NumPy, in float64 or
float32, with no fusion and no streaming beyond chunking token rows to bound
memory. Sources (the nanochat explainer page, cloudtoid llm-book):

* "Architecture Choices": a decoder-only GPT of the modern family with RoPE,
  RMSNorm, ReLU-squared, QK-norm and untied embeddings.
* "RoPE Intuition": q and k are rotated by angles proportional to position,
  so that q.k depends only on the relative distance.
* "ReLU^2 Sparsity": relu(x)^2 zeroes negatives and squares positives.
* "How dimensions are derived": d_model = 64 depth, heads of width 128, FFN
  width 4 d_model.
* "The Full Pipeline" / "Pretraining": next-token prediction, cross-entropy
  between the logits and the actual next tokens.
* "Multi-Head Attention (what nanochat uses)": full MHA, one K/V per head.

Readings where the pages are silent (each is listed in the design notes):
pre-norm blocks and a final norm before lm_head; no norm after the embedding;
parameter-free RMSNorm with eps 1e-6 inside the square root (also for
QK-norm); RoPE in the half-split pairing (dim j pairs with j + 64), angle
pos * 10000^(-j/64), positions from 0 in every sequence, angles formed in
float64; attention scale 1/sqrt(128); no biases, dropout or logit capping;
loss = mean over all B*T positions in nats; argmax = lowest index among ties.

Token input ("Streaming Tokenization": the shards hold packed 16-bit token
ids that the loader reads as they are; "Pretraining": the target of each
position is the next token): a row of T+1 ids gives the inputs ids[0..T-1]
and the targets ids[1..T] (split_packed).

Several batches, one update ("Distributed Training": every GPU runs the step
on its own shard and the gradients are averaged by an all-reduce after the
backward): step_accumulated averages the losses and gradients of n
micro-batches, which is what n accumulating backward passes with scale 1/n
produce on one GPU.

The supervised fine-tuning variant ("Supervised Fine-Tuning (SFT)": the same
cross-entropy, but only on the assistant's response tokens; the prompt tokens
are masked from the loss) is expressed by the target id IGNORE (-1): such a
position contributes no loss and no gradient, and the loss is the mean over
the remaining positions (0 when there are none).
"""

from __future__ import annotations

import dataclasses

import numpy as np

EPS = 1e-6
ROPE_BASE = 10000.0
HEAD_DIM = 128
IGNORE = -1


@dataclasses.dataclass(frozen=True)
class Shape:
    depth: int
    d_model: int
    n_head: int
    vocab: int

    @property
    def ffn(self) -> int:
        return 4 * self.d_model


def layout(s: Shape):
    """Flat parameter layout: list of (name, offset, rows, cols).

    wte[V,d]; per layer w_qkv[3d,d] (q rows, then k, then v; row h*128+j is
    dim j of head h), w_o[d,d], w_fc[4d,d], w_proj[d,4d]; lm_head[V,d].
    Every matrix is [out, in], so a linear layer is y = x W^T.
    """
    d, V, F = s.d_model, s.vocab, s.ffn
    blocks = [("wte", V, d)]
    for l in range(s.depth):
        blocks += [(f"h{l}.w_qkv", 3 * d, d), (f"h{l}.w_o", d, d),
                   (f"h{l}.w_fc", F, d), (f"h{l}.w_proj", d, F)]
    blocks.append(("lm_head", V, d))
    out, off = [], 0
    for name, r, c in blocks:
        out.append((name, off, r, c))
        off += r * c
    return out


def param_count(s: Shape) -> int:
    name, off, r, c = layout(s)[-1]
    return off + r * c


def unpack(params: np.ndarray, s: Shape, dtype=np.float64):
    p = np.asarray(params)
    out = {}
    for name, off, r, c in layout(s):
        out[name] = p[off:off + r * c].reshape(r, c).astype(dtype, copy=False)
    return out


# ---------------------------------------------------------------- pieces

def rmsnorm(z: np.ndarray, eps: float = EPS):
    """Parameter-free RMSNorm over the last axis: y = z / sqrt(mean z^2 + eps).

    Returns (y, r) with r = 1/sqrt(mean z^2 + eps) (the "RMSNorm" entry of
    "Architecture Choices"; no gain, eps inside the root).
    """
    ms = np.mean(z * z, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(ms + eps)
    return z * r, r


def rmsnorm_backward(dy: np.ndarray, y: np.ndarray, r: np.ndarray):
    """Gradient through y = z * r(z): dz = r * (dy - y * mean(dy * y))."""
    return r * (dy - y * np.mean(dy * y, axis=-1, keepdims=True))


def rope_angles(T: int, D: int = HEAD_DIM, base: float = ROPE_BASE, offset: int = 0):
    """cos, sin of pos * base^(-j/(D/2)) for pos in offset..offset+T-1,
    j in 0..D/2-1, formed in float64 ("RoPE Intuition": angles proportional
    to position)."""
    half = D // 2
    j = np.arange(half, dtype=np.float64)
    theta = base ** (-j / half)
    pos = np.arange(offset, offset + T, dtype=np.float64)
    ang = pos[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)


def rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray):
    """Rotate pairs (j, j + D/2) of the last axis by the angle of each
    position. x is [..., T, H, D]; cos/sin are [T, D/2]."""
    half = x.shape[-1] // 2
    c = cos[:, None, :].astype(x.dtype)
    s = sin[:, None, :].astype(x.dtype)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def rope_backward(g: np.ndarray, cos: np.ndarray, sin: np.ndarray):
    """Transpose of the rotation: rotate by the negative angle."""
    half = g.shape[-1] // 2
    c = cos[:, None, :].astype(g.dtype)
    s = sin[:, None, :].astype(g.dtype)
    g1, g2 = g[..., :half], g[..., half:]
    return np.concatenate([g1 * c + g2 * s, -g1 * s + g2 * c], axis=-1)


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """Causal softmax attention for one sequence, all heads.

    q, k, v: [T, H, D]. s = q k^T / sqrt(D), keys after the query masked,
    p = softmax over keys, o = p v. Returns o [T, H, D] and lse [H, T].
    """
    T, H, D = q.shape
    scale = 1.0 / np.sqrt(D)
    qh = q.transpose(1, 0, 2)
    kh = k.transpose(1, 0, 2)
    vh = v.transpose(1, 0, 2)
    s = np.matmul(qh, kh.transpose(0, 2, 1)) * q.dtype.type(scale)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(mask[None], -np.inf, s)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=-1, keepdims=True)
    p = e / z
    o = np.matmul(p, vh)
    lse = (m + np.log(z))[..., 0]
    return o.transpose(1, 0, 2), lse


def causal_attention_backward(q, k, v, do):
    """Analytic backward of causal_attention for one sequence.

    dv = p^T do; dp = do v^T; ds = p * (dp - rowsum(dp * p));
    dq = ds k / sqrt(D); dk = ds^T q / sqrt(D). p is recomputed from q, k.
    """
    T, H, D = q.shape
    scale = q.dtype.type(1.0 / np.sqrt(D))
    qh, kh, vh = (a.transpose(1, 0, 2) for a in (q, k, v))
    doh = do.transpose(1, 0, 2)
    s = np.matmul(qh, kh.transpose(0, 2, 1)) * scale
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(mask[None], -np.inf, s)
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    p = e / np.sum(e, axis=-1, keepdims=True)
    dv = np.matmul(p.transpose(0, 2, 1), doh)
    dp = np.matmul(doh, vh.transpose(0, 2, 1))
    ds = p * (dp - np.sum(dp * p, axis=-1, keepdims=True))
    dq = np.matmul(ds, kh) * scale
    dk = np.matmul(ds.transpose(0, 2, 1), qh) * scale
    return (dq.transpose(1, 0, 2), dk.transpose(1, 0, 2), dv.transpose(1, 0, 2))


def relu2(u):
    """ReLU-squared ("ReLU^2 Sparsity"): max(u, 0)^2, exact zero for u <= 0."""
    return np.square(np.maximum(u, 0))


def relu2_backward(da, u):
    """d/du max(u,0)^2 = 2 max(u,0); zero at u = 0."""
    return da * (2 * np.maximum(u, 0))


def cross_entropy_rows(hf, w_lm, tgt, chunk: int = 2048):
    """Per-position logsumexp, loss and argmax of logits = hf W_lm^T.

    ("Pretraining": cross-entropy between the predicted logits and the actual
    next tokens.) Rows are processed in chunks only to bound memory.
    Returns lse [M], nll [M], argmax [M] (lowest index on ties). A target of
    IGNORE gives nll 0 at that row (lse and argmax are still those of the row).
    """
    M = hf.shape[0]
    lse = np.empty(M, dtype=hf.dtype)
    nll = np.empty(M, dtype=hf.dtype)
    amax = np.empty(M, dtype=np.int64)
    for s in range(0, M, chunk):
        e = min(M, s + chunk)
        logits = hf[s:e] @ w_lm.T
        m = np.max(logits, axis=-1, keepdims=True)
        z = np.log(np.sum(np.exp(logits - m), axis=-1, keepdims=True)) + m
        lse[s:e] = z[:, 0]
        t = tgt[s:e]
        keep = t != IGNORE
        picked = logits[np.arange(e - s), np.where(keep, t, 0)]
        nll[s:e] = np.where(keep, z[:, 0] - picked, 0.0)
        amax[s:e] = np.argmax(logits, axis=-1)
    return lse, nll, amax


def cross_entropy_backward(hf, w_lm, tgt, lse, chunk: int = 2048):
    """g = (softmax(logits) - onehot(tgt)) / n on the n rows whose target is
    not IGNORE, 0 on the others; dW_lm = g^T hf; dhf = g W_lm."""
    M = hf.shape[0]
    n = int(np.count_nonzero(np.asarray(tgt) != IGNORE))
    dhf = np.empty_like(hf)
    dw = np.zeros_like(w_lm)
    for s in range(0, M, chunk):
        e = min(M, s + chunk)
        logits = hf[s:e] @ w_lm.T
        t = tgt[s:e]
        keep = t != IGNORE
        g = np.exp(logits - lse[s:e, None])
        g[np.arange(e - s)[keep], t[keep]] -= 1
        g[~keep] = 0
        if n:
            g /= n
        dhf[s:e] = g @ w_lm
        dw += g.T @ hf[s:e]
    return dhf, dw


# ---------------------------------------------------------------- step

def forward(params, tokens, targets, s: Shape, dtype=np.float64, keep=True):
    """Forward pass and mean next-token loss.

    tokens, targets: int [B, T]. Returns (loss, cache); cache holds what the
    backward needs (or None when keep is False) plus per-position lse, nll,
    argmax.
    """
    P = unpack(params, s, dtype)
    tok = np.asarray(tokens)
    tgt = np.asarray(targets)
    B, T = tok.shape
    d, H, D = s.d_model, s.n_head, HEAD_DIM
    cos, sin = rope_angles(T, D)
    x = P["wte"][tok]                       # [B, T, d]; no scaling or norm
    layers = []
    for l in range(s.depth):
        Wqkv, Wo = P[f"h{l}.w_qkv"], P[f"h{l}.w_o"]
        Wfc, Wproj = P[f"h{l}.w_fc"], P[f"h{l}.w_proj"]
        xn1, r1 = rmsnorm(x)
        qkv = xn1 @ Wqkv.T                  # [B, T, 3d]
        q = qkv[..., :d].reshape(B, T, H, D)
        k = qkv[..., d:2 * d].reshape(B, T, H, D)
        v = qkv[..., 2 * d:].reshape(B, T, H, D)
        qn, rq = rmsnorm(q)                 # QK-norm per head
        kn, rk = rmsnorm(k)
        qr = rope(qn, cos, sin)
        kr = rope(kn, cos, sin)
        o = np.empty_like(q)
        for b in range(B):
            o[b], _ = causal_attention(qr[b], kr[b], v[b])
        o = o.reshape(B, T, d)
        x = x + o @ Wo.T
        xn2, r2 = rmsnorm(x)
        u = xn2 @ Wfc.T
        a = relu2(u)
        x = x + a @ Wproj.T
        if keep:
            layers.append(dict(xn1=xn1, r1=r1, qn=qn, rq=rq, kn=kn, rk=rk,
                               qr=qr, kr=kr, v=v, o=o, xn2=xn2, r2=r2, u=u, a=a))
    hf, rf = rmsnorm(x)
    M = B * T
    lse, nll, amax = cross_entropy_rows(hf.reshape(M, d), P["lm_head"], tgt.reshape(M))
    valid = tgt.reshape(M) != IGNORE
    loss = float(np.sum(nll[valid]) / np.count_nonzero(valid)) if valid.any() else 0.0
    cache = dict(P=P, tok=tok, tgt=tgt, layers=layers, hf=hf, rf=rf, lse=lse,
                 nll=nll, argmax=amax, cos=cos, sin=sin, shape=s, dtype=dtype)
    return loss, cache


def backward(cache):
    """Analytic gradient of the mean loss w.r.t. every parameter, returned as
    one flat vector in the layout of `layout` (dtype of the forward)."""
    P, s = cache["P"], cache["shape"]
    tok, tgt = cache["tok"], cache["tgt"]
    B, T = tok.shape
    d, H, D = s.d_model, s.n_head, HEAD_DIM
    M = B * T
    cos, sin = cache["cos"], cache["sin"]
    grads = {}
    hf = cache["hf"].reshape(M, d)
    dhf, grads["lm_head"] = cross_entropy_backward(hf, P["lm_head"], tgt.reshape(M), cache["lse"])
    dx = rmsnorm_backward(dhf.reshape(B, T, d), cache["hf"], cache["rf"])
    for l in reversed(range(s.depth)):
        c = cache["layers"][l]
        Wqkv, Wo = P[f"h{l}.w_qkv"], P[f"h{l}.w_o"]
        Wfc, Wproj = P[f"h{l}.w_fc"], P[f"h{l}.w_proj"]
        # MLP: x = x + relu2(rmsnorm(x) Wfc^T) Wproj^T
        grads[f"h{l}.w_proj"] = dx.reshape(M, d).T @ c["a"].reshape(M, -1)
        da = dx @ Wproj
        du = relu2_backward(da, c["u"])
        grads[f"h{l}.w_fc"] = du.reshape(M, -1).T @ c["xn2"].reshape(M, d)
        dxn2 = du @ Wfc
        dx = dx + rmsnorm_backward(dxn2, c["xn2"], c["r2"])
        # attention: x = x + attn(rmsnorm(x)) Wo^T
        grads[f"h{l}.w_o"] = dx.reshape(M, d).T @ c["o"].reshape(M, d)
        do = (dx @ Wo).reshape(B, T, H, D)
        dqr = np.empty_like(do)
        dkr = np.empty_like(do)
        dv = np.empty_like(do)
        for b in range(B):
            dqr[b], dkr[b], dv[b] = causal_attention_backward(c["qr"][b], c["kr"][b], c["v"][b], do[b])
        dqn = rope_backward(dqr, cos, sin)
        dkn = rope_backward(dkr, cos, sin)
        dq = rmsnorm_backward(dqn, c["qn"], c["rq"])
        dk = rmsnorm_backward(dkn, c["kn"], c["rk"])
        dqkv = np.concatenate([dq.reshape(B, T, d), dk.reshape(B, T, d), dv.reshape(B, T, d)], axis=-1)
        grads[f"h{l}.w_qkv"] = dqkv.reshape(M, 3 * d).T @ c["xn1"].reshape(M, d)
        dxn1 = dqkv @ Wqkv
        dx = dx + rmsnorm_backward(dxn1, c["xn1"], c["r1"])
    # embedding: row id receives the sum of dx over the positions holding id
    dwte = np.zeros_like(P["wte"])
    np.add.at(dwte, tok.reshape(M), dx.reshape(M, d))
    grads["wte"] = dwte
    out = np.empty(param_count(s), dtype=cache["dtype"])
    for name, off, r, cc in layout(s):
        out[off:off + r * cc] = grads[name].reshape(-1)
    return out


def step(params, tokens, targets, s: Shape, dtype=np.float64):
    """Convenience: (loss, flat grads, cache)."""
    loss, cache = forward(params, tokens, targets, s, dtype)
    return loss, backward(cache), cache


def split_packed(packed):
    """Packed token rows [B, T+1] -> (inputs [B, T], next-token targets
    [B, T]) as int32: position t of row b reads id t and predicts id t+1."""
    ids = np.asarray(packed).astype(np.int64)
    return ids[:, :-1].astype(np.int32), ids[:, 1:].astype(np.int32)


def step_accumulated(params, micro_batches, s: Shape, dtype=np.float64):
    """Mean loss and mean gradient over micro-batches [(tokens, targets), ...],
    each micro-batch's loss being its own mean over its positions: the
    gradient that shard-wise averaging (or accumulation with scale 1/n) forms."""
    n = len(micro_batches)
    loss_sum, grad_sum = 0.0, None
    for tok, tgt in micro_batches:
        loss, g, _ = step(params, tok, tgt, s, dtype)
        loss_sum += loss
        grad_sum = g.astype(np.float64) if grad_sum is None else grad_sum + g
    return loss_sum / n, grad_sum / n
