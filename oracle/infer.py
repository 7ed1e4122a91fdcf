"""CPU oracle of generation with a KV cache: the prefill of a prompt and
one-token decode steps.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module;
only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
It shares no code with the CUDA library.

Source: nanochat explainer (cloudtoid llm-book), "Inference & KV Cache":
generation runs in two phases. Prefill processes the whole prompt at once,
every token attending to every earlier one, and fills the cache with the key
and value of every layer and position. Decode then produces one token at a
time: the new token's query attends to the cached keys and values, and its
own key and value are appended, so a step costs O(N) instead of
re-processing the prefix. The model is the one of oracle.model (keys are
cached after QK-norm and RoPE, i.e. as the attention uses them).

Readings: the next token is the argmax of the last position's logits
(greedy; the pages name no sampling rule); decode positions continue the
prompt's positions (the new token at position T0 + i); the cache holds
k_hat (normed and rotated) and v per layer, sequence, head and position.
"""

from __future__ import annotations

import numpy as np

from .model import HEAD_DIM, Shape, causal_attention, relu2, rmsnorm, rope, rope_angles, unpack


def _block_inputs(P, l):
    return P[f"h{l}.w_qkv"], P[f"h{l}.w_o"], P[f"h{l}.w_fc"], P[f"h{l}.w_proj"]


def prefill(params, tokens, s: Shape, dtype=np.float64):
    """Run the prompt tokens [B, T0] through the model.

    Returns (cache, logits) with logits [B, V] of the last position and cache
    = {"k": [L arrays [B, T0, H, D]], "v": [...], "pos": T0}.
    """
    P = unpack(params, s, dtype)
    tok = np.asarray(tokens)
    B, T0 = tok.shape
    d, H, D = s.d_model, s.n_head, HEAD_DIM
    cos, sin = rope_angles(T0, D)
    x = P["wte"][tok]
    ks, vs = [], []
    for l in range(s.depth):
        Wqkv, Wo, Wfc, Wproj = _block_inputs(P, l)
        xn, _ = rmsnorm(x)
        qkv = xn @ Wqkv.T
        q = rope(rmsnorm(qkv[..., :d].reshape(B, T0, H, D))[0], cos, sin)
        k = rope(rmsnorm(qkv[..., d:2 * d].reshape(B, T0, H, D))[0], cos, sin)
        v = qkv[..., 2 * d:].reshape(B, T0, H, D)
        o = np.empty_like(q)
        for b in range(B):
            o[b], _ = causal_attention(q[b], k[b], v[b])
        x = x + o.reshape(B, T0, d) @ Wo.T
        xn2, _ = rmsnorm(x)
        x = x + relu2(xn2 @ Wfc.T) @ Wproj.T
        ks.append(k)
        vs.append(v)
    hf, _ = rmsnorm(x[:, -1])
    return {"k": ks, "v": vs, "pos": T0}, hf @ P["lm_head"].T


def decode_step(params, cache, tokens, s: Shape, dtype=np.float64):
    """One decode step: tokens [B] at position cache["pos"] attend to the
    cached keys/values of positions < pos and to their own. Returns
    (new cache, logits [B, V]); the input cache is not modified."""
    P = unpack(params, s, dtype)
    tok = np.asarray(tokens)
    B = tok.shape[0]
    d, H, D = s.d_model, s.n_head, HEAD_DIM
    pos = cache["pos"]
    cos, sin = rope_angles(1, D, offset=pos)
    x = P["wte"][tok]                                        # [B, d]
    ks, vs = [], []
    for l in range(s.depth):
        Wqkv, Wo, Wfc, Wproj = _block_inputs(P, l)
        xn, _ = rmsnorm(x)
        qkv = xn @ Wqkv.T
        # rope works on [..., T, H, D]: here T = 1
        q = rope(rmsnorm(qkv[:, :d].reshape(B, 1, H, D))[0], cos, sin)[:, 0]
        k = rope(rmsnorm(qkv[:, d:2 * d].reshape(B, 1, H, D))[0], cos, sin)
        v = qkv[:, 2 * d:].reshape(B, 1, H, D)
        K = np.concatenate([cache["k"][l], k], axis=1)       # [B, pos+1, H, D]
        Vv = np.concatenate([cache["v"][l], v], axis=1)
        sc = np.einsum("bhd,bthd->bht", q, K) / np.sqrt(D)  # every cached position is visible
        p = np.exp(sc - sc.max(axis=-1, keepdims=True))
        p /= p.sum(axis=-1, keepdims=True)
        o = np.einsum("bht,bthd->bhd", p, Vv).reshape(B, d)
        x = x + o @ Wo.T
        xn2, _ = rmsnorm(x)
        x = x + relu2(xn2 @ Wfc.T) @ Wproj.T
        ks.append(K)
        vs.append(Vv)
    hf, _ = rmsnorm(x)
    return {"k": ks, "v": vs, "pos": pos + 1}, hf @ P["lm_head"].T


def generate(params, prompt, steps: int, s: Shape, dtype=np.float64):
    """Greedy generation: prefill, then `steps` decode steps, each feeding
    the previous argmax. Returns the generated ids [B, steps + 1] (the first
    comes from the prefill) and the logits of every produced position."""
    cache, logits = prefill(params, prompt, s, dtype)
    out, all_logits = [np.argmax(logits, axis=-1)], [logits]
    for _ in range(steps):
        cache, logits = decode_step(params, cache, out[-1], s, dtype)
        out.append(np.argmax(logits, axis=-1))
        all_logits.append(logits)
    return np.stack(out, axis=1), all_logits
