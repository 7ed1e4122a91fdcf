"""CPU oracle of the optimizer step that completes a pretraining step: global
gradient clipping, AdamW on the embedding and unembedding, Muon on every 2-D
block matrix, and the learning-rate schedule.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module;
only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
It shares no code with the CUDA library.

Sources:

* nanochat explainer (cloudtoid llm-book), "The Full Pipeline" / "Pretraining":
  Muon for the matrix (2-D) weights plus AdamW for the embedding and
  unembedding, a cosine learning-rate schedule with warmup, gradient clipping
  at 1.0 and weight decay 0.1.
* "Karpathy Built a Full ChatGPT Clone in 8,000 Lines of Code" (topaiproduct),
  "What the Community Is Saying": Muon (Bernstein's optimizer, in Keller
  Jordan's implementation) for the matrix-multiplication parameters, AdamW for
  the embeddings and unembeddings.

The pages name the methods and nothing more. Readings taken (each is listed in
the design notes):

* Clipping: one L2 norm over every gradient of the model; every gradient is
  multiplied by min(1, max_norm / (norm + 1e-6)) before either optimizer sees it.
* AdamW is Adam with decoupled weight decay (Loshchilov & Hutter): first and
  second moments with bias correction, defaults beta1 0.9, beta2 0.999,
  eps 1e-8 (Kingma & Ba), and p <- p (1 - lr wd) - lr m_hat / (sqrt(v_hat) + eps).
* Muon as Keller Jordan published it: Nesterov momentum mu = 0.95
  (buf <- mu buf + g, u = g + mu buf); u is orthogonalised by five steps of the
  quintic Newton-Schulz iteration X <- a X + (b A + c A^2) X, A = X X^T,
  (a, b, c) = (3.4445, -4.7750, 2.0315), started from X = u / (||u||_F + 1e-7)
  in the wide orientation (the transpose when rows > cols); the step is
  -lr sqrt(max(1, rows / cols)) X, with the same decoupled weight decay as
  AdamW. Every block matrix (w_qkv, w_o, w_fc, w_proj of each layer) is one
  Muon matrix, as stored ([out, in]).
* Weight decay 0.1 applies to both parameter groups.
* The optimizer keeps fp32 master weights; the bf16 parameters the step reads
  are their round-to-nearest-even image.
* Schedule: linear warmup to the peak over `warmup` steps, then a half cosine
  from the peak down to final_frac * peak at step `total`.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

from .model import Shape, layout

CLIP_EPS = 1e-6
NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_EPS = 1e-7


@dataclasses.dataclass(frozen=True)
class Hyper:
    lr_adamw: float = 3e-3
    lr_muon: float = 2e-2
    weight_decay: float = 0.1
    max_grad_norm: float = 1.0
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    momentum: float = 0.95
    ns_steps: int = 5


def groups(s: Shape):
    """Split the flat layout into the two optimizer groups.

    Returns (adamw, muon): lists of (name, offset, rows, cols). AdamW takes the
    embedding (wte) and the unembedding (lm_head); Muon takes every 2-D block
    matrix.
    """
    adamw, muon = [], []
    for name, off, r, c in layout(s):
        (adamw if name in ("wte", "lm_head") else muon).append((name, off, r, c))
    return adamw, muon


def clip_scale(grads: np.ndarray, max_norm: float):
    """Global L2 norm of every gradient and the factor that clips it."""
    g = grads.astype(np.float64)
    norm = math.sqrt(float(np.dot(g, g)))
    return norm, min(1.0, max_norm / (norm + CLIP_EPS))


def adamw(p, g, m, v, t: int, lr: float, beta1: float, beta2: float, eps: float, wd: float):
    """One AdamW step (decoupled decay) at 1-based step t. Returns p, m, v."""
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    p = p * (1.0 - lr * wd) - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p, m, v


def newton_schulz(G: np.ndarray, steps: int = 5, coeffs=NS_COEFFS, eps: float = NS_EPS):
    """Quintic Newton-Schulz orthogonalisation of a 2-D matrix.

    Works on the wide orientation (rows <= cols), normalised to unit Frobenius
    norm; each step is X <- a X + (b A + c A A) X with A = X X^T.
    """
    a, b, c = coeffs
    X = np.asarray(G, dtype=np.float64)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    X = X / (np.linalg.norm(X) + eps)
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if tall else X


def muon(p, g, buf, lr: float, momentum: float, wd: float, ns_steps: int = 5):
    """One Muon step on one matrix p [rows, cols]. Returns p, buf."""
    buf = momentum * buf + g
    u = g + momentum * buf
    O = newton_schulz(u, ns_steps)
    rows, cols = p.shape
    scale = math.sqrt(max(1.0, rows / cols))
    p = p * (1.0 - lr * wd) - lr * scale * O
    return p, buf


def lr_at(step: int, warmup: int, total: int, peak: float, final_frac: float = 0.0):
    """Learning rate at 0-based step: linear warmup, then cosine decay."""
    if step < warmup:
        return peak * (step + 1) / warmup
    progress = min(1.0, max(0.0, (step - warmup) / max(1, total - warmup)))
    return peak * (final_frac + (1.0 - final_frac) * 0.5 * (1.0 + math.cos(math.pi * progress)))


def init_state(master: np.ndarray, s: Shape):
    """Zero moments for every parameter of both groups."""
    adamw_g, muon_g = groups(s)
    st = {"t": 0}
    for name, off, r, c in adamw_g:
        st["m:" + name] = np.zeros((r, c))
        st["v:" + name] = np.zeros((r, c))
    for name, off, r, c in muon_g:
        st["buf:" + name] = np.zeros((r, c))
    return st


def optimizer_step(master: np.ndarray, grads: np.ndarray, state: dict, s: Shape, h: Hyper):
    """One optimizer step on flat float64 master weights.

    Returns (new master, new state, grad norm, clip factor). The state's step
    counter t is 1-based after the call.
    """
    norm, k = clip_scale(grads, h.max_grad_norm)
    g_all = grads.astype(np.float64) * k
    out = np.array(master, dtype=np.float64, copy=True)
    st = {key: (val.copy() if isinstance(val, np.ndarray) else val) for key, val in state.items()}
    st["t"] = t = state["t"] + 1
    adamw_g, muon_g = groups(s)
    for name, off, r, c in adamw_g:
        n = r * c
        p, m, v = adamw(out[off:off + n].reshape(r, c), g_all[off:off + n].reshape(r, c), st["m:" + name],
                        st["v:" + name], t, h.lr_adamw, h.beta1, h.beta2, h.eps, h.weight_decay)
        out[off:off + n] = p.reshape(-1)
        st["m:" + name], st["v:" + name] = m, v
    for name, off, r, c in muon_g:
        n = r * c
        p, buf = muon(out[off:off + n].reshape(r, c), g_all[off:off + n].reshape(r, c), st["buf:" + name],
                      h.lr_muon, h.momentum, h.weight_decay, h.ns_steps)
        out[off:off + n] = p.reshape(-1)
        st["buf:" + name] = buf
    return out, st, norm, k
