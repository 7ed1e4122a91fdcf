"""Seeded synthetic workloads for the nanochat pretraining step.

This module only draws data. It holds none of the model's arithmetic, so both
the CPU oracle and the CUDA library can consume the same arrays without
sharing any code that computes the method.

Workloads (shapes follow the depth dial of the nanochat explainer, "The 'One
Dial' Design" / "How dimensions are derived": d_model = 64 * depth,
n_head = d_model / 128, head_dim 128, FFN width 4 * d_model; vocabulary
65,536 from the same page's "Tokenizer Training" stage):

  tiny        depth 2,  d_model 128 (1 head), seq 64,   batch 4,  fp32
  small       depth 4,  d_model 256 (2 heads), seq 512,  batch 8,  bf16
  gpt2_small  depth 12, d_model 768 (6 heads), seq 2048, batch 8,  bf16
  d20         depth 20, d_model 1280 (10 heads), seq 2048, batch 16, bf16
  d26         depth 26, d_model 1664 (13 heads), seq 2048, batch 16, bf16

The tiny workload breaks the 64*depth rule on purpose (depth 2, width 128)
so that a single 128-wide head exists.

Parameter recipe: numpy Generator(PCG64(seed)) float32 standard normals,
drawn in the order of the flat parameter layout, scaled by 0.02 (the tiny workload scales
its lm_head block by 0.001 instead). bf16 workloads round every parameter to
bf16 (round to nearest even) and both sides read the rounded values.

Token recipe: ids follow a Zipf law with exponent 1.1 over ranks 1..V
(p_k proportional to k^-1.1, id = k - 1, so small ids are frequent), drawn by
inverse CDF from Generator(PCG64(seed + 1)). B*(T+1) ids are drawn and
reshaped to [B, T+1]; tokens are [:, :T] and targets the next token [:, 1:].
This stands in for the FineWeb-EDU token stream the pages pretrain on.
"""

from __future__ import annotations

import dataclasses

import numpy as np

VOCAB = 65536
HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    depth: int
    d_model: int
    n_head: int
    seq_len: int
    batch: int
    vocab: int = VOCAB
    dtype: str = "bf16"          # "bf16" or "fp32" storage of params/activations
    lm_head_std: float = 0.02
    std: float = 0.02

    @property
    def ffn(self) -> int:
        return 4 * self.d_model

    @property
    def tokens(self) -> int:
        return self.batch * self.seq_len

    def with_batch(self, batch: int) -> "Workload":
        return dataclasses.replace(self, batch=batch)

    def with_vocab(self, vocab: int) -> "Workload":
        return dataclasses.replace(self, vocab=vocab)

    def with_seq(self, seq_len: int) -> "Workload":
        return dataclasses.replace(self, seq_len=seq_len)


WORKLOADS = {
    "tiny": Workload("tiny", 2, 128, 1, 64, 4, dtype="fp32", lm_head_std=0.001),
    "small": Workload("small", 4, 256, 2, 512, 8),
    "gpt2_small": Workload("gpt2_small", 12, 768, 6, 2048, 8),
    "d20": Workload("d20", 20, 1280, 10, 2048, 16),
    "d26": Workload("d26", 26, 1664, 13, 2048, 16),
}


def segments(w: Workload):
    """(name, rows, cols) of every parameter block, in flat-buffer order.

    Order: wte[V,d]; per layer w_qkv[3d,d], w_o[d,d], w_fc[4d,d],
    w_proj[d,4d]; lm_head[V,d].
    """
    d, V, F = w.d_model, w.vocab, w.ffn
    out = [("wte", V, d)]
    for l in range(w.depth):
        out += [(f"h{l}.w_qkv", 3 * d, d), (f"h{l}.w_o", d, d),
                (f"h{l}.w_fc", F, d), (f"h{l}.w_proj", d, F)]
    out.append(("lm_head", V, d))
    return out


def n_params(w: Workload) -> int:
    return sum(r * c for _, r, c in segments(w))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest bf16 (ties to even), as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    xf, of = x.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for s in range(0, xf.size, step):
        u = xf[s:s + step].view(np.uint32)
        r = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
        of[s:s + step] = (r & np.uint32(0xFFFF0000)).view(np.float32)
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of float32 values that are already bf16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def make_params(w: Workload, seed: int = 0) -> np.ndarray:
    """Flat float32 parameter vector (bf16-rounded for bf16 workloads)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    total = n_params(w)
    out = np.empty(total, dtype=np.float32)
    off = 0
    for name, r, c in segments(w):
        n = r * c
        std = w.lm_head_std if name == "lm_head" else w.std
        blk = out[off:off + n]
        step = 1 << 24
        for s in range(0, n, step):
            e = min(n, s + step)
            rng.standard_normal(e - s, dtype=np.float32, out=blk[s:e])
            blk[s:e] *= np.float32(std)
        off += n
    if w.dtype == "bf16":
        out = round_bf16(out)
    return out


def make_grads(w: Workload, seed: int = 100, std: float = 1e-3) -> np.ndarray:
    """Flat float32 stand-in for a backward's output, for the optimizer step:
    N(0, std^2) draws from PCG64(seed) in layout order; the wte rows of the
    upper half of the vocabulary are zero, as rows of ids absent from a batch
    are in a real gradient."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty(n_params(w), dtype=np.float32)
    step = 1 << 24
    for s in range(0, out.size, step):
        e = min(out.size, s + step)
        rng.standard_normal(e - s, dtype=np.float32, out=out[s:e])
        out[s:e] *= np.float32(std)
    V, d = w.vocab, w.d_model
    out[(V // 2) * d:V * d] = 0.0
    return out


def make_sft_targets(targets: np.ndarray, seed: int = 200, mean_turn: int = 128) -> np.ndarray:
    """Targets of the supervised fine-tuning variant: every sequence is a run
    of alternating prompt and response turns, starting with a prompt, with
    turn lengths uniform in [mean_turn / 4, 7 mean_turn / 4); targets inside
    prompt turns become -1 (no loss there). Draws from PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.array(targets, dtype=np.int32, copy=True)
    B, T = out.shape
    lo, hi = max(1, mean_turn // 4), max(2, (7 * mean_turn) // 4)
    for b in range(B):
        t, prompt = 0, True
        while t < T:
            n = int(rng.integers(lo, hi))
            if prompt:
                out[b, t:t + n] = -1
            t += n
            prompt = not prompt
    return out


def make_decode_tokens(w: Workload, steps: int, seed: int = 300) -> np.ndarray:
    """Tokens fed to `steps` decode steps after a prompt, int32 [B, steps]:
    Zipf(1.1) ids like the prompts', from PCG64(seed)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    cdf = zipf_cdf(w.vocab)
    ids = np.searchsorted(cdf, rng.random(w.batch * steps), side="right")
    return np.minimum(ids, w.vocab - 1).astype(np.int32).reshape(w.batch, steps)


def zipf_cdf(vocab: int, s: float = 1.1) -> np.ndarray:
    k = np.arange(1, vocab + 1, dtype=np.float64)
    p = k ** (-s)
    c = np.cumsum(p)
    return c / c[-1]


def _token_rows(w: Workload, seed: int):
    """[B, T+1] Zipf(1.1) ids (int64), one row of T+1 ids per sequence."""
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    cdf = zipf_cdf(w.vocab)
    u = rng.random(w.batch * (w.seq_len + 1))
    ids = np.searchsorted(cdf, u, side="right")
    ids = np.minimum(ids, w.vocab - 1)
    return ids.reshape(w.batch, w.seq_len + 1)


def make_tokens(w: Workload, seed: int = 0):
    """(tokens, targets) int32 [B, T]: Zipf(1.1) ids, targets = next token."""
    ids = _token_rows(w, seed).astype(np.int32)
    return np.ascontiguousarray(ids[:, :-1]), np.ascontiguousarray(ids[:, 1:])


def make_packed_tokens(w: Workload, seed: int = 0):
    """The same draw as make_tokens(w, seed), as packed uint16 rows [B, T+1]
    (the token-shard format: ids of a vocabulary of at most 65,536 entries)."""
    if w.vocab > 65536:
        raise ValueError("uint16 rows need vocab <= 65536")
    return np.ascontiguousarray(_token_rows(w, seed).astype(np.uint16))


def model_flops_per_token(w: Workload) -> float:
    """Algorithmic training FLOPs per token (forward + backward).

    6 * (12 L d^2 + d V) for the linear layers (QKV, out-proj, MLP up/down and
    lm_head) plus 6 L d T for causal attention (QK^T and PV over the lower
    triangle, about T/2 keys per query, times 3 for forward + backward). The
    embedding gather counts zero.
    """
    L, d, V, T = w.depth, w.d_model, w.vocab, w.seq_len
    return 6.0 * (12 * L * d * d + d * V) + 6.0 * L * d * T
