"""Seeded synthetic inputs for the TTT-E2E inner loop.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Both the float64 oracle and the CUDA path (its tests and
the benchmark) take their inputs from here, so the two sides start from
bit-identical token ids and fp32 weights.

Token stream (stands in for the Books / DCLM text the TTT-E2E pages train and
evaluate on, which is not available here): ranks drawn from a Zipf(1.1) law
truncated to the vocabulary by inverse CDF on the explicit pmf, mapped to ids
through a seeded permutation, then 32-token spans copied to random later
offsets (T // 128 copies) so that the stream contains exact repeats the fast
weights can learn.

Weights: every matrix N(0, 0.02), drawn as float32 standard normals from
``default_rng(seed)`` in blob order and scaled in float32; RMSNorm gains are 1
and are not drawn.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

__all__ = ["Shape", "SHAPES", "blob_layout", "blob_size", "zipf_tokens",
           "weight_blob", "sequence_tokens"]


@dataclass(frozen=True)
class Shape:
    """Model shape and run hyper-parameters of one workload."""
    n_layers: int
    d_model: int
    n_heads: int
    d_ff: int
    vocab: int
    window: int
    chunk: int
    rope_theta: float
    eta: float
    seq_len: int
    n_seqs: int = 1
    compute: str = "bf16"          # "fp32" or "bf16"
    rms_eps: float = 1e-6
    dual_mlp: bool = False         # trainable blocks carry a frozen static MLP beside the fast one

    @property
    def n_trainable(self) -> int:
        return self.n_layers // 4

    @property
    def d_head(self) -> int:
        return self.d_model // self.n_heads

    def replace(self, **kw) -> "Shape":
        d = dict(self.__dict__)
        d.update(kw)
        return Shape(**d)


# The five workloads: tiny fp32, 125M/760M/3B shapes in bf16 with fp32 fast
# weights, and the 760M-shape window/chunk sweep (4 sequences of 65536).
SHAPES = {
    "tiny": Shape(4, 128, 4, 512, 512, 128, 64, 1e4, 1e-2, 512, compute="fp32"),
    "125m": Shape(12, 768, 12, 3072, 32000, 8192, 1024, 1e6, 1e-3, 32768),
    "760m": Shape(24, 1536, 16, 6144, 32000, 8192, 1024, 1e7, 1e-3, 131072),
    "3b": Shape(28, 3072, 24, 12288, 32000, 8192, 1024, 1e7, 5e-4, 131072),
}
for _k in (2048, 8192, 32768):
    for _b in (256, 1024, 2048):
        if _k >= _b:
            SHAPES[f"sweep_k{_k}_b{_b}"] = SHAPES["760m"].replace(
                window=_k, chunk=_b, seq_len=65536, n_seqs=4)


def blob_layout(shape: Shape):
    """(name, shape, is_gain) for every tensor of the fp32 weight blob, in order.

    Order: E[V][d]; per layer g_attn[d], Wq, Wk, Wv, Wo [d][d], g_mlp[d],
    W_up[d][f], W_down[f][d] (with dual_mlp, the trainable layers then add the
    static pair W_up_s[d][f], W_down_s[f][d]); g_final[d]; W_lm[d][V].
    Row-major, y = x.W.
    """
    d, f, V = shape.d_model, shape.d_ff, shape.vocab
    out = [("E", (V, d), False)]
    for l in range(shape.n_layers):
        out += [(f"g_attn.{l}", (d,), True),
                (f"Wq.{l}", (d, d), False), (f"Wk.{l}", (d, d), False),
                (f"Wv.{l}", (d, d), False), (f"Wo.{l}", (d, d), False),
                (f"g_mlp.{l}", (d,), True),
                (f"W_up.{l}", (d, f), False), (f"W_down.{l}", (f, d), False)]
        if shape.dual_mlp and l >= shape.n_layers - shape.n_trainable:
            out += [(f"W_up_s.{l}", (d, f), False), (f"W_down_s.{l}", (f, d), False)]
    out += [("g_final", (d,), True), ("W_lm", (d, V), False)]
    return out


def blob_size(shape: Shape) -> int:
    return sum(int(np.prod(s)) for _, s, _ in blob_layout(shape))


def weight_blob(shape: Shape, seed: int = 0, std: float = 0.02) -> np.ndarray:
    """fp32 weight blob: N(0, std) matrices, unit gains."""
    rng = np.random.default_rng(seed)
    blob = np.empty(blob_size(shape), dtype=np.float32)
    off = 0
    for _, s, is_gain in blob_layout(shape):
        n = int(np.prod(s))
        if is_gain:
            blob[off:off + n] = 1.0
        else:
            seg = blob[off:off + n]
            rng.standard_normal(n, dtype=np.float32, out=seg)
            seg *= np.float32(std)
        off += n
    return blob


def zipf_tokens(T: int, vocab: int, seed: int, s: float = 1.1,
                span: int = 32, copies: int | None = None) -> np.ndarray:
    """int32[T] Zipf(s) token ids with ``copies`` (default T//128) repeated spans."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(vocab)
    pmf = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(pmf)
    cdf /= cdf[-1]
    u = rng.random(T)
    r = np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1)
    tok = perm[r].astype(np.int32)
    if copies is None:
        copies = T // 128
    if T >= 2 * span:
        for _ in range(copies):
            src = int(rng.integers(0, T - 2 * span + 1))
            dst = int(rng.integers(src + span, T - span + 1))
            tok[dst:dst + span] = tok[src:src + span].copy()
    return tok


def sequence_tokens(shape: Shape, seq: int = 0, T: int | None = None) -> np.ndarray:
    """Tokens of sequence ``seq`` (seed 1000 + seq), full length unless T given."""
    full = zipf_tokens(shape.seq_len, shape.vocab, 1000 + seq)
    return full if T is None else full[:T].copy()


def n_chunks(T: int, b: int) -> int:
    return int(math.ceil(T / b))
