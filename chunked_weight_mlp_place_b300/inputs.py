"""Seeded synthetic inputs for the In-Place TTT fast-weight layer.

This module only draws random arrays; it performs none of the layer's
arithmetic (no gate, conv, projection or fast-weight update).  Both the float64
CPU oracle (through the tests) and the CUDA library (through the tests and the
benchmark) are fed from here, so the two sides see bit-identical inputs.

Shapes and distributions follow the workloads of the In-Place TTT write-ups: a
gated MLP ``(SiLU(x W_g) * (x W_u)) W_o`` at the 500M / 1.5B / 4B model scales
(experiments section: from-scratch 500M and 1.5B models, plug-in Qwen3-4B), long
contexts up to 128k tokens and chunk sizes 64..4096 (chunk-size ablation,
Fig. 3b).  The pages publish no dataset the kernels could consume, so Gaussian
stand-ins are used:

* X  ~ N(0, 1) per element, then RMS-normalised per token (eps 1e-6, no gain);
* token ids uniform over the vocabulary; embedding table ~ N(0, 1/d);
  E = table[ids] (the embedding lookup is input preparation);
* W_g, W_u ~ N(0, 1/d); W_o0 ~ N(0, 1/d_ff); conv weights ~ N(0, 1/2);
  P ~ N(0, 1/d).  The second argument of N is the variance.

Every tensor has its own counter-independent PCG64 stream spawned from one
``SeedSequence``, so any tensor (or the first rows of X / ids) can be drawn
without drawing the others.  Values are produced in float32 and, for the bf16
workloads, rounded to bfloat16 (round to nearest even) *before* they are handed
to either side, so parity measures compute error, not input rounding.  The
fast weight W_o0 and the conv weights stay float32 in every workload.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence

import numpy as np

__all__ = ["Workload", "WORKLOADS", "generate", "round_to_bf16", "workload", "doc_boundaries", "DOC_MIXES"]

# Stream indices inside the spawned SeedSequence; fixed so that adding a tensor
# never changes the values of the others (new streams go at the end).
_STREAMS = ("ids", "table", "X", "W_g", "W_u", "W_o0", "conv_w", "P", "doc_len")


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload of the fast-weight layer.

    ``B`` is the chunk size (tokens per fast-weight update); ``L`` the sequence
    length; ``batch`` the number of independent sequences.
    """

    name: str
    batch: int
    L: int
    B: int
    d: int
    d_ff: int
    vocab: int
    dtype: str  # "fp32" or "bf16" (activations); the fast weight is always fp32
    eta: float
    rules: Sequence[str]

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def K(self) -> int:
        return self.L // self.B


# The five workloads: a tiny fp32 check, then 500M-, 1.5B- and 4B-scale layers
# and the chunk-size / rule sweep at the 4B shape.
WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 256, 64, 64, 256, 512, "fp32", 0.1, ("mse", "add")),
    "500m": Workload("500m", 8, 4096, 512, 1024, 4096, 512, "bf16", 0.05, ("mse",)),
    "1p5b": Workload("1p5b", 1, 32768, 1024, 2048, 8192, 512, "bf16", 0.02, ("mse",)),
    "4b": Workload("4b", 1, 131072, 1024, 2560, 9728, 151936, "bf16", 0.01, ("mse",)),
    # chunk sizes swept: 64, 256, 512, 1024, 4096 (B below is the default point)
    "4b_sweep": Workload("4b_sweep", 1, 32768, 1024, 2560, 9728, 512, "bf16", 0.01, ("mse", "add")),
}
SWEEP_CHUNKS = (64, 256, 512, 1024, 4096)


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return w.replace(**overrides) if overrides else w


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32.

    Inputs are finite and far from the float32 range limits.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def _streams(seed: int) -> Dict[str, np.random.Generator]:
    children = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    return {name: np.random.Generator(np.random.PCG64(c)) for name, c in zip(_STREAMS, children)}


def _normal(rng: np.random.Generator, shape, var: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(np.sqrt(var))
    return a


def generate(w: Workload, seed: int = 0, n_tokens: Optional[int] = None,
             want: Sequence[str] = ("X", "E", "W_g", "W_u", "W_o0", "conv_w", "P")) -> Dict[str, np.ndarray]:
    """Draw the inputs of workload ``w``.

    Returns float32 arrays (values exactly representable in ``w.dtype``):
    ``X`` and ``E`` of shape (batch*L, d) (token-major, sequence s occupies rows
    s*L .. s*L+L-1); ``W_g``, ``W_u`` (d, d_ff); ``W_o0`` (d_ff, d); ``conv_w``
    (d, 4); ``P`` (d, d); also ``ids`` (batch*L,) when E is requested.

    ``n_tokens`` limits X / ids / E to the first ``n_tokens`` rows of the
    flattened token axis (the same values a full draw would give there).
    """
    T = w.batch * w.L if n_tokens is None else int(n_tokens)
    if not 0 <= T <= w.batch * w.L:
        raise ValueError("n_tokens out of range")
    rng = _streams(seed)
    q = round_to_bf16 if w.dtype == "bf16" else (lambda a: np.ascontiguousarray(a, np.float32))
    out: Dict[str, np.ndarray] = {}
    if "X" in want:
        X = rng["X"].standard_normal(size=(T, w.d), dtype=np.float32)
        ms = np.mean(np.square(X, dtype=np.float64), axis=1, keepdims=True)
        X = (X / np.sqrt(ms + 1e-6)).astype(np.float32)
        out["X"] = q(X)
    if "E" in want or "ids" in want:
        ids = rng["ids"].integers(0, w.vocab, size=w.batch * w.L, dtype=np.int64)[:T]
        out["ids"] = ids
        if "E" in want:
            table = q(_normal(rng["table"], (w.vocab, w.d), 1.0 / w.d))
            out["E"] = np.ascontiguousarray(table[ids])
    if "W_g" in want:
        out["W_g"] = q(_normal(rng["W_g"], (w.d, w.d_ff), 1.0 / w.d))
    if "W_u" in want:
        out["W_u"] = q(_normal(rng["W_u"], (w.d, w.d_ff), 1.0 / w.d))
    if "W_o0" in want:
        out["W_o0"] = _normal(rng["W_o0"], (w.d_ff, w.d), 1.0 / w.d_ff)
    if "conv_w" in want:
        out["conv_w"] = _normal(rng["conv_w"], (w.d, 4), 0.5)
    if "P" in want:
        out["P"] = q(_normal(rng["P"], (w.d, w.d), 1.0 / w.d))
    return out


# Packed-document length mixes (min, max tokens), log-uniform between them: a
# long-tailed spread of document lengths, so that most documents end inside a
# chunk and a few span many chunks.  "long128k" packs 128k tokens of documents
# from 256 tokens to 32k (the long-context range of the write-ups' experiments).
DOC_MIXES: Dict[str, tuple] = {
    "long128k": (256, 32768),
    "short": (1, 600),
}


def doc_boundaries(n_tokens: int, seed: int = 0, mix: str = "long128k") -> np.ndarray:
    """Boundaries cu_seqlens (int64, 0 .. n_tokens, strictly rising) of documents
    packed back to back: lengths drawn log-uniformly in the mix's range until
    n_tokens is filled, the last one cut to fit."""
    lo, hi = DOC_MIXES[mix]
    rng = _streams(seed)["doc_len"]
    cu = [0]
    while cu[-1] < n_tokens:
        n = int(round(float(np.exp(rng.uniform(np.log(lo), np.log(hi))))))
        cu.append(min(n_tokens, cu[-1] + max(1, n)))
    return np.asarray(cu, dtype=np.int64)
