"""Float64 CPU oracle of the In-Place TTT fast-weight layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  The CUDA library never calls it and shares no code with it.

It is the method written out plainly, in the order the pages give it, with a
library matmul as the only building block:

* gated MLP ``MLP(x) = (SiLU(x W_g) * (x W_u)) W_o`` with W_g, W_u frozen and
  the final projection W_o used as the fast weight -- In-Place TTT write-up
  (itsolotime), §2.1 "core insight", the gated-MLP formula; su666666 write-up,
  "first axe" (the down projection is the fast weight);
* the target ``V = Proj(Conv(E))`` built from token embeddings E -- itsolotime
  §2.3 "LM-aligned objective"; su666666 "second axe";
* the chunk-wise apply-then-update loop: split the activations (the pages'
  "A", here Z) and targets V into K = L/B chunks; for chunk k first apply the
  current fast weight, then take one gradient step on that chunk --
  itsolotime §2.2 "large-chunk update" and Fig. 1; su666666 "third axe"
  (outputs of the whole chunk first, then the gradient accumulated over the
  chunk, one update).

Readings where the pages leave a step open:

* loss: ``l_k(W) = ||Z_k W - V_k||_F^2 / (2B)`` ("make W z_t close to v_t",
  su666666 "second axe"), so one gradient step is
  ``W <- W - (eta/B) Z_k^T (Z_k W - V_k)`` (the MSE rule);
* the additive rule ``W <- W + (eta/B) Z_k^T V_k`` is the step of the inner
  product ("simple similarity measure") loss ``-<Z_k W, V_k>/B`` whose updates
  only accumulate (itsolotime §2.3 last paragraph, and the open questions in
  the conclusion);
* the conv is depthwise, width 4, tap j multiplies E[t+j], no bias, and it
  reads zeros past the end of the token's own chunk, so no update reads past
  its chunk (itsolotime §2.3: the conv lets V carry future tokens; the
  next-token example puts a one at the next position);
* the step is normalised by the chunk size B;
* SiLU(a) = a * sigmoid(a), computed with an exact float64 exp.

Parity pins (tests/test_oracle_pins.py) tie every function here to something
other than itself: a hand-worked example, finite differences, per-token brute
force, closed forms, library routines and the pages' special cases.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

__all__ = [
    "silu", "gated_activation", "chunk_conv", "make_targets", "mse_loss",
    "chunk_step", "chunk_engine", "layer_forward", "layer_forward_varlen", "layers_forward",
]


def silu(a: np.ndarray) -> np.ndarray:
    """SiLU(a) = a / (1 + exp(-a)), the gate activation of the gated MLP
    (itsolotime §2.1, gated-MLP formula)."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def gated_activation(X: np.ndarray, W_g: np.ndarray, W_u: np.ndarray) -> np.ndarray:
    """Z = SiLU(X W_g) * (X W_u): the activation that enters the fast weight W_o
    (itsolotime §2.1; the pages' "A", su666666's "z").  X is (T, d)."""
    X = np.asarray(X, np.float64)
    return silu(X @ np.asarray(W_g, np.float64)) * (X @ np.asarray(W_u, np.float64))


def chunk_conv(E: np.ndarray, conv_w: np.ndarray, B: int) -> np.ndarray:
    """Depthwise width-4 conv over positions t..t+3, zero past each chunk's end.

    ``C[t, c] = sum_{j=0..3} conv_w[c, j] * E[t+j, c]`` where ``E[t+j]`` counts
    as zero once ``t+j`` leaves the chunk of B tokens that holds t.  E is
    (L, d) for one sequence, L a multiple of B (itsolotime §2.3 "Conv"; the
    chunk-end padding keeps every update inside its own chunk).
    """
    E = np.asarray(E, np.float64)
    w = np.asarray(conv_w, np.float64)
    L, d = E.shape
    if L % B:
        raise ValueError("L must be a multiple of B")
    C = np.zeros((L, d), np.float64)
    for c0 in range(0, L, B):
        Ek = E[c0:c0 + B]
        Ck = C[c0:c0 + B]
        for j in range(4):
            if j < B:
                Ck[:B - j] += Ek[j:] * w[:, j]
    return C


def make_targets(E: np.ndarray, conv_w: np.ndarray, P: np.ndarray, B: int) -> np.ndarray:
    """V = Proj(Conv(E)) = chunk_conv(E) @ P (itsolotime §2.3)."""
    return chunk_conv(E, conv_w, B) @ np.asarray(P, np.float64)


def mse_loss(Z_k: np.ndarray, V_k: np.ndarray, W: np.ndarray) -> float:
    """l_k(W) = ||Z_k W - V_k||_F^2 / (2B), the chunk loss of the MSE rule."""
    R = np.asarray(Z_k, np.float64) @ np.asarray(W, np.float64) - np.asarray(V_k, np.float64)
    return float(np.sum(R * R) / (2.0 * Z_k.shape[0]))


def chunk_step(Z_k: np.ndarray, V_k: np.ndarray, W: np.ndarray, eta: float,
               rule: str = "mse") -> Tuple[np.ndarray, np.ndarray]:
    """One chunk: apply the current fast weight, then one gradient step.

    Returns (O_k, W_next) with O_k = Z_k W (itsolotime §2.2 step 1 "apply") and
    W_next from the chunk's gradient (§2.2 step 2 "update").
    """
    Z_k = np.asarray(Z_k, np.float64)
    V_k = np.asarray(V_k, np.float64)
    B = Z_k.shape[0]
    O_k = Z_k @ W
    if rule == "mse":
        W_next = W - (eta / B) * (Z_k.T @ (O_k - V_k))
    elif rule == "add":
        W_next = W + (eta / B) * (Z_k.T @ V_k)
    else:
        raise ValueError(f"unknown rule {rule!r}")
    return O_k, W_next


def chunk_engine(Z: np.ndarray, V: np.ndarray, W_o0: np.ndarray, B: int, eta: float,
                 rule: str = "mse", max_chunks: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """The apply-then-update loop over the K = L/B chunks of one sequence.

    Z is (L, d_ff), V is (L, d), W_o0 is (d_ff, d).  Returns O (rows of the
    processed chunks) and the fast weight after the last processed chunk.
    """
    L = Z.shape[0]
    if L % B:
        raise ValueError("L must be a multiple of B")
    K = L // B if max_chunks is None else min(L // B, max_chunks)
    W = np.array(W_o0, np.float64, copy=True)
    O = np.zeros((K * B, V.shape[1]), np.float64)
    for k in range(K):
        sl = slice(k * B, (k + 1) * B)
        O[sl], W = chunk_step(Z[sl], V[sl], W, eta, rule)
    return O, W


def layer_forward(X: np.ndarray, E: np.ndarray, W_g: np.ndarray, W_u: np.ndarray,
                  W_o0: np.ndarray, conv_w: np.ndarray, P: np.ndarray, L: int, B: int,
                  eta: float, rule: str = "mse", max_chunks: Optional[int] = None,
                  ) -> Tuple[np.ndarray, np.ndarray]:
    """The whole fast-weight layer for ``batch = X.shape[0] // L`` sequences.

    Chunk by chunk, in the method's own order: Z_k from X_k, V_k from E_k (the
    conv only reads its own chunk), O_k = Z_k W_k, then the update.  Memory is
    O(B) per sequence, like the method's (su666666 "third axe").

    X, E are (batch*L, d), token-major per sequence.  W_o0 is (d_ff, d) shared
    by all sequences, or (batch, d_ff, d).  Returns O (batch*K'*B, d) for the
    processed chunks K' = min(K, max_chunks) and W_final (batch, d_ff, d).
    """
    X = np.asarray(X, np.float64)
    E = np.asarray(E, np.float64)
    if L % B or X.shape[0] % L:
        raise ValueError("rows must be batch*L with L a multiple of B")
    batch = X.shape[0] // L
    K = L // B if max_chunks is None else min(L // B, max_chunks)
    W0 = np.asarray(W_o0, np.float64)
    d = E.shape[1]
    O = np.zeros((batch * K * B, d), np.float64)
    W_fin = np.zeros((batch,) + W0.shape[-2:], np.float64)
    for s in range(batch):
        W = np.array(W0[s] if W0.ndim == 3 else W0, np.float64, copy=True)
        for k in range(K):
            rows = slice(s * L + k * B, s * L + (k + 1) * B)
            Z_k = gated_activation(X[rows], W_g, W_u)
            V_k = make_targets(E[rows], conv_w, P, B)
            O[s * K * B + k * B: s * K * B + (k + 1) * B], W = chunk_step(Z_k, V_k, W, eta, rule)
        W_fin[s] = W
    return O, W_fin


def layer_forward_varlen(X: np.ndarray, E: np.ndarray, W_g: np.ndarray, W_u: np.ndarray,
                         W_o0: np.ndarray, conv_w: np.ndarray, P: np.ndarray, cu_seqlens,
                         B: int, eta: float, rule: str = "mse") -> Tuple[np.ndarray, np.ndarray]:
    """The layer over packed documents, with the fast weight reset at every
    document boundary (itsolotime §3.2, "boundary reset": back to the
    pretrained initial value, so no document sees another's updates).

    Document i holds rows cu_seqlens[i] .. cu_seqlens[i+1]-1 of X and E.
    Readings where the pages are silent:

    * a document's chunks start at its first token: B tokens each, the last one
      holding what is left (1 .. B tokens);
    * that last chunk's step is normalised by its own token count (the chunk
      loss is the mean over the chunk's tokens, as for full chunks);
    * the conv reads zeros past the document's end, as past any chunk's end.

    W_o0 is (d_ff, d) shared by all documents, or (n_docs, d_ff, d).  Returns
    O (T, d) and W_final (n_docs, d_ff, d).
    """
    X = np.asarray(X, np.float64)
    E = np.asarray(E, np.float64)
    cu = [int(c) for c in cu_seqlens]
    n_docs = len(cu) - 1
    if n_docs < 0 or cu[0] != 0 or cu[-1] != X.shape[0] or any(b <= a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must rise strictly from 0 to the number of rows")
    W0 = np.asarray(W_o0, np.float64)
    O = np.zeros((X.shape[0], E.shape[1]), np.float64)
    W_fin = np.zeros((n_docs,) + W0.shape[-2:], np.float64)
    for i in range(n_docs):
        W = np.array(W0[i] if W0.ndim == 3 else W0, np.float64, copy=True)
        for c0 in range(cu[i], cu[i + 1], B):
            rows = slice(c0, min(c0 + B, cu[i + 1]))
            n = rows.stop - rows.start
            Z_k = gated_activation(X[rows], W_g, W_u)
            V_k = make_targets(E[rows], conv_w, P, n)  # the whole (possibly short) chunk is one conv chunk
            O[rows], W = chunk_step(Z_k, V_k, W, eta, rule)
        W_fin[i] = W
    return O, W_fin


def layers_forward(X: np.ndarray, E: np.ndarray, W_g: np.ndarray, W_u: np.ndarray, W_o0: np.ndarray,
                   conv_w: np.ndarray, P: np.ndarray, L: int, B: int, eta: float,
                   rule: str = "mse") -> Tuple[np.ndarray, np.ndarray]:
    """Several layers' fast-weight MLPs over the same tokens: layer l takes its
    own hidden states X[l] and its own W_g, W_u, W_o0, conv_w and P, and every
    layer's target is built from the same token embeddings E (the In-Place TTT
    layer is the MLP block of each layer it is put in: itsolotime §2.1; the
    target of §2.3 reads the token embeddings).  Layers do not interact here.

    X is (n_layers, batch*L, d); E (batch*L, d); W_g, W_u (n_layers, d, d_ff);
    W_o0 (n_layers, d_ff, d) or (n_layers, batch, d_ff, d); conv_w
    (n_layers, d, 4); P (n_layers, d, d).  Returns O (n_layers, batch*L, d) and
    W_final (n_layers, batch, d_ff, d).
    """
    X = np.asarray(X, np.float64)
    n = X.shape[0]
    outs = [layer_forward(X[l], E, W_g[l], W_u[l], W_o0[l], conv_w[l], P[l], L, B, eta, rule) for l in range(n)]
    return np.stack([o for o, _ in outs]), np.stack([w for _, w in outs])
