"""The additive rule over one sequence split across GPUs (context parallelism).

Each rank holds a run of whole chunks of every sequence: rank r the tokens
r*L .. r*L+L-1 of a sequence of world*L tokens, L a multiple of the chunk size
B (the conv pads at chunk ends, so no rank needs its neighbour's tokens).  The
additive rule is associative (In-Place TTT write-up, itsolotime §2.3; §3.2:
parallel equals serial): the fast weight after a run of chunks is the weight
before it plus (eta/B) times the run's sum of Z_k^T V_k.  So

1. every rank builds Z and V of its tokens and the sum S_r of Z_k^T V_k over its
   chunks (one GEMM);
2. one exchange: the ranks all-gather their sums (torch.distributed; NCCL on
   GPUs, gloo on CPUs);
3. rank r starts from W_0 + (eta/B) * sum of S_r' over the ranks r' < r and
   runs its own chunks with the additive rule.

The last rank's W_final is the sequence's.  Every step's arithmetic runs in the
library (``LibraryBackend``); the exchange moves batch x d_ff x d fp32 sums
once.  The MSE rule has no such split (its chunks are sequential), so it is not
offered here.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _lib as ip

__all__ = ["LibraryBackend", "additive_forward", "allgather_earlier"]


class LibraryBackend:
    """The steps of one rank through the library's C-ABI (CUDA tensors)."""

    def gate_targets(self, X, E, W_g, W_u, conv_w, P, L, B):
        Z = torch.empty(X.shape[0], W_g.shape[1], dtype=X.dtype, device=X.device)
        V = torch.empty_like(E)
        ip.gate_up(X, W_g, W_u, Z)
        ip.make_targets(E, conv_w, P, V, L, B)
        return Z, V

    def sums(self, Z, V, L):
        S = torch.empty(Z.shape[0] // L, Z.shape[1], V.shape[1], dtype=torch.float32, device=Z.device)
        ip.additive_sums(Z, V, L, S)
        return S

    def start(self, W_o0, batch, B):
        """Every sequence's copy of W_o0 ((d_ff, d), or per sequence (batch, d_ff, d))."""
        W = torch.empty((batch,) + tuple(W_o0.shape[-2:]), dtype=torch.float32, device=W_o0.device)
        ip.copy_weights(W_o0, W)
        return W

    def axpy(self, W, S, alpha):
        ip.weight_axpy(W, S, alpha)

    def chunk_forward(self, Z, V, W_start, L, B, eta, O, W_final):
        ip.chunk_forward(Z, V, W_start, L, B, eta, "add", O, W_final)


def allgather_earlier(S, group=None):
    """The chunk sums of the ranks before this one, by one all-gather over `group`
    (every rank receives world - 1 sums of batch x d_ff x d fp32); none without
    an initialised process group."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return []
    gathered = [torch.empty_like(S) for _ in range(dist.get_world_size(group))]
    dist.all_gather(gathered, S, group=group)
    return gathered[:dist.get_rank(group)]


def additive_forward(X, E, W_g, W_u, W_o0, conv_w, P, L: int, B: int, eta: float, O, W_final, group=None,
                     backend=None, exchange=None) -> None:
    """This rank's part of the additive rule over sequences split across the ranks of `group`.

    X, E: this rank's run of every sequence, (batch*L, d), sequence s in rows
    s*L .. s*L+L-1; W_g, W_u, conv_w, P, W_o0 as in ipttt_layer_forward (the
    same on every rank).  O (batch*L, d): this rank's outputs; W_final
    (batch, d_ff, d): the fast weight after this rank's chunks (the sequence's
    final weight on the last rank).

    ``exchange(S, group)`` returns the chunk sums of the earlier ranks given this
    rank's own; the default is :func:`allgather_earlier` (without an initialised
    process group: none, so the call is the plain additive rule).  Passing one
    lets the ranks run in turn in one process, each handing its sum to the next.
    """
    be = backend if backend is not None else LibraryBackend()
    Z, V = be.gate_targets(X, E, W_g, W_u, conv_w, P, L, B)
    S = be.sums(Z, V, L)
    W_start = be.start(W_o0, S.shape[0], B)
    for S_r in (exchange or allgather_earlier)(S, group):
        be.axpy(W_start, S_r, eta / B)
    be.chunk_forward(Z, V, W_start, L, B, eta, O, W_final)
