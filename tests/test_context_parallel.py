"""Context-parallel additive rule (chunked_weight_mlp_place_b300.context_parallel)
as two and three gloo ranks on CPU, each holding a run of every sequence, against the
float64 oracle's one-pass additive layer.  Each rank's steps run on a float64
stand-in of the library built from the oracle's functions; the exchange and the
start weights are the module's own."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class OracleBackend:
    """The steps of one rank in float64 on the host (test stand-in of the library)."""

    def gate_targets(self, X, E, W_g, W_u, conv_w, P, L, B):
        from oracle import ipttt_oracle as orc
        n = X.shape[0] // L
        Z = orc.gated_activation(X.numpy(), W_g.numpy(), W_u.numpy())
        V = np.concatenate([orc.make_targets(E.numpy()[s * L:(s + 1) * L], conv_w.numpy(), P.numpy(), B)
                            for s in range(n)])
        return torch.from_numpy(Z), torch.from_numpy(V)

    def sums(self, Z, V, L):
        n = Z.shape[0] // L
        return torch.stack([Z[s * L:(s + 1) * L].T @ V[s * L:(s + 1) * L] for s in range(n)])

    def start(self, W_o0, batch, B):
        return W_o0.expand(batch, *W_o0.shape[-2:]).clone() if W_o0.dim() == 2 else W_o0.clone()

    def axpy(self, W, S, alpha):
        W.add_(S, alpha=alpha)

    def chunk_forward(self, Z, V, W_start, L, B, eta, O, W_final):
        from oracle import ipttt_oracle as orc
        for s in range(Z.shape[0] // L):
            r = slice(s * L, (s + 1) * L)
            o, w = orc.chunk_engine(Z[r].numpy(), V[r].numpy(), W_start[s].numpy(), B, eta, "add")
            O[r] = torch.from_numpy(o)
            W_final[s] = torch.from_numpy(w)


def _inputs(batch, L_full, d, d_ff, seed=5):
    rng = np.random.default_rng(seed)
    return dict(X=rng.standard_normal((batch * L_full, d)), E=rng.standard_normal((batch * L_full, d)),
                W_g=rng.standard_normal((d, d_ff)) / np.sqrt(d), W_u=rng.standard_normal((d, d_ff)) / np.sqrt(d),
                W_o0=rng.standard_normal((d_ff, d)) / np.sqrt(d_ff), conv_w=rng.standard_normal((d, 4)) * 0.7,
                P=rng.standard_normal((d, d)) / np.sqrt(d))


def _local(a, k, rank, batch, L):
    """Rank `rank`'s run of L tokens of every sequence."""
    L_full = a[k].shape[0] // batch
    return torch.from_numpy(np.concatenate([a[k][s * L_full + rank * L: s * L_full + (rank + 1) * L]
                                            for s in range(batch)]))


def _worker(rank, world, port, cfg, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from chunked_weight_mlp_place_b300 import context_parallel as cp

    batch, L, B, d, d_ff, eta = cfg
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        a = _inputs(batch, world * L, d, d_ff)
        t = {k: torch.from_numpy(a[k]) for k in ("W_g", "W_u", "W_o0", "conv_w", "P")}
        O = torch.empty(batch * L, d, dtype=torch.float64)
        W_final = torch.empty(batch, d_ff, d, dtype=torch.float64)
        cp.additive_forward(_local(a, "X", rank, batch, L), _local(a, "E", rank, batch, L), t["W_g"], t["W_u"],
                            t["W_o0"], t["conv_w"], t["P"], L, B, eta, O, W_final, backend=OracleBackend())
        q.put((rank, O.numpy(), W_final.numpy()))
    finally:
        dist.destroy_process_group()


def _run(world, cfg):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    procs = [ctx.Process(target=_worker, args=(r, world, port, cfg, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict((r, (o, w)) for r, o, w in (q.get(timeout=120) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


@pytest.mark.parametrize("world,batch", [(2, 2), (3, 1)])
def test_ranks_equal_the_one_pass_additive_layer(world, batch):
    from oracle import ipttt_oracle as orc
    L, B, d, d_ff, eta = 12, 4, 5, 7, 0.2
    got = _run(world, (batch, L, B, d, d_ff, eta))
    a = _inputs(batch, world * L, d, d_ff)
    O_ref, W_ref = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"],
                                     world * L, B, eta, "add")
    O_ref = O_ref.reshape(batch, world, L, d)
    for r in range(world):
        np.testing.assert_allclose(got[r][0].reshape(batch, L, d), O_ref[:, r], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got[world - 1][1], W_ref, rtol=1e-12, atol=1e-12)
    # the first rank's weight is the one after its own chunks only
    O_half, W_half = orc.layer_forward(_local(a, "X", 0, batch, L).numpy(), _local(a, "E", 0, batch, L).numpy(),
                                       a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], L, B, eta, "add")
    np.testing.assert_allclose(got[0][1], W_half, rtol=1e-12, atol=1e-12)
