"""GPU checks of the context-parallel additive rule's pieces: the chunk-sum GEMM
(ipttt_additive_sums) and the weight update (ipttt_weight_axpy) against
float64 sums, and one rank of chunked_weight_mlp_place_b300.context_parallel
(no process group) against the oracle's additive layer."""
import numpy as np
import pytest
import torch

import chunked_weight_mlp_place_b300 as ip
from chunked_weight_mlp_place_b300 import context_parallel as cp
from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, down, rel, up
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu


def test_additive_sums_and_weight_axpy():
    rng = np.random.default_rng(3)
    batch, L, d, d_ff = 2, 256, 136, 264
    Z = inputs.round_to_bf16(rng.standard_normal((batch * L, d_ff)).astype(np.float32))
    V = inputs.round_to_bf16(rng.standard_normal((batch * L, d)).astype(np.float32))
    S = torch.empty(batch, d_ff, d, device="cuda")
    ip.additive_sums(up(Z, torch.bfloat16), up(V, torch.bfloat16), L, S)
    ref = np.stack([Z[s * L:(s + 1) * L].astype(np.float64).T @ V[s * L:(s + 1) * L] for s in range(batch)])
    assert rel(down(S), ref) <= 1e-5
    W = rng.standard_normal((batch, d_ff, d)).astype(np.float32)
    Wt = torch.from_numpy(W).cuda()
    ip.weight_axpy(Wt, S, 0.3)
    assert ip.sync_status() == 0
    np.testing.assert_allclose(down(Wt), W + 0.3 * down(S), rtol=1e-6, atol=1e-6)


def test_one_rank_is_the_additive_layer():
    w = inputs.workload("tiny", batch=2, L=256, B=64, d=128, d_ff=256, dtype="bf16", eta=0.05)
    a = inputs.generate(w, seed=11)
    t = {k: up(a[k], torch.bfloat16) for k in ("X", "E", "W_g", "W_u", "P")}
    O = torch.empty(w.batch * w.L, w.d, dtype=torch.bfloat16, device="cuda")
    Wf = torch.empty(w.batch, w.d_ff, w.d, device="cuda")
    cp.additive_forward(t["X"], t["E"], t["W_g"], t["W_u"], torch.from_numpy(a["W_o0"]).cuda(),
                        torch.from_numpy(a["conv_w"]).cuda(), t["P"], w.L, w.B, w.eta, O, Wf)
    assert ip.sync_status() == 0
    Oref, Wref = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], w.L, w.B,
                                   w.eta, "add")
    assert rel(down(O), Oref) <= TOL["bf16"]
    assert rel(down(Wf), Wref) <= TOL["bf16"]
    assert rel(down(Wf) - a["W_o0"], Wref - a["W_o0"]) <= TOL["bf16"]


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_in_turn_through_the_library_equal_the_one_pass_additive_layer(world):
    """The sequence split into `world` runs of whole chunks; the ranks run one after
    another in this process, every step through the library (LibraryBackend), each
    rank's chunk sum handed to the later ranks by the exchange.  The concatenated
    outputs and the last rank's W_final equal the oracle's one-pass additive layer;
    the first rank's W_final equals the oracle's over its own chunks only."""
    batch, L, B, d, d_ff = 2, 256, 64, 128, 256
    w = inputs.workload("tiny", batch=batch, L=world * L, B=B, d=d, d_ff=d_ff, dtype="bf16", eta=0.05)
    a = inputs.generate(w, seed=20 + world)
    t = {k: up(a[k], torch.bfloat16) for k in ("W_g", "W_u", "P")}
    W0 = torch.from_numpy(a["W_o0"]).cuda()
    cw = torch.from_numpy(a["conv_w"]).cuda()

    def run_of(k, r):  # rank r's run of L tokens of every sequence
        x = a[k].reshape(batch, world, L, d)[:, r].reshape(batch * L, d)
        return np.ascontiguousarray(x)

    sums = []

    def exchange(S, group):  # the earlier ranks' sums; this rank's kept for the later ones
        earlier = list(sums)
        sums.append(S.clone())
        return earlier

    Os, Wfs = [], []
    for r in range(world):
        O = torch.empty(batch * L, d, dtype=torch.bfloat16, device="cuda")
        Wf = torch.empty(batch, d_ff, d, device="cuda")
        cp.additive_forward(up(run_of("X", r), torch.bfloat16), up(run_of("E", r), torch.bfloat16), t["W_g"],
                            t["W_u"], W0, cw, t["P"], L, B, w.eta, O, Wf, exchange=exchange)
        assert ip.sync_status() == 0
        Os.append(down(O).reshape(batch, L, d))
        Wfs.append(down(Wf))
    Oref, Wref = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], world * L, B,
                                   w.eta, "add")
    O_cat = np.concatenate(Os, axis=1).reshape(batch * world * L, d)
    assert rel(O_cat, Oref) <= TOL["bf16"], rel(O_cat, Oref)
    assert rel(Wfs[-1], Wref) <= TOL["bf16"]
    assert rel(Wfs[-1] - a["W_o0"], Wref - a["W_o0"]) <= TOL["bf16"]
    O0, W0ref = orc.layer_forward(run_of("X", 0), run_of("E", 0), a["W_g"], a["W_u"], a["W_o0"], a["conv_w"],
                                  a["P"], L, B, w.eta, "add")
    assert rel(Os[0].reshape(batch * L, d), O0) <= TOL["bf16"]
    assert rel(Wfs[0] - a["W_o0"], W0ref - a["W_o0"]) <= TOL["bf16"]
