"""GPU parity of the multi-layer call (ipttt_layers_forward: several layers'
fast-weight MLPs over the same tokens in one launch per step) against the
float64 oracle's layers_forward on the same seeded inputs.  Tolerances as for
one layer: relative Frobenius error <= 1e-2 (bf16) and <= 1e-4 (fp32) on O,
W_final and the accumulated update W_final - W_o0."""
import numpy as np
import pytest
import torch

import chunked_weight_mlp_place_b300 as ip
from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, down, rel, tdtype, up
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu


def _inputs(dtype, n_layers, batch, d, d_ff, L, B, eta=0.05):
    w = inputs.workload("tiny", batch=batch, L=L, B=B, d=d, d_ff=d_ff, dtype=dtype, eta=eta)
    per = [inputs.generate(w, seed=100 + l) for l in range(n_layers)]
    a = {k: np.stack([p[k] for p in per]) for k in ("X", "W_g", "W_u", "W_o0", "conv_w", "P")}
    a["E"] = inputs.generate(w, seed=7)["E"]
    return w, a


def _run(w, a, rule, W0=None):
    dt = tdtype(w)
    n = a["X"].shape[0]
    t = {k: up(a[k], dt) for k in ("X", "E", "W_g", "W_u", "P")}
    W0t = torch.from_numpy(np.ascontiguousarray(a["W_o0"] if W0 is None else W0, np.float32)).cuda()
    O = torch.empty(n, w.batch * w.L, w.d, dtype=dt, device="cuda")
    Wf = torch.empty(n, w.batch, w.d_ff, w.d, dtype=torch.float32, device="cuda")
    ip.layers_forward(t["X"], t["E"], t["W_g"], t["W_u"], W0t, up(a["conv_w"], torch.float32), t["P"], w.L, w.B,
                      w.eta, rule, O, Wf)
    assert ip.sync_status() == 0
    return down(O), down(Wf)


def _check(O, Wf, Oref, Wref, W0, tol):
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Wf))
    assert rel(O, Oref) <= tol, rel(O, Oref)
    assert rel(Wf, Wref) <= tol, rel(Wf, Wref)
    assert rel(Wf - W0, Wref - W0) <= tol, rel(Wf - W0, Wref - W0)


@pytest.mark.parametrize("dtype,n_layers,batch,d,d_ff,L,B", [
    ("bf16", 3, 2, 128, 256, 256, 64),     # per-layer W_o0 shared by two sequences
    ("bf16", 2, 1, 256, 512, 512, 128),    # one sequence: W_o0 is already per entry
    ("bf16", 4, 1, 136, 264, 96, 16),      # d, d_ff off the tile sizes, B = 16
    ("fp32", 3, 2, 40, 72, 30, 5),         # fp32 mode, any sizes
])
@pytest.mark.parametrize("rule", ["mse", "add"])
def test_layers_match_oracle(dtype, n_layers, batch, d, d_ff, L, B, rule):
    w, a = _inputs(dtype, n_layers, batch, d, d_ff, L, B)
    O, Wf = _run(w, a, rule)
    Oref, Wref = orc.layers_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], L, B,
                                    w.eta, rule)
    _check(O, Wf, Oref, Wref, a["W_o0"][:, None], TOL[dtype])


def test_layers_per_sequence_initial_weights_and_launches():
    w, a = _inputs("bf16", 3, 2, 128, 256, 256, 64)
    rng = np.random.default_rng(9)
    W0 = (a["W_o0"][:, None] + 0.05 * rng.standard_normal((3, 2) + a["W_o0"].shape[1:])).astype(np.float32)
    O, Wf = _run(w, a, "mse", W0=W0)
    # gate + conv + proj (one launch each for all layers) + split + K * (apply + residual + update) + merge
    assert ip.last_launch_count() == 3 + 1 + 3 * (w.L // w.B) + 1
    Oref, Wref = orc.layers_forward(a["X"], a["E"], a["W_g"], a["W_u"], W0, a["conv_w"], a["P"], w.L, w.B, w.eta,
                                    "mse")
    _check(O, Wf, Oref, Wref, W0, TOL["bf16"])
    # a per-layer W_o0 shared by the sequences adds one copy per layer
    _run(w, a, "mse")
    assert ip.last_launch_count() == 3 + 3 + 1 + 3 * (w.L // w.B) + 1
