"""GPU parity of the persistent MSE chunk engine (the whole chunk loop as one
kernel, used in bf16 mode when B, d and d_ff are multiples of 256) against the
float64 oracle, at sizes that exercise its work split: several chunks (the
apply of chunk k+1 waiting for the update rows of chunk k), d_ff cut into
uneven slices, two sequences, one chunk, several column blocks and token tiles.
Tolerance: relative Frobenius error <= 1e-2 on O (whole and per chunk),
W_final and the accumulated update W_final - W_o0."""
import numpy as np
import pytest
import torch

import chunked_weight_mlp_place_b300 as ip
from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, down, rel, run_layer, up
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu


def _check(O, Wf, Oref, Wref, W0, w):
    tol = TOL["bf16"]
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Wf))
    assert rel(O, Oref) <= tol, rel(O, Oref)
    Oc, Rc = O.reshape(-1, w.B, w.d), Oref.reshape(-1, w.B, w.d)
    worst = max(rel(Oc[i], Rc[i]) for i in range(Oc.shape[0]))
    assert worst <= tol, worst
    assert rel(Wf, Wref) <= tol, rel(Wf, Wref)
    assert rel(Wf - W0, Wref - W0) <= tol, rel(Wf - W0, Wref - W0)


# Chunks below 1024 tokens run in windows of chunks where a window fits (test_gpu_windows.py);
# the lengths here fit none, so the engine runs on the chunks themselves.
@pytest.mark.parametrize("batch,L,B,d,d_ff", [
    (1, 3840, 256, 512, 1024),    # 15 chunks, two column blocks, d_ff in 4 slices of one tile
    (2, 768, 256, 256, 768),      # two sequences, d_ff in 3 slices
    (1, 1536, 512, 768, 1280),    # two token tiles per chunk, d_ff in slices of 1, 1, 1, 2 tiles
    (1, 1024, 1024, 256, 256),    # one chunk, one slice
    (1, 8192, 1024, 2560, 9728),  # the 4B shape, 8 chunks
])
def test_engine_matches_oracle(batch, L, B, d, d_ff):
    w = inputs.workload("500m", batch=batch, L=L, B=B, d=d, d_ff=d_ff, eta=0.05, vocab=512)
    a = inputs.generate(w, seed=B + d)
    O, Wf = run_layer(w, a, "mse")
    Oref, Wref = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], L, B,
                                   w.eta, "mse")
    _check(O, Wf, Oref, Wref, a["W_o0"][None], w)
    assert ip.last_launch_count() <= 8  # gate, conv, proj, split, engine, merge (+ memsets are not kernels)


def test_engine_repeated_runs_agree():
    """The engine's reductions are fp32 additions in whatever order the slices
    finish: repeated runs agree to the tolerance, and each matches the oracle."""
    w = inputs.workload("500m", batch=1, L=1280, B=256, d=512, d_ff=1024, eta=0.05)
    a = inputs.generate(w, seed=5)
    Oref, Wref = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], w.L, w.B,
                                   w.eta, "mse")
    for _ in range(4):
        O, Wf = run_layer(w, a, "mse")
        _check(O, Wf, Oref, Wref, a["W_o0"][None], w)


def test_engine_per_sequence_initial_weights():
    w = inputs.workload("500m", batch=2, L=768, B=256, d=256, d_ff=512, eta=0.05)
    a = inputs.generate(w, seed=9)
    rng = np.random.default_rng(1)
    W0 = (rng.standard_normal((2, w.d_ff, w.d)) * w.d_ff ** -0.5).astype(np.float32)
    O, Wf = run_layer(w, a, "mse", W0=W0)
    Oref, Wref = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], W0, a["conv_w"], a["P"], w.L, w.B, w.eta,
                                   "mse")
    _check(O, Wf, Oref, Wref, W0, w)
