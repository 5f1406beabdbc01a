"""GPU parity of IPTTT_RULE_ADD_BLOCKCAUSAL (the additive rule's outputs from its
block-causal quadratic form O = Z W_0 + (eta/B) mask(Z Z^T) V, W_final = W_0 +
(eta/B) Z^T V) against the float64 oracle's additive rule, and against the
library's own scan-based additive rule at a full sweep size.  Tolerances as for
the layer: relative Frobenius error <= 1e-2 (bf16) and <= 1e-4 (fp32) on O,
W_final and the accumulated update W_final - W_o0."""
import numpy as np
import pytest

from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, rel, run_layer
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu


def _check(O, Wf, Oref, Wref, W0, tol):
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Wf))
    assert rel(O, Oref) <= tol, rel(O, Oref)
    assert rel(Wf, Wref) <= tol, rel(Wf, Wref)
    assert rel(Wf - W0, Wref - W0) <= tol, rel(Wf - W0, Wref - W0)


@pytest.mark.parametrize("dtype,batch,L,B,d,d_ff", [
    ("bf16", 2, 256, 64, 128, 256),       # two sequences, several score tiles
    ("bf16", 1, 512, 16, 136, 264),       # B = 16, d and d_ff off the tile sizes
    ("bf16", 1, 1024, 128, 512, 1024),    # diagonal tiles cut by the mask inside a 128 x 256 tile
    ("fp32", 1, 60, 5, 40, 72),           # fp32 mode, any sizes
])
def test_blockcausal_matches_oracle_additive(dtype, batch, L, B, d, d_ff):
    w = inputs.workload("tiny", batch=batch, L=L, B=B, d=d, d_ff=d_ff, dtype=dtype, eta=0.05)
    a = inputs.generate(w, seed=L + d)
    O, Wf = run_layer(w, a, "add_blockcausal")
    Oref, Wref = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], L, B,
                                   w.eta, "add")
    _check(O, Wf, Oref, Wref, a["W_o0"][None], TOL[dtype])
