"""GPU parity of the packed-document layer (ipttt_layer_forward_varlen: the
fast weight reset to W_o0 at every document boundary, itsolotime §3.2) against
the float64 oracle on the same seeded inputs.  Tolerances as for the batched
layer: relative Frobenius error <= 1e-2 (bf16) and <= 1e-4 (fp32) on O,
W_final and the accumulated update W_final - W_o0."""
import numpy as np
import pytest
import torch

import chunked_weight_mlp_place_b300 as ip
from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, down, rel, tdtype, up
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu


def run_varlen(w, a, cu, rule, W0=None, out_dtype=torch.float64):
    dt = tdtype(w)
    X, E = up(a["X"], dt), up(a["E"], dt)
    n = len(cu) - 1
    W0t = torch.from_numpy(np.ascontiguousarray(a["W_o0"] if W0 is None else W0, np.float32)).cuda()
    O = torch.empty(X.shape[0], w.d, dtype=dt, device="cuda")
    Wf = torch.empty(n, w.d_ff, w.d, dtype=torch.float32, device="cuda")
    ip.layer_forward_varlen(X, E, up(a["W_g"], dt), up(a["W_u"], dt), W0t, up(a["conv_w"], torch.float32),
                            up(a["P"], dt), cu, w.B, w.eta, rule, O, Wf)
    assert ip.sync_status() == 0
    return down(O, out_dtype), down(Wf, out_dtype)


def _case(dtype, d, d_ff, B, lengths, eta=0.05, seed=0):
    T = int(sum(lengths))
    w = inputs.workload("tiny", batch=1, L=T, B=B, d=d, d_ff=d_ff, dtype=dtype, eta=eta)
    a = inputs.generate(w, seed=seed)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return w, a, cu


def _check(O, Wf, Oref, Wref, W0, tol):
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Wf))
    assert rel(O, Oref) <= tol, rel(O, Oref)
    assert rel(Wf, Wref) <= tol, rel(Wf, Wref)
    assert rel(Wf - W0, Wref - W0) <= tol, rel(Wf - W0, Wref - W0)


@pytest.mark.parametrize("dtype,d,d_ff,B,lengths", [
    ("bf16", 128, 256, 64, [150, 64, 17, 300, 1]),      # ragged, whole, short, long, one token
    ("bf16", 512, 1024, 256, [1000, 700, 256, 33]),     # several tiles per operand, ragged tails
    ("bf16", 136, 264, 16, [40, 7, 16, 100]),           # d, d_ff off the tile sizes, B = 16
    ("fp32", 40, 72, 5, [13, 4, 9, 1, 25]),             # fp32 mode, any sizes
])
@pytest.mark.parametrize("rule", ["mse", "add"])
def test_varlen_matches_oracle(dtype, d, d_ff, B, lengths, rule):
    w, a, cu = _case(dtype, d, d_ff, B, lengths, seed=len(lengths) + d)
    O, Wf = run_varlen(w, a, cu, rule)
    Oref, Wref = orc.layer_forward_varlen(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], cu,
                                          B, w.eta, rule)
    _check(O, Wf, Oref, Wref, a["W_o0"][None], TOL[dtype])


def test_varlen_per_document_initial_weights():
    """W_o0 given per document (document order, not the longest-first order
    the engine runs them in)."""
    lengths = [70, 300, 20, 150]
    w, a, cu = _case("bf16", 128, 256, 64, lengths, seed=3)
    rng = np.random.default_rng(5)
    W0 = (a["W_o0"][None] + 0.05 * rng.standard_normal((len(lengths),) + a["W_o0"].shape)).astype(np.float32)
    O, Wf = run_varlen(w, a, cu, "mse", W0=W0)
    Oref, Wref = orc.layer_forward_varlen(a["X"], a["E"], a["W_g"], a["W_u"], W0, a["conv_w"], a["P"], cu,
                                          w.B, w.eta, "mse")
    _check(O, Wf, Oref, Wref, W0, TOL["bf16"])


def test_varlen_launches_and_a_single_document():
    lengths = [300, 100, 64]
    w, a, cu = _case("bf16", 128, 256, 64, lengths, seed=6)
    run_varlen(w, a, cu, "mse")
    k_max = -(-max(lengths) // w.B)
    # gate + conv + proj + split of W_o0 + k_max * (apply + residual + update) + one merge per document
    assert ip.last_launch_count() == 3 + 1 + 3 * k_max + len(lengths)
    # one document of whole chunks is the batched layer with batch 1
    w1, a1, cu1 = _case("bf16", 128, 256, 64, [256], seed=7)
    O, Wf = run_varlen(w1, a1, cu1, "mse")
    Oref, Wref = orc.layer_forward(a1["X"], a1["E"], a1["W_g"], a1["W_u"], a1["W_o0"], a1["conv_w"], a1["P"],
                                   256, 64, w1.eta, "mse")
    _check(O, Wf, Oref, Wref, a1["W_o0"][None], TOL["bf16"])


def test_varlen_full_size_4b_documents():
    """128k tokens at the 4B shape (d=2560, d_ff=9728, B=1024) packed as the
    long128k document mix.  The oracle follows every chunk of the two shortest
    documents (one short chunk; several chunks ending in a short one) and the
    first chunk of the longest."""
    w = inputs.workload("4b")
    a = inputs.generate(w, seed=0)
    cu = inputs.doc_boundaries(w.L, seed=0, mix="long128k")
    O, Wf = run_varlen(w, a, cu, "mse", out_dtype=torch.float32)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Wf))
    lens = np.diff(cu)
    by_len = np.argsort(lens, kind="stable")
    picks = [int(by_len[0])] + [int(i) for i in by_len if w.B < lens[i] <= 3 * w.B][:1]
    for i in picks:
        r = slice(int(cu[i]), int(cu[i + 1]))
        Oref, Wref = orc.layer_forward_varlen(a["X"][r], a["E"][r], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"],
                                              a["P"], [0, int(lens[i])], w.B, w.eta, "mse")
        _check(O[r], Wf[i][None], Oref, Wref, a["W_o0"][None], TOL["bf16"])
    j = int(by_len[-1])
    r = slice(int(cu[j]), int(cu[j]) + w.B)
    Oref, _ = orc.layer_forward_varlen(a["X"][r], a["E"][r], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"],
                                       [0, w.B], w.B, w.eta, "mse")
    assert rel(O[r], Oref) <= TOL["bf16"]
