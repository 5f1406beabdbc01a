"""GPU parity at the workloads' full sizes, every chunk against the oracle.

The layer runs through ipttt_layer_forward at each workload's full shape (the
4B-scale one is exactly the launch configuration the benchmark times) and the
float64 oracle runs the same seeded inputs over the whole sequence.  Compared:

* O over the whole sequence, and chunk by chunk: the worst chunk, and the worst
  (chunk, 256-column block) piece, so that one bad tile of one late chunk cannot
  hide in the norm of the whole array;
* W_final after the last chunk, and the accumulated update W_final - W_o0
  (W_final alone is close to W_o0 and would hide update errors).

Tolerance: relative Frobenius error <= 1e-2 in bf16 mode on each of those.  The
chunk-size sweep (L = 32768 at the 4B shape, B in {64, 256, 512, 1024, 4096},
both rules: the chunk-size ablation of the write-ups, itsolotime Fig. 3b) shares
one oracle Z; the block-causal additive form is checked against the same oracle
results as the scan-based additive rule.  A property that holds at any size is
also checked at the 4B shape: two half-length runs chained through W_final equal
one full-length run (serial chunk updates compose, itsolotime §3.2).
"""
import functools

import numpy as np
import pytest
import torch

from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, run_layer
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu

TOL_BF16 = TOL["bf16"]
COL_BLOCK = 256


def rel(a, b, block=1 << 22):
    """Relative Frobenius error ||a - b|| / ||b||, accumulated in float64 block by block."""
    a = np.asarray(a).reshape(-1)
    b = np.asarray(b).reshape(-1)
    num = den = 0.0
    for i in range(0, b.size, block):
        x = a[i:i + block].astype(np.float64)
        y = b[i:i + block].astype(np.float64)
        num += float(np.sum((x - y) ** 2))
        den += float(np.sum(y * y))
    return (num / den) ** 0.5 if den > 0 else num ** 0.5


def piece_errors(O, Oref, L, B, d):
    """Relative error of every chunk of every sequence, and of every (chunk, column block)."""
    O = np.asarray(O).reshape(-1, B, d)
    Oref = np.asarray(Oref).reshape(-1, B, d)
    per_chunk = np.empty(O.shape[0])
    per_piece = []
    for i in range(O.shape[0]):
        diff = O[i].astype(np.float64) - Oref[i]
        per_chunk[i] = np.linalg.norm(diff) / np.linalg.norm(Oref[i])
        for c in range(0, d, COL_BLOCK):
            den = np.linalg.norm(Oref[i][:, c:c + COL_BLOCK])
            per_piece.append(np.linalg.norm(diff[:, c:c + COL_BLOCK]) / den if den > 0 else 0.0)
    return per_chunk, np.asarray(per_piece)


def check_all(name, O, Wf, Oref, Wref, W0, w):
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Wf)), name
    e_o = rel(O, Oref)
    chunks, pieces = piece_errors(O, Oref, w.L, w.B, w.d)
    e_w = rel(Wf, Wref)
    e_u = rel(np.asarray(Wf, np.float64) - W0, np.asarray(Wref, np.float64) - W0)
    msg = (f"{name}: O {e_o:.3g} (worst chunk {chunks.max():.3g} at {int(chunks.argmax())}, worst piece "
           f"{pieces.max():.3g}), W_final {e_w:.3g}, update {e_u:.3g}")
    print(msg)
    assert e_o <= TOL_BF16, msg
    assert chunks.max() <= TOL_BF16, msg
    assert pieces.max() <= TOL_BF16, msg
    assert e_w <= TOL_BF16, msg
    assert e_u <= TOL_BF16, msg


def _prefix(w, a, n, start=0):
    """Tokens start .. start+n-1 of every sequence of arrays `a`."""
    out = dict(a)
    for k in ("X", "E"):
        out[k] = np.ascontiguousarray(a[k].reshape(w.batch, w.L, -1)[:, start:start + n].reshape(w.batch * n, -1))
    return out


def _run(w, a, rule, **kw):
    return run_layer(w, a, rule, out_dtype=torch.float32, **kw)


def _full_case(w, rule, resume=False):
    a = inputs.generate(w, seed=0)
    O, Wf = _run(w, a, rule)
    Oref, Wref = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], w.L, w.B,
                                   w.eta, rule)
    check_all(f"{w.name} B={w.B} {rule}", O, Wf, Oref, Wref, a["W_o0"][None], w)
    del Oref, Wref
    if resume:
        h = (w.L // w.B // 2) * w.B
        O1, W1 = _run(w, _prefix(w, a, h), rule, L=h)
        O2, W2 = _run(w, _prefix(w, a, w.L - h, start=h), rule, L=w.L - h, W0=W1)
        Ocat = np.concatenate([O1.reshape(w.batch, h, w.d), O2.reshape(w.batch, w.L - h, w.d)], axis=1)
        assert rel(Ocat, O) <= TOL_BF16, "resume: O of two chained halves"
        assert rel(W2, Wf) <= TOL_BF16, "resume: W_final of two chained halves"
        assert rel(W2 - a["W_o0"][None], Wf - a["W_o0"][None]) <= TOL_BF16, "resume: update"


def test_4b_layer_full_size_mse():
    """d=2560, d_ff=9728, L=131072, B=1024, vocab 151936: the benchmarked workload, all 128 chunks."""
    _full_case(inputs.workload("4b"), "mse", resume=True)


def test_1p5b_layer_full_size_mse():
    """d=2048, d_ff=8192, L=32768, B=1024: all 32 chunks."""
    _full_case(inputs.workload("1p5b"), "mse")


def test_500m_layer_full_size_mse():
    """batch 8, L=4096, B=512, d=1024, d_ff=4096: every chunk of every sequence."""
    _full_case(inputs.workload("500m"), "mse")


# ---------------------------------------------------------- chunk-size sweep
@functools.lru_cache(maxsize=1)
def _sweep_inputs():
    w = inputs.workload("4b_sweep")
    a = inputs.generate(w, seed=0)
    Z = orc.gated_activation(a["X"], a["W_g"], a["W_u"])  # independent of B and of the rule
    return a, Z


@functools.lru_cache(maxsize=1)
def _sweep_targets(B):
    a, _ = _sweep_inputs()
    return orc.make_targets(a["E"], a["conv_w"], a["P"], B)


@functools.lru_cache(maxsize=2)
def _sweep_oracle(B, rule):
    a, Z = _sweep_inputs()
    w = inputs.workload("4b_sweep", B=B)
    return orc.chunk_engine(Z, _sweep_targets(B), a["W_o0"], B, w.eta, rule)


@pytest.mark.parametrize("B,rule", [(64, "mse"), (64, "add"), (256, "mse"), (256, "add"), (512, "mse"),
                                    (512, "add"), (1024, "mse"), (1024, "add"), (4096, "mse"), (4096, "add")])
def test_4b_chunk_sweep_full_size(B, rule):
    """L=32768 at the 4B shape: every chunk at every swept chunk size, both rules."""
    w = inputs.workload("4b_sweep", B=B)
    a, _ = _sweep_inputs()
    O, Wf = _run(w, a, rule)
    Oref, Wref = _sweep_oracle(B, rule)
    check_all(f"4b_sweep B={B} {rule}", O, Wf, Oref, Wref[None], a["W_o0"][None], w)


@pytest.mark.parametrize("B", [64, 256])
def test_blockcausal_full_sweep_size(B):
    """The additive rule in its block-causal form at L=32768, 4B shape, against the
    oracle's additive rule over every chunk."""
    w = inputs.workload("4b_sweep", B=B)
    a, _ = _sweep_inputs()
    O, Wf = _run(w, a, "add_blockcausal")
    Oref, Wref = _sweep_oracle(B, "add")
    check_all(f"4b_sweep B={B} add_blockcausal", O, Wf, Oref, Wref[None], a["W_o0"][None], w)
