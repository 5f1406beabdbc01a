"""GPU parity at the workloads' full sizes.

The layer runs through ipttt_layer_forward at each workload's full shape (the
4B-scale one is exactly the launch configuration the benchmark times).  The
float64 oracle cannot follow a 128k-token sequence chunk by chunk in seconds,
so the check is split in two:

* sampled outputs the oracle computes directly: the leading chunks of O (the
  oracle runs the same chunks of the same seeded inputs), and the fast weight
  after those chunks (a GPU run over that prefix, with the same per-chunk
  kernels and tile shapes as the full run);
* properties that hold at any size, between GPU runs: the full run's leading
  chunks equal the prefix run's, and two half-length runs chained through
  W_final equal one full-length run (serial chunk updates compose, itsolotime
  §3.2).

Tolerances are the ones the layer is specified to: relative Frobenius error
<= 1e-2 in bf16 mode on O, W_final and the accumulated update W_final - W_o0.
"""
import numpy as np
import pytest
import torch

from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, run_layer
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu


def _prefix(w, a, n, start=0):
    """Tokens start .. start+n-1 of every sequence of arrays `a`."""
    out = dict(a)
    for k in ("X", "E"):
        out[k] = np.ascontiguousarray(a[k].reshape(w.batch, w.L, -1)[:, start:start + n].reshape(w.batch * n, -1))
    return out


def _oracle(w, a, rule, n_chunks, seqs=None):
    """Oracle O (leading n_chunks of each listed sequence) and the fast weight after them."""
    seqs = range(w.batch) if seqs is None else seqs
    O, W = [], []
    for s in seqs:
        rows = slice(s * w.L, s * w.L + n_chunks * w.B)
        o, wf = orc.layer_forward(a["X"][rows], a["E"][rows], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"],
                                  n_chunks * w.B, w.B, w.eta, rule)
        O.append(o)
        W.append(wf[0])
    return O, W


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


def _run(w, a, rule, **kw):
    return run_layer(w, a, rule, out_dtype=torch.float32, **kw)


def _check(name, got, ref, W0=None):
    e = rel(got, ref)
    assert np.all(np.isfinite(got)), name
    assert e <= TOL["bf16"], f"{name}: rel err {e:.3g}"
    if W0 is not None:
        eu = rel(np.asarray(got, np.float64) - W0, np.asarray(ref, np.float64) - W0)
        assert eu <= TOL["bf16"], f"{name} update: rel err {eu:.3g}"


def _full_size_case(w, rule, n_chunks, seqs=None, resume=True):
    a = inputs.generate(w, seed=0)
    seqs = list(range(w.batch)) if seqs is None else seqs
    O, Wf = _run(w, a, rule)                           # the full-size run
    O = O.reshape(w.batch, w.L, w.d)
    n = n_chunks * w.B
    Oref, Wref = _oracle(w, a, rule, n_chunks, seqs)
    for s, o_ref in zip(seqs, Oref):
        _check(f"O leading {n_chunks} chunks, sequence {s}", O[s, :n], o_ref)
    # fast weight after the leading chunks: a prefix run, same kernels per chunk
    Op, Wp = _run(w, _prefix(w, a, n), rule, L=n)
    Op = Op.reshape(w.batch, n, w.d)
    for s, w_ref in zip(seqs, Wref):
        _check(f"W after {n_chunks} chunks, sequence {s}", Wp[s], w_ref, a["W_o0"])
    # property: the full run's leading chunks are the prefix run's
    _check("prefix consistency", O[:, :n], Op)
    if resume and w.L // w.B >= 2:
        h = (w.L // w.B // 2) * w.B
        O1, W1 = _run(w, _prefix(w, a, h), rule, L=h)
        O2, W2 = _run(w, _prefix(w, a, w.L - h, start=h), rule, L=w.L - h, W0=W1)
        Ocat = np.concatenate([O1.reshape(w.batch, h, w.d), O2.reshape(w.batch, w.L - h, w.d)], axis=1)
        del O1, O2
        _check("resume: O of two chained halves", Ocat, O)
        _check("resume: W_final of two chained halves", W2, Wf, a["W_o0"][None])


def test_4b_layer_full_size_mse():
    """d=2560, d_ff=9728, L=131072, B=1024, vocab 151936: the benchmarked workload."""
    _full_size_case(inputs.workload("4b"), "mse", n_chunks=4)


def test_1p5b_layer_full_size_mse():
    _full_size_case(inputs.workload("1p5b"), "mse", n_chunks=4)


def test_500m_layer_full_size_mse():
    """batch 8: every chunk of the first and last sequence against the oracle."""
    w = inputs.workload("500m")
    _full_size_case(w, "mse", n_chunks=w.L // w.B, seqs=[0, w.batch - 1], resume=False)


@pytest.mark.parametrize("B,rule,n_chunks", [(64, "mse", 16), (64, "add", 16), (1024, "add", 4),
                                             (4096, "mse", 2), (4096, "add", 2)])
def test_4b_chunk_sweep_full_size(B, rule, n_chunks):
    """L=32768 at the 4B shape, the chunk-size / rule sweep points at both ends."""
    _full_size_case(inputs.workload("4b_sweep", B=B), rule, n_chunks=n_chunks)
