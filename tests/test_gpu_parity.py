"""GPU parity: the CUDA path through the C-ABI against the float64 oracle on the
same seeded inputs.  Tolerance: relative Frobenius error <= 1e-2 (bf16
operands, fp32 accumulation) and <= 1e-4 (fp32 mode), on O, W_final and the
accumulated update W_final - W_o0."""
import numpy as np
import pytest
import torch

import chunked_weight_mlp_place_b300 as ip
from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, down, rel, run_layer, tdtype, up
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu


def _q(a, dtype):
    return inputs.round_to_bf16(a) if dtype == "bf16" else np.asarray(a, np.float32)


def _rand(rng, shape, scale, dtype):
    return _q((rng.standard_normal(shape) * scale).astype(np.float32), dtype)


def _check_engine(O, Wf, Oref, Wref, W0, tol):
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Wf))
    assert rel(O, Oref) <= tol, rel(O, Oref)
    assert rel(Wf, Wref) <= tol, rel(Wf, Wref)
    assert rel(Wf - W0, Wref - W0) <= tol, rel(Wf - W0, Wref - W0)


# ---------------------------------------------------------------- gate / targets
@pytest.mark.parametrize("dtype,T,d,d_ff", [("bf16", 300, 136, 264), ("bf16", 128, 64, 128),
                                            ("bf16", 1000, 512, 1024), ("fp32", 50, 37, 90),
                                            ("fp32", 256, 64, 256)])
def test_gate_up(dtype, T, d, d_ff):
    rng = np.random.default_rng(T + d)
    X = _rand(rng, (T, d), 1.0, dtype)
    Wg = _rand(rng, (d, d_ff), d ** -0.5, dtype)
    Wu = _rand(rng, (d, d_ff), d ** -0.5, dtype)
    dt = tdtype(dtype)
    Z = torch.empty(T, d_ff, dtype=dt, device="cuda")
    ip.gate_up(up(X, dt), up(Wg, dt), up(Wu, dt), Z)
    assert ip.sync_status() == 0
    ref = orc.gated_activation(X, Wg, Wu)
    assert rel(down(Z), ref) <= TOL[dtype], rel(down(Z), ref)


@pytest.mark.parametrize("dtype,batch,L,B,d", [("bf16", 2, 192, 64, 264), ("bf16", 1, 512, 16, 64),
                                               ("fp32", 2, 30, 5, 37), ("fp32", 1, 256, 64, 64)])
def test_make_targets(dtype, batch, L, B, d):
    rng = np.random.default_rng(L + d)
    E = _rand(rng, (batch * L, d), d ** -0.5, dtype)
    w = (rng.standard_normal((d, 4)) * 0.5 ** 0.5).astype(np.float32)
    P = _rand(rng, (d, d), d ** -0.5, dtype)
    dt = tdtype(dtype)
    V = torch.empty(batch * L, d, dtype=dt, device="cuda")
    ip.make_targets(up(E, dt), up(w, torch.float32), up(P, dt), V, L, B)
    assert ip.sync_status() == 0
    ref = np.concatenate([orc.make_targets(E[s * L:(s + 1) * L], w, P, B) for s in range(batch)])
    assert rel(down(V), ref) <= TOL[dtype], rel(down(V), ref)


def test_next_token_target_is_exact_on_gpu():
    """conv one-hot at tap 1 and P = I give V_t = E_{t+1}, zero at chunk ends:
    exact in bf16 (itsolotime §2.3 example)."""
    rng = np.random.default_rng(0)
    L, B, d = 256, 64, 64
    E = _rand(rng, (L, d), 1.0, "bf16")
    w = np.zeros((d, 4), np.float32)
    w[:, 1] = 1
    V = torch.empty(L, d, dtype=torch.bfloat16, device="cuda")
    ip.make_targets(up(E, torch.bfloat16), up(w, torch.float32), up(np.eye(d), torch.bfloat16), V, L, B)
    assert ip.sync_status() == 0
    ref = orc.make_targets(E, w, np.eye(d), B)
    np.testing.assert_array_equal(down(V), ref)


# ------------------------------------------------------------------- chunk engine
ENGINE_CASES = [
    # dtype, batch, L, B, d, d_ff, eta
    ("bf16", 1, 256, 64, 256, 256, 0.1),
    ("bf16", 2, 512, 64, 264, 200, 0.05),    # ragged d / d_ff tails, 2 sequences
    ("bf16", 1, 1024, 64, 128, 384, 0.05),   # K = 16 chunks: additive scan with groups of 2
    ("bf16", 1, 576, 64, 128, 128, 0.05),    # K = 9: additive groups of 3
    ("bf16", 1, 480, 16, 64, 128, 0.02),     # smallest chunk the tensor cores take
    ("bf16", 1, 256, 256, 256, 512, 0.1),    # one chunk (B = L)
    ("fp32", 1, 256, 64, 64, 256, 0.1),
    ("fp32", 2, 60, 5, 37, 90, 0.2),         # ragged everything
    ("fp32", 1, 112, 7, 16, 24, 0.1),        # K = 16 with B = 7
]


@pytest.mark.parametrize("rule", ["mse", "add"])
@pytest.mark.parametrize("case", ENGINE_CASES)
def test_chunk_engine(case, rule):
    dtype, batch, L, B, d, d_ff, eta = case
    rng = np.random.default_rng(L * 7 + d + d_ff)
    Z = _rand(rng, (batch * L, d_ff), 0.6, dtype)
    V = _rand(rng, (batch * L, d), 0.5, dtype)
    W0 = (rng.standard_normal((d_ff, d)) * d_ff ** -0.5).astype(np.float32)
    dt = tdtype(dtype)
    O = torch.empty(batch * L, d, dtype=dt, device="cuda")
    Wf = torch.empty(batch, d_ff, d, dtype=torch.float32, device="cuda")
    ip.chunk_forward(up(Z, dt), up(V, dt), up(W0, torch.float32), L, B, eta, rule, O, Wf)
    assert ip.sync_status() == 0
    Oref, Wref = [], []
    for s in range(batch):
        o, wr = orc.chunk_engine(Z[s * L:(s + 1) * L], V[s * L:(s + 1) * L], W0, B, eta, rule)
        Oref.append(o)
        Wref.append(wr)
    _check_engine(down(O), down(Wf), np.concatenate(Oref), np.stack(Wref), W0[None], TOL[dtype])


# -------------------------------------------------------------------- whole layer
def _oracle_layer(w, a, rule, L=None, W0=None, max_chunks=None):
    L = w.L if L is None else L
    return orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"] if W0 is None else W0, a["conv_w"],
                             a["P"], L, w.B, w.eta, rule, max_chunks=max_chunks)


@pytest.mark.parametrize("rule", ["mse", "add"])
def test_tiny_workload_fp32(rule):
    w = inputs.workload("tiny")
    a = inputs.generate(w, seed=0)
    O, Wf = run_layer(w, a, rule)
    Oref, Wref = _oracle_layer(w, a, rule)
    _check_engine(O, Wf, Oref, Wref, a["W_o0"][None], TOL["fp32"])


SMALL_BF16 = [
    inputs.workload("500m", batch=2, L=512, B=128, d=256, d_ff=1024),
    inputs.workload("4b", batch=1, L=1024, B=256, d=320, d_ff=1216, vocab=512),
]


@pytest.mark.parametrize("rule", ["mse", "add"])
@pytest.mark.parametrize("w", SMALL_BF16, ids=["500m-shape-small", "4b-ratio-small"])
def test_small_workloads_bf16(w, rule):
    a = inputs.generate(w, seed=0)
    O, Wf = run_layer(w, a, rule)
    Oref, Wref = _oracle_layer(w, a, rule)
    _check_engine(O, Wf, Oref, Wref, a["W_o0"][None], TOL["bf16"])


# ---------------------------------------------------------------------- edge cases
def test_eta_zero_is_the_gated_mlp_and_keeps_the_weight():
    w = inputs.workload("500m", batch=1, L=256, B=64, d=128, d_ff=256, eta=0.0)
    a = inputs.generate(w, seed=1)
    O, Wf = run_layer(w, a, "mse")
    Z = orc.gated_activation(a["X"], a["W_g"], a["W_u"])
    assert rel(O, Z @ a["W_o0"]) <= TOL["bf16"]
    np.testing.assert_array_equal(Wf[0], a["W_o0"].astype(np.float64))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_empty_sequence_copies_the_initial_weight(dtype):
    dt = tdtype(dtype)
    W0 = torch.randn(128, 64, device="cuda")
    Wf = torch.empty(2, 128, 64, device="cuda")
    X = torch.empty(0, 64, dtype=dt, device="cuda")
    ip.chunk_forward(torch.empty(0, 128, dtype=dt, device="cuda"), X, W0, 0, 64, 0.1, "mse", X, Wf)
    assert ip.sync_status() == 0
    assert torch.equal(Wf[0], W0) and torch.equal(Wf[1], W0)


@pytest.mark.parametrize("rule", ["mse", "add"])
def test_resume_from_w_final_matches_one_pass(rule):
    """forward(L) == forward(first half) then forward(second half) from W_final
    (per-sequence initial weights), and matches the oracle."""
    w = inputs.workload("500m", batch=2, L=512, B=64, d=128, d_ff=256)
    a = inputs.generate(w, seed=2)
    O, Wf = run_layer(w, a, rule)
    h = w.L // 2
    first = {k: (v.reshape(2, w.L, -1)[:, :h].reshape(2 * h, -1) if k in ("X", "E") else v) for k, v in a.items()}
    second = {k: (v.reshape(2, w.L, -1)[:, h:].reshape(2 * h, -1) if k in ("X", "E") else v) for k, v in a.items()}
    O1, W1 = run_layer(w, first, rule, L=h)
    O2, W2 = run_layer(w, second, rule, L=h, W0=W1.astype(np.float32))
    Ocat = np.concatenate([O1.reshape(2, h, -1), O2.reshape(2, h, -1)], axis=1).reshape(O.shape)
    assert rel(Ocat, O) <= 1e-3 and rel(W2, Wf) <= 1e-4
    Oref, Wref = _oracle_layer(w, a, rule)
    _check_engine(Ocat, W2, Oref, Wref, a["W_o0"][None], TOL["bf16"])


def test_causality_on_gpu():
    """Changing X or E in later chunks leaves earlier outputs unchanged."""
    w = inputs.workload("500m", batch=1, L=512, B=128, d=128, d_ff=256)
    a = inputs.generate(w, seed=3)
    O, _ = run_layer(w, a, "mse")
    b = dict(a)
    b["X"] = a["X"].copy()
    b["E"] = a["E"].copy()
    b["X"][256:] = inputs.round_to_bf16(b["X"][256:] * 2)
    b["E"][128:] = inputs.round_to_bf16(b["E"][128:] * -3)
    O2, _ = run_layer(w, b, "mse")
    assert rel(O2[:256], O[:256]) <= 1e-3  # fp32 atomics may reorder; nothing else differs
    assert rel(O2[256:], O[256:]) > 1e-2


def test_launch_count_and_no_host_fallback():
    w = inputs.workload("500m", batch=1, L=256, B=64, d=128, d_ff=256)
    a = inputs.generate(w, seed=4)
    run_layer(w, a, "mse")
    # gate + conv + proj + split of W_o0 + K * (apply + residual + update) + merge into W_final
    assert ip.last_launch_count() == 3 + 1 + 3 * (w.L // w.B) + 1


@pytest.mark.parametrize("rule", ["mse", "add"])
@pytest.mark.parametrize("shape", [(1024, 64, 128, 384), (576, 64, 128, 128), (1024, 256, 320, 1216)])
def test_repeated_runs_stay_within_tolerance(shape, rule):
    """Every one of several back-to-back runs matches the oracle.  Guards the
    cross-CTA split-K reductions and the shared-memory slot reuse of the update
    epilogue, whose ordering faults showed up only in some runs."""
    L, B, d, d_ff = shape
    rng = np.random.default_rng(11)
    Z = _rand(rng, (L, d_ff), 0.6, "bf16")
    V = _rand(rng, (L, d), 0.5, "bf16")
    W0 = (rng.standard_normal((d_ff, d)) * d_ff ** -0.5).astype(np.float32)
    Oref, Wref = orc.chunk_engine(Z, V, W0, B, 0.05, rule)
    Zt, Vt, W0t = up(Z, torch.bfloat16), up(V, torch.bfloat16), up(W0, torch.float32)
    for _ in range(8):
        O = torch.empty(L, d, dtype=torch.bfloat16, device="cuda")
        Wf = torch.empty(1, d_ff, d, dtype=torch.float32, device="cuda")
        ip.chunk_forward(Zt, Vt, W0t, L, B, 0.05, rule, O, Wf)
        assert ip.sync_status() == 0
        _check_engine(down(O), down(Wf), Oref, Wref[None], W0[None], TOL["bf16"])


def test_pool_limit_refuses_a_call_before_queuing_anything():
    w = inputs.workload("500m", batch=1, L=256, B=64, d=128, d_ff=256)
    a = inputs.generate(w, seed=12)
    ip.set_pool_limit(4096)
    try:
        with pytest.raises(ip.IptttError) as e:
            run_layer(w, a, "mse")
        assert e.value.status == ip._lib.ERR_ALLOC
        assert ip.last_launch_count() == 0
    finally:
        ip.set_pool_limit(0)
    O, Wf = run_layer(w, a, "mse")
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Wf))
