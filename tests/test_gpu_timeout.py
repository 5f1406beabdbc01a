"""Failure detection on the GPU without a fault: the pipeline waits of the
tensor-core kernels are capped, and a wait that runs past its limit is reported
as IPTTT_ERR_TIMEOUT by ipttt_sync_status, with the kernel ending cleanly and
the context left usable.

Nothing is withheld and no kernel is broken: the soft limit is set below the
length of the waits a normal call makes (ipttt_set_wait_limit, a few hundred
nanoseconds), so the detection fires on waits that would have completed.  The
CTAs that see it stop issuing MMAs and writing results but complete their
handshakes, so every copy and MMA in flight finishes before they exit.  After
the default is restored the next call is checked against the oracle."""
import numpy as np
import pytest
import torch

import chunked_weight_mlp_place_b300 as ip
from chunked_weight_mlp_place_b300 import inputs
from gpu_util import TOL, down, rel, up
from oracle import ipttt_oracle as orc

pytestmark = pytest.mark.gpu


def _engine_case(B, L):
    rng = np.random.default_rng(7)
    d, d_ff = 512, 1024
    Z = inputs.round_to_bf16((rng.standard_normal((L, d_ff)) * 0.6).astype(np.float32))
    V = inputs.round_to_bf16((rng.standard_normal((L, d)) * 0.5).astype(np.float32))
    W0 = (rng.standard_normal((d_ff, d)) * d_ff ** -0.5).astype(np.float32)
    return L, B, Z, V, W0


def _run(L, B, Z, V, W0, rule):
    O = torch.empty(L, V.shape[1], dtype=torch.bfloat16, device="cuda")
    Wf = torch.empty(1, Z.shape[1], V.shape[1], device="cuda")
    ip.chunk_forward(up(Z, torch.bfloat16), up(V, torch.bfloat16), up(W0, torch.float32), L, B, 0.05, rule, O, Wf)
    return O, Wf


@pytest.mark.parametrize("rule,B,L", [("mse", 128, 1152), ("add", 128, 1024), ("mse", 256, 768), ("mse", 64, 1024)])
def test_a_wait_past_the_limit_is_reported_and_the_next_call_is_exact(rule, B, L):
    """MSE with 9 chunks of 128 (no window fits) and the additive rule: the per-chunk
    GEMM kernels; MSE with 3 chunks of 256: the persistent chunk engine on chunks (its
    waits on other CTAs' counters included); MSE with chunks of 64: windows of 1024
    tokens (the window GEMMs, then the engine on windows)."""
    L, B, Z, V, W0 = _engine_case(B, L)
    assert ip.sync_status() == ip._lib.OK
    ip.set_wait_limit(200)  # ns: far below the waits of a real pipeline
    try:
        _run(L, B, Z, V, W0, rule)
        status = ip.sync_status()
    finally:
        ip.set_wait_limit(0)
    assert status == ip._lib.ERR_TIMEOUT, ip.status_string(status)
    assert ip.sync_status() == ip._lib.OK  # the word was cleared by the read; the context works
    O, Wf = _run(L, B, Z, V, W0, rule)
    assert ip.sync_status() == ip._lib.OK
    Oref, Wref = orc.chunk_engine(Z, V, W0, B, 0.05, rule)
    assert rel(down(O), Oref) <= TOL["bf16"]
    assert rel(down(Wf)[0], Wref) <= TOL["bf16"]
    assert rel(down(Wf)[0] - W0, Wref - W0) <= TOL["bf16"]


def test_the_default_limit_reports_nothing_on_a_whole_layer():
    w = inputs.workload("500m", batch=1, L=1024, B=256, d=512, d_ff=1024)
    a = inputs.generate(w, seed=3)
    dt = torch.bfloat16
    O = torch.empty(w.L, w.d, dtype=dt, device="cuda")
    Wf = torch.empty(1, w.d_ff, w.d, device="cuda")
    ip.layer_forward(up(a["X"], dt), up(a["E"], dt), up(a["W_g"], dt), up(a["W_u"], dt),
                     up(a["W_o0"], torch.float32), up(a["conv_w"], torch.float32), up(a["P"], dt), w.L, w.B, w.eta,
                     "mse", O, Wf)
    assert ip.sync_status() == ip._lib.OK
