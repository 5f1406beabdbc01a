"""The benchmark's roofline arithmetic on CPU: the work it charges per launch
adds up to the layer's algorithmic FLOPs and weight bytes, and the layer's
roofline at the 4B workload is the one derived by hand from the measured peaks."""
import importlib.util
import os

import numpy as np
import pytest

from chunked_weight_mlp_place_b300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(spec)
spec.loader.exec_module(bench)


def test_per_launch_work_adds_up_to_the_layer():
    w = inputs.workload("4b")
    T, K = w.batch * w.L, w.L // w.B
    launches = {"gate_up": 1, "proj": 1, "apply": K, "update": K}
    total = sum(bench.kernel_work(w, k)[0] * n for k, n in launches.items())
    # 4 d d_ff (gate+up) + 2 d d_ff (apply) + 2 d d_ff (update) + 2 d^2 (proj) per token
    assert total == pytest.approx((8 * w.d * w.d_ff + 2 * w.d * w.d) * T, rel=1e-12)
    assert bench.kernel_work(w, "update")[1] * K == pytest.approx(K * 2 * w.d_ff * w.d * 4, rel=1e-12)
    # the persistent engine: the apply and update of every chunk in its one launch
    launches = {"gate_up": 1, "proj": 1, "engine": 1}
    total = sum(bench.kernel_work(w, k)[0] * n for k, n in launches.items())
    assert total == pytest.approx((8 * w.d * w.d_ff + 2 * w.d * w.d) * T, rel=1e-12)
    assert bench.kernel_work(w, "engine")[1] == pytest.approx(K * 2 * w.d_ff * w.d * 4, rel=1e-12)


def test_layer_roofline_at_the_4b_workload():
    peaks = {"bf16_tflops": 1785.8, "hbm_gbs": 6493.7}
    tps, bound = bench.roofline_tokens_per_s(inputs.workload("4b"), peaks)
    # 27.8 TFLOP at 1785.8 TFLOP/s = 15.6 ms > 25.5 GB of W traffic at 6493.7 GB/s = 3.9 ms
    assert bound == "tensor"
    assert tps == pytest.approx(131072 / (212.3e6 * 131072 / 1785.8e12), rel=2e-3)
    w64 = inputs.workload("4b_sweep", B=64)
    tps64, bound64 = bench.roofline_tokens_per_s(w64, peaks)
    assert bound64 == "hbm"
    assert tps64 == pytest.approx(32768 / (512 * 2 * 9728 * 2560 * 4 / 6493.7e9), rel=1e-9)


def test_packed_documents_count_each_documents_chunks():
    w = inputs.workload("4b_sweep", B=1024)
    cu = np.array([0, 1000, 1024, 5000, 32768])
    n = bench.chunk_counts(w, cu)
    np.testing.assert_array_equal(n, [1, 1, 4, 28])  # 1000, 24, 3976, 27768 tokens
    fl, by = bench.kernel_work(w, "update", cu)
    assert by * n.max() == pytest.approx(n.sum() * 2 * w.d_ff * w.d * 4, rel=1e-12)
    assert fl * n.max() == pytest.approx(2 * w.d * w.d_ff * w.L, rel=1e-12)


def test_several_layers_and_the_block_causal_form():
    w = inputs.workload("4b_sweep", B=64)
    assert bench.kernel_work(w, "gate_up", layers=8)[0] == 8 * bench.kernel_work(w, "gate_up")[0]
    K = w.L // w.B
    pairs = w.B * w.B * K * (K - 1) / 2  # kept (query, key) pairs: keys of earlier chunks only
    assert pairs == pytest.approx(sum(q * w.B * w.B for q in range(K)), rel=1e-12)
    assert bench.kernel_work(w, "scores", rule="add_blockcausal")[0] == pytest.approx(2 * w.d_ff * pairs)


def test_windowed_form_accounting():
    """Chunks below 1024 tokens run in windows (the MSE rule, bf16): the engine then moves
    the fast weight once per window, and the window GEMMs add FLOPs counted here by brute
    force over the chunk pairs of a window."""
    for B, W in [(64, 1024), (128, 1024), (256, 1024), (512, 1024), (1024, 0), (4096, 0)]:
        assert bench.window_tokens(inputs.workload("4b_sweep", B=B)) == W
    assert bench.window_tokens(inputs.workload("4b_sweep", B=64), rule="add") == 0
    assert bench.window_tokens(inputs.workload("4b", L=1536, B=128)) == 768
    assert bench.window_tokens(inputs.workload("500m")) == 0  # d = 1024, two chunks a window: not taken
    assert bench.window_tokens(inputs.workload("500m", B=256)) == 1024
    w = inputs.workload("4b_sweep", B=64)
    W, B = 1024, 64
    nwin = w.L // W
    assert bench.kernel_work(w, "engine")[1] == pytest.approx(nwin * 2 * w.d_ff * w.d * 4, rel=1e-12)
    m = W // B
    gram = sum(2 * w.d_ff * B * B for j in range(m) for i in range(j))  # chunk i < chunk j
    inv = sum(2 * B * (j * B) * (j * B) for j in range(1, m))  # row block j: B x jB times jB x jB
    per_window = gram + inv + 2 * W * W * w.d_ff + 2 * W * W * w.d
    assert bench.kernel_work(w, "window")[0] == pytest.approx(nwin * per_window, rel=1e-12)
