"""Seeded input generator: determinism, partial draws and bf16 rounding (CPU)."""
import numpy as np
import torch

from chunked_weight_mlp_place_b300 import inputs


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        np.array([1.0, -1.0, 0.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -9], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(inputs.round_to_bf16(x), ref)


def test_generation_is_deterministic_and_prefix_consistent():
    w = inputs.workload("500m", batch=2, L=256, B=64, d=64, d_ff=128)
    a = inputs.generate(w, seed=3)
    b = inputs.generate(w, seed=3)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    p = inputs.generate(w, seed=3, n_tokens=100)
    np.testing.assert_array_equal(p["X"], a["X"][:100])
    np.testing.assert_array_equal(p["E"], a["E"][:100])
    np.testing.assert_array_equal(p["W_g"], a["W_g"])
    c = inputs.generate(w, seed=4)
    assert not np.array_equal(c["X"], a["X"])


def test_shapes_distributions_and_representability():
    w = inputs.workload("500m", batch=2, L=512, B=64, d=128, d_ff=256)
    a = inputs.generate(w)
    assert a["X"].shape == (1024, 128) and a["E"].shape == (1024, 128)
    assert a["W_g"].shape == (128, 256) and a["W_o0"].shape == (256, 128)
    assert a["conv_w"].shape == (128, 4) and a["P"].shape == (128, 128)
    # RMS-normalised tokens
    np.testing.assert_allclose(np.sqrt(np.mean(a["X"].astype(np.float64) ** 2, axis=1)), 1.0, rtol=1e-2)
    # variances of the weights (second argument of N is the variance)
    assert abs(a["W_g"].var() * 128 - 1) < 0.05
    assert abs(a["W_o0"].var() * 256 - 1) < 0.05
    assert abs(a["conv_w"].var() / 0.5 - 1) < 0.2
    # bf16 activations and projection are exactly representable; fp32 fast weight is not rounded
    for k in ("X", "E", "W_g", "W_u", "P"):
        np.testing.assert_array_equal(inputs.round_to_bf16(a[k]), a[k])
    assert not np.array_equal(inputs.round_to_bf16(a["W_o0"]), a["W_o0"])
    # E is the embedding-table gather of the ids
    assert a["ids"].min() >= 0 and a["ids"].max() < w.vocab


def test_doc_boundaries_are_seeded_rising_and_cover_the_tokens():
    for mix, (lo, hi) in inputs.DOC_MIXES.items():
        cu = inputs.doc_boundaries(50000, seed=3, mix=mix)
        np.testing.assert_array_equal(cu, inputs.doc_boundaries(50000, seed=3, mix=mix))
        assert cu[0] == 0 and cu[-1] == 50000 and cu.dtype == np.int64
        lens = np.diff(cu)
        assert np.all(lens >= 1)
        assert np.all(lens[:-1] >= lo) and np.all(lens <= hi + 1)   # the last one is cut to fit
        assert not np.array_equal(cu, inputs.doc_boundaries(50000, seed=4, mix=mix))
    # the document stream was appended: X still comes from the third of the
    # original eight spawned streams
    w = inputs.workload("tiny")
    a = inputs.generate(w, seed=0, want=("X",))
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(0).spawn(8)[2]))
    X = g.standard_normal(size=(w.L, w.d), dtype=np.float32)
    X = (X / np.sqrt(np.mean(np.square(X, dtype=np.float64), axis=1, keepdims=True) + 1e-6)).astype(np.float32)
    np.testing.assert_array_equal(a["X"], X)
