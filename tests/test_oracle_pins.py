"""Pins of the float64 oracle to things other than itself (CPU only).

Each test ties one oracle function to a hand-worked example, a library routine,
finite differences, an independent brute force, a closed form, or one of the
special cases the In-Place TTT pages spell out.  A plausible slip in the oracle
(a dropped term, a wrong sign, index or scale, a transposed operand, the update
applied before the output) fails at least one of them.
"""
import numpy as np
import pytest
import scipy.special
import torch

from conftest import load_golden, rel_err
from oracle import ipttt_oracle as orc
from chunked_weight_mlp_place_b300 import inputs


def _tiny(seed=1, L=24, B=6, d=5, d_ff=7, batch=1):
    rng = np.random.default_rng(seed)
    return dict(
        X=rng.standard_normal((batch * L, d)),
        E=rng.standard_normal((batch * L, d)),
        W_g=rng.standard_normal((d, d_ff)) / np.sqrt(d),
        W_u=rng.standard_normal((d, d_ff)) / np.sqrt(d),
        W_o0=rng.standard_normal((d_ff, d)) / np.sqrt(d_ff),
        conv_w=rng.standard_normal((d, 4)) * np.sqrt(0.5),
        P=rng.standard_normal((d, d)) / np.sqrt(d),
        L=L, B=B,
    )


# ---------------------------------------------------------------- hand-worked
@pytest.mark.parametrize("name", ["chunk_engine_d1.txt", "chunk_engine_d2.txt"])
@pytest.mark.parametrize("rule", ["mse", "add"])
def test_golden_chunk_engine(name, rule):
    g = load_golden(name)
    O, W = orc.chunk_engine(g["Z"], g["V"], g["W0"], int(g["B"]), g["eta"], rule)
    np.testing.assert_array_equal(O, g[f"{rule}_O"])
    np.testing.assert_array_equal(W, g[f"{rule}_W"])


def test_golden_targets():
    g = load_golden("targets_conv_proj.txt")
    B = int(g["B"])
    np.testing.assert_array_equal(orc.chunk_conv(g["E"], g["conv_w"], B), g["C"])
    np.testing.assert_array_equal(orc.make_targets(g["E"], g["conv_w"], g["P"], B), g["V"])


# ------------------------------------------------------------ library routines
def test_silu_matches_expit():
    a = np.concatenate([np.linspace(-40, 40, 2001), [-800.0, -100.0, 0.0, 100.0, 800.0]])
    np.testing.assert_allclose(orc.silu(a), a * scipy.special.expit(a), rtol=1e-14, atol=1e-300)
    assert np.all(np.isfinite(orc.silu(a)))


def test_gated_activation_matches_torch():
    t = _tiny()
    Z = orc.gated_activation(t["X"], t["W_g"], t["W_u"])
    X = torch.from_numpy(t["X"])
    ref = torch.nn.functional.silu(X @ torch.from_numpy(t["W_g"])) * (X @ torch.from_numpy(t["W_u"]))
    np.testing.assert_allclose(Z, ref.numpy(), rtol=1e-13, atol=1e-14)


def test_conv_matches_numpy_correlate_per_chunk():
    rng = np.random.default_rng(3)
    L, B, d = 40, 8, 3
    E = rng.standard_normal((L, d))
    w = rng.standard_normal((d, 4))
    C = orc.chunk_conv(E, w, B)
    for c in range(d):
        for k in range(L // B):
            e = np.concatenate([E[k * B:(k + 1) * B, c], np.zeros(3)])  # zeros past the chunk end
            ref = np.correlate(e, w[c], mode="valid")  # sum_j w[j] e[t+j]
            np.testing.assert_allclose(C[k * B:(k + 1) * B, c], ref, rtol=1e-13, atol=1e-14)


def test_mse_update_matches_autograd():
    """One chunk step equals W - eta * grad of ||ZW - V||^2/(2B) from torch autograd."""
    rng = np.random.default_rng(4)
    B, d_ff, d, eta = 9, 6, 4, 0.3
    Z, V, W = rng.standard_normal((B, d_ff)), rng.standard_normal((B, d)), rng.standard_normal((d_ff, d))
    Wt = torch.tensor(W, requires_grad=True)
    loss = ((torch.from_numpy(Z) @ Wt - torch.from_numpy(V)) ** 2).sum() / (2 * B)
    loss.backward()
    O, W1 = orc.chunk_step(Z, V, W, eta, "mse")
    np.testing.assert_allclose(W1, W - eta * Wt.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(O, Z @ W, rtol=1e-13)


def test_additive_update_matches_autograd_of_similarity_loss():
    rng = np.random.default_rng(5)
    B, d_ff, d, eta = 7, 5, 3, 0.2
    Z, V, W = rng.standard_normal((B, d_ff)), rng.standard_normal((B, d)), rng.standard_normal((d_ff, d))
    Wt = torch.tensor(W, requires_grad=True)
    loss = -(torch.from_numpy(Z) @ Wt * torch.from_numpy(V)).sum() / B
    loss.backward()
    _, W1 = orc.chunk_step(Z, V, W, eta, "add")
    np.testing.assert_allclose(W1, W - eta * Wt.grad.numpy(), rtol=1e-12, atol=1e-14)


# --------------------------------------------------------- finite differences
def test_mse_gradient_finite_differences():
    rng = np.random.default_rng(6)
    B, d_ff, d, eta = 16, 12, 10, 0.05
    Z, V, W = rng.standard_normal((B, d_ff)), rng.standard_normal((B, d)), rng.standard_normal((d_ff, d))
    _, W1 = orc.chunk_step(Z, V, W, eta, "mse")
    grad = (W - W1) / eta
    h = 1e-5
    picks = rng.choice(d_ff * d, size=32, replace=False)
    for p in picks:
        i, j = divmod(int(p), d)
        Wp, Wm = W.copy(), W.copy()
        Wp[i, j] += h
        Wm[i, j] -= h
        fd = (orc.mse_loss(Z, V, Wp) - orc.mse_loss(Z, V, Wm)) / (2 * h)
        assert abs(fd - grad[i, j]) <= 1e-6 * max(1.0, abs(grad[i, j])), (i, j, fd, grad[i, j])


# -------------------------------------------------------------- brute force
def _brute_force(Z, V, W0, B, eta, rule):
    """Pure-Python per-token loops, accumulating each token's gradient and
    applying the sum, over the chunk's token count, at the end of its chunk
    (B=1: one update per token; a short last chunk averages its own tokens)."""
    Z, V = Z.tolist(), V.tolist()
    W = [list(r) for r in W0.tolist()]
    d_ff, d = len(W), len(W[0])
    O = []
    for c0 in range(0, len(Z), B):
        G = [[0.0] * d for _ in range(d_ff)]
        n = min(B, len(Z) - c0)
        for t in range(c0, c0 + n):
            o = [sum(Z[t][i] * W[i][j] for i in range(d_ff)) for j in range(d)]
            O.append(o)
            e = [o[j] - V[t][j] for j in range(d)] if rule == "mse" else [-V[t][j] for j in range(d)]
            for i in range(d_ff):
                for j in range(d):
                    G[i][j] += Z[t][i] * e[j]
        for i in range(d_ff):
            for j in range(d):
                W[i][j] -= eta / n * G[i][j]
    return np.array(O), np.array(W)


@pytest.mark.parametrize("B", [1, 3, 4])
@pytest.mark.parametrize("rule", ["mse", "add"])
def test_chunk_engine_matches_brute_force(B, rule):
    rng = np.random.default_rng(7 + B)
    L, d_ff, d, eta = 12, 5, 3, 0.3
    Z, V, W0 = rng.standard_normal((L, d_ff)), rng.standard_normal((L, d)), rng.standard_normal((d_ff, d))
    O, W = orc.chunk_engine(Z, V, W0, B, eta, rule)
    Ob, Wb = _brute_force(Z, V, W0, B, eta, rule)
    np.testing.assert_allclose(O, Ob, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(W, Wb, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------- closed forms
def test_additive_closed_form_and_block_causal_form():
    """W_k = W_0 + (eta/B) Z_{<k}^T V_{<k}, O_k = Z_k W_0 + (eta/B) (Z_k Z_{<k}^T) V_{<k}."""
    rng = np.random.default_rng(8)
    L, B, d_ff, d, eta = 40, 8, 6, 4, 0.1
    Z, V, W0 = rng.standard_normal((L, d_ff)), rng.standard_normal((L, d)), rng.standard_normal((d_ff, d))
    O, W = orc.chunk_engine(Z, V, W0, B, eta, "add")
    np.testing.assert_allclose(W, W0 + eta / B * Z.T @ V, rtol=1e-12, atol=1e-12)
    for k in range(L // B):
        s = slice(k * B, (k + 1) * B)
        p = slice(0, k * B)
        ref = Z[s] @ W0 + eta / B * (Z[s] @ Z[p].T) @ V[p]
        np.testing.assert_allclose(O[s], ref, rtol=1e-12, atol=1e-12)
        _, Wk = orc.chunk_engine(Z[:k * B], V[:k * B], W0, B, eta, "add") if k else (None, W0)
        np.testing.assert_allclose(Wk, W0 + eta / B * Z[p].T @ V[p], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("B,m", [(4, 6), (8, 2), (1, 5)])
def test_mse_loop_equals_its_window_solve(B, m):
    """The MSE rule over m consecutive chunks from the window's start weight W_k, restated as one
    solve: with alpha = -eta/B, A = alpha mask(Z Z^T) (token pairs in different chunks, the later
    row), Y = Z W_k - V and X = (I - A)^-1, the window's residuals are R = X Y, its outputs O = R + V
    and the next weight W_k + alpha (X^T Z)^T Y.  X is built row block by row block as
    X_j = e_j + A_{j,<j} X_{<j} and checked against a dense inverse.  Equal to the oracle's chunk
    loop up to float64 rounding (the same identity the GPU's windowed form computes in bf16)."""
    rng = np.random.default_rng(9 + B)
    W, d_ff, d, eta = B * m, 7, 5, 0.3
    nwin = 3
    L = W * nwin
    Z, V, W0 = rng.standard_normal((L, d_ff)) * 0.5, rng.standard_normal((L, d)), rng.standard_normal((d_ff, d))
    O_ref, W_ref = orc.chunk_engine(Z, V, W0, B, eta, "mse")
    alpha = -eta / B
    chunk = np.arange(W) // B
    later = chunk[:, None] > chunk[None, :]
    Wk = W0.copy()
    O = np.zeros_like(V)
    for w in range(nwin):
        s = slice(w * W, (w + 1) * W)
        Zw, Vw = Z[s], V[s]
        A = alpha * (Zw @ Zw.T) * later
        X = np.eye(W)
        for j in range(1, m):
            r = slice(j * B, (j + 1) * B)
            X[r, :j * B] = A[r, :j * B] @ X[:j * B, :j * B]
        np.testing.assert_allclose(X, np.linalg.inv(np.eye(W) - A), rtol=1e-10, atol=1e-12)
        Y = Zw @ Wk - Vw
        O[s] = X @ Y + Vw
        Wk = Wk + alpha * (X.T @ Zw).T @ Y
    np.testing.assert_allclose(O, O_ref, rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(Wk, W_ref, rtol=1e-9, atol=1e-10)


def test_eta_zero_is_the_plain_gated_mlp():
    t = _tiny(batch=2)
    O, W = orc.layer_forward(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"],
                             t["L"], t["B"], 0.0, "mse")
    X = torch.from_numpy(t["X"])
    mlp = (torch.nn.functional.silu(X @ torch.from_numpy(t["W_g"])) * (X @ torch.from_numpy(t["W_u"]))) \
        @ torch.from_numpy(t["W_o0"])
    np.testing.assert_allclose(O, mlp.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(W, np.stack([t["W_o0"]] * 2))


def test_first_chunk_and_single_chunk_use_the_initial_weight():
    """O_0 = Z_0 W_0 always; with B = L the final weight is one step from W_0."""
    t = _tiny(L=12, B=12)
    O, W = orc.layer_forward(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"],
                             12, 12, 0.2, "mse")
    Z = orc.gated_activation(t["X"], t["W_g"], t["W_u"])
    V = orc.make_targets(t["E"], t["conv_w"], t["P"], 12)
    np.testing.assert_allclose(O, Z @ t["W_o0"], rtol=1e-12, atol=1e-13)
    Wt = torch.tensor(t["W_o0"], requires_grad=True)
    (((torch.from_numpy(Z) @ Wt - torch.from_numpy(V)) ** 2).sum() / 24).backward()
    np.testing.assert_allclose(W[0], t["W_o0"] - 0.2 * Wt.grad.numpy(), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------ the pages' special cases
def test_next_token_target():
    """One-hot conv at the next position and P = I give V_t = E_{t+1}, and zero
    on each chunk's last row because of the chunk-end padding (itsolotime §2.3)."""
    rng = np.random.default_rng(9)
    L, B, d = 20, 5, 4
    E = rng.standard_normal((L, d))
    w = np.zeros((d, 4))
    w[:, 1] = 1.0
    V = orc.make_targets(E, w, np.eye(d), B)
    for t in range(L):
        if (t + 1) % B == 0:
            np.testing.assert_array_equal(V[t], 0.0)
        else:
            np.testing.assert_array_equal(V[t], E[t + 1])


def test_no_conv_no_proj_target_is_the_embedding():
    """The ablation without conv and projection (tap 0 only, P = I) gives V = E."""
    rng = np.random.default_rng(10)
    E = rng.standard_normal((16, 3))
    w = np.zeros((3, 4))
    w[:, 0] = 1.0
    np.testing.assert_array_equal(orc.make_targets(E, w, np.eye(3), 4), E)


# ------------------------------------------------------------------ invariants
@pytest.mark.parametrize("rule", ["mse", "add"])
def test_causality_future_tokens_do_not_reach_earlier_outputs(rule):
    """O for chunks <= k does not change when X or E change in chunks > k, and
    E changes in chunk k itself do not reach O_k (apply-then-update, and the
    conv padding stops at the chunk end: itsolotime §2.2, §3.2)."""
    t = _tiny(L=24, B=6)
    args = lambda X, E: orc.layer_forward(X, E, t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"],
                                          24, 6, 0.3, rule)
    O, _ = args(t["X"], t["E"])
    k = 2
    X2, E2 = t["X"].copy(), t["E"].copy()
    X2[(k + 1) * 6:] += 1.0
    E2[k * 6:] -= 2.0  # includes the first rows of chunk k, the ones an unpadded conv would leak
    O2, _ = args(X2, E2)
    np.testing.assert_array_equal(O2[:(k + 1) * 6], O[:(k + 1) * 6])
    assert np.max(np.abs(O2[(k + 1) * 6:] - O[(k + 1) * 6:])) > 1e-3


@pytest.mark.parametrize("rule", ["mse", "add"])
def test_resume_equals_single_pass(rule):
    """Running the first half, then the second half from W_final, equals one pass
    (the chunked algorithm is the serial one, itsolotime §3.2)."""
    t = _tiny(L=24, B=4, batch=2)
    L, B = 24, 4
    X, E = t["X"].reshape(2, L, -1), t["E"].reshape(2, L, -1)
    f = lambda X, E, W0, L: orc.layer_forward(X.reshape(-1, X.shape[-1]), E.reshape(-1, E.shape[-1]),
                                              t["W_g"], t["W_u"], W0, t["conv_w"], t["P"], L, B, 0.25, rule)
    O, W = f(X, E, t["W_o0"], L)
    O1, W1 = f(X[:, :12], E[:, :12], t["W_o0"], 12)
    O2, W2 = f(X[:, 12:], E[:, 12:], W1, 12)
    Ocat = np.concatenate([O1.reshape(2, 12, -1), O2.reshape(2, 12, -1)], axis=1).reshape(O.shape)
    np.testing.assert_allclose(Ocat, O, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(W2, W, rtol=1e-12, atol=1e-13)


def test_sequences_are_independent():
    t = _tiny(batch=3)
    L = t["L"]
    O, W = orc.layer_forward(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"], L, 6, 0.2)
    for s in range(3):
        r = slice(s * L, (s + 1) * L)
        Os, Ws = orc.layer_forward(t["X"][r], t["E"][r], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"],
                                   L, 6, 0.2)
        np.testing.assert_array_equal(O[r], Os)
        np.testing.assert_array_equal(W[s], Ws[0])


def test_layer_forward_equals_engine_on_precomputed_Z_V_and_prefix():
    t = _tiny(L=30, B=5)
    Z = orc.gated_activation(t["X"], t["W_g"], t["W_u"])
    V = orc.make_targets(t["E"], t["conv_w"], t["P"], 5)
    O, W = orc.layer_forward(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"], 30, 5, 0.3)
    Oe, We = orc.chunk_engine(Z, V, t["W_o0"], 5, 0.3)
    np.testing.assert_allclose(O, Oe, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(W[0], We, rtol=1e-13, atol=1e-14)
    Op, Wp = orc.layer_forward(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"], 30, 5, 0.3,
                               max_chunks=2)
    Oe2, We2 = orc.chunk_engine(Z, V, t["W_o0"], 5, 0.3, max_chunks=2)
    np.testing.assert_allclose(Op, Oe2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(Wp[0], We2, rtol=1e-13, atol=1e-14)


def test_tiny_workload_is_stable_and_finite():
    """Guard, not a pin: eta * lambda_max(Z_k^T Z_k / B) < 2 on the tiny workload,
    so the MSE recursion contracts and the oracle's outputs stay finite."""
    w = inputs.workload("tiny")
    a = inputs.generate(w, seed=0)
    Z = orc.gated_activation(a["X"], a["W_g"], a["W_u"])
    for k in range(w.K):
        Zk = Z[k * w.B:(k + 1) * w.B]
        lam = np.linalg.eigvalsh(Zk.T @ Zk / w.B).max()
        assert w.eta * lam < 2.0
    for rule in w.rules:
        O, W = orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"],
                                 w.L, w.B, w.eta, rule)
        assert np.all(np.isfinite(O)) and np.all(np.isfinite(W))


# ------------------------------------------------- packed documents (varlen)
def _targets_per_token(E, conv_w, P, starts, ends, B):
    """v_t = (sum_j conv_w[:, j] * E[t+j]) P over the taps that stay inside t's
    chunk, chunks of B tokens counted from each document's first token and cut
    at its last: a per-token loop, independent of the oracle's chunk slicing."""
    V = np.zeros_like(E)
    for a, b in zip(starts, ends):
        for t in range(a, b):
            end = min(a + ((t - a) // B + 1) * B, b)
            c = np.zeros(E.shape[1])
            for j in range(4):
                if t + j < end:
                    c += conv_w[:, j] * E[t + j]
            V[t] = c @ P
    return V


def _docs(lengths, seed=11, d=4, d_ff=6):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    t = dict(X=rng.standard_normal((T, d)), E=rng.standard_normal((T, d)),
             W_g=rng.standard_normal((d, d_ff)) / np.sqrt(d), W_u=rng.standard_normal((d, d_ff)) / np.sqrt(d),
             W_o0=rng.standard_normal((d_ff, d)) / np.sqrt(d_ff), conv_w=rng.standard_normal((d, 4)) * np.sqrt(0.5),
             P=rng.standard_normal((d, d)) / np.sqrt(d))
    t["cu"] = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return t


def _varlen(t, B, eta, rule="mse", W0=None):
    return orc.layer_forward_varlen(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"] if W0 is None else W0,
                                    t["conv_w"], t["P"], t["cu"], B, eta, rule)


@pytest.mark.parametrize("rule", ["mse", "add"])
def test_varlen_whole_chunk_documents_equal_the_batched_layer(rule):
    """Documents of whole chunks, all of one length: the batched layer, each
    sequence restarting from W_o0 (the reset is the batched layer's own)."""
    t = _docs([12, 12, 12])
    O, W = _varlen(t, 4, 0.2, rule)
    Ob, Wb = orc.layer_forward(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"], 12, 4, 0.2, rule)
    np.testing.assert_allclose(O, Ob, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(W, Wb, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("rule", ["mse", "add"])
def test_varlen_ragged_documents_match_per_token_brute_force(rule):
    """Ragged last chunks (13 = 4+4+4+1, 6 = 4+2) and a document shorter than B:
    per-token outputs and gradients, the fast weight reset per document, each
    chunk's step averaged over its own tokens."""
    lengths, B, eta = [13, 3, 6], 4, 0.25
    t = _docs(lengths)
    O, W = _varlen(t, B, eta, rule)
    cu = t["cu"]
    Z = orc.gated_activation(t["X"], t["W_g"], t["W_u"])
    V = _targets_per_token(t["E"], t["conv_w"], t["P"], cu[:-1], cu[1:], B)
    for i in range(len(lengths)):
        r = slice(cu[i], cu[i + 1])
        Ob, Wb = _brute_force(Z[r], V[r], t["W_o0"], B, eta, rule)
        np.testing.assert_allclose(O[r], Ob, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(W[i], Wb, rtol=1e-12, atol=1e-12)


def test_varlen_short_document_closed_form():
    """One document of n < B tokens is one chunk: O = MLP(x) with W_o0 (two
    plain matmuls and the logistic function), and
    W_final = W_o0 - (eta/n) Z^T (Z W_o0 - V)."""
    n, B, eta = 5, 8, 0.3
    t = _docs([n], seed=12)
    O, W = _varlen(t, B, eta)
    a = t["X"] @ t["W_g"]
    Z = a * scipy.special.expit(a) * (t["X"] @ t["W_u"])
    V = _targets_per_token(t["E"], t["conv_w"], t["P"], [0], [n], B)
    np.testing.assert_allclose(O, Z @ t["W_o0"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(W[0], t["W_o0"] - (eta / n) * Z.T @ (Z @ t["W_o0"] - V), rtol=1e-12, atol=1e-13)


def test_varlen_documents_are_isolated():
    """Changing one document's tokens changes nothing in the others (the reset
    at each boundary, and no conv tap reads across one)."""
    lengths, B = [9, 7, 10], 4
    t = _docs(lengths)
    O, W = _varlen(t, B, 0.2)
    cu = t["cu"]
    t2 = dict(t)
    t2["X"] = t["X"].copy()
    t2["E"] = t["E"].copy()
    t2["X"][cu[1]:cu[2]] += 1.0
    t2["E"][cu[1]:cu[2]] -= 0.5
    O2, W2 = _varlen(t2, B, 0.2)
    for i in (0, 2):
        np.testing.assert_array_equal(O2[cu[i]:cu[i + 1]], O[cu[i]:cu[i + 1]])
        np.testing.assert_array_equal(W2[i], W[i])
    assert not np.allclose(O2[cu[1]:cu[2]], O[cu[1]:cu[2]])
    assert not np.allclose(W2[1], W[1])


def test_varlen_rejects_bad_boundaries():
    t = _docs([4, 4])
    for cu in ([0, 4, 4, 8], [1, 8], [0, 4, 9]):
        with pytest.raises(ValueError):
            orc.layer_forward_varlen(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"], cu, 4, 0.1)


# --------------------------------------------------- several layers at once
def _layers(n=3, seed=21, L=12, d=4, d_ff=6, batch=2):
    rng = np.random.default_rng(seed)
    T = batch * L
    return dict(X=rng.standard_normal((n, T, d)), E=rng.standard_normal((T, d)),
                W_g=rng.standard_normal((n, d, d_ff)) / np.sqrt(d), W_u=rng.standard_normal((n, d, d_ff)) / np.sqrt(d),
                W_o0=rng.standard_normal((n, d_ff, d)) / np.sqrt(d_ff),
                conv_w=rng.standard_normal((n, d, 4)) * np.sqrt(0.5), P=rng.standard_normal((n, d, d)) / np.sqrt(d),
                L=L)


@pytest.mark.parametrize("rule", ["mse", "add"])
def test_layers_match_per_layer_brute_force(rule):
    """Each layer is its own gated MLP with its own fast weight: per layer and
    sequence, the per-token brute force on that layer's Z (two matmuls and the
    logistic function) and targets (per-token conv of the shared E)."""
    t, B, eta = _layers(), 4, 0.2
    L = t["L"]
    O, W = orc.layers_forward(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"], L, B, eta, rule)
    assert O.shape == t["X"].shape and W.shape == (3, 2) + t["W_o0"].shape[1:]
    for l in range(3):
        a = t["X"][l] @ t["W_g"][l]
        Z = a * scipy.special.expit(a) * (t["X"][l] @ t["W_u"][l])
        starts = np.arange(0, 2 * L, L)
        V = _targets_per_token(t["E"], t["conv_w"][l], t["P"][l], starts, starts + L, B)
        for s in range(2):
            r = slice(s * L, (s + 1) * L)
            Ob, Wb = _brute_force(Z[r], V[r], t["W_o0"][l], B, eta, rule)
            np.testing.assert_allclose(O[l][r], Ob, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(W[l][s], Wb, rtol=1e-12, atol=1e-12)


def test_layers_do_not_interact():
    t = _layers()
    O, W = orc.layers_forward(t["X"], t["E"], t["W_g"], t["W_u"], t["W_o0"], t["conv_w"], t["P"], t["L"], 4, 0.2)
    t2 = dict(t)
    t2["W_g"] = t["W_g"].copy()
    t2["W_g"][1] *= 1.5
    t2["P"] = t["P"].copy()
    t2["P"][1] *= -1.0
    O2, W2 = orc.layers_forward(t2["X"], t2["E"], t2["W_g"], t2["W_u"], t2["W_o0"], t2["conv_w"], t2["P"],
                                t["L"], 4, 0.2)
    for l in (0, 2):
        np.testing.assert_array_equal(O2[l], O[l])
        np.testing.assert_array_equal(W2[l], W[l])
    assert not np.allclose(O2[1], O[1])
