"""Helpers shared by the GPU parity tests: upload seeded inputs, call the C-ABI
through the binding, and bring results back as float64."""
import numpy as np
import torch

import chunked_weight_mlp_place_b300 as ip

# Relative Frobenius tolerances on O and W_final: 1e-2 for bf16 operands with
# fp32 accumulation, 1e-4 for the fp32 mode.
TOL = {"bf16": 1e-2, "fp32": 1e-4}


def tdtype(w_or_name):
    name = w_or_name if isinstance(w_or_name, str) else w_or_name.dtype
    return torch.bfloat16 if name == "bf16" else torch.float32


def up(a, dtype, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev).to(dtype).contiguous()


def down(t, dtype=torch.float64):
    return t.detach().to(dtype).cpu().numpy()


def rel(a, b):
    den = np.linalg.norm(b)
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / (den if den > 0 else 1.0))


def run_layer(w, a, rule, L=None, W0=None, stream=None, out_dtype=torch.float64):
    """Run ipttt_layer_forward on arrays ``a`` (from inputs.generate) for workload w;
    O and W_final come back as numpy arrays of ``out_dtype``."""
    dt = tdtype(w)
    L = w.L if L is None else L
    X, E = up(a["X"], dt), up(a["E"], dt)
    batch = X.shape[0] // L
    W0t = torch.from_numpy(np.ascontiguousarray(a["W_o0"] if W0 is None else W0, np.float32)).cuda()
    O = torch.empty(batch * L, w.d, dtype=dt, device="cuda")
    Wf = torch.empty(batch, w.d_ff, w.d, dtype=torch.float32, device="cuda")
    ip.layer_forward(X, E, up(a["W_g"], dt), up(a["W_u"], dt), W0t, up(a["conv_w"], torch.float32),
                     up(a["P"], dt), L, w.B, w.eta, rule, O, Wf, stream=stream)
    assert ip.sync_status() == 0
    return down(O, out_dtype), down(Wf, out_dtype)
