"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments with a status code before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from chunked_weight_mlp_place_b300 import _lib
from chunked_weight_mlp_place_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build()
    return _lib.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "ipttt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ipttt_\w+)\s*\(", src)))


def test_header_and_binding_agree():
    assert _declared() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert _lib.version() == 100
    for s in range(7):
        assert _lib.status_string(s)
    assert "unknown" in _lib.status_string(99)


def _dims(batch=1, d=64, d_ff=256, dtype=_lib.BF16, w0=0):
    return _lib.dims(batch, d, d_ff, dtype, w0)


FAKE = 1 << 20  # aligned, non-null, never dereferenced: host checks fail first or no device is found


def _layer(L, dm, Lseq=256, B=64, eta=0.1, rule=0, ptrs=None, pdims=True):
    p = ptrs if ptrs is not None else [FAKE] * 9
    return L.ipttt_layer_forward(p[0], p[1], p[2], p[3], p[4], p[5], p[6], Lseq, B, eta, rule, p[7], p[8],
                                 ctypes.byref(dm) if pdims else None, None)


def test_invalid_arguments_are_rejected_on_the_host(L):
    E = _lib.ERR_INVALID_ARG
    assert _layer(L, _dims(), pdims=False) == E                        # no dims
    assert _layer(L, _dims(), Lseq=250, B=64) == E                     # L % B != 0
    assert _layer(L, _dims(), B=0) == E                                # B < 1
    assert _layer(L, _dims(), Lseq=-64) == E                           # L < 0
    assert _layer(L, _dims(d=60)) == E                                 # bf16 needs d % 8 == 0
    assert _layer(L, _dims(d_ff=100)) == E                             # bf16 needs d_ff % 8 == 0
    assert _layer(L, _dims(), Lseq=240, B=24) == E                     # bf16 needs B % 16 == 0
    assert _layer(L, _dims(dtype=7)) == E                              # unknown dtype
    assert _layer(L, _dims(d=0)) == E
    assert _layer(L, _dims(batch=-1)) == E
    assert _layer(L, _dims(w0=2)) == E
    assert _layer(L, _dims(), rule=5) == E                             # unknown rule
    assert _layer(L, _dims(), eta=float("nan")) == E
    ptrs = [FAKE] * 9
    ptrs[3] = 0
    assert _layer(L, _dims(), ptrs=ptrs) == E                          # null pointer
    ptrs[3] = FAKE + 4
    assert _layer(L, _dims(), ptrs=ptrs) == E                          # misaligned pointer
    dm = _dims()
    assert L.ipttt_make_targets(FAKE, FAKE, FAKE, FAKE, 100, 64, ctypes.byref(dm), None) == E
    assert L.ipttt_gate_up(FAKE, FAKE, FAKE, FAKE, -1, ctypes.byref(dm), None) == E
    assert L.ipttt_chunk_forward(FAKE, FAKE, FAKE, 256, 48, 0.1, 0, FAKE, FAKE, ctypes.byref(dm), None) == E


def _varlen(L, dm, cu, B=64, eta=0.1, rule=0):
    arr = (ctypes.c_int64 * max(1, len(cu)))(*cu) if cu is not None else None
    return L.ipttt_layer_forward_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, arr, max(0, len(cu or []) - 1),
                                        B, eta, rule, FAKE, FAKE, ctypes.byref(dm), None)


def test_varlen_arguments_are_checked_on_the_host(L):
    E = _lib.ERR_INVALID_ARG
    dm = _dims()
    assert _varlen(L, dm, None) == E                                   # no boundaries
    assert _varlen(L, dm, [1, 64]) == E                                # must start at 0
    assert _varlen(L, dm, [0, 64, 64, 128]) == E                       # empty document
    assert _varlen(L, dm, [0, 100, 90]) == E                           # falling boundary
    assert _varlen(L, dm, [0, 64], B=24) == E                          # bf16 needs B % 16 == 0
    assert _varlen(L, dm, [0, 64], B=0) == E
    assert _varlen(L, dm, [0, 64], rule=3) == E
    assert _varlen(L, dm, [0, 64], eta=float("inf")) == E
    assert _varlen(L, dm, [0]) == _lib.OK                              # no documents: nothing to do
    # valid boundaries, ragged lengths: the call reaches the device check
    st = _varlen(L, dm, [0, 70, 75, 300])
    assert st in (_lib.ERR_UNSUPPORTED, _lib.OK, _lib.ERR_INVALID_ARG)


def test_layers_arguments_are_checked_on_the_host(L):
    E = _lib.ERR_INVALID_ARG
    dm = _dims(batch=2)

    def call(n_layers=3, Lseq=256, B=64, eta=0.1, rule=0, d=dm):
        return L.ipttt_layers_forward(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, n_layers, Lseq, B, eta, rule,
                                      FAKE, FAKE, ctypes.byref(d), None)

    assert call(n_layers=-1) == E
    assert call(Lseq=250) == E                                          # L % B != 0
    assert call(B=24) == E                                              # bf16 needs B % 16 == 0
    assert call(rule=7) == E
    assert call(eta=float("nan")) == E
    assert call(d=_dims(d=60)) == E
    assert call(n_layers=0) == _lib.OK                                  # nothing to do
    assert call(d=_dims(batch=0)) == _lib.OK
    assert call() in (_lib.ERR_UNSUPPORTED, _lib.OK, _lib.ERR_INVALID_ARG)  # reaches the device check


def test_context_parallel_pieces_are_checked_on_the_host(L):
    E = _lib.ERR_INVALID_ARG
    dm = _dims(batch=2)
    assert L.ipttt_additive_sums(FAKE, FAKE, 100, FAKE, ctypes.byref(dm), None) == E   # bf16: L % 16
    assert L.ipttt_additive_sums(FAKE, FAKE, -16, FAKE, ctypes.byref(dm), None) == E
    assert L.ipttt_additive_sums(FAKE, FAKE, 64, FAKE, None, None) == E
    assert L.ipttt_additive_sums(FAKE, FAKE, 64, FAKE, ctypes.byref(_dims(batch=0)), None) == _lib.OK
    assert L.ipttt_weight_axpy(FAKE, FAKE, 0.5, -1, None) == E
    assert L.ipttt_weight_axpy(FAKE, FAKE, float("nan"), 8, None) == E
    assert L.ipttt_weight_axpy(FAKE, FAKE, 0.5, 0, None) == _lib.OK
    assert L.ipttt_weight_axpy(0, FAKE, 0.5, 8, None) == E                              # null pointer


def test_pool_limit_is_host_only(L):
    assert L.ipttt_set_pool_limit(1 << 20) == _lib.OK
    assert L.ipttt_set_pool_limit(0) == _lib.OK


def test_fp32_mode_takes_any_sizes_on_the_host_checks(L):
    # fp32 accepts ragged sizes; with valid arguments the call reaches the device
    # check, which on a machine without a B300 says "unsupported".
    dm = _dims(d=37, d_ff=90, dtype=_lib.FP32)
    st = _layer(L, dm, Lseq=30, B=5)
    assert st in (_lib.ERR_UNSUPPORTED, _lib.OK, _lib.ERR_INVALID_ARG)
    try:
        import torch
        if not torch.cuda.is_available():
            assert st == _lib.ERR_UNSUPPORTED
    except ImportError:
        pass


def test_empty_inputs_are_no_ops(L):
    dm = _dims(batch=0)
    assert _layer(L, dm) == _lib.OK
    assert L.ipttt_gate_up(0, 0, 0, 0, 0, ctypes.byref(_dims()), None) == _lib.OK
    assert L.ipttt_make_targets(0, 0, 0, 0, 256, 64, ctypes.byref(_dims(batch=0)), None) == _lib.OK


def test_workspace_size_is_host_only(L):
    out = ctypes.c_size_t()
    dm = _dims(batch=1, d=2560, d_ff=9728)
    assert L.ipttt_workspace_size(ctypes.byref(dm), 131072, 1024, 0, 1, ctypes.byref(out)) == _lib.OK
    T = 131072
    act = T * 9728 * 2 + 2 * T * 2560 * 2
    # fp32 partial sums and bf16 residual of one chunk, the fast weight's split hi/lo planes, and
    # the persistent engine's counters: per chunk and 256-column block, three per 256-token tile
    # (two halves' applies, the residual) and one per d_ff slice (4)
    eng = 1024 * 2560 * 4 + 1024 * 2560 * 2 + 2 * 9728 * 2560 * 2 + 128 * 10 * (3 * 4 + 4) * 4
    assert act + eng <= out.value <= act + eng + 4096
    assert L.ipttt_workspace_size(ctypes.byref(dm), 131072, 1024, 0, 0, ctypes.byref(out)) == _lib.OK
    assert eng <= out.value <= eng + 4096
    # additive scan: 8 groups of fp32 sums + split hi/lo states
    assert L.ipttt_workspace_size(ctypes.byref(dm), 32768, 64, 1, 0, ctypes.byref(out)) == _lib.OK
    assert out.value >= 8 * 9728 * 2560 * 8
    # block-causal additive form: [Z | S] (L x (d_ff + L)) and [W_0 ; V] ((d_ff + L) x d) act, Z^T V fp32
    assert L.ipttt_workspace_size(ctypes.byref(dm), 32768, 64, 2, 0, ctypes.byref(out)) == _lib.OK
    kc = 9728 + 32768
    quad = 32768 * kc * 2 + kc * 2560 * 2 + 9728 * 2560 * 4
    assert quad <= out.value <= quad + 4096
    # MSE with chunks of 64 tokens: windows of 1024 tokens (16 chunks): the engine's sums, counters
    # and planes for 1024-token chunks, every window's Y, Zt, and the Gram and X of each of the 32
    # windows (1024 x 1024 bf16)
    assert L.ipttt_workspace_size(ctypes.byref(dm), 32768, 64, 0, 0, ctypes.byref(out)) == _lib.OK
    win = (1024 * 2560 * 4 + 32768 * 2560 * 2 + 2 * 9728 * 2560 * 2 + 32 * 10 * (3 * 4 + 4) * 4
           + 2 * 32 * 1024 * 1024 * 2 + 32768 * 9728 * 2)
    assert win <= out.value <= win + 4096
    # d = 1024 with two chunks a window: no windows (d (m - 1) < 2 W), the engine on 512-token chunks
    dm5 = _dims(batch=8, d=1024, d_ff=4096)
    assert L.ipttt_workspace_size(ctypes.byref(dm5), 4096, 512, 0, 0, ctypes.byref(out)) == _lib.OK
    eng5 = 8 * (512 * 1024 * 4 + 512 * 1024 * 2 + 2 * 4096 * 1024 * 2) + 8 * 8 * 4 * (3 * 2 + 4) * 4
    assert eng5 <= out.value <= eng5 + 4096
    assert L.ipttt_workspace_size(ctypes.byref(dm), 100, 64, 0, 0, ctypes.byref(out)) == _lib.ERR_INVALID_ARG
    assert L.ipttt_workspace_size(None, 128, 64, 0, 0, ctypes.byref(out)) == _lib.ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        _lib.gate_up(x, torch.zeros(8, 8, dtype=torch.bfloat16), torch.zeros(8, 8, dtype=torch.bfloat16),
                     torch.zeros(4, 8, dtype=torch.bfloat16))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libipttt.so"))
    with pytest.raises(ImportError):
        _lib.lib()


def test_noalloc_targets_size_limit_is_checked_on_the_host(L):
    dm = _dims(batch=1, d=2560)
    # 4096 tokens x 2560 bf16 = 20 MiB > the 16 MiB fixed scratch: rejected before any device call
    assert L.ipttt_make_targets_noalloc(FAKE, FAKE, FAKE, FAKE, 4096, 1024, ctypes.byref(dm), None) == \
        _lib.ERR_INVALID_ARG
    assert L.ipttt_make_targets_noalloc(FAKE, FAKE, FAKE, FAKE, 100, 64, ctypes.byref(dm), None) == \
        _lib.ERR_INVALID_ARG
    assert L.ipttt_make_targets_noalloc(0, 0, 0, 0, 0, 64, ctypes.byref(dm), None) == _lib.OK


def test_header_is_plain_c_and_the_library_links_from_c(tmp_path):
    """The boundary is a C ABI: a C program (gcc, not a C++ compiler) includes the
    header, links against the built library and calls its host-only functions."""
    import shutil
    import subprocess

    build()
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    src = tmp_path / "use_ipttt.c"
    src.write_text(
        '#include <stdio.h>\n#include "ipttt.h"\n'
        "int main(void) {\n"
        "  ipttt_dims dm = {1, 64, 256, IPTTT_BF16, 0};\n"
        "  size_t bytes = 0;\n"
        "  if (ipttt_workspace_size(&dm, 256, 64, IPTTT_RULE_MSE, 1, &bytes) != IPTTT_OK || bytes == 0) return 1;\n"
        "  if (ipttt_layer_forward(0, 0, 0, 0, 0, 0, 0, 250, 64, 0.1f, IPTTT_RULE_MSE, 0, 0, &dm, 0)\n"
        "      != IPTTT_ERR_INVALID_ARG) return 2;\n"
        '  printf("%d %s\\n", ipttt_version(), ipttt_status_string(IPTTT_ERR_TIMEOUT));\n'
        "  return 0;\n}\n")
    exe = tmp_path / "use_ipttt"
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe), "-L", libdir, "-lipttt", "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == _lib.lib().ipttt_version() and "wait" in " ".join(out[1:])


def test_noalloc_and_pooled_targets_give_the_same_status_for_the_same_bad_argument(L):
    """Both target builders validate through the same checks: each bad argument
    below is refused on the host, with the same status, by both entry points."""
    cases = [
        (_dims(d_ff=0), FAKE, 256, 64),          # d_ff < 1
        (_dims(w0=2), FAKE, 256, 64),            # w0_per_seq outside 0/1
        (_dims(dtype=7), FAKE, 256, 64),         # unknown dtype
        (_dims(d=60), FAKE, 256, 64),            # bf16 mode, d not a multiple of 8
        (_dims(), FAKE, 250, 64),                # L not a multiple of B
        (_dims(), FAKE, 256, 24),                # bf16 mode, B not a multiple of 16
        (_dims(batch=-1), FAKE, 256, 64),        # negative batch
        (_dims(), 0, 256, 64),                   # null pointer
        (_dims(), FAKE + 8, 256, 64),            # pointer not 16-byte aligned
    ]
    for dm, ptr, Lseq, B in cases:
        a = L.ipttt_make_targets(ptr, FAKE, FAKE, FAKE, Lseq, B, ctypes.byref(dm), None)
        b = L.ipttt_make_targets_noalloc(ptr, FAKE, FAKE, FAKE, Lseq, B, ctypes.byref(dm), None)
        assert a == b == _lib.ERR_INVALID_ARG, (dm.d, dm.d_ff, dm.dtype, Lseq, B, ptr, a, b)
    assert L.ipttt_make_targets(FAKE, FAKE, FAKE, FAKE, 256, 64, None, None) == \
        L.ipttt_make_targets_noalloc(FAKE, FAKE, FAKE, FAKE, 256, 64, None, None) == _lib.ERR_INVALID_ARG


def test_binding_checks_shapes_before_the_call():
    """The C-ABI takes sizes, not tensors, so the binding checks the tensors' shapes
    against them first (a tensor smaller than the sizes say would be read or
    written past its end on the device)."""
    import torch
    E = torch.zeros(256, 64, dtype=torch.bfloat16)
    ok = dict(conv_w=torch.zeros(64, 4), P=torch.zeros(64, 64, dtype=torch.bfloat16),
              V=torch.zeros(256, 64, dtype=torch.bfloat16))
    for fn in (_lib.make_targets, _lib.make_targets_noalloc):
        for bad in (dict(V=torch.zeros(128, 64, dtype=torch.bfloat16)), dict(P=torch.zeros(32, 64, dtype=torch.bfloat16)),
                    dict(conv_w=torch.zeros(64, 3))):
            kw = dict(ok, **bad)
            with pytest.raises(ValueError, match="shape"):
                fn(E, kw["conv_w"], kw["P"], kw["V"], 128, 64)
        with pytest.raises(ValueError, match="whole number"):
            fn(E, ok["conv_w"], ok["P"], ok["V"], 96, 32)  # 256 rows are not sequences of 96
    Z = torch.zeros(256, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="shape"):
        _lib.chunk_forward(Z, torch.zeros(256, 64, dtype=torch.bfloat16), torch.zeros(128, 64), 128, 64, 0.1, "mse",
                           torch.zeros(256, 64, dtype=torch.bfloat16), torch.zeros(1, 128, 64))  # W_final: batch 2


@pytest.mark.parametrize("d,d_ff,Lseq,B", [
    (2560, 9728, 32768, 64), (2560, 9728, 32768, 512), (1024, 4096, 4096, 512), (1024, 4096, 4096, 256),
    (512, 1024, 1536, 128), (256, 512, 1536, 128), (256, 256, 512, 64), (2560, 9728, 4096, 1024),
    (384, 1024, 2048, 64), (256, 768, 768, 256),
])
def test_the_benchmark_sees_the_windows_the_library_takes(L, d, d_ff, Lseq, B):
    """bench.py's mirror of the window rule (its roofline accounting depends on it) against the
    library's own choice, read off the MSE workspace: besides the fast weight's planes (at least
    4 d d_ff bytes) a window's layout holds every chunk's Y and Zt (L (d + d_ff) bf16), where the
    chunk layout holds one chunk's sums and R and the counters."""
    import importlib.util

    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    from chunked_weight_mlp_place_b300 import inputs

    W = bench.window_tokens(inputs.workload("4b", L=Lseq, B=B, d=d, d_ff=d_ff))
    out = ctypes.c_size_t()
    assert L.ipttt_workspace_size(ctypes.byref(_dims(batch=1, d=d, d_ff=d_ff)), Lseq, B, 0, 0,
                                  ctypes.byref(out)) == _lib.OK
    assert (out.value >= 4 * d * d_ff + Lseq * (d + d_ff) * 2) == bool(W), (W, out.value)
