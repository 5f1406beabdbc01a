"""The allocation-free target builder, ipttt_make_targets_noalloc.

It is meant for callers that cannot allocate device memory while they build
targets: their GPU memory is already handed out by another allocator, or they
cannot afford a cudaMalloc / cudaFree that may synchronise the device.  It must
give the same targets as ipttt_make_targets, which draws the same scratch
from the library's cudaMalloc-grown pool, call after call even though every
call reuses the same fixed array.  (This file is collected last on purpose.)
"""
import numpy as np
import pytest
import torch

import chunked_weight_mlp_place_b300 as ip
from chunked_weight_mlp_place_b300 import inputs
from chunked_weight_mlp_place_b300.build import build
from gpu_util import down, up

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    ip.lib()


@pytest.mark.parametrize("dtype,batch,L,B,d", [("bf16", 2, 1024, 256, 1024), ("bf16", 1, 3072, 1024, 2560),
                                               ("fp32", 2, 96, 24, 120)])
def test_noalloc_targets_match_the_pooled_entry_point(dtype, batch, L, B, d):
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = inputs.round_to_bf16 if dtype == "bf16" else (lambda a: a.astype(np.float32))
    for call in range(2):  # two calls in a row: the second reuses the array the first filled
        rng = np.random.default_rng(100 * call + d)
        E = up(q((rng.standard_normal((batch * L, d)) * d ** -0.5).astype(np.float32)), dt)
        w = up((rng.standard_normal((d, 4)) * 0.5 ** 0.5).astype(np.float32), torch.float32)
        P = up(q((rng.standard_normal((d, d)) * d ** -0.5).astype(np.float32)), dt)
        V_pool = torch.empty(batch * L, d, dtype=dt, device="cuda")
        V_fixed = torch.full((batch * L, d), float("nan"), dtype=dt, device="cuda")
        ip.make_targets(E, w, P, V_pool, L, B)
        ip.make_targets_noalloc(E, w, P, V_fixed, L, B)
        assert ip.sync_status() == 0
        a, b = down(V_fixed), down(V_pool)
        assert np.all(np.isfinite(a))
        # the same kernels on the same inputs with a deterministic store epilogue: bit for bit equal
        np.testing.assert_array_equal(a, b, err_msg=f"call {call}")


def test_noalloc_targets_refuse_more_than_the_fixed_scratch():
    d, B = 2560, 1024
    L = 4 * B  # 4096 x 2560 bf16 = 20 MiB of conv output > 16 MiB
    E = torch.zeros(L, d, dtype=torch.bfloat16, device="cuda")
    V = torch.empty(L, d, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(d, 4, device="cuda")
    P = torch.zeros(d, d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ip.IptttError, match="fixed"):
        ip.make_targets_noalloc(E, w, P, V, L, B)
    assert ip.sync_status() == 0
