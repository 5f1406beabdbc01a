"""libipttt for B300: the fast-weight hot path of In-Place Test-Time Training.

The compute lives in ``libipttt.so`` (hand-written sm_103a CUDA kernels behind
the C-ABI of ``include/ipttt.h``); this package holds its ctypes binding, the
in-tree build script and the seeded synthetic input generator.
"""
from ._lib import (  # noqa: F401
    BF16, FP32, RULE_ADD, RULE_MSE, IptttError, additive_sums, chunk_forward, copy_weights, gate_up, kernel_timing,
    kernel_timing_read, weight_axpy,
    last_launch_count, layer_forward, layer_forward_varlen, layers_forward,
    lib, make_targets, make_targets_noalloc, release, set_pool_limit, set_wait_limit, status_string, sync_status,
    version,
    workspace_size,
)
