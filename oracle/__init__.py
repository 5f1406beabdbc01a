"""Float64 CPU oracle of the In-Place TTT fast-weight layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package; the CUDA library never does.
"""
from .ipttt_oracle import *  # noqa: F401,F403
from .ipttt_oracle import __all__  # noqa: F401
