"""CPU oracle of the top-k routed MoE FFN layer (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` import this package. The product (the CUDA library and its
binding) never does.
"""
from . import moe_oracle  # noqa: F401
