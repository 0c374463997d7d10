"""fp64 CPU oracle of the compressed-sparse-attention path.

TEST INFRASTRUCTURE: only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm import this package. The CUDA library never does.
"""
from .csa_oracle import *  # noqa: F401,F403
from .csa_oracle import __all__  # noqa: F401
