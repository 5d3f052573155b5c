"""CPU oracle of the GPTQ per-layer path -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import or run anything in this package. The CUDA library and its
Python binding never import it, and it imports nothing from them.
"""
from .gptq_oracle import *  # noqa: F401,F403
