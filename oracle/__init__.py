"""CPU oracle of the quantized attention recipe (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path never does.
"""
from .qattn_oracle import *  # noqa: F401,F403
from . import qattn_oracle  # noqa: F401
