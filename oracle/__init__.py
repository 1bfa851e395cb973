"""fp64 CPU oracle of the quantized MoE decode layer.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  See ``moe_oracle`` for
the definition it follows and the readings it takes where the pages are open.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import __all__  # noqa: F401
