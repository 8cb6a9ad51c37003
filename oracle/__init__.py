"""CPU oracle for the int4-weight quantized linear layer.

TEST INFRASTRUCTURE ONLY. Nothing in the product package imports, calls or
links anything here; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it. It
shares no code with the CUDA path.

The oracle proper is plain numpy in float64 / int64 (``w4_oracle.py``). The W4A16
layer is also stated in plain C (``w4_oracle_c.c``, called through
``c_oracle.py``) for timing the CPU baseline on the host's cores; the tests pin it
to the numpy statement.
"""
from .w4_oracle import *  # noqa: F401,F403
