"""fp64 CPU oracle for the BackLite attention hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the library.  It shares no
code with the CUDA path.

* ``attention``  -- exact forward, per-tile LSE statistics, masked backward.
* ``mask_spec``  -- the canonical tile-selection rule (mask_from_stats).
* ``varlen``     -- the three steps over packed variable-length batches.
"""
from . import attention, mask_spec, varlen  # noqa: F401
