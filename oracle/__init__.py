"""Float64 CPU oracle for the HSQ compressed-KV path.

TEST INFRASTRUCTURE ONLY.  This package is imported by the test-suite, by
``__graft_entry__.smoke()`` (to check one small GPU run) and by the
CPU-baseline / reference leg of ``bench.py``.  The CUDA library and its
Python binding never import, call or link anything in here, and nothing in
here imports them.
"""

from .hsq_oracle import *  # noqa: F401,F403
from .hsq_oracle import __all__  # noqa: F401
