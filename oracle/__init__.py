"""Float64 CPU oracle of the OSCAR two-bit rotated KV-cache path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
anything in this package; only the tests, `__graft_entry__.smoke()` and the
CPU-baseline leg of `bench.py` use it.  It shares no code with the CUDA
library: it is plain numpy, written from the pages' description of the
method, and serves as the checker the CUDA path is compared against.
"""
from .oscar_oracle import *  # noqa: F401,F403
