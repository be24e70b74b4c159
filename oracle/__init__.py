"""CPU oracle for the DLite round. TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
leg may import this package. The product path (the CUDA library and its
binding) never imports, links or runs anything here.
"""
from . import philox  # noqa: F401
from . import dlite_oracle  # noqa: F401
