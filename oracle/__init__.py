"""CPU oracle for the grouped MXFP8 MoE expert MLP — test infrastructure.

Plain, slow, fp64 restatement of the method from the pages, pinned by the
``-m "not gpu"`` tests in tests/test_oracle_*.py.  Only tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline leg may import it; the
product path (mxfp8_grouped_gemm_gb300) never does, and this package imports
nothing from the product path.
"""
from . import mx, moe  # noqa: F401
