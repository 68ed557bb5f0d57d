"""CPU oracle of the decode KV swap-in: TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or calls anything here.
"""
from .oracle import Oracle, build_oracle, page_table, NUM_STATS, STAT_NAMES  # noqa: F401
