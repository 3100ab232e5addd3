"""CPU oracle (f64) of the DFlash drafter round -- test infrastructure only.

Only the test suite, the package's smoke check and the benchmark's CPU
baseline leg may import this package; the product path never does.
"""
from .dflash_oracle import *  # noqa: F401,F403
