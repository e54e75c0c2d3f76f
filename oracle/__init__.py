"""CPU oracle (float64, unchunked) for the LM-head objectives.

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline leg use it.  The product path never imports it.
"""
from .lmhead import *  # noqa: F401,F403
