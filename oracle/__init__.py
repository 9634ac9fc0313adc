"""CPU oracle for the 'store sharded, compute full' weight path.

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline use it. The CUDA library never imports or calls it.
"""
from .sws_oracle import *  # noqa: F401,F403
