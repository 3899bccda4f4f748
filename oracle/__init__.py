"""fp64 CPU oracle of the Medusa decode step.  Test infrastructure only.

Only tests, the smoke check and the benchmark's CPU-baseline leg import this package;
the library never does.
"""
from .medusa_oracle import *  # noqa: F401,F403
