"""CPU oracle for the Beam MoE sublayer (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
package. The CUDA path never does.
"""
from .beam_oracle import *  # noqa: F401,F403
