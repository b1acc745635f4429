"""CPU oracle (NumPy, fp64) of the MTP drafter step, draft block and greedy verify.

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and the
benchmark's CPU-baseline / reference leg, never by the CUDA library. It shares no code with
the CUDA path. Pinned by the not-gpu tests; the composition of a whole drafter step is
"parity unpinned" beyond the pinned pieces (no published logits or tokens exist).
"""
from .mtp_oracle import *  # noqa: F401,F403
from .mtp_oracle import MASK_VALUE  # noqa: F401
