"""CPU oracle for the ConvRot W4A8 linear layer -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the package smoke check and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never calls into it, and it shares no code with that path.
"""
from .convrot_oracle import *  # noqa: F401,F403
from .convrot_oracle import __all__  # noqa: F401
