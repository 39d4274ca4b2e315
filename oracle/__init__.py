"""fp64 CPU oracle for block-sparse paged MSA.  Test infrastructure only: used by
tests/, the smoke check and the bench's CPU-baseline leg, never by the CUDA path."""
from .msa_oracle import *  # noqa: F401,F403
from .msa_oracle import __all__  # noqa: F401
