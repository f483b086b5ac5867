"""fp64 CPU oracle for paged-KV attention (test infrastructure only; parity pinned by
``tests/test_oracle_*.py``). Never imported by the CUDA library."""
from .oracle import *  # noqa: F401,F403
from .oracle import build, default_threads  # noqa: F401
