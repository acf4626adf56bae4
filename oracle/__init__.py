"""CPU oracle for the decode GEMV (test infrastructure only; see oracle.py)."""
from .oracle import (RTOL, accept, build, default_threads, gemv, gemv_one,  # noqa: F401
                     gemv_rmsnorm, gemv_w4, load)
