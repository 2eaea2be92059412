"""Per-frame SSIMULACRA2 scoring of YUV frame pairs on NVIDIA GB300 (sm_103a).

The compute path is libss2 (CUDA kernels behind the C ABI in include/ss2.h);
this package holds the ctypes binding (``ss2``) and the in-tree build
(``_build``).
"""
from .ss2 import (MSSSIM, NPARAMS, Cambi, NVALUES, FloatSSIM, Scorer, SS2Error,  # noqa: F401
                  default_params, host_tables, last_error, lib)

__all__ = ["Scorer", "FloatSSIM", "MSSSIM", "Cambi", "SS2Error", "default_params", "host_tables", "last_error",
           "lib", "NPARAMS", "NVALUES"]
