"""GB300-native (sm_103a) KDA gated delta-rule serving step.

The product is the C-ABI library libkda_gb300.so (include/kda.h): kda_decode,
kda_verify and kda_verify_ring. This package holds its CUDA sources (csrc/),
its in-tree build (_build.py), a ctypes binding with the same names (kda.py)
and seeded synthetic workloads (workloads.py).
"""

from . import kda, workloads  # noqa: F401
from .kda import (  # noqa: F401
    KdaError,
    kda_decode,
    kda_verify,
    kda_verify_ring,
    kda_select_config,
    kda_num_configs,
    kda_config_tile_v,
    kda_last_error,
    load_library,
)
