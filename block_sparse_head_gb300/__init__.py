"""Layout-driven block-sparse multi-head attention forward for GB300 (sm_103a).

The compute runs in ``libbsa.so`` (C ABI, hand-written CUDA); this package holds
the ctypes binding (``binding``) and the seeded synthetic workloads (``workloads``).
"""

from .binding import (  # noqa: F401
    BSA_ORDER_GLOBAL,
    BSA_ORDER_GROUPED,
    BsaError,
    Lut,
    backward,
    build_lut,
    forward,
    forward_ext,
    library_path,
    load_library,
    topk_forward,
)
