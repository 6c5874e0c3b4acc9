"""decode_context_mla_gb300: striped absorbed-MLA decode with an exact LSE merge on one GB300.

The compute path is libdcpmla (C ABI in include/dcpmla.h, CUDA kernels for
sm_103a); this package holds its in-tree build, its Python binding (same
names as the C calls) and a small host-side runner that strings the calls
together.  Importing the package does not load the library; the first call
does, and raises if it is missing -- there is no CPU fallback.
"""
from .binding import *  # noqa: F401,F403
from .binding import DcpmlaError  # noqa: F401
