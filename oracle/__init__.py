"""fp64 CPU oracle (test infrastructure only; never imported by the library).

See dcp_oracle for what it computes and which passages each function follows.
Every function here is pinned by tests against values and identities the
pages or the mathematics fix; none is marked "parity unpinned".
"""
from .dcp_oracle import *  # noqa: F401,F403
