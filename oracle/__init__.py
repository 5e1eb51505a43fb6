"""Float64 CPU oracle for the MHLA forward pass.

Test infrastructure: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA library (``token_level_head_phi_gb300``) and imports only numpy.
"""

from .mhla_oracle import *  # noqa: F401,F403
from .mhla_oracle import __all__  # noqa: F401
