"""CPU oracle for routed block-sparse self-attention: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import anything here. The CUDA library never does, and the
two share no code. See ``sa_oracle`` for the arithmetic and its citations.
"""

from .sa_oracle import *  # noqa: F401,F403
from .sa_oracle import BLOCK, TIE_WINDOW  # noqa: F401
