"""CPU fp64 oracle for the FlashAttention-2 forward pass — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. The product (``attention_forward_03_gb300``)
never imports it, and the two share no code: the only common module is
``workloads`` (seeded input generation, no attention arithmetic).

Contents
  attention_fwd   the definition of the forward pass (C, fp64), all rows or a
                  sample of rows. See ``fa2_oracle.c`` for the formula and
                  its sources.
  online_merge    the tile-by-tile (m, l) recurrence of the pages, in numpy
                  fp64, used only to pin the definition against the method's
                  own recurrence.
  attention_bwd   the gradient of the forward definition w.r.t. Q, K, V for
                  an upstream gradient dO (C, fp64). See ``fa2_bwd_oracle.c``.

Every function here is pinned by ``tests/test_oracle_pins.py`` (forward) and
``tests/test_oracle_bwd_pins.py`` (gradient).
"""
from .reference import attention_fwd, sample_rows, default_threads  # noqa: F401
from .online import online_merge  # noqa: F401
from .gradient import attention_bwd  # noqa: F401
