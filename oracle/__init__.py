"""CPU oracle of the Gated DeltaNet recurrence.  TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GPU library and its Python binding
never import it; the two share no code.

* :mod:`oracle.recurrence` -- the fp64 token-by-token loop (C, OpenMP), the
  definition every GPU result is compared against;
* :mod:`oracle.chunked` -- an independent fp64 numpy statement of the
  chunk-parallel (WY/UT) form, used only to pin that the chunk algebra equals
  the token loop.
"""
from .recurrence import build, forward, decode_step, max_threads  # noqa: F401
