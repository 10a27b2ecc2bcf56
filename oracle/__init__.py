"""fp64 CPU oracle of the UPipe attention layer -- test infrastructure only.

Imported by the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s
cpu baseline / reference arm, never by the CUDA library.
"""
from . import upipe_oracle  # noqa: F401
