"""CPU oracle for batched paged-KV attention — test infrastructure only.

Imported by the test-suite, by ``__graft_entry__.smoke()`` and by the CPU
baseline leg of ``bench.py``; never by the library's product path.  See
``oracle/ref.py`` for what it computes and which page each function follows.
"""
from .ref import *  # noqa: F401,F403
