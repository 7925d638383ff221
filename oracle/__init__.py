"""Float64 CPU oracle (test infrastructure; see ``oracle/ref.py`` header).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this package."""
from .ref import *  # noqa: F401,F403
from .ref import IGNORE_INDEX  # noqa: F401
