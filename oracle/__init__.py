"""Reference oracle for the sparse offloaded-KV decode step.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA library (``sparse_kv_cache_landmark_gb300/csrc``) and imports nothing
from it.
"""
from .kvo_oracle import *  # noqa: F401,F403
