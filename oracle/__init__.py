"""fp64 CPU oracle for the multi-LoRA delta (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library in ``lora_serving_gb300/``.
"""
from .oracle import *  # noqa: F401,F403
