"""GB300-native multi-LoRA delta (SGMV / BGMV) behind a C ABI.

The CUDA library ``liblora.so`` (include/lora.h) does all of the work; the
Python side marshals arguments (``abi``), manages device memory for the
adapter store and metadata (``store``) and draws seeded synthetic inputs
(``synth``).
"""
from .build import build  # noqa: F401

__all__ = ["build", "abi", "store", "synth"]
