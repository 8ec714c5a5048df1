"""GB300-native compressed-KV sparse attention path (DeepSeek-V4-style).

The compute lives in libds4c.so (hand-written CUDA for sm_103a behind the C ABI
of include/ds4c.h).  ``abi`` binds it with ctypes under the ABI's own names;
``layer.DeviceLayer`` owns a layer's device tensors and calls the ABI;
``configs`` and ``synth`` describe the synthetic workloads.
"""

from . import configs, synth  # noqa: F401

__all__ = ["configs", "synth", "abi", "layer", "build"]
