"""BF16 weight-streaming decode chain for NVIDIA GB300 (sm_103a).

The compute path is the CUDA library ``lib/libwsgemv.so`` (C ABI in
``include/wsgemv.h``), reached through the thin ctypes layer in
``binding``.  ``synth`` holds the seeded synthetic inputs; ``workloads``
builds the pages' workloads on the device.
"""
from ._build import build  # noqa: F401
