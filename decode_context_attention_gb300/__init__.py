"""GB300-native (sm_103a) DCP LSE merge: pack, combine and fused unpack+combine.

The compute lives in ``libdcp_gb300.so`` (hand-written CUDA behind a C ABI,
declared in ``include/dcp.h``); ``binding`` is a thin ctypes layer over it.
There is no CPU fallback: calling into the binding without the built library
raises.
"""
from .workloads import WORKLOADS, Workload, generate, sweep_points  # noqa: F401
