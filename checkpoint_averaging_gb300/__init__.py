"""GB300-native DiLoCo outer merge.

``checkpoint_averaging_gb300.binding`` is the Python face of libcam (C ABI in
include/cam.h); importing this package does not load the CUDA library, so the
seeded workload generator (``workloads``) is usable on machines without a GPU.
"""
__version__ = "0.1.0"
