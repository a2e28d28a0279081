"""GB300-native (sm_103a) FMPQ W4Ax GEMM: fused activation quantizer, offline INT4 weight
packing and the mixed INT4/INT8-activation x INT4-weight GEMM, behind a C ABI
(include/fmpq.h). ``fmpq`` is the thin Python binding; ``workloads`` draws seeded inputs."""
from . import workloads  # noqa: F401  (no CUDA dependency)

__all__ = ["workloads", "fmpq", "build"]
