"""Seeded synthetic inputs shared by the CUDA library's tests and the oracle.

Holds no arithmetic of the attention method (see ``gen`` and ``workloads``).
"""
from . import gen, workloads  # noqa: F401
