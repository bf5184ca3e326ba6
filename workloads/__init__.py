"""Seeded synthetic inputs for paged GQA decode with block scoring.

This module is the one piece shared by the CUDA path's tests/bench and the
CPU oracle.  It holds shapes, sequence lengths, seeds and random tensors only:
none of the method's arithmetic (no attention, no mass, no scoring) lives here.
"""
from .gen import (  # noqa: F401
    Workload,
    WORKLOADS,
    workload,
    unit_dirs,
    kv_tokens,
    queries,
    kv_stream,
    BOOST_C,
    synthetic_masses,
)
