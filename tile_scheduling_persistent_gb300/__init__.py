"""Deterministic attention backward (DASH tile schedules) for GB300 / sm_103a.

The compute lives in ``libdash.so`` (hand-written CUDA, C ABI declared in
``include/dash.h``); ``tile_scheduling_persistent_gb300.dash`` is the thin
ctypes binding.  Importing this package does not load the library; the first
call into ``dash`` does, and fails loudly if it has not been built.
"""
from .inputs import SCHEDULE_IDS, WORKLOADS, make_qkvdo, make_workload_inputs  # noqa: F401
