"""Seeded synthetic inputs (workload tables, top-K streams, row contents) shared by the tests,
the oracle runs and bench.py.  Holds no resolver arithmetic."""
from . import content, workloads  # noqa: F401
