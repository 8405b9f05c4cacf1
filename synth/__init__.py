"""Seeded synthetic inputs shared by tests, bench.py and the smoke check."""
from .inputs import WORKLOADS, Workload, make_inputs, small_workload, to_numpy_bits  # noqa: F401
