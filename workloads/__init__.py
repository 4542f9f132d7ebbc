"""Seeded synthetic workloads shared by tests and bench (inputs only)."""
from .configs import ALL, C0, C1, C2, C3, C4, Workload  # noqa: F401
