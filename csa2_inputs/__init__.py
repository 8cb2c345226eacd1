"""Seeded synthetic inputs for CSA2 (shared by the tests, the bench and the oracle).

Holds none of the method's arithmetic: see ``rng`` (counter-based generator)
and ``workloads`` (shapes, seeds, length mixes, page tables, raw tensors).
"""
from . import rng, workloads  # noqa: F401
