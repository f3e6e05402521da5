"""Seeded synthetic operands shared by the tests, the bench and the oracle runs.

Holds none of the GEMM's arithmetic: it only draws random values, rounds them
to the 16-bit input format and lays them out in memory in the requested operand
orientation.
"""
from .inputs import K_MAJOR, MN_MAJOR, Problem, WORKLOADS, make_problem, workload  # noqa: F401
