"""Seeded synthetic workloads shared by the tests, the oracle runs and bench.py.

This package only draws random numbers and lays them out; it holds none of the
attention arithmetic (no slot formula, no normalisation, no softmax).
"""
from .workloads import CONFIGS, Workload, make_workload, bf16_bits_from_f32, f32_from_bf16_bits

__all__ = ["CONFIGS", "Workload", "make_workload", "bf16_bits_from_f32", "f32_from_bf16_bits"]
