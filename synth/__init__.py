"""Seeded synthetic workloads shared by the tests, the oracle runs and bench.py.

This package only draws random numbers and lays them out; it holds none of the
attention arithmetic (no slot formula, no normalisation, no softmax).
"""
from .workloads import (CONFIG_ORDER, CONFIGS, Workload, bf16_bits_from_f32, f32_from_bf16_bits, make_workload,
                        to_torch)

__all__ = ["CONFIG_ORDER", "CONFIGS", "Workload", "make_workload", "bf16_bits_from_f32", "f32_from_bf16_bits",
           "to_torch"]
