"""Seeded synthetic inputs for the tiered KV-cache decode step.

Shared by the CPU oracle (tests), the CUDA path's tests and bench.py. It holds
none of the method's arithmetic: only generators of inputs that are pure
functions of (seed, indices), identical on CPU and CUDA tensors.
"""
from .philox import normal_f32, normal_table, philox4x32, uniform_u16, uniform_u32
from .workloads import (BATCH32, CHAIN7B, MHA16K, TINY, WORKLOADS, Workload,
                        long128k)

__all__ = ["philox4x32", "uniform_u16", "uniform_u32", "normal_f32", "normal_table",
           "Workload", "TINY", "CHAIN7B", "BATCH32", "MHA16K", "long128k", "WORKLOADS"]
