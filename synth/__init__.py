"""Seeded synthetic inputs shared by the oracle, the tests and the bench.

This package holds random-number generation and workload shapes only: none of
the attention arithmetic lives here, so the oracle and the CUDA path can both
consume its output without sharing any of the method's code.
"""
from .rng import normal, splitmix64_outputs, uniform01
from .workloads import WORKLOADS, Inputs, Workload, make_inputs, bf16_round, bf16_bits_to_f32, f32_to_bf16_bits
from .workloads import MSA_WORKLOADS, MsaInputs, MsaWorkload, make_msa_inputs, with_affine_params

__all__ = [
    "normal", "splitmix64_outputs", "uniform01",
    "WORKLOADS", "Inputs", "Workload", "make_inputs",
    "bf16_round", "bf16_bits_to_f32", "f32_to_bf16_bits",
    "MSA_WORKLOADS", "MsaInputs", "MsaWorkload", "make_msa_inputs", "with_affine_params",
]
