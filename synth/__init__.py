"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA library's callers."""
from .generate import (WORKLOADS, Inputs, Workload, bf16_bits_to_f32, feature_weight, normal_reference, ar1_reference,
                       gauss_inputs, make_inputs, normal, to_bf16_bits, uniform_bits, uniform, HolaInputs, hola_inputs,
                       HOLA_WORKLOAD)

__all__ = ["WORKLOADS", "Inputs", "Workload", "bf16_bits_to_f32", "feature_weight", "normal_reference", "ar1_reference", "gauss_inputs",
           "make_inputs", "normal", "to_bf16_bits", "uniform_bits", "uniform", "HolaInputs", "hola_inputs",
           "HOLA_WORKLOAD"]
