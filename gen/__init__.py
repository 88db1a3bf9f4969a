"""Seeded synthetic workload generator shared by the oracle and the CUDA path (inputs only)."""
from .workload import LayerShape, config, make_shape, make_inputs, make_bias, zipf_bias, bf16_to_f32_np, E384_SWEEP  # noqa: F401
