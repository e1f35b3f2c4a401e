"""Seeded synthetic inputs for the weight-stream workloads.

This module is the only code shared by the CUDA path's callers and the CPU
oracle. It draws random numbers and nothing else: no quantization, no
dequantization, no products. Every generator is keyed by (seed, stream id) so
the same tensor can be regenerated on either side.

Distributions follow the workloads the pages measure (weights ~ N(0, 0.02),
activations ~ N(0, 1) in BF16, top-8 routing over 512 experts drawn uniformly
at random because no trained router exists here).
"""
from .gen import (  # noqa: F401
    stream_seed,
    weight_fp32,
    activation_bf16,
    expert_ids,
    route_weights,
)
