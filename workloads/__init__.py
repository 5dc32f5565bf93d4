"""Seeded synthetic inputs for the AKV hot path.

This package only draws random numbers and lays out requests: message
lengths, the cache-operation log a harness policy would issue, raw Q/K/V,
decode pools and model weights.  It holds none of the method's arithmetic
(no rotation, no attention, no visibility rule); the oracle and the CUDA
library both consume the arrays it returns.
"""
from .gen import (  # noqa: F401
    Trajectory,
    DecodeWorkload,
    ModelWorkload,
    bf16_bits,
    tiny_config,
    agent_trajectory,
    rolling_drop_config,
    repos_config,
    decode_workload,
    shared_prefix_batch,
    model_workload,
    random_request,
)
