"""Seeded synthetic inputs for the KDA hot path (shared input data only)."""
from .generator import (  # noqa: F401
    Workload, workload, custom, prefill_inputs, decode_inputs, initial_state,
    splitmix64, splitmix64_int, uniform, normal, raw_bits, STREAMS,
)
