"""Seeded synthetic inputs for the P-EAGLE drafting workloads.

This package only draws random numbers and lays them out. It holds none of
the method's arithmetic: no norm, projection, attention, COD rule or verify
step lives here. Both the CPU oracle (through the tests) and the CUDA path
receive the arrays it returns.
"""
from .workloads import WORKLOADS, Workload, workload
from .generate import (
    bf16_round,
    make_weights,
    make_decode_inputs,
    make_train_inputs,
    make_targets_with_accept,
    make_request_cache,
    draw_accept_lengths,
)

__all__ = [
    "WORKLOADS", "Workload", "workload", "bf16_round", "make_weights",
    "make_decode_inputs", "make_train_inputs", "make_targets_with_accept",
    "make_request_cache", "draw_accept_lengths",
]
