"""Seeded synthetic inputs for the verify step (shared by tests and the bench).

This package holds none of the method's arithmetic: it draws Gaussian logits
and picks the shapes, per-row K and peaked token ids of each workload.  The
draft tokens (and, for the LM-head workload, the draft probabilities) are not
made here: they come from a draft-side sampler, the oracle's in the tests and
the library's in the bench.
"""
from .synth import (CONFIGS, Workload, bf16_bits_to_f32, f32_to_bf16_bits, make_config,
                    make_workload)

__all__ = ["CONFIGS", "Workload", "bf16_bits_to_f32", "f32_to_bf16_bits", "make_config",
           "make_workload"]
