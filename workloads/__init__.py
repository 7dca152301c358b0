"""Seeded synthetic inputs for the multi-adapter LoRA linear layer.

This package only draws random numbers and lays them out; it performs none of
the layer's arithmetic.  Both the CUDA path (tests, bench) and the float64
oracle read their inputs from here, so the two sides always see the same
values.  Random draws use numpy's PCG64 seeded through ``SeedSequence``; every
tensor comes from its own spawned stream so that adding a tensor never shifts
another one.
"""

from .configs import (  # noqa: F401
    CONFIG_NAMES,
    WIDENING_NAMES,
    Projection,
    Workload,
    bf16_round,
    bf16_bits,
    make_config,
    synth,
)
