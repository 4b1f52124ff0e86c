"""Oracle: a plain, slow, obviously correct CPU implementation of one training step.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(the CUDA library and its Python binding) never imports it and shares no code
with it; the two meet only in the seeded input generators of ``synth``.

What it computes is the plain definition of one training step of the method
described in "MegaTrain: Full Precision Training of 100B+ Parameter Large
Language Models on a Single GPU" (chatpaper abstract; chestersoft digest,
"Methodik"): the layer-wise streaming, double buffering, stateless templates
and packed blocks are an exact re-scheduling, so the oracle runs the model
whole, with no streaming. Floating point is numpy, float64 by default (any
dtype may be passed). Matrix products use ``numpy.matmul`` as the library
primitive; everything else is written out step by step.

Pins (tests/test_oracle_*.py): float64 central finite differences, closed-form
losses, attention special cases and brute force, torch-autograd cross-check,
Adam closed forms, independent layout arithmetic. No function here is
"parity unpinned".
"""
from .model import (  # noqa: F401
    Config,
    adam_update,
    bf16_bits_to_float,
    float_to_bf16_bits,
    forward_backward,
    init_params,
    layout,
    loss_only,
    pack_arena,
    train_step,
    unpack_arena,
)
