"""CPU oracle for the DoRA factored row norm and stable compose.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference legs, never by the library.
"""
from .dora_oracle import (  # noqa: F401
    BF16, F32, compose, compose_backward, compose_backward_stored, compose_inner,
    compose_inner_stored, compose_stored, decode, dense_ba_bytes, factored_intermediate_bytes,
    magnitude_grad, magnitude_grad_stored, magnitude_scale, naive_compose_f32, norm_and_scale,
    norm_from_partials, norm_partials,
    round_to, round_to_bf16_bits, row_norm,
)
