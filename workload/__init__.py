"""Seeded synthetic inputs for the routed mixture-of-experts FFN.

This package only draws random numbers and encodes them into the storage
formats the method consumes (int4 affine groups, fp16 router weights, bf16
hidden states, logit-bias traces).  It holds none of the method's arithmetic:
no router, no top-k, no dequantised matvec, no combine.  Both the CPU oracle
(``oracle/``) and the CUDA library consume what it produces.
"""

from .gen import (  # noqa: F401
    Shape,
    TINY,
    FULL,
    derive_seed,
    quantise_rows,
    gen_layer,
    gen_hidden,
    zipf_reuse_targets,
    mixture_targets,
    bias_from_targets,
)
