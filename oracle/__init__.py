"""CPU oracle for the dequant-GEMV path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The CUDA library never calls it and
shares no code with it.
"""
from .ggml_oracle import (  # noqa: F401
    fp16_bits_to_f64,
    q8_0_dequant,
    q4k_scales_mins,
    q4k_dequant,
    q6k_quants,
    q6k_dequant,
    get_rows,
    gemv,
    silu,
    swiglu,
    ffn_residual,
    qkv,
    logits_argmax,
    logits_topk,
    gemm_batch,
)
