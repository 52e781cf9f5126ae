"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module only draws random numbers and lays them out as raw GGML block
bytes; it holds none of the dequantisation or GEMV arithmetic.  Both the CPU
oracle (``oracle/``) and the CUDA path (``ggml_quantized_dequant_gb300``) read
the bytes it produces, each with its own decoder.

Block encodings (GGML, little-endian), as the workload descriptions state them:

* Q8_0 block, 34 bytes for 32 weights: fp16 scale ``d`` at byte 0, then 32
  signed int8 quants ``q`` at bytes 2..33; weight ``k`` of block ``b`` is column
  ``32*b + k`` of its row.
* Q4_K superblock, 144 bytes for 256 weights: fp16 ``d`` at byte 0, fp16
  ``dmin`` at byte 2, 12 bytes packing eight 6-bit scales and eight 6-bit mins
  at bytes 4..15, 128 bytes of 4-bit quants at bytes 16..143.
* Q6_K superblock, 210 bytes for 256 weights: 128 bytes of low 4-bit quant parts
  at bytes 0..127, 64 bytes of high 2-bit parts at bytes 128..191, sixteen int8
  scales at bytes 192..207, fp16 ``d`` at bytes 208..209.

Drawing the 12 scale bytes and the 128 quant bytes as independent uniform
bytes makes every 6-bit scale, 6-bit min and 4-bit quant uniform over its whole
range, because each of those fields is a fixed set of distinct bits; the
generator therefore never has to pack a field.  The same holds for the Q6_K
quant bytes (every 6-bit quant uniform over 0..63).

Seeds: every array is drawn from ``numpy.random.default_rng([config, *path])``
(``rng_for``), so each workload matrix has its own reproducible stream.
Within one matrix the draw order is: scale plane(s), then quant bytes.
"""
from __future__ import annotations

import numpy as np

Q8_0_BLOCK_ELEMS = 32
Q8_0_BLOCK_BYTES = 34
Q4K_BLOCK_ELEMS = 256
Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_ELEMS = 256
Q6K_BLOCK_BYTES = 210


def rng_for(config: int, *path: int) -> np.random.Generator:
    """The generator for one array of one workload: ``default_rng([config, *path])``."""
    return np.random.default_rng([int(config), *[int(p) for p in path]])


def _fp16_le_bytes(values: np.ndarray) -> np.ndarray:
    """Round to IEEE binary16 (numpy's round-to-nearest-even cast) and return the LE bytes."""
    h = np.asarray(values, dtype=np.float64).astype("<f2")
    return h.view(np.uint8).reshape(*h.shape, 2)


def q8_0_blocks(rng: np.random.Generator, n_out: int, n_in: int,
                d_range=(1e-3, 2e-2), q_range=(-127, 127)) -> np.ndarray:
    """Random GGML Q8_0 matrix as raw bytes, shape ``(n_out, n_in//32*34)`` uint8.

    ``d`` ~ U[d_range] cast to fp16; ``q`` ~ U{q_range} (inclusive) as int8.
    """
    if n_in % Q8_0_BLOCK_ELEMS:
        raise ValueError("n_in must be a multiple of 32 for Q8_0")
    nb = n_in // Q8_0_BLOCK_ELEMS
    d = rng.uniform(d_range[0], d_range[1], size=(n_out, nb))
    q = rng.integers(q_range[0], q_range[1] + 1, size=(n_out, nb, Q8_0_BLOCK_ELEMS), dtype=np.int8)
    out = np.empty((n_out, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    out[..., 0:2] = _fp16_le_bytes(d)
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(n_out, nb * Q8_0_BLOCK_BYTES)


def q4k_blocks(rng: np.random.Generator, n_out: int, n_in: int,
               d_range=(1e-3, 1e-2), dmin_range=(1e-3, 1e-2)) -> np.ndarray:
    """Random GGML Q4_K matrix as raw bytes, shape ``(n_out, n_in//256*144)`` uint8.

    ``d``, ``dmin`` ~ U[range] cast to fp16; the 12 scale/min bytes and the 128
    quant bytes are uniform random bytes (so every 6-bit scale/min and every
    4-bit quant is uniform over its range).
    """
    if n_in % Q4K_BLOCK_ELEMS:
        raise ValueError("n_in must be a multiple of 256 for Q4_K")
    nb = n_in // Q4K_BLOCK_ELEMS
    d = rng.uniform(d_range[0], d_range[1], size=(n_out, nb))
    dmin = rng.uniform(dmin_range[0], dmin_range[1], size=(n_out, nb))
    scales = rng.integers(0, 256, size=(n_out, nb, 12), dtype=np.uint8)
    qs = rng.integers(0, 256, size=(n_out, nb, 128), dtype=np.uint8)
    out = np.empty((n_out, nb, Q4K_BLOCK_BYTES), dtype=np.uint8)
    out[..., 0:2] = _fp16_le_bytes(d)
    out[..., 2:4] = _fp16_le_bytes(dmin)
    out[..., 4:16] = scales
    out[..., 16:] = qs
    return out.reshape(n_out, nb * Q4K_BLOCK_BYTES)


def q6k_blocks(rng: np.random.Generator, n_out: int, n_in: int,
               d_range=(1e-3, 1e-2), scale_range=(-128, 127)) -> np.ndarray:
    """Random GGML Q6_K matrix as raw bytes, shape ``(n_out, n_in//256*210)`` uint8.

    ``d`` ~ U[d_range] cast to fp16; the sixteen int8 scales ~ U{scale_range}; the
    192 quant bytes are uniform random bytes (every 6-bit quant uniform over 0..63).
    Draw order: d, scales, quant bytes.
    """
    if n_in % Q6K_BLOCK_ELEMS:
        raise ValueError("n_in must be a multiple of 256 for Q6_K")
    nb = n_in // Q6K_BLOCK_ELEMS
    d = rng.uniform(d_range[0], d_range[1], size=(n_out, nb))
    sc = rng.integers(scale_range[0], scale_range[1] + 1, size=(n_out, nb, 16), dtype=np.int8)
    qs = rng.integers(0, 256, size=(n_out, nb, 192), dtype=np.uint8)
    out = np.empty((n_out, nb, Q6K_BLOCK_BYTES), dtype=np.uint8)
    out[..., 0:192] = qs
    out[..., 192:208] = sc.view(np.uint8)
    out[..., 208:210] = _fp16_le_bytes(d)
    return out.reshape(n_out, nb * Q6K_BLOCK_BYTES)


def activations(rng: np.random.Generator, rows: int, n: int) -> np.ndarray:
    """f32 activations ~ N(0, 1), shape ``(rows, n)``."""
    return rng.standard_normal(size=(rows, n)).astype(np.float32)


# ---------------------------------------------------------------------------
# The workloads (shapes, distributions and seeds), one function per config.
# ---------------------------------------------------------------------------

#: Config 0: Q8_0 GEMV, batch 1, W 256 x 512, seed 0.
C0 = dict(n_out=256, n_in=512)
#: 3B-class decode shapes: hidden 3072, FFN 8192.
N_EMBD = 3072
N_FF = 8192
#: Distinct matrices per set in the cycled workloads (one per layer).
N_LAYERS = 28


def config0():
    """Config 0: ``(W_bytes, x)`` with W 256x512 Q8_0 and x (1, 512); all from seed 0."""
    rng = np.random.default_rng(0)
    w = q8_0_blocks(rng, C0["n_out"], C0["n_in"])
    x = activations(rng, 1, C0["n_in"])
    return w, x


def config1_up(t: int) -> np.ndarray:
    """Config 1, layer ``t``'s up matrix: Q8_0, n_in=3072 -> n_out=8192."""
    return q8_0_blocks(rng_for(1, 0, t), N_FF, N_EMBD)


def config1_down(t: int) -> np.ndarray:
    """Config 1, layer ``t``'s down matrix: Q8_0, n_in=8192 -> n_out=3072."""
    return q8_0_blocks(rng_for(1, 1, t), N_EMBD, N_FF)


def config1_x() -> np.ndarray:
    """Config 1 activation (1, 3072)."""
    return activations(rng_for(1, 2), 1, N_EMBD)


def config2_w(t: int) -> np.ndarray:
    """Config 2, copy ``t``: Q4_K, n_in=3072 -> n_out=8192."""
    return q4k_blocks(rng_for(2, 0, t), N_FF, N_EMBD)


def config2_x() -> np.ndarray:
    """Config 2 activation (1, 3072)."""
    return activations(rng_for(2, 1), 1, N_EMBD)


def config3_layer(t: int):
    """Config 3, layer ``t``: ``(W_gate, W_up, W_down)`` Q4_K bytes (3072->8192, 3072->8192, 8192->3072)."""
    return (q4k_blocks(rng_for(3, 0, t), N_FF, N_EMBD),
            q4k_blocks(rng_for(3, 1, t), N_FF, N_EMBD),
            q4k_blocks(rng_for(3, 2, t), N_EMBD, N_FF))


def config3_x_residual():
    """Config 3 ``(x, residual)``, each (1, 3072) ~ N(0, 1)."""
    return activations(rng_for(3, 3), 1, N_EMBD), activations(rng_for(3, 4), 1, N_EMBD)


#: Fused QKV workload: 3B-class grouped-query attention, 24 query heads and 8 KV heads of 128.
N_Q = 3072
N_KV = 1024


def qkv_layer(t: int):
    """QKV layer ``t``: ``(W_q, W_k, W_v)`` Q4_K bytes (3072->3072, 3072->1024, 3072->1024)."""
    return (q4k_blocks(rng_for(5, 0, t), N_Q, N_EMBD),
            q4k_blocks(rng_for(5, 1, t), N_KV, N_EMBD),
            q4k_blocks(rng_for(5, 2, t), N_KV, N_EMBD))


#: Output projection workload: a 3B-class vocabulary.
N_VOCAB = 128256


def output_projection():
    """Output projection ``(W, x)``: Q8_0 bytes 3072 -> 128256 (config-1 distributions) and x (1, 3072)."""
    return q8_0_blocks(rng_for(6, 0), N_VOCAB, N_EMBD), activations(rng_for(6, 1), 1, N_EMBD)


#: Config 4 token counts.
C4_M = (16, 64, 512)


def config4_w(kind: int, t: int = 0) -> np.ndarray:
    """Config 4 weight: ``kind`` 0 = 3072->8192, 1 = 8192->3072 (Q8_0, config-1 distributions)."""
    if kind == 0:
        return q8_0_blocks(rng_for(4, 0, t), N_FF, N_EMBD)
    return q8_0_blocks(rng_for(4, 1, t), N_EMBD, N_FF)


def config4_x(kind: int, m: int) -> np.ndarray:
    """Config 4 activations ``(m, n_in)`` for weight ``kind``."""
    n_in = N_EMBD if kind == 0 else N_FF
    return activations(rng_for(4, 2 + kind, m), m, n_in)


def q6k_output_projection():
    """Q6_K output projection ``(W, x)``: 3072 -> 128256 (a 3B-class vocabulary, Q6_K
    as quantised files keep the output and embedding tables) and x (1, 3072)."""
    return q6k_blocks(rng_for(7, 0), N_VOCAB, N_EMBD), activations(rng_for(7, 1), 1, N_EMBD)


def token_ids(rng: np.random.Generator, n: int, n_vocab: int = N_VOCAB) -> np.ndarray:
    """``n`` token ids uniform over the vocabulary (int32), for embedding lookups."""
    return rng.integers(0, n_vocab, size=n).astype(np.int32)
