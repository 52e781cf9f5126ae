"""Plain, slow, obviously-correct CPU oracle for GGML Q8_0 / Q4_K dequant-GEMV.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  It shares no code, tables or constants with the CUDA library;
both sides read the raw GGML bytes that ``synth`` draws.

Sources (the pages are rustdoc for the ``qualia_core_db`` crate):

* "Module cuda_lane", *Functions: q8_0_gemv_oracle_into* -- the idea of a CPU
  twin that decodes a row-major GGML Q8_0 matrix and multiplies it by x.
* "Module cuda_lane", *Functions: try_q4k_soa_gemv / try_q4k_soa_fused_swiglu /
  try_q4k_soa_ffn_block_residual* -- Q4_K GEMV, the SwiGLU expansion
  ``out[i] = silu(gate_row_i . x) * (up_row_i . x)`` and ``out = residual + FFN(x)``.
* "Module cuda_lane", *Functions: try_q4k_soa_qkv* -- Q, K and V projected from
  the same activation; with grouped-query attention K and V exist only for the
  first n_kv rows.
* "QTensorEngine", *dispatch_output_top1_chunked* / *dispatch_output_topk_chunked*
  -- the output projection with an on-device argmax (k = 1) or top-k epilogue:
  only the winning (id, logit) candidates are read back instead of the logits.
* "weight_cache.rs", *try_cuda_batch_gemv* doc comment -- layouts: W is
  row-major ``n_out x n_in`` (rows = outputs, GGML convention); activations are
  packed ``batch x n_in``; outputs are ``batch x n_out``.
* The block encodings (Q8_0: fp16 d + 32 int8 q, value d*q; Q4_K: fp16 d, fp16
  dmin, 12 bytes of 6-bit scales/mins, 128 bytes of 4-bit quants, value
  ``d*sc_j*q - dmin*m_j``) come from the workload definitions; the pages only
  name ``Q8_0_BLOCK_BYTES`` / ``Q8_0_BLOCK_ELEMS`` ("Module cuda_lane",
  *Constants*).  The byte positions inside a Q4_K superblock follow the
  standard GGML layout (the reading the design notes record).

Precision: dequantised weights are produced in f32 exactly as the definition
states (see each function); every dot product is accumulated in float64 from
exact float64 products of f32 weights and f32 activations.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# IEEE 754 binary16 decoding (own decoder; pinned against numpy's float16 cast
# over all 65536 bit patterns in the oracle tests).
# ---------------------------------------------------------------------------


def fp16_bits_to_f64(bits) -> np.ndarray:
    """Decode IEEE binary16 bit patterns (uint16) to float64.

    sign = bit 15, exponent e = bits 14..10 (bias 15), fraction f = bits 9..0:
      e == 0           -> (-1)^s * 2^-14 * f/1024         (zero / subnormal)
      0 < e < 31       -> (-1)^s * 2^(e-15) * (1 + f/1024)
      e == 31, f == 0  -> (-1)^s * inf
      e == 31, f != 0  -> NaN
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    s = (b >> 15) & 1
    e = (b >> 10) & 0x1F
    f = b & 0x3FF
    sign = np.where(s == 1, -1.0, 1.0)
    sub = sign * np.ldexp(f.astype(np.float64), -24)                     # 2^-14 * f/2^10
    nrm = sign * np.ldexp((1024 + f).astype(np.float64), (e - 25).astype(np.int64))  # 2^(e-15) * (1024+f)/2^10
    inf = sign * np.inf
    out = np.where(e == 0, sub, nrm)
    out = np.where((e == 31) & (f == 0), inf, out)
    out = np.where((e == 31) & (f != 0), np.nan, out)
    return out


def _le_u16(lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    return lo.astype(np.uint16) | (hi.astype(np.uint16) << 8)


# ---------------------------------------------------------------------------
# Q8_0
# ---------------------------------------------------------------------------


def q8_0_dequant(raw, n_out: int, n_in: int) -> np.ndarray:
    """Dequantise a row-major GGML Q8_0 matrix to f32, shape ``(n_out, n_in)``.

    Each 34-byte block: bytes 0..1 = little-endian fp16 ``d``, bytes 2..33 =
    int8 ``q[0..31]``; weight ``k`` of block ``b`` in a row is column ``32b+k``
    and equals ``d * q[k]``.  ``d`` has at most 11 significant bits and ``q``
    at most 8, so the product is exact in f32 (computed here in float64 and
    stored as f32 without rounding).
    """
    if n_in % 32:
        raise ValueError("Q8_0 rows are whole 32-element blocks")
    nb = n_in // 32
    blk = np.asarray(raw, dtype=np.uint8).reshape(n_out, nb, 34)
    d = fp16_bits_to_f64(_le_u16(blk[..., 0], blk[..., 1]))               # (n_out, nb)
    q = blk[..., 2:].view(np.int8).astype(np.float64)                     # (n_out, nb, 32)
    w = d[..., None] * q
    return w.reshape(n_out, n_in).astype(np.float32)


# ---------------------------------------------------------------------------
# Q4_K
# ---------------------------------------------------------------------------


def q4k_scales_mins(scales12: np.ndarray):
    """Unpack the 12 scale bytes of Q4_K superblocks into eight 6-bit scales and mins.

    ``scales12``: uint8 array ``(..., 12)``.  Returns ``(sc, m)``, each ``(..., 8)`` int64.
    For sub-block j < 4:  sc_j = s[j] & 63,  m_j = s[j+4] & 63.
    For sub-block j >= 4: sc_j = (s[j+4] & 0x0F) | ((s[j-4] >> 6) << 4),
                          m_j  = (s[j+4] >> 4)   | ((s[j]   >> 6) << 4).
    """
    s = np.asarray(scales12, dtype=np.uint8).astype(np.int64)
    sc = np.empty(s.shape[:-1] + (8,), dtype=np.int64)
    m = np.empty_like(sc)
    for j in range(8):
        if j < 4:
            sc[..., j] = s[..., j] & 63
            m[..., j] = s[..., j + 4] & 63
        else:
            sc[..., j] = (s[..., j + 4] & 0x0F) | ((s[..., j - 4] >> 6) << 4)
            m[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    return sc, m


def q4k_dequant(raw, n_out: int, n_in: int) -> np.ndarray:
    """Dequantise a row-major GGML Q4_K matrix to f32, shape ``(n_out, n_in)``.

    Superblock of 144 bytes for 256 weights: ``d`` fp16 @0, ``dmin`` fp16 @2,
    12 packed scale/min bytes @4, 128 quant bytes ``qs`` @16.  The 256 weights
    are four 64-weight chunks c = 0..3 using ``qs[32c .. 32c+31]``: weight
    ``64c + l`` (l < 32) is the low nibble of ``qs[32c+l]`` in sub-block
    ``j = 2c``; weight ``64c + 32 + l`` is the high nibble, sub-block ``2c+1``.
    Weight value: ``d*sc_j*q - dmin*m_j`` with q in 0..15.

    Rounding: ``a = d*sc_j*q`` (<= 21 significant bits) and ``b = dmin*m_j``
    (<= 17 bits) are exact in f32; the only rounding is the f32 subtraction
    ``RN_f32(a - b)``.  Here ``a - b`` is formed in float64 and rounded to f32
    once; when the exponents of ``a`` and ``b`` are within 29 bits the float64
    difference is exact, and otherwise the smaller term lies far below half an
    f32 ulp of the larger, so in every case the result equals the correctly
    rounded f32 difference.
    """
    if n_in % 256:
        raise ValueError("Q4_K rows are whole 256-element superblocks")
    nb = n_in // 256
    blk = np.asarray(raw, dtype=np.uint8).reshape(n_out, nb, 144)
    d = fp16_bits_to_f64(_le_u16(blk[..., 0], blk[..., 1]))               # (n_out, nb)
    dmin = fp16_bits_to_f64(_le_u16(blk[..., 2], blk[..., 3]))
    sc, m = q4k_scales_mins(blk[..., 4:16])                               # (n_out, nb, 8)
    qs = blk[..., 16:].astype(np.int64)                                   # (n_out, nb, 128)

    q = np.empty((n_out, nb, 256), dtype=np.int64)
    sub = np.empty((256,), dtype=np.int64)                                # sub-block index of each weight
    for c in range(4):
        chunk = qs[..., 32 * c: 32 * c + 32]
        q[..., 64 * c: 64 * c + 32] = chunk & 0x0F
        q[..., 64 * c + 32: 64 * c + 64] = chunk >> 4
        sub[64 * c: 64 * c + 32] = 2 * c
        sub[64 * c + 32: 64 * c + 64] = 2 * c + 1

    sc_e = sc[..., sub].astype(np.float64)                                # (n_out, nb, 256)
    m_e = m[..., sub].astype(np.float64)
    a = d[..., None] * sc_e * q.astype(np.float64)
    b = dmin[..., None] * m_e
    w = (a - b).astype(np.float32)
    return w.reshape(n_out, n_in)


# ---------------------------------------------------------------------------
# Q6_K
# ---------------------------------------------------------------------------


def q6k_quants(ql: np.ndarray, qh: np.ndarray) -> np.ndarray:
    """The 6-bit quants ``q`` (0..63) of Q6_K superblocks, ``(..., 256)`` int64.

    ``ql``: ``(..., 128)`` bytes of low 4-bit parts, ``qh``: ``(..., 64)`` bytes of
    high 2-bit parts.  The superblock is two halves h = 0, 1 of 128 weights, each
    using ``ql[64h .. 64h+63]`` and ``qh[32h .. 32h+31]``; inside a half, weight
    ``32t + l`` (t = 0..3, l = 0..31) takes
      low 4 bits:  t = 0: low nibble of ql[64h + l],   t = 1: low nibble of ql[64h + 32 + l],
                   t = 2: high nibble of ql[64h + l],  t = 3: high nibble of ql[64h + 32 + l];
      high 2 bits: bits 2t, 2t+1 of qh[32h + l].
    """
    ql = np.asarray(ql, dtype=np.uint8).astype(np.int64)
    qh = np.asarray(qh, dtype=np.uint8).astype(np.int64)
    q = np.empty(ql.shape[:-1] + (256,), dtype=np.int64)
    for h in range(2):
        for t in range(4):
            lo_src = ql[..., 64 * h + 32 * (t & 1): 64 * h + 32 * (t & 1) + 32]
            lo = (lo_src & 0x0F) if t < 2 else (lo_src >> 4)
            hi = (qh[..., 32 * h: 32 * h + 32] >> (2 * t)) & 3
            q[..., 128 * h + 32 * t: 128 * h + 32 * t + 32] = lo | (hi << 4)
    return q


def q6k_dequant(raw, n_out: int, n_in: int) -> np.ndarray:
    """Dequantise a row-major GGML Q6_K matrix to f32, shape ``(n_out, n_in)``.

    Superblock of 210 bytes for 256 weights: ``ql`` (128 bytes of low 4-bit
    parts) @0, ``qh`` (64 bytes of high 2-bit parts) @128, sixteen int8 scales
    @192, fp16 ``d`` @208.  Weight ``e`` of the superblock has the 6-bit quant
    ``q_e`` of :func:`q6k_quants` and belongs to the 16-weight sub-block
    ``e // 16``: its value is ``d * scales[e // 16] * (q_e - 32)``.

    Exactness: ``d`` has at most 11 significant bits, ``|scale| <= 128`` and
    ``|q - 32| <= 32``, so the product has at most 23 significant bits and is
    exact in f32 (formed here in float64 and stored without rounding).
    """
    if n_in % 256:
        raise ValueError("Q6_K rows are whole 256-element superblocks")
    nb = n_in // 256
    blk = np.asarray(raw, dtype=np.uint8).reshape(n_out, nb, 210)
    q = q6k_quants(blk[..., 0:128], blk[..., 128:192])                    # (n_out, nb, 256)
    sc = blk[..., 192:208].view(np.int8).astype(np.float64)                # (n_out, nb, 16)
    d = fp16_bits_to_f64(_le_u16(blk[..., 208], blk[..., 209]))           # (n_out, nb)
    sub = np.arange(256) // 16
    w = d[..., None] * sc[..., sub] * (q - 32).astype(np.float64)
    return w.reshape(n_out, n_in).astype(np.float32)


def get_rows(w: np.ndarray, ids) -> np.ndarray:
    """Embedding lookup: rows ``ids`` of the dequantised matrix ``w``, shape ``(len(ids), n_in)``.

    An id outside ``[0, n_rows)`` has no row; its output row is NaN.
    """
    w = np.asarray(w, dtype=np.float32)
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    out = np.full((ids.size, w.shape[1]), np.nan, dtype=np.float32)
    for i, t in enumerate(ids):
        if 0 <= t < w.shape[0]:
            out[i] = w[t]
    return out


# ---------------------------------------------------------------------------
# GEMV / GEMM / SwiGLU / FFN (float64 accumulation)
# ---------------------------------------------------------------------------


def gemv(w: np.ndarray, x: np.ndarray):
    """``y[b, r] = sum_k w[r, k] * x[b, k]`` in float64, plus ``A[b, r] = sum_k |w[r, k]| |x[b, k]|``.

    ``w``: ``(n_out, n_in)`` f32 dequantised weights (row-major, rows = outputs).
    ``x``: ``(batch, n_in)`` f32 (or float64, used as given, e.g. an exact
    intermediate).  Returns ``(y, A)``, each ``(batch, n_out)`` float64.
    The products of two f32 values are exact in float64; einsum without
    ``optimize`` runs a plain sum-of-products loop on one thread.
    """
    w64 = np.asarray(w, dtype=np.float32).astype(np.float64)
    x64 = np.atleast_2d(np.asarray(x)).astype(np.float64)
    if x64.shape[1] != w64.shape[1]:
        raise ValueError("x has %d columns, W has %d" % (x64.shape[1], w64.shape[1]))
    y = np.einsum("rk,bk->br", w64, x64, optimize=False)
    a = np.einsum("rk,bk->br", np.abs(w64), np.abs(x64), optimize=False)
    return y, a


def silu(z):
    """``silu(z) = z * sigmoid(z) = z / (1 + exp(-z))`` in float64 (math.exp per element)."""
    z = np.asarray(z, dtype=np.float64)
    flat = z.reshape(-1)
    out = np.empty_like(flat)
    for i, v in enumerate(flat):
        v = float(v)
        if v < -709.0:           # exp(-v) overflows float64; silu -> -0 from below
            out[i] = v * math.exp(v) / (1.0 + math.exp(v))
        else:
            out[i] = v / (1.0 + math.exp(-v))
    return out.reshape(z.shape)


def swiglu(w_gate: np.ndarray, w_up: np.ndarray, x: np.ndarray):
    """SwiGLU expansion ``mid[b, i] = silu(g[b, i]) * u[b, i]``, ``g = W_gate x``, ``u = W_up x``.

    Returns a dict with ``mid``, ``g``, ``u``, ``A_g``, ``A_u`` (float64, ``(batch, n_ff)``).
    """
    g, ag = gemv(w_gate, x)
    u, au = gemv(w_up, x)
    return dict(mid=silu(g) * u, g=g, u=u, A_g=ag, A_u=au)


def ffn_residual(w_gate, w_up, w_down, x, residual):
    """Pre-norm-free FFN block with residual: ``out = residual + W_down . swiglu(W_gate x, W_up x)``.

    ``mid`` is the exact (float64) SwiGLU result; ``out`` is float64.  Returns a
    dict with ``out``, ``mid`` and the intermediate quantities of ``swiglu``.
    """
    s = swiglu(w_gate, w_up, x)
    down, a_down = gemv(w_down, s["mid"])  # float64 mid fed straight in
    res = np.atleast_2d(np.asarray(residual, dtype=np.float32)).astype(np.float64)
    s.update(out=res + down, down=down, A_down=a_down)
    return s


def qkv(w_q: np.ndarray, w_k: np.ndarray, w_v: np.ndarray, x: np.ndarray):
    """QKV projection from one activation: ``q = W_q x``, ``k = W_k x``, ``v = W_v x``.

    ``W_q`` is ``n_q x n_in``; ``W_k`` and ``W_v`` are ``n_kv x n_in`` with
    ``n_kv <= n_q`` (grouped-query attention: K and V rows stop at n_kv).  Returns
    a dict with ``q``, ``k``, ``v`` and their ``A_q``, ``A_k``, ``A_v``
    (``sum |w||x|``), all float64.
    """
    if w_k.shape != w_v.shape or w_k.shape[1] != w_q.shape[1] or w_k.shape[0] > w_q.shape[0]:
        raise ValueError("W_k and W_v must be n_kv x n_in with n_kv <= n_q")
    q, a_q = gemv(w_q, x)
    k, a_k = gemv(w_k, x)
    v, a_v = gemv(w_v, x)
    return dict(q=q, k=k, v=v, A_q=a_q, A_k=a_k, A_v=a_v)


def logits_argmax(w: np.ndarray, x: np.ndarray):
    """Output projection with argmax: ``logits = W x`` and, per activation row, the first
    index of the largest logit and that logit.

    A NaN logit counts as larger than every number, so the first NaN wins (the
    numpy.argmax convention).  Returns a dict with ``logits``, ``A`` (``sum |w||x|``),
    ``index`` (int64) and ``value`` (float64).
    """
    logits, a = gemv(w, x)
    index = np.empty(logits.shape[0], dtype=np.int64)
    value = np.empty(logits.shape[0], dtype=np.float64)
    for b, row in enumerate(logits):
        nan = np.flatnonzero(np.isnan(row))
        i = int(nan[0]) if nan.size else int(np.flatnonzero(row == row.max())[0])
        index[b], value[b] = i, row[i]
    return dict(logits=logits, A=a, index=index, value=value)


def logits_topk(w: np.ndarray, x: np.ndarray, k: int):
    """Output projection with top-k: ``logits = W x``; per activation row, the ``k``
    first (index, logit) pairs of the order NaN first, then larger logit first, then
    smaller index first -- the k = 1 case is :func:`logits_argmax`.

    Selection by k passes: each pass takes, among the logits not yet taken, the first
    NaN if there is one, else the first index holding the largest value.  Returns a
    dict with ``logits``, ``A``, ``index`` (int64, ``(batch, k)``) and ``value``
    (float64, ``(batch, k)``).
    """
    logits, a = gemv(w, x)
    n = logits.shape[1]
    if not 1 <= k <= n:
        raise ValueError("k must be in 1..n_vocab")
    index = np.empty((logits.shape[0], k), dtype=np.int64)
    value = np.empty((logits.shape[0], k), dtype=np.float64)
    for b, row in enumerate(logits):
        free = np.ones(n, dtype=bool)
        nan = np.isnan(row)
        for j in range(k):
            cand_nan = np.flatnonzero(free & nan)
            if cand_nan.size:
                i = int(cand_nan[0])
            else:
                top = row[free].max()
                i = int(np.flatnonzero(free & (row == top))[0])
            free[i] = False
            index[b, j], value[b, j] = i, row[i]
    return dict(logits=logits, A=a, index=index, value=value)


def gemm_batch(w: np.ndarray, x: np.ndarray):
    """Batch-prefill GEMM ``Y[m, r] = sum_k X[m, k] * W[r, k]`` in float64 on UNROUNDED f32 X.

    Same definition as :func:`gemv` with ``M`` activation rows; returns ``(Y, A)``.
    """
    return gemv(w, x)
