"""Error bounds the GPU results are held to (derived from the f32 arithmetic).

GEMV: |y - y_ref| <= 1e-5 * A, A = sum_k |w_k| |x_k| (the stated GEMV bound).

SwiGLU: mid = silu(g) * u with g, u each within 1e-5 * A_g, 1e-5 * A_u of the
exact values; |silu'| <= 1.1 everywhere, and expf adds a few ulp:
    eps_mid = 1.1 |u| 1e-5 A_g + |silu(g)| 1e-5 A_u + 1e-6 |mid|.

FFN: out = residual + W_down . mid.  The down GEMV on the f32 mid adds
1e-5 * sum_j |Wd_rj| |mid_j|, the mid error propagates through |Wd|, and the
final residual add rounds once:
    |out - out_ref| <= 1e-5 sum_j |Wd_rj| |mid_j| + sum_j |Wd_rj| eps_mid_j + 2^-24 |out_ref|.

Batch GEMM (bf16 operands, f32 accumulation): |Y - Y_ref| <= 4e-3 * A.
"""
import numpy as np

import oracle


def gemv_excess(y, y_ref, a, rel=1e-5):
    """Largest |y - y_ref| / (rel * A) (<= 1 passes); exact zeros are required where A == 0."""
    y = np.asarray(y, dtype=np.float64).reshape(y_ref.shape)
    err = np.abs(y - y_ref)
    bound = rel * a
    if np.any((bound == 0) & (err != 0)):
        return np.inf
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.where(bound > 0, err / np.where(bound > 0, bound, 1), 0.0)
    return float(r.max()) if r.size else 0.0


def swiglu_eps(s):
    return (1.1 * np.abs(s["u"]) * 1e-5 * s["A_g"] + np.abs(oracle.silu(s["g"])) * 1e-5 * s["A_u"]
            + 1e-6 * np.abs(s["mid"]))


def ffn_bound(o, wd_deq):
    eps = swiglu_eps(o)                                     # (batch, n_ff)
    _, a_mid = oracle.gemv(wd_deq, np.abs(o["mid"]))        # sum_j |Wd_rj| |mid_j|
    _, a_eps = oracle.gemv(wd_deq, eps)                     # sum_j |Wd_rj| eps_j
    return 1e-5 * a_mid + a_eps + 2.0 ** -24 * np.abs(o["out"])
