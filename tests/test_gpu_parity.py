"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bars (stated in the workload definition):
* dequantised weights: bit-exact (compared as raw f32 bits);
* GEMV / SwiGLU / FFN: |y - y_ref| <= 1e-5 * sum|w||x| (FFN / SwiGLU with the
  propagated bound of tests/_bounds.py);
* tensor-core batch GEMM: |Y - Y_ref| <= 4e-3 * sum|w||x| against the fp64
  oracle on the unrounded activations.
Shapes cover several tiles plus ragged tails, batch 1..8, and the full
workload sizes in the launch configuration the bench times.
"""
import numpy as np
import pytest

import oracle
import synth
from _bounds import ffn_bound, gemv_excess, swiglu_eps

pytestmark = pytest.mark.gpu


def _dev():
    import torch
    return torch.device("cuda")


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(_dev())


def _nan(*shape):
    import torch
    return torch.full(shape, float("nan"), dtype=torch.float32, device=_dev())


def _np(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


# ------------------------------------------------------------------ dequant

@pytest.mark.parametrize("n_out,n_in", [(256, 512), (3, 96), (37, 1056), (8192, 3072)])
def test_q8_0_dequant_bit_exact(cuda_lib, n_out, n_in):
    qdq = cuda_lib
    wb = synth.q8_0_blocks(np.random.default_rng(n_out * 7 + n_in), n_out, n_in)
    W = qdq.upload_q8_0(wb, n_out, n_in)
    out = _nan(n_out, n_in)
    qdq.q8_0_dequant(W, out, n_out, n_in)
    ref = oracle.q8_0_dequant(wb, n_out, n_in)
    assert np.array_equal(_np(out).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("n_out,n_in", [(3, 256), (37, 768), (8192, 3072)])
def test_q4k_dequant_bit_exact(cuda_lib, n_out, n_in):
    qdq = cuda_lib
    wb = synth.q4k_blocks(np.random.default_rng(n_out * 5 + n_in), n_out, n_in)
    W = qdq.upload_q4k(wb, n_out, n_in)
    out = _nan(n_out, n_in)
    qdq.q4k_dequant(W, out, n_out, n_in)
    ref = oracle.q4k_dequant(wb, n_out, n_in)
    assert np.array_equal(_np(out).view(np.uint32), ref.view(np.uint32))


def test_q4k_dequant_extreme_scales_bit_exact(cuda_lib):
    # largest dmin and smallest d: the f32 subtraction has to round
    qdq = cuda_lib
    wb = synth.q4k_blocks(np.random.default_rng(3), 16, 512, d_range=(6e-5, 6e-5), dmin_range=(6e4, 6e4))
    W = qdq.upload_q4k(wb, 16, 512)
    out = _nan(16, 512)
    qdq.q4k_dequant(W, out, 16, 512)
    assert np.array_equal(_np(out).view(np.uint32), oracle.q4k_dequant(wb, 16, 512).view(np.uint32))


# ------------------------------------------------------------------ GEMV

Q8_SHAPES = [(256, 512, 1), (1, 32, 1), (3, 96, 1), (157, 800, 1), (300, 4096, 3), (64, 512, 8),
             (33, 8192, 8), (1000, 1024, 2),
             # the largest row the batch-1 pipeline takes (16 slice warps), rows it hands to the
             # general kernel (n_in % 256 != 0, n_in > 16384), and the largest n_in accepted
             (40, 16384, 1), (150, 20000, 1), (24, 32768, 1), (16, 32768, 8)]


@pytest.mark.parametrize("n_out,n_in,batch", Q8_SHAPES)
def test_q8_0_gemv_parity(cuda_lib, n_out, n_in, batch):
    qdq = cuda_lib
    rng = np.random.default_rng(n_out + 3 * n_in + batch)
    wb = synth.q8_0_blocks(rng, n_out, n_in)
    x = synth.activations(rng, batch, n_in)
    W = qdq.upload_q8_0(wb, n_out, n_in)
    y = _nan(batch, n_out)
    qdq.q8_0_gemv(W, _t(x), y, n_out, n_in, batch)
    y_ref, a = oracle.gemv(oracle.q8_0_dequant(wb, n_out, n_in), x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


def test_q8_0_gemv_config0_seed0(cuda_lib):
    qdq = cuda_lib
    wb, x = synth.config0()
    W = qdq.upload_q8_0(wb, 256, 512)
    y = _nan(1, 256)
    qdq.q8_0_gemv(W, _t(x), y, 256, 512, 1)
    y_ref, a = oracle.gemv(oracle.q8_0_dequant(wb, 256, 512), x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


@pytest.mark.parametrize("which", ["up", "down"])
def test_q8_0_gemv_full_size(cuda_lib, which):
    qdq = cuda_lib
    if which == "up":
        n_out, n_in, wb, x = 8192, 3072, synth.config1_up(0), synth.config1_x()
    else:
        n_out, n_in, wb = 3072, 8192, synth.config1_down(0)
        x = synth.activations(synth.rng_for(1, 3), 1, 8192)
    W = qdq.upload_q8_0(wb, n_out, n_in)
    y = _nan(1, n_out)
    qdq.q8_0_gemv(W, _t(x), y, n_out, n_in, 1)
    y_ref, a = oracle.gemv(oracle.q8_0_dequant(wb, n_out, n_in), x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


def test_q8_0_gemv_extreme_quants(cuda_lib):
    # q = -128 and +127, negative and large scales
    qdq = cuda_lib
    n_out, n_in = 40, 256
    wb = synth.q8_0_blocks(np.random.default_rng(5), n_out, n_in, d_range=(-3e4, 3e4), q_range=(-128, 127))
    blk = wb.reshape(n_out, n_in // 32, 34)
    blk[::2, :, 2:] = np.uint8(0x80)  # every other row all -128
    x = synth.activations(np.random.default_rng(6), 2, n_in)
    W = qdq.upload_q8_0(wb, n_out, n_in)
    y = _nan(2, n_out)
    qdq.q8_0_gemv(W, _t(x), y, n_out, n_in, 2)
    y_ref, a = oracle.gemv(oracle.q8_0_dequant(wb, n_out, n_in), x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


def test_gemv_zero_x_gives_exact_zero(cuda_lib):
    qdq = cuda_lib
    wb = synth.q8_0_blocks(np.random.default_rng(8), 64, 512)
    W = qdq.upload_q8_0(wb, 64, 512)
    y = _nan(1, 64)
    qdq.q8_0_gemv(W, _t(np.zeros((1, 512), np.float32)), y, 64, 512, 1)
    assert np.all(_np(y) == 0.0)


Q4_SHAPES = [(1, 256, 1), (5, 512, 1), (157, 2048, 1), (300, 3072, 4), (64, 512, 8), (33, 8192, 8),
             (1000, 1280, 2), (40, 16384, 1), (24, 32768, 1), (16, 32768, 8)]


@pytest.mark.parametrize("n_out,n_in,batch", Q4_SHAPES)
def test_q4k_gemv_parity(cuda_lib, n_out, n_in, batch):
    qdq = cuda_lib
    rng = np.random.default_rng(n_out + 5 * n_in + batch)
    wb = synth.q4k_blocks(rng, n_out, n_in)
    x = synth.activations(rng, batch, n_in)
    W = qdq.upload_q4k(wb, n_out, n_in)
    y = _nan(batch, n_out)
    qdq.q4k_gemv(W, _t(x), y, n_out, n_in, batch)
    y_ref, a = oracle.gemv(oracle.q4k_dequant(wb, n_out, n_in), x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


def test_q4k_gemv_full_size_config2(cuda_lib):
    qdq = cuda_lib
    wb, x = synth.config2_w(0), synth.config2_x()
    W = qdq.upload_q4k(wb, 8192, 3072)
    y = _nan(1, 8192)
    qdq.q4k_gemv(W, _t(x), y, 8192, 3072, 1)
    y_ref, a = oracle.gemv(oracle.q4k_dequant(wb, 8192, 3072), x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


def test_q4k_gemv_cancelling_weights(cuda_lib):
    # d*sc*q close to dmin*m for most weights: sum|w||x| is small relative to the
    # separate terms, the hard case for the factored sub-block sum
    qdq = cuda_lib
    n_out, n_in = 64, 1024
    rng = np.random.default_rng(11)
    wb = synth.q4k_blocks(rng, n_out, n_in, d_range=(1e-2, 1e-2), dmin_range=(1e-2, 1e-2))
    sb = wb.reshape(n_out, n_in // 256, 144)
    # every sc_j = 4 and m_j = 32 (bytes 0..3: sc 4; bytes 4..7: m 32 plus the top bits 2 of
    # m_4..7; bytes 8..11: low nibbles sc 4, m 0), d == dmin, so a quant of 8 gives exactly 0
    sb[..., 4:16] = np.array([4, 4, 4, 4, 160, 160, 160, 160, 4, 4, 4, 4], dtype=np.uint8)
    sb[..., 16:] = np.where(rng.random(sb[..., 16:].shape) < 0.8, 0x88, sb[..., 16:]).astype(np.uint8)
    x = synth.activations(rng, 1, n_in)
    W = qdq.upload_q4k(wb, n_out, n_in)
    y = _nan(1, n_out)
    qdq.q4k_gemv(W, _t(x), y, n_out, n_in, 1)
    w = oracle.q4k_dequant(wb, n_out, n_in)
    y_ref, a = oracle.gemv(w, x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


# ------------------------------------------------------------------ SwiGLU / FFN

@pytest.mark.parametrize("n_ff,n_embd,batch", [(512, 256, 1), (1000, 512, 3), (8192, 3072, 1)])
def test_q4k_swiglu_parity(cuda_lib, n_ff, n_embd, batch):
    qdq = cuda_lib
    rng = np.random.default_rng(n_ff + n_embd + batch)
    g, u = synth.q4k_blocks(rng, n_ff, n_embd), synth.q4k_blocks(rng, n_ff, n_embd)
    x = synth.activations(rng, batch, n_embd)
    Wg, Wu = qdq.upload_q4k(g, n_ff, n_embd), qdq.upload_q4k(u, n_ff, n_embd)
    mid = _nan(batch, n_ff)
    qdq.q4k_swiglu(Wg, Wu, _t(x), mid, n_ff, n_embd, batch)
    s = oracle.swiglu(oracle.q4k_dequant(g, n_ff, n_embd), oracle.q4k_dequant(u, n_ff, n_embd), x)
    err = np.abs(_np(mid) - s["mid"])
    assert np.all(err <= swiglu_eps(s))


def _ffn_case(qdq, n_embd, n_ff, batch, seed, in_place=False, layer=None):
    if layer is not None:
        g, u, d = synth.config3_layer(layer)
        x, res = synth.config3_x_residual()
    else:
        rng = np.random.default_rng(seed)
        g, u, d = (synth.q4k_blocks(rng, n_ff, n_embd), synth.q4k_blocks(rng, n_ff, n_embd),
                   synth.q4k_blocks(rng, n_embd, n_ff))
        x, res = synth.activations(rng, batch, n_embd), synth.activations(rng, batch, n_embd)
    Wg, Wu, Wd = qdq.upload_q4k(g, n_ff, n_embd), qdq.upload_q4k(u, n_ff, n_embd), qdq.upload_q4k(d, n_embd, n_ff)
    mid = _nan(batch, n_ff)
    res_d = _t(res)
    out = res_d if in_place else _nan(batch, n_embd)
    qdq.q4k_ffn_residual(Wg, Wu, Wd, _t(x), res_d, out, mid, n_embd, n_ff, batch)
    wd = oracle.q4k_dequant(d, n_embd, n_ff)
    o = oracle.ffn_residual(oracle.q4k_dequant(g, n_ff, n_embd), oracle.q4k_dequant(u, n_ff, n_embd), wd, x, res)
    err = np.abs(_np(out) - o["out"])
    assert np.all(err <= ffn_bound(o, wd))
    assert np.all(np.abs(_np(mid) - o["mid"]) <= swiglu_eps(o))


@pytest.mark.parametrize("n_embd,n_ff,batch", [(256, 512, 1), (512, 1280, 2), (768, 2048, 5), (512, 1024, 8)])
def test_q4k_ffn_residual_parity(cuda_lib, n_embd, n_ff, batch):
    _ffn_case(cuda_lib, n_embd, n_ff, batch, seed=n_embd + n_ff + batch)


def test_q4k_ffn_residual_in_place(cuda_lib):
    _ffn_case(cuda_lib, 512, 1024, 2, seed=99, in_place=True)


def test_q4k_ffn_residual_full_size_config3(cuda_lib):
    _ffn_case(cuda_lib, 3072, 8192, 1, seed=0, layer=0)


# ------------------------------------------------------------------ batch GEMM (tensor cores)

def _gemm_case(qdq, n_out, n_in, M, wb=None, X=None, sample_rows=None, seed=0):
    import torch
    rng = np.random.default_rng(seed)
    if wb is None:
        wb = synth.q8_0_blocks(rng, n_out, n_in)
    if X is None:
        X = synth.activations(rng, M, n_in)
    W = qdq.upload_q8_0(wb, n_out, n_in)
    Y = _nan(M, n_out)
    ws = torch.zeros(qdq.gemm_batch_workspace_bytes(M, n_out, n_in), dtype=torch.uint8, device=_dev())
    qdq.q8_0_gemm_batch(W, _t(X), Y, ws, n_out, n_in, M)
    Yh = _np(Y)
    rows = np.arange(M) if sample_rows is None else sample_rows
    Y_ref, A = oracle.gemm_batch(oracle.q8_0_dequant(wb, n_out, n_in), X[rows])
    assert gemv_excess(Yh[rows], Y_ref, A, rel=4e-3) <= 1.0
    assert qdq.pipeline_timeouts() == 0


@pytest.mark.parametrize("M", [1, 16, 20, 32, 64, 100, 200, 257, 512, 1000])
def test_q8_0_gemm_batch_parity_small(cuda_lib, M):
    _gemm_case(cuda_lib, 256, 512, M, seed=M)


@pytest.mark.parametrize("n_out,n_in,M", [(384, 1024, 33), (128, 64, 16), (1024, 2048, 130), (256, 320, 40),
                                           (128, 448, 17), (512, 192, 300), (128, 64, 40), (256, 192, 48)])
def test_q8_0_gemm_batch_parity_shapes(cuda_lib, n_out, n_in, M):
    _gemm_case(cuda_lib, n_out, n_in, M, seed=n_out + M)


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("M", [16, 32, 64, 512])
def test_q8_0_gemm_batch_full_size_config4(cuda_lib, kind, M):
    n_out, n_in = (8192, 3072) if kind == 0 else (3072, 8192)
    # M = 512: 32 rows from each 256-token tile (every output column, so every weight
    # tile and K split, enters each sampled row)
    sample = None if M <= 64 else np.sort(np.concatenate(
        [t * 256 + np.random.default_rng(M + t).choice(256, 32, replace=False) for t in range(M // 256)]))
    _gemm_case(cuda_lib, n_out, n_in, M, wb=synth.config4_w(kind), X=synth.config4_x(kind, M),
               sample_rows=sample)


@pytest.mark.parametrize("n_out,n_in,M", [(8192, 3072, 600), (3072, 8192, 384), (1024, 1024, 160)])
def test_q8_0_gemm_batch_token_tiles(cuda_lib, n_out, n_in, M):
    # above 128 tokens the token tile is 128, 192 or 256, whichever the launch plan
    # estimates fastest: 8192 x 600 has more output tiles than SMs (no K split, two
    # waves), 3072 x 384 takes 192-token tiles, 160 tokens one partial 192-token tile.
    # 24 sampled rows spread over the tokens
    sample = np.sort(np.random.default_rng(M).choice(M, min(M, 24), replace=False))
    _gemm_case(cuda_lib, n_out, n_in, M, sample_rows=sample, seed=n_out + M)


def test_q8_0_gemm_batch_m1_matches_gemv_within_bf16_bound(cuda_lib):
    qdq = cuda_lib
    import torch
    wb, x = synth.config0()
    W = qdq.upload_q8_0(wb, 256, 512)
    y = _nan(1, 256)
    Y = _nan(1, 256)
    qdq.q8_0_gemv(W, _t(x), y, 256, 512, 1)
    ws = torch.zeros(qdq.gemm_batch_workspace_bytes(1, 256, 512), dtype=torch.uint8, device=_dev())
    qdq.q8_0_gemm_batch(W, _t(x), Y, ws, 256, 512, 1)
    _, a = oracle.gemv(oracle.q8_0_dequant(wb, 256, 512), x)
    assert np.all(np.abs(_np(Y) - _np(y)) <= 4e-3 * a)


# ------------------------------------------------------------------ fused QKV

def _qkv_case(qdq, n_q, n_kv, n_embd, batch, seed):
    rng = np.random.default_rng(seed)
    bq, bk, bv = (synth.q4k_blocks(rng, n_q, n_embd), synth.q4k_blocks(rng, n_kv, n_embd),
                  synth.q4k_blocks(rng, n_kv, n_embd))
    x = synth.activations(rng, batch, n_embd)
    Wq, Wk, Wv = qdq.upload_q4k(bq, n_q, n_embd), qdq.upload_q4k(bk, n_kv, n_embd), qdq.upload_q4k(bv, n_kv, n_embd)
    q, k, v = _nan(batch, n_q), _nan(batch, n_kv), _nan(batch, n_kv)
    qdq.q4k_qkv(Wq, Wk, Wv, _t(x), q, k, v, n_q, n_kv, n_embd, batch)
    o = oracle.qkv(oracle.q4k_dequant(bq, n_q, n_embd), oracle.q4k_dequant(bk, n_kv, n_embd),
                   oracle.q4k_dequant(bv, n_kv, n_embd), x)
    for name, got in (("q", q), ("k", k), ("v", v)):
        assert gemv_excess(_np(got), o[name], o["A_" + name]) <= 1.0, name
    assert qdq.pipeline_timeouts() == 0


# 3B-class GQA (24 heads / 8 KV heads of 128), Q->K and K->V boundaries inside a 4-row stage,
# n_kv == n_q, a single K/V row, 16 slice warps per row, batch 3 (three GEMV launches)
QKV_SHAPES = [(3072, 1024, 3072, 1), (256, 64, 512, 1), (101, 37, 1024, 1), (50, 50, 256, 1), (7, 1, 256, 1),
              (64, 16, 16384, 1), (40, 8, 768, 3)]


@pytest.mark.parametrize("n_q,n_kv,n_embd,batch", QKV_SHAPES)
def test_q4k_qkv_parity(cuda_lib, n_q, n_kv, n_embd, batch):
    _qkv_case(cuda_lib, n_q, n_kv, n_embd, batch, seed=n_q + 7 * n_kv + n_embd + batch)


def test_q4k_qkv_float_x_parity(cuda_lib):
    qdq = cuda_lib
    old = qdq.set_option(qdq.QDQ_OPT_XS_FLOAT_X, 1)
    try:
        _qkv_case(qdq, 101, 37, 1024, 1, seed=5)
    finally:
        qdq.set_option(qdq.QDQ_OPT_XS_FLOAT_X, old)


def test_q4k_qkv_rows_equal_the_separate_gemvs(cuda_lib):
    # the fused kernel reduces each row exactly as the Q4_K GEMV kernel does
    qdq = cuda_lib
    n_q, n_kv, n_embd = 301, 77, 2048
    rng = np.random.default_rng(8)
    bq, bk, bv = (synth.q4k_blocks(rng, n_q, n_embd), synth.q4k_blocks(rng, n_kv, n_embd),
                  synth.q4k_blocks(rng, n_kv, n_embd))
    x = _t(synth.activations(rng, 1, n_embd))
    Wq, Wk, Wv = qdq.upload_q4k(bq, n_q, n_embd), qdq.upload_q4k(bk, n_kv, n_embd), qdq.upload_q4k(bv, n_kv, n_embd)
    q, k, v = _nan(1, n_q), _nan(1, n_kv), _nan(1, n_kv)
    qdq.q4k_qkv(Wq, Wk, Wv, x, q, k, v, n_q, n_kv, n_embd, 1)
    for W, got, n in ((Wq, q, n_q), (Wk, k, n_kv), (Wv, v, n_kv)):
        y = _nan(1, n)
        qdq.q4k_gemv(W, x, y, n, n_embd, 1)
        assert np.allclose(_np(got), _np(y), rtol=0, atol=1e-5 * float(np.abs(_np(y)).max()))


# ------------------------------------------------------------------ output projection + argmax

def _check_argmax(qdq, wb, x, n_vocab, n_in, batch):
    import torch
    W = qdq.upload_q8_0(wb, n_vocab, n_in)
    logits = _nan(batch, n_vocab)
    idx = torch.full((batch,), -1, dtype=torch.int32, device=_dev())
    val = _nan(batch)
    qdq.q8_0_logits_argmax(W, _t(x), logits, idx, val, n_vocab, n_in, batch)
    lg, ix, vl = _np(logits), _np(idx), _np(val)
    o = oracle.logits_argmax(oracle.q8_0_dequant(wb, n_vocab, n_in), x)
    return lg, ix, vl, o


# a 3B-class vocabulary (128256 x 3072), ragged sizes, batch 3 (general GEMV + argmax)
@pytest.mark.parametrize("n_vocab,n_in,batch", [(128256, 3072, 1), (1000, 512, 1), (5003, 2048, 3), (1, 32, 1)])
def test_logits_argmax_parity(cuda_lib, n_vocab, n_in, batch):
    rng = np.random.default_rng(n_vocab + n_in + batch)
    wb, x = synth.q8_0_blocks(rng, n_vocab, n_in), synth.activations(rng, batch, n_in)
    lg, ix, vl, o = _check_argmax(cuda_lib, wb, x, n_vocab, n_in, batch)
    assert gemv_excess(lg, o["logits"], o["A"]) <= 1.0
    for b in range(batch):
        # unique: the first maximum of the logits the GPU computed, and that logit bit for bit
        assert ix[b] == int(np.argmax(lg[b])) and vl[b].view(np.uint32) == lg[b, ix[b]].view(np.uint32)
        # valid: within the GEMV bound of the exact maximum
        assert o["logits"][b, ix[b]] >= o["value"][b] - 2e-5 * o["A"][b].max()


def test_logits_argmax_first_of_equal_rows(cuda_lib):
    # identical rows give identical logits; the first of the maximal pair wins
    n_vocab, n_in = 4000, 1024
    rng = np.random.default_rng(81)
    wb, x = synth.q8_0_blocks(rng, n_vocab, n_in), synth.activations(rng, 1, n_in)
    y, _ = oracle.gemv(oracle.q8_0_dequant(wb, n_vocab, n_in), x)
    top = int(np.argmax(y[0]))
    wb[3001] = wb[top]
    wb[17] = wb[top]
    lg, ix, vl, o = _check_argmax(cuda_lib, wb, x, n_vocab, n_in, 1)
    assert lg[0, 17] == lg[0, top] == lg[0, 3001]
    assert ix[0] == min(17, top) and o["index"][0] == min(17, top)


def test_logits_argmax_nan_activation(cuda_lib):
    n_vocab, n_in = 700, 512
    rng = np.random.default_rng(82)
    wb, x = synth.q8_0_blocks(rng, n_vocab, n_in), synth.activations(rng, 2, n_in)
    x[1, 7] = np.nan
    lg, ix, vl, o = _check_argmax(cuda_lib, wb, x, n_vocab, n_in, 2)
    assert ix[1] == 0 and np.isnan(vl[1]) and np.all(np.isnan(lg[1]))
    assert ix[0] == o["index"][0] or o["logits"][0, ix[0]] >= o["value"][0] - 2e-5 * o["A"][0].max()


# ------------------------------------------------------------------ batch-1 arithmetic
# The batch-1 kernels multiply in 24-bit block fixed point by default (the integer
# byte dot products); QDQ_OPT_XS_FLOAT_X = 1 selects f32 arithmetic.  Their error
# bounds (include/qdq.h):
#   fixed:  2^-22 sum_b max_{j in b} |x_j| sum_{j in b} |w_j| + f32 rounding
#   float:  1e-5 sum |w||x|

class _FloatX:
    def __init__(self, qdq, value):
        self.qdq, self.value = qdq, value

    def __enter__(self):
        self.old = self.qdq.set_option(self.qdq.QDQ_OPT_XS_FLOAT_X, self.value)

    def __exit__(self, *exc):
        self.qdq.set_option(self.qdq.QDQ_OPT_XS_FLOAT_X, self.old)


def _gemv1(qdq, fmt, wb, x, n_out, n_in):
    W = qdq.upload_q8_0(wb, n_out, n_in) if fmt == "q8_0" else qdq.upload_q4k(wb, n_out, n_in)
    y = _nan(1, n_out)
    (qdq.q8_0_gemv if fmt == "q8_0" else qdq.q4k_gemv)(W, _t(x), y, n_out, n_in, 1)
    return _np(y)


def _blocks(fmt, rng, n_out, n_in):
    return synth.q8_0_blocks(rng, n_out, n_in) if fmt == "q8_0" else synth.q4k_blocks(rng, n_out, n_in)


def _deq(fmt, wb, n_out, n_in):
    return oracle.q8_0_dequant(wb, n_out, n_in) if fmt == "q8_0" else oracle.q4k_dequant(wb, n_out, n_in)


@pytest.mark.parametrize("fmt", ["q8_0", "q4k"])
@pytest.mark.parametrize("n_out,n_in", [(256, 512), (157, 3072), (40, 16384), (8192, 3072)])
def test_batch1_float_x_parity(cuda_lib, fmt, n_out, n_in):
    qdq = cuda_lib
    rng = np.random.default_rng(n_out + n_in + len(fmt))
    wb, x = _blocks(fmt, rng, n_out, n_in), synth.activations(rng, 1, n_in)
    with _FloatX(qdq, 1):
        y = _gemv1(qdq, fmt, wb, x, n_out, n_in)
    y_ref, a = oracle.gemv(_deq(fmt, wb, n_out, n_in), x)
    assert gemv_excess(y, y_ref, a) <= 1.0


def test_batch1_float_x_ffn_parity(cuda_lib):
    with _FloatX(cuda_lib, 1):
        _ffn_case(cuda_lib, 768, 2048, 1, seed=77)


@pytest.mark.parametrize("fmt", ["q8_0", "q4k"])
def test_batch1_outlier_channels(cuda_lib, fmt):
    # residual-stream-like activations: 1 % of the channels 300x larger than the rest.
    # Weights that do not single out the outliers keep the fixed-point error far inside
    # the 1e-5 bar, whichever arithmetic runs.
    qdq = cuda_lib
    n_out, n_in = 512, 3072
    rng = np.random.default_rng(31)
    wb, x = _blocks(fmt, rng, n_out, n_in), synth.activations(rng, 1, n_in)
    x[:, rng.choice(n_in, n_in // 100, replace=False)] *= 300.0
    y_ref, a = oracle.gemv(_deq(fmt, wb, n_out, n_in), x)
    for fx in (0, 1):
        with _FloatX(qdq, fx):
            assert gemv_excess(_gemv1(qdq, fmt, wb, x, n_out, n_in), y_ref, a) <= 1.0


def test_batch1_fixed_x_stated_bound(cuda_lib):
    # Adversarial for block fixed point: one activation per 32-block is 1e4 and its
    # weights are all zero; the rest are ~1e-2.  The default (f32) arithmetic meets the
    # 1e-5 sum|w||x| bound here as everywhere; the opt-in fixed-point path stays within
    # its own stated bound, which is relative to each block's largest activation.
    qdq = cuda_lib
    n_out, n_in = 96, 1024
    rng = np.random.default_rng(41)
    wb = synth.q8_0_blocks(rng, n_out, n_in)
    j0 = rng.integers(0, 32, n_in // 32)
    blk = wb.reshape(n_out, n_in // 32, 34)
    blk[:, np.arange(n_in // 32), 2 + j0] = 0
    x = 1e-2 * synth.activations(rng, 1, n_in)
    x[0, 32 * np.arange(n_in // 32) + j0] = 1e4
    w = oracle.q8_0_dequant(wb, n_out, n_in)
    y_ref, a = oracle.gemv(w, x)
    assert gemv_excess(_gemv1(qdq, "q8_0", wb, x, n_out, n_in), y_ref, a) <= 1.0   # the default path
    m_b = np.abs(x[0]).reshape(-1, 32).max(axis=1)                       # max |x| per block
    w_b = np.abs(w.astype(np.float64)).reshape(n_out, -1, 32).sum(axis=2)  # sum |w| per row and block
    fixed_bound = 2.0 ** -22 * (w_b * m_b).sum(axis=1) + 1e-5 * a[0]
    with _FloatX(qdq, 0):
        y = _gemv1(qdq, "q8_0", wb, x, n_out, n_in)
    assert np.all(np.abs(y[0].astype(np.float64) - y_ref[0]) <= fixed_bound)


def _cancelling_q4k(rng, n_out, n_in, frac_zero, d=1e-2, dmin=1e-2):
    """Q4_K rows whose sub-blocks have sc_j = 4, m_j = 32 everywhere: with d == dmin a
    quant of 8 dequantises to exactly 0, and `frac_zero` of the quant bytes are 0x88."""
    wb = synth.q4k_blocks(rng, n_out, n_in, d_range=(d, d), dmin_range=(dmin, dmin))
    sb = wb.reshape(n_out, n_in // 256, 144)
    # bytes 0..3: sc_0..3 = 4; 4..7: m_0..3 = 32 with the top bits (2) of m_4..7; 8..11:
    # low nibbles sc_4..7 = 4 and m_4..7 = 0 (m_4..7 = 0 | 2 << 4 = 32)
    sb[..., 4:16] = np.array([4, 4, 4, 4, 160, 160, 160, 160, 4, 4, 4, 4], dtype=np.uint8)
    keep = rng.random(sb[..., 16:].shape) >= frac_zero
    sb[..., 16:] = np.where(keep, sb[..., 16:], 0x88).astype(np.uint8)
    return wb


@pytest.mark.parametrize("batch", [1, 4])
@pytest.mark.parametrize("frac_zero", [1.0, 0.99])
def test_q4k_gemv_cancelling_rows(cuda_lib, batch, frac_zero):
    # d*sc_j*q == dmin*m_j for 100 % / 99 % of the weights: sum|w||x| is a tiny part of
    # the two regrouped terms; a row of zero weights must give exactly 0
    qdq = cuda_lib
    n_out, n_in = 200, 2048
    rng = np.random.default_rng(int(frac_zero * 100) + batch)
    wb = _cancelling_q4k(rng, n_out, n_in, frac_zero)
    x = synth.activations(rng, batch, n_in)
    W = qdq.upload_q4k(wb, n_out, n_in)
    y = _nan(batch, n_out)
    qdq.q4k_gemv(W, _t(x), y, n_out, n_in, batch)
    w = oracle.q4k_dequant(wb, n_out, n_in)
    y_ref, a = oracle.gemv(w, x)
    if frac_zero == 1.0:
        assert np.all(w == 0) and np.all(_np(y) == 0.0)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


def test_q4k_gemv_near_cancelling_adjacent_scales(cuda_lib):
    # dmin one fp16 step above d: every weight of a quant-8 sub-block is the same tiny
    # value 32 (d - dmin); the regrouped terms are ~10^3 times larger than the weights
    qdq = cuda_lib
    n_out, n_in = 64, 1024
    d = 1e-2
    dmin = float(np.nextafter(np.float16(d), np.float16(1)))
    rng = np.random.default_rng(12)
    wb = _cancelling_q4k(rng, n_out, n_in, 1.0, d=d, dmin=dmin)
    x = synth.activations(rng, 1, n_in)
    W = qdq.upload_q4k(wb, n_out, n_in)
    y = _nan(1, n_out)
    qdq.q4k_gemv(W, _t(x), y, n_out, n_in, 1)
    w = oracle.q4k_dequant(wb, n_out, n_in)
    assert np.all(w != 0) and np.abs(w).max() < 1e-3 * (4 * d * 8)   # 1000x below d*sc*q
    y_ref, a = oracle.gemv(w, x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


def test_q4k_fixed_x_zero_rows_stay_zero(cuda_lib):
    # the opt-in fixed-point path applies the sub-block shift to exact integer sums:
    # weights that are all exactly zero still give exactly zero
    qdq = cuda_lib
    rng = np.random.default_rng(13)
    wb = _cancelling_q4k(rng, 64, 1024, 1.0)
    x = synth.activations(rng, 1, 1024)
    with _FloatX(qdq, 0):
        y = _gemv1(qdq, "q4k", wb, x, 64, 1024)
    assert np.all(y == 0.0)


@pytest.mark.parametrize("fx", [0, 1])
def test_batch1_chain_reads_the_previous_output(cuda_lib, fx):
    # up then down back to back on one stream (the down kernel starts early under
    # programmatic dependent launch), the intermediate freshly filled with NaN each
    # time: the down kernel must read h only after the up kernel wrote it
    qdq = cuda_lib
    n_embd, n_ff = 3072, 8192
    up, dn = synth.config1_up(0), synth.config1_down(0)
    Wu, Wd = qdq.upload_q8_0(up, n_ff, n_embd), qdq.upload_q8_0(dn, n_embd, n_ff)
    x = synth.config1_x()
    wd = oracle.q8_0_dequant(dn, n_embd, n_ff)
    with _FloatX(qdq, fx):
        for _ in range(4):
            h, y = _nan(1, n_ff), _nan(1, n_embd)
            qdq.q8_0_gemv(Wu, _t(x), h, n_ff, n_embd, 1)
            qdq.q8_0_gemv(Wd, h, y, n_embd, n_ff, 1)
            hh = _np(h)
            assert np.all(np.isfinite(hh))
            y_ref, a = oracle.gemv(wd, hh)
            assert gemv_excess(_np(y), y_ref, a) <= 1.0


@pytest.mark.parametrize("fx", [0, 1])
def test_batch1_one_hot_x_extracts_column(cuda_lib, fx):
    # x = e_k: y is column k of W exactly (d q is exact in f32; X_k = 2^21 exactly)
    qdq = cuda_lib
    n_out, n_in = 200, 2048
    wb = synth.q8_0_blocks(np.random.default_rng(51), n_out, n_in)
    w = oracle.q8_0_dequant(wb, n_out, n_in)
    for k in (0, 31, 1000, 2047):
        x = np.zeros((1, n_in), np.float32)
        x[0, k] = 1.0
        with _FloatX(qdq, fx):
            y = _gemv1(qdq, "q8_0", wb, x, n_out, n_in)
        assert np.array_equal(y[0], w[:, k])


@pytest.mark.parametrize("fx", [0, 1])
@pytest.mark.parametrize("fmt", ["q8_0", "q4k"])
def test_batch1_nan_activation_gives_nan_rows(cuda_lib, fmt, fx):
    qdq = cuda_lib
    n_out, n_in = 64, 512
    rng = np.random.default_rng(61)
    wb, x = _blocks(fmt, rng, n_out, n_in), synth.activations(rng, 1, n_in)
    x[0, 300] = np.nan
    with _FloatX(qdq, fx):
        y = _gemv1(qdq, fmt, wb, x, n_out, n_in)
    assert np.all(np.isnan(y))


# ------------------------------------------------------------------ launch options, errors

def test_launch_options_do_not_change_results(cuda_lib):
    qdq = cuda_lib
    rng = np.random.default_rng(21)
    wb = synth.q4k_blocks(rng, 700, 2048)
    x = synth.activations(rng, 1, 2048)
    W = qdq.upload_q4k(wb, 700, 2048)
    outs = []
    for pdl, pf in [(1, 1), (0, 0), (1, 0), (0, 1), (1, 2), (0, 2), (1, 3)]:
        old_pdl = qdq.set_option(qdq.QDQ_OPT_PDL, pdl)
        old_pf = qdq.set_option(qdq.QDQ_OPT_L2_PREFETCH, pf)
        y = _nan(1, 700)
        qdq.q4k_gemv(W, _t(x), y, 700, 2048, 1)
        outs.append(_np(y))
        qdq.set_option(qdq.QDQ_OPT_PDL, old_pdl)
        qdq.set_option(qdq.QDQ_OPT_L2_PREFETCH, old_pf)
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def test_ctas_per_sm_does_not_change_ffn_results(cuda_lib):
    # a row's sum does not depend on which CTA computes it: every split of the rows
    # between CTAs gives the same bits
    qdq = cuda_lib
    import torch
    rng = np.random.default_rng(23)
    g, u, d = synth.q4k_blocks(rng, 2048, 1024), synth.q4k_blocks(rng, 2048, 1024), synth.q4k_blocks(rng, 1024, 2048)
    x, res = synth.activations(rng, 1, 1024), synth.activations(rng, 1, 1024)
    Wg, Wu, Wd = qdq.upload_q4k(g, 2048, 1024), qdq.upload_q4k(u, 2048, 1024), qdq.upload_q4k(d, 1024, 2048)
    outs = []
    for cps in (0, 1, 2, 3):
        old = qdq.set_option(qdq.QDQ_OPT_CTAS_PER_SM, cps)
        try:
            out, mid = _nan(1, 1024), torch.empty((1, 2048), device=_dev())
            qdq.q4k_ffn_residual(Wg, Wu, Wd, _t(x), _t(res), out, mid, 1024, 2048, 1)
            outs.append(_np(out))
        finally:
            qdq.set_option(qdq.QDQ_OPT_CTAS_PER_SM, old)
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    assert qdq.pipeline_timeouts() == 0


def test_error_leaves_outputs_untouched(cuda_lib):
    qdq = cuda_lib
    import torch
    wb = synth.q8_0_blocks(np.random.default_rng(1), 64, 256)
    W = qdq.upload_q8_0(wb, 64, 256)
    x = _t(synth.activations(np.random.default_rng(2), 1, 256))
    y = _nan(1, 64)
    with pytest.raises(qdq.QdqError) as e:
        qdq.q8_0_gemv(W, int(x.data_ptr()) + 4, y, 64, 256, 1)   # misaligned x
    assert e.value.status == qdq.QDQ_ERR_ALIGN
    with pytest.raises(qdq.QdqError) as e:
        qdq.q8_0_gemv(W, x, y, 64, 256, 9)                        # batch too large
    assert e.value.status == qdq.QDQ_ERR_DIMS
    assert np.all(np.isnan(_np(y)))
    torch.cuda.synchronize()


# ------------------------------------------------------------------ batch-1 pipeline shapes

@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("n_out,groups", [(2053, 0), (2053, 3), (1001, 2), (1001, 5), (152 * 9 + 151, 0)])
def test_batch1_uneven_group_rows(cuda_lib, n_out, groups, kernel):
    # rows of a CTA are split between its consumer groups; uneven splits end each
    # group with a partial stage, which must neither be lost nor spill into the next
    # group (both batch-1 kernels: 0 direct load, 1 shared-memory ring)
    qdq = cuda_lib
    old_k = qdq.set_option(qdq.QDQ_OPT_BATCH1_KERNEL, kernel)
    rng = np.random.default_rng(n_out + 7 * groups)
    wq = synth.q8_0_blocks(rng, n_out, 3072)
    g, u, d = synth.q4k_blocks(rng, n_out, 3072), synth.q4k_blocks(rng, n_out, 3072), synth.q4k_blocks(rng, n_out, 3072)
    x, res = synth.activations(rng, 1, 3072), synth.activations(rng, 1, n_out)
    Wq, Wg, Wu, Wd = (qdq.upload_q8_0(wq, n_out, 3072), qdq.upload_q4k(g, n_out, 3072),
                      qdq.upload_q4k(u, n_out, 3072), qdq.upload_q4k(d, n_out, 3072))
    old_g = qdq.set_option(qdq.QDQ_OPT_XS_GROUPS, groups)
    try:
        y, mid, y4 = _nan(1, n_out), _nan(1, n_out), _nan(1, n_out)
        qdq.q8_0_gemv(Wq, _t(x), y, n_out, 3072, 1)
        qdq.q4k_swiglu(Wg, Wu, _t(x), mid, n_out, 3072, 1)
        qdq.q4k_gemv(Wd, _t(x), y4, n_out, 3072, 1)
        yh, mh, y4h = _np(y), _np(mid), _np(y4)
    finally:
        qdq.set_option(qdq.QDQ_OPT_BATCH1_KERNEL, old_k)
        qdq.set_option(qdq.QDQ_OPT_XS_GROUPS, old_g)
    y_ref, a = oracle.gemv(oracle.q8_0_dequant(wq, n_out, 3072), x)
    assert gemv_excess(yh, y_ref, a) <= 1.0
    s = oracle.swiglu(oracle.q4k_dequant(g, n_out, 3072), oracle.q4k_dequant(u, n_out, 3072), x)
    assert np.all(np.abs(mh - s["mid"]) <= swiglu_eps(s))
    y4_ref, a4 = oracle.gemv(oracle.q4k_dequant(d, n_out, 3072), x)
    assert gemv_excess(y4h, y4_ref, a4) <= 1.0
    assert qdq.pipeline_timeouts() == 0


@pytest.mark.parametrize("kernel,groups,slots", [(1, 1, 1), (1, 1, 2), (1, 2, 1), (1, 3, 4), (1, 5, 2), (1, 4, 3),
                                                (0, 1, 1), (0, 1, 2), (0, 2, 1), (0, 3, 2), (0, 5, 1), (0, 4, 2)])
def test_batch1_pipeline_shapes(cuda_lib, kernel, groups, slots):
    # the ring kernel (kernel 1) streams weights through per-group shared-memory rings
    # (slots = ring slots per group); the direct-load kernel (kernel 0) holds one or two
    # stages of registers per warp (slots = that depth): every shape must give the
    # same sums within the bound
    qdq = cuda_lib
    old_k = qdq.set_option(qdq.QDQ_OPT_BATCH1_KERNEL, kernel)
    rng = np.random.default_rng(100 + 10 * groups + slots)
    wq = synth.q8_0_blocks(rng, 600, 3072)
    g, u = synth.q4k_blocks(rng, 600, 3072), synth.q4k_blocks(rng, 600, 3072)
    x = synth.activations(rng, 1, 3072)
    Wq, Wg, Wu = qdq.upload_q8_0(wq, 600, 3072), qdq.upload_q4k(g, 600, 3072), qdq.upload_q4k(u, 600, 3072)
    old_g = qdq.set_option(qdq.QDQ_OPT_XS_GROUPS, groups)
    old_s = qdq.set_option(qdq.QDQ_OPT_XS_STAGES, slots)
    try:
        y, mid = _nan(1, 600), _nan(1, 600)
        qdq.q8_0_gemv(Wq, _t(x), y, 600, 3072, 1)
        qdq.q4k_swiglu(Wg, Wu, _t(x), mid, 600, 3072, 1)
        yh, mh = _np(y), _np(mid)
    finally:
        qdq.set_option(qdq.QDQ_OPT_XS_GROUPS, old_g)
        qdq.set_option(qdq.QDQ_OPT_XS_STAGES, old_s)
        qdq.set_option(qdq.QDQ_OPT_BATCH1_KERNEL, old_k)
    y_ref, a = oracle.gemv(oracle.q8_0_dequant(wq, 600, 3072), x)
    assert gemv_excess(yh, y_ref, a) <= 1.0
    s = oracle.swiglu(oracle.q4k_dequant(g, 600, 3072), oracle.q4k_dequant(u, 600, 3072), x)
    assert np.all(np.abs(mh - s["mid"]) <= swiglu_eps(s))
    assert qdq.pipeline_timeouts() == 0
