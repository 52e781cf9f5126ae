"""GPU parity of the Q6_K path and the on-device top-k (through the C ABI).

Bars:
* Q6_K dequantised weights and embedding rows: bit-exact (d*scale*(q-32) is
  exact in f32);
* Q6_K GEMV: |y - y_ref| <= 1e-5 * sum|w||x| against the float64 oracle;
* top-k: the indices and values are unique given the logits, so they are
  compared with the stable top-k of the logits the GPU computed (value bits
  included), and every returned logit must be within the GEMV bound of the
  oracle's k-th best logit.
"""
import numpy as np
import pytest

import oracle
import synth
from _bounds import gemv_excess

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


# ------------------------------------------------------------------ Q6_K

@pytest.mark.parametrize("n_out,n_in", [(1, 256), (37, 768), (5, 3072), (300, 2048), (1000, 8192)])
def test_q6k_dequant_bit_exact(cuda_lib, n_out, n_in):
    qdq = cuda_lib
    wb = synth.q6k_blocks(np.random.default_rng(n_out + n_in), n_out, n_in)
    W = qdq.upload_q6k(wb, n_out, n_in)
    out = _nan(n_out, n_in)
    qdq.q6k_dequant(W, out, n_out, n_in)
    assert np.array_equal(_np(out).view(np.uint32), oracle.q6k_dequant(wb, n_out, n_in).view(np.uint32))


def test_q6k_dequant_extreme_scales_bit_exact(cuda_lib):
    # largest fp16 d, scales -128 / 127, every quant 0 or 63
    qdq = cuda_lib
    rng = np.random.default_rng(4)
    wb = synth.q6k_blocks(rng, 16, 512, d_range=(65504.0, 65504.0))
    sb = wb.reshape(16, 2, 210)
    sb[..., 192:208] = np.where(rng.random((16, 2, 16)) < 0.5, 0x80, 0x7F).astype(np.uint8)
    sb[..., 0:192] = np.where(rng.random((16, 2, 192)) < 0.5, 0x00, 0xFF).astype(np.uint8)
    W = qdq.upload_q6k(wb, 16, 512)
    out = _nan(16, 512)
    qdq.q6k_dequant(W, out, 16, 512)
    assert np.array_equal(_np(out).view(np.uint32), oracle.q6k_dequant(wb, 16, 512).view(np.uint32))


Q6_SHAPES = [(1, 256, 1), (5, 512, 1), (157, 3072, 1), (64, 512, 8), (33, 8192, 3), (1000, 1280, 2),
             (40, 16384, 1), (24, 32768, 1), (16, 32768, 8), (3001, 4096, 1)]


@pytest.mark.parametrize("n_out,n_in,batch", Q6_SHAPES)
def test_q6k_gemv_parity(cuda_lib, n_out, n_in, batch):
    qdq = cuda_lib
    rng = np.random.default_rng(n_out + 7 * n_in + batch)
    wb = synth.q6k_blocks(rng, n_out, n_in)
    x = synth.activations(rng, batch, n_in)
    W = qdq.upload_q6k(wb, n_out, n_in)
    y = _nan(batch, n_out)
    qdq.q6k_gemv(W, _t(x), y, n_out, n_in, batch)
    y_ref, a = oracle.gemv(oracle.q6k_dequant(wb, n_out, n_in), x)
    assert gemv_excess(_np(y), y_ref, a) <= 1.0


def test_q6k_gemv_output_projection_full_size(cuda_lib):
    # the 3B-class vocabulary projection (128256 x 3072), checked on every row
    qdq = cuda_lib
    wb, x = synth.q6k_output_projection()
    W = qdq.upload_q6k(wb, synth.N_VOCAB, synth.N_EMBD)
    y = _nan(1, synth.N_VOCAB)
    qdq.q6k_gemv(W, _t(x), y, synth.N_VOCAB, synth.N_EMBD, 1)
    yh = _np(y)
    rows = wb.reshape(synth.N_VOCAB, -1)
    for r0 in range(0, synth.N_VOCAB, 16032):   # the oracle in row blocks (bounded host memory)
        r1 = min(r0 + 16032, synth.N_VOCAB)
        y_ref, a = oracle.gemv(oracle.q6k_dequant(rows[r0:r1], r1 - r0, synth.N_EMBD), x)
        assert gemv_excess(yh[:, r0:r1], y_ref, a) <= 1.0


def test_q6k_gemv_one_hot_extracts_column(cuda_lib):
    qdq = cuda_lib
    wb = synth.q6k_blocks(np.random.default_rng(17), 200, 2048)
    W = qdq.upload_q6k(wb, 200, 2048)
    w = oracle.q6k_dequant(wb, 200, 2048)
    for k in (0, 15, 16, 1000, 2047):
        x = np.zeros((1, 2048), np.float32)
        x[0, k] = 1.0
        y = _nan(1, 200)
        qdq.q6k_gemv(W, _t(x), y, 200, 2048, 1)
        assert np.array_equal(_np(y)[0], w[:, k])


def test_q6k_get_rows_bit_exact(cuda_lib):
    # embedding lookup on the vocabulary table: repeated, first and last ids, and ids
    # outside the table (a NaN row each)
    import torch
    qdq = cuda_lib
    n_rows, n_in = 4096, 3072
    wb = synth.q6k_blocks(np.random.default_rng(18), n_rows, n_in)
    W = qdq.upload_q6k(wb, n_rows, n_in)
    ids = np.concatenate([synth.token_ids(np.random.default_rng(19), 29, n_rows), [0, n_rows - 1, 7, 7, -1, n_rows]])
    ids = ids.astype(np.int32)
    out = _nan(len(ids), n_in)
    qdq.q6k_get_rows(W, torch.from_numpy(ids).to(_dev()), out, len(ids), n_rows, n_in)
    ref = oracle.get_rows(oracle.q6k_dequant(wb, n_rows, n_in), ids)
    got = _np(out)
    ok = ~np.isnan(ref[:, 0])
    assert np.array_equal(got[ok].view(np.uint32), ref[ok].view(np.uint32))
    assert np.all(np.isnan(got[~ok]))


# ------------------------------------------------------------------ top-k

def _stable_topk(row, k):
    """Top-k of one logits row in the stated order (NaN first, larger, smaller index)."""
    nan = np.isnan(row)
    key = np.where(nan, np.inf, row.astype(np.float64))
    order = np.lexsort((np.arange(row.size), ~nan, -key))   # NaN group first, then value desc, index asc
    return order[:k]


def _topk_case(qdq, wb, x, n_vocab, n_in, batch, k, fused=True):
    """`wb`: raw Q8_0 bytes, or a matrix already uploaded (a torch tensor)."""
    import torch
    W = wb if isinstance(wb, torch.Tensor) else qdq.upload_q8_0(wb, n_vocab, n_in)
    logits = _nan(batch, n_vocab)
    ws = torch.empty(qdq.topk_workspace_bytes(n_vocab, batch, k), dtype=torch.uint8, device=_dev())
    idx = torch.full((batch, k), -1, dtype=torch.int32, device=_dev())
    val = _nan(batch, k)
    if fused:
        qdq.q8_0_logits_topk(W, _t(x), logits, ws, idx, val, n_vocab, n_in, batch, k)
    else:
        qdq.q8_0_gemv(W, _t(x), logits, n_vocab, n_in, batch)
        qdq.topk_rows(logits, n_vocab, batch, k, ws, idx, val)
    return _np(logits), _np(idx), _np(val)


def test_topk_full_vocabulary(cuda_lib):
    # the 3B-class vocabulary (128256 x 3072 Q8_0), k = 1, 8, 40 and the largest k
    qdq = cuda_lib
    wb, x = synth.output_projection()
    n_vocab, n_in = synth.N_VOCAB, synth.N_EMBD
    rows = wb.reshape(n_vocab, -1)
    ref, a = np.empty((1, n_vocab)), np.empty((1, n_vocab))
    for r0 in range(0, n_vocab, 16032):        # oracle logits in row blocks (bounded host memory)
        r1 = min(r0 + 16032, n_vocab)
        ref[:, r0:r1], a[:, r0:r1] = oracle.gemv(oracle.q8_0_dequant(rows[r0:r1], r1 - r0, n_in), x)
    kmax = qdq.QDQ_MAX_TOPK
    W = qdq.upload_q8_0(wb, n_vocab, n_in)
    exact_order = np.lexsort((np.arange(n_vocab), -ref[0]))[:kmax]            # exact top-k of the oracle logits
    for k in (1, 8, 40, kmax):
        lg, ix, vl = _topk_case(qdq, W, x, n_vocab, n_in, 1, k)
        order = _stable_topk(lg[0], k)
        assert np.array_equal(ix[0], order)                                # unique given the logits
        assert np.array_equal(vl[0].view(np.uint32), lg[0, order].view(np.uint32))
        tol = 2e-5 * a[0].max()
        assert np.all(ref[0, ix[0]] >= ref[0, exact_order[k - 1]] - tol)   # valid: near the exact top-k
        assert np.all(np.abs(vl[0] - ref[0, ix[0]]) <= 1e-5 * a[0, ix[0]])


@pytest.mark.parametrize("n_vocab,n_in,batch,k", [(1000, 512, 1, 8), (5003, 2048, 3, 40), (64, 32, 2, 64),
                                                  (1, 32, 1, 1), (9000, 256, 8, 17)])
def test_topk_shapes(cuda_lib, n_vocab, n_in, batch, k):
    qdq = cuda_lib
    rng = np.random.default_rng(n_vocab + k)
    wb, x = synth.q8_0_blocks(rng, n_vocab, n_in), synth.activations(rng, batch, n_in)
    lg, ix, vl = _topk_case(qdq, wb, x, n_vocab, n_in, batch, k, fused=(batch % 2 == 1))
    for b in range(batch):
        order = _stable_topk(lg[b], k)
        assert np.array_equal(ix[b], order)
        assert np.array_equal(vl[b].view(np.uint32), lg[b, order].view(np.uint32))


def test_topk_ties_nans_and_signed_zeros(cuda_lib):
    # logits written directly: runs of equal values across chunk borders, NaNs, +0 / -0
    import torch
    qdq = cuda_lib
    n, k = 5000, 40
    rng = np.random.default_rng(23)
    lg = rng.integers(-5, 6, size=(2, n)).astype(np.float32)   # many ties
    lg[0, [17, 1023, 1024, 4999]] = 5.0
    lg[1, [3000, 12]] = np.nan
    lg[1, 100:200] = -0.0
    lg[1, 200:300] = 0.0
    logits = _t(lg)
    ws = torch.empty(qdq.topk_workspace_bytes(n, 2, k), dtype=torch.uint8, device=_dev())
    idx = torch.full((2, k), -1, dtype=torch.int32, device=_dev())
    val = _nan(2, k)
    qdq.topk_rows(logits, n, 2, k, ws, idx, val)
    ix, vl = _np(idx), _np(val)
    for b in range(2):
        order = _stable_topk(lg[b], k)
        assert np.array_equal(ix[b], order)
        assert np.array_equal(vl[b].view(np.uint32), lg[b, order].view(np.uint32))
    assert list(ix[1, :2]) == [12, 3000]
    # the oracle's selection on the same logits (row 0: an identity projection reproduces them)
    o = oracle.logits_topk(np.eye(n, dtype=np.float32), lg[:1], k)
    assert np.array_equal(o["index"][0], ix[0].astype(np.int64))


# ------------------------------------------------------------------ Q4_K batch GEMM / SwiGLU on tensor cores

def _gemm_q4k(qdq, wb, X, n_out, n_in, M):
    import torch
    W = qdq.upload_q4k(wb, n_out, n_in)
    Y = _nan(M, n_out)
    ws = torch.zeros(qdq.gemm_batch_workspace_bytes(M, n_out, n_in), dtype=torch.uint8, device=_dev())
    qdq.q4k_gemm_batch(W, _t(X), Y, ws, n_out, n_in, M)
    return _np(Y)


def _tile_sample(M, seed):
    """All rows for small M, else 32 rows from each 256-token tile."""
    if M <= 64:
        return np.arange(M)
    return np.sort(np.concatenate([t * 256 + np.random.default_rng(seed + t).choice(min(256, M - t * 256),
                                                                                   min(32, M - t * 256), replace=False)
                                   for t in range((M + 255) // 256)]))


@pytest.mark.parametrize("n_out,n_in,M", [(256, 512, 1), (256, 512, 16), (256, 512, 20), (256, 512, 64),
                                          (256, 512, 100), (256, 512, 257), (384, 1024, 33), (128, 256, 16),
                                          (1024, 2048, 130), (512, 768, 300), (128, 256, 40), (128, 768, 32)])
def test_q4k_gemm_batch_parity(cuda_lib, n_out, n_in, M):
    rng = np.random.default_rng(n_out + n_in + M)
    wb, X = synth.q4k_blocks(rng, n_out, n_in), synth.activations(rng, M, n_in)
    Y = _gemm_q4k(cuda_lib, wb, X, n_out, n_in, M)
    Y_ref, A = oracle.gemm_batch(oracle.q4k_dequant(wb, n_out, n_in), X)
    assert gemv_excess(Y, Y_ref, A, rel=4e-3) <= 1.0
    assert cuda_lib.pipeline_timeouts() == 0


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("M", [16, 64, 512])
def test_q4k_gemm_batch_full_size(cuda_lib, kind, M):
    # the config-2/3 shapes: 3072 -> 8192 (gate / up) and 8192 -> 3072 (down)
    n_out, n_in = (8192, 3072) if kind == 0 else (3072, 8192)
    rng = np.random.default_rng(70 + kind)
    wb, X = synth.q4k_blocks(rng, n_out, n_in), synth.activations(rng, M, n_in)
    Y = _gemm_q4k(cuda_lib, wb, X, n_out, n_in, M)
    rows = _tile_sample(M, M)
    Y_ref, A = oracle.gemm_batch(oracle.q4k_dequant(wb, n_out, n_in), X[rows])
    assert gemv_excess(Y[rows], Y_ref, A, rel=4e-3) <= 1.0


@pytest.mark.parametrize("n_out,n_in,M", [(8192, 3072, 600), (3072, 8192, 384)])
def test_q4k_gemm_batch_token_tiles(cuda_lib, n_out, n_in, M):
    # 8192 x 600: more output tiles than SMs (no K split, two waves); 3072 x 384: 192-token tiles
    rng = np.random.default_rng(n_out + M)
    wb, X = synth.q4k_blocks(rng, n_out, n_in), synth.activations(rng, M, n_in)
    Y = _gemm_q4k(cuda_lib, wb, X, n_out, n_in, M)
    rows = np.sort(rng.choice(M, 24, replace=False))
    Y_ref, A = oracle.gemm_batch(oracle.q4k_dequant(wb, n_out, n_in), X[rows])
    assert gemv_excess(Y[rows], Y_ref, A, rel=4e-3) <= 1.0
    assert cuda_lib.pipeline_timeouts() == 0


def test_q4k_gemm_batch_m1_matches_gemv_within_bf16_bound(cuda_lib):
    qdq = cuda_lib
    rng = np.random.default_rng(72)
    wb, x = synth.q4k_blocks(rng, 512, 1024), synth.activations(rng, 1, 1024)
    Y = _gemm_q4k(qdq, wb, x, 512, 1024, 1)
    W = qdq.upload_q4k(wb, 512, 1024)
    y = _nan(1, 512)
    qdq.q4k_gemv(W, _t(x), y, 512, 1024, 1)
    _, a = oracle.gemv(oracle.q4k_dequant(wb, 512, 1024), x)
    assert np.all(np.abs(Y - _np(y)) <= 4e-3 * a)


@pytest.mark.parametrize("fmt", ["q8_0", "q4k"])
def test_gemm_batch_split_k_is_deterministic(cuda_lib, fmt):
    # small M on a 3072-row matrix splits K across CTAs; the partials are added in a
    # fixed order, so two calls give the same bits
    import torch
    qdq = cuda_lib
    n_out, n_in, M = 3072, 8192, 16
    rng = np.random.default_rng(73)
    X = _t(synth.activations(rng, M, n_in))
    if fmt == "q8_0":
        W, f = qdq.upload_q8_0(synth.q8_0_blocks(rng, n_out, n_in), n_out, n_in), qdq.q8_0_gemm_batch
    else:
        W, f = qdq.upload_q4k(synth.q4k_blocks(rng, n_out, n_in), n_out, n_in), qdq.q4k_gemm_batch
    ws = torch.zeros(qdq.gemm_batch_workspace_bytes(M, n_out, n_in), dtype=torch.uint8, device=_dev())
    outs = []
    for _ in range(3):
        Y = _nan(M, n_out)
        f(W, X, Y, ws, n_out, n_in, M)
        outs.append(_np(Y))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[2].view(np.uint32))


def test_gemm_batch_workspace_reused_across_shapes(cuda_lib):
    # one workspace serves calls of different shapes and token counts (different split-K
    # cluster sizes, in-kernel or separate X conversion) back to back
    import torch
    qdq = cuda_lib
    rng = np.random.default_rng(74)
    cases = [(3072, 8192, 16), (8192, 3072, 16), (3072, 8192, 40), (384, 1024, 33), (3072, 8192, 64),
             (1024, 2048, 130), (3072, 8192, 16)]
    size = max(qdq.gemm_batch_workspace_bytes(M, n_out, n_in) for n_out, n_in, M in cases)
    ws = torch.zeros(size, dtype=torch.uint8, device=_dev())
    for n_out, n_in, M in cases:
        wb, X = synth.q8_0_blocks(rng, n_out, n_in), synth.activations(rng, M, n_in)
        W = qdq.upload_q8_0(wb, n_out, n_in)
        Y = _nan(M, n_out)
        qdq.q8_0_gemm_batch(W, _t(X), Y, ws, n_out, n_in, M)
        rows = np.arange(0, M, max(1, M // 8))
        Y_ref, A = oracle.gemm_batch(oracle.q8_0_dequant(wb, n_out, n_in), X[rows])
        assert gemv_excess(_np(Y)[rows], Y_ref, A, rel=4e-3) <= 1.0, (n_out, n_in, M)
    assert qdq.pipeline_timeouts() == 0


def _swiglu_batch_bound(s, rel=4e-3):
    # the batch bound through silu (|silu'| <= 1.1) and the product, plus expf's ulp
    return (1.1 * np.abs(s["u"]) * rel * s["A_g"] + np.abs(oracle.silu(s["g"])) * rel * s["A_u"]
            + 1e-6 * np.abs(s["mid"]))


@pytest.mark.parametrize("n_ff,n_embd,M", [(512, 256, 20), (1024, 512, 130), (256, 1024, 1), (8192, 3072, 64),
                                           (1024, 512, 192), (3072, 1024, 600), (256, 256, 17), (384, 768, 32),
                                           (128, 256, 16)])
def test_q4k_swiglu_batch_parity(cuda_lib, n_ff, n_embd, M):
    import torch
    qdq = cuda_lib
    rng = np.random.default_rng(n_ff + n_embd + M)
    g, u = synth.q4k_blocks(rng, n_ff, n_embd), synth.q4k_blocks(rng, n_ff, n_embd)
    X = synth.activations(rng, M, n_embd)
    Wg, Wu = qdq.upload_q4k(g, n_ff, n_embd), qdq.upload_q4k(u, n_ff, n_embd)
    mid = _nan(M, n_ff)
    ws = torch.zeros(qdq.q4k_swiglu_batch_workspace_bytes(M, n_ff, n_embd), dtype=torch.uint8, device=_dev())
    qdq.q4k_swiglu_batch(Wg, Wu, _t(X), mid, ws, n_ff, n_embd, M)
    rows = _tile_sample(M, 5)[:16]
    s = oracle.swiglu(oracle.q4k_dequant(g, n_ff, n_embd), oracle.q4k_dequant(u, n_ff, n_embd), X[rows])
    assert np.all(np.abs(_np(mid)[rows] - s["mid"]) <= _swiglu_batch_bound(s))
    assert qdq.pipeline_timeouts() == 0


def _topk_direct(qdq, lg, k):
    import torch
    batch, n = lg.shape
    ws = torch.empty(qdq.topk_workspace_bytes(n, batch, k), dtype=torch.uint8, device=_dev())
    idx = torch.full((batch, k), -1, dtype=torch.int32, device=_dev())
    val = _nan(batch, k)
    qdq.topk_rows(_t(lg), n, batch, k, ws, idx, val)
    ix, vl = _np(idx), _np(val)
    for b in range(batch):
        order = _stable_topk(lg[b], k)
        assert np.array_equal(ix[b], order), b
        assert np.array_equal(vl[b].view(np.uint32), lg[b, order].view(np.uint32)), b


def test_topk_adversarial_rows(cuda_lib):
    # full-vocabulary rows whose top values cluster in one 1024-logit chunk, ascending and descending
    # rows (every chunk's candidates matter / none do), all equal (ties broken by index), NaNs spread
    # over every chunk, runs of equal values across chunk borders
    n, k = 128256, 64
    rng = np.random.default_rng(31)
    rows = []
    r = rng.standard_normal(n).astype(np.float32)
    lo7 = 7 * n // 8
    r[lo7 + 5 + 64 * np.arange(15)] = 100.0 + np.arange(15, dtype=np.float32)  # one chunk
    rows.append(r)
    rows.append(np.arange(n, dtype=np.float32))            # ascending: every CTA's threshold differs
    rows.append(-np.arange(n, dtype=np.float32))           # descending
    rows.append(np.full(n, 2.5, dtype=np.float32))         # all equal: ties broken by index
    r = rng.standard_normal(n).astype(np.float32)
    r[::997] = np.nan
    rows.append(r)
    r = np.repeat(rng.integers(-3, 4, size=n // 64 + 1), 64)[:n].astype(np.float32)  # runs of equal values
    rows.append(r)
    _topk_direct(cuda_lib, np.stack(rows), k)
    _topk_direct(cuda_lib, np.ascontiguousarray(np.stack(rows)[:, :100000]), 33)
    _topk_direct(cuda_lib, np.stack(rows), 1)


def test_top1_is_the_argmax(cuda_lib):
    # k = 1 takes the argmax kernel: same index and value bits as the argmax entry point and the
    # stated order on rows whose best entries are NaNs, -0 before +0, ties and -inf only
    import torch
    qdq = cuda_lib
    n = 70001
    rng = np.random.default_rng(33)
    rows = [rng.standard_normal(n).astype(np.float32) for _ in range(6)]
    rows[0][[70000, 40000]] = np.nan
    rows[1][:] = -1.0
    rows[1][[5000, 3]] = -0.0
    rows[1][[60000, 100]] = 0.0
    rows[2][:] = -np.inf
    rows[3][[12345, 54321]] = 9.0
    rows[4][-1] = 50.0
    lg = np.stack(rows)
    _topk_direct(qdq, lg, 1)
    # the fused projection + top-1 against the projection + argmax on the same weights
    n_vocab, n_in, batch = 5003, 1024, 3
    wb, x = synth.q8_0_blocks(rng, n_vocab, n_in), synth.activations(rng, batch, n_in)
    W = qdq.upload_q8_0(wb, n_vocab, n_in)
    lg1, ix1, vl1 = _topk_case(qdq, W, x, n_vocab, n_in, batch, 1, fused=True)
    logits = _nan(batch, n_vocab)
    idx = torch.full((batch,), -1, dtype=torch.int32, device=_dev())
    val = _nan(batch)
    qdq.q8_0_logits_argmax(W, _t(x), logits, idx, val, n_vocab, n_in, batch)
    assert np.array_equal(_np(logits).view(np.uint32), lg1.view(np.uint32))
    assert np.array_equal(_np(idx), ix1[:, 0]) and np.array_equal(_np(val).view(np.uint32), vl1[:, 0].view(np.uint32))


def test_topk_very_long_row(cuda_lib):
    # 1.5 M logits: 1465 chunk lists, so three merge rounds (46 CTAs, 2, 1); a second row of
    # equal values (ties by index)
    rng = np.random.default_rng(34)
    lg = rng.standard_normal((2, 1_500_001)).astype(np.float32)
    lg[0, 7::300000] = np.nan
    lg[1, :] = 1.0
    _topk_direct(cuda_lib, lg, 64)
    _topk_direct(cuda_lib, lg, 7)


def test_topk_repeated_calls_reuse_the_workspace(cuda_lib):
    # back-to-back calls (fused projection and separate top-k, different k and row counts)
    # on one workspace stay exact
    import torch
    qdq = cuda_lib
    rng = np.random.default_rng(35)
    n_vocab, n_in = 40000, 1024
    wb, x = synth.q8_0_blocks(rng, n_vocab, n_in), synth.activations(rng, 1, n_in)
    W = qdq.upload_q8_0(wb, n_vocab, n_in)
    ws = torch.empty(max(qdq.topk_workspace_bytes(n_vocab, 3, 64), qdq.topk_workspace_bytes(n_vocab, 1, 64)),
                     dtype=torch.uint8, device=_dev())
    ws.fill_(0xAB)  # arbitrary scratch contents before the first call
    lg3 = rng.standard_normal((3, n_vocab)).astype(np.float32)
    for k in (40, 64, 3, 40):
        logits = _nan(1, n_vocab)
        idx = torch.full((1, k), -1, dtype=torch.int32, device=_dev())
        val = _nan(1, k)
        qdq.q8_0_logits_topk(W, _t(x), logits, ws, idx, val, n_vocab, n_in, 1, k)
        lg = _np(logits)
        assert np.array_equal(_np(idx)[0], _stable_topk(lg[0], k))
        idx3 = torch.full((3, k), -1, dtype=torch.int32, device=_dev())
        val3 = _nan(3, k)
        qdq.topk_rows(_t(lg3), n_vocab, 3, k, ws, idx3, val3)
        for b in range(3):
            assert np.array_equal(_np(idx3)[b], _stable_topk(lg3[b], k))


def test_topk_long_rows(cuda_lib):
    # 300001 logits: three merge rounds (1024-logit chunks, 2048-key merges), a ragged last chunk
    rng = np.random.default_rng(32)
    lg = rng.standard_normal((2, 300001)).astype(np.float32)
    lg[1, 5::50000] = np.nan
    _topk_direct(cuda_lib, lg, 40)


@pytest.mark.parametrize("n_vocab,n_in,k", [(100, 256, 64), (1000, 512, 1), (5003, 2048, 40), (33333, 1024, 17),
                                            (40000, 3072, 40), (128256, 3072, 64)])
def test_logits_topk_fused_equals_separate(cuda_lib, n_vocab, n_in, k):
    # batch 1 selects from the projection's per-CTA candidates; the separate GEMV + top-k
    # path must give the same indices and value bits (also for rows shorter than k per CTA)
    qdq = cuda_lib
    rng = np.random.default_rng(n_vocab + k)
    wb, x = synth.q8_0_blocks(rng, n_vocab, n_in), synth.activations(rng, 1, n_in)
    import torch
    W = qdq.upload_q8_0(wb, n_vocab, n_in)
    lg1, ix1, vl1 = _topk_case(qdq, W, x, n_vocab, n_in, 1, k, fused=True)
    lg2, ix2, vl2 = _topk_case(qdq, W, x, n_vocab, n_in, 1, k, fused=False)
    assert np.array_equal(lg1.view(np.uint32), lg2.view(np.uint32))
    assert np.array_equal(ix1, ix2)
    assert np.array_equal(vl1.view(np.uint32), vl2.view(np.uint32))
    order = _stable_topk(lg1[0], k)
    assert np.array_equal(ix1[0], order)


@pytest.mark.parametrize("k", [40, 64])
def test_logits_topk_fused_many_candidates(cuda_lib, k):
    # every third row has a large logit, so that each CTA of the projection holds fewer
    # than k large rows and every CTA's candidate list mixes large and small logits; the
    # merge of the lists and the separate GEMV + top-k path must agree bit for bit
    qdq = cuda_lib
    n_vocab, n_in = 40000, 3072
    rng = np.random.default_rng(91 + k)
    wb = synth.q8_0_blocks(rng, n_vocab, n_in).reshape(n_vocab, n_in // 32, 34)
    wb[0::3, :, 2:] = 127  # int8 quants 127 on every third row
    wb = wb.reshape(n_vocab, -1)
    x = np.abs(synth.activations(rng, 1, n_in))
    W = qdq.upload_q8_0(wb, n_vocab, n_in)
    lg1, ix1, vl1 = _topk_case(qdq, W, x, n_vocab, n_in, 1, k, fused=True)
    lg2, ix2, vl2 = _topk_case(qdq, W, x, n_vocab, n_in, 1, k, fused=False)
    assert np.array_equal(ix1, ix2)
    assert np.array_equal(vl1.view(np.uint32), vl2.view(np.uint32))
    order = _stable_topk(lg1[0], k)
    assert np.array_equal(ix1[0], order)
    assert np.all(ix1[0] % 3 == 0)
