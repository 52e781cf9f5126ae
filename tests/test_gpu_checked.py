"""The debug build (-DQDQ_CHECKS) on the GPU: every guard holds on valid inputs.

The checked library guards the indices the kernels compute (weight rows and
blocks, shared-memory partial sums, output rows, top-k ids, bulk-copy
alignment): an index out of bounds would skip its access and set a bit of a
device status word instead of faulting.  Here each entry point runs on
several-tile shapes with ragged tails through both builds; the results must be
bit-identical (the guards add no arithmetic) and the status word must stay 0.
"""
import contextlib
import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked(cuda_lib):
    from ggml_quantized_dequant_gb300 import _build
    qdq = cuda_lib
    dbg = ctypes.CDLL(_build.build(checks=True))
    for name, (res, args) in qdq.SIGNATURES.items():
        fn = getattr(dbg, name)
        fn.restype = res
        fn.argtypes = args
    assert dbg.qdq_checks_enabled() == 1
    assert dbg.qdq_check_status() == 0
    return dbg


@contextlib.contextmanager
def _using(qdq, handle):
    old = qdq._lib
    qdq._lib = handle
    try:
        yield
    finally:
        qdq._lib = old


def _dev():
    import torch
    return torch.device("cuda")


def _t(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(_dev())


def _nan(*shape):
    import torch
    return torch.full(shape, float("nan"), dtype=torch.float32, device=_dev())


def _ws(nbytes):
    import torch
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=_dev())


def _same(qdq, dbg, run):
    """run(qdq) -> list of output tensors; both builds must give the same bits."""
    import torch
    ref = [t.cpu().numpy().copy() for t in run(qdq)]
    torch.cuda.synchronize()
    with _using(qdq, dbg):
        got = [t.cpu().numpy().copy() for t in run(qdq)]
        torch.cuda.synchronize()
        assert dbg.qdq_check_status() == 0
        assert dbg.qdq_pipeline_timeouts() == 0
    for a, b in zip(ref, got):
        assert a.dtype == b.dtype and a.shape == b.shape
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def _set_both(qdq, dbg, key, value):
    qdq.set_option(key, value)
    dbg.qdq_set_option(key, value)


@pytest.mark.parametrize("kernel", [0, 1])
@pytest.mark.parametrize("fmt", ["q8_0", "q4k"])
@pytest.mark.parametrize("n_out,n_in,batch", [(2053, 3072, 1), (157, 8192, 1), (300, 1024, 3)])
def test_checked_gemv(cuda_lib, checked, kernel, fmt, n_out, n_in, batch):
    qdq = cuda_lib
    rng = np.random.default_rng(n_out + n_in + batch)
    if fmt == "q8_0":
        W = qdq.upload_q8_0(synth.q8_0_blocks(rng, n_out, n_in), n_out, n_in)
        fn = qdq.q8_0_gemv
    else:
        W = qdq.upload_q4k(synth.q4k_blocks(rng, n_out, n_in), n_out, n_in)
        fn = qdq.q4k_gemv
    x = _t(synth.activations(rng, batch, n_in))

    def run(q):
        y = _nan(batch, n_out)
        fn(W, x, y, n_out, n_in, batch)
        return [y]

    _set_both(qdq, checked, qdq.QDQ_OPT_BATCH1_KERNEL, kernel)
    try:
        _same(qdq, checked, run)
    finally:
        _set_both(qdq, checked, qdq.QDQ_OPT_BATCH1_KERNEL, 0)


@pytest.mark.parametrize("batch", [1, 2])
def test_checked_ffn_and_qkv(cuda_lib, checked, batch):
    qdq = cuda_lib
    rng = np.random.default_rng(11 + batch)
    n_embd, n_ff, n_q, n_kv = 768, 2048, 768, 256
    Wg, Wu = (qdq.upload_q4k(synth.q4k_blocks(rng, n_ff, n_embd), n_ff, n_embd) for _ in range(2))
    Wd = qdq.upload_q4k(synth.q4k_blocks(rng, n_embd, n_ff), n_embd, n_ff)
    Wq = qdq.upload_q4k(synth.q4k_blocks(rng, n_q, n_embd), n_q, n_embd)
    Wk, Wv = (qdq.upload_q4k(synth.q4k_blocks(rng, n_kv, n_embd), n_kv, n_embd) for _ in range(2))
    x = _t(synth.activations(rng, batch, n_embd))
    res = _t(synth.activations(rng, batch, n_embd))

    def run(q):
        out, mid = _nan(batch, n_embd), _nan(batch, n_ff)
        q.q4k_ffn_residual(Wg, Wu, Wd, x, res, out, mid, n_embd, n_ff, batch)
        qq, kk, vv = _nan(batch, n_q), _nan(batch, n_kv), _nan(batch, n_kv)
        q.q4k_qkv(Wq, Wk, Wv, x, qq, kk, vv, n_q, n_kv, n_embd, batch)
        return [out, mid, qq, kk, vv]

    _same(qdq, checked, run)


def test_checked_q6k(cuda_lib, checked):
    import torch
    qdq = cuda_lib
    rng = np.random.default_rng(6)
    n_out, n_in = 3001, 3072
    W = qdq.upload_q6k(synth.q6k_blocks(rng, n_out, n_in), n_out, n_in)
    x1 = _t(synth.activations(rng, 1, n_in))
    x4 = _t(synth.activations(rng, 4, n_in))
    # the two bad ids are rejected by design (NaN rows), not by a guard
    ids = torch.tensor([0, 3000, 17, -1, 3001, 5], dtype=torch.int32, device=_dev())

    def run(q):
        y1, y4, rows = _nan(1, n_out), _nan(4, n_out), _nan(6, n_in)
        q.q6k_gemv(W, x1, y1, n_out, n_in, 1)
        q.q6k_gemv(W, x4, y4, n_out, n_in, 4)
        q.q6k_get_rows(W, ids, rows, 6, n_out, n_in)
        return [y1, y4, rows]

    _same(qdq, checked, run)


@pytest.mark.parametrize("n_in", [1024, 3072])
@pytest.mark.parametrize("batch", [1, 2])
@pytest.mark.parametrize("k", [1, 40, 64])
def test_checked_topk_and_argmax(cuda_lib, checked, k, batch, n_in):
    # batch 1: the projection writes per-CTA candidates (CTAs of fewer than k rows at
    # n_in = 1024, of more at 3072), then the merge rounds; batch 2: the chunked path
    import torch
    qdq = cuda_lib
    rng = np.random.default_rng(40 + k)
    n_vocab = 50003
    W = qdq.upload_q8_0(synth.q8_0_blocks(rng, n_vocab, n_in), n_vocab, n_in)
    x = _t(synth.activations(rng, batch, n_in))

    def run(q):
        logits = _nan(batch, n_vocab)
        idx = torch.full((batch, k), -7, dtype=torch.int32, device=_dev())
        val = _nan(batch, k)
        ws = _ws(q.topk_workspace_bytes(n_vocab, batch, k))
        q.q8_0_logits_topk(W, x, logits, ws, idx, val, n_vocab, n_in, batch, k)
        ai = torch.full((batch,), -7, dtype=torch.int32, device=_dev())
        av = _nan(batch)
        q.q8_0_logits_argmax(W, x, _nan(batch, n_vocab), ai, av, n_vocab, n_in, batch)
        return [logits, idx, val, ai, av]

    _same(qdq, checked, run)


@pytest.mark.parametrize("M", [1, 40, 130, 300])
def test_checked_gemm(cuda_lib, checked, M):
    qdq = cuda_lib
    rng = np.random.default_rng(100 + M)
    n_out, n_in, n_ff = 384, 1024, 512
    W8 = qdq.upload_q8_0(synth.q8_0_blocks(rng, n_out, n_in), n_out, n_in)
    W4 = qdq.upload_q4k(synth.q4k_blocks(rng, n_out, n_in), n_out, n_in)
    Wg, Wu = (qdq.upload_q4k(synth.q4k_blocks(rng, n_ff, n_in), n_ff, n_in) for _ in range(2))
    X = _t(synth.activations(rng, M, n_in))

    def run(q):
        Y8, Y4, mid = _nan(M, n_out), _nan(M, n_out), _nan(M, n_ff)
        ws = _ws(q.gemm_batch_workspace_bytes(M, n_out, n_in))
        q.q8_0_gemm_batch(W8, X, Y8, ws, n_out, n_in, M)
        q.q4k_gemm_batch(W4, X, Y4, ws, n_out, n_in, M)
        ws2 = _ws(q.q4k_swiglu_batch_workspace_bytes(M, n_ff, n_in))
        q.q4k_swiglu_batch(Wg, Wu, X, mid, ws2, n_ff, n_in, M)
        return [Y8, Y4, mid]

    _same(qdq, checked, run)
