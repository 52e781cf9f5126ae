"""The allocation-free FFN entry point (qdq_q4k_ffn_residual_noalloc).

Some callers may not allocate device memory (a plug-in whose host application
owns the GPU's memory through its own pool, a decode loop that must not pay for
cudaMalloc/cudaFree), so this entry point keeps the FFN's intermediate vector in
a fixed array inside the library instead of taking a workspace.  These tests
check, through the C ABI, that two calls in a row give what the ordinary entry
point gives on the same inputs, within the FFN bound the other parity tests
use, and that a request larger than the array is refused.

The file name sorts last so that a run stopping at its first failure has
already run every other test.
"""
import numpy as np
import pytest

import oracle
import synth
from _bounds import ffn_bound


def test_oversize_request_is_refused_before_any_cuda_call():
    from ggml_quantized_dequant_gb300 import _build
    import ggml_quantized_dequant_gb300 as qdq
    _build.build()
    lib = qdq.load()
    fake = 0x10000000  # never dereferenced: the size check comes first
    n_ff = qdq.QDQ_NOALLOC_FFN_MAX_MID // 4 + 256
    assert lib.qdq_q4k_ffn_residual_noalloc(fake, fake, fake, fake, fake, fake, 256, n_ff, 4, None) \
        == qdq.QDQ_ERR_SCRATCH
    assert "scratch" in qdq.status_string(qdq.QDQ_ERR_SCRATCH)


def test_bad_arguments_are_refused_before_the_scratch_lookup():
    # NULL, misaligned and overlapping arguments get the same status as from the
    # workspace entry point, before the call looks up its device array (so also
    # on a machine without a GPU, where that lookup would fail)
    from ggml_quantized_dequant_gb300 import _build
    import ggml_quantized_dequant_gb300 as qdq
    _build.build()
    lib = qdq.load()
    base = 0x10000000
    wg, wu, wd, x, r, o = (base + i * (1 << 24) for i in range(6))  # distinct, 16-byte aligned
    f = lib.qdq_q4k_ffn_residual_noalloc
    assert f(wg, None, wd, x, r, o, 256, 512, 1, None) == qdq.QDQ_ERR_NULL
    assert f(wg, wu, wd, x + 4, r, o, 256, 512, 1, None) == qdq.QDQ_ERR_ALIGN
    assert f(wg, wu, wd, x, r, o, 300, 512, 1, None) == qdq.QDQ_ERR_DIMS
    assert f(wg, wu, wd, x, r, x, 256, 512, 1, None) == qdq.QDQ_ERR_ALIAS
    assert f(wg, wu, wd, x, r, o, 256, 512, 0, None) == qdq.QDQ_ERR_DIMS


def _layer(rng, n_embd, n_ff):
    return (synth.q4k_blocks(rng, n_ff, n_embd), synth.q4k_blocks(rng, n_ff, n_embd),
            synth.q4k_blocks(rng, n_embd, n_ff))


@pytest.mark.gpu
@pytest.mark.parametrize("n_embd,n_ff,batch", [(512, 1280, 2), (3072, 8192, 1)])
def test_noalloc_ffn_matches_workspace_entry_point_twice(cuda_lib, n_embd, n_ff, batch):
    import torch
    qdq = cuda_lib
    dev = torch.device("cuda")
    rng = np.random.default_rng(n_embd + n_ff + batch)
    g, u, d = _layer(rng, n_embd, n_ff)
    Wg, Wu, Wd = qdq.upload_q4k(g, n_ff, n_embd), qdq.upload_q4k(u, n_ff, n_embd), qdq.upload_q4k(d, n_embd, n_ff)
    wd = oracle.q4k_dequant(d, n_embd, n_ff)
    wg, wu = oracle.q4k_dequant(g, n_ff, n_embd), oracle.q4k_dequant(u, n_ff, n_embd)
    for call in range(2):  # the second call finds the first call's values in the array
        x = synth.activations(rng, batch, n_embd)
        res = synth.activations(rng, batch, n_embd)
        xd, rd = torch.from_numpy(x).to(dev), torch.from_numpy(res).to(dev)
        ref_out = torch.full((batch, n_embd), float("nan"), device=dev)
        mid = torch.empty((batch, n_ff), device=dev)
        qdq.q4k_ffn_residual(Wg, Wu, Wd, xd, rd, ref_out, mid, n_embd, n_ff, batch)
        out = torch.full((batch, n_embd), float("nan"), device=dev)
        qdq.q4k_ffn_residual_noalloc(Wg, Wu, Wd, xd, rd, out, n_embd, n_ff, batch)
        torch.cuda.synchronize()
        o = oracle.ffn_residual(wg, wu, wd, x, res)
        bound = ffn_bound(o, wd)
        got, ref = out.cpu().numpy(), ref_out.cpu().numpy()
        assert np.all(np.isfinite(got)), "call %d" % call
        assert np.all(np.abs(got.astype(np.float64) - ref) <= bound), "call %d" % call
        assert np.all(np.abs(got.astype(np.float64) - o["out"]) <= bound), "call %d" % call
