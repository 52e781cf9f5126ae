"""Host-side checks of the C-ABI library that need no GPU.

* the shared library loads and exports every function ``include/qdq.h``
  declares, and the Python binding declares a signature for each of them;
* argument validation: NULL pointers, bad dimensions, misaligned pointers and
  aliasing outputs are rejected with the documented status before anything
  touches CUDA (fake, never-dereferenced addresses are enough here);
* the packed-size helpers return the GGML byte counts.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qdq.h")


@pytest.fixture(scope="module")
def lib():
    from ggml_quantized_dequant_gb300 import _build
    import ggml_quantized_dequant_gb300 as qdq
    _build.build()
    return qdq.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qdq_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["qdq_q8_0_gemv", "qdq_q4k_gemv", "qdq_q4k_swiglu", "qdq_q4k_ffn_residual",
                 "qdq_q8_0_gemm_batch", "qdq_q8_0_pack", "qdq_q4k_pack"]:
        assert must in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    import ggml_quantized_dequant_gb300 as qdq
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in qdq.SIGNATURES, name


def test_no_cuda_symbols_in_signatures_are_torch_types():
    # the C ABI uses plain pointers and sizes only
    src = open(HEADER).read()
    assert "torch" not in src.lower().replace("torch types", "")


GOOD = 0x10000000  # a 256-byte aligned fake device address (never dereferenced)


def test_packed_sizes(lib):
    assert lib.qdq_q8_0_packed_bytes(8192, 3072) == 8192 * 3072 // 32 * 34
    assert lib.qdq_q4k_packed_bytes(8192, 3072) == 8192 * 3072 // 256 * 144
    assert lib.qdq_q8_0_packed_bytes(4, 33) == 0
    assert lib.qdq_q4k_packed_bytes(4, 300) == 0
    assert lib.qdq_q8_0_packed_bytes(0, 32) == 0
    # the GEMM workspace size needs a device to query: 0 without one, else X in bf16 above
    # 32 tokens (the SwiGLU: above 16), and a token 256 bytes below
    ws = lib.qdq_gemm_batch_workspace_bytes(16, 8192, 3072)
    assert ws == 0 or ws == 256
    ws = lib.qdq_gemm_batch_workspace_bytes(32, 8192, 3072)
    assert ws == 0 or ws == 256
    ws = lib.qdq_gemm_batch_workspace_bytes(33, 8192, 3072)
    assert ws == 0 or ws >= 33 * 3072 * 2
    ws = lib.qdq_q4k_swiglu_batch_workspace_bytes(17, 8192, 3072)
    assert ws == 0 or ws >= 17 * 3072 * 2
    ws = lib.qdq_gemm_batch_workspace_bytes(512, 8192, 3072)
    assert ws == 0 or ws >= 512 * 3072 * 2
    assert lib.qdq_gemm_batch_workspace_bytes(0, 8192, 3072) == 0


def test_gemv_argument_validation(lib):
    import ggml_quantized_dequant_gb300 as qdq
    W, x, y = GOOD, GOOD + (1 << 28), GOOD + (2 << 28)
    assert lib.qdq_q8_0_gemv(None, x, y, 64, 64, 1, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q8_0_gemv(W, x, y, 64, 48, 1, None) == qdq.QDQ_ERR_DIMS      # n_in % 32
    assert lib.qdq_q8_0_gemv(W, x, y, 0, 64, 1, None) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_q8_0_gemv(W, x, y, 64, 64, 0, None) == qdq.QDQ_ERR_DIMS      # batch 0
    assert lib.qdq_q8_0_gemv(W, x, y, 64, 64, 9, None) == qdq.QDQ_ERR_DIMS      # batch > 8
    assert lib.qdq_q8_0_gemv(W + 8, x, y, 64, 64, 1, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q8_0_gemv(W, x + 4, y, 64, 64, 1, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q8_0_gemv(W, x, y + 2, 64, 64, 1, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q8_0_gemv(W, x, W + 64, 64, 64, 1, None) == qdq.QDQ_ERR_ALIAS  # y inside W
    assert lib.qdq_q8_0_gemv(W, x, x, 64, 64, 1, None) == qdq.QDQ_ERR_ALIAS
    assert lib.qdq_q8_0_gemv(W, x, y, 64, 1 << 20, 1, None) == qdq.QDQ_ERR_UNSUPPORTED
    assert lib.qdq_q4k_gemv(W, x, y, 64, 128, 1, None) == qdq.QDQ_ERR_DIMS       # n_in % 256
    assert lib.qdq_q4k_gemv(W, None, y, 64, 256, 1, None) == qdq.QDQ_ERR_NULL


def test_swiglu_and_ffn_validation(lib):
    import ggml_quantized_dequant_gb300 as qdq
    Wg, Wu, Wd = GOOD, GOOD + (1 << 28), GOOD + (2 << 28)
    x, res, out, mid = GOOD + (3 << 28), GOOD + (4 << 28), GOOD + (5 << 28), GOOD + (6 << 28)
    assert lib.qdq_q4k_swiglu(Wg, None, x, mid, 512, 256, 1, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q4k_swiglu(Wg, Wu, x, mid, 512, 255, 1, None) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_q4k_swiglu(Wg, Wu + 4, x, mid, 512, 256, 1, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q4k_swiglu(Wg, Wu, x, Wu + 16, 512, 256, 1, None) == qdq.QDQ_ERR_ALIAS
    args = dict(n_embd=256, n_ff=512, batch=1)
    f = lambda *p: lib.qdq_q4k_ffn_residual(*p, args["n_embd"], args["n_ff"], args["batch"], None)  # noqa: E731
    assert f(Wg, Wu, Wd, x, res, out, None) == qdq.QDQ_ERR_NULL
    assert f(Wg, Wu, Wd, x, res, out, mid + 4) == qdq.QDQ_ERR_ALIGN
    assert f(Wg, Wu, Wd, x, res, out, x) == qdq.QDQ_ERR_ALIAS            # mid overlaps x
    assert f(Wg, Wu, Wd, x, res, res + 4, mid) == qdq.QDQ_ERR_ALIAS      # partial overlap with residual
    assert f(Wg, Wu, Wd, x, res, x, mid) == qdq.QDQ_ERR_ALIAS            # out over x
    assert lib.qdq_q4k_ffn_residual(Wg, Wu, Wd, x, res, out, mid, 256, 500, 1, None) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_q4k_ffn_residual(Wg, Wu, Wd, x, res, out, mid, 256, 512, 9, None) == qdq.QDQ_ERR_DIMS


def test_qkv_validation(lib):
    import ggml_quantized_dequant_gb300 as qdq
    Wq, Wk, Wv = GOOD, GOOD + (1 << 28), GOOD + (2 << 28)
    x, q, k, v = GOOD + (3 << 28), GOOD + (4 << 28), GOOD + (5 << 28), GOOD + (6 << 28)
    f = lambda *p, n_q=512, n_kv=128, n_embd=256, batch=1: lib.qdq_q4k_qkv(  # noqa: E731
        *p, n_q, n_kv, n_embd, batch, None)
    assert f(Wq, Wk, None, x, q, k, v) == qdq.QDQ_ERR_NULL
    assert f(Wq, Wk, Wv, x, q, k, None) == qdq.QDQ_ERR_NULL
    assert f(Wq, Wk, Wv, x, q, k, v, n_embd=255) == qdq.QDQ_ERR_DIMS
    assert f(Wq, Wk, Wv, x, q, k, v, n_kv=0) == qdq.QDQ_ERR_DIMS
    assert f(Wq, Wk, Wv, x, q, k, v, n_kv=513) == qdq.QDQ_ERR_DIMS         # K/V wider than Q
    assert f(Wq, Wk, Wv, x, q, k, v, batch=9) == qdq.QDQ_ERR_DIMS
    assert f(Wq, Wk + 8, Wv, x, q, k, v) == qdq.QDQ_ERR_ALIGN
    assert f(Wq, Wk, Wv, x + 4, q, k, v) == qdq.QDQ_ERR_ALIGN
    assert f(Wq, Wk, Wv, x, q, k, v + 2) == qdq.QDQ_ERR_ALIGN
    assert f(Wq, Wk, Wv, x, q, q + 4 * 100, v) == qdq.QDQ_ERR_ALIAS        # k inside q
    assert f(Wq, Wk, Wv, x, q, k, Wv + 64) == qdq.QDQ_ERR_ALIAS            # v inside W_v
    assert f(Wq, Wk, Wv, x, x, k, v) == qdq.QDQ_ERR_ALIAS                  # q over x
    assert f(Wq, Wk, Wv, x, q, k, v, n_embd=1 << 20) == qdq.QDQ_ERR_UNSUPPORTED


def test_logits_argmax_validation(lib):
    import ggml_quantized_dequant_gb300 as qdq
    W, x, lg, idx, val = GOOD, GOOD + (1 << 28), GOOD + (2 << 28), GOOD + (3 << 28), GOOD + (4 << 28)
    f = lib.qdq_q8_0_logits_argmax
    assert f(W, x, lg, None, val, 1000, 512, 1, None) == qdq.QDQ_ERR_NULL
    assert f(W, x, lg, idx, val, 1000, 500, 1, None) == qdq.QDQ_ERR_DIMS
    assert f(W, x, lg, idx, val, 1000, 512, 9, None) == qdq.QDQ_ERR_DIMS
    assert f(W, x, lg, idx + 2, val, 1000, 512, 1, None) == qdq.QDQ_ERR_ALIGN
    assert f(W, x, lg, idx, lg + 40, 1000, 512, 1, None) == qdq.QDQ_ERR_ALIAS     # value inside logits
    assert f(W, x, lg, idx, idx + 2 * 4 - 4, 1000, 512, 2, None) == qdq.QDQ_ERR_ALIAS  # index/value overlap
    assert f(W, x, x, idx, val, 1000, 512, 1, None) == qdq.QDQ_ERR_ALIAS          # logits over x


def test_gemm_validation(lib):
    import ggml_quantized_dequant_gb300 as qdq
    W, X, Y, ws = GOOD, GOOD + (1 << 28), GOOD + (2 << 28), GOOD + (3 << 28)
    assert lib.qdq_q8_0_gemm_batch(W, X, Y, None, 256, 512, 16, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q8_0_gemm_batch(W, X, Y, ws, 256, 512, 0, None) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_q8_0_gemm_batch(W, X, Y, ws, 256, 480, 16, None) == qdq.QDQ_ERR_UNSUPPORTED  # n_in % 64
    assert lib.qdq_q8_0_gemm_batch(W, X, Y, ws, 200, 512, 16, None) == qdq.QDQ_ERR_UNSUPPORTED  # n_out % 128
    assert lib.qdq_q8_0_gemm_batch(W, X, Y, ws + 64, 256, 512, 16, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q8_0_gemm_batch(W, X, X, ws, 256, 512, 16, None) == qdq.QDQ_ERR_ALIAS


def test_pack_validation(lib):
    import ggml_quantized_dequant_gb300 as qdq
    assert lib.qdq_q8_0_pack(GOOD, None, 4, 32, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q8_0_pack(GOOD, GOOD + 8, 4, 32, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q8_0_pack(GOOD, GOOD + 16, 4, 32, None) == qdq.QDQ_ERR_ALIAS
    assert lib.qdq_q4k_pack(GOOD, GOOD + (1 << 20), 4, 100, None) == qdq.QDQ_ERR_DIMS


def test_options_and_strings(lib):
    import ggml_quantized_dequant_gb300 as qdq
    assert lib.qdq_set_option(99, 1) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_set_option(qdq.QDQ_OPT_CTAS_PER_SM, 9) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_set_option(qdq.QDQ_OPT_XS_FLOAT_X, 2) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_set_option(qdq.QDQ_OPT_XS_FLOAT_X, 0) == 1  # the f32 arithmetic is the default
    assert lib.qdq_set_option(qdq.QDQ_OPT_XS_FLOAT_X, 1) == 0
    prev = lib.qdq_set_option(qdq.QDQ_OPT_PDL, 0)
    assert prev in (0, 1)
    assert lib.qdq_set_option(qdq.QDQ_OPT_PDL, prev) == 0
    assert b"QDQ_ERR_ALIAS" in lib.qdq_status_string(qdq.QDQ_ERR_ALIAS)
    assert lib.qdq_last_cuda_error() == 0
    assert b"sm_103a" in lib.qdq_version()


def test_q6k_validation_and_sizes(lib):
    import ggml_quantized_dequant_gb300 as qdq
    # packed rows: 210 bytes per 256 weights padded to 16 bytes (none at n_in % 2048 == 0)
    assert lib.qdq_q6k_packed_bytes(5, 3072) == 5 * 2528
    assert lib.qdq_q6k_packed_bytes(5, 8192) == 5 * 8192 // 256 * 210
    assert lib.qdq_q6k_packed_bytes(5, 300) == 0
    W, x, y, ids = GOOD, GOOD + (1 << 28), GOOD + (2 << 28), GOOD + (3 << 28)
    assert lib.qdq_q6k_pack(GOOD, None, 4, 256, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q6k_pack(GOOD, GOOD + 16 * 1024, 4, 255, None) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_q6k_pack(GOOD, GOOD + 8, 4, 256, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q6k_pack(GOOD, GOOD + 16, 4, 256, None) == qdq.QDQ_ERR_ALIAS
    assert lib.qdq_q6k_gemv(W, x, y, 64, 300, 1, None) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_q6k_gemv(W, x, y, 64, 256, 9, None) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_q6k_gemv(W, x + 4, y, 64, 256, 1, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q6k_gemv(W, x, W + 16, 64, 256, 1, None) == qdq.QDQ_ERR_ALIAS
    assert lib.qdq_q6k_dequant(W, None, 64, 256, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q6k_get_rows(W, None, y, 4, 64, 256, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q6k_get_rows(W, ids, y, -1, 64, 256, None) == qdq.QDQ_ERR_DIMS
    assert lib.qdq_q6k_get_rows(W, ids + 2, y, 4, 64, 256, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q6k_get_rows(W, ids, ids, 4, 64, 256, None) == qdq.QDQ_ERR_ALIAS
    assert lib.qdq_q6k_get_rows(W, ids, y, 0, 64, 256, None) == qdq.QDQ_OK   # empty: nothing launched


def test_topk_validation_and_sizes(lib):
    import ggml_quantized_dequant_gb300 as qdq
    # two rounds of candidate keys: batch * ceil(n / 1024) * k 8-byte keys each
    assert lib.qdq_topk_workspace_bytes(128256, 2, 40) == 2 * 2 * 126 * 40 * 8
    assert lib.qdq_topk_workspace_bytes(100, 1, 101) == 0
    assert lib.qdq_topk_workspace_bytes(1000, 1, qdq.QDQ_MAX_TOPK + 1) == 0
    lg, ws, idx, val = GOOD, GOOD + (1 << 28), GOOD + (2 << 28), GOOD + (3 << 28)
    f = lib.qdq_topk_rows
    assert f(lg, 1000, 1, 8, None, idx, val, None) == qdq.QDQ_ERR_NULL
    assert f(lg, 1000, 1, 0, ws, idx, val, None) == qdq.QDQ_ERR_DIMS
    assert f(lg, 5, 1, 6, ws, idx, val, None) == qdq.QDQ_ERR_DIMS             # k > n
    assert f(lg, 1000, 0, 8, ws, idx, val, None) == qdq.QDQ_ERR_DIMS
    assert f(lg, 1000, 1, 65, ws, idx, val, None) == qdq.QDQ_ERR_UNSUPPORTED
    assert f(lg, 1000, 1, 8, ws + 8, idx, val, None) == qdq.QDQ_ERR_ALIGN
    assert f(lg, 1000, 1, 8, ws, idx, lg + 64, None) == qdq.QDQ_ERR_ALIAS    # value inside the logits
    assert f(lg, 1000, 1, 8, ws, idx, idx + 16, None) == qdq.QDQ_ERR_ALIAS   # value over index
    assert f(lg, 1000, 1, 8, lg + 16, idx, val, None) == qdq.QDQ_ERR_ALIAS   # workspace over the logits
    W, x = GOOD + (4 << 28), GOOD + (5 << 28)
    g = lib.qdq_q8_0_logits_topk
    assert g(W, x, lg, ws, idx, val, 1000, 500, 1, 8, None) == qdq.QDQ_ERR_DIMS
    assert g(W, x, lg, ws, idx, val, 1000, 512, 1, 0, None) == qdq.QDQ_ERR_DIMS
    assert g(W, x, lg, ws, idx, x, 1000, 512, 1, 8, None) == qdq.QDQ_ERR_ALIAS   # value over x
    assert g(W, x, lg, W + 16, idx, val, 1000, 512, 1, 8, None) == qdq.QDQ_ERR_ALIAS


def test_q4k_gemm_and_swiglu_batch_validation(lib):
    import ggml_quantized_dequant_gb300 as qdq
    W, X, Y, ws, W2 = GOOD, GOOD + (1 << 28), GOOD + (2 << 28), GOOD + (3 << 28), GOOD + (4 << 28)
    assert lib.qdq_q4k_gemm_batch(W, X, Y, None, 256, 512, 16, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q4k_gemm_batch(W, X, Y, ws, 256, 320, 16, None) == qdq.QDQ_ERR_DIMS       # n_in % 256
    assert lib.qdq_q4k_gemm_batch(W, X, Y, ws, 200, 512, 16, None) == qdq.QDQ_ERR_UNSUPPORTED  # n_out % 128
    assert lib.qdq_q4k_gemm_batch(W, X, Y, ws + 128, 256, 512, 16, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q4k_gemm_batch(W, X, W + 16, ws, 256, 512, 16, None) == qdq.QDQ_ERR_ALIAS
    assert lib.qdq_q4k_swiglu_batch(W, None, X, Y, ws, 512, 256, 16, None) == qdq.QDQ_ERR_NULL
    assert lib.qdq_q4k_swiglu_batch(W, W2 + 8, X, Y, ws, 512, 256, 16, None) == qdq.QDQ_ERR_ALIGN
    assert lib.qdq_q4k_swiglu_batch(W, W2, X, W2 + 64, ws, 512, 256, 16, None) == qdq.QDQ_ERR_ALIAS
    assert lib.qdq_q4k_swiglu_batch(W, W2, X, Y, ws, 512, 256, 0, None) == qdq.QDQ_ERR_DIMS


def test_normal_build_has_no_checks(lib):
    # the guards compile to nothing in the normal build: no status word, nothing to read
    assert lib.qdq_checks_enabled() == 0
    assert lib.qdq_check_status() == 0


def test_checked_build_links_and_exports_the_same_symbols():
    import ctypes
    from ggml_quantized_dequant_gb300 import _build
    path = _build.build(checks=True)
    assert path != _build.LIB
    dbg = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(dbg, name), name
    dbg.qdq_checks_enabled.restype = ctypes.c_int
    assert dbg.qdq_checks_enabled() == 1
