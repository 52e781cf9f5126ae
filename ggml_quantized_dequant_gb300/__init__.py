"""Python binding of the qdq CUDA library (libqdq.so): argument marshalling only.

Every function here takes torch CUDA tensors (or raw device pointers as ints),
passes their addresses, sizes and the current CUDA stream to the C ABI declared
in ``include/qdq.h``, and raises :class:`QdqError` on a non-zero status.  All
arithmetic runs in the CUDA kernels; there is no CPU path.  The library is
built in-tree by ``__graft_entry__.build()`` (or ``python -m
ggml_quantized_dequant_gb300._build``); loading fails loudly if it is absent.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqdq.so")

QDQ_OK = 0
QDQ_ERR_NULL = -1
QDQ_ERR_DIMS = -2
QDQ_ERR_ALIGN = -3
QDQ_ERR_UNSUPPORTED = -4
QDQ_ERR_CUDA = -5
QDQ_ERR_ALIAS = -6
QDQ_ERR_SCRATCH = -7
QDQ_NOALLOC_FFN_MAX_MID = 262144
QDQ_MAX_GEMV_BATCH = 8
QDQ_MAX_TOPK = 64
QDQ_MAX_GEMV_N_IN = 32768
QDQ_OPT_PDL = 1
QDQ_OPT_L2_PREFETCH = 2
QDQ_OPT_CTAS_PER_SM = 3
QDQ_OPT_XS_GROUPS = 4
QDQ_OPT_XS_STAGES = 5
QDQ_OPT_XS_FLOAT_X = 6
QDQ_OPT_BATCH1_KERNEL = 7

_c_int, _c_size, _c_vp, _c_char_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_char_p

# name -> (restype, argtypes); mirrors include/qdq.h
SIGNATURES = {
    "qdq_status_string": (_c_char_p, [_c_int]),
    "qdq_last_cuda_error": (_c_int, []),
    "qdq_version": (_c_char_p, []),
    "qdq_q8_0_packed_bytes": (_c_size, [_c_int, _c_int]),
    "qdq_q4k_packed_bytes": (_c_size, [_c_int, _c_int]),
    "qdq_q8_0_pack": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_vp]),
    "qdq_q4k_pack": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_vp]),
    "qdq_q8_0_dequant": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_vp]),
    "qdq_q4k_dequant": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_vp]),
    "qdq_q8_0_gemv": (_c_int, [_c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q4k_gemv": (_c_int, [_c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q4k_swiglu": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q8_0_logits_argmax": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q4k_qkv": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int,
                             _c_vp]),
    "qdq_q4k_ffn_residual": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                      _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q4k_ffn_residual_noalloc": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                              _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q6k_packed_bytes": (_c_size, [_c_int, _c_int]),
    "qdq_q6k_pack": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_vp]),
    "qdq_q6k_dequant": (_c_int, [_c_vp, _c_vp, _c_int, _c_int, _c_vp]),
    "qdq_q6k_gemv": (_c_int, [_c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q6k_get_rows": (_c_int, [_c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_topk_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "qdq_topk_rows": (_c_int, [_c_vp, _c_int, _c_int, _c_int, _c_vp, _c_vp, _c_vp, _c_vp]),
    "qdq_q8_0_logits_topk": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_int,
                                      _c_vp]),
    "qdq_gemm_batch_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "qdq_q8_0_gemm_batch": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q4k_gemm_batch": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_q4k_swiglu_batch_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "qdq_q4k_swiglu_batch": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_int, _c_int, _c_int, _c_vp]),
    "qdq_pipeline_timeouts": (_c_int, []),
    "qdq_noop": (_c_int, [_c_vp]),
    "qdq_check_status": (_c_int, []),
    "qdq_checks_enabled": (_c_int, []),
    "qdq_set_option": (_c_int, [_c_int, _c_int]),
}

_lib = None


class QdqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = "%s failed: %s" % (fn, status_string(status))
        if status == QDQ_ERR_CUDA and _lib is not None:
            msg += " (cudaError %d)" % _lib.qdq_last_cuda_error()
        super().__init__(msg)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libqdq.so (once) and declare every entry point's signature."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("libqdq.so is not built (%s); run __graft_entry__.build()" % p)
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def lib() -> ctypes.CDLL:
    return load()


def status_string(status: int) -> str:
    if _lib is None:
        return str(status)
    return _lib.qdq_status_string(int(status)).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) or None
    if isinstance(stream, int):
        return stream or None
    return int(stream.cuda_stream) or None


def _check(name: str, status: int):
    if status != QDQ_OK:
        raise QdqError(name, status)


# ---------------------------------------------------------------- C-ABI mirrors

def q8_0_packed_bytes(n_out: int, n_in: int) -> int:
    return int(lib().qdq_q8_0_packed_bytes(n_out, n_in))


def q4k_packed_bytes(n_out: int, n_in: int) -> int:
    return int(lib().qdq_q4k_packed_bytes(n_out, n_in))


def q8_0_pack(ggml, packed, n_out: int, n_in: int, stream=None):
    _check("qdq_q8_0_pack", lib().qdq_q8_0_pack(_ptr(ggml), _ptr(packed), n_out, n_in, _stream(stream)))


def q4k_pack(ggml, packed, n_out: int, n_in: int, stream=None):
    _check("qdq_q4k_pack", lib().qdq_q4k_pack(_ptr(ggml), _ptr(packed), n_out, n_in, _stream(stream)))


def q8_0_dequant(W, out, n_out: int, n_in: int, stream=None):
    _check("qdq_q8_0_dequant", lib().qdq_q8_0_dequant(_ptr(W), _ptr(out), n_out, n_in, _stream(stream)))


def q4k_dequant(W, out, n_out: int, n_in: int, stream=None):
    _check("qdq_q4k_dequant", lib().qdq_q4k_dequant(_ptr(W), _ptr(out), n_out, n_in, _stream(stream)))


def q8_0_gemv(W, x, y, n_out: int, n_in: int, batch: int = 1, stream=None):
    _check("qdq_q8_0_gemv", lib().qdq_q8_0_gemv(_ptr(W), _ptr(x), _ptr(y), n_out, n_in, batch, _stream(stream)))


def q4k_gemv(W, x, y, n_out: int, n_in: int, batch: int = 1, stream=None):
    _check("qdq_q4k_gemv", lib().qdq_q4k_gemv(_ptr(W), _ptr(x), _ptr(y), n_out, n_in, batch, _stream(stream)))


def q4k_swiglu(Wg, Wu, x, mid, n_ff: int, n_embd: int, batch: int = 1, stream=None):
    _check("qdq_q4k_swiglu", lib().qdq_q4k_swiglu(_ptr(Wg), _ptr(Wu), _ptr(x), _ptr(mid), n_ff, n_embd, batch,
                                                  _stream(stream)))


def q8_0_logits_argmax(W, x, logits, index, value, n_vocab: int, n_in: int, batch: int = 1, stream=None):
    """Output projection plus on-device argmax: ``index`` (int32) and ``value`` (f32) per batch row."""
    _check("qdq_q8_0_logits_argmax",
           lib().qdq_q8_0_logits_argmax(_ptr(W), _ptr(x), _ptr(logits), _ptr(index), _ptr(value), n_vocab, n_in,
                                        batch, _stream(stream)))


def q4k_qkv(Wq, Wk, Wv, x, q, k, v, n_q: int, n_kv: int, n_embd: int, batch: int = 1, stream=None):
    _check("qdq_q4k_qkv", lib().qdq_q4k_qkv(_ptr(Wq), _ptr(Wk), _ptr(Wv), _ptr(x), _ptr(q), _ptr(k), _ptr(v),
                                            n_q, n_kv, n_embd, batch, _stream(stream)))


def q4k_ffn_residual(Wg, Wu, Wd, x, residual, out, mid_workspace, n_embd: int, n_ff: int, batch: int = 1,
                     stream=None):
    _check("qdq_q4k_ffn_residual",
           lib().qdq_q4k_ffn_residual(_ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(x), _ptr(residual), _ptr(out),
                                      _ptr(mid_workspace), n_embd, n_ff, batch, _stream(stream)))


def q4k_ffn_residual_noalloc(Wg, Wu, Wd, x, residual, out, n_embd: int, n_ff: int, batch: int = 1, stream=None):
    """The FFN block with its intermediate vector in the library's fixed device array (no allocation).

    For callers that may not allocate device memory.  batch * n_ff must not exceed
    QDQ_NOALLOC_FFN_MAX_MID; calls that overlap on the GPU share the array and race.
    """
    _check("qdq_q4k_ffn_residual_noalloc",
           lib().qdq_q4k_ffn_residual_noalloc(_ptr(Wg), _ptr(Wu), _ptr(Wd), _ptr(x), _ptr(residual), _ptr(out),
                                              n_embd, n_ff, batch, _stream(stream)))


def q6k_packed_bytes(n_out: int, n_in: int) -> int:
    return int(lib().qdq_q6k_packed_bytes(n_out, n_in))


def q6k_pack(ggml, packed, n_out: int, n_in: int, stream=None):
    _check("qdq_q6k_pack", lib().qdq_q6k_pack(_ptr(ggml), _ptr(packed), n_out, n_in, _stream(stream)))


def q6k_dequant(W, out, n_out: int, n_in: int, stream=None):
    _check("qdq_q6k_dequant", lib().qdq_q6k_dequant(_ptr(W), _ptr(out), n_out, n_in, _stream(stream)))


def q6k_gemv(W, x, y, n_out: int, n_in: int, batch: int = 1, stream=None):
    _check("qdq_q6k_gemv", lib().qdq_q6k_gemv(_ptr(W), _ptr(x), _ptr(y), n_out, n_in, batch, _stream(stream)))


def q6k_get_rows(W, ids, out, n_ids: int, n_rows: int, n_in: int, stream=None):
    """Embedding lookup: ``out[i] = dequantised row ids[i]`` (int32 ids on the device)."""
    _check("qdq_q6k_get_rows", lib().qdq_q6k_get_rows(_ptr(W), _ptr(ids), _ptr(out), n_ids, n_rows, n_in,
                                                      _stream(stream)))


def topk_workspace_bytes(n: int, batch: int, k: int) -> int:
    return int(lib().qdq_topk_workspace_bytes(n, batch, k))


def topk_rows(logits, n: int, batch: int, k: int, workspace, index, value, stream=None):
    """Per row of ``logits``: the k best (index, value) pairs, NaN first, larger first, smaller index on ties."""
    _check("qdq_topk_rows", lib().qdq_topk_rows(_ptr(logits), n, batch, k, _ptr(workspace), _ptr(index), _ptr(value),
                                                _stream(stream)))


def q8_0_logits_topk(W, x, logits, workspace, index, value, n_vocab: int, n_in: int, batch: int, k: int,
                     stream=None):
    _check("qdq_q8_0_logits_topk",
           lib().qdq_q8_0_logits_topk(_ptr(W), _ptr(x), _ptr(logits), _ptr(workspace), _ptr(index), _ptr(value),
                                      n_vocab, n_in, batch, k, _stream(stream)))


def gemm_batch_workspace_bytes(M: int, n_out: int, n_in: int) -> int:
    """Workspace bytes of the tensor-core batch GEMMs on the current device (the bf16 copy of X)."""
    return int(lib().qdq_gemm_batch_workspace_bytes(M, n_out, n_in))


def q8_0_gemm_batch(W, X, Y, workspace, n_out: int, n_in: int, M: int, stream=None):
    _check("qdq_q8_0_gemm_batch", lib().qdq_q8_0_gemm_batch(_ptr(W), _ptr(X), _ptr(Y), _ptr(workspace), n_out,
                                                            n_in, M, _stream(stream)))


def q4k_gemm_batch(W, X, Y, workspace, n_out: int, n_in: int, M: int, stream=None):
    _check("qdq_q4k_gemm_batch", lib().qdq_q4k_gemm_batch(_ptr(W), _ptr(X), _ptr(Y), _ptr(workspace), n_out,
                                                          n_in, M, _stream(stream)))


def q4k_swiglu_batch_workspace_bytes(M: int, n_ff: int, n_embd: int) -> int:
    return int(lib().qdq_q4k_swiglu_batch_workspace_bytes(M, n_ff, n_embd))


def q4k_swiglu_batch(Wg, Wu, X, mid, workspace, n_ff: int, n_embd: int, M: int, stream=None):
    _check("qdq_q4k_swiglu_batch", lib().qdq_q4k_swiglu_batch(_ptr(Wg), _ptr(Wu), _ptr(X), _ptr(mid),
                                                              _ptr(workspace), n_ff, n_embd, M, _stream(stream)))


def noop(stream=None):
    """One empty kernel on the stream (for the launch round-trip measurement)."""
    _check("qdq_noop", lib().qdq_noop(_stream(stream)))


def pipeline_timeouts() -> int:
    return int(lib().qdq_pipeline_timeouts())


def set_option(key: int, value: int) -> int:
    r = int(lib().qdq_set_option(key, value))
    if r < 0:
        raise QdqError("qdq_set_option", r)
    return r


# ---------------------------------------------------------------- upload helpers
# (device memory comes from torch; the repack itself runs in the CUDA kernels)

def upload_q8_0(ggml_bytes, n_out: int, n_in: int, device="cuda", stream=None):
    """Copy raw GGML Q8_0 bytes (numpy uint8 or torch) to the device and repack them; returns the packed tensor."""
    import torch
    raw = torch.as_tensor(ggml_bytes, dtype=torch.uint8).reshape(-1).to(device)
    packed = torch.empty(q8_0_packed_bytes(n_out, n_in), dtype=torch.uint8, device=device)
    q8_0_pack(raw, packed, n_out, n_in, stream)
    return packed


def upload_q6k(ggml_bytes, n_out: int, n_in: int, device="cuda", stream=None):
    """Copy raw GGML Q6_K bytes (numpy uint8 or torch) to the device and repack them; returns the packed tensor."""
    import torch
    raw = torch.as_tensor(ggml_bytes, dtype=torch.uint8).reshape(-1).to(device)
    packed = torch.empty(q6k_packed_bytes(n_out, n_in), dtype=torch.uint8, device=device)
    q6k_pack(raw, packed, n_out, n_in, stream)
    return packed


def upload_q4k(ggml_bytes, n_out: int, n_in: int, device="cuda", stream=None):
    """Copy raw GGML Q4_K bytes (numpy uint8 or torch) to the device and repack them; returns the packed tensor."""
    import torch
    raw = torch.as_tensor(ggml_bytes, dtype=torch.uint8).reshape(-1).to(device)
    packed = torch.empty(q4k_packed_bytes(n_out, n_in), dtype=torch.uint8, device=device)
    q4k_pack(raw, packed, n_out, n_in, stream)
    return packed
