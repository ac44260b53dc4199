"""Thin ctypes binding of libqvg.so (include/qvg.h): argument marshalling only.

Every function has the C name and forwards to the C ABI; torch tensors supply
device memory and the current CUDA stream.  Nothing here computes: a missing
library raises, there is no fallback path.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqvg.so")

QVG_OK, QVG_ERR_INVALID_ARG, QVG_ERR_UNSUPPORTED, QVG_ERR_CAPACITY, QVG_ERR_CUDA, QVG_ERR_TIMEOUT = range(6)

EXPORTS = [
    "qvg_last_error", "qvg_version", "qvg_encoded_bytes", "qvg_workspace_bytes", "qvg_fit_stats",
    "qvg_fit_centroids",
    "qvg_assign", "qvg_update", "qvg_encode", "qvg_decode", "qvg_append_chunk", "qvg_decode_cache",
    "coral_predict_encode", "coral_predict_decode", "coral_predict_encode_static", "coral_fit_block",
    "coral_prepared_bytes", "coral_prepare_predictor",
    "coral_sas_workspace_bytes", "coral_sas_encode", "coral_sas_decode", "qvg_attention_decode",
    "qvg_attention_workspace_bytes", "qvg_attention_decode_staged", "qvg_compress_host",
    "qvg_device_error", "qvg_debug_set_wait",
]


class QvgError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"qvg status {status}: {msg}")
        self.status = status


class qvg_config(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("num_clusters", ctypes.c_int32), ("lloyd_iters", ctypes.c_int32),
                ("num_stages", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("group_size", ctypes.c_int32)]


class qvg_cache(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("meta", ctypes.c_void_p), ("ids", ctypes.c_void_p),
                ("centroids", ctypes.c_void_p), ("chunk_offset", ctypes.c_void_p),
                ("chunk_version", ctypes.c_void_p), ("capacity", ctypes.c_int64),
                ("max_versions", ctypes.c_int32), ("max_chunks", ctypes.c_int32),
                ("n_used", ctypes.c_int64), ("n_versions", ctypes.c_int32), ("n_chunks", ctypes.c_int32)]


class coral_predictor(ctypes.Structure):
    _fields_ = [("B", ctypes.c_void_p), ("U", ctypes.c_void_p), ("W", ctypes.c_void_p),
                ("rank", ctypes.c_int32), ("prepared", ctypes.c_void_p)]


class qvg_encoded_view(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("meta", ctypes.c_void_p), ("ids", ctypes.c_void_p),
                ("centroids", ctypes.c_void_p)]


_lib = None
P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
PCFG = ctypes.POINTER(qvg_config)
PSZ = ctypes.POINTER(ctypes.c_size_t)


def load(path=LIB_PATH):
    """Load libqvg.so (built by ``build.py`` / ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m kv_cache_quantization_means_b300.build`")
    L = ctypes.CDLL(path)
    L.qvg_last_error.restype = ctypes.c_char_p
    L.qvg_version.restype = ctypes.c_char_p
    L.qvg_encoded_bytes.argtypes = [PCFG, I64, I32, PSZ, PSZ, PSZ, PSZ]
    L.qvg_workspace_bytes.argtypes = [PCFG, I64, PSZ]
    L.qvg_fit_stats.argtypes = [PCFG, I64, P, SZ, ctypes.POINTER(ctypes.c_uint64), P]
    L.qvg_fit_centroids.argtypes = [PCFG, P, I64, I64, I64, P, P, P, I64, I64, P, SZ, P]
    L.qvg_assign.argtypes = [PCFG, P, I64, I64, I64, P, P, I64, I64, P, SZ, P]
    L.qvg_update.argtypes = [PCFG, P, I64, I64, I64, P, I64, I64, P, P, SZ, P]
    L.qvg_encode.argtypes = [PCFG, P, I64, I64, I64, P, I32, P, P, P, I64, I64, P, SZ, P]
    L.qvg_decode.argtypes = [PCFG, P, P, P, P, I64, I64, I64, P, I64, I64, P]
    L.qvg_append_chunk.argtypes = [PCFG, ctypes.POINTER(qvg_cache), P, I64, I64, I64, I32, P, SZ, P]
    L.qvg_decode_cache.argtypes = [PCFG, ctypes.POINTER(qvg_cache), I64, I64, P, I64, I64, P]
    L.coral_predict_encode.argtypes = [PCFG, ctypes.POINTER(coral_predictor), P, P, I64, P, P, P, P, P, SZ, P]
    L.coral_predict_encode_static.argtypes = [PCFG, ctypes.POINTER(coral_predictor), P, P, I64, P, P, P, P, P]
    L.coral_predict_decode.argtypes = [PCFG, ctypes.POINTER(coral_predictor), P, I64, P, P, P, P, P, SZ, P]
    L.coral_fit_block.argtypes = [PCFG, ctypes.POINTER(coral_predictor), P, P, I64, P, P, SZ, P]
    L.coral_prepared_bytes.argtypes = [PCFG, I32, PSZ]
    L.coral_prepare_predictor.argtypes = [PCFG, ctypes.POINTER(coral_predictor), P, SZ, P]
    L.coral_sas_workspace_bytes.argtypes = [PCFG, I64, PSZ]
    L.coral_sas_encode.argtypes = [PCFG, ctypes.POINTER(coral_predictor), P, P, I64, P, P, P, P, P, P, P, SZ, P]
    L.coral_sas_decode.argtypes = [PCFG, ctypes.POINTER(coral_predictor), P, I64, P, P, P, P, P, P, P, SZ, P]
    L.qvg_attention_decode.argtypes = [PCFG, P, I64, I64, I64, ctypes.POINTER(qvg_encoded_view),
                                       ctypes.POINTER(qvg_encoded_view), I64, I64, ctypes.c_float, P, I64, I64, P]
    L.qvg_attention_workspace_bytes.argtypes = [PCFG, I64, PSZ]
    L.qvg_attention_decode_staged.argtypes = [PCFG, P, I64, I64, I64, ctypes.POINTER(qvg_encoded_view),
                                              ctypes.POINTER(qvg_encoded_view), I64, I64, ctypes.c_float, P, I64,
                                              I64, P, ctypes.c_size_t, P]
    L.qvg_compress_host.argtypes = [PCFG, P, P, I64, I64, I64, P, P, P, P, P, P, P, SZ, P, SZ, P]
    L.qvg_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), I32, P]
    L.qvg_debug_set_wait.argtypes = [ctypes.c_uint64, ctypes.c_uint32, P]
    for name in EXPORTS[2:]:
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(st):
    if st != QVG_OK:
        raise QvgError(st, load().qvg_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def config(num_heads, head_dim, num_clusters, lloyd_iters, num_stages, group_size, bits=2):
    return qvg_config(num_heads, head_dim, num_clusters, lloyd_iters, num_stages, bits, group_size)


# ------------------------------------------------------------ the C calls --

def qvg_version():
    return load().qvg_version().decode()


def qvg_encoded_bytes(cfg, capacity, n_versions=1):
    out = [ctypes.c_size_t() for _ in range(4)]
    _check(load().qvg_encoded_bytes(ctypes.byref(cfg), capacity, n_versions, *[ctypes.byref(o) for o in out]))
    return tuple(o.value for o in out)


def qvg_workspace_bytes(cfg, n_tokens):
    b = ctypes.c_size_t()
    _check(load().qvg_workspace_bytes(ctypes.byref(cfg), n_tokens, ctypes.byref(b)))
    return b.value


def qvg_fit_stats(cfg, n_tokens, workspace, stream=None, with_status=False):
    """The four counters; with_status=True returns (status, counters) and
    accepts QVG_ERR_TIMEOUT (error word set) instead of raising."""
    out = (ctypes.c_uint64 * 4)()
    st = load().qvg_fit_stats(ctypes.byref(cfg), n_tokens, _ptr(workspace), _nbytes(workspace), out,
                              _stream(stream))
    if not (with_status and st == QVG_ERR_TIMEOUT):
        _check(st)
    stats = tuple(int(v) for v in out)
    return (st, stats) if with_status else stats


def qvg_device_error(clear=False, stream=None):
    """(status, error word): QVG_ERR_TIMEOUT with the word when it was set."""
    out = ctypes.c_uint32(0)
    st = load().qvg_device_error(ctypes.byref(out), 1 if clear else 0, _stream(stream))
    if st not in (QVG_OK, QVG_ERR_TIMEOUT):
        _check(st)
    return st, out.value


def qvg_debug_set_wait(wait_limit_ns, flags=0, stream=None):
    _check(load().qvg_debug_set_wait(wait_limit_ns, flags, _stream(stream)))


def qvg_fit_centroids(cfg, x, n_tokens, head_stride, token_stride, warm_start, centroids, ids, capacity,
                      tok_offset, workspace, stream=None):
    _check(load().qvg_fit_centroids(ctypes.byref(cfg), _ptr(x), n_tokens, head_stride, token_stride,
                                    _ptr(warm_start), _ptr(centroids), _ptr(ids), capacity, tok_offset,
                                    _ptr(workspace), _nbytes(workspace), _stream(stream)))


def qvg_assign(cfg, x, n_tokens, head_stride, token_stride, centroids, ids, capacity, tok_offset, workspace,
               stream=None):
    _check(load().qvg_assign(ctypes.byref(cfg), _ptr(x), n_tokens, head_stride, token_stride, _ptr(centroids),
                             _ptr(ids), capacity, tok_offset, _ptr(workspace), _nbytes(workspace), _stream(stream)))


def qvg_update(cfg, x, n_tokens, head_stride, token_stride, ids, capacity, tok_offset, centroids, workspace,
               stream=None):
    _check(load().qvg_update(ctypes.byref(cfg), _ptr(x), n_tokens, head_stride, token_stride, _ptr(ids), capacity,
                             tok_offset, _ptr(centroids), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def qvg_encode(cfg, x, n_tokens, head_stride, token_stride, centroids, assign, codes, meta, ids, capacity,
               tok_offset, workspace=None, stream=None):
    _check(load().qvg_encode(ctypes.byref(cfg), _ptr(x), n_tokens, head_stride, token_stride, _ptr(centroids),
                             int(assign), _ptr(codes), _ptr(meta), _ptr(ids), capacity, tok_offset,
                             _ptr(workspace), _nbytes(workspace), _stream(stream)))


def qvg_decode(cfg, codes, meta, ids, centroids, capacity, tok_begin, tok_end, out, out_head_stride,
               out_token_stride, stream=None):
    _check(load().qvg_decode(ctypes.byref(cfg), _ptr(codes), _ptr(meta), _ptr(ids), _ptr(centroids), capacity,
                             tok_begin, tok_end, _ptr(out), out_head_stride, out_token_stride, _stream(stream)))


def qvg_append_chunk(cfg, cache, x, n_new, head_stride, token_stride, refit, workspace, stream=None):
    _check(load().qvg_append_chunk(ctypes.byref(cfg), ctypes.byref(cache), _ptr(x), n_new, head_stride,
                                   token_stride, int(refit), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def qvg_decode_cache(cfg, cache, tok_begin, tok_end, out, out_head_stride, out_token_stride, stream=None):
    _check(load().qvg_decode_cache(ctypes.byref(cfg), ctypes.byref(cache), tok_begin, tok_end, _ptr(out),
                                   out_head_stride, out_token_stride, _stream(stream)))


def coral_predict_encode(cfg, pred, xhat_prev, x_next, n_tokens, codes, meta, xhat_next, pred_out=None,
                         workspace=None, stream=None):
    _check(load().coral_predict_encode(ctypes.byref(cfg), ctypes.byref(pred) if pred is not None else None,
                                       _ptr(xhat_prev), _ptr(x_next), n_tokens, _ptr(codes), _ptr(meta),
                                       _ptr(xhat_next), _ptr(pred_out), _ptr(workspace), _nbytes(workspace),
                                       _stream(stream)))


def coral_predict_encode_static(cfg, pred, xhat_prev, x_next, n_tokens, codes, meta, xhat_next, pred_out=None,
                                stream=None):
    """coral_predict_encode without a workspace (built-in fixed scratch)."""
    _check(load().coral_predict_encode_static(ctypes.byref(cfg), ctypes.byref(pred) if pred is not None else None,
                                              _ptr(xhat_prev), _ptr(x_next), n_tokens, _ptr(codes), _ptr(meta),
                                              _ptr(xhat_next), _ptr(pred_out), _stream(stream)))


def coral_prepared_bytes(cfg, rank=32):
    b = ctypes.c_size_t()
    _check(load().coral_prepared_bytes(ctypes.byref(cfg), rank, ctypes.byref(b)))
    return b.value


def coral_prepare_predictor(cfg, pred, prepared, stream=None):
    """Lays pred's U and W out once into `prepared` (a device buffer of
    coral_prepared_bytes); set pred.prepared to it afterwards."""
    _check(load().coral_prepare_predictor(ctypes.byref(cfg), ctypes.byref(pred), _ptr(prepared), _nbytes(prepared),
                                          _stream(stream)))


def coral_fit_block(cfg, pred, xhat_prev, x_next, n_tokens, B_out, workspace, stream=None):
    """Adapted block predictors: per head the ridge least-squares B_h (bf16
    [H][D][D]) for this layer pair; pred supplies U and W."""
    _check(load().coral_fit_block(ctypes.byref(cfg), ctypes.byref(pred) if pred is not None else None,
                                  _ptr(xhat_prev), _ptr(x_next), n_tokens, _ptr(B_out), _ptr(workspace),
                                  _nbytes(workspace), _stream(stream)))


def coral_predict_decode(cfg, pred, xhat_prev, n_tokens, codes, meta, xhat_next, pred_out=None, workspace=None,
                         stream=None):
    _check(load().coral_predict_decode(ctypes.byref(cfg), ctypes.byref(pred) if pred is not None else None,
                                       _ptr(xhat_prev), n_tokens, _ptr(codes), _ptr(meta), _ptr(xhat_next),
                                       _ptr(pred_out), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def coral_sas_workspace_bytes(cfg, n_tokens):
    b = ctypes.c_size_t(0)
    _check(load().coral_sas_workspace_bytes(ctypes.byref(cfg), n_tokens, ctypes.byref(b)))
    return b.value


def coral_sas_encode(cfg, pred, xhat_prev, x_next, n_tokens, codes, meta, ids, centroids, xhat_next, workspace,
                     pred_out=None, stream=None):
    """Coral-KV + SAS hybrid, one layer: k-means smoothing and PRQ of the
    bf16 prediction residual; xhat_next = bf16(pred + decoded residual)."""
    _check(load().coral_sas_encode(ctypes.byref(cfg), ctypes.byref(pred) if pred is not None else None,
                                   _ptr(xhat_prev), _ptr(x_next), n_tokens, _ptr(codes), _ptr(meta), _ptr(ids),
                                   _ptr(centroids), _ptr(xhat_next), _ptr(pred_out), _ptr(workspace),
                                   _nbytes(workspace), _stream(stream)))


def coral_sas_decode(cfg, pred, xhat_prev, n_tokens, codes, meta, ids, centroids, xhat_next, workspace,
                     pred_out=None, stream=None):
    _check(load().coral_sas_decode(ctypes.byref(cfg), ctypes.byref(pred) if pred is not None else None,
                                   _ptr(xhat_prev), n_tokens, _ptr(codes), _ptr(meta), _ptr(ids), _ptr(centroids),
                                   _ptr(xhat_next), _ptr(pred_out), _ptr(workspace), _nbytes(workspace),
                                   _stream(stream)))


def encoded_view(bufs):
    """qvg_encoded_view of a dict with "codes", "meta" and optionally "ids" and
    "centroids" device tensors (as alloc_encoded returns)."""
    return qvg_encoded_view(codes=_ptr(bufs["codes"]), meta=_ptr(bufs["meta"]), ids=_ptr(bufs.get("ids")),
                            centroids=_ptr(bufs.get("centroids")))


def qvg_attention_decode(cfg, q, n_queries, q_head_stride, q_token_stride, k, v, capacity, n_keys, scale, out,
                         out_head_stride, out_token_stride, stream=None):
    """k, v: qvg_encoded_view structs (see encoded_view)."""
    _check(load().qvg_attention_decode(ctypes.byref(cfg), _ptr(q), n_queries, q_head_stride, q_token_stride,
                                       ctypes.byref(k), ctypes.byref(v), capacity, n_keys, float(scale), _ptr(out),
                                       out_head_stride, out_token_stride, _stream(stream)))


def qvg_compress_host(cfg, x_host, x_dev, n_tokens, head_stride, token_stride, warm_start, centroids, ids, codes,
                      meta, out_dev, host_out, workspace, stream=None):
    """x_host, host_out: (pinned) host tensors; the rest device tensors (out_dev may be None)."""
    _check(load().qvg_compress_host(ctypes.byref(cfg), _ptr(x_host), _ptr(x_dev), n_tokens, head_stride, token_stride,
                                    _ptr(warm_start), _ptr(centroids), _ptr(ids), _ptr(codes), _ptr(meta),
                                    _ptr(out_dev), _ptr(host_out), _nbytes(host_out), _ptr(workspace),
                                    _nbytes(workspace), _stream(stream)))


def qvg_attention_workspace_bytes(cfg, n_keys):
    b = ctypes.c_size_t(0)
    _check(load().qvg_attention_workspace_bytes(ctypes.byref(cfg), n_keys, ctypes.byref(b)))
    return b.value


def qvg_attention_decode_staged(cfg, q, n_queries, q_head_stride, q_token_stride, k, v, capacity, n_keys, scale,
                                out, out_head_stride, out_token_stride, workspace, stream=None):
    """k, v: qvg_encoded_view structs; workspace: a device buffer of at least
    qvg_attention_workspace_bytes (or None when that is 0)."""
    _check(load().qvg_attention_decode_staged(ctypes.byref(cfg), _ptr(q), n_queries, q_head_stride, q_token_stride,
                                              ctypes.byref(k), ctypes.byref(v), capacity, n_keys, float(scale),
                                              _ptr(out), out_head_stride, out_token_stride, _ptr(workspace),
                                              _nbytes(workspace), _stream(stream)))


# -------------------------------------------------- allocation conveniences --

def alloc_encoded(cfg, capacity, n_versions=1, device="cuda"):
    """Device buffers for one encoded (layer, tensor), sized by qvg_encoded_bytes."""
    cb, mb, ib, xb = qvg_encoded_bytes(cfg, capacity, n_versions)
    return {
        "codes": torch.empty(cb // 4, dtype=torch.int32, device=device),
        "meta": torch.empty(mb // 4, dtype=torch.int32, device=device),
        "ids": torch.empty(max(ib, 1), dtype=torch.uint8, device=device),
        "centroids": torch.empty(max(xb // 2, 8), dtype=torch.int16, device=device),
    }


def alloc_workspace(cfg, n_tokens, device="cuda"):
    return torch.empty(qvg_workspace_bytes(cfg, n_tokens), dtype=torch.uint8, device=device)


def make_cache(cfg, capacity, max_versions, max_chunks, device="cuda"):
    """A streaming cache: device buffers (kept alive in the returned dict) and
    the qvg_cache struct pointing at them."""
    bufs = alloc_encoded(cfg, capacity, max_versions, device)
    bufs["chunk_offset"] = torch.zeros(max_chunks + 1, dtype=torch.int64, device=device)
    bufs["chunk_version"] = torch.zeros(max_chunks, dtype=torch.int32, device=device)
    c = qvg_cache(codes=_ptr(bufs["codes"]), meta=_ptr(bufs["meta"]), ids=_ptr(bufs["ids"]),
                  centroids=_ptr(bufs["centroids"]), chunk_offset=_ptr(bufs["chunk_offset"]),
                  chunk_version=_ptr(bufs["chunk_version"]), capacity=capacity, max_versions=max_versions,
                  max_chunks=max_chunks, n_used=0, n_versions=0, n_chunks=0)
    return c, bufs
