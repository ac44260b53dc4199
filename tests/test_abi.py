"""The C-ABI library loads, exports every symbol include/qvg.h declares, and
rejects bad arguments on the host before launching anything (no GPU needed:
every call here fails validation or is a host-only size query)."""
import ctypes
import os
import re
from fractions import Fraction

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def Q():
    import kv_cache_quantization_means_b300 as Q
    from kv_cache_quantization_means_b300 import build as B
    B.build()
    Q.load()
    return Q


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "qvg.h")).read()
    return sorted(set(re.findall(r"QVG_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ["qvg_fit_centroids", "qvg_encode", "qvg_append_chunk", "qvg_decode", "coral_predict_encode"]:
        assert name in syms


def test_library_exports_every_declared_symbol(Q):
    lib = ctypes.CDLL(Q.qvg.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert sorted(Q.EXPORTS) == declared_symbols()


def test_version(Q):
    assert "sm_103a" in Q.qvg_version()


def cfg(Q, H=2, D=64, C=16, T=3, S=2, G=64, bits=2):
    return Q.config(H, D, C, T, S, G, bits)


@pytest.mark.parametrize("kw,status", [
    (dict(bits=3), 2), (dict(bits=8), 2), (dict(D=48), 2), (dict(G=48), 2), (dict(D=64, G=128), 1), (dict(S=0), 2),
    (dict(S=5), 2), (dict(C=300), 2), (dict(C=-1), 2), (dict(D=256, C=16), 2), (dict(H=0), 1),
])
def test_bad_configs_rejected(Q, kw, status):
    with pytest.raises(Q.QvgError) as e:
        Q.qvg_encoded_bytes(cfg(Q, **kw), 100)
    assert e.value.status == status


def test_encoded_bytes_closed_form(Q):
    """Buffer sizes from the ABI equal the closed form S*b + 32*S/G + 8/D +
    16*C*V/N bits per element."""
    for (H, D, C, S, G, N, V, b) in [(2, 64, 16, 2, 64, 1560, 1, 2), (12, 128, 256, 2, 64, 32760, 1, 2),
                                     (12, 128, 256, 2, 64, 187200, 5, 2), (40, 128, 256, 3, 128, 81920, 1, 2),
                                     (16, 128, 0, 2, 64, 16384, 1, 2), (12, 128, 256, 1, 128, 32760, 1, 4),
                                     (2, 32, 0, 4, 16, 777, 1, 4)]:
        c = Q.config(H, D, C, 1, S, G, b)
        cb, mb, ib, xb = Q.qvg_encoded_bytes(c, N, V)
        bits = Fraction(8 * (cb + mb + ib + xb), H * N * D)
        want = Fraction(b * S) + Fraction(32 * S, G) + ((Fraction(8, D) + Fraction(16 * C * V, N)) if C else 0)
        assert bits == want


def test_cross_layer_codec_is_two_bit(Q):
    """4-bit codes are a QVG option; the cross-layer codec refuses them on
    the host, before any launch."""
    c = Q.config(2, 128, 0, 0, 2, 64, 4)
    with pytest.raises(Q.QvgError) as e:
        Q.coral_predict_encode(c, None, None, None, 0, None, None, None, stream=0)
    assert e.value.status == 2


def test_workspace_bytes_monotone(Q):
    c = cfg(Q)
    a, b = Q.qvg_workspace_bytes(c, 100), Q.qvg_workspace_bytes(c, 10000)
    assert 0 < a < b and a % 256 == 0


def _raw(Q):
    return Q.load()


def test_invalid_arguments_fail_before_launch(Q):
    L = _raw(Q)
    c = cfg(Q)
    b = ctypes.byref(c)
    # NULL input
    assert L.qvg_encode(b, None, 10, 640, 64, None, 0, None, None, None, 10, 0, None, 0, None) == 1
    # misaligned input pointer
    assert L.qvg_encode(b, 8, 10, 640, 64, 16, 0, 16, 16, 16, 10, 0, None, 0, None) == 1
    # strides not multiples of 8
    assert L.qvg_encode(b, 16, 10, 644, 64, 16, 0, 16, 16, 16, 10, 0, None, 0, None) == 1
    # rows beyond capacity
    assert L.qvg_encode(b, 16, 10, 640, 64, 16, 0, 16, 16, 16, 15, 6, None, 0, None) == 3
    # assign without workspace
    assert L.qvg_encode(b, 16, 10, 640, 64, 16, 1, 16, 16, 16, 10, 0, None, 0, None) == 1
    # workspace too small / unaligned
    assert L.qvg_fit_centroids(b, 16, 10, 640, 64, None, 16, 16, 10, 0, 256, 16, None) == 1
    assert L.qvg_fit_centroids(b, 16, 10, 640, 64, None, 16, 16, 10, 0, 264, 1 << 30, None) == 1
    # fit with no tokens / no clusters
    assert L.qvg_fit_centroids(b, 16, 0, 640, 64, None, 16, 16, 10, 0, 256, 1 << 30, None) == 1
    c0 = cfg(Q, C=0)
    assert L.qvg_fit_centroids(ctypes.byref(c0), 16, 10, 640, 64, None, 16, 16, 10, 0, 256, 1 << 30, None) == 1
    # decode range outside capacity
    assert L.qvg_decode(b, 16, 16, 16, 16, 10, 5, 11, 16, 640, 64, None) == 1
    assert L.qvg_decode(b, 16, 16, 16, 16, 10, 6, 5, 16, 640, 64, None) == 1
    # the message names the problem
    assert L.qvg_decode(b, 16, 16, 16, 16, 10, 5, 11, 16, 640, 64, None) == 1
    assert b"outside" in L.qvg_last_error()
    assert L.qvg_encode(b, 16, 10, 640, 64, 16, 0, 16, 16, 16, 15, 6, None, 0, None) == 3
    assert b"capacity" in L.qvg_last_error()


def test_empty_calls_are_no_ops(Q):
    L = _raw(Q)
    c = cfg(Q)
    b = ctypes.byref(c)
    # empty decode range and empty encode return OK without touching the GPU
    assert L.qvg_decode(b, 16, 16, 16, 16, 10, 4, 4, 16, 640, 64, None) == 0
    c0 = cfg(Q, C=0)
    assert L.qvg_encode(ctypes.byref(c0), None, 0, 0, 0, None, 0, 16, 16, None, 0, 0, None, 0, None) == 0


def test_append_chunk_capacity_checks(Q):
    L = _raw(Q)
    c = cfg(Q)
    cache = Q.qvg.qvg_cache(codes=16, meta=16, ids=16, centroids=16, chunk_offset=16, chunk_version=16,
                            capacity=100, max_versions=1, max_chunks=2, n_used=0, n_versions=0, n_chunks=0)
    cp = ctypes.byref(cache)
    # first chunk must refit
    assert L.qvg_append_chunk(ctypes.byref(c), cp, 16, 50, 6400, 64, 0, 256, 1 << 30, None) == 1
    # overflowing rows
    assert L.qvg_append_chunk(ctypes.byref(c), cp, 16, 150, 9600, 64, 1, 256, 1 << 30, None) == 3
    cache.n_versions, cache.n_chunks, cache.n_used = 1, 2, 60
    assert L.qvg_append_chunk(ctypes.byref(c), cp, 16, 10, 640, 64, 0, 256, 1 << 30, None) == 3   # chunks full
    cache.n_chunks = 1
    assert L.qvg_append_chunk(ctypes.byref(c), cp, 16, 10, 640, 64, 1, 256, 1 << 30, None) == 3   # versions full
    assert cache.n_used == 60 and cache.n_chunks == 1   # failed calls change nothing


def test_coral_argument_checks(Q):
    L = _raw(Q)
    c = Q.config(4, 128, 0, 0, 2, 64)
    pred = Q.qvg.coral_predictor(B=16, U=16, W=16, rank=24)
    args = (ctypes.byref(c), ctypes.byref(pred), 16, 16, 10, 16, 16, 16, None, 256, 1 << 20, None)
    assert L.coral_predict_encode(*args) == 2          # rank not a multiple of 16
    pred.rank = 32
    assert L.coral_predict_encode(ctypes.byref(c), ctypes.byref(pred), 16, 16, 10, 16, 16, 16, None, 256, 8,
                                  None) == 1         # workspace too small
    cq = Q.config(4, 128, 16, 1, 2, 64)
    assert L.coral_predict_encode(ctypes.byref(cq), *args[1:]) == 1   # clusters must be 0


def test_coral_prepared_layout_checks(Q):
    """The prepared predictor layout: its size, and the argument checks of
    coral_prepare_predictor and of a predictor that carries one (all refused
    on the host, nothing launched)."""
    L = _raw(Q)
    c = Q.config(4, 128, 0, 0, 2, 64)
    sz = ctypes.c_size_t(0)
    assert L.coral_prepared_bytes(ctypes.byref(c), 32, ctypes.byref(sz)) == 0
    HD = 4 * 128
    a256 = lambda v: (v + 255) // 256 * 256
    assert sz.value == a256(32 * HD * 2) + a256(HD * 64 * 2)              # Wt, then [U | U]
    assert L.coral_prepared_bytes(ctypes.byref(c), 16, ctypes.byref(sz)) == 2      # rank 32 only
    c64 = Q.config(4, 64, 0, 0, 2, 64)
    assert L.coral_prepared_bytes(ctypes.byref(c64), 32, ctypes.byref(sz)) == 2    # head_dim 128 only
    need = Q.coral_prepared_bytes(c)
    buf = 1 << 20                                                            # a 256-byte aligned address
    pred = Q.qvg.coral_predictor(B=16, U=16, W=16, rank=32)
    prep = lambda p, ptr=buf, n=need: L.coral_prepare_predictor(ctypes.byref(c), ctypes.byref(p), ptr, n, None)
    assert prep(pred, ptr=None) == 1                                         # no buffer
    assert prep(pred, ptr=buf + 16) == 1                                     # not 256-byte aligned
    assert prep(pred, n=need - 1) == 1                                       # too small
    assert prep(Q.qvg.coral_predictor(B=16, U=None, W=16, rank=32)) == 1     # U missing
    assert prep(Q.qvg.coral_predictor(B=16, U=16, W=16, rank=16)) == 2       # rank 32 only
    # a predictor carrying a layout it cannot use is refused by the codec calls
    bad = Q.qvg.coral_predictor(B=16, U=16, W=16, rank=32, prepared=buf + 16)
    ws = 1 << 24                                                             # workspace bytes claimed: enough
    assert L.coral_predict_encode(ctypes.byref(c), ctypes.byref(bad), 16, 16, 10, 16, 16, 16, None, 256, ws,
                                  None) == 1                                 # layout not 256-byte aligned
    bad16 = Q.qvg.coral_predictor(B=16, U=16, W=16, rank=16, prepared=buf)
    assert L.coral_predict_encode(ctypes.byref(c), ctypes.byref(bad16), 16, 16, 10, 16, 16, 16, None, 256, ws,
                                  None) == 2                                 # layout with rank 16


def test_coral_sas_argument_checks(Q):
    """The Coral + SAS hybrid validates its configuration, buffers and
    workspace on the host and launches nothing when they are wrong."""
    L = Q.load()
    sz = ctypes.c_size_t(0)
    c0 = Q.config(4, 128, 0, 4, 2, 64)              # no clusters: the hybrid needs some
    assert L.coral_sas_workspace_bytes(ctypes.byref(c0), 100, ctypes.byref(sz)) == 1
    c = Q.config(4, 128, 16, 3, 2, 64)
    assert L.coral_sas_workspace_bytes(ctypes.byref(c), 100, ctypes.byref(sz)) == 0
    need = sz.value
    assert need >= Q.qvg_workspace_bytes(c, 100) + 100 * 4 * 128 * (4 + 2)    # fit + prediction + residual
    assert Q.coral_sas_workspace_bytes(c, 10000) > need                      # grows with the tokens
    ws = 1 << 20                                                             # a 256-byte aligned address

    def enc(cfg, n=100, wbytes=None, x_next=16, codes=16, ids=16, ws_ptr=ws):
        return L.coral_sas_encode(ctypes.byref(cfg), None, None, x_next, n, codes, 16, ids, 16, 16, None, ws_ptr,
                                  need if wbytes is None else wbytes, None)

    assert enc(c0) == 1                                  # no clusters
    c4 = Q.config(4, 128, 16, 3, 2, 64, 4)
    assert enc(c4) == 2                                  # 2-bit codes only
    cT = Q.config(4, 128, 16, 0, 2, 64)
    assert enc(cT) == 1                                  # lloyd_iters must be >= 1
    assert enc(c, n=0) == 1                              # needs tokens
    assert enc(c, wbytes=need - 1) == 1                  # workspace too small
    assert enc(c, ws_ptr=ws + 16) == 1                   # workspace not 256-byte aligned
    assert enc(c, x_next=None) == 1                      # buffer missing
    assert enc(c, ids=None) == 1
    assert enc(c, codes=24) == 1                         # codes not 16-byte aligned
    assert L.coral_sas_decode(ctypes.byref(c), None, None, 100, None, 16, 16, 16, 16, None, ws, need, None) == 1
    assert "NULL" in L.qvg_last_error().decode() or "null" in L.qvg_last_error().decode().lower()
    # a predicted layer needs a predictor
    assert L.coral_sas_encode(ctypes.byref(c), None, 16, 16, 100, 16, 16, 16, 16, 16, None, ws, need, None) == 1


def test_attention_argument_checks(Q):
    """The fused attention call validates shapes, buffers, strides and the
    key range on the host; every case here fails validation (or is the empty
    no-op) and launches nothing."""
    L = Q.load()
    V = Q.qvg.qvg_encoded_view
    kv = V(codes=16, meta=16, ids=16, centroids=16)
    c = Q.config(2, 128, 16, 1, 2, 64)

    def call(cfg=c, q=16, nq=10, qhs=1280, qts=128, k=kv, v=kv, cap=100, nk=50, scale=0.088, out=16, ohs=1280,
             ots=128):
        kp = None if k is None else ctypes.byref(k)
        vp = None if v is None else ctypes.byref(v)
        return L.qvg_attention_decode(ctypes.byref(cfg), q, nq, qhs, qts, kp, vp, cap, nk, ctypes.c_float(scale),
                                      out, ohs, ots, None)

    assert call(cfg=Q.config(2, 256, 0, 1, 2, 64)) == 2            # head_dim 256 not supported
    assert call(cfg=Q.config(2, 32, 0, 1, 2, 16)) == 2             # nor 32
    assert call(nk=0) == 1                                         # needs a key
    assert call(nk=101) == 1                                       # beyond capacity
    assert b"n_keys" in L.qvg_last_error()
    assert call(nq=-1) == 1
    assert call(scale=float("inf")) == 1
    assert call(scale=float("nan")) == 1
    assert call(k=None) == 1
    assert call(v=V(codes=None, meta=16, ids=16, centroids=16)) == 1
    assert call(k=V(codes=16, meta=24, ids=16, centroids=16)) == 1  # meta not 16-byte aligned
    assert call(k=V(codes=16, meta=16, ids=None, centroids=16)) == 1  # C > 0 needs ids
    assert call(v=V(codes=16, meta=16, ids=16, centroids=None)) == 1
    assert call(q=None) == 1
    assert call(q=24) == 1                                         # q not 16-byte aligned
    assert call(qts=132) == 1                                      # q stride not a multiple of 8
    assert call(out=None) == 1
    assert call(out=8) == 1                                        # out not 16-byte aligned
    assert call(ots=130) == 1                                      # out stride not a multiple of 4
    assert call(cfg=Q.config(2, 128, 16, 1, 2, 48)) == 2           # group size outside 16, 32, 64, 128
    # no clusters: ids and centroids may be NULL; still fails on the key range
    c0 = Q.config(2, 128, 0, 0, 2, 64)
    assert call(cfg=c0, k=V(codes=16, meta=16, ids=None, centroids=None), nk=0) == 1
    # no queries: nothing to do, and nothing launched
    assert call(nq=0, q=None, out=None) == 0


def test_static_coral_encode_refuses_scratch_beyond_its_array(Q):
    """The allocation-free Coral encode checks on the host that its scratch
    fits the built-in 4 MiB array: 128 heads of 128 channels at 16,384 tokens
    need 128*N + 192*H*D bytes > 4 MiB for the tensor-core path, so the call
    returns QVG_ERR_CAPACITY before touching the GPU (the pointers are never
    dereferenced)."""
    c = Q.config(128, 128, 0, 0, 2, 64)
    fake = 1 << 20
    pred = Q.qvg.coral_predictor(B=fake, U=fake, W=fake, rank=32)
    with pytest.raises(Q.QvgError) as e:
        Q.coral_predict_encode_static(c, pred, fake, fake, 16384, fake, fake, fake, None, stream=0)
    assert e.value.status == 3
