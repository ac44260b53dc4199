"""ctypes front end of the CPU oracle (``qvg_oracle.cpp``) -- test
infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  Arrays are numpy; bf16 tensors travel as
their uint16 bit patterns.  Layouts are per head unit (``[N][D]`` rows); the
tests reshape the CUDA library's ``[S][H][N][...]`` buffers to compare.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qvg_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force=False):
    """Compile the oracle with g++ (-O2, no FMA contraction, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", _LIB + ".tmp", _SRC]
    subprocess.check_call(cmd)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.or_to_bf16.argtypes = [ctypes.c_double]
        L.or_to_bf16.restype = ctypes.c_uint16
        L.or_to_f16.argtypes = [ctypes.c_float]
        L.or_to_f16.restype = ctypes.c_uint16
        L.or_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.or_f16_to_f32.restype = ctypes.c_float
        L.or_kmeans_init.argtypes = [P, I64, I32, I32, P]
        L.or_assign.argtypes = [P, I64, I32, P, I32, P, P]
        L.or_update.argtypes = [P, I64, I32, P, I32, P, P]
        L.or_fit.argtypes = [P, I64, I32, I32, I32, P, P, P]
        L.or_prq_encode.argtypes = [P, I64, I32, P, P, I32, I32, I32, P, P]
        L.or_decode.argtypes = [P, P, P, P, I64, I32, I32, I32, I32, P]
        L.or_stream.argtypes = [P, I64, I32, I32, I32, I32, I32, I32, I32, I32, P, P, P, P, P]
        L.or_stream.restype = I32
        L.or_coral_predict.argtypes = [P, I64, I32, I32, P, P, P, I32, P]
        L.or_coral_encode_layer.argtypes = [P, P, I64, I32, I32, P, P, P, I32, P, I32, I32, P, P, P, P]
        L.or_coral_decode_layer.argtypes = [P, I64, I32, I32, P, P, P, I32, P, I32, I32, P, P, P]
        L.or_bits_per_element.argtypes = [I32, I32, I32, I32, I32, I64, I32]
        L.or_coral_fit_block.argtypes = [P, P, I64, I32, I32, P, P, I32, P, P]
        L.or_bits_per_element.restype = ctypes.c_double
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- formats --

def to_bf16(v):
    return lib().or_to_bf16(float(v))


def to_f16(v):
    return lib().or_to_f16(float(np.float32(v)))


def f16_to_f32(h):
    return lib().or_f16_to_f32(int(h))


# ------------------------------------------------------------------ k-means --

def kmeans_init(x, C):
    x = _c(x, np.uint16)
    N, D = x.shape
    cent = np.empty((C, D), np.uint16)
    lib().or_kmeans_init(_p(x), N, D, C, _p(cent))
    return cent


def assign(x, cent, return_dist=False):
    x = _c(x, np.uint16)
    cent = _c(cent, np.uint16)
    N, D = x.shape
    ids = np.empty(N, np.int32)
    dmin = np.empty(N, np.float64)
    lib().or_assign(_p(x), N, D, _p(cent), cent.shape[0], _p(ids), _p(dmin))
    return (ids, dmin) if return_dist else ids


def update(x, ids, cent):
    x = _c(x, np.uint16)
    ids = _c(ids, np.int32)
    out = _c(cent, np.uint16).copy()
    N, D = x.shape
    counts = np.empty(out.shape[0], np.int64)
    lib().or_update(_p(x), N, D, _p(ids), out.shape[0], _p(out), _p(counts))
    return out, counts


def fit(x, C, T, warm=None):
    x = _c(x, np.uint16)
    N, D = x.shape
    cent = np.empty((C, D), np.uint16)
    ids = np.empty(N, np.int32)
    w = None if warm is None else _c(warm, np.uint16)
    lib().or_fit(_p(x), N, D, C, T, _p(w), _p(cent), _p(ids))
    return cent, ids


# --------------------------------------------------------------------- PRQ --

def prq_encode(x, cent, ids, S, G, b=2):
    """codes [S][N][D*b/32] uint32 (element e at bits b*e of its row, least
    significant first), meta [S][N][D/G] uint32 (lo = fp16 scale, hi = fp16
    zero).  b = 2 (QVG) or 4 (the PRQ_INT4 variant)."""
    x = _c(x, np.uint16)
    N, D = x.shape
    codes = np.empty((S, N, D * b // 32), np.uint32)
    meta = np.empty((S, N, D // G), np.uint32)
    c = None if cent is None else _c(cent, np.uint16)
    i = None if ids is None else _c(ids, np.int32)
    lib().or_prq_encode(_p(x), N, D, _p(c), _p(i), S, G, b, _p(codes), _p(meta))
    return codes, meta


def decode(codes, meta, ids, cent, G, b=2):
    codes = _c(codes, np.uint32)
    meta = _c(meta, np.uint32)
    S, N, W = codes.shape
    D = W * 32 // b
    out = np.empty((N, D), np.uint16)
    c = None if cent is None else _c(cent, np.uint16)
    i = None if ids is None else _c(ids, np.int32)
    lib().or_decode(_p(codes), _p(meta), _p(i), _p(c), N, D, S, G, b, _p(out))
    return out


def stream(x, chunk, steps, refit_every, C, T, S, G, b=2):
    x = _c(x, np.uint16)
    D = x.shape[1]
    Ntot = chunk * steps
    versions = np.zeros((steps, C, D), np.uint16)
    cver = np.empty(steps, np.int32)
    ids = np.empty(Ntot, np.int32)
    codes = np.empty((S, Ntot, D * b // 32), np.uint32)
    meta = np.empty((S, Ntot, D // G), np.uint32)
    nv = lib().or_stream(_p(x), chunk, steps, refit_every, D, C, T, S, G, b, _p(versions),
                         _p(cver), _p(ids), _p(codes), _p(meta))
    return versions[:nv], cver, ids, codes, meta


# ------------------------------------------------------------------- Coral --

def coral_predict(xh, B, U, W, H, D):
    xh = _c(xh, np.uint16)
    N = xh.shape[0]
    R = U.shape[1]
    pred = np.empty((N, H * D), np.float64)
    lib().or_coral_predict(_p(xh), N, H, D, _p(_c(B, np.uint16)), _p(_c(U, np.uint16)),
                           _p(_c(W, np.uint16)), R, _p(pred))
    return pred


def coral_encode_layer(xh_prev, x_next, B, U, W, H, D, S, G, pred_in=None):
    x_next = _c(x_next, np.uint16)
    N = x_next.shape[0]
    R = 0 if U is None else U.shape[1]
    codes = np.empty((S, H, N, D // 16), np.uint32)
    meta = np.empty((S, H, N, D // G), np.uint32)
    xh_next = np.empty((N, H * D), np.uint16)
    pred_out = np.empty((N, H * D), np.float32)
    xp = None if xh_prev is None else _c(xh_prev, np.uint16)
    pi = None if pred_in is None else _c(pred_in, np.float32)
    cv = (lambda a: None if a is None else _c(a, np.uint16))
    lib().or_coral_encode_layer(_p(xp), _p(x_next), N, H, D, _p(cv(B)), _p(cv(U)), _p(cv(W)), R,
                                _p(pi), S, G, _p(codes), _p(meta), _p(xh_next), _p(pred_out))
    return codes, meta, xh_next, pred_out


def coral_decode_layer(xh_prev, codes, meta, B, U, W, H, D, G, pred_in=None):
    codes = _c(codes, np.uint32)
    meta = _c(meta, np.uint32)
    S, _, N, _ = codes.shape
    R = 0 if U is None else U.shape[1]
    xh_next = np.empty((N, H * D), np.uint16)
    xp = None if xh_prev is None else _c(xh_prev, np.uint16)
    pi = None if pred_in is None else _c(pred_in, np.float32)
    cv = (lambda a: None if a is None else _c(a, np.uint16))
    lib().or_coral_decode_layer(_p(xp), N, H, D, _p(cv(B)), _p(cv(U)), _p(cv(W)), R, _p(pi), S, G,
                                _p(codes), _p(meta), _p(xh_next))
    return xh_next


def coral_fit_block(xh, y, U, W, H, D):
    """Adapted block predictors (Coral-KV adapted configuration): per head
    the ridge-regularised least-squares B_h for y - U_h t = B_h x_hat.
    Returns (B bf16 bits [H][D][D], Z = B^T before rounding, fp64 [H][D][D]
    laid out as B[h][o][i])."""
    xh = _c(xh, np.uint16)
    y = _c(y, np.uint16)
    N = xh.shape[0]
    R = 0 if U is None else U.shape[1]
    B = np.empty((H, D, D), np.uint16)
    Z = np.empty((H, D, D), np.float64)
    cv = (lambda a: None if a is None else _c(a, np.uint16))
    lib().or_coral_fit_block(_p(xh), _p(y), N, H, D, _p(cv(U)), _p(cv(W)), R, _p(B), _p(Z))
    return B, Z


def bits_per_element(S, b, G, C, D, N, V=1):
    return lib().or_bits_per_element(S, b, G, C, D, N, V)


# ------------------------------------------------------ Coral + SAS hybrid --

def f32_to_bf16_bits(a):
    """bf16 bit patterns of finite float32 values, round to nearest even:
    add 0x7FFF plus the lowest kept bit, then drop the low 16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def coral_sas_layer(xh_prev, x_next, B, U, W, H, D, C, T, S, G, pred_in=None):
    """Coral-KV prediction with the k-means smoothing of its residual, one
    layer.  The pages do not describe the combination; this is the plain
    reading the library implements:
      pred  = the block-DPLR prediction of layer l+1 from x_hat_l: fp32, taken
              from pred_in when given (the GPU's own, for staged checks), else
              the fp64 prediction rounded to fp32; zero without x_hat_l;
      r     = bf16(fp32(x_next - pred));
      per head: centroids, ids = fit(r_h, C, T); codes, meta = prq_encode of
              r_h - c[id]; r_hat_h = decode of them;
      x_hat = bf16(fp32(pred + r_hat)).
    Returns (centroids [H][C][D], ids [H][N], codes [S][H][N][D/16],
    meta [S][H][N][D/G], x_hat [N][H*D], pred fp32 [N][H*D])."""
    x_next = _c(x_next, np.uint16)
    N = x_next.shape[0]
    if pred_in is not None:
        pred = _c(pred_in, np.float32)
    elif xh_prev is None:
        pred = np.zeros((N, H * D), np.float32)
    else:
        pred = coral_predict(xh_prev, B, U, W, H, D).astype(np.float32)
    r = f32_to_bf16_bits(bf16_bits_to_f32(x_next) - pred)
    cent = np.empty((H, C, D), np.uint16)
    ids = np.empty((H, N), np.int32)
    codes = np.empty((S, H, N, D // 16), np.uint32)
    meta = np.empty((S, H, N, D // G), np.uint32)
    rhat = np.empty((N, H * D), np.uint16)
    for h in range(H):
        rh = np.ascontiguousarray(r[:, h * D:(h + 1) * D])
        cent[h], ids[h] = fit(rh, C, T)
        codes[:, h], meta[:, h] = prq_encode(rh, cent[h], ids[h], S, G)
        rhat[:, h * D:(h + 1) * D] = decode(codes[:, h], meta[:, h], ids[h], cent[h], G)
    x_hat = f32_to_bf16_bits(pred + bf16_bits_to_f32(rhat))
    return cent, ids, codes, meta, x_hat, pred


# ------------------------------------------- attention over the decoded cache --

def attention(q, k_hat, v_hat, scale):
    """Softmax attention of one head over decoded K/V rows, in fp64: the plain
    definition of what a consumer of the cache computes (Quant VideoGen
    explainer, sec. 3: dequantisation fused into the kernels that use the
    cache; the 33-method Self-Forcing KV-cache study, abstract: attention over
    the rebuilt BF16 keys and values).  Non-causal: every query sees every key.
      s[i, n] = scale * <q_i, k_n>,
      o_i     = sum_n exp(s[i, n]) v_n / sum_n exp(s[i, n]).
    Subtracting each row's largest score before the exponential leaves o
    unchanged and keeps exp from overflowing.
    q [Nq][D], k_hat and v_hat [N][D] as bf16 bits (uint16), N >= 1; scale is
    used as given (a float32 value converts exactly).  Returns fp64 [Nq][D]."""
    Qf = bf16_bits_to_f32(q).astype(np.float64)
    Kf = bf16_bits_to_f32(k_hat).astype(np.float64)
    Vf = bf16_bits_to_f32(v_hat).astype(np.float64)
    s = float(scale) * (Qf @ Kf.T)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    return (p @ Vf) / p.sum(axis=1, keepdims=True)
