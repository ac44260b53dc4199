"""Device-side generation of the synthetic caches (CUDA twin of synth.py).

``mixture_layer_gpu`` writes exactly the bytes ``synth.mixture_layer`` would,
straight into a device tensor, so the full-size workloads need no host
round trip.  Cross-layer (Coral) inputs beyond layer 0 are built on the device
with torch matmuls (``coral_chain_gpu``); those follow the same recipe but are
not bit-identical to the numpy chain, and no test compares them with it.
"""
import ctypes
import os
import subprocess

import numpy as np
import torch

from . import synth as SY

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gpu.cu")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force=False):
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                           "-Xcompiler", "-fPIC", "-shared", "-o", _LIB + ".tmp", _SRC])
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            raise ImportError(f"{_LIB} missing: run synth.gpu.build()")
        L = ctypes.CDLL(_LIB)
        L.synth_mixture.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                    ctypes.c_double, ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
        L.synth_mixture.restype = ctypes.c_int
        _lib = L
    return _lib


def unit_keys(wl, layer, tensor):
    """[H][8] uint64: centres, assign, drift, noise keys and the outlier mask."""
    k = np.zeros((wl.heads, 8), dtype=np.uint64)
    for h in range(wl.heads):
        k[h, 0] = SY.stream_key(wl.seed, layer, tensor, h, SY.P_CENTERS)
        k[h, 1] = SY.stream_key(wl.seed, layer, tensor, h, SY.P_ASSIGN)
        k[h, 2] = SY.stream_key(wl.seed, layer, tensor, h, SY.P_DRIFT)
        k[h, 3] = SY.stream_key(wl.seed, layer, tensor, h, SY.P_NOISE)
        if tensor == SY.K_TENSOR and wl.outlier_channels:
            k[h, 4:8] = SY.outlier_mask(wl, layer, h)
    return k


def mixture_layer_gpu(wl, layer, tensor, out=None, tok_begin=0, tok_end=None, layout="hnd", stream=None,
                      with_outliers=True):
    """bf16 bits (as an int16 tensor) of all heads of one (layer, tensor) for
    tokens [tok_begin, tok_end), layout ``hnd`` ([H][n][D]) or ``nhd``."""
    if tok_end is None:
        tok_end = wl.tokens
    n = tok_end - tok_begin
    H, D, M = wl.heads, wl.head_dim, wl.centers
    shape = (H, n, D) if layout == "hnd" else (n, H, D)
    if out is None:
        out = torch.empty(shape, dtype=torch.int16, device="cuda")
    hs, ts = (n * D, D) if layout == "hnd" else (D, H * D)
    F = max(1, (tok_end - 1) // wl.frame_tokens + 1)
    keys = unit_keys(wl, layer, tensor)
    if not with_outliers:
        keys[:, 4:8] = 0
    kt = torch.from_numpy(keys.view(np.int64)).to("cuda")
    tab = torch.empty(H * F * M * D, dtype=torch.float64, device="cuda")
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    st = lib().synth_mixture(kt.data_ptr(), H, M, D, F, wl.frame_tokens, tok_begin, n, wl.noise_std,
                             wl.drift_std, wl.outlier_factor, tab.data_ptr(), out.data_ptr(), hs, ts, s)
    if st != 0:
        raise RuntimeError(f"synth_mixture failed: cuda error {st}")
    torch.cuda.current_stream().synchronize()
    return out


def coral_chain_gpu(wl, tensor, n_layers=None):
    """Token-major bf16 bits [L][N][H*D] of one tensor for the cross-layer
    workload, built on the device: layer 0 from the mixture generator, then
    x_{l+1} = bf16(A_l x_l + next_noise_std * z) with A_l from
    ``synth.coral_predictor`` and z a seeded torch normal draw."""
    L = wl.layers if n_layers is None else n_layers
    H, D, N = wl.heads, wl.head_dim, wl.tokens
    out = torch.empty((L, N, H * D), dtype=torch.int16, device="cuda")
    mixture_layer_gpu(wl, 0, tensor, out=out[0].view(N, H, D), layout="nhd")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(wl.seed * 100 + tensor)
    for l in range(L - 1):
        B, U, W = coral_predictor_device(wl, l)
        x = out[l].view(torch.bfloat16).float().view(N, H, D)
        blk = torch.einsum("hoi,nhi->nho", B.view(torch.bfloat16).float(), x).reshape(N, H * D)
        low = (x.reshape(N, H * D) @ W.view(torch.bfloat16).float()) @ U.view(torch.bfloat16).float().T
        z = torch.randn((N, H * D), device="cuda", generator=gen)
        out[l + 1] = (blk + low + wl.next_noise_std * z).to(torch.bfloat16).view(torch.int16)
    return out


_pred_cache = {}


def coral_predictor_device(wl, layer):
    key = (wl.name, layer)
    if key not in _pred_cache:
        B, U, W = SY.coral_predictor(wl, layer)
        _pred_cache[key] = tuple(torch.from_numpy(a.view(np.int16)).to("cuda") for a in (B, U, W))
    return _pred_cache[key]
