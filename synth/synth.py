"""Seeded, counter-based generator of synthetic bf16 KV caches (numpy side).

This module produces inputs only; it holds none of the codec's arithmetic.  A
CUDA twin (``synth_gpu.cu``) computes the same recipe byte for byte so that the
big configurations can be drawn straight into device memory; the two are
checked against each other on sampled rows.

Recipe (every step is exact integer arithmetic or a single IEEE fp64 operation
in a fixed order, so both sides agree bit for bit):

* ``mix64`` is the SplitMix64 output function (Steele, Lea & Flood, 2014):
  xor-shift 30, multiply 0xBF58476D1CE4E5B9, xor-shift 27, multiply
  0x94D049BB133111EB, xor-shift 31.  The i-th draw of a stream with key k is
  ``mix64(k + (i + 1) * 0x9E3779B97F4A7C15)`` (mod 2**64).
* Stream keys: ``k = mix64(seed + gamma)``, then for each field f of
  (layer, tensor, head, purpose): ``k = mix64((k ^ f) + gamma)``.
* Approximate N(0,1) from one draw h: the four 16-bit fields of h are summed
  (Irwin-Hall of 4 uniforms), ``z = (S - 131070) * (sqrt(3) / 65536)`` in fp64.
* Mixture per (layer, tensor, head): M centres ``mu0[m,d] = z``; per latent
  frame f >= 1 the centres drift, ``mu_f = mu_{f-1} + drift * z`` (fp64, frame
  by frame).  Token n picks centre ``draw % M``, sits in frame
  ``n // frame_tokens`` and gets ``x = mu_f[m,d] + noise * z`` (fp64 multiply,
  then add).  On K only, ``outlier_channels`` channels (the ones with the
  smallest draws of the outlier stream, ties by index) are multiplied by
  ``outlier_factor`` (fp64).  The value is rounded fp64 -> fp32 -> bf16, each
  round-to-nearest-even.
"""
import numpy as np

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MUL1 = 0xBF58476D1CE4E5B9
MUL2 = 0x94D049BB133111EB
NORM_SCALE = float.fromhex("0x1.bb67ae8584caap-16")   # sqrt(3) / 65536, rounded to fp64

P_CENTERS, P_ASSIGN, P_DRIFT, P_NOISE, P_OUTLIER = 1, 2, 3, 4, 5
P_CORAL_B, P_CORAL_U, P_CORAL_W, P_CORAL_NOISE = 6, 7, 8, 9

K_TENSOR, V_TENSOR = 0, 1
Q_TENSOR = 2        # queries of an attention consumer, drawn like K and V (no outliers)
P_ENC_CODES, P_ENC_META, P_ENC_IDS, P_ENC_CENT = 10, 11, 12, 13


def mix64_int(z):
    z &= M64
    z = ((z ^ (z >> 30)) * MUL1) & M64
    z = ((z ^ (z >> 27)) * MUL2) & M64
    return z ^ (z >> 31)


def stream_key(seed, *fields):
    k = mix64_int(seed + GAMMA)
    for f in fields:
        k = mix64_int(((k ^ (int(f) & M64)) + GAMMA) & M64)
    return k


def _mix64_np(z):
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= np.uint64(MUL1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(MUL2)
    z ^= z >> np.uint64(31)
    return z


def draws(key, idx):
    """Draws ``idx`` (uint64 array of counters) of the stream ``key``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (idx + np.uint64(1)) * np.uint64(GAMMA)
    return _mix64_np(z)


def normals(key, idx):
    h = draws(key, idx)
    m16 = np.uint64(0xFFFF)
    s = ((h & m16) + ((h >> np.uint64(16)) & m16) + ((h >> np.uint64(32)) & m16)
         + (h >> np.uint64(48))).astype(np.int64)
    return (s - 131070).astype(np.float64) * NORM_SCALE


def f64_to_bf16_bits(x):
    """fp64 -> fp32 (RN-even) -> bf16 (RN-even), as uint16 bit patterns."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(wl, layer, head):
    if wl.outlier_channels == 0:
        return np.zeros(0, dtype=np.int64)
    key = stream_key(wl.seed, layer, K_TENSOR, head, P_OUTLIER)
    d = np.arange(wl.head_dim, dtype=np.uint64)
    h = draws(key, d)
    order = np.lexsort((np.arange(wl.head_dim), h))
    return np.sort(order[: wl.outlier_channels]).astype(np.int64)


def outlier_mask(wl, layer, head):
    """Per-channel multiplier bitmask as 4 uint64 words (channels < 256)."""
    words = [0, 0, 0, 0]
    for c in outlier_channels(wl, layer, head):
        words[c // 64] |= 1 << (c % 64)
    return words


def center_table(wl, layer, tensor, head, n_frames):
    """Centres of every frame, fp64 [n_frames][M][D]."""
    M, D = wl.centers, wl.head_dim
    kc = stream_key(wl.seed, layer, tensor, head, P_CENTERS)
    kd = stream_key(wl.seed, layer, tensor, head, P_DRIFT)
    idx = np.arange(M * D, dtype=np.uint64)
    tab = np.empty((n_frames, M, D), dtype=np.float64)
    tab[0] = normals(kc, idx).reshape(M, D)
    for f in range(1, n_frames):
        z = normals(kd, np.uint64(f * M * D) + idx).reshape(M, D)
        tab[f] = tab[f - 1] + wl.drift_std * z
    return tab


def mixture_unit(wl, layer, tensor, head, tok_begin=0, tok_end=None, tokens=None):
    """bf16 bits [n][D] of one (layer, tensor, head) unit for tokens
    [tok_begin, tok_end) (or for the explicit token indices ``tokens``)."""
    D, M = wl.head_dim, wl.centers
    if tokens is None:
        if tok_end is None:
            tok_end = wl.tokens
        tokens = np.arange(tok_begin, tok_end, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    if tokens.size == 0:
        return np.zeros((0, D), dtype=np.uint16)
    n_frames = int(tokens.max()) // wl.frame_tokens + 1
    tab = center_table(wl, layer, tensor, head, n_frames)
    ka = stream_key(wl.seed, layer, tensor, head, P_ASSIGN)
    kn = stream_key(wl.seed, layer, tensor, head, P_NOISE)
    m = (draws(ka, tokens.astype(np.uint64)) % np.uint64(M)).astype(np.int64)
    f = tokens // wl.frame_tokens
    idx = (tokens.astype(np.uint64)[:, None] * np.uint64(D)
           + np.arange(D, dtype=np.uint64)[None, :])
    z = normals(kn, idx)
    x = tab[f, m, :] + wl.noise_std * z
    if tensor == K_TENSOR and wl.outlier_channels:
        ch = outlier_channels(wl, layer, head)
        x[:, ch] = x[:, ch] * wl.outlier_factor
    return f64_to_bf16_bits(x)


def mixture_layer(wl, layer, tensor, tok_begin=0, tok_end=None, layout="hnd"):
    """bf16 bits of all heads of one (layer, tensor): ``hnd`` -> [H][n][D],
    ``nhd`` -> [n][H][D]."""
    units = [mixture_unit(wl, layer, tensor, h, tok_begin, tok_end) for h in range(wl.heads)]
    a = np.stack(units, axis=0)
    if layout == "nhd":
        a = np.ascontiguousarray(a.transpose(1, 0, 2))
    return a


# ---------------------------------------------------------------------------
# Cross-layer workload: layer l+1 = A_l . layer l + noise, A_l block-diagonal
# per head plus a global low-rank term.  Inputs only; the codec never sees A_l
# except as the given predictor.
# ---------------------------------------------------------------------------

def coral_predictor(wl, layer):
    """bf16 bits of (B [H][D][D] out x in, U [H*D][R], W [H*D][R]) for the map
    layer -> layer + 1.  B entries have variance 1/D, U and W 1/(H*D)."""
    H, D, R = wl.heads, wl.head_dim, wl.rank
    HD = H * D
    kb = stream_key(wl.seed, layer, 0, 0, P_CORAL_B)
    ku = stream_key(wl.seed, layer, 0, 0, P_CORAL_U)
    kw = stream_key(wl.seed, layer, 0, 0, P_CORAL_W)
    sb = float(np.sqrt(1.0 / D))
    sl = float(np.sqrt(1.0 / HD))
    B = f64_to_bf16_bits(normals(kb, np.arange(H * D * D, dtype=np.uint64)) * sb).reshape(H, D, D)
    U = f64_to_bf16_bits(normals(ku, np.arange(HD * R, dtype=np.uint64)) * sl).reshape(HD, R)
    W = f64_to_bf16_bits(normals(kw, np.arange(HD * R, dtype=np.uint64)) * sl).reshape(HD, R)
    return B, U, W


def coral_layers(wl, tensor, tok_begin=0, tok_end=None, n_layers=None):
    """bf16 bits [L][n][H*D] (token-major) of one tensor across layers for
    tokens [tok_begin, tok_end).  Layer 0 is the mixture (no drift, no
    outliers); layer l+1 = bf16(A_l x_l + next_noise_std * z) with A_l x_l
    evaluated in fp64 (block part plus U (W^T x))."""
    H, D = wl.heads, wl.head_dim
    HD = H * D
    if tok_end is None:
        tok_end = wl.tokens
    L = wl.layers if n_layers is None else n_layers
    tokens = np.arange(tok_begin, tok_end, dtype=np.int64)
    n = tokens.size
    out = np.empty((L, n, HD), dtype=np.uint16)
    x0 = np.stack([mixture_unit(wl, 0, tensor, h, tokens=tokens) for h in range(H)], axis=1)
    out[0] = x0.reshape(n, HD)
    for l in range(L - 1):
        B, U, W = coral_predictor(wl, l)
        x = bf16_bits_to_f32(out[l]).astype(np.float64).reshape(n, H, D)
        Bf = bf16_bits_to_f32(B).astype(np.float64)
        blk = np.einsum("hoi,nhi->nho", Bf, x).reshape(n, HD)
        Uf = bf16_bits_to_f32(U).astype(np.float64)
        Wf = bf16_bits_to_f32(W).astype(np.float64)
        low = (x.reshape(n, HD) @ Wf) @ Uf.T
        kz = stream_key(wl.seed, l + 1, tensor, 0, P_CORAL_NOISE)
        idx = tokens.astype(np.uint64)[:, None] * np.uint64(HD) + np.arange(HD, dtype=np.uint64)[None, :]
        z = normals(kz, idx)
        out[l + 1] = f64_to_bf16_bits(blk + low + wl.next_noise_std * z)
    return out


# ---------------------------------------------------------------------------
# Arbitrary encoded caches: every bit pattern of this form is a legal
# encoding, so these stand in for a compressed history without running any
# encoder.  Inputs only.
# ---------------------------------------------------------------------------

def random_encoding(seed, tensor, H, cap, D, S, G, C, bits=2):
    """Bit patterns of one encoded (layer, tensor) with ``cap`` rows per head:
    codes uint32 [S][H][cap][D*bits/32], uniform words; meta uint32
    [S][H][cap][D/G], low half an fp16 scale in [2^-6, 2^-5) (exponent field
    9, uniform mantissa), high half an fp16 zero-point of magnitude in
    [2^-4, 2^-3) (exponent field 11) with a uniform sign; ids uint8 [H][cap]
    uniform in [0, C); centroids bf16 [H][C][D] from the approximate normals.
    ids and centroids are None when C == 0."""
    W = D * bits // 32
    kc = stream_key(seed, tensor, P_ENC_CODES)
    codes = (draws(kc, np.arange(S * H * cap * W, dtype=np.uint64)) & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    km = stream_key(seed, tensor, P_ENC_META)
    d = draws(km, np.arange(S * H * cap * (D // G), dtype=np.uint64))
    scale = np.uint64(0x2400) | (d & np.uint64(0x3FF))
    zero = (((d >> np.uint64(10)) & np.uint64(1)) << np.uint64(15)) | np.uint64(0x2C00) | ((d >> np.uint64(11)) & np.uint64(0x3FF))
    meta = (scale | (zero << np.uint64(16))).astype(np.uint32)
    codes = codes.reshape(S, H, cap, W)
    meta = meta.reshape(S, H, cap, D // G)
    if C == 0:
        return codes, meta, None, None
    ki = stream_key(seed, tensor, P_ENC_IDS)
    ids = (draws(ki, np.arange(H * cap, dtype=np.uint64)) % np.uint64(C)).astype(np.uint8).reshape(H, cap)
    kx = stream_key(seed, tensor, P_ENC_CENT)
    cent = f64_to_bf16_bits(normals(kx, np.arange(H * C * D, dtype=np.uint64))).reshape(H, C, D)
    return codes, meta, ids, cent
