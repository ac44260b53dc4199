"""GPU parity of attention over a compressed K/V history (qvg_attention_decode:
the decode fused into the consumer, no bf16 K/V buffer) against the oracle,
which decodes the same encodings to bf16 rows and evaluates softmax attention
in fp64 (oracle.attention).

Tolerance, per query row i and channel d, derived from the kernel's
arithmetic (its decoded K/V rows are the decoder's, bit for bit):
  w_n        the oracle's softmax weights of row i, Ew[.] = sum_n w_n (.)
  scores     bf16 products are exact in fp32; a D-term fp32 sum errs by at
             most D * 2^-24 * sum_d |q_d k_d| under round-to-nearest; allowing
             8x that for the tensor cores' accumulation order gives
             E_i = |scale| * D * 2^-21 * max_n sum_d |q_id k_nd|, plus
             2^-20 * max_n |s_in| for the fp32 scale multiply and exp2f.
             Weights move by a factor within exp(+-2 E_i), and since the
             weight changes sum to zero, o_d moves by at most
             (exp(2 E_i) - 1) * Ew|v_d - o_d|.
  bf16 P     probabilities are rounded to bf16 (relative 2^-9) before the
             product with V while the denominator sums them unrounded:
             at most 2^-9 * Ew|v_d|.
  sums       fp32 accumulation of P V and of the denominator: four MMA
             accumulations and one rescale per 64-key tile, plus exp2f's
             2 ulps: (5 * tiles + 16) * 2^-23 * Ew|v_d|, tiles = n_keys / 64
             rounded up.  The tensor-core path accumulates eight K = 16
             products and at most one rescale per 128-key tile (9 roundings
             per 128 keys, within the 10 allowed) and sums each tile's
             probabilities in four partial sums of 32 before adding them to
             the denominator ((34 + n_keys / 128) * 2^-24 relative, within
             the same allowance).
"""
import numpy as np
import pytest
import torch

from synth import synth as SY
from synth import workloads as WL
from gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


def tolerance(q, k, v, o_ref, scale, n_keys):
    """Per-element bound of |o_gpu - o_ref| (module docstring)."""
    Qf = SY.bf16_bits_to_f32(q).astype(np.float64)
    Kf = SY.bf16_bits_to_f32(k).astype(np.float64)
    Vf = SY.bf16_bits_to_f32(v).astype(np.float64)
    D = Qf.shape[1]
    s = scale * (Qf @ Kf.T)
    w = np.exp(s - s.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    A = (np.abs(Qf) @ np.abs(Kf).T).max(axis=1)
    E = abs(scale) * D * 2.0 ** -21 * A + 2.0 ** -20 * np.abs(s).max(axis=1)
    assert E.max() < 0.05, "tolerance derivation assumes small score errors"
    tiles = (n_keys + 63) // 64
    ew_abs = w @ np.abs(Vf)
    ew_dev = np.einsum("in,ind->id", w, np.abs(Vf[None, :, :] - o_ref[:, None, :]))
    return (2.0 ** -9 + (5 * tiles + 16) * 2.0 ** -23) * ew_abs + np.expm1(2 * E)[:, None] * ew_dev + 1e-30


def mixture(rng, N, D, M=8, noise=0.15):
    centres = rng.standard_normal((M, D))
    return SY.f64_to_bf16_bits(centres[rng.integers(0, M, N)] + noise * rng.standard_normal((N, D)))


def oracle_encoding(oracle, x, C, S, G, b):
    """Per head: fit (C > 0) and PRQ-encode x [H][N][D] on the CPU; returns
    codes [S][H][N][W], meta [S][H][N][D/G], ids [H][N], centroids [H][C][D]
    and the decoded rows [H][N][D]."""
    H, N, D = x.shape
    codes = np.empty((S, H, N, D * b // 32), np.uint32)
    meta = np.empty((S, H, N, D // G), np.uint32)
    ids = np.zeros((H, N), np.uint8) if C else None
    cent = np.zeros((H, C, D), np.uint16) if C else None
    dec = np.empty((H, N, D), np.uint16)
    for h in range(H):
        oc, oi = oracle.fit(x[h], C, 2) if C else (None, None)
        codes[:, h], meta[:, h] = oracle.prq_encode(x[h], oc, oi, S, G, b)
        dec[h] = oracle.decode(codes[:, h], meta[:, h], oi, oc, G, b)
        if C:
            ids[h], cent[h] = oi, oc
    return codes, meta, ids, cent, dec


def pad_rows(a, cap, rng, axis):
    """Extends the token axis of an encoded buffer to `cap` rows filled with
    random words (rows past n_keys must never be read)."""
    shape = list(a.shape)
    extra = cap - shape[axis]
    if extra == 0:
        return a
    shape[axis] = extra
    junk = rng.integers(0, 256 if a.dtype == np.uint8 else 2 ** 32, size=shape, dtype=np.uint64).astype(a.dtype)
    return np.concatenate([a, junk], axis=axis)


def device_views(Q, codes, meta, ids, cent):
    bufs = {"codes": to_dev(codes.reshape(-1)), "meta": to_dev(meta.reshape(-1))}
    if ids is not None:
        bufs["ids"] = to_dev(ids.reshape(-1))
        bufs["centroids"] = to_dev(cent.reshape(-1))
    return bufs, Q.encoded_view(bufs)


def attend(Q, cfg, q, Nq, qhs, qts, kb, vb, cap, n_keys, scale, out, ohs, ots, staged):
    """qvg_attention_decode, or qvg_attention_decode_staged with a working
    buffer of the size the library asks for."""
    if not staged:
        Q.qvg_attention_decode(cfg, q, Nq, qhs, qts, kb[1], vb[1], cap, n_keys, scale, out, ohs, ots)
        return
    nb = Q.qvg_attention_workspace_bytes(cfg, n_keys)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda") if nb else None
    Q.qvg_attention_decode_staged(cfg, q, Nq, qhs, qts, kb[1], vb[1], cap, n_keys, scale, out, ohs, ots, ws)


def run_attention(Q, cfg, q_nhd, kb, vb, cap, n_keys, scale, token_major=True, out_pad=0, staged=False):
    """q_nhd: bf16 bits [Nq][H][D].  Returns fp32 [H][Nq][D]."""
    Nq, H, D = q_nhd.shape
    if token_major:
        q = to_dev(np.ascontiguousarray(q_nhd).reshape(-1))
        qhs, qts = D, H * D
        ots = H * D + out_pad
        out = torch.full((Nq * ots + 4,), float("nan"), dtype=torch.float32, device="cuda")
        ohs = D
    else:
        q = to_dev(np.ascontiguousarray(q_nhd.transpose(1, 0, 2)).reshape(-1))
        qhs, qts = Nq * D, D
        ohs, ots = Nq * D + out_pad, D
        out = torch.full((H * ohs + 4,), float("nan"), dtype=torch.float32, device="cuda")
    attend(Q, cfg, q, Nq, qhs, qts, kb, vb, cap, n_keys, scale, out, ohs, ots, staged)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    res = np.empty((H, Nq, D))
    for h in range(H):
        for i in range(Nq):
            res[h, i] = o[h * ohs + i * ots: h * ohs + i * ots + D]
    return res, o, (ohs, ots)


CASES = [  # D, bits, S, G, C, token-major
    (128, 2, 2, 64, 16, True),
    (128, 4, 2, 64, 16, False),
    (64, 2, 1, 32, 0, True),
    (64, 4, 3, 16, 8, False),
    (128, 2, 4, 128, 0, True),
    # 4-bit, one stage: the kernel's prefetching specialisation
    (128, 4, 1, 64, 16, True),
    (64, 4, 1, 16, 0, False),
    # with the rows above, every (bits, S) form of the tensor-core path's staging decode
    (128, 2, 1, 32, 8, False),
    (128, 2, 3, 16, 16, True),
    (128, 4, 3, 128, 0, False),
    (128, 4, 4, 64, 8, True),
]


@pytest.mark.parametrize("staged", [False, True])
@pytest.mark.parametrize("D,bits,S,G,C,token_major", CASES)
def test_attention_matches_oracle(qvg, oracle, D, bits, S, G, C, token_major, staged):
    """Two heads, 300 keys (four full 64-key tiles and a ragged one; two full
    128-key tiles and a ragged one) inside a 320-row encoding whose last 20
    rows hold random words, 100 queries (one full 64-query tile and a ragged
    one; one ragged 128-query tile).  staged: the tensor-core entry point
    (head_dim 64 takes its fallback to the fused kernel)."""
    rng = np.random.default_rng(1000 + D + 10 * bits + S + G + C)
    H, N, cap, Nq = 2, 300, 320, 100
    cfg = qvg.config(H, D, C, 2, S, G, bits)
    xk = np.stack([mixture(rng, N, D) for _ in range(H)])
    xv = np.stack([mixture(rng, N, D) for _ in range(H)])
    kc, km, ki, kx, kdec = oracle_encoding(oracle, xk, C, S, G, bits)
    vc, vm, vi, vx, vdec = oracle_encoding(oracle, xv, C, S, G, bits)
    kb = device_views(qvg, pad_rows(kc, cap, rng, 2), pad_rows(km, cap, rng, 2),
                      None if ki is None else pad_rows(ki, cap, rng, 1), kx)
    vb = device_views(qvg, pad_rows(vc, cap, rng, 2), pad_rows(vm, cap, rng, 2),
                      None if vi is None else pad_rows(vi, cap, rng, 1), vx)
    q = np.stack([mixture(rng, Nq, D) for _ in range(H)], axis=1)     # [Nq][H][D]
    scale = float(np.float32(D ** -0.5))
    got, raw, (ohs, ots) = run_attention(qvg, cfg, q, kb, vb, cap, N, scale, token_major, out_pad=4, staged=staged)
    for h in range(H):
        ref = oracle.attention(q[:, h], kdec[h], vdec[h], scale)
        tol = tolerance(q[:, h], kdec[h], vdec[h], ref, scale, N)
        err = np.abs(got[h] - ref)
        assert np.all(err <= tol), f"head {h}: max err {err.max():.3g}, worst err/tol {(err / tol).max():.3g}"
    # padding between output rows is never written
    written = np.zeros(raw.shape, bool)
    for h in range(H):
        for i in range(Nq):
            written[h * ohs + i * ots: h * ohs + i * ots + D] = True
    assert np.all(np.isnan(raw[~written]))


@pytest.mark.parametrize("staged", [False, True])
def test_attention_single_key_is_exact(qvg, oracle, staged):
    """With one key every weight is exactly 1 (exp2(0) = 1, bf16(1) = 1), so
    every output row is the decoded value row, bit for bit in fp32."""
    rng = np.random.default_rng(5)
    H, D, S, G, C, cap = 3, 128, 2, 64, 16, 64
    cfg = qvg.config(H, D, C, 2, S, G)
    xk = np.stack([mixture(rng, cap, D) for _ in range(H)])
    xv = np.stack([mixture(rng, cap, D) for _ in range(H)])
    kc, km, ki, kx, _ = oracle_encoding(oracle, xk, C, S, G, 2)
    vc, vm, vi, vx, vdec = oracle_encoding(oracle, xv, C, S, G, 2)
    kb, vb = device_views(qvg, kc, km, ki, kx), device_views(qvg, vc, vm, vi, vx)
    q = np.stack([mixture(rng, 70, D) for _ in range(H)], axis=1)
    got, _, _ = run_attention(qvg, cfg, q, kb, vb, cap, 1, 0.3, staged=staged)
    for h in range(H):
        np.testing.assert_array_equal(got[h], np.broadcast_to(SY.bf16_bits_to_f32(vdec[h, 0]), got[h].shape))


def test_attention_zero_queries_and_mean(qvg, oracle):
    """n_queries = 0 writes nothing; all-zero queries weigh every key equally,
    so the output is the mean of the decoded value rows (within the bound)."""
    rng = np.random.default_rng(6)
    H, D, S, G, C, N = 2, 64, 2, 32, 0, 130
    cfg = qvg.config(H, D, C, 0, S, G)
    xk = np.stack([mixture(rng, N, D) for _ in range(H)])
    xv = np.stack([mixture(rng, N, D) for _ in range(H)])
    kc, km, _, _, kdec = oracle_encoding(oracle, xk, C, S, G, 2)
    vc, vm, _, _, vdec = oracle_encoding(oracle, xv, C, S, G, 2)
    kb, vb = device_views(qvg, kc, km, None, None), device_views(qvg, vc, vm, None, None)
    out = torch.full((16,), 7.0, dtype=torch.float32, device="cuda")
    qvg.qvg_attention_decode(cfg, None, 0, 0, 0, kb[1], vb[1], N, N, 0.125, out, 0, 0)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    q = np.zeros((5, H, D), np.uint16)
    got, _, _ = run_attention(qvg, cfg, q, kb, vb, N, N, 0.125)
    for h in range(H):
        ref = oracle.attention(q[:, h], kdec[h], vdec[h], 0.125)
        np.testing.assert_allclose(ref, np.broadcast_to(SY.bf16_bits_to_f32(vdec[h]).astype(np.float64).mean(0),
                                                        ref.shape), rtol=0, atol=1e-12)
        assert np.all(np.abs(got[h] - ref) <= tolerance(q[:, h], kdec[h], vdec[h], ref, 0.125, N))


@pytest.mark.parametrize("staged", [False, True])
def test_attention_full_size_sampled_rows(qvg, oracle, staged):
    """The Wan2.1 shape in the bench's launch configuration: 12 heads, a chunk
    of 4680 queries (token-major) over 32760 compressed keys (C = 256, S = 2,
    G = 64), random but legal encodings.  Sampled query rows of every head are
    checked against the oracle.  Three of them are probes: in head 0, 1 and 2
    one key (the first key, the first key of the ragged last tile, the last
    key) has its zero-points set to 4.0, which lifts each of its elements by
    8, and the probe row of that head is 0.25 in every channel; that key's
    score then leads all others by about 20, so the output is its value row
    and a skipped or misplaced tile fails."""
    wl = WL.WAN
    H, D, N, Nq, S, G, C = wl.heads, wl.head_dim, wl.tokens, 4680, wl.stages, wl.group_size, wl.clusters
    cfg = qvg.config(H, D, C, wl.lloyd_iters, S, G)
    kc, km, ki, kx = SY.random_encoding(wl.seed, SY.K_TENSOR, H, N, D, S, G, C)
    vc, vm, vi, vx = SY.random_encoding(wl.seed, SY.V_TENSOR, H, N, D, S, G, C)
    last_tile = (N - 1) // 64 * 64
    probes = [(0, 1, 0), (1, Nq - 3, last_tile), (2, Nq - 1, N - 1)]        # (head, query row, key)
    for h, _, key in probes:
        km[:, h, key, :] = (km[:, h, key, :] & np.uint32(0xFFFF)) | np.uint32(0x4400 << 16)
    kdec = np.stack([oracle.decode(kc[:, h], km[:, h], ki[h].astype(np.int32), kx[h], G) for h in range(H)])
    vdec = np.stack([oracle.decode(vc[:, h], vm[:, h], vi[h].astype(np.int32), vx[h], G) for h in range(H)])
    q = np.stack([SY.mixture_unit(wl, 0, SY.Q_TENSOR, h, 0, Nq) for h in range(H)], axis=1)   # [Nq][H][D]
    for h, row, _ in probes:
        q[row, h] = 0x3E80                                                   # 0.25
    kb, vb = device_views(qvg, kc, km, ki, kx), device_views(qvg, vc, vm, vi, vx)
    scale = float(np.float32(D ** -0.5))
    qd = to_dev(np.ascontiguousarray(q).reshape(-1))
    out = torch.empty((Nq, H, D), dtype=torch.float32, device="cuda")
    attend(qvg, cfg, qd, Nq, D, H * D, kb, vb, N, N, scale, out, D, H * D, staged)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    rows = sorted({0, 63, 64, 2345, 4607, 4608} | {row for _, row, _ in probes})
    for h in range(H):
        qs = q[rows, h]
        ref = oracle.attention(qs, kdec[h], vdec[h], scale)
        tol = tolerance(qs, kdec[h], vdec[h], ref, scale, N)
        err = np.abs(got[rows, h] - ref)
        assert np.all(err <= tol), f"head {h}: max err {err.max():.3g}, worst err/tol {(err / tol).max():.3g}"
    for h, row, key in probes:
        r = rows.index(row)
        vkey = SY.bf16_bits_to_f32(vdec[h, key]).astype(np.float64)
        ref = oracle.attention(q[row:row + 1, h], kdec[h], vdec[h], scale)[0]
        assert np.abs(ref - vkey).max() < 1e-3, "probe key does not dominate"
        assert np.abs(got[row, h] - vkey).max() < 1e-2, f"probe of key {key} (head {h})"
    assert np.isfinite(got).all()
