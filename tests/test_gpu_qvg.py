"""GPU parity of the QVG path (k-means fit, assign, update, PRQ encode and
decode) against the CPU oracle, element by element, through the C ABI.

Integer outputs (ids, codes, meta words) and bf16 outputs (centroids,
reconstructions) must be bit-exact: the CUDA path takes every decision in the
arithmetic the oracle uses (exact argmin, exact cluster sums, fp32 quantiser).
"""
import numpy as np
import pytest
import torch

from synth import synth as SY
from synth import workloads as WL
from gpu_helpers import Encoded, run_fit_encode_decode, to_dev, u16

pytestmark = pytest.mark.gpu


def mixture(rng, N, D, M=8, spread=1.0, noise=0.1):
    centres = rng.standard_normal((M, D)) * spread
    lab = rng.integers(0, M, N)
    return SY.f64_to_bf16_bits(centres[lab] + noise * rng.standard_normal((N, D)))


def check_unit(oracle, xh, enc, dec, h, C, T, S, G, offset=0, n=None, warm=None, b=2):
    n = xh.shape[0] if n is None else n
    sl = slice(offset, offset + n)
    if C > 0:
        oc, oi = oracle.fit(xh, C, T, warm=warm)
        np.testing.assert_array_equal(enc.centroids()[0, h], oc, err_msg=f"centroids head {h}")
        np.testing.assert_array_equal(enc.ids()[h, sl], oi, err_msg=f"ids head {h}")
    else:
        oc, oi = None, None
    rc, rm = oracle.prq_encode(xh, oc, oi, S, G, b)
    np.testing.assert_array_equal(enc.codes()[:, h, sl], rc, err_msg=f"codes head {h}")
    np.testing.assert_array_equal(enc.meta()[:, h, sl], rm, err_msg=f"meta head {h}")
    np.testing.assert_array_equal(dec[h], oracle.decode(rc, rm, oi, oc, G, b), err_msg=f"decode head {h}")


@pytest.mark.parametrize("tensor", [SY.K_TENSOR, SY.V_TENSOR])
def test_tiny_workload_bit_exact(qvg, oracle, tensor):
    wl = WL.TINY
    H, D, N = wl.heads, wl.head_dim, wl.tokens
    xb = SY.mixture_layer(wl, 0, tensor)
    cfg = qvg.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D)
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size)


@pytest.mark.parametrize("D,G,S,C", [
    (64, 64, 1, 0), (128, 64, 2, 0), (128, 128, 3, 0), (128, 16, 4, 0), (256, 128, 2, 0), (32, 16, 2, 0),
    (32, 32, 1, 5), (64, 32, 2, 16), (128, 64, 2, 256), (128, 128, 3, 100), (64, 16, 4, 64), (128, 32, 1, 1),
])
def test_shape_variants_bit_exact(qvg, oracle, D, G, S, C):
    rng = np.random.default_rng(D * 7 + G + S * 3 + C)
    H, N, T = 3, 777, 2                      # ragged: not a multiple of any tile
    xb = np.stack([mixture(rng, N, D, M=12, spread=1.5, noise=0.2) for _ in range(H)])
    cfg = qvg.config(H, D, C, T, S, G)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D)
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, C, T, S, G)


@pytest.mark.parametrize("D,C", [(64, 120), (64, 200), (64, 256), (128, 150), (128, 192), (128, 65)])
def test_assign_tile_widths_bit_exact(qvg, oracle, D, C):
    """The tensor-core assign at each padded centroid count it is built for
    (C rounded up to a multiple of 64: 128, 192 and 256 with D = 64; 192 with
    D = 128; and 128 with 63 padding columns, whose scores must never win): a
    fit's centroids and ids, the encode and the decode bit-exact against the
    oracle on 1500 tokens per head (a ragged last tile)."""
    rng = np.random.default_rng(D * 1000 + C)
    H, N, T, S, G = 2, 1500, 2, 2, 64
    xb = np.stack([mixture(rng, N, D, M=max(8, C // 2), spread=1.0, noise=0.15) for _ in range(H)])
    cfg = qvg.config(H, D, C, T, S, G)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D)
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, C, T, S, G)


def test_token_major_layout_offsets_and_subrange_decode(qvg, oracle):
    """[N][H][D] input (head_stride = D, token_stride = H*D), rows written at an
    offset inside a larger buffer, and a decode of a sub-range."""
    rng = np.random.default_rng(11)
    H, D, N, C, T, S, G = 4, 128, 1000, 32, 2, 2, 64
    xb = np.stack([mixture(rng, N, D, M=20) for _ in range(H)])          # [H][N][D]
    xt = np.ascontiguousarray(xb.transpose(1, 0, 2))                    # [N][H][D]
    cfg = qvg.config(H, D, C, T, S, G)
    off, cap = 300, 1500
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xt), N, D, H * D, capacity=cap, offset=off,
                                     decode_range=(off + 100, off + 617))
    for h in range(H):
        oc, oi = oracle.fit(xb[h], C, T)
        np.testing.assert_array_equal(enc.centroids()[0, h], oc)
        np.testing.assert_array_equal(enc.ids()[h, off:off + N], oi)
        rc, rm = oracle.prq_encode(xb[h], oc, oi, S, G)
        np.testing.assert_array_equal(enc.codes()[:, h, off:off + N], rc)
        np.testing.assert_array_equal(enc.meta()[:, h, off:off + N], rm)
        np.testing.assert_array_equal(dec[h], oracle.decode(rc, rm, oi, oc, G)[100:617])
    # rows outside [off, off + N) were not touched
    assert np.all(enc.codes()[:, :, :off] == 0xFFFFFFFF) and np.all(enc.codes()[:, :, off + N:] == 0xFFFFFFFF)
    assert np.all(enc.ids()[:, :off] == 255)


def test_staged_assign_and_update(qvg, oracle):
    """assign given the oracle's centroids, update given the oracle's ids."""
    rng = np.random.default_rng(12)
    H, D, N, C = 2, 128, 3000, 256
    xb = np.stack([mixture(rng, N, D, M=64, spread=1.0, noise=0.15) for _ in range(H)])
    cent = np.stack([oracle.kmeans_init(xb[h], C) for h in range(H)])
    cfg = qvg.config(H, D, C, 1, 2, 64)
    x = to_dev(xb)
    ids = torch.full((H * N,), 255, dtype=torch.uint8, device="cuda")
    ws = qvg.alloc_workspace(cfg, N)
    qvg.qvg_assign(cfg, x, N, N * D, D, to_dev(cent), ids, N, 0, ws)
    torch.cuda.synchronize()
    gids = ids.cpu().numpy().reshape(H, N).astype(np.int32)
    for h in range(H):
        np.testing.assert_array_equal(gids[h], oracle.assign(xb[h], cent[h]))
    # update with the oracle's ids of the next-to-initial centroids
    oids = np.stack([oracle.assign(xb[h], cent[h]) for h in range(H)])
    c_dev = to_dev(cent)
    qvg.qvg_update(cfg, x, N, N * D, D, to_dev(oids.astype(np.uint8)), N, 0, c_dev, ws)
    torch.cuda.synchronize()
    got = u16(c_dev).reshape(H, C, D)
    for h in range(H):
        want, counts = oracle.update(xb[h], oids[h], cent[h])
        np.testing.assert_array_equal(got[h], want)


@pytest.mark.parametrize("D,C,N,big", [
    (128, 2, 9000, False),     # one cluster of ~6300 tokens: more than one shared-memory list
    (128, 2, 9000, True),      # the same with values >= 2^14 (128-bit sums over several lists)
    (64, 3, 7001, False),
    (32, 1, 5003, True),
    (128, 40, 3001, True),     # values >= 2^14 in short clusters (one list)
])
def test_update_long_clusters_and_large_values(qvg, oracle, D, C, N, big):
    """The update alone, given ids with clusters longer than one list of
    tokens, values of magnitude >= 2^14, and id rows that start off a 16-byte
    boundary (capacity and offset not multiples of 16)."""
    rng = np.random.default_rng(D + 10 * C + N + big)
    H, cap, off = 2, N + 37, 5
    x = rng.standard_normal((H, N, D))
    if big:
        m = rng.random((H, N, D)) < 0.002
        x[m] = rng.choice([-1.0, 1.0], m.sum()) * 2.0 ** rng.integers(14, 18, m.sum())
    xb = SY.f64_to_bf16_bits(x)
    p = rng.random(C) + 0.1
    p[0] += 4.0                                    # cluster 0 holds most tokens
    oids = np.stack([rng.choice(C, N, p=p / p.sum()) for _ in range(H)]).astype(np.int32)
    cent = SY.f64_to_bf16_bits(rng.standard_normal((H, C, D)))
    ids = np.full((H, cap), 255, np.uint8)
    ids[:, off:off + N] = oids
    cfg = qvg.config(H, D, C, 1, 2, 32)
    c_dev = to_dev(cent)
    ws = qvg.alloc_workspace(cfg, N)
    qvg.qvg_update(cfg, to_dev(xb), N, N * D, D, to_dev(ids.reshape(-1)), cap, off, c_dev, ws)
    torch.cuda.synchronize()
    got = u16(c_dev).reshape(H, C, D)
    for h in range(H):
        want, counts = oracle.update(xb[h], oids[h], cent[h])
        if C <= 3:
            assert counts.max() > 4096
        np.testing.assert_array_equal(got[h], want)


@pytest.mark.parametrize("D,C", [(128, 16), (64, 40)])
def test_fit_with_values_beyond_the_first_window(qvg, oracle, D, C):
    """A fit whose later updates apply only the changed ids to the stored
    exact sums: head 0 has a few values of magnitude 2^14..2^16 (those groups
    take 128-bit sums and full updates), head 1 has none."""
    rng = np.random.default_rng(D + C)
    H, N, T, S, G = 2, 2500, 4, 2, 64
    xb = np.stack([mixture(rng, N, D, M=24, spread=1.5, noise=0.3) for _ in range(H)])
    xf = SY.bf16_bits_to_f32(xb).astype(np.float64)
    m = rng.random((N, D)) < 0.0005
    xf[0][m] = rng.choice([-1.0, 1.0], m.sum()) * 2.0 ** rng.integers(14, 17, m.sum())
    xb = SY.f64_to_bf16_bits(xf)
    cfg = qvg.config(H, D, C, T, S, G)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D)
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, C, T, S, G)


def test_update_means_at_rounding_midpoints(qvg, oracle):
    """Cluster means that are exact bf16 rounding midpoints (ties to even),
    or lie just off them, or next to a power of two, next to ordinary
    clusters and an empty one: the rounding is decided exactly there."""
    rng = np.random.default_rng(77)
    D, C = 64, 8
    def nxt(b, k=1):                       # the k-th bf16 pattern above b (positive values)
        return (b.astype(np.int64) + k).astype(np.uint16)
    a = SY.f64_to_bf16_bits(np.abs(rng.standard_normal((6, D))) + 0.1)
    edge = np.full(D, 0x3FFF, np.uint16)   # 1.9921875, the last bf16 below 2
    rows, lab = [], []
    def add(k, *vals):
        for v in vals:
            rows.append(v); lab.append(k)
    add(0, a[0], nxt(a[0]))                          # mean = midpoint
    add(1, a[1], a[1], nxt(a[1]), nxt(a[1]))         # midpoint from four tokens
    add(2, a[2], a[2], nxt(a[2], 2))                 # a + 2/3 ulp
    add(3, *([a[3]] * 3 + [nxt(a[3])] * 3))          # midpoint from six
    for v in SY.f64_to_bf16_bits(rng.standard_normal((1000, D))):
        add(4, v)                                    # an ordinary cluster
    add(5, a[5], a[5] ^ np.uint16(0x8000))           # mean 0
    add(6, edge, nxt(edge))                          # midpoint below 2.0
    x = np.stack(rows).astype(np.uint16)
    ids = np.array(lab, np.int32)
    perm = rng.permutation(len(ids))
    x, ids = x[perm], ids[perm]
    N = len(ids)
    cent = SY.f64_to_bf16_bits(rng.standard_normal((C, D)))
    cfg = qvg.config(1, D, C, 1, 2, 32)
    c_dev = to_dev(cent[None])
    ws = qvg.alloc_workspace(cfg, N)
    qvg.qvg_update(cfg, to_dev(x[None]), N, N * D, D, to_dev(ids.astype(np.uint8)), N, 0, c_dev, ws)
    torch.cuda.synchronize()
    want, counts = oracle.update(x, ids, cent)
    assert counts[7] == 0
    np.testing.assert_array_equal(u16(c_dev).reshape(C, D), want)


def test_compress_host_matches_device_calls(qvg):
    """qvg_compress_host (host buffers in and out) gives the bytes of the
    separate device calls: fit, encode, decode, then the encoding copied back."""
    rng = np.random.default_rng(31)
    H, D, N, C, T, S, G = 3, 128, 1111, 32, 3, 2, 64
    xb = np.stack([mixture(rng, N, D, M=12) for _ in range(H)])          # [H][N][D]
    xt = np.ascontiguousarray(xb.transpose(1, 0, 2))                    # token-major [N][H][D]
    cfg = qvg.config(H, D, C, T, S, G)
    x_dev = to_dev(xt.reshape(-1))
    ref = Encoded(qvg, cfg, N)
    ws = qvg.alloc_workspace(cfg, N)
    ref_out = torch.empty((N, H, D), dtype=torch.int16, device="cuda")
    qvg.qvg_fit_centroids(cfg, x_dev, N, D, H * D, None, ref["centroids"], ref["ids"], N, 0, ws)
    qvg.qvg_encode(cfg, x_dev, N, D, H * D, ref["centroids"], 0, ref["codes"], ref["meta"], ref["ids"], N, 0, ws)
    qvg.qvg_decode(cfg, ref["codes"], ref["meta"], ref["ids"], ref["centroids"], N, 0, N, ref_out, D, H * D)
    torch.cuda.synchronize()
    host_x = torch.from_numpy(xt.reshape(-1).view(np.int16)).pin_memory()
    cb, mb, ib, xbytes = qvg.qvg_encoded_bytes(cfg, N, 1)
    host_out = torch.full((cb + mb + ib + xbytes,), 0xAB, dtype=torch.uint8).pin_memory()
    got = Encoded(qvg, cfg, N)
    staging = torch.empty_like(x_dev)
    out = torch.empty_like(ref_out)
    qvg.qvg_compress_host(cfg, host_x, staging, N, D, H * D, None, got["centroids"], got["ids"], got["codes"],
                          got["meta"], out, host_out, ws)
    torch.cuda.synchronize()
    assert torch.equal(staging, x_dev)
    assert torch.equal(out, ref_out)
    want = b"".join(ref[k].cpu().numpy().tobytes()[:n] for k, n in
                    (("codes", cb), ("meta", mb), ("ids", ib), ("centroids", xbytes)))
    assert host_out.numpy().tobytes() == want


@pytest.mark.parametrize("D", [64, 128])
def test_ties_and_degenerate_inputs(qvg, oracle, D):
    """Exact duplicate tokens (ties at distance 0 between equal centroids),
    fewer tokens than clusters (duplicate initial centroids), constant rows
    (zero scale) and a single token (one partial tile)."""
    rng = np.random.default_rng(13 + D)
    G, S = 32, 2
    base = mixture(rng, 40, D, M=3)
    cases = [
        np.concatenate([base, base, base[:7]]),                        # duplicates
        base[:5],                                                        # N < C
        np.tile(SY.f64_to_bf16_bits(np.full((1, D), 0.75)), (50, 1)),   # constant rows
        base[:1],                                                        # one token
    ]
    for k, xh in enumerate(cases):
        N = xh.shape[0]
        for C in (1, 8):
            cfg = qvg.config(1, D, C, 3, S, G)
            enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xh[None]), N, N * D, D)
            check_unit(oracle, xh, enc, dec, 0, C, 3, S, G)


def test_outlier_and_wide_range_values(qvg, oracle):
    """Large outlier channels, tiny magnitudes and exact zeros."""
    rng = np.random.default_rng(14)
    H, D, N, C, S, G = 2, 128, 900, 16, 3, 64
    x = rng.standard_normal((H, N, D))
    x[:, :, 3] *= 60.0
    x[:, :, 100] *= 1e-7
    x[:, ::7, 50] = 0.0
    xb = SY.f64_to_bf16_bits(x)
    cfg = qvg.config(H, D, C, 3, S, G)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D)
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, C, 3, S, G)


def test_warm_start_fit(qvg, oracle):
    rng = np.random.default_rng(15)
    H, D, N, C, T = 2, 64, 1200, 16, 2
    xb = np.stack([mixture(rng, N, D, M=16) for _ in range(H)])
    warm = np.stack([SY.f64_to_bf16_bits(rng.standard_normal((C, D))) for _ in range(H)])
    cfg = qvg.config(H, D, C, T, 2, 64)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D, warm=to_dev(warm))
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, C, T, 2, 64, warm=warm[h])


def test_encode_with_device_assign(qvg, oracle):
    """qvg_encode(assign=1): ids computed on the fly against given centroids."""
    rng = np.random.default_rng(16)
    H, D, N, C, S, G = 3, 128, 2049, 64, 2, 64
    xb = np.stack([mixture(rng, N, D, M=30) for _ in range(H)])
    cent = np.stack([oracle.fit(xb[h][:500], C, 2)[0] for h in range(H)])
    cfg = qvg.config(H, D, C, 2, S, G)
    enc = Encoded(qvg, cfg, N)
    ws = qvg.alloc_workspace(cfg, N)
    enc["centroids"][: cent.size].copy_(to_dev(cent.reshape(-1)))
    qvg.qvg_encode(cfg, to_dev(xb), N, N * D, D, enc["centroids"], 1, enc["codes"], enc["meta"], enc["ids"], N, 0,
                   ws)
    torch.cuda.synchronize()
    for h in range(H):
        oi = oracle.assign(xb[h], cent[h])
        np.testing.assert_array_equal(enc.ids()[h], oi)
        rc, rm = oracle.prq_encode(xb[h], cent[h], oi, S, G)
        np.testing.assert_array_equal(enc.codes()[:, h], rc)
        np.testing.assert_array_equal(enc.meta()[:, h], rm)


def test_repeated_calls_are_deterministic(qvg):
    wl = WL.TINY
    H, D, N = wl.heads, wl.head_dim, wl.tokens
    x = to_dev(SY.mixture_layer(wl, 0, 0))
    cfg = qvg.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size)
    runs = [run_fit_encode_decode(qvg, cfg, x, N, N * D, D) for _ in range(3)]
    for enc, dec in runs[1:]:
        assert np.array_equal(enc.codes(), runs[0][0].codes())
        assert np.array_equal(enc.centroids(), runs[0][0].centroids())
        assert np.array_equal(dec, runs[0][1])


@pytest.mark.parametrize("G", [16, 32, 64, 128])
def test_quantiser_half_integer_ties(qvg, oracle, G):
    """Values on a coarse grid make t = (r - z) / s land exactly on k + 1/2
    (or within half an ulp of it) for many elements, so rint(t) is decided by
    the rounding of the product alone: any fusion of the multiply with the
    rounding addition, or any skipped clamp that matters, changes codes here."""
    rng = np.random.default_rng(4242 + G)
    H, N, D, S = 2, 513, 128, 3
    grid = rng.integers(-24, 25, size=(H, N, D)).astype(np.float64) / 16.0
    # a few groups with a far outlier, so the clamp path is taken as well
    grid[:, ::37, 5] = 900.0
    xb = SY.f64_to_bf16_bits(grid)
    cfg = qvg.config(H, D, 0, 0, S, G)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D)
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, 0, 0, S, G)


@pytest.mark.parametrize("D,G,S,C", [
    (128, 64, 2, 0), (128, 128, 1, 0), (128, 16, 3, 0), (64, 32, 2, 16), (32, 16, 4, 0), (256, 64, 2, 0),
    (128, 64, 2, 256), (128, 128, 3, 100),
])
def test_four_bit_codes_bit_exact(qvg, oracle, D, G, S, C):
    """4-bit codes (the PRQ_INT4 variant): fit, encode and decode match the
    oracle bit for bit on ragged shapes (777 tokens)."""
    rng = np.random.default_rng(D * 3 + G + S + C + 4)
    H, N, T = 3, 777, 2
    xb = np.stack([mixture(rng, N, D, M=12, spread=1.5, noise=0.2) for _ in range(H)])
    cfg = qvg.config(H, D, C, T, S, G, 4)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D)
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, C, T, S, G, b=4)


@pytest.mark.parametrize("G", [16, 64, 128])
def test_four_bit_half_integer_ties(qvg, oracle, G):
    """The coarse-grid tie case of the quantiser, with 15 steps."""
    rng = np.random.default_rng(99 + G)
    H, N, D, S = 2, 300, 128, 2
    grid = rng.integers(-40, 41, size=(H, N, D)).astype(np.float64) / 8.0
    grid[:, ::29, 7] = -700.0
    xb = SY.f64_to_bf16_bits(grid)
    cfg = qvg.config(H, D, 0, 0, S, G, 4)
    enc, dec = run_fit_encode_decode(qvg, cfg, to_dev(xb), N, N * D, D)
    for h in range(H):
        check_unit(oracle, xb[h], enc, dec, h, 0, 0, S, G, b=4)


def test_fit_reuses_workspace_without_stale_norms(qvg, oracle):
    """A fit keeps ||x||^2 per token in the workspace for its later assign
    steps; a second fit on other data in the same workspace must not use the
    first fit's norms.  The first fit runs on x / 64 (exact in bf16), so stale
    norms would shrink the screen's error bound on the second."""
    rng = np.random.default_rng(31)
    H, D, N, C, T = 2, 128, 3000, 64, 3
    xb = np.stack([mixture(rng, N, D, M=48, spread=1.0, noise=0.2) for _ in range(H)])
    small = SY.f64_to_bf16_bits(SY.bf16_bits_to_f32(xb).astype(np.float64) / 64.0)
    cfg = qvg.config(H, D, C, T, 2, 64)
    ws = qvg.alloc_workspace(cfg, N)
    cent = torch.empty(H * C * D, dtype=torch.int16, device="cuda")
    ids = torch.empty(H * N, dtype=torch.uint8, device="cuda")
    qvg.qvg_fit_centroids(cfg, to_dev(small), N, N * D, D, None, cent, ids, N, 0, ws)
    qvg.qvg_fit_centroids(cfg, to_dev(xb), N, N * D, D, None, cent, ids, N, 0, ws)
    torch.cuda.synchronize()
    got_c = u16(cent).reshape(H, C, D)
    got_i = ids.cpu().numpy().reshape(H, N).astype(np.int32)
    for h in range(H):
        oc, oi = oracle.fit(xb[h], C, T)
        np.testing.assert_array_equal(got_c[h], oc, err_msg=f"centroids head {h}")
        np.testing.assert_array_equal(got_i[h], oi, err_msg=f"ids head {h}")
    assert qvg.qvg_fit_stats(cfg, N, ws)[3] == 0


def test_empty_inputs_write_nothing(qvg):
    """Zero tokens: assign, update, encode, an empty decode range, the
    cross-layer codec and attention with no queries return OK and write
    nothing; the calls that need a token (fit, append, the hybrid) refuse
    with an argument error and write nothing either."""
    H, D, C, T, S, G = 2, 128, 16, 2, 2, 64
    cap = 300
    cfg = qvg.config(H, D, C, T, S, G)
    enc = qvg.alloc_encoded(cfg, cap)
    for k, t in enc.items():
        t.fill_(0xFF if t.dtype == torch.uint8 else -1)
    x = torch.zeros((cap, H, D), dtype=torch.int16, device="cuda")
    ws = qvg.alloc_workspace(cfg, cap)
    out = torch.full((cap, H, D), -1, dtype=torch.int16, device="cuda")
    before = {k: t.clone() for k, t in enc.items()}
    qvg.qvg_assign(cfg, x, 0, D, H * D, enc["centroids"], enc["ids"], cap, 0, ws)
    qvg.qvg_update(cfg, x, 0, D, H * D, enc["ids"], cap, 0, enc["centroids"], ws)
    qvg.qvg_encode(cfg, x, 0, D, H * D, enc["centroids"], 1, enc["codes"], enc["meta"], enc["ids"], cap, 0, ws)
    qvg.qvg_decode(cfg, enc["codes"], enc["meta"], enc["ids"], enc["centroids"], cap, 7, 7, out, D, H * D)
    with pytest.raises(qvg.QvgError):
        qvg.qvg_fit_centroids(cfg, x, 0, D, H * D, None, enc["centroids"], enc["ids"], cap, 0, ws)
    # cross-layer codec (no clusters) with no tokens
    ccfg = qvg.config(H, D, 0, 0, S, G)
    cws = qvg.alloc_workspace(ccfg, cap)
    xh = torch.full((cap, H * D), -1, dtype=torch.int16, device="cuda")
    qvg.coral_predict_encode(ccfg, None, None, x.view(cap, H * D), 0, enc["codes"], enc["meta"], xh, None, cws)
    qvg.coral_predict_decode(ccfg, None, None, 0, enc["codes"], enc["meta"], xh, None, cws)
    sws = torch.empty(qvg.coral_sas_workspace_bytes(cfg, cap), dtype=torch.uint8, device="cuda")
    with pytest.raises(qvg.QvgError):
        qvg.coral_sas_encode(cfg, None, None, x.view(cap, H * D), 0, enc["codes"], enc["meta"], enc["ids"],
                             enc["centroids"], xh, sws)
    # attention with no queries over a one-key history
    q = torch.zeros((4, H, D), dtype=torch.int16, device="cuda")
    ao = torch.full((4, H, D), float("nan"), dtype=torch.float32, device="cuda")
    view = qvg.encoded_view(enc)
    qvg.qvg_attention_decode(cfg, q, 0, D, H * D, view, view, cap, 1, 0.1, ao, D, H * D)
    aws = torch.empty(max(1, qvg.qvg_attention_workspace_bytes(cfg, 1)), dtype=torch.uint8, device="cuda")
    qvg.qvg_attention_decode_staged(cfg, q, 0, D, H * D, view, view, cap, 1, 0.1, ao, D, H * D, aws)
    torch.cuda.synchronize()
    for k, t in enc.items():
        assert torch.equal(t, before[k]), k
    assert bool((out == -1).all()) and bool((xh == -1).all()) and bool(torch.isnan(ao).all())
