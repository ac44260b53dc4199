"""GPU parity of the streaming append path (centroid caching): chunks are
fitted (warm-started) every k-th step and only assigned otherwise; the whole
history decodes against each chunk's own centroid version."""
import numpy as np
import pytest
import torch

from synth import synth as SY
from synth import workloads as WL
from gpu_helpers import to_dev, u16, u32

pytestmark = pytest.mark.gpu


def run_stream(qvg, cfg, xb, chunk, steps, every, layout="hnd"):
    H, N, D = xb.shape
    cache, bufs = qvg.make_cache(cfg, chunk * steps, max_versions=(steps + every - 1) // every,
                                 max_chunks=steps)
    ws = qvg.alloc_workspace(cfg, chunk)
    x = to_dev(xb if layout == "hnd" else np.ascontiguousarray(xb.transpose(1, 0, 2)))
    hs, ts = (N * D, D) if layout == "hnd" else (D, H * D)
    for t in range(steps):
        xt = x[:, t * chunk:] if layout == "hnd" else x[t * chunk:]
        qvg.qvg_append_chunk(cfg, cache, xt, chunk, hs, ts, t % every == 0, ws)
    assert cache.n_used == chunk * steps and cache.n_chunks == steps
    out = torch.full((H, chunk * steps, D), -1, dtype=torch.int16, device="cuda")
    qvg.qvg_decode_cache(cfg, cache, 0, chunk * steps, out, chunk * steps * D, D)
    # a partial window across a chunk boundary too
    w0, w1 = chunk - 9, min(2 * chunk + 8, chunk * steps)
    out2 = torch.full((H, w1 - w0, D), -1, dtype=torch.int16, device="cuda")
    qvg.qvg_decode_cache(cfg, cache, w0, w1, out2, (w1 - w0) * D, D)
    torch.cuda.synchronize()
    return cache, bufs, u16(out), u16(out2)


@pytest.mark.parametrize("layout,b", [("hnd", 2), ("nhd", 2), ("nhd", 4)])
def test_stream_matches_oracle(qvg, oracle, layout, b):
    wl = WL.STREAM
    H, D, C, T, S, G = 2, 64, 32, 2, 2, 64
    chunk, steps, every = 390, 6, 3
    n = chunk * steps
    rng = np.random.default_rng(21)
    # a drifting mixture: the tiny workload's units with drift
    xb = np.stack([SY.mixture_unit(WL.TINY, 0, 0, h, 0, n) for h in range(H)])
    xb = SY.f64_to_bf16_bits(SY.bf16_bits_to_f32(xb).astype(np.float64)
                             + np.linspace(0, 1, n)[None, :, None] * rng.standard_normal((H, 1, D)))
    cfg = qvg.config(H, D, C, T, S, G, b)
    cache, bufs, dec, dec2 = run_stream(qvg, cfg, xb, chunk, steps, every, layout)
    V = cache.n_versions
    assert V == 2
    codes = u32(bufs["codes"]).reshape(S, H, n, D * b // 32)
    meta = u32(bufs["meta"]).reshape(S, H, n, D // G)
    ids = bufs["ids"].cpu().numpy()[: H * n].reshape(H, n).astype(np.int32)
    cents = u16(bufs["centroids"])[: V * H * C * D].reshape(V, H, C, D)
    cver = bufs["chunk_version"].cpu().numpy()[:steps]
    coff = bufs["chunk_offset"].cpu().numpy()[: steps + 1]
    assert list(coff) == [chunk * t for t in range(steps + 1)]
    for h in range(H):
        vers, ov, oi, oc, om = oracle.stream(xb[h], chunk, steps, every, C, T, S, G, b)
        assert list(cver) == list(ov)
        for v in range(V):
            np.testing.assert_array_equal(cents[v, h], vers[v])
        np.testing.assert_array_equal(ids[h], oi)
        np.testing.assert_array_equal(codes[:, h], oc)
        np.testing.assert_array_equal(meta[:, h], om)
        want = np.concatenate([oracle.decode(oc[:, t * chunk:(t + 1) * chunk], om[:, t * chunk:(t + 1) * chunk],
                                             oi[t * chunk:(t + 1) * chunk], vers[ov[t]], G, b) for t in range(steps)])
        np.testing.assert_array_equal(dec[h], want)
        np.testing.assert_array_equal(dec2[h], want[chunk - 9:min(2 * chunk + 8, n)])


def test_stream_wan_shape_first_chunks(qvg, oracle):
    """Two real 4680-token chunks of the streaming workload (Wan2.1 shape, C=256,
    T=4): chunk 0 refits cold, chunk 1 assigns to the cached table."""
    wl = WL.STREAM
    H, D, chunk = 2, wl.head_dim, wl.chunk_tokens
    n = 2 * chunk
    xb = np.stack([SY.mixture_unit(wl, 0, 0, h, 0, n) for h in range(H)])
    cfg = qvg.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size)
    cache, bufs, dec, _ = run_stream(qvg, cfg, xb, chunk, 2, wl.refit_every)
    S, G, C = wl.stages, wl.group_size, wl.clusters
    codes = u32(bufs["codes"]).reshape(S, H, n, D // 16)
    cents = u16(bufs["centroids"])[: H * C * D].reshape(H, C, D)
    for h in range(H):
        vers, ov, oi, oc, om = oracle.stream(xb[h], chunk, 2, wl.refit_every, C, wl.lloyd_iters, S, G)
        np.testing.assert_array_equal(cents[h], vers[0])
        np.testing.assert_array_equal(codes[:, h], oc)
        want = oracle.decode(oc, om, oi, vers[0], G)
        np.testing.assert_array_equal(dec[h], want)


def test_stream_wan_shape_through_a_warm_refit(qvg, oracle):
    """Ten real 4680-token chunks of the streaming workload (Wan2.1 shape,
    C = 256, T = 4, refit every 8th chunk): chunk 0 refits cold, chunks 1-7
    assign to that table, chunk 8 refits warm-started from it (a second
    version), chunk 9 assigns to the new one.  Centroid versions, ids, codes,
    scale/zero words and the decode of the whole history -- and of a window
    across the version change -- are compared with the oracle bit for bit on
    head 0 (two heads run on the GPU)."""
    wl = WL.STREAM
    H, D, chunk, steps = 2, wl.head_dim, wl.chunk_tokens, 10
    n = chunk * steps
    S, G, C, T = wl.stages, wl.group_size, wl.clusters, wl.lloyd_iters
    xb = np.stack([SY.mixture_unit(wl, 0, SY.K_TENSOR, h, 0, n) for h in range(H)])
    cfg = qvg.config(H, D, C, T, S, G)
    cache, bufs, dec, _ = run_stream(qvg, cfg, xb, chunk, steps, wl.refit_every)
    assert cache.n_versions == 2
    w0, w1 = 7 * chunk + 100, 9 * chunk + 50          # chunk 7 (version 0) .. chunk 9 (version 1)
    win = torch.full((H, w1 - w0, D), -1, dtype=torch.int16, device="cuda")
    qvg.qvg_decode_cache(cfg, cache, w0, w1, win, (w1 - w0) * D, D)
    torch.cuda.synchronize()
    win = u16(win)
    codes = u32(bufs["codes"]).reshape(S, H, n, D // 16)
    meta = u32(bufs["meta"]).reshape(S, H, n, D // G)
    ids = bufs["ids"].cpu().numpy()[: H * n].reshape(H, n).astype(np.int32)
    cents = u16(bufs["centroids"])[: 2 * H * C * D].reshape(2, H, C, D)
    h = 0
    vers, ov, oi, oc, om = oracle.stream(xb[h], chunk, steps, wl.refit_every, C, T, S, G)
    assert list(ov) == [0] * 8 + [1] * 2
    for v in range(2):
        np.testing.assert_array_equal(cents[v, h], vers[v], err_msg=f"version {v}")
    np.testing.assert_array_equal(ids[h], oi)
    np.testing.assert_array_equal(codes[:, h], oc)
    np.testing.assert_array_equal(meta[:, h], om)
    want = np.concatenate([oracle.decode(oc[:, t * chunk:(t + 1) * chunk], om[:, t * chunk:(t + 1) * chunk],
                                         oi[t * chunk:(t + 1) * chunk], vers[ov[t]], G) for t in range(steps)])
    np.testing.assert_array_equal(dec[h], want)
    np.testing.assert_array_equal(win[h], want[w0:w1])
