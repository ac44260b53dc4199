"""Failure path of the bounded waits in the persistent decoder and the
tensor-core k-means assign, exercised
without a GPU fault: a test flag makes each CTA's copy producer withhold its
first copy, so the consumers' first wait runs out after a short limit.  The
kernel must then record the error word (0x7E000000), drain the copies it did
issue and return, leaving the context usable; the library reports the word as
QVG_ERR_TIMEOUT.  Nothing here traps, faults or waits without a limit."""
import numpy as np
import pytest
import torch

from synth import synth as SY
from gpu_helpers import Encoded, to_dev, u16

pytestmark = pytest.mark.gpu

ERR_TIMEOUT_WORD = 0x7E000000


def _case(qvg, C):
    rng = np.random.default_rng(5 + C)
    H, D, N, S, G = 3, 128, 1000, 2, 64
    xb = SY.f64_to_bf16_bits(rng.standard_normal((H, N, D)))
    cfg = qvg.config(H, D, C, 2, S, G)
    return cfg, to_dev(xb), H, D, N


@pytest.mark.parametrize("C", [0, 16])
def test_withheld_copy_expires_the_wait_and_reports_timeout(qvg, C):
    cfg, x, H, D, N = _case(qvg, C)
    enc = Encoded(qvg, cfg, N)
    ws = qvg.alloc_workspace(cfg, N)
    if C:
        qvg.qvg_fit_centroids(cfg, x, N, N * D, D, None, enc["centroids"], enc["ids"], N, 0, ws)
    # a clean run first: the reference outputs, and no error word
    qvg.qvg_device_error(clear=True)
    qvg.qvg_encode(cfg, x, N, N * D, D, enc["centroids"], 0, enc["codes"], enc["meta"], enc["ids"], N, 0, ws)
    ref = torch.empty((H, N, D), dtype=torch.int16, device="cuda")
    qvg.qvg_decode(cfg, enc["codes"], enc["meta"], enc["ids"], enc["centroids"], N, 0, N, ref, N * D, D)
    torch.cuda.synchronize()
    assert qvg.qvg_device_error() == (qvg.QVG_OK, 0)
    codes_ref = enc["codes"].clone()
    try:
        qvg.qvg_debug_set_wait(20_000_000, 1)      # 20 ms, first copy withheld
        out = torch.empty_like(ref)
        qvg.qvg_decode(cfg, enc["codes"], enc["meta"], enc["ids"], enc["centroids"], N, 0, N, out, N * D, D)
        torch.cuda.synchronize()
        assert qvg.qvg_device_error(clear=True) == (qvg.QVG_ERR_TIMEOUT, ERR_TIMEOUT_WORD)
    finally:
        qvg.qvg_debug_set_wait(0, 0)
    # the context still works: a normal encode and decode reproduce the clean run
    # (the encoder has no waits: the flag leaves it unchanged)
    qvg.qvg_encode(cfg, x, N, N * D, D, enc["centroids"], 0, enc["codes"], enc["meta"], enc["ids"], N, 0, ws)
    out = torch.empty_like(ref)
    qvg.qvg_decode(cfg, enc["codes"], enc["meta"], enc["ids"], enc["centroids"], N, 0, N, out, N * D, D)
    torch.cuda.synchronize()
    assert qvg.qvg_device_error() == (qvg.QVG_OK, 0)
    assert torch.equal(enc["codes"], codes_ref)
    assert np.array_equal(u16(out), u16(ref))


def test_assign_withheld_tile_expires_the_wait_and_reports_timeout(qvg, oracle):
    """The tensor-core k-means assign (inside a fit) under the same flag: each
    CTA's token producer withholds its first tile, so the MMA issuer's and the
    epilogue's waits on it run out after 20 ms.  The kernel records
    0x7E000000 in the workspace's error word, drains the copies it issued,
    frees its tensor memory and returns; qvg_fit_stats reports the word as
    QVG_ERR_TIMEOUT, and the next fit, with the flag cleared, matches the
    oracle."""
    rng = np.random.default_rng(9)
    H, D, N, C, T = 2, 128, 1500, 16, 2
    xb = SY.f64_to_bf16_bits(rng.standard_normal((H, N, D)))
    cfg = qvg.config(H, D, C, T, 2, 64)
    x = to_dev(xb)
    enc = Encoded(qvg, cfg, N)
    ws = qvg.alloc_workspace(cfg, N)
    try:
        qvg.qvg_debug_set_wait(20_000_000, 1)
        qvg.qvg_fit_centroids(cfg, x, N, N * D, D, None, enc["centroids"], enc["ids"], N, 0, ws)
        torch.cuda.synchronize()
        st, stats = qvg.qvg_fit_stats(cfg, N, ws, with_status=True)
        assert (st, stats[3]) == (qvg.QVG_ERR_TIMEOUT, ERR_TIMEOUT_WORD)
    finally:
        qvg.qvg_debug_set_wait(0, 0)
    qvg.qvg_fit_centroids(cfg, x, N, N * D, D, None, enc["centroids"], enc["ids"], N, 0, ws)
    torch.cuda.synchronize()
    st, stats = qvg.qvg_fit_stats(cfg, N, ws, with_status=True)
    assert st == qvg.QVG_OK and stats[3] == 0
    for h in range(H):
        oc, oi = oracle.fit(xb[h], C, T)
        np.testing.assert_array_equal(enc.centroids()[0, h], oc)
        np.testing.assert_array_equal(enc.ids()[h], oi)
