"""GPU parity of the Coral-KV cross-layer codec.

The prediction is a tensor-core fp32 contraction, so it is compared with the
oracle's fp64 prediction within an accumulation bound; every integer decision
after it is then checked bit-exactly by driving the oracle's quantiser with
the GPU's own fp32 prediction (staged parity).  Encoder and decoder
reconstructions must be bit-identical.  The closed-loop chain over several
layers is also run on both sides independently and compared in relative MSE.
"""
import numpy as np
import pytest
import torch

from synth import synth as SY
from synth import workloads as WL
from gpu_helpers import to_dev, u16, u32

pytestmark = pytest.mark.gpu

GAMMA = 2.0 ** -13


def pred_bound(xh, B, U, W, H, D):
    f = lambda a: np.abs(SY.bf16_bits_to_f32(a).astype(np.float64))
    x = f(xh).reshape(-1, H, D)
    blk = np.einsum("hoi,nhi->nho", f(B), x).reshape(x.shape[0], H * D)
    t_abs = x.reshape(x.shape[0], H * D) @ f(W)
    low = t_abs @ f(U).T
    return GAMMA * (blk + low) + 1e-6


def gpu_layer(qvg, cfg, pred, xprev_dev, xnext_dev, N, encode=True, codes=None, meta=None):
    H, D, S, G = cfg.num_heads, cfg.head_dim, cfg.num_stages, cfg.group_size
    if encode:
        codes = torch.full((S * H * N * D // 16,), -1, dtype=torch.int32, device="cuda")
        meta = torch.full((S * H * N * D // G,), -1, dtype=torch.int32, device="cuda")
    xh = torch.full((N, H * D), -1, dtype=torch.int16, device="cuda")
    pout = torch.empty((N, H * D), dtype=torch.float32, device="cuda")
    ws = qvg.alloc_workspace(cfg, N)
    if encode:
        qvg.coral_predict_encode(cfg, pred, xprev_dev, xnext_dev, N, codes, meta, xh, pout, ws)
    else:
        qvg.coral_predict_decode(cfg, pred, xprev_dev, N, codes, meta, xh, pout, ws)
    torch.cuda.synchronize()
    assert qvg.qvg_fit_stats(cfg, N, ws)[3] == 0      # no bounded wait expired
    return codes, meta, xh, pout


def predictor(qvg, B, U, W):
    dev = [to_dev(a) for a in (B, U, W)]
    p = qvg.qvg.coral_predictor(B=dev[0].data_ptr(), U=dev[1].data_ptr(), W=dev[2].data_ptr(), rank=U.shape[1])
    return p, dev


# (tokens, rank, heads, group size, stages): rank 32 runs the tcgen05 path
# (token tiles of 128 with a ragged last tile), the other ranks the general
# one; the last three rows give the tcgen05 path's other stage counts
@pytest.mark.parametrize("N,R,H,G,S", [(300, 32, 4, None, None), (64, 16, 4, None, None), (129, 0, 4, None, None),
                                       (300, 32, 4, 16, None), (300, 32, 4, 64, None), (1100, 32, 8, None, None),
                                       (300, 32, 4, None, 1), (300, 32, 4, 16, 3), (129, 32, 4, 64, 4)])
def test_coral_chain_staged_parity(qvg, oracle, N, R, H, G, S):
    wl = WL.CORAL
    D, L = wl.head_dim, 4
    S = S or wl.stages
    G = G or wl.group_size
    small = WL.Workload(**{**wl.__dict__, "heads": H, "tokens": N, "layers": L, "rank": max(R, 16)})
    xs = SY.coral_layers(small, SY.K_TENSOR, 0, N)              # [L][N][H*D]
    cfg = qvg.config(H, D, 0, 0, S, G)
    # layer 0: plain PRQ, bit-exact
    codes, meta, xh, _ = gpu_layer(qvg, cfg, None, None, to_dev(xs[0]), N)
    oc, om, oxh, _ = oracle.coral_encode_layer(None, xs[0], None, None, None, H, D, S, G)
    np.testing.assert_array_equal(u32(codes).reshape(oc.shape), oc)
    np.testing.assert_array_equal(u32(meta).reshape(om.shape), om)
    np.testing.assert_array_equal(u16(xh), oxh)
    prev = u16(xh)
    for l in range(L - 1):
        B, U, W = SY.coral_predictor(small, l)
        if R == 0:
            U = np.zeros((H * D, 0), np.uint16)
            W = U
        pred, keep = predictor(qvg, B, U, W)
        codes, meta, xh, pout = gpu_layer(qvg, cfg, pred, to_dev(prev), to_dev(xs[l + 1]), N)
        gp = pout.cpu().numpy()
        # 1. prediction within the fp32 accumulation bound of the fp64 value
        p64 = oracle.coral_predict(prev, B, U if R else np.zeros((H * D, 16), np.uint16),
                                   W if R else np.zeros((H * D, 16), np.uint16), H, D)
        bound = pred_bound(prev, B, U if R else np.zeros((H * D, 1), np.uint16),
                           W if R else np.zeros((H * D, 1), np.uint16), H, D)
        assert np.all(np.abs(gp - p64) <= bound), np.max(np.abs(gp - p64) / bound)
        # 2. quantiser and reconstruction bit-exact given the GPU's prediction
        oc, om, oxh, _ = oracle.coral_encode_layer(prev, xs[l + 1], B, U, W, H, D, S, G, pred_in=gp)
        np.testing.assert_array_equal(u32(codes).reshape(oc.shape), oc)
        np.testing.assert_array_equal(u32(meta).reshape(om.shape), om)
        np.testing.assert_array_equal(u16(xh), oxh)
        # 3. the decoder rebuilds the encoder's reconstruction exactly
        _, _, dxh, dp = gpu_layer(qvg, cfg, pred, to_dev(prev), None, N, encode=False, codes=codes, meta=meta)
        np.testing.assert_array_equal(u16(dxh), u16(xh))
        np.testing.assert_array_equal(dp.cpu().numpy(), gp)
        prev = u16(xh)


def test_coral_closed_loop_end_to_end(qvg, oracle):
    """Both sides run the whole chain on their own; reconstructions agree in
    relative MSE within 1% at every layer.  At the first predicted layer the
    codes are identical except where the fp32 and fp64 predictions straddle a
    rounding boundary; after that a single differing code changes the next
    prediction of its whole token (the low-rank term mixes all heads), so the
    two chains are compared in quality only -- their per-layer exactness is
    the staged test above."""
    wl = WL.CORAL
    H, D, S, G, L, N = 16, wl.head_dim, wl.stages, wl.group_size, 6, 256
    small = WL.Workload(**{**wl.__dict__, "tokens": N, "layers": L})
    xs = SY.coral_layers(small, SY.V_TENSOR, 0, N)
    cfg = qvg.config(H, D, 0, 0, S, G)
    g_prev = o_prev = None
    total = diff = 0
    for l in range(L):
        if l == 0:
            codes, meta, xh, _ = gpu_layer(qvg, cfg, None, None, to_dev(xs[0]), N)
            oc, om, oxh, _ = oracle.coral_encode_layer(None, xs[0], None, None, None, H, D, S, G)
        else:
            B, U, W = SY.coral_predictor(small, l - 1)
            pred, keep = predictor(qvg, B, U, W)
            codes, meta, xh, _ = gpu_layer(qvg, cfg, pred, to_dev(g_prev), to_dev(xs[l]), N)
            oc, om, oxh, _ = oracle.coral_encode_layer(o_prev, xs[l], B, U, W, H, D, S, G)
        gc = u32(codes).reshape(oc.shape)
        if l <= 1:
            total += gc.size
            diff += int(np.sum(gc != oc))
        g_prev, o_prev = u16(xh), oxh
        x = SY.bf16_bits_to_f32(xs[l]).astype(np.float64)
        eg = np.mean((SY.bf16_bits_to_f32(g_prev) - x) ** 2)
        eo = np.mean((SY.bf16_bits_to_f32(o_prev) - x) ** 2)
        assert abs(eg - eo) <= 0.01 * eo, (l, eg, eo)
    assert diff <= 1e-3 * total, (diff, total)


@pytest.mark.parametrize("N,H", [(1100, 4), (9000, 4)])
def test_coral_fit_block_parity(qvg, oracle, N, H):
    """Adapted block predictors: the GPU's least-squares B_h (fp32 sums and
    fp32 Cholesky solve) against the oracle's fp64 solution Z.  Bound, from
    the arithmetic: rounding to bf16 (8 significant bits) errs by at most
    2^-8 |Z|; the fp32 solve by the first-order Cholesky bound
    cond(G_h) * D * 2^-24 of the block's scale (taken twice), with cond(G_h)
    computed here from the ridge-regularised Gram matrix.  The layer is then
    encoded with the fitted block and checked bit-exactly given its
    prediction (staged parity)."""
    wl = WL.CORAL
    S, D, G = wl.stages, wl.head_dim, wl.group_size
    small = WL.Workload(**{**wl.__dict__, "heads": H, "tokens": N, "layers": 2})
    xs = SY.coral_layers(small, SY.K_TENSOR, 0, N)
    _, U, W = SY.coral_predictor(small, 0)
    cfg = qvg.config(H, D, 0, 0, S, G)
    ws = qvg.alloc_workspace(cfg, N)
    Ud, Wd = to_dev(U), to_dev(W)
    Bout = torch.full((H * D * D,), -1, dtype=torch.int16, device="cuda")
    fitpred = qvg.qvg.coral_predictor(B=Bout.data_ptr(), U=Ud.data_ptr(), W=Wd.data_ptr(), rank=U.shape[1])
    xprev, xnext = to_dev(xs[0]), to_dev(xs[1])
    qvg.coral_fit_block(cfg, fitpred, xprev, xnext, N, Bout, ws)
    torch.cuda.synchronize()
    assert qvg.qvg_fit_stats(cfg, N, ws)[3] == 0
    Bg = u16(Bout).reshape(H, D, D)
    Bo, Z = oracle.coral_fit_block(xs[0], xs[1], U, W, H, D)
    bg = SY.bf16_bits_to_f32(Bg).astype(np.float64)
    scale = np.abs(Z).max(axis=(1, 2), keepdims=True)
    x = SY.bf16_bits_to_f32(xs[0]).astype(np.float64)
    kappa = np.empty((H, 1, 1))
    for h in range(H):
        Gh = x[:, h * D:(h + 1) * D].T @ x[:, h * D:(h + 1) * D]
        ev = np.linalg.eigvalsh(Gh + np.ldexp(np.trace(Gh) / D, -20) * np.eye(D))
        kappa[h] = ev[-1] / ev[0]
    tol = 2.0 ** -8 * np.abs(Z) + 2 * kappa * D * 2.0 ** -24 * scale
    assert np.all(np.abs(bg - Z) <= tol), np.max(np.abs(bg - Z) / tol)
    assert np.mean(Bg == Bo) >= 0.5, np.mean(Bg == Bo)
    # encode this layer with the fitted block; the oracle quantises with the GPU's prediction
    codes, meta, xh, pout = gpu_layer(qvg, cfg, fitpred, xprev, xnext, N)
    gp = pout.cpu().numpy()
    oc, om, oxh, _ = oracle.coral_encode_layer(xs[0], xs[1], Bg, U, W, H, D, S, G, pred_in=gp)
    np.testing.assert_array_equal(u32(codes).reshape(oc.shape), oc)
    np.testing.assert_array_equal(u32(meta).reshape(om.shape), om)
    np.testing.assert_array_equal(u16(xh), oxh)
    p64 = oracle.coral_predict(xs[0], Bg, U, W, H, D)
    assert np.all(np.abs(gp - p64) <= pred_bound(xs[0], Bg, U, W, H, D))


def test_prepared_predictor_is_bit_identical(qvg):
    """A predictor that carries its prepared U/W layout (coral_prepare_predictor)
    gives, bit for bit, what one without it gives: codes, meta, reconstruction
    and prediction of the encoder and the decoder, the refit block, and the
    Coral + SAS hybrid's outputs."""
    wl = WL.CORAL
    H, D, S, G, N = 4, wl.head_dim, wl.stages, wl.group_size, 300
    small = WL.Workload(**{**wl.__dict__, "heads": H, "tokens": N, "layers": 2, "rank": 32})
    xs = SY.coral_layers(small, SY.K_TENSOR, 0, N)
    cfg = qvg.config(H, D, 0, 0, S, G)
    B, U, W = SY.coral_predictor(small, 0)
    plain, keep = predictor(qvg, B, U, W)
    lay = torch.empty(qvg.coral_prepared_bytes(cfg), dtype=torch.uint8, device="cuda")
    qvg.coral_prepare_predictor(cfg, plain, lay)
    prepared = qvg.qvg.coral_predictor(B=plain.B, U=plain.U, W=plain.W, rank=32, prepared=lay.data_ptr())
    prev, nxt = to_dev(xs[0]), to_dev(xs[1])
    e1 = gpu_layer(qvg, cfg, plain, prev, nxt, N)
    e2 = gpu_layer(qvg, cfg, prepared, prev, nxt, N)
    for u, v in zip(e1, e2):
        assert torch.equal(u, v)
    d1 = gpu_layer(qvg, cfg, plain, prev, None, N, encode=False, codes=e1[0], meta=e1[1])
    d2 = gpu_layer(qvg, cfg, prepared, prev, None, N, encode=False, codes=e1[0], meta=e1[1])
    assert torch.equal(d1[2], d2[2]) and torch.equal(d1[3], d2[3]) and torch.equal(d1[2], e1[2])
    # the block refit (its low-rank projection uses the layout too)
    ws = qvg.alloc_workspace(cfg, N)
    outs = []
    for p in (plain, prepared):
        Bout = torch.full((H * D * D,), -1, dtype=torch.int16, device="cuda")
        fp = qvg.qvg.coral_predictor(B=Bout.data_ptr(), U=p.U, W=p.W, rank=32, prepared=p.prepared)
        qvg.coral_fit_block(cfg, fp, prev, nxt, N, Bout, ws)
        torch.cuda.synchronize()
        outs.append(Bout.clone())
    assert torch.equal(outs[0], outs[1])
    # the hybrid, both directions
    scfg = qvg.config(H, D, 16, 2, S, G)
    sws = torch.empty(qvg.coral_sas_workspace_bytes(scfg, N), dtype=torch.uint8, device="cuda")
    r1 = sas_gpu_layer(qvg, scfg, plain, prev, nxt, N, sws)
    r2 = sas_gpu_layer(qvg, scfg, prepared, prev, nxt, N, sws)
    for k in r1[0]:
        assert torch.equal(r1[0][k], r2[0][k]), k
    assert torch.equal(r1[1], r2[1]) and torch.equal(r1[2], r2[2])
    q1 = sas_gpu_layer(qvg, scfg, plain, prev, None, N, sws, bufs=r1[0])
    q2 = sas_gpu_layer(qvg, scfg, prepared, prev, None, N, sws, bufs=r1[0])
    assert torch.equal(q1[1], q2[1]) and torch.equal(q1[1], r1[1])


def test_coral_fit_block_zero_input(qvg):
    wl = WL.CORAL
    H, D, N = 2, wl.head_dim, 500
    small = WL.Workload(**{**wl.__dict__, "heads": H, "tokens": N, "layers": 2})
    _, U, W = SY.coral_predictor(small, 0)
    cfg = qvg.config(H, D, 0, 0, wl.stages, wl.group_size)
    ws = qvg.alloc_workspace(cfg, N)
    Ud, Wd = to_dev(U), to_dev(W)
    Bout = torch.full((H * D * D,), -1, dtype=torch.int16, device="cuda")
    pred = qvg.qvg.coral_predictor(B=Bout.data_ptr(), U=Ud.data_ptr(), W=Wd.data_ptr(), rank=U.shape[1])
    zeros = torch.zeros((N, H * D), dtype=torch.int16, device="cuda")
    y = to_dev(SY.coral_layers(small, SY.K_TENSOR, 0, N)[1])
    qvg.coral_fit_block(cfg, pred, zeros, y, N, Bout, ws)
    torch.cuda.synchronize()
    assert np.all(u16(Bout) == 0)


def sas_gpu_layer(qvg, cfg, pred, xprev_dev, xnext_dev, N, ws, bufs=None, want_pred=True):
    """One layer of the Coral-KV + SAS hybrid through the C ABI: encode when
    bufs is None (fresh poisoned outputs), else decode from bufs.  want_pred
    False passes no prediction buffer (the decoder then stores none)."""
    H, D, S, G, C = cfg.num_heads, cfg.head_dim, cfg.num_stages, cfg.group_size, cfg.num_clusters
    xh = torch.full((N, H * D), -1, dtype=torch.int16, device="cuda")
    pout = torch.empty((N, H * D), dtype=torch.float32, device="cuda")
    if bufs is None:
        bufs = {"codes": torch.full((S * H * N * D // 16,), -1, dtype=torch.int32, device="cuda"),
                "meta": torch.full((S * H * N * D // G,), -1, dtype=torch.int32, device="cuda"),
                "ids": torch.full((H * N,), 255, dtype=torch.uint8, device="cuda"),
                "cent": torch.full((H * C * D,), -1, dtype=torch.int16, device="cuda")}
        qvg.coral_sas_encode(cfg, pred, xprev_dev, xnext_dev, N, bufs["codes"], bufs["meta"], bufs["ids"],
                             bufs["cent"], xh, ws, pred_out=pout)
    else:
        qvg.coral_sas_decode(cfg, pred, xprev_dev, N, bufs["codes"], bufs["meta"], bufs["ids"], bufs["cent"], xh,
                             ws, pred_out=pout if want_pred else None)
    torch.cuda.synchronize()
    assert qvg.qvg_fit_stats(cfg, N, ws)[3] == 0      # no bounded wait expired
    return bufs, xh, pout


# rank 32 runs the tensor-core prediction (ragged last token tile), rank 16 the general one
@pytest.mark.parametrize("N,R,H", [(300, 32, 4), (129, 16, 4)])
def test_coral_sas_hybrid_staged_parity(qvg, oracle, N, R, H):
    """Coral-KV + SAS hybrid over three closed-loop layers: given the GPU's
    fp32 prediction, the residual's centroids, ids, codes, meta and the
    reconstruction are bit-exact against the oracle, and the decoder rebuilds
    the encoder's reconstruction exactly.  Layer 0 has no prediction."""
    wl = WL.CORAL
    D, S, G, C, T, L = wl.head_dim, wl.stages, wl.group_size, 16, 3, 3
    small = WL.Workload(**{**wl.__dict__, "heads": H, "tokens": N, "layers": L, "rank": R})
    xs = SY.coral_layers(small, SY.K_TENSOR, 0, N)
    cfg = qvg.config(H, D, C, T, S, G)
    ws = torch.empty(qvg.coral_sas_workspace_bytes(cfg, N), dtype=torch.uint8, device="cuda")
    prev = pred = keep = B = U = W = None
    for l in range(L):
        if l > 0:
            B, U, W = SY.coral_predictor(small, l - 1)
            pred, keep = predictor(qvg, B, U, W)
        bufs, xh, pout = sas_gpu_layer(qvg, cfg, pred, None if prev is None else to_dev(prev), to_dev(xs[l]), N, ws)
        gp = pout.cpu().numpy()
        if l == 0:
            assert np.all(gp == 0)
        oc, oi, ocodes, ometa, oxh, _ = oracle.coral_sas_layer(prev, xs[l], B, U, W, H, D, C, T, S, G, pred_in=gp)
        np.testing.assert_array_equal(u16(bufs["cent"]).reshape(H, C, D), oc, err_msg=f"centroids layer {l}")
        np.testing.assert_array_equal(bufs["ids"].cpu().numpy().reshape(H, N).astype(np.int32), oi,
                                      err_msg=f"ids layer {l}")
        np.testing.assert_array_equal(u32(bufs["codes"]).reshape(ocodes.shape), ocodes, err_msg=f"codes layer {l}")
        np.testing.assert_array_equal(u32(bufs["meta"]).reshape(ometa.shape), ometa, err_msg=f"meta layer {l}")
        np.testing.assert_array_equal(u16(xh), oxh, err_msg=f"reconstruction layer {l}")
        _, dxh, dp = sas_gpu_layer(qvg, cfg, pred, None if prev is None else to_dev(prev), None, N, ws, bufs=bufs)
        np.testing.assert_array_equal(u16(dxh), u16(xh))
        np.testing.assert_array_equal(dp.cpu().numpy(), gp)
        # and without a prediction buffer (nothing but x_hat stored)
        _, dxh2, _ = sas_gpu_layer(qvg, cfg, pred, None if prev is None else to_dev(prev), None, N, ws, bufs=bufs,
                                   want_pred=False)
        np.testing.assert_array_equal(u16(dxh2), u16(xh))
        prev = u16(xh)
