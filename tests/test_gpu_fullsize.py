"""Full-size parity in the launch configuration the bench times.

The CUDA path processes a whole layer of the Wan2.1-shaped and the large
workloads (token-major [N][H][D] cache, all heads in one call); sampled
(tensor, head) units are recomputed by the CPU oracle from the numpy twin of
the generator and must match bit for bit.  The cross-layer workload runs
all 16,384 tokens of every layer on the GPU and is compared on token slices.
"""
import numpy as np
import pytest
import torch

from synth import gpu as SG
from synth import synth as SY
from synth import workloads as WL
from gpu_helpers import Encoded, to_dev, u16, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _synth_lib():
    SG.build()


def run_layer(qvg, wl, tensor, layer=0):
    H, D, N = wl.heads, wl.head_dim, wl.tokens
    x = SG.mixture_layer_gpu(wl, layer, tensor, layout="nhd")          # [N][H][D]
    cfg = qvg.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size)
    enc = Encoded(qvg, cfg, N)
    ws = qvg.alloc_workspace(cfg, N)
    qvg.qvg_fit_centroids(cfg, x, N, D, H * D, None, enc["centroids"], enc["ids"], N, 0, ws)
    stats = qvg.qvg_fit_stats(cfg, N, ws)
    assert stats[3] == 0, "a k-means kernel gave up a wait"
    print(f"\n{wl.name} tensor {tensor}: {wl.lloyd_iters} Lloyd assigns re-ranked {stats[0]} of {wl.lloyd_iters * H * N} rows exactly "
          f"({stats[0] / (wl.lloyd_iters * H * N):.4f}), {stats[1]} settled in fp64")
    qvg.qvg_encode(cfg, x, N, D, H * D, enc["centroids"], 0, enc["codes"], enc["meta"], enc["ids"], N, 0, ws)
    out = torch.empty((N, H, D), dtype=torch.int16, device="cuda")
    qvg.qvg_decode(cfg, enc["codes"], enc["meta"], enc["ids"], enc["centroids"], N, 0, N, out, D, H * D)
    torch.cuda.synchronize()
    return x, enc, out


def check_heads(oracle, wl, tensor, x, enc, out, heads, layer=0):
    D, S, G, C, T = wl.head_dim, wl.stages, wl.group_size, wl.clusters, wl.lloyd_iters
    xg = u16(x)
    dec = u16(out)
    for h in heads:
        xh = SY.mixture_unit(wl, layer, tensor, h)
        np.testing.assert_array_equal(xg[:, h, :], xh, err_msg="device generator differs from numpy")
        oc, oi = oracle.fit(xh, C, T)
        np.testing.assert_array_equal(enc.centroids()[0, h], oc, err_msg=f"centroids head {h}")
        np.testing.assert_array_equal(enc.ids()[h], oi, err_msg=f"ids head {h}")
        rc, rm = oracle.prq_encode(xh, oc, oi, S, G)
        np.testing.assert_array_equal(enc.codes()[:, h], rc, err_msg=f"codes head {h}")
        np.testing.assert_array_equal(enc.meta()[:, h], rm, err_msg=f"meta head {h}")
        np.testing.assert_array_equal(dec[:, h, :], oracle.decode(rc, rm, oi, oc, G), err_msg=f"decode head {h}")


@pytest.mark.parametrize("tensor,heads", [(SY.K_TENSOR, [0, 11]), (SY.V_TENSOR, [5])])
def test_wan_layer_sampled_heads(qvg, oracle, tensor, heads):
    wl = WL.WAN
    x, enc, out = run_layer(qvg, wl, tensor)
    check_heads(oracle, wl, tensor, x, enc, out, heads)


def test_wan_layer_properties_all_heads(qvg):
    """Properties that hold for every head of the full layer: ids in range,
    every decoded value within the last stage's error bound of the input, and
    the reconstruction error well below the input variance.  Bound per
    element: s/2 (round to nearest) + 2^-9 s (fp16 rounding of the scale, x3
    levels) + 2^-11 |z| (fp16 rounding of the zero-point) + 2^-8 max(|x|,
    |x_hat|) (bf16 rounding of the output)."""
    wl = WL.WAN
    x, enc, out = run_layer(qvg, wl, SY.K_TENSOR, layer=7)
    ids = enc.ids()
    assert ids.max() < wl.clusters
    xf = x.view(torch.bfloat16).float()
    of = out.view(torch.bfloat16).float()
    meta = enc.meta()
    def per_elem(bits):
        v = torch.from_numpy(bits.astype(np.uint16).view(np.float16).astype(np.float32)).cuda()
        return v.repeat_interleave(wl.group_size, dim=-1).permute(1, 0, 2)        # [N][H][D]
    s_last, z_last = per_elem(meta[-1] & 0xFFFF), per_elem(meta[-1] >> 16)
    err = (of - xf).abs()
    bound = s_last / 2 + s_last * 2 ** -9 + z_last.abs() * 2 ** -11 + torch.maximum(xf.abs(), of.abs()) * 2 ** -8
    assert torch.all(err <= bound + 1e-6)
    rel = (err ** 2).mean() / (xf ** 2).mean()
    assert rel < 1e-3


@pytest.mark.slow
def test_large_layer_sampled_heads(qvg, oracle):
    wl = WL.LARGE
    x, enc, out = run_layer(qvg, wl, SY.V_TENSOR, layer=47)
    check_heads(oracle, wl, SY.V_TENSOR, x, enc, out, [39], layer=47)


def test_coral_full_size_token_slices(qvg, oracle):
    """All 16,384 tokens of a 4-layer chain through the device codec; the
    first and last 128 token rows come from the numpy generator and are
    compared with the oracle (staged: the oracle quantises the GPU's fp32
    prediction)."""
    wl = WL.CORAL
    H, D, S, G, N = wl.heads, wl.head_dim, wl.stages, wl.group_size, wl.tokens
    L = 4
    sl = 128
    fill = SG.coral_chain_gpu(wl, SY.K_TENSOR, n_layers=L)            # [L][N][HD] device
    a = SY.coral_layers(wl, SY.K_TENSOR, 0, sl, n_layers=L)
    b = SY.coral_layers(wl, SY.K_TENSOR, N - sl, N, n_layers=L)
    fill[:, :sl] = to_dev(a)
    fill[:, N - sl:] = to_dev(b)
    cfg = qvg.config(H, D, 0, 0, S, G)
    ws = qvg.alloc_workspace(cfg, N)
    prev = None
    for l in range(L):
        codes = torch.empty(S * H * N * D // 16, dtype=torch.int32, device="cuda")
        meta = torch.empty(S * H * N * D // G, dtype=torch.int32, device="cuda")
        xh = torch.empty((N, H * D), dtype=torch.int16, device="cuda")
        pout = torch.empty((N, H * D), dtype=torch.float32, device="cuda")
        if l == 0:
            qvg.coral_predict_encode(cfg, None, None, fill[0], N, codes, meta, xh, pout, ws)
            Bm = Um = Wm = None
        else:
            Bm, Um, Wm = SY.coral_predictor(wl, l - 1)
            Bd, Ud, Wd = SG.coral_predictor_device(wl, l - 1)
            pred = qvg.qvg.coral_predictor(B=Bd.data_ptr(), U=Ud.data_ptr(), W=Wd.data_ptr(), rank=wl.rank)
            qvg.coral_predict_encode(cfg, pred, prev, fill[l], N, codes, meta, xh, pout, ws)
        torch.cuda.synchronize()
        gc = u32(codes).reshape(S, H, N, D // 16)
        gm = u32(meta).reshape(S, H, N, D // G)
        gx = u16(xh)
        gp = pout.cpu().numpy()
        gprev = None if prev is None else u16(prev)
        for lo, src in ((0, a), (N - sl, b)):
            rows = slice(lo, lo + sl)
            pin = None if l == 0 else gp[rows]
            xprev = None if l == 0 else gprev[rows]
            oc, om, ox, _ = oracle.coral_encode_layer(xprev, src[l], Bm, Um, Wm, H, D, S, G, pred_in=pin)
            np.testing.assert_array_equal(gc[:, :, rows], oc)
            np.testing.assert_array_equal(gm[:, :, rows], om)
            np.testing.assert_array_equal(gx[rows], ox)
            if l > 0:
                p64 = oracle.coral_predict(xprev, Bm, Um, Wm, H, D)
                assert np.max(np.abs(gp[rows] - p64)) < 1e-3
        prev = xh


def test_coral_sas_full_size_decoder_rebuilds_encoder(qvg):
    """The Coral-KV + SAS hybrid at the bench's layer size (16 heads x 16,384
    tokens, C = 256, T = 4), two layers: the decoder, with and without a
    prediction buffer, rebuilds the encoder's reconstruction bit for bit and
    the same fp32 prediction, and the reconstruction is close to the input
    (relative MSE below 1e-2)."""
    wl = WL.CORAL
    H, D, S, G, N = wl.heads, wl.head_dim, wl.stages, wl.group_size, wl.tokens
    C, T, L = 256, 4, 2
    xs = SG.coral_chain_gpu(wl, SY.K_TENSOR, n_layers=L)             # [L][N][HD] device
    cfg = qvg.config(H, D, C, T, S, G)
    ws = torch.empty(qvg.coral_sas_workspace_bytes(cfg, N), dtype=torch.uint8, device="cuda")
    prev, pred = None, None
    for l in range(L):
        if l > 0:
            Bd, Ud, Wd = SG.coral_predictor_device(wl, l - 1)
            pred = qvg.qvg.coral_predictor(B=Bd.data_ptr(), U=Ud.data_ptr(), W=Wd.data_ptr(), rank=wl.rank)
        codes = torch.empty(S * H * N * D // 16, dtype=torch.int32, device="cuda")
        meta = torch.empty(S * H * N * D // G, dtype=torch.int32, device="cuda")
        ids = torch.empty(H * N, dtype=torch.uint8, device="cuda")
        cent = torch.empty(H * C * D, dtype=torch.int16, device="cuda")
        xh = torch.empty((N, H * D), dtype=torch.int16, device="cuda")
        pe = torch.empty((N, H * D), dtype=torch.float32, device="cuda")
        qvg.coral_sas_encode(cfg, pred, prev, xs[l], N, codes, meta, ids, cent, xh, ws, pred_out=pe)
        dx1 = torch.empty_like(xh)
        pd = torch.empty_like(pe)
        qvg.coral_sas_decode(cfg, pred, prev, N, codes, meta, ids, cent, dx1, ws, pred_out=pd)
        dx2 = torch.empty_like(xh)
        qvg.coral_sas_decode(cfg, pred, prev, N, codes, meta, ids, cent, dx2, ws)
        torch.cuda.synchronize()
        assert qvg.qvg_fit_stats(cfg, N, ws)[3] == 0
        assert torch.equal(dx1, xh) and torch.equal(dx2, xh), f"layer {l}"
        assert torch.equal(pd, pe), f"layer {l}"
        x = SY.bf16_bits_to_f32(u16(xs[l])).astype(np.float64)
        r = SY.bf16_bits_to_f32(u16(xh)).astype(np.float64)
        assert np.mean((x - r) ** 2) / np.mean(x ** 2) < 1e-2, f"layer {l}"
        prev = xh


def test_bench_step_on_four_streams_matches_one_stream(qvg, oracle):
    """The bench times the Wan2.1 step with its (layer, tensor) units spread
    over four streams, a workspace per stream.  Four layers of that step must
    give, unit for unit, the bytes of the same units run in order on one
    stream; one head of the last unit is checked against the oracle."""
    import bench
    wl = bench.workload("wan")
    L, H, D, N = 4, wl.heads, wl.head_dim, wl.tokens
    runs = []
    for streams in (4, 1):
        st = bench.QvgStep(qvg, wl, L, streams=streams)
        st.step()
        torch.cuda.synchronize()
        res = {(l, t): {k: st.enc[l][t][k].cpu().clone() for k in ("codes", "meta", "ids", "centroids")}
               for l in range(L) for t in (0, 1)}
        last = st.out[st.slot(L - 1, 1)].cpu().clone()
        runs.append((res, last))
        del st
        torch.cuda.empty_cache()
    (a, la), (b, lb) = runs
    for key in a:
        for k in a[key]:
            assert torch.equal(a[key][k], b[key][k]), f"unit {key}: {k} differs between four streams and one"
    assert torch.equal(la, lb), "decoded output differs between four streams and one"
    h = 3
    xh = SY.mixture_unit(wl, L - 1, 1, h)
    oc, oi = oracle.fit(xh, wl.clusters, wl.lloyd_iters)
    got = a[(L - 1, 1)]
    np.testing.assert_array_equal(got["centroids"].numpy().view(np.uint16).reshape(H, wl.clusters, D)[h], oc)
    np.testing.assert_array_equal(got["ids"].numpy().reshape(H, N)[h].astype(np.int32), oi)
