"""Small fixed cases of the codec's kernels, for timing and for profilers.

    python -m kv_cache_quantization_means_b300.profile_case unit [time]
    python -m kv_cache_quantization_means_b300.profile_case coral [time]
    python -m kv_cache_quantization_means_b300.profile_case coral_fit [time]
    python -m kv_cache_quantization_means_b300.profile_case coral_sas [time]
    python -m kv_cache_quantization_means_b300.profile_case attn [time]

`unit` runs one (layer, tensor) of the Wan2.1-shaped cache (12 heads x 32760
tokens x 128, C = 256, T = 4, S = 2, G = 64): a fit, then one more assign,
update, encode and decode.  `attn` runs the attention over a compressed history, the tensor-core
(staged) entry point and the in-CTA fused one.  `coral` runs one cross-layer layer (16 heads x
16384 tokens x 128, rank 32, S = 2, G = 64): encode then decode, and checks
that both rebuild the same x_hat.  Without `time` each kernel runs once (the
form to put under a profiler); with `time` each call is replayed from a CUDA
graph and its mean device time printed.  Inputs come from the seeded
synthetic generators.
"""
import sys

import torch

from . import qvg as Q
from synth import gpu as SG
from synth import workloads as WL


def _graph_time_us(f, reps=20, inner=10):
    f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(inner):
            f()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps / inner * 1e3


def unit_case(timed):
    wl = WL.WAN
    H, D, N = wl.heads, wl.head_dim, wl.tokens
    cfg = Q.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size)
    x = SG.mixture_layer_gpu(wl, 0, 1, layout="nhd")
    e = Q.alloc_encoded(cfg, N)
    ws = Q.alloc_workspace(cfg, N)
    out = torch.empty((N, H, D), dtype=torch.int16, device="cuda")
    calls = {
        "fit": lambda: Q.qvg_fit_centroids(cfg, x, N, D, H * D, None, e["centroids"], e["ids"], N, 0, ws),
        "assign": lambda: Q.qvg_assign(cfg, x, N, D, H * D, e["centroids"], e["ids"], N, 0, ws),
        "update": lambda: Q.qvg_update(cfg, x, N, D, H * D, e["ids"], N, 0, e["centroids"], ws),
        "encode": lambda: Q.qvg_encode(cfg, x, N, D, H * D, e["centroids"], 0, e["codes"], e["meta"], e["ids"],
                                       N, 0, ws),
        "decode": lambda: Q.qvg_decode(cfg, e["codes"], e["meta"], e["ids"], e["centroids"], N, 0, N, out, D,
                                       H * D),
    }
    for f in calls.values():
        f()
    torch.cuda.synchronize()
    stats = Q.qvg_fit_stats(cfg, N, ws)
    assert stats[3] == 0, stats
    print("re-rank stats (rows re-ranked, exact, channel-order fp64, error word):", stats)
    if timed:
        for name in ("assign", "update", "encode", "decode", "fit"):
            print(f"{name:8s} {_graph_time_us(calls[name]):9.1f} us")


def coral_case(timed):
    wl = WL.CORAL
    H, D, N, S, G = wl.heads, wl.head_dim, wl.tokens, wl.stages, wl.group_size
    cfg = Q.config(H, D, 0, 0, S, G)
    xs = SG.coral_chain_gpu(wl, 0, n_layers=2)
    B, U, W = SG.coral_predictor_device(wl, 0)
    pred = Q.coral_predictor(B=B.data_ptr(), U=U.data_ptr(), W=W.data_ptr(), rank=wl.rank)
    codes = torch.empty(S * H * N * D // 16, dtype=torch.int32, device="cuda")
    meta = torch.empty(S * H * N * D // G, dtype=torch.int32, device="cuda")
    xh = torch.empty((N, H * D), dtype=torch.int16, device="cuda")
    dec = torch.empty((N, H * D), dtype=torch.int16, device="cuda")
    ws = Q.alloc_workspace(cfg, N)
    enc = lambda: Q.coral_predict_encode(cfg, pred, xs[0], xs[1], N, codes, meta, xh, None, ws)
    dcd = lambda: Q.coral_predict_decode(cfg, pred, xs[0], N, codes, meta, dec, None, ws)
    enc()
    dcd()
    torch.cuda.synchronize()
    assert torch.equal(xh, dec), "encoder and decoder reconstructions differ"
    assert Q.qvg_fit_stats(cfg, N, ws)[3] == 0
    if timed:
        el = N * H * D
        # algorithmic bytes per element: encode reads x_hat_l and x_{l+1},
        # writes x_hat_{l+1}, S stages of 2-bit codes and one 4-byte scale/zero
        # word per G elements and stage
        for name, f, byt in (("encode", enc, 6.0 + S * (0.25 + 4.0 / G)), ("decode", dcd, 4.0 + S * (0.25 + 4.0 / G))):
            t = _graph_time_us(f)
            print(f"{name:8s} {t:9.1f} us   {el * byt / t / 1e3:8.1f} GB/s algorithmic")


def coral_fit_case(timed):
    """The adapted configuration's block refit on one Coral layer pair."""
    wl = WL.CORAL
    H, D, N, S, G = wl.heads, wl.head_dim, wl.tokens, wl.stages, wl.group_size
    cfg = Q.config(H, D, 0, 0, S, G)
    xs = SG.coral_chain_gpu(wl, 0, n_layers=2)
    _, U, W = SG.coral_predictor_device(wl, 0)
    B = torch.empty(H * D * D, dtype=torch.int16, device="cuda")
    pred = Q.coral_predictor(B=B.data_ptr(), U=U.data_ptr(), W=W.data_ptr(), rank=wl.rank)
    ws = Q.alloc_workspace(cfg, N)
    fit = lambda: Q.coral_fit_block(cfg, pred, xs[0], xs[1], N, B, ws)
    fit()
    torch.cuda.synchronize()
    assert Q.qvg_fit_stats(cfg, N, ws)[3] == 0
    if timed:
        print(f"fit      {_graph_time_us(fit):9.1f} us")


def coral_sas_case(timed):
    """One layer of the Coral-KV + SAS hybrid (C = 256, T = 4 on the residual):
    encode then decode, checking that both rebuild the same x_hat."""
    wl = WL.CORAL
    H, D, N, S, G = wl.heads, wl.head_dim, wl.tokens, wl.stages, wl.group_size
    cfg = Q.config(H, D, 256, 4, S, G)
    xs = SG.coral_chain_gpu(wl, 0, n_layers=2)
    B, U, W = SG.coral_predictor_device(wl, 0)
    pred = Q.coral_predictor(B=B.data_ptr(), U=U.data_ptr(), W=W.data_ptr(), rank=wl.rank)
    codes = torch.empty(S * H * N * D // 16, dtype=torch.int32, device="cuda")
    meta = torch.empty(S * H * N * D // G, dtype=torch.int32, device="cuda")
    ids = torch.empty(H * N, dtype=torch.uint8, device="cuda")
    cent = torch.empty(H * 256 * D, dtype=torch.int16, device="cuda")
    xh = torch.empty((N, H * D), dtype=torch.int16, device="cuda")
    dec = torch.empty((N, H * D), dtype=torch.int16, device="cuda")
    ws = torch.empty(Q.coral_sas_workspace_bytes(cfg, N), dtype=torch.uint8, device="cuda")
    enc = lambda: Q.coral_sas_encode(cfg, pred, xs[0], xs[1], N, codes, meta, ids, cent, xh, ws)
    dcd = lambda: Q.coral_sas_decode(cfg, pred, xs[0], N, codes, meta, ids, cent, dec, ws)
    enc()
    dcd()
    torch.cuda.synchronize()
    assert torch.equal(xh, dec), "encoder and decoder reconstructions differ"
    assert Q.qvg_fit_stats(cfg, N, ws)[3] == 0
    if timed:
        for name, f in (("encode", enc), ("decode", dcd)):
            print(f"{name:8s} {_graph_time_us(f):9.1f} us")


def attn_case(timed):
    """One layer of attention over the compressed Wan2.1 cache: 12 heads, a
    3-frame chunk of 4680 queries over 32760 keys (K and V fitted with C = 256,
    T = 4 and encoded with S = 2, G = 64 by the library first)."""
    import numpy as np
    from synth import synth as SY
    wl = WL.WAN
    H, D, N, Nq = wl.heads, wl.head_dim, wl.tokens, 3 * wl.frame_tokens
    cfg = Q.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size)
    ws = Q.alloc_workspace(cfg, N)
    views, keep = [], []
    for t in (SY.K_TENSOR, SY.V_TENSOR):
        x = SG.mixture_layer_gpu(wl, 0, t, layout="nhd")
        e = Q.alloc_encoded(cfg, N)
        Q.qvg_fit_centroids(cfg, x, N, D, H * D, None, e["centroids"], e["ids"], N, 0, ws)
        Q.qvg_encode(cfg, x, N, D, H * D, e["centroids"], 0, e["codes"], e["meta"], e["ids"], N, 0, ws)
        keep.append(e)
        views.append(Q.encoded_view(e))
    q = np.stack([SY.mixture_unit(wl, 0, SY.Q_TENSOR, h, 0, Nq) for h in range(H)], axis=1)
    qd = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).cuda()
    out = torch.empty((Nq, H, D), dtype=torch.float32, device="cuda")
    scale = float(np.float32(D ** -0.5))
    aws = torch.empty(Q.qvg_attention_workspace_bytes(cfg, N), dtype=torch.uint8, device="cuda")
    calls = {
        "staged": lambda: Q.qvg_attention_decode_staged(cfg, qd, Nq, D, H * D, views[0], views[1], N, N, scale, out,
                                                        D, H * D, aws),
        "fused": lambda: Q.qvg_attention_decode(cfg, qd, Nq, D, H * D, views[0], views[1], N, N, scale, out, D, H * D),
    }
    for f in calls.values():
        f()
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    if timed:
        for name, f in calls.items():
            t = _graph_time_us(f, reps=5, inner=3)
            print(f"attention ({name}) {t:9.1f} us   {4.0 * H * Nq * N * D / t / 1e6:8.1f} TFLOP/s   "
                  f"{2 * H * N * D * 2 / t / 1e3:8.1f} GB/s of bf16 K+V attended")


def main(argv):
    case = argv[1] if len(argv) > 1 else "unit"
    timed = len(argv) > 2 and argv[2] == "time"
    {"unit": unit_case, "coral": coral_case, "coral_fit": coral_fit_case, "coral_sas": coral_sas_case,
     "attn": attn_case}[case](timed)


if __name__ == "__main__":
    main(sys.argv)
