"""The allocation-free Coral encode (coral_predict_encode_static).

Some callers cannot allocate device memory or hand the library a workspace:
a runtime whose allocator owns every byte of device memory, a plugin that
must keep a fixed footprint, or code that may not call cudaMalloc where the
encode happens.  For them the library keeps the encode's only scratch (the
low-rank projection, 64 floats per token, at most 16,384 tokens) in a fixed
device array of its own.

This checks, through the C ABI, that two calls in a row of the
allocation-free entry point give exactly what the workspace entry point gives
on the same inputs (codes, scales/zero-points and reconstruction bit for bit,
the fp32 prediction too), and that a size beyond the built-in scratch is
refused on the host.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from synth import synth as SY
from synth import workloads as WL
from gpu_helpers import to_dev, u16, u32

pytestmark = pytest.mark.gpu


def _predictor(qvg, wl, layer):
    B, U, W = SY.coral_predictor(wl, layer)
    dev = [to_dev(a) for a in (B, U, W)]
    p = qvg.qvg.coral_predictor(B=dev[0].data_ptr(), U=dev[1].data_ptr(), W=dev[2].data_ptr(), rank=U.shape[1])
    return p, dev


def _outputs(cfg, N):
    H, D, S, G = cfg.num_heads, cfg.head_dim, cfg.num_stages, cfg.group_size
    return (torch.full((S * H * N * D // 16,), -1, dtype=torch.int32, device="cuda"),
            torch.full((S * H * N * D // G,), -1, dtype=torch.int32, device="cuda"),
            torch.full((N, H * D), -1, dtype=torch.int16, device="cuda"),
            torch.full((N, H * D), float("nan"), dtype=torch.float32, device="cuda"))


def test_static_scratch_encode_matches_workspace_encode(qvg):
    wl = WL.CORAL
    H, D, S, G, N = 4, wl.head_dim, wl.stages, wl.group_size, 1000
    small = WL.Workload(**{**wl.__dict__, "heads": H, "tokens": N, "layers": 3})
    xs = SY.coral_layers(small, SY.V_TENSOR, 0, N)            # [3][N][H*D] bf16 bits
    cfg = qvg.config(H, D, 0, 0, S, G)
    ws = qvg.alloc_workspace(cfg, N)
    x = [to_dev(a) for a in xs]
    # layer 0 (no prediction) gives the previous reconstruction of layer 1
    c0, m0, xh0, _ = _outputs(cfg, N)
    qvg.coral_predict_encode(cfg, None, None, x[0], N, c0, m0, xh0, None, ws)
    prev = xh0
    for layer in (1, 2):                                       # two calls in a row
        pred, keep = _predictor(qvg, small, layer - 1)
        ref = _outputs(cfg, N)
        qvg.coral_predict_encode(cfg, pred, prev, x[layer], N, ref[0], ref[1], ref[2], ref[3], ws)
        got = _outputs(cfg, N)
        qvg.coral_predict_encode_static(cfg, pred, prev, x[layer], N, got[0], got[1], got[2], got[3])
        torch.cuda.synchronize()
        np.testing.assert_array_equal(u32(got[0]), u32(ref[0]), err_msg=f"codes, layer {layer}")
        np.testing.assert_array_equal(u32(got[1]), u32(ref[1]), err_msg=f"meta, layer {layer}")
        np.testing.assert_array_equal(u16(got[2]), u16(ref[2]), err_msg=f"reconstruction, layer {layer}")
        np.testing.assert_array_equal(got[3].cpu().numpy(), ref[3].cpu().numpy(), err_msg=f"prediction, layer {layer}")
        prev = ref[2]


def test_static_scratch_rejects_oversized_calls(qvg):
    H, D, S, G = 4, 128, 2, 64
    cfg = qvg.config(H, D, 0, 0, S, G)
    N = 16385
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    pred = qvg.qvg.coral_predictor(B=dummy.data_ptr(), U=dummy.data_ptr(), W=dummy.data_ptr(), rank=32)
    with pytest.raises(qvg.QvgError) as ei:
        qvg.coral_predict_encode_static(cfg, pred, dummy, dummy, N, dummy, dummy, dummy, None)
    assert ei.value.status == qvg.QVG_ERR_CAPACITY


def test_static_scratch_encode_at_its_token_limit(qvg):
    """At the cross-layer workload's own shape -- 16 heads of 128 channels and
    16,384 tokens, the most the built-in scratch takes -- the allocation-free
    encode still gives exactly what the workspace entry point gives, on two
    layers in a row, and leaves the device error word clear."""
    from synth import gpu as SG
    wl = WL.CORAL
    H, D, S, G, N = wl.heads, wl.head_dim, wl.stages, wl.group_size, wl.tokens
    assert N == 16384
    cfg = qvg.config(H, D, 0, 0, S, G)
    xs = SG.coral_chain_gpu(wl, SY.V_TENSOR, n_layers=3)     # [3][N][H*D] bf16 bits, on the device
    ws = qvg.alloc_workspace(cfg, N)
    qvg.qvg_device_error(clear=True)
    prev = xs[0]
    for layer in (1, 2):
        B, U, W = SG.coral_predictor_device(wl, layer - 1)
        pred = qvg.qvg.coral_predictor(B=B.data_ptr(), U=U.data_ptr(), W=W.data_ptr(), rank=wl.rank)
        ref = _outputs(cfg, N)
        qvg.coral_predict_encode(cfg, pred, prev, xs[layer], N, ref[0], ref[1], ref[2], None, ws)
        got = _outputs(cfg, N)
        qvg.coral_predict_encode_static(cfg, pred, prev, xs[layer], N, got[0], got[1], got[2], None)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref[0]), f"codes, layer {layer}"
        assert torch.equal(got[1], ref[1]), f"meta, layer {layer}"
        assert torch.equal(got[2], ref[2]), f"reconstruction, layer {layer}"
        prev = ref[2]
    assert qvg.qvg_device_error() == (qvg.QVG_OK, 0)
