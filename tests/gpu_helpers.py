"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and
bring its buffers back as numpy arrays in the oracle's per-head layouts."""
import numpy as np
import torch


def to_dev(a):
    """numpy uint16/uint32 array -> device tensor with the same bytes."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda()
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).cuda()
    if a.dtype == np.uint8:
        return torch.from_numpy(a).cuda()
    return torch.from_numpy(a).cuda()


def u16(t):
    return t.cpu().numpy().view(np.uint16)


def u32(t):
    return t.cpu().numpy().view(np.uint32)


class Encoded:
    """Device buffers of one encoded (layer, tensor) plus numpy views."""

    def __init__(self, Q, cfg, capacity, versions=1):
        self.Q, self.cfg, self.cap, self.V = Q, cfg, capacity, versions
        self.bufs = Q.alloc_encoded(cfg, capacity, versions)
        # poison the outputs so an unwritten element cannot pass as correct
        for k in ("codes", "meta"):
            self.bufs[k].fill_(-1)
        self.bufs["ids"].fill_(255)

    def __getitem__(self, k):
        return self.bufs[k]

    def codes(self):
        c = self.cfg
        return u32(self.bufs["codes"]).reshape(c.num_stages, c.num_heads, self.cap, c.head_dim * c.bits // 32)

    def meta(self):
        c = self.cfg
        return u32(self.bufs["meta"]).reshape(c.num_stages, c.num_heads, self.cap, c.head_dim // c.group_size)

    def ids(self):
        c = self.cfg
        return self.bufs["ids"].cpu().numpy()[: c.num_heads * self.cap].reshape(c.num_heads, self.cap).astype(np.int32)

    def centroids(self):
        c = self.cfg
        n = self.V * c.num_heads * c.num_clusters * c.head_dim
        return u16(self.bufs["centroids"])[:n].reshape(self.V, c.num_heads, c.num_clusters, c.head_dim)


def run_fit_encode_decode(Q, cfg, x_dev, n, head_stride, token_stride, capacity=None, offset=0, warm=None,
                          decode_range=None):
    cap = n + offset if capacity is None else capacity
    enc = Encoded(Q, cfg, cap)
    ws = Q.alloc_workspace(cfg, n)
    if cfg.num_clusters > 0:
        Q.qvg_fit_centroids(cfg, x_dev, n, head_stride, token_stride, warm, enc["centroids"], enc["ids"], cap,
                            offset, ws)
        assert Q.qvg_fit_stats(cfg, n, ws)[3] == 0, "a k-means kernel gave up a wait"
    Q.qvg_encode(cfg, x_dev, n, head_stride, token_stride, enc["centroids"], 0, enc["codes"], enc["meta"],
                 enc["ids"], cap, offset, ws)
    b, e = decode_range if decode_range else (offset, offset + n)
    H, D = cfg.num_heads, cfg.head_dim
    out = torch.full((H, max(e - b, 0), D), -1, dtype=torch.int16, device="cuda")
    Q.qvg_decode(cfg, enc["codes"], enc["meta"], enc["ids"], enc["centroids"], cap, b, e, out, max(e - b, 0) * D, D)
    torch.cuda.synchronize()
    return enc, u16(out)
