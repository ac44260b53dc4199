"""Throughput of the KV-cache codec on one B300 (or N independent replicas).

One step = the whole hot path over one Wan2.1-1.3B-shaped cache: for each of
the 30 layers and both K and V (token-major [32760][12][128] bf16), the
per-head k-means fit (C=256, 4 Lloyd iterations), the 2-stage 2-bit PRQ
encode and the decode back to bf16.  value = bf16 KV bytes processed per
second (6.04 GB per step), inputs resident in HBM; every layer's input
(201 MB) is larger than L2.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config wan|large|stream|coral|tiny]
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV-cache 2-bit encode/decode GB/s of bf16 KV; % of B300 HBM peak"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def source_hash(*files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# The files each timed kernel is built from; a stored ncu traffic figure is
# used only while all of them are unchanged.
_CS = "kv_cache_quantization_means_b300/csrc/"
KERNEL_SOURCES = {
    "assign": [_CS + "assign_tc.cu", _CS + "tc_common.cuh", _CS + "common.cuh", _CS + "kernels.h"],
    "encode": [_CS + "prq.cu", _CS + "prq16.cuh", _CS + "common.cuh",
               _CS + "tc_common.cuh", _CS + "kernels.h"],
    "decode": [_CS + "prq_decode_tma.cu", _CS + "prq16.cuh", _CS + "common.cuh",
               _CS + "tc_common.cuh", _CS + "kernels.h"],
    "coral_predict": [_CS + "coral_tc.cu", _CS + "prq16.cuh", _CS + "tc_common.cuh", _CS + "common.cuh",
                      _CS + "kernels.h"],
}


def traffic_for(kernel, src_files):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source has not changed since it was captured; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t[kernel]
        if e["source_hash"] != source_hash(*src_files):
            return None
        return e["dram_bytes_per_launch"]
    except Exception:
        return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        self.first = 0
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # the timed region starts once the sampler is running; samples taken
            # before it (the first one) are not counted
            deadline = time.monotonic() + 3.0
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.005)
            self.first = len(self.lines)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.first:]:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 8:
                continue
            try:
                sm.append(float(p[0]))
                mx = float(p[1])
            except ValueError:
                continue
            for name, v in zip(names, p[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- workload --

def max_over_ranks(t, world, device):
    """The slowest rank's step time: each rank times its own GPU's step, and
    the job is done when the last one is."""
    if world <= 1:
        return t
    import torch
    import torch.distributed as dist
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_throughput(bytes_per_rank_step, world, t):
    """Whole-job GB/s: every rank processes its own replica of the step."""
    return bytes_per_rank_step * world / t / 1e9


def workload(name, bits=None):
    import dataclasses
    from synth import workloads as WL
    wl = WL.SHORT["wan" if name == "attn" else name]
    return wl if bits is None else dataclasses.replace(wl, bits=bits)


class QvgStep:
    """Device buffers and the launch sequence of one step of the QVG path."""

    def __init__(self, Q, wl, layers, streams=4):
        import torch
        from synth import gpu as SG
        self.Q, self.wl, self.L = Q, wl, layers
        H, D, N = wl.heads, wl.head_dim, wl.tokens
        self.cfg = Q.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size, wl.bits)
        self.x = [[SG.mixture_layer_gpu(wl, l, t, layout="nhd") for t in (0, 1)] for l in range(layers)]
        self.enc = [[Q.alloc_encoded(self.cfg, N) for _ in (0, 1)] for _ in range(layers)]
        # units run concurrently on `streams` streams, each with its own
        # workspace and decode-output buffer: unit (l, t) goes to stream
        # (2 l + t) mod streams
        self.nstreams = streams
        self.ws = [Q.alloc_workspace(self.cfg, N) for _ in range(streams)]
        self.sides = [torch.cuda.Stream() for _ in range(streams - 1)]
        self.out = [torch.empty((N, H, D), dtype=torch.int16, device="cuda") for _ in range(streams)]
        self.N, self.H, self.D = N, H, D
        self.bytes_per_step = 2 * layers * N * H * D * 2

    def fit(self, l, t):
        e, N, D, H = self.enc[l][t], self.N, self.D, self.H
        self.Q.qvg_fit_centroids(self.cfg, self.x[l][t], N, D, H * D, None, e["centroids"], e["ids"], N, 0,
                                 self.ws[self.slot(l, t)])

    def assign(self, l, t):
        e, N, D, H = self.enc[l][t], self.N, self.D, self.H
        self.Q.qvg_assign(self.cfg, self.x[l][t], N, D, H * D, e["centroids"], e["ids"], N, 0, self.ws[self.slot(l, t)])

    def encode(self, l, t):
        e, N, D, H = self.enc[l][t], self.N, self.D, self.H
        self.Q.qvg_encode(self.cfg, self.x[l][t], N, D, H * D, e["centroids"], 0, e["codes"], e["meta"], e["ids"],
                          N, 0, self.ws[self.slot(l, t)])

    def update(self, l, t):
        e, N, D, H = self.enc[l][t], self.N, self.D, self.H
        self.Q.qvg_update(self.cfg, self.x[l][t], N, D, H * D, e["ids"], N, 0, e["centroids"], self.ws[self.slot(l, t)])

    def decode(self, l, t):
        e, N, D, H = self.enc[l][t], self.N, self.D, self.H
        self.Q.qvg_decode(self.cfg, e["codes"], e["meta"], e["ids"], e["centroids"], N, 0, N,
                          self.out[self.slot(l, t)], D, H * D)

    def slot(self, l, t):
        return (2 * l + t) % self.nstreams

    def step(self):
        """Units spread over the streams: they are independent, so the small
        kernels of one run beside another's work."""
        import torch
        cur = torch.cuda.current_stream()
        streams = [cur] + self.sides
        for sd in self.sides:
            sd.wait_stream(cur)
        for l in range(self.L):
            for t in (0, 1):
                with torch.cuda.stream(streams[self.slot(l, t)]):
                    self.fit(l, t)
                    self.encode(l, t)
                    self.decode(l, t)
        for sd in self.sides:
            cur.wait_stream(sd)

    def compressed_bytes(self):
        cb, mb, ib, xb = self.Q.qvg_encoded_bytes(self.cfg, self.N, 1)
        return cb + mb + ib + xb


class CoralStep:
    """Cross-layer closed loop of the Coral-KV workload (24 layers x 16 heads x
    128 x 16,384 tokens, K and V): per tensor, layer 0 is PRQ-coded, then for
    each l the block-DPLR prediction from the reconstructed layer l is
    subtracted from layer l+1 and the residual PRQ-coded (encoder), and the
    chain is decoded back (decoder)."""

    def __init__(self, Q, wl, layers, adapted=False, sas=False, sas_clusters=256, sas_iters=4):
        import torch
        from synth import gpu as SG
        self.Q, self.wl, self.L, self.adapted, self.sas = Q, wl, layers, adapted, sas
        H, D, N, S, G = wl.heads, wl.head_dim, wl.tokens, wl.stages, wl.group_size
        self.cfg = Q.config(H, D, 0, 0, S, G)
        self.N, self.H, self.D, self.HD = N, H, D, H * D
        self.x = [SG.coral_chain_gpu(wl, t, n_layers=layers) for t in (0, 1)]        # [L][N][HD]
        self.preds, self.keep, self.layouts = [], [], []
        for l in range(layers - 1):
            B, U, W = SG.coral_predictor_device(wl, l)
            self.keep.append((B, U, W))
            p = Q.qvg.coral_predictor(B=B.data_ptr(), U=U.data_ptr(), W=W.data_ptr(), rank=wl.rank)
            # the predictor's U/W layout for the tensor cores, prepared once when it is loaded
            lay = torch.empty(Q.coral_prepared_bytes(self.cfg, wl.rank), dtype=torch.uint8, device="cuda")
            Q.coral_prepare_predictor(self.cfg, p, lay)
            p.prepared = lay.data_ptr()
            self.layouts.append(lay)
            self.preds.append(p)
        torch.cuda.synchronize()
        # adapted configuration: per tensor and layer a block refit into its own buffer
        self.fit_B, self.fit_preds = [], []
        if adapted:
            for t in (0, 1):
                bs = [torch.empty(H * D * D, dtype=torch.int16, device="cuda") for _ in range(layers - 1)]
                self.fit_B.append(bs)
                self.fit_preds.append([Q.qvg.coral_predictor(B=bs[l].data_ptr(), U=self.keep[l][1].data_ptr(),
                                                             W=self.keep[l][2].data_ptr(), rank=wl.rank,
                                                             prepared=self.layouts[l].data_ptr())
                                       for l in range(layers - 1)])
        self.codes = [[torch.empty(S * H * N * D // 16, dtype=torch.int32, device="cuda") for _ in range(layers)]
                      for _ in (0, 1)]
        self.meta = [[torch.empty(S * H * N * D // G, dtype=torch.int32, device="cuda") for _ in range(layers)]
                     for _ in (0, 1)]
        self.xh = [torch.empty((layers, N, H * D), dtype=torch.int16, device="cuda") for _ in (0, 1)]
        self.dec = [torch.empty((layers, N, H * D), dtype=torch.int16, device="cuda") for _ in (0, 1)]
        # one workspace per tensor: the K and V chains run concurrently on two streams
        self.ws = [Q.alloc_workspace(self.cfg, N) for _ in (0, 1)]
        self.side = torch.cuda.Stream()
        self.bytes_per_step = 2 * layers * N * H * D * 2
        # per tensor and direction: layer 0 (one kernel), then low-rank + predict per layer (the
        # predictors' layouts are prepared at load); adapted: + low-rank + Gram + reduce + solve per
        # encoded layer
        self.launches_per_step = 2 * (1 + 2 * (layers - 1)) * 2 + (2 * 4 * (layers - 1) if adapted else 0)
        if sas:
            # Coral-KV + SAS hybrid: the residual of every layer is k-means smoothed (C, T) and PRQ-coded
            C, T = sas_clusters, sas_iters
            self.cfg_s = Q.config(H, D, C, T, S, G)
            self.ws_s = [torch.empty(Q.coral_sas_workspace_bytes(self.cfg_s, N), dtype=torch.uint8, device="cuda")
                         for _ in (0, 1)]
            self.ids = [[torch.empty(H * N, dtype=torch.uint8, device="cuda") for _ in range(layers)] for _ in (0, 1)]
            self.cents = [[torch.empty(H * C * D, dtype=torch.int16, device="cuda") for _ in range(layers)]
                          for _ in (0, 1)]
            # encode per layer: prediction (1 kernel at layer 0, else low-rank + predict), residual,
            # k-means init + T x (assign + update), PRQ encode, decode, reconstruction;
            # decode per layer: the prediction alone, whose kernel also decodes the residual
            # and forms x_hat = bf16(pred + r_hat)
            enc = (1 + 5 + 2 * T) + (layers - 1) * (2 + 5 + 2 * T)
            dec = 1 + (layers - 1) * 2
            self.launches_per_step = 2 * (enc + dec)

    def pred(self, t, l):
        return self.fit_preds[t][l - 1] if self.adapted else self.preds[l - 1]

    def encode(self, t, l):
        prev = None if l == 0 else self.xh[t][l - 1]
        pred = None if l == 0 else self.pred(t, l)
        if self.sas:
            self.Q.coral_sas_encode(self.cfg_s, pred, prev, self.x[t][l], self.N, self.codes[t][l], self.meta[t][l],
                                    self.ids[t][l], self.cents[t][l], self.xh[t][l], self.ws_s[t])
            return
        if self.adapted and l > 0:
            self.Q.coral_fit_block(self.cfg, pred, prev, self.x[t][l], self.N, self.fit_B[t][l - 1], self.ws[t])
        self.Q.coral_predict_encode(self.cfg, pred, prev, self.x[t][l], self.N, self.codes[t][l], self.meta[t][l],
                                    self.xh[t][l], None, self.ws[t])

    def decode(self, t, l):
        prev = None if l == 0 else self.dec[t][l - 1]
        pred = None if l == 0 else self.pred(t, l)
        if self.sas:
            self.Q.coral_sas_decode(self.cfg_s, pred, prev, self.N, self.codes[t][l], self.meta[t][l],
                                    self.ids[t][l], self.cents[t][l], self.dec[t][l], self.ws_s[t])
            return
        self.Q.coral_predict_decode(self.cfg, pred, prev, self.N, self.codes[t][l], self.meta[t][l],
                                    self.dec[t][l], None, self.ws[t])

    def step(self):
        """The K chain, then the V chain.  In the adapted configuration the V
        chain runs on a second stream beside the K chain: the block refit's
        one-CTA-per-head solve leaves most SMs idle.  (The reusable
        configuration's persistent predict kernels already fill every SM, and
        two chains only compete.)"""
        import torch
        cur = torch.cuda.current_stream()
        two = self.adapted or self.sas
        if two:
            self.side.wait_stream(cur)
        for t in (0, 1):
            with torch.cuda.stream(self.side if (two and t == 1) else cur):
                for l in range(self.L):
                    self.encode(t, l)
                for l in range(self.L):
                    self.decode(t, l)
        if two:
            cur.wait_stream(self.side)


class StreamStep:
    """Streaming rollout on the Wan2.1 shape (30 layers x 12 heads x 128): 40
    steps, each appending a 3-frame chunk of 4680 tokens per layer and tensor
    (a warm-started refit every 8th chunk, assign-only otherwise) and then
    decoding the whole history of every layer, layer by layer, into one
    reused bf16 buffer.  One bench step = the whole rollout."""

    def __init__(self, Q, wl, layers):
        import torch
        from synth import gpu as SG
        self.Q, self.wl, self.L = Q, wl, layers
        H, D, N = wl.heads, wl.head_dim, wl.tokens
        self.cfg = Q.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size, wl.bits)
        self.N, self.H, self.D = N, H, D
        self.chunk, self.steps, self.every = wl.chunk_tokens, wl.steps, wl.refit_every
        self.x = [[SG.mixture_layer_gpu(wl, l, t, layout="nhd") for t in (0, 1)] for l in range(layers)]
        vmax = (self.steps + self.every - 1) // self.every
        self.caches = [[Q.make_cache(self.cfg, N, vmax, self.steps) for _ in (0, 1)] for _ in range(layers)]
        self.ws = Q.alloc_workspace(self.cfg, self.chunk)
        self.out = torch.empty((N, H, D), dtype=torch.int16, device="cuda")
        per_tok = H * D * 2
        # per (layer, tensor) and step: refit (init + T x (assign + update)) or assign, encode, chunk-table
        # update, then the history decode
        T = wl.lloyd_iters
        self.launches_per_step = 2 * layers * sum((1 + 2 * T if k % self.every == 0 else 1) + 2 + 1
                                                  for k in range(self.steps))
        self.enc_bytes = 2 * layers * N * per_tok
        self.dec_bytes = 2 * layers * per_tok * self.chunk * sum(range(1, self.steps + 1))
        self.bytes_per_step = self.enc_bytes + self.dec_bytes

    def reset(self):
        for row in self.caches:
            for c, _ in row:
                c.n_used = 0
                c.n_versions = 0
                c.n_chunks = 0

    def step(self):
        self.reset()
        H, D, ch = self.H, self.D, self.chunk
        for k in range(self.steps):
            for l in range(self.L):
                for t in (0, 1):
                    c, _ = self.caches[l][t]
                    xs = self.x[l][t][k * ch:(k + 1) * ch]
                    self.Q.qvg_append_chunk(self.cfg, c, xs, ch, D, H * D, k % self.every == 0, self.ws)
                    self.Q.qvg_decode_cache(self.cfg, c, 0, c.n_used, self.out, D, H * D)


class AttnStep:
    """Attention of one 3-frame chunk's queries over the compressed history,
    Wan2.1 shape: per layer, 12 heads x 4680 queries x 32760 keys x 128, with
    K and V of every layer fitted (C = 256, T = 4) and encoded (S = 2, G = 64)
    by the library once, outside the timed region.  A step is one
    qvg_attention_decode_staged per layer: per group of four heads the keys
    and values are decoded once into an L2-sized working buffer, then 128-query
    tiles attend to it on the tensor cores; no bf16 K/V of the layer is
    formed."""

    def __init__(self, Q, wl, layers):
        import numpy as np
        import torch
        from synth import gpu as SG
        from synth import synth as SY
        self.Q, self.wl, self.L = Q, wl, layers
        H, D, N = wl.heads, wl.head_dim, wl.tokens
        self.H, self.D, self.N, self.Nq = H, D, N, 3 * wl.frame_tokens
        self.cfg = Q.config(H, D, wl.clusters, wl.lloyd_iters, wl.stages, wl.group_size, wl.bits)
        ws = Q.alloc_workspace(self.cfg, N)
        self.enc = []
        for l in range(layers):
            pair = []
            for t in (SY.K_TENSOR, SY.V_TENSOR):
                x = SG.mixture_layer_gpu(wl, l, t, layout="nhd")
                e = Q.alloc_encoded(self.cfg, N)
                Q.qvg_fit_centroids(self.cfg, x, N, D, H * D, None, e["centroids"], e["ids"], N, 0, ws)
                Q.qvg_encode(self.cfg, x, N, D, H * D, e["centroids"], 0, e["codes"], e["meta"], e["ids"], N, 0, ws)
                pair.append((e, Q.encoded_view(e)))
            self.enc.append(pair)
        torch.cuda.synchronize()
        del ws
        q = np.stack([SY.mixture_unit(wl, 0, SY.Q_TENSOR, h, 0, self.Nq) for h in range(H)], axis=1)
        self.q = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).cuda()
        self.out = torch.empty((self.Nq, H, D), dtype=torch.float32, device="cuda")
        self.scale = float(np.float32(D ** -0.5))
        self.aws = torch.empty(Q.qvg_attention_workspace_bytes(self.cfg, N), dtype=torch.uint8, device="cuda")
        groups = (H + 3) // 4
        self.launches_per_step = layers * 2 * groups        # a staging decode and an attention kernel per group
        self.kv_bytes = 2 * H * N * D * 2                   # bf16 K + V of one layer
        self.bytes_per_step = layers * self.kv_bytes
        self.flops_per_launch = 4.0 * H * self.Nq * N * D   # Q K^T and P V

    def layer(self, l):
        (_, kv), (_, vv) = self.enc[l]
        self.Q.qvg_attention_decode_staged(self.cfg, self.q, self.Nq, self.D, self.H * self.D, kv, vv, self.N,
                                           self.N, self.scale, self.out, self.D, self.H * self.D, self.aws)

    def step(self):
        for l in range(self.L):
            self.layer(l)


def attn_config_block(wl):
    return {"workload": f"attention over the compressed {wl.name} cache: {wl.layers} layers x {wl.heads} heads, "
                        f"{3 * wl.frame_tokens} queries (one 3-frame chunk) x {wl.tokens} keys x head_dim "
                        f"{wl.head_dim}, K and V encoded with C={wl.clusters} T={wl.lloyd_iters} S={wl.stages} "
                        f"b={wl.bits} G={wl.group_size}; value counts the bf16 K+V bytes attended per second"}


def _oracle_attn_sample(args):
    """One head of the attention workload on the CPU: the oracle decodes the
    head's 32760 K and V rows and attends `nq` queries over them."""
    seed, head, nq = args
    import time as _t
    from oracle import oracle as O
    from synth import synth as SY
    wl = workload("wan")
    H, D, N, S, G, C = 1, wl.head_dim, wl.tokens, wl.stages, wl.group_size, wl.clusters
    kc, km, ki, kx = SY.random_encoding(seed + head, SY.K_TENSOR, H, N, D, S, G, C)
    vc, vm, vi, vx = SY.random_encoding(seed + head, SY.V_TENSOR, H, N, D, S, G, C)
    q = SY.mixture_unit(wl, 0, SY.Q_TENSOR, head, 0, nq)
    t0 = _t.perf_counter()
    kd = O.decode(kc[:, 0], km[:, 0], ki[0].astype("int32"), kx[0], G)
    vd = O.decode(vc[:, 0], vm[:, 0], vi[0].astype("int32"), vx[0], G)
    O.attention(q, kd, vd, D ** -0.5)
    return _t.perf_counter() - t0


def cpu_baseline_attn(nq=512):
    """The oracle on this host's cores: one head per process (decode of the
    head's K and V, then attention of nq of the chunk's 4680 queries), all in
    parallel; the bytes credited are the head's bf16 K + V times nq / 4680."""
    import multiprocessing as mp
    from oracle import oracle as O
    O.build()
    wl = workload("wan")
    n = host_workers()
    ctx = mp.get_context("spawn")
    # one BLAS thread per worker, so that `cores` counts the threads used
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    os.environ.update({k: "1" for k in saved})
    try:
        with ctx.Pool(n) as pool:
            walls = pool.map(_oracle_attn_sample, [(wl.seed, h % wl.heads, nq) for h in range(n)])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    wall = max(walls)
    nbytes = n * 2 * wl.tokens * wl.head_dim * 2 * nq / (3 * wl.frame_tokens)
    return {"value": nbytes / wall / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{n} heads, each: oracle decode of {wl.tokens} K and V rows + fp64 attention of {nq} of the "
                      f"{3 * wl.frame_tokens} queries; one head per process, all concurrent; slowest {wall:.1f} s"}


def time_fn(fn, reps, stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(reps):
        fn()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps / 1e3


def graph_time(fn, reps):
    """Device time of fn() per call: fn is captured once in a CUDA graph and
    the graph is replayed, so host-side launch cost does not enter."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    torch.cuda.synchronize()
    return time_fn(g.replay, reps)


def kernel_rooflines(st, peaks, reps=3):
    """Average per-launch device time of each kernel family over all
    (layer, tensor) units, and its algorithmic bytes or flops per launch."""
    hbm, tf_burst, tf_sus, kind = peaks
    wl, L = st.wl, st.L
    elems = st.N * st.H * st.D                      # one tensor of one layer
    S, G, C, D = wl.stages, wl.group_size, wl.clusters, wl.head_dim
    code_b = S * (wl.bits / 8 + 4 / G)              # code + meta bytes per element
    id_b = 1 / D
    units = [(l, t) for l in range(L) for t in (0, 1)]

    def over_units(f):
        return lambda: [f(l, t) for (l, t) in units]

    t_dec = graph_time(over_units(st.decode), reps) / len(units)
    t_enc = graph_time(over_units(st.encode), reps) / len(units)
    t_asg = graph_time(over_units(st.assign), reps) / len(units)
    t_upd = graph_time(over_units(st.update), reps) / len(units)
    t_fit = graph_time(over_units(st.fit), 1) / len(units)
    dec_bytes = elems * (code_b + id_b + 2)
    enc_bytes = elems * (2 + id_b + code_b)
    asg_flops = 2.0 * C * elems                     # token-by-centroid distance GEMM
    upd_bytes = elems * (2 + id_b)                  # reads every token once (plus ids)
    out = {
        "decode": {"bound": "hbm", "achieved": dec_bytes / t_dec / 1e9, "peak": hbm, "unit": "GB/s",
                   "time_us": t_dec * 1e6, "algorithmic_bytes": dec_bytes},
        "encode": {"bound": "hbm", "achieved": enc_bytes / t_enc / 1e9, "peak": hbm, "unit": "GB/s",
                   "time_us": t_enc * 1e6, "algorithmic_bytes": enc_bytes},
        "assign": {"bound": "tensor", "achieved": asg_flops / t_asg / 1e12, "peak": tf_burst, "unit": "TFLOP/s",
                   "time_us": t_asg * 1e6, "algorithmic_flops": asg_flops},
        "update": {"bound": "hbm", "achieved": upd_bytes / t_upd / 1e9, "peak": hbm, "unit": "GB/s",
                   "time_us": t_upd * 1e6, "algorithmic_bytes": upd_bytes},
        "fit": {"bound": "tensor", "achieved": wl.lloyd_iters * asg_flops / t_fit / 1e12, "peak": tf_sus,
                "unit": "TFLOP/s", "time_us": t_fit * 1e6},
    }
    for v in out.values():
        v["frac"] = v["achieved"] / v["peak"]
        v["peak_kind"] = kind
    out["decode"]["bf16_gbs"] = elems * 2 / t_dec / 1e9
    out["encode"]["bf16_gbs"] = elems * 2 / t_enc / 1e9
    return out


# ------------------------------------------------------------ CPU oracle --

def _oracle_unit(args):
    name, bits, layer, tensor, head = args
    import time as _t
    from oracle import oracle as O
    from synth import synth as SY
    wl = workload(name, bits)
    x = SY.mixture_unit(wl, layer, tensor, head)
    t0 = _t.perf_counter()
    cent, ids = O.fit(x, wl.clusters, wl.lloyd_iters)
    codes, meta = O.prq_encode(x, cent, ids, wl.stages, wl.group_size, wl.bits)
    O.decode(codes, meta, ids, cent, wl.group_size, wl.bits)
    return _t.perf_counter() - t0, x.size * 2


def host_workers():
    """Worker processes of the CPU oracle: one per core this process may run
    on (both the cpu_baseline leg and --impl reference use this count)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(name, bits=None):
    """The oracle as it stands on this host's cores: one (layer, tensor, head)
    unit per worker process, one process per core, all units in parallel;
    throughput = bf16 bytes of the units / wall time."""
    import multiprocessing as mp
    from oracle import oracle as O
    O.build()
    wl = workload(name, bits)
    n = host_workers()
    units = [(name, bits, (i * 7) % wl.layers, i % 2, (i * 5) % wl.heads) for i in range(n)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(n) as pool:
        res = pool.map(_oracle_unit, units)
    wall = max(r[0] for r in res)
    nbytes = sum(r[1] for r in res)
    return {"value": nbytes / wall / 1e9, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"{n} (layer, tensor, head) units of {wl.name} ({wl.tokens} tokens x {wl.head_dim}), "
                      f"fit T={wl.lloyd_iters} + encode + decode, one unit per process, all concurrent; "
                      f"slowest unit {wall:.1f} s (timed inside the worker, generation excluded)"}


# ------------------------------------------------------------------ main --

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    name = args.config
    wl = workload(name, args.bits)
    t0 = time.perf_counter()
    per_step = []
    # the same sample, on the same number of cores, as the cpu_baseline leg
    base = (lambda: cpu_baseline_attn()) if name == "attn" else (lambda: cpu_baseline(name, bits=args.bits))
    for _ in range(args.warmup):
        base()
    for _ in range(args.steps):
        per_step.append(base())
    wall = time.perf_counter() - t0
    v = statistics.median(p["value"] for p in per_step)
    cb = dict(per_step[-1])
    cb["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / max(1, args.steps + args.warmup) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32",
            "data": "synthetic", "config": attn_config_block(wl) if name == "attn" else config_block(wl, args),
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def config_block(wl, args):
    return {"workload": f"{wl.name}: {wl.layers} layers x {wl.heads} heads x head_dim {wl.head_dim} x {wl.tokens} "
                        f"tokens, K and V bf16 token-major; C={wl.clusters} T={wl.lloyd_iters} S={wl.stages} "
                        f"b={wl.bits} G={wl.group_size}",
            "layers": wl.layers, "heads": wl.heads, "head_dim": wl.head_dim, "tokens": wl.tokens,
            "clusters": wl.clusters, "lloyd_iters": wl.lloyd_iters, "stages": wl.stages, "group_size": wl.group_size,
            "bits": wl.bits, "streams": getattr(args, "streams", 1),
            "l2": "inputs larger than L2 (one layer's K or V is %.0f MB)" % (wl.tokens * wl.heads * wl.head_dim * 2 / 1e6),
            "parallelism": f"replicas x{args.gpus}"}


def run_aux(args, Q, wl, peaks, world, rank, local):
    """Bench line of the cross-layer (coral) or streaming (stream) workload:
    whole step captured in one CUDA graph, device-timed; the roofline is that
    of the step's dominant kernel family."""
    import torch
    hbm = peaks[0]
    if args.config == "coral":
        st = CoralStep(Q, wl, wl.layers, adapted=args.adapted, sas=args.sas)
    elif args.config == "attn":
        st = AttnStep(Q, wl, wl.layers)
    else:
        st = StreamStep(Q, wl, wl.layers)
    st.step()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    with ClockSampler(local) as clk:
        t_step = graph_time(st.step, max(1, args.steps))
    if world > 1:
        dist.barrier()
    if args.config == "coral":
        L, n = st.L, st.N * st.HD
        t_dec = graph_time(lambda: [st.decode(t, l) for t in (0, 1) for l in range(L)], 3) / (2 * L)
        dec_bytes = n * (2 + wl.stages * (2 / 8 + 4 / wl.group_size) + 2)   # read x_hat_l, codes+meta; write x_hat_l+1
        if args.sas:
            dec_bytes += n / wl.head_dim                                      # + the residual's cluster ids
        dom = {"kernel": ("coral+sas decode (prediction, residual decode and reconstruction in one kernel per "
                          "layer, after the low-rank projection)" if args.sas
                          else "coral decode (low-rank + predict/decode per layer)"), "bound": "hbm",
               "achieved": dec_bytes / t_dec / 1e9, "peak": hbm, "unit": "GB/s", "time_us": t_dec * 1e6}
        cfgb = {"workload": f"{wl.name}: {wl.layers} layers x {wl.heads} heads x head_dim {wl.head_dim} x {wl.tokens} "
                            f"tokens, K and V, closed-loop block-DPLR (rank {wl.rank}; U/W layouts prepared at load) + PRQ S={wl.stages} G={wl.group_size}, "
                            "encode chain + decode chain" + ("; adapted: each layer's block predictors refit "
                                                              "(least squares) before it is encoded" if args.adapted else "")
                            + ("; hybrid: each layer's bf16 prediction residual k-means smoothed (C=256 T=4) before "
                               "its PRQ" if args.sas else "")}
    elif args.config == "attn":
        t_att = graph_time(lambda: st.layer(0), 3)
        dom = {"kernel": "attn_stage_kernel + attn_fa_kernel (per 4-head group: K/V decoded once into an L2-sized "
                         "buffer; tcgen05 S=QK^T and O+=PV in tensor memory)",
               "bound": "tensor", "achieved": st.flops_per_launch / t_att / 1e12, "peak": peaks[1],
               "unit": "TFLOP/s", "time_us": t_att * 1e6}
        cfgb = attn_config_block(wl)
    else:
        c = st.caches[-1][-1][0]
        lens = [st.chunk * (k + 1) for k in range(st.steps)]
        t_dec = graph_time(lambda: [Q.qvg_decode_cache(st.cfg, c, 0, n, st.out, st.D, st.H * st.D) for n in lens], 3)
        el = sum(lens) * st.H * st.D
        b = el * (wl.stages * (wl.bits / 8 + 4 / wl.group_size) + 1 / wl.head_dim + 2)
        dom = {"kernel": "prq_decode (versioned history decode)", "bound": "hbm", "achieved": b / t_dec / 1e9,
               "peak": hbm, "unit": "GB/s", "time_us": t_dec / st.steps * 1e6}
        cfgb = {"workload": f"{wl.name}: {wl.layers} layers x {wl.heads} heads x head_dim {wl.head_dim}; {wl.steps} steps "
                            f"of {wl.chunk_tokens}-token chunks (refit every {wl.refit_every}, C={wl.clusters} "
                            f"T={wl.lloyd_iters}), full-history decode of every layer per step; value counts bf16 bytes "
                            f"encoded ({st.enc_bytes / 1e9:.1f} GB) + decoded ({st.dec_bytes / 1e9:.1f} GB)"}
    dom["frac"] = dom["achieved"] / dom["peak"]
    dom["traffic"] = None
    dom["peak_kind"] = peaks[3]
    t_step = max_over_ranks(t_step, world, "cuda")
    value = job_throughput(st.bytes_per_step, world, t_step)
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfgb, "roofline": dom,
            "cpu_baseline": None, "e2e": None, "gpu_launches": st.launches_per_step * args.steps, "cuda_graph": True,
            "clocks": clk.summary()}
    if args.config == "attn":
        line["dtype"] = "bf16 x bf16 -> f32"
        if rank == 0 and not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline_attn()
    if rank == 0:
        print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="wan", choices=["wan", "large", "coral", "stream", "attn"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--streams", type=int, default=4,
                    help="QVG workloads: (layer, tensor) units run concurrently on this many streams")
    ap.add_argument("--adapted", action="store_true",
                    help="coral: refit each layer's block predictors for the current video before encoding it")
    ap.add_argument("--sas", action="store_true",
                    help="coral: Coral-KV + SAS hybrid, k-means smoothing of each layer's prediction residual")
    ap.add_argument("--bits", type=int, default=None, choices=[2, 4],
                    help="code width of the QVG workloads (default: the workload's, 2)")
    args = ap.parse_args()
    if args.bits is not None and args.config == "coral" and args.bits != 2:
        ap.error("the cross-layer codec uses 2-bit codes")
    if args.sas and (args.config != "coral" or args.adapted):
        ap.error("--sas is a mode of the coral workload (and not combined with --adapted)")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            dist.barrier()

    import __graft_entry__ as GE
    GE.build()
    import kv_cache_quantization_means_b300 as Q
    Q.load()
    wl = workload(args.config, args.bits)
    peaks = load_peaks()
    if args.config in ("coral", "stream", "attn"):
        return run_aux(args, Q, wl, peaks, world, rank, local)
    layers = wl.layers if args.config == "wan" else 2
    st = QvgStep(Q, wl, layers, streams=args.streams)
    torch.cuda.synchronize()

    graph = None
    if not args.no_graph:
        st.step()                                   # eager warm-up (sets kernel attributes)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            st.step()
        run = graph.replay
    else:
        run = st.step
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    barrier()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier()
        s = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(args.steps):
            run()
        b.record(s)
        torch.cuda.synchronize()
        barrier()
    t = max_over_ranks(a.elapsed_time(b) / 1e3 / args.steps, world, "cuda")
    value = job_throughput(st.bytes_per_step, world, t)
    # per (layer, tensor): init + T x (assign, update) + encode + decode
    launches_per_step = 2 * layers * (1 + wl.lloyd_iters * 2 + 2)

    roof = kernel_rooflines(st, peaks)

    # end to end through the C ABI with host buffers: for every (layer,
    # tensor), qvg_compress_host copies its K or V from pinned host memory,
    # fits, encodes and decodes it, and copies the compressed stream back.
    e2e = None
    if not args.no_e2e:
        units = [(l, t) for l in range(layers) for t in (0, 1)]
        host_x = {u: st.x[u[0]][u[1]].cpu().pin_memory() for u in units}
        host_out = {u: torch.empty(st.compressed_bytes(), dtype=torch.uint8).pin_memory() for u in units}
        comp = torch.cuda.current_stream()
        # one qvg_compress_host call per unit (host->device copy, fit, encode,
        # decode, device->host copy of the encoding, all on the unit's stream),
        # units dealt round-robin to three streams so that one unit's copies
        # overlap another's kernels
        lanes = [torch.cuda.Stream() for _ in range(3)]
        N, D, H = st.N, st.D, st.H

        def e2e_step():
            for ln in lanes:
                ln.wait_stream(comp)                  # nothing starts before the timed region
            for i, u in enumerate(units):
                l, t = u
                e, ln = st.enc[l][t], lanes[i % len(lanes)]
                Q.qvg_compress_host(st.cfg, host_x[u], st.x[l][t], N, D, H * D, None, e["centroids"], e["ids"],
                                    e["codes"], e["meta"], st.out[i % len(lanes)], host_out[u], st.ws[i % len(lanes)],
                                    stream=ln)
            for ln in lanes:
                comp.wait_stream(ln)                  # the timed region ends after the last read-back
        e2e_step()
        te = time_fn(e2e_step, max(1, min(args.steps, 3)))
        te = max_over_ranks(te, world, "cuda")
        e2e = {"value": job_throughput(st.bytes_per_step, world, te), "unit": "GB/s",
               "h2d_bytes_per_step": st.bytes_per_step, "d2h_bytes_per_step": 2 * layers * st.compressed_bytes(),
               "pipelined": "qvg_compress_host per (layer, tensor): host->device copy, fit, encode, decode, "
                            "device->host copy of the encoding; units round-robin on three streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(args.config, bits=args.bits)

    dom = max(("assign", "decode", "encode"), key=lambda k: roof[k]["time_us"])
    src = {k: KERNEL_SOURCES[k] for k in ("assign", "decode", "encode")}
    rl = {k: roof[dom][k] for k in ("bound", "achieved", "peak", "unit", "frac")}
    rl["kernel"] = dom
    rl["traffic"] = traffic_for(dom, src[dom])
    rl["peak_kind"] = roof[dom]["peak_kind"]
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded mixture-of-Gaussians bf16 KV cache)",
            "config": config_block(wl, args), "roofline": rl,
            "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                        for k, v in roof.items()},
            "hbm_frac_of_nominal_8tbs": {k: roof[k]["achieved"] / 8000.0 for k in ("decode", "encode")},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(), "cuda_graph": graph is not None}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
