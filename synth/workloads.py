"""Synthetic workload definitions: shapes and generator parameters only.

These are the five cache shapes the codec is exercised on.  They stand in for
the caches of the pages' host models (a Wan2.1 self-forcing stack, long
LongCat/HY-WorldPlay rollouts, MAGI-1 for the cross-layer predictor), none of
which is available here: every tensor is drawn from the seeded generator in
``synth.synth``.  Nothing in this module does any of the codec's arithmetic.
"""
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layers: int
    heads: int
    head_dim: int
    tokens: int              # tokens per layer (for streaming: the final history length)
    frame_tokens: int        # tokens per latent frame (drift step)
    centers: int             # mixture components per (layer, tensor, head)
    noise_std: float
    drift_std: float
    outlier_channels: int    # key channels scaled (K only)
    outlier_factor: float
    # codec parameters
    clusters: int            # C (0 = no smoothing)
    lloyd_iters: int         # T
    stages: int              # S
    bits: int
    group_size: int          # G
    # streaming
    chunk_tokens: int = 0
    steps: int = 0
    refit_every: int = 0
    # cross-layer predictor
    rank: int = 0
    next_noise_std: float = 0.0
    extra: dict = field(default_factory=dict)

    @property
    def elems_per_layer(self):
        """K + V elements of one layer."""
        return 2 * self.heads * self.tokens * self.head_dim


TINY = Workload(
    name="tiny", seed=1000, layers=1, heads=2, head_dim=64, tokens=1560,
    frame_tokens=1560, centers=8, noise_std=0.1, drift_std=0.0,
    outlier_channels=2, outlier_factor=8.0,
    clusters=16, lloyd_iters=3, stages=2, bits=2, group_size=64)

WAN = Workload(
    name="wan2.1-1.3b", seed=1001, layers=30, heads=12, head_dim=128, tokens=32760,
    frame_tokens=1560, centers=64, noise_std=0.15, drift_std=0.02,
    outlier_channels=4, outlier_factor=10.0,
    clusters=256, lloyd_iters=4, stages=2, bits=2, group_size=64)

STREAM = Workload(
    name="streaming-wan", seed=1002, layers=30, heads=12, head_dim=128, tokens=187200,
    frame_tokens=1560, centers=64, noise_std=0.15, drift_std=0.02,
    outlier_channels=4, outlier_factor=10.0,
    clusters=256, lloyd_iters=4, stages=2, bits=2, group_size=64,
    chunk_tokens=4680, steps=40, refit_every=8)

LARGE = Workload(
    name="large", seed=1003, layers=48, heads=40, head_dim=128, tokens=81920,
    frame_tokens=4096, centers=128, noise_std=0.15, drift_std=0.02,
    outlier_channels=8, outlier_factor=12.0,
    clusters=256, lloyd_iters=3, stages=3, bits=2, group_size=128)

CORAL = Workload(
    name="coral-blockdplr", seed=1004, layers=24, heads=16, head_dim=128, tokens=16384,
    frame_tokens=16384, centers=64, noise_std=0.15, drift_std=0.0,
    outlier_channels=0, outlier_factor=1.0,
    clusters=0, lloyd_iters=0, stages=2, bits=2, group_size=64,
    rank=32, next_noise_std=0.05)

ALL = {w.name: w for w in (TINY, WAN, STREAM, LARGE, CORAL)}
SHORT = {"tiny": TINY, "wan": WAN, "stream": STREAM, "large": LARGE, "coral": CORAL}
