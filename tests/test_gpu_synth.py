"""The device generator writes the same bytes as the numpy generator."""
import numpy as np
import pytest

from synth import gpu as SG
from synth import synth as SY
from synth import workloads as WL
from gpu_helpers import u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,layer,tensor,tb,te", [
    ("tiny", 0, 0, 0, 1560), ("tiny", 0, 1, 17, 1000), ("wan2.1-1.3b", 3, 0, 30000, 32760),
    ("large", 5, 0, 40000, 41000), ("streaming-wan", 2, 1, 180000, 187200),
])
def test_gpu_generator_matches_numpy(name, layer, tensor, tb, te):
    SG.build()
    wl = WL.ALL[name]
    for layout in ("hnd", "nhd"):
        g = u16(SG.mixture_layer_gpu(wl, layer, tensor, tok_begin=tb, tok_end=te, layout=layout))
        if layout == "nhd":
            g = g.transpose(1, 0, 2)
        for h in sorted({0, wl.heads - 1}):
            np.testing.assert_array_equal(g[h], SY.mixture_unit(wl, layer, tensor, h, tb, te))
