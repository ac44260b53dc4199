"""B300-native KV-cache codec: Quant VideoGen (k-means smoothing + progressive
2-bit residual quantisation) and Coral-KV cross-layer residual coding, as
hand-written sm_103a CUDA kernels behind the C ABI in include/qvg.h."""
from .qvg import *  # noqa: F401,F403
from .qvg import load, QvgError, config, alloc_encoded, alloc_workspace, make_cache, EXPORTS  # noqa: F401
