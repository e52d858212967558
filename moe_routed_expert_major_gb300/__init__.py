"""GB300 routed-expert MoE over MXFP4 weights: a C-ABI CUDA library (libtfx_moe.so,
sm_103a) and its thin Python binding (``tfx``)."""
from . import tfx  # noqa: F401
