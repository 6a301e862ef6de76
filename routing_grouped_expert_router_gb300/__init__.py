"""GB300-native (sm_103a) MoE FFN layer: router, dispatch, SwiGLU GroupedGEMM
experts and combine, forward and backward, behind a C ABI."""
from . import configs, metrics, synth  # noqa: F401
