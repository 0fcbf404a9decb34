"""GB300-native single-GPU MoE layer forward (routing -> FP8 quant -> FC1 +
SwiGLU -> FC2 -> combine) behind the C ABI of include/megamoe.h."""
from . import binding
from .layer import MegaMoELayer, sf_atom_rows

__all__ = ["binding", "MegaMoELayer", "sf_atom_rows"]
