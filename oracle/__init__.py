"""Plain fp64 CPU oracle of the decoder hot path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
import this package; the CUDA library never does.
"""
from .decoder import (Oracle, argmax_lowest, assemble_prompt, attention, greedy, linear,
                      perception_projection, rms_norm, rope_neox, silu, swiglu_ffn)

__all__ = ["Oracle", "argmax_lowest", "assemble_prompt", "attention", "greedy", "linear",
           "perception_projection", "rms_norm", "rope_neox", "silu", "swiglu_ffn"]
