"""Plain fp64 CPU oracle of the decoder hot path (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
import this package; the CUDA library never does.
"""
from .decoder import (Oracle, argmax_lowest, assemble_prompt, attention, decode_budget, greedy, linear,
                      perception_projection, rms_norm, rope_neox, silu, swiglu_ffn)
from .e4m3 import e4m3_decode, e4m3_round, e4m3_weights, quantize_rows, row_scales

__all__ = ["Oracle", "argmax_lowest", "assemble_prompt", "attention", "decode_budget", "greedy", "linear",
           "perception_projection", "rms_norm", "rope_neox", "silu", "swiglu_ffn",
           "e4m3_decode", "e4m3_round", "e4m3_weights", "quantize_rows", "row_scales"]
