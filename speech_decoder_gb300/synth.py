"""Seeded synthetic inputs for the Qwen3-style speech decoder.

This module only *generates data*: the shapes of the five workloads, random
weights, prompt token ids and audio-encoder rows.  It holds no step of the
decoder's arithmetic, so both the plain CPU oracle (``oracle/``) and the CUDA
path can draw their inputs from it without sharing any method code.

Weights follow the random-init recipe of the workloads: every matrix and the
token embedding is N(0, 0.02); RMSNorm weights are 1 for the tiny block and
1 + 0.1*N(0,1) elsewhere (so that a dropped norm weight shows up in parity).
For bf16 workloads each value is rounded to the nearest bf16 (ties to even)
*here*, so both sides read exactly the same numbers.

Prompt layout follows the pages' audio injection (prefix token rows |
encoder rows | suffix token rows): the canary-qwen layout of 9 prefix ids and
5 suffix ids around 138 encoder rows (transcribe.cpp src/arch/canary_qwen/
model.cpp, prompt construction), the qwen3_asr 9 + 6 layout
(transcribe-cpp-sys src/arch/qwen3_asr/model.cpp, build_prompt_tokens).
Encoder rows are N(0, 1).
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "ModelSpec", "Prompt", "Workload", "WORKLOADS", "model_weights", "prompt_inputs",
    "round_bf16", "bf16_bits", "workload", "small_spec",
]


@dataclasses.dataclass(frozen=True)
class ModelSpec:
    """Shape and numeric format of a Qwen3-style decoder."""
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    weight_dtype: str = "bf16"      # "bf16", "e4m3" (bf16 in; the library rounds rows to e4m3) or "f32"
    kv_dtype: str = "f16"           # "f16" or "f32"
    norm_init: str = "jitter"       # "ones" or "jitter"
    w_std: float = 0.02


@dataclasses.dataclass(frozen=True)
class Prompt:
    """One utterance: prefix ids | n_audio encoder rows | suffix ids."""
    prefix_len: int
    n_audio: int
    suffix_len: int

    @property
    def T(self) -> int:
        return self.prefix_len + self.n_audio + self.suffix_len


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    model: ModelSpec
    prompts: tuple          # tuple[Prompt, ...]; batch = len(prompts)
    steps: int              # greedy dec_step calls after the prefill
    seed: int = 0
    eos_id: int = -1

    @property
    def batch(self) -> int:
        return len(self.prompts)


QWEN3_0_6B = ModelSpec("qwen3-0.6b-shape", 28, 1024, 16, 8, 128, 3072, 151936)
QWEN3_1_7B = ModelSpec("qwen3-1.7b-shape", 28, 2048, 16, 8, 128, 6144, 151936)
TINY = ModelSpec("tiny-block", 1, 256, 4, 2, 64, 768, 1024, weight_dtype="f32",
                 kv_dtype="f32", norm_init="ones")


def _batch32_prompts(seed: int = 0) -> tuple:
    rng = np.random.default_rng([seed, 4032])
    n_audio = rng.integers(50, 751, size=32)
    return tuple(Prompt(9, int(n), 6) for n in n_audio)


WORKLOADS = {
    "tiny": Workload("tiny", TINY, (Prompt(0, 16, 0),), steps=8),
    "qwen3-0.6b-t153": Workload("qwen3-0.6b-t153", QWEN3_0_6B, (Prompt(10, 138, 5),), steps=64),
    "qwen3-1.7b-t152": Workload("qwen3-1.7b-t152", QWEN3_1_7B, (Prompt(9, 138, 5),), steps=256),
    "qwen3-1.7b-b32": Workload("qwen3-1.7b-b32", QWEN3_1_7B, _batch32_prompts(), steps=256),
    "qwen3-1.7b-t8015": Workload("qwen3-1.7b-t8015", QWEN3_1_7B, (Prompt(9, 8000, 6),), steps=128),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def small_spec(**kw) -> ModelSpec:
    """A reduced model for fast tests (defaults: 2 layers, GQA group 2)."""
    base = dict(name="small", n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64,
                ffn=512, vocab=1000)
    base.update(kw)
    return ModelSpec(**base)


# ---------------------------------------------------------------- bf16 helpers
def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), in place; returns a."""
    assert a.dtype == np.float32 and a.flags.c_contiguous
    u = a.view(np.uint32)
    u += np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    u &= np.uint32(0xFFFF0000)
    return a


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """The bf16 bit patterns of float32 values that are already bf16-exact."""
    assert a.dtype == np.float32
    return (np.ascontiguousarray(a).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------- weights
_TENSORS = ("attn_norm", "q", "k", "v", "o", "q_norm", "k_norm", "ffn_norm", "gate", "up", "down")


def _shape(spec: ModelSpec, name: str) -> tuple:
    H, nq, nkv, d, F = spec.hidden, spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.ffn
    return {
        "attn_norm": (H,), "ffn_norm": (H,), "q_norm": (d,), "k_norm": (d,),
        "q": (nq * d, H), "k": (nkv * d, H), "v": (nkv * d, H), "o": (H, nq * d),
        "gate": (F, H), "up": (F, H), "down": (H, F),
        "embed": (spec.vocab, H), "final_norm": (H,),
    }[name]


def _gen(spec: ModelSpec, seed: int, layer: int, name: str) -> np.ndarray:
    # One independent stream per (seed, layer, tensor): generation order and
    # thread count never change the values.
    tid = (_TENSORS + ("embed", "final_norm")).index(name)
    rng = np.random.default_rng([seed, layer + 1, tid, 7919])
    shape = _shape(spec, name)
    if name.endswith("norm"):
        if spec.norm_init == "ones":
            a = np.ones(shape, np.float32)
        else:
            a = (1.0 + 0.1 * rng.standard_normal(shape, dtype=np.float32)).astype(np.float32)
    else:
        a = rng.standard_normal(shape, dtype=np.float32)
        a *= np.float32(spec.w_std)
    if spec.weight_dtype in ("bf16", "e4m3"):
        round_bf16(a)
    return a


def model_weights(spec: ModelSpec, seed: int = 0, threads: int = 16) -> dict:
    """Random weights in the HF [out, in] layout, float32 arrays.

    Returns {"embed": [V,H], "final_norm": [H], "layers": [ {name: array} ]}.
    Values are bf16-exact when spec.weight_dtype is "bf16" or "e4m3".
    """
    jobs = [(-1, "embed"), (-1, "final_norm")]
    jobs += [(l, n) for l in range(spec.n_layers) for n in _TENSORS]
    with ThreadPoolExecutor(max(1, threads)) as ex:
        arrays = list(ex.map(lambda j: _gen(spec, seed, j[0], j[1]), jobs))
    out = {"embed": arrays[0], "final_norm": arrays[1], "layers": []}
    k = 2
    for _ in range(spec.n_layers):
        out["layers"].append(dict(zip(_TENSORS, arrays[k:k + len(_TENSORS)])))
        k += len(_TENSORS)
    return out


# ---------------------------------------------------------------- prompts
def prompt_inputs(spec: ModelSpec, prompt: Prompt, seed: int = 0, item: int = 0) -> dict:
    """Token ids and encoder rows of one utterance.

    Returns {"ids": int32 [prefix_len + suffix_len], "audio": float32 [n_audio, H],
    "prefix_len": int}.  ids[:prefix_len] precede the audio rows and
    ids[prefix_len:] follow them.
    """
    rng = np.random.default_rng([seed, 1000 + item, 31])
    ids = rng.integers(0, spec.vocab, size=prompt.prefix_len + prompt.suffix_len).astype(np.int32)
    audio = rng.standard_normal((prompt.n_audio, spec.hidden), dtype=np.float32)
    return {"ids": ids, "audio": audio, "prefix_len": prompt.prefix_len}
