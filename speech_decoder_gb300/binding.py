"""Python binding of libdec.so: argument marshalling only.

Every step of the decoder runs in the library's CUDA kernels; this module
allocates the device workspace through PyTorch, passes pointers and sizes,
and converts status codes into exceptions.  There is no fallback path: if
the library is missing, construction fails.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, byref, c_char_p, c_float, c_int32, c_int64, c_size_t, c_void_p

import numpy as np

from . import synth

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdec.so")

DEC_OK, DEC_ERR_INVALID_ARG, DEC_ERR_OOM, DEC_ERR_INPUT_TOO_LONG = 0, 1, 2, 3
DEC_ERR_OUTPUT_TRUNCATED, DEC_ERR_CUDA, DEC_ERR_STATE, DEC_ERR_DEVICE = 4, 5, 6, 7
DEC_BF16, DEC_F32, DEC_F16, DEC_E4M3 = 0, 1, 2, 3

EXPORTS = [
    "dec_workspace_size", "dec_create", "dec_destroy", "dec_reset", "dec_prefill", "dec_prefill_chunk", "dec_prefill_ids",
    "dec_prefill_batch", "dec_prefill_ids_batch", "dec_step", "dec_step_batch", "dec_generate", "dec_generate_batch",
    "dec_debug_logits", "dec_set_dumps", "dec_debug_dump", "dec_launch_count", "dec_last_timings",
    "dec_last_error", "dec_status_string", "dec_profile_kernel", "dec_attn_decode_scratch_size",
    "dec_attn_decode", "dec_attn_decode_noalloc", "dec_debug_gemm", "dec_perception_project",
    "dec_quantize_e4m3_rows", "dec_decode_budget",
]


class dec_hparams(ctypes.Structure):
    _fields_ = [("n_layers", c_int32), ("hidden", c_int32), ("n_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("ffn", c_int32), ("vocab", c_int32), ("rms_eps", c_float),
                ("rope_theta", c_float), ("max_ctx", c_int32), ("max_batch", c_int32),
                ("max_tokens", c_int32), ("max_new", c_int32), ("eos_id", c_int32),
                ("weight_dtype", c_int32), ("kv_dtype", c_int32)]


_LAYER_FIELDS = ("attn_norm", "q", "k", "v", "o", "q_norm", "k_norm", "ffn_norm", "gate", "up", "down")


class dec_layer_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in _LAYER_FIELDS]


class dec_weights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("final_norm", c_void_p), ("layers", POINTER(dec_layer_weights))]


class DecError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None


def load_library():
    """Load libdec.so and declare its signatures (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    H = c_void_p
    sig = {
        "dec_workspace_size": ([POINTER(dec_hparams), POINTER(c_size_t)], c_int32),
        "dec_create": ([POINTER(dec_hparams), POINTER(dec_weights), c_void_p, c_size_t, c_void_p,
                        POINTER(c_void_p)], c_int32),
        "dec_destroy": ([H], None),
        "dec_reset": ([H], c_int32),
        "dec_prefill": ([H, c_void_p, c_int32, c_int32, POINTER(c_int32)], c_int32),
        "dec_prefill_chunk": ([H, c_void_p, c_int32, c_int32, c_int32, POINTER(c_int32)], c_int32),
        "dec_prefill_ids": ([H, c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int32, POINTER(c_int32)],
                            c_int32),
        "dec_prefill_batch": ([H, c_void_p, c_void_p, c_int32, c_int32, c_void_p], c_int32),
        "dec_prefill_ids_batch": ([H, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p],
                                  c_int32),
        "dec_step": ([H, c_int32, POINTER(c_int32)], c_int32),
        "dec_step_batch": ([H, c_void_p, c_void_p, c_void_p], c_int32),
        "dec_generate": ([H, c_int32, c_void_p, POINTER(c_int32)], c_int32),
        "dec_generate_batch": ([H, c_int32, c_void_p, c_void_p, c_void_p], c_int32),
        "dec_debug_logits": ([H, c_void_p, c_int32], c_int32),
        "dec_set_dumps": ([H, c_int32], c_int32),
        "dec_debug_dump": ([H, c_char_p, c_void_p, c_size_t], c_int32),
        "dec_launch_count": ([H, POINTER(c_int64)], c_int32),
        "dec_last_timings": ([H, POINTER(c_float), POINTER(c_float)], c_int32),
        "dec_profile_kernel": ([H, c_int32, c_int32, POINTER(c_float), POINTER(ctypes.c_double)], c_int32),
        "dec_attn_decode_scratch_size": ([c_int32, c_int32, c_int32, c_int32, POINTER(c_size_t)], c_int32),
        "dec_attn_decode": ([c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_int32, c_int32,
                             c_int32, c_int32, c_void_p, c_void_p, c_size_t, c_void_p], c_int32),
        "dec_attn_decode_noalloc": ([c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_int32,
                                     c_int32, c_int32, c_int32, c_void_p, c_void_p], c_int32),
        "dec_debug_gemm": ([c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int32, c_void_p,
                            c_int32, c_int32, c_int32, c_void_p, c_size_t, c_void_p], c_int32),
        "dec_perception_project": ([c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                                    c_size_t, c_void_p], c_int32),
        "dec_quantize_e4m3_rows": ([c_void_p, c_int64, c_int32, c_void_p, c_void_p, c_void_p, c_void_p], c_int32),
        "dec_decode_budget": ([c_int32, c_int32, c_int32, c_int32, POINTER(c_int32)], c_int32),
        "dec_last_error": ([H], c_char_p),
        "dec_status_string": ([c_int32], c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def hparams_for(spec: "synth.ModelSpec", *, max_ctx: int, max_batch: int = 1, max_tokens: int | None = None,
                max_new: int = 256, eos_id: int = -1) -> dec_hparams:
    return dec_hparams(
        n_layers=spec.n_layers, hidden=spec.hidden, n_heads=spec.n_heads, n_kv_heads=spec.n_kv_heads,
        head_dim=spec.head_dim, ffn=spec.ffn, vocab=spec.vocab, rms_eps=spec.rms_eps,
        rope_theta=spec.rope_theta, max_ctx=max_ctx, max_batch=max_batch,
        max_tokens=max_tokens if max_tokens is not None else max_ctx, max_new=max_new, eos_id=eos_id,
        weight_dtype={"bf16": DEC_BF16, "e4m3": DEC_E4M3, "f32": DEC_F32}[spec.weight_dtype],
        kv_dtype=DEC_F16 if spec.kv_dtype == "f16" else DEC_F32)


def workspace_size(hp: dec_hparams) -> int:
    lib = load_library()
    n = c_size_t()
    st = lib.dec_workspace_size(byref(hp), byref(n))
    if st != DEC_OK:
        raise DecError(st, "unsupported hyper-parameters")
    return n.value


def _host_f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def decode_budget(n_audio: int, T_prompt: int, ceiling: int, floor_new: int = 256) -> int:
    """dec_decode_budget: the generation budget of a run (raises DecError)."""
    lib = load_library()
    out = c_int32()
    st = lib.dec_decode_budget(int(n_audio), int(T_prompt), int(floor_new), int(ceiling), byref(out))
    if st != DEC_OK:
        raise DecError(st, lib.dec_status_string(st).decode())
    return out.value


class Decoder:
    """One decoder instance on one CUDA device (owns its workspace tensor)."""

    def __init__(self, spec, weights: dict, *, max_ctx: int, max_batch: int = 1, max_tokens: int | None = None,
                 max_new: int = 256, eos_id: int = -1, device: str = "cuda:0"):
        import torch
        self.torch = torch
        self.lib = load_library()
        self.spec = spec
        self.hp = hparams_for(spec, max_ctx=max_ctx, max_batch=max_batch, max_tokens=max_tokens,
                              max_new=max_new, eos_id=eos_id)
        self.device = torch.device(device)
        size = workspace_size(self.hp)
        self.workspace = torch.empty(size, dtype=torch.uint8, device=self.device)
        # a dedicated stream: the library captures CUDA graphs on it, which the
        # legacy default stream does not allow
        self.stream = torch.cuda.Stream(device=self.device)
        bf16 = spec.weight_dtype in ("bf16", "e4m3")
        keep = []

        def host(a):
            arr = synth.bf16_bits(a) if bf16 else _host_f32(a)
            arr = np.ascontiguousarray(arr)
            keep.append(arr)
            return arr.ctypes.data

        layers = (dec_layer_weights * spec.n_layers)()
        for i, L in enumerate(weights["layers"]):
            for n in _LAYER_FIELDS:
                setattr(layers[i], n, host(L[n]))
        w = dec_weights(embed=host(weights["embed"]), final_norm=host(weights["final_norm"]), layers=layers)
        handle = c_void_p()
        with torch.cuda.device(self.device):
            st = self.lib.dec_create(byref(self.hp), byref(w), c_void_p(self.workspace.data_ptr()), size,
                                     c_void_p(self.stream.cuda_stream), byref(handle))
        del keep
        if st != DEC_OK:
            raise DecError(st, f"dec_create failed: {self._name(st)}")
        self.h = handle

    # ------------------------------------------------------------ helpers
    def _name(self, st):
        return self.lib.dec_status_string(st).decode()

    def _check(self, st, allow=(DEC_OK,)):
        if st not in allow:
            msg = self.lib.dec_last_error(self.h).decode() if getattr(self, "h", None) else ""
            raise DecError(st, f"{self._name(st)}: {msg}")
        return st

    def _rows(self, a):
        """(pointer, on_device, keepalive) of float32 rows from numpy or torch."""
        t = self.torch
        if isinstance(a, t.Tensor):
            assert a.dtype == t.float32 and a.is_contiguous()
            if a.is_cuda:
                # order the library's stream after the work that produced `a`
                self.stream.wait_stream(t.cuda.current_stream(a.device))
            return a.data_ptr(), int(a.is_cuda), a
        arr = _host_f32(a)
        return arr.ctypes.data, 0, arr

    # ------------------------------------------------------------ API
    def prefill(self, embeds) -> int:
        p, dev, keep = self._rows(embeds)
        tok = c_int32()
        self._check(self.lib.dec_prefill(self.h, p, int(embeds.shape[0]), dev, byref(tok)))
        return tok.value

    def prefill_chunk(self, embeds, final: bool = False):
        """Next rows of a chunked prompt; returns the prompt's first token on
        the final chunk, None before it."""
        p, dev, keep = self._rows(embeds)
        tok = c_int32()
        self._check(self.lib.dec_prefill_chunk(self.h, p, int(embeds.shape[0]), dev, int(bool(final)), byref(tok)))
        return tok.value if final else None

    def prefill_ids(self, ids, audio, prefix_len: int) -> int:
        """ids and audio both on the device (torch CUDA tensors) or both on the
        host (numpy arrays or torch CPU tensors, pinned or not)."""
        t = self.torch
        p, dev, keep = self._rows(audio)
        if dev:
            ids_t = ids if isinstance(ids, t.Tensor) else t.from_numpy(np.ascontiguousarray(ids, np.int32))
            ids_t = ids_t.to(device=self.device, dtype=t.int32).contiguous()
            self.stream.wait_stream(t.cuda.current_stream(self.device))
            ip, n_ids = ids_t.data_ptr(), ids_t.numel()
        elif isinstance(ids, t.Tensor):
            ids_t = ids.to(t.int32).contiguous()
            ip, n_ids = ids_t.data_ptr(), ids_t.numel()
        else:
            ids_t = np.ascontiguousarray(ids, dtype=np.int32)
            ip, n_ids = ids_t.ctypes.data, ids_t.size
        tok = c_int32()
        self._check(self.lib.dec_prefill_ids(self.h, ip, n_ids, p, int(audio.shape[0]), prefix_len, dev,
                                             byref(tok)))
        return tok.value

    def prefill_ids_batch(self, ids_list, audio_list, prefix_lens, on_device: bool = False) -> np.ndarray:
        """Ragged batch of (ids, encoder rows, prefix_len) items, assembled on the device."""
        t = self.torch
        cu_ids = np.zeros(len(ids_list) + 1, np.int32)
        cu_ids[1:] = np.cumsum([len(i) for i in ids_list])
        cu_au = np.zeros(len(audio_list) + 1, np.int32)
        cu_au[1:] = np.cumsum([int(a.shape[0]) for a in audio_list])
        pre = np.ascontiguousarray(prefix_lens, dtype=np.int32)
        ids = np.concatenate([np.asarray(i, np.int32) for i in ids_list]).astype(np.int32)
        audio = np.concatenate([np.asarray(a, np.float32) for a in audio_list]).astype(np.float32)
        if on_device:
            ids_t = t.from_numpy(ids).to(self.device)
            au_t = t.from_numpy(audio).to(self.device)
            self.stream.wait_stream(t.cuda.current_stream(self.device))
            ip, ap, keep = ids_t.data_ptr(), au_t.data_ptr(), (ids_t, au_t)
        else:
            ip, ap, keep = ids.ctypes.data, audio.ctypes.data, (ids, audio)
        out = np.zeros(len(ids_list), np.int32)
        self._check(self.lib.dec_prefill_ids_batch(self.h, ip, cu_ids.ctypes.data, ap, cu_au.ctypes.data,
                                                   pre.ctypes.data, len(ids_list), int(on_device),
                                                   out.ctypes.data))
        return out

    def prefill_ids_batch_ptr(self, ids_ptr, cu_ids, audio_ptr, cu_audio, prefix_lens, on_device: int) -> np.ndarray:
        """Same, with caller-owned data pointers (device or pinned host)."""
        cu_ids = np.ascontiguousarray(cu_ids, np.int32)
        cu_audio = np.ascontiguousarray(cu_audio, np.int32)
        pre = np.ascontiguousarray(prefix_lens, np.int32)
        out = np.zeros(len(pre), np.int32)
        self._check(self.lib.dec_prefill_ids_batch(self.h, ids_ptr, cu_ids.ctypes.data, audio_ptr,
                                                   cu_audio.ctypes.data, pre.ctypes.data, len(pre), on_device,
                                                   out.ctypes.data))
        return out

    def prefill_batch(self, embeds_list) -> np.ndarray:
        lens = [int(e.shape[0]) for e in embeds_list]
        cu = np.zeros(len(lens) + 1, np.int32)
        cu[1:] = np.cumsum(lens)
        if isinstance(embeds_list[0], self.torch.Tensor):
            cat = self.torch.cat(list(embeds_list)).contiguous()
        else:
            cat = np.concatenate([_host_f32(e) for e in embeds_list])
        return self.prefill_concat(cat, cu)

    def prefill_concat(self, cat, cu: np.ndarray) -> np.ndarray:
        cu = np.ascontiguousarray(cu, dtype=np.int32)
        p, dev, keep = self._rows(cat)
        out = np.zeros(len(cu) - 1, np.int32)
        self._check(self.lib.dec_prefill_batch(self.h, p, cu.ctypes.data, len(cu) - 1, dev, out.ctypes.data))
        return out

    def step(self, token: int) -> int:
        nxt = c_int32()
        self._check(self.lib.dec_step(self.h, int(token), byref(nxt)))
        return nxt.value

    def step_batch(self, tokens, active=None) -> np.ndarray:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        act = None if active is None else np.ascontiguousarray(active, dtype=np.uint8)
        out = np.zeros(len(tokens), np.int32)
        self._check(self.lib.dec_step_batch(self.h, tokens.ctypes.data, None if act is None else act.ctypes.data,
                                            out.ctypes.data))
        return out

    def generate(self, max_new: int):
        out = np.zeros(max_new, np.int32)
        n = c_int32()
        st = self._check(self.lib.dec_generate(self.h, max_new, out.ctypes.data, byref(n)),
                         allow=(DEC_OK, DEC_ERR_OUTPUT_TRUNCATED))
        return [int(v) for v in out[:n.value]], st == DEC_ERR_OUTPUT_TRUNCATED

    def generate_batch(self, max_new: int, n_seq: int):
        out = np.zeros((n_seq, max_new), np.int32)
        n = np.zeros(n_seq, np.int32)
        tr = np.zeros(n_seq, np.int32)
        self._check(self.lib.dec_generate_batch(self.h, max_new, out.ctypes.data, n.ctypes.data, tr.ctypes.data))
        return [([int(v) for v in out[b, :n[b]]], bool(tr[b])) for b in range(n_seq)]

    def logits(self, rows: int = 1) -> np.ndarray:
        out = np.zeros((rows, self.spec.vocab), np.float32)
        self._check(self.lib.dec_debug_logits(self.h, out.ctypes.data, rows))
        return out

    def set_dumps(self, on: bool):
        self._check(self.lib.dec_set_dumps(self.h, int(on)))

    def dump(self, name: str, shape) -> np.ndarray:
        out = np.zeros(shape, np.float32)
        self._check(self.lib.dec_debug_dump(self.h, name.encode(), out.ctypes.data, out.size))
        return out

    def launch_count(self) -> int:
        n = c_int64()
        self._check(self.lib.dec_launch_count(self.h, byref(n)))
        return n.value

    def timings(self):
        a, b = c_float(), c_float()
        self._check(self.lib.dec_last_timings(self.h, byref(a), byref(b)))
        return a.value, b.value

    def profile_kernel(self, op: int, iters: int):
        """(mean ms per launch, algorithmic bytes per launch) of one kernel family."""
        ms, nb = c_float(), ctypes.c_double()
        self._check(self.lib.dec_profile_kernel(self.h, op, iters, byref(ms), byref(nb)))
        return ms.value, nb.value

    def reset(self):
        self._check(self.lib.dec_reset(self.h))

    def close(self):
        if getattr(self, "h", None):
            self.lib.dec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
