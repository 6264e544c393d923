"""The C-ABI library builds, loads, and exports every symbol include/dec.h
declares.  Host-side validation runs without a GPU; no kernel is launched."""
import ctypes
import os
import re

import pytest

from speech_decoder_gb300 import binding, build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dec_[a-z0-9_]+)\s*\(", src)))


def test_header_matches_binding_list():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.dec_status_string(0) == b"DEC_OK"
    assert lib.dec_status_string(3) == b"DEC_ERR_INPUT_TOO_LONG"


def _hp(**kw):
    spec = synth.QWEN3_1_7B
    hp = binding.hparams_for(spec, max_ctx=1024, max_batch=32, max_tokens=24576)
    for k, v in kw.items():
        setattr(hp, k, v)
    return hp


def test_workspace_size_and_validation(lib):
    n = ctypes.c_size_t()
    assert lib.dec_workspace_size(ctypes.byref(_hp()), ctypes.byref(n)) == 0
    # weights 3.44 GB + KV 28 layers x 8 heads x 32768 slots x 128 x 2 B x 2
    assert n.value > 3.44e9 + 3.7e9
    for bad in (dict(head_dim=96), dict(n_heads=12, n_kv_heads=8), dict(ffn=1000), dict(hidden=1000),
                dict(max_batch=0), dict(max_batch=65), dict(max_ctx=200, max_new=256), dict(eos_id=151936),
                dict(weight_dtype=binding.DEC_BF16, kv_dtype=binding.DEC_F32), dict(n_layers=0)):
        assert lib.dec_workspace_size(ctypes.byref(_hp(**bad)), ctypes.byref(n)) == binding.DEC_ERR_INVALID_ARG, bad


def test_null_arguments_rejected(lib):
    out = ctypes.c_void_p()
    assert lib.dec_create(None, None, None, 0, None, ctypes.byref(out)) == binding.DEC_ERR_INVALID_ARG
    assert lib.dec_workspace_size(None, None) == binding.DEC_ERR_INVALID_ARG
    assert lib.dec_reset(None) == binding.DEC_ERR_INVALID_ARG
    assert lib.dec_step(None, 0, None) == binding.DEC_ERR_INVALID_ARG


def test_decode_budget_matches_oracle_reading(lib):
    """dec_decode_budget is host arithmetic: compare it with the oracle's
    reading of the page's budget on a grid, and its status codes with the
    oracle's rejections."""
    import oracle as O
    out = ctypes.c_int32()
    for ceiling in (600, 4096, 8271, 40960):
        for n_audio in range(0, 9000, 97):
            for extra in (1, 15, 300):
                T = n_audio + extra
                st = lib.dec_decode_budget(n_audio, T, 256, ceiling, ctypes.byref(out))
                try:
                    want = O.decode_budget(n_audio, T, ceiling)
                except ValueError:
                    assert st == binding.DEC_ERR_INPUT_TOO_LONG, (n_audio, T, ceiling)
                    continue
                assert st == binding.DEC_OK and out.value == want, (n_audio, T, ceiling)
    assert lib.dec_decode_budget(-1, 10, 256, 1000, ctypes.byref(out)) == binding.DEC_ERR_INVALID_ARG
    assert lib.dec_decode_budget(10, 0, 256, 1000, ctypes.byref(out)) == binding.DEC_ERR_INVALID_ARG
    assert lib.dec_decode_budget(10, 20, 256, 1000, None) == binding.DEC_ERR_INVALID_ARG
