"""dec_attn_decode_noalloc: the scratch-free variant of the decode attention
for callers that cannot allocate device memory (an engine or plugin that owns
all device memory, a loop that must not call cudaMalloc).  Its output must
match dec_attn_decode, which takes caller-allocated scratch, on two calls in a
row (the second call reuses the shared array the first one left behind).

This file sorts last so that a run stopping at the first failure has already
run every other test."""
import numpy as np
import pytest

from _parity import rel_err
from test_gpu_ops import attn_case, run_op

pytestmark = pytest.mark.gpu

TOL = 1e-4     # the fp32 tolerance of the other parity tests


@pytest.fixture(scope="module")
def lib():
    from speech_decoder_gb300 import binding, build
    build.build()
    return binding.load_library()


def test_noalloc_matches_scratch_entry_point_twice(lib):
    cases = [
        (3, 16, 8, 128, 2048, [5, 152, 700], [0, 10, 1000], True),
        (2, 8, 2, 64, 512, [300, 33], [0, 300], False),
    ]
    for B, nq, nkv, d, slots, lens, offs, f16 in cases:
        q, K, V, lens_a, offs_a = attn_case(21, B, nq, nkv, d, slots, lens, offs, f16)
        ref = run_op(lib, q, K, V, lens_a, offs_a, f16, fn="dec_attn_decode")
        for _ in range(2):
            got = run_op(lib, q, K, V, lens_a, offs_a, f16, fn="dec_attn_decode_noalloc")
            assert rel_err(got.reshape(B, -1), ref.reshape(B, -1)) <= TOL


def test_noalloc_rejects_oversized_shapes(lib):
    from speech_decoder_gb300.binding import DEC_ERR_OOM
    # 4096 sequences x 8 KV heads x 1 split x 2 query heads x (128 + 2) floats:
    # about 34 MB of partials, far above the 4 MiB array
    st = lib.dec_attn_decode_noalloc(1, 1, 1, 2, 100, 1, 1, 4096, 16, 8, 128, 1, None)
    assert st == DEC_ERR_OOM
    # the limit of that shape is 502 sequences: 503 no longer fits
    assert lib.dec_attn_decode_noalloc(1, 1, 1, 2, 100, 1, 1, 503, 16, 8, 128, 1, None) == DEC_ERR_OOM
