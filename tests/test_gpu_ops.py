"""Kernel-level parity through the C ABI: the standalone split-KV decode
attention against the oracle's attention on the same (fp16-rounded) keys."""
import ctypes

import numpy as np
import pytest

import oracle as O
from _parity import rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from speech_decoder_gb300 import binding, build
    build.build()
    return binding.load_library()


def attn_case(seed, B, nq, nkv, d, slots, lens, offs, kv_f16):
    rng = np.random.default_rng(seed)
    kv_np = np.float16 if kv_f16 else np.float32
    K = rng.standard_normal((nkv, slots, d)).astype(kv_np)
    V = rng.standard_normal((nkv, slots, d)).astype(kv_np)
    q = (rng.standard_normal((B, nq, d)) * 0.3).astype(np.float32)
    return q, K, V, np.array(lens, np.int32), np.array(offs, np.int32)


def run_op(lib, q, K, V, lens, offs, kv_f16, fn="dec_attn_decode"):
    import torch
    from speech_decoder_gb300.binding import DEC_F16, DEC_F32
    B, nq, d = q.shape
    nkv, slots, _ = K.shape
    dev = "cuda:0"
    tq, tK, tV = (torch.from_numpy(a).to(dev) for a in (q, K, V))
    toff, tlen = torch.from_numpy(offs).to(dev), torch.from_numpy(lens).to(dev)
    out = torch.full((B, nq, d), 7.0, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    args = [tq.data_ptr(), tK.data_ptr(), tV.data_ptr(), DEC_F16 if kv_f16 else DEC_F32, slots, toff.data_ptr(),
            tlen.data_ptr(), B, nq, nkv, d, out.data_ptr()]
    if fn == "dec_attn_decode":
        n = ctypes.c_size_t()
        assert lib.dec_attn_decode_scratch_size(B, nq, nkv, d, ctypes.byref(n)) == 0
        scratch = torch.empty(n.value, dtype=torch.uint8, device=dev)
        st = lib.dec_attn_decode(*args, scratch.data_ptr(), n.value, stream.cuda_stream)
    else:
        st = getattr(lib, fn)(*args, stream.cuda_stream)
    assert st == 0, st
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_attn(q, K, V, lens, offs):
    out = []
    for b in range(q.shape[0]):
        L, o = int(lens[b]), int(offs[b])
        Kb = np.transpose(K[:, o:o + L, :].astype(np.float64), (1, 0, 2))
        Vb = np.transpose(V[:, o:o + L, :].astype(np.float64), (1, 0, 2))
        out.append(O.attention(q[b][None].astype(np.float64), Kb, Vb, np.array([L - 1]))[0])
    return np.stack(out)


CASES = [
    # B, nq, nkv, d, slots, lens, offs, kv_f16
    (1, 16, 8, 128, 8192, [8143], [0], True),
    (3, 16, 8, 128, 2048, [1, 152, 700], [0, 10, 1000], True),
    (4, 8, 1, 64, 600, [33, 1, 257, 64], [0, 40, 80, 400], False),
    (2, 4, 4, 64, 100, [17, 50], [0, 50], True),
    (5, 32, 4, 128, 3000, [2999, 1, 2, 500, 1000], [0, 0, 0, 0, 1500], True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}q{c[1]}kv{c[2]}d{c[3]}{'f16' if c[7] else 'f32'}" for c in CASES])
def test_attn_decode_op_matches_oracle(lib, case):
    B, nq, nkv, d, slots, lens, offs, f16 = case
    q, K, V, lens, offs = attn_case(11, B, nq, nkv, d, slots, lens, offs, f16)
    got = run_op(lib, q, K, V, lens, offs, f16)
    ref = oracle_attn(q, K, V, lens, offs)
    assert rel_err(got.reshape(B, -1), ref.reshape(B, -1)) <= 1e-4


def test_attn_decode_op_skips_invalid_rows(lib):
    q, K, V, lens, offs = attn_case(12, 3, 4, 2, 64, 64, [0, 10, 60], [0, 0, 10], True)
    got = run_op(lib, q, K, V, lens, offs, True)
    assert np.all(got[0] == 7.0) and np.all(got[2] == 7.0)          # len 0 and out-of-pool rows untouched
    ref = oracle_attn(q[1:2], K, V, lens[1:2], offs[1:2])
    assert rel_err(got[1].reshape(1, -1), ref.reshape(1, -1)) <= 1e-4
