"""Parity of the e4m3 weight format (bf16 weights rounded row by row to
2^e * e4m3; the single-sequence step GEMVs stream the 1-byte codes).

* dec_quantize_e4m3_rows against the oracle's rounding, bit for bit: codes
  (by value), row scales and the rounded bf16 weights, in place and not;
* a decoder created with DEC_E4M3 against the fp64 oracle given the same
  rounded weights: prefill logits and teacher-forced steps (relative error
  <= 2e-2), the greedy loop, and batched steps (which take the rounded bf16
  copy);
* the step GEMVs really stream one byte per weight (the profiler's
  algorithmic bytes of the projection GEMVs halve against the bf16 decoder).
"""
import ctypes

import numpy as np
import pytest

import oracle as O
from _parity import prompt_rows, rel_err, teacher_forced, token_ok
from speech_decoder_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2

SPEC = synth.small_spec(n_layers=2, hidden=1024, n_heads=16, n_kv_heads=8, head_dim=128, ffn=3072,
                        vocab=32768, weight_dtype="e4m3")


@pytest.fixture(scope="module", autouse=True)
def built():
    from speech_decoder_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def weights():
    return synth.model_weights(SPEC, seed=51)


@pytest.fixture(scope="module")
def rounded(weights):
    return O.e4m3_weights(weights)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def special_rows(cols: int, rng) -> np.ndarray:
    w = (rng.standard_normal((300, cols)) * 0.02).astype(np.float32)
    w[0] = 0.0                                            # all-zero row: scale 1
    w[1] = 0.0
    w[1, 5] = 56.0                                        # max exactly 448 * 2^-3
    w[2] = 0.0
    w[2, 9] = -56.25                                      # just above: scale 2^-2
    w[3] *= np.float32(1e-30)                             # tiny row
    w[4, 11] = 1000.0                                     # one outlier: most values round to 0
    w[5] = np.abs(w[5])
    w[6] = -np.abs(w[6])
    w[7] = ((np.arange(cols) % 29) - 14) * np.float32(0.37)   # a spread of magnitudes
    w[8, :] = 17.0 / 32          # scale 2^-9: 17/32 * 2^9 = 272, a midpoint of 256 and 288 (ties to even: 256)
    synth.round_bf16(w)
    return w


@pytest.mark.parametrize("cols", [1024, 6144, 48])
def test_quantize_op_bit_exact(cols):
    import torch
    from speech_decoder_gb300.binding import load_library
    lib = load_library()
    w = special_rows(cols, np.random.default_rng(52 + cols))
    ref_r, ref_s, ref_q = O.quantize_rows(w)
    wb = torch.from_numpy(synth.bf16_bits(w).view(np.int16)).cuda()
    codes = torch.empty(w.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(w.shape[0], dtype=torch.float32, device="cuda")
    out = torch.empty_like(wb)
    assert lib.dec_quantize_e4m3_rows(ctypes.c_void_p(wb.data_ptr()), w.shape[0], cols,
                                      ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scales.data_ptr()),
                                      ctypes.c_void_p(out.data_ptr()), None) == 0
    torch.cuda.synchronize()
    assert np.array_equal(scales.cpu().numpy(), ref_s)
    got_q = O.e4m3_decode(codes.cpu().numpy())
    assert np.array_equal(got_q, ref_q), np.argwhere(got_q != ref_q)[:5]
    assert np.array_equal(bf16_values(out.cpu().numpy().view(np.uint16)), ref_r)
    # in place: the rounded values overwrite the input
    assert lib.dec_quantize_e4m3_rows(ctypes.c_void_p(wb.data_ptr()), w.shape[0], cols,
                                      ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scales.data_ptr()),
                                      ctypes.c_void_p(wb.data_ptr()), None) == 0
    torch.cuda.synchronize()
    assert np.array_equal(bf16_values(wb.cpu().numpy().view(np.uint16)), ref_r)


def test_quantize_op_rejects_bad_arguments():
    from speech_decoder_gb300.binding import DEC_ERR_INVALID_ARG, load_library
    lib = load_library()
    p = ctypes.c_void_p(16)
    assert lib.dec_quantize_e4m3_rows(None, 4, 16, p, p, p, None) == DEC_ERR_INVALID_ARG
    assert lib.dec_quantize_e4m3_rows(p, 0, 16, p, p, p, None) == DEC_ERR_INVALID_ARG
    assert lib.dec_quantize_e4m3_rows(p, 4, 0, p, p, p, None) == DEC_ERR_INVALID_ARG


def make(w, **kw):
    from speech_decoder_gb300.binding import Decoder
    return Decoder(SPEC, w, **kw)


@pytest.mark.parametrize("prompt", [synth.Prompt(4, 150, 3), synth.Prompt(0, 1, 0), synth.Prompt(9, 600, 5)],
                         ids=["T157", "T1", "T614"])
def test_e4m3_teacher_forced(weights, rounded, prompt):
    emb, _ = prompt_rows(SPEC, rounded, prompt, seed=53)
    dec = make(weights, max_ctx=prompt.T + 24, max_new=12)
    worst, _ = teacher_forced(dec, O.Oracle(SPEC, rounded, prompt.T + 12), emb, 10, TOL)
    dec.close()
    print(f"T={prompt.T}: worst rel logit err {worst:.2e}")


def test_e4m3_greedy_equals_oracle(weights, rounded):
    prompt = synth.Prompt(3, 200, 2)
    emb, _ = prompt_rows(SPEC, rounded, prompt, seed=54)
    n = 24
    dec = make(weights, max_ctx=prompt.T + n + 8, max_new=n)
    dec.prefill(emb)
    ids, _ = dec.generate(n)
    dec.close()
    ref, _, _ = O.greedy(O.Oracle(SPEC, rounded, prompt.T + n), emb.astype(np.float64), n)
    assert ids == ref


def test_e4m3_batched_steps(weights, rounded):
    """Several sequences per step take the rounded bf16 weights: the same model."""
    prompts = [synth.Prompt(2, 40, 1), synth.Prompt(5, 333, 4), synth.Prompt(0, 7, 0)]
    embs = [prompt_rows(SPEC, rounded, p, seed=55, item=i)[0] for i, p in enumerate(prompts)]
    dec = make(weights, max_ctx=400, max_batch=3, max_tokens=512, max_new=8)
    dec.prefill_batch(embs)
    orcs = [O.Oracle(SPEC, rounded, e.shape[0] + 8) for e in embs]
    toks = [O.argmax_lowest(o.prefill(e)) for o, e in zip(orcs, embs)]
    for step in range(4):
        nxt = dec.step_batch(np.array(toks, np.int32), np.ones(3, np.uint8))
        got = dec.logits(3)
        for b in range(3):
            ref = orcs[b].step(toks[b])
            assert rel_err(got[b], ref) <= TOL, (step, b)
            assert token_ok(int(nxt[b]), ref, got[b])
            toks[b] = O.argmax_lowest(ref)
    dec.close()


def test_e4m3_steps_stream_one_byte_per_weight(weights):
    """dec_profile_kernel(op 0) runs the step's projection GEMVs as the step
    launches them; their algorithmic bytes count one byte per weight."""
    import dataclasses
    emb = np.random.default_rng(56).standard_normal((16, SPEC.hidden)).astype(np.float32)
    a = make(weights, max_ctx=64, max_new=8)
    bspec = dataclasses.replace(SPEC, weight_dtype="bf16")
    from speech_decoder_gb300.binding import Decoder
    b = Decoder(bspec, weights, max_ctx=64, max_new=8)
    a.prefill(emb)
    b.prefill(emb)
    _, bytes_a = a.profile_kernel(0, 2)
    _, bytes_b = b.profile_kernel(0, 2)
    a.close()
    b.close()
    H, F, d = SPEC.hidden, SPEC.ffn, SPEC.head_dim
    w_elems = ((SPEC.n_heads + 2 * SPEC.n_kv_heads) * d * H + H * SPEC.n_heads * d + 2 * F * H + H * F) / 4
    assert bytes_b - bytes_a == pytest.approx(w_elems, rel=1e-6)
