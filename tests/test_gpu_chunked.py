"""Chunked prefill through the C ABI: prompt rows fed in pieces against the
growing KV cache must give the logits, first token and greedy run of a
single whole-prompt prefill (the oracle pins chunked == single-shot in
test_oracle_pins), on both prompt-attention paths (tensor cores for
head_dim 128 with fp16 KV, CUDA cores for head_dim 64)."""
import numpy as np
import pytest

import oracle as O
from _parity import prompt_rows, rel_err, token_ok
from speech_decoder_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from speech_decoder_gb300 import build
    build.build()


def make(spec, w, **kw):
    from speech_decoder_gb300.binding import Decoder
    return Decoder(spec, w, **kw)


SPECS = [
    dict(n_layers=2, hidden=512, n_heads=4, n_kv_heads=2, head_dim=128, ffn=1024, vocab=2048),
    dict(n_layers=2, hidden=512, n_heads=8, n_kv_heads=2, head_dim=64, ffn=768, vocab=1500),
]


@pytest.mark.parametrize("kw", SPECS, ids=["d128", "d64"])
@pytest.mark.parametrize("cuts", [(100, 177), (1, 2, 130, 290)], ids=["3chunks", "5chunks"])
def test_chunked_equals_single(kw, cuts):
    spec = synth.small_spec(**kw)
    w = synth.model_weights(spec, seed=41)
    emb, _ = prompt_rows(spec, w, synth.Prompt(5, 290, 5), seed=42)
    T = emb.shape[0]
    a = make(spec, w, max_ctx=T + 32, max_tokens=T, max_new=12)
    t_single = a.prefill(emb)
    l_single = a.logits(1)[0]
    ids_single, _ = a.generate(12)
    b = make(spec, w, max_ctx=T + 32, max_tokens=T, max_new=12)
    bounds = [0, *cuts, T]
    for i in range(len(bounds) - 1):
        last = i == len(bounds) - 2
        tok = b.prefill_chunk(emb[bounds[i]:bounds[i + 1]], final=last)
        assert (tok is None) != last
    l_chunk = b.logits(1)[0]
    assert rel_err(l_chunk, l_single) <= 1e-3
    assert tok == t_single
    ids_chunk, _ = b.generate(12)
    assert ids_chunk == ids_single
    ref = O.Oracle(spec, w, T + 4).prefill(emb.astype(np.float64))
    assert rel_err(l_chunk, ref) <= TOL_BF16 and token_ok(tok, ref, l_chunk)


def test_chunk_state_and_limits():
    from speech_decoder_gb300.binding import DEC_ERR_INPUT_TOO_LONG, DEC_ERR_STATE, DecError
    spec = synth.small_spec(**SPECS[0])
    w = synth.model_weights(spec, seed=43)
    emb, _ = prompt_rows(spec, w, synth.Prompt(2, 60, 2), seed=44)
    dec = make(spec, w, max_ctx=80, max_tokens=64, max_new=8)
    assert dec.prefill_chunk(emb[:30]) is None
    with pytest.raises(DecError) as e:
        dec.step(1)                                  # not prefilled until the final chunk
    assert e.value.status == DEC_ERR_STATE
    with pytest.raises(DecError) as e:
        dec.prefill_chunk(emb[:50], final=True)      # 30 + 50 + 8 > 80
    assert e.value.status == DEC_ERR_INPUT_TOO_LONG
    # the failed call abandoned the chunked prompt: a new one starts at position 0
    assert dec.prefill_chunk(emb[:40]) is None
    tok = dec.prefill_chunk(emb[40:], final=True)
    ref = O.Oracle(spec, w, 80).prefill(emb.astype(np.float64))
    assert token_ok(tok, ref, dec.logits(1)[0])
    ids, _ = dec.generate(8)
    assert len(ids) == 8
