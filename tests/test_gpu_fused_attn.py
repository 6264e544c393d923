"""Parity of the single-sequence decode step whose q|k|v GEMV finishes each KV
head's attention itself (the CTA that completes a head's q, k and v rows runs
the head's attention over every key) against the fp64 oracle and against the
separate split-KV attention kernel (the default; SPEECH_DECODER_STEP_ATTN=fused
selects the fused step).

Contexts cover one key tile (256 keys), a step whose appended key opens a new
tile (no key of that tile comes from the pool), and four tiles.  The q|k|v
rows (4096) split over one CTA per SM, so most CTAs hold rows of two heads and
every head's rows are completed by several CTAs."""
import os

import numpy as np
import pytest

import oracle as O
from _parity import prompt_rows, rel_err, teacher_forced
from speech_decoder_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2

SPEC = synth.small_spec(n_layers=2, hidden=1024, n_heads=16, n_kv_heads=8, head_dim=128, ffn=3072,
                        vocab=32768)


@pytest.fixture(scope="module", autouse=True)
def built():
    from speech_decoder_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def weights():
    return synth.model_weights(SPEC, seed=41)


def make(w, split=False, **kw):
    from speech_decoder_gb300.binding import Decoder
    old = os.environ.get("SPEECH_DECODER_STEP_ATTN")
    if split:
        os.environ.pop("SPEECH_DECODER_STEP_ATTN", None)
    else:
        os.environ["SPEECH_DECODER_STEP_ATTN"] = "fused"
    try:
        return Decoder(SPEC, w, **kw)
    finally:
        if old is None:
            os.environ.pop("SPEECH_DECODER_STEP_ATTN", None)
        else:
            os.environ["SPEECH_DECODER_STEP_ATTN"] = old


CASES = [(synth.Prompt(4, 150, 3), 10), (synth.Prompt(4, 240, 6), 12), (synth.Prompt(9, 855, 6), 40)]
IDS = ["T157-1tile", "T250-newtile", "T870-4tiles"]


@pytest.mark.parametrize("prompt,steps", CASES, ids=IDS)
def test_fused_teacher_forced(weights, prompt, steps):
    emb, _ = prompt_rows(SPEC, weights, prompt, seed=42)
    dec = make(weights, max_ctx=prompt.T + steps + 8, max_new=steps + 2)
    worst, _ = teacher_forced(dec, O.Oracle(SPEC, weights, prompt.T + steps), emb, steps, TOL_BF16)
    dec.close()
    print(f"T={prompt.T}: worst rel logit err {worst:.2e}")


@pytest.mark.parametrize("prompt,steps", CASES, ids=IDS)
def test_fused_matches_split(weights, prompt, steps):
    emb, _ = prompt_rows(SPEC, weights, prompt, seed=43)
    kw = dict(max_ctx=prompt.T + steps + 8, max_new=steps + 2)
    a, b = make(weights, **kw), make(weights, split=True, **kw)
    ta, tb = a.prefill(emb), b.prefill(emb)
    assert ta == tb
    tok = ta
    la0, lb0 = a.launch_count(), b.launch_count()
    for i in range(steps):
        na, nb = a.step(tok), b.step(tok)
        ga, gb = a.logits(1), b.logits(1)
        # the same attention arithmetic, one split against several: fp32 rounding
        assert rel_err(ga, gb) <= 1e-4, i
        assert na == nb, i
        tok = na
    # the fused step has no attention launch: one launch fewer per layer and step
    assert (b.launch_count() - lb0) - (a.launch_count() - la0) == SPEC.n_layers * steps
    a.close()
    b.close()


def test_fused_greedy_equals_oracle(weights):
    """The CUDA-graph greedy loop (the benchmark's path) on the fused step."""
    prompt = synth.Prompt(3, 200, 2)
    emb, _ = prompt_rows(SPEC, weights, prompt, seed=44)
    n = 24
    dec = make(weights, max_ctx=prompt.T + n + 8, max_new=n)
    dec.prefill(emb)
    ids, _ = dec.generate(n)
    dec.close()
    ref, _, _ = O.greedy(O.Oracle(SPEC, weights, prompt.T + n), emb.astype(np.float64), n)
    assert ids == ref
