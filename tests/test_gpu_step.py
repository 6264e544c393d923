"""Parity of the persistent decode step (one cooperative launch per greedy
step) with the fp64 oracle and with the per-op kernel sequence.

The model is sized so that every CTA owns many ring chunks per projection
(the lm_head gives each CTA more chunks than the ring has stages and the CTA
has consumer warps), which is where the step kernel's chunk hand-off between
the producer and the consumer warps wraps around the ring several times."""
import os

import numpy as np
import pytest

import oracle as O
from _parity import prompt_rows, rel_err, teacher_forced, token_ok
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
    return synth.model_weights(SPEC, seed=31)


def make(w, kernels=False, **kw):
    from speech_decoder_gb300.binding import Decoder
    old = os.environ.get("SPEECH_DECODER_STEP")
    os.environ["SPEECH_DECODER_STEP"] = "kernels" if kernels else "persistent"
    try:
        return Decoder(SPEC, w, **kw)
    finally:
        if old is None:
            os.environ.pop("SPEECH_DECODER_STEP", None)
        else:
            os.environ["SPEECH_DECODER_STEP"] = old


def steps_launches(dec, emb, n):
    dec.prefill(emb)
    before = dec.launch_count()
    ids, _ = dec.generate(n)
    return ids, dec.launch_count() - before


@pytest.mark.parametrize("prompt", [synth.Prompt(4, 150, 3), synth.Prompt(0, 1, 0), synth.Prompt(9, 600, 5)],
                         ids=["T157", "T1", "T614"])
def test_step_teacher_forced(weights, prompt):
    emb, _ = prompt_rows(SPEC, weights, prompt, seed=32)
    dec = make(weights, max_ctx=prompt.T + 24, max_new=12)
    teacher_forced(dec, O.Oracle(SPEC, weights, prompt.T + 12), emb, 10, TOL_BF16)


def test_step_matches_kernel_sequence(weights):
    emb, _ = prompt_rows(SPEC, weights, synth.Prompt(3, 200, 2), seed=33)
    a = make(weights, max_ctx=256, max_new=16)
    b = make(weights, kernels=True, max_ctx=256, max_new=16)
    ids_a, la = steps_launches(a, emb, 16)
    ids_b, lb = steps_launches(b, emb, 16)
    # the persistent path launches far fewer kernels per step than the per-op sequence
    assert la < lb, (la, lb)
    ref, _, _ = O.greedy(O.Oracle(SPEC, weights, emb.shape[0] + 16), emb, 16)
    assert ids_a == ref and ids_b == ref
    # single steps: logits of the two paths agree to fp32 rounding of different summation orders
    a.prefill(emb)
    b.prefill(emb)
    tok = ref[0]
    for _ in range(4):
        ta, tb = a.step(tok), b.step(tok)
        la_, lb_ = a.logits(1), b.logits(1)
        assert rel_err(la_, lb_) <= 1e-4
        assert ta == tb
        tok = ta


def test_step_batched_rows(weights):
    prompts = [synth.Prompt(2, 40, 1), synth.Prompt(5, 333, 4), synth.Prompt(0, 7, 0), synth.Prompt(1, 90, 2)]
    embs = [prompt_rows(SPEC, weights, p, seed=34, item=i)[0] for i, p in enumerate(prompts)]
    dec = make(weights, max_ctx=400, max_batch=4, max_tokens=512, max_new=8)
    dec.prefill_batch(embs)
    orcs = [O.Oracle(SPEC, weights, e.shape[0] + 8) for e in embs]
    toks = [O.argmax_lowest(o.prefill(e)) for o, e in zip(orcs, embs)]
    for step in range(5):
        active = np.array([1, 0 if step == 2 else 1, 1, 1], np.uint8)
        nxt = dec.step_batch(np.array(toks, np.int32), active)
        got = dec.logits(4)
        for b in range(4):
            if not active[b]:
                assert nxt[b] == -1
                continue
            ref = orcs[b].step(toks[b])
            assert rel_err(got[b], ref) <= TOL_BF16, (step, b)
            assert token_ok(int(nxt[b]), ref, got[b])
            toks[b] = O.argmax_lowest(ref)
