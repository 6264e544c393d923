"""The cluster step attention (one thread-block cluster per sequence and KV
head, the keys split over the cluster's CTAs and combined through
distributed shared memory) against the oracle and against the split-KV
attention kernel, for every cluster size the context capacity selects
(1, 2, 4, 8 CTAs, and 8 CTAs holding up to 128 keys each) and 1, 2 and 4
query heads per KV head."""
import os

import numpy as np
import pytest

import oracle as O
from _parity import prompt_rows, rel_err, teacher_forced
from speech_decoder_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from speech_decoder_gb300 import build
    build.build()


def make(spec, w, attn=None, **kw):
    from speech_decoder_gb300.binding import Decoder
    old = os.environ.get("SPEECH_DECODER_STEP_ATTN")
    try:
        if attn:
            os.environ["SPEECH_DECODER_STEP_ATTN"] = attn
        return Decoder(spec, w, **kw)
    finally:
        if old is None:
            os.environ.pop("SPEECH_DECODER_STEP_ATTN", None)
        else:
            os.environ["SPEECH_DECODER_STEP_ATTN"] = old


HEADS = [(2, 2), (4, 2), (8, 2)]            # (query heads, KV heads): n_rep 1, 2, 4
# (prompt, context capacity): one, two, four and eight CTAs per cluster (up to 64 keys each while
# the cluster can grow), and eight CTAs of up to 128 keys each
SIZES = [(synth.Prompt(3, 40, 2), 60), (synth.Prompt(3, 60, 2), 100), (synth.Prompt(5, 170, 4), 250),
         (synth.Prompt(9, 400, 6), 500), (synth.Prompt(9, 850, 6), 1000)]


@pytest.mark.parametrize("heads", HEADS, ids=[f"q{a}kv{b}" for a, b in HEADS])
@pytest.mark.parametrize("size", SIZES, ids=["S1", "S2", "S4", "S8", "S8full"])
def test_cluster_attention_teacher_forced(heads, size):
    nq, nkv = heads
    prompt, cap = size
    spec = synth.small_spec(n_layers=2, hidden=256, n_heads=nq, n_kv_heads=nkv, head_dim=128, ffn=512, vocab=997)
    w = synth.model_weights(spec, seed=61)
    emb, _ = prompt_rows(spec, w, prompt, seed=62)
    steps = 6
    dec = make(spec, w, max_ctx=cap, max_new=cap - prompt.T)
    worst, _ = teacher_forced(dec, O.Oracle(spec, w, prompt.T + steps + 1), emb, steps, TOL)
    # the same steps on the split-KV kernel: equal up to fp32 rounding order
    ref = make(spec, w, attn="split", max_ctx=cap, max_new=cap - prompt.T)
    dec.prefill(emb)
    ref.prefill(emb)
    tok = 5
    for _ in range(steps):
        a = dec.step(tok)
        b = ref.step(tok)
        assert rel_err(dec.logits(1)[0], ref.logits(1)[0]) <= 1e-4
        assert a == b
        tok = a
    dec.close()
    ref.close()
    print(f"{nq}/{nkv} heads, capacity {cap}: worst rel err vs oracle {worst:.2e}")


def test_cluster_attention_batched_rows():
    """Up to four sequences of different lengths in one launch (one cluster
    per sequence and KV head), teacher-forced against the oracle."""
    spec = synth.small_spec(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=128, ffn=512, vocab=997)
    w = synth.model_weights(spec, seed=71)
    prompts = [synth.Prompt(2, 30, 1), synth.Prompt(4, 300, 3), synth.Prompt(1, 7, 0), synth.Prompt(6, 480, 2)]
    embs = [prompt_rows(spec, w, p, seed=72, item=i)[0] for i, p in enumerate(prompts)]
    dec = make(spec, w, max_ctx=500, max_batch=4, max_tokens=1024, max_new=8)
    first = dec.prefill_batch(embs)
    orcs = [O.Oracle(spec, w, e.shape[0] + 8) for e in embs]
    refs = [o.prefill(e) for o, e in zip(orcs, embs)]
    got = dec.logits(4)
    toks = []
    for b in range(4):
        assert rel_err(got[b], refs[b]) <= TOL
        toks.append(O.argmax_lowest(refs[b]))
    for _ in range(5):
        dec.step_batch(np.array(toks, np.int32))
        got = dec.logits(4)
        for b in range(4):
            ref = orcs[b].step(toks[b])
            assert rel_err(got[b], ref) <= TOL, b
            toks[b] = O.argmax_lowest(ref)
    dec.close()
