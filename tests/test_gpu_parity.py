"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on small
models: several shapes, ragged prompts, batched rows, greedy loops, dumps and
error paths.  Tolerances: max relative logit error 1e-4 for the fp32 build
and 2e-2 for the bf16 build; greedy tokens must equal the oracle's unless the
oracle's top-2 gap lies inside twice the observed logit error."""
import numpy as np
import pytest

import oracle as O
from _parity import prompt_rows, rel_err, teacher_forced, token_ok
from speech_decoder_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from speech_decoder_gb300 import build
    build.build()


def make(spec, w, **kw):
    from speech_decoder_gb300.binding import Decoder
    return Decoder(spec, w, **kw)


# ------------------------------------------------------------------ tiny block (fp32 build)
@pytest.fixture(scope="module")
def tiny():
    wl = synth.workload("tiny")
    w = synth.model_weights(wl.model)
    emb, _ = prompt_rows(wl.model, w, wl.prompts[0])
    return wl, w, emb


def test_tiny_fp32_teacher_forced(tiny):
    wl, w, emb = tiny
    dec = make(wl.model, w, max_ctx=64, max_new=16)
    worst, ties = teacher_forced(dec, O.Oracle(wl.model, w, emb.shape[0] + 16), emb, wl.steps, TOL_F32)
    assert ties == 0
    print(f"tiny fp32 worst rel err {worst:.2e}")


def test_tiny_fp32_greedy_generate(tiny):
    wl, w, emb = tiny
    dec = make(wl.model, w, max_ctx=64, max_new=16)
    dec.prefill(emb)
    ids, trunc = dec.generate(wl.steps + 1)
    ref, rtrunc, _ = O.greedy(O.Oracle(wl.model, w, emb.shape[0] + 16), emb, wl.steps + 1)
    assert ids == ref and trunc == rtrunc


def test_tiny_bf16_teacher_forced(tiny):
    wl, _, _ = tiny
    spec = synth.ModelSpec("tiny-bf16", 1, 256, 4, 2, 64, 768, 1024, norm_init="ones")
    w = synth.model_weights(spec)
    emb, _ = prompt_rows(spec, w, wl.prompts[0])
    dec = make(spec, w, max_ctx=64, max_new=16)
    teacher_forced(dec, O.Oracle(spec, w, emb.shape[0] + 16), emb, wl.steps, TOL_BF16)


# ------------------------------------------------------------------ small bf16 models
SMALL = [
    dict(n_layers=2, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn=512, vocab=1000),
    dict(n_layers=3, hidden=512, n_heads=4, n_kv_heads=2, head_dim=128, ffn=1408, vocab=3001),
    dict(n_layers=2, hidden=512, n_heads=8, n_kv_heads=1, head_dim=64, ffn=768, vocab=777),
    dict(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=384, vocab=513),
]


@pytest.mark.parametrize("kw", SMALL, ids=[f"L{k['n_layers']}H{k['hidden']}q{k['n_heads']}kv{k['n_kv_heads']}d{k['head_dim']}" for k in SMALL])
@pytest.mark.parametrize("prompt", [synth.Prompt(3, 40, 2), synth.Prompt(0, 1, 0), synth.Prompt(9, 150, 5)],
                         ids=["T45", "T1", "T164"])
def test_small_bf16_teacher_forced(kw, prompt):
    spec = synth.small_spec(**kw)
    w = synth.model_weights(spec, seed=1)
    emb, _ = prompt_rows(spec, w, prompt, seed=2)
    dec = make(spec, w, max_ctx=prompt.T + 24, max_new=12)
    teacher_forced(dec, O.Oracle(spec, w, prompt.T + 12), emb, 10, TOL_BF16)


def test_small_f32_teacher_forced():
    spec = synth.small_spec(weight_dtype="f32", kv_dtype="f32", head_dim=128, hidden=512, ffn=1024)
    w = synth.model_weights(spec, seed=4)
    emb, _ = prompt_rows(spec, w, synth.Prompt(5, 60, 3), seed=5)
    dec = make(spec, w, max_ctx=128, max_new=12)
    worst, ties = teacher_forced(dec, O.Oracle(spec, w, 80), emb, 10, TOL_F32)
    assert ties == 0


# ------------------------------------------------------------------ dumps, assembly, consistency
@pytest.fixture(scope="module")
def small():
    spec = synth.small_spec(n_layers=3, hidden=512, n_heads=4, n_kv_heads=2, head_dim=128, ffn=1024, vocab=2048)
    return spec, synth.model_weights(spec, seed=7)


def test_dump_points(small):
    spec, w = small
    emb, _ = prompt_rows(spec, w, synth.Prompt(4, 50, 3), seed=8)
    dec = make(spec, w, max_ctx=128, max_new=8)
    dec.set_dumps(True)
    dec.prefill(emb)
    T, H = emb.shape
    inj = dec.dump("dec.audio_injected", (T, H))
    assert np.array_equal(inj, emb)
    orc = O.Oracle(spec, w, 128)
    x0 = orc.block(0, emb.astype(np.float64), np.arange(T))
    b0 = dec.dump("dec.block.0.out", (T, H))
    assert rel_err(b0, x0) <= TOL_BF16
    orc2 = O.Oracle(spec, w, 128)
    xl = orc2.forward(emb)
    last = dec.dump("dec.block.last.out", (1, H))
    assert rel_err(last, xl[-1:]) <= TOL_BF16
    yb = dec.dump("dec.out_before_head", (1, H))
    assert rel_err(yb, O.rms_norm(xl[-1:], w["final_norm"], spec.rms_eps)) <= TOL_BF16


def test_prefill_ids_matches_host_assembly(small):
    spec, w = small
    emb, p = prompt_rows(spec, w, synth.Prompt(6, 30, 4), seed=9)
    a = make(spec, w, max_ctx=128, max_new=8)
    t1 = a.prefill(emb)
    l1 = a.logits(1)
    t2 = a.prefill_ids(p["ids"], p["audio"], p["prefix_len"])
    l2 = a.logits(1)
    assert t1 == t2 and np.array_equal(l1, l2)


def test_prefill_then_step_equals_longer_prefill(small):
    spec, w = small
    emb, _ = prompt_rows(spec, w, synth.Prompt(2, 40, 2), seed=10)
    a = make(spec, w, max_ctx=128, max_new=8)
    a.prefill(emb)
    tok = 17
    t_step = a.step(tok)
    l_step = a.logits(1)
    ext = np.concatenate([emb, w["embed"][tok][None, :]]).astype(np.float32)
    t_pre = a.prefill(ext)
    l_pre = a.logits(1)
    assert rel_err(l_step, l_pre) <= TOL_BF16
    assert token_ok(t_step, l_pre[0].astype(np.float64), l_step[0])


# ------------------------------------------------------------------ batched rows
def test_batched_prefill_steps_and_active_mask(small):
    spec, w = small
    prompts = [synth.Prompt(2, 3, 0), synth.Prompt(4, 29, 3), synth.Prompt(0, 1, 0), synth.Prompt(9, 61, 6)]
    embs = [prompt_rows(spec, w, p, seed=11, item=i)[0] for i, p in enumerate(prompts)]
    dec = make(spec, w, max_ctx=128, max_batch=4, max_tokens=256, max_new=8)
    first = dec.prefill_batch(embs)
    got = dec.logits(4)
    orcs = [O.Oracle(spec, w, e.shape[0] + 8) for e in embs]
    refs = [o.prefill(e) for o, e in zip(orcs, embs)]
    toks = []
    for b in range(4):
        assert rel_err(got[b], refs[b]) <= TOL_BF16
        assert token_ok(int(first[b]), refs[b], got[b])
        toks.append(O.argmax_lowest(refs[b]))
    for step in range(5):
        active = np.array([1, 1, 0 if step % 2 else 1, 1], np.uint8)
        nxt = dec.step_batch(np.array(toks, np.int32), active)
        got = dec.logits(4)
        for b in range(4):
            if not active[b]:
                assert nxt[b] == -1
                continue
            ref = orcs[b].step(toks[b])
            assert rel_err(got[b], ref) <= TOL_BF16
            assert token_ok(int(nxt[b]), ref, got[b])
            toks[b] = O.argmax_lowest(ref)


def test_batched_equals_serial(small):
    spec, w = small
    prompts = [synth.Prompt(3, 20, 2), synth.Prompt(1, 47, 0), synth.Prompt(5, 8, 5)]
    embs = [prompt_rows(spec, w, p, seed=12, item=i)[0] for i, p in enumerate(prompts)]
    dec = make(spec, w, max_ctx=128, max_batch=3, max_tokens=128, max_new=8)
    first = dec.prefill_batch(embs)
    lb = dec.logits(3)
    for b, e in enumerate(embs):
        t = dec.prefill(e)
        assert t == first[b]
        assert rel_err(dec.logits(1)[0], lb[b]) <= 1e-5


def test_generate_batch_per_item_eos(small):
    spec, w = small
    prompts = [synth.Prompt(2, 12, 1), synth.Prompt(3, 30, 2), synth.Prompt(0, 5, 0)]
    embs = [prompt_rows(spec, w, p, seed=13, item=i)[0] for i, p in enumerate(prompts)]
    # EOS = the first token of item 0's oracle run that did not occur before it,
    # so item 0 stops early after k ids
    probe, _, _ = O.greedy(O.Oracle(spec, w, 64), embs[0], 12)
    ks = [i for i in range(1, len(probe)) if probe[i] not in probe[:i]]
    assert ks, "item 0 repeats one token; pick another seed"
    k = ks[0]
    eos = probe[k]
    refs = [O.greedy(O.Oracle(spec, w, e.shape[0] + 12), e, 12, eos_id=eos) for e in embs]
    dec = make(spec, w, max_ctx=128, max_batch=3, max_tokens=128, max_new=12, eos_id=eos)
    dec.prefill_batch(embs)
    out = dec.generate_batch(12, 3)
    for b in range(3):
        ids, trunc = out[b]
        rids, rtrunc, _ = refs[b]
        assert ids == rids and trunc == rtrunc, (b, ids, rids)
    assert not out[0][1] and len(out[0][0]) == k


# ------------------------------------------------------------------ errors
def test_error_paths(small):
    from speech_decoder_gb300.binding import (DEC_ERR_INPUT_TOO_LONG, DEC_ERR_INVALID_ARG, DEC_ERR_STATE,
                                              DecError)
    spec, w = small
    dec = make(spec, w, max_ctx=64, max_new=8)
    with pytest.raises(DecError) as e:
        dec.step(1)
    assert e.value.status == DEC_ERR_STATE
    with pytest.raises(DecError) as e:
        dec.prefill(np.zeros((57, spec.hidden), np.float32))      # 57 + 8 > 64
    assert e.value.status == DEC_ERR_INPUT_TOO_LONG
    emb, _ = prompt_rows(spec, w, synth.Prompt(2, 10, 2), seed=14)
    dec.prefill(emb)
    with pytest.raises(DecError) as e:
        dec.step(spec.vocab)
    assert e.value.status == DEC_ERR_INVALID_ARG
    with pytest.raises(DecError) as e:
        dec.generate(9)
    assert e.value.status == DEC_ERR_INVALID_ARG
    dec.reset()
    with pytest.raises(DecError) as e:
        dec.step(1)
    assert e.value.status == DEC_ERR_STATE


def test_budget_and_kv_full(small):
    from speech_decoder_gb300.binding import DEC_ERR_INPUT_TOO_LONG, DecError
    spec, w = small
    emb, _ = prompt_rows(spec, w, synth.Prompt(2, 10, 2), seed=15)
    dec = make(spec, w, max_ctx=64, max_new=8)
    dec.prefill(emb)
    ids, trunc = dec.generate(8)
    ref, rtrunc, _ = O.greedy(O.Oracle(spec, w, emb.shape[0] + 8), emb, 8)
    assert ids == ref and trunc and rtrunc and len(ids) == 8
    # the sequence owns T + max_new slots: max_new single steps fit, the next one does not
    dec.prefill(emb)
    for _ in range(8):
        dec.step(3)
    with pytest.raises(DecError) as e:
        dec.step(3)
    assert e.value.status == DEC_ERR_INPUT_TOO_LONG


# ------------------------------------------------------------------ batched rows on the tensor-core path (B > 4)
def test_batched_tc_path_prefill_steps_generate(small):
    spec, w = small
    rng = np.random.default_rng(21)
    prompts = [synth.Prompt(int(rng.integers(0, 5)), int(rng.integers(1, 90)), int(rng.integers(0, 4)))
               for _ in range(7)]
    embs = [prompt_rows(spec, w, p, seed=22, item=i)[0] for i, p in enumerate(prompts)]
    dec = make(spec, w, max_ctx=128, max_batch=8, max_tokens=1024, max_new=10)
    first = dec.prefill_batch(embs)
    got = dec.logits(7)
    orcs = [O.Oracle(spec, w, e.shape[0] + 10) for e in embs]
    refs = [o.prefill(e) for o, e in zip(orcs, embs)]
    toks = []
    for b in range(7):
        assert rel_err(got[b], refs[b]) <= TOL_BF16
        assert token_ok(int(first[b]), refs[b], got[b])
        toks.append(O.argmax_lowest(refs[b]))
    for step in range(4):
        active = np.ones(7, np.uint8)
        active[step % 7] = 0
        nxt = dec.step_batch(np.array(toks, np.int32), active)
        got = dec.logits(7)
        for b in range(7):
            if not active[b]:
                assert nxt[b] == -1
                continue
            ref = orcs[b].step(toks[b])
            assert rel_err(got[b], ref) <= TOL_BF16, (step, b)
            assert token_ok(int(nxt[b]), ref, got[b])
            toks[b] = O.argmax_lowest(ref)
    # greedy loop with per-item EOS on the same path
    probe, _, _ = O.greedy(O.Oracle(spec, w, embs[2].shape[0] + 10), embs[2], 10)
    ks = [i for i in range(1, len(probe)) if probe[i] not in probe[:i]]
    eos = probe[ks[0]] if ks else -1
    dec2 = make(spec, w, max_ctx=128, max_batch=8, max_tokens=1024, max_new=10, eos_id=eos)
    dec2.prefill_batch(embs)
    out = dec2.generate_batch(10, 7)
    for b in range(7):
        rids, rtrunc, _ = O.greedy(O.Oracle(spec, w, embs[b].shape[0] + 10), embs[b], 10, eos_id=eos)
        assert out[b][0] == rids and out[b][1] == rtrunc, (b, out[b], rids)


# ------------------------------------------------------------------ argmax ties on the device
def _tie_weights(spec, w, tops, used, near):
    """A copy of the weights in which, for each top token t in `tops`, a lower
    index j (t - 1 when `near`, else the lowest index not in `used`) gets the
    embedding row of t: logit j then equals logit t exactly, at every
    position (the lm_head is the tied embedding), so the lowest-index rule
    must pick j.  Returns (weights, {t: j})."""
    w2 = dict(w)
    E = np.array(w["embed"], copy=True)
    pairs, taken = {}, set(used) | set(tops)
    for t in sorted(set(tops)):
        if near:
            j = t - 1
            assert j >= 0 and j not in taken
        else:
            j = next(i for i in range(t) if i not in taken)
        E[j] = E[t]
        pairs[t] = j
        taken.add(j)
    w2["embed"] = E
    return w2, pairs


@pytest.mark.parametrize("near", [True, False], ids=["same-warp", "across-ctas"])
def test_argmax_tie_single_sequence(small, near):
    """The lm_head GEMV's argmax (one sequence) returns the lower index of two
    equal logits, within a warp's rows and across CTAs (model.cpp, run: the
    strict '>' scan keeps the first maximum)."""
    spec, w = small
    emb, item = prompt_rows(spec, w, synth.Prompt(3, 30, 2), seed=31)
    t = O.argmax_lowest(O.Oracle(spec, w, emb.shape[0] + 2).prefill(emb))
    used = set(int(v) for v in item["ids"])
    if near and (t == 0 or t - 1 in used):
        pytest.skip("no free neighbour below the top token for this seed")
    w2, pairs = _tie_weights(spec, w, [t], used, near)
    j = pairs[t]
    if not near:
        assert t - j > spec.vocab // 152, "the two rows must sit in different CTAs"
    emb2, _ = prompt_rows(spec, w2, synth.Prompt(3, 30, 2), seed=31)
    ref = O.Oracle(spec, w2, emb2.shape[0] + 2).prefill(emb2)
    assert ref[j] == ref[t] and O.argmax_lowest(ref) == j
    dec = make(spec, w2, max_ctx=64, max_new=2)
    tok = dec.prefill(emb2)
    got = dec.logits(1)[0]
    dec.close()
    assert got[j] == got[t], "the duplicated rows must give identical logits"
    assert tok == j, f"tie of rows {j} and {t}: the device picked {tok}"


def test_argmax_tie_batched_rows(small):
    """Same rule for the batched head (more rows than one GEMV CTA holds: the
    tensor-core lm_head and the row-wise argmax kernel)."""
    spec, w = small
    prompts = [synth.Prompt(2, 10 + 7 * i, 1) for i in range(6)]
    rows = [prompt_rows(spec, w, p, seed=41, item=i) for i, p in enumerate(prompts)]
    tops = [O.argmax_lowest(O.Oracle(spec, w, e.shape[0] + 2).prefill(e)) for e, _ in rows]
    used = set(int(v) for _, it in rows for v in it["ids"])
    w2, pairs = _tie_weights(spec, w, tops, used, near=False)
    embs = [prompt_rows(spec, w2, p, seed=41, item=i)[0] for i, p in enumerate(prompts)]
    dec = make(spec, w2, max_ctx=128, max_batch=8, max_tokens=1024, max_new=2)
    first = dec.prefill_batch(embs)
    got = dec.logits(6)
    dec.close()
    for b, e in enumerate(embs):
        ref = O.Oracle(spec, w2, e.shape[0] + 2).prefill(e)
        j = O.argmax_lowest(ref)
        assert j in pairs.values() and ref[j] == ref[tops[b]], b
        assert got[b][j] == got[b][tops[b]], f"item {b}: duplicated rows differ on the device"
        assert int(first[b]) == j, f"item {b}: tie of rows {j} and {tops[b]}, device picked {first[b]}"


# ------------------------------------------------------------------ decode budget (moss/model.cpp, run)
def test_greedy_stops_at_decode_budget(small):
    """A greedy run given the generation budget of dec_decode_budget stops
    exactly there, with the oracle's tokens."""
    from speech_decoder_gb300.binding import decode_budget
    spec, w = small
    prompt = synth.Prompt(9, 70, 6)
    emb, _ = prompt_rows(spec, w, prompt, seed=51)
    ceiling = prompt.T + 300
    budget = decode_budget(prompt.n_audio, prompt.T, ceiling)
    assert budget == O.decode_budget(prompt.n_audio, prompt.T, ceiling) == 268
    dec = make(spec, w, max_ctx=ceiling, max_new=300)
    dec.prefill(emb)
    ids, trunc = dec.generate(budget)
    ref, rtrunc, hist = O.greedy(O.Oracle(spec, w, ceiling), emb, budget, keep_logits=True)
    assert len(ids) == budget and trunc and rtrunc
    # tokens equal the oracle's up to the first tie inside the observed error:
    # at a difference, replay the GPU's tokens up to it for its logits there
    k = next((i for i, (a, b) in enumerate(zip(ids, ref)) if a != b), None)
    if k is not None:
        dec.prefill(emb)
        for i in range(k):
            dec.step(ids[i])
        got = dec.logits(1)[0]
        assert token_ok(ids[k], hist[k], got), f"token {k}: GPU {ids[k]}, oracle {ref[k]}"
    dec.close()
