"""Parity at the full sizes of the benchmark workloads, through the same calls
and decoder configuration the benchmark times (prefill from token ids and
encoder rows on the device, then the CUDA-graph greedy loop).

For every workload:

* the greedy run's tokens come from ``dec_generate`` (``dec_generate_batch``);
* the oracle runs ONE pass over the prompt rows followed by the embeddings of
  the tokens the GPU generated, so its row T - 1 + i holds the logits that
  predict generated token i (fed the GPU's own tokens: no oracle input comes
  from anything but the seeded inputs and the ids);
* the GPU's logits of every position come from a replay of the same tokens
  through ``dec_step`` (``dec_step_batch``), one step at a time, reading
  ``dec_debug_logits`` after each; each replayed step must return exactly the
  token the greedy loop produced (same kernels, same arithmetic);
* every position's logits must be within 2e-2 relative error of the
  oracle's (max |gpu - ref| / max |ref|), and every GPU token must be the
  oracle's argmax unless the oracle's top-2 gap at that position lies within
  twice the logit error observed there (a tie inside the bf16 error).

The 8015-row workload is checked twice: the full prompt with two blocks over
all 128 steps, and all 28 blocks teacher-forced for four steps.  The batched
workload checks six items spread over the length range (the two shortest,
two of median length, the two longest) against the oracle, and a second run
with an end-of-stream id against the first: every row must stop exactly at
its first end-of-stream token, with the tokens before it unchanged.
"""
import numpy as np
import pytest

import oracle as O
from _parity import rel_err, token_ok
from speech_decoder_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from speech_decoder_gb300 import build
    build.build()


def make(spec, w, **kw):
    from speech_decoder_gb300.binding import Decoder
    return Decoder(spec, w, **kw)


def item_rows(spec, w, prompt, seed, item):
    p = synth.prompt_inputs(spec, prompt, seed=seed, item=item)
    emb = O.assemble_prompt(w["embed"], p["ids"], p["audio"], p["prefix_len"])
    return p, emb


def oracle_sequence(spec, w, emb, gpu_ids):
    """Oracle logits for the prompt's last row and every generated position,
    fed the GPU's own tokens; returns float64 [len(gpu_ids), vocab]."""
    T = emb.shape[0]
    rows = [np.asarray(emb, np.float64)]
    if len(gpu_ids) > 1:
        rows.append(np.asarray(w["embed"][np.asarray(gpu_ids[:-1], np.int64)], np.float64))
    ext = np.concatenate(rows)
    orc = O.Oracle(spec, w, ext.shape[0])
    x = orc.forward(ext)[T - 1:]
    y = O.rms_norm(x, w["final_norm"], spec.rms_eps)
    return O.linear(y, w["embed"])


class Tally:
    """Worst relative logit error and tie-bound token mismatches of one run."""

    def __init__(self, name):
        self.name, self.worst, self.ties, self.n = name, 0.0, 0, 0

    def check(self, i, tok, got, ref):
        e = rel_err(got, ref)
        self.worst = max(self.worst, e)
        self.n += 1
        assert e <= TOL, f"{self.name} position {i}: logits rel err {e:.3e}"
        assert token_ok(tok, ref, got), (f"{self.name} position {i}: GPU {tok}, oracle {O.argmax_lowest(ref)}, "
                                         f"gap {float(ref[O.argmax_lowest(ref)] - ref[tok]):.3e}")
        self.ties += int(tok != O.argmax_lowest(ref))

    def report(self):
        print(f"{self.name}: {self.n} positions, worst logits rel err {self.worst:.2e}, "
              f"{self.ties} tie-bound token mismatches")


def run_single(wl, spec, n_steps):
    import torch
    w = synth.model_weights(spec, seed=wl.seed)
    prompt = wl.prompts[0]
    p, emb = item_rows(spec, w, prompt, wl.seed, 0)
    max_new = n_steps + 1
    dec = make(spec, w, max_ctx=prompt.T + max_new, max_batch=1, max_tokens=prompt.T, max_new=max_new,
               eos_id=wl.eos_id)
    ids_dev = torch.from_numpy(np.asarray(p["ids"], np.int32)).cuda()
    audio_dev = torch.from_numpy(np.asarray(p["audio"], np.float32)).cuda()
    first = dec.prefill_ids(ids_dev, audio_dev, int(p["prefix_len"]))
    got = [dec.logits(1)[0]]
    dec.prefill_ids(ids_dev, audio_dev, int(p["prefix_len"]))
    ids, trunc = dec.generate(max_new)
    assert ids[0] == first and len(ids) == max_new and trunc
    # replay the greedy run one step at a time for every position's logits
    dec.prefill_ids(ids_dev, audio_dev, int(p["prefix_len"]))
    for i in range(len(ids) - 1):
        nxt = dec.step(ids[i])
        assert nxt == ids[i + 1], f"replayed step {i} gave {nxt}, the greedy loop {ids[i + 1]}"
        got.append(dec.logits(1)[0])
    dec.close()
    ref = oracle_sequence(spec, w, emb, ids)
    t = Tally(wl.name if spec is wl.model else f"{wl.name} ({spec.n_layers} blocks)")
    for i, tok in enumerate(ids):
        t.check(i, tok, got[i], ref[i])
    t.report()


def test_qwen3_06b_t153_full():
    wl = synth.workload("qwen3-0.6b-t153")
    run_single(wl, wl.model, wl.steps)


def test_qwen3_17b_t152_full():
    wl = synth.workload("qwen3-1.7b-t152")
    run_single(wl, wl.model, wl.steps)


def test_qwen3_17b_t8015_two_blocks():
    wl = synth.workload("qwen3-1.7b-t8015")
    m = wl.model
    spec = synth.ModelSpec("qwen3-1.7b-shape-2blocks", 2, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.ffn,
                           m.vocab)
    run_single(wl, spec, wl.steps)


@pytest.mark.slow
def test_qwen3_17b_t8015_teacher_forced():
    """All 28 blocks at the full 8015-row prompt, then four steps fed the
    oracle's tokens on both sides."""
    import torch
    wl = synth.workload("qwen3-1.7b-t8015")
    spec = wl.model
    w = synth.model_weights(spec, seed=wl.seed)
    prompt = wl.prompts[0]
    p, emb = item_rows(spec, w, prompt, wl.seed, 0)
    steps = 4
    dec = make(spec, w, max_ctx=prompt.T + steps + 1, max_batch=1, max_tokens=prompt.T, max_new=steps + 1)
    g_tok = dec.prefill_ids(torch.from_numpy(np.asarray(p["ids"], np.int32)).cuda(),
                            torch.from_numpy(np.asarray(p["audio"], np.float32)).cuda(), int(p["prefix_len"]))
    got = dec.logits(1)[0]
    orc = O.Oracle(spec, w, prompt.T + steps + 1)
    ref = orc.prefill(emb)
    t = Tally(f"{wl.name} teacher-forced")
    t.check(0, g_tok, got, ref)
    tok = O.argmax_lowest(ref)
    for i in range(steps):
        g_tok = dec.step(tok)
        got = dec.logits(1)[0]
        ref = orc.step(tok)
        t.check(i + 1, g_tok, got, ref)
        tok = O.argmax_lowest(ref)
    dec.close()
    t.report()


def _batch_inputs(wl, spec):
    import torch
    B = wl.batch
    items = [synth.prompt_inputs(spec, pr, seed=wl.seed, item=i) for i, pr in enumerate(wl.prompts)]
    ids_np = np.concatenate([it["ids"] for it in items]).astype(np.int32)
    audio_np = np.concatenate([it["audio"] for it in items]).astype(np.float32)
    cu_ids = np.zeros(B + 1, np.int32)
    cu_ids[1:] = np.cumsum([len(it["ids"]) for it in items])
    cu_au = np.zeros(B + 1, np.int32)
    cu_au[1:] = np.cumsum([it["audio"].shape[0] for it in items])
    pre_lens = np.array([it["prefix_len"] for it in items], np.int32)
    ids_dev = torch.from_numpy(ids_np).cuda()
    audio_dev = torch.from_numpy(audio_np).cuda()

    def prefill(dec):
        return dec.prefill_ids_batch_ptr(ids_dev.data_ptr(), cu_ids, audio_dev.data_ptr(), cu_au, pre_lens, 1)

    return prefill, (ids_dev, audio_dev)


def test_qwen3_17b_b32_full():
    wl = synth.workload("qwen3-1.7b-b32")
    spec = wl.model
    w = synth.model_weights(spec, seed=wl.seed)
    B = wl.batch
    Ts = [pr.T for pr in wl.prompts]
    max_new = wl.steps + 1
    order = sorted(range(B), key=lambda i: (Ts[i], i))
    checked = sorted(set(order[:2] + order[B // 2 - 1:B // 2 + 1] + order[-2:]))
    assert len(checked) == 6
    prefill, keep = _batch_inputs(wl, spec)
    dec = make(spec, w, max_ctx=max(Ts) + max_new, max_batch=B, max_tokens=sum(Ts), max_new=max_new, eos_id=-1)
    first = prefill(dec)
    got = {b: [dec.logits(B)[b]] for b in checked}
    prefill(dec)
    out = dec.generate_batch(max_new, B)
    for b in range(B):
        assert len(out[b][0]) == max_new and out[b][1] and out[b][0][0] == first[b]
    # replay all rows step by step; keep the checked items' logits
    prefill(dec)
    for i in range(max_new - 1):
        nxt = dec.step_batch(np.array([out[b][0][i] for b in range(B)], np.int32))
        assert [int(v) for v in nxt] == [out[b][0][i + 1] for b in range(B)], f"replayed step {i}"
        lg = dec.logits(B)
        for b in checked:
            got[b].append(lg[b].copy())
    dec.close()
    ref_best = {}
    for b in checked:
        _, emb = item_rows(spec, w, wl.prompts[b], wl.seed, b)
        ref = oracle_sequence(spec, w, emb, out[b][0])
        t = Tally(f"b32 item {b} (T={Ts[b]})")
        for i, tok in enumerate(out[b][0]):
            t.check(i, tok, got[b][i], ref[i])
        t.report()
        ref_best[b] = [O.argmax_lowest(r) for r in ref]
        del ref, got[b]

    # per-item end-of-stream masking at full size: the most frequent generated
    # token (after the first position) becomes the end-of-stream id
    gen = np.concatenate([np.asarray(out[b][0][1:]) for b in range(B)])
    vals, counts = np.unique(gen, return_counts=True)
    eos = int(vals[np.argmax(counts)])
    want, stops = [], []
    for b in range(B):
        seq = out[b][0]
        k = seq.index(eos) if eos in seq else len(seq)
        want.append((seq[:k], k == len(seq)))
        stops.append(k)
    assert len(set(stops)) > 2 and min(stops) < max_new, f"end-of-stream id {eos} stops too few rows: {stops}"
    dec = make(spec, w, max_ctx=max(Ts) + max_new, max_batch=B, max_tokens=sum(Ts), max_new=max_new, eos_id=eos)
    prefill(dec)
    res = dec.generate_batch(max_new, B)
    dec.close()
    for b in range(B):
        assert res[b][0] == want[b][0], f"item {b}: stopped after {len(res[b][0])} ids, expected {len(want[b][0])}"
        assert res[b][1] == want[b][1], f"item {b}: truncated flag"
    # the oracle-checked items stop where the oracle's greedy loop with this
    # end-of-stream id stops (its argmax sequence, fed the same tokens, up to
    # the first tie-bound difference)
    for b in checked:
        best, seq = ref_best[b], out[b][0]
        diff = next((i for i in range(len(seq)) if seq[i] != best[i]), len(seq))
        o_stop = best.index(eos) if eos in best else len(best)
        if o_stop <= diff:
            assert stops[b] == o_stop, f"item {b}: GPU stops after {stops[b]} ids, the oracle after {o_stop}"
    print(f"b32 end-of-stream id {eos}: rows stop after {sorted(stops)} ids")
