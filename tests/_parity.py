"""Helpers shared by the GPU parity tests (oracle side and comparison rules)."""
import numpy as np

import oracle as O
from speech_decoder_gb300 import synth


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max_i |got_i - ref_i| / max_i |ref_i| (per row, the worst row)."""
    got = np.atleast_2d(np.asarray(got, np.float64))
    ref = np.atleast_2d(np.asarray(ref, np.float64))
    return float(np.max(np.max(np.abs(got - ref), axis=1) / np.max(np.abs(ref), axis=1)))


def token_ok(gpu_tok: int, ref_logits: np.ndarray, got_logits: np.ndarray) -> bool:
    """The GPU's argmax must be the oracle's, unless the oracle's top-2 gap is
    within twice the observed logit error (a tie inside the error bound)."""
    ref_tok = O.argmax_lowest(ref_logits)
    if gpu_tok == ref_tok:
        return True
    bound = 2.0 * float(np.max(np.abs(np.asarray(got_logits, np.float64) - ref_logits)))
    return float(ref_logits[ref_tok] - ref_logits[gpu_tok]) <= bound


def prompt_rows(spec, weights, prompt, seed=0, item=0):
    p = synth.prompt_inputs(spec, prompt, seed=seed, item=item)
    emb = O.assemble_prompt(weights["embed"], p["ids"], p["audio"], p["prefix_len"])
    return emb.astype(np.float32), p


def teacher_forced(dec, orc, emb, steps, tol):
    """Prefill both sides, then feed the oracle's greedy tokens to both.
    Returns (worst relative logit error, number of tie-bound token mismatches)."""
    worst, ties = 0.0, 0
    g_tok = dec.prefill(emb)
    ref = orc.prefill(emb.astype(np.float64))
    got = dec.logits(1)[0]
    e = rel_err(got, ref)
    worst = max(worst, e)
    assert e <= tol, f"prefill logits rel err {e:.3e} > {tol}"
    assert token_ok(g_tok, ref, got), f"prefill token {g_tok} vs oracle {O.argmax_lowest(ref)}"
    ties += g_tok != O.argmax_lowest(ref)
    tok = O.argmax_lowest(ref)
    for i in range(steps):
        g_tok = dec.step(tok)
        ref = orc.step(tok)
        got = dec.logits(1)[0]
        e = rel_err(got, ref)
        worst = max(worst, e)
        assert e <= tol, f"step {i} logits rel err {e:.3e} > {tol}"
        assert token_ok(g_tok, ref, got), f"step {i} token {g_tok} vs oracle {O.argmax_lowest(ref)}"
        ties += g_tok != O.argmax_lowest(ref)
        tok = O.argmax_lowest(ref)
    return worst, ties
