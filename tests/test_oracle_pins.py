"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong head mapping) fails it.
None of them retypes the oracle's own formula: they use closed-form values,
invariants, special cases and a brute-force evaluator on tiny inputs.
"""
import math

import numpy as np
import pytest

import oracle as O
from speech_decoder_gb300 import synth


# ------------------------------------------------------------------ RMSNorm
def test_rms_norm_unit_rms_per_row():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 96)) * np.array([[0.01], [1.0], [3.0], [100.0], [7.0]])
    y = O.rms_norm(x, np.ones(96), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-12)


def test_rms_norm_closed_forms():
    # constant row c: mean(x^2) = c^2 -> c / sqrt(c^2 + eps)
    y = O.rms_norm(np.full((1, 8), 3.0), np.ones(8), 7.0)
    assert np.allclose(y, 3.0 / 4.0, atol=0, rtol=1e-15)
    # zero row stays zero (eps keeps it finite)
    assert np.all(O.rms_norm(np.zeros((1, 4)), np.ones(4), 1e-6) == 0.0)
    # the weight scales elementwise
    w = np.array([1.0, -2.0, 0.5, 0.0])
    y = O.rms_norm(np.array([[2.0, 2.0, 2.0, 2.0]]), w, 0.0)
    assert np.array_equal(y, w[None, :])


def test_rms_norm_is_per_head_on_reshaped_qk():
    # the Q/K norm runs over head_dim per head: two heads with very different
    # scales both come out with unit RMS
    rng = np.random.default_rng(2)
    q = rng.standard_normal((3, 2, 16)) * np.array([1e-3, 1e3])[None, :, None]
    y = O.rms_norm(q, np.ones(16), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-12)


# ------------------------------------------------------------------ linear
def test_linear_orientation_out_in():
    W = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])      # [out=2, in=3]
    assert np.array_equal(O.linear(np.array([[1.0, 0.0, -1.0]]), W), [[-2.0, -2.0]])
    assert np.array_equal(O.linear(np.array([[1.0, 1.0, 1.0]]), W), [[6.0, 15.0]])


# ------------------------------------------------------------------ RoPE
COS1, SIN1 = 0.5403023058681398, 0.8414709848078965      # cos(1), sin(1)


def _unit(d, i):
    z = np.zeros((1, 1, d))
    z[0, 0, i] = 1.0
    return z


def test_rope_position_zero_is_identity():
    z = np.random.default_rng(3).standard_normal((1, 4, 64))
    assert np.array_equal(O.rope_neox(z, np.array([0]), 1e6), z)


def test_rope_neox_pairing_and_direction():
    d = 128
    # frequency index 0 has angle = position; e_0 at p=1 goes to (cos 1) e_0 + (sin 1) e_{d/2}
    y = O.rope_neox(_unit(d, 0), np.array([1]), 1e6)[0, 0]
    exp = np.zeros(d)
    exp[0], exp[d // 2] = COS1, SIN1
    assert np.allclose(y, exp, atol=1e-15)
    # e_{d/2} at p=1 goes to (-sin 1) e_0 + (cos 1) e_{d/2}
    y = O.rope_neox(_unit(d, d // 2), np.array([1]), 1e6)[0, 0]
    exp = np.zeros(d)
    exp[0], exp[d // 2] = -SIN1, COS1
    assert np.allclose(y, exp, atol=1e-15)


@pytest.mark.parametrize("d,i", [(128, 32), (64, 16)])
def test_rope_frequency_exponent(d, i):
    # theta^(-2i/d) with theta = 1e6 and 2i/d = 1/2 is exactly 1e-3, so at
    # position 1000 pair i turns by exactly one radian
    y = O.rope_neox(_unit(d, i), np.array([1000]), 1e6)[0, 0]
    assert abs(y[i] - COS1) < 1e-12 and abs(y[i + d // 2] - SIN1) < 1e-12
    assert np.count_nonzero(np.abs(y) > 1e-12) == 2


def test_rope_preserves_head_norm_and_relative_position():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 3, 128))
    k = rng.standard_normal((1, 3, 128))
    for p in (1, 17, 4097, 8142):
        qr = O.rope_neox(q, np.array([p]), 1e6)
        assert np.allclose(np.linalg.norm(qr, axis=-1), np.linalg.norm(q, axis=-1), rtol=1e-13)
    # <R_p q, R_r k> depends only on p - r
    dots = []
    for p, r in ((10, 3), (110, 103), (5007, 5000)):
        qr = O.rope_neox(q, np.array([p]), 1e6)
        kr = O.rope_neox(k, np.array([r]), 1e6)
        dots.append(np.sum(qr * kr, axis=-1))
    assert np.allclose(dots[0], dots[1], atol=1e-10) and np.allclose(dots[0], dots[2], atol=1e-9)


# ------------------------------------------------------------------ attention
def test_attention_single_key_returns_v():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 32))
    K = rng.standard_normal((1, 2, 32))
    V = rng.standard_normal((1, 2, 32))
    out = O.attention(q, K, V, np.array([0]))
    assert np.allclose(out[0], np.repeat(V[0], 2, axis=0), atol=1e-15)


def test_attention_identical_keys_average_v():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 2, 16))
    K = np.tile(rng.standard_normal((1, 1, 16)), (5, 1, 1))
    V = rng.standard_normal((5, 1, 16))
    out = O.attention(q, K, V, np.array([4]))
    assert np.allclose(out[0, 0], V[:, 0].mean(axis=0), atol=1e-14)
    assert np.allclose(out[0, 1], V[:, 0].mean(axis=0), atol=1e-14)


def test_attention_scale_closed_form():
    # score of key 0 = (ln 3 e_0) . (sqrt(d) e_0) / sqrt(d) = ln 3, key 1 scores 0:
    # softmax weights are exactly 3/4 and 1/4
    d = 64
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = math.log(3.0)
    K = np.zeros((2, 1, d))
    K[0, 0, 0] = math.sqrt(d)
    V = np.zeros((2, 1, d))
    V[0, 0, :] = 1.0
    V[1, 0, :] = -3.0
    out = O.attention(q, K, V, np.array([1]))
    assert np.allclose(out[0, 0], 0.75 * 1.0 + 0.25 * -3.0, atol=1e-14)


def test_attention_causal():
    rng = np.random.default_rng(7)
    T = 6
    q = rng.standard_normal((T, 2, 8))
    K = rng.standard_normal((T, 1, 8))
    V = rng.standard_normal((T, 1, 8))
    out = O.attention(q, K, V, np.arange(T))
    assert np.allclose(out[0, :, :], V[0, 0][None, :], atol=1e-15)      # row 0 sees only key 0
    K2, V2 = K.copy(), V.copy()
    K2[4:] += 10.0
    V2[4:] -= 10.0
    out2 = O.attention(q, K2, V2, np.arange(T))
    assert np.array_equal(out[:4], out2[:4])                              # future keys invisible


def test_gqa_equals_mha_with_repeated_kv():
    rng = np.random.default_rng(8)
    T, nq, nkv, d = 5, 6, 2, 16
    q = rng.standard_normal((T, nq, d))
    K = rng.standard_normal((T, nkv, d))
    V = rng.standard_normal((T, nkv, d))
    rep = nq // nkv
    # HF repeat_kv: KV head g serves query heads g*rep .. g*rep + rep - 1
    Kr = np.repeat(K, rep, axis=1)
    Vr = np.repeat(V, rep, axis=1)
    assert np.allclose(O.attention(q, K, V, np.arange(T)), O.attention(q, Kr, Vr, np.arange(T)),
                       atol=1e-14)


# ------------------------------------------------------------------ SwiGLU
def test_perception_projection_closed_forms():
    """W = 0 gives the bias on every row; a one-hot W row copies one input
    column; bias is per output feature (not per row)."""
    rng = np.random.default_rng(21)
    enc = rng.standard_normal((5, 8))
    bias = rng.standard_normal(6)
    assert np.array_equal(O.perception_projection(enc, np.zeros((6, 8)), bias), np.tile(bias, (5, 1)))
    W = np.zeros((6, 8))
    W[2, 7] = 1.0
    W[4, 0] = -2.0
    y = O.perception_projection(enc, W, np.zeros(6))
    assert np.array_equal(y[:, 2], enc[:, 7]) and np.array_equal(y[:, 4], -2.0 * enc[:, 0])
    assert np.count_nonzero(y[:, [0, 1, 3, 5]]) == 0


def test_silu_values():
    assert O.silu(np.array(0.0)) == 0.0
    assert abs(O.silu(np.array(1.0)) - 0.7310585786300049) < 1e-15
    assert abs(O.silu(np.array(-1.0)) + 0.2689414213699951) < 1e-15
    assert abs(O.silu(np.array(40.0)) - 40.0) < 1e-12


def test_swiglu_gate_up_roles():
    # gate reads x0, up reads x1, down is the identity on the single feature
    Wg = np.array([[1.0, 0.0]])
    Wu = np.array([[0.0, 1.0]])
    Wd = np.array([[1.0], [0.0]])
    y = O.swiglu_ffn(np.array([[1.0, 2.0]]), Wg, Wu, Wd)
    assert abs(y[0, 0] - 2.0 * 0.7310585786300049) < 1e-15   # silu(1) * 2, not silu(2) * 1
    assert y[0, 1] == 0.0


# ------------------------------------------------------------------ argmax
def test_argmax_lowest_index_on_ties():
    v = np.zeros(100)
    v[37] = 5.0
    assert O.argmax_lowest(v) == 37
    v[12] = 5.0
    v[90] = 5.0
    assert O.argmax_lowest(v) == 12
    v = np.full(10, -3.0)
    assert O.argmax_lowest(v) == 0
    with pytest.raises(ValueError):
        O.argmax_lowest(np.array([1.0, np.nan]))


# ------------------------------------------------------------------ model level
def _tiny(**kw):
    spec = synth.small_spec(**kw)
    return spec, synth.model_weights(spec, seed=kw.get("seed_", 0), threads=4)


def test_prompt_assembly_order():
    E = np.arange(10 * 3, dtype=np.float32).reshape(10, 3)
    audio = -np.ones((2, 3), np.float32)
    x = O.assemble_prompt(E, np.array([4, 1, 7]), audio, prefix_len=1)
    assert np.array_equal(x, np.stack([E[4], audio[0], audio[1], E[1], E[7]]))


def test_zero_out_projections_make_block_identity():
    spec, w = _tiny(n_layers=1)
    for name in ("o", "down"):
        w["layers"][0][name] = np.zeros_like(w["layers"][0][name])
    orc = O.Oracle(spec, w, 16)
    x = np.random.default_rng(9).standard_normal((5, spec.hidden))
    assert np.array_equal(orc.forward(x), x)


def test_tied_head_reads_embedding_rows():
    spec = synth.small_spec(n_layers=1, hidden=16, n_heads=2, n_kv_heads=1, head_dim=8, ffn=128,
                            vocab=16, norm_init="ones")
    w = synth.model_weights(spec, threads=2)
    w["embed"] = np.eye(16, dtype=np.float32) * 2.0
    orc = O.Oracle(spec, w, 4)
    x = np.random.default_rng(10).standard_normal(16)
    y = x / np.sqrt(np.mean(x * x) + spec.rms_eps)
    assert np.allclose(orc.head(x), 2.0 * y, atol=1e-14)


def test_prefill_then_step_equals_longer_prefill():
    spec, w = _tiny()
    rng = np.random.default_rng(11)
    emb = rng.standard_normal((7, spec.hidden))
    tok = 123
    a = O.Oracle(spec, w, 16)
    a.prefill(emb)
    la = a.step(tok)
    b = O.Oracle(spec, w, 16)
    lb = b.prefill(np.concatenate([emb, w["embed"][tok][None, :].astype(np.float64)]))
    assert np.allclose(la, lb, atol=1e-11, rtol=0)
    for l in range(spec.n_layers):
        assert np.allclose(a.K[l][:8], b.K[l][:8], atol=1e-12)


def test_chunked_forward_equals_single_forward():
    """Chunked prefill (rows fed in pieces against the growing KV cache) gives
    the hidden states of a single pass over all rows: the pin for the CUDA
    path's dec_prefill_chunk."""
    spec, w = _tiny()
    rng = np.random.default_rng(13)
    emb = rng.standard_normal((23, spec.hidden))
    one = O.Oracle(spec, w, 32)
    h1 = one.forward(emb)
    chunked = O.Oracle(spec, w, 32)
    parts = [chunked.forward(emb[a:b]) for a, b in ((0, 5), (5, 16), (16, 23))]
    assert np.allclose(np.concatenate(parts), h1, atol=1e-11, rtol=0)
    for l in range(spec.n_layers):
        assert np.allclose(chunked.K[l][:23], one.K[l][:23], atol=1e-12)


def test_model_is_causal():
    spec, w = _tiny()
    rng = np.random.default_rng(12)
    emb = rng.standard_normal((9, spec.hidden))
    h1 = O.Oracle(spec, w, 16).forward(emb)
    emb2 = emb.copy()
    emb2[6:] = rng.standard_normal((3, spec.hidden))
    h2 = O.Oracle(spec, w, 16).forward(emb2)
    assert np.array_equal(h1[:6], h2[:6]) and not np.allclose(h1[6:], h2[6:])


def test_model_gqa_equals_mha_with_repeated_kv_weights():
    spec, w = _tiny(n_heads=4, n_kv_heads=2)
    mha = synth.small_spec(n_heads=4, n_kv_heads=4)
    w2 = {"embed": w["embed"], "final_norm": w["final_norm"], "layers": []}
    d = spec.head_dim
    for L in w["layers"]:
        L2 = dict(L)
        for name in ("k", "v"):
            heads = L[name].reshape(2, d, spec.hidden)
            L2[name] = np.repeat(heads, 2, axis=0).reshape(4 * d, spec.hidden)
        w2["layers"].append(L2)
    emb = np.random.default_rng(13).standard_normal((6, spec.hidden))
    a = O.Oracle(spec, w, 8).prefill(emb)
    b = O.Oracle(mha, w2, 8).prefill(emb)
    assert np.allclose(a, b, atol=1e-12)


# ------------------------------------------------------------------ brute force
def _brute_logits(spec, w, emb):
    """Scalar Python evaluation of the whole model (explicit loops, math module,
    full score matrix, explicit KV repetition)."""
    H, nq, nkv, d, F = spec.hidden, spec.n_heads, spec.n_kv_heads, spec.head_dim, spec.ffn
    eps, theta = spec.rms_eps, spec.rope_theta
    T = len(emb)
    X = [[float(v) for v in row] for row in emb]

    def norm(vec, wt):
        r = math.sqrt(sum(v * v for v in vec) / len(vec) + eps)
        return [vec[j] / r * float(wt[j]) for j in range(len(vec))]

    def mv(Wm, vec):
        return [sum(float(Wm[o][i]) * vec[i] for i in range(len(vec))) for o in range(len(Wm))]

    def rot(vec, p):
        out = list(vec)
        for i in range(d // 2):
            ang = p / (theta ** (2.0 * i / d))
            c, s = math.cos(ang), math.sin(ang)
            out[i] = vec[i] * c - vec[i + d // 2] * s
            out[i + d // 2] = vec[i + d // 2] * c + vec[i] * s
        return out

    for L in w["layers"]:
        Q, K, V = [], [], []
        for t in range(T):
            xn = norm(X[t], L["attn_norm"])
            qf, kf, vf = mv(L["q"], xn), mv(L["k"], xn), mv(L["v"], xn)
            Q.append([rot(norm(qf[h * d:(h + 1) * d], L["q_norm"]), t) for h in range(nq)])
            ks = [rot(norm(kf[g * d:(g + 1) * d], L["k_norm"]), t) for g in range(nkv)]
            vs = [vf[g * d:(g + 1) * d] for g in range(nkv)]
            # explicit repetition of KV heads to query heads
            K.append([ks[h * nkv // nq] for h in range(nq)])
            V.append([vs[h * nkv // nq] for h in range(nq)])
        newX = []
        for t in range(T):
            o = []
            for h in range(nq):
                sc = [sum(Q[t][h][j] * K[u][h][j] for j in range(d)) / math.sqrt(d) for u in range(t + 1)]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                z = sum(e)
                o += [sum(e[u] / z * V[u][h][j] for u in range(t + 1)) for j in range(d)]
            x1 = [X[t][i] + v for i, v in enumerate(mv(L["o"], o))]
            xn = norm(x1, L["ffn_norm"])
            g, u = mv(L["gate"], xn), mv(L["up"], xn)
            hdn = [g[j] / (1.0 + math.exp(-g[j])) * u[j] for j in range(F)]
            newX.append([x1[i] + v for i, v in enumerate(mv(L["down"], hdn))])
        X = newX
    y = norm(X[-1], w["final_norm"])
    return np.array(mv(w["embed"], y))


def test_brute_force_tiny_model():
    spec = synth.small_spec(n_layers=2, hidden=12, n_heads=4, n_kv_heads=2, head_dim=6, ffn=10,
                            vocab=9)
    w = synth.model_weights(spec, seed=5, threads=2)
    emb = np.random.default_rng(14).standard_normal((4, 12))
    ref = _brute_logits(spec, w, emb)
    got = O.Oracle(spec, w, 8).prefill(emb)
    assert np.allclose(got, ref, atol=1e-12, rtol=0)


# ------------------------------------------------------------------ greedy loop
class _Scripted:
    """A stand-in model that returns scripted argmax tokens."""

    def __init__(self, toks, capacity, T):
        self.toks = list(toks)
        self.capacity = capacity
        self.n_past = 0
        self.T = T

    def _logits(self):
        v = np.zeros(50)
        v[self.toks.pop(0)] = 1.0
        return v

    def prefill(self, emb):
        self.n_past = self.T
        return self._logits()

    def step(self, tok):
        self.n_past += 1
        return self._logits()


def test_greedy_stops_at_eos_and_strips_it():
    ids, trunc, _ = O.greedy(_Scripted([5, 6, 7, 3, 9, 9], 100, 4), None, max_new=256, eos_id=3)
    assert ids == [5, 6, 7] and not trunc


def test_greedy_budget_counts_prefill_token():
    ids, trunc, _ = O.greedy(_Scripted([1] * 20, 100, 4), None, max_new=5, eos_id=3)
    assert ids == [1] * 5 and trunc


def test_greedy_stops_when_kv_full():
    # prompt of 4 in a 7-slot cache: three steps write slots 4, 5, 6
    ids, trunc, _ = O.greedy(_Scripted([2] * 20, 7, 4), None, max_new=256, eos_id=3)
    assert ids == [2] * 4 and trunc


def test_greedy_eos_first_token():
    ids, trunc, _ = O.greedy(_Scripted([3, 4], 100, 4), None, max_new=256, eos_id=3)
    assert ids == [] and not trunc


# ------------------------------------------------------------------ decode budget
# moss/model.cpp (transcribe-cpp-sys 0.4.1), run: the budget asked for is twice
# the audio rows plus 128, the 256-token generation reserve is the floor, the
# context left after the prompt the cap; a prompt that cannot take the reserve
# is rejected before.  Values worked by hand from that reading.
@pytest.mark.parametrize("n_audio,T,ceiling,want", [
    (138, 152, 8192, 404),        # the JFK prompt: 2 * 138 + 128 = 404 (above the floor, far below the cap)
    (50, 65, 8192, 256),          # 2 * 50 + 128 = 228 < 256: the reserve is the floor
    (64, 79, 8192, 256),          # 2 * 64 + 128 = 256 exactly
    (65, 80, 8192, 258),          # one audio row above that: two more tokens
    (4000, 4015, 8192, 4177),     # 8128 asked, 8192 - 4015 = 4177 left: the cap
    (8000, 8015, 8271, 256),      # cap = 256 = the floor: the gate's boundary case
])
def test_decode_budget_worked_values(n_audio, T, ceiling, want):
    assert O.decode_budget(n_audio, T, ceiling) == want


def test_decode_budget_gate_and_invariants():
    with pytest.raises(ValueError):
        O.decode_budget(8000, 8015, 8270)        # 8015 + 256 > 8270: input too long
    with pytest.raises(ValueError):
        O.decode_budget(-1, 10, 1000)
    for n in range(0, 3000, 7):
        T = n + 15
        b = O.decode_budget(n, T, 4096)
        assert 256 <= b and T + b <= 4096
        # more audio never lowers the budget for the same prompt length
        assert O.decode_budget(n + 1, T, 4096) >= b


# ------------------------------------------------------------------ synth
def test_round_bf16_ties_to_even_and_exact():
    a = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], np.float32)
    synth.round_bf16(a)
    assert list(a) == [1.0, 1.0, 1.0 + 2 ** -6, -2.5, 1.0]
    assert list(synth.bf16_bits(np.array([1.0, -2.0], np.float32))) == [0x3F80, 0xC000]


def test_synth_is_deterministic_and_thread_independent():
    spec = synth.small_spec()
    a = synth.model_weights(spec, seed=3, threads=1)
    b = synth.model_weights(spec, seed=3, threads=8)
    assert np.array_equal(a["embed"], b["embed"])
    assert np.array_equal(a["layers"][1]["down"], b["layers"][1]["down"])
    p = synth.prompt_inputs(spec, synth.Prompt(9, 20, 5), seed=0, item=2)
    assert p["ids"].shape == (14,) and p["audio"].shape == (20, 256)
