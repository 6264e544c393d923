"""Plain fp64 CPU oracle of the Qwen3-style speech-LLM decoder.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call
this module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library; the
only thing both sides take from a common module is the seeded input data
(``speech_decoder_gb300.synth``), which holds none of the arithmetic below.

Every step is written out in the order the pages state it, in float64, with
numpy's matmul as the only library primitive.  Sources (page titles as they
appear on docs.rs):

* qwen3_asr/decoder.cpp (transcribe-cpp-sys 0.2.0), file header: the block is
  pre-LN RMSNorm, GQA with per-head Q/K RMSNorm, NeoX RoPE at theta = 1e6,
  KV write/read, SwiGLU on a packed gate_up projection.
* same page, build_prefill_graph: token-embedding gather, audio injection by
  3-way concat (prefix | enc_out | suffix), block stack, final RMSNorm,
  tied lm_head on the last position.
* same page, build_step_graph: one token at position cur_past, KV written at
  index cur_past, final RMSNorm, tied lm_head, argmax of the logits directly
  (no softmax: it would not change which logit is largest).
* qwen3_asr/model.cpp (transcribe-cpp-sys 0.2.0), run: causal prefill mask
  (key c visible to query r iff c <= r), host argmax with strict '>' (lowest
  index wins a tie), the greedy loop (stop at EOS, at max_new generated ids
  counting the prefill's token, or when the KV width is full), truncation
  when no EOS was produced, and stripping of a trailing EOS.

Readings where the pages are silent (also listed in the design notes):
attention scale 1/sqrt(head_dim); Q/K-norm weight is one [head_dim] vector
shared by all heads with the same eps; Q/K-norm before RoPE; RoPE frequency
theta^(-2i/d) with NeoX half-split pairing (i, i + d/2); 1-D positions equal
to the token index (the MRoPE sections coincide for a single position
stream); GQA query head h reads KV head h // (n_heads / n_kv_heads); the
new token's K/V are written before attention so a query sees itself.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------- ops
def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis, then the elementwise weight.

    ggml's rms_norm followed by mul (decoder.cpp, build_step_graph: final
    norm; the same pre-LN norm opens each block): x / sqrt(mean(x^2) + eps) * w.
    """
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(w)


def linear(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    """y = x W^T with W in the [out, in] layout (ggml mul_mat of a weight)."""
    return _f64(x) @ _f64(W).T


def rope_neox(z: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """NeoX rotary embedding (decoder.cpp, file header: NeoX-style RoPE with
    base theta = 1e6).

    z: [T, heads, d]; pos: [T] absolute token positions.  For i < d/2 the
    pair (z_i, z_{i+d/2}) is rotated by the angle pos * theta^(-2i/d).
    """
    z = _f64(z)
    d = z.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=F64)
    inv_freq = np.power(F64(theta), -2.0 * i / d)
    ang = _f64(pos)[:, None] * inv_freq[None, :]             # [T, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a = z[..., :half]
    b = z[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, q_pos: np.ndarray) -> np.ndarray:
    """Causal grouped-query attention.

    q: [T, n_heads, d] at absolute positions q_pos; K, V: [S, n_kv_heads, d]
    for key positions 0..S-1.  Key j is visible to a query at position p iff
    j <= p (the causal mask of qwen3_asr/model.cpp, run; the step mask opens
    [0, cur_past]).  Scores are q.k / sqrt(d); query head h uses KV head
    h // (n_heads / n_kv_heads).
    """
    q, K, V = _f64(q), _f64(K), _f64(V)
    T, nq, d = q.shape
    S, nkv, _ = K.shape
    n_rep = nq // nkv
    scale = 1.0 / np.sqrt(F64(d))
    visible = np.arange(S)[None, :] <= _f64(q_pos)[:, None]  # [T, S]
    out = np.empty((T, nq, d), F64)
    for h in range(nq):
        g = h // n_rep
        s = (q[:, h, :] @ K[:, g, :].T) * scale
        s = np.where(visible, s, -np.inf)
        s = s - np.max(s, axis=1, keepdims=True)
        p = np.exp(s)
        p = p / np.sum(p, axis=1, keepdims=True)
        out[:, h, :] = p @ V[:, g, :]
    return out


def perception_projection(enc: np.ndarray, W: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """The step just before the decoder (canary_qwen/model.cpp, forward shape:
    the perception projection is a linear layer from 1024 to 2048 features
    with a bias): encoder rows enc [T, d_in] to prompt rows W enc + bias, W in
    the [out, in] layout."""
    return linear(enc, W) + _f64(bias)[None, :]


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + exp(-z))."""
    z = _f64(z)
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(xn: np.ndarray, W_gate, W_up, W_down) -> np.ndarray:
    """down( silu(gate(xn)) * up(xn) ).  The pages pack gate and up into one
    matrix (model.cpp, load: pack_gate_up); packing is a layout choice and the
    oracle keeps the two halves separate."""
    return linear(silu(linear(xn, W_gate)) * linear(xn, W_up), W_down)


def argmax_lowest(logits: np.ndarray) -> int:
    """Index of the maximum; on a tie the lowest index wins (strict '>' scan
    of qwen3_asr/model.cpp, run)."""
    v = _f64(logits)
    if np.isnan(v).any():
        raise ValueError("NaN logit")
    # the strict '>' scan keeps the first index that attains the maximum
    return int(np.flatnonzero(v == np.max(v))[0])


def assemble_prompt(embed: np.ndarray, ids: np.ndarray, audio: np.ndarray, prefix_len: int) -> np.ndarray:
    """Audio injection by 3-way concat (decoder.cpp, build_prefill_graph):
    rows = embed[ids[:prefix_len]] | audio | embed[ids[prefix_len:]]."""
    ids = np.asarray(ids)
    pre = _f64(embed[ids[:prefix_len]])
    suf = _f64(embed[ids[prefix_len:]])
    return np.concatenate([pre, _f64(audio), suf], axis=0)


# --------------------------------------------------------------------- model
class Oracle:
    """One sequence of the decoder with its own fp64 KV cache.

    spec: a synth.ModelSpec (only shapes, eps and theta are read);
    weights: synth.model_weights() layout; capacity: KV slots.
    """

    def __init__(self, spec, weights: dict, capacity: int):
        self.spec = spec
        self.w = weights
        self.capacity = int(capacity)
        L, nkv, d = spec.n_layers, spec.n_kv_heads, spec.head_dim
        self.K = [np.zeros((self.capacity, nkv, d), F64) for _ in range(L)]
        self.V = [np.zeros((self.capacity, nkv, d), F64) for _ in range(L)]
        self.n_past = 0
        self.last_hidden = None

    # one decoder block over rows at absolute positions pos (contiguous, ending
    # at the newest token); qwen3_asr/decoder.cpp header
    def block(self, l: int, x: np.ndarray, pos: np.ndarray) -> np.ndarray:
        sp, W = self.spec, self.w["layers"][l]
        T = x.shape[0]
        nq, nkv, d, eps = sp.n_heads, sp.n_kv_heads, sp.head_dim, sp.rms_eps
        xn = rms_norm(x, W["attn_norm"], eps)
        q = linear(xn, W["q"]).reshape(T, nq, d)
        k = linear(xn, W["k"]).reshape(T, nkv, d)
        v = linear(xn, W["v"]).reshape(T, nkv, d)
        q = rms_norm(q, W["q_norm"], eps)
        k = rms_norm(k, W["k_norm"], eps)
        q = rope_neox(q, pos, sp.rope_theta)
        k = rope_neox(k, pos, sp.rope_theta)
        self.K[l][pos] = k
        self.V[l][pos] = v
        S = int(pos[-1]) + 1
        o = attention(q, self.K[l][:S], self.V[l][:S], pos)
        x = x + linear(o.reshape(T, nq * d), W["o"])
        xn = rms_norm(x, W["ffn_norm"], eps)
        return x + swiglu_ffn(xn, W["gate"], W["up"], W["down"])

    def forward(self, x: np.ndarray) -> np.ndarray:
        T = x.shape[0]
        if self.n_past + T > self.capacity:
            raise ValueError("KV capacity exceeded")
        pos = np.arange(self.n_past, self.n_past + T)
        x = _f64(x)
        for l in range(self.spec.n_layers):
            x = self.block(l, x, pos)
        self.n_past += T
        return x

    def head(self, x_row: np.ndarray) -> np.ndarray:
        """Final RMSNorm + tied lm_head (logits = embed . y)."""
        y = rms_norm(x_row, self.w["final_norm"], self.spec.rms_eps)
        self.last_hidden = y
        return linear(y[None, :], self.w["embed"])[0]

    def prefill(self, embeds: np.ndarray) -> np.ndarray:
        """Run all prompt rows; return the last position's logits."""
        x = self.forward(embeds)
        return self.head(x[-1])

    def step(self, token: int) -> np.ndarray:
        """One greedy step: the token's embedding at position n_past."""
        x = _f64(self.w["embed"][int(token)])[None, :]
        x = self.forward(x)
        return self.head(x[0])


def decode_budget(n_audio: int, T_prompt: int, ceiling: int, floor_new: int = 256) -> int:
    """Generation budget of one run (moss/model.cpp of transcribe-cpp-sys
    0.4.1, run: the budget passed to the greedy loop; run_batch takes the
    same call with the batch's longest audio and longest prompt).

    The page first rejects a prompt whose rows plus the fixed 256-token
    generation reserve exceed the context ceiling, then asks for twice the
    audio rows plus 128 tokens (room above the plain audio-token count for
    the transcript's markers), with the 256-token reserve as the floor and the
    context left after the prompt as the cap.  The helper's body is not on
    the page; the reading taken is the plain clamp
    min(max(2 n_audio + 128, floor_new), ceiling - T_prompt).
    Raises ValueError where the page returns its input-too-long status.
    """
    n_audio, T_prompt, ceiling, floor_new = int(n_audio), int(T_prompt), int(ceiling), int(floor_new)
    if n_audio < 0 or T_prompt < 1 or floor_new < 1 or ceiling < 1:
        raise ValueError("invalid argument")
    if T_prompt + floor_new > ceiling:
        raise ValueError("input too long")
    want = 2 * n_audio + 128
    return min(max(want, floor_new), ceiling - T_prompt)


def greedy(oracle: Oracle, embeds: np.ndarray, max_new: int, eos_id: int = -1,
           keep_logits: bool = False):
    """The greedy loop of qwen3_asr/model.cpp, run.

    Returns (ids, truncated, logits_list).  ids holds at most max_new tokens,
    the first one from the prefill; a trailing EOS is stripped; truncated is
    True when the loop stopped without producing EOS.
    """
    logits = oracle.prefill(embeds)
    hist = [logits] if keep_logits else []
    tok = argmax_lowest(logits)
    ids = [tok]
    while tok != eos_id and len(ids) < max_new and oracle.n_past + 1 <= oracle.capacity:
        logits = oracle.step(tok)
        if keep_logits:
            hist.append(logits)
        tok = argmax_lowest(logits)
        ids.append(tok)
    truncated = tok != eos_id
    if ids and ids[-1] == eos_id:
        ids.pop()
    return ids, truncated, hist
