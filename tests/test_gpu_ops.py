"""Kernel-level parity through the C ABI: the standalone split-KV decode
attention against the oracle's attention on the same (fp16-rounded) keys."""
import ctypes

import numpy as np
import pytest

import oracle as O
from _parity import rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from speech_decoder_gb300 import binding, build
    build.build()
    return binding.load_library()


def attn_case(seed, B, nq, nkv, d, slots, lens, offs, kv_f16):
    rng = np.random.default_rng(seed)
    kv_np = np.float16 if kv_f16 else np.float32
    K = rng.standard_normal((nkv, slots, d)).astype(kv_np)
    V = rng.standard_normal((nkv, slots, d)).astype(kv_np)
    q = (rng.standard_normal((B, nq, d)) * 0.3).astype(np.float32)
    return q, K, V, np.array(lens, np.int32), np.array(offs, np.int32)


def run_op(lib, q, K, V, lens, offs, kv_f16, fn="dec_attn_decode"):
    import torch
    from speech_decoder_gb300.binding import DEC_F16, DEC_F32
    B, nq, d = q.shape
    nkv, slots, _ = K.shape
    dev = "cuda:0"
    tq, tK, tV = (torch.from_numpy(a).to(dev) for a in (q, K, V))
    toff, tlen = torch.from_numpy(offs).to(dev), torch.from_numpy(lens).to(dev)
    out = torch.full((B, nq, d), 7.0, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    args = [tq.data_ptr(), tK.data_ptr(), tV.data_ptr(), DEC_F16 if kv_f16 else DEC_F32, slots, toff.data_ptr(),
            tlen.data_ptr(), B, nq, nkv, d, out.data_ptr()]
    if fn == "dec_attn_decode":
        n = ctypes.c_size_t()
        assert lib.dec_attn_decode_scratch_size(B, nq, nkv, d, ctypes.byref(n)) == 0
        scratch = torch.empty(n.value, dtype=torch.uint8, device=dev)
        st = lib.dec_attn_decode(*args, scratch.data_ptr(), n.value, stream.cuda_stream)
    else:
        st = getattr(lib, fn)(*args, stream.cuda_stream)
    assert st == 0, st
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_attn(q, K, V, lens, offs):
    out = []
    for b in range(q.shape[0]):
        L, o = int(lens[b]), int(offs[b])
        Kb = np.transpose(K[:, o:o + L, :].astype(np.float64), (1, 0, 2))
        Vb = np.transpose(V[:, o:o + L, :].astype(np.float64), (1, 0, 2))
        out.append(O.attention(q[b][None].astype(np.float64), Kb, Vb, np.array([L - 1]))[0])
    return np.stack(out)


CASES = [
    # B, nq, nkv, d, slots, lens, offs, kv_f16
    (1, 16, 8, 128, 8192, [8143], [0], True),
    (3, 16, 8, 128, 2048, [1, 152, 700], [0, 10, 1000], True),
    (4, 8, 1, 64, 600, [33, 1, 257, 64], [0, 40, 80, 400], False),
    (2, 4, 4, 64, 100, [17, 50], [0, 50], True),
    (5, 32, 4, 128, 3000, [2999, 1, 2, 500, 1000], [0, 0, 0, 0, 1500], True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}q{c[1]}kv{c[2]}d{c[3]}{'f16' if c[7] else 'f32'}" for c in CASES])
def test_attn_decode_op_matches_oracle(lib, case):
    B, nq, nkv, d, slots, lens, offs, f16 = case
    q, K, V, lens, offs = attn_case(11, B, nq, nkv, d, slots, lens, offs, f16)
    got = run_op(lib, q, K, V, lens, offs, f16)
    ref = oracle_attn(q, K, V, lens, offs)
    assert rel_err(got.reshape(B, -1), ref.reshape(B, -1)) <= 1e-4


def test_attn_decode_op_skips_invalid_rows(lib):
    q, K, V, lens, offs = attn_case(12, 3, 4, 2, 64, 64, [0, 10, 60], [0, 0, 10], True)
    got = run_op(lib, q, K, V, lens, offs, True)
    assert np.all(got[0] == 7.0) and np.all(got[2] == 7.0)          # len 0 and out-of-pool rows untouched
    ref = oracle_attn(q[1:2], K, V, lens[1:2], offs[1:2])
    assert rel_err(got[1].reshape(1, -1), ref.reshape(1, -1)) <= 1e-4


# ------------------------------------------------------------------ prefill GEMM (tcgen05 / CUDA cores)
def _bf16(a):
    from speech_decoder_gb300 import synth
    a = np.ascontiguousarray(a, np.float32).copy()
    synth.round_bf16(a)
    return a


def run_gemm(lib, X, W, epi, use_tc, splits=0, C0=None):
    import torch
    from speech_decoder_gb300 import synth
    dev = "cuda:0"
    T, K = X.shape
    N = W.shape[0]
    xt = torch.from_numpy(synth.bf16_bits(X).view(np.int16)).to(dev)
    wt = torch.from_numpy(synth.bf16_bits(W).view(np.int16)).to(dev)
    scratch = torch.zeros(64 << 20, dtype=torch.uint8, device=dev)
    if epi == 2:
        out = torch.zeros((T, N // 2), dtype=torch.int16, device=dev)
        st = lib.dec_debug_gemm(xt.data_ptr(), T, wt.data_ptr(), N, K, 2, None, 0, out.data_ptr(), N // 2, 1,
                                splits, scratch.data_ptr(), scratch.numel(), torch.cuda.current_stream().cuda_stream)
        assert st == 0, st
        torch.cuda.synchronize()
        bits = out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16
        return bits.view(np.float32)
    C = torch.from_numpy(np.zeros((T, N), np.float32) if C0 is None else C0.copy()).to(dev)
    st = lib.dec_debug_gemm(xt.data_ptr(), T, wt.data_ptr(), N, K, epi, C.data_ptr(), N, None, 0, use_tc, splits,
                            scratch.data_ptr(), scratch.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, st
    torch.cuda.synchronize()
    return C.cpu().numpy()


GEMMS = [  # T, N, K, splits (0 = automatic)
    (16, 512, 256, 0), (152, 4096, 2048, 0), (152, 2048, 6144, 0), (1, 256, 512, 0), (700, 1024, 512, 0),
    (8015, 256, 256, 0), (37, 384, 1408, 3), (152, 128, 64, 1), (300, 768, 192, 2),
    # split-K: 5 splits of uneven length, two prompt-row tiles (the second ragged) with 8 splits,
    # 12 splits of the down projection's K
    (152, 4096, 2048, 5), (400, 384, 1024, 0), (152, 2048, 6144, 12),
    # long prompts: the persistent kernel (tiles of 256 weight rows x 128 prompt rows, several per CTA;
    # ragged last prompt-row tile; K = 6144 as in the down projection)
    (8015, 12288, 2048, 0), (2048, 4096, 2048, 0), (1500, 2048, 6144, 0),
    # a short batch of rows against many weight rows (the vocabulary projection of a batch): the
    # persistent kernel with 32- and 48-row tiles, the last 256-row weight tile half outside the matrix
    (32, 39040, 256, 0), (17, 39040, 256, 0), (48, 39040, 512, 0),
]


@pytest.mark.parametrize("shape", GEMMS, ids=[f"T{s[0]}N{s[1]}K{s[2]}s{s[3]}" for s in GEMMS])
def test_gemm_tc_matches_oracle_linear(lib, shape):
    T, N, K, splits = shape
    rng = np.random.default_rng(T * 7 + N)
    X = _bf16(rng.standard_normal((T, K)))
    W = _bf16(rng.standard_normal((N, K)) * 0.02)
    ref = O.linear(X, W)
    got = run_gemm(lib, X, W, 0, 1, splits)
    assert rel_err(got, ref) <= 1e-5
    C0 = rng.standard_normal((T, N)).astype(np.float32)
    got = run_gemm(lib, X, W, 1, 1, splits, C0=C0)                      # residual add
    assert rel_err(got, C0 + ref) <= 1e-5


@pytest.mark.parametrize("shape", [(152, 1536, 512, 0), (16, 512, 256, 2), (500, 768, 256, 0), (8015, 12288, 2048, 0),
                                   (1100, 4096, 1024, 0)],
                         ids=["T152F768", "T16F256s2", "T500F384", "T8015F6144", "T1100F2048"])
def test_gemm_tc_swiglu_matches_oracle(lib, shape):
    T, N2, K, splits = shape
    F = N2 // 2
    rng = np.random.default_rng(N2 + T)
    X = _bf16(rng.standard_normal((T, K)))
    Wg = _bf16(rng.standard_normal((F, K)) * 0.05)
    Wu = _bf16(rng.standard_normal((F, K)) * 0.05)
    # pack as the library does: blocks of 128 gate rows then the same 128 features' up rows
    packed = np.concatenate([np.concatenate([Wg[j:j + 128], Wu[j:j + 128]]) for j in range(0, F, 128)])
    got = run_gemm(lib, X, packed, 2, 1, splits)
    g, u = O.linear(X, Wg), O.linear(X, Wu)
    ref = O.silu(g) * u
    # output rounded to bf16 (relative error up to 2^-9 of each value, 2^-8
    # allowed), plus the fp32 accumulation error of gate and up (well below
    # 1e-5 absolute for K <= 2048 at these magnitudes), carried through the
    # product: it dominates where one factor is near zero
    assert np.all(np.abs(got - ref) <= 2 ** -8 * np.abs(ref) + 1e-5 * (np.abs(O.silu(g)) + np.abs(u)))


def test_gemm_simt_matches_oracle_linear(lib):
    rng = np.random.default_rng(5)
    X = _bf16(rng.standard_normal((45, 512)))
    W = _bf16(rng.standard_normal((384, 512)) * 0.02)
    assert rel_err(run_gemm(lib, X, W, 0, 0), O.linear(X, W)) <= 1e-5


# ------------------------------------------------------------------ perception projection
@pytest.mark.parametrize("T", [1, 138, 301])
def test_perception_projection_matches_oracle(lib, T):
    """Linear(1024, 2048) + bias of encoder rows (bf16 weights, fp32 rows) on
    the tensor cores against the oracle's fp64 projection of the same values."""
    import torch
    from speech_decoder_gb300 import synth
    rng = np.random.default_rng(50 + T)
    d_in, d_out = 1024, 2048
    enc = rng.standard_normal((T, d_in)).astype(np.float32)
    W = synth.round_bf16((rng.standard_normal((d_out, d_in)) * 0.02).astype(np.float32))
    bias = rng.standard_normal(d_out).astype(np.float32)
    dev = "cuda:0"
    t_enc = torch.from_numpy(enc).to(dev)
    t_W = torch.from_numpy(W).to(torch.bfloat16).to(dev)
    t_b = torch.from_numpy(bias).to(dev)
    out = torch.full((T, d_out), 3.0, dtype=torch.float32, device=dev)
    n = 2 * ((T * d_in * 2 + 255) // 256 * 256) + (16 << 20)
    scratch = torch.empty(n, dtype=torch.uint8, device=dev)
    st = lib.dec_perception_project(t_enc.data_ptr(), T, d_in, t_W.data_ptr(), t_b.data_ptr(), d_out, out.data_ptr(),
                                    scratch.data_ptr(), n, torch.cuda.current_stream().cuda_stream)
    assert st == 0, st
    torch.cuda.synchronize()
    ref = O.perception_projection(enc.astype(np.float64), W.astype(np.float64), bias)
    e = rel_err(out.cpu().numpy(), ref)
    assert e <= 1e-4, e
    # too little scratch is refused before any work
    assert lib.dec_perception_project(t_enc.data_ptr(), T, d_in, t_W.data_ptr(), t_b.data_ptr(), d_out,
                                      out.data_ptr(), scratch.data_ptr(), 1024,
                                      torch.cuda.current_stream().cuda_stream) == 2
