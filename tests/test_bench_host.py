"""Host-side logic of bench.py (no GPU): the algorithmic byte count of a
decode step, the workload options, and the hash that keys the committed ncu
traffic record to the GEMV sources."""
import argparse
import os
import shutil

import pytest

import bench
from speech_decoder_gb300 import synth


def weight_count(spec):
    H, F, d = spec.hidden, spec.ffn, spec.head_dim
    per_layer = (spec.n_heads + 2 * spec.n_kv_heads) * d * H + H * spec.n_heads * d + 2 * F * H + H * F
    return spec.n_layers * per_layer + spec.vocab * H


def test_decode_bytes_per_step_counts_every_weight_once():
    spec = synth.QWEN3_1_7B
    # 1.7B shape: 3.441 GB of bf16 weights per token, 114,688 B of fp16 K and V per cached token
    assert bench.decode_bytes_per_step(spec, 0.0) == 2 * weight_count(spec)
    assert abs(2 * weight_count(spec) / 1e9 - 3.441) < 1e-3
    per_tok = bench.decode_bytes_per_step(spec, 1.0) - bench.decode_bytes_per_step(spec, 0.0)
    assert per_tok == 114688
    assert bench.decode_bytes_per_step(spec, 10.0, batch=4) - bench.decode_bytes_per_step(spec, 0.0, batch=4) \
        == 4 * 10 * 114688


def test_decode_bytes_e4m3_single_sequence_only():
    import dataclasses
    spec = dataclasses.replace(synth.QWEN3_1_7B, weight_dtype="e4m3")
    # one sequence streams one byte per weight; batched steps take the bf16 copy
    assert bench.decode_bytes_per_step(spec, 0.0) == weight_count(spec)
    assert bench.decode_bytes_per_step(spec, 0.0, batch=2) == 2 * weight_count(spec)


def _args(**kw):
    a = argparse.Namespace(workload="qwen3-1.7b-t152", layers=0, weights="bf16")
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_workload_options():
    wl = bench.workload_for(_args())
    assert wl.name == "qwen3-1.7b-t152" and wl.model.weight_dtype == "bf16" and wl.model.n_layers == 28
    wl = bench.workload_for(_args(weights="e4m3"))
    assert wl.name == "qwen3-1.7b-t152-e4m3" and wl.model.weight_dtype == "e4m3"
    wl = bench.workload_for(_args(layers=2))
    assert wl.model.n_layers == 2 and wl.name.endswith("-2blocks")


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = os.path.join(bench.ROOT, "speech_decoder_gb300", "csrc")
    dst = tmp_path / "speech_decoder_gb300" / "csrc"
    shutil.copytree(csrc, dst)
    base = bench.kernel_sha()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_sha() == base
    f = dst / "gemv_stream.cu"
    src = f.read_text()
    f.write_text("// a new comment line\n" + src.replace("namespace dec {", "namespace dec {  /* inline note */", 1))
    assert bench.kernel_sha() == base
    f.write_text(src.replace("constexpr int kAutoStages = 12;", "constexpr int kAutoStages = 11;", 1))
    assert "kAutoStages = 11" in f.read_text()
    assert bench.kernel_sha() != base
    # a record keyed to other sources is not reported
    assert bench.ncu_traffic(synth.workload("qwen3-1.7b-t152").model) is None


def test_traffic_record_is_well_formed():
    import json
    with open(os.path.join(bench.ROOT, "profiles", "gemv_traffic.json")) as fh:
        d = json.load(fh)
    assert set(d["per_launch_bytes"]) == {"qkv", "o", "gate_up_swiglu", "down"}
    assert d["dram_bytes_per_launch"] == pytest.approx(sum(d["per_launch_bytes"].values()) / 4, abs=1)
    # DRAM bytes are at least the algorithmic bytes (weights are read once)
    assert d["dram_bytes_per_launch"] >= d["algorithmic_bytes_per_launch"]
    assert "--clock-control none" in d["command"]
    t = bench.ncu_traffic(synth.workload("qwen3-1.7b-t152").model)
    assert t is None or t == d["dram_bytes_per_launch"]
    # only reported for the projection shapes it was captured on
    assert bench.ncu_traffic(synth.workload("qwen3-0.6b-t153").model) is None


def test_prefill_work_counts_rows_pairs_and_slice_last():
    """FLOPs of a prefill counted by brute force over rows and causal
    (query, key) pairs, with the last block on the last row only."""
    spec = synth.small_spec(n_layers=3, hidden=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn=96, vocab=50)
    H, F, d, nq, nkv, V = spec.hidden, spec.ffn, spec.head_dim, spec.n_heads, spec.n_kv_heads, spec.vocab
    qkv = (nq + 2 * nkv) * d * H
    rest = H * nq * d + 2 * F * H + H * F
    for Ts in ([1], [7], [5, 9]):
        want = 0
        for T in Ts:
            pairs = sum(t + 1 for t in range(T))          # causal (query, key) pairs
            want += (spec.n_layers - 1) * (2 * T * (qkv + rest) + 4 * nq * d * pairs)
            want += 2 * T * qkv + 2 * rest + 4 * nq * d * T  # last block: keys of every row, one query row
            want += 2 * V * H                                 # tied lm_head on the last row
        flops, nbytes = bench.prefill_work(spec, Ts)
        assert flops == want
        kv = sum(Ts) * spec.n_layers * 2 * nkv * d * 2
        assert nbytes == 2 * weight_count(spec) + kv + sum(Ts) * H * 4


def test_prefill_roofline_picks_the_bound():
    spec = synth.QWEN3_1_7B
    # 152 rows: about 125 FLOP per byte, below the ridge (HBM); 8015 rows: far above (tensor cores)
    r = bench.prefill_roofline(spec, [152], 1.0, 6793.1, 1701.1)
    assert r["bound"] == "hbm" and r["frac"] == r["hbm_frac"]
    r = bench.prefill_roofline(spec, [8015], 30.0, 6793.1, 1701.1)
    assert r["bound"] == "tensor" and r["frac"] == r["tc_frac"]
    assert 28e12 < r["flops"] < 30.1e12
