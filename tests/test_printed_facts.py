"""The benchmark workloads and the perception projection against the facts
the source pages print (tests/golden/printed_facts.json, each entry under its
page and section)."""
import json
import os

from speech_decoder_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "printed_facts.json")


def facts():
    with open(GOLDEN) as fh:
        return json.load(fh)


def canary():
    return facts()["canary_qwen/model.cpp (transcribe.cpp), file header, forward shape"]


def test_qwen3_17b_shape_matches_the_canary_page():
    c = canary()
    m = synth.QWEN3_1_7B
    assert m.hidden == c["decoder_hidden"] and m.n_layers == c["decoder_blocks"]
    assert c["decoder"].startswith("Qwen3-1.7B")


def test_t152_prompt_is_the_jfk_prompt_with_the_placeholder_replaced():
    c = canary()
    wl = synth.workload("qwen3-1.7b-t152")
    (p,) = wl.prompts
    assert p.n_audio == c["encoder_rows_jfk"]
    # the one placeholder id becomes the encoder rows; the other ids stay
    assert p.prefix_len + p.suffix_len == c["prompt_ids_jfk"] - c["audio_placeholders_in_prompt"]
    assert p.T == 152 and wl.model is synth.QWEN3_1_7B


def test_rope_theta_of_every_workload():
    f = facts()["qwen3_asr/decoder.cpp (transcribe-cpp-sys 0.2.0), file header"]
    for name in ("qwen3-0.6b-t153", "qwen3-1.7b-t152", "qwen3-1.7b-b32", "qwen3-1.7b-t8015"):
        assert synth.workload(name).model.rope_theta == f["rope_theta"], name


def test_perception_projection_shape_matches_the_canary_page():
    c = canary()
    d_in, d_out = c["perception_projection_in_out"]
    # the projection's output rows are the decoder's input rows
    assert d_out == synth.QWEN3_1_7B.hidden and d_in == 1024 and c["perception_projection_bias"]


def test_moss_decoder_is_the_small_shape():
    f = facts()["moss/model.cpp (transcribe-cpp-sys 0.4.1), file header"]
    assert f["decoder"] == "Qwen3-0.6B"
    assert synth.QWEN3_0_6B.name.startswith("qwen3-0.6b")
