#!/usr/bin/env python
"""Throughput of the Qwen3-style speech decoder on GB300: decode tok/s and
prefill tok/s, with the roofline fraction of the dominant kernel.

One bench step is one utterance of the workload: a prefill over the
audio-injected prompt, then the greedy step loop (all rows of the hot path).
Inputs (token ids and encoder rows) are resident in HBM before the timed
region; every step streams the full 3.4 GB of weights, far more than the
129 MB L2, so no step is served from cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the
decoder has no data-path exchange); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import csv
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speech_decoder_gb300 import synth  # noqa: E402

METRIC = "decode tok/s & prefill tok/s (Qwen3-1.7B shape, 1 GB300); % HBM/TC roofline"
DEFAULT_WORKLOAD = "qwen3-1.7b-t152"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-long-prefill", action="store_true",
                   help="skip the timed 8015-row prompt of the same model")
    p.add_argument("--cpu-sample", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--weights", choices=["bf16", "e4m3"], default="bf16",
                   help="e4m3: the library rounds the weights row by row to 2^e * e4m3 and the single-sequence "
                        "step GEMVs stream 1-byte codes (not the benchmark's bf16 configuration)")
    p.add_argument("--layers", type=int, default=0,
                   help="profiling only: keep the workload's shapes but run this many blocks "
                        "(the JSON line then names the reduced model and is not a benchmark value)")
    return p.parse_args()


# ---------------------------------------------------------------- environment
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def combine_ranks(times_ms, counts, world, device="cpu"):
    """Whole-job numbers of independent replicas: the slowest rank's times
    (max over ranks) and the units of all ranks (sum).  world == 1 returns the
    inputs; otherwise every rank must call it (torch.distributed collective)."""
    import torch
    t = torch.tensor(list(times_ms), dtype=torch.float64, device=device)
    c = torch.tensor(list(counts), dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(c, op=torch.distributed.ReduceOp.SUM)
    return t.tolist(), c.tolist()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        hbm = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
        bf16 = d.get("bf16_tflops_sustained") or d.get("bf16_tflops")
        if hbm:
            return float(hbm), float(bf16) if bf16 else 1714.0, "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu_index
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for row in csv.reader(f):
                if len(row) < 9:
                    continue
                try:
                    sm.append(float(row[1]))
                    mx.append(float(row[2]))
                except ValueError:
                    continue
                for n, v in zip(names, row[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_for(args):
    wl = synth.workload(args.workload)
    if getattr(args, "weights", "bf16") == "e4m3":
        m = dataclasses.replace(wl.model, weight_dtype="e4m3", name=f"{wl.model.name}-e4m3")
        wl = dataclasses.replace(wl, model=m, name=f"{wl.name}-e4m3")
    if args.layers > 0:
        m = dataclasses.replace(wl.model, n_layers=args.layers, name=f"{wl.model.name}-{args.layers}blocks")
        wl = dataclasses.replace(wl, model=m, name=f"{wl.name}-{args.layers}blocks")
    return wl


def kernel_sha() -> str:
    """Hash of the sources the GEMV is compiled from, comments and whitespace
    removed (the code, not its commentary, decides the kernel's traffic)."""
    h = hashlib.sha256()
    for f in ("gemv.cu", "gemv_stream.cu", "attn_step.cuh", "decode.cuh", "common.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "speech_decoder_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(spec):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when the kernel source changed since it was taken or the
    model's projection shapes differ from the captured ones."""
    path = os.path.join(ROOT, "profiles", "gemv_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_sha") != kernel_sha():
        return None
    shape = d.get("shape", {})
    if any(getattr(spec, k) != v for k, v in shape.items()) or not shape:
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- workload
def workload_inputs(wl, w):
    items = []
    for i, pr in enumerate(wl.prompts):
        items.append(synth.prompt_inputs(wl.model, pr, seed=wl.seed, item=i))
    return items


def decode_bytes_per_step(spec, kv_len_mean: float, batch: int = 1) -> float:
    """Algorithmic HBM bytes of one decode step: every weight once (bf16; one
    byte for the e4m3 format's single-sequence steps) plus the K and V rows
    each sequence's attention reads (fp16)."""
    H, F, d, nq, nkv, L = spec.hidden, spec.ffn, spec.head_dim, spec.n_heads, spec.n_kv_heads, spec.n_layers
    wb = 1 if spec.weight_dtype == "e4m3" and batch == 1 else 2
    per_layer = ((nq + 2 * nkv) * d * H + H * nq * d + 2 * F * H + H * F) * wb
    return L * per_layer + spec.vocab * H * wb + batch * L * 2 * nkv * d * 2 * kv_len_mean


def prefill_work(spec, Ts) -> tuple:
    """Algorithmic work of one prefill of the prompts Ts (one sequence each):
    (FLOPs, HBM bytes).

    FLOPs follow the method as this library runs it: every block but the
    last takes all prompt rows (2 T N K per projection, 4 nq d T (T + 1) / 2
    for the causal attention); the last block writes every row's keys and
    values (its q|k|v projection on all rows) and runs the attention query,
    o projection and FFN on the last row only (slice_last), and the tied
    lm_head runs on that row.  Bytes: every weight once (the prompt is one
    pass over the model) plus the fp16 K/V rows written and the fp32 prompt
    rows read."""
    H, F, d, nq, nkv, L, V = (spec.hidden, spec.ffn, spec.head_dim, spec.n_heads, spec.n_kv_heads,
                              spec.n_layers, spec.vocab)
    qkv_n = (nq + 2 * nkv) * d
    rest = H * nq * d + 2 * F * H + H * F             # o, gate|up, down weights
    flops = 0.0
    for T in Ts:
        flops += 2.0 * T * (qkv_n * H + rest) * (L - 1) + 4.0 * nq * d * T * (T + 1) / 2 * (L - 1)
        flops += 2.0 * T * qkv_n * H + 2.0 * rest + 4.0 * nq * d * T
        flops += 2.0 * V * H
    wbytes = L * (qkv_n * H + rest) * 2 + V * H * 2
    nbytes = wbytes + sum(Ts) * (L * 2 * nkv * d * 2 + H * 4)
    return flops, float(nbytes)


def prefill_roofline(spec, Ts, ms, hbm, tc_peak) -> dict:
    """Achieved rates of one prefill against both ceilings; `bound` names
    the one the arithmetic intensity selects (FLOPs per byte below the ridge
    tc_peak / hbm: HBM)."""
    flops, nbytes = prefill_work(spec, Ts)
    gbs = nbytes / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    bound = "hbm" if flops / nbytes < tc_peak * 1e12 / (hbm * 1e9) else "tensor"
    return {"bound": bound, "flops": flops, "bytes": int(nbytes),
            "achieved_gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
            "achieved_tflops": round(tfs, 2), "tc_frac": round(tfs / tc_peak, 4),
            "frac": round(gbs / hbm if bound == "hbm" else tfs / tc_peak, 4)}


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()
    from speech_decoder_gb300.binding import Decoder

    wl = workload_for(args)
    spec = wl.model
    w = synth.model_weights(spec, seed=wl.seed)
    items = workload_inputs(wl, w)
    B = wl.batch
    Ts = [p.T for p in wl.prompts]
    T_all = sum(Ts)
    max_new = wl.steps + 1                      # the prefill's token counts toward the budget
    dec = Decoder(spec, w, max_ctx=max(Ts) + max_new, max_batch=B, max_tokens=T_all, max_new=max_new,
                  eos_id=wl.eos_id, device=dev)
    del w
    stream = dec.stream
    ids_np = np.concatenate([it["ids"] for it in items]).astype(np.int32)
    audio_np = np.concatenate([it["audio"] for it in items]).astype(np.float32)
    cu_ids = np.zeros(B + 1, np.int32)
    cu_ids[1:] = np.cumsum([len(it["ids"]) for it in items])
    cu_au = np.zeros(B + 1, np.int32)
    cu_au[1:] = np.cumsum([it["audio"].shape[0] for it in items])
    pre_lens = np.array([it["prefix_len"] for it in items], np.int32)
    ids_dev = torch.from_numpy(ids_np).to(dev)
    audio_dev = torch.from_numpy(audio_np).to(dev)
    torch.cuda.synchronize()

    def utterance(ids, audio, on_device):
        """One pass of the hot path: prefill every item, then the greedy loop."""
        if B == 1:
            dec.prefill_ids(ids, audio, int(pre_lens[0]))
            out, _ = dec.generate(max_new)
            return len(out) - 1
        dec.prefill_ids_batch_ptr(ids.data_ptr(), cu_ids, audio.data_ptr(), cu_au, pre_lens, int(on_device))
        res = dec.generate_batch(max_new, B)
        return sum(len(r[0]) - 1 for r in res)

    for _ in range(args.warmup):
        utterance(ids_dev, audio_dev, True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local) if rank == 0 else None
    n0 = dec.launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pre_ms, gen_ms, n_tok = 0.0, 0.0, 0
    e0.record(stream)
    for _ in range(args.steps):
        n = utterance(ids_dev, audio_dev, True)
        p, g = dec.timings()
        pre_ms += p
        gen_ms += g
        n_tok += n
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    launches = dec.launch_count() - n0
    clk = clocks.stop() if clocks else None
    total_ms = e0.elapsed_time(e1)
    (total_ms, gen_ms, pre_ms), (n_tok_all, n_pre_all) = combine_ranks(
        [total_ms, gen_ms, pre_ms], [n_tok, args.steps * T_all], world, dev)
    decode_tok_s = n_tok_all / (gen_ms / 1e3)
    prefill_tok_s = n_pre_all / (pre_ms / 1e3)

    # dominant kernel: the projection kernel of the decode step, timed alone
    hbm, bf16_peak, peak_kind = peaks()
    utterance(ids_dev, audio_dev, True)
    if B == 1:
        dec.prefill_ids(ids_dev, audio_dev, int(pre_lens[0]))
        impl = os.environ.get("SPEECH_DECODER_GEMV", "stream")
        kname = ("k_gemv_stream" if impl == "stream" else "k_gemv_ldg") + \
            " (the step's q|k|v, o, gate|up+SwiGLU and down GEMVs, every layer in order)"
    else:
        dec.prefill_ids_batch_ptr(ids_dev.data_ptr(), cu_ids, audio_dev.data_ptr(), cu_au, pre_lens, 1)
        kname = "k_gemm_tc + k_splitk_reduce (q|k|v and gate|up projections of %d rows, per projection)" % B
    kms, kbytes = dec.profile_kernel(0, 10)
    achieved = kbytes / (kms / 1e3) / 1e9
    roof = {"kernel": kname, "bound": "hbm",
            "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
            "peak_source": peak_kind, "bytes_per_launch": int(kbytes), "avg_launch_us": round(kms * 1e3, 2),
            "traffic": ncu_traffic(spec) if B == 1 and spec.weight_dtype == "bf16" else None}
    kv_mean = float(np.mean([t + wl.steps / 2 for t in Ts]))
    step_bytes = decode_bytes_per_step(spec, kv_mean, B)
    steps_done = n_tok / B
    step_ms = gen_ms / max(1.0, steps_done)
    step_roof = {"bytes_per_step": int(step_bytes), "achieved": round(step_bytes / (step_ms / 1e3) / 1e9, 1),
                 "frac": round(step_bytes / (step_ms / 1e3) / 1e9 / hbm, 4)}

    e2e = None
    if not args.no_e2e:
        ids_h = torch.from_numpy(ids_np).pin_memory()
        audio_h = torch.from_numpy(audio_np).pin_memory()
        utterance(ids_h, audio_h, False)
        torch.cuda.synchronize()
        t_pre, t_gen, n_e = 0.0, 0.0, 0
        reps = max(1, args.steps)
        for _ in range(reps):
            t0 = time.perf_counter()
            if B == 1:
                dec.prefill_ids(ids_h, audio_h, int(pre_lens[0]))
            else:
                dec.prefill_ids_batch_ptr(ids_h.data_ptr(), cu_ids, audio_h.data_ptr(), cu_au, pre_lens, 0)
            t1 = time.perf_counter()
            if B == 1:
                out, _ = dec.generate(max_new)
                n_e += len(out) - 1
            else:
                n_e += sum(len(r[0]) - 1 for r in dec.generate_batch(max_new, B))
            t2 = time.perf_counter()
            t_pre += t1 - t0
            t_gen += t2 - t1
        e2e = {"value": round(n_e * world / t_gen, 1), "unit": "tok/s",
               "prefill_tok_s": round(reps * T_all * world / t_pre, 1),
               "h2d_bytes_per_step": int(ids_h.numel() * 4 + audio_h.numel() * 4),
               "d2h_bytes_per_step": int(B * (4 + 4 * max_new))}

    pre_roof = prefill_roofline(spec, Ts, pre_ms / args.steps, hbm, bf16_peak)
    pre_roof["peak_gbs"], pre_roof["peak_tflops"], pre_roof["peak_source"] = hbm, bf16_peak, peak_kind

    long = None
    if B == 1 and not args.no_long_prefill and args.layers == 0:
        long = long_prefill(args, hbm, bf16_peak, peak_kind, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(decode_tok_s, 1), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if spec.weight_dtype == "bf16" else "e4m3 weights (per-row power-of-two scale), fp32 accumulate",
            "data": "synthetic (seeded random-init weights N(0,0.02), encoder rows N(0,1))",
            "config": {"workload": wl.name, "prompt_rows": T_all,
                       "layout": [[p.prefix_len, p.n_audio, p.suffix_len] for p in wl.prompts][:4],
                       "decode_steps": wl.steps, "batch": wl.batch, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: every step streams %.1f GB of weights" % (
                           decode_bytes_per_step(spec, 0.0, 1) / 1e9)},
            "prefill": {"value": round(prefill_tok_s, 1), "unit": "tok/s", "ms": round(pre_ms / args.steps, 3),
                        "roofline": pre_roof},
            "prefill_long": long,
            "decode_ms_per_step": round(step_ms, 4),
            "roofline": roof, "step_roofline": step_roof, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clk, "gpu_launches": int(launches),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- long prompt
LONG_WORKLOAD = "qwen3-1.7b-t8015"


def long_prefill(args, hbm, bf16_peak, peak_kind, dev, reps=3):
    """The tensor-core-bound prefill: the 8015-row prompt (9 | 8000 encoder
    rows | 6) of the same model, timed with CUDA events on the decoder's
    stream (prefill only; one untimed warm-up)."""
    import torch
    from speech_decoder_gb300.binding import Decoder
    lw = synth.workload(LONG_WORKLOAD)
    spec = lw.model
    if args.weights == "e4m3":
        spec = dataclasses.replace(spec, weight_dtype="e4m3", name=f"{spec.name}-e4m3")
    pr = lw.prompts[0]
    w = synth.model_weights(spec, seed=lw.seed)
    it = synth.prompt_inputs(spec, pr, seed=lw.seed, item=0)
    dec = Decoder(spec, w, max_ctx=pr.T + lw.steps + 1, max_batch=1, max_tokens=pr.T, max_new=lw.steps + 1,
                  device=dev)
    del w
    ids = torch.from_numpy(np.asarray(it["ids"], np.int32)).to(dev)
    audio = torch.from_numpy(np.asarray(it["audio"], np.float32)).to(dev)
    dec.prefill_ids(ids, audio, int(it["prefix_len"]))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(dec.stream)
    for _ in range(reps):
        dec.prefill_ids(ids, audio, int(it["prefix_len"]))
    e1.record(dec.stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    dec.close()
    del dec
    torch.cuda.empty_cache()
    roof = prefill_roofline(spec, [pr.T], ms, hbm, bf16_peak)
    roof["peak_gbs"], roof["peak_tflops"], roof["peak_source"] = hbm, bf16_peak, peak_kind
    return {"workload": lw.name, "prompt_rows": pr.T, "reps": reps, "ms": round(ms, 3),
            "value": round(pr.T / (ms / 1e3), 1), "unit": "tok/s", "roofline": roof}


# ---------------------------------------------------------------- oracle timings
def oracle_sample(wl, rows: int, steps: int) -> dict:
    """The fp64 oracle, as it stands: a prefill of the first `rows` prompt
    rows of item 0, then `steps` greedy steps of the full model."""
    import oracle as O
    spec = wl.model
    w = synth.model_weights(spec, seed=wl.seed)
    item = synth.prompt_inputs(spec, wl.prompts[0], seed=wl.seed, item=0)
    emb = O.assemble_prompt(w["embed"], item["ids"], item["audio"], item["prefix_len"])[:rows]
    orc = O.Oracle(spec, w, rows + steps + 1)
    t0 = time.perf_counter()
    logits = orc.prefill(emb)
    t1 = time.perf_counter()
    tok = O.argmax_lowest(logits)
    for _ in range(steps):
        tok = O.argmax_lowest(orc.step(tok))
    t2 = time.perf_counter()
    return {"value": round(steps / (t2 - t1), 4), "prefill_tok_s": round(rows / (t1 - t0), 3),
            "rows": rows, "steps": steps}


def _sample_in_child(wl, threads: int, rows: int, steps: int) -> dict:
    """oracle_sample in a child process whose BLAS runs on `threads` threads."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-sample", str(threads), "--workload", wl.name,
           "--steps", str(steps), "--warmup", str(rows), "--weights", "bf16"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(f"oracle sample failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(wl) -> dict:
    """The oracle timed on the host cores, as a reported baseline: on every
    core, the whole prompt's prefill and 3 greedy steps; on one thread, an
    8-row prefill and 1 step (bounded samples of the same workload)."""
    cores = os.cpu_count() or 1
    T0 = wl.prompts[0].T
    allc = _sample_in_child(wl, cores, T0, 3)
    one = _sample_in_child(wl, 1, 8, 1)
    note = "; the oracle's time does not depend on the weights' rounding" if wl.model.weight_dtype == "e4m3" else ""
    return {"value": allc["value"], "unit": "tok/s", "cores": cores, "kind": "oracle",
            "prefill_tok_s": allc["prefill_tok_s"],
            "sample": f"{wl.name}: prefill of the whole {T0}-row prompt, then 3 greedy steps of all "
                      f"{wl.model.n_layers} layers (numpy fp64, BLAS on {cores} threads{note})",
            "one_thread": {"value": one["value"], "unit": "tok/s", "cores": 1, "prefill_tok_s": one["prefill_tok_s"],
                           "sample": f"{wl.name}: prefill of the first 8 prompt rows, then 1 greedy step "
                                     f"(numpy fp64, BLAS on 1 thread)"}}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import oracle as O
    wl = workload_for(args)
    spec = wl.model
    w = synth.model_weights(spec, seed=wl.seed)
    item = synth.prompt_inputs(spec, wl.prompts[0], seed=wl.seed, item=0)
    rows = 8
    emb = O.assemble_prompt(w["embed"], item["ids"], item["audio"], item["prefix_len"])[:rows]
    orc = O.Oracle(spec, w, rows + args.warmup + args.steps + 1)
    tok = O.argmax_lowest(orc.prefill(emb))
    for _ in range(args.warmup):
        tok = O.argmax_lowest(orc.step(tok))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tok = O.argmax_lowest(orc.step(tok))
    dt = time.perf_counter() - t0
    v = args.steps / dt
    sample = (f"{wl.name}: each step is one greedy decode step of all {spec.n_layers} layers after an untimed "
              f"{rows}-row prefill (numpy fp64 oracle, BLAS on all host cores)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "prompt_rows": wl.prompts[0].T, "decode_steps": wl.steps},
        "cpu_baseline": {"value": round(v, 4), "unit": "tok/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.cpu_sample:
        # child of cpu_baseline: --warmup carries the prefill rows, --steps the greedy steps
        print(json.dumps(oracle_sample(workload_for(a), a.warmup, a.steps)), flush=True)
    elif a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
