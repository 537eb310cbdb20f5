#!/usr/bin/env python3
"""Dual-AR frame-decode benchmark: frames/s, RTF and fraction of the HBM roofline.

Default workload (one GPU): the full S2-Pro-shaped model at batch 1 -- a
512-token prompt, then 256 frames (warm-up + timed) with seeded uniforms,
T = 0.8, top-p 0.8, repetition-aware window 10, <|im_end|> excluded so every
frame runs.  A step is one frame: q0 draw, ten fast-AR passes, fusion, one
slow position with the restricted head.  Weights (9.1 GB) exceed L2, so no
flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (torchrun) every rank runs an independent replica (no collective
on the data path); the value is the frames of all ranks over the slowest
rank's time.  `--impl reference` times the CPU oracle on the same workload.
"""
from __future__ import annotations

import argparse
import atexit
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dualar_inputs import CONFIGS, FRAMES_PER_AUDIO_SECOND  # noqa: E402
from dualar_inputs import generators as gen  # noqa: E402

METRIC = "Dual-AR frames/s (and RTF) at batch 1 and 64 on 1 GB300; % of HBM roofline"

WORKLOADS = {
    "s2pro_b1": dict(cfg="s2pro", batch=1, prompt=512, frames=256, temperature=0.8, top_p=0.8,
                     ras_win=10, desc="full S2-Pro-shaped Dual-AR, batch 1, 512-token prompt, "
                                       "T=0.8 top-p 0.8 RAS window 10"),
    "s2pro_l1_b1": dict(cfg="s2pro_l1", batch=1, prompt=512, frames=16, temperature=0.8, top_p=0.8,
                        ras_win=10, desc="one-layer S2-Pro-shaped profiling case, batch 1, 512-token prompt"),
    "s2pro_b64": dict(cfg="s2pro", batch=64, prompt=0, frames=28, temperature=0.8, top_p=0.8, ras_win=10,
                      desc="full S2-Pro-shaped Dual-AR, batch 64, contexts uniform in [1024, 4096]"),
    "s2pro_l1_b64": dict(cfg="s2pro_l1", batch=64, prompt=0, frames=8, temperature=0.8, top_p=0.8, ras_win=10,
                         desc="one-layer S2-Pro-shaped profiling case, batch 64, contexts uniform in [1024, 4096]"),
    "s2pro_b128_replace": dict(cfg="s2pro", batch=128, prompt=0, frames=64, temperature=0.8, top_p=0.8,
                               ras_win=10, desc="full S2-Pro-shaped Dual-AR, batch 128: 124 contexts uniform in "
                                                "[2048, 4096] that finish at seeded frames (uniform in [1, 64]) and "
                                                "are replaced from a seeded queue, plus 4 resident contexts of 16384"),
    "s2pro_b64_two_streams": dict(cfg="s2pro", batch=64, prompt=0, frames=20, temperature=0.8, top_p=0.8,
                                  ras_win=10, desc="full S2-Pro-shaped Dual-AR, batch 64 (contexts uniform in "
                                                   "[1024, 4096]) as one decoder, then as two decoders of 32 on "
                                                   "two CUDA streams (co-scheduling the fast AR of one group with "
                                                   "the slow step of the other)"),
    "tiny_b1": dict(cfg="tiny", batch=1, prompt=32, frames=16, temperature=0.8, top_p=0.8, ras_win=10,
                    desc="tiny Dual-AR, batch 1, 32-token prompt"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="s2pro_b1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-batches", action="store_true",
                    help="skip the batch-16, batch-64 and batch-128 measurements")
    ap.add_argument("--no-w4a16", action="store_true", help="skip the 4-bit-weight measurement")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


MEGA_SOURCES = ["dual_ar_tts_frame_gb300/csrc/mega.cu", "dual_ar_tts_frame_gb300/csrc/gemv.cuh",
                "dual_ar_tts_frame_gb300/csrc/ops.cuh", "dual_ar_tts_frame_gb300/csrc/common.cuh",
                "dual_ar_tts_frame_gb300/csrc/internal.h", "dual_ar_tts_frame_gb300/csrc/mega.h"]


def sources_sha256(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()


def traffic_record():
    """ncu DRAM bytes per launch of the persistent frame kernel
    (profiles/mega_traffic.json), if they were taken on the current sources
    of that kernel; None otherwise."""
    p = os.path.join(ROOT, "profiles", "mega_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p))
    return rec if rec.get("sources_sha256") == sources_sha256(rec.get("sources", MEGA_SOURCES)) else None


class ClockSampler:
    """nvidia-smi samples every 20 ms, started before the warm-up (the tool
    takes a while to come up); summary() keeps the samples read between
    mark_start() and mark_end(), the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.lines = []   # (host time of reading, line)
        self.t0 = None
        self.t1 = None

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
            atexit.register(self.__exit__, None, None, None)   # never left running
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def __exit__(self, *a):
        if self.proc:
            proc, self.proc = self.proc, None
            proc.terminate()
            try:
                proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                proc.kill()
            self.th.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            if self.t0 is not None and self.t1 is not None and not (self.t0 <= t <= self.t1 + 0.02):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    """The largest x of all ranks of the initialised process group (the
    slowest replica's time); device: where the group's collectives run
    ("cuda" for NCCL, "cpu" for gloo)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, world_size: int, slowest_s: float) -> float:
    """Whole-job throughput of independent replicas: the units all ranks
    processed over the slowest rank's time."""
    return units_per_rank * world_size / slowest_s


# ---------------------------------------------------------------------------
# CPU oracle timing (the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def time_oracle(o, wl, prompt, uniforms, n_frames, budget_s):
    """The oracle's decode frames/s on one sequence after a prefill of the
    workload's prompt (prefill untimed)."""
    from oracle import Sampling as OSampling
    seq = o.prefill(prompt)
    smp = OSampling(temperature=wl["temperature"], top_p=wl["top_p"], ras_win=wl["ras_win"], allow_eos=False)
    done = 0
    t0 = time.perf_counter()
    for f in range(n_frames):
        o.decode_frame(seq, uniforms[f, 0], smp)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return done, el


def oracle_synthetic_sequence(o, cfg, n_tokens: int, seed: int):
    """An oracle sequence holding a context of n_tokens positions without a
    prefill (a 36-layer prefill of thousands of tokens takes the host far
    longer than the decode it precedes): cached K/V values seeded in [-1, 1)
    and rounded to bf16 (one layer's worth, which every layer starts from:
    the oracle appends by copying and never writes a cache in place), the
    held hidden state seeded in [-1, 1) and the held logits the restricted
    head's of it.  The values do not matter for timing; the shapes are the
    workload's."""
    from oracle import SeqState
    u = gen.gen_uniform((2, n_tokens, cfg.n_kv_head, cfg.head_dim), seed, "oracle_ctx:kv")
    x = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits((2.0 * u - 1.0).astype(np.float32)))
    kv = [[x[0], x[1]] for _ in range(cfg.n_layer)]
    h = (2.0 * gen.gen_uniform((cfg.dim,), seed, "oracle_ctx:h") - 1.0).astype(np.float32)
    return SeqState(kv=kv, pos=n_tokens, h_last=h, z_last=o.restricted_logits(h))


def time_oracle_batch(o, cfg, contexts, frames: int, budget_s: float) -> dict:
    """Teacher-forced oracle frames on sequences of the given context lengths,
    one after another (the oracle decodes a batch one sequence at a time, so
    its batch throughput is its per-sequence rate)."""
    from oracle import Sampling as OSampling
    smp = OSampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    per, total_f, total_s = [], 0, 0.0
    for i, n in enumerate(contexts):
        seq = oracle_synthetic_sequence(o, cfg, int(n), seed=7000 + i)
        forced = gen.make_forced_codes(frames, 1, cfg, seed=8000 + i)
        uni = gen.make_uniforms(frames, 1, cfg, seed=9000 + i)
        done = 0
        t0 = time.perf_counter()
        for f in range(frames):
            o.decode_frame(seq, uni[f, 0], smp, forced=forced[f, 0])
            done += 1
            if time.perf_counter() - t0 > budget_s / len(contexts):
                break
        el = time.perf_counter() - t0
        per.append({"context": int(n), "frames": done, "frames_per_s": done / el})
        total_f += done
        total_s += el
        del seq
    return {"value": total_f / total_s, "unit": "frames/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{total_f} teacher-forced frames over {len(contexts)} sequences of contexts "
                      f"{', '.join(str(int(c)) for c in contexts)} (synthetic cached K/V, no prefill), "
                      f"NumPy fp32 on {os.cpu_count()} host threads",
            "per_sequence": per}


# ---------------------------------------------------------------------------

BATCH_CONTEXTS = {
    16: dict(lo=512, hi=2048, seed=2, stream="ctx_b16"),
    64: dict(lo=1024, hi=4096, seed=3, stream="ctx_b64"),
}


def batch_contexts(b: int) -> np.ndarray:
    c = BATCH_CONTEXTS[b]
    return gen.make_lengths(b, c["lo"], c["hi"], seed=c["seed"], stream=c["stream"])


def measure_batch(cfg, w, b: int, frames: int, warmup: int, peak: float) -> dict:
    """A continuous batch of b sequences (b = 16: contexts uniform in [512,
    2,048], seed 2; b = 64: [1,024, 4,096], seed 3) set up by the
    synthetic-context hook (seeded K/V and held state, no prefill), then
    `warmup` + `frames` decode steps with seeded uniforms (seed 1), T 0.8,
    top-p 0.8, resample window 10, <|im_end|> excluded.  Device-timed with
    CUDA events."""
    import torch
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling
    from dual_ar_tts_frame_gb300 import bytemodel
    ctx = batch_contexts(b)
    lim = BATCH_CONTEXTS[b]
    max_ctx = int(ctx.max()) + warmup + frames + 8
    pages = sum(-(-(int(c) + warmup + frames + 1) // cfg.page_tokens) for c in ctx) + 8
    dec = DualARDecoder(cfg, w, max_pages=pages, max_seqs=b, max_ctx=max_ctx)
    for s in range(b):
        dec.synthetic_context(s, int(ctx[s]), seed=1000 + s)
    dec.sync()
    smp = Sampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    uni = torch.from_numpy(gen.make_uniforms(warmup + frames, b, cfg, seed=1)).cuda()
    codes = torch.empty((b, cfg.n_codebooks), dtype=torch.int32, device="cuda")
    status = torch.empty((b,), dtype=torch.int32, device="cuda")
    slots = list(range(b))
    stream = torch.cuda.current_stream()
    for f in range(warmup):
        dec.decode_frame(slots, uni[f], smp, codes, status)
    dec.sync()
    launches = dec.last_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for f in range(warmup, warmup + frames):
        dec.decode_frame(slots, uni[f], smp, codes, status)
    ev1.record(stream)
    torch.cuda.synchronize()
    dec.sync()
    ms = ev0.elapsed_time(ev1)
    assert int(status.max().item()) == 0
    bytes_total = sum(bytemodel.frame_bytes(cfg, [int(c) + f + 1 for c in ctx]) for f in range(warmup, warmup + frames))
    gbs = bytes_total / (ms / 1000.0) / 1e9
    dec.close()
    return {"workload": f"full S2-Pro-shaped Dual-AR, batch {b}, contexts uniform in [{lim['lo']}, {lim['hi']}] "
                        f"(seed {lim['seed']}, synthetic K/V and held state, no prefill), T=0.8 top-p 0.8 "
                        f"RAS window 10; {warmup + frames} steps ({warmup} warm-up, {frames} timed)",
            "value": b * frames / (ms / 1000.0), "unit": "frames/s", "steps": frames, "warmup": warmup,
            "ms_per_step": ms / frames, "rtf": FRAMES_PER_AUDIO_SECOND / (frames / (ms / 1000.0)),
            "frame_bytes_per_step": bytes_total / frames,
            "frame_roofline": {"achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak},
            "gpu_launches_per_step": launches}


def measure_batch64(cfg, w, frames: int, warmup: int, peak: float) -> dict:
    return measure_batch(cfg, w, 64, frames, warmup, peak)


def measure_two_streams(cfg, w, frames: int, warmup: int) -> dict:
    """The batch-64 workload (contexts uniform in [1,024, 4,096], seed 3,
    synthetic K/V) decoded by one decoder, then split into two decoders of
    32 sequences on two CUDA streams whose steps run concurrently (with an
    offset of 0 or 1 step), so the fast AR of one group can overlap the slow
    step of the other.  Device-timed from one event before both streams to
    one after both; frames/s over all 64 sequences."""
    import torch
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling
    ctx = batch_contexts(64)
    smp = Sampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    uni = torch.from_numpy(gen.make_uniforms(warmup + frames, 64, cfg, seed=1)).cuda()

    def make(cs, stream, seed0):
        pages = sum(-(-(int(c) + warmup + frames + 2) // cfg.page_tokens) for c in cs) + 8
        d = DualARDecoder(cfg, w, max_pages=pages, max_seqs=len(cs), max_ctx=int(max(cs)) + warmup + frames + 8,
                          stream=stream)
        for s in range(len(cs)):
            d.synthetic_context(s, int(cs[s]), seed=seed0 + s)
        return d

    def bufs(b):
        return (torch.empty((b, cfg.n_codebooks), dtype=torch.int32, device="cuda"),
                torch.empty((b,), dtype=torch.int32, device="cuda"))

    out = {}
    st = torch.cuda.Stream()
    d = make(ctx, st, 1000)
    c, s_ = bufs(64)
    with torch.cuda.stream(st):
        for f in range(warmup):
            d.decode_frame(list(range(64)), uni[f], smp, c, s_)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    with torch.cuda.stream(st):
        for f in range(warmup, warmup + frames):
            d.decode_frame(list(range(64)), uni[f], smp, c, s_)
    e1.record(st)
    torch.cuda.synchronize()
    d.sync()
    d.close()
    ms = e0.elapsed_time(e1)
    out["one_decoder_b64"] = {"frames_per_s": 64 * frames / (ms / 1000.0), "ms_per_step": ms / frames}
    torch.cuda.empty_cache()
    for off in (0, 1):
        sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
        da, db = make(ctx[:32], sa, 1000), make(ctx[32:], sb, 1032)
        ua, ub = uni[:, :32].contiguous(), uni[:, 32:].contiguous()
        (ca, sa_), (cb, sb_) = bufs(32), bufs(32)
        for f in range(warmup):
            with torch.cuda.stream(sa):
                da.decode_frame(list(range(32)), ua[f], smp, ca, sa_)
            with torch.cuda.stream(sb):
                db.decode_frame(list(range(32)), ub[f], smp, cb, sb_)
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea, eb = torch.cuda.Event(), torch.cuda.Event()
        t0.record(cur)
        sa.wait_event(t0)
        sb.wait_event(t0)
        for f in range(warmup, warmup + frames):
            with torch.cuda.stream(sa):
                da.decode_frame(list(range(32)), ua[f], smp, ca, sa_)
            if f - warmup >= off:
                with torch.cuda.stream(sb):
                    db.decode_frame(list(range(32)), ub[f - off], smp, cb, sb_)
        for f in range(warmup + frames - off, warmup + frames):
            with torch.cuda.stream(sb):
                db.decode_frame(list(range(32)), ub[f], smp, cb, sb_)
        ea.record(sa)
        eb.record(sb)
        cur.wait_event(ea)
        cur.wait_event(eb)
        t1.record(cur)
        torch.cuda.synchronize()
        da.sync()
        db.sync()
        da.close()
        db.close()
        ms = t0.elapsed_time(t1)
        out[f"two_decoders_b32_offset{off}"] = {"frames_per_s": 64 * frames / (ms / 1000.0),
                                                "ms_per_pair_of_steps": ms / frames}
        torch.cuda.empty_cache()
    return out


def measure_replacement(cfg, w, frames: int, peak: float, with_prefill: bool) -> dict:
    """Batch 128 with replacement: 124 contexts uniform in [2,048, 4,096] and
    4 of 16,384 (seed 4), set up by the synthetic-context hook; every step
    decodes all 128 slots, then each sequence whose seeded finish frame has
    come is released and its slot restarted from the queue.  The decode steps
    are device-timed one by one (CUDA events around each call), so the
    replacements' set-up is excluded; with_prefill restarts slots with a real
    prefill of a seeded prompt of the queued length and also reports the
    wall time of the whole loop, prefill included."""
    import torch
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling
    from dual_ar_tts_frame_gb300 import bytemodel
    b = 128
    wl = gen.make_replacement_workload(b, 4, 4 * b, seed=4)
    ctx = [int(c) for c in wl["ctx"]]
    max_ctx = max(ctx) + frames + 16
    # every short slot may hold a 4,096-token context plus its growth at any time
    per = lambda n: -(-(n + frames + 4) // cfg.page_tokens)  # noqa: E731
    pages = (b - 4) * per(4096) + sum(per(c) for c in ctx[-4:]) + 8
    dec = DualARDecoder(cfg, w, max_pages=pages, max_seqs=b, max_ctx=max_ctx)
    for s in range(b):
        dec.synthetic_context(s, ctx[s], seed=3000 + s)
    dec.sync()
    smp = Sampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    uni = torch.from_numpy(gen.make_uniforms(frames, b, cfg, seed=1)).cuda()
    codes = torch.empty((b, cfg.n_codebooks), dtype=torch.int32, device="cuda")
    status = torch.empty((b,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    slots = list(range(b))
    length = list(ctx)
    finish = [int(f) for f in wl["finish"]]
    q = 0
    step_ms = 0.0
    step_bytes = 0
    replaced = 0
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(frames)]
    for f in range(3):   # untimed warm-up steps before the schedule starts
        dec.decode_frame(slots, uni[f], smp, codes, status)
        length = [n + 1 for n in length]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for f in range(frames):
        step_bytes += bytemodel.frame_bytes(cfg, [n + 1 for n in length])
        evs[f][0].record(stream)
        dec.decode_frame(slots, uni[f], smp, codes, status)
        evs[f][1].record(stream)
        for s in slots:
            length[s] += 1
            if finish[s] == f + 1:
                dec.release(s)
                n = int(wl["queue_ctx"][q])
                if with_prefill:
                    dec.prefill(s, gen.make_prompt(cfg, n, seed=5000 + q))
                else:
                    dec.synthetic_context(s, n, seed=5000 + q)
                length[s] = n
                finish[s] = f + 1 + int(wl["queue_finish"][q])
                q += 1
                replaced += 1
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    dec.sync()
    step_ms = sum(a.elapsed_time(z) for a, z in evs)
    dec.close()
    gbs = step_bytes / (step_ms / 1000.0) / 1e9
    r = {"workload": WORKLOADS["s2pro_b128_replace"]["desc"] + " (synthetic K/V and held state for the "
                     "initial contexts" + ("; replacements prefilled" if with_prefill else "; replacements "
                     "set up by the synthetic-context hook") + ")",
         "value": b * frames / (step_ms / 1000.0), "unit": "frames/s", "steps": frames,
         "ms_per_step": step_ms / frames, "replaced_sequences": replaced,
         "frame_bytes_per_step": step_bytes / frames,
         "frame_roofline": {"achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak}}
    if with_prefill:
        r["prefill_included"] = {"value": b * frames / wall, "unit": "frames/s", "wall_s": wall,
                                 "note": "host wall clock of the whole loop: decode steps plus the "
                                         "replacements' prefills"}
    return r


def measure_w4a16(cfg, w, prompt, frames: int, warmup: int, peak: float) -> dict:
    """Batch 1 with 4-bit weights: the "late12attn" plan (every projection
    packed except the query/key/value and output projections of the last 12
    slow layers; embeddings, norms and heads bf16), packed on the GPU from
    the same bf16 weights.  The benchmark's 512-token prompt is prefilled
    through the packed weights, then `warmup` + `frames` frames (seed-1
    uniforms, T 0.8, top-p 0.8, RAS 10, <|im_end|> excluded), device-timed;
    then a few frames with every GEMV launch bracketed by events for the
    GEMV kernel's own roofline."""
    import torch
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling, late_attn_keys, pack_w4a16
    from dual_ar_tts_frame_gb300 import bytemodel
    keys = late_attn_keys(cfg.n_layer, cfg.fast_n_layer, 12)
    packed = {k: pack_w4a16(w[k]) for k in keys}
    max_ctx = len(prompt) + warmup + frames + 16
    dec = DualARDecoder(cfg, w, max_pages=(max_ctx + 63) // 64 + 2, max_seqs=1, max_ctx=max_ctx)
    dec.set_w4a16(packed)
    stream = torch.cuda.current_stream()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    dec.prefill(0, prompt)
    p1.record(stream)
    dec.sync()
    prefill_ms = p0.elapsed_time(p1)
    smp = Sampling(temperature=0.8, top_p=0.8, ras_win=10, allow_eos=False)
    n_prof = 4
    uni = torch.from_numpy(gen.make_uniforms(warmup + frames + n_prof, 1, cfg, seed=1)).cuda()
    codes = torch.empty((1, cfg.n_codebooks), dtype=torch.int32, device="cuda")
    status = torch.empty((1,), dtype=torch.int32, device="cuda")
    for f in range(warmup):
        dec.decode_frame([0], uni[f], smp, codes, status)
    dec.sync()
    launches = dec.last_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for f in range(warmup, warmup + frames):
        dec.decode_frame([0], uni[f], smp, codes, status)
    ev1.record(stream)
    torch.cuda.synchronize()
    dec.sync()
    ms = ev0.elapsed_time(ev1)
    assert int(status.item()) == 0
    dec.profile(True)
    for f in range(warmup + frames, warmup + frames + n_prof):
        dec.decode_frame([0], uni[f], smp, codes, status)
    dec.profile(False)
    prof = dec.profile_read()
    dec.close()
    att = [len(prompt) + f + 1 for f in range(warmup, warmup + frames)]
    bytes_total = sum(bytemodel.frame_bytes(cfg, [a], keys) for a in att)
    gbs = bytes_total / (ms / 1000.0) / 1e9
    # the dominant kernel of the profiled frames: the persistent frame kernel
    # (one launch per frame, no GEMV bytes recorded; its algorithmic bytes
    # are the frame's) or, per op, the GEMV launches
    persistent = prof["total_bytes"] == 0.0 and prof["launches"] == n_prof
    prof_att = [len(prompt) + f + 1 for f in range(warmup + frames, warmup + frames + n_prof)]
    if persistent:
        kname = "mega_kernel (persistent frame kernel, 4-bit variant)"
        kbytes = sum(bytemodel.frame_bytes(cfg, [a], keys) for a in prof_att)
    else:
        kname = "gemv_kernel (4-bit and bf16 weight-streaming GEMV)"
        kbytes = prof["total_bytes"]
    k_gbs = kbytes / (prof["total_ms"] / 1000.0) / 1e9 if prof["total_ms"] > 0 else None
    return {"workload": f"full S2-Pro-shaped Dual-AR, batch 1, {len(prompt)}-token prompt, 4-bit weights "
                        f"(late12attn plan: {len(keys)} of {5 * (cfg.n_layer + cfg.fast_n_layer)} block projections packed, "
                        "group 128, bf16 scales), "
                        "T=0.8 top-p 0.8 RAS window 10",
            "value": frames / (ms / 1000.0), "unit": "frames/s", "steps": frames, "warmup": warmup,
            "ms_per_step": ms / frames, "rtf": FRAMES_PER_AUDIO_SECOND / (frames / (ms / 1000.0)),
            "packed_projections": len(keys), "frame_bytes_per_step": bytes_total / frames,
            "frame_roofline": {"achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak},
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": k_gbs, "peak": peak, "unit": "GB/s",
                         "frac": (k_gbs / peak) if k_gbs else None, "launches": prof["launches"],
                         "frames": n_prof, "bytes_per_frame": kbytes / n_prof,
                         "ms_per_frame": prof["total_ms"] / n_prof},
            "prefill_ms": prefill_ms, "gpu_launches_per_step": launches}


def main():
    args = parse()
    wl = WORKLOADS[args.workload]
    cfg = CONFIGS[wl["cfg"]]
    ws, rank, local = dist_env()
    W = args.warmup if args.warmup is not None else min(16, wl["frames"] // 4)
    K = args.steps if args.steps is not None else wl["frames"] - W
    assert W >= 0 and K >= 1
    prompt = gen.make_prompt(cfg, wl["prompt"], seed=0)
    uni_all = gen.make_uniforms(W + K, wl["batch"], cfg, seed=1)
    config = {"workload": f"{args.workload}: {wl['desc']}; {W + K} frames ({W} warm-up, {K} timed)",
              "batch": wl["batch"],
              "prompt_tokens": wl["prompt"], "frames": W + K,
              "l2": "inputs larger than L2 (9.1 GB of weights streamed per frame); no flush"}
    if args.workload != "s2pro_b1":
        config["l2"] = "small profiling/parity workload, not a bench line"

    if args.workload == "s2pro_b128_replace":
        # the batch-128 replacement workload alone (not part of the default line)
        import torch
        from dual_ar_tts_frame_gb300 import build, upload_weights
        torch.cuda.set_device(local)
        build()
        w = upload_weights(gen.make_weights(cfg, seed=0))
        peak, _ = peaks()
        for with_prefill in (False, True):
            r = measure_replacement(cfg, w, frames=W + K, peak=peak, with_prefill=with_prefill)
            print(json.dumps({"metric": METRIC, "impl": "ours", "config": {"workload": r["workload"]}, **r}),
                  flush=True)
        return

    if args.workload == "s2pro_b64_two_streams":
        # the co-scheduling comparison alone (not part of the default line)
        import torch
        from dual_ar_tts_frame_gb300 import build, upload_weights
        torch.cuda.set_device(local)
        build()
        w = upload_weights(gen.make_weights(cfg, seed=0))
        r = measure_two_streams(cfg, w, frames=K, warmup=max(W, 3))
        print(json.dumps({"metric": METRIC, "impl": "ours", "unit": "frames/s",
                          "config": {"workload": f"{args.workload}: {wl['desc']}; {K} timed steps"}, **r}), flush=True)
        return

    if args.workload in ("s2pro_b64", "s2pro_l1_b64"):
        # the batch-64 measurement alone (also part of the default line)
        import torch
        from dual_ar_tts_frame_gb300 import build, upload_weights
        torch.cuda.set_device(local)
        build()
        w = upload_weights(gen.make_weights(cfg, seed=0))
        peak, _ = peaks()
        r = measure_batch64(cfg, w, frames=K, warmup=W, peak=peak)
        print(json.dumps({"metric": METRIC, "impl": "ours", "config": {"workload": r["workload"]}, **r}), flush=True)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        bits = gen.make_weights(cfg, seed=0)
        from oracle import DualAROracle
        o = DualAROracle(cfg, bits, max_pos=wl["prompt"] + W + K + 8)
        done, el = time_oracle(o, wl, prompt, uni_all, W + K, budget_s=150.0)
        fps = done / el
        cores = os.cpu_count()
        line = {"impl": "reference", "metric": METRIC, "value": fps, "unit": "frames/s", "n_gpus": ws,
                "steps": done, "warmup": 0, "ms_per_step": 1000.0 * el / done, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": fps, "unit": "frames/s", "cores": cores, "kind": "oracle",
                                 "sample": f"{done} frames after a {wl['prompt']}-token prefill "
                                           f"(prefill untimed), NumPy fp32 on {cores} host threads"},
                "e2e": {"value": fps, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from dual_ar_tts_frame_gb300 import DualARDecoder, Sampling, build, upload_weights
    from dual_ar_tts_frame_gb300 import bytemodel
    build()
    # the clock sampler starts now (nvidia-smi takes a while to come up) and
    # keeps only the samples of the timed region below
    clk = ClockSampler(local).__enter__()
    bits = gen.make_weights(cfg, seed=0)
    w = upload_weights(bits)
    if ws > 1 or args.no_cpu_baseline:
        del bits
        bits = None
    b = wl["batch"]
    max_ctx = wl["prompt"] + W + K + 8
    pages_per = (max_ctx + cfg.page_tokens - 1) // cfg.page_tokens
    dec = DualARDecoder(cfg, w, max_pages=2 * b * pages_per + 2, max_seqs=2 * b, max_ctx=max_ctx)
    smp = Sampling(temperature=wl["temperature"], top_p=wl["top_p"], ras_win=wl["ras_win"], allow_eos=False)
    slots = list(range(b))
    for s in slots:
        dec.prefill(s, prompt)
    dec.sync()
    uni = torch.from_numpy(uni_all).cuda()
    codes = torch.empty((b, cfg.n_codebooks), dtype=torch.int32, device="cuda")
    status = torch.empty((b,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    for f in range(W):
        dec.decode_frame(slots, uni[f], smp, codes, status)
    dec.sync()
    launches_per_frame = dec.last_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    dec.profile(True)
    clk.mark_start()
    ev0.record(stream)
    for f in range(W, W + K):
        dec.decode_frame(slots, uni[f], smp, codes, status)
    ev1.record(stream)
    torch.cuda.synchronize()
    clk.mark_end()
    clk.__exit__(None, None, None)
    dec.profile(False)
    dec.sync()
    prof = dec.profile_read()
    ms = ev0.elapsed_time(ev1)
    if ws > 1:
        ms = max_over_ranks(ms, "cuda")
    value = replica_throughput(b * K, ws, ms / 1000.0)
    ms_per_step = ms / K
    # byte model over the timed frames: contexts grow by one per frame
    att = [wl["prompt"] + f + 1 for f in range(W, W + K)]
    bytes_total = sum(bytemodel.frame_bytes(cfg, [a] * b) for a in att)
    peak, peak_src = peaks()
    frame_gbs = bytes_total / (ms / 1000.0) / 1e9
    tr = traffic_record()
    persistent = prof["total_bytes"] == 0.0 and prof["launches"] == K
    if persistent:
        # the persistent frame kernel is the dominant (only) kernel of a step:
        # its algorithmic bytes are the frame's (byte model), its time the
        # CUDA-event duration of its launches
        kname = "mega_kernel (persistent frame kernel)"
        kbytes = bytes_total / K
    else:
        kname = "gemv_kernel (weight-streaming GEMV)"
        kbytes = prof["total_bytes"] / max(1, prof["launches"])
    avg_us = 1000.0 * prof["total_ms"] / max(1, prof["launches"])
    kgbs = kbytes / (avg_us * 1e-6) / 1e9 if avg_us > 0 else None
    e2e = None
    prefill = None
    if not args.no_e2e:
        # end to end through the public API: pinned host uniforms in, codes and
        # status out, the host reading each frame's result before the next
        eslots = [b + s for s in slots]
        pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pe0.record(stream)
        for s in eslots:
            dec.prefill(s, prompt)
        pe1.record(stream)
        dec.sync()
        prefill = {"prompt_tokens": wl["prompt"], "ms_per_sequence": pe0.elapsed_time(pe1) / len(eslots),
                   "note": "the prompt's prefill (chunks of up to 128 rows on the tensor cores), device-timed; "
                           "the first audio frame follows one decode step later"}
        prefill["tokens_per_s"] = wl["prompt"] / (prefill["ms_per_sequence"] / 1000.0)
        hu = torch.from_numpy(uni_all).pin_memory()
        du = torch.empty((b, cfg.n_codebooks + 1), dtype=torch.float32, device="cuda")
        hc = torch.empty((b, cfg.n_codebooks), dtype=torch.int32).pin_memory()
        hs = torch.empty((b,), dtype=torch.int32).pin_memory()
        for f in range(W):
            du.copy_(hu[f], non_blocking=True)
            dec.decode_frame(eslots, du, smp, codes, status)
            hc.copy_(codes, non_blocking=True)
            hs.copy_(status, non_blocking=True)
            stream.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for f in range(W, W + K):
            du.copy_(hu[f], non_blocking=True)
            dec.decode_frame(eslots, du, smp, codes, status)
            hc.copy_(codes, non_blocking=True)
            hs.copy_(status, non_blocking=True)
            stream.synchronize()
            assert int(hs[0]) == 0
        el = time.perf_counter() - t0
        if ws > 1:
            el = max_over_ranks(el, "cuda")
        e2e = {"value": replica_throughput(b * K, ws, el), "unit": "frames/s", "h2d_bytes_per_step": hu[0].numel() * 4,
               "d2h_bytes_per_step": hc.numel() * 4 + hs.numel() * 4}

    dec.close()
    b16 = b64 = b128 = None
    if args.workload == "s2pro_b1" and not args.no_batches:
        b16 = measure_batch(cfg, w, 16, frames=24, warmup=4, peak=peak)
        b64 = measure_batch64(cfg, w, frames=24, warmup=4, peak=peak)
        b128 = {"decode": measure_replacement(cfg, w, frames=64, peak=peak, with_prefill=False),
                "prefill_included": measure_replacement(cfg, w, frames=64, peak=peak, with_prefill=True)}
    w4 = None
    if args.workload in ("s2pro_b1", "s2pro_l1_b1") and not args.no_w4a16:
        w4 = measure_w4a16(cfg, w, prompt, frames=64, warmup=8, peak=peak)

    cpu = cpu_batch = None
    if rank == 0 and ws == 1 and bits is not None:
        from oracle import DualAROracle
        n_or = 8 if cfg.name == "s2pro" else 16
        o = DualAROracle(cfg, bits, max_pos=max(16_400, wl["prompt"] + n_or + 8))
        done, el = time_oracle(o, wl, prompt, uni_all, n_or, budget_s=25.0)
        cpu = {"value": done / el, "unit": "frames/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{done} frames of this workload after a {wl['prompt']}-token prefill "
                         f"(prefill untimed), batch 1, NumPy fp32"}
        if args.workload == "s2pro_b1" and not args.no_batches:
            repl = gen.make_replacement_workload(128, 4, 512, seed=4)["ctx"]
            cpu_batch = {"batch16": time_oracle_batch(o, cfg, batch_contexts(16)[:2], 8, budget_s=12.0),
                         "batch64": time_oracle_batch(o, cfg, batch_contexts(64)[:2], 8, budget_s=12.0),
                         "batch128_replace": time_oracle_batch(o, cfg, [repl[0], repl[-1]], 8, budget_s=16.0)}
        del o

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "weights_dtype": "bf16",
            "data": "synthetic: seeded random-init weights N(0,0.02) (norm gains 1+N(0,0.02)), "
                    "uniform prompt ids, counter-based uniforms",
            "config": config,
            "rtf": FRAMES_PER_AUDIO_SECOND / (value / (b * ws)),
            "frame_bytes_per_step": bytes_total / K,
            "frame_roofline": {"achieved": frame_gbs, "peak": peak, "unit": "GB/s",
                               "frac": frame_gbs / peak},
            "roofline": {"bound": "hbm", "kernel": kname,
                         "achieved": kgbs, "peak": peak, "unit": "GB/s",
                         "frac": (kgbs / peak) if kgbs else None,
                         "traffic": tr["dram_bytes_per_launch"] if (tr and tr.get("kernel") == kname) else None,
                         "bytes_per_launch": kbytes, "avg_launch_us": avg_us,
                         "launches": prof["launches"], "share_of_step": prof["total_ms"] / ms,
                         "peak_source": peak_src},
            "e2e": e2e,
            "prefill": prefill,
            "gpu_launches": launches_per_frame * K,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "cpu_baseline_batch": cpu_batch,
            "batch16": b16,
            "batch64": b64,
            "batch128_replace": b128,
            "w4a16": w4,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
