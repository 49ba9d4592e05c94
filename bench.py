#!/usr/bin/env python3
"""Benchmark: GPT-2 124M cachedStep decode tokens/s on one GB300, and the
achieved HBM bandwidth of the step kernel against the measured peak.

Workload (one bench step): GPT-2 124M shapes, binary32 packed checkpoint with
N(0, 0.02) weights from a fixed seed (synthetic: no pretrained weights exist
here); 16 uniform random prompt tokens fill positions 0..15 once; each bench
step rewinds the session to position 16 and runs 112 greedy cachedStep
decode steps (positions 16..127) as ONE persistent kernel launch, the next
token chosen on the device.  The weights (495 MB per token) are larger than
the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quant f32|int8]

Multi-GPU runs (torchrun) are independent replicas: one session per GPU, no
data exchange; value = all tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GPT-2 124M cachedStep tokens/s on 1 GB300; achieved HBM GB/s vs peak"
PROMPT = 16
DECODE = 112  # decode positions per bench step (--decode-steps)
KV_ROW_BYTES = 12 * 1536 * 4  # one cached position (README cachedStep paragraph)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def step_bytes(shape, quant: str, p: int) -> int:
    """Algorithmic HBM bytes of one cachedStep at position p: every weight the
    step needs once (block matrices, LayerNorm parameters, biases, the tied
    vocabulary matrix, one position row), the KV cache read at positions
    0..p-1, this position's KV write and the logits write."""
    d, F, L, V = shape.d_model, shape.d_ff, shape.n_layer, shape.vocab
    params = L * (2 * d + 3 * d + d + 2 * d + F + d) + 2 * d + d  # LN, biases, final LN, one wpe row
    if quant in ("f32", "f16"):
        mats = L * (d * 3 * d + d * d + d * F + F * d) + V * d
        weights = (4 if quant == "f32" else 2) * mats + 4 * params
    elif quant in ("int8_row", "int8_row_act"):
        rb = lambda K: K + 4  # one scale per row (the device copy repeats it per group)
        mats = L * (3 * d * rb(d) + d * rb(d) + F * rb(d) + d * rb(F)) + V * rb(d)
        weights = mats + 4 * params
    else:
        rb = lambda K: K + (K // 64) * 4
        mats = L * (3 * d * rb(d) + d * rb(d) + F * rb(d) + d * rb(F)) + V * rb(d)
        weights = mats + 4 * params
    return weights + KV_ROW_BYTES * p + KV_ROW_BYTES + 4 * V


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                self.rows.append(f)

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def combine_replicas(ms_local: float, ws: int):
    """Whole-job figures of N independent replicas: the slowest rank's ms per
    launch (max over ranks, gloo) and the tokens of all ranks over that time."""
    ms = ms_local
    if ws > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_local], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, ws * DECODE / (ms * 1e-3)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def oracle_decode_rate(shape, w, toks, quant: int, n_decode: int, passes: int = 1):
    """Times the oracle (single-threaded C) on the decode workload: the prompt
    cache is built untimed, then `passes` runs of n_decode greedy steps from
    it are timed."""
    from oracle import Oracle
    om = Oracle().model(shape, w, quant=quant)
    _, ch, cache0 = om.session(list(toks), PROMPT)
    t0 = time.perf_counter()
    for _ in range(passes):
        cache, tok = cache0, int(ch[-1])
        for i in range(n_decode):
            st, lg, cache = om.cached_step(cache, tok, PROMPT + i)
            tok = int(np.argmax(lg))
    dt = time.perf_counter() - t0
    om.close()
    return passes * n_decode / dt, dt


def reference_arm(args, shape, w, toks):
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    quant = {"f32": 0, "int8": 1, "f16": 2, "int8_row": 3, "int8_row_act": 4}[args.quant]
    per_step = 2
    from oracle import Oracle
    om = Oracle().model(shape, w, quant=quant)
    _, ch, cache0 = om.session(list(toks), PROMPT)
    tok0 = int(ch[-1])

    def one_step():
        cache, tok = cache0, tok0
        for i in range(per_step):
            st, lg, cache = om.cached_step(cache, tok, PROMPT + i)
            tok = int(np.argmax(lg))

    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    sample = f"{per_step} teacher-free greedy oracle steps at positions 16..{16 + per_step - 1} per bench step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": args.quant, "data": "synthetic",
            "config": workload_config(args),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(args):
    return {"workload": f"gpt2-124m {args.quant} cachedStep greedy decode, 16-token prompt then {DECODE} steps "
                        f"(positions 16..{15 + DECODE}), one persistent launch per {DECODE} steps",
            "tokens_per_step": DECODE, "positions": f"16..{15 + DECODE}", "model_shape": "12x768, 12 heads, ffn 3072, "
            "vocab 50257", "l2": "inputs larger than L2 (weights 495 MB f32 / 249 MB f16 / 132 MB int8 per token)",
            "parallelism": f"replicas x{args.gpus}"}


def traffic_from_profiles(kernel_src_hash: str, quant: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "step_kernel_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(quant)
        if e and e.get("kernel_sha256") == kernel_src_hash:
            return e["dram_bytes_per_launch_112_steps"]
    except Exception:
        pass
    return None


# Sources of each step kernel (the traffic record is keyed by their hash).
KERNEL_SOURCES = {"cluster": ("cstep.cu", "cstep.cuh", "gpt2_dev.cuh"), "phase": ("decode.cu", "gpt2_dev.cuh")}
KERNEL_NAMES = {"cluster": "cstep_kernel", "phase": "step_kernel"}


def kernel_hash(kind: str = "phase"):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "stream_decode_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


PREFILL_GFLOP_128 = 21.82  # GEMMs (2 x 128 x 85M block weights) + attention + the last row's head


def prefill_rate(g, torch, shape, w, n: int = 128, reps: int = 10):
    """The 128-token full-prefix pass (gpt2_session_prefill, tensor cores):
    median ms over `reps` calls (CUDA events on the launching stream, the
    session rewound to position 0 between calls) and algorithmic TFLOP/s."""
    from stream_decode_gb300 import synth
    model = g.Model(shape, w)
    sess = g.Session(model)
    toks = torch.tensor(synth.tokens(shape.vocab, n, seed=11).astype(np.int32), device="cuda")
    lg = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(3):
        assert sess.rewind(0) == "ok" and sess.prefill(toks, n, lg, None, st) == "ok"
    assert sess.sync() == "ok"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(reps):
        assert sess.rewind(0) == "ok"
        e0.record(st)
        assert sess.prefill(toks, n, lg, None, st) == "ok"
        e1.record(st)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    assert sess.sync() == "ok"
    sess.close()
    model.close()
    ms = float(np.median(times))
    return {"tokens": n, "ms_per_infer": ms, "TFLOP_per_s": PREFILL_GFLOP_128 * (n / 128) / ms,
            "arith": "3xTF32 tcgen05 GEMMs, binary32 elsewhere"}


def measure_decode(g, torch, shape, w, toks, quant: str, args, rank_sync):
    """Returns (ms per bench step, launches, session) after W warm-ups and K timed steps."""
    q = {"f32": g.F32, "int8": g.INT8_G64, "f16": g.F16, "int8_row": g.INT8_ROW, "int8_row_act": g.INT8_ROW_ACT}[quant]
    model = g.Model(shape, w, quant=q)
    sess = g.Session(model)
    V = shape.vocab
    stream = torch.cuda.current_stream()
    d_prompt = torch.tensor(np.asarray(toks, np.int32), device="cuda")
    tout = torch.empty(max(PROMPT, DECODE), dtype=torch.int32, device="cuda")  # the prompt run writes PROMPT ids
    assert sess.run(d_prompt, PROMPT, None, 0, tout) == "ok"
    assert sess.sync() == "ok"
    first = int(tout[PROMPT - 1].item())
    tin = torch.full((DECODE,), -1, dtype=torch.int32, device="cuda")
    tin[0] = first
    logits = torch.empty(V, dtype=torch.float32, device="cuda")

    def one():
        assert sess.rewind(PROMPT) == "ok"
        assert sess.run(tin, DECODE, logits, 0, tout, stream) == "ok"

    for _ in range(args.warmup):
        one()
    assert sess.sync() == "ok"
    torch.cuda.synchronize()
    rank_sync()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id(torch)) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            one()
        e1.record(stream)
        torch.cuda.synchronize()
    rank_sync()
    st = sess.sync()
    assert st == "ok", st
    ms = e0.elapsed_time(e1) / args.steps
    return ms, args.steps, model, sess, first, clk.summary()


def gpu_id(torch) -> str:
    """nvidia-smi --id of the current device (its UUID when torch knows it)."""
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(torch.cuda.current_device())


def measure_e2e(g, sess, shape, first, n_steps):
    """Host buffers through the C ABI, one call per bench step
    (gpt2_session_run_host): the step's token ids go in from pinned host
    memory, one persistent launch decodes them, and every position's logits
    and greedy choice come back to pinned host memory before the call
    returns.  Wall clock over n_steps calls (after one untimed call)."""
    import torch
    tin = torch.full((DECODE,), -1, dtype=torch.int32, pin_memory=True)
    tin[0] = first
    logits = torch.empty((DECODE, shape.vocab), dtype=torch.float32, pin_memory=True)
    tout = torch.zeros(DECODE, dtype=torch.int32, pin_memory=True)
    assert sess.rewind(PROMPT) == "ok" and sess.run_host(tin, DECODE, logits, tout) == "ok"
    t0 = time.perf_counter()
    for _ in range(n_steps):
        assert sess.rewind(PROMPT) == "ok"
        st = sess.run_host(tin, DECODE, logits, tout)
        assert st == "ok", st
    dt = time.perf_counter() - t0
    return DECODE * n_steps / dt, dt


def measure_e2e_per_token(g, sess, shape, first, n_steps):
    """Interactive use: one gpt2_session_step_host call per token (token in
    as a call argument, that step's logits and choice back in pinned host
    memory), the next token taken from the returned choice on the host."""
    import torch
    host = torch.empty(shape.vocab, dtype=torch.float32, pin_memory=True)
    nxt = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    t0 = time.perf_counter()
    for _ in range(n_steps):
        assert sess.rewind(PROMPT) == "ok"
        tok = first
        for i in range(DECODE):
            st = sess.step_host(tok, host, nxt)
            assert st == "ok", st
            tok = int(nxt.item()) & 0xFFFFFFFF
    dt = time.perf_counter() - t0
    return DECODE * n_steps / dt, dt


def long_context(g, torch, w, reps=20):
    """µs per cachedStep at p = 128, 512, 1023 over a cache of uniform random
    tokens (the long-context configuration)."""
    from stream_decode_gb300 import synth
    s = synth.GPT2_124M_LONG
    model = g.Model(s, w)
    sess = g.Session(model)
    toks = synth.tokens(s.vocab, 1024, seed=1234)
    d = torch.tensor(toks.astype(np.int32), device="cuda")
    assert sess.run(d, 1023, None, 0, None) == "ok"
    assert sess.sync() == "ok"
    row = g.cache_words_per_position(s)
    cache = sess.read_cache()  # positions 0..1022, for the oracle's step below
    assert cache.size == 1023 * row
    out = {}
    stream = torch.cuda.current_stream()
    # a session rewinds only backwards: the positions are timed in descending
    # order (a step at p rewrites row p with the same token's key and value)
    for p in (1023, 512, 128):
        tin = d[p:p + 1]
        for _ in range(3):
            assert sess.rewind(p) == "ok"
            assert sess.run(tin, 1, None, 0, None, stream) == "ok"
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            sess.rewind(p)
            sess.run(tin, 1, None, 0, None, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        assert sess.sync() == "ok"
        us = 1e3 * e0.elapsed_time(e1) / reps
        by = step_bytes(s, "f32", p)
        out[f"p{p}"] = {"us_per_step": us, "GB_per_s": by / us * 1e-3, "bytes": by}
    # the oracle's step at position 1023 on the cache the GPU built
    # (single-threaded C on one host core): the long-context CPU baseline
    sess.close()
    model.close()
    from oracle import Oracle
    om = Oracle().model(s, w)
    t0 = time.perf_counter()
    st, lg, _ = om.cached_step(cache, int(toks[1023]), 1023)
    dt = time.perf_counter() - t0
    om.close()
    assert st == "ok", st
    out["oracle_p1023"] = {"tokens_per_s": 1.0 / dt, "s_per_step": dt, "cores": 1,
                           "sample": "one cachedStep at position 1023 over the GPU-built 1023-position cache"}
    return out


BLOCK_PARAMS_124M = 12 * (768 * 2304 + 768 * 768 + 768 * 3072 + 3072 * 768)  # block-matrix weights


def batched_decode(g, torch, shape, w, B: int, reps: int = 5):
    """B independent sessions (gpt2_batch_run): a 16-token teacher-forced
    prompt each, then 112 greedy steps at positions 16..127 per timed run
    (the batch rewound to 16 before each run, logits written every step).
    Returns tokens/s over all sessions and the algorithmic bytes and flops:
    the binary32 weights once per step for all B rows, each session's KV
    rows and logits; 2 flops per weight per session plus attention."""
    from stream_decode_gb300 import synth
    model = g.Model(shape, w)
    bt = g.Batch(model, B)
    V = shape.vocab
    prompt = synth.tokens(V, PROMPT * B, seed=77).reshape(PROMPT, B).astype(np.int32)
    d_prompt = torch.tensor(prompt, device="cuda")
    pout = torch.zeros((PROMPT, B), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    assert bt.run(d_prompt, PROMPT, None, 0, pout, stream) == "ok"
    assert bt.sync() == "ok"
    dec = torch.full((DECODE, B), -1, dtype=torch.int32, device="cuda")
    dec[0] = pout[PROMPT - 1]
    dout = torch.zeros((DECODE, B), dtype=torch.int32, device="cuda")
    logits = torch.empty((B, V), dtype=torch.float32, device="cuda")

    def one():
        assert bt.rewind(PROMPT, stream) == "ok"
        assert bt.run(dec, DECODE, logits, 0, dout, stream) == "ok"

    for _ in range(3):
        one()
    assert bt.sync() == "ok"
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    assert bt.sync() == "ok"
    ms = e0.elapsed_time(e1) / reps
    bt.close()
    model.close()
    d, L = shape.d_model, shape.n_layer
    weights = step_bytes(shape, "f32", 0) - KV_ROW_BYTES - 4 * V
    by = DECODE * weights + B * sum(KV_ROW_BYTES * (p + 1) + 4 * V for p in range(PROMPT, PROMPT + DECODE))
    fl = sum(B * (2 * (BLOCK_PARAMS_124M + V * d) + L * 4 * d * (p + 1)) for p in range(PROMPT, PROMPT + DECODE))
    return {"sessions": B, "tokens_per_s": B * DECODE / (ms * 1e-3), "ms_per_112_steps": ms,
            "us_per_step": 1e3 * ms / DECODE, "GB_per_s": by / (ms * 1e-3) / 1e9,
            "TFLOP_per_s": fl / (ms * 1e-3) / 1e12,
            "arith": "3xTF32 tcgen05 projections (vocabulary included), binary32 elsewhere"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quant", choices=["f32", "int8", "f16", "int8_row", "int8_row_act"], default="f32")
    ap.add_argument("--no-extra", action="store_true", help="skip the int8, binary16, long-context and prefill extras")
    ap.add_argument("--prefill-only", action="store_true",
                    help="only the 128-token prefill leg (3 warm-up calls, --steps timed calls); prints its JSON")
    ap.add_argument("--batch-only", type=int, default=0, metavar="B",
                    help="only the batched leg with B sessions (3 warm-up runs, --steps timed runs); prints its JSON")
    ap.add_argument("--decode-steps", type=int, default=112,
                    help="decode positions per bench step (112 = positions 16..127)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    global DECODE
    DECODE = max(1, min(112, args.decode_steps))

    from stream_decode_gb300 import synth
    shape = synth.GPT2_124M
    w = synth.checkpoint(shape, synth.SEED_124M)
    toks = synth.tokens(shape.vocab, PROMPT)

    if args.impl == "reference":
        reference_arm(args, shape, w, toks)
        return

    import torch
    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    if args.prefill_only:
        from stream_decode_gb300 import gpt2 as g
        print(json.dumps(prefill_rate(g, torch, shape, w, reps=max(1, args.steps))), flush=True)
        return
    if args.batch_only:
        from stream_decode_gb300 import gpt2 as g
        print(json.dumps(batched_decode(g, torch, shape, w, args.batch_only, reps=max(1, args.steps))), flush=True)
        return
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        rank_sync = dist.barrier
    else:
        rank_sync = lambda: None
    from stream_decode_gb300 import gpt2 as g

    ms, launches, model, sess, first, clocks = measure_decode(g, torch, shape, w, toks, args.quant, args, rank_sync)
    ms, value = combine_replicas(ms, ws)

    peak, peak_kind = _peaks()
    launch_bytes = sum(step_bytes(shape, args.quant, p) for p in range(PROMPT, PROMPT + DECODE))
    achieved = launch_bytes / (ms * 1e-3) / 1e9
    # which step kernel the model runs, and the committed traffic record of
    # one 112-step launch (positions 16..127) if it was taken on that source
    kkind = model.step_kernel[0]
    traffic = traffic_from_profiles(kernel_hash(kkind), args.quant) if DECODE == 112 else None

    e2e_rate, _ = measure_e2e(g, sess, shape, first, 5)
    e2e_tok_rate, _ = measure_e2e_per_token(g, sess, shape, first, 2)
    sess.close()
    model.close()

    extra = {}
    if rank == 0 and not args.no_extra:
        if args.quant == "f32":
            ms8, _, m8, s8, _, _ = measure_decode(g, torch, shape, w, toks, "int8", args, lambda: None)
            b8 = sum(step_bytes(shape, "int8", p) for p in range(PROMPT, PROMPT + DECODE))
            extra["int8_decode"] = {"tokens_per_s": DECODE / (ms8 * 1e-3), "ms_per_step": ms8,
                                    "GB_per_s": b8 / (ms8 * 1e-3) / 1e9,
                                    "frac_of_peak": b8 / (ms8 * 1e-3) / 1e9 / peak}
            s8.close()
            m8.close()
            ms16, _, m16, s16, _, _ = measure_decode(g, torch, shape, w, toks, "f16", args, lambda: None)
            b16 = sum(step_bytes(shape, "f16", p) for p in range(PROMPT, PROMPT + DECODE))
            extra["f16_decode"] = {"tokens_per_s": DECODE / (ms16 * 1e-3), "ms_per_step": ms16,
                                   "GB_per_s": b16 / (ms16 * 1e-3) / 1e9,
                                   "frac_of_peak": b16 / (ms16 * 1e-3) / 1e9 / peak,
                                   "weights": "block matrices and tied embedding in binary16, rest binary32"}
            s16.close()
            m16.close()
            msr, _, mr, sr, _, _ = measure_decode(g, torch, shape, w, toks, "int8_row", args, lambda: None)
            br = sum(step_bytes(shape, "int8_row", p) for p in range(PROMPT, PROMPT + DECODE))
            extra["int8_row_decode"] = {"tokens_per_s": DECODE / (msr * 1e-3), "ms_per_step": msr,
                                        "GB_per_s": br / (msr * 1e-3) / 1e9,
                                        "frac_of_peak": br / (msr * 1e-3) / 1e9 / peak,
                                        "weights": "int8, one scale per output row; group-64 activation scales"}
            sr.close()
            mr.close()
            msa, _, ma, sa, _, _ = measure_decode(g, torch, shape, w, toks, "int8_row_act", args, lambda: None)
            extra["int8_row_act_decode"] = {"tokens_per_s": DECODE / (msa * 1e-3), "ms_per_step": msa,
                                            "GB_per_s": br / (msa * 1e-3) / 1e9,
                                            "frac_of_peak": br / (msa * 1e-3) / 1e9 / peak,
                                            "weights": "int8, one scale per output row; one scale per "
                                                       "activation vector"}
            sa.close()
            ma.close()
        extra["long_context_f32"] = long_context(g, torch, w)
        extra["batched_f32"] = [batched_decode(g, torch, shape, w, B) for B in (16, 64, 256)]
        extra["prefill_f32"] = prefill_rate(g, torch, shape, w)

    cpu = None
    if rank == 0 and not args.no_extra and args.quant == "f32":
        # the int8 workload's CPU baseline: the oracle's int8 model, same sample
        r8, dt8 = oracle_decode_rate(shape, w, toks, 1, DECODE, 2)
        extra["cpu_baseline_int8"] = {"value": r8, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                      "sample": f"two runs of the workload's {DECODE} int8 greedy decode steps "
                                                f"(positions 16..127) after an untimed 16-token prompt ({dt8:.1f} s)"}
    if rank == 0:
        rate, dt = oracle_decode_rate(shape, w, toks, {"f32": 0, "int8": 1, "f16": 2, "int8_row": 3,
                                                       "int8_row_act": 4}[args.quant],
                                      DECODE, 2)
        cpu = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"two runs of the workload's {DECODE} greedy decode steps (positions 16..127) after an "
                         f"untimed 16-token prompt ({dt:.1f} s of single-threaded C on {cpu_cores()} available "
                         f"host cores)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": args.quant, "data": "synthetic (seeded N(0,0.02) weights, "
                "uniform random prompt tokens)", "config": workload_config(args),
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "traffic": traffic, "kernel": KERNEL_NAMES[kkind],
                             "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                             "algorithmic_bytes_per_launch": launch_bytes},
                "cpu_baseline": cpu,
                "e2e": {"value": ws * e2e_rate, "unit": "tokens/s", "h2d_bytes_per_step": 4 * DECODE,
                        "d2h_bytes_per_step": DECODE * (4 * shape.vocab + 4),
                        "api": f"gpt2_session_run_host, one call per bench step ({DECODE} tokens), pinned host buffers",
                        "per_token_calls": {"value": ws * e2e_tok_rate, "unit": "tokens/s",
                                            "api": "gpt2_session_step_host, one call per token"}},
                "gpu_launches": launches, "clocks": clocks, "extra": extra}
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
