#!/usr/bin/env python3
"""Benchmark of the KDA mixer core on one GB300 (or N independent replicas).

Headline workload: one KDA layer, batched decode of B=256 independent
sequences, 96 heads x 128, FP32 recurrent state (~1.6 GB, larger than L2),
BF16 inputs/outputs. One step = one decode token for the whole batch (one
launch of the fused decode kernel). Beside it, the chunked prefill of one
sequence of T=8192 tokens (same geometry) is timed and reported under
"prefill".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kda|reference]

--impl reference times the FP64 CPU oracle (the only other implementation of
this path) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA tokens/s: decode B=256 (HBM GB/s, % peak); prefill T=8192 (% TC peak)"
H, DH, KCONV, CHUNK = 96, 128, 4, 64
D = H * DH
B_DEC = 256
T_PRE = 8192
# algorithmic bytes per (sequence, head, token) of decode with BF16 I/O:
# state read + write, q,k,v,z,g in, b in, out, conv history read + write
DEC_BYTES_PER_UNIT = 2 * DH * DH * 4 + 5 * DH * 2 + 2 + DH * 2 + 2 * 3 * (KCONV - 1) * DH * 2
# algorithmic FLOPs per (token, head) of chunked prefill at C = 64: 2 (3 d^2 + 5 C d)
PRE_FLOP_PER_TOKEN_HEAD = 2 * (3 * DH * DH + 5 * CHUNK * DH)
# algorithmic bytes per token of prefill with BF16 I/O: q,k,v,z,g,b in, out
PRE_BYTES_PER_TOKEN = (5 * D + H + D) * 2
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode launch at B=256, from
# one ncu capture of the decode kernel built from the sources below, whose SHA-256 (over the
# files in this order) is recorded with it. The line reports null when the sources differ, and
# a CPU test fails until the capture is taken again.
DEC_TRAFFIC_B256 = 1_699_825_664 + 1_612_125_184
DEC_TRAFFIC_SOURCES = ("linear_attention_mixer_gb300/csrc/kda_decode.cu",
                       "linear_attention_mixer_gb300/csrc/kda_decode_common.cuh",
                       "linear_attention_mixer_gb300/csrc/kda_ptx.cuh",
                       "linear_attention_mixer_gb300/csrc/kda_internal.cuh")
DEC_TRAFFIC_SRC_SHA256 = "3f0ea532124da2c4f17d78e6a3791603693172d9a59f7042cc0e85c46bfc1bbc"


def decode_sources_sha256() -> str:
    """SHA-256 of the decode kernel's source files, in DEC_TRAFFIC_SOURCES order."""
    import hashlib
    h = hashlib.sha256()
    for rel in DEC_TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region (read-only)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.f is None:
            return None
        try:
            self.f.flush()
            rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
            os.unlink(self.f.name)
        except Exception:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for nm, val in zip(names, r[5:9]):
                    if val.strip().lower() == "active":
                        reasons.add(nm)
            except Exception:
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ reference arm

def _oracle_decode_sample(n_seq: int, steps: int, seed: int = 2, nthreads: int = 0):
    """Time the FP64 oracle on n_seq sequences x 96 heads for `steps` decode tokens
    (nthreads 0: every host core)."""
    import numpy as np

    import kda_inputs as KI
    from oracle import oracle as O
    O.build()
    p = KI.make_params(H, DH, KCONV, seed)
    S_all = KI.make_state(n_seq, H, DH, seed, std=0.05).astype(np.float64)
    tail_all = KI.make_tail(n_seq, H, DH, KCONV, seed, bf16=True).astype(np.float64)
    tok = KI.make_tokens(n_seq * steps, H, DH, seed, bf16=True)
    oc = O.OracleCfg(H=H, d=DH)
    slots = np.arange(n_seq, dtype=np.int32)
    nt = nthreads or O.max_threads()
    times = []
    for s in range(steps):
        rows = slice(s * n_seq, (s + 1) * n_seq)
        t0 = time.perf_counter()
        O.decode_batch(oc, p, S_all, tail_all, slots, {k: v[rows] for k, v in tok.items()}, nthreads=nt)
        times.append(time.perf_counter() - t0)
    return times, nt


def _oracle_prefill_sample(T: int, n_heads: int, seed: int = 3, nthreads: int = 0):
    import numpy as np

    import kda_inputs as KI
    from oracle import oracle as O
    O.build()
    p = KI.make_params(n_heads, DH, KCONV, seed)
    tok = KI.make_tokens(T, n_heads, DH, seed, bf16=True)
    oc = O.OracleCfg(H=n_heads, d=DH)
    S, tail = O.new_state(oc)
    nt = nthreads or O.max_threads()
    t0 = time.perf_counter()
    O.sequence(oc, p, S, tail, tok, nthreads=nt)
    return time.perf_counter() - t0, nt


def cpu_baseline_decode(target_s: float = 12.0):
    """Bounded sample: n_seq sequences x 96 heads, as many decode steps as fit ~target_s."""
    n_seq = 32
    t1, nt = _oracle_decode_sample(n_seq, 1)
    steps = max(1, min(20, int(target_s / max(t1[0], 1e-3))))
    times, nt = _oracle_decode_sample(n_seq, steps)
    tot = sum(times)
    n1, s1 = 4, 2  # single thread: a smaller sample of the same shape
    t_one, _ = _oracle_decode_sample(n1, s1, nthreads=1)
    return {"value": n_seq * steps / tot, "unit": "tokens/s", "cores": nt, "kind": "oracle",
            "sample": f"FP64 oracle, {steps} decode steps x {n_seq} sequences x {H} heads x {DH} "
                      f"(B=256 workload shape), OpenMP over (sequence, head) units",
            "value_1thread": n1 * s1 / sum(t_one),
            "sample_1thread": f"FP64 oracle on one core, {s1} decode steps x {n1} sequences x {H} heads"}


def cpu_baseline_prefill():
    """Bounded sample: 2048 tokens x 32 heads of the T=8192 prefill, scaled to 96 heads."""
    T, nh = 2048, 32
    t, nt = _oracle_prefill_sample(T, nh)
    T1 = 256
    t1, _ = _oracle_prefill_sample(T1, 1, nthreads=1)
    return {"value": T / (t * H / nh), "unit": "tokens/s", "cores": nt, "kind": "oracle",
            "sample": f"FP64 oracle, sequential per token, {T} tokens x {nh} heads (scaled to {H} heads), "
                      f"OpenMP over heads",
            "value_1thread": T1 / (t1 * H),
            "sample_1thread": f"FP64 oracle on one core, {T1} tokens x 1 head (scaled to {H} heads)"}


def cpu_baseline_gate_proj(T: int = 2048):
    """Bounded sample: the FP64 projection oracle (numpy matmuls) on T tokens at hidden 7168, 96 heads."""
    import os
    import kda_inputs as KI
    from oracle.gate_proj import gate_proj
    inp = KI.make_gate_proj(T, HIDDEN, H, DH, seed=6)
    gate_proj(inp["x"][:64], inp["w_fa"], inp["w_fb"], inp["w_b"])  # warm-up
    t0 = time.perf_counter()
    gate_proj(inp["x"], inp["w_fa"], inp["w_fb"], inp["w_b"])
    t = time.perf_counter() - t0
    try:
        from threadpoolctl import threadpool_info
        cores = max(i.get("num_threads", 1) for i in threadpool_info()) or os.cpu_count()
    except Exception:  # threadpoolctl absent: numpy's BLAS uses every core by default
        cores = os.cpu_count()
    return {"value": T / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"FP64 projection oracle (numpy BLAS matmuls), {T} tokens x hidden {HIDDEN}, {H} heads"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    n_seq = 8
    _oracle_decode_sample(n_seq, max(1, min(args.warmup, 3)))  # warm-up (untimed)
    times, nt = _oracle_decode_sample(n_seq, args.steps)
    tot = sum(times)
    val = n_seq * args.steps / tot
    line = {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "decode B=256, 96 heads x 128, 1 KDA layer (each step: a sample of "
                                   f"{n_seq} sequences)", "batch": B_DEC, "heads": H, "head_dim": DH,
                       "io_dtype": "bf16", "state_dtype": "f64"},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": nt, "kind": "oracle",
                             "sample": f"FP64 oracle, {n_seq} sequences x {H} heads per step"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ CUDA arm

def _fill_state_random(K, cfg, st, n_slots, gen, dev):
    """Fill S ~ N(0, 0.05^2) and the conv history ~ N(0, 1) (BF16) through a device blob."""
    import torch
    sb = H * DH * DH * 4
    tb = 3 * (KCONV - 1) * D * 2
    blob = torch.empty(64 + n_slots * (sb + tb), dtype=torch.uint8, device=dev)
    hdr = K.kda_blob_header()
    hdr.magic, hdr.version = K.KDA_BLOB_MAGIC, K.KDA_BLOB_VERSION
    hdr.num_heads, hdr.head_dim, hdr.conv_kernel, hdr.io_dtype, hdr.n_slots = H, DH, KCONV, cfg.io_dtype, n_slots
    hdr.state_bytes_per_slot, hdr.tail_bytes_per_slot = sb, tb
    blob[:64].copy_(torch.frombuffer(bytearray(bytes(hdr)), dtype=torch.uint8))
    body = blob[64:].view(n_slots, sb + tb)
    for s in range(n_slots):
        body[s, :sb].view(torch.float32).copy_(torch.randn(sb // 4, generator=gen, device=dev) * 0.05)
        body[s, sb:].view(torch.bfloat16).copy_(torch.randn(tb // 2, generator=gen, device=dev).to(torch.bfloat16))
    K.kda_state_restore(st, list(range(n_slots)), blob)
    torch.cuda.synchronize()
    del blob


def _params(K, gen, dev):
    import torch
    conv_w = (torch.randn(3, D, KCONV, generator=gen, device=dev) * 0.5).contiguous()
    dt_bias = torch.randn(D, generator=gen, device=dev) * math.sqrt(0.5)
    A_log = torch.rand(H, generator=gen, device=dev) * math.log(16.0)
    norm_w = 1.0 + torch.randn(DH, generator=gen, device=dev) * math.sqrt(0.1)
    return K.kda_layer_params_from(conv_w, dt_bias, A_log, norm_w)


def _inputs(rows, gen, dev, dtype):
    import torch
    return {n: torch.randn(rows, H if n == "b" else D, generator=gen, device=dev).to(dtype).contiguous()
            for n in ("q", "k", "v", "z", "b", "g")}


def _time_decode(K, args, cfg, params, gen, dev, stream, ws, local):
    """Decode of args.batch sequences: device-resident timing, per-launch events, e2e."""
    import torch
    Bd = args.batch
    st = K.kda_state_alloc(cfg, Bd)
    _fill_state_random(K, cfg, st, Bd, gen, dev)
    ring_n = 16  # 16 distinct input sets (~0.5 GB at B=256), cycled
    ring = [_inputs(Bd, gen, dev, torch.bfloat16) for _ in range(ring_n)]
    slots = torch.arange(Bd, dtype=torch.int32, device=dev)
    out = torch.empty(Bd, D, dtype=torch.bfloat16, device=dev)

    def dec_step(i):
        x = ring[i % ring_n]
        K.kda_decode_token(cfg, params, st, slots, x["q"], x["k"], x["v"], x["z"], x["b"], x["g"], out, stream)

    for i in range(32):  # the states are further filled by random decode steps (untimed)
        dec_step(i)
    for i in range(args.warmup):
        dec_step(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            dec_step(i)
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    _barrier(ws)
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    assert K.kda_state_poll_error(st) == 0

    # e2e through the public API: pinned host inputs copied in, result copied out, every step
    e2e_steps = min(args.steps, 100)
    host = [{n: t.cpu().pin_memory() for n, t in ring[j].items()} for j in range(4)]
    dbuf = {n: torch.empty_like(t) for n, t in ring[0].items()}
    hout = torch.empty(Bd, D, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host[0].values())
    d2h = hout.numel() * hout.element_size()

    def e2e_step(i):
        hx = host[i % 4]
        for n in dbuf:
            dbuf[n].copy_(hx[n], non_blocking=True)
        K.kda_decode_token(cfg, params, st, slots, dbuf["q"], dbuf["k"], dbuf["v"], dbuf["z"], dbuf["b"],
                           dbuf["g"], out, stream)
        hout.copy_(out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    _barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = e0.elapsed_time(e1)

    # the same steps pipelined the way a serving loop runs them: step i+1's inputs are copied in
    # (copy stream) and step i-1's output copied out (output stream) while step i's kernel runs;
    # inputs and outputs are double-buffered and ordered by events. Every copy is inside the
    # timed region.
    cs, ds = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    dbufs = [{n: torch.empty_like(t) for n, t in ring[0].items()} for _ in range(2)]
    outs = [torch.empty(Bd, D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    houts = [torch.empty(Bd, D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]    # slot's inputs have landed
    ev_used = [torch.cuda.Event() for _ in range(2)]  # slot's kernel is done (inputs free, output ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]   # slot's output has reached the host

    def piped_step(i):
        j = i & 1
        with torch.cuda.stream(cs):
            if i >= 2:
                cs.wait_event(ev_used[j])
            hx = host[i % 4]
            for n, t in dbufs[j].items():
                t.copy_(hx[n], non_blocking=True)
            ev_in[j].record(cs)
        stream.wait_event(ev_in[j])
        if i >= 2:
            stream.wait_event(ev_out[j])
        x = dbufs[j]
        K.kda_decode_token(cfg, params, st, slots, x["q"], x["k"], x["v"], x["z"], x["b"], x["g"], outs[j], stream)
        ev_used[j].record(stream)
        with torch.cuda.stream(ds):
            ds.wait_event(ev_used[j])
            houts[j].copy_(outs[j], non_blocking=True)
            ev_out[j].record(ds)

    for i in range(4):
        piped_step(i)
    torch.cuda.synchronize()
    _barrier(ws)
    e0.record(stream)
    cs.wait_event(e0)
    for i in range(e2e_steps):
        piped_step(i)
    for j in range(2):
        stream.wait_event(ev_out[j])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    assert K.kda_state_poll_error(st) == 0
    K.kda_state_free(st)
    del ring, host, dbuf, dbufs, outs, houts
    torch.cuda.empty_cache()
    return {"total_ms": total_ms, "launch_ms": launch_ms, "clocks": clk.summary(), "e2e_ms": e2e_ms,
            "e2e_serial_ms": e2e_serial_ms, "e2e_steps": e2e_steps, "h2d": h2d, "d2h": d2h}


def _time_decode_b1(K, cfg, params, gen, dev, stream):
    """Batch-1 decode latency with the L2 flushed between steps."""
    import torch
    st1 = K.kda_state_alloc(cfg, 1)
    _fill_state_random(K, cfg, st1, 1, gen, dev)
    x1 = [_inputs(1, gen, dev, torch.bfloat16) for _ in range(8)]
    s1 = torch.zeros(1, dtype=torch.int32, device=dev)
    o1 = torch.empty(1, D, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # 256 MB > L2

    def b1_step(i):
        x = x1[i % 8]
        K.kda_decode_token(cfg, params, st1, s1, x["q"], x["k"], x["v"], x["z"], x["b"], x["g"], o1, stream)

    for i in range(10):
        b1_step(i)
    b1_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(200)]
    for i in range(200):
        flush.fill_(i & 0xFF)  # evict the 6.3 MB state from L2 between steps
        b1_ev[i][0].record(stream)
        b1_step(i)
        b1_ev[i][1].record(stream)
    torch.cuda.synchronize()
    b1_us = 1e3 * statistics.median(a.elapsed_time(b) for a, b in b1_ev)
    # host time of one kda_decode_token call (CPU clock, no synchronisation): the C entry point
    # called through ctypes with its arguments built once, so the figure is the library's own
    # host path (checks, launch) plus one ctypes call
    import ctypes
    x = x1[0]
    args_c = (ctypes.byref(cfg), ctypes.byref(params), st1, ctypes.c_void_p(s1.data_ptr()), 1,
              *(ctypes.c_void_p(x[n].data_ptr()) for n in ("q", "k", "v", "z", "b", "g")),
              ctypes.c_void_p(o1.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    fn = K.lib().kda_decode_token
    host_us = []
    for rep in range(5):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(100):
            rc = fn(*args_c)
        host_us.append((time.perf_counter() - t0) / 100 * 1e6)
        assert rc == 0
    torch.cuda.synchronize()
    K.kda_state_free(st1)
    del flush
    return b1_us, statistics.median(host_us)


def _time_decode_multi(K, cfg, params, gen, dev, stream, Bd, n, reps=50):
    """kda_decode_tokens: n tokens for each of Bd sequences per call (one pass over the
    states). Returns ms per call (median of per-call events; inputs cycle over a ring and
    the 1.6 GB of state is larger than L2)."""
    import torch
    st = K.kda_state_alloc(cfg, Bd)
    _fill_state_random(K, cfg, st, Bd, gen, dev)
    ring = [_inputs(Bd * n, gen, dev, torch.bfloat16) for _ in range(4)]
    slots = torch.arange(Bd, dtype=torch.int32, device=dev)
    out = torch.empty(Bd * n, D, dtype=torch.bfloat16, device=dev)

    def call(i):
        x = ring[i % 4]
        K.kda_decode_tokens(cfg, params, st, slots, n, x["q"], x["k"], x["v"], x["z"], x["b"], x["g"], out, stream)

    for i in range(5):
        call(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        ev[i][0].record(stream)
        call(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    assert K.kda_state_poll_error(st) == 0
    K.kda_state_free(st)
    del ring, out
    torch.cuda.empty_cache()
    return ms


def _time_prefill(K, args, cfg, params, gen, dev, stream):
    import torch
    Tp = args.prefill_tokens
    pst = K.kda_state_alloc(cfg, 1)
    px = _inputs(Tp, gen, dev, torch.bfloat16)
    pout = torch.empty(Tp, D, dtype=torch.bfloat16, device=dev)
    pslots = torch.zeros(1, dtype=torch.int32, device=dev)
    cu_h = [0, Tp]
    cu = torch.tensor(cu_h, dtype=torch.int32, device=dev)

    def pre_call():
        K.kda_prefill(cfg, params, pst, pslots, cu, cu_h, px["q"], px["k"], px["v"], px["z"], px["b"], px["g"],
                      pout, stream)

    for _ in range(3):
        K.kda_state_reset(pst, [0], stream)
        pre_call()
    torch.cuda.synchronize()
    reps = args.prefill_reps
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        K.kda_state_reset(pst, [0], stream)
        pev[i][0].record(stream)
        pre_call()
        pev[i][1].record(stream)
    torch.cuda.synchronize()
    pre_ms = statistics.median(a.elapsed_time(b) for a, b in pev)
    assert K.kda_state_poll_error(pst) == 0
    K.kda_state_free(pst)
    del px
    torch.cuda.empty_cache()
    return pre_ms


HIDDEN = 7168  # Kimi K3 hidden width (the input side of the gate/beta projections)


def _time_gate_proj(K, args, gen, dev, stream, reps=20):
    """kda_gate_proj on T = prefill-length tokens at hidden 7168, 96 heads; L2 flushed
    (256 MB written) before every timed call, so each call reads x and the weights from HBM."""
    import torch
    T = args.prefill_tokens
    bf = torch.bfloat16
    gcfg = K.kda_config(H, DH, K.KDA_BF16)
    x = torch.randn(T, HIDDEN, generator=gen, device=dev).to(bf)
    fa = (torch.randn(DH, HIDDEN, generator=gen, device=dev) * HIDDEN ** -0.5).to(bf)
    fb = (torch.randn(D, DH, generator=gen, device=dev) * DH ** -0.5).to(bf)
    bp = (torch.randn(H, HIDDEN, generator=gen, device=dev) * HIDDEN ** -0.5).to(bf)
    z = torch.empty(T, D, dtype=bf, device=dev)
    b = torch.empty(T, H, dtype=bf, device=dev)
    ws = torch.empty(K.kda_gate_proj_workspace_bytes(gcfg, HIDDEN, T), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        K.kda_gate_proj(gcfg, x, fa, fb, bp, z, b, ws, stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        K.kda_gate_proj(gcfg, x, fa, fb, bp, z, b, ws, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(c) for a, c in ev)
    assert int(ws[:4].view(torch.int32).item()) == 0
    flop = 2 * T * (HIDDEN * (DH + H) + DH * D)
    nbytes = 2 * (T * HIDDEN + T * D + T * H + (DH + H) * HIDDEN + D * DH)
    peaks = _peaks()
    src = "of measured" if peaks["source"] == "measured" else "of fallback"
    tf, gbs = flop / (ms / 1e3) / 1e12, nbytes / (ms / 1e3) / 1e9
    del x, z, ws, flush
    torch.cuda.empty_cache()
    return {"workload": f"kda_gate_proj: z = W_fb(W_fa x), b = W_b x for T={T} tokens, hidden {HIDDEN}, "
                        f"96 heads x 128, BF16 in/out, FP32 accumulation (L2 flushed before each call)",
            "ms": ms, "value": T / (ms / 1e3), "unit": "tokens/s", "reps": reps,
            "gpu_launches_per_call": 2,  # gp_in_kernel, gp_out_kernel (+ a 4-byte memset)
            "roofline_hbm": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": gbs / peaks["hbm_gbs"], "bytes_per_call": nbytes, "peak_note": src},
            "roofline_tensor": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                                "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"], "flop_per_call": flop,
                                "peak_note": src}}


KDA_LAYERS = 69  # KDA layers of the Kimi K3 stack (the header comment's architecture block)


def _time_layer_stack(K, args, cfg, gen, dev, stream, reps=5):
    """Whole KDA layers at decode B=256 (hidden 7168, 96 heads x 128): per layer one product
    with the stacked W_q/W_k/W_v/W_g, the gate/beta projections, the mixer and W_o with the
    residual, all on the library's kernels with synthetic random-init weights. Times one layer
    (per-stage CUDA events, so the mixer's share is known) and the 69-layer stack (as many
    layers as device memory holds, stated). Weights and states (0.9 GB + 1.7 GB per layer) are
    far larger than L2."""
    import torch

    from linear_attention_mixer_gb300.layer import KdaLayerRunner, random_layer_weights
    Bd = args.batch
    runner = KdaLayerRunner(cfg, HIDDEN, Bd, dev)
    slots = torch.arange(Bd, dtype=torch.int32, device=dev)
    per_layer = (4 * D * HIDDEN + DH * HIDDEN + D * DH + H * HIDDEN + HIDDEN * D) * 2 + \
        Bd * (H * DH * DH * 4 + 3 * (KCONV - 1) * D * 2)
    free, _ = torch.cuda.mem_get_info(dev)
    n_layers = int(max(1, min(args.stack_layers, (free - (8 << 30)) // per_layer)))
    layers, states = [], []
    try:
        for _ in range(n_layers):
            layers.append(random_layer_weights(H, DH, HIDDEN, gen, dev))
            states.append(K.kda_state_alloc(cfg, Bd))
        x0 = torch.randn(Bd, HIDDEN, generator=gen, device=dev).to(torch.bfloat16)
        bufs = [torch.empty_like(x0), torch.empty_like(x0)]

        def stack_step():
            x = x0
            for li in range(n_layers):
                y = bufs[li & 1]
                runner.decode(layers[li], states[li], slots, x, y, stream)
                x = y

        # one layer, stage by stage
        lw, st = layers[0], states[0]
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        stage = {"qkvg_proj": [], "gate_proj": [], "mixer": [], "out_proj": [], "layer": []}
        D4 = runner.qkvg.view(4, Bd, D)
        for rep in range(reps + 2):
            ev[0].record(stream)
            K.kda_linear(x0, lw.w_qkvg, D4, runner.ws_lin, ysplit=D, stream=stream)
            ev[1].record(stream)
            K.kda_gate_proj(cfg, x0, lw.w_fa, lw.w_fb, lw.w_b, runner.z, runner.b, runner.ws_gp, stream)
            ev[2].record(stream)
            K.kda_decode_token(cfg, lw.params, st, slots, D4[0], D4[1], D4[2], runner.z, runner.b, D4[3],
                               runner.o, stream)
            ev[3].record(stream)
            K.kda_linear(runner.o, lw.w_o, bufs[0], runner.ws_lin, r=x0, stream=stream)
            ev[4].record(stream)
            torch.cuda.synchronize()
            if rep >= 2:
                for key, a, b in (("qkvg_proj", 0, 1), ("gate_proj", 1, 2), ("mixer", 2, 3), ("out_proj", 3, 4),
                                  ("layer", 0, 4)):
                    stage[key].append(ev[a].elapsed_time(ev[b]))
        med = {k: statistics.median(v) for k, v in stage.items()}
        # the stack
        stack_step()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            stack_step()
        t1.record(stream)
        torch.cuda.synchronize()
        stack_ms = t0.elapsed_time(t1) / reps
        for st_ in states:
            assert K.kda_state_poll_error(st_) == 0
    finally:
        for st_ in states:
            K.kda_state_free(st_)
        del layers
        torch.cuda.empty_cache()
    peaks = _peaks()
    w_qkvg, w_o = 4 * D * HIDDEN * 2, HIDDEN * D * 2
    gbs = lambda nbytes, ms: nbytes / (ms / 1e3) / 1e9
    return {"workload": f"KDA layer decode, B={Bd} sequences, hidden {HIDDEN}, 96 heads x 128, BF16 I/O, FP32 state: "
                        "stacked W_q/W_k/W_v/W_g product, gate/beta projections, mixer, W_o with the residual "
                        "(synthetic random-init weights)",
            "layer_ms": med["layer"], "layer_tokens_per_s": Bd / (med["layer"] / 1e3),
            "stage_ms": {k: med[k] for k in ("qkvg_proj", "gate_proj", "mixer", "out_proj")},
            "mixer_share": med["mixer"] / med["layer"],
            "qkvg_proj_gbs": gbs(w_qkvg + Bd * HIDDEN * 2 + 4 * Bd * D * 2, med["qkvg_proj"]),
            "out_proj_gbs": gbs(w_o + Bd * D * 2 + 2 * Bd * HIDDEN * 2, med["out_proj"]),
            "hbm_peak_gbs": peaks["hbm_gbs"],
            "stack_layers": n_layers, "stack_ms": stack_ms, "stack_tokens_per_s": Bd / (stack_ms / 1e3),
            "stack_note": f"{n_layers} of the model's {KDA_LAYERS} KDA layers chained (each layer's output is the "
                          "next one's input), one decode token for all sequences per step, mean of "
                          f"{reps} steps"}


def _time_gate_prefill(K, args, cfg, params, gen, dev, stream, reps=10):
    """From the hidden state to the mixer output for one sequence of T tokens (hidden 7168, 96
    heads): kda_gate_proj then kda_prefill (z written and read back), against kda_gate_proj_in
    then kda_prefill_gate_fused (z formed inside the prefill). L2 flushed before each call."""
    import torch
    T = args.prefill_tokens
    bf = torch.bfloat16
    x = torch.randn(T, HIDDEN, generator=gen, device=dev).to(bf)
    fa = (torch.randn(DH, HIDDEN, generator=gen, device=dev) * HIDDEN ** -0.5).to(bf)
    fb = (torch.randn(D, DH, generator=gen, device=dev) * DH ** -0.5).to(bf)
    bp = (torch.randn(H, HIDDEN, generator=gen, device=dev) * HIDDEN ** -0.5).to(bf)
    px = _inputs(T, gen, dev, bf)
    z = torch.empty(T, D, dtype=bf, device=dev)
    f = torch.empty(T, DH, dtype=bf, device=dev)
    b = torch.empty(T, H, dtype=bf, device=dev)
    out = torch.empty(T, D, dtype=bf, device=dev)
    ws = torch.empty(K.kda_gate_proj_workspace_bytes(cfg, HIDDEN, T), dtype=torch.uint8, device=dev)
    st = K.kda_state_alloc(cfg, 1)
    slots = torch.zeros(1, dtype=torch.int32, device=dev)
    cu_h = [0, T]
    cu = torch.tensor(cu_h, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def separate():
        K.kda_gate_proj(cfg, x, fa, fb, bp, z, b, ws, stream)
        K.kda_prefill(cfg, params, st, slots, cu, cu_h, px["q"], px["k"], px["v"], z, b, px["g"], out, stream)

    def fused():
        K.kda_gate_proj_in(cfg, x, fa, bp, f, b, ws, stream)
        K.kda_prefill_gate_fused(cfg, params, st, slots, cu, cu_h, px["q"], px["k"], px["v"], f, fb, b, px["g"],
                                 out, stream)

    res = {}
    for name, fn in (("separate", separate), ("fused", fused)):
        for _ in range(3):
            K.kda_state_reset(st, [0], stream)
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i in range(reps):
            K.kda_state_reset(st, [0], stream)
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        res[name] = statistics.median(a.elapsed_time(c) for a, c in ev)
    assert K.kda_state_poll_error(st) == 0 and int(ws[:4].view(torch.int32).item()) == 0
    K.kda_state_free(st)
    del x, px, z, f, out, ws, flush
    torch.cuda.empty_cache()
    return {"workload": f"hidden state -> mixer output, 1 sequence T={T}, hidden {HIDDEN}, 96 heads x 128, BF16 I/O "
                        "(L2 flushed before each call)",
            "separate_ms": res["separate"], "fused_ms": res["fused"],
            "separate_calls": "kda_gate_proj + kda_prefill (z written, 24 KB per token, and read back)",
            "fused_calls": "kda_gate_proj_in + kda_prefill_gate_fused (z = W_fb f formed in the prefill)",
            "fused_vs_separate": res["separate"] / res["fused"]}


def _time_varlen(K, args, cfg, params, gen, dev, stream):
    """Varlen workload: 16 sequences ~U[512, 16384] (seeded lengths), prefill all, snapshot /
    reset / restore sequences 0-7, then 128 batched decode steps; tokens/s of both phases."""
    import numpy as np
    import torch

    import kda_inputs as KI
    c = KI.CONFIGS["varlen"]
    N, steps = c["n_seq"], c["decode_steps"]
    lens = KI.varlen_lengths(N, c["len_lo"], c["len_hi"], c["seed"])
    cu_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu_h[-1])
    x = _inputs(T, gen, dev, torch.bfloat16)
    out = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    st = K.kda_state_alloc(cfg, N)
    slots = torch.arange(N, dtype=torch.int32, device=dev)
    cu = torch.tensor(cu_h, device=dev)
    reps = max(1, min(3, args.prefill_reps))
    times = []
    for r in range(reps + 1):
        K.kda_state_reset(st, list(range(N)), stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        K.kda_prefill(cfg, params, st, slots, cu, cu_h, x["q"], x["k"], x["v"], x["z"], x["b"], x["g"], out, stream)
        b.record(stream)
        torch.cuda.synchronize()
        if r > 0:  # the first call grows the workspace
            times.append(a.elapsed_time(b))
    del x, out
    half = list(range(N // 2))
    blob = torch.empty(K.kda_state_blob_bytes(st, len(half)), dtype=torch.uint8, device=dev)
    K.kda_state_snapshot(st, half, blob, stream)
    K.kda_state_reset(st, half, stream)
    K.kda_state_restore(st, half, blob, stream)
    ring = [_inputs(N, gen, dev, torch.bfloat16) for _ in range(steps)]
    o = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s in range(steps):
        y = ring[s]
        K.kda_decode_token(cfg, params, st, slots, y["q"], y["k"], y["v"], y["z"], y["b"], y["g"], o, stream)
    b.record(stream)
    torch.cuda.synchronize()
    dec_ms = a.elapsed_time(b)
    assert K.kda_state_poll_error(st) == 0
    K.kda_state_free(st)
    del ring, blob
    torch.cuda.empty_cache()
    pre_ms = statistics.median(times)
    return {"workload": f"16 sequences, lengths ~U[512,16384] (seeded), {T} tokens, 96 heads x 128, BF16 I/O; "
                        "prefill all, snapshot/reset/restore 8, then 128 batched decode steps",
            "total_tokens": T, "prefill_ms": pre_ms, "prefill_tokens_per_s": T / (pre_ms / 1e3),
            "decode_ms_per_step": dec_ms / steps, "decode_tokens_per_s": N * steps / (dec_ms / 1e3)}


def _time_photo(K, cfg, params, gen, dev, stream, prefill_ms):
    """Photo take and restore of one sequence slot (96 heads x 128, one layer), in pinned host
    memory and parked in a file, against re-prefilling the T-token prompt it stands for. The
    calls synchronise their stream, so they are timed on the host clock (median)."""
    import shutil

    import torch
    st = K.kda_state_alloc(cfg, 2)
    _fill_state_random(K, cfg, st, 2, gen, dev)
    torch.cuda.synchronize()
    tokens = list(range(4096))
    res = {"photo_bytes": K.kda_state_blob_bytes(st, 1)}
    tmp = tempfile.mkdtemp(prefix="kda_photo_bench_")
    try:
        for mode, d, reps in (("ram", None, 20), ("file", tmp, 5)):
            ps = K.kda_photo_store_create(2, d)
            try:
                pid = K.kda_photo_take(ps, [st], 0, tokens, stream)  # first take allocates
                K.kda_photo_restore(ps, pid, [st], 1, stream)
                tt, tr = [], []
                for _ in range(reps):
                    t0 = time.perf_counter()
                    pid = K.kda_photo_take(ps, [st], 0, tokens, stream)
                    t1 = time.perf_counter()
                    K.kda_photo_restore(ps, pid, [st], 1, stream)
                    t2 = time.perf_counter()
                    tt.append((t1 - t0) * 1e3)
                    tr.append((t2 - t1) * 1e3)
            finally:
                K.kda_photo_store_free(ps)
            res[f"{mode}_take_ms"] = statistics.median(tt)
            res[f"{mode}_restore_ms"] = statistics.median(tr)
            res[f"{mode}_restore_gbs"] = res["photo_bytes"] / (res[f"{mode}_restore_ms"] / 1e3) / 1e9
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
        K.kda_state_free(st)
    res["workload"] = ("kda_photo take/restore of one sequence slot (96 heads x 128, 1 KDA layer, FP32 state + "
                       "BF16 conv history), pinned host memory and a parked file; host clock, median")
    if prefill_ms is not None:
        res["reprefill_ms"] = prefill_ms
        res["reprefill_tokens"] = T_PRE
        res["ram_restore_vs_reprefill"] = prefill_ms / res["ram_restore_ms"]
    return res


def run_kda(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from linear_attention_mixer_gb300 import build as KB
    KB.build()
    import linear_attention_mixer_gb300 as K
    peaks = _peaks()
    src = "of measured" if peaks["source"] == "measured" else "of fallback"
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)
    stream = torch.cuda.current_stream()
    cfg = K.kda_config(H, DH, K.KDA_BF16)
    params = _params(K, gen, dev)
    Bd, Tp = args.batch, args.prefill_tokens

    line = {"metric": METRIC, "value": None, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"decode B={Bd}, 96 heads x 128, 1 KDA layer", "batch": Bd, "heads": H,
                       "head_dim": DH, "io_dtype": "bf16", "state_dtype": "f32",
                       "l2": f"inputs larger than L2 ({Bd * H * DH * DH * 4 / 1e9:.2f} GB of state per step)",
                       "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"}}
    if args.only in ("all", "decode"):
        r = _time_decode(K, args, cfg, params, gen, dev, stream, ws, local)
        total_ms_max = _max_over_ranks(r["total_ms"], ws, dev)
        e2e_ms_max = _max_over_ranks(r["e2e_ms"], ws, dev)
        e2e_serial_max = _max_over_ranks(r["e2e_serial_ms"], ws, dev)
        dec_bytes = DEC_BYTES_PER_UNIT * Bd * H
        achieved = dec_bytes / (r["launch_ms"] / 1e3) / 1e9
        line.update({
            "value": Bd * args.steps * ws / (total_ms_max / 1e3),
            "ms_per_step": total_ms_max / args.steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": (DEC_TRAFFIC_B256 if Bd == B_DEC and decode_sources_sha256() == DEC_TRAFFIC_SRC_SHA256
                                     else None),
                         "kernel": "decode_persistent_kernel<bf16,3>", "bytes_per_launch": dec_bytes,
                         "launch_ms": r["launch_ms"], "peak_note": src},
            "e2e": {"value": Bd * r["e2e_steps"] * ws / (e2e_ms_max / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "steps": r["e2e_steps"],
                    "mode": "copies of step i+1 (in) and i-1 (out) overlap step i's kernel on two copy streams, "
                            "double-buffered, all inside the timed region",
                    "serial_value": Bd * r["e2e_steps"] * ws / (e2e_serial_max / 1e3),
                    "serial_mode": "copy in, kernel, copy out on one stream"},
            "gpu_launches": args.steps,
            "clocks": r["clocks"],
        })
        if args.only == "all":
            b1_us, host_us = _time_decode_b1(K, cfg, params, gen, dev, stream)
            line["decode_b1"] = {"workload": "decode B=1, 96 heads x 128, BF16 I/O, FP32 state "
                                             "(L2 flushed between steps)",
                                 "latency_us": b1_us, "host_us_per_call": host_us,
                                 "host_note": "CPU clock per kda_decode_token call, no synchronisation, "
                                              "100 calls back to back through ctypes, median of 5",
                                 "bytes_per_step": DEC_BYTES_PER_UNIT * H,
                                 "achieved_gbs": DEC_BYTES_PER_UNIT * H / (b1_us / 1e6) / 1e9}
            # speculative-verify style decode: n tokens per sequence per call, one state pass
            line["decode_multi"] = []
            for n in (4, 8):
                mms = _time_decode_multi(K, cfg, params, gen, dev, stream, Bd, n)
                mbytes = Bd * H * (2 * DH * DH * 4 + n * (5 * DH * 2 + 2 + DH * 2) + 2 * 3 * (KCONV - 1) * DH * 2)
                line["decode_multi"].append({
                    "workload": f"kda_decode_tokens, B={Bd} sequences x n={n} tokens per call, 96 heads x 128, "
                                f"BF16 I/O, FP32 state",
                    "n": n, "ms_per_call": mms, "tokens_per_s": Bd * n / (mms / 1e3),
                    "vs_n_single_token_calls": n * line["ms_per_step"] / mms,
                    "achieved_gbs": mbytes / (mms / 1e3) / 1e9, "bytes_per_call": mbytes})
    if args.only == "decode_multi":
        line["decode_multi"] = []
        for n in (4, 8):
            mms = _time_decode_multi(K, cfg, params, gen, dev, stream, Bd, n)
            line["decode_multi"].append({"n": n, "ms_per_call": mms, "tokens_per_s": Bd * n / (mms / 1e3)})
        line["value"] = line["decode_multi"][-1]["tokens_per_s"]
        line["ms_per_step"] = line["decode_multi"][-1]["ms_per_call"]
    if args.only in ("all", "prefill"):
        pre_ms = _time_prefill(K, args, cfg, params, gen, dev, stream)
        pre_flop = PRE_FLOP_PER_TOKEN_HEAD * Tp * H
        pre_bytes = PRE_BYTES_PER_TOKEN * Tp
        pre_tflops = pre_flop / (pre_ms / 1e3) / 1e12
        pre_gbs = pre_bytes / (pre_ms / 1e3) / 1e9
        line["prefill"] = {
            "workload": f"prefill 1 sequence T={Tp}, 96 heads x 128, chunk 64, BF16 I/O",
            "value": Tp / (pre_ms / 1e3), "unit": "tokens/s", "ms": pre_ms, "reps": args.prefill_reps,
            "gpu_launches_per_call": 3,  # chunk table, prep_tc, state_tc
            "roofline_tensor": {"bound": "tensor", "achieved": pre_tflops, "peak": peaks["bf16_tflops"],
                                "unit": "TFLOP/s", "frac": pre_tflops / peaks["bf16_tflops"],
                                "flop_per_call": pre_flop, "peak_note": src},
            "roofline_hbm": {"bound": "hbm", "achieved": pre_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": pre_gbs / peaks["hbm_gbs"], "bytes_per_call": pre_bytes, "peak_note": src}}
        if args.only == "prefill":
            line["value"] = Tp / (pre_ms / 1e3)
            line["ms_per_step"] = pre_ms
            line["gpu_launches"] = 3 * args.prefill_reps
    if args.only in ("all", "gate_proj"):
        line["gate_proj"] = _time_gate_proj(K, args, gen, dev, stream)
        line["gate_prefill"] = _time_gate_prefill(K, args, cfg, params, gen, dev, stream)
        if args.only == "gate_proj":
            line["value"] = line["gate_proj"]["value"]
            line["ms_per_step"] = line["gate_proj"]["ms"]
            line["gpu_launches"] = 2 * line["gate_proj"]["reps"]
    if args.only in ("all", "layer"):
        line["layer"] = _time_layer_stack(K, args, cfg, gen, dev, stream)
        if args.only == "layer":
            line["value"] = line["layer"]["stack_tokens_per_s"]
            line["ms_per_step"] = line["layer"]["stack_ms"]
    if args.only == "all":
        line["varlen"] = _time_varlen(K, args, cfg, params, gen, dev, stream)
        line["photo"] = _time_photo(K, cfg, params, gen, dev, stream,
                                    line["prefill"]["ms"] if Tp == T_PRE else None)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode()
        if "prefill" in line:
            line["prefill"]["cpu_baseline"] = cpu_baseline_prefill()
        if "gate_proj" in line:
            line["gate_proj"]["cpu_baseline"] = cpu_baseline_gate_proj()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _self_launch(n: int, argv) -> int:
    """--gpus N > 1 without a launcher: re-run this script under torch.distributed.run,
    one process per GPU on this node (independent replicas), rendezvous on 127.0.0.1.
    Rank 0 prints the JSON line; the return code is the launcher's."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__)] + list(argv)
    return subprocess.run(cmd, cwd=ROOT).returncode


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--prefill-reps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "decode", "decode_multi", "prefill", "gate_proj", "layer"], default="all",
                    help="time one part only (small profiling runs); the JSON line keeps its keys")
    ap.add_argument("--batch", type=int, default=B_DEC, help="decode batch (profiling runs)")
    ap.add_argument("--prefill-tokens", type=int, default=T_PRE, help="prefill length (profiling runs)")
    ap.add_argument("--stack-layers", type=int, default=KDA_LAYERS,
                    help="KDA layers in the layer-stack leg (profiling runs; the model has 69)")
    args = ap.parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return _self_launch(args.gpus, argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_kda(args)


if __name__ == "__main__":
    sys.exit(main())
