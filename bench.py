"""Benchmark of the packed prefix-tree attention path on one GB300 (or N, one per rank).

One step = the whole hot path over one synthetic batch:
  plan (host C++ planner) -> plan upload -> tree RoPE -> tree attention -> readout/calibration.

Default workload: the Llama-1B-shaped batch -- 8 rows, each a 128-token resident
template -> 512-token document -> 4 question blocks of 48 -> 2 option leaves of
40 (depth 4), 8192 forward tokens, 32 q heads / 8 kv heads, head dim 64, RoPE
theta 500000, 4-6 letters per question, T in {0.7, 1.0, 1.3}.

Printed (rank 0, one JSON line): tokens/s of the whole job, the attention
kernel's TFLOP/s against the measured tensor peak (roofline), an end-to-end
figure through tree_runtime_step_host (inputs from page-locked host memory,
decisions back, every copy inside the timed region) beside the measured
host-to-device link rate, SM clocks sampled during the timed region, RoPE and
readout against HBM (back to back, from a CUDA graph, and one call alone), and
the CPU oracle timed on the host as a baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 2] [--impl reference]
  python bench.py --only attn|rope|readout|layer|model [--workload N] [--steps K] [--warmup W] [--sets S]

--only times one kernel (or the Llama layer, or the whole decision forward) by
itself (CUDA events, rotating input sets) and prints one JSON line for it; it is
also the small, fixed command that profiler captures are taken on.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "packed tree-attention tokens/s & TFLOP/s (8192-tok forward), % of f16 TC peak"
UNIT = "tokens/s"
N_SETS = 4  # rotating input sets: 4 x ~81 MB > 129 MB L2

# DRAM bytes per attention launch from one ncu capture, valid only for the
# kernel source it was taken on (sha256 of csrc/attn.cu, first 16 hex digits).
ATTN_TRAFFIC = {(2, "95cf95238ad36d73"): 53639424, (2, "5196ae79ce41ba40"): 53936896,
                (2, "bf00683af88959fd"): 52984576, (2, "02ab9c012a8bcad5"): 53109760}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return dict(hbm=float(m["hbm_gbs"]), tc=float(m["bf16_tflops_sustained"]),
                    tc_burst=float(m["bf16_tflops"]), src="measured")
    except Exception:
        return dict(hbm=6800.0, tc=1700.0, tc_burst=1900.0, src="fallback")


def _src_hash(name):
    with open(os.path.join(ROOT, "prefix_tree_packed_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ GPU arm

class Batch:
    """One workload resident on the device (N_SETS rotating copies of Q/K/V/O).

    A step goes through ``tree_runtime_step``: the host planner packs the batch, and the plan
    transfer, RoPE, attention and readout run as one chain of kernels on the stream, with the
    plan buffers alternating so that the host plans step s+1 while the GPU runs step s.
    """

    def __init__(self, lib, torch, w: synth.Workload, dev, n_sets=N_SETS, tiling=0, pack_heads=0):
        self.lib, self.torch, self.w, self.dev = lib, torch, w, dev
        kw = dict(leaf1=w.leaf1, leaf2=w.leaf2) if w.leaf1 is not None else {}
        self.kw = kw
        self.spec = lib.Spec.from_forest(w.forest, max_fwd=w.max_fwd, tiling=tiling, pack_heads=pack_heads, **kw)
        self.plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd, tiling=tiling, pack_heads=pack_heads, **kw)
        i = self.plan.info
        self.info = i
        self.rt = lib.Runtime(i.dev_bytes + 4096, max(i.n_chunks, 1))
        # a plan on the device for the single-kernel measurements
        self.pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
        self.plan.upload(self.pdev, i.dev_bytes, torch.cuda.current_stream())
        q, k, v = synth.draw_qkv(i.n_fwd, i.n_tot, w.hq, w.hkv, w.d, w.seed)
        self.host = dict(q=q, k=k, v=v)
        self.sets = []
        for s in range(n_sets):
            self.sets.append(dict(q=torch.from_numpy(q).to(dev), k=torch.from_numpy(k).to(dev),
                                  v=torch.from_numpy(v).to(dev),
                                  o=torch.empty((i.n_fwd, w.hq, w.d), dtype=torch.float16, device=dev)))
        self.tab = torch.from_numpy(lib.rope_table(i.max_pos, w.d, w.theta)).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.nq = i.n_questions
        self.logits = self.nl = self.T = self.p_cal = self.choice = None
        if self.nq:
            stride = w.letter_stride
            logits = synth.draw_logits(i.n_slots, stride, w.logit_sigma, w.seed)
            self.host.update(logits=logits, n=w.n_letters, T=w.temperature)
            self.logits = torch.from_numpy(logits).to(dev)
            self.nl = torch.from_numpy(w.n_letters).to(dev)
            self.T = torch.from_numpy(w.temperature).to(dev)
            self.p_cal = torch.empty((self.nq, stride), device=dev)
            self.choice = torch.empty(self.nq, dtype=torch.int32, device=dev)
        self.chunks = [self.plan.chunk(c) for c in range(i.n_chunks)]
        # per input set and chunk: the chunk's query / output rows (views made once)
        self.views = [[(b["q"][ci.q0 - i.n_res: ci.q1 - i.n_res], b["o"][ci.q0 - i.n_res: ci.q1 - i.n_res])
                       for ci in self.chunks] for b in self.sets]

    def step(self, s, stream, ev=None, bufs=None):
        """Enqueue one whole-path step on `stream` using input set s (or `bufs`).

        ev: optional pair of CUDA events, recorded around the step's attention launches.
        """
        w, i = self.w, self.info
        b = bufs if bufs is not None else self.sets[s]
        self.rt.step(self.spec, b["q"], b["k"], b["v"], b["o"], self.tab, i.max_pos, w.hq, w.hkv, w.d,
                     logits=b.get("logits", self.logits), stride=w.letter_stride, n_letters=b.get("n", self.nl),
                     temperature=b.get("T", self.T), p_cal=self.p_cal, choice=self.choice, status=self.status,
                     stream=stream, attn_events=ev)

    def launches_per_step(self):
        # plan transfer, RoPE and attention per chunk, readout
        return 1 + 2 * len(self.chunks) + (1 if self.nq else 0)


def measure_rope(lib, torch, B, stream, reps=40, warmup=None, keys_only=False, timing_forms=False):
    """tree_rope alone over the rotating input sets (Q and K, or K only): algorithmic GB/s."""
    w, i = B.w, B.info
    n_sets = len(B.sets)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def run(s, st=None):
        for c in range(len(B.chunks)):
            lib.tree_rope(B.plan, B.pdev, c, None if keys_only else B.views[s][c][0], B.sets[s]["k"], w.hq, w.hkv,
                          w.d, B.tab, i.max_pos, stream if st is None else st)
    for s in range(n_sets if warmup is None else warmup):
        run(s % n_sets)
    ev[0].record(stream)
    for r in range(reps):
        run(r % n_sets)
    ev[1].record(stream)
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / reps
    # read + write of every forward row rotated, plus its position
    heads = w.hkv if keys_only else w.hq + w.hkv
    nbytes = 2 * i.n_fwd * heads * w.d * 2 + 4 * i.n_fwd
    if not timing_forms:
        return ms, nbytes
    fns = [lambda st, x=x: run(x, st) for x in range(n_sets)]
    return ms, nbytes, graph_ms(torch, fns, reps), single_call_us(torch, fns[0], stream)


def measure_readout(lib, torch, dev, stream, reps=64, n_sets=None, warmup=None, n_questions=65536, timing_forms=False):
    """readout_decide on n_questions (2-10 letters each) over rotating buffer sets: algorithmic GB/s.

    n_sets None: enough sets that their buffers span three times the L2 cache (at least 2)."""
    b = synth.draw_readout_batch(n_questions)
    nq, stride = len(b["r1"]), b["stride"]
    set_bytes = 4 * (b["logits"].size + nq * stride) + 4 * 5 * nq   # logits, p_cal; r1, r2, n, T, choice
    if n_sets is None:
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        n_sets = max(2, -(-3 * l2 // set_bytes))
    sets = []
    for _ in range(n_sets):
        sets.append(dict(logits=torch.from_numpy(b["logits"]).to(dev), r1=torch.from_numpy(b["r1"]).to(dev),
                         r2=torch.from_numpy(b["r2"]).to(dev), n=torch.from_numpy(b["n_letters"]).to(dev),
                         T=torch.from_numpy(b["temperature"]).to(dev),
                         pc=torch.empty((nq, stride), device=dev), ch=torch.empty(nq, dtype=torch.int32, device=dev)))

    def run(x, st=None):
        lib.readout_decide(x["logits"], stride, x["r1"], x["r2"], x["n"], x["T"], nq, x["pc"], None, x["ch"], None,
                           stream if st is None else st)
    for r in range(n_sets if warmup is None else warmup):
        run(sets[r % n_sets])
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    for r in range(reps):
        run(sets[r % n_sets])
    ev[1].record(stream)
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / reps
    n = b["n_letters"].astype(np.int64)
    # logits of both orders, r1/r2/n/T, the zero-padded p_cal row, the choice
    nbytes = int((2 * n * 4).sum() + 16 * nq + 4 * stride * nq + 4 * nq)
    if not timing_forms:
        return ms, nbytes
    fns = [lambda st, x=x: run(x, st) for x in sets]
    return ms, nbytes, graph_ms(torch, fns, reps), single_call_us(torch, fns[0], stream), (n_sets, n_sets * set_bytes)


def graph_ms(torch, fns, reps):
    """Mean time of one call when the calls `fns` (launchers taking a stream, one per rotating input
    set) run back to back from a captured CUDA graph, free of host launch overhead: ms."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in fns:
            f(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for f in fns:
            f(cs)
    g.replay()
    torch.cuda.synchronize()
    n = max(1, reps // len(fns))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    cur = torch.cuda.current_stream()
    ev[0].record(cur)
    for _ in range(n):
        g.replay()
    ev[1].record(cur)
    torch.cuda.synchronize()
    return ev[0].elapsed_time(ev[1]) / (n * len(fns))


def single_call_us(torch, f, stream, n=21):
    """Median device time of one call issued alone (the stream idle before it, launch latency included)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ts = []
    for _ in range(n):
        torch.cuda.synchronize()
        ev[0].record(stream)
        f(stream)
        ev[1].record(stream)
        torch.cuda.synchronize()
        ts.append(ev[0].elapsed_time(ev[1]))
    return statistics.median(ts) * 1e3


def measure_h2d(torch, dev, stream, nbytes, reps=10):
    """Host -> device copy rate from page-locked memory (one cudaMemcpyAsync per rep): GB/s."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        ev[1].record(stream)
    torch.cuda.synchronize()
    return nbytes * reps / (ev[0].elapsed_time(ev[1]) * 1e6)


def measure_attn(lib, torch, B, stream, reps, warmup):
    """tree_attn_fwd alone over the rotating input sets, one work counter per chunk.

    Returns the mean time of one whole forward (all chunks) in ms.
    """
    w = B.w
    n_sets = len(B.sets)
    work = torch.zeros(2 * len(B.chunks), dtype=torch.int32, device=B.dev)

    def fwd(s):
        for c in range(len(B.chunks)):
            qv, ov = B.views[s][c]
            lib.tree_attn_fwd(B.plan, B.pdev, c, qv, B.sets[s]["k"], B.sets[s]["v"], ov, None, w.hq, w.hkv, w.d,
                              status=B.status, stream=stream, work=work[2 * c: 2 * c + 2])
    for r in range(warmup):
        fwd(r % n_sets)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    for r in range(reps):
        fwd(r % n_sets)
    ev[1].record(stream)
    torch.cuda.synchronize()
    assert int(B.status.item()) == 0, "device status word set"
    return ev[0].elapsed_time(ev[1]) / reps


# model width and MLP width of the Llama layer around each workload's attention shape
LAYER_DIMS = {1: (256, 512), 2: (2048, 8192), 3: (4096, 14336), 4: (4096, 14336), 5: (4096, 14336)}


def measure_layer(lib, torch, w, dev, stream, reps, warmup):
    """tree_layer_fwd over the workload's batch with random-init weights, plus each projection GEMM alone.

    Returns a dict: ms per layer, tokens, FLOPs (projections + visible attention pairs) and per-GEMM figures.
    """
    hidden, ffn = LAYER_DIMS[w.number]
    plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd)
    i = plan.info
    n_fwd, n_res = i.n_tot - i.n_res, i.n_res
    wts, x, rk, rv = synth.draw_layer(n_fwd, n_res, hidden, w.hq, w.hkv, w.d, ffn, w.seed)
    td = {k: torch.from_numpy(v).to(dev) for k, v in wts.items()}
    lw = lib.layer_weights(hidden, w.hq, w.hkv, w.d, ffn, td)
    nbytes = lib.layer_workspace_bytes(plan, lw)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
    plan.upload(pdev, i.dev_bytes, stream)
    tab = torch.from_numpy(lib.rope_table(i.max_pos, w.d, w.theta)).to(dev)
    qd, kvd = w.hq * w.d, w.hkv * w.d
    tx = torch.from_numpy(x).to(dev)
    kc = torch.zeros(i.n_tot, kvd, dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    kc[:n_res] = torch.from_numpy(rk).to(dev)
    vc[:n_res] = torch.from_numpy(rv).to(dev)
    y = torch.empty_like(tx)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    work = torch.zeros(2 * i.n_chunks, dtype=torch.int32, device=dev)

    def run():
        lib.layer_fwd(plan, pdev, lw, tx, kc, vc, y, tab, i.max_pos, ws, nbytes, work=work, status=st, stream=stream)

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(stream)
        for _ in range(n):
            fn()
        ev[1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / n

    ms = timed(run, reps)
    assert int(st.item()) == 0, "device status word set"
    m = n_fwd
    gemms = {"qkv": (m, qd + 2 * kvd, hidden), "o": (m, hidden, qd), "gate_up": (m, 2 * ffn, hidden),
             "down": (m, hidden, ffn)}
    gemm_flops = sum(2.0 * a * b * c for a, b, c in gemms.values())
    attn_flops = 4.0 * w.d * w.hq * i.pairs
    # each projection alone, on the workspace buffers (same shapes and epilogues as in the layer)
    a_ = torch.randn(m, max(hidden, ffn, qd), device=dev, dtype=torch.float16)
    out = torch.empty(m, max(hidden, ffn, qd + 2 * kvd), device=dev, dtype=torch.float16)
    per = {}
    for name, (mm, n, k) in gemms.items():
        if name == "gate_up":
            b_, epi, nn, r = td["wgu"], lib.GEMM_SWIGLU, ffn, None
        elif name == "qkv":
            b_, epi, nn, r = td["wqkv"], lib.GEMM_STORE, n, None
        else:
            b_, epi, nn, r = (td["wo"] if name == "o" else td["wd"]), lib.GEMM_RESIDUAL, n, out
        av = a_[:, :k].contiguous()
        t = timed(lambda: lib.gemm(av, b_, out, mm, nn, k, epi, r=r, status=st, stream=stream), reps)
        per[name] = dict(m=mm, n=n, k=k, us=round(t * 1e3, 1), tflops=round(2.0 * mm * n * k / t / 1e9, 1))
    return dict(ms=ms, tokens=n_fwd, hidden=hidden, ffn=ffn, flops=gemm_flops + attn_flops, gemm_flops=gemm_flops,
                attn_flops=attn_flops, gemms=per)


def decision_forest():
    """The page's six-prompt example as one request: template 53 (resident) -> state 120 ->
    3 questions of 24 -> 2 option orders of 18; 4 letters per question."""
    parent, length, resident = [-1, 0], [53, 120], [1, 0]
    leaf1, leaf2 = [], []
    for _ in range(3):
        parent.append(1)
        length.append(24)
        resident.append(0)
        qb = len(parent) - 1
        for o in range(2):
            parent.append(qb)
            length.append(18)
            resident.append(0)
            (leaf1 if o == 0 else leaf2).append(len(parent) - 1)
    return dict(parent=parent, length=length, resident=resident, leaf1=leaf1, leaf2=leaf2,
                n_letters=np.full(3, 4, np.int32), temperature=np.ones(3, np.float32))


def measure_model(lib, torch, dev, stream, spec: dict, d: int, hq: int, hkv: int, theta: float, n_layers: int,
                  reps: int, warmup: int, seed: int, stride: int = 8):
    """tree_model_fwd + readout_decide on one planned batch; random-init weights drawn on the device."""
    hidden, ffn = (2048, 8192) if d == 64 else (4096, 14336)
    plan = lib.Plan(spec["parent"], spec["length"], spec.get("key"), spec["resident"], spec["leaf1"], spec["leaf2"])
    i = plan.info
    n_fwd, n_res = i.n_tot - i.n_res, i.n_res
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def rnd(*shape, scale=1.0, off=0.0):
        return (torch.randn(*shape, generator=g, device=dev, dtype=torch.float32) * scale + off).to(torch.float16)

    qd, kvd = hq * d, hkv * d
    keep, layers, kcs, vcs = [], [], [], []
    for _ in range(n_layers):
        t = {"w_in": rnd(hidden, scale=0.1, off=1.0), "wqkv": rnd(qd + 2 * kvd, hidden, scale=hidden ** -0.5),
             "wo": rnd(hidden, qd, scale=qd ** -0.5), "w_post": rnd(hidden, scale=0.1, off=1.0),
             "wgu": rnd(2 * ffn, hidden, scale=hidden ** -0.5), "wd": rnd(hidden, ffn, scale=ffn ** -0.5)}
        keep.append(t)
        layers.append(lib.layer_weights(hidden, hq, hkv, d, ffn, t))
        kcs.append(rnd(i.n_tot, kvd))
        vcs.append(rnd(i.n_tot, kvd))
    w_final, w_letters = rnd(hidden, scale=0.1, off=1.0), rnd(stride, hidden, scale=hidden ** -0.5)
    x = rnd(n_fwd, hidden)
    pdev = torch.empty(i.dev_bytes, dtype=torch.uint8, device=dev)
    plan.upload(pdev, i.dev_bytes, stream)
    tab = torch.from_numpy(lib.rope_table(i.max_pos, d, theta)).to(dev)
    nb = lib.model_workspace_bytes(plan, layers[0])
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    logits = torch.empty((i.n_slots, stride), device=dev)
    p_cal = torch.empty((i.n_questions, stride), device=dev)
    choice = torch.empty(i.n_questions, dtype=torch.int32, device=dev)
    has_q = spec["leaf1"] is not None and spec["n_letters"] is not None and i.n_questions > 0
    nl = torch.from_numpy(spec["n_letters"]).to(dev) if has_q else None
    temp = torch.from_numpy(spec["temperature"]).to(dev) if has_q else None
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    work = torch.zeros(2 * i.n_chunks, dtype=torch.int32, device=dev)
    base = pdev.data_ptr()

    def run():
        lib.model_fwd(plan, pdev, layers, x, kcs, vcs, tab, i.max_pos, w_final, w_letters, stride, logits, ws, nb,
                      work=work, status=st, stream=stream)
        if has_q:
            lib.readout_decide(logits, stride, base + i.off_r1, base + i.off_r2, nl, temp, i.n_questions, p_cal,
                               None, choice, st, stream)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record(stream)
    for _ in range(reps):
        run()
    ev[1].record(stream)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status word set"
    ms = ev[0].elapsed_time(ev[1]) / reps
    return dict(ms=ms, tokens=n_fwd, resident=n_res, questions=i.n_questions if has_q else 0, hidden=hidden, ffn=ffn)


def run_only(args):
    """One kernel by itself on cuda:0: a JSON line with its time and roofline."""
    import torch
    import prefix_tree_packed_gb300 as lib
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks = _peaks()
    line = {"kernel": args.only, "steps": args.steps, "warmup": args.warmup}
    if args.only == "model":
        w = synth.workload(args.workload)
        spec = dict(parent=w.forest.parent, length=w.forest.length, key=w.forest.key, resident=w.forest.resident,
                    leaf1=w.leaf1,
                    leaf2=w.leaf2, n_letters=w.n_letters, temperature=w.temperature)
        batch = measure_model(lib, torch, dev, stream, spec, w.d, w.hq, w.hkv, w.theta, args.layers, args.steps,
                              args.warmup, seed=w.seed)
        one = measure_model(lib, torch, dev, stream, decision_forest(), w.d, w.hq, w.hkv, w.theta, args.layers,
                            args.steps, args.warmup, seed=w.seed + 1)
        line.update(workload=w.name, layers=args.layers, hidden=batch["hidden"], ffn=batch["ffn"],
                    weights="random init (no trained weights)",
                    batch=dict(ms=round(batch["ms"], 3), forward_tokens=batch["tokens"], questions=batch["questions"],
                               tokens_per_s=round(batch["tokens"] / (batch["ms"] / 1e3), 1),
                               decisions_per_s=round(batch["questions"] / (batch["ms"] / 1e3), 1),
                               readout_slots=int(lib.Plan(spec["parent"], spec["length"], spec["key"],
                                                          spec["resident"]).info.n_slots)),
                    one_request=dict(what="the page's six-prompt example: template 53 resident, state 120, "
                                          "3 questions x (24 + 2 orders x 18), 4 letters",
                                     ms=round(one["ms"], 3), forward_tokens=one["tokens"], questions=one["questions"]))
        line["peak_source"] = peaks["src"]
        print(json.dumps(line), flush=True)
        return
    if args.only == "readout":
        ms, nbytes, gms, one_us, rot = measure_readout(lib, torch, dev, stream, reps=args.steps,
                                                       n_sets=args.sets or None, warmup=args.warmup,
                                                       n_questions=args.questions, timing_forms=True)
        gbs = nbytes / ms / 1e6
        line.update(workload=f"{args.questions:,} questions, 2-10 letters", sets=rot[0],
                    rotating_mb=round(rot[1] / 1e6, 1), us=round(ms * 1e3, 2), bytes=nbytes,
                    achieved=round(gbs, 1), unit="GB/s", peak=peaks["hbm"], frac=round(gbs / peaks["hbm"], 4),
                    graph_us=round(gms * 1e3, 2), graph_frac=round(nbytes / gms / 1e6 / peaks["hbm"], 4),
                    single_call_us=round(one_us, 2))
    else:
        w = synth.workload(args.workload)
        B = Batch(lib, torch, w, dev, n_sets=args.sets or N_SETS, tiling=args.tiling, pack_heads=args.pack)
        B.plan.upload(B.pdev, B.info.dev_bytes, stream)
        line.update(workload=w.name, sets=len(B.sets), tiling=args.tiling, pack_heads=B.info.pack_heads)
        if args.only == "layer":
            r = measure_layer(lib, torch, w, dev, stream, args.steps, args.warmup)
            tf = r["flops"] / (r["ms"] / 1e3) / 1e12
            line.update(us_per_layer=round(r["ms"] * 1e3, 1), tokens=r["tokens"],
                        tokens_per_s=round(r["tokens"] / (r["ms"] / 1e3), 1), hidden=r["hidden"], ffn=r["ffn"],
                        flops=r["flops"], attn_flops=r["attn_flops"], achieved=round(tf, 1), unit="TFLOP/s",
                        peak=peaks["tc"], frac=round(tf / peaks["tc"], 4), gemms=r["gemms"],
                        weights="random init (no trained weights)")
        elif args.only == "rope":
            ms, nbytes, gms, one_us = measure_rope(lib, torch, B, stream, reps=args.steps, warmup=args.warmup,
                                                   keys_only=args.keys_only, timing_forms=True)
            line["keys_only"] = args.keys_only
            gbs = nbytes / ms / 1e6
            line.update(us=round(ms * 1e3, 2), bytes=nbytes, achieved=round(gbs, 1), unit="GB/s",
                        peak=peaks["hbm"], frac=round(gbs / peaks["hbm"], 4), graph_us=round(gms * 1e3, 2),
                        graph_frac=round(nbytes / gms / 1e6 / peaks["hbm"], 4), single_call_us=round(one_us, 2))
        else:
            ms = measure_attn(lib, torch, B, stream, reps=args.steps, warmup=args.warmup)
            i = B.info
            flops = 4.0 * w.d * w.hq * i.pairs
            tf = flops / (ms / 1e3) / 1e12
            # Q and O of every forward row, K and V of every key row, the plan image: each once
            nbytes = 2 * i.n_fwd * w.hq * w.d * 2 + 2 * i.n_tot * w.hkv * w.d * 2 + i.dev_bytes
            gbs = nbytes / ms / 1e6
            ridge = peaks["tc_burst"] * 1e12 / (peaks["hbm"] * 1e9)  # flop per byte where the two roofs meet
            line.update(us_per_forward=round(ms * 1e3, 2), chunks=len(B.chunks), visible_pairs=i.pairs,
                        achieved=round(tf, 2), unit="TFLOP/s", peak=peaks["tc_burst"],
                        frac=round(tf / peaks["tc_burst"], 4), frac_of_sustained=round(tf / peaks["tc"], 4),
                        bytes=nbytes, flop_per_byte=round(flops / nbytes, 1), gbs=round(gbs, 1),
                        hbm_frac=round(gbs / peaks["hbm"], 4),
                        bound="tensor" if flops / nbytes >= ridge else "hbm")
    line["peak_source"] = peaks["src"]
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ every workload

def oracle_sample(w, budget_s: float, seed: int = 0):
    """The oracle (plan, f64 RoPE, per-prompt attention, readout) on workload w: the whole workload,
    repeated while under budget_s, where one pass is a few seconds of host time (attention work up
    to 1e11 pair-head-dims); otherwise on random forward rows, in growing batches until budget_s is
    spent, the rate per row extrapolating to the batch (rows are drawn uniformly)."""
    from oracle import plan as oplan
    p, _ = oplan.plan_forest(w.forest, max_fwd=w.max_fwd)
    if p.pairs * w.hq * w.d <= 1e11:
        t = time.perf_counter()
        n, reps = 0, 0
        while reps == 0 or (time.perf_counter() - t < budget_s and reps < 50):
            n += _oracle_step(w)
            reps += 1
        dt = time.perf_counter() - t
        return {"tokens_per_s": round(n / dt, 2), "rows": int(n), "seconds": round(dt, 2), "cores": _threads(),
                "sample": f"{reps} x the whole workload ({p.n_fwd} forward rows): materialised prompts, dense "
                          f"attention per prompt"}
    rng = np.random.default_rng(seed)
    t = time.perf_counter()
    n, batch = 0, 4
    while True:
        rows = np.sort(rng.choice(p.n_fwd, min(batch, p.n_fwd), replace=False))
        n += _oracle_step(w, rows)
        if time.perf_counter() - t >= budget_s:
            break
        batch = min(2 * batch, 256)
    dt = time.perf_counter() - t
    return {"tokens_per_s": round(n / dt, 2), "rows": int(n), "seconds": round(dt, 2), "cores": _threads(),
            "sample": f"{n} random forward rows of {p.n_fwd}, each attending over its own prompt's keys; the "
                      f"rate per row extrapolates to the batch"}


def measure_configs(lib, torch, dev, stream, peaks, oracle_s: float, numbers=(1, 2, 3, 4, 5)):
    """tree_attn_fwd (and tree_rope) on every workload, each over rotating input sets larger than L2
    where the workload allows, with the oracle's rate on a sample of the same workload beside it."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    ridge = peaks["tc_burst"] * 1e12 / (peaks["hbm"] * 1e9)
    out = {}
    for n in numbers:
        w = synth.workload(n)
        plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd)
        i = plan.info
        set_bytes = 2 * i.n_fwd * w.hq * w.d * 2 + 2 * i.n_tot * w.hkv * w.d * 2
        n_sets = int(min(8, max(2, -(-3 * l2 // set_bytes))))
        B = Batch(lib, torch, w, dev, n_sets=n_sets)
        flops = 4.0 * w.d * w.hq * i.pairs
        # attention bytes: Q and O of every forward row, K and V of every key row, the plan image
        nbytes = set_bytes + i.dev_bytes
        probe = measure_attn(lib, torch, B, stream, reps=2, warmup=3)
        reps = int(min(2000, max(5, 0.25 / max(probe * 1e-3, 1e-6))))
        ms = measure_attn(lib, torch, B, stream, reps=reps, warmup=3)
        tf = flops / (ms / 1e3) / 1e12
        gbs = nbytes / ms / 1e6
        bound = "tensor" if flops / nbytes >= ridge else "hbm"
        r_ms, r_bytes = measure_rope(lib, torch, B, stream, reps=max(20, reps // 4))
        r_gbs = r_bytes / r_ms / 1e6
        e = {"forward_tokens": i.n_fwd, "resident_tokens": i.n_res, "chunks": i.n_chunks,
             "heads": f"{w.hq}/{w.hkv}", "head_dim": w.d, "visible_pairs_per_head": int(i.pairs),
             "rotating_sets": n_sets, "rotating_mb": round(n_sets * set_bytes / 1e6, 1),
             "tree_attn_fwd": {"us_per_forward": round(ms * 1e3, 2), "launches": i.n_chunks, "reps": reps,
                               "tokens_per_s": round(i.n_fwd / (ms / 1e3), 1), "flops": flops,
                               "tflops": round(tf, 2), "frac_of_burst": round(tf / peaks["tc_burst"], 4),
                               "bytes": int(nbytes), "gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm"], 4),
                               "flop_per_byte": round(flops / nbytes, 1), "bound": bound},
             "tree_rope": {"us": round(r_ms * 1e3, 2), "bytes": int(r_bytes), "gbs": round(r_gbs, 1),
                           "hbm_frac": round(r_gbs / peaks["hbm"], 4)}}
        e["roofline_frac"] = e["tree_attn_fwd"]["frac_of_burst" if bound == "tensor" else "hbm_frac"]
        del B
        torch.cuda.empty_cache()
        # gathered key tiles with the q heads of a kv head packed into one MMA tile (tiling 2), timed
        # where they cut the MMA tiles visited: per kv head a packed entry meets each of the R q
        # heads, a gathered one the two halves of its query tile
        R = w.hq // w.hkv
        if R in (2, 4, 8):
            g_plan = lib.Plan.from_forest(w.forest, max_fwd=w.max_fwd, tiling=2, pack_heads=R)
            if g_plan.info.n_entries * 2 < 0.8 * i.n_entries * R:
                Bg = Batch(lib, torch, w, dev, n_sets=n_sets, tiling=2, pack_heads=R)
                gms = measure_attn(lib, torch, Bg, stream, reps=reps, warmup=3)
                gbs_g = (set_bytes + Bg.info.dev_bytes) / gms / 1e6
                tf_g = flops / (gms / 1e3) / 1e12
                e["tree_attn_fwd_gathered"] = {
                    "plan": f"tiling 2, pack_heads {R}", "us_per_forward": round(gms * 1e3, 2),
                    "mma_tile_pairs_per_kv_head": int(g_plan.info.n_entries * 2),
                    "packed_mma_tile_pairs_per_kv_head": int(i.n_entries * R),
                    "tokens_per_s": round(i.n_fwd / (gms / 1e3), 1), "tflops": round(tf_g, 2),
                    "frac_of_burst": round(tf_g / peaks["tc_burst"], 4), "gbs": round(gbs_g, 1),
                    "hbm_frac": round(gbs_g / peaks["hbm"], 4)}
                g_frac = e["tree_attn_fwd_gathered"]["frac_of_burst" if bound == "tensor" else "hbm_frac"]
                if g_frac > e["roofline_frac"]:
                    e["roofline_frac"] = g_frac
                    e["roofline_from"] = "tree_attn_fwd_gathered"
                del Bg
                torch.cuda.empty_cache()
        if oracle_s > 0:
            e["oracle"] = oracle_sample(w, oracle_s, seed=n)
            e["oracle"]["kind"] = "oracle"
        out[w.name] = e
    return out


# ------------------------------------------------------------------ ranks (one GPU each)

def job_batch(n: int, world: int):
    """The whole job's batch: `world` copies of workload n's rows (copy c's letters and temperatures
    drawn with seed n + 101 c), the resident template shared.  Returns the workload of copy 0 and
    the batch as (parent, length, key, resident, leaf1, leaf2, n_letters, temperature)."""
    copies = [synth.workload(n, seed=n + 101 * c) for c in range(world)]
    w0 = copies[0]
    f, nb = w0.forest, w0.forest.n_blocks
    res = f.resident.astype(bool)
    parent = np.concatenate([np.where(f.parent >= 0, f.parent + c * nb, -1) for c in range(world)]).astype(np.int32)
    # keys of copied rows must not make them merge with the other copies; the template's may
    key = np.concatenate([np.where(res | (f.key == 0), f.key, f.key + (np.uint64(c) << np.uint64(40)))
                          for c in range(world)]).astype(np.uint64)
    batch = dict(parent=parent, length=np.tile(f.length, world), key=key, resident=np.tile(f.resident, world))
    if w0.leaf1 is not None:
        batch.update(leaf1=np.concatenate([w0.leaf1 + c * nb for c in range(world)]).astype(np.int32),
                     leaf2=np.concatenate([w0.leaf2 + c * nb for c in range(world)]).astype(np.int32),
                     n_letters=np.concatenate([c.n_letters for c in copies]).astype(np.int32),
                     temperature=np.concatenate([c.temperature for c in copies]).astype(np.float32))
    return w0, batch


def rank_workload(n: int, rank: int, world: int = 1):
    """This rank's share of the job's batch: its rows as split by tree_shard_rows (visible pairs,
    longest first), the resident template kept by every rank.  Rows are independent trees, so no
    data moves between ranks; decisions are gathered on the host afterwards.

    Returns (workload, question_index): the share as a workload (inputs seeded per rank) and the
    job-wide index of each of its questions."""
    import prefix_tree_packed_gb300 as lib
    w0, b = job_batch(n, world)
    spec = lib.Spec(b["parent"], b["length"], b["key"], b["resident"], b.get("leaf1"), b.get("leaf2"),
                    max_fwd=w0.max_fwd)
    block_rank, question_rank, _ = lib.shard_rows(spec, world)
    sel = lib.shard_select(spec, block_rank, question_rank, rank)
    qi = sel["question_index"]
    has_q = "leaf1" in b and len(qi) > 0
    w = synth.Workload(n, w0.name, synth.Forest(sel["parent"], sel["length"], sel["key"], sel["resident"]),
                       hq=w0.hq, hkv=w0.hkv, d=w0.d, theta=w0.theta, seed=n + 101 * rank,
                       leaf1=sel["leaf1"] if has_q else None, leaf2=sel["leaf2"] if has_q else None,
                       n_letters=b["n_letters"][qi] if has_q else None,
                       temperature=b["temperature"][qi] if has_q else None,
                       logit_sigma=w0.logit_sigma, letter_stride=w0.letter_stride, max_fwd=w0.max_fwd)
    return w, qi


def max_over_ranks(dist, values, device):
    """Elementwise max of per-rank timings (the only collective, outside the timed region)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_value(tokens_per_step: int, world: int, steps: int, ms: float) -> float:
    """Whole-job tokens/s when every rank runs tokens_per_step: all ranks' tokens over the slowest
    rank's time."""
    return tokens_per_step * world * steps / (ms / 1e3)


def job_tokens(dist, n_fwd: int, device) -> int:
    """Forward tokens of one job step: the sum over ranks of their shares."""
    import torch
    t = torch.tensor([n_fwd], dtype=torch.int64, device=device)
    if dist is not None:
        dist.all_reduce(t)
    return int(t.item())


def gather_decisions(dist, world: int, q_index, choices):
    """Every rank's (job-wide question index, choice) pairs, assembled on the host: one choice per
    question of the job, or None where a question was not answered."""
    parts = [(np.asarray(q_index), np.asarray(choices))]
    if dist is not None:
        parts = [None] * world
        dist.all_gather_object(parts, (np.asarray(q_index), np.asarray(choices)))
    n = sum(len(q) for q, _ in parts)
    out = np.full(n, -2, np.int32)
    for q, c in parts:
        out[q] = c
    return out


def run_gpu(args):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import prefix_tree_packed_gb300 as lib

    # every rank plans and runs its share of the job's rows: rows are independent, no data exchange
    w, q_index = rank_workload(args.workload, rank, world)
    B = Batch(lib, torch, w, dev)
    i = B.info
    stream = torch.cuda.current_stream()
    for s in range(args.warmup):
        B.step(s % N_SETS, stream)
    # event pairs around each step's attention launches, created before the timed region
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in evs:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize()

    # ---- device-resident timed region (events around every step's attention launches)
    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    h0 = time.perf_counter()
    for s in range(args.steps):
        B.step(s % N_SETS, stream, ev=evs[s])
    host_ms = (time.perf_counter() - h0) * 1e3
    t1.record(stream)
    torch.cuda.synchronize()
    total_ms = t0.elapsed_time(t1)
    clk = clocks.stop()
    attn_ms = [a.elapsed_time(b) for a, b in evs]
    assert int(B.status.item()) == 0, "device status word set"

    # ---- end to end: inputs from pinned host memory, decisions back to the host, through
    # tree_runtime_step_host: the runtime uploads each step's inputs into one of its two
    # device sets on its own copy stream (while the previous step computes) and copies the
    # decisions back on the compute stream; every copy lies inside the timed region.
    h = B.host
    pin = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in h.items()}
    B.rt.attach_io(max_fwd=i.n_fwd, max_tot=i.n_tot, hq=w.hq, hkv=w.hkv, d=w.d,
                   stride=w.letter_stride if B.nq else 0, max_slots=i.n_slots if B.nq else 0,
                   max_questions=B.nq)
    out_pc = torch.empty(tuple(B.p_cal.shape), dtype=torch.float32).pin_memory() if B.nq else None
    out_ch = torch.empty(B.nq, dtype=torch.int32).pin_memory() if B.nq else None
    h2d = sum(v.numel() * v.element_size() for v in pin.values()) + i.dev_bytes
    d2h = (out_pc.numel() * 4 + out_ch.numel() * 4) if B.nq else 0

    def e2e_step():
        B.rt.step_host(B.spec, pin["q"], pin["k"], pin["v"], B.tab, i.max_pos, logits=pin.get("logits"),
                       n_letters=pin.get("n"), temperature=pin.get("T"), p_cal=out_pc, choice=out_ch,
                       status=B.status, stream=stream)

    for s in range(max(2, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    torch.cuda.synchronize()  # the runtime's copy stream starts the first upload after `a`
    for s in range(args.steps):
        e2e_step()
    b.record(stream)  # after the last step's copies back (the step waited for its uploads)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b)
    assert int(B.status.item()) == 0, "device status word set"
    link_gbs = measure_h2d(torch, dev, stream, int(h2d))

    # ---- decisions of the last step gathered on the host (outside the timed regions)
    decisions = gather_decisions(dist, world, q_index, out_ch.numpy() if B.nq else np.zeros(0, np.int32))

    # ---- max over ranks
    total_ms, e2e_ms = max_over_ranks(dist, [total_ms, e2e_ms], dev)
    toks_step = job_tokens(dist, i.n_fwd, dev)
    value = toks_step * args.steps / (total_ms / 1e3)
    e2e_value = toks_step * args.steps / (e2e_ms / 1e3)

    peaks = _peaks()
    flops = 4.0 * w.d * w.hq * i.pairs                      # QK^T + PV on visible pairs only
    attn_launch_ms = statistics.mean(attn_ms) / len(B.chunks)  # the pair spans the step's attention launches
    flops_launch = flops / len(B.chunks)
    achieved = flops_launch / (attn_launch_ms / 1e3) / 1e12
    h_attn = _src_hash("attn.cu")
    traffic = ATTN_TRAFFIC.get((args.workload, h_attn))

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 (f32 accumulate)",
        "data": "synthetic (seeded N(0,1) Q/K/V, N(0,sigma) letter logits)",
        "config": {"workload": w.name, "forward_tokens": i.n_fwd, "resident_tokens": i.n_res,
                   "rows": 8 if args.workload == 2 else None, "q_heads": w.hq, "kv_heads": w.hkv,
                   "head_dim": w.d, "visible_pairs_per_head": i.pairs, "chunks": len(B.chunks),
                   "questions": B.nq, "l2": f"{N_SETS} rotating input sets (> L2)",
                   "step": "tree_runtime_step: plan (host) + plan transfer + rope + attention + readout, one kernel chain",
                   "parallelism": f"dp{world} (the job's {world} x 8 rows split by visible pairs; template on "
                                  f"every rank; decisions gathered on the host)"},
        "tflops_attention": round(achieved, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["tc_burst"], "unit": "TFLOP/s",
                     "frac": round(achieved / peaks["tc_burst"], 4), "traffic": traffic,
                     "kernel": "tree_attn_fwd",
                     "peak_source": f"{peaks['src']} bf16 burst x 1 (f16 = bf16 rate; the launch is timed in a "
                                    f"region of milliseconds at full clock)",
                     "frac_of_sustained": round(achieved / peaks["tc"], 4),
                     "launch_ms": round(attn_launch_ms, 5)},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms / args.steps, 4),
                "call": "tree_runtime_step_host (page-locked host inputs, decisions back to the host)",
                "h2d_link_gbs": round(link_gbs, 1),
                "frac_of_link": round(h2d / (e2e_ms / args.steps * 1e6) / link_gbs, 4)},
        "decisions": {"questions": int(len(decisions)), "answered": int((decisions >= 0).sum()),
                      "gathered_from_ranks": world},
        "gpu_launches": B.launches_per_step() * args.steps,
        "host_enqueue_ms_per_step": round(host_ms / args.steps, 4),
        "clocks": clk,
    }
    rope_ms, rope_bytes, rope_gms, rope_one = measure_rope(lib, torch, B, stream, timing_forms=True)
    ro_ms, ro_bytes, ro_gms, ro_one, ro_rot = measure_readout(lib, torch, dev, stream, timing_forms=True)
    rot_mb = N_SETS * (2 * i.n_fwd * w.hq * w.d * 2 + 2 * i.n_tot * w.hkv * w.d * 2) / 1e6  # Q, O, K, V per set
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    line["kernels"] = {
        "tree_rope": {"bound": "hbm", "us": round(rope_ms * 1e3, 2), "bytes": rope_bytes,
                      "achieved": round(rope_bytes / rope_ms / 1e6, 1), "peak": peaks["hbm"], "unit": "GB/s",
                      "frac": round(rope_bytes / rope_ms / 1e6 / peaks["hbm"], 4),
                      "graph_us": round(rope_gms * 1e3, 2), "single_call_us": round(rope_one, 2),
                      "note": f"{N_SETS} rotating Q/K/V/O sets ({rot_mb:.0f} MB, {rot_mb * 1e6 / l2_bytes:.1f} x L2); "
                              "us: launches back to back on the stream, "
                              "graph_us: the same from a CUDA graph, single_call_us: one launch on an idle stream"},
        "readout_decide_65536q": {"bound": "hbm", "us": round(ro_ms * 1e3, 2), "bytes": ro_bytes,
                                  "achieved": round(ro_bytes / ro_ms / 1e6, 1), "peak": peaks["hbm"],
                                  "unit": "GB/s", "frac": round(ro_bytes / ro_ms / 1e6 / peaks["hbm"], 4),
                                  "graph_us": round(ro_gms * 1e3, 2), "single_call_us": round(ro_one, 2),
                                  "note": f"65,536 questions, 2-10 letters, {ro_rot[0]} rotating buffer sets "
                                          f"({ro_rot[1] / 1e6:.0f} MB, {ro_rot[1] / l2_bytes:.1f} x L2)"},
        "tree_attn_fwd": {"bound": "tensor", "us": round(attn_launch_ms * 1e3, 2), "flops": flops_launch,
                          "achieved": round(achieved, 2), "peak": peaks["tc_burst"], "unit": "TFLOP/s",
                          "frac": round(achieved / peaks["tc_burst"], 4)},
    }
    if rank == 0 and not args.no_configs:
        line["configs"] = measure_configs(lib, torch, dev, stream, peaks,
                                          0.0 if (world > 1 or args.no_cpu_baseline) else args.oracle_budget)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------------ CPU oracle arm

def _oracle_step(w, rows=None):
    """The oracle's whole path over the workload, or over forward rows `rows` of it.

    With `rows`, RoPE is applied to those query rows and to the key rows their
    prompts reach, attention is computed for those rows only, and the readout
    runs on the workload's questions.
    """
    from oracle import attention as oatt
    from oracle import plan as oplan
    from oracle import readout as ordo
    from oracle import rope as orope
    f = w.forest
    kw = dict(leaf1=w.leaf1, leaf2=w.leaf2) if w.leaf1 is not None else {}
    p, qm = oplan.plan_forest(f, max_fwd=w.max_fwd, **kw)
    q, k, v = synth.draw_qkv(p.n_fwd, p.n_tot, w.hq, w.hkv, w.d, w.seed)
    if rows is None:
        qr, kr = orope.apply_plan(p, q, k, w.theta)
        oatt.attend_paths(p, qr, kr, v)
        n_tok = p.n_fwd
    else:
        need = np.zeros(p.n_tot, bool)
        blk = np.searchsorted(p.blk_start, np.arange(p.n_tot), side="right") - 1
        for r in rows:
            b = int(blk[r + p.n_res])
            while b >= 0:
                need[p.blk_start[b]:p.blk_start[b] + p.blk_len[b]] = True
                b = int(p.blk_parent[b])
        fwd = np.nonzero(need[p.n_res:])[0] + p.n_res
        qr = q.copy()
        kr = k.copy()
        qr[rows] = orope.rope_f16(q[rows], p.pos[rows + p.n_res], w.theta)
        kr[fwd] = orope.rope_f16(k[fwd], p.pos[fwd], w.theta)
        oatt.attend_rows(p, qr, kr, v, rows)
        n_tok = len(rows)
    if qm:
        logits = synth.draw_logits(p.n_slots, w.letter_stride, w.logit_sigma, w.seed)
        ordo.decide(logits, qm["r1"], qm["r2"], w.n_letters, w.temperature, w.letter_stride)
    return n_tok


def _threads():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


def cpu_baseline(w, budget_s=15.0):
    t = time.perf_counter()
    n = _oracle_step(w)
    dt = time.perf_counter() - t
    reps = 1
    while time.perf_counter() - t + dt < budget_s and reps < 20:
        n += _oracle_step(w)
        reps += 1
    dt = time.perf_counter() - t
    return {"value": round(n / dt, 2), "unit": UNIT, "cores": _threads(), "kind": "oracle",
            "sample": f"{reps} x the whole workload ({w.name}): host plan, f64 RoPE, per-prompt dense "
                      f"attention, readout; numpy float64, BLAS threads = cores",
            "seconds": round(dt, 2)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = synth.workload(args.workload)
    # each step: the oracle on the first row's worth of forward tokens (one prompt tree)
    from oracle import plan as oplan
    p, _ = oplan.plan_forest(w.forest, max_fwd=w.max_fwd)
    rows = np.arange(min(p.n_fwd, 256))
    for _ in range(args.warmup):
        _oracle_step(w, rows)
    t = time.perf_counter()
    n = 0
    for _ in range(args.steps):
        n += _oracle_step(w, rows)
    dt = time.perf_counter() - t
    value = n / dt
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "sample_rows": int(len(rows))},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": _threads(), "kind": "oracle",
                             "sample": f"per step: plan, f64 RoPE and per-row attention of the first "
                                       f"{len(rows)} forward rows (and the keys of their prompts), readout "
                                       f"({w.name})"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload kernel and oracle figures")
    ap.add_argument("--oracle-budget", type=float, default=4.0, help="host seconds of oracle per workload")
    ap.add_argument("--only", choices=["attn", "rope", "readout", "layer", "model"], default=None)
    ap.add_argument("--layers", type=int, default=16, help="layers for --only model (Llama-1B: 16)")
    ap.add_argument("--sets", type=int, default=0, help="rotating input sets for --only (0: default)")
    ap.add_argument("--questions", type=int, default=65536, help="questions for --only readout")
    ap.add_argument("--keys-only", action="store_true", help="--only rope: rotate the keys alone")
    ap.add_argument("--tiling", type=int, default=0, choices=[0, 1, 2],
                    help="--only attn: key tiles of 128 packed keys (0), by position (1, batch-invariant) or "
                         "gathered (2: the keys some query of the tile sees)")
    ap.add_argument("--pack", type=int, default=0, choices=[0, 1, 2, 4, 8],
                    help="--only attn with --tiling 2: q heads packed into one MMA tile (the q/kv head ratio)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.only and args.impl == "native":
        run_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
