"""Benchmark: decode-step products against a 4B-class Q4_K_M decoder on GB300.

One step = one token through the whole weight stream of a 36-layer dense
decoder (hidden 2560; q 2560->4096, k/v 2560->1024, o 4096->2560, gate/up
2560->9728, down 9728->2560; LM head 2560->151936), Q4_K everywhere except
Q6_K for v_proj and down_proj on even layers and for the LM head, in decode
order (q, k, v share an input; gate, up share an input; each stage waits for
the previous one).  Three ways to run the step through libkq are timed, each
captured in a CUDA graph whose kernels are chained with programmatic
dependent launch:
  launches: one kq_matvec per matrix (253 launches);
  stages:   one launch per stage -- a barrier-free kq_chain_run for q|k|v and
            gate|up, kq_matvec for o, down and the head (145 launches);
  chain:    one kq_chain_run of all 253 products with a grid barrier before
            every stage (one persistent launch per step).
The headline value is the fastest; all are reported.

Prints one JSON line.  `value` is quantized-weight GB/s (stored weight bytes
read per second); tok/s-equivalent = steps per second.  Inputs are synthetic
(seeded), weights resident in HBM before timing; the weight set (2.49 GB) is
far larger than L2, so no flushing is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kq|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
import zlib

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-weight GB/s and equiv. decode tok/s vs 8 TB/s HBM roofline"
WORKLOAD = "4B-class dense decoder, 36 layers + LM head, Q4_K_M mix (Q6_K v/down on even layers and head), M=1, bf16 x"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def max_over_ranks(torch, dist, value, device):
    """The largest of every rank's value, on every rank (the slowest replica
    sets the whole job's time); dist None: one process."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_replica, world, ms):
    """Whole-job throughput: every replica reads its own weights once per step."""
    return bytes_per_replica * world / (ms * 1e-3) / 1e9


def build_model(torch, synth, seed=0, n_stages=None):
    """Weights and per-stage inputs/outputs for one token of the sweep (its
    first n_stages stages only, when given)."""
    stages = synth.dense_layer_sweep()
    if n_stages is not None:
        stages = stages[:n_stages]
    dev = torch.device("cuda")
    mats, xs = [], []
    # every stage's x is a view of one device buffer (xs[0]._base), so a
    # step's inputs arrive with one host-to-device copy
    xbuf = torch.empty(sum(st[0][3] for st in stages), dtype=torch.bfloat16, device=dev)
    off = 0
    for si, st in enumerate(stages):
        K = st[0][3]
        g = synth.rng(seed, 1000 + si)
        xv = xbuf[off:off + K].view(1, K)
        xv.copy_(torch.from_numpy(synth.gen_x(1, K, g, "bf16").view(np.int16)).to(dev).view(torch.bfloat16))
        xs.append(xv)
        off += K
        for (name, qt, N, K_) in st:
            gm = synth.rng(seed, 1000 + si, zlib.crc32(name.encode()) & 0xFFFF)
            kw = {"q6_scale_range": (-32, 31)} if qt == synth.Q6_K else {}
            W = torch.from_numpy(synth.gen_matrix(qt, N, K_, gm, **kw)).to(dev)
            y = torch.empty(N, dtype=torch.float32, device=dev)
            mats.append({"name": name, "type": qt, "N": N, "K": K_, "W": W, "stage": si, "y": y,
                         "bytes": synth.matrix_bytes(qt, N, K_)})
    return stages, mats, xs


def record_step(kq, torch, mats, xs, stream, only_type=None):
    for m in mats:
        if only_type is not None and m["type"] != only_type:
            continue
        kq.kq_matvec(m["type"], m["W"], xs[m["stage"]], kq.KQ_BF16, m["y"], m["N"], m["K"], 1, stream)


def make_chain(kq, mats, xs, only_type=None):
    """The step as one chain: a grid barrier before the first product of every stage."""
    ops, last_stage = [], None
    for m in mats:
        if only_type is not None and m["type"] != only_type:
            continue
        ops.append({"type": m["type"], "x_dtype": kq.KQ_BF16, "W": m["W"], "x": xs[m["stage"]], "y": m["y"],
                    "N": m["N"], "K": m["K"], "wait_previous": int(bool(ops) and m["stage"] != last_stage)})
        last_stage = m["stage"]
    return kq.Chain(ops)


def device_info(torch) -> dict:
    """GPU name, SM count, L2 bytes, CUDA runtime and driver versions, host
    cores (what a measurement was taken on); fields it cannot read are left out."""
    info = {"host_cores": os.cpu_count()}
    try:
        p = torch.cuda.get_device_properties(torch.cuda.current_device())
        info["name"] = p.name
        info["sms"] = p.multi_processor_count
        l2 = getattr(p, "L2_cache_size", None)
        if l2:
            info["l2_bytes"] = int(l2)
        info["cuda"] = torch.version.cuda
    except Exception:
        pass
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=10)
        if out.returncode == 0 and out.stdout.strip():
            info["driver"] = out.stdout.strip().splitlines()[0]
    except Exception:
        pass
    return info


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm the path once outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm = [float(r[0]) for r in self.rows if r and r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if len(r) > 1 and r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            for i, n in enumerate(names):
                if len(r) > 3 + i and r[3 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "interval_ms": 20}


def cpu_baseline(mats_host, seconds=12.0):
    """The oracle (fp64 C, all host cores) on a bounded sample of the step:
    the first layer's matrices in decode order, repeated until ~`seconds` of
    CPU work."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    done_bytes, passes, t0 = 0, 0, time.perf_counter()
    while True:
        for (name, qt, N, K, W, x) in mats_host:
            oracle.matvec(qt, W, N, K, x, threads=threads)
            done_bytes += W.size
        passes += 1
        if time.perf_counter() - t0 > seconds:
            break
    dt = time.perf_counter() - t0
    names = [m[0] for m in mats_host]
    return {"value": done_bytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(names)} matrices of layer 0 ({names[0]}..{names[-1]}) x {passes} passes, "
                      f"{done_bytes / 1e6:.0f} MB, {dt:.1f} s"}


def host_sample(synth, n_mats=7, seed=0):
    """The first layer's matrices (and inputs) on the host, for the CPU legs."""
    out = []
    for si, st in enumerate(synth.dense_layer_sweep()):
        K = st[0][3]
        x = synth.gen_x(1, K, synth.rng(seed, 1000 + si), "bf16")
        for (name, qt, N, K_) in st:
            gm = synth.rng(seed, 1000 + si, zlib.crc32(name.encode()) & 0xFFFF)
            kw = {"q6_scale_range": (-32, 31)} if qt == synth.Q6_K else {}
            out.append((name, qt, N, K_, synth.gen_matrix(qt, N, K_, gm, **kw), x))
            if len(out) >= n_mats:
                return out
    return out


def run_reference(args, rank, world):
    """Reference arm: the oracle itself (plain fp64 C on the host cores)."""
    from gguf_quant_weight_super_gb300 import synth
    if rank != 0:
        return
    sample = host_sample(synth, n_mats=4)
    total_bytes = sum(s[4].size for s in sample)
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    for _ in range(max(0, args.warmup)):
        pass  # the oracle has no state to warm; warm-up steps would only burn CPU time
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for (name, qt, N, K, W, x) in sample:
            oracle.matvec(qt, W, N, K, x, threads=threads)
    dt = time.perf_counter() - t0
    v = total_bytes * args.steps / dt / 1e9
    line = {"metric": METRIC, "value": v, "unit": "GB/s", "impl": "reference", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD + " (bounded sample: first 4 matrices of layer 0 per step)",
                       "l2": "inputs larger than L2 on the GPU arm"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"4 matrices of layer 0, {total_bytes / 1e6:.1f} MB per step"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_single(args):
    """One product of a given shape, `--steps` times (for profiler captures)."""
    import torch
    from gguf_quant_weight_super_gb300 import build, kq, synth
    build.build()
    spec = args.single.split(":")
    if spec[0] == "moe_ffn":  # moe_ffn:<type>:<M>: one MoE layer's router + expert FFN (128 experts top-8)
        return run_single_ffn(args, spec)
    if spec[0] == "dequant":  # dequant:<type>:<N>x<K>:<fp32|bf16>: expansion of a whole matrix
        return run_single_dequant(args, spec)
    if spec[0] == "chain":  # chain:<layers>: the dense sweep's first layers as one chain launch
        return run_single_chain(args, int(spec[1]) if len(spec) > 1 else 1)
    qt = {"Q4_K": synth.Q4_K, "Q5_K": synth.Q5_K, "Q6_K": synth.Q6_K, "IA4": synth.IA4}[spec[0]]
    N, K = (int(v) for v in spec[1].split("x"))
    M = int(spec[2]) if len(spec) > 2 else 1
    xd = spec[3] if len(spec) > 3 else "bf16"
    g = synth.rng(0, qt, N, K)
    W = torch.from_numpy(synth.gen_matrix(qt, N, K, g)).cuda()
    xn = synth.gen_x(M, K, g, xd)
    x = torch.from_numpy(xn.view(np.int16)).cuda().view(torch.bfloat16) if xd == "bf16" else torch.from_numpy(xn).cuda()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for _ in range(args.steps):
        kq.kq_matvec(qt, W, x, kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32, y, N, K, M)
    torch.cuda.synchronize()
    assert kq.kq_device_error() == 0
    print(json.dumps({"single": args.single, "runs": args.steps, "ok": True}))


def run_single_chain(args, layers):
    """The first `layers` layers of the dense sweep (4 dependent stages each)
    as one chain launch, `--steps` times (for profiler captures)."""
    import torch
    from gguf_quant_weight_super_gb300 import kq, synth
    stages, keep, xs = build_model(torch, synth, n_stages=4 * layers)
    chain = make_chain(kq, keep, xs)
    for _ in range(args.steps):
        chain.run()
    torch.cuda.synchronize()
    assert kq.kq_device_error() == 0
    print(json.dumps({"single": args.single, "runs": args.steps, "ok": True,
                      "weight_bytes": int(sum(m["bytes"] for m in keep))}))


def run_single_dequant(args, spec):
    """Dequantize one N x K matrix to fp32 or bf16, `--steps` times."""
    import torch
    from gguf_quant_weight_super_gb300 import kq, synth
    qt = {"Q4_K": synth.Q4_K, "Q5_K": synth.Q5_K, "Q6_K": synth.Q6_K, "IA4": synth.IA4}[spec[1]]
    N, K = (int(v) for v in spec[2].split("x"))
    W = torch.from_numpy(synth.gen_matrix(qt, N, K, synth.rng(0, qt, N, K))).cuda()
    bf = len(spec) > 3 and spec[3] == "bf16"
    out = torch.empty(N * K, dtype=torch.bfloat16 if bf else torch.float32, device="cuda")
    for _ in range(args.steps):
        (kq.kq_dequant_bf16 if bf else kq.kq_dequant)(qt, W, out, N * K)
    torch.cuda.synchronize()
    assert kq.kq_device_error() == 0
    print(json.dumps({"single": args.single, "runs": args.steps, "ok": True}))


def run_single_ffn(args, spec):
    """One MoE layer of the MoE benchmark (router, then the expert FFN's two
    launches), `--steps` times, eagerly (for profiler captures)."""
    import torch
    from gguf_quant_weight_super_gb300 import kq, synth
    qt = {"Q4_K": synth.Q4_K, "IA4": synth.IA4}[spec[1]]
    M = int(spec[2]) if len(spec) > 2 else 1
    E, H, F, SH, top_k = 128, 2816, 704, 2112, 8
    g = synth.rng(2, M)
    mats = [torch.from_numpy(synth.gen_matrix(qt, N, K, g)).cuda()
            for N, K in ((E * F, H), (E * F, H), (E * H, F), (SH, H), (SH, H), (H, SH))]
    w = kq.ffn_weights(qt, qt, E, kq.KQ_ACT_GELU_TANH, F, mats[0], mats[1], mats[2], SH, mats[3], mats[4], mats[5])
    logits = torch.from_numpy(synth.gen_logits(M, E, g)).cuda()
    x = torch.from_numpy(synth.gen_x(M, H, g, "bf16").view(np.int16)).cuda().view(torch.bfloat16)
    ids = torch.empty((M, top_k), dtype=torch.int32, device="cuda")
    gate = torch.empty((M, top_k), dtype=torch.float32, device="cuda")
    y = torch.empty((M, H), dtype=torch.float32, device="cuda")
    ws = kq.moe_ffn_workspace(H, F, SH, M, top_k, E)
    for _ in range(args.steps):
        kq.kq_moe_route(logits, M, E, top_k, ids, gate, None)
        kq.kq_moe_ffn(w, ids, gate, x, kq.KQ_BF16, y, H, M, top_k, ws, ws.numel())
    torch.cuda.synchronize()
    kq.kq_moe_check(ws)
    assert kq.kq_device_error() == 0
    print(json.dumps({"single": args.single, "runs": args.steps, "ok": True}))


def run_timeline(args):
    """Per-stage breakdown of the dense sweep as one chain launch, from the
    timeline library's per-CTA global-timer stamps (one untimed step after
    warm-up; the stamps themselves cost a few store instructions per op)."""
    import torch
    from gguf_quant_weight_super_gb300 import kq, synth
    L = kq.use_timeline_library()
    stages, mats, xs = build_model(torch, synth)
    chain = make_chain(kq, mats, xs)
    stream = torch.cuda.Stream()
    for _ in range(max(3, args.warmup) + 1):
        chain.run(stream)
    torch.cuda.synchronize()
    assert kq.kq_device_error() == 0
    G = torch.cuda.get_device_properties(0).multi_processor_count
    CT, OPS = 160, 512
    buf = np.zeros(CT * OPS * 4, dtype=np.uint64)
    assert L.kq_timeline_read(buf.ctypes.data, buf.nbytes) == 0
    ts = buf.reshape(CT, OPS, 4).astype(np.int64)[:G] / 1e3  # us
    starts = [i for i, m in enumerate(mats) if i == 0 or m["stage"] != mats[i - 1]["stage"]] + [len(mats)]
    rows = []
    for si in range(len(starts) - 1):
        i, j = starts[si], starts[si + 1]
        start, done = ts[:, i, 1], ts[:, j, 3]
        r = {"stage": si, "ops": "+".join(m["name"].split(".")[-1] for m in mats[i:j]),
             "bytes": int(sum(m["bytes"] for m in mats[i:j])),
             "consume_med_us": float(np.median(done - start)),
             "tail_us": float(done.max() - np.median(done))}
        if si > 0:
            r["staging_med_us"] = float(np.median(start - ts[:, i, 0]))
            r["barrier_us"] = float(ts[:, i, 0].min() - ts[:, i, 3].max())
            r["stage_us"] = float(done.max() - ts[:, i, 3].max())  # last arrival before to last arrival after
        rows.append(r)
    total = float(ts[:, len(mats), 3].max() - ts[:, 0, 1].min())
    groups = {}
    for r in rows[1:]:
        groups.setdefault(r["ops"], []).append(r)
    out = {"workload": WORKLOAD + ", one chain launch, per-stage means over the layers (us)", "step_us": total,
           "stages": len(rows)}
    out["by_stage"] = {k: {f: round(float(np.mean([r[f] for r in v])), 3)
                           for f in ("bytes", "barrier_us", "staging_med_us", "consume_med_us", "tail_us", "stage_us")}
                       for k, v in groups.items()}
    print(json.dumps(out), flush=True)


def _timed_graph(torch, fn, stream, steps, warmup):
    g = capture(torch, fn, stream)
    for _ in range(max(3, warmup)):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def dev_matrix(torch, synth, qt, N, K, gen):
    """N x ceil(K/256) blocks generated on the device by the input recipe of
    synth.gen_blocks (uniform code, scale and min bytes; d, dmin =
    fp16(|N(0, 0.002)|); Q6_K scales over the full int8 range), flattened to
    bytes.  For the large benchmark weight sets, which would take minutes to
    draw on the host; a different random stream from the host generator."""
    nbl = N * synth.n_blocks_per_row(K)
    raw = torch.randint(0, 256, (nbl, synth.BLOCK_BYTES[qt]), dtype=torch.uint8, device="cuda", generator=gen)

    def half_bytes():
        h = (torch.randn(nbl, device="cuda", generator=gen) * 0.002).abs().half()
        return h.view(torch.uint8).view(nbl, 2)
    if qt in (synth.Q4_K, synth.Q5_K):
        raw[:, 0:2] = half_bytes()
        raw[:, 2:4] = half_bytes()
    elif qt == synth.Q6_K:
        raw[:, 208:210] = half_bytes()
    else:
        raise ValueError("device generation covers the k-quant formats")
    return raw.view(-1)


def graph_ms(torch, fn, stream, steps, warmup):
    return _timed_graph(torch, fn, stream, steps, warmup)


def dense_case(torch, kq, synth, qt, N, K, M, xd, seed, steps, warmup, stream, span=320 << 20, min_copies=1):
    """One product repeated over enough distinct weight copies that every
    replay reads HBM; returns (weight bytes, ms per product)."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    W0 = dev_matrix(torch, synth, qt, N, K, gen)
    ncopy = max(min_copies, -(-span // W0.numel()))
    Ws = [W0] + [W0.clone() for _ in range(ncopy - 1)]
    x = torch.randn((M, K), device="cuda", generator=gen)
    x = x.to(torch.bfloat16) if xd == "bf16" else x
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    xdt = kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32

    def step():
        for W in Ws:
            kq.kq_matvec(qt, W, x, xdt, y, N, K, M, stream)
    ms = graph_ms(torch, step, stream, steps, warmup) / ncopy
    del Ws
    return synth.matrix_bytes(qt, N, K), ms


def moe_case(torch, kq, synth, M, steps, warmup, stream, rho=0.0, layers=30, seed=2):
    """The routed-MoE decode step of the MoE workload: 30 layers of router +
    expert FFN (128 experts, top-8, gate/up 2816->704, down 704->2816) + a
    shared FFN 2816->2112->2816, Q4_K, bf16 x; weights generated on the
    device.  Returns the step's ms, stored bytes read (distinct routed experts
    + shared FFN) and the experts per layer."""
    qt, E, H, F, SH, top_k = synth.Q4_K, 128, 2816, 704, 2112, 8
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    per = []
    for li in range(layers):
        L = {"Wg": dev_matrix(torch, synth, qt, E * F, H, gen), "Wu": dev_matrix(torch, synth, qt, E * F, H, gen),
             "Wd": dev_matrix(torch, synth, qt, E * H, F, gen), "Sg": dev_matrix(torch, synth, qt, SH, H, gen),
             "Su": dev_matrix(torch, synth, qt, SH, H, gen), "Sd": dev_matrix(torch, synth, qt, H, SH, gen)}
        z = torch.randn((M, E), device="cuda", generator=gen)
        if rho:  # a per-layer component shared by the tokens of the block (correlated routing)
            z = (rho ** 0.5) * torch.randn((1, E), device="cuda", generator=gen) + ((1 - rho) ** 0.5) * z
        L["logits"] = z.contiguous()
        L["ids"] = torch.empty((M, top_k), dtype=torch.int32, device="cuda")
        L["gate"] = torch.empty((M, top_k), dtype=torch.float32, device="cuda")
        L["ffn"] = kq.ffn_weights(qt, qt, E, kq.KQ_ACT_GELU_TANH, F, L["Wg"], L["Wu"], L["Wd"], SH, L["Sg"],
                                  L["Su"], L["Sd"])
        per.append(L)
    x = torch.randn((M, H), device="cuda", generator=gen).to(torch.bfloat16)
    y = torch.empty((M, H), dtype=torch.float32, device="cuda")
    ws = kq.moe_ffn_workspace(H, F, SH, M, top_k, E)

    def step():
        for L in per:
            kq.kq_moe_route(L["logits"], M, E, top_k, L["ids"], L["gate"], None, stream)
            kq.kq_moe_ffn(L["ffn"], L["ids"], L["gate"], x, kq.KQ_BF16, y, H, M, top_k, ws, ws.numel(), stream)
    ms = graph_ms(torch, step, stream, steps, warmup)
    kq.kq_moe_check(ws)
    eb = synth.matrix_bytes(qt, F, H) * 2 + synth.matrix_bytes(qt, H, F)
    sb = synth.matrix_bytes(qt, SH, H) * 2 + synth.matrix_bytes(qt, H, SH)
    nexp = [int(torch.unique(L["ids"]).numel()) for L in per]
    nbytes = sum(n * eb + sb for n in nexp)
    del per
    torch.cuda.empty_cache()
    return ms, nbytes, sum(nexp) / layers


def other_configs(torch, kq, synth, stream, steps, warmup, peak):
    """The benchmark's other configurations, measured in the same run after
    the headline: ms per step and GB/s of stored weight bytes each."""
    out = {}

    def rec(b, ms, **kw):
        r = {"ms": round(ms, 5), "GB/s": round(b / (ms * 1e-3) / 1e9, 1), "frac_of_hbm_peak": round(b / (ms * 1e-3) / 1e9 / peak, 4)}
        r.update(kw)
        return r
    b, ms = dense_case(torch, kq, synth, synth.Q4_K, 4096, 4096, 1, "f32", 0, steps, warmup, stream, span=0,
                       min_copies=64)
    out["single_q4k_4096x4096_f32x"] = rec(b, ms)
    sweep = {}
    for qt, nm in ((synth.Q4_K, "Q4_K"), (synth.Q5_K, "Q5_K"), (synth.Q6_K, "Q6_K")):
        for M in (1, 2, 4, 8):
            b, ms = dense_case(torch, kq, synth, qt, 4096, 14336, M, "bf16", 1, steps, warmup, stream)
            sweep[f"{nm}/M={M}"] = rec(b, ms)
    out["format_sweep_4096x14336_bf16x"] = sweep
    tb, tms = 0, 0.0
    for N, K in ((14336, 4096), (14336, 4096), (4096, 14336)):
        b, ms = dense_case(torch, kq, synth, synth.Q4_K, N, K, 16, "bf16", 3, steps, warmup, stream)
        tb, tms = tb + b, tms + ms
    out["verify_block_m16_gate_up_down"] = rec(tb, tms, tok_s_equiv=round(16e3 / tms, 1))
    # M = 8 with correlated routing: a speculative verify block (about 29
    # distinct experts per layer for 8 tokens)
    for M, rho, tag in ((1, 0.0, "m1"), (8, 0.62, "m8_verify"), (16, 0.0, "m16")):
        ms, b, ne = moe_case(torch, kq, synth, M, min(steps, 10), warmup, stream, rho=rho)
        out[f"moe_30_layers_{tag}"] = rec(b, ms, tok_s_equiv=round(M * 1e3 / ms, 1), experts_per_layer=round(ne, 1))
    return out


def run_workload(args):
    """The other benchmark configurations, one JSON line each (measurements
    behind the design notes; the default run is the dense sweep).  Inputs
    smaller than L2 rotate through enough copies that every step reads HBM."""
    import torch
    from gguf_quant_weight_super_gb300 import build, kq, synth
    build.build()
    kq.lib()
    dev = torch.device("cuda")
    stream = torch.cuda.Stream()
    peak, peak_kind = load_peaks()
    L2_SPAN = 320 << 20  # bytes of distinct weights cycled through per replay

    def bf16(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    def line(name, nbytes, ms, extra):
        gbs = nbytes / (ms * 1e-3) / 1e9
        out = {"workload": name, "metric": METRIC, "value": gbs, "unit": "GB/s", "ms_per_step": ms,
               "weight_bytes_per_step": nbytes, "frac_of_hbm_peak": gbs / peak, "peak": peak,
               "peak_kind": peak_kind, "tok_s_equiv": 1e3 / ms}
        out.update(extra)
        print(json.dumps(out), flush=True)

    def dense(qt, N, K, M, xd, seed, label):
        g = synth.rng(seed, qt, N, K)
        W0 = synth.gen_matrix(qt, N, K, g)
        ncopy = max(1, -(-L2_SPAN // W0.size))
        Ws = [torch.from_numpy(W0).to(dev) for _ in range(ncopy)]
        xn = synth.gen_x(M, K, g, xd)
        x = bf16(xn) if xd == "bf16" else torch.from_numpy(xn).to(dev)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        xdt = kq.KQ_BF16 if xd == "bf16" else kq.KQ_F32

        def step():
            for W in Ws:
                kq.kq_matvec(qt, W, x, xdt, y, N, K, M, stream)
        ms = _timed_graph(torch, step, stream, args.steps, args.warmup) / ncopy
        return W0.size, ms

    wl = args.workload
    if wl == "q4k_4096":
        b, ms = dense(synth.Q4_K, 4096, 4096, 1, "f32", 0, "q4k")
        line("single Q4_K 4096x4096, fp32 x, M=1", b, ms, {})
    elif wl == "format_sweep":
        res = {}
        for qt, nm in ((synth.Q4_K, "Q4_K"), (synth.Q5_K, "Q5_K"), (synth.Q6_K, "Q6_K"), (synth.IA4, "IA4")):
            for M in (1, 2, 4, 8):
                b, ms = dense(qt, 4096, 14336, M, "bf16", 1, nm)
                res[f"{nm}/M={M}"] = {"ms": ms, "GB/s": b / (ms * 1e-3) / 1e9, "bytes": b}
        tot_b = sum(r["bytes"] for r in res.values())
        tot_ms = sum(r["ms"] for r in res.values())
        line("format sweep 4096x14336, Q4_K/Q5_K/Q6_K/IA4, M=1,2,4,8, bf16 x", tot_b, tot_ms, {"cases": res})
    elif wl == "verify16":
        res, tot_b, tot_ms = {}, 0, 0.0
        for nm, N, K in (("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)):
            b, ms = dense(synth.Q4_K, N, K, 16, "bf16", 3, nm)
            res[nm] = {"ms": ms, "GB/s": b / (ms * 1e-3) / 1e9}
            tot_b += b
            tot_ms += ms
        line("verify block M=16, gate/up 4096->14336, down 14336->4096, Q4_K, bf16 x", tot_b, tot_ms,
             {"cases": res, "tok_s_equiv": 16e3 / tot_ms})
    elif wl == "dequant":
        # expansion to fp32 / bf16 (the dequantizing load path): bytes read + written per second
        res = {}
        for qt, nm in ((synth.Q4_K, "Q4_K"), (synth.Q5_K, "Q5_K"), (synth.Q6_K, "Q6_K")):
            N, K = 14336, 4096
            W0 = synth.gen_matrix(qt, N, K, synth.rng(6, qt))
            ncopy = max(2, -(-L2_SPAN // W0.size))
            Ws = [torch.from_numpy(W0).to(dev) for _ in range(ncopy)]
            out32 = torch.empty(N * K, dtype=torch.float32, device=dev)
            out16 = torch.empty(N * K, dtype=torch.bfloat16, device=dev)
            for tag, out, fn, ob in (("fp32", out32, kq.kq_dequant, 4), ("bf16", out16, kq.kq_dequant_bf16, 2)):
                def step(out=out, fn=fn):
                    for W in Ws:
                        fn(qt, W, out, N * K, stream)
                ms = _timed_graph(torch, step, stream, args.steps, args.warmup) / ncopy
                moved = W0.size + N * K * ob
                res[f"{nm}/{tag}"] = {"ms": ms, "GB/s": moved / (ms * 1e-3) / 1e9, "read": W0.size, "written": N * K * ob}
        tot_b = sum(v["read"] + v["written"] for v in res.values())
        tot_ms = sum(v["ms"] for v in res.values())
        line("dequant 14336x4096 to fp32 and bf16, Q4_K/Q5_K/Q6_K (GB/s of bytes read + written)", tot_b, tot_ms,
             {"cases": res})
    elif wl == "moe":
        E, H, F, SH, top_k, layers = 128, 2816, 704, 2112, 8, 30

        def mat(qt, N, K, g):
            # IA4: drawn in MLX's group-affine layout and regrouped on the device (load time, untimed)
            if qt == synth.IA4:
                q, sc, bi = synth.gen_ia4_mlx(N, K, g)
                return kq.ia4_pack(torch.from_numpy(q.view(np.int32)).to(dev),
                                   torch.from_numpy(sc.view(np.int16)).to(dev),
                                   torch.from_numpy(bi.view(np.int16)).to(dev))
            return torch.from_numpy(synth.gen_matrix(qt, N, K, g)).to(dev)

        # M = 8: a verify block's correlated routing; IA4: the group-affine INT4 experts of an MLX checkpoint
        for M, rho, qt in ((1, 0.0, synth.Q4_K), (1, 0.0, synth.IA4), (8, 0.62, synth.Q4_K), (8, 0.62, synth.IA4),
                           (16, 0.0, synth.Q4_K)):
            g = synth.rng(2, M)
            Wg0 = mat(qt, E * F, H, g)
            Wd0 = mat(qt, E * H, F, g)
            per_layer = []
            for li in range(layers):
                gl = synth.rng(2, M, li)
                lay = {"Wg": Wg0.clone(), "Wu": Wg0.clone(), "Wd": Wd0.clone(),
                       "logits": torch.from_numpy(synth.gen_logits(M, E, gl, rho=rho)).to(dev),
                       "ids": torch.empty((M, top_k), dtype=torch.int32, device=dev),
                       "gate": torch.empty((M, top_k), dtype=torch.float32, device=dev),
                       "Sg": mat(qt, SH, H, gl), "Su": mat(qt, SH, H, gl), "Sd": mat(qt, H, SH, gl)}
                per_layer.append(lay)
            del Wg0, Wd0
            x = bf16(synth.gen_x(M, H, g, "bf16"))
            xs = bf16(synth.gen_x(M * top_k, F, g, "bf16"))
            xsh = bf16(synth.gen_x(M, SH, g, "bf16"))
            yg = torch.empty((M, top_k, F), dtype=torch.float32, device=dev)
            yu = torch.empty_like(yg)
            yd = torch.empty((M, H), dtype=torch.float32, device=dev)
            ysg = torch.empty((M, SH), dtype=torch.float32, device=dev)
            ysu = torch.empty_like(ysg)
            ysd = torch.empty((M, H), dtype=torch.float32, device=dev)
            wsg = kq.moe_workspace(F, M, top_k, E)
            wsd = kq.moe_workspace(H, M, top_k, E)
            use_chain = M == 1 and qt != synth.IA4  # chains take the k-quants only
            if use_chain:  # one token: the shared gate|up (same x) as one barrier-free chain launch
                for L in per_layer:
                    L["shared_gu"] = kq.Chain([
                        {"type": qt, "x_dtype": kq.KQ_BF16, "W": L["Sg"], "x": x, "y": ysg, "N": SH, "K": H},
                        {"type": qt, "x_dtype": kq.KQ_BF16, "W": L["Su"], "x": x, "y": ysu, "N": SH, "K": H}])

            def route_all():
                for L in per_layer:
                    kq.kq_moe_route(L["logits"], M, E, top_k, L["ids"], L["gate"], None, stream)

            def step():
                for L in per_layer:
                    kq.kq_moe_route(L["logits"], M, E, top_k, L["ids"], L["gate"], None, stream)
                    kq.kq_moe_matvec(qt, L["Wg"], E, L["ids"], None, x, kq.KQ_BF16, 0, yg, F, H, M, top_k,
                                     wsg, wsg.numel(), stream)
                    kq.kq_moe_matvec(qt, L["Wu"], E, L["ids"], None, x, kq.KQ_BF16, 0, yu, F, H, M, top_k,
                                     wsg, wsg.numel(), stream)
                    kq.kq_moe_matvec(qt, L["Wd"], E, L["ids"], L["gate"], xs, kq.KQ_BF16, 1, yd, H, F, M,
                                     top_k, wsd, wsd.numel(), stream)
                    if use_chain:
                        L["shared_gu"].run(stream)
                    else:
                        kq.kq_matvec(qt, L["Sg"], x, kq.KQ_BF16, ysg, SH, H, M, stream)
                        kq.kq_matvec(qt, L["Su"], x, kq.KQ_BF16, ysu, SH, H, M, stream)
                    kq.kq_matvec(qt, L["Sd"], xsh, kq.KQ_BF16, ysd, H, SH, M, stream)
            # the layer as one expert FFN: router, gate|up + activation, down + combine + shared (3 launches)
            wsf = kq.moe_ffn_workspace(H, F, SH, M, top_k, E)
            yf = torch.empty((M, H), dtype=torch.float32, device=dev)
            for L in per_layer:
                L["ffn"] = kq.ffn_weights(qt, qt, E, kq.KQ_ACT_GELU_TANH, F, L["Wg"], L["Wu"],
                                          L["Wd"], SH, L["Sg"], L["Su"], L["Sd"])

            def step_ffn():
                for L in per_layer:
                    kq.kq_moe_route(L["logits"], M, E, top_k, L["ids"], L["gate"], None, stream)
                    kq.kq_moe_ffn(L["ffn"], L["ids"], L["gate"], x, kq.KQ_BF16, yf, H, M, top_k, wsf, wsf.numel(),
                                  stream)
            ms_sep = _timed_graph(torch, step, stream, args.steps, args.warmup)
            kq.kq_moe_check(wsg)
            kq.kq_moe_check(wsd)
            ms = _timed_graph(torch, step_ffn, stream, args.steps, args.warmup)
            kq.kq_moe_check(wsf)
            route_ms = _timed_graph(torch, route_all, stream, args.steps, args.warmup)
            for L in per_layer:  # distinct experts the router picked (the expert bytes a step reads)
                L["nexp"] = int(torch.unique(L["ids"]).numel())
            eb = synth.matrix_bytes(qt, F, H) * 2 + synth.matrix_bytes(qt, H, F)
            sb = synth.matrix_bytes(qt, SH, H) * 2 + synth.matrix_bytes(qt, H, SH)
            nbytes = sum(L["nexp"] * eb + sb for L in per_layer)
            # the same without the padding of the last block of rows whose K is not a multiple of 256
            ub = lambda N, K: N * K * synth.BLOCK_BYTES[qt] // 256  # noqa: E731
            nbytes_unpadded = sum(L["nexp"] * (2 * ub(F, H) + ub(H, F)) + 2 * ub(SH, H) + ub(H, SH) for L in per_layer)
            line(f"routed MoE decode, 30 layers: router + expert FFN (128 experts top-8, GELU-gated) + shared FFN, "
                 f"{synth.TYPE_NAMES[qt]}, M={M}" + (f", correlated routing (rho {rho})" if rho else ""), nbytes, ms,
                 {"tok_s_equiv": M * 1e3 / ms, "distinct_experts_per_layer": sum(L["nexp"] for L in per_layer) / layers,
                  "weight_bytes_unpadded_per_step": nbytes_unpadded,
                  "launches_per_step": 3 * layers, "router_us_per_layer": route_ms * 1e3 / layers,
                  "separate_products": {"ms_per_step": ms_sep, "GB/s": nbytes / (ms_sep * 1e-3) / 1e9,
                                        "launches_per_step": (6 if M == 1 else 7) * layers}})
            del per_layer
            torch.cuda.empty_cache()
    else:
        raise SystemExit(f"unknown workload {wl}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kq", choices=["kq", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other configurations in the JSON line")
    ap.add_argument("--single", default=None,
                    help="profiling helper: run one product TYPE:NxK[:M[:f32|bf16]] (e.g. Q4_K:19456x2560), one MoE layer moe_ffn:TYPE:M, one expansion dequant:TYPE:NxK:fp32|bf16, or the dense sweep's first layers as a chain chain:LAYERS, --steps times")
    ap.add_argument("--timeline", action="store_true",
                    help="per-stage breakdown of the dense sweep's chain from per-CTA timer stamps (timeline library)")
    ap.add_argument("--workload", default=None, choices=["q4k_4096", "format_sweep", "verify16", "moe", "dequant"],
                    help="time another configuration instead of the dense sweep (one JSON line each)")
    args = ap.parse_args()
    if args.workload:
        run_workload(args)
        return
    if args.single:
        run_single(args)
        return
    if args.timeline:
        run_timeline(args)
        return

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from gguf_quant_weight_super_gb300 import build, kq, synth
    build.build()
    kq.lib()
    torch.manual_seed(0)

    stages, mats, xs = build_model(torch, synth, seed=rank)
    total_bytes = sum(m["bytes"] for m in mats)
    launches_per_step = len(mats)
    stream = torch.cuda.Stream()

    chain = make_chain(kq, mats, xs)
    # the independent products of a stage (q|k|v, gate|up) as one launch each
    stage_runs = []
    for si in range(len(stages)):
        sm = [m for m in mats if m["stage"] == si]
        if len(sm) == 1:
            m = sm[0]
            stage_runs.append(lambda m=m: kq.kq_matvec(m["type"], m["W"], xs[m["stage"]], kq.KQ_BF16, m["y"], m["N"],
                                                        m["K"], 1, stream))
        else:
            ch = make_chain(kq, sm, xs)
            stage_runs.append(lambda ch=ch: ch.run(stream))
    graphs = {"launches": capture(torch, lambda: record_step(kq, torch, mats, xs, stream), stream),
              "stages": capture(torch, lambda: [r() for r in stage_runs], stream),
              "chain": capture(torch, lambda: chain.run(stream), stream)}
    launches = {"launches": launches_per_step, "stages": len(stage_runs), "chain": 1}

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(graph, steps, clk=None):
        for _ in range(max(3, args.warmup)):
            graph.replay()
        barrier()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(steps):
                graph.replay()
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / steps

    variants = {}
    with ClockSampler(local) as clk:
        for name, graph in graphs.items():
            variants[name] = max_over_ranks(torch, dist, timed(graph, args.steps), "cuda")
    assert kq.kq_device_error() == 0, "device error word set"
    best = min(variants, key=variants.get)
    ms = variants[best]
    step_graph = graphs[best]

    # spread of single steps of the best variant (each replay between its own
    # pair of events, after the timed region; the value above is the mean)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for a, b in pairs:
            a.record(stream)
            step_graph.replay()
            b.record(stream)
    torch.cuda.synchronize()
    per = sorted(a.elapsed_time(b) for a, b in pairs)
    pick = lambda q: per[min(len(per) - 1, int(q * len(per)))]  # noqa: E731
    spread = {"p10": pick(0.1), "p50": pick(0.5), "p90": pick(0.9), "n": len(per)}

    # dominant kernel: prog_kernel.  For the chain, one launch is the whole
    # step; for separate launches, the Q4_K products of a step timed alone
    # (same order, same chaining).
    peak, peak_kind = load_peaks()
    if best in ("chain", "stages"):
        q4_bytes, n_q4, q4_ms = total_bytes, launches[best], ms
        rf_kernel = ("prog_kernel (chain: all 253 products of a step, one launch)" if best == "chain" else
                     "prog_kernel (one launch per stage: q|k|v, o, gate|up, down; 145 per step)")
    else:
        q4 = [m for m in mats if m["type"] == synth.Q4_K]
        q4_bytes, n_q4 = sum(m["bytes"] for m in q4), len(q4)
        q4_graph = capture(torch, lambda: record_step(kq, torch, mats, xs, stream, only_type=synth.Q4_K), stream)
        q4_ms = timed(q4_graph, args.steps)
        rf_kernel = "prog_kernel (all Q4_K products of a step, one launch each)"
    achieved = q4_bytes / (q4_ms * 1e-3) / 1e9
    traffic = None
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            tr = json.load(f)
        if tr.get("kernel_build") == kq.build_id("prog_kernel") and best in tr.get("variants", []):
            # DRAM bytes per launch from one ncu capture (ratio to the weight
            # bytes), scaled to the average launch of this variant
            traffic = tr["dram_bytes_ratio"] * q4_bytes / n_q4
    except Exception:
        traffic = None

    # end to end: per step, H2D of the step's inputs from pinned host memory,
    # the step, and D2H of the logits (the step's result)
    xbuf = xs[0]._base  # all stages' x, contiguous
    x_host = xbuf.cpu().pin_memory()
    logits = mats[-1]["y"]
    logits_host = torch.empty_like(logits, device="cpu").pin_memory()
    h2d = x_host.numel() * x_host.element_size()
    d2h = logits.numel() * logits.element_size()

    def e2e_step():
        xbuf.copy_(x_host, non_blocking=True)
        step_graph.replay()
        logits_host.copy_(logits, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
    torch.cuda.synchronize()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(torch, dist, e0.elapsed_time(e1) / args.steps, "cuda")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(host_sample(synth, n_mats=7))
    configs = None
    if not args.no_configs:
        del graphs, step_graph, chain, stage_runs
        torch.cuda.empty_cache()
        configs = other_configs(torch, kq, synth, stream, min(args.steps, 20), args.warmup, load_peaks()[0])

    if rank == 0:
        gbs = job_gbs(total_bytes, world, ms)
        line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": max(3, args.warmup), "ms_per_step": ms, "ms_per_step_spread": spread,
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "u8 codes x bf16 x, int32/fp32 accumulate", "data": "synthetic",
                "tok_s_equiv": world * 1e3 / ms, "roofline_tok_s_equiv": peak * 1e9 / total_bytes,
                "frac_of_hbm_peak": gbs / world / peak,
                "config": {"workload": WORKLOAD, "weight_bytes_per_step": total_bytes, "variant": best,
                           "launches_per_step": launches[best],
                           "graph": "CUDA graph per step (launches: programmatic dependent launch)",
                           "l2": "inputs larger than L2 (2.49 GB of weights per step, read once)",
                           "parallelism": f"replicas x{world}"},
                "variants": {k: {"ms_per_step": v, "GB/s": total_bytes * world / (v * 1e-3) / 1e9,
                                 "launches_per_step": launches[k]} for k, v in variants.items()},
                "roofline": {"bound": "hbm", "kernel": rf_kernel,
                             "achieved": achieved, "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs",
                             "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                             "launches": n_q4, "bytes_per_launch": q4_bytes / n_q4,
                             "avg_launch_us": q4_ms * 1e3 / n_q4},
                "e2e": {"value": total_bytes * world / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
                "gpu_launches": launches[best] * args.steps,
                "clocks": clk.summary(), "device": device_info(torch)}
        if line["clocks"]["sm_mhz"]:  # the step in SM clock cycles at the median clock of the timed region
            line["clocks"]["mcycles_per_step"] = round(ms * line["clocks"]["sm_mhz"] * 1e-3, 4)
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if configs is not None:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
