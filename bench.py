#!/usr/bin/env python3
"""Benchmark of the KDA core (libkda) on GB300.

A step is one chunked KDA prefill of the 4k workload (B=1, T=4096, H=32,
K=V=128, bf16 q/k/v, fp32 g/beta, zero initial state, output + final fp32
state) through the C ABI: kda_chunk_intra then kda_chunk_scan on one stream.
Inputs are resident in HBM when the timed region starts; they (plus the
workspace) exceed the 129 MB L2, so no flush is needed between steps.  The
same line also carries the decode half of the metric: the 256 x 32 decode
step (512 MiB fp32 state pool, 64 consecutive steps), in microseconds.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the fp64 CPU
oracle instead (a bounded sample of the same workload on the host cores).

Multi-GPU (torchrun, one rank per GPU): each rank runs its own copy of the
workload (independent sequences; the KDA core needs no exchange), so the
scaling is weak and there is no collective on the data path; only the
timing barrier and a max-reduction of the times.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import kda_inputs  # noqa: E402

METRIC = "KDA prefill tokens/s (T=4096,H=32,K=V=128) & decode step us; % roofline"
T_4K, H, K, V = 4096, 32, 128, 128
DEC_N, DEC_STEPS = 256, 64
L2_BYTES = 129 * 1024 * 1024
KERNELS_PER_PREFILL = 4   # chunk index, state scan (launched first, running alongside the
                          # prep), main prep, strong-decay prep (exits at once when nothing
                          # is deferred)
KERNELS_PER_DECODE = 1


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--precise", action="store_true", help="fp32 CUDA-core chunk path")
    p.add_argument("--no-gated", action="store_true", help="skip the raw-gate prefill sub-run")
    p.add_argument("--no-conv", action="store_true", help="skip the short-convolution sub-run")
    p.add_argument("--no-varlen", action="store_true", help="skip the varlen_8 prefill sub-run")
    p.add_argument("--no-long", action="store_true",
                   help="skip the long_131k prefill + hand-off decode sub-run")
    p.add_argument("--phases", action="store_true",
                   help="run each step as its two phases (the prep, then the scan after it) "
                        "instead of one forward, and skip the sub-runs that need the whole "
                        "forward: the form a kernel profiler can capture (it serialises "
                        "kernels, and the forward's scan waits for records of a prep that "
                        "runs beside it)")
    a = p.parse_args()
    if a.phases:
        a.no_e2e = a.no_gated = a.no_varlen = a.no_long = True
    return a


# ---- distributed plumbing --------------------------------------------------

def free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_ranks(n, script, argv, env=None, timeout=None):
    """Run `script argv` as n local ranks (one process per GPU) under
    torch.distributed.run on 127.0.0.1; each rank reads RANK / LOCAL_RANK /
    WORLD_SIZE / MASTER_* from its environment.  Returns the launcher's exit
    code; the ranks' stdout (rank 0's JSON line) passes through."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1",
           "--nproc-per-node", str(n), "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()), script, *argv]
    return subprocess.run(cmd, env=env, timeout=timeout).returncode


def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return rank, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device=None):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- peaks, clocks, profiles ----------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


class Clocks:
    """nvidia-smi sampled every 50 ms while the benchmark runs; the samples
    inside a wall-clock window are summarised afterwards."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.t0 = time.time()
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-i", str(gpu_index), "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.p = None

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = []
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append(dict(t=ts + frac, sm=float(parts[2]), smax=float(parts[3]),
                                 power=float(parts[4]) if parts[4] not in ("[N/A]", "N/A") else None,
                                 reasons=parts[5], hw=parts[6], hwt=parts[7], swt=parts[8],
                                 swp=parts[9]))
            except (ValueError, IndexError):
                continue
        self.rows = rows
        os.unlink(self.f.name)
        return rows

    def summary(self, t_start, t_end):
        rows = getattr(self, "rows", [])
        win = [r for r in rows if t_start - 0.06 <= r["t"] <= t_end + 0.06]
        if not win and rows:  # the window was shorter than one sample period
            mid = 0.5 * (t_start + t_end)
            win = sorted(rows, key=lambda r: abs(r["t"] - mid))[:2]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        reasons = set()
        for r in win:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in win),
                "sm_max_mhz": max(r["smax"] for r in win), "reasons": sorted(reasons),
                "samples": len(win),
                "power_w_max": max((r["power"] for r in win if r["power"] is not None), default=None)}


def traffic_from_profiles(kernel_key):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, or
    None if there is none or the kernel's source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path)).get(kernel_key)
    except (ValueError, OSError):
        return None
    if not d:
        return None
    import hashlib
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["source_sha"]:
        return None
    return float(d["bytes_per_launch"])


# ---- algorithmic bytes -----------------------------------------------------

def prefill_bytes(T, H, elem=2):
    qkv = 3 * T * H * K * elem
    g = T * H * K * 4
    beta = T * H * 4
    o = T * H * V * elem
    state = H * V * K * 4          # final state written (zero initial state not read)
    return dict(intra=qkv + g + beta, scan=o + state, step=qkv + g + beta + o + state)


def gated_prefill_bytes(T, H, elem=2):
    """Raw gates in the q/k/v dtype (plus A_log, dt_bias) instead of fp32 g, beta."""
    qkv = 3 * T * H * K * elem
    gate = T * H * K * elem + T * H * elem + H * 4 + H * K * 4
    o = T * H * V * elem
    state = H * V * K * 4
    return qkv + gate + o + state


def run_gated(args, kda, dev, stream, ws):
    """The 4k prefill from the model's raw gates (bf16 raw gate and beta, lower
    bound -5), activated in-kernel: one kda_chunk_fwd_gated call per step."""
    y = kda_inputs.prefill_4k_gated()
    d = {n: y[n].to(dev) for n in ("q", "k", "v", "raw_gate", "raw_beta", "a_log", "dt_bias")}
    o = torch.empty((T_4K, H, V), dtype=torch.bfloat16, device=dev)
    sf = torch.empty((1, H, V, K), dtype=torch.float32, device=dev)
    need = kda.kda_chunk_workspace_bytes(T_4K, 1, H, flags=kda.KDA_CHUNK_GATED)
    work = torch.empty(need, dtype=torch.uint8, device=dev)

    ye = kda_inputs.with_output_gate(y, seed=6)
    og, nw = ye["out_gate"].to(dev), ye["norm_weight"].to(dev)

    def step(epi=False):
        kda.kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["raw_gate"], d["raw_beta"], d["a_log"],
                                d["dt_bias"], lower_bound=y["lower_bound"], o=o, final_state=sf,
                                workspace=work, stream=stream,
                                out_gate=og if epi else None, norm_weight=nw if epi else None,
                                norm_eps=ye["norm_eps"])

    def timed(epi):
        for _ in range(max(3, args.warmup)):
            step(epi)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(ws)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(args.steps):
            step(epi)
        b.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b), ws, dev) / args.steps

    ms = timed(False)
    status = kda.kda_workspace_status(work, stream)
    ms_epi = timed(True)
    byt = gated_prefill_bytes(T_4K, H)
    pk = peaks()
    return {"workload": "prefill_4k_gated", "tokens_per_s": round(T_4K * ws / (ms / 1e3), 1),
            "ms_per_step": round(ms, 4), "steps": args.steps,
            "with_output_epilogue": {"tokens_per_s": round(T_4K * ws / (ms_epi / 1e3), 1),
                                     "ms_per_step": round(ms_epi, 4),
                                     "epilogue": "RMSNorm(o) * weight * sigmoid(out_gate), eps 1e-5"},
            "gate": "raw bf16 gate + dt_bias, exp(A_log) scale, lower bound -5; raw bf16 beta",
            "workspace_status": status,
            "roofline": {"bound": "hbm", "algorithmic_bytes": byt,
                         "achieved": round(byt / (ms / 1e3) / 1e9, 1), "peak": pk["hbm"],
                         "unit": "GB/s", "frac": round(byt / (ms / 1e3) / 1e9 / pk["hbm"], 4)}}


def time_phases(kda, d, steps, **kw):
    """Device time of the two phases of the chunked forward, each run alone
    (kda_chunk_intra, then kda_chunk_scan: the scan after the prep, not
    alongside it), ms per call; CUDA events on the launch stream."""
    stream = kw["stream"]

    def split(ev=None):
        if ev is not None:
            ev[0].record(stream)
        kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], phase="intra", **kw)
        if ev is not None:
            ev[1].record(stream)
        kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], phase="scan", **kw)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        split()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        split(evs[i])
    torch.cuda.synchronize()
    return (statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
            statistics.mean(e[1].elapsed_time(e[2]) for e in evs))


def time_prefill(kda, d, cu, init, steps, warmup, stream, ws, fin=None, idx=None):
    """Device time of the chunked forward on resident inputs (one call per
    step, CUDA events on the launch stream between steps), ms per call as the
    median step (so that one disturbed step does not move it), and of its two
    phases run alone."""
    T, Hh, _ = d["q"].shape
    N = cu.numel() - 1
    o = torch.empty((T, Hh, V), dtype=torch.bfloat16, device=d["q"].device)
    if fin is None:
        fin = torch.empty((N, Hh, V, K), dtype=torch.float32, device=d["q"].device)
    need = kda.kda_chunk_workspace_bytes(T, N, Hh)
    work = torch.empty(need, dtype=torch.uint8, device=d["q"].device)
    kw = dict(cu_seqlens=cu, initial_state=init, o=o, final_state=fin, state_indices=idx,
              workspace=work, stream=stream)

    def step():
        kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], **kw)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    barrier(ws)
    torch.cuda.synchronize()
    evs[0].record(stream)
    for i in range(steps):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(steps))
    ms = max_over_ranks(per[steps // 2], ws, d["q"].device)
    status = kda.kda_workspace_status(work, stream)
    intra, scan = time_phases(kda, d, steps, **kw)
    del work
    return ms, intra, scan, o, fin, status


def _hbm_roof(nbytes, ms, pk):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "algorithmic_bytes": int(nbytes), "achieved": round(gbs, 1),
            "peak": pk["hbm"], "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4)}


def _oracle_tokens_per_s(x, heads, t_max=None):
    """The oracle (fp64 recurrence, OpenMP over sequence x head) on the listed
    heads of the first t_max tokens of each sequence; all-head tokens/s."""
    import oracle
    oracle.build()
    cu = x["cu_seqlens"].numpy()
    if t_max is not None:
        lens = [min(int(cu[i + 1] - cu[i]), t_max) for i in range(len(cu) - 1)]
        rows = torch.cat([torch.arange(int(cu[i]), int(cu[i]) + lens[i]) for i in range(len(lens))])
        sub_cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
        sub_cu[1:] = torch.cumsum(torch.tensor(lens), 0)
    else:
        rows, sub_cu = torch.arange(int(cu[-1])), torch.tensor(cu, dtype=torch.int64)
    sub = {n: x[n][rows][:, heads].contiguous() for n in ("q", "k", "v", "g", "beta")}
    s0 = x.get("initial_state")
    s0 = None if s0 is None else torch.swapaxes(s0[:, heads], -1, -2).double().numpy()
    cores = oracle.max_threads()
    t = time.perf_counter()
    oracle.recurrence(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"],
                      cu_seqlens=sub_cu.numpy().astype(np.int32), initial_state=s0, n_threads=cores)
    dt = time.perf_counter() - t
    tokens = rows.numel() * len(heads) / x["H"]
    return {"value": round(tokens / dt, 1), "unit": "tokens/s", "kind": "oracle",
            "cores": min(cores, len(heads) * (len(sub_cu) - 1)), "seconds": round(dt, 3),
            "sample": (f"{len(heads)} of {x['H']} heads x "
                       f"{'all' if t_max is None else f'the first {t_max}'} tokens of each of "
                       f"{len(sub_cu) - 1} sequence(s), fp64 token recurrence, OpenMP over "
                       f"(sequence, head)")}


def run_varlen(args, kda, dev, stream, pk, ws, rank):
    """varlen_8: 8 packed sequences, lengths U{512..8192} (seeded), H=32, bf16,
    nonzero fp32 initial states: one chunked forward over all of them."""
    x = kda_inputs.varlen_8()
    d = {n: x[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    cu, s0 = x["cu_seqlens"].to(dev), x["initial_state"].to(dev)
    T, N = int(x["cu_seqlens"][-1]), len(x["lengths"])
    ms, intra, scan, o, fin, status = time_prefill(kda, d, cu, s0, args.steps, args.warmup,
                                                   stream, ws)
    nb = prefill_bytes(T, H)["intra"] + T * H * V * 2 + 2 * N * H * V * K * 4
    wide = N * H * 4 > torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"workload": "varlen_8", "lengths": x["lengths"], "T": T, "H": H,
           "tokens_per_s": round(T * ws / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
           "kernels_ms": {"kda_chunk_intra": round(intra, 4), "kda_chunk_scan": round(scan, 4)},
           "scan_layout": "wide (one CTA per sequence x head)" if wide else "split",
           "roofline": dict(_hbm_roof(nb, ms, pk), note="q,k,v,g,beta,o + initial and final states"),
           "workspace_status": status, "steps": args.steps}
    del d, o, fin
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = _oracle_tokens_per_s(x, heads=[0, 1])
    return out


def run_long(args, kda, dev, stream, pk, ws, rank):
    """long_131k: B=1, T=131072, H=32, bf16, decay mix 90% U[-0.01,-1e-5] /
    10% U[-3,-1]; the final state is handed into slot 1 of a 2-slot pool and
    256 decode steps continue from it (fresh seeded tokens per step, all
    pre-staged on the device), replayed from one CUDA graph."""
    x = kda_inputs.long_131k()
    d = {n: x[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    cu = x["cu_seqlens"].to(dev)
    T = int(x["cu_seqlens"][-1])
    pool = torch.zeros((2, H, V, K), dtype=torch.float32, device=dev)
    idx = torch.tensor([1], dtype=torch.int32, device=dev)
    steps = max(2, min(args.steps, 5))
    ms, intra, scan, o, _, status = time_prefill(kda, d, cu, None, steps, min(args.warmup, 3),
                                                 stream, ws, fin=pool, idx=idx)
    nb = prefill_bytes(T, H)["step"]
    del d, o
    # hand-off decode: B=1, 32 heads, state slot 1 (2 MiB, resident in L2)
    toks = [kda_inputs.decode_tokens(1, H=H, seed=4, step=t, g_mixed=True) for t in range(256)]
    toks = [{n: t[n].to(dev) for n in ("q", "k", "v", "g", "beta")} for t in toks]
    o1 = torch.empty((256, 1, H, V), dtype=torch.bfloat16, device=dev)

    def dstep(i, st):
        t = toks[i]
        kda.kda_recurrent_step(t["q"], t["k"], t["v"], t["g"], t["beta"], pool, state_indices=idx,
                               o=o1[i], stream=st)

    for i in range(3):
        dstep(i, stream)
    torch.cuda.synchronize()
    us = _graph_us(dstep, 256, stream, reps=3)
    out = {"workload": "long_131k", "T": T, "H": H,
           "prefill": {"tokens_per_s": round(T * ws / (ms * 1e-3), 1), "ms_per_step": round(ms, 4),
                       "kernels_ms": {"kda_chunk_intra": round(intra, 4),
                                      "kda_chunk_scan": round(scan, 4)},
                       "roofline": dict(_hbm_roof(nb, ms, pk),
                                        note="bound in practice by 2048 sequential chunk steps per head"),
                       "workspace_status": status, "steps": steps},
           "handoff_decode": {"steps": 256, "us_per_step": round(us, 3),
                              "timing": "256 steps from the handed-off pool slot, one CUDA graph replay",
                              "l2_resident": "the 2 MiB state and 40 KB of inputs per step stay in L2",
                              "launches_per_step": 1}}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = _oracle_tokens_per_s(x, heads=list(range(16)), t_max=8192)
    return out


def _graph_us(fn, n, stream, reps=5):
    """Per-call device time of fn(0..n-1) captured in one CUDA graph and
    replayed: no host launch gaps inside the timed region."""
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()  # capture needs a side stream
    cs.wait_stream(stream)
    with torch.cuda.graph(g, stream=cs):
        for i in range(n):
            fn(i, cs)
    times = []
    with torch.cuda.stream(stream):
        g.replay()
        torch.cuda.synchronize()
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e3 / n)
    del g
    return statistics.median(times)


def run_conv(args, kda, dev, stream, pk):
    """The short causal convolution on the fused q/k/v projection (D = 3 x 32
    x 128 = 12288 channels, ks = 4, SiLU, bf16): prefill over the 4k sequence
    (x and y 96 MiB each, above L2) and one decode update for 256 sequences,
    rotating over 8 input/pool sets (about 250 MB) so that no step finds its
    data in L2.  Both are timed as CUDA-graph replays of 16 / 32 calls (the
    decode update is shorter than a host launch)."""
    c = kda_inputs.conv_inputs([T_4K], seed=83)
    D, ks = c["D"], c["ks"]
    x, w, cu = c["x"].to(dev), c["weight"].to(dev), c["cu_seqlens"].to(dev)
    y = torch.empty_like(x)
    fin = torch.empty((1, ks - 1, D), dtype=x.dtype, device=dev)

    def pre(i, st=stream):
        kda.kda_short_conv_fwd(x, w, cu_seqlens=cu, final_states=fin, y=y, stream=st)

    for i in range(3):
        pre(i)
    torch.cuda.synchronize()
    us_pre = _graph_us(pre, 16, stream)
    b_pre = 2 * T_4K * D * 2 + ks * D * 2 + (ks - 1) * D * 2
    del x, y
    sets = []
    for j in range(8):
        g = torch.Generator().manual_seed(8300 + j)
        sets.append((torch.randn((DEC_N, D), generator=g).to(torch.bfloat16).to(dev),
                     torch.randn((DEC_N, ks - 1, D), generator=g).to(torch.bfloat16).to(dev),
                     torch.empty((DEC_N, D), dtype=torch.bfloat16, device=dev)))

    def upd(i, st=stream):
        xt, pool, yt = sets[i % len(sets)]
        kda.kda_short_conv_update(xt, w, pool, y=yt, stream=st)

    for i in range(8):
        upd(i)
    torch.cuda.synchronize()
    us_upd = _graph_us(upd, 32, stream)
    b_upd = DEC_N * D * 2 * 2 + 2 * DEC_N * (ks - 1) * D * 2 + ks * D * 2
    # speculative verify width 4: per-token state slots, accepted counts 1..4
    SV = 4
    spec = []
    for j in range(4):
        g = torch.Generator().manual_seed(8400 + j)
        spec.append((torch.randn((DEC_N, SV, D), generator=g).to(torch.bfloat16).to(dev),
                     torch.randn((DEC_N * SV, ks - 1, D), generator=g).to(torch.bfloat16).to(dev),
                     torch.empty((DEC_N, SV, D), dtype=torch.bfloat16, device=dev)))
    sidx = torch.arange(DEC_N * SV, dtype=torch.int32, device=dev).view(DEC_N, SV)
    sacc = (torch.arange(DEC_N, dtype=torch.int32, device=dev) % SV) + 1

    def spec_upd(i, st=stream):
        xt, pool, yt = spec[i % len(spec)]
        kda.kda_short_conv_multi_update(xt, w, pool, sidx, num_accepted=sacc, y=yt, stream=st)

    for i in range(4):
        spec_upd(i)
    torch.cuda.synchronize()
    us_spec = _graph_us(spec_upd, 32, stream)
    b_spec = DEC_N * SV * D * 2 * 2 + (1 + SV) * DEC_N * (ks - 1) * D * 2 + ks * D * 2
    del sets, spec
    roof = lambda b, us: {"bound": "hbm", "algorithmic_bytes": b,
                          "achieved": round(b / (us * 1e-6) / 1e9, 1), "peak": pk["hbm"],
                          "unit": "GB/s", "frac": round(b / (us * 1e-6) / 1e9 / pk["hbm"], 4)}
    pre_roof = dict(roof(b_pre, us_pre), kernel="conv_prefill_kernel",
                    traffic=traffic_from_profiles("conv_prefill"))
    return {"workload": "short_conv_qkv", "D": D, "ks": ks, "activation": "silu", "dtype": "bf16",
            "timing": "CUDA graph replay, per call",
            "prefill": {"T": T_4K, "us_per_call": round(us_pre, 2), "launches_per_call": 1,
                        "tokens_per_s": round(T_4K / (us_pre * 1e-6), 1),
                        "roofline": pre_roof},
            "decode_update": {"N": DEC_N, "us_per_call": round(us_upd, 2), "launches_per_call": 1,
                              "roofline": roof(b_upd, us_upd)},
            "speculative_update": {"N": DEC_N, "verify_width": SV, "us_per_call": round(us_spec, 2),
                                   "launches_per_call": 1, "roofline": roof(b_spec, us_spec)}}


def decode_bytes(N, H, elem=2):
    state = 2 * N * H * V * K * 4  # read + write
    io = N * H * (2 * K * elem + V * elem + K * 4 + 4 + V * elem)
    return state + io


# ---- our arm ---------------------------------------------------------------

def run_ours(args, rank, ws):
    import kimi_delta_attention_07_gb300 as kda
    kda.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    pk = peaks()

    x = kda_inputs.prefill_4k()
    d = {n: x[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    flags = kda.KDA_CHUNK_PRECISE if args.precise else 0
    ws_bytes = kda.kda_chunk_workspace_bytes(T_4K, 1, H, K, V, kda.KDA_BF16, flags)
    work = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    o = torch.empty((T_4K, H, V), dtype=torch.bfloat16, device=dev)
    sf = torch.empty((1, H, V, K), dtype=torch.float32, device=dev)
    kw = dict(o=o, final_state=sf, workspace=work, precise=args.precise, stream=stream)

    def step():  # the whole forward: one kda_chunk_fwd call (or its two phases)
        if args.phases:
            kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], phase="intra", **kw)
            kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], phase="scan", **kw)
        else:
            kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], **kw)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    clocks = Clocks(dev.index) if rank == 0 else None
    time.sleep(0.15)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(ws)
    total_ms = start.elapsed_time(end)
    # the kernels alone, for the breakdown: the prep phase (chunk index, main
    # and strong-decay prep) and the scan after it
    intra_ms, scan_ms = time_phases(kda, d, args.steps, **kw)
    total_ms = max_over_ranks(total_ms, ws, dev)
    ms_per_step = total_ms / args.steps
    tokens = T_4K * args.steps * ws
    value = tokens / (total_ms / 1e3)

    nb = prefill_bytes(T_4K, H)
    kernels = {
        "kda_chunk_intra": dict(ms=intra_ms, algorithmic_bytes=nb["intra"],
                                gbs=nb["intra"] / (intra_ms * 1e-3) / 1e9),
        "kda_chunk_scan": dict(ms=scan_ms, algorithmic_bytes=nb["scan"],
                               gbs=nb["scan"] / (scan_ms * 1e-3) / 1e9),
    }
    tot = intra_ms + scan_ms
    for v_ in kernels.values():
        v_["share"] = v_["ms"] / tot
    dom = max(kernels, key=lambda n: kernels[n]["ms"])
    dk = kernels[dom]
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(dk["gbs"], 1),
                "peak": pk["hbm"], "unit": "GB/s", "frac": round(dk["gbs"] / pk["hbm"], 4),
                "traffic": traffic_from_profiles(dom + ("_precise" if args.precise else "")),
                "peak_source": pk["source"] + " (burst HBM copy)",
                "timing": "the kernel alone (phase-split calls); in the step the scan runs "
                          "alongside the prep"}
    step_gbs = nb["step"] / (ms_per_step * 1e-3) / 1e9
    step_roofline = {"bound": "hbm", "algorithmic_bytes": nb["step"], "achieved": round(step_gbs, 1),
                     "peak": pk["hbm"], "unit": "GB/s", "frac": round(step_gbs / pk["hbm"], 4)}

    if rank == 0:
        clocks.stop()
        clk = clocks.summary(t_wall0, t_wall1)
    else:
        clk = None

    e2e = None if args.no_e2e else run_e2e(args, kda, x, dev, stream, work, flags, ws)
    dec = None if args.no_decode else run_decode(args, kda, dev, stream, pk, ws)
    gated = None if (args.no_gated or args.precise) else run_gated(args, kda, dev, stream, ws)
    conv = None if args.no_conv else run_conv(args, kda, dev, stream, pk)
    varlen = None if (args.no_varlen or args.precise) else run_varlen(args, kda, dev, stream, pk, ws, rank)
    long_ = None if (args.no_long or args.precise) else run_long(args, kda, dev, stream, pk, ws, rank)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x, sample_heads=H)

    launches = KERNELS_PER_PREFILL * args.steps
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp32" if args.precise else "bf16",
            "data": "synthetic (seeded, torch.Generator on CPU)",
            "config": {"workload": "prefill_4k", "B": 1, "T": T_4K, "H": H, "K": K, "V": V,
                       "chunk": 64, "io_dtype": "bf16", "g_beta_state": "fp32",
                       "global_batch_tokens": T_4K * ws, "parallelism": f"replicas{ws}",
                       "l2": "inputs + workspace > 129 MB L2, no flush",
                       "path": "fp32 CUDA-core (precise)" if args.precise else "default",
                       "step": ("the two phases run one after the other" if args.phases else
                                "one forward: the scan runs alongside the prep")},
            "roofline": roofline, "step_roofline": step_roofline, "kernels": kernels,
            "e2e": e2e, "gpu_launches": launches, "clocks": clk,
            "decode": dec, "gated": gated, "short_conv": conv, "varlen_8": varlen,
            "long_131k": long_, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_e2e(args, kda, x, dev, stream, work, flags, ws):
    """Same metric through the public call with HOST buffers: every step copies
    its inputs in from pinned host memory, runs the chunked forward and copies
    the output and final state back, all inside the timed region.  Steps are
    pipelined the way a serving loop would run them: the inputs of step i+1
    are copied in (two copy streams) while step i computes and step i-1's
    results are copied out (a third stream); device input buffers are
    double-buffered."""
    names = ("q", "k", "v", "g", "beta")
    host = {n: x[n].pin_memory() for n in names}
    nbuf = 2
    d = [{n: torch.empty_like(host[n], device=dev) for n in names} for _ in range(nbuf)]
    o = [torch.empty((T_4K, H, V), dtype=torch.bfloat16, device=dev) for _ in range(nbuf)]
    sf = [torch.empty((1, H, V, K), dtype=torch.float32, device=dev) for _ in range(nbuf)]
    o_h = torch.empty((T_4K, H, V), dtype=torch.bfloat16).pin_memory()
    s_h = torch.empty((1, H, V, K), dtype=torch.float32).pin_memory()
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = o_h.numel() * 2 + s_h.numel() * 4
    copy_in = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
    copy_out = torch.cuda.Stream(device=dev)
    lanes = (("q", "g"), ("k", "v", "beta"))  # bytes split about evenly over the copy streams

    def ev():
        return torch.cuda.Event(enable_timing=False)

    def run(steps, start_ev=None, end_ev=None):
        in_done = [[ev() for _ in copy_in] for _ in range(steps)]
        done = [ev() for _ in range(steps)]
        out_done = [ev() for _ in range(steps)]
        if start_ev is not None:
            start_ev.record(stream)
            for cs in (*copy_in, copy_out):
                cs.wait_stream(stream)
        for i in range(steps):
            b = i % nbuf
            for li, cs in enumerate(copy_in):
                if i >= nbuf:
                    cs.wait_event(done[i - nbuf])  # buffer b is free again
                with torch.cuda.stream(cs):
                    for n in lanes[li]:
                        d[b][n].copy_(host[n], non_blocking=True)
                in_done[i][li].record(cs)
            for e_ in in_done[i]:
                stream.wait_event(e_)
            if i >= nbuf:
                stream.wait_event(out_done[i - nbuf])  # o / final state of buffer b read out
            kda.kda_chunk_fwd(d[b]["q"], d[b]["k"], d[b]["v"], d[b]["g"], d[b]["beta"], o=o[b],
                              final_state=sf[b], workspace=work, precise=bool(flags), stream=stream)
            done[i].record(stream)
            copy_out.wait_event(done[i])
            with torch.cuda.stream(copy_out):
                o_h.copy_(o[b], non_blocking=True)
                s_h.copy_(sf[b], non_blocking=True)
            out_done[i].record(copy_out)
        if end_ev is not None:
            for cs in (*copy_in, copy_out):
                stream.wait_stream(cs)
            end_ev.record(stream)

    run(3)
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 20))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    run(steps, a, b)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), ws, dev)
    return {"value": round(T_4K * steps * ws / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "pipelined": "copy-in of step i+1 and copy-out of step i-1 overlap step i"}


def run_decode(args, kda, dev, stream, pk, ws):
    """256 sequences x 32 heads, 512 MiB fp32 state pool, 64 consecutive decode
    steps with fresh bf16 tokens each step (all inputs pre-staged on the device)."""
    pool = kda_inputs.decode_pool(DEC_N, H=H, seed=3).to(dev)
    toks = [kda_inputs.decode_tokens(DEC_N, H=H, seed=3, step=t) for t in range(DEC_STEPS)]
    toks = [{n: t[n].to(dev) for n in ("q", "k", "v", "g", "beta")} for t in toks]
    o = torch.empty((DEC_N, H, V), dtype=torch.bfloat16, device=dev)
    for t in range(3):  # warm-up on a scratch copy so the timed 64 steps start from the seed pool
        scratch = pool.clone()
        kda.kda_recurrent_step(*(toks[t][n] for n in ("q", "k", "v", "g", "beta")), scratch, o=o,
                               stream=stream)
        del scratch
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(DEC_STEPS)]
    barrier(ws)
    torch.cuda.synchronize()
    for t in range(DEC_STEPS):
        evs[t][0].record(stream)
        kda.kda_recurrent_step(*(toks[t][n] for n in ("q", "k", "v", "g", "beta")), pool, o=o,
                               stream=stream)
        evs[t][1].record(stream)
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    med = max_over_ranks(statistics.median(us), ws, dev)
    nbytes = decode_bytes(DEC_N, H)
    gbs = nbytes / (med * 1e-6) / 1e9
    # the model's decode path: raw gates in, output epilogue out (same pool, continued)
    gtoks = [kda_inputs.with_output_gate(kda_inputs.with_raw_gates(
        kda_inputs.decode_tokens(DEC_N, H=H, seed=3, step=DEC_STEPS + t), seed=5), seed=6)
        for t in range(8)]
    names = ("q", "k", "v", "raw_gate", "raw_beta", "a_log", "dt_bias")
    gd = [{n: t[n].to(dev) for n in names + ("out_gate", "norm_weight")} for t in gtoks]

    def gstep(t):
        kda.kda_recurrent_step_gated(*(gd[t][n] for n in names), pool, lower_bound=-5.0,
                                     out_gate=gd[t]["out_gate"], norm_weight=gd[t]["norm_weight"],
                                     norm_eps=1e-5, o=o, stream=stream)

    gstep(0)
    torch.cuda.synchronize()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(8)]
    for t in range(8):
        gev[t][0].record(stream)
        gstep(t)
        gev[t][1].record(stream)
    torch.cuda.synchronize()
    gus = statistics.median([a.elapsed_time(b) * 1e3 for a, b in gev])
    del gd, gtoks
    spec = run_spec_decode(kda, dev, stream, pk)
    return {"workload": "decode_256", "us_per_step": round(med, 2),
            "gated_epilogue_us_per_step": round(gus, 2), "speculative": spec,
            "us_min": round(min(us), 2), "tokens_per_s": round(DEC_N * ws / (med * 1e-6), 1),
            "steps": DEC_STEPS, "launches": DEC_STEPS * KERNELS_PER_DECODE,
            "roofline": {"kernel": "recurrent_step_kernel", "bound": "hbm",
                         "algorithmic_bytes": nbytes, "achieved": round(gbs, 1),
                         "peak": pk["hbm"], "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4),
                         "traffic": traffic_from_profiles("recurrent_step_kernel")}}


def run_spec_decode(kda, dev, stream, pk, S=4, steps=16):
    """Speculative decode with a verify width of S: 256 sequences x 32 heads,
    S draft tokens each, per-token slots in a pool of 256 S slots, accepted
    counts cycling 1..S.  The state is read once and written S times."""
    slots = DEC_N * S
    pool = kda_inputs.decode_pool(slots, H=H, seed=73).to(dev)
    idx = torch.arange(slots, dtype=torch.int32, device=dev).view(DEC_N, S)
    acc = (torch.arange(DEC_N, dtype=torch.int32, device=dev) % S) + 1
    toks = [{n: t.to(dev) for n, t in kda_inputs.spec_tokens(DEC_N, S, H=H, seed=73, step=i).items()}
            for i in range(4)]
    o = torch.empty((DEC_N, S, H, V), dtype=torch.bfloat16, device=dev)

    def one(i):
        t = toks[i % len(toks)]
        kda.kda_recurrent_multi_step(t["q"], t["k"], t["v"], t["g"], t["beta"], pool, idx,
                                     num_accepted=acc, o=o, stream=stream)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        evs[i][0].record(stream)
        one(i)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    us = statistics.median([a.elapsed_time(b) * 1e3 for a, b in evs])
    nbytes = (1 + S) * DEC_N * H * V * K * 4 + S * DEC_N * H * (3 * K * 2 + K * 4 + 4 + V * 2)
    gbs = nbytes / (us * 1e-6) / 1e9
    # the model's form: raw gates in, output epilogue out (same pool, continued)
    gtoks = [kda_inputs.with_output_gate(kda_inputs.with_raw_gates(t, seed=74), seed=75) for t in
             (kda_inputs.spec_tokens(DEC_N, S, H=H, seed=74, step=i) for i in range(2))]
    names = ("q", "k", "v", "raw_gate", "raw_beta", "a_log", "dt_bias")
    gd = [{n: t[n].to(dev) for n in names + ("out_gate", "norm_weight")} for t in gtoks]

    def gone(i):
        t = gd[i % len(gd)]
        kda.kda_recurrent_multi_step_gated(*(t[n] for n in names), pool, idx, num_accepted=acc,
                                           lower_bound=-5.0, out_gate=t["out_gate"],
                                           norm_weight=t["norm_weight"], norm_eps=1e-5, o=o,
                                           stream=stream)

    for i in range(2):
        gone(i)
    torch.cuda.synchronize()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(8)]
    for i in range(8):
        gev[i][0].record(stream)
        gone(i)
        gev[i][1].record(stream)
    torch.cuda.synchronize()
    gus = statistics.median([a.elapsed_time(b) * 1e3 for a, b in gev])
    del pool, gd, gtoks
    return {"verify_width": S, "us_per_step": round(us, 2), "gated_epilogue_us_per_step": round(gus, 2),
            "tokens_per_s": round(DEC_N * S / (us * 1e-6), 1),
            "roofline": {"bound": "hbm", "algorithmic_bytes": nbytes, "achieved": round(gbs, 1),
                         "peak": pk["hbm"], "unit": "GB/s", "frac": round(gbs / pk["hbm"], 4)}}


# ---- the oracle as the CPU baseline / reference arm ------------------------

def cpu_baseline(x, sample_heads, min_seconds=1.0, max_reps=8):
    """The oracle on the host cores: the whole 4k workload (all heads), run
    until at least min_seconds of wall time (about 10-30 core-seconds on a
    16-core Grace host)."""
    import oracle
    heads = list(range(sample_heads))
    sub = {n: x[n][:, heads].contiguous() for n in ("q", "k", "v", "g", "beta")}
    cores = oracle.max_threads()
    reps, dt = 0, 0.0
    while reps < max_reps and (reps == 0 or dt < min_seconds):
        t = time.perf_counter()
        oracle.recurrence(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], n_threads=cores)
        dt += time.perf_counter() - t
        reps += 1
    tokens = reps * x["q"].shape[0] * len(heads) / H  # in units of full (all-head) tokens
    used = min(cores, len(heads))
    return {"value": round(tokens / dt, 1), "unit": "tokens/s", "cores": used,
            "kind": "oracle", "seconds": round(dt, 3), "core_seconds": round(dt * used, 1),
            "sample": f"prefill_4k x {reps}, {len(heads)} of {H} heads x {x['q'].shape[0]} "
                      f"tokens, fp64 token recurrence, OpenMP over heads"}


def run_reference(args, rank, ws):
    if rank != 0:
        return
    import oracle
    oracle.build()
    x = kda_inputs.prefill_4k()
    cores = oracle.max_threads()
    heads = list(range(min(H, max(cores, 1))))
    sub = {n: x[n][:, heads].contiguous() for n in ("q", "k", "v", "g", "beta")}

    def step():
        oracle.recurrence(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], n_threads=cores)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    tokens = T_4K * len(heads) / H * args.steps
    value = tokens / dt
    sample = (f"prefill_4k, {len(heads)} of {H} heads x {T_4K} tokens per step, fp64 token "
              f"recurrence (the oracle), OpenMP over heads")
    line = {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "prefill_4k", "B": 1, "T": T_4K, "H": H, "K": K, "V": V},
            "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s",
                             "cores": min(cores, len(heads)), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # `bench.py --gpus N` started directly: launch the N ranks ourselves
        if args.impl != "reference" and torch.cuda.device_count() < args.gpus:
            sys.exit(f"bench.py: --gpus {args.gpus} but only {torch.cuda.device_count()} "
                     f"CUDA device(s) are visible")
        sys.exit(spawn_ranks(args.gpus, os.path.abspath(__file__), sys.argv[1:]))
    if int(os.environ.get("WORLD_SIZE", "1")) != args.gpus:
        sys.exit(f"bench.py: WORLD_SIZE={os.environ.get('WORLD_SIZE')} but --gpus {args.gpus}")
    if args.impl == "reference":
        rank, ws = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
        run_reference(args, rank, ws)
        return
    rank, ws = dist_setup("nccl")
    try:
        run_ours(args, rank, ws)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
