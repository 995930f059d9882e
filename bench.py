#!/usr/bin/env python
"""Benchmark of causal log-linear Mamba-2 attention on one GB300 per rank.

One step = one lla_forward over the mid-size prefill workload (B=4, H=16,
T=8192, dk=128, dv=64, bf16 q/k/v, chunk 64), inputs resident in HBM (434 MB,
larger than L2, so no flush between steps). The same run also times the
recurrent decode workload (64 sequences x 16 heads, t ~ U[1, 65536), 1000
one-token steps) and reports its HBM bandwidth. Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lla|reference]

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from log_linear_attention_gb300 import inputs  # noqa: E402

METRIC = "log-linear attn fwd tokens/s & TFLOP/s vs bf16 peak @T=8192; decode GB/s vs HBM"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# fp32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 flop x 2.07 GHz (maximum SM clock)
ALU_F32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


# ----------------------------------------------------------------------------- work model

def popcount_sum(n: int) -> int:
    return sum(bin(j).count("1") for j in range(n))


def prefill_work(cfg: inputs.PrefillConfig) -> dict:
    """Algorithmic flops and minimum bytes of one prefill call: causal pairs only,
    nonempty Fenwick levels only, each input read once and the output written once."""
    BH = cfg.B * cfg.H
    C, dk, dv, T = cfg.chunk, cfg.dk, cfg.dv, cfg.T
    N = T // C
    esz = 2 if cfg.dtype == "bf16" else 4
    intra = BH * N * C * (C + 1) // 2 * 2 * (dk + dv)
    state = BH * N * 2 * C * dk * dv
    level = BH * popcount_sum(N) * 2 * C * dk * dv
    in_bytes = BH * T * (2 * dk + dv) * esz + BH * T * 4 + BH * T * cfg.L * 4
    out_bytes = BH * T * dv * esz
    return dict(intra=intra, state=state, level=level, flops=intra + state + level,
                in_bytes=in_bytes, out_bytes=out_bytes, bytes=in_bytes + out_bytes)


def kernel_work(name: str, cfg: inputs.PrefillConfig) -> dict:
    """Per-launch algorithmic work of each kernel the forward launches, and its bound."""
    w = prefill_work(cfg)
    BH = cfg.B * cfg.H
    T, dk, dv = cfg.T, cfg.dk, cfg.dv
    esz = 2 if cfg.dtype == "bf16" else 4
    q_b = BH * T * dk * esz
    k_b = BH * T * dk * esz
    v_b = BH * T * dv * esz
    a_b = BH * T * 4
    lam_b = BH * T * cfg.L * 4
    if name == "simt_output":
        return dict(bound="alu", flops=w["intra"] + w["level"],
                    bytes=q_b + k_b + v_b + a_b + lam_b + w["out_bytes"])
    if name == "simt_chunk_state":
        return dict(bound="alu", flops=w["state"], bytes=k_b + v_b + a_b + BH * (T // cfg.chunk) * dk * dv * 4)
    if name == "tc_output":
        return dict(bound="hbm", flops=w["intra"] + w["level"],
                    bytes=q_b + k_b + v_b + a_b + lam_b + w["out_bytes"])
    if name == "tc_nodes":
        return dict(bound="hbm", flops=w["state"], bytes=k_b + v_b + a_b)
    return dict(bound="hbm", flops=0, bytes=a_b)


def backward_work(cfg: inputs.PrefillConfig) -> dict:
    """Algorithmic work of one lla_backward call (causal pairs and nonempty levels only):
    in-chunk pairs need q.k, dO.v, and the dq, dk, dv products (3 dk + 2 dv multiply-adds);
    the forward nodes are rebuilt (state); every level read appears twice (B dO for dq and
    the node gradient q dO^T); the key side applies C_i twice (dk and dv)."""
    w = prefill_work(cfg)
    BH = cfg.B * cfg.H
    C = min(cfg.chunk, 64)
    N = cfg.T // C
    intra = BH * N * C * (C + 1) // 2 * 2 * (3 * cfg.dk + 2 * cfg.dv)
    state = BH * N * 2 * C * cfg.dk * cfg.dv
    level = BH * sum(bin(j).count("1") for j in range(N)) * 2 * C * cfg.dk * cfg.dv
    keyside = 2 * state
    esz = 2 if cfg.dtype == "bf16" else 4
    nbytes = (w["in_bytes"] + BH * cfg.T * cfg.dv * esz  # inputs + dout
              + BH * cfg.T * (2 * cfg.dk + cfg.dv) * esz + BH * cfg.T * 4 * (1 + cfg.L))  # gradients
    return dict(flops=intra + state + 2 * level + keyside, bytes=nbytes)


def decode_bytes(t: np.ndarray, H: int, dk: int, dv: int, Lmax: int, esz: int = 2) -> int:
    """Bytes one decode step must move: every nonempty state level read once
    (popcount(t-1) + 1 of them) and every level held after the step written once
    (popcount(t) + 1), fp32; plus the token vectors, lambda, log_a and the output."""
    total = 0
    for x in t.tolist():
        reads = (bin(x - 1).count("1") + 1) if x > 0 else 0
        writes = bin(x).count("1") + 1
        total += H * 4 * dk * dv * (reads + writes)
    total += len(t) * H * ((2 * dk + dv) * esz + 4 + Lmax * 4 + dv * esz) + len(t) * 8
    return total


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = dict(hbm_gbs=FALLBACK_HBM_GBS, bf16_tflops=FALLBACK_BF16_TFLOPS,
                 bf16_tflops_sustained=1700.0, source="fallback")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k_, v_ in x.items():
                        walk(v_, f"{pre}{k_}.")
                else:
                    flat[pre[:-1]] = x
            walk(d)
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                for fk, fv in flat.items():
                    if fk.split(".")[-1] == key and isinstance(fv, (int, float)):
                        peaks[key] = float(fv)
            peaks["source"] = "measured"
        except Exception:
            pass
    return peaks


def traffic_record(name: str):
    """DRAM bytes per launch from the committed ncu summary (profiles/ncu_traffic.txt), if the
    kernel's source still has the hash recorded at capture time; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    try:
        for line in open(path):
            parts = line.split()
            if not parts or parts[0].startswith("#") or parts[0] != name or len(parts) != 4:
                continue
            # the kernel's source files, '+'-joined: their concatenation is what was hashed
            h = hashlib.sha256()
            for src in parts[1].split("+"):
                h.update(open(os.path.join(ROOT, src), "rb").read())
            if h.hexdigest() != parts[2]:
                return None
            return float(parts[3])
    except OSError:
        return None
    return None


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        time.sleep(0.15)
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [l for (ts, l) in self.lines if self.t0 is not None and self.t0 <= ts <= (self.t1 or ts)]
        adjacent = False
        if not inside and self.lines:
            # region shorter than the sampling period: take the samples nearest to it
            mid = ((self.t0 or 0) + (self.t1 or 0)) / 2
            inside = [l for _, l in sorted(self.lines, key=lambda x: abs(x[0] - mid))[:3]]
            adjacent = True
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in inside:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, p in zip(names, parts[5:9]):
                if p.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "adjacent_samples": adjacent}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device: str = "cuda") -> float:
    """The slowest rank's time: every rank's timing scalar reduced with MAX (the only
    collective of the benchmark; the workload itself has no data-path exchange)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(tokens_per_rank: int, ms_max: float, ws: int) -> float:
    """Whole-job throughput under weak scaling: every rank processes its own full
    workload, so the job moves ws * tokens_per_rank tokens in the slowest rank's time."""
    return ws * tokens_per_rank / (ms_max / 1e3)


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- oracle (CPU baseline)

def oracle_tokens_per_s(cfg: inputs.PrefillConfig, inp: inputs.PrefillInputs, budget_s: float, T_sample=None):
    """Time the fp64 oracle (recurrent form, one core) on whole heads of the workload
    until ``budget_s`` elapses; returns (tokens/s in whole-token units, sample text)."""
    import oracle
    T = cfg.T if T_sample is None else T_sample
    heads = 0
    t0 = time.perf_counter()
    for bh in range(cfg.B * cfg.H):
        b, h = divmod(bh, cfg.H)
        sl = (slice(b, b + 1), slice(h, h + 1), slice(0, T))
        lam = inp.lam[sl][..., :inputs.num_levels(T)]
        oracle.recurrent(inp.q[sl], inp.k[sl], inp.v[sl], inp.log_a[sl], lam)
        heads += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    tokens = heads * T / cfg.H  # a token of the workload carries all H heads
    return tokens / dt, f"{heads} of {cfg.B * cfg.H} heads x {T} tokens (recurrent form), scaled by 1/H", dt


def cpu_info() -> dict:
    """Host CPU model and core count (the CPU baseline runs on these cores)."""
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":")[0].strip().lower()
            if key in ("model name", "cpu model", "hardware"):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if not model:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or "unknown"}


def oracle_tokens_per_s_all_cores(cfg: inputs.PrefillConfig, inp: inputs.PrefillInputs, budget_s: float):
    """The same oracle (single-threaded C, unchanged) on every host core at once: a thread
    pool over independent (b, h) heads (the ctypes calls release the GIL). Returns
    (tokens/s in whole-token units, threads used, sample text)."""
    import concurrent.futures
    import oracle
    n = os.cpu_count() or 1
    T = cfg.T
    L = inputs.num_levels(T)

    def one(bh):
        b, h = divmod(bh, cfg.H)
        sl = (slice(b, b + 1), slice(h, h + 1), slice(0, T))
        oracle.recurrent(inp.q[sl], inp.k[sl], inp.v[sl], inp.log_a[sl], inp.lam[sl][..., :L])
        return 1

    heads = 0
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        nxt = 0
        while nxt < cfg.B * cfg.H and time.perf_counter() - t0 < budget_s:
            batch = list(range(nxt, min(nxt + n, cfg.B * cfg.H)))
            nxt += len(batch)
            heads += sum(ex.map(one, batch))
    dt = time.perf_counter() - t0
    return heads * T / cfg.H / dt, n, f"{heads} of {cfg.B * cfg.H} heads x {T} tokens (recurrent form) on {n} threads"


def run_reference(args, cfg):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = inputs.make_prefill(cfg, seed=0, B=1, H=1)
    one = inputs.PrefillConfig(**{**cfg.__dict__, "B": 1, "H": 1})
    # size each step so that warmup + steps end within about two minutes
    est_per_token = 2.5e-4
    T_sample = cfg.T
    while T_sample > 1024 and (args.steps + args.warmup) * T_sample * est_per_token > 120:
        T_sample //= 2
    for _ in range(args.warmup):
        oracle_tokens_per_s(one, inp, 0.0, T_sample)
    times = []
    for _ in range(args.steps):
        _, sample, dt = oracle_tokens_per_s(one, inp, 0.0, T_sample)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = (T_sample / cfg.H) / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "B": cfg.B, "H": cfg.H, "T": cfg.T, "dk": cfg.dk, "dv": cfg.dv,
                   "chunk": cfg.chunk},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step: 1 head x {T_sample} tokens of the workload (recurrent form, fp64), "
                                   f"scaled by 1/H"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm

def cuda_time(fn, steps, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


VARLEN = dict(n_seq=32, H=16, dk=128, dv=64, min_len=256, max_len=8192, chunk=64)


def bench_varlen(args, dev, stream, rank):
    """Packed prefill and hand-off of a serving-like mix: VARLEN["n_seq"] sequences with lengths
    uniform in [min_len, max_len] (seeded), headline distributions, drawn on the device."""
    import torch
    from log_linear_attention_gb300 import binding
    c = VARLEN
    lengths = np.random.default_rng(1234 + rank).integers(c["min_len"], c["max_len"] + 1, size=c["n_seq"])
    total, max_T = int(lengths.sum()), int(lengths.max())
    H, dk, dv = c["H"], c["dk"], c["dv"]
    L = inputs.num_levels(max_T)
    g = torch.Generator(device=dev)
    g.manual_seed(4321 + rank)
    q = torch.randn((H, total, dk), device=dev, generator=g)
    q = (q / q.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    k = torch.randn((H, total, dk), device=dev, generator=g)
    k = (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    v = torch.randn((H, total, dv), device=dev, generator=g).to(torch.bfloat16)
    la = -torch.nn.functional.softplus(torch.randn((H, total), device=dev, generator=g) - 2.0)
    lam = torch.nn.functional.softplus(torch.randn((H, total, L), device=dev, generator=g))
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).to(dev)
    out = torch.empty((H, total, dv), dtype=torch.bfloat16, device=dev)
    states = torch.empty((c["n_seq"], H, L, dk, dv), dtype=torch.float32, device=dev)

    def fstep():
        binding.forward_varlen(q, k, v, la, lam, cu, max_T, c["chunk"], out=out)

    def hstep():
        binding.prefill_state_varlen(k, v, la, cu, max_T, states)

    for _ in range(3):
        fstep()
        hstep()
    n = max(3, min(args.steps, 10))
    f_ms = cuda_time(fstep, n, stream) / n
    h_ms = cuda_time(hstep, n, stream) / n
    assert binding.device_error() == 0
    return dict(workload=f"{c['n_seq']} packed sequences x {H} heads, lengths U[{c['min_len']},{c['max_len']}] "
                         f"(total {total}, max {max_T}), dk={dk} dv={dv} bf16",
                prefill_ms=f_ms, prefill_tokens_per_s=total / (f_ms / 1e3),
                handoff_ms=h_ms, handoff_tokens_per_s=total / (h_ms / 1e3),
                layout="packed: each sequence's own 128-token tiles (no padded copy) on the tensor-core path",
                tile_overhead=float(sum((int(x) + 127) // 128 * 128 for x in lengths)) / total)


def bench_decode(args, dev, stream, rank, ws):
    """Time args.decode_steps one-token decode steps of the decode workload; returns
    (total ms, algorithmic bytes moved, steps)."""
    import torch
    from log_linear_attention_gb300 import binding

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    dcfg = inputs.DECODE_CONFIG
    dsteps = args.decode_steps
    t0v = inputs.make_positions(dcfg, rank)
    t_all_np = t0v[None, :] + np.arange(dsteps + max(args.warmup, 3), dtype=np.int64)[:, None]
    t_all = torch.from_numpy(t_all_np).to(dev)
    n_tok = 32
    toks = [inputs.make_decode_token(dcfg, rank * 1000 + i) for i in range(n_tok)]
    dq_s = [(bf16(tk.bits["q"]).to(dev), bf16(tk.bits["k"]).to(dev), bf16(tk.bits["v"]).to(dev),
             torch.from_numpy(tk.log_a).to(dev), torch.from_numpy(tk.lam).to(dev)) for tk in toks]
    states = torch.randn((dcfg.batch, dcfg.H, dcfg.Lmax, dcfg.dk, dcfg.dv), device=dev,
                         generator=torch.Generator(device=dev).manual_seed(rank)) * (dcfg.dk ** -0.5)
    dout = torch.empty((dcfg.batch, dcfg.H, dcfg.dv), dtype=torch.bfloat16, device=dev)
    counter = [0]

    def dstep():
        i = counter[0]
        x = dq_s[i % n_tok]
        binding.decode_step(*x, states, t_all[i], out=dout)
        counter[0] += 1

    for _ in range(max(args.warmup, 3)):
        dstep()
    first = counter[0]
    d_ms_total = cuda_time(dstep, dsteps, stream)
    d_ms_total = max_over_ranks(d_ms_total, ws)
    assert binding.device_error() == 0
    dbytes = sum(decode_bytes(t_all_np[i], dcfg.H, dcfg.dk, dcfg.dv, dcfg.Lmax) for i in range(first, first + dsteps))

    return d_ms_total, dbytes, dsteps


def gdn_work(cfg: inputs.PrefillConfig) -> dict:
    """Algorithmic flops of one log-linear Gated DeltaNet prefill (the chunkwise algorithm, chunk
    C = min(chunk, 64)): per chunk the causal halves of Q K^T and K K^T, the two unit-triangular
    inverses (C^3/6 multiply-adds each), W, Q~ and the pseudo-values, the in-chunk attention
    matrix and its product with V, the chunk state; per Fenwick level read the node read
    (2 C dk dv) and its carry through the chunk (4 C dk dv)."""
    BH = cfg.B * cfg.H
    C = min(cfg.chunk, 64)
    N = cfg.T // C
    dk, dv = cfg.dk, cfg.dv
    tri = C * (C + 1) // 2
    chunk = (2 * tri * 2 * dk + 2 * C ** 3 // 3 + tri * 2 * (2 * dk + dv) + C ** 3 // 3 + tri * 2 * dv
             + 2 * C * dk * dv)
    reads = popcount_sum(N)
    flops = BH * (N * chunk + reads * 6 * C * dk * dv)
    esz = 2 if cfg.dtype == "bf16" else 4
    nbytes = BH * cfg.T * ((2 * dk + 2 * dv) * esz + 8 + cfg.L * 4)
    return dict(flops=flops, bytes=nbytes)


def gdn_device_inputs(cfg: inputs.PrefillConfig, dev, seed: int = 99):
    """One Gated DeltaNet prefill problem drawn on the device with the config's distributions
    (unit-norm q/k rows, beta = sigmoid(N(0,1))): q, k, v, log_a, beta, lambda, out."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    shp = (cfg.B, cfg.H, cfg.T)

    def unit(x):
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)

    q = unit(torch.randn(shp + (cfg.dk,), device=dev, generator=g))
    k = unit(torch.randn(shp + (cfg.dk,), device=dev, generator=g))
    v = torch.randn(shp + (cfg.dv,), device=dev, generator=g).to(torch.bfloat16)
    la = -torch.nn.functional.softplus(torch.randn(shp, device=dev, generator=g) + cfg.log_a_mu)
    bt = torch.sigmoid(torch.randn(shp, device=dev, generator=g))
    lam = torch.nn.functional.softplus(torch.randn(shp + (cfg.L,), device=dev, generator=g))
    out = torch.empty(shp + (cfg.dv,), dtype=torch.bfloat16, device=dev)
    return q, k, v, la, bt, lam, out


def bench_gdn(args, dev, stream, peaks) -> dict:
    """The log-linear Gated DeltaNet: prefill of the headline-shaped workload (B4 H16 T8192 dk128
    dv64, unit-norm q/k, beta = sigmoid(N(0,1))) and the decode step of the decode workload."""
    import torch
    from log_linear_attention_gb300 import binding
    cfg = inputs.GDN_CONFIGS["gdn-headline"]
    g = torch.Generator(device=dev)
    g.manual_seed(98)
    q, k, v, la, bt, lam, out = gdn_device_inputs(cfg, dev)

    def unit(x):
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)

    def step():
        binding.gdn_forward(q, k, v, la, bt, lam, cfg.chunk, out=out)

    step()
    n = 3
    ms = cuda_time(step, n, stream) / n
    per = {}
    for kname, kms in binding.gdn_forward_profile(q, k, v, la, bt, lam, cfg.chunk, out):
        per[kname] = per.get(kname, 0.0) + kms
    work = gdn_work(cfg)
    tfl = work["flops"] / (ms / 1e3) / 1e12
    tf32_peak = peaks["bf16_tflops"] / 2
    # decode: the decode workload's shapes and positions, random states
    dcfg = inputs.DECODE_CONFIG
    pos = torch.from_numpy(inputs.make_positions(dcfg, 0)).to(dev)
    states = torch.randn((dcfg.batch, dcfg.H, dcfg.Lmax, dcfg.dk, dcfg.dv), device=dev, generator=g) * dcfg.dk ** -0.5
    dq = torch.randn((dcfg.batch, dcfg.H, dcfg.dk), device=dev, generator=g).to(torch.bfloat16)
    dk_ = unit(torch.randn((dcfg.batch, dcfg.H, dcfg.dk), device=dev, generator=g))
    dv_ = torch.randn((dcfg.batch, dcfg.H, dcfg.dv), device=dev, generator=g).to(torch.bfloat16)
    dla = -torch.nn.functional.softplus(torch.randn((dcfg.batch, dcfg.H), device=dev, generator=g))
    dbt = torch.sigmoid(torch.randn((dcfg.batch, dcfg.H), device=dev, generator=g))
    dlam = torch.nn.functional.softplus(torch.randn((dcfg.batch, dcfg.H, dcfg.Lmax), device=dev, generator=g))
    dout = torch.empty((dcfg.batch, dcfg.H, dcfg.dv), dtype=torch.bfloat16, device=dev)
    t_np = pos.cpu().numpy()
    nsteps = 200
    ts = [pos + i for i in range(nsteps + 3)]

    counter = [0]

    def dstep():
        binding.gdn_decode_step(dq, dk_, dv_, dla, dbt, dlam, states, ts[counter[0]], out=dout)
        counter[0] += 1

    for _ in range(3):
        dstep()
    d_ms = cuda_time(dstep, nsteps, stream)
    dbytes = sum(decode_bytes(t_np + i, dcfg.H, dcfg.dk, dcfg.dv, dcfg.Lmax) + len(t_np) * dcfg.H * 4
                 for i in range(3, 3 + nsteps))
    assert binding.device_error() == 0
    d_gbs = dbytes / (d_ms / 1e3) / 1e9
    return {"prefill": {"workload": f"{cfg.name}: B={cfg.B} H={cfg.H} T={cfg.T} dk={cfg.dk} dv={cfg.dv} "
                                    f"chunk={cfg.chunk}, bf16 q/k/v (unit-norm q, k), fp32 log_a/beta/lambda",
                        "ms": ms, "tokens_per_s": cfg.tokens / (ms / 1e3), "algorithmic_gflop": work["flops"] / 1e9,
                        "kernels_ms": per,
                        "roofline": {"bound": "tensor", "achieved": tfl, "peak": tf32_peak, "unit": "TFLOP/s",
                                     "frac": tfl / tf32_peak,
                                     "peak_source": f"{peaks['source']} bf16 x 1/2 (tf32, the dtype of the level "
                                                    "pass's dominant MMA)",
                                     "hbm_frac_of_call": work["bytes"] / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]}},
            "decode": {"workload": "64 sequences x 16 heads, dk=128 dv=64, t ~ U[1,65536), fp32 states (18 slots)",
                       "steps": nsteps, "us_per_step": 1e3 * d_ms / nsteps, "gbs": d_gbs,
                       "frac_of_hbm": d_gbs / peaks["hbm_gbs"],
                       "convention": "eager: nonempty levels read once, held levels written once"}}


def bench_prefill_config(args, dev, stream, name, peaks) -> dict:
    """One more prefill workload of the stated configs (inputs drawn on the device with that
    config's distributions): time per call, throughput, and the roofline of its dominant
    kernel, measured the same way as the headline."""
    import torch
    from log_linear_attention_gb300 import binding
    cfg = inputs.PREFILL_CONFIGS[name]
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    shp = (cfg.B, cfg.H, cfg.T)

    def qk():
        x = torch.randn(shp + (cfg.dk,), device=dev, generator=g)
        x = x / x.norm(dim=-1, keepdim=True) if cfg.qk_unit_rows else x * cfg.dk ** -0.5
        return x.to(torch.bfloat16)

    q, k = qk(), qk()
    v = torch.randn(shp + (cfg.dv,), device=dev, generator=g).to(torch.bfloat16)
    la = -torch.nn.functional.softplus(torch.randn(shp, device=dev, generator=g) + cfg.log_a_mu)
    lam = torch.nn.functional.softplus(torch.randn(shp + (cfg.L,), device=dev, generator=g))
    out = torch.empty(shp + (cfg.dv,), dtype=torch.bfloat16, device=dev)

    def step():
        binding.forward(q, k, v, la, lam, cfg.chunk, out=out)

    for _ in range(max(args.warmup, 3)):
        step()
    n = max(5, min(args.steps, 30))
    ms = cuda_time(step, n, stream) / n
    per = {}
    for _ in range(max(3, min(args.steps, 10))):
        for kname, kms in binding.forward_profile(q, k, v, la, lam, cfg.chunk, out):
            per.setdefault(kname, []).append(kms)
    assert binding.device_error() == 0
    kavg = {kn: sum(x) / len(x) for kn, x in per.items()}
    top = max(kavg, key=kavg.get)
    kw = kernel_work(top, cfg)
    work = prefill_work(cfg)
    if kw["bound"] == "hbm":
        achieved, peak, unit = kw["bytes"] / (kavg[top] / 1e3) / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = kw["flops"] / (kavg[top] / 1e3) / 1e12, ALU_F32_TFLOPS, "TFLOP/s"
    return {"workload": f"{cfg.name} prefill: B={cfg.B} H={cfg.H} T={cfg.T} dk={cfg.dk} dv={cfg.dv} "
                        f"chunk={cfg.chunk}, bf16 q/k/v ({cfg.L} levels), inputs drawn on the device",
            "ms": ms, "tokens_per_s": cfg.tokens / (ms / 1e3),
            "tflops": work["flops"] / (ms / 1e3) / 1e12, "algorithmic_gflop": work["flops"] / 1e9,
            "frac_of_bf16_peak": work["flops"] / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
            "hbm_frac_of_call": work["bytes"] / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
            "roofline": {"kernel": top, "bound": kw["bound"], "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak, "kernel_ms": kavg[top]},
            "kernels_ms": kavg}


def run_lla(args, cfg):
    import torch
    from log_linear_attention_gb300 import binding

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    if args.mode == "gdn":
        # Gated DeltaNet prefill launches only (a short target for profilers)
        gcfg = inputs.GDN_CONFIGS["gdn-headline"]
        if args.batch:
            gcfg = dataclasses.replace(gcfg, B=args.batch)
        q, k, v, la, bt, lam, gout = gdn_device_inputs(gcfg, dev)
        gstep = lambda: binding.gdn_forward(q, k, v, la, bt, lam, gcfg.chunk, out=gout)  # noqa: E731
        for _ in range(max(args.warmup, 3)):
            gstep()
        g_ms = cuda_time(gstep, args.steps, stream) / args.steps
        assert binding.device_error() == 0
        if rank == 0:
            print(json.dumps({"mode": "gdn", "workload": f"{gcfg.name} B={gcfg.B}", "ms": g_ms, "steps": args.steps}))
        return 0
    if args.mode == "decode":
        # decode launches only (a short target for profilers); not the benchmark line
        d_ms_total, dbytes, dsteps = bench_decode(args, dev, stream, rank, ws)
        if rank == 0:
            print(json.dumps({"mode": "decode", "us_per_step": 1e3 * d_ms_total / dsteps,
                              "gbs": dbytes / (d_ms_total / 1e3) / 1e9, "steps": dsteps}))
        return 0

    # ---- inputs (per-rank seed: every rank runs the full workload: weak scaling)
    inp = inputs.make_prefill(cfg, seed=rank)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    host = [bf16(inp.bits["q"]), bf16(inp.bits["k"]), bf16(inp.bits["v"]),
            torch.from_numpy(inp.log_a), torch.from_numpy(inp.lam)]
    host = [h.pin_memory() for h in host]
    dq, dk_, dv_, da, dl = (h.to(dev) for h in host)
    out = torch.empty((cfg.B, cfg.H, cfg.T, cfg.dv), dtype=torch.bfloat16, device=dev)
    if args.mode == "backward":
        # backward launches only (a short target for profilers)
        gout = torch.randn((cfg.B, cfg.H, cfg.T, cfg.dv), device=dev).to(torch.bfloat16)
        for _ in range(max(args.warmup, 3)):
            binding.backward(dq, dk_, dv_, da, dl, gout, cfg.chunk)
        b_ms = cuda_time(lambda: binding.backward(dq, dk_, dv_, da, dl, gout, cfg.chunk), args.steps, stream) / args.steps
        assert binding.device_error() == 0
        if rank == 0:
            print(json.dumps({"mode": "backward", "config": cfg.name, "ms": b_ms, "steps": args.steps}))
        return 0
    if args.mode == "varlen":
        vl = bench_varlen(args, dev, stream, rank)
        if rank == 0:
            print(json.dumps({"mode": "varlen", **vl}))
        return 0
    if args.mode == "handoff":
        # prefill -> decode hand-off launches only (a short target for profilers)
        hstates = torch.empty((cfg.B, cfg.H, inputs.num_levels(cfg.T + 1), cfg.dk, cfg.dv), dtype=torch.float32,
                              device=dev)
        for _ in range(max(args.warmup, 3)):
            binding.prefill_state(dk_, dv_, da, hstates)
        h_ms = cuda_time(lambda: binding.prefill_state(dk_, dv_, da, hstates), args.steps, stream) / args.steps
        assert binding.device_error() == 0
        if rank == 0:
            print(json.dumps({"mode": "handoff", "config": cfg.name, "ms": h_ms, "steps": args.steps}))
        return 0
    work = prefill_work(cfg)

    def step():
        binding.forward(dq, dk_, dv_, da, dl, cfg.chunk, out=out)

    for _ in range(max(args.warmup, 3)):
        step()
    assert binding.device_error() == 0
    if args.mode == "prefill":
        # prefill launches only (a short target for profilers); not the benchmark line
        ms = cuda_time(step, args.steps, stream) / args.steps
        assert binding.device_error() == 0
        if rank == 0:
            print(json.dumps({"mode": "prefill", "config": cfg.name, "ms_per_step": ms, "steps": args.steps}))
        return 0

    clocks = ClockSampler(local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize()
    clocks.mark("start")
    ms_total = cuda_time(step, args.steps, stream)
    clocks.mark("end")
    clk = clocks.stop()
    ms_total = max_over_ranks(ms_total, ws)
    ms = ms_total / args.steps
    tokens_per_s = aggregate_tokens_per_s(cfg.tokens, ms, ws)
    tflops = work["flops"] / (ms / 1e3) / 1e12

    # ---- per-kernel device times (CUDA events recorded by the library between its launches)
    per_kernel = {}
    nprof = max(3, min(args.steps, 20))
    launches_per_step = 0
    for _ in range(nprof):
        rec = binding.forward_profile(dq, dk_, dv_, da, dl, cfg.chunk, out)
        launches_per_step = len(rec)
        for name, kms in rec:
            per_kernel.setdefault(name, []).append(kms)
    kavg = {n: sum(v) / len(v) for n, v in per_kernel.items()}
    top = max(kavg, key=kavg.get)
    kw = kernel_work(top, cfg)
    t_top = kavg[top] / 1e3
    if kw["bound"] == "hbm":
        achieved, peak, unit = kw["bytes"] / t_top / 1e9, peaks["hbm_gbs"], "GB/s"
    elif kw["bound"] == "tensor":
        achieved, peak, unit = kw["flops"] / t_top / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved, peak, unit = kw["flops"] / t_top / 1e12, ALU_F32_TFLOPS, "TFLOP/s"
    roofline = {"bound": kw["bound"], "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": traffic_record(top), "kernel": top, "kernel_ms": kavg[top],
                "algorithmic_bytes": kw["bytes"], "algorithmic_flops": kw["flops"],
                "peak_source": peaks["source"] if kw["bound"] != "alu" else "derived: 152 SM x 128 FMA x 2.07 GHz",
                "kernel_share": kavg[top] / sum(kavg.values()),
                "kernels_ms": kavg}

    # ---- end to end: pinned host buffers -> device -> lla_forward -> host, every step
    # the call's host output buffer is the caller's (lla_forward_host writes into it): pinned and
    # allocated once, as a serving caller holds it, so that no step pays a pinned allocation
    host_out = torch.empty((cfg.B, cfg.H, cfg.T, cfg.dv), dtype=torch.bfloat16, pin_memory=True)

    def e2e_step():
        return binding.forward(*host, cfg.chunk, out=host_out)

    e2e_step()
    torch.cuda.synchronize()
    n_e2e = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    ms_e2e = cuda_time(e2e_step, n_e2e, stream) / n_e2e
    wall_e2e = (time.perf_counter() - t0) / n_e2e * 1e3
    ms_e2e = max(ms_e2e, wall_e2e)
    ms_e2e = max_over_ranks(ms_e2e, ws)
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = out.numel() * out.element_size()

    # pinned host <-> device copy rates on this machine: the ceiling of the e2e number
    cbuf_h = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    cbuf_d = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(2):
        cbuf_d.copy_(cbuf_h, non_blocking=True)
        cbuf_h.copy_(cbuf_d, non_blocking=True)
    h2d_ms = cuda_time(lambda: cbuf_d.copy_(cbuf_h, non_blocking=True), 5, stream) / 5
    d2h_ms = cuda_time(lambda: cbuf_h.copy_(cbuf_d, non_blocking=True), 5, stream) / 5
    del cbuf_h, cbuf_d

    d_ms_total, dbytes, dsteps = bench_decode(args, dev, stream, rank, ws)
    d_gbs = ws * dbytes / (d_ms_total / 1e3) / 1e9
    sub = {name: bench_prefill_config(args, dev, stream, name, peaks) for name in ("small", "long")}
    gdn = bench_gdn(args, dev, stream, peaks)

    # ---- prefill -> decode hand-off: the state set after the whole prompt
    hL = inputs.num_levels(cfg.T + 1)
    hstates = torch.empty((cfg.B, cfg.H, hL, cfg.dk, cfg.dv), dtype=torch.float32, device=dev)

    def hstep():
        binding.prefill_state(dk_, dv_, da, hstates)

    for _ in range(3):
        hstep()
    n_h = max(3, min(args.steps, 20))
    h_ms = cuda_time(hstep, n_h, stream) / n_h
    held = 1 + bin(cfg.T - 1).count("1")

    # ---- backward: gradients of sum(dout * out) for the same problem
    gout = torch.randn((cfg.B, cfg.H, cfg.T, cfg.dv), device=dev).to(torch.bfloat16)

    def bstep():
        binding.backward(dq, dk_, dv_, da, dl, gout, cfg.chunk)

    for _ in range(3):
        bstep()
    n_b = max(3, min(args.steps, 10))
    b_ms = cuda_time(bstep, n_b, stream) / n_b
    assert binding.device_error() == 0
    bw = backward_work(cfg)
    vl = bench_varlen(args, dev, stream, rank)
    h_bytes = (cfg.B * cfg.H * cfg.T * ((cfg.dk + cfg.dv) * 2 + 4) + cfg.B * cfg.H * held * cfg.dk * cfg.dv * 4)

    line = None
    if rank == 0:
        # CPU baseline: the oracle as it stands, on the host cores, bounded sample
        cpu_val, cpu_sample, _ = oracle_tokens_per_s(cfg, inp, args.cpu_budget)
        cpu_all, cpu_threads, cpu_all_sample = oracle_tokens_per_s_all_cores(cfg, inp, args.cpu_budget)
        cpu = cpu_info()
        line = {
            "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{cfg.name} prefill: B={cfg.B} H={cfg.H} T={cfg.T} dk={cfg.dk} dv={cfg.dv} "
                                   f"chunk={cfg.chunk}, bf16 q/k/v, fp32 log_a/lambda ({cfg.L} levels)",
                       "global_batch": cfg.B * ws, "seq_len": cfg.T, "parallelism": f"heads-replicated x{ws}",
                       "l2": "inputs (434 MB) exceed L2; no flush"},
            "tflops": {"value": tflops, "algorithmic_gflop_per_step": work["flops"] / 1e9,
                       "frac_of_bf16_peak": tflops / peaks["bf16_tflops"], "peak_source": peaks["source"]},
            "hbm": {"min_bytes_per_step": work["bytes"], "gbs_at_min_bytes": work["bytes"] / (ms / 1e3) / 1e9,
                    "frac": work["bytes"] / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]},
            "roofline": roofline,
            "decode": {"workload": "64 sequences x 16 heads, dk=128 dv=64, t ~ U[1,65536), fp32 states (18 slots), "
                                   "bf16 q/k/v", "steps": dsteps, "us_per_step": 1e3 * d_ms_total / dsteps,
                       "gbs": d_gbs, "frac_of_hbm": d_gbs / peaks["hbm_gbs"],
                       "bytes_per_step": dbytes / dsteps, "convention": "eager: nonempty levels read once, "
                                                                         "held levels written once"},
            "handoff": {"workload": f"state set after the {cfg.T}-token prompt of every (b, h) (lla_prefill_state)",
                        "ms": h_ms, "gbs": h_bytes / (h_ms / 1e3) / 1e9,
                        "frac_of_hbm": h_bytes / (h_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                        "bytes": h_bytes, "convention": "k, v, log_a read once; held state slots written once"},
            "backward": {"workload": f"lla_backward of the same {cfg.name} problem (dq, dk, dv, dlog_a, dlambda)",
                         "ms": b_ms, "tokens_per_s": cfg.tokens / (b_ms / 1e3),
                         "tflops": bw["flops"] / (b_ms / 1e3) / 1e12,
                         "algorithmic_gflop": bw["flops"] / 1e9,
                         "frac_of_bf16_peak": bw["flops"] / (b_ms / 1e3) / 1e12 / peaks["bf16_tflops"],
                         "bound": "hbm", "algorithmic_bytes": bw["bytes"],
                         "gbs": bw["bytes"] / (b_ms / 1e3) / 1e9,
                         "frac_of_hbm": bw["bytes"] / (b_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                         "peak_source": peaks["source"]},
            "varlen": vl,
            "small": sub["small"],
            "long": sub["long"],
            "gdn": gdn,
            "e2e": {"value": ws * cfg.tokens / (ms_e2e / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                    "pinned_copy_gbs": {"h2d": (256 << 20) / (h2d_ms / 1e3) / 1e9,
                                        "d2h": (256 << 20) / (d2h_ms / 1e3) / 1e9},
                    "copy_bound_ms": h2d / ((256 << 20) / (h2d_ms / 1e3)) * 1e3},
            "cpu_baseline": {"value": cpu_val, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": cpu_sample, **cpu,
                             "all_cores": {"value": cpu_all, "unit": "tokens/s", "cores": cpu_threads,
                                           "sample": cpu_all_sample}},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "peaks": {k_: peaks[k_] for k_ in ("hbm_gbs", "bf16_tflops", "source")},
        }
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["lla", "reference"], default="lla")
    ap.add_argument("--config", default="headline", choices=sorted(inputs.PREFILL_CONFIGS))
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--mode", choices=["all", "prefill", "decode", "handoff", "backward", "varlen", "gdn"],
                    default="all",
                    help="prefill / decode / handoff / backward / varlen / gdn: run only that workload's launches "
                         "(profiling targets)")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling modes only: the config's shapes with this many sequences (a smaller case)")
    args = ap.parse_args()
    cfg = inputs.PREFILL_CONFIGS[args.config]
    if args.batch:
        if args.mode == "all":
            ap.error("--batch applies to the profiling modes only, not to the benchmark line")
        cfg = dataclasses.replace(cfg, B=args.batch)
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_lla(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
