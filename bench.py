"""Benchmark of the KDA serving hot path on GB300.

Prints ONE JSON line (rank 0).  Workload: the decode step (batch 64 requests, H=32, dk=dv=128, conv
width 4, fp32 states in a 4096-slot pool, a fresh random draw of 64 distinct slots every step, in place).
`value` = decode tokens/s over all ranks, with inputs resident in HBM; `e2e` = the same through the
C-ABI call with the step's token inputs copied from pinned host memory and y copied back inside the
timed region.  `prefill` adds the chunked-prefill workload (4 sequences of 2048/4096/8192/8192 tokens,
chunk 64, checkpoints every 128 tokens into pool slots) timed the same way.  `cpu_baseline` times the
fp64 oracle on this host's cores on a bounded sample of the decode workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Multi-GPU (weak scaling, one independent batch per rank, no collective on the data path):
  python -m torch.distributed.run --nproc-per-node N --master-addr 127.0.0.1 ... bench.py --gpus N
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import kda_inputs as ki  # noqa: E402

METRIC = "KDA decode tokens/s + state GB/s vs HBM peak; chunked-prefill tokens/s"
H, DK, DV, W = 32, 128, 128, 4
DEC_N, DEC_SLOTS = 64, 4096
PRE_LENS, PRE_CHUNK, PRE_INTERVAL = (2048, 4096, 8192, 8192), 64, 128
DECODE_BYTES_PER_HEAD_TOKEN = 2 * DK * DV * 4 + 2 * (W - 1) * (2 * DK + DV) * 2 + (3 * DK + DK + DV + DV) * 2 + 2
PREFILL_IO_BYTES_PER_HEAD_TOKEN = (2 * DK + DV + DK + DV + DV) * 2 + 2
CKPT_BYTES = DK * DV * 4 + (W - 1) * (2 * DK + DV) * 2


# ----------------------------------------------------------------------------- multi-rank plumbing
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    """Slowest rank's value (the whole job is as slow as its slowest rank)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def rank_seed(base: int, rank: int) -> int:
    """Each rank serves an independent batch (weak scaling)."""
    return base + 7919 * rank


# ----------------------------------------------------------------------------- peaks and clocks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0) or 0), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while a region runs."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + ",".join(self.FIELDS),
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def file_sha(*paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_values(name: str, sha: str) -> dict:
    """The key: value lines of profiles/<name>_traffic.txt when its kernel_source_sha matches `sha`, else {}."""
    path = os.path.join(ROOT, "profiles", f"{name}_traffic.txt")
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        return kv if kv.get("kernel_source_sha") == sha else {}
    except Exception:
        return {}


def profiled_traffic(name: str, sha: str):
    """dram bytes per launch recorded in profiles/<name>_traffic.txt for this exact kernel source, else None."""
    path = os.path.join(ROOT, "profiles", f"{name}_traffic.txt")
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha") == sha:
            return float(kv["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------- CPU oracle (baseline / reference)
class OracleDecodeSample:
    """One decode step of the fp64 oracle for a sample of n requests (all heads) of the decode workload."""

    def __init__(self, n: int, seed: int = 2):
        import oracle
        oracle.build()
        self.oracle, self.n = oracle, n
        self.cfg = oracle.Cfg(H=H, dk=DK, dv=DV, W=W)
        self.wts = ki.layer_weights(seed, H, DK, DV, W)
        tok = ki.token_inputs(seed, n, H, DK, DV)
        self.f = {k: ki.bf16_bits_to_f64(v) for k, v in tok.items()}
        S_h, C_h = ki.pool_tiles(seed, H, DK, DV, W, np.arange(n * H))
        self.S0 = S_h.reshape(n, H, DK, DV).astype(np.float64)
        self.C0 = ki.bf16_bits_to_f64(C_h).reshape(n, H, W - 1, 2 * DK + DV)
        self.cu, self.sp = np.arange(n + 1), np.zeros(n, dtype=np.int64)

    def step(self) -> float:
        f = self.f
        t0 = time.perf_counter()
        self.oracle.forward(self.cfg, self.cu, self.sp, f["q"], f["k"], f["v"], f["a"], f["b"], f["z"],
                            self.wts["conv_w"], self.wts["norm_w"], self.S0, self.C0)
        return time.perf_counter() - t0


def oracle_decode_rate(seconds: float, seed: int = 2) -> dict:
    """fp64 oracle on this host: repeated decode steps of 16 of the 64 requests, for about `seconds`."""
    smp = OracleDecodeSample(16, seed)
    reps, dt = 0, 0.0
    while dt < seconds:
        dt += smp.step()
        reps += 1
    return {"value": reps * smp.n / dt, "unit": "tokens/s", "cores": smp.oracle.num_threads(), "kind": "oracle",
            "sample": f"{reps} repetitions of one decode step for {smp.n} of the 64 requests (all {H} heads, "
                      f"dk=dv={DK}, 4096-slot pool contents), fp64, {dt:.1f} s"}


def run_reference(args):
    """The reference arm: the fp64 oracle as it stands, timed on this host's cores, each step one oracle
    decode call on a sample of the decode workload sized so that the whole run takes a few minutes."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    probe = OracleDecodeSample(16)
    t16 = min(probe.step() for _ in range(3))
    total = args.steps + args.warmup
    n = 16 if total * t16 <= 150.0 else max(1, int(16 * 150.0 / (total * t16)))
    smp = probe if n == 16 else OracleDecodeSample(n)
    for _ in range(args.warmup):
        smp.step()
    dt = sum(smp.step() for _ in range(args.steps))
    val = args.steps * n / dt
    sample = (f"each step: one fp64 oracle decode step for {n} of the 64 requests (all {H} heads, dk=dv={DK}); "
              f"{args.steps} steps in {dt:.1f} s")
    line = {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "decode step: batch 64 requests, H=32, dk=dv=128, conv width 4, 4096-slot "
                                   "pool (bounded sample per step, see cpu_baseline)"},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": smp.oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
def bf16_dev(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def run_gpu(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    import hybrid_linear_attention_decode_gb300 as kda
    try:
        kda.load_library()
    except RuntimeError:
        from hybrid_linear_attention_decode_gb300 import build as kbuild
        kbuild.build()
        kda.load_library()
    hbm_peak, _, _, peak_kind = measured_peaks()
    seed = rank_seed(2, rank)
    stream = torch.cuda.current_stream(dev)

    # ---- decode workload
    pool = kda.StatePool.empty(DEC_SLOTS, H, DK, DV, W, device=dev)
    ki.fill_device_pool(pool.S, pool.conv, seed)
    wts = ki.layer_weights(seed, H, DK, DV, W)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).to(dev), torch.from_numpy(wts["norm_w"]).to(dev))
    tok = ki.token_inputs(seed, DEC_N, H, DK, DV)
    d = {k: bf16_dev(v, dev) for k, v in tok.items()}
    y = torch.empty(DEC_N, H, DV, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    K, Wm = args.steps, args.warmup
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    nd = Wm + K
    slots = torch.rand(nd, DEC_SLOTS, device=dev, generator=g).argsort(dim=1)[:, :DEC_N].to(torch.int32).contiguous()

    def dec(i, st=stream):
        s = slots[i % nd]
        kda.kda_decode_step(pool, prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, s, s, status, st)

    for i in range(Wm):
        dec(i)
    torch.cuda.synchronize()
    # per-launch kernel time from events around eager launches (diagnostic)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
    for i, (a, b) in enumerate(ev):
        a.record(stream)
        dec(i)
        b.record(stream)
    torch.cuda.synchronize()
    eager_launch_ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
    # the timed region: one replay of a captured graph of exactly K decode steps (fresh slots per step)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(K):
            dec(Wm + i, None)
    graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    region_ms = start.elapsed_time(end)
    launch_ms = region_ms / K
    # keep the GPU busy (untimed) until the sampler has seen over a second of load
    while time.time() - t_wall0 < 1.5:
        graph.replay()
        torch.cuda.synchronize()
    t_wall2 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall2)
    del graph
    assert int(status.item()) == 0, f"decode status {int(status.item())}"
    region_ms = max_over_ranks(region_ms, ws)
    dec_tokens = DEC_N * ws
    value = dec_tokens * K / (region_ms / 1000.0)
    bytes_per_launch = DECODE_BYTES_PER_HEAD_TOKEN * DEC_N * H
    achieved = bytes_per_launch / (launch_ms / 1000.0) / 1e9
    state_gbs = 2 * DK * DV * 4 * DEC_N * H / (launch_ms / 1000.0) / 1e9
    dec_sha = file_sha("hybrid_linear_attention_decode_gb300/csrc/kda_decode.cu",
                       "hybrid_linear_attention_decode_gb300/csrc/kda_device.cuh")
    traffic = profiled_traffic("kda_decode", dec_sha)

    # ---- end to end through the C ABI: token inputs from pinned host memory, y back to the host.
    # Each step's token inputs sit in one pinned buffer (q|k|v|a|z|b, 16-byte aligned pieces) plus its slot
    # ids; the device side is double-buffered, so step i+1's inputs arrive (copy stream) while step i runs
    # and y of step i returns (output stream) while step i+1 runs.  A serving loop drives decode through
    # CUDA graphs (full-decode graphs), and so does this measurement: one graph of Ke pipelined steps,
    # replayed once inside the timed region.
    names = ["q", "k", "v", "a", "z", "b"]
    offs, total = {}, 0
    for nm in names:
        offs[nm] = total
        total += (tok[nm].size + 7) // 8 * 8
    host_pack = torch.empty(total, dtype=torch.int16).pin_memory()
    for nm in names:
        host_pack[offs[nm]:offs[nm] + tok[nm].size] = torch.from_numpy(
            np.ascontiguousarray(tok[nm]).reshape(-1).view(np.int16))
    dev_pack = [torch.empty(total, dtype=torch.int16, device=dev) for _ in range(2)]
    dviews = [{nm: dev_pack[j][offs[nm]:offs[nm] + tok[nm].size].view(torch.bfloat16).view(tok[nm].shape)
               for nm in names} for j in range(2)]
    host_slots = slots.cpu().pin_memory()
    dev_slot = [torch.empty(DEC_N, dtype=torch.int32, device=dev) for _ in range(2)]
    ydev = [torch.empty(DEC_N, H, DV, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    host_y = torch.empty(DEC_N, H, DV, dtype=torch.bfloat16).pin_memory()
    h2d = total * 2 + DEC_N * 4
    d2h = host_y.numel() * host_y.element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_steps(i0, n):
        cur = torch.cuda.current_stream(dev)
        s_in.wait_stream(cur)
        s_out.wait_stream(cur)
        ev_k, ev_o = [None] * n, [None] * n
        for i in range(n):
            jb = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_k[i - 2])  # the kernel that read this buffer is done
                dev_pack[jb].copy_(host_pack, non_blocking=True)
                dev_slot[jb].copy_(host_slots[(i0 + i) % nd], non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            cur.wait_event(ev_in)
            if i >= 2:
                cur.wait_event(ev_o[i - 2])  # y of this buffer has been copied out
            dv_ = dviews[jb]
            kda.kda_decode_step(pool, prm, dv_["q"], dv_["k"], dv_["v"], dv_["a"], dv_["b"], dv_["z"], ydev[jb],
                                dev_slot[jb], dev_slot[jb], status, None)
            ev_k[i] = torch.cuda.Event()
            ev_k[i].record(cur)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_k[i])
                host_y.copy_(ydev[jb], non_blocking=True)
                ev_o[i] = torch.cuda.Event()
                ev_o[i].record(s_out)
        cur.wait_stream(s_in)
        cur.wait_stream(s_out)

    e2e_steps(0, Wm)
    torch.cuda.synchronize()
    Ke = max(3, min(K, 500))
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph):
        e2e_steps(Wm, Ke)
    e2e_graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del e2e_graph
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    e2e_val = dec_tokens * Ke / (e2e_ms / 1000.0)

    # ---- the decode step at batch 64, 128 and 256: the fixed cost of a step
    decode_sweep = run_decode_sweep(args, kda, torch, dev, stream, pool, prm, seed, hbm_peak, ws)

    # ---- the same decode step on a bf16 state pool
    decode_bf16 = run_decode_bf16(args, kda, torch, dev, stream, prm, d, seed, hbm_peak, ws)

    # ---- speculative verification: 5 tokens per request, every position kept
    decode_multi = run_decode_multi(args, kda, torch, dev, stream, pool, prm, seed, hbm_peak, ws)

    # ---- the input projections feeding the prefill workload
    projection = run_project(args, kda, torch, dev, stream, seed, ws)

    # ---- the long-context workload (prefill of one 131072-token sequence, then decode at batch 256)
    long_context = run_long_context(args, kda, torch, dev, stream, pool, prm, seed, hbm_peak, ws)

    # ---- chunked prefill workload
    prefill = run_prefill(args, kda, torch, dev, stream, pool, prm, seed, hbm_peak, ws)

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": Wm,
            "ms_per_step": region_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp32", "data": "synthetic",
            "config": {"workload": "decode step: batch 64 requests, H=32, dk=dv=128, conv width 4, fp32 state "
                                   "pool of 4096 slots (8 GiB), 64 distinct random slots per step, in place",
                       "global_batch": DEC_N * ws, "per_gpu_batch": DEC_N, "heads": H, "dk": DK, "dv": DV,
                       "l2": "inputs larger than L2: every step draws fresh random slots from an 8 GiB pool",
                       "parallelism": f"replicas x{ws} (independent batches per GPU)"},
            "state_gbs": state_gbs,
            "roofline": {"bound": "hbm", "kernel": "kda_decode_kernel", "achieved": achieved, "peak": hbm_peak,
                         "unit": "GB/s", "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                         "traffic": traffic, "algorithmic_bytes_per_launch": bytes_per_launch,
                         "launch_ms": launch_ms, "eager_launch_ms_median": eager_launch_ms},
            "clocks": clocks,
            "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": Ke, "mode": "one CUDA-graph replay of the pipelined steps: per step the packed token "
                                         "inputs and slot ids copied from pinned host memory, the C-ABI decode "
                                         "call, y copied back to pinned host memory; copies of neighbouring "
                                         "steps overlap the kernel"},
            "gpu_launches": K,
            "decode_batch_sweep": decode_sweep,
            "decode_bf16_state": decode_bf16,
            "decode_multi_verify": decode_multi,
            "projection": projection,
            "prefill": prefill,
            "long_context": long_context}
    if rank == 0:
        if ws == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_decode_rate(args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


PROJ_HIDDEN = 4096  # hidden size of the synthetic layer whose projections feed the prefill workload


def run_project(args, kda, torch, dev, stream, seed, ws):
    """The six input projections of the prefill workload's 22528 tokens (hidden 4096 -> q, k, v, a, z, b for
    H = 32, d = 128: 20512 features) as one GEMM, against the measured dense bf16 peak."""
    T = int(sum(PRE_LENS))
    N = kda.projection_width(H, DK, DV)
    x_bits, w_bits = ki.projection_inputs(seed + 5, T, PROJ_HIDDEN, N)
    x = bf16_dev(x_bits, dev)
    w = bf16_dev(w_bits, dev)
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device=dev)  # noqa: E731
    q, k, v, a, z, b = e(T, H, DK), e(T, H, DK), e(T, H, DV), e(T, H, DK), e(T, H, DV), e(T, H)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def run():
        kda.kda_project_inputs(x, w, H, DK, DV, q, k, v, a, b, z, status, stream)

    K, Wm = max(3, min(args.steps, 20)), max(3, args.warmup)
    for _ in range(Wm):
        run()
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws) / K
    if int(status.item()) != 0:
        return {"error": f"device status {int(status.item())}"}
    flops = 2.0 * T * PROJ_HIDDEN * N
    tf = flops / (ms / 1000.0) / 1e12
    _, bf16_peak, _, kind = measured_peaks()
    return {"workload": f"input projections: {T} tokens x hidden {PROJ_HIDDEN} -> q, k, v, a, z, b for H=32, "
                        f"d=128 ({N} features) in one GEMM, bf16 in, fp32 accumulate, bf16 out",
            "tokens_per_s": T * ws / (ms / 1000.0), "ms_per_call": ms, "steps": K, "tflops": tf,
            "bf16_peak_tflops": bf16_peak, "peak_kind": kind, "tensor_frac": tf / bf16_peak}


def run_decode_sweep(args, kda, torch, dev, stream, pool, prm, seed, hbm_peak, ws):
    """The decode step at batch 64, 128 and 256 on the decode workload's pool (fresh random slots every step,
    one graph replay of K steps each), and a least-squares fit of time per step = fixed + per_item * items
    (items = batch x heads): the fixed part is what a step costs beyond streaming its items."""
    K = max(3, min(args.steps, 300))
    rows = []
    for N in (64, 128, 256):
        tok = ki.token_inputs(seed + 20, N, H, DK, DV)
        d = {k: bf16_dev(v, dev) for k, v in tok.items()}
        y = torch.empty(N, H, DV, dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed + N)
        sl = torch.rand(K + 3, DEC_SLOTS, device=dev, generator=g).argsort(dim=1)[:, :N].to(torch.int32).contiguous()

        def dec(i, st=stream):
            kda.kda_decode_step(pool, prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, sl[i], sl[i], status,
                                st)
        for i in range(3):
            dec(i)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for i in range(K):
                dec(3 + i, None)
        gr.replay()
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gr.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = max_over_ranks(e0.elapsed_time(e1), ws) / K * 1000.0
        del gr
        if int(status.item()) != 0:
            return {"error": f"device status {int(status.item())} at batch {N}"}
        rows.append((N, us))
    items = np.array([n * H for n, _ in rows], dtype=np.float64)
    t = np.array([u for _, u in rows])
    per_item, fixed = np.polyfit(items, t, 1)
    per_item_bytes = DECODE_BYTES_PER_HEAD_TOKEN
    return {"workload": "decode step at batch 64 / 128 / 256, H=32, dk=dv=128, fp32 pool of 4096 slots, fresh "
                        "random slots per step",
            "us_per_step": {str(n): u for n, u in rows},
            "hbm_frac": {str(n): per_item_bytes * n * H / (u / 1e6) / 1e9 / hbm_peak for n, u in rows},
            "fit": {"fixed_us": float(fixed), "per_item_ns": float(per_item * 1000.0),
                    "streaming_gbs": per_item_bytes / (per_item * 1e-6) / 1e9},
            "steps": K}


MULTI_L = 5  # verify step: 4 draft tokens + 1


def run_decode_multi(args, kda, torch, dev, stream, pool, prm, seed, hbm_peak, ws):
    """Speculative verification on the decode workload's fp32 pool: 64 requests x 5 tokens in one launch,
    the state after every position kept in its own slot; each step draws 64 + 320 fresh distinct slots."""
    L = MULTI_L
    tok = ki.token_inputs(seed + 3, DEC_N * L, H, DK, DV)
    d = {k: bf16_dev(v, dev) for k, v in tok.items()}
    y = torch.empty(DEC_N * L, H, DV, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    K, Wm = max(3, min(args.steps, 500)), args.warmup
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 3)
    draw = torch.rand(K + Wm, DEC_SLOTS, device=dev, generator=g).argsort(dim=1)[:, :DEC_N * (L + 1)]
    draw = draw.to(torch.int32)
    src = draw[:, :DEC_N].contiguous()
    dst = draw[:, DEC_N:].contiguous()

    def step(i, st=stream):
        kda.kda_decode_multi(pool, prm, L, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, src[i], dst[i], status,
                             st)

    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(K):
            step(Wm + i, None)
    graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws) / K
    del graph
    if int(status.item()) != 0:
        return {"error": f"device status {int(status.item())}"}
    # per (request, head): one state + window read, L state + window writes, L tokens of q,k,v,a,z,y,b
    per_item = (1 + L) * DK * DV * 4 + (1 + L) * (W - 1) * (2 * DK + DV) * 2 + L * ((3 * DK + DK + DV + DV) * 2 + 2)
    gbs = per_item * DEC_N * H / (ms / 1000.0) / 1e9
    return {"workload": "verify step: 64 requests x 5 tokens (4 draft + 1), H=32, dk=dv=128, fp32 pool of 4096 "
                        "slots, the state after every position kept in its own slot, fresh random slots per step",
            "tokens_per_s": DEC_N * L * ws / (ms / 1000.0), "ms_per_step": ms, "steps": K,
            "algorithmic_bytes_per_launch": per_item * DEC_N * H, "achieved_gbs": gbs, "hbm_frac": gbs / hbm_peak,
            "traffic": profiled_traffic("kda_decode_multi", file_sha(
                "hybrid_linear_attention_decode_gb300/csrc/kda_decode_multi.cu",
                "hybrid_linear_attention_decode_gb300/csrc/kda_device.cuh"))}


def run_decode_bf16(args, kda, torch, dev, stream, prm, d, seed, hbm_peak, ws):
    """The decode-step workload on a bf16 state pool (states stored in bf16, computed in fp32): 32 KiB of
    state per (request, head) instead of 64 KiB."""
    pool = kda.StatePool.empty(DEC_SLOTS, H, DK, DV, W, device=dev, state_dtype=torch.bfloat16)
    ki.fill_device_pool(pool.S, pool.conv, seed)
    K, Wm = max(3, min(args.steps, 1000)), args.warmup
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 1)
    slots = torch.rand(K + Wm, DEC_SLOTS, device=dev, generator=g).argsort(dim=1)[:, :DEC_N].to(torch.int32)
    slots = slots.contiguous()
    y = torch.empty(DEC_N, H, DV, dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def dec(i, st=stream):
        s_ = slots[i]
        kda.kda_decode_step(pool, prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, s_, s_, status, st)

    for i in range(Wm):
        dec(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(K):
            dec(Wm + i, None)
    graph.replay()
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws) / K
    del graph
    if int(status.item()) != 0:
        return {"error": f"device status {int(status.item())}"}
    per_ht = 2 * DK * DV * 2 + 2 * (W - 1) * (2 * DK + DV) * 2 + (3 * DK + DK + DV + DV) * 2 + 2
    gbs = per_ht * DEC_N * H / (ms / 1000.0) / 1e9
    sha = file_sha("hybrid_linear_attention_decode_gb300/csrc/kda_decode.cu",
                   "hybrid_linear_attention_decode_gb300/csrc/kda_device.cuh")
    return {"workload": "decode step as above on a bf16 state pool (4096 slots, 4 GiB)",
            "tokens_per_s": DEC_N * ws / (ms / 1000.0), "ms_per_step": ms, "steps": K,
            "algorithmic_bytes_per_launch": per_ht * DEC_N * H, "achieved_gbs": gbs, "hbm_frac": gbs / hbm_peak,
            "traffic": profiled_traffic("kda_decode_bf16", sha)}


LONG_T, LONG_INTERVAL, LONG_DEC_N = 131072, 32768, 256


def run_long_context(args, kda, torch, dev, stream, pool, prm, seed, hbm_peak, ws, prefill_only=False,
                     tokens=LONG_T):
    """The long-context workload: one 131072-token prefill (H=32, d=128, chunk 64, checkpoints every 32768
    tokens) into the pool, then a batch-256 decode step in which request 0 continues that sequence from its
    final state and 255 requests use other random slots.  Token inputs are drawn on the device (seeded torch
    generator, the distributions of the other workloads); 5 GB of them would be slow to draw on the host.
    prefill_only: two prefill calls and nothing else (the profile case)."""
    T, C, I = tokens, PRE_CHUNK, LONG_INTERVAL
    ns = int(pool.S.shape[0])
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 11)

    def draw(*shape, shift=0.0):
        return (torch.randn(*shape, generator=g, device=dev) + shift).to(torch.bfloat16)
    q, k, v, z = draw(T, H, DK), draw(T, H, DK), draw(T, H, DV), draw(T, H, DV)
    a, b = draw(T, H, DK, shift=3.0), draw(T, H)
    y = torch.empty(T, H, DV, dtype=torch.bfloat16, device=dev)
    perm = torch.randperm(ns, generator=g, device=dev).to(torch.int32)
    nck = T // I
    dst = perm[:1].contiguous()
    ck = perm[1:1 + nck].contiguous()
    i32 = lambda x: torch.tensor(x, dtype=torch.int32, device=dev)  # noqa: E731
    cu, offs, src = i32([0, T]), i32([0, nck]), i32([-1])
    sp = torch.zeros(1, dtype=torch.int64, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws_buf = torch.empty(kda.kda_prefill_workspace_bytes(pool, 1, T, C), dtype=torch.uint8, device=dev)

    def pre():
        kda.kda_prefill_chunked(pool, prm, cu, sp, src, dst, C, I, offs, ck, q, k, v, a, b, z, y, ws_buf, status,
                                stream)
    pre()
    torch.cuda.synchronize()
    barrier(ws)
    Kp = 1 if prefill_only else 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(Kp):
        pre()
    e1.record(stream)
    torch.cuda.synchronize()
    pre_ms = max_over_ranks(e0.elapsed_time(e1), ws) / Kp
    del ws_buf, q, k, v, a, z, b, y
    if prefill_only:
        return {"prefill_ms": pre_ms, "status": int(status.item())}
    # decode at batch 256: request 0 continues the long sequence (in place), the rest use other slots
    N = LONG_DEC_N
    others = perm[1 + nck:1 + nck + N - 1]
    slots = torch.cat([dst, others]).contiguous()
    dq, dk_, dv_, dz = draw(N, H, DK), draw(N, H, DK), draw(N, H, DV), draw(N, H, DV)
    da, db = draw(N, H, DK, shift=3.0), draw(N, H)
    yd = torch.empty(N, H, DV, dtype=torch.bfloat16, device=dev)
    Kd = 200

    def dec(st_=None):
        kda.kda_decode_step(pool, prm, dq, dk_, dv_, da, db, dz, yd, slots, slots, status, st_)
    for _ in range(3):
        dec(stream)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for _ in range(Kd):
            dec()
    gr.replay()
    torch.cuda.synchronize()
    barrier(ws)
    e0.record(stream)
    gr.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    dec_ms = max_over_ranks(e0.elapsed_time(e1), ws) / Kd
    del gr
    if int(status.item()) != 0:
        return {"error": f"device status {int(status.item())}"}
    dec_bytes = DECODE_BYTES_PER_HEAD_TOKEN * N * H
    pre_io = PREFILL_IO_BYTES_PER_HEAD_TOKEN * T * H + CKPT_BYTES * (nck + 1) * H
    return {"workload": f"long context: one {T}-token prefill (H=32, d=128, chunk 64, checkpoints every {I} "
                        f"tokens), then a batch-{N} decode step continuing it plus {N - 1} other slots",
            "prefill_ms": pre_ms, "prefill_tokens_per_s": T * ws / (pre_ms / 1000.0),
            "prefill_roofline": prefill_roofline(pre_ms, T * H, pre_io, "kda_prefill_long"),
            "decode_us": dec_ms * 1000.0, "decode_tokens_per_s": N * ws / (dec_ms / 1000.0),
            "decode_hbm_frac": dec_bytes / (dec_ms / 1000.0) / 1e9 / hbm_peak}


# Useful floating-point work of the chunked form per (token, head) at chunk C = 64, dk = dv = d = 128 (2 flops
# per multiply-add): the intra-chunk products A, Qk, W, U' and Qk U (5 x 2 C d), the state-side products W S,
# Q+ S and K~^T U (3 x 2 d^2), and the triangular inverse (2 C^2 / 3 per token).
PREFILL_FLOPS_PER_HEAD_TOKEN = 5 * 2 * PRE_CHUNK * DK + 3 * 2 * DK * DV + 2 * PRE_CHUNK ** 2 / 3
PREFILL_SOURCES = ("hybrid_linear_attention_decode_gb300/csrc/kda_prefill.cu",
                   "hybrid_linear_attention_decode_gb300/csrc/kda_device.cuh",
                   "hybrid_linear_attention_decode_gb300/csrc/kda_umma.cuh")


def prefill_roofline(ms: float, head_tokens: int, algorithmic_bytes: float, profile: str) -> dict:
    """Three views of one prefill call against the measured peaks: useful flops / bf16 peak, algorithmic bytes /
    HBM peak, and useful flops / the rate the byte roofline allows at this arithmetic intensity; plus the
    tensor-pipe activity and DRAM traffic of an ncu capture of the same kernels, when it matches them."""
    hbm_peak, bf16_peak, _, kind = measured_peaks()
    flops = PREFILL_FLOPS_PER_HEAD_TOKEN * head_tokens
    tflops = flops / (ms / 1000.0) / 1e12
    gbs = algorithmic_bytes / (ms / 1000.0) / 1e9
    intensity = flops / algorithmic_bytes
    attainable = min(bf16_peak, intensity * hbm_peak / 1000.0)
    prof = profiled_values(profile, file_sha(*PREFILL_SOURCES))
    num = lambda k: float(prof[k]) if k in prof else None  # noqa: E731
    return {"bound": "hbm" if intensity * hbm_peak / 1000.0 < bf16_peak else "tensor",
            "useful_flop_per_head_token": PREFILL_FLOPS_PER_HEAD_TOKEN, "useful_tflops": tflops,
            "useful_flop_frac": tflops / bf16_peak, "achieved_gbs": gbs, "byte_frac": gbs / hbm_peak,
            "flop_per_byte": intensity, "attainable_tflops": attainable, "attainable_frac": tflops / attainable,
            "tensor_pipe_frac": {k[len("tensor_pipe_frac_"):]: float(v) for k, v in prof.items()
                                 if k.startswith("tensor_pipe_frac_")} or None,
            "traffic": num("dram_bytes_per_call"), "peak_bf16_tflops": bf16_peak, "peak_hbm_gbs": hbm_peak,
            "peak_kind": kind}


def prefill_problem(seed: int, lens, chunk: int, interval: int, num_slots: int):
    """Token inputs, tables and slot plan of a varlen prefill from empty prefixes."""
    T = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sp = np.zeros(len(lens), dtype=np.int64)
    counts = [(l // interval) if interval else 0 for l in lens]
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    nck = int(offs[-1])
    perm = ki.permutation(seed, ki.STREAM["slots"] + 77, num_slots)
    dst = perm[:len(lens)].astype(np.int32)
    ck = perm[len(lens):len(lens) + nck].astype(np.int32)
    return T, cu, sp, dst, offs, ck


def run_prefill(args, kda, torch, dev, stream, pool, prm, seed, hbm_peak, ws):
    T, cu, sp, dst, offs, ck = prefill_problem(seed, PRE_LENS, PRE_CHUNK, PRE_INTERVAL, int(pool.S.shape[0]))
    tok = ki.token_inputs(seed + 1, T, H, DK, DV)
    d = {k: bf16_dev(v, dev) for k, v in tok.items()}
    y = torch.empty(T, H, DV, dtype=torch.bfloat16, device=dev)
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    cu_d, sp_d, dst_d, offs_d, ck_d = t(cu, 0), t(sp, 0), t(dst, 0), t(offs, 0), t(ck, 0)
    src_d = torch.full((len(PRE_LENS),), -1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    try:
        nbytes = kda.kda_prefill_workspace_bytes(pool, len(PRE_LENS), T, PRE_CHUNK)
        if nbytes == 0:
            return None
        ws_buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def pre():
            kda.kda_prefill_chunked(pool, prm, cu_d, sp_d, src_d, dst_d, PRE_CHUNK, PRE_INTERVAL, offs_d, ck_d,
                                    d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, ws_buf, status, stream)
        Kp, Wp = max(3, min(args.steps, 20)), max(3, args.warmup)
        for _ in range(Wp):
            pre()
        torch.cuda.synchronize()
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(Kp):
            pre()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), ws) / Kp
    except kda.KdaError as e:
        return {"error": str(e)}
    if int(status.item()) != 0:
        return {"error": f"device status {int(status.item())}"}
    io = PREFILL_IO_BYTES_PER_HEAD_TOKEN * T * H + CKPT_BYTES * int(offs[-1]) * H + len(PRE_LENS) * H * CKPT_BYTES
    return {"workload": "chunked prefill: 4 sequences of 2048/4096/8192/8192 tokens from empty prefixes, H=32, "
                        "dk=dv=128, chunk 64, checkpoints every 128 tokens (176 x 32 heads) into pool slots",
            "tokens_per_s": T * ws / (ms / 1000.0), "ms_per_call": ms, "steps": Kp,
            "status": int(status.item()),
            "hbm_frac_of_algorithmic_bytes": io / (ms / 1000.0) / 1e9 / hbm_peak,
            "algorithmic_bytes_per_call": io,
            "roofline": prefill_roofline(ms, T * H, io, "kda_prefill_varlen4")}


def run_profile_case(args):
    """Small case for ncu captures of one kernel: decode on a 768-slot pool (1.5 GiB fp32 or 0.8 GiB bf16
    states, larger than L2), batch 64, a fresh slot draw per launch; the 5-token verify step on the same
    pool; one prefill call of the benchmark's prefill workload; or two calls of the long-context prefill
    (one 131072-token sequence, launched in segments; for a launch list, not a multi-pass capture)."""
    import torch
    import hybrid_linear_attention_decode_gb300 as kda
    kda.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    seed = 2
    wts = ki.layer_weights(seed, H, DK, DV, W)
    prm = kda.LayerParams(torch.from_numpy(wts["conv_w"]).to(dev), torch.from_numpy(wts["norm_w"]).to(dev))
    if args.profile in ("decode", "decode_bf16"):
        slots_n = 768
        sdt = torch.bfloat16 if args.profile == "decode_bf16" else torch.float32
        pool = kda.StatePool.empty(slots_n, H, DK, DV, W, device=dev, state_dtype=sdt)
        ki.fill_device_pool(pool.S, pool.conv, seed)
        tok = ki.token_inputs(seed, DEC_N, H, DK, DV)
        d = {k: bf16_dev(v, dev) for k, v in tok.items()}
        y = torch.empty(DEC_N, H, DV, dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        n = args.warmup + args.steps
        slots = torch.rand(n, slots_n, device=dev, generator=g).argsort(dim=1)[:, :DEC_N].to(torch.int32).contiguous()
        for i in range(n):
            kda.kda_decode_step(pool, prm, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y, slots[i], slots[i],
                                status, stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        print(f"profile case {args.profile}: {n} launches")
    elif args.profile == "decode_multi":
        slots_n, L = 768, MULTI_L
        pool = kda.StatePool.empty(slots_n, H, DK, DV, W, device=dev)
        ki.fill_device_pool(pool.S, pool.conv, seed)
        tok = ki.token_inputs(seed, DEC_N * L, H, DK, DV)
        d = {k: bf16_dev(v, dev) for k, v in tok.items()}
        y = torch.empty(DEC_N * L, H, DV, dtype=torch.bfloat16, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        n = args.warmup + args.steps
        draw = torch.rand(n, slots_n, device=dev, generator=g).argsort(dim=1)[:, :DEC_N * (L + 1)].to(torch.int32)
        for i in range(n):
            kda.kda_decode_multi(pool, prm, L, d["q"], d["k"], d["v"], d["a"], d["b"], d["z"], y,
                                 draw[i, :DEC_N].contiguous(), draw[i, DEC_N:].contiguous(), status, stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        print(f"profile case decode_multi: {n} launches")
    elif args.profile == "project":
        r = run_project(argparse.Namespace(steps=args.steps, warmup=args.warmup), kda, torch, dev, stream, seed, 1)
        print(f"profile case project: {r}")
    elif args.profile in ("long_prefill", "long_prefill_small"):
        # the small case: one 32768-token sequence (512 chunks, launched in segments like the full one, one
        # checkpoint), for captures whose per-chunk traffic scales to the 131072-token workload
        pool = kda.StatePool.empty(16, H, DK, DV, W, device=dev)
        T = LONG_T if args.profile == "long_prefill" else LONG_T // 4
        r = run_long_context(args, kda, torch, dev, stream, pool, prm, seed, measured_peaks()[0], 1,
                             prefill_only=True, tokens=T)
        assert r["status"] == 0
        print(f"profile case {args.profile}: {r}")
    else:
        pool = kda.StatePool.empty(512, H, DK, DV, W, device=dev)
        r = run_prefill(argparse.Namespace(steps=1, warmup=args.warmup), kda, torch, dev, stream, pool, prm, seed,
                        measured_peaks()[0], 1)
        print(f"profile case prefill: {r}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", choices=["decode", "decode_bf16", "decode_multi", "project", "prefill",
                                              "long_prefill", "long_prefill_small"], default=None,
                    help="run a small case of one kernel for an ncu capture and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
