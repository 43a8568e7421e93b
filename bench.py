"""WKV7 forward + backward throughput on the RWKV-7 1.5B-shaped layer scan.

One step = the forward scan (y, s_final and checkpoints) plus the backward
(dr, dw, dk, dv, da, db, dS_init) over B=4, T=4096, H=32, N=64 with bf16
inputs and fp32 state and gradients, inputs resident in HBM. Prints one JSON
line. `--impl reference` times the CPU oracle on a bounded sample of the same
workload instead.

Multi-GPU (torchrun, one process per GPU): every rank scans its own batch of
the same shape (independent (b, h) problems, no data-path collective); the
slowest rank's time counts and `value` is the tokens of all ranks per second.
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

METRIC = "WKV7 fwd+bwd tokens/s (B·T) at 1.5B shape; achieved % of roofline"
FP32_LANES_PER_SM = 128  # Blackwell SM: 4 partitions x 32 FP32 lanes

# The backward call (wkv7_backward_bf16) launches two kernels: the carry chain and the
# per-chunk output pass. DRAM bytes (read + write) per token-head of the two together, from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum at T=1024, divided by B*T*H;
# traffic grows in proportion to T). It is valid only for the kernel sources it was taken on: a
# change to any of them makes the report carry null instead.
TRAFFIC = {
    "kernel": "wkv7_bwd4_carry_kernel + wkv7_bwd4_out_kernel (one wkv7_backward_bf16 call)",
    "sources": ("wkv7_bwd4.cu", "wkv7_common.cuh", "wkv7_scaled.cuh", "wkv7_mma.cuh", "wkv7_mma16.cuh",
                "wkv7_launch.h", "wkv7_decay.cuh", "wkv7_tmem.cuh"),
    "sha256": "899673a9c877216d7d4638a15cfe0470ba169a470784601a014ef8795cd281da",
    "bytes_per_token_head": (83.937280e6 + 28.293376e6 + 318.861312e6 + 161.522944e6) / 131072,
}


# The fp32 backward (wkv7_backward at N = 64, 16-step checkpoints) runs the carry chain and the
# per-chunk output pass in split bf16; their DRAM bytes per token-head from one ncu capture of the
# 8 x 1024 x 12 case (dram__bytes_read.sum + dram__bytes_write.sum / (B*T*H)), null once their
# sources change.
TRAFFIC_FP32 = {
    "kernel": "wkv7_bwd4_carry_kernel<float> + wkv7_bwd4_out_f32_kernel (one wkv7_backward call, fp32 inputs)",
    "sources": ("wkv7_bwd4.cu", "wkv7_bwd4_f32.cu", "wkv7_common.cuh", "wkv7_scaled.cuh", "wkv7_mma.cuh",
                "wkv7_mma16.cuh", "wkv7_launch.h", "wkv7_decay.cuh", "wkv7_tmem.cuh"),
    "sha256": "bdbcc5c26ae502ad4d5d4b1223b836964b52e925b2f3a7a2221892e6647700dd",
    "N": 64,
    "bytes_per_token_head": (125.889792e6 + 60.157952e6 + 377.625344e6 + 123.926272e6) / 98304,
}


def configs_bench_workload() -> str:
    from linear_rnn_state_gb300 import configs

    return configs.BENCH_WORKLOAD


def measured_traffic_fp32(token_heads: int, N: int):
    t = TRAFFIC_FP32
    if not t["sha256"] or N != t["N"] or sources_sha256(t["sources"]) != t["sha256"]:
        return None
    return t["bytes_per_token_head"] * token_heads


def sources_sha256(names) -> str:
    import hashlib

    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "linear_rnn_state_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(token_heads: int):
    """Per-launch DRAM bytes of the dominant kernel, or None if its sources changed since."""
    if not TRAFFIC["sha256"] or sources_sha256(TRAFFIC["sources"]) != TRAFFIC["sha256"]:
        return None
    return TRAFFIC["bytes_per_token_head"] * token_heads


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "sm_max_mhz": float(p.get("sm_max_mhz", 2070.0)),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "sm_max_mhz": 2070.0, "source": "fallback"}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_seed(rank: int) -> int:
    """Each rank scans its own batch: the generator is seeded with the rank."""
    return rank


def head_shard(B: int, H: int, rank: int, world: int):
    """The (b, h) heads rank `rank` of `world` owns when one batch of B x H
    heads is split across ranks: a contiguous run of the B*H heads in (b, h)
    order, as even as the division allows. Heads are independent (each runs
    its own scan and its own backward), so a split by (b, h) needs no
    exchange; this is the only split the path uses."""
    n = B * H
    lo, hi = rank * n // world, (rank + 1) * n // world
    return [(i // H, i % H) for i in range(lo, hi)]


def reduce_max(value: float, dist, device=None) -> float:
    """Slowest rank's value (max over ranks); identity on one process."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def allreduce_param_grad(t, dist):
    """Sum of a parameter gradient over ranks (in place); identity on one
    process. The RWKV-8 decay is one parameter shared by every batch row, so
    ranks that shard the batch add their ddecay: the path's one exchange."""
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return t


def aggregate_tokens_per_s(world: int, B: int, T: int, ms_per_step: float) -> float:
    """Tokens of all ranks (each B*T per step) per second of the slowest rank."""
    return world * B * T / (ms_per_step * 1e-3)


def _init_pg(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist if world > 1 else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, path: str | None = None):
        """`path`: where the raw samples go ("{rank}" is replaced by the device
        index); a temporary file when None."""
        self.dev = device_index
        self.proc = None
        if path:
            self.path = path.replace("{rank}", str(device_index))
        else:
            fd, self.path = tempfile.mkstemp(prefix=f"clocks_rank{device_index}_", suffix=".csv")
            os.close(fd)

    def __enter__(self):
        try:
            if os.path.dirname(self.path):
                os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.dev)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _work_per_token_head(N, C, in_bytes):
    """Algorithmic FLOP and bytes per token-head (fwd, bwd).

    FLOP: 4 N^2 multiply-adds forward (sa, v k^T, sa b^T, y) and 12 N^2
    backward, each counted as 2 FLOP. Bytes: forward reads r, w, k, v, a, b
    and writes y and 1/C of a checkpoint; backward reads r, w, k, v, a, b,
    dy and 1/C of a checkpoint and writes six fp32 gradients.
    """
    f_flop, b_flop = 8 * N * N, 24 * N * N
    ck = 4 * N * N / C
    f_bytes = 7 * N * in_bytes + ck
    b_bytes = 7 * N * in_bytes + ck + 6 * N * 4
    return f_flop, b_flop, f_bytes, b_bytes


# Host memory the timed oracle sample may hold: its backward keeps every state of a
# head (T N^2 doubles) while it walks back, one head per thread.
ORACLE_SAMPLE_BYTES = 16e9


def cpu_sample_heads(wl, cores):
    """How many (b, h) heads the timed oracle sample takes: every head, unless
    their state histories would not fit the host-memory budget (the 65536-step
    workload), then as many as fit, at most one per core."""
    per_head = wl.T * wl.N * wl.N * 8
    fit = max(1, int(ORACLE_SAMPLE_BYTES // per_head))
    return wl.B * wl.H if fit >= min(wl.B * wl.H, cores) else min(fit, cores)


def cpu_baseline_sample(wl, d, heads, nthreads=0):
    """Time the oracle (fwd + bwd, fp64) on the first `heads` (b, h) heads of
    the workload, each over its whole sequence, on every host core (at most
    one thread per head)."""
    import numpy as np

    import oracle
    from linear_rnn_state_gb300 import inputs

    P = min(wl.B * wl.H, heads)
    cores = min(nthreads or len(os.sched_getaffinity(0)), P)
    heads = [(i // wl.H, i % wl.H) for i in range(P)]
    o = {n: inputs.as_f64(d[n], wl.storage) for n in ("r", "w", "k", "v", "a", "b", "dy")}
    sel = {n: np.stack([o[n][bi, :, hi, :] for bi, hi in heads])[:, :, None, :] for n in o}
    t0 = time.perf_counter()
    oracle.forward(*(sel[n] for n in ("r", "w", "k", "v", "a", "b")), nthreads=cores)
    oracle.backward(*(sel[n] for n in ("r", "w", "k", "v", "a", "b", "dy")), nthreads=cores)
    dt = time.perf_counter() - t0
    tokens = wl.T * P / wl.H  # one head is 1/H of a batch row's tokens
    return tokens / dt, cores, P, dt


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    from linear_rnn_state_gb300 import configs, inputs

    wl = configs.WORKLOADS[args.shape]
    d = inputs.generate(wl.B, wl.T, wl.H, wl.N, wl.storage, wl.s_init_std, seed=0)
    # each step: the whole workload (every (b, h) head over its full sequence), or on the
    # 65536-step workload the heads whose state histories fit the host-memory budget
    P = cpu_sample_heads(wl, len(os.sched_getaffinity(0)))
    for _ in range(args.warmup):
        cpu_baseline_sample(wl, d, P)
    times, toks = [], 0.0
    for _ in range(args.steps):
        v, used, P, dt = cpu_baseline_sample(wl, d, P)
        times.append(dt)
        toks += wl.T * P / wl.H
    value = toks / sum(times)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "H": wl.H, "N": wl.N, "storage": wl.storage},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": f"{P} of {wl.B * wl.H} (b,h) heads, full T={wl.T}, fwd+bwd in fp64 per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import numpy as np
    import torch

    from linear_rnn_state_gb300 import configs, inputs, wkv7

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = _init_pg(world, "nccl")
    wkv7.load()
    dev = torch.device("cuda", local)
    wl = configs.WORKLOADS[args.shape]
    B, T, H, N = wl.B, wl.T, wl.H, wl.N
    if args.T:  # shorter sequence of the same layer shape, for profiler captures
        T = args.T
    bf16 = wl.storage == "bf16"
    if args.workload != "wkv7" and not bf16:
        raise RuntimeError(f"--workload {args.workload} runs on bf16 inputs only")
    # bf16 at N = 64: the chunked kernels' 16-step checkpoints; fp32: the workload's interval
    C = wkv7.wkv7_default_ckpt_every(N, bf16) if bf16 else wl.ckpt_every
    names = ("r", "w", "k", "v", "a", "b", "dy")
    d = inputs.generate(B, T, H, N, wl.storage, wl.s_init_std, seed=shard_seed(rank))
    logit = args.workload == "wkv7-logit"  # the decay given as logits z, w formed in the kernels
    if logit:
        d["w"] = inputs.generate_logits(B, T, H, N, wl.storage, seed=shard_seed(rank))

    def to_dev(x):
        t = torch.from_numpy(x)
        return (t.view(torch.bfloat16) if bf16 else t).to(dev)

    t_in = {n: to_dev(d[n]) for n in names}
    tdt = torch.bfloat16 if bf16 else torch.float32
    y = torch.empty((B, T, H, N), dtype=tdt, device=dev)
    s_final = torch.empty((B, H, N, N), dtype=torch.float32, device=dev)
    nck = (T + C - 1) // C
    ckpt = torch.empty((B, H, nck, N, N), dtype=torch.float32, device=dev)
    grads = {n: torch.empty((B, T, H, N), dtype=torch.float32, device=dev) for n in ("dr", "dw", "dk", "dv", "da", "db")}
    dS = torch.empty((B, H, N, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    fwd = wkv7.wkv7_forward_bf16 if bf16 else wkv7.wkv7_forward
    bwd = wkv7.wkv7_backward_bf16 if bf16 else wkv7.wkv7_backward
    if logit:
        if not (bf16 and N == 64 and C == 16):
            raise RuntimeError("the decay-logit workload needs bf16 inputs, N = 64 and 16-step checkpoints")
        fwd, bwd = wkv7.wkv7_forward_logit_bf16, wkv7.wkv7_backward_logit_bf16
    epilogue = args.workload == "wkv7-epilogue"
    if epilogue:
        # the forward with the group-norm + bonus epilogue fused (out, nv and stats written) and
        # its backward (the group-norm gradient pass, the scan's backward, the bonus terms)
        rng = np.random.default_rng(0)
        epi_p = [torch.from_numpy(x.astype(np.float32)).to(dev) for x in (
            rng.uniform(0.5, 1.5, (H, N)), 0.1 * rng.standard_normal((H, N)), 0.5 * rng.standard_normal((H, N)))]
        nv = torch.empty_like(y)
        stats = torch.empty((B, T, H, 2), dtype=torch.float32, device=dev)
        pgrads = [torch.empty((H, N), dtype=torch.float32, device=dev) for _ in range(3)]
        fwd, bwd = wkv7.wkv7_forward_epilogue_bf16, wkv7.wkv7_backward_epilogue_bf16

    def build_args(tin, yb, gb, dSb):
        """The forward's and backward's C arguments on one set of input and
        output buffers (the checkpoints, s_final and the epilogue's nv and
        stats are written and read within a step, so every set shares them)."""
        g6 = [gb[n].data_ptr() for n in ("dr", "dw", "dk", "dv", "da", "db")]
        if epilogue:
            fa = [tin[n].data_ptr() for n in names[:6]] + [None] + [x.data_ptr() for x in epi_p] + [
                yb.data_ptr(), nv.data_ptr(), stats.data_ptr(), s_final.data_ptr(), ckpt.data_ptr(), C, 0, B, T, H,
                N, sp]
            ba = [tin[n].data_ptr() for n in names] + [nv.data_ptr(), stats.data_ptr(), epi_p[0].data_ptr(),
                                                       epi_p[2].data_ptr(), None, None, ckpt.data_ptr(), C, 0] + g6 + [
                dSb.data_ptr()] + [x.data_ptr() for x in pgrads] + [B, T, H, N, sp]
            return fa, ba
        fa = [tin[n].data_ptr() for n in names[:6]] + [None, yb.data_ptr(), s_final.data_ptr(), ckpt.data_ptr(),
                                                       C, B, T, H, N, sp]
        ba = [tin[n].data_ptr() for n in names] + [None, ckpt.data_ptr(), C] + g6 + [dSb.data_ptr(), B, T, H, N, sp]
        if logit:
            ba = ba[:8] + [None] + ba[8:]  # dS_final: none
        return fa, ba

    fwd_args, bwd_args = build_args(t_in, y, grads, dS)

    def step(ev=None, fa=None, ba=None):
        if ev is not None:
            ev[0].record(stream)
        rc = fwd(*(fa or fwd_args))
        if ev is not None:
            ev[1].record(stream)
        rc2 = bwd(*(ba or bwd_args))
        if ev is not None:
            ev[2].record(stream)
        if rc or rc2:
            raise RuntimeError(wkv7.last_error())

    for _ in range(args.warmup):
        step()
    wkv7.status()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local, args.clock_csv) as clocks:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(args.steps):
            step(events[k])
        end.record(stream)
        torch.cuda.synchronize()
    wkv7.status()
    if dist:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in events)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in events)
    ms = reduce_max(total_ms / args.steps, dist, dev)

    if args.no_e2e:
        e2e_ms = None
    else:
        e2e_ms = _e2e(args, d, names, t_in, grads, y, dS, step, build_args, stream, dist, dev)
    if rank != 0:
        return 0
    return _report(args, wl, world, B, T, H, N, C, bf16, ms, fwd_ms, bwd_ms, e2e_ms, ckpt, d, clocks, dev)


def _pipelined_e2e(args, host_in, sets, step_on, stream, dist, dev):
    """End-to-end steps through the C ABI with pinned host buffers: every step
    copies its inputs in, runs forward + backward and copies every output
    back. `sets` holds two (device inputs, device outputs) buffer sets keyed
    like `host_in`; `step_on(i)` enqueues one step on set i. Steps alternate
    between the sets: step k's host-to-device copies (one copy stream)
    overlap step k-1's compute, and its device-to-host copies (another
    stream) overlap step k+1's, ordered by events so that no buffer is
    rewritten before it has been read. Returns (ms per step, bytes in, bytes
    out per step)."""
    import torch

    host_out = {n: torch.empty(x.shape, dtype=x.dtype).pin_memory() for n, x in sets[0][1].items()}
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in host_out.values())
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    n_steps = max(2, min(args.steps, 20))

    def run(k, ev_in, ev_done, ev_out):
        dev_in, dev_out = sets[k % 2]
        if k >= 2:
            s_in.wait_event(ev_done[k - 2])  # step k-2 has read this set's inputs
        with torch.cuda.stream(s_in):
            for n, src in host_in.items():
                dst = dev_in[n]
                if dst.dtype != src.dtype:  # bf16 buffers take the raw 16-bit host words
                    dst, src = dst.view(torch.int16), src.view(torch.int16)
                dst.copy_(src, non_blocking=True)
        ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if k >= 2:
            stream.wait_event(ev_out[k - 2])  # step k-2's outputs have left this set
        step_on(k % 2)
        ev_done[k].record(stream)
        s_out.wait_event(ev_done[k])
        with torch.cuda.stream(s_out):
            for n, x in dev_out.items():
                host_out[n].copy_(x, non_blocking=True)
        ev_out[k].record(s_out)

    def events(n):
        return [torch.cuda.Event() for _ in range(n)]

    run(0, *(events(1) for _ in range(3)))  # warm-up of the copy paths
    torch.cuda.synchronize()
    ev_in, ev_done, ev_out = events(n_steps), events(n_steps), events(n_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for k in range(n_steps):
        run(k, ev_in, ev_done, ev_out)
    s_in.wait_event(ev_out[n_steps - 1])
    e1.record(s_in)
    torch.cuda.synchronize()
    return reduce_max(e0.elapsed_time(e1) / n_steps, dist, dev), h2d, d2h


def _e2e(args, d, names, t_in, grads, y, dS, step, build_args, stream, dist, dev):
    """The WKV7 step end to end (see _pipelined_e2e): inputs in, every gradient,
    y and dS_init out."""
    import torch

    host_in = {n: torch.from_numpy(d[n]).pin_memory() for n in names}
    t1 = {n: torch.empty_like(t_in[n]) for n in names}
    g1 = {n: torch.empty_like(grads[n]) for n in grads}
    y1, dS1 = torch.empty_like(y), torch.empty_like(dS)
    sets = [(t_in, {**grads, "y": y, "dS_init": dS}), (t1, {**g1, "y": y1, "dS_init": dS1})]
    set_args = [build_args(t_in, y, grads, dS), build_args(t1, y1, g1, dS1)]
    return _pipelined_e2e(args, host_in, sets, lambda i: step(fa=set_args[i][0], ba=set_args[i][1]), stream, dist,
                          dev)


def _report(args, wl, world, B, T, H, N, C, bf16, ms, fwd_ms, bwd_ms, e2e, ckpt, d, clocks, dev):
    import torch

    peaks = _peaks()
    BTH = B * T * H
    f_flop, b_flop, f_bytes, b_bytes = _work_per_token_head(N, C, 2 if bf16 else 4)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_flops = sms * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6
    achieved = b_flop * BTH / (bwd_ms * 1e-3)
    t_roof = max((f_flop + b_flop) * BTH / peak_flops, (f_bytes + b_bytes) * BTH / (peaks["hbm_gbs"] * 1e9))
    value = aggregate_tokens_per_s(world, B, T, ms)
    with_cpu = not args.no_cpu_baseline and T == wl.T and args.workload == "wkv7"  # the plain scan's oracle
    cpu_v, cpu_cores, cpu_P, cpu_dt = cpu_baseline_sample(
        wl, d, cpu_sample_heads(wl, len(os.sched_getaffinity(0)))) if with_cpu else (None, 0, 0, 0.0)
    chunked = bf16 and N == 64
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if (bf16 and N == 64) else "f32", "data": "synthetic",
        "arithmetic": ("tensor-core products with fp32 accumulation: bf16 operands in the forward (the fp32 state "
                       "rounded to bf16 where it enters a product; the state update's scaled k and b as bf16 hi + lo "
                       "pairs), bf16 operands in the backward's carry chain (the fp32 carry rounded to bf16 where it "
                       "enters a product) and in its per-chunk gradient products (the carry "
                       "stored as bf16 between the two backward kernels, the fp32 checkpoint rounded to bf16 "
                       "there); fp32 accumulation, state and element-wise math" if chunked else
                       ("tensor-core products in split bf16 (each operand a bf16 hi + lo pair, three products per "
                        "fp32 product, fp32 accumulation) in the forward, the backward's carry chain and its "
                        "per-chunk output pass; the state, the carried gradient (stored as fp32 between the two "
                        "backward kernels) and every element-wise step fp32"
                        if N == 64 and C == 16 else "fp32 FMA throughout (scalar kernels)"))
                      + "; inputs, dy and y stored in " + wl.storage,
        "config": {"workload": (wl.name + {"wkv7-logit": "-decay-logits", "wkv7-epilogue": "-with-epilogue"}.get(
                       args.workload, ""))
                   if T == wl.T else f"{wl.name} (T={T})", "B": B, "T": T, "H": H, "N": N, "storage": wl.storage, "ckpt_every": C,
                   "l2": "no flush: inputs, checkpoints and gradients (%.1f GB) exceed the 129 MB L2"
                         % ((7 * BTH * N * (2 if bf16 else 4) + ckpt.numel() * 4 + 6 * BTH * N * 4) / 1e9)},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "step_roofline_frac": t_roof / (ms * 1e-3),
        "roofline": {"bound": "alu", "achieved": achieved / 1e12, "peak": peak_flops / 1e12, "unit": "TFLOP/s",
                     "frac": achieved / peak_flops,
                     "traffic": measured_traffic(BTH) if chunked else measured_traffic_fp32(BTH, N) if C == 16 else None,
                     "kernel": TRAFFIC["kernel"] if chunked else TRAFFIC_FP32["kernel"] if N == 64 and C == 16
                     else "wkv7_bwd2_kernel (one wkv7_backward call)",
                     "note": ("the backward call (its two kernels, timed together with CUDA events around the "
                              "call): algorithmic FLOP of the recurrence (24 N^2 per token-head) against the FP32 "
                              "CUDA-core peak, the roofline the metric names; the kernels form them as tensor-core "
                              "products with bf16 operands") if chunked else
                             ("the backward call (its two kernels, timed together with CUDA events around the call): "
                              "algorithmic FLOP of the recurrence (24 N^2 per token-head) against the FP32 CUDA-core "
                              "peak; the kernels form them as split-bf16 tensor-core products")
                             if N == 64 and C == 16 else
                             ("the backward call (one kernel, timed with CUDA events around the call): algorithmic "
                              "FLOP of the recurrence (24 N^2 per token-head) against the FP32 CUDA-core peak"),
                     "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz",
                     "hbm_gbs_achieved": b_bytes * BTH / (bwd_ms * 1e-3) / 1e9, "hbm_peak_gbs": peaks["hbm_gbs"]},
        "e2e": None if e2e is None else {
            "value": aggregate_tokens_per_s(world, B, T, e2e[0]), "unit": "tokens/s", "h2d_bytes_per_step": e2e[1],
            "d2h_bytes_per_step": e2e[2]},
        # bf16 at N = 64: forward, carry chain, output pass (+ the epilogue's parameter sum); fp32 at
        # N = 64 with 16-step checkpoints the same three; otherwise the scalar forward and backward
        "gpu_launches": (4 if args.workload == "wkv7-epilogue" else 3 if N == 64 and C == 16 else 2) * args.steps,
        "clocks": clocks.summary(),
    }
    if args.workload == "wkv7-epilogue":
        line["note"] = ("forward with the group-norm + bonus epilogue fused (out, normalized y and per-row stats "
                        "written in the place of y); backward with the epilogue's gradient fused into the scan's "
                        "split backward (dy formed where the carry and output kernels read it, the bonus terms "
                        "added to the output pass's stores) plus one small kernel summing the parameters' terms")
    elif args.workload == "wkv7-logit":
        line["note"] = "the decay given as logits z and formed inside the scan kernels; dz returned in the place of dw"
    if wl.name != configs_bench_workload():
        line["note"] = (f"the {wl.name} workload (B={B}, T={T}, H={H}, N={N}, {wl.storage}); the metric's own "
                        "workload is the default run")
    if cpu_v is not None:
        line["cpu_baseline"] = {"value": cpu_v, "unit": "tokens/s", "cores": cpu_cores, "kind": "oracle",
                                "sample": f"{cpu_P} of {B * H} (b,h) heads, full T={T}, fwd+bwd fp64 ({cpu_dt:.1f} s)"}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ RWKV-8 ---
# `--workload rwkv8`: the RWKV-8 normalized recurrence (include/rwkv8.h), fp32,
# B=4, T=4096, H=32 heads of L = E = 64 with one value row per head. The pages
# give no sizes for it; this reuses the RWKV-7 layer's B, T, H and head size.

RWKV8_METRIC = "RWKV-8 normalized recurrence fwd+bwd tokens/s (B·T), B=4 T=4096 H=32 L=E=64 fp32; achieved % of roofline"
RWKV8_SHAPE = {"B": 4, "T": 4096, "H": 32, "Hv": 32, "L": 64, "E": 64}

# DRAM bytes per token-head of one rwkv8_backward call (its kernel; the ddecay sum moves 32 KB), from one
# ncu capture at T=1024 (dram__bytes_read.sum + dram__bytes_write.sum / (B*T*H)); null once the
# kernel sources change.
RWKV8_TRAFFIC = {
    "kernel": "rwkv8_bwd_kernel (one rwkv8_backward call)",
    "sources": ("rwkv8_bwd.cu", "rwkv8_launch.h"),
    "sha256": "b03718f14002a3d822decece8bbc3a53d86c81c7b71b6f81396feef18a60800f",
    "bytes_per_token_head": (237.082624e6 + 46.064896e6) / 131072,
}


def _rwkv8_env(name):
    return os.environ.get(name, "").startswith("1")


def _rwkv8_work_per_token_head(L, E, C=16):
    """Algorithmic FLOP and bytes per token-head (fwd, bwd) of the RWKV-8
    recurrence, from its step-by-step definition: forward 3 L E multiply-adds
    (readout, decay, q v^T), backward 6 L E (carry decay, U dy^T, <rho, dy>,
    G v, G^T q, G . rho), each 2 FLOP. Bytes: forward reads q, v and writes y
    and 1/C of a checkpoint (rho and rho_norm); backward reads q, v, dy and
    the checkpoint share and writes dq and dv (fp32 throughout)."""
    ck = 4 * (L * E + L) / C
    return 6 * L * E, 12 * L * E, 4 * (L + 2 * E) + ck, 4 * (L + 2 * E) + ck + 4 * (L + E)


def _rwkv8_oracle_sample(d, heads, T):
    """Time the RWKV-8 oracle (fwd + bwd, fp64) on the first `heads` heads of
    batch row 0, each over the whole sequence."""
    import importlib.util

    import numpy as np

    spec = importlib.util.spec_from_file_location("rwkv8_oracle", os.path.join(ROOT, "oracle", "rwkv8_oracle.py"))
    orc = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(orc)
    sl = (slice(0, 1), slice(0, heads))
    o = {k: d[k][sl].astype(np.float64) for k in ("q", "v", "dy")}
    dec = d["decay"][:heads].astype(np.float64)
    t0 = time.perf_counter()
    orc.forward(o["q"], o["v"], dec)
    orc.backward(o["q"], o["v"], dec, o["dy"])
    dt = time.perf_counter() - t0
    return T * heads / RWKV8_SHAPE["H"] / dt, dt


def run_rwkv8(args):
    world, rank, local = _dist()
    if args.impl == "reference":
        if rank != 0:
            return 0
        from linear_rnn_state_gb300 import inputs

        sh = RWKV8_SHAPE
        d = inputs.generate_rwkv8(1, sh["T"], sh["H"], sh["Hv"], sh["L"], sh["E"], "f32", seed=0)
        heads = 8
        for _ in range(args.warmup):
            _rwkv8_oracle_sample(d, heads, sh["T"])
        times = [_rwkv8_oracle_sample(d, heads, sh["T"])[1] for _ in range(args.steps)]
        value = sh["T"] * heads / sh["H"] * len(times) / sum(times)
        line = {
            "metric": RWKV8_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "rwkv8-4x4096x32-l64e64-f32", **sh},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{heads} of {sh['B'] * sh['H']} heads, full T={sh['T']}, fwd+bwd fp64 "
                                       "per step (numpy, one thread)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return 0

    import torch

    from linear_rnn_state_gb300 import inputs, rwkv8, wkv7

    torch.cuda.set_device(local)
    dist = _init_pg(world, "nccl")
    rwkv8.load()
    dev = torch.device("cuda", local)
    sh = dict(RWKV8_SHAPE)
    if args.T:
        sh["T"] = args.T
    B, T, H, Hv, L, E = (sh[k] for k in ("B", "T", "H", "Hv", "L", "E"))
    d = inputs.generate_rwkv8(B, T, H, Hv, L, E, "f32", seed=shard_seed(rank))
    t_in = {k: torch.from_numpy(d[k]).to(dev) for k in ("q", "v", "decay", "dy")}
    if dist:  # the decay is a parameter: one copy for every rank (rank 0's)
        dist.broadcast(t_in["decay"], src=0)
    f32 = dict(dtype=torch.float32, device=dev)
    y = torch.empty((B, H, T, E), **f32)
    rf, nf = torch.empty((B, H, L, E), **f32), torch.empty((B, H, L), **f32)
    ckpt = torch.empty(rwkv8.rwkv8_ckpt_bytes(B, T, H, L, E) // 4, **f32)
    g = {"dq": torch.empty((B, H, T, L), **f32), "dv": torch.empty((B, Hv, T, E), **f32),
         "ddecay": torch.empty((H, L), **f32), "d_rho_init": torch.empty((B, H, L, E), **f32),
         "d_rho_norm_init": torch.empty((B, H, L), **f32)}
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    fargs = [t_in["q"].data_ptr(), t_in["v"].data_ptr(), t_in["decay"].data_ptr(), None, None, y.data_ptr(),
             rf.data_ptr(), nf.data_ptr(), ckpt.data_ptr(), B, T, H, Hv, L, E, sp]
    bargs = [t_in["q"].data_ptr(), t_in["v"].data_ptr(), t_in["decay"].data_ptr(), t_in["dy"].data_ptr(), None, None,
             None, None, ckpt.data_ptr()] + [g[k].data_ptr() for k in g] + [B, T, H, Hv, L, E, sp]

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        rc = rwkv8.rwkv8_forward(*fargs)
        if ev is not None:
            ev[1].record(stream)
        rc2 = rwkv8.rwkv8_backward(*bargs)
        allreduce_param_grad(g["ddecay"], dist)
        if ev is not None:
            ev[2].record(stream)
        if rc or rc2:
            raise RuntimeError(wkv7.last_error())

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local, args.clock_csv) as clocks:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(args.steps):
            step(events[k])
        end.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = reduce_max(start.elapsed_time(end) / args.steps, dist, dev)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in events)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in events)

    e2e = None
    if not args.no_e2e:
        # inputs q, v, dy in and y and every gradient out, pipelined over two buffer sets (the decay
        # is a parameter and stays resident; checkpoints and final states never leave the device)
        names = ("q", "v", "dy")
        host_in = {k: torch.from_numpy(d[k]).pin_memory() for k in names}
        t1 = {k: torch.empty_like(t_in[k]) for k in names}
        g1 = {k: torch.empty_like(x) for k, x in g.items()}
        sets = [({k: t_in[k] for k in names}, {**g, "y": y}), (t1, {**g1, "y": torch.empty_like(y)})]

        def set_args(i):
            tin, out = sets[i]
            fa = [tin["q"].data_ptr(), tin["v"].data_ptr(), t_in["decay"].data_ptr(), None, None,
                  out["y"].data_ptr(), rf.data_ptr(), nf.data_ptr(), ckpt.data_ptr(), B, T, H, Hv, L, E, sp]
            ba = [tin["q"].data_ptr(), tin["v"].data_ptr(), t_in["decay"].data_ptr(), tin["dy"].data_ptr(), None,
                  None, None, None, ckpt.data_ptr()] + [out[k].data_ptr() for k in g] + [B, T, H, Hv, L, E, sp]
            return fa, ba

        pargs = [set_args(0), set_args(1)]

        def step_on(i):
            rc = rwkv8.rwkv8_forward(*pargs[i][0])
            rc2 = rwkv8.rwkv8_backward(*pargs[i][1])
            allreduce_param_grad(sets[i][1]["ddecay"], dist)
            if rc or rc2:
                raise RuntimeError(wkv7.last_error())

        e2e = _pipelined_e2e(args, host_in, sets, step_on, stream, dist, dev)
    if rank != 0:
        return 0

    peaks = _peaks()
    BTH = B * T * H
    f_flop, b_flop, f_bytes, b_bytes = _rwkv8_work_per_token_head(L, E)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_flops = sms * FP32_LANES_PER_SM * 2 * peaks["sm_max_mhz"] * 1e6
    achieved = b_flop * BTH / (bwd_ms * 1e-3)
    t_roof = max((f_flop + b_flop) * BTH / peak_flops, (f_bytes + b_bytes) * BTH / (peaks["hbm_gbs"] * 1e9))
    traffic = None
    split_bwd = _rwkv8_env("RWKV8_SPLIT_BACKWARD") and not _rwkv8_env("RWKV8_SEQUENTIAL")
    bwd_kernel = ("rwkv8_bwd_r0_kernel + rwkv8_bwd_chain_kernel + rwkv8_bwd_chunk_kernel (one rwkv8_backward call)"
                  if split_bwd
                  else RWKV8_TRAFFIC["kernel"])
    if (not split_bwd and RWKV8_TRAFFIC["sha256"]
            and sources_sha256(RWKV8_TRAFFIC["sources"]) == RWKV8_TRAFFIC["sha256"]):
        traffic = RWKV8_TRAFFIC["bytes_per_token_head"] * BTH
    line = {
        "metric": RWKV8_METRIC, "value": aggregate_tokens_per_s(world, B, T, ms), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "arithmetic": "fp32 FFMA on the CUDA cores; the forward's chain and readout products on the tensor cores "
                      "in split tf32 (three tf32 products per fp32 product, fp32 accumulation)",
        "config": {"workload": "rwkv8-4x4096x32-l64e64-f32" if T == RWKV8_SHAPE["T"] else f"rwkv8 (T={T})", **sh,
                   "ckpt_every": 16,
                   "l2": "no flush: inputs, checkpoints and gradients (%.1f GB) exceed the 129 MB L2"
                         % ((3 * BTH * 64 * 4 + ckpt.numel() * 4 + 3 * BTH * 64 * 4) / 1e9)},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "step_roofline_frac": t_roof / (ms * 1e-3),
        "roofline": {"bound": "alu", "achieved": achieved / 1e12, "peak": peak_flops / 1e12, "unit": "TFLOP/s",
                     "frac": achieved / peak_flops, "traffic": traffic, "kernel": bwd_kernel,
                     "note": "the backward call timed with CUDA events around it: algorithmic FLOP of the "
                             "recurrence (12 L E per token-head) against the FP32 CUDA-core peak",
                     "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {peaks['sm_max_mhz']:.0f} MHz",
                     "hbm_gbs_achieved": b_bytes * BTH / (bwd_ms * 1e-3) / 1e9, "hbm_peak_gbs": peaks["hbm_gbs"]},
        "e2e": None if e2e is None else {
            "value": aggregate_tokens_per_s(world, B, T, e2e[0]), "unit": "tokens/s", "h2d_bytes_per_step": e2e[1],
            "d2h_bytes_per_step": e2e[2]},
        # forward: the chain and the per-chunk readout (one kernel with RWKV8_SEQUENTIAL=1); backward: its
        # kernel and the ddecay sum over b (RWKV8_SPLIT_BACKWARD=1: the R0 pass, the chain, the
        # per-chunk kernel and the sums over the chunks and over b); for a shared value row, one dv sum
        # per batch row
        "gpu_launches": ((1 if _rwkv8_env("RWKV8_SEQUENTIAL") else 2)
                         + (5 if _rwkv8_env("RWKV8_SPLIT_BACKWARD") and not _rwkv8_env("RWKV8_SEQUENTIAL") else 2)
                         + (B if Hv == 1 and H > 1 else 0)) * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline and T == RWKV8_SHAPE["T"]:
        heads = 16
        v, dt = _rwkv8_oracle_sample(d, heads, T)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                "sample": f"{heads} of {B * H} heads, full T={T}, fwd+bwd fp64 ({dt:.1f} s, numpy)"}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--clock-csv", default=None,
                    help="file for the raw nvidia-smi samples of the timed region ({rank} = device index); "
                         "a temporary file by default")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the timed oracle sample")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--T", type=int, default=0, help="override T (profiler captures of a smaller case)")
    ap.add_argument("--workload", choices=["wkv7", "wkv7-logit", "wkv7-epilogue", "rwkv8"], default="wkv7",
                    help="wkv7: the RWKV-7 1.5B-shaped layer (default); wkv7-logit: the same with the decay "
                         "given as logits and formed inside the kernels; wkv7-epilogue: the same step with the "
                         "group-norm + bonus epilogue (fused into the forward) and its backward; rwkv8: the "
                         "RWKV-8 recurrence")
    ap.add_argument("--shape", default=None,
                    help="WKV7 workload by name (linear_rnn_state_gb300/configs.py): rwkv7-1.5b-layer-bf16 "
                         "(default, the metric's), rwkv7-0.1b-layer-fp32, long-carry-fp32, small-fp32-carry, "
                         "tiny-fp32")
    args = ap.parse_args()
    from linear_rnn_state_gb300 import configs

    args.shape = args.shape or configs.BENCH_WORKLOAD
    if args.shape not in configs.WORKLOADS:
        ap.error(f"unknown --shape {args.shape}; one of {', '.join(configs.WORKLOADS)}")
    if args.workload == "rwkv8":
        return run_rwkv8(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
