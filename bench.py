"""Benchmark of the ZeroS causal forward: B8 H8 N4096 d64, bf16, RoPE, one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload causal|encoder|long|decode|sm] [--path auto|simt|chunk]
                    [--pass fwd|bwd] [--ln]

One step = one pass of the whole hot path (logits, prefix scans, zero-sum weights, angular
factor, state scan and readout: one zeros_fwd call) over one batch of device-resident
synthetic inputs.  Each step is timed with CUDA events on the launching stream; L2 is flushed
(a 256 MB write) before every step, outside the timed events.  Prints ONE JSON line (rank 0).

N > 1 (torchrun): every rank runs its own copy of the workload on its own GPU (the B x H
sequences are independent: weak scaling, no data-path collective); value = tokens of all
ranks / max-over-ranks time.

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import zeros_inputs as zi  # noqa: E402

METRIC = "ZeroS fwd tokens/s (B8·H8·N4096·d64 bf16) and % of roofline on 1 GB300"
WORKLOADS = {
    "causal": zi.CAUSAL_ROPE_B8H8N4096D64,
    "encoder": zi.ENCODER_VIT_B256H3N197D64,
    "long": zi.LONG_ROPE_B2H16N65536D128,
    "decode": zi.DECODE_B256H32D128,
    "sm": zi.CAUSAL_ROPE_B8H8N4096D64,  # ZeroS-SM on the causal RoPE workload's q, k, v, gates
}
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes (read + write) of one forward call (the scalar pass and the d = 64 forward kernel),
# from the committed ncu summaries of this workload, keyed by a fingerprint of the kernel
# sources they were measured on; reported as null once the sources change.
CHUNK_SOURCES = ["zero_sum_prefix_gb300/csrc/zs_walk.cu", "zero_sum_prefix_gb300/csrc/zs_scalars.cu",
                 "zero_sum_prefix_gb300/csrc/zs_range.cuh", "zero_sum_prefix_gb300/csrc/zs_sm100.cuh",
                 "zero_sum_prefix_gb300/csrc/zs_common.cuh"]
MEASURED_TRAFFIC = {"2990ea0b17be6957": 33602816 + 0 + 111005952 + 9714944}
# the ZeroS-SM workload's dominant kernel (sm1_kernel): DRAM bytes read + written per launch
SM_SOURCES = ["zero_sum_prefix_gb300/csrc/zs_sm.cu", "zero_sum_prefix_gb300/csrc/zs_sm100.cuh",
              "zero_sum_prefix_gb300/csrc/zs_common.cuh"]
MEASURED_SM_TRAFFIC = {"72bcbcc9246ff7f2": 180504064 + 17020416}


def kernel_fingerprint(sources=None) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in (sources or CHUNK_SOURCES):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def algorithmic_bytes(w: zi.Workload) -> int:
    """Bytes the method must move per forward: read q, k, v, u and the two gate logits, write
    out (per token-head 4 d b_in + 8 + d b_out)."""
    b = 2 if w.dtype == "bf16" else 4
    return w.B * w.H * w.N * (4 * w.d * b + 8 + w.d * b)


def decode_bytes(w: zi.Workload) -> int:
    """Bytes one decode step must move: every sequence's three fp32 d x d states read and
    written, plus its running sum and scalars, plus the token (q, k, v, u, gates) and out."""
    b = 2 if w.dtype == "bf16" else 4
    per = 2 * (12 * w.d * w.d + 4 * w.d + 16) + 4 * w.d * b + 8 + w.d * b
    return w.B * w.H * per


def backward_bytes(w: zi.Workload) -> int:
    """Bytes the backward must move: read q, k, v, u, dout and the two gate logits, write the
    fp32 gradients dq, dk, dv, du, dg1, dgh (per token-head 5 d b_in + 8 + 16 d + 8)."""
    b = 2 if w.dtype == "bf16" else 4
    return w.B * w.H * w.N * (5 * w.d * b + 8 + 16 * w.d + 8)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    """Rank / world from the torchrun environment.  One process per GPU over NCCL; on a host
    without CUDA (the multi-process tests) the same code runs over gloo."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cuda = torch.cuda.is_available()
    if world > 1:
        import torch.distributed as dist
        if cuda:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif cuda:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: float, ms_per_rank: float, world: int) -> tuple:
    """Whole-job throughput: the units every rank processed / the slowest rank's time."""
    ms = max_over_ranks(ms_per_rank, world)
    return units_per_rank * world / (ms / 1e3), ms


# ---------------------------------------------------------------------------------------------
def pipelined_e2e(host_in: dict, step, steps: int, world: int) -> float:
    """End-to-end time per step through the public API with host buffers: every step copies its
    inputs from pinned host memory (``host_in``) to the device, runs ``step(dev_inputs)`` (which
    returns the device result tensors) and copies the results back to pinned host memory.  Three
    streams and two buffer sets let step i+1's host-to-device copy, step i's kernels and step
    i-1's device-to-host copy run at the same time (a streaming pipeline; each buffer set is
    reused only after its previous step's kernels and copy-back finished).  Returns ms per step
    (max over ranks)."""
    sets = [{n: torch.empty_like(t, device="cuda") for n, t in host_in.items()} for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    host_out = [None, None]
    held = [None, None]  # results of a set's last step, alive until its copy-back is ordered

    def run(n_steps):
        for i in range(n_steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_cmp[b])
                for n, t in host_in.items():
                    sets[b][n].copy_(t, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[b])
                if i >= 2:
                    s_cmp.wait_event(ev_out[b])
                res = step(sets[b])
                held[b] = res
                ev_cmp[b].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[b])
                if host_out[b] is None:
                    host_out[b] = [torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in res]
                for h, r in zip(host_out[b], res):
                    h.copy_(r, non_blocking=True)
                ev_out[b].record(s_out)

    run(4)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    run(steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize()
    return max_over_ranks(e0.elapsed_time(e1) / steps, world)


def oracle_rate(w: zi.Workload, inp_cpu: dict, seqs: int, tokens: int, nthreads: int,
                min_seconds: float = 0.0):
    """Run the fp64 oracle on `seqs` sequences x `tokens` tokens, repeated until `min_seconds`
    of wall time have passed; return (tokens/s, seconds, threads, passes).  Throughput is
    counted in the metric's token unit (one (b, n) position carries H heads, so seqs*tokens
    token-heads count as seqs*tokens/H tokens)."""
    import oracle
    pick = [(i // w.H, i % w.H) for i in range(seqs)]
    sel = lambda t: torch.stack([t[b, h, :tokens] for b, h in pick])[None]  # noqa: E731
    q, k, v, u = (sel(inp_cpu[n]) for n in ("q", "k", "v", "u"))
    g1, gh = sel(inp_cpu["g1"]), sel(inp_cpu["gh"])
    # one head's prior for the whole sample (the cost does not depend on which head)
    mu = inp_cpu["mu"][:1].repeat(seqs, 1)
    tau = inp_cpu["tau"][:1].repeat(seqs)
    args = [x.double().numpy() for x in (q[0][None], k[0][None], v[0][None], u[0][None])]
    q64, k64, v64, u64 = (a.reshape(1, seqs, tokens, w.d) for a in args)
    g164 = g1.double().numpy().reshape(1, seqs, tokens)
    gh64 = gh.double().numpy().reshape(1, seqs, tokens)
    mu64, tau64 = mu.double().numpy(), tau.double().numpy()
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle.forward(q64, k64, v64, u64, g164, gh64, mu64, tau64, causal=w.causal,
                       rope=w.rope, rope_base=w.rope_base, nthreads=nthreads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= 50:
            break
    token_heads = seqs * tokens * passes
    return token_heads / w.H / dt, dt, min(nthreads, seqs), passes


def reference_arm(args, w: zi.Workload):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = oracle.threads()
    seqs = min(cores, w.B * w.H)
    tokens = min(w.N, 512)
    inp = zi.make(w, "cpu", N=tokens)
    for _ in range(args.warmup):
        oracle_rate(w, inp, seqs, tokens, cores)
    times = []
    for _ in range(args.steps):
        _, dt, used, _ = oracle_rate(w, inp, seqs, tokens, cores)
        times.append(dt)
    sec = sum(times) / len(times)
    value = seqs * tokens / w.H / sec
    sample = (f"{seqs} of the {w.B * w.H} (b,h) sequences x first {tokens} tokens of "
              f"{w.name}, fp64 recurrent oracle, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------------------------
def ours_forward(args, w: zi.Workload):
    world, rank, local = dist_setup()
    import zero_sum_prefix_gb300 as zs
    zs.load()
    dev = torch.device("cuda", local)
    inp = zi.make(w, dev)
    out = torch.empty_like(inp["q"])
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    ln = {}
    if args.ln:  # fused output LayerNorm with a per-head gain and bias
        gen = torch.Generator(device="cpu").manual_seed(w.seed + 17)
        ln = dict(ln=True, ln_w=(1.0 + 0.1 * torch.randn((w.H, w.d), generator=gen)).to(dev),
                  ln_b=(0.1 * torch.randn((w.H, w.d), generator=gen)).to(dev))

    def step():
        zs.fwd(inp["q"], inp["k"], inp["v"], inp["u"], inp["g1"], inp["gh"], inp["mu"],
               inp["tau"], causal=w.causal, rope=w.rope, rope_base=w.rope_base, out=out,
               path=args.path, **ln)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if zs.get_status() != 0:
        raise RuntimeError("device status after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = zs.kernel_launches()
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = zs.kernel_launches() - launches0
    barrier(world)
    clk = clocks.stop()
    if zs.get_status() != 0:
        raise RuntimeError("device status after the timed region")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    tokens = w.B * w.N
    value, ms = aggregate_rate(tokens, sum(per) / len(per), world)

    hbm, peak_kind = peaks()
    alg = algorithmic_bytes(w)
    achieved = alg / (ms / 1e3) / 1e9

    # ---- end to end through the public API with host buffers (pipelined over steps) ----
    names = ("q", "k", "v", "u", "g1", "gh", "mu", "tau")
    host = {n: inp[n].cpu().pin_memory() for n in names}
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = out.numel() * out.element_size()
    outs = {}

    def e2e_step(src):
        o = outs.setdefault(src["q"].data_ptr(), torch.empty_like(out))
        zs.fwd(src["q"], src["k"], src["v"], src["u"], src["g1"], src["gh"], src["mu"],
               src["tau"], causal=w.causal, rope=w.rope, rope_base=w.rope_base, out=o,
               path=args.path, **ln)
        return [o]

    e2e_ms = pipelined_e2e(host, e2e_step, max(3, min(args.steps, 20)), world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = oracle.threads()
        inp_cpu = {n: t.cpu() for n, t in inp.items()}
        seqs = min(w.B * w.H, max(cores, 1) * 4)
        rate, dt, used, reps = oracle_rate(w, inp_cpu, seqs, w.N, cores, min_seconds=1.5)
        cpu = {"value": rate, "unit": "tokens/s", "cores": used, "kind": "oracle",
               "sample": f"{seqs} of {w.B * w.H} (b,h) sequences x all {w.N} tokens, fp64 "
                         f"recurrent oracle, {reps} passes ({dt:.1f} s wall)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "rope": w.rope, "rope_base": w.rope_base,
                       "path": args.path, "parallelism": f"replicas x{world}",
                       "output_layernorm": bool(args.ln),
                       "l2": "flushed before every step (256 MB write, outside the events)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm,
                         "traffic": (MEASURED_TRAFFIC.get(kernel_fingerprint())
                                     if w is zi.CAUSAL_ROPE_B8H8N4096D64 and args.path != "simt"
                                     and not args.ln else None),
                         "peak_source": peak_kind,
                         "algorithmic_bytes_per_launch": alg,
                         "timed": ("the whole zeros_fwd call: scalar pass + forward kernel"
                                   if args.path != "simt" else "the whole zeros_fwd call")},
            "cpu_baseline": cpu,
            "e2e": {"value": tokens * world / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line))


def ours_backward(args, w: zi.Workload):
    """Backward of the causal layer (zeros_bwd): one step = the gradients of sum(out * dout)
    with respect to every input, for the whole batch."""
    if not w.causal:
        raise SystemExit("the backward pass is defined for the causal workloads")
    world, rank, local = dist_setup()
    import zero_sum_prefix_gb300 as zs
    zs.load()
    dev = torch.device("cuda", local)
    inp = zi.make(w, dev)
    gen = torch.Generator(device="cpu").manual_seed(w.seed * 7 + 3)
    dout = torch.randn(inp["q"].shape, generator=gen).to(dev, inp["q"].dtype)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    names = ("q", "k", "v", "u", "g1", "gh", "mu", "tau")

    def step(src, do):
        return zs.bwd(*(src[n] for n in names), do, rope=w.rope, rope_base=w.rope_base)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step(inp, dout)
    torch.cuda.synchronize()
    if zs.get_status() != 0:
        raise RuntimeError("device status after warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    l0 = zs.kernel_launches()
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step(inp, dout)
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = zs.kernel_launches() - l0
    barrier(world)
    clk = clocks.stop()
    if zs.get_status() != 0:
        raise RuntimeError("device status after the timed region")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    tokens = w.B * w.N
    value, ms = aggregate_rate(tokens, sum(per) / len(per), world)
    hbm, kind = peaks()
    alg = backward_bytes(w)

    # end to end with host buffers: inputs and dout in, every gradient out (pipelined)
    host = {n: inp[n].cpu().pin_memory() for n in names}
    host["dout"] = dout.cpu().pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    grads = step(inp, dout)
    d2h = sum(t.numel() * t.element_size() for t in grads.values())

    def e2e_step(src):
        return list(step(src, src["dout"]).values())

    e2e_ms = pipelined_e2e(host, e2e_step, max(3, min(args.steps, 10)), world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle import grad as ograd
        toks = min(w.N, 1024)
        c = {n: inp[n].cpu() for n in names}
        sl = lambda t: t[:1, :, :toks]  # noqa: E731
        t0 = time.perf_counter()
        reps = 0
        while True:
            ograd.backward(sl(c["q"]), sl(c["k"]), sl(c["v"]), sl(c["u"]), sl(c["g1"]),
                           sl(c["gh"]), c["mu"], c["tau"], sl(dout.cpu()), rope=w.rope,
                           rope_base=w.rope_base)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= 1.5 or reps >= 20:
                break
        cpu = {"value": toks * reps / (dt), "unit": "tokens/s", "cores": torch.get_num_threads(),
               "kind": "oracle",
               "sample": f"batch 1 (all {w.H} heads) x first {toks} tokens, fp64 autograd of "
                         f"the O(N^2) definition, {reps} passes ({dt:.1f} s wall)"}
    if rank == 0:
        print(json.dumps({
            "metric": f"ZeroS backward tokens/s ({w.name})", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "rope": w.rope, "pass": "backward",
                       "l2": "flushed before every step (256 MB write, outside the events)"},
            "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": alg / (ms / 1e3) / 1e9 / hbm, "traffic": None,
                         "peak_source": kind, "algorithmic_bytes_per_launch": alg},
            "cpu_baseline": cpu,
            "e2e": {"value": tokens * world / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches, "clocks": clk}))


def sm_flops(w: zi.Workload) -> float:
    """Algorithmic flops of ZeroS-SM: the logits Q K^T and the weighted sum W V over the visible
    (query, key) pairs, 2 d flops per pair each (causal: N (N + 1) / 2 pairs per sequence)."""
    pairs = w.N * (w.N + 1) / 2 if w.causal else float(w.N) * w.N
    return w.B * w.H * pairs * 4.0 * w.d


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def ours_sm(args, w: zi.Workload):
    """ZeroS-SM, the quadratic variant (zeros_sm_fwd): one step = one forward of the batch."""
    world, rank, local = dist_setup()
    import zero_sum_prefix_gb300 as zs
    zs.load()
    dev = torch.device("cuda", local)
    inp = zi.make(w, dev)
    names = ("q", "k", "v", "g1", "gh")
    out = torch.empty_like(inp["q"])
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(src):
        return zs.sm_fwd(*(src[n] for n in names), causal=w.causal, rope=w.rope,
                         rope_base=w.rope_base, out=out)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1.0)
        step(inp)
    torch.cuda.synchronize()
    if zs.get_status() != 0:
        raise RuntimeError("device status after warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    l0 = zs.kernel_launches()
    for i in range(args.steps):
        flush.fill_(float(i))
        starts[i].record(stream)
        step(inp)
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = zs.kernel_launches() - l0
    barrier(world)
    clk = clocks.stop()
    if zs.get_status() != 0:
        raise RuntimeError("device status after the timed region")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    tokens = w.B * w.N
    value, ms = aggregate_rate(tokens, sum(per) / len(per), world)
    peak, kind = bf16_peak()
    achieved = sm_flops(w) / (ms / 1e3) / 1e12

    host = {n: inp[n].cpu().pin_memory() for n in names}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out.numel() * out.element_size()
    outs = {}

    def e2e_step(src):
        o = outs.setdefault(src["q"].data_ptr(), torch.empty_like(out))
        zs.sm_fwd(*(src[n] for n in names), causal=w.causal, rope=w.rope,
                  rope_base=w.rope_base, out=o)
        return [o]

    e2e_ms = pipelined_e2e(host, e2e_step, max(3, min(args.steps, 10)), world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        toks = min(w.N, 1024)
        sel = {n: inp[n][:1, :, :toks].cpu() for n in names}
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.sm(*(sel[n] for n in names), causal=w.causal, rope=w.rope,
                      rope_base=w.rope_base, nthreads=oracle.threads())
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= 1.5 or reps >= 20:
                break
        cpu = {"value": toks * reps / dt, "unit": "tokens/s",
               "cores": min(oracle.threads(), w.H), "kind": "oracle",
               "sample": f"batch 1 (all {w.H} heads) x first {toks} tokens, fp64 O(N^2) "
                         f"oracle, {reps} passes ({dt:.1f} s wall)"}
    if rank == 0:
        print(json.dumps({
            "metric": f"ZeroS-SM fwd tokens/s ({w.name})", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "rope": w.rope, "variant": "ZeroS-SM",
                       "l2": "flushed before every step (256 MB write, outside the events)"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak,
                         "traffic": (MEASURED_SM_TRAFFIC.get(kernel_fingerprint(SM_SOURCES))
                                     if w is zi.CAUSAL_ROPE_B8H8N4096D64 else None),
                         "peak_source": kind, "algorithmic_flops_per_launch": sm_flops(w),
                         "timed": "the whole zeros_sm_fwd call: statistics and rotary pass + "
                                  "attention kernel"},
            "cpu_baseline": cpu,
            "e2e": {"value": tokens * world / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches, "clocks": clk}))


def ours_decode(args, w: zi.Workload):
    """Recurrent decode: prefill 8192 tokens (zeros_fwd_ex final_state), then time decode
    steps; one step advances all B x H sequences by one token."""
    world, rank, local = dist_setup()
    import zero_sum_prefix_gb300 as zs
    zs.load()
    dev = torch.device("cuda", local)
    st = torch.empty(zs.state_bytes(w.B, w.H, w.d), dtype=torch.uint8, device=dev)
    # prefill in batch slices to bound the memory held by inputs
    slice_b = 16
    mu = tau = None
    for b0 in range(0, w.B, slice_b):
        part = zi.make(w.with_(seed=w.seed * 131 + b0), dev, B=min(slice_b, w.B - b0))
        if mu is None:
            mu, tau = part["mu"], part["tau"]
        nb = part["q"].shape[0]
        sub = torch.empty(zs.state_bytes(nb, w.H, w.d), dtype=torch.uint8, device=dev)
        zs.fwd(part["q"], part["k"], part["v"], part["u"], part["g1"], part["gh"], mu, tau,
               causal=True, rope=w.rope, rope_base=w.rope_base, final_state=sub)
        rb = zs.record_bytes(w.d)
        st[256 + b0 * w.H * rb: 256 + (b0 + nb) * w.H * rb].copy_(sub[256:])
        if b0 == 0:
            st[:256].copy_(sub[:256])
        del part, sub
    # the header records B; rewrite it for the full batch
    hdr = st[:256].view(torch.int32)
    hdr[2] = w.B
    steps_tok = [zi.decode_tokens(w, i, dev) for i in range(8)]
    out = torch.empty((w.B, w.H, w.d), dtype=torch.bfloat16, device=dev)

    def step(i):
        tk = steps_tok[i % len(steps_tok)]
        zs.decode_step(st, tk["q"], tk["k"], tk["v"], tk["u"], tk["g1"], tk["gh"], out=out)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    l0 = zs.kernel_launches()
    for i in range(args.steps):
        starts[i].record(stream)
        step(i)
        ends[i].record(stream)
    torch.cuda.synchronize()
    launches = zs.kernel_launches() - l0
    clk = clocks.stop()
    if zs.get_status() != 0:
        raise RuntimeError("device status after decode")
    per = sorted(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms = max_over_ranks(statistics.median(per), world)
    hbm, kind = peaks()
    alg = decode_bytes(w)
    achieved = alg / (ms / 1e3) / 1e9

    # end to end: each step's token (q, k, v, u, gates) copied in from pinned host memory and its
    # output copied back; the recurrent state stays resident on the device
    tk0 = steps_tok[0]
    host = {n: tk0[n].cpu().pin_memory() for n in ("q", "k", "v", "u", "g1", "gh")}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out.numel() * out.element_size()
    outs = {}

    def e2e_step(src):
        o = outs.setdefault(src["q"].data_ptr(), torch.empty_like(out))
        zs.decode_step(st, src["q"], src["k"], src["v"], src["u"], src["g1"], src["gh"], out=o)
        return [o]

    e2e_ms = pipelined_e2e(host, e2e_step, max(3, min(args.steps, 50)), world)
    if zs.get_status() != 0:
        raise RuntimeError("device status after the end-to-end decode steps")
    if rank == 0:
        print(json.dumps({
            "metric": "ZeroS decode step tokens/s (B256 H32 d128, fp32 state, after 8192-token "
                      "prefill)", "value": w.B * world / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "d": w.d,
                       "l2": "state (3.2 GB) larger than L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": None, "peak_source": kind,
                         "algorithmic_bytes_per_launch": alg},
            "e2e": {"value": w.B * world / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches, "clocks": clk}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # default: 1500 steps (the default workload's timed region is then about a quarter of a
    # second, so the clock samples, every 50 ms, come from a sustained run); 30 for the
    # reference arm, whose steps run the CPU oracle
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="causal", choices=sorted(WORKLOADS))
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "chunk"])
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd"])
    ap.add_argument("--ln", action="store_true", help="fuse the output LayerNorm (forward)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 30 if args.impl == "reference" else 1500
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, w)
    elif args.workload == "sm":
        ours_sm(args, w)
    elif args.pass_ == "bwd":
        ours_backward(args, w)
    elif args.workload == "decode":
        ours_decode(args, w)
    else:
        ours_forward(args, w)


if __name__ == "__main__":
    main()
