"""Benchmark: useful TFLOP/s of jagged attention forward + backward on GB300.

One step = the whole hot path over one batch of the GEM-shaped workload
(B=1024 sequences, lognormal lengths median 256 / sigma 0.8 clipped to
[1, 2048], H=4, D=128, bf16, int64 offsets): host LPT + zigzag schedule of
the batch's offsets, upload of the tile lists, jagged forward (O, LSE) and
jagged backward (dQ, dK, dV). Inputs are resident in HBM and larger than
L2 (4 x 363 MB), so no explicit L2 flush is needed between steps.

Prints ONE JSON line (rank 0). With --impl reference, the CPU fp64 oracle
is timed instead on a bounded sample of the same workload.

Multi-GPU (torchrun): every rank runs its own batch (seed + rank); the
sequences are independent, so there is no collective on the data path
("scaling": "weak"); value = all ranks' useful FLOPs / max rank time.
"""

import argparse
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


# DRAM bytes (read + write) of one GEM backward launch, from an ncu capture of
# the first 256 sequences (dram__bytes_read.sum + dram__bytes_write.sum)
# scaled by the processed (key tile, query block) pairs. Reset to None
# whenever the backward kernel changes until it is measured again.
BWD_GEM_TRAFFIC = 4.22e9


def _spin(stream, cycles=2_000_000):
    """Queue about 1 ms of device-side idling on `stream` (no memory traffic)."""
    import torch
    with torch.cuda.stream(stream):
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(cycles)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(local_flops, local_ms, ws, dev):
    """Whole-job figures of a weak-scaling run: the useful FLOPs of every rank's
    own batch summed, and the slowest rank's time. One process per GPU; with
    ws == 1 the local values are returned unchanged."""
    if ws == 1:
        return float(local_flops), float(local_ms)
    import torch
    import torch.distributed as dist
    f = torch.tensor([float(local_flops)], dtype=torch.float64, device=dev)
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(f, op=dist.ReduceOp.SUM)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(f.item()), float(t.item())


def _gem_lengths(seed_offset=0):
    from jagged_flash_attention_flashattention_gb300 import workloads as W
    if seed_offset == 0:
        return W.lengths_for("gem")
    return W.lengths_for("gem", seed=W.SEEDS["gem"] + 7919 * seed_offset)


def cpu_baseline(budget_s=12.0, lengths=None, H=4, D=128):
    """Times the fp64 oracle (fwd + bwd) on a prefix of the GEM batch."""
    import torch

    from jagged_flash_attention_flashattention_gb300 import workloads as W
    from oracle import attention as A

    L = (_gem_lengths() if lengths is None else lengths)[:256]
    inp = W.jagged_inputs(L, H, D, W.SEEDS["gem"], device="cpu")
    q, k, v, do = (inp[n].double().numpy() for n in ("q", "k", "v", "do"))
    offs = W.offsets_of(L)
    s = 1 / np.sqrt(D)
    t0 = time.perf_counter()
    flops = 0.0
    n = 0
    while n < len(L) and time.perf_counter() - t0 < budget_s:
        a, e = int(offs[n]), int(offs[n + 1])
        for h in range(H):
            A.seq_fwd(q[a:e, h], k[a:e, h], v[a:e, h], s)
            A.seq_bwd(q[a:e, h], k[a:e, h], v[a:e, h], do[a:e, h], s)
        flops += 3.5 * 4.0 * H * D * float(e - a) ** 2
        n += 1
    dt = time.perf_counter() - t0
    threads = torch.get_num_threads()
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        threads = max((i.get("num_threads", 0) for i in info), default=threads)
    except Exception:
        pass
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": int(threads), "kind": "oracle",
            "sample": "fp64 NumPy oracle fwd+bwd on the first %d GEM sequences x %d heads "
                      "(%.1f s wall, %d host cores visible)" % (n, H, dt, os.cpu_count())}


METRIC = "useful TFLOP/s fwd+bwd (jagged attention, bf16) and % of GB300 bf16 tensor peak"


def _gem_desc(L, H=4, D=128):
    return "gem: B=%d, T=%d, H=%d, D=%d, max len %d" % (len(L), int(np.sum(L)), H, D, int(max(L)))


def run_reference(args):
    """The reference arm: the pages publish no runnable code, so the fp64 CPU
    oracle stands in for it. W untimed and K timed steps; a step is the oracle's
    forward + backward over a bounded prefix of the GEM batch (the same prefix
    every step), sized so the whole run stays within about two minutes."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import torch

    from jagged_flash_attention_flashattention_gb300 import workloads as W
    from oracle import attention as A

    H, D = 4, 128
    L_all = _gem_lengths()
    L = L_all[:256]
    inp = W.jagged_inputs(L, H, D, W.SEEDS["gem"], device="cpu")
    q, k, v, do = (inp[n].double().numpy() for n in ("q", "k", "v", "do"))
    offs = W.offsets_of(L)
    sc = 1 / np.sqrt(D)

    def seq(n):
        a, e = int(offs[n]), int(offs[n + 1])
        for h in range(H):
            A.seq_fwd(q[a:e, h], k[a:e, h], v[a:e, h], sc)
            A.seq_bwd(q[a:e, h], k[a:e, h], v[a:e, h], do[a:e, h], sc)
        return 3.5 * 4.0 * H * D * float(e - a) ** 2

    # size the step: as many leading sequences as fit in the per-step budget
    budget = min(6.0, 120.0 / max(1, args.steps + args.warmup))
    t0 = time.perf_counter()
    n_seq = 0
    while n_seq < len(L) and time.perf_counter() - t0 < budget:
        seq(n_seq)
        n_seq += 1
    step_flops = sum(3.5 * 4.0 * H * D * float(offs[n + 1] - offs[n]) ** 2 for n in range(n_seq))
    for _ in range(args.warmup - 1):
        for n in range(n_seq):
            seq(n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for n in range(n_seq):
            seq(n)
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    value = step_flops / (ms * 1e-3) / 1e12
    threads = torch.get_num_threads()
    try:
        import threadpoolctl
        threads = max((i.get("num_threads", 0) for i in threadpoolctl.threadpool_info()),
                      default=threads)
    except Exception:
        pass
    sample = ("fp64 NumPy oracle fwd+bwd on the first %d of the %d GEM sequences x %d heads per step "
              "(%.2f s per step)" % (n_seq, len(L_all), H, ms * 1e-3))
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _gem_desc(L_all, H, D), "parallelism": "replicas (one batch per GPU)",
                   "l2": "inputs larger than L2 (no flush)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": int(threads), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _setup(name, rank, dev, seqs=0):
    """Inputs and one hot-path step for a named workload. Returns a dict."""
    import torch

    import jagged_flash_attention_flashattention_gb300 as jfa
    from jagged_flash_attention_flashattention_gb300 import workloads as W

    cfg = W.WORKLOADS[name]
    H, D = cfg["H"], cfg["D"]
    st = {"H": H, "D": D, "kind": cfg["kind"]}
    if cfg["kind"] == "jagged":
        L = _gem_lengths(rank) if name == "gem" else W.lengths_for(name)
        if seqs:
            L = L[:seqs]
        off_host = W.offsets_of(L, cfg["offsets_dtype"])
        inp = W.jagged_inputs(L, H, D, W.SEEDS[name] + 1000 * rank, device=dev)
        off = torch.from_numpy(off_host).to(dev)
        ws_buf = jfa.Plan(off, H, D, host_offsets=off_host).workspace
        st["fwd_flops"] = W.useful_flops("jagged", L, H=H, D=D)
        st["desc"] = "%s: B=%d, T=%d, H=%d, D=%d, max len %d" % (name, len(L), int(off_host[-1]), H, D, int(max(L)))

        def fwd():
            st["plan"] = jfa.Plan(off, H, D, host_offsets=off_host, workspace=ws_buf)
            st["o"], st["lse"] = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=st["plan"])

        def bwd():
            jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], st["o"], st["lse"], inp["do"], off, plan=st["plan"])

        st["check"] = lambda: st["plan"].check()
    elif cfg["kind"] == "bcast":
        L = W.lengths_for(name)
        Lq = cfg["Lq"]
        off_host = W.offsets_of(L, cfg["offsets_dtype"])
        inp = W.bcast_inputs(L, Lq, H, D, W.SEEDS[name] + 1000 * rank, device=dev)
        off = torch.from_numpy(off_host).to(dev)
        st["fwd_flops"] = W.useful_flops("bcast", L, H=H, D=D, Lq=Lq)
        st["desc"] = "bcast: Lq=%d, B=%d, Tk=%d, H=%d, D=%d" % (Lq, len(L), int(off_host[-1]), H, D)

        def fwd():
            st["plan"] = jfa.Plan(off, H, D, kind="bcast", Lq=Lq, host_offsets=off_host)
            st["o"], st["lse"] = jfa.jfa_bcastq_fwd(inp["q"], inp["k"], inp["v"], off, plan=st["plan"])

        def bwd():
            jfa.jfa_bcastq_bwd(inp["q"], inp["k"], inp["v"], st["o"], st["lse"], inp["do"], off,
                               plan=st["plan"])

        st["check"] = lambda: st["plan"].check()
    else:
        B, L = (seqs or cfg["B"]), cfg["L"]
        inp = W.blockdiag_inputs(B, L, H, D, W.SEEDS[name] + 1000 * rank, device=dev)
        st["fwd_flops"] = W.useful_flops("blockdiag", H=H, D=D, B=B, L=L)
        st["fwd_bytes"] = 4 * B * L * H * D * 2
        st["bwd_bytes"] = 7 * B * L * H * D * 2
        st["desc"] = "blockdiag: B=%d, L=%d, H=%d, D=%d, 64-token blocks" % (B, L, H, D)

        def fwd():
            jfa.blockdiag_fwd(inp["q"], inp["k"], inp["v"])

        def bwd():
            jfa.blockdiag_bwd(inp["q"], inp["k"], inp["v"], inp["do"])

        st["check"] = lambda: jfa.check_status(device=dev)
    st["inp"] = inp
    st["fwd"], st["bwd"] = fwd, bwd
    st["bwd_flops"] = 2.5 * st["fwd_flops"]
    return st


def run_ours(args):
    import torch
    import torch.distributed as dist

    import jagged_flash_attention_flashattention_gb300 as jfa
    from jagged_flash_attention_flashattention_gb300 import workloads as W

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, tc_peak, tc_sust, peak_src = _peaks()

    st = _setup(args.config, rank, dev, args.seqs)
    fwd_flops, bwd_flops = st["fwd_flops"], st["bwd_flops"]
    stream = torch.cuda.current_stream()

    def step(timing=None):
        if timing is not None:
            timing["e0"].record(stream)
        st["fwd"]()
        if timing is not None:
            timing["e1"].record(stream)
        st["bwd"]()
        if timing is not None:
            timing["e2"].record(stream)

    for _ in range(args.warmup):
        step()
    st["check"]()

    evs = [{n: torch.cuda.Event(enable_timing=True) for n in ("e0", "e1", "e2")}
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # A short device-side spin before the start event lets the host queue the
    # timed steps ahead of the GPU, so host launch latency stays out of the
    # timed region (it holds only the steps' own kernels).
    _spin(stream)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    st["check"]()
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = statistics.median(e["e0"].elapsed_time(e["e1"]) for e in evs)
    bwd_ms = statistics.median(e["e1"].elapsed_time(e["e2"]) for e in evs)
    job_flops, t_max = aggregate_over_ranks(fwd_flops + bwd_flops, total_ms, ws, dev)
    ms_per_step = t_max / args.steps
    value = job_flops / (ms_per_step * 1e-3) / 1e12

    e2e = None
    if args.config == "gem" and not args.seqs:
        e2e = _e2e_gem(args, st, dev, ws)

    if rank == 0:
        bwd_tf = bwd_flops / (bwd_ms * 1e-3) / 1e12
        fwd_tf = fwd_flops / (fwd_ms * 1e-3) / 1e12
        peak = tc_peak  # a short run of back-to-back steps: the burst figure
        if st["kind"] == "blockdiag":
            bw = st["bwd_bytes"] / (bwd_ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "kernel": "blockdiag_bwd", "achieved": round(bw, 1),
                    "peak": hbm_peak, "unit": "GB/s", "frac": round(bw / hbm_peak, 4),
                    "traffic": None, "peak_source": peak_src + " HBM copy"}
        else:
            roof = {"bound": "tensor", "kernel": "jfa_bwd (bwd kernel + dQ cast)",
                    "achieved": round(bwd_tf, 1), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(bwd_tf / peak, 4),
                    "traffic": BWD_GEM_TRAFFIC if args.config == "gem" and not args.seqs else None,
                    "peak_source": peak_src + " bf16 burst (cuBLAS)"}
        line = {
            "metric": METRIC,
            "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": st["desc"], "parallelism": "replicas (one batch per GPU)",
                       "l2": "inputs larger than L2 (no flush)"},
            "fwd": {"ms": round(fwd_ms, 4), "tflops": round(fwd_tf, 1),
                    "frac_of_peak": round(fwd_tf / peak, 4)},
            "bwd": {"ms": round(bwd_ms, 4), "tflops": round(bwd_tf, 1),
                    "frac_of_peak": round(bwd_tf / peak, 4)},
            "pct_of_peak": round(100 * value / peak, 2),
            "roofline": roof,
            "clocks": clk,
            "gpu_launches": (4 if st["kind"] == "jagged" else 2) * args.steps,
        }
        if st["kind"] == "blockdiag":
            line["fwd"]["gbps"] = round(st["fwd_bytes"] / (fwd_ms * 1e-3) / 1e9, 1)
            line["bwd"]["gbps"] = round(st["bwd_bytes"] / (bwd_ms * 1e-3) / 1e9, 1)
        if e2e is not None:
            line["e2e"] = e2e
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _e2e_gem(args, st, dev, ws):
    """Same metric through the public API with host (pinned) buffers: every
    step copies q, k, v, dO and the offsets in and O, dQ, dK, dV out. Steps
    are pipelined the way a training input pipeline would run them: the
    host-to-device copy of step n+1 and the device-to-host copy of step n-1
    run on their own streams while step n's kernels run (two device buffer
    sets; every step still moves all of its own bytes in both directions)."""
    import torch
    import torch.distributed as dist

    import jagged_flash_attention_flashattention_gb300 as jfa

    H, D = st["H"], st["D"]
    inp = st["inp"]
    off_host = st["plan"].host_offsets
    hq, hk, hv, hdo = (inp[n].cpu().pin_memory() for n in ("q", "k", "v", "do"))
    h_off = torch.from_numpy(off_host).pin_memory()
    h_out = [[torch.empty_like(hq).pin_memory() for _ in range(4)] for _ in range(2)]
    d_in = [[torch.empty_like(inp[n]) for n in ("q", "k", "v", "do")] for _ in range(2)]
    d_off = [torch.empty_like(h_off, device=dev) for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo)) + off_host.nbytes
    d2h = 4 * hq.numel() * hq.element_size()
    ws_buf = st["plan"].workspace
    comp = torch.cuda.current_stream()
    # One stream per tensor and direction, so the copies spread over the copy engines.
    s_in = [torch.cuda.Stream() for _ in range(4)]
    s_out = [torch.cuda.Stream() for _ in range(4)]
    ev_in = [[torch.cuda.Event() for _ in range(4)] for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [[torch.cuda.Event() for _ in range(4)] for _ in range(2)]

    def e2e_step(n):
        b = n & 1
        for j, (dst, src) in enumerate(zip(d_in[b], (hq, hk, hv, hdo))):
            with torch.cuda.stream(s_in[j]):
                if n >= 2:
                    s_in[j].wait_event(ev_comp[b])  # step n-2 has finished reading buffer set b
                dst.copy_(src, non_blocking=True)
                if j == 0:
                    d_off[b].copy_(h_off, non_blocking=True)
                ev_in[b][j].record(s_in[j])
        for e in ev_in[b]:
            comp.wait_event(e)
        q_, k_, v_, do_ = d_in[b]
        p2 = jfa.Plan(d_off[b], H, D, host_offsets=off_host, workspace=ws_buf)
        o_, l_ = jfa.jfa_fwd(q_, k_, v_, d_off[b], plan=p2)
        g = jfa.jfa_bwd(q_, k_, v_, o_, l_, do_, d_off[b], plan=p2)
        ev_comp[b].record(comp)
        for j, (dst, src) in enumerate(zip(h_out[b], (o_,) + tuple(g))):
            with torch.cuda.stream(s_out[j]):
                s_out[j].wait_event(ev_comp[b])
                dst.copy_(src, non_blocking=True)
                src.record_stream(s_out[j])
                ev_out[b][j].record(s_out[j])

    for n in range(2):
        e2e_step(n)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    n_steps = max(2, min(args.steps, 20))
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(comp)
    for si in s_in:
        si.wait_event(a0)
    for n in range(n_steps):
        e2e_step(n)
    for e in ev_out[(n_steps - 1) & 1]:
        comp.wait_event(e)
    a1.record(comp)
    torch.cuda.synchronize()
    job_flops, ms = aggregate_over_ranks(st["fwd_flops"] + st["bwd_flops"],
                                         a0.elapsed_time(a1) / n_steps, ws, dev)
    val = job_flops / (ms * 1e-3) / 1e12
    return {"value": round(val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 3),
            "overlap": "h2d of step n+1 and d2h of step n-1 run beside step n's kernels"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seqs", type=int, default=0,
                    help="keep only the first N sequences (jagged) or N batch rows (block-diagonal): "
                         "a small profiling case")
    ap.add_argument("--config", default="gem",
                    choices=["gem", "stress", "bcast", "blockdiag", "blockdiag64", "tiny"])
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
