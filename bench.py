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
BWD_GEM_TRAFFIC = 4.224e9  # 680.6 + 327.1 MB on 256 sequences, x 4.1917 (129,708 / 30,944 pairs)

# Nominal dense bf16 tensor peak of one GB300 (NVIDIA's figure without 2:4
# sparsity), the second denominator reported next to the measured cuBLAS peak.
SPEC_BF16_TFLOPS = 2250.0


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
    """Times the fp64 oracle (fwd + bwd, and each separately) on a prefix of the GEM batch."""
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
    t_fwd = t_bwd = 0.0
    n = 0
    while n < len(L) and time.perf_counter() - t0 < budget_s:
        a, e = int(offs[n]), int(offs[n + 1])
        for h in range(H):
            t1 = time.perf_counter()
            A.seq_fwd(q[a:e, h], k[a:e, h], v[a:e, h], s)
            t2 = time.perf_counter()
            A.seq_bwd(q[a:e, h], k[a:e, h], v[a:e, h], do[a:e, h], s)
            t_fwd += t2 - t1
            t_bwd += time.perf_counter() - t2
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
    fwd_flops = flops / 3.5
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": int(threads), "kind": "oracle",
            "fwd_tflops": fwd_flops / max(t_fwd, 1e-9) / 1e12,
            "bwd_tflops": 2.5 * fwd_flops / max(t_bwd, 1e-9) / 1e12,
            "sample": "fp64 NumPy oracle fwd+bwd on the first %d GEM sequences x %d heads "
                      "(%.1f s wall: fwd %.1f s, bwd %.1f s; %d host cores visible)"
                      % (n, H, dt, t_fwd, t_bwd, os.cpu_count())}


def scheduler_times(dev, reps=10):
    """Host time of planning the GEM batch: the C scheduler alone (forward and
    backward tile lists), and a whole Plan (both lists, pinned staging and the
    asynchronous upload, synchronised), for self-attention and for the
    block-sparse masks of the gem_sparse workload. Medians over `reps`."""
    import torch

    import jagged_flash_attention_flashattention_gb300 as jfa
    from jagged_flash_attention_flashattention_gb300 import workloads as W

    L = _gem_lengths()
    H, D = 4, 128
    off_host = W.offsets_of(L)
    off = torch.from_numpy(off_host).to(dev)
    masks = jfa.pack_block_masks(W.block_masks(L, L, W.MASK_SEEDS["gem_sparse"], density=0.5),
                                 off_host, off_host)
    n_sms = jfa.num_sms()
    ws = jfa.Plan(off, H, D, host_offsets=off_host).workspace

    def med(fn):
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            ts.append((time.perf_counter() - t0) * 1e3)
        return round(statistics.median(ts), 3)

    def plan(**kw):
        jfa.Plan(off, H, D, host_offsets=off_host, workspace=ws, **kw)
        torch.cuda.synchronize()

    return {
        "workload": _gem_desc(L, H, D),
        "sched_ms": med(lambda: (jfa.schedule(off_host, H, jfa.tile_rows(jfa.OP_FWD, D), n_sms),
                                 jfa.schedule(off_host, H, jfa.tile_rows(jfa.OP_BWD, D), n_sms))),
        "plan_with_upload_ms": med(plan),
        "sparse_sched_ms": med(lambda: (jfa.schedule_sparse(off_host, off_host, H, jfa.OP_FWD, n_sms, masks),
                                        jfa.schedule_sparse(off_host, off_host, H, jfa.OP_BWD, n_sms, masks))),
        "sparse_plan_with_upload_ms": med(lambda: plan(kind="sparse", block_masks=masks)),
    }


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


def _setup(name, rank, dev, seqs=0, zigzag=True):
    """Inputs and one hot-path step for a named workload. Returns a dict."""
    import torch

    import jagged_flash_attention_flashattention_gb300 as jfa
    from jagged_flash_attention_flashattention_gb300 import workloads as W

    cfg = W.WORKLOADS[name]
    H, D = cfg["H"], cfg["D"]
    st = {"H": H, "D": D, "kind": cfg["kind"]}
    if cfg["kind"] == "jagged":
        lname = cfg.get("lengths", name)
        L = _gem_lengths(rank) if lname == "gem" else W.lengths_for(lname)
        if seqs:
            L = L[:seqs]
        off_host = W.offsets_of(L, cfg["offsets_dtype"])
        inp = W.jagged_inputs(L, H, D, W.SEEDS[name] + 1000 * rank, device=dev)
        off = torch.from_numpy(off_host).to(dev)
        ws_buf = jfa.Plan(off, H, D, host_offsets=off_host, zigzag=zigzag).workspace
        st["fwd_flops"] = W.useful_flops("jagged", L, H=H, D=D)
        st["desc"] = "%s: B=%d, T=%d, H=%d, D=%d, max len %d" % (name, len(L), int(off_host[-1]), H, D, int(max(L)))

        def fwd():
            st["plan"] = jfa.Plan(off, H, D, host_offsets=off_host, workspace=ws_buf, zigzag=zigzag)
            st["o"], st["lse"] = jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=st["plan"])

        def bwd():
            jfa.jfa_bwd(inp["q"], inp["k"], inp["v"], st["o"], st["lse"], inp["do"], off, plan=st["plan"])

        if cfg.get("rotary"):
            # rotary layer (q and k rotated at their positions in their
            # sequences), forward on the rotated rows, and the backward with
            # the rotary backward fused into its closing cast (dQ and dK)
            cos, sin = W.rotary_tables(int(max(L)), D, device=dev)
            st["desc"] += ", rotary (fp32 tables [max len, D/2])"

            def fwd():  # noqa: F811
                st["plan"] = jfa.Plan(off, H, D, host_offsets=off_host, workspace=ws_buf, zigzag=zigzag)
                st["qr"] = jfa.jfa_rope(inp["q"], off, cos, sin, plan=st["plan"])
                st["kr"] = jfa.jfa_rope(inp["k"], off, cos, sin, plan=st["plan"])
                st["o"], st["lse"] = jfa.jfa_fwd(st["qr"], st["kr"], inp["v"], off, plan=st["plan"])

            def bwd():  # noqa: F811
                jfa.jfa_rotary_bwd(st["qr"], st["kr"], inp["v"], st["o"], st["lse"], inp["do"], off,
                                   cos, sin, plan=st["plan"])

        st["check"] = lambda: st["plan"].check()
    elif cfg["kind"] == "varlen":
        L = _gem_lengths(rank) if cfg["lengths"] == "gem" else W.lengths_for(cfg["lengths"])
        if seqs:
            L = L[:seqs]
        win, det = cfg["window"], cfg["deterministic"]
        off_host = W.offsets_of(L, cfg["offsets_dtype"])
        inp = W.jagged_inputs(L, H, D, W.SEEDS[cfg["lengths"]] + 1000 * rank, device=dev)
        off = torch.from_numpy(off_host).to(dev)
        if cfg.get("kv_seed"):  # cross attention: key/value lengths of their own
            Lk = W.lengths_for(cfg["lengths"], seed=cfg["kv_seed"] + 1000 * rank)[:len(L)]
            koff_host = W.offsets_of(Lk, cfg["offsets_dtype"])
            kv = W.jagged_inputs(Lk, H, D, W.SEEDS[cfg["lengths"]] + 500 + 1000 * rank, device=dev)
            inp["k"], inp["v"] = kv["k"], kv["v"]
            koff = torch.from_numpy(koff_host).to(dev)
            st["fwd_flops"] = W.useful_flops("cross", (L, Lk), H=H, D=D)
            st["desc"] = "%s: B=%d, Tq=%d, Tk=%d, H=%d, D=%d, separate q/kv offsets, no mask" % (
                name, len(L), int(off_host[-1]), int(koff_host[-1]), H, D)
        else:
            koff_host, koff = off_host, off
            st["fwd_flops"] = W.useful_flops("varlen", L, H=H, D=D, window=win)
            st["desc"] = "%s: B=%d, T=%d, H=%d, D=%d, window %s, %s dQ" % (
                name, len(L), int(off_host[-1]), H, D, tuple(win), "ordered" if det else "atomic")
        ws_buf = jfa.Plan(koff, H, D, kind="varlen", q_offsets=off, host_offsets=koff_host,
                          host_q_offsets=off_host, window=win, deterministic=det).workspace

        def fwd():
            st["plan"] = jfa.Plan(koff, H, D, kind="varlen", q_offsets=off, host_offsets=koff_host,
                                  host_q_offsets=off_host, window=win, deterministic=det,
                                  workspace=ws_buf, zigzag=zigzag)
            st["o"], st["lse"] = jfa.jfa_varlen_fwd(inp["q"], inp["k"], inp["v"], off, koff,
                                                    window=win, plan=st["plan"])

        def bwd():
            jfa.jfa_varlen_bwd(inp["q"], inp["k"], inp["v"], st["o"], st["lse"], inp["do"], off, koff,
                               window=win, deterministic=det, plan=st["plan"])

        st["check"] = lambda: st["plan"].check()
    elif cfg["kind"] == "sparse":
        L = _gem_lengths(rank) if cfg["lengths"] == "gem" else W.lengths_for(cfg["lengths"])
        if seqs:
            L = L[:seqs]
        off_host = W.offsets_of(L, cfg["offsets_dtype"])
        masks = W.block_masks(L, L, W.MASK_SEEDS[name] + 1000 * rank, density=cfg["density"])
        flat = jfa.pack_block_masks(masks, off_host, off_host)  # an input, like the host offsets
        inp = W.jagged_inputs(L, H, D, W.SEEDS[name] + 1000 * rank, device=dev)
        off = torch.from_numpy(off_host).to(dev)
        ws_buf = jfa.Plan(off, H, D, kind="sparse", host_offsets=off_host, block_masks=flat).workspace
        st["fwd_flops"] = W.useful_flops("sparse", L, H=H, D=D, masks=masks)
        kept = sum(int(m.sum()) for m in masks)
        st["desc"] = ("%s: B=%d, T=%d, H=%d, D=%d, block-causal 128x128 block masks, off-diagonal "
                      "blocks kept with p=%.2f (%d of %d blocks)" % (
                          name, len(L), int(off_host[-1]), H, D, cfg["density"], kept,
                          sum(m.size for m in masks)))

        def fwd():
            st["plan"] = jfa.Plan(off, H, D, kind="sparse", host_offsets=off_host, block_masks=flat,
                                  workspace=ws_buf, zigzag=zigzag)
            kfwd()

        def kfwd():
            st["o"], st["lse"] = jfa.jfa_sparse_fwd(inp["q"], inp["k"], inp["v"], off, off,
                                                    plan=st["plan"])

        def bwd():
            jfa.jfa_sparse_bwd(inp["q"], inp["k"], inp["v"], st["o"], st["lse"], inp["do"], off, off,
                               plan=st["plan"])

        # The kernels alone, on the plan of the last step: the block lists are
        # built on the host in every step (about 3 ms for this batch), longer
        # than the kernels, so the step times above include host time.
        st["kernels"] = (kfwd, bwd)

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
            st["plan"] = jfa.Plan(off, H, D, kind="bcast", Lq=Lq, host_offsets=off_host, zigzag=zigzag)
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
        if cfg.get("rotary"):
            # The forward writes the rotated rows (a rotary layer's saved
            # output): a rotary pass on q and k and the plain forward on them;
            # the backward reads those and rotates dQ, dK back in its
            # epilogue. Modelled bytes are the operation's own (q, k, v read,
            # o, q_rot, k_rot written: 6 tiles); the two-pass forward moves 8.
            # The fp32 tables (2 x L x D/2 x 4 bytes) stay in L2.
            cos, sin = W.rotary_tables(L, D, device=dev)
            st["fwd_bytes"] = 6 * B * L * H * D * 2
            st["desc"] += (", rotary (fp32 tables [L, D/2]; forward: rotary pass writing q_rot, k_rot, "
                           "then the plain forward; backward: rotation fused in its epilogue)")

            def fwd():
                st["o"], st["q_rot"], st["k_rot"] = jfa.blockdiag_rotary_fwd(
                    inp["q"], inp["k"], inp["v"], cos, sin, return_rotated=True)

            def bwd():
                jfa.blockdiag_rotary_bwd(st["q_rot"], st["k_rot"], inp["v"], inp["do"], cos, sin)
        else:
            def fwd():
                jfa.blockdiag_fwd(inp["q"], inp["k"], inp["v"])

            def bwd():
                jfa.blockdiag_bwd(inp["q"], inp["k"], inp["v"], inp["do"])

        st["check"] = lambda: jfa.check_status(device=dev)
    st["inp"] = inp
    st["fwd"], st["bwd"] = fwd, bwd
    st["bwd_flops"] = 2.5 * st["fwd_flops"]
    return st


def _time_steps(st, steps, warmup, stream, sampler=None, barrier=None):
    """Times `steps` fwd+bwd steps of a set-up workload after `warmup` untimed
    ones, with CUDA events on `stream`; `barrier` (multi-rank runs) is called
    on both sides of the timed region. Returns (total ms, median fwd ms,
    median bwd ms, clocks or None)."""
    import torch

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        st["fwd"]()
        if ev is not None:
            ev[1].record(stream)
        st["bwd"]()
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        step()
    st["check"]()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if barrier is not None:
        barrier()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
    # A short device-side spin before the start event lets the host queue the
    # timed steps ahead of the GPU, so host launch latency stays out of the
    # timed region (it holds only the steps' own kernels).
    _spin(stream)
    t0.record(stream)
    for i in range(steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    clk = sampler.stop() if sampler is not None else None
    if barrier is not None:
        barrier()
    st["check"]()
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    return t0.elapsed_time(t1), fwd_ms, bwd_ms, clk


def _fracs(tflops, peak, spec=SPEC_BF16_TFLOPS):
    return {"tflops": round(tflops, 1), "frac_of_peak": round(tflops / peak, 4),
            "frac_of_spec_peak": round(tflops / spec, 4)}


def _dynamic_fwd_ms(st, steps, warmup, stream):
    """Median forward kernel time of a jagged workload under the host static
    schedule (LPT + zigzag lists) and under device-side dynamic scheduling
    with both claim orders, each launched the same way: plans built first,
    W warm-up launches, then K launches queued behind a device-side spin and
    timed with CUDA events."""
    import torch

    import jagged_flash_attention_flashattention_gb300 as jfa

    inp, off = st["inp"], st["plan"].offsets
    H, D = st["H"], st["D"]
    host = st["plan"].host_offsets
    static_plan = jfa.Plan(off, H, D, host_offsets=host)
    runs = {"static": lambda: jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=static_plan)}
    for order in ("device", "lpt"):
        plan = jfa.DynamicPlan(off, H, D, order=order, host_offsets=host)
        runs[order] = (lambda pl: lambda: jfa.jfa_fwd_dynamic(inp["q"], inp["k"], inp["v"], off,
                                                              plan=pl))(plan)
    res = {}
    for name, fn in runs.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        _spin(stream)
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        res[name] = statistics.median(a.elapsed_time(b) for a, b in evs)
    jfa.check_status(static_plan.workspace)
    return res


def _pair_fwd_ms(st, steps, warmup, stream):
    """Median forward kernel time of a jagged D = 128 workload on single CTAs
    (jfa_fwd) and on CTA pairs (jfa_fwd_pair), each launched the same way as
    in _dynamic_fwd_ms."""
    import torch

    import jagged_flash_attention_flashattention_gb300 as jfa

    inp, off = st["inp"], st["plan"].offsets
    H, D = st["H"], st["D"]
    host = st["plan"].host_offsets
    plans = {"single": jfa.Plan(off, H, D, host_offsets=host),
             "pair": jfa.Plan(off, H, D, host_offsets=host, pair=True)}
    res = {}
    for name, plan in plans.items():
        fn = (lambda pl: lambda: jfa.jfa_fwd(inp["q"], inp["k"], inp["v"], off, plan=pl))(plan)
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        _spin(stream)
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        res[name] = statistics.median(a.elapsed_time(b) for a, b in evs)
        plan.check()
    return res


def _kernel_ms(st, steps, warmup, stream):
    """Median fwd and bwd times of a workload's kernel calls on a plan built
    beforehand (st["kernels"]), each call bracketed by CUDA events."""
    import torch

    res = {}
    for op, fn in zip(("fwd", "bwd"), st["kernels"]):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        _spin(stream)
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        res[op] = statistics.median(a.elapsed_time(b) for a, b in evs)
    st["check"]()
    return res


def _other_configs(args, dev, peaks):
    """Every other workload of the method, each timed like the headline one
    (W warm-up and K timed fwd+bwd steps, CUDA events, median per op), plus the
    stress workload under the naive tile order for the LPT + zigzag A/B."""
    import torch

    hbm_peak, tc_peak = peaks
    stream = torch.cuda.current_stream()
    steps, warmup = max(3, min(args.steps, 10)), 3
    out = {}
    for name in ("stress", "bcast", "blockdiag", "blockdiag64", "blockdiag_rotary", "gem_causal",
                 "gem_det", "gem_cross", "gem_rotary", "gem_sparse"):
        st = _setup(name, 0, dev)
        _, f_ms, b_ms, _ = _time_steps(st, steps, warmup, stream)
        ff, bf = st["fwd_flops"], st["bwd_flops"]
        rec = {"workload": st["desc"], "steps": steps,
               "fwd": dict(ms=round(f_ms, 4), **_fracs(ff / f_ms / 1e9, tc_peak)),
               "bwd": dict(ms=round(b_ms, 4), **_fracs(bf / b_ms / 1e9, tc_peak))}
        if st["kind"] == "blockdiag":
            for op, nbytes, ms in (("fwd", st["fwd_bytes"], f_ms), ("bwd", st["bwd_bytes"], b_ms)):
                gbs = nbytes / (ms * 1e-3) / 1e9
                rec[op]["gbps"] = round(gbs, 1)
                rec[op]["frac_of_hbm_peak"] = round(gbs / hbm_peak, 4)
            rec["bytes_note"] = ("modelled bytes (inputs read once, outputs written once) over "
                                 "the measured copy peak")
        if "kernels" in st:  # step times include host-side planning: the kernels alone as well
            km = _kernel_ms(st, steps, warmup, stream)
            rec["kernels_only"] = {
                "note": "plan (host block lists) built before the timed calls",
                "fwd": dict(ms=round(km["fwd"], 4), **_fracs(ff / km["fwd"] / 1e9, tc_peak)),
                "bwd": dict(ms=round(km["bwd"], 4), **_fracs(bf / km["bwd"] / 1e9, tc_peak))}
        out[name] = rec
        if name == "stress":
            dyn = _dynamic_fwd_ms(st, steps, warmup, stream)
            nv = _setup(name, 0, dev, zigzag=False)
            _, nf_ms, nb_ms, _ = _time_steps(nv, steps, warmup, stream)
            out["schedule_ab"] = {
                "workload": st["desc"],
                "fwd_ms_zigzag": round(f_ms, 4), "fwd_ms_naive": round(nf_ms, 4),
                "bwd_ms_zigzag": round(b_ms, 4), "bwd_ms_naive": round(nb_ms, 4),
                "fwd_naive_over_zigzag": round(nf_ms / f_ms, 3),
                "bwd_naive_over_zigzag": round(nb_ms / b_ms, 3),
                # forward kernel alone, each launched the same way: the host
                # LPT + zigzag lists against device-side dynamic scheduling
                # (CTAs claim tiles at run time) in two claim orders
                "fwd_kernel_ms_static_zigzag": round(dyn["static"], 4),
                "fwd_kernel_ms_dynamic_device_order": round(dyn["device"], 4),
                "fwd_kernel_ms_dynamic_lpt_order": round(dyn["lpt"], 4),
                "fwd_dynamic_device_over_static": round(dyn["device"] / dyn["static"], 3),
                "fwd_dynamic_lpt_over_static": round(dyn["lpt"] / dyn["static"], 3)}
            del nv
        if name == "stress":
            out["pair_ab"] = {}
            for pname, pst in (("gem", None), ("stress", st)):
                if pst is None:
                    pst = _setup("gem", 0, dev)
                    pst["fwd"]()  # builds the workload's plan (its host offsets)
                pr = _pair_fwd_ms(pst, steps, warmup, stream)
                # forward kernel alone on single CTAs against CTA pairs
                # (cta_group::2 products, 512-row tiles)
                out["pair_ab"][pname] = {
                    "fwd_kernel_ms_single": round(pr["single"], 4),
                    "fwd_kernel_ms_pair": round(pr["pair"], 4),
                    "pair_over_single": round(pr["pair"] / pr["single"], 3)}
                del pst
        del st
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, tc_peak, tc_sust, peak_src = _peaks()

    st = _setup(args.config, rank, dev, args.seqs, zigzag=args.schedule == "zigzag")
    fwd_flops, bwd_flops = st["fwd_flops"], st["bwd_flops"]
    stream = torch.cuda.current_stream()
    total_ms, fwd_ms, bwd_ms, clk = _time_steps(st, args.steps, args.warmup, stream,
                                                ClockSampler(local),
                                                dist.barrier if ws > 1 else None)
    job_flops, t_max = aggregate_over_ranks(fwd_flops + bwd_flops, total_ms, ws, dev)
    ms_per_step = t_max / args.steps
    value = job_flops / (ms_per_step * 1e-3) / 1e12

    full_gem = args.config == "gem" and not args.seqs
    e2e = _e2e_gem(args, st, dev, ws, ms_per_step) if full_gem else None
    configs = None
    if full_gem and rank == 0 and not args.no_configs:
        del st["inp"]
        configs = _other_configs(args, dev, (hbm_peak, tc_peak))

    if rank == 0:
        bwd_tf = bwd_flops / (bwd_ms * 1e-3) / 1e12
        fwd_tf = fwd_flops / (fwd_ms * 1e-3) / 1e12
        peak = tc_peak  # a short run of back-to-back steps: the burst figure
        if st["kind"] == "blockdiag":
            bw = st["bwd_bytes"] / (bwd_ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "kernel": "blockdiag_bwd", "achieved": round(bw, 1),
                    "peak": hbm_peak, "unit": "GB/s", "frac": round(bw / hbm_peak, 4),
                    "traffic": None, "peak_source": peak_src + " HBM copy",
                    "achieved_note": "modelled bytes (inputs read once, outputs written once) / "
                                     "CUDA-event time; the measured copy peak is not a ceiling"}
        else:
            roof = {"bound": "tensor", "kernel": "jfa_bwd (bwd kernel + dQ cast)",
                    "achieved": round(bwd_tf, 1), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(bwd_tf / peak, 4),
                    "frac_of_spec_peak": round(bwd_tf / SPEC_BF16_TFLOPS, 4),
                    "traffic": BWD_GEM_TRAFFIC if full_gem else None,
                    "peak_source": peak_src + " bf16 burst (cuBLAS); spec peak %.0f TFLOP/s"
                                   % SPEC_BF16_TFLOPS}
        line = {
            "metric": METRIC,
            "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": st["desc"], "parallelism": "replicas (one batch per GPU)",
                       "l2": "inputs larger than L2 (no flush)", "schedule": args.schedule},
            "fwd": dict(ms=round(fwd_ms, 4), **_fracs(fwd_tf, peak)),
            "bwd": dict(ms=round(bwd_ms, 4), **_fracs(bwd_tf, peak)),
            "pct_of_peak": round(100 * value / peak, 2),
            "pct_of_spec_peak": round(100 * value / SPEC_BF16_TFLOPS, 2),
            "roofline": roof,
            "clocks": clk,
            "gpu_launches": (4 if st["kind"] in ("jagged", "varlen", "sparse") else 2) * args.steps,
        }
        if full_gem:
            line["targets"] = {
                op: {"target_frac": tgt, "frac_of_peak": line[op]["frac_of_peak"],
                     "frac_of_spec_peak": line[op]["frac_of_spec_peak"],
                     "met_vs_measured_peak": line[op]["frac_of_peak"] >= tgt,
                     "met_vs_spec_peak": line[op]["frac_of_spec_peak"] >= tgt}
                for op, tgt in (("fwd", 0.50), ("bwd", 0.35))}
        if st["kind"] == "blockdiag":
            line["fwd"]["gbps"] = round(st["fwd_bytes"] / (fwd_ms * 1e-3) / 1e9, 1)
            line["bwd"]["gbps"] = round(st["bwd_bytes"] / (bwd_ms * 1e-3) / 1e9, 1)
        if e2e is not None:
            line["e2e"] = e2e
        if configs is not None:
            line["configs"] = configs
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        if full_gem and not args.no_configs:
            line["scheduler"] = scheduler_times(dev)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _gpu_local_cpus(dev):
    """CPUs on the host NUMA node next to the GPU (from sysfs), or None."""
    import torch
    bus = None
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        try:
            r = subprocess.run(["nvidia-smi", "-i", str(dev.index or 0), "--query-gpu=pci.bus_id",
                                "--format=csv,noheader"], capture_output=True, text=True, timeout=10)
            dom, rest = r.stdout.strip().split(":", 1)
            bus = "%04x:%s" % (int(dom, 16), rest.lower())
        except Exception:
            return None
    try:
        with open("/sys/bus/pci/devices/%s/local_cpulist" % bus) as f:
            text = f.read().strip()
    except Exception:
        return None
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus or None


def _copy_rates(pairs_in, pairs_out, s_in, s_out, reps=3):
    """Bare pinned copies, no kernels: host-to-device alone, device-to-host
    alone and both at once, each over every buffer on its own stream. Returns
    GB/s for each (best of `reps`)."""
    import torch

    def run(groups):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            cur = torch.cuda.current_stream()
            a.record(cur)
            nbytes = 0
            for pairs, streams in groups:
                for (dst, src), sj in zip(pairs, streams):
                    sj.wait_event(a)
                    with torch.cuda.stream(sj):
                        dst.copy_(src, non_blocking=True)
                    nbytes += src.numel() * src.element_size()
            for pairs, streams in groups:
                for sj in streams[:len(pairs)]:
                    cur.wait_stream(sj)
            b.record(cur)
            torch.cuda.synchronize()
            gbs = nbytes / (a.elapsed_time(b) * 1e-3) / 1e9
            best = gbs if best is None else max(best, gbs)
        return best

    return (run([(pairs_in, s_in)]), run([(pairs_out, s_out)]),
            run([(pairs_in, s_in), (pairs_out, s_out)]))


def _e2e_gem(args, st, dev, ws, kernel_ms):
    """Same metric through the public API with host (pinned) buffers: every
    step copies q, k, v, dO and the offsets in and O, dQ, dK, dV out. Steps
    are pipelined the way a training input pipeline would run them: the
    host-to-device copy of step n+1 and the device-to-host copy of step n-1
    run on their own streams while step n's kernels run (two device buffer
    sets; every step still moves all of its own bytes in both directions).
    The same run also times the bare copies with no kernels, so the line
    shows the bound the host link puts on the end-to-end figure."""
    import torch
    import torch.distributed as dist

    import jagged_flash_attention_flashattention_gb300 as jfa

    H, D = st["H"], st["D"]
    inp = st["inp"]
    off_host = st["plan"].host_offsets
    # Pinned buffers on the host NUMA node next to the GPU when sysfs names one
    # (pages are placed where the allocating thread runs).
    affinity = "unchanged"
    local = _gpu_local_cpus(dev)
    try:
        allowed = os.sched_getaffinity(0)
        if local and (local & allowed) and (local & allowed) != allowed:
            os.sched_setaffinity(0, local & allowed)
            affinity = "gpu-local cpus %d of %d" % (len(local & allowed), len(allowed))
        elif local:
            affinity = "all %d allowed cpus are gpu-local" % len(allowed) if local >= allowed else \
                "no gpu-local cpu allowed"
        else:
            affinity = "gpu-local cpus unknown"
    except Exception:
        pass
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

    dev_out = [torch.empty_like(hq, device=dev) for _ in range(4)]
    h2d_gbs, d2h_gbs, both_gbs = _copy_rates(list(zip(d_in[0], (hq, hk, hv, hdo))),
                                             list(zip(h_out[0], dev_out)), s_in, s_out)
    del dev_out
    copy_ms = max(h2d / h2d_gbs, d2h / d2h_gbs, (h2d + d2h) / both_gbs) / 1e6

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
    hidden = (copy_ms + kernel_ms - ms) / min(copy_ms, kernel_ms)
    return {"value": round(val, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 3),
            "overlap": "h2d of step n+1 and d2h of step n-1 run beside step n's kernels",
            "copy_gbps": {"h2d": round(h2d_gbs, 1), "d2h": round(d2h_gbs, 1),
                          "both_directions": round(both_gbs, 1)},
            "copy_bound_ms": round(copy_ms, 3), "kernel_ms": round(kernel_ms, 3),
            "hidden_fraction": round(max(0.0, min(1.0, hidden)), 3),
            "bound": "host link" if copy_ms > kernel_ms else "kernels",
            "host_buffers": affinity}


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
                    choices=["gem", "stress", "bcast", "blockdiag", "blockdiag64", "tiny",
                             "gem_causal", "gem_det", "blockdiag_rotary", "gem_rotary",
                             "gem_sparse", "gem_cross"])
    ap.add_argument("--schedule", default="zigzag", choices=["zigzag", "naive"],
                    help="tile order: host LPT + zigzag deal, or the unsorted round-robin deal")
    ap.add_argument("--no-configs", action="store_true",
                    help="with the GEM workload, skip timing the other workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
