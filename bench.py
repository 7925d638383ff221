#!/usr/bin/env python
"""Benchmark: one step = the whole hot path of the vocab-parallel LM head on
one batch -- embedding gather of the batch's ids, fused LM head + CE forward,
and its backward (dX, dW) -- on seeded synthetic inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload v128k] [--path fused|split] [--no-cpu-baseline]

``--path fused`` (default) runs the LM head as one vp_lmhead_ce_fwd_bwd call
(tile probabilities saved in fp16, 3 GEMMs per step); ``--path split`` runs
vp_lmhead_ce_fwd + vp_lmhead_ce_bwd (logits recomputed, 4 GEMMs per step).
The other path is also timed briefly after the timed region and reported
under ``other_path`` (not part of ``value``).

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs the same
step on its own seeded batch (weak scaling, no collective on the data path;
the only collectives are the timing barrier and the max over ranks).

``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (the baseline these pages give no faster
implementation of); only rank 0 runs it.
"""
import argparse
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

METRIC = "fused LM-head+CE fwd+bwd tokens/s and % of bf16 tensor peak at V=128256"
UNIT = "tokens/s"
GEMM_STAGES = {"split": ("lse_stats_gemm", "dz_recompute_gemm", "dw_gemm", "dx_gemm"),
               "fused": ("lse_p_gemm", "dw_gemm", "dx_gemm")}
# library stages of the LM head's forward and backward (the gather is timed apart)
FWD_STAGES = ("lse_stats_gemm", "lse_p_gemm", "lse_merge", "loss_mean", "upstream_scale")
BWD_STAGES = ("dz_recompute_gemm", "dz_from_p", "x_transpose", "dw_gemm", "dx_gemm")


def fwd_bwd_ms(stages, steps):
    """(forward ms, backward ms) per step from the library's per-kernel events.
    In the fused call the upstream scale runs with the forward; the p -> dZ
    pass and the two gradient GEMMs are its backward."""
    f = sum(stages.get(s, (0.0, 0))[0] for s in FWD_STAGES) / steps
    b = sum(stages.get(s, (0.0, 0))[0] for s in BWD_STAGES) / steps
    return round(f, 4), round(b, 4)


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="v128k")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU work budget of the oracle baseline")
    p.add_argument("--e2e-steps", type=int, default=0,
                   help="steps of the end-to-end loop (0: as many as the timed region, so both see the same "
                        "power-capped clocks)")
    p.add_argument("--path", choices=["fused", "split"], default="fused",
                   help="fused: one fwd+bwd call with saved probabilities; split: fwd, then bwd with recompute")
    p.add_argument("--other-path-steps", type=int, default=5, help="timed steps of the other path (0: skip)")
    p.add_argument("--embed-iters", type=int, default=20, help="launches per case of the gather microbench (0: skip)")
    p.add_argument("--gemm-variant", choices=["single", "pair", "single128", "mcast"], default="single",
                   help="tcgen05 GEMM form: the default (one SM per logits and dX tile, dW^T on SM pairs), SM "
                        "pairs for every GEMM, 128x256 tiles on one SM for every GEMM, or the default with the "
                        "logits GEMMs in TMA-multicast clusters")
    p.add_argument("--token-chunk", type=int, default=0,
                   help="fused path: token rows per chunk the workspace is sized for (0: the library's bounded "
                        "default, saved probabilities <= 1.25 GiB; N: all tokens at once)")
    p.add_argument("--vocab-chunk", type=int, default=0,
                   help="split path: vocab ids per backward chunk (0: the library's default, one shard V/T; "
                        "V: the whole vocabulary at once)")
    p.add_argument("--unbounded-steps", type=int, default=5,
                   help="timed steps of each path with one chunk (all N tokens / all V ids) for comparison (0: skip)")
    p.add_argument("--configs", default="minimind,v32k,v128k,v152k",
                   help="workloads of the per-config throughput table ('' to skip)")
    args = p.parse_args()
    if args.e2e_steps <= 0:
        args.e2e_steps = args.steps
    return args


# DRAM bytes (read + write) per GEMM stage (one 2NHV contraction, summed over
# its token-chunk launches) of the tcgen05 GEMM kernels in the fused v128k step
# with the default bounded workspace, from one ncu capture
# (profiles/launches_fused_step_v128k.md: mean of the three stages over four
# steps).  They describe the kernels built from the sources hashed here; once
# those change, `traffic` is reported as null until a new capture replaces the
# number.
GEMM_TRAFFIC = {"workload": "v128k", "path": "fused", "gemm_variant": "single", "token_chunk": 0,
                "bytes_per_stage": 17.25e9,
                "by_stage": {"lse_p_gemm": 9.06e9, "dw_gemm": 28.07e9, "dx_gemm": 14.63e9},
                "sources": ("vocab_lm_head_vp_b300/csrc/ce_bf16.cu", "vocab_lm_head_vp_b300/csrc/ptx.cuh",
                            "vocab_lm_head_vp_b300/csrc/umma_gemm.cuh", "vocab_lm_head_vp_b300/csrc/umma_gemm_2sm.cuh"),
                "sha256": "df4529958c82f8e67c44fe513afdfe4a481f4678d5a030decd4806fe63e306d3"}


def gemm_traffic(workload, path, variant, token_chunk):
    """ncu DRAM bytes per GEMM stage if they were taken on this kernel and step, else None."""
    import hashlib
    t = GEMM_TRAFFIC
    if (workload, path, variant, token_chunk) != (t["workload"], t["path"], t["gemm_variant"], t["token_chunk"]):
        return None
    h = hashlib.sha256()
    for f in t["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return t["bytes_per_stage"] if h.hexdigest() == t["sha256"] else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.out = None

    def start(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        sm, smax, power, reasons = [], [], [], set()
        for line in self.out.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, v in zip(self.REASONS, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.out.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


# ------------------------------------------------------------------ ranks
def rank_env():
    """(rank, world size, local rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(wl, rank):
    """Each rank draws its own batch: weak scaling over independent batches."""
    return wl.seed + rank


def max_over_ranks(x, world, device=None):
    """The slowest rank's time (the job's time); a no-op on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, steps, seconds):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / seconds


# ------------------------------------------------------------------ oracle timing (host cores)
def oracle_tokens_per_s(inp, budget_s):
    """Time the float64 oracle (fwd + bwd, exactly as it stands) on a leading
    sample of the batch's tokens sized to about budget_s seconds."""
    import oracle.ref as ref
    wl = inp.wl
    W64 = np.asarray(inp.W, dtype=np.float64)   # input preparation, not timed
    X64 = np.asarray(inp.X, dtype=np.float64)

    def run(n):
        t0 = time.perf_counter()
        ref.lmhead_ce_backward(X64[:n], W64, inp.targets[:n], wl.V)
        return time.perf_counter() - t0

    n = 2
    t = run(n)
    while t < budget_s / 8 and n < wl.N:
        n = min(wl.N, n * 4)
        t = run(n)
    if t < budget_s / 2 and n < wl.N:
        n = min(wl.N, max(n + 1, int(n * budget_s / max(t, 1e-3) * 0.7)))
        t = run(n)
    return n / t, n, t


def embed_roofline(in_step_gbs, micro, peaks):
    """The gather's bandwidth: the uniform-id V128k launch with L2 flushed is the
    headline (no row repeats); the Zipf and V152k cases and the in-step figure
    (event overhead included, L2 warm) are reported beside it."""
    r = {"kernel": "embed_gather_kernel", "bound": "hbm", "unit": "GB/s", "peak": peaks["hbm_gbs"],
         "in_step_gbs": in_step_gbs}
    if micro:
        a = micro["v128k_uniform"]["GB/s"]
        r.update({"achieved": a, "frac": a / peaks["hbm_gbs"], "frac_of_8TBs": a / 8000.0,
                  "workload": ("v128k shape (N=16384, H=4096, V=128256), uniform ids, L2 flushed before each "
                               "launch, differential timing (flush+gather minus flush)"),
                  "cases": micro})
    else:
        r.update({"achieved": in_step_gbs, "frac": in_step_gbs / peaks["hbm_gbs"],
                  "workload": "in-step launch, Zipf ids (repeated rows hit in L2)"})
    return r


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    import synth
    rank, _, _ = rank_env()
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(wl)
    # each step: the oracle on a bounded sample sized so that the run ends in a few minutes
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    _, n, _ = oracle_tokens_per_s(inp, per_step)
    import oracle.ref as ref
    W64 = np.asarray(inp.W, dtype=np.float64)
    X64 = np.asarray(inp.X[:n], dtype=np.float64)
    for _ in range(args.warmup):
        ref.lmhead_ce_backward(X64, W64, inp.targets[:n], wl.V)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ref.lmhead_ce_backward(X64, W64, inp.targets[:n], wl.V)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    sample = f"first {n} of {wl.N} tokens per step, full H={wl.H} and V={wl.V}, float64 NumPy fwd+bwd"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores_used(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def workload_config(wl):
    return {"workload": f"{wl.name}: N={wl.N} H={wl.H} V={wl.V} T={wl.T} {wl.dtype}, targets {wl.targets}"
                        + (f", {int(wl.ignore_frac * 100)}% ignore_index" if wl.ignore_frac else ""),
            "N": wl.N, "H": wl.H, "V": wl.V, "T": wl.T, "dtype": wl.dtype,
            "l2": ("no flush: inputs larger than L2 (W %.2f GB, X %.0f MB; L2 126 MB)" if wl.V * wl.H * 2 > 126e6
                   else "inputs fit in L2 (W %.2f GB, X %.0f MB); no flush") % (wl.V * wl.H * 2 / 1e9,
                                                                                 wl.N * wl.H * 2 / 1e6)}


# ------------------------------------------------------------------ embedding gather alone
def embed_microbench(vp, dev, iters=20):
    """vp_embed_fwd at the V128k and V152k shapes, uniform and Zipf(1.1) ids,
    with the L2 flushed (a 256 MB write) before every launch.  Differential
    timing on the launching stream: `iters` x (flush, gather) between one pair
    of CUDA events, minus `iters` x flush alone, so per-launch event overhead
    (several microseconds against a ~40 us kernel) stays out.  Algorithmic
    bytes per launch: read N rows + write N rows + N int64 ids."""
    import torch
    import synth
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for name in ("v128k", "v152k"):
        wl = synth.WORKLOADS[name]
        g = torch.Generator(device=dev).manual_seed(wl.seed)
        W = torch.randn(wl.V, wl.H, generator=g, device=dev).to(torch.bfloat16)
        o = torch.empty((wl.N, wl.H), dtype=torch.bfloat16, device=dev)
        rng = np.random.default_rng(wl.seed)
        for kind, ids in (("uniform", rng.integers(0, wl.V, wl.N)), ("zipf", synth.zipf_ids(rng, wl.N, wl.V, 1.1))):
            idt = torch.from_numpy(ids).to(dev)

            def loop(with_gather):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record()
                for _ in range(iters):
                    flush.zero_()
                    if with_gather:
                        vp.embed_fwd(idt, W, wl.T, out=o)
                e1.record()
                torch.cuda.synchronize()
                return e0.elapsed_time(e1)

            loop(True)   # warm-up
            both = [loop(True) for _ in range(3)]
            alone = [loop(False) for _ in range(3)]
            ms = (statistics.median(both) - statistics.median(alone)) / iters
            nbytes = 2.0 * wl.N * wl.H * 2 + 8.0 * wl.N
            out[f"{name}_{kind}"] = {"N": wl.N, "H": wl.H, "V": wl.V, "ms": ms, "GB/s": nbytes / (ms / 1e3) / 1e9,
                                     "rate": ("L2-assisted: repeated Zipf ids hit rows already in L2, so this is "
                                              "not an HBM rate" if kind == "zipf" else
                                              "HBM: distinct rows, L2 flushed before each launch")}
        del W, o
    return out


def embed_bwd_microbench(vp, dev, iters=20):
    """vp_embed_bwd (accumulate into the tied weight's fp32 gradient) at the
    V128k shape with the workload's Zipf ids and with uniform ids, L2 flushed
    before every call, differential timing as in embed_microbench.
    Algorithmic bytes: read dOut (N x H bf16) and the ids, read and write
    every touched fp32 row of dW once."""
    import torch
    import synth
    wl = synth.WORKLOADS["v128k"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    G = torch.randn(wl.N, wl.H, generator=g, device=dev).to(torch.bfloat16)
    dW = torch.zeros((wl.V, wl.H), dtype=torch.float32, device=dev)
    ws = torch.empty(vp._load().vp_embed_bwd_workspace_size(wl.N, wl.H, wl.V, wl.T, vp.VP_BF16),
                     dtype=torch.uint8, device=dev)
    rng = np.random.default_rng(wl.seed)
    out = {}
    for kind, ids in (("zipf", synth.zipf_ids(rng, wl.N, wl.V, 1.1)), ("uniform", rng.integers(0, wl.V, wl.N))):
        idt = torch.from_numpy(ids).to(dev)

        def loop(what):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            for _ in range(iters):
                flush.zero_()
                if what == "call":
                    vp.embed_bwd(idt, G, wl.V, wl.T, dW=dW, accumulate=True, workspace=ws)
                elif what == "planned":
                    vp.embed_bwd_planned(ws, G, wl.V, wl.T, dW=dW, accumulate=True)
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)

        loop("call")   # warm-up; leaves the plan of these ids in ws
        call = [loop("call") for _ in range(3)]
        planned = [loop("planned") for _ in range(3)]
        alone = [loop(None) for _ in range(3)]
        ms = (statistics.median(call) - statistics.median(alone)) / iters
        ms_sums = (statistics.median(planned) - statistics.median(alone)) / iters
        distinct = len(np.unique(ids))
        nbytes = wl.N * wl.H * 2.0 + 8.0 * wl.N + 2.0 * distinct * wl.H * 4
        out[kind] = {"ms": ms, "distinct_ids": distinct, "alg_bytes": nbytes, "GB/s": nbytes / (ms / 1e3) / 1e9,
                     "sums_ms": ms_sums, "sums_GB/s": (nbytes - 8.0 * wl.N) / (ms_sums / 1e3) / 1e9,
                     "note": "ms / GB/s: the whole vp_embed_bwd call (sort of the ids + sums); sums_*: "
                             "vp_embed_bwd_planned alone, the sort done ahead by vp_embed_bwd_plan"}
    del G, dW, ws
    return out


# ------------------------------------------------------------------ every config's throughput
def config_table(vp, dev, names, rank, world, barrier):
    """Both LM-head paths at each named workload's shape with the library's
    default (bounded) workspaces: tokens/s, algorithmic (6NHV) and executed
    TFLOP/s, % of the measured bf16 burst peak.  X and W are drawn on the device
    from a seeded generator (N(0,1) and N(0,0.02^2), rounded to bf16), targets on
    the host (uniform or Zipf(1.1), ignored positions) -- the workloads'
    distributions; parity of these shapes is the tests' business.  Each case runs
    about half a second of steps."""
    import torch
    import synth
    if not names:
        return None
    peaks = load_peaks()
    rows = []
    for name in names:
        wl = synth.WORKLOADS[name]
        N, H, V, T = wl.N, wl.H, wl.V, wl.T
        g = torch.Generator(device=dev).manual_seed(wl.seed + rank)
        X = torch.randn(N, H, generator=g, device=dev).to(torch.bfloat16)
        W = (torch.randn(V, H, generator=g, device=dev) * wl.w_std).to(torch.bfloat16)
        rng = np.random.default_rng(wl.seed + rank)
        yn = synth.zipf_ids(rng, N, V, wl.zipf_s) if wl.targets == "zipf" else rng.integers(0, V, N)
        if wl.ignore_frac:
            yn[rng.choice(N, int(wl.ignore_frac * N), replace=False)] = synth.IGNORE_INDEX
        y = torch.from_numpy(yn.astype(np.int64)).to(dev)
        o = {"loss": torch.empty(N, device=dev), "lse": torch.empty(N, device=dev),
             "mean": torch.empty(1, device=dev), "n_bad": torch.empty(1, dtype=torch.int32, device=dev),
             "dX": torch.empty_like(X), "dW": torch.empty((V, H), device=dev)}
        for path in ("fused", "split"):
            if path == "fused":
                ws = [torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 2), dtype=torch.uint8, device=dev)]
                run = lambda: vp.lmhead_ce_fwd_bwd(X, W, y, T, workspace=ws[0], out=o)
            else:
                ws = [torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 0), dtype=torch.uint8, device=dev),
                      torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 1), dtype=torch.uint8, device=dev)]

                def run():
                    vp.lmhead_ce_fwd(X, W, y, T, workspace=ws[0], out=o)
                    vp.lmhead_ce_bwd(X, W, y, o["lse"], T, workspace=ws[1], dX=o["dX"], dW=o["dW"])
            for _ in range(3):
                run()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize()
            steps = int(min(200, max(3, 500.0 / max(e0.elapsed_time(e1), 1e-3))))
            barrier()
            e0.record()
            for _ in range(steps):
                run()
            e1.record()
            torch.cuda.synchronize()
            ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
            assert all(vp.read_device_status(w) == 0 for w in ws)
            # the same step captured once in a CUDA graph and replayed: the launches
            # cost no host time, so a small workload shows its device time
            graph = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(side):
                run()
            torch.cuda.current_stream(dev).wait_stream(side)
            with torch.cuda.graph(graph):
                run()
            graph.replay()
            torch.cuda.synchronize()
            barrier()
            e0.record()
            for _ in range(steps):
                graph.replay()
            e1.record()
            torch.cuda.synchronize()
            ms_graph = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
            assert all(vp.read_device_status(w) == 0 for w in ws)
            del graph
            alg = 6.0 * N * H * V / (ms / 1e3) / 1e12
            exe = (6.0 if path == "fused" else 8.0) * N * H * V / (ms / 1e3) / 1e12
            rows.append({"workload": name, "path": path, "N": N, "H": H, "V": V, "T": T, "steps": steps,
                         "ms_per_step": ms, "tokens_per_s": job_tokens_per_s(N, world, 1, ms / 1e3),
                         "tflops_algorithmic": alg, "tflops_executed": exe,
                         "pct_bf16_burst_algorithmic": 100.0 * alg / peaks["bf16_tflops"],
                         "pct_bf16_burst_executed": 100.0 * exe / peaks["bf16_tflops"],
                         "ms_per_step_graph": ms_graph,
                         "pct_bf16_burst_algorithmic_graph": 100.0 * 6.0 * N * H * V / (ms_graph / 1e3) / 1e12
                         / peaks["bf16_tflops"],
                         "workspace_bytes": int(sum(w.numel() for w in ws)),
                         "l2": "inputs fit in L2" if (N + V) * H * 2 < 100e6 else "inputs larger than L2"})
            del ws, run
        del X, W, y, o
        torch.cuda.empty_cache()
    return {"note": "library default workspaces (fused: saved probabilities <= 1.25 GiB; split: one shard's dZ); "
                    "X, W drawn on the device; no L2 flush (MiniMind's inputs stay in L2); ms_per_step: the "
                    "calls issued from Python every step; ms_per_step_graph: the same calls captured once in a "
                    "CUDA graph and replayed", "rows": rows}


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    import synth
    import vocab_lm_head_vp_b300 as vp
    from vocab_lm_head_vp_b300 import build

    rank, world, local = rank_env()
    if rank == 0:
        build.build()   # libvp.so is a build product: make it if missing or stale (no-op otherwise)
    if world > 1:
        # the other ranks wait (bounded) until rank 0's build is in place
        t_wait = time.time()
        while not build.up_to_date():
            if time.time() - t_wait > 900:
                raise RuntimeError("libvp.so was not built by rank 0 within 900 s")
            time.sleep(1.0)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    vp.set_gemm_variant({"single": 0, "pair": 1, "single128": 2, "mcast": 3}[args.gemm_variant])
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    wl = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(wl, seed=rank_seed(wl, rank))
    N, H, V, T = wl.N, wl.H, wl.V, wl.T
    to = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    X = to(inp.X_bits).to(dev)
    W = to(inp.W_bits).to(dev)
    y = torch.from_numpy(inp.targets).to(dev)
    emb = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
    fo = {"loss": torch.empty(N, dtype=torch.float32, device=dev),
          "lse": torch.empty(N, dtype=torch.float32, device=dev),
          "mean": torch.empty(1, dtype=torch.float32, device=dev),
          "n_bad": torch.empty(1, dtype=torch.int32, device=dev)}
    dX = torch.empty_like(X)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    fo["dX"], fo["dW"] = dX, dW

    def make_step(path, chunk=None):
        """One step of the given path and the workspaces it uses.  chunk: token
        rows (fused) or vocab ids (split) the workspace is sized for; None takes
        the command line's, 0 the library's bounded default."""
        if path == "fused":
            tc = args.token_chunk if chunk is None else chunk
            ws = torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 2, tc), dtype=torch.uint8, device=dev)

            def step(Xs, ys):
                vp.embed_fwd(ys, W, T, out=emb)
                vp.lmhead_ce_fwd_bwd(Xs, W, ys, T, workspace=ws, out=fo)
            return step, [ws]
        vc = args.vocab_chunk if chunk is None else chunk
        wsf = torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 0), dtype=torch.uint8, device=dev)
        wsb = torch.empty(vp.workspace_size(N, H, V, T, vp.VP_BF16, 1, vc), dtype=torch.uint8, device=dev)

        def step(Xs, ys):
            vp.embed_fwd(ys, W, T, out=emb)
            vp.lmhead_ce_fwd(Xs, W, ys, T, workspace=wsf, out=fo)
            vp.lmhead_ce_bwd(Xs, W, ys, fo["lse"], T, workspace=wsb, dX=dX, dW=dW)
        return step, [wsf, wsb]

    def time_path(path, chunk, steps):
        """Brief timing of one path: ms per step, forward / backward ms, GEMM
        chunks per step, workspace bytes."""
        ostep, ows = make_step(path, chunk)
        for _ in range(2):
            ostep(X, y)
        torch.cuda.synchronize()
        barrier()
        vp.stage_timing_enable(256 * steps + 64)
        e0.record()
        for _ in range(steps):
            ostep(X, y)
        e1.record()
        torch.cuda.synchronize()
        ost = vp.stage_timing_read()
        vp.stage_timing_enable(0)
        oms = max_over_ranks(e0.elapsed_time(e1), world, dev) / steps
        assert all(vp.read_device_status(w) == 0 for w in ows)
        ofwd, obwd = fwd_bwd_ms(ost, steps)
        r = {"path": path, "steps": steps, "ms_per_step": oms, "value": job_tokens_per_s(N, world, 1, oms / 1e3),
             "unit": UNIT, "fwd_ms": ofwd, "bwd_ms": obwd, "chunks": ost.get("dw_gemm", (0, 0))[1] / steps,
             "workspace_bytes": int(sum(w.numel() for w in ows)),
             "pct_bf16_burst_algorithmic": 100.0 * 6.0 * N * H * V / (oms / 1e3) / 1e12 / load_peaks()["bf16_tflops"],
             "stages_ms_per_step": {k: round(v[0] / steps, 4) for k, v in ost.items() if v[1]}}
        del ostep, ows
        torch.cuda.empty_cache()
        return r

    step, workspaces = make_step(args.path)
    ws_bytes = int(sum(w.numel() for w in workspaces))
    for _ in range(args.warmup):
        step(X, y)
    torch.cuda.synchronize()
    assert all(vp.read_device_status(w) == 0 for w in workspaces)

    # ---------------- timed region
    uuid = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else None)
    vp.stage_timing_enable(256 * args.steps + 64)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        step(X, y)
    e1.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    stages = vp.stage_timing_read()
    vp.stage_timing_enable(0)
    ms = max_over_ranks(ms, world, dev)

    # ---------------- end to end through host buffers (X, targets in; loss out)
    # As a training loop would: step i+1's inputs are copied from pinned host
    # memory on a copy stream into the other of two device buffers while step i
    # computes; each step's per-token loss and mean are read back to the host.
    Xh = to(inp.X_bits).pin_memory()
    yh = torch.from_numpy(inp.targets).pin_memory()
    loss_h = torch.empty(N, dtype=torch.float32).pin_memory()
    mean_h = torch.empty(1, dtype=torch.float32).pin_memory()
    Xd = [torch.empty_like(X) for _ in range(2)]
    yd = [torch.empty_like(y) for _ in range(2)]
    ready = [torch.cuda.Event() for _ in range(2)]   # inputs of a buffer have landed
    free = [torch.cuda.Event() for _ in range(2)]    # the step reading a buffer has finished
    compute, copier = torch.cuda.current_stream(dev), torch.cuda.Stream(dev)

    def copy_in(b):
        with torch.cuda.stream(copier):
            copier.wait_event(free[b])
            Xd[b].copy_(Xh, non_blocking=True)
            yd[b].copy_(yh, non_blocking=True)
            ready[b].record(copier)

    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    copy_in(0)
    for i in range(args.e2e_steps):
        b = i % 2
        compute.wait_event(ready[b])
        step(Xd[b], yd[b])
        free[b].record(compute)
        if i + 1 < args.e2e_steps:
            copy_in(1 - b)
        loss_h.copy_(fo["loss"], non_blocking=True)
        mean_h.copy_(fo["mean"], non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, dev)
    h2d = Xh.numel() * 2 + yh.numel() * 8
    d2h = loss_h.numel() * 4 + 4
    assert all(vp.read_device_status(w) == 0 for w in workspaces)

    emb_micro = embed_microbench(vp, dev, args.embed_iters) if args.embed_iters > 0 else None
    emb_bwd_micro = embed_bwd_microbench(vp, dev, args.embed_iters) if args.embed_iters > 0 else None

    # ---------------- the other path, briefly (reported beside, not in `value`)
    other = None
    if args.other_path_steps > 0:
        opath = "split" if args.path == "fused" else "fused"
        other = time_path(opath, 0, args.other_path_steps)
    # ---------------- both paths with one chunk (all N tokens, all V ids): the memory bound's cost
    unbounded = None
    if args.unbounded_steps > 0:
        unbounded = {"fused": time_path("fused", N, args.unbounded_steps),
                     "split": time_path("split", V, args.unbounded_steps)}
    del step, workspaces
    torch.cuda.empty_cache()
    table = config_table(vp, dev, [c for c in args.configs.split(",") if c], rank, world, barrier)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks = load_peaks()
    sec = ms / 1e3
    value = job_tokens_per_s(N, world, args.steps, sec)
    alg = 6.0 * N * H * V          # fwd 2NHV + dX 2NHV + dW 2NHV
    # the split path also recomputes the logits in the backward
    exe = (8.0 if args.path == "split" else 6.0) * N * H * V
    gstages = GEMM_STAGES[args.path]
    gemm_ms = sum(stages[s][0] for s in gstages)
    gemm_n = sum(stages[s][1] for s in gstages)
    # every step's GEMM launches together do 2NHV per stage (a stage may run as several
    # token or vocab chunks): achieved = those flops / the launches' time
    gemm_flops = 2.0 * N * H * V * len(gstages) * args.steps
    achieved = gemm_flops / (gemm_ms / 1e3) / 1e12
    emb_ms, emb_n = stages["embed_gather"]
    emb_bytes = 2.0 * N * H * 2 + 8.0 * N
    emb_gbs = emb_bytes / (emb_ms / max(1, emb_n) / 1e3) / 1e9
    # operands once + outputs once, averaged over the step's GEMM launches
    lse_b = N * H * 2 + V * H * 2 + (N * V * 2 if args.path == "fused" else 0)
    dz_b = N * H * 2 + V * H * 2 + N * V * 2               # split path's recompute launch
    dw_b = N * V * 2 + N * H * 2 + V * H * 4
    dx_b = N * V * 2 + V * H * 2 + N * H * 2
    gemm_alg_bytes = ((lse_b + dw_b + dx_b) / 3 if args.path == "fused" else (lse_b + dz_b + dw_b + dx_b) / 4)
    gemm_launches_per_stage = gemm_n / max(1, len(gstages) * args.steps)   # > 1 when a stage runs in chunks
    extra = {}
    if args.path == "fused" and stages.get("dz_from_p", (0.0, 0))[1] > 0:
        dzp_ms, dzp_n = stages["dz_from_p"]
        valid_rows = int(((inp.targets >= 0) & (inp.targets < V)).sum())
        # read fp16 p, one fp32 tile maximum per 256 columns, and write bf16 dZ for valid rows;
        # write zeros for ignored ones
        dzp_bytes = (4.0 * valid_rows + 2.0 * (N - valid_rows)) * V + 4.0 * valid_rows * -(-V // 256)
        # those bytes are the whole batch's, moved by the step's launches (one per token chunk)
        dzp_gbs = dzp_bytes * args.steps / (dzp_ms / 1e3) / 1e9
        extra["roofline_dz_from_p"] = {"kernel": "dz_from_p_kernel", "bound": "hbm", "achieved": dzp_gbs,
                                       "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": dzp_gbs / peaks["hbm_gbs"]}
    launches = sum(c for _, c in stages.values())
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) X, N(0,0.02^2) W, Zipf targets)",
        "config": dict(workload_config(wl), parallelism=f"replicas x{world}, no data-path collective",
                       path=args.path, gemm_variant=args.gemm_variant, workspace_bytes=ws_bytes,
                       chunks_per_step=gemm_launches_per_stage,
                       chunking=("token chunks; saved fp16 probabilities bounded by the workspace"
                                 if args.path == "fused" else "vocab chunks; bf16 dZ of one chunk at a time")),
        "tflops_algorithmic": alg * args.steps / sec / 1e12,
        "tflops_executed": exe * args.steps / sec / 1e12,
        "pct_bf16_peak_algorithmic": 100.0 * alg * args.steps / sec / 1e12 / peaks["bf16_tflops"],
        "pct_bf16_peak_executed": 100.0 * exe * args.steps / sec / 1e12 / peaks["bf16_tflops"],
        "roofline": {"kernel": ("umma_gemm_kernel (tcgen05; 3 launches/step: lse stats + saved p, dW, dX)"
                                if args.path == "fused" else
                                "umma_gemm_kernel (tcgen05; 4 launches/step: lse stats, dZ recompute, dW, dX)"),
                     "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "peak_kind": f"bf16 burst ({peaks['source']})",
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "peak_sustained": peaks["bf16_tflops_sustained"],
                     "traffic": gemm_traffic(wl.name, args.path, args.gemm_variant, args.token_chunk),
                     "launches_per_gemm_stage": gemm_launches_per_stage,
                     "traffic_unit": "bytes per GEMM stage (one 2NHV contraction; ncu dram read + write, "
                                     "summed over the stage's launches)",
                     "algorithmic_bytes_per_stage": gemm_alg_bytes},
        "roofline_embed": embed_roofline(emb_gbs, emb_micro, peaks),
        "embed_bwd": None if emb_bwd_micro is None else {
            "kernel": "vp_embed_bwd (key sort + run sums + cross-run sums), accumulate into fp32 dW",
            "workload": "v128k shape, L2 flushed before each call, differential timing", "bound": "hbm",
            "unit": "GB/s",
            "peak": peaks["hbm_gbs"], "cases": emb_bwd_micro},
        **extra,
        "stages_ms_per_step": {k: round(v[0] / args.steps, 4) for k, v in stages.items() if v[1]},
        "fwd_ms_per_step": fwd_bwd_ms(stages, args.steps)[0],
        "bwd_ms_per_step": fwd_bwd_ms(stages, args.steps)[1],
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": {"value": job_tokens_per_s(N, world, args.e2e_steps, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "X and targets copied from pinned host memory every step (on a copy stream, into the "
                        "other of two device buffers while the previous step computes) and the loss read back "
                        "every step; the weight W is model state resident in HBM"},
        "other_path": other,
        "unbounded": unbounded,
        "configs": table,
    }
    if world == 1 and not args.no_cpu_baseline:
        v, n, t = oracle_tokens_per_s(inp, args.cpu_seconds)
        result["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores_used(), "kind": "oracle",
                                  "sample": f"first {n} of {N} tokens, full H and V, float64 NumPy fwd+bwd, "
                                            f"{t:.1f} s"}
    print(json.dumps(result))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
