"""Benchmark of one SGA layer (compaction + attention) on B300: prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload headline|vggt|long|tiny]
                    [--impl ours|reference] [--no-e2e] [--no-cpu]

A step is one pass of the whole hot path over one layer of synthetic input: the compaction of
K/V into the kept set (plus the dropped-row sums) and the attention over the kept set with the
diagonal and mean components.  Inputs are resident in HBM when the timed region starts; they
are larger than L2, so no flush is needed between steps.  Times are CUDA events on the launching
stream, bracketed by a barrier and a device synchronise, max over ranks.

Multi-GPU (torchrun, one rank per GPU): the layers of different batch elements are independent
problems, so each rank runs its own layer (weak scaling) and the only collective is the timing
reduction.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (the method has no public implementation to run).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SGA ms/layer and effective TFLOP/s at 800 frames, σ=4 (fraction of bf16 peak)"

WORKLOADS = {
    "headline": dict(desc="SGA layer: N=800 frames x 1374 tokens (37x37 patches + 5 special), H=16, d=64, "
                          "bf16, sigma=4 (2,2), frame 0 and special tokens dense, diagonal + mean "
                          "(leave-one-out, ln count bias)",
                     cfg=dict(B=1, H=16, N=800, sigma=4)),
    "vggt": dict(desc="SGA layer: N=32 frames x 1374 tokens, H=16, d=64, bf16, sigma=4, diag+mean",
                 cfg=dict(B=1, H=16, N=32, sigma=4)),
    "long": dict(desc="SGA layer: N=200 frames x 1374 tokens, H=16, d=64, bf16, sigma=9 (3,3), diag+mean",
                 cfg=dict(B=1, H=16, N=200, sigma=9)),
    "tiny": dict(desc="SGA layer: N=4 frames x 69 tokens (8x8 + 5), H=2, d=64, fp32, sigma=4, diag+mean",
                 cfg=dict(B=1, H=2, N=4, grid_h=8, grid_w=8, sigma=4, dtype="f32")),
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p["bf16_tflops_sustained"]), source="measured")
    except Exception:
        return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:8]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    return rank, world, local


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def layer_flops(cfg, S: int) -> float:
    """Effective FLOPs of one layer: 4 * T * (|S| + 2) * d per (batch, head) with the diagonal
    and mean components (QK^T and PV, 2 FLOP per multiply-add)."""
    extra = 2 if (cfg.diag or cfg.mean) else 0
    return 4.0 * cfg.T * (S + extra) * 64 * cfg.H * cfg.B


def compaction_bytes(cfg, S: int) -> float:
    """Algorithmic HBM bytes of the compaction: read K and V, write K_S and V_S (sums negligible)."""
    es = 2 if cfg.dtype == "bf16" else 4
    return (2.0 * cfg.T + 2.0 * S) * 64 * es * cfg.H * cfg.B


def cpu_oracle_sample(cfg, q, k, v, target_s: float = 12.0, h: int = 0, max_rows: int = 4096):
    """Time the fp64 oracle on sampled query rows of one (batch, head); returns a dict."""
    import oracle
    from subsampled_global_attention_sga_b300.inputs import sample_rows
    s_h, s_w = cfg.s_hw
    op = oracle.plan(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, s_h, s_w, cfg.phase_shift, cfg.ref_frame_dense)
    qh, kh, vh = (x[0, h].float().cpu().numpy() for x in (q, k, v))
    t0 = time.perf_counter()
    sums = oracle.dropped_sums(op, kh, vh)
    t_sums = time.perf_counter() - t0
    calib = min(64, cfg.T)
    rows = sample_rows(cfg.T, cfg.L, calib, seed=77).numpy()
    t0 = time.perf_counter()
    oracle.sga_rows(op, qh[rows], kh, vh, rows, diag=cfg.diag, mean=cfg.mean, sums=sums)
    t_cal = time.perf_counter() - t0
    n = int(max(calib, min(max_rows, cfg.T, calib * max(1.0, (target_s - t_cal) / max(t_cal, 1e-6)))))
    rows = sample_rows(cfg.T, cfg.L, n, seed=78).numpy()
    t0 = time.perf_counter()
    oracle.sga_rows(op, qh[rows], kh, vh, rows, diag=cfg.diag, mean=cfg.mean, sums=sums)
    t_rows = time.perf_counter() - t0
    n = len(rows)
    extra = 2 if (cfg.diag or cfg.mean) else 0
    flops = 4.0 * n * (op.S + extra) * 64
    # per-(batch, head) sums are amortised over all rows of that head in a full layer
    ms_layer = (t_rows / n * cfg.T + t_sums) * cfg.H * cfg.B * 1e3
    return {"value": flops / t_rows / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} query rows of head {h} (of {cfg.T} x {cfg.H}); fp64 C oracle, OpenMP",
            "seconds": t_rows, "extrapolated_ms_per_layer": ms_layer}


def run_ours(args):
    import subsampled_global_attention_sga_b300 as sga
    from subsampled_global_attention_sga_b300.inputs import correlated_qkv

    rank, world, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload]
    cfg = sga.SGAConfig(**wl["cfg"])
    tdt = cfg.torch_dtype
    # each rank its own batch element: independent seeds
    q, k, v = correlated_qkv(1, cfg.H, cfg.N, cfg.L, 64, seed=3 * rank, dtype=tdt, device=dev)
    plan = sga.Plan(cfg, dev)
    K_S, V_S, k_sum, v_sum = plan.compact(k, v)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        plan.compact(k, v, K_S, V_S, k_sum, v_sum)
        if ev is not None:
            ev[1].record(stream)
        plan.forward(q, k, v, K_S, V_S, k_sum, v_sum, out=out)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if sga.device_status(dev) != 0:
        raise RuntimeError("device status not OK after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize(dev)
    with Clocks(dev.index) as clk:
        # a short device-side spin before the first event lets the host enqueue the steps ahead
        # of the GPU, so no event interval contains host launch overhead
        torch.cuda._sleep(int(2e6 * (2 + args.steps)))
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    _barrier(world)
    status = sga.device_status(dev)
    total_ms = _max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    comp_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    clocks = clk.summary()

    flops = layer_flops(cfg, plan.S)
    ms_step = total_ms / args.steps
    value = world * flops / (ms_step * 1e-3) / 1e12
    peaks = _peaks()
    attn_tflops = flops / (attn_ms * 1e-3) / 1e12
    comp_gbs = compaction_bytes(cfg, plan.S) / (comp_ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        qh, kh, vh = (x.cpu().pin_memory() for x in (q, k, v))
        oh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        for _ in range(2):
            sga.layer_from_host(plan, qh, kh, vh, out_host=oh)
        torch.cuda.synchronize(dev)
        _barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            sga.layer_from_host(plan, qh, kh, vh, out_host=oh)
        b.record(stream)
        torch.cuda.synchronize(dev)
        _barrier(world)
        e_ms = _max_over_ranks(a.elapsed_time(b), world, dev) / args.steps
        e2e = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (qh, kh, vh)),
               "d2h_bytes_per_step": oh.numel() * oh.element_size()}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_oracle_sample(cfg, q, k, v)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": wl["desc"], "B_per_rank": cfg.B, "H": cfg.H, "N": cfg.N, "L": cfg.L, "T": cfg.T,
                   "S": plan.S, "sigma": cfg.sigma, "flops_per_layer": flops,
                   "l2": "inputs larger than L2 (Q, K, V %.2f GB each); no flush" % (q.numel() * q.element_size() / 1e9),
                   "parallelism": f"dp{world} (independent layers per rank)"},
        "roofline": {"bound": "tensor", "kernel": "sga::tc::attn_tc_kernel", "achieved": attn_tflops,
                     "peak": peaks["bf16_sus"], "unit": "TFLOP/s", "frac": attn_tflops / peaks["bf16_sus"],
                     "peak_kind": f"bf16 dense sustained ({peaks['source']})",
                     "frac_of_burst": attn_tflops / peaks["bf16"], "traffic": None,
                     "attention_ms": attn_ms},
        "compaction": {"ms": comp_ms, "achieved_gbs": comp_gbs, "bytes": compaction_bytes(cfg, plan.S),
                       "frac_hbm": comp_gbs / peaks["hbm"], "frac_8tbs": comp_gbs / 8000.0,
                       "peak_source": peaks["source"]},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The fp64 CPU oracle, as it stands, on a bounded sample of the workload (rank 0 only)."""
    rank, world, _ = (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0)
    if rank != 0:
        return
    import oracle
    import subsampled_global_attention_sga_b300 as sga
    from subsampled_global_attention_sga_b300.inputs import correlated_qkv
    wl = WORKLOADS[args.workload]
    cfg = sga.SGAConfig(**wl["cfg"])
    # one (batch, head) of the same workload, generated on the host
    q, k, v = correlated_qkv(1, 1, cfg.N, cfg.L, 64, seed=0, dtype=cfg.torch_dtype, device="cpu")
    one = sga.SGAConfig(**dict(wl["cfg"], H=1))
    s_h, s_w = cfg.s_hw
    S = oracle.plan(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, s_h, s_w, cfg.phase_shift, cfg.ref_frame_dense).S
    per_step = max(2.0, min(15.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_sample(one, q, k, v, target_s=per_step / 4)
    vals, secs, rows_ms = [], [], []
    for _ in range(args.steps):
        r = cpu_oracle_sample(one, q, k, v, target_s=per_step)
        vals.append(r["value"])
        secs.append(r["seconds"])
        rows_ms.append(r["extrapolated_ms_per_layer"] * cfg.H)
    value = statistics.mean(vals)
    ms_layer = statistics.mean(rows_ms)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_layer, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl["desc"], "H": cfg.H, "N": cfg.N, "T": cfg.T, "S": S,
                   "flops_per_layer": layer_flops(cfg, S),
                   "note": "each step times the oracle on sampled query rows of one head; ms_per_step is "
                           "extrapolated to the full layer"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{args.steps} steps x sampled query rows of one head, ~{per_step:.0f} s each"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="headline")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
