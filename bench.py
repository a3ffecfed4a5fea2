"""Benchmark of one SGA layer (compaction + attention) on B300: prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME | --workload sweep]
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SGA ms/layer and effective TFLOP/s at 800 frames, σ=4 (fraction of bf16 peak)"

WORKLOADS = {
    "headline": dict(kind="sga",
                     desc="SGA layer: N=800 frames x 1374 tokens (37x37 patches + 5 special), H=16, d=64, "
                          "bf16, sigma=4 (2,2), frame 0 and special tokens dense, diagonal + mean "
                          "(leave-one-out, ln count bias)",
                     cfg=dict(B=1, H=16, N=800, sigma=4)),
    "headline_phase": dict(kind="sga",
                           desc="SGA layer with the per-frame phase-shifted grid: N=800 frames x 1374 tokens, "
                                "H=16, d=64, bf16, sigma=4 (2,2), frame 0 and special tokens dense, diagonal + mean",
                           cfg=dict(B=1, H=16, N=800, sigma=4, phase_shift=True)),
    "vggt": dict(kind="sga", desc="SGA layer: N=32 frames x 1374 tokens, H=16, d=64, bf16, sigma=4, diag+mean",
                 cfg=dict(B=1, H=16, N=32, sigma=4)),
    "long": dict(kind="sga", desc="SGA layer: N=200 frames x 1374 tokens, H=16, d=64, bf16, sigma=9 (3,3), diag+mean",
                 cfg=dict(B=1, H=16, N=200, sigma=9)),
    "tiny": dict(kind="sga", desc="SGA layer: N=4 frames x 69 tokens (8x8 + 5), H=2, d=64, fp32, sigma=4, diag+mean",
                 cfg=dict(B=1, H=2, N=4, grid_h=8, grid_w=8, sigma=4, dtype="f32")),
    "general": dict(kind="sga",
                    desc="SGA layer, generalised kept set: N=200 frames x 1374 tokens, H=16, d=64, bf16, "
                         "per-axis sigma_b = 1.3 with phase shift, frame 0 + special tokens dense, 10 % of "
                         "the tokens protected, diagonal + mean",
                    cfg=dict(B=1, H=16, N=200), general=dict(sigma=(13, 10), phase=True, protected=0.10)),
    "rope": dict(kind="sga",
                 desc="SGA layer with fused 2D RoPE (base 100, position offset 1): N=800 frames x 1374 "
                      "tokens, H=16, d=64, bf16, sigma=4, diag+mean",
                 cfg=dict(B=1, H=16, N=800, sigma=4, rope=True, rope_base=100.0, rope_pos_offset=1)),
    "rope_long": dict(kind="sga",
                      desc="SGA layer with fused 2D RoPE: N=200 frames x 1374 tokens, H=16, d=64, bf16, "
                           "sigma=9, diag+mean",
                      cfg=dict(B=1, H=16, N=200, sigma=9, rope=True, rope_base=100.0, rope_pos_offset=1)),
    "httm": dict(kind="merge",
                 desc="head-wise temporal token merging (HTTM-style): 200 frames x 1374 tokens, H=16, d=64, "
                      "bf16; keys/values merged per head in blocks of 4 frames x 37 patches, 50 % of the "
                      "sources merged into the first frame of the chunk, then size-aware attention (ln g) "
                      "of all 274,800 queries over the merged keys",
                 mcfg=dict(B=1, H=16, N=200, n_t=4, n_s=37, r_permille=500)),
    "merged": dict(kind="bias",
                   desc="size-aware attention: 274,800 queries (200 frames x 1374) against 137,400 merged "
                        "keys standing for 1-3 tokens each (bias ln g), H=16, d=64, bf16",
                   shape=dict(H=16, Tq=274800, Tk=137400)),
    "dense": dict(kind="dense", desc="dense global attention (sigma = 1): N=32 frames x 1374 tokens, H=16, d=64, bf16",
                  shape=dict(H=16, N=32, L=1374)),
    "frame": dict(kind="frame", desc="frame-local attention (Global-to-Frame): N=100 frames x 1374 tokens, H=16, "
                                     "d=64, bf16", shape=dict(H=16, N=100, L=1374)),
}

# DRAM traffic of the dominant kernel per launch, measured with
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum (one pass) on this file's default
# workload, keyed by a fingerprint of the kernel's sources; reported only while they are unchanged.
KERNEL_SOURCES = ("subsampled_global_attention_sga_b300/csrc/attn_tc.cuh",
                  "subsampled_global_attention_sga_b300/csrc/common.cuh",
                  "subsampled_global_attention_sga_b300/csrc/extras.cuh")
TRAFFIC_GB = {
    # attn_tc_kernel<false> on the 800-frame sigma = 4 layer: 379.49 GB read + 2.71 GB written
    "40917419ae2423cb": {"headline": 382.20},
    # after the size-aware and rotary variants were added (same main path): 304.64 + 2.71 GB
    "585bb52597cd6808": {"headline": 307.35},
    # key tiles swept in alternating directions per round of units: 92.52 + 2.44 GB
    "ae0006a668381cc7": {"headline": 94.96},
    # Q tiles released at the unit's last key tile, plus the self-test's skipped-tile hook (off
    # in this launch): 170.49 + 2.44 GB; same 1.38 s, the kernel is not bound by DRAM
    "58b57bb8c27c1a5d": {"headline": 172.93},
    # slots numbered across units, mixed units, the epilogue forms, whole-sector output stores:
    # 114.51 + 3.40 GB (1.15 s; L2 evict-last hints on the K/V tiles left it at 116.8 GB)
    "094d1d58d00a412f": {"headline": 117.91},
}


def _kernel_fingerprint() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


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


def _percentiles(xs):
    """p10 / p50 / p90 (linear interpolation) and the mean of a list of times."""
    a = np.sort(np.asarray(xs, dtype=np.float64))
    q = lambda f: float(np.interp(f * (len(a) - 1), np.arange(len(a)), a))
    return {"p10": q(0.1), "p50": q(0.5), "p90": q(0.9), "mean": float(a.mean()), "n": int(len(a))}


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


class Job:
    """One workload on the device: stages run in order per step, FLOPs per step, the dominant
    stage (name, roofline bound, algorithmic amount per launch) and an end-to-end call."""

    def __init__(self, sga, wl, dev, rank):
        from subsampled_global_attention_sga_b300.inputs import correlated_qkv
        self.sga, self.wl, self.dev, self.kind = sga, wl, dev, wl["kind"]
        self.launches = None                    # kernels per step, when not one per stage
        seed = 3 * rank
        if self.kind == "sga":
            cfg = sga.SGAConfig(**wl["cfg"])
            self.cfg = cfg
            q, k, v = correlated_qkv(cfg.B, cfg.H, cfg.N, cfg.L, 64, seed=seed, dtype=cfg.torch_dtype, device=dev)
            if "general" in wl:
                g = wl["general"]
                prot = np.random.default_rng(seed).integers(0, cfg.T, size=int(g["protected"] * cfg.T))
                kv, _, _ = sga.plan_host_general(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, sigma_h=g["sigma"],
                                                 sigma_w=g["sigma"], phase_shift=g["phase"],
                                                 ref_frame_dense=cfg.ref_frame_dense, protected=prot)
                self.plan = sga.Plan(cfg, dev, kv_index=kv)
                self.kv_index = kv
            else:
                self.plan = sga.Plan(cfg, dev)
                self.kv_index = None
            self.inputs = (q, k, v)
            self.bufs = self.plan.compact(k, v)
            self.out = torch.empty_like(q)
            plan, bufs, out = self.plan, self.bufs, self.out
            self.stages = [("compaction", lambda: plan.compact(k, v, *bufs)),
                           ("attention", lambda: plan.forward(q, k, v, *bufs, out=out))]
            self.flops = layer_flops(cfg, plan.S)
            self.dominant = ("attention", "tensor", self.flops, "sga::tc::attn_tc_kernel<false>")
            ck = "sga::cr::compact_rope_kernel" if (cfg.rope and cfg.dtype == "bf16") else "sga::compact_kernel"
            self.secondary = ("compaction", "hbm", compaction_bytes(cfg, plan.S), ck)
            self.launches = 3                   # the compaction, its sums, the attention
            self.dtype = cfg.dtype
            self.config = {"B_per_rank": cfg.B, "H": cfg.H, "N": cfg.N, "L": cfg.L, "T": cfg.T, "S": plan.S,
                           "sigma": cfg.sigma, "flops_per_layer": self.flops}
        elif self.kind == "bias":
            sh = wl["shape"]
            H, Tq, Tk = sh["H"], sh["Tq"], sh["Tk"]
            q, _, _ = correlated_qkv(1, H, 1, Tq, 64, seed=seed, dtype=torch.bfloat16, device=dev)
            _, k, v = correlated_qkv(1, H, 1, Tk, 64, seed=seed + 1, dtype=torch.bfloat16, device=dev)
            gen = torch.Generator(device=dev).manual_seed(seed + 2)
            bias = torch.log(torch.randint(1, 4, (1, H, Tk), generator=gen, device=dev).float()).contiguous()
            self.inputs = (q, k, v, bias)
            self.out = torch.empty_like(q)
            out = self.out
            self.stages = [("attention", lambda: sga.bias_forward(q, k, v, bias, out=out))]
            self.flops = 4.0 * Tq * Tk * 64 * H
            self.dominant = ("attention", "tensor", self.flops, "sga::tc::attn_tc_kernel<true>")
            self.secondary = None
            self.dtype = "bf16"
            self.config = {"H": H, "Tq": Tq, "Tk": Tk, "flops_per_layer": self.flops}
        elif self.kind == "merge":
            mc = sga.MergeConfig(**wl["mcfg"])
            L = mc.n_special + mc.grid_h * mc.grid_w
            q, k, v = correlated_qkv(mc.B, mc.H, mc.N, L, 64, seed=seed, dtype=torch.bfloat16, device=dev)
            M = sga.merge_size(mc)
            bufs = sga.merge(mc, k, v)
            self.mcfg, self.inputs = mc, (q, k, v)
            self.out = torch.empty_like(q)
            out = self.out
            self.stages = [("merge", lambda: sga.merge(mc, k, v, out=bufs)),
                           ("attention", lambda: sga.bias_forward(q, bufs[0], bufs[1], bufs[2], out=out))]
            self.flops = 4.0 * mc.T * M * 64 * mc.H * mc.B
            self.dominant = ("attention", "tensor", self.flops, "sga::tc::attn_tc_kernel<true, false>")
            self.secondary = None
            self.merge_stage = True
            self.dtype = "bf16"
            self.config = {"H": mc.H, "N": mc.N, "T": mc.T, "M": M, "n_t": mc.n_t, "n_s": mc.n_s,
                           "r_permille": mc.r_permille, "flops_per_layer": self.flops}
        else:
            sh = wl["shape"]
            H, N, L = sh["H"], sh["N"], sh["L"]
            q, k, v = correlated_qkv(1, H, N, L, 64, seed=seed, dtype=torch.bfloat16, device=dev)
            self.inputs = (q, k, v)
            self.out = torch.empty_like(q)
            out = self.out
            if self.kind == "dense":
                self.stages = [("attention", lambda: sga.dense_forward(q, k, v, out=out))]
                self.flops = 4.0 * (N * L) ** 2 * 64 * H
            else:
                self.stages = [("attention", lambda: sga.frame_forward(q, k, v, N, L, out=out))]
                self.flops = 4.0 * N * L * L * 64 * H
            self.dominant = ("attention", "tensor", self.flops, "sga::tc::attn_tc_kernel<false>")
            self.secondary = None
            self.dtype = "bf16"
            self.config = {"H": H, "N": N, "L": L, "T": N * L, "flops_per_layer": self.flops}

    def step(self, ev=None, stream=None):
        for i, (_, fn) in enumerate(self.stages):
            if ev is not None:
                ev[i].record(stream)
            fn()
        if ev is not None:
            ev[len(self.stages)].record(stream)

    def e2e_call(self, host_in, out_host):
        """Copy this step's inputs from pinned host memory, run the layer, copy the result back."""
        sga, dev = self.sga, self.dev
        if self.kind == "sga":
            return sga.layer_from_host(self.plan, *host_in, out_host=out_host)
        if self.kind == "merge":
            q, k, v = [x.to(dev, non_blocking=True) for x in host_in]
            out_host.copy_(sga.merged_attention(self.mcfg, q, k, v), non_blocking=True)
            return out_host
        dev_in = [x.to(dev, non_blocking=True) for x in host_in]
        if self.kind == "bias":
            o = sga.bias_forward(*dev_in)
        elif self.kind == "dense":
            o = sga.dense_forward(*dev_in)
        else:
            sh = self.wl["shape"]
            o = sga.frame_forward(*dev_in, sh["N"], sh["L"])
        out_host.copy_(o, non_blocking=True)
        return out_host

    def cpu_sample(self, target_s=12.0, h=0, max_rows=4096):
        """Time the fp64 oracle on sampled query rows of one (batch, head)."""
        import oracle
        from subsampled_global_attention_sga_b300.inputs import sample_rows
        kind = self.kind
        hx = [x[0, h].float().cpu().numpy() for x in self.inputs[:3]]
        qh, kh, vh = hx
        Tq = qh.shape[0]
        extra_t, pre = 0.0, None
        if kind == "sga":
            cfg = self.cfg
            if self.kv_index is None:
                s_h, s_w = cfg.s_hw
                op = oracle.plan(cfg.N, cfg.grid_h, cfg.grid_w, cfg.n_special, s_h, s_w, cfg.phase_shift,
                                 cfg.ref_frame_dense)
            else:
                kept = np.zeros(cfg.T, dtype=np.uint8)
                kept[self.kv_index] = 1
                op = oracle.Plan(T=cfg.T, L=cfg.L, kept=kept, kv_index=self.kv_index,
                                 frame_off=np.searchsorted(self.kv_index, np.arange(cfg.N + 1) * cfg.L).astype(np.int32))
            if cfg.rope:
                qh = oracle.rope2d(qh, cfg.L, cfg.n_special, cfg.grid_w, cfg.rope_base, cfg.rope_pos_offset).astype(np.float32)
                kh = oracle.rope2d(kh, cfg.L, cfg.n_special, cfg.grid_w, cfg.rope_base, cfg.rope_pos_offset).astype(np.float32)
            t0 = time.perf_counter()
            sums = oracle.dropped_sums(op, kh, vh)
            extra_t = time.perf_counter() - t0
            n_keys = op.S + (2 if (cfg.diag or cfg.mean) else 0)
            run = lambda rows: oracle.sga_rows(op, qh[rows], kh, vh, rows, diag=cfg.diag, mean=cfg.mean, sums=sums)
            L = cfg.L
        elif kind == "merge":
            mc = self.mcfg
            t0 = time.perf_counter()
            m = oracle.merge_match(kh, mc.N, mc.grid_h, mc.grid_w, mc.n_special, mc.n_t, mc.n_s, mc.r_permille)
            kept, gid, sizes = oracle.merge_groups(m)
            km, vm = oracle.merge_apply(kh, gid, len(kept)), oracle.merge_apply(vh, gid, len(kept))
            extra_t = time.perf_counter() - t0
            b = np.log(sizes)
            n_keys = len(kept)
            run = lambda rows: oracle.biased_attention_rows(qh[rows], km, vm, b)
            L = mc.n_special + mc.grid_h * mc.grid_w
        elif kind == "bias":
            b = self.inputs[3][0, h].double().cpu().numpy()
            n_keys = kh.shape[0]
            run = lambda rows: oracle.biased_attention_rows(qh[rows], kh, vh, b)
            L = 1374
        else:
            L = self.wl["shape"]["L"]
            fl = L if kind == "frame" else 0
            n_keys = L if kind == "frame" else kh.shape[0]
            run = lambda rows: oracle.attention_rows(qh[rows], kh, vh, rows, frame_len=fl)
        calib = min(64, Tq)
        rows = sample_rows(Tq, L, calib, seed=77).numpy()
        t0 = time.perf_counter()
        run(rows)
        t_cal = time.perf_counter() - t0
        n = int(max(calib, min(max_rows, Tq, calib * max(1.0, (target_s - t_cal) / max(t_cal, 1e-6)))))
        rows = sample_rows(Tq, L, n, seed=78).numpy()
        t0 = time.perf_counter()
        run(rows)
        t_rows = time.perf_counter() - t0
        n = len(rows)
        flops = 4.0 * n * n_keys * 64
        heads = self.flops / (4.0 * Tq * n_keys * 64)
        ms_layer = (t_rows / n * Tq + extra_t) * heads * 1e3
        return {"value": flops / t_rows / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                "sample": f"{n} query rows of head {h} (of {Tq} rows x {heads:.0f} heads); fp64 C oracle, OpenMP",
                "seconds": t_rows, "extrapolated_ms_per_layer": ms_layer}


def run_ours(args):
    import subsampled_global_attention_sga_b300 as sga

    rank, world, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload]
    job = Job(sga, wl, dev, rank)
    stream = torch.cuda.current_stream(dev)
    n_st = len(job.stages)

    for _ in range(args.warmup):
        job.step()
    torch.cuda.synchronize(dev)
    if sga.device_status(dev) != 0:
        raise RuntimeError("device status not OK after warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_st + 1)] for _ in range(args.steps)]
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
            job.step(evs[i], stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    _barrier(world)
    status = sga.device_status(dev)
    total_ms = _max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    stage_ms = {name: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i, (name, _) in enumerate(job.stages)}
    # spread of the per-step device times (every step bracketed by its own events)
    step_times = [e[0].elapsed_time(e[n_st]) for e in evs]
    spread = {"step": _percentiles(step_times)}
    for i, (name, _) in enumerate(job.stages):
        spread[name] = _percentiles([e[i].elapsed_time(e[i + 1]) for e in evs])
    clocks = clk.summary()

    ms_step = total_ms / args.steps
    value = world * job.flops / (ms_step * 1e-3) / 1e12
    peaks = _peaks()
    d_name, d_bound, d_amount, d_kernel = job.dominant
    d_ms = stage_ms[d_name]
    achieved = d_amount / (d_ms * 1e-3) / 1e12
    fp = _kernel_fingerprint()
    traffic = TRAFFIC_GB.get(fp, {}).get(args.workload)
    # the dominant kernel runs back to back for seconds inside the timed steps, so its peak is
    # the sustained (power-capped) bf16 figure; the burst fraction is given beside it
    roofline = {"bound": d_bound, "kernel": d_kernel, "achieved": achieved, "peak": peaks["bf16_sus"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_sus"],
                "peak_kind": f"bf16 dense sustained ({peaks['source']})",
                "frac_of_burst": achieved / peaks["bf16"], "burst_peak": peaks["bf16"],
                "traffic": traffic * 1e9 if traffic is not None else None,
                "traffic_unit": "bytes per launch (dram read + write, ncu)", "kernel_fingerprint": fp,
                "kernel_ms": d_ms, "kernel_ms_p50": spread[d_name]["p50"]}
    secondary = None
    if "merge" in stage_ms:
        secondary = {"kernel": "sga::merge_kernel<bf16>", "ms": stage_ms["merge"]}
    if job.secondary is not None:
        s_name, _, s_bytes, s_kernel = job.secondary
        s_ms = stage_ms[s_name]
        gbs = s_bytes / (s_ms * 1e-3) / 1e9
        secondary = {"kernel": s_kernel, "ms": s_ms, "achieved_gbs": gbs, "bytes": s_bytes,
                     "frac_hbm": gbs / peaks["hbm"], "frac_8tbs": gbs / 8000.0, "peak_source": peaks["source"]}

    e2e = None
    if not args.no_e2e:
        host_in = [x.cpu().pin_memory() for x in job.inputs]
        oh = torch.empty(job.out.shape, dtype=job.out.dtype, pin_memory=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if job.kind in ("sga", "dense", "frame", "bias"):
            # streamed: batch i+1's inputs are copied in and batch i-1's output copied out while
            # batch i is computed (the library's host-streaming executor); every step still moves
            # all its bytes
            if job.kind == "sga":
                hs = job.sga.HostStream(job.plan)
                submit = lambda: hs.submit(*host_in, oh)
            else:
                sh = job.wl["shape"]
                if job.kind == "bias":
                    hs = job.sga.PlainHostStream("bias", 1, sh["H"], sh["Tq"], Tk=sh["Tk"])
                    submit = lambda: hs.submit(*host_in[:3], oh, bias_host=host_in[3])
                else:
                    T = sh["N"] * sh["L"]
                    hs = job.sga.PlainHostStream(job.kind, 1, sh["H"], T, N=sh["N"], L=sh["L"])
                    submit = lambda: hs.submit(*host_in, oh)
            for _ in range(2):
                submit()
            hs.synchronize()
            torch.cuda.synchronize(dev)
            _barrier(world)
            a.record(hs.h2d)
            for _ in range(args.steps):
                submit()
            b.record(hs.d2h)
            e2e_mode = "streamed (host-streaming executor: copies overlap the previous/next step's compute)"
        else:
            for _ in range(2):
                job.e2e_call(host_in, oh)
            torch.cuda.synchronize(dev)
            _barrier(world)
            a.record(stream)
            for _ in range(args.steps):
                job.e2e_call(host_in, oh)
            b.record(stream)
            e2e_mode = "serial (copy in, compute, copy out on one stream)"
        torch.cuda.synchronize(dev)
        _barrier(world)
        e_ms = _max_over_ranks(a.elapsed_time(b), world, dev) / args.steps
        if job.kind in ("sga", "dense", "frame", "bias"):
            hs.synchronize()
            hs.close()
        h2d = sum(x.numel() * x.element_size() for x in host_in)
        d2h = oh.numel() * oh.element_size()
        # with copies overlapping compute a step costs max(copy-in time, compute, copy-out time):
        # when the step takes well over the device time, the host link is what binds
        bound = "copies (host link)" if e_ms > 1.25 * ms_step else "compute"
        e2e = {"value": world * job.flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "mode": e2e_mode, "bound": bound,
               "h2d_gbs": h2d / (e_ms * 1e-3) / 1e9, "device_ms_per_step": ms_step}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = job.cpu_sample()

    if rank != 0:
        return
    q = job.inputs[0]
    metric = METRIC if args.workload == "headline" else f"{args.workload}: ms/layer and effective TFLOP/s"
    config = {"workload": wl["desc"], **job.config,
              "l2": "inputs larger than L2 (Q %.2f GB); no flush" % (q.numel() * q.element_size() / 1e9)
              if q.numel() * q.element_size() > 126e6 else "inputs smaller than L2: steady-state, L2-warm",
              "parallelism": f"dp{world} (independent layers per rank)", "stage_ms": stage_ms,
              "ms_spread": spread}
    line = {
        "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if job.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config, "roofline": roofline, "compaction": secondary, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (job.launches if job.launches is not None else n_st) * args.steps,
        "clocks": clocks, "device_status": status,
    }
    print(json.dumps(line), flush=True)


def _time_stages(stages, warmup, steps, dev):
    """Per-step CUDA-event times (ms) of each stage, on the current stream, after `warmup` steps."""
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        for _, fn in stages:
            fn()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(steps)]
    torch.cuda._sleep(int(2e6 * (2 + steps)))
    for e in evs:
        for i, (_, fn) in enumerate(stages):
            e[i].record(stream)
            fn()
        e[len(stages)].record(stream)
    torch.cuda.synchronize(dev)
    return {name: [e[i].elapsed_time(e[i + 1]) for e in evs] for i, (name, _) in enumerate(stages)}


SWEEP_N, SWEEP_H, SWEEP_SIGMAS = 100, 16, (1, 2, 4, 6, 9)


def run_sweep(args):
    """The 100-frame sweep: sigma in {1, 2, 4, 6, 9} x fixed / phase-shifted grid x diagonal and
    mean terms on / off, plus frame-local attention as the dense-per-frame baseline.  One JSON
    line per configuration (median of the per-step device times), then a summary line with the
    measured dense / SGA time ratios beside the FLOP ratios that bound them."""
    import subsampled_global_attention_sga_b300 as sga
    from subsampled_global_attention_sga_b300.inputs import correlated_qkv
    rank, world, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = _peaks()
    N, H = SWEEP_N, SWEEP_H
    L = sga.SGAConfig(B=1, H=H, N=N).L
    q, k, v = correlated_qkv(1, H, N, L, 64, seed=3 * rank, dtype=torch.bfloat16, device=dev)
    cases = [(s_, ph, terms) for s_ in SWEEP_SIGMAS for ph in (False, True) for terms in (True, False)
             if not (s_ == 1 and ph)]
    lines, att_ms = [], {}
    with Clocks(dev.index) as clk:
        for sigma, ph, terms in cases:
            cfg = sga.SGAConfig(B=1, H=H, N=N, sigma=sigma, phase_shift=ph, diag=terms, mean=terms)
            plan = sga.Plan(cfg, dev)
            bufs = plan.compact(k, v)
            out = torch.empty_like(q)
            t = _time_stages([("compaction", lambda: plan.compact(k, v, *bufs)),
                              ("attention", lambda: plan.forward(q, k, v, *bufs, out=out))],
                             args.warmup, args.steps, dev)
            if sga.device_status(dev) != 0:
                raise RuntimeError("device status not OK")
            flops = layer_flops(cfg, plan.S)
            a50, c50 = _percentiles(t["attention"])["p50"], _percentiles(t["compaction"])["p50"]
            att_ms[(sigma, ph, terms)] = a50
            lines.append({
                "metric": f"sweep N={N}: SGA ms/layer and effective TFLOP/s", "sigma": sigma, "phase_shift": ph,
                "diag_mean": terms, "T": cfg.T, "S": plan.S, "flops_per_layer": flops,
                "ms_per_layer": a50 + c50, "attention_ms": _percentiles(t["attention"]),
                "compaction_ms": _percentiles(t["compaction"]), "tflops": flops / ((a50 + c50) * 1e-3) / 1e12,
                "attention_tflops": flops / (a50 * 1e-3) / 1e12,
                "frac_of_burst": flops / (a50 * 1e-3) / 1e12 / peaks["bf16"],
                "frac_of_sustained": flops / (a50 * 1e-3) / 1e12 / peaks["bf16_sus"],
                "compaction_gbs": compaction_bytes(cfg, plan.S) / (c50 * 1e-3) / 1e9})
            plan.close()
            del bufs, out
        out = torch.empty_like(q)
        t = _time_stages([("attention", lambda: sga.frame_forward(q, k, v, N, L, out=out))], args.warmup,
                         args.steps, dev)
        f50 = _percentiles(t["attention"])["p50"]
        fflops = 4.0 * N * L * L * 64 * H
        lines.append({"metric": f"sweep N={N}: frame-local attention ms/layer and TFLOP/s", "kind": "frame-local",
                      "T": N * L, "flops_per_layer": fflops, "ms_per_layer": f50,
                      "attention_ms": _percentiles(t["attention"]), "tflops": fflops / (f50 * 1e-3) / 1e12,
                      "frac_of_burst": fflops / (f50 * 1e-3) / 1e12 / peaks["bf16"]})
    if rank != 0:
        return
    for ln in lines:
        print(json.dumps(ln), flush=True)
    dense = att_ms[(1, False, True)]
    ratios = {}
    for sigma in SWEEP_SIGMAS[1:]:
        for ph in (False, True):
            key = (sigma, ph, True)
            row = next(x for x in lines if x.get("sigma") == sigma and x.get("phase_shift") == ph and x.get("diag_mean"))
            dense_row = next(x for x in lines if x.get("sigma") == 1)
            ratios[f"sigma{sigma}{'_phase' if ph else ''}"] = {
                "measured_dense_over_sga": dense / att_ms[key],
                "flop_bound": dense_row["flops_per_layer"] / row["flops_per_layer"]}
    print(json.dumps({"metric": f"sweep N={N}: dense / SGA attention time", "ratios": ratios,
                      "frame_local_over_dense": f50 / dense, "clocks": clk.summary(), "steps": args.steps,
                      "warmup": args.warmup, "peaks": peaks}), flush=True)


def run_reference(args):
    """The fp64 CPU oracle, as it stands, on a bounded sample of the workload (rank 0 only)."""
    rank, world, _ = (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0)
    if rank != 0:
        return
    import oracle
    import subsampled_global_attention_sga_b300 as sga
    from subsampled_global_attention_sga_b300.inputs import correlated_qkv
    wl = WORKLOADS.get(args.workload, {"kind": "sweep"})
    if wl["kind"] != "sga":
        print(json.dumps({"impl": "reference", "unavailable": "the CPU reference arm covers the SGA workloads"}))
        return
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
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["sweep"], default="headline")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "sweep":
        run_sweep(args)
    else:
        run_ours(args)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
