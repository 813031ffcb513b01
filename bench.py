"""Benchmark of the BackLite hot path on one GB300 (or N, one process each).

One step = exact forward that reduces the tile weights in its epilogue ->
mask from the tile weights -> block-sparse backward, on the video-DiT-shaped
workload (B=1, H=Hk=40, n=32760 = 21x30x52 latent grid, d=128, 128x128
tiles, negl_prob=0.05, clustered synthetic inputs, seed 0).  Inputs are
resident in HBM and larger than the 129 MB L2 (Q alone is 335 MB), so no
flush is needed between steps.  The unfused path (forward writing the full
statistics, bl_mask_from_stats reading them; the same lists) is timed beside
it under "unfused".

Printed JSON line (rank 0): ``value`` = attention-backward milliseconds per
step (mask + backward, CUDA events on the launch stream, max over ranks),
with dense-equivalent TFLOP/s, skipped-tile fraction and the fraction of the
measured bf16 tensor peak on the computed tiles beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload (query tiles of a few heads) and scales it to the full
backward in the same unit.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn bwd ms + dense-equiv TFLOP/s at n=32k,d=128; skip %; % bf16 tensor peak"
WORKLOAD = "video_n32760_d128"
NEGL = 0.05


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16": d["bf16_tflops"], "bf16_sustained": d.get("bf16_tflops_sustained"),
                "hbm": d["hbm_gbs"], "src": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "src": "fallback"}


class ClockSampler:
    """SM clocks, power and throttle reasons sampled during the timed region.

    Reads NVML through ctypes from a background thread (no child processes, so
    nothing forks the CUDA process while kernels run); falls back to
    nvidia-smi only if libnvidia-ml cannot be loaded.  Only reads settings."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_id: str, period_s: float = 0.05):
        self.gpu_id = gpu_id
        self.period = period_s
        self.rows = []
        self._stop = threading.Event()
        self._t = None
        self._nvml = None
        self._dev = None
        self.max_mhz = None
        try:
            import ctypes
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() == 0:
                dev = ctypes.c_void_p()
                if lib.nvmlDeviceGetHandleByUUID(gpu_id.encode(), ctypes.byref(dev)) == 0:
                    self._nvml, self._dev = lib, dev
                    mx = ctypes.c_uint()
                    if lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = float(mx.value)
        except OSError:
            self._nvml = None

    def _sample_nvml(self):
        import ctypes
        lib, dev = self._nvml, self._dev
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        lib.nvmlDeviceGetClockInfo(dev, 1, ctypes.byref(clk))          # NVML_CLOCK_SM
        lib.nvmlDeviceGetPowerUsage(dev, ctypes.byref(pw))
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(dev, ctypes.byref(rs))
        return float(clk.value), pw.value / 1000.0, int(rs.value)

    def _sample_smi(self):
        q = ("clocks.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap,clocks.max.sm")
        out = subprocess.run(["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={q}",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True,
                             timeout=5).stdout.strip().split(",")
        bits = [0x8, 0x40, 0x20, 0x4]
        rs = sum(b for b, v in zip(bits, out[2:6]) if v.strip().lower() == "active")
        self.max_mhz = float(out[6])
        return float(out[0]), float(out[1]), rs

    def _run(self):
        while not self._stop.is_set():
            try:
                self.rows.append(self._sample_nvml() if self._nvml else self._sample_smi())
            except Exception:
                pass
            self._stop.wait(self.period)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        self._t.join(timeout=10)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"]}
        reasons = sorted({name for _, _, r in self.rows for bit, name in self.REASONS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(r[0] for r in self.rows),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.rows),
                "power_w_max": max(r[1] for r in self.rows),
                "source": "nvml" if self._nvml else "nvidia-smi"}


def _smi_id(dev):
    """nvidia-smi --id for a torch device: its UUID (independent of
    CUDA_VISIBLE_DEVICES renumbering), else the visible index."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in vis.split(",") if p.strip()]
    idx = dev.index or 0
    return parts[idx].strip() if idx < len(parts) else str(idx)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_reference_sample(w, q, k, v, go, budget_s=15.0, max_tiles=256):
    """Time the oracle's backward for whole query tiles of the workload.

    For each sampled (head, query tile) the oracle forms the tile's exact
    forward rows (LSE and tile statistics against every key), applies the
    selection rule to that tile's row of key tiles and computes G_Q for the
    tile's rows with the masked backward.  Returns (ms for the full backward
    extrapolated over all B*H*T_r query tiles, description, tiles, seconds).
    """
    import numpy as np

    from oracle import attention as A
    from oracle import mask_spec as M

    rng = np.random.default_rng(1)
    T_r = w.T_r
    t0 = time.perf_counter()
    done = 0
    qn = q.float().numpy()
    kn = k.float().numpy()
    vn = v.float().numpy()
    gn = go.float().numpy()
    while done < max_tiles and time.perf_counter() - t0 < budget_s:
        h = int(rng.integers(w.H))
        hk = h // (w.H // w.Hk)
        i = int(rng.integers(T_r))
        rows = np.arange(i * w.block_q, min(w.n, (i + 1) * w.block_q))
        qh = qn[0, :, h].astype(np.float64)
        kh = kn[0, :, hk].astype(np.float64)
        vh = vn[0, :, hk].astype(np.float64)
        o_r, l_r, st_r = A.forward_head(qh, kh, vh, w.scale, rows=rows, block_k=w.block_k,
                                        causal=w.causal, window=w.window)
        d = M.tile_weights(st_r.astype(np.float32), l_r.astype(np.float32), len(rows), w.block_q)
        act, _ = M.select_row(d[0], M.threshold(NEGL))
        tm = np.zeros((T_r, w.T_c), dtype=np.uint8)
        tm[i] = act
        tm[M.structurally_empty(T_r, w.T_c, w.n, w.block_q, w.block_k, w.causal, w.window)] = 0
        o_full = np.zeros_like(qh)
        o_full[rows] = o_r
        lse_full = np.zeros(w.n)
        lse_full[rows] = l_r
        A.backward_head(qh, kh, vh, o_full, gn[0, :, h].astype(np.float64), lse_full, w.scale,
                        tm, w.block_q, w.block_k, rows=rows, causal=w.causal, window=w.window)
        done += 1
    el = time.perf_counter() - t0
    total_tiles = w.B * w.H * T_r
    ms_full = el / done * total_tiles * 1e3
    desc = (f"{done} random (head, query tile) pairs of {total_tiles}: exact forward rows, "
            f"tile stats, selection and G_Q in fp64, extrapolated to the full backward")
    return ms_full, desc, done, el


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    from block_sparse_attention_fwd_gb300 import inputs
    w = inputs.WORKLOADS[WORKLOAD]
    q, k, v, go = inputs.generate(w, seed=0)
    cores = os.cpu_count()
    vals = []
    for s in range(args.warmup + args.steps):
        ms, desc, tiles, el = cpu_reference_sample(w, q, k, v, go, budget_s=args.ref_budget,
                                                   max_tiles=args.ref_tiles)
        if s >= args.warmup:
            vals.append(ms)
    val = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "ms",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": val,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "B": w.B, "n": w.n, "H": w.H,
                                            "Hk": w.Hk, "d": w.d, "tiles": "128x128",
                                            "negl_prob": NEGL},
            "cpu_baseline": {"value": val, "unit": "ms", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": val, "unit": "ms", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    from block_sparse_attention_fwd_gb300 import _lib, build, inputs

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = inputs.WORKLOADS[args.workload]
    negl = args.negl
    # weak scaling: every rank runs its own independent problem (seed = rank)
    q, k, v, go = inputs.generate(w, seed=rank)
    shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)
    T_r, T_c = _lib.tiles(shape)
    qd, kd, vd, god = (x.to(dev) for x in (q, k, v, go))
    o = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.n), dtype=torch.float32, device=dev)
    logw = torch.empty((w.B, w.H, T_r, T_c), dtype=torch.float32, device=dev)
    fws = torch.empty(_lib.fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    lists = _lib.alloc_lists(shape, dev)
    g_q, g_k, g_v = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    wsb = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # one step: the forward reduces the tile weights in its epilogue (the
    # statistics rows stay in its scratch slots), the mask reads the weights,
    # then the block-sparse backward
    def step(ev=None):
        if ev:
            ev[0].record(stream)
        _lib.attn_fwd_tile_weights(shape, qd, kd, vd, w.scale, o, lse, logw, workspace=fws)
        if ev:
            ev[1].record(stream)
        _lib.mask_from_tile_weights(shape, logw, negl, lists)
        if ev:
            ev[2].record(stream)
        _lib.attn_bwd(shape, qd, kd, vd, o, god, lse, w.scale, lists, g_q, g_k, g_v, wsb)
        if ev:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if _lib.bwd_check_status(shape, wsb) != 0:
        raise RuntimeError("backward reported corrupt tile lists")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(_smi_id(dev)) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for s in range(args.steps):
            step(evs[s])
        t_end.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    mask_ms = [e[1].elapsed_time(e[2]) for e in evs]
    bwd_ms = [e[2].elapsed_time(e[3]) for e in evs]
    attn_bwd = [m + b for m, b in zip(mask_ms, bwd_ms)]
    step_ms = total_ms / args.steps
    vals = torch.tensor([statistics.mean(attn_bwd), step_ms], dtype=torch.float64, device=dev)
    if ws > 1:
        torch.distributed.all_reduce(vals, op=torch.distributed.ReduceOp.MAX)
    attn_bwd_ms, step_ms = float(vals[0]), float(vals[1])

    # sparsity of this step's mask
    mask = lists["mask"]
    n_active = int(mask.sum(dtype=torch.int64).item())
    n_tiles = mask.numel()
    skip = 1.0 - n_active / n_tiles

    # dense backward at the same shape (lists = NULL), same timing method
    dense_ms = []
    for _ in range(args.dense_iters):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        _lib.attn_bwd(shape, qd, kd, vd, o, god, lse, w.scale, None, g_q, g_k, g_v, wsb)
        b.record(stream)
        torch.cuda.synchronize()
        dense_ms.append(a.elapsed_time(b))
    # the unfused path beside it: the forward writing the full statistics and
    # the mask pass reading them (the same lists, bit for bit)
    def timed_call(fn, reps=3):
        ts = []
        for _ in range(reps + 1):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts[1:])

    stats = torch.empty((w.B, w.H, T_c, T_r * w.block_q), dtype=torch.float32, device=dev)
    fwd_stats_ms = timed_call(lambda: _lib.attn_fwd(shape, qd, kd, vd, w.scale, o, lse, stats))
    lists2 = _lib.alloc_lists(shape, dev)
    mask_stats_ms = timed_call(lambda: _lib.mask_from_stats(shape, stats, lse, negl, lists2))
    if not torch.equal(lists2["mask"], lists["mask"]):
        raise RuntimeError("the mask from the tile weights differs from the mask from the stats")
    del stats, lists2

    pk = _peaks()
    dense_flop = w.dense_bwd_flop()
    # computed-tile work: 10*Br*Bc*d per active (head, q tile, k tile) triple,
    # counting only the valid rows/keys of ragged edge tiles
    computed_flop = _active_flop(mask, w)
    bwd_only = statistics.mean(bwd_ms)
    fwd_only = statistics.mean(fwd_ms)
    achieved_tf = computed_flop / (bwd_only * 1e-3) / 1e12
    fwd_tf = w.dense_fwd_flop() / (fwd_only * 1e-3) / 1e12
    traffic = _traffic(args.workload)
    line = {
        "metric": METRIC, "value": attn_bwd_ms, "unit": "ms", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded clustered generator, video-grid clusters)",
        "config": {"workload": args.workload, "B": w.B, "n": w.n, "H": w.H, "Hk": w.Hk,
                   "d": w.d, "tiles": f"{w.block_q}x{w.block_k}", "negl_prob": negl,
                   "l2": "inputs larger than L2 (no flush)"},
        "fwd_ms": statistics.mean(fwd_ms), "mask_ms": statistics.mean(mask_ms),
        "bwd_kernels_ms": bwd_only,
        "dense_bwd_ms": statistics.median(dense_ms) if dense_ms else None,
        "dense_equiv_tflops": dense_flop / (attn_bwd_ms * 1e-3) / 1e12,
        "skip_frac": skip,
        "frac_bf16_peak_computed_tiles": achieved_tf / pk["bf16"],
        # the step's dominant kernel (by time): the forward with tile statistics
        "roofline": {"bound": "tensor", "achieved": fwd_tf, "peak": pk["bf16"],
                     "unit": "TFLOP/s", "frac": fwd_tf / pk["bf16"],
                     "traffic": traffic.get("fwd_tc_kernel"),
                     "kernel": "fwd_tc_kernel with the tile-weight epilogue "
                               "(4*B*H*n^2*d per launch)",
                     "peak_src": pk["src"] + " burst"},
        # the metric's own kernel: the block-sparse backward on computed tiles
        "roofline_bwd": {"bound": "tensor", "achieved": achieved_tf, "peak": pk["bf16"],
                         "unit": "TFLOP/s", "frac": achieved_tf / pk["bf16"],
                         "traffic": _sum_or_none(traffic, ("bwd_pre_kernel", "bwd_tc_kernel",
                                                           "dq_convert_kernel")),
                         "kernel": "bl_attn_bwd call (D pass, which also zeroes the dQ "
                                   "accumulator, + bwd_tc_kernel + dQ convert), 10*d*valid rows*"
                                   "valid keys per kept tile; traffic summed over the three",
                         "peak_src": pk["src"] + " burst"},
        "roofline_mask": {"bound": "hbm",
                          "achieved": _mask_bytes(w, True) / (statistics.mean(mask_ms) * 1e-3) / 1e9,
                          "peak": pk["hbm"], "unit": "GB/s",
                          "frac": _mask_bytes(w, True) / (statistics.mean(mask_ms) * 1e-3) / 1e9 / pk["hbm"],
                          "traffic": _sum_or_none(traffic, ("mask_rows_warp_kernel",
                                                            "q_lists_kernel")),
                          "kernel": "bl_mask_from_tile_weights call (mask_rows_warp_kernel + "
                                    "q_lists_kernel) reading the forward's tile weights"},
        "unfused": {"fwd_with_stats_ms": fwd_stats_ms, "mask_from_stats_ms": mask_stats_ms,
                    "mask_from_stats_gbs": _mask_bytes(w) / (mask_stats_ms * 1e-3) / 1e9,
                    "what": "forward writing the full tile statistics + bl_mask_from_stats "
                            "(same lists); not part of value"},
        # per step: forward 1, mask 2, backward 3 (D pass, tcgen05 pass, dQ convert)
        "gpu_launches": 6 * args.steps,
    }
    clk_s = clk.summary()
    line["clocks"] = clk_s

    if not args.no_e2e:
        line["e2e"] = _e2e(args, w, shape, q, k, v, go, negl, dev)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        ms_cpu, desc, tiles, el = cpu_reference_sample(w, q, k, v, go, budget_s=args.ref_budget,
                                                       max_tiles=args.ref_tiles)
        line["cpu_baseline"] = {"value": ms_cpu, "unit": "ms", "cores": os.cpu_count(),
                                "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def _mask_bytes(w, from_weights=False):
    """Algorithmic bytes of the mask pass: read the tile statistics and the
    LSE (bl_mask_from_stats) or the tile weights (bl_mask_from_tile_weights),
    write mask, kv_idx, kv_cnt, q_idx, q_cnt."""
    if from_weights:
        inp = w.B * w.H * w.T_r * w.T_c * 4
    else:
        inp = w.B * w.H * w.T_c * w.T_r * w.block_q * 4 + w.B * w.H * w.n * 4
    lists = w.B * w.H * w.T_r * w.T_c * (1 + 4 + 4) + w.B * w.H * (w.T_r + w.T_c) * 4
    return inp + lists


def _sum_or_none(traffic, kernels):
    """Summed per-launch traffic of the kernels of one call, or None unless all
    of them have a current measurement."""
    vals = [traffic.get(k) for k in kernels]
    return None if any(v is None for v in vals) else sum(vals)


def _traffic(workload):
    """Per-launch DRAM bytes (read + write) of the kernels on this workload from
    the committed ncu summary, for every kernel whose source is unchanged since
    the counters were taken (same SHA-256 of its .cu file); else absent."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return {}
    d = json.load(open(p))
    out = {}
    for kernel, rec in d.get(workload, {}).items():
        src = os.path.join(ROOT, "block_sparse_attention_fwd_gb300", "csrc", rec["source"])
        if os.path.exists(src) and \
                hashlib.sha256(open(src, "rb").read()).hexdigest() == rec["sha256"]:
            out[kernel] = rec["dram_bytes_per_launch"]
    return out


def _active_flop(mask, w):
    import torch
    T_r, T_c = mask.shape[2], mask.shape[3]
    rows = torch.full((T_r,), w.block_q, dtype=torch.float64)
    rows[-1] = w.n - (T_r - 1) * w.block_q
    cols = torch.full((T_c,), w.block_k, dtype=torch.float64)
    cols[-1] = w.n - (T_c - 1) * w.block_k
    m = mask.to("cpu", torch.float64)
    return float(10.0 * w.d * torch.einsum("bhij,i,j->", m, rows, cols))


def _e2e(args, w, shape, q, k, v, go, negl, dev):
    """Same step through the public API with host buffers: pinned H2D copies of
    Q, K, V, G_O and D2H copies of G_Q, G_K, G_V inside the timed region, every
    step.  The copies are pipelined with the compute like a loader's prefetch:
    inputs and gradients are double-buffered on the device, step t+1's inputs
    upload on one copy stream while step t computes, and step t's gradients
    download on another while step t+1 computes; the timed region ends when the
    last step's gradients have reached the host."""
    import torch

    from block_sparse_attention_fwd_gb300 import _lib
    hq, hk, hv, hg = (x.pin_memory() for x in (q, k, v, go))
    outs = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in (q, k, v)]
            for _ in range(2)]
    ins = [[torch.empty(x.shape, dtype=x.dtype, device=dev) for x in (q, k, v, go)]
           for _ in range(2)]
    grads = [[torch.empty(x.shape, dtype=x.dtype, device=dev) for x in (q, k, v)]
             for _ in range(2)]
    o = torch.empty(q.shape, dtype=q.dtype, device=dev)
    lse = torch.empty((w.B, w.H, w.n), dtype=torch.float32, device=dev)
    T_r, T_c = _lib.tiles(shape)
    logw = torch.empty((w.B, w.H, T_r, T_c), dtype=torch.float32, device=dev)
    fws = torch.empty(_lib.fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    lists = _lib.alloc_lists(shape, dev)
    wsb = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
    main = torch.cuda.current_stream(dev)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]

    def upload(t):
        i = t % 2
        up.wait_event(computed[i])          # step t-2 has finished reading buffer i
        with torch.cuda.stream(up):
            for dst, src in zip(ins[i], (hq, hk, hv, hg)):
                dst.copy_(src, non_blocking=True)
            in_ready[i].record(up)

    def compute(t):
        i = t % 2
        dq, dk, dv, dg = ins[i]
        gq, gk, gv = grads[i]
        main.wait_event(in_ready[i])
        main.wait_event(downloaded[i])      # step t-2's gradients have left buffer i
        _lib.attn_fwd_tile_weights(shape, dq, dk, dv, w.scale, o, lse, logw, workspace=fws)
        _lib.mask_from_tile_weights(shape, logw, negl, lists)
        _lib.attn_bwd(shape, dq, dk, dv, o, dg, lse, w.scale, lists, gq, gk, gv, wsb)
        computed[i].record(main)

    def download(t):
        i = t % 2
        down.wait_event(computed[i])
        with torch.cuda.stream(down):
            for dst, src in zip(outs[i], grads[i]):
                dst.copy_(src, non_blocking=True)
            downloaded[i].record(down)

    def run(n):
        upload(0)
        for t in range(n):
            if t + 1 < n:
                upload(t + 1)
            compute(t)
            download(t)
        main.wait_stream(down)

    for e in computed + downloaded:
        e.record(main)
    run(2)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    n = max(2, min(args.steps, 6))
    a.record(main)
    run(n)
    b.record(main)
    torch.cuda.synchronize()
    h2d = sum(x.numel() * x.element_size() for x in (q, k, v, go))
    d2h = sum(x.numel() * x.element_size() for x in grads[0])
    # the copy bandwidth alone (one direction at a time, same buffers)
    bw = {}
    for name, fn, nbytes in (("h2d", lambda: [d.copy_(s_, non_blocking=True) for d, s_ in
                                              zip(ins[0], (hq, hk, hv, hg))], h2d),
                             ("d2h", lambda: [d.copy_(s_, non_blocking=True) for d, s_ in
                                              zip(outs[0], grads[0])], d2h)):
        fn()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(main)
        fn()
        c1.record(main)
        torch.cuda.synchronize()
        bw[name + "_gbs"] = nbytes / (c0.elapsed_time(c1) * 1e-3) / 1e9
    return {"value": a.elapsed_time(b) / n, "unit": "ms",
            "what": "H2D inputs + fwd + mask + bwd + D2H gradients, ms per step, the copies "
                    "of neighbouring steps overlapped with the compute",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "copy_bandwidth": bw}


def run_all_configs(args):
    """One JSON line per workload (and negl_prob) with the per-kernel times;
    these fill the per-configuration table, they are not the contract line."""
    import torch

    from block_sparse_attention_fwd_gb300 import _lib, build, inputs
    build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pk = _peaks()
    def timed(fn, reps):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    names = [x for x in args.configs.split(",") if x] if args.configs else [
        "tiny_n256_d64", "clustered_n4096_d64", "gqa_n8192_d128", "video_n32760_d128",
        "long_n131072_d128", "llm_causal_n16384_d128", "llm_window2048_n16384_d128"]
    for name in names:
        w = inputs.WORKLOADS[name]
        q, k, v, go = inputs.generate(w, seed=0)
        shape = _lib.make_shape(w.B, w.n, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window)
        T_r, T_c = _lib.tiles(shape)
        qd, kd, vd, god = (x.to(dev) for x in (q, k, v, go))
        o = torch.empty_like(qd)
        lse = torch.empty((w.B, w.H, w.n), dtype=torch.float32, device=dev)
        stats = torch.empty((w.B, w.H, T_c, T_r * w.block_q), dtype=torch.float32, device=dev)
        lists = _lib.alloc_lists(shape, dev)
        g_q, g_k, g_v = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        wsb = torch.empty(_lib.bwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)

        reps = 3 if w.n >= 100000 else 5
        # the tile-weights path (128 x 128 tiles): forward with the reduction
        # epilogue, statistics rows in the scratch slots only
        tw = _lib.fwd_workspace_bytes(shape) > 0
        if tw:
            logw = torch.empty((w.B, w.H, T_r, T_c), dtype=torch.float32, device=dev)
            fws = torch.empty(_lib.fwd_workspace_bytes(shape), dtype=torch.uint8, device=dev)
            fwd_tw = timed(lambda: _lib.attn_fwd_tile_weights(shape, qd, kd, vd, w.scale, o, lse,
                                                              logw, workspace=fws), reps)
        fwd = timed(lambda: _lib.attn_fwd(shape, qd, kd, vd, w.scale, o, lse, stats), reps)
        dense = timed(lambda: _lib.attn_bwd(shape, qd, kd, vd, o, god, lse, w.scale, None, g_q,
                                            g_k, g_v, wsb), reps)
        for negl in w.negl_probs:
            mask_ms = timed(lambda: _lib.mask_from_stats(shape, stats, lse, negl, lists), reps)
            bwd = timed(lambda: _lib.attn_bwd(shape, qd, kd, vd, o, god, lse, w.scale, lists, g_q,
                                              g_k, g_v, wsb), reps)
            mask = lists["mask"]
            skip = 1.0 - float(mask.float().mean())
            comp = _active_flop(mask, w)
            tw_line = {}
            if tw:
                lists_w = _lib.alloc_lists(shape, dev)
                mask_tw = timed(lambda: _lib.mask_from_tile_weights(shape, logw, negl, lists_w),
                                reps)
                if not torch.equal(lists_w["mask"], mask):
                    raise RuntimeError(f"{name}: tile-weight mask differs from the stats mask")
                tw_line = {"fwd_tw_ms": fwd_tw, "fwd_tw_frac_peak":
                           w.dense_fwd_flop() / fwd_tw / 1e9 / pk["bf16"],
                           "mask_tw_ms": mask_tw, "attn_bwd_tw_ms": mask_tw + bwd}
                del lists_w
            line = {"workload": name, "negl_prob": negl, "fwd_ms": fwd,
                    "fwd_tflops": w.dense_fwd_flop() / fwd / 1e9,
                    "mask_ms": mask_ms, "mask_gbs": _mask_bytes(w) / mask_ms / 1e6,
                    "bwd_ms": bwd, "attn_bwd_ms": mask_ms + bwd,
                    "dense_equiv_tflops": w.dense_bwd_flop() / (mask_ms + bwd) / 1e9,
                    "skip_frac": skip,
                    "frac_bf16_peak_computed_tiles": comp / bwd / 1e9 / pk["bf16"],
                    "dense_bwd_ms": dense,
                    "dense_bwd_frac_peak": w.dense_bwd_flop() / dense / 1e9 / pk["bf16"],
                    **tw_line}
            if not args.no_cpu_baseline:
                ms_cpu, desc, tiles, el = cpu_reference_sample(w, q, k, v, go, budget_s=5.0,
                                                               max_tiles=64)
                line["oracle_bwd_ms_extrapolated"] = ms_cpu
                line["oracle_sample"] = f"{tiles} query tiles in {el:.1f} s, {os.cpu_count()} cores"
            print(json.dumps(line), flush=True)
        if name == "video_n32760_d128":
            # LSE-combine of two partial results of this shape (HBM-bound)
            parts = 2
            op = torch.empty((parts,) + tuple(o.shape), dtype=torch.bfloat16, device=dev)
            op[0].copy_(o)
            op[1].copy_(o)
            lp = torch.stack([lse, lse]).contiguous()
            oc, lc = torch.empty_like(o), torch.empty_like(lse)
            cm = timed(lambda: _lib.lse_combine(op, lp, oc, lc), reps)
            rows = w.B * w.n * w.H
            nbytes = parts * rows * (2 * w.d + 4) + rows * (2 * w.d + 4)
            print(json.dumps({"workload": name, "kernel": "bl_lse_combine", "parts": parts,
                              "ms": cm, "gbs": nbytes / cm / 1e6,
                              "frac_hbm": nbytes / cm / 1e6 / pk["hbm"]}), flush=True)
            del op, lp, oc, lc
        del qd, kd, vd, god, o, lse, stats, lists, g_q, g_k, g_v, wsb
        if tw:
            del logw, fws
        torch.cuda.empty_cache()
    packed = [x for x in args.packed.split(",") if x] if args.packed else list(inputs.PACKED)
    for name in packed:
        _run_packed(inputs.PACKED[name], pk, timed, dev)
    return 0


def _packed_active_flop(mask, p, H):
    """10*d*rows*cols summed over the kept tiles of every packed sequence."""
    import torch
    w, off, total = p.base, 0, 0.0
    m = mask.to("cpu", torch.float64)
    for n in p.lengths:
        if n == 0:
            continue
        T_r, T_c = -(-n // w.block_q), -(-n // w.block_k)
        blk = m[off:off + H * T_r * T_c].view(H, T_r, T_c)
        off += H * T_r * T_c
        rows = torch.full((T_r,), w.block_q, dtype=torch.float64)
        rows[-1] = n - (T_r - 1) * w.block_q
        cols = torch.full((T_c,), w.block_k, dtype=torch.float64)
        cols[-1] = n - (T_c - 1) * w.block_k
        total += float(10.0 * w.d * torch.einsum("hij,i,j->", blk, rows, cols))
    return total


def _run_packed(p, pk, timed, dev):
    """One JSON line per packed variable-length workload: the three calls with
    the runs spread over the library's side streams (default) and one after
    another on the caller's stream (streams = 1)."""
    import torch

    from block_sparse_attention_fwd_gb300 import _lib, inputs
    w = p.base
    cu, q, k, v, go = inputs.generate_packed(w, p.lengths, seed=0)
    qd, kd, vd, god = (x.to(dev) for x in (q, k, v, go))
    line = {"workload": p.name, "sequences": len(p.lengths), "total_tokens": p.total,
            "lengths": list(p.lengths), "negl_prob": w.negl_probs[0]}
    for streams in (0, 1):
        vl = _lib.Varlen(cu, w.H, w.Hk, w.d, w.block_q, w.block_k, w.causal, w.window, streams)
        o = torch.empty_like(qd)
        lse = torch.empty(vl.sizes["lse"], dtype=torch.float32, device=dev)
        stats = torch.empty(vl.sizes["tile_stats"], dtype=torch.float32, device=dev)
        lists = _lib.alloc_varlen_lists(vl, dev)
        g = [torch.empty_like(x) for x in (qd, kd, vd)]
        ws = torch.empty(vl.sizes["bwd_workspace_bytes"], dtype=torch.uint8, device=dev)
        negl = w.negl_probs[0]
        fwd = timed(lambda: _lib.attn_fwd_varlen(vl, qd, kd, vd, w.scale, o, lse, stats), 5)
        mask_ms = timed(lambda: _lib.mask_from_stats_varlen(vl, stats, lse, negl, lists), 5)
        bwd = timed(lambda: _lib.attn_bwd_varlen(vl, qd, kd, vd, o, god, lse, w.scale, lists,
                                                 *g, ws), 5)
        dense = timed(lambda: _lib.attn_bwd_varlen(vl, qd, kd, vd, o, god, lse, w.scale, None,
                                                   *g, ws), 5)
        if _lib.varlen_bwd_check_status(vl, ws) != 0:
            raise RuntimeError("packed backward reported a bad status")
        tag = "" if streams == 0 else "_serial"
        line.update({f"fwd_ms{tag}": fwd, f"mask_ms{tag}": mask_ms, f"bwd_ms{tag}": bwd,
                     f"dense_bwd_ms{tag}": dense})
        if streams == 0:
            comp = _packed_active_flop(lists["mask"], p, w.H)
            line.update({"launch_groups": vl.sizes["groups"],
                         "fwd_frac_peak": p.dense_fwd_flop() / fwd / 1e9 / pk["bf16"],
                         "skip_frac": 1.0 - float(lists["mask"].float().mean()),
                         "frac_bf16_peak_computed_tiles": comp / bwd / 1e9 / pk["bf16"],
                         "dense_bwd_frac_peak": p.dense_bwd_flop() / dense / 1e9 / pk["bf16"]})
        del o, lse, stats, lists, g, ws
    print(json.dumps(line), flush=True)
    del qd, kd, vd, god
    torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--negl", type=float, default=NEGL)
    ap.add_argument("--dense-iters", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=15.0)
    ap.add_argument("--ref-tiles", type=int, default=256)
    ap.add_argument("--configs", default="",
                    help="comma-separated workloads for --all-configs (default: all)")
    ap.add_argument("--packed", default="",
                    help="comma-separated packed workloads for --all-configs (default: all)")
    ap.add_argument("--all-configs", action="store_true",
                    help="per-workload kernel times (not the contract line)")
    args = ap.parse_args()
    if args.all_configs:
        return run_all_configs(args)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
