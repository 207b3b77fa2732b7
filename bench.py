"""Benchmark of the masked attention forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--quick]

One step = one masked attention forward over the headline workload (the
128K-token block-sparse causal prefill: B1 H32 N131072 d128 bf16, block 128,
diagonal + first column kept, other causal blocks Bernoulli(0.5)), i.e. the
whole hot path: device tile walk, TMA loads, Q K^T, boundary masking, online
softmax, P V, epilogue.  Metric: effective TFLOP/s = 4 * d * (exact unmasked
query-key pairs) / time.  The other workloads (tiny fp32 ViT, 896^2 and
1792^2 ViT layers, head-wise causal windows with sinks) are timed kernel by
kernel and reported under "workloads".

With --gpus N > 1 (launched by torchrun) every rank runs an independent
replica of the step on its own GPU (the path has no exchange step); the time
is the max over ranks and value = all ranks' units / that time ("weak").
--impl reference times the fp64 CPU oracle (the reference arm here) on a
bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "effective attention TFLOP/s (unmasked FLOPs) and % of GB300 BF16 peak"
HEADLINE = ("bsparse128k", "block128")
KERNEL_SOURCES = ["block_sparse_attention_masked_gb300/csrc/attention_fwd.cu",
                  "block_sparse_attention_masked_gb300/csrc/attention_tiles.cuh",
                  "block_sparse_attention_masked_gb300/csrc/ptx.cuh",
                  "block_sparse_attention_masked_gb300/csrc/plan_rules.h",
                  "block_sparse_attention_masked_gb300/csrc/tile_mma.cuh"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def profile_traffic(workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it matches the
    current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"attention_fwd_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return int(float(vals["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ masks and counts
def spec_head(spec, h: int):
    """The mask of head h alone (a one-head MaskSpec for the oracle)."""
    from workloads import MaskSpec

    pick = lambda xs: None if xs is None else [xs[h]]  # noqa: E731
    blk = None
    if spec.block is not None:
        b = np.asarray(spec.block)
        blk = b[h:h + 1] if b.ndim == 3 else b
    sink = None if spec.sink is None else np.asarray(spec.sink)[h:h + 1]
    return MaskSpec(spec.kind, [spec.head_param[h]], perm=pick(spec.perm), perm_grid=pick(spec.perm_grid),
                    block=blk, sink=sink, sink_tokens=getattr(spec, "sink_tokens", 0))


def block_mask_pairs(spec, N: int, B: int = 1) -> int:
    """Visible (query, key) pairs of a block-selection mask with N a multiple
    of the block size: a kept block below the diagonal has Bs^2 pairs, a kept
    diagonal block Bs (Bs + 1) / 2 (causality inside it); blocks above the
    diagonal count nothing.  The unit count of the FLOP metric for the
    reference arm, which does not load the library."""
    blk = np.asarray(spec.block, dtype=bool)
    if blk.ndim == 2:
        blk = blk[None]
    total = 0
    for h in range(len(spec.head_param)):
        bh = blk[h] if blk.shape[0] > 1 else blk[0]
        bs = int(spec.head_param[h])
        if N % bs:
            raise ValueError("N must be a multiple of the block size")
        total += int(np.tril(bh, -1).sum()) * bs * bs + int(np.diag(bh).sum()) * bs * (bs + 1) // 2
    return B * total


def cpu_info() -> dict:
    """The host cores this process may use and the BLAS thread pool size."""
    info = {"affinity": len(os.sched_getaffinity(0)), "nproc": os.cpu_count()}
    try:
        import threadpoolctl

        pools = threadpoolctl.threadpool_info()
        info["blas_threads"] = max((i.get("num_threads", 0) for i in pools), default=0)
    except Exception:
        info["blas_threads"] = None
    return info


def numa_info(gpu_index: int) -> dict:
    """NUMA node of the GPU (sysfs) and the nodes of the host."""
    out = {}
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.strip().lower()
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{dom[-4:]}:{rest}/numa_node"
        with open(path) as f:
            out["gpu_node"] = int(f.read().strip())
    except Exception:
        out["gpu_node"] = None
    try:
        out["host_nodes"] = len([n for n in os.listdir("/sys/devices/system/node") if n.startswith("node")])
    except Exception:
        out["host_nodes"] = None
    return out


def headline_config(wl, mask_name: str, pairs: int, world: int) -> dict:
    """The `config` of the benchmark line, the same in both arms."""
    in_bytes = wl.B * (wl.H + 2 * (wl.kv_heads or wl.H)) * wl.N * wl.d * (4 if wl.dtype == "f32" else 2)
    l2 = (f"inputs larger than L2 ({in_bytes / 2**30:.2f} GiB)" if in_bytes > 2 * 129e6
          else "flushed (512 MiB write) before each run")
    return {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d, "mask": mask_name,
            "mask_detail": wl.description, "pairs": int(pairs), "l2": l2,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ------------------------------------------------------------------ distributed
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    _n = 0

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        ClockSampler._n += 1  # one file per sampler: several may be open in one process
        self.path = os.path.join("/tmp", f"mattn_clocks_{os.getpid()}_{ClockSampler._n}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, maxes, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.remove(self.path)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------------ GPU arm
def effective_flops(pairs: int, d: int) -> float:
    return 4.0 * d * pairs


def time_kernel(fn, iters: int, warmup: int, flush=None):
    """Median CUDA-event time (ms) of fn() over iters runs, L2 flushed before each."""
    import torch

    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        if flush is not None:
            flush()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    return statistics.median(times), times


def run_gpu(args):
    import torch

    import block_sparse_attention_masked_gb300 as mattn
    from workloads import WORKLOADS, make_mask, make_workload_inputs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    mattn.lib()
    peaks = measured_peaks()
    dev = f"cuda:{local}"

    # ---------------- headline step
    wl_name, mask_name = args.workload or HEADLINE[0], args.mask or HEADLINE[1]
    wl = WORKLOADS[wl_name]
    if args.n or args.heads:  # same recipe at a smaller size (profiling cases)
        import dataclasses

        wl = dataclasses.replace(wl, N=args.n or wl.N, H=args.heads or wl.H)
    q, k, v = make_workload_inputs(wl, seed=0, device=dev)
    spec = make_mask(wl, mask_name, seed=0)
    mask = mattn.prepare(spec, wl.H, wl.N, device=dev)
    pairs = mattn.count_pairs(spec, wl.B, wl.H, wl.N)
    if spec.kind == "block" and pairs != block_mask_pairs(spec, wl.N, wl.B):
        raise RuntimeError("the library's pair count differs from the bitmap's")
    flops = effective_flops(pairs, wl.d)
    o = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        mattn.attention(q, k, v, mask, out=o, lse=lse)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    rc, word = mattn.device_status()
    if rc != 0:
        raise RuntimeError(f"device error word {word:#x} after warm-up")
    with ClockSampler(local) as clk:
        barrier(dist)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        t0 = time.perf_counter()
        for s, e in ev:
            s.record(stream)
            step()
            e.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        barrier(dist)
    clocks = clk.summary()  # the timed region's samples, read before any other sampler runs
    step_ms = [s.elapsed_time(e) for s, e in ev]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(dist, total_ms, device=dev)
    ms_per_step = total_ms / args.steps
    rc, word = mattn.device_status()
    if rc != 0:
        raise RuntimeError(f"device error word {word:#x} after timed steps")
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12
    per_launch_ms = statistics.mean(step_ms)
    achieved = flops / (per_launch_ms * 1e-3) / 1e12
    traffic = profile_traffic(wl_name)

    # ---------------- end to end through the host-buffer entry point (before the
    # oracle's host work below, which would share the host with its copies)
    e2e = None
    if not args.quick:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32).pin_memory()
        hmask = mattn.PreparedMask(spec, wl.H, wl.N, host_side=True)
        for _ in range(max(1, min(args.warmup, 2))):
            mattn.attention_host(qh, kh, vh, hmask, out=oh, lse=lh)
        e2e_steps = max(1, min(args.steps, 10))
        barrier(dist)
        torch.cuda.synchronize()
        with ClockSampler(local) as e2e_clk:
            t0 = time.perf_counter()
            call_ms = []
            for _ in range(e2e_steps):
                tc = time.perf_counter()
                mattn.attention_host(qh, kh, vh, hmask, out=oh, lse=lh)
                call_ms.append(round(1e3 * (time.perf_counter() - tc), 3))
            e2e_s = max_over_ranks(dist, time.perf_counter() - t0, device=dev)
        barrier(dist)
        tensor_bytes = q.numel() * q.element_size()
        bits_bytes = int(hmask.block_words_host.nbytes) if spec.kind == "block" else 0
        # the host link alone: one pinned copy of q in and of o out, timed on the device
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        q.copy_(qh, non_blocking=True)
        s1.record()
        s1.synchronize()
        h2d_gbs = tensor_bytes / (s0.elapsed_time(s1) * 1e-3) / 1e9
        s0.record()
        oh.copy_(o, non_blocking=True)
        s1.record()
        s1.synchronize()
        d2h_gbs = tensor_bytes / (s0.elapsed_time(s1) * 1e-3) / 1e9
        e2e_ms = 1e3 * e2e_s / e2e_steps
        in_bytes, out_bytes = 3 * tensor_bytes + bits_bytes, tensor_bytes + lse.numel() * 4
        e2e = {"value": round(world * flops * e2e_steps / e2e_s / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "ms_per_step": round(e2e_ms, 3), "calls_ms": call_ms, "clocks": e2e_clk.summary(),
               "entry_point": "mattn_fwd_host",
               "h2d_gbs": round(h2d_gbs, 1), "d2h_gbs": round(d2h_gbs, 1),
               "copy_ms_at_those_rates": round(1e3 * (in_bytes / (h2d_gbs * 1e9) + out_bytes / (d2h_gbs * 1e9)), 2),
               "device_ms_per_step": round(ms_per_step, 3), "kernel_share": round(ms_per_step / e2e_ms, 3),
               "numa": numa_info(local), "host_cpus": cpu_info(),
               "host_buffers_pinned": all(t.is_pinned() for t in (qh, kh, vh, oh, lh))}
        del qh, kh, vh, oh, lh

    # ---------------- the oracle on the GPU arm's own inputs (sampled rows)
    parity = {}
    cpu = None
    if rank == 0 and world == 1 and not args.quick:
        rows = sampled_rows(wl.N, 128, seed=1, extra=55)
        heads = [0, wl.H - 1]
        chk, secs, pr = oracle_check(q, k, v, o, lse, spec, heads, rows)
        parity[f"{wl_name}/{mask_name}"] = chk
        st_rows = rows[:16]
        st_secs = oracle_single_thread(q, k, v, spec, 0, st_rows)
        st_pairs = rows_pairs(spec, 0, wl.N, st_rows)
        ci = cpu_info()
        cpu = {"value": round(effective_flops(pr, wl.d) / secs / 1e12, 6), "unit": "TFLOP/s",
               "cores": ci["affinity"], "cores_detail": ci, "kind": "oracle",
               "sample": f"{wl_name}/{mask_name}: heads {heads}, {len(rows)} query rows each (first, last, block "
                         f"edges, middle, random), every key scored in fp64 (numpy), {secs:.2f} s on all "
                         f"{ci['affinity']} cores",
               "single_thread": None if st_secs is None else {
                   "value": round(effective_flops(st_pairs, wl.d) / st_secs / 1e12, 6), "unit": "TFLOP/s",
                   "sample": f"head 0, {len(st_rows)} rows, one BLAS thread, {st_secs:.2f} s"}}

    del q, k, v, o, lse
    torch.cuda.empty_cache()

    # ---------------- every workload, kernel by kernel
    workloads = {}
    if not args.quick:
        flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

        def flush():
            flush_buf.zero_()

        for name, wlx in WORKLOADS.items():
            if name.startswith("decode"):
                workloads.update(decode_sweep(name, wlx, dev, peaks))
                continue
            qx, kx, vx = make_workload_inputs(wlx, seed=0, device=dev)
            in_bytes = (qx.numel() + kx.numel() + vx.numel()) * qx.element_size()
            for m in wlx.masks:
                sp = make_mask(wlx, m, seed=0)
                mk = mattn.prepare(sp, wlx.H, wlx.N, device=dev)
                ox = torch.empty_like(qx)
                lx = torch.empty((wlx.B, wlx.H, wlx.N), dtype=torch.float32, device=dev)
                pr = mattn.count_pairs(sp, wlx.B, wlx.H, wlx.N)
                fl = effective_flops(pr, wlx.d)
                iters = 5 if name == "bsparse128k" else 20
                med, _ = time_kernel(lambda: mattn.attention(qx, kx, vx, mk, out=ox, lse=lx), iters, 3,
                                     flush=None if in_bytes > 2 * 129e6 else flush)
                out_bytes = ox.numel() * ox.element_size() + lx.numel() * 4
                tf = fl / (med * 1e-3) / 1e12
                t_flop = fl / (peaks["bf16_tflops"] * 1e12)
                t_byte = (in_bytes + out_bytes) / (peaks["hbm_gbs"] * 1e9)
                workloads[f"{name}/{m}"] = {
                    "ms": round(med, 4), "tflops": round(tf, 1), "pct_peak": round(100 * tf / peaks["bf16_tflops"], 1),
                    "pct_own_roofline": round(100 * max(t_flop, t_byte) / (med * 1e-3), 1),
                    "roofline_bound": "tensor" if t_flop >= t_byte else "hbm",
                    "schedule": mattn.plan_schedule(mk, wlx.B, wlx.N, wlx.d,
                                                    mattn.F32 if wlx.dtype == "f32" else mattn.BF16),
                    "pairs": pr, "hbm_gbs_min_traffic": round((in_bytes + out_bytes) / (med * 1e-3) / 1e9, 1),
                    "l2": "inputs > L2" if in_bytes > 2 * 129e6 else "flushed (512 MiB write) before each run"}
                if rank == 0 and name == "vit16384" and m == "sliding256_rowcol":
                    # raster heads 0 and 7, column-major heads 8 and 15
                    rows = sampled_rows(wlx.N, 256, seed=2, extra=40)
                    chk, _, _ = oracle_check(qx, kx, vx, ox, lx, sp, [0, 7, 8, 15], rows)
                    parity[f"{name}/{m}"] = chk
            if name == "bsparse128k":
                # RRAttention's block selection on the same inputs (stride 8,
                # block 128, tau 0.95): algorithmic work = Eq. 8's product,
                # 2 d (L/S)^2 FLOPs per head (the kernel forms it twice:
                # one pass for the row log-sum-exp, one for the block sums)
                S_rr, bs_rr, tau_rr = 8, 128, 0.95
                med, _ = time_kernel(lambda: mattn.rr_select(qx, kx, S_rr, bs_rr, tau_rr), 5, 3)
                ns = wlx.N // S_rr
                fl = 2.0 * wlx.d * ns * ns * wlx.B * wlx.H
                bits, _ = mattn.rr_select(qx, kx, S_rr, bs_rr, tau_rr)
                nbk = wlx.N // bs_rr
                kept = int(np.unpackbits(bits.cpu().numpy().view(np.uint8)).sum())
                workloads[f"{name}/rr_select_s8_b128_tau0.95"] = {
                    "ms": round(med, 4), "tflops_eq8": round(fl / (med * 1e-3) / 1e12, 1),
                    "kept_causal_block_fraction": round(kept / (wlx.B * wlx.H * nbk * (nbk + 1) / 2), 4),
                    "share_of_attention_step": round(med / workloads[f"{name}/{wlx.masks[0]}"]["ms"], 4),
                    "l2": "inputs > L2"}
                del bits
            if name in ("bsparse128k", "vit16384"):
                # received attention (column sums of the attention matrix) of
                # the workload's first mask, from the forward's LSE: one
                # QK^T product per visible pair, 2 d FLOPs
                m0 = wlx.masks[0]
                mk = mattn.prepare(make_mask(wlx, m0, seed=0), wlx.H, wlx.N, device=dev)
                _, lx = mattn.attention(qx, kx, vx, mk)
                rx = torch.empty_like(lx)
                med, _ = time_kernel(lambda: mattn.received(qx, kx, lx, mk, out=rx), 5 if name == "bsparse128k" else 20,
                                     3, flush=None if name == "bsparse128k" else flush)
                pr = workloads[f"{name}/{m0}"]["pairs"]
                workloads[f"{name}/received_{m0}"] = {
                    "ms": round(med, 4), "tflops_qk": round(2.0 * wlx.d * pr / (med * 1e-3) / 1e12, 1),
                    "pct_peak": round(100 * 2.0 * wlx.d * pr / (med * 1e-3) / 1e12 / peaks["bf16_tflops"], 1)}
                del lx, rx
            del qx, kx, vx
            torch.cuda.empty_cache()
        rc, word = mattn.device_status()
        if rc != 0:
            raise RuntimeError(f"device error word {word:#x} after the workload sweep")


    sched = mattn.plan_schedule(mask, wl.B, wl.N, wl.d, mattn.F32 if wl.dtype == "f32" else mattn.BF16)
    family = {"paired": "attention_fwd_kernel", "split": "attention_fwd_kernel",
              "persistent": "attention_persist_kernel", "single": "attention_sp_kernel"}.get(sched, sched)
    headline_kernel = f"{family}<{wl.d}> ({sched} schedule)"
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": headline_config(wl, mask_name, pairs, world),
            "pct_of_peak": round(100 * value / world / peaks["bf16_tflops"], 1),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "traffic": traffic,
                         "traffic_source": (None if traffic is None else
                                            f"carried from the committed ncu capture profiles/attention_fwd_{wl_name}.md "
                                            f"(kernel source hash {kernel_source_hash()}); not measured in this run"),
                         "peak_source": peaks["source"] + " burst bf16 (cuBLAS)",
                         "kernel": headline_kernel},
            "cpu_baseline": cpu,
            "parity": parity,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clocks,
            "wall_s_timed": round(wall, 3),
            "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------ oracle comparison and CPU baseline
def sampled_rows(N: int, edge: int, seed: int, extra: int) -> np.ndarray:
    """Query rows the oracle checks: the first and last rows, rows on both
    sides of a block / window edge and of the middle, and `extra` random
    ones (seeded)."""
    rng = np.random.default_rng(seed)
    edges = [0, 1, edge - 1, edge, N // 2 - 1, N // 2, N - edge - 1, N - edge, N - 1]
    rows = {int(r) for r in edges if 0 <= r < N}
    rows |= {int(r) for r in rng.choice(N, extra, replace=False)}
    return np.array(sorted(rows), dtype=np.int64)


def oracle_check(q, k, v, o, lse, spec, heads, rows):
    """The fp64 oracle on the GPU arm's own inputs, for the given heads and
    query rows, against the GPU's outputs.  Returns the errors (max abs and
    relative L2 over O, max abs over the LSE), the oracle's seconds and the
    visible pairs of the rows (the FLOP metric's units)."""
    from oracle import dense

    num = den = 0.0
    max_abs = lse_err = 0.0
    secs = 0.0
    pairs = 0
    group = q.shape[1] // k.shape[1]
    for h in heads:
        qh = q[0, h].float().cpu().numpy()[None, None]
        kh = k[0, h // group].float().cpu().numpy()[None, None]
        vh = v[0, h // group].float().cpu().numpy()[None, None]
        sub = spec_head(spec, h)
        t0 = time.perf_counter()
        ro, rl = dense.attention(qh, kh, vh, sub, rows=rows)
        secs += time.perf_counter() - t0
        go = o[0, h].float().cpu().numpy()[rows].astype(np.float64)
        gl = lse[0, h].cpu().numpy()[rows].astype(np.float64)
        diff = go - ro[0]
        max_abs = max(max_abs, float(np.abs(diff).max()))
        num += float((diff ** 2).sum())
        den += float((ro[0] ** 2).sum())
        fin = np.isfinite(rl[0])
        if fin.any():
            lse_err = max(lse_err, float(np.abs(gl[fin] - rl[0][fin]).max()))
        pairs += rows_pairs(spec, h, q.shape[2], rows)
    return {"max_abs": max_abs, "rel_l2": (num / den) ** 0.5 if den > 0 else 0.0, "lse_max_abs": lse_err,
            "rows": int(len(rows)), "heads": [int(h) for h in heads]}, secs, pairs


def rows_pairs(spec, h: int, N: int, rows) -> int:
    """Visible pairs of the given caller-order query rows of head h."""
    from oracle import dense

    sub = spec_head(spec, h)
    pos = dense.inverse_permutation(dense._head_perm(sub, 0), N)
    return sum(int(dense.dense_mask_strip(sub, 0, N, int(pos[r]), int(pos[r]) + 1).sum()) for r in rows)


SINGLE_THREAD_CHILD = r"""
import sys, time, numpy as np
sys.path.insert(0, sys.argv[1])
from oracle import dense
import pickle
d = np.load(sys.argv[2], allow_pickle=False)
with open(sys.argv[3], "rb") as f:
    spec = pickle.load(f)
t0 = time.perf_counter()
dense.attention(d["q"], d["k"], d["v"], spec, rows=d["rows"])
print(time.perf_counter() - t0)
"""


def oracle_single_thread(q, k, v, spec, h, rows):
    """Seconds of the oracle on one head's rows in a child process whose BLAS
    runs one thread (the thread count of a numpy BLAS is fixed at import)."""
    import pickle
    import tempfile

    with tempfile.TemporaryDirectory() as tmp:
        group = q.shape[1] // k.shape[1]
        data = os.path.join(tmp, "d.npz")
        np.savez(data, q=q[0, h].float().cpu().numpy()[None, None], k=k[0, h // group].float().cpu().numpy()[None, None],
                 v=v[0, h // group].float().cpu().numpy()[None, None], rows=rows)
        sp = os.path.join(tmp, "s.pkl")
        with open(sp, "wb") as f:
            pickle.dump(spec_head(spec, h), f)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                   BLIS_NUM_THREADS="1")
        res = subprocess.run([sys.executable, "-c", SINGLE_THREAD_CHILD, ROOT, data, sp], capture_output=True,
                             text=True, env=env, timeout=600)
        if res.returncode != 0:
            return None
        return float(res.stdout.strip().splitlines()[-1])


# ------------------------------------------------------------------ other stages (profiling aid)
def decode_visible_keys(spec, h: int, length: int) -> int:
    """Keys the decode query (position length - 1) of head h sees."""
    if spec.kind == "full":
        return length
    w = int(spec.head_param[h])
    win = min(w, length)
    return win + max(0, min(int(spec.sink_tokens or 0), length - win))


def decode_sweep(name, wl, dev, peaks):
    """Decode steps of a workload: one query per sequence against a full
    cache of wl.N tokens.  HBM-bound: the K and V rows each step reads."""
    import torch
    import block_sparse_attention_masked_gb300 as mattn
    from workloads import make_decode_inputs, make_mask

    q, k, v = make_decode_inputs(wl, seed=0, device=dev)
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    out = {}
    kv = wl.kv_heads or wl.H
    for m in wl.masks:
        sp = make_mask(wl, m, seed=0)
        mk = mattn.prepare(sp, wl.H, wl.N, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((wl.B, wl.H), dtype=torch.float32, device=dev)
        # distinct K/V rows read: the union of the group's visible keys (the
        # heads of a group share one window size here)
        rows = wl.B * kv * decode_visible_keys(sp, 0, wl.N)
        big = rows * wl.d * 4 > 2 * 129e6
        med, _ = time_kernel(lambda: mattn.decode(q, k, v, mk, out=o, lse=lse), 20, 3,
                             flush=None if big else (lambda: flush_buf.zero_()))
        pairs = wl.B * sum(decode_visible_keys(sp, h, wl.N) for h in range(wl.H))
        group = wl.H // kv
        bytes_rw = 2 * rows * wl.d * 2 + q.numel() * 2 * 2 + lse.numel() * 4
        gbs = bytes_rw / (med * 1e-3) / 1e9
        out[f"{name}/{m}"] = {
            "ms": round(med, 4), "tflops": round(4.0 * wl.d * pairs / (med * 1e-3) / 1e12, 2),
            "hbm_gbs": round(gbs, 1), "pct_hbm": round(100 * gbs / peaks["hbm_gbs"], 1),
            "kv_rows_read": rows, "query_heads_per_kv_head": group,
            "l2": "rows read larger than L2" if big else "flushed (512 MiB write) before each run"}
    del q, k, v, flush_buf
    torch.cuda.empty_cache()
    return out


def run_stage(args):
    """Time RRAttention's block selection (stride 8, block 128, tau 0.95) or
    the received attention on the headline workload's inputs: warm-up, then
    ``steps`` timed calls; one short JSON line."""
    import dataclasses

    import torch

    import block_sparse_attention_masked_gb300 as mattn
    from workloads import WORKLOADS, make_mask, make_workload_inputs

    torch.cuda.set_device(0)
    if args.stage == "decode":
        from workloads import make_decode_inputs

        wl = WORKLOADS[args.workload or "decode128k"]
        if args.n:
            wl = dataclasses.replace(wl, N=args.n)
        q, k, v = make_decode_inputs(wl, seed=0, device="cuda")
        dmask = mattn.prepare(make_mask(wl, args.mask or wl.masks[0], seed=0), wl.H, wl.N)
        o = torch.empty_like(q)
        lse = torch.empty((wl.B, wl.H), dtype=torch.float32, device="cuda")
        med, _ = time_kernel(lambda: mattn.decode(q, k, v, dmask, out=o, lse=lse), args.steps, args.warmup)
        rc, word = mattn.device_status()
        if rc != 0:
            raise RuntimeError(f"device error word {word:#x}")
        print(json.dumps({"stage": "decode", "workload": wl.name, "mask": args.mask or wl.masks[0], "L": wl.N,
                          "H": wl.H, "H_kv": wl.kv_heads, "d": wl.d, "ms_median": round(med, 4),
                          "steps": args.steps}), flush=True)
        return
    wl = WORKLOADS[args.workload or HEADLINE[0]]
    if args.n or args.heads:
        wl = dataclasses.replace(wl, N=args.n or wl.N, H=args.heads or wl.H)
    q, k, v = make_workload_inputs(wl, seed=0, device="cuda")
    if args.stage == "rr_select":
        def fn():
            mattn.rr_select(q, k, 8, 128, 0.95)
    else:
        mask = mattn.prepare(make_mask(wl, args.mask or HEADLINE[1], seed=0), wl.H, wl.N)
        _, lse = mattn.attention(q, k, v, mask)
        r = torch.empty_like(lse)

        def fn():
            mattn.received(q, k, lse, mask, out=r)
    med, times = time_kernel(fn, args.steps, args.warmup)
    rc, word = mattn.device_status()
    if rc != 0:
        raise RuntimeError(f"device error word {word:#x}")
    print(json.dumps({"stage": args.stage, "workload": wl.name,
                      "N": wl.N, "H": wl.H, "d": wl.d, "ms_median": round(med, 4), "steps": args.steps}), flush=True)


# ------------------------------------------------------------------ oracle (CPU) arm
def oracle_sample(seconds_target: float = 15.0):
    """Time the oracle on sampled rows of head 0 of the headline workload.

    Inputs are drawn with the workload recipe on the CPU (same shapes and
    distribution); returns (effective TFLOP/s, seconds, rows, description)."""
    import torch

    from oracle import dense
    from workloads import WORKLOADS, make_mask

    wl_name, mask_name = HEADLINE
    wl = WORKLOADS[wl_name]
    g = torch.Generator().manual_seed(0)
    shape = (1, 1, wl.N, wl.d)
    q, k, v = (torch.randn(shape, generator=g).to(torch.bfloat16).float().numpy() for _ in range(3))
    spec = make_mask(wl, mask_name, seed=0, heads=1)
    rng = np.random.default_rng(0)
    rows_all = rng.permutation(wl.N)
    done_rows, t_total, pairs = 0, 0.0, 0
    chunk = 32
    while t_total < seconds_target and done_rows + chunk <= wl.N:
        rows = np.sort(rows_all[done_rows:done_rows + chunk])
        t0 = time.perf_counter()
        dense.attention(q, k, v, spec, rows=rows)
        t_total += time.perf_counter() - t0
        blk = np.asarray(spec.block)[0]
        bs = spec.head_param[0]
        for r in rows:  # allowed keys of row r (counted outside the timed region)
            m = r // bs
            kept = np.nonzero(blk[m, :m])[0]
            pairs += len(kept) * bs + (r - m * bs + 1) * int(blk[m, m])
        done_rows += chunk
    tf = effective_flops(pairs, wl.d) / t_total / 1e12
    desc = (f"{wl_name}/{mask_name}: {done_rows} random query rows of head 0, all {wl.N} keys scored in fp64 "
            f"(numpy), {t_total:.1f} s")
    return tf, t_total, done_rows, desc


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        oracle_sample(0.5)
    vals, secs = [], 0.0
    rows_total = 0
    for _ in range(args.steps):
        tf, s, rows, desc = oracle_sample(per_step)
        vals.append(tf)
        secs += s
        rows_total += rows
    value = statistics.mean(vals)
    from workloads import WORKLOADS, make_mask

    wl = WORKLOADS[HEADLINE[0]]
    spec = make_mask(wl, HEADLINE[1], seed=0)
    ci = cpu_info()
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * secs / args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": headline_config(wl, HEADLINE[1], block_mask_pairs(spec, wl.N, wl.B), world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": ci["affinity"], "cores_detail": ci,
                         "kind": "oracle",
                         "sample": f"{rows_total} sampled query rows of head 0 over {args.steps} steps"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline step only (no e2e, sweep or oracle)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--workload", default=None, help="headline workload name (default bsparse128k)")
    ap.add_argument("--mask", default=None, help="mask of that workload")
    ap.add_argument("--n", type=int, default=0, help="shrink N (profiling cases)")
    ap.add_argument("--heads", type=int, default=0, help="shrink H (profiling cases)")
    ap.add_argument("--stage", default="attention", choices=["attention", "rr_select", "received", "decode"],
                    help="profiling aid: time one other stage on the headline inputs instead of the step "
                         "(prints a short line, not the benchmark record)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.stage != "attention":
        run_stage(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
