"""Benchmark: 3D-RoPE full spatiotemporal attention on the Wan-14B 720p shape (B=2, 40 heads,
d=128, latent grid 21x45x80 = 75600 tokens, bf16), one call = one step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints one JSON line.  `value` is achieved TFLOP/s (4*B*H*N^2*d per call) summed over ranks,
timed with CUDA events on the launching stream over K back-to-back calls whose inputs are
already resident in HBM (each of q, k, v is 1.55 GB, far larger than the 129 MB L2, so no L2
flush is needed).  `e2e` times the same call through the public API with the inputs copied
from pinned host memory and the output and lse copied back inside the timed region.  With
N > 1 (torchrun) every rank runs an independent replica of the whole workload.
`--impl reference` times the fp64 CPU oracle on a bounded sample of rows instead.
"""
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

from video_diffusion_transformer_rope_gb300 import configs, synth  # noqa: E402

KERNEL_SRC = os.path.join(ROOT, "video_diffusion_transformer_rope_gb300", "csrc", "attn_fwd_sm103.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_bf16_sm103_traffic.txt")
METRIC = "3D-RoPE attention TFLOP/s (4*B*H*N^2*d per call), Wan-14B 720p shape, 1 GB300"
L2_BYTES = 129 * 2**20


def metric_for(w):
    """The headline metric string for the Wan-14B 720p workload; the same metric named after
    the shape for the other workloads."""
    if w.name == configs.WAN14B_720P.name:
        return METRIC
    return (f"3D-RoPE attention TFLOP/s (4*B*H*N^2*d per call), {w.name} shape "
            f"(B={w.B}, H={w.H}, N={w.N}), 1 GB300")


def _l2_note(w):
    each = w.B * w.N * w.H * w.d * (4 if w.dtype == "f32" else 2)
    if each > L2_BYTES:
        return f"inputs larger than L2 (q, k, v {each / 1e9:.2f} GB each); no flush"
    return f"inputs smaller than L2 (q, k, v {each / 1e6:.2f} MB each): L2-resident across calls"


METRIC_WINDOW = "windowed 3D-RoPE attention TFLOP/s (4*d per kept query-key pair), 1 GB300"
METRIC_SUBSET = "active-query 3D-RoPE attention TFLOP/s (4*d per active query-key pair), 1 GB300"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0) or 0), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def _source_hash():
    """Hash of the attention kernel's code with comments and blank space removed, so that a
    stored DRAM-traffic figure stays attached to the code it was measured on."""
    import hashlib
    import re
    with open(KERNEL_SRC) as f:
        src = f.read()
    src = re.sub(r"//[^\n]*", "", src)
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = "\n".join(line.strip() for line in src.splitlines() if line.strip())
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def _traffic_per_launch(workload, kernel, k_rope="prepass"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel
    (same source, same kernel variant and K rotation mode, same workload)."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    key, val = line.split(":", 1)
                    kv[key.strip()] = val.strip()
        if (kv.get("kernel_source_sha256_16") != _source_hash() or kv.get("workload") != workload or
                kv.get("kernel", "single") != kernel or kv.get("k_rope", "prepass") != k_rope):
            return None
        return float(kv["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.out,
                stderr=subprocess.DEVNULL)
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
            self.out.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                try:
                    pw.append(float(parts[3]))
                except ValueError:
                    pw.append(float("nan"))
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        watts = [w for w in pw if w == w]
        out = {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "samples": len(sm),
               "reasons": sorted(reasons)}
        if watts:
            out["power_w_median"] = statistics.median(watts)
            out["power_w_max"] = max(watts)
        return out


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max_over_ranks(x, ws, device):
    """Largest x over all ranks (the slowest rank's time); identity on one rank."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(work_per_rank, ms_per_step_max, ws):
    """Whole-job throughput: every rank runs its own replica of `work_per_rank` FLOP per step;
    the job takes as long as the slowest rank."""
    return ws * work_per_rank / (ms_per_step_max * 1e-3) / 1e12


# One oracle sample: ORACLE_HEADS (b, h) pairs x ORACLE_ROWS query rows each.  The CPU
# baseline leg of the GPU run and the reference arm time the very same samples, so their
# TFLOP/s agree up to noise (the oracle rotates a head's K once per sample, so the per-row
# cost depends on the rows per head).
ORACLE_HEADS, ORACLE_ROWS = 2, 512


def _cpu_oracle_sample(w, q, k, v, seed=0):
    """Time the oracle (as it stands) on one sample of the workload, inputs already on the
    host.  Returns (seconds, rows)."""
    import numpy as np
    import oracle.fp64 as O
    rng = np.random.default_rng(seed)
    rows = []
    for i in range(ORACLE_HEADS):
        b, h = ((seed + i) % w.B), ((seed + i) * 7) % w.H
        for n in rng.choice(w.N, ORACLE_ROWS, replace=False):
            rows.append((b, h, int(n)))
    t0 = time.perf_counter()
    O.rope3d_attention_rows(q, k, v, (w.T, w.Hg, w.Wg), rows, w.sections, w.theta)
    return time.perf_counter() - t0, len(rows)


def _oracle_tflops(w, seconds, rows):
    return 4.0 * w.N * w.d * rows / seconds / 1e12


def _sample_text(w, samples, seconds):
    return (f"{samples} sample(s) of {ORACLE_HEADS * ORACLE_ROWS} query rows ({ORACLE_HEADS} heads x "
            f"{ORACLE_ROWS}) of the {w.name} workload, fp64 NumPy oracle, {seconds:.1f} s in all; "
            f"TFLOP/s = 4*N*d per row / time")


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import torch
    if torch.cuda.is_available():    # the seeded draw is faster on a device; values go to the host
        q, k, v = (t.cpu() for t in synth.make_qkv(w, device="cuda"))
    else:
        q, k, v = synth.make_qkv(w, device="cpu")
    for i in range(args.warmup):
        _cpu_oracle_sample(w, q, k, v, seed=1000 + i)
    total_s, total_rows = 0.0, 0
    for s in range(args.steps):
        dt, rows = _cpu_oracle_sample(w, q, k, v, seed=s)
        total_s += dt
        total_rows += rows
    tflops = _oracle_tflops(w, total_s, total_rows)
    per_step_ms = total_s / args.steps * 1e3
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": metric_for(w), "value": tflops, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step_ms,
        "ms_per_step_extrapolated": w.flops / (tflops * 1e12) * 1e3,
        "step": f"one sample of {ORACLE_HEADS * ORACLE_ROWS} query rows (measured); "
                "ms_per_step_extrapolated = the time of a full call at the same rate",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), bf16-rounded)",
        "config": _config(w),
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": _sample_text(w, args.steps, total_s)},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline(w, q, k, v, min_seconds=8.0, max_samples=16):
    """The same oracle samples as the reference arm, timed until min_seconds have passed."""
    total_s, total_rows, n = 0.0, 0, 0
    while n < max_samples and (total_s < min_seconds or n == 0):
        dt, rows = _cpu_oracle_sample(w, q, k, v, seed=n)
        total_s += dt
        total_rows += rows
        n += 1
    return {"value": _oracle_tflops(w, total_s, total_rows), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "sample": _sample_text(w, n, total_s)}


def _config(w, k_rope="prepass", kernel="default"):
    return {"workload": w.name, "k_rope": k_rope, "qk_operands": w.qk, "kernel": kernel, "B": w.B,
            "heads": w.H, "head_dim": w.d,
            "grid": f"{w.T}x{w.Hg}x{w.Wg}", "N": w.N,
            "sections": "/".join(map(str, w.sections)), "theta": w.theta,
            "l2": _l2_note(w),
            "parallelism": "replicas (one independent call per GPU)"}


def _e2e_leg(w, q, k, v, out, lse, hq, hk, hv, call, stream, dev, barrier, max_over_ranks, work,
             ws, steps):
    """End to end through the public API: every step copies its inputs from pinned host memory
    and its out + lse back, inside the timed region.  Pipelined as a serving loop would run:
    two device buffer sets; step i+1's upload (H2D stream) and step i-1's download (D2H
    stream) overlap step i's kernels."""
    import torch
    import video_diffusion_transformer_rope_gb300 as vdx
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hout = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    hlse = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True) for _ in range(2)]
    dq, dk, dv = [q, torch.empty_like(q)], [k, torch.empty_like(k)], [v, torch.empty_like(v)]
    dout, dlse = [out, torch.empty_like(out)], [lse, torch.empty_like(lse)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(1, steps)
    # per-step timestamps on each stream (read after the timed region) to show how far the
    # copies overlapped the kernels
    mark = {k: [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
            for k in ("up0", "up1", "run0", "run1", "down0", "down1")}

    def upload(i):
        sl = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(computed[sl])          # the kernel that read this slot is done
            mark["up0"][i].record(s_in)
            dq[sl].copy_(hq, non_blocking=True)
            dk[sl].copy_(hk, non_blocking=True)
            dv[sl].copy_(hv, non_blocking=True)
            mark["up1"][i].record(s_in)
            in_ready[sl].record(s_in)

    barrier()
    start.record(stream)
    s_in.wait_stream(stream)
    s_out.wait_stream(stream)
    upload(0)
    for i in range(e2e_steps):
        sl = i % 2
        if i + 1 < e2e_steps:
            upload(i + 1)
        stream.wait_event(in_ready[sl])
        if i >= 2:
            stream.wait_event(drained[sl])             # this slot's previous result is home
        mark["run0"][i].record(stream)
        call(dq[sl], dk[sl], dv[sl], dout[sl], dlse[sl])
        mark["run1"][i].record(stream)
        computed[sl].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[sl])
            mark["down0"][i].record(s_out)
            hout[sl].copy_(dout[sl], non_blocking=True)
            hlse[sl].copy_(dlse[sl], non_blocking=True)
            mark["down1"][i].record(s_out)
            drained[sl].record(s_out)
    stream.wait_stream(s_in)
    stream.wait_stream(s_out)
    end.record(stream)
    barrier()
    vdx.sync_check(stream)
    e2e_ms = max_over_ranks(start.elapsed_time(end) / e2e_steps)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = hout[0].numel() * hout[0].element_size() + hlse[0].numel() * hlse[0].element_size()

    mean = lambda a, b: statistics.mean(mark[a][i].elapsed_time(mark[b][i]) for i in range(e2e_steps))
    streams = {"upload_ms": mean("up0", "up1"), "kernels_ms": mean("run0", "run1"),
               "download_ms": mean("down0", "down1")}
    streams["upload_gbs"] = h2d / streams["upload_ms"] / 1e6
    streams["download_gbs"] = d2h / streams["download_ms"] / 1e6
    return {"value": job_tflops(work, e2e_ms, ws), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
            "per_stream_mean": streams,
            "copies": "pinned host memory, H2D and D2H streams overlapping compute "
                      "(double-buffered device inputs and outputs)"}


def _kernel_used(args, w):
    """Which attention kernel runs the timed calls (the library's default rule for dense calls:
    CTA pairs with the fused K rotation, with split operands, or with fp16 operands and
    N >= 65536)."""
    if args.kernel != "default":
        return args.kernel
    dense = not args.window and not args.subset
    return "pair" if dense and (args.k_rope == "fused" or w.qk == "split" or w.N >= 65536) else "single"


def run_ours(args, w):
    import torch
    import video_diffusion_transformer_rope_gb300 as vdx
    from video_diffusion_transformer_rope_gb300 import _build

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    if rank == 0:
        _build.build()
    if ws > 1:
        torch.distributed.barrier()
    vdx.lib()
    dev = torch.device("cuda", torch.cuda.current_device())

    q, k, v = synth.make_qkv(w, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    grid = (w.T, w.Hg, w.Wg)
    stream = torch.cuda.current_stream()

    k_mode = {"prepass": vdx.K_ROPE_PREPASS, "fused": vdx.K_ROPE_FUSED}[args.k_rope]
    qk = vdx.QK_MODES[w.qk]
    k_ws = torch.empty(vdx.workspace_bytes(w.B, w.H, grid, w.d, qk) // 2, dtype=torch.float16,
                       device=dev) if args.k_rope == "prepass" else None

    work = w.flops                       # FLOP per call (dense: 4*B*H*N^2*d)
    if args.window:
        # windowed (block-sparse) attention: count only the query-key pairs the mask keeps
        import numpy as np
        win = tuple(int(x) for x in args.window.split(","))
        words = vdx.window_block_mask(grid, win)
        nk = (w.N + vdx.SPARSE_KBLOCK - 1) // vdx.SPARSE_KBLOCK
        bits = ((words[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(words.shape[0], -1)[:, :nk]
        qrows = np.minimum(vdx.SPARSE_QBLOCK, w.N - np.arange(words.shape[0]) * vdx.SPARSE_QBLOCK)
        kcols = np.minimum(vdx.SPARSE_KBLOCK, w.N - np.arange(nk) * vdx.SPARSE_KBLOCK)
        pairs = float((qrows[:, None] * bits * kcols[None, :]).sum())
        work = 4.0 * w.B * w.H * pairs * w.d
        mask_dev = torch.from_numpy(words.astype(np.int32)).to(dev)

        def call(qq, kk, vv, oo, ll):
            vdx.rope3d_attn_sparse(qq, kk, vv, grid, mask_dev, w.sections, w.theta, out=oo, lse=ll,
                                   stream=stream, workspace=k_ws, qk_precision=qk)
    elif args.subset:
        # active-query subset: a seeded fraction of the tokens attends to every key
        frac = float(args.subset)
        nq = max(1, int(round(frac * w.N)))
        gsub = torch.Generator(device="cpu").manual_seed(w.seed + 3000)
        idx = torch.randperm(w.N, generator=gsub)[:nq].sort().values.to(torch.int32).to(dev)
        work = 4.0 * w.B * w.H * float(nq) * w.N * w.d

        def call(qq, kk, vv, oo, ll):
            vdx.rope3d_attn_subset(qq, kk, vv, grid, idx, oo, ll, w.sections, w.theta,
                                   stream=stream, workspace=k_ws, qk_precision=qk)
    else:
        kern = {"default": vdx.KERNEL_DEFAULT, "single": vdx.KERNEL_SINGLE, "pair": vdx.KERNEL_PAIR}[args.kernel]

        def call(qq, kk, vv, oo, ll):
            vdx.rope3d_attn(qq, kk, vv, grid, w.sections, w.theta, out=oo, lse=ll, stream=stream,
                            k_rope=k_mode, workspace=k_ws, qk_precision=qk, kernel=kern)

    def step():
        call(q, k, v, out, lse)

    for _ in range(args.warmup):
        step()
    vdx.sync_check(stream)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x):
        return reduce_max_over_ranks(x, ws, dev)

    # ---- device-resident timed region
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        smi_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        smi_id = str(dev.index)
    with ClockSampler(smi_id) as clk:
        barrier()
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        barrier()
    vdx.sync_check(stream)
    ms = max_over_ranks(start.elapsed_time(end) / args.steps)
    clocks = clk.summary()

    # ---- end to end through the public API: every step copies its inputs from pinned host
    # memory and its out + lse back, inside the timed region.  Pipelined as a serving loop
    # would run: two device buffer sets; step i+1's upload (H2D stream) and step i-1's
    # download (D2H stream) overlap step i's kernels.
    e2e = None
    hq = hk = hv = None
    if not args.no_e2e:
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        e2e = _e2e_leg(w, q, k, v, out, lse, hq, hk, hv, call, stream, dev, barrier, max_over_ranks,
                       work, ws, args.steps)
    elif rank == 0 and ws == 1 and not args.no_cpu_baseline:
        hq, hk, hv = (t.cpu() for t in (q, k, v))

    tflops_rank = job_tflops(work, ms, 1)
    value = job_tflops(work, ms, ws)
    peak, peak_sus, peak_src = _peaks()
    traffic = _traffic_per_launch(w.name, _kernel_used(args, w), args.k_rope)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not args.window and not args.subset:
        cpu = cpu_baseline(w, hq, hk, hv)

    if rank == 0:
        line = {
            "metric": METRIC_WINDOW if args.window else (METRIC_SUBSET if args.subset else metric_for(w)),
            "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) on device, bf16)",
            "config": dict(_config(w, args.k_rope, _kernel_used(args, w)), **({"window": args.window,
                                                         "mask_density": work / w.flops}
                                                        if args.window else {}),
                           **({"active_query_fraction": float(args.subset)} if args.subset else {})),
            "e2e": e2e,
            "gpu_launches": args.steps * (2 if args.k_rope == "prepass" else 1),
            "roofline": {"bound": "tensor", "achieved": tflops_rank, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops_rank / peak, "traffic": traffic,
                         "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)",
                         "frac_of_sustained": (tflops_rank / peak_sus) if peak_sus else None,
                         "kernel": (f"attn_fwd_sm103, {_kernel_used(args, w)} (+ rope3d_qk_prepass)"
                                    if args.k_rope == "prepass" else f"attn_fwd_sm103, {_kernel_used(args, w)}, fused K rotation")},
            "cpu_baseline": cpu,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=configs.WAN14B_720P.name, choices=sorted(configs.BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--window", default=None,
                    help="wt,wh,ww: windowed 3D attention through the block-sparse path; value "
                         "counts only the query-key pairs the window's block mask keeps")
    ap.add_argument("--subset", default=None,
                    help="fraction: active-query subset (that share of tokens, seeded) attends to "
                         "every key; value counts 4*d per active query-key pair")
    ap.add_argument("--k-rope", choices=["prepass", "fused"], default="prepass",
                    help="K rotated once by a prepass kernel (default) or per tile inside the "
                         "attention kernel")
    ap.add_argument("--kernel", choices=["default", "single", "pair"], default="default",
                    help="attention kernel for dense calls: the library's choice, one CTA per 256 "
                         "query rows, or CTA pairs sharing each K/V tile")
    ap.add_argument("--qk", choices=["fp16", "split"], default=None,
                    help="QK operand precision (default: the workload's own: split for the "
                         "long-clip stress workload, fp16 for the others)")
    ap.add_argument("--batch", type=int, default=None,
                    help="profiling runs only: override the workload's batch size B")
    ap.add_argument("--heads", type=int, default=None,
                    help="profiling runs only: override the workload's head count H")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end leg (profiling runs: halves the device memory)")
    args = ap.parse_args()
    ws_env = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != ws_env:
        ap.error(f"--gpus {args.gpus} but {ws_env} process(es) were launched: run N > 1 under "
                 "torchrun (one process per GPU)")
    w = configs.BY_NAME[args.workload]
    if args.qk:
        import dataclasses
        w = dataclasses.replace(w, qk=args.qk)
    if args.batch or args.heads:
        import dataclasses
        B, H = args.batch or w.B, args.heads or w.H
        w = dataclasses.replace(w, B=B, H=H, name=f"{w.name}_B{B}_H{H}")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
