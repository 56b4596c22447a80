"""Benchmark: one decode step of paged-KV attention on GB300.

A step is the whole hot path for one batch: write the step's new K/V token
per sequence into the paged cache, then paged decode attention with its
split-K combine, through pkv_decode_step + pkv_decode_combine: for fp16/bf16
caches the write is folded into the split kernel (2 launches), for INT8
caches one append kernel writes the rows (3 launches). --unfused runs
pkv_append + pkv_decode_split + pkv_decode_combine (3 launches; INT8: 4).
Default workload: the GQA Llama-3-8B-shape batch (B=256, 32 q / 8 kv heads,
D=128, bf16, L~U[128,4096]).

    python bench.py [--gpus N --steps K --warmup W] [--config NAME] [--impl reference]

Prints one JSON line. `value` is the decode-attention HBM throughput of the
whole step: algorithmic bytes (KV + q + block tables, per the workload) over
the step time, summed over ranks. The KV cache (2.3 GB) is far larger than L2,
so no flush is needed between steps. `--impl reference` times the CPU oracle
(float64 NumPy) on the host cores over a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_decode_05_gb300.workloads import (CONFIGS, DESCRIPTIONS,  # noqa: E402
                                                algorithmic_bytes, make_workload)

METRIC = "paged decode-attn achieved HBM GB/s (% of GB300 peak) and decode tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")
# Kernel-timing pass: CUDA events around every kernel of each step. Events
# between two launches stop the second from overlapping the first (programmatic
# dependent launch), so this pass is separate from the timed region; its first
# KERNEL_PASS_SKIP steps are dropped and the median is reported.
KERNEL_PASS_MIN_STEPS = 200
KERNEL_PASS_MIN_MS = 1000.0
KERNEL_PASS_MAX_STEPS = 20000
KERNEL_PASS_SKIP = 5
# Parity bound of the bench's parity leg: bf16 / fp16 KV elementwise
# |g - o| <= 2e-3 + 1e-2 |o|; INT8 KV |g - o| <= 2e-2 against the oracle on
# the dequantised cache.
TOL_ABS, TOL_REL, TOL_I8 = 2e-3, 1e-2, 2e-2


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--config", default="gqa8b", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--op", default="decode_step",
                    choices=["decode_step", "copy_blocks", "multiquery"],
                    help="decode_step: the hot path (default); copy_blocks: copy-on-write "
                         "block copy of --copy-pairs random blocks of the workload's pool; "
                         "multiquery: append of the q_len new tokens + causal multi-query "
                         "attention (use --config spec_verify or prefill_chunk)")
    ap.add_argument("--copy-pairs", type=int, default=4096)
    ap.add_argument("--unfused", action="store_true",
                    help="step = pkv_append + split + combine (3 launches; INT8: 4) instead of "
                         "pkv_decode_step (16-bit: split with the append folded in; INT8: the "
                         "step's append kernel + split) + combine")
    ap.add_argument("--graph", action="store_true",
                    help="replay the step from a captured CUDA graph instead of eager launches")
    ap.add_argument("--num-parts", type=int, default=0, help="worker warps (0 = device default)")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-steps", type=int, default=0,
                    help="steps of the kernel-timing pass that follows the timed region "
                         "(0: at least %d steps and about %.0f s of work)"
                         % (KERNEL_PASS_MIN_STEPS, KERNEL_PASS_MIN_MS / 1e3))
    return ap.parse_args(argv)


def load_peaks():
    """HBM roofline denominator: the measured copy bandwidth if present."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_tensor_peak():
    """Dense bf16 tensor roofline denominator (TFLOP/s, burst) if measured."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


_CODE_TOKENS = re.compile(rb'("(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\')|/\*.*?\*/|//[^\n]*',
                          re.S)


def code_only(text: bytes) -> bytes:
    """C++ source without its comments, whitespace runs collapsed to one
    space: what the compiler sees, up to formatting."""
    text = _CODE_TOKENS.sub(lambda m: m.group(1) if m.group(1) else b" ", text)
    return re.sub(rb"\s+", b" ", text).strip()


def mq_kernel_for(kv_dtype: str, head_dim: int, rows: int):
    """The multi-query kernel pkv_multiquery_attn runs for ``rows`` = q_len x
    group size (q and out 16-byte aligned), and the sources its device code
    comes from: the library's dispatch rule, checked against the library's
    own planner by tests/test_bench_host.py."""
    i8 = kv_dtype == "i8"
    if not i8 and rows >= 128:
        return "mq_tc_kernel", ("mq_split.cuh", "mq.cu")
    if rows <= 24 and (not i8 or head_dim == 128):
        return ("mqt_i8_split_kernel" if i8 else "mqt_split_kernel"), ("mq_split.cuh", "mq_t.cu")
    return "mq_split_kernel", ("mq_split.cuh",)


def kernel_source_hash(source="decode.cu") -> str:
    """sha256 (first 16 hex digits) of the device code a kernel is built from:
    each file of ``source`` (a name or a tuple of names) up to its host-code
    marker line (``// ---- ... host ---``), followed by common.cuh, comments
    and formatting left out (:func:`code_only`). Host-side edits below the
    marker, and comment-only edits, leave it alone."""
    import hashlib
    csrc = os.path.join(ROOT, "paged_kv_decode_05_gb300", "csrc")
    text = b""
    for name in ((source,) if isinstance(source, str) else tuple(source)):
        with open(os.path.join(csrc, name), "rb") as f:
            part = f.read()
        m = re.search(rb"^// -+ host -+$", part, re.M)
        text += code_only(part[:m.start()] if m else part) + b"\n"
    with open(os.path.join(csrc, "common.cuh"), "rb") as f:
        text += code_only(f.read())
    return hashlib.sha256(text).hexdigest()[:16]


def recorded_traffic(kernel: str, config: str, source: str = "decode.cu"):
    """DRAM bytes per launch from the committed ncu summary, if still current.

    profiles/<kernel>_<config>.md carries a line
    ``traffic_bytes_per_launch: N source_sha256: H``; it counts only while H
    matches :func:`kernel_source_hash` of ``source``.
    """
    path = os.path.join(ROOT, "profiles", f"{kernel}_{config}.md")
    try:
        h = kernel_source_hash(source)
        for line in open(path):
            if line.startswith("traffic_bytes_per_launch:"):
                parts = line.split()
                if parts[3] == h:
                    return int(parts[1])
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float, timed=None):
        """Median SM clock and the throttle reasons seen in the window [t0, t1]
        (host wall time). ``timed``: the timed region's (start, end) inside
        that window; its sample count is reported beside the window's (a short
        timed region can fall between two 100 ms samples, so the window also
        covers the warm-up and the kernel-timing pass around it)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons, n, n_timed = [], None, set(), 0, 0
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < len(self.FIELDS):
                continue
            try:
                sm.append(float(f[0]))
                smax = float(f[1])
            except ValueError:
                continue
            n += 1
            if timed is not None and timed[0] <= ts <= timed[1]:
                n_timed += 1
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), f[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
               "reasons": sorted(reasons), "samples": n}
        if timed is not None:
            out["samples_in_timed_region"] = n_timed
            out["window_s"] = round(t1 - t0, 3)
            out["window"] = "warm-up, timed steps and kernel-timing pass"
        return out


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def oracle_sample(w, budget_s: float, first: int = 0):
    """Time the CPU oracle on whole sequences until ~budget_s (at least one).

    Returns (seconds, algorithmic bytes covered, sequences, threads).
    """
    import oracle
    cfg = w.cfg
    shape = (w.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    if cfg.kv_dtype == "i8":
        k = np.zeros(shape, np.int8); v = np.zeros(shape, np.int8)
        ks = np.zeros(shape[:2], np.float32); vs = np.zeros(shape[:2], np.float32)
        oracle.append_int8(k, v, ks, vs, w.k_fill, w.v_fill, w.fill_slots)
        oracle.append_int8(k, v, ks, vs, w.k_step, w.v_step, w.step_slots)
    else:
        dt = np.uint16 if cfg.kv_dtype == "bf16" else np.float16
        k = np.zeros(shape, dt); v = np.zeros(shape, dt); ks = vs = None
        oracle.append_copy(k, v, w.k_fill, w.v_fill, w.fill_slots)
        oracle.append_copy(k, v, w.k_step, w.v_step, w.step_slots)
    seqs, outs, t_total = [], {}, 0.0
    b = first
    while len(seqs) < cfg.batch and (t_total < budget_s or not seqs):
        t0 = time.perf_counter()
        o = oracle.paged_decode_attention(w.q, k, v, w.block_tables, w.context_lens,
                                          cfg.softmax_scale, ks, vs, seqs=[b])
        t_total += time.perf_counter() - t0
        outs[b] = o[0]
        seqs.append(b)
        b = (b + 1) % cfg.batch
    lens = w.context_lens[seqs]
    from paged_kv_decode_05_gb300.workloads import variant
    byts = algorithmic_bytes(variant(cfg, batch=len(seqs)), lens)
    return t_total, byts, seqs, _threads(), outs


def parity_report(got: dict, want: dict, int8: bool) -> dict:
    """Element-wise comparison of the GPU output rows with the oracle's on the
    sampled sequences: max |g - o|, max |g - o| / |o| over |o| >= 0.2, and
    whether every element meets the workload's bound."""
    g = np.concatenate([np.asarray(got[b], np.float64).ravel() for b in sorted(want)])
    o = np.concatenate([np.asarray(want[b], np.float64).ravel() for b in sorted(want)])
    err = np.abs(g - o)
    big = np.abs(o) >= 0.2
    ok = bool(np.all(err <= TOL_I8)) if int8 else bool(np.all(err <= TOL_ABS + TOL_REL * np.abs(o)))
    return {"sequences": len(want), "elements": int(g.size),
            "max_abs": float(err.max()) if g.size else 0.0,
            "max_rel_where_abs_o_ge_0.2": float((err[big] / np.abs(o[big])).max()) if big.any()
            else 0.0,
            "bound": "|g-o| <= 2e-2" if int8 else "|g-o| <= 2e-3 + 1e-2|o|", "pass": ok,
            "against": "float64 oracle" + (" on the dequantised cache" if int8 else "")}


def _threads() -> int:
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 1) for d in threadpool_info()]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def _gpu_state(w, device):
    """Device tensors for one workload: cache filled by pkv_append, step inputs."""
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    cfg = w.cfg

    def dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    shape = (w.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    st = {"status": torch.zeros(1, dtype=torch.int32, device=device)}
    if cfg.kv_dtype == "i8":
        st["k_cache"] = torch.zeros(shape, dtype=torch.int8, device=device)
        st["v_cache"] = torch.zeros(shape, dtype=torch.int8, device=device)
        st["k_scales"] = torch.zeros(shape[:2], dtype=torch.float32, device=device)
        st["v_scales"] = torch.zeros(shape[:2], dtype=torch.float32, device=device)
        n = B.pkv_append_workspace_size(st["k_cache"])
        st["append_ws"] = torch.zeros(n, dtype=torch.uint8, device=device)   # zeroed once
    else:
        dt = torch.bfloat16 if cfg.kv_dtype == "bf16" else torch.float16
        st["k_cache"] = torch.zeros(shape, dtype=dt, device=device)
        st["v_cache"] = torch.zeros(shape, dtype=dt, device=device)
        st["k_scales"] = st["v_scales"] = st["append_ws"] = None
    B.pkv_append(dev(w.k_fill), dev(w.v_fill), dev(w.fill_slots), st["k_cache"], st["v_cache"],
                 st["k_scales"], st["v_scales"], st["append_ws"], st["status"])
    st["q"] = dev(w.q)
    st["k_step"], st["v_step"] = dev(w.k_step), dev(w.v_step)
    st["step_slots"] = dev(w.step_slots)
    st["block_tables"], st["context_lens"] = dev(w.block_tables), dev(w.context_lens)
    st["out"] = torch.empty_like(st["q"])
    torch.cuda.synchronize(device)
    return st


def out_to_f64(t) -> np.ndarray:
    """A CUDA output tensor (fp16 / bf16) as float64 on the host, exactly."""
    return t.float().cpu().numpy().astype(np.float64)


def kernel_pass(step, n: int, device, names=("append", "split", "combine")) -> dict:
    """Run ``n`` steps, each ``step(ev)`` recording len(names) + 1 CUDA events
    on the launching stream around its kernels, and return the median, mean,
    min and max of each kernel's time in ms over the steps after the first
    KERNEL_PASS_SKIP."""
    import torch
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1))
           for _ in range(n)]
    torch.cuda.synchronize(device)
    for e in evs:
        step(e)
    torch.cuda.synchronize(device)
    skip = min(KERNEL_PASS_SKIP, max(0, n - 1))
    res = {"steps": n - skip, "skipped": skip}
    for i, name in enumerate(names):
        t = [e[i].elapsed_time(e[i + 1]) for e in evs[skip:]]
        res[name] = {"median": statistics.median(t), "mean": sum(t) / len(t),
                     "min": min(t), "max": max(t)}
    return res


def _step(st, cfg, ws, parts, ev=None, fused=None):
    """One decode step: the new token's cache write, split, combine.

    Unfused: pkv_append, pkv_decode_split, pkv_decode_combine (3 launches; 4
    for INT8). Fused: pkv_decode_step's split phase (16-bit caches: the split
    kernel writes the new rows itself; INT8: the step's append kernel, then
    the split), then pkv_decode_combine (2 launches; 3 for INT8).
    ``ev``: optional 4 CUDA events recorded before the append, before the
    split, before the combine and after it (the first two coincide if fused).
    """
    from paged_kv_decode_05_gb300 import binding as B
    if fused is None:
        fused = st.get("fused", False)
    if ev is not None:
        ev[0].record()
    if not fused:
        B.pkv_append(st["k_step"], st["v_step"], st["step_slots"], st["k_cache"],
                     st["v_cache"], st["k_scales"], st["v_scales"], st["append_ws"],
                     st["status"])
    if ev is not None:
        ev[1].record()
    if fused:
        B.pkv_decode_step(st["q"], st["k_step"], st["v_step"], st["k_cache"], st["v_cache"],
                          st["block_tables"], st["context_lens"], cfg.softmax_scale, st["out"],
                          ws, parts, st["status"], run_combine=False, k_scales=st["k_scales"],
                          v_scales=st["v_scales"])
    else:
        B.pkv_decode_split(st["q"], st["k_cache"], st["v_cache"], st["block_tables"],
                           st["context_lens"], cfg.softmax_scale, st["out"], ws,
                           st["k_scales"], st["v_scales"], parts, st["status"])
    if ev is not None:
        ev[2].record()
    B.pkv_decode_combine(st["out"], st["k_cache"], ws, parts)
    if ev is not None:
        ev[3].record()


def run_native(args):
    import torch
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from paged_kv_decode_05_gb300 import binding as B
    from paged_kv_decode_05_gb300.build import build
    if rank == 0:
        build()
    barrier(world, device)
    B.lib()

    cfg = CONFIGS[args.config]
    w = make_workload(cfg, seed=cfg.seed + rank)   # one replica per rank (weak scaling)
    st = _gpu_state(w, device)
    parts = args.num_parts or B.pkv_decode_default_parts(cfg.batch, cfg.num_q_heads,
                                                         st["k_cache"], device.index)
    ws = torch.empty(B.pkv_decode_workspace_size(cfg.batch, cfg.num_q_heads, st["k_cache"], parts),
                     dtype=torch.uint8, device=device)
    alg = algorithmic_bytes(cfg, w.context_lens)
    st["fused"] = not args.unfused
    launches_per_step = (2 if st["fused"] else 3) + (1 if cfg.kv_dtype == "i8" else 0)
    K, W = args.steps, args.warmup

    props = torch.cuda.get_device_properties(device)
    sampler = ClockSampler(str(getattr(props, "uuid", local)).strip())
    if str(sampler.gpu_id) and not str(sampler.gpu_id).startswith("GPU-"):
        sampler.gpu_id = "GPU-" + sampler.gpu_id
    sampler.start()
    time.sleep(0.3)                 # nvidia-smi is up before the GPU work starts
    wall_w = time.time()
    for _ in range(W):
        _step(st, cfg, ws, parts)
    torch.cuda.synchronize(device)
    graph = None
    if args.graph:  # one captured step, replayed in the timed loop
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            _step(st, cfg, ws, parts)
        for _ in range(W):
            graph.replay()
        torch.cuda.synchronize(device)

    # ---- device-timed region: K steps, inputs resident in HBM, no events
    # between the launches
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    wall0 = time.time()
    t_start.record()
    for _ in range(K):
        if graph is not None:
            graph.replay()
        else:
            _step(st, cfg, ws, parts)
    t_end.record()
    torch.cuda.synchronize(device)
    wall1 = time.time()
    barrier(world, device)
    ms_total = reduce_max(t_start.elapsed_time(t_end), world, device)
    out_timed = st["out"].clone()
    status = int(st["status"].item())

    # ---- kernel-timing pass: events around every kernel of each step
    n_kp = args.kernel_steps or int(min(KERNEL_PASS_MAX_STEPS,
                                        max(KERNEL_PASS_MIN_STEPS,
                                            KERNEL_PASS_MIN_MS * K / max(ms_total, 1e-6))))
    # INT8: pkv_decode_step runs its append kernel and the split in one call,
    # so this pass times the steps through pkv_append + split + combine (the
    # same split and combine kernels; pkv_append writes the same codes and
    # scales as the step's append kernel, so the cache state is unchanged)
    kp_fused = st["fused"] and cfg.kv_dtype != "i8"
    kp = kernel_pass(lambda ev: _step(st, cfg, ws, parts, ev, fused=kp_fused), n_kp, device)
    if st["fused"] and not kp_fused:
        kp["append_timed_as"] = "pkv_append (two kernels) in place of the step's append kernel"
    wall2 = time.time()

    # ---- end-to-end through the C ABI with host buffers (H2D inputs, D2H output)
    e2e = _e2e(st, w, cfg, ws, parts, device, min(K, args.e2e_steps), world)
    time.sleep(0.2)
    clocks = sampler.stop(wall_w, wall2, timed=(wall0, wall1))

    step_s = ms_total / 1e3 / K
    value = alg * world / step_s / 1e9
    peak, peak_src = load_peaks()
    split_ms = kp["split"]["median"]
    achieved = alg / (split_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(ms_total / K, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": cfg.kv_dtype, "data": "synthetic (seeded N(0,1) K/V/q, shuffled block pool)",
        "config": {**workload_config(args.config, w, alg), "workers": parts,
                   "l2": "no flush: the KV cache read each step (%.2f GB) is far larger than "
                         "the 129 MB L2" % (alg / 1e9),
                   "parallelism": f"replicas x{world}",
                   "step": (("pkv_decode_step split phase (the step's INT8 append kernel, "
                             "then the split) + pkv_decode_combine" if cfg.kv_dtype == "i8" else
                             "pkv_decode_step split phase (new K/V rows written by the split "
                             "kernel) + pkv_decode_combine") if st["fused"] else
                            "pkv_append + pkv_decode_split + pkv_decode_combine")},
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * value / world / peak, 2),
        "decode_tokens_per_s": round(cfg.batch * world / step_s, 1),
        "kv_tokens_per_s": round(w.total_tokens * world / step_s, 1),
        "roofline": {"kernel": "decode_split_kernel", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic("decode_split_kernel", args.config),
                     "algorithmic_bytes_per_launch": alg,
                     "split_ms": round(split_ms, 6),
                     "split_share_of_step": round(split_ms / (ms_total / K), 4)},
        "kernel_ms": {**{k: {kk: round(vv, 6) for kk, vv in v.items()}
                         for k, v in kp.items() if isinstance(v, dict)},
                      "steps": kp["steps"], "skipped": kp["skipped"],
                      **({"append_timed_as": kp["append_timed_as"]}
                         if "append_timed_as" in kp else {}),
                      "how": "separate pass after the timed region: CUDA events around each "
                             "kernel of every step (the first steps dropped), median"},
        "launch_mode": "cuda_graph" if graph is not None else "eager",
        "e2e": e2e, "gpu_launches": K * launches_per_step, "clocks": clocks,
        "device_status": status,
    }
    if rank == 0 and not args.no_cpu_baseline:
        t, byts, seqs, thr, want = oracle_sample(w, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": round(byts / t / 1e9, 4), "unit": "GB/s", "cores": thr,
                                "kind": "oracle",
                                "sample": f"float64 oracle attention over {len(seqs)} of "
                                          f"{cfg.batch} sequences ({t:.1f} s), same workload"}
        got = out_to_f64(out_timed)
        line["parity"] = parity_report({b: got[b] for b in want}, want, cfg.kv_dtype == "i8")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _e2e(st, w, cfg, ws, parts, device, K, world):
    """Same metric through the C ABI, with every step's inputs copied from
    pinned host memory and its output copied back inside the timed region.

    Served the way a decode loop runs: the inputs and the output are double
    buffered on the device, the host-to-device copies of step n+1 run on one
    stream and the device-to-host copy of step n on another while step n+1
    computes; events keep a buffer from being refilled before the step that
    reads it has finished, or overwritten before its copy-out has."""
    import torch
    names = ["q", "k_step", "v_step", "step_slots", "block_tables", "context_lens"]
    host = {n: st[n].cpu().pin_memory() for n in names}
    out_host = torch.empty(st["out"].shape, dtype=st["out"].dtype).pin_memory()
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = out_host.numel() * out_host.element_size()
    sets = [dict(st), dict(st)]
    for n in names + ["out"]:
        sets[1][n] = torch.empty_like(st[n])
    comp = torch.cuda.current_stream(device)
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ready = [torch.cuda.Event() for _ in range(2)]    # inputs of the set copied in
    done = [torch.cuda.Event() for _ in range(2)]     # the step using the set finished
    drained = [torch.cuda.Event() for _ in range(2)]  # the set's output copied out

    def step(n):
        i = n % 2
        with torch.cuda.stream(up):
            if n >= 2:
                up.wait_event(done[i])
            for name in names:
                sets[i][name].copy_(host[name], non_blocking=True)
            ready[i].record(up)
        comp.wait_event(ready[i])
        if n >= 2:
            comp.wait_event(drained[i])
        _step(sets[i], cfg, ws, parts)
        done[i].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(done[i])
            out_host.copy_(sets[i]["out"], non_blocking=True)
            drained[i].record(down)

    for n in range(4):
        step(n)
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    for n in range(K):
        step(n)
    comp.wait_event(drained[(K - 1) % 2])
    b.record(comp)
    torch.cuda.synchronize(device)
    ms = reduce_max(a.elapsed_time(b), world, device)
    alg = algorithmic_bytes(cfg, w.context_lens)
    return {"value": round(alg * world / (ms / 1e3 / K) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": K,
            "ms_per_step": round(ms / K, 6),
            "how": "inputs and output double buffered; copies on two side streams overlap "
                   "the neighbouring steps' kernels"}


def workload_config(name, w, alg):
    """The keys that identify a decode workload, shared by both arms' lines
    (algorithmic bytes of one pass over the whole batch: the native arm's step)."""
    cfg = w.cfg
    return {"workload": DESCRIPTIONS[name], "name": name, "batch": cfg.batch,
            "num_q_heads": cfg.num_q_heads, "num_kv_heads": cfg.num_kv_heads,
            "head_dim": cfg.head_dim, "block_size": cfg.block_size,
            "total_context_tokens": w.total_tokens, "algorithmic_bytes_per_batch": alg}


def run_reference(args):
    """The CPU oracle as the reference arm: each step is the oracle's decode of
    one sequence of the workload (cycling through the batch), on host cores."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    cfg = CONFIGS[args.config]
    w = make_workload(cfg)
    # one oracle-built cache, then K timed steps of one sequence each
    import oracle
    shape = (w.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    if cfg.kv_dtype == "i8":
        k = np.zeros(shape, np.int8); v = np.zeros(shape, np.int8)
        ks = np.zeros(shape[:2], np.float32); vs = np.zeros(shape[:2], np.float32)
        oracle.append_int8(k, v, ks, vs, w.k_fill, w.v_fill, w.fill_slots)
        oracle.append_int8(k, v, ks, vs, w.k_step, w.v_step, w.step_slots)
    else:
        dt = np.uint16 if cfg.kv_dtype == "bf16" else np.float16
        k = np.zeros(shape, dt); v = np.zeros(shape, dt); ks = vs = None
        oracle.append_copy(k, v, w.k_fill, w.v_fill, w.fill_slots)
        oracle.append_copy(k, v, w.k_step, w.v_step, w.step_slots)
    from paged_kv_decode_05_gb300.workloads import variant

    def one(b):
        oracle.paged_decode_attention(w.q, k, v, w.block_tables, w.context_lens,
                                      cfg.softmax_scale, ks, vs, seqs=[b])

    for i in range(args.warmup):
        one(i % cfg.batch)
    seqs = [(args.warmup + i) % cfg.batch for i in range(args.steps)]
    t0 = time.perf_counter()
    for b in seqs:
        one(b)
    t = time.perf_counter() - t0
    byts = algorithmic_bytes(variant(cfg, batch=len(seqs)), w.context_lens[seqs])
    value = byts / t / 1e9
    cores = _threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**workload_config(args.config, w, algorithmic_bytes(cfg, w.context_lens)),
                   "step": "oracle decode of one sequence of the batch, cycling"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{len(seqs)} single-sequence float64 oracle decodes "
                                   f"({t:.1f} s)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_copy_blocks(args):
    """Copy-on-write block copy throughput on the workload's pool (1 GPU)."""
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    from paged_kv_decode_05_gb300.build import build
    build()
    device = torch.device("cuda", 0)
    cfg = CONFIGS[args.config]
    w = make_workload(cfg)
    st = _gpu_state(w, device)
    rng = np.random.default_rng(1)
    n = min(args.copy_pairs, w.num_blocks // 2)
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    src = torch.from_numpy(perm[:n].copy()).to(device)
    dst = torch.from_numpy(perm[n:2 * n].copy()).to(device)
    esz = 1 if cfg.kv_dtype == "i8" else 2
    block_bytes = cfg.num_kv_heads * cfg.block_size * cfg.head_dim * esz
    moved = 2 * n * 2 * block_bytes + (2 * 2 * n * cfg.num_kv_heads * 4 if esz == 1 else 0)
    for _ in range(args.warmup):
        B.pkv_copy_blocks(st["k_cache"], st["v_cache"], src, dst, st["k_scales"], st["v_scales"])
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        B.pkv_copy_blocks(st["k_cache"], st["v_cache"], src, dst, st["k_scales"], st["v_scales"])
    b.record()
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / args.steps
    peak, src_name = load_peaks()
    gbs = moved / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": "copy-on-write block copy HBM GB/s (read + write)", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 6), "higher_is_better": True, "dtype": cfg.kv_dtype,
        "data": "synthetic", "config": {"workload": DESCRIPTIONS[args.config], "pairs": n,
                                        "bytes_per_pair": 2 * block_bytes},
        "roofline": {"kernel": "copy_blocks_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                     "peak": peak, "peak_source": src_name, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "traffic": None},
        "gpu_launches": args.steps}), flush=True)


def run_multiquery(args):
    """Speculative verification / prefill chunk step on 1 GPU."""
    import torch
    from paged_kv_decode_05_gb300 import binding as B
    from paged_kv_decode_05_gb300.build import build
    build()
    device = torch.device("cuda", 0)
    cfg = CONFIGS[args.config]
    w = make_workload(cfg)
    st = _gpu_state(w, device)
    cu = torch.from_numpy(w.cu_q).to(device)
    nq = cfg.q_len
    ws = torch.empty(B.pkv_multiquery_workspace_size(cfg.batch, cfg.num_q_heads, nq,
                                                     st["k_cache"], args.num_parts),
                     dtype=torch.uint8, device=device)
    out = torch.empty_like(st["q"])

    def step(ev=None):
        if ev is not None:
            ev[0].record()
        B.pkv_append(st["k_step"], st["v_step"], st["step_slots"], st["k_cache"], st["v_cache"],
                     st["k_scales"], st["v_scales"], st["append_ws"], st["status"])
        if ev is not None:
            ev[1].record()
        B.pkv_multiquery_attn(st["q"], cu, nq, st["k_cache"], st["v_cache"], st["block_tables"],
                              st["context_lens"], cfg.softmax_scale, out, ws, args.num_parts,
                              st["status"], k_scales=st["k_scales"], v_scales=st["v_scales"])
        if ev is not None:
            ev[2].record()

    props = torch.cuda.get_device_properties(device)
    sampler = ClockSampler(str(getattr(props, "uuid", 0)).strip())
    if str(sampler.gpu_id) and not str(sampler.gpu_id).startswith("GPU-"):
        sampler.gpu_id = "GPU-" + sampler.gpu_id
    sampler.start()
    time.sleep(0.3)
    wall_w = time.time()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize(device)
    wall1 = time.time()
    ms = a.elapsed_time(b) / args.steps
    n_kp = args.kernel_steps or int(min(KERNEL_PASS_MAX_STEPS, max(
        KERNEL_PASS_MIN_STEPS, KERNEL_PASS_MIN_MS / max(ms, 1e-6))))
    kp = kernel_pass(step, n_kp, device, names=("append", "attn"))
    wall2 = time.time()
    time.sleep(0.2)
    clocks = sampler.stop(wall_w, wall2, timed=(wall0, wall1))
    attn_ms = kp["attn"]["median"]
    alg = algorithmic_bytes(cfg, w.context_lens)
    lens = w.context_lens.astype(np.int64)
    # causal FLOPs: query i of a sequence attends to L - nq + i + 1 tokens, 4 D flops each head
    flops = int(sum(4 * cfg.head_dim * cfg.num_q_heads * (nq * (L - nq) + nq * (nq + 1) // 2)
                    for L in lens))
    peak, src_name = load_peaks()
    tpeak, tsrc = load_tensor_peak()
    gbs = alg / (attn_ms / 1e3) / 1e9
    tflops = flops / (attn_ms / 1e3) / 1e12
    # The library's dispatch rule: runs over fp16 / bf16 caches that fill
    # 128-row tiles (q_len x the group size) take the tcgen05 kernel, one
    # launch; runs of at most 24 rows take a short-run split kernel (fp16 /
    # bf16 caches, and INT8 caches at head_dim 128) and the combine, other
    # runs the 16-rows-per-warp split kernel and the combine, two launches
    # each. Plus the append (two kernels for INT8).
    g = cfg.num_q_heads // cfg.num_kv_heads
    kernel, src = mq_kernel_for(cfg.kv_dtype, cfg.head_dim, nq * g)
    tc = kernel == "mq_tc_kernel"
    launches = (1 if tc else 2) + (2 if cfg.kv_dtype == "i8" else 1)
    traffic = recorded_traffic(kernel, args.config, src)
    # Bound: the workload's FLOP/byte against the machine balance (measured
    # tensor peak / measured HBM bandwidth). Long prefill chunks are dense
    # contractions; verification of a few draft tokens streams the cache.
    if flops / alg > tpeak * 1e12 / (peak * 1e9):
        roof = {"kernel": kernel, "bound": "tensor", "achieved": round(tflops, 1),
                "peak": tpeak, "peak_source": tsrc, "unit": "TFLOP/s",
                "frac": round(tflops / tpeak, 4), "traffic": traffic,
                "note": ("tcgen05.mma (bf16 in, fp32 accumulate in TMEM)" if tc else
                         "mma.sync m16n8k16 (bf16 in, fp32 accumulate)") +
                        " against the dense bf16 GEMM peak"}
    else:
        roof = {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1),
                "peak": peak, "peak_source": src_name, "unit": "GB/s",
                "frac": round(gbs / peak, 4), "traffic": traffic}
    print(json.dumps({
        "metric": "multi-query paged attention HBM GB/s (causal, q_len new tokens/sequence)",
        "value": round(alg / (ms / 1e3) / 1e9, 1), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "dtype": cfg.kv_dtype, "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.config], "name": args.config, "q_len": nq,
                   "algorithmic_bytes_per_step": alg, "attention_flops": flops},
        "attn_ms_avg": round(attn_ms, 6), "attn_tflops": round(tflops, 1),
        "query_tokens_per_s": round(cfg.batch * nq / (ms / 1e3), 1),
        "roofline": roof,
        "clocks": clocks,
        "device_status": int(st["status"].item()),
        "gpu_launches": args.steps * launches}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "copy_blocks":
        run_copy_blocks(args)
    elif args.op == "multiquery":
        run_multiquery(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
