"""Benchmark of the paged MLA decode hot path on one or more GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

A step is one full decode call (split-K segments + merge, through the C ABI)
over one batch of the DeepSeek-V3-shaped bf16 workload: 64 requests, 128
heads, qlen 1, seq_lens uniform in [1024, 8192], block 64, values ~N(0, 1),
random page permutation, segments chosen by the planner. With the planner's
balanced schedule a call is three launches: the work list from the lengths,
the decode over it, and the merge of the rows the list split. Inputs are
seeded and synthetic. L2 is flushed (a 256 MiB write) before every timed
step, and only the step itself is inside its CUDA events. The roofline's
kernel time is the decode launch alone, timed the same way on the same work
list; its bound is HBM when the launch's algorithmic bytes at the measured
copy rate take longer than its flops at the dense tensor peak of its dtype
(e4m3: the measured bf16 peak times the nominal 2x), else the tensor pipe.

The default line also carries ``workloads``: the other workload shapes (the
tiny batch, the e4m3 batch at 16 and 128 heads, multi-token rows with
sinks, the sparse top-k decode), each timed in the same run the same way,
with its per-call and decode times, both roofline fractions and its bound.

Under torchrun (N > 1) every rank decodes its own batch of the same shape
(weak scaling, no collective on the data path); the per-step time is the max
over ranks and ``value`` counts the KV tokens of all ranks.

``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload) and prints the same JSON line with
``"impl": "reference"``.
"""
from __future__ import annotations

import argparse
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("MLA decode µs/call & KV tokens/s; HBM GB/s or MMA util as % of GB300 "
          "roofline")
UNIT = "KV tokens/s"
WORKLOADS = {
    "dsv3": "dsv3_bf16: DeepSeek-V3-shaped bf16 MLA decode, batch {b}, 128 heads, qlen 1, "
            "seq_lens uniform in [1024, 8192], block_size 64, q/cache ~N(0,1) bf16, "
            "scale 1/sqrt(192), random page permutation, segments chosen by the planner",
    "tiny": "tiny_dense: batch 2, 16 heads, qlen 1, seq_lens {{37,130}}, block_size 16, "
            "q/cache bf16 ~N(0,0.5^2), 4 segments, tile 16",
    "fp8": "fp8_decode: e4m3 q+KV with per-tensor scales, batch {b}, qlen 1, 16384 KV "
           "tokens/request, block_size 64, {h} heads",
    "mtp": "mtp_sinks: multi-token causal decode with sinks, batch {b}, 128 heads, qlen 2-4, "
           "seq_lens lognormal(median 4096, sigma 1) clipped to [128, 32768], bf16",
    "sparse": "sparse_topk: 128 tokens over 16 requests, 128 heads, bf16, 65536-token cache "
              "per request at block_size 64, top-2048 distinct indices with -1 padding",
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def _build_workload(name, seed_offset=0, batch=None, heads=128):
    from paged_mla_decode_06_gb300 import inputs as I
    if name == "dsv3":
        b = batch or 64
        return I.dsv3_bf16(seed=2 + seed_offset, batch=b), WORKLOADS[name].format(b=b)
    if name == "tiny":
        return I.tiny_dense(seed=1 + seed_offset), WORKLOADS[name].format()
    if name == "fp8":
        b = batch or 52
        return I.fp8_decode(heads, seed=3 + seed_offset, batch=b), \
            WORKLOADS[name].format(b=b, h=heads)
    if name == "mtp":
        b = batch or 32
        return I.mtp_sinks(seed=4 + seed_offset, batch=b), WORKLOADS[name].format(b=b)
    if name == "sparse":
        return I.sparse_topk(seed=5 + seed_offset), WORKLOADS[name].format()
    raise ValueError(name)


def _row_bytes(w):
    return 576 * (2 if w.kv_dtype == "bf16" else 1)


def _kv_keys(w):
    """KV tokens attended once per request (dense) or valid slots (sparse)."""
    import numpy as np
    if w.sparse:
        return int((w.topk_indices >= 0).sum())
    return int(w.seq_lens.astype(np.int64).sum())


def _flops(w):
    """2176 flop per (visible key, query row): 1152 for q.k over 576 columns,
    1024 for p.v over 512 (causally masked keys are not counted)."""
    import numpy as np
    H = w.num_heads
    if w.sparse:
        return float((w.topk_indices >= 0).sum()) * H * 2176.0
    if w.qo_indptr is None:
        return float(w.seq_lens.astype(np.int64).sum()) * H * 2176.0
    tot = 0
    for r in range(w.num_reqs):
        ql = int(w.qo_indptr[r + 1] - w.qo_indptr[r])
        L = int(w.seq_lens[r])
        tot += sum(max(0, L - ql + j + 1) for j in range(ql))
    return float(tot) * H * 2176.0


# DRAM bytes (read + write) per algorithmic byte of a decode kernel, from one
# ncu capture each (the profile summaries under profiles/ name the commands
# and the numbers), valid only for the kernel source each was taken on and
# the workload it was taken on: (kernel id, workload, heads) -> record.
PROFILED_TRAFFIC = {
    (4, "dsv3", None): {  # decode_tc.cu, DeepSeek-V3-shaped batch (profiles/decode_tc_dsv3.md)
        "source": "decode_tc.cu",
        "code_sha256": "8627e3e3dff2a7f099e4577878849af60304b92bd461a6cd133bfca0f5975a21",
        "dram_per_alg_byte": (139.609088 + 3.360256) / 138.103440,
    },
    (5, "fp8", 16): {  # decode_hn.cu, e4m3 batch at 16 heads (profiles/decode_hn_fp8.md)
        "source": "decode_hn.cu",
        "code_sha256": "b27dd235d6d48fcd1daf6457f627d20b78edd5858b4d37eb289261f2ff1ad65b",
        "dram_per_alg_byte": (226.828800 + 3.769344) / 226.738272,
    },
    (5, "fp8", 128): {  # decode_hn.cu on CTA-pair clusters, e4m3 batch at 128 heads (same file)
        "source": "decode_hn.cu",
        "code_sha256": "b27dd235d6d48fcd1daf6457f627d20b78edd5858b4d37eb289261f2ff1ad65b",
        "dram_per_alg_byte": (228.402432 + 4.709632) / 228.286560,
    },
}


def _code_digest(path):
    """sha256 of a source file's code: `//` comments and blank lines dropped,
    so that editing a comment does not disown a profile of the same code."""
    import hashlib
    import re
    lines = []
    with open(path) as f:
        for line in f:
            code = re.sub(r"//.*$", "", line.rstrip("\n")).rstrip()
            if code.strip():
                lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def _profiled_traffic(alg_bytes, kernel_id, workload_name, heads=None):
    """DRAM bytes of one launch scaled from the capture, or None once the
    kernel source differs from the one profiled, or for a kernel and
    workload no capture covers."""
    rec = PROFILED_TRAFFIC.get((kernel_id, workload_name, heads if workload_name == "fp8" else None))
    if rec is None:
        return None
    src = os.path.join(ROOT, "paged_mla_decode_06_gb300", "csrc", rec["source"])
    try:
        digest = _code_digest(src)
    except OSError:
        return None
    if digest != rec["code_sha256"]:
        return None
    return alg_bytes * rec["dram_per_alg_byte"]


def _alg_bytes_decode(w):
    """Algorithmic bytes of one decode launch: every KV row once per request
    (or valid sparse slot), q once, the block-table entries or slot list read.
    Segment partials are not algorithmic."""
    import numpy as np
    qb = w.num_tokens * w.num_heads * 576 * (2 if w.q_dtype == "bf16" else 1)
    if w.sparse:
        return _kv_keys(w) * _row_bytes(w) + qb + w.topk_indices.size * 4
    blocks = int(((w.seq_lens.astype(np.int64) + w.block_size - 1) // w.block_size).sum())
    return _kv_keys(w) * _row_bytes(w) + qb + blocks * 4 + w.num_reqs * 4


def smi_gpu_id(dev) -> str:
    """The GPU as nvidia-smi names it: its UUID (or PCI bus id), not the CUDA
    ordinal, which CUDA_VISIBLE_DEVICES renumbers."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    u = str(getattr(props, "uuid", "") or "")
    if len(u) == 36 and u.count("-") == 4:
        return "GPU-" + u
    try:
        return f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    except AttributeError:
        return str(dev.index or 0)


class ClockSampler:
    """nvidia-smi sampled every 100 ms while the timed region runs (read-only
    queries of the one GPU the benchmark runs on)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, log_path: str | None = None):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []
        self.log_path = log_path

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        if self.log_path:
            with open(self.log_path, "w") as f:
                f.write(self.FIELDS + "\n" + "\n".join(self.lines) + "\n")
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s >= 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on the host cores
# ---------------------------------------------------------------------------

def _oracle_worker(budget_s, n_steps, q):
    """Time the oracle on bounded samples of the workload: each step runs
    requests (continuing round-robin through the batch) until ``budget_s``
    seconds have passed, at least one request per step."""
    import numpy as np
    import oracle as O
    from paged_mla_decode_06_gb300 import inputs as I

    w = I.dsv3_bf16()
    blas = "unknown"
    try:
        cfg = np.show_config(mode="dicts")
        blas = cfg.get("Build Dependencies", {}).get("blas", {}).get("name", "unknown")
    except Exception:  # noqa: BLE001
        pass
    r = 0
    out = []
    for _ in range(n_steps):
        keys = 0
        done = 0
        t0 = time.perf_counter()
        while True:
            O.mla_decode(w.q[r:r + 1], "bf16", 1.0, w.cache, "bf16", 1.0,
                         w.block_table[r:r + 1], w.seq_lens[r:r + 1], w.softmax_scale,
                         block_size=w.block_size)
            keys += int(w.seq_lens[r])
            done += 1
            r = (r + 1) % w.num_reqs
            if time.perf_counter() - t0 >= budget_s:
                break
        out.append({"keys": keys, "requests": done, "seconds": time.perf_counter() - t0})
    q.put({"steps": out, "blas": blas, "total_requests": w.num_reqs})


def cpu_baseline_steps(budget_s=20.0, n_steps=1):
    """Run the oracle in a fresh (spawned) process whose BLAS uses every host
    core; returns one record per step."""
    cores = os.cpu_count() or 1
    env_keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = str(cores)
    try:
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        p = ctx.Process(target=_oracle_worker, args=(budget_s, n_steps, q))
        p.start()
        res = q.get(timeout=1800)
        p.join(timeout=60)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    recs = []
    for st in res["steps"]:
        recs.append({"value": st["keys"] / st["seconds"], "unit": UNIT, "cores": cores,
                     "kind": "oracle",
                     "sample": (f"fp64 numpy oracle, {st['requests']} request decodes taken "
                                f"round-robin from the {res['total_requests']}-request batch "
                                f"({st['keys']} KV tokens, {st['seconds']:.1f} s, "
                                f"BLAS {res['blas']} with {cores} threads)"),
                     "seconds": st["seconds"]})
    return recs


def _tiny_worker(q, reps):
    import oracle as O
    from paged_mla_decode_06_gb300 import inputs as I
    w = I.tiny_dense()
    t0 = time.perf_counter()
    for _ in range(reps):
        O.mla_decode(w.q, "bf16", 1.0, w.cache, "bf16", 1.0, w.block_table, w.seq_lens,
                     w.softmax_scale, block_size=w.block_size)
    q.put({"seconds": time.perf_counter() - t0, "keys": reps * int(w.seq_lens.sum())})


def cpu_baseline_tiny_1core(reps=20):
    """The oracle on the tiny batch (2 requests, 16 heads, 167 keys) in a
    spawned process limited to one BLAS thread."""
    env_keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        p = ctx.Process(target=_tiny_worker, args=(q, reps))
        p.start()
        r = q.get(timeout=600)
        p.join(timeout=60)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return {"value": r["keys"] / r["seconds"], "unit": UNIT, "cores": 1, "kind": "oracle",
            "us_per_call": r["seconds"] / reps * 1e6,
            "sample": f"fp64 numpy oracle, tiny_dense whole batch x {reps}, one BLAS thread"}


def cpu_baseline(budget_s=20.0):
    return cpu_baseline_steps(budget_s, 1)[0]


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def aggregate_over_ranks(times_ms, units, device=None):
    """Whole-job numbers from per-rank ones: every time is the max over ranks
    (the slowest replica bounds the job), the work units are summed. Without
    an initialised process group (one rank) the inputs come back unchanged."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(times_ms), float(units)
    dev = device if device is not None else torch.device("cpu")
    t = torch.tensor(list(times_ms), dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([float(units)], dtype=torch.float64, device=dev)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.tolist()], float(u.item())


def tensor_peak_tflops(peaks, kv_dtype):
    """Dense tensor peak for the arithmetic a workload runs: the measured bf16
    GEMM peak, times the nominal e4m3:bf16 ratio (4.5 / 2.25 PFLOP/s dense)
    for an e4m3 cache."""
    return float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * (
        2.0 if kv_dtype == "fp8" else 1.0)


def roofline_of(w, kernel_us, peaks):
    """Both fractions of one decode launch and the bound that applies: HBM when
    its algorithmic bytes at the measured copy rate take longer than its
    flops at the dtype's dense peak, else the tensor pipe."""
    alg = _alg_bytes_decode(w)
    flops = _flops(w)
    bw = float(peaks["hbm_gbs"])
    tp = tensor_peak_tflops(peaks, w.kv_dtype)
    t_mem_us = alg / (bw * 1e9) * 1e6
    t_tc_us = flops / (tp * 1e12) * 1e6
    gbs = alg / (kernel_us * 1e-6) / 1e9
    tfs = flops / (kernel_us * 1e-6) / 1e12
    return {"bound": "hbm" if t_mem_us >= t_tc_us else "tensor",
            "hbm_gbs": gbs, "hbm_frac": gbs / bw, "tensor_tflops": tfs,
            "tensor_peak_tflops": tp, "tensor_frac": tfs / tp,
            "algorithmic_bytes": alg, "algorithmic_flops": flops}


def make_decode_only(B, dw, w, plan):
    """The decode launch of one step alone: the kernel over the step's work
    list (balanced plans) or the split-K stage writing its partials."""
    import torch
    dev = dw.device
    T, H, NS = w.num_tokens, w.num_heads, plan.num_segments
    so = torch.empty((T, H, NS, 512), dtype=torch.float32, device=dev)
    sm = torch.empty((T, H, NS), dtype=torch.float32, device=dev)
    se = torch.empty((T, H, NS), dtype=torch.float32, device=dev)
    if w.sparse:
        dw.convert()
    balanced = plan.schedule == 1
    if balanced:  # the work list a step computes, for the same lengths
        B.mla_decode_schedule(plan, seq_lens=None if w.sparse else dw.seq_lens,
                              qo_indptr=dw.qo_indptr, workspace=dw.workspace)

    def decode_only():
        if balanced:
            B.mla_decode_items(plan, dw.q, dw.cache,
                               block_table=None if w.sparse else dw.block_table,
                               seq_lens=None if w.sparse else dw.seq_lens,
                               qo_indptr=dw.qo_indptr, sparse_slots=dw.slots,
                               softmax_scale=w.softmax_scale, q_scale=w.q_scale,
                               kv_scale=w.kv_scale, sinks=dw.sinks, workspace=dw.workspace,
                               out=dw.out, lse=dw.lse)
            return
        B.mla_decode_segments(plan, dw.q, dw.cache,
                              block_table=None if w.sparse else dw.block_table,
                              seq_lens=None if w.sparse else dw.seq_lens,
                              qo_indptr=dw.qo_indptr, sparse_slots=dw.slots,
                              softmax_scale=w.softmax_scale, q_scale=w.q_scale,
                              kv_scale=w.kv_scale, segm_output=so, segm_max=sm, segm_expsum=se)
    return decode_only


def time_loop(fn, steps, flush, stream):
    """Per-call device times (ms) of fn, L2 flushed before each, CUDA events on
    the launching stream. All calls are queued before the one synchronisation
    at the end, so that the host's launch work (and any pause of the host
    thread) overlaps queued device work instead of falling between a call's
    two events."""
    import torch
    evs = []
    for _ in range(steps):
        flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


# The other workload shapes, timed in the same run as the headline: the
# small-case check, the e4m3 batch at the two head counts the pages quote,
# multi-token rows with sinks, and the sparse top-k decode.
SIDE_WORKLOADS = [("tiny", 16), ("fp8", 16), ("fp8", 128), ("mtp", 128), ("sparse", 128)]


def side_workloads(B, dev, flush, stream, peaks, steps):
    import torch
    res = {}
    for name, heads in SIDE_WORKLOADS:
        w, desc = _build_workload(name, heads=heads)
        dw = B.DeviceWorkload(w, device=dev)
        plan = dw.plan
        for _ in range(3):
            dw.forward()
        torch.cuda.synchronize(dev)
        step = time_loop(dw.forward, steps, flush, stream)
        dec_fn = make_decode_only(B, dw, w, plan)
        for _ in range(3):
            dec_fn()
        dec = time_loop(dec_fn, steps, flush, stream)
        us = statistics.mean(step) * 1e3
        dus = statistics.mean(dec) * 1e3
        key = f"{name}_h{heads}" if name == "fp8" else name
        res[key] = {"workload": desc, "us_per_call": us, "decode_us": dus,
                    "kv_tokens_per_s": _kv_keys(w) / (us * 1e-6),
                    "kernel": int(plan.kernel), "rows_per_cta": int(plan.rows_per_cta),
                    "schedule": "balanced" if plan.schedule == 1 else "uniform",
                    "num_segments": int(plan.num_segments), "status_word": dw.status(),
                    "traffic": _profiled_traffic(_alg_bytes_decode(w), int(plan.kernel), name, heads),
                    **roofline_of(w, dus, peaks)}
        del dw, dec_fn
        torch.cuda.empty_cache()
    return res


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from paged_mla_decode_06_gb300 import binding as B
    from paged_mla_decode_06_gb300 import build as BUILD

    BUILD.build()
    B.load_library()
    w, workload = _build_workload(args.workload, seed_offset=rank, batch=args.batch,
                                  heads=args.heads)
    kern = {"auto": B.MLA_KERNEL_AUTO, "mma": B.MLA_KERNEL_WARP_MMA,
            "tc": B.MLA_KERNEL_TCGEN05}[args.kernel]
    dw = B.DeviceWorkload(w, device=dev, kernel=kern,
                          num_segments=args.num_segments if args.num_segments else None)
    plan = dw.plan
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- device-resident timing of the whole step
    for _ in range(args.warmup):
        dw.forward()
    barrier()
    # the raw clock samples go to a CSV only when MLA_BENCH_CLOCKS_CSV names one
    sampler = ClockSampler(smi_gpu_id(dev), os.environ.get("MLA_BENCH_CLOCKS_CSV") or None)
    sampler.start()
    barrier()
    t_wall = time.perf_counter()
    step_ms = time_loop(dw.forward, args.steps, flush, stream)
    barrier()
    wall = time.perf_counter() - t_wall

    # ---- the decode kernel alone (same launch as inside the step)
    T, H, NS = w.num_tokens, w.num_heads, plan.num_segments
    balanced = plan.schedule == 1
    decode_only = make_decode_only(B, dw, w, plan)
    for _ in range(3):
        decode_only()
    dec_ms = time_loop(decode_only, args.steps, flush, stream)
    clocks = sampler.stop()

    # ---- end to end through the C ABI with host buffers: every step copies
    # the step's inputs (q, block table / top-k indices, lengths) from pinned
    # host memory and the output and LSE back; the cache is device-resident.
    pairs = [(dw.q, torch.from_numpy(w.q.view(np.int16 if w.q_dtype == "bf16" else np.uint8)))]
    if w.sparse:
        pairs += [(dw.topk_indices, torch.from_numpy(w.topk_indices)),
                  (dw.req_id, torch.from_numpy(w.req_id_per_token))]
    else:
        pairs += [(dw.block_table, torch.from_numpy(w.block_table)),
                  (dw.seq_lens, torch.from_numpy(w.seq_lens))]
        if dw.qo_indptr is not None:
            pairs.append((dw.qo_indptr, torch.from_numpy(w.qo_indptr)))
    pairs = [(d, h.pin_memory()) for d, h in pairs]
    h_out = torch.empty((T, H, 512), dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty((T, H), dtype=torch.float32).pin_memory()
    h2d = sum(h.numel() * h.element_size() for _, h in pairs)
    d2h = h_out.numel() * 2 + h_lse.numel() * 4

    def e2e_step():
        for d, h in pairs:
            d.copy_(h.view(d.dtype) if h.dtype != d.dtype else h, non_blocking=True)
        dw.forward()
        h_out.copy_(dw.out, non_blocking=True)
        h_lse.copy_(dw.lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ms = []
    for _ in range(args.steps):
        flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))

    keys_rank = float(_kv_keys(w))
    (ms, dms, ems), keys_total = aggregate_over_ranks(
        [statistics.mean(step_ms), statistics.mean(dec_ms), statistics.mean(e2e_ms)],
        keys_rank, dev if world > 1 else None)

    if rank == 0:
        peaks, src = _peaks()
        alg = _alg_bytes_decode(w)
        rf = roofline_of(w, dms * 1e3, peaks)
        kname = {4: "decode_tc_kernel (tcgen05 CTA pair, rows as M)",
                 5: "decode_hn_kernel (tcgen05, rows as N)"}.get(int(plan.kernel),
                                                                "decode_mma_kernel (warp MMA)")
        if rf["bound"] == "hbm":
            roof = {"bound": "hbm", "achieved": rf["hbm_gbs"], "peak": float(peaks["hbm_gbs"]),
                    "unit": "GB/s", "frac": rf["hbm_frac"], "peak_source": f"hbm_gbs of {src}"}
        else:
            roof = {"bound": "tensor", "achieved": rf["tensor_tflops"], "peak": rf["tensor_peak_tflops"],
                    "unit": "TFLOP/s", "frac": rf["tensor_frac"],
                    "peak_source": f"bf16_tflops (burst) of {src}" +
                                   (" x 2 (nominal e4m3:bf16)" if w.kv_dtype == "fp8" else "")}
        roof.update({"traffic": _profiled_traffic(alg, int(plan.kernel), args.workload, args.heads),
                     "kernel": kname, "kernel_us": dms * 1e3, "algorithmic_bytes": alg,
                     "algorithmic_flops": rf["algorithmic_flops"],
                     "hbm_frac": rf["hbm_frac"], "tensor_tflops": rf["tensor_tflops"],
                     "tensor_frac": rf["tensor_frac"]})
        line = {
            "metric": METRIC,
            "value": keys_total / (ms * 1e-3),
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "us_per_call": ms * 1e3,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16" if w.kv_dtype == "bf16" else "e4m3 (fp32 accumulate, bf16 out)",
            "data": "synthetic (seeded numpy; no dataset or weights)",
            "config": {"workload": workload, "num_segments": NS, "tile_size": plan.tile_size,
                       "schedule": "balanced" if balanced else "uniform",
                       "rows_per_cta": plan.rows_per_cta, "kernel": int(plan.kernel),
                       "kv_tokens_per_gpu": int(keys_rank),
                       "l2": "flushed (256 MiB write) before every timed step",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof,
            "clocks": clocks,
            "e2e": {"value": keys_total / (ems * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": ems},
            "gpu_launches": args.steps * ((3 if balanced else 1 + (1 if NS > 1 else 0)) +
                                          (1 if w.sparse else 0)),
            "status_word": dw.status(),
            "wall_s_timed_region": wall,
        }
        default_line = world == 1 and args.workload == "dsv3" and not args.batch
        if default_line and not args.no_workloads:
            line["workloads"] = side_workloads(B, dev, flush, stream, peaks,
                                               min(args.steps, args.side_steps))
        if default_line and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.cpu_budget)
            line["cpu_baseline"]["tiny_1core"] = cpu_baseline_tiny_1core()
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    n = args.warmup + args.steps
    budget = min(10.0, max(1.0, 90.0 / n))
    recs = cpu_baseline_steps(budget, n)[args.warmup:]
    value = statistics.mean(r["value"] for r in recs)
    ms = statistics.mean(1e3 * r["seconds"] for r in recs)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded numpy; no dataset or weights)",
        "config": {"workload": WORKLOADS["dsv3"].format(b=64),
                   "sample": f"each step a bounded sample (~{budget:.1f} s) of the batch"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": recs[0]["cores"],
                         "kind": "oracle", "sample": recs[-1]["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_kernels_once():
    """One launch of every library kernel on inputs above the 129 MB L2, for
    a profiler's counter pass (no timing, no JSON line): the e4m3 decode at
    128 heads (schedule, rows-as-N decode on CTA-pair clusters, merge; then
    the CTA-pair kernel with the rows as M), the sparse decode (index
    conversion, schedule, decode, merge), the e4m3 decode at 16 heads on the
    warp-MMA kernel and on the rows-as-N kernel, the multi-token decode with
    sinks, the q concat/quantisation, the per-shard LSE merge, the sparse
    list lengths and the fixed-width fit."""
    import torch
    from paged_mla_decode_06_gb300 import binding as B
    from paged_mla_decode_06_gb300 import build as BUILD
    from paged_mla_decode_06_gb300 import inputs as I
    BUILD.build()
    B.load_library()
    dev = torch.device("cuda")
    wf = I.fp8_decode(128, batch=16)                    # 16 x 16384 x 576 B = 151 MB
    ws = I.sparse_topk(num_reqs=8, cache_tokens=32768)  # 64 tokens x 2048 rows x 1152 B
    wm = I.fp8_decode(16, batch=16)
    wt = I.mtp_sinks(batch=16)                          # multi-token rows: 2-4 row tiles per request
    dwf = B.DeviceWorkload(wf, device=dev)
    dwp = B.DeviceWorkload(wf, device=dev, kernel=B.MLA_KERNEL_TCGEN05)
    dws = B.DeviceWorkload(ws, device=dev)
    dwm = B.DeviceWorkload(wm, device=dev, kernel=B.MLA_KERNEL_WARP_MMA)
    dwn = B.DeviceWorkload(wm, device=dev)              # the rows-as-N kernel on the same batch
    dwt = B.DeviceWorkload(wt, device=dev)
    g = torch.Generator(device=dev).manual_seed(11)
    T, H = 1024, 128
    nope = torch.randn(T, H, 512, device=dev, generator=g).to(torch.bfloat16)
    pe = torch.randn(T, H, 64, device=dev, generator=g).to(torch.bfloat16)
    qout = torch.empty(T, H, 576, dtype=torch.uint8, device=dev)
    sh_out = torch.randn(4, 256, 128, 512, device=dev, generator=g).to(torch.bfloat16)
    sh_lse = torch.randn(4, 256, 128, device=dev, generator=g)
    mo = torch.empty(256, 128, 512, dtype=torch.bfloat16, device=dev)
    ml = torch.empty(256, 128, device=dev)
    R = 8192
    qsl = torch.arange(0, 2 * R + 1, 2, dtype=torch.int32, device=dev)
    seq = torch.randint(0, 8192, (R,), dtype=torch.int32, device=dev, generator=g)
    ptr = torch.empty(2 * R + 1, dtype=torch.int32, device=dev)
    ti = torch.randint(-1, 1 << 20, (16384, 2112), dtype=torch.int32, device=dev, generator=g)
    fit = torch.empty(16384, 2048, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    dwf.forward()
    dwp.forward()
    dws.forward()
    dwm.forward()
    dwn.forward()
    dwt.forward()
    B.mla_concat_quant_q(nope, pe, out=qout, q_scale=0.05)
    B.mla_merge_lse(sh_out, sh_lse, out=mo, lse=ml)
    B.mla_sparse_seqlen(qsl, seq, topk=2048, indptr=ptr)
    B.mla_fit_kpool_indices(ti, topk=2048, out=fit)
    torch.cuda.synchronize()
    if any(d.status() != 0 for d in (dwf, dwp, dws, dwn, dwt)):
        raise RuntimeError("device status word set")
    print("kernels-once ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workload shapes on the default line")
    ap.add_argument("--side-steps", type=int, default=100,
                    help="timed calls per workload of the workloads object")
    ap.add_argument("--kernel", default="auto", choices=["auto", "mma", "tc"],
                    help="decode kernel variant (default: the planner's choice)")
    ap.add_argument("--num-segments", type=int, default=0,
                    help="split-K segments (default: the planner's choice)")
    ap.add_argument("--workload", default="dsv3", choices=sorted(WORKLOADS),
                    help="dsv3 (the measured default), tiny, fp8, mtp or sparse")
    ap.add_argument("--batch", type=int, default=0,
                    help="requests per batch (0: the workload's own; smaller batches of the "
                         "same shape are for profiler captures)")
    ap.add_argument("--heads", type=int, default=128, help="heads of the fp8 workload")
    ap.add_argument("--kernels-once", action="store_true",
                    help="launch every library kernel once (for a profiler pass) and exit")
    args = ap.parse_args()
    if args.kernels_once:
        run_kernels_once()
        return
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
