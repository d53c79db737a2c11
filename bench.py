"""Benchmark one packed paged-attention step (KV append + attention) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference] [--config NAME] [--only]

A step is one pass of the whole path over one synthetic batch: KV append of
the step's new tokens, split-KV attention with its LSE merge, and the
tensor-core prefill tiles when present.  The step plan (host step metadata) is
an input like the block tables: resident in HBM for `value`, computed and
uploaded per step inside `e2e`.

The line's workload is the high-concurrency decode step (256 sequences, 3.4 GB
of KV), the largest of the five step shapes the metric is quoted on; the other
four (tiny decode, small-model decode, the agent-shaped mixed step, the
shared-prefix verify step) are timed in the same process, the same way, and
reported under `configs`, each with its own e2e (--only skips them).

* value: KV tokens/s = sum(context_lens) / device time per step, inputs resident
  in HBM, the step replayed from a CUDA graph, L2 flushed before every timed
  step (a 256 MB buffer written, then another 256 MB read, so L2 holds only
  clean unrelated lines) and the flush kept outside the per-step CUDA-event pairs.
* roofline: the dominant kernel alone (split-KV decode: bytes vs the measured
  HBM copy bandwidth; tensor-core prefill: FLOPs vs the measured bf16 peak),
  timed with CUDA events recorded on its launch stream around each launch
  (library profiling hook), algorithmic bytes or FLOPs / mean duration.  The
  split-KV kernel's bytes are the K/V blocks its plan streams (a shared prefix
  the plan reads once per CTA counted once, one gathered onto the tensor cores
  not at all) plus q, out and metadata; the tensor-core kernel's FLOPs are
  4 * D * (query row, key) pairs: the causal pairs of prefill-class sequences
  plus the gathered shared-prefix pairs.  A step with tensor-core work also
  reports the step against both roofs (step_roofline: t = max(bytes / BW,
  FLOPs / peak) over the measured step time).
* e2e: the same metric through the public API from pinned HOST buffers: every
  step copies q, the new K/V, slot mapping, metadata and the plan host->device
  (one pinned buffer, one transfer), plans on the host from the caller's host
  arrays into pinned memory (on the library's planning thread, while the copy
  and the KV append are queued), runs append + attention and copies out back
  (wall time per step).
* cpu_baseline / --impl reference: the fp64 CPU oracle as it stands, on the
  host cores, on a bounded sample of the same workload.
"""

from __future__ import annotations

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

import workloads  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
METRIC = "paged-attention step: KV tokens/s and achieved HBM GB/s vs peak on 1 GB300"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


PREFILL_MIN_Q = 64   # sequences with at least this many query tokens run on the tensor-core kernel


# Sources that decide what a kernel does for a given workload: its own file,
# the planner (its work lists), the entry points and the shared headers.
KERNEL_SOURCES = {
    "decode_kernel": ["pkv_decode.cu", "pkv_plan.cpp"],
    "prefill_kernel": ["pkv_prefill.cu", "pkv_plan.cpp"],
    "state_checkpoint_kernel": ["pkv_state.cu"],
}
COMMON_SOURCES = ["pkv_api.cu", "pkv_device.cuh", "pkv_tc.cuh", "pkv_internal.h"]


def source_sha256(kernel: str) -> str:
    """Hash of the sources behind one kernel, as recorded next to its ncu traffic."""
    import hashlib
    d = os.path.join(ROOT, "paged_kv_attention_append_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(KERNEL_SOURCES[kernel] + COMMON_SOURCES):
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(ROOT, "include", "pkv.h"), "rb") as fh:
        h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(kernel: str, workload: str):
    """ncu DRAM bytes per launch for this kernel/workload, or None when no capture
    exists or the kernels changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{kernel}/{workload}")
        if rec and rec.get("source_sha256") == source_sha256(kernel):
            return int(rec["dram_bytes"])
    except Exception:
        pass
    return None


def algorithmic_bytes(meta, prefill=None) -> int:
    """KV + Q + O + metadata bytes of one attention pass (split-KV scratch excluded).

    prefill=None counts every sequence; False only the split-KV (decode-class)
    sequences; True only the tensor-core (prefill-class) ones."""
    d, hq, hkv = meta.head_dim, meta.num_q_heads, meta.num_kv_heads
    live = meta.q_lens > 0
    if prefill is not None:
        live &= (meta.q_lens >= PREFILL_MIN_Q) == prefill
    kv = int(meta.context_lens[live].astype(np.int64).sum()) * 2 * hkv * d * 2
    qo = 2 * int(meta.q_lens[live].astype(np.int64).sum()) * hq * d * 2
    nb = int(((meta.context_lens[live].astype(np.int64) + 15) // 16).sum())
    return kv + qo + 4 * (2 * int(live.sum()) + 1) + 4 * nb


def decode_kernel_bytes(meta, info) -> int:
    """Bytes the split-KV kernel must move for one launch of this plan: the K and V
    of every (KV block, KV head) pair it streams (a prefix the plan reads once per
    shared-prefix CTA counted once; a prefix gathered onto the tensor cores not at
    all), plus the q and out rows of the split-KV sequences and their metadata."""
    d, hq = meta.head_dim, meta.num_q_heads
    live = (meta.q_lens > 0) & (meta.q_lens < PREFILL_MIN_Q)
    kv = int(info.decode_blocks) * 16 * 2 * d * 2
    qo = 2 * int(meta.q_lens[live].astype(np.int64).sum()) * hq * d * 2
    nb = int(((meta.context_lens[live].astype(np.int64) + 15) // 16).sum())
    return kv + qo + 4 * (2 * int(live.sum()) + 1) + 4 * nb


def unique_bytes(meta) -> int:
    d, hq, hkv = meta.head_dim, meta.num_q_heads, meta.num_kv_heads
    return meta.unique_blocks() * 16 * 2 * hkv * d * 2 + 2 * meta.total_q * hq * d * 2


def prefill_flops(meta) -> int:
    """4*D*Hq*(visible (q, k) pairs) over the tensor-core (prefill-class) sequences."""
    pairs = 0
    for s in range(meta.num_seqs):
        qs, ctx = int(meta.q_lens[s]), int(meta.context_lens[s])
        if qs >= PREFILL_MIN_Q:
            pairs += sum(ctx - qs + i + 1 for i in range(qs))
    return 4 * meta.head_dim * meta.num_q_heads * pairs


class ClockSampler:
    """nvidia-smi sampling in the background during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or self.file is None:
            return None
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


ORACLE_MAX_KV_TOKENS = 60000   # bound on the oracle sample's pool (host memory and set-up time)


def oracle_sample_step(meta):
    """The workload itself, or its first sequences up to ORACLE_MAX_KV_TOKENS of
    context (same shapes and length distribution, a smaller pool)."""
    if meta.kv_tokens() <= ORACLE_MAX_KV_TOKENS:
        return meta, "full step"
    n, tok = 0, 0
    while n < meta.num_seqs and (n == 0 or tok + int(meta.context_lens[n]) <= ORACLE_MAX_KV_TOKENS):
        tok += int(meta.context_lens[n])
        n += 1
    sub = workloads.build_step(meta.name, meta.seed, meta.q_lens[:n], meta.context_lens[:n],
                               meta.num_q_heads, meta.num_kv_heads, meta.head_dim,
                               scale=meta.scale)
    return sub, f"first {n} of {meta.num_seqs} sequences"


def run_oracle_sample(meta, target_s=10.0, max_reps=1000, num_threads=0):
    """Time the oracle (append + attention) on whole steps of a bounded sample of the
    workload, or on a fixed subset of its query rows when even one step would take
    longer than about target_s.  Reports KV tokens/s of the work actually done."""
    import oracle
    step, what = oracle_sample_step(meta)
    q, k, v, pool = workloads.make_values(step, device="cpu")
    rows_total = step.total_q * step.num_q_heads
    # cost model: one row costs ~ its visible keys
    t0 = time.perf_counter()
    probe_rows = np.arange(0, rows_total, max(1, rows_total // 64), dtype=np.int64)
    oracle.run_step(step, q, k, v, pool, rows=probe_rows, num_threads=num_threads)
    per_row = (time.perf_counter() - t0) / len(probe_rows)
    full = per_row * rows_total
    if full <= target_s:
        reps, rows = min(max(1, int(target_s / max(full, 1e-6))), max_reps), None
        sample = what
    else:
        n = max(1, int(rows_total * target_s / full))
        rows = np.sort(np.random.default_rng(0).choice(rows_total, size=n, replace=False)).astype(np.int64)
        reps, sample = 1, f"{what}, {n} of {rows_total} query rows"
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.run_step(step, q, k, v, pool, rows=rows, num_threads=num_threads)
    dt = time.perf_counter() - t0
    if rows is None:
        kv_tok = step.kv_tokens() * reps
    else:   # credit each sampled row with its share of the step's KV tokens
        kv_tok = step.kv_tokens() * len(rows) / rows_total
    cores = num_threads if num_threads > 0 else oracle.max_threads()
    return {"value": kv_tok / dt, "unit": "KV tokens/s", "cores": cores,
            "kind": "oracle", "seconds": dt,
            "sample": f"{meta.name}: {sample} x {reps} (fp64 C oracle, OpenMP, {cores} threads)"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _dist_active() -> bool:
    import torch.distributed as dist
    return dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1


def barrier():
    """Barrier over all ranks (no-op in a single process)."""
    if _dist_active():
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank scalar (a step time) over all ranks; identity in one process."""
    if not _dist_active():
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world_size: int, seconds: float) -> float:
    """Whole-job throughput of independent replicas: every rank processes the same
    number of units (weak scaling) and the job takes the slowest rank's time."""
    return world_size * units_per_rank / seconds


def bench_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    meta = workloads.make_config(args.config)
    for _ in range(args.warmup):
        run_oracle_sample(meta, target_s=0.5, max_reps=1)
    times, vals = [], []
    for _ in range(args.steps):
        r = run_oracle_sample(meta, target_s=2.0, max_reps=1)
        vals.append(r["value"])
    v = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "KV tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": meta.kv_tokens() / v * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(meta, ws),
            "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": v, "unit": "KV tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    line["cpu_baseline"]["value"] = v
    print(json.dumps(line), flush=True)


L2_NOTE = (f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MB written, then "
           f"{L2_FLUSH_BYTES >> 20} MB read)")
TIMING_NOTE = ("CUDA graph replay per step, CUDA events per step; kernel intervals from event "
               "nodes captured around each kernel (second graph, no programmatic launch)")
# the five step shapes the metric is quoted on (the first is correctness-only
# and launch-bound); the line's own workload is the largest that fits one GPU
BASELINE_CONFIGS = ["tiny_decode", "small_decode", "agent_mixed", "high_conc_decode",
                    "shared_prefix_verify"]
HEADLINE = "high_conc_decode"


def config_of(meta, ws: int) -> dict:
    """The workload keys of a bench line (identical for the pkv and reference arms)."""
    nch = workloads.chain_steps(meta)
    return {**workloads.describe(meta), **({"chain_steps": nch} if nch > 1 else {}),
            "parallelism": f"replicas x{ws}" if ws > 1 else "single"}


class StepBench:
    """One workload resident on the GPU: its inputs, plan, a CUDA graph of one
    step, and the timings of the step and of each kernel in it."""

    def __init__(self, pkv, meta, dev, stream):
        import torch
        self.pkv, self.meta, self.dev, self.stream = pkv, meta, dev, stream
        nch = self.nch = workloads.chain_steps(meta)
        self.metas = [workloads.chain_step(meta, meta.context_lens, t) for t in range(nch)]
        q, k, v, pool = workloads.make_values(meta, device=dev)
        self.pool = pool
        self.vals = [(q, k, v)] + [tuple(workloads.make_values(m, seed=meta.seed + t, device=dev)[:3])
                                   for t, m in enumerate(self.metas) if t > 0]
        self.slots0 = torch.from_numpy(meta.slot_mapping).to(dev)
        self.slots = self.slots0.clone()
        self.cu_d = torch.from_numpy(meta.cu_q_lens).to(dev)
        self.ctx0_d = torch.from_numpy(meta.context_lens).to(dev)
        self.ctx_d = self.ctx0_d.clone()
        self.bt_d = torch.from_numpy(meta.block_tables).to(dev)
        self.outs = [torch.empty_like(x[0]) for x in self.vals]
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.chain_arg = nch if nch > 1 else None
        self.info, self.host_plan = pkv.plan_step(
            meta.cu_q_lens, meta.context_lens, meta.num_q_heads, pool, upload=False,
            chain_steps=self.chain_arg, block_tables=meta.block_tables)
        self.plan = pkv.StepPlan(self.info, self.host_plan, dev)

    def host_plan_us(self, reps=50):
        """Host planning per step as the e2e loop does it: one bound planner call
        (pkv_plan_step_ex) over the step's int32 arrays into a reused buffer."""
        import numpy as np
        import torch
        m = self.meta
        cu = np.ascontiguousarray(m.cu_q_lens, dtype=np.int32)
        ctx = np.ascontiguousarray(m.context_lens, dtype=np.int32)
        bt = np.ascontiguousarray(m.block_tables, dtype=np.int32)
        out = np.zeros(((int(self.info.plan_bytes) + 4095) // 4096 + 1) * 1024, dtype=np.int32)
        planner = self.pkv.BoundPlan(
            cu, ctx, m.num_q_heads, self.pool, out, chain_steps=self.chain_arg, block_tables=bt,
            num_sms=torch.cuda.get_device_properties(self.dev).multi_processor_count)
        planner.run()
        t0 = time.perf_counter()
        for _ in range(reps):
            planner.run()
        return (time.perf_counter() - t0) / reps * 1e6

    def step(self):
        # the plan is a step input like the block tables: uploaded before the
        # timed region (StepPlan); host planning and its upload are timed in e2e
        pkv, m = self.pkv, self.meta
        if self.nch > 1:
            self.ctx_d.copy_(self.ctx0_d)
            self.slots.copy_(self.slots0)
        for t, (qt, kt, vt) in enumerate(self.vals):
            pkv.paged_kv_append(kt, vt, self.slots, self.pool, dev_status=self.status)
            pkv.paged_varlen_attention(qt, self.cu_d, self.ctx_d, self.bt_d, self.pool, m.scale,
                                       plan=self.plan, out=self.outs[t], dev_status=self.status)
            if t + 1 < self.nch:
                pkv.decode_advance(self.ctx_d, self.slots, self.cu_d, self.bt_d, self.pool,
                                   dev_status=self.status)

    def measure(self, args, flush_l2, clock_sampler=None):
        """Step time (graph replay, L2 flushed before each) and per-kernel times
        (event nodes around each kernel in a second graph)."""
        import torch
        pkv, dev, stream = self.pkv, self.dev, self.stream
        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup)):
                self.step()
        torch.cuda.synchronize(dev)
        assert int(self.status.item()) == 0, f"device status {int(self.status.item())}"
        launches_before = pkv.kernel_launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self.step()
        self.launches_per_step = pkv.kernel_launch_count() - launches_before
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                flush_l2()
                graph.replay()
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        with (clock_sampler if clock_sampler is not None else _nullctx()):
            with torch.cuda.stream(stream):
                for a, b in ev:
                    flush_l2()
                    a.record(stream)
                    graph.replay()
                    b.record(stream)
            torch.cuda.synchronize(dev)
            info = self.info
            present = {"append": True, "decode": info.num_decode_warps + info.num_shared_ctas > 0,
                       "merge": info.num_kernels > (1 if info.num_decode_warps + info.num_shared_ctas > 0 else 0)
                       + (1 if info.num_prefill_tiles > 0 else 0),
                       "prefill": info.num_prefill_tiles > 0}
            k_ev = {n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for n in present}
            samples = {n: [] for n in present}
            with torch.cuda.stream(stream):
                for a, b in k_ev.values():
                    a.record(stream)
                    b.record(stream)
                torch.cuda.synchronize(dev)
                for name, (a, b) in k_ev.items():
                    pkv.set_profile_events(name, a, b)
                graph_k = torch.cuda.CUDAGraph()
                try:
                    with torch.cuda.graph(graph_k, stream=stream):
                        self.step()
                finally:
                    for name in k_ev:
                        pkv.set_profile_events(name)
                for i in range(args.warmup + args.steps):
                    flush_l2()
                    graph_k.replay()
                    stream.synchronize()
                    if i >= args.warmup:
                        for name, (a, b) in k_ev.items():
                            if present[name]:
                                samples[name].append(a.elapsed_time(b))
            torch.cuda.synchronize(dev)
        self.step_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / args.steps, dev)
        self.kern_ms = {n: (statistics.mean(samples[n]) if present[n] and samples[n] else 0.0)
                        for n in k_ev}
        assert int(self.status.item()) == 0, f"device status {int(self.status.item())}"
        # warm: the same step replayed back to back without the L2 flush
        ev_w = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            graph.replay()
            for a, b in ev_w:
                a.record(stream)
                graph.replay()
                b.record(stream)
        torch.cuda.synchronize(dev)
        self.warm_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev_w) / args.steps, dev)
        self.graph = graph

    def summary(self, ws: int, steps: int) -> dict:
        """Throughput, the dominant kernel's roofline, per-kernel times; for a step
        with tensor-core work, the step-level pair of fractions."""
        meta, info, pk = self.meta, self.info, peaks()
        kv_tok = sum(m.kv_tokens() for m in self.metas)          # over the chain's steps
        bytes_alg = sum(algorithmic_bytes(m) for m in self.metas)
        # kernel events keep the last launch of a chain: its step's bytes (the
        # plan of a chain is sized for its last step)
        dec_bytes = decode_kernel_bytes(self.metas[-1], info)
        # tensor-core work: prefill-class sequences and gathered shared-prefix rows
        fl = prefill_flops(meta) + 4 * meta.head_dim * int(info.gather_pairs)
        km = self.kern_ms
        decode_ms, prefill_ms = km["decode"], km["prefill"]
        kernels = {"append_kernel": {"ms_per_launch": km["append"]}}
        if km["merge"]:
            kernels["merge_kernel"] = {"ms_per_launch": km["merge"]}
        if decode_ms:
            kernels["decode_kernel"] = {"ms_per_launch": decode_ms, "bytes_per_launch": dec_bytes,
                                        "gbs": dec_bytes / (decode_ms * 1e-3) / 1e9,
                                        "frac_hbm": dec_bytes / (decode_ms * 1e-3) / 1e9 / pk["hbm_gbs"]}
        if prefill_ms:
            kernels["prefill_kernel"] = {"ms_per_launch": prefill_ms, "flops_per_launch": fl,
                                         "tflops": fl / (prefill_ms * 1e-3) / 1e12,
                                         "frac_bf16": fl / (prefill_ms * 1e-3) / 1e12 / pk["bf16_tflops"]}
        if prefill_ms > decode_ms:     # the dominant kernel is a dense contraction
            achieved = fl / (prefill_ms * 1e-3) / 1e12
            roofline = {"bound": "tensor", "kernel": "prefill_kernel", "achieved": achieved,
                        "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                        "traffic": recorded_traffic("prefill_kernel", meta.name),
                        "flops_per_launch": fl, "ms_per_launch": prefill_ms,
                        "peak_source": pk["source"] + " (bf16 burst)",
                        "frac_sustained": achieved / (pk["bf16_tflops_sustained"] or pk["bf16_tflops"])}
        elif decode_ms:
            achieved = dec_bytes / (decode_ms * 1e-3) / 1e9
            roofline = {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved,
                        "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                        "traffic": recorded_traffic("decode_kernel", meta.name),
                        "bytes_per_launch": dec_bytes, "ms_per_launch": decode_ms,
                        "peak_source": pk["source"]}
        else:
            roofline = None
        out = {
            "value": job_throughput(kv_tok, ws, self.step_ms * 1e-3), "unit": "KV tokens/s",
            "ms_per_step": self.step_ms, "roofline": roofline, "kernels": kernels,
            "step_gbs": bytes_alg / (self.step_ms * 1e-3) / 1e9,
            "step_frac_hbm": bytes_alg / (self.step_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "gpu_launches": self.launches_per_step * steps,
            "warm": {"value": job_throughput(kv_tok, ws, self.warm_ms * 1e-3),
                     "ms_per_step": self.warm_ms, "l2": "not flushed: the step replayed back to back"},
            "plan": {"decode_warps": info.num_decode_warps, "decode_pieces": info.num_decode_pieces,
                     "merge_groups": info.num_merge_groups, "prefill_tiles": info.num_prefill_tiles,
                     "shared_prefix_ctas": info.num_shared_ctas, "kernels_per_call": info.num_kernels,
                     "gathered_rows": info.num_gather_rows * (meta.num_q_heads // meta.num_kv_heads)},
        }
        if fl:
            # the step as a whole against both roofs: t_roofline = max(bytes / BW, flops / peak),
            # bytes counting blocks several sequences share once (what HBM must deliver)
            step_bytes = min(bytes_alg, unique_bytes(meta)) if self.nch == 1 else bytes_alg
            t_b = step_bytes / (pk["hbm_gbs"] * 1e9)
            t_f = fl / (pk["bf16_tflops"] * 1e12)
            t_s = self.step_ms * 1e-3
            out["step_roofline"] = {
                "bytes": step_bytes, "flops": fl, "t_bytes_ms": t_b * 1e3, "t_flops_ms": t_f * 1e3,
                "t_roofline_ms": max(t_b, t_f) * 1e3, "frac": max(t_b, t_f) / t_s,
                "frac_hbm": t_b / t_s, "frac_tensor": t_f / t_s,
                "bound": "tensor" if t_f >= t_b else "hbm"}
            out["prefill_tflops_step"] = fl / t_s / 1e12
        if meta.unique_blocks() * 16 < kv_tok and decode_ms:
            out["unique_gbs"] = unique_bytes(meta) / (decode_ms * 1e-3) / 1e9
        return out

    def e2e(self, args, ws):
        """Wall time per step through the public API from pinned host buffers (a
        chained workload: all its steps' inputs in, one plan, every output back).
        The step's int32 metadata, every step's bf16 q/k/v and, last, the plan
        (written by the host planner each step) share one pinned buffer, so one
        copy carries all of them.  The planner reads the caller's own host
        arrays (lengths and block tables), not their staging copies in that
        buffer: on Grace, host reads of pinned lines the device copy has just
        read run slower (a 256-sequence plan 56-58 us from the staging copies,
        43 us from the caller's arrays, the copy running or not)."""
        import torch
        pkv, dev, stream, meta, info = self.pkv, self.dev, self.stream, self.meta, self.info

        def packed(parts):
            offs, n = [], 0
            for t in parts:
                offs.append(n)
                n += (t.numel() * t.element_size() + 15) // 16 * 16
            hbuf = torch.zeros(max(n, 16), dtype=torch.uint8).pin_memory()
            dbuf = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
            dviews, hviews = [], []
            for t, o in zip(parts, offs):
                nb = t.numel() * t.element_size()
                hv = hbuf[o:o + nb].view(t.dtype).view(t.shape)
                hv.copy_(t.cpu())
                dviews.append(dbuf[o:o + nb].view(t.dtype).view(t.shape))
                hviews.append(hv)
            return hbuf, dbuf, dviews, hviews

        plan_words = ((int(info.plan_bytes) + 4095) // 4096 + 1) * 1024
        qkv_parts = [x for qkv in self.vals for x in qkv]
        buf_h, buf_d, dviews, hviews = packed(
            [self.slots0, self.cu_d, self.ctx0_d, self.bt_d] + qkv_parts +
            [torch.zeros(plan_words, dtype=torch.int32)])
        ds, dcu, dctx, dbt = dviews[:4]
        dplan = dviews[-1]
        cu_h, ctx_h, bt_h, plan_hv = hviews[1], hviews[2], hviews[3], hviews[-1]
        plan_off = plan_hv.data_ptr() - buf_h.data_ptr()          # bytes, 16-byte aligned
        qkv_dv = dviews[4:-1]
        dvals = [tuple(qkv_dv[3 * t:3 * t + 3]) for t in range(len(self.vals))]
        plan_np = plan_hv.numpy()
        cu_np = np.ascontiguousarray(self.meta.cu_q_lens, dtype=np.int32)
        ctx_np = np.ascontiguousarray(self.meta.context_lens, dtype=np.int32)
        bt_np = np.ascontiguousarray(self.meta.block_tables, dtype=np.int32)
        assert (np.array_equal(cu_np, cu_h.numpy()) and np.array_equal(ctx_np, ctx_h.numpy())
                and np.array_equal(bt_np, bt_h.numpy()))
        num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        outs_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in self.outs]
        h2d = (plan_off + int(info.plan_bytes) + 15) // 16 * 16  # bytes copied per step
        plan_e2e = pkv.StepPlan(info, self.host_plan, dev)
        plan_e2e.dev = dplan.view(torch.uint8)
        d2h = sum(o.numel() * o.element_size() for o in outs_h)
        # every step reuses the same host and device buffers: the planner call,
        # the copies and the kernel calls have their arguments bound once
        bound = [pkv.BoundStep(dk, dv, ds, dq, dcu, dctx, dbt, self.pool, meta.scale, plan_e2e,
                               self.outs[t], dev_status=self.status, stream=stream)
                 for t, (dq, dk, dv) in enumerate(dvals)]
        planner = pkv.BoundPlan(cu_np, ctx_np, meta.num_q_heads, self.pool, plan_np,
                                num_sms=num_sms, chain_steps=self.chain_arg, block_tables=bt_np,
                                spin_us=2000)
        up = pkv.BoundCopy(buf_d, buf_h, stream=stream)
        down = [pkv.BoundCopy(oh, o, stream=stream) for oh, o in zip(outs_h, self.outs)]
        times = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                torch.cuda.synchronize(dev)
                t0 = time.perf_counter()
                # the library's planning thread plans the step while this one
                # queues the inputs' copy and the first step's KV append (it
                # needs no plan); the plan follows them up
                planner.post()
                up.run(plan_off)
                bound[0].run_append()
                inf2, plan_nb = planner.wait()
                n = (plan_off + plan_nb + 15) // 16 * 16
                up.run(n - plan_off, plan_off)
                plan_e2e.info = inf2
                for t, b in enumerate(bound):
                    if t > 0:
                        b.run_append()
                    b.run_attention()
                    if t + 1 < self.nch:
                        pkv.decode_advance(dctx, ds, dcu, dbt, self.pool, dev_status=self.status)
                for d in down:
                    d.run()
                stream.synchronize()
                if i >= args.warmup:
                    times.append(time.perf_counter() - t0)
        planner.close()
        assert int(self.status.item()) == 0, f"device status {int(self.status.item())}"
        e2e_s = max_over_ranks(statistics.mean(times), dev)
        kv_tok = sum(m.kv_tokens() for m in self.metas)
        return {"value": job_throughput(kv_tok, ws, e2e_s), "unit": "KV tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3}


class _nullctx:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def bench_pkv(args):
    import torch
    import paged_kv_attention_append_gb300 as pkv

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_acc = torch.zeros((), dtype=torch.float32, device=dev)

    def flush_l2():
        flush_w.zero_()                          # write more than L2 holds ...
        torch.sum(flush_r, dim=0, out=flush_acc)  # ... then read more, leaving clean lines
    stream = torch.cuda.Stream(dev)

    # the other configurations first, each timed the same way and then freed
    others = {}
    if not args.only:
        for name in BASELINE_CONFIGS:
            if name == args.config:
                continue
            b = StepBench(pkv, workloads.make_config(name), dev, stream)
            b.measure(args, flush_l2)
            others[name] = b.summary(ws, args.steps)
            others[name]["e2e"] = b.e2e(args, ws)
            del b
            torch.cuda.empty_cache()

    meta = workloads.make_config(args.config)
    b = StepBench(pkv, meta, dev, stream)
    host_plan_us = b.host_plan_us()
    with ClockSampler(local) as clk:
        b.measure(args, flush_l2, None)
    clocks = clk.summary()
    head = b.summary(ws, args.steps)
    e2e = b.e2e(args, ws)
    cpu = cpu1 = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = run_oracle_sample(meta)                                   # all host cores
        cpu1 = run_oracle_sample(meta, target_s=3.0, num_threads=1)     # one core
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": head["value"], "unit": "KV tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shapes of the named workload)",
        "config": config_of(meta, ws),
        "l2": L2_NOTE, "timing": TIMING_NOTE,
        "gpu_launches": head["gpu_launches"],
        "roofline": head["roofline"],
        "kernels": head["kernels"],
        "step_gbs": head["step_gbs"], "step_frac_hbm": head["step_frac_hbm"],
        "warm": head["warm"],
        "host_plan_us": host_plan_us,
        "e2e": e2e,
        "clocks": clocks,
        "cpu_baseline": None if cpu is None else {
            **{k2: cpu[k2] for k2 in ("value", "unit", "cores", "kind", "sample")},
            "value_1core": cpu1["value"], "sample_1core": cpu1["sample"]},
        "plan": head["plan"],
    }
    for k2 in ("step_roofline", "prefill_tflops_step", "unique_gbs"):
        if k2 in head:
            line[k2] = head[k2]
    if others:
        line["configs"] = {meta.name: {k2: head[k2] for k2 in
                                       ("value", "ms_per_step", "roofline", "kernels", "step_gbs",
                                        "step_frac_hbm", "plan", *[x for x in ("step_roofline",
                                                                               "unique_gbs")
                                                                   if x in head])}}
        line["configs"][meta.name]["e2e"] = e2e
        line["configs"].update({n: {**o, "config": config_of(workloads.make_config(n), ws)}
                                for n, o in others.items()})
    print(json.dumps(line), flush=True)


STATE_POOL_SLOTS = 1650        # ~1,650 cached blocks ...
STATE_ROW_BYTES = 1 << 20      # ... of ~1 MiB state rows: a ~1.6 GiB pool
STATE_ROWS_PER_CALL = 64       # sequences checkpointing at a block boundary in one step


def bench_state_checkpoint(args):
    """State-row checkpoint (in-place row writes into a state pool): bytes read +
    written per second against the measured copy bandwidth.  The pool has the
    page's size; each call writes STATE_ROWS_PER_CALL rows to random slots."""
    import torch
    import paged_kv_attention_append_gb300 as pkv
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(1242)
    pool = torch.randint(0, 256, (STATE_POOL_SLOTS, STATE_ROW_BYTES), dtype=torch.uint8, device=dev,
                         generator=g)
    src = torch.randint(0, 256, (STATE_ROWS_PER_CALL, STATE_ROW_BYTES), dtype=torch.uint8, device=dev,
                        generator=g)
    slots = torch.randperm(STATE_POOL_SLOTS, device=dev, generator=g)[:STATE_ROWS_PER_CALL].to(torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_acc = torch.zeros((), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def flush_l2():
        flush_w.zero_()
        torch.sum(flush_r, dim=0, out=flush_acc)

    def step():
        pkv.state_checkpoint(src, slots, pool, dev_status=status)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2()
            step()
    torch.cuda.synchronize(dev)
    launches_before = pkv.kernel_launch_count()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    pkv.set_profile_events("state", a, b)
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph, stream=stream):
            step()
    finally:
        pkv.set_profile_events("state")
    launches = pkv.kernel_launch_count() - launches_before
    times = []
    barrier()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                flush_l2()
                graph.replay()
                stream.synchronize()
                times.append(a.elapsed_time(b))
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0
    ms = max_over_ranks(statistics.mean(times), dev)
    nbytes = 2 * STATE_ROWS_PER_CALL * STATE_ROW_BYTES
    gbs = nbytes / (ms * 1e-3) / 1e9
    # end to end: host rows pinned -> device, checkpoint, read one row back
    src_h = src.cpu().pin_memory()
    back = torch.empty(STATE_ROW_BYTES, dtype=torch.uint8).pin_memory()
    src_d = torch.empty_like(src)
    e2e = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            src_d.copy_(src_h, non_blocking=True)
            pkv.state_checkpoint(src_d, slots, pool, dev_status=status)
            back.copy_(pool[int(slots[0])], non_blocking=True)
            stream.synchronize()
            if i >= args.warmup:
                e2e.append(time.perf_counter() - t0)
    e2e_s = max_over_ranks(statistics.mean(e2e), dev)
    pk = peaks()
    if rank != 0:
        return
    line = {
        "metric": "state-row checkpoint: GB/s (bytes read + written) vs peak on 1 GB300",
        "value": job_throughput(nbytes / 1e9, ws, ms * 1e-3), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded random bytes)",
        "config": {"workload": "state_checkpoint", "pool_slots": STATE_POOL_SLOTS,
                   "row_bytes": STATE_ROW_BYTES, "rows_per_call": STATE_ROWS_PER_CALL,
                   "l2": f"flushed before every timed call ({L2_FLUSH_BYTES >> 20} MB written, then read)",
                   "timing": "CUDA graph replay per call, event nodes around the kernel"},
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "kernel": "state_checkpoint_kernel", "achieved": gbs,
                     "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                     "traffic": recorded_traffic("state_checkpoint_kernel", "state_checkpoint"),
                     "bytes_per_launch": nbytes, "ms_per_launch": ms, "peak_source": pk["source"]},
        "e2e": {"value": job_throughput(nbytes / 1e9, ws, e2e_s), "unit": "GB/s",
                "h2d_bytes_per_step": src_h.numel(), "d2h_bytes_per_step": back.numel(),
                "ms_per_step": e2e_s * 1e3},
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--config", default=HEADLINE,
                    choices=list(workloads.CONFIGS) + ["state_checkpoint"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", action="store_true",
                    help="time the named workload alone (no per-configuration summary)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.config == "state_checkpoint":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the state checkpoint has no "
                              "oracle arm in the benchmark (its parity tests use the oracle)"}))
            return
        bench_state_checkpoint(args)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_pkv(args)


if __name__ == "__main__":
    main()
