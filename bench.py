"""Benchmark one packed paged-attention step (KV append + attention) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl pkv|reference] [--config NAME]

A step is one pass of the whole path over one synthetic batch: KV append of
the step's new tokens, split-KV attention and its LSE merge, and the
tensor-core prefill tiles when present.  The step plan (host step metadata) is
an input like the block tables: resident in HBM for `value`, computed and
uploaded per step inside `e2e`.

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
  plus the gathered shared-prefix pairs.
* e2e: the same metric through the public API from pinned HOST buffers: every
  step copies q, the new K/V, slot mapping and metadata host->device (two pinned
  buffers, one transfer each), plans on the host into pinned memory and uploads
  the plan asynchronously, runs append + attention and copies out back (wall
  time per step).
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
            "config": {"workload": meta.name, **workloads.describe(meta)},
            "cpu_baseline": {k: r[k] for k in ("value", "unit", "cores", "kind", "sample")},
            "e2e": {"value": v, "unit": "KV tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    line["cpu_baseline"]["value"] = v
    print(json.dumps(line), flush=True)


def bench_pkv(args):
    import torch
    import paged_kv_attention_append_gb300 as pkv

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    meta = workloads.make_config(args.config)
    # a chained workload runs nch decode steps per timed unit (one graph), with
    # the contexts and slots moved on by the device between steps
    nch = workloads.chain_steps(meta)
    metas = [workloads.chain_step(meta, meta.context_lens, t) for t in range(nch)]
    q, k, v, pool = workloads.make_values(meta, device=dev)
    vals = [(q, k, v)] + [tuple(workloads.make_values(m, seed=meta.seed + t, device=dev)[:3])
                          for t, m in enumerate(metas) if t > 0]
    slots0 = torch.from_numpy(meta.slot_mapping).to(dev)
    slots = slots0.clone()
    cu_d = torch.from_numpy(meta.cu_q_lens).to(dev)
    ctx0_d = torch.from_numpy(meta.context_lens).to(dev)
    ctx_d = ctx0_d.clone()
    bt_d = torch.from_numpy(meta.block_tables).to(dev)
    outs = [torch.empty_like(x[0]) for x in vals]
    out = outs[0]
    flush_w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_acc = torch.zeros((), dtype=torch.float32, device=dev)

    def flush_l2():
        flush_w.zero_()                          # write more than L2 holds ...
        torch.sum(flush_r, dim=0, out=flush_acc)  # ... then read more, leaving clean lines
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    chain_arg = nch if nch > 1 else None
    info, host_plan = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, pool,
                                    upload=False, chain_steps=chain_arg,
                                    block_tables=meta.block_tables)
    t0 = time.perf_counter()
    for _ in range(50):
        pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, pool, upload=False,
                      chain_steps=chain_arg, block_tables=meta.block_tables)
    host_plan_us = (time.perf_counter() - t0) / 50 * 1e6
    plan = pkv.StepPlan(info, host_plan, dev)

    def step():
        # the plan is a step input like the block tables: uploaded before the timed
        # region (StepPlan); host planning and its upload are timed inside e2e
        if nch > 1:
            ctx_d.copy_(ctx0_d)
            slots.copy_(slots0)
        for t, (qt, kt, vt) in enumerate(vals):
            pkv.paged_kv_append(kt, vt, slots, pool, dev_status=status)
            pkv.paged_varlen_attention(qt, cu_d, ctx_d, bt_d, pool, meta.scale, plan=plan,
                                       out=outs[t], dev_status=status)
            if t + 1 < nch:
                pkv.decode_advance(ctx_d, slots, cu_d, bt_d, pool, dev_status=status)

    # warm up eagerly, then capture one step into a CUDA graph
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            step()
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    launches_before = pkv.kernel_launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    launches_per_step = pkv.kernel_launch_count() - launches_before
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
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            for a, b in ev:
                flush_l2()
                a.record(stream)
                graph.replay()
                b.record(stream)
        torch.cuda.synchronize(dev)
        # kernel-only timing (roofline): the library records our events around each
        # launch; captured into a second graph they are event nodes beside the
        # kernels, so an interval holds the kernel and no host launch gap.  L2 is
        # flushed before every replay, as for the step.
        present = {"append": True, "decode": info.num_decode_warps > 0,
                   "merge": info.num_merge_groups > 0, "prefill": info.num_prefill_tiles > 0}
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
                    step()
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
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    kern_ms = {n: (statistics.mean(samples[n]) if present[n] else 0.0) for n in k_ev}
    decode_ms, prefill_ms = kern_ms["decode"], kern_ms["prefill"]
    clocks = clk.summary()
    step_ms = max_over_ranks(step_ms, dev)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    # warm: the same step replayed back to back without the L2 flush (the
    # flushed figure above is the headline)
    ev_w = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        graph.replay()
        for a, b in ev_w:
            a.record(stream)
            graph.replay()
            b.record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev_w) / args.steps, dev)

    # ---- end to end from pinned host buffers through the public API (a chained
    # workload: all its steps' inputs in, one plan, every step's output back).  The
    # step's host inputs sit in two pinned buffers -- the int32 metadata (slots,
    # cu_q_lens, context_lens, block tables) and every step's bf16 q/k/v -- each
    # copied in one transfer; the plan is written straight into pinned memory and
    # uploaded asynchronously.
    def packed(parts):
        """One pinned host byte buffer holding `parts` (any dtypes, each start
        16-byte aligned), the matching device buffer, and the device and host
        views of each part."""
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

    # the step's int32 metadata, every step's bf16 q/k/v and, last, the plan
    # (written by the host planner each step) share one pinned buffer, so one
    # copy carries all of them
    plan_words = ((int(info.plan_bytes) + 4095) // 4096 + 1) * 1024
    qkv_parts = [x for qkv in vals for x in qkv]
    buf_h, buf_d, dviews, hviews = packed(
        [slots0, cu_d, ctx0_d, bt_d] + qkv_parts + [torch.zeros(plan_words, dtype=torch.int32)])
    ds, dcu, dctx, dbt = dviews[:4]
    dplan = dviews[-1]
    cu_h, ctx_h, bt_h, plan_hv = hviews[1], hviews[2], hviews[3], hviews[-1]
    plan_off = plan_hv.data_ptr() - buf_h.data_ptr()          # bytes, 16-byte aligned
    qkv_dv = dviews[4:-1]
    dvals = [tuple(qkv_dv[3 * t:3 * t + 3]) for t in range(len(vals))]
    cu_np, ctx_np, bt_np, plan_np = cu_h.numpy(), ctx_h.numpy(), bt_h.numpy(), plan_hv.numpy()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    outs_h = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    h2d = (plan_off + int(info.plan_bytes) + 15) // 16 * 16  # bytes copied per step
    # one copy after planning, or -- when the step's inputs are large enough for
    # their transfer to matter -- the inputs first, overlapping the planning,
    # then the plan
    split_copy = plan_off > (4 << 20)
    plan_e2e = pkv.StepPlan(info, host_plan, dev)
    plan_e2e.dev = dplan.view(torch.uint8)
    d2h = sum(o.numel() * o.element_size() for o in outs_h)
    e2e_times = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            if split_copy:  # large inputs go up while the host plans
                buf_d[:plan_off].copy_(buf_h[:plan_off], non_blocking=True)
            inf2, hp2 = pkv.plan_step(cu_np, ctx_np, meta.num_q_heads, pool, upload=False,
                                      chain_steps=chain_arg, block_tables=bt_np,
                                      num_sms=num_sms, out=plan_np)
            n = (plan_off + hp2.nbytes + 15) // 16 * 16
            n0 = plan_off if split_copy else 0
            buf_d[n0:n].copy_(buf_h[n0:n], non_blocking=True)
            plan_e2e.info = inf2
            for t, (dq, dk, dv) in enumerate(dvals):
                pkv.paged_kv_append(dk, dv, ds, pool, dev_status=status)
                pkv.paged_varlen_attention(dq, dcu, dctx, dbt, pool, meta.scale, plan=plan_e2e,
                                           out=outs[t], dev_status=status)
                if t + 1 < nch:
                    pkv.decode_advance(dctx, ds, dcu, dbt, pool, dev_status=status)
            for oh, o in zip(outs_h, outs):
                oh.copy_(o, non_blocking=True)
            stream.synchronize()
            if i >= args.warmup:
                e2e_times.append(time.perf_counter() - t0)
    e2e_s = max_over_ranks(statistics.mean(e2e_times), dev)

    pk = peaks()
    kv_tok = sum(m.kv_tokens() for m in metas)          # over the chain's steps
    bytes_alg = sum(algorithmic_bytes(m) for m in metas)
    # kernel events keep the last launch of a chain: its step's bytes (the plan
    # of a chain is sized for its last step)
    dec_bytes = decode_kernel_bytes(metas[-1], info)
    # tensor-core work: prefill-class sequences and gathered shared-prefix rows
    fl = prefill_flops(meta) + 4 * meta.head_dim * int(info.gather_pairs)
    kernels = {"append_kernel": {"ms_per_launch": kern_ms["append"]}}
    if kern_ms["merge"]:
        kernels["merge_kernel"] = {"ms_per_launch": kern_ms["merge"]}
    if decode_ms:
        kernels["decode_kernel"] = {"ms_per_launch": decode_ms, "bytes_per_launch": dec_bytes,
                                    "gbs": dec_bytes / (decode_ms * 1e-3) / 1e9}
    if prefill_ms:
        kernels["prefill_kernel"] = {"ms_per_launch": prefill_ms, "flops_per_launch": fl,
                                     "tflops": fl / (prefill_ms * 1e-3) / 1e12}
    if prefill_ms > decode_ms:     # the dominant kernel is a dense contraction
        achieved = fl / (prefill_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": "prefill_kernel", "achieved": achieved,
                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                    "traffic": recorded_traffic("prefill_kernel", meta.name), "flops_per_launch": fl, "ms_per_launch": prefill_ms,
                    "peak_source": pk["source"] + " (bf16 burst)"}
    else:
        achieved = dec_bytes / (decode_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved,
                    "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                    "traffic": recorded_traffic("decode_kernel", meta.name), "bytes_per_launch": dec_bytes, "ms_per_launch": decode_ms,
                    "peak_source": pk["source"]}
    cpu = cpu1 = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = run_oracle_sample(meta)                                   # all host cores
        cpu1 = run_oracle_sample(meta, target_s=3.0, num_threads=1)     # one core
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": job_throughput(kv_tok, ws, step_ms * 1e-3), "unit": "KV tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shapes of the named workload)",
        "config": {**workloads.describe(meta), **({"chain_steps": nch} if nch > 1 else {}),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single",
                   "l2": f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MB written, then "
                         f"{L2_FLUSH_BYTES >> 20} MB read)",
                   "timing": "CUDA graph replay per step, CUDA events per step; kernel "
                             "intervals from event nodes captured around each kernel "
                             "(second graph, no programmatic launch)"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roofline,
        "kernels": kernels,
        "step_gbs": bytes_alg / (step_ms * 1e-3) / 1e9,
        "warm": {"value": job_throughput(kv_tok, ws, warm_ms * 1e-3), "ms_per_step": warm_ms,
                 "l2": "not flushed: the step replayed back to back"},
        "host_plan_us": host_plan_us,
        "e2e": {"value": job_throughput(kv_tok, ws, e2e_s), "unit": "KV tokens/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3},
        "clocks": clocks,
        "cpu_baseline": None if cpu is None else {
            **{k2: cpu[k2] for k2 in ("value", "unit", "cores", "kind", "sample")},
            "value_1core": cpu1["value"], "sample_1core": cpu1["sample"]},
        "plan": {"decode_warps": info.num_decode_warps, "decode_pieces": info.num_decode_pieces,
                 "merge_groups": info.num_merge_groups, "prefill_tiles": info.num_prefill_tiles,
                 "shared_prefix_ctas": info.num_shared_ctas,
                 "gathered_rows": info.num_gather_rows * (meta.num_q_heads // meta.num_kv_heads)},
    }
    if meta.unique_blocks() * 16 < kv_tok and decode_ms:
        line["unique_gbs"] = unique_bytes(meta) / (decode_ms * 1e-3) / 1e9
    if fl:
        line["prefill_tflops_step"] = fl / (step_ms * 1e-3) / 1e12
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
    ap.add_argument("--config", default="small_decode",
                    choices=list(workloads.CONFIGS) + ["state_checkpoint"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
