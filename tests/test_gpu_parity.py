"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle.

Bars: KV append bit-exact over the whole pool; attention within max-abs 2e-2 and
mean-abs 2e-3 of the oracle (bf16 output, fp32 accumulation), and within the
bf16-floor bar of tests/parity_bar.py on every compared element (the bar that
sees a dropped block of keys at long context).  Every call through gpu_step
also checks guard bands: canary rows before and after `out`, and canary bytes
before and after the workspace, must be unchanged.
"""

import numpy as np
import pytest
import torch

import oracle
import parity_bar
import workloads

pytestmark = pytest.mark.gpu

MAX_ABS = parity_bar.MAX_ABS
MEAN_ABS = parity_bar.MEAN_ABS
OUT_GUARD_ROWS = 3
OUT_CANARY = 0x7FC1            # a bf16 NaN no kernel writes
WS_GUARD_BYTES = 4096          # keeps the workspace 256-byte aligned
WS_CANARY = 0xA5


@pytest.fixture(scope="module")
def pkv(cuda_device):
    import paged_kv_attention_append_gb300 as m
    m.build()
    return m


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def guarded_out(shape, dev):
    """An output tensor inside a buffer with canary rows on both sides."""
    buf = torch.full((shape[0] + 2 * OUT_GUARD_ROWS, *shape[1:]), OUT_CANARY,
                     dtype=torch.int16, device=dev).view(torch.bfloat16)
    return buf, buf[OUT_GUARD_ROWS:OUT_GUARD_ROWS + shape[0]]


def guarded_workspace(plan, dev):
    """Replace the plan's workspace by one inside a buffer with canary bytes on
    both sides (the workspace itself starts filled with canary bytes too: its
    contents on entry must not matter)."""
    n = int(plan.info.workspace_bytes)
    buf = torch.full((n + 2 * WS_GUARD_BYTES,), WS_CANARY, dtype=torch.uint8, device=dev)
    plan.workspace = buf[WS_GUARD_BYTES:WS_GUARD_BYTES + n]
    return buf


def check_guards(out_buf, ws_buf, what=""):
    g = OUT_GUARD_ROWS
    ob = out_buf.view(torch.int16)
    canary = torch.tensor(OUT_CANARY, dtype=torch.int16, device=ob.device)
    assert bool((ob[:g] == canary).all()) and bool((ob[ob.shape[0] - g:] == canary).all()), \
        f"{what}: a kernel wrote outside out"
    wb = ws_buf
    assert bool((wb[:WS_GUARD_BYTES] == WS_CANARY).all()) and \
        bool((wb[wb.shape[0] - WS_GUARD_BYTES:] == WS_CANARY).all()), \
        f"{what}: a kernel wrote outside the workspace"


def gpu_step(pkv, meta, q, k, v, pool, dev, *, num_sms=None, check_status=True, tables=True,
             prefill_min_q=None):
    """Append + attention on the GPU; returns (out bf16 cpu tensor, pool after, status).
    tables=True plans with the host block tables (first block ids in the plan,
    shared-prefix CTAs where sequences share leading blocks).  out and the
    workspace sit between guard bands that are checked after the call."""
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    pd = pool.to(dev) if pool.device != dev else pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_kv_append(kd, vd, torch.from_numpy(meta.slot_mapping).to(dev), pd, dev_status=status)
    plan = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, pd, num_sms=num_sms,
                         block_tables=meta.block_tables if tables else None,
                         prefill_min_q=prefill_min_q)
    ws_buf = guarded_workspace(plan, dev)
    out_buf, out = guarded_out(tuple(qd.shape), dev)
    pkv.paged_varlen_attention(qd, meta.cu_q_lens, meta.context_lens,
                               torch.from_numpy(meta.block_tables).to(dev), pd, meta.scale,
                               plan=plan, out=out, dev_status=status)
    torch.cuda.synchronize(dev)
    st = int(status.item())
    if check_status:
        assert st == 0, f"device status {st}: {pkv.DEV_STATUS.get(st)}"
        check_guards(out_buf, ws_buf, meta.name)
    return out.cpu(), pd, st


def assert_close(got_bf16, want, what=""):
    r = parity_bar.check(got_bf16, want, what, head_dim=want.shape[-1])
    return r["max_abs"], r["mean_abs"]


def sample_rows(meta, rng, n):
    total = meta.total_q * meta.num_q_heads
    rows = set(rng.choice(total, size=min(n, total), replace=False).tolist())
    # every sequence's first and last query token, all heads of one of them
    for s in range(meta.num_seqs):
        for t in (int(meta.cu_q_lens[s]), int(meta.cu_q_lens[s + 1]) - 1):
            if t >= int(meta.cu_q_lens[s]):
                rows.add(t * meta.num_q_heads + int(rng.integers(meta.num_q_heads)))
    return np.array(sorted(rows), dtype=np.int64)


def tile_rows(meta, rng, tile=128):
    """One random row of every (128-token tile, query head) of every sequence,
    plus each sequence's first and last token on every head."""
    rows = set()
    hq = meta.num_q_heads
    for s in range(meta.num_seqs):
        c0, c1 = int(meta.cu_q_lens[s]), int(meta.cu_q_lens[s + 1])
        for t0 in range(c0, c1, tile):
            t1 = min(c1, t0 + tile)
            for h in range(hq):
                rows.add(int(rng.integers(t0, t1)) * hq + h)
        if c1 > c0:
            for h in range(hq):
                rows.add(c0 * hq + h)
                rows.add((c1 - 1) * hq + h)
    return np.array(sorted(rows), dtype=np.int64)


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_append_bit_exact_full_size(pkv, cuda_device, name):
    meta = workloads.make_config(name)
    big = name in ("high_conc_decode", "long_context_mix")
    q, k, v, pool = workloads.make_values(meta, device=cuda_device if big else "cpu")
    pool_host = pool.cpu()
    want, bad = oracle.paged_kv_append(pool_host, k.cpu(), v.cpu(), meta.slot_mapping, block_size=16)
    assert bad == 0
    pd = pool.to(cuda_device) if not big else pool
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.paged_kv_append(k.to(cuda_device), v.to(cuda_device),
                        torch.from_numpy(meta.slot_mapping).to(cuda_device), pd, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(pd), want)


def test_append_padding_and_bad_slot_reported(pkv, cuda_device):
    meta = workloads.tiny_decode()
    q, k, v, pool = workloads.make_values(meta)
    slots = meta.slot_mapping.copy()
    slots[1] = -1
    slots[2] = meta.num_blocks * 16 + 5
    want, bad = oracle.paged_kv_append(pool, k, v, slots, block_size=16)
    assert bad == 1
    pd = pool.to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.paged_kv_append(k.to(cuda_device), v.to(cuda_device), torch.from_numpy(slots).to(cuda_device),
                        pd, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert np.array_equal(bits(pd), want)


# ------------------------------------------------------------------ attention, full oracle

@pytest.mark.parametrize("name", ["tiny_decode", "small_decode", "shared_prefix_verify", "mtp_draft",
                                  "wide_verify"])
def test_attention_matches_oracle_every_row(pkv, cuda_device, name):
    meta = workloads.make_config(name)
    q, k, v, pool = workloads.make_values(meta)
    want, pool_want = oracle.run_step(meta, q, k, v, pool)
    out, pd, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
    assert np.array_equal(bits(pd), pool_want)
    assert_close(out, want, f"{name} (every row)")


@pytest.mark.parametrize("seed", range(16))
def test_attention_random_mixed_steps(pkv, cuda_device, seed):
    rng = np.random.default_rng(1000 + seed)
    meta = workloads.random_step(rng, max_ctx=int(rng.choice([40, 300, 1500])))
    q, k, v, pool = workloads.make_values(meta)
    want, _ = oracle.run_step(meta, q, k, v, pool)
    out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device,
                         num_sms=int(rng.choice([1, 8, 152])))
    assert_close(out, want, f"seed {seed}")


# ------------------------------------------------------------------ attention, full size

@pytest.mark.parametrize("name", ["agent_mixed", "high_conc_decode"])
def test_attention_full_size_every_row(pkv, cuda_device, name):
    """The mixed step (a 2048-token chunk beside three decodes) and the
    high-concurrency step (256 decodes, 3.4 GB of KV), inputs drawn on the GPU,
    in the launch configuration the benchmark times; every output row against
    the oracle."""
    meta = workloads.make_config(name)
    q, k, v, pool = workloads.make_values(meta, device=cuda_device)
    qh, kh, vh, ph = q.cpu(), k.cpu(), v.cpu(), pool.cpu()
    out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
    del pool
    want, _ = oracle.run_step(meta, qh, kh, vh, ph)
    assert_close(out, want, f"{name} (every row)")


@pytest.mark.parametrize("name", ["shared_prefix_verify", "small_decode", "long_context_mix"])
def test_attention_full_size_sampled_rows(pkv, cuda_device, name):
    """Full-size steps with inputs drawn on the GPU.  The long-context step
    (30 000 + 5 000 + 10 prefill rows, ~9.5 TFLOP) is beyond the oracle row by
    row, so one random row of every (128-token tile, query head) is checked,
    plus every head of each sequence's first and last token."""
    meta = workloads.make_config(name)
    q, k, v, pool = workloads.make_values(meta, device=cuda_device)
    qh, kh, vh, ph = q.cpu(), k.cpu(), v.cpu(), pool.cpu()
    out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
    rng = np.random.default_rng(5)
    rows = tile_rows(meta, rng) if name == "long_context_mix" else sample_rows(meta, rng, 3000)
    want, _ = oracle.run_step(meta, qh, kh, vh, ph, rows=rows)
    got = out.view(-1, meta.head_dim)[torch.from_numpy(rows)]
    assert_close(got, want, f"{name} ({len(rows)} rows)")


# ------------------------------------------------------------------ invariants on the GPU

def test_split_count_invariance(pkv, cuda_device):
    meta = workloads.small_decode()
    q, k, v, pool = workloads.make_values(meta)
    a, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, num_sms=1)      # one split each
    b, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, num_sms=1000)   # many splits
    diff = (a.double() - b.double()).abs()
    assert float(diff.max()) <= 2e-2 and float(diff.mean()) <= 2e-3


def test_block_permutation_is_bitwise_invariant(pkv, cuda_device):
    rng = np.random.default_rng(3)
    meta = workloads.random_step(rng, num_seqs=5, max_ctx=700)
    q, k, v, pool = workloads.make_values(meta)
    a, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
    perm = rng.permutation(meta.num_blocks)
    pool2 = torch.empty_like(pool)
    pool2[torch.from_numpy(perm)] = pool
    tables2 = np.where(meta.block_tables >= 0, perm[np.maximum(meta.block_tables, 0)], -1).astype(np.int32)
    meta2 = workloads.StepMeta(**{**meta.__dict__, "block_tables": tables2,
                                  "slot_mapping": (perm[meta.slot_mapping // 16] * 16 +
                                                   meta.slot_mapping % 16).astype(np.int32)})
    b, _, _ = gpu_step(pkv, meta2, q, k, v, pool2, cuda_device)
    assert torch.equal(a, b)


def test_constant_v_and_single_key(pkv, cuda_device):
    meta = workloads.build_step("t", 9, [1, 1, 3], [1, 200, 3], 8, 2, 128, pool_blocks=30)
    q, k, v, pool = workloads.make_values(meta)
    want, _ = oracle.run_step(meta, q, k, v, pool)
    out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
    assert_close(out, want)
    # a single visible key returns its V exactly (weight 1, one bf16 rounding of an exact value)
    assert torch.equal(out[0].float(), v[0].repeat_interleave(4, dim=0).float())
    vv = v.clone()
    vv[:] = 0.375
    pool_c = pool.clone()
    pool_c[:, 1] = 0.375
    out2, _, _ = gpu_step(pkv, meta, q, k, vv, pool_c, cuda_device)
    assert torch.all(out2.float() == 0.375)


def test_edge_shapes(pkv, cuda_device):
    cases = [
        ([1], [1], 16, 1, 128),          # group 16, single key
        ([1], [32768], 32, 8, 128),      # longest context of the high-concurrency mix
        ([64], [64], 4, 4, 64),          # prefill from an empty cache (q_len = ctx)
        ([0, 2, 0, 1], [5, 48, 7, 16], 8, 2, 64),   # q_len 0 sequences, block-aligned ctx
        ([2] * 9, [17, 18, 31, 32, 33, 47, 48, 49, 2], 32, 8, 128),  # verify pairs on block edges
    ]
    for i, (ql, cl, hq, hkv, d) in enumerate(cases):
        meta = workloads.build_step("edge", 40 + i, ql, cl, hq, hkv, d)
        q, k, v, pool = workloads.make_values(meta)
        want, _ = oracle.run_step(meta, q, k, v, pool)
        out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
        assert_close(out, want, f"edge case {i}")


def test_empty_step_is_a_no_op(pkv, cuda_device):
    pool = torch.zeros(4, 2, 2, 16, 64, dtype=torch.bfloat16, device=cuda_device)
    q = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device=cuda_device)
    before = pkv.kernel_launch_count()
    out = pkv.paged_varlen_attention(q, np.array([0], np.int32), np.array([], np.int32),
                                     torch.zeros(0, 1, dtype=torch.int32, device=cuda_device), pool, 0.1)
    assert out.shape == (0, 4, 64) and pkv.kernel_launch_count() == before


def test_bad_block_id_is_reported_not_faulted(pkv, cuda_device):
    meta = workloads.build_step("t", 12, [1, 1], [100, 60], 8, 2, 128, pool_blocks=20)
    q, k, v, pool = workloads.make_values(meta)
    tables = meta.block_tables.copy()
    tables[0, 3] = meta.num_blocks + 7      # outside the pool
    bad = workloads.StepMeta(**{**meta.__dict__, "block_tables": tables})
    out, _, st = gpu_step(pkv, bad, q, k, v, pool, cuda_device, check_status=False)
    assert st == 2
    # the other sequence is unaffected
    want, _ = oracle.run_step(meta, q, k, v, pool)
    assert_close(out[1:], want[1:])


def test_attention_on_a_side_stream_with_host_arrays(pkv, cuda_device):
    """The call runs on a non-default stream with host cu_q_lens / context_lens /
    block tables: the arrays it copies to the device and the output it
    allocates belong to that stream, so the result read after syncing that
    stream alone matches the oracle."""
    meta = workloads.build_step("side", 61, [1, 3, 130], [700, 90, 400], 8, 2, 128)
    q, k, v, pool = workloads.make_values(meta)
    want, pool_want = oracle.run_step(meta, q, k, v, pool)
    dev = cuda_device
    pd = torch.from_numpy(pool_want.view(np.int16)).view(torch.bfloat16).to(dev)
    s = torch.cuda.Stream(dev)
    qd = q.to(dev)
    torch.cuda.synchronize(dev)
    outs = []
    for _ in range(3):      # temporaries freed between calls may be reused by the next
        outs.append(pkv.paged_varlen_attention(qd, meta.cu_q_lens, meta.context_lens,
                                               meta.block_tables, pd, meta.scale, stream=s))
    s.synchronize()
    for o in outs:
        assert_close(o.cpu(), want, "side stream")


def test_bound_step_matches_the_plain_calls(pkv, cuda_device):
    """A BoundStep (arguments checked once, replayed per step) gives the same
    pool and output bits as the plain append + attention calls, across two
    steps whose plans differ (a new plan summary each run)."""
    dev = cuda_device
    meta = workloads.build_step("bound", 71, [1, 2, 1], [300, 900, 45], 16, 4, 128)
    q, k, v, pool = workloads.make_values(meta)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    cu = torch.from_numpy(meta.cu_q_lens).to(dev)
    ctx = torch.from_numpy(meta.context_lens).to(dev)
    bt = torch.from_numpy(meta.block_tables).to(dev)
    sl = torch.from_numpy(meta.slot_mapping).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pa, pb = pool.to(dev), pool.to(dev)
    plan = pkv.plan_step(meta.cu_q_lens, meta.context_lens, 16, pa, block_tables=meta.block_tables)
    ref = [None, None]
    out_b = torch.empty_like(qd)
    b = pkv.BoundStep(kd, vd, sl, qd, cu, ctx, bt, pb, meta.scale, plan, out_b, dev_status=status)
    for step, sms in enumerate((152, 5)):      # the second step has another plan
        p2 = pkv.plan_step(meta.cu_q_lens, meta.context_lens, 16, pa, num_sms=sms,
                           block_tables=meta.block_tables)
        pkv.paged_kv_append(kd, vd, sl, pa, dev_status=status)
        ref[step] = pkv.paged_varlen_attention(qd, cu, ctx, bt, pa, meta.scale, plan=p2,
                                               dev_status=status)
        plan.info, plan.dev, plan.workspace = p2.info, p2.dev, p2.workspace
        b.run()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out_b, ref[step]) and torch.equal(pa, pb)


def test_bound_copies_and_planner_serve_a_step_from_host_buffers(pkv, cuda_device):
    """The serving loop through the library alone: pinned inputs go up with one
    bound copy, the plan is made by the bound planner on its own thread (while
    the copy and the append are queued) into the same pinned buffer and goes up
    behind them, the bound step runs and a bound copy brings
    out back.  The result has the bits of the plain calls, and copy_async moves
    bytes both ways unchanged."""
    dev = cuda_device
    g = torch.Generator().manual_seed(3)
    src = torch.randint(0, 255, (12345,), dtype=torch.uint8, generator=g).pin_memory()
    mid = torch.empty(12345, dtype=torch.uint8, device=dev)
    back = torch.zeros(12345, dtype=torch.uint8).pin_memory()
    pkv.copy_async(mid, src)
    pkv.copy_async(back, mid, 12000)
    torch.cuda.synchronize()
    assert torch.equal(back[:12000], src[:12000]) and int(back[12000:].sum()) == 0

    meta = workloads.build_step("serve", 72, [1, 2, 1, 1], [300, 900, 45, 2000], 16, 4, 128)
    q, k, v, pool = workloads.make_values(meta)
    parts = [torch.from_numpy(meta.slot_mapping), torch.from_numpy(meta.cu_q_lens),
             torch.from_numpy(meta.context_lens), torch.from_numpy(meta.block_tables), q, k, v,
             torch.zeros(1 << 15, dtype=torch.int32)]
    offs, n = [], 0
    for t in parts:
        offs.append(n)
        n += (t.numel() * t.element_size() + 15) // 16 * 16
    hbuf = torch.zeros(n, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(n, dtype=torch.uint8, device=dev)
    hv, dv = [], []
    for t, o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        h = hbuf[o:o + nb].view(t.dtype).view(t.shape)
        h.copy_(t)
        hv.append(h)
        dv.append(dbuf[o:o + nb].view(t.dtype).view(t.shape))
    ds, dcu, dctx, dbt, dq, dk, dvv, dplan = dv
    pool_a, pool_b = pool.to(dev), pool.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    planner = pkv.BoundPlan(hv[1].numpy(), hv[2].numpy(), 16, pool_b, hv[-1].numpy(),
                            block_tables=hv[3].numpy(), spin_us=500)
    info, plan_nb = planner.run()
    plan = pkv.StepPlan(info, hv[-1].numpy().view(np.uint8)[:plan_nb].view(np.int32), dev)
    plan.dev = dplan.view(torch.uint8)
    out_b = torch.empty_like(dq)
    out_h = torch.empty(out_b.shape, dtype=out_b.dtype).pin_memory()
    up = pkv.BoundCopy(dbuf, hbuf)
    down = pkv.BoundCopy(out_h, out_b)
    step = pkv.BoundStep(dk, dvv, ds, dq, dcu, dctx, dbt, pool_b, meta.scale, plan, out_b,
                         dev_status=status)
    hv[-1].zero_()
    planner.post()                   # planned on the library's thread meanwhile:
    up.run(offs[-1])                 # the inputs, then the append (it needs no plan)
    step.run_append()
    info2, plan_nb = planner.wait()
    assert info2.plan_bytes == info.plan_bytes
    up.run(plan_nb, offs[-1])        # the plan behind them
    step.run_attention()
    down.run()
    torch.cuda.synchronize()
    pkv.paged_kv_append(k.to(dev), v.to(dev), torch.from_numpy(meta.slot_mapping).to(dev), pool_a)
    ref = pkv.paged_varlen_attention(q.to(dev), meta.cu_q_lens, meta.context_lens,
                                     torch.from_numpy(meta.block_tables).to(dev), pool_a,
                                     meta.scale, plan=pkv.plan_step(
                                         meta.cu_q_lens, meta.context_lens, 16, pool_a,
                                         block_tables=meta.block_tables))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out_h, ref.cpu()) and torch.equal(pool_a, pool_b)


def test_in_tree_library_is_loaded(pkv):
    import os
    assert os.path.exists(pkv.library_path())
    maps = open("/proc/self/maps").read()
    assert pkv.library_path() in maps


# ------------------------------------------------------------------ tensor-core prefill path

@pytest.mark.parametrize("ql,cl,hq,hkv,d", [
    ([128], [128], 1, 1, 128),                  # one exact tile, prefill from an empty cache
    ([64], [64], 2, 1, 64),                     # D = 64, group 2
    ([200], [700], 5, 1, 128),                  # ragged tile, context before the chunk
    ([130, 1, 300], [900, 50, 301], 8, 2, 128), # prefill + decode in one step
    ([256], [4096 + 256], 4, 1, 128),           # long context, several key tiles
])
def test_prefill_kernel_matches_oracle(pkv, cuda_device, ql, cl, hq, hkv, d):
    meta = workloads.build_step("prefill", 77 + len(ql), ql, cl, hq, hkv, d)
    q, k, v, pool = workloads.make_values(meta)
    plan_info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, hq, pkv.pool_desc(pool),
                                 upload=False)
    assert plan_info.num_prefill_tiles > 0
    want, _ = oracle.run_step(meta, q, k, v, pool)
    out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
    assert_close(out, want, f"prefill {ql} {cl}")


@pytest.mark.parametrize("d", [128, 64])
def test_prefill_rescales_when_scores_grow_along_the_keys(pkv, cuda_device, d):
    """Scores that grow from one 128-key tile to the next by more than 2^8 (in
    the exponent's log2 units) make every row's running max jump at each tile,
    so the tensor-core softmax takes its rescale path (O and l rescaled, the
    tile's exponentials redone) on every tile after the first; the result
    still matches the oracle."""
    meta = workloads.build_step("grow", 131, [640], [640], 4, 2, d)   # prefill from empty, 5 key tiles
    q, k, v, pool = workloads.make_values(meta)
    g = torch.Generator().manual_seed(5)
    q.copy_((1.0 + 0.1 * torch.randn(q.shape, generator=g)).to(torch.bfloat16))
    tile = (torch.arange(meta.total_q) // 128).to(torch.float32)
    # score of key p for any row: about scale * D * 0.9 * tile(p) -> +(0.9 * sqrt(D) / ln 2) log2 units per tile (> 10)
    k.copy_((0.9 * tile[:, None, None] + 0.3 * torch.randn(k.shape, generator=g)).to(torch.bfloat16))
    plan_info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads,
                                 pkv.pool_desc(pool), upload=False)
    assert plan_info.num_prefill_tiles > 0
    want, _ = oracle.run_step(meta, q, k, v, pool)
    out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
    assert_close(out, want, f"growing scores D={d}")


def test_prefill_and_split_kv_paths_agree(pkv, cuda_device):
    meta = workloads.build_step("paths", 91, [300, 2, 1], [1000, 500, 40], 8, 2, 128)
    q, k, v, pool = workloads.make_values(meta)
    tc_out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device)
    info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, 8, pkv.pool_desc(pool), upload=False,
                            prefill_min_q=-1)   # every row on the split-KV kernel
    assert info.num_prefill_tiles == 0
    kv_out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, prefill_min_q=-1)
    diff = (tc_out.double() - kv_out.double()).abs()
    assert float(diff.max()) <= MAX_ABS and float(diff.mean()) <= MEAN_ABS


@pytest.mark.parametrize("num_sms", [1, 5, 7, 19])
def test_prefill_split_kv_and_persistent_items_match_oracle(pkv, cuda_device, num_sms):
    """Persistent prefill CTAs: with few SMs one CTA runs many work items in a
    row (barrier phases carried across items); with an odd split of the work the
    leftover query tiles are cut along their keys into partials that the merge
    kernel combines.  Every row is checked against the oracle."""
    meta = workloads.build_step("split_prefill", 123 + num_sms, [384, 1, 200], [3000, 700, 900],
                                8, 2, 128)
    q, k, v, pool = workloads.make_values(meta)
    info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, 8, pkv.pool_desc(pool),
                            num_sms=num_sms, upload=False)
    # the persistent CTAs take the SMs the split-KV work leaves (at least one)
    assert 1 <= info.num_prefill_ctas <= min(num_sms, info.num_prefill_tiles)
    if num_sms in (7, 19):
        assert info.num_prefill_merges > 0      # some query tiles are cut along their keys
    want, _ = oracle.run_step(meta, q, k, v, pool)
    out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, num_sms=num_sms)
    assert_close(out, want, f"split prefill on {num_sms} SMs")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("num_sms", [1, 3, 152])
def test_prefill_whole_sub_tiles_short_passes_match_oracle(pkv, cuda_device, d, num_sms):
    """Whole 128-token sub-tiles leave the tensor-core kernel through a V-ring
    slot and a bulk tensor store, ragged ones row by row.  Passes of one to
    three key tiles, many of them on one CTA (one or three SMs), put the
    output's staging slots next to one another in the ring.  Every row of the
    step (whole, ragged and decode) is checked against the oracle; out starts
    as NaN canaries, so a row left unwritten fails, and the guard rows around
    out show any store past its ends."""
    ql = [128, 128, 256, 128, 200, 128, 1]
    cl = [128, 200, 256, 300, 260, 384, 90]
    meta = workloads.build_step("whole_tiles", 17 + d + num_sms, ql, cl, 8, 2, d)
    q, k, v, pool = workloads.make_values(meta)
    info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, 8, pkv.pool_desc(pool),
                            num_sms=num_sms, upload=False)
    assert info.num_prefill_tiles > 0
    want, _ = oracle.run_step(meta, q, k, v, pool)
    out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, num_sms=num_sms)
    assert_close(out, want, f"whole sub-tiles D={d} on {num_sms} SMs")


# ------------------------------------------------------------------ state-row checkpoint

@pytest.mark.parametrize("num_slots,row_bytes,n", [
    (40, 16, 7),            # the smallest row
    (300, 4096, 64),        # many short rows
    (96, 1 << 20, 24),      # MiB rows, as in the page's state pools
    (8, 48, 0),             # nothing to write
])
def test_state_checkpoint_bit_exact(pkv, cuda_device, num_slots, row_bytes, n):
    rng = np.random.default_rng(row_bytes + n)
    pool = rng.integers(0, 256, size=(num_slots, row_bytes), dtype=np.uint8)
    src = rng.integers(0, 256, size=(n, row_bytes), dtype=np.uint8)
    slots = rng.permutation(num_slots)[:n].astype(np.int32)
    if n > 3:
        slots[1] = -1
    want, bad = oracle.state_checkpoint(pool, src, slots)
    assert bad == 0
    pd = torch.from_numpy(pool).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.state_checkpoint(torch.from_numpy(src).to(cuda_device), torch.from_numpy(slots).to(cuda_device),
                         pd, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(pd.cpu().numpy(), want)


def test_state_checkpoint_bad_slot_reported_and_skipped(pkv, cuda_device):
    rng = np.random.default_rng(11)
    pool = rng.integers(0, 256, size=(20, 64), dtype=np.uint8)
    src = rng.integers(0, 256, size=(3, 64), dtype=np.uint8)
    slots = np.array([5, 20, 7], dtype=np.int32)          # 20 is past the pool
    want, bad = oracle.state_checkpoint(pool, src, slots)
    assert bad == 1
    pd = torch.from_numpy(pool).to(cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkv.state_checkpoint(torch.from_numpy(src).to(cuda_device), torch.from_numpy(slots).to(cuda_device),
                         pd, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert np.array_equal(pd.cpu().numpy(), want)


def test_state_checkpoint_full_size_pool(pkv, cuda_device):
    """The page's pool size: about 1,650 cached blocks of ~1 MiB state rows
    (~1.6 GiB); 64 rows written, checked row by row, other rows unchanged."""
    num_slots, row_bytes, n = 1650, 1 << 20, 64
    g = torch.Generator(device=cuda_device).manual_seed(5)
    pool = torch.randint(0, 256, (num_slots, row_bytes), dtype=torch.uint8, device=cuda_device,
                         generator=g)
    before = pool.clone()
    src = torch.randint(0, 256, (n, row_bytes), dtype=torch.uint8, device=cuda_device, generator=g)
    slots = torch.randperm(num_slots, device=cuda_device, generator=g)[:n].to(torch.int32)
    pkv.state_checkpoint(src, slots, pool)
    torch.cuda.synchronize()
    written = torch.zeros(num_slots, dtype=torch.bool, device=cuda_device)
    written[slots.long()] = True
    assert torch.equal(pool[slots.long()], src)
    assert torch.equal(pool[~written], before[~written])


# ------------------------------------------------------------------ chained decode

def _chain_case(steps, seed=77, window=False):
    """A decode batch whose tables already hold the blocks of the chain's last step,
    and the per-step (context_lens, slot_mapping) the chain must go through.
    window: an 8-token verify window (two row groups: a shared-block item) rides
    along too."""
    ctx0 = np.array([15, 16, 17, 100, 31, 255, 2] + ([300] if window else []), dtype=np.int32)
    ql = np.array([1, 1, 1, 2, 1, 1, 1] + ([8] if window else []), dtype=np.int32)
    last = ctx0 + (steps - 1) * ql
    meta = workloads.build_step("chain", seed, ql, last, 8, 2, 128)
    per_step = []
    for t in range(steps):
        ctx = ctx0 + t * ql
        slots = []
        for s in range(len(ql)):
            for i in range(int(ql[s])):
                pos = int(ctx[s]) - int(ql[s]) + i
                slots.append(int(meta.block_tables[s, pos // 16]) * 16 + pos % 16)
        per_step.append(workloads.StepMeta(**{**meta.__dict__, "context_lens": ctx.astype(np.int32),
                                              "slot_mapping": np.array(slots, dtype=np.int32)}))
    return meta, per_step


@pytest.mark.parametrize("window", [False, True])
def test_decode_chain_matches_oracle_every_step(pkv, cuda_device, window):
    steps = 6
    meta, per_step = _chain_case(steps, window=window)
    _, _, _, pool = workloads.make_values(per_step[0])
    vals = [workloads.make_values(m, seed=500 + t)[:3] for t, m in enumerate(per_step)]
    # oracle: append then attend, step by step
    pool_o = pool
    want = []
    for m, (q, k, v) in zip(per_step, vals):
        out, pool_o = oracle.run_step(m, q, k, v, pool_o)
        want.append(out)
    # GPU: one chain plan, device-side advance between steps
    dev = cuda_device
    pd = pool.to(dev)
    cu = torch.from_numpy(meta.cu_q_lens).to(dev)
    ctx = torch.from_numpy(per_step[0].context_lens).to(dev)
    slots = torch.from_numpy(per_step[0].slot_mapping).to(dev)
    bt = torch.from_numpy(meta.block_tables).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    plan = pkv.plan_step(per_step[0].cu_q_lens, per_step[0].context_lens, 8, pd, chain_steps=steps)
    assert (plan.info.num_shared_ctas > 0) == window
    outs = []
    for t, (q, k, v) in enumerate(vals):
        pkv.paged_kv_append(k.to(dev), v.to(dev), slots, pd, dev_status=status)
        outs.append(pkv.paged_varlen_attention(q.to(dev), cu, ctx, bt, pd, meta.scale, plan=plan,
                                               dev_status=status))
        if t + 1 < steps:
            pkv.decode_advance(ctx, slots, cu, bt, pd, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(ctx.cpu().numpy(), per_step[-1].context_lens)
    assert np.array_equal(slots.cpu().numpy(), per_step[-1].slot_mapping)
    assert np.array_equal(bits(pd), pool_o)
    for t in range(steps):
        assert_close(outs[t].cpu(), want[t], f"chain step {t}")


def test_decode_chain_graph_replay_matches_eager(pkv, cuda_device):
    """The whole chain (append, attention, advance per step) captured once into a
    CUDA graph, with the first step's lengths restored at its start, replays to
    the same bits as the eager chain."""
    steps = 4
    meta, per_step = _chain_case(steps, seed=78)
    _, _, _, pool = workloads.make_values(per_step[0])
    dev = cuda_device
    vals = [tuple(x.to(dev) for x in workloads.make_values(m, seed=600 + t)[:3])
            for t, m in enumerate(per_step)]
    cu = torch.from_numpy(meta.cu_q_lens).to(dev)
    ctx0 = torch.from_numpy(per_step[0].context_lens).to(dev)
    slots0 = torch.from_numpy(per_step[0].slot_mapping).to(dev)
    bt = torch.from_numpy(meta.block_tables).to(dev)
    plan = pkv.plan_step(per_step[0].cu_q_lens, per_step[0].context_lens, 8, pool.to(dev),
                         chain_steps=steps)
    ctx, slots = ctx0.clone(), slots0.clone()
    outs = [torch.empty_like(v[0]) for v in vals]

    def chain(pd):
        ctx.copy_(ctx0)
        slots.copy_(slots0)
        for t, (q, k, v) in enumerate(vals):
            pkv.paged_kv_append(k, v, slots, pd)
            pkv.paged_varlen_attention(q, cu, ctx, bt, pd, meta.scale, plan=plan, out=outs[t])
            if t + 1 < steps:
                pkv.decode_advance(ctx, slots, cu, bt, pd)
    pd_e = pool.to(dev)
    chain(pd_e)
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    pd_g = pool.to(dev)
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        chain(pd_g)                          # warm-up on the capture stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain(pd_g)
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for t in range(steps):
        assert torch.equal(outs[t], eager[t])
    assert torch.equal(pd_g, pd_e)


def test_plan_with_block_tables_same_result_and_mismatch_reported(pkv, cuda_device):
    """A plan that carries the first block ids (from the host tables) gives the
    same bits as one that does not; host tables that disagree with the device
    copy are reported as a plan mismatch (the ids are range-checked first, so
    only in-pool blocks are read), and no output row is built from the blocks
    the plan named: every row is either left as it was or correct."""
    meta = workloads.small_decode()
    q, k, v, pool = workloads.make_values(meta)
    dev = cuda_device
    pd = pool.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.paged_kv_append(k.to(dev), v.to(dev), torch.from_numpy(meta.slot_mapping).to(dev), pd,
                        dev_status=status)
    bt = torch.from_numpy(meta.block_tables).to(dev)
    qd = q.to(dev)
    outs = []
    for tables in (None, meta.block_tables):
        plan = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, pd,
                             block_tables=tables)
        outs.append(pkv.paged_varlen_attention(qd, meta.cu_q_lens, meta.context_lens, bt, pd,
                                               meta.scale, plan=plan, dev_status=status))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(outs[0], outs[1])
    wrong = np.roll(meta.block_tables, 1, axis=0)          # other sequences' blocks
    plan = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, pd,
                         block_tables=wrong)
    out_buf, out = guarded_out(tuple(qd.shape), dev)
    pkv.paged_varlen_attention(qd, meta.cu_q_lens, meta.context_lens, bt, pd, meta.scale,
                               plan=plan, out=out, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 4      # PKV_DEV_PLAN_MISMATCH
    ob = out.view(torch.int16).cpu().reshape(-1, meta.head_dim)
    untouched = (ob == OUT_CANARY).all(dim=1).numpy()
    assert untouched.sum() > 0
    want, _ = oracle.run_step(meta, q, k, v, pool)
    got = out.cpu().reshape(-1, meta.head_dim)
    written = ~untouched
    if written.any():
        parity_bar.check(got[torch.from_numpy(written)], want.reshape(-1, meta.head_dim)[written],
                         "rows written under a plan mismatch")


@pytest.mark.parametrize("name,num_sms", [("shared_prefix_verify", 152), ("mtp_draft", 152),
                                          ("shared_prefix_verify", 7)])
def test_shared_prefix_ctas_match_oracle_and_per_warp_path(pkv, cuda_device, name, num_sms):
    """Sequences sharing leading blocks read them once per work unit (here the
    tensor-core gathered sub-tiles); the result matches the oracle on every row and
    the per-warp plan (no tables)."""
    meta = workloads.make_config(name)
    q, k, v, pool = workloads.make_values(meta)
    info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads,
                            pkv.pool_desc(pool), num_sms=num_sms, upload=False,
                            block_tables=meta.block_tables)
    assert info.num_gather_rows > 0
    want, _ = oracle.run_step(meta, q, k, v, pool)
    shared, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, num_sms=num_sms)
    per_warp, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, num_sms=num_sms, tables=False)
    assert_close(shared, want, f"{name} shared-prefix CTAs")
    diff = (shared.double() - per_warp.double()).abs()
    assert float(diff.max()) <= MAX_ABS and float(diff.mean()) <= MEAN_ABS


@pytest.mark.parametrize("seed,num_seqs,group,hkv,d,pre", [
    (0, 40, 1, 2, 128, 8), (1, 40, 2, 1, 64, 20), (2, 24, 4, 2, 128, 33), (3, 12, 8, 1, 64, 20),
    (4, 70, 1, 1, 128, 17), (5, 6, 2, 2, 128, 16)])
def test_shared_prefix_random_steps_match_oracle(pkv, cuda_device, seed, num_seqs, group, hkv, d, pre):
    """Random steps whose sequences share a prefix: gathered tensor-core sub-tiles
    (G = 1 .. 8, so 128 .. 16 tokens per sub-tile, one or two per item) or, for a
    small group, the split-KV shared-prefix CTAs; against the oracle on every row."""
    rng = np.random.default_rng(500 + seed)
    meta = workloads.random_step(rng, num_seqs=num_seqs, group=group, hkv=hkv, d=d, max_q=3,
                                 max_ctx=pre * 16 + 700, shared_prefix_blocks=pre)
    q, k, v, pool = workloads.make_values(meta)
    info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads,
                            pkv.pool_desc(pool), upload=False, block_tables=meta.block_tables)
    assert info.num_gather_rows > 0 or info.num_shared_ctas > 0
    want, _ = oracle.run_step(meta, q, k, v, pool)
    for sms in (152, 9):
        out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, num_sms=sms)
        assert_close(out, want, f"seed {seed} sms {sms}")


@pytest.mark.parametrize("seed", [0, 1])
def test_verify_windows_chained_shared_items_match_oracle(pkv, cuda_device, seed):
    """Verify windows of 8 tokens (two row groups that read the same blocks) go to
    shared-block CTAs whose warp pairs run chains of items (items that split a
    window's blocks between pairs; with 1 or 3 SMs the planner keeps the windows
    on the per-warp ranges instead).  Every row against the oracle, and the
    chains really occur."""
    rng = np.random.default_rng(900 + seed)
    n = 12
    q_lens = [8 if i % 2 == 0 else 4 for i in range(n)]
    ctx = [int(c) for c in rng.integers(160, 1500, size=n)]
    meta = workloads.build_step("windows", 77 + seed, q_lens, ctx, 8, 2, 128, rng=rng)
    q, k, v, pool = workloads.make_values(meta)
    want, _ = oracle.run_step(meta, q, k, v, pool)
    chained = False
    for sms in (1, 3, 9, 37, 152):
        info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads,
                                pkv.pool_desc(pool), num_sms=sms, upload=False,
                                block_tables=meta.block_tables)
        assert info.num_shared_ctas > 0 or sms < 9
        chained |= info.num_shared_items > 2 * info.num_shared_ctas
        out, _, _ = gpu_step(pkv, meta, q, k, v, pool, cuda_device, num_sms=sms)
        assert_close(out, want, f"windows seed {seed} sms {sms}")
    assert chained


@pytest.mark.parametrize("window", [False, True])
def test_planning_thread_serves_consecutive_steps(pkv, cuda_device, window):
    """A serving loop over several decode steps whose contexts grow (plans of
    changing size): each step is planned on the library's planning thread while
    the step's KV append is queued, then attended with that plan; every step
    matches the oracle and the pool ends bit-exact."""
    steps = 5
    meta, per_step = _chain_case(steps, seed=91, window=window)
    _, _, _, pool = workloads.make_values(per_step[0])
    vals = [workloads.make_values(m, seed=700 + t)[:3] for t, m in enumerate(per_step)]
    pool_o, want = pool, []
    for m, (q, k, v) in zip(per_step, vals):
        out, pool_o = oracle.run_step(m, q, k, v, pool_o)
        want.append(out)
    dev = cuda_device
    pd = pool.to(dev)
    cu_h = meta.cu_q_lens.astype(np.int32).copy()
    ctx_h = per_step[0].context_lens.astype(np.int32).copy()
    bt_h = meta.block_tables.astype(np.int32).copy()
    plan_h = np.zeros(1 << 18, np.int32)
    planner = pkv.BoundPlan(cu_h, ctx_h, meta.num_q_heads, pd, plan_h, block_tables=bt_h,
                            spin_us=200)
    cu = torch.from_numpy(cu_h).to(dev)
    bt = torch.from_numpy(bt_h).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sizes = set()
    for t, (m, (q, k, v)) in enumerate(zip(per_step, vals)):
        ctx_h[:] = m.context_lens
        planner.post()
        ctx = torch.from_numpy(m.context_lens).to(dev)
        slots = torch.from_numpy(m.slot_mapping).to(dev)
        pkv.paged_kv_append(k.to(dev), v.to(dev), slots, pd, dev_status=status)
        info, nb = planner.wait()
        sizes.add(int(info.plan_bytes))
        plan = pkv.StepPlan(info, plan_h.view(np.uint8)[:nb].view(np.int32), dev)
        out = pkv.paged_varlen_attention(q.to(dev), cu, ctx, bt, pd, meta.scale, plan=plan,
                                         dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(out.cpu(), want[t], f"planning thread step {t}")
    planner.close()
    assert len(sizes) > 1          # the plans did change from step to step
    assert np.array_equal(bits(pd), pool_o)
