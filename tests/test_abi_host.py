"""Host-side tests of the C ABI (no GPU needed): exported symbols, the step
planner's tiling invariants, and argument validation that returns before any
CUDA call."""

import ctypes
import os
import re

import numpy as np
import pytest

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_attention_append_gb300 as m
    m.build()
    return m


def test_library_exports_every_declared_symbol(pkv):
    with open(os.path.join(ROOT, "include", "pkv.h")) as f:
        hdr = f.read()
    names = re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", hdr)
    assert len(names) >= 6, names
    lib = ctypes.CDLL(pkv.library_path())
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pkv.h but not exported"


def test_version_and_status_strings(pkv):
    assert pkv.version() >= 100
    for s in range(11):
        assert pkv.status_string(s).startswith("PKV_")
    assert pkv.status_string(11) == "unknown pkv status"


# ---------------------------------------------------------------- planner

def parse_plan(info, host):
    words = host.view(np.int32)
    hdr = words[:16]
    assert hdr[0] == 0x33564B50
    nw, npc, nm, npf = (info.num_decode_warps, info.num_decode_pieces, info.num_merge_groups,
                        info.num_prefill_tiles)
    off_w = 16
    off_first = off_w + ((nw + 1 + 7) // 8) * 8
    off_p = off_first + 12 * nw
    off_m = off_p + 8 * npc
    ncta = info.num_prefill_ctas
    nsh = info.num_shared_ctas
    nitems = info.num_shared_items
    assert nitems >= 2 * nsh             # two warp pairs per shared CTA, each starting a chain
    off_s = off_m + 8 * nm
    off_b = off_s + 24 * nitems          # 96-byte items
    off_f = off_b + (((ncta + 1 + 7) // 8) * 8 if ncta else 0)
    off_g = off_f + 16 * npf
    ng = info.num_gather_rows
    assert hdr[12] == ng
    assert info.plan_bytes == 4 * (off_g + 4 * ng)
    wb = words[off_w:off_w + nw + 1]
    pieces = words[off_p:off_m].reshape(npc, 8)
    heads = words[off_first:off_p].reshape(nw, 12)
    if nw:
        assert np.array_equal(heads[:, :8], pieces[wb[:-1]])  # each warp's first piece, copied
    mer = words[off_m:off_s].reshape(nm, 8)
    pre = words[off_f:off_g].reshape(npf, 16)
    parse_plan.gather = words[off_g:off_g + 4 * ng].reshape(ng, 4)
    parse_plan.shared = words[off_s:off_b].reshape(nitems, 24)
    if nitems:
        # every item is on exactly one pair's chain: pair k starts at item k and
        # each `next` (word 5) names a later item or is -1
        seen = np.zeros(nitems, bool)
        for k in range(2 * nsh):
            i = k
            while i >= 0:
                assert not seen[i]
                seen[i] = True
                nxt = int(parse_plan.shared[i, 5])
                assert nxt == -1 or i < nxt < nitems
                if nxt != -1:
                    assert nxt >= 2 * nsh        # the chains' other items follow the heads
                i = nxt
        assert seen.all()
    pb = words[off_b:off_b + ncta + 1] if ncta else np.zeros(1, np.int32)
    if ncta:
        assert pb[0] == 0 and pb[-1] == npf and np.all(np.diff(pb) >= 1)   # no CTA without work
    return hdr, wb, pieces, mer, pre


def check_prefill_items(meta, pre, mer, s):
    """Work items of prefill-class sequence s:
    (seq, h, hq0, hq1, qi0_0, qi0_1, n0, n1, kt0, kt1, part0, part1).
    Every (query head, 128-token tile) unit sees each of its key tiles in exactly
    one item; both sub-tiles of an item read KV head h; a unit whose key tiles
    span several items has one partial slot per item and one merge group (kind
    1) naming exactly those slots; a unit in one item writes out directly."""
    g = meta.num_q_heads // meta.num_kv_heads
    qs, ctx = int(meta.q_lens[s]), int(meta.context_lens[s])
    items = pre[(pre[:, 0] == s) & (pre[:, 12] < 0)]     # contiguous sub-tiles only
    seen = {}    # (hq, q0) -> list of (kt0, kt1, part)
    for it in items:
        _, h, hq0, hq1, qa, qb, na, nb, kt0, kt1, pa, pb = (int(v) for v in it[:12])
        assert it[13] < 0
        assert 1 <= na <= 128 and 0 <= nb <= 128 and 0 <= kt0 < kt1
        for hq, q0, n, part in [(hq0, qa, na, pa)] + ([(hq1, qb, nb, pb)] if nb else []):
            assert hq // g == h and q0 % 128 == 0 and n == min(128, qs - q0)
            nt = (ctx - qs + q0 + n - 1) // 128 + 1
            assert kt0 < nt
            seen.setdefault((hq, q0), []).append((kt0, min(kt1, nt), part, nt))
    expect = [(hq, q0) for hq in range(meta.num_q_heads) for q0 in range(0, qs, 128)]
    assert sorted(seen) == sorted(expect)
    pm = mer[(mer[:, 0] == s) & (mer[:, 6] == 1)]
    for (hq, q0), rs in seen.items():
        rs.sort()
        nt = rs[0][3]
        assert rs[0][0] == 0 and rs[-1][1] == nt
        assert all(rs[i][1] == rs[i + 1][0] for i in range(len(rs) - 1))   # no gap, no overlap
        m = pm[(pm[:, 3] == hq) & (pm[:, 1] == q0)]
        if len(rs) == 1:
            assert rs[0][2] == -1 and len(m) == 0
        else:
            parts = sorted(r[2] for r in rs)
            assert len(m) == 1 and m[0, 5] == len(rs) and parts == list(range(m[0, 4], m[0, 4] + len(rs)))
    return len(items)


def sum_segment_blocks(meta):
    """Blocks over all (row group, KV head) segments of the decode-class rows."""
    g = meta.num_q_heads // meta.num_kv_heads
    nq_tile = max(1, 16 // g)
    tot = 0
    for s in range(meta.num_seqs):
        qs, ctx = int(meta.q_lens[s]), int(meta.context_lens[s])
        if qs == 0 or qs >= 64:
            continue
        for qi0 in range(0, qs, nq_tile):
            n_q = min(nq_tile, qs - qi0)
            tot += ((ctx - qs + qi0 + n_q - 1) // 16 + 1) * meta.num_kv_heads
    return tot


def check_plan(meta, info, host, num_sms):
    hdr, wb, pieces, mer, pre = parse_plan(info, host)
    g = meta.num_q_heads // meta.num_kv_heads
    hkv = meta.num_kv_heads
    nq_tile = max(1, 16 // g)
    assert info.total_q == meta.total_q
    assert info.kv_tokens == int(meta.context_lens[meta.q_lens > 0].astype(np.int64).sum())
    # warp ranges: contiguous, cover all pieces, equal cost: 2 per block plus 6
    # per segment start; each of a range's two ends may be off by one block and
    # one segment start
    # shared-block items (verify windows wider than one row group): as pieces
    # (seq, qi0, n_q, h, kb_begin, kb_end, part, q_row0), one per row group
    sh = parse_plan.shared
    rows = []
    for it in sh:
        for w in range(int(it[4])):
            rg = it[8 + 8 * w:16 + 8 * w]
            rows.append([rg[0], rg[1], rg[2], it[1], it[2], it[3], rg[3], rg[4]])
    sh_pieces = np.array(rows, dtype=np.int32).reshape(-1, 8)
    nw = info.num_decode_warps
    if nw:
        assert wb[0] == 0 and wb[-1] == len(pieces) and np.all(np.diff(wb) >= 1)
        per_warp = [int((pieces[wb[w]:wb[w + 1], 5] - pieces[wb[w]:wb[w + 1], 4]).sum())
                    for w in range(nw)]
        sh_blocks = int((sh_pieces[:, 5] - sh_pieces[:, 4]).sum())
        assert sum(per_warp) + sh_blocks == sum_segment_blocks(meta)
        if not len(sh_pieces):
            cost = [2 * per_warp[w] + 6 * int((pieces[wb[w]:wb[w + 1], 4] == 0).sum())
                    for w in range(nw)]
            assert max(cost) - min(cost) <= 2 * (2 + 6)
        if num_sms is not None:      # warp slots: independent warps, then two per pair
            assert nw + 2 * 2 * info.num_shared_ctas <= num_sms * 8
    assert np.all(pieces[:, 5] > pieces[:, 4])
    pieces = np.concatenate([pieces, sh_pieces])
    # every decode segment (row group x KV head) is covered exactly once, in order
    prefill_seqs = set(int(x) for x in pre[pre[:, 12] < 0, 0]) if len(pre) else set()
    seen_parts = set()
    total_blocks = 0
    for s in range(meta.num_seqs):
        qs, ctx = int(meta.q_lens[s]), int(meta.context_lens[s])
        mine = pieces[pieces[:, 0] == s]
        if qs == 0:
            assert len(mine) == 0 and s not in prefill_seqs
            continue
        if s in prefill_seqs:
            assert len(mine) == 0
            check_prefill_items(meta, pre, mer, s)
            continue
        for qi0 in range(0, qs, nq_tile):
            n_q = min(nq_tile, qs - qi0)
            nb = (ctx - qs + qi0 + n_q - 1) // 16 + 1
            for h in range(hkv):
                seg = mine[(mine[:, 1] == qi0) & (mine[:, 3] == h)]
                assert len(seg) >= 1 and np.all(seg[:, 2] == n_q)
                seg = seg[np.argsort(seg[:, 4])]
                assert seg[0, 4] == 0 and seg[-1, 5] == nb
                assert np.all(seg[1:, 4] == seg[:-1, 5])
                total_blocks += nb
                if len(seg) == 1:
                    assert seg[0, 6] == -1
                else:
                    parts = list(seg[:, 6])
                    assert parts == list(range(parts[0], parts[0] + len(parts)))
                    assert not (set(parts) & seen_parts)
                    seen_parts |= set(parts)
                    m = mer[(mer[:, 0] == s) & (mer[:, 1] == qi0) & (mer[:, 3] == h) & (mer[:, 6] == 0)]
                    assert len(m) == 1 and m[0, 2] == n_q and m[0, 4] == parts[0] and m[0, 5] == len(parts)
    assert total_blocks == sum_segment_blocks(meta)
    # the split-KV kernel's attended blocks, each (sequence, block, KV head) once
    dec = [s for s in range(meta.num_seqs) if 0 < meta.q_lens[s] and s not in prefill_seqs]
    assert info.decode_blocks == hkv * sum((int(meta.context_lens[s]) + 15) // 16 for s in dec)
    assert len(seen_parts) == info.num_partials
    d = meta.head_dim
    a = lambda x: (x + 255) // 256 * 256
    pp = info.num_prefill_partials
    ws = a(info.num_partials * 16 * d * 4) + a(info.num_partials * 16 * 8) + \
        a(pp * 128 * d * 4) + a(pp * 128 * 8)
    assert info.workspace_bytes == ws
    nm = info.num_merge_groups
    assert np.array_equal(mer[:, 7], meta.cu_q_lens[mer[:, 0]] + mer[:, 1])   # packed first row
    assert info.num_prefill_merges == int((mer[:, 6] == 1).sum())
    assert np.all(mer[:nm - info.num_prefill_merges, 6] == 0)   # decode groups first
    dmer = mer[:nm - info.num_prefill_merges]
    g = meta.num_q_heads // meta.num_kv_heads
    # the merge launch covers the largest decode group's rows (n_q tokens x G heads)
    assert info.merge_rows == (int(dmer[:, 2].max()) * g if len(dmer) else 0)
    assert info.merge_rows <= 16
    assert info.num_kernels == (info.num_decode_warps > 0) + (info.num_merge_groups > 0) + \
        (info.num_prefill_tiles > 0)


@pytest.mark.parametrize("name", list(workloads.CONFIGS))
def test_planner_tiles_cover_every_config(pkv, name):
    meta = workloads.make_config(name)
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    for sms in (152, 20):
        info, host = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                                   num_sms=sms, upload=False)
        check_plan(meta, info, host, sms)


@pytest.mark.parametrize("seed", range(20))
def test_planner_random_steps(pkv, seed):
    rng = np.random.default_rng(seed)
    meta = workloads.random_step(rng, max_ctx=3000)
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    info, host = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                               num_sms=int(rng.integers(1, 200)), upload=False)
    check_plan(meta, info, host, None)


def test_planner_handles_zero_length_queries_and_empty_steps(pkv):
    desc = pkv.PoolDesc(10, 16, 2, 64)
    info, host = pkv.plan_step(np.array([0, 0, 3, 3], np.int32), np.array([5, 40, 7], np.int32), 4,
                               desc, num_sms=152, upload=False)
    hdr, wb, pieces, mer, pre = parse_plan(info, host)
    assert set(pieces[:, 0]) == {1}
    info, host = pkv.plan_step(np.array([0], np.int32), np.array([], np.int32), 4, desc,
                               num_sms=152, upload=False)
    assert info.num_decode_warps == 0 and info.num_kernels == 0 and info.workspace_bytes == 0
    # a step of prefill chunks only: no split-KV warps at all
    info, host = pkv.plan_step(np.array([0, 300, 500], np.int32), np.array([300, 900], np.int32), 4,
                               pkv.PoolDesc(200, 16, 2, 64), num_sms=152, upload=False)
    assert info.num_decode_warps == 0 and info.num_prefill_tiles > 0


@pytest.mark.parametrize("cu,ctx,hq,desc,err", [
    ([1, 2], [4], 4, (10, 16, 2, 64), "SHAPE"),             # cu[0] != 0
    ([0, 3, 2], [4, 4], 4, (10, 16, 2, 64), "SHAPE"),       # not monotone
    ([0, 5], [4], 4, (10, 16, 2, 64), "RANGE"),             # q_len > ctx
    ([0, 1], [-1], 4, (10, 16, 2, 64), "RANGE"),            # negative ctx
    ([0, 1], [4], 4, (10, 16, 2, 96), "UNSUPPORTED"),       # head_dim 96
    ([0, 1], [4], 4, (10, 8, 2, 64), "UNSUPPORTED"),        # block size 8
    ([0, 1], [4], 5, (10, 16, 2, 64), "SHAPE"),             # Hq % Hkv
    ([0, 1], [4], 64, (10, 16, 2, 64), "UNSUPPORTED"),      # group 32 > 16
])
def test_planner_rejects_bad_steps(pkv, cu, ctx, hq, desc, err):
    with pytest.raises(pkv.PkvError) as ei:
        pkv.plan_step(np.array(cu, np.int32), np.array(ctx, np.int32), hq, pkv.PoolDesc(*desc),
                      num_sms=152, upload=False)
    assert err in str(ei.value)


def test_planner_reports_small_plan_buffer(pkv):
    lib = ctypes.CDLL(pkv.library_path())
    lib.pkv_plan_step.restype = ctypes.c_int32
    cu = np.array([0, 1, 2], np.int32)
    ctx = np.array([100, 200], np.int32)
    desc = pkv.PoolDesc(100, 16, 2, 64)
    info = pkv.PlanInfo()
    buf = np.zeros(4, np.int32)
    st = lib.pkv_plan_step(cu.ctypes.data_as(ctypes.c_void_p), ctx.ctypes.data_as(ctypes.c_void_p),
                           2, 4, ctypes.byref(desc), 152, buf.ctypes.data_as(ctypes.c_void_p),
                           ctypes.c_int64(buf.nbytes), ctypes.byref(info))
    assert st == 5 and info.plan_bytes > buf.nbytes


# ---------------------------------------------------------------- entry-point validation

def _raw(pkv):
    lib = ctypes.CDLL(pkv.library_path())
    lib.pkv_paged_kv_append.restype = ctypes.c_int32
    lib.pkv_paged_varlen_attention.restype = ctypes.c_int32
    return lib


FAKE = 0x7F0000001000  # never dereferenced: every call below returns before touching the GPU


def test_append_validation_returns_before_launch(pkv):
    lib = _raw(pkv)
    P = ctypes.c_void_p
    ok = pkv.PoolDesc(10, 16, 2, 64)
    # zero tokens: nothing to do
    assert lib.pkv_paged_kv_append(None, None, None, 0, None, ctypes.byref(ok), None, None) == 0
    assert lib.pkv_paged_kv_append(P(FAKE), P(FAKE), None, 3, P(FAKE), ctypes.byref(ok), None, None) == 1
    assert lib.pkv_paged_kv_append(P(FAKE), P(FAKE), P(FAKE), 3, P(FAKE), None, None, None) == 1
    bad = pkv.PoolDesc(10, 32, 2, 64)
    assert lib.pkv_paged_kv_append(P(FAKE), P(FAKE), P(FAKE), 3, P(FAKE), ctypes.byref(bad), None, None) == 4
    assert lib.pkv_paged_kv_append(P(FAKE + 8), P(FAKE), P(FAKE), 3, P(FAKE), ctypes.byref(ok), None, None) == 8
    assert lib.pkv_paged_kv_append(P(FAKE), P(FAKE), P(FAKE), -1, P(FAKE), ctypes.byref(ok), None, None) == 2
    huge = pkv.PoolDesc(1 << 27, 16, 8, 128)   # 2^31 pool rows: TMA coordinates would overflow
    assert lib.pkv_paged_kv_append(P(FAKE), P(FAKE), P(FAKE), 3, P(FAKE), ctypes.byref(huge), None, None) == 4


def test_attention_validation_returns_before_launch(pkv):
    lib = _raw(pkv)
    P = ctypes.c_void_p
    meta = workloads.small_decode()
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    info, host = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                               num_sms=152, upload=False)

    def call(info_=info, desc_=desc, scale=0.1, maxb=meta.max_blocks, ws=P(FAKE), wsb=1 << 30, q=P(FAKE)):
        return lib.pkv_paged_varlen_attention(q, P(FAKE), P(FAKE), P(FAKE), maxb, P(FAKE),
                                              ctypes.byref(desc_), ctypes.c_float(scale),
                                              ctypes.byref(info_), P(FAKE), P(FAKE), ws,
                                              ctypes.c_int64(wsb), None, None)
    assert call(q=None) == 1
    assert call(scale=float("nan")) == 3
    assert call(maxb=info.max_blocks_needed - 1) == 3
    if info.workspace_bytes:
        assert call(wsb=info.workspace_bytes - 1) == 5
    assert call(ws=P(FAKE + 16)) == 8        # workspace must be 256-byte aligned
    other = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, 64)
    assert call(desc_=other) == 2
    empty, _ = pkv.plan_step(np.array([0], np.int32), np.array([], np.int32), meta.num_q_heads,
                             desc, num_sms=152, upload=False)
    assert call(info_=empty, q=None) == 0    # nothing to compute


def test_state_checkpoint_argument_checks_return_before_any_cuda_call(pkv):
    lib = ctypes.CDLL(pkv.library_path())
    f = lib.pkv_state_checkpoint
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    f.restype = ctypes.c_int32
    fake = ctypes.c_void_p(0x1000)     # never dereferenced: every case returns before a launch
    assert f(fake, fake, 4, fake, 10, 24, None, None) == 2       # row_bytes not a multiple of 16
    assert f(fake, fake, 4, fake, 10, 0, None, None) == 2        # empty rows
    assert f(fake, fake, -1, fake, 10, 32, None, None) == 2      # negative count
    assert f(None, None, 0, None, 10, 32, None, None) == 0       # nothing to do
    assert f(None, fake, 4, fake, 10, 32, None, None) == 1       # NULL src
    assert f(ctypes.c_void_p(0x1008), fake, 4, fake, 10, 32, None, None) == 8   # misaligned src


def test_decode_chain_plan_covers_the_last_step(pkv):
    """A chain plan for S steps is a single-step plan of the last step's contexts
    (each step adds q_len tokens), with lookahead S - 1; prefill rows are refused."""
    meta = workloads.small_decode()
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    steps = 7
    info, host = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                               num_sms=152, upload=False, chain_steps=steps)
    last = meta.context_lens + (steps - 1) * meta.q_lens
    info1, host1 = pkv.plan_step(meta.cu_q_lens, last, meta.num_q_heads, desc, num_sms=152,
                                 upload=False)
    assert info.lookahead == steps - 1 and info1.lookahead == 0
    assert info.decode_blocks == info1.decode_blocks
    assert info.kv_tokens == int(meta.context_lens.sum())
    assert np.array_equal(host[16:], host1[16:])          # same work lists after the header
    with pytest.raises(pkv.PkvError):                       # prefill-class rows
        pkv.plan_step([0, 100], [300], 8, pkv.PoolDesc(100, 16, 2, 128), upload=False, chain_steps=2)
    with pytest.raises(pkv.PkvError):
        pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc, upload=False,
                      chain_steps=0)


def test_plan_carries_first_block_ids_when_given_the_tables(pkv):
    meta = workloads.small_decode()
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    info, host = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                               num_sms=152, upload=False, block_tables=meta.block_tables)
    info0, host0 = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                                 num_sms=152, upload=False)
    nw = info.num_decode_warps
    off = 16 + ((nw + 1 + 7) // 8) * 8
    heads = host.view(np.int32)[off:off + 12 * nw].reshape(nw, 12)
    heads0 = host0.view(np.int32)[off:off + 12 * nw].reshape(nw, 12)
    assert np.array_equal(heads[:, :8], heads0[:, :8]) and np.all(heads0[:, 8:] == -1)
    for w in range(nw):
        seq, kb0, kb1 = heads[w, 0], heads[w, 4], heads[w, 5]
        for i in range(3):
            want = meta.block_tables[seq, kb0 + i] if kb0 + i < kb1 else -1
            assert heads[w, 8 + i] == want
        assert heads[w, 11] == -1



def test_shared_prefix_items_cover_the_shared_blocks(pkv):
    """With the host tables, sequences whose tables start with the same blocks get
    shared-prefix CTAs over those blocks; every (row group, KV head) result is then
    its shared chunks over [0, L) plus its suffix pieces over [L, nb), with one
    merge group naming exactly those parts."""
    # a small group (under 64 query rows per KV head) stays on the split-KV CTAs
    meta = workloads.random_step(np.random.default_rng(11), num_seqs=6, group=2, max_q=2,
                                 max_ctx=600, shared_prefix_blocks=16)
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    info, host = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                               num_sms=152, upload=False, block_tables=meta.block_tables)
    assert info.num_shared_ctas > 0 and info.num_gather_rows == 0
    hdr, wb, pieces, mer, pre = parse_plan(info, host)
    sh = parse_plan.shared
    g = meta.num_q_heads // meta.num_kv_heads
    nq_tile = max(1, 16 // g)
    # shared chunks per (seq, qi0, h): list of (kb_begin, kb_end, part)
    got = {}
    for it in sh:
        seq0, h, kb0, kb1, nrg = (int(x) for x in it[:5])
        if nrg == 0:                              # an empty item (pads a CTA's pair)
            continue
        assert 1 <= nrg <= 2 and 0 <= kb0 < kb1
        # the blocks are the same physical blocks in every member's table
        for w in range(nrg):
            seq, qi0, n_q, part, qrow = (int(x) for x in it[8 + 8 * w: 13 + 8 * w])
            assert np.array_equal(meta.block_tables[seq, kb0:kb1], meta.block_tables[seq0, kb0:kb1])
            assert qrow == meta.cu_q_lens[seq] + qi0
            got.setdefault((seq, qi0, h), []).append((kb0, kb1, part))
    assert got
    for (seq, qi0, h), chunks in got.items():
        chunks.sort()
        L = chunks[-1][1]
        assert chunks[0][0] == 0 and all(chunks[i][1] == chunks[i + 1][0] for i in range(len(chunks) - 1))
        qs, ctx = int(meta.q_lens[seq]), int(meta.context_lens[seq])
        n_q = min(nq_tile, qs - qi0)
        nb = (ctx - qs + qi0 + n_q - 1) // 16 + 1
        assert L <= (ctx - qs + 1) // 16          # every row sees the shared blocks in full
        mine = pieces[(pieces[:, 0] == seq) & (pieces[:, 1] == qi0) & (pieces[:, 3] == h)]
        mine = mine[np.argsort(mine[:, 4])]
        if len(mine):
            assert mine[0, 4] == L and mine[-1, 5] == nb
            assert np.all(mine[1:, 4] == mine[:-1, 5])
        parts = sorted([c[2] for c in chunks] + [int(x) for x in mine[:, 6]])
        m = mer[(mer[:, 0] == seq) & (mer[:, 1] == qi0) & (mer[:, 3] == h) & (mer[:, 6] == 0)]
        if len(parts) > 1:
            assert len(m) == 1 and m[0, 5] == len(parts)
            assert parts == list(range(m[0, 4], m[0, 4] + len(parts)))
        else:
            assert parts == [-1] and len(m) == 0


def check_gathered_prefix(meta, info, host):
    """Gathered sub-tiles (a prefix many query rows share, on the tensor cores):
    every token of every sharing sequence appears once per KV head and key chunk,
    at the right row of its row group's partial slot; each (row group, KV head)
    has its prefix key tiles [0, KT) covered once, by chunks whose slots are
    consecutive from its merge group's first slot, and its suffix pieces cover
    blocks [8 KT, nb); the gathered keys are the same physical blocks in every
    member's table.  Returns the number of (row group, KV head) pairs covered."""
    hdr, wb, pieces, mer, pre = parse_plan(info, host)
    gat = parse_plan.gather
    g = meta.num_q_heads // meta.num_kv_heads
    nq_tile = max(1, 16 // g)
    cu = meta.cu_q_lens
    items = pre[pre[:, 12] >= 0]
    assert len(items) and info.num_gather_rows == len(gat)
    cover = {}   # (seq, qi0, h) -> list of (kt0, kt1, slot)
    for it in items:
        seq0, h, kt0, kt1 = int(it[0]), int(it[1]), int(it[8]), int(it[9])
        assert 0 <= kt0 < kt1
        for x in range(2):
            n, c, g0 = int(it[6 + x]), int(it[10 + x]), int(it[12 + x])
            if n == 0:
                assert x == 1 and g0 < 0
                continue
            assert 1 <= n * g <= 128 and c >= 0 and g0 >= 0
            toks = gat[g0:g0 + n, 0]
            run = bool(np.all(np.diff(toks) == 1))
            assert bool(it[14] >> x & 1) == run          # consecutive tokens: one q box
            if run:
                assert it[4 + x] == toks[0]
            for q_tok, part0, row0, _ in gat[g0:g0 + n]:
                s = int(np.searchsorted(cu, q_tok, side="right")) - 1
                i = int(q_tok - cu[s])
                qi0 = i // nq_tile * nq_tile
                assert row0 == (i - qi0) * g
                assert np.array_equal(meta.block_tables[s, 8 * kt0:8 * kt1],
                                      meta.block_tables[seq0, 8 * kt0:8 * kt1])
                qs, ctx = int(meta.q_lens[s]), int(meta.context_lens[s])
                assert 128 * kt1 <= ctx - qs + 1          # every row sees these keys
                cover.setdefault((s, qi0, h), {}).setdefault(i, []).append((kt0, kt1, part0 + c))
    for (s, qi0, h), per_tok in cover.items():
        qs, ctx = int(meta.q_lens[s]), int(meta.context_lens[s])
        n_q = min(nq_tile, qs - qi0)
        assert sorted(per_tok) == list(range(qi0, qi0 + n_q))   # every token of the row group
        chunks = sorted(set(per_tok[qi0]))
        assert all(sorted(set(v)) == chunks for v in per_tok.values())
        assert chunks[0][0] == 0 and all(chunks[k][1] == chunks[k + 1][0] for k in range(len(chunks) - 1))
        kt = chunks[-1][1]
        slots = [c[2] for c in chunks]
        m = mer[(mer[:, 0] == s) & (mer[:, 1] == qi0) & (mer[:, 3] == h) & (mer[:, 6] == 0)]
        assert len(m) == 1 and slots == list(range(m[0, 4], m[0, 4] + len(slots)))
        nb = (ctx - qs + qi0 + n_q - 1) // 16 + 1
        mine = pieces[(pieces[:, 0] == s) & (pieces[:, 1] == qi0) & (pieces[:, 3] == h)]
        mine = mine[np.argsort(mine[:, 4])]
        if 8 * kt < nb:
            assert mine[0, 4] == 8 * kt and mine[-1, 5] == nb and np.all(mine[1:, 4] == mine[:-1, 5])
        assert m[0, 5] == len(slots) + len(mine)
        if len(mine):
            assert sorted(mine[:, 6]) == list(range(m[0, 4] + len(slots), m[0, 4] + m[0, 5]))
    return len(cover)


@pytest.mark.parametrize("name", ["shared_prefix_verify", "mtp_draft"])
def test_gathered_prefix_items_cover_every_row_group(pkv, name):
    meta = workloads.make_config(name)
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    for sms in (152, 13):
        info, host = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                                   num_sms=sms, upload=False, block_tables=meta.block_tables)
        assert info.num_shared_ctas == 0 and info.num_gather_rows > 0
        g = meta.num_q_heads // meta.num_kv_heads
        units = sum((int(q) + max(1, 16 // g) - 1) // max(1, 16 // g) for q in meta.q_lens)
        assert check_gathered_prefix(meta, info, host) == units * meta.num_kv_heads


def test_step_generator_slots_are_distinct():
    """Every generated step appends each new token to its own slot (a slot written
    twice would make the pool depend on write order), also when sequences share
    prefix blocks."""
    metas = [workloads.make_config(n) for n in workloads.CONFIGS]
    for seed in range(30):
        rng = np.random.default_rng(900 + seed)
        metas.append(workloads.random_step(rng, num_seqs=int(rng.integers(2, 40)), max_q=3,
                                           shared_prefix_blocks=int(rng.choice([0, 3, 8, 20])),
                                           max_ctx=500))
    for meta in metas:
        sl = meta.slot_mapping[meta.slot_mapping >= 0]
        assert len(np.unique(sl)) == len(sl), meta.name


def test_workspace_size_matches_the_plan_summary(pkv):
    for name in ("small_decode", "agent_mixed", "tiny_decode"):
        meta = workloads.make_config(name)
        desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
        info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc,
                                num_sms=152, upload=False)
        assert pkv.workspace_size(info) == info.workspace_bytes
    lib = ctypes.CDLL(pkv.library_path())
    lib.pkv_workspace_size.restype = ctypes.c_size_t
    assert lib.pkv_workspace_size(None) == 0


@pytest.mark.parametrize("name", ["small_decode", "agent_mixed", "shared_prefix_verify",
                                  "decode_chain"])
def test_bound_planner_writes_the_plan_step_bytes(pkv, name):
    """BoundPlan is argument marshalling only: over the same arrays it writes the
    bytes plan_step writes, run after run, and follows in-place edits of them."""
    meta = workloads.make_config(name)
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    cu, ctx = meta.cu_q_lens.astype(np.int32).copy(), meta.context_lens.astype(np.int32).copy()
    bt = meta.block_tables.astype(np.int32).copy()
    chain = 3 if name == "decode_chain" else None
    out = np.zeros(1 << 17, np.int32)
    bp = pkv.BoundPlan(cu, ctx, meta.num_q_heads, desc, out, num_sms=152, block_tables=bt,
                       chain_steps=chain)
    for step in range(2):
        info, nb = bp.run()
        want_info, want = pkv.plan_step(cu, ctx, meta.num_q_heads, desc, upload=False,
                                        num_sms=152, block_tables=bt, chain_steps=chain)
        assert nb == want.nbytes and info.plan_bytes == want_info.plan_bytes
        assert np.array_equal(out.view(np.uint8)[:nb], want.view(np.uint8)[:nb])
        assert info.workspace_bytes == want_info.workspace_bytes
        if name != "decode_chain":
            ctx[-1] += 16   # the next step: one sequence gains a block
    with pytest.raises(TypeError):
        pkv.BoundPlan(cu.astype(np.int64), ctx, meta.num_q_heads, desc, out, num_sms=152)
    with pytest.raises(ValueError):
        pkv.BoundPlan(cu[:-1], ctx, meta.num_q_heads, desc, out, num_sms=152)


def test_copy_entry_point_checks_its_arguments(pkv):
    """pkv_copy_async's argument errors come back without touching a device."""
    lib = ctypes.CDLL(pkv.library_path())
    P = ctypes.c_void_p
    lib.pkv_copy_async.argtypes = [P, P, ctypes.c_int64, P]
    buf = ctypes.create_string_buffer(64)
    assert lib.pkv_copy_async(None, None, 0, None) == 0                  # nothing queued
    assert lib.pkv_copy_async(None, ctypes.addressof(buf), 16, None) == 1  # PKV_ERR_NULL
    assert lib.pkv_copy_async(ctypes.addressof(buf), None, 16, None) == 1
    assert lib.pkv_copy_async(ctypes.addressof(buf), ctypes.addressof(buf), -1, None) == 3


def test_prefill_min_q_is_a_planner_argument(pkv):
    meta = workloads.build_step("pmq", 5, [300, 200, 1], [900, 700, 50], 8, 2, 128)
    desc = pkv.PoolDesc(meta.num_blocks, 16, 2, 128)

    def tiles(pmq):
        info, host = pkv.plan_step(meta.cu_q_lens, meta.context_lens, 8, desc, num_sms=152,
                                   upload=False, prefill_min_q=pmq)
        pf = parse_plan(info, host)[4]
        return sorted({int(t[0]) for t in pf}), info
    assert tiles(None)[0] == [0, 1]      # default: from 64 query tokens
    assert tiles(250)[0] == [0]
    seqs, info = tiles(-1)               # none: every row on the split-KV kernel
    assert seqs == [] and info.num_prefill_tiles == 0 and info.num_decode_warps > 0


def test_planner_asks_the_device_for_its_sm_count(pkv):
    """num_sms <= 0 means "the current device's SM count"; with no device the
    planner says so instead of guessing."""
    meta = workloads.tiny_decode()
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    with pytest.raises(pkv.PkvError) as e:
        pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, desc, num_sms=0,
                      upload=False)
    assert e.value.status == 6      # PKV_ERR_CUDA


def test_split_kv_warps_beside_a_prefill(pkv):
    """Behind a prefill whose persistent CTAs take every SM the split-KV work goes
    to half the warp slots (the CTAs that start first, as those CTAs exit); a
    small prefill chunk beside many decodes leaves SMs free from the start and
    keeps every slot; with gathered prefix items only, the split-KV work goes to
    the warp slots of the SMs the items leave free."""
    desc = pkv.PoolDesc(60000, 16, 8, 128)
    # 200 decodes at 2000 keys + a 64-token chunk at 1000: few prefill CTAs
    q = [1] * 200 + [64]
    ctx = [2000] * 200 + [1000]
    cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
    info, _ = pkv.plan_step(cu, np.array(ctx, np.int32), 40, desc, num_sms=152, upload=False)
    assert 0 < info.num_prefill_ctas < 152 and info.num_decode_warps == 152 * 8
    # the agent-shaped step: a 2048-token chunk whose tiles fill every SM
    meta = workloads.make_config("agent_mixed")
    info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads,
                            pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim),
                            num_sms=152, upload=False, block_tables=meta.block_tables)
    assert info.num_prefill_ctas == 152 and info.num_decode_warps == 152 * 8 // 2
    # gathered prefix items only
    meta = workloads.make_config("shared_prefix_verify")
    info, _ = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads,
                            pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim),
                            num_sms=152, upload=False, block_tables=meta.block_tables)
    assert info.num_gather_rows > 0 and info.num_shared_ctas == 0
    assert info.num_decode_warps == (152 - info.num_prefill_ctas) * 8


def test_planning_from_several_threads_gives_each_its_own_plan(pkv):
    """Plans made at the same time on several host threads (the library call
    releases the GIL) are each identical, byte for byte, to the plan made alone."""
    import threading
    steps = [workloads.make_config(n) for n in ("small_decode", "agent_mixed", "wide_verify")]
    descs = [pkv.PoolDesc(m.num_blocks, 16, m.num_kv_heads, m.head_dim) for m in steps]
    alone = [pkv.plan_step(m.cu_q_lens, m.context_lens, m.num_q_heads, d, num_sms=152,
                           upload=False, block_tables=m.block_tables)[1].copy()
             for m, d in zip(steps, descs)]
    bad = []

    def worker(i):
        m, d = steps[i % 3], descs[i % 3]
        for _ in range(30):
            _, host = pkv.plan_step(m.cu_q_lens, m.context_lens, m.num_q_heads, d, num_sms=152,
                                    upload=False, block_tables=m.block_tables)
            if not np.array_equal(host, alone[i % 3]):
                bad.append(i)
    threads = [threading.Thread(target=worker, args=(i,)) for i in range(6)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not bad


@pytest.mark.parametrize("spin_us", [0, 2000])
def test_planning_thread_writes_the_plan_run_writes(pkv, spin_us):
    """post()/wait() run the same planner call on the library's planning thread:
    byte for byte the plan run() writes, step after step, whether the thread was
    polling (spin_us 2000) or asleep (spin_us 0, and after a pause) when the job
    came."""
    import time
    for name in ("small_decode", "agent_mixed", "shared_prefix_verify", "decode_chain"):
        meta = workloads.make_config(name)
        desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
        cu, ctx = meta.cu_q_lens.astype(np.int32).copy(), meta.context_lens.astype(np.int32).copy()
        bt = meta.block_tables.astype(np.int32).copy()
        chain = 3 if name == "decode_chain" else None
        out_a, out_b = np.zeros(1 << 17, np.int32), np.zeros(1 << 17, np.int32)
        sync = pkv.BoundPlan(cu, ctx, meta.num_q_heads, desc, out_a, num_sms=152, block_tables=bt,
                             chain_steps=chain)
        thr = pkv.BoundPlan(cu, ctx, meta.num_q_heads, desc, out_b, num_sms=152, block_tables=bt,
                            chain_steps=chain, spin_us=spin_us)
        for step in range(4):
            want_info, want_nb = sync.run()
            want_ws = want_info.workspace_bytes
            out_b[:] = -1
            thr.post()
            if step == 2:
                time.sleep(0.01)        # the thread has gone to sleep by now
            info, nb = thr.wait()
            assert nb == want_nb and info.workspace_bytes == want_ws
            assert info.num_decode_warps == want_info.num_decode_warps
            assert np.array_equal(out_b.view(np.uint8)[:nb], out_a.view(np.uint8)[:nb])
            if name != "decode_chain":
                ctx[-1] += 16
        thr.close()
        with pytest.raises(RuntimeError):
            thr.post()


def test_planning_thread_reports_errors_and_misuse(pkv):
    """The job's own status comes back from wait(); a second post before wait, or
    a wait with nothing posted, is PKV_ERR_STATE, and the planner stays usable."""
    meta = workloads.tiny_decode()
    desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
    cu, ctx = meta.cu_q_lens.astype(np.int32).copy(), meta.context_lens.astype(np.int32).copy()
    out = np.zeros(1 << 14, np.int32)
    bp = pkv.BoundPlan(cu, ctx, meta.num_q_heads, desc, out, num_sms=152, spin_us=100)
    with pytest.raises(pkv.PkvError) as e:
        bp.wait()
    assert e.value.status == 9                      # PKV_ERR_STATE: nothing posted
    bp.post()
    with pytest.raises(pkv.PkvError) as e:
        bp.post()
    assert e.value.status == 9                      # PKV_ERR_STATE: still pending
    info, nb = bp.wait()
    assert info.num_seqs == len(ctx) and nb > 0
    good = ctx.copy()
    ctx[0] = -1                                     # an invalid step: PKV_ERR_RANGE from the job
    bp.post()
    with pytest.raises(pkv.PkvError) as e:
        bp.wait()
    assert e.value.status == 3
    ctx[:] = good
    bp.post()                                       # usable again
    assert bp.wait()[0].num_seqs == len(ctx)
    no_thread = pkv.BoundPlan(cu, ctx, meta.num_q_heads, desc, out, num_sms=152)
    with pytest.raises(RuntimeError):
        no_thread.post()


def test_planning_thread_entry_points_check_their_arguments(pkv):
    lib = ctypes.CDLL(pkv.library_path())
    P = ctypes.c_void_p
    lib.pkv_planner_create.argtypes = [ctypes.c_int32, ctypes.POINTER(P)]
    lib.pkv_planner_destroy.argtypes = [P]
    lib.pkv_planner_destroy.restype = None
    lib.pkv_planner_wait.argtypes = [P]
    h = P()
    assert lib.pkv_planner_create(0, None) == 1                  # PKV_ERR_NULL
    assert lib.pkv_planner_create(2000000, ctypes.byref(h)) == 3  # PKV_ERR_RANGE
    assert lib.pkv_planner_wait(None) == 1
    lib.pkv_planner_destroy(None)                                  # no-op
    for spin in (0, 50, 1000):                                     # created and destroyed idle
        assert lib.pkv_planner_create(spin, ctypes.byref(h)) == 0 and h.value
        lib.pkv_planner_destroy(h)


def test_two_planning_threads_at_once(pkv):
    """Two planners, each with its own thread, posted to and waited on from two
    Python threads at the same time: every plan is byte for byte the one the
    synchronous call writes for the same step."""
    import threading
    names = ("small_decode", "shared_prefix_verify")
    cases = []
    for name in names:
        meta = workloads.make_config(name)
        desc = pkv.PoolDesc(meta.num_blocks, 16, meta.num_kv_heads, meta.head_dim)
        cu, ctx = meta.cu_q_lens.astype(np.int32).copy(), meta.context_lens.astype(np.int32).copy()
        bt = meta.block_tables.astype(np.int32).copy()
        ref_info, ref = pkv.plan_step(cu, ctx, meta.num_q_heads, desc, num_sms=152, upload=False,
                                      block_tables=bt)
        out = np.zeros(1 << 17, np.int32)
        bp = pkv.BoundPlan(cu, ctx, meta.num_q_heads, desc, out, num_sms=152, block_tables=bt,
                           spin_us=500)
        cases.append((bp, out, ref.view(np.uint8)[:ref_info.plan_bytes].copy()))
    bad = []

    def loop(i):
        bp, out, ref = cases[i]
        for _ in range(40):
            out[:] = 0
            bp.post()
            _, nb = bp.wait()
            if not np.array_equal(out.view(np.uint8)[:len(ref)], ref):
                bad.append(i)
    threads = [threading.Thread(target=loop, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    for bp, _, _ in cases:
        bp.close()
    assert not bad
