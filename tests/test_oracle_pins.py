"""Pins for the CPU oracle, checked against things other than the oracle itself.

* brute force by a second, independent route: the padded dense rectangle
  [B, H, T, D] with an explicit boolean mask (the stock layout the vllm-metal
  page contrasts with its packed varlen step, "Replacing attention, reusing the
  rest"), gathered with numpy fancy indexing and evaluated by torch's float64
  scaled_dot_product_attention on the CPU;
* hand-derived closed forms under tests/golden/;
* invariants the definition fixes: block-permutation invariance, constant V,
  single visible key, scale 0 = mean, one-hot argmax, shared prefix = unshared
  copies, decode row = last prefill row, chunk-split invariance, batch
  composition;
* append: a numpy scatter as the second route, padding skips, range errors.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# helpers (second route: numpy gather + torch SDPA)
# ----------------------------------------------------------------------------

def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def brute_force(meta, q, pool, scale=None):
    """Padded-rectangle attention in float64 via torch SDPA with a boolean mask."""
    scale = meta.scale if scale is None else scale
    B = meta.num_seqs
    hq, hkv, d, bs = meta.num_q_heads, meta.num_kv_heads, meta.head_dim, meta.block_size
    g = hq // hkv
    tmax = int(meta.context_lens.max())
    qmax = int(meta.q_lens.max())
    poolf = pool.to(torch.float64)
    K = torch.zeros(B, hkv, tmax, d, dtype=torch.float64)
    V = torch.zeros_like(K)
    Q = torch.zeros(B, hq, qmax, d, dtype=torch.float64)
    mask = torch.zeros(B, 1, qmax, tmax, dtype=torch.bool)
    qf = q.to(torch.float64)
    for s in range(B):
        ctx = int(meta.context_lens[s])
        qs = int(meta.q_lens[s])
        pos = np.arange(ctx)
        phys = meta.block_tables[s, pos // bs]
        off = pos % bs
        K[s, :, :ctx] = poolf[phys, 0, :, off, :].permute(1, 0, 2)
        V[s, :, :ctx] = poolf[phys, 1, :, off, :].permute(1, 0, 2)
        c0 = int(meta.cu_q_lens[s])
        Q[s, :, :qs] = qf[c0:c0 + qs].permute(1, 0, 2)
        for i in range(qs):
            mask[s, 0, i, :ctx - qs + i + 1] = True
    Kx = K.repeat_interleave(g, dim=1)
    Vx = V.repeat_interleave(g, dim=1)
    O = torch.nn.functional.scaled_dot_product_attention(Q, Kx, Vx, attn_mask=mask, scale=scale)
    out = torch.zeros(meta.total_q, hq, d, dtype=torch.float64)
    for s in range(B):
        c0, qs = int(meta.cu_q_lens[s]), int(meta.q_lens[s])
        out[c0:c0 + qs] = O[s, :, :qs].permute(1, 0, 2)
    return out.numpy()


def run_oracle(meta, q, pool, scale=None, **kw):
    return oracle.paged_varlen_attention(q, meta.cu_q_lens, meta.context_lens, meta.block_tables,
                                         pool, meta.scale if scale is None else scale, **kw)


# ----------------------------------------------------------------------------
# brute force
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(12))
def test_oracle_matches_padded_sdpa(seed):
    rng = np.random.default_rng(100 + seed)
    meta = workloads.random_step(rng, max_ctx=90)
    q, _, _, pool = workloads.make_values(meta)
    got = run_oracle(meta, q, pool)
    ref = brute_force(meta, q, pool)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_oracle_tiny_decode_matches_padded_sdpa():
    meta = workloads.tiny_decode()
    q, _, _, pool = workloads.make_values(meta)
    np.testing.assert_allclose(run_oracle(meta, q, pool), brute_force(meta, q, pool), rtol=0, atol=1e-12)


def test_oracle_row_subset_equals_full():
    rng = np.random.default_rng(7)
    meta = workloads.random_step(rng, num_seqs=4, max_ctx=70)
    q, _, _, pool = workloads.make_values(meta)
    full = run_oracle(meta, q, pool).reshape(-1, meta.head_dim)
    rows = rng.choice(full.shape[0], size=min(25, full.shape[0]), replace=False)
    sub = run_oracle(meta, q, pool, rows=rows)
    np.testing.assert_array_equal(sub, full[rows])


def test_oracle_thread_count_does_not_change_bits():
    rng = np.random.default_rng(8)
    meta = workloads.random_step(rng, num_seqs=5, max_ctx=120)
    q, _, _, pool = workloads.make_values(meta)
    np.testing.assert_array_equal(run_oracle(meta, q, pool, num_threads=1),
                                  run_oracle(meta, q, pool, num_threads=3))


# ----------------------------------------------------------------------------
# hand-derived fixtures
# ----------------------------------------------------------------------------

def _golden_cases():
    with open(os.path.join(GOLDEN, "closed_form_cases.json")) as f:
        return json.load(f)["cases"]


def _scale(s):
    return {"ln3": math.log(3.0), "ln2": math.log(2.0)}.get(s, None) or float(s)


def _vec(sparse, d, dtype=np.float32):
    v = np.zeros(d, dtype=dtype)
    for k, x in sparse.items():
        v[int(k)] = x
    return v


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_oracle_golden_closed_forms(case):
    hq, hkv, d, bs, nb = (case[k] for k in ("num_q_heads", "num_kv_heads", "head_dim", "block_size", "num_blocks"))
    seqs = case["seqs"]
    q_lens = [s["q_len"] for s in seqs]
    ctx = [s["ctx"] for s in seqs]
    maxb = max(len(s["block_table"]) for s in seqs)
    tables = np.full((len(seqs), maxb), -1, np.int32)
    for i, s in enumerate(seqs):
        tables[i, :len(s["block_table"])] = s["block_table"]
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    poolf = np.full((nb, 2, hkv, bs, d), 99.0, np.float32)   # garbage in unused slots
    for si, s in enumerate(seqs):
        for h in range(hkv):
            for p in range(s["ctx"]):
                b, o = s["block_table"][p // bs], p % bs
                poolf[b, 0, h, o] = _vec(case["keys"][si][h][p], d)
                poolf[b, 1, h, o] = _vec(case["values"][si][h][p], d)
    qf = np.stack([np.stack([_vec(case["q"][t][h], d) for h in range(hq)]) for t in range(int(cu[-1]))])
    pool = torch.from_numpy(poolf).to(torch.bfloat16)
    q = torch.from_numpy(qf).to(torch.bfloat16)
    assert torch.equal(pool.float(), torch.from_numpy(poolf)), "fixture values must be bf16-exact"
    got = oracle.paged_varlen_attention(q, cu, np.asarray(ctx, np.int32), tables, pool, _scale(case["scale"]))
    exp = np.stack([np.stack([_vec(case["expected"][t][h], d, np.float64) for h in range(hq)])
                    for t in range(int(cu[-1]))])
    np.testing.assert_allclose(got, exp, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------
# invariants
# ----------------------------------------------------------------------------

def test_block_permutation_invariance():
    rng = np.random.default_rng(11)
    meta = workloads.random_step(rng, num_seqs=5, max_ctx=150)
    q, _, _, pool = workloads.make_values(meta)
    base = run_oracle(meta, q, pool)
    perm = rng.permutation(meta.num_blocks)          # new physical id of old block b
    pool2 = torch.empty_like(pool)
    pool2[torch.from_numpy(perm)] = pool
    tables2 = np.where(meta.block_tables >= 0, perm[np.maximum(meta.block_tables, 0)], -1).astype(np.int32)
    got = oracle.paged_varlen_attention(q, meta.cu_q_lens, meta.context_lens, tables2, pool2, meta.scale)
    np.testing.assert_array_equal(got, base)


def test_constant_v_returns_constant():
    rng = np.random.default_rng(12)
    meta = workloads.random_step(rng, num_seqs=4, max_ctx=120)
    q, _, _, pool = workloads.make_values(meta)
    pool[:, 1] = -0.6875
    got = run_oracle(meta, q, pool)
    np.testing.assert_allclose(got, -0.6875, rtol=0, atol=1e-14)


def test_single_visible_key_returns_its_value():
    # ctx = 1 decode, and the first query of a chunk that covers the whole context
    meta = workloads.build_step("t", 5, [1, 7], [1, 7], 4, 2, 64, pool_blocks=6)
    q, _, _, pool = workloads.make_values(meta)
    out = run_oracle(meta, q, pool)
    for s, tok in ((0, 0), (1, int(meta.cu_q_lens[1]))):
        b = int(meta.block_tables[s, 0])
        for hq in range(4):
            np.testing.assert_array_equal(out[tok, hq], pool[b, 1, hq // 2, 0].to(torch.float64).numpy())


def test_scale_zero_gives_mean_of_visible_values():
    rng = np.random.default_rng(13)
    meta = workloads.random_step(rng, num_seqs=4, max_ctx=100)
    q, _, _, pool = workloads.make_values(meta)
    got = run_oracle(meta, q, pool, scale=0.0)
    g = meta.num_q_heads // meta.num_kv_heads
    pf = pool.to(torch.float64).numpy()
    for s in range(meta.num_seqs):
        ctx, qs, c0 = int(meta.context_lens[s]), int(meta.q_lens[s]), int(meta.cu_q_lens[s])
        for i in range(qs):
            n = ctx - qs + i + 1
            pos = np.arange(n)
            vals = pf[meta.block_tables[s, pos // 16], 1, :, pos % 16, :]   # [n, hkv, d]
            mean = vals.mean(axis=0)
            for hq in range(meta.num_q_heads):
                np.testing.assert_allclose(got[c0 + i, hq], mean[hq // g], rtol=0, atol=1e-13)


def test_one_hot_query_with_large_scale_picks_argmax_key():
    meta = workloads.build_step("t", 9, [1], [40], 2, 1, 64, pool_blocks=5)
    q, _, _, pool = workloads.make_values(meta)
    q.zero_()
    q[0, :, 17] = 1.0
    pool[:, 0, :, :, 17] = 0.5
    target = 29
    b, o = int(meta.block_tables[0, target // 16]), target % 16
    pool[b, 0, 0, o, 17] = 1.0
    out = run_oracle(meta, q, pool, scale=5000.0)
    want = pool[b, 1, 0, o].to(torch.float64).numpy()
    for hq in range(2):
        np.testing.assert_array_equal(out[0, hq], want)


def test_shared_prefix_equals_unshared_copies():
    rng = np.random.default_rng(14)
    meta = workloads.random_step(rng, num_seqs=4, max_ctx=100, shared_prefix_blocks=3)
    q, _, _, pool = workloads.make_values(meta)
    shared = run_oracle(meta, q, pool)
    # give every sequence its own copy of the prefix blocks
    extra = 3 * meta.num_seqs
    pool2 = torch.cat([pool, torch.zeros((extra,) + tuple(pool.shape[1:]), dtype=pool.dtype)])
    tables2 = meta.block_tables.copy()
    nxt = meta.num_blocks
    for s in range(meta.num_seqs):
        for j in range(3):
            pool2[nxt] = pool[meta.block_tables[s, j]]
            tables2[s, j] = nxt
            nxt += 1
    assert len({int(meta.block_tables[s, 0]) for s in range(meta.num_seqs)}) == 1
    got = oracle.paged_varlen_attention(q, meta.cu_q_lens, meta.context_lens, tables2, pool2, meta.scale)
    np.testing.assert_array_equal(got, shared)


def test_decode_row_equals_last_prefill_row():
    pre = workloads.build_step("t", 21, [9], [30], 6, 3, 128, pool_blocks=4)
    q, _, _, pool = workloads.make_values(pre)
    full = run_oracle(pre, q, pool)
    dec_cu = np.array([0, 1], np.int32)
    got = oracle.paged_varlen_attention(q[8:9], dec_cu, pre.context_lens, pre.block_tables, pool, pre.scale)
    np.testing.assert_array_equal(got[0], full[8])


def test_chunk_split_invariance():
    """A prefill chunk computed in one step equals the same chunk computed in two
    consecutive steps (the chunk-boundary caveat of the vllm-ios page's prefix
    caching note concerns greedy downstream ties, not the attention values)."""
    meta = workloads.build_step("t", 22, [37], [50], 8, 2, 64, pool_blocks=6)
    q, _, _, pool = workloads.make_values(meta)
    full = run_oracle(meta, q, pool)
    n1 = 15
    a = oracle.paged_varlen_attention(q[:n1], np.array([0, n1], np.int32), np.array([50 - 37 + n1], np.int32),
                                      meta.block_tables, pool, meta.scale)
    b = oracle.paged_varlen_attention(q[n1:], np.array([0, 37 - n1], np.int32), meta.context_lens,
                                      meta.block_tables, pool, meta.scale)
    np.testing.assert_array_equal(np.concatenate([a, b]), full)


def test_batch_composition_invariance():
    rng = np.random.default_rng(15)
    meta = workloads.random_step(rng, num_seqs=5, max_ctx=80)
    q, _, _, pool = workloads.make_values(meta)
    full = run_oracle(meta, q, pool)
    for s in range(meta.num_seqs):
        c0, c1 = int(meta.cu_q_lens[s]), int(meta.cu_q_lens[s + 1])
        alone = oracle.paged_varlen_attention(q[c0:c1], np.array([0, c1 - c0], np.int32),
                                              meta.context_lens[s:s + 1], meta.block_tables[s:s + 1],
                                              pool, meta.scale)
        np.testing.assert_array_equal(alone, full[c0:c1])


def test_rejects_bad_metadata():
    meta = workloads.build_step("t", 23, [2], [20], 2, 1, 64, pool_blocks=4)
    q, _, _, pool = workloads.make_values(meta)
    with pytest.raises(ValueError):   # q_len > ctx
        oracle.paged_varlen_attention(q, meta.cu_q_lens, np.array([1], np.int32), meta.block_tables, pool, 1.0)
    bt = meta.block_tables.copy()
    bt[0, 1] = 4                      # block id outside the pool
    with pytest.raises(ValueError):
        oracle.paged_varlen_attention(q, meta.cu_q_lens, meta.context_lens, bt, pool, 1.0)
    assert oracle.check_step(np.array([1, 2], np.int32), meta.context_lens, bt, 4, 16) != 0


# ----------------------------------------------------------------------------
# append
# ----------------------------------------------------------------------------

def numpy_scatter(pool_bits, kb, vb, slots, bs):
    out = pool_bits.copy()
    for t, slot in enumerate(slots):
        if slot < 0 or slot >= out.shape[0] * bs:
            continue
        out[slot // bs, 0, :, slot % bs, :] = kb[t]
        out[slot // bs, 1, :, slot % bs, :] = vb[t]
    return out


@pytest.mark.parametrize("name", ["tiny_decode", "small_decode", "agent_mixed", "shared_prefix_verify"])
def test_append_matches_numpy_scatter(name):
    meta = workloads.make_config(name)
    _, k, v, pool = workloads.make_values(meta)
    got, bad = oracle.paged_kv_append(pool, k, v, meta.slot_mapping, block_size=meta.block_size)
    assert bad == 0
    want = numpy_scatter(bits(pool), bits(k), bits(v), meta.slot_mapping, meta.block_size)
    np.testing.assert_array_equal(got, want)
    # round trip: gathering the appended slots returns k and v bit for bit
    sl = meta.slot_mapping
    np.testing.assert_array_equal(got[sl // 16, 0, :, sl % 16, :], bits(k))
    np.testing.assert_array_equal(got[sl // 16, 1, :, sl % 16, :], bits(v))


def test_append_padding_and_out_of_range_slots():
    meta = workloads.tiny_decode()
    _, k, v, pool = workloads.make_values(meta)
    slots = meta.slot_mapping.copy()
    slots[1] = -1
    slots[2] = meta.num_blocks * 16        # first slot past the pool
    got, bad = oracle.paged_kv_append(pool, k, v, slots, block_size=16)
    assert bad == 1
    want = numpy_scatter(bits(pool), bits(k), bits(v), slots, 16)
    np.testing.assert_array_equal(got, want)
    # tokens 1 and 2 were not written anywhere
    changed = np.any(got != bits(pool), axis=(1, 2, 3, 4))
    assert set(np.nonzero(changed)[0]) <= {int(meta.slot_mapping[0]) // 16, int(meta.slot_mapping[3]) // 16}


def test_append_then_attend_sees_new_token():
    """A decode whose new token is its only key returns the appended V row."""
    meta = workloads.build_step("t", 31, [1], [1], 2, 1, 64, pool_blocks=3)
    q, k, v, pool = workloads.make_values(meta)
    out, pool_after = oracle.run_step(meta, q, k, v, pool)
    np.testing.assert_array_equal(out[0, 0], v[0, 0].to(torch.float64).numpy())
    np.testing.assert_array_equal(out[0, 1], v[0, 0].to(torch.float64).numpy())


# ------------------------------------------------------------------ state checkpoint

def test_state_checkpoint_equals_indexed_assignment():
    """Rows land where their slots say, byte for byte, by a second route (numpy
    indexed assignment); negative slots write nothing; other rows are untouched."""
    rng = np.random.default_rng(7)
    num_slots, row_bytes, n = 50, 48, 20
    pool = rng.integers(0, 256, size=(num_slots, row_bytes), dtype=np.uint8)
    src = rng.integers(0, 256, size=(n, row_bytes), dtype=np.uint8)
    slots = rng.permutation(num_slots)[:n].astype(np.int32)
    slots[[3, 11]] = -1
    got, bad = oracle.state_checkpoint(pool, src, slots)
    want = pool.copy()
    keep = slots >= 0
    want[slots[keep]] = src[keep]
    assert bad == 0 and np.array_equal(got, want)
    untouched = np.setdiff1d(np.arange(num_slots), slots[keep])
    assert np.array_equal(got[untouched], pool[untouched])


def test_state_checkpoint_bad_slots_and_empty():
    pool = np.arange(4 * 16, dtype=np.uint8).reshape(4, 16)
    src = np.full((3, 16), 255, dtype=np.uint8)
    got, bad = oracle.state_checkpoint(pool, src, np.array([4, -1, 1], dtype=np.int32))
    assert bad == 1                                  # slot 4 is past the pool: skipped
    want = pool.copy()
    want[1] = 255
    assert np.array_equal(got, want)
    got0, bad0 = oracle.state_checkpoint(pool, src[:0], np.zeros(0, dtype=np.int32))
    assert bad0 == 0 and np.array_equal(got0, pool)
