"""Seeded synthetic inputs for one packed attention step over a paged KV cache.

This module is shared by the tests, the benchmark and the oracle's callers.  It
builds the *inputs* of a step only -- sequence lengths, block tables, slot
mappings and bf16 tensors drawn from N(0, 1) -- and holds none of the method's
arithmetic (no gather, no softmax, no append).

The five named workloads follow the step shapes of the vllm-metal v0.4.0 release
page ("Replacing attention, reusing the rest": a packed query axis with
cu_seqlens, KV in fixed-size pages located through per-request block tables,
one launch covering prefill chunks, decode tokens and speculative-verify
windows).  The numeric shapes (head counts, length distributions, pool sizing)
are the benchmark configurations of this library; readings the pages leave open
are stated beside each one.

Conventions used everywhere in this repository:

* ``q``      bf16 ``[total_q, Hq, D]``, packed in sequence order.
* ``k_new``, ``v_new`` bf16 ``[total_q, Hkv, D]``: this step's keys/values.
* ``kv_pool`` bf16 ``[num_blocks, 2, Hkv, block_size, D]`` (index 0 = K, 1 = V).
* ``cu_q_lens`` int32 ``[num_seqs + 1]``, ``context_lens`` int32 ``[num_seqs]``
  (context length *including* this step's new tokens).
* ``block_tables`` int32 ``[num_seqs, max_blocks_per_seq]``, unused entries -1.
* ``slot_mapping`` int32 ``[total_q]``: physical slot ``block * block_size +
  offset`` of each new token; a negative slot means "skip" (padding).
* Query token ``i`` of sequence ``s`` sits at position ``ctx_s - q_s + i`` and
  sees keys ``0 .. ctx_s - q_s + i`` (causal within the query chunk).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK_SIZE = 16


@dataclasses.dataclass
class StepMeta:
    """Host-side description of one packed step (all arrays are numpy)."""

    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q_lens: np.ndarray          # int32 [num_seqs]
    context_lens: np.ndarray    # int32 [num_seqs]
    cu_q_lens: np.ndarray       # int32 [num_seqs + 1]
    block_tables: np.ndarray    # int32 [num_seqs, max_blocks]
    slot_mapping: np.ndarray    # int32 [total_q]
    scale: float
    notes: str = ""

    @property
    def num_seqs(self) -> int:
        return int(self.q_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.cu_q_lens[-1])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    def kv_tokens(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())

    def unique_blocks(self) -> int:
        """Distinct physical blocks read by the step (shared prefixes counted once)."""
        used = set()
        for s in range(self.num_seqs):
            nb = -(-int(self.context_lens[s]) // self.block_size)
            used.update(int(b) for b in self.block_tables[s, :nb])
        return len(used)


def _cu(q_lens: np.ndarray) -> np.ndarray:
    cu = np.zeros(len(q_lens) + 1, dtype=np.int64)
    np.cumsum(q_lens, out=cu[1:])
    return cu.astype(np.int32)


def _slots(q_lens, ctx_lens, tables, bs) -> np.ndarray:
    out = []
    for s in range(len(q_lens)):
        for i in range(int(q_lens[s])):
            pos = int(ctx_lens[s]) - int(q_lens[s]) + i
            out.append(int(tables[s, pos // bs]) * bs + pos % bs)
    return np.asarray(out, dtype=np.int32)


def build_step(name, seed, q_lens, ctx_lens, hq, hkv, d, *, pool_blocks=None,
               shared_prefix_blocks=0, bs=BLOCK_SIZE, scale=None, notes="",
               rng=None, append=True) -> StepMeta:
    """Assign physical blocks by a seeded random permutation and derive slots.

    ``shared_prefix_blocks`` > 0 makes every sequence's first that many logical
    blocks point at the same physical blocks (a shared prompt prefix).
    ``pool_blocks`` defaults to the distinct blocks needed + 10 %.
    ``append=False`` marks every query token's slot as skip (-1): the step
    attends over K/V already in the pool and writes none (a draft pass over the
    target's cache).
    """
    rng = np.random.default_rng(seed) if rng is None else rng
    q_lens = np.asarray(q_lens, dtype=np.int32)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
    assert np.all(q_lens <= ctx_lens)
    nblk = [-(-int(c) // bs) for c in ctx_lens]
    private = [max(0, n - shared_prefix_blocks) for n in nblk]
    needed = shared_prefix_blocks + sum(private)
    if pool_blocks is None:
        pool_blocks = int(math.ceil(needed * 1.1))
    assert pool_blocks >= needed
    perm = rng.permutation(pool_blocks).astype(np.int32)
    max_blocks = max(nblk) if nblk else 1
    tables = np.full((len(q_lens), max_blocks), -1, dtype=np.int32)
    shared = perm[:shared_prefix_blocks]
    nxt = shared_prefix_blocks
    for s, n in enumerate(nblk):
        k = min(n, shared_prefix_blocks)
        tables[s, :k] = shared[:k]
        tables[s, k:n] = perm[nxt:nxt + (n - k)]
        nxt += n - k
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return StepMeta(name=name, seed=seed, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=d, block_size=bs, num_blocks=pool_blocks,
                    q_lens=q_lens, context_lens=ctx_lens, cu_q_lens=_cu(q_lens),
                    block_tables=tables,
                    slot_mapping=(_slots(q_lens, ctx_lens, tables, bs) if append else
                                  np.full(int(q_lens.sum()), -1, dtype=np.int32)),
                    scale=float(scale), notes=notes)


# ---------------------------------------------------------------------------
# The five benchmark workloads.  Seed = 1234 + index unless given.
# ---------------------------------------------------------------------------

def tiny_decode(seed=1234):
    """4 decodes, contexts {17,33,64,100}, 8 q heads / 2 KV heads, D=64,
    a 64-block pool placed by a seeded random permutation, scale 1/sqrt(64)."""
    return build_step("tiny_decode", seed, [1, 1, 1, 1], [17, 33, 64, 100], 8, 2, 64,
                      pool_blocks=64)


def small_decode(seed=1235):
    """16 decodes, contexts uniform integer in [512, 4096], 16 q / 8 KV heads,
    D=128, pool = distinct blocks + 10 %."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(512, 4096, size=16, endpoint=True)
    return build_step("small_decode", seed, [1] * 16, ctx, 16, 8, 128, rng=rng)


def agent_mixed(seed=1236):
    """A 2048-token chunked-prefill query at prior context 2560 (ctx 4608, causal
    within the chunk) packed with 3 decodes whose contexts are N(4600, 800)
    clipped to [2048, 8192]; 40 q / 8 KV heads, D=128."""
    rng = np.random.default_rng(seed)
    dec = np.clip(np.rint(rng.normal(4600.0, 800.0, size=3)), 2048, 8192).astype(np.int32)
    return build_step("agent_mixed", seed, [2048, 1, 1, 1], [2560 + 2048, *dec], 40, 8, 128,
                      rng=rng)


LOGNORMAL_SIGMA = 1.0


def high_conc_decode(seed=1237, num_seqs=256):
    """256 decodes, contexts lognormal with median 2048 (sigma = 1.0 in log space,
    a reading: the spread is not given), rounded and clipped to [64, 32768];
    32 q / 8 KV heads, D=128, blocks scattered over a pool of distinct + 10 %."""
    rng = np.random.default_rng(seed)
    ctx = np.clip(np.rint(rng.lognormal(math.log(2048.0), LOGNORMAL_SIGMA, size=num_seqs)),
                  64, 32768).astype(np.int32)
    return build_step("high_conc_decode", seed, [1] * num_seqs, ctx, 32, 8, 128, rng=rng,
                      notes=f"lognormal sigma={LOGNORMAL_SIGMA}")


def shared_prefix_verify(seed=1238, num_seqs=64):
    """64 sequences whose first 256 blocks (a 4096-token prefix) are the same
    physical blocks, each with a private suffix of uniform length in [0, 1024]
    followed by 2 query tokens (a draft-verify pair, causal within the pair);
    32 q / 8 KV heads, D=128."""
    rng = np.random.default_rng(seed)
    suffix = rng.integers(0, 1024, size=num_seqs, endpoint=True)
    ctx = 4096 + suffix + 2
    return build_step("shared_prefix_verify", seed, [2] * num_seqs, ctx, 32, 8, 128,
                      shared_prefix_blocks=256, rng=rng)


def long_context_mix(seed=1239):
    """The vllm-metal page's packed-step example, "30,000 + 5,000 + 10" tokens
    ("Replacing attention, reusing the rest", the padded-rectangle figure): three
    requests prefilled in one step, each from an empty cache (context = query
    length; a reading, the page gives only the token counts), with the mixed
    step's model shape, 40 q / 8 KV heads, D=128 (also a reading: the example
    names no model)."""
    return build_step("long_context_mix", seed, [30000, 5000, 10], [30000, 5000, 10], 40, 8, 128)


def mtp_draft(seed=1240, num_seqs=64):
    """The batched draft pass of the vllm-metal page ("Batched MTP under
    concurrent load"): every request's seed token in one packed dispatch against
    the target's shared KV cache, nothing appended (the seed's K/V is already
    cached).  The shared-prefix step's shapes: 64 requests on a shared 4096-token
    prefix plus a private suffix U[0, 1024], 1 query each, 32 q / 8 KV heads,
    D=128."""
    rng = np.random.default_rng(seed)
    suffix = rng.integers(0, 1024, size=num_seqs, endpoint=True)
    ctx = 4096 + suffix + 1
    return build_step("mtp_draft", seed, [1] * num_seqs, ctx, 32, 8, 128,
                      shared_prefix_blocks=256, rng=rng, append=False)


def wide_verify(seed=1241, num_seqs=64):
    """Verify windows wider than the page's 2 ("values above 1 are ignored" in
    its MTP runs): 64 requests, alternately 4 and 8 query tokens (3 or 7 draft
    tokens plus the seed, causal within the window), contexts uniform in
    [1024, 8192], 32 q / 8 KV heads, D=128."""
    rng = np.random.default_rng(seed)
    ql = np.array([4, 8] * (num_seqs // 2), dtype=np.int32)
    ctx = rng.integers(1024, 8192, size=num_seqs, endpoint=True)
    return build_step("wide_verify", seed, ql, ctx, 32, 8, 128, rng=rng)


def decode_chain(seed=1243, steps=8):
    """The small-model decode batch run as a chain of `steps` decode steps in one
    graph (the vllm-metal page's "Chained greedy decode", 4-8 tokens a chunk):
    16 decodes, first-step contexts uniform in [512, 4096], 16 q / 8 KV heads,
    D=128; block tables already hold the blocks of the last step.  Returns the
    first step; each later step adds one token per sequence."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(512, 4096, size=16, endpoint=True).astype(np.int32)
    last = build_step("decode_chain", seed, [1] * 16, ctx + (steps - 1), 16, 8, 128, rng=rng,
                      notes=f"chain_steps={steps}")
    return chain_step(last, ctx, 0)


def chain_step(last: StepMeta, ctx0, t: int) -> StepMeta:
    """Step t of a decode chain whose last step is `last` and whose first-step
    contexts are ctx0: contexts ctx0 + t * q_len, slots of the new positions."""
    ctx = (np.asarray(ctx0, dtype=np.int32) + t * last.q_lens).astype(np.int32)
    slots = []
    for s in range(last.num_seqs):
        for i in range(int(last.q_lens[s])):
            pos = int(ctx[s]) - int(last.q_lens[s]) + i
            slots.append(int(last.block_tables[s, pos // last.block_size]) * last.block_size +
                         pos % last.block_size)
    return StepMeta(**{**last.__dict__, "context_lens": ctx,
                       "slot_mapping": np.array(slots, dtype=np.int32)})


def chain_steps(meta: StepMeta) -> int:
    """Chain length recorded in a chained workload's notes (1 for a single step)."""
    for tok in meta.notes.split():
        if tok.startswith("chain_steps="):
            return int(tok.split("=", 1)[1])
    return 1


CONFIGS = {
    "tiny_decode": tiny_decode,
    "small_decode": small_decode,
    "agent_mixed": agent_mixed,
    "high_conc_decode": high_conc_decode,
    "shared_prefix_verify": shared_prefix_verify,
    "long_context_mix": long_context_mix,
    "mtp_draft": mtp_draft,
    "wide_verify": wide_verify,
    "decode_chain": decode_chain,
}


def make_config(name: str, seed: int | None = None) -> StepMeta:
    fn = CONFIGS[name]
    return fn() if seed is None else fn(seed)


def random_step(rng: np.random.Generator, *, num_seqs=None, hkv=None, group=None, d=None,
                max_ctx=200, max_q=None, pool_extra=1.3, shared_prefix_blocks=0) -> StepMeta:
    """A small random mixed step for property tests (decodes, verifies, prefills)."""
    num_seqs = int(rng.integers(1, 6)) if num_seqs is None else num_seqs
    hkv = int(rng.choice([1, 2, 4])) if hkv is None else hkv
    group = int(rng.choice([1, 2, 3, 4, 5, 8])) if group is None else group
    d = int(rng.choice([64, 128])) if d is None else d
    ctx = rng.integers(1, max_ctx + 1, size=num_seqs)
    if shared_prefix_blocks:
        ctx = np.maximum(ctx, shared_prefix_blocks * BLOCK_SIZE + 1)
    q = []
    for c in ctx:
        kind = rng.integers(0, 3)
        mq = int(c) if max_q is None else min(int(c), max_q)
        q.append(1 if kind == 0 else min(int(c), 2) if kind == 1 else int(rng.integers(1, mq + 1)))
    if shared_prefix_blocks:
        # the step's new tokens land past the shared blocks: two sequences never
        # write the same slot of a block they share
        ctx = np.maximum(ctx, shared_prefix_blocks * BLOCK_SIZE + np.array(q))
    nb = sum(-(-int(c) // BLOCK_SIZE) for c in ctx)
    return build_step("random", int(rng.integers(1 << 30)), q, ctx, hkv * group, hkv, d,
                      pool_blocks=int(nb * pool_extra) + 2,
                      shared_prefix_blocks=shared_prefix_blocks, rng=rng)


# ---------------------------------------------------------------------------
# Tensor values.  bf16 N(0, 1): float32 normals rounded to bf16.
# ---------------------------------------------------------------------------

def _normal_bf16(rng, shape):
    import torch
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def make_values(meta: StepMeta, seed: int | None = None, device="cpu"):
    """Return (q, k_new, v_new, kv_pool) as bf16 torch tensors.

    On the CPU the values come from numpy's PCG64 stream (reproducible across
    machines).  On a CUDA device they come from torch's seeded CUDA generator,
    which fills multi-GB pools in milliseconds; callers that need the same
    values on the host copy the device tensors back.
    """
    import torch
    seed = meta.seed if seed is None else seed
    shp_q = (meta.total_q, meta.num_q_heads, meta.head_dim)
    shp_kv = (meta.total_q, meta.num_kv_heads, meta.head_dim)
    shp_pool = (meta.num_blocks, 2, meta.num_kv_heads, meta.block_size, meta.head_dim)
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = np.random.default_rng(seed + 7919)
        return (_normal_bf16(rng, shp_q), _normal_bf16(rng, shp_kv),
                _normal_bf16(rng, shp_kv), _normal_bf16(rng, shp_pool))
    g = torch.Generator(device=dev)
    g.manual_seed(seed + 7919)
    out = []
    for shp in (shp_q, shp_kv, shp_kv, shp_pool):
        t = torch.empty(shp, dtype=torch.bfloat16, device=dev)
        flat = t.view(-1)
        chunk = 1 << 28
        for i in range(0, flat.numel(), chunk):
            n = min(chunk, flat.numel() - i)
            flat[i:i + n] = torch.randn(n, generator=g, device=dev, dtype=torch.float32)
        out.append(t)
    return tuple(out)


def describe(meta: StepMeta) -> dict:
    return {
        "workload": meta.name,
        "seed": meta.seed,
        "num_seqs": meta.num_seqs,
        "total_q": meta.total_q,
        "kv_tokens": meta.kv_tokens(),
        "num_q_heads": meta.num_q_heads,
        "num_kv_heads": meta.num_kv_heads,
        "head_dim": meta.head_dim,
        "block_size": meta.block_size,
        "num_blocks": meta.num_blocks,
        **({"notes": meta.notes} if meta.notes else {}),
    }
