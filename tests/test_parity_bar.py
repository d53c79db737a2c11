"""The bf16-floor parity bar, pinned on the CPU.

The GPU parity tests apply two bars (tests/parity_bar.py).  These checks show
the floor bar does what it is for:

* it accepts the oracle rounded once to bf16 (an ideal kernel's output);
* it accepts an fp32 evaluation with P rounded to bf16 before the P V product
  (the arithmetic the kernels use), written here with numpy for a few rows;
* it rejects the oracle's result for the same rows with one 16-key block
  dropped (the mistake planted in the oracle's input: each row's context cut
  by one block), at contexts where the acceptance bar alone lets it through.
"""

import numpy as np
import pytest
import torch

import oracle
import parity_bar
import workloads


def _decode_step(ctx, seed):
    # one KV head, 4 query heads, one decode token per sequence, D = 128
    return workloads.build_step("bar", seed, [1] * len(ctx), ctx, 4, 1, 128)


def _kernel_like(meta, q, pool):
    """fp32 scores and softmax, P rounded to bf16 for P V, fp32 sums, output
    rounded to bf16: decode rows only (q_len = 1), all keys visible."""
    d, g = meta.head_dim, meta.num_q_heads // meta.num_kv_heads
    out = np.zeros((meta.total_q, meta.num_q_heads, d))
    qf = q.to(torch.float32).numpy()
    pf = pool.to(torch.float32).numpy()
    for s in range(meta.num_seqs):
        ctx = int(meta.context_lens[s])
        nb = -(-ctx // 16)
        blocks = meta.block_tables[s, :nb]
        for hq in range(meta.num_q_heads):
            h = hq // g
            kk = pf[blocks, 0, h].reshape(-1, d)[:ctx]
            vv = pf[blocks, 1, h].reshape(-1, d)[:ctx]
            x = (kk @ qf[s, hq]).astype(np.float32) * np.float32(meta.scale)
            p = np.exp(x - x.max()).astype(np.float32)
            l = p.sum(dtype=np.float32)
            pb = torch.from_numpy(p).to(torch.bfloat16).to(torch.float32).numpy()
            o = (pb @ vv).astype(np.float32) / l
            out[s, hq] = torch.from_numpy(o).to(torch.bfloat16).to(torch.float64).numpy()
    return out


@pytest.mark.parametrize("ctx", [[4000, 4100], [8000], [30000, 32768]])
def test_floor_bar_rejects_a_dropped_block(ctx):
    meta = _decode_step(ctx, 11 + len(ctx))
    q, k, v, pool = workloads.make_values(meta)
    want, pool_after = oracle.run_step(meta, q, k, v, pool)
    pool_t = torch.from_numpy(pool_after.view(np.int16)).view(torch.bfloat16).reshape(pool.shape)

    ideal = parity_bar.evaluate(parity_bar.bf16_round(want), want)
    assert ideal["acceptance_ok"] and ideal["floor_ok"], ideal
    assert ideal["floor_ratio"] == pytest.approx(1.0)

    emul = parity_bar.evaluate(_kernel_like(meta, q, pool_t), want)
    assert emul["acceptance_ok"] and emul["floor_ok"], emul

    # the planted mistake: every row misses its last 16 keys
    short = workloads.StepMeta(**{**meta.__dict__,
                                  "context_lens": (meta.context_lens - 16).astype(np.int32),
                                  "slot_mapping": np.full(meta.total_q, -1, np.int32)})
    dropped, _ = oracle.run_step(short, q, k, v, pool_t)
    bad = parity_bar.evaluate(parity_bar.bf16_round(dropped), want)
    assert not bad["floor_ok"], bad
    if min(ctx) >= 8000:
        # the acceptance bar alone does not see it at these contexts
        assert bad["acceptance_ok"], bad


def test_bf16_round_is_round_to_nearest_even():
    # values exactly between two bf16 numbers go to the one with an even mantissa
    one_ulp = 2.0 ** -7
    x = np.array([1.0 + one_ulp / 2, 1.0 + 3 * one_ulp / 2, -(1.0 + one_ulp / 2),
                  1.0 + one_ulp / 2 + 1e-12, 3.0e-3, 0.0, 1234.5])
    r = parity_bar.bf16_round(x)
    assert r[0] == 1.0 and r[1] == 1.0 + 2 * one_ulp and r[2] == -1.0
    assert r[3] == 1.0 + one_ulp
    # agrees with torch's float32 -> bf16 rounding where the value is a float32
    f = np.float64(np.float32(3.0e-3))
    assert parity_bar.bf16_round(np.array([f]))[0] == float(
        torch.tensor([f], dtype=torch.float32).to(torch.bfloat16).double())
    assert r[5] == 0.0 and r[6] == 1232.0
