"""The allocation-free attention entry point, called through the C ABI.

pkv_paged_varlen_attention_noalloc serves callers that cannot allocate device
memory (no cudaMalloc available or allowed): its split-KV scratch is a fixed
array in the library's device image instead of a caller workspace.  This test
checks that two calls in a row (the second one sees the first one's leftover
scratch contents) give the same output as the workspace entry point, within
the attention tolerance used by the other GPU tests.  It lives in its own file,
collected last, and needs no state from other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
NOALLOC_LIMIT = 16 * 1024 * 1024


@pytest.fixture(scope="module")
def pkv(cuda_device):
    import paged_kv_attention_append_gb300 as m
    m.build()
    return m


def _noalloc_fn(pkv):
    lib = ctypes.CDLL(pkv.library_path())
    fn = lib.pkv_paged_varlen_attention_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [P, P, P, P, ctypes.c_int32, P, ctypes.POINTER(pkv.PoolDesc), ctypes.c_float,
                   ctypes.POINTER(pkv.PlanInfo), P, P, P, P]
    fn.restype = ctypes.c_int32
    return fn


def _step(pkv, meta, dev):
    q, k, v, pool = workloads.make_values(meta, device=dev)
    pkv.paged_kv_append(k, v, torch.from_numpy(meta.slot_mapping).to(dev), pool)
    cu = torch.from_numpy(meta.cu_q_lens).to(dev)
    ctx = torch.from_numpy(meta.context_lens).to(dev)
    bt = torch.from_numpy(meta.block_tables).to(dev)
    plan = pkv.plan_step(meta.cu_q_lens, meta.context_lens, meta.num_q_heads, pool)
    return q, pool, cu, ctx, bt, plan


def _call(fn, pkv, meta, q, pool, cu, ctx, bt, plan, out, status, stream):
    desc = pkv.pool_desc(pool)
    return fn(q.data_ptr(), cu.data_ptr(), ctx.data_ptr(), bt.data_ptr(), bt.shape[1],
              pool.data_ptr(), ctypes.byref(desc), meta.scale, ctypes.byref(plan.info),
              plan.dev.data_ptr(), out.data_ptr(), status.data_ptr(), stream.cuda_stream)


def _close(a, b):
    d = (a.double() - b.double()).abs()
    assert torch.isfinite(a.double()).all()
    assert float(d.max()) <= MAX_ABS and float(d.mean()) <= MEAN_ABS, (float(d.max()), float(d.mean()))


def test_noalloc_matches_workspace_entry_point_twice(pkv, cuda_device):
    fn = _noalloc_fn(pkv)
    stream = torch.cuda.current_stream(cuda_device)
    steps = [workloads.small_decode(), workloads.shared_prefix_verify()]
    results = []
    for meta in steps:
        q, pool, cu, ctx, bt, plan = _step(pkv, meta, cuda_device)
        assert 0 < plan.info.workspace_bytes <= NOALLOC_LIMIT, plan.info.workspace_bytes
        ref = pkv.paged_varlen_attention(q, cu, ctx, bt, pool, meta.scale, plan=plan)
        out = torch.full_like(q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        st = _call(fn, pkv, meta, q, pool, cu, ctx, bt, plan, out, status, stream)
        assert st == 0, pkv.status_string(st)
        results.append((ref, out, status))
    torch.cuda.synchronize(cuda_device)
    for ref, out, status in results:
        assert int(status.item()) == 0
        _close(out, ref)
        assert torch.equal(out, ref)   # same kernels, same plan: identical bits


def test_noalloc_rejects_steps_beyond_its_scratch(pkv, cuda_device):
    fn = _noalloc_fn(pkv)
    meta = workloads.small_decode()
    q, pool, cu, ctx, bt, plan = _step(pkv, meta, cuda_device)
    big = pkv.PlanInfo.from_buffer_copy(plan.info)
    big.workspace_bytes = NOALLOC_LIMIT + 256
    out = torch.zeros_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    desc = pkv.pool_desc(pool)
    st = fn(q.data_ptr(), cu.data_ptr(), ctx.data_ptr(), bt.data_ptr(), bt.shape[1],
            pool.data_ptr(), ctypes.byref(desc), meta.scale, ctypes.byref(big),
            plan.dev.data_ptr(), out.data_ptr(), status.data_ptr(),
            torch.cuda.current_stream(cuda_device).cuda_stream)
    assert st == 5    # PKV_ERR_WORKSPACE
    torch.cuda.synchronize(cuda_device)
    assert torch.count_nonzero(out) == 0
