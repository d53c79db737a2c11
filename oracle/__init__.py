"""CPU fp64 oracle for paged KV append and packed varlen attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product path.  It shares no code with
the CUDA library (``paged_kv_attention_append_gb300``) and neither imports the
other.  The arithmetic lives in ``pkv_oracle.c`` (plain C, OpenMP, doubles); this
module only compiles it with gcc and marshals arrays.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (brute force through a second route, closed forms,
invariants and a hand-derived fixture under ``tests/golden/``).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_SHAPE, ERR_RANGE = 0, 2, 3


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c with gcc (-O2, OpenMP, strict IEEE: no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_paged_kv_append.argtypes = [P, i32, i32, i32, i32, P, P, P, i32]
            lib.oracle_paged_kv_append.restype = i32
            lib.oracle_state_checkpoint.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, P,
                                                    ctypes.c_int64]
            lib.oracle_state_checkpoint.restype = ctypes.c_int64
            lib.oracle_check_step.argtypes = [i32, P, P, P, i32, i32, i32]
            lib.oracle_check_step.restype = i32
            lib.oracle_paged_varlen_attention.argtypes = [P, i32, i32, P, P, i32, P, i32, P, i32,
                                                          i32, i32, i32, f64, P, i64, P, i32]
            lib.oracle_paged_varlen_attention.restype = i32
            lib.oracle_max_threads.restype = i32
            _lib = lib
    return _lib


def _u16(t) -> np.ndarray:
    """bf16 torch tensor or uint16 array -> contiguous uint16 numpy array of raw bits."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(a) -> np.ndarray:
    if not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def paged_kv_append(pool_bits: np.ndarray, k, v, slot_mapping, *, block_size: int):
    """Return (new_pool_bits, n_bad_slots).  pool_bits: uint16 [nb, 2, Hkv, bs, D]."""
    pool = np.array(_u16(pool_bits), copy=True)
    nb, two, hkv, bs, d = pool.shape
    assert two == 2 and bs == block_size
    kb, vb, sm = _u16(k), _u16(v), _i32(slot_mapping)
    n = sm.shape[0]
    assert kb.shape == (n, hkv, d) and vb.shape == (n, hkv, d)
    bad = _load().oracle_paged_kv_append(_ptr(pool), nb, bs, hkv, d, _ptr(kb), _ptr(vb), _ptr(sm), n)
    return pool, int(bad)


def state_checkpoint(pool_bytes: np.ndarray, src_bytes: np.ndarray, slots):
    """Return (new_pool, n_bad_slots).  pool_bytes: uint8 [num_slots, row_bytes];
    src_bytes: uint8 [n_rows, row_bytes]; slots: int32 [n_rows] (negative = skip)."""
    pool = np.array(np.ascontiguousarray(pool_bytes, dtype=np.uint8), copy=True)
    src = np.ascontiguousarray(src_bytes, dtype=np.uint8)
    sl = _i32(slots)
    assert pool.ndim == 2 and src.ndim == 2 and src.shape[1] == pool.shape[1]
    assert sl.shape == (src.shape[0],)
    bad = _load().oracle_state_checkpoint(_ptr(pool), pool.shape[0], pool.shape[1], _ptr(src),
                                          _ptr(sl), src.shape[0])
    return pool, int(bad)


def check_step(cu_q_lens, context_lens, block_tables, num_blocks, block_size) -> int:
    cu, ctx, bt = _i32(cu_q_lens), _i32(context_lens), _i32(block_tables)
    return int(_load().oracle_check_step(ctx.shape[0], _ptr(cu), _ptr(ctx), _ptr(bt),
                                         bt.shape[1] if bt.ndim == 2 else 0, num_blocks, block_size))


def paged_varlen_attention(q, cu_q_lens, context_lens, block_tables, pool_bits, scale: float,
                           *, rows=None, num_threads: int = 0) -> np.ndarray:
    """fp64 attention.  Returns [total_q, Hq, D] (rows=None) or [len(rows), D].

    rows: optional int64 array of flat row ids ``token * Hq + q_head``.
    """
    qb, pool = _u16(q), _u16(pool_bits)
    cu, ctx, bt = _i32(cu_q_lens), _i32(context_lens), _i32(block_tables)
    total_q, hq, d = qb.shape
    nb, two, hkv, bs, d2 = pool.shape
    assert d2 == d and two == 2
    if bt.ndim != 2:
        bt = bt.reshape(ctx.shape[0], -1)
    if rows is None:
        n_rows, rp = total_q * hq, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows, rp = rows.shape[0], _ptr(rows)
    out = np.zeros((max(n_rows, 1), d), dtype=np.float64)
    rc = _load().oracle_paged_varlen_attention(
        _ptr(qb), total_q, hq, _ptr(cu), _ptr(ctx), ctx.shape[0], _ptr(bt), bt.shape[1], _ptr(pool),
        nb, bs, hkv, d, float(scale), rp, n_rows, _ptr(out), int(num_threads))
    if rc != OK:
        raise ValueError(f"oracle rejected the step (code {rc})")
    out = out[:n_rows]
    return out.reshape(total_q, hq, d) if rows is None else out


def run_step(meta, q, k_new, v_new, pool, *, rows=None, num_threads: int = 0):
    """Append this step's K/V into a copy of ``pool``, then attend.  Returns (out, pool_after)."""
    pool_after, bad = paged_kv_append(pool, k_new, v_new, meta.slot_mapping, block_size=meta.block_size)
    if bad:
        raise ValueError(f"{bad} slots outside the pool")
    out = paged_varlen_attention(q, meta.cu_q_lens, meta.context_lens, meta.block_tables, pool_after,
                                 meta.scale, rows=rows, num_threads=num_threads)
    return out, pool_after
