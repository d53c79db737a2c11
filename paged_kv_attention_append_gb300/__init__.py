"""Paged KV append + packed varlen attention for one GB300 (sm_103a).

A thin binding over the C ABI in ``include/pkv.h`` (``_lib/libpkv.so``): it
checks torch tensors, passes their device pointers and the current CUDA stream,
and allocates the caller-owned buffers (plan copy, workspace, output).  Every
step of the computation runs in the library's CUDA kernels; there is no other
implementation here.  If the library is missing, every call raises.

    kv_pool = torch.empty(num_blocks, 2, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    paged_kv_append(k_new, v_new, slot_mapping, kv_pool)
    out = paged_varlen_attention(q, cu_q_lens, context_lens, block_tables, kv_pool, scale)
"""

from __future__ import annotations

import ctypes
import os
import threading
import weakref

import numpy as np
import torch

__all__ = [
    "PkvError", "PoolDesc", "PlanInfo", "StepPlan", "build", "library_path", "version",
    "status_string", "kernel_launch_count", "paged_kv_append", "plan_step",
    "paged_varlen_attention", "DEV_STATUS", "workspace_size", "BoundStep", "BoundPlan",
    "BoundCopy", "copy_async",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libpkv.so")
_lock = threading.Lock()
_lib = None

DEV_STATUS = {0: "ok", 1: "bad slot", 2: "bad block id", 3: "pipeline wait timed out",
              4: "plan does not match device metadata"}


class PkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "total_q", "num_decode_warps",
        "num_decode_pieces", "num_merge_groups", "num_partials", "num_prefill_tiles", "num_kernels",
        "max_blocks_needed", "num_prefill_ctas", "num_prefill_partials", "num_prefill_merges",
        "lookahead", "num_shared_ctas", "num_gather_rows", "merge_rows", "num_shared_items")] + [
            (n, ctypes.c_int64) for n in (
            "kv_tokens", "decode_blocks", "plan_bytes", "workspace_bytes", "gather_pairs")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


def build(verbose: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a) and return its path."""
    from . import _build
    return _build.build(verbose=verbose)


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"{_LIB_PATH} is missing: build the CUDA library first "
                    "(paged_kv_attention_append_gb300.build()); there is no fallback path")
            lib = ctypes.CDLL(_LIB_PATH)
            P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            lib.pkv_version.restype = i32
            lib.pkv_status_string.argtypes = [i32]
            lib.pkv_status_string.restype = ctypes.c_char_p
            lib.pkv_kernel_launch_count.restype = i64
            lib.pkv_paged_kv_append.argtypes = [P, P, P, i32, P, ctypes.POINTER(PoolDesc), P, P]
            lib.pkv_paged_kv_append.restype = i32
            lib.pkv_plan_step.argtypes = [P, P, i32, i32, ctypes.POINTER(PoolDesc), i32, P, i64,
                                          ctypes.POINTER(PlanInfo)]
            lib.pkv_plan_step.restype = i32
            lib.pkv_paged_varlen_attention.argtypes = [P, P, P, P, i32, P, ctypes.POINTER(PoolDesc),
                                                       ctypes.c_float, ctypes.POINTER(PlanInfo), P, P,
                                                       P, i64, P, P]
            lib.pkv_paged_varlen_attention.restype = i32
            lib.pkv_state_checkpoint.argtypes = [P, P, i32, P, i64, i64, P, P]
            lib.pkv_state_checkpoint.restype = i32
            lib.pkv_plan_decode_chain.argtypes = [P, P, i32, i32, ctypes.POINTER(PoolDesc), i32,
                                                  i32, P, i64, ctypes.POINTER(PlanInfo)]
            lib.pkv_plan_decode_chain.restype = i32
            lib.pkv_plan_step_ex.argtypes = [P, P, i32, i32, ctypes.POINTER(PoolDesc), i32, i32,
                                             P, i32, i32, P, i64, ctypes.POINTER(PlanInfo)]
            lib.pkv_plan_step_ex.restype = i32
            lib.pkv_decode_advance.argtypes = [P, P, P, P, i32, i32, ctypes.POINTER(PoolDesc), P,
                                               P]
            lib.pkv_decode_advance.restype = i32
            lib.pkv_set_profile_events.argtypes = [i32, P, P]
            lib.pkv_set_profile_events.restype = i32
            lib.pkv_workspace_size.argtypes = [ctypes.POINTER(PlanInfo)]
            lib.pkv_workspace_size.restype = ctypes.c_size_t
            lib.pkv_copy_async.argtypes = [P, P, i64, P]
            lib.pkv_copy_async.restype = i32
            lib.pkv_planner_create.argtypes = [i32, ctypes.POINTER(P)]
            lib.pkv_planner_create.restype = i32
            lib.pkv_planner_destroy.argtypes = [P]
            lib.pkv_planner_destroy.restype = None
            lib.pkv_planner_post.argtypes = [P, P, P, i32, i32, ctypes.POINTER(PoolDesc), i32, i32,
                                             P, i32, i32, P, i64, ctypes.POINTER(PlanInfo)]
            lib.pkv_planner_post.restype = i32
            lib.pkv_planner_wait.argtypes = [P]
            lib.pkv_planner_wait.restype = i32
            _lib = lib
    return _lib


def version() -> int:
    return int(_load().pkv_version())


def status_string(status: int) -> str:
    return _load().pkv_status_string(int(status)).decode()


def kernel_launch_count() -> int:
    return int(_load().pkv_kernel_launch_count())


KERNEL_IDS = {"append": 0, "decode": 1, "merge": 2, "prefill": 3, "state": 4}


def set_profile_events(kernel: str, start=None, stop=None):
    """Record torch.cuda.Event `start`/`stop` around every launch of `kernel` made
    from this thread (None, None turns it off).  Events must have been recorded once."""
    st = _load().pkv_set_profile_events(KERNEL_IDS[kernel],
                                        None if start is None else start.cuda_event,
                                        None if stop is None else stop.cuda_event)
    if st:
        raise PkvError(st, "pkv_set_profile_events")


# The per-call wrappers below sit on the host side of every step, so they keep
# Python work small: pointers go to ctypes as plain ints (the prototypes say
# void*), the current stream comes from torch's raw-stream query, and a pool's
# descriptor is built once per pool shape.
def _ptr(t):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, t):
    """Raw handle of `stream`, else of the current stream of tensor t's device."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(t.get_device())
    return torch.cuda.current_stream(t.device).cuda_stream


def _check_cuda(name, t, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


_desc_cache: dict = {}


def pool_desc(kv_pool: torch.Tensor) -> PoolDesc:
    shape = kv_pool.shape
    d = _desc_cache.get(shape)
    if d is not None:
        return d
    if len(shape) != 5 or shape[1] != 2:
        raise ValueError("kv_pool must be [num_blocks, 2, num_kv_heads, block_size, head_dim]")
    nb, _, hkv, bs, hd = shape
    d = PoolDesc(nb, bs, hkv, hd)
    if len(_desc_cache) < 64:
        _desc_cache[shape] = d
    return d


def paged_kv_append(k, v, slot_mapping, kv_pool, *, dev_status=None, stream=None):
    """Write this step's K/V rows into the pool slots named by slot_mapping (negative = skip).

    k, v: bf16 [n, Hkv, D]; slot_mapping: int32 [n]; kv_pool: bf16 [nb, 2, Hkv, 16, D].
    """
    _check_cuda("kv_pool", kv_pool, torch.bfloat16, 5)
    _check_cuda("k", k, torch.bfloat16, 3)
    _check_cuda("v", v, torch.bfloat16, 3)
    _check_cuda("slot_mapping", slot_mapping, torch.int32, 1)
    desc = pool_desc(kv_pool)
    n = slot_mapping.shape[0]
    if k.shape != (n, desc.num_kv_heads, desc.head_dim) or v.shape != k.shape:
        raise ValueError(f"k/v must be [{n}, {desc.num_kv_heads}, {desc.head_dim}]")
    if dev_status is not None:
        _check_cuda("dev_status", dev_status, torch.int32)
    st = _load().pkv_paged_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), n, _ptr(kv_pool),
                                     ctypes.byref(desc), _ptr(dev_status),
                                     _stream(stream, kv_pool))
    if st:
        raise PkvError(st, "pkv_paged_kv_append")


def state_checkpoint(src, dst_slots, pool, *, dev_status=None, stream=None):
    """Write row i of src into pool row dst_slots[i] in place (negative = skip).

    src: [n, ...] and pool: [num_slots, ...] contiguous CUDA tensors whose rows
    (everything after the first axis) have the same byte size, a multiple of 16;
    dst_slots: int32 [n].  Rows are copied as raw bytes, whatever the dtype.
    """
    for name, t in (("src", src), ("pool", pool)):
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda" or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA tensor")
    _check_cuda("dst_slots", dst_slots, torch.int32, 1)
    n = dst_slots.shape[0]
    if src.dim() < 1 or pool.dim() < 1 or src.shape[0] != n:
        raise ValueError("src must have one row per dst_slots entry")
    row_bytes = src[0].numel() * src.element_size() if n else 0
    pool_row = pool[0].numel() * pool.element_size() if pool.shape[0] else 0
    if n and row_bytes != pool_row:
        raise ValueError(f"row sizes differ: src {row_bytes} B, pool {pool_row} B")
    if dev_status is not None:
        _check_cuda("dev_status", dev_status, torch.int32)
    st = _load().pkv_state_checkpoint(_ptr(src), _ptr(dst_slots), n, _ptr(pool), pool.shape[0],
                                      max(row_bytes, 16), _ptr(dev_status),
                                      _stream(stream, pool))
    if st:
        raise PkvError(st, "pkv_state_checkpoint")


def _host_i32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=np.int32)


def workspace_size(info: PlanInfo) -> int:
    """Device workspace bytes the attention call needs for this plan."""
    return int(_load().pkv_workspace_size(ctypes.byref(info)))


def _buffer_span(t):
    """(address, bytes) of a contiguous tensor or numpy array."""
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            raise ValueError("copy buffers must be contiguous")
        return t.data_ptr(), t.numel() * t.element_size()
    a = np.asarray(t)
    if not a.flags.c_contiguous:
        raise ValueError("copy buffers must be contiguous")
    return a.ctypes.data, a.nbytes


def copy_async(dst, src, nbytes=None, *, stream=None) -> None:
    """Queue a copy of nbytes (default: all of src) from src to dst on `stream`
    (pkv_copy_async): host<->device or device<->device, the direction from the
    pointers; asynchronous for pinned host memory.  dst and src: contiguous
    tensors (or numpy arrays on the host side)."""
    BoundCopy(dst, src, stream=stream).run(nbytes)


class BoundCopy:
    """pkv_copy_async between two fixed buffers with its arguments marshalled
    once: run(nbytes, offset) copies src[offset : offset + nbytes] to the same
    byte range of dst on the bound stream (the whole of src by default).  For a
    loop that moves each step's inputs up and its output back through the same
    pinned and device buffers."""

    def __init__(self, dst, src, *, stream=None):
        self._dst, dn = _buffer_span(dst)
        self._src, sn = _buffer_span(src)
        self._n = min(dn, sn)
        dev_t = dst if isinstance(dst, torch.Tensor) and dst.is_cuda else src
        if not (isinstance(dev_t, torch.Tensor) and dev_t.is_cuda):
            raise ValueError("one side of the copy must be a CUDA tensor")
        self._keep = (dst, src)
        self._stream = ctypes.c_void_p(_stream(stream, dev_t))
        self._f = _load().pkv_copy_async

    def run(self, nbytes=None, offset: int = 0) -> None:
        n = self._n - offset if nbytes is None else int(nbytes)
        if offset < 0 or n < 0 or offset + n > self._n:
            raise ValueError(f"copy of {n} bytes at {offset} exceeds the bound buffers ({self._n})")
        st = self._f(self._dst + offset, self._src + offset, n, self._stream)
        if st:
            raise PkvError(st, "pkv_copy_async")


class StepPlan:
    """Host step metadata plus its device copy and the workspace it needs."""

    def __init__(self, info: PlanInfo, host: np.ndarray, device: torch.device, stream=None):
        self.info = info
        self.host = host
        self.device = device
        self.dev = None
        self.workspace = None
        self.upload(stream)

    def upload(self, stream=None):
        """Copy the plan to the device and make sure the workspace is big enough.
        With `stream`, the copy and the allocations are made on that stream."""
        dev = torch.device(self.device)
        nbytes = max(int(self.info.plan_bytes), 16)
        src = torch.from_numpy(self.host.view(np.uint8)[:nbytes])
        with torch.cuda.stream(stream) if stream is not None else _nullcontext():
            if self.dev is None or self.dev.numel() < nbytes:
                self.dev = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            self.dev[:nbytes].copy_(src, non_blocking=False)
            wsb = workspace_size(self.info)
            if wsb > 0 and (self.workspace is None or self.workspace.numel() < wsb):
                self.workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
        return self


class _nullcontext:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


_tls = threading.local()   # per thread: the size of its last plan, to size the next buffer


def plan_step(cu_q_lens, context_lens, num_q_heads: int, kv_pool_or_desc, *, num_sms=None,
              device=None, upload=True, stream=None, chain_steps=None,
              block_tables=None, prefill_min_q=None, out=None) -> StepPlan | tuple:
    """Build the host plan for one step (pkv_plan_step_ex) and upload it.

    cu_q_lens / context_lens: host arrays or tensors (copied to the host if on a GPU).
    chain_steps: plan a chain of that many decode steps instead.
    block_tables: the step's block tables (host copy) -- lets the plan carry each
    split-KV warp's first block ids (checked on the device against the tables)
    and read blocks that sequences share once per work unit.
    prefill_min_q: query tokens from which a sequence runs on the tensor-core
    kernel (None or 0: the library's default; negative: no sequence does).
    out (with upload=False): a writable host buffer (numpy array or CPU tensor,
    e.g. pinned memory for an asynchronous upload) the plan is written into; the
    returned host bytes are then a view of it.
    Returns a StepPlan (or (info, host_bytes) when upload=False).
    """
    desc = kv_pool_or_desc if isinstance(kv_pool_or_desc, PoolDesc) else pool_desc(kv_pool_or_desc)
    if device is None:
        device = kv_pool_or_desc.device if isinstance(kv_pool_or_desc, torch.Tensor) else "cuda"
    cu = _host_i32(cu_q_lens)
    ctx = _host_i32(context_lens)
    if cu.ndim != 1 or ctx.ndim != 1 or cu.shape[0] != ctx.shape[0] + 1:
        raise ValueError("cu_q_lens must have num_seqs + 1 entries and context_lens num_seqs")
    if num_sms is None:
        num_sms = (torch.cuda.get_device_properties(torch.device(device)).multi_processor_count
                   if torch.cuda.is_available() else 152)
    info = PlanInfo()
    lib = _load()
    name = "pkv_plan_step_ex"
    bt = None
    if block_tables is not None:
        bt = _host_i32(block_tables)
        if bt.ndim != 2 or bt.shape[0] != ctx.shape[0]:
            raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    pmq = 0 if prefill_min_q is None else int(prefill_min_q)

    def call(buf, cap):
        return lib.pkv_plan_step_ex(
            cu.ctypes.data_as(ctypes.c_void_p), ctx.ctypes.data_as(ctypes.c_void_p), ctx.shape[0],
            int(num_q_heads), ctypes.byref(desc), int(num_sms),
            1 if chain_steps is None else int(chain_steps),
            None if bt is None else bt.ctypes.data_as(ctypes.c_void_p),
            0 if bt is None else bt.shape[1], pmq, buf, cap, ctypes.byref(info))
    if out is not None and not upload:
        buf = out.numpy() if isinstance(out, torch.Tensor) else out
        if not buf.flags.c_contiguous or not buf.flags.writeable:
            raise ValueError("out must be a contiguous writable host buffer")
        st = call(buf.ctypes.data_as(ctypes.c_void_p), buf.nbytes)
        if st:
            raise PkvError(st, name)
        n = (max(int(info.plan_bytes), 16) + 15) // 16 * 16
        return info, buf.reshape(-1).view(np.uint8)[:n].view(np.int32)
    # one planning pass into a fresh buffer sized from this thread's last plan
    # (planned again only when the plan outgrows it); the buffer is the plan's
    cap = getattr(_tls, "plan_cap", 1 << 16)
    host = np.empty(cap // 4, dtype=np.int32)
    st = call(host.ctypes.data_as(ctypes.c_void_p), host.nbytes)
    if st == 5 and int(info.plan_bytes) > host.nbytes:   # PKV_ERR_WORKSPACE: grow and redo
        host = np.empty((int(info.plan_bytes) + 15) // 16 * 4, dtype=np.int32)
        st = call(host.ctypes.data_as(ctypes.c_void_p), host.nbytes)
    if st:
        raise PkvError(st, name)
    n = (max(int(info.plan_bytes), 16) + 15) // 16 * 16
    _tls.plan_cap = max(1 << 12, (n * 5 // 4 + 4095) // 4096 * 4096)
    host = host[:n // 4]
    if not upload:
        return info, host
    return StepPlan(info, host, torch.device(device), stream)


class BoundPlan:
    """pkv_plan_step_ex over fixed host arrays with its arguments marshalled once.

    For a serving loop that rewrites the step's metadata in place (e.g. views of
    one pinned buffer) and plans every step into the same host buffer `out`:
    run() is one call into the planner; it returns (info, nbytes), info being
    this object's PlanInfo (overwritten by the next run) and nbytes the plan's
    size in `out`.  The arrays must be C-contiguous int32 numpy arrays whose
    shapes stay fixed (their contents may change between runs); the other
    arguments mean what they mean for plan_step.

    With `spin_us` set, the object also owns a planning thread (pkv_planner_*):
    post() starts the same call there and returns at once, so the caller can
    queue the step's input copy and KV append meanwhile; wait() returns what
    run() returns once it has finished.  spin_us is how long the thread polls
    for the next post before it sleeps.  The arrays and `out` must stay
    unchanged from post() to wait().
    """

    def __init__(self, cu_q_lens, context_lens, num_q_heads: int, kv_pool_or_desc, out, *,
                 num_sms=None, chain_steps=None, block_tables=None, prefill_min_q=None,
                 spin_us=None):
        arrays = [("cu_q_lens", cu_q_lens), ("context_lens", context_lens)]
        if block_tables is not None:
            arrays.append(("block_tables", block_tables))
        for name, a in arrays:
            if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous):
                raise TypeError(f"{name} must be a C-contiguous int32 numpy array")
        if cu_q_lens.ndim != 1 or context_lens.ndim != 1 or \
                cu_q_lens.shape[0] != context_lens.shape[0] + 1:
            raise ValueError("cu_q_lens must have num_seqs + 1 entries and context_lens num_seqs")
        if block_tables is not None and (block_tables.ndim != 2 or
                                         block_tables.shape[0] != context_lens.shape[0]):
            raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
        buf = out.numpy() if isinstance(out, torch.Tensor) else out
        if not (isinstance(buf, np.ndarray) and buf.flags.c_contiguous and buf.flags.writeable):
            raise ValueError("out must be a contiguous writable host buffer")
        self.desc = (kv_pool_or_desc if isinstance(kv_pool_or_desc, PoolDesc)
                     else pool_desc(kv_pool_or_desc))
        if num_sms is None:
            device = (kv_pool_or_desc.device if isinstance(kv_pool_or_desc, torch.Tensor)
                      else "cuda")
            num_sms = (torch.cuda.get_device_properties(torch.device(device)).multi_processor_count
                       if torch.cuda.is_available() else 152)
        self.info = PlanInfo()
        self._keep = (cu_q_lens, context_lens, block_tables, buf)
        self._out = buf.reshape(-1).view(np.uint8)
        vp = ctypes.c_void_p
        self._args = (vp(cu_q_lens.ctypes.data), vp(context_lens.ctypes.data),
                      ctypes.c_int32(context_lens.shape[0]), ctypes.c_int32(int(num_q_heads)),
                      ctypes.byref(self.desc), ctypes.c_int32(int(num_sms)),
                      ctypes.c_int32(1 if chain_steps is None else int(chain_steps)),
                      vp(None if block_tables is None else block_tables.ctypes.data),
                      ctypes.c_int32(0 if block_tables is None else block_tables.shape[1]),
                      ctypes.c_int32(0 if prefill_min_q is None else int(prefill_min_q)),
                      vp(buf.ctypes.data), ctypes.c_int64(buf.nbytes), ctypes.byref(self.info))
        self._f = _load().pkv_plan_step_ex
        self._worker = None
        if spin_us is not None:
            lib = _load()
            handle = ctypes.c_void_p()
            st = lib.pkv_planner_create(int(spin_us), ctypes.byref(handle))
            if st:
                raise PkvError(st, "pkv_planner_create")
            self._worker = handle
            self._post, self._wait = lib.pkv_planner_post, lib.pkv_planner_wait
            self._fin = weakref.finalize(self, lib.pkv_planner_destroy, handle)

    def run(self):
        st = self._f(*self._args)
        if st:
            raise PkvError(st, "pkv_plan_step_ex")
        return self.info, (max(int(self.info.plan_bytes), 16) + 15) // 16 * 16

    def post(self) -> None:
        if self._worker is None:
            raise RuntimeError("BoundPlan was made without spin_us: it has no planning thread")
        st = self._post(self._worker, *self._args)
        if st:
            raise PkvError(st, "pkv_planner_post")

    def wait(self):
        if self._worker is None:
            raise RuntimeError("BoundPlan was made without spin_us: it has no planning thread")
        st = self._wait(self._worker)
        if st:
            raise PkvError(st, "pkv_planner_wait")
        return self.info, (max(int(self.info.plan_bytes), 16) + 15) // 16 * 16

    def close(self) -> None:
        """Stop and join the planning thread (also done when the object is collected)."""
        if self._worker is not None:
            self._fin()
            self._worker = None


def decode_advance(context_lens, slot_mapping, cu_q_lens, block_tables, kv_pool, *,
                   dev_status=None, stream=None):
    """Move a decode chain to its next step on the device (pkv_decode_advance):
    context_lens += q_len and slot_mapping <- the slots of the new positions.
    All four arrays are device int32 tensors; context_lens and slot_mapping are
    updated in place."""
    _check_cuda("context_lens", context_lens, torch.int32, 1)
    _check_cuda("slot_mapping", slot_mapping, torch.int32, 1)
    _check_cuda("cu_q_lens", cu_q_lens, torch.int32, 1)
    _check_cuda("block_tables", block_tables, torch.int32, 2)
    desc = pool_desc(kv_pool)
    n = context_lens.shape[0]
    if cu_q_lens.shape[0] != n + 1 or block_tables.shape[0] != n:
        raise ValueError("cu_q_lens needs num_seqs + 1 entries and block_tables num_seqs rows")
    if dev_status is not None:
        _check_cuda("dev_status", dev_status, torch.int32)
    st = _load().pkv_decode_advance(_ptr(context_lens), _ptr(slot_mapping), _ptr(cu_q_lens),
                                    _ptr(block_tables), block_tables.shape[1], n,
                                    ctypes.byref(desc), _ptr(dev_status),
                                    _stream(stream, context_lens))
    if st:
        raise PkvError(st, "pkv_decode_advance")


def _dev_i32(x, device, name):
    if isinstance(x, torch.Tensor) and x.is_cuda:
        _check_cuda(name, x, torch.int32)
        return x
    return torch.from_numpy(_host_i32(x)).to(device)


def paged_varlen_attention(q, cu_q_lens, context_lens, block_tables, kv_pool, scale: float, *,
                           plan: StepPlan | None = None, out=None, dev_status=None, stream=None):
    """Packed varlen causal attention over the paged pool; returns out [total_q, Hq, D] bf16.

    cu_q_lens / context_lens may be host or device arrays; a plan is built from
    host copies when none is given.  block_tables: int32 [num_seqs, max_blocks].
    stream: run on this CUDA stream instead of the current one; the arrays this
    call copies to the device, the workspace and `out` (when allocated here) are
    then allocated on that stream, and the caller orders its use of `out` after it.
    """
    _check_cuda("q", q, torch.bfloat16, 3)
    _check_cuda("kv_pool", kv_pool, torch.bfloat16, 5)
    desc = pool_desc(kv_pool)
    dev = q.device
    ctx_mgr = torch.cuda.stream(stream) if stream is not None else _nullcontext()
    with ctx_mgr:
        if plan is None:
            plan = plan_step(cu_q_lens, context_lens, q.shape[1], desc, device=dev, stream=stream)
        info = plan.info
        if q.shape[0] != info.total_q or q.shape[1] != info.num_q_heads or q.shape[2] != desc.head_dim:
            raise ValueError(f"q shape {tuple(q.shape)} does not match the plan "
                             f"({info.total_q}, {info.num_q_heads}, {desc.head_dim})")
        cu_d = _dev_i32(cu_q_lens, dev, "cu_q_lens")
        ctx_d = _dev_i32(context_lens, dev, "context_lens")
        bt_d = _dev_i32(block_tables, dev, "block_tables")
        if bt_d.dim() != 2 or bt_d.shape[0] != info.num_seqs:
            raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
        if out is None:
            out = torch.empty_like(q)
        else:
            _check_cuda("out", out, torch.bfloat16, 3)
            if out.shape != q.shape:
                raise ValueError("out must have q's shape")
        if dev_status is not None:
            _check_cuda("dev_status", dev_status, torch.int32)
        ws = plan.workspace
        st = _load().pkv_paged_varlen_attention(
            _ptr(q), _ptr(cu_d), _ptr(ctx_d), _ptr(bt_d), bt_d.shape[1], _ptr(kv_pool),
            ctypes.byref(desc), float(scale), ctypes.byref(info), _ptr(plan.dev), _ptr(out),
            _ptr(ws), 0 if ws is None else ws.numel(), _ptr(dev_status), _stream(stream, q))
    if st:
        raise PkvError(st, "pkv_paged_varlen_attention")
    return out


class BoundStep:
    """One step's KV append and attention with their arguments checked once.

    A serving loop that reuses the same device buffers every step (inputs copied
    into them, the plan re-made into the same pinned buffer) binds them here and
    calls run() per step: each run is two calls into the library with
    pre-marshalled arguments, no tensor checks and no allocation.  `plan` is
    read at run time (plan.info, plan.dev and plan.workspace may be replaced
    between runs, e.g. with each step's new plan summary), so the step's shape
    may change as long as the bound buffers stay large enough for it: run()
    re-checks the sizes the plan states against the bound tensors.
    """

    def __init__(self, k, v, slot_mapping, q, cu_q_lens, context_lens, block_tables, kv_pool,
                 scale: float, plan: StepPlan, out, *, dev_status=None, stream=None):
        _check_cuda("kv_pool", kv_pool, torch.bfloat16, 5)
        for name, t, ndim in (("k", k, 3), ("v", v, 3), ("q", q, 3), ("out", out, 3)):
            _check_cuda(name, t, torch.bfloat16, ndim)
        for name, t, ndim in (("slot_mapping", slot_mapping, 1), ("cu_q_lens", cu_q_lens, 1),
                              ("context_lens", context_lens, 1), ("block_tables", block_tables, 2)):
            _check_cuda(name, t, torch.int32, ndim)
        if dev_status is not None:
            _check_cuda("dev_status", dev_status, torch.int32)
        desc = pool_desc(kv_pool)
        if k.shape[1:] != (desc.num_kv_heads, desc.head_dim) or v.shape != k.shape:
            raise ValueError("k/v must be [n, num_kv_heads, head_dim] of the pool")
        if out.shape != q.shape or q.shape[2] != desc.head_dim:
            raise ValueError("out must have q's shape, [total_q, num_q_heads, head_dim]")
        if slot_mapping.shape[0] != k.shape[0]:
            raise ValueError("slot_mapping needs one entry per new token")
        self.plan = plan
        self._tensors = (k, v, slot_mapping, q, cu_q_lens, context_lens, block_tables, kv_pool,
                         out, dev_status)   # kept alive while bound
        self._desc = desc
        self._lib = _load()
        self._stream = _stream(stream, q)
        self._n_new = k.shape[0]
        self._shape = (q.shape[0], q.shape[1], cu_q_lens.shape[0], block_tables.shape[0],
                       block_tables.shape[1])
        vp = ctypes.c_void_p
        self._append = (vp(k.data_ptr()), vp(v.data_ptr()), vp(slot_mapping.data_ptr()),
                        ctypes.c_int32(self._n_new), vp(kv_pool.data_ptr()), ctypes.byref(desc),
                        vp(_ptr(dev_status)), vp(self._stream))
        self._attn_head = (vp(q.data_ptr()), vp(cu_q_lens.data_ptr()), vp(context_lens.data_ptr()),
                           vp(block_tables.data_ptr()), ctypes.c_int32(block_tables.shape[1]),
                           vp(kv_pool.data_ptr()), ctypes.byref(desc), ctypes.c_float(scale))
        self._out = vp(out.data_ptr())
        self._tail = (vp(_ptr(dev_status)), vp(self._stream))

    def run(self) -> None:
        """Enqueue this step's append and attention on the bound stream."""
        self.run_append()
        self.run_attention()

    def run_append(self) -> None:
        """Enqueue the step's KV append alone: it needs no plan, so a serving loop
        may queue it as soon as the step's new K/V are on the device and plan the
        step meanwhile (run_attention then follows it on the same stream)."""
        st = self._lib.pkv_paged_kv_append(*self._append)
        if st:
            raise PkvError(st, "pkv_paged_kv_append")

    def run_attention(self) -> None:
        """Enqueue the step's attention with the plan as it stands now."""
        info = self.plan.info
        total_q, hq, n_cu, n_bt, max_blocks = self._shape
        if (info.total_q != total_q or info.num_q_heads != hq or info.num_seqs + 1 != n_cu or
                info.num_seqs != n_bt):
            raise ValueError("the plan does not match the bound buffers")
        ws = self.plan.workspace
        st = self._lib.pkv_paged_varlen_attention(
            *self._attn_head, ctypes.byref(info), ctypes.c_void_p(self.plan.dev.data_ptr()),
            self._out, ctypes.c_void_p(None if ws is None else ws.data_ptr()),
            ctypes.c_int64(0 if ws is None else ws.numel()), *self._tail)
        if st:
            raise PkvError(st, "pkv_paged_varlen_attention")
