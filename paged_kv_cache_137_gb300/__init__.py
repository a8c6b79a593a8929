"""GB300-native paged KV cache: Python binding of libpkv.so.

The functions below carry the names of the C ABI in ``include/pkv.h`` and do
argument marshalling only (tensor checks, pointers, the current CUDA stream);
every step of the data path runs in the library's CUDA kernels or its native
host allocator.  Device memory comes from PyTorch tensors owned by the caller.
There is no fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from ._build import LIB, build  # noqa: F401

PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_OUT_OF_BLOCKS, PKV_ERR_UNKNOWN_SEQ, PKV_ERR_UNSUPPORTED, \
    PKV_ERR_CUDA = range(6)
PKV_F32, PKV_F16, PKV_BF16, PKV_E4M3 = range(4)
PKV_KERNEL_AUTO, PKV_KERNEL_SIMT, PKV_KERNEL_TENSOR_CORE = range(3)
KERNEL_OF_NAME = {"auto": PKV_KERNEL_AUTO, "simt": PKV_KERNEL_SIMT, "tc": PKV_KERNEL_TENSOR_CORE}

STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "OUT_OF_BLOCKS", 3: "UNKNOWN_SEQ", 4: "UNSUPPORTED",
                5: "CUDA"}
DTYPE_OF_NAME = {"f32": PKV_F32, "f16": PKV_F16, "bf16": PKV_BF16, "e4m3": PKV_E4M3}
TORCH_OF_DTYPE = {PKV_F32: torch.float32, PKV_F16: torch.float16, PKV_BF16: torch.bfloat16,
                  PKV_E4M3: torch.uint8}


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.code = STATUS_NAMES.get(status, str(status))


class pkv_kv_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("head_scales", ctypes.c_void_p)]

    @property
    def elem_bytes(self) -> int:
        return {PKV_F32: 4, PKV_F16: 2, PKV_BF16: 2, PKV_E4M3: 1}[self.kv_dtype]

    @property
    def torch_dtype(self):
        return TORCH_OF_DTYPE[self.kv_dtype]

    @property
    def cache_shape(self):
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)


def kv_desc(num_blocks, num_kv_heads, head_dim, block_size, kv_dtype, head_scales=None) -> pkv_kv_desc:
    """The cache descriptor.  head_scales (E4M3 caches): a contiguous float32
    device tensor [4, num_kv_heads] holding each KV head's K scale, V scale,
    K inverse and V inverse scale; the descriptor keeps a reference to it."""
    if isinstance(kv_dtype, str):
        kv_dtype = DTYPE_OF_NAME[kv_dtype]
    d = pkv_kv_desc(num_blocks, num_kv_heads, head_dim, block_size, kv_dtype)
    if head_scales is not None:
        if (not isinstance(head_scales, torch.Tensor) or not head_scales.is_cuda
                or head_scales.dtype != torch.float32 or tuple(head_scales.shape) != (4, num_kv_heads)
                or not head_scales.is_contiguous()):
            raise ValueError("head_scales must be a contiguous float32 CUDA tensor [4, num_kv_heads]")
        d.head_scales = head_scales.data_ptr()
        d._head_scales = head_scales
    return d


def with_head_scales(desc: pkv_kv_desc, head_scales) -> pkv_kv_desc:
    """A copy of ``desc`` with per-KV-head E4M3 scales (see kv_desc)."""
    return kv_desc(desc.num_blocks, desc.num_kv_heads, desc.head_dim, desc.block_size, desc.kv_dtype,
                   head_scales)


_lib = None
_P = ctypes.c_void_p
_I32, _I64, _U64, _F = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
_PI32, _PI64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
_PDESC = ctypes.POINTER(pkv_kv_desc)

_SIGNATURES = {
    "pkv_block_bytes": (_U64, [_I32, _I32, _I32, _I32, _I32]),
    "pkv_num_blocks_for_budget": (_U64, [_U64, _U64]),
    "pkv_dtype_bytes": (_I32, [_I32]),
    "pkv_pool_create": (_I32, [_I32, _I32, _PI32, ctypes.POINTER(_P)]),
    "pkv_pool_destroy": (None, [_P]),
    "pkv_seq_create": (_I32, [_P, _I64]),
    "pkv_seq_append": (_I32, [_P, _I64, _I32, _PI64, _PI32, _I32, _PI32]),
    "pkv_batch_append": (_I32, [_P, _PI64, _I32, _PI64, _PI32, _I32, _PI32]),
    "pkv_seq_fork": (_I32, [_P, _I64, _I64]),
    "pkv_seq_free": (_I32, [_P, _I64]),
    "pkv_seq_table": (_I32, [_P, _I64, _PI32, _I32, _PI32, _PI64]),
    "pkv_block_tables": (_I32, [_P, _PI64, _I32, _I32, _PI32, _PI32]),
    "pkv_block_tables_update": (_I32, [_P, _PI64, _I32, _I32, _PI32, _PI64, _PI32]),
    "pkv_block_refcount": (_I32, [_P, _I32, _PI32]),
    "pkv_num_free_blocks": (_I32, [_P]),
    "pkv_free_stack": (_I32, [_P, _PI32, _I32, _PI32]),
    "pkv_pool_usage": (_I32, [_P, _PI64, _PI64, _PI64]),
    "pkv_write": (_I32, [_P, _P, _P, _P, _I32, _P, _I32, _PDESC, _F, _F, _P]),
    "pkv_copy_blocks": (_I32, [ctypes.POINTER(_P), ctypes.POINTER(_P), _I32, _PI32, _I32, _PDESC, _P]),
    "pkv_attention_workspace_bytes": (ctypes.c_size_t, [_I32, _I32, _I32, _PDESC, _I32]),
    "pkv_attention_partition": (_I32, [_I32, _I32, _PDESC, _I32]),
    "pkv_attention_decode": (_I32, [_P, _P, _I32, _P, _P, _P, _I32, _P, _I32, _I32, _PDESC, _F, _F, _F,
                                    _I32, _P, ctypes.c_size_t, _P]),
    "pkv_set_attention_kernel": (_I32, [_I32]),
    "pkv_set_prefill_kernel": (_I32, [_I32]),
    "pkv_attention_decode_noalloc": (_I32, [_P, _P, _I32, _P, _P, _P, _I32, _P, _I32, _I32, _PDESC, _F,
                                            _F, _F, _I32, _P]),
    "pkv_attention_prefill": (_I32, [_P, _P, _I32, _P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32,
                                     _PDESC, _F, _F, _F, _P]),
    "pkv_pool_enable_prefix_cache": (_I32, [_P]),
    "pkv_seq_create_cached": (_I32, [_P, _I64, _PI32, _I32, _PI32]),
    "pkv_seq_append_tokens": (_I32, [_P, _I64, _PI32, _I32, _PI64, _PI32, _I32, _PI32]),
    "pkv_prefix_cache_stats": (_I32, [_P, _PI64, _PI64, _PI64, _PI64]),
    "pkv_reusable_blocks": (_I32, [_P, _PI32, _I32, _PI32]),
    "pkv_batch_append_preempt": (_I32, [_P, _PI64, _I32, _PI64, _PI32, _I32, _PI32, _PI64, _PI32]),
    "pkv_seq_admit": (_I32, [_P, _I64, _I32, _I32, _PI64]),
    "pkv_decode_step": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _PDESC, _F, _F,
                               _F, _F, _F, _I32, _P, ctypes.c_size_t, _P]),
    "pkv_shared_prefix_blocks": (_I32, [_P, _PI64, _I32, _PI32]),
    "pkv_shared_prefix_workspace_bytes": (ctypes.c_size_t, [_I32, _I32, _I32, _PDESC, _I32, _I32]),
    "pkv_attention_decode_shared_prefix": (_I32, [_P, _P, _I32, _P, _P, _P, _I32, _P, _I32, _I32, _PDESC,
                                                  _I32, _F, _F, _F, _I32, _P, ctypes.c_size_t, _P]),
    "pkv_decode_step_shared_prefix": (_I32, [_P, _P, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32,
                                             _PDESC, _I32, _F, _F, _F, _F, _F, _I32, _P,
                                             ctypes.c_size_t, _P]),
    "pkv_device_status": (_I32, [_PI32, _I32, _P]),
    "pkv_set_stage_wait_limit": (_I32, [_U64]),
    "pkv_last_error": (ctypes.c_char_p, []),
}
NOALLOC_SCRATCH_BYTES = 16 << 20
# device error bits (pkv_device_status)
PKV_DEVICE_BAD_LENGTH, PKV_DEVICE_BAD_TABLE, PKV_DEVICE_WAIT_TIMEOUT, PKV_DEVICE_BAD_SHARED_PREFIX = 1, 2, 4, 8
EXPORTED = tuple(_SIGNATURES)


def lib():
    """The loaded libpkv (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: build it with paged_kv_cache_137_gb300.build()")
        handle = ctypes.CDLL(LIB)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


_FAST = {}


def _fast(name: str):
    """The C function with its pointer arguments taken as plain addresses
    (c_void_p) instead of typed pointers, for the allocator's per-step calls:
    building a typed pointer per argument costs more than the call itself."""
    f = _FAST.get(name)
    if f is None:
        restype, argtypes = _SIGNATURES[name]
        f = lib()[name]  # a separate function object; the typed one stays as it is
        f.restype = restype
        f.argtypes = [_P if t in (_PI32, _PI64) else t for t in argtypes]
        _FAST[name] = f
    return f


def _host_i32_address(x, shape, what: str) -> int:
    """Address of a C-contiguous int32 host buffer of the given shape (a
    NumPy array or a CPU tensor); ValueError otherwise."""
    if isinstance(x, np.ndarray):
        ok = x.dtype == np.int32 and x.flags.c_contiguous and x.flags.writeable
        addr = x.ctypes.data
    else:
        import torch
        ok = (isinstance(x, torch.Tensor) and x.device.type == "cpu" and x.dtype == torch.int32
              and x.is_contiguous())
        addr = x.data_ptr() if ok else 0
    if not ok or tuple(x.shape) != tuple(shape):
        raise ValueError(f"{what} must be a C-contiguous int32 host buffer of shape {tuple(shape)}")
    return addr


def _check(status: int):
    if status != PKV_OK:
        raise PkvError(status, lib().pkv_last_error().decode())


def _i32p(a: np.ndarray):
    return a.ctypes.data_as(_PI32)


def _i64p(a: np.ndarray):
    return a.ctypes.data_as(_PI64)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    m = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}
    if t.dtype not in m:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


# ------------------------------------------------------------------ sizing
def pkv_block_bytes(num_layers, num_kv_heads, head_dim, block_size, elem_bytes) -> int:
    return int(lib().pkv_block_bytes(num_layers, num_kv_heads, head_dim, block_size, elem_bytes))


def pkv_num_blocks_for_budget(budget_bytes, block_bytes) -> int:
    return int(lib().pkv_num_blocks_for_budget(int(budget_bytes), int(block_bytes)))


def pkv_dtype_bytes(dtype) -> int:
    return int(lib().pkv_dtype_bytes(DTYPE_OF_NAME.get(dtype, dtype)))


# --------------------------------------------------------------- allocator
class BlockTableRows:
    """A batch's block tables kept on the host across decode steps and
    brought up to date by pkv_block_tables_update: each step rewrites only
    the entries that can have changed (a row's last entry and what was
    appended), or the whole row when it now holds another sequence.

    tables: int32 CPU tensor [capacity, max_blocks]; context_lens: int32
    [capacity] (pinned if asked, so that they reach the device by one copy
    each).  update(seq_ids) fills their first len(seq_ids) rows and returns
    those views.  The rows belong to this object: writing them otherwise
    needs reset()."""

    def __init__(self, pool: "Pool", capacity: int, max_blocks: int, pin_memory: bool = False):
        self.pool, self.capacity, self.max_blocks = pool, int(capacity), int(max_blocks)
        self.tables = torch.full((self.capacity, self.max_blocks), -1, dtype=torch.int32,
                                 pin_memory=pin_memory)
        self.context_lens = torch.zeros(self.capacity, dtype=torch.int32, pin_memory=pin_memory)
        self._rows = np.zeros((self.capacity, 2), dtype=np.int64)
        self._addr = (self.tables.data_ptr(), self._rows.ctypes.data, self.context_lens.data_ptr())
        self._views = {}   # n -> (tables[:n], context_lens[:n]): slicing a tensor costs µs

    def reset(self):
        """Forget what the rows hold: the next update rewrites them whole."""
        self._rows[:] = 0

    def update(self, seq_ids):
        n = len(seq_ids)
        if n > self.capacity:
            raise ValueError(f"{n} sequences exceed the {self.capacity} rows")
        ids, ids_p = self.pool._buf("ids", n, np.int64)
        ids[:n] = seq_ids
        t_p, r_p, c_p = self._addr
        _check(_fast("pkv_block_tables_update")(self.pool._h.value, ids_p, n, self.max_blocks, t_p,
                                                r_p, c_p))
        v = self._views.get(n)
        if v is None:
            v = self._views[n] = (self.tables[:n], self.context_lens[:n])
        return v


class Pool:
    """A native block allocator (free stack, tables, reference counts)."""

    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        h = _P()
        order = None
        if initial_free_order is not None:
            order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
            if order.shape != (self.num_blocks,):
                raise ValueError("initial_free_order must hold num_blocks ids")
        _check(lib().pkv_pool_create(self.num_blocks, self.block_size,
                                     _i32p(order) if order is not None else None, ctypes.byref(h)))
        self._h = h
        self._bufs = {}    # per-step scratch (a handle is used from one thread)

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pkv_pool_destroy(self._h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def seq_create(self, seq_id: int):
        _check(lib().pkv_seq_create(self._h, int(seq_id)))

    def seq_append(self, seq_id: int, n_new: int):
        """-> (slots int64[n_new], cow pairs int32[n, 2])"""
        slots = np.empty(max(n_new, 1), dtype=np.int64)
        cow = np.empty(2, dtype=np.int32)
        n_cow = ctypes.c_int32(0)
        _check(lib().pkv_seq_append(self._h, int(seq_id), int(n_new), _i64p(slots), _i32p(cow), 1,
                                    ctypes.byref(n_cow)))
        return slots[:n_new], cow[:2 * n_cow.value].reshape(-1, 2)

    def _buf(self, name: str, n: int, dtype):
        """A reusable host buffer of at least n elements and its address."""
        b = self._bufs.get(name)
        if b is None or b[0].size < n:
            arr = np.empty(max(n, 64), dtype=dtype)
            b = self._bufs[name] = (arr, arr.ctypes.data)
        return b

    def batch_append(self, seq_ids):
        """One token per sequence, all-or-nothing -> (slots int64[B], cow int32[n, 2])"""
        n = len(seq_ids)
        ids, ids_p = self._buf("ids", n, np.int64)
        ids[:n] = seq_ids
        slots, slots_p = self._buf("slots", n, np.int64)
        cow, cow_p = self._buf("cow", 2 * n, np.int32)
        ncow, ncow_p = self._buf("ncow", 1, np.int32)
        _check(_fast("pkv_batch_append")(self._h.value, ids_p, n, slots_p, cow_p, n, ncow_p))
        k = int(ncow[0])
        return slots[:n].copy(), cow[:2 * k].reshape(-1, 2).copy()

    def seq_fork(self, parent: int, child: int):
        _check(lib().pkv_seq_fork(self._h, int(parent), int(child)))

    def seq_free(self, seq_id: int):
        _check(lib().pkv_seq_free(self._h, int(seq_id)))

    def seq_table(self, seq_id: int):
        """-> (table int32[n_blocks], context_len)"""
        n = ctypes.c_int32(0)
        ln = ctypes.c_int64(0)
        _check(lib().pkv_seq_table(self._h, int(seq_id), None, 0, ctypes.byref(n), ctypes.byref(ln)))
        out = np.empty(max(n.value, 1), dtype=np.int32)
        _check(lib().pkv_seq_table(self._h, int(seq_id), _i32p(out), len(out), ctypes.byref(n),
                                   ctypes.byref(ln)))
        return out[:n.value], ln.value

    def block_tables(self, seq_ids, max_blocks: int, out=None):
        """-> (tables int32[B, max_blocks] padded with -1, context_lens int32[B])

        out: optional (tables, context_lens) to fill instead of fresh arrays:
        C-contiguous int32 host arrays or CPU tensors (pinned ones can go
        to the device by one copy each) of exactly those shapes; returned as
        given.  On an error neither is written."""
        n = len(seq_ids)
        ids, ids_p = self._buf("ids", n, np.int64)
        ids[:n] = seq_ids
        if out is None:
            tables = np.empty((n, max_blocks), dtype=np.int32)
            ctx = np.empty(n, dtype=np.int32)
            t_p, c_p = tables.ctypes.data, ctx.ctypes.data
        else:
            tables, ctx = out
            t_p = _host_i32_address(tables, (n, int(max_blocks)), "tables")
            c_p = _host_i32_address(ctx, (n,), "context_lens")
        _check(_fast("pkv_block_tables")(self._h.value, ids_p, n, int(max_blocks), t_p, c_p))
        return tables, ctx

    def block_tables_rows(self, capacity: int, max_blocks: int, pin_memory: bool = False):
        """Host buffers for pkv_block_tables_update, kept across decode steps
        (see BlockTableRows)."""
        return BlockTableRows(self, capacity, max_blocks, pin_memory)

    def shared_prefix_blocks(self, seq_ids) -> int:
        """Leading table entries every listed sequence maps to the same
        physical blocks, short of each one's last position
        (pkv_shared_prefix_blocks)."""
        n = len(seq_ids)
        ids, ids_p = self._buf("ids", n, np.int64)
        ids[:n] = seq_ids
        k = ctypes.c_int32(0)
        _check(lib().pkv_shared_prefix_blocks(self._h, ids.ctypes.data_as(_PI64), n, ctypes.byref(k)))
        return k.value

    def block_refcount(self, block: int) -> int:
        rc = ctypes.c_int32(0)
        _check(lib().pkv_block_refcount(self._h, int(block), ctypes.byref(rc)))
        return rc.value

    def num_free_blocks(self) -> int:
        return int(lib().pkv_num_free_blocks(self._h))

    def free_stack(self) -> np.ndarray:
        """The free stack, top first."""
        n = ctypes.c_int32(0)
        _check(lib().pkv_free_stack(self._h, None, 0, ctypes.byref(n)))
        out = np.empty(max(n.value, 1), dtype=np.int32)
        _check(lib().pkv_free_stack(self._h, _i32p(out), len(out), ctypes.byref(n)))
        return out[:n.value]

    # --- prefix caching
    def enable_prefix_cache(self):
        _check(lib().pkv_pool_enable_prefix_cache(self._h))

    def seq_create_cached(self, seq_id: int, token_ids) -> int:
        """Create a sequence from a prompt; -> tokens served from the cache."""
        ids = np.ascontiguousarray(token_ids, dtype=np.int32)
        n = ctypes.c_int32(0)
        _check(lib().pkv_seq_create_cached(self._h, int(seq_id), _i32p(ids), len(ids),
                                           ctypes.byref(n)))
        return n.value

    def seq_append_tokens(self, seq_id: int, token_ids):
        """Append tokens with their ids -> (slots int64[n], cow pairs int32[n, 2])"""
        ids = np.ascontiguousarray(token_ids, dtype=np.int32)
        n_new = len(ids)
        slots = np.empty(max(n_new, 1), dtype=np.int64)
        cow = np.empty(2, dtype=np.int32)
        n_cow = ctypes.c_int32(0)
        _check(lib().pkv_seq_append_tokens(self._h, int(seq_id), _i32p(ids), n_new, _i64p(slots),
                                           _i32p(cow), 1, ctypes.byref(n_cow)))
        return slots[:n_new], cow[:2 * n_cow.value].reshape(-1, 2)

    def prefix_cache_stats(self):
        """-> (published blocks, reusable blocks, cached prompt tokens served, evictions)"""
        v = [ctypes.c_int64() for _ in range(4)]
        _check(lib().pkv_prefix_cache_stats(self._h, *[ctypes.byref(x) for x in v]))
        return tuple(x.value for x in v)

    def reusable_blocks(self) -> np.ndarray:
        """Published blocks at count 0, first to be evicted first."""
        n = ctypes.c_int32(0)
        _check(lib().pkv_reusable_blocks(self._h, None, 0, ctypes.byref(n)))
        out = np.empty(max(n.value, 1), dtype=np.int32)
        _check(lib().pkv_reusable_blocks(self._h, _i32p(out), len(out), ctypes.byref(n)))
        return out[:n.value]

    # --- preemption
    def batch_append_preempt(self, seq_ids):
        """One token per sequence in priority order, preempting the lowest
        priority when the pool runs dry -> (slots int64[B] (-1 = preempted),
        cow int32[n, 2], preempted ids)"""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = len(ids)
        slots = np.empty(max(n, 1), dtype=np.int64)
        cow = np.empty(2 * max(n, 1), dtype=np.int32)
        pre = np.empty(max(n, 1), dtype=np.int64)
        n_cow, n_pre = ctypes.c_int32(0), ctypes.c_int32(0)
        _check(lib().pkv_batch_append_preempt(self._h, _i64p(ids), n, _i64p(slots), _i32p(cow), n,
                                              ctypes.byref(n_cow), _i64p(pre), ctypes.byref(n_pre)))
        return slots[:n], cow[:2 * n_cow.value].reshape(-1, 2), list(pre[:n_pre.value])

    def seq_admit(self, seq_id: int, n_tokens: int, watermark_blocks: int = 0):
        """Create + append n_tokens if watermark_blocks stay free -> slots"""
        slots = np.empty(max(n_tokens, 1), dtype=np.int64)
        _check(lib().pkv_seq_admit(self._h, int(seq_id), int(n_tokens), int(watermark_blocks),
                                   _i64p(slots)))
        return slots[:n_tokens]

    def usage(self):
        """-> (live sequences, live tokens, blocks in use)"""
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().pkv_pool_usage(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
        return a.value, b.value, c.value


def pkv_pool_create(num_blocks, block_size, initial_free_order=None) -> Pool:
    return Pool(num_blocks, block_size, initial_free_order)


# ------------------------------------------------------------------ device
def empty_cache(desc: pkv_kv_desc, device="cuda", fill_byte: int | None = None):
    """One layer's (K, V) cache tensors [num_blocks, N_kv, T, D]."""
    k = torch.empty(desc.cache_shape, dtype=desc.torch_dtype, device=device)
    v = torch.empty_like(k)
    if fill_byte is not None:
        k.view(torch.uint8).fill_(fill_byte)
        v.view(torch.uint8).fill_(fill_byte)
    return k, v


def pkv_write(k_cache, v_cache, k, v, slot_mapping, desc: pkv_kv_desc, k_inv_scale=1.0,
              v_inv_scale=1.0, stream=None):
    """Write each token's K/V [n, N_kv, D] into its slot (slot_mapping int64[n])."""
    n = k.shape[0]
    if k.shape != (n, desc.num_kv_heads, desc.head_dim) or v.shape != k.shape or v.dtype != k.dtype:
        raise ValueError("k and v must be [n_tokens, num_kv_heads, head_dim] of one dtype")
    if slot_mapping.shape != (n,):
        raise ValueError("slot_mapping must be int64[n_tokens]")
    for t, name in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        if tuple(t.shape) != desc.cache_shape or t.dtype != desc.torch_dtype:
            raise ValueError(f"{name} must be {desc.torch_dtype}{desc.cache_shape}")
    _check(lib().pkv_write(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _dev(k, "k"),
                           _dev(v, "v"), _dtype_code(k), _dev(slot_mapping, "slot_mapping", torch.int64),
                           n, ctypes.byref(desc), float(k_inv_scale), float(v_inv_scale),
                           _stream(stream)))


def _copy_blocks_args(k_caches, v_caches, src_dst, desc):
    pairs = np.ascontiguousarray(np.asarray(src_dst, dtype=np.int32).reshape(-1))
    n = len(pairs) // 2
    if n == 0:
        return None
    if len(k_caches) != len(v_caches):
        raise ValueError("k_caches and v_caches differ in length")
    for t in list(k_caches) + list(v_caches):
        if tuple(t.shape) != desc.cache_shape or t.dtype != desc.torch_dtype:
            raise ValueError("cache tensors do not match desc")
    kp = (_P * len(k_caches))(*[_dev(t, "k_cache") for t in k_caches])
    vp = (_P * len(v_caches))(*[_dev(t, "v_cache") for t in v_caches])
    return (kp, vp, len(k_caches), _i32p(pairs), n, ctypes.byref(desc)), (pairs, kp, vp, desc)


def pkv_copy_blocks(k_caches, v_caches, src_dst, desc: pkv_kv_desc, stream=None):
    """Copy blocks src -> dst in every layer; src_dst is a host int32 [n, 2]."""
    a = _copy_blocks_args(k_caches, v_caches, src_dst, desc)
    if a is not None:
        _check(lib().pkv_copy_blocks(*a[0], _stream(stream)))


def prepare_copy_blocks(k_caches, v_caches, src_dst, desc: pkv_kv_desc):
    """pkv_copy_blocks on these caches and pairs as a Prepared call (None when
    there are no pairs: nothing to launch)."""
    a = _copy_blocks_args(k_caches, v_caches, src_dst, desc)
    return None if a is None else Prepared(lib().pkv_copy_blocks, a[0], (a[1], list(k_caches),
                                                                           list(v_caches)))


def pkv_attention_workspace_bytes(num_seqs, num_q_heads, max_blocks, desc: pkv_kv_desc,
                                  partition_tokens=0) -> int:
    return int(lib().pkv_attention_workspace_bytes(num_seqs, num_q_heads, max_blocks,
                                                   ctypes.byref(desc), partition_tokens))


def pkv_attention_partition(num_seqs, max_blocks, desc: pkv_kv_desc, partition_tokens=0) -> int:
    return int(lib().pkv_attention_partition(num_seqs, max_blocks, ctypes.byref(desc), partition_tokens))


def pkv_set_attention_kernel(kind) -> None:
    """Process-wide decode kernel choice: "auto", "simt" or "tc"."""
    _check(lib().pkv_set_attention_kernel(KERNEL_OF_NAME.get(kind, kind)))


PREFILL_KERNEL_OF_NAME = {"auto": 0, "mma_sync": 1, "tcgen05": 2}


def pkv_set_prefill_kernel(kind) -> None:
    """Process-wide prefill kernel choice: "auto", "mma_sync" or "tcgen05"."""
    _check(lib().pkv_set_prefill_kernel(PREFILL_KERNEL_OF_NAME.get(kind, kind)))


def workspace_for(num_seqs, num_q_heads, max_blocks, desc, partition_tokens=0, device="cuda"):
    """A zero-filled workspace tensor of the size the decode call needs (None if 0)."""
    n = pkv_attention_workspace_bytes(num_seqs, num_q_heads, max_blocks, desc, partition_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


def pkv_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, desc: pkv_kv_desc,
                         softmax_scale, k_scale=1.0, v_scale=1.0, partition_tokens=0,
                         workspace=None, stream=None):
    """Decode attention of q [B, Hq, D] through block tables int32[B, max_blocks]."""
    b, hq, d = q.shape
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    if block_tables.dim() != 2 or block_tables.shape[0] != b:
        raise ValueError("block_tables must be int32[B, max_blocks]")
    if context_lens.shape != (b,):
        raise ValueError("context_lens must be int32[B]")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    _check(lib().pkv_attention_decode(
        _dev(out, "out"), _dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache", desc.torch_dtype),
        _dev(v_cache, "v_cache", desc.torch_dtype), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), b, hq,
        ctypes.byref(desc), float(softmax_scale), float(k_scale), float(v_scale),
        int(partition_tokens), ws_ptr, ws_bytes, _stream(stream)))
    return out


def _decode_step_args(out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                      desc, prefix_blocks, softmax_scale, k_scale, v_scale, k_inv_scale,
                      v_inv_scale, partition_tokens, workspace):
    """The checked, marshalled arguments of pkv_decode_step (prefix_blocks
    None) or pkv_decode_step_shared_prefix, without the stream."""
    b, hq, d = q.shape
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    if k_new.shape != v_new.shape or k_new.shape[0] != b or k_new.dtype != q.dtype:
        raise ValueError("k_new, v_new must be [B, N_kv, D] in q's dtype")
    if block_tables.dim() != 2 or block_tables.shape[0] != b or context_lens.shape != (b,):
        raise ValueError("block_tables int32[B, max_blocks], context_lens int32[B] expected")
    ws_ptr, ws_bytes = _ws(workspace)
    head = (_dev(out, "out"), _dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache", desc.torch_dtype),
            _dev(v_cache, "v_cache", desc.torch_dtype), _dev(k_new, "k_new"), _dev(v_new, "v_new"),
            _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
            _dev(context_lens, "context_lens", torch.int32), b, hq, ctypes.byref(desc))
    tail = (float(softmax_scale), float(k_scale), float(v_scale), float(k_inv_scale),
            float(v_inv_scale), int(partition_tokens), ws_ptr, ws_bytes)
    if prefix_blocks is None:
        return lib().pkv_decode_step, head + tail
    return lib().pkv_decode_step_shared_prefix, head + (int(prefix_blocks),) + tail


class Prepared:
    """A library call whose arguments were checked and marshalled once, for a
    loop that repeats it on the same buffers (a serving step re-issued with
    new contents in the same device memory).  ``call(stream)`` launches it on
    ``stream`` (a torch stream, a raw cudaStream_t as int, or None for the
    current stream).  The buffers must stay alive and keep their shapes."""

    def __init__(self, fn, args, keep):
        self._fn, self._args, self._keep = fn, args, keep

    def __call__(self, stream=None):
        _check(self._fn(*self._args, stream if isinstance(stream, int) else _stream(stream)))


def pkv_decode_step(out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                    desc: pkv_kv_desc, softmax_scale, k_scale=1.0, v_scale=1.0, k_inv_scale=1.0,
                    v_inv_scale=1.0, partition_tokens=0, workspace=None, stream=None):
    """The step's K/V written at position ctx - 1 of each sequence, then decode
    attention (one launch where the tensor-core split kernel applies)."""
    fn, args = _decode_step_args(out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                                 desc, None, softmax_scale, k_scale, v_scale, k_inv_scale,
                                 v_inv_scale, partition_tokens, workspace)
    _check(fn(*args, _stream(stream)))
    return out


def prepare_decode_step(out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                        desc: pkv_kv_desc, softmax_scale, k_scale=1.0, v_scale=1.0,
                        k_inv_scale=1.0, v_inv_scale=1.0, partition_tokens=0, workspace=None,
                        prefix_blocks=None) -> Prepared:
    """pkv_decode_step (or, with prefix_blocks, pkv_decode_step_shared_prefix)
    as a Prepared call on these buffers."""
    fn, args = _decode_step_args(out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                                 desc, prefix_blocks, softmax_scale, k_scale, v_scale, k_inv_scale,
                                 v_inv_scale, partition_tokens, workspace)
    return Prepared(fn, args, (out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                               desc, workspace))


def pkv_attention_prefill(out, q, k_cache, v_cache, block_tables, context_lens, query_start,
                          desc: pkv_kv_desc, softmax_scale, max_query_len=None, k_scale=1.0,
                          v_scale=1.0, stream=None):
    """Prefill attention of packed chunks q [total_q, Hq, D]; query_start
    int32[B + 1] (device) gives each sequence's rows.  ``max_query_len``
    defaults to the longest chunk (read back from query_start)."""
    total_q, hq, d = q.shape
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    b = context_lens.shape[0]
    if block_tables.dim() != 2 or block_tables.shape[0] != b or query_start.shape != (b + 1,):
        raise ValueError("block_tables int32[B, max_blocks], query_start int32[B + 1] expected")
    if max_query_len is None:
        max_query_len = int((query_start[1:] - query_start[:-1]).max().item()) if b else 0
    _check(lib().pkv_attention_prefill(
        _dev(out, "out"), _dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache", desc.torch_dtype),
        _dev(v_cache, "v_cache", desc.torch_dtype), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32),
        _dev(query_start, "query_start", torch.int32), b, total_q, int(max_query_len), hq,
        ctypes.byref(desc), float(softmax_scale), float(k_scale), float(v_scale), _stream(stream)))
    return out


def pkv_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                 desc: pkv_kv_desc, softmax_scale, k_scale=1.0, v_scale=1.0,
                                 partition_tokens=0, stream=None):
    """Decode attention for callers that cannot allocate device memory (for
    example a plug-in whose host owns all device memory, or a loop that must
    not call cudaMalloc): the split-K scratch is the library's own fixed
    16 MiB device array.  Same result as pkv_attention_decode; sizes that need
    more scratch raise INVALID_ARG."""
    b, hq, d = q.shape
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    if block_tables.dim() != 2 or block_tables.shape[0] != b or context_lens.shape != (b,):
        raise ValueError("block_tables must be int32[B, max_blocks], context_lens int32[B]")
    _check(lib().pkv_attention_decode_noalloc(
        _dev(out, "out"), _dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache", desc.torch_dtype),
        _dev(v_cache, "v_cache", desc.torch_dtype), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), b, hq,
        ctypes.byref(desc), float(softmax_scale), float(k_scale), float(v_scale),
        int(partition_tokens), _stream(stream)))
    return out


def pkv_shared_prefix_workspace_bytes(num_seqs, num_q_heads, max_blocks, desc: pkv_kv_desc,
                                      prefix_blocks, partition_tokens=0) -> int:
    return int(lib().pkv_shared_prefix_workspace_bytes(num_seqs, num_q_heads, max_blocks,
                                                       ctypes.byref(desc), int(prefix_blocks),
                                                       partition_tokens))


def shared_prefix_workspace_for(num_seqs, num_q_heads, max_blocks, desc, prefix_blocks,
                                partition_tokens=0, device="cuda"):
    """A zero-filled workspace for the shared-prefix decode calls (None if 0)."""
    n = pkv_shared_prefix_workspace_bytes(num_seqs, num_q_heads, max_blocks, desc, prefix_blocks,
                                          partition_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()


def pkv_attention_decode_shared_prefix(out, q, k_cache, v_cache, block_tables, context_lens,
                                       desc: pkv_kv_desc, prefix_blocks, softmax_scale, k_scale=1.0,
                                       v_scale=1.0, partition_tokens=0, workspace=None, stream=None):
    """Decode attention whose first ``prefix_blocks`` table entries are the
    same blocks in every row: the prefix is attended once for all sequences
    (pkv_attention_decode_shared_prefix)."""
    b, hq, d = q.shape
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    if block_tables.dim() != 2 or block_tables.shape[0] != b or context_lens.shape != (b,):
        raise ValueError("block_tables int32[B, max_blocks], context_lens int32[B] expected")
    ws_ptr, ws_bytes = _ws(workspace)
    _check(lib().pkv_attention_decode_shared_prefix(
        _dev(out, "out"), _dev(q, "q"), _dtype_code(q), _dev(k_cache, "k_cache", desc.torch_dtype),
        _dev(v_cache, "v_cache", desc.torch_dtype), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), b, hq,
        ctypes.byref(desc), int(prefix_blocks), float(softmax_scale), float(k_scale), float(v_scale),
        int(partition_tokens), ws_ptr, ws_bytes, _stream(stream)))
    return out


def pkv_decode_step_shared_prefix(out, q, k_cache, v_cache, k_new, v_new, block_tables,
                                  context_lens, desc: pkv_kv_desc, prefix_blocks, softmax_scale,
                                  k_scale=1.0, v_scale=1.0, k_inv_scale=1.0, v_inv_scale=1.0,
                                  partition_tokens=0, workspace=None, stream=None):
    """pkv_decode_step over a shared prefix (pkv_decode_step_shared_prefix)."""
    fn, args = _decode_step_args(out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens,
                                 desc, prefix_blocks, softmax_scale, k_scale, v_scale, k_inv_scale,
                                 v_inv_scale, partition_tokens, workspace)
    _check(fn(*args, _stream(stream)))
    return out


def pkv_device_status(clear: bool = False, stream=None) -> int:
    """The current device's error word (PKV_DEVICE_* bits), after
    synchronising ``stream``; ``clear`` resets it."""
    flags = ctypes.c_int32(0)
    _check(lib().pkv_device_status(ctypes.byref(flags), 1 if clear else 0, _stream(stream)))
    return flags.value


def pkv_set_stage_wait_limit(nanoseconds: int) -> None:
    """Give-up limit of the decode kernels' stage waits (default 50 ms)."""
    _check(lib().pkv_set_stage_wait_limit(int(nanoseconds)))
