"""Python binding of libkvx.so: the C ABI of ``include/kvx.h`` under the same names.

Argument marshalling only: every step of a copy (validation, chunking,
packing, upload, the copy kernel) runs inside libkvx.so. Descriptor arrays
are numpy ``uint64`` arrays (or anything ``np.asarray`` turns into one);
streams are ``torch.cuda.Stream`` objects, raw ``cudaStream_t`` integers, or
``None`` for the legacy default stream. A non-OK status raises ``KvxError``
carrying the status and the library's message.

The library must have been built (``__graft_entry__.build()`` or
``python -m expert_host_block_gb300.build``); importing this module without
it raises at once. There is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB_PATH

KVX_H2D, KVX_D2H, KVX_D2D = 0, 1, 2
DIRS = {"h2d": KVX_H2D, "d2h": KVX_D2H, "d2d": KVX_D2D}
KVX_VARIANT_AUTO, KVX_VARIANT_LDG, KVX_VARIANT_BULK, KVX_VARIANT_STAGE = 0, 1, 2, 3
VARIANTS = {"auto": KVX_VARIANT_AUTO, "ldg": KVX_VARIANT_LDG, "bulk": KVX_VARIANT_BULK,
            "stage": KVX_VARIANT_STAGE}
KVX_ASSIGN_AUTO, KVX_ASSIGN_STATIC, KVX_ASSIGN_DYNAMIC = 0, 1, 2
ASSIGNS = {"auto": KVX_ASSIGN_AUTO, "static": KVX_ASSIGN_STATIC, "dynamic": KVX_ASSIGN_DYNAMIC}

KVX_OK = 0
KVX_ERR_INVALID_ARG = 1
KVX_ERR_ALIGN = 2
KVX_ERR_OVERLAP = 3
KVX_ERR_CAPACITY = 4
KVX_ERR_NOT_MAPPED = 5
KVX_ERR_CUDA = 6
KVX_ERR_TIMEOUT = 7
KVX_ERR_DEVICE_FAULT = 8
KVX_ERR_CAPTURE = 9

# the C ABI version this binding's structures follow (KVX_VERSION_MAJOR * 100 + KVX_VERSION_MINOR)
KVX_VERSION = 4

KVX_CHUNK_BYTES = 16384
KVX_MAX_CHUNKS = 1 << 22

CHUNK_DTYPE = np.dtype([("src", "<u8"), ("dst", "<u8"), ("len", "<u4"), ("desc", "<u4"),
                        ("reserved", "<u8")])

# Every symbol include/kvx.h declares.
EXPORTS = (
    "kvx_copy_batch", "kvx_copy_batch_ex", "kvx_desc_buf_create", "kvx_upload_descriptors",
    "kvx_copy_uploaded", "kvx_copy_uploaded_ex", "kvx_desc_buf_info", "kvx_desc_buf_destroy",
    "kvx_validate", "kvx_plan_chunks", "kvx_default_launch", "kvx_set_validate_level",
    "kvx_get_validate_level", "kvx_status_string", "kvx_last_error", "kvx_version", "kvx_select_launch",
    "kvx_stream_check", "kvx_host_alloc", "kvx_host_free", "kvx_copy_batch_memcpy",
    "kvx_copy_contiguous", "kvx_copy_batch_noalloc", "kvx_selftest_wait_timeout", "kvx_debug_bounds",
    "kvx_devlist_create", "kvx_devlist_destroy", "kvx_copy_device_list",
    "kvx_transfer_create", "kvx_transfer_start", "kvx_transfer_poll", "kvx_transfer_progress",
    "kvx_transfer_destroy", "kvx_auto_path", "kvx_copy_batch_auto", "kvx_device_query",
    "kvx_status_enqueue", "kvx_status_wait", "kvx_status_query",
    # include/kvx_standin.h
    "kvx_standin_gemv_bf16",
)


class kvx_status_token(ctypes.Structure):
    _fields_ = [("slot", ctypes.c_uint64), ("gen", ctypes.c_uint64), ("device", ctypes.c_int)]


class kvx_launch(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("cta_budget", ctypes.c_int), ("threads", ctypes.c_int),
                ("unroll", ctypes.c_int), ("stages", ctypes.c_int), ("store_policy", ctypes.c_int),
                ("assign", ctypes.c_int)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


class KvxError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.name = status_string(status) if _lib is not None else str(status)
        super().__init__(f"{self.name}: {message}")


_lib = None
_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_u64 = ctypes.c_uint64
_int = ctypes.c_int


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'` (no fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "kvx_copy_batch": ([_vp, _vp, _vp, _sz, _int, _int, _vp], _int),
        "kvx_copy_batch_ex": ([_vp, _vp, _vp, _sz, _int, ctypes.POINTER(kvx_launch), _vp], _int),
        "kvx_desc_buf_create": ([_sz, ctypes.POINTER(_vp)], _int),
        "kvx_upload_descriptors": ([_vp, _vp, _vp, _vp, _sz, _int, _vp], _int),
        "kvx_copy_uploaded": ([_vp, _int, _vp], _int),
        "kvx_copy_uploaded_ex": ([_vp, ctypes.POINTER(kvx_launch), _vp], _int),
        "kvx_desc_buf_info": ([_vp, ctypes.POINTER(_sz), ctypes.POINTER(_u64), ctypes.POINTER(kvx_launch)], _int),
        "kvx_desc_buf_destroy": ([_vp], _int),
        "kvx_validate": ([_vp, _vp, _vp, _sz, _int, _int], _int),
        "kvx_plan_chunks": ([_vp, _vp, _vp, _sz, _vp, _sz, ctypes.POINTER(_sz)], _int),
        "kvx_default_launch": ([_int, _u64, ctypes.POINTER(kvx_launch)], _int),
        "kvx_select_launch": ([_vp, _vp, _vp, _sz, _int, ctypes.POINTER(kvx_launch),
                               ctypes.POINTER(kvx_launch)], _int),
        "kvx_set_validate_level": ([_int], _int),
        "kvx_get_validate_level": ([], _int),
        "kvx_status_string": ([_int], ctypes.c_char_p),
        "kvx_last_error": ([], ctypes.c_char_p),
        "kvx_version": ([], _int),
        "kvx_stream_check": ([_vp], _int),
        "kvx_host_alloc": ([_sz, ctypes.POINTER(_vp)], _int),
        "kvx_host_free": ([_vp], _int),
        "kvx_copy_batch_memcpy": ([_vp, _vp, _vp, _sz, _int, _vp, ctypes.POINTER(_sz)], _int),
        "kvx_copy_contiguous": ([_u64, _u64, _u64, _int, _vp], _int),
        "kvx_selftest_wait_timeout": ([_u64, _vp], _int),
        "kvx_debug_bounds": ([_vp, _vp, _sz], _int),
        "kvx_copy_batch_noalloc": ([_vp, _vp, _vp, _sz, _int, _int, _vp], _int),
        "kvx_devlist_create": ([ctypes.c_uint32, ctypes.POINTER(_vp)], _int),
        "kvx_transfer_create": ([ctypes.POINTER(_vp)], _int),
        "kvx_transfer_start": ([_vp, _vp, _vp, _vp, _sz, _int, _sz, ctypes.POINTER(kvx_launch), _vp], _int),
        "kvx_transfer_poll": ([_vp, ctypes.POINTER(_int)], _int),
        "kvx_transfer_progress": ([_vp, ctypes.POINTER(_sz), ctypes.POINTER(_sz)], _int),
        "kvx_transfer_destroy": ([_vp], _int),
        "kvx_auto_path": ([_vp, _vp, _vp, _sz, _int, _int, ctypes.POINTER(_int)], _int),
        "kvx_device_query": ([ctypes.POINTER(_int), ctypes.POINTER(_sz), ctypes.POINTER(_sz), ctypes.POINTER(_sz)],
                             _int),
        "kvx_status_enqueue": ([_vp, ctypes.POINTER(kvx_status_token)], _int),
        "kvx_status_wait": ([ctypes.POINTER(kvx_status_token)], _int),
        "kvx_status_query": ([ctypes.POINTER(kvx_status_token), ctypes.POINTER(_int)], _int),
        "kvx_copy_batch_auto": ([_vp, _vp, _vp, _sz, _int, _int, _vp, ctypes.POINTER(_int)], _int),
        "kvx_devlist_destroy": ([_vp], _int),
        "kvx_copy_device_list": ([_vp, _u64, _u64, _u64, _u64, _int, ctypes.POINTER(kvx_launch), _vp], _int),
        "kvx_standin_gemv_bf16": ([_u64, _u64, _u64, _u64, ctypes.c_uint32, _int, _vp], _int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if lib.kvx_version() != KVX_VERSION:
        raise RuntimeError(f"{LIB_PATH} implements C ABI version {lib.kvx_version()}, this binding "
                           f"version {KVX_VERSION}: rebuild the library")
    _lib = lib
    return lib


def lib():
    """The loaded ctypes library (raises if it was not built)."""
    return _load()


def status_string(status: int) -> str:
    return _load().kvx_status_string(status).decode()


def last_error() -> str:
    return _load().kvx_last_error().decode()


def _check(status: int) -> None:
    if status != KVX_OK:
        raise KvxError(status, last_error())


def _u64arr(a) -> np.ndarray:
    if isinstance(a, np.ndarray) and a.dtype == np.uint64 and a.flags.c_contiguous:
        return a
    if hasattr(a, "numpy") and not isinstance(a, np.ndarray):  # torch CPU tensor
        a = a.numpy()
    return np.ascontiguousarray(np.asarray(a).astype(np.uint64, copy=False).reshape(-1))


def _stream(s) -> int:
    if s is None:
        return 0
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError(f"not a stream: {s!r}")


def _triple(src_addrs, dst_addrs, sizes, n):
    s, d, z = _u64arr(src_addrs), _u64arr(dst_addrs), _u64arr(sizes)
    if n is None:
        n = z.size
    if not (s.size >= n and d.size >= n and z.size >= n):
        raise ValueError(f"descriptor arrays shorter than n = {n}")
    return s, d, z, int(n)


def _launch(launch) -> kvx_launch | None:
    if launch is None:
        return None
    if isinstance(launch, kvx_launch):
        return launch
    v = dict(launch)
    if isinstance(v.get("variant"), str):
        v["variant"] = VARIANTS[v["variant"]]
    if isinstance(v.get("assign"), str):
        v["assign"] = ASSIGNS[v["assign"]]
    return kvx_launch(**v)


def _dir(d) -> int:
    return DIRS[d] if isinstance(d, str) else int(d)


# ---- the batch copy --------------------------------------------------------

def kvx_copy_batch(src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, cta_budget=0, stream=None) -> None:
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    _check(_load().kvx_copy_batch(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir),
                                  int(cta_budget), _stream(stream)))


def kvx_copy_batch_ex(src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, launch=None, stream=None) -> None:
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    lp = _launch(launch)
    _check(_load().kvx_copy_batch_ex(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir),
                                     ctypes.byref(lp) if lp is not None else None, _stream(stream)))


class Descriptors:
    """Reusable descriptor arrays with their addresses taken once.

    The vLLM offloading connector keeps its descriptor arrays as buffers it
    allocates once and refills for every transfer (vLLM PR #42212 report,
    §实现拆解 item 3). This is that pattern on the Python side: three uint64
    arrays of a fixed capacity whose addresses are looked up at construction,
    so a call only marshals integers. Fill ``src``, ``dst`` and ``sizes``
    (directly, or with ``set``), then call ``copy_batch``.
    """

    def __init__(self, capacity: int):
        self.capacity = int(capacity)
        self.src = np.zeros(self.capacity, dtype=np.uint64)
        self.dst = np.zeros(self.capacity, dtype=np.uint64)
        self.sizes = np.zeros(self.capacity, dtype=np.uint64)
        self.n = 0
        self._ptrs = (self.src.ctypes.data, self.dst.ctypes.data, self.sizes.ctypes.data)
        self._fn = _load().kvx_copy_batch

    def set(self, src_addrs, dst_addrs, sizes) -> "Descriptors":
        n = len(sizes)
        if n > self.capacity:
            raise ValueError(f"{n} descriptors exceed capacity {self.capacity}")
        self.src[:n] = src_addrs
        self.dst[:n] = dst_addrs
        self.sizes[:n] = sizes
        self.n = n
        return self

    def copy_batch(self, dir, cta_budget: int = 0, stream=None) -> None:
        """kvx_copy_batch over the first ``n`` descriptors."""
        ps, pd, pz = self._ptrs
        st = self._fn(ps, pd, pz, self.n, DIRS[dir] if isinstance(dir, str) else dir, cta_budget,
                      _stream(stream))
        if st != KVX_OK:
            raise KvxError(st, last_error())


# ---- descriptor buffers ----------------------------------------------------

def kvx_desc_buf_create(max_chunks: int) -> int:
    h = _vp()
    _check(_load().kvx_desc_buf_create(int(max_chunks), ctypes.byref(h)))
    return h.value


def kvx_upload_descriptors(buf: int, src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, stream=None) -> None:
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    _check(_load().kvx_upload_descriptors(buf, s.ctypes.data, d.ctypes.data, z.ctypes.data, n,
                                          _dir(dir), _stream(stream)))


def kvx_copy_uploaded(buf: int, cta_budget=0, stream=None) -> None:
    _check(_load().kvx_copy_uploaded(buf, int(cta_budget), _stream(stream)))


def kvx_copy_uploaded_ex(buf: int, launch=None, stream=None) -> None:
    lp = _launch(launch)
    _check(_load().kvx_copy_uploaded_ex(buf, ctypes.byref(lp) if lp is not None else None,
                                        _stream(stream)))


def kvx_desc_buf_info(buf: int):
    """(n_chunks, payload_bytes, selected launch as a dict)."""
    n, p, l = _sz(), _u64(), kvx_launch()
    _check(_load().kvx_desc_buf_info(buf, ctypes.byref(n), ctypes.byref(p), ctypes.byref(l)))
    return n.value, p.value, l.as_dict()


def kvx_desc_buf_destroy(buf: int) -> None:
    _check(_load().kvx_desc_buf_destroy(buf))


class DescBuf:
    """A kvx_desc_buf owned by a Python object."""

    def __init__(self, max_chunks: int):
        self.handle = kvx_desc_buf_create(max_chunks)
        self.max_chunks = int(max_chunks)

    def upload(self, src_addrs, dst_addrs, sizes, dir, stream=None):
        kvx_upload_descriptors(self.handle, src_addrs, dst_addrs, sizes, None, dir, stream)

    def copy(self, cta_budget=0, stream=None, launch=None):
        if launch is None:
            kvx_copy_uploaded(self.handle, cta_budget, stream)
        else:
            kvx_copy_uploaded_ex(self.handle, launch, stream)

    def info(self):
        return kvx_desc_buf_info(self.handle)

    def close(self):
        if self.handle:
            kvx_desc_buf_destroy(self.handle)
            self.handle = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- descriptor lists that live on the device --------------------------------

def kvx_devlist_create(max_n: int) -> int:
    h = _vp()
    _check(_load().kvx_devlist_create(int(max_n), ctypes.byref(h)))
    return h.value


def kvx_devlist_destroy(handle: int) -> None:
    _check(_load().kvx_devlist_destroy(handle))


def kvx_copy_device_list(handle: int, d_src: int, d_dst: int, d_sizes: int, d_count: int, dir,
                         launch=None, stream=None) -> None:
    """Copy the list whose arrays and count are in device memory (device addresses)."""
    lp = _launch(launch)
    _check(_load().kvx_copy_device_list(handle, int(d_src), int(d_dst), int(d_sizes), int(d_count), _dir(dir),
                                        ctypes.byref(lp) if lp is not None else None, _stream(stream)))


class DeviceList:
    """A kvx_devlist owned by a Python object."""

    def __init__(self, max_n: int):
        self.handle = kvx_devlist_create(max_n)
        self.max_n = int(max_n)

    def copy(self, d_src: int, d_dst: int, d_sizes: int, d_count: int, dir, launch=None, stream=None):
        kvx_copy_device_list(self.handle, d_src, d_dst, d_sizes, d_count, dir, launch, stream)

    def close(self):
        if self.handle:
            kvx_devlist_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- Auto policy ----------------------------------------------------------------

KVX_POLICY_THROUGHPUT, KVX_POLICY_TAIL = 0, 1
POLICIES = {"throughput": KVX_POLICY_THROUGHPUT, "tail": KVX_POLICY_TAIL}
KVX_PATH_KERNEL_LDG, KVX_PATH_KERNEL_BULK, KVX_PATH_DMA, KVX_PATH_KERNEL_STAGE = 1, 2, 3, 4
PATHS = {KVX_PATH_KERNEL_LDG: "kernel_ldg", KVX_PATH_KERNEL_BULK: "kernel_bulk", KVX_PATH_DMA: "dma",
         KVX_PATH_KERNEL_STAGE: "kernel_stage"}


def _policy(p) -> int:
    return POLICIES[p] if isinstance(p, str) else int(p)


def kvx_auto_path(src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, policy="throughput") -> str:
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    out = _int()
    _check(_load().kvx_auto_path(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir), _policy(policy),
                                 ctypes.byref(out)))
    return PATHS[out.value]


def kvx_copy_batch_auto(src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, policy="throughput", stream=None) -> str:
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    out = _int()
    _check(_load().kvx_copy_batch_auto(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir),
                                       _policy(policy), _stream(stream), ctypes.byref(out)))
    return PATHS[out.value]


# ---- tail-bounded submission ---------------------------------------------------

class Transfer:
    """A kvx_transfer: a batch submitted in pieces, each after the previous one completed."""

    def __init__(self):
        h = _vp()
        _check(_load().kvx_transfer_create(ctypes.byref(h)))
        self.handle = h.value
        self._done = _int()

    def start(self, src_addrs, dst_addrs, sizes, dir, chunk_descriptors=0, launch=None, stream=None):
        s, d, z, n = _triple(src_addrs, dst_addrs, sizes, None)
        lp = _launch(launch)
        _check(_load().kvx_transfer_start(self.handle, s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir),
                                          int(chunk_descriptors), ctypes.byref(lp) if lp is not None else None,
                                          _stream(stream)))

    def poll(self) -> bool:
        """Submit the next piece if the last one completed; True once all pieces completed."""
        _check(_load().kvx_transfer_poll(self.handle, ctypes.byref(self._done)))
        return bool(self._done.value)

    def progress(self):
        a, b = _sz(), _sz()
        _check(_load().kvx_transfer_progress(self.handle, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def close(self):
        if self.handle:
            _check(_load().kvx_transfer_destroy(self.handle))
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- host-only helpers -----------------------------------------------------

def kvx_validate(src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, level=0) -> int:
    """The status kvx_copy_batch would return before enqueuing (does not raise)."""
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    return int(_load().kvx_validate(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir), int(level)))


def kvx_plan_chunks(src_addrs, dst_addrs, sizes, n=None) -> np.ndarray:
    """The chunk table (structured array of CHUNK_DTYPE) kvx would upload."""
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    cnt = _sz()
    L = _load()
    _check(L.kvx_plan_chunks(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, None, 0, ctypes.byref(cnt)))
    out = np.zeros(cnt.value, dtype=CHUNK_DTYPE)
    _check(L.kvx_plan_chunks(s.ctypes.data, d.ctypes.data, z.ctypes.data, n,
                             out.ctypes.data if out.size else None, out.size, ctypes.byref(cnt)))
    return out


def kvx_default_launch(dir, mean_chunk_bytes: int) -> dict:
    l = kvx_launch()
    _check(_load().kvx_default_launch(_dir(dir), int(mean_chunk_bytes), ctypes.byref(l)))
    return l.as_dict()


def kvx_select_launch(src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, launch=None) -> dict:
    """The launch kvx_copy_batch_ex would make for this batch (host only, no device needed)."""
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    lp = _launch(launch)
    out = kvx_launch()
    _check(_load().kvx_select_launch(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir),
                                     ctypes.byref(lp) if lp is not None else None, ctypes.byref(out)))
    return out.as_dict()


def kvx_set_validate_level(level: int) -> None:
    _check(_load().kvx_set_validate_level(int(level)))


def kvx_get_validate_level() -> int:
    return int(_load().kvx_get_validate_level())


def kvx_version() -> int:
    return int(_load().kvx_version())


# ---- device status, memory -------------------------------------------------

def kvx_stream_check(stream=None) -> None:
    _check(_load().kvx_stream_check(_stream(stream)))


def kvx_status_enqueue(stream=None) -> kvx_status_token:
    """Mark the current end of `stream`'s work (an event); returns the token whose wait reads the device's errors."""
    tok = kvx_status_token()
    _check(_load().kvx_status_enqueue(_stream(stream), ctypes.byref(tok)))
    return tok


def kvx_status_wait(tok: kvx_status_token) -> None:
    """Block until the stream reached the token, then read the device's errors; raises like kvx_stream_check."""
    _check(_load().kvx_status_wait(ctypes.byref(tok)))


def kvx_status_query(tok: kvx_status_token) -> bool:
    """True once the stream reached the token (raising if the device reported an error); False while pending."""
    r = _int()
    _check(_load().kvx_status_query(ctypes.byref(tok), ctypes.byref(r)))
    return bool(r.value)


def kvx_device_query() -> dict:
    """SM count, per-thread stack limit and free / total memory of the current device."""
    sms, stack, free, total = _int(), _sz(), _sz(), _sz()
    _check(_load().kvx_device_query(ctypes.byref(sms), ctypes.byref(stack), ctypes.byref(free), ctypes.byref(total)))
    return {"sm_count": sms.value, "stack_bytes_per_thread": stack.value, "free_bytes": free.value,
            "total_bytes": total.value}


def kvx_host_alloc(nbytes: int) -> int:
    p = _vp()
    _check(_load().kvx_host_alloc(int(nbytes), ctypes.byref(p)))
    return p.value


def kvx_host_free(addr: int) -> None:
    _check(_load().kvx_host_free(addr))


class HostBuffer:
    """Mapped pinned host memory from kvx_host_alloc, viewable as a numpy array."""

    def __init__(self, nbytes: int):
        self.nbytes = int(nbytes)
        self.addr = kvx_host_alloc(self.nbytes)
        self._view = np.ctypeslib.as_array((ctypes.c_uint8 * self.nbytes).from_address(self.addr))

    def numpy(self) -> np.ndarray:
        return self._view

    def close(self):
        if self.addr:
            self._view = None
            kvx_host_free(self.addr)
            self.addr = 0

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---- baselines -------------------------------------------------------------

def kvx_copy_batch_memcpy(src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, stream=None) -> int:
    """Per-range directional cudaMemcpyAsync; returns the number of memcpy calls."""
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    r = _sz()
    _check(_load().kvx_copy_batch_memcpy(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir),
                                         _stream(stream), ctypes.byref(r)))
    return r.value


def kvx_copy_contiguous(dst: int, src: int, nbytes: int, dir, stream=None) -> None:
    _check(_load().kvx_copy_contiguous(int(dst), int(src), int(nbytes), _dir(dir), _stream(stream)))


KVX_NOALLOC_MAX_CHUNKS = 65536


def kvx_copy_batch_noalloc(src_addrs, dst_addrs, sizes, n=None, dir=KVX_H2D, cta_budget=0, stream=None) -> None:
    """kvx_copy_batch for callers that cannot allocate at copy time (two fixed 2 MiB device tables).

    At most KVX_NOALLOC_MAX_CHUNKS chunks per call; not allowed during stream
    capture. Calls on one stream or on several are ordered by the library: each
    upload waits for the last copy that read its table (see include/kvx.h).
    """
    s, d, z, n = _triple(src_addrs, dst_addrs, sizes, n)
    _check(_load().kvx_copy_batch_noalloc(s.ctypes.data, d.ctypes.data, z.ctypes.data, n, _dir(dir),
                                          int(cta_budget), _stream(stream)))


KVX_DEBUG_BOUNDS_MAX = 64


def kvx_debug_bounds(lo, hi) -> None:
    """Register the address ranges [lo[i], hi[i]) every copy must stay inside (empty: check off)."""
    a = np.ascontiguousarray(np.asarray(lo, dtype=np.uint64).reshape(-1))
    b = np.ascontiguousarray(np.asarray(hi, dtype=np.uint64).reshape(-1))
    if a.size != b.size:
        raise ValueError("lo and hi differ in length")
    _check(_load().kvx_debug_bounds(a.ctypes.data if a.size else None, b.ctypes.data if b.size else None,
                                    a.size))


def kvx_selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(_load().kvx_selftest_wait_timeout(int(timeout_ns), _stream(stream)))


# ---- decode stand-in (include/kvx_standin.h) -------------------------------

def kvx_standin_gemv_bf16(W: int, x: int, y: int, rows: int, cols: int, ctas: int = 0, stream=None) -> None:
    """y = W @ x with W (rows x cols) and x in bf16, fp32 accumulation; device addresses."""
    st = _load().kvx_standin_gemv_bf16(int(W), int(x), int(y), int(rows), int(cols), int(ctas),
                                       _stream(stream))
    if st != KVX_OK:
        raise KvxError(st, "kvx_standin_gemv_bf16: bad arguments or launch failure")
