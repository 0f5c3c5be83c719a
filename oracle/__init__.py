"""kvx oracle: the plain CPU definition of a batched descriptor copy.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product (``expert_host_block_gb300``) never imports it, and this
package imports nothing from the product.

The arithmetic lives in ``kvx_oracle.c`` (plain C, compiled with gcc into
``oracle/_build/liboracle.so``). This module only marshals numpy arrays into
it. Every function works on host snapshots: byte pools as ``np.uint8`` arrays
and descriptors as ``np.uint64`` offsets into those pools.

Citations (what each function follows):

* ``copy_batch`` / ``copy_batch_bytewise``: the batch copy replaces one
  directional memcpy per fragment and must move the same bytes (PegaFlow issue
  #408, "Kernel transfer backend causes decode TPOT tail spikes under
  concurrent KV transfers", §Summary; vLLM PR #42212 report, §实现拆解 item 4;
  FreeToken issue #751, §What we changed).
* ``range_checksums``: the per-descriptor checksum invariant (64-bit FNV-1a,
  its published parameters).
* ``ranges_disjoint``: the reading that destination ranges of one batch do not
  overlap (the pages are silent; see the C file's header).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvx_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u64p = ctypes.POINTER(ctypes.c_uint64)


def build(force: bool = False) -> str:
    """Compile ``kvx_oracle.c`` with gcc (plain -O2, no target-specific flags)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC],
                       check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_copy_batch.argtypes = [_u8p, _u8p, _u64p, _u64p, _u64p, ctypes.c_size_t]
        lib.oracle_copy_batch.restype = None
        lib.oracle_copy_batch_bytewise.argtypes = [
            _u8p, ctypes.c_size_t, _u8p, _u64p, _u64p, _u64p, ctypes.c_size_t]
        lib.oracle_copy_batch_bytewise.restype = None
        lib.oracle_fnv1a64.argtypes = [_u8p, ctypes.c_size_t]
        lib.oracle_fnv1a64.restype = ctypes.c_uint64
        lib.oracle_range_checksums.argtypes = [_u8p, _u64p, _u64p, ctypes.c_size_t, _u64p]
        lib.oracle_range_checksums.restype = None
        lib.oracle_ranges_disjoint.argtypes = [_u64p, _u64p, ctypes.c_size_t]
        lib.oracle_ranges_disjoint.restype = ctypes.c_int
        _lib = lib
        return lib


def _bytes(a: np.ndarray) -> np.ndarray:
    if a.dtype != np.uint8 or a.ndim != 1 or not a.flags.c_contiguous:
        raise TypeError("byte pools must be contiguous 1-D np.uint8 arrays")
    return a


def _u64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint64).reshape(-1))


def _check_bounds(pool_bytes: int, off: np.ndarray, sizes: np.ndarray, what: str) -> None:
    if off.size and int((off + sizes).max()) > pool_bytes:
        raise ValueError(f"a {what} range ends past its pool ({pool_bytes} bytes)")


def copy_batch(dst_pool: np.ndarray, src_pool: np.ndarray, src_off, dst_off, sizes) -> None:
    """In place: for each i, ``dst_pool[dst_off[i]:+sizes[i]] = src_pool[src_off[i]:+sizes[i]]``.

    ``dst_pool`` and ``src_pool`` may be the same array (a copy inside one pool)
    when no destination range overlaps a source range.
    """
    lib = _load()
    _bytes(dst_pool), _bytes(src_pool)
    s, d, z = _u64(src_off), _u64(dst_off), _u64(sizes)
    if not (s.size == d.size == z.size):
        raise ValueError("src_off, dst_off and sizes differ in length")
    _check_bounds(src_pool.size, s, z, "source")
    _check_bounds(dst_pool.size, d, z, "destination")
    lib.oracle_copy_batch(dst_pool.ctypes.data_as(_u8p), src_pool.ctypes.data_as(_u8p),
                          s.ctypes.data_as(_u64p), d.ctypes.data_as(_u64p),
                          z.ctypes.data_as(_u64p), s.size)


def copy_batch_bytewise(dst_pool: np.ndarray, src_pool: np.ndarray, src_off, dst_off, sizes) -> None:
    """The per-output-byte formulation of ``copy_batch`` (quadratic; tiny pools only)."""
    lib = _load()
    _bytes(dst_pool), _bytes(src_pool)
    s, d, z = _u64(src_off), _u64(dst_off), _u64(sizes)
    if not (s.size == d.size == z.size):
        raise ValueError("src_off, dst_off and sizes differ in length")
    _check_bounds(src_pool.size, s, z, "source")
    _check_bounds(dst_pool.size, d, z, "destination")
    lib.oracle_copy_batch_bytewise(dst_pool.ctypes.data_as(_u8p), dst_pool.size,
                                   src_pool.ctypes.data_as(_u8p), s.ctypes.data_as(_u64p),
                                   d.ctypes.data_as(_u64p), z.ctypes.data_as(_u64p), s.size)


def fnv1a64(data) -> int:
    """64-bit FNV-1a of a bytes-like object or a uint8 array."""
    lib = _load()
    a = np.frombuffer(bytes(data), dtype=np.uint8) if not isinstance(data, np.ndarray) else _bytes(data)
    a = np.ascontiguousarray(a)
    return int(lib.oracle_fnv1a64(a.ctypes.data_as(_u8p), a.size))


def range_checksums(pool: np.ndarray, off, sizes) -> np.ndarray:
    """FNV-1a of each range ``pool[off[i]:off[i]+sizes[i]]`` as a uint64 array."""
    lib = _load()
    _bytes(pool)
    o, z = _u64(off), _u64(sizes)
    _check_bounds(pool.size, o, z, "checksum")
    out = np.zeros(o.size, dtype=np.uint64)
    lib.oracle_range_checksums(pool.ctypes.data_as(_u8p), o.ctypes.data_as(_u64p),
                               z.ctypes.data_as(_u64p), o.size, out.ctypes.data_as(_u64p))
    return out


def ranges_disjoint(off, sizes) -> bool:
    """True when the non-empty ranges ``[off[i], off[i]+sizes[i])`` share no byte."""
    lib = _load()
    o, z = _u64(off), _u64(sizes)
    r = lib.oracle_ranges_disjoint(o.ctypes.data_as(_u64p), z.ctypes.data_as(_u64p), o.size)
    if r < 0:
        raise MemoryError("oracle_ranges_disjoint: out of memory")
    return bool(r)
