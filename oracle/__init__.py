"""CPU oracle of the compressed stream (bf16, fp16, fp32) and the fused compressed reduce.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg (``bench.py``) may import this package.  The GPU
library never imports, links or calls it, and it shares no code with the GPU
library.

The arithmetic lives in ``cccl_oracle.c`` (plain single-threaded C, built with
``-O2 -ffp-contract=off``, no fast-math).  This module only builds it and
marshals numpy arrays.  Method source: "CCCL: In-GPU Compression-Coupled
Collective Communication", sections 4.1, 4.3, 4.4 and 5, and Figure 2.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cccl_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_CORRUPT = 0, 1, 2, 3
CHUNK_ELEMS = 4096


def build(force: bool = False) -> str:
    """Compile ``cccl_oracle.c`` into ``liboracle.so`` next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
             "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    sz, u8p, u16p = ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p
    lib.oracle_n_chunks.argtypes = [sz]
    lib.oracle_n_chunks.restype = sz
    lib.oracle_data_start.argtypes = [sz]
    lib.oracle_data_start.restype = sz
    lib.oracle_compress_bound.argtypes = [sz]
    lib.oracle_compress_bound.restype = sz
    lib.oracle_plane_position.argtypes = [ctypes.c_uint, ctypes.POINTER(ctypes.c_uint),
                                          ctypes.POINTER(ctypes.c_uint)]
    lib.oracle_plane_element.argtypes = [ctypes.c_uint, ctypes.c_uint]
    lib.oracle_plane_element.restype = ctypes.c_uint
    lib.oracle_chunk_choice.argtypes = [u16p, sz] + [ctypes.POINTER(ctypes.c_uint)] * 3 + \
        [ctypes.POINTER(sz)] * 2
    lib.oracle_encode_chunk.argtypes = [u16p, sz, u8p, ctypes.POINTER(sz)]
    lib.oracle_compress.argtypes = [u16p, sz, u8p, sz, ctypes.POINTER(sz)]
    lib.oracle_decompress.argtypes = [u8p, sz, u16p, sz]
    lib.oracle_round_bf16.argtypes = [ctypes.c_float]
    lib.oracle_round_bf16.restype = ctypes.c_uint16
    lib.oracle_sum_ranks.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, sz, u16p]
    lib.oracle_reduce.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(sz), ctypes.c_int, sz,
                                  u8p, sz, ctypes.POINTER(sz)]
    lib.oracle_reduce_mixed.argtypes = [u16p, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(sz), ctypes.c_int,
                                        sz, u8p, sz, ctypes.POINTER(sz)]
    lib.oracle_reduce_op.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(sz), ctypes.c_int, sz,
                                     ctypes.c_int, u8p, sz, ctypes.POINTER(sz)]
    lib.oracle_compress_window.argtypes = [u16p, sz, u8p, sz, ctypes.POINTER(sz)]
    lib.oracle_compress_paged.argtypes = [u16p, sz, ctypes.c_void_p, sz, u8p, sz, ctypes.POINTER(sz)]
    lib.oracle_decompress_paged.argtypes = [u8p, sz, u16p, sz, ctypes.c_void_p, sz]
    vp, ip = ctypes.c_void_p, ctypes.c_int
    lib.oracle_compress_bound_typed.argtypes = [ip, sz]
    lib.oracle_compress_bound_typed.restype = sz
    lib.oracle_chunk_choice_typed.argtypes = [ip, vp, sz] + [ctypes.POINTER(ctypes.c_uint)] * 3 + \
        [ctypes.POINTER(sz)] * 2
    lib.oracle_encode_chunk_typed.argtypes = [ip, vp, sz, u8p, ctypes.POINTER(sz)]
    lib.oracle_compress_typed.argtypes = [ip, vp, sz, u8p, sz, ctypes.POINTER(sz), ip]
    lib.oracle_decompress_typed.argtypes = [ip, u8p, sz, vp, sz]
    lib.oracle_sum_ranks_typed.argtypes = [ip, ctypes.POINTER(ctypes.c_void_p), ip, sz, vp]
    lib.oracle_reduce_typed.argtypes = [ip, ip, vp, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(sz), ip, sz,
                                        u8p, sz, ctypes.POINTER(sz)]
    lib.oracle_round_fp16.argtypes = [ctypes.c_float]
    lib.oracle_round_fp16.restype = ctypes.c_uint16
    lib.oracle_fp16_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_fp16_to_float.restype = ctypes.c_float
    for f in ("oracle_chunk_choice_typed", "oracle_encode_chunk_typed", "oracle_compress_typed",
              "oracle_decompress_typed", "oracle_sum_ranks_typed", "oracle_reduce_typed",
              "oracle_chunk_choice", "oracle_encode_chunk", "oracle_compress", "oracle_decompress",
              "oracle_reduce", "oracle_reduce_mixed", "oracle_compress_paged", "oracle_decompress_paged",
              "oracle_compress_window", "oracle_reduce_op"):
        getattr(lib, f).restype = ctypes.c_int
    lib.oracle_sum_ranks.restype = None
    lib.oracle_plane_position.restype = None
    return lib


_lib = None
_override = None  # a library built from another source (the mutation tests use it)


def _load():
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        _lib = _bind(build())
    return _lib


class use_library:
    """Context manager: route this module's calls to another build of the
    oracle source (used only to check that the pins catch planted mistakes)."""

    def __init__(self, path: str):
        self.lib = _bind(path)

    def __enter__(self):
        global _override
        _override = self.lib
        return self

    def __exit__(self, *exc):
        global _override
        _override = None
        return False


def build_from(src: str, out: str) -> str:
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                           "-w", "-o", out, src, "-lm"])
    return out


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed with status %d" % (what, status))
        self.status = status


def _u16(x) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        a = a.view(np.uint16) if a.dtype.itemsize == 2 else a.astype(np.uint16)
    return a


def n_chunks(n: int) -> int:
    return _load().oracle_n_chunks(n)


def data_start(n: int) -> int:
    return _load().oracle_data_start(n)


def compress_bound(n: int) -> int:
    return _load().oracle_compress_bound(n)


def plane_position(i: int) -> tuple[int, int]:
    w, b = ctypes.c_uint(), ctypes.c_uint()
    _load().oracle_plane_position(i, ctypes.byref(w), ctypes.byref(b))
    return w.value, b.value


def plane_element(word: int, bit: int) -> int:
    return int(_load().oracle_plane_element(word, bit))


def chunk_choice(x) -> dict:
    """Encoding decision for one chunk: raw, k, base, n_esc, bytes."""
    a = _u16(x)
    raw, k, base = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
    n_esc, nbytes = ctypes.c_size_t(), ctypes.c_size_t()
    st = _load().oracle_chunk_choice(a.ctypes.data, a.size, ctypes.byref(raw), ctypes.byref(k), ctypes.byref(base),
                                     ctypes.byref(n_esc), ctypes.byref(nbytes))
    if st != OK:
        raise OracleError(st, "oracle_chunk_choice")
    return dict(raw=raw.value, k=k.value, base=base.value, n_esc=n_esc.value, bytes=nbytes.value)


def encode_chunk(x) -> bytes:
    """One chunk (header included) encoded on its own."""
    a = _u16(x)
    out = np.zeros(16 + 2 * CHUNK_ELEMS, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_encode_chunk(a.ctypes.data, a.size, out.ctypes.data, ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_encode_chunk")
    return out[:nb.value].tobytes()


def compress(x) -> np.ndarray:
    """bf16 bits (uint16 array) -> compressed stream (uint8 array)."""
    a = _u16(x).reshape(-1)
    cap = compress_bound(a.size)
    out = np.empty(cap, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_compress(a.ctypes.data, a.size, out.ctypes.data, cap, ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_compress")
    return out[:nb.value]


def decompress(s, n: int) -> np.ndarray:
    """Compressed stream -> n bf16 bit patterns; raises OracleError on a bad stream."""
    b = np.ascontiguousarray(np.frombuffer(bytes(s), np.uint8) if isinstance(s, (bytes, bytearray)) else s,
                             dtype=np.uint8)
    out = np.empty(n, np.uint16)
    st = _load().oracle_decompress(b.ctypes.data, b.size, out.ctypes.data, n)
    if st != OK:
        raise OracleError(st, "oracle_decompress")
    return out


def decompress_status(s, n: int) -> int:
    try:
        decompress(s, n)
        return OK
    except OracleError as e:
        return e.status


def round_bf16(f: float) -> int:
    return int(_load().oracle_round_bf16(ctypes.c_float(f)))


def sum_ranks(xs) -> np.ndarray:
    """Element-wise binary32 sum in rank order, rounded once to bf16."""
    arrs = [_u16(x).reshape(-1) for x in xs]
    n = arrs[0].size
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    out = np.empty(n, np.uint16)
    _load().oracle_sum_ranks(ptrs, len(arrs), n, out.ctypes.data)
    return out


def reduce_mixed(local, streams, n: int) -> np.ndarray:
    """Local uncompressed operand (rank 0) and compressed streams (ranks 1..)
    -> compressed stream of their rounded binary32 sum."""
    loc = _u16(local).reshape(-1)
    if loc.size != n:
        raise ValueError("local operand must hold n values")
    bs = [np.ascontiguousarray(s, dtype=np.uint8) for s in streams]
    ptrs = (ctypes.c_void_p * max(len(bs), 1))(*[b.ctypes.data for b in bs])
    sizes = (ctypes.c_size_t * max(len(bs), 1))(*[b.size for b in bs])
    cap = compress_bound(n)
    out = np.empty(cap, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_reduce_mixed(loc.ctypes.data, ptrs, sizes, len(bs), n, out.ctypes.data, cap,
                                     ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_reduce_mixed")
    return out[:nb.value]


def compress_window(x) -> np.ndarray:
    """Window-base variant (stream version 2) of compress."""
    x = _u16(x).reshape(-1)
    cap = compress_bound(x.size)
    out = np.empty(cap, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_compress_window(x.ctypes.data, x.size, out.ctypes.data, cap, ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_compress_window")
    return out[:nb.value]


def compress_paged(pool, block_elems: int, table) -> np.ndarray:
    """Stream of the blocks pool[table[i]] (block_elems values each), in order."""
    pool = _u16(pool).reshape(-1)
    tab = np.ascontiguousarray(table, dtype=np.int32)
    n = tab.size * block_elems
    cap = compress_bound(n)
    out = np.empty(cap, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_compress_paged(pool.ctypes.data, block_elems, tab.ctypes.data, tab.size, out.ctypes.data,
                                       cap, ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_compress_paged")
    return out[:nb.value]


def decompress_paged(s, pool, block_elems: int, table) -> np.ndarray:
    """A copy of ``pool`` with the stream's blocks written where the table says."""
    b = np.ascontiguousarray(s, dtype=np.uint8)
    out = _u16(pool).reshape(-1).copy()
    tab = np.ascontiguousarray(table, dtype=np.int32)
    st = _load().oracle_decompress_paged(b.ctypes.data, b.size, out.ctypes.data, block_elems, tab.ctypes.data, tab.size)
    if st != OK:
        raise OracleError(st, "oracle_decompress_paged")
    return out


OP_SUM, OP_MIN, OP_MAX = 0, 1, 2


def reduce_op(streams, n: int, op: int) -> np.ndarray:
    """reduce with op OP_SUM, OP_MIN or OP_MAX."""
    bs = [np.ascontiguousarray(s, dtype=np.uint8) for s in streams]
    ptrs = (ctypes.c_void_p * len(bs))(*[b.ctypes.data for b in bs])
    sizes = (ctypes.c_size_t * len(bs))(*[b.size for b in bs])
    cap = compress_bound(n)
    out = np.empty(cap, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_reduce_op(ptrs, sizes, len(bs), n, op, out.ctypes.data, cap, ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_reduce_op")
    return out[:nb.value]


def reduce(streams, n: int) -> np.ndarray:
    """R compressed streams -> compressed stream of their rounded binary32 sum."""
    bs = [np.ascontiguousarray(s, dtype=np.uint8) for s in streams]
    ptrs = (ctypes.c_void_p * len(bs))(*[b.ctypes.data for b in bs])
    sizes = (ctypes.c_size_t * len(bs))(*[b.size for b in bs])
    cap = compress_bound(n)
    out = np.empty(cap, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_reduce(ptrs, sizes, len(bs), n, out.ctypes.data, cap, ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_reduce")
    return out[:nb.value]


# ---------------------------------------------------------------------------
# element types: bf16, fp16, fp32 (the same split with 8-, 5- and 8-bit
# exponents).  Values travel as their bit patterns: uint16 for bf16 and fp16,
# uint32 for fp32.
# ---------------------------------------------------------------------------
DTYPE_BF16, DTYPE_FP16, DTYPE_FP32 = 1, 2, 3
_BITS = {DTYPE_BF16: np.uint16, DTYPE_FP16: np.uint16, DTYPE_FP32: np.uint32}


def _bits(dtype: int, x) -> np.ndarray:
    want = _BITS[dtype]
    a = np.ascontiguousarray(x)
    if a.dtype != want:
        a = a.view(want) if a.dtype.itemsize == np.dtype(want).itemsize else a.astype(want)
    return a.reshape(-1)


def compress_bound_typed(dtype: int, n: int) -> int:
    return _load().oracle_compress_bound_typed(dtype, n)


def chunk_choice_typed(dtype: int, x) -> dict:
    a = _bits(dtype, x)
    raw, k, base = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
    n_esc, nbytes = ctypes.c_size_t(), ctypes.c_size_t()
    st = _load().oracle_chunk_choice_typed(dtype, a.ctypes.data, a.size, ctypes.byref(raw), ctypes.byref(k),
                                           ctypes.byref(base), ctypes.byref(n_esc), ctypes.byref(nbytes))
    if st != OK:
        raise OracleError(st, "oracle_chunk_choice_typed")
    return dict(raw=raw.value, k=k.value, base=base.value, n_esc=n_esc.value, bytes=nbytes.value)


def encode_chunk_typed(dtype: int, x) -> bytes:
    a = _bits(dtype, x)
    out = np.zeros(16 + 4 * CHUNK_ELEMS, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_encode_chunk_typed(dtype, a.ctypes.data, a.size, out.ctypes.data, ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_encode_chunk_typed")
    return out[:nb.value].tobytes()


def compress_typed(dtype: int, x, window: bool = False) -> np.ndarray:
    """Bit patterns of one element type -> compressed stream (uint8 array)."""
    a = _bits(dtype, x)
    cap = compress_bound_typed(dtype, a.size)
    out = np.empty(cap, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_compress_typed(dtype, a.ctypes.data, a.size, out.ctypes.data, cap, ctypes.byref(nb),
                                       1 if window else 0)
    if st != OK:
        raise OracleError(st, "oracle_compress_typed")
    return out[:nb.value]


def decompress_typed(dtype: int, s, n: int) -> np.ndarray:
    b = np.ascontiguousarray(np.frombuffer(bytes(s), np.uint8) if isinstance(s, (bytes, bytearray)) else s,
                             dtype=np.uint8)
    out = np.empty(n, _BITS[dtype])
    st = _load().oracle_decompress_typed(dtype, b.ctypes.data, b.size, out.ctypes.data, n)
    if st != OK:
        raise OracleError(st, "oracle_decompress_typed")
    return out


def decompress_typed_status(dtype: int, s, n: int) -> int:
    try:
        decompress_typed(dtype, s, n)
        return OK
    except OracleError as e:
        return e.status


def sum_ranks_typed(dtype: int, xs) -> np.ndarray:
    arrs = [_bits(dtype, x) for x in xs]
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    out = np.empty(arrs[0].size, _BITS[dtype])
    st = _load().oracle_sum_ranks_typed(dtype, ptrs, len(arrs), arrs[0].size, out.ctypes.data)
    if st != OK:
        raise OracleError(st, "oracle_sum_ranks_typed")
    return out


def reduce_typed(dtype: int, streams, n: int, op: int = 0, local=None) -> np.ndarray:
    """Reduce (op OP_SUM, OP_MIN, OP_MAX) of an optional local operand (rank
    0) and compressed streams -> compressed stream of the result."""
    bs = [np.ascontiguousarray(s, dtype=np.uint8) for s in streams]
    ptrs = (ctypes.c_void_p * max(len(bs), 1))(*[b.ctypes.data for b in bs])
    sizes = (ctypes.c_size_t * max(len(bs), 1))(*[b.size for b in bs])
    loc = None
    if local is not None:
        loc = _bits(dtype, local)
        if loc.size != n:
            raise ValueError("local operand must hold n values")
    cap = compress_bound_typed(dtype, n)
    out = np.empty(cap, np.uint8)
    nb = ctypes.c_size_t()
    st = _load().oracle_reduce_typed(dtype, op, None if loc is None else loc.ctypes.data, ptrs, sizes, len(bs), n,
                                     out.ctypes.data, cap, ctypes.byref(nb))
    if st != OK:
        raise OracleError(st, "oracle_reduce_typed")
    return out[:nb.value]


def round_fp16(f: float) -> int:
    return int(_load().oracle_round_fp16(ctypes.c_float(f)))


def fp16_to_float(h: int) -> float:
    return float(_load().oracle_fp16_to_float(h))
