"""Python binding of libcccl: compressed bf16 (and fp16, fp32) communication
buffers and the fused compressed reduce, on one GB300 GPU.

Every function here marshals arguments for the C ABI of ``include/cccl.h``
(same names) and calls it; all compute runs in the library's sm_103a kernels.
torch supplies device memory and streams only.  There is no fallback: importing
this package raises ImportError when ``libcccl.so`` has not been built.
"""

from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcccl.so")

CCCL_OK = 0
CCCL_ERR_INVALID_ARG = 1
CCCL_ERR_CAPACITY = 2
CCCL_ERR_CORRUPT = 3
CCCL_ERR_TIMEOUT = 4
CCCL_ERR_CUDA = 5
CCCL_ERR_UNIMPLEMENTED = 6
CHUNK_ELEMS = 4096
CCCL_OP_SUM, CCCL_OP_MIN, CCCL_OP_MAX = 0, 1, 2
CCCL_DTYPE_BF16, CCCL_DTYPE_FP16, CCCL_DTYPE_FP32 = 1, 2, 3
MAX_RANKS = 64

if not os.path.exists(LIB_PATH):
    raise ImportError("libcccl.so is not built (run __graft_entry__.build() or "
                      "python compression_coupled_collectives_gb300/build.py)")

_lib = ctypes.CDLL(LIB_PATH)
_sz, _vp, _i = ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
_lib.cccl_compress_bound.argtypes = [_sz]
_lib.cccl_compress_bound.restype = _sz
_lib.cccl_workspace_bytes.argtypes = [_sz]
_lib.cccl_workspace_bytes.restype = _sz
_lib.cccl_compress.argtypes = [_vp, _sz, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_compress.restype = _i
_lib.cccl_compress_window.argtypes = [_vp, _sz, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_compress_window.restype = _i
_lib.cccl_compress_noalloc.argtypes = [_vp, _sz, _vp, _sz, _vp]
_lib.cccl_compress_noalloc.restype = _i
_lib.cccl_decompress.argtypes = [_vp, _sz, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_decompress.restype = _i
_lib.cccl_reduce_compressed.argtypes = [ctypes.POINTER(_vp), ctypes.POINTER(_sz), _i, _sz, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_reduce_compressed.restype = _i
_lib.cccl_compress_paged.argtypes = [_vp, _sz, _sz, _vp, _sz, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_compress_paged.restype = _i
_lib.cccl_decompress_paged.argtypes = [_vp, _sz, _vp, _sz, _sz, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_decompress_paged.restype = _i
_lib.cccl_reduce_op.argtypes = [ctypes.POINTER(_vp), ctypes.POINTER(_sz), _i, _sz, _i, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_reduce_op.restype = _i
_lib.cccl_reduce_mixed.argtypes = [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_sz), _i, _sz, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_reduce_mixed.restype = _i
_lib.cccl_compress_bound_typed.argtypes = [_i, _sz]
_lib.cccl_compress_bound_typed.restype = _sz
_lib.cccl_compress_typed.argtypes = [_i, _vp, _sz, _vp, _sz, _vp, _sz, _i, _vp]
_lib.cccl_compress_typed.restype = _i
_lib.cccl_decompress_typed.argtypes = [_i, _vp, _sz, _vp, _sz, _vp, _sz, _vp]
_lib.cccl_decompress_typed.restype = _i
_lib.cccl_reduce_typed.argtypes = [_i, _i, _vp, ctypes.POINTER(_vp), ctypes.POINTER(_sz), _i, _sz, _vp, _sz, _vp,
                                   _sz, _vp]
_lib.cccl_reduce_typed.restype = _i
_lib.cccl_get_result.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(_i)]
_lib.cccl_get_result.restype = _i
_lib.cccl_selftest_timeouts.argtypes = [_vp, _sz, _vp]
_lib.cccl_selftest_timeouts.restype = _i
_lib.cccl_selftest_lookback.argtypes = [_vp, ctypes.c_uint32, ctypes.c_uint32, _i, _vp, _vp, _sz, _vp]
_lib.cccl_selftest_lookback.restype = _i
LOOKBACK_POISON = 0xC000000000000000
_lib.cccl_status_string.argtypes = [_i]
_lib.cccl_status_string.restype = ctypes.c_char_p


class CcclError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s" % (what, cccl_status_string(status)))
        self.status = status


def cccl_status_string(status: int) -> str:
    return _lib.cccl_status_string(int(status)).decode()


def cccl_compress_bound(n_elems: int) -> int:
    return int(_lib.cccl_compress_bound(n_elems))


def cccl_workspace_bytes(n_elems: int) -> int:
    return int(_lib.cccl_workspace_bytes(n_elems))


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str) -> None:
    if status != CCCL_OK:
        raise CcclError(status, what)


def _bf16_bits(x: torch.Tensor) -> torch.Tensor:
    if x.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError("expected bf16 values (bfloat16, or their int16/uint16 bit patterns)")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x


def cccl_compress(x: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """Enqueue compression of ``x`` (n bf16 values) into ``out`` (uint8, at least
    cccl_compress_bound(n) bytes) using workspace ``ws``."""
    x = _bf16_bits(x)
    _check(_lib.cccl_compress(x.data_ptr(), x.numel(), out.data_ptr(), out.numel() * out.element_size(),
                              ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)), "cccl_compress")


def cccl_compress_window(x: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    """Enqueue the window-base variant of compression (stream version 2)."""
    x = _bf16_bits(x)
    _check(_lib.cccl_compress_window(x.data_ptr(), x.numel(), out.data_ptr(), out.numel() * out.element_size(),
                                     ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "cccl_compress_window")


def cccl_compress_noalloc(x: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Enqueue the same compression as cccl_compress using the library's static
    device scratch instead of a caller workspace (nothing is allocated).  The
    stream size is then bytes 32..39 of ``out``; no device status is reported
    (see include/cccl.h)."""
    x = _bf16_bits(x)
    _check(_lib.cccl_compress_noalloc(x.data_ptr(), x.numel(), out.data_ptr(), out.numel() * out.element_size(),
                                      _stream(stream)), "cccl_compress_noalloc")


def cccl_decompress(s: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, in_bytes: int | None = None,
                    stream=None) -> None:
    """Enqueue decompression of stream ``s`` into ``out`` (out.numel() bf16 values)."""
    out = _bf16_bits(out)
    nbytes = s.numel() * s.element_size() if in_bytes is None else int(in_bytes)
    _check(_lib.cccl_decompress(s.data_ptr(), nbytes, out.data_ptr(), out.numel(), ws.data_ptr(),
                                ws.numel() * ws.element_size(), _stream(stream)), "cccl_decompress")


def cccl_reduce_compressed(ins: Sequence[torch.Tensor], n_elems: int, out: torch.Tensor, ws: torch.Tensor,
                           in_bytes: Sequence[int] | None = None, stream=None) -> None:
    """Enqueue the fused decompress -> binary32 sum in rank order -> bf16 ->
    compress of the R streams ``ins`` into ``out``."""
    R = len(ins)
    ptrs = (_vp * max(R, 1))(*[t.data_ptr() for t in ins])
    sizes = [t.numel() * t.element_size() for t in ins] if in_bytes is None else list(in_bytes)
    szs = (_sz * max(R, 1))(*sizes)
    _check(_lib.cccl_reduce_compressed(ptrs, szs, R, n_elems, out.data_ptr(), out.numel() * out.element_size(),
                                       ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "cccl_reduce_compressed")


def cccl_compress_paged(pool: torch.Tensor, block_elems: int, table: torch.Tensor, out: torch.Tensor,
                        ws: torch.Tensor, stream=None) -> None:
    """Enqueue compression of the pool blocks named by ``table`` (int32, on the
    device), in table order; ``pool`` holds whole blocks of block_elems values."""
    pool = _bf16_bits(pool)
    if table.dtype != torch.int32 or not table.is_contiguous():
        raise TypeError("expected a contiguous int32 block table")
    _check(_lib.cccl_compress_paged(pool.data_ptr(), pool.numel() // block_elems, block_elems, table.data_ptr(),
                                    table.numel(), out.data_ptr(), out.numel() * out.element_size(), ws.data_ptr(),
                                    ws.numel() * ws.element_size(), _stream(stream)), "cccl_compress_paged")


def cccl_decompress_paged(s: torch.Tensor, pool: torch.Tensor, block_elems: int, table: torch.Tensor,
                          ws: torch.Tensor, in_bytes: int | None = None, stream=None) -> None:
    """Enqueue decompression of stream ``s`` into the pool blocks named by ``table``."""
    pool = _bf16_bits(pool)
    if table.dtype != torch.int32 or not table.is_contiguous():
        raise TypeError("expected a contiguous int32 block table")
    nbytes = s.numel() * s.element_size() if in_bytes is None else int(in_bytes)
    _check(_lib.cccl_decompress_paged(s.data_ptr(), nbytes, pool.data_ptr(), pool.numel() // block_elems,
                                      block_elems, table.data_ptr(), table.numel(), ws.data_ptr(),
                                      ws.numel() * ws.element_size(), _stream(stream)), "cccl_decompress_paged")


def cccl_reduce_op(ins: Sequence[torch.Tensor], n_elems: int, op: int, out: torch.Tensor, ws: torch.Tensor,
                   in_bytes: Sequence[int] | None = None, stream=None) -> None:
    """Enqueue the compressed reduce with operator ``op`` (CCCL_OP_SUM, _MIN or _MAX)."""
    R = len(ins)
    ptrs = (_vp * max(R, 1))(*[t.data_ptr() for t in ins])
    sizes = [t.numel() * t.element_size() for t in ins] if in_bytes is None else list(in_bytes)
    szs = (_sz * max(R, 1))(*sizes)
    _check(_lib.cccl_reduce_op(ptrs, szs, R, n_elems, op, out.data_ptr(), out.numel() * out.element_size(),
                               ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)), "cccl_reduce_op")


def cccl_reduce_mixed(local: torch.Tensor, remote: Sequence[torch.Tensor], out: torch.Tensor, ws: torch.Tensor,
                      in_bytes: Sequence[int] | None = None, stream=None) -> None:
    """Enqueue the selective-compression reduce: the uncompressed bf16 buffer
    ``local`` (rank 0) plus the compressed streams ``remote`` (ranks 1..)."""
    local = _bf16_bits(local)
    n = len(remote)
    ptrs = (_vp * max(n, 1))(*[t.data_ptr() for t in remote])
    sizes = [t.numel() * t.element_size() for t in remote] if in_bytes is None else list(in_bytes)
    szs = (_sz * max(n, 1))(*sizes)
    _check(_lib.cccl_reduce_mixed(local.data_ptr(), ptrs, szs, n, local.numel(), out.data_ptr(),
                                  out.numel() * out.element_size(), ws.data_ptr(), ws.numel() * ws.element_size(),
                                  _stream(stream)), "cccl_reduce_mixed")


# torch dtypes accepted for each element type (the values or their bit patterns)
_TYPED = {CCCL_DTYPE_BF16: (torch.bfloat16, torch.int16, torch.uint16),
          CCCL_DTYPE_FP16: (torch.float16, torch.int16, torch.uint16),
          CCCL_DTYPE_FP32: (torch.float32, torch.int32, torch.uint32)}


def _typed(dtype: int, x: torch.Tensor) -> torch.Tensor:
    if dtype not in _TYPED:
        raise ValueError("unknown element type %r" % (dtype,))
    if x.dtype not in _TYPED[dtype]:
        raise TypeError("expected values of element type %d or their bit patterns, got %s" % (dtype, x.dtype))
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x


def cccl_compress_bound_typed(dtype: int, n_elems: int) -> int:
    return int(_lib.cccl_compress_bound_typed(dtype, n_elems))


def cccl_compress_typed(dtype: int, x: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, window: bool = False,
                        stream=None) -> None:
    """Enqueue compression of ``x`` (values of element type ``dtype``)."""
    x = _typed(dtype, x)
    _check(_lib.cccl_compress_typed(dtype, x.data_ptr(), x.numel(), out.data_ptr(), out.numel() * out.element_size(),
                                    ws.data_ptr(), ws.numel() * ws.element_size(), 1 if window else 0,
                                    _stream(stream)), "cccl_compress_typed")


def cccl_decompress_typed(dtype: int, s: torch.Tensor, out: torch.Tensor, ws: torch.Tensor,
                          in_bytes: int | None = None, stream=None) -> None:
    """Enqueue decompression of stream ``s`` into ``out`` (out.numel() values of ``dtype``)."""
    out = _typed(dtype, out)
    nbytes = s.numel() * s.element_size() if in_bytes is None else int(in_bytes)
    _check(_lib.cccl_decompress_typed(dtype, s.data_ptr(), nbytes, out.data_ptr(), out.numel(), ws.data_ptr(),
                                      ws.numel() * ws.element_size(), _stream(stream)), "cccl_decompress_typed")


def cccl_reduce_typed(dtype: int, op: int, local: torch.Tensor | None, ins: Sequence[torch.Tensor], n_elems: int,
                      out: torch.Tensor, ws: torch.Tensor, in_bytes: Sequence[int] | None = None,
                      stream=None) -> None:
    """Enqueue the compressed reduce (op CCCL_OP_*) of the optional
    uncompressed ``local`` operand (rank 0) and the streams ``ins``."""
    if local is not None:
        local = _typed(dtype, local)
    n = len(ins)
    ptrs = (_vp * max(n, 1))(*[t.data_ptr() for t in ins])
    sizes = [t.numel() * t.element_size() for t in ins] if in_bytes is None else list(in_bytes)
    szs = (_sz * max(n, 1))(*sizes)
    _check(_lib.cccl_reduce_typed(dtype, op, None if local is None else local.data_ptr(), ptrs, szs, n, n_elems,
                                  out.data_ptr(), out.numel() * out.element_size(), ws.data_ptr(),
                                  ws.numel() * ws.element_size(), _stream(stream)), "cccl_reduce_typed")


def cccl_get_result(ws: torch.Tensor, stream=None) -> tuple[int, int]:
    """Synchronise ``stream``; return (stream bytes of the last compress/reduce, device status)."""
    nbytes = ctypes.c_uint64(0)
    dev = ctypes.c_int(0)
    _check(_lib.cccl_get_result(ws.data_ptr(), _stream(stream), ctypes.byref(nbytes), ctypes.byref(dev)),
           "cccl_get_result")
    return int(nbytes.value), int(dev.value)


def cccl_selftest_lookback(sizes: torch.Tensor, result: torch.Tensor, ws: torch.Tensor, poison_unit: int | None = None,
                           concurrent: bool = False, stream=None) -> None:
    """Enqueue the look-back self test over len(sizes) units (int32 device
    tensor of sizes below 2^17); `result` (int64 device tensor, one per unit)
    receives each unit's offset (4096 + the sizes before it), or
    LOOKBACK_POISON from the poisoned unit on."""
    n = sizes.numel()
    p = n if poison_unit is None else poison_unit
    _check(_lib.cccl_selftest_lookback(sizes.data_ptr(), n, p, 1 if concurrent else 0, result.data_ptr(),
                                       ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "cccl_selftest_lookback")


def cccl_selftest_timeouts(ws: torch.Tensor, stream=None) -> None:
    """Enqueue the bounded-wait self test (an mbarrier wait and a look-back
    that never complete); cccl_get_result then reports CCCL_ERR_TIMEOUT."""
    _check(_lib.cccl_selftest_timeouts(ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "cccl_selftest_timeouts")


# ---------------------------------------------------------------- conveniences
def empty_stream(n_elems: int, device=None) -> torch.Tensor:
    """A uint8 buffer large enough for any stream of n_elems values."""
    return torch.empty(cccl_compress_bound(n_elems), dtype=torch.uint8, device=device or "cuda")


def empty_workspace(n_elems: int, device=None) -> torch.Tensor:
    return torch.empty(cccl_workspace_bytes(n_elems), dtype=torch.uint8, device=device or "cuda")


def compress(x: torch.Tensor, stream=None) -> torch.Tensor:
    """Compress and wait; returns the stream trimmed to its size."""
    out = empty_stream(x.numel(), x.device)
    ws = empty_workspace(x.numel(), x.device)
    cccl_compress(x, out, ws, stream)
    nbytes, dev = cccl_get_result(ws, stream)
    _check(dev, "cccl_compress (device)")
    return out[:nbytes]


def compress_window(x: torch.Tensor, stream=None) -> torch.Tensor:
    """Window-base variant of compress; waits and returns the trimmed stream."""
    out = empty_stream(x.numel(), x.device)
    ws = empty_workspace(x.numel(), x.device)
    cccl_compress_window(x, out, ws, stream)
    nbytes, dev = cccl_get_result(ws, stream)
    _check(dev, "cccl_compress_window (device)")
    return out[:nbytes]


def decompress(s: torch.Tensor, n_elems: int, stream=None) -> torch.Tensor:
    """Decompress and wait; returns n_elems bf16 bit patterns (int16)."""
    out = torch.empty(n_elems, dtype=torch.int16, device=s.device)
    ws = empty_workspace(n_elems, s.device)
    cccl_decompress(s, out, ws, stream=stream)
    _, dev = cccl_get_result(ws, stream)
    _check(dev, "cccl_decompress (device)")
    return out


def reduce_mixed(local: torch.Tensor, remote: Sequence[torch.Tensor], stream=None) -> torch.Tensor:
    """Selective-compression reduce and wait; returns the output stream trimmed."""
    n = local.numel()
    out = empty_stream(n, local.device)
    ws = empty_workspace(n, local.device)
    cccl_reduce_mixed(local, remote, out, ws, stream=stream)
    nbytes, dev = cccl_get_result(ws, stream)
    _check(dev, "cccl_reduce_mixed (device)")
    return out[:nbytes]


def reduce_compressed(streams: Sequence[torch.Tensor], n_elems: int, stream=None) -> torch.Tensor:
    """Fused compressed reduce and wait; returns the output stream trimmed."""
    dev0 = streams[0].device
    out = empty_stream(n_elems, dev0)
    ws = empty_workspace(n_elems, dev0)
    cccl_reduce_compressed(streams, n_elems, out, ws, stream=stream)
    nbytes, dev = cccl_get_result(ws, stream)
    _check(dev, "cccl_reduce_compressed (device)")
    return out[:nbytes]


_BITS_OF = {CCCL_DTYPE_BF16: torch.int16, CCCL_DTYPE_FP16: torch.int16, CCCL_DTYPE_FP32: torch.int32}


def empty_stream_typed(dtype: int, n_elems: int, device=None) -> torch.Tensor:
    return torch.empty(cccl_compress_bound_typed(dtype, n_elems), dtype=torch.uint8, device=device or "cuda")


def compress_typed(dtype: int, x: torch.Tensor, window: bool = False, stream=None) -> torch.Tensor:
    """Compress values of element type ``dtype`` and wait; returns the trimmed stream."""
    out = empty_stream_typed(dtype, x.numel(), x.device)
    ws = empty_workspace(x.numel(), x.device)
    cccl_compress_typed(dtype, x, out, ws, window, stream)
    nbytes, dev = cccl_get_result(ws, stream)
    _check(dev, "cccl_compress_typed (device)")
    return out[:nbytes]


def decompress_typed(dtype: int, s: torch.Tensor, n_elems: int, stream=None) -> torch.Tensor:
    """Decompress and wait; returns n_elems bit patterns (int16, or int32 for fp32)."""
    out = torch.empty(n_elems, dtype=_BITS_OF[dtype], device=s.device)
    ws = empty_workspace(n_elems, s.device)
    cccl_decompress_typed(dtype, s, out, ws, stream=stream)
    _, dev = cccl_get_result(ws, stream)
    _check(dev, "cccl_decompress_typed (device)")
    return out


def reduce_typed(dtype: int, streams: Sequence[torch.Tensor], n_elems: int, op: int = CCCL_OP_SUM,
                 local: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Compressed reduce of any element type and wait; returns the trimmed stream."""
    dev0 = local.device if local is not None else streams[0].device
    out = empty_stream_typed(dtype, n_elems, dev0)
    ws = empty_workspace(n_elems, dev0)
    cccl_reduce_typed(dtype, op, local, streams, n_elems, out, ws, stream=stream)
    nbytes, dev = cccl_get_result(ws, stream)
    _check(dev, "cccl_reduce_typed (device)")
    return out[:nbytes]
