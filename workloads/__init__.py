"""Seeded synthetic inputs for the five workloads (bf16 bit patterns as uint16;
``generate_typed`` gives the same recipes as fp16 or fp32 bit patterns).

Shared by the tests, the smoke check and the benchmark.  It holds none of the
compression method's arithmetic: a counter-based SplitMix64 stream, uniforms,
Box-Muller normals (``wl_gen.c``) and the recipes below.  Rounding of the
synthetic binary32 values to bf16 is done by torch's CPU conversion (round to
nearest even), not by any code of the method.

Seed of rank r in workload w: ``1000 * w + r``.  Every recipe is counter-based,
so ``generate(w, r, start, count)`` returns exactly the slice
``generate(w, r)[start:start + count]`` without producing the rest.

Workloads (sizes in bf16 elements, 4096-element chunks):
  1. 1,048,576 values ~ N(0, 0.02); two ranks for the reduce.
  2. 33,554,432 values ~ N(0, 1e-3); each position independently, with
     probability 1/100, multiplied by 100 in binary32 before rounding
     (gradient-like buffer with escapes).
  3. 8 ranks x 134,217,728 values ~ N(0, 0.02).
  4. KV-cache tensor [32 layers, 2 (K/V), 4096 tokens, 8 heads, 128 dim]
     (268,435,456 values): N(0, 1) times a per-(layer, K/V, head) scale
     10^U(-1, 1), i.e. log-uniform in [0.1, 10] (512 scales).
  5. 268,435,456 values: first half uniformly random 16-bit patterns; second
     half N(0, 1) where each position independently is, with probability
     1/1000 each, a NaN (random sign, random nonzero payload), +-Inf, +-0 or a
     subnormal (random sign, fraction 1..127); four ranks for the reduce.
"""

from __future__ import annotations

import concurrent.futures as _cf
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wl_gen.c")
_LIB = os.path.join(_HERE, "libwl_gen.so")

SIZES = {1: 1 << 20, 2: 1 << 25, 3: 1 << 27, 4: 1 << 28, 5: 1 << 28}
RANKS = {1: 2, 2: 1, 3: 8, 4: 1, 5: 4}
KV_SHAPE = (32, 2, 4096, 8, 128)

# stream ids inside one seed
_S_VALUE, _S_AUX, _S_CAT, _S_BITS = 0, 1, 2, 3
_BLOCK = 1 << 22


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-o", tmp, _SRC,
                               "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None
_lib_lock = threading.Lock()


def _load():
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u64 = ctypes.c_uint64
        for f in ("wl_u64", "wl_uniform", "wl_normal"):
            getattr(lib, f).argtypes = [u64, u64, u64, u64, ctypes.c_void_p]
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill(fn: str, dtype, seed: int, stream: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype)
    f = getattr(_load(), fn)
    if count <= _BLOCK:
        f(seed, stream, start, count, out.ctypes.data)
        return out
    base = out.ctypes.data
    item = out.itemsize
    jobs = [(o, min(_BLOCK, count - o)) for o in range(0, count, _BLOCK)]
    with _cf.ThreadPoolExecutor(_threads()) as ex:  # ctypes releases the GIL
        list(ex.map(lambda j: f(seed, stream, start + j[0], j[1], base + j[0] * item), jobs))
    return out


def u64(seed, stream, start, count):
    return _fill("wl_u64", np.uint64, seed, stream, start, count)


def uniform(seed, stream, start, count):
    return _fill("wl_uniform", np.float64, seed, stream, start, count)


def normal(seed, stream, start, count):
    return _fill("wl_normal", np.float64, seed, stream, start, count)


def to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    """binary32 -> bf16 bit patterns via torch's CPU conversion (RNE)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def seed_of(workload: int, rank: int) -> int:
    return 1000 * workload + rank


DTYPE_BF16, DTYPE_FP16, DTYPE_FP32 = 1, 2, 3
# per element type: bit-pattern dtype, sign bit, exponent-all-ones pattern, fraction mask
_TYPE = {DTYPE_BF16: (np.uint16, 0x8000, 0x7F80, 0x7F), DTYPE_FP16: (np.uint16, 0x8000, 0x7C00, 0x3FF),
         DTYPE_FP32: (np.uint32, 0x80000000, 0x7F800000, 0x7FFFFF)}


def to_fp16_bits(f32: np.ndarray) -> np.ndarray:
    """binary32 -> IEEE fp16 bit patterns via torch's CPU conversion (RNE)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)


def _to_bits(dtype: int, f32: np.ndarray) -> np.ndarray:
    if dtype == DTYPE_BF16:
        return to_bf16_bits(f32)
    if dtype == DTYPE_FP16:
        return to_fp16_bits(f32)
    return np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)


def generate(workload: int, rank: int = 0, start: int = 0, count: int | None = None,
             n: int | None = None) -> np.ndarray:
    """bf16 bits of ``workload``'s rank ``rank``, elements [start, start+count).

    ``n`` overrides the workload's element count (same recipe, other size);
    recipes that depend on the position (workloads 4 and 5) use it.
    """
    return generate_typed(DTYPE_BF16, workload, rank, start, count, n)


def generate_typed(dtype: int, workload: int, rank: int = 0, start: int = 0, count: int | None = None,
                   n: int | None = None) -> np.ndarray:
    """Bit patterns of ``workload``'s rank ``rank`` in element type ``dtype``
    (1 bf16, 2 fp16: uint16; 3 fp32: uint32).  The same binary32 values as the
    bf16 recipe, rounded by torch to the type (fp32: kept); workload 5's
    incompressible half is random patterns of the type's width and its special
    values use the type's fields (NaN payload, subnormal fraction: 1 .. all
    fraction bits)."""
    bits_t, sign_bit, exp_ones, frac_mask = _TYPE[dtype]
    total = SIZES[workload] if n is None else n
    if count is None:
        count = total - start
    if start < 0 or count < 0 or start + count > total:
        raise ValueError("slice out of range")
    seed = seed_of(workload, rank)
    if count == 0:
        return np.empty(0, bits_t)
    if count > 2 * _BLOCK:
        # large requests: slices of one block each, on host threads (numpy and
        # torch release the GIL); every recipe is counter-based, so the slices
        # join into exactly the same bits
        out = np.empty(count, bits_t)

        def part(o):
            m = min(_BLOCK, count - o)
            out[o:o + m] = generate_typed(dtype, workload, rank, start + o, m, total)

        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(part, range(0, count, _BLOCK)))
        return out
    if workload in (1, 3):
        return _to_bits(dtype, (0.02 * normal(seed, _S_VALUE, start, count)).astype(np.float32))
    if workload == 2:
        x = (1e-3 * normal(seed, _S_VALUE, start, count)).astype(np.float32)
        hot = uniform(seed, _S_AUX, start, count) <= 0.01
        x[hot] = x[hot] * np.float32(100.0)
        return _to_bits(dtype, x)
    if workload == 4:
        idx = np.arange(start, start + count, dtype=np.int64)
        head = (idx // KV_SHAPE[4]) % KV_SHAPE[3]
        slab = idx // (KV_SHAPE[2] * KV_SHAPE[3] * KV_SHAPE[4])  # layer * 2 + kv
        scale_idx = slab * KV_SHAPE[3] + head
        slab_elems = KV_SHAPE[2] * KV_SHAPE[3] * KV_SHAPE[4]
        n_scales = -(-total // slab_elems) * KV_SHAPE[3]
        scales = 10.0 ** (-1.0 + 2.0 * uniform(seed, _S_AUX, 0, int(n_scales)))
        return _to_bits(dtype, (normal(seed, _S_VALUE, start, count) * scales[scale_idx]).astype(np.float32))
    if workload == 5:
        half = total // 2
        out = np.empty(count, bits_t)
        width_mask = np.uint64(0xFFFF if bits_t == np.uint16 else 0xFFFFFFFF)
        lo = max(start, 0)
        a_end = min(start + count, half)
        if a_end > lo:  # incompressible half
            out[:a_end - lo] = (u64(seed, _S_BITS, lo, a_end - lo) & width_mask).astype(bits_t)
        b_start = max(start, half)
        if start + count > b_start:
            m = start + count - b_start
            o = b_start - start
            vals = _to_bits(dtype, normal(seed, _S_VALUE, b_start, m).astype(np.float32))
            cat = uniform(seed, _S_CAT, b_start, m)
            bits = u64(seed, _S_AUX, b_start, m)
            sign = (((bits >> np.uint64(63)) * np.uint64(sign_bit))).astype(bits_t)
            fm = np.uint64(frac_mask)
            frac = ((bits & fm) % fm + np.uint64(1)).astype(bits_t)  # 1 .. frac_mask
            nan = cat <= 0.001
            inf = (cat > 0.001) & (cat <= 0.002)
            zero = (cat > 0.002) & (cat <= 0.003)
            sub = (cat > 0.003) & (cat <= 0.004)
            vals[nan] = sign[nan] | bits_t(exp_ones) | frac[nan]
            vals[inf] = sign[inf] | bits_t(exp_ones)
            vals[zero] = sign[zero]
            vals[sub] = sign[sub] | frac[sub]
            out[o:] = vals
        return out
    raise ValueError("unknown workload %r" % (workload,))
