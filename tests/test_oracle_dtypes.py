"""Pins of the oracle's fp16 and fp32 element types (the bf16 split of
section 4.1 with a 5-bit and an 8-bit exponent) against things other than
itself:

- losslessness over every fp16 bit pattern and over random fp32 patterns;
- the independent Python reading of the typed format (tests/pyformat.py),
  whose encoder tries every code width;
- hand-derived chunk decisions, one of them between fp16's raw threshold
  (2560 bytes) and bf16's (4096);
- the binary16 conversions against numpy's IEEE conversions;
- the binary32 sums, rounded once, against numpy; min and max against an
  independent total-order key;
- corrupt streams.
"""

import struct

import numpy as np
import pytest

import pyformat as pf

CHUNK = 4096
BF16, FP16, FP32 = 1, 2, 3


def _rup16(v):
    return -(-v // 16) * 16


def _fp16_chunk(exponents, rng):
    e = np.asarray(exponents, np.uint16)
    rest = rng.integers(0, 1 << 16, e.size).astype(np.uint16) & np.uint16(0x83FF)
    return rest | (e << 10)


def _fp32_chunk(exponents, rng):
    e = np.asarray(exponents, np.uint32)
    rest = rng.integers(0, 1 << 32, e.size, dtype=np.uint64).astype(np.uint32) & np.uint32(0x807FFFFF)
    return rest | (e << 23)


# ---------------------------------------------------------------- binary16 conversions
def _float32_probes():
    rng = np.random.default_rng(11)
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = h.view(np.float16).astype(np.float32)
    finite = vals[np.isfinite(vals)]
    with np.errstate(over="ignore"):
        nxt = np.nextafter(finite.astype(np.float16), np.float16(np.inf)).astype(np.float32)
    ok = np.isfinite(nxt)
    mid = ((finite[ok].astype(np.float64) + nxt[ok].astype(np.float64)) / 2).astype(np.float32)  # exact ties
    around = np.concatenate([mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(-np.inf))])
    rand = rng.integers(0, 1 << 32, 1 << 18, dtype=np.uint64).astype(np.uint32).view(np.float32)
    edges = np.array([65504, 65505, 65519.99, 65520, 65536, 1e9, 2.0 ** -24, 2.0 ** -25, 2.0 ** -26,
                      3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, np.inf], np.float32)
    out = np.concatenate([finite, around, rand, edges, -edges])
    return out[~np.isnan(out)]


def test_round_fp16_matches_numpy_on_ties_subnormals_and_overflow(orc):
    f = _float32_probes()
    with np.errstate(over="ignore"):
        want = f.astype(np.float16).view(np.uint16)
    lib = orc._load()
    got = np.array([lib.oracle_round_fp16(float(v)) for v in f], np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(f[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_round_fp16_nan_is_canonical(orc):
    for bits in (0x7FC00000, 0xFFC00001, 0x7F800001, 0xFFFFFFFF):
        f = np.array([bits], np.uint32).view(np.float32)[0]
        assert orc.round_fp16(float(f)) == 0x7E00


def test_fp16_to_float_matches_numpy_on_every_pattern(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = h.view(np.float16).astype(np.float32)
    lib = orc._load()
    got = np.array([lib.oracle_fp16_to_float(int(v)) for v in h], np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


# ---------------------------------------------------------------- lossless, independent reading
@pytest.mark.parametrize("seed", [1, 2])
def test_all_fp16_patterns_round_trip(orc, seed):
    x = np.random.default_rng(seed).permutation(65536).astype(np.uint16)
    s = orc.compress_typed(FP16, x)
    assert np.array_equal(orc.decompress_typed(FP16, s, x.size), x)
    assert np.array_equal(pf.decode_stream_typed(FP16, s.tobytes(), x.size), x)
    assert s.tobytes() == pf.encode_stream_typed(FP16, x)


def test_random_fp32_patterns_round_trip(orc):
    rng = np.random.default_rng(3)
    x = rng.integers(0, 1 << 32, 5 * CHUNK + 333, dtype=np.uint64).astype(np.uint32)
    x[:CHUNK] = (x[:CHUNK] & np.uint32(0x807FFFFF)) | (np.uint32(120 + (np.arange(CHUNK) % 5)) << 23)
    s = orc.compress_typed(FP32, x)
    assert np.array_equal(orc.decompress_typed(FP32, s, x.size), x)
    assert s.tobytes() == pf.encode_stream_typed(FP32, x)
    assert pf.chunk_headers(s.tobytes())[0][1] == 0  # the narrow chunk is packed


def _typed_samples(wl, dtype):
    yield "n01", wl.generate_typed(dtype, 1, 0, count=6 * CHUNK)
    yield "grad", wl.generate_typed(dtype, 2, 0, count=6 * CHUNK + 1000)
    yield "kv", wl.generate_typed(dtype, 4, 0, count=6 * CHUNK, n=1 << 22)
    yield "mixed", wl.generate_typed(dtype, 5, 0, start=(1 << 27) - 3 * CHUNK, count=6 * CHUNK)


@pytest.mark.parametrize("dtype", [FP16, FP32])
@pytest.mark.parametrize("window", [False, True])
def test_oracle_matches_the_independent_encoder(orc, wl, dtype, window):
    for name, x in _typed_samples(wl, dtype):
        s = orc.compress_typed(dtype, x, window=window)
        assert s.tobytes() == pf.encode_stream_typed(dtype, x, window=window), name
        assert np.array_equal(orc.decompress_typed(dtype, s, x.size), x), name


def test_bf16_typed_is_the_bf16_stream(orc, wl):
    x = wl.generate(2, 0, count=4 * CHUNK + 5)
    assert np.array_equal(orc.compress_typed(BF16, x), orc.compress(x))
    assert np.array_equal(orc.compress_typed(BF16, x, window=True), orc.compress_window(x))


# ---------------------------------------------------------------- hand-derived decisions
def test_fp16_hand_case_narrow_chunk(orc):
    """Exponents 10 (4000 times) and 11 (96): k = 1 costs 512 + 96 = 608 bytes,
    k = 2 costs 1024; packed size 16 + 4096 + 3 * 512 + 512 + 96 = 6256."""
    rng = np.random.default_rng(5)
    e = np.array([10] * 4000 + [11] * 96)[rng.permutation(CHUNK)]
    ch = orc.chunk_choice_typed(FP16, _fp16_chunk(e, rng))
    assert ch == dict(raw=0, k=1, base=10, n_esc=96, bytes=6256)


def test_fp16_hand_case_between_the_two_raw_thresholds(orc):
    """Exponents 0..15 (200 each) and 16..19 (224 each).  k = 4 leaves the
    1096 exponents >= 15 as escapes: 2048 + pad16(1096) = 3152 bytes, the
    best width, which does not beat fp16's 5-bit exponents (2560 bytes):
    raw, although it is below bf16's 4096."""
    rng = np.random.default_rng(6)
    e = np.array(sum(([v] * 200 for v in range(16)), []) + sum(([v] * 224 for v in range(16, 20)), []))
    assert e.size == CHUNK
    x = _fp16_chunk(e[rng.permutation(CHUNK)], rng)
    ch = orc.chunk_choice_typed(FP16, x)
    assert ch == dict(raw=1, k=0, base=0, n_esc=0, bytes=16 + 2 * CHUNK)


def test_fp16_hand_case_widest_code(orc):
    """Exponents 0..14, 273 times each, and one 15 (4096 = 15 * 273 + 1):
    k = 4 (sentinel 15) escapes only the 15, 2048 + 16 = 2064 bytes; k = 3
    escapes the 2185 exponents >= 7, 1536 + 2192 = 3728 bytes."""
    rng = np.random.default_rng(7)
    e = np.array(sum(([v] * 273 for v in range(15)), []) + [15])[rng.permutation(CHUNK)]
    ch = orc.chunk_choice_typed(FP16, _fp16_chunk(e, rng))
    assert ch == dict(raw=0, k=4, base=0, n_esc=1, bytes=16 + 5632 + 2048 + 16)


def test_fp32_hand_case(orc):
    """Exponents 120 (4000) and 121 (96), as the bf16 hand case: k = 1 with 96
    escapes; size 16 + 4096 + 8192 + 512 + 96 = 12912."""
    rng = np.random.default_rng(8)
    e = np.array([120] * 4000 + [121] * 96)[rng.permutation(CHUNK)]
    ch = orc.chunk_choice_typed(FP32, _fp32_chunk(e, rng))
    assert ch == dict(raw=0, k=1, base=120, n_esc=96, bytes=12912)


def test_fp16_body_layout_by_hand(orc):
    """One chunk of a single exponent (k = 0): the body is the low bytes, then
    the planes of fraction bit 8, fraction bit 9 and the sign."""
    i = np.arange(CHUNK)
    x = ((i & 0xFF) | (((i >> 1) & 1) << 8) | (((i >> 2) & 1) << 9) | (((i >> 3) & 1) << 15) | (7 << 10))
    x = x.astype(np.uint16)
    c = orc.encode_chunk_typed(FP16, x)
    assert struct.unpack_from("<BBBBHHII", c, 0) == (0, 0, 7, 0, CHUNK, 0, 16 + 4096 + 1536, 0)
    assert c[16:16 + 4096] == bytes((i & 0xFF).astype(np.uint8))
    words = np.frombuffer(c[16 + 4096:], "<u4").reshape(3, 128)
    for t, shift in enumerate((1, 2, 3)):
        for el in (0, 2, 5, 4095, 1234):
            w, b = orc.plane_position(el)
            assert (words[t, w] >> b) & 1 == (el >> shift) & 1


def test_fp32_body_layout_by_hand(orc):
    """k = 0 fp32 chunk: the byte plane is sign and fraction bits 16..22, the
    lower halves follow verbatim."""
    i = np.arange(CHUNK, dtype=np.uint32)
    x = (np.uint32(100) << 23) | (i * np.uint32(2654435761) & np.uint32(0x807FFFFF))
    c = orc.encode_chunk_typed(FP32, x)
    assert struct.unpack_from("<BBBBHHII", c, 0)[:3] == (0, 0, 100)
    hi = x >> 16
    assert c[16:16 + 4096] == bytes((((hi >> 8) & 0x80) | (hi & 0x7F)).astype(np.uint8))
    assert c[16 + 4096:16 + 4096 + 8192] == (x & 0xFFFF).astype("<u2").tobytes()


# ---------------------------------------------------------------- reduce
def _np_sum(dtype, xs):
    with np.errstate(over="ignore", invalid="ignore"):
        if dtype == FP16:
            acc = xs[0].view(np.float16).astype(np.float32)
            for x in xs[1:]:
                acc = acc + x.view(np.float16).astype(np.float32)
            out = acc.astype(np.float16).view(np.uint16).copy()
            out[np.isnan(acc)] = 0x7E00
            return out
        acc = xs[0].view(np.float32).copy()
        for x in xs[1:]:
            acc = acc + x.view(np.float32)
        out = acc.view(np.uint32).copy()
        out[np.isnan(acc)] = 0x7FC00000
        return out


@pytest.mark.parametrize("dtype", [FP16, FP32])
def test_sum_ranks_matches_numpy(orc, wl, dtype):
    rng = np.random.default_rng(9)
    width = 16 if dtype == FP16 else 32
    rand = [rng.integers(0, 1 << width, 1 << 15, dtype=np.uint64).astype(np.uint16 if width == 16 else np.uint32)
            for _ in range(3)]
    assert np.array_equal(orc.sum_ranks_typed(dtype, rand), _np_sum(dtype, rand))
    ws = [wl.generate_typed(dtype, 5, r, start=(1 << 27) - CHUNK, count=3 * CHUNK) for r in range(4)]
    assert np.array_equal(orc.sum_ranks_typed(dtype, ws), _np_sum(dtype, ws))


def test_fp16_sum_rounds_once_after_binary32(orc):
    """1 + 2^-11 + 2^-11: binary32 keeps 1 + 2^-10 (fp16 0x3C01); rounding
    after every add would give 1 twice (ties to even)."""
    one, tiny = np.array([0x3C00], np.uint16), np.array([0x1000], np.uint16)  # 2^-11
    assert orc.sum_ranks_typed(FP16, [one, tiny, tiny])[0] == 0x3C01
    # overflow of a finite sum to Inf, and Inf - Inf to the canonical NaN
    big = np.array([0x7BFF], np.uint16)  # 65504
    assert orc.sum_ranks_typed(FP16, [big, big])[0] == 0x7C00
    assert orc.sum_ranks_typed(FP16, [np.array([0x7C00], np.uint16), np.array([0xFC00], np.uint16)])[0] == 0x7E00


def test_fp32_sum_keeps_subnormals_and_order(orc):
    sub = np.array([1], np.uint32)  # 2^-149
    assert orc.sum_ranks_typed(FP32, [sub, sub])[0] == 2
    a, b, c = (np.array([v], np.float32).view(np.uint32) for v in (2.0 ** 30, -(2.0 ** 30), 1.0))
    assert orc.sum_ranks_typed(FP32, [a, b, c])[0] == 0x3F800000
    assert orc.sum_ranks_typed(FP32, [a, c, b])[0] == 0  # 2^30 + 1 rounds back to 2^30


def _order_key(dtype, x):
    width = 16 if dtype == FP16 else 32
    x = x.astype(np.uint64)
    sign = np.uint64(1 << (width - 1))
    full = np.uint64((1 << width) - 1)
    return np.where(x & sign, ~x & full, x | sign)


@pytest.mark.parametrize("dtype", [FP16, FP32])
@pytest.mark.parametrize("op", [1, 2])
def test_min_max_match_an_independent_total_order(orc, wl, dtype, op):
    xs = [wl.generate_typed(dtype, 5, r, start=(1 << 27) - CHUNK, count=3 * CHUNK) for r in range(3)]
    n = xs[0].size
    out = orc.decompress_typed(dtype, orc.reduce_typed(dtype, [orc.compress_typed(dtype, x) for x in xs], n, op), n)
    keys = np.stack([_order_key(dtype, x) for x in xs])
    pick = np.argmin(keys, 0) if op == 1 else np.argmax(keys, 0)
    want = np.stack(xs)[pick, np.arange(n)]
    if dtype == FP16:
        nan = np.any(np.stack([(x & 0x7FFF) > 0x7C00 for x in xs]), 0)
        want[nan] = 0x7E00
    else:
        nan = np.any(np.stack([(x & 0x7FFFFFFF) > 0x7F800000 for x in xs]), 0)
        want[nan] = 0x7FC00000
    assert nan.any() and np.array_equal(out, want)


@pytest.mark.parametrize("dtype", [FP16, FP32])
def test_reduce_is_compress_of_the_reduced_values(orc, wl, dtype):
    xs = [wl.generate_typed(dtype, 2, r, count=5 * CHUNK + 17) for r in range(3)]
    n = xs[0].size
    streams = [orc.compress_typed(dtype, x) for x in xs]
    assert np.array_equal(orc.reduce_typed(dtype, streams, n), orc.compress_typed(dtype, _np_sum(dtype, xs)))
    # the local operand as rank 0 is the same as its stream
    assert np.array_equal(orc.reduce_typed(dtype, streams[1:], n, local=xs[0]), orc.reduce_typed(dtype, streams, n))


# ---------------------------------------------------------------- corrupt streams
def _packed_fp16_chunk_stream(orc, rng):
    e = np.array([3] * 4000 + [4] * 96)[rng.permutation(CHUNK)]
    x = _fp16_chunk(e, rng)
    return x, bytearray(orc.compress_typed(FP16, x).tobytes())


def test_typed_decoder_rejects_other_dtypes(orc, wl):
    x = wl.generate_typed(FP16, 1, 0, count=CHUNK)
    s = orc.compress_typed(FP16, x)
    assert orc.decompress_typed_status(BF16, s, x.size) == orc.ERR_CORRUPT
    assert orc.decompress_typed_status(FP32, s, x.size) == orc.ERR_CORRUPT
    assert orc.decompress_status(s, x.size) == orc.ERR_CORRUPT


def test_fp16_exponent_out_of_range_is_corrupt(orc):
    rng = np.random.default_rng(12)
    x, s = _packed_fp16_chunk_stream(orc, rng)
    off = pf.chunk_headers(bytes(s))[0][0]
    assert s[off + 1] == 1 and s[off + 2] == 3
    s2 = bytearray(s)
    s2[off + 2] = 31  # base 31: the only non-sentinel code (0) gives 31, still a 5-bit exponent
    assert orc.decompress_typed_status(FP16, s2, CHUNK) == orc.OK
    s3 = bytearray(s)
    s3[off + 2] = 32  # a base no 5-bit exponent can have
    assert orc.decompress_typed_status(FP16, s3, CHUNK) == orc.ERR_CORRUPT
    s4 = bytearray(s)
    esc_at = off + 16 + 5632 + 512
    s4[esc_at] = 32  # an escaped exponent above 31
    assert orc.decompress_typed_status(FP16, s4, CHUNK) == orc.ERR_CORRUPT


def test_fp16_width_five_is_corrupt(orc):
    rng = np.random.default_rng(13)
    x, s = _packed_fp16_chunk_stream(orc, rng)
    off = pf.chunk_headers(bytes(s))[0][0]
    s[off + 1] = 5
    assert orc.decompress_typed_status(FP16, s, CHUNK) == orc.ERR_CORRUPT
