"""Pins of the CPU oracle against things other than itself.

- losslessness over every one of the 65,536 bf16 bit patterns;
- a second, independent Python reading of the format (decoder, and a
  brute-force encoder that tries every code width k);
- hand-derived chunk decisions (tests/golden/chunk_choices.txt);
- closed-form sizes and offsets of every chunk;
- the binary32 sum and the bf16 rounding against numpy and torch;
- the special cases of the reduce.
"""

import os
import struct
import zlib

import numpy as np
import pytest
import torch

import pyformat as pf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "chunk_choices.txt")
CHUNK = 4096


def _rup16(v):
    return -(-v // 16) * 16


# ---------------------------------------------------------------- lossless
def test_all_bf16_patterns_round_trip_in_order(orc):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    s = orc.compress(x)
    assert np.array_equal(orc.decompress(s, x.size), x)
    assert np.array_equal(pf.decode_stream(s.tobytes(), x.size), x)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_all_bf16_patterns_round_trip_shuffled(orc, seed):
    x = np.random.default_rng(seed).permutation(65536).astype(np.uint16)
    s = orc.compress(x)
    assert np.array_equal(orc.decompress(s, x.size), x)
    assert np.array_equal(pf.decode_stream(s.tobytes(), x.size), x)


def test_sorted_patterns_use_every_mode(orc):
    """Chunks of consecutive bit patterns (one exponent pair per chunk) give
    packed chunks; their round trip pins sign and fraction bits."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    hdrs = pf.chunk_headers(orc.compress(x).tobytes())
    # 4096 consecutive patterns = 32 exponents x 128: width 5 with escapes
    assert {h[1] for h in hdrs} == {0} and {h[2] for h in hdrs} == {5}


# ---------------------------------------------------------------- independent reading
def _samples(wl):
    rng = np.random.default_rng(7)
    yield "n01", wl.generate(1, 0, count=16 * CHUNK)
    yield "n2", wl.generate(2, 0, count=16 * CHUNK)
    yield "kv", wl.generate(4, 0, count=16 * CHUNK, n=1 << 22)
    yield "worst_lo", wl.generate(5, 0, count=8 * CHUNK, n=1 << 20)
    yield "worst_hi", wl.generate(5, 0, start=1 << 19, count=8 * CHUNK, n=1 << 20)
    yield "uniform_bits", rng.integers(0, 65536, 4 * CHUNK).astype(np.uint16)
    yield "const", np.full(3 * CHUNK, 0x3F80, np.uint16)
    yield "zeros", np.zeros(2 * CHUNK + 5, np.uint16)
    few = rng.choice(np.array([0x3C00, 0x3C80, 0x3D00, 0xBC00, 0x4000], np.uint16), 5 * CHUNK + 77)
    yield "few_symbols", few


def test_oracle_matches_brute_force_stream(orc, wl):
    for name, x in _samples(wl):
        s = orc.compress(x).tobytes()
        assert s == pf.encode_stream(x), name
        assert np.array_equal(pf.decode_stream(s, x.size), x), name
        assert np.array_equal(orc.decompress(np.frombuffer(s, np.uint8), x.size), x), name


def test_brute_force_choice_on_random_exponent_mixes(orc):
    """Random chunks built from 1 to 4 exponent clusters with random counts:
    the oracle's choice equals encoding at every k and keeping the shortest."""
    rng = np.random.default_rng(11)
    for trial in range(300):
        n_sym = rng.integers(1, 5)
        exps = rng.choice(256, n_sym, replace=False)
        weights = rng.dirichlet(np.ones(n_sym) * rng.choice([0.05, 0.5, 5.0]))
        e = rng.choice(exps, CHUNK, p=weights).astype(np.uint16)
        sm = rng.integers(0, 256, CHUNK).astype(np.uint16)
        x = ((sm & 0x80) << 8) | (e << 7) | (sm & 0x7F)
        mode, k, enc = pf.brute_force_chunk(x)
        got = orc.encode_chunk(x)
        assert got == enc, (trial, mode, k)
        ch = orc.chunk_choice(x)
        assert ch["bytes"] == len(enc)
        assert ch["raw"] == (mode == "raw")
        if mode == "packed":
            assert ch["k"] == k


# ---------------------------------------------------------------- golden, hand derived
def _golden_cases():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest, "n": CHUNK}
                cases.append(cur)
            elif key == "n":
                cur["n"] = int(rest)
            elif key == "groups":
                cur["groups"] = [tuple(int(v) for v in g.split(":")) for g in rest.split()]
            elif key == "expect":
                parts = rest.split()
                cur["mode"] = parts[0]
                cur.update({kv.split("=")[0]: int(kv.split("=")[1]) for kv in parts[1:]})
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_chunk_choice(orc, case):
    rng = np.random.default_rng(zlib.crc32(case["name"].encode()))
    e = np.concatenate([np.full(c, ex, np.uint16) for ex, c in case["groups"]])
    assert e.size == case["n"]
    e = e[rng.permutation(e.size)]
    sm = rng.integers(0, 256, e.size).astype(np.uint16)
    x = ((sm & 0x80) << 8) | (e << 7) | (sm & 0x7F)
    ch = orc.chunk_choice(x)
    assert ch["raw"] == (case["mode"] == "raw")
    assert ch["bytes"] == case["bytes"]
    if case["mode"] == "packed":
        assert (ch["k"], ch["base"], ch["n_esc"]) == (case["k"], case["base"], case["n_esc"])
    enc = orc.encode_chunk(x)
    mode, k, base, _, n_c, n_esc, nbytes, _ = struct.unpack_from("<BBBBHHII", enc, 0)
    assert (mode, n_c, nbytes, len(enc)) == (1 if case["mode"] == "raw" else 0, case["n"], case["bytes"],
                                             case["bytes"])
    assert np.array_equal(pf.decode_chunk(enc, case["n"]), x)


# ---------------------------------------------------------------- closed-form sizes
@pytest.mark.parametrize("n", [1, 2, 7, 4095, 4096, 4097, 8191, 8192, 12289, 65536 + 3])
def test_closed_form_sizes_and_offsets(orc, wl, n):
    x = wl.generate(2, 0, count=n, n=max(n, 1))
    s = orc.compress(x).tobytes()
    magic, ver, dt, ce, res, n_el, nch, total = struct.unpack_from("<IHHIIQQQ", s, 0)
    assert (magic, ver, dt, ce, res, n_el) == (0x31424343, 1, 1, CHUNK, 0, n)
    assert nch == -(-n // CHUNK) and total == len(s)
    assert s[40:64] == bytes(24)
    start = 64 + _rup16(8 * nch)
    assert orc.data_start(n) == start
    assert s[64 + 8 * nch:start] == bytes(start - 64 - 8 * nch)
    pos = start
    for c, (off, mode, k, base, n_c, n_esc, nbytes) in enumerate(pf.chunk_headers(s)):
        assert off == pos and off % 16 == 0
        assert n_c == min(CHUNK, n - c * CHUNK)
        if mode == 1:
            assert (k, base, n_esc) == (0, 0, 0)
            assert nbytes == 16 + _rup16(2 * n_c)
        else:
            assert n_c == CHUNK and k <= 7
            assert nbytes == 16 + 4096 + 512 * k + _rup16(n_esc)
        pos += nbytes
    assert pos == total
    assert total <= orc.compress_bound(n)


def test_bound_is_reached_by_incompressible_input(orc):
    rng = np.random.default_rng(5)
    for n in (4096, 3 * 4096 + 11):
        x = rng.integers(0, 65536, n).astype(np.uint16)
        x[::64] = 0  # exponent 0 next to exponent 255 in every chunk
        x[1::64] = 0x7F80
        assert orc.compress(x).size == orc.compress_bound(n)


def test_padding_and_reserved_bytes_are_zero(orc, wl):
    x = wl.generate(2, 0, count=40 * CHUNK + 123, n=1 << 20)
    s = orc.compress(x).tobytes()
    for off, mode, k, base, n_c, n_esc, nbytes in pf.chunk_headers(s):
        assert s[off + 3] == 0 and s[off + 12:off + 16] == bytes(4)
        used = 2 * n_c if mode == 1 else 4096 + 512 * k + n_esc
        assert s[off + 16 + used:off + nbytes] == bytes(nbytes - 16 - used)


def test_plane_position_is_a_permutation(orc):
    seen = set()
    for i in range(CHUNK):
        w, b = orc.plane_position(i)
        assert 0 <= w < 128 and 0 <= b < 32
        seen.add(32 * w + b)
        assert (w, b) == (pf.WORD_OF[i], pf.BIT_OF[i])
    assert len(seen) == CHUNK


def test_single_escape_lands_where_defined(orc):
    """One element one exponent above the rest: k=1, its plane-0 bit and its
    escape byte are the only non-zero bytes after the sign+fraction plane."""
    for i in (0, 1, 4, 7, 8, 255, 256, 1023, 1024, 4095):
        x = np.full(CHUNK, 0x3F00, np.uint16)  # exponent 126, fraction 0
        x[i] = 0x3F80  # exponent 127
        enc = orc.encode_chunk(x)
        mode, k, base, _, n_c, n_esc, nbytes, _ = struct.unpack_from("<BBBBHHII", enc, 0)
        assert (mode, k, base, n_esc, nbytes) == (0, 1, 126, 1, 16 + 4096 + 512 + 16)
        plane = np.frombuffer(enc[16 + 4096:16 + 4096 + 512], "<u4")
        w, b = orc.plane_position(i)
        want = np.zeros(128, np.uint32)
        want[w] = 1 << b
        assert np.array_equal(plane, want)
        assert enc[16 + 4096 + 512] == 127 and enc[16 + 4096 + 513:] == bytes(15)


def test_escapes_in_bit_plane_order(orc):
    """Escapes follow the order of their elements' bits in the planes: plane
    word (q, l) = 32 q + l, then bit 8 b + m.  Hand-placed: element 9 (row 0,
    lane 1, s 1: word 1, bit 8), element 3 (lane 0, s 3: word 0, bit 24),
    element 700 (row 2, lane 23, s 4: word 23, bit 5), element 2048 (row 8:
    word 64, bit 0), element 4000 (row 15, lane 20, s 0: word 3*32+20 = 116,
    bit 2*(15 % 4) = 6)."""
    x = np.full(CHUNK, 0x3F00, np.uint16)
    placed = {9: 130, 3: 140, 700: 150, 2048: 160, 4000: 170}
    for p, e in placed.items():
        x[p] = e << 7
    enc = orc.encode_chunk(x)
    _, k, base, _, _, n_esc, _, _ = struct.unpack_from("<BBBBHHII", enc, 0)
    assert (k, base, n_esc) == (1, 126, 5)
    # by (word, bit): 3 (0, 24), 9 (1, 8), 700 (23, 5), 2048 (64, 0), 4000 (116, 6)
    assert list(enc[16 + 4096 + 512:16 + 4096 + 512 + 5]) == [140, 130, 150, 160, 170]
    for i, (w, b) in {3: (0, 24), 9: (1, 8), 700: (23, 5), 2048: (64, 0), 4000: (116, 6)}.items():
        assert orc.plane_position(i) == (w, b)
        assert orc.plane_element(w, b) == i


def test_plane_element_inverts_plane_position(orc):
    for i in range(CHUNK):
        assert orc.plane_element(*orc.plane_position(i)) == i


# ---------------------------------------------------------------- reduce arithmetic
def _f32(x):
    return (x.astype(np.uint32) << 16).view(np.float32)


def _torch_bf16(f32):
    return torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def test_round_bf16_matches_torch_on_every_upper_half(orc):
    """Every binary32 whose low 16 bits sit at the rounding boundaries (and
    random ones), for all 65,536 upper halves: equal to torch's RNE
    conversion; NaNs become 0x7FC0."""
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], np.uint32)
    u = (hi[:, None] | lows[None, :]).reshape(-1)
    f = u.view(np.float32)
    ref = _torch_bf16(f)
    nan = np.isnan(f)
    ref[nan] = 0x7FC0
    got = np.array([orc.round_bf16(v) for v in f[::7]], np.uint16)  # C call per value: sample
    assert np.array_equal(got, ref[::7])
    # the vectorised path of the oracle: R=1 sum of bf16 values is the identity
    xs = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    out = orc.sum_ranks([xs])
    want = xs.copy()
    want[np.isnan(_f32(xs))] = 0x7FC0
    assert np.array_equal(out, want)


def test_sum_of_two_matches_binary64_then_round(orc):
    """R=2: binary32 a+b equals (float)((double)a + (double)b), because
    binary64 carries more than 2*24+2 bits (double rounding is innocuous for
    a single addition); then torch rounds it to bf16."""
    rng = np.random.default_rng(3)
    a = rng.integers(0, 65536, 1 << 20).astype(np.uint16)
    b = rng.integers(0, 65536, 1 << 20).astype(np.uint16)
    with np.errstate(over="ignore", invalid="ignore"):
        exact = (_f32(a).astype(np.float64) + _f32(b).astype(np.float64)).astype(np.float32)
    want = _torch_bf16(exact)
    want[np.isnan(exact)] = 0x7FC0
    assert np.array_equal(orc.sum_ranks([a, b]), want)


def test_sum_of_many_is_sequential_binary32(orc, wl):
    R = 8
    xs = [wl.generate(3, r, count=1 << 16) for r in range(R)]
    acc = _f32(xs[0]).copy()
    for r in range(1, R):
        acc = (acc + _f32(xs[r])).astype(np.float32)  # numpy binary32 add, RNE
    assert np.array_equal(orc.sum_ranks(xs), _torch_bf16(acc))


def test_sum_rank_order_matters_and_is_kept(orc):
    """(big + -big) + small != big + (-big + small) in binary32: the result
    must be the rank-0-first order."""
    big, small = np.float32(2.0 ** 30), np.float32(1.0)
    bits = lambda f: np.array([np.float32(f)]).view(np.uint32)[0] >> 16
    a = np.array([bits(big)], np.uint16)
    b = np.array([bits(-big)], np.uint16)
    c = np.array([bits(small)], np.uint16)
    assert orc.sum_ranks([a, b, c])[0] == 0x3F80  # (2^30 - 2^30) + 1 = 1
    assert orc.sum_ranks([b, c, a])[0] == 0x0000  # (-2^30 + 1) + 2^30 = 0 in binary32


def test_reduce_special_values(orc):
    pinf, ninf, pz, nz, one = 0x7F80, 0xFF80, 0x0000, 0x8000, 0x3F80
    a = np.array([pinf, pz, nz, nz, 0x7F7F, 0x7FC1, 0x0001, one], np.uint16)
    b = np.array([ninf, nz, nz, pz, 0x7F7F, one, 0x0001, 0xFFC0], np.uint16)
    want = np.array([0x7FC0, 0x0000, 0x8000, 0x0000, 0x7F80, 0x7FC0, 0x0002, 0x7FC0], np.uint16)
    assert np.array_equal(orc.sum_ranks([a, b]), want)


def test_reduce_single_rank_is_identity_without_nan(orc, wl):
    x = wl.generate(1, 0, count=8 * CHUNK + 100)
    s = orc.compress(x)
    assert np.array_equal(orc.reduce([s], x.size), s)


def test_reduce_equals_compress_of_rounded_sum(orc, wl):
    n = 10 * CHUNK + 17
    xs = [wl.generate(5, r, count=n, start=(1 << 19) - 5 * CHUNK, n=1 << 20) for r in range(4)]
    streams = [orc.compress(x) for x in xs]
    out = orc.reduce(streams, n)
    assert np.array_equal(out, orc.compress(orc.sum_ranks(xs)))
    dec = pf.decode_stream(out.tobytes(), n)
    acc = _f32(xs[0]).copy()
    with np.errstate(over="ignore", invalid="ignore"):
        for x in xs[1:]:
            acc = (acc + _f32(x)).astype(np.float32)
    want = _torch_bf16(acc)
    want[np.isnan(acc)] = 0x7FC0
    assert np.array_equal(dec, want)


def test_reduce_mixed_is_reduce_with_the_local_operand_compressed(orc, wl):
    """Compression is lossless, so merging the local uncompressed operand with
    compressed remote ranks equals the plain reduce with the local operand
    compressed first, as rank 0."""
    for n, R in [(5 * CHUNK + 33, 3), (CHUNK, 2), (100, 4), (2 * CHUNK, 1)]:
        xs = [wl.generate(5, r, count=n, start=(1 << 19) - 2 * CHUNK, n=1 << 20) for r in range(R)]
        streams = [orc.compress(x) for x in xs]
        assert np.array_equal(orc.reduce_mixed(xs[0], streams[1:], n), orc.reduce(streams, n))


def test_reduce_mixed_matches_sequential_binary32_from_the_local_operand(orc, wl):
    n = 6 * CHUNK + 5
    xs = [wl.generate(1, r, count=n) for r in range(2)] + [wl.generate(2, 0, count=n)]
    streams = [orc.compress(x) for x in xs[1:]]
    dec = pf.decode_stream(orc.reduce_mixed(xs[0], streams, n).tobytes(), n)
    acc = _f32(xs[0]).copy()
    for x in xs[1:]:
        acc = (acc + _f32(x)).astype(np.float32)
    assert np.array_equal(dec, _torch_bf16(acc))


def test_reduce_mixed_order_and_nan(orc):
    big, one = 0x4E80, 0x3F80  # 2^30, 1
    local = np.array([big | 0x8000, 0x7FC1, 0x0000], np.uint16)  # -2^30, NaN, +0
    r1 = np.array([one, one, 0x8000], np.uint16)
    r2 = np.array([big, one, 0x8000], np.uint16)
    out = orc.decompress(orc.reduce_mixed(local, [orc.compress(r1), orc.compress(r2)], 3), 3)
    # (-2^30 + 1) + 2^30 = 0 in binary32; NaN + 1 + 1 -> 0x7FC0; +0 + -0 + -0 = +0
    assert np.array_equal(out, np.array([0x0000, 0x7FC0, 0x0000], np.uint16))
    x = np.array([0x7FC1, 0x3F80, 0xFFFF], np.uint16)
    assert np.array_equal(orc.decompress(orc.reduce_mixed(x, [], 3), 3), np.array([0x7FC0, 0x3F80, 0x7FC0], np.uint16))


def test_paged_compress_is_compress_of_the_gathered_blocks(orc, wl):
    B = 4 * CHUNK  # 16 tokens x 8 heads x 128 dim of the KV-cache shape
    pool = wl.generate(4, 0, count=9 * B)
    for table in ([0, 1, 2], [7, 2, 2, 0, 8], list(range(9))[::-1]):
        tab = np.array(table, np.int32)
        gathered = pool.reshape(-1, B)[tab].reshape(-1)
        assert np.array_equal(orc.compress_paged(pool, B, tab), orc.compress(gathered))
    with pytest.raises(orc.OracleError):
        orc.compress_paged(pool, B + 8, np.array([0], np.int32))


def test_paged_round_trip_writes_only_the_named_blocks(orc, wl):
    B = 2 * CHUNK
    pool = wl.generate(4, 1, count=10 * B)
    tab = np.array([6, 1, 9, 3], np.int32)
    s = orc.compress_paged(pool, B, tab)
    target = np.full(10 * B, 0x1234, np.uint16)
    out = orc.decompress_paged(s, target, B, tab).reshape(-1, B)
    want = target.reshape(-1, B).copy()
    want[tab] = pool.reshape(-1, B)[tab]
    assert np.array_equal(out, want)


# ---------------------------------------------------------------- min / max reduce ops
def _order_key(x):
    """bf16 bits -> unsigned key in IEEE total order (-0 below +0)."""
    x = x.astype(np.uint32)
    return np.where(x & 0x8000, (~x) & 0xFFFF, x | 0x8000)


def _minmax_numpy(xs, op):
    keys = np.stack([_order_key(x) for x in xs])
    pick = keys.argmin(0) if op == 1 else keys.argmax(0)
    out = np.stack(xs)[pick, np.arange(xs[0].size)].astype(np.uint16)
    nan = np.zeros(xs[0].size, bool)
    for x in xs:
        nan |= (x & 0x7FFF) > 0x7F80
    out[nan] = 0x7FC0
    return out


@pytest.mark.parametrize("op", [1, 2])
def test_reduce_min_max_match_an_independent_total_order(orc, wl, op):
    n = 5 * CHUNK + 3
    xs = [wl.generate(5, r, start=(1 << 27) - 2 * CHUNK, count=n) for r in range(3)]
    rng = np.random.default_rng(op)
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC1, 0x0001, 0x8001, 0x3F80, 0xBF80], np.uint16)
    xs.append(rng.choice(specials, n).astype(np.uint16))
    got = orc.decompress(orc.reduce_op([orc.compress(x) for x in xs], n, op), n)
    assert np.array_equal(got, _minmax_numpy(xs, op))


def test_reduce_min_max_single_rank_and_signed_zero(orc):
    x = np.array([0x8000, 0x0000, 0x7FC1, 0x3F80], np.uint16)
    s = [orc.compress(x)]
    for op in (1, 2):
        assert np.array_equal(orc.decompress(orc.reduce_op(s, 4, op), 4), np.array([0x8000, 0x0000, 0x7FC0, 0x3F80]))
    a, b = orc.compress(np.array([0x0000], np.uint16)), orc.compress(np.array([0x8000], np.uint16))
    assert orc.decompress(orc.reduce_op([a, b], 1, 1), 1)[0] == 0x8000  # min(+0, -0) = -0
    assert orc.decompress(orc.reduce_op([b, a], 1, 2), 1)[0] == 0x0000  # max(-0, +0) = +0


# ---------------------------------------------------------------- window-base variant (version 2)
def test_window_variant_matches_the_independent_encoder(orc, wl):
    """Every (k, base) escape count is recounted in numpy (pyformat.window_table)
    and the stream rebuilt from those choices, byte for byte."""
    samples = [wl.generate(5, 0, start=(1 << 27) - 2 * CHUNK, count=6 * CHUNK),  # uniform | specials half
               wl.generate(2, 0, count=5 * CHUNK + 77), wl.generate(4, 0, count=4 * CHUNK),
               np.random.default_rng(3).permutation(65536).astype(np.uint16)[:8 * CHUNK]]
    for x in samples:
        assert orc.compress_window(x).tobytes() == pf.encode_stream_window(x)


def test_window_variant_is_lossless_and_never_larger(orc, wl):
    allp = np.random.default_rng(11).permutation(65536).astype(np.uint16)
    assert np.array_equal(orc.decompress(orc.compress_window(allp), allp.size), allp)
    for x in (wl.generate(5, 1, start=1 << 27, count=16 * CHUNK), wl.generate(2, 1, count=16 * CHUNK)):
        v1, v2 = orc.compress(x), orc.compress_window(x)
        assert np.array_equal(orc.decompress(v2, x.size), x)
        s1, s2 = pf.chunk_headers(v1.tobytes()), pf.chunk_headers(v2.tobytes())
        assert all(b[6] <= a[6] for a, b in zip(s1, s2))  # chunk by chunk
        assert v2[4] == 2 and v1[4] == 1


def test_window_variant_hand_case(orc):
    """4090 exponents spread over 124..130 and 6 zeros: version 1 must take the
    base 0 and goes raw (every offset >= 124 escapes even at k = 7); the window
    [124, 130] at k = 3 leaves only the 6 zeros: 3 * 512 + pad16(6) = 1552."""
    e = np.concatenate([np.arange(4090) % 7 + 124, np.zeros(6, np.int64)]).astype(np.uint16)
    e = e[np.random.default_rng(5).permutation(e.size)]
    x = ((e << 7) | 0x35).astype(np.uint16)
    v1 = pf.chunk_headers(orc.compress(x).tobytes())[0]
    v2 = pf.chunk_headers(orc.compress_window(x).tobytes())[0]
    assert v1[1:3] == (1, 0)  # raw
    assert v2[1:4] == (0, 3, 124) and v2[5:7] == (6, 16 + 4096 + 1552)


def test_window_variant_base_tie_takes_the_smallest(orc):
    """Exponents 100..110, evenly: at k = 4 (15 codes) every window starting at
    96..100 holds them all (no escapes, 2048 bytes, the best size), and the
    smallest start wins."""
    e = (np.arange(CHUNK) % 11 + 100).astype(np.uint16)
    h = pf.chunk_headers(orc.compress_window((e << 7) | 0x11).tobytes())[0]
    assert h[1:4] == (0, 4, 96) and h[5] == 0


# ---------------------------------------------------------------- corrupt streams
def _corrupt_cases(orc, wl):
    x = wl.generate(2, 0, count=3 * CHUNK + 10, n=1 << 20)
    s = bytearray(orc.compress(x).tobytes())
    hdrs = pf.chunk_headers(bytes(s))
    packed = next(h for h in hdrs if h[1] == 0)
    o = packed[0]

    def mut(fn):
        t = bytearray(s)
        fn(t)
        return bytes(t)

    yield "magic", mut(lambda t: t.__setitem__(0, 0))
    yield "version", mut(lambda t: t.__setitem__(4, 3))
    yield "n_elems", mut(lambda t: struct.pack_into("<Q", t, 16, x.size + 1))
    yield "total_bytes", mut(lambda t: struct.pack_into("<Q", t, 32, len(s) + 16))
    yield "offset_misaligned", mut(lambda t: struct.pack_into("<Q", t, 64 + 8, hdrs[1][0] + 8))
    yield "k_too_big", mut(lambda t: t.__setitem__(o + 1, 8))
    yield "mode_bad", mut(lambda t: t.__setitem__(o, 2))
    yield "n_esc_wrong", mut(lambda t: struct.pack_into("<H", t, o + 6, packed[5] + 16))
    yield "chunk_bytes_wrong", mut(lambda t: struct.pack_into("<I", t, o + 8, packed[6] + 16))
    yield "tail_n_c", mut(lambda t: struct.pack_into("<H", t, hdrs[-1][0] + 4, 11))
    yield "truncated", bytes(s[:-16])


def test_oracle_rejects_corrupt_streams(orc, wl):
    for name, bad in _corrupt_cases(orc, wl):
        assert orc.decompress_status(np.frombuffer(bad, np.uint8), 3 * CHUNK + 10) == orc.ERR_CORRUPT, name


def test_oracle_rejects_packed_chunk_not_smaller_than_raw(orc):
    """k=7 with 512 escapes is 4096 bytes of exponents: an encoder stores that
    chunk raw, so a packed one is malformed even though it could be decoded."""
    rng = np.random.default_rng(8)
    e = np.full(CHUNK, 10, np.uint16)
    e[rng.choice(CHUNK, 600, replace=False)] = 200
    x = (e << 7).astype(np.uint16)
    enc = pf.encode_chunk_at(x, 7)
    assert len(enc) == 16 + 4096 + 3584 + 608
    body = enc.ljust(len(enc), b"\0")
    start = 64 + 16
    total = start + len(body)
    hdr = struct.pack("<IHHIIQQQ", 0x31424343, 1, 1, CHUNK, 0, CHUNK, 1, total).ljust(64, b"\0")
    table = struct.pack("<Q", start).ljust(16, b"\0")
    s = hdr + table + body
    assert np.array_equal(pf.decode_stream(s, CHUNK), x)  # decodable in principle
    assert orc.decompress_status(np.frombuffer(s, np.uint8), CHUNK) == orc.ERR_CORRUPT


def test_oracle_rejects_exponent_overflow(orc):
    """base + code above 255 cannot come from an encoder: reported corrupt."""
    x = np.full(CHUNK, 250 << 7, np.uint16)
    x[:2096] = 251 << 7  # k=2 (1024) beats k=1 (512 + 2096): offsets 0 and 1 are plain codes
    s = bytearray(orc.compress(x).tobytes())
    o = pf.chunk_headers(bytes(s))[0][0]
    assert s[o + 1] == 2
    s[o + 2] = 255  # base 255: code 1 -> exponent 256
    assert orc.decompress_status(np.frombuffer(bytes(s), np.uint8), CHUNK) == orc.ERR_CORRUPT
