"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch each one.  The mistakes are planted in C source copied to a temporary
directory and built there; the committed oracle is never modified.
"""

import os
import zlib

import numpy as np
import pytest
import torch

import pyformat as pf

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "cccl_oracle.c")
CHUNK = 4096

MUTATIONS = [
    ("tie_keeps_larger_k", "if (!have || size < best_size) { /* strict: ties keep the smaller k */",
     "if (!have || size <= best_size) { /* strict: ties keep the smaller k */"),
    ("raw_tie_goes_packed", "if (best_size >= raw_exponent_bytes(dt)) /* no gain over the verbatim exponents: raw (ties too) */",
     "if (best_size > raw_exponent_bytes(dt)) /* no gain over the verbatim exponents: raw (ties too) */"),
    ("sign_bit_dropped", "return ((b >> 8) & 0x80u) | (b & 0x7Fu);", "return (b & 0x7Fu);"),
    ("plane_bit_order_swapped", "*bit = 8 * (s % 4) + 2 * (j % 4) + s / 4;", "*bit = 8 * (s % 4) + 2 * (s / 4) + j % 4;"),
    ("plane_word_order_swapped", "*word = (j / 4) * 32 + l;", "*word = l * 4 + j / 4;"),
    ("escape_padding_dropped", "dt->resid_bytes + (size_t)BIT_PLANE_BYTES * k + pad16(n_esc);",
     "dt->resid_bytes + (size_t)BIT_PLANE_BYTES * k + n_esc;"),
    ("escape_padding_ignored_in_choice", "size_t size = (size_t)BIT_PLANE_BYTES * k + pad16(n_esc);",
     "size_t size = (size_t)BIT_PLANE_BYTES * k + n_esc;"),
    ("escape_threshold_off_by_one", "if (e - ch.base >= sentinel)", "if (e - ch.base > sentinel)"),
    ("escapes_in_element_order", "unsigned e = exponent_of(dt, elem(dt, x, element_at[pos]));",
     "unsigned e = exponent_of(dt, elem(dt, x, pos));"),
    ("count_threshold_off_by_one", "count_at_or_above(dt, x, n_c, emin, sentinel);",
     "count_at_or_above(dt, x, n_c, emin, sentinel + 1);"),
    ("rounding_half_up", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    ("nan_not_canonical", "if ((u & 0x7FFFFFFFu) > 0x7F800000u)\n        return 0x7FC0;", ""),
    ("accumulate_from_zero", "float acc = to_binary32(dt, elem(dt, xs[0], i));\n        for (int r = 1; r < R; r++)",
     "float acc = 0.0f;\n        for (int r = 0; r < R; r++)"),
    ("rank_order_reversed", "acc = acc + to_binary32(dt, elem(dt, xs[r], i));",
     "acc = acc + to_binary32(dt, elem(dt, xs[R - r], i));"),
    ("tail_chunk_packed", "if (n_c != CHUNK_ELEMS) /* a partial chunk travels raw (section 5) */",
     "if (n_c == 0)"),
    ("minimum_not_tracked", "        if (e < emin)\n            emin = e;\n        if (e > emax)\n            emax = e;\n    }\n\n    /* size",
     "        if (e > emin)\n            emin = e;\n        if (e > emax)\n            emax = e;\n    }\n\n    /* size"),
    ("offset_table_relative", "put_u64(out + STREAM_HEADER_BYTES + 8 * c, pos);",
     "put_u64(out + STREAM_HEADER_BYTES + 8 * c, pos - start);"),
    ("remote_ranks_reversed", "st = decompress_stream(dt, ins[r - first], in_bytes[r - first], x, n);",
     "st = decompress_stream(dt, ins[R - 1 - r], in_bytes[R - 1 - r], x, n);"),
    ("window_tie_keeps_larger_base", "if (b == 0 || n_esc < k_esc) {", "if (b == 0 || n_esc <= k_esc) {"),
    ("window_one_too_narrow", "unsigned top = b + S < n_sym ? b + S : n_sym;",
     "unsigned top = b + S - 1 < n_sym ? b + S - 1 : n_sym;"),
    ("min_signed_zero_order", "        return na; /* negative (including -0) below positive (including +0) */",
     "        return nb; /* negative (including -0) below positive (including +0) */"),
    ("minmax_nan_dropped", "            if (is_nan_elem(dt, acc) || is_nan_elem(dt, b))\n                acc = dt->nan;\n            else if",
     "            if (0)\n                acc = dt->nan;\n            else if"),
    ("paged_gather_ignores_table", "memcpy(x + i * block_elems, pool + (size_t)table[i] * block_elems,",
     "memcpy(x + i * block_elems, pool + i * block_elems,"),
    ("paged_scatter_ignores_table", "memcpy(pool + (size_t)table[i] * block_elems, x + i * block_elems,",
     "memcpy(pool + i * block_elems, x + i * block_elems,"),
    ("mixed_local_added_last", "            sum_ranks(dt, xs, R, n, res);",
     "{ const void *t = xs[0]; for (int q = 0; q + 1 < R; q++) xs[q] = xs[q + 1]; xs[R - 1] = t; "
     "sum_ranks(dt, xs, R, n, res); for (int q = R - 1; q > 0; q--) xs[q] = xs[q - 1]; xs[0] = t; }"),
    # element types
    ("fp16_plane_bits_swapped", "FP16_PLANE_BITS[3] = {8, 9, 15};", "FP16_PLANE_BITS[3] = {9, 8, 15};"),
    ("fp16_sign_not_stored", "FP16_PLANE_BITS[3] = {8, 9, 15};", "FP16_PLANE_BITS[3] = {8, 9, 14};"),
    ("fp32_low_half_dropped", "put_u16(body + SM_PLANE_BYTES + 2 * i, elem(dt, x, i) & 0xFFFFu);",
     "put_u16(body + SM_PLANE_BYTES + 2 * i, 0);"),
    ("raw_threshold_of_bf16", "return (size_t)BIT_PLANE_BYTES * dt->exp_bits;", "return SM_PLANE_BYTES;"),
    ("fp16_round_ties_away", "if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0))", "if (frac >= 0.5)"),
    ("fp16_overflow_at_max", "if (a >= 65520.0) /* halfway", "if (a > 65504.0) /* halfway"),
    ("fp16_subnormal_quantum", "E = -14; /* subnormal range: quantum 2^-24 */", "E = -15; /* subnormal range: quantum 2^-24 */"),
    ("fp16_to_float_bias", "mag = ldexpf((float)(1024u + m), (int)e - 25);", "mag = ldexpf((float)(1024u + m), (int)e - 24);"),
    ("fp32_sum_rounded_to_bf16", "        memcpy(&u, &f, sizeof u);\n        return u;",
     "        return (uint32_t)oracle_round_bf16(f) << 16;"),
    ("sign_bit_of_two_bytes", "return 1u << (8 * dt->elem_bytes - 1);", "return 0x8000u;"),
    ("fp16_exponent_range_unchecked", "        if (e >= n_symbols(dt))\n            return ORC_ERR_CORRUPT;", ""),
]


def _f32(x):
    return (x.astype(np.uint32) << 16).view(np.float32)


def _torch_bf16(f32):
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16)
    out = t.view(torch.int16).numpy().view(np.uint16).copy()
    out[np.isnan(f32)] = 0x7FC0
    return out


def _golden_like_chunks():
    rng = np.random.default_rng(99)
    groups = [
        [(120, 4000), (121, 96)], [(100, 3599), (101, 497)], [(100, 3583), (101, 513)],
        [(0, 512), (1, 512), (3, 512), (7, 512), (15, 512), (31, 512), (63, 512), (200, 512)],
        [(0, 528), (1, 512), (3, 512), (7, 512), (15, 512), (31, 512), (63, 512), (200, 496)],
        [(e, 292) for e in range(50, 64)] + [(64, 7), (65, 1)],
        [(0, 513), (1, 512), (3, 512), (7, 512), (15, 512), (31, 512), (63, 512), (200, 511)],
    ]
    for g in groups:
        e = np.concatenate([np.full(c, v, np.uint16) for v, c in g])
        e = e[rng.permutation(e.size)]
        sm = rng.integers(0, 256, e.size).astype(np.uint16)
        yield ((sm & 0x80) << 8) | (e << 7) | (sm & 0x7F)


def _battery(orc, wl):
    """Run the pins; return the names of the ones that fail."""
    failed = []

    def check(name, fn):
        try:
            if not fn():
                failed.append(name)
        except Exception:  # a crash in the mutant counts as caught
            failed.append(name)

    allp = np.random.default_rng(1).permutation(65536).astype(np.uint16)
    check("lossless_all_patterns", lambda: np.array_equal(orc.decompress(orc.compress(allp), allp.size), allp))
    check("python_decoder", lambda: np.array_equal(pf.decode_stream(orc.compress(allp).tobytes(), allp.size), allp))
    samples = [wl.generate(1, 0, count=8 * CHUNK), wl.generate(2, 0, count=8 * CHUNK + 99)]
    samples += list(_golden_like_chunks())
    check("brute_force_streams", lambda: all(orc.compress(x).tobytes() == pf.encode_stream(x) for x in samples))
    rng = np.random.default_rng(4)
    a = rng.integers(0, 65536, 1 << 16).astype(np.uint16)
    b = rng.integers(0, 65536, 1 << 16).astype(np.uint16)
    with np.errstate(over="ignore", invalid="ignore"):
        exact = (_f32(a).astype(np.float64) + _f32(b).astype(np.float64)).astype(np.float32)
    check("sum_two_vs_binary64", lambda: np.array_equal(orc.sum_ranks([a, b]), _torch_bf16(exact)))
    sp_a = np.array([0x7F80, 0x8000, 0x7FC1, 0x4E80], np.uint16)
    sp_b = np.array([0xFF80, 0x8000, 0x3F80, 0xCE80], np.uint16)
    sp_c = np.array([0x0000, 0x8000, 0x0000, 0x3F80], np.uint16)
    check("special_values", lambda: np.array_equal(orc.sum_ranks([sp_a, sp_b, sp_c]),
                                                   np.array([0x7FC0, 0x8000, 0x7FC0, 0x3F80], np.uint16)))
    check("rank_order", lambda: orc.sum_ranks([sp_b[3:], sp_c[3:], sp_a[3:]])[0] == 0)
    # local 2^30, remote -2^30 then 1: (2^30 - 2^30) + 1 = 1 only in this order
    check("mixed_rank_order", lambda: orc.decompress(
        orc.reduce_mixed(sp_a[3:], [orc.compress(sp_b[3:]), orc.compress(sp_c[3:])], 1), 1)[0] == 0x3F80)
    mm = [np.array([0x0000, 0x3F80, 0x7FC1, 0x8000], np.uint16), np.array([0x8000, 0xBF80, 0x3F80, 0x0000], np.uint16)]
    check("min_max", lambda: (lambda s: orc.decompress(orc.reduce_op(s, 4, 1), 4).tolist() ==
                              [0x8000, 0xBF80, 0x7FC0, 0x8000] and
                              orc.decompress(orc.reduce_op(s, 4, 2), 4).tolist() ==
                              [0x0000, 0x3F80, 0x7FC0, 0x0000])([orc.compress(v) for v in mm]))
    wx = wl.generate(5, 0, start=(1 << 27) - 2 * CHUNK, count=4 * CHUNK)
    check("window_variant", lambda: orc.compress_window(wx).tobytes() == pf.encode_stream_window(wx))
    te = (np.arange(CHUNK) % 11 + 100).astype(np.uint16)  # exponents 100..110: k = 4 from any base 96..100
    check("window_base_tie", lambda: pf.chunk_headers(orc.compress_window((te << 7) | 0x11).tobytes())[0][3] == 96)
    pool = np.arange(6 * CHUNK, dtype=np.uint16) * 7 + 1
    tab = np.array([4, 1, 3], np.int32)
    check("paged_gather", lambda: np.array_equal(orc.compress_paged(pool, CHUNK, tab),
                                                 orc.compress(pool.reshape(-1, CHUNK)[tab].reshape(-1))))
    check("paged_scatter", lambda: np.array_equal(
        orc.decompress_paged(orc.compress(pool[:3 * CHUNK]), np.zeros_like(pool), CHUNK, tab).reshape(-1, CHUNK)[tab],
        pool[:3 * CHUNK].reshape(-1, CHUNK)))
    # element types
    h16 = np.random.default_rng(2).permutation(65536).astype(np.uint16)
    check("fp16_lossless", lambda: np.array_equal(orc.decompress_typed(2, orc.compress_typed(2, h16), h16.size), h16))
    typed = [(d, wl.generate_typed(d, w, 0, start=s0, count=3 * CHUNK))
             for d in (2, 3) for w, s0 in ((2, 0), (5, (1 << 27) - CHUNK))]
    typed.append((2, h16[:3 * CHUNK]))
    check("typed_independent_encoder", lambda: all(orc.compress_typed(d, x).tobytes() == pf.encode_stream_typed(d, x)
                                                   for d, x in typed))
    check("typed_independent_decoder", lambda: all(np.array_equal(
        pf.decode_stream_typed(d, orc.compress_typed(d, x).tobytes(), x.size), x) for d, x in typed))
    tw = wl.generate_typed(2, 5, 0, start=(1 << 27) - CHUNK, count=3 * CHUNK)
    check("typed_window", lambda: orc.compress_typed(2, tw, window=True).tobytes() ==
          pf.encode_stream_typed(2, tw, window=True))
    probes = np.concatenate([np.array([65504, 65519, 65520, 65521, 2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -14,
                                       1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 3e-6, -7e-7], np.float32),
                             np.random.default_rng(6).standard_normal(4000).astype(np.float32) * 1e-4])
    with np.errstate(over="ignore"):
        probes16 = probes.astype(np.float16).view(np.uint16).tolist()
    check("fp16_rounding", lambda: [orc.round_fp16(float(v)) for v in probes] == probes16)
    h_all = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    h_fin = h_all[(h_all & 0x7C00) != 0x7C00]
    check("fp16_widening", lambda: [orc.fp16_to_float(int(v)) for v in h_fin[::7]] ==
          h_fin[::7].view(np.float16).astype(np.float32).tolist())
    f32 = [np.array(v, np.float32).view(np.uint32)
           for v in ([2.0 ** 30, 1e-39], [-(2.0 ** 30), 1e-39], [1 + 2.0 ** -20, 3.0])]
    check("fp32_sum", lambda: orc.sum_ranks_typed(3, f32).tolist() ==
          np.array([1 + 2.0 ** -20, 3.0], np.float32).view(np.uint32).tolist())
    mm32 = [np.array([0x80000000, 0x7FC00001, 0x3F800000], np.uint32), np.array([0, 0, 0xBF800000], np.uint32)]
    check("fp32_min", lambda: orc.decompress_typed(3, orc.reduce_typed(3, [orc.compress_typed(3, v) for v in mm32], 3, 1),
                                                   3).tolist() == [0x80000000, 0x7FC00000, 0xBF800000])
    check("reduce_rank_order", lambda: orc.decompress(  # 2^30, -2^30, 1 in that order
        orc.reduce([orc.compress(v) for v in (sp_a[3:], sp_b[3:], sp_c[3:])], 1), 1)[0] == 0x3F80)
    def escape_range():
        bad = bytearray(orc.compress_typed(2, ((np.arange(CHUNK) % 64 == 0) + 3).astype(np.uint16) << 10).tobytes())
        off = pf.chunk_headers(bytes(bad))[0][0]
        bad[off + 16 + 5632 + 512] = 40  # an escaped exponent no 5-bit field holds
        return orc.decompress_typed_status(2, bad, CHUNK) == orc.ERR_CORRUPT
    check("fp16_escape_range", escape_range)
    return failed


@pytest.fixture(scope="module")
def source():
    with open(ORACLE_SRC) as f:
        return f.read()


def test_unmutated_oracle_passes_battery(orc, wl):
    assert _battery(orc, wl) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(orc, wl, source, tmp_path, name, old, new):
    assert source.count(old) == 1, "mutation anchor not found: " + name
    src = tmp_path / ("oracle_%08x.c" % zlib.crc32(name.encode()))
    src.write_text(source.replace(old, new))
    lib = orc.build_from(str(src), str(tmp_path / "mutant.so"))
    with orc.use_library(lib):
        failed = _battery(orc, wl)
    assert failed, "planted mistake %r was not caught by any pin" % name
