"""GPU path vs the CPU oracle for the fp16 and fp32 element types, byte for
byte (tolerance 0), through the C ABI's typed entry points: compress (both
table choices), decompress, and the fused reduce with every operator and the
local operand; ragged sizes, every fp16 bit pattern, crafted chunks at every
width boundary, the workloads' recipes at full size, special values and
corrupt streams.
"""

import concurrent.futures as cf

import numpy as np
import pytest
import torch

import pyformat as pf

pytestmark = pytest.mark.gpu
CHUNK = 4096
BF16, FP16, FP32 = 1, 2, 3
WIDTH = {BF16: 16, FP16: 16, FP32: 32}


@pytest.fixture(scope="session")
def cc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import compression_coupled_collectives_gb300 as m

    torch.cuda.set_device(0)
    return m


def dev(dtype, x: np.ndarray) -> torch.Tensor:
    x = np.ascontiguousarray(x)
    return torch.from_numpy(x.view(np.int32 if WIDTH[dtype] == 32 else np.int16)).cuda()


def host(dtype, t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32 if WIDTH[dtype] == 32 else np.uint16)


def check_round_trip(cc, orc, dtype, x, window=False, what=""):
    s = cc.compress_typed(dtype, dev(dtype, x), window=window)
    got = s.cpu().numpy()
    ref = orc.compress_typed(dtype, x, window=window)
    if not np.array_equal(got, ref):
        m = min(got.size, ref.size)
        diff = np.nonzero(got[:m] != ref[:m])[0]
        raise AssertionError("%s: stream differs (gpu %d bytes, oracle %d, first diff at %s)"
                             % (what, got.size, ref.size, diff[:1]))
    back = host(dtype, cc.decompress_typed(dtype, s, x.size))
    assert np.array_equal(back, x), what
    return s


def _rand_bits(dtype, n, seed):
    rng = np.random.default_rng(seed)
    if WIDTH[dtype] == 32:
        return rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    return rng.integers(0, 1 << 16, n).astype(np.uint16)


# ---------------------------------------------------------------- compress / decompress
@pytest.mark.parametrize("dtype", [FP16, FP32])
@pytest.mark.parametrize("window", [False, True])
@pytest.mark.parametrize("n", [1, 3, 4095, 4096, 4097, 8192, 5 * 4096 + 77, 37 * 4096 + 1])
def test_sizes_and_tails(cc, orc, wl, dtype, window, n):
    check_round_trip(cc, orc, dtype, wl.generate_typed(dtype, 2, 0, count=n, n=max(n, 1)), window, "n=%d" % n)


@pytest.mark.parametrize("window", [False, True])
def test_every_fp16_pattern(cc, orc, window):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    check_round_trip(cc, orc, FP16, x, window, "in order")
    for seed in (1, 2):
        check_round_trip(cc, orc, FP16, np.random.default_rng(seed).permutation(65536).astype(np.uint16), window,
                         "seed %d" % seed)


@pytest.mark.parametrize("window", [False, True])
def test_random_fp32_patterns(cc, orc, window):
    check_round_trip(cc, orc, FP32, _rand_bits(FP32, 40 * CHUNK + 3, 5), window, "random")


def _crafted(dtype, seed):
    """Chunks at every width's boundaries and random skewed tables, for the
    type's exponent field."""
    rng = np.random.default_rng(seed)
    ebits = 5 if dtype == FP16 else 8
    nsym = 1 << ebits
    chunks = []
    for _ in range(120):
        n_sym = rng.integers(1, 6)
        exps = rng.choice(nsym, n_sym, replace=False)
        w = rng.dirichlet(np.ones(n_sym) * rng.choice([0.05, 0.5, 5.0]))
        chunks.append(rng.choice(exps, CHUNK, p=w))
    base = 3 if dtype == FP16 else 40
    for k in range(1, ebits):
        for extra in (0, 1, 15, 16, 17, 511, 512, 513):
            e = np.full(CHUNK, base)
            e[rng.choice(CHUNK, 1500, replace=False)] = base + (1 << k) - 2
            if extra:
                e[rng.choice(CHUNK, extra, replace=False)] = min(base + (1 << k) - 1 + rng.integers(0, 3), nsym - 1)
            chunks.append(e)
    # low outliers below a narrow window (the window variant's case)
    for lo in (0, 1):
        e = np.full(CHUNK, nsym - 4)
        e[rng.choice(CHUNK, 40, replace=False)] = lo
        chunks.append(e)
    e = np.concatenate(chunks)
    rest = _rand_bits(dtype, e.size, seed + 1)
    if dtype == FP16:
        return ((rest & np.uint16(0x83FF)) | (e.astype(np.uint16) << 10)).astype(np.uint16)
    return ((rest & np.uint32(0x807FFFFF)) | (e.astype(np.uint32) << 23)).astype(np.uint32)


@pytest.mark.parametrize("dtype", [FP16, FP32])
@pytest.mark.parametrize("window", [False, True])
def test_crafted_chunks_every_decision(cc, orc, dtype, window):
    x = _crafted(dtype, 30 + dtype)
    s = check_round_trip(cc, orc, dtype, x, window, "crafted")
    hdrs = pf.chunk_headers(s.cpu().numpy().tobytes())
    assert len({(h[1], h[2]) for h in hdrs}) >= (5 if dtype == FP16 or window else 8)  # raw and many widths
    assert any(h[5] > 0 for h in hdrs)


def test_bf16_typed_is_the_bf16_path(cc, orc, wl):
    x = wl.generate(2, 0, count=9 * CHUNK + 5, n=1 << 20)
    d = dev(BF16, x)
    assert np.array_equal(cc.compress_typed(BF16, d).cpu().numpy(), cc.compress(d).cpu().numpy())
    assert np.array_equal(cc.compress_typed(BF16, d, window=True).cpu().numpy(), cc.compress_window(d).cpu().numpy())
    s = cc.compress(d)
    assert np.array_equal(host(BF16, cc.decompress_typed(BF16, s, x.size)), x)


# ---------------------------------------------------------------- fused reduce
def check_reduce(cc, orc, dtype, xs, op=0, local=False, window_inputs=False, what=""):
    n = xs[0].size
    refs = [orc.compress_typed(dtype, x, window=window_inputs) for x in xs]
    streams = [torch.from_numpy(r).cuda() for r in refs]
    if local:
        got = cc.reduce_typed(dtype, streams[1:], n, op, local=dev(dtype, xs[0])).cpu().numpy()
        want = orc.reduce_typed(dtype, refs[1:], n, op, local=xs[0])
    else:
        got = cc.reduce_typed(dtype, streams, n, op).cpu().numpy()
        want = orc.reduce_typed(dtype, refs, n, op)
    assert np.array_equal(got, want), "%s: reduced stream differs (%d vs %d bytes)" % (what, got.size, want.size)
    return got


@pytest.mark.parametrize("dtype", [FP16, FP32])
@pytest.mark.parametrize("op", [0, 1, 2])
@pytest.mark.parametrize("R", [1, 2, 3, 8])
def test_reduce_ranks_and_ops(cc, orc, wl, dtype, op, R):
    n = 10 * CHUNK + 55
    check_reduce(cc, orc, dtype, [wl.generate_typed(dtype, 3, r, count=n) for r in range(R)], op, what="R=%d" % R)


@pytest.mark.parametrize("dtype", [FP16, FP32])
@pytest.mark.parametrize("op", [0, 1, 2])
def test_reduce_local_operand(cc, orc, wl, dtype, op):
    for n in (7 * CHUNK, 7 * CHUNK + 901):
        xs = [wl.generate_typed(dtype, 2, r, count=n, n=1 << 20) for r in range(3)]
        check_reduce(cc, orc, dtype, xs, op, local=True, what="n=%d" % n)
    xs = [wl.generate_typed(dtype, 2, 0, count=3 * CHUNK, n=1 << 20)]
    check_reduce(cc, orc, dtype, xs, op, local=True, what="local only")


@pytest.mark.parametrize("dtype", [FP16, FP32])
def test_reduce_special_values_and_raw_chunks(cc, orc, dtype):
    rng = np.random.default_rng(50 + dtype)
    n = 9 * CHUNK + 1
    if dtype == FP16:
        specials = np.array([0x7C00, 0xFC00, 0x0000, 0x8000, 0x7E01, 0xFFFF, 0x0001, 0x8001, 0x03FF, 0x7BFF, 0xFBFF,
                             0x0400, 0x3C00, 0xBC00], np.uint16)
    else:
        specials = np.array([0x7F800000, 0xFF800000, 0, 0x80000000, 0x7FC00001, 0xFFFFFFFF, 1, 0x80000001,
                             0x007FFFFF, 0x7F7FFFFF, 0xFF7FFFFF, 0x00800000, 0x3F800000, 0xBF800000], np.uint32)
    xs = []
    for r in range(4):
        x = rng.choice(specials, n)
        x[:2 * CHUNK] = _rand_bits(dtype, 2 * CHUNK, 60 + r)  # raw chunks
        xs.append(x.astype(specials.dtype))
    for op in (0, 1, 2):
        check_reduce(cc, orc, dtype, xs, op, what="specials op %d" % op)


def test_fp16_reduce_exact_cases(cc, orc):
    cases = [
        (0x7C00, 0xFC00, 0x7E00),  # Inf + -Inf
        (0x0000, 0x8000, 0x0000),  # +0 + -0
        (0x8000, 0x8000, 0x8000),  # -0 + -0
        (0x7BFF, 0x7BFF, 0x7C00),  # 65504 + 65504 overflows
        (0x0001, 0x0001, 0x0002),  # subnormals kept
        (0x7E01, 0x3C00, 0x7E00),  # NaN payload canonical
        (0x3C00, 0x1000, 0x3C00),  # 1 + 2^-11: a tie, stays 1 (even)
        (0x3C01, 0x1000, 0x3C02),  # 1 + 2^-10 + 2^-11: a tie, rounds to even
    ]
    a = np.full(CHUNK, 0x3C00, np.uint16)
    xa, xb = a.copy(), a.copy()
    for i, (u, v, _) in enumerate(cases):
        xa[i], xb[i] = u, v
    got = check_reduce(cc, orc, FP16, [xa, xb])
    dec = pf.decode_stream_typed(FP16, got.tobytes(), CHUNK)
    for i, (_, _, w) in enumerate(cases):
        assert dec[i] == w, (i, hex(dec[i]), hex(w))


@pytest.mark.parametrize("dtype", [FP16, FP32])
def test_reduce_reads_window_streams(cc, orc, wl, dtype):
    xs = [wl.generate_typed(dtype, 5, r, start=(1 << 27) - 4 * CHUNK, count=8 * CHUNK) for r in range(3)]
    check_reduce(cc, orc, dtype, xs, 0, window_inputs=True, what="window inputs")


# ---------------------------------------------------------------- full-size workloads
def _par(fn, items):
    with cf.ThreadPoolExecutor(8) as ex:
        return list(ex.map(fn, items))


@pytest.mark.parametrize("dtype", [FP16, FP32])
@pytest.mark.parametrize("workload", [1, 2, 5])
def test_full_size_workload(cc, orc, wl, dtype, workload):
    n, R = wl.SIZES[workload], max(2, wl.RANKS[workload])
    if workload == 5:
        n, R = 1 << 25, 2  # the same recipe over 2^25 values (both halves)
    xs = _par(lambda r: wl.generate_typed(dtype, workload, r, n=n), range(R))
    refs = _par(lambda x: orc.compress_typed(dtype, x), xs)
    streams = []
    for x, ref in zip(xs, refs):
        s = cc.compress_typed(dtype, dev(dtype, x))
        assert np.array_equal(s.cpu().numpy(), ref), "workload %d compress" % workload
        assert np.array_equal(host(dtype, cc.decompress_typed(dtype, s, n)), x), "workload %d decompress" % workload
        streams.append(s)
    got = cc.reduce_typed(dtype, streams, n).cpu().numpy()
    want = orc.reduce_typed(dtype, refs, n)
    assert np.array_equal(got, want), "workload %d reduce" % workload
    del streams
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- corrupt streams
def _bad_variants(orc, wl, dtype):
    n = 3 * CHUNK + 10
    x = wl.generate_typed(dtype, 2, 0, count=n, n=1 << 20)
    s = bytearray(orc.compress_typed(dtype, x).tobytes())
    hdrs = pf.chunk_headers(bytes(s))
    packed = next(h for h in hdrs if h[1] == 0 and h[2] > 0)
    o = packed[0]

    def mut(fn):
        t = bytearray(s)
        fn(t)
        return bytes(t)

    other = FP32 if dtype == FP16 else FP16
    yield "dtype", mut(lambda t: t.__setitem__(6, other))
    yield "k_too_big", mut(lambda t: t.__setitem__(o + 1, 5 if dtype == FP16 else 8))
    if dtype == FP16:
        yield "base_above_31", mut(lambda t: t.__setitem__(o + 2, 32))
        if packed[5] > 0:
            resid = 4096 + 1536
            yield "escape_above_31", mut(lambda t: t.__setitem__(o + 16 + resid + 512 * packed[2], 40))
    yield "chunk_bytes_wrong", mut(lambda t: t.__setitem__(o + 8, (t[o + 8] + 16) & 0xFF))
    yield "truncated", bytes(s[:-16])


@pytest.mark.parametrize("dtype", [FP16, FP32])
def test_decompress_and_reduce_reject_corrupt_streams(cc, orc, wl, dtype):
    n = 3 * CHUNK + 10
    good = torch.from_numpy(orc.compress_typed(dtype, wl.generate_typed(dtype, 2, 0, count=n, n=1 << 20))).cuda()
    for name, bad in _bad_variants(orc, wl, dtype):
        assert orc.decompress_typed_status(dtype, np.frombuffer(bad, np.uint8), n) == orc.ERR_CORRUPT, name
        d = torch.from_numpy(np.frombuffer(bad, np.uint8).copy()).cuda()
        out = torch.empty(n, dtype=torch.int32 if dtype == FP32 else torch.int16, device="cuda")
        ws = cc.empty_workspace(n)
        cc.cccl_decompress_typed(dtype, d, out, ws)
        assert cc.cccl_get_result(ws)[1] == cc.CCCL_ERR_CORRUPT, name
        rout = cc.empty_stream_typed(dtype, n)
        cc.cccl_reduce_typed(dtype, 0, None, [good, d], n, rout, ws)
        assert cc.cccl_get_result(ws)[1] == cc.CCCL_ERR_CORRUPT, name
