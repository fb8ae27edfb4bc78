"""GPU path vs the CPU oracle, byte for byte (tolerance 0), through the C ABI.

Compressed streams, decompressed values and reduced streams must be identical
to the oracle's on the same seeded inputs: small and ragged sizes, every bf16
bit pattern, crafted chunks at every decision boundary, the five workloads at
full size, special values, corrupt streams and argument errors.
"""

import concurrent.futures as cf
import struct

import numpy as np
import pytest
import torch

import pyformat as pf

pytestmark = pytest.mark.gpu
CHUNK = 4096


@pytest.fixture(scope="session")
def cc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import compression_coupled_collectives_gb300 as m

    torch.cuda.set_device(0)
    return m


def dev(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def gpu_compress(cc, x):
    s = cc.compress(dev(x))
    return s, s.cpu().numpy()


def check_round_trip(cc, orc, x, what=""):
    s, got = gpu_compress(cc, x)
    ref = orc.compress(x)
    if not np.array_equal(got, ref):
        diff = np.nonzero(got[:min(got.size, ref.size)] != ref[:min(got.size, ref.size)])[0]
        raise AssertionError("%s: stream differs (gpu %d bytes, oracle %d, first diff at %s)"
                             % (what, got.size, ref.size, diff[:1]))
    back = host_u16(cc.decompress(s, x.size))
    assert np.array_equal(back, x), what
    return s


# ---------------------------------------------------------------- compress / decompress
@pytest.mark.parametrize("n", [1, 2, 7, 100, 4095, 4096, 4097, 8191, 8192, 3 * 4096 + 11, 40 * 4096 + 5])
def test_sizes_and_tails(cc, orc, wl, n):
    check_round_trip(cc, orc, wl.generate(2, 0, count=n, n=max(n, 1)), "n=%d" % n)


def test_every_bf16_pattern(cc, orc):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    check_round_trip(cc, orc, x, "in order")
    for seed in (1, 2, 3):
        check_round_trip(cc, orc, np.random.default_rng(seed).permutation(65536).astype(np.uint16), "seed %d" % seed)


def _crafted_chunks():
    rng = np.random.default_rng(21)
    chunks = []
    for trial in range(240):
        n_sym = rng.integers(1, 6)
        exps = rng.choice(256, n_sym, replace=False)
        weights = rng.dirichlet(np.ones(n_sym) * rng.choice([0.05, 0.5, 5.0]))
        e = rng.choice(exps, CHUNK, p=weights).astype(np.uint16)
        sm = rng.integers(0, 256, CHUNK).astype(np.uint16)
        chunks.append(((sm & 0x80) << 8) | (e << 7) | (sm & 0x7F))
    # every width's boundaries: offsets 2^k - 2 (a code) and 2^k - 1 (an escape)
    for k in range(1, 8):
        for extra in (0, 1, 15, 16, 17, 511, 512, 513):
            e = np.full(CHUNK, 40, np.uint16)
            e[rng.choice(CHUNK, 1500, replace=False)] = 40 + (1 << k) - 2
            if extra:
                e[rng.choice(CHUNK, extra, replace=False)] = 40 + (1 << k) - 1 + rng.integers(0, 3)
            sm = rng.integers(0, 256, CHUNK).astype(np.uint16)
            chunks.append(((sm & 0x80) << 8) | (e << 7) | (sm & 0x7F))
    return np.concatenate(chunks).astype(np.uint16)


def test_crafted_chunks_every_decision(cc, orc):
    x = _crafted_chunks()
    s = check_round_trip(cc, orc, x, "crafted")
    hdrs = pf.chunk_headers(s.cpu().numpy().tobytes())
    ks = {(h[1], h[2]) for h in hdrs}
    assert len(ks) >= 8  # raw and many widths were exercised
    assert any(h[5] > 0 for h in hdrs)


def test_golden_chunks(cc, orc):
    from test_oracle_pins import _golden_cases
    import zlib

    for case in _golden_cases():
        rng = np.random.default_rng(zlib.crc32(case["name"].encode()))
        e = np.concatenate([np.full(c, ex, np.uint16) for ex, c in case["groups"]])
        e = e[rng.permutation(e.size)]
        sm = rng.integers(0, 256, e.size).astype(np.uint16)
        x = ((sm & 0x80) << 8) | (e << 7) | (sm & 0x7F)
        s = check_round_trip(cc, orc, x.astype(np.uint16), case["name"])
        hdr = pf.chunk_headers(s.cpu().numpy().tobytes())[0]
        assert hdr[6] == case["bytes"], case["name"]


@pytest.mark.parametrize("workload,start,count", [
    (1, 0, 1 << 20),
    (2, 0, 1 << 21),
    (4, 3 << 22, 1 << 21),
    (5, 0, 1 << 20),
    (5, (1 << 27) - (1 << 19), 1 << 20),  # across the boundary of the two halves
    (5, 1 << 27, 1 << 20),
])
def test_workload_slices(cc, orc, wl, workload, start, count):
    check_round_trip(cc, orc, wl.generate(workload, 0, start=start, count=count), "w%d" % workload)


def test_repeated_calls_reuse_workspace_and_buffers(cc, orc, wl):
    n = 20 * CHUNK + 3
    out = cc.empty_stream(n)
    ws = cc.empty_workspace(n)
    for seed in range(3):
        x = wl.generate(2, seed, count=n, n=n)
        cc.cccl_compress(dev(x), out, ws)
        nbytes, st = cc.cccl_get_result(ws)
        assert st == 0
        assert np.array_equal(out[:nbytes].cpu().numpy(), orc.compress(x))


def test_two_streams_two_workspaces(cc, orc, wl):
    n = 300 * CHUNK
    xs = [wl.generate(3, r, count=n) for r in range(2)]
    outs = [cc.empty_stream(n) for _ in xs]
    wss = [cc.empty_workspace(n) for _ in xs]
    streams = [torch.cuda.Stream() for _ in xs]
    d = [dev(x) for x in xs]
    torch.cuda.synchronize()
    for i in range(2):
        cc.cccl_compress(d[i], outs[i], wss[i], stream=streams[i])
    for i in range(2):
        nbytes, st = cc.cccl_get_result(wss[i], stream=streams[i])
        assert st == 0
        assert np.array_equal(outs[i][:nbytes].cpu().numpy(), orc.compress(xs[i]))


# ---------------------------------------------------------------- fused reduce
def check_reduce(cc, orc, xs, what=""):
    n = xs[0].size
    refs = [orc.compress(x) for x in xs]
    streams = [cc.compress(dev(x)) for x in xs]
    for s, r in zip(streams, refs):
        assert np.array_equal(s.cpu().numpy(), r)
    got = cc.reduce_compressed(streams, n).cpu().numpy()
    want = orc.reduce(refs, n)
    assert np.array_equal(got, want), "%s: reduced stream differs (%d vs %d bytes)" % (what, got.size, want.size)
    return got


@pytest.mark.parametrize("R", [1, 2, 3, 5, 8, 17, 64])
def test_reduce_ranks(cc, orc, wl, R):
    n = 12 * CHUNK + 77
    check_reduce(cc, orc, [wl.generate(3, r, count=n) for r in range(R)], "R=%d" % R)


def test_reduce_special_values(cc, orc):
    rng = np.random.default_rng(5)
    n = 9 * CHUNK + 1
    specials = np.array([0x7F80, 0xFF80, 0x0000, 0x8000, 0x7FC1, 0xFFFF, 0x0001, 0x8001, 0x007F, 0x7F7F, 0xFF7F,
                         0x0080, 0x3F80, 0xBF80], np.uint16)
    xs = []
    for r in range(4):
        x = rng.choice(specials, n).astype(np.uint16)
        x[: 2 * CHUNK] = rng.integers(0, 65536, 2 * CHUNK).astype(np.uint16)  # raw chunks
        xs.append(x)
    check_reduce(cc, orc, xs, "specials")


def test_reduce_exact_cases(cc, orc):
    n = CHUNK
    a = np.full(n, 0x3F80, np.uint16)
    cases = [
        (0x7F80, 0xFF80, 0x7FC0),  # Inf + -Inf
        (0x0000, 0x8000, 0x0000),  # +0 + -0
        (0x8000, 0x8000, 0x8000),  # -0 + -0
        (0x7F7F, 0x7F7F, 0x7F80),  # overflow to Inf
        (0x0001, 0x0001, 0x0002),  # subnormals, no flush to zero
        (0x7FC1, 0x3F80, 0x7FC0),  # NaN payload canonical
        (0xFFC0, 0x3F80, 0x7FC0),  # negative NaN canonical
        (0x3F80, 0x3B80, 0x3F80),  # 1 + 2^-8: tie to even stays 1
        (0x3F81, 0x3B80, 0x3F82),  # tie to even rounds up
    ]
    xa, xb = a.copy(), a.copy()
    for i, (u, v, _) in enumerate(cases):
        xa[i], xb[i] = u, v
    got = check_reduce(cc, orc, [xa, xb])
    dec = pf.decode_stream(got.tobytes(), n)
    for i, (_, _, w) in enumerate(cases):
        assert dec[i] == w, (i, hex(dec[i]), hex(w))


def test_reduce_single_rank_is_identity(cc, orc, wl):
    x = wl.generate(1, 0, count=30 * CHUNK + 9)
    s = cc.compress(dev(x))
    out = cc.reduce_compressed([s], x.size)
    assert np.array_equal(out.cpu().numpy(), s.cpu().numpy())


# ---------------------------------------------------------------- full-size workloads
def _par(fn, items):
    with cf.ThreadPoolExecutor(8) as ex:
        return list(ex.map(fn, items))


@pytest.mark.parametrize("workload", [1, 2, 3, 4, 5])
def test_full_size_workload(cc, orc, wl, workload):
    n, R = wl.SIZES[workload], wl.RANKS[workload]
    xs = _par(lambda r: wl.generate(workload, r), range(R))
    refs = _par(orc.compress, xs)
    streams = []
    for x, ref in zip(xs, refs):
        s = cc.compress(dev(x))
        assert np.array_equal(s.cpu().numpy(), ref), "workload %d compress" % workload
        if workload != 3:
            assert np.array_equal(host_u16(cc.decompress(s, n)), x), "workload %d decompress" % workload
        streams.append(s)
    if R > 1:
        got = cc.reduce_compressed(streams, n).cpu().numpy()
        want = orc.reduce(refs, n)
        assert np.array_equal(got, want), "workload %d reduce" % workload
    del streams
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- corrupt streams and errors
def _corrupt_variants(orc, wl):
    n = 3 * CHUNK + 10
    x = wl.generate(2, 0, count=n, n=1 << 20)
    s = bytearray(orc.compress(x).tobytes())
    hdrs = pf.chunk_headers(bytes(s))
    packed = next(h for h in hdrs if h[1] == 0 and h[2] > 0)
    o = packed[0]

    def mut(fn):
        t = bytearray(s)
        fn(t)
        return bytes(t)

    yield "magic", mut(lambda t: t.__setitem__(0, 0))
    yield "n_elems", mut(lambda t: struct.pack_into("<Q", t, 16, n + 1))
    yield "total_bytes", mut(lambda t: struct.pack_into("<Q", t, 32, len(s) + 16))
    yield "offset_misaligned", mut(lambda t: struct.pack_into("<Q", t, 64 + 8, hdrs[1][0] + 8))
    yield "offset_backwards", mut(lambda t: struct.pack_into("<Q", t, 64 + 16, hdrs[1][0]))
    yield "offset_huge", mut(lambda t: struct.pack_into("<Q", t, 64 + 8, 1 << 40))
    yield "next_offset_unaligned", mut(lambda t: struct.pack_into("<Q", t, 64 + 16, hdrs[2][0] + 4))
    yield "k_too_big", mut(lambda t: t.__setitem__(o + 1, 8))
    yield "mode_bad", mut(lambda t: t.__setitem__(o, 2))
    yield "n_esc_wrong", mut(lambda t: struct.pack_into("<H", t, o + 6, packed[5] + 16))
    yield "chunk_bytes_wrong", mut(lambda t: struct.pack_into("<I", t, o + 8, packed[6] + 16))
    yield "tail_n_c", mut(lambda t: struct.pack_into("<H", t, hdrs[-1][0] + 4, 11))
    # one extra sentinel: set every plane bit of an element whose code is not
    # the sentinel
    k = packed[2]
    words = np.frombuffer(bytes(s[o + 16 + 4096:o + 16 + 4096 + 512 * k]), "<u4").reshape(k, 128)
    code = sum(((words[p, pf.WORD_OF] >> pf.BIT_OF.astype(np.uint32)) & 1) << p for p in range(k))
    victim = int(np.nonzero(code != (1 << k) - 1)[0][0])
    w, b = int(pf.WORD_OF[victim]), int(pf.BIT_OF[victim])

    def extra_sentinel(t):
        for p in range(k):
            t[o + 16 + 4096 + 512 * p + 4 * w + b // 8] |= 1 << (b % 8)

    yield "sentinel_count", mut(extra_sentinel)
    yield "truncated", bytes(s[:-16])


def test_decompress_rejects_corrupt_streams(cc, orc, wl):
    n = 3 * CHUNK + 10
    for name, bad in _corrupt_variants(orc, wl):
        want = orc.decompress_status(np.frombuffer(bad, np.uint8), n)
        assert want == orc.ERR_CORRUPT, name
        d = torch.from_numpy(np.frombuffer(bad, np.uint8).copy()).cuda()
        out = torch.empty(n, dtype=torch.int16, device="cuda")
        ws = cc.empty_workspace(n)
        cc.cccl_decompress(d, out, ws)
        _, st = cc.cccl_get_result(ws)
        assert st == cc.CCCL_ERR_CORRUPT, name


def test_reduce_rejects_corrupt_input(cc, orc, wl):
    n = 3 * CHUNK + 10
    good = torch.from_numpy(orc.compress(wl.generate(2, 0, count=n, n=1 << 20))).cuda()
    for name, bad in _corrupt_variants(orc, wl):
        d = torch.from_numpy(np.frombuffer(bad, np.uint8).copy()).cuda()
        out = cc.empty_stream(n)
        ws = cc.empty_workspace(n)
        cc.cccl_reduce_compressed([good, d, good], n, out, ws)
        _, st = cc.cccl_get_result(ws)
        assert st == cc.CCCL_ERR_CORRUPT, name


# ---------------------------------------------------------------- min / max reduce ops
@pytest.mark.parametrize("op", [1, 2])
@pytest.mark.parametrize("R", [1, 2, 3, 7])
def test_reduce_min_max(cc, orc, wl, op, R):
    n = 11 * CHUNK + 123
    rng = np.random.default_rng(10 * op + R)
    specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC1, 0xFFFF, 0x0001, 0x8001, 0x3F80, 0xBF80], np.uint16)
    xs = []
    for r in range(R):
        x = wl.generate(3, r, count=n)
        idx = rng.choice(n, 300, replace=False)
        x[idx] = rng.choice(specials, idx.size)
        xs.append(x)
    refs = [orc.compress(x) for x in xs]
    streams = [torch.from_numpy(rf).cuda() for rf in refs]
    out = cc.empty_stream(n)
    ws = cc.empty_workspace(n)
    cc.cccl_reduce_op(streams, n, op, out, ws)
    nbytes, st = cc.cccl_get_result(ws)
    assert st == 0
    assert np.array_equal(out[:nbytes].cpu().numpy(), orc.reduce_op(refs, n, op))


def test_reduce_op_sum_is_reduce_compressed(cc, orc, wl):
    n = 7 * CHUNK + 1
    refs = [orc.compress(wl.generate(2, r, count=n, n=1 << 20)) for r in range(2)]
    streams = [torch.from_numpy(rf).cuda() for rf in refs]
    out = cc.empty_stream(n)
    ws = cc.empty_workspace(n)
    cc.cccl_reduce_op(streams, n, cc.CCCL_OP_SUM, out, ws)
    nbytes, _ = cc.cccl_get_result(ws)
    assert np.array_equal(out[:nbytes].cpu().numpy(), orc.reduce(refs, n))


# ---------------------------------------------------------------- selective-compression reduce
def check_reduce_mixed(cc, orc, local, xs, what=""):
    n = local.size
    refs = [orc.compress(x) for x in xs]
    streams = [cc.compress(dev(x)) for x in xs]
    got = cc.reduce_mixed(dev(local), streams).cpu().numpy()
    want = orc.reduce_mixed(local, refs, n)
    assert np.array_equal(got, want), "%s: reduced stream differs (%d vs %d bytes)" % (what, got.size, want.size)


@pytest.mark.parametrize("n_remote", [0, 1, 2, 4, 9])
@pytest.mark.parametrize("n", [100, CHUNK, 7 * CHUNK + 33, 40 * CHUNK])
def test_reduce_mixed(cc, orc, wl, n_remote, n):
    local = wl.generate(3, 7, count=n)
    xs = [wl.generate(3, r, count=n) for r in range(n_remote)]
    check_reduce_mixed(cc, orc, local, xs, "n=%d remote=%d" % (n, n_remote))


def test_reduce_mixed_special_and_raw_chunks(cc, orc, wl):
    n = 9 * CHUNK + 1001
    start = (1 << 27) - 4 * CHUNK  # across the uniform / special-value boundary of workload 5
    local = wl.generate(5, 0, start=start, count=n)
    xs = [wl.generate(5, r, start=start, count=n) for r in range(1, 4)]
    check_reduce_mixed(cc, orc, local, xs, "workload 5")


def test_reduce_mixed_full_gradient_buffer(cc, orc, wl):
    n = 1 << 22  # 128 chunk groups of the 64 MiB gradient-like workload
    local = wl.generate(2, 0, count=n)
    check_reduce_mixed(cc, orc, local, [wl.generate(3, 1, count=n)], "gradient")


def test_reduce_mixed_rejects_corrupt_remote(cc, orc, wl):
    n = 3 * CHUNK + 10
    local = dev(wl.generate(2, 0, count=n, n=1 << 20))
    good = torch.from_numpy(orc.compress(wl.generate(2, 0, count=n, n=1 << 20))).cuda()
    for name, bad in _corrupt_variants(orc, wl):
        d = torch.from_numpy(np.frombuffer(bad, np.uint8).copy()).cuda()
        out = cc.empty_stream(n)
        ws = cc.empty_workspace(n)
        cc.cccl_reduce_mixed(local, [good, d], out, ws)
        _, st = cc.cccl_get_result(ws)
        assert st == cc.CCCL_ERR_CORRUPT, name


# ---------------------------------------------------------------- window-base variant (version 2)
@pytest.mark.parametrize("workload,start,count", [
    (1, 0, 40 * CHUNK + 9), (2, 0, 64 * CHUNK), (4, 0, 32 * CHUNK),
    (5, (1 << 27) - 16 * CHUNK, 48 * CHUNK),  # uniform patterns, then N(0, 1) with specials
])
def test_window_variant(cc, orc, wl, workload, start, count):
    x = wl.generate(workload, 0, start=start, count=count)
    got = cc.compress_window(dev(x)).cpu().numpy()
    want = orc.compress_window(x)
    assert np.array_equal(got, want)
    assert np.array_equal(host_u16(cc.decompress(torch.from_numpy(got).cuda(), x.size)), x)


def test_window_variant_every_pattern_and_crafted(cc, orc):
    allp = np.random.default_rng(2).permutation(65536).astype(np.uint16)
    assert np.array_equal(cc.compress_window(dev(allp)).cpu().numpy(), orc.compress_window(allp))
    rng = np.random.default_rng(8)
    chunks = []
    for lo, hi, n_out in [(124, 130, 6), (100, 110, 0), (0, 3, 40), (250, 255, 7), (60, 70, 1000)]:
        e = rng.integers(lo, hi + 1, CHUNK)
        e[rng.choice(CHUNK, n_out, replace=False)] = rng.integers(0, 256, n_out)
        sm = rng.integers(0, 256, CHUNK)
        chunks.append((((sm & 0x80) << 8) | (e << 7) | (sm & 0x7F)).astype(np.uint16))
    x = np.concatenate(chunks)
    assert np.array_equal(cc.compress_window(dev(x)).cpu().numpy(), orc.compress_window(x))


def test_reduce_reads_window_streams(cc, orc, wl):
    n = 9 * CHUNK + 5
    xs = [wl.generate(5, r, start=1 << 27, count=n) for r in range(3)]
    ins = [cc.compress_window(dev(x)) for x in xs]
    got = cc.reduce_compressed(ins, n).cpu().numpy()
    assert np.array_equal(got, orc.reduce([orc.compress_window(x) for x in xs], n))


# ---------------------------------------------------------------- paged payload
KV_BLOCK = 16 * 8 * 128  # 16 tokens x 8 heads x 128 dim of the KV-cache shape = 4 chunks


@pytest.mark.parametrize("n_pool,n_blocks,seed", [(8, 3, 0), (64, 40, 1), (2048, 1024, 2)])
def test_paged_compress_and_decompress(cc, orc, wl, n_pool, n_blocks, seed):
    rng = np.random.default_rng(seed)
    pool = wl.generate(4, 0, count=n_pool * KV_BLOCK)
    table = rng.permutation(n_pool)[:n_blocks].astype(np.int32)
    if n_blocks > 2:
        table[-1] = table[0]  # compress may read a block twice
    dpool = dev(pool)
    dtab = torch.from_numpy(table).cuda()
    n = n_blocks * KV_BLOCK
    out = cc.empty_stream(n)
    ws = cc.empty_workspace(n)
    cc.cccl_compress_paged(dpool, KV_BLOCK, dtab, out, ws)
    nbytes, st = cc.cccl_get_result(ws)
    assert st == 0
    got = out[:nbytes].cpu().numpy()
    want = orc.compress_paged(pool, KV_BLOCK, table)
    assert np.array_equal(got, want)
    # decompress into distinct blocks of another pool
    dtab2 = torch.from_numpy(rng.permutation(n_pool)[:n_blocks].astype(np.int32)).cuda()
    target = np.full(n_pool * KV_BLOCK, 0x3C00, np.uint16)
    dtarget = dev(target)
    cc.cccl_decompress_paged(out[:nbytes], dtarget, KV_BLOCK, dtab2, ws)
    _, st = cc.cccl_get_result(ws)
    assert st == 0
    want_pool = orc.decompress_paged(want, target, KV_BLOCK, dtab2.cpu().numpy())
    assert np.array_equal(host_u16(dtarget), want_pool)


def test_paged_table_entry_outside_the_pool(cc, orc, wl):
    pool = dev(wl.generate(4, 0, count=4 * KV_BLOCK))
    n = 2 * KV_BLOCK
    out = cc.empty_stream(n)
    ws = cc.empty_workspace(n)
    for bad in ([0, 4], [-1, 1]):
        dtab = torch.tensor(bad, dtype=torch.int32, device="cuda")
        cc.cccl_compress_paged(pool, KV_BLOCK, dtab, out, ws)
        _, st = cc.cccl_get_result(ws)
        assert st == cc.CCCL_ERR_INVALID_ARG
    good = cc.compress(pool[:n])
    dtab = torch.tensor([1, 7], dtype=torch.int32, device="cuda")
    cc.cccl_decompress_paged(good, pool, KV_BLOCK, dtab, ws)
    _, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_ERR_INVALID_ARG


def test_argument_errors(cc):
    n = 5 * CHUNK
    x = torch.zeros(n, dtype=torch.int16, device="cuda")
    out = cc.empty_stream(n)
    ws = cc.empty_workspace(n)
    with pytest.raises(cc.CcclError) as e:
        cc.cccl_compress(x, out[: cc.cccl_compress_bound(n) - 16], ws)
    assert e.value.status == cc.CCCL_ERR_CAPACITY
    with pytest.raises(cc.CcclError) as e:
        cc.cccl_compress(x, out, ws[:16])
    assert e.value.status == cc.CCCL_ERR_INVALID_ARG
    big = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    with pytest.raises(cc.CcclError) as e:
        cc.cccl_compress(big[1:n + 1], out, ws)  # 2-byte misaligned input
    assert e.value.status == cc.CCCL_ERR_INVALID_ARG
    # a size larger than the device allocation is refused before any launch
    # (the check works at allocation granularity: torch sub-allocates tensors
    # from larger segments, so claim more than any segment holds)
    small_out = torch.empty(1024, dtype=torch.uint8, device="cuda")
    r = cc._lib.cccl_compress(x.data_ptr(), n, small_out.data_ptr(), 1 << 40, ws.data_ptr(), ws.numel(), None)
    assert r == cc.CCCL_ERR_INVALID_ARG
    r = cc._lib.cccl_decompress(out.data_ptr(), 1 << 40, x.data_ptr(), n, ws.data_ptr(), ws.numel(), None)
    assert r == cc.CCCL_ERR_INVALID_ARG
    host = np.zeros(n + 8, np.uint16)
    hp = (host.ctypes.data + 15) // 16 * 16  # aligned, but pageable host memory
    r = cc._lib.cccl_compress(hp, n, out.data_ptr(), out.numel(), ws.data_ptr(), ws.numel(), None)
    assert r == cc.CCCL_ERR_INVALID_ARG
    with pytest.raises(cc.CcclError) as e:
        cc.cccl_reduce_compressed([], n, out, ws)
    assert e.value.status == cc.CCCL_ERR_INVALID_ARG
    with pytest.raises(cc.CcclError) as e:
        cc.cccl_reduce_compressed([out] * 65, n, out, ws)
    assert e.value.status == cc.CCCL_ERR_INVALID_ARG
    # the library still works after all of that
    cc.cccl_compress(x, out, ws)
    nbytes, st = cc.cccl_get_result(ws)
    assert st == 0 and nbytes > 0


# ---------------------------------------------------------------- CUDA graphs
def test_step_captured_in_a_cuda_graph(cc, orc, wl):
    """The C ABI calls only enqueue work on the given stream (no host sync, no
    allocation), so a whole step (two compressions, the fused reduce and the
    decompression, each with its workspace clear) can be captured in a CUDA
    graph and replayed; every replay reproduces the oracle's streams."""
    n = 23 * CHUNK + 5
    xs_host = [wl.generate(2, r, count=n, n=1 << 20) for r in range(2)]
    xs = [dev(x) for x in xs_host]
    outs = [cc.empty_stream(n) for _ in xs]
    red = cc.empty_stream(n)
    y = torch.empty(n, dtype=torch.int16, device="cuda")
    wss = [cc.empty_workspace(n) for _ in range(4)]
    sizes = []
    for x, o, w in zip(xs, outs, wss):  # a first, uncaptured call of each entry point
        cc.cccl_compress(x, o, w)
        sizes.append(cc.cccl_get_result(w)[0])
    cc.cccl_reduce_compressed(outs, n, red, wss[2])
    cc.cccl_get_result(wss[2])
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        s = torch.cuda.current_stream()
        for x, o, w in zip(xs, outs, wss):
            cc.cccl_compress(x, o, w, stream=s)
        cc.cccl_reduce_compressed(outs, n, red, wss[2], stream=s)
        cc.cccl_decompress(red, y, wss[3], stream=s)
    refs = [orc.compress(x) for x in xs_host]
    want_red = orc.reduce(refs, n)
    for rep in range(3):
        for o in outs:
            o.zero_()
        red.zero_()
        y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for o, w, ref in zip(outs, wss, refs):
            nb, st = cc.cccl_get_result(w)
            assert st == 0 and np.array_equal(o[:nb].cpu().numpy(), ref), rep
        nb, st = cc.cccl_get_result(wss[2])
        assert st == 0 and np.array_equal(red[:nb].cpu().numpy(), want_red), rep
        assert np.array_equal(host_u16(y), orc.decompress(want_red, n)), rep


def test_full_size_step_in_a_cuda_graph(cc, orc, wl):
    """The benchmark's step as it times it: workload 2 at full size on two
    simulated ranks, captured once as a CUDA graph and replayed.  Every replay
    gives the same bytes as the plain calls (whose streams the full-size
    workload test checks against the oracle), and sampled chunks match the
    oracle directly."""
    n = wl.SIZES[2]
    xs_host = [wl.generate(2, r) for r in range(2)]
    xs = [dev(x) for x in xs_host]
    outs = [cc.empty_stream(n) for _ in xs]
    red = cc.empty_stream(n)
    y = torch.empty(n, dtype=torch.int16, device="cuda")
    wss = [cc.empty_workspace(n) for _ in range(4)]

    def step(s=None):
        for x, o, w in zip(xs, outs, wss):
            cc.cccl_compress(x, o, w, stream=s)
        cc.cccl_reduce_compressed(outs, n, red, wss[2], stream=s)
        cc.cccl_decompress(red, y, wss[3], stream=s)

    step()
    plain = [o[:cc.cccl_get_result(w)[0]].clone() for o, w in zip(outs + [red], wss[:3])]
    y_plain = y.clone()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        step(torch.cuda.current_stream())
    for rep in range(2):
        for t in outs + [red, y]:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for o, w, p in zip(outs + [red], wss[:3], plain):
            nb, st = cc.cccl_get_result(w)
            assert st == 0 and nb == p.numel() and torch.equal(o[:nb], p), rep
        assert torch.equal(y, y_plain), rep
    # sampled chunks of the replayed streams against the oracle
    head = outs[0][:64 + 8 * (n // CHUNK)].cpu().numpy().tobytes()
    for c in (0, 1, 4095, n // CHUNK - 1):
        o0, o1 = struct.unpack_from("<QQ", head, 64 + 8 * c) if c + 1 < n // CHUNK else (
            struct.unpack_from("<Q", head, 64 + 8 * c)[0], plain[0].numel())
        got = outs[0][o0:o1].cpu().numpy().tobytes()
        assert got == bytes(orc.encode_chunk(xs_host[0][c * CHUNK:(c + 1) * CHUNK])), c
    want = orc.sum_ranks([x[:8 * CHUNK] for x in xs_host])
    assert np.array_equal(host_u16(y[:8 * CHUNK]), want)


# ---------------------------------------------------------------- streams past 4 GiB
def test_streams_past_4_gib(cc, orc, wl):
    """3 x 2^30 + 3 chunks + 5 values per rank (about 6 GiB of bf16; the
    streams, about 5 GB, pass 2^32 bytes): the offset table, compress,
    decompress and the fused reduce must carry 64-bit offsets and element
    indices.  The input tiles one
    seeded 2^20-value block; every chunk's bytes depend only on its own
    values, so sampled chunks are checked against the oracle chunk by chunk,
    the offset table against the chunk sizes, and the round trip in full on
    the device."""
    import struct

    tile = 1 << 20
    n = 3 * (1 << 30) + 3 * CHUNK + 5
    base = [wl.generate(2, r, count=tile, n=tile) for r in range(2)]
    reps = -(-n // tile)
    xs = [dev(b).repeat(reps)[:n].contiguous() for b in base]
    streams = [cc.compress(x) for x in xs]
    red = cc.reduce_compressed(streams, n)
    nch = -(-n // CHUNK)
    samples = [0, 1, 255, 256, nch // 2, nch - 3, nch - 2, nch - 1]
    for s_dev, b in zip(streams + [red], base + [None]):
        total = int(s_dev.numel())
        head = s_dev[:64].cpu().numpy().tobytes()
        assert struct.unpack_from("<QQQ", head, 16) == (n, nch, total)
        assert total > (1 << 32)
        offs = s_dev[64:64 + 8 * nch].cpu().numpy().view(np.uint64).astype(np.int64)
        ends = np.append(offs[1:], total)
        sizes = ends - offs
        assert (sizes > 0).all() and (sizes % 16 == 0).all() and offs[0] == 64 + -(-8 * nch // 16) * 16
        for c in samples:
            got = s_dev[int(offs[c]):int(ends[c])].cpu().numpy().tobytes()
            lo = c * CHUNK
            n_c = min(CHUNK, n - lo)
            if b is not None:
                want = orc.encode_chunk(b[lo % tile:lo % tile + n_c])
            else:  # the reduce: chunk c of the sum of chunk c of both ranks
                parts = [orc.compress(bb[lo % tile:lo % tile + n_c]) for bb in base]
                one = orc.reduce(parts, n_c)
                o0 = struct.unpack_from("<Q", one.tobytes(), 64)[0]
                want = one.tobytes()[o0:]
            assert got == want, "chunk %d" % c
    for x, s_dev in zip(xs, streams):
        assert torch.equal(cc.decompress(s_dev, n), x)
    del xs, streams, red
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- bounded waits
def test_bounded_waits_time_out_and_the_context_survives(cc, orc, wl):
    """An mbarrier no thread arrives on and a look-back whose predecessor never
    publishes: both waits give up after the 2 s limit and report TIMEOUT on the
    host; the context stays usable for the next call."""
    import time

    ws = cc.empty_workspace(8192)
    t0 = time.time()
    cc.cccl_selftest_timeouts(ws)
    nbytes, st = cc.cccl_get_result(ws)
    took = time.time() - t0
    assert st == cc.CCCL_ERR_TIMEOUT
    assert nbytes == 0
    assert 1.5 < took < 30.0
    # the look-back poisoned its own unit for its successors
    status = ws[16:32].cpu().numpy().view(np.uint64)
    assert int(status[1]) >> 62 == 3
    x = wl.generate(2, 0, count=3 * CHUNK + 7, n=1 << 20)
    assert np.array_equal(cc.compress(dev(x)).cpu().numpy(), orc.compress(x))
