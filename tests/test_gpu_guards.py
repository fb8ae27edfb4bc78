"""Guard bands around every buffer the library writes (the stand-in for a
memory checker on this GPU): outputs, workspaces and decoded values sit in
larger allocations filled with a pattern, the library is given only the
inner part, and afterwards every byte past what the call may write must
still hold the pattern.  Ragged sizes (one value, a partial chunk, several
chunks and a tail), every element type, the table-driven paged payload, and
the entry point that uses its own static scratch."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

GUARD = 4096        # bytes of pattern past each buffer
PAT_OUT, PAT_WS, PAT_VAL = 0xA5, 0x5A, 0x3C
SIZES = [1, 4095, 3 * 4096 + 7, 40 * 4096 + 5]


@pytest.fixture(scope="module")
def cc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import compression_coupled_collectives_gb300 as m

    torch.cuda.set_device(0)
    return m


def guarded(nbytes: int, pattern: int) -> tuple[torch.Tensor, torch.Tensor]:
    """A uint8 device buffer of nbytes + GUARD bytes, all `pattern`, and its first nbytes."""
    full = torch.full((nbytes + GUARD,), pattern, dtype=torch.uint8, device="cuda")
    return full, full[:nbytes]


def untouched(full: torch.Tensor, start: int, pattern: int) -> bool:
    return bool((full[start:] == pattern).all())


def ws_guarded(cc, n):
    # a workspace 64 bytes larger than needed, so that its tail is checked too
    need = cc.cccl_workspace_bytes(n)
    full, ws = guarded(need + 64, PAT_WS)
    used = 16 + 8 * (-(-n // 4096))
    return full, ws, used


def values(wl, w, r, n, dtype=None):
    if dtype is None:
        return torch.from_numpy(wl.generate(w, r, count=n, n=max(n, 1 << 20)).view(np.int16)).cuda()
    bits = np.int16 if dtype != 3 else np.int32
    return torch.from_numpy(wl.generate_typed(dtype, w, r, count=n, n=max(n, 1 << 20)).view(bits)).cuda()


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("window", [False, True])
def test_compress_writes_only_its_stream(cc, wl, n, window):
    x = values(wl, 2, 0, n)
    full, out = guarded(cc.cccl_compress_bound(n), PAT_OUT)
    wfull, ws, used = ws_guarded(cc, n)
    (cc.cccl_compress_window if window else cc.cccl_compress)(x, out, ws)
    total, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_OK and 0 < total <= out.numel()
    assert untouched(full, total, PAT_OUT)       # [total, capacity) and past the buffer
    assert untouched(wfull, used, PAT_WS)        # the workspace past what the call uses


@pytest.mark.parametrize("n", SIZES)
def test_decompress_writes_only_n_values(cc, wl, n):
    x = values(wl, 2, 1, n)
    s = cc.compress(x)
    full = torch.full((n + GUARD,), PAT_VAL * 0x0101, dtype=torch.int16, device="cuda")
    wfull, ws, _ = ws_guarded(cc, n)
    cc.cccl_decompress(s, full[:n], ws)
    _, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_OK
    assert torch.equal(full[:n], x)
    assert bool((full[n:] == PAT_VAL * 0x0101).all())
    assert untouched(wfull, 16, PAT_WS)          # decompress uses the 16-byte header only


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("R", [1, 3, 8])
def test_reduce_writes_only_its_stream(cc, wl, n, R):
    streams = [cc.compress(values(wl, 1, r, n)) for r in range(R)]
    full, out = guarded(cc.cccl_compress_bound(n), PAT_OUT)
    wfull, ws, used = ws_guarded(cc, n)
    cc.cccl_reduce_compressed(streams, n, out, ws)
    total, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_OK
    assert untouched(full, total, PAT_OUT)
    assert untouched(wfull, used, PAT_WS)
    # min over the same streams: same guard
    full2, out2 = guarded(cc.cccl_compress_bound(n), PAT_OUT)
    cc.cccl_reduce_op(streams, n, cc.CCCL_OP_MIN, out2, ws)
    total2, st2 = cc.cccl_get_result(ws)
    assert st2 == cc.CCCL_OK and untouched(full2, total2, PAT_OUT)


@pytest.mark.parametrize("n", SIZES)
def test_reduce_mixed_writes_only_its_stream(cc, wl, n):
    local = values(wl, 2, 0, n)
    remote = [cc.compress(values(wl, 2, r, n)) for r in (1, 2)]
    full, out = guarded(cc.cccl_compress_bound(n), PAT_OUT)
    wfull, ws, used = ws_guarded(cc, n)
    cc.cccl_reduce_mixed(local, remote, out, ws)
    total, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_OK
    assert untouched(full, total, PAT_OUT)
    assert untouched(wfull, used, PAT_WS)


@pytest.mark.parametrize("dtype", [2, 3])
@pytest.mark.parametrize("n", SIZES)
def test_typed_calls_write_only_their_buffers(cc, wl, dtype, n):
    xs = [values(wl, 2, r, n, dtype) for r in range(2)]
    item = 2 if dtype == 2 else 4
    wfull, ws, used = ws_guarded(cc, n)
    streams = []
    for x in xs:
        full, out = guarded(cc.cccl_compress_bound_typed(dtype, n), PAT_OUT)
        cc.cccl_compress_typed(dtype, x, out, ws)
        total, st = cc.cccl_get_result(ws)
        assert st == cc.CCCL_OK and untouched(full, total, PAT_OUT) and untouched(wfull, used, PAT_WS)
        streams.append(out[:total])
    full, out = guarded(cc.cccl_compress_bound_typed(dtype, n), PAT_OUT)
    cc.cccl_reduce_typed(dtype, cc.CCCL_OP_SUM, xs[0], streams[1:], n, out, ws)
    total, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_OK and untouched(full, total, PAT_OUT) and untouched(wfull, used, PAT_WS)
    vfull = torch.full(((n * item + GUARD) // item,), 0, dtype=xs[0].dtype, device="cuda")
    vfull.view(torch.uint8).fill_(PAT_VAL)
    cc.cccl_decompress_typed(dtype, streams[0], vfull[:n], ws)
    _, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_OK and torch.equal(vfull[:n], xs[0])
    assert bool((vfull.view(torch.uint8)[n * item:] == PAT_VAL).all())


def test_paged_calls_write_only_their_blocks(cc, wl):
    block = 2 * 4096
    n_pool, n_blk = 64, 20
    pool = torch.from_numpy(wl.generate(4, 0, count=n_pool * block).view(np.int16)).cuda()
    table = torch.from_numpy(np.random.default_rng(3).permutation(n_pool)[:n_blk].astype(np.int32)).cuda()
    n = n_blk * block
    full, out = guarded(cc.cccl_compress_bound(n), PAT_OUT)
    wfull, ws, used = ws_guarded(cc, n)
    cc.cccl_compress_paged(pool, block, table, out, ws)
    total, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_OK and untouched(full, total, PAT_OUT) and untouched(wfull, used, PAT_WS)
    # decompress into a second pool: the named blocks get their values, every
    # other block and the bytes past the pool keep the pattern
    tfull = torch.full((n_pool * block + GUARD // 2,), PAT_VAL * 0x0101, dtype=torch.int16, device="cuda")
    target = tfull[:n_pool * block]
    cc.cccl_decompress_paged(out[:total], target, block, table, ws)
    _, st = cc.cccl_get_result(ws)
    assert st == cc.CCCL_OK
    tb = target.view(n_pool, block)
    named = torch.zeros(n_pool, dtype=torch.bool, device="cuda")
    named[table.long()] = True
    assert torch.equal(tb[table.long()], pool.view(n_pool, block)[table.long()])
    assert bool((tb[~named] == PAT_VAL * 0x0101).all())
    assert bool((tfull[n_pool * block:] == PAT_VAL * 0x0101).all())


@pytest.mark.parametrize("n", SIZES)
def test_noalloc_writes_only_its_stream(cc, wl, n):
    x = values(wl, 2, 3, n)
    full, out = guarded(cc.cccl_compress_bound(n), PAT_OUT)
    cc.cccl_compress_noalloc(x, out)
    torch.cuda.synchronize()
    total = int(out[32:40].cpu().numpy().view(np.uint64)[0])
    assert 0 < total <= out.numel()
    assert untouched(full, total, PAT_OUT)
