"""The decoupled look-back that places the compress and reduce kernels'
variable-size units (groups of chunks) densely in the stream, run through the
library's own self test: every unit's offset must be the exclusive prefix sum
of the sizes before it, whether each unit has to walk back over thousands of
predecessors that published only their sizes (many 256-unit windows) or the
units publish concurrently in a scrambled order with late publishers; a
poisoned unit must stop every unit after it.  Bounded waits only: nothing
can hang, and no wait runs out (the status stays OK)."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import compression_coupled_collectives_gb300 as m

    torch.cuda.set_device(0)
    return m


def _run(cc, sizes_np, poison=None, concurrent=False):
    n = sizes_np.size
    sizes = torch.from_numpy(sizes_np.astype(np.int32)).cuda()
    result = torch.full((n,), -1, dtype=torch.int64, device="cuda")
    ws = torch.empty(16 + 8 * n + 16, dtype=torch.uint8, device="cuda")
    cc.cccl_selftest_lookback(sizes, result, ws, poison_unit=poison, concurrent=concurrent)
    _, st = cc.cccl_get_result(ws)
    return result.cpu().numpy().view(np.uint64), st


def _expected(sizes_np, poison=None):
    want = (4096 + np.concatenate([[0], np.cumsum(sizes_np.astype(np.uint64))[:-1]])).astype(np.uint64)
    if poison is not None:
        want[poison:] = np.uint64(0xC000000000000000)
    return want


def _sizes(n, seed):
    # units of 3 to 8 chunks, each 16 + 4096 + 512 k + escapes bytes or raw: 16-byte multiples below 2^17
    return np.random.default_rng(seed).integers(1, 8192, size=n).astype(np.uint32) * 16


@pytest.mark.parametrize("n", [1, 2, 257, 5000])
def test_serial_walks_over_every_predecessor(cc, n):
    sizes = _sizes(n, n)
    got, st = _run(cc, sizes)
    assert st == cc.CCCL_OK
    assert np.array_equal(got, _expected(sizes))


def test_serial_poison_stops_every_later_unit(cc):
    n, p = 3000, 1234
    sizes = _sizes(n, 7)
    got, st = _run(cc, sizes, poison=p)
    assert st == cc.CCCL_OK
    assert np.array_equal(got, _expected(sizes, p))


@pytest.mark.parametrize("n", [1000, 20000])
def test_concurrent_scrambled_publication(cc, n):
    sizes = _sizes(n, 11 + n)
    got, st = _run(cc, sizes, concurrent=True)
    assert st == cc.CCCL_OK
    assert np.array_equal(got, _expected(sizes))


def test_concurrent_poison_stops_every_later_unit(cc):
    n, p = 4000, 999
    sizes = _sizes(n, 5)
    got, st = _run(cc, sizes, poison=p, concurrent=True)
    assert st == cc.CCCL_OK
    assert np.array_equal(got, _expected(sizes, p))
