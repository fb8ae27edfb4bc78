"""cccl_compress_noalloc: compression for callers that cannot allocate device
memory (another component owns the memory pool, cudaMalloc is not allowed or
would synchronise at that point, or there is no allocator at all).  Its
scratch is a static device array inside the library, so the caller passes only
the input and the output.  Checked through the C ABI against cccl_compress,
byte for byte, on two calls in a row that share that scratch.

This file is collected last so that a failure here, under -x, comes after
every other test has run."""

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


def _stream_size(out: torch.Tensor) -> int:
    return int(out[32:40].cpu().numpy().view(np.uint64)[0])


def test_noalloc_matches_compress_on_two_calls_in_a_row(cc, wl):
    n = 2000 * 4096 + 777  # many groups and a raw partial chunk
    xs = [torch.from_numpy(wl.generate(2, r, count=n, n=n).view(np.int16)).cuda() for r in range(2)]
    refs = [cc.compress(x) for x in xs]  # the existing entry point, with its own workspace
    outs = [cc.empty_stream(n) for _ in xs]
    for x, out in zip(xs, outs):  # back to back on one stream: the scratch is reused in order
        cc.cccl_compress_noalloc(x, out)
    torch.cuda.synchronize()
    for out, ref in zip(outs, refs):
        size = _stream_size(out)
        assert size == ref.numel()
        assert torch.equal(out[:size], ref)  # tolerance 0: identical bytes


def test_noalloc_larger_call_then_smaller_call(cc, wl):
    """The scratch keeps the previous call's placement words; a smaller call
    after a larger one must clear what it uses and give the same bytes as the
    entry point with its own workspace."""
    sizes = [2000 * 4096 + 777, 3 * 4096 + 5, 1]
    for n in sizes:
        x = torch.from_numpy(wl.generate(2, 5, count=n, n=1 << 24).view(np.int16)).cuda()
        ref = cc.compress(x)
        out = cc.empty_stream(n)
        cc.cccl_compress_noalloc(x, out)
        torch.cuda.synchronize()
        size = _stream_size(out)
        assert size == ref.numel()
        assert torch.equal(out[:size], ref)


def test_noalloc_rejects_sizes_beyond_its_scratch(cc):
    x = torch.zeros(16, dtype=torch.int16, device="cuda")
    out = torch.zeros(64, dtype=torch.uint8, device="cuda")
    limit = 1 << 30
    r = cc._lib.cccl_compress_noalloc(x.data_ptr(), limit + 1, out.data_ptr(), 1 << 40, None)
    assert r == cc.CCCL_ERR_INVALID_ARG
    r = cc._lib.cccl_compress_noalloc(x.data_ptr(), 0, out.data_ptr(), 64, None)
    assert r == cc.CCCL_ERR_INVALID_ARG
