"""The C ABI library on a machine without a GPU: it loads, exports every entry
point that include/cccl.h declares, and its pure host functions and host-side
argument checks behave as documented (no compute is launched)."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cccl.h")


@pytest.fixture(scope="module")
def cc():
    import __graft_entry__

    __graft_entry__.build()
    import compression_coupled_collectives_gb300 as m

    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cccl_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    assert names == sorted(["cccl_compress_bound", "cccl_workspace_bytes", "cccl_compress", "cccl_compress_noalloc",
                            "cccl_decompress", "cccl_reduce_compressed", "cccl_reduce_mixed", "cccl_get_result",
                            "cccl_status_string", "cccl_compress_paged", "cccl_decompress_paged",
                            "cccl_compress_window", "cccl_reduce_op", "cccl_compress_bound_typed",
                            "cccl_compress_typed", "cccl_decompress_typed", "cccl_reduce_typed",
                            "cccl_selftest_timeouts", "cccl_selftest_lookback"]), names


def test_library_exports_every_declared_symbol(cc):
    lib = ctypes.CDLL(cc.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name


@pytest.mark.parametrize("n", [1, 2, 4095, 4096, 4097, 1 << 20, (1 << 28) + 3])
def test_bound_matches_oracle(cc, orc, n):
    assert cc.cccl_compress_bound(n) == orc.compress_bound(n)
    nch = -(-n // 4096)
    assert cc.cccl_workspace_bytes(n) == -(-(16 + 8 * nch) // 16) * 16


@pytest.mark.parametrize("dtype", [1, 2, 3])
@pytest.mark.parametrize("n", [1, 4095, 4096, 4097, 1 << 20, (1 << 26) + 5])
def test_typed_bound_matches_oracle(cc, orc, dtype, n):
    assert cc.cccl_compress_bound_typed(dtype, n) == orc.compress_bound_typed(dtype, n)


def test_typed_bound_limits(cc):
    assert cc.cccl_compress_bound_typed(1, 12345) == cc.cccl_compress_bound(12345)
    assert cc.cccl_compress_bound_typed(0, 4096) == 0
    assert cc.cccl_compress_bound_typed(4, 4096) == 0
    assert cc.cccl_compress_bound_typed(3, 0) == 0
    assert cc.cccl_compress_bound_typed(2, (1 << 40) + 1) == 0


def test_bound_and_workspace_limits(cc):
    assert cc.cccl_compress_bound(0) == 0
    assert cc.cccl_workspace_bytes(0) == 0
    assert cc.cccl_compress_bound((1 << 40) + 1) == 0
    assert cc.cccl_compress_bound(1 << 40) > 0


def test_status_strings(cc):
    for code, name in [(0, "CCCL_OK"), (1, "CCCL_ERR_INVALID_ARG"), (2, "CCCL_ERR_CAPACITY"),
                       (3, "CCCL_ERR_CORRUPT"), (4, "CCCL_ERR_TIMEOUT"), (5, "CCCL_ERR_CUDA"),
                       (6, "CCCL_ERR_UNIMPLEMENTED"), (99, "CCCL_ERR_UNKNOWN")]:
        assert cc.cccl_status_string(code) == name


def test_host_side_argument_checks(cc):
    """Errors found before anything is enqueued; none of these touch a GPU."""
    lib = cc._lib
    n = 10 * 4096
    bound, wsb = cc.cccl_compress_bound(n), cc.cccl_workspace_bytes(n)
    A, B, W = 0x10000, 0x20000, 0x30000  # aligned addresses that are never dereferenced
    assert lib.cccl_compress(A, 0, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress(A + 2, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress(A, n, B + 8, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress(A, n, B, bound, W, wsb - 16, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress(A, n, B, bound - 1, W, wsb, None) == cc.CCCL_ERR_CAPACITY
    assert lib.cccl_compress(None, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress(A, (1 << 40) + 1, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_decompress(A, 0, B, n, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_decompress(A, 4096, B, n, W, 8, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_decompress(A, 4096, B + 2, n, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    ptrs = (ctypes.c_void_p * 2)(A, A + 0x1000)
    sizes = (ctypes.c_size_t * 2)(100, 100)
    assert lib.cccl_reduce_compressed(ptrs, sizes, 0, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_compressed(ptrs, sizes, 65, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_compressed(None, sizes, 2, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_compressed(ptrs, sizes, 2, n, B, bound - 1, W, wsb, None) == cc.CCCL_ERR_CAPACITY
    bad = (ctypes.c_void_p * 2)(A, A + 8)
    assert lib.cccl_reduce_compressed(bad, sizes, 2, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_mixed(A, ptrs, sizes, -1, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_mixed(A, ptrs, sizes, 64, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_mixed(A, None, sizes, 2, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_mixed(A + 2, ptrs, sizes, 2, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_mixed(None, None, None, 0, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_mixed(A, ptrs, sizes, 2, 0, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_mixed(A, ptrs, sizes, 2, n, B, bound - 1, W, wsb, None) == cc.CCCL_ERR_CAPACITY
    assert lib.cccl_reduce_mixed(A, ptrs, sizes, 2, n, B, bound, W, wsb - 16, None) == cc.CCCL_ERR_INVALID_ARG
    BE, T = 4 * 4096, 0x40000
    pb = cc.cccl_compress_bound(3 * BE)
    assert lib.cccl_compress_paged(A, 8, BE + 8, T, 3, B, pb, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_paged(A, 8, 0, T, 3, B, pb, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_paged(A, 0, BE, T, 3, B, pb, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_paged(A, 8, BE, T, 0, B, pb, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_paged(A, 8, BE, None, 3, B, pb, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_paged(A, 8, BE, T + 2, 3, B, pb, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_paged(A + 2, 8, BE, T, 3, B, pb, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_decompress_paged(B, 0, A, 8, BE, T, 3, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_decompress_paged(B, 4096, A, 8, BE + 16, T, 3, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_window(A, 0, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_window(A + 2, n, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_window(A, n, B, bound - 1, W, wsb, None) == cc.CCCL_ERR_CAPACITY
    assert lib.cccl_reduce_op(ptrs, sizes, 2, n, 3, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_op(ptrs, sizes, 2, n, -1, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_op(ptrs, sizes, 0, n, 1, B, bound, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    b32 = cc.cccl_compress_bound_typed(3, n)
    assert lib.cccl_compress_typed(4, A, n, B, b32, W, wsb, 0, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_typed(0, A, n, B, b32, W, wsb, 0, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_typed(3, A, 0, B, b32, W, wsb, 0, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_typed(3, A + 4, n, B, b32, W, wsb, 0, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_typed(3, A, n, B, b32, W, wsb - 16, 0, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_compress_typed(3, A, n, B, bound, W, wsb, 0, None) == cc.CCCL_ERR_CAPACITY  # bf16's bound
    assert lib.cccl_compress_typed(2, A, n, B, bound - 1, W, wsb, 1, None) == cc.CCCL_ERR_CAPACITY
    assert lib.cccl_decompress_typed(5, A, 4096, B, n, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_decompress_typed(3, A, 0, B, n, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_decompress_typed(3, A, 4096, B + 8, n, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_decompress_typed(2, A, 4096, B, n, W, 8, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_typed(4, 0, None, ptrs, sizes, 2, n, B, b32, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_typed(3, 3, None, ptrs, sizes, 2, n, B, b32, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_typed(3, 0, None, ptrs, sizes, 0, n, B, b32, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_typed(3, 0, A, ptrs, sizes, 64, n, B, b32, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_typed(3, 0, None, ptrs, sizes, 65, n, B, b32, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_typed(3, 0, None, None, sizes, 2, n, B, b32, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_typed(3, 0, A + 4, ptrs, sizes, 2, n, B, b32, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_reduce_typed(3, 0, None, ptrs, sizes, 2, n, B, b32 - 1, W, wsb, None) == cc.CCCL_ERR_CAPACITY
    assert lib.cccl_reduce_typed(3, 1, None, bad, sizes, 2, n, B, b32, W, wsb, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_get_result(None, None, None, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_get_result(W + 4, None, None, None) == cc.CCCL_ERR_INVALID_ARG


def test_host_pointers_are_refused(cc):
    """Without a device allocation behind them, buffers are refused on the host
    (a kernel is never handed a host address)."""
    n = 4096
    x = np.zeros(n + 16, np.uint16)
    out = np.zeros(cc.cccl_compress_bound(n) + 16, np.uint8)
    ws = np.zeros(cc.cccl_workspace_bytes(n) + 16, np.uint8)
    al = lambda a: (a.ctypes.data + 15) // 16 * 16
    r = cc._lib.cccl_compress(al(x), n, al(out), cc.cccl_compress_bound(n), al(ws), cc.cccl_workspace_bytes(n), None)
    assert r == cc.CCCL_ERR_INVALID_ARG


def test_selftest_timeouts_argument_checks(cc):
    lib = cc._lib
    need = cc.cccl_workspace_bytes(8192)
    ws = np.zeros(need + 16, np.uint8)
    base = (ws.ctypes.data + 15) // 16 * 16
    assert lib.cccl_selftest_timeouts(None, need, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_selftest_timeouts(base + 4, need, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_selftest_timeouts(base, need - 16, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_selftest_timeouts(base, need, None) == cc.CCCL_ERR_INVALID_ARG  # host memory


def test_kernel_set_up_is_kept_per_device(tmp_path):
    """The launchers set a kernel's shared-memory limit through PerDeviceOnce:
    the step runs once for each device (an attribute belongs to the device's
    context), is retried after a failure, and a second device is not taken as
    done because the first one is."""
    import shutil
    import subprocess

    gxx = shutil.which("g++")
    cuda_inc = "/usr/local/cuda/include"
    if gxx is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    src = tmp_path / "once.cpp"
    src.write_text(r'''
#include <cstdio>
#include "cccl_launch.h"
int main() {
    cccl::PerDeviceOnce once;
    int calls[4] = {0, 0, 0, 0};
    auto step = [&](int dev, int slot, cudaError_t result) {
        return (int)once.run(dev, [&] { ++calls[slot]; return result; });
    };
    int r[8];
    r[0] = step(0, 0, cudaSuccess);
    r[1] = step(0, 0, cudaSuccess);           // device 0 is done: not run again
    r[2] = step(1, 1, cudaSuccess);           // device 1 is set up on its own
    r[3] = step(2, 2, cudaErrorInvalidValue); // a failure is returned and not remembered
    r[4] = step(2, 2, cudaSuccess);
    r[5] = step(2, 2, cudaSuccess);
    r[6] = step(70, 3, cudaSuccess);          // beyond 64 devices: run every time
    r[7] = step(70, 3, cudaSuccess);
    std::printf("%d %d %d %d", calls[0], calls[1], calls[2], calls[3]);
    for (int x : r) std::printf(" %d", x);
    std::printf("\n");
    return 0;
}
''')
    exe = tmp_path / "once"
    csrc = os.path.join(ROOT, "compression_coupled_collectives_gb300", "csrc")
    subprocess.check_call([gxx, "-std=c++17", "-I", csrc, "-I", cuda_inc, str(src), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split()
    calls, results = [int(v) for v in out[:4]], [int(v) for v in out[4:]]
    assert calls == [1, 1, 2, 2]
    assert results == [0, 0, 0, 1, 0, 0, 0, 0]  # 1 = cudaErrorInvalidValue


def test_selftest_lookback_argument_checks(cc):
    lib = cc._lib
    n = 100
    sizes = np.zeros(n + 4, np.uint32)
    res = np.zeros(n + 2, np.uint64)
    ws = np.zeros(16 + 8 * n + 16, np.uint8)
    base = (ws.ctypes.data + 15) // 16 * 16
    s_ptr, r_ptr = (sizes.ctypes.data + 3) // 4 * 4, (res.ctypes.data + 7) // 8 * 8
    assert lib.cccl_selftest_lookback(s_ptr, 0, n, 0, r_ptr, base, 16 + 8 * n, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_selftest_lookback(s_ptr, (1 << 20) + 1, n, 0, r_ptr, base, 1 << 30, None) == \
        cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_selftest_lookback(None, n, n, 0, r_ptr, base, 16 + 8 * n, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_selftest_lookback(s_ptr, n, n, 0, r_ptr, base + 4, 16 + 8 * n, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_selftest_lookback(s_ptr, n, n, 0, r_ptr, base, 8 * n, None) == cc.CCCL_ERR_INVALID_ARG
    assert lib.cccl_selftest_lookback(s_ptr, n, n, 0, r_ptr, base, 16 + 8 * n, None) == \
        cc.CCCL_ERR_INVALID_ARG  # host memory
