"""tcgen05 self-check: the library's shared-memory operand layouts, MMA issue and
TMEM read-back against a reference matrix product (bf16 in, fp32 out)."""

import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_delta_rule_06_gb300 import build, ops

    build.build()
    L = ops.load_library()
    L.gdn_selftest_mma.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p] * 4
    L.gdn_selftest_mma.restype = ctypes.c_int
    L.gdn_selftest_mma_m64_rows.argtypes = [ctypes.c_int] * 2 + [ctypes.c_void_p] * 4
    L.gdn_selftest_mma_m64_rows.restype = ctypes.c_int
    L.gdn_selftest_mma_tmem_a.argtypes = [ctypes.c_int] * 3 + [ctypes.c_void_p] * 4
    L.gdn_selftest_mma_tmem_a.restype = ctypes.c_int
    L.gdn_selftest_tma_tile.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int] * 5 + [ctypes.c_void_p] * 3
    L.gdn_selftest_tma_tile.restype = ctypes.c_int
    L.gdn_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    L.gdn_device_error.restype = ctypes.c_int
    return L


def _run(lib, M, N, K, amn, bmn, seed=0):
    g = torch.Generator().manual_seed(seed + M + N + K)
    A = torch.randn((M, K), generator=g).to(torch.bfloat16).cuda()
    B = torch.randn((K, N), generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    rc = lib.gdn_selftest_mma(M, N, K, amn, bmn, ctypes.c_void_p(A.data_ptr()),
                              ctypes.c_void_p(B.data_ptr()), ctypes.c_void_p(D.data_ptr()),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    ref = A.float() @ B.float()
    return D, ref


def _lanes_m64():
    # accumulator row r of an M = 64 MMA sits in TMEM lane 32 * (r // 16) + r % 16
    return torch.tensor([32 * (r // 16) + r % 16 for r in range(64)])


@pytest.mark.parametrize("amn", [0, 1])
@pytest.mark.parametrize("bmn", [0, 1])
@pytest.mark.parametrize("N,K", [(64, 16), (64, 192), (128, 64), (192, 128), (256, 32)])
def test_m128(lib, amn, bmn, N, K):
    D, ref = _run(lib, 128, N, K, amn, bmn)
    torch.testing.assert_close(D, ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("amn", [0, 1])
@pytest.mark.parametrize("bmn", [0, 1])
@pytest.mark.parametrize("N,K", [(64, 64), (192, 32), (128, 16)])
def test_m64_lane_placement(lib, amn, bmn, N, K):
    D, ref = _run(lib, 64, N, K, amn, bmn)
    got = D[_lanes_m64().cuda()]
    torch.testing.assert_close(got, ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("N,K", [(32, 16), (64, 64), (192, 128), (256, 32)])
def test_m64_rows_16x32bx2(lib, N, K):
    # thread t < 16 of warp w holds row 16 (w % 4) + t, columns c .. c + 15;
    # thread t + 16 the same row at columns c + 16 .. c + 31
    g = torch.Generator().manual_seed(3 + N + K)
    A = torch.randn((64, K), generator=g).to(torch.bfloat16).cuda()
    B = torch.randn((K, N), generator=g).to(torch.bfloat16).cuda()
    D = torch.full((64, N), float("nan"), device="cuda")
    rc = lib.gdn_selftest_mma_m64_rows(N, K, ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
                                       ctypes.c_void_p(D.data_ptr()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    torch.testing.assert_close(D, -(A.float() @ B.float()), rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("bmn", [0, 1])
@pytest.mark.parametrize("N,K", [(64, 32), (64, 192), (192, 64), (128, 256)])
def test_a_from_tmem(lib, bmn, N, K):
    g = torch.Generator().manual_seed(7 + N + K)
    A = torch.randn((128, K), generator=g).to(torch.bfloat16).cuda()
    B = torch.randn((K, N), generator=g).to(torch.bfloat16).cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    rc = lib.gdn_selftest_mma_tmem_a(N, K, bmn, ctypes.c_void_p(A.data_ptr()),
                                     ctypes.c_void_p(B.data_ptr()), ctypes.c_void_p(D.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    torch.testing.assert_close(D, A.float() @ B.float(), rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("B,T,H,D,cols,b,t0,h,xg0", [
    (2, 200, 3, 192, 192, 1, 128, 2, 0),   # full width, ragged last tile (rows 200.. zero)
    (1, 64, 1, 64, 64, 0, 0, 0, 0),
    (2, 130, 4, 256, 128, 0, 64, 3, 16),   # column sub-tile starting at column 128
    (1, 300, 2, 128, 128, 0, 256, 1, 0),   # 44 valid rows
])
def test_tma_row_tile(lib, B, T, H, D, cols, b, t0, h, xg0):
    g = torch.Generator().manual_seed(B * T + D)
    x = torch.randn((B, T, H, D), generator=g).to(torch.bfloat16).cuda()
    out = torch.full((64 * cols,), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.gdn_selftest_tma_tile(B, T, H, D, cols, b, t0, h, xg0, ctypes.c_void_p(x.data_ptr()),
                                   ctypes.c_void_p(out.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    rows = torch.zeros((64, cols), dtype=torch.bfloat16)
    nv = max(0, min(64, T - t0))
    rows[:nv] = x[b, t0:t0 + nv, h, 8 * xg0:8 * xg0 + cols].cpu()
    # panel layout: [column group][row][8 elements]
    want = rows.reshape(64, cols // 8, 8).permute(1, 0, 2).reshape(-1)
    assert torch.equal(out.cpu(), want)


def test_no_wait_timeouts(lib):
    flag = ctypes.c_uint(123)
    assert lib.gdn_device_error(ctypes.byref(flag)) == 0
    assert flag.value == 0


@pytest.mark.parametrize("mode", [0, 1])
def test_bounded_wait_gives_up_and_reports(lib, mode):
    """A wait that nothing completes (mode 0: an mbarrier phase; mode 1: a
    progress word left at 0) gives up after its limit (1 ms here): the kernel
    returns, the timeout bit of the device error word is set and then cleared
    by reading it, the kernel freed its tensor memory before returning, and the
    next launches run normally."""
    import time

    from gated_delta_rule_06_gb300 import workloads as wl
    from parity_util import TOL, check, gpu_backward, gpu_forward, oracle_backward, \
        oracle_forward, to_dev

    lib.gdn_selftest_wait_timeout.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]
    lib.gdn_selftest_wait_timeout.restype = ctypes.c_int
    flag = ctypes.c_uint(123)
    assert lib.gdn_device_error(ctypes.byref(flag)) == 0 and flag.value == 0
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.gdn_selftest_wait_timeout(mode, 1_000_000, ctypes.c_void_p(word.data_ptr()),
                                       ctypes.c_void_p(out.data_ptr()), stream)
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 0.5, elapsed  # 1 ms limit (plus launch): far below the kernels' 1 s
    assert out.tolist() == [0, 1]  # gave up; tensor memory freed before returning
    assert lib.gdn_device_error(ctypes.byref(flag)) == 0
    assert flag.value & 1, flag.value
    assert lib.gdn_device_error(ctypes.byref(flag)) == 0 and flag.value == 0  # cleared
    # bad arguments are refused before any launch
    assert lib.gdn_selftest_wait_timeout(2, 1_000_000, None, ctypes.c_void_p(out.data_ptr()),
                                         stream) != 0
    assert lib.gdn_selftest_wait_timeout(0, 10 ** 10, None, ctypes.c_void_p(out.data_ptr()),
                                         stream) != 0
    # the context is intact: the tensor-core self-check and a forward + backward pass
    D, ref = _run(lib, 128, 64, 64, 0, 0, seed=5)
    torch.testing.assert_close(D, ref, rtol=1e-5, atol=1e-4)
    w = wl.custom("after_timeout", 1, 130, 2, 4, 64, 64, dtype=torch.bfloat16, seed=41)
    x = wl.make_inputs(w)
    xd = to_dev(x)
    o, sT, saved = gpu_forward(xd)
    g = gpu_backward(xd, saved)
    torch.cuda.synchronize()
    o_r, _ = oracle_forward(x)
    check("o", o, o_r, TOL[torch.bfloat16])
    gr = oracle_backward(x)
    check("dk", g["dk"], gr["dk"], TOL[torch.bfloat16])
    assert lib.gdn_device_error(ctypes.byref(flag)) == 0 and flag.value == 0
