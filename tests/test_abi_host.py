"""The C ABI on the host (no GPU needed): the library loads, exports every
function include/pq2.h declares, and rejects invalid arguments before any
CUDA call.  Also the launch geometry of pq2_mmv, which must not depend on M."""
import ctypes
import os
import re

import pytest

from ternary_weight_int8_gb300 import build, pq2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pq2.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(pq2.LIB_PATH):
        build.build()
    return pq2.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pq2_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["pq2_prepare", "pq2_quantize_act", "pq2_mmv", "pq2_mm"]:
        assert required in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert names
    for name in names:
        assert hasattr(L, name), name
        assert name in pq2.SIGNATURES, f"binding lacks {name}"


def test_status_strings_and_sizes(L):
    for s in range(0, 9):
        assert L.pq2_status_string(s)
    assert L.pq2_status_string(12345) == b"unknown status"
    assert L.pq2_layout_version() >= 1
    assert L.pq2_prepared_bytes(17408, 5120) == 17408 * 5120 * 34 // 128
    assert L.pq2_prepared_bytes(10, 100) == 0
    assert L.pq2_prepared_bytes(0, 128) == 0


A = 1 << 20   # a 16-byte aligned fake address: never dereferenced


def test_prepare_validation(L):
    assert L.pq2_prepare(None, 34, 1, 128, A, A, None) == pq2.PQ2_ERR_NULL
    assert L.pq2_prepare(A, 33, 1, 128, A, A, None) == pq2.PQ2_ERR_SHAPE
    assert L.pq2_prepare(A, 34, 0, 128, A, A, None) == pq2.PQ2_ERR_SHAPE
    assert L.pq2_prepare(A, 34, 1, 129, A, A, None) == pq2.PQ2_ERR_SHAPE
    assert L.pq2_prepare(A, 34, 1, 128, A + 8, A, None) == pq2.PQ2_ERR_ALIGN
    assert L.pq2_prepare(A, 34, 1, 128, A, A + 1, None) == pq2.PQ2_ERR_ALIGN


def test_quantize_validation(L):
    f = L.pq2_quantize_act
    assert f(None, 0, 128, 1, 128, A, 1, A, A, None) == pq2.PQ2_ERR_NULL
    assert f(A, 3, 128, 1, 128, A, 1, A, A, None) == pq2.PQ2_ERR_DTYPE
    assert f(A, 0, 128, 1, 128, A, 5, A, A, None) == pq2.PQ2_ERR_DTYPE
    assert f(A, 0, 127, 1, 128, A, 1, A, A, None) == pq2.PQ2_ERR_SHAPE
    assert f(A, 0, 128, 0, 128, A, 1, A, A, None) == pq2.PQ2_ERR_SHAPE
    assert f(A, 0, 256, 1, 192, A, 1, A, A, None) == pq2.PQ2_ERR_SHAPE
    assert f(A + 1, 0, 128, 1, 128, A, 1, A, A, None) == pq2.PQ2_ERR_ALIGN
    assert f(A, 2, 128, 1, 128, A, 1, A + 2, A, None) == pq2.PQ2_ERR_ALIGN
    assert f(A, 0, 128, 1, 128, A + 4, 1, A, A, None) == pq2.PQ2_ERR_ALIGN


def test_mmv_validation(L):
    f = L.pq2_mmv
    ok = [A, A, A, A, A, A, pq2.PQ2_F32, 1, 10, 128, None, None]
    for i in range(6):
        bad = list(ok); bad[i] = None
        assert f(*bad) == pq2.PQ2_ERR_NULL
    for idx, val, err in [(7, 0, pq2.PQ2_ERR_SHAPE), (7, 9, pq2.PQ2_ERR_SHAPE),
                          (8, 0, pq2.PQ2_ERR_SHAPE), (9, 64, pq2.PQ2_ERR_SHAPE),
                          (6, pq2.PQ2_F16, pq2.PQ2_ERR_DTYPE), (0, A + 4, pq2.PQ2_ERR_ALIGN),
                          (3, A + 8, pq2.PQ2_ERR_ALIGN), (1, A + 2, pq2.PQ2_ERR_ALIGN),
                          (4, A + 1, pq2.PQ2_ERR_ALIGN), (5, A + 2, pq2.PQ2_ERR_ALIGN)]:
        bad = list(ok); bad[idx] = val
        assert f(*bad) == err, (idx, val)
    ex = ok[:10] + [5, 0] + ok[10:]
    assert L.pq2_mmv_ex(*ex) == pq2.PQ2_ERR_DTYPE
    ex = ok[:10] + [pq2.PQ2_DECODE_PLANES, 8] + ok[10:]
    assert L.pq2_mmv_ex(*ex) == pq2.PQ2_ERR_DTYPE


def test_linear_validation(L):
    f = L.pq2_linear
    ws = L.pq2_linear_workspace_bytes(4, 5120)
    assert ws >= 4 * 5120 + 2 * 4 * 40 * 4 and ws % 4 == 0
    assert L.pq2_linear_workspace_bytes(0, 5120) == 0
    assert L.pq2_linear_workspace_bytes(4, 100) == 0
    ok = [A, pq2.PQ2_BF16, 5120, 4, 64, 5120, A, A, A, pq2.PQ2_F32, A, ws, None, None]
    for i in (0, 6, 7, 8, 10):
        bad = list(ok); bad[i] = None
        assert f(*bad) == pq2.PQ2_ERR_NULL, i
    for idx, val, err in [(3, (1 << 20) + 1, pq2.PQ2_ERR_SHAPE), (3, 0, pq2.PQ2_ERR_SHAPE),
                          (2, 5000, pq2.PQ2_ERR_SHAPE), (11, ws - 1, pq2.PQ2_ERR_SHAPE),
                          (1, 9, pq2.PQ2_ERR_DTYPE), (9, pq2.PQ2_F16, pq2.PQ2_ERR_DTYPE),
                          (10, A + 16, pq2.PQ2_ERR_ALIGN), (6, A + 8, pq2.PQ2_ERR_ALIGN),
                          (0, A + 1, pq2.PQ2_ERR_ALIGN)]:
        bad = list(ok); bad[idx] = val
        assert f(*bad) == err, (idx, val)


def test_mm_and_debug_validation(L):
    assert L.pq2_mm(A, A, A, A, A, A, 2, 0, 10, 128, None, None) == pq2.PQ2_ERR_SHAPE
    assert L.pq2_mm(A, A, A, A, A, A, 2, (1 << 20) + 1, 10, 128, None, None) == pq2.PQ2_ERR_SHAPE
    assert L.pq2_mm(A, A, A, A, A, None, 2, 16, 10, 128, None, None) == pq2.PQ2_ERR_NULL
    assert L.pq2_mm(A, A, None, A, A, A, 2, 16, 10, 128, None, None) == pq2.PQ2_ERR_NULL
    assert L.pq2_mm(A + 2, A, A, A, A, A, 2, 16, 10, 128, None, None) == pq2.PQ2_ERR_ALIGN
    assert L.pq2_debug_group_dots(A, None, A, 16, 10, 128, 1, A, None, None) == pq2.PQ2_ERR_NULL
    d = L.pq2_debug_group_dots
    assert d(A, None, A, 1, 10, 128, 7, A, None, None) == pq2.PQ2_ERR_DTYPE
    assert d(A, None, A, 1, 10, 128, 2, A, None, None) == pq2.PQ2_ERR_NULL
    assert d(A, A, A, 9, 10, 128, 0, A, None, None) == pq2.PQ2_ERR_SHAPE
    assert d(A, A, A, 0, 10, 128, 1, A, None, None) == pq2.PQ2_ERR_SHAPE


def test_valid_call_without_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert L.pq2_mmv(A, A, A, A, A, A, pq2.PQ2_F32, 1, 10, 128, None, None) in (
        pq2.PQ2_ERR_CUDA, pq2.PQ2_ERR_ARCH)


@pytest.mark.parametrize("N,K", [(14336, 4096), (10240, 5120), (17408, 5120), (5120, 17408),
                                 (6144, 5120), (5, 384), (1, 128), (100000, 1024),
                                 (153, 17408)])
@pytest.mark.parametrize("sms", [152, 148, 8])
def test_mmv_geometry(L, N, K, sms):
    ctas, threads, splits, rows_max = pq2.mmv_geometry(N, K, sms)
    G = K // 128
    assert 1 <= ctas and rows_max == -(-N // ctas)
    assert ctas <= max(sms, -(-N // 256)) and rows_max <= 256
    assert threads % 32 == 0 and 32 <= threads <= 288
    # each consumer thread owns two rows of one split
    pairs = -(-rows_max // 2)
    assert pairs * splits <= threads < pairs * splits + 32
    # a row's splits share one warp: S is a power of two dividing 32
    assert 1 <= splits <= min(G, 16) and 32 % splits == 0
    # every row is covered: the CTA row ranges tile [0, N)
    bounds = [N * c // ctas for c in range(ctas + 1)]
    assert bounds[0] == 0 and bounds[-1] == N
    assert max(b - a for a, b in zip(bounds, bounds[1:])) == rows_max


def test_mmv_geometry_fills_the_gb300_shapes(L):
    """On 152 SMs the configured projection shapes keep >= 87% of the
    consumer lanes (two rows each) and steps busy."""
    for N, K in [(14336, 4096), (10240, 5120), (17408, 5120), (5120, 17408), (6144, 5120)]:
        ctas, threads, splits, R = pq2.mmv_geometry(N, K, 152)
        G = K // 128
        steps = -(-G // splits)
        eff = (-(-R // 2) * splits / threads) * (G / (splits * steps))
        assert ctas == 152 and eff >= 0.87, (N, K, eff)


def test_mm_f8_validation(L):
    f = L.pq2_mm_f8
    assert f(A, A, A, A, A, A, 2, 0, 10, 128, None, None) == pq2.PQ2_ERR_SHAPE
    assert f(None, A, A, A, A, A, 2, 16, 10, 128, None, None) == pq2.PQ2_ERR_NULL
    assert f(A, A, None, A, A, A, 2, 16, 10, 128, None, None) == pq2.PQ2_ERR_NULL
    assert f(A, A, A, A, A, A, 1, 16, 10, 128, None, None) == pq2.PQ2_ERR_DTYPE
    assert f(A + 8, A, A, A, A, A, 2, 16, 10, 128, None, None) == pq2.PQ2_ERR_ALIGN
    assert f(A, A, A, A, A, A, 2, 16, 10, 200, None, None) == pq2.PQ2_ERR_SHAPE
    d = L.pq2_debug_group_dots
    assert d(A, None, A, 16, 10, 128, pq2.PQ2_PATH_MM_F8, A, None, None) == pq2.PQ2_ERR_NULL
    assert d(A, A, A, 0, 10, 128, pq2.PQ2_PATH_MM_F8, A, None, None) == pq2.PQ2_ERR_SHAPE
    assert d(A, A, A, 16, 10, 128, 5, A, None, None) == pq2.PQ2_ERR_DTYPE
    # the tensor-core GEMV path takes M = 1..8 and its corrections
    assert d(A, A, A, 16, 10, 128, pq2.PQ2_PATH_MMV_TC, A, None, None) == pq2.PQ2_ERR_SHAPE
    assert d(A, None, A, 4, 10, 128, pq2.PQ2_PATH_MMV_TC, A, None, None) == pq2.PQ2_ERR_NULL


def test_grouped_validation(L):
    q = L.pq2_quantize_act_grouped
    ok = [A, pq2.PQ2_BF16, 256, 2, 256, 32, A, pq2.PQ2_Q_PLANES, A, A, None]
    for idx, val, err in [(5, 16, pq2.PQ2_ERR_SHAPE), (5, 96, pq2.PQ2_ERR_SHAPE),
                          (7, 5, pq2.PQ2_ERR_DTYPE), (1, 9, pq2.PQ2_ERR_DTYPE),
                          (7, pq2.PQ2_Q_MMV16, pq2.PQ2_ERR_SHAPE),
                          (6, None, pq2.PQ2_ERR_NULL), (0, None, pq2.PQ2_ERR_NULL),
                          (6, A + 4, pq2.PQ2_ERR_ALIGN), (4, 200, pq2.PQ2_ERR_SHAPE)]:
        bad = list(ok); bad[idx] = val
        assert q(*bad) == err, (idx, val)
    m = L.pq2_mmv_grouped
    ok = [A, A, A, A, A, A, pq2.PQ2_F32, 4, 10, 256, 32, 0, None, None]
    for idx, val, err in [(7, 9, pq2.PQ2_ERR_SHAPE), (10, 16, pq2.PQ2_ERR_SHAPE),
                          (11, 8, pq2.PQ2_ERR_DTYPE), (2, None, pq2.PQ2_ERR_NULL),
                          (3, A + 8, pq2.PQ2_ERR_ALIGN)]:
        bad = list(ok); bad[idx] = val
        assert m(*bad) == err, (idx, val)


def test_mm_grouped_validation(L):
    for f in (L.pq2_mm_grouped, L.pq2_mm_f8_grouped):
        ok = [A, A, A, A, A, A, pq2.PQ2_F32, 16, 10, 256, 64, None, None]
        for idx, val, err in [(10, 16, pq2.PQ2_ERR_SHAPE), (10, 96, pq2.PQ2_ERR_SHAPE),
                              (7, 0, pq2.PQ2_ERR_SHAPE), (9, 200, pq2.PQ2_ERR_SHAPE),
                              (6, 1, pq2.PQ2_ERR_DTYPE), (0, None, pq2.PQ2_ERR_NULL),
                              (2, None, pq2.PQ2_ERR_NULL), (0, A + 8, pq2.PQ2_ERR_ALIGN),
                              (4, A + 1, pq2.PQ2_ERR_ALIGN)]:
            bad = list(ok); bad[idx] = val
            assert f(*bad) == err, (f, idx, val)
    d = L.pq2_debug_mm_dots_grouped
    ok = [A, pq2.PQ2_PATH_MM_F8, A, 16, 10, 256, 32, A, None, None]
    for idx, val, err in [(1, pq2.PQ2_PATH_MMV_PLANES, pq2.PQ2_ERR_DTYPE),
                          (6, 128 + 32, pq2.PQ2_ERR_SHAPE), (3, 0, pq2.PQ2_ERR_SHAPE),
                          (7, None, pq2.PQ2_ERR_NULL), (7, A + 2, pq2.PQ2_ERR_ALIGN)]:
        bad = list(ok); bad[idx] = val
        assert d(*bad) == err, (idx, val)


def test_linear_grouped_validation(L):
    wb = L.pq2_linear_grouped_workspace_bytes
    # q (int8 planes up to M = 8, two e4m3 planes from M = 9), s_x, sum(q)
    assert wb(4, 256, 32) == 4 * 256 + 256 + 4 * 8 * 4
    assert wb(9, 256, 64) == 9 * 512 + 256 + 9 * 4 * 4
    assert wb(4, 256, 16) == 0 and wb(0, 256, 32) == 0 and wb(4, 200, 32) == 0
    f = L.pq2_linear_grouped
    need = wb(16, 256, 64)
    ok = [A, pq2.PQ2_BF16, 256, 16, 10, 256, A, A, 64, A, pq2.PQ2_F32, A, need, None, None]
    for idx, val, err in [(8, 16, pq2.PQ2_ERR_SHAPE), (12, need - 1, pq2.PQ2_ERR_SHAPE),
                          (2, 255, pq2.PQ2_ERR_SHAPE), (1, 7, pq2.PQ2_ERR_DTYPE),
                          (10, pq2.PQ2_F16, pq2.PQ2_ERR_DTYPE), (11, None, pq2.PQ2_ERR_NULL),
                          (11, A + 16, pq2.PQ2_ERR_ALIGN), (6, A + 4, pq2.PQ2_ERR_ALIGN)]:
        bad = list(ok); bad[idx] = val
        assert f(*bad) == err, (idx, val)


def test_ptq_validation(L):
    p = L.pq2_ptq_prepare
    assert p(A, 56, 1, 384, A, A, None) == pq2.PQ2_ERR_SHAPE       # K % 256
    assert p(A, 55, 1, 256, A, A, None) == pq2.PQ2_ERR_SHAPE       # row stride < 28 K/128
    assert p(None, 56, 1, 256, A, A, None) == pq2.PQ2_ERR_NULL
    assert p(A, 56, 1, 256, A + 8, A, None) == pq2.PQ2_ERR_ALIGN
    assert p(A, 56, 1, 256, A, A + 4, None) == pq2.PQ2_ERR_ALIGN
    m = L.pq2_ptq_mmv
    ok = [A, A, A, A, A, A, pq2.PQ2_F32, 4, 10, 512, 32, 0, None]
    for idx, val, err in [(7, 5, pq2.PQ2_ERR_SHAPE), (9, 384, pq2.PQ2_ERR_SHAPE),
                          (10, 16, pq2.PQ2_ERR_SHAPE), (11, 8, pq2.PQ2_ERR_DTYPE),
                          (6, pq2.PQ2_F16, pq2.PQ2_ERR_DTYPE), (2, None, pq2.PQ2_ERR_NULL),
                          (1, None, pq2.PQ2_ERR_NULL), (3, A + 8, pq2.PQ2_ERR_ALIGN),
                          (4, A + 4, pq2.PQ2_ERR_ALIGN)]:
        bad = list(ok); bad[idx] = val
        assert m(*bad) == err, (idx, val)
    wsb = L.pq2_ptq_linear_workspace_bytes
    n = wsb(4, 512, 32)
    assert n >= 4 * 512 + 2 * 4 * 16 * 4
    assert wsb(5, 512, 32) == 0 and wsb(4, 384, 32) == 0 and wsb(4, 512, 16) == 0
    lin = L.pq2_ptq_linear
    ok = [A, pq2.PQ2_BF16, 512, 4, 10, 512, A, A, 32, A, pq2.PQ2_F32, A, n, None]
    for idx, val, err in [(12, n - 1, pq2.PQ2_ERR_SHAPE), (3, 5, pq2.PQ2_ERR_SHAPE),
                          (2, 500, pq2.PQ2_ERR_SHAPE), (1, 9, pq2.PQ2_ERR_DTYPE),
                          (11, A + 64, pq2.PQ2_ERR_ALIGN), (0, None, pq2.PQ2_ERR_NULL)]:
        bad = list(ok); bad[idx] = val
        assert lin(*bad) == err, (idx, val)
    d = L.pq2_debug_ptq_dots
    assert d(A, A, A, A, 5, 10, 512, 32, A, None) == pq2.PQ2_ERR_SHAPE
    assert d(A, A, A, A, 4, 10, 512, 32, None, None) == pq2.PQ2_ERR_NULL


def test_drop_arrival_validation(L):
    """The bounded-wait test entry: a device status is required and the wait
    limit must lie in 1000 .. 2^32 clocks; all rejected before any CUDA call."""
    f = L.pq2_debug_mmv_drop_arrival
    ok = [A, A, A, A, A, A, pq2.PQ2_F32, 1, 10, 128, 20000, A, None]
    bad = list(ok)
    bad[11] = None
    assert f(*bad) == pq2.PQ2_ERR_NULL
    for lim in (0, 999, (1 << 32) + 1):
        bad = list(ok)
        bad[10] = lim
        assert f(*bad) == pq2.PQ2_ERR_SHAPE, lim
    bad = list(ok)
    bad[11] = A + 2
    assert f(*bad) == pq2.PQ2_ERR_ALIGN
    bad = list(ok)
    bad[7] = 9
    assert f(*bad) == pq2.PQ2_ERR_SHAPE
    bad = list(ok)
    bad[0] = None
    assert f(*bad) == pq2.PQ2_ERR_NULL


def test_linear_static_error_order(L):
    """pq2_linear_static reports errors in pq2_linear's order: a bad dtype
    before an oversized shape, before any CUDA call."""
    f = L.pq2_linear_static
    big = 123392  # M = 8 needs more than the static scratch at this K
    assert f(A, 7, big, 8, 4, big, A, A, A, pq2.PQ2_F32, None, None) == pq2.PQ2_ERR_DTYPE
    assert f(A, pq2.PQ2_BF16, big, 8, 4, big, A, A, A, 9, None, None) == pq2.PQ2_ERR_DTYPE
    assert f(A, pq2.PQ2_BF16, big, 8, 4, big, A, A, A, pq2.PQ2_F32, None, None) == \
        pq2.PQ2_ERR_SHAPE
    assert f(None, pq2.PQ2_BF16, 128, 1, 4, 128, A, A, A, pq2.PQ2_F32, None, None) == \
        pq2.PQ2_ERR_NULL


def test_mmv_tc_validation(L):
    """pq2_mmv_tc rejects what pq2_mmv_ex rejects, before any CUDA call."""
    f = L.pq2_mmv_tc
    ok = [A, A, A, A, A, A, pq2.PQ2_F32, 4, 10, 128, 0, None, None]
    for idx, val, err in [(0, None, pq2.PQ2_ERR_NULL), (2, None, pq2.PQ2_ERR_NULL),
                          (7, 9, pq2.PQ2_ERR_SHAPE), (7, 0, pq2.PQ2_ERR_SHAPE),
                          (9, 200, pq2.PQ2_ERR_SHAPE), (6, 1, pq2.PQ2_ERR_DTYPE),
                          (10, 4, pq2.PQ2_ERR_DTYPE), (0, A + 8, pq2.PQ2_ERR_ALIGN),
                          (5, A + 2, pq2.PQ2_ERR_ALIGN)]:
        bad = list(ok); bad[idx] = val
        assert f(*bad) == err, (idx, val)
    # the GEMV choice of pq2_linear: dp4a for M <= 4, tensor cores from M = 6,
    # at M = 5 only for slabs of at most 72 rows in at most 8 splits
    for M in range(1, 5):
        assert L.pq2_linear_tensor_gemv(M, 10240, 5120, 152) == 0
    for M in range(6, 9):
        for N, K in [(10240, 5120), (17408, 5120), (5120, 17408), (6144, 5120)]:
            assert L.pq2_linear_tensor_gemv(M, N, K, 152) == 1
    assert L.pq2_linear_tensor_gemv(5, 10240, 5120, 152) == 1   # 68 rows, 8 splits
    assert L.pq2_linear_tensor_gemv(5, 6144, 5120, 152) == 1    # 41 rows, 8 splits
    assert L.pq2_linear_tensor_gemv(5, 17408, 5120, 152) == 0   # 115 rows
    assert L.pq2_linear_tensor_gemv(5, 5120, 17408, 152) == 0   # 16 splits
    assert L.pq2_linear_tensor_gemv(16, 10240, 5120, 152) == 0
    assert L.pq2_linear_tensor_gemv(9, 10240, 5120, 152) == 0
