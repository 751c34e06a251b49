"""pq2_linear_static (include/pq2.h): the allocation-free variant of
pq2_linear for callers that cannot allocate device memory, whose workspace
is a static device array.  Two calls in a row through the C ABI must give
exactly pq2_linear's bits (both run the same kernels in the same order, only
the workspace differs), each within the tolerance the parity tests use
against the oracle, |y - y64| <= 1e-5 * sum_g |s_x s_w dot|, and a warmed-up
call must leave the device's free memory unchanged."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from ternary_weight_int8_gb300 import pq2, synth  # noqa: E402
import gpu_util as U  # noqa: E402

pytestmark = pytest.mark.gpu


def _oracle_bound(x, codes_o, scales_o):
    _, _, _, _, _, y64, bound = U.oracle_reference(x, codes_o, scales_o)
    return y64, bound


@pytest.mark.parametrize("M,N,K", [(3, 1000, 1152), (16, 300, 1024)])
def test_static_matches_linear_twice_in_a_row(M, N, K):
    lib = pq2.lib()
    stream = torch.cuda.current_stream().cuda_stream
    raw, codes_o, scales_o = U.weights(N, K, seed=321 + M)
    codes, scales = pq2.pq2_prepare(raw, K)
    xs = [synth.activations(M, K, seed=900 + M + i, device="cuda", outlier_frac=0.01)
          for i in range(2)]
    ys_static = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in xs]
    ys_linear = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in xs]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # two calls in a row on one stream, no synchronisation between them
    for x, y in zip(xs, ys_static):
        st = lib.pq2_linear_static(x.data_ptr(), pq2.PQ2_BF16, K, M, N, K, codes.data_ptr(),
                                   scales.data_ptr(), y.data_ptr(), pq2.PQ2_F32,
                                   status.data_ptr(), stream)
        assert st == pq2.PQ2_OK, st
    ws = torch.empty(pq2.linear_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    for x, y in zip(xs, ys_linear):
        st = lib.pq2_linear(x.data_ptr(), pq2.PQ2_BF16, K, M, N, K, codes.data_ptr(),
                            scales.data_ptr(), y.data_ptr(), pq2.PQ2_F32, ws.data_ptr(),
                            ws.numel(), status.data_ptr(), stream)
        assert st == pq2.PQ2_OK, st
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for x, ys, yl in zip(xs, ys_static, ys_linear):
        assert torch.equal(ys.view(torch.int32), yl.view(torch.int32))
        y64, bound = _oracle_bound(x, codes_o, scales_o)
        ok, worst = U.O.within_bound(ys.cpu().numpy(), y64, bound)
        assert ok, worst


def test_static_call_allocates_nothing():
    lib = pq2.lib()
    stream = torch.cuda.current_stream().cuda_stream
    M, N, K = 4, 2048, 5120
    raw, _, _ = U.weights(N, K, seed=77)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=78, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def call():
        st = lib.pq2_linear_static(x.data_ptr(), pq2.PQ2_BF16, K, M, N, K, codes.data_ptr(),
                                   scales.data_ptr(), y.data_ptr(), pq2.PQ2_BF16, None, stream)
        assert st == pq2.PQ2_OK, st
        torch.cuda.synchronize()

    call()  # warm-up: the first call on a device looks up the scratch address
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        call()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_static_rejects_shapes_beyond_its_scratch():
    lib = pq2.lib()
    # the largest K whose workspace fits the static scratch at M = 8
    K = 128
    while pq2.linear_workspace_bytes(8, K + 128) <= pq2.PQ2_STATIC_SCRATCH_BYTES:
        K += 128
    big = K + 128
    assert pq2.linear_workspace_bytes(8, big) > pq2.PQ2_STATIC_SCRATCH_BYTES
    x = torch.zeros((8, big), dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros((4, big // 4), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((4, big // 128), dtype=torch.int16, device="cuda")
    y = torch.empty((8, 4), dtype=torch.float32, device="cuda")
    st = lib.pq2_linear_static(x.data_ptr(), pq2.PQ2_BF16, big, 8, 4, big,
                               codes.data_ptr(), scales.data_ptr(), y.data_ptr(), pq2.PQ2_F32,
                               None, torch.cuda.current_stream().cuda_stream)
    assert st == pq2.PQ2_ERR_SHAPE
