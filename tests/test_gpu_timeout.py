"""The bounded device waits, driven to their limit on the GPU without a fault
or a hang: pq2_debug_mmv_drop_arrival runs the small-batch GEMV with one
consumer warp withholding its release of the first ring slot and the
producer's wait for that slot limited to ~10 us.  The wait must give up,
the kernel must record PQ2_ERR_TIMEOUT in the device status and return
promptly (every copy it issued landed first, so nothing outlives the CTA),
and the context must stay usable: a plain pq2_mmv afterwards gives the
same bits as before."""
import time

import pytest
import torch

from ternary_weight_int8_gb300 import pq2, synth
import gpu_util as U

pytestmark = pytest.mark.gpu

# Shapes whose weight pipeline reuses ring slots (the producer waits for a
# release), the first one that the library accepts is used.
SHAPES = [(10240, 5120), (5120, 17408), (2048, 17408)]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pq2.lib()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [1, 4])
def test_dropped_release_times_out_and_returns(M):
    lib = pq2.lib()
    for N, K in SHAPES:
        raw, _, _ = U.weights(N, K, seed=N + K)
        codes, scales = pq2.pq2_prepare(raw, K)
        x = synth.activations(M, K, seed=M, device="cuda")
        q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
        y_ref = pq2.pq2_mmv(q, sx, qs, codes, scales)
        torch.cuda.synchronize()
        y = torch.empty_like(y_ref)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        t0 = time.perf_counter()
        st = lib.pq2_debug_mmv_drop_arrival(q.data_ptr(), sx.data_ptr(), qs.data_ptr(),
                                            codes.data_ptr(), scales.data_ptr(), y.data_ptr(),
                                            pq2.PQ2_F32, M, N, K, 20000, status.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
        if st == pq2.PQ2_ERR_SHAPE:
            continue  # no reused slot at this shape
        assert st == pq2.PQ2_OK
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert int(status.item()) == pq2.PQ2_ERR_TIMEOUT
        assert elapsed < 1.0, elapsed  # the limit, not the ~2 s default, ended it
        # the context is intact and the normal path unchanged
        y2 = pq2.pq2_mmv(q, sx, qs, codes, scales)
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        pq2.pq2_mmv(q, sx, qs, codes, scales, y=y2, status=st2)
        torch.cuda.synchronize()
        assert int(st2.item()) == 0
        assert torch.equal(y2.view(torch.int32), y_ref.view(torch.int32))
        return
    pytest.fail("no configured shape reuses a ring slot")
