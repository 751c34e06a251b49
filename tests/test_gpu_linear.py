"""pq2_linear for M = 1..8 (quantisation, then the GEMV streaming its
weights meanwhile) against the same two steps called one by one: the same
bits for every activation type, row stride and alignment, degenerate
groups and chains of dependent calls; and against the oracle's bound.
Quantisation of quotients on and near half-integers against the oracle."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from ternary_weight_int8_gb300 import pq2, synth
import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pq2.lib()
    yield
    torch.cuda.synchronize()


def _weights(N, K, seed):
    return pq2.pq2_prepare(synth.raw_weights(N, K, seed=seed, device="cuda"), K)


def _two_kernel(x, codes, scales, out_dtype=torch.float32):
    q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
    return pq2.pq2_mmv(q, sx, qs, codes, scales, out_dtype=out_dtype)


def _x(M, K, dtype, seed, ld_pad=0, offset=0):
    """Activations [M][K] of `dtype` inside a [M][K + ld_pad + offset] buffer,
    starting `offset` elements in (offset 1 defeats vector loads)."""
    base = synth.activations(M, K, seed=seed, device="cuda", outlier_frac=0.01).to(dtype)
    buf = torch.zeros((M, K + ld_pad + offset), dtype=dtype, device="cuda")
    buf[:, offset:offset + K] = base
    return buf[:, offset:offset + K]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("M,N,K,ld_pad,offset", [
    (1, 10240, 5120, 0, 0), (4, 10240, 5120, 0, 0), (8, 10240, 5120, 0, 0),
    (3, 1000, 1152, 5, 0), (5, 333, 384, 0, 1), (2, 7, 128, 3, 1), (1, 5120, 17408, 0, 0),
    (6, 152, 640, 8, 0),
])
def test_linear_matches_two_kernels(dtype, M, N, K, ld_pad, offset):
    codes, scales = _weights(N, K, seed=N + 17 * M)
    x = _x(M, K, dtype, seed=M + K, ld_pad=ld_pad, offset=offset)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_lin = pq2.pq2_linear(x, codes, scales, status=status)
    y_lin_b = pq2.pq2_linear(x, codes, scales, out_dtype=torch.bfloat16)
    y_two = _two_kernel(x, codes, scales)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(y_lin.view(torch.int32), y_two.view(torch.int32))
    assert torch.equal(y_lin_b.view(torch.int16), y_two.to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("M", [1, 4, 8])
def test_linear_against_oracle(M):
    N, K = 1000, 4096
    raw, codes_o, scales_o = U.weights(N, K, seed=77 + M)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=500 + M, device="cuda", outlier_frac=0.01)
    y = pq2.pq2_linear(x, codes, scales)
    torch.cuda.synchronize()
    _, _, _, _, _, y64, bound = U.oracle_reference(x, codes_o, scales_o)
    diff = np.abs(y.cpu().numpy().astype(np.float64) - y64)
    assert np.all(diff <= 1e-5 * bound), float((diff - 1e-5 * bound).max())


@pytest.mark.parametrize("M", [9, 12, 15])
def test_linear_between_gemv_and_prefill_sizes(M):
    """M = 9..15 run the prefill GEMM's 8-bit path as one partial token tile:
    bit-identical to quantising to PQ2_Q_F8 and calling pq2_mm_f8, and within
    the oracle's bound."""
    N, K = 1000, 4096
    raw, codes_o, scales_o = U.weights(N, K, seed=91 + M)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=600 + M, device="cuda", outlier_frac=0.01)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = pq2.pq2_linear(x, codes, scales, status=status)
    q8, sx8, qs8 = pq2.pq2_quantize_act(x, pq2.PQ2_Q_F8)
    y_two = pq2.pq2_mm_f8(q8, sx8, qs8, codes, scales)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(y.view(torch.int32), y_two.view(torch.int32))
    _, _, _, _, _, y64, bound = U.oracle_reference(x, codes_o, scales_o)
    diff = np.abs(y.cpu().numpy().astype(np.float64) - y64)
    assert np.all(diff <= 1e-5 * bound), float((diff - 1e-5 * bound).max())


def test_all_zero_and_single_outlier_groups():
    """Degenerate groups: all zeros (s = 0, q = 0) and one large value among
    zeros (q = +-127 there, 0 elsewhere)."""
    M, N, K = 3, 500, 1024
    codes, scales = _weights(N, K, seed=5)
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    x[1, 200] = 3.0e4
    x[2, 7] = -1.0e-30
    x[2, 900:1024] = 0.5
    y_lin = pq2.pq2_linear(x, codes, scales)
    y_two = _two_kernel(x, codes, scales)
    torch.cuda.synchronize()
    assert torch.equal(y_lin.view(torch.int32), y_two.view(torch.int32))
    assert torch.count_nonzero(y_lin[0]) == 0


def test_chain_fp32_each_call_reads_previous_output():
    """Calls whose x is the previous call's fp32 y, launched back to back,
    match the same chain of separate quantise and GEMV calls."""
    K = 2048
    mats = [_weights(K, K, seed=40 + i) for i in range(3)]
    x0 = synth.activations(4, K, seed=9, device="cuda").float()

    def chain(step):
        x = x0
        for c, sc in mats * 4:
            x = step(x, c, sc)
        torch.cuda.synchronize()
        return x

    a = chain(lambda x, c, sc: pq2.pq2_linear(x, c, sc))
    b = chain(lambda x, c, sc: _two_kernel(x, c, sc))
    assert torch.isfinite(a).all()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quotients_at_and_near_half_integers(dtype):
    """Groups whose a / s fall on or within 3e-5 of half-integers, where
    round-half-to-even and the last bit of the quotient decide q: q, s_x and
    sum(q) bit-exact against the oracle."""
    M, K = 4, 2048
    G = K // 128
    gen = torch.Generator().manual_seed(5)
    x = torch.empty((M, K), dtype=torch.float32)
    for m in range(M):
        for g in range(G):
            s = 1.0 if m == 0 else float(torch.rand(1, generator=gen)) * 4 + 1e-3
            k = torch.randint(-127, 127, (128,), generator=gen).float()
            delta = (torch.rand(128, generator=gen) - 0.5) * 6e-5 * (m - 1 if m > 1 else 0)
            v = (k + 0.5 + delta) * s
            v[0] = 127.0 * s  # the group maximum: s_x = 127 s / 127
            x[m, g * 128:(g + 1) * 128] = v
    x = x.to(dtype)
    q_o, sx_o = O.quantize(O.widen(U.x_bits(x), U.kind(x)))
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_ROWS)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_o.view(np.uint32))
    assert np.array_equal(qs.cpu().numpy(), O.qsum(q_o))


@pytest.mark.parametrize("M", [1, 3, 8, 48])
def test_linear_on_mapped_host_buffers(M):
    """pq2_linear reading x from, and writing y to, pinned host memory the
    device addresses directly: bit-identical to the same call on device
    buffers (GEMV for M <= 8, the 8-bit prefill path above)."""
    N, K = 1000, 2048
    raw = synth.raw_weights(N, K, seed=M + 1, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M, outlier_frac=0.01)
    hx = x.pin_memory()
    hy = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    if not (U.host_mapped(hx) and U.host_mapped(hy)):
        pytest.skip("pinned host memory is not device-addressable here")
    lib = pq2.lib()
    ws = torch.empty(pq2.linear_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = lib.pq2_linear(hx.data_ptr(), pq2.PQ2_BF16, K, M, N, K, codes.data_ptr(),
                        scales.data_ptr(), hy.data_ptr(), pq2.PQ2_BF16, ws.data_ptr(), ws.numel(),
                        status.data_ptr(), None)
    assert st == pq2.PQ2_OK
    yd = pq2.linear(x.cuda(), codes, scales, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(hy.view(torch.int16), yd.cpu().view(torch.int16))
