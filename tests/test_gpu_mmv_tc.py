"""The small-batch GEMV on the legacy tensor-core path (pq2_mmv_tc, mma.sync
with fp16 operands) through the C ABI: the quantiser's PQ2_Q_MMV16 bytes and
corrections against an independent host construction of the documented
layout; the per-group dots bit-exact against the oracle (the extremes
included); y bit-identical to the dp4a GEMV pq2_mmv for every M = 1..8, both
output types and every call flag (same split, same fp32 order), hence within
the bound and batch invariant; pq2_linear's tensor-core M bit-identical to
quantise + pq2_mmv."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from ternary_weight_int8_gb300 import pq2, synth
import gpu_util as U

pytestmark = pytest.mark.gpu
G = 128


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pq2.lib()
    yield
    torch.cuda.synchronize()


# (N, K): ragged slabs, every split count the geometry picks (S = 1..16), the
# four layer shapes and 4096 x 14336
SHAPES = [(1, 128), (7, 256), (300, 1152), (1000, 640), (2048, 17408), (10240, 5120),
          (6144, 5120), (17408, 5120), (5120, 17408), (14336, 4096)]


def _prep(N, K, seed, code_values=3):
    raw, codes_o, scales_o = U.weights(N, K, seed, code_values=code_values)
    codes, scales = pq2.pq2_prepare(raw, K)
    return codes, scales, codes_o, scales_o


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("M,K", [(1, 128), (3, 384), (8, 5120), (5, 17408)])
def test_quantize_mmv16_layout(dtype, M, K):
    x = synth.activations(M, K, seed=M + K, outlier_frac=0.01).to(dtype)
    q_o, sx_o = O.quantize(O.widen(U.x_bits(x), U.kind(x)))
    q, sx, corr = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_MMV16)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy().view(np.uint16), U.mmv16_layout(q_o).view(np.uint16))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_o.view(np.uint32))
    assert np.array_equal(corr.cpu().numpy(), U.mmv16_correction(q_o))


def test_quantize_mmv16_rejects_small_groups():
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((2, 256), dtype=torch.float16, device="cuda")
    sx = torch.empty((2, 8), dtype=torch.float32, device="cuda")
    qs = torch.empty((2, 8), dtype=torch.int32, device="cuda")
    st = pq2.lib().pq2_quantize_act_grouped(x.data_ptr(), pq2.PQ2_BF16, 256, 2, 256, 32,
                                            q.data_ptr(), pq2.PQ2_Q_MMV16, sx.data_ptr(),
                                            qs.data_ptr(), None)
    assert st == pq2.PQ2_ERR_SHAPE


@pytest.mark.parametrize("M", [1, 2, 4, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 128), (300, 1152), (1000, 640), (2048, 17408)])
def test_tc_group_dots_bitexact(M, N, K):
    codes, _, codes_o, scales_o = _prep(N, K, seed=M + N + K, code_values=4)
    x = synth.activations(M, K, seed=M * 3 + K, outlier_frac=0.01)
    _, _, _, dots_o, *_ = U.oracle_reference(x, codes_o, scales_o)
    q, _, corr = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_MMV16)
    dots, back, guard = U.guarded((M, N, K // G), torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pq2.pq2_debug_group_dots(q, codes, pq2.PQ2_PATH_MMV_TC, qsum=corr, dots=dots, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(dots.cpu().numpy(), dots_o)
    assert U.guards_intact(back, guard)


def test_tc_extreme_dots_exact():
    """|dot| = 32512 (code 3, weight +2, against q = +-127) and the largest
    corrections stay exact on the fp16 tensor path."""
    M, N, K = 8, 64, 512
    codes_np = np.full((N, K), 3, np.uint8)
    codes_np[1::2, :] = 0
    codes_np[2::4, ::2] = 2
    sbits = torch.full((N, K // G), 0.02, dtype=torch.float16).view(torch.int16)
    raw = synth.raw_from_parts(torch.from_numpy(codes_np), sbits)
    codes, _ = pq2.pq2_prepare(raw.cuda(), K)
    x = torch.full((M, K), 127.0)
    x[1::3] = -127.0
    x[2::5, ::3] = 63.0
    x = x.to(torch.bfloat16)
    q, _, corr = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_MMV16)
    dots = pq2.pq2_debug_group_dots(q, codes, pq2.PQ2_PATH_MMV_TC, qsum=corr)
    torch.cuda.synchronize()
    codes_o, _ = O.prepare(raw.numpy(), K)
    q_o, _ = O.quantize(O.widen(synth.bits_u16(x), "bf16"))
    dots_o = O.group_dots(q_o, codes_o)
    assert np.abs(dots_o).max() == 32512
    assert np.array_equal(dots.cpu().numpy(), dots_o)


def _both(x, codes, scales, out_dtype, flags=0):
    qp, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
    qt, sx2, corr = pq2.pq2_quantize_act(x, pq2.PQ2_Q_MMV16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    yt = pq2.pq2_mmv_tc(qt, sx2, corr, codes, scales, out_dtype=out_dtype, flags=flags,
                        status=status)
    yd = pq2.pq2_mmv(qp, sx, qs, codes, scales, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return yt, yd


@pytest.mark.parametrize("N,K", SHAPES)
def test_tc_equals_dp4a_every_m(N, K):
    codes, scales, codes_o, scales_o = _prep(N, K, seed=N ^ K)
    x8 = synth.activations(8, K, seed=N + 3 * K, device="cuda", outlier_frac=0.01)
    for M in range(1, 9):
        for dt in (torch.float32, torch.bfloat16):
            yt, yd = _both(x8[:M], codes, scales, dt)
            ib = torch.int32 if dt == torch.float32 else torch.int16
            assert torch.equal(yt.view(ib), yd.view(ib)), (M, dt)
    # and against the oracle at one M (the dp4a GEMV is checked the same way)
    if N * K <= 4_000_000:
        *_, y64, bound = U.oracle_reference(x8[:3].cpu(), codes_o, scales_o)
        yt, _ = _both(x8[:3], codes, scales, torch.float32)
        ok, worst = O.within_bound(yt.cpu().numpy(), y64, bound)
        assert ok, worst


@pytest.mark.parametrize("flags", [pq2.PQ2_MMV_OVERLAP_WEIGHTS, pq2.PQ2_MMV_INDEPENDENT])
def test_tc_flags_same_bits(flags):
    N, K = 10240, 5120
    codes, scales, _, _ = _prep(N, K, seed=5)
    x = synth.activations(6, K, seed=6, device="cuda")
    yt, yd = _both(x, codes, scales, torch.float32, flags=flags)
    assert torch.equal(yt.view(torch.int32), yd.view(torch.int32))


@pytest.mark.parametrize("M", [1, 3, 5, 8])
def test_linear_tensor_path_bit_identical(M):
    """pq2_linear on the M where it runs the tensor-core GEMV equals
    quantise + pq2_mmv, in a chain of dependent calls."""
    N, K = 6144, 5120
    codes, scales, _, _ = _prep(N, K, seed=M)
    xs = [synth.activations(M, K, seed=40 + M + i, device="cuda") for i in range(3)]
    ys = [pq2.linear(x, codes, scales) for x in xs]
    torch.cuda.synchronize()
    for x, y in zip(xs, ys):
        q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
        yd = pq2.pq2_mmv(q, sx, qs, codes, scales)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), yd.view(torch.int32))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert pq2.lib().pq2_linear_tensor_gemv(M, N, K, sms) == (1 if M >= 5 else 0)


def test_prep_writes_mmv16():
    """The fused preparation writes the same PQ2_Q_MMV16 bytes and corrections
    as quantising its own q (it shares the store)."""
    M, K = 5, 2048
    g = torch.Generator().manual_seed(3)
    x = synth.activations(M, K, seed=4, outlier_frac=0.01).to(torch.bfloat16).cuda()
    w = (torch.randn(K, generator=g) * 0.1).to(torch.bfloat16).cuda()
    sign = (torch.randint(0, 2, (K,), generator=g) * 2 - 1).to(torch.int8).cuda()
    qt, _, corr, _, _ = pq2.pq2_norm_hadamard_quantize(x, w, sign, 1e-6,
                                                       layout=pq2.PQ2_Q_MMV16)
    qr, _, _, _, _ = pq2.pq2_norm_hadamard_quantize(x, w, sign, 1e-6, layout=pq2.PQ2_Q_ROWS)
    torch.cuda.synchronize()
    qr = qr.cpu().numpy()
    assert np.array_equal(qt.cpu().numpy().view(np.uint16), U.mmv16_layout(qr).view(np.uint16))
    assert np.array_equal(corr.cpu().numpy(), U.mmv16_correction(qr))
