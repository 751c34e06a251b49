"""Activation groups of 64 and 32 (page "Kernel experiments: recorded
evidence", Test 9): pq2_quantize_act_grouped and pq2_mmv_grouped through the
C ABI against the oracle's grouped functions.

Bit-exact: q (every layout), s_x, sum(q) per activation group, the partial
dots.  Fp32 y: |y - y64| <= 1e-5 * sum_{g,h} |s_x[gh] * s_w[g] * dot_gh|
(the oracle's grouped bound); bf16 y: the same plus half a bf16 ulp.  Batch
invariance for M = 1..4.  act_group = 128 gives the plain path's bytes."""
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


SHAPES = [(1, 128), (5, 384), (153, 256), (1000, 1152), (2048, 4096), (613, 17408)]


def _oracle(x, codes_o, scales_o, A):
    a = O.widen(U.x_bits(x), U.kind(x))
    q, sx = O.quantize_grouped(a, A)
    dots = O.group_dots_grouped(q, codes_o, A)
    y32, y64, bound = O.scale_accumulate_grouped(dots, sx, scales_o, A)
    return q, sx, O.qsum_grouped(q, A), dots, y32, y64, bound


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("M,K", [(1, 128), (3, 384), (4, 5120), (8, 1152), (64, 2048),
                                 (13001, 384)])
@pytest.mark.parametrize("A", [64, 32])
def test_quantize_grouped_bitexact(dtype, M, K, A):
    x = synth.activations(M, K, seed=M * 7 + K + A, outlier_frac=0.01).to(dtype)
    a = O.widen(U.x_bits(x), U.kind(x))
    q_o, sx_o = O.quantize_grouped(a, A)
    qs_o = O.qsum_grouped(q_o, A)
    for layout in (pq2.PQ2_Q_ROWS, pq2.PQ2_Q_PLANES, pq2.PQ2_Q_F16, pq2.PQ2_Q_F8):
        q, sx, qs = pq2.pq2_quantize_act_grouped(x.cuda(), A, layout)
        torch.cuda.synchronize()
        if layout == pq2.PQ2_Q_ROWS:
            assert np.array_equal(q.cpu().numpy(), q_o)
        elif layout == pq2.PQ2_Q_PLANES:
            assert np.array_equal(q.cpu().numpy(), O.q_planes(q_o))
        elif layout == pq2.PQ2_Q_F8:
            assert np.array_equal(q.cpu().numpy(), U.mm_operand_order_f8(q_o))
        else:
            assert np.array_equal(q.cpu().float().numpy(),
                                  U.mm_operand_order(q_o).astype(np.float32))
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_o.view(np.uint32))
        assert np.array_equal(qs.cpu().numpy(), qs_o)


@pytest.mark.parametrize("M,K", [(1, 128), (4, 5120), (8, 1152)])
def test_quantize_grouped_128_is_the_plain_quantiser(M, K):
    x = synth.activations(M, K, seed=K + M, device="cuda", outlier_frac=0.01)
    for layout in (pq2.PQ2_Q_ROWS, pq2.PQ2_Q_PLANES, pq2.PQ2_Q_F16):
        a = pq2.pq2_quantize_act_grouped(x, 128, layout)
        b = pq2.pq2_quantize_act(x, layout)
        torch.cuda.synchronize()
        assert torch.equal(a[0].view(torch.int8), b[0].view(torch.int8))
        assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
        assert torch.equal(a[2], b[2])


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("A", [64, 32])
def test_grouped_partial_dots_bitexact(N, K, M, A):
    raw, codes_o, scales_o = U.weights(N, K, seed=N * 3 + K + M + A, code_values=4)
    codes, _ = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=N + K + A, outlier_frac=0.01)
    _, _, _, dots_o, *_ = _oracle(x, codes_o, scales_o, A)
    q, _, qs = pq2.pq2_quantize_act_grouped(x.cuda(), A, pq2.PQ2_Q_PLANES)
    dots = pq2.pq2_debug_group_dots_grouped(q, qs, codes, A)
    torch.cuda.synchronize()
    assert np.array_equal(dots.cpu().numpy(), dots_o)


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 6, 8])
@pytest.mark.parametrize("A", [64, 32])
def test_mmv_grouped_within_bound(N, K, M, A):
    raw, codes_o, scales_o = U.weights(N, K, seed=N + 5 * K + M + A)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=K + 3 * M + A, outlier_frac=0.01)
    *_, y64, bound = _oracle(x, codes_o, scales_o, A)
    q, sx, qs = pq2.pq2_quantize_act_grouped(x.cuda(), A, pq2.PQ2_Q_PLANES)
    bits = []
    for flags in (0, pq2.PQ2_MMV_OVERLAP_WEIGHTS, pq2.PQ2_MMV_INDEPENDENT):
        y, y_b, yg = U.guarded((M, N), torch.float32)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pq2.pq2_mmv_grouped(q, sx, qs, codes, scales, A, y=y, flags=flags, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert U.guards_intact(y_b, yg)
        ok, worst = O.within_bound(y.cpu().numpy(), y64, bound)
        assert ok, f"flags {flags}: worst error / bound = {worst}"
        bits.append(y.cpu().numpy().view(np.uint32))
    assert all(np.array_equal(bits[0], b) for b in bits[1:])
    yb = pq2.pq2_mmv_grouped(q, sx, qs, codes, scales, A, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ok, worst = O.bf16_within_bound(yb.cpu().float().numpy(), y64, bound)
    assert ok, worst
    assert np.array_equal(yb.cpu().view(torch.int16).numpy().view(np.uint16),
                          O.float_to_bf16_rne(bits[0].view(np.float32)))


@pytest.mark.parametrize("N,K", [(1000, 1152), (5120, 5120)])
def test_mmv_grouped_128_is_the_plain_gemv(N, K):
    raw = synth.raw_weights(N, K, seed=N, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    for M in (1, 4):
        x = synth.activations(M, K, seed=M + K, device="cuda", outlier_frac=0.01)
        q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
        a = pq2.pq2_mmv_grouped(q, sx, qs, codes, scales, 128)
        b = pq2.pq2_mmv(q, sx, qs, codes, scales, decode=pq2.PQ2_DECODE_PLANES)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("N,K", [(10240, 5120), (17408, 5120), (5120, 17408), (1000, 1152)])
@pytest.mark.parametrize("A", [64, 32])
def test_mmv_grouped_batch_invariance(N, K, A):
    """Row j of the output is bit-identical for every M in 1..8 (M > 4 runs
    as two passes), and equal to the same activation row alone."""
    raw = synth.raw_weights(N, K, seed=N + A, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x8 = synth.activations(8, K, seed=K + A, device="cuda", outlier_frac=0.01)
    ref = None
    for M in range(1, 9):
        q, sx, qs = pq2.pq2_quantize_act_grouped(x8[:M].contiguous(), A, pq2.PQ2_Q_PLANES)
        y = pq2.pq2_mmv_grouped(q, sx, qs, codes, scales, A)
        torch.cuda.synchronize()
        bits = y.cpu().numpy().view(np.uint32)
        if ref is None:
            ref = bits[0].copy()
        assert np.array_equal(bits[0], ref), M
    q, sx, qs = pq2.pq2_quantize_act_grouped(x8, A, pq2.PQ2_Q_PLANES)
    all8 = pq2.pq2_mmv_grouped(q, sx, qs, codes, scales, A).cpu().numpy().view(np.uint32)
    for j in range(8):
        q, sx, qs = pq2.pq2_quantize_act_grouped(x8[j:j + 1].contiguous(), A, pq2.PQ2_Q_PLANES)
        one = pq2.pq2_mmv_grouped(q, sx, qs, codes, scales, A).cpu().numpy().view(np.uint32)
        assert np.array_equal(one[0], all8[j]), j


@pytest.mark.parametrize("A", [64, 32])
def test_mmv_grouped_full_size_sampled(A):
    """ffn_up at full size (N = 17408, K = 5120), M = 1 and 4: a sample of
    output rows from the oracle within the bound."""
    N, K = 17408, 5120
    raw = synth.raw_weights(N, K, seed=91, device="cpu")
    codes, scales = pq2.pq2_prepare(raw.cuda(), K)
    rng = np.random.default_rng(A)
    rows = np.unique(np.concatenate([rng.choice(N, 96, replace=False), [0, N - 1]]))
    codes_o, scales_o = O.prepare(raw.numpy()[rows], K)
    for M in (1, 4):
        x = synth.activations(M, K, seed=M + A, device="cuda", outlier_frac=0.01)
        q, sx, qs = pq2.pq2_quantize_act_grouped(x, A, pq2.PQ2_Q_PLANES)
        y = pq2.pq2_mmv_grouped(q, sx, qs, codes, scales, A)
        torch.cuda.synchronize()
        *_, y64, bound = _oracle(x, codes_o, scales_o, A)
        ok, worst = O.within_bound(y.cpu().numpy()[:, rows], y64, bound)
        assert ok, worst


def test_grouped_rejects_bad_arguments():
    lib = pq2.lib()
    M, N, K = 9, 8, 256
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sx = torch.zeros((M, 8), dtype=torch.float32, device="cuda")
    qs = torch.zeros((M, 8), dtype=torch.int32, device="cuda")
    codes = torch.zeros((N, K // 4), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((N, 2), dtype=torch.int16, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")

    def quant(A, layout=pq2.PQ2_Q_PLANES):
        return lib.pq2_quantize_act_grouped(x.data_ptr(), pq2.PQ2_BF16, K, M, K, A,
                                            q.data_ptr(), layout, sx.data_ptr(), qs.data_ptr(),
                                            None)

    def mmv(Mc, A, flags=0):
        return lib.pq2_mmv_grouped(q.data_ptr(), sx.data_ptr(), qs.data_ptr(), codes.data_ptr(),
                                   scales.data_ptr(), y.data_ptr(), pq2.PQ2_F32, Mc, N, K, A,
                                   flags, None, None)
    assert quant(16) == pq2.PQ2_ERR_SHAPE
    assert quant(96) == pq2.PQ2_ERR_SHAPE
    assert quant(32, layout=9) == pq2.PQ2_ERR_DTYPE
    assert quant(32) == pq2.PQ2_OK
    assert mmv(9, 32) == pq2.PQ2_ERR_SHAPE
    assert mmv(4, 16) == pq2.PQ2_ERR_SHAPE
    assert mmv(4, 32, flags=64) == pq2.PQ2_ERR_DTYPE
    assert mmv(4, 32) == pq2.PQ2_OK
    torch.cuda.synchronize()
