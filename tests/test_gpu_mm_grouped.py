"""The prefill GEMM with activation groups of 64 and 32 (page "Kernel
experiments: recorded evidence", Test 9, "Smaller Q8 activation groups"):
pq2_mm_grouped (fp16 operands), pq2_mm_f8_grouped (e4m3 planes) and
pq2_linear_grouped through the C ABI against the oracle's grouped functions.

Bit-exact: the partial dots of every (weight group, activation group) pair,
read out of the tensor-core accumulator.  Fp32 y within
|y - y64| <= 1e-5 * sum_{g,h} |s_x[gh] * s_w[g] * dot_gh| (the oracle's
grouped bound), bf16 y within that plus half a bf16 ulp.  The two tensor
paths give the same bits; act_group = 128 gives pq2_mm's bits."""
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


# (M, N, K): partial token and row tiles, K from one to 40 weight groups
# (odd group counts take the scale warp's element-wise staging).
SHAPES = [(16, 128, 128), (128, 128, 384), (200, 300, 1152), (384, 1000, 640),
          (130, 136, 2048), (1, 256, 640), (9, 300, 1152), (257, 384, 5120)]

PATHS = [(pq2.PQ2_PATH_MM, pq2.PQ2_Q_F16), (pq2.PQ2_PATH_MM_F8, pq2.PQ2_Q_F8)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("A", [64, 32])
@pytest.mark.parametrize("path,layout", PATHS)
def test_mm_grouped_partial_dots_bitexact(M, N, K, A, path, layout):
    raw, codes_o, scales_o = U.weights(N, K, seed=M + N + K + A, code_values=4)
    codes, _ = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M * 3 + K + A, outlier_frac=0.01)
    _, _, _, dots_o, *_ = U.oracle_reference_grouped(x, codes_o, scales_o, A)
    q, _, _ = pq2.pq2_quantize_act_grouped(x.cuda(), A, layout)
    dots, back, guard = U.guarded((M, N, K // A), torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pq2.pq2_debug_mm_dots_grouped(q, codes, path, A, dots=dots, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert U.guards_intact(back, guard)
    assert np.array_equal(dots.cpu().numpy(), dots_o)


def test_mm_grouped_extreme_dots_exact():
    """The largest partial dots (|dot| = A * 127 * 2) on both tensor paths."""
    M, N, K = 128, 128, 512
    codes_np = np.full((N, K), 3, np.uint8)
    codes_np[1::2, :] = 0
    codes_np[2::4, ::2] = 2
    sbits = torch.full((N, K // 128), 0.02, dtype=torch.float16).view(torch.int16)
    raw = synth.raw_from_parts(torch.from_numpy(codes_np), sbits)
    codes, _ = pq2.pq2_prepare(raw.cuda(), K)
    codes_o, _ = O.prepare(raw.numpy(), K)
    x = torch.full((M, K), 127.0)
    x[1::3] = -127.0
    x[2::5, ::3] = 63.0
    x = x.to(torch.bfloat16)
    for A in (64, 32):
        q_o, _ = O.quantize_grouped(O.widen(synth.bits_u16(x), "bf16"), A)
        dots_o = O.group_dots_grouped(q_o, codes_o, A)
        assert np.abs(dots_o).max() == A * 127 * 2
        for path, layout in PATHS:
            q, _, _ = pq2.pq2_quantize_act_grouped(x.cuda(), A, layout)
            dots = pq2.pq2_debug_mm_dots_grouped(q, codes, path, A)
            torch.cuda.synchronize()
            assert np.array_equal(dots.cpu().numpy(), dots_o), (A, path)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("A", [64, 32])
def test_mm_grouped_y_within_bound(M, N, K, A):
    raw, codes_o, scales_o = U.weights(N, K, seed=7 * M + N + A)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M + 5 + A, outlier_frac=0.01)
    *_, y64, bound = U.oracle_reference_grouped(x, codes_o, scales_o, A)
    q16, sx, qs = pq2.pq2_quantize_act_grouped(x.cuda(), A, pq2.PQ2_Q_F16)
    q8, sx8, qs8 = pq2.pq2_quantize_act_grouped(x.cuda(), A, pq2.PQ2_Q_F8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, back, guard = U.guarded((M, N), torch.float32)
    pq2.pq2_mm_grouped(q16, sx, qs, codes, scales, A, y=y, status=status)
    y8 = pq2.pq2_mm_f8_grouped(q8, sx8, qs8, codes, scales, A, status=status)
    yb = pq2.pq2_mm_f8_grouped(q8, sx8, qs8, codes, scales, A, out_dtype=torch.bfloat16,
                               status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert U.guards_intact(back, guard)
    ok, worst = O.within_bound(y.cpu().numpy(), y64, bound)
    assert ok, worst
    assert torch.equal(y.view(torch.int32), y8.view(torch.int32))
    ok, worst = O.bf16_within_bound(yb.cpu().float().numpy(), y64, bound)
    assert ok, worst
    assert np.array_equal(yb.cpu().view(torch.int16).numpy().view(np.uint16),
                          O.float_to_bf16_rne(y8.cpu().numpy()))


@pytest.mark.parametrize("M,N,K", [(16, 128, 128), (200, 300, 1152), (4096, 17408, 5120)])
def test_mm_grouped_128_is_pq2_mm(M, N, K):
    raw = synth.raw_weights(N, K, seed=N + M, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M, device="cuda")
    for mm, mmg, layout in ((pq2.pq2_mm, pq2.pq2_mm_grouped, pq2.PQ2_Q_F16),
                            (pq2.pq2_mm_f8, pq2.pq2_mm_f8_grouped, pq2.PQ2_Q_F8)):
        q, sx, qs = pq2.pq2_quantize_act(x, layout)
        a = mm(q, sx, qs, codes, scales, out_dtype=torch.bfloat16)
        b = mmg(q, sx, qs, codes, scales, 128, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M", [128, 512, 4096])
@pytest.mark.parametrize("A", [64, 32])
def test_mm_grouped_prefill_ffn_up_against_oracle(M, A):
    """ffn_up K = 5120, N = 17408 at the sizes the pages time grouped calls
    (M = 128, 512) and at M = 4096, in the benchmark's launch configuration
    (pq2_linear_grouped: grouped quantiser, then the 8-bit grouped GEMM):
    every token row up to M = 512, above that at least 64 seeded rows
    covering every 128-token tile, against every output column."""
    N, K = 17408, 5120
    raw, codes_o, scales_o = U.weights(N, K, seed=2025)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M + A)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = pq2.pq2_linear_grouped(x.cuda(), codes, scales, A, status=status)
    yb = pq2.pq2_linear_grouped(x.cuda(), codes, scales, A, out_dtype=torch.bfloat16,
                                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = U.tile_rows(M, seed=M + A)
    assert len(rows) == M or (len(rows) >= 64 and
                              len(set((rows // 128).tolist())) == (M + 127) // 128)
    y64, bound = U.oracle_rows_grouped(x, rows, codes_o, scales_o, A)
    ok, worst = O.within_bound(y.cpu().numpy()[rows], y64, bound)
    assert ok, worst
    ok, worst = O.bf16_within_bound(yb.cpu().float().numpy()[rows], y64, bound)
    assert ok, worst


@pytest.mark.parametrize("M", [1, 3, 4, 6, 8, 9, 15, 48])
@pytest.mark.parametrize("A", [128, 64, 32])
def test_linear_grouped_is_its_two_calls(M, A):
    """pq2_linear_grouped equals the grouped quantiser followed by the grouped
    GEMV (M <= 8) or the grouped 8-bit GEMM (M >= 9), bit for bit, and is
    within the oracle's grouped bound."""
    N, K = 384, 1152
    raw, codes_o, scales_o = U.weights(N, K, seed=M + A)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=2 * M + A, outlier_frac=0.01)
    xd = x.cuda()
    y = pq2.pq2_linear_grouped(xd, codes, scales, A)
    if M <= 8:
        q, sx, qs = pq2.pq2_quantize_act_grouped(xd, A, pq2.PQ2_Q_PLANES)
        ref = pq2.pq2_mmv_grouped(q, sx, qs, codes, scales, A)
    else:
        q, sx, qs = pq2.pq2_quantize_act_grouped(xd, A, pq2.PQ2_Q_F8)
        ref = pq2.pq2_mm_f8_grouped(q, sx, qs, codes, scales, A)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), ref.view(torch.int32))
    *_, y64, bound = U.oracle_reference_grouped(x, codes_o, scales_o, A)
    ok, worst = O.within_bound(y.cpu().numpy(), y64, bound)
    assert ok, worst


@pytest.mark.parametrize("M", [9, 16, 300])
def test_prefill_kernels_are_deterministic(M):
    """Repeated calls give the same bits: the grouped GEMM on both tensor
    paths (A = 64, 32) and the A = 128 kernels, including the narrow kernel
    at M <= 16 (fixed reduction order, no atomics)."""
    N, K = 1000, 1152
    raw = synth.raw_weights(N, K, seed=M, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M + 1, device="cuda", outlier_frac=0.01)
    for A in (128, 64, 32):
        for mm, layout in ((pq2.pq2_mm_grouped, pq2.PQ2_Q_F16),
                           (pq2.pq2_mm_f8_grouped, pq2.PQ2_Q_F8)):
            q, sx, qs = pq2.pq2_quantize_act_grouped(x, A, layout)
            ys = [mm(q, sx, qs, codes, scales, A) for _ in range(3)]
            torch.cuda.synchronize()
            assert all(torch.equal(ys[0].view(torch.int32), y.view(torch.int32)) for y in ys[1:])
