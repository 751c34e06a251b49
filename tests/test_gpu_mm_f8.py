"""The 8-bit prefill path pq2_mm_f8 (weights decoded to e4m3, q as the two
exact e4m3 planes of PQ2_Q_F8) through the C ABI: the quantiser's PQ2_Q_F8
bytes against an independent construction, the per-group dots bit-exact
against the oracle, and y bit-identical to the fp16 path pq2_mm (both form
the exact group dots, and the epilogue is shared), hence within the bound."""
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


SHAPES = [(16, 128, 128), (128, 128, 384), (200, 300, 1152), (384, 1000, 640), (130, 136, 2048),
          (1, 256, 640), (9, 300, 1152)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,K", [(1, 128), (3, 384), (16, 5120), (130, 1152)])
def test_quantize_f8_layout(dtype, M, K):
    x = synth.activations(M, K, seed=M + K, outlier_frac=0.01).to(dtype)
    q_o, sx_o = O.quantize(O.widen(U.x_bits(x), U.kind(x)))
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_F8)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), U.mm_operand_order_f8(q_o))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_o.view(np.uint32))
    assert np.array_equal(qs.cpu().numpy(), O.qsum(q_o))


def test_prep_f8_layout():
    """The fused preparation writes the same PQ2_Q_F8 bytes as quantising its
    own q (it shares the store)."""
    M, K = 5, 2048
    g = torch.Generator().manual_seed(3)
    x = synth.activations(M, K, seed=4, outlier_frac=0.01).to(torch.bfloat16).cuda()
    w = (torch.randn(K, generator=g) * 0.1).to(torch.bfloat16).cuda()
    sign = (torch.randint(0, 2, (K,), generator=g) * 2 - 1).to(torch.int8).cuda()
    q8, _, _, _, _ = pq2.pq2_norm_hadamard_quantize(x, w, sign, 1e-6, layout=pq2.PQ2_Q_F8)
    qr, _, _, _, _ = pq2.pq2_norm_hadamard_quantize(x, w, sign, 1e-6, layout=pq2.PQ2_Q_ROWS)
    torch.cuda.synchronize()
    assert np.array_equal(q8.cpu().numpy(), U.mm_operand_order_f8(qr.cpu().numpy()))


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_mm_f8_group_dots_bitexact(M, N, K):
    raw, codes_o, scales_o = U.weights(N, K, seed=M + N + K, code_values=4)
    codes, _ = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M * 3 + K, outlier_frac=0.01)
    q_o, _, _, dots_o, *_ = U.oracle_reference(x, codes_o, scales_o)
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_F8)
    dots, back, guard = U.guarded((M, N, K // G), torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pq2.pq2_debug_group_dots(q, codes, pq2.PQ2_PATH_MM_F8, qsum=qs, dots=dots, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(dots.cpu().numpy(), dots_o)
    assert U.guards_intact(back, guard)


@pytest.mark.parametrize("M", [128, 16, 9])
def test_mm_f8_extreme_dots_exact(M):
    """|dot| = 32512 (weight +2 from code 3 against q = 127) and q = -127
    (16a = -128, b = 1) stay exact on the 8-bit path."""
    N, K = 128, 512
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
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_F8)
    dots = pq2.pq2_debug_group_dots(q, codes, pq2.PQ2_PATH_MM_F8, qsum=qs)
    torch.cuda.synchronize()
    codes_o, _ = O.prepare(raw.numpy(), K)
    q_o, _ = O.quantize(O.widen(synth.bits_u16(x), "bf16"))
    dots_o = O.group_dots(q_o, codes_o)
    assert np.abs(dots_o).max() == 32512
    assert np.array_equal(dots.cpu().numpy(), dots_o)


def _both(M, N, K, seed, out_dtype):
    raw, codes_o, scales_o = U.weights(N, K, seed=seed)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=seed + 1, outlier_frac=0.01)
    q8, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_F8)
    q16, _, _ = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_F16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y8 = pq2.pq2_mm_f8(q8, sx, qs, codes, scales, out_dtype=out_dtype, status=status)
    y16 = pq2.pq2_mm(q16, sx, qs, codes, scales, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return x, codes_o, scales_o, y8, y16


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_mm_f8_y_equals_fp16_path(M, N, K):
    x, codes_o, scales_o, y8, y16 = _both(M, N, K, 11 * M + N, torch.float32)
    assert torch.equal(y8.view(torch.int32), y16.view(torch.int32))
    *_, y64, bound = U.oracle_reference(x, codes_o, scales_o)
    ok, worst = O.within_bound(y8.cpu().numpy(), y64, bound)
    assert ok, worst
    _, _, _, b8, b16 = _both(M, N, K, 11 * M + N, torch.bfloat16)
    assert torch.equal(b8.view(torch.int16), b16.view(torch.int16))


@pytest.mark.parametrize("M", [16, 512, 4096])
def test_mm_f8_prefill_ffn_up_equals_fp16_path(M):
    """ffn_up K=5120, N=17408 at benchmark sizes: bit-identical to pq2_mm."""
    N, K = 17408, 5120
    raw = synth.raw_weights(N, K, seed=2024, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M, device="cuda")
    q8, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_F8)
    q16, _, _ = pq2.pq2_quantize_act(x, pq2.PQ2_Q_F16)
    y8 = pq2.pq2_mm_f8(q8, sx, qs, codes, scales, out_dtype=torch.bfloat16)
    y16 = pq2.pq2_mm(q16, sx, qs, codes, scales, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(y8.view(torch.int16), y16.view(torch.int16))
