"""Prefill path pq2_mm (tcgen05) against the CPU oracle, through the C ABI.

Bit-exact: the per-group int32 dots the tensor cores form (the debug path
reads them straight out of the MMA accumulator).  Fp32 y within
|y - y64| <= 1e-5 * sum_g |s_x * s_w * dot_g|; bf16 y within that plus half
a bf16 ulp.
"""
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


def _prep(N, K, seed, code_values=3):
    raw, codes_o, scales_o = U.weights(N, K, seed, code_values=code_values)
    codes, scales = pq2.pq2_prepare(raw, K)
    return codes, scales, codes_o, scales_o


SHAPES = [(16, 128, 128), (128, 128, 384), (200, 300, 1152), (384, 1000, 640), (130, 136, 2048),
          (1, 256, 640), (9, 300, 1152)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_mm_group_dots_bitexact(M, N, K):
    codes, scales, codes_o, scales_o = _prep(N, K, seed=M + N + K, code_values=4)
    x = synth.activations(M, K, seed=M * 3 + K, outlier_frac=0.01)
    q_o, _, _, dots_o, *_ = U.oracle_reference(x, codes_o, scales_o)
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_F16)
    dots, back, guard = U.guarded((M, N, K // G), torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pq2.pq2_debug_group_dots(q, codes, pq2.PQ2_PATH_MM, qsum=qs, dots=dots, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(dots.cpu().numpy(), dots_o)
    assert U.guards_intact(back, guard)


@pytest.mark.parametrize("M", [128, 16, 9])
def test_mm_extreme_dots_exact(M):
    """The largest group dots (|dot| = 128 * 127 * 2 = 32512) and alternating
    signs stay exact on the fp16 tensor path."""
    N, K = 128, 512
    codes_np = np.full((N, K), 3, np.uint8)          # weight +2 everywhere
    codes_np[1::2, :] = 0                            # odd rows: weight -1
    codes_np[2::4, ::2] = 2                          # some +1
    sbits = torch.full((N, K // G), 0.02, dtype=torch.float16).view(torch.int16)
    raw = synth.raw_from_parts(torch.from_numpy(codes_np), sbits)
    codes, scales = pq2.pq2_prepare(raw.cuda(), K)
    x = torch.full((M, K), 127.0)
    x[1::3] = -127.0
    x[2::5, ::3] = 63.0
    x = x.to(torch.bfloat16)
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_F16)
    dots = pq2.pq2_debug_group_dots(q, codes, pq2.PQ2_PATH_MM, qsum=qs)
    torch.cuda.synchronize()
    codes_o, scales_o = O.prepare(raw.numpy(), K)
    q_o, _ = O.quantize(O.widen(synth.bits_u16(x), "bf16"))
    dots_o = O.group_dots(q_o, codes_o)
    assert np.abs(dots_o).max() == 32512
    assert np.array_equal(dots.cpu().numpy(), dots_o)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_mm_y_within_bound(M, N, K):
    codes, scales, codes_o, scales_o = _prep(N, K, seed=7 * M + N)
    x = synth.activations(M, K, seed=M + 5, outlier_frac=0.01)
    *_, y64, bound = U.oracle_reference(x, codes_o, scales_o)
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_F16)
    y, back, guard = U.guarded((M, N), torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pq2.pq2_mm(q, sx, qs, codes, scales, y=y, status=status)
    yb = pq2.pq2_mm(q, sx, qs, codes, scales, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert U.guards_intact(back, guard)
    ok, worst = O.within_bound(y.cpu().numpy(), y64, bound)
    assert ok, worst
    ok, worst = O.bf16_within_bound(yb.cpu().float().numpy(), y64, bound)
    assert ok, worst


@pytest.mark.parametrize("M", [16, 128, 512, 2048, 4096])
def test_mm_prefill_ffn_up_against_oracle(M):
    """Prefill ffn_up K=5120, N=17408 at the benchmark's M values, in the
    benchmark's launch configuration: every token row up to M = 512, and
    above that at least 64 seeded rows covering every 128-token tile, against
    every output column, for pq2_mm (fp16 operands) and pq2_mm_f8 (e4m3
    planes); fp32 and bf16 outputs."""
    N, K = 17408, 5120
    codes, scales, codes_o, scales_o = _prep(N, K, seed=2024)
    x = synth.activations(M, K, seed=M)
    xd = x.cuda()
    q, sx, qs = pq2.pq2_quantize_act(xd, pq2.PQ2_Q_F16)
    q8, _, _ = pq2.pq2_quantize_act(xd, pq2.PQ2_Q_F8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = pq2.pq2_mm(q, sx, qs, codes, scales, status=status)
    y8 = pq2.pq2_mm_f8(q8, sx, qs, codes, scales, status=status)
    yb = pq2.pq2_mm_f8(q8, sx, qs, codes, scales, out_dtype=torch.bfloat16, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = U.tile_rows(M, seed=M)
    assert len(rows) == M or (len(rows) >= 64 and
                              len(set((rows // 128).tolist())) == (M + 127) // 128)
    y64, bound = U.oracle_rows(x, rows, codes_o, scales_o)
    for got in (y, y8):
        ok, worst = O.within_bound(got.cpu().numpy()[rows], y64, bound)
        assert ok, worst
    ok, worst = O.bf16_within_bound(yb.cpu().float().numpy()[rows], y64, bound)
    assert ok, worst


@pytest.mark.parametrize("M", [12, 48, 300])
def test_linear_dispatches_to_mm_for_prefill(M):
    N, K = 384, 1024
    codes, scales, codes_o, scales_o = _prep(N, K, seed=9)
    x = synth.activations(M, K, seed=10)
    y = pq2.linear(x.cuda(), codes, scales)
    torch.cuda.synchronize()
    *_, y64, bound = U.oracle_reference(x, codes_o, scales_o)
    assert O.within_bound(y.cpu().numpy(), y64, bound)[0]
