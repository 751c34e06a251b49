"""pq2_mmv_gated / pq2_linear_gated (the gate/up projection with its gated
activation silu(gate) * up in the GEMV's epilogue) against the oracle's fp64
silu(gate) * up within the bound ``oracle.gated_bound`` derives from the y
rule, batch invariance for M = 1..8, and the complete call against its two
steps."""
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


def _case(I, K, M, seed):
    raw, codes_o, scales_o = U.weights(2 * I, K, seed=seed)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=seed + 1, device="cuda", outlier_frac=0.01)
    return codes, scales, codes_o, scales_o, x


@pytest.mark.parametrize("I,K", [(7, 128), (150, 384), (300, 1152), (1000, 4096),
                                 (2500, 2048), (613, 5120)])
@pytest.mark.parametrize("M", [1, 3, 4, 8])
def test_gated_against_oracle(I, K, M):
    codes, scales, codes_o, scales_o, x = _case(I, K, M, seed=I + 7 * M)
    q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pq2.pq2_mmv_gated(q, sx, qs, codes, scales, status=status)
    out_b = pq2.pq2_mmv_gated(q, sx, qs, codes, scales, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _, _, _, _, _, y64, bound = U.oracle_reference(x, codes_o, scales_o)
    out64 = O.gated(y64)
    gb = O.gated_bound(y64, bound)
    ok, worst = O.gated_within_bound(out.cpu().numpy(), out64, gb)
    assert ok, worst
    ok, worst = O.gated_within_bound(out_b.float().cpu().numpy(), out64, gb, bf16=True)
    assert ok, worst


@pytest.mark.parametrize("I,K,M", [(1000, 4096, 1), (2500, 2048, 4), (613, 5120, 8)])
def test_gated_uses_the_gemv_rows(I, K, M):
    """silu(gate) * up from pq2_mmv's own y (fp32 on the host) agrees with the
    gated kernel to a few fp32 ulps: the gate and up sums are pq2_mmv's."""
    codes, scales, _, _, x = _case(I, K, M, seed=5 * I + M)
    q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
    out = pq2.pq2_mmv_gated(q, sx, qs, codes, scales)
    y = pq2.pq2_mmv(q, sx, qs, codes, scales)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    g, u = y[:, :I], y[:, I:]
    ref = (g / (np.float32(1) + np.exp(-g))) * u
    o = out.cpu().numpy()
    assert np.all(np.abs(o - ref) <= 8 * np.spacing(np.abs(ref).astype(np.float32)) + 1e-30)


@pytest.mark.parametrize("I,K", [(5120, 5120), (2560, 17408), (1000, 1152)])
def test_gated_batch_invariance(I, K):
    """Column j is bit-identical for every M in 1..8 (and every column of an
    M-row call equals the same row alone)."""
    raw = synth.raw_weights(2 * I, K, seed=I, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x8 = synth.activations(8, K, seed=K, device="cuda", outlier_frac=0.01)
    ref = None
    for M in range(1, 9):
        q, sx, qs = pq2.pq2_quantize_act(x8[:M].contiguous(), pq2.PQ2_Q_PLANES)
        out = pq2.pq2_mmv_gated(q, sx, qs, codes, scales)
        torch.cuda.synchronize()
        bits = out.cpu().numpy().view(np.uint32)
        if ref is None:
            ref = bits[0].copy()
        assert np.array_equal(bits[0], ref), M
    q, sx, qs = pq2.pq2_quantize_act(x8, pq2.PQ2_Q_PLANES)
    all8 = pq2.pq2_mmv_gated(q, sx, qs, codes, scales).cpu().numpy().view(np.uint32)
    for j in range(8):
        q, sx, qs = pq2.pq2_quantize_act(x8[j:j + 1].contiguous(), pq2.PQ2_Q_PLANES)
        one = pq2.pq2_mmv_gated(q, sx, qs, codes, scales).cpu().numpy().view(np.uint32)
        assert np.array_equal(one[0], all8[j]), j


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_linear_gated_matches_two_calls(M):
    I, K = 3000, 5120
    raw = synth.raw_weights(2 * I, K, seed=M, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=100 + M, device="cuda", outlier_frac=0.01)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = pq2.pq2_linear_gated(x, codes, scales, status=status)
    ab = pq2.pq2_linear_gated(x, codes, scales, out_dtype=torch.bfloat16)
    q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
    b = pq2.pq2_mmv_gated(q, sx, qs, codes, scales)
    bb = pq2.pq2_mmv_gated(q, sx, qs, codes, scales, out_dtype=torch.bfloat16,
                           flags=pq2.PQ2_MMV_INDEPENDENT)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(ab.view(torch.int16), bb.view(torch.int16))


def test_gated_full_size_sampled():
    """ffn gate/up at full size (K=5120, 2 x 17408 rows), M = 1 and 4: a
    sample of output rows (gate and up rows from the oracle) within the
    bound."""
    I, K = 17408, 5120
    raw = synth.raw_weights(2 * I, K, seed=77, device="cpu")
    codes, scales = pq2.pq2_prepare(raw.cuda(), K)
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(I, 96, replace=False))
    rows = np.unique(np.concatenate([rows, [0, I - 1]]))
    sub = np.concatenate([rows, rows + I])
    codes_o, scales_o = O.prepare(raw.numpy()[sub], K)
    for M in (1, 4):
        x = synth.activations(M, K, seed=M, device="cuda", outlier_frac=0.01)
        q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
        out = pq2.pq2_mmv_gated(q, sx, qs, codes, scales)
        torch.cuda.synchronize()
        _, _, _, _, _, y64, bound = U.oracle_reference(x, codes_o, scales_o)
        out64 = O.gated(y64)
        ok, worst = O.gated_within_bound(out.cpu().numpy()[:, rows], out64,
                                         O.gated_bound(y64, bound))
        assert ok, worst


def test_gated_rejects_odd_n_and_bad_flags():
    lib = pq2.lib()
    K, M = 256, 2
    q = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sx = torch.zeros((M, 2), dtype=torch.float32, device="cuda")
    qs = torch.zeros((M, 2), dtype=torch.int32, device="cuda")
    codes = torch.zeros((9, K // 4), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((9, 2), dtype=torch.int16, device="cuda")
    out = torch.empty((M, 8), dtype=torch.float32, device="cuda")
    args = (q.data_ptr(), sx.data_ptr(), qs.data_ptr(), codes.data_ptr(), scales.data_ptr(),
            out.data_ptr(), pq2.PQ2_F32, M)
    assert lib.pq2_mmv_gated(*args, 9, K, 0, None, None) == pq2.PQ2_ERR_SHAPE
    assert lib.pq2_mmv_gated(*args, 8, K, 4, None, None) == pq2.PQ2_ERR_DTYPE
    assert lib.pq2_mmv_gated(*args, 8, K, 0, None, None) == pq2.PQ2_OK
    torch.cuda.synchronize()
