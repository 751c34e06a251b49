"""PTQ1_0 weights (page "KERNEL_REPORT: PTQ1_0 small-batch decoding on the
PrismML fork, RTX 3060 12GB"): pq2_ptq_prepare and pq2_ptq_mmv through the C
ABI against the oracle (block decode ``oracle.ptq_unpack``, then the grouped
quantiser, partial dots and fp64 scale-accumulate).

Bit-exact: the prepared planes (a byte move), the partial dots.  Fp32 y:
|y - y64| <= 1e-5 * sum_{g,h} |s_x * d * dot|; bf16 y: the same plus half a
bf16 ulp and equal to the RNE of the fp32 result.  Batch invariance for
M = 1..4."""
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


SHAPES = [(1, 256), (5, 512), (153, 1024), (1000, 1280), (2048, 4096), (613, 17408)]


def _weights(N, K, seed):
    raw = synth.ptq_raw_weights(N, K, seed=seed)
    codes_o, scales_o = O.ptq_unpack(raw.numpy(), K)
    qs, side = pq2.pq2_ptq_prepare(raw.cuda(), K)
    return raw, qs, side, codes_o, scales_o


def _oracle(x, codes_o, scales_o, A):
    a = O.widen(U.x_bits(x), U.kind(x))
    q, sx = O.quantize_grouped(a, A)
    dots = O.group_dots_grouped(q, codes_o, A)
    _, y64, bound = O.scale_accumulate_grouped(dots, sx, scales_o, A)
    return dots, y64, bound


@pytest.mark.parametrize("N,K,pad", [(1, 256, 0), (7, 512, 5), (300, 1280, 0), (64, 17408, 3)])
def test_ptq_prepare_is_a_byte_move(N, K, pad):
    raw = synth.ptq_raw_weights(N, K, seed=N + K)
    G = K // 128
    dev = torch.zeros((N, raw.shape[1] + pad), dtype=torch.uint8)
    dev[:, :raw.shape[1]] = raw
    qs, side = pq2.pq2_ptq_prepare(dev.cuda()[:, :raw.shape[1]], K)
    torch.cuda.synchronize()
    blocks = raw.numpy().reshape(N, G, 28)
    assert np.array_equal(qs.cpu().numpy(), blocks[:, :, :24].reshape(N, 24 * G))
    want = blocks[:, :, 24:28].copy().view("<u4").reshape(N, G)
    assert np.array_equal(side.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("A", [128, 64, 32])
def test_ptq_partial_dots_bitexact(N, K, M, A):
    _, qs, side, codes_o, scales_o = _weights(N, K, seed=N * 5 + K + A)
    x = synth.activations(M, K, seed=N + M + A, outlier_frac=0.01)
    dots_o, _, _ = _oracle(x, codes_o, scales_o, A)
    q, _, qsum = pq2.pq2_quantize_act_grouped(x.cuda(), A, pq2.PQ2_Q_ROWS)
    dots = pq2.pq2_debug_ptq_dots(q, qsum, qs, side, A)
    torch.cuda.synchronize()
    assert np.array_equal(dots.cpu().numpy(), dots_o)


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("A", [128, 32])
def test_ptq_mmv_within_bound(N, K, M, A):
    _, qs, side, codes_o, scales_o = _weights(N, K, seed=N + 3 * K + A)
    x = synth.activations(M, K, seed=K + 7 * M + A, outlier_frac=0.01)
    _, y64, bound = _oracle(x, codes_o, scales_o, A)
    q, sx, qsum = pq2.pq2_quantize_act_grouped(x.cuda(), A, pq2.PQ2_Q_ROWS)
    bits = []
    for flags in (0, pq2.PQ2_MMV_OVERLAP_WEIGHTS, pq2.PQ2_MMV_INDEPENDENT):
        y, y_b, yg = U.guarded((M, N), torch.float32)
        pq2.pq2_ptq_mmv(q, sx, qsum, qs, side, A, y=y, flags=flags)
        torch.cuda.synchronize()
        assert U.guards_intact(y_b, yg)
        ok, worst = O.within_bound(y.cpu().numpy(), y64, bound)
        assert ok, f"flags {flags}: worst error / bound = {worst}"
        bits.append(y.cpu().numpy().view(np.uint32))
    assert all(np.array_equal(bits[0], b) for b in bits[1:])
    yb = pq2.pq2_ptq_mmv(q, sx, qsum, qs, side, A, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ok, worst = O.bf16_within_bound(yb.cpu().float().numpy(), y64, bound)
    assert ok, worst
    assert np.array_equal(yb.cpu().view(torch.int16).numpy().view(np.uint16),
                          O.float_to_bf16_rne(bits[0].view(np.float32)))


@pytest.mark.parametrize("N,K", [(10240, 5120), (14336, 4096), (5120, 17408), (1000, 1280)])
@pytest.mark.parametrize("A", [128, 32])
def test_ptq_batch_invariance(N, K, A):
    """Row j of the output is bit-identical for every M in 1..4, and equal to
    the same activation row alone."""
    raw = synth.ptq_raw_weights(N, K, seed=N + A, device="cuda")
    qs, side = pq2.pq2_ptq_prepare(raw, K)
    x4 = synth.activations(4, K, seed=K + A, device="cuda", outlier_frac=0.01)
    ref = None
    for M in range(1, 5):
        q, sx, qsum = pq2.pq2_quantize_act_grouped(x4[:M].contiguous(), A, pq2.PQ2_Q_ROWS)
        y = pq2.pq2_ptq_mmv(q, sx, qsum, qs, side, A)
        torch.cuda.synchronize()
        bits = y.cpu().numpy().view(np.uint32)
        if ref is None:
            ref = bits[0].copy()
        assert np.array_equal(bits[0], ref), M
    q, sx, qsum = pq2.pq2_quantize_act_grouped(x4, A, pq2.PQ2_Q_ROWS)
    all4 = pq2.pq2_ptq_mmv(q, sx, qsum, qs, side, A).cpu().numpy().view(np.uint32)
    for j in range(4):
        q, sx, qsum = pq2.pq2_quantize_act_grouped(x4[j:j + 1].contiguous(), A, pq2.PQ2_Q_ROWS)
        one = pq2.pq2_ptq_mmv(q, sx, qsum, qs, side, A).cpu().numpy().view(np.uint32)
        assert np.array_equal(one[0], all4[j]), j


@pytest.mark.parametrize("name,N,K", [("attn_qkv", 10240, 5120), ("ffn_up", 17408, 5120),
                                      ("ffn_down", 5120, 17408)])
def test_ptq_full_size_sampled(name, N, K):
    """The pages' PTQ1_0 shapes at full size, M = 1 and 4, A = 32 and 128: a
    sample of output rows from the oracle within the bound."""
    raw = synth.ptq_raw_weights(N, K, seed=N + 1, device="cpu")
    qs, side = pq2.pq2_ptq_prepare(raw.cuda(), K)
    rng = np.random.default_rng(N)
    rows = np.unique(np.concatenate([rng.choice(N, 64, replace=False), [0, N - 1]]))
    codes_o, scales_o = O.ptq_unpack(raw.numpy()[rows], K)
    for A in (32, 128):
        for M in (1, 4):
            x = synth.activations(M, K, seed=M + A, device="cuda", outlier_frac=0.01)
            q, sx, qsum = pq2.pq2_quantize_act_grouped(x, A, pq2.PQ2_Q_ROWS)
            y = pq2.pq2_ptq_mmv(q, sx, qsum, qs, side, A, flags=pq2.PQ2_MMV_INDEPENDENT)
            torch.cuda.synchronize()
            _, y64, bound = _oracle(x, codes_o, scales_o, A)
            ok, worst = O.within_bound(y.cpu().numpy()[:, rows], y64, bound)
            assert ok, (A, M, worst)


def test_ptq_rejects_bad_arguments():
    lib = pq2.lib()
    M, N, K = 4, 8, 512
    raw = torch.zeros((N, 28 * K // 128), dtype=torch.uint8, device="cuda")
    qs = torch.zeros((N, 24 * K // 128), dtype=torch.uint8, device="cuda")
    side = torch.zeros((N, K // 128), dtype=torch.int32, device="cuda")
    q = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sx = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    qsum = torch.zeros((M, K // 32), dtype=torch.int32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")

    def prep(K_, stride=raw.shape[1], qs_p=qs.data_ptr()):
        return lib.pq2_ptq_prepare(raw.data_ptr(), stride, N, K_, qs_p, side.data_ptr(), None)

    def mmv(M_, K_, A, flags=0, qs_p=qs.data_ptr()):
        return lib.pq2_ptq_mmv(q.data_ptr(), sx.data_ptr(), qsum.data_ptr(), qs_p,
                               side.data_ptr(), y.data_ptr(), pq2.PQ2_F32, M_, N, K_, A, flags,
                               None)
    assert prep(384) == pq2.PQ2_ERR_SHAPE
    assert prep(K, stride=10) == pq2.PQ2_ERR_SHAPE
    assert prep(K, qs_p=qs.data_ptr() + 8) == pq2.PQ2_ERR_ALIGN
    assert prep(K) == pq2.PQ2_OK
    assert mmv(5, K, 32) == pq2.PQ2_ERR_SHAPE
    assert mmv(M, 384, 32) == pq2.PQ2_ERR_SHAPE
    assert mmv(M, K, 16) == pq2.PQ2_ERR_SHAPE
    assert mmv(M, K, 32, flags=8) == pq2.PQ2_ERR_DTYPE
    assert mmv(M, K, 32, qs_p=qs.data_ptr() + 4) == pq2.PQ2_ERR_ALIGN
    assert mmv(M, K, 32) == pq2.PQ2_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [1, 2, 4])
@pytest.mark.parametrize("A", [128, 32])
def test_ptq_linear_matches_two_calls(M, A):
    """pq2_ptq_linear is bit-identical to pq2_quantize_act_grouped (rows)
    followed by pq2_ptq_mmv, for fp32 and bf16 outputs."""
    N, K = 3000, 5120
    raw = synth.ptq_raw_weights(N, K, seed=M + A, device="cuda")
    qs, side = pq2.pq2_ptq_prepare(raw, K)
    x = synth.activations(M, K, seed=A + 3 * M, device="cuda", outlier_frac=0.01)
    for out_dtype in (torch.float32, torch.bfloat16):
        a = pq2.pq2_ptq_linear(x, qs, side, A, out_dtype=out_dtype)
        q, sx, qsum = pq2.pq2_quantize_act_grouped(x, A, pq2.PQ2_Q_ROWS)
        b = pq2.pq2_ptq_mmv(q, sx, qsum, qs, side, A, out_dtype=out_dtype)
        torch.cuda.synchronize()
        iv = torch.int32 if out_dtype == torch.float32 else torch.int16
        assert torch.equal(a.view(iv), b.view(iv))


def test_ptq_linear_rejects_small_workspace():
    lib = pq2.lib()
    M, N, K = 2, 8, 512
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    qs = torch.zeros((N, 24 * K // 128), dtype=torch.uint8, device="cuda")
    side = torch.zeros((N, K // 128), dtype=torch.int32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    need = lib.pq2_ptq_linear_workspace_bytes(M, K, 32)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (x.data_ptr(), pq2.PQ2_BF16, K, M, N, K, qs.data_ptr(), side.data_ptr(), 32,
            y.data_ptr(), pq2.PQ2_F32, ws.data_ptr())
    assert lib.pq2_ptq_linear(*args, need - 1, None) == pq2.PQ2_ERR_SHAPE
    assert lib.pq2_ptq_linear_workspace_bytes(5, K, 32) == 0
    assert lib.pq2_ptq_linear(*args, need, None) == pq2.PQ2_OK
    torch.cuda.synchronize()
