"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Bit-exact: prepared planes, q (every layout), s_x, sum(q), per-group int32
dots.  Fp32 y: |y - y64| <= 1e-5 * sum_g |s_x * s_w * dot_g|; bf16 y: the
same plus half a bf16 ulp.  Batch invariance: column j bit-identical for
every M in 1..8.
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


# ------------------------------------------------------------- preparation
@pytest.mark.parametrize("N,K,pad", [(1, 128, 0), (7, 384, 6), (300, 1152, 0),
                                     (1000, 5120, 10)])
def test_prepare_bitexact(N, K, pad):
    raw, codes_o, scales_o = U.weights(N, K, seed=N + K, code_values=4, raw_pad=pad)
    codes, codes_b, cg = U.guarded((N, K // 4), torch.uint8)
    scales, scales_b, sg = U.guarded((N, K // G), torch.int16)
    pq2.pq2_prepare(raw, K, codes=codes, scales=scales.view(torch.float16))
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), codes_o)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), scales_o)
    assert U.guards_intact(codes_b, cg) and U.guards_intact(scales_b, sg)


# ------------------------------------------------------------ quantisation
def _tie_rows(K, dtype):
    x = torch.zeros((3, K))
    x[0, :9] = torch.tensor([127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, -1.5, 126.5])
    x[1, :] = 0.0                                              # zero groups
    for j, amax in enumerate([2.734375, 4.75, 6.5]):           # near-ties
        x[2, j * G] = amax
        x[2, j * G + 1] = amax / 2
        x[2, j * G + 2] = -amax / 2
    return x.to(dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("M,K,ld_pad", [(1, 128, 0), (3, 384, 0), (5, 1152, 3),
                                        (8, 5120, 8), (64, 4096, 0)])
def test_quantize_bitexact(dtype, M, K, ld_pad):
    x = synth.activations(M, K, seed=M * 7 + K, outlier_frac=0.01, dtype=torch.float32)
    if M >= 3:
        x[:3] = _tie_rows(K, torch.float32)
    x = x.to(dtype)
    xs = torch.zeros((M, K + ld_pad), dtype=dtype, device="cuda")
    xs[:, :K] = x.cuda()
    xv = xs[:, :K]
    q_o, sx_o = O.quantize(O.widen(U.x_bits(x), U.kind(x)))
    qs_o = O.qsum(q_o)
    for layout in (pq2.PQ2_Q_ROWS, pq2.PQ2_Q_PLANES, pq2.PQ2_Q_F16):
        q, sx, qs = pq2.pq2_quantize_act(xv, layout)
        torch.cuda.synchronize()
        if layout == pq2.PQ2_Q_ROWS:
            assert np.array_equal(q.cpu().numpy(), q_o)
        elif layout == pq2.PQ2_Q_PLANES:
            assert np.array_equal(q.cpu().numpy(), O.q_planes(q_o))
        else:
            assert np.array_equal(q.cpu().float().numpy(),
                                  U.mm_operand_order(q_o).astype(np.float32))
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_o.view(np.uint32))
        assert np.array_equal(qs.cpu().numpy(), qs_o)



@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("M,K,ld_pad", [(13001, 384, 0), (13001, 384, 3), (1024, 5120, 0),
                                        (410, 5120, 8)])
def test_quantize_batched_bitexact(dtype, M, K, ld_pad):
    """Enough groups for the many-row quantiser (eight lanes per group, four
    groups per warp): 39,003 groups (a ragged last warp), 40,960 and 16,400
    groups of full rows, and a row stride that is not a multiple of 16 bytes
    (which keeps one warp per group).  The same bytes as the oracle in every
    layout."""
    x = synth.activations(M, K, seed=M + K, outlier_frac=0.01, dtype=torch.float32)
    x[:3] = _tie_rows(K, torch.float32)
    x = x.to(dtype)
    xs = torch.zeros((M, K + ld_pad), dtype=dtype, device="cuda")
    xs[:, :K] = x.cuda()
    xv = xs[:, :K]
    q_o, sx_o = O.quantize(O.widen(U.x_bits(x), U.kind(x)))
    qs_o = O.qsum(q_o)
    for layout in (pq2.PQ2_Q_ROWS, pq2.PQ2_Q_PLANES, pq2.PQ2_Q_F16, pq2.PQ2_Q_F8):
        q, sx, qs = pq2.pq2_quantize_act(xv, layout)
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

# ----------------------------------------------------------------- mmv
MMV_SHAPES = [(1, 128), (5, 384), (153, 256), (1000, 1152), (2048, 4096), (613, 17408)]


def _setup(N, K, M, seed, code_values=3, outliers=0.0):
    raw, codes_o, scales_o = U.weights(N, K, seed, code_values=code_values)
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=seed + 1, outlier_frac=outliers)
    return codes, scales, codes_o, scales_o, x


@pytest.mark.parametrize("N,K", MMV_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 8])
def test_mmv_group_dots_bitexact(N, K, M):
    codes, scales, codes_o, scales_o, x = _setup(N, K, M, seed=N * 31 + K + M, code_values=4)
    q_o, _, _, dots_o, *_ = U.oracle_reference(x, codes_o, scales_o)
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_PLANES)
    for path in (pq2.PQ2_PATH_MMV_ADDXOR, pq2.PQ2_PATH_MMV_PLANES):
        dots, dots_b, dg = U.guarded((M, N, K // G), torch.int32)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pq2.pq2_debug_group_dots(q, codes, path, qsum=qs, dots=dots, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(dots.cpu().numpy(), dots_o), path
        assert U.guards_intact(dots_b, dg)


@pytest.mark.parametrize("N,K", MMV_SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_mmv_y_within_bound(N, K, M):
    codes, scales, codes_o, scales_o, x = _setup(N, K, M, seed=N + 17 * K + M, outliers=0.01)
    *_, y32_o, y64, bound = U.oracle_reference(x, codes_o, scales_o)
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_PLANES)
    outs = {}
    for dec in (pq2.PQ2_DECODE_ADDXOR, pq2.PQ2_DECODE_PLANES):
        y, y_b, yg = U.guarded((M, N), torch.float32)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pq2.pq2_mmv(q, sx, qs, codes, scales, y=y, decode=dec, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert U.guards_intact(y_b, yg)
        ok, worst = O.within_bound(y.cpu().numpy(), y64, bound)
        assert ok, f"decode {dec}: worst error / bound = {worst}"
        outs[dec] = y.cpu().numpy().view(np.uint32)
    assert np.array_equal(outs[0], outs[1])   # exact dots -> identical bits
    yb = pq2.pq2_mmv(q, sx, qs, codes, scales, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ok, worst = O.bf16_within_bound(yb.cpu().float().numpy(), y64, bound)
    assert ok, worst
    # bf16 output is the RNE rounding of the fp32 result
    assert np.array_equal(yb.cpu().view(torch.int16).numpy().view(np.uint16),
                          O.float_to_bf16_rne(outs[0].view(np.float32)))


@pytest.mark.parametrize("N,K", [(10240, 5120), (6144, 5120), (17408, 5120), (5120, 17408),
                                 (777, 1280)])
def test_mmv_batch_invariance(N, K):
    """Column j of the M=1 output is bit-identical to column j at M = 2..8
    (layer sweep shapes, seeded bf16 N(0,1) activations)."""
    raw = synth.raw_weights(N, K, seed=N ^ K, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x8 = synth.activations(8, K, seed=K + 3, device="cuda")
    ref = None
    for M in range(1, 9):
        # the same eight activation rows, presented with a batch of M: row j
        # of every batch is row j of x8 (rows beyond M are absent)
        q, sx, qs = pq2.pq2_quantize_act(x8[:M].contiguous(), pq2.PQ2_Q_PLANES)
        y = pq2.pq2_mmv(q, sx, qs, codes, scales)
        torch.cuda.synchronize()
        yy = y.cpu().numpy().view(np.uint32)
        if ref is None:
            ref = {}
        for j in range(M):
            if j in ref:
                assert np.array_equal(yy[j], ref[j]), (M, j)
            else:
                ref[j] = yy[j].copy()
    # and every row j as the single row of an M = 1 call
    for j in range(8):
        q, sx, qs = pq2.pq2_quantize_act(x8[j:j + 1].contiguous(), pq2.PQ2_Q_PLANES)
        y = pq2.pq2_mmv(q, sx, qs, codes, scales)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32)[0], ref[j]), j


@pytest.mark.parametrize("N,K", [(10240, 5120), (5120, 17408), (1000, 1152)])
@pytest.mark.parametrize("M", [1, 3, 4, 8])
def test_overlap_and_linear_match_plain_calls(N, K, M):
    """The overlapped GEMV and the fused complete call give the same bits as
    quantise + plain pq2_mmv."""
    raw = synth.raw_weights(N, K, seed=N + M, device="cuda")
    codes, scales = pq2.pq2_prepare(raw, K)
    x = synth.activations(M, K, seed=M, device="cuda", outlier_frac=0.01)
    q, sx, qs = pq2.pq2_quantize_act(x, pq2.PQ2_Q_PLANES)
    y_plain = pq2.pq2_mmv(q, sx, qs, codes, scales)
    y_over = pq2.pq2_mmv(q, sx, qs, codes, scales, flags=pq2.PQ2_MMV_OVERLAP_WEIGHTS)
    y_ind = pq2.pq2_mmv(q, sx, qs, codes, scales, flags=pq2.PQ2_MMV_INDEPENDENT)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_lin = pq2.pq2_linear(x, codes, scales, status=status)
    y_lin_b = pq2.pq2_linear(x, codes, scales, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(y_over.view(torch.int32), y_plain.view(torch.int32))
    assert torch.equal(y_ind.view(torch.int32), y_plain.view(torch.int32))
    assert torch.equal(y_lin.view(torch.int32), y_plain.view(torch.int32))
    assert torch.equal(y_lin_b.view(torch.int16), y_plain.to(torch.bfloat16).view(torch.int16))


def test_linear_back_to_back_chain():
    """A chain of complete calls on one stream, each consuming the previous
    output (so every call depends on the one before), matches the same chain
    run call by call with synchronisation in between."""
    N = K = 4096
    mats = [pq2.pq2_prepare(synth.raw_weights(N, K, seed=i, device="cuda"), K) for i in range(4)]
    x0 = synth.activations(2, K, seed=11, device="cuda")

    def chain(sync):
        x = x0
        for c, sc in mats * 3:
            x = pq2.pq2_linear(x, c, sc, out_dtype=torch.bfloat16)
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return x

    a = chain(False)
    b = chain(True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_mmv_deterministic_repeats():
    N, K, M = 5120, 17408, 4
    codes, scales, *_ , x = _setup(N, K, M, seed=99)
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_PLANES)
    first = pq2.pq2_mmv(q, sx, qs, codes, scales).clone()
    for _ in range(20):
        y = pq2.pq2_mmv(q, sx, qs, codes, scales)
        assert torch.equal(y.view(torch.int32), first.view(torch.int32))


def test_mmv_special_codes():
    """All-code-1 weights give exactly 0; all-code-2 weights give
    sum_g sum(q) * s_x * s_w within the bound."""
    N, K, M = 300, 1024, 3
    for code, expect_zero in [(1, True), (2, False)]:
        codes_np = np.full((N, K), code, np.uint8)
        sbits = torch.full((N, K // G), 0.03, dtype=torch.float16).view(torch.int16)
        raw = synth.raw_from_parts(torch.from_numpy(codes_np), sbits)
        codes, scales = pq2.pq2_prepare(raw.cuda(), K)
        x = synth.activations(M, K, seed=5)
        q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_PLANES)
        y = pq2.pq2_mmv(q, sx, qs, codes, scales)
        torch.cuda.synchronize()
        if expect_zero:
            assert not y.any()
        else:
            codes_o, scales_o = O.prepare(raw.numpy(), K)
            *_, y64, bound = U.oracle_reference(x, codes_o, scales_o)
            assert O.within_bound(y.cpu().numpy(), y64, bound)[0]


def test_mmv_rejects_bad_arguments_without_launch():
    N, K, M = 64, 256, 2
    codes, scales, *_, x = _setup(N, K, M, seed=3)
    q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_PLANES)
    L = pq2.lib()
    y = torch.empty((M, N), device="cuda")
    base = [q.data_ptr(), sx.data_ptr(), qs.data_ptr(), codes.data_ptr(), scales.data_ptr(),
            y.data_ptr(), pq2.PQ2_F32, M, N, K, None, None]
    assert L.pq2_mmv(*base) == pq2.PQ2_OK
    bad = list(base); bad[7] = 9
    assert L.pq2_mmv(*bad) == pq2.PQ2_ERR_SHAPE
    bad = list(base); bad[9] = 200
    assert L.pq2_mmv(*bad) == pq2.PQ2_ERR_SHAPE
    bad = list(base); bad[0] = q.data_ptr() + 4
    assert L.pq2_mmv(*bad) == pq2.PQ2_ERR_ALIGN
    bad = list(base); bad[6] = 7
    assert L.pq2_mmv(*bad) == pq2.PQ2_ERR_DTYPE
    bad = list(base); bad[2] = None
    assert L.pq2_mmv(*bad) == pq2.PQ2_ERR_NULL
    torch.cuda.synchronize()


# ------------------------------------------------- full-size workloads
FULL = [
    # (name, N, K, Ms, outliers)
    ("gemv_4096x14336", 14336, 4096, [1], 0.0),
    ("attn_qkv", 10240, 5120, [1, 2, 3, 4], 0.01),
    ("ffn_up", 17408, 5120, [1, 2, 3, 4, 8], 0.0),
    ("ffn_down", 5120, 17408, [1, 2, 3, 4, 8], 0.0),
]


@pytest.mark.parametrize("name,N,K,Ms,outliers", FULL, ids=[f[0] for f in FULL])
def test_full_size_against_oracle(name, N, K, Ms, outliers):
    """Full shapes in the launch configuration the benchmark times: every
    group dot bit-exact, every output within the bound."""
    raw, codes_o, scales_o = U.weights(N, K, seed=len(name) * 1000 + N)
    codes, scales = pq2.pq2_prepare(raw, K)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), codes_o)
    for M in Ms:
        x = synth.activations(M, K, seed=M + N, outlier_frac=outliers)
        q_o, sx_o, qs_o, dots_o, y32_o, y64, bound = U.oracle_reference(x, codes_o, scales_o)
        q, sx, qs = pq2.pq2_quantize_act(x.cuda(), pq2.PQ2_Q_PLANES)
        path = (pq2.PQ2_PATH_MMV_ADDXOR if pq2.mmv_decoder(M) == pq2.PQ2_DECODE_ADDXOR
                else pq2.PQ2_PATH_MMV_PLANES)
        dots = pq2.pq2_debug_group_dots(q, codes, path, qsum=qs)
        y = pq2.pq2_mmv(q, sx, qs, codes, scales)
        torch.cuda.synchronize()
        assert np.array_equal(q.cpu().numpy(), O.q_planes(q_o))
        assert np.array_equal(sx.cpu().numpy(), sx_o)
        assert np.array_equal(dots.cpu().numpy(), dots_o)
        ok, worst = O.within_bound(y.cpu().numpy(), y64, bound)
        assert ok, (M, worst)
