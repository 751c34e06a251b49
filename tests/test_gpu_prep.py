"""pq2_norm_hadamard_quantize (RMSNorm + signs + 1024-point Walsh-Hadamard +
group-128 INT8 in one kernel) against the CPU oracle, bit for bit: q in every
layout, s_x, sum(q), the normalised row and the residual output."""
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


def _inputs(M, K, seed, residual):
    g = torch.Generator().manual_seed(seed)
    x = synth.activations(M, K, seed=seed, outlier_frac=0.01).to(torch.bfloat16)
    r = (torch.randn((M, K), generator=g) * 0.5).to(torch.bfloat16) if residual else None
    w = (torch.randn(K, generator=g) * 0.1).to(torch.bfloat16)
    sign = (torch.randint(0, 2, (K,), generator=g) * 2 - 1).to(torch.int8)
    return x, r, w, sign


def _oracle(x, r, w, sign, eps, rows=None):
    xb = synth.bits_u16(x)
    rb = None if r is None else synth.bits_u16(r)
    if rows is not None:
        xb = xb[rows]
        rb = None if rb is None else rb[rows]
    return O.norm_hadamard_quantize(xb, rb, synth.bits_u16(w), sign.numpy(), eps)


@pytest.mark.parametrize("M,K", [(1, 1024), (3, 5120), (8, 17408), (64, 2048), (2, 32768),
                                 (2, 10240), (1, 16384), (5, 9216)])
@pytest.mark.parametrize("residual", [False, True])
def test_prep_bitexact(M, K, residual):
    eps = 1e-6
    x, r, w, sign = _inputs(M, K, seed=M * 31 + K, residual=residual)
    q_o, sx_o, nb_o, rb_o = _oracle(x, r, w, sign, eps)
    dev = lambda t: None if t is None else t.cuda()
    for layout in (pq2.PQ2_Q_ROWS, pq2.PQ2_Q_PLANES, pq2.PQ2_Q_F16):
        q, sx, qs, nb, rb = pq2.pq2_norm_hadamard_quantize(
            dev(x), dev(w), dev(sign), eps, residual=dev(r), layout=layout,
            want_norm=True, want_residual=residual)
        torch.cuda.synchronize()
        if layout == pq2.PQ2_Q_ROWS:
            assert np.array_equal(q.cpu().numpy(), q_o)
        elif layout == pq2.PQ2_Q_PLANES:
            assert np.array_equal(q.cpu().numpy(), O.q_planes(q_o))
        else:
            assert np.array_equal(q.cpu().float().numpy(),
                                  U.mm_operand_order(q_o).astype(np.float32))
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_o.view(np.uint32))
        assert np.array_equal(qs.cpu().numpy(), O.qsum(q_o))
        assert np.array_equal(synth.bits_u16(nb.cpu()), nb_o)
        if residual:
            assert np.array_equal(synth.bits_u16(rb.cpu()), rb_o)


@pytest.mark.parametrize("M", [4096, 700])
def test_prep_prefill_rows_sampled(M):
    """Many rows (the kernel with one 256-thread CTA per row; M = 4096, K = 5120
    is the prefill shape): sampled rows bit-exact in every q layout, with
    sum(q) (the tensor-core GEMV's correction for PQ2_Q_MMV16)."""
    K, eps = 5120, 1e-5
    x, r, w, sign = _inputs(M, K, seed=11 + M, residual=True)
    rows = np.array([0, 1, 333, M // 2, M - 1])
    q_o, sx_o, _, _ = _oracle(x, r, w, sign, eps, rows=rows)
    for layout in (pq2.PQ2_Q_ROWS, pq2.PQ2_Q_PLANES, pq2.PQ2_Q_F16, pq2.PQ2_Q_F8,
                   pq2.PQ2_Q_MMV16):
        q, sx, qs, _, _ = pq2.pq2_norm_hadamard_quantize(
            x.cuda(), w.cuda(), sign.cuda(), eps, residual=r.cuda(), layout=layout)
        torch.cuda.synchronize()
        qh = q.cpu()
        if layout == pq2.PQ2_Q_ROWS:
            assert np.array_equal(qh.numpy()[rows], q_o)
        elif layout == pq2.PQ2_Q_PLANES:
            assert np.array_equal(qh.numpy()[rows], O.q_planes(q_o))
        elif layout == pq2.PQ2_Q_F16:
            assert np.array_equal(qh.float().numpy()[rows],
                                  U.mm_operand_order(q_o).astype(np.float32))
        elif layout == pq2.PQ2_Q_F8:
            assert np.array_equal(qh.numpy()[rows], U.mm_operand_order_f8(q_o))
        else:
            assert np.array_equal(qh.float().numpy()[rows], U.mmv16_layout(q_o))
        assert np.array_equal(sx.cpu().numpy()[rows].view(np.uint32), sx_o.view(np.uint32))
        qs_o = U.mmv16_correction(q_o) if layout == pq2.PQ2_Q_MMV16 else O.qsum(q_o)
        assert np.array_equal(qs.cpu().numpy()[rows], qs_o)


@pytest.mark.parametrize("K", [1024, 5120, 16384, 32768])
def test_prep_many_rows_every_output(K):
    """The many-row kernel (M = 608, the smallest M it runs) with one to 32
    transform blocks per row: q in the four register-path layouts and the
    tensor-core GEMV's, s_x, sum(q), the normalised row and the residual
    output bit-exact on sampled rows."""
    M, eps = 608, 1e-6
    x, r, w, sign = _inputs(M, K, seed=K + 7, residual=True)
    rows = np.array([0, 5, 301, M - 1])
    q_o, sx_o, nb_o, rb_o = _oracle(x, r, w, sign, eps, rows=rows)
    for layout in (pq2.PQ2_Q_ROWS, pq2.PQ2_Q_PLANES, pq2.PQ2_Q_F16, pq2.PQ2_Q_F8,
                   pq2.PQ2_Q_MMV16):
        q, sx, qs, nb, rb = pq2.pq2_norm_hadamard_quantize(
            x.cuda(), w.cuda(), sign.cuda(), eps, residual=r.cuda(), layout=layout,
            want_norm=True, want_residual=True)
        torch.cuda.synchronize()
        qh = q.cpu()
        if layout == pq2.PQ2_Q_ROWS:
            assert np.array_equal(qh.numpy()[rows], q_o)
        elif layout == pq2.PQ2_Q_PLANES:
            assert np.array_equal(qh.numpy()[rows], O.q_planes(q_o))
        elif layout == pq2.PQ2_Q_F16:
            assert np.array_equal(qh.float().numpy()[rows],
                                  U.mm_operand_order(q_o).astype(np.float32))
        elif layout == pq2.PQ2_Q_F8:
            assert np.array_equal(qh.numpy()[rows], U.mm_operand_order_f8(q_o))
        else:
            assert np.array_equal(qh.float().numpy()[rows], U.mmv16_layout(q_o))
        assert np.array_equal(sx.cpu().numpy()[rows].view(np.uint32), sx_o.view(np.uint32))
        qs_o = U.mmv16_correction(q_o) if layout == pq2.PQ2_Q_MMV16 else O.qsum(q_o)
        assert np.array_equal(qs.cpu().numpy()[rows], qs_o)
        assert np.array_equal(synth.bits_u16(nb.cpu())[rows], nb_o)
        assert np.array_equal(synth.bits_u16(rb.cpu())[rows], rb_o)


def _walsh(k):
    """Walsh function k of length 1024: (-1)^popcount(j & k)."""
    j = np.arange(1024)
    bits = np.array([bin(v).count("1") for v in (j & k)])
    return np.where(bits % 2 == 0, 1.0, -1.0)


def test_prep_many_rows_near_tie():
    """A quotient on a half-integer in the many-row kernel: x = 1, eps = 0
    (so inv = 1), w + 1 and the signs shaped so that each block's input is
    W_a + W_b / 2 (two Walsh functions of the same 128-group).  The
    transform then gives 32 at a and 16 at b, so q(16) = 16 / fl(32/127),
    within 1e-4 of 63.5, which takes the IEEE-division branch; the other
    elements are 0.  Bit-exact against the oracle on the first and last row."""
    M, K = 608, 5120
    w = np.empty(K, np.float32)
    sign = np.empty(K, np.int8)
    for blk in range(K // 1024):
        a = 128 * (blk % 8) + 3 + blk
        b = a + 64 + blk
        v = _walsh(a) + 0.5 * _walsh(b)
        w[1024 * blk:1024 * (blk + 1)] = np.abs(v) - 1.0   # w + 1 = |v|: 1.5 or 0.5
        sign[1024 * blk:1024 * (blk + 1)] = np.where(v > 0, 1, -1)
    x = torch.ones((M, K), dtype=torch.bfloat16)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    st = torch.from_numpy(sign)
    rows = np.array([0, M - 1])
    q_o, sx_o, _, _ = _oracle(x, None, wt, st, 0.0, rows=rows)
    assert set(np.unique(np.abs(q_o)).tolist()) <= {0, 63, 64, 127} and (np.abs(q_o) == 127).any()
    assert ((np.abs(q_o) == 63) | (np.abs(q_o) == 64)).any()
    for layout in (pq2.PQ2_Q_ROWS, pq2.PQ2_Q_F8):
        q, sx, qs, _, _ = pq2.pq2_norm_hadamard_quantize(x.cuda(), wt.cuda(), st.cuda(), 0.0,
                                                         layout=layout)
        torch.cuda.synchronize()
        if layout == pq2.PQ2_Q_ROWS:
            assert np.array_equal(q.cpu().numpy()[rows], q_o)
        else:
            assert np.array_equal(q.cpu().numpy()[rows], U.mm_operand_order_f8(q_o))
        assert np.array_equal(sx.cpu().numpy()[rows].view(np.uint32), sx_o.view(np.uint32))
        assert np.array_equal(qs.cpu().numpy()[rows], O.qsum(q_o))


def test_prep_rows_are_independent():
    """Row j of an 8-row call equals the same row prepared alone."""
    K, eps = 5120, 1e-6
    x, r, w, sign = _inputs(8, K, seed=5, residual=False)
    xc, wc, sc = x.cuda(), w.cuda(), sign.cuda()
    q8, sx8, _, _, _ = pq2.pq2_norm_hadamard_quantize(xc, wc, sc, eps)
    for j in range(8):
        q1, sx1, _, _, _ = pq2.pq2_norm_hadamard_quantize(xc[j:j + 1].contiguous(), wc, sc, eps)
        torch.cuda.synchronize()
        assert torch.equal(q1[0], q8[j]) and torch.equal(sx1[0].view(torch.int32), sx8[j].view(torch.int32))


def test_prep_rejects_bad_arguments():
    lib = pq2.lib()
    M, K = 2, 1024
    x = torch.zeros((M, 4 * K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(4 * K, dtype=torch.bfloat16, device="cuda")
    sign = torch.ones(4 * K, dtype=torch.int8, device="cuda")
    q = torch.empty((M, 4 * K), dtype=torch.int8, device="cuda")
    sx = torch.empty((M, 32), dtype=torch.float32, device="cuda")

    def call(K_, eps=0.0, layout=pq2.PQ2_Q_PLANES, xp=x.data_ptr(), qp=q.data_ptr()):
        return lib.pq2_norm_hadamard_quantize(xp, None, None, w.data_ptr(), sign.data_ptr(),
                                              eps, M, K_, None, qp, layout, sx.data_ptr(),
                                              None, None)
    assert call(1536) == pq2.PQ2_ERR_SHAPE
    assert call(512) == pq2.PQ2_ERR_SHAPE
    assert call(40960) == pq2.PQ2_ERR_SHAPE
    assert call(1024, eps=-1.0) == pq2.PQ2_ERR_SHAPE
    assert call(1024, eps=float("nan")) == pq2.PQ2_ERR_SHAPE
    assert call(1024, layout=7) == pq2.PQ2_ERR_DTYPE
    assert call(1024, xp=None) == pq2.PQ2_ERR_NULL
    assert call(1024, qp=q.data_ptr() + 4) == pq2.PQ2_ERR_ALIGN
    assert call(1024) == pq2.PQ2_OK
    torch.cuda.synchronize()
