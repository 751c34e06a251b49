"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, not against the oracle's own formulas.

Each ``pin_*`` takes a loaded oracle library (ctypes handle) and raises
AssertionError on a mismatch.  ``tests/test_oracle_pins.py`` runs them against
the real oracle; ``tests/test_oracle_mutants.py`` runs them against copies of
the oracle with planted mistakes and requires that some pin fails for each.

Sources: page "Kernel experiments: recorded evidence" (KE) and page
"Baseline and the integer breakthrough" (BIB).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
G = 128


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f16_bits(v: float) -> int:
    return int(np.array([v], np.float16).view(np.uint16)[0])


def _pack(codes: np.ndarray) -> np.ndarray:
    """codes u8[N][K] (0..3) -> code plane u8[N][K/4], weight k in bits
    2(k%4) of byte k/4 (KE Test 1 block format)."""
    c = codes.astype(np.uint8).reshape(codes.shape[0], -1, 4)
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def _unpack_numpy(plane: np.ndarray) -> np.ndarray:
    """Independent decode through numpy's little-endian bit unpacking:
    field i of a byte = bit(2i) + 2*bit(2i+1); weight = field - 1."""
    bits = np.unpackbits(plane[..., None], axis=-1, bitorder="little")
    fields = bits[..., 0::2].astype(np.int16) + 2 * bits[..., 1::2].astype(np.int16)
    return (fields.reshape(plane.shape[0], -1) - 1).astype(np.int64)


# ------------------------------------------------------------------ decode
def pin_worked_example_unit(lib):
    """BIB 'Calculate with small integers': [-1,0,+1,+1] . [20,30,40,10] = 30;
    at activation scale 0.1 and weight scale 0.5 the contribution is 1.5."""
    ex = _golden("worked_example.json")
    codes = np.ones((1, G), np.uint8)          # code 1 = weight 0 elsewhere
    codes[0, :4] = ex["codes"]
    plane = _pack(codes)
    w = O.decode_matrix(plane, G, lib=lib)
    assert list(w[0, :4]) == ex["weights"], w[0, :4]
    q = np.zeros((1, G), np.int8)
    q[0, :4] = ex["q"]
    dots = O.group_dots(q, plane, lib=lib)
    assert int(dots[0, 0, 0]) == ex["dot"], dots
    sx = np.array([[ex["activation_scale"]]], np.float32)
    sw = np.array([[_f16_bits(ex["weight_scale"])]], np.uint16)
    y32, y64, bound = O.scale_accumulate(dots, sx, sw, lib=lib)
    assert abs(float(y32[0, 0]) - ex["contribution"]) <= 4e-7 * ex["contribution"], y32
    assert abs(float(y64[0, 0]) - ex["contribution"]) <= 1e-7, y64
    assert abs(bound[0, 0] - abs(y64[0, 0])) <= 1e-15


def pin_worked_example_end_to_end(lib):
    """The worked example through the quantiser: with an element of
    magnitude 127 in the group the scale is exactly 1, so q equals x; the
    codes [0,1,2,2] at weight scale 0.5 give exactly 30 * 1 * 0.5 = 15."""
    ex = _golden("worked_example.json")
    x = np.zeros((1, G), np.float32)
    x[0, :4] = ex["q"]
    x[0, 4] = 127.0
    q, sx = O.quantize(x, lib=lib)
    assert sx[0, 0] == np.float32(1.0), sx
    assert list(q[0, :5]) == ex["q"] + [127]
    codes = np.ones((1, G), np.uint8)
    codes[0, :4] = ex["codes"]
    plane = _pack(codes)
    dots = O.group_dots(q, plane, lib=lib)
    y32, y64, _ = O.scale_accumulate(dots, sx, np.array([[_f16_bits(0.5)]], np.uint16), lib=lib)
    assert int(dots[0, 0, 0]) == 30
    assert y32[0, 0] == np.float32(15.0) and y64[0, 0] == 15.0, (y32, y64)


def pin_decode_all_bytes(lib):
    """All 256 packed byte values (KE Test 1: 'separate checks cover all
    packed byte values').  The oracle's field decode must equal (a) the
    pages' add/XOR fast path with its stated byte map, and (b) numpy's
    little-endian bit unpacking, including the field order."""
    tab = _golden("decode_table.json")
    add_c, xor_c = tab["add_constant"], tab["xor_constant"]
    biased = {int(k): v for k, v in tab["biased_byte_to_signed"].items()}
    code_map = {int(k): v for k, v in tab["code_to_weight"].items()}
    plane = np.arange(256, dtype=np.uint8).reshape(256, 1)
    via_numpy = _unpack_numpy(plane)                     # [256][4]
    for p in range(256):
        spread = (p & 3) | ((p << 6) & 0x300) | ((p << 12) & 0x30000) | ((p << 18) & 0x3000000)
        word = ((spread + add_c) & 0xFFFFFFFF)
        fast = []
        for i in range(4):
            byte = (word >> (8 * i)) & 0xFF
            assert byte in biased, (p, i, byte)
            fast.append(biased[byte])
        signed = [((((word ^ xor_c) >> (8 * i)) & 0xFF) ^ 0x80) - 0x80 for i in range(4)]
        assert fast == signed
        got = [O.decode_field(p, i, lib=lib) for i in range(4)]
        assert got == fast, (p, got, fast)
        assert got == list(via_numpy[p]), (p, got, via_numpy[p])
        assert got == [code_map[(p >> (2 * i)) & 3] for i in range(4)]
    assert [O.decode_field(0xFF, i, lib=lib) for i in range(4)] == [2, 2, 2, 2]


def pin_decode_matrix_order(lib):
    """Weight k of a group comes from field k%4 of code byte k/4: the pages'
    byte-expanded MMQ reshapes (byte, shift) to k = 4*byte + shift."""
    rng = np.random.default_rng(11)
    plane = rng.integers(0, 256, size=(3, 2 * 32), dtype=np.uint8)
    w = O.decode_matrix(plane, 2 * G, lib=lib).astype(np.int64)
    assert np.array_equal(w, _unpack_numpy(plane))


# --------------------------------------------------------------- floats
def pin_half_to_float_all(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = O.half_to_float(bits, lib=lib)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_bf16_conversions(lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = O.bf16_to_float(bits, lib=lib)
    nan = np.isnan(ref)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10,
        # exact ties: bf16 value + half an ulp, both parities of the last bit
        (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        ((np.arange(1, 200, dtype=np.uint32) + 0x3F80) << 16 | 0x8000).view(np.float32),
    ])
    ref16 = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.float_to_bf16_rne(vals, lib=lib), ref16)


# -------------------------------------------------------------- quantiser
def pin_quantize_ties_zero_clamp(lib):
    """KE Test 6 _quantize: scale = max|x|/127, IEEE division, round half to
    even, clamp at +-127; a zero group keeps scale 0 and all-zero q."""
    x = np.zeros((3, G), np.float32)
    x[0, :9] = [127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, -1.5, 126.5]
    x[2, :3] = [-254.0, 1.0, 3.0]            # scale 2: 1/2 -> 0, 3/2 -> 2
    q, sx = O.quantize(x, lib=lib)
    assert sx[0, 0] == np.float32(1.0)
    assert list(q[0, :9]) == [127, 2, 4, -2, 0, 2, 0, -2, 126]
    assert sx[1, 0] == 0.0 and not q[1].any()
    assert sx[2, 0] == np.float32(2.0)
    assert list(q[2, :3]) == [-127, 0, 2]


def pin_quantize_properties(lib):
    """Properties fixed by the definition on random data: the max-abs element
    maps to +-127, |q*s - a| <= s/2*(1+2^-16), s = amax/127 within one fp32
    rounding, negating x negates q and keeps s, and scaling x by a power of
    two scales s by it and leaves q unchanged."""
    rng = np.random.default_rng(7)
    a = rng.standard_normal((4, 6 * G)).astype(np.float32)
    a[1, G:2 * G] *= 20.0
    a[2, 2 * G:3 * G] *= 1e-30                       # subnormal-scale group
    q, sx = O.quantize(a, lib=lib)
    grp = a.reshape(4, 6, G)
    amax = np.abs(grp).max(-1)
    assert np.all(np.abs(sx.astype(np.float64) - amax / 127.0) <= amax / 127.0 * 2.0 ** -23)
    qg = q.reshape(4, 6, G).astype(np.int32)
    arg = np.abs(grp).argmax(-1)
    picked = np.take_along_axis(qg, arg[..., None], -1)[..., 0]
    assert np.all(np.abs(picked) == 127)
    err = np.abs(qg * sx[..., None].astype(np.float64) - grp)
    assert np.all(err <= sx[..., None] / 2 * (1 + 2.0 ** -16) + 1e-45)
    qn, sxn = O.quantize(-a, lib=lib)
    assert np.array_equal(qn, -q) and np.array_equal(sxn, sx)
    q4, sx4 = O.quantize(a * np.float32(4.0), lib=lib)
    normal = amax.ravel() > 1e-30
    assert np.array_equal(q4.reshape(4, 6, G)[normal.reshape(4, 6)],
                          q.reshape(4, 6, G)[normal.reshape(4, 6)])
    assert np.array_equal(sx4.ravel()[normal], (sx * np.float32(4.0)).ravel()[normal])


def pin_quantize_vs_numpy(lib):
    """The same definition evaluated with numpy's float32 division and
    round-half-even (np.rint), on bf16-valued N(0,1) data with outliers."""
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((5, 4 * G)).astype(np.float32))
    x[:, rng.choice(4 * G, 5, replace=False)] *= 20
    # near-tie groups: x = amax/2 lands next to 63.5, where dividing by the
    # scale and multiplying by its fp32 reciprocal round to different codes
    for r, amax in enumerate([2.734375, 4.75, 6.5, 6.71875, 9.375]):
        x[r, 3 * G:4 * G] = 0.0
        x[r, 3 * G] = amax
        x[r, 3 * G + 1:3 * G + 8] = torch.tensor([amax / 2, -amax / 2, amax / 4,
                                                    amax / 3, amax / 5, 1.0, -1.0])
    a = x.to(torch.bfloat16).float().numpy()
    q, sx = O.quantize(a, lib=lib)
    grp = a.reshape(5, 4, G)
    s = (np.abs(grp).max(-1) / np.float32(127.0)).astype(np.float32)
    d = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    r = np.clip(np.rint((grp / d[..., None]).astype(np.float32)), -127, 127)
    assert np.array_equal(sx, s)
    assert np.array_equal(q.reshape(5, 4, G), r.astype(np.int8))


def pin_q_planes(lib):
    """KE Test 21 plane-order store: element i of a group goes to
    (i%4)*32 + i//4."""
    q = np.tile(np.arange(G, dtype=np.int64) - 64, (2, 2)).astype(np.int8)
    qp = O.q_planes(q, lib=lib)
    for grp in range(2):
        for i in range(G):
            assert qp[0, grp * G + (i % 4) * 32 + i // 4] == q[0, grp * G + i]
    assert list(qp[1, :4]) == [-64, -60, -56, -52]
    assert qp[1, 32] == -63
    T = O.qsum(q, lib=lib)
    assert np.array_equal(T, np.full((2, 2), sum(range(-64, 64)), np.int32))


# ------------------------------------------------------------- group dots
def pin_group_dots_brute_force(lib):
    """dot[m][n][g] against an int64 matmul of numpy-decoded weights, on
    random codes including code 3 (+2)."""
    rng = np.random.default_rng(1)
    for (M, N, K) in [(1, 1, 128), (2, 5, 256), (3, 4, 384), (8, 3, 512)]:
        plane = rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)
        q = rng.integers(-127, 128, size=(M, K), dtype=np.int64).astype(np.int8)
        w = _unpack_numpy(plane)
        ref = np.einsum("mgk,ngk->mng", q.reshape(M, -1, G).astype(np.int64),
                        w.reshape(N, -1, G))
        got = O.group_dots(q, plane, lib=lib)
        assert np.array_equal(got, ref), (M, N, K)


def pin_group_dots_special(lib):
    """All code 1 -> 0; all code 2 -> sum q; all code 0 -> -sum q;
    all code 3 -> 2 sum q (per group)."""
    rng = np.random.default_rng(2)
    q = rng.integers(-127, 128, size=(2, 3 * G)).astype(np.int8)
    T = q.reshape(2, 3, G).astype(np.int64).sum(-1)
    for code, mult in [(1, 0), (2, 1), (0, -1), (3, 2)]:
        plane = _pack(np.full((1, 3 * G), code, np.uint8))
        d = O.group_dots(q, plane, lib=lib)[:, 0, :]
        assert np.array_equal(d, mult * T), code


# -------------------------------------------------------- scale/accumulate
def _dense_fp64(q, sx, plane, scales_bits, K):
    """fp64 reconstruction (KE Test 8 CPU replay): x_hat = q * s_x,
    W = (c - 1) * s_w, y = x_hat @ W^T."""
    M = q.shape[0]
    N = plane.shape[0]
    xh = (q.reshape(M, -1, G).astype(np.float64) * sx[..., None].astype(np.float64)).reshape(M, K)
    sw = scales_bits.view(np.float16).astype(np.float64)
    W = (_unpack_numpy(plane).reshape(N, -1, G) * sw[..., None]).reshape(N, K)
    return xh @ W.T


def pin_pipeline_fp64(lib):
    """Tiny shapes end to end: the oracle's fp64 value matches the fp64 dense
    reconstruction to 1e-12 (the pages' CPU replay tolerance), and its fp32
    sequential value lies inside the accepted bound."""
    rng = np.random.default_rng(4)
    for (M, N, K) in [(1, 1, 128), (2, 5, 256), (3, 4, 384), (3, 5, 384)]:
        codes = rng.integers(0, 3, size=(N, K), dtype=np.uint8)
        plane = _pack(codes)
        sbits = rng.uniform(0.005, 0.05, size=(N, K // G)).astype(np.float16).view(np.uint16)
        x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16)
        a = O.widen(x.view(torch.int16).numpy().view(np.uint16), "bf16", lib=lib)
        assert np.array_equal(a, x.float().numpy())
        q, sx = O.quantize(a, lib=lib)
        dots = O.group_dots(q, plane, lib=lib)
        y32, y64, bound = O.scale_accumulate(dots, sx, sbits, lib=lib)
        ref = _dense_fp64(q, sx, plane, sbits, K)
        assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), (M, N, K)
        ok, _ = O.within_bound(y32, y64, bound)
        assert ok
        assert np.all(bound >= np.abs(y64) * (1 - 1e-12))
        ylin = O.linear(x.view(torch.int16).numpy().view(np.uint16), "bf16", plane, sbits, lib=lib)
        assert np.array_equal(ylin, y32)


def pin_scale_linearity(lib):
    """Doubling every weight scale doubles y32 bit for bit (a power-of-two
    factor commutes with every fp32 rounding); codes all 1 give exact 0."""
    rng = np.random.default_rng(9)
    M, N, K = 2, 3, 512
    plane = _pack(rng.integers(0, 3, size=(N, K), dtype=np.uint8))
    sw = rng.uniform(0.005, 0.05, size=(N, K // G)).astype(np.float16)
    q = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    sx = rng.uniform(0.001, 0.1, size=(M, K // G)).astype(np.float32)
    dots = O.group_dots(q, plane, lib=lib)
    y1, _, _ = O.scale_accumulate(dots, sx, sw.view(np.uint16), lib=lib)
    y2, _, _ = O.scale_accumulate(dots, sx, (sw * np.float16(2)).view(np.uint16), lib=lib)
    assert np.array_equal(y2, y1 * np.float32(2))
    zero = O.group_dots(q, _pack(np.ones((N, K), np.uint8)), lib=lib)
    yz, _, _ = O.scale_accumulate(zero, sx, sw.view(np.uint16), lib=lib)
    assert not yz.any()


def pin_prepare(lib):
    """KE Test 1 prepare_pq2 (separate): bytes 0-1 of each 34-byte block are
    the little-endian fp16 scale, bytes 2..33 the 32 code bytes."""
    N, K = 3, 256
    raw = np.zeros((N, 2 * 34 + 6), np.uint8)      # row stride with padding
    for n in range(N):
        for g in range(2):
            raw[n, g * 34 + 0] = 0x00
            raw[n, g * 34 + 1] = 0x38                # 0x3800 = 0.5
            raw[n, g * 34 + 2:g * 34 + 34] = (np.arange(32) + 40 * n + 7 * g) & 0xFF
    codes, scales = O.prepare(raw, K, lib=lib)
    assert np.all(scales == 0x3800)
    assert O.half_to_float(scales[:1, :1], lib=lib)[0, 0] == 0.5
    for n in range(N):
        for g in range(2):
            assert np.array_equal(codes[n, g * 32:(g + 1) * 32],
                                  (np.arange(32) + 40 * n + 7 * g) & 0xFF)


# ------------------------------------------------------------------ gated
# KE Test 12: the gate/up projection's output is split in halves, gate
# first, and the gated result is silu(gate) * up, silu(v) = v * sigmoid(v).
# Logistic values (sigmoid(v) = 1 / (1 + e^-v)) to double precision:
SIGMOID = {1.0: 0.7310585786300049, 1.5: 0.8175744761936437, -2.0: 0.11920292202211755}


def pin_gated_values(lib):
    """Known logistic values, gate columns before up columns."""
    y = np.array([[1.0, 1.5, -2.0, 2.0, 3.0, 0.5]])
    out = O.gated(y, lib=lib)
    want = [1.0 * SIGMOID[1.0] * 2.0, 1.5 * SIGMOID[1.5] * 3.0, -2.0 * SIGMOID[-2.0] * 0.5]
    assert out.shape == (1, 3)
    assert np.allclose(out[0], want, rtol=1e-15, atol=0), (out, want)


def pin_gated_identities(lib):
    """silu(0) = 0; silu(v) - silu(-v) = v (sigmoid(v) + sigmoid(-v) = 1);
    silu(40) = 40 and |silu(-40)| < 1e-15 to double precision."""
    vs = np.array([0.0, 0.25, 1.0, 3.0, 7.5, 40.0])
    y = np.concatenate([vs, -vs, np.ones(12)])[None, :]
    out = O.gated(y, lib=lib)[0]
    n = len(vs)
    assert out[0] == 0.0 and out[n] == 0.0
    assert np.allclose(out[:n] - out[n:], vs, rtol=1e-14, atol=1e-300), out
    assert out[n - 1] == 40.0 and abs(out[2 * n - 1]) < 1e-15


def pin_gated_end_to_end(lib):
    """Two weight rows through the whole oracle: x = the worked example plus a
    127 (so s_x = 1, q = x), gate row codes [0,1,2,2] (dot 30), up row codes
    [2,2,2,2] (dot 20+30+40+10 = 100), weight scale 0.5: gate = 15, up = 50,
    gated = 15 * sigmoid(15) * 50 with sigmoid(15) = 1 / (1 + 3.059023205018258e-7)."""
    ex = _golden("worked_example.json")
    x = np.zeros((1, G), np.float32)
    x[0, :4] = ex["q"]
    x[0, 4] = 127.0
    q, sx = O.quantize(x, lib=lib)
    codes = np.ones((2, G), np.uint8)
    codes[0, :4] = ex["codes"]
    codes[1, :4] = 2
    dots = O.group_dots(q, _pack(codes), lib=lib)
    _, y64, _ = O.scale_accumulate(dots, sx, np.full((2, 1), _f16_bits(0.5), np.uint16), lib=lib)
    assert list(y64[0]) == [15.0, 50.0], y64
    out = O.gated(y64, lib=lib)
    want = 15.0 / (1.0 + 3.059023205018258e-7) * 50.0
    assert abs(out[0, 0] - want) <= 1e-13, (out, want)


# ------------------------------------------ activation groups (KE Test 9)
def pin_grouped_quantize_scales(lib):
    """A = 64 and 32: each activation group gets its own max|x| / 127.  Group
    maxima 127, 63.5, 31.75 and 100 (a later group larger than an earlier one)
    give s = 1, 1/2, 1/4 and 100/127, and q = x / s."""
    x = np.zeros((1, 128), np.float32)
    x[0, 0:4] = [127.0, 10.0, -3.0, 0.0]
    x[0, 32:35] = [63.5, 5.0, -2.5]
    x[0, 64:66] = [31.75, 1.25]
    x[0, 96:98] = [100.0, 40.0]
    s100 = np.float32(100.0) / np.float32(127.0)
    q64, s64 = O.quantize_grouped(x, 64, lib=lib)
    assert list(s64[0]) == [1.0, s100], s64
    q32, s32 = O.quantize_grouped(x, 32, lib=lib)
    assert list(s32[0]) == [1.0, 0.5, 0.25, s100], s32
    assert list(q32[0, 0:4]) == [127, 10, -3, 0]
    assert list(q32[0, 32:35]) == [127, 10, -5]
    assert list(q32[0, 64:66]) == [127, 5]
    assert list(q32[0, 96:98]) == [127, 51]          # 40 * 127 / 100 = 50.8
    assert list(O.qsum_grouped(q32, 32, lib=lib)[0]) == [134, 132, 132, 178]


def pin_grouped_128_is_the_plain_path(lib):
    """A = 128 reproduces the (separately pinned) ungrouped functions."""
    rng = np.random.default_rng(9)
    M, N, K = 2, 5, 384
    a = (rng.standard_normal((M, K)) * 3).astype(np.float32)
    q1, s1 = O.quantize(a, lib=lib)
    q2, s2 = O.quantize_grouped(a, 128, lib=lib)
    assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
    plane = _pack(rng.integers(0, 3, (N, K)).astype(np.uint8))
    d1 = O.group_dots(q1, plane, lib=lib)
    d2 = O.group_dots_grouped(q1, plane, 128, lib=lib)
    assert np.array_equal(d1, d2)
    sw = rng.uniform(0.005, 0.05, (N, K // G)).astype(np.float16).view(np.uint16)
    y1 = O.scale_accumulate(d1, s1, sw, lib=lib)
    y2 = O.scale_accumulate_grouped(d2, s2, sw, 128, lib=lib)
    assert all(np.array_equal(u, v) for u, v in zip(y1, y2))


def pin_grouped_dots_brute_force(lib):
    """Partial dots against numpy's own decode (int64), and summed over a
    128-group's partials they give the group's dot."""
    rng = np.random.default_rng(4)
    M, N, K = 3, 4, 256
    q = rng.integers(-127, 128, (M, K)).astype(np.int8)
    plane = _pack(rng.integers(0, 3, (N, K)).astype(np.uint8))
    w = _unpack_numpy(plane)
    for A in (64, 32):
        d = O.group_dots_grouped(q, plane, A, lib=lib)
        ref = np.einsum("nk,mk->mnk", w, q.astype(np.int64)).reshape(M, N, K // A, A).sum(-1)
        assert np.array_equal(d, ref), A
        full = O.group_dots(q, plane, lib=lib)
        assert np.array_equal(d.reshape(M, N, K // G, G // A).sum(-1), full), A
        # fp64 scale-accumulate against a dense numpy evaluation: activation
        # group j belongs to weight group j // (128 / A)
        sx = rng.uniform(0.01, 0.1, (M, K // A)).astype(np.float32)
        sw = rng.uniform(0.005, 0.05, (N, K // G)).astype(np.float16)
        _, y64, _ = O.scale_accumulate_grouped(d, sx, sw.view(np.uint16), A, lib=lib)
        wg = sw.astype(np.float64)[:, np.arange(K // A) // (G // A)]
        ref = np.einsum("mnj,mj,nj->mn", d.astype(np.float64), sx.astype(np.float64), wg)
        assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12), A


def pin_grouped_worked_example(lib):
    """The worked example in both halves of a 128-group at A = 64: half 0
    holds x = [20,30,40,10] with a 127 (s = 1, q = x), half 1 holds
    [10,15,20,5] with a 63.5 (s = 1/2, q = [20,30,40,10]); codes [0,1,2,2]
    in both halves give partial dots 30 and 30, and at weight scale 0.5
    y = (30 * 1) * 0.5 + (30 * 0.5) * 0.5 = 22.5."""
    ex = _golden("worked_example.json")
    x = np.zeros((1, G), np.float32)
    x[0, 0:4] = ex["q"]
    x[0, 4] = 127.0
    x[0, 64:68] = np.array(ex["q"], np.float32) / 2
    x[0, 68] = 63.5
    q, sx = O.quantize_grouped(x, 64, lib=lib)
    assert list(sx[0]) == [1.0, 0.5]
    codes = np.ones((1, G), np.uint8)
    codes[0, 0:4] = ex["codes"]
    codes[0, 64:68] = ex["codes"]
    d = O.group_dots_grouped(q, _pack(codes), 64, lib=lib)
    assert list(d[0, 0]) == [ex["dot"], ex["dot"]]
    y32, y64, b = O.scale_accumulate_grouped(d, sx, np.array([[_f16_bits(0.5)]], np.uint16), 64,
                                             lib=lib)
    assert y32[0, 0] == np.float32(22.5) and y64[0, 0] == 22.5 and b[0, 0] == 22.5


# ------------------------------------------- fused preparation (KE Test 18)
def _walsh(k: int) -> np.ndarray:
    """Column k of the Sylvester Hadamard matrix of order 1024: entry j is
    (-1)^popcount(j & k)."""
    j = np.arange(1024)
    bits = np.array([bin(v).count("1") for v in (j & k)])
    return np.where(bits % 2 == 0, 1.0, -1.0)


def _bf16_bits(values) -> np.ndarray:
    return synth_bits(np.asarray(values, np.float32))


def synth_bits(a: np.ndarray) -> np.ndarray:
    """bf16 bits of fp32 values that bf16 represents exactly."""
    b = np.ascontiguousarray(a, np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "not exact in bf16"
    return (b >> 16).astype(np.uint16)


def pin_fwht_columns(lib):
    """H e_k = column k of the Sylvester matrix / 32 (closed form)."""
    for k in (0, 1, 5, 513, 1023):
        e = np.zeros(1024, np.float32)
        e[k] = 1.0
        assert np.array_equal(O.fwht1024(e, lib=lib), (_walsh(k) / 32.0).astype(np.float32)), k


def pin_fwht_involution(lib):
    """The orthonormal transform is its own inverse; for small integers every
    partial sum is exact, so H(H(v)) == v bit for bit."""
    v = (np.arange(1024) * 37 % 201 - 100).astype(np.float32)
    assert np.array_equal(O.fwht1024(O.fwht1024(v, lib=lib), lib=lib), v)


def pin_sumsq_structure(lib):
    """2048 strided fp32 partials, then a tree: with h[0]^2 = 2^24 and
    h[1], h[2], h[3] = 1 the tree adds 1 + 1 before meeting 2^24 and keeps
    2^24 + 2; a sequential fp32 sum would round each +1 away (2^24).  The
    squares of small integers sum exactly otherwise."""
    h = np.zeros(4096, np.float32)
    h[0], h[1], h[2], h[3] = 4096.0, 1.0, 1.0, 1.0
    assert O.sumsq2048(h, lib=lib) == 16777218.0
    g = (np.arange(5120) % 7).astype(np.float32)
    assert O.sumsq2048(g, lib=lib) == float(np.sum((np.arange(5120) % 7) ** 2))


def pin_norm_hadamard_constant_row(lib):
    """x = 3, residual = -1 (h = 2), w = 0, signs +1, eps = 0, K = 2048:
    mean h^2 = 4, inv = 1/2, n = 1; the transform of a constant block is
    32 e_0, so each 1024-block quantises to q = 127 at its first element
    (s_x = 32/127) and zeros elsewhere (s_x = 0); the residual output is 2."""
    K = 2048
    x = _bf16_bits(np.full((1, K), 3.0))
    r = _bf16_bits(np.full((1, K), -1.0))
    w = _bf16_bits(np.zeros(K))
    q, sx, nb, rb = O.norm_hadamard_quantize(x, r, w, np.ones(K, np.int8), 0.0, lib=lib)
    assert np.all(nb == _bf16_bits([1.0])[0]) and np.all(rb == _bf16_bits([2.0])[0])
    want = np.zeros((1, K), np.int8)
    want[0, 0] = want[0, 1024] = 127
    assert np.array_equal(q, want), np.nonzero(q)
    s = np.zeros((1, K // G), np.float32)
    s[0, 0] = s[0, 8] = np.float32(32.0) / np.float32(127.0)
    assert np.array_equal(sx, s), sx


def pin_norm_hadamard_sign_pattern(lib):
    """Signs equal to Walsh function k and a constant row: v = column k, and
    its transform is 32 e_k, so q = 127 exactly at element k; the norm
    weight enters as w + 1 (w = 0.5 gives n = 1.5 for h * inv = 1)."""
    K, k = 1024, 300
    x = _bf16_bits(np.full((1, K), 1.0))
    w = _bf16_bits(np.full(K, 0.5))
    sign = _walsh(k).astype(np.int8)
    q, sx, nb, _ = O.norm_hadamard_quantize(x, None, w, sign, 0.0, lib=lib)
    assert np.all(nb == _bf16_bits([1.5])[0])
    want = np.zeros((1, K), np.int8)
    want[0, k] = 127
    assert np.array_equal(q, want), np.nonzero(q)
    assert sx[0, k // G] == np.float32(48.0) / np.float32(127.0)


def pin_norm_eps(lib):
    """eps enters under the root: x = 1, eps = 3 gives inv = 1/2, n = 0.5."""
    K = 1024
    x = _bf16_bits(np.full((1, K), 1.0))
    w = _bf16_bits(np.zeros(K))
    _, _, nb, _ = O.norm_hadamard_quantize(x, None, w, np.ones(K, np.int8), 3.0, lib=lib)
    assert np.all(nb == _bf16_bits([0.5])[0])


# -------------------------------------------------- PTQ1_0 weights (KR)
# Page "KERNEL_REPORT: PTQ1_0 small-batch decoding on the PrismML fork, RTX
# 3060 12GB" (KR), "What the source said": 28-byte blocks of 128 weights,
# 24 qs bytes of five trits, 2 qh bytes with 8 more trits, fp16 d last.

def _ptq_byte(trits) -> int:
    """The byte whose repeated x3 expansion gives `trits` (first trit most
    significant): the base-3 fraction 0.t0t1t2t3t4 rounded up to 1/256ths,
    ceil(256 V / 243) with V the base-3 value of the five trits."""
    t = list(trits) + [0] * (5 - len(trits))
    V = sum(d * 3 ** (4 - i) for i, d in enumerate(t))
    return (256 * V + 242) // 243


def _ptq_position(k: int):
    """Reading taken for the weight order: trit n of qs byte j is weight
    24n + j; trit n of qh byte j is weight 120 + 2n + j.  -> (byte, trit)."""
    if k < 120:
        return k % 24, k // 24
    return 24 + (k - 120) % 2, (k - 120) // 2


def _ptq_block(trits128, d_bits: int) -> np.ndarray:
    """28 bytes for one block from 128 trits (0..2) and an fp16 bit pattern."""
    per_byte = [[0] * 5 for _ in range(26)]
    for k in range(G):
        b, n = _ptq_position(k)
        per_byte[b][n] = int(trits128[k])
    blk = np.zeros(28, np.uint8)
    for b in range(26):
        blk[b] = _ptq_byte(per_byte[b])
    blk[26], blk[27] = d_bits & 0xFF, d_bits >> 8
    return blk


def pin_ptq_trit_closed_form(lib):
    """Trit n of byte b is the (n+1)-th base-3 digit of the fraction b/256,
    floor(b * 3^(n+1) / 256) mod 3, for every byte and level; and every
    five-trit value V comes back from its byte ceil(256 V / 243)."""
    for b in range(256):
        for n in range(5):
            assert O.ptq_trit(b, n, lib=lib) == (b * 3 ** (n + 1) // 256) % 3, (b, n)
    for V in range(243):
        digits = [(V // 3 ** (4 - i)) % 3 for i in range(5)]
        b = _ptq_byte(digits)
        assert [O.ptq_trit(b, n, lib=lib) for n in range(5)] == digits, V


def pin_ptq_weight_positions(lib):
    """A block with one +1 weight (trit 2) at k and 0 (trit 1) elsewhere
    unpacks to the unit vector e_k, for every k; the scale is bytes 26-27."""
    raw = np.stack([_ptq_block(np.where(np.arange(G) == k, 2, 1), 0x3C00 + k) for k in range(G)])
    codes, scales = O.ptq_unpack(raw, G, lib=lib)
    w = _unpack_numpy(codes)
    assert np.array_equal(w, np.eye(G, dtype=np.int64)), np.argwhere(w != np.eye(G))[:4]
    assert list(scales[:, 0]) == [0x3C00 + k for k in range(G)]


def pin_ptq_random_blocks(lib):
    """Random trits through independently built blocks (three rows of three
    blocks, rows padded to a longer stride) come back as code = trit."""
    rng = np.random.default_rng(21)
    N, K = 3, 384
    trits = rng.integers(0, 3, (N, K))
    dbits = rng.integers(0, 0x7C00, (N, K // G))
    raw = np.zeros((N, 3 * 28 + 5), np.uint8)
    for n in range(N):
        for g in range(K // G):
            raw[n, 28 * g:28 * g + 28] = _ptq_block(trits[n, g * G:(g + 1) * G], int(dbits[n, g]))
    codes, scales = O.ptq_unpack(raw, K, lib=lib)
    assert np.array_equal(_unpack_numpy(codes), trits - 1)
    assert np.array_equal(scales, dbits.astype(np.uint16))


def pin_ptq_worked_example(lib):
    """BIB 'Calculate with small integers' in PTQ1_0 form: weights
    [-1, 0, +1, +1] at k = 0..3, d = 0.5, x = [20, 30, 40, 10, 127, 0...]:
    y = 15 with activation groups of 128 and of 32; all-(+1) and all-(-1)
    blocks give +sum(q) and -sum(q)."""
    ex = _golden("worked_example.json")
    trits = np.ones(G, np.int64)
    trits[:4] = ex["codes"]
    raw = _ptq_block(trits, _f16_bits(0.5))[None, :]
    codes, scales = O.ptq_unpack(raw, G, lib=lib)
    x = np.zeros((1, G), np.float32)
    x[0, :4] = ex["q"]
    x[0, 4] = 127.0
    for A in (128, 32):
        q, sx = O.quantize_grouped(x, A, lib=lib)
        d = O.group_dots_grouped(q, codes, A, lib=lib)
        _, y64, _ = O.scale_accumulate_grouped(d, sx, scales, A, lib=lib)
        assert y64[0, 0] == 15.0, (A, y64)
    q = np.random.default_rng(2).integers(-127, 128, (1, G)).astype(np.int8)
    for t, sign in ((2, 1), (0, -1)):
        c, _ = O.ptq_unpack(_ptq_block(np.full(G, t), 0)[None, :], G, lib=lib)
        assert O.group_dots(q, c, lib=lib)[0, 0, 0] == sign * int(q.astype(np.int64).sum())


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
