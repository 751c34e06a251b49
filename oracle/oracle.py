"""ctypes marshalling for the C oracle in ``pq2_oracle.c``.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Every function here
converts numpy arrays, calls the matching ``orc_*`` C function and returns
numpy arrays; none of the method's arithmetic is done in Python except the
acceptance checks (``within_bound`` / ``bf16_within_bound``), which state the
error bound of the scale-accumulate step:
  |y - y64| <= 1e-5 * B,  B = sum_g |s_x * s_w * dot_g|            (fp32 out)
  |y - y64| <= 1e-5 * B * (1 + 2^-8) + 2^-8 * |y64|                (bf16 out)
and of the gated output (``gated_within_bound``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pq2_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None

GROUP = 128
KIND = {"bf16": 0, "f16": 1, "f32": 2}


def build_oracle(force: bool = False, extra_flags=()) -> str:
    """Compile pq2_oracle.c with gcc into oracle/liboracle.so (if stale)."""
    out = _LIB_PATH if not extra_flags else os.path.join(
        _HERE, "liboracle_" + "_".join(f.strip("-").replace("=", "") for f in extra_flags) + ".so")
    stale = (not os.path.exists(out)
             or os.path.getmtime(out) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, *extra_flags, _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) the oracle library and declare signatures."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build_oracle())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        sigs = {
            "orc_decode_field": (I, [ctypes.c_uint8, I]),
            "orc_half_to_float": (ctypes.c_float, [ctypes.c_uint16]),
            "orc_bf16_to_float": (ctypes.c_float, [ctypes.c_uint16]),
            "orc_float_to_bf16_rne": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_prepare": (None, [P, I64, I64, I64, P, P]),
            "orc_ptq_trit": (I, [ctypes.c_uint8, I]),
            "orc_ptq_unpack": (None, [P, I64, I64, I64, P, P]),
            "orc_decode_matrix": (None, [P, I64, I64, P]),
            "orc_quantize": (None, [P, I64, I64, P, P]),
            "orc_widen": (None, [P, I, I64, I64, I64, P]),
            "orc_q_planes": (None, [P, I64, I64, P]),
            "orc_qsum": (None, [P, I64, I64, P]),
            "orc_group_dots": (None, [P, P, I64, I64, I64, P]),
            "orc_scale_accumulate": (None, [P, P, P, I64, I64, I64, P, P, P]),
            "orc_linear": (None, [P, I, I64, I64, I64, I64, P, P, P, P, P, P, P]),
            "orc_gated": (None, [P, I64, I64, P]),
            "orc_quantize_grouped": (None, [P, I64, I64, I, P, P]),
            "orc_qsum_grouped": (None, [P, I64, I64, I, P]),
            "orc_group_dots_grouped": (None, [P, P, I64, I64, I64, I, P]),
            "orc_scale_accumulate_grouped": (None, [P, P, P, I64, I64, I64, I, P, P, P]),
            "orc_fwht1024": (None, [P]),
            "orc_sumsq2048": (ctypes.c_float, [P, I64]),
            "orc_norm_hadamard_quantize": (None, [P, P, P, P, ctypes.c_float, I64, I64,
                                                  P, P, P, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


# ------------------------------------------------------------------ scalars
def decode_field(byte: int, field: int, lib=None) -> int:
    return (lib or load()).orc_decode_field(byte, field)


def half_to_float(bits: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.orc_half_to_float(int(b)) for b in np.asarray(bits).ravel()],
                    dtype=np.float32).reshape(np.shape(bits))


def bf16_to_float(bits: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.orc_bf16_to_float(int(b)) for b in np.asarray(bits).ravel()],
                    dtype=np.float32).reshape(np.shape(bits))


def float_to_bf16_rne(values: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    vals = np.asarray(values, dtype=np.float32)
    return np.array([lib.orc_float_to_bf16_rne(float(v)) for v in vals.ravel()],
                    dtype=np.uint16).reshape(vals.shape)


# ------------------------------------------------------------- preparation
def prepare(raw: np.ndarray, K: int, lib=None):
    """raw u8[N][>= K/128*34] -> (codes u8[N][K/4], scales u16[N][K/128])."""
    lib = lib or load()
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    N = raw.shape[0]
    codes = np.empty((N, K // 4), np.uint8)
    scales = np.empty((N, K // GROUP), np.uint16)
    lib.orc_prepare(_p(raw), raw.shape[1], N, K, _p(codes), _p(scales))
    return codes, scales


def decode_matrix(codes: np.ndarray, K: int, lib=None) -> np.ndarray:
    lib = lib or load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    w = np.empty((codes.shape[0], K), np.int8)
    lib.orc_decode_matrix(_p(codes), codes.shape[0], K, _p(w))
    return w


def ptq_trit(byte: int, level: int, lib=None) -> int:
    lib = lib or load()
    return int(lib.orc_ptq_trit(byte, level))


def ptq_unpack(raw: np.ndarray, K: int, lib=None):
    """PTQ1_0 rows u8[N][>= K/128*28] -> (code plane u8[N][K/4] with code =
    trit, fp16 scale bits u16[N][K/128])."""
    lib = lib or load()
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    N = raw.shape[0]
    codes = np.empty((N, K // 4), np.uint8)
    scales = np.empty((N, K // GROUP), np.uint16)
    lib.orc_ptq_unpack(_p(raw), raw.shape[1], N, K, _p(codes), _p(scales))
    return codes, scales


# ------------------------------------------------------------ quantisation
def widen(x_bits: np.ndarray, kind: str, lib=None) -> np.ndarray:
    """bf16/f16 bit patterns (u16) or f32 values -> f32 [M][K]."""
    lib = lib or load()
    x = np.ascontiguousarray(x_bits)
    M, K = x.shape
    a = np.empty((M, K), np.float32)
    lib.orc_widen(_p(x), KIND[kind], K, M, K, _p(a))
    return a


def quantize(a: np.ndarray, lib=None):
    """f32 a[M][K] -> (q i8[M][K], sx f32[M][K/128])."""
    lib = lib or load()
    a = np.ascontiguousarray(a, dtype=np.float32)
    M, K = a.shape
    q = np.empty((M, K), np.int8)
    sx = np.empty((M, K // GROUP), np.float32)
    lib.orc_quantize(_p(a), M, K, _p(q), _p(sx))
    return q, sx


def q_planes(q: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    qp = np.empty_like(q)
    lib.orc_q_planes(_p(q), q.shape[0], q.shape[1], _p(qp))
    return qp


def qsum(q: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    T = np.empty((q.shape[0], q.shape[1] // GROUP), np.int32)
    lib.orc_qsum(_p(q), q.shape[0], q.shape[1], _p(T))
    return T


# ----------------------------------------------------------- matmul pieces
def group_dots(q: np.ndarray, codes: np.ndarray, lib=None) -> np.ndarray:
    """q i8[M][K], codes u8[N][K/4] -> int32 dots[M][N][K/128]."""
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    M, K = q.shape
    N = codes.shape[0]
    dots = np.empty((M, N, K // GROUP), np.int32)
    lib.orc_group_dots(_p(q), _p(codes), M, N, K, _p(dots))
    return dots


def scale_accumulate(dots: np.ndarray, sx: np.ndarray, scales: np.ndarray,
                     lib=None):
    """-> (y32 f32[M][N], y64 f64[M][N], bound f64[M][N])."""
    lib = lib or load()
    dots = np.ascontiguousarray(dots, dtype=np.int32)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    M, N, G = dots.shape
    y32 = np.empty((M, N), np.float32)
    y64 = np.empty((M, N), np.float64)
    bound = np.empty((M, N), np.float64)
    lib.orc_scale_accumulate(_p(dots), _p(sx), _p(scales), M, N, G * GROUP,
                             _p(y32), _p(y64), _p(bound))
    return y32, y64, bound


def linear(x_bits: np.ndarray, kind: str, codes: np.ndarray,
           scales: np.ndarray, lib=None) -> np.ndarray:
    """Whole path (widen, quantise, group dots, scale) -> y32 f32[M][N]."""
    lib = lib or load()
    x = np.ascontiguousarray(x_bits)
    M, K = x.shape
    N = codes.shape[0]
    a = np.empty((M, K), np.float32)
    q = np.empty((M, K), np.int8)
    sx = np.empty((M, K // GROUP), np.float32)
    dots = np.empty((M, N, K // GROUP), np.int32)
    y = np.empty((M, N), np.float32)
    lib.orc_linear(_p(x), KIND[kind], K, M, N, K, _p(np.ascontiguousarray(codes)),
                   _p(np.ascontiguousarray(scales)), _p(a), _p(q), _p(sx),
                   _p(dots), _p(y))
    return y


def quantize_grouped(a: np.ndarray, A: int, lib=None):
    """f32 a[M][K], activation group A (128, 64, 32) -> (q i8[M][K],
    sx f32[M][K/A])."""
    lib = lib or load()
    a = np.ascontiguousarray(a, dtype=np.float32)
    M, K = a.shape
    q = np.empty((M, K), np.int8)
    sx = np.empty((M, K // A), np.float32)
    lib.orc_quantize_grouped(_p(a), M, K, A, _p(q), _p(sx))
    return q, sx


def group_dots_grouped(q: np.ndarray, codes: np.ndarray, A: int, lib=None) -> np.ndarray:
    """q i8[M][K], codes u8[N][K/4] -> int32 partial dots [M][N][K/A]."""
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    M, K = q.shape
    N = codes.shape[0]
    dots = np.empty((M, N, K // A), np.int32)
    lib.orc_group_dots_grouped(_p(q), _p(codes), M, N, K, A, _p(dots))
    return dots


def scale_accumulate_grouped(dots: np.ndarray, sx: np.ndarray, scales: np.ndarray, A: int,
                             lib=None):
    """-> (y32 f32[M][N], y64 f64[M][N], bound f64[M][N])."""
    lib = lib or load()
    dots = np.ascontiguousarray(dots, dtype=np.int32)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    M, N, GA = dots.shape
    K = GA * A
    y32 = np.empty((M, N), np.float32)
    y64 = np.empty((M, N), np.float64)
    bound = np.empty((M, N), np.float64)
    lib.orc_scale_accumulate_grouped(_p(dots), _p(sx), _p(scales), M, N, K, A, _p(y32),
                                     _p(y64), _p(bound))
    return y32, y64, bound


def qsum_grouped(q: np.ndarray, A: int, lib=None) -> np.ndarray:
    """Sum of q over each A-group, int32 [M][K/A]."""
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    M, K = q.shape
    T = np.empty((M, K // A), np.int32)
    lib.orc_qsum_grouped(_p(q), M, K, A, _p(T))
    return T


def gated(y64: np.ndarray, lib=None) -> np.ndarray:
    """y64 f64[M][N] (gate columns, then up columns) -> silu(gate) * up,
    f64[M][N/2]."""
    lib = lib or load()
    y64 = np.ascontiguousarray(y64, dtype=np.float64)
    M, N = y64.shape
    out = np.empty((M, N // 2), np.float64)
    lib.orc_gated(_p(y64), M, N, _p(out))
    return out


def fwht1024(v: np.ndarray, lib=None) -> np.ndarray:
    """Orthonormal 1024-point Walsh-Hadamard transform (fp32), a copy."""
    lib = lib or load()
    out = np.ascontiguousarray(v, dtype=np.float32).copy()
    assert out.shape == (1024,)
    lib.orc_fwht1024(_p(out))
    return out


def sumsq2048(h: np.ndarray, lib=None) -> float:
    """Sum of squares in the 2048-partial reduction structure (fp32)."""
    lib = lib or load()
    h = np.ascontiguousarray(h, dtype=np.float32)
    return float(lib.orc_sumsq2048(_p(h), h.shape[0]))


def norm_hadamard_quantize(x_bits: np.ndarray, residual_bits, w_bits: np.ndarray,
                           sign: np.ndarray, eps: float, lib=None):
    """bf16 x [M][K] (bits), optional bf16 residual (bits), bf16 norm weight
    w [K] (bits, applied as w + 1), sign [K] (+1/-1), eps ->
    (q i8[M][K], sx f32[M][K/128], norm bits u16[M][K], residual-out bits
    u16[M][K] or None)."""
    lib = lib or load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x.shape
    r = None if residual_bits is None else np.ascontiguousarray(residual_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    sg = np.ascontiguousarray(sign, dtype=np.int8)
    q = np.empty((M, K), np.int8)
    sx = np.empty((M, K // GROUP), np.float32)
    nb = np.empty((M, K), np.uint16)
    rb = np.empty((M, K), np.uint16) if r is not None else None
    lib.orc_norm_hadamard_quantize(_p(x), None if r is None else _p(r), _p(w), _p(sg),
                                   ctypes.c_float(eps), M, K, _p(nb),
                                   None if rb is None else _p(rb), _p(q), _p(sx))
    return q, sx, nb, rb


# --------------------------------------------------------- acceptance rules
REL_BOUND = 1e-5


def within_bound(y: np.ndarray, y64: np.ndarray, bound: np.ndarray):
    """fp32 output rule: |y - y64| <= 1e-5 * B (elementwise). Returns
    (ok, worst ratio |y-y64| / (1e-5*B), with 0/0 counted as 0)."""
    err = np.abs(np.asarray(y, np.float64) - y64)
    lim = REL_BOUND * bound
    ratio = np.where(lim > 0, err / np.where(lim > 0, lim, 1.0),
                     np.where(err > 0, np.inf, 0.0))
    return bool(np.all(err <= lim)), float(ratio.max(initial=0.0))


def bf16_within_bound(y: np.ndarray, y64: np.ndarray, bound: np.ndarray):
    """bf16 output rule: the fp32 result y32 obeys |y32 - y64| <= 1e-5*B and
    round-to-nearest-even to bf16 moves it by at most half an ulp,
    2^-8*|y32| <= 2^-8*(|y64| + 1e-5*B).  Hence
    |y - y64| <= 1e-5*B*(1 + 2^-8) + 2^-8*|y64|."""
    err = np.abs(np.asarray(y, np.float64) - y64)
    lim = REL_BOUND * bound * (1.0 + 2.0 ** -8) + np.abs(y64) * 2.0 ** -8
    ratio = np.where(lim > 0, err / np.where(lim > 0, lim, 1.0),
                     np.where(err > 0, np.inf, 0.0))
    return bool(np.all(err <= lim)), float(ratio.max(initial=0.0))


SILU_SLOPE = 1.1  # max |d silu / dx| = 1.09984, at x ~ 2.3994
GATED_ROUND = 2.0 ** -20  # fp32 expf (2 ulp), add, divide, multiply: <= 1.75 * 2^-22


def gated_bound(y64: np.ndarray, bound: np.ndarray) -> np.ndarray:
    """Error bound of an fp32 gated output silu(g) * u whose g and u obey
    the fp32 output rule |g - g64| <= Bg = 1e-5 * B_gate, |u - u64| <= Bu:
      |silu(g) u - silu(g64) u64| <= SILU_SLOPE * Bg * (|u64| + Bu)
                                     + |silu(g64)| * Bu                  (E)
    plus the fp32 rounding of silu and the product, relative <= 2^-20 of
    (|out64| + E).  Returns that bound, f64[M][N/2]."""
    M, N = y64.shape
    I = N // 2
    g, u = y64[:, :I], y64[:, I:]
    bg, bu = REL_BOUND * bound[:, :I], REL_BOUND * bound[:, I:]
    silu = g / (1.0 + np.exp(-g))
    e = SILU_SLOPE * bg * (np.abs(u) + bu) + np.abs(silu) * bu
    return e + GATED_ROUND * (np.abs(silu * u) + e)


def gated_within_bound(out: np.ndarray, out64: np.ndarray, gbound: np.ndarray,
                       bf16: bool = False):
    """|out - out64| <= gbound (fp32), or + 2^-8 * (|out64| + gbound) for a
    bf16 output (round to nearest even).  Returns (ok, worst ratio)."""
    err = np.abs(np.asarray(out, np.float64) - out64)
    lim = gbound + (2.0 ** -8 * (np.abs(out64) + gbound) if bf16 else 0.0)
    ratio = np.where(lim > 0, err / np.where(lim > 0, lim, 1.0),
                     np.where(err > 0, np.inf, 0.0))
    return bool(np.all(err <= lim)), float(ratio.max(initial=0.0))
