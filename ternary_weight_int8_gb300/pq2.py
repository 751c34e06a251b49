"""Thin Python binding of libpq2 (ctypes).  Argument marshalling only: every
step of the path runs in the library's CUDA kernels.  torch supplies device
memory and streams.  There is no fallback: if libpq2.so is missing or a call
fails, an exception is raised.

Two levels:
  * ``lib()`` — the raw C functions with their exact C signatures (pointers
    as integers), used by tests that exercise the C ABI directly;
  * ``pq2_prepare``, ``pq2_quantize_act``, ``pq2_mmv``, ``pq2_mm``,
    ``pq2_debug_group_dots`` — the same names taking torch tensors, allocating
    outputs with torch when not given, and passing the current torch stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpq2.so")

PQ2_OK, PQ2_ERR_NULL, PQ2_ERR_SHAPE, PQ2_ERR_ALIGN, PQ2_ERR_DTYPE = 0, 1, 2, 3, 4
PQ2_ERR_ARCH, PQ2_ERR_LAUNCH, PQ2_ERR_TIMEOUT, PQ2_ERR_CUDA = 5, 6, 7, 8
PQ2_BF16, PQ2_F16, PQ2_F32 = 0, 1, 2
PQ2_Q_ROWS, PQ2_Q_PLANES, PQ2_Q_F16, PQ2_Q_F8, PQ2_Q_MMV16 = 0, 1, 2, 3, 4
PQ2_DECODE_ADDXOR, PQ2_DECODE_PLANES = 0, 1
PQ2_PATH_MMV_ADDXOR, PQ2_PATH_MM, PQ2_PATH_MMV_PLANES, PQ2_PATH_MM_F8, PQ2_PATH_MMV_TC = \
    0, 1, 2, 3, 4
PQ2_MMV_OVERLAP_WEIGHTS, PQ2_MMV_INDEPENDENT = 1, 2
PQ2_STATIC_SCRATCH_BYTES = 1 << 20
GROUP = 128

# C signatures, mirroring include/pq2.h.
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
SIGNATURES = {
    "pq2_layout_version": (_I, []),
    "pq2_status_string": (ctypes.c_char_p, [_I]),
    "pq2_prepared_bytes": (_SZ, [_I64, _I64]),
    "pq2_prepare": (_I, [_P, _I64, _I64, _I64, _P, _P, _P]),
    "pq2_quantize_act": (_I, [_P, _I, _I64, _I64, _I64, _P, _I, _P, _P, _P]),
    "pq2_mmv": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _P]),
    "pq2_mmv_ex": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _I, _P, _P]),
    "pq2_mmv_tc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _P, _P]),
    "pq2_linear_tensor_gemv": (_I, [_I64, _I64, _I64, _I]),
    "pq2_linear": (_I, [_P, _I, _I64, _I64, _I64, _I64, _P, _P, _P, _I, _P, _SZ, _P, _P]),
    "pq2_linear_workspace_bytes": (_SZ, [_I64, _I64]),
    "pq2_linear_static": (_I, [_P, _I, _I64, _I64, _I64, _I64, _P, _P, _P, _I, _P, _P]),
    "pq2_mmv_gated": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _P, _P]),
    "pq2_quantize_act_grouped": (_I, [_P, _I, _I64, _I64, _I64, _I, _P, _I, _P, _P, _P]),
    "pq2_ptq_prepare": (_I, [_P, _I64, _I64, _I64, _P, _P, _P]),
    "pq2_ptq_linear_workspace_bytes": (_SZ, [_I64, _I64, _I]),
    "pq2_ptq_linear": (_I, [_P, _I, _I64, _I64, _I64, _I64, _P, _P, _I, _P, _I, _P, _SZ, _P]),
    "pq2_ptq_mmv": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _I, _P]),
    "pq2_debug_ptq_dots": (_I, [_P, _P, _P, _P, _I64, _I64, _I64, _I, _P, _P]),
    "pq2_mmv_grouped": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _I, _P, _P]),
    "pq2_debug_group_dots_grouped": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _P, _P, _P]),
    "pq2_norm_hadamard_quantize": (_I, [_P, _P, _P, _P, _P, ctypes.c_float, _I64, _I64, _P,
                                        _P, _I, _P, _P, _P]),
    "pq2_linear_gated": (_I, [_P, _I, _I64, _I64, _I64, _I64, _P, _P, _P, _I, _P, _SZ, _P, _P]),
    "pq2_mmv_decoder": (_I, [_I64]),
    "pq2_mm": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _P]),
    "pq2_mm_f8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _P]),
    "pq2_debug_group_dots": (_I, [_P, _P, _P, _I64, _I64, _I64, _I, _P, _P, _P]),
    "pq2_mm_grouped": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _P, _P]),
    "pq2_mm_f8_grouped": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _P, _P]),
    "pq2_debug_mm_dots_grouped": (_I, [_P, _I, _P, _I64, _I64, _I64, _I, _P, _P, _P]),
    "pq2_linear_grouped_workspace_bytes": (_SZ, [_I64, _I64, _I]),
    "pq2_linear_grouped": (_I, [_P, _I, _I64, _I64, _I64, _I64, _P, _P, _I, _P, _I, _P, _SZ, _P,
                                _P]),
    "pq2_mmv_geometry": (_I, [_I64, _I64, _I, _P, _P, _P, _P]),
    "pq2_debug_mmv_drop_arrival": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I64, _P,
                                        _P]),
}

_lock = threading.Lock()
_lib = None


class Pq2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().pq2_status_string(status).decode()
        super().__init__(f"{fn} failed with status {status}: {msg}")


def lib():
    """Load libpq2.so (it must have been built, see build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"libpq2.so not found at {LIB_PATH}; build it with "
                    "`python -m ternary_weight_int8_gb300.build`")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def _check(fn: str, status: int):
    if status != PQ2_OK:
        raise Pq2Error(fn, status)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


_DT = {torch.bfloat16: PQ2_BF16, torch.float16: PQ2_F16, torch.float32: PQ2_F32}


def prepared_bytes(N: int, K: int) -> int:
    return lib().pq2_prepared_bytes(N, K)


def pq2_prepare(raw: torch.Tensor, K: int, codes=None, scales=None, stream=None):
    """Raw blocks u8[N][>=K/128*34] (CUDA) -> (codes u8[N][K/4], scales fp16[N][K/128])."""
    N = raw.shape[0]
    if raw.dtype != torch.uint8 or raw.dim() != 2 or raw.stride(1) != 1:
        raise ValueError("raw must be a 2-D uint8 tensor with unit column stride")
    if codes is None:
        codes = torch.empty((N, K // 4), dtype=torch.uint8, device=raw.device)
    if scales is None:
        scales = torch.empty((N, K // GROUP), dtype=torch.float16, device=raw.device)
    _check("pq2_prepare", lib().pq2_prepare(_ptr(raw), raw.stride(0), N, K, _ptr(codes),
                                            _ptr(scales), _stream(stream)))
    return codes, scales


def pq2_quantize_act(x: torch.Tensor, layout: int = PQ2_Q_PLANES, q=None, sx=None,
                     qsum=None, want_qsum: bool = True, stream=None):
    """x[M][K] (bf16/f16/f32, CUDA, unit column stride) -> (q, sx, qsum)."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    if q is None:
        q = q_buffer(M, K, layout, x.device)
    if sx is None:
        sx = torch.empty((M, K // GROUP), dtype=torch.float32, device=x.device)
    if qsum is None and want_qsum:
        qsum = torch.empty((M, K // GROUP), dtype=torch.int32, device=x.device)
    _check("pq2_quantize_act",
           lib().pq2_quantize_act(_ptr(x), _DT[x.dtype], x.stride(0), M, K, _ptr(q), layout,
                                  _ptr(sx), _ptr(qsum), _stream(stream)))
    return q, sx, qsum


def pq2_mmv(q_planes, sx, qsum, codes, scales, y=None, out_dtype=torch.float32,
            decode=None, flags=0, status=None, stream=None):
    """Small-batch GEMV, M = 1..8: y[M][N] = sum_g dot * s_x * s_w."""
    M, K = q_planes.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=q_planes.device)
    yd = _DT[y.dtype]
    args = (_ptr(q_planes), _ptr(sx), _ptr(qsum), _ptr(codes), _ptr(scales), _ptr(y), yd, M,
            N, K)
    if decode is None and not flags:
        st = lib().pq2_mmv(*args, _ptr(status), _stream(stream))
    else:
        dec = mmv_decoder(M) if decode is None else decode
        st = lib().pq2_mmv_ex(*args, dec, flags, _ptr(status), _stream(stream))
    _check("pq2_mmv", st)
    return y


def pq2_mmv_tc(q_mmv16, sx, qcorr, codes, scales, y=None, out_dtype=torch.float32, flags=0,
               status=None, stream=None):
    """Small-batch GEMV on the tensor-core path, M = 1..8, q from
    pq2_quantize_act(PQ2_Q_MMV16) and its corrections; same bits as pq2_mmv."""
    M, K = q_mmv16.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=q_mmv16.device)
    _check("pq2_mmv_tc", lib().pq2_mmv_tc(_ptr(q_mmv16), _ptr(sx), _ptr(qcorr), _ptr(codes),
                                          _ptr(scales), _ptr(y), _DT[y.dtype], M, N, K, flags,
                                          _ptr(status), _stream(stream)))
    return y


def linear_workspace_bytes(M: int, K: int) -> int:
    return lib().pq2_linear_workspace_bytes(M, K)


def pq2_linear(x, codes, scales, y=None, out_dtype=torch.float32, workspace=None,
               status=None, stream=None):
    """Complete projection: quantise x, then the GEMV for M = 1..8 (streaming
    its weights while the quantisation runs) or the prefill GEMM from M = 9."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    wb = linear_workspace_bytes(M, K)
    if workspace is None:
        workspace = torch.empty(wb, dtype=torch.uint8, device=x.device)
    _check("pq2_linear", lib().pq2_linear(
        _ptr(x), _DT[x.dtype], x.stride(0), M, N, K, _ptr(codes), _ptr(scales), _ptr(y),
        _DT[y.dtype], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream)))
    return y


def pq2_quantize_act_grouped(x: torch.Tensor, act_group: int, layout: int = PQ2_Q_PLANES,
                             stream=None):
    """x[M][K] -> (q, sx [M][K/A], qsum [M][K/A]) with activation groups of A."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    q = q_buffer(M, K, layout, x.device)
    sx = torch.empty((M, K // act_group), dtype=torch.float32, device=x.device)
    qsum = torch.empty((M, K // act_group), dtype=torch.int32, device=x.device)
    _check("pq2_quantize_act_grouped", lib().pq2_quantize_act_grouped(
        _ptr(x), _DT[x.dtype], x.stride(0), M, K, act_group, _ptr(q), layout, _ptr(sx),
        _ptr(qsum), _stream(stream)))
    return q, sx, qsum


def pq2_mmv_grouped(q_planes, sx, qsum, codes, scales, act_group: int, y=None,
                    out_dtype=torch.float32, flags=0, status=None, stream=None):
    """GEMV with activation groups of A (M = 1..4)."""
    M, K = q_planes.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=q_planes.device)
    _check("pq2_mmv_grouped", lib().pq2_mmv_grouped(
        _ptr(q_planes), _ptr(sx), _ptr(qsum), _ptr(codes), _ptr(scales), _ptr(y), _DT[y.dtype],
        M, N, K, act_group, flags, _ptr(status), _stream(stream)))
    return y


def pq2_debug_group_dots_grouped(q_planes, qsum, codes, act_group: int, stream=None):
    """Exact partial dots [M][N][K/A] of the grouped GEMV's device code."""
    M, K = q_planes.shape
    N = codes.shape[0]
    dots = torch.empty((M, N, K // act_group), dtype=torch.int32, device=q_planes.device)
    _check("pq2_debug_group_dots_grouped", lib().pq2_debug_group_dots_grouped(
        _ptr(q_planes), _ptr(qsum), _ptr(codes), M, N, K, act_group, _ptr(dots), None,
        _stream(stream)))
    return dots


def pq2_ptq_prepare(raw: torch.Tensor, K: int, stream=None):
    """Raw PTQ1_0 rows u8[N][>= 28 K/128] (CUDA, unit column stride) ->
    (qs u8[N][24 K/128], side i32[N][K/128]: qh | d << 16)."""
    if raw.dim() != 2 or raw.stride(1) != 1 or raw.dtype != torch.uint8:
        raise ValueError("Expected a CUDA uint8 PTQ1_0 matrix")
    N = raw.shape[0]
    qs = torch.empty((N, K // GROUP * 24), dtype=torch.uint8, device=raw.device)
    side = torch.empty((N, K // GROUP), dtype=torch.int32, device=raw.device)
    _check("pq2_ptq_prepare", lib().pq2_ptq_prepare(_ptr(raw), raw.stride(0), N, K, _ptr(qs),
                                                     _ptr(side), _stream(stream)))
    return qs, side


def pq2_ptq_mmv(q_rows, sx, qsum, qs, side, act_group: int, y=None, out_dtype=torch.float32,
                flags=0, stream=None):
    """PTQ1_0 GEMV (M = 1..4) on row-layout grouped activations."""
    M, K = q_rows.shape
    N = qs.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=q_rows.device)
    _check("pq2_ptq_mmv", lib().pq2_ptq_mmv(
        _ptr(q_rows), _ptr(sx), _ptr(qsum), _ptr(qs), _ptr(side), _ptr(y), _DT[y.dtype], M, N,
        K, act_group, flags, _stream(stream)))
    return y


def pq2_ptq_linear(x, qs, side, act_group: int, y=None, out_dtype=torch.float32, stream=None):
    """Complete PTQ1_0 projection (M = 1..4): grouped quantisation + GEMV."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    N = qs.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    nbytes = lib().pq2_ptq_linear_workspace_bytes(M, K, act_group)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=x.device)
    _check("pq2_ptq_linear", lib().pq2_ptq_linear(
        _ptr(x), _DT[x.dtype], x.stride(0), M, N, K, _ptr(qs), _ptr(side), act_group, _ptr(y),
        _DT[y.dtype], _ptr(ws), ws.numel(), _stream(stream)))
    return y


def pq2_debug_ptq_dots(q_rows, qsum, qs, side, act_group: int, stream=None):
    """Exact partial dots [M][N][K/A] of the PTQ1_0 GEMV's device code."""
    M, K = q_rows.shape
    N = qs.shape[0]
    dots = torch.empty((M, N, K // act_group), dtype=torch.int32, device=q_rows.device)
    _check("pq2_debug_ptq_dots", lib().pq2_debug_ptq_dots(
        _ptr(q_rows), _ptr(qsum), _ptr(qs), _ptr(side), M, N, K, act_group, _ptr(dots),
        _stream(stream)))
    return dots


def pq2_mmv_gated(q_planes, sx, qsum, codes, scales, out=None, out_dtype=torch.float32,
                  flags=0, status=None, stream=None):
    """Gate/up GEMV with its gated activation, M = 1..8: codes/scales hold N
    rows (gate rows, then up rows); out[M][N/2] = silu(gate) * up."""
    M, K = q_planes.shape
    N = codes.shape[0]
    if out is None:
        out = torch.empty((M, N // 2), dtype=out_dtype, device=q_planes.device)
    _check("pq2_mmv_gated", lib().pq2_mmv_gated(
        _ptr(q_planes), _ptr(sx), _ptr(qsum), _ptr(codes), _ptr(scales), _ptr(out),
        _DT[out.dtype], M, N, K, flags, _ptr(status), _stream(stream)))
    return out


def pq2_linear_gated(x, codes, scales, out=None, out_dtype=torch.float32, workspace=None,
                     status=None, stream=None):
    """Complete gated call for M = 1..8: quantise x, then pq2_mmv_gated."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    N = codes.shape[0]
    if out is None:
        out = torch.empty((M, N // 2), dtype=out_dtype, device=x.device)
    if workspace is None:
        workspace = torch.empty(linear_workspace_bytes(M, K), dtype=torch.uint8,
                                device=x.device)
    _check("pq2_linear_gated", lib().pq2_linear_gated(
        _ptr(x), _DT[x.dtype], x.stride(0), M, N, K, _ptr(codes), _ptr(scales), _ptr(out),
        _DT[out.dtype], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream)))
    return out


def pq2_norm_hadamard_quantize(x, w, sign, eps, residual=None, layout: int = PQ2_Q_PLANES,
                               want_norm=False, want_residual=False, stream=None):
    """x bf16 [M][K] (CUDA), norm weight w bf16 [K], sign int8 [K] (+-1) ->
    (q, sx, qsum, norm_out or None, residual_out or None): RMSNorm, signs,
    1024-point Walsh-Hadamard and group-128 quantisation in one kernel."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D bf16 tensor")
    M, K = x.shape
    q = q_buffer(M, K, layout, x.device)
    sx = torch.empty((M, K // GROUP), dtype=torch.float32, device=x.device)
    qsum = torch.empty((M, K // GROUP), dtype=torch.int32, device=x.device)
    norm = torch.empty_like(x) if want_norm else None
    rout = torch.empty_like(x) if want_residual else None
    _check("pq2_norm_hadamard_quantize", lib().pq2_norm_hadamard_quantize(
        _ptr(x), _ptr(residual), _ptr(rout), _ptr(w), _ptr(sign), float(eps), M, K,
        _ptr(norm), _ptr(q), layout, _ptr(sx), _ptr(qsum), _stream(stream)))
    return q, sx, qsum, norm, rout


def q_buffer(M: int, K: int, layout: int, device):
    """Output buffer of the quantiser for `layout`: fp16 [M][K] (PQ2_Q_F16,
    PQ2_Q_MMV16), uint8 [M][2K] (the two e4m3 planes of PQ2_Q_F8) or int8
    [M][K]."""
    if layout in (PQ2_Q_F16, PQ2_Q_MMV16):
        return torch.empty((M, K), dtype=torch.float16, device=device)
    if layout == PQ2_Q_F8:
        return torch.empty((M, 2 * K), dtype=torch.uint8, device=device)
    return torch.empty((M, K), dtype=torch.int8, device=device)


def pq2_mm_f8(q_f8, sx, qsum, codes, scales, y=None, out_dtype=torch.float32, status=None,
              stream=None):
    """Prefill matmul (M >= 16; any M >= 1) on the 8-bit tcgen05 path (q from PQ2_Q_F8)."""
    M, K = q_f8.shape[0], q_f8.shape[1] // 2
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=q_f8.device)
    _check("pq2_mm_f8", lib().pq2_mm_f8(_ptr(q_f8), _ptr(sx), _ptr(qsum), _ptr(codes),
                                        _ptr(scales), _ptr(y), _DT[y.dtype], M, N, K,
                                        _ptr(status), _stream(stream)))
    return y


def pq2_mm(q_f16, sx, qsum, codes, scales, y=None, out_dtype=torch.float32, status=None,
           stream=None):
    """Prefill matmul (M >= 16; any M >= 1) on tcgen05 tensor cores."""
    M, K = q_f16.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=q_f16.device)
    _check("pq2_mm", lib().pq2_mm(_ptr(q_f16), _ptr(sx), _ptr(qsum), _ptr(codes), _ptr(scales),
                                  _ptr(y), _DT[y.dtype], M, N, K, _ptr(status),
                                  _stream(stream)))
    return y


def pq2_debug_group_dots(q, codes, path: int, qsum=None, dots=None, status=None,
                         stream=None):
    """Exact int32 group dots [M][N][K/128] from the kernels' own decode/dot code."""
    M, K = q.shape
    if path == PQ2_PATH_MM_F8:
        K //= 2
    N = codes.shape[0]
    if dots is None:
        dots = torch.empty((M, N, K // GROUP), dtype=torch.int32, device=q.device)
    _check("pq2_debug_group_dots",
           lib().pq2_debug_group_dots(_ptr(q), _ptr(qsum), _ptr(codes), M, N, K, path,
                                      _ptr(dots), _ptr(status), _stream(stream)))
    return dots


def pq2_mm_grouped(q_f16, sx, qsum, codes, scales, act_group: int, y=None,
                   out_dtype=torch.float32, status=None, stream=None):
    """Prefill matmul with activation groups of A (q from
    pq2_quantize_act_grouped, PQ2_Q_F16)."""
    M, K = q_f16.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=q_f16.device)
    _check("pq2_mm_grouped", lib().pq2_mm_grouped(
        _ptr(q_f16), _ptr(sx), _ptr(qsum), _ptr(codes), _ptr(scales), _ptr(y), _DT[y.dtype],
        M, N, K, act_group, _ptr(status), _stream(stream)))
    return y


def pq2_mm_f8_grouped(q_f8, sx, qsum, codes, scales, act_group: int, y=None,
                      out_dtype=torch.float32, status=None, stream=None):
    """pq2_mm_grouped on the 8-bit tensor path (q PQ2_Q_F8)."""
    M, K = q_f8.shape[0], q_f8.shape[1] // 2
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=q_f8.device)
    _check("pq2_mm_f8_grouped", lib().pq2_mm_f8_grouped(
        _ptr(q_f8), _ptr(sx), _ptr(qsum), _ptr(codes), _ptr(scales), _ptr(y), _DT[y.dtype],
        M, N, K, act_group, _ptr(status), _stream(stream)))
    return y


def pq2_debug_mm_dots_grouped(q, codes, path: int, act_group: int, dots=None, status=None,
                              stream=None):
    """Exact partial dots [M][N][K/A] of the grouped prefill kernels."""
    M, K = q.shape
    if path == PQ2_PATH_MM_F8:
        K //= 2
    N = codes.shape[0]
    if dots is None:
        dots = torch.empty((M, N, K // act_group), dtype=torch.int32, device=q.device)
    _check("pq2_debug_mm_dots_grouped", lib().pq2_debug_mm_dots_grouped(
        _ptr(q), path, _ptr(codes), M, N, K, act_group, _ptr(dots), _ptr(status),
        _stream(stream)))
    return dots


def linear_grouped_workspace_bytes(M: int, K: int, act_group: int) -> int:
    return lib().pq2_linear_grouped_workspace_bytes(M, K, act_group)


def pq2_linear_grouped(x, codes, scales, act_group: int, y=None, out_dtype=torch.float32,
                       workspace=None, status=None, stream=None):
    """Complete projection with activation groups of A: the grouped quantiser,
    then the grouped GEMV (M = 1..8) or the grouped prefill GEMM (M >= 9)."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    N = codes.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if workspace is None:
        workspace = torch.empty(linear_grouped_workspace_bytes(M, K, act_group),
                                dtype=torch.uint8, device=x.device)
    _check("pq2_linear_grouped", lib().pq2_linear_grouped(
        _ptr(x), _DT[x.dtype], x.stride(0), M, N, K, _ptr(codes), _ptr(scales), act_group,
        _ptr(y), _DT[y.dtype], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream)))
    return y


def mmv_geometry(N: int, K: int, sm_count: int):
    """(ctas, threads, splits, rows_max) of pq2_mmv for (N, K) — host only."""
    out = [ctypes.c_int() for _ in range(4)]
    _check("pq2_mmv_geometry", lib().pq2_mmv_geometry(
        N, K, sm_count, *[ctypes.addressof(o) for o in out]))
    return tuple(o.value for o in out)


def mmv_decoder(M: int) -> int:
    return lib().pq2_mmv_decoder(M)


def linear(x, codes, scales, out_dtype=torch.float32, stream=None):
    """The complete projection: pq2_linear (the GEMV for M <= 8, the
    prefill GEMM from M = 9)."""
    return pq2_linear(x, codes, scales, out_dtype=out_dtype, stream=stream)
