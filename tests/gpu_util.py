"""Helpers for the GPU parity tests: seeded inputs on the device, oracle
references on the host, guard-banded output buffers."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from ternary_weight_int8_gb300 import synth

G = 128


def weights(N, K, seed, code_values=3, device="cuda", raw_pad=0):
    """Raw blocks on the device (row stride padded by raw_pad bytes) and the
    oracle's planes of the same bytes."""
    raw = synth.raw_weights(N, K, seed, device="cpu", code_values=code_values)
    if raw_pad:
        padded = torch.zeros((N, raw.shape[1] + raw_pad), dtype=torch.uint8)
        padded[:, :raw.shape[1]] = raw
        raw_dev = padded.to(device)[:, :raw.shape[1]]
    else:
        raw_dev = raw.to(device)
    codes_o, scales_o = O.prepare(raw.numpy(), K)
    return raw_dev, codes_o, scales_o


def guarded(shape, dtype, device="cuda", guard=64, fill=None):
    """A tensor view with `guard` elements of poison on both sides; returns
    (view, backing, poison value)."""
    n = int(np.prod(shape))
    backing = torch.empty(n + 2 * guard, dtype=dtype, device=device)
    if dtype.is_floating_point:
        poison = float("nan") if fill is None else fill
    else:
        poison = -0x5A5A5A5A if dtype == torch.int32 else (0x5A if dtype == torch.uint8 else -91)
    backing.fill_(poison)
    view = backing[guard:guard + n].view(shape)
    return view, backing, guard


def guards_intact(backing, guard):
    b = backing.detach().cpu()
    head, tail = b[:guard], b[-guard:]
    if b.dtype.is_floating_point:
        return bool(torch.isnan(head).all() and torch.isnan(tail).all())
    return bool((head == head[0]).all() and (tail == head[0]).all())


def x_bits(x):
    return synth.bits_u16(x) if x.dtype in (torch.bfloat16, torch.float16) else \
        x.detach().cpu().float().numpy()


def kind(x):
    return {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[x.dtype]


def oracle_reference(x, codes_o, scales_o):
    """(q, sx, qsum, dots, y32, y64, bound) from the oracle for activations x."""
    a = O.widen(x_bits(x), kind(x))
    q, sx = O.quantize(a)
    dots = O.group_dots(q, codes_o)
    y32, y64, bound = O.scale_accumulate(dots, sx, scales_o)
    return q, sx, O.qsum(q), dots, y32, y64, bound


def oracle_rows(x, rows, codes_o, scales_o, chunk=16, threads=None):
    """(y64, bound) of the oracle for the activation rows `rows` of x against
    every output row of the prepared planes, formed in chunks of `chunk`
    activation rows (the int32 dots of one chunk stay small) on a pool of
    host threads.  Quantisation is per row, so each chunk is the oracle's
    result for those rows exactly; the oracle's C calls release the
    interpreter lock."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    xs = x[torch.as_tensor(np.asarray(rows))]
    n = xs.shape[0]
    pieces = [(i, min(i + chunk, n)) for i in range(0, n, chunk)]

    def one(ab):
        a, b = ab
        *_, y64, bound = oracle_reference(xs[a:b], codes_o, scales_o)
        return y64, bound

    threads = threads or max(1, min(len(pieces), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(one, pieces))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def oracle_reference_grouped(x, codes_o, scales_o, A):
    """(q, sx, qsum, dots, y32, y64, bound) of the oracle with activation
    groups of A elements."""
    a = O.widen(x_bits(x), kind(x))
    q, sx = O.quantize_grouped(a, A)
    dots = O.group_dots_grouped(q, codes_o, A)
    y32, y64, bound = O.scale_accumulate_grouped(dots, sx, scales_o, A)
    return q, sx, O.qsum_grouped(q, A), dots, y32, y64, bound


def oracle_rows_grouped(x, rows, codes_o, scales_o, A, chunk=16, threads=None):
    """oracle_rows with activation groups of A elements."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    xs = x[torch.as_tensor(np.asarray(rows))]
    n = xs.shape[0]
    pieces = [(i, min(i + chunk, n)) for i in range(0, n, chunk)]

    def one(ab):
        a, b = ab
        *_, y64, bound = oracle_reference_grouped(xs[a:b], codes_o, scales_o, A)
        return y64, bound

    threads = threads or max(1, min(len(pieces), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(one, pieces))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def tile_rows(M, tile=128, total=64, seed=0):
    """Rows to compare at a large M: every row up to M = 512; above that,
    `total` seeded rows spread so that every tile of `tile` rows holds at
    least one (the first and last row always included)."""
    if M <= 512:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    tiles = (M + tile - 1) // tile
    per = max(1, -(-total // tiles))
    rows = {0, M - 1}
    for t in range(tiles):
        lo, hi = t * tile, min(M, (t + 1) * tile)
        rows.update(rng.choice(np.arange(lo, hi), min(per, hi - lo), replace=False).tolist())
    return np.array(sorted(rows))


def mm_operand_order(q: np.ndarray) -> np.ndarray:
    """The PQ2_Q_F16 layout (include/pq2.h): inside every 16 consecutive
    elements, element 4b + s goes to position 4s + 2(b & 1) + (b >> 1)."""
    M, K = q.shape
    out = np.empty_like(q)
    for i in range(16):
        b, s = i // 4, i % 4
        p = 4 * s + 2 * (b & 1) + (b >> 1)
        out[:, p::16] = q[:, i::16]
    return out


def mm_operand_order_f8(q: np.ndarray) -> np.ndarray:
    """The PQ2_Q_F8 layout (include/pq2.h) as bytes [M][2K]: per 128-group the
    e4m3 plane of 16a, then the e4m3 plane of b (q = 16a + b, b = q & 15);
    inside every 16 elements, element 8h + 2e + o sits at 4(2h + o) + e.
    The e4m3 bytes come from torch's float8_e4m3fn conversion."""
    M, K = q.shape
    qi = q.astype(np.int64)
    planes = [(qi >> 4) * 16, qi & 15]
    i = np.arange(16)
    pos = 4 * (2 * (i // 8) + (i % 2)) + (i % 8) // 2
    out = np.empty((M, K // G, 2, G), np.uint8)
    for p, v in enumerate(planes):
        b = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        b = b.reshape(M, K // 16, 16)
        r = np.empty_like(b)
        r[:, :, pos] = b
        out[:, :, p, :] = r.reshape(M, K // G, G)
    return out.reshape(M, 2 * K)


def mmv16_layout(q: np.ndarray) -> np.ndarray:
    """The PQ2_Q_MMV16 layout (include/pq2.h) as fp16 [M][K], built on the
    host from int8 q: inside every 128-group, position 32t + 4j + 2r + e
    holds element 16(t + 4(j // 4)) + 8e + f, f = 2(j % 4) + r, divided by
    4^f (f <= 4) or 4^(f - 3) (f >= 5)."""
    M, K = q.shape
    qg = q.reshape(M, K // G, G).astype(np.float64)
    out = np.empty((M, K // G, G), np.float64)
    for P in range(G):
        t, j, r, e = P // 32, (P % 32) // 4, (P % 4) // 2, P % 2
        f = 2 * (j % 4) + r
        i = 16 * (t + 4 * (j // 4)) + 8 * e + f
        out[:, :, P] = qg[:, :, i] / 4.0 ** (f if f <= 4 else f - 3)
    return out.astype(np.float16).reshape(M, K)


def mmv16_correction(q: np.ndarray) -> np.ndarray:
    """The PQ2_Q_MMV16 group corrections: sum over the group of
    q_i * (1 + 1024 / scale_i), scale_i the divisor of element i (its field
    f = i % 8 as above)."""
    M, K = q.shape
    f = np.arange(G) % 8
    wt = 1 + 1024 // 4 ** np.where(f <= 4, f, f - 3)
    return (q.reshape(M, K // G, G).astype(np.int64) * wt).sum(-1).astype(np.int32)


def host_mapped(t) -> bool:
    """True when the pinned host tensor `t` is addressable by the device at
    its own address (asked of the CUDA runtime, not by touching it)."""
    import ctypes

    class Attr(ctypes.Structure):
        _fields_ = [("type", ctypes.c_int), ("device", ctypes.c_int),
                    ("devicePointer", ctypes.c_void_p), ("hostPointer", ctypes.c_void_p),
                    ("reserved", ctypes.c_long * 16)]
    rt = None
    for name in ("libcudart.so", "libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    if rt is None:
        return False
    a = Attr()
    rc = rt.cudaPointerGetAttributes(ctypes.byref(a), ctypes.c_void_p(t.data_ptr()))
    return rc == 0 and a.type == 1 and a.devicePointer == t.data_ptr()
