"""Host-side logic of bench.py (no GPU): the all-core oracle baseline splits
the output rows over threads and must equal the single-threaded oracle bit
for bit; the ncu traffic figure is reported only while the GEMV sources are
those it was captured from; the rotation rule keeps every call's weights out
of L2."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_threaded_oracle_call_equals_single_thread(orc):
    from oracle import oracle as O
    from ternary_weight_int8_gb300 import synth
    N, K = 37, 512
    raw = synth.raw_weights(N, K, seed=3)
    codes, scales = O.prepare(raw.numpy(), K)
    for M in (1, 3):
        x = synth.bits_u16(synth.activations(M, K, seed=9 + M, outlier_frac=0.01))
        y1 = O.linear(x, "bf16", codes, scales)
        for threads in (2, 5, 8):
            yt = bench.oracle_linear_threads(O, x, codes, scales, threads)
            assert yt.shape == (M, N)
            assert np.array_equal(yt.view(np.uint32), y1.view(np.uint32)), threads


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    assert isinstance(bench.recorded_traffic(), (int, type(None)))
    # a profile whose hash matches the given sources is reported ...
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel v1")
    import hashlib
    h = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    prof = tmp_path / "p.md"
    prof.write_text("# capture\n\ntraffic-record: kernel=x sources_sha256_16=%s "
                    "dram_bytes_per_launch=1234 algorithmic_bytes=1000\n" % h)
    monkeypatch.setattr(bench, "MMV_PROFILE", str(prof))
    monkeypatch.setattr(bench, "MMV_SOURCES", (str(src),))
    monkeypatch.setattr(bench, "ROOT", "/")
    assert bench.recorded_traffic() == 1234
    # ... and nulled once the source changes
    src.write_bytes(b"kernel v2")
    assert bench.recorded_traffic() is None
    # no record at all
    prof.write_text("# capture without a record\n")
    assert bench.recorded_traffic() is None


@pytest.mark.parametrize("l2,b,want", [(129 << 20, 13_926_400, 39), (129 << 20, 23_674_880, 23),
                                       (129 << 20, 47_349_760, 16), (1 << 20, 10 << 20, 16)])
def test_rotation_count(l2, b, want):
    n = bench.rotation_count(l2, b)
    assert n == want
    assert n >= 16 and n * b >= 4 * l2


def test_compact_summary_is_short():
    by_m = {str(M): {"mmv_us": 3.123 + M, "mmv_frac": 0.6543} for M in range(1, 9)}
    s = bench.compact(by_m, "mmv_us", "mmv_frac")
    assert s.startswith("1:4.12/0.65 2:5.12/0.65")
    assert len(s) <= 120
