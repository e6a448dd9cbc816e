"""bench.py's host-side arithmetic, on the CPU: the algorithmic bytes of a layer,
the roofline bound of a call, and the parsing of the clock samples taken during
the timed region.
"""
import pytest

import bench


@pytest.mark.parametrize("K,N,mb", [
    # Llama-2 projection shapes with their algorithmic bytes in MB (packed int4
    # K*N/2, bf16/fp16 scales G*N*2, 4-bit zeros G*N/2, G = K/128)
    (4096, 12288, 26.15), (4096, 4096, 8.72), (4096, 22016, 46.85), (11008, 4096, 23.43),
    (5120, 15360, 40.86), (5120, 27648, 73.54), (13824, 5120, 36.77),
    (8192, 10240, 43.58), (8192, 57344, 244.06), (28672, 8192, 122.03),
])
def test_alg_bytes_of_the_decode_layers(K, N, mb):
    assert round(bench.alg_bytes(K, N) / 1e6, 2) == mb


def test_alg_bytes_terms():
    # one group of 128 rows, 8 columns: 512 bytes of codes, 16 of scales, 4 of zeros
    assert bench.alg_bytes(128, 8) == 128 * 8 // 2 + 8 * 2 + 8 // 2
    # group -1 is one group over K
    assert bench.alg_bytes(4096, 16, group=4096) == 4096 * 16 // 2 + 16 * 2 + 16 // 2


def test_roofline_bound_flips_at_the_ridge():
    K, N, hbm, tc = 4096, 4096, 6791.4, 1902.7
    ridge = bench.alg_bytes(K, N) * tc * 1e12 / (hbm * 1e9 * 2.0 * N * K)
    assert 60 < ridge < 80
    for M in (1, 16, 64):
        bound, frac = bench.roofline_point(K, N, M, 1e-5, hbm, tc)
        assert bound == "hbm"
        assert frac == pytest.approx(bench.alg_bytes(K, N) / (hbm * 1e9) / 1e-5)
    for M in (128, 2048):
        bound, frac = bench.roofline_point(K, N, M, 1e-3, hbm, tc)
        assert bound == "tensor"
        assert frac == pytest.approx(2.0 * M * N * K / (tc * 1e12) / 1e-3)


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def test_clock_samples_are_parsed():
    s = bench.ClockSampler(0)
    s.proc = _FakeProc()
    s.lines = [
        "2070, 2070, 910.2, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "1995, 2070, 1350.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2040, 2070, 1200.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    out = s.stop()
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2040
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi():
    s = bench.ClockSampler(0)  # never started
    out = s.stop()
    assert out["sm_mhz"] is None and out["reasons"] == ["nvidia-smi unavailable"]
