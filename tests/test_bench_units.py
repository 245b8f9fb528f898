"""The benchmark's algorithmic units, against sizes worked out by hand from
the workload definitions (tensor shapes x element sizes; five matrix products
over the causal half)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_decode_step_bytes():
    # K and V bf16 [64][1024][5][128] read: 2 * 83,886,080 B; dK and dV f32
    # written: 2 * 167,772,160 B; q, dout read and dq written, f32
    # [64][20][128]: 3 * 655,360 B
    assert bench.decode_bytes() == 2 * 83_886_080 + 2 * 167_772_160 + 3 * 655_360 == 505_282_560
    # an f32 cache doubles the K/V reads only
    assert bench.decode_bytes(kv_es=4) - bench.decode_bytes() == 2 * 83_886_080


def test_rmsnorm_step_bytes():
    # 64 rows of 2560: x, dy read and dx written (f32), gamma read once
    assert bench.rmsnorm_bytes(64, 2560) == 64 * 2560 * 12 + 2560 * 4 == 1_976_320


@pytest.mark.parametrize("B,T,H,D,flops", [
    (4, 2048, 20, 128, 214_748_364_800.0),      # the T = 2048 workload, 2.147e11
    (1, 8192, 32, 128, 1_374_389_534_720.0),    # the long-context workload, 1.374e12
    (2, 512, 20, 128, 6_710_886_400.0),         # one layer of the chain, 6.71e9
])
def test_causal_flops(B, T, H, D, flops):
    # five products of 2 * D flops per (query, key) pair over T^2 / 2 pairs
    assert bench.causal_flops(B, T, H, D) == flops


def test_job_rate_units():
    # 505,282,560 B in 0.1116 ms is 4.53 TB/s
    assert bench.job_rate(505_282_560, 1, 0.1116) / 1e9 == pytest.approx(4527.6, rel=1e-4)


def test_recorded_traffic_is_keyed_to_the_kernel_sources():
    # a record is used only while the hash of its kernel's source files matches
    assert bench.recorded_traffic("decode_bwd_kernel", ["rows.cu"]) is None
    assert bench.recorded_traffic("no_such_kernel", ["decode.cu"]) is None
    for key, files in (("decode_bwd_kernel", ["decode.cu", "abw_device.cuh"]),
                       ("causal_kv_tc_kernel", ["causal.cu", "abw_device.cuh", "tcgen05.cuh"])):
        v = bench.recorded_traffic(key, files)
        assert v is None or (isinstance(v, int) and v > 0)
