"""Host-side bookkeeping pinned against numbers the pages print."""
import os

import pytest

from exact_io_aware_flash_gb300 import flops

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def test_flop_count_reproduces_sm75_throughput_tables():
    n = 0
    for d, causal, N, ms, tflops in _rows("sm75_throughput.txt"):
        f = flops.forward_flops(1, 8, int(N), int(d), bool(int(causal)))
        got = f / (float(ms) * 1e-3) / 1e12
        # printed to two decimals
        assert abs(got - float(tflops)) <= 0.0051, (d, causal, N, got, tflops)
        n += 1
    assert n == 9


def test_materialised_score_memory_matches_worked_example():
    scale = {"MB": 1e6, "GB": 1e9, "MiB": 2 ** 20}
    for N, heads, value, unit in _rows("score_matrix_memory.txt"):
        got = flops.materialised_score_bytes(int(N), int(heads)) / scale[unit]
        # the pages round to two significant figures ("~ 8.6 GB", "~ 550 GB")
        assert got == pytest.approx(float(value), rel=0.02), (N, heads, got, value, unit)


def test_backward_is_two_and_a_half_forwards():
    assert flops.backward_flops(2, 3, 100, 64, True) == 2.5 * flops.forward_flops(2, 3, 100, 64, True)
