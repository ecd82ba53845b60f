"""Host-side FLOP bookkeeping of the sliding-window workload, checked by brute force."""
import numpy as np

from exact_io_aware_flash_gb300.flops import (backward_flops_window, forward_flops,
                                              forward_flops_window, window_pairs)


def brute_pairs(N, W):
    i = np.arange(N)[:, None]
    k = np.arange(N)[None, :]
    return int(((k <= i) & (k > i - W)).sum())


def test_window_pairs_brute_force():
    for N in (1, 2, 7, 128, 129, 300):
        for W in (1, 2, 5, 127, 128, 129, 299, 300, 301, 1000):
            assert window_pairs(N, W) == brute_pairs(N, W), (N, W)


def test_window_flops_limits():
    # width 1: each row sees itself only
    assert forward_flops_window(2, 3, 50, 64, 1) == 4.0 * 64 * 2 * 3 * 50
    # W >= N: the causal pair count N(N+1)/2 (the causal convention N^2/2 differs by N/2)
    N, d = 4096, 128
    assert window_pairs(N, N) == N * (N + 1) // 2
    assert abs(forward_flops_window(1, 1, N, d, N) - forward_flops(1, 1, N, d, True)) == 4.0 * d * N / 2
    assert backward_flops_window(1, 2, 300, 64, 100) == 2.5 * forward_flops_window(1, 2, 300, 64, 100)
